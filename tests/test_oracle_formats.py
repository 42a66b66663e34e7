"""Pins for the oracle's FP8 / BF16 format code, against things other than the
oracle itself: closed forms of the format definitions ("FP8 Formats for Deep
Learning", abstract / core claim), the E4M3 code-gap figure ("Characterization
and Mitigation of Training Instabilities in Microscaling Formats", Figure 5),
and torch's own CPU float8 casts where the definitions coincide."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import E4M3, E5M2

TORCH_DT = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}


def _torch_decode(fmt):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(TORCH_DT[fmt]).to(torch.float64).numpy()


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_decode_matches_torch_for_all_256_codes(fmt):
    ours = oracle.decode_table(fmt)
    ref = _torch_decode(fmt)
    nan_o, nan_r = np.isnan(ours), np.isnan(ref)
    assert (nan_o == nan_r).all()
    assert np.array_equal(ours[~nan_o], ref[~nan_r])
    # signed zero of 0x80
    assert math.copysign(1.0, ours[0x80]) == -1.0


def test_e4m3_closed_forms():
    t = oracle.decode_table(E4M3)
    assert t[0x7E] == 448.0 == 1.75 * 2 ** 8
    assert t[0x08] == 2.0 ** -6          # smallest normal
    assert t[0x01] == 2.0 ** -9          # smallest subnormal
    assert t[0x07] == 7 * 2.0 ** -9
    assert t[0x38] == 1.0                # exponent field 7 = bias
    nan_codes = [c for c in range(256) if math.isnan(t[c])]
    assert nan_codes == [0x7F, 0xFF]     # a single NaN mantissa pattern per sign
    assert not np.isinf(t).any()         # no infinities
    assert np.isfinite(t).sum() == 254
    assert oracle.fp8_max(E4M3) == 448.0


def test_e5m2_closed_forms():
    t = oracle.decode_table(E5M2)
    assert t[0x7B] == 57344.0 == 1.75 * 2 ** 15
    assert t[0x04] == 2.0 ** -14
    assert t[0x01] == 2.0 ** -16
    assert t[0x3C] == 1.0
    assert t[0x7C] == math.inf and t[0xFC] == -math.inf
    nan_codes = [c for c in range(256) if math.isnan(t[c])]
    assert nan_codes == [0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF]
    assert np.isfinite(t).sum() == 248
    assert oracle.fp8_max(E5M2) == 57344.0


def test_e4m3_code_gap_figure():
    """Relative gap between successive positive normal E4M3 codes runs from
    12.5% (1/8) down to about 6.6% (1/15) within every binade."""
    t = oracle.decode_table(E4M3)
    for ef in range(1, 16):
        gaps = []
        for m in range(8):
            c = (ef << 3) | m
            if c + 1 > 0x7E:
                break
            gaps.append((t[c + 1] - t[c]) / t[c])
        assert gaps[0] == 1 / 8
        if len(gaps) == 8:
            assert gaps[-1] == pytest.approx(1 / 15, rel=0, abs=1e-15)
        assert all(a > b for a, b in zip(gaps, gaps[1:]))


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_encode_decode_round_trip_all_codes(fmt):
    t = oracle.decode_table(fmt)
    for c in range(256):
        if math.isnan(t[c]):
            assert oracle.fp8_encode(t[c], fmt) == 0x7F
        else:
            assert oracle.fp8_encode(t[c], fmt) == c, hex(c)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_rne_midpoints_and_neighbours(fmt):
    t = oracle.decode_table(fmt)
    maxc = 0x7E if fmt == E4M3 else 0x7B
    for c in range(maxc):
        lo, hi = t[c], t[c + 1]
        mid = (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        assert oracle.fp8_encode(mid, fmt) == even
        assert oracle.fp8_encode(np.nextafter(mid, np.inf), fmt) == c + 1
        assert oracle.fp8_encode(np.nextafter(mid, -np.inf), fmt) == c
        assert oracle.fp8_encode(-mid, fmt) == (even | 0x80)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_encode_matches_torch_cast_in_range(fmt):
    """Random float32 values inside the format's range, rounded by torch's
    CPU float8 cast (a library implementation of the same RNE rule)."""
    g = torch.Generator().manual_seed(11 + fmt)
    fmax = 448.0 if fmt == E4M3 else 57344.0
    mag = torch.exp2(torch.rand(20000, generator=g) * (math.log2(fmax) + 20) - 20)
    sign = torch.where(torch.rand(20000, generator=g) < 0.5, -1.0, 1.0)
    y = (mag * sign).float().clamp(-fmax, fmax)
    ref = y.to(TORCH_DT[fmt]).view(torch.uint8).numpy()
    ours = np.array([oracle.fp8_encode(float(v), fmt) for v in y.tolist()], np.uint8)
    assert np.array_equal(ours, ref)


def test_signed_zero_and_underflow():
    assert oracle.fp8_encode(-0.0, E4M3) == 0x80
    assert oracle.fp8_encode(0.0, E4M3) == 0x00
    assert oracle.fp8_encode(-(2.0 ** -12), E4M3) == 0x80
    assert oracle.fp8_encode(2.0 ** -12, E4M3) == 0x00
    assert oracle.fp8_encode(-(2.0 ** -18), E5M2) == 0x80


def test_overflow_rules():
    # saturating (MX clamp): anything beyond the largest value gives it
    assert oracle.fp8_encode(1000.0, E4M3, saturate=True) == 0x7E
    assert oracle.fp8_encode(-1e6, E4M3, saturate=True) == 0xFE
    assert oracle.fp8_encode(1e9, E5M2, saturate=True) == 0x7B
    assert oracle.fp8_encode(-1e9, E5M2, saturate=True) == 0xFB
    # non-saturating: below the midpoint past the max rounds down to the max
    assert oracle.fp8_encode(460.0, E4M3) == 0x7E
    assert oracle.fp8_encode(464.0, E4M3) == 0x7F        # no infinity: NaN
    assert oracle.fp8_encode(61439.0, E5M2) == 0x7B
    assert oracle.fp8_encode(61440.0, E5M2) == 0x7C      # IEEE-like: infinity
    assert oracle.fp8_encode(-61440.0, E5M2) == 0xFC


def test_bf16_decode_matches_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    sample = np.random.default_rng(0).choice(65536, 4000, replace=False)
    sample = np.concatenate([sample, [0, 1, 0x7F, 0x80, 0x7F80, 0xFF80, 0x7FC0, 0x8000, 0x8001]])
    for b in sample:
        ours = oracle.bf16_to_double(int(bits[b]))
        r = ref[b]
        if math.isnan(r):
            assert math.isnan(ours)
        else:
            assert ours == r and math.copysign(1, ours) == math.copysign(1, r)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_ue8m0_exponent_is_the_tight_round_up(fmt):
    """The round-up rule is the unique e with FMAX/2 < amax/2^e <= FMAX
    (unless clamped at -127); checked on random BF16 magnitudes."""
    fmax = oracle.fp8_max(fmt)
    rng = np.random.default_rng(5 + fmt)
    bits = rng.integers(0, 0x7F80, 5000).astype(np.uint16)
    for b in bits:
        amax = oracle.bf16_to_double(int(b))
        e = oracle.ue8m0_exp(amax, fmt)
        assert -127 <= e <= 127
        r = amax / 2.0 ** e
        assert r <= fmax
        if e > -127:
            assert r > fmax / 2
    assert oracle.ue8m0_exp(0.0, fmt) == -127
    assert oracle.ue8m0_exp(math.nan, fmt) == 128
    assert oracle.ue8m0_exp(math.inf, fmt) == 128
    assert oracle.ue8m0_exp(fmax, fmt) == 0
    assert oracle.ue8m0_exp(np.nextafter(fmax, np.inf), fmt) == 1


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_mx_exponent_floor_rule(fmt):
    """MX: 2^emax <= amax/2^e < 2^(emax+1) whenever e is not clamped."""
    emax = 8 if fmt == E4M3 else 15
    rng = np.random.default_rng(7 + fmt)
    bits = rng.integers(1, 0x7F80, 5000).astype(np.uint16)
    for b in bits:
        amax = oracle.bf16_to_double(int(b))
        e = oracle.mx_exp(amax, fmt)
        r = amax / 2.0 ** e
        if -127 < e < 127:
            assert 2.0 ** emax <= r < 2.0 ** (emax + 1)
        else:
            assert e == -127 and r < 2.0 ** (emax + 1)
    assert oracle.mx_exp(1.0, E4M3) == -8
    assert oracle.mx_exp(0.0, fmt) == -127
