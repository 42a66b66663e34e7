"""Pins for the oracle's quantizers: hand-worked examples (tests/golden/),
invariants the recipe states (UE8M0 scales rounded up so the range is never
exceeded; MX blocks clamp beyond the largest code), exact FP8 inputs
quantizing to themselves, and torch's float8 cast as a library special case."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import E4M3, E5M2
from golden_io import load_quant_examples
from fp8_hybrid_granularity_gb300 import workloads

TORCH_DT = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}
FMT = {"e4m3": E4M3, "e5m2": E5M2}


def _decode(q, fmt):
    """Decode codes with torch's float8 view (independent of the oracle)."""
    return torch.from_numpy(np.ascontiguousarray(q)).view(TORCH_DT[fmt]).to(torch.float64).numpy()


def _bits_to_f64(x_bits):
    return workloads.from_bits(x_bits).to(torch.float64).numpy()


@pytest.mark.parametrize("case", load_quant_examples(), ids=lambda c: c["case"])
def test_hand_worked_examples(case):
    x = case["x"][None, :]
    fmt = FMT[case["fmt"]]
    if case["mode"] == "row":
        q, s = oracle.quant_token(x, 0, fmt)
        clamped = 0
    else:
        q, s, clamped = oracle.quant_mx32(x, fmt)
    assert s.ravel().tolist() == [case["scale"]]
    assert q.ravel().tolist() == case["q"].tolist(), [hex(v) for v in q.ravel()]
    assert clamped == case["clamped"]


def _exact_fp8_groups(rng, rows, cols, fmt, k_per_row):
    """BF16 inputs that are FP8 grid values times 2^k, with the row max in
    (FMAX/2, FMAX]*2^k, so that a per-row UE8M0 quantization must return the
    same codes and scale byte k+127."""
    top = 0x70 if fmt == E4M3 else 0x74   # codes of 256 / 32768 (> FMAX/2)
    maxc = 0x7E if fmt == E4M3 else 0x7B
    codes = rng.integers(0, maxc + 1, (rows, cols)).astype(np.uint8)
    codes[:, rng.integers(0, cols)] = rng.integers(top, maxc + 1, rows)
    codes |= (rng.integers(0, 2, (rows, cols)) << 7).astype(np.uint8)
    vals = _decode(codes, fmt) * np.exp2(k_per_row)[:, None]
    bits = workloads.bf16_bits(torch.from_numpy(vals).to(torch.bfloat16))
    assert np.array_equal(_bits_to_f64(bits), vals)       # exactly representable
    return bits, codes


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_exact_fp8_inputs_quantize_to_themselves(fmt):
    rng = np.random.default_rng(21 + fmt)
    k = rng.integers(-20, 20, 64)
    bits, codes = _exact_fp8_groups(rng, 64, 96, fmt, k)
    q, s = oracle.quant_token(bits, 0, fmt)
    assert np.array_equal(s[:, 0].astype(int), k + 127)
    # +-0 codes: the oracle keeps the sign of a zero input, which is what the
    # BF16 input carries
    assert np.array_equal(q, codes)


def _random_act(rows, cols, seed, kind="act"):
    t = workloads.make_tensor(kind, rows, cols, seed, "pin")
    return workloads.bf16_bits(t)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("group", [0, 128])
def test_token_quant_invariants(fmt, group):
    x = _random_act(64, 512, 3 + fmt + group)
    q, s = oracle.quant_token(x, group, fmt)
    xf = _bits_to_f64(x)
    fmax = oracle.fp8_max(fmt)
    deq_codes = _decode(q, fmt)
    g = 512 if group == 0 else group
    e = s.astype(np.int64) - 127
    e_full = np.repeat(e, g, axis=1)
    # scale: power of two rounded up -> tight bound on the group amax
    amax = np.abs(xf).reshape(64, -1, g).max(axis=2)
    r = amax / np.exp2(e)
    assert (r <= fmax).all() and (r > fmax / 2).all()
    # codes never saturate or go NaN in the UE8M0 mode
    assert np.isfinite(deq_codes).all() and (np.abs(deq_codes) <= fmax).all()
    # error bound of one rounding: half a code spacing at the value
    xhat = deq_codes * np.exp2(e_full)
    mbits = 3 if fmt == E4M3 else 2
    min_normal_exp = -6 if fmt == E4M3 else -14
    spacing_exp = np.maximum(np.floor(np.log2(np.maximum(np.abs(xf), 1e-300))) - e_full,
                             min_normal_exp) - mbits
    assert (np.abs(xf - xhat) <= np.exp2(spacing_exp + e_full - 1)).all()
    # sign symmetry
    qn, sn = oracle.quant_token(x ^ np.uint16(0x8000), group, fmt)
    assert np.array_equal(sn, s) and np.array_equal(qn, q ^ np.uint8(0x80))
    # monotone within each group
    for row in range(0, 64, 7):
        order = np.argsort(xf[row, :g], kind="stable")
        assert (np.diff(deq_codes[row, :g][order]) >= 0).all()


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_token_quant_matches_torch_cast(fmt):
    """With the scale fixed by the rule, codes = torch's RNE cast of x*2^-e."""
    x = _random_act(32, 1024, 9 + fmt)
    q, s = oracle.quant_token(x, 128, fmt)
    xf = torch.from_numpy(_bits_to_f64(x)).float()
    e = torch.from_numpy(s.astype(np.int64) - 127).repeat_interleave(128, dim=1)
    y = xf * torch.exp2(-e.float())            # exact power-of-two scaling
    ref = y.to(TORCH_DT[fmt]).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)


def test_group_structure():
    """A 1x128 group equals the per-row quantization of that 128-wide slice;
    the transposed variant equals the plain one applied to x^T."""
    x = _random_act(256, 384, 31)
    q, s = oracle.quant_token(x, 128, E4M3)
    for j in range(3):
        qj, sj = oracle.quant_token(np.ascontiguousarray(x[:, 128 * j:128 * (j + 1)]), 0, E4M3)
        assert np.array_equal(q[:, 128 * j:128 * (j + 1)], qj)
        assert np.array_equal(s[:, j], sj[:, 0])
    qt, st = oracle.quant_token(x, 128, E4M3, transpose=True)
    q2, s2 = oracle.quant_token(np.ascontiguousarray(x.T), 128, E4M3)
    assert np.array_equal(qt, q2) and np.array_equal(st, s2)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_block128(fmt):
    x = workloads.bf16_bits(workloads.make_tensor("weight", 256, 384, 4, "pin"))
    q, s, qt, st = oracle.quant_block128(x, fmt, transposed_copy=True)
    assert np.array_equal(qt, q.T) and np.array_equal(st, s.T)
    # each block = per-row quantization of the flattened block (one group)
    for rb in range(2):
        for cb in range(3):
            blk = np.ascontiguousarray(x[128 * rb:128 * (rb + 1), 128 * cb:128 * (cb + 1)])
            qb, sb = oracle.quant_token(blk.reshape(1, -1), 0, fmt)
            assert sb[0, 0] == s[rb, cb]
            assert np.array_equal(qb.reshape(128, 128), q[128 * rb:128 * (rb + 1), 128 * cb:128 * (cb + 1)])
    # the amax must see the whole block: one large value moves the whole block's scale
    x2 = x.copy()
    x2[5, 7] = 0x4300  # 128.0
    q2, s2, _, _ = oracle.quant_block128(x2, fmt)
    assert s2[0, 0] != s[0, 0] and (s2[0, 1:] == s[0, 1:]).all() and (s2[1] == s[1]).all()


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_mx32_rules(fmt):
    x = _random_act(64, 256, 41, kind="mx_ln_clamp")
    q, s, clamped = oracle.quant_mx32(x, fmt)
    xf = _bits_to_f64(x)
    fmax = oracle.fp8_max(fmt)
    emax = 8 if fmt == E4M3 else 15
    e = s.astype(np.int64) - 127
    amax = np.abs(xf).reshape(64, -1, 32).max(axis=2)
    r = amax / np.exp2(e)
    assert ((r >= 2.0 ** emax) & (r < 2.0 ** (emax + 1))).all()
    y = np.abs(xf) / np.exp2(np.repeat(e, 32, axis=1))
    maxc = 0x7E if fmt == E4M3 else 0x7B
    assert clamped == int((y > fmax).sum())
    # top code iff the scaled magnitude reaches the RNE midpoint below the max
    t = oracle.decode_table(fmt)
    top_mid = (t[maxc] + t[maxc - 1]) / 2
    top = (q & 0x7F) == maxc
    # a tie at the midpoint goes to the even mantissa: the top code for E4M3
    # (0x7E, mantissa 110), the code below it for E5M2 (0x7B has mantissa 11)
    expect = (y > top_mid) | ((y == top_mid) & (maxc % 2 == 0))
    assert np.array_equal(top, expect)
    # saturated elements are exactly those beyond the maximum
    assert np.array_equal((y > fmax), top & (y > fmax))


def test_mx32_layernorm_rows():
    """The layer-norm-like rows at 1 +- 1e-3 all collapse to one code
    (amax > 1 so the block's power of two is 2^0 and every value rounds to
    256 * 2^-8); rows at [0.998, 1.0] clamp entirely to the top code."""
    x = _random_act(8, 64, 43, kind="mx_ln")
    q, s, clamped = oracle.quant_mx32(x, E4M3)
    xf = _bits_to_f64(x)
    ln = xf[:4]
    rows_gt1 = (np.abs(ln).reshape(4, -1, 32).max(axis=2) >= 1.0)
    assert (s[:4][rows_gt1] == 119).all()
    xc = _random_act(8, 64, 44, kind="mx_ln_clamp")
    qc, sc, cc = oracle.quant_mx32(xc, E4M3)
    amaxc = np.abs(_bits_to_f64(xc)[:4]).reshape(4, -1, 32).max(axis=2)
    assert (amaxc < 1.0).all()
    assert ((qc[:4] & 0x7F) == 0x7E).all()


def test_nonfinite_groups():
    x = _random_act(2, 256, 50)
    x[0, 3] = 0x7FC0   # NaN
    x[1, 200] = 0xFF80  # -inf
    q, s = oracle.quant_token(x, 128, E4M3)
    assert s[0, 0] == 0xFF and (q[0, :128] == 0x7F).all()
    assert s[0, 1] != 0xFF
    assert s[1, 1] == 0xFF and (q[1, 128:] == 0x7F).all()
    qm, sm, _ = oracle.quant_mx32(x, E5M2)
    assert sm[0, 0] == 0xFF and (qm[0, :32] == 0x7F).all() and sm[0, 1] != 0xFF


def test_zero_group():
    x = np.zeros((1, 128), np.uint16)
    x[0, 1] = 0x8000
    q, s = oracle.quant_token(x, 128, E4M3)
    assert s[0, 0] == 0 and q[0, 0] == 0 and q[0, 1] == 0x80
    q, s, _ = oracle.quant_mx32(x, E4M3)
    assert (s == 0).all()
