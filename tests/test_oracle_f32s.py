"""Pins for the oracle's FP32-scale variant: hand-worked cases
(tests/golden/f32_scale_examples.txt), an independent route through numpy's
single-precision arithmetic and torch's FP8 casts, the reduction to the UE8M0
quantizer when every group's amax is FMAX times a power of two, and the
one-rounding error bound."""
import numpy as np
import pytest
import torch

import oracle
from oracle import E4M3, E5M2, GRAN_ROW, GRAN_1x128, GRAN_128x128
from fp8_hybrid_granularity_gb300 import workloads
from golden_io import load_quant_examples

FMT = {"e4m3": E4M3, "e5m2": E5M2}
TORCH_FP8 = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}


@pytest.mark.parametrize("case", load_quant_examples("f32_scale_examples.txt"),
                         ids=lambda c: c["case"])
def test_hand_worked(case):
    fmt = FMT[case["fmt"]]
    q, s = oracle.quant_token_f32s(case["x"].reshape(1, -1), 0, fmt)
    assert np.array_equal(q.ravel(), case["q"])
    assert int(s.view(np.uint32)[0, 0]) == case["scale_f32"]


def _numpy_torch_route(xb, group, fmt):
    """The same definition through numpy float32 arithmetic and torch's
    (round-to-nearest-even) FP8 cast."""
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).float().numpy()
    rows, cols = x.shape
    g = cols if group == 0 else group
    fmax = np.float32(oracle.fp8_max(fmt))
    xg = x.reshape(rows, cols // g, g)
    amax = np.abs(xg).max(axis=2).astype(np.float32)
    safe = np.where(amax == 0, np.float32(1), amax)
    d = np.where(amax == 0, np.float32(1), safe / fmax).astype(np.float32)
    m = np.where(amax == 0, np.float32(1), fmax / safe).astype(np.float32)
    y = (xg * m[:, :, None]).astype(np.float32)
    y = np.clip(y, -fmax, fmax)                      # saturation (never reached but defined)
    q = torch.from_numpy(y.reshape(rows, cols)).to(TORCH_FP8[fmt]).view(torch.uint8).numpy()
    return q, d


@pytest.mark.parametrize("group", [0, 128])
@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_independent_route(group, fmt):
    x = workloads.bf16_bits(workloads.make_tensor("act", 64, 512, 50 + group + fmt, "f32s"))
    q, s = oracle.quant_token_f32s(x, group, fmt)
    q2, d2 = _numpy_torch_route(x, group, fmt)
    assert np.array_equal(q, q2)
    assert np.array_equal(s.view(np.uint32), d2.view(np.uint32))


def test_block_route_and_transposed_copy():
    w = workloads.bf16_bits(workloads.make_tensor("weight", 256, 384, 52, "f32b"))
    q, s, qt, st = oracle.quant_block128_f32s(w, E4M3, transposed_copy=True)
    for rb in range(2):
        for cb in range(3):
            blk = w[128 * rb:128 * rb + 128, 128 * cb:128 * cb + 128]
            q2, d2 = _numpy_torch_route(blk.reshape(1, -1), 0, E4M3)
            assert np.array_equal(q[128 * rb:128 * rb + 128, 128 * cb:128 * cb + 128].ravel(), q2.ravel())
            assert s[rb, cb] == d2[0, 0] and st[cb, rb] == d2[0, 0]
    assert np.array_equal(qt, q.T)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_power_of_two_ratio_reduces_to_ue8m0(fmt):
    """Scale each row so its amax is exactly FMAX * 2^k: then d = 2^k and
    m = 2^-k exactly, and the codes must be the UE8M0 quantizer's."""
    x = workloads.make_tensor("act", 32, 256, 53, "p2").float()
    k = torch.arange(-8, 24).float()[:, None]
    amax = x.abs().amax(dim=1, keepdim=True)
    fmax = oracle.fp8_max(fmt)
    xs = (x / amax * fmax * torch.pow(2.0, k)).to(torch.bfloat16)
    # keep only rows whose amax survived the BF16 rounding exactly
    ok = (xs.float().abs().amax(dim=1) == (fmax * torch.pow(2.0, k[:, 0])))
    xb = workloads.bf16_bits(xs[ok])
    q, s = oracle.quant_token_f32s(xb, 0, fmt)
    qu, su = oracle.quant_token(xb, 0, fmt)
    assert ok.sum() >= 16
    assert np.array_equal(q, qu)
    assert np.array_equal(s[:, 0].astype(np.float64), np.exp2(su[:, 0].astype(np.float64) - 127))


def test_error_bound_and_range():
    """|x - decode(q) * d| is at most half the FP8 spacing at |x|/d (one
    rounding, widened by the FP32 rounding of m and of x*m), and every code is
    finite."""
    x = workloads.bf16_bits(workloads.make_tensor("grad", 64, 512, 54, "eb"))
    for fmt in (E4M3, E5M2):
        q, s = oracle.quant_token_f32s(x, 128, fmt)
        xd = oracle.dequant_f32s(q, s, GRAN_1x128, fmt)
        xv = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy()
        dec = oracle.decode_table(fmt)
        assert np.isfinite(dec[q]).all()
        grid = np.sort(dec[:128][np.isfinite(dec[:128])])
        d = np.repeat(s.astype(np.float64), 128, axis=1)
        y = np.abs(xv) / d
        k = np.minimum(np.searchsorted(grid, y), len(grid) - 1)
        step = grid[k] - grid[np.maximum(k - 1, 0)]
        assert (np.abs(xv - xd) <= (0.5 * step * (1 + 2.0 ** -20) + 2.0 ** -20 * y) * d).all()


def test_dequant_layouts():
    q = np.full((256, 256), 0x38, np.uint8)          # 1.0 everywhere
    srow = np.arange(1, 257, dtype=np.float32)[:, None]
    assert np.array_equal(oracle.dequant_f32s(q, srow, GRAN_ROW, E4M3)[:, 0], srow[:, 0])
    sblk = np.array([[1, 2], [3, 4]], np.float32)
    d = oracle.dequant_f32s(q, sblk, GRAN_128x128, E4M3)
    assert d[0, 0] == 1 and d[0, 200] == 2 and d[200, 0] == 3 and d[255, 255] == 4
