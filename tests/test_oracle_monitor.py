"""Pins for the oracle's MX clamp monitor: a hand-worked fixture
(tests/golden/mx_monitor_examples.txt), the closed forms of the two
layer-norm-like workloads, an independent threshold characterization of the
last bin on random data, and consistency with the plain MX quantizer."""
import math

import numpy as np
import pytest

import oracle
from oracle import E4M3, E5M2
from fp8_hybrid_granularity_gb300 import workloads
from golden_io import load_quant_examples


def test_hand_worked_fixture():
    (c,) = load_quant_examples("mx_monitor_examples.txt")
    x = c["x"].reshape(c["rows"], -1)
    q, s, st, rs = oracle.mx32_monitor(x, E4M3)
    for k in oracle.MX_STAT_NAMES:
        assert st[k] == c[k], k
    assert list(rs) == c["row_sat"]


def _ln_rows(lo, hi, rows, cols, seed):
    import torch
    g = torch.Generator().manual_seed(seed)
    t = lo + (hi - lo) * torch.rand(rows, cols, generator=g)
    return workloads.bf16_bits(t.to(torch.bfloat16))


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_layernorm_rows_collapse_without_clamping(fmt):
    """Values 1 +- 1e-3: a block's amax is just above 1, so e = -emax and every
    scaled value lies within 0.1% of 2^emax, inside one rounding interval of
    the code for 2^emax (E4M3 spacing 32 around 256, E5M2 8192 around 32768):
    every block collapses onto that code and nothing saturates.  (A block
    whose 32 values all fell below 1 would saturate as a whole and still
    collapse; at this seed none does.)"""
    x = _ln_rows(0.999, 1.001, 64, 512, 5)
    q, s, st, rs = oracle.mx32_monitor(x, fmt)
    nblk = x.size // 32
    assert st["blocks_collapsed"] == nblk
    assert st["saturated"] == 0 and st["top_code"] == 0 and st["blocks_saturated"] == 0
    one = oracle.fp8_encode(2.0 ** (8 if fmt == E4M3 else 15), fmt)
    assert (q == one).all()
    assert not rs.any()


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_clamp_rows_saturate_entirely(fmt):
    """Values in [0.990, 0.997]: amax < 1 so e = -1 - emax; scaled values lie
    in [0.99, 0.997] * 2^(emax+1), above FMAX = 1.75 * 2^emax: every element
    saturates to the largest code, every block is saturated and collapsed."""
    rows, cols = 16, 256
    x = _ln_rows(0.990, 0.997, rows, cols, 6)
    q, s, st, rs = oracle.mx32_monitor(x, fmt)
    top = oracle.fp8_encode(oracle.fp8_max(fmt), fmt)
    assert (q == top).all()
    assert st == {"saturated": x.size, "top_code": x.size, "blocks_saturated": x.size // 32,
                  "blocks_collapsed": x.size // 32}
    assert (rs == cols).all()


def test_last_bin_threshold_on_random_blocks():
    """Independent route: with X = 2^(floor(log2 amax) - 8), an E4M3 element
    lands in the last bin iff |x|/X >= 432 (the midpoint of 416 and 448; the
    tie rounds to 448's even mantissa) and saturates iff |x|/X > 448."""
    x = workloads.bf16_bits(workloads.make_tensor("normal", 48, 1024, 9, "mon"))
    _, _, st, rs = oracle.mx32_monitor(x, E4M3)
    sat = top = bsat = 0
    row_sat = []
    for r in range(x.shape[0]):
        rsum = 0
        for c0 in range(0, x.shape[1], 32):
            v = [oracle.bf16_to_double(b) for b in x[r, c0:c0 + 32]]
            amax = max(abs(t) for t in v)
            m, ex = math.frexp(amax)           # amax = m * 2^ex, m in [0.5, 1)
            X = 2.0 ** ((ex - 1) - 8)
            ns = sum(abs(t) / X > 448 for t in v)
            top += sum(abs(t) / X >= 432 for t in v)
            sat += ns
            rsum += ns
            bsat += ns > 0
        row_sat.append(rsum)
    assert sat > 0 and top > sat                 # the sample exercises both
    assert (st["saturated"], st["top_code"], st["blocks_saturated"]) == (sat, top, bsat)
    assert st["blocks_collapsed"] == 0
    assert list(rs) == row_sat


def test_monitor_quantizes_like_mx32():
    x = workloads.bf16_bits(workloads.workload_tensor("mxfp8_4096", "A_clamp")[2040:2056, :512])
    for fmt in (E4M3, E5M2):
        q, s, st, rs = oracle.mx32_monitor(x, fmt)
        q2, s2, cnt = oracle.quant_mx32(x, fmt)
        assert np.array_equal(q, q2) and np.array_equal(s, s2)
        assert st["saturated"] == cnt == int(rs.sum())
        assert st["saturated"] <= st["top_code"]
