"""Pins for the oracle's scaled GEMM: exact rational arithmetic on tiny shapes
(every dequantized operand is an integer times a power of two, so the dot
product is exact in Python integers), and a closed-form special case with
unit scales and small-integer codes.  Operands are decoded here with torch's
float8 view, not with the oracle's decoder."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import E4M3, E5M2, GRAN_ROW, GRAN_1x128, GRAN_128x128, GRAN_MX32

TORCH_DT = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}


def _decode(q, fmt):
    return torch.from_numpy(np.ascontiguousarray(q)).view(TORCH_DT[fmt]).to(torch.float64).numpy()


def _scale_grid(scale, gran, rows, K):
    """Per-element scale byte, expanded independently of the oracle."""
    if gran == GRAN_ROW:
        return np.repeat(scale[:, :1], K, axis=1)
    if gran == GRAN_1x128:
        return np.repeat(scale[:, :K // 128], 128, axis=1)
    if gran == GRAN_128x128:
        return np.repeat(np.repeat(scale[:rows // 128, :K // 128], 128, axis=0), 128, axis=1)
    return np.repeat(scale[:, :K // 32], 32, axis=1)


def _exact_values(q, scale, gran, fmt):
    rows, K = q.shape
    v = _decode(q, fmt)
    e = _scale_grid(scale, gran, rows, K).astype(np.int64) - 127
    return v, e


def _exact_dot(va, ea, vb, eb):
    """Exact sum of va*2^ea * vb*2^eb as a Python Fraction-free integer pair
    (numerator, exponent)."""
    base = -400
    tot = 0
    for x, a, y, b in zip(va, ea, vb, eb):
        if x == 0 or y == 0:
            continue
        mx, px = math.frexp(x)       # x = mx * 2^px, mx has <= 53 bits
        my, py = math.frexp(y)
        ix = int(mx * 2 ** 53)
        iy = int(my * 2 ** 53)
        sh = px + py + int(a) + int(b) - 106 - base
        assert sh >= 0
        tot += (ix * iy) << sh
    return tot, base


def _to_float(num, base):
    return math.ldexp(float(num), base) if abs(num) < 2 ** 1000 else float(num) * 2.0 ** base


def _random_operand(rng, rows, K, gran, fmt):
    maxc = 0x7E if fmt == E4M3 else 0x7B
    q = rng.integers(0, maxc + 1, (rows, K)).astype(np.uint8)
    q |= (rng.integers(0, 2, (rows, K)) << 7).astype(np.uint8)
    if gran == GRAN_ROW:
        s = rng.integers(100, 140, (rows, 1))
    elif gran == GRAN_1x128:
        s = rng.integers(100, 140, (rows, K // 128))
    elif gran == GRAN_128x128:
        s = rng.integers(100, 140, (rows // 128, K // 128))
    else:
        s = rng.integers(100, 140, (rows, K // 32))
    return q, s.astype(np.uint8)


CASES = [
    (GRAN_ROW, E4M3, GRAN_128x128, E4M3),
    (GRAN_1x128, E5M2, GRAN_128x128, E4M3),
    (GRAN_1x128, E4M3, GRAN_1x128, E4M3),
    (GRAN_MX32, E4M3, GRAN_MX32, E5M2),
]


@pytest.mark.parametrize("ga,fa,gb,fb", CASES)
def test_gemm_ref_exact_on_tiny_shapes(ga, fa, gb, fb):
    rng = np.random.default_rng(ga * 10 + gb)
    M, N, K = 6, 128, 256
    qa, sa = _random_operand(rng, M, K, ga, fa)
    qb, sb = _random_operand(rng, N, K, gb, fb)
    va, ea = _exact_values(qa, sa, ga, fa)
    vb, eb = _exact_values(qb, sb, gb, fb)
    jj = np.array([0, 1, 5, 64, 127, 100, 33])
    ii = np.array([0, 5, 3, 2, 1, 4, 0])
    c, s = oracle.gemm_ref_pairs(qa, sa, ga, fa, qb, sb, gb, fb, ii, jj)
    for t, (i, j) in enumerate(zip(ii, jj)):
        num, base = _exact_dot(va[i], ea[i], vb[j], eb[j])
        exact = _to_float(num, base)
        # fp64 accumulation of K terms: |err| <= K * 2^-53 * S
        assert abs(c[t] - exact) <= K * 2.0 ** -53 * s[t] + 1e-300
        # S is the sum of magnitudes
        absnum = 0
        for x, a, y, b in zip(va[i], ea[i], vb[j], eb[j]):
            absnum += abs(x * y) * 2.0 ** (int(a) + int(b))
        assert s[t] == pytest.approx(absnum, rel=1e-12)


def test_gemm_ref_unit_scales_small_integers():
    """Codes of the integers -8..8 with scale byte 127 (2^0): C is an exact
    integer matrix product."""
    rng = np.random.default_rng(3)
    ints = np.arange(-8, 9)
    codes = torch.tensor(ints, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    M, N, K = 8, 128, 256
    ia = rng.integers(0, len(ints), (M, K))
    ib = rng.integers(0, len(ints), (N, K))
    qa, qb = codes[ia], codes[ib]
    sa = np.full((M, K // 128), 127, np.uint8)
    sb = np.full((1, K // 128), 127, np.uint8)
    ii, jj = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    c, s = oracle.gemm_ref_pairs(qa, sa, GRAN_1x128, E4M3, qb, sb, GRAN_128x128, E4M3,
                                 ii.ravel(), jj.ravel())
    exact = ints[ia].astype(np.int64) @ ints[ib].astype(np.int64).T
    assert np.array_equal(c.reshape(M, N), exact.astype(np.float64))
    absx = np.abs(ints[ia]).astype(np.int64) @ np.abs(ints[ib]).astype(np.int64).T
    assert np.array_equal(s.reshape(M, N), absx.astype(np.float64))


def test_dense_and_pairs_agree_and_scale_index():
    """gemm_ref_dense over oracle.dequant equals gemm_ref_pairs; scales that
    vary along K (MX) are applied per 32-wide block."""
    rng = np.random.default_rng(9)
    M, N, K = 4, 3, 128
    qa, sa = _random_operand(rng, M, K, GRAN_MX32, E4M3)
    qb, sb = _random_operand(rng, N, K, GRAN_MX32, E4M3)
    a = oracle.dequant(qa, sa, GRAN_MX32, E4M3)
    b = oracle.dequant(qb, sb, GRAN_MX32, E4M3)
    va, ea = _exact_values(qa, sa, GRAN_MX32, E4M3)
    assert np.array_equal(a, va * np.exp2(ea))
    c, s = oracle.gemm_ref_dense(a, b)
    ii, jj = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    c2, s2 = oracle.gemm_ref_pairs(qa, sa, GRAN_MX32, E4M3, qb, sb, GRAN_MX32, E4M3,
                                   ii.ravel(), jj.ravel())
    assert np.array_equal(c.ravel(), c2) and np.array_equal(s.ravel(), s2)


def test_tolerance_helper():
    assert oracle.bf16_ulp(np.array([1.0]))[0] == 2.0 ** -7
    assert oracle.bf16_ulp(np.array([-3.0]))[0] == 2.0 ** -6
    assert oracle.bf16_ulp(np.array([0.0]))[0] == 2.0 ** -133
    tol = oracle.gemm_tolerance(np.array([1.0]), np.array([10.0]))
    assert tol[0] == 4e-3 * 10 + 2.0 ** -7
