"""GPU parity of the block-scaled FP8 GEMM against the oracle's fp64 product of
the dequantized operands:

    |C_gpu - C_ref| <= 4e-3 * sum_k |a_ik * b_jk| + one BF16 ulp of |C_ref|

The operands are quantized by the ORACLE and uploaded, so these tests check
the GEMM alone; test_gpu_pipeline checks quantizers + GEMM end to end."""
import numpy as np
import pytest
import torch

import oracle
from oracle import E4M3, E5M2, GRAN_ROW, GRAN_1x128, GRAN_128x128, GRAN_MX32
import fp8_hybrid_granularity_gb300 as fp8hg
from fp8_hybrid_granularity_gb300 import workloads, FPROP, DGRAD, WGRAD
from helpers import oracle_quant, to_qtensor, check_gemm

pytestmark = pytest.mark.gpu


def _operand(kind, rows, k, gran, fmt, seed):
    bits = workloads.bf16_bits(workloads.make_tensor(kind, rows, k, seed, "gpu-gemm"))
    q, s = oracle_quant(bits, gran, fmt)
    return q, s


def _ref(qa, sa, ga, fa, qb, sb, gb, fb):
    a = oracle.dequant(qa, sa, ga, fa)
    b = oracle.dequant(qb, sb, gb, fb)
    return oracle.gemm_ref_dense(a, b)


CASES = [
    # op, (gran_a, fmt_a, kind_a), (gran_b, fmt_b, kind_b), M, N, K
    (FPROP, (GRAN_ROW, E4M3, "act_tiny"), (GRAN_128x128, E4M3, "weight"), 256, 512, 512),
    (FPROP, (GRAN_1x128, E4M3, "act"), (GRAN_128x128, E4M3, "weight"), 384, 384, 640),
    (DGRAD, (GRAN_ROW, E5M2, "grad"), (GRAN_128x128, E4M3, "weight"), 256, 640, 384),
    (DGRAD, (GRAN_1x128, E4M3, "grad"), (GRAN_128x128, E4M3, "weight"), 128, 256, 1152),
    (WGRAD, (GRAN_1x128, E5M2, "grad"), (GRAN_1x128, E4M3, "act"), 256, 256, 1024),
    (FPROP, (GRAN_MX32, E4M3, "mx_ln"), (GRAN_MX32, E4M3, "mx_ln"), 256, 512, 512),
    (FPROP, (GRAN_MX32, E5M2, "mx_ln_clamp"), (GRAN_MX32, E4M3, "normal"), 128, 384, 256),
    # E5M2 on the B side (instruction-descriptor bits 10-12), alone and with E5M2 A
    (FPROP, (GRAN_ROW, E4M3, "act"), (GRAN_128x128, E5M2, "weight"), 256, 384, 512),
    (WGRAD, (GRAN_1x128, E4M3, "act"), (GRAN_1x128, E5M2, "grad"), 256, 640, 640),
    (DGRAD, (GRAN_ROW, E5M2, "grad"), (GRAN_128x128, E5M2, "weight"), 512, 256, 384),
    (FPROP, (GRAN_MX32, E4M3, "normal"), (GRAN_MX32, E5M2, "mx_ln"), 256, 256, 384),
    # several n-tiles of every shape, the last one ragged (1152 = 2 x 448 + 256 =
    # 5 x 224 + 32 = 4 x 256 + 128)
    (FPROP, (GRAN_ROW, E4M3, "act"), (GRAN_128x128, E4M3, "weight"), 512, 1152, 384),
]


TILES = [1, 2, 3]   # 128 x 256 tiles; 256 x 224 tiles with two accumulators; CTA pairs (256 x 448)


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"op{c[0]}-{c[1][0]}{c[1][1]}-{c[2][0]}{c[2][1]}-{c[3]}x{c[4]}x{c[5]}")
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("tile", TILES)
def test_gemm_matches_oracle(cuda_lib, case, out_dtype, tile):
    op, (ga, fa, ka), (gb, fb, kb), M, N, K = case
    if tile >= 2 and M % 256:
        pytest.skip("256-row tiles need M % 256 == 0")
    qa, sa = _operand(ka, M, K, ga, fa, M + K)
    qb, sb = _operand(kb, N, K, gb, fb, N + 3 * K)
    c = fp8hg.fp8_gemm_scaled(op, to_qtensor(qa, sa, fa, ga), to_qtensor(qb, sb, fb, gb),
                              out_dtype=out_dtype, tile=tile)
    assert fp8hg.fp8hg_get_device_error() == 0
    c_ref, s_abs = _ref(qa, sa, ga, fa, qb, sb, gb, fb)
    check_gemm(c.float().cpu().numpy(), c_ref, s_abs, "gemm")


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_gemm_accumulate(cuda_lib, tile, out_dtype):
    """C = A1 B^T, then C += A2 B^T; N = 384 leaves a ragged last tile for
    every tile shape (384 = 256 + 128 = 224 + 160; 384 < 448)."""
    M, N, K = 256, 384, 512
    qa, sa = _operand("act", M, K, GRAN_1x128, E4M3, 1)
    qb, sb = _operand("weight", N, K, GRAN_128x128, E4M3, 2)
    qa2, sa2 = _operand("act", M, K, GRAN_1x128, E4M3, 3)
    a, b, a2 = to_qtensor(qa, sa, E4M3, GRAN_1x128), to_qtensor(qb, sb, E4M3, GRAN_128x128), \
        to_qtensor(qa2, sa2, E4M3, GRAN_1x128)
    c = fp8hg.fp8_gemm_scaled(FPROP, a, b, out_dtype=out_dtype, tile=tile)
    c1 = c.float().cpu().numpy()                   # the first product as stored
    fp8hg.fp8_gemm_scaled(FPROP, a2, b, out=c, accumulate=True, tile=tile)
    r1, s1 = _ref(qa, sa, GRAN_1x128, E4M3, qb, sb, GRAN_128x128, E4M3)
    r2, s2 = _ref(qa2, sa2, GRAN_1x128, E4M3, qb, sb, GRAN_128x128, E4M3)
    check_gemm(c1, r1, s1, "first product")
    # the sum is rounded once more to the output type (BF16: one more ulp)
    check_gemm(c.float().cpu().numpy(), r1 + r2, s1 + s2 + np.abs(r1), "accumulate")


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("fmt_a,fmt_b", [(E4M3, E4M3), (E4M3, E5M2), (E5M2, E5M2)])
def test_gemm_unit_scales_exact(cuda_lib, tile, fmt_a, fmt_b):
    """Small-integer codes with unit scales: the product is an exact integer
    matrix that FP32 accumulation represents exactly.  Every integer in
    [-8, 8] is exact in both encodings, so a wrong format field decodes
    different values and breaks the equality."""
    rng = np.random.default_rng(0)
    ints = np.arange(-8, 9)
    f8 = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}
    enc = lambda f: torch.tensor(ints, dtype=torch.float32).to(f8[f]).view(torch.uint8).numpy()
    M, N, K = 256, 256, 256
    ia, ib = rng.integers(0, 17, (M, K)), rng.integers(0, 17, (N, K))
    qa, qb = enc(fmt_a)[ia], enc(fmt_b)[ib]
    sa = np.full((M, K // 128), 127, np.uint8)
    sb = np.full((N // 128, K // 128), 127, np.uint8)
    c = fp8hg.fp8_gemm_scaled(FPROP, to_qtensor(qa, sa, fmt_a, GRAN_1x128),
                              to_qtensor(qb, sb, fmt_b, GRAN_128x128), out_dtype=torch.float32,
                              tile=tile)
    exact = ints[ia].astype(np.int64) @ ints[ib].astype(np.int64).T
    assert np.array_equal(c.cpu().numpy().astype(np.int64), exact)


@pytest.mark.parametrize("tile", TILES)
def test_gemm_distinct_row_scales(cuda_lib, tile):
    """Unit codes, a distinct power-of-two scale per A row and per 128-row B
    block, and per-32-K MX scales: any mix-up of scale rows, blocks or K slots
    changes the product by a power of two."""
    rng = np.random.default_rng(1)
    M, N, K = 256, 256, 256
    one = 0x38  # E4M3 code of 1.0
    qa = np.full((M, K), one, np.uint8)
    qb = np.full((N, K), one, np.uint8)
    sa = (100 + rng.integers(0, 40, (M, K // 32))).astype(np.uint8)
    sb = (100 + rng.integers(0, 40, (N, K // 32))).astype(np.uint8)
    c = fp8hg.fp8_gemm_scaled(FPROP, to_qtensor(qa, sa, E4M3, GRAN_MX32),
                              to_qtensor(qb, sb, E4M3, GRAN_MX32), out_dtype=torch.float32,
                              tile=tile)
    c_ref, s_abs = _ref(qa, sa, GRAN_MX32, E4M3, qb, sb, GRAN_MX32, E4M3)
    check_gemm(c.cpu().numpy(), c_ref, s_abs, "distinct scales")


@pytest.mark.parametrize("tile", TILES)
def test_gemm_timeout_path(cuda_lib, tile):
    """A host-injected missing arrival makes the first pipeline wait run out:
    the kernel returns, the status reads TIMEOUT, and the next call works."""
    M, N, K = 256, 256, 256
    qa, sa = _operand("act", M, K, GRAN_1x128, E4M3, 5)
    qb, sb = _operand("weight", N, K, GRAN_128x128, E4M3, 6)
    a, b = to_qtensor(qa, sa, E4M3, GRAN_1x128), to_qtensor(qb, sb, E4M3, GRAN_128x128)
    fp8hg.fp8_gemm_scaled(FPROP, a, b, wait_limit_ns=20_000_000, inject_fault=1, tile=tile)
    assert fp8hg.fp8hg_get_device_error() == 6  # FP8HG_ERR_TIMEOUT
    c = fp8hg.fp8_gemm_scaled(FPROP, a, b, out_dtype=torch.float32, tile=tile)
    assert fp8hg.fp8hg_get_device_error() == 0
    c_ref, s_abs = _ref(qa, sa, GRAN_1x128, E4M3, qb, sb, GRAN_128x128, E4M3)
    check_gemm(c.cpu().numpy(), c_ref, s_abs, "after timeout")


@pytest.mark.parametrize("tile", TILES)
def test_gemm_strided_operands(cuda_lib, tile):
    """Operands and scales that are views into wider buffers (row strides
    ld > K and ld_scale > the scale columns): the tensor maps and the scale
    reads follow the strides."""
    M, N, K = 256, 384, 640
    qa, sa = _operand("act", M, K, GRAN_1x128, E4M3, 41)
    qb, sb = _operand("weight", N, K, GRAN_128x128, E4M3, 42)

    def strided(q, s, fmt, gran, pad_k, pad_s):
        cb = torch.zeros((q.shape[0], q.shape[1] + pad_k), dtype=torch.uint8, device="cuda")
        cb[:, :q.shape[1]] = torch.from_numpy(np.ascontiguousarray(q)).cuda()
        ncs = s.shape[1]
        sbuf = torch.full((s.shape[0], ncs + pad_s), 0x7F, dtype=torch.uint8, device="cuda")
        sbuf[:, :ncs] = torch.from_numpy(np.ascontiguousarray(s)).cuda()
        return fp8hg.QTensor(cb[:, :q.shape[1]], sbuf, fmt, gran, ncs)

    a = strided(qa, sa, E4M3, GRAN_1x128, 256, 15)          # ld = K + 256, ld_scale = 5 + 15
    b = strided(qb, sb, E4M3, GRAN_128x128, 128, 11)        # ld = K + 128, ld_scale = 5 + 11
    assert a.codes.stride(0) == K + 256 and b.codes.stride(0) == K + 128
    c = fp8hg.fp8_gemm_scaled(FPROP, a, b, out_dtype=torch.float32, tile=tile)
    assert fp8hg.fp8hg_get_device_error() == 0
    c_ref, s_abs = _ref(qa, sa, GRAN_1x128, E4M3, qb, sb, GRAN_128x128, E4M3)
    check_gemm(c.cpu().numpy(), c_ref, s_abs, "strided operands")
