"""Split-K GEMM (fp8_gemm_scaled_splitk) against the oracle's fp64 product of
the dequantized operands, with the tolerance of the unsplit GEMM:

    |C_gpu - C_ref| <= 4e-3 * sum_k |a_ik * b_jk| + one BF16 ulp of |C_ref|

Each tile's K range is split over 2-4 CTAs; the first part adds the others'
FP32 partial tiles in part order, so repeated calls are bit-identical."""
import numpy as np
import pytest
import torch

import oracle
from oracle import E4M3, E5M2, GRAN_ROW, GRAN_1x128, GRAN_128x128, GRAN_MX32
import fp8_hybrid_granularity_gb300 as fp8hg
from fp8_hybrid_granularity_gb300 import workloads, FPROP, DGRAD, WGRAD
from helpers import oracle_quant, to_qtensor, check_gemm

pytestmark = pytest.mark.gpu

TIMEOUT = 6


def _operand(kind, rows, k, gran, fmt, seed):
    bits = workloads.bf16_bits(workloads.make_tensor(kind, rows, k, seed, "gpu-splitk"))
    return oracle_quant(bits, gran, fmt)


def _case(op, ga, fa, ka, gb, fb, kb, M, N, K):
    qa, sa = _operand(ka, M, K, ga, fa, M + K)
    qb, sb = _operand(kb, N, K, gb, fb, N + 3 * K)
    ref = oracle.gemm_ref_dense(oracle.dequant(qa, sa, ga, fa), oracle.dequant(qb, sb, gb, fb))
    return to_qtensor(qa, sa, fa, ga), to_qtensor(qb, sb, fb, gb), ref


CASES = [
    # op, A (gran, fmt, kind), B (gran, fmt, kind), M, N, K; N = 384 ends inside
    # the second 224-column tile
    (FPROP, (GRAN_ROW, E4M3, "act"), (GRAN_128x128, E4M3, "weight"), 512, 384, 2048),
    (DGRAD, (GRAN_1x128, E5M2, "grad"), (GRAN_128x128, E4M3, "weight"), 256, 640, 1536),
    (WGRAD, (GRAN_1x128, E4M3, "act"), (GRAN_1x128, E5M2, "grad"), 256, 384, 2560),
    (FPROP, (GRAN_MX32, E4M3, "mx_ln"), (GRAN_MX32, E4M3, "mx_ln"), 256, 512, 1024),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"op{c[0]}-{c[1][0]}-{c[2][0]}-{c[3]}x{c[4]}x{c[5]}")
@pytest.mark.parametrize("split", [2, 3, 4])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_splitk_matches_oracle(cuda_lib, case, split, out_dtype):
    op, (ga, fa, ka), (gb, fb, kb), M, N, K = case
    a, b, (c_ref, s_abs) = _case(op, ga, fa, ka, gb, fb, kb, M, N, K)
    ws = fp8hg.splitk_workspace(M, N, K, split)
    c = fp8hg.fp8_gemm_scaled_splitk(op, a, b, out_dtype=out_dtype, split_k=split, workspace=ws)
    assert fp8hg.fp8hg_get_device_error() == 0
    check_gemm(c.float().cpu().numpy(), c_ref, s_abs, f"split {split}")
    # the call leaves the per-tile counters at zero and a second call on the
    # same workspace gives the same bits
    tiles = (M // 256) * ((N + 223) // 224)
    assert int(ws[:tiles * 32].count_nonzero()) == 0
    c2 = fp8hg.fp8_gemm_scaled_splitk(op, a, b, out_dtype=out_dtype, split_k=split, workspace=ws)
    assert fp8hg.fp8hg_get_device_error() == 0
    assert torch.equal(c.view(torch.int16 if out_dtype == torch.bfloat16 else torch.int32),
                       c2.view(torch.int16 if out_dtype == torch.bfloat16 else torch.int32))


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_splitk_accumulate(cuda_lib, out_dtype):
    """C = A1 B^T unsplit, then C += A2 B^T split in three."""
    M, N, K = 512, 384, 1536
    a, b, (r1, s1) = _case(FPROP, GRAN_1x128, E4M3, "act", GRAN_128x128, E4M3, "weight", M, N, K)
    qa2, sa2 = _operand("act", M, K, GRAN_1x128, E4M3, 77)
    a2 = to_qtensor(qa2, sa2, E4M3, GRAN_1x128)
    qb, sb = _operand("weight", N, K, GRAN_128x128, E4M3, N + 3 * K)
    r2, s2 = oracle.gemm_ref_dense(oracle.dequant(qa2, sa2, GRAN_1x128, E4M3),
                                   oracle.dequant(qb, sb, GRAN_128x128, E4M3))
    c = fp8hg.fp8_gemm_scaled(FPROP, a, b, out_dtype=out_dtype)
    ws = fp8hg.splitk_workspace(M, N, K, 3)
    fp8hg.fp8_gemm_scaled_splitk(FPROP, a2, b, out=c, accumulate=True, split_k=3, workspace=ws)
    assert fp8hg.fp8hg_get_device_error() == 0
    ref = r1 + r2
    s_abs = s1 + s2
    if out_dtype == torch.bfloat16:
        # the first product is rounded to BF16 before the second is added
        s_abs = s_abs + np.abs(r1)
    check_gemm(c.float().cpu().numpy(), ref, s_abs, "split accumulate")


def test_splitk_full_size_1p5b_down(cuda_lib):
    """The 1.5B down projection at M = 8192 (K = 8960, N = 1536) split in two:
    sampled rows against the oracle at full K; the library's own choice for
    this shape is not to split (the exchange would cost more than the fuller
    last wave gains)."""
    M, N, K = 8192, 1536, 8960
    assert fp8hg.splitk_workspace(M, N, K, 0) is None
    ws = fp8hg.splitk_workspace(M, N, K, 2)
    h = workloads.make_tensor("act", M, K, 5, "H-1p5b", device="cuda")
    w = workloads.make_tensor("weight", N, K, 6, "W_down-1p5b", device="cuda")
    a = fp8hg.fp8_quant_token(h, 0, E4M3)
    b = fp8hg.fp8_quant_block128(w, E4M3)
    c = fp8hg.fp8_gemm_scaled_splitk(FPROP, a, b, split_k=2, workspace=ws)
    assert fp8hg.fp8hg_get_device_error() == 0
    rng = np.random.default_rng(3)
    rows = np.concatenate([[0, M - 1], rng.choice(np.arange(1, M - 1), 14, replace=False)])
    qa = a.codes.cpu().numpy()[rows]
    sa = a.scales().cpu().numpy()[rows]
    qb, sb = b.codes.cpu().numpy(), b.scales().cpu().numpy()
    c_ref, s_abs = oracle.gemm_ref_dense(oracle.dequant(qa, sa, GRAN_ROW, E4M3),
                                         oracle.dequant(qb, sb, GRAN_128x128, E4M3))
    check_gemm(c.float().cpu().numpy()[rows], c_ref, s_abs, "split 2, sampled rows")


def test_splitk_auto_few_tiles_long_k(cuda_lib):
    """Two output tiles over K = 32768 (a weight gradient of a small layer
    over many tokens): the library's choice splits it; against the oracle."""
    M, N, K = 256, 256, 32768
    ws = fp8hg.splitk_workspace(M, N, K, 0)
    assert ws is not None, "the library's choice should split this shape"
    a, b, (c_ref, s_abs) = _case(WGRAD, GRAN_1x128, E5M2, "grad", GRAN_1x128, E4M3, "act",
                                 M, N, K)
    c = fp8hg.fp8_gemm_scaled_splitk(WGRAD, a, b, out_dtype=torch.float32, split_k=0,
                                     workspace=ws)
    assert fp8hg.fp8hg_get_device_error() == 0
    check_gemm(c.float().cpu().numpy(), c_ref, s_abs, "auto split")


def test_splitk_timeout_path(cuda_lib):
    """A withheld part count: the first part's wait runs out, the status reads
    TIMEOUT once; with the workspace cleared, the next call is right."""
    M, N, K = 256, 384, 1024
    a, b, (c_ref, s_abs) = _case(FPROP, GRAN_ROW, E4M3, "act", GRAN_128x128, E4M3, "weight",
                                 M, N, K)
    ws = fp8hg.splitk_workspace(M, N, K, 2)
    fp8hg.fp8_gemm_scaled_splitk(FPROP, a, b, split_k=2, workspace=ws, wait_limit_ns=20_000_000,
                                 inject_fault=2)
    assert fp8hg.fp8hg_get_device_error() == TIMEOUT
    ws.zero_()
    c = fp8hg.fp8_gemm_scaled_splitk(FPROP, a, b, split_k=2, workspace=ws)
    assert fp8hg.fp8hg_get_device_error() == 0
    check_gemm(c.float().cpu().numpy(), c_ref, s_abs, "after timeout")


def test_splitk_output_canary(cuda_lib):
    """Strided output inside a 0xAB-filled buffer: nothing written outside."""
    from test_gpu_canary import canvas, assert_canary
    M, N, K = 256, 384, 1024
    a, b, (c_ref, s_abs) = _case(FPROP, GRAN_ROW, E4M3, "act", GRAN_128x128, E4M3, "weight",
                                 M, N, K)
    ws = fp8hg.splitk_workspace(M, N, K, 4)
    for dtype in (torch.bfloat16, torch.float32):
        cbuf, c = canvas(M, N, N + 64, dtype=dtype)
        fp8hg.fp8_gemm_scaled_splitk(FPROP, a, b, out=c, split_k=4, workspace=ws)
        assert fp8hg.fp8hg_get_device_error() == 0
        check_gemm(c.float().cpu().numpy(), c_ref, s_abs, "canary")
        assert_canary(cbuf, M, N, "C")
