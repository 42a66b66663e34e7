"""End to end on the GPU: BF16 inputs -> GPU quantizers -> GPU GEMM, against
the oracle's own quantization and fp64 GEMM of the same BF16 inputs.  Covers
the tiny forward layer in full, the 1.5B layer shapes (gate/up, down, QKV
forward; down data-gradient with E5M2 gradients) on sampled outputs, and the
MXFP8 4096^3 case including its clamp count."""
import zlib

import numpy as np
import pytest
import torch

import oracle
from oracle import E4M3, E5M2, GRAN_ROW, GRAN_128x128, GRAN_MX32
import fp8_hybrid_granularity_gb300 as fp8hg
from fp8_hybrid_granularity_gb300 import workloads
from helpers import np_u8, assert_codes_equal, check_gemm

pytestmark = pytest.mark.gpu


def _bits(t):
    return workloads.bf16_bits(t.detach().cpu())


def test_tiny_fprop_full(cuda_lib):
    x = workloads.workload_tensor("tiny_fprop", "X")
    w = workloads.workload_tensor("tiny_fprop", "W")
    xq = fp8hg.fp8_quant_token(x.cuda(), 0, E4M3)
    wq = fp8hg.fp8_quant_block128(w.cuda(), E4M3)
    y = fp8hg.fp8_gemm_scaled(fp8hg.FPROP, xq, wq)
    qx, sx = oracle.quant_token(_bits(x), 0, E4M3)
    qw, sw, _, _ = oracle.quant_block128(_bits(w), E4M3)
    assert_codes_equal(np_u8(xq.codes), qx, "X codes")
    assert_codes_equal(np_u8(wq.codes), qw, "W codes")
    c_ref, s_abs = oracle.gemm_ref_dense(oracle.dequant(qx, sx, GRAN_ROW, E4M3),
                                         oracle.dequant(qw, sw, GRAN_128x128, E4M3))
    check_gemm(y.float().cpu().numpy(), c_ref, s_abs, "tiny fprop")


def _sampled_fprop(a_bf16, w_bf16, fmt_a, rng, nrows=24, nblocks=3):
    """GPU: per-token A x 128x128-block W over the whole tensors; oracle: the
    sampled rows of A and whole 128-row blocks of W."""
    aq = fp8hg.fp8_quant_token(a_bf16, 0, fmt_a)
    wq = fp8hg.fp8_quant_block128(w_bf16, E4M3)
    y = fp8hg.fp8_gemm_scaled(fp8hg.FPROP, aq, wq)
    assert fp8hg.fp8hg_get_device_error() == 0
    M, N = a_bf16.shape[0], w_bf16.shape[0]
    ii = rng.choice(M, nrows, replace=False)
    qa, sa = oracle.quant_token(_bits(a_bf16[torch.from_numpy(ii).cuda()]), 0, fmt_a)
    assert_codes_equal(np_u8(aq.codes[torch.from_numpy(ii).cuda()]), qa, "A codes (sampled rows)")
    c_gpu, c_ref, s_abs = [], [], []
    for b in rng.choice(N // 128, nblocks, replace=False):
        qb, sb, _, _ = oracle.quant_block128(_bits(w_bf16[128 * b:128 * b + 128]), E4M3)
        jj = rng.choice(128, 8, replace=False)
        I, J = np.meshgrid(np.arange(nrows), jj, indexing="ij")
        c, s = oracle.gemm_ref_pairs(qa, sa, GRAN_ROW, fmt_a, qb, sb, GRAN_128x128, E4M3,
                                     I.ravel(), J.ravel())
        c_ref.append(c)
        s_abs.append(s)
        g = y[torch.from_numpy(ii).cuda()][:, torch.from_numpy(128 * b + jj).cuda()]
        c_gpu.append(g.float().cpu().numpy().ravel())
    return np.concatenate(c_gpu), np.concatenate(c_ref), np.concatenate(s_abs)


@pytest.mark.parametrize("a_name,w_name", [("X", "W_gate"), ("X", "W_up"), ("H", "W_down"),
                                           ("X", "W_qkv")])
def test_fprop_1p5b_layers(cuda_lib, a_name, w_name):
    a = workloads.workload_tensor("fprop_1p5b", a_name, device="cuda")
    w = workloads.workload_tensor("fprop_1p5b", w_name, device="cuda")
    rng = np.random.default_rng(zlib.crc32((a_name + w_name).encode()))
    check_gemm(*_sampled_fprop(a, w, E4M3, rng), f"fprop {w_name}")


@pytest.mark.parametrize("tile", [0, 2])
def test_fprop_1p5b_gate_up_stacked(cuda_lib, tile):
    """The gate and up weights quantized by one batched call into the two
    halves of one stacked buffer, then one GEMM over the stack: its output
    holds the two projections side by side, the same bytes as one GEMM per
    weight (both halves' tiles are the separate GEMMs' tiles), and sampled
    outputs of the up half agree with the oracle."""
    x = workloads.workload_tensor("fprop_1p5b", "X", device="cuda")
    wg = workloads.workload_tensor("fprop_1p5b", "W_gate", device="cuda")
    wu = workloads.workload_tensor("fprop_1p5b", "W_up", device="cuda")
    n, k = wg.shape
    both, _ = fp8hg.alloc_block128(2 * n, k, E4M3, False, x.device)
    halves = [fp8hg.QTensor(both.codes[h * n:(h + 1) * n], both.scale[h * n // 128:(h + 1) * n // 128],
                            E4M3, GRAN_128x128, k // 128) for h in (0, 1)]
    fp8hg.fp8_quant_block128_batch([wg, wu], E4M3, outs=[(q, None) for q in halves])
    xq = fp8hg.fp8_quant_token(x, 0, E4M3)
    y = fp8hg.fp8_gemm_scaled(fp8hg.FPROP, xq, both, tile=tile)
    yg = fp8hg.fp8_gemm_scaled(fp8hg.FPROP, xq, fp8hg.fp8_quant_block128(wg, E4M3), tile=tile)
    yu = fp8hg.fp8_gemm_scaled(fp8hg.FPROP, xq, fp8hg.fp8_quant_block128(wu, E4M3), tile=tile)
    assert fp8hg.fp8hg_get_device_error() == 0
    assert torch.equal(y[:, :n], yg) and torch.equal(y[:, n:], yu)
    rng = np.random.default_rng(23)
    c_gpu, c_ref, s_abs = _sampled_fprop(x, wu, E4M3, rng)
    check_gemm(c_gpu, c_ref, s_abs, "stacked up half (via the separate GEMM)")


def test_dgrad_1p5b_e5m2(cuda_lib):
    """dX = dY W_gate: dY [8192, 8960] per token E5M2, B = W_gate^T from the
    block quantizer's transposed copy."""
    dev = torch.device("cuda", 0)
    dy = workloads.make_tensor("grad", 8192, 8960, 1, "dY_gate", device=dev)
    w = workloads.workload_tensor("fprop_1p5b", "W_gate", device="cuda")   # [8960, 1536]
    dyq = fp8hg.fp8_quant_token(dy, 0, E5M2)
    _, wt = fp8hg.fp8_quant_block128(w, E4M3, transposed_copy=True)      # [1536, 8960]
    dx = fp8hg.fp8_gemm_scaled(fp8hg.DGRAD, dyq, wt)
    rng = np.random.default_rng(7)
    ii = rng.choice(8192, 16, replace=False)
    qa, sa = oracle.quant_token(_bits(dy[torch.from_numpy(ii).cuda()]), 0, E5M2)
    b = int(rng.integers(1536 // 128))
    _, _, qbt, sbt = oracle.quant_block128(_bits(w[:, 128 * b:128 * b + 128]), E4M3,
                                           transposed_copy=True)
    jj = rng.choice(128, 8, replace=False)
    I, J = np.meshgrid(np.arange(16), jj, indexing="ij")
    c_ref, s_abs = oracle.gemm_ref_pairs(qa, sa, GRAN_ROW, E5M2, qbt, sbt, GRAN_128x128, E4M3,
                                         I.ravel(), J.ravel())
    g = dx[torch.from_numpy(ii).cuda()][:, torch.from_numpy(128 * b + jj).cuda()]
    check_gemm(g.float().cpu().numpy().ravel(), c_ref, s_abs, "dgrad e5m2")


@pytest.mark.parametrize("a_name", ["A", "A_clamp"])
def test_mxfp8_4096(cuda_lib, a_name):
    a = workloads.workload_tensor("mxfp8_4096", a_name, device="cuda")
    b = workloads.workload_tensor("mxfp8_4096", "B", device="cuda")
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
    aq = fp8hg.fp8_quant_mx32(a, E4M3, clamp_count=cnt)
    bq = fp8hg.fp8_quant_mx32(b, E4M3)
    c = fp8hg.fp8_gemm_scaled(fp8hg.FPROP, aq, bq)
    assert fp8hg.fp8hg_get_device_error() == 0
    # clamp count over the whole tensor, codes on sampled rows
    _, _, clamped = oracle.quant_mx32(_bits(a), E4M3)
    assert int(cnt.item()) == clamped
    if a_name == "A_clamp":
        assert clamped > 0
    rng = np.random.default_rng(11)
    ii = np.concatenate([rng.choice(2048, 8, replace=False), 2048 + rng.choice(2048, 8, replace=False)])
    jj = np.concatenate([rng.choice(2048, 4, replace=False), 2048 + rng.choice(2048, 4, replace=False)])
    qa, sa, _ = oracle.quant_mx32(_bits(a[torch.from_numpy(ii).cuda()]), E4M3)
    qb, sb, _ = oracle.quant_mx32(_bits(b[torch.from_numpy(jj).cuda()]), E4M3)
    assert_codes_equal(np_u8(aq.codes[torch.from_numpy(ii).cuda()]), qa, "MX codes")
    I, J = np.meshgrid(np.arange(len(ii)), np.arange(len(jj)), indexing="ij")
    c_ref, s_abs = oracle.gemm_ref_pairs(qa, sa, GRAN_MX32, E4M3, qb, sb, GRAN_MX32, E4M3,
                                         I.ravel(), J.ravel())
    g = c[torch.from_numpy(ii).cuda()][:, torch.from_numpy(jj).cuda()].float().cpu().numpy().ravel()
    check_gemm(g, c_ref, s_abs, "mx gemm")
