"""The FP32-scale variant on the GPU against the oracle: quantizer codes and
FP32 scale bits bit for bit; the promotion GEMM within the GEMM tolerance."""
import numpy as np
import pytest
import torch

import oracle
from oracle import E4M3, E5M2, GRAN_ROW, GRAN_1x128, GRAN_128x128
import fp8_hybrid_granularity_gb300 as fp8hg
from fp8_hybrid_granularity_gb300 import workloads
from helpers import np_u8, assert_codes_equal, check_gemm

pytestmark = pytest.mark.gpu


def _f32_bits(t):
    return t.detach().cpu().contiguous().view(torch.int32).numpy().view(np.uint32)


def _bits(t):
    return workloads.bf16_bits(t.detach().cpu())


@pytest.mark.parametrize("rows,cols", [(64, 512), (33, 4096), (16, 8960), (8, 18944)])
@pytest.mark.parametrize("group", [0, 128])
@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_token_quant(cuda_lib, rows, cols, group, fmt):
    """Short rows (registers), long rows (staged in shared memory), 1x128."""
    x = workloads.make_tensor("act", rows, cols, 60 + group + fmt, f"f32q{cols}")
    x[0, :] = 0.0                                      # an all-zero group: d = 1
    if rows > 3:
        x[3, 7] = float("nan")                         # a non-finite group: d = NaN
    q = fp8hg.fp8_quant_token_f32s(x.cuda(), group, fmt)
    qo, so = oracle.quant_token_f32s(_bits(x), group, fmt)
    assert_codes_equal(np_u8(q.codes), qo, "codes")
    assert np.array_equal(_f32_bits(q.scale), so.view(np.uint32)), "scale bits"


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_block128_quant(cuda_lib, fmt):
    w = workloads.make_tensor("weight", 384, 640, 62 + fmt, "f32b")
    w[128:256, 0:128] = 0.0
    q, qt = fp8hg.fp8_quant_block128_f32s(w.cuda(), fmt, transposed_copy=True)
    qo, so, qto, sto = oracle.quant_block128_f32s(_bits(w), fmt, transposed_copy=True)
    assert_codes_equal(np_u8(q.codes), qo, "codes")
    assert_codes_equal(np_u8(qt.codes), qto, "codes^T")
    assert np.array_equal(_f32_bits(q.scale), so.view(np.uint32))
    assert np.array_equal(_f32_bits(qt.scale), sto.view(np.uint32))


def _upload(q, s, fmt, gran):
    return fp8hg.QTensor(torch.from_numpy(np.ascontiguousarray(q)).cuda(),
                         torch.from_numpy(np.ascontiguousarray(s)).cuda(), fmt, gran, s.shape[1])


@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (256, 384, 640), (384, 256, 1152)])
@pytest.mark.parametrize("group", [0, 128])
def test_gemm_vs_oracle(cuda_lib, M, N, K, group):
    """Several tiles and k-block groups (K/128 = 1, 5 and 9 blocks: a partial
    group of scale factors), per-token and 1x128 A."""
    a = workloads.make_tensor("act", M, K, 64 + K, "f32a")
    b = workloads.make_tensor("weight", N, K, 65 + K, "f32w")
    qa, sa = oracle.quant_token_f32s(_bits(a), group, E4M3)
    qb, sb, _, _ = oracle.quant_block128_f32s(_bits(b), E4M3)
    ga = GRAN_ROW if group == 0 else GRAN_1x128
    c = fp8hg.fp8_gemm_scaled_f32s(fp8hg.FPROP, _upload(qa, sa, E4M3, ga),
                                   _upload(qb, sb, E4M3, GRAN_128x128), out_dtype=torch.float32)
    assert fp8hg.fp8hg_get_device_error() == 0
    c_ref, s_abs = oracle.gemm_ref_dense(oracle.dequant_f32s(qa, sa, ga, E4M3),
                                         oracle.dequant_f32s(qb, sb, GRAN_128x128, E4M3))
    check_gemm(c.cpu().numpy(), c_ref, s_abs, f"f32s gemm {M}x{N}x{K}")


def test_dgrad_e5m2_bf16_out(cuda_lib):
    """dX = dY W: dY per token in E5M2, W^T from the block quantizer's
    transposed copy, BF16 out."""
    dy = workloads.make_tensor("grad", 256, 512, 66, "f32dy")
    w = workloads.make_tensor("weight", 512, 384, 67, "f32wd")           # [N_out=512, K=384]
    qd, sd = oracle.quant_token_f32s(_bits(dy), 0, E5M2)
    _, _, qwt, swt = oracle.quant_block128_f32s(_bits(w), E4M3, transposed_copy=True)   # [384, 512]
    dx = fp8hg.fp8_gemm_scaled_f32s(fp8hg.DGRAD, _upload(qd, sd, E5M2, GRAN_ROW),
                                    _upload(qwt, swt, E4M3, GRAN_128x128))
    c_ref, s_abs = oracle.gemm_ref_dense(oracle.dequant_f32s(qd, sd, GRAN_ROW, E5M2),
                                         oracle.dequant_f32s(qwt, swt, GRAN_128x128, E4M3))
    check_gemm(dx.float().cpu().numpy(), c_ref, s_abs, "f32s dgrad")


def test_pipeline_1p5b_gate_sampled(cuda_lib):
    """GPU quantizers + promotion GEMM on X [8192, 1536] x W_gate [8960, 1536],
    against the oracle's quantization and GEMM on sampled rows and blocks."""
    x = workloads.workload_tensor("fprop_1p5b", "X", device="cuda")
    w = workloads.workload_tensor("fprop_1p5b", "W_gate", device="cuda")
    xq = fp8hg.fp8_quant_token_f32s(x, 0, E4M3)
    wq = fp8hg.fp8_quant_block128_f32s(w, E4M3)
    y = fp8hg.fp8_gemm_scaled_f32s(fp8hg.FPROP, xq, wq)
    assert fp8hg.fp8hg_get_device_error() == 0
    rng = np.random.default_rng(12)
    ii = rng.choice(8192, 16, replace=False)
    qa, sa = oracle.quant_token_f32s(_bits(x[torch.from_numpy(ii).cuda()]), 0, E4M3)
    for bidx in rng.choice(8960 // 128, 3, replace=False):
        qb, sb, _, _ = oracle.quant_block128_f32s(_bits(w[128 * bidx:128 * bidx + 128]), E4M3)
        c_ref, s_abs = oracle.gemm_ref_dense(oracle.dequant_f32s(qa, sa, GRAN_ROW, E4M3),
                                             oracle.dequant_f32s(qb, sb, GRAN_128x128, E4M3))
        g = y[torch.from_numpy(ii).cuda()][:, 128 * bidx:128 * bidx + 128].float().cpu().numpy()
        check_gemm(g, c_ref, s_abs, f"f32s pipeline block {bidx}")
