"""The timeout path of every kernel that waits on copies, made to run out by
a host-chosen missing copy (fp8hg_wait_opts.inject_fault = 1) and a short
wait limit.  Nothing faults, traps or hangs: the kernel gives up after the
limit, records FP8HG_ERR_TIMEOUT in the device error word and returns; the
status reads TIMEOUT once, and the next call on the same context is correct.
(The main GEMM's own timeout path is tested in test_gpu_gemm.py.)"""
import numpy as np
import pytest
import torch

import oracle
from oracle import E4M3, E5M2, GRAN_ROW, GRAN_1x128, GRAN_128x128
import fp8_hybrid_granularity_gb300 as fp8hg
from fp8_hybrid_granularity_gb300 import workloads
from helpers import np_u8, assert_codes_equal, check_gemm

pytestmark = pytest.mark.gpu

TIMEOUT = 6          # FP8HG_ERR_TIMEOUT
LIMIT_NS = 20_000_000  # 20 ms


def test_token_quant_row_kernel_timeout(cuda_lib):
    """Per-token quantization of 16 KB rows runs the bulk-copy row kernel."""
    x = workloads.make_tensor("act", 512, 8192, 70, "timeout-row")
    xd = x.cuda()
    fp8hg.fp8_quant_token(xd, 0, E4M3, wait_limit_ns=LIMIT_NS, inject_fault=1)
    assert fp8hg.fp8hg_get_device_error() == TIMEOUT
    assert fp8hg.fp8hg_get_device_error() == 0      # reading clears the word
    q = fp8hg.fp8_quant_token(xd, 0, E4M3)
    assert fp8hg.fp8hg_get_device_error() == 0
    qo, so = oracle.quant_token(workloads.bf16_bits(x), 0, E4M3)
    assert_codes_equal(np_u8(q.codes), qo, "codes after timeout")
    assert_codes_equal(np_u8(q.scales()), so, "scales after timeout")


def test_requant_timeout(cuda_lib):
    x = workloads.make_tensor("act", 1024, 512, 71, "timeout-rq")
    src = fp8hg.fp8_quant_token(x.cuda(), 0, E4M3)
    fp8hg.fp8_requant_t(src, E5M2, wait_limit_ns=LIMIT_NS, inject_fault=1)
    assert fp8hg.fp8hg_get_device_error() == TIMEOUT
    out = fp8hg.fp8_requant_t(src, E5M2)
    assert fp8hg.fp8hg_get_device_error() == 0
    qs, ss = oracle.quant_token(workloads.bf16_bits(x), 0, E4M3)
    qo, so = oracle.requant_t(qs, ss, GRAN_ROW, E4M3, E5M2)
    assert_codes_equal(np_u8(out.codes), qo, "codes after timeout")
    assert_codes_equal(np_u8(out.scales()), so, "scales after timeout")


def test_f32s_gemm_timeout(cuda_lib):
    M, N, K = 256, 256, 384
    xa = workloads.bf16_bits(workloads.make_tensor("act", M, K, 72, "timeout-a"))
    xw = workloads.bf16_bits(workloads.make_tensor("weight", N, K, 73, "timeout-b"))
    qa, sa = oracle.quant_token_f32s(xa, 128, E4M3)
    qb, sb, _, _ = oracle.quant_block128_f32s(xw, E4M3)
    up = lambda q, s, g: fp8hg.QTensor(torch.from_numpy(np.ascontiguousarray(q)).cuda(),
                                       torch.from_numpy(np.ascontiguousarray(s)).cuda(), E4M3, g,
                                       s.shape[1])
    a, b = up(qa, sa, GRAN_1x128), up(qb, sb, GRAN_128x128)
    fp8hg.fp8_gemm_scaled_f32s(fp8hg.FPROP, a, b, wait_limit_ns=LIMIT_NS, inject_fault=1)
    assert fp8hg.fp8hg_get_device_error() == TIMEOUT
    c = fp8hg.fp8_gemm_scaled_f32s(fp8hg.FPROP, a, b, out_dtype=torch.float32)
    assert fp8hg.fp8hg_get_device_error() == 0
    c_ref, s_abs = oracle.gemm_ref_dense(oracle.dequant_f32s(qa, sa, GRAN_1x128, E4M3),
                                         oracle.dequant_f32s(qb, sb, GRAN_128x128, E4M3))
    check_gemm(c.cpu().numpy(), c_ref, s_abs, "f32s GEMM after timeout")
