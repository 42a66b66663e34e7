"""Parity at the ends of the throughput sweep: BF16 [R, 4096] tensors from
1 MB (R = 128, checked whole) to 4 GB (R = 524288, checked on sampled rows and
blocks) through all three granularities, and the down-projection GEMM at
M = 4096 and 65536 (16384 is in test_gpu_fullsize.py) on sampled outputs."""
import numpy as np
import pytest
import torch

import oracle
from oracle import E4M3, GRAN_ROW, GRAN_128x128
import fp8_hybrid_granularity_gb300 as fp8hg
from fp8_hybrid_granularity_gb300 import workloads
from helpers import np_u8, assert_codes_equal, check_gemm

pytestmark = pytest.mark.gpu
C = 4096


def _bits(t):
    return workloads.bf16_bits(t.detach().cpu())


def test_sweep_smallest_whole(cuda_lib):
    x = workloads.make_tensor("act", 128, C, 4, "sweep", device="cuda")
    xb = _bits(x)
    q = fp8hg.fp8_quant_token(x, 0, E4M3)
    qo, so = oracle.quant_token(xb, 0, E4M3)
    assert_codes_equal(np_u8(q.codes), qo, "token")
    assert_codes_equal(np_u8(q.scales()), so, "token scales")
    q = fp8hg.fp8_quant_token(x, 128, E4M3)
    qo, so = oracle.quant_token(xb, 128, E4M3)
    assert_codes_equal(np_u8(q.codes), qo, "1x128")
    assert_codes_equal(np_u8(q.scales()), so, "1x128 scales")
    q = fp8hg.fp8_quant_block128(x, E4M3)
    qo, so, _, _ = oracle.quant_block128(xb, E4M3)
    assert_codes_equal(np_u8(q.codes), qo, "128x128")
    assert_codes_equal(np_u8(q.scales()), so, "128x128 scales")


def test_sweep_largest_sampled(cuda_lib):
    R = 128 * 4 ** 6                                   # 4 GB of BF16
    x = workloads.make_tensor("act", R, C, 4, "sweep", device="cuda")
    rng = np.random.default_rng(21)
    rows = np.concatenate([[0, R - 1], rng.choice(R, 30, replace=False)])
    idx = torch.from_numpy(rows).cuda()
    xb = _bits(x[idx])
    q = fp8hg.fp8_quant_token(x, 0, E4M3)
    qo, so = oracle.quant_token(xb, 0, E4M3)
    assert_codes_equal(np_u8(q.codes[idx]), qo, "token")
    assert_codes_equal(np_u8(q.scales()[idx]), so, "token scales")
    del q
    q = fp8hg.fp8_quant_token(x, 128, E4M3)
    qo, so = oracle.quant_token(xb, 128, E4M3)
    assert_codes_equal(np_u8(q.codes[idx]), qo, "1x128")
    assert_codes_equal(np_u8(q.scales()[idx]), so, "1x128 scales")
    del q
    q = fp8hg.fp8_quant_block128(x, E4M3)
    for rb in [0, R // 128 - 1] + list(rng.choice(R // 128, 4, replace=False)):
        r0 = 128 * int(rb)
        qo, so, _, _ = oracle.quant_block128(_bits(x[r0:r0 + 128]), E4M3)
        assert_codes_equal(np_u8(q.codes[r0:r0 + 128]), qo, f"block row {rb}")
        assert_codes_equal(np_u8(q.scales()[int(rb)]), so[0], f"block scales {rb}")
    assert fp8hg.fp8hg_get_device_error() == 0


@pytest.mark.parametrize("M", [4096, 65536])
def test_down_projection_sweep_sizes(cuda_lib, M):
    HID, MLP = 3584, 18944
    w = workloads.make_tensor("weight", HID, MLP, 4, "W_down", device="cuda")
    h = workloads.make_tensor("act", M, MLP, 4, "H", device="cuda")
    y = fp8hg.fp8_gemm_scaled(fp8hg.FPROP, fp8hg.fp8_quant_token(h, 0, E4M3),
                              fp8hg.fp8_quant_block128(w, E4M3))
    assert fp8hg.fp8hg_get_device_error() == 0
    rng = np.random.default_rng(M)
    ii = np.concatenate([[0, M - 1], rng.choice(M, 10, replace=False)])
    qa, sa = oracle.quant_token(_bits(h[torch.from_numpy(ii).cuda()]), 0, E4M3)
    c_gpu, c_ref, s_abs = [], [], []
    for b in [0, HID // 128 - 1, int(rng.integers(HID // 128))]:
        qb, sb, _, _ = oracle.quant_block128(_bits(w[128 * b:128 * b + 128]), E4M3)
        jj = rng.choice(128, 4, replace=False)
        I, J = np.meshgrid(np.arange(len(ii)), jj, indexing="ij")
        c, s = oracle.gemm_ref_pairs(qa, sa, GRAN_ROW, E4M3, qb, sb, GRAN_128x128, E4M3,
                                     I.ravel(), J.ravel())
        c_ref.append(c)
        s_abs.append(s)
        g = y[torch.from_numpy(ii).cuda()][:, torch.from_numpy(128 * b + jj).cuda()]
        c_gpu.append(g.float().cpu().numpy().ravel())
    check_gemm(np.concatenate(c_gpu), np.concatenate(c_ref), np.concatenate(s_abs), f"down M={M}")
