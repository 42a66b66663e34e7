"""The GEMM with its output quantized in the epilogue (fp8_gemm_scaled_q).

The codes are decided on the GPU's FP32 accumulator, which differs from the
oracle's fp64 sum by accumulation order, so two kinds of check are used:
  * exact products (small-integer codes, power-of-two scales): the FP32
    accumulator equals the oracle's C exactly, and the codes and scales must
    equal the oracle's quantization of C bit for bit;
  * general products: every scale byte is the oracle's round-up exponent of
    the group's amax (or its neighbour when the amax lies within the GEMM
    tolerance of a power-of-two boundary), and every code is the oracle's
    round-to-nearest-even encoding of some value within the GEMM tolerance of
    the oracle's C under that scale: the encoder is monotonic, so the code
    must lie between the encodings of (C - tol) / 2^e and (C + tol) / 2^e.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import E4M3, E5M2, GRAN_ROW, GRAN_1x128, GRAN_128x128, GRAN_MX32
import fp8_hybrid_granularity_gb300 as fp8hg
from fp8_hybrid_granularity_gb300 import workloads
from helpers import np_u8, to_qtensor, assert_codes_equal, oracle_quant, check_gemm

pytestmark = pytest.mark.gpu

ONE = {E4M3: 0x38, E5M2: 0x3C}          # FP8 codes of 1.0


def _int_operands(rng, M, N, K):
    """Codes of -1 / 0 / +1, per-row A scales and per-block B scales that are
    constant along K, so C[i, j] = 2^(ea_i + eb_j) * (integer of magnitude <= K)."""
    va = rng.integers(-1, 2, (M, K))
    vb = rng.integers(-1, 2, (N, K))
    va[5] = 0                                            # an all-zero row of C
    enc = lambda v: np.where(v > 0, ONE[E4M3], np.where(v < 0, ONE[E4M3] | 0x80, 0)).astype(np.uint8)
    sa = (124 + rng.integers(0, 7, (M, 1))).astype(np.uint8)
    sb_rows = (125 + rng.integers(0, 5, (N // 128, 1))).astype(np.uint8)
    sb = np.repeat(sb_rows, K // 128, axis=1)
    return enc(va), sa, enc(vb), sb


def _bf16_exact(c):
    t = torch.from_numpy(c)
    b = t.to(torch.bfloat16)
    assert torch.equal(b.to(torch.float64), t)
    return workloads.bf16_bits(b)


@pytest.mark.parametrize("fmt_c", [E4M3, E5M2])
def test_exact_products_bit_exact(cuda_lib, fmt_c):
    rng = np.random.default_rng(40 + fmt_c)
    M, N, K = 256, 384, 256                              # N: one full and one half n-tile
    qa, sa, qb, sb = _int_operands(rng, M, N, K)
    a = to_qtensor(qa, sa, E4M3, GRAN_ROW)
    b = to_qtensor(qb, sb, E4M3, GRAN_128x128)
    out = fp8hg.fp8_gemm_scaled_q(fp8hg.FPROP, a, b, fmt_c)
    assert fp8hg.fp8hg_get_device_error() == 0
    c_ref, _ = oracle.gemm_ref_dense(oracle.dequant(qa, sa, GRAN_ROW, E4M3),
                                     oracle.dequant(qb, sb, GRAN_128x128, E4M3))
    qo, so = oracle.quant_token(_bf16_exact(c_ref), 128, fmt_c)
    assert_codes_equal(np_u8(out.codes), qo, "codes")
    assert_codes_equal(np_u8(out.scales()), so, "scales")
    assert (so[5] == 0).all()                            # zero group: exponent -127

    # the quantized C is a 1x128 operand: feed it to a second GEMM
    qw, sw = oracle_quant(workloads.bf16_bits(workloads.make_tensor("weight", 256, N, 41, "W2")),
                          GRAN_128x128, E4M3)
    y = fp8hg.fp8_gemm_scaled(fp8hg.FPROP, out, to_qtensor(qw, sw, E4M3, GRAN_128x128))
    y_ref, s_abs = oracle.gemm_ref_dense(oracle.dequant(qo, so, GRAN_1x128, fmt_c),
                                         oracle.dequant(qw, sw, GRAN_128x128, E4M3))
    check_gemm(y.float().cpu().numpy(), y_ref, s_abs, "chained GEMM")


def _positive_grid(fmt):
    t = oracle.decode_table(fmt)[:128]
    return np.sort(t[np.isfinite(t)])


def check_quantized_output(codes, scales, c_ref, s_abs, fmt, what):
    """codes [r, n], scales [r, n/128] from the GPU; c_ref, s_abs [r, n] fp64."""
    tol = oracle.gemm_tolerance(c_ref, s_abs)
    grid = _positive_grid(fmt)
    dec = oracle.decode_table(fmt)
    r, n = c_ref.shape
    for i in range(r):
        for g in range(n // 128):
            cs = slice(128 * g, 128 * g + 128)
            amax = np.abs(c_ref[i, cs]).max()
            slack = tol[i, cs].max()
            allowed = {oracle.ue8m0_exp(max(amax - slack, 0.0), fmt),
                       oracle.ue8m0_exp(amax, fmt), oracle.ue8m0_exp(amax + slack, fmt)}
            e = int(scales[i, g]) - 127
            assert e in allowed, f"{what}: row {i} group {g}: exponent {e}, expected {allowed}"
            y_hi = (np.abs(c_ref[i, cs]) + tol[i, cs]) * 2.0 ** -e
            k = np.minimum(np.searchsorted(grid, y_hi), len(grid) - 1)
            step = grid[k] - grid[np.maximum(k - 1, 0)]          # spacing just above y_hi
            x_hat = dec[codes[i, cs]] * 2.0 ** e
            err = np.abs(x_hat - c_ref[i, cs])
            bound = tol[i, cs] + 0.5 * step * 2.0 ** e
            bad = ~(err <= bound)
            assert not bad.any(), (f"{what}: row {i} col {128 * g + np.argmax(bad)}: "
                                   f"{x_hat[bad][0]} vs {c_ref[i, cs][bad][0]}")
            # the code is the RNE encoding of a value within tolerance of C
            enc = lambda y: dec[oracle.fp8_encode(float(y), fmt, True)]
            lo = np.array([enc(y) for y in (c_ref[i, cs] - tol[i, cs]) * 2.0 ** -e])
            hi = np.array([enc(y) for y in (c_ref[i, cs] + tol[i, cs]) * 2.0 ** -e])
            got = dec[codes[i, cs]]
            bad = ~((lo <= got) & (got <= hi))
            assert not bad.any(), (f"{what}: row {i} col {128 * g + np.argmax(bad)}: code value "
                                   f"{got[bad][0]} outside [{lo[bad][0]}, {hi[bad][0]}]")


@pytest.mark.parametrize("fmt_c", [E4M3, E5M2])
def test_tiny_fprop_tolerance(cuda_lib, fmt_c):
    x = workloads.workload_tensor("tiny_fprop", "X")
    w = workloads.workload_tensor("tiny_fprop", "W")
    qx, sx = oracle.quant_token(workloads.bf16_bits(x), 0, E4M3)
    qw, sw, _, _ = oracle.quant_block128(workloads.bf16_bits(w), E4M3)
    out = fp8hg.fp8_gemm_scaled_q(fp8hg.FPROP, to_qtensor(qx, sx, E4M3, GRAN_ROW),
                                  to_qtensor(qw, sw, E4M3, GRAN_128x128), fmt_c)
    assert fp8hg.fp8hg_get_device_error() == 0
    c_ref, s_abs = oracle.gemm_ref_dense(oracle.dequant(qx, sx, GRAN_ROW, E4M3),
                                         oracle.dequant(qw, sw, GRAN_128x128, E4M3))
    check_quantized_output(np_u8(out.codes), np_u8(out.scales()), c_ref, s_abs, fmt_c, "tiny")


def test_1p5b_gate_sampled_rows(cuda_lib):
    """X [8192, 1536] x W_gate [8960, 1536]^T, C quantized E4M3; 6 sampled rows
    (all 8960 columns, 70 groups each)."""
    x = workloads.workload_tensor("fprop_1p5b", "X")
    w = workloads.workload_tensor("fprop_1p5b", "W_gate")
    qx, sx = oracle.quant_token(workloads.bf16_bits(x), 0, E4M3)
    qw, sw, _, _ = oracle.quant_block128(workloads.bf16_bits(w), E4M3)
    out = fp8hg.fp8_gemm_scaled_q(fp8hg.FPROP, to_qtensor(qx, sx, E4M3, GRAN_ROW),
                                  to_qtensor(qw, sw, E4M3, GRAN_128x128), E4M3)
    assert fp8hg.fp8hg_get_device_error() == 0
    rows = np.array([0, 8191] + list(np.random.default_rng(9).choice(8192, 4, replace=False)))
    codes = np_u8(out.codes[torch.from_numpy(rows).cuda()])
    scales = np_u8(out.scales()[torch.from_numpy(rows).cuda()])
    I, J = np.meshgrid(np.arange(len(rows)), np.arange(8960), indexing="ij")
    c_ref, s_abs = oracle.gemm_ref_pairs(qx[rows], sx[rows], GRAN_ROW, E4M3, qw, sw,
                                         GRAN_128x128, E4M3, I.ravel(), J.ravel())
    check_quantized_output(codes, scales, c_ref.reshape(len(rows), 8960),
                           s_abs.reshape(len(rows), 8960), E4M3, "1.5B gate")


@pytest.mark.parametrize("fmt_c", [E4M3, E5M2])
def test_mx32_operands_exact_products(cuda_lib, fmt_c):
    """MX32 x MX32 operands (the G = 4 instantiation of the quantized epilogue):
    codes -1 / 0 / +1 and per-32-K scale bytes that are the row's byte in every
    block, so C is exact in FP32 and BF16 and its quantization must equal the
    oracle's bit for bit; a wrong scale slot or byte changes C by a power of two."""
    rng = np.random.default_rng(60 + fmt_c)
    M, N, K = 256, 384, 256
    qa, sa_row, qb, sb_blk = _int_operands(rng, M, N, K)
    sa = np.repeat(sa_row, K // 32, axis=1)                      # [M, K/32]
    sb = np.repeat(np.repeat(sb_blk[:, :1], 128, axis=0), K // 32, axis=1)  # [N, K/32]
    a = to_qtensor(qa, sa, E4M3, GRAN_MX32)
    b = to_qtensor(qb, sb, E4M3, GRAN_MX32)
    out = fp8hg.fp8_gemm_scaled_q(fp8hg.FPROP, a, b, fmt_c)
    assert fp8hg.fp8hg_get_device_error() == 0
    c_ref, _ = oracle.gemm_ref_dense(oracle.dequant(qa, sa, GRAN_MX32, E4M3),
                                     oracle.dequant(qb, sb, GRAN_MX32, E4M3))
    qo, so = oracle.quant_token(_bf16_exact(c_ref), 128, fmt_c)
    assert_codes_equal(np_u8(out.codes), qo, "codes")
    assert_codes_equal(np_u8(out.scales()), so, "scales")


@pytest.mark.parametrize("fmt_c", [E4M3, E5M2])
def test_mx32_operands_tolerance(cuda_lib, fmt_c):
    """MX32 x MX32 on the MX workload's layer-norm-like and normal rows (scales
    that differ from block to block along K), C quantized in the epilogue."""
    M, N, K = 256, 256, 512
    xa = workloads.bf16_bits(workloads.make_tensor("mx_ln", M, K, 61, "qa"))
    xb = workloads.bf16_bits(workloads.make_tensor("normal", N, K, 62, "qb"))
    qa, sa = oracle_quant(xa, GRAN_MX32, E4M3)
    qb, sb = oracle_quant(xb, GRAN_MX32, E5M2)
    out = fp8hg.fp8_gemm_scaled_q(fp8hg.FPROP, to_qtensor(qa, sa, E4M3, GRAN_MX32),
                                  to_qtensor(qb, sb, E5M2, GRAN_MX32), fmt_c)
    assert fp8hg.fp8hg_get_device_error() == 0
    c_ref, s_abs = oracle.gemm_ref_dense(oracle.dequant(qa, sa, GRAN_MX32, E4M3),
                                         oracle.dequant(qb, sb, GRAN_MX32, E5M2))
    check_quantized_output(np_u8(out.codes), np_u8(out.scales()), c_ref, s_abs, fmt_c, "mx32")
