"""Out-of-bounds write check with canary bytes (no sanitizer is available).

Every output buffer handed to a kernel is a view into a larger buffer filled
with 0xAB: the row stride is wider than the row (ld > cols), the scale arrays
have padding columns, and two guard rows follow the last row.  After the
call, the view must hold the oracle's result and every byte outside it must
still read 0xAB.  This catches a kernel that writes past `cols` into the
stride gap, past the scale array's meaningful columns, or past the last row.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import E4M3, E5M2, GRAN_ROW, GRAN_1x128, GRAN_128x128, GRAN_MX32
import fp8_hybrid_granularity_gb300 as fp8hg
from fp8_hybrid_granularity_gb300 import workloads
from helpers import np_u8, assert_codes_equal, oracle_quant, to_qtensor, check_gemm

pytestmark = pytest.mark.gpu

CANARY = 0xAB
GUARD = 2


def canvas(rows, cols, ld, dtype=torch.uint8):
    """A [rows + GUARD, ld] buffer of canary bytes and its [rows, cols] view."""
    nbytes = torch.tensor([], dtype=dtype).element_size()
    buf = torch.full(((rows + GUARD) * ld * nbytes,), CANARY, dtype=torch.uint8, device="cuda")
    buf = buf.view(dtype).view(rows + GUARD, ld)
    return buf, buf[:rows, :cols]


def assert_canary(buf, rows, cols, what):
    b = buf.cpu().view(torch.uint8).numpy()
    nbytes = buf.element_size()
    outside = np.ones(b.shape, bool)
    outside[:rows, :cols * nbytes] = False
    bad = np.argwhere(outside & (b != CANARY))
    assert len(bad) == 0, f"{what}: {len(bad)} bytes written outside the output, first at {tuple(bad[0])}"


def _x(kind, rows, cols, seed):
    t = workloads.make_tensor(kind, rows, cols, seed, "canary")
    return t, workloads.bf16_bits(t)


@pytest.mark.parametrize("rows,cols,group", [(256, 384, 0), (128, 8192, 0), (256, 384, 128),
                                             (128, 8192, 128)])
@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_token_quant_canary(cuda_lib, rows, cols, group, fmt):
    """Per-token (short rows: register kernel; 16 KB rows: the bulk-copy row
    kernel) and 1x128 quantization."""
    x, xb = _x("act", rows, cols, rows + cols + group)
    ncs = 1 if group == 0 else cols // 128
    qbuf, q = canvas(rows, cols, cols + 48)
    sbuf, s = canvas(rows, ncs, ncs + 5)
    out = fp8hg.QTensor(q, s, fmt, GRAN_ROW if group == 0 else GRAN_1x128, ncs)
    fp8hg.fp8_quant_token(x.cuda(), group, fmt, out=out)
    assert fp8hg.fp8hg_get_device_error() == 0
    qo, so = oracle.quant_token(xb, group, fmt)
    assert_codes_equal(np_u8(q), qo, "codes")
    assert_codes_equal(np_u8(s), so, "scales")
    assert_canary(qbuf, rows, cols, "codes")
    assert_canary(sbuf, rows, ncs, "scales")


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_transposed_quant_canary(cuda_lib, fmt):
    rows, cols = 384, 192
    x, xb = _x("grad", rows, cols, 7)
    qbuf, q = canvas(cols, rows, rows + 48)
    sbuf, s = canvas(cols, rows // 128, rows // 128 + 5)
    out = fp8hg.QTensor(q, s, fmt, GRAN_1x128, rows // 128)
    fp8hg.fp8_quant_token(x.cuda(), 128, fmt, transpose=True, out=out)
    assert fp8hg.fp8hg_get_device_error() == 0
    qo, so = oracle.quant_token(xb, 128, fmt, transpose=True)
    assert_codes_equal(np_u8(q), qo, "codes")
    assert_codes_equal(np_u8(s), so, "scales")
    assert_canary(qbuf, cols, rows, "codes")
    assert_canary(sbuf, cols, rows // 128, "scales")


def test_block128_canary(cuda_lib):
    rows, cols = 256, 384
    x, xb = _x("weight", rows, cols, 8)
    qbuf, q = canvas(rows, cols, cols + 48)
    sbuf, s = canvas(rows // 128, cols // 128, cols // 128 + 5)
    qtbuf, qt = canvas(cols, rows, rows + 32)
    stbuf, st = canvas(cols // 128, rows // 128, rows // 128 + 3)
    fp8hg.fp8_quant_block128(x.cuda(), E4M3, True,
                             out=fp8hg.QTensor(q, s, E4M3, GRAN_128x128, cols // 128),
                             out_t=fp8hg.QTensor(qt, st, E4M3, GRAN_128x128, rows // 128))
    assert fp8hg.fp8hg_get_device_error() == 0
    qo, so, qto, sto = oracle.quant_block128(xb, E4M3, transposed_copy=True)
    for got, ref, what in ((q, qo, "codes"), (s, so, "scales"), (qt, qto, "codes^T"),
                           (st, sto, "scales^T")):
        assert_codes_equal(np_u8(got), ref, what)
    assert_canary(qbuf, rows, cols, "codes")
    assert_canary(sbuf, rows // 128, cols // 128, "scales")
    assert_canary(qtbuf, cols, rows, "codes^T")
    assert_canary(stbuf, cols // 128, rows // 128, "scales^T")


@pytest.mark.parametrize("monitor", [False, True])
def test_mx32_canary(cuda_lib, monitor):
    rows, cols = 256, 416                      # 13 MX blocks per row
    x, xb = _x("mx_ln_clamp", rows, cols, 9)
    qbuf, q = canvas(rows, cols, cols + 32)
    sbuf, s = canvas(rows, cols // 32, cols // 32 + 6)
    out = fp8hg.QTensor(q, s, E4M3, GRAN_MX32, cols // 32)
    if monitor:
        fp8hg.fp8_quant_mx32_monitor(x.cuda(), E4M3, out=out)
    else:
        fp8hg.fp8_quant_mx32(x.cuda(), E4M3, out=out)
    assert fp8hg.fp8hg_get_device_error() == 0
    qo, so, _ = oracle.quant_mx32(xb, E4M3)
    assert_codes_equal(np_u8(q), qo, "codes")
    assert_codes_equal(np_u8(s), so, "scales")
    assert_canary(qbuf, rows, cols, "codes")
    assert_canary(sbuf, rows, cols // 32, "scales")


def test_requant_canary(cuda_lib):
    rows, cols = 256, 384
    x, xb = _x("act", rows, cols, 10)
    src = fp8hg.fp8_quant_token(x.cuda(), 0, E4M3)
    qbuf, q = canvas(cols, rows, rows + 48)
    sbuf, s = canvas(cols, rows // 128, rows // 128 + 5)
    fp8hg.fp8_requant_t(src, E5M2, out=fp8hg.QTensor(q, s, E5M2, GRAN_1x128, rows // 128))
    assert fp8hg.fp8hg_get_device_error() == 0
    qs, ss = oracle.quant_token(xb, 0, E4M3)
    qo, so = oracle.requant_t(qs, ss, GRAN_ROW, E4M3, E5M2)
    assert_codes_equal(np_u8(q), qo, "codes")
    assert_codes_equal(np_u8(s), so, "scales")
    assert_canary(qbuf, cols, rows, "codes")
    assert_canary(sbuf, cols, rows // 128, "scales")


def test_f32s_token_canary(cuda_lib):
    rows, cols = 256, 384
    x, xb = _x("act", rows, cols, 11)
    qbuf, q = canvas(rows, cols, cols + 48)
    sbuf, s = canvas(rows, cols // 128, cols // 128 + 3, dtype=torch.float32)
    fp8hg.fp8_quant_token_f32s(x.cuda(), 128, E4M3,
                               out=fp8hg.QTensor(q, s, E4M3, GRAN_1x128, cols // 128))
    assert fp8hg.fp8hg_get_device_error() == 0
    qo, so = oracle.quant_token_f32s(xb, 128, E4M3)
    assert_codes_equal(np_u8(q), qo, "codes")
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))
    assert_canary(qbuf, rows, cols, "codes")
    assert_canary(sbuf, rows, cols // 128, "scales")


def _gemm_operands(M, N, K):
    xa = workloads.bf16_bits(workloads.make_tensor("act", M, K, 12, "canary-a"))
    xw = workloads.bf16_bits(workloads.make_tensor("weight", N, K, 13, "canary-b"))
    qa, sa = oracle_quant(xa, GRAN_ROW, E4M3)
    qb, sb = oracle_quant(xw, GRAN_128x128, E4M3)
    ref = oracle.gemm_ref_dense(oracle.dequant(qa, sa, GRAN_ROW, E4M3),
                                oracle.dequant(qb, sb, GRAN_128x128, E4M3))
    return to_qtensor(qa, sa, E4M3, GRAN_ROW), to_qtensor(qb, sb, E4M3, GRAN_128x128), ref


@pytest.mark.parametrize("tile", [1, 2, 3])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("accumulate", [False, True])
def test_gemm_output_canary(cuda_lib, tile, dtype, accumulate):
    """N = 384 ends inside every tile shape's last n-tile (256 + 128, 224 + 160, 448)."""
    M, N, K = 256, 384, 256
    a, b, (c_ref, s_abs) = _gemm_operands(M, N, K)
    cbuf, c = canvas(M, N, N + 64, dtype=dtype)
    if accumulate:
        c.zero_()
    fp8hg.fp8_gemm_scaled(fp8hg.FPROP, a, b, out=c, accumulate=accumulate, tile=tile)
    assert fp8hg.fp8hg_get_device_error() == 0
    check_gemm(c.float().cpu().numpy(), c_ref, s_abs, "gemm")
    assert_canary(cbuf, M, N, "C")


@pytest.mark.parametrize("fmt_c", [E4M3, E5M2])
def test_gemm_q_canary(cuda_lib, fmt_c):
    M, N, K = 256, 384, 256
    a, b, _ = _gemm_operands(M, N, K)
    qbuf, q = canvas(M, N, N + 48)
    sbuf, s = canvas(M, N // 128, N // 128 + 3)
    fp8hg.fp8_gemm_scaled_q(fp8hg.FPROP, a, b, fmt_c,
                            out=fp8hg.QTensor(q, s, fmt_c, GRAN_1x128, N // 128))
    assert fp8hg.fp8hg_get_device_error() == 0
    assert_canary(qbuf, M, N, "codes")
    assert_canary(sbuf, M, N // 128, "scales")
