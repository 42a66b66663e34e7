"""The C-ABI library loads without a GPU, exports every function the header
declares, and rejects bad arguments before launching anything.  No call here
reaches the device."""
import ctypes

import pytest

import fp8_hybrid_granularity_gb300 as fp8hg
from fp8_hybrid_granularity_gb300 import Operand, E4M3, GRAN_ROW, GRAN_1x128, GRAN_128x128, GRAN_MX32

EXPECTED = {"fp8_quant_token", "fp8_quant_block128", "fp8_quant_mx32", "fp8_quant_mx32_monitor",
            "fp8_requant_t", "fp8_gemm_scaled_q", "fp8_quant_token_f32s",
            "fp8_quant_block128_f32s", "fp8_gemm_scaled_f32s",
            "fp8_gemm_scaled",
            "fp8_gemm_scaled_ex", "fp8hg_get_device_error", "fp8hg_status_str", "fp8hg_version",
            "fp8_quant_token_ex", "fp8_requant_t_ex", "fp8_gemm_scaled_f32s_ex",
            "fp8_quant_token_dual", "fp8_quant_token_dual_workspace",
            "fp8_quant_token_dual_noalloc", "fp8_gemm_scaled_splitk",
            "fp8_gemm_splitk_workspace", "fp8_quant_block128_batch"}

OK, INVALID, ALIGN, SHAPE, UNSUP = 0, 1, 2, 3, 4
FAKE = 0x10000  # never dereferenced: every call below fails validation first


@pytest.fixture(scope="module")
def lib():
    return fp8hg.load_library()


def test_header_declares_the_expected_api():
    assert set(fp8hg.declared_functions()) == EXPECTED


def test_library_exports_every_declared_symbol(lib):
    for name in fp8hg.declared_functions():
        assert hasattr(lib, name), name
    assert lib.fp8hg_version() == (1 << 16)


def test_status_strings(lib):
    for code, name in fp8hg.STATUS.items():
        assert lib.fp8hg_status_str(code).decode() == name
    assert lib.fp8hg_status_str(99).decode() == "FP8HG_UNKNOWN_STATUS"


def test_quant_token_validation(lib):
    q = lib.fp8_quant_token
    assert q(None, 4, 128, 128, 0, 0, E4M3, FAKE, 128, FAKE, 1, None) == INVALID
    assert q(FAKE, 4, 128, 128, 64, 0, E4M3, FAKE, 128, FAKE, 1, None) == INVALID     # group
    assert q(FAKE, 4, 128, 128, 0, 0, 7, FAKE, 128, FAKE, 1, None) == INVALID         # fmt
    assert q(FAKE + 8, 4, 128, 128, 0, 0, E4M3, FAKE, 128, FAKE, 1, None) == ALIGN    # x align
    assert q(FAKE, 4, 128, 130, 0, 0, E4M3, FAKE, 128, FAKE, 1, None) == ALIGN        # ld_x
    assert q(FAKE, 4, 100, 104, 0, 0, E4M3, FAKE, 112, FAKE, 1, None) == SHAPE        # cols
    assert q(FAKE, 4, 128, 128, 0, 1, E4M3, FAKE, 128, FAKE, 1, None) == UNSUP        # ROW^T
    assert q(FAKE, 100, 128, 128, 128, 1, E4M3, FAKE, 128, FAKE, 1, None) == SHAPE    # rows%128
    assert q(FAKE, 4, 256, 128, 0, 0, E4M3, FAKE, 256, FAKE, 1, None) == INVALID      # ld_x < cols
    assert q(FAKE, 4, 256, 256, 128, 0, E4M3, FAKE, 256, FAKE, 1, None) == INVALID    # ld_s < 2


def test_block128_and_mx_validation(lib):
    b = lib.fp8_quant_block128
    assert b(FAKE, 100, 128, 128, E4M3, FAKE, 128, FAKE, 1, None, 0, None, 0, None) == SHAPE
    assert b(FAKE, 128, 128, 128, E4M3, FAKE, 128, FAKE, 1, FAKE, 128, None, 0, None) == INVALID
    assert b(FAKE, 128, 128, 128, E4M3, FAKE, 128, FAKE, 1, FAKE + 4, 128, FAKE, 1, None) == ALIGN
    m = lib.fp8_quant_mx32
    assert m(FAKE, 4, 48, 48, E4M3, FAKE, 48, FAKE, 2, None, None) == SHAPE
    assert m(FAKE, 4, 64, 64, E4M3, FAKE, 64, FAKE, 2, FAKE + 4, None) == ALIGN
    mon = lib.fp8_quant_mx32_monitor
    assert mon(FAKE, 4, 64, 64, E4M3, FAKE, 64, FAKE, 2, None, None, None) == INVALID  # stats
    assert mon(FAKE, 4, 48, 48, E4M3, FAKE, 48, FAKE, 2, FAKE, None, None) == SHAPE
    assert mon(FAKE, 4, 64, 64, E4M3, FAKE, 64, FAKE, 2, FAKE + 4, None, None) == ALIGN
    assert mon(FAKE, 4, 64, 64, E4M3, FAKE, 64, FAKE, 2, FAKE, FAKE + 2, None) == ALIGN
    assert mon(FAKE, 4, 64, 64, E4M3, FAKE, 64, FAKE, 1, FAKE, None, None) == INVALID  # ld_s
    assert mon(FAKE, 0, 64, 64, E4M3, FAKE, 64, FAKE, 2, FAKE, None, None) == OK       # empty


def test_block128_batch_validation(lib):
    """Every job is checked before anything is launched; none of these reaches
    the device (the ones that pass validation have no blocks to launch)."""
    J = fp8hg._Block128Job

    def job(rows=128, cols=128, ld_x=128, q=FAKE, ld_q=128, s=FAKE, ld_s=1, qt=None, ld_qt=0,
            st=None, ld_st=0, x=FAKE):
        return J(x, rows, cols, ld_x, q, ld_q, s, ld_s, qt, ld_qt, st, ld_st)

    def call(*jobs, n=None, fmt=E4M3):
        arr = (J * max(len(jobs), 1))(*jobs)
        return lib.fp8_quant_block128_batch(ctypes.addressof(arr), len(jobs) if n is None else n,
                                            fmt, None)

    assert call(n=0) == OK                                    # nothing to do
    assert call(job(), n=-1) == INVALID
    assert call(*[job()] * 9) == INVALID                      # more than FP8HG_BATCH_MAX
    assert lib.fp8_quant_block128_batch(None, 1, E4M3, None) == INVALID
    assert call(job(), fmt=7) == INVALID
    assert call(job(rows=0), job(cols=0)) == OK               # empty jobs are skipped
    assert call(job(), job(rows=100)) == SHAPE                # the second job's shape
    assert call(job(), job(x=FAKE + 8)) == ALIGN
    assert call(job(), job(ld_x=64)) == INVALID               # ld_x < cols
    assert call(job(), job(ld_s=0)) == INVALID
    assert call(job(qt=FAKE, ld_qt=128)) == INVALID           # q_t without scale_t
    # the transposed copy for every job or for none
    assert call(job(qt=FAKE, ld_qt=128, st=FAKE, ld_st=1), job()) == INVALID
    assert call(job(qt=FAKE + 4, ld_qt=128, st=FAKE, ld_st=1)) == ALIGN
    assert call(job(qt=FAKE, ld_qt=136, st=FAKE, ld_st=1)) == ALIGN       # ld_qt % 16 != 0
    assert call(job(qt=FAKE, ld_qt=112, st=FAKE, ld_st=1)) == INVALID     # ld_qt < rows


def test_requant_validation(lib):
    r = lib.fp8_requant_t

    def call(rows=256, cols=256, ld_q=256, ld_s=2, gran=GRAN_1x128, fi=E4M3, fo=E4M3, q=FAKE,
             qt=FAKE, ld_qt=256, ld_st=2, s=FAKE, st=FAKE):
        return r(q, rows, cols, ld_q, s, ld_s, gran, fi, fo, qt, ld_qt, st, ld_st, None)

    assert call(gran=GRAN_128x128) == UNSUP
    assert call(fi=5) == INVALID
    assert call(fo=-1) == INVALID
    assert call(rows=0) == OK                       # empty: nothing read or written
    assert call(q=None) == INVALID
    assert call(st=None) == INVALID
    assert call(q=FAKE + 8) == ALIGN
    assert call(ld_qt=264) == ALIGN
    assert call(rows=200, ld_qt=208) == SHAPE
    assert call(cols=192, ld_q=192) == SHAPE
    assert call(ld_q=128) == INVALID                # ld_q < cols
    assert call(ld_s=1) == INVALID                  # 1x128 needs cols/128 scale columns
    assert call(ld_st=1) == INVALID                 # rows/128 output scale columns


def _op(rows=256, k=256, gran=GRAN_1x128, ld=None, lds=4, fmt=E4M3, scale=FAKE):
    return Operand(FAKE, scale, rows, k, ld if ld is not None else k, lds, fmt, gran)


def test_gemm_q_validation(lib):
    g = lib.fp8_gemm_scaled_q
    blk = dict(gran=GRAN_128x128, lds=4)

    def call(a=None, b=None, c=FAKE, ldc=256, cs=FAKE, ldcs=4, fmt=E4M3, op=0):
        a = a or _op()
        b = b or _op(**blk)
        return g(op, ctypes.byref(a), ctypes.byref(b), c, ldc, cs, ldcs, fmt, None)

    assert call(fmt=3) == INVALID
    assert call(c=None) == INVALID
    assert call(cs=None) == INVALID
    assert call(c=FAKE + 8) == ALIGN
    assert call(ldc=264) == ALIGN
    assert call(ldc=128) == INVALID                 # ldc < N
    assert call(ldcs=1) == INVALID                  # N/128 = 2 scale columns
    assert call(b=_op(gran=GRAN_1x128)) == UNSUP    # fprop needs block B
    assert call(a=_op(rows=200)) == SHAPE
    assert call(op=7) == INVALID


def test_f32s_validation(lib):
    qt = lib.fp8_quant_token_f32s
    assert qt(FAKE, 4, 128, 128, 64, E4M3, FAKE, 128, FAKE, 1, None) == INVALID    # group
    assert qt(FAKE, 4, 128, 128, 0, E4M3, FAKE, 128, FAKE + 2, 1, None) == ALIGN   # scale align
    assert qt(FAKE, 4, 96, 96, 0, E4M3, FAKE, 112, FAKE, 1, None) == SHAPE
    assert qt(FAKE, 4, 256, 256, 128, E4M3, FAKE, 256, FAKE, 1, None) == INVALID   # ld_s
    qb = lib.fp8_quant_block128_f32s
    assert qb(FAKE, 100, 128, 128, E4M3, FAKE, 128, FAKE, 1, None, 0, None, 0, None) == SHAPE
    assert qb(FAKE, 128, 128, 128, E4M3, FAKE, 128, FAKE, 1, FAKE, 128, None, 0, None) == INVALID
    g = lib.fp8_gemm_scaled_f32s

    def call(a, b, op=0, c=FAKE, ldc=256, out=0):
        return g(op, ctypes.byref(a), ctypes.byref(b), c, ldc, out, None)

    blk = dict(gran=GRAN_128x128, lds=2)
    assert call(_op(gran=GRAN_ROW, lds=1), _op(**blk), op=2) == UNSUP     # wgrad
    assert call(_op(), _op(gran=GRAN_1x128, lds=2)) == UNSUP             # B must be blocks
    assert call(_op(gran=GRAN_MX32, lds=8), _op(**blk)) == UNSUP
    assert call(_op(rows=200), _op(**blk)) == SHAPE
    assert call(_op(lds=1), _op(**blk)) == INVALID                       # 1x128 needs K/128
    assert call(_op(scale=FAKE + 2), _op(**blk)) == ALIGN
    assert call(_op(), _op(**blk), out=2) == INVALID
    assert call(_op(), _op(**blk), ldc=100) == INVALID


def test_gemm_options_validation(lib):
    g = lib.fp8_gemm_scaled_ex
    blk = dict(gran=GRAN_128x128, lds=4)

    def call(a, opts):
        return g(0, ctypes.byref(a), ctypes.byref(_op(**blk)), FAKE, 256, 0, 0,
                 ctypes.byref(opts), None)

    assert call(_op(), fp8hg.GemmOpts(0, 0, 4)) == INVALID        # tile selector
    assert call(_op(), fp8hg.GemmOpts(0, 0, -1)) == INVALID
    assert call(_op(), fp8hg.GemmOpts(0, 2, 0)) == INVALID        # inject_fault
    assert call(_op(rows=128), fp8hg.GemmOpts(0, 0, 2)) == UNSUP  # 256-row tiles, M = 128
    assert call(_op(rows=384), fp8hg.GemmOpts(0, 0, 3)) == UNSUP  # CTA pairs, M % 256 != 0


def test_splitk_validation(lib):
    """fp8_gemm_scaled_splitk: split_k in 0..8 and at most K/128, forced
    splits only on 256-row tiles with a large enough, 256-byte aligned
    workspace, inject_fault 2 only with a split; the workspace size
    function's layout (flags padded to 256 bytes, then FP32 partial tiles)."""
    g = lib.fp8_gemm_scaled_splitk
    W = 1 << 40                      # "large enough" (never touched)

    def sc(k):                        # scale columns, padded to four
        return (k // 128 + 3) // 4 * 4

    def call(a=None, split=2, ws=FAKE * 256, wsb=W, opts=None, k=1024):
        a = a or _op(rows=512, k=k, lds=sc(k))
        b = _op(rows=384, k=k, gran=GRAN_128x128, lds=sc(k))
        return g(0, ctypes.byref(a), ctypes.byref(b), FAKE, 384, 0, 0,
                 split, ws, wsb, ctypes.byref(opts) if opts else None, None)

    assert call(split=9) == INVALID
    assert call(split=-1) == INVALID
    assert call(split=4, k=384) == SHAPE                          # more parts than k-blocks
    assert call(a=_op(rows=384, k=1024, lds=8)) == UNSUP          # M % 256
    assert call(opts=fp8hg.GemmOpts(0, 0, 1)) == UNSUP            # forced 128 x 256 tiles
    assert call(ws=None) == INVALID
    assert call(wsb=1000) == INVALID
    assert call(ws=FAKE * 256 + 16) == ALIGN
    assert call(opts=fp8hg.GemmOpts(0, 3, 0)) == INVALID          # inject_fault
    assert call(split=1, opts=fp8hg.GemmOpts(0, 2, 0)) == UNSUP   # injection needs a split
    ws = lib.fp8_gemm_splitk_workspace
    tiles = 2 * 2                                                  # 512 / 256 x ceil(384 / 224)
    assert ws(512, 384, 2048, 2) == 256 + tiles * 1 * 256 * 224 * 4
    assert ws(512, 384, 2048, 3) == 256 + tiles * 2 * 256 * 224 * 4
    assert ws(512, 384, 2048, 1) == 0
    assert ws(384, 384, 2048, 2) == 0                             # M % 256
    assert ws(512, 384, 256, 3) == 0                              # more parts than k-blocks


def test_gemm_validation(lib):
    g = lib.fp8_gemm_scaled
    C = FAKE

    def call(a, b, op=0, ldc=256, out=0, acc=0, c=C):
        return g(op, ctypes.byref(a), ctypes.byref(b), c, ldc, out, acc, None)

    blk = dict(gran=GRAN_128x128, lds=4)
    assert call(_op(rows=200), _op(**blk)) == SHAPE
    assert call(_op(k=200), _op(k=200, **blk)) == SHAPE
    assert call(_op(k=256), _op(k=384, **blk)) == SHAPE
    assert call(_op(ld=264), _op(**blk)) == ALIGN                  # ld % 16
    assert call(_op(lds=2), _op(**blk)) == ALIGN                   # ld_scale % 4
    assert call(_op(scale=FAKE + 1), _op(**blk)) == ALIGN          # scale alignment
    assert call(_op(), _op(gran=GRAN_1x128)) == UNSUP              # fprop needs block B
    assert call(_op(gran=GRAN_MX32, lds=8), _op(**blk)) == UNSUP   # MX only with MX
    assert call(_op(gran=GRAN_ROW, lds=1), _op(**blk), op=2) == UNSUP  # wgrad needs 1x128
    assert call(_op(), _op(**blk), op=5) == INVALID
    assert call(_op(), _op(**blk), out=3) == INVALID
    assert call(_op(), _op(**blk), c=None) == INVALID
    assert call(_op(), _op(**blk), c=FAKE + 8) == ALIGN
    assert call(_op(), _op(**blk), ldc=100) == INVALID
    assert call(_op(), _op(**blk), ldc=260) == ALIGN
    a = _op()
    a.fmt = 9
    assert call(a, _op(**blk)) == INVALID


def test_wait_options_validation(lib):
    """fp8hg_wait_opts: inject_fault in {0, 1}, reserved 0, and fault injection
    only where the kernel waits on copies (per-token rows of more than 4096
    elements for fp8_quant_token_ex)."""
    W = fp8hg.WaitOpts
    qx = lib.fp8_quant_token_ex

    def tok(opts, cols=8192, group=0, transpose=0):
        return qx(FAKE, 128, cols, cols, group, transpose, E4M3, FAKE, cols, FAKE,
                  cols // 128, ctypes.byref(opts), None)

    assert tok(W(0, 2, 0)) == INVALID
    assert tok(W(0, 0, 1)) == INVALID                       # reserved
    assert tok(W(0, 1, 0), cols=1024) == UNSUP               # 2 KB rows: register kernel, no wait
    assert tok(W(0, 1, 0), group=128) == UNSUP               # 1x128: no wait
    assert tok(W(0, 1, 0), group=128, transpose=1) == UNSUP  # transposed: no wait
    assert qx(FAKE, 0, 8192, 8192, 0, 0, E4M3, FAKE, 8192, FAKE, 1,
              ctypes.byref(W(5, 1, 0)), None) == OK           # empty: nothing launched
    r = lib.fp8_requant_t_ex
    assert r(FAKE, 256, 256, 256, FAKE, 2, GRAN_1x128, E4M3, E4M3, FAKE, 256, FAKE, 2,
             ctypes.byref(W(0, 3, 0)), None) == INVALID
    g = lib.fp8_gemm_scaled_f32s_ex
    blk = dict(gran=GRAN_128x128, lds=2)
    assert g(0, ctypes.byref(_op()), ctypes.byref(_op(**blk)), FAKE, 256, 0,
             ctypes.byref(W(0, -1, 0)), None) == INVALID


def test_dual_quant_validation(lib):
    d = lib.fp8_quant_token_dual
    ws_need = lib.fp8_quant_token_dual_workspace(256, 256)
    assert ws_need >= 4 * (256 + 2) and ws_need % 256 == 0
    assert lib.fp8_quant_token_dual_workspace(0, 256) == 0

    def call(rows=256, cols=256, fmt=E4M3, fmt_t=E4M3, ws=FAKE, wsb=None, qt=FAKE, ld_qt=256,
             ld_st=2, st=FAKE, x=FAKE, opts=None):
        wsb = ws_need if wsb is None else wsb
        return d(x, rows, cols, cols, fmt, FAKE, cols, FAKE, 1, fmt_t, qt, ld_qt, st, ld_st, ws,
                 wsb, opts, None)

    assert call(fmt_t=4) == INVALID
    assert call(ws=None) == INVALID
    assert call(wsb=ws_need - 1) == INVALID
    assert call(ws=FAKE + 4) == ALIGN
    assert call(qt=FAKE + 8) == ALIGN
    assert call(rows=200, ld_qt=208) == SHAPE
    assert call(cols=192) == SHAPE
    assert call(ld_st=1) == INVALID
    assert call(st=None) == INVALID
    assert call(rows=0) == OK
    assert call(opts=ctypes.byref(fp8hg.WaitOpts(0, 7, 0))) == INVALID
