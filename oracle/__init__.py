"""CPU oracle for hybrid-granularity FP8 quantization and the scaled GEMM.

TEST INFRASTRUCTURE ONLY: imported by the test suite, the package smoke check
and the bench's CPU-baseline / reference arm, never by the product path.  The
arithmetic lives in ``fp8hg_oracle.c`` (plain C, fp64); this module only
compiles it with gcc and marshals numpy arrays through ctypes.

Definitions followed (see the C file for the per-function citations):
  * "FP8 Formats for Deep Learning" -- E4M3 / E5M2 encodings, RNE rounding.
  * "A Comprehensive FP8 Training Recipe for Reasoning-Enhanced Language
    Models" -- hybrid granularity, UE8M0 round-up scales.
  * "Characterization and Mitigation of Training Instabilities in Microscaling
    Formats" -- MX shared scale and saturating clamp.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

E4M3, E5M2 = 0, 1
GRAN_ROW, GRAN_1x128, GRAN_128x128, GRAN_MX32 = 0, 1, 2, 3

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8hg_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``liboracle.so`` (plain gcc, no fast-math)."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)
                 or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
        if force or stale:
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared",
                                   "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        lib.orc_bf16_to_double.restype = ctypes.c_double
        lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.orc_fp8_decode.restype = ctypes.c_double
        lib.orc_fp8_decode.argtypes = [ctypes.c_uint8, I]
        lib.orc_fp8_encode.restype = ctypes.c_uint8
        lib.orc_fp8_encode.argtypes = [ctypes.c_double, I, I]
        lib.orc_fp8_max.restype = ctypes.c_double
        lib.orc_fp8_max.argtypes = [I]
        lib.orc_ue8m0_exp.restype = I
        lib.orc_ue8m0_exp.argtypes = [ctypes.c_double, I]
        lib.orc_mx_exp.restype = I
        lib.orc_mx_exp.argtypes = [ctypes.c_double, I]
        lib.orc_quant_token.restype = I
        lib.orc_quant_token.argtypes = [P, I64, I64, I64, I, I, I, P, I64, P, I64]
        lib.orc_quant_block128.restype = I
        lib.orc_quant_block128.argtypes = [P, I64, I64, I64, I, P, I64, P, I64, P, I64, P, I64]
        lib.orc_quant_mx32.restype = I
        lib.orc_quant_mx32.argtypes = [P, I64, I64, I64, I, P, I64, P, I64, P]
        lib.orc_mx32_monitor.restype = I
        lib.orc_mx32_monitor.argtypes = [P, I64, I64, I64, I, P, I64, P, I64, P, P]
        lib.orc_requant_t.restype = I
        lib.orc_requant_t.argtypes = [P, I64, I64, I64, P, I64, I, I, I, P, I64, P, I64]
        lib.orc_quant_token_f32s.restype = I
        lib.orc_quant_token_f32s.argtypes = [P, I64, I64, I64, I, I, P, I64, P, I64]
        lib.orc_quant_block128_f32s.restype = I
        lib.orc_quant_block128_f32s.argtypes = [P, I64, I64, I64, I, P, I64, P, I64, P, I64, P, I64]
        lib.orc_dequant_f32s.restype = I
        lib.orc_dequant_f32s.argtypes = [P, I64, P, I64, I, I, I64, I64, P]
        lib.orc_dequant.restype = I
        lib.orc_dequant.argtypes = [P, I64, P, I64, I, I, I64, I64, P]
        lib.orc_gemm_ref_pairs.restype = I
        lib.orc_gemm_ref_pairs.argtypes = [P, I64, P, I64, I, I, P, I64, P, I64, I, I, I64,
                                           P, P, I64, P, P]
        lib.orc_gemm_ref_dense.restype = I
        lib.orc_gemm_ref_dense.argtypes = [P, P, I64, I64, I64, P, P]
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _u16(x):
    x = np.asarray(x)
    if x.dtype != np.uint16:
        raise TypeError("BF16 inputs are passed as uint16 bit patterns")
    return np.ascontiguousarray(x)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what}: bad arguments (rc={rc})")


# --- scalar format helpers -------------------------------------------------

def bf16_to_double(bits: int) -> float:
    return _load().orc_bf16_to_double(int(bits))


def fp8_decode(code: int, fmt: int) -> float:
    return _load().orc_fp8_decode(int(code), int(fmt))


def fp8_encode(y: float, fmt: int, saturate: bool = False) -> int:
    return int(_load().orc_fp8_encode(float(y), int(fmt), 1 if saturate else 0))


def fp8_max(fmt: int) -> float:
    return _load().orc_fp8_max(int(fmt))


def ue8m0_exp(amax: float, fmt: int) -> int:
    return int(_load().orc_ue8m0_exp(float(amax), int(fmt)))


def mx_exp(amax: float, fmt: int) -> int:
    return int(_load().orc_mx_exp(float(amax), int(fmt)))


def decode_table(fmt: int) -> np.ndarray:
    """All 256 code values as float64 (NaN / inf where the format says so)."""
    return np.array([fp8_decode(c, fmt) for c in range(256)], dtype=np.float64)


# --- quantizers -------------------------------------------------------------

def quant_token(x, group: int, fmt: int, transpose: bool = False):
    """Returns (q, scale).  group 0 = per row (token), 128 = per 1x128 group.

    transpose=True: groups of 128 along the rows; q is [cols, rows],
    scale is [cols, rows/128]."""
    x = _u16(x)
    rows, cols = x.shape
    if transpose:
        q = np.empty((cols, rows), np.uint8)
        s = np.empty((cols, rows // 128), np.uint8)
    else:
        ng = 1 if group == 0 else cols // group
        q = np.empty((rows, cols), np.uint8)
        s = np.empty((rows, ng), np.uint8)
    rc = _load().orc_quant_token(_ptr(x), rows, cols, cols, int(group), 1 if transpose else 0,
                                 int(fmt), _ptr(q), q.shape[1], _ptr(s), s.shape[1])
    _check(rc, "quant_token")
    return q, s


def quant_block128(x, fmt: int, transposed_copy: bool = False):
    """Returns (q, scale, q_t, scale_t); q_t / scale_t are None unless asked."""
    x = _u16(x)
    rows, cols = x.shape
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows // 128, cols // 128), np.uint8)
    qt = st = None
    if transposed_copy:
        qt = np.empty((cols, rows), np.uint8)
        st = np.empty((cols // 128, rows // 128), np.uint8)
    rc = _load().orc_quant_block128(_ptr(x), rows, cols, cols, int(fmt), _ptr(q), cols,
                                    _ptr(s), s.shape[1], _ptr(qt), rows,
                                    _ptr(st), rows // 128)
    _check(rc, "quant_block128")
    return q, s, qt, st


def quant_mx32(x, fmt: int):
    """Returns (q, scale, clamp_count)."""
    x = _u16(x)
    rows, cols = x.shape
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows, cols // 32), np.uint8)
    cnt = np.zeros(1, np.uint64)
    rc = _load().orc_quant_mx32(_ptr(x), rows, cols, cols, int(fmt), _ptr(q), cols,
                                _ptr(s), s.shape[1], _ptr(cnt))
    _check(rc, "quant_mx32")
    return q, s, int(cnt[0])


MX_STAT_NAMES = ("saturated", "top_code", "blocks_saturated", "blocks_collapsed")


def mx32_monitor(x, fmt: int):
    """MX quantization with the clamp monitor's counts.  Returns
    (q, scale, stats dict, per-row saturated counts)."""
    x = _u16(x)
    rows, cols = x.shape
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows, cols // 32), np.uint8)
    st = np.zeros(4, np.uint64)
    rs = np.zeros(rows, np.uint64)
    rc = _load().orc_mx32_monitor(_ptr(x), rows, cols, cols, int(fmt), _ptr(q), cols,
                                  _ptr(s), s.shape[1], _ptr(st), _ptr(rs))
    _check(rc, "mx32_monitor")
    return q, s, dict(zip(MX_STAT_NAMES, (int(v) for v in st))), rs


# --- dequantization and GEMM ------------------------------------------------

def dequant(q, scale, gran: int, fmt: int) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    scale = np.ascontiguousarray(scale, dtype=np.uint8)
    rows, k = q.shape
    out = np.empty((rows, k), np.float64)
    _load().orc_dequant(_ptr(q), k, _ptr(scale), scale.shape[1], int(gran), int(fmt),
                        rows, k, _ptr(out))
    return out


def quant_token_f32s(x, group: int, fmt: int):
    """FP32-scale variant: (q [rows, cols], scale float32 [rows, ngroups])."""
    x = _u16(x)
    rows, cols = x.shape
    ng = 1 if group == 0 else cols // 128
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows, ng), np.float32)
    rc = _load().orc_quant_token_f32s(_ptr(x), rows, cols, cols, int(group), int(fmt), _ptr(q),
                                      cols, _ptr(s), ng)
    _check(rc, "quant_token_f32s")
    return q, s


def quant_block128_f32s(x, fmt: int, transposed_copy: bool = False):
    """FP32-scale variant: (q, scale float32 [rows/128, cols/128], q_t, scale_t)."""
    x = _u16(x)
    rows, cols = x.shape
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows // 128, cols // 128), np.float32)
    qt = st = None
    if transposed_copy:
        qt = np.empty((cols, rows), np.uint8)
        st = np.empty((cols // 128, rows // 128), np.float32)
    rc = _load().orc_quant_block128_f32s(_ptr(x), rows, cols, cols, int(fmt), _ptr(q), cols,
                                         _ptr(s), s.shape[1], _ptr(qt), rows, _ptr(st),
                                         rows // 128)
    _check(rc, "quant_block128_f32s")
    return q, s, qt, st


def dequant_f32s(q, scale, gran: int, fmt: int) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    scale = np.ascontiguousarray(scale, dtype=np.float32)
    rows, k = q.shape
    out = np.empty((rows, k), np.float64)
    rc = _load().orc_dequant_f32s(_ptr(q), k, _ptr(scale), scale.shape[1], int(gran), int(fmt),
                                  rows, k, _ptr(out))
    _check(rc, "dequant_f32s")
    return out


def requant_t(q, scale, gran: int, fmt_in: int, fmt_out: int):
    """Stored FP8 operand q [tokens, cols] (ROW or 1x128-along-K scales) ->
    1x128 groups along the tokens, transposed: (q_t [cols, tokens],
    scale_t [cols, tokens/128])."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    scale = np.ascontiguousarray(scale, dtype=np.uint8)
    rows, cols = q.shape
    qt = np.empty((cols, rows), np.uint8)
    st = np.empty((cols, rows // 128), np.uint8)
    rc = _load().orc_requant_t(_ptr(q), rows, cols, cols, _ptr(scale), scale.shape[1], int(gran),
                               int(fmt_in), int(fmt_out), _ptr(qt), rows, _ptr(st), rows // 128)
    _check(rc, "requant_t")
    return qt, st


def gemm_ref_dense(a_hat, b_hat):
    """C_ref = a_hat @ b_hat.T and S = |a_hat| @ |b_hat|.T, in fp64 loops."""
    a = np.ascontiguousarray(a_hat, dtype=np.float64)
    b = np.ascontiguousarray(b_hat, dtype=np.float64)
    M, K = a.shape
    N = b.shape[0]
    c = np.empty((M, N), np.float64)
    s = np.empty((M, N), np.float64)
    _load().orc_gemm_ref_dense(_ptr(a), _ptr(b), M, N, K, _ptr(c), _ptr(s))
    return c, s


def gemm_ref_pairs(qa, sa, gran_a, fmt_a, qb, sb, gran_b, fmt_b, ii, jj):
    """C_ref and S at the output positions (ii[t], jj[t]) of C = A * B^T."""
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qb = np.ascontiguousarray(qb, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=np.uint8)
    sb = np.ascontiguousarray(sb, dtype=np.uint8)
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    K = qa.shape[1]
    assert qb.shape[1] == K and ii.shape == jj.shape
    c = np.empty(ii.shape, np.float64)
    s = np.empty(ii.shape, np.float64)
    _load().orc_gemm_ref_pairs(_ptr(qa), K, _ptr(sa), sa.shape[1], int(gran_a), int(fmt_a),
                               _ptr(qb), K, _ptr(sb), sb.shape[1], int(gran_b), int(fmt_b), K,
                               _ptr(ii), _ptr(jj), ii.size, _ptr(c), _ptr(s))
    return c, s


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """One BF16 ulp at |x| (the spacing of BF16 values in x's binade);
    the smallest BF16 subnormal, 2^-133, where x is zero or subnormal."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    _, p = np.frexp(ax)               # ax = f * 2^p, f in [0.5, 1)
    ulp = np.ldexp(1.0, p - 1 - 7)    # 7 stored mantissa bits
    return np.where(ax < 2.0 ** -126, 2.0 ** -133, ulp)


def gemm_tolerance(c_ref, s_abs):
    """|C_gpu - C_ref| <= 4e-3 * S + one BF16 ulp of |C_ref|."""
    return 4e-3 * np.asarray(s_abs) + bf16_ulp(c_ref)
