"""Hybrid-granularity FP8 quantization and block-scaled FP8 GEMM for GB300.

Python binding of the C ABI in ``include/fp8hg.h`` (library ``libfp8hg.so``,
built in-tree from ``csrc/``).  This module only marshals arguments: every
step of the computation runs in the CUDA kernels.  PyTorch supplies device
memory and the current stream.  There is no CPU fallback: if the library is
missing or fails to load, every call raises.

Tensor-level API (same names as the C entry points):

  fp8_quant_token(x, group=0|128, fmt, transpose=False) -> QTensor
  fp8_quant_token_dual(x, fmt, fmt_t)                   -> QTensor, QTensor^T (one read)
  fp8_quant_block128(x, fmt, transposed_copy=False)     -> QTensor[, QTensor]
  fp8_quant_mx32(x, fmt, clamp_count=None)              -> QTensor
  fp8_quant_mx32_monitor(x, fmt, stats=None, row_saturated=None) -> QTensor, stats
  fp8_requant_t(src QTensor, fmt)                       -> QTensor (transposed)
  fp8_gemm_scaled(op, a, b, out=None, out_dtype=bf16, accumulate=False)
  fp8_gemm_scaled_q(op, a, b, fmt)                      -> QTensor (1x128 along N)
  fp8_quant_token_f32s / fp8_quant_block128_f32s / fp8_gemm_scaled_f32s
                                                        the FP32-scale variant
  fp8hg_get_device_error(stream=None)

Scale arrays are allocated with their column count rounded up to a multiple
of four (the GEMM reads scale bytes four at a time); ``QTensor.scales()``
returns the unpadded view.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
from dataclasses import dataclass
from typing import Optional

from . import build as _build

E4M3, E5M2 = 0, 1
GRAN_ROW, GRAN_1x128, GRAN_128x128, GRAN_MX32 = 0, 1, 2, 3
FPROP, DGRAD, WGRAD = 0, 1, 2
OUT_BF16, OUT_FP32 = 0, 1

STATUS = {0: "FP8HG_OK", 1: "FP8HG_ERR_INVALID_ARG", 2: "FP8HG_ERR_ALIGNMENT",
          3: "FP8HG_ERR_SHAPE", 4: "FP8HG_ERR_UNSUPPORTED", 5: "FP8HG_ERR_CUDA",
          6: "FP8HG_ERR_TIMEOUT"}

HEADER = os.path.join(_build.INCLUDE, "fp8hg.h")


class Fp8hgError(RuntimeError):
    def __init__(self, what: str, status: int):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


class Operand(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("k", ctypes.c_int64), ("ld", ctypes.c_int64),
                ("ld_scale", ctypes.c_int64), ("fmt", ctypes.c_int32), ("gran", ctypes.c_int32)]


class GemmOpts(ctypes.Structure):
    _fields_ = [("wait_limit_ns", ctypes.c_uint64), ("inject_fault", ctypes.c_int32),
                ("tile", ctypes.c_int32)]


class WaitOpts(ctypes.Structure):
    _fields_ = [("wait_limit_ns", ctypes.c_uint64), ("inject_fault", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


def _wait_opts(wait_limit_ns: int, inject_fault: int):
    """A WaitOpts by reference, or None (library defaults) when both are 0."""
    if not wait_limit_ns and not inject_fault:
        return None
    return ctypes.byref(WaitOpts(wait_limit_ns, inject_fault, 0))


_lib = None
_lock = threading.Lock()


def declared_functions():
    """Names of the functions include/fp8hg.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)


def load_library(build_if_stale: bool = True):
    """Load libfp8hg.so (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build_if_stale and _build.is_stale():
            _build.build()
        if not os.path.exists(_build.LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {_build.LIB_PATH}")
        lib = ctypes.CDLL(_build.LIB_PATH)
        P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.fp8_quant_token.argtypes = [P, I64, I64, I64, I, I, I, P, I64, P, I64, P]
        lib.fp8_quant_token_ex.argtypes = [P, I64, I64, I64, I, I, I, P, I64, P, I64, P, P]
        lib.fp8_quant_token_dual.argtypes = [P, I64, I64, I64, I, P, I64, P, I64, I, P, I64, P,
                                             I64, P, ctypes.c_size_t, P, P]
        lib.fp8_quant_token_dual_workspace.argtypes = [I64, I64]
        lib.fp8_quant_token_dual_workspace.restype = ctypes.c_size_t
        lib.fp8_requant_t_ex.argtypes = [P, I64, I64, I64, P, I64, I, I, I, P, I64, P, I64, P, P]
        lib.fp8_gemm_scaled_f32s_ex.argtypes = [I, ctypes.POINTER(Operand),
                                                ctypes.POINTER(Operand), P, I64, I, P, P]
        lib.fp8_quant_block128.argtypes = [P, I64, I64, I64, I, P, I64, P, I64, P, I64, P, I64, P]
        lib.fp8_quant_block128_batch.argtypes = [P, I, I, P]
        lib.fp8_quant_mx32.argtypes = [P, I64, I64, I64, I, P, I64, P, I64, P, P]
        lib.fp8_quant_mx32_monitor.argtypes = [P, I64, I64, I64, I, P, I64, P, I64, P, P, P]
        lib.fp8_requant_t.argtypes = [P, I64, I64, I64, P, I64, I, I, I, P, I64, P, I64, P]
        lib.fp8_gemm_scaled_q.argtypes = [I, ctypes.POINTER(Operand), ctypes.POINTER(Operand), P,
                                          I64, P, I64, I, P]
        lib.fp8_quant_token_f32s.argtypes = [P, I64, I64, I64, I, I, P, I64, P, I64, P]
        lib.fp8_quant_block128_f32s.argtypes = [P, I64, I64, I64, I, P, I64, P, I64, P, I64, P,
                                                I64, P]
        # fp8hg_operand_f32s has the layout of fp8hg_operand (float scale pointer)
        lib.fp8_gemm_scaled_f32s.argtypes = [I, ctypes.POINTER(Operand), ctypes.POINTER(Operand),
                                             P, I64, I, P]
        lib.fp8_gemm_scaled.argtypes = [I, ctypes.POINTER(Operand), ctypes.POINTER(Operand), P,
                                        I64, I, I, P]
        lib.fp8_gemm_scaled_ex.argtypes = [I, ctypes.POINTER(Operand), ctypes.POINTER(Operand), P,
                                           I64, I, I, ctypes.POINTER(GemmOpts), P]
        lib.fp8_gemm_scaled_splitk.argtypes = [I, ctypes.POINTER(Operand), ctypes.POINTER(Operand),
                                               P, I64, I, I, I, P, ctypes.c_size_t,
                                               ctypes.POINTER(GemmOpts), P]
        lib.fp8_gemm_splitk_workspace.argtypes = [I64, I64, I64, I]
        lib.fp8_gemm_splitk_workspace.restype = ctypes.c_size_t
        lib.fp8hg_get_device_error.argtypes = [P]
        lib.fp8hg_status_str.restype = ctypes.c_char_p
        lib.fp8hg_status_str.argtypes = [I]
        for fn in ("fp8_quant_token", "fp8_quant_block128", "fp8_quant_mx32", "fp8_gemm_scaled",
                   "fp8_gemm_scaled_ex", "fp8hg_get_device_error", "fp8hg_version",
                   "fp8_quant_token_ex", "fp8_requant_t_ex", "fp8_gemm_scaled_f32s_ex",
                   "fp8_quant_token_dual", "fp8_gemm_scaled_splitk"):
            getattr(lib, fn).restype = I
        _lib = lib
        return lib


def lib():
    return _lib if _lib is not None else load_library()


def _check(rc: int, what: str):
    if rc != 0:
        raise Fp8hgError(what, rc)


def _stream(stream):
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _round4(n: int) -> int:
    return (n + 3) // 4 * 4


@dataclass
class QTensor:
    """FP8 codes [rows, k] (K-contiguous) and their scale bytes.

    ``scale`` holds the padded storage; ``ncols_scale`` its meaningful
    columns.  ``gran`` says how scale bytes map onto elements."""
    codes: "object"
    scale: "object"
    fmt: int
    gran: int
    ncols_scale: int

    def scales(self):
        return self.scale[:, :self.ncols_scale]

    def operand(self) -> Operand:
        c, s = self.codes, self.scale
        return Operand(c.data_ptr(), s.data_ptr(), c.shape[0], c.shape[1], c.stride(0),
                       s.stride(0), self.fmt, self.gran)


def _check_bf16(x):
    import torch
    if x.dtype != torch.bfloat16 or not x.is_cuda or x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D CUDA bfloat16 tensor with unit column stride")


def fp8_quant_token(x, group: int = 0, fmt: int = E4M3, transpose: bool = False,
                    out: Optional[QTensor] = None, stream=None, wait_limit_ns: int = 0,
                    inject_fault: int = 0) -> QTensor:
    """Per-token (group=0) or per-1x128 (group=128) UE8M0 quantization;
    transpose=True quantizes 128-row groups and writes [cols, rows].
    out: optional preallocated QTensor (e.g. from alloc_token).
    wait_limit_ns / inject_fault: see fp8hg_wait_opts (tests of the timeout path)."""
    _check_bf16(x)
    rows, cols = x.shape
    out = out if out is not None else alloc_token(rows, cols, group, fmt, transpose, x.device)
    rc = lib().fp8_quant_token_ex(_ptr(x), rows, cols, x.stride(0), group, 1 if transpose else 0,
                                  fmt, _ptr(out.codes), out.codes.stride(0), _ptr(out.scale),
                                  out.scale.stride(0), _wait_opts(wait_limit_ns, inject_fault),
                                  _stream(stream))
    _check(rc, "fp8_quant_token")
    return out


def dual_workspace(rows: int, cols: int, device="cuda"):
    """Scratch for fp8_quant_token_dual on [rows, cols] (a uint8 CUDA tensor)."""
    import torch
    n = int(lib().fp8_quant_token_dual_workspace(rows, cols))
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


def fp8_quant_token_dual(x, fmt: int = E4M3, fmt_t: Optional[int] = None,
                         out: Optional[QTensor] = None, out_t: Optional[QTensor] = None,
                         workspace=None, stream=None, wait_limit_ns: int = 0,
                         inject_fault: int = 0):
    """Per-token codes (as fp8_quant_token(x, 0, fmt)) and transposed 1x128
    codes along the tokens (as fp8_quant_token(x, 128, fmt_t, transpose=True))
    from one read of x.  Returns (QTensor, QTensor).  workspace: optional
    tensor from dual_workspace (allocated per call if None)."""
    _check_bf16(x)
    rows, cols = x.shape
    fmt_t = fmt if fmt_t is None else fmt_t
    out = out if out is not None else alloc_token(rows, cols, 0, fmt, False, x.device)
    out_t = out_t if out_t is not None else alloc_token(rows, cols, 128, fmt_t, True, x.device)
    ws = workspace if workspace is not None else dual_workspace(rows, cols, x.device)
    rc = lib().fp8_quant_token_dual(
        _ptr(x), rows, cols, x.stride(0), fmt, _ptr(out.codes), out.codes.stride(0),
        _ptr(out.scale), out.scale.stride(0), fmt_t, _ptr(out_t.codes), out_t.codes.stride(0),
        _ptr(out_t.scale), out_t.scale.stride(0), _ptr(ws), ws.numel() * ws.element_size(),
        _wait_opts(wait_limit_ns, inject_fault), _stream(stream))
    _check(rc, "fp8_quant_token_dual")
    return out, out_t


def fp8_quant_token_dual_noalloc(x, fmt: int = E4M3, fmt_t: Optional[int] = None,
                                 out: Optional[QTensor] = None, out_t: Optional[QTensor] = None,
                                 stream=None):
    """fp8_quant_token_dual for callers that cannot provide device scratch:
    the library's fixed scratch is used instead (at most 65536 tokens; calls
    that may overlap on the GPU must not use it concurrently)."""
    _check_bf16(x)
    rows, cols = x.shape
    fmt_t = fmt if fmt_t is None else fmt_t
    out = out if out is not None else alloc_token(rows, cols, 0, fmt, False, x.device)
    out_t = out_t if out_t is not None else alloc_token(rows, cols, 128, fmt_t, True, x.device)
    f = lib().fp8_quant_token_dual_noalloc
    P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    f.argtypes = [P, I64, I64, I64, I, P, I64, P, I64, I, P, I64, P, I64, P, P]
    f.restype = I
    rc = f(_ptr(x), rows, cols, x.stride(0), fmt, _ptr(out.codes), out.codes.stride(0),
           _ptr(out.scale), out.scale.stride(0), fmt_t, _ptr(out_t.codes), out_t.codes.stride(0),
           _ptr(out_t.scale), out_t.scale.stride(0), None, _stream(stream))
    _check(rc, "fp8_quant_token_dual_noalloc")
    return out, out_t


def fp8_quant_block128(x, fmt: int = E4M3, transposed_copy: bool = False, out=None,
                       out_t=None, stream=None):
    """Per-128x128-block UE8M0 quantization; with transposed_copy=True also
    returns the codes of x^T and the transposed scale grid.  out / out_t:
    optional preallocated QTensors (e.g. from alloc_block128)."""
    _check_bf16(x)
    rows, cols = x.shape
    if out is None or (transposed_copy and out_t is None):
        out, out_t2 = alloc_block128(rows, cols, fmt, transposed_copy, x.device)
        out_t = out_t if out_t is not None else out_t2
    qt = out_t.codes if transposed_copy else None
    st = out_t.scale if transposed_copy else None
    rc = lib().fp8_quant_block128(_ptr(x), rows, cols, x.stride(0), fmt, _ptr(out.codes),
                                  out.codes.stride(0), _ptr(out.scale), out.scale.stride(0),
                                  _ptr(qt), qt.stride(0) if qt is not None else 0,
                                  _ptr(st), st.stride(0) if st is not None else 0, _stream(stream))
    _check(rc, "fp8_quant_block128")
    if transposed_copy:
        return out, out_t
    return out


BATCH_MAX = 8   # FP8HG_BATCH_MAX


class _Block128Job(ctypes.Structure):
    """fp8hg_block128_job of the C header."""
    _fields_ = [("x", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("ld_x", ctypes.c_int64), ("q", ctypes.c_void_p), ("ld_q", ctypes.c_int64),
                ("scale", ctypes.c_void_p), ("ld_s", ctypes.c_int64), ("q_t", ctypes.c_void_p),
                ("ld_qt", ctypes.c_int64), ("scale_t", ctypes.c_void_p), ("ld_st", ctypes.c_int64)]


def fp8_quant_block128_batch(xs, fmt: int = E4M3, transposed_copy: bool = False, outs=None,
                             stream=None):
    """fp8_quant_block128 on up to BATCH_MAX tensors in one launch.  Returns a
    list with, per tensor, what fp8_quant_block128 returns.  outs: optional
    list of preallocated (QTensor, QTensor or None) pairs (alloc_block128)."""
    if len(xs) > BATCH_MAX:
        raise ValueError(f"at most {BATCH_MAX} tensors per batch")
    jobs = (_Block128Job * max(len(xs), 1))()
    res = []
    for i, x in enumerate(xs):
        _check_bf16(x)
        rows, cols = x.shape
        if outs is not None and outs[i] is not None:
            out, out_t = outs[i]
        else:
            out, out_t = alloc_block128(rows, cols, fmt, transposed_copy, x.device)
        qt = out_t.codes if transposed_copy else None
        st = out_t.scale if transposed_copy else None
        jobs[i] = _Block128Job(_ptr(x), rows, cols, x.stride(0), _ptr(out.codes),
                               out.codes.stride(0), _ptr(out.scale), out.scale.stride(0),
                               _ptr(qt), qt.stride(0) if qt is not None else 0,
                               _ptr(st), st.stride(0) if st is not None else 0)
        res.append((out, out_t) if transposed_copy else out)
    rc = lib().fp8_quant_block128_batch(ctypes.addressof(jobs), len(xs), fmt, _stream(stream))
    _check(rc, "fp8_quant_block128_batch")
    return res


def alloc_block128(rows: int, cols: int, fmt: int = E4M3, transposed_copy: bool = False,
                   device="cuda"):
    """Output buffers for fp8_quant_block128: (QTensor, QTensor or None)."""
    import torch
    q = torch.empty((rows, cols), dtype=torch.uint8, device=device)
    s = torch.empty((max(rows // 128, 1), _round4(max(cols // 128, 1))), dtype=torch.uint8,
                    device=device)
    out = QTensor(q, s, fmt, GRAN_128x128, cols // 128)
    if not transposed_copy:
        return out, None
    qt = torch.empty((cols, rows), dtype=torch.uint8, device=device)
    st = torch.empty((max(cols // 128, 1), _round4(max(rows // 128, 1))), dtype=torch.uint8,
                     device=device)
    return out, QTensor(qt, st, fmt, GRAN_128x128, rows // 128)


def alloc_token(rows: int, cols: int, group: int = 0, fmt: int = E4M3, transpose: bool = False,
                device="cuda") -> QTensor:
    """Output buffers for fp8_quant_token (shape of the result, padded scales)."""
    import torch
    if transpose:
        q = torch.empty((cols, rows), dtype=torch.uint8, device=device)
        s = torch.empty((cols, _round4(rows // 128)), dtype=torch.uint8, device=device)
        return QTensor(q, s, fmt, GRAN_1x128, rows // 128)
    q = torch.empty((rows, cols), dtype=torch.uint8, device=device)
    if group == 0:
        return QTensor(q, torch.empty((rows, 1), dtype=torch.uint8, device=device), fmt,
                       GRAN_ROW, 1)
    s = torch.empty((rows, _round4(cols // 128)), dtype=torch.uint8, device=device)
    return QTensor(q, s, fmt, GRAN_1x128, cols // 128)


def alloc_mx32(rows: int, cols: int, fmt: int = E4M3, device="cuda") -> QTensor:
    import torch
    q = torch.empty((rows, cols), dtype=torch.uint8, device=device)
    s = torch.empty((rows, _round4(cols // 32)), dtype=torch.uint8, device=device)
    return QTensor(q, s, fmt, GRAN_MX32, cols // 32)


def fp8_quant_mx32(x, fmt: int = E4M3, clamp_count=None, out=None, stream=None) -> QTensor:
    """MXFP8 quantization (32-element blocks, saturating).  clamp_count: an
    optional int64 CUDA tensor of one element that receives (+=) the number
    of clamped elements."""
    _check_bf16(x)
    rows, cols = x.shape
    out = out if out is not None else alloc_mx32(rows, cols, fmt, x.device)
    rc = lib().fp8_quant_mx32(_ptr(x), rows, cols, x.stride(0), fmt, _ptr(out.codes),
                              out.codes.stride(0), _ptr(out.scale), out.scale.stride(0),
                              _ptr(clamp_count), _stream(stream))
    _check(rc, "fp8_quant_mx32")
    return out


def fp8_requant_t(src: QTensor, fmt: int = E4M3, out: Optional[QTensor] = None,
                  stream=None, wait_limit_ns: int = 0, inject_fault: int = 0) -> QTensor:
    """Re-quantize a stored per-token or 1x128 operand [tokens, cols] into
    1x128 groups along the tokens, transposed ([cols, tokens]): the
    weight-gradient operand, from the FP8 codes instead of the BF16 source."""
    if src.gran not in (GRAN_ROW, GRAN_1x128):
        raise ValueError("source must have per-token or 1x128 scales")
    rows, cols = src.codes.shape
    out = out if out is not None else alloc_token(rows, cols, 128, fmt, True, src.codes.device)
    rc = lib().fp8_requant_t_ex(_ptr(src.codes), rows, cols, src.codes.stride(0), _ptr(src.scale),
                                src.scale.stride(0), src.gran, src.fmt, fmt, _ptr(out.codes),
                                out.codes.stride(0), _ptr(out.scale), out.scale.stride(0),
                                _wait_opts(wait_limit_ns, inject_fault), _stream(stream))
    _check(rc, "fp8_requant_t")
    return out


MX_STAT_NAMES = ("saturated", "top_code", "blocks_saturated", "blocks_collapsed")


def fp8_quant_mx32_monitor(x, fmt: int = E4M3, stats=None, row_saturated=None, out=None,
                           stream=None):
    """MXFP8 quantization that also counts the last-bin population.

    stats: int64 CUDA tensor of 4 (saturated, top_code, blocks_saturated,
    blocks_collapsed); allocated zeroed if None.  row_saturated: optional
    int32 CUDA tensor [rows] of per-row saturated counts.  Both receive +=.
    Returns (QTensor, stats)."""
    import torch
    _check_bf16(x)
    rows, cols = x.shape
    if stats is None:
        stats = torch.zeros(4, dtype=torch.int64, device=x.device)
    if stats.dtype != torch.int64 or stats.numel() != 4 or not stats.is_contiguous():
        raise ValueError("stats must be a contiguous int64 tensor of 4 elements")
    if row_saturated is not None and (row_saturated.dtype != torch.int32 or
                                      row_saturated.numel() != rows or
                                      not row_saturated.is_contiguous()):
        raise ValueError("row_saturated must be a contiguous int32 tensor of `rows` elements")
    out = out if out is not None else alloc_mx32(rows, cols, fmt, x.device)
    rc = lib().fp8_quant_mx32_monitor(_ptr(x), rows, cols, x.stride(0), fmt, _ptr(out.codes),
                                      out.codes.stride(0), _ptr(out.scale), out.scale.stride(0),
                                      _ptr(stats), _ptr(row_saturated), _stream(stream))
    _check(rc, "fp8_quant_mx32_monitor")
    return out, stats


# --- FP32-scale variant ("FP8 w. FP32 scale") -------------------------------
# QTensors of this variant hold float32 scales ([rows, 1], [rows, cols/128]
# or [rows/128, cols/128]); the GEMM takes them through fp8_gemm_scaled_f32s.

def fp8_quant_token_f32s(x, group: int = 0, fmt: int = E4M3, out: Optional[QTensor] = None,
                         stream=None) -> QTensor:
    import torch
    _check_bf16(x)
    rows, cols = x.shape
    if out is None:
        q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
        ng = 1 if group == 0 else cols // 128
        out = QTensor(q, torch.empty((rows, ng), dtype=torch.float32, device=x.device), fmt,
                      GRAN_ROW if group == 0 else GRAN_1x128, ng)
    rc = lib().fp8_quant_token_f32s(_ptr(x), rows, cols, x.stride(0), group, fmt, _ptr(out.codes),
                                    out.codes.stride(0), _ptr(out.scale), out.scale.stride(0),
                                    _stream(stream))
    _check(rc, "fp8_quant_token_f32s")
    return out


def fp8_quant_block128_f32s(x, fmt: int = E4M3, transposed_copy: bool = False, stream=None):
    import torch
    _check_bf16(x)
    rows, cols = x.shape
    dev = x.device
    out = QTensor(torch.empty((rows, cols), dtype=torch.uint8, device=dev),
                  torch.empty((rows // 128, cols // 128), dtype=torch.float32, device=dev), fmt,
                  GRAN_128x128, cols // 128)
    out_t = None
    if transposed_copy:
        out_t = QTensor(torch.empty((cols, rows), dtype=torch.uint8, device=dev),
                        torch.empty((cols // 128, rows // 128), dtype=torch.float32, device=dev),
                        fmt, GRAN_128x128, rows // 128)
    rc = lib().fp8_quant_block128_f32s(
        _ptr(x), rows, cols, x.stride(0), fmt, _ptr(out.codes), out.codes.stride(0),
        _ptr(out.scale), out.scale.stride(0), _ptr(out_t.codes) if out_t else None,
        out_t.codes.stride(0) if out_t else 0, _ptr(out_t.scale) if out_t else None,
        out_t.scale.stride(0) if out_t else 0, _stream(stream))
    _check(rc, "fp8_quant_block128_f32s")
    return (out, out_t) if transposed_copy else out


def fp8_gemm_scaled_f32s(op: int, a: QTensor, b: QTensor, out=None, out_dtype=None, stream=None,
                         wait_limit_ns: int = 0, inject_fault: int = 0):
    """C = A * B^T on FP8 operands with FP32 scales (promotion GEMM)."""
    import torch
    if out is None:
        dt = out_dtype if out_dtype is not None else torch.bfloat16
        out = torch.empty((a.codes.shape[0], b.codes.shape[0]), dtype=dt, device=a.codes.device)
    if out.dtype == torch.bfloat16:
        kind = OUT_BF16
    elif out.dtype == torch.float32:
        kind = OUT_FP32
    else:
        raise ValueError("out must be bfloat16 or float32")
    if a.scale.dtype != torch.float32 or b.scale.dtype != torch.float32:
        raise ValueError("operands must carry float32 scales")
    oa, ob = a.operand(), b.operand()
    rc = lib().fp8_gemm_scaled_f32s_ex(op, ctypes.byref(oa), ctypes.byref(ob), _ptr(out),
                                       out.stride(0), kind, _wait_opts(wait_limit_ns, inject_fault),
                                       _stream(stream))
    _check(rc, "fp8_gemm_scaled_f32s")
    return out


def fp8_gemm_scaled_q(op: int, a: QTensor, b: QTensor, fmt: int = E4M3,
                      out: Optional[QTensor] = None, stream=None) -> QTensor:
    """C = A * B^T with C quantized in the GEMM's epilogue: FP8 codes [M, N]
    with one UE8M0 scale per 128 columns of a row (a 1x128 operand)."""
    M, N = a.codes.shape[0], b.codes.shape[0]
    out = out if out is not None else alloc_token(M, N, 128, fmt, False, a.codes.device)
    oa, ob = a.operand(), b.operand()
    rc = lib().fp8_gemm_scaled_q(op, ctypes.byref(oa), ctypes.byref(ob), _ptr(out.codes),
                                 out.codes.stride(0), _ptr(out.scale), out.scale.stride(0), fmt,
                                 _stream(stream))
    _check(rc, "fp8_gemm_scaled_q")
    return out


def fp8_gemm_scaled(op: int, a: QTensor, b: QTensor, out=None, out_dtype=None,
                    accumulate: bool = False, wait_limit_ns: int = 0, inject_fault: int = 0,
                    tile: int = 0, stream=None):
    """C = A * B^T (or C += A * B^T) on block-scaled FP8 operands.  tile: 0 =
    library's choice, 1 = 128 x 256 tiles, 2 = 256 x 224 tiles (M % 256 == 0)."""
    import torch
    if out is None:
        dt = out_dtype if out_dtype is not None else torch.bfloat16
        out = torch.empty((a.codes.shape[0], b.codes.shape[0]), dtype=dt, device=a.codes.device)
    if out.dtype == torch.bfloat16:
        kind = OUT_BF16
    elif out.dtype == torch.float32:
        kind = OUT_FP32
    else:
        raise ValueError("out must be bfloat16 or float32")
    oa, ob = a.operand(), b.operand()
    if wait_limit_ns or inject_fault or tile:
        opts = GemmOpts(wait_limit_ns, inject_fault, tile)
        rc = lib().fp8_gemm_scaled_ex(op, ctypes.byref(oa), ctypes.byref(ob), _ptr(out),
                                      out.stride(0), kind, 1 if accumulate else 0,
                                      ctypes.byref(opts), _stream(stream))
    else:
        rc = lib().fp8_gemm_scaled(op, ctypes.byref(oa), ctypes.byref(ob), _ptr(out),
                                   out.stride(0), kind, 1 if accumulate else 0, _stream(stream))
    _check(rc, "fp8_gemm_scaled")
    return out


def splitk_workspace(M: int, N: int, K: int, split_k: int = 0, device="cuda"):
    """Zero-filled scratch for fp8_gemm_scaled_splitk on an [M, K] x [N, K]^T
    product with split_k parts (0 = what the library's choice needs); None
    when that choice would not split."""
    import torch
    n = int(lib().fp8_gemm_splitk_workspace(M, N, K, split_k))
    if n == 0:
        return None
    return torch.zeros(n, dtype=torch.uint8, device=device)


def fp8_gemm_scaled_splitk(op: int, a: QTensor, b: QTensor, out=None, out_dtype=None,
                           accumulate: bool = False, split_k: int = 0, workspace=None,
                           wait_limit_ns: int = 0, inject_fault: int = 0, tile: int = 0,
                           stream=None):
    """fp8_gemm_scaled with each tile's K range split over split_k CTAs (0 =
    the library's choice, given a workspace from splitk_workspace)."""
    import torch
    if out is None:
        dt = out_dtype if out_dtype is not None else torch.bfloat16
        out = torch.empty((a.codes.shape[0], b.codes.shape[0]), dtype=dt, device=a.codes.device)
    if out.dtype == torch.bfloat16:
        kind = OUT_BF16
    elif out.dtype == torch.float32:
        kind = OUT_FP32
    else:
        raise ValueError("out must be bfloat16 or float32")
    oa, ob = a.operand(), b.operand()
    opts = GemmOpts(wait_limit_ns, inject_fault, tile)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib().fp8_gemm_scaled_splitk(op, ctypes.byref(oa), ctypes.byref(ob), _ptr(out),
                                      out.stride(0), kind, 1 if accumulate else 0, split_k,
                                      _ptr(workspace), ws_bytes, ctypes.byref(opts),
                                      _stream(stream))
    _check(rc, "fp8_gemm_scaled_splitk")
    return out


def fp8hg_get_device_error(stream=None) -> int:
    """Synchronize and return (and clear) the device error status."""
    return int(lib().fp8hg_get_device_error(_stream(stream)))


def fp8hg_status_str(status: int) -> str:
    return lib().fp8hg_status_str(int(status)).decode()
