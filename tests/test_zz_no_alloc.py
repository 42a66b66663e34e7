"""The entry point that allocates nothing (fp8_quant_token_dual_noalloc).

Some callers cannot give the library device memory: code running under a
framework whose memory pool owns the device, code inside an allocator's own
callbacks, or hot paths that must not pay for the synchronization a
cudaMalloc can cause.  For them the single-read dual quantizer has a variant
whose scratch is a fixed array inside the library.  These tests call it
through the C ABI (ctypes on the library symbol) and require the same bytes
as the regular entry point, fp8_quant_token_dual, on two calls in a row: the
second call must not see the first call's maxima in the shared scratch.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.  It also passes alone, in a
fresh process (the fixture loads the library itself).
"""
import ctypes

import pytest
import torch

import fp8_hybrid_granularity_gb300 as fp8hg
from fp8_hybrid_granularity_gb300 import workloads, E4M3, E5M2

pytestmark = pytest.mark.gpu

P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
FP8HG_ERR_SHAPE = 3


def _noalloc(lib):
    f = lib.fp8_quant_token_dual_noalloc
    f.argtypes = [P, I64, I64, I64, I, P, I64, P, I64, I, P, I64, P, I64, P, P]
    f.restype = I
    return f


def _call(f, x, fmt, fmt_t):
    rows, cols = x.shape
    tok = fp8hg.alloc_token(rows, cols, 0, fmt, False, x.device)
    tr = fp8hg.alloc_token(rows, cols, 128, fmt_t, True, x.device)
    stream = torch.cuda.current_stream().cuda_stream
    rc = f(x.data_ptr(), rows, cols, x.stride(0), fmt, tok.codes.data_ptr(), tok.codes.stride(0),
           tok.scale.data_ptr(), tok.scale.stride(0), fmt_t, tr.codes.data_ptr(),
           tr.codes.stride(0), tr.scale.data_ptr(), tr.scale.stride(0), None, stream)
    return rc, tok, tr


def test_noalloc_matches_the_workspace_entry_point(cuda_lib):
    f = _noalloc(cuda_lib.lib())
    # two calls in a row: large magnitudes first, then small ones (stale
    # maxima left in the shared scratch would inflate the second call's scales)
    inputs = [(workloads.make_tensor("act", 1024, 640, 80, "noalloc-1") * 500, E4M3, E4M3),
              (workloads.make_tensor("grad", 768, 512, 81, "noalloc-2"), E5M2, E4M3)]
    for x_cpu, fmt, fmt_t in inputs:
        x = x_cpu.cuda()
        rc, tok, tr = _call(f, x, fmt, fmt_t)
        assert rc == 0
        assert fp8hg.fp8hg_get_device_error() == 0
        ref_tok, ref_tr = fp8hg.fp8_quant_token_dual(x, fmt, fmt_t)
        assert fp8hg.fp8hg_get_device_error() == 0
        assert torch.equal(tok.codes, ref_tok.codes)
        assert torch.equal(tok.scales(), ref_tok.scales())
        assert torch.equal(tr.codes, ref_tr.codes)
        assert torch.equal(tr.scales(), ref_tr.scales())


def test_noalloc_rejects_more_rows_than_its_scratch(cuda_lib):
    """65536 tokens at most; the check comes before anything is launched."""
    f = _noalloc(cuda_lib.lib())
    rows, cols = 65536 + 128, 128
    fake = 0x10000
    rc = f(fake, rows, cols, cols, E4M3, fake, cols, fake, 1, E4M3, fake, rows, fake, rows // 128,
           None, None)
    assert rc == FP8HG_ERR_SHAPE
