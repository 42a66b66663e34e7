"""Shared helpers for the GPU parity tests: move oracle results to the GPU
and compare GPU results with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import fp8_hybrid_granularity_gb300 as fp8hg
from fp8_hybrid_granularity_gb300 import workloads

GRAN_NAMES = {0: "row", 1: "1x128", 2: "128x128", 3: "mx32"}


def bits_to_cuda(bits: np.ndarray) -> torch.Tensor:
    return workloads.from_bits(bits).cuda()


def np_u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().astype(np.uint8)


def oracle_quant(bits, gran, fmt, transpose=False):
    """Oracle codes and scales for one operand (numpy uint8)."""
    if gran == oracle.GRAN_ROW:
        return oracle.quant_token(bits, 0, fmt)
    if gran == oracle.GRAN_1x128:
        return oracle.quant_token(bits, 128, fmt, transpose=transpose)
    if gran == oracle.GRAN_128x128:
        q, s, qt, st = oracle.quant_block128(bits, fmt, transposed_copy=transpose)
        return (qt, st) if transpose else (q, s)
    q, s, _ = oracle.quant_mx32(bits, fmt)
    return q, s


def to_qtensor(q: np.ndarray, s: np.ndarray, fmt: int, gran: int) -> fp8hg.QTensor:
    """Upload oracle codes / scales as a GEMM operand (scale columns padded to 4)."""
    ncs = s.shape[1]
    pad = ncs if gran == oracle.GRAN_ROW else (ncs + 3) // 4 * 4
    sp = np.zeros((s.shape[0], pad), np.uint8)
    sp[:, :ncs] = s
    return fp8hg.QTensor(torch.from_numpy(np.ascontiguousarray(q)).cuda(),
                         torch.from_numpy(sp).cuda(), fmt, gran, ncs)


def assert_codes_equal(gpu: np.ndarray, ref: np.ndarray, what: str):
    if not np.array_equal(gpu, ref):
        bad = np.argwhere(gpu != ref)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} mismatches, first at {i}: "
                             f"gpu {gpu[i]:#04x} oracle {ref[i]:#04x}")


def check_gemm(c_gpu: np.ndarray, c_ref: np.ndarray, s_abs: np.ndarray, what: str):
    """|C_gpu - C_ref| <= 4e-3 * sum_k |a*b| + one BF16 ulp of |C_ref|."""
    tol = oracle.gemm_tolerance(c_ref, s_abs)
    err = np.abs(c_gpu.astype(np.float64) - c_ref)
    bad = ~(err <= tol)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first {i}: "
                             f"gpu {c_gpu[i]!r} ref {c_ref[i]!r} tol {tol[i]!r}")
    return float((err / np.maximum(s_abs, 1e-300)).max())
