"""The quantized-epilogue GEMM's checker, pinned on the CPU: it accepts the
oracle's own 1x128 quantization of C and rejects a code one step off, a
wrong scale byte and a code from the wrong side of a rounding tie."""
import numpy as np
import pytest

import oracle
from oracle import E4M3, E5M2
from test_gpu_gemm_q import check_quantized_output


def _quantize_rows(c, fmt):
    """1x128 groups along each row: round-up UE8M0 scale of the group's amax,
    codes the RNE encoding of c / 2^e (the oracle's scalar routines)."""
    r, n = c.shape
    codes = np.zeros((r, n), np.uint8)
    scales = np.zeros((r, n // 128), np.uint8)
    for i in range(r):
        for g in range(n // 128):
            cs = slice(128 * g, 128 * g + 128)
            e = oracle.ue8m0_exp(float(np.abs(c[i, cs]).max()), fmt)
            scales[i, g] = e + 127
            codes[i, cs] = [oracle.fp8_encode(float(y) * 2.0 ** -e, fmt) for y in c[i, cs]]
    return codes, scales


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_checker_pins(fmt):
    rng = np.random.default_rng(11)
    c = rng.normal(size=(2, 256)) * 5.0
    s_abs = np.abs(c)                      # tolerance ~0.4 % of |C|: far below an FP8 step
    codes, scales = _quantize_rows(c, fmt)
    check_quantized_output(codes, scales, c, s_abs, fmt, "oracle")

    # a code one step away from the RNE one (same sign, larger magnitude), at
    # an element whose tolerance interval does not straddle a rounding
    # midpoint (there both neighbours are the RNE code of a value within
    # tolerance, and both are accepted)
    e0 = int(scales[0, 0]) - 127
    tol = oracle.gemm_tolerance(c, s_abs)
    dec = oracle.decode_table(fmt)
    unique = [j for j in range(128)
              if oracle.fp8_encode((c[0, j] - tol[0, j]) * 2.0 ** -e0, fmt)
              == oracle.fp8_encode((c[0, j] + tol[0, j]) * 2.0 ** -e0, fmt)
              and dec[codes[0, j] + 1] < np.inf]
    j = unique[0]
    bad = codes.copy()
    bad[0, j] += 1
    with pytest.raises(AssertionError):
        check_quantized_output(bad, scales, c, s_abs, fmt, "off by one")

    # a scale byte one binade off (codes re-encoded under it)
    e = int(scales[1, 1]) - 127 + 2
    bad_s = scales.copy()
    bad_s[1, 1] = e + 127
    bad_c = codes.copy()
    bad_c[1, 128:] = [oracle.fp8_encode(float(y) * 2.0 ** -e, fmt) for y in c[1, 128:]]
    with pytest.raises(AssertionError):
        check_quantized_output(bad_c, bad_s, c, s_abs, fmt, "scale")
