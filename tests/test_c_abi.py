"""The boundary is a C ABI: include/fp8hg.h compiles as strict C99 and a plain
C program links libfp8hg.so and calls it.  Only calls that fail validation
(or need no device) are made, so no GPU is needed."""
import os
import shutil
import subprocess

import pytest

import fp8_hybrid_granularity_gb300 as fp8hg
from fp8_hybrid_granularity_gb300 import build as fp8_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdint.h>
#include <stdio.h>
#include <string.h>
#include "fp8hg.h"

int main(void) {
    uint16_t *x = (uint16_t *)(uintptr_t)0x10000;   /* never dereferenced */
    uint8_t *q = (uint8_t *)(uintptr_t)0x10000;
    fp8hg_operand a = {q, q, 256, 256, 256, 4, FP8HG_E4M3, FP8HG_GRAN_1x128};
    fp8hg_operand b = a;
    fp8hg_gemm_opts opts = {0, 0, 7};
    if (fp8hg_version() != (1 << 16)) return 1;
    if (strcmp(fp8hg_status_str(FP8HG_ERR_TIMEOUT), "FP8HG_ERR_TIMEOUT") != 0) return 2;
    if (fp8_quant_token(NULL, 4, 128, 128, 0, 0, FP8HG_E4M3, q, 128, q, 1, NULL) !=
        FP8HG_ERR_INVALID_ARG) return 3;
    if (fp8_quant_token(x, 4, 100, 104, 0, 0, FP8HG_E4M3, q, 112, q, 1, NULL) != FP8HG_ERR_SHAPE)
        return 4;
    if (fp8_quant_block128(x, 128, 128, 128, FP8HG_E4M3, q + 4, 128, q, 1, NULL, 0, NULL, 0,
                           NULL) != FP8HG_ERR_ALIGNMENT) return 5;
    /* the forward GEMM needs 128x128-block weights */
    if (fp8_gemm_scaled(FP8HG_FPROP, &a, &b, q, 256, FP8HG_OUT_BF16, 0, NULL) !=
        FP8HG_ERR_UNSUPPORTED) return 6;
    if (fp8_gemm_scaled_ex(FP8HG_WGRAD, &a, &b, q, 256, FP8HG_OUT_FP32, 0, &opts, NULL) !=
        FP8HG_ERR_INVALID_ARG) return 7;
    /* empty tensors: nothing is read or written */
    if (fp8_quant_mx32(x, 0, 64, 64, FP8HG_E4M3, q, 64, q, 2, NULL, NULL) != FP8HG_OK) return 8;
    puts("ok");
    return 0;
}
"""


def test_header_is_c99_and_library_links_from_c(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fp8hg.load_library()                      # builds libfp8hg.so if it is missing
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(fp8_build.LIB_PATH)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                        "-L", libdir, "-lfp8hg", "-Wl,-rpath," + libdir],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
