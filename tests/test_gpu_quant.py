"""GPU parity of the quantizer kernels against the CPU oracle: codes and scale
bytes must match bit for bit.  Small shapes span several tiles / groups and a
ragged tail (rows not a multiple of any launch width, columns that leave idle
threads in the per-row kernel); special values cover zeros, signed zeros,
subnormals, the clamp ends of the exponent range, NaN and infinity."""
import numpy as np
import pytest
import torch

import oracle
from oracle import E4M3, E5M2
import fp8_hybrid_granularity_gb300 as fp8hg
from fp8_hybrid_granularity_gb300 import workloads
from helpers import bits_to_cuda, np_u8, assert_codes_equal

pytestmark = pytest.mark.gpu

FMTS = [E4M3, E5M2]


def _bits(kind, rows, cols, seed):
    return workloads.bf16_bits(workloads.make_tensor(kind, rows, cols, seed, "gpu-quant"))


def _special(rows, cols, seed):
    """Random activations with special values planted in some groups."""
    x = _bits("act", rows, cols, seed).copy()
    rng = np.random.default_rng(seed)
    x[0, :] = 0                                             # all-zero row / groups
    if rows > 1:
        x[1, :] = 0x8000                                    # all -0
    if rows > 2:
        x[2, :] = rng.integers(1, 0x80, cols) | (rng.integers(0, 2, cols) << 15)  # subnormals
    if rows > 3:
        x[3, :] = 0x7F7F                                    # largest finite BF16
        x[3, ::3] = 0xFF7F
    if rows > 5:
        x[5, 7] = 0x7FC0                                    # NaN
        x[5, cols - 1] = 0xFF80                             # -inf
    if rows > 6:
        x[6, :] = 0x0001                                    # smallest subnormal
        x[6, 1] = 0x3F80                                    # ... and one 1.0
    return x


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("rows,cols", [(1, 128), (37, 512), (300, 1536), (5, 8960), (3, 18944),
                                       (2, 131072 + 128)])
def test_quant_token_row(cuda_lib, fmt, rows, cols):
    x = _special(rows, cols, rows + cols)
    qg = fp8hg.fp8_quant_token(bits_to_cuda(x), 0, fmt)
    q, s = oracle.quant_token(x, 0, fmt)
    assert_codes_equal(np_u8(qg.scales()), s, "scale")
    assert_codes_equal(np_u8(qg.codes), q, "codes")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("rows,cols", [(1, 128), (300, 384), (1000, 1536), (7, 8960)])
def test_quant_token_1x128(cuda_lib, fmt, rows, cols):
    x = _special(rows, cols, 3 * rows + cols)
    qg = fp8hg.fp8_quant_token(bits_to_cuda(x), 128, fmt)
    q, s = oracle.quant_token(x, 128, fmt)
    assert_codes_equal(np_u8(qg.scales()), s, "scale")
    assert_codes_equal(np_u8(qg.codes), q, "codes")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("rows,cols", [(128, 64), (384, 192), (256, 3584 // 4)])
def test_quant_token_transposed(cuda_lib, fmt, rows, cols):
    x = _special(rows, cols, rows + 7 * cols)
    qg = fp8hg.fp8_quant_token(bits_to_cuda(x), 128, fmt, transpose=True)
    q, s = oracle.quant_token(x, 128, fmt, transpose=True)
    assert_codes_equal(np_u8(qg.scales()), s, "scale")
    assert_codes_equal(np_u8(qg.codes), q, "codes")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("rows,cols", [(128, 128), (384, 640), (256, 1536)])
@pytest.mark.parametrize("trans", [False, True])
def test_quant_block128(cuda_lib, fmt, rows, cols, trans):
    x = _bits("weight", rows, cols, rows * cols + fmt).copy()
    if rows > 130:
        x[130, 5] = 0x7FC0                                  # one NaN block
    x[3, 200 % cols] = 0x0000
    res = fp8hg.fp8_quant_block128(bits_to_cuda(x), fmt, transposed_copy=trans)
    q, s, qt, st = oracle.quant_block128(x, fmt, transposed_copy=trans)
    g = res[0] if trans else res
    assert_codes_equal(np_u8(g.scales()), s, "scale")
    assert_codes_equal(np_u8(g.codes), q, "codes")
    if trans:
        assert_codes_equal(np_u8(res[1].scales()), st, "scale_t")
        assert_codes_equal(np_u8(res[1].codes), qt, "codes_t")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("trans", [False, True])
def test_quant_block128_batch(cuda_lib, fmt, trans):
    """Several tensors in one launch (shapes of one, a few and many blocks, one
    of them a strided column slice, one with a NaN block, an empty one): each
    tensor's codes, scales and transposed copy equal the oracle's for that
    tensor alone."""
    shapes = [(384, 640), (128, 128), (256, 1536), (128, 256), (0, 256), (1280, 384)]
    xs_bits = [_bits("weight", r, c, 1000 + i + fmt) if r else np.zeros((0, c), np.uint16)
               for i, (r, c) in enumerate(shapes)]
    xs_bits[0] = xs_bits[0].copy()
    xs_bits[0][130, 5] = 0x7FC0                              # one NaN block
    xs = [bits_to_cuda(b) if b.shape[0] else torch.empty(b.shape, dtype=torch.bfloat16, device="cuda")
          for b in xs_bits]
    wide = _bits("weight", 128, 512, 4242 + fmt)             # strided: the middle 256 columns
    xs.append(bits_to_cuda(wide)[:, 128:384])
    xs_bits.append(np.ascontiguousarray(wide[:, 128:384]))
    res = fp8hg.fp8_quant_block128_batch(xs, fmt, transposed_copy=trans)
    assert fp8hg.fp8hg_get_device_error() == 0
    for i, (b, r) in enumerate(zip(xs_bits, res)):
        if b.shape[0] == 0:
            continue
        q, s, qt, st = oracle.quant_block128(b, fmt, transposed_copy=trans)
        g = r[0] if trans else r
        assert_codes_equal(np_u8(g.scales()), s, f"job {i} scale")
        assert_codes_equal(np_u8(g.codes), q, f"job {i} codes")
        if trans:
            assert_codes_equal(np_u8(r[1].scales()), st, f"job {i} scale_t")
            assert_codes_equal(np_u8(r[1].codes), qt, f"job {i} codes_t")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("kind,rows,cols", [("mx_ln", 64, 4096), ("mx_ln_clamp", 64, 4096),
                                            ("act", 33, 96), ("act", 1, 32),
                                            # rows longer than 8 KB: the multi-row kernel
                                            ("mx_ln_clamp", 16, 4608), ("act", 5, 8224)])
def test_quant_mx32(cuda_lib, fmt, kind, rows, cols):
    x = _bits(kind, rows, cols, rows + cols + fmt).copy()
    if rows > 5:
        x[5, 3] = 0x7FC0
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
    qg = fp8hg.fp8_quant_mx32(bits_to_cuda(x), fmt, clamp_count=cnt)
    q, s, clamped = oracle.quant_mx32(x, fmt)
    assert_codes_equal(np_u8(qg.scales()), s, "scale")
    assert_codes_equal(np_u8(qg.codes), q, "codes")
    assert int(cnt.item()) == clamped


def test_empty_inputs(cuda_lib):
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    qg = fp8hg.fp8_quant_token(x, 128, E4M3)
    assert qg.codes.shape == (0, 256)
    qm = fp8hg.fp8_quant_mx32(x, E4M3)
    assert qm.codes.shape == (0, 256)
    torch.cuda.synchronize()


def test_strided_input(cuda_lib):
    """Row stride larger than the row (a column slice of a wider tensor)."""
    full = _bits("act", 64, 1024, 77)
    xg = bits_to_cuda(full)[:, 256:768]
    qg = fp8hg.fp8_quant_token(xg, 128, E4M3)
    q, s = oracle.quant_token(np.ascontiguousarray(full[:, 256:768]), 128, E4M3)
    assert_codes_equal(np_u8(qg.codes), q, "codes")
    assert_codes_equal(np_u8(qg.scales()), s, "scale")
