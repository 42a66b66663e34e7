"""The single-read dual quantizer (fp8_quant_token_dual) against the oracle:
per-token codes and scales as orc_quant_token(x, 0, fmt), transposed 1x128
codes and scales as orc_quant_token(x, 128, fmt_t, transpose), bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from oracle import E4M3, E5M2
import fp8_hybrid_granularity_gb300 as fp8hg
from fp8_hybrid_granularity_gb300 import workloads
from helpers import np_u8, assert_codes_equal

pytestmark = pytest.mark.gpu

TIMEOUT = 6


def _check(x_cpu, tok, tr, fmt, fmt_t, what=""):
    xb = workloads.bf16_bits(x_cpu)
    qo, so = oracle.quant_token(xb, 0, fmt)
    qto, sto = oracle.quant_token(xb, 128, fmt_t, transpose=True)
    assert_codes_equal(np_u8(tok.codes), qo, f"{what} per-token codes")
    assert_codes_equal(np_u8(tok.scales()), so, f"{what} per-token scales")
    assert_codes_equal(np_u8(tr.codes), qto, f"{what} transposed codes")
    assert_codes_equal(np_u8(tr.scales()), sto, f"{what} transposed scales")


@pytest.mark.parametrize("rows,cols", [(128, 128), (256, 384), (640, 256), (384, 1024)])
@pytest.mark.parametrize("fmt,fmt_t", [(E4M3, E4M3), (E5M2, E5M2), (E4M3, E5M2)])
def test_dual_matches_oracle(cuda_lib, rows, cols, fmt, fmt_t):
    """One tile to several stripes and tiles per stripe (the first and second
    passes interleave differently), with a zero row, a NaN and an infinity."""
    x = workloads.make_tensor("act", rows, cols, rows * 7 + cols + fmt + 3 * fmt_t, "dual")
    x[1, :] = 0.0                                      # a zero token: scale 2^-127
    x[rows - 2, cols // 2] = float("nan")              # a NaN: its token and 1x128 group
    x[rows // 2 + 3, 5] = float("inf")
    x[7, 130 % cols] = -3.0e4                          # a large outlier
    tok, tr = fp8hg.fp8_quant_token_dual(x.cuda(), fmt, fmt_t)
    assert fp8hg.fp8hg_get_device_error() == 0
    _check(x, tok, tr, fmt, fmt_t)


@pytest.mark.parametrize("rows,cols", [(8192, 1024), (2560, 2560), (256, 18944), (128, 19584)])
def test_dual_many_tiles_per_cta(cuda_lib, rows, cols):
    """More tiles than the grid has CTAs, so each CTA streams several tiles
    and casts each per token a few tiles after its first pass: 16 to 296
    tiles per stripe (18944 columns: a stripe nearly one round of the grid
    wide), and 19584 columns (306 tiles, wider than a round: the two
    quantizers run instead).  A NaN and a zero token included."""
    x = workloads.make_tensor("act", rows, cols, rows + cols, "dual-many")
    x[rows - 1, :] = 0.0
    x[rows // 3, cols - 1] = float("nan")
    tok, tr = fp8hg.fp8_quant_token_dual(x.cuda(), E4M3, E5M2)
    assert fp8hg.fp8hg_get_device_error() == 0
    _check(x, tok, tr, E4M3, E5M2, f"{rows}x{cols}")


def test_dual_equals_the_two_quantizers(cuda_lib):
    """[4096, 3584] (the 7B hidden size): the same bytes as the per-token
    quantizer and the transposed 1x128 quantizer, called separately."""
    x = workloads.make_tensor("act", 4096, 3584, 11, "dual-eq", device="cuda")
    tok, tr = fp8hg.fp8_quant_token_dual(x, E4M3)
    a = fp8hg.fp8_quant_token(x, 0, E4M3)
    b = fp8hg.fp8_quant_token(x, 128, E4M3, transpose=True)
    assert fp8hg.fp8hg_get_device_error() == 0
    assert torch.equal(tok.codes, a.codes) and torch.equal(tok.scales(), a.scales())
    assert torch.equal(tr.codes, b.codes) and torch.equal(tr.scales(), b.scales())
    rows = np.array([0, 1, 2047, 4095])
    ri = torch.from_numpy(rows).cuda()
    qo, so = oracle.quant_token(workloads.bf16_bits(x[ri].cpu()), 0, E4M3)
    assert_codes_equal(np_u8(tok.codes[ri]), qo, "sampled rows")
    assert_codes_equal(np_u8(tok.scales()[ri]), so, "sampled row scales")


def test_dual_workspace_reused(cuda_lib):
    """Two calls with one workspace on different tensors: the second call's
    maxima start from zero (the call clears the workspace)."""
    ws = fp8hg.dual_workspace(512, 512)
    big = workloads.make_tensor("act", 512, 512, 12, "dual-ws1") * 1000
    small = workloads.make_tensor("grad", 512, 512, 13, "dual-ws2")
    fp8hg.fp8_quant_token_dual(big.cuda(), E4M3, workspace=ws)
    tok, tr = fp8hg.fp8_quant_token_dual(small.cuda(), E5M2, workspace=ws)
    assert fp8hg.fp8hg_get_device_error() == 0
    _check(small, tok, tr, E5M2, E5M2, "second call")


def test_dual_full_size_7b(cuda_lib):
    """H [16384, 18944] as the step quantizes it: sampled tokens (all 18944
    columns) and sampled columns (all 16384 tokens) against the oracle."""
    M, C = 16384, 18944
    h = workloads.make_tensor("act", M, C, 2, "H", device="cuda")
    tok, tr = fp8hg.fp8_quant_token_dual(h, E4M3)
    assert fp8hg.fp8hg_get_device_error() == 0
    rng = np.random.default_rng(14)
    rows = np.concatenate([[0, M - 1], rng.choice(np.arange(1, M - 1), 30, replace=False)])
    ri = torch.from_numpy(rows).cuda()
    qo, so = oracle.quant_token(workloads.bf16_bits(h[ri].cpu()), 0, E4M3)
    assert_codes_equal(np_u8(tok.codes[ri]), qo, "sampled tokens")
    assert_codes_equal(np_u8(tok.scales()[ri]), so, "sampled token scales")
    cols = np.sort(np.concatenate([[0, C - 1], rng.choice(np.arange(1, C - 1), 24, replace=False)]))
    ci = torch.from_numpy(cols).cuda()
    qto, sto = oracle.quant_token(workloads.bf16_bits(h[:, ci].cpu()), 128, E4M3, transpose=True)
    assert_codes_equal(np_u8(tr.codes[ci]), qto, "sampled columns")
    assert_codes_equal(np_u8(tr.scales()[ci]), sto, "sampled column scales")


def test_dual_timeout_path(cuda_lib):
    """A withheld tile completion: the second pass of its stripe waits out the
    limit, the status reads TIMEOUT once, and the next call is exact."""
    x = workloads.make_tensor("act", 512, 512, 15, "dual-timeout")
    xd = x.cuda()
    fp8hg.fp8_quant_token_dual(xd, E4M3, wait_limit_ns=20_000_000, inject_fault=1)
    assert fp8hg.fp8hg_get_device_error() == TIMEOUT
    tok, tr = fp8hg.fp8_quant_token_dual(xd, E4M3)
    assert fp8hg.fp8hg_get_device_error() == 0
    _check(x, tok, tr, E4M3, E4M3, "after timeout")


def test_dual_canary(cuda_lib):
    """Strided outputs inside 0xAB-filled buffers: nothing written outside."""
    from test_gpu_canary import canvas, assert_canary
    rows, cols = 384, 256
    x = workloads.make_tensor("act", rows, cols, 16, "dual-canary")
    qb, q = canvas(rows, cols, cols + 48)
    sb, s = canvas(rows, 1, 7)
    qtb, qt = canvas(cols, rows, rows + 32)
    stb, st = canvas(cols, rows // 128, rows // 128 + 5)
    tok, tr = fp8hg.fp8_quant_token_dual(
        x.cuda(), E4M3, out=fp8hg.QTensor(q, s, E4M3, fp8hg.GRAN_ROW, 1),
        out_t=fp8hg.QTensor(qt, st, E4M3, fp8hg.GRAN_1x128, rows // 128))
    assert fp8hg.fp8hg_get_device_error() == 0
    _check(x, tok, tr, E4M3, E4M3, "canary")
    for buf, r, c, what in ((qb, rows, cols, "codes"), (sb, rows, 1, "scales"),
                            (qtb, cols, rows, "codes^T"), (stb, cols, rows // 128, "scales^T")):
        assert_canary(buf, r, c, what)


def test_dual_strided_input(cuda_lib):
    """x a view into a wider buffer (ld_x = cols + 64): the copies follow the
    row stride."""
    rows, cols = 384, 512
    full = workloads.make_tensor("act", rows, cols + 64, 17, "dual-strided")
    x = full.cuda()[:, :cols]
    assert x.stride(0) == cols + 64
    tok, tr = fp8hg.fp8_quant_token_dual(x, E4M3, E5M2)
    assert fp8hg.fp8hg_get_device_error() == 0
    _check(full[:, :cols].contiguous(), tok, tr, E4M3, E5M2, "strided")
