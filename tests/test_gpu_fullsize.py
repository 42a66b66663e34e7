"""Parity at the full 7B step sizes, in the launch configuration bench.py
times (same entry points, same shapes, inputs drawn on the GPU by the seeded
generators).  Every output is produced by the GPU over the whole tensor; the
oracle recomputes sampled rows, columns, blocks and output elements, each of
which depends only on the slice of input it is given:

  per-token codes    -> sampled rows of the input
  1x128 transposed   -> sampled columns of the input (all 16384 tokens)
  128x128 blocks     -> sampled 128x128 blocks (and their transposed copies)
  GEMM outputs       -> sampled (i, j), from the oracle's own quantization of
                        row i of A's source and the block / column slice of B
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import E4M3, E5M2, GRAN_ROW, GRAN_1x128, GRAN_128x128
import fp8_hybrid_granularity_gb300 as fp8hg
from fp8_hybrid_granularity_gb300 import workloads
from helpers import np_u8, assert_codes_equal, check_gemm

pytestmark = pytest.mark.gpu

M, HID, MLP = 16384, 3584, 18944


@pytest.fixture(scope="module")
def data(cuda_lib):
    dev = torch.device("cuda", 0)
    mk = lambda kind, r, c, n: workloads.make_tensor(kind, r, c, 2, n, device=dev)
    d = {"H": mk("act", M, MLP, "H"), "X": mk("act", M, HID, "X"),
         "W_down": mk("weight", HID, MLP, "W_down"), "dY_gate": mk("grad", M, MLP, "dY_gate"),
         "dY_down": mk("grad", M, HID, "dY_down"), "W_gate": mk("weight", MLP, HID, "W_gate"),
         "W_up": mk("weight", MLP, HID, "W_up"), "dY_up": mk("grad", M, MLP, "dY_up")}
    yield d
    del d
    torch.cuda.empty_cache()


def _bits(t):
    return workloads.bf16_bits(t.detach().cpu())


def test_token_quant_full_size(data):
    h = data["H"]
    q = fp8hg.fp8_quant_token(h, 0, E4M3)
    rows = np.random.default_rng(0).choice(M, 48, replace=False)
    rows = np.concatenate([rows, [0, M - 1]])
    hb = _bits(h[torch.from_numpy(rows).cuda()])
    qo, so = oracle.quant_token(hb, 0, E4M3)
    assert_codes_equal(np_u8(q.codes[torch.from_numpy(rows).cuda()]), qo, "codes")
    assert_codes_equal(np_u8(q.scales()[torch.from_numpy(rows).cuda()]), so, "scales")


def test_transposed_quant_full_size(data):
    dy = data["dY_gate"]
    q = fp8hg.fp8_quant_token(dy, 128, E5M2, transpose=True)
    cols = np.sort(np.random.default_rng(1).choice(MLP, 40, replace=False))
    cols = np.concatenate([cols, [MLP - 1]])
    idx = torch.from_numpy(cols).cuda()
    xb = _bits(dy[:, idx])                       # [16384, ncols]
    qo, so = oracle.quant_token(xb, 128, E5M2, transpose=True)
    assert_codes_equal(np_u8(q.codes[idx]), qo, "codes")
    assert_codes_equal(np_u8(q.scales()[idx]), so, "scales")


def test_block128_full_size(data):
    w = data["W_down"]
    q, qt = fp8hg.fp8_quant_block128(w, E4M3, transposed_copy=True)
    rng = np.random.default_rng(2)
    blocks = [(0, 0), (HID // 128 - 1, MLP // 128 - 1)] + \
        [(int(rng.integers(HID // 128)), int(rng.integers(MLP // 128))) for _ in range(4)]
    for rb, cb in blocks:
        r0, c0 = 128 * rb, 128 * cb
        xb = _bits(w[r0:r0 + 128, c0:c0 + 128])
        qo, so, qto, sto = oracle.quant_block128(xb, E4M3, transposed_copy=True)
        assert_codes_equal(np_u8(q.codes[r0:r0 + 128, c0:c0 + 128]), qo, f"block {rb},{cb}")
        assert int(q.scales()[rb, cb]) == int(so[0, 0])
        assert_codes_equal(np_u8(qt.codes[c0:c0 + 128, r0:r0 + 128]), qto, f"block^T {rb},{cb}")
        assert int(qt.scales()[cb, rb]) == int(sto[0, 0])


# tile 0: the library's choice (the 256 x 224 kernel at these shapes, as the
# step runs); tile 3: the CTA-pair kernel (256 x 448 tiles, opt-in)
@pytest.mark.parametrize("tile", [0, 3])
def test_fprop_down_gemm_full_size(data, tile):
    """Y = H W_down^T, M=16384, K=18944, N=3584; 256 sampled outputs."""
    h, w = data["H"], data["W_down"]
    y = fp8hg.fp8_gemm_scaled(fp8hg.FPROP, fp8hg.fp8_quant_token(h, 0, E4M3),
                              fp8hg.fp8_quant_block128(w, E4M3), tile=tile)
    assert fp8hg.fp8hg_get_device_error() == 0
    rng = np.random.default_rng(3)
    ii = rng.choice(M, 16, replace=False)
    jb = rng.choice(HID // 128, 4, replace=False)      # B row blocks
    qa, sa = oracle.quant_token(_bits(h[torch.from_numpy(ii).cuda()]), 0, E4M3)
    c_gpu, c_ref, s_abs = [], [], []
    for b in jb:
        qb, sb, _, _ = oracle.quant_block128(_bits(w[128 * b:128 * b + 128]), E4M3)
        jj = rng.choice(128, 4, replace=False)
        I, J = np.meshgrid(np.arange(len(ii)), jj, indexing="ij")
        c, s = oracle.gemm_ref_pairs(qa, sa, GRAN_ROW, E4M3, qb, sb, GRAN_128x128, E4M3,
                                     I.ravel(), J.ravel())
        c_ref.append(c)
        s_abs.append(s)
        g = y[torch.from_numpy(ii).cuda()][:, torch.from_numpy(128 * b + jj).cuda()]
        c_gpu.append(g.float().cpu().numpy().ravel())
    check_gemm(np.concatenate(c_gpu), np.concatenate(c_ref), np.concatenate(s_abs), "fprop down")


def test_wgrad_gemm_full_size(data):
    """dW_gate = dY_gate^T X: contraction over 16384 tokens, FP32 out."""
    dy, x = data["dY_gate"], data["X"]
    a = fp8hg.fp8_quant_token(dy, 128, E5M2, transpose=True)
    b = fp8hg.fp8_quant_token(x, 128, E4M3, transpose=True)
    dw = fp8hg.fp8_gemm_scaled(fp8hg.WGRAD, a, b, out_dtype=torch.float32)
    assert fp8hg.fp8hg_get_device_error() == 0
    rng = np.random.default_rng(4)
    ii = np.sort(rng.choice(MLP, 12, replace=False))
    jj = np.sort(rng.choice(HID, 12, replace=False))
    qa, sa = oracle.quant_token(_bits(dy[:, torch.from_numpy(ii).cuda()]), 128, E5M2, transpose=True)
    qb, sb = oracle.quant_token(_bits(x[:, torch.from_numpy(jj).cuda()]), 128, E4M3, transpose=True)
    I, J = np.meshgrid(np.arange(len(ii)), np.arange(len(jj)), indexing="ij")
    c_ref, s_abs = oracle.gemm_ref_pairs(qa, sa, GRAN_1x128, E5M2, qb, sb, GRAN_1x128, E4M3,
                                         I.ravel(), J.ravel())
    g = dw[torch.from_numpy(ii).cuda()][:, torch.from_numpy(jj).cuda()].cpu().numpy().ravel()
    check_gemm(g, c_ref, s_abs, "wgrad")


def _dgrad_ref(dy, w, ii, b, jj, fmt_dy):
    """Oracle C_ref, S for dX[ii, 128 b + jj] of dX = dY W: A = dY rows ii
    quantized per token, B rows = columns 128b..128b+127 of W, i.e. the
    transposed copy of W's 128x128 blocks in that block column."""
    qa, sa = oracle.quant_token(_bits(dy[torch.from_numpy(ii).cuda()]), 0, fmt_dy)
    _, _, qbt, sbt = oracle.quant_block128(_bits(w[:, 128 * b:128 * b + 128]), E4M3,
                                           transposed_copy=True)
    I, J = np.meshgrid(np.arange(len(ii)), jj, indexing="ij")
    return oracle.gemm_ref_pairs(qa, sa, GRAN_ROW, fmt_dy, qbt, sbt, GRAN_128x128, E4M3,
                                 I.ravel(), J.ravel())


@pytest.mark.parametrize("tile", [0, 3])
def test_dgrad_down_gemm_full_size(data, tile):
    """dH = dY_down W_down as the step runs it: A = dY_down [16384, 3584] per
    token E5M2, B = W_down^T [18944, 3584] (the transposed block copy);
    contraction 3584, N = 18944, BF16 out; 192 sampled outputs, including the
    last 128-column block (inside the ragged last n-tile of both tile shapes:
    18944 = 84 x 224 + 128 = 42 x 448 + 128)."""
    dy, w = data["dY_down"], data["W_down"]
    a = fp8hg.fp8_quant_token(dy, 0, E5M2)
    _, bt = fp8hg.fp8_quant_block128(w, E4M3, transposed_copy=True)
    dh = fp8hg.fp8_gemm_scaled(fp8hg.DGRAD, a, bt, tile=tile)
    assert dh.shape == (M, MLP)
    assert fp8hg.fp8hg_get_device_error() == 0
    rng = np.random.default_rng(5)
    ii = np.concatenate([[0, M - 1], rng.choice(np.arange(1, M - 1), 10, replace=False)])
    c_gpu, c_ref, s_abs = [], [], []
    for b in [0, MLP // 128 - 1] + list(rng.choice(np.arange(1, MLP // 128 - 1), 2, replace=False)):
        jj = np.concatenate([[0, 127], rng.choice(np.arange(1, 127), 2, replace=False)])
        c, s = _dgrad_ref(dy, w, ii, int(b), jj, E5M2)
        c_ref.append(c)
        s_abs.append(s)
        g = dh[torch.from_numpy(ii).cuda()][:, torch.from_numpy(128 * int(b) + jj).cuda()]
        c_gpu.append(g.float().cpu().numpy().ravel())
    check_gemm(np.concatenate(c_gpu), np.concatenate(c_ref), np.concatenate(s_abs), "dgrad down")


def test_dgrad_accumulate_full_size(data):
    """dX = dY_gate W_gate + dY_up W_up in BF16, the second product accumulated
    onto the first (C += A B^T) exactly as the step launches it: contraction
    18944, N = 3584.  The stored first product is rounded to BF16 once more
    before the sum, which the |C_ref(gate)| term of the tolerance covers."""
    dyg, dyu, wg, wu = data["dY_gate"], data["dY_up"], data["W_gate"], data["W_up"]
    ag, au = fp8hg.fp8_quant_token(dyg, 0, E5M2), fp8hg.fp8_quant_token(dyu, 0, E5M2)
    _, btg = fp8hg.fp8_quant_block128(wg, E4M3, transposed_copy=True)
    _, btu = fp8hg.fp8_quant_block128(wu, E4M3, transposed_copy=True)
    dx = fp8hg.fp8_gemm_scaled(fp8hg.DGRAD, ag, btg)
    fp8hg.fp8_gemm_scaled(fp8hg.DGRAD, au, btu, out=dx, accumulate=True)
    assert fp8hg.fp8hg_get_device_error() == 0
    rng = np.random.default_rng(6)
    ii = np.concatenate([[0, M - 1], rng.choice(np.arange(1, M - 1), 8, replace=False)])
    c_gpu, c_ref, s_abs = [], [], []
    for b in [0, HID // 128 - 1, int(rng.integers(1, HID // 128 - 1))]:
        jj = np.concatenate([[0, 127], rng.choice(np.arange(1, 127), 2, replace=False)])
        r1, s1 = _dgrad_ref(dyg, wg, ii, b, jj, E5M2)
        r2, s2 = _dgrad_ref(dyu, wu, ii, b, jj, E5M2)
        c_ref.append(r1 + r2)
        s_abs.append(s1 + s2 + np.abs(r1))
        g = dx[torch.from_numpy(ii).cuda()][:, torch.from_numpy(128 * b + jj).cuda()]
        c_gpu.append(g.float().cpu().numpy().ravel())
    check_gemm(np.concatenate(c_gpu), np.concatenate(c_ref), np.concatenate(s_abs),
               "dgrad accumulate")
