"""Re-quantization of stored FP8 codes (fp8_requant_t) on the GPU against the
oracle, bit for bit.  The stored codes fed to both sides are the oracle's own
quantization of seeded BF16 inputs."""
import numpy as np
import pytest
import torch

import oracle
from oracle import E4M3, E5M2, GRAN_ROW, GRAN_1x128
import fp8_hybrid_granularity_gb300 as fp8hg
from fp8_hybrid_granularity_gb300 import workloads
from golden_io import load_quant_examples
from helpers import np_u8, assert_codes_equal

pytestmark = pytest.mark.gpu

FMT = {"e4m3": E4M3, "e5m2": E5M2}
GRAN = {"row": GRAN_ROW, "1x128": GRAN_1x128}


def _src(q, s, gran, fmt, ld=None):
    """Upload oracle codes / scales as a QTensor (scale columns padded to 4),
    optionally inside a wider row stride."""
    rows, cols = q.shape
    ld = ld or cols
    buf = torch.zeros((rows, ld), dtype=torch.uint8, device="cuda")
    buf[:, :cols] = torch.from_numpy(q).cuda()
    ns = s.shape[1]
    sb = torch.zeros((rows, (ns + 3) // 4 * 4), dtype=torch.uint8, device="cuda")
    sb[:, :ns] = torch.from_numpy(np.ascontiguousarray(s)).cuda()
    return fp8hg.QTensor(buf[:, :cols], sb, fmt, gran, ns)


def _gpu_requant(q, s, gran, fmt_in, fmt_out, ld=None):
    out = fp8hg.fp8_requant_t(_src(q, s, gran, fmt_in, ld), fmt_out)
    torch.cuda.synchronize()
    return np_u8(out.codes), np_u8(out.scales())


@pytest.mark.parametrize("case", load_quant_examples("requant_examples.txt"),
                         ids=lambda c: c["case"])
def test_hand_worked(cuda_lib, case):
    rows = case["rows"]
    q = case["q_in"].reshape(rows, -1)
    s = case["s_in"].reshape(rows, -1)
    if q.shape[1] < 128:                   # the kernel works on 128-column tiles
        q = np.concatenate([q, np.zeros((rows, 128 - q.shape[1]), np.uint8)], axis=1)
    qt, st = _gpu_requant(q, s, GRAN[case["gran"]], FMT[case["fmt_in"]], FMT[case["fmt_out"]])
    n = case["q_out"].size // rows
    assert_codes_equal(qt[:n].ravel(), case["q_out"], case["case"])
    assert_codes_equal(st[:n].ravel(), case["s_out"], case["case"] + " scales")


@pytest.mark.parametrize("gran", [GRAN_ROW, GRAN_1x128])
@pytest.mark.parametrize("fmt_in,fmt_out", [(E4M3, E4M3), (E5M2, E5M2), (E5M2, E4M3),
                                            (E4M3, E5M2)])
def test_parity_multi_tile_strided(cuda_lib, gran, fmt_in, fmt_out):
    """3 x 5 tiles, source rows inside a wider stride; activations and
    Student-t gradients."""
    kind = "grad" if fmt_in == E5M2 else "act"
    x = workloads.make_tensor(kind, 384, 640, 31 + gran, f"rq{fmt_in}{fmt_out}")
    q, s = oracle.quant_token(workloads.bf16_bits(x), 0 if gran == GRAN_ROW else 128, fmt_in)
    qt, st = _gpu_requant(q, s, gran, fmt_in, fmt_out, ld=768)
    qo, so = oracle.requant_t(q, s, gran, fmt_in, fmt_out)
    assert_codes_equal(qt, qo, "codes")
    assert_codes_equal(st, so, "scales")


def test_extreme_scales_and_specials(cuda_lib):
    """Stored values across the whole scale range (bytes 0..240, so x_hat
    reaches FP32 subnormals), zeros, a NaN scale and NaN codes."""
    rng = np.random.default_rng(5)
    rows, cols = 256, 256
    q = rng.integers(0, 256, (rows, cols), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x3C                       # no NaN codes except below
    s = rng.integers(0, 241, (rows, 2), dtype=np.uint8)
    s[:128, 0] = rng.integers(0, 8, 128)               # tiny scales: subnormal x_hat
    s[130, 1] = 0xFF                                   # NaN scale: groups of token 130
    q[200, 17] = 0x7F                                  # NaN code in column 17
    q[:, 40] = 0                                       # an all-zero column
    qt, st = _gpu_requant(q, s, GRAN_1x128, E4M3, E4M3)
    qo, so = oracle.requant_t(q, s, GRAN_1x128, E4M3, E4M3)
    assert_codes_equal(qt, qo, "codes")
    assert_codes_equal(st, so, "scales")
    assert so[17, 1] == 0xFF and so[200, 1] == 0xFF and so[40, 0] == 0


def test_full_1p5b_activation_sampled(cuda_lib):
    """H [8192, 8960] stored per token (E4M3): the whole tensor re-quantized on
    the GPU, compared on 6 sampled 128-column slices (all 8192 tokens)."""
    h = workloads.workload_tensor("fprop_1p5b", "H")
    q, s = oracle.quant_token(workloads.bf16_bits(h), 0, E4M3)
    qt, st = _gpu_requant(q, s, GRAN_ROW, E4M3, E4M3)
    rng = np.random.default_rng(8)
    blocks = sorted(set([0, 8960 // 128 - 1] + list(rng.choice(8960 // 128, 4, replace=False))))
    for b in blocks:
        cs = slice(128 * b, 128 * b + 128)
        qo, so = oracle.requant_t(q[:, cs], s, GRAN_ROW, E4M3, E4M3)
        assert_codes_equal(qt[cs], qo, f"cols {cs}")
        assert_codes_equal(st[cs], so, f"scales {cs}")


def test_empty(cuda_lib):
    q = torch.empty((0, 128), dtype=torch.uint8, device="cuda")
    src = fp8hg.QTensor(q, torch.empty((0, 4), dtype=torch.uint8, device="cuda"), E4M3,
                        GRAN_ROW, 1)
    out = fp8hg.fp8_requant_t(src, E4M3)
    assert out.codes.shape == (128, 0)
