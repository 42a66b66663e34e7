"""Pins for the oracle's re-quantization of stored FP8 codes along the tokens:
hand-worked cases (tests/golden/requant_examples.txt), and the reduction to
the BF16 transposed quantizer when the stored values are exact in BF16."""
import numpy as np
import pytest
import torch

import oracle
from oracle import E4M3, E5M2, GRAN_ROW, GRAN_1x128
from fp8_hybrid_granularity_gb300 import workloads
from golden_io import load_quant_examples

FMT = {"e4m3": E4M3, "e5m2": E5M2}
GRAN = {"row": GRAN_ROW, "1x128": GRAN_1x128}


@pytest.mark.parametrize("case", load_quant_examples("requant_examples.txt"),
                         ids=lambda c: c["case"])
def test_hand_worked(case):
    rows = case["rows"]
    q = case["q_in"].reshape(rows, -1)
    s = case["s_in"].reshape(rows, -1)
    qt, st = oracle.requant_t(q, s, GRAN[case["gran"]], FMT[case["fmt_in"]], FMT[case["fmt_out"]])
    assert np.array_equal(qt.ravel(), case["q_out"])
    assert np.array_equal(st.ravel(), case["s_out"])


def _exact_bf16(x_hat):
    """x_hat as BF16 bit patterns, asserting the conversion is exact."""
    t = torch.from_numpy(x_hat)
    b = t.to(torch.bfloat16)
    assert torch.equal(b.to(torch.float64), t), "stored value not exact in BF16"
    return workloads.bf16_bits(b)


@pytest.mark.parametrize("gran", [GRAN_ROW, GRAN_1x128])
@pytest.mark.parametrize("fmt_in,fmt_out", [(E4M3, E4M3), (E5M2, E5M2), (E4M3, E5M2)])
def test_reduces_to_bf16_transposed_quantizer(gran, fmt_in, fmt_out):
    """Every stored value decode(q) * 2^e of these tensors is exact in BF16
    (3 or 2 mantissa bits, exponents well inside BF16's range), so quantizing
    the stored values from BF16 with 1x128 groups along the rows, transposed,
    must give the same codes and scales as the re-quantizer."""
    x = workloads.make_tensor("act", 256, 384, 21, "rq")
    xb = workloads.bf16_bits(x)
    q, s = oracle.quant_token(xb, 0 if gran == GRAN_ROW else 128, fmt_in)
    x_hat = oracle.dequant(q, s, gran, fmt_in)
    qt, st = oracle.requant_t(q, s, gran, fmt_in, fmt_out)
    qr, sr = oracle.quant_token(_exact_bf16(x_hat), 128, fmt_out, transpose=True)
    assert np.array_equal(qt, qr)
    assert np.array_equal(st, sr)


def test_scale_is_the_tight_round_up():
    """Each output group's scale is the smallest power of two that keeps the
    group's largest stored magnitude within FMAX: FMAX/2 < amax/2^e <= FMAX."""
    x = workloads.make_tensor("grad", 384, 256, 22, "rq2")
    q, s = oracle.quant_token(workloads.bf16_bits(x), 128, E5M2)
    x_hat = oracle.dequant(q, s, GRAN_1x128, E5M2)
    for fmt in (E4M3, E5M2):
        qt, st = oracle.requant_t(q, s, GRAN_1x128, E5M2, fmt)
        fmax = oracle.fp8_max(fmt)
        amax = np.abs(x_hat).reshape(3, 128, 256).max(axis=1).T      # [cols, groups]
        ratio = amax / np.exp2(st.astype(np.float64) - 127)
        nz = amax > 0
        assert (ratio[nz] <= fmax).all() and (ratio[nz] > fmax / 2).all()


def test_rejects_bad_shapes():
    q = np.zeros((100, 128), np.uint8)
    with pytest.raises(ValueError):
        oracle.requant_t(q, np.zeros((100, 1), np.uint8), GRAN_ROW, E4M3, E4M3)
