"""The MX clamp monitor on the GPU against the oracle: codes and scales bit
for bit, the four counts and the per-row saturated counts exactly."""
import numpy as np
import pytest
import torch

import oracle
from oracle import E4M3, E5M2
import fp8_hybrid_granularity_gb300 as fp8hg
from fp8_hybrid_granularity_gb300 import workloads
from golden_io import load_quant_examples
from helpers import np_u8, assert_codes_equal

pytestmark = pytest.mark.gpu


def _run(x_dev, fmt, with_rows=True):
    rows = x_dev.shape[0]
    rs = torch.zeros(rows, dtype=torch.int32, device=x_dev.device) if with_rows else None
    q, st = fp8hg.fp8_quant_mx32_monitor(x_dev, fmt, row_saturated=rs)
    torch.cuda.synchronize()
    stats = dict(zip(fp8hg.MX_STAT_NAMES, (int(v) for v in st.cpu())))
    return q, stats, (rs.cpu().numpy() if with_rows else None)


def _check(x_bits, x_dev, fmt, what):
    q, stats, rs = _run(x_dev, fmt)
    qo, so, sto, rso = oracle.mx32_monitor(x_bits, fmt)
    assert_codes_equal(np_u8(q.codes), qo, f"{what} codes")
    assert_codes_equal(np_u8(q.scales()), so, f"{what} scales")
    assert stats == sto, what
    assert np.array_equal(rs.astype(np.uint64), rso), what
    return stats


def test_hand_worked_fixture(cuda_lib):
    (c,) = load_quant_examples("mx_monitor_examples.txt")
    x = c["x"].reshape(c["rows"], -1)
    xd = workloads.from_bits(x).cuda()
    st = _check(x, xd, E4M3, "fixture")
    assert st["saturated"] == c["saturated"] and st["blocks_collapsed"] == c["blocks_collapsed"]


@pytest.mark.parametrize("name", ["A", "A_clamp"])
@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_mx_workload_full_tensor(cuda_lib, name, fmt):
    """The 4096x4096 MX inputs: layer-norm-like rows [0, 2048) (collapse, or
    saturation in the clamp variant), N(0,1) rows [2048, 4096)."""
    x = workloads.workload_tensor("mxfp8_4096", name)
    st = _check(workloads.bf16_bits(x), x.cuda(), fmt, name)
    if name == "A_clamp":
        assert st["saturated"] >= 2048 * 4096
    assert st["blocks_collapsed"] >= 2048 * 4096 // 32


@pytest.mark.parametrize("rows,cols,ld", [(77, 1056, 1120), (1, 32, 32), (5, 4128, 4136)])
def test_ragged_and_strided(cuda_lib, rows, cols, ld):
    full = workloads.make_tensor("normal", rows, ld, 13, f"mon{cols}") * 3.0
    full[:, : cols // 2] = 1.0 + 1e-3 * full[:, : cols // 2]     # a clustered half
    full = full.to(torch.bfloat16)
    xd = full.cuda()[:, :cols]
    _check(workloads.bf16_bits(full[:, :cols].contiguous()), xd, E4M3, f"{rows}x{cols}")


def test_matches_plain_mx32_and_accumulates(cuda_lib):
    x = workloads.workload_tensor("mxfp8_4096", "A_clamp")[1984:2112].cuda()
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
    q1 = fp8hg.fp8_quant_mx32(x, E4M3, clamp_count=cnt)
    st = torch.zeros(4, dtype=torch.int64, device="cuda")
    q2, _ = fp8hg.fp8_quant_mx32_monitor(x, E4M3, stats=st)
    assert torch.equal(q1.codes, q2.codes) and torch.equal(q1.scale, q2.scale)
    assert int(st[0]) == int(cnt.item()) > 0
    first = st.clone()
    fp8hg.fp8_quant_mx32_monitor(x, E4M3, stats=st)
    assert torch.equal(st, 2 * first)


def test_empty_is_a_no_op(cuda_lib):
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    _, st = fp8hg.fp8_quant_mx32_monitor(x, E4M3)
    assert int(st.abs().sum()) == 0
