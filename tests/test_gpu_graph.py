"""The library's calls can be captured into a CUDA graph and replayed: the
block quantizer, the single-read dual quantizer (cooperative launch, with its
workspace clear), the GEMM, and the split-K GEMM (cooperative launch).  The
replay of the captured sequence on new inputs gives the same bytes as the
same calls made one by one."""
import pytest
import torch

import fp8_hybrid_granularity_gb300 as fp8hg
from fp8_hybrid_granularity_gb300 import workloads, FPROP, E4M3

pytestmark = pytest.mark.gpu


def test_captured_sequence_matches_eager(cuda_lib):
    M, N, K = 512, 384, 2048
    dev = torch.device("cuda")
    x = workloads.make_tensor("act", M, K, 21, "graph-x", device=dev)
    w = workloads.make_tensor("weight", N, K, 22, "graph-w", device=dev)
    tok = fp8hg.alloc_token(M, K, 0, E4M3, False, dev)
    tr = fp8hg.alloc_token(M, K, 128, E4M3, True, dev)
    wq, _ = fp8hg.alloc_block128(N, K, E4M3, False, dev)
    ws_dual = fp8hg.dual_workspace(M, K, dev)
    ws_split = fp8hg.splitk_workspace(M, N, K, 2, dev)
    c = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    c2 = torch.empty((M, N), dtype=torch.bfloat16, device=dev)

    def step():
        fp8hg.fp8_quant_block128(w, E4M3, out=wq)
        fp8hg.fp8_quant_token_dual(x, E4M3, out=tok, out_t=tr, workspace=ws_dual)
        fp8hg.fp8_gemm_scaled(FPROP, tok, wq, out=c)
        fp8hg.fp8_gemm_scaled_splitk(FPROP, tok, wq, out=c2, split_k=2, workspace=ws_split)

    step()                                   # first calls (library set-up) outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=side):
        step()
    # new inputs in the captured buffers, then one replay
    x.copy_(workloads.make_tensor("act", M, K, 23, "graph-x2", device=dev))
    w.copy_(workloads.make_tensor("weight", N, K, 24, "graph-w2", device=dev))
    g.replay()
    torch.cuda.synchronize()
    assert fp8hg.fp8hg_get_device_error() == 0
    got = [t.clone() for t in (tok.codes, tok.scale, tr.codes, tr.scale, wq.codes, wq.scale, c, c2)]
    step()                                   # the same calls, eagerly, on the same inputs
    torch.cuda.synchronize()
    assert fp8hg.fp8hg_get_device_error() == 0
    want = (tok.codes, tok.scale, tr.codes, tr.scale, wq.codes, wq.scale, c, c2)
    names = ("codes", "scales", "codes^T", "scales^T", "W codes", "W scales", "C", "C split")
    for a, b, n in zip(got, want, names):
        assert torch.equal(a.view(torch.uint8) if a.dtype != torch.uint8 else a,
                           b.view(torch.uint8) if b.dtype != torch.uint8 else b), n
