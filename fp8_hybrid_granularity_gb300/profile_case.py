"""Small single-kernel cases for profiling (ncu) and quick timing.

    python -m fp8_hybrid_granularity_gb300.profile_case gemm --m 4096
    python -m fp8_hybrid_granularity_gb300.profile_case quant_row --m 4096

Each case builds seeded synthetic inputs at the 7B shapes (reduced token
count M), runs `--warmup` untimed launches and `--iters` timed launches of one
kernel, and prints the mean launch time from CUDA events.  Cases:

  gemm       fprop down projection: A = H [M, 18944] per token, B = W_down
             [3584, 18944] 128x128 blocks, BF16 out
  gemm_gate  fprop gate projection: A = X [M, 3584] per token, B = W_gate
             [18944, 3584] 128x128 blocks, BF16 out
  gemm_gate_q  the same with the output quantized in the epilogue (E4M3,
             1x128 along N)
  gemm_gate_f32s  the gate projection with FP32 scales (promotion GEMM)
  gemm_f32s  the down projection with FP32 scales
  quant_row_f32s  per-token quantization of H with FP32 scales
  wgrad      gate weight gradient: A = dY^T [18944, M] 1x128 E5M2, B = X^T
             [3584, M] 1x128 E4M3, FP32 out
  quant_row  per-token quantization of H [M, 18944]
  quant_1x128  1x128 quantization of H [M, 18944]
  quant_t    1x128-along-tokens transposed quantization of H [M, 18944]
  block128   128x128 quantization (+ transposed copy) of W_down [3584, 18944]
  mx32       MXFP8 quantization of [M, 4096]
  gemm_shape fprop on any shape: A [M, K] per token, B [N, K] 128x128 blocks,
             BF16 out (--n, --k; e.g. the 1.5B layers at M = 8192)
  gemm_mx    MXFP8 x MXFP8 GEMM: A [M, 4096], B [4096, 4096] (layer-norm-like
             and normal rows), both quantized in 32-element blocks, BF16 out
  mx32_mon   the same with the clamp monitor's counts
  requant    stored per-token FP8 codes of H [M, 18944] -> 1x128 along the
             tokens, transposed (the weight-gradient operand)
  sweep      quantizer bandwidth for BF16 [R, 4096] tensors, R = 128 * 4^i
             (1 MB to 4 GB), per token, 1x128 and 128x128, with L2 flushed
             before every timed launch (and L2-warm for tensors <= 64 MB);
             then the down-projection GEMM at M = 4096, 16384, 65536.  One
             JSON line per point (--m is ignored).
"""
from __future__ import annotations

import argparse
import json

import torch

import fp8_hybrid_granularity_gb300 as fp8hg
from fp8_hybrid_granularity_gb300 import workloads

HID, MLP = 3584, 18944


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["gemm", "gemm_gate", "gemm_gate_q", "gemm_gate_f32s", "gemm_f32s",
                                     "quant_row_f32s", "wgrad", "quant_row", "quant_1x128", "quant_t", "block128", "gemm_mx", "gemm_shape",
                                     "mx32", "mx32_mon", "requant", "sweep"])
    ap.add_argument("--m", type=int, default=4096)
    ap.add_argument("--warmup", type=int, default=2)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--n", type=int, default=HID)
    ap.add_argument("--k", type=int, default=MLP)
    args = ap.parse_args()
    fp8hg.load_library()
    dev = torch.device("cuda", 0)
    if args.case == "sweep":
        return sweep(dev, max(args.iters, 3))
    M = args.m
    mk = lambda kind, r, c, n: workloads.make_tensor(kind, r, c, 4, n, device=dev)
    E4 = fp8hg.E4M3
    if args.case == "gemm":
        h = mk("act", M, MLP, "H")
        w = mk("weight", HID, MLP, "W_down")
        a = fp8hg.fp8_quant_token(h, 0, E4)
        b = fp8hg.fp8_quant_block128(w, E4)
        out = torch.empty((M, HID), dtype=torch.bfloat16, device=dev)
        fn = lambda: fp8hg.fp8_gemm_scaled(fp8hg.FPROP, a, b, out=out)
        work, unit = 2.0 * M * HID * MLP, "flop"
    elif args.case in ("gemm_gate", "gemm_gate_q"):
        x = mk("act", M, HID, "X")
        w = mk("weight", MLP, HID, "W_gate")
        a = fp8hg.fp8_quant_token(x, 0, E4)
        b = fp8hg.fp8_quant_block128(w, E4)
        if args.case == "gemm_gate_q":
            out = fp8hg.alloc_token(M, MLP, 128, E4, False, dev)
            fn = lambda: fp8hg.fp8_gemm_scaled_q(fp8hg.FPROP, a, b, E4, out=out)
        else:
            out = torch.empty((M, MLP), dtype=torch.bfloat16, device=dev)
            fn = lambda: fp8hg.fp8_gemm_scaled(fp8hg.FPROP, a, b, out=out)
        work, unit = 2.0 * M * HID * MLP, "flop"
    elif args.case in ("gemm_gate_f32s", "gemm_f32s"):
        gate = args.case == "gemm_gate_f32s"
        a_src = mk("act", M, HID if gate else MLP, "X" if gate else "H")
        w = mk("weight", MLP if gate else HID, HID if gate else MLP, "W_gate" if gate else "W_down")
        a = fp8hg.fp8_quant_token_f32s(a_src, 0, E4)
        b = fp8hg.fp8_quant_block128_f32s(w, E4)
        out = torch.empty((M, w.shape[0]), dtype=torch.bfloat16, device=dev)
        fn = lambda: fp8hg.fp8_gemm_scaled_f32s(fp8hg.FPROP, a, b, out=out)
        work, unit = 2.0 * M * HID * MLP, "flop"
    elif args.case == "quant_row_f32s":
        h = mk("act", M, MLP, "H")
        out = fp8hg.QTensor(torch.empty((M, MLP), dtype=torch.uint8, device=dev),
                            torch.empty((M, 1), dtype=torch.float32, device=dev), E4, 0, 1)
        fn = lambda: fp8hg.fp8_quant_token_f32s(h, 0, E4, out=out)
        work, unit = 3.0 * M * MLP + 4 * M, "byte"
    elif args.case == "wgrad":
        dy = mk("grad", M, MLP, "dY_gate")
        x = mk("act", M, HID, "X")
        a = fp8hg.fp8_quant_token(dy, 128, fp8hg.E5M2, transpose=True)
        b = fp8hg.fp8_quant_token(x, 128, E4, transpose=True)
        out = torch.empty((MLP, HID), dtype=torch.float32, device=dev)
        fn = lambda: fp8hg.fp8_gemm_scaled(fp8hg.WGRAD, a, b, out=out)
        work, unit = 2.0 * M * HID * MLP, "flop"
    elif args.case in ("quant_row", "quant_1x128", "quant_t"):
        h = mk("act", M, MLP, "H")
        group = 0 if args.case == "quant_row" else 128
        tr = args.case == "quant_t"
        out = fp8hg.alloc_token(M, MLP, group, E4, tr, dev)
        fn = lambda: fp8hg.fp8_quant_token(h, group, E4, tr, out=out)
        work, unit = 3.0 * M * MLP + (M if group == 0 else M * MLP / 128), "byte"
    elif args.case == "gemm_shape":
        a = fp8hg.fp8_quant_token(mk("act", M, args.k, "A"), 0, E4)
        b = fp8hg.fp8_quant_block128(mk("weight", args.n, args.k, "W"), E4)
        out = torch.empty((M, args.n), dtype=torch.bfloat16, device=dev)
        fn = lambda: fp8hg.fp8_gemm_scaled(fp8hg.FPROP, a, b, out=out)
        work, unit = 2.0 * M * args.n * args.k, "flop"
    elif args.case == "gemm_mx":
        a = fp8hg.fp8_quant_mx32(mk("mx_ln", M, 4096, "A"), E4)
        b = fp8hg.fp8_quant_mx32(mk("mx_ln", 4096, 4096, "B"), E4)
        out = torch.empty((M, 4096), dtype=torch.bfloat16, device=dev)
        fn = lambda: fp8hg.fp8_gemm_scaled(fp8hg.FPROP, a, b, out=out)
        work, unit = 2.0 * M * 4096 * 4096, "flop"
    elif args.case == "block128":
        w = mk("weight", HID, MLP, "W_down")
        o, ot = fp8hg.alloc_block128(HID, MLP, E4, True, dev)
        fn = lambda: fp8hg.fp8_quant_block128(w, E4, True, out=o, out_t=ot)
        work, unit = 4.0 * HID * MLP + 2.0 * HID * MLP / 16384, "byte"
    elif args.case == "requant":
        h = mk("act", M, MLP, "H")
        src = fp8hg.fp8_quant_token(h, 0, E4)
        o = fp8hg.alloc_token(M, MLP, 128, E4, True, dev)
        fn = lambda: fp8hg.fp8_requant_t(src, E4, out=o)
        work, unit = 2.0 * M * MLP + M + M * MLP / 128, "byte"
    else:
        x = mk("mx_ln", M, 4096, "A")
        o = fp8hg.alloc_mx32(M, 4096, E4, dev)
        if args.case == "mx32_mon":
            st = torch.zeros(4, dtype=torch.int64, device=dev)
            rs = torch.zeros(M, dtype=torch.int32, device=dev)
            fn = lambda: fp8hg.fp8_quant_mx32_monitor(x, E4, stats=st, row_saturated=rs, out=o)
        else:
            fn = lambda: fp8hg.fp8_quant_mx32(x, E4, out=o)
        work, unit = 3.0 * M * 4096 + M * 4096 / 32, "byte"
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    evs = []
    for _ in range(args.iters):
        a0, b0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record()
        fn()
        b0.record()
        evs.append((a0, b0))
    torch.cuda.synchronize()
    status = fp8hg.fp8hg_get_device_error()
    if status != 0:
        raise SystemExit(f"device error {fp8hg.fp8hg_status_str(status)}")
    ms = sum(a0.elapsed_time(b0) for a0, b0 in evs) / len(evs)
    rate = work / (ms * 1e-3) / (1e12 if unit == "flop" else 1e9)
    print(json.dumps({"case": args.case, "m": M, **({"n": args.n, "k": args.k} if args.case == "gemm_shape" else {}), "ms": ms,
                      ("tflops" if unit == "flop" else "gbs"): rate}))


def _time(fn, iters, flush=None):
    """Mean CUDA-event time of fn over iters launches (ms); flush() runs
    untimed before each launch when given."""
    total = 0.0
    for _ in range(iters):
        if flush is not None:
            flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        total += a.elapsed_time(b)
    return total / iters


def sweep(dev, iters):
    E4 = fp8hg.E4M3
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    scratch = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    flush = lambda: scratch.fill_(1)
    for i in range(7):
        R, C = 128 * 4 ** i, 4096
        x = workloads.make_tensor("act", R, C, 4, "sweep", device=dev)
        outs = {"token": fp8hg.alloc_token(R, C, 0, E4, False, dev),
                "1x128": fp8hg.alloc_token(R, C, 128, E4, False, dev),
                "128x128": fp8hg.alloc_block128(R, C, E4, False, dev)[0]}
        fns = {"token": lambda: fp8hg.fp8_quant_token(x, 0, E4, out=outs["token"]),
               "1x128": lambda: fp8hg.fp8_quant_token(x, 128, E4, out=outs["1x128"]),
               "128x128": lambda: fp8hg.fp8_quant_block128(x, E4, out=outs["128x128"])}
        groups = {"token": R, "1x128": R * C / 128, "128x128": R * C / 16384}
        for g, fn in fns.items():
            fn()
            torch.cuda.synchronize()
            nbytes = 3.0 * R * C + groups[g]
            line = {"case": "sweep_quant", "gran": g, "rows": R, "cols": C,
                    "tensor_mb": 2.0 * R * C / 2 ** 20, "bytes": nbytes}
            ms = _time(fn, iters, flush)
            line.update(ms_flushed=ms, gbs_flushed=nbytes / ms / 1e6)
            if 2 * R * C <= 64 * 2 ** 20:
                ms_w = _time(fn, iters)
                line.update(ms_l2warm=ms_w, gbs_l2warm=nbytes / ms_w / 1e6)
            print(json.dumps(line), flush=True)
        del x, outs, fns
        torch.cuda.empty_cache()
    assert fp8hg.fp8hg_get_device_error() == 0
    w = workloads.make_tensor("weight", HID, MLP, 4, "W_down", device=dev)
    b = fp8hg.fp8_quant_block128(w, E4)
    for M in (4096, 16384, 65536):
        h = workloads.make_tensor("act", M, MLP, 4, "H", device=dev)
        a = fp8hg.fp8_quant_token(h, 0, E4)
        del h
        out = torch.empty((M, HID), dtype=torch.bfloat16, device=dev)
        fn = lambda: fp8hg.fp8_gemm_scaled(fp8hg.FPROP, a, b, out=out)
        fn()
        torch.cuda.synchronize()
        ms = _time(fn, iters, flush)
        print(json.dumps({"case": "sweep_gemm_down", "m": M, "k": MLP, "n": HID, "ms": ms,
                          "tflops": 2.0 * M * HID * MLP / ms / 1e9}), flush=True)
        del a, out
        torch.cuda.empty_cache()
    status = fp8hg.fp8hg_get_device_error()
    if status != 0:
        raise SystemExit(f"device error {fp8hg.fp8hg_status_str(status)}")


if __name__ == "__main__":
    main()
