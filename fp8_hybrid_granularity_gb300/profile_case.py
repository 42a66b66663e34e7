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
  mx32_mon   the same with the clamp monitor's counts
  requant    stored per-token FP8 codes of H [M, 18944] -> 1x128 along the
             tokens, transposed (the weight-gradient operand)
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
                                     "quant_row_f32s", "wgrad", "quant_row", "quant_1x128", "quant_t", "block128",
                                     "mx32", "mx32_mon", "requant"])
    ap.add_argument("--m", type=int, default=4096)
    ap.add_argument("--warmup", type=int, default=2)
    ap.add_argument("--iters", type=int, default=3)
    args = ap.parse_args()
    fp8hg.load_library()
    dev = torch.device("cuda", 0)
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
    print(json.dumps({"case": args.case, "m": M, "ms": ms,
                      ("tflops" if unit == "flop" else "gbs"): rate}))


if __name__ == "__main__":
    main()
