"""Benchmark of the hybrid-granularity FP8 hot path on GB300.

One step = one Qwen2.5-7B-shaped MLP block (gate, up, down linears) at
M = 16384 tokens, hidden 3584, MLP width 18944, run through the C ABI:

  quantize   W_gate, W_up, W_down   128x128 blocks, E4M3 (+ transposed copies)
             X, H                   per token, E4M3
             dY_gate, dY_up, dY_down per token, E5M2
             X^T, H^T, dY^T (x3)    1x128 groups along tokens (wgrad layout)
  fprop      Y_g = X W_g^T, Y_u = X W_u^T, Y_d = H W_d^T           (BF16 out)
  dgrad      dX = dY_g W_g + dY_u W_u (accumulated), dH = dY_d W_d (BF16 out)
  wgrad      dW_g = dY_g^T X, dW_u = dY_u^T X, dW_d = dY_d^T H       (FP32 out)

13 quantizer launches + 9 GEMM launches per step.  The headline value is
total GEMM FLOP / step time (TFLOP/s including every quantization pass).
Inputs are seeded synthetic BF16 tensors with the recipe's distributions,
resident in HBM; every step touches ~15 GB, far more than the 126 MB L2, so
no explicit flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--impl reference times the CPU oracle (plain C, fp64, single-threaded) on a
bounded sample of the same step, in one process per host core: a 32x32 block
of outputs of each of the 9 GEMMs at full K, including the oracle's
quantization of the operand slices that block needs.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from fp8_hybrid_granularity_gb300 import replicas  # noqa: E402

METRIC = "scaled-FP8 GEMM TFLOP/s incl. quant (% FP8 peak); quantizer GB/s (% HBM) at 7B shapes"
M_TOK, HID, MLP = 16384, 3584, 18944
WORKLOAD = (f"linear_step_7b: Qwen2.5-7B MLP block (gate/up/down) fprop+dgrad+wgrad, "
            f"M={M_TOK} tokens, hidden {HID}, MLP {MLP}; per-token E4M3 activations, "
            f"128x128-block E4M3 weights, per-token E5M2 output grads, 1x128 wgrad re-quant")
GEMM_FLOP = 2.0 * M_TOK * HID * MLP          # every GEMM of the step has this size
N_GEMM, N_QUANT = 9, 13
GEMM_NAMES = ["fprop_gate", "fprop_up", "fprop_down", "dgrad_gate", "dgrad_up", "dgrad_down",
              "wgrad_gate", "wgrad_up", "wgrad_down"]
QUANT_NAMES = ["W_gate_blk", "W_up_blk", "W_down_blk", "X_tok", "H_tok", "dYg_tok", "dYu_tok",
               "dYd_tok", "X_t", "H_t", "dYg_t", "dYu_t", "dYd_t"]
GEMM_SRC = os.path.join(ROOT, "fp8_hybrid_granularity_gb300", "csrc", "gemm.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gemm_mxf8_linear_step_7b.md")


def _parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sus=float(p["bf16_tflops_sustained"]), src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def _gemm_traffic():
    """Per-launch DRAM bytes of the GEMM from the committed ncu summary, or
    None when the kernel source changed since the capture."""
    try:
        text = open(TRAFFIC_FILE).read()
        sha = re.search(r"gemm\.cu sha256: ([0-9a-f]{64})", text).group(1)
        nbytes = float(re.search(r"traffic per full-size launch \(bytes\): ([0-9.e+]+)", text).group(1))
    except Exception:
        return None
    cur = hashlib.sha256(open(GEMM_SRC, "rb").read()).hexdigest()
    return nbytes if cur == sha else None


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc, self.lines = index, None, []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self._t.join(timeout=2)
        mhz, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                mx.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        loaded = [m for m, p in zip(mhz, power) if p > 300.0] or mhz
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(mhz), "power_w_max": max(power) if power else None}


# ----------------------------------------------------------------- GPU step
# The step's inputs in the order its launches first read them.
INPUT_ORDER = ["W_gate", "W_up", "W_down", "X", "H", "dY_gate", "dY_up", "dY_down"]


class Step:
    """Preallocated buffers and the launch sequence of one step."""

    def __init__(self, torch, fp8hg, workloads, device, seed_offset=0):
        self.torch, self.f = torch, fp8hg
        seed = replicas.replica_seed(2, seed_offset)
        T = lambda kind, r, c, name: workloads.make_tensor(kind, r, c, seed, name,
                                                           device=device)
        self.inp = {
            "X": T("act", M_TOK, HID, "X"), "H": T("act", M_TOK, MLP, "H"),
            "W_gate": T("weight", MLP, HID, "W_gate"), "W_up": T("weight", MLP, HID, "W_up"),
            "W_down": T("weight", HID, MLP, "W_down"),
            "dY_gate": T("grad", M_TOK, MLP, "dY_gate"), "dY_up": T("grad", M_TOK, MLP, "dY_up"),
            "dY_down": T("grad", M_TOK, HID, "dY_down"),
        }
        E4, E5 = fp8hg.E4M3, fp8hg.E5M2
        at, ab = fp8hg.alloc_token, fp8hg.alloc_block128
        self.wq = {n: ab(*self.inp[n].shape, E4, True, device) for n in ("W_gate", "W_up", "W_down")}
        self.xq = at(M_TOK, HID, 0, E4, False, device)
        self.hq = at(M_TOK, MLP, 0, E4, False, device)
        self.dyq = {n: at(*self.inp[n].shape, 0, E5, False, device)
                    for n in ("dY_gate", "dY_up", "dY_down")}
        self.xt = at(M_TOK, HID, 128, E4, True, device)
        self.ht = at(M_TOK, MLP, 128, E4, True, device)
        self.dyt = {n: at(*self.inp[n].shape, 128, E5, True, device)
                    for n in ("dY_gate", "dY_up", "dY_down")}
        bf, f32 = torch.bfloat16, torch.float32
        e = lambda shape, dt: torch.empty(shape, dtype=dt, device=device)
        self.out = {"Y_gate": e((M_TOK, MLP), bf), "Y_up": e((M_TOK, MLP), bf),
                    "Y_down": e((M_TOK, HID), bf), "dX": e((M_TOK, HID), bf),
                    "dH": e((M_TOK, MLP), bf), "dW_gate": e((MLP, HID), f32),
                    "dW_up": e((MLP, HID), f32), "dW_down": e((HID, MLP), f32)}
        n_el = lambda t: t.numel()
        i = self.inp
        # algorithmic bytes of the quantizer passes: 2 B read + 1 B written per
        # element (+1 B more for the transposed weight copy) + 1 B per scale
        qb = 0.0
        for n in ("W_gate", "W_up", "W_down"):
            qb += 4.0 * n_el(i[n]) + 2.0 * n_el(i[n]) / 16384
        for n in ("X", "H", "dY_gate", "dY_up", "dY_down"):
            qb += 3.0 * n_el(i[n]) + i[n].shape[0]          # per token
            qb += 3.0 * n_el(i[n]) + n_el(i[n]) / 128       # 1x128 along tokens
        self.quant_bytes = qb
        self.in_bytes = sum(t.numel() * t.element_size() for t in i.values())
        self.out_bytes = sum(t.numel() * t.element_size() for t in self.out.values())

    def run(self, ev=None, ready=None, done=None):
        """Enqueue one step on the current stream.  ev: optional list that
        receives (kind, start_event, end_event) per launch.  ready: optional
        {input name: event}, waited on before the first launch that reads the
        input.  done: optional dict that receives {output name: event},
        recorded after the output's last write."""
        f, i, o = self.f, self.inp, self.out
        torch = self.torch
        waited = set()

        def need(*names):
            if ready is None:
                return
            for n in names:
                if n not in waited:
                    torch.cuda.current_stream().wait_event(ready[n])
                    waited.add(n)

        def finished(*names):
            if done is None:
                return
            for n in names:
                e = torch.cuda.Event()
                e.record()
                done[n] = e

        def timed(kind, fn):
            if ev is None:
                fn()
                return
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            ev.append((kind, a, b))

        E4, E5 = f.E4M3, f.E5M2
        for n in ("W_gate", "W_up", "W_down"):
            w, wt = self.wq[n]
            need(n)
            timed("quant", lambda: f.fp8_quant_block128(i[n], E4, True, out=w, out_t=wt))
        need("X")
        timed("quant", lambda: f.fp8_quant_token(i["X"], 0, E4, out=self.xq))
        need("H")
        timed("quant", lambda: f.fp8_quant_token(i["H"], 0, E4, out=self.hq))
        for n in ("dY_gate", "dY_up", "dY_down"):
            need(n)
            timed("quant", lambda: f.fp8_quant_token(i[n], 0, E5, out=self.dyq[n]))
        timed("quant", lambda: f.fp8_quant_token(i["X"], 128, E4, True, out=self.xt))
        timed("quant", lambda: f.fp8_quant_token(i["H"], 128, E4, True, out=self.ht))
        for n in ("dY_gate", "dY_up", "dY_down"):
            timed("quant", lambda: f.fp8_quant_token(i[n], 128, E5, True, out=self.dyt[n]))
        W = self.wq
        g = f.fp8_gemm_scaled
        timed("gemm", lambda: g(f.FPROP, self.xq, W["W_gate"][0], out=o["Y_gate"]))
        finished("Y_gate")
        timed("gemm", lambda: g(f.FPROP, self.xq, W["W_up"][0], out=o["Y_up"]))
        finished("Y_up")
        timed("gemm", lambda: g(f.FPROP, self.hq, W["W_down"][0], out=o["Y_down"]))
        finished("Y_down")
        timed("gemm", lambda: g(f.DGRAD, self.dyq["dY_gate"], W["W_gate"][1], out=o["dX"]))
        timed("gemm", lambda: g(f.DGRAD, self.dyq["dY_up"], W["W_up"][1], out=o["dX"],
                                accumulate=True))
        finished("dX")
        timed("gemm", lambda: g(f.DGRAD, self.dyq["dY_down"], W["W_down"][1], out=o["dH"]))
        finished("dH")
        timed("gemm", lambda: g(f.WGRAD, self.dyt["dY_gate"], self.xt, out=o["dW_gate"]))
        finished("dW_gate")
        timed("gemm", lambda: g(f.WGRAD, self.dyt["dY_up"], self.xt, out=o["dW_up"]))
        finished("dW_up")
        timed("gemm", lambda: g(f.WGRAD, self.dyt["dY_down"], self.ht, out=o["dW_down"]))
        finished("dW_down")


# ---------------------------------------------------------- oracle sample
def oracle_sample_step(tile: int = 32, barrier=None):
    """The oracle on one tile x tile block of outputs of each of the step's 9
    GEMMs at full K, quantizing the operand slices that block needs (whole
    128-row weight blocks, whole 128-token groups).  Returns (flop, seconds).
    barrier: waited on after the inputs are generated, before the clock starts
    (several processes then time the same interval)."""
    import oracle
    from fp8_hybrid_granularity_gb300 import workloads as wl
    oracle.build()
    gen = lambda kind, r, c, name: wl.bf16_bits(wl.make_tensor(kind, r, c, 2, "sample-" + name))
    E4, E5 = oracle.E4M3, oracle.E5M2
    t = tile
    # input slices (generated before timing starts)
    xs, hs = gen("act", t, HID, "X"), gen("act", t, MLP, "H")          # t tokens
    wg_rows, wu_rows = gen("weight", 128, HID, "Wg"), gen("weight", 128, HID, "Wu")
    wd_rows = gen("weight", 128, MLP, "Wd")                             # one block row
    wg_cols, wu_cols = gen("weight", MLP, 128, "Wgc"), gen("weight", MLP, 128, "Wuc")
    wd_cols = gen("weight", HID, 128, "Wdc")                            # one block column
    dyg, dyu, dyd = gen("grad", t, MLP, "dYg"), gen("grad", t, MLP, "dYu"), gen("grad", t, HID, "dYd")
    dyg_c, dyu_c = gen("grad", M_TOK, t, "dYgc"), gen("grad", M_TOK, t, "dYuc")
    dyd_c = gen("grad", M_TOK, t, "dYdc")                               # t channels, all tokens
    x_c, h_c = gen("act", M_TOK, t, "Xc"), gen("act", M_TOK, t, "Hc")
    R, B128, T = oracle.GRAN_ROW, oracle.GRAN_128x128, oracle.GRAN_1x128
    if barrier is not None:
        barrier.wait(timeout=600)

    def gemm(qa, sa, ga, fa, qb, sb, gb, fb):
        qa, qb = qa[:t], qb[:t]
        sa = sa[:t] if ga != B128 else sa[:1]
        sb = sb[:t] if gb != B128 else sb[:1]
        oracle.gemm_ref_dense(oracle.dequant(qa, sa, ga, fa), oracle.dequant(qb, sb, gb, fb))
        return 2.0 * qa.shape[0] * qb.shape[0] * qa.shape[1]

    t0 = time.perf_counter()
    flop = 0.0
    qx, sx = oracle.quant_token(xs, 0, E4)
    qh, sh = oracle.quant_token(hs, 0, E4)
    for w in (wg_rows, wu_rows):                                       # gate, up fprop
        qw, sw, _, _ = oracle.quant_block128(w, E4)
        flop += gemm(qx, sx, R, E4, qw, sw, B128, E4)
    qw, sw, _, _ = oracle.quant_block128(wd_rows, E4)                   # down fprop
    flop += gemm(qh, sh, R, E4, qw, sw, B128, E4)
    for dy, w in ((dyg, wg_cols), (dyu, wu_cols), (dyd, wd_cols)):      # dgrad
        _, _, qwt, swt = oracle.quant_block128(w, E4, transposed_copy=True)
        qd, sd = oracle.quant_token(dy, 0, E5)
        flop += gemm(qd, sd, R, E5, qwt, swt, B128, E4)
    qxt, sxt = oracle.quant_token(x_c, 128, E4, transpose=True)
    qht, sht = oracle.quant_token(h_c, 128, E4, transpose=True)
    for dyc, (qb, sb) in ((dyg_c, (qxt, sxt)), (dyu_c, (qxt, sxt)), (dyd_c, (qht, sht))):
        qd, sd = oracle.quant_token(dyc, 128, E5, transpose=True)       # wgrad
        flop += gemm(qd, sd, T, E5, qb, sb, T, E4)
    return flop, time.perf_counter() - t0


def _oracle_worker(barrier, queue, steps):
    try:
        queue.put([oracle_sample_step(barrier=barrier) for _ in range(steps)])
    except Exception as e:  # reported by the parent
        queue.put(("error", repr(e)))


def oracle_all_cores(steps: int = 1, skip: int = 0):
    """The oracle sample step in one spawned process per host core, `steps`
    times, every process starting each step's clock together (a barrier).
    Returns (flop of all processes over the last steps - skip steps, the sum
    over those steps of the slowest process's seconds, processes), or None if
    the processes could not be run."""
    import multiprocessing as mp
    import queue as _queue
    import oracle
    oracle.build()
    n = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    if n < 2:
        return None
    ctx = mp.get_context("spawn")
    barrier, q = ctx.Barrier(n), ctx.Queue()
    procs = [ctx.Process(target=_oracle_worker, args=(barrier, q, steps), daemon=True)
             for _ in range(n)]
    for p in procs:
        p.start()
    res = []
    try:
        for _ in range(n):
            res.append(q.get(timeout=900))
    except _queue.Empty:
        res = []
    for p in procs:
        p.join(timeout=60)
        if p.is_alive():
            p.terminate()
    if len(res) != n or any(r[0] == "error" for r in res):
        return None
    flop = sum(r[i][0] for r in res for i in range(skip, steps))
    secs = sum(max(r[i][1] for r in res) for i in range(skip, steps))
    return flop, secs, n


def cpu_baseline_entry():
    """cpu_baseline: the oracle on all host cores (one process per core), with
    the single-thread figure beside it."""
    flop1, secs1 = oracle_sample_step()
    one = {"value": flop1 / secs1 / 1e12, "unit": "TFLOP/s", "cores": 1, "seconds": secs1}
    allc = oracle_all_cores()
    if allc is None:
        return dict(one, kind="oracle", sample=SAMPLE_DESC)
    flop, secs, n = allc
    return {"value": flop / secs / 1e12, "unit": "TFLOP/s", "cores": n, "kind": "oracle",
            "sample": SAMPLE_DESC_ALL.format(n=n), "seconds": secs, "single_thread": one}


SAMPLE_DESC_ALL = ("{n} processes at once (one per host core), each running the oracle (plain C, "
                   "fp64, 1 thread) on a 32x32 block of outputs of each of the step's 9 GEMMs at "
                   "full K, including quantizing the operand slices it needs (whole 128-row "
                   "weight blocks, whole 128-token groups)")

SAMPLE_DESC = ("oracle (plain C, fp64, 1 thread) on a 32x32 block of outputs of each of the "
               "step's 9 GEMMs at full K, including quantizing the operand slices it needs "
               "(whole 128-row weight blocks, whole 128-token groups)")


def run_reference(args):
    """The oracle as it stands on the host cores: one process per core, each
    running the sample step; W untimed steps, then K timed ones."""
    if not replicas.rank_info().is_root:
        return
    allc = oracle_all_cores(args.warmup + args.steps, skip=args.warmup)
    if allc is not None:
        flop, secs, cores = allc
        sample = SAMPLE_DESC_ALL.format(n=cores)
    else:   # processes could not be started: one thread, in this process
        for _ in range(args.warmup):
            oracle_sample_step()
        flop, secs, cores = 0.0, 0.0, 1
        for _ in range(args.steps):
            f, s = oracle_sample_step()
            flop += f
            secs += s
        sample = SAMPLE_DESC
    tf = flop / secs / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": tf, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": "32x32 outputs per GEMM at full K"},
            "cpu_baseline": {"value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": tf, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------- main
def main():
    args = _parse()
    if args.impl == "reference":
        run_reference(args)
        return
    import torch
    import torch.distributed as dist
    import fp8_hybrid_granularity_gb300 as fp8hg
    from fp8_hybrid_granularity_gb300 import workloads

    ri = replicas.rank_info()
    world, rank, local = ri.world, ri.rank, ri.local
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    fp8hg.load_library()
    peaks = _peaks()

    step = Step(torch, fp8hg, workloads, dev, seed_offset=rank)
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(max(args.warmup, 3)):
        step.run()
    assert fp8hg.fp8hg_get_device_error() == 0, "device error during warm-up"
    barrier()

    # ---------------- timed region: K steps, every launch bracketed by events
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.2)
    events = []
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    t_start.record()
    for _ in range(args.steps):
        step.run(events)
    t_end.record()
    barrier()
    clk = clocks.stop()
    ms = t_start.elapsed_time(t_end) / args.steps
    status = fp8hg.fp8hg_get_device_error()
    if status != 0:
        raise RuntimeError(f"device error: {fp8hg.fp8hg_status_str(status)}")
    ms = replicas.max_over_ranks(ms, dist, dev)

    gemm_ms = [a.elapsed_time(b) for k, a, b in events if k == "gemm"]
    per_gemm = [sum(gemm_ms[j::N_GEMM]) / args.steps for j in range(N_GEMM)]
    per_quant = [sum(v[j::N_QUANT]) / args.steps
                 for v in [[a.elapsed_time(b) for k, a, b in events if k == "quant"]]
                 for j in range(N_QUANT)]
    quant_ms = [a.elapsed_time(b) for k, a, b in events if k == "quant"]
    gemm_avg = sum(gemm_ms) / len(gemm_ms)
    quant_step_ms = sum(quant_ms) / args.steps
    value = replicas.job_throughput(world, N_GEMM * GEMM_FLOP, ms)
    gemm_tf = GEMM_FLOP / (gemm_avg * 1e-3) / 1e12
    quant_gbs = step.quant_bytes / (quant_step_ms * 1e-3) / 1e9
    fp8_peak = 2.0 * peaks["bf16_sus"]   # fp8 dense = 2x bf16 dense (nominal ratio)

    # ---------------- end to end: host buffers in, results back, every step
    # Each step's inputs are copied host -> device from pinned memory and all
    # of its outputs device -> host, inside the timed region.  Three device
    # buffer sets let step i+1's inputs arrive and step i-1's outputs leave
    # while step i computes (copy engines and SMs work concurrently); with
    # two sets a step's input copy would wait for the output copy of the
    # step before last, and the chain copy-in -> compute -> copy-out would
    # set the period instead of the copy bandwidth.  Per-tensor events let a
    # launch start once its own inputs have arrived and an output leave as
    # soon as it is final.
    e2e = None
    if not args.no_e2e:
        host_in = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in step.inp.items()}
        for k, v in step.inp.items():
            host_in[k].copy_(v)
        host_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
                    for k, v in step.out.items()}
        n_sets = 3
        sets = [step] + [Step(torch, fp8hg, workloads, dev, seed_offset=rank)
                         for _ in range(n_sets - 1)]
        s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        ke = max(4, min(args.steps, 30))
        for st_ in sets[1:]:
            st_.run()
        barrier()

        def pipelined(nsteps):
            """nsteps end-to-end steps; returns the elapsed milliseconds."""
            freed = [None] * n_sets  # event: buffer set's outputs copied back
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.current_stream().wait_stream(s_in)
            a.record()
            for st_ in (s_in, s_cmp, s_out):
                st_.wait_event(a)
            for i in range(nsteps):
                cur = sets[i % n_sets]
                # inputs in the order the step first reads them, each with its
                # own event; outputs copied back as soon as each is final
                with torch.cuda.stream(s_in):
                    if freed[i % n_sets] is not None:
                        s_in.wait_event(freed[i % n_sets])
                    ready = {}
                    for k in INPUT_ORDER:
                        cur.inp[k].copy_(host_in[k], non_blocking=True)
                        ready[k] = torch.cuda.Event()
                        ready[k].record(s_in)
                with torch.cuda.stream(s_cmp):
                    if freed[i % n_sets] is not None:
                        s_cmp.wait_event(freed[i % n_sets])
                    done = {}
                    cur.run(ready=ready, done=done)
                with torch.cuda.stream(s_out):
                    for k, v in cur.out.items():
                        s_out.wait_event(done[k])
                        host_out[k].copy_(v, non_blocking=True)
                    ev_out = torch.cuda.Event()
                    ev_out.record(s_out)
                    freed[i % n_sets] = ev_out
            cs = torch.cuda.current_stream()
            for st_ in (s_in, s_cmp, s_out):
                cs.wait_stream(st_)
            b.record()
            barrier()
            return a.elapsed_time(b)

        pipelined(max(args.warmup, 3))   # untimed warm-up of the copy pipeline
        e_total = pipelined(ke)
        e_ms = e_total / ke
        e_ms = replicas.max_over_ranks(e_ms, dist, dev)
        e2e = {"value": replicas.job_throughput(world, N_GEMM * GEMM_FLOP, e_ms), "unit": "TFLOP/s",
               "h2d_bytes_per_step": step.in_bytes, "d2h_bytes_per_step": step.out_bytes,
               "ms_per_step": e_ms, "steps": ke,
               "note": ("pinned host buffers; three device buffer sets; each input copied in the "
                        "order the step reads it and each output copied back once final, "
                        "overlapped with compute")}
        del sets

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_entry()

    if rank == 0:
        traffic = _gemm_traffic()
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp8", "data": "synthetic (seeded; Qwen2.5-7B MLP shapes, recipe distributions)",
            "config": {"workload": WORKLOAD, "tokens": M_TOK, "hidden": HID, "mlp": MLP,
                       "gemms_per_step": N_GEMM, "quant_launches_per_step": N_QUANT,
                       "l2": "inputs larger than L2 (each step streams ~15 GB); no flush",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": {"bound": "tensor", "kernel": "k_gemm_wide", "achieved": gemm_tf,
                         "peak": fp8_peak, "unit": "TFLOP/s", "frac": gemm_tf / fp8_peak,
                         "traffic": traffic,
                         "peak_source": f"{peaks['src']} bf16 sustained x2 (nominal fp8/bf16 ratio)",
                         "per_launch_flop": GEMM_FLOP, "avg_launch_ms": gemm_avg},
            "frac_fp8_peak_incl_quant": value / world / fp8_peak,
            "gemm_only_tflops": gemm_tf,
            "quant": {"gbs": quant_gbs, "frac_hbm": quant_gbs / peaks["hbm"],
                      "hbm_peak_gbs": peaks["hbm"], "bytes_per_step": step.quant_bytes,
                      "ms_per_step": quant_step_ms},
            "per_launch_ms": {
                "gemm": dict(zip(GEMM_NAMES, [round(x, 4) for x in per_gemm])),
                "quant": dict(zip(QUANT_NAMES, [round(x, 4) for x in per_quant]))},
            "gpu_launches": (N_GEMM + N_QUANT) * args.steps,
            "clocks": clk,
            "cpu_baseline": cpu,
            "e2e": e2e,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
