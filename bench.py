"""Benchmark of the hybrid-granularity FP8 hot path on GB300.

  python bench.py [--config NAME] [--gpus N] [--steps K] [--warmup W]
                  [--impl reference] [--kernel CASE]

--config (default linear_step_7b, the headline):

  linear_step_7b  one Qwen2.5-7B-shaped MLP block (gate, up, down) at
                  M = 16384 tokens, hidden 3584, MLP width 18944, run through
                  the C ABI:
                    quantize  W_gate, W_up, W_down   128x128 blocks, E4M3 (+ transposed copies),
                                                     one batched launch
                              X, H                   per token, E4M3
                              dY_gate, dY_up, dY_down per token, E5M2
                              X^T, H^T, dY^T (x3)    1x128 groups along tokens (wgrad layout)
                    fprop     Y_g = X W_g^T, Y_u = X W_u^T, Y_d = H W_d^T      (BF16 out)
                    dgrad     dX = dY_g W_g + dY_u W_u (accumulated), dH = dY_d W_d (BF16)
                    wgrad     dW_g = dY_g^T X, dW_u = dY_u^T X, dW_d = dY_d^T H  (FP32 out)
                  6 quantizer launches (both activation layouts from one read
                  each; 11 with --act-quant separate) + 9 GEMM launches per step.
  fprop_1p5b      Qwen2.5-1.5B layer fprop at M = 8192: X, H per token, the
                  gate / up / down / QKV weights in 128x128 blocks (one batched
                  launch, gate and up written into one stacked buffer), three
                  GEMMs: gate and up as one (--gate-up separate: four GEMMs).
  tiny_fprop      X [256 x 512] per token, W [512 x 512] blocks, one GEMM.
  mxfp8_4096      MXFP8: A, B [4096 x 4096] (layer-norm-like and normal rows)
                  quantized in 32-element blocks (clamps counted), C = A B^T.
  sweep           quantizer bandwidth on BF16 [R x 4096], R = 128 * 4^i
                  (1 MB .. 4 GB), per token / 1x128 / 128x128, L2 flushed
                  before every timed launch (and L2-warm up to 64 MB); then
                  the down-projection GEMM at M = 4096, 16384, 65536.

A step's value is its GEMM FLOP over the step time (TFLOP/s with every
quantization pass inside the timed region); the sweep's is the quantizers'
algorithmic bytes over their time (GB/s).  Inputs are seeded synthetic BF16
tensors resident in HBM.  The JSON line carries the roofline of the dominant
kernel against a dense FP8 peak measured in the same run (cuBLAS E4M3 8192^3
through torch._scaled_mm, best single launch), the quantizers' GB/s against the
measured HBM copy rate, an end-to-end figure with host buffers, the SM clocks
seen, and the CPU oracle's rate on a bounded sample of the same work.

--impl reference times the CPU oracle (plain C, fp64) on that bounded sample,
in one process per host core.  --kernel CASE runs one kernel on a small case
(for ncu captures; see KERNEL_CASES).  With --gpus N > 1 and no torchrun
environment, N replicas are started here, one process per local GPU.
"""
from __future__ import annotations

import argparse
import functools
import hashlib
import json
import os
import socket
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from fp8_hybrid_granularity_gb300 import replicas  # noqa: E402

METRIC = "scaled-FP8 GEMM TFLOP/s incl. quant (% FP8 peak); quantizer GB/s (% HBM) at 7B shapes"
CONFIGS = ("linear_step_7b", "fprop_1p5b", "tiny_fprop", "mxfp8_4096", "sweep")
M_TOK, HID, MLP = 16384, 3584, 18944
GEMM_SRC = os.path.join(ROOT, "fp8_hybrid_granularity_gb300", "csrc", "gemm.cu")
TENSOR_FLOP_PER_CYCLE_SM = 16384      # dense FP8 MMA rate of one SM (128x256x32 per 128 cycles)

# DRAM bytes per GEMM launch of the 7B step (dram__bytes_read.sum +
# dram__bytes_write.sum): the mean of one full-size launch of each of the
# step's three GEMM classes (gate-like, down-like, weight gradient; three
# launches each), captured with ncu; valid only for the gemm.cu it was taken
# on; any other source gives traffic null.
GEMM_TRAFFIC = {"gemm_sha256": "049612a6325dec498219e97a8dba1ce109ceac11442ef70db564936bb2264adb",
                "bytes_per_launch": 1.1031e9}


def _parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--config", default="linear_step_7b", choices=CONFIGS)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--launch", default="graph", choices=["eager", "graph"],
                    help="timed steps replayed from one CUDA graph (default), or launched one by one")
    ap.add_argument("--act-quant", default="dual", choices=["dual", "separate"],
                    help="7B step: both activation layouts from one read, or one call each")
    ap.add_argument("--gate-up", default="merged", choices=["merged", "separate"],
                    help="1.5B forward: the gate and up projections as one GEMM over their "
                         "stacked weights, or one GEMM each")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-peak-probe", action="store_true")
    ap.add_argument("--kernel", default=None, help="single-kernel case (see KERNEL_CASES)")
    ap.add_argument("--m", type=int, default=4096, help="tokens of a --kernel case")
    ap.add_argument("--n", type=int, default=HID, help="N of the gemm_shape case")
    ap.add_argument("--k", type=int, default=MLP, help="K of the gemm_shape case")
    ap.add_argument("--split", type=int, default=1,
                    help="K parts of the gemm_shape case (1 = no split, 0 = the library's choice)")
    ap.add_argument("--tile", type=int, default=0,
                    help="GEMM tile of a --kernel case or of every GEMM of a step config "
                         "(0 = the library's choice; see fp8hg_gemm_opts)")
    return ap.parse_args(argv)


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sus=float(p["bf16_tflops_sustained"]), src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def _gemm_traffic():
    sha = hashlib.sha256(open(GEMM_SRC, "rb").read()).hexdigest()
    if GEMM_TRAFFIC["gemm_sha256"] == sha:
        return GEMM_TRAFFIC["bytes_per_launch"]
    return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling while a region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 20):
        self.index, self.period, self.proc, self.lines = index, period_ms, None, []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", str(self.period), "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None
        return self

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


# ------------------------------------------------------------------ steps
class StepBase:
    """Preallocated buffers and the launch sequence of one step of a config.

    Subclasses fill `inp` (BF16 inputs, in the order the step first reads
    them: INPUT_ORDER), `out` (results), `quant_bytes` (algorithmic bytes of
    the quantizer launches), `gemm_flop` (FLOP of each GEMM launch, in launch
    order) and implement `launches(L)`, which enqueues the step through the
    launch helper L."""
    INPUT_ORDER: list = []
    GEMM_NAMES: list = []
    QUANT_NAMES: list = []
    WORKLOAD = ""
    DESC: dict = {}
    TILE = 0      # GEMM tile of every GEMM in the step (0 = the library's choice)

    def __init__(self, torch, f, device):
        self.torch, self.f, self.dev = torch, f, device

    def _sizes(self):
        self.in_bytes = sum(t.numel() * t.element_size() for t in self.inp.values())
        self.out_bytes = sum(t.numel() * t.element_size() for t in self.out.values())
        self.flop = float(sum(self.gemm_flop))

    def run(self, ev=None, ready=None, done=None, external=False, mark=None):
        """Enqueue one step on the current stream.  ev: optional list that
        receives (kind, start_event, end_event) per launch.  ready: optional
        {input name: event}, waited on before the first launch that reads the
        input.  done: optional dict that receives {output name: event},
        recorded after the output's last write.  external: the timing events
        are recorded as event nodes of a graph being captured.  mark:
        optional list that receives one event recorded before the step's
        first GEMM (every step quantizes first, then multiplies)."""
        self.launches(_Launcher(self.torch, ev, ready, done, external, mark))


class _Launcher:
    def __init__(self, torch, ev, ready, done, external=False, mark=None):
        self.torch, self.ev, self.ready, self.done, self.waited = torch, ev, ready, done, set()
        self.ekw = {"enable_timing": True, "external": True} if external else {"enable_timing": True}
        self.mark = mark        # list: receives one event recorded before the first GEMM

    def need(self, *names):
        if self.ready is None:
            return
        for n in names:
            if n not in self.waited:
                self.torch.cuda.current_stream().wait_event(self.ready[n])
                self.waited.add(n)

    def finished(self, *names):
        if self.done is None:
            return
        for n in names:
            e = self.torch.cuda.Event()
            e.record()
            self.done[n] = e

    def timed(self, kind, fn):
        if self.mark is not None and kind == "gemm" and not self.mark:
            e = self.torch.cuda.Event(**self.ekw)
            e.record()
            self.mark.append(e)
        if self.ev is None:
            fn()
            return
        a = self.torch.cuda.Event(**self.ekw)
        b = self.torch.cuda.Event(**self.ekw)
        a.record()
        fn()
        b.record()
        self.ev.append((kind, a, b))


def _tok_bytes(n_el, rows):        # per token: 2 B read + 1 B written + 1 B per row
    return 3.0 * n_el + rows


def _g128_bytes(n_el):             # 1x128 groups (either direction): + 1 B per 128
    return 3.0 * n_el + n_el / 128.0


def _dual_bytes(n_el, rows):        # both layouts from one read: 2 B read + 2 x 1 B written
    return 4.0 * n_el + rows + n_el / 128.0


def _blk_bytes(n_el, transposed):  # 128x128 blocks (+ transposed copy and its scales)
    return (4.0 if transposed else 3.0) * n_el + (2.0 if transposed else 1.0) * n_el / 16384.0


class LinearStep7B(StepBase):
    INPUT_ORDER = ["W_gate", "W_up", "W_down", "X", "H", "dY_gate", "dY_up", "dY_down"]
    GEMM_NAMES = ["fprop_gate", "fprop_up", "fprop_down", "dgrad_gate", "dgrad_up", "dgrad_down",
                  "wgrad_gate", "wgrad_up", "wgrad_down"]
    ACTS = ("X", "H", "dY_gate", "dY_up", "dY_down")
    # dual: each activation's per-token and transposed 1x128 codes from one
    # read (fp8_quant_token_dual); separate: one quantizer call per layout
    # the three weights in one batched launch (fp8_quant_block128_batch)
    QUANT_NAMES_DUAL = ["W_blk_batch", "X_dual", "H_dual", "dYg_dual", "dYu_dual", "dYd_dual"]
    QUANT_NAMES_SEPARATE = ["W_blk_batch", "X_tok", "H_tok", "dYg_tok", "dYu_tok", "dYd_tok",
                            "X_t", "H_t", "dYg_t", "dYu_t", "dYd_t"]
    ACT_QUANT = "dual"
    WORKLOAD = (f"linear_step_7b: Qwen2.5-7B MLP block (gate/up/down) fprop+dgrad+wgrad, "
                f"M={M_TOK} tokens, hidden {HID}, MLP {MLP}; per-token E4M3 activations, "
                f"128x128-block E4M3 weights, per-token E5M2 output grads, 1x128 wgrad re-quant")
    DESC = {"tokens": M_TOK, "hidden": HID, "mlp": MLP}

    def __init__(self, torch, f, workloads, device, seed_offset=0):
        super().__init__(torch, f, device)
        seed = replicas.replica_seed(2, seed_offset)
        T = lambda kind, r, c, name: workloads.make_tensor(kind, r, c, seed, name, device=device)
        self.inp = {
            "X": T("act", M_TOK, HID, "X"), "H": T("act", M_TOK, MLP, "H"),
            "W_gate": T("weight", MLP, HID, "W_gate"), "W_up": T("weight", MLP, HID, "W_up"),
            "W_down": T("weight", HID, MLP, "W_down"),
            "dY_gate": T("grad", M_TOK, MLP, "dY_gate"), "dY_up": T("grad", M_TOK, MLP, "dY_up"),
            "dY_down": T("grad", M_TOK, HID, "dY_down"),
        }
        E4, E5 = f.E4M3, f.E5M2
        at, ab = f.alloc_token, f.alloc_block128
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
        i = self.inp
        self.dual = self.ACT_QUANT == "dual"
        self.QUANT_NAMES = self.QUANT_NAMES_DUAL if self.dual else self.QUANT_NAMES_SEPARATE
        self.ws = f.dual_workspace(M_TOK, MLP, device) if self.dual else None
        qb = sum(_blk_bytes(i[n].numel(), True) for n in ("W_gate", "W_up", "W_down"))
        for n in self.ACTS:
            if self.dual:
                qb += _dual_bytes(i[n].numel(), i[n].shape[0])
            else:
                qb += _tok_bytes(i[n].numel(), i[n].shape[0]) + _g128_bytes(i[n].numel())
        self.quant_bytes = qb
        self.gemm_flop = [2.0 * M_TOK * HID * MLP] * 9
        self._sizes()

    def launches(self, L):
        f, i, o, W = self.f, self.inp, self.out, self.wq
        E4, E5 = f.E4M3, f.E5M2
        wn = ("W_gate", "W_up", "W_down")
        L.need(*wn)
        L.timed("quant", lambda: f.fp8_quant_block128_batch([i[n] for n in wn], E4, True,
                                                            outs=[W[n] for n in wn]))
        tok = {"X": (self.xq, self.xt, E4), "H": (self.hq, self.ht, E4)}
        tok.update({n: (self.dyq[n], self.dyt[n], E5) for n in ("dY_gate", "dY_up", "dY_down")})
        if self.dual:
            for n in self.ACTS:
                q, qt, fmt = tok[n]
                L.need(n)
                L.timed("quant", lambda: f.fp8_quant_token_dual(i[n], fmt, out=q, out_t=qt,
                                                                workspace=self.ws))
        else:
            for n in self.ACTS:
                q, _, fmt = tok[n]
                L.need(n)
                L.timed("quant", lambda: f.fp8_quant_token(i[n], 0, fmt, out=q))
            for n in self.ACTS:
                _, qt, fmt = tok[n]
                L.timed("quant", lambda: f.fp8_quant_token(i[n], 128, fmt, True, out=qt))
        g = functools.partial(f.fp8_gemm_scaled, tile=self.TILE)
        L.timed("gemm", lambda: g(f.FPROP, self.xq, W["W_gate"][0], out=o["Y_gate"]))
        L.finished("Y_gate")
        L.timed("gemm", lambda: g(f.FPROP, self.xq, W["W_up"][0], out=o["Y_up"]))
        L.finished("Y_up")
        L.timed("gemm", lambda: g(f.FPROP, self.hq, W["W_down"][0], out=o["Y_down"]))
        L.finished("Y_down")
        L.timed("gemm", lambda: g(f.DGRAD, self.dyq["dY_gate"], W["W_gate"][1], out=o["dX"]))
        L.timed("gemm", lambda: g(f.DGRAD, self.dyq["dY_up"], W["W_up"][1], out=o["dX"],
                                  accumulate=True))
        L.finished("dX")
        L.timed("gemm", lambda: g(f.DGRAD, self.dyq["dY_down"], W["W_down"][1], out=o["dH"]))
        L.finished("dH")
        L.timed("gemm", lambda: g(f.WGRAD, self.dyt["dY_gate"], self.xt, out=o["dW_gate"]))
        L.finished("dW_gate")
        L.timed("gemm", lambda: g(f.WGRAD, self.dyt["dY_up"], self.xt, out=o["dW_up"]))
        L.finished("dW_up")
        L.timed("gemm", lambda: g(f.WGRAD, self.dyt["dY_down"], self.ht, out=o["dW_down"]))
        L.finished("dW_down")


class FpropStep(StepBase):
    """Forward linears only: activations per token, weights in 128x128 blocks
    (no transposed copy), one BF16 GEMM per weight.  gemms: list of
    (weight name, activation name).  merge: groups of weights applied to the
    same activation (the MLP's gate and up projections) whose codes are
    written into one buffer, one after another, and multiplied by one GEMM
    whose output holds the group's outputs side by side (MERGE = False: one
    GEMM each)."""
    MERGE = True

    def __init__(self, torch, f, workloads, device, workload, gemms, seed_offset=0, merge=()):
        super().__init__(torch, f, device)
        spec = workloads.WORKLOADS[workload]
        seed = replicas.replica_seed(spec["seed"], seed_offset)
        self.inp = {n: workloads.make_tensor(kind, r, c, seed, n, device=device)
                    for (n, kind, r, c) in spec["tensors"]}
        acts = sorted({a for _, a in gemms}, key=[a for _, a in gemms].index)
        weights = [w for w, _ in gemms]
        self.INPUT_ORDER = weights + acts
        E4 = f.E4M3
        self.wq = {w: f.alloc_block128(*self.inp[w].shape, E4, False, device)[0] for w in weights}
        self.aq = {a: f.alloc_token(*self.inp[a].shape, 0, E4, False, device) for a in acts}
        # the B operand of each GEMM: one weight's codes, or a merged group's
        self.bq = dict(self.wq)
        run = list(gemms)
        for group in (merge if self.MERGE else ()):
            a = dict(gemms)[group[0]]
            rows = [self.inp[w].shape[0] for w in group]
            cols = self.inp[group[0]].shape[1]
            both, _ = f.alloc_block128(sum(rows), cols, E4, False, device)
            r0 = 0
            for w, r in zip(group, rows):
                self.wq[w] = f.QTensor(both.codes[r0:r0 + r], both.scale[r0 // 128:(r0 + r) // 128],
                                       E4, f.GRAN_128x128, cols // 128)
                del self.bq[w]
                r0 += r
            name = "+".join(group)
            self.bq[name] = both
            run = [(name, a)] + [(w, x) for w, x in run if w not in group]
        self.gemms = run
        self.out = {f"Y_{w}": torch.empty((self.inp[a].shape[0], self.bq[w].codes.shape[0]),
                                          dtype=torch.bfloat16, device=device) for w, a in run}
        # several weights: one batched launch (fp8_quant_block128_batch)
        self.batch_w = len(weights) > 1
        self.QUANT_NAMES = (["W_blk_batch"] if self.batch_w else [f"{w}_blk" for w in weights]) + \
            [f"{a}_tok" for a in acts]
        self.GEMM_NAMES = [f"fprop_{w}" for w, _ in run]
        self.quant_bytes = (sum(_blk_bytes(self.inp[w].numel(), False) for w in weights) +
                            sum(_tok_bytes(self.inp[a].numel(), self.inp[a].shape[0]) for a in acts))
        self.gemm_flop = [2.0 * self.inp[a].shape[0] * self.bq[w].codes.shape[0] * self.inp[a].shape[1]
                          for w, a in run]
        self._sizes()

    def launches(self, L):
        f, i = self.f, self.inp
        if self.batch_w:
            ws = list(self.wq)
            L.need(*ws)
            L.timed("quant", lambda: f.fp8_quant_block128_batch(
                [i[w] for w in ws], f.E4M3, outs=[(self.wq[w], None) for w in ws]))
        else:
            for w, q in self.wq.items():
                L.need(w)
                L.timed("quant", lambda: f.fp8_quant_block128(i[w], f.E4M3, out=q))
        for a, q in self.aq.items():
            L.need(a)
            L.timed("quant", lambda: f.fp8_quant_token(i[a], 0, f.E4M3, out=q))
        for w, a in self.gemms:
            L.timed("gemm", lambda: f.fp8_gemm_scaled(f.FPROP, self.aq[a], self.bq[w],
                                                      out=self.out[f"Y_{w}"], tile=self.TILE))
            L.finished(f"Y_{w}")


class Fprop1p5B(FpropStep):
    WORKLOAD = ("fprop_1p5b: Qwen2.5-1.5B layer fprop, M=8192 tokens, hidden 1536, MLP 8960, "
                "QKV 2048; per-token E4M3 activations, 128x128-block E4M3 weights, BF16 out; "
                "gate and up projections as one GEMM over their stacked weights")
    DESC = {"tokens": 8192, "hidden": 1536, "mlp": 8960, "qkv": 2048}

    def __init__(self, torch, f, workloads, device, seed_offset=0):
        super().__init__(torch, f, workloads, device, "fprop_1p5b",
                         [("W_gate", "X"), ("W_up", "X"), ("W_down", "H"), ("W_qkv", "X")],
                         seed_offset, merge=(("W_gate", "W_up"),))


class TinyFprop(FpropStep):
    WORKLOAD = ("tiny_fprop: X [256x512] per-token E4M3 (N(0,1), 0.1% outliers x50), "
                "W [512x512] 128x128-block E4M3, Y = X W^T in BF16")
    DESC = {"tokens": 256, "k": 512, "n": 512}

    def __init__(self, torch, f, workloads, device, seed_offset=0):
        super().__init__(torch, f, workloads, device, "tiny_fprop", [("W", "X")], seed_offset)


class Mxfp8Step(StepBase):
    INPUT_ORDER = ["A", "B"]
    GEMM_NAMES = ["mx_gemm"]
    QUANT_NAMES = ["AB_mx32"]
    WORKLOAD = ("mxfp8_4096: A, B [4096x4096] MXFP8 E4M3 (32-element blocks, E8M0 floor scales, "
                "saturating), rows [0,2048) layer-norm-like 1 +- 1e-3, rows [2048,4096) N(0,1); "
                "C = A B^T in BF16; A and B stored as the halves of one [8192x4096] buffer and "
                "quantized by one call")
    DESC = {"m": 4096, "n": 4096, "k": 4096, "block": 32}

    def __init__(self, torch, f, workloads, device, seed_offset=0):
        super().__init__(torch, f, device)
        spec = workloads.WORKLOADS["mxfp8_4096"]
        seed = replicas.replica_seed(spec["seed"], seed_offset)
        # A and B live in the two halves of one [8192 x 4096] buffer and are
        # quantized by one call (each element still every step); the GEMM
        # reads the two halves of the codes and scales
        self.ab = torch.empty((8192, 4096), dtype=torch.bfloat16, device=device)
        self.inp = {"A": self.ab[:4096], "B": self.ab[4096:]}
        for (n, kind, r, c) in spec["tensors"]:
            if n in ("A", "B"):
                self.inp[n].copy_(workloads.make_tensor(kind, r, c, seed, n, device=device))
        self.qab = f.alloc_mx32(8192, 4096, f.E4M3, device)
        self.q = {n: f.QTensor(self.qab.codes[h], self.qab.scale[h], f.E4M3, f.GRAN_MX32, 4096 // 32)
                  for n, h in (("A", slice(0, 4096)), ("B", slice(4096, 8192)))}
        self.clamps = torch.zeros(1, dtype=torch.int64, device=device)
        self.out = {"C": torch.empty((4096, 4096), dtype=torch.bfloat16, device=device)}
        self.quant_bytes = 2 * (3.0 * 4096 * 4096 + 4096 * 4096 / 32.0)
        self.gemm_flop = [2.0 * 4096 ** 3]
        self._sizes()

    def launches(self, L):
        f = self.f
        L.need("A", "B")
        L.timed("quant", lambda: f.fp8_quant_mx32(self.ab, f.E4M3, clamp_count=self.clamps,
                                                  out=self.qab))
        L.timed("gemm", lambda: f.fp8_gemm_scaled(f.FPROP, self.q["A"], self.q["B"],
                                                  out=self.out["C"], tile=self.TILE))
        L.finished("C")


L2_FLUSHED = ("tiny_fprop", "mxfp8_4096")
L2_NOTE = {"linear_step_7b": "inputs larger than L2 (each step streams ~15 GB); no flush",
           "fprop_1p5b": "inputs larger than L2 (each step streams ~0.9 GB); no flush",
           "tiny_fprop": "L2 flushed (512 MB write) before every timed step, outside its timing",
           "mxfp8_4096": "L2 flushed (512 MB write) before every timed step, outside its timing"}
STEPS = {"linear_step_7b": LinearStep7B, "fprop_1p5b": Fprop1p5B, "tiny_fprop": TinyFprop,
         "mxfp8_4096": Mxfp8Step}


# ------------------------------------------------------------ FP8 peak probe
def fp8_peak_probe(torch, dev, n=8192, sustain_s=4.0):
    """Dense FP8 peak of this GPU, measured: cuBLAS E4M3 x E4M3 -> BF16 at
    n^3 through torch._scaled_mm (tensor-wise unit scales).  Burst = best of
    the single launches timed over ~0.4 s (at least 20); sustained =
    back-to-back launches for ~sustain_s
    seconds, with the SM clocks sampled meanwhile.  None if unavailable."""
    try:
        a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        one = torch.ones((), dtype=torch.float32, device=dev)
        f = lambda: torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one,
                                     out_dtype=torch.bfloat16, use_fast_accum=True)
        for _ in range(5):
            f()
        torch.cuda.synchronize()
        flop = 2.0 * n ** 3
        # burst: single launches, each timed alone, for ~0.4 s (at least 20)
        # so that the clock sampler sees the same interval
        clk = ClockSampler(dev.index or 0, period_ms=20).start()
        time.sleep(0.1)
        best, count, t0 = float("inf"), 0, time.perf_counter()
        while count < 20 or time.perf_counter() - t0 < 0.4:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            f()
            e1.record()
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1))
            count += 1
        burst_clk = clk.stop()
        iters = max(10, int(sustain_s * 1e3 / best))
        clk = ClockSampler(dev.index or 0).start()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(iters):
            f()
        e1.record()
        e1.synchronize()
        sus_clk = clk.stop()
        del a, b
        return {"burst_tflops": flop / best / 1e9, "sustained_tflops": flop * iters / e0.elapsed_time(e1) / 1e9,
                "burst_ms": best, "burst_launches": count, "sustained_launches": iters,
                "burst_clocks": burst_clk,
                "sustained_clocks": sus_clk,
                "how": f"cuBLAS E4M3 x E4M3 -> BF16, {n}^3, torch._scaled_mm with tensor-wise unit "
                       f"scales: best of {count} single launches over ~0.4 s (burst) and {iters} "
                       f"back-to-back launches (sustained)"}
    except Exception as e:   # reported in the line; the fallback denominator is used
        return {"error": repr(e)}


def _fp8_peak(peaks, probe):
    """(peak TFLOP/s, source) for kernels timed per launch (the burst case)."""
    if probe and "burst_tflops" in probe:
        return probe["burst_tflops"], ("measured fp8 burst in this run: " + probe["how"])
    return 2.0 * peaks["bf16"], (f"{peaks['src']} bf16 burst x 2 (nominal fp8/bf16 ratio; the fp8 "
                                 f"probe failed: {probe.get('error') if probe else 'not run'})")


# ------------------------------------------------------------ oracle samples
# A GEMM operand of the oracle's bounded sample: (mode, kind, source rows,
# source cols, fmt).  mode tok: rows of the source quantized per token (K =
# source cols); blk: one 128-row block row of the weight; blkT: one 128-column
# block column of the weight, its transposed copy (K = source rows); tokT: t
# columns of the source quantized in 1x128 groups along its rows, transposed
# (K = source rows); mx: rows quantized in 32-element MX blocks.
E4M3_, E5M2_ = 0, 1
SAMPLE_GEMMS = {
    "linear_step_7b": [
        (("tok", "act", M_TOK, HID, E4M3_), ("blk", "weight", MLP, HID, E4M3_)),
        (("tok", "act", M_TOK, HID, E4M3_), ("blk", "weight", MLP, HID, E4M3_)),
        (("tok", "act", M_TOK, MLP, E4M3_), ("blk", "weight", HID, MLP, E4M3_)),
        (("tok", "grad", M_TOK, MLP, E5M2_), ("blkT", "weight", MLP, HID, E4M3_)),
        (("tok", "grad", M_TOK, MLP, E5M2_), ("blkT", "weight", MLP, HID, E4M3_)),
        (("tok", "grad", M_TOK, HID, E5M2_), ("blkT", "weight", HID, MLP, E4M3_)),
        (("tokT", "grad", M_TOK, MLP, E5M2_), ("tokT", "act", M_TOK, HID, E4M3_)),
        (("tokT", "grad", M_TOK, MLP, E5M2_), ("tokT", "act", M_TOK, HID, E4M3_)),
        (("tokT", "grad", M_TOK, HID, E5M2_), ("tokT", "act", M_TOK, MLP, E4M3_)),
    ],
    "fprop_1p5b": [
        (("tok", "act", 8192, 1536, E4M3_), ("blk", "weight", 8960, 1536, E4M3_)),
        (("tok", "act", 8192, 1536, E4M3_), ("blk", "weight", 8960, 1536, E4M3_)),
        (("tok", "act", 8192, 8960, E4M3_), ("blk", "weight", 1536, 8960, E4M3_)),
        (("tok", "act", 8192, 1536, E4M3_), ("blk", "weight", 2048, 1536, E4M3_)),
    ],
    "tiny_fprop": [(("tok", "act_tiny", 256, 512, E4M3_), ("blk", "weight", 512, 512, E4M3_))],
    "mxfp8_4096": [(("mx", "mx_ln", 4096, 4096, E4M3_), ("mx", "mx_ln", 4096, 4096, E4M3_))],
}
# The quantizer passes of a step, sampled: (mode, kind, rows, cols, fmt) with
# the sample's own (rows, cols): per token and MX on a few whole rows, 1x128
# transposed on 128 tokens x a few columns, block128 on one block row.
SAMPLE_QUANTS = {
    "linear_step_7b": [("blkT", "weight", 128, HID, E4M3_), ("blkT", "weight", 128, MLP, E4M3_),
                       ("tok", "act", 16, HID, E4M3_), ("tok", "act", 16, MLP, E4M3_),
                       ("tok", "grad", 16, MLP, E5M2_), ("tokT", "act", 128, 512, E4M3_),
                       ("tokT", "grad", 128, 512, E5M2_)],
    "fprop_1p5b": [("blk", "weight", 128, 1536, E4M3_), ("blk", "weight", 128, 8960, E4M3_),
                   ("tok", "act", 32, 1536, E4M3_), ("tok", "act", 32, 8960, E4M3_)],
    "tiny_fprop": [("blk", "weight", 128, 512, E4M3_), ("tok", "act_tiny", 256, 512, E4M3_)],
    "mxfp8_4096": [("mx", "mx_ln", 64, 4096, E4M3_), ("mx", "mx_ln", 64, 4096, E4M3_)],
    "sweep": [("tok", "act", 64, 4096, E4M3_), ("g128", "act", 64, 4096, E4M3_),
              ("blk", "act", 128, 4096, E4M3_)],
}
SAMPLE_TILE = 32


def _sample_operand(oracle, wl, spec, t, tag):
    mode, kind, rows, cols, fmt = spec
    gen = lambda r, c: wl.bf16_bits(wl.make_tensor(kind, r, c, 2, f"sample-{tag}"))
    if mode == "tok":
        return ("tok", gen(t, cols), fmt)
    if mode == "blk":
        return ("blk", gen(128, cols), fmt)
    if mode == "blkT":
        return ("blkT", gen(rows, 128), fmt)
    if mode == "tokT":
        return ("tokT", gen(rows, t), fmt)
    return ("mx", gen(t, cols), fmt)


def _quantize(oracle, op, t):
    """The oracle's quantization of one sampled operand -> (q, s, gran, fmt)."""
    mode, bits, fmt = op
    if mode == "tok":
        q, s = oracle.quant_token(bits, 0, fmt)
        return q, s, oracle.GRAN_ROW, fmt
    if mode == "blk":
        q, s, _, _ = oracle.quant_block128(bits, fmt)
        return q[:t], s, oracle.GRAN_128x128, fmt
    if mode == "blkT":
        _, _, qt, st = oracle.quant_block128(bits, fmt, transposed_copy=True)
        return qt[:t], st, oracle.GRAN_128x128, fmt
    if mode == "tokT":
        q, s = oracle.quant_token(bits, 128, fmt, transpose=True)
        return q, s, oracle.GRAN_1x128, fmt
    q, s, _ = oracle.quant_mx32(bits, fmt)
    return q, s, oracle.GRAN_MX32, fmt


def oracle_gemm_sample(config, t=SAMPLE_TILE, barrier=None):
    """The oracle on a t x t block of outputs of each GEMM of the config's step
    at full K, including the quantization of the operand slices that block
    needs.  Returns (flop, seconds)."""
    import oracle
    from fp8_hybrid_granularity_gb300 import workloads as wl
    oracle.build()
    ops = [(_sample_operand(oracle, wl, a, t, f"a{j}"), _sample_operand(oracle, wl, b, t, f"b{j}"))
           for j, (a, b) in enumerate(SAMPLE_GEMMS[config])]
    if barrier is not None:
        barrier.wait(timeout=600)
    t0 = time.perf_counter()
    flop = 0.0
    for a, b in ops:
        qa, sa, ga, fa = _quantize(oracle, a, t)
        qb, sb, gb, fb = _quantize(oracle, b, t)
        oracle.gemm_ref_dense(oracle.dequant(qa, sa, ga, fa), oracle.dequant(qb, sb, gb, fb))
        flop += 2.0 * qa.shape[0] * qb.shape[0] * qa.shape[1]
    return flop, time.perf_counter() - t0


def oracle_quant_sample(config, barrier=None):
    """The oracle's quantizers on the config's sampled slices.  Returns
    (algorithmic bytes, seconds): 2 B read + 1 B written per element, + 1 B
    per scale (+ 1 B per element and the scales again for a transposed
    weight copy)."""
    import oracle
    from fp8_hybrid_granularity_gb300 import workloads as wl
    oracle.build()
    xs = [(mode, wl.bf16_bits(wl.make_tensor(kind, r, c, 2, f"qsample-{j}")), fmt)
          for j, (mode, kind, r, c, fmt) in enumerate(SAMPLE_QUANTS[config])]
    if barrier is not None:
        barrier.wait(timeout=600)
    t0 = time.perf_counter()
    nbytes = 0.0
    for mode, x, fmt in xs:
        n = x.size
        if mode == "tok":
            oracle.quant_token(x, 0, fmt)
            nbytes += _tok_bytes(n, x.shape[0])
        elif mode == "g128":
            oracle.quant_token(x, 128, fmt)
            nbytes += _g128_bytes(n)
        elif mode == "tokT":
            oracle.quant_token(x, 128, fmt, transpose=True)
            nbytes += _g128_bytes(n)
        elif mode in ("blk", "blkT"):
            oracle.quant_block128(x, fmt, transposed_copy=mode == "blkT")
            nbytes += _blk_bytes(n, mode == "blkT")
        else:
            oracle.quant_mx32(x, fmt)
            nbytes += 3.0 * n + n / 32.0
    return nbytes, time.perf_counter() - t0


def _oracle_worker(barrier, queue, steps, config):
    try:
        res = []
        for _ in range(steps):
            g = oracle_gemm_sample(config, barrier=barrier) if config in SAMPLE_GEMMS else (0.0, 0.0)
            q = oracle_quant_sample(config, barrier=barrier)
            res.append((g, q))
        queue.put(res)
    except Exception as e:  # reported by the parent
        queue.put(("error", repr(e)))


def _host_cores():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def oracle_all_cores(config, steps=1, skip=0):
    """The config's oracle samples in one spawned process per host core,
    `steps` times, every process starting each timed phase together (a
    barrier).  Returns {"gemm": (flop, s), "quant": (bytes, s), "cores": n},
    totals over all processes for the last steps - skip steps with the
    slowest process's seconds, or None if the processes could not be run."""
    import multiprocessing as mp
    import queue as _queue
    import oracle
    oracle.build()
    n = _host_cores()
    if n < 2:
        return None
    ctx = mp.get_context("spawn")
    barrier, q = ctx.Barrier(n), ctx.Queue()
    procs = [ctx.Process(target=_oracle_worker, args=(barrier, q, steps, config), daemon=True)
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
    out = {"cores": n}
    for k, name in ((0, "gemm"), (1, "quant")):
        work = sum(r[i][k][0] for r in res for i in range(skip, steps))
        secs = sum(max(r[i][k][1] for r in res) for i in range(skip, steps))
        out[name] = (work, secs)
    return out


def _sample_desc(config, cores):
    who = f"{cores} processes at once (one per host core)" if cores > 1 else "one process"
    gem = (f"a {SAMPLE_TILE}x{SAMPLE_TILE} block of outputs of each of the step's "
           f"{len(SAMPLE_GEMMS[config])} GEMMs at full K, including quantizing the operand slices "
           f"it needs" if config in SAMPLE_GEMMS else "no GEMM")
    qs = ", ".join(f"{m} {r}x{c}" for (m, _, r, c, _) in SAMPLE_QUANTS[config])
    return (f"{who}, each running the oracle (plain C, fp64, 1 thread) on {gem}; quantizers on "
            f"slices of the step's tensors: {qs}")


def cpu_baseline_entry(config):
    """cpu_baseline: the oracle on all host cores (one process per core), with
    the single-thread figures beside it.  value: GEMM sample TFLOP/s (sweep:
    quantizer GB/s)."""
    one_q = oracle_quant_sample(config)
    one = {"quant_gbs": one_q[0] / one_q[1] / 1e9, "quant_seconds": one_q[1]}
    if config in SAMPLE_GEMMS:
        one_g = oracle_gemm_sample(config)
        one.update(value=one_g[0] / one_g[1] / 1e12, unit="TFLOP/s", seconds=one_g[1])
    allc = oracle_all_cores(config)
    if allc is None:
        v = one.get("value", one["quant_gbs"])
        return {"value": v, "unit": "TFLOP/s" if config in SAMPLE_GEMMS else "GB/s", "cores": 1,
                "kind": "oracle", "sample": _sample_desc(config, 1),
                "quant": {"gbs": one["quant_gbs"], "cores": 1}}
    qb, qs = allc["quant"]
    quant = {"gbs": qb / qs / 1e9, "cores": allc["cores"], "single_thread_gbs": one["quant_gbs"]}
    if config in SAMPLE_GEMMS:
        gf, gs = allc["gemm"]
        return {"value": gf / gs / 1e12, "unit": "TFLOP/s", "cores": allc["cores"],
                "kind": "oracle", "sample": _sample_desc(config, allc["cores"]),
                "single_thread": {"value": one["value"], "unit": "TFLOP/s", "cores": 1},
                "quant": quant}
    return {"value": quant["gbs"], "unit": "GB/s", "cores": allc["cores"], "kind": "oracle",
            "sample": _sample_desc(config, allc["cores"]),
            "single_thread": {"value": one["quant_gbs"], "unit": "GB/s", "cores": 1}, "quant": quant}


def run_reference(args):
    """The oracle as it stands on the host cores: one process per core, each
    running the config's sample step; W untimed steps, then K timed ones."""
    if not replicas.rank_info().is_root:
        return
    cfg = args.config
    gemm = cfg in SAMPLE_GEMMS
    allc = oracle_all_cores(cfg, args.warmup + args.steps, skip=args.warmup)
    if allc is not None:
        work, secs = allc["gemm"] if gemm else allc["quant"]
        cores = allc["cores"]
    else:   # processes could not be started: one thread, in this process
        for _ in range(args.warmup):
            oracle_gemm_sample(cfg) if gemm else oracle_quant_sample(cfg)
        work = secs = 0.0
        for _ in range(args.steps):
            w, s = oracle_gemm_sample(cfg) if gemm else oracle_quant_sample(cfg)
            work += w
            secs += s
        cores = 1
    value = work / secs / (1e12 if gemm else 1e9)
    unit = "TFLOP/s" if gemm else "GB/s"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg, "sample": _sample_desc(cfg, cores)},
            "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                             "sample": _sample_desc(cfg, cores)},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# -------------------------------------------------------- replica launcher
def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def spawn_replicas(n, argv, script=None, env=None):
    """Start `n` copies of `script` (this file by default) as ranks 0..n-1 of
    one job on this node, the way torch.distributed.run would: RANK,
    LOCAL_RANK, WORLD_SIZE, LOCAL_WORLD_SIZE, MASTER_ADDR = 127.0.0.1 and a
    free MASTER_PORT in each process's environment.  Each rank uses the GPU
    of its local rank; only rank 0 prints.  Returns the first non-zero exit
    code, or 0."""
    script = script or os.path.abspath(__file__)
    port = _free_port()
    base = dict(os.environ if env is None else env)
    procs = []
    for r in range(n):
        e = dict(base, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(n),
                 LOCAL_WORLD_SIZE=str(n), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, script] + list(argv), env=e))
    # A rank that fails would leave the others waiting in a collective: once
    # any rank exits non-zero, the remaining ones are stopped.
    rc = 0
    while None in [p.poll() for p in procs]:      # poll every rank each pass
        failed = [p.returncode for p in procs if p.returncode not in (None, 0)]
        if failed:
            rc = failed[0]
            for p in procs:
                if p.poll() is None:
                    p.terminate()
            for p in procs:
                try:
                    p.wait(timeout=30)
                except subprocess.TimeoutExpired:
                    p.kill()
            break
        time.sleep(0.1)
    for p in procs:
        rc = rc or (p.wait() or 0)
    return rc


# ------------------------------------------------------------- GPU arm
def _pipelined_e2e(torch, make_step, step, nsets, nsteps_warm, nsteps, barrier):
    """End to end: every step's inputs copied host -> device from pinned
    memory and all of its outputs device -> host, inside the timed region.
    `nsets` device buffer sets let step i+1's inputs arrive and step i-1's
    outputs leave while step i computes (copy engines and SMs work
    concurrently); per-tensor events let a launch start once its own inputs
    have arrived and an output leave as soon as it is final.  Returns the
    mean milliseconds per step."""
    host_in = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in step.inp.items()}
    for k, v in step.inp.items():
        host_in[k].copy_(v)
    host_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in step.out.items()}
    sets = [step] + [make_step() for _ in range(nsets - 1)]
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    for st_ in sets[1:]:
        st_.run()
    barrier()

    def pipelined(n):
        freed = [None] * nsets
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.current_stream().wait_stream(s_in)
        a.record()
        for st_ in (s_in, s_cmp, s_out):
            st_.wait_event(a)
        for i in range(n):
            cur = sets[i % nsets]
            with torch.cuda.stream(s_in):
                if freed[i % nsets] is not None:
                    s_in.wait_event(freed[i % nsets])
                ready = {}
                for k in cur.INPUT_ORDER:
                    cur.inp[k].copy_(host_in[k], non_blocking=True)
                    ready[k] = torch.cuda.Event()
                    ready[k].record(s_in)
            with torch.cuda.stream(s_cmp):
                if freed[i % nsets] is not None:
                    s_cmp.wait_event(freed[i % nsets])
                done = {}
                cur.run(ready=ready, done=done)
            with torch.cuda.stream(s_out):
                for k, v in cur.out.items():
                    s_out.wait_event(done[k])
                    host_out[k].copy_(v, non_blocking=True)
                ev_out = torch.cuda.Event()
                ev_out.record(s_out)
                freed[i % nsets] = ev_out
        cs = torch.cuda.current_stream()
        for st_ in (s_in, s_cmp, s_out):
            cs.wait_stream(st_)
        b.record()
        barrier()
        return a.elapsed_time(b)

    pipelined(nsteps_warm)
    ms = pipelined(nsteps) / nsteps
    del sets
    return ms


def host_link_probe(torch, dev, nbytes=1 << 30, reps=3):
    """Copy rates between pinned host memory and the device on this machine: host
    -> device alone, device -> host alone, and both at once (half the bytes
    each way on two streams), best of `reps`, GB/s."""
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    h.fill_(1)
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    rates = {}
    for name in ("h2d", "d2h", "both"):
        best = float("inf")
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            if name == "h2d":
                d.copy_(h, non_blocking=True)
            elif name == "d2h":
                h.copy_(d, non_blocking=True)
            else:
                half = nbytes // 2
                for st_ in (s1, s2):
                    st_.wait_event(a)
                with torch.cuda.stream(s1):
                    d[:half].copy_(h[:half], non_blocking=True)
                with torch.cuda.stream(s2):
                    h[half:].copy_(d[half:], non_blocking=True)
                torch.cuda.current_stream().wait_stream(s1)
                torch.cuda.current_stream().wait_stream(s2)
            b.record()
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b))
        rates[name] = nbytes / (best * 1e-3) / 1e9
    del h, d
    return rates


def link_floor_ms(in_bytes, out_bytes, rates):
    """Lower bound on a step whose inputs cross the host link in and whose
    outputs cross it out: each direction at its own rate, and all bytes at
    the rate of both directions together."""
    return 1e3 * max(in_bytes / (rates["h2d"] * 1e9), out_bytes / (rates["d2h"] * 1e9),
                     (in_bytes + out_bytes) / (rates["both"] * 1e9))


def run_step_config(args, torch, dist, fp8hg, workloads, ri, dev, peaks):
    world, rank = ri.world, ri.rank
    cls = STEPS[args.config]
    if hasattr(cls, "ACT_QUANT"):
        cls.ACT_QUANT = args.act_quant
    if hasattr(cls, "MERGE"):
        cls.MERGE = args.gate_up == "merged"
    cls.TILE = args.tile
    step = cls(torch, fp8hg, workloads, dev, seed_offset=rank)
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(max(args.warmup, 3)):
        step.run()
    if fp8hg.fp8hg_get_device_error() != 0:
        raise RuntimeError("device error during warm-up")
    barrier()

    # ---------------- timed region: K steps as a user runs them, with three
    # events per step (start, before the first GEMM, end): an event pair
    # around every launch would cost the small configs 7-40 % (each record
    # orders the stream, so a launch can no longer start while the one before
    # drains).  The quantizers' time and the GEMMs' mean launch time come from
    # these marks; the per-launch breakdown from an instrumented pass after.
    # Steps whose tensors fit in L2 (tiny, MX) are each preceded by a 512 MB
    # write that flushes L2, outside the step's events.
    flush = (torch.empty(512 * 2 ** 20 // 4, dtype=torch.float32, device=dev)
             if args.config in L2_FLUSHED else None)

    def enqueue_timed(per_step, external):
        for _ in range(args.steps):
            if flush is not None:
                flush.fill_(1.0)
            a = torch.cuda.Event(enable_timing=True, external=external)
            b = torch.cuda.Event(enable_timing=True, external=external)
            mark = []
            a.record()
            step.run(external=external, mark=mark)
            b.record()
            per_step.append((a, mark[0], b))

    # Graph launch: the K timed steps are captured once, with the events as
    # event nodes, and the timed region is one replay.
    launch = args.launch
    graph = None
    if launch == "graph":
        try:
            per_step = []
            graph = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.graph(graph, stream=side):
                enqueue_timed(per_step, True)
            graph.replay()                      # untimed: uploads the graph
            barrier()
        except (TypeError, RuntimeError) as e:  # no external events in this torch
            graph, launch = None, f"eager (graph capture failed: {type(e).__name__})"
    if graph is None:
        per_step = []
    clocks = ClockSampler(ri.local).start()
    time.sleep(0.2)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    t_start.record()
    if graph is not None:
        graph.replay()
    else:
        enqueue_timed(per_step, False)
    t_end.record()
    barrier()
    if flush is None:
        ms = t_start.elapsed_time(t_end) / args.steps
    else:
        ms = sum(a.elapsed_time(b) for a, _, b in per_step) / args.steps
    clk = clocks.stop()
    status = fp8hg.fp8hg_get_device_error()
    if status != 0:
        raise RuntimeError(f"device error: {fp8hg.fp8hg_status_str(status)}")
    ms = replicas.max_over_ranks(ms, dist, dev)

    ng, nq = len(step.GEMM_NAMES), len(step.QUANT_NAMES)
    quant_step_ms = sum(a.elapsed_time(m) for a, m, _ in per_step) / args.steps
    gemm_step_ms = sum(m.elapsed_time(b) for _, m, b in per_step) / args.steps
    value = replicas.job_throughput(world, step.flop, ms)
    gemm_tf = step.flop / (gemm_step_ms * 1e-3) / 1e12
    quant_gbs = step.quant_bytes / (quant_step_ms * 1e-3) / 1e9

    # per-launch breakdown: an instrumented pass (an event pair around every
    # launch), outside the timed region
    events = []
    n_inst = max(1, min(args.steps, 10))
    for _ in range(n_inst):
        if flush is not None:
            flush.fill_(1.0)
        step.run(events)
    torch.cuda.synchronize()
    del flush
    gemm_ms = [a.elapsed_time(b) for k, a, b in events if k == "gemm"]
    quant_ms = [a.elapsed_time(b) for k, a, b in events if k == "quant"]
    per_gemm = [sum(gemm_ms[j::ng]) / n_inst for j in range(ng)]
    per_quant = [sum(quant_ms[j::nq]) / n_inst for j in range(nq)]

    e2e = None
    if not args.no_e2e:
        make = lambda: cls(torch, fp8hg, workloads, dev, seed_offset=rank)
        n_e2e = max(4, min(args.steps, 30))
        e_ms = _pipelined_e2e(torch, make, step, 3, max(args.warmup, 3), n_e2e, barrier)
        e_ms = replicas.max_over_ranks(e_ms, dist, dev)
        link = host_link_probe(torch, dev)
        floor = link_floor_ms(step.in_bytes, step.out_bytes, link)
        e2e = {"value": replicas.job_throughput(world, step.flop, e_ms), "unit": "TFLOP/s",
               "h2d_bytes_per_step": step.in_bytes, "d2h_bytes_per_step": step.out_bytes,
               "ms_per_step": e_ms, "steps": n_e2e,
               "host_link_gbs": {k: round(v, 1) for k, v in link.items()},
               "link_floor_ms": floor, "frac_of_link_floor": floor / e_ms,
               "note": ("pinned host buffers; three device buffer sets; each input copied in the "
                        "order the step reads it and each output copied back once final, "
                        "overlapped with compute")}

    probe = None
    if rank == 0 and not args.no_peak_probe:
        probe = fp8_peak_probe(torch, dev)
    barrier()
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_entry(args.config)
    if rank != 0:
        return None

    fp8_peak, peak_src = _fp8_peak(peaks, probe)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = clk.get("sm_mhz")
    at_clock = TENSOR_FLOP_PER_CYCLE_SM * sms * mhz * 1e6 / 1e12 if mhz else None
    gemm_kernel = {1: "k_gemm_mxf8", 2: "k_gemm_wide", 3: "k_gemm_pair"}.get(
        cls.TILE, "k_gemm_wide" if args.config == "linear_step_7b" else
        "fp8_gemm_scaled (k_gemm_wide or k_gemm_mxf8 by the library's tile rule)")
    return {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8", "data": "synthetic (seeded; recipe distributions)",
        "config": dict({"workload": cls.WORKLOAD, "name": args.config,
                        "gemms_per_step": ng, "quant_launches_per_step": nq,
                        "l2": L2_NOTE[args.config], "launch": launch,
                        "act_quant": getattr(cls, "ACT_QUANT", None), "gemm_tile": cls.TILE,
                        "gate_up": (("merged" if cls.MERGE else "separate")
                                    if args.config == "fprop_1p5b" else None),
                        "parallelism": "replicas" if world > 1 else "single GPU"}, **cls.DESC),
        "roofline": {"bound": "tensor", "kernel": gemm_kernel, "achieved": gemm_tf,
                     "peak": fp8_peak, "unit": "TFLOP/s", "frac": gemm_tf / fp8_peak,
                     "traffic": (_gemm_traffic() if args.config == "linear_step_7b" and cls.TILE in (0, 2)
                                 else None),
                     "peak_source": peak_src,
                     "per_launch_flop": step.flop / ng, "avg_launch_ms": gemm_step_ms / ng,
                     "timing": ("GEMM phase of every timed step (first GEMM to step end, "
                                "CUDA events on the launching stream) / GEMMs per step"),
                     "clock_normalised": {"sm_mhz": mhz, "sms": sms,
                                          "flop_per_cycle_sm": TENSOR_FLOP_PER_CYCLE_SM,
                                          "peak_at_clock": at_clock,
                                          "frac": gemm_tf / at_clock if at_clock else None},
                     "bf16x2": {"peak": 2.0 * peaks["bf16"], "frac": gemm_tf / (2.0 * peaks["bf16"]),
                                "source": f"{peaks['src']} bf16 burst x 2 (nominal ratio)"}},
        "frac_fp8_peak_incl_quant": value / world / fp8_peak,
        "gemm_only_tflops": gemm_tf,
        "quant": {"gbs": quant_gbs, "frac_hbm": quant_gbs / peaks["hbm"],
                  "hbm_peak_gbs": peaks["hbm"], "bytes_per_step": step.quant_bytes,
                  "ms_per_step": quant_step_ms,
                  "bytes_counted": ("dual activation quantizer: 2 B read + 2 B written per "
                                    "element (both layouts from one read); block weights: "
                                    "3-4 B per element; + scales"
                                    if getattr(step, "dual", False) else
                                    "per call: 2 B read + 1 B written per element + scales")},
        "per_launch_ms": {"gemm": dict(zip(step.GEMM_NAMES, [round(x, 4) for x in per_gemm])),
                          "quant": dict(zip(step.QUANT_NAMES, [round(x, 4) for x in per_quant])),
                          "note": (f"instrumented pass of {n_inst} steps after the timed region "
                                   "(an event pair around every launch); the timed region "
                                   "records only step start, first GEMM and step end")},
        "gpu_launches": (ng + nq) * args.steps,
        "clocks": clk,
        "fp8_peak_probe": probe,
        "cpu_baseline": cpu,
        "e2e": e2e,
    }


# ------------------------------------------------------------------ sweep
SWEEP_ROWS = [128 * 4 ** i for i in range(7)]       # [R x 4096] BF16: 1 MB .. 4 GB
SWEEP_GEMM_M = [4096, 16384, 65536]


def run_sweep(args, torch, dist, fp8hg, workloads, ri, dev, peaks):
    """Quantizer bandwidth over tensor sizes (L2 flushed before each timed
    launch, and L2-warm for tensors up to 64 MB), then the down-projection
    GEMM at three token counts.  value = the quantizers' algorithmic bytes
    over their time at every flushed point (GB/s)."""
    world, rank = ri.world, ri.rank
    E4 = fp8hg.E4M3
    flush = torch.empty(512 * 2 ** 20 // 4, dtype=torch.float32, device=dev)   # 512 MB > L2
    reps = max(args.steps, 3)

    def timed(fn, flush_l2):
        for _ in range(max(args.warmup, 3)):
            fn()
        ts = []
        for _ in range(reps):
            if flush_l2:
                flush.fill_(1.0)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    clocks = ClockSampler(ri.local).start()
    points, tot_bytes, tot_ms = [], 0.0, 0.0
    big = None
    for R in SWEEP_ROWS:
        x = workloads.make_tensor("act", R, 4096, replicas.replica_seed(4, rank), f"sweep{R}",
                                  device=dev)
        n = x.numel()
        q_tok = fp8hg.alloc_token(R, 4096, 0, E4, False, dev)
        q_128 = fp8hg.alloc_token(R, 4096, 128, E4, False, dev)
        q_blk, _ = fp8hg.alloc_block128(R, 4096, E4, False, dev)
        cases = [("token", lambda: fp8hg.fp8_quant_token(x, 0, E4, out=q_tok), _tok_bytes(n, R)),
                 ("1x128", lambda: fp8hg.fp8_quant_token(x, 128, E4, out=q_128), _g128_bytes(n)),
                 ("128x128", lambda: fp8hg.fp8_quant_block128(x, E4, out=q_blk),
                  _blk_bytes(n, False))]
        for gran, fn, nbytes in cases:
            ms = timed(fn, True)
            p = {"bytes_in": 2 * n, "gran": gran, "ms": ms, "gbs": nbytes / ms / 1e6,
                 "frac_hbm": nbytes / ms / 1e6 / peaks["hbm"], "l2": "flushed"}
            if 2 * n <= 64 * 2 ** 20:
                ms_w = timed(fn, False)
                p["l2_warm"] = {"ms": ms_w, "gbs": nbytes / ms_w / 1e6}
            points.append(p)
            tot_bytes += nbytes
            tot_ms += ms
            if R == SWEEP_ROWS[-1] and gran == "token":
                big = p
        del x, q_tok, q_128, q_blk
        torch.cuda.empty_cache()
    gemm_points = []
    w = workloads.make_tensor("weight", HID, MLP, replicas.replica_seed(4, rank), "W_down", device=dev)
    wq = fp8hg.fp8_quant_block128(w, E4)
    del w
    for M in SWEEP_GEMM_M:
        h = workloads.make_tensor("act", M, MLP, replicas.replica_seed(4, rank), "H", device=dev)
        hq = fp8hg.fp8_quant_token(h, 0, E4)
        del h
        y = torch.empty((M, HID), dtype=torch.bfloat16, device=dev)
        ms = timed(lambda: fp8hg.fp8_gemm_scaled(fp8hg.FPROP, hq, wq, out=y), M <= 16384)
        gemm_points.append({"m": M, "k": MLP, "n": HID, "ms": ms,
                            "tflops": 2.0 * M * HID * MLP / ms / 1e9})
        del hq, y
        torch.cuda.empty_cache()
    clk = clocks.stop()
    if fp8hg.fp8hg_get_device_error() != 0:
        raise RuntimeError("device error in the sweep")
    gbs = tot_bytes / tot_ms / 1e6
    gbs = replicas.max_over_ranks(-gbs, dist, dev) * -1.0      # slowest rank
    # end to end: the 1 GB per-token point with the input copied in from
    # pinned host memory and the codes and scales copied back, every launch
    e2e = None
    if not args.no_e2e:
        R = 131072
        xh = workloads.make_tensor("act", R, 4096, 4, "sweep-e2e").pin_memory()
        xd = torch.empty_like(xh, device=dev)
        qd = fp8hg.alloc_token(R, 4096, 0, E4, False, dev)
        qh = torch.empty(qd.codes.shape, dtype=torch.uint8, pin_memory=True)
        sh = torch.empty(qd.scale.shape, dtype=torch.uint8, pin_memory=True)

        def e2e_step():
            xd.copy_(xh, non_blocking=True)
            fp8hg.fp8_quant_token(xd, 0, E4, out=qd)
            qh.copy_(qd.codes, non_blocking=True)
            sh.copy_(qd.scale, non_blocking=True)
        ms = timed(e2e_step, False)
        nb = _tok_bytes(R * 4096, R)
        e2e = {"value": nb / ms / 1e6, "unit": "GB/s", "h2d_bytes_per_step": xh.numel() * 2,
               "d2h_bytes_per_step": qh.numel() + sh.numel(), "ms_per_step": ms,
               "note": "per-token quantizer on [131072 x 4096] BF16 (1 GB), input copied in "
                       "and codes + scales copied back every launch (serial, one stream)"}
        del xh, xd, qd, qh, sh
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_entry("sweep")
    if rank != 0:
        return None
    return {
        "metric": METRIC, "value": gbs * world, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp8",
        "data": "synthetic (seeded; activation distribution of the 1.5B/7B configs)",
        "config": {"workload": "sweep: quantizers on BF16 [R x 4096], R = 128*4^i (1 MB..4 GB), "
                               "per token / 1x128 / 128x128; fprop down GEMM at M = 4096, 16384, "
                               "65536 (K = 18944, N = 3584)",
                   "name": "sweep", "l2": "flushed (512 MB write) before every timed quantizer "
                                          "launch; L2-warm also reported up to 64 MB",
                   "reps_per_point": reps, "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "kernel": "k_quant_row (per token, 4 GB)",
                     "achieved": big["gbs"], "peak": peaks["hbm"], "unit": "GB/s",
                     "frac": big["gbs"] / peaks["hbm"], "traffic": None,
                     "peak_source": f"{peaks['src']} HBM copy (MEASURED_PEAKS.json)",
                     "per_launch_bytes": _tok_bytes(SWEEP_ROWS[-1] * 4096, SWEEP_ROWS[-1]),
                     "avg_launch_ms": big["ms"]},
        "points": points, "gemm_points": gemm_points,
        "gpu_launches": len(points) * reps + len(gemm_points) * reps,
        "clocks": clk, "cpu_baseline": cpu, "e2e": e2e,
    }


# -------------------------------------------------------- single kernels
KERNEL_CASES = {
    "gemm_down": "fprop down projection: A = H [M, 18944] per token, B = W_down [3584, 18944] "
                 "128x128 blocks, BF16 out",
    "gemm_gate": "fprop gate projection: A = X [M, 3584] per token, B = W_gate [18944, 3584], BF16",
    "gemm_gate_q": "the gate projection with the output quantized in the epilogue (E4M3, 1x128)",
    "wgrad": "gate weight gradient: A = dY^T [18944, M] 1x128 E5M2, B = X^T [3584, M] 1x128, FP32",
    "gemm_shape": "fprop on A [M, --k] per token x B [--n, --k] 128x128 blocks, BF16 out",
    "gemm_mx": "MXFP8 x MXFP8: A [M, 4096] (layer-norm-like and normal rows), B [4096, 4096]",
    "gemm_f32s": "the down projection with FP32 scales (promotion GEMM)",
    "quant_row": "per-token quantization of H [M, 18944]",
    "quant_1x128": "1x128 quantization of H [M, 18944]",
    "quant_t": "1x128-along-tokens transposed quantization of H [M, 18944]",
    "quant_dual": "both quantizations of H [M, 18944] (per token, 1x128 along tokens "
                  "transposed) from one read",
    "block128": "128x128 quantization (+ transposed copy) of W_down [3584, 18944]",
    "mx32": "MXFP8 quantization of [M, 4096]",
    "mx32_mon": "MXFP8 quantization of [M, 4096] with the clamp monitor's counts",
    "requant": "stored per-token FP8 codes of H [M, 18944] -> 1x128 along tokens, transposed",
}


def run_kernel_case(args):
    """One kernel, W untimed and K timed launches on a small case; prints the
    mean launch time (CUDA events).  Meant for ncu captures."""
    import torch
    import fp8_hybrid_granularity_gb300 as fp8hg
    from fp8_hybrid_granularity_gb300 import workloads
    if args.kernel not in KERNEL_CASES:
        raise SystemExit(f"unknown --kernel {args.kernel}; one of {sorted(KERNEL_CASES)}")
    fp8hg.load_library()
    dev = torch.device("cuda", 0)
    M, c = args.m, args.kernel
    mk = lambda kind, r, cc, n: workloads.make_tensor(kind, r, cc, 4, n, device=dev)
    E4, E5 = fp8hg.E4M3, fp8hg.E5M2
    bf = torch.bfloat16
    if c in ("gemm_down", "gemm_f32s"):
        h, w = mk("act", M, MLP, "H"), mk("weight", HID, MLP, "W_down")
        y = torch.empty((M, HID), dtype=bf, device=dev)
        if c == "gemm_down":
            a, b = fp8hg.fp8_quant_token(h, 0, E4), fp8hg.fp8_quant_block128(w, E4)
            fn = lambda: fp8hg.fp8_gemm_scaled(fp8hg.FPROP, a, b, out=y, tile=args.tile)
        else:
            a, b = fp8hg.fp8_quant_token_f32s(h, 0, E4), fp8hg.fp8_quant_block128_f32s(w, E4)
            fn = lambda: fp8hg.fp8_gemm_scaled_f32s(fp8hg.FPROP, a, b, out=y)
        work, unit = 2.0 * M * HID * MLP, "flop"
    elif c in ("gemm_gate", "gemm_gate_q"):
        x, w = mk("act", M, HID, "X"), mk("weight", MLP, HID, "W_gate")
        a, b = fp8hg.fp8_quant_token(x, 0, E4), fp8hg.fp8_quant_block128(w, E4)
        if c == "gemm_gate":
            y = torch.empty((M, MLP), dtype=bf, device=dev)
            fn = lambda: fp8hg.fp8_gemm_scaled(fp8hg.FPROP, a, b, out=y, tile=args.tile)
        else:
            yq = fp8hg.alloc_token(M, MLP, 128, E4, False, dev)
            fn = lambda: fp8hg.fp8_gemm_scaled_q(fp8hg.FPROP, a, b, E4, out=yq)
        work, unit = 2.0 * M * HID * MLP, "flop"
    elif c == "wgrad":
        dy, x = mk("grad", M, MLP, "dY"), mk("act", M, HID, "X")
        a, b = fp8hg.fp8_quant_token(dy, 128, E5, True), fp8hg.fp8_quant_token(x, 128, E4, True)
        y = torch.empty((MLP, HID), dtype=torch.float32, device=dev)
        fn = lambda: fp8hg.fp8_gemm_scaled(fp8hg.WGRAD, a, b, out=y, tile=args.tile)
        work, unit = 2.0 * M * HID * MLP, "flop"
    elif c == "gemm_shape":
        x, w = mk("act", M, args.k, "X"), mk("weight", args.n, args.k, "W")
        a, b = fp8hg.fp8_quant_token(x, 0, E4), fp8hg.fp8_quant_block128(w, E4)
        y = torch.empty((M, args.n), dtype=bf, device=dev)
        if args.split == 1:
            fn = lambda: fp8hg.fp8_gemm_scaled(fp8hg.FPROP, a, b, out=y, tile=args.tile)
        else:
            ws = fp8hg.splitk_workspace(M, args.n, args.k, args.split, dev)
            fn = lambda: fp8hg.fp8_gemm_scaled_splitk(fp8hg.FPROP, a, b, out=y, split_k=args.split,
                                                      workspace=ws, tile=args.tile)
        work, unit = 2.0 * M * args.n * args.k, "flop"
    elif c == "gemm_mx":
        xa, xb = mk("mx_ln", M, 4096, "A"), mk("mx_ln", 4096, 4096, "B")
        a, b = fp8hg.fp8_quant_mx32(xa, E4), fp8hg.fp8_quant_mx32(xb, E4)
        y = torch.empty((M, 4096), dtype=bf, device=dev)
        fn = lambda: fp8hg.fp8_gemm_scaled(fp8hg.FPROP, a, b, out=y, tile=args.tile)
        work, unit = 2.0 * M * 4096 * 4096, "flop"
    elif c == "quant_dual":
        h = mk("act", M, MLP, "H")
        n = h.numel()
        o = fp8hg.alloc_token(M, MLP, 0, E4, False, dev)
        ot = fp8hg.alloc_token(M, MLP, 128, E4, True, dev)
        ws = fp8hg.dual_workspace(M, MLP, dev)
        fn = lambda: fp8hg.fp8_quant_token_dual(h, E4, out=o, out_t=ot, workspace=ws)
        work, unit = _dual_bytes(n, M), "bytes"
    elif c in ("quant_row", "quant_1x128", "quant_t", "requant"):
        h = mk("act", M, MLP, "H")
        n = h.numel()
        if c == "quant_row":
            o = fp8hg.alloc_token(M, MLP, 0, E4, False, dev)
            fn, work = lambda: fp8hg.fp8_quant_token(h, 0, E4, out=o), _tok_bytes(n, M)
        elif c == "quant_1x128":
            o = fp8hg.alloc_token(M, MLP, 128, E4, False, dev)
            fn, work = lambda: fp8hg.fp8_quant_token(h, 128, E4, out=o), _g128_bytes(n)
        elif c == "quant_t":
            o = fp8hg.alloc_token(M, MLP, 128, E4, True, dev)
            fn, work = lambda: fp8hg.fp8_quant_token(h, 128, E4, True, out=o), _g128_bytes(n)
        else:
            src = fp8hg.fp8_quant_token(h, 0, E4)
            o = fp8hg.alloc_token(M, MLP, 128, E4, True, dev)
            fn, work = lambda: fp8hg.fp8_requant_t(src, E4, out=o), 2.0 * n + M + n / 128.0
        unit = "bytes"
    elif c == "block128":
        w = mk("weight", HID, MLP, "W_down")
        o, ot = fp8hg.alloc_block128(HID, MLP, E4, True, dev)
        fn = lambda: fp8hg.fp8_quant_block128(w, E4, True, out=o, out_t=ot)
        work, unit = _blk_bytes(w.numel(), True), "bytes"
    else:  # mx32, mx32_mon
        x = mk("mx_ln", M, 4096, "A")
        o = fp8hg.alloc_mx32(M, 4096, E4, dev)
        if c == "mx32":
            fn = lambda: fp8hg.fp8_quant_mx32(x, E4, out=o)
        else:
            st = torch.zeros(4, dtype=torch.int64, device=dev)
            fn = lambda: fp8hg.fp8_quant_mx32_monitor(x, E4, stats=st, out=o)
        work, unit = 3.0 * x.numel() + x.numel() / 32.0, "bytes"
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(args.steps):
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_.record()
        fn()
        b_.record()
        b_.synchronize()
        ts.append(a_.elapsed_time(b_))
    if fp8hg.fp8hg_get_device_error() != 0:
        raise RuntimeError("device error")
    ms = sum(ts) / len(ts)
    rate = work / ms / (1e9 if unit == "flop" else 1e6)
    print(json.dumps({"kernel_case": c, "what": KERNEL_CASES[c], "m": M, "launches": len(ts),
                      "mean_ms": ms, "min_ms": min(ts),
                      ("tflops" if unit == "flop" else "gbs"): rate}), flush=True)


# ------------------------------------------------------------------- main
def main(argv=None):
    args = _parse(argv)
    if args.impl == "reference":
        run_reference(args)
        return 0
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        return spawn_replicas(args.gpus, sys.argv[1:] if argv is None else argv)
    if args.kernel:
        run_kernel_case(args)
        return 0
    import torch
    import torch.distributed as dist
    import fp8_hybrid_granularity_gb300 as fp8hg
    from fp8_hybrid_granularity_gb300 import workloads

    ri = replicas.rank_info()
    if ri.world > 1 and torch.cuda.device_count() <= ri.local:
        raise SystemExit(f"rank {ri.rank}: local rank {ri.local} has no GPU "
                         f"({torch.cuda.device_count()} visible)")
    torch.cuda.set_device(ri.local)
    if ri.world > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", ri.local)
    fp8hg.load_library()
    peaks = _peaks()
    run = run_sweep if args.config == "sweep" else run_step_config
    line = run(args, torch, dist, fp8hg, workloads, ri, dev, peaks)
    if line is not None:
        print(json.dumps(line), flush=True)
    if ri.world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
