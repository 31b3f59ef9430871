#!/usr/bin/env python
"""Benchmark of the Q4_K / Q5_K / Q6_K x Q8 path on GB300 at 7B shapes.  Prints ONE JSON line.

Step (the headline `value`): one 7B FFN prefill at the pages' 3314-token prompt length
(3314 tokens), every row of the hot path:
    RMSNorm-fused Q8 quantize (x_hidden 3314 x 3584)
    -> Q4_K tensor-core GEMM gate (18944 x 3584)  -> Q4_K GEMM up (18944 x 3584)
    -> plain Q8 quantize (x_ffn 3314 x 18944)      -> Q6_K GEMM down (3584 x 18944)
value = 2*M*N*K integer ops summed over the three GEMMs / step time, in TOPS.
The step's footprint (weights 132 MB, activations 298 MB, outputs 549 MB) is far larger
than the 129 MB L2, so consecutive steps do not hit L2 for their inputs (no flush).

Also reported, measured in the same run:
  "decode":  the decode sweep, one decode token through all 196 per-layer matmuls of a 28-layer
             7B q4_K_m stack (Q8 quantize + dp4a GEMV each, captured in one CUDA graph): one
             grouped GEMV launch per layer level (q|k|v, o, gate|up, down), the K = 3584 levels
             quantizing their activation inside the GEMV, down's through a quantize launch;
             the variants (a quantize launch before every level, per-matrix launches on
             parallel branches, one linear chain as "serial") are reported beside it; weight
             GB/s and tok/s; 3.9 GB of weights, far larger than L2.
  "lm_head": the 152064 x 3584 Q6_K LM head at M = 1 (GEMV) and M = 16 (GEMV and GEMM).
  "gemm_q5k", "gemv_q5k": the Q5_K prefill GEMM on the gate shape and the Q5_K decode GEMV on a
             matrix of the LM-head shape (synthetic Q5_K weights).
  "gate_up_swiglu": the fused gate|up GEMM with the SwiGLU epilogue writing the down
             projection's plane, against the unfused chain, alone and inside the whole FFN.
  "gemv_b32", "gemm_b32": the decode GEMV of each 32-value block format (Q4_0, Q4_1, Q5_0, Q5_1,
             Q8_0) on a matrix of the LM-head shape, and its prefill GEMM on the gate shape
             (synthetic weights).
  "roofline": the dominant kernel (Q4_K GEMM) against the measured dense bf16 tensor peak
             (f16 MMA rate = bf16 rate); "roofline_decode": the LM-head GEMV against the
             measured HBM copy bandwidth.
  "e2e":     the same step through the C ABI from pinned host buffers, with the activation
             copies in and the three outputs copied back inside the timed region (the copies
             on their own streams, overlapping the GEMMs that do not need them).
  "cpu_baseline": the CPU oracle on this host's cores on a token slice of the same step.

--impl reference times the CPU oracle itself on the same workload (a token slice per step).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Q4_K/Q6_K MMQ prefill int8 TOPS + MMVQ decode weight GB/s at 7B shapes"
L2_BYTES = 129 * 1024 * 1024


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["mq", "reference"], default="mq")
    ap.add_argument("--skip-decode", action="store_true", help="prefill step only")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU-baseline sample budget")
    ap.add_argument("--case", choices=sorted(CASES), help="run one kernel of the path a few times (profiling)")
    ap.add_argument("--reps", type=int, default=3, help="launches of --case after 2 warm-up launches")
    return ap.parse_args()


# DRAM bytes (read + write) of one launch of the roofline kernels, from one ncu capture of the
# current kernels (dram__bytes_read.sum + dram__bytes_write.sum); set to None whenever a kernel
# changes until it is captured again.
TRAFFIC_GEMM_Q4K_GATE = 97.276928e6 + 209.093120e6      # 18944x3584 Q4_K, M=3314 (Y is 251 MB)
TRAFFIC_GEMM_Q6K_DOWN = 420.704000e6 + 43.702784e6      # 3584x18944 Q6_K, M=3314
TRAFFIC_GEMV_Q6K_LMHEAD = 447.188736e6 + 3.509760e6     # 152064x3584 Q6_K, M=1
# the legacy int8 tensor instruction's measured peak on this GPU (mma.sync.m16n8k32.s8, 152 SMs): context
# only -- the GEMM does not use that instruction
INT8_MMA_SYNC_PEAK_TOPS = 158.1
# the instruction the GEMM does use, tcgen05.mma kind::f16 issued back to back from shared memory on all
# 152 SMs (a probe of this project, profiles/probes_gb300_peaks.md): the kernel's own instruction ceiling,
# reported beside the cuBLAS bf16 denominator
TCGEN05_F16_PROBE_TFLOPS = 2400.4

# single-kernel cases for profiler captures: name -> (config, kernel); inputs of the named config
CASES = {
    "gemm_q4k_gate": "7B FFN prefill gate GEMM: Q4_K 18944x3584, M=3314",
    "gemm_q6k_down": "7B FFN prefill down GEMM: Q6_K 3584x18944, M=3314",
    "gemm_q4k_qproj": "7B q_proj prefill GEMM: Q4_K 3584x3584, M=512",
    "gemv_q6k_lmhead": "LM head GEMV: Q6_K 152064x3584, M=1",
    "small_q6k_lmhead": "LM head small-M tensor-core GEMM: Q6_K 152064x3584, M=16",
    "small_q4k_vocab": "small-M tensor-core GEMM of the LM-head shape: 152064x3584 synthetic Q4_K weights, M=16",
    "gemv_q4k_gate": "decode sweep layer-1 gate GEMV: Q4_K 18944x3584, M=1",
    "gemv_q5k_vocab": "Q5_K GEMV of the LM-head shape: 152064x3584 synthetic Q5_K weights, M=1",
    **{f"gemv_{f}_vocab": f"{f.upper()} GEMV of the LM-head shape: 152064x3584 synthetic {f.upper()} weights, M=1"
       for f in ("q4_0", "q4_1", "q5_0", "q5_1", "q8_0")},
    **{f"gemm_{f}_gate": f"{f.upper()} GEMM of the gate shape: 18944x3584 synthetic {f.upper()} weights, M=3314"
       for f in ("q4_0", "q4_1", "q5_0", "q5_1", "q8_0")},
    "gemm_swiglu_ffn": "7B FFN prefill fused gate|up GEMM: Q4_K 2 x 18944x3584, M=3314, SwiGLU epilogue -> down plane",
    "quantize_rms": "7B FFN prefill RMSNorm-fused Q8 quantize: 3314x3584",
    "decode_sweep": "decode sweep: the 196 quantize + GEMV pairs of one decode token, plain launches",
    "decode_sweep_grouped": "decode sweep: one decode token with one grouped quantize and one grouped GEMV launch per "
                            "layer level and format (238 launches), plain launches",
    "decode_sweep_fused": "decode sweep: one decode token, the K = 3584 levels' activations quantized inside their "
                          "grouped GEMVs, down's by a grouped quantize launch (154 launches), plain launches",
    "quantize_ffn": "7B FFN prefill plain Q8 quantize: 3314x18944",
}


def run_case(args):
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from quantized_q8_activation_quantize_gb300 import binding as B
    from quantized_q8_activation_quantize_gb300 import inputs as I
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    name = args.case
    if name == "decode_sweep":
        sw = DecodeSweep(torch, B, I)
        for _ in range(1 + args.reps):
            sw.run(True)
        torch.cuda.synchronize()
        B.mq_device_status()
        print(json.dumps({"case": name, "what": CASES[name], "launches": (1 + args.reps) * 2 * len(sw.items)}))
        return
    if name in ("decode_sweep_grouped", "decode_sweep_fused"):
        sw = DecodeSweep(torch, B, I)
        for _ in range(1 + args.reps):
            sw.run_grouped(True, I.HIDDEN if name == "decode_sweep_fused" else 0)
        torch.cuda.synchronize()
        B.mq_device_status()
        print(json.dumps({"case": name, "what": CASES[name]}))
        return
    if name.startswith("gemm_q4k_gate") or name.startswith("gemm_q6k_down") or name.startswith("quantize"):
        c = I.ffn_prefill()
        M = c["x_hidden"].shape[0]
        if name == "gemm_q6k_down" or name == "quantize_ffn":
            x, K, N, w, fmt, rms = c["x_ffn"], I.FFN, I.HIDDEN, c["w_down"], "q6k", None
        else:
            x, K, N, w, fmt, rms = c["x_hidden"], I.HIDDEN, I.FFN, c["w_gate"], "q4k", c["rms_w"]
    elif name == "gemm_q4k_qproj":
        c = I.qproj_prefill()
        x, w, fmt, rms = c["x"], c["w"], "q4k", None
        M, K, N = x.shape[0], x.shape[1], w.shape[0]
    elif name == "gemv_q6k_lmhead":
        x, w, fmt, rms = I.lm_head_x(1), I.lm_head_weights(), "q6k", None
        M, K, N = 1, I.HIDDEN, I.VOCAB
    elif name == "small_q6k_lmhead":
        x, w, fmt, rms = I.lm_head_x(16), I.lm_head_weights(), "q6k", None
        M, K, N = 16, I.HIDDEN, I.VOCAB
    elif name == "small_q4k_vocab":
        x, w, fmt, rms = I.lm_head_x(16), I.q4k_weights(I.rng(4, I.STREAM_W, 1), I.VOCAB, I.HIDDEN), "q4k", None
        M, K, N = 16, I.HIDDEN, I.VOCAB
    elif name == "gemv_q5k_vocab":
        x, w, fmt, rms = I.lm_head_x(1), I.q5k_vocab_weights(), "q5k", None
        M, K, N = 1, I.HIDDEN, I.VOCAB
    elif name == "gemm_swiglu_ffn" or (name.startswith("gemm_q") and name[5:-5] in I.B32_BYTES):
        c = I.ffn_prefill()
        x, rms, K, N = c["x_hidden"], c["rms_w"], I.HIDDEN, I.FFN
        M = x.shape[0]
        if name == "gemm_swiglu_ffn":
            fmt, w, w2 = "q4k", c["w_gate"], c["w_up"]
        else:
            fmt, w2 = name[5:-5], None
            w = I.b32_weights(I.rng(2, I.STREAM_W, 6 + list(I.B32_BYTES).index(fmt)), N, K, fmt)
    elif name.startswith("gemv_q") and name[5:-6] in I.B32_BYTES:
        fmt = name[5:-6]
        x, w, rms = I.lm_head_x(1), I.b32_vocab_weights(fmt), None
        M, K, N = 1, I.HIDDEN, I.VOCAB
    else:
        c = I.decode_matrix(1, 4)
        x, w, fmt, rms = c["x"], c["w"], "q4k", None
        M, K, N = 1, I.HIDDEN, I.FFN
    xd, wd = dev(x), dev(w.reshape(N, -1))
    rd = dev(rms) if rms is not None else None
    plane = B.alloc_plane(M, K)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    B.mq_quantize_q8(xd, M, K, rd, 1e-6, plane)
    if name.startswith("quantize"):
        fn = lambda: B.mq_quantize_q8_ex(xd, M, K, rd, 1e-6, B.PLANE_FOR_GEMM, plane)
    elif name == "gemm_swiglu_ffn":
        w2d, po = dev(w2.reshape(N, -1)), B.alloc_plane(M, N)
        fn = lambda: B.mq_gemm_q4k_swiglu(wd, w2d, N, K, plane, M, po)
    else:
        f = (B.GEMM_SMALL if name.startswith("small") else B.GEMM if name.startswith("gemm") else B.GEMV)[fmt]
        fn = lambda: f(wd, N, K, plane, M, y)
    for _ in range(2 + args.reps):
        fn()
    torch.cuda.synchronize()
    B.mq_device_status()
    print(json.dumps({"case": name, "what": CASES[name], "launches": 2 + args.reps}))


# ------------------------------------------------------------------------------ distributed ---

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, use_cuda: bool):
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend="nccl" if use_cuda else "gloo")
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if self.pg is None:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64, device="cuda" if self.pg.get_backend() == "nccl" else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())


# ----------------------------------------------------------------------------------- clocks ---

class Clocks:
    """nvidia-smi sampler running only while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ln in open(self.path):
            p = [s.strip() for s in ln.split(",")]
            if len(p) >= 9:
                rows.append(p)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "reasons": reasons, "samples": len(rows)}


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------------------------- workloads ---

def ffn_ops(M):
    from quantized_q8_activation_quantize_gb300 import inputs as I
    return 2 * M * (2 * I.FFN * I.HIDDEN + I.HIDDEN * I.FFN)


class Prefill:
    """The 7B FFN prefill step at M = 3314, device-resident inputs."""

    def __init__(self, torch, B, I):
        self.torch, self.B = torch, B
        c = I.ffn_prefill()
        self.M, self.H, self.F = c["x_hidden"].shape[0], I.HIDDEN, I.FFN
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        self.w_gate = dev(c["w_gate"].reshape(self.F, -1))
        self.w_up = dev(c["w_up"].reshape(self.F, -1))
        self.w_down = dev(c["w_down"].reshape(self.H, -1))
        self.host_x_h = torch.from_numpy(c["x_hidden"]).pin_memory()
        self.host_x_f = torch.from_numpy(c["x_ffn"]).pin_memory()
        self.x_h, self.x_f = self.host_x_h.cuda(), self.host_x_f.cuda()
        self.rms_w = dev(c["rms_w"])
        self.eps = float(c["eps"])
        self.p_h = B.alloc_plane(self.M, self.H)
        self.p_f = B.alloc_plane(self.M, self.F)
        self.y_gate = torch.empty((self.M, self.F), dtype=torch.float32, device="cuda")
        self.y_up = torch.empty_like(self.y_gate)
        self.y_down = torch.empty((self.M, self.H), dtype=torch.float32, device="cuda")
        self.ops = ffn_ops(self.M)
        self.gemm_q4k_ops = 2 * self.M * self.F * self.H
        self.gemm_q6k_ops = 2 * self.M * self.H * self.F
        self.launches = 5

    def step(self, ev=None):
        """One pass; with `ev` (list of 6 events) records event boundaries between launches."""
        B, M, H, F = self.B, self.M, self.H, self.F
        rec = (lambda i: ev[i].record()) if ev is not None else (lambda i: None)
        rec(0)
        B.mq_quantize_q8_ex(self.x_h, M, H, self.rms_w, self.eps, B.PLANE_FOR_GEMM, self.p_h)
        rec(1)
        B.mq_gemm_q4k(self.w_gate, F, H, self.p_h, M, self.y_gate)
        rec(2)
        B.mq_gemm_q4k(self.w_up, F, H, self.p_h, M, self.y_up)
        rec(3)
        B.mq_quantize_q8_ex(self.x_f, M, F, None, 0.0, B.PLANE_FOR_GEMM, self.p_f)
        rec(4)
        B.mq_gemm_q6k(self.w_down, H, F, self.p_f, M, self.y_down)
        rec(5)

    def e2e_setup(self):
        t = self.torch
        self.host_y = [t.empty(tuple(y.shape), dtype=t.float32).pin_memory() for y in (self.y_gate, self.y_up, self.y_down)]
        self.h2d = self.host_x_h.numel() * 4 + self.host_x_f.numel() * 4
        self.d2h = sum(y.numel() * 4 for y in self.host_y)
        self.s_in, self.s_out = t.cuda.Stream(), t.cuda.Stream()

    def e2e_step(self):
        """The step from pinned host inputs to pinned host outputs, copies on their own streams:
        x_ffn goes up while the gate / up GEMMs run, y_gate and y_up come back while the later
        GEMMs run; the step ends (on the calling stream) when all three outputs are on the host."""
        t, B, M, H, F = self.torch, self.B, self.M, self.H, self.F
        cs = t.cuda.current_stream()
        ev = lambda s: (lambda e: (e.record(s), e)[1])(t.cuda.Event())
        self.s_in.wait_event(ev(cs))                      # the previous step is done with x_h / x_f
        with t.cuda.stream(self.s_in):
            self.x_h.copy_(self.host_x_h, non_blocking=True)
            e_xh = ev(self.s_in)
            self.x_f.copy_(self.host_x_f, non_blocking=True)
            e_xf = ev(self.s_in)
        cs.wait_event(e_xh)
        B.mq_quantize_q8_ex(self.x_h, M, H, self.rms_w, self.eps, B.PLANE_FOR_GEMM, self.p_h)
        B.mq_gemm_q4k(self.w_gate, F, H, self.p_h, M, self.y_gate)
        e_g = ev(cs)
        B.mq_gemm_q4k(self.w_up, F, H, self.p_h, M, self.y_up)
        e_u = ev(cs)
        cs.wait_event(e_xf)
        B.mq_quantize_q8_ex(self.x_f, M, F, None, 0.0, B.PLANE_FOR_GEMM, self.p_f)
        B.mq_gemm_q6k(self.w_down, H, F, self.p_f, M, self.y_down)
        e_d = ev(cs)
        with t.cuda.stream(self.s_out):
            for e, h, d in ((e_g, self.host_y[0], self.y_gate), (e_u, self.host_y[1], self.y_up),
                            (e_d, self.host_y[2], self.y_down)):
                self.s_out.wait_event(e)
                h.copy_(d, non_blocking=True)
            e_out = ev(self.s_out)
        cs.wait_event(e_out)


class DecodeSweep:
    """The decode sweep: one decode token through the 196 matmuls of a 28-layer 7B q4_K_m stack."""

    def __init__(self, torch, B, I):
        self.torch, self.B = torch, B
        self.items = []
        self.weight_bytes = 0
        self.bytes = 0
        for (layer, idx, name, fmt, n, k) in I.decode_layout():
            c = I.decode_matrix(layer, idx)
            w = torch.from_numpy(c["w"].reshape(n, -1)).cuda()
            x = torch.from_numpy(c["x"]).cuda()
            plane = B.alloc_plane(1, k)
            y = torch.empty((1, n), dtype=torch.float32, device="cuda")
            self.items.append((fmt, w, x, plane, y, n, k))
            self.weight_bytes += w.numel()
            self.bytes += w.numel() + 1.25 * k + 4 * n + 4 * k     # weights + plane + output + activation
        self.graph = None

    def _one(self, item, quantize):
        fmt, w, x, plane, y, n, k = item
        if quantize:
            self.B.mq_quantize_q8_ex(x, 1, k, None, 0.0, self.B.PLANE_FOR_GEMV, plane)
        self.B.GEMV[fmt](w, n, k, plane, 1, y)

    def run(self, quantize=True, branches=False):
        """The sweep in layer order.  branches=True: a layer's independent matmuls -- q, k, v (all
        from the layer input) and gate, up (both from the post-attention input) -- go to parallel
        streams, joined before o and before down, the dependency structure of a real layer."""
        if not branches:
            for item in self.items:
                self._one(item, quantize)
            return
        t = self.torch
        main = t.cuda.current_stream()
        if not hasattr(self, "side"):
            self.side = [t.cuda.Stream(), t.cuda.Stream()]
        for layer in range(len(self.items) // 7):
            li = self.items[7 * layer:7 * layer + 7]           # q, k, v, o, gate, up, down
            for group in (li[0:3], li[3:4], li[4:6], li[6:7]):
                if len(group) == 1:
                    self._one(group[0], quantize)
                    continue
                fork = t.cuda.Event()
                fork.record(main)
                for i in range(len(group) - 1):
                    self.side[i].wait_event(fork)
                    with t.cuda.stream(self.side[i]):
                        self._one(group[1 + i], quantize)
                self._one(group[0], quantize)
                for i in range(len(group) - 1):
                    join = t.cuda.Event()
                    join.record(self.side[i])
                    main.wait_event(join)

    def _gemv_group(self, group):
        if len(group) == 1:
            fmt, w, x, plane, y, n, k = group[0]
            self.B.GEMV[fmt](w, n, k, plane, 1, y)
        else:
            self.B.GEMV_GROUPED[group[0][0]]([(w, n, plane, y) for (_, w, _, plane, y, n, _) in group], group[0][6], 1)

    def _gemv_group_x(self, group):
        fmt, k = group[0][0], group[0][6]
        self.B.GEMV_GROUPED_X[fmt]([(w, n, x, y) for (_, w, x, _, y, n, _) in group], k)

    def run_grouped(self, quantize=True, xq_max_k=0):
        """The sweep with one launch per layer level and weight format: q|k|v from the layer input (one
        grouped quantize; one grouped Q4_K GEMV, and in the Q6_K layers v's GEMV on a parallel branch),
        then o, gate|up (grouped quantize and GEMV), down -- the dependency order of a real layer.
        Levels with K <= xq_max_k skip the quantize launch: their grouped GEMV quantizes the f32
        activations itself (mq_gemv_grouped_x_*)."""
        t, B = self.torch, self.B
        main = t.cuda.current_stream()
        if not hasattr(self, "side"):
            self.side = [t.cuda.Stream(), t.cuda.Stream()]
        for layer in range(len(self.items) // 7):
            li = self.items[7 * layer:7 * layer + 7]           # q, k, v, o, gate, up, down
            for group in (li[0:3], li[3:4], li[4:6], li[6:7]):
                fused = quantize and group[0][6] <= xq_max_k
                gemv = self._gemv_group_x if fused else self._gemv_group
                if quantize and not fused:
                    B.mq_quantize_q8_grouped([(it[2], it[3]) for it in group], 1, group[0][6], B.PLANE_FOR_GEMV)
                by_fmt = {}
                for it in group:
                    by_fmt.setdefault(it[0], []).append(it)
                if len(by_fmt) == 1:
                    gemv(group)
                    continue
                fork = t.cuda.Event()
                fork.record(main)
                self.side[0].wait_event(fork)
                with t.cuda.stream(self.side[0]):
                    gemv(by_fmt["q6k"])
                gemv(by_fmt["q4k"])
                join = t.cuda.Event()
                join.record(self.side[0])
                main.wait_event(join)

    def capture_grouped(self, quantize=True, xq_max_k=0):
        t = self.torch
        s = t.cuda.Stream()
        s.wait_stream(t.cuda.current_stream())
        with t.cuda.stream(s):
            self.run_grouped(True, xq_max_k)
        t.cuda.current_stream().wait_stream(s)
        t.cuda.synchronize()
        g = t.cuda.CUDAGraph()
        with t.cuda.graph(g):
            self.run_grouped(quantize, xq_max_k)
        t.cuda.synchronize()
        return g

    def capture(self, quantize=True, branches=False):
        """One CUDA graph of the sweep: Q8 quantize + GEMV per matmul, or the GEMVs alone
        (on the planes the last quantizing run left)."""
        t = self.torch
        s = t.cuda.Stream()
        s.wait_stream(t.cuda.current_stream())
        with t.cuda.stream(s):
            self.run(True, branches)       # warm the launch path (and fill the planes) outside the capture
        t.cuda.current_stream().wait_stream(s)
        t.cuda.synchronize()
        g = t.cuda.CUDAGraph()
        with t.cuda.graph(g):
            self.run(quantize, branches)
        t.cuda.synchronize()
        return g


def time_events(torch, fn, steps, warmup):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


# ------------------------------------------------------------------------------ CPU oracle ---

def cpu_oracle_ffn(budget_s: float, threads: int):
    """The oracle on token slices of the FFN prefill step until `budget_s` is spent."""
    import oracle
    from quantized_q8_activation_quantize_gb300 import inputs as I
    c = I.ffn_prefill()
    t_done, ops, tokens = 0.0, 0, 0
    chunk = 4
    while t_done < budget_s and tokens < c["x_hidden"].shape[0]:
        n = min(chunk, c["x_hidden"].shape[0] - tokens)       # the last slice may be short
        sl = slice(tokens, tokens + n)
        t0 = time.perf_counter()
        ph = oracle.quantize_q8(c["x_hidden"][sl], c["rms_w"], float(c["eps"]))
        oracle.matmul(c["w_gate"], "q4k", ph, threads=threads)
        oracle.matmul(c["w_up"], "q4k", ph, threads=threads)
        pf = oracle.quantize_q8(c["x_ffn"][sl])
        oracle.matmul(c["w_down"], "q6k", pf, threads=threads)
        t_done += time.perf_counter() - t0
        ops += ffn_ops(n)
        tokens += n
    return ops / t_done / 1e12, tokens, t_done


# ------------------------------------------------------------------------------------ main ---

def run_reference(args, dist):
    if dist.rank != 0:
        return
    threads = os.cpu_count() or 1
    per_step = []
    tokens = 0
    budget = max(0.5, min(args.cpu_seconds, 20.0, 120.0 / max(1, args.steps + args.warmup)))
    for i in range(args.warmup + args.steps):
        v, tok, t = cpu_oracle_ffn(budget, threads)
        if i >= args.warmup:
            per_step.append((v, tok, t))
            tokens = tok
    value = statistics.mean(v for v, _, _ in per_step)
    ms = statistics.mean(t for _, _, t in per_step) * 1e3
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int8 dots, f64 scaling (CPU oracle)",
            "data": "synthetic (seeded, 7B q4_K_m shapes)",
            "config": {"workload": "7B FFN prefill, 3314 tokens: RMSNorm-Q8, gate/up Q4_K 18944x3584, "
                                   "Q8, down Q6_K 3584x18944", "tokens_per_step_sample": tokens},
            "cpu_baseline": {"value": value, "unit": "TOPS", "cores": threads, "kind": "oracle",
                             "sample": f"first {tokens} of 3314 tokens of the FFN step per timed step"},
            "e2e": {"value": value, "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def bind_gpu_local_cpus(torch, dev):
    """Run this process (and so first-touch its pinned host buffers) on the CPUs local to the GPU, as
    sysfs lists them for the GPU's PCI function; returns that CPU list, or None where it is not known."""
    try:
        pr = torch.cuda.get_device_properties(dev)
        bus = f"{pr.pci_domain_id:04x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"
        with open(f"/sys/bus/pci/devices/{bus}/local_cpulist") as f:
            spec = f.read().strip()
        cpus = set()
        for part in spec.split(","):
            if "-" in part:
                a, b = part.split("-")
                cpus.update(range(int(a), int(b) + 1))
            elif part:
                cpus.add(int(part))
        cpus &= os.sched_getaffinity(0)
        if not cpus:
            return None
        os.sched_setaffinity(0, cpus)
        return spec
    except (AttributeError, OSError, ValueError):
        return None


def main():
    args = parse_args()
    if args.case:
        run_case(args)
        return
    dist = Dist()
    if args.impl == "reference":
        dist.init(use_cuda=False)
        run_reference(args, dist)
        return
    import torch
    torch.cuda.set_device(dist.local)
    dist.init(use_cuda=True)
    host_cpus = bind_gpu_local_cpus(torch, dist.local)
    import __graft_entry__
    __graft_entry__.build()
    from quantized_q8_activation_quantize_gb300 import binding as B
    from quantized_q8_activation_quantize_gb300 import inputs as I

    hbm_peak, bf16_peak, peak_kind = measured_peaks()
    W = max(3, args.warmup)
    K = max(1, args.steps)

    # ---------------- prefill step (headline)
    pf = Prefill(torch, B, I)
    for _ in range(W):
        pf.step()
    torch.cuda.synchronize()
    B.mq_device_status()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    clocks = Clocks(torch.cuda.current_device())
    clocks.start()
    dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record()
    for k in range(K):
        pf.step(evs[k])
    t_end.record()
    torch.cuda.synchronize()
    dist.barrier()
    clk = clocks.stop()
    B.mq_device_status()
    ms_step = dist.max(t_start.elapsed_time(t_end) / K)
    per = np.array([[e[i].elapsed_time(e[i + 1]) for i in range(5)] for e in evs])   # ms per launch
    k_ms = per.mean(axis=0)
    value = dist.world * pf.ops / (ms_step * 1e-3) / 1e12

    gemm_q4k_ms = (k_ms[1] + k_ms[2]) / 2
    q4k_tflops = pf.gemm_q4k_ops / (gemm_q4k_ms * 1e-3) / 1e12
    q6k_tflops = pf.gemm_q6k_ops / (k_ms[4] * 1e-3) / 1e12
    # algorithmic bytes of a quantizer: 4 B in and 1.25 B out per value (+ the RMSNorm weight)
    qrms_gbs = (pf.M * pf.H * 5.25 + pf.H * 4) / (k_ms[0] * 1e-3) / 1e9
    q_gbs = pf.M * pf.F * 5.25 / (k_ms[3] * 1e-3) / 1e9
    # the SwiGLU producer (NEXT row, not part of the FFN prefill step): the down projection's plane
    # from this step's gate / up outputs
    swiglu_ms = time_events(torch, lambda: B.mq_quantize_swiglu_q8_ex(pf.y_gate, pf.y_up, pf.M, pf.F, B.PLANE_FOR_GEMM,
                                                                      pf.p_f), K, W)
    swiglu_gbs = pf.M * pf.F * 9.25 / (swiglu_ms * 1e-3) / 1e9
    # the fused gate|up GEMM (NEXT row): gate and up in one kernel whose epilogue writes the down
    # projection's plane, against the unfused chain (two GEMMs, then the SwiGLU producer), and the
    # whole SwiGLU FFN both ways (RMSNorm-Q8 -> gate|up -> down)
    def unfused_gu():
        B.mq_gemm_q4k(pf.w_gate, pf.F, pf.H, pf.p_h, pf.M, pf.y_gate)
        B.mq_gemm_q4k(pf.w_up, pf.F, pf.H, pf.p_h, pf.M, pf.y_up)
        B.mq_quantize_swiglu_q8_ex(pf.y_gate, pf.y_up, pf.M, pf.F, B.PLANE_FOR_GEMM, pf.p_f)

    def fused_gu():
        B.mq_gemm_q4k_swiglu(pf.w_gate, pf.w_up, pf.F, pf.H, pf.p_h, pf.M, pf.p_f)

    def ffn(gu):
        def run():
            B.mq_quantize_q8_ex(pf.x_h, pf.M, pf.H, pf.rms_w, pf.eps, B.PLANE_FOR_GEMM, pf.p_h)
            gu()
            B.mq_gemm_q6k(pf.w_down, pf.H, pf.F, pf.p_f, pf.M, pf.y_down)
        return run

    gu_unfused_ms = time_events(torch, unfused_gu, K, W)
    gu_fused_ms = time_events(torch, fused_gu, K, W)
    ffn_unfused_ms = time_events(torch, ffn(unfused_gu), K, W)
    ffn_fused_ms = time_events(torch, ffn(fused_gu), K, W)
    B.mq_device_status()
    fused = {"what": "7B SwiGLU FFN at 3314 tokens: gate|up Q4_K 2 x 18944 x 3584 -> silu(gate) * up as the "
                     "down projection's Q8 plane; fused = one kernel, unfused = two GEMMs + the SwiGLU producer",
             "gate_up_fused_ms": gu_fused_ms, "gate_up_unfused_ms": gu_unfused_ms,
             "gate_up_fused_TOPS": 2 * pf.gemm_q4k_ops / (gu_fused_ms * 1e-3) / 1e12,
             "ffn_fused_ms": ffn_fused_ms, "ffn_unfused_ms": ffn_unfused_ms,
             "ffn_fused_TOPS": pf.ops / (ffn_fused_ms * 1e-3) / 1e12}
    # the Q5_K prefill GEMM on the gate shape (synthetic Q5_K weights), from the step's plane
    w5g = torch.from_numpy(I.q5k_weights(I.rng(2, I.STREAM_W, 5), pf.F, pf.H).reshape(pf.F, -1)).cuda()
    q5_ms = time_events(torch, lambda: B.mq_gemm_q5k(w5g, pf.F, pf.H, pf.p_h, pf.M, pf.y_gate), K, W)
    del w5g
    gemm_b32 = {}
    for i, fmt in enumerate(I.B32_BYTES):
        wb = torch.from_numpy(I.b32_weights(I.rng(2, I.STREAM_W, 6 + i), pf.F, pf.H, fmt).reshape(pf.F, -1)).cuda()
        ms_b = time_events(torch, lambda: B.GEMM[fmt](wb, pf.F, pf.H, pf.p_h, pf.M, pf.y_gate), K, W)
        gemm_b32[fmt] = {"ms": ms_b, "TOPS": 2 * pf.M * pf.F * pf.H / (ms_b * 1e-3) / 1e12}
        del wb

    # ---------------- e2e through host buffers
    pf.e2e_setup()
    e2e_ms = time_events(torch, pf.e2e_step, max(2, K // 2), 1)
    e2e_ms = dist.max(e2e_ms)
    # the overlapped copies must deliver exactly what the device-resident step computes
    torch.cuda.synchronize()
    pf.step()
    torch.cuda.synchronize()
    for h, d in zip(pf.host_y, (pf.y_gate, pf.y_up, pf.y_down)):
        if not torch.equal(h, d.cpu()):
            raise RuntimeError("e2e outputs differ from the device-resident step")
    e2e = {"value": dist.world * pf.ops / (e2e_ms * 1e-3) / 1e12, "unit": "TOPS", "ms_per_step": e2e_ms,
           "h2d_bytes_per_step": pf.h2d, "d2h_bytes_per_step": pf.d2h}

    line = {
        "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": dist.world, "steps": K, "warmup": W,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8 (exact integer block dots on f16 tensor-core MMA) + f32 scaling",
        "data": "synthetic (seeded, 7B q4_K_m shapes)",
        "config": {"workload": "7B FFN prefill, 3314 tokens: RMSNorm-Q8, gate/up Q4_K 18944x3584, "
                               "Q8, down Q6_K 3584x18944", "tokens": pf.M, "l2": "inputs larger than L2 (no flush)",
                   "parallelism": f"replicas x{dist.world}", "host_cpus": host_cpus},
        "prefill_tok_per_s": dist.world * pf.M / (ms_step * 1e-3),
        "kernels_ms": {"rms_quantize": k_ms[0], "gemm_q4k_gate": k_ms[1], "gemm_q4k_up": k_ms[2],
                       "quantize": k_ms[3], "gemm_q6k_down": k_ms[4]},
        "kernels_rate": {"gemm_q4k_tops": q4k_tflops, "gemm_q6k_tops": q6k_tflops,
                         "rms_quantize_gbs": qrms_gbs, "quantize_gbs": q_gbs},
        "swiglu_quantize": {"what": "SwiGLU-fused Q8 producer of the down projection, 3314 x 18944 "
                                    "(gate / up outputs of the step)", "ms": swiglu_ms, "GB/s": swiglu_gbs},
        "gemm_q5k": {"what": "Q5_K GEMM on the gate shape 18944 x 3584, M = 3314 (synthetic Q5_K weights)",
                     "ms": q5_ms, "TOPS": pf.gemm_q4k_ops / (q5_ms * 1e-3) / 1e12},
        "gate_up_swiglu": fused,
        "gemm_b32": {"what": "GEMM on the gate shape 18944 x 3584, M = 3314, per 32-value block format "
                             "(synthetic weights)", **gemm_b32},
        "roofline": {"bound": "tensor", "kernel": "mq_gemm_q4k (18944x3584, M=3314)", "achieved": q4k_tflops,
                     "peak": bf16_peak, "unit": "TFLOP/s", "frac": q4k_tflops / bf16_peak,
                     "traffic": TRAFFIC_GEMM_Q4K_GATE,
                     "peak_kind": f"{peak_kind} dense bf16 (f16 MMA has the same nominal rate)",
                     "peak_probe": TCGEN05_F16_PROBE_TFLOPS, "frac_of_probe": q4k_tflops / TCGEN05_F16_PROBE_TFLOPS,
                     "vs_int8_mma_sync_peak": q4k_tflops / INT8_MMA_SYNC_PEAK_TOPS,
                     "vs_int8_mma_sync_note": "context only: the legacy int8 instruction is not what the kernel runs"},
        "roofline_q6k": {"bound": "tensor", "kernel": "mq_gemm_q6k (3584x18944, M=3314)", "achieved": q6k_tflops,
                         "peak": bf16_peak, "unit": "TFLOP/s", "frac": q6k_tflops / bf16_peak,
                         "traffic": TRAFFIC_GEMM_Q6K_DOWN,
                         "peak_kind": f"{peak_kind} dense bf16 (f16 MMA has the same nominal rate)"},
        "e2e": e2e, "gpu_launches": pf.launches * K, "clocks": clk,
    }

    # ---------------- decode: LM head GEMV and the 28-layer sweep
    if not args.skip_decode:
        lm_w = torch.from_numpy(I.lm_head_weights().reshape(I.VOCAB, -1)).cuda()
        lm = {}
        for m, paths in ((1, ("gemv",)), (4, ("gemv", "small")), (16, ("gemv", "gemm", "small")),
                         (32, ("small",)), (I.PREFILL_TOKENS, ("gemm",))):
            x = torch.from_numpy(I.lm_head_x(m)).cuda()
            plane = B.alloc_plane(m, I.HIDDEN)
            B.mq_quantize_q8(x, m, I.HIDDEN, None, 0.0, plane)
            y = torch.empty((m, I.VOCAB), dtype=torch.float32, device="cuda")
            for path in paths:
                f = {"gemv": B.GEMV, "gemm": B.GEMM, "small": B.GEMM_SMALL}[path]["q6k"]
                reps = max(5, K) if m < 1000 else 3            # M = 3314 writes a 2 GB output per launch
                ms = time_events(torch, lambda: f(lm_w, I.VOCAB, I.HIDDEN, plane, m, y), reps, min(W, 3))
                gbs = (lm_w.numel() + B.mq_q8_plane_bytes(m, I.HIDDEN) + 4 * m * I.VOCAB) / (ms * 1e-3) / 1e9
                lm[f"m{m}_{path}"] = {"ms": ms, "GB/s": gbs, "TOPS": 2 * m * I.VOCAB * I.HIDDEN / (ms * 1e-3) / 1e12}
            del x, plane, y
        line["lm_head"] = lm
        # the Q5_K decode GEMV on a matrix of the LM-head shape (synthetic Q5_K weights)
        w5 = torch.from_numpy(I.q5k_vocab_weights().reshape(I.VOCAB, -1)).cuda()
        x = torch.from_numpy(I.lm_head_x(1)).cuda()
        plane = B.alloc_plane(1, I.HIDDEN)
        B.mq_quantize_q8(x, 1, I.HIDDEN, None, 0.0, plane)
        y = torch.empty((1, I.VOCAB), dtype=torch.float32, device="cuda")
        ms = time_events(torch, lambda: B.GEMV["q5k"](w5, I.VOCAB, I.HIDDEN, plane, 1, y), max(5, K), min(W, 3))
        gbs = (w5.numel() + B.mq_q8_plane_bytes(1, I.HIDDEN) + 4 * I.VOCAB) / (ms * 1e-3) / 1e9
        line["gemv_q5k"] = {"what": "Q5_K GEMV 152064 x 3584, M = 1 (synthetic Q5_K weights, 374.7 MB)",
                            "ms": ms, "GB/s": gbs, "frac_of_hbm": gbs / hbm_peak}
        # the 32-value block formats' decode GEMV on the same shape
        b32 = {}
        for fmt in I.B32_BYTES:
            wb = torch.from_numpy(I.b32_vocab_weights(fmt).reshape(I.VOCAB, -1)).cuda()
            ms = time_events(torch, lambda: B.GEMV[fmt](wb, I.VOCAB, I.HIDDEN, plane, 1, y), max(5, K), min(W, 3))
            gbs = (wb.numel() + B.mq_q8_plane_bytes(1, I.HIDDEN) + 4 * I.VOCAB) / (ms * 1e-3) / 1e9
            b32[fmt] = {"ms": ms, "GB/s": gbs, "frac_of_hbm": gbs / hbm_peak, "weight_MB": wb.numel() / 1e6}
            del wb
        line["gemv_b32"] = {"what": "GEMV 152064 x 3584, M = 1, per 32-value block format (synthetic weights)",
                            **b32}
        del w5, x, plane, y
        g = lm["m1_gemv"]["GB/s"]
        line["roofline_decode"] = {"bound": "hbm", "kernel": "mq_gemv_q6k (152064x3584, M=1)", "achieved": g,
                                   "peak": hbm_peak, "unit": "GB/s", "frac": g / hbm_peak,
                                   "traffic": TRAFFIC_GEMV_Q6K_LMHEAD,
                                   "peak_kind": f"{peak_kind} HBM copy"}
        del lm_w
        torch.cuda.empty_cache()
        sw = DecodeSweep(torch, B, I)
        ms = time_events(torch, sw.capture(True).replay, max(5, K), W)
        ms_gemv = time_events(torch, sw.capture(False).replay, max(5, K), W)
        ms_br = time_events(torch, sw.capture(True, True).replay, max(5, K), W)
        ms_br_gemv = time_events(torch, sw.capture(False, True).replay, max(5, K), W)
        ms_gr = time_events(torch, sw.capture_grouped(True).replay, max(5, K), W)
        ms_gr_gemv = time_events(torch, sw.capture_grouped(False).replay, max(5, K), W)
        # the grouped sweep computes what the per-matrix one does, bit for bit
        outs = [it[4].clone() for it in sw.items]
        for it in sw.items:
            it[4].fill_(float("nan"))
        sw.run(True)
        torch.cuda.synchronize()
        if not all(torch.equal(a, it[4]) for a, it in zip(outs, sw.items)):
            raise RuntimeError("grouped decode sweep differs from the per-matrix sweep")
        # the sweep with the activations of the K = 3584 levels (q|k|v, o, gate|up) quantized inside
        # their grouped GEMVs, and with every level's (down too): the same outputs, bit for bit
        xq = {}
        for xk in (I.HIDDEN, I.FFN):
            gx = sw.capture_grouped(True, xk)
            for it in sw.items:
                it[4].fill_(float("nan"))
            gx.replay()
            torch.cuda.synchronize()
            if not all(torch.equal(a, it[4]) for a, it in zip(outs, sw.items)):
                raise RuntimeError("decode sweep with in-GEMV quantization differs from the per-matrix sweep")
            xq[xk] = time_events(torch, gx.replay, max(5, K), W)
            del gx
        B.mq_device_status()
        gemv_bytes = sw.bytes - 4 * sum(k for *_, k in sw.items)          # without the f32 activations
        lm_ms = lm["m1_gemv"]["ms"]
        n_layers = len(sw.items) // 7
        gr_launches = 4 * n_layers + 4 * n_layers + (n_layers + 1) // 2      # quantize + GEMV per level (+ v)
        gx_launches = gr_launches - 3 * n_layers                             # no quantize launch before q|k|v, o, gate|up
        ms_gx = xq[I.HIDDEN]
        line["decode"] = {"workload": "7B decode sweep: 28 layers x 7 matmuls, M=1, Q8 quantize + GEMV each, one CUDA graph; "
                                      "one grouped GEMV launch per layer level and format (q|k|v from the layer input, o, "
                                      "gate|up from the post-attention input, down), v's Q6_K GEMV on a parallel branch; the "
                                      "K = 3584 levels quantize their activation inside the GEMV, down's takes a quantize launch",
                          "ms_per_token": ms_gx, "tok_per_s": 1e3 / ms_gx, "weight_bytes": sw.weight_bytes,
                          "GB/s": sw.bytes / (ms_gx * 1e-3) / 1e9,
                          "frac_of_hbm": sw.bytes / (ms_gx * 1e-3) / 1e9 / hbm_peak,
                          "launches_per_token": gx_launches,
                          "gemv_only": {"what": "the grouped GEMVs alone (planes already quantized)",
                                        "ms_per_token": ms_gr_gemv, "GB/s": gemv_bytes / (ms_gr_gemv * 1e-3) / 1e9,
                                        "tok_per_s_with_lm_head": 1e3 / (ms_gr_gemv + lm_ms)},
                          "quantize_launches": {"what": "a grouped quantize launch before every grouped GEMV",
                                                "ms_per_token": ms_gr, "launches_per_token": gr_launches},
                          "in_gemv_quantize_all_levels": {"what": "down's activation quantized inside its GEMV too",
                                                          "ms_per_token": xq[I.FFN]},
                          "per_matrix": {"what": "one quantize + one GEMV launch per matmul (392 launches), "
                                                 "q|k|v and gate|up on parallel branches",
                                         "ms_per_token": ms_br, "GB/s": sw.bytes / (ms_br * 1e-3) / 1e9,
                                         "gemv_only_ms_per_token": ms_br_gemv},
                          "serial": {"what": "the 392 per-matrix launches as one linear chain",
                                     "ms_per_token": ms, "GB/s": sw.bytes / (ms * 1e-3) / 1e9,
                                     "gemv_only_ms_per_token": ms_gemv}}

    # ---------------- CPU baseline (oracle on the host cores, rank 0 only)
    if dist.rank == 0 and dist.world == 1:
        threads = os.cpu_count() or 1
        v, tokens, secs = cpu_oracle_ffn(args.cpu_seconds, threads)
        v1, tokens1, secs1 = cpu_oracle_ffn(max(0.5, args.cpu_seconds / 2), 1)
        line["cpu_baseline"] = {"value": v, "unit": "TOPS", "cores": threads, "kind": "oracle",
                                "sample": f"first {tokens} of 3314 tokens of the FFN step ({secs:.1f} s)",
                                "single_core": {"value": v1, "unit": "TOPS", "cores": 1,
                                                "sample": f"first {tokens1} of 3314 tokens ({secs1:.1f} s)"}}
    if dist.rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
