#!/usr/bin/env python
"""Benchmark of the RVQ MoE expert-FFN decode layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step = one whole MoE layer (router logits -> top-k + grouping -> gate/up
LUT-GEMV -> SwiGLU reduction -> down LUT-GEMV -> combine + residual) over one
batch.  Default workload: the K3-shaped decode layer (d=7168, f=2048, 256
experts, top-16, 4.23 GB of RVQ codes resident in HBM) at batch 1; each step
takes the next token of a seeded pool, so the routed experts change every
step and the codes stream from HBM (inputs larger than L2).

Workload k3_prefill2048: the same layer shape over a 2048-token chunk with the
Zipf-skewed router bias; every expert group runs on the tensor-core path (RVQ
tiles decoded to bf16 in shared memory, tcgen05 GEMMs).  Its roofline is the
tensor pipe: useful FLOPs (2 per multiply-add of gate, up and down over every
routed token) per launch of the gate/up GEMM.

Prints one JSON line (rank 0).  Multi-GPU (torchrun): independent replicas,
no collective on the data path; value = all ranks' weights / max time.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synth import workloads as W  # noqa: E402

METRIC = "RVQ expert-FFN Gweights/s and code-byte HBM GB/s vs ~8 TB/s peak; layer tok/s"
UNIT = "Gweights/s"
WORKLOADS = {
    # name: (config, batch[, experts in the bank])
    "k3_decode_b1": (2, 1),
    "k3_decode_b1_e64": (2, 1, 64),   # profiling case: same experts, 1.06 GB bank
    "k3_decode_b8": (2, 8),
    "k3_decode_b16": (2, 16),
    "k3_decode_b32": (2, 32),
    "k3_decode_b64": (2, 64),
    "k3_decode_b64_e64": (2, 64, 64),  # profiling case: the two-token GEMV on a 1.06 GB bank
    "decode_d2048_b1": (1, 1),
    "decode_d2048_b4": (1, 4),
    "decode_d2048_b16": (1, 16),
    "k3_prefill2048": (4, 2048),
    "k3_stack8_b1": (3, 1),
    "k3_stack8_b32": (3, 32),
    "k3_prefill512_e64": (4, 512, 64),  # profiling case: ~128 tokens per expert, 1.06 GB bank
    "k3_stack8_prefill2048": (5, 2048),
    # the decode layer on a bank whose codes come from the offline encoder
    # (N(0, 0.02^2) weights, 2 Lloyd rounds per stage) instead of uniform codes
    "k3_decode_b1_encoded": (2, 1, None, "encoded"),
}
# tiered expert store: (config, batch, HBM cache slots, router lookahead per token):
# the 8 K3-shaped layers' records in pinned host memory (34 GB), 256 slots of
# HBM cache (4.25 GB), streamed per layer (moe_layer_forward_streamed)
STREAM_WORKLOADS = {
    "k3_stream8_b1": (3, 1, 256, 0),
    "k3_stream8_b1_lookahead6": (3, 1, 256, 6),
}
# offline encoder: (rows, cols, Lloyd rounds per stage) of one expert matrix,
# Gaussian weights (sigma 0.02); a step encodes the whole matrix
ENCODE_WORKLOADS = {
    "k3_encode_2048x7168_iters8": (2048, 7168, 8),
}
ENCODE_UNIT = "Mweights/s"
# one RVQ matrix times one input vector: (rows, cols, n); the 73.7 KB of codes
# and codebooks stay in L2, so the call is bound by launch latency, not HBM
GEMV_WORKLOADS = {
    "gemv_256x512": (256, 512, 1),
}
ENCODE_METRIC = "offline RVQ encoder: weights encoded per second (3 stages x 256 codewords)"
KERNELS = ["router_logits", "route", "lut_plan", "lut_gemv_gate_up", "swiglu_reduce",
           "lut_gemv_down", "combine"]
DOMINANT = "lut_gemv_gate_up"
L2_BYTES = 129 * 10**6   # GB300 L2
BANK_COPIES = 4          # rotated bank copies for a single layer whose bank is under 2 x L2
# event intervals of the layer call when every expert takes the tensor-core path
KERNELS_TC = ["router_logits", "route", "lut_experts", "prefill_gate_up", "prefill_down",
              "unused", "combine"]
DOMINANT_TC = "prefill_gate_up"
# router logits, top-k selection, grouping, gate/up GEMM, down GEMM, combine
TC_LAUNCHES_PER_STEP = 6


def router_launches(n, E, d):
    """Launches of the layer's router logits: the tensor-core GEMM for a
    prefill-sized bf16 batch (n >= 128, E % 128 == 0, d % 256 == 0) adds the
    split of Wr into three bf16 terms."""
    return 2 if n >= 128 and E % 128 == 0 and d % 256 == 0 else 1


def load_traffic(name):
    """DRAM bytes per launch of `name` from the committed ncu summary, or None
    when a source the kernel is built from changed since that capture."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "lut_gemv_traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(name)
    if not rec:
        return None
    h = hashlib.sha1()
    for rel in rec["sources"]:
        src = os.path.join(ROOT, rel)
        if not os.path.exists(src):
            return None
        h.update(open(src, "rb").read())
    if h.hexdigest() != rec["sources_sha1"]:
        return None
    return int(rec["dram_bytes_per_launch"])


def load_peaks(kind="hbm"):
    """(peak, source): HBM GB/s, or sustained dense bf16 TFLOP/s (the kernels
    are timed inside a seconds-long loop of steps)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        if kind == "tensor":
            return (float(d["bf16_tflops_sustained"]),
                    "measured (sustained bf16; fp16 has the same nominal dense rate)")
        return float(d["hbm_gbs"]), "measured"
    return ((1700.0, "fallback (sustained bf16; fp16 has the same nominal dense rate)")
            if kind == "tensor" else (6800.0, "fallback"))


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML (ctypes on the
    driver's libnvidia-ml) every ~2 ms; reads only."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index: int):
        self.samples = []
        self.ok = False
        self.max_mhz = None
        try:
            import torch
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            uuid = "GPU-" + str(torch.cuda.get_device_properties(cuda_index).uuid)
            self.h = ctypes.c_void_p()
            if self.nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) != 0:
                return
            m = ctypes.c_uint()
            if self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(m)) == 0:
                self.max_mhz = int(m.value)
            self.ok = True
        except Exception:
            self.ok = False

    def _one(self):
        c, r = ctypes.c_uint(), ctypes.c_ulonglong()
        if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(c)) != 0:
            return None
        fn = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nv.nvmlDeviceGetCurrentClocksThrottleReasons
        if fn(self.h, ctypes.byref(r)) != 0:
            r.value = 0
        return (time.perf_counter(), int(c.value), int(r.value))

    def start(self):
        self._stop = threading.Event()
        if not self.ok:
            return

        def run():
            while not self._stop.is_set():
                s = self._one()
                if s:
                    self.samples.append(s)
                time.sleep(0.002)
        self.th = threading.Thread(target=run, daemon=True)
        self.th.start()

    def stop(self):
        self._stop.set()
        if self.ok:
            self.th.join()

    def summary(self, t0, t1):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [],
                    "note": "NVML unavailable"}
        win = [s for s in self.samples if t0 <= s[0] <= t1] or self.samples
        bits = 0
        for s in win:
            bits |= s[2]
        return {"sm_mhz": statistics.median(s[1] for s in win), "sm_max_mhz": self.max_mhz,
                "reasons": [n for b, n in self.REASONS.items() if bits & b],
                "samples": len(win)}


# ---------------------------------------------------------------- GPU arm
def workload_shape(name):
    spec = WORKLOADS[name]
    config, batch = spec[0], spec[1]
    s = W.WORKLOADS[config].shape
    if len(spec) > 2 and spec[2] is not None:
        s = W.LayerShape(s.d, s.f, spec[2], s.k)
    return config, batch, s


def encoded_bank(name):
    spec = WORKLOADS.get(name, ())
    return len(spec) > 3 and spec[3] == "encoded"


def router_bias(config, src):
    wl = W.WORKLOADS[config]
    if not wl.is_prefill:
        return None
    return W.zipf_bias(src.lseed, src.shape.E, wl.zipf_beta)


def build_layer(config, device, k=None, shape=None, layer=0, encoded=False):
    from moe_expert_ffn_router_gb300.layer import MoeLayer
    s = shape or W.WORKLOADS[config].shape
    src = W.ExpertSource(config, layer, s)
    L = MoeLayer(s.E, s.d, s.f, k or s.k, layer=layer, device=device)
    if encoded:
        encode_experts(L, s, device, seed=1000 * layer + config)
    for e in range(s.E if encoded else 0, s.E):
        mats = [(src.codes(e, m), src.codebooks(e, m)) for m in range(3)]
        L.load_expert(e, mats[0][0], mats[1][0], mats[2][0], np.stack([c for _, c in mats]))
    L.set_router(src.router_weight(), router_bias(config, src))
    L.validate()
    return L, src


def encode_experts(L, s, device, seed, iters=2, sigma=0.02):
    """Every expert's gate, up and down matrix drawn N(0, sigma^2) on the
    device (a seeded generator per matrix) and encoded by rvq_encode."""
    import torch
    import moe_expert_ffn_router_gb300 as rvq
    shapes = [(s.f, s.d), (s.f, s.d), (s.d, s.f)]
    ws = torch.empty(max(rvq.rvq_encode_workspace_bytes(r, c) for r, c in shapes),
                     dtype=torch.uint8, device=device)
    gen = torch.Generator(device=device)
    for e in range(s.E):
        codes, cbs = [], []
        for m, (r, c) in enumerate(shapes):
            gen.manual_seed(seed * 1_000_003 + e * 3 + m)
            w = torch.randn((r, c), generator=gen, device=device) * sigma
            cd = torch.empty((r, c // 8, 3), dtype=torch.uint8, device=device)
            cb = torch.empty((3, 256, 8), dtype=torch.float32, device=device)
            rvq.rvq_encode(w, r, c, iters, cd, cb, ws)
            codes.append(cd)
            cbs.append(cb)
        L.load_expert(e, codes[0], codes[1], codes[2], torch.stack(cbs))
    torch.cuda.synchronize(device)


def replica_max_ms(ms, world, device):
    """The slowest replica's time in ms: the whole job ends when its last
    rank does (replicas only; the one collective of the bench)."""
    if world <= 1:
        return float(ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, world, ms):
    """Whole-job throughput: the units all ranks processed over the slowest
    rank's time (every replica runs the same seeded workload)."""
    return units_per_rank * world / (ms / 1e3)


def run_gpu(args, rank, world, local_rank):
    import torch
    import moe_expert_ffn_router_gb300 as rvq

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    config, batch, s = workload_shape(args.workload)
    prefill = W.WORKLOADS[config].is_prefill
    tc_min = 1 if prefill else 0
    if args.tc_min_tokens is not None:
        tc_min = args.tc_min_tokens
    kernels = KERNELS_TC if tc_min > 0 else KERNELS
    n_layers = W.WORKLOADS[config].n_layers
    encoded = encoded_bank(args.workload)
    weights_per_expert = 3 * s.d * s.f
    code_bytes_per_expert = 3 * (3 * s.d * s.f // 8)
    # a single layer whose bank is under twice the L2 is timed on BANK_COPIES
    # seeded copies (other seeds, the same shapes), step i on copy i mod
    # BANK_COPIES, so that a step does not find the previous steps' experts in L2
    rot = BANK_COPIES if n_layers == 1 and code_bytes_per_expert * s.E < 2 * L2_BYTES else 1
    built = [build_layer(config, dev, shape=s, layer=i, encoded=encoded)
             for i in range(max(n_layers, rot))]
    L, src = built[0]
    from moe_expert_ffn_router_gb300.layer import MoeStack
    stack = MoeStack([b[0] for b in built[:n_layers]])
    copies = [b[0] for b in built] if n_layers == 1 else [L]
    copy_bufs = [stack.buffers(batch)[0]] + [Lc.buffers(batch) for Lc in copies[1:]]
    if prefill:
        pool_bits = src.tokens_bf16(2 * batch)          # two chunks, alternating
    else:
        pool = max(64, 4 * batch)
        pool_bits = src.tokens_bf16(pool * batch if batch > 1 else pool)
    xs = torch.from_numpy(pool_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    xs = xs.reshape(-1, batch, s.d)
    nsteps = xs.shape[0]
    assert nsteps % rot == 0, "each token-pool entry keeps one bank copy"
    cb_bytes_per_expert = 3 * rvq.RVQ_CODEBOOK_BYTES

    def forward(x, events=None, r=0):
        # one layer: the layer itself (router -> top-k -> FFN -> combine +
        # residual), on bank copy r; a stack: pre-norm + layer, per layer
        if n_layers == 1:
            return [copies[r].forward(x, copy_bufs[r], events=events, tc_min_tokens=tc_min)]
        return stack.forward(x, events=events, tc_min_tokens=tc_min)

    def step(i, events=None):
        return forward(xs[i % nsteps], events=events, r=i % rot)

    # unique experts per step, summed over the layers (from the routing the
    # GPU computed); the pool is replayed identically in the timed loop, so
    # count once per pool entry
    uniq, uniq0 = [], []
    for i in range(nsteps):
        bl = step(i)
        torch.cuda.synchronize()
        per = [len(set(b["idx"].cpu().numpy().reshape(-1).tolist())) for b in bl]
        uniq.append(sum(per))
        uniq0.append(per[0])
    for Lx in stack.layers + copies[1:]:
        rc, bits = Lx.status(batch)
        if rc != 0:
            raise RuntimeError(f"device status {rc} bits {bits:#x}")

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(run_step):
        for i in range(args.warmup):
            run_step(i)
        barrier()
        e0.record()
        for i in range(args.steps):
            run_step(args.warmup + i)
        e1.record()
        barrier()
        return replica_max_ms(e0.elapsed_time(e1), world, dev)

    # A single layer is also timed as one CUDA graph per step
    # (moe_layer_graph_launch: the layer's launches recorded once per
    # token-pool entry and replayed).  The kernel launches, with programmatic
    # dependent launch between them and from one step into the next, are the
    # timed value unless --graph: a graph boundary ends that overlap (the next
    # step's router cannot start behind the previous step's combine), and the
    # replays measured slower (0.092-0.099 against 0.089 ms per K3 decode step).
    graphs = ([copies[j % rot].graph(xs[j], copy_bufs[j % rot], tc_min_tokens=tc_min)
               for j in range(nsteps)] if n_layers == 1 else [])
    use_graph = bool(graphs) and args.graph
    ms_other = timed(step if use_graph else (lambda i: graphs[i % nsteps].launch())) \
        if graphs else None
    sampler = ClockSampler(local_rank)
    sampler.start()
    t0w = time.perf_counter()
    ms = timed((lambda i: graphs[i % nsteps].launch()) if use_graph else step)
    t1w = time.perf_counter()
    sampler.stop()
    clocks = sampler.summary(t0w, t1w)
    for g in graphs:
        g.close()

    steps_idx = [(args.warmup + i) % nsteps for i in range(args.steps)]
    experts_total = sum(uniq[j] for j in steps_idx)
    value = job_rate(experts_total * weights_per_expert, world, ms) / 1e9
    code_gbs = job_rate(experts_total * (code_bytes_per_expert + cb_bytes_per_expert), world,
                        ms) / 1e9
    tok_s = job_rate(batch * args.steps, world, ms)

    # ---- per-kernel durations (events between kernels, same steps) ----
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(rvq.MOE_LAYER_EVENTS)]
    for e in evs:
        e.record()
    torch.cuda.synchronize()
    per = {k: [] for k in kernels}
    for i in range(args.steps):
        step(args.warmup + i, events=evs)
        torch.cuda.synchronize()
        for j, name in enumerate(kernels):
            per[name].append(evs[j].elapsed_time(evs[j + 1]))
    avg = {k: float(np.mean(v)) for k, v in per.items() if k != "unused"}
    # decode batches on lookup tables: the routing launch writes the pair plan
    # and the down GEMV reduces its own SwiGLU inputs, so those two event
    # intervals hold no launch
    fused = tc_min == 0 and batch <= 16
    fused_swiglu = fused and s.d // 256 <= 32 and batch <= 4
    if fused:
        avg.pop("lut_plan", None)
    if fused_swiglu:
        avg.pop("swiglu_reduce", None)
    if tc_min > 0:
        # useful FLOPs: 2 per multiply-add, gate + up (2 d f) then down (d f)
        # for each of the n k routed (token, expert) pairs
        pairs = batch * s.k
        gu_flops = 2.0 * 2 * s.d * s.f * pairs
        dn_flops = 2.0 * s.d * s.f * pairs
        peak, peak_kind = load_peaks("tensor")
        achieved = gu_flops / (avg[DOMINANT_TC] / 1e3) / 1e12
        ffn_tflops = (gu_flops + dn_flops) / (
            (avg["prefill_gate_up"] + avg["prefill_down"]) / 1e3) / 1e12
        roofline = {"kernel": DOMINANT_TC, "bound": "tensor", "achieved": round(achieved, 1),
                    "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                    "peak_source": peak_kind, "traffic": None,
                    "algorithmic_flops_per_launch": int(gu_flops),
                    "avg_launch_us": round(avg[DOMINANT_TC] * 1e3, 2),
                    "timing": "a second pass over the timed steps with an event between "
                              "kernels (serialised, programmatic dependent launch off); "
                              "launch latency included",
                    "ffn_tflops": round(ffn_tflops, 1),
                    "ffn_frac": round(ffn_tflops / peak, 4)}
    else:
        # algorithmic bytes of the gate/up launch: gate + up codes and
        # codebooks of every unique selected expert
        gu_bytes = np.mean([uniq0[j] for j in steps_idx]) * 2 * (
            3 * s.d * s.f // 8 + rvq.RVQ_CODEBOOK_BYTES)
        peak, peak_kind = load_peaks()
        achieved = gu_bytes / (avg[DOMINANT] / 1e3) / 1e9
        roofline = {"kernel": DOMINANT, "bound": "hbm", "achieved": round(achieved, 1),
                    "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                    "peak_source": peak_kind,
                    "traffic": load_traffic(DOMINANT) if (s.E == 256 and batch == 1
                                                          and n_layers == 1) else None,
                    "algorithmic_bytes_per_launch": int(gu_bytes),
                    "avg_launch_us": round(avg[DOMINANT] * 1e3, 2),
                    "timing": "a second pass over the timed steps with an event between "
                              "kernels (serialised, programmatic dependent launch off); "
                              "launch latency included"}

    # ---- end to end through host buffers ----
    pinned_in = torch.from_numpy(pool_bits.view(np.int16).copy()).reshape(-1, batch, s.d)
    pinned_in = pinned_in.pin_memory()
    pinned_out = torch.empty((batch, s.d), dtype=torch.float32).pin_memory()
    xbuf = torch.empty((batch, s.d), dtype=torch.bfloat16, device=dev)
    out_last = stack.buffers(batch)[-1]["out"]

    pin_bf16 = pinned_in.view(torch.bfloat16)

    def e2e_step(i):
        if n_layers == 1:
            # the library's host-buffer layer call (moe_layer_forward_host)
            r = i % rot
            copies[r].forward_host(pin_bf16[i % nsteps], pinned_out, copy_bufs[r],
                                   tc_min_tokens=tc_min)
            return
        # a stack: its input copied in and its output copied back around it
        xbuf.view(torch.int16).copy_(pinned_in[i % nsteps], non_blocking=True)
        forward(xbuf)
        pinned_out.copy_(out_last, non_blocking=True)

    if use_graph:
        # the copies in and out recorded in each step's graph
        graphs = [copies[j % rot].graph(xbuf, copy_bufs[j % rot], x_host=pin_bf16[j],
                                        out_host=pinned_out, tc_min_tokens=tc_min)
                  for j in range(nsteps)]
        ms_e2e = timed(lambda i: graphs[i % nsteps].launch())
        for g in graphs:
            g.close()
    else:
        ms_e2e = timed(e2e_step)
    e2e = {"value": round(job_rate(experts_total * weights_per_expert, world, ms_e2e) / 1e9, 2),
           "unit": UNIT,
           "h2d_bytes_per_step": batch * s.d * 2, "d2h_bytes_per_step": batch * s.d * 4}
    for Lx in stack.layers + copies[1:]:
        rc, bits = Lx.status(batch)
        if rc != 0:
            raise RuntimeError(f"device status {rc} bits {bits:#x}")
    launch = {"mode": "one CUDA graph per step (moe_layer_graph_launch)" if use_graph
              else "the layer's kernel launches, programmatic dependent launch between them"}
    if ms_other is not None:
        launch["kernel_launches_ms_per_step" if use_graph else "graph_ms_per_step"] = round(
            ms_other / args.steps, 4)
    res = dict(value=value, ms=ms, code_gbs=code_gbs, tok_s=tok_s, roofline=roofline, e2e=e2e,
               launch=launch,
               clocks=clocks, kernels_us={k: round(v * 1e3, 2) for k, v in avg.items()},
               uniq_mean=float(np.mean([uniq[j] for j in steps_idx])),
               launches=((TC_LAUNCHES_PER_STEP if tc_min == 1 else len(KERNELS) if tc_min == 0
                          else len(KERNELS) + TC_LAUNCHES_PER_STEP - 3)
                         + router_launches(batch, s.E, s.d) - 1
                         # a stack's pre-norm: inside the router launch for one token
                         + (1 if n_layers > 1 and batch > 1 else 0)
                         # decode batches on lookup tables: the pair plan inside the routing
                         # launch, the SwiGLU reduction inside the down GEMV
                         - (1 if fused else 0) - (1 if fused_swiglu else 0))
                        * args.steps * n_layers,
               config=config, batch=batch, shape=s, prefill=prefill, layers=n_layers,
               bank_copies=rot)
    del L, stack, built, copies, copy_bufs
    return res


# ------------------------------------------------------------- CPU oracle
def host_cores():
    """Host cores this process may run on (its CPU affinity)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OracleBatch:
    """One batch of the workload through the oracle as it stands: router
    logits and top-k for the batch, every (token, expert) pair's expert FFN
    (explicit dequantisation, fp64 matmuls), the weighted combine.  The pairs
    run on a thread pool in this harness (the C oracle releases the GIL); the
    oracle itself is single-threaded code."""

    def __init__(self, config, shape, tokens_bf16):
        import oracle
        import synth
        self.oracle = oracle
        self.s = s = shape
        self.src = src = W.ExpertSource(config, 0, s)
        self.wr = src.router_weight()
        self.bias = router_bias(config, src)
        self.x64 = synth.bf16_to_f32(tokens_bf16).astype(np.float64)
        lg = oracle.router_logits(self.wr, self.x64, self.bias).astype(np.float32)
        self.idx, _, _ = oracle.route(lg, s.k)
        self.mats = {}

    def experts(self, rows):
        """Generate (outside any timing) the experts the given tokens route to."""
        for t in rows:
            for e in self.idx[t]:
                e = int(e)
                if e not in self.mats:
                    self.mats[e] = tuple((self.src.codes(e, m), self.src.codebooks(e, m))
                                         for m in range(3))

    def run(self, rows, pairs=None, threads=1):
        """The oracle layer on tokens `rows` (all their pairs, or the first
        `pairs` of them when given: a bounded sample).  Returns seconds."""
        from concurrent.futures import ThreadPoolExecutor
        o, s = self.oracle, self.s
        self.experts(rows)
        t0 = time.perf_counter()
        x = self.x64[rows]
        lg = o.router_logits(self.wr, x, self.bias).astype(np.float32)
        idx, w, _ = o.route(lg, s.k)
        work = [(i, int(e)) for i in range(len(rows)) for e in idx[i]]
        if pairs is not None:
            work = work[:pairs]

        def ffn(item):
            i, e = item
            return o.expert_ffn(*self.mats[e], s.d, s.f, x[i])

        if threads > 1:
            with ThreadPoolExecutor(max_workers=threads) as ex:
                ys = list(ex.map(ffn, work))
        else:
            ys = [ffn(it) for it in work]
        if pairs is None:
            o.combine(np.stack(ys), w, x)
        return time.perf_counter() - t0


def oracle_baseline(config, shape, batch, layers, uniq_mean, tokens_bf16):
    """cpu_baseline of the GPU arm: the oracle on the host's cores (threads over
    the (token, expert) pairs of one batch), and on one core (a sample of
    pairs), scaled to the workload's batch, layers and distinct experts."""
    s = shape
    cores = host_cores()
    pairs_batch = batch * s.k
    ob = OracleBatch(config, s, tokens_bf16)
    rows = list(range(min(batch, max(1, (4 * cores) // s.k))))
    ob.experts(rows)
    # all cores: whole tokens (every pair of each) while that stays bounded
    t_all = ob.run(rows, threads=cores)
    pairs_all = len(rows) * s.k
    step_all = t_all / pairs_all * pairs_batch * layers
    # one core: two pairs of the first token
    t_one = ob.run([0], pairs=2, threads=1)
    step_one = t_one / 2 * pairs_batch * layers
    weights = uniq_mean * layers * 3 * s.d * s.f   # every layer's distinct experts
    return {"value": round(weights / step_all / 1e9, 6), "unit": UNIT, "cores": cores,
            "kind": "oracle",
            "single_thread": {"value": round(weights / step_one / 1e9, 6), "cores": 1,
                              "s_per_pair": round(t_one / 2, 3)},
            "sample": f"{len(rows)} token(s), {pairs_all} (token, expert) pairs through the "
                      f"oracle layer on {cores} threads ({t_all:.2f} s; one core: 2 pairs, "
                      f"{t_one:.2f} s), scaled to the {batch}-token batch ({pairs_batch} pairs), "
                      f"{layers} layer(s) and {uniq_mean:.1f} distinct experts per layer"}


def oracle_unique_experts(config, batch, src, s):
    """Distinct experts the oracle router selects for the workload's first batch."""
    import oracle
    import synth
    x64 = synth.bf16_to_f32(src.tokens_bf16(batch)).astype(np.float64)
    lg = oracle.router_logits(src.router_weight(), x64, router_bias(config, src))
    idx, _, _ = oracle.route(lg.astype(np.float32), s.k)
    return len(set(idx.reshape(-1).tolist()))


def reference_arm(args, rank):
    """The oracle as the reference implementation, on the host's cores (threads
    over the (token, expert) pairs in this harness).  A step is one batch of
    the workload through the oracle layer: every pair when the batch has at
    most 4 pairs per core, otherwise a stated sample of 4 pairs per core
    (value scaled to the whole batch).  steps / ms_per_step report what ran:
    when the requested steps would take more than ~150 s, fewer run."""
    if rank != 0:
        return
    if args.workload in GEMV_WORKLOADS:
        return reference_gemv(args)
    config, batch, s = workload_shape(args.workload)
    src = W.ExpertSource(config, 0, s)
    cores = host_cores()
    layers = W.WORKLOADS[config].n_layers
    pool = max(8, args.steps + args.warmup)
    bits = src.tokens_bf16(pool * batch).reshape(pool, batch, s.d)
    full = batch * s.k <= 4 * cores
    sample_pairs = None if full else 4 * cores
    ob = OracleBatch(config, s, bits.reshape(-1, s.d))
    uniq = layers * (s.k if batch == 1 else oracle_unique_experts(config, batch, src, s))
    budget_s = 150.0
    times, ran = [], 0
    t_start = time.perf_counter()
    total = args.warmup + args.steps
    for i in range(total):
        # the whole batch, or its first tokens up to 4 pairs per core
        rows = list(range(i * batch, i * batch + (batch if full else
                                                    max(1, sample_pairs // s.k))))
        dt = ob.run(rows, pairs=sample_pairs, threads=cores)
        if i >= args.warmup:
            times.append(dt)
            ran += 1
        elapsed = time.perf_counter() - t_start
        if ran >= 1 and elapsed + dt > budget_s:  # the next step would pass the budget
            break
    per_step = float(np.mean(times))                    # seconds per step as run
    npairs = batch * s.k if full else sample_pairs
    step_s = per_step / npairs * batch * s.k * layers   # the whole batch, every layer
    value = uniq * 3 * s.d * s.f / step_s / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
            "n_gpus": args.gpus, "steps": ran, "warmup": args.warmup,
            "steps_requested": args.steps, "ms_per_step": round(per_step * 1e3, 2),
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload + ":" + W.WORKLOADS[config].name,
                       "batch": batch, "experts": s.E, "layers": layers},
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores,
                             "kind": "oracle",
                             "sample": (f"every step is one whole {batch}-token batch "
                                        f"({batch * s.k} (token, expert) pairs) of layer 0"
                                        if full else
                                        f"every step is {sample_pairs} of the batch's "
                                        f"{batch * s.k} (token, expert) pairs")
                                       + f" on {cores} threads; value scaled to "
                                       f"{layers} layer(s) and {uniq} distinct experts"
                                       + ("" if full else " and the whole batch")},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def gemv_inputs(rows, cols, n):
    """The single-matrix workload's seeded inputs: canonical codes, codebooks
    and fp32 x (N(0, 1)), from the generator of the layer workloads."""
    import synth
    mseed = W.matrix_seed(W.layer_seed(0, 0), 0, 0)
    codes = W.codes(mseed, rows, cols)
    cb = W.codebooks(mseed)
    x = W.tokens_f32(W.layer_seed(0, 0), n, cols)
    return codes, cb, x


def run_gemv(args, rank, world, local_rank):
    """rvq_gemv on one 256 x 512 matrix (fp32 input, batch 1) per step: the
    single-GEMV configuration.  L2-resident, so the figure is latency, not a
    fraction of HBM bandwidth (reported as such)."""
    import torch
    import moe_expert_ffn_router_gb300 as rvq
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    rows, cols, n = GEMV_WORKLOADS[args.workload]
    codes, cb, x = gemv_inputs(rows, cols, n)
    packed = torch.empty(rvq.rvq_code_bytes(rows, cols), dtype=torch.uint8, device=dev)
    rvq.rvq_pack(torch.from_numpy(codes).to(dev), rows, cols, packed)
    cbp = torch.empty(6144, dtype=torch.float32, device=dev)
    rvq.rvq_pack_codebooks(torch.from_numpy(cb).to(dev), cbp)
    xd = torch.from_numpy(x).to(dev)
    y = torch.empty((n, rows), dtype=torch.float32, device=dev)
    ws = torch.empty(rvq.rvq_gemv_workspace_bytes(rows, cols, n), dtype=torch.uint8, device=dev)
    rvq.rvq_ws_clear(ws)
    for _ in range(args.warmup):
        rvq.rvq_gemv(packed, cbp, rows, cols, xd, n, y, ws)
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank)
    sampler.start()
    t0w = time.perf_counter()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        rvq.rvq_gemv(packed, cbp, rows, cols, xd, n, y, ws)
    e1.record()
    torch.cuda.synchronize()
    t1w = time.perf_counter()
    sampler.stop()
    ms = replica_max_ms(e0.elapsed_time(e1), world, dev)
    rc, bits = rvq.rvq_ws_status(ws)
    if rc != 0:
        raise RuntimeError(f"device status {rc} bits {bits:#x}")
    # end to end: x from pinned host memory, y back, each step
    xh = torch.from_numpy(x).pin_memory()
    yh = torch.empty((n, rows), dtype=torch.float32).pin_memory()
    e0.record()
    for _ in range(args.steps):
        xd.copy_(xh, non_blocking=True)
        rvq.rvq_gemv(packed, cbp, rows, cols, xd, n, y, ws)
        yh.copy_(y, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    ms_e2e = replica_max_ms(e0.elapsed_time(e1), world, dev)
    weights = rows * cols * n
    us = ms / args.steps * 1e3
    algo_bytes = 3 * rows * cols // 8 + rvq.RVQ_CODEBOOK_BYTES + n * cols * 4
    peak, peak_kind = load_peaks()
    ach = algo_bytes / (us / 1e6) / 1e9
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        reps = 20
        t0 = time.perf_counter()
        for _ in range(reps):
            oracle.rvq_gemv(codes, cb, rows, cols, x.astype(np.float64))
        dt = (time.perf_counter() - t0) / reps
        cpu = {"value": round(weights / dt / 1e9, 6), "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"the oracle GEMV (explicit dequant, fp64) on the same matrix, "
                         f"{reps} calls, {dt * 1e3:.2f} ms per call"}
    line = {
        "metric": METRIC, "value": round(job_rate(weights * args.steps, world, ms) / 1e9, 3),
        "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms / args.steps, 5), "us_per_call": round(us, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": args.workload + ":" + W.WORKLOADS[0].name, "rows": rows,
                   "cols": cols, "batch": n,
                   "l2": "L2-resident: 73.7 KB of codes and codebooks, reused every step",
                   "parallelism": f"replicas{world}", "path": "fp32 lookup tables"},
        "roofline": {"bound": "hbm", "achieved": round(ach, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(ach / peak, 5), "peak_source": peak_kind, "traffic": None,
                     "algorithmic_bytes_per_launch": algo_bytes,
                     "note": "L2-resident and launch-latency bound: the fraction is "
                             "reported, not a target"},
        "cpu_baseline": cpu,
        "e2e": {"value": round(job_rate(weights * args.steps, world, ms_e2e) / 1e9, 3),
                "unit": UNIT, "h2d_bytes_per_step": n * cols * 4,
                "d2h_bytes_per_step": n * rows * 4,
                "note": "x copied from pinned host memory and y back around each call"},
        "clocks": sampler.summary(t0w, t1w),
        # plan, GEMV, slot reduction
        "gpu_launches": 3 * args.steps * world,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def reference_gemv(args):
    """The oracle GEMV (explicit dequantisation, fp64 dot products) per step."""
    import oracle
    rows, cols, n = GEMV_WORKLOADS[args.workload]
    codes, cb, x = gemv_inputs(rows, cols, n)
    x64 = x.astype(np.float64)
    for _ in range(args.warmup):
        oracle.rvq_gemv(codes, cb, rows, cols, x64)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.rvq_gemv(codes, cb, rows, cols, x64)
    dt = (time.perf_counter() - t0) / args.steps
    value = rows * cols * n / dt / 1e9
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "rows": rows, "cols": cols, "batch": n},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": "the whole workload, every step"},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}), flush=True)


def run_stream(args, rank, world, local_rank):
    """The tiered expert store: every layer's records in pinned host memory, an
    HBM cache of record slots, misses copied per layer after routing (and the
    next layer's predicted experts prefetched with lookahead).  A step is one
    batch through the whole stack, host reads of the routing included."""
    import torch
    import moe_expert_ffn_router_gb300 as rvq
    from moe_expert_ffn_router_gb300.layer import MoeStreamedStack
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    config, batch, slots, lookahead = STREAM_WORKLOADS[args.workload]
    wl = W.WORKLOADS[config]
    s = wl.shape
    layers = [build_layer(config, dev, shape=s, layer=i)[0] for i in range(wl.n_layers)]
    src = W.ExpertSource(config, 0, s)
    st = MoeStreamedStack(layers, slots=slots, lookahead=lookahead)
    del layers
    torch.cuda.empty_cache()
    pool = max(64, 4 * batch)
    bits = src.tokens_bf16(pool * batch)
    host_x = torch.from_numpy(bits.view(np.int16)).reshape(pool, batch, s.d).pin_memory()
    xbuf = torch.empty((batch, s.d), dtype=torch.bfloat16, device=dev)
    out_host = torch.empty((batch, s.d), dtype=torch.float32).pin_memory()
    uniq = []

    def step(i, count=False):
        xbuf.view(torch.int16).copy_(host_x[i % pool], non_blocking=True)
        bufs = st.forward(xbuf)
        out_host.copy_(bufs[-1]["out"], non_blocking=True)
        if count:
            uniq.append(sum(int((torch.diff(b["offsets"]) > 0).sum()) for b in bufs))

    sampler = ClockSampler(local_rank)
    sampler.start()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    s0 = st.stats()
    t0w = time.perf_counter()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        step(args.warmup + i)
    e1.record()
    torch.cuda.synchronize()
    t1w = time.perf_counter()
    sampler.stop()
    ms = replica_max_ms(e0.elapsed_time(e1), world, dev)
    s1 = st.stats()
    for i in range(args.steps):  # the routed experts of the same steps (not timed)
        step(args.warmup + i, count=True)
    torch.cuda.synchronize()
    rc, bits_st = st.status(batch)
    if rc != 0:
        raise RuntimeError(f"device status {rc} bits {bits_st:#x}")
    d = {k: s1[k] - s0[k] for k in ("hits", "misses", "prefetched", "prefetch_used",
                                     "bytes_copied")}
    experts_total = sum(uniq)
    weights = experts_total * 3 * s.d * s.f
    value = job_rate(weights, world, ms) / 1e9
    rb = st.host.numel() // (wl.n_layers * s.E)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": args.workload + ":" + wl.name, "batch": batch,
                   "layers": wl.n_layers, "d": s.d, "f": s.f, "experts": s.E, "top_k": s.k,
                   "host_bank_gb": round(st.host.numel() / 1e9, 2),
                   "hbm_cache_slots": slots, "hbm_cache_gb": round(slots * rb / 1e9, 2),
                   "lookahead": lookahead,
                   "l2": "records stream from host memory every step (4.25 GB cache, 34 GB bank)",
                   "parallelism": f"replicas{world}", "path": "fp32 lookup tables, streamed"},
        "tok_s": round(job_rate(batch * args.steps, world, ms), 2),
        "stream": {"hit_rate": round(d["hits"] / max(1, d["hits"] + d["misses"]), 4),
                   "misses_per_step": round(d["misses"] / args.steps, 2),
                   "prefetched_per_step": round(d["prefetched"] / args.steps, 2),
                   "prefetch_used": d["prefetch_used"],
                   "h2d_gbs": round(d["bytes_copied"] / (ms / 1e3) / 1e9, 1)},
        "roofline": None,
        "roofline_note": "bound by the host -> HBM record copies (h2d_gbs), not a kernel",
        "cpu_baseline": None,
        "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step":
                batch * s.d * 2 + d["bytes_copied"] // args.steps,
                "d2h_bytes_per_step": batch * s.d * 4},
        "clocks": sampler.summary(t0w, t1w),
        # per layer: norm, router, top-k, pair plan, 2 GEMVs, SwiGLU, combine (+ the
        # lookahead router of the next layer)
        # per layer: norm, router logits, route, pair plan, gate/up GEMV,
        # SwiGLU reduction (inside the down GEMV up to 4 tokens), down GEMV,
        # combine; lookahead adds the next layer's router
        "gpu_launches": args.steps * (wl.n_layers * (7 if batch <= 4 and s.d // 256 <= 32 else 8)
                                      + (wl.n_layers - 1 if lookahead else 0)),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    st.close()


def encode_ops_per_step(rows, cols, iters):
    """fp32 lane operations of the nearest-codeword search per step: 8
    subtractions and 8 fused multiply-adds per (sub-vector, codeword), 256
    codewords, iters + 1 searches per stage, 3 stages."""
    return rows * cols // 8 * 256 * 16 * (iters + 1) * 3


def run_encode(args, rank, world, local_rank):
    """The offline RVQ encoder over one K3 expert matrix per step (inputs in
    HBM; the 58.7 MB matrix and its residual stay in L2 between passes, which
    is the kernel's own reuse, not a cache carried over from the last step:
    each step starts from w)."""
    import torch
    import moe_expert_ffn_router_gb300 as rvq
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    rows, cols, iters = ENCODE_WORKLOADS[args.workload]
    w_host = torch.from_numpy(np.random.default_rng(2024).normal(
        0, 0.02, size=(rows, cols)).astype(np.float32)).pin_memory()
    w = w_host.to(dev)
    codes = torch.empty((rows, cols // 8, 3), dtype=torch.uint8, device=dev)
    cb = torch.empty((3, 256, 8), dtype=torch.float32, device=dev)
    ws = torch.empty(rvq.rvq_encode_workspace_bytes(rows, cols), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # > L2, written between steps
    codes_host = torch.empty(codes.shape, dtype=torch.uint8).pin_memory()
    stream = torch.cuda.current_stream(dev)

    def timed(k, e2e):
        evs = []
        tot = 0.0
        for i in range(k):
            flush.fill_(i & 0xFF)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            if e2e:
                w.copy_(w_host, non_blocking=True)
            rvq.rvq_encode(w, rows, cols, iters, codes, cb, ws, stream=stream)
            if e2e:
                codes_host.copy_(codes, non_blocking=True)
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize()
        for a, b in evs:
            tot += a.elapsed_time(b)
        return tot

    for _ in range(args.warmup):
        rvq.rvq_encode(w, rows, cols, iters, codes, cb, ws, stream=stream)
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank)
    sampler.start()
    t0w = time.perf_counter()
    ms = replica_max_ms(timed(args.steps, False), world, dev)
    t1w = time.perf_counter()
    sampler.stop()
    ms_e2e = replica_max_ms(timed(args.steps, True), world, dev)
    weights = rows * cols
    value = job_rate(weights * args.steps, world, ms) / 1e6
    clocks = sampler.summary(t0w, t1w)
    ops = encode_ops_per_step(rows, cols, iters)
    peak = 152 * 128 * 2070e6 / 1e12  # fp32 lanes x maximum SM clock, T lane-ops/s
    ach = ops / (ms / args.steps / 1e3) / 1e12
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = encode_cpu_sample(cols, iters)
    line = {
        "metric": ENCODE_METRIC, "value": round(value, 2), "unit": ENCODE_UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": args.workload, "rows": rows, "cols": cols, "iters": iters,
                   "weights": "Gaussian, sigma 0.02, seed 2024",
                   "l2": "a 256 MB buffer is written between timed steps (flush)",
                   "parallelism": f"replicas{world}"},
        "roofline": {"bound": "alu", "achieved": round(ach, 2), "peak": round(peak, 2),
                     "unit": "T fp32 lane-ops/s", "frac": round(ach / peak, 3), "traffic": None,
                     "scope": "whole step (nearest-codeword search ops / step time); the "
                              "search kernel is nearly all of the step",
                     "peak_source": "152 SMs x 128 fp32 lanes x 2070 MHz maximum SM clock"},
        "cpu_baseline": cpu,
        "e2e": {"value": round(job_rate(weights * args.steps, world, ms_e2e) / 1e6, 2),
                "unit": ENCODE_UNIT, "h2d_bytes_per_step": weights * 4,
                "d2h_bytes_per_step": weights // 8 * 3},
        "clocks": clocks,
        # copy of w into the workspace is a memcpy; per stage: init, (iters) x
        # (search + update), last search, finish
        "gpu_launches": args.steps * 3 * (2 * iters + 3),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def encode_cpu_sample(cols, iters, rows=512):
    """The oracle encoder on a rows x cols slice of the same kind of matrix (the
    search cost per weight does not depend on the row count)."""
    import oracle
    w = np.random.default_rng(2024).normal(0, 0.02, size=(rows, cols)).astype(np.float32)
    t0 = time.perf_counter()
    oracle.rvq_encode(w, iters)
    dt = time.perf_counter() - t0
    return {"value": round(rows * cols / dt / 1e6, 4), "unit": ENCODE_UNIT, "cores": 1,
            "kind": "oracle",
            "sample": f"oracle encoder on a {rows} x {cols} slice, {iters} rounds "
                      f"({dt:.1f} s)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 200; 10 for --impl reference, whose steps "
                         "take about a second of CPU time each)")
    ap.add_argument("--warmup", type=int, default=None, help="untimed steps (default 10; 3)")
    ap.add_argument("--workload", default="k3_decode_b1",
                    choices=sorted(WORKLOADS) + sorted(STREAM_WORKLOADS) +
                    sorted(ENCODE_WORKLOADS) + sorted(GEMV_WORKLOADS))
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--tc-min-tokens", type=int, default=None,
                    help="experts with at least this many tokens take the tensor-core path "
                         "(default: 1 for the prefill workload, 0 = lookup tables only, otherwise)")
    ap.add_argument("--graph", action="store_true",
                    help="time one CUDA graph per step (moe_layer_graph_launch) instead of the "
                         "layer's kernel launches")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle timing (profiling runs)")
    args = ap.parse_args()
    ref = args.impl == "reference"
    if args.steps is None:
        args.steps = 10 if ref else 200
    if args.warmup is None:
        args.warmup = 3 if ref else 10
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference" and args.workload in ENCODE_WORKLOADS:
        if rank == 0:
            rows, cols, iters = ENCODE_WORKLOADS[args.workload]
            cpu = encode_cpu_sample(cols, iters)
            print(json.dumps({
                "impl": "reference", "metric": ENCODE_METRIC, "value": cpu["value"],
                "unit": ENCODE_UNIT, "n_gpus": args.gpus, "steps": 1, "warmup": 0,
                "ms_per_step": round(rows * cols / cpu["value"] / 1e3, 1),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f32", "data": "synthetic",
                "config": {"workload": args.workload, "rows": rows, "cols": cols, "iters": iters},
                "cpu_baseline": cpu,
                "e2e": {"value": cpu["value"], "unit": ENCODE_UNIT, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}), flush=True)
        return
    if args.impl == "reference":
        reference_arm(args, rank)
        return
    if args.workload in ENCODE_WORKLOADS:
        run_encode(args, rank, world, local_rank)
        return
    if args.workload in GEMV_WORKLOADS:
        run_gemv(args, rank, world, local_rank)
        return
    if args.workload in STREAM_WORKLOADS:
        run_stream(args, rank, world, local_rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    r = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        s = r["shape"]
        cpu = None
        if not args.no_cpu_baseline:
            src = W.ExpertSource(r["config"], 0, s)
            cpu = oracle_baseline(r["config"], s, r["batch"], r["layers"],
                                  r["uniq_mean"] / r["layers"], src.tokens_bf16(r["batch"]))
        line = {
            "metric": METRIC, "value": round(r["value"], 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(r["ms"] / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16" if r["prefill"] else "f32",
            "data": "synthetic",
            "config": {"workload": args.workload + ":" + W.WORKLOADS[r["config"]].name,
                       "batch": r["batch"], "layers": r["layers"],
                       "d": s.d, "f": s.f, "experts": s.E, "top_k": s.k,
                       "codes_bytes": 3 * (3 * s.d * s.f // 8) * s.E * r["layers"],
                       "l2": (f"inputs larger than L2: "
                              f"{3 * (3 * s.d * s.f // 8) * s.E * r['layers'] / 1e9:.2f} "
                              "GB code bank (L2 129 MB); token pool rotates routing every step")
                             if r["bank_copies"] == 1 else
                             (f"{r['bank_copies']} seeded copies of the "
                              f"{3 * (3 * s.d * s.f // 8) * s.E / 1e6:.0f} MB code bank "
                              f"({r['bank_copies'] * 3 * (3 * s.d * s.f // 8) * s.E / 1e9:.2f} "
                              "GB, L2 129 MB), step i on copy i mod "
                              f"{r['bank_copies']}; token pool rotates routing every step"),
                       "bank_copies": r["bank_copies"],
                       "parallelism": f"replicas{world}",
                       "path": ("tensor cores for every expert group (fp16 operands: "
                                "bf16 tokens and fp16 codeword sums, fp32 accumulate)")
                               if r["prefill"] else
                               "fp32 lookup tables",
                       "codes": ("encoded from N(0, 0.02^2) weights by rvq_encode, 2 Lloyd "
                                 "rounds per stage") if encoded_bank(args.workload) else
                                "uniform random (seeded)"},
            "code_byte_gbs": round(r["code_gbs"], 1),
            "layer_tok_s": round(r["tok_s"], 1),
            "unique_experts_per_step": round(r["uniq_mean"], 2),
            "kernels_us": r["kernels_us"],
            "roofline": r["roofline"], "cpu_baseline": cpu, "e2e": r["e2e"], "launch": r["launch"],
            "clocks": r["clocks"], "gpu_launches": r["launches"] * world,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
