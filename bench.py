#!/usr/bin/env python3
"""Benchmark: batched GDN decode on one GB300 (dense and DeltaLog append-merge).

Default workload (``headline``): B=128 requests, H=32 heads, dk=dv=128, fp32
state (256 MiB), bf16 q/k/v, per-head log-decay log(sigmoid(randn+3)), beta =
sigmoid(randn); DeltaLog merge interval M=8.

One benchmark *step* is one full append-merge cycle: M decode steps (M-1
appends and one merge) over M batches of synthetic input, so every path of
the decode step runs in every timed step and the figure is cycle-amortised.
``value`` is head-steps/s = B * H * M * K / t over K timed steps, inputs
already resident in HBM (a 16-step ring of pre-generated inputs). The state
(256 MiB) is larger than L2, so no flush is needed between steps.

Also reported: the dense mode on the same inputs, per-kernel CUDA-event
durations with the algorithmic bytes each launch moves (roofline against the
measured HBM copy bandwidth, and the fraction of the nominal ~8 TB/s beside it),
the read / write traffic by phase and its reduction against dense (algorithmic
model, and ncu-measured when a capture of the current kernel sources is
committed), an end-to-end figure through the public API with pinned host
buffers, the SM clocks sampled during the timed region, dense-vs-M sweeps over
the suite's decode workloads, the chunked prefill and the speculative-decoding
verify on the same shape, and the fp64 CPU oracle timed on the host cores (a
baseline, not the target).

``--impl reference`` times the fp64 CPU oracle alone on the same metric.
Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GDN decode head-steps/s and achieved HBM GB/s (% of GB300 peak), dense vs M"
UNIT = "head-steps/s"
RING = 16
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 126 * 2**20   # GB300 L2 (~126 MiB)
SPEC_HBM_GBS = 8000.0   # nominal HBM3e bandwidth of a GB300 (~8 TB/s), reported beside the measured peak
KERNEL_SOURCES = ("gdn_decode.cu", "gdn_device.cuh", "gdn_internal.h")


# ----------------------------------------------------------------------------- helpers

def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_timing(elapsed_s: float, units: float, device=None):
    """Max of the elapsed time and sum of the work over all ranks (identity when not
    distributed). Uses the default process group (NCCL on GPUs, gloo on CPU)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return elapsed_s, units
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    """Hash of the kernel sources' code: line comments and blank space are dropped, so a
    comment edit keeps a capture's counters valid while any code change drops them."""
    import re
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "linear_attention_decode_gdn_gb300", "csrc", name)) as f:
            code = re.sub(r"//[^\n]*", "", f.read())
        h.update(" ".join(code.split()).encode())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 50):
        self.gpu, self.ms, self.proc, self.lines = gpu_index, interval_ms, None, []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", f"-lms={self.ms}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except (ValueError, IndexError):
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- traffic model

def head_bytes_rw(mode: str, n: int, w, klb=2, conv=False, ulb=4):
    """Algorithmic DRAM (read, write) bytes one decode launch moves per (request, head),
    following the traffic model of the DeltaLog notes (Sec. 2.5, Eqs. (8)-(11)): inputs and
    output, the state read (and write for dense / merge), the n log entries replayed, the
    entry an append writes, and the decay metadata."""
    D = w.dk
    e = 2 if w.qkv_bf16 else 4
    dlam = w.dlam
    rd = 3 * D * e + 4 * dlam + (0 if w.raw_value else 4)   # q, k, v, lambda, beta
    if w.kda_full:
        rd += 4 * D                                         # output-gate logits
    wr = 4 * D                                              # o
    if conv:
        rd += 3 * D * 3 * e + 3 * D * 16                    # conv cache, weights
        wr += 3 * D * 3 * e                                 # conv cache shifted
    state = 4 * D * D
    entry = D * klb + ulb * D + 4 * dlam                    # one log position
    if mode == "dense":
        return rd + state, wr + state
    meta = 4 * dlam + 4                                     # ell and L read
    if mode == "append":
        return rd + state + n * entry + meta, wr + entry + 4 * dlam + 4
    return rd + state + n * entry + meta, wr + state + 4 * dlam + 4  # merge: base r+w


def head_bytes(mode: str, n: int, w, klb=2, conv=False, ulb=4) -> int:
    """Algorithmic DRAM bytes (read + write) of one decode launch per (request, head)."""
    r, wr = head_bytes_rw(mode, n, w, klb, conv, ulb)
    return r + wr


# ----------------------------------------------------------------------------- GPU arm

# Prefill on the other tensor-core prefill kernels, measured beside the headline one:
# (workload, positions per request) -- the fused conv, and the per-key decay with the KDA gate
# and output epilogue.
PREFILL_CONFIGS = (("small_conv", 256), ("kda_full", 128))


def run_prefill_configs(args, dev, stream, gdn, runner=None):
    """The prefill leg on each of PREFILL_CONFIGS; a leg that raises is reported as
    unavailable, with the error, instead of ending the run. Returns (legs, launches)."""
    import argparse
    from linear_attention_decode_gdn_gb300 import workloads as wl
    runner = runner or run_prefill
    legs, launches = {}, 0
    for name, T in PREFILL_CONFIGS:
        w = wl.WORKLOADS[name]
        leg_args = argparse.Namespace(**dict(vars(args), prefill=T))
        try:
            leg = runner(leg_args, w, decode_flags(gdn, w), dev, stream, gdn)
        except Exception as e:  # noqa: BLE001 -- one leg's failure must not cost the bench line
            leg = {"unavailable": f"{type(e).__name__}: {e}"}
        launches += int(leg.get("launches", 0))
        legs[f"{name}/T{T}"] = dict(leg, workload=f"{name}: {w.description}")
    return legs, launches


def decode_flags(gdn, w, klog_prenorm=False) -> int:
    flags = (gdn.QKV_BF16 if w.qkv_bf16 else 0) | (gdn.FUSE_CONV if w.conv else 0)
    if klog_prenorm:
        flags |= gdn.KLOG_PRENORM
    if w.raw_value:  # the RWKV6 instantiation: b = v (beta NULL), raw q/k, bf16 value log
        flags |= gdn.PLAIN_UPDATE | gdn.NO_QK_L2NORM | gdn.ULOG_BF16
    if w.kda_full:   # the KDA gate parametrisation and output epilogue
        flags |= gdn.GATE_KDA | gdn.OUT_NORM_GATE
    return flags


class DecodeRunner:
    """One workload's decode launches through the C ABI: a ring of pre-generated decode
    steps resident in HBM, the dense state pool and one DeltaLog pool set per merge
    interval (allocated on first use), and timed sequences of launches."""

    def __init__(self, gdn, lib, w, dev, stream, rank, ring=RING, klog_prenorm=False, keep_host=False,
                 extra_flags=0, use_step=False, stagger=False):
        import torch
        from linear_attention_decode_gdn_gb300 import workloads as wl
        self.gdn, self.lib, self.w, self.dev, self.stream = gdn, lib, w, dev, stream
        self.sptr = ctypes.c_void_p(stream.cuda_stream)
        self.flags = decode_flags(gdn, w, klog_prenorm) | extra_flags
        self.kda_dev = {}
        if w.kda_full:
            kp = wl.kda_gate_params(w)
            self.kda_dev = {n: torch.from_numpy(kp[n]).to(dev) for n in ("a_log", "dt_bias", "out_norm_w")}
        self.ring, self.host_ring = [], []
        for t in range(ring):
            x = wl.step_inputs(w, t + 1000 * rank)
            d = {}
            if w.conv:
                d["mixed_qkv"] = torch.from_numpy(x["mixed_bits"].view(np.int16)).view(torch.bfloat16)
            else:
                for n_ in ("q", "k", "v"):
                    d[n_] = (torch.from_numpy(x[n_ + "_bits"].view(np.int16)).view(torch.bfloat16)
                             if w.qkv_bf16 else torch.from_numpy(x[n_]))
            if w.kda_full:
                d["log_decay"] = torch.from_numpy(x["f"])
                d["beta"] = torch.from_numpy(x["b_raw"])
                d["out_gate"] = torch.from_numpy(x["out_gate"])
            else:
                d["log_decay"] = torch.from_numpy(x["lam"])
                if not w.raw_value:
                    d["beta"] = torch.from_numpy(x["beta"])
            if keep_host:
                self.host_ring.append({k: v.pin_memory() for k, v in d.items()})
            self.ring.append({k: v.to(dev) for k, v in d.items()})
        self.slot = torch.arange(w.batch, dtype=torch.int32, device=dev)
        self.conv_w = torch.from_numpy(wl.conv_weights(w)).to(dev) if w.conv else None
        self.o = torch.zeros((w.batch, w.num_heads, w.dv), dtype=torch.float32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.sets = {}
        self.launches = 0
        # every DeltaLog launch through gdn_decode_step (each slot-head picks append or merge
        # from its own log length) instead of the phase-specific entries; with `stagger`,
        # request b enters the timed steps with b % M entries in its log, so every launch
        # mixes appends and merges (about one request in M merging)
        self.use_step, self.stagger, self.staggered = use_step, stagger, set()

    def _set(self, M):
        """(dims, pools, per-ring-step inputs, log) of merge interval M (0: dense)."""
        if M not in self.sets:
            gdn, w = self.gdn, self.w
            dims = gdn.make_dims(w.batch, w.num_heads, w.dk, num_slots=w.batch,
                                 decay_per_key=w.decay_per_key, log_capacity=max(M - 1, 0), flags=self.flags)
            pools = gdn.Pools.allocate(dims, device=self.dev, conv=w.conv, deltalog=M > 0)
            ins = []
            for r in range(len(self.ring)):
                d = dict(self.ring[r], **self.kda_dev)
                if w.conv:
                    d.update(conv_w=self.conv_w, conv_pool=pools.conv)
                ins.append(gdn.make_inputs(slot=self.slot, **d))
            self.sets[M] = (dims, pools, ins, pools.log() if M > 0 else None)
        return self.sets[M]

    def launch(self, kind, r, M):
        P = ctypes.byref
        if kind == "dense":
            dims, pools, ins, _ = self._set(0)
            rc = self.lib.gdn_decode_dense(P(dims), P(ins[r]), pools.state.data_ptr(), self.o.data_ptr(),
                                           self.status.data_ptr(), self.sptr)
        else:
            dims, pools, ins, log = self._set(M)
            fn = (self.lib.gdn_decode_step if self.use_step
                  else self.lib.gdn_decode_append if kind == "append" else self.lib.gdn_decode_merge)
            rc = fn(P(dims), P(ins[r]), pools.state.data_ptr(), P(log), self.o.data_ptr(),
                    self.status.data_ptr(), self.sptr)
        if rc:
            self.gdn._abi.check(rc, kind)
        self.launches += 1

    @staticmethod
    def cycle_kinds(mode, M):
        if mode == "dense":
            return ["dense"] * M
        return ["append"] * (M - 1) + ["merge"]

    def timed(self, mode, M, steps, warmup, per_kernel=False):
        """Times `steps` cycles of M decode steps after `warmup` cycles. Back to back
        (per_kernel False) or with an event pair around every launch."""
        import torch
        kinds = self.cycle_kinds(mode, M)
        r, n = 0, len(self.ring)
        self._set(0 if mode == "dense" else M)  # allocate outside the timed region
        if self.stagger and mode != "dense" and M not in self.staggered:
            self._stagger(M)
        for _ in range(warmup):
            for k in kinds:
                self.launch(k, r % n, M)
                r += 1
        torch.cuda.synchronize(self.dev)
        barrier()
        torch.cuda.synchronize(self.dev)
        evs = []
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(self.stream)
        for _ in range(steps):
            for k in kinds:
                if per_kernel:
                    a = torch.cuda.Event(enable_timing=True)
                    b = torch.cuda.Event(enable_timing=True)
                    a.record(self.stream)
                    self.launch(k, r % n, M)
                    b.record(self.stream)
                    evs.append((k, a, b))
                else:
                    self.launch(k, r % n, M)
                r += 1
        t1.record(self.stream)
        torch.cuda.synchronize(self.dev)
        barrier()
        elapsed = t0.elapsed_time(t1) / 1e3
        per = {}
        for k, a, b in evs:
            per.setdefault(k, []).append(a.elapsed_time(b) / 1e3)
        if int(self.status.item()) != 0:
            raise RuntimeError(f"device status {int(self.status.item())} in the {self.w.name} run")
        return elapsed, per

    def _stagger(self, M):
        """Pre-roll of the staggered phases: M - 1 steps in which only the requests with
        b % M > r take part (the others are padding, slot -1)."""
        import torch
        dims, pools, _, log = self._set(M)
        P = ctypes.byref
        b = torch.arange(self.w.batch, device=self.dev)
        for r in range(M - 1):
            sl = torch.where(b % M > r, self.slot, torch.full_like(self.slot, -1))
            d = dict(self.ring[r % len(self.ring)], **self.kda_dev)
            if self.w.conv:
                d.update(conv_w=self.conv_w, conv_pool=pools.conv)
            ins = self.gdn.make_inputs(slot=sl, **d)
            rc = self.lib.gdn_decode_step(P(dims), P(ins), pools.state.data_ptr(), P(log), self.o.data_ptr(),
                                          self.status.data_ptr(), self.sptr)
            if rc:
                self.gdn._abi.check(rc, "step")
            self.launches += 1
        torch.cuda.synchronize(self.dev)
        self.staggered.add(M)

    def free(self):
        import torch
        self.sets.clear()
        self.ring.clear()
        torch.cuda.empty_cache()


def layout_bytes(flags, gdn):
    """Bytes per element of the key log and the value log under `flags`."""
    klb = 4 if flags & gdn.KLOG_FP32 else 2
    ulb = 2 if flags & gdn.ULOG_BF16 else 4
    return klb, ulb


def cycle_bytes_per_head(w, M, klb, ulb):
    """Algorithmic bytes of one cycle of M decode steps per (request, head): dense M steps
    for M = 1 (the dense kernel), else M - 1 appends entering with L = 0 .. M-2 and the
    merge entering with L = M - 1."""
    if M == 1:
        return head_bytes("dense", 0, w, klb, w.conv, ulb)
    return (sum(head_bytes("append", n, w, klb, w.conv, ulb) for n in range(M - 1))
            + head_bytes("merge", M - 1, w, klb, w.conv, ulb))


def fractions(gbs, peak):
    return {"frac_of_peak": gbs / peak, "frac_of_spec": gbs / SPEC_HBM_GBS}


# Decode-step sweeps reported beside the headline value (dense vs the merge interval on the
# suite's decode workloads); M = 1 is the dense kernel. "split_dv": each head on two CTAs, one
# per half of the value columns (GDN_SPLIT_DV), beside the one-CTA-per-head default. "step": the
# same cycle through gdn_decode_step, the entry for batches whose requests sit at different
# points of their cycle (each slot-head appends or merges by its own log length);
# "step_staggered": the same with request b's cycle offset by b % M steps, so that every launch
# mixes appends and merges (the serving case).
SWEEPS = (("headline", (1, 2, 4, 8, 16), ""), ("high_concurrency", (1, 2, 4, 8, 16), ""), ("kda", (1, 8), ""),
          ("small_conv", (1, 8), ""), ("kda_full", (1, 8), ""), ("rwkv6", (1, 4), ""),
          ("headline", (1, 8), "split_dv"), ("small_conv", (1, 8), "split_dv"), ("headline", (8,), "step"),
          ("headline", (8,), "step_staggered"))
SWEEP_DECODE_STEPS = 256   # timed decode steps per sweep point (whole cycles)
SWEEP_RING = 8


def run_sweeps(gdn, lib, dev, stream, rank, world, peak):
    """Every (workload, M) point of SWEEPS: head-steps/s, us per decode step and algorithmic
    GB/s of launches back to back over SWEEP_DECODE_STEPS decode steps after 3 warm-up cycles."""
    from linear_attention_decode_gdn_gb300 import workloads as wl
    out, launches = {}, 0
    for name, Ms, variant in SWEEPS:
        w = wl.WORKLOADS[name]
        extra = gdn.SPLIT_DV if variant == "split_dv" else 0
        run = DecodeRunner(gdn, lib, w, dev, stream, rank, ring=SWEEP_RING, extra_flags=extra,
                           use_step=variant.startswith("step"), stagger=variant == "step_staggered")
        klb, ulb = layout_bytes(run.flags, gdn)
        heads = w.batch * w.num_heads
        leg = {"batch": w.batch, "num_heads": w.num_heads, "dk": w.dk, "dv": w.dv,
               # a state that fits in L2 is partly re-read from L2: its algorithmic GB/s is no
               # HBM figure and may exceed the copy peak
               "state_fits_in_l2": w.state_bytes < L2_BYTES}
        for M in Ms:
            cycles = max(1, SWEEP_DECODE_STEPS // M)
            mode = "dense" if M == 1 else "deltalog"
            el, _ = run.timed(mode, M, cycles, 3)
            el, units = reduce_timing(el, heads * M * cycles, device=dev)
            nbytes = heads * cycle_bytes_per_head(w, M, klb, ulb) * cycles * world
            gbs = nbytes / el / 1e9
            leg["dense" if M == 1 else f"M{M}"] = {
                "head_steps_per_s": units / el, "us_per_decode_step": el / (cycles * M) * 1e6,
                "algorithmic_bytes_per_decode_step": nbytes / (cycles * M * world),
                "algorithmic_gbs": gbs, **fractions(gbs, peak)}
            run.sets.clear()
        best = max((k for k in leg if k.startswith("M")), key=lambda k: leg[k]["head_steps_per_s"])
        if "dense" in leg:
            leg["speedup_best_M_vs_dense"] = {"M": int(best[1:]),
                                              "speedup": leg[best]["head_steps_per_s"] / leg["dense"]["head_steps_per_s"]}
        launches += run.launches
        run.free()
        out[name + (f"/{variant}" if variant else "")] = leg
    return out, launches


def measured_traffic(workload: str, M: int, path=None):
    """Per-launch DRAM bytes from the committed ncu capture of one whole decode cycle
    (appends entering with L = 0 .. M-2, the merge, one dense launch), when it was taken on
    the current kernel sources: {(kernel, L): (read, write)}; else None."""
    path = path or os.path.join(ROOT, "profiles", "decode_traffic_headline.txt")
    if not os.path.exists(path):
        return None
    src = kernel_source_hash()
    got = {}
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        f = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
        if f.get("workload") != workload or f.get("src") != src or int(f.get("M", -1)) != M:
            continue
        got[(f["kernel"], int(f.get("L", 0)))] = (float(f["read"]), float(f["write"]))
    need = [("append", n) for n in range(M - 1)] + [("merge", M - 1), ("dense", 0)]
    return got if all(k in got for k in need) else None


def measured_summary(meas, M):
    """The DeltaLog notes' Fig. 8 view of a measured cycle: read / write per launch for the
    first and last append, the merge and dense; per decode step the cycle's bytes / M
    against one dense launch; the write and total reductions."""
    mr = sum(meas[("append", n)][0] for n in range(M - 1)) + meas[("merge", M - 1)][0]
    mw = sum(meas[("append", n)][1] for n in range(M - 1)) + meas[("merge", M - 1)][1]
    d_r, d_w = meas[("dense", 0)]
    sel = [("append", 0), ("append", M - 2), ("merge", M - 1), ("dense", 0)]
    return {
        "per_launch": {(f"{k}_L{n}" if k != "dense" else k): {"read": meas[(k, n)][0], "write": meas[(k, n)][1]}
                       for k, n in sel},
        "per_decode_step": {f"deltalog_M{M}": {"read": mr / M, "write": mw / M},
                            "dense": {"read": d_r, "write": d_w}},
        "write_reduction": d_w / (mw / M), "total_reduction": (d_r + d_w) / ((mr + mw) / M),
        "source": "ncu dram__bytes_read.sum / dram__bytes_write.sum of one whole cycle "
                  "(profiles/decode_traffic_headline.txt, taken on the current kernel sources)"}


def run_gpu(args, rank, local_rank, world):
    import torch
    import linear_attention_decode_gdn_gb300 as gdn
    from linear_attention_decode_gdn_gb300 import build as gbuild
    from linear_attention_decode_gdn_gb300 import workloads as wl

    if local_rank == 0:  # one build per node; the other ranks wait for it
        gbuild.build()
    barrier()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = wl.WORKLOADS[args.workload]
    M = args.merge_interval
    B, H, D = w.batch, w.num_heads, w.dk
    lib = gdn._abi.load()
    stream = torch.cuda.current_stream(dev)
    main = DecodeRunner(gdn, lib, w, dev, stream, rank, klog_prenorm=args.klog_prenorm,
                        keep_host=not args.no_e2e)
    flags = main.flags

    # ---- warm both modes, then the timed regions (clocks sampled meanwhile). The
    # throughput comes from launches back to back (nothing between them, so a launch can
    # overlap the tail of the previous one); the per-kernel durations from a second
    # region with an event pair around every launch (which serialises the launches).
    res, per = {}, {}
    with ClockSampler(local_rank) as clocks:
        res["deltalog"] = main.timed("deltalog", M, args.steps, args.warmup)
        res["dense"] = main.timed("dense", M, args.steps, args.warmup)
        per["deltalog"] = main.timed("deltalog", M, args.steps, args.warmup, per_kernel=True)
        per["dense"] = main.timed("dense", M, args.steps, args.warmup, per_kernel=True)

    peak, peak_kind = measured_peaks()
    heads = B * H
    klb, ulb = layout_bytes(flags, gdn)
    avg_n = (M - 2) / 2 if M > 1 else 0.0    # appends enter with L = 0 .. M-2
    bytes_per_launch = {
        "dense": heads * head_bytes("dense", 0, w, klb, w.conv, ulb),
        "append": heads * head_bytes("append", avg_n, w, klb, w.conv, ulb),
        "merge": heads * head_bytes("merge", M - 1, w, klb, w.conv, ulb),
    }
    kernels = {}
    for mode in ("deltalog", "dense"):
        for k, durs in per[mode][1].items():
            tot = float(np.sum(durs))
            avg = tot / len(durs)
            achieved = bytes_per_launch[k] / avg / 1e9
            kernels[k] = {"launches": len(durs), "avg_us": avg * 1e6, "total_ms": tot * 1e3,
                          "algorithmic_bytes_per_launch": bytes_per_launch[k],
                          "achieved_gbs": achieved, **fractions(achieved, peak)}
    lt, lu = reduce_timing(res["deltalog"][0], heads * M * args.steps, device=dev)
    dt, du = reduce_timing(res["dense"][0], heads * M * args.steps, device=dev)
    value = lu / lt
    cycle_bytes = heads * cycle_bytes_per_head(w, M, klb, ulb)
    dense_bytes = M * bytes_per_launch["dense"]
    modes = {}
    for name, (el, units), nbytes in ((f"deltalog_M{M}", (lt, lu), cycle_bytes),
                                      ("dense", (dt, du), dense_bytes)):
        gbs = nbytes * args.steps * world / el / 1e9
        modes[name] = {"head_steps_per_s": units / el,
                       "us_per_decode_step": el / (args.steps * M) * 1e6,
                       "algorithmic_bytes_per_decode_step": nbytes / M,
                       "algorithmic_gbs": gbs, **fractions(gbs, peak)}
    modes["speedup_deltalog_vs_dense"] = value / (du / dt)
    # read / write bytes per launch by phase (the DeltaLog notes' Fig. 8 split) and per
    # decode step, with the write and total reductions of the log against dense: from the
    # algorithmic model, and measured by ncu when a capture of the current sources exists
    phases = {"dense": head_bytes_rw("dense", 0, w, klb, w.conv, ulb)}
    if M > 1:
        phases["append_L0"] = head_bytes_rw("append", 0, w, klb, w.conv, ulb)
        phases[f"append_L{M - 2}"] = head_bytes_rw("append", M - 2, w, klb, w.conv, ulb)
    phases[f"merge_L{M - 1}"] = head_bytes_rw("merge", M - 1, w, klb, w.conv, ulb)
    cyc = [head_bytes_rw("append", n, w, klb, w.conv, ulb) for n in range(M - 1)] + \
        [head_bytes_rw("merge", M - 1, w, klb, w.conv, ulb)]
    step_r, step_w = sum(c[0] for c in cyc) * heads / M, sum(c[1] for c in cyc) * heads / M
    dense_r, dense_w = phases["dense"][0] * heads, phases["dense"][1] * heads
    traffic = {"model": {
        "per_launch": {k: {"read": v[0] * heads, "write": v[1] * heads} for k, v in phases.items()},
        "per_decode_step": {f"deltalog_M{M}": {"read": step_r, "write": step_w},
                            "dense": {"read": dense_r, "write": dense_w}},
        "write_reduction": dense_w / step_w, "total_reduction": (dense_r + dense_w) / (step_r + step_w),
        "source": "algorithmic model (DeltaLog notes Sec. 2.5, Eqs. (8)-(11))"}}
    meas = measured_traffic(args.workload, M) if (M > 1 and not args.klog_prenorm) else None
    traffic["measured"] = measured_summary(meas, M) if meas is not None else None
    modes["traffic"] = traffic

    # dominant kernel of the timed DeltaLog cycle: largest share of device time
    dom = max(per["deltalog"][1], key=lambda k: kernels[k]["total_ms"])
    kd = kernels[dom]
    dom_traffic = None
    if meas is not None:
        if dom == "append":
            dom_traffic = sum(sum(meas[("append", n)]) for n in range(M - 1)) / (M - 1)
        else:
            dom_traffic = sum(meas[("merge", M - 1)])
    roofline = {"bound": "hbm", "kernel": dom, "achieved": kd["achieved_gbs"], "peak": peak,
                "peak_kind": f"{peak_kind} (hbm_gbs of MEASURED_PEAKS.json)" if peak_kind == "measured"
                else "fallback 6.8 TB/s", "unit": "GB/s", "frac": kd["achieved_gbs"] / peak,
                "frac_of_spec": kd["achieved_gbs"] / SPEC_HBM_GBS, "spec_gbs": SPEC_HBM_GBS,
                "traffic": dom_traffic,
                "algorithmic_bytes_per_launch": kd["algorithmic_bytes_per_launch"],
                "duration": "CUDA events around every launch of the second timed region "
                            "(serialised launches: no overlap with the previous grid)"}

    # ---- end to end through the public API: pinned host inputs in, o back to pinned host
    e2e = None
    if not args.no_e2e:
        dims_log, pools_l, _, _ = main._set(M)
        e2e = run_e2e(args, w, M, dims_log, pools_l, main.host_ring, main.slot, main.conv_w, dev, stream, gdn,
                      main.kda_dev)
    launches_main = main.launches
    main.free()

    sweeps, sweep_launches, sweep_clocks = None, 0, None
    if not args.no_sweeps:
        with ClockSampler(local_rank) as sclocks:
            sweeps, sweep_launches = run_sweeps(gdn, lib, dev, stream, rank, world, peak)
        sweep_clocks = sclocks.summary()
    verify = run_verify(args, w, flags, dev, stream, gdn, peak) if args.verify else None
    prefill = run_prefill(args, w, flags, dev, stream, gdn) if args.prefill else None
    # (one GPU only: a leg that failed on one rank would leave the others in its collective)
    prefill_configs, pc_launches = None, 0
    if args.prefill and not args.no_sweeps and args.workload == "headline" and world == 1:
        prefill_configs, pc_launches = run_prefill_configs(args, dev, stream, gdn)

    launches = (launches_main + (e2e["launches"] if e2e else 0) + (verify["launches"] if verify else 0)
                + (prefill.get("launches", 0) if prefill else 0) + sweep_launches + pc_launches)
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": lt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.description}", "batch": B, "num_heads": H, "dk": D,
                   "dv": w.dv, "merge_interval": M, "decode_steps_per_step": M,
                   "inputs": ("bf16" if w.qkv_bf16 else "fp32") + " q/k/v"
                   + (" through the fused width-4 conv" if w.conv else "")
                   + (", fp32 log-decay, raw-value update (beta = 1); fp32 state, bf16 key and value logs"
                      if w.raw_value else
                      ", fp32 log-decay and beta; fp32 state and log values, "
                      + ("bf16 pre-normalisation" if args.klog_prenorm else "bf16") + " key log"),
                   "l2": f"state {w.state_bytes / 2**20:.0f} MiB > L2 (inputs larger than L2, no flush)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "modes": modes,
        "kernels": kernels,
        "roofline": roofline,
        "e2e": e2e,
        **({"sweeps": dict(sweeps, clocks=sweep_clocks)} if sweeps else {}),
        **({"verify": verify} if verify else {}),
        **({"prefill": prefill} if prefill else {}),
        **({"prefill_configs": prefill_configs} if prefill_configs else {}),
        "pages_context": PAGES_CONTEXT,
        "gpu_launches": launches,
        "clocks": {k: v for k, v in clocks.summary().items()},
    }
    return out


# The pages' own measurements, quoted beside this bench's as context only: other hardware,
# other kernels, not the target (DeltaLog reading notes, Sec. 4.1 Figs. 6-7, Sec. 4.2 Fig. 8,
# Sec. 4.4 Fig. 10, Sec. 4.6 Table 4). This bench's counterparts: `modes.speedup_deltalog_vs_dense`,
# the measured `modes.traffic` reductions and `modes.deltalog_M8.us_per_decode_step`.
PAGES_CONTEXT = {
    "note": "the pages' numbers on other GPUs, against other kernels; context, not the target",
    "deltalog_speedup_vs_fla_rtx4090_gdn_m8": "up to 1.86x (B = 64 .. 512)",
    "deltalog_speedup_vs_fla_h200_gdn_m8": "1.34 / 1.45 / 1.53 / 1.60x at B = 64 / 128 / 256 / 512",
    "write_traffic_reduction_vs_dense_h200_b128_m8": 7.83,
    "total_traffic_reduction_vs_dense_h200_b128_m8": 1.64,
    "end_to_end_tpot_speedup_h200": "1.05 - 1.20x (two hybrid models; needs trained weights, not run here)",
    "amortised_step_latency_h200_b128_m8_ms": 0.103,
}


def _packed(arrays: dict, align: int = 256):
    """Byte offsets of `arrays` packed into one buffer (each start 256-byte aligned)."""
    offs, off = {}, 0
    for k, t in arrays.items():
        offs[k] = off
        off += (t.numel() * t.element_size() + align - 1) // align * align
    return offs, off


def _views(buf, offs, like: dict):
    return {k: buf[offs[k]:offs[k] + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
            for k, t in like.items()}


def run_verify(args, w, flags, dev, stream, gdn, peak):
    """Speculative-decoding verify on the same workload: T = args.verify positions per
    request (the last token and T-1 drafts) through gdn_decode_verify, the state after
    every position written to its own pool row, the initial row chosen by a seeded
    acceptance count. Unit: positions x heads per second."""
    import torch
    B, H, D, T = w.batch, w.num_heads, w.dk, args.verify
    vflags = flags & ~(gdn.KLOG_PRENORM | gdn.ULOG_BF16 | gdn.GATE_KDA | gdn.OUT_NORM_GATE)
    rng = np.random.default_rng(w.seed + 77)
    S = B * T
    conv = {}
    if w.conv:  # q, k, v from the conv of mixed_qkv through the widened window [S][channels][T+2]
        conv["conv_w"] = torch.from_numpy(wl_conv_weights(w)).to(dev)
        conv["conv_pool"] = torch.zeros((S, w.channels, T + 2), dtype=torch.bfloat16 if w.qkv_bf16
                                        else torch.float32, device=dev)
    ring = []
    for t in range(RING):
        x = dict(conv)
        if w.conv:
            a = rng.standard_normal((B, T, w.channels), dtype=np.float32)
            bits, _ = wl_bf16(a)
            x["mixed_qkv"] = torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16) if w.qkv_bf16 \
                else torch.from_numpy(a).to(dev)
        for n in (() if w.conv else ("q", "k", "v")):
            a = rng.standard_normal((B, T, H, D), dtype=np.float32) * np.float32(1.0 if n == "v" else w.qk_mult)
            bits, _ = wl_bf16(a)
            x[n] = torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16) if w.qkv_bf16 \
                else torch.from_numpy(a).to(dev)
        a_raw = rng.standard_normal((B, T, H, w.dlam), dtype=np.float32) + np.float32(3)
        x["log_decay"] = torch.from_numpy((-np.log1p(np.exp(-a_raw))).astype(np.float32)).to(dev)
        if not w.raw_value:
            b_raw = rng.standard_normal((B, T, H), dtype=np.float32)
            x["beta"] = torch.from_numpy((1 / (1 + np.exp(-b_raw))).astype(np.float32)).to(dev)
        acc = torch.from_numpy(rng.integers(1, T + 1, size=B).astype(np.int32)).to(dev)
        ring.append((gdn.make_inputs(**x), acc, x))
    dims = gdn.make_dims(B, H, D, num_slots=S, decay_per_key=w.decay_per_key, flags=vflags)
    pool = torch.zeros((S, H, D, D), dtype=torch.float32, device=dev)
    idx = torch.arange(S, dtype=torch.int32, device=dev).view(B, T)
    o = torch.zeros((B, T, H, D), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    calls = max(50, args.steps // 4)

    def go(n, r0=0):
        for i in range(n):
            inp, acc, _ = ring[(r0 + i) % RING]
            gdn.decode_verify(dims, T, inp, idx, acc, pool, o, status, stream=stream)

    go(max(3, args.warmup))
    torch.cuda.synchronize(dev)
    barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    go(calls)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the verify run")
    el, units = reduce_timing(t0.elapsed_time(t1) / 1e3, B * H * T * calls, device=dev)
    e = 2 if w.qkv_bf16 else 4
    per_head = 4 * D * D * (1 + T) + T * (3 * D * e + 4 * w.dlam + (0 if w.raw_value else 4) + 4 * D) + 8
    if w.conv:  # the window: three inputs read, T + 2 written, per channel; the weights
        per_head += 3 * D * ((3 + T + 2) * e + 16)
    gbs = B * H * per_head * calls / el / 1e9
    return {"value": units / el, "unit": "positions x heads / s", "positions_per_request": T,
            "us_per_call": el / calls * 1e6, "calls": calls, "launches": calls + max(3, args.warmup),
            "algorithmic_bytes_per_call": B * H * per_head, "algorithmic_gbs": gbs, **fractions(gbs, peak),
            "state_rows": "one read + T writes of the 64 KiB state per (request, head)"}


FP32_FMA_PER_SM_CLK = 128   # GB300 SM: 4 partitions x 32 FP32 lanes
TF32_PER_BF16 = 1.1 / 2.25  # nominal dense tensor-core rates of a GB300, TF32 : BF16
FALLBACK_BF16_TFLOPS = 1900.0
GB300_SMS = 152
GB300_MAX_SM_MHZ = 2070.0


def prefill_chunk_fmas(D: int, C: int, plain: bool) -> int:
    """Algorithmic FMAs of one chunk of C positions of one head in the WY/UT prefill:
    pair sums (A strictly lower unless plain, P lower with the diagonal), [Ktil; Qtil] S0
    (only Qtil under the plain update), the forward substitution, the readout P B and
    Khat^T B. Elementwise scalings are left out."""
    pairs_p = C * (C + 1) // 2
    pairs_a = 0 if plain else C * (C - 1) // 2
    gemm1 = (1 if plain else 2) * C * D * D
    subst = 0 if plain else C * (C - 1) // 2 * D
    return (pairs_a + pairs_p) * D + gemm1 + subst + pairs_p * D + D * D * C


def run_prefill(args, w, flags, dev, stream, gdn):
    """Chunked prefill on the workload's batch shape: T = args.prefill positions per request
    from a zero state, through gdn_prefill. Compute-bound: reported against the FP32 ALU peak
    derived from the SM count, the FP32 lanes per SM and the maximum SM clock."""
    import torch
    B, H, D, T = w.batch, w.num_heads, w.dk, args.prefill
    pflags = flags & (gdn.QKV_BF16 | gdn.NO_QK_L2NORM | gdn.PLAIN_UPDATE | gdn.FUSE_CONV)
    rng = np.random.default_rng(w.seed + 99)
    x = {}
    if w.conv:
        # mixed_qkv rows [B][T][channels] through the width-4 conv, the workload's conv weights,
        # a zero conv state (each call leaves the prompt's last three inputs there)
        from linear_attention_decode_gdn_gb300 import workloads as wl
        a = rng.standard_normal((B, T, w.channels), dtype=np.float32)
        bits, _ = wl_bf16(a)
        x["mixed_qkv"] = torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16) if w.qkv_bf16 \
            else torch.from_numpy(a).to(dev)
        x["conv_w"] = torch.from_numpy(wl.conv_weights(w)).to(dev)
        x["conv_pool"] = torch.zeros((B, w.channels, 3), device=dev,
                                     dtype=torch.bfloat16 if w.qkv_bf16 else torch.float32)
    else:
        for n in ("q", "k", "v"):
            a = rng.standard_normal((B, T, H, D), dtype=np.float32) * np.float32(1.0 if n == "v" else w.qk_mult)
            bits, _ = wl_bf16(a)
            x[n] = torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16) if w.qkv_bf16 \
                else torch.from_numpy(a).to(dev)
    a_raw = rng.standard_normal((B, T, H, w.dlam), dtype=np.float32) + np.float32(3)
    b_raw = rng.standard_normal((B, T, H), dtype=np.float32)
    if w.kda_full:
        # the KDA gate parametrisation (raw gate f = decay draw - 3, write logit) and the
        # output epilogue, as in the decode workload
        from linear_attention_decode_gdn_gb300 import workloads as wl
        pflags |= gdn.GATE_KDA | gdn.OUT_NORM_GATE
        kp = wl.kda_gate_params(w)
        x.update({n: torch.from_numpy(kp[n]).to(dev) for n in ("a_log", "dt_bias", "out_norm_w")})
        x["log_decay"] = torch.from_numpy(a_raw - np.float32(3)).to(dev)
        x["beta"] = torch.from_numpy(b_raw).to(dev)
        x["out_gate"] = torch.from_numpy(rng.standard_normal((B, T, H, D), dtype=np.float32)).to(dev)
    else:
        x["log_decay"] = torch.from_numpy((-np.log1p(np.exp(-a_raw))).astype(np.float32)).to(dev)
        if not w.raw_value:
            x["beta"] = torch.from_numpy((1 / (1 + np.exp(-b_raw))).astype(np.float32)).to(dev)
    slot = torch.arange(B, dtype=torch.int32, device=dev)
    inp = gdn.make_inputs(slot=slot, **x)
    dims = gdn.make_dims(B, H, D, num_slots=B, decay_per_key=w.decay_per_key, flags=pflags)
    pool = torch.zeros((B, H, D, D), dtype=torch.float32, device=dev)
    o = torch.zeros((B, T, H, D), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    calls = max(3, min(20, args.steps // 100))
    for _ in range(max(2, args.warmup // 2)):
        gdn.prefill(dims, T, inp, pool, o, status=status, stream=stream)
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(calls):
        gdn.prefill(dims, T, inp, pool, o, status=status, stream=stream)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the prefill run")
    el, units = reduce_timing(t0.elapsed_time(t1) / 1e3, B * H * T * calls, device=dev)
    chunks = -(-T // 32)
    flops = 2.0 * prefill_chunk_fmas(D, 32, bool(pflags & gdn.PLAIN_UPDATE)) * chunks * B * H
    tflops = flops * calls / el / 1e12
    alu_peak = GB300_SMS * FP32_FMA_PER_SM_CLK * 2 * GB300_MAX_SM_MHZ * 1e6 / 1e12
    out = {"value": units / el, "unit": "positions x heads / s", "positions_per_request": T,
           "ms_per_call": el / calls * 1e3, "calls": calls, "launches": calls + max(2, args.warmup // 2)}
    if prefill_on_tensor_cores(D, w.decay_per_key, pflags, gdn, B, T):
        # the products run as kind::tf32 MMAs, three per fp32-accurate product (3xTF32)
        bf16, kind = measured_bf16_tflops()
        tf32 = bf16 * TF32_PER_BF16
        peak = tf32 / 3.0
        out["kernel"] = ("gdn_prefill_tc_pk_kernel" if w.decay_per_key else "gdn_prefill_tc_kernel") + \
            (" with the fused conv" if pflags & gdn.FUSE_CONV else "") + " (tcgen05 kind::tf32, 3xTF32)"
        out["roofline"] = {
            "bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s (fp32-accurate, 3xTF32)",
            "frac": tflops / peak,
            "peak_derivation": f"{kind} bf16 {bf16:.0f} TFLOP/s x {TF32_PER_BF16:.3f} (nominal TF32/BF16 dense "
                               f"ratio 1.1/2.25) = {tf32:.0f} TF32 TFLOP/s, / 3 MMAs per fp32-accurate product",
            "frac_of_fp32_alu_peak": tflops / alu_peak, "fp32_alu_peak": alu_peak,
            "algorithmic_flops_per_call": flops}
    else:
        out["kernel"] = "gdn_prefill_kernel (FP32 CUDA cores)"
        out["roofline"] = {"bound": "alu", "achieved": tflops, "peak": alu_peak, "unit": "TFLOP/s (fp32)",
                           "frac": tflops / alu_peak,
                           "peak_derivation": "152 SMs x 128 FP32 FMA/clk x 2 FLOP x 2070 MHz",
                           "algorithmic_flops_per_call": flops}
    return out


def prefill_on_tensor_cores(D, decay_per_key, flags, gdn, B=1, T=1) -> bool:
    """The library's choice of prefill kernel: a tcgen05 one for 128-wide heads (and B * T
    below 2^31, the 32-bit position coordinate of its token copies): with a per-head decay and
    no KDA gate / epilogue (the fused conv with bf16 mixed_qkv included), or a per-key decay
    with bf16 q, k, v and no fused conv."""
    if D != 128 or B * T >= 2 ** 31:
        return False
    if decay_per_key:  # bf16 q, k, v; the KDA gate and epilogue included
        return bool(flags & gdn.QKV_BF16) and not flags & gdn.FUSE_CONV
    if flags & gdn.FUSE_CONV and not flags & gdn.QKV_BF16:
        return False
    return not flags & (gdn.GATE_KDA | gdn.OUT_NORM_GATE)


def measured_bf16_tflops():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def wl_bf16(a):
    from linear_attention_decode_gdn_gb300 import workloads as wl
    return wl.bf16_round(a)


def wl_conv_weights(w):
    from linear_attention_decode_gdn_gb300 import workloads as wl
    return wl.conv_weights(w)


class _Cudart:
    """The few CUDA runtime calls the end-to-end loop issues per step, bound through
    ctypes (the runtime the decode library itself links), so the host side of a step
    costs a handful of microseconds."""
    H2D, D2H = 1, 2

    def __init__(self):
        self.lib = ctypes.CDLL("libcudart.so.13")
        for name, args in (("cudaMemcpyAsync", [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                                 ctypes.c_int, ctypes.c_void_p]),
                           ("cudaEventRecord", [ctypes.c_void_p, ctypes.c_void_p]),
                           ("cudaStreamWaitEvent", [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]),
                           ("cudaEventCreateWithFlags", [ctypes.c_void_p, ctypes.c_uint]),
                           ("cudaEventDestroy", [ctypes.c_void_p])):
            fn = getattr(self.lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int

    def event(self):
        e = ctypes.c_void_p()
        self._ok(self.lib.cudaEventCreateWithFlags(ctypes.byref(e), 2), "cudaEventCreateWithFlags")
        return e

    @staticmethod
    def _ok(rc, what):
        if rc != 0:
            raise RuntimeError(f"{what} failed with CUDA error {rc}")


def run_e2e(args, w, M, dims, pools, host_ring, slot, conv_w, dev, stream, gdn, kda_dev=None):
    """Same metric through the C ABI with host buffers. Every bench step (one append-merge
    cycle of M decode steps) copies its inputs host -> device (one pinned buffer holding
    the M decode steps' q/k/v or conv input, log-decay, beta, ...), runs its M decode
    calls back to back, and copies their M output rows back to pinned host memory. The
    copies run on their own streams, double-buffered against the decode kernels and
    ordered by events, the way a serving loop overlaps the next step's upload and the
    last step's readback with the current step."""
    import torch
    rt = _Cudart()
    offs, nbytes = _packed(host_ring[0])
    ncyc = max(1, len(host_ring) // M)        # distinct cycles of inputs in the ring
    host_cyc = []
    for c in range(ncyc):
        hb = torch.empty(M * nbytes, dtype=torch.uint8).pin_memory()
        for j in range(M):
            src = host_ring[(c * M + j) % len(host_ring)]
            for k, v in _views(hb[j * nbytes:(j + 1) * nbytes], offs, src).items():
                v.copy_(src[k])
        host_cyc.append(hb)
    stage = [torch.empty(M * nbytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    o = [torch.zeros((M, w.batch, w.num_heads, w.dv), dtype=torch.float32, device=dev) for _ in range(2)]
    o_host = [torch.empty_like(o[0], device="cpu").pin_memory() for _ in range(2)]
    log = pools.log()
    extra = dict(conv_w=conv_w, conv_pool=pools.conv) if w.conv else {}
    extra.update(kda_dev or {})  # per-head parameters stay resident; per-step inputs are copied
    inputs = [[gdn.make_inputs(slot=slot, **_views(stage[b][j * nbytes:(j + 1) * nbytes], offs, host_ring[0]),
                               **extra) for j in range(M)] for b in range(2)]
    h2d = M * nbytes
    d2h = o[0].numel() * o[0].element_size()
    gdn.slot_reset(dims, slot, w.batch, log, pools.conv, None, stream=stream)
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    sc, si, so = (ctypes.c_void_p(x.cuda_stream) for x in (stream, s_in, s_out))
    ev_in = [rt.event() for _ in range(2)]
    ev_k = [rt.event() for _ in range(2)]
    ev_out = [rt.event() for _ in range(2)]
    lib = gdn._abi.load()
    P = ctypes.byref
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    base_ptr, st_ptr = ctypes.c_void_p(pools.state.data_ptr()), ctypes.c_void_p(status.data_ptr())
    # the decode calls' arguments, built once: (entry point, inputs, o row) per buffer and step
    calls = [[(lib.gdn_decode_append if j < M - 1 else lib.gdn_decode_merge, P(inputs[b][j]),
               ctypes.c_void_p(o[b][j].data_ptr())) for j in range(M)] for b in range(2)]
    hp = [ctypes.c_void_p(t.data_ptr()) for t in host_cyc]
    sp = [ctypes.c_void_p(t.data_ptr()) for t in stage]
    op = [ctypes.c_void_p(t.data_ptr()) for t in o]
    ohp = [ctypes.c_void_p(t.data_ptr()) for t in o_host]
    dims_p, log_p = P(dims), P(log)
    steps, c, launches = args.e2e_steps or args.steps, 0, 0
    memcpy, record, wait = rt.lib.cudaMemcpyAsync, rt.lib.cudaEventRecord, rt.lib.cudaStreamWaitEvent

    def one_step():
        nonlocal c, launches
        b = c & 1
        if c >= 2:
            wait(si, ev_k[b], 0)                  # the kernels of step c-2 have consumed stage[b]
        memcpy(sp[b], hp[c % ncyc], h2d, rt.H2D, si)
        record(ev_in[b], si)
        wait(sc, ev_in[b], 0)
        if c >= 2:
            wait(sc, ev_out[b], 0)                # o[b] of step c-2 has been read back
        for fn, inp, optr in calls[b]:
            rc = fn(dims_p, inp, base_ptr, log_p, optr, st_ptr, sc)
            if rc:
                gdn._abi.check(rc, "decode")
        record(ev_k[b], sc)
        wait(so, ev_k[b], 0)
        memcpy(ohp[b], op[b], d2h, rt.D2H, so)
        record(ev_out[b], so)
        c += 1
        launches += M

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize(dev)
    barrier()
    launches = 0
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    s_in.wait_event(t0)
    s_out.wait_event(t0)
    for _ in range(steps):
        one_step()
    for e in ev_out:
        wait(sc, e, 0)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the end-to-end run")
    if not bool(torch.isfinite(o_host[(c - 1) & 1]).all()):
        raise RuntimeError("non-finite output read back in the end-to-end run")
    for e in ev_in + ev_k + ev_out:
        rt.lib.cudaEventDestroy(e)
    el, units = reduce_timing(t0.elapsed_time(t1) / 1e3, w.batch * w.num_heads * M * steps, device=dev)
    return {"value": units / el, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps, "launches": launches,
            "pipeline": "per step: one H2D of the cycle's inputs, M decode calls back to back, one D2H of "
                        "the M output rows; copies on their own streams, double-buffered, event-ordered",
            "api": "gdn_decode_append / gdn_decode_merge (C ABI), host copies through the CUDA runtime"}


# ----------------------------------------------------------------------------- CPU oracle

def oracle_sample(w, steps_budget_s: float, max_steps: int, batch: int, warm=1):
    """Times the fp64 oracle (dense recurrence, OpenMP over (request, head)) on a bounded
    sample: `batch` requests of the workload, consecutive decode steps."""
    import oracle
    from linear_attention_decode_gdn_gb300 import workloads as wl
    lib = oracle.load()
    H, D = w.num_heads, w.dk
    flags = (oracle.PLAIN if w.raw_value else oracle.L2NORM) | (oracle.CONV if w.conv else 0)
    kp = None
    if w.kda_full:
        flags |= oracle.GATE_KDA | oracle.OUT_NORM_GATE
        kp = wl.kda_gate_params(w)
    cfg = dict(batch=batch, num_heads=H, dk=D, dv=w.dv, num_slots=batch, dlam=w.dlam,
               log_capacity=0, flags=flags, q_scale=1.0, l2_eps=1e-6)
    st = oracle.BatchState(batch, H, D, w.dv, w.dlam, 0, nch=w.channels)
    slot = np.arange(batch, dtype=np.int32)
    cw = wl.conv_weights(w).astype(np.float64) if w.conv else None
    inputs = []
    for t in range(min(max_steps, RING)):
        x = wl.step_inputs(w, t, batch=batch)
        kw = dict(lam=x["lam"].astype(np.float64), beta=x["beta"].astype(np.float64))
        if kp is not None:
            kw = dict(lam=x["f"].astype(np.float64), beta=x["b_raw"].astype(np.float64),
                      out_gate=x["out_gate"].astype(np.float64), lower_bound=kp["lower_bound"],
                      **{n: kp[n].astype(np.float64) for n in ("a_log", "dt_bias", "out_norm_w")})
        if w.conv:
            kw.update(mixed=x["mixed"].astype(np.float64), conv_w=cw)
        else:
            kw.update(q=x["q"].astype(np.float64), k=x["k"].astype(np.float64),
                      v=x["v"].astype(np.float64))
        inputs.append(kw)
    for t in range(warm):
        oracle.step_batch(cfg, "dense", st, slot, lib=lib, **inputs[t % len(inputs)])
    n, t0 = 0, time.perf_counter()
    while n < max_steps:
        oracle.step_batch(cfg, "dense", st, slot, lib=lib, **inputs[n % len(inputs)])
        n += 1
        if time.perf_counter() - t0 >= steps_budget_s:
            break
    el = time.perf_counter() - t0
    return batch * H * n / el, n, el, oracle.num_threads(lib)


def cpu_baseline(w, budget_s=12.0):
    batch = min(w.batch, 32)
    v, n, el, cores = oracle_sample(w, budget_s, 10_000, batch)
    return {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} decode steps of {batch} requests x {w.num_heads} heads of the {w.name} "
                      f"workload (dk=dv={w.dk}), fp64 dense recurrence, {el:.1f} s"}


def run_reference(args, rank):
    """The CPU oracle as it stands, on this arm's metric: each step is one cycle of M decode
    steps over a bounded sample (8 requests x H heads) of the workload."""
    if rank != 0:
        return None
    from linear_attention_decode_gdn_gb300 import workloads as wl
    import oracle
    w = wl.WORKLOADS[args.workload]
    M = args.merge_interval
    batch = min(8, w.batch)
    oracle_sample(w, 0.0, max(1, args.warmup) * M, batch)  # warm-up
    v, n, el, cores = oracle_sample(w, 1e30, args.steps * M, batch, warm=0)
    sample = (f"{args.steps} steps x {M} decode steps of {batch} requests x {w.num_heads} heads "
              f"(dk=dv={w.dk}) of the {w.name} workload, fp64 dense recurrence")
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": f"{w.name}: {w.description}", "merge_interval": M,
                       "decode_steps_per_step": M, "sample_batch": batch},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


# ----------------------------------------------------------------------------- main

def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000, help="timed steps (append-merge cycles)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gdn", "reference"], default="gdn")
    ap.add_argument("--workload", default="headline")
    ap.add_argument("--merge-interval", type=int, default=8)
    ap.add_argument("--klog-prenorm", action="store_true",
                    help="key log keeps the pre-normalisation bf16 key (exact factor)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefill", type=int, default=256,
                    help="also time the chunked prefill with this many positions per request (0: off)")
    ap.add_argument("--verify", type=int, default=4,
                    help="also time the speculative-decoding verify path with this many positions (0: off)")
    ap.add_argument("--no-sweeps", action="store_true",
                    help="skip the dense-vs-M sweeps over the suite's decode workloads")
    args = ap.parse_args(argv)

    world, rank, local = dist_info()
    if args.impl == "reference":
        line = run_reference(args, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    out = run_gpu(args, rank, local, world)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            from linear_attention_decode_gdn_gb300 import workloads as wl
            out["cpu_baseline"] = cpu_baseline(wl.WORKLOADS[args.workload])
        else:
            out["cpu_baseline"] = None
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
