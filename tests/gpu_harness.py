"""Lockstep parity runner: the CUDA path (through the C ABI) beside the fp64 oracle.

Both sides are fed the same seeded inputs from ``workloads``; the GPU sees the
bf16 / fp32 values, the oracle their exact fp64 upcasts. The oracle's dense
recurrence is the reference for every GPU mode (dense and DeltaLog): the
DeltaLog logical state must equal it. Error metric: max|gpu - ref| / max|ref|
over the whole output tensor [T, B, H, dv], and separately over the final state.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

import oracle
import linear_attention_decode_gdn_gb300 as gdn
from linear_attention_decode_gdn_gb300 import workloads as wl

F64 = np.float64


def dev_f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda")


def dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to("cuda").view(torch.bfloat16)


def dev_i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to("cuda")


def base_flags(w: wl.Workload, gate_raw=False) -> int:
    f = 0
    if w.qkv_bf16:
        f |= gdn.QKV_BF16
    if w.conv:
        f |= gdn.FUSE_CONV
    if gate_raw:
        f |= gdn.GATE_RAW
    if w.raw_value:  # the RWKV6 instantiation: b = v, raw q/k, bf16 value log
        f |= gdn.PLAIN_UPDATE | gdn.NO_QK_L2NORM | gdn.ULOG_BF16
    if w.kda_full:   # the KDA gate parametrisation and output epilogue
        f |= gdn.GATE_KDA | gdn.OUT_NORM_GATE
    return f


def oracle_flags(w: wl.Workload, gpu_flags: int) -> int:
    f = 0
    if w.conv:
        f |= oracle.CONV
    if not gpu_flags & gdn.NO_QK_L2NORM:
        f |= oracle.L2NORM
    if gpu_flags & gdn.PLAIN_UPDATE:
        f |= oracle.PLAIN
    if gpu_flags & gdn.GATE_RAW:
        f |= oracle.GATE_RAW
    if gpu_flags & gdn.GATE_KDA:
        f |= oracle.GATE_KDA
    if gpu_flags & gdn.OUT_NORM_GATE:
        f |= oracle.OUT_NORM_GATE
    return f


@dataclass
class Variant:
    """One GPU configuration run in lockstep with the oracle."""
    mode: str                 # 'dense' | 'deltalog'
    M: int = 1                # merge interval (deltalog)
    entry: str = "split"      # deltalog: 'split' = append/merge chosen on the host, 'step' = gdn_decode_step
    extra_flags: int = 0
    name: str = ""
    drop_flags: int = 0       # flags of the workload this variant runs without
    max_err: float = 0.0
    max_ref: float = 0.0
    state_err: float = float("nan")
    state_ref: float = float("nan")
    outputs: list = field(default_factory=list)

    def setup(self, w: wl.Workload, B, num_slots, q_scale, l2_eps, gate_raw):
        self.C = self.M - 1 if self.mode == "deltalog" else 0
        self.dims = gdn.make_dims(B, w.num_heads, w.dk, w.dv, num_slots, decay_per_key=w.decay_per_key,
                                  log_capacity=self.C,
                                  flags=(base_flags(w, gate_raw) | self.extra_flags) & ~self.drop_flags,
                                  q_scale=q_scale, l2_eps=l2_eps)
        self.pools = gdn.Pools.allocate(self.dims, conv=w.conv, deltalog=self.mode == "deltalog")
        self.o = torch.zeros((B, w.num_heads, w.dv), dtype=torch.float32, device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.t = 0
        if not self.name:
            self.name = self.mode if self.mode == "dense" else f"M={self.M}/{self.entry}"

    def step(self, inputs):
        if self.mode == "dense":
            gdn.decode_dense(self.dims, inputs, self.pools.state, self.o, self.status)
        elif self.entry == "step":
            gdn.decode_step(self.dims, inputs, self.pools.state, self.pools.log(), self.o, self.status)
        elif (self.t + 1) % self.M == 0:
            gdn.decode_merge(self.dims, inputs, self.pools.state, self.pools.log(), self.o, self.status)
        else:
            gdn.decode_append(self.dims, inputs, self.pools.state, self.pools.log(), self.o, self.status)
        self.t += 1

    @property
    def rel_err(self):
        return self.max_err / self.max_ref if self.max_ref > 0 else self.max_err

    @property
    def state_rel_err(self):
        return self.state_err / self.state_ref if self.state_ref > 0 else self.state_err


class Lockstep:
    """Steps the oracle (dense, fp64) and a set of GPU variants on identical inputs."""

    def __init__(self, w: wl.Workload, variants, *, batch=None, slot=None, num_slots=None,
                 q_scale=1.0, l2_eps=1e-6, gate_raw=False, extra_oracle_flags=0, keep_outputs=False):
        self.w = w
        self.B = w.batch if batch is None else batch
        self.slot = wl.identity_slots(self.B) if slot is None else np.asarray(slot, dtype=np.int32)
        self.num_slots = num_slots or max(1, int(self.slot.max()) + 1)
        self.gate_raw = gate_raw
        self.keep = keep_outputs
        self.variants = variants
        gpu_flags0 = base_flags(w, gate_raw) | (variants[0].extra_flags if variants else 0)
        gpu_flags0 &= ~(variants[0].drop_flags if variants else 0)
        self.cfg = dict(batch=self.B, num_heads=w.num_heads, dk=w.dk, dv=w.dv, num_slots=self.num_slots,
                        dlam=w.dlam, log_capacity=0,
                        flags=oracle_flags(w, gpu_flags0) | extra_oracle_flags,
                        q_scale=q_scale, l2_eps=l2_eps)
        self.ost = oracle.BatchState(self.num_slots, w.num_heads, w.dk, w.dv, w.dlam, 0, nch=w.channels)
        for v in variants:
            v.setup(w, self.B, self.num_slots, q_scale, l2_eps, gate_raw)
        self.slot_dev = dev_i32(self.slot)
        if w.conv:
            cw = wl.conv_weights(w)
            self.conv_w = cw.astype(F64)
            self.conv_w_dev = dev_f32(cw)
        self.kda = wl.kda_gate_params(w) if w.kda_full else None
        if self.kda:
            self.kda_dev = {n: dev_f32(self.kda[n]) for n in ("a_log", "dt_bias", "out_norm_w")}
        self.t = 0
        self.ref_outputs = []

    def gates(self, x):
        """(log_decay input, beta input) as both sides receive them."""
        if self.w.kda_full:
            return x["f"], x["b_raw"]
        if self.gate_raw:
            return x["a_raw"], x["b_raw"]
        return x["lam"], x["beta"]

    def device_inputs(self, x, v: Variant):
        w = self.w
        lam, beta = self.gates(x)
        # raw-value workloads pass no beta (NULL: beta = 1); the oracle gets ones
        d = dict(log_decay=dev_f32(lam), beta=None if w.raw_value else dev_f32(beta), slot=self.slot_dev)
        if w.conv:
            d["mixed_qkv"] = dev_bf16(x["mixed_bits"]) if w.qkv_bf16 else dev_f32(x["mixed"])
            d["conv_w"] = self.conv_w_dev
            d["conv_pool"] = v.pools.conv
        else:
            for n in ("q", "k", "v"):
                d[n] = dev_bf16(x[n + "_bits"]) if w.qkv_bf16 else dev_f32(x[n])
        if w.kda_full:
            d.update(self.kda_dev, out_gate=dev_f32(x["out_gate"]))
        return d

    def step(self):
        w = self.w
        x = wl.step_inputs(w, self.t, batch=self.B)
        lam, beta = self.gates(x)
        kw = dict(lam=lam.astype(F64), beta=beta.astype(F64))
        if w.kda_full:
            kw.update(a_log=self.kda["a_log"].astype(F64), dt_bias=self.kda["dt_bias"].astype(F64),
                      out_norm_w=self.kda["out_norm_w"].astype(F64), out_gate=x["out_gate"].astype(F64),
                      lower_bound=self.kda["lower_bound"])
        if w.conv:
            kw.update(mixed=x["mixed"].astype(F64), conv_w=self.conv_w)
        else:
            kw.update(q=x["q"].astype(F64), k=x["k"].astype(F64), v=x["v"].astype(F64))
        o_ref = oracle.step_batch(self.cfg, "dense", self.ost, self.slot, **kw)
        live = self.slot >= 0
        keep_alive = []
        for v in self.variants:
            d = self.device_inputs(x, v)
            keep_alive.append(d)
            v.step(gdn.make_inputs(**d))
        torch.cuda.synchronize()
        for v in self.variants:
            o = v.o.cpu().numpy().astype(F64)
            v.max_err = max(v.max_err, float(np.max(np.abs(o[live] - o_ref[live]), initial=0.0)))
            v.max_ref = max(v.max_ref, float(np.max(np.abs(o_ref[live]), initial=0.0)))
            if self.keep:
                v.outputs.append(o)
        if self.keep:
            self.ref_outputs.append(o_ref.copy())
        self.t += 1
        return x

    def run(self, steps=None):
        for _ in range(self.w.steps if steps is None else steps):
            self.step()
        return self

    def compare_states(self):
        """Final state (dense) / base (DeltaLog, valid after whole cycles) vs the oracle."""
        S_ref = self.ost.S
        used = sorted({int(s) for s in self.slot if s >= 0})
        for v in self.variants:
            if v.mode == "deltalog" and (v.t % v.M) != 0:
                continue
            S = v.pools.state.cpu().numpy().astype(F64)
            v.state_err = float(np.max(np.abs(S[used] - S_ref[used])))
            v.state_ref = float(np.max(np.abs(S_ref[used])))
        return self

    def status(self, v: Variant) -> int:
        return int(v.status.item())
