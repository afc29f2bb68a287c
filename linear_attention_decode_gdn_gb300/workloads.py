"""Seeded synthetic inputs for the batched GDN decode step.

This module only draws random numbers and shapes them; it holds none of the
decode arithmetic, so the CUDA path and the CPU oracle can both be fed from it
without sharing any computation. numpy only (no torch), so it also runs where
no GPU or CUDA library is present.

Draw recipe (per workload, per decode step t):
  * generator: numpy PCG64 seeded with SeedSequence([seed, t]); conv weights
    use SeedSequence([seed, 1 << 20]).
  * order: (q, k, v) -- or mixed_qkv when the short conv is fused -- then the
    decay draw, then the write-gate draw.
  * q, k ~ N(0,1) * qk_mult, v ~ N(0,1); for bf16 workloads each value is
    rounded to bf16 (round-to-nearest-even) and both sides see that value.
  * alpha = sigmoid(N(0,1) + 3), lambda = log(alpha) (per head, or per key
    channel for the per-key-decay workload); beta = sigmoid(N(0,1)); both fp32.
  * conv weights N(0,1) * 0.5 (standard deviation 0.5), fp32, no bias.
  * raw-value workloads (the RWKV6 instantiation): the write-gate draw is made and
    discarded, beta = 1; q and k are not L2-normalised, so they are drawn with
    qk_mult = 1/sqrt(dk) (unit expected norm).
  * workloads with the full KDA gate and output epilogue: the forget pre-activation
    is f = (decay draw) - 3 ~ N(0,1), the write logit is the raw write-gate draw, and
    the output-gate logits g ~ N(0,1) [B,H,dv] are drawn after them. Per-head
    parameters come once from SeedSequence([seed, 2 << 20]): A_log = log U(1, 16)
    [H], dt_bias = -4 + 0.5 N(0,1) [H, dlam], RMSNorm weight 1 + 0.1 N(0,1) [dv];
    lower bound -5. With these, alpha = exp(lambda) lies mostly in (0.9, 1).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_heads: int
    dk: int
    dv: int
    steps: int
    merge_intervals: tuple
    qkv_bf16: bool
    conv: bool
    decay_per_key: bool
    seed: int
    qk_mult: float = 1.0
    conv_w_std: float = 0.5
    raw_value: bool = False  # RWKV6 update S <- D(lambda) S + k v^T: beta = 1, no correction
                             # and no L2 norm; K and U logs bf16
    kda_full: bool = False   # KDA gate parametrisation and output epilogue (RMSNorm, gate)
    description: str = field(default="", compare=False)

    @property
    def dlam(self) -> int:
        return self.dk if self.decay_per_key else 1

    @property
    def channels(self) -> int:
        return 2 * self.num_heads * self.dk + self.num_heads * self.dv

    @property
    def state_bytes(self) -> int:
        return 4 * self.batch * self.num_heads * self.dk * self.dv


WORKLOADS = {
    w.name: w
    for w in (
        Workload("tiny", 1, 2, 16, 16, 64, (4,), False, False, False, 1001, qk_mult=0.25,
                 description="B=1, H=2, dk=dv=16, fp32 q/k/v (randn/4, L2-normalised), 64 steps, M=4"),
        Workload("small_conv", 64, 16, 128, 128, 128, (8,), True, True, False, 1002,
                 description="B=64, H=16, dk=dv=128, bf16 mixed_qkv through the width-4 conv, 128 steps, M=8"),
        Workload("headline", 128, 32, 128, 128, 128, (1, 8), True, False, False, 1003,
                 description="B=128, H=32, dk=dv=128, fp32 state 256 MiB, bf16 q/k/v, 128 steps, M in {1, 8}"),
        Workload("high_concurrency", 512, 32, 128, 128, 128, (1, 2, 4, 8, 16), True, False, False,
                 1004, description="B=512, H=32, dk=dv=128, fp32 state 1 GiB, 128 steps, M in {1,2,4,8,16}"),
        Workload("kda", 256, 32, 128, 128, 128, (8,), True, False, True, 1005,
                 description="B=256, H=32, dk=dv=128, per-key-channel log decay (width 128), 128 steps, M=8"),
        Workload("kda_full", 256, 32, 128, 128, 128, (8,), True, False, True, 1007, kda_full=True,
                 description="B=256, H=32, dk=dv=128, KDA with its gate parametrisation "
                             "(lower_bound sigmoid(exp(A_log)(f + dt_bias))) and output epilogue "
                             "(RMSNorm, sigmoid output gate), 128 steps, M=8"),
        Workload("rwkv6", 128, 32, 128, 128, 128, (1, 4), True, False, True, 1006, qk_mult=128 ** -0.5,
                 raw_value=True,
                 description="B=128, H=32, dk=dv=128, per-key-channel log decay, raw-value update "
                             "(beta = 1, no correction, no L2 norm), bf16 K and U logs, 128 steps, M in {1, 4}"),
    )
}


def bf16_round(x: np.ndarray):
    """Round float32 values to bf16 (nearest-even). Returns (uint16 bits, float32 values)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    bits = rounded.astype(np.uint16)
    vals = (bits.astype(np.uint32) << 16).view(np.float32)
    return bits, vals


def _rng(seed: int, t: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, t])))


def _gates(rng, w: Workload, batch: int):
    a_raw = rng.standard_normal((batch, w.num_heads, w.dlam)) + 3.0
    b_raw = rng.standard_normal((batch, w.num_heads))
    lam = (-np.log1p(np.exp(-a_raw))).astype(np.float32)      # log(sigmoid(a_raw))
    beta = (1.0 / (1.0 + np.exp(-b_raw))).astype(np.float32)   # sigmoid(b_raw)
    return lam, beta, a_raw.astype(np.float32), b_raw.astype(np.float32)


def step_inputs(w: Workload, t: int, batch: int | None = None) -> dict:
    """Inputs of decode step ``t`` (0-based). ``batch`` overrides the workload's B
    (a prefix of the same draw is NOT implied: a different B is a different draw).

    Returned keys (numpy):
      q, k, v          float32 [B,H,d] (exact values; bf16-representable for bf16 workloads)
      q_bits, k_bits, v_bits  uint16 bf16 bit patterns (bf16 workloads only)
      mixed, mixed_bits  float32 / uint16 [B, channels] (conv workloads only)
      lam              float32 [B,H,dlam]   log-decay
      beta             float32 [B,H]
      a_raw, b_raw     float32 raw gate draws (lam = logsigmoid(a_raw), beta = sigmoid(b_raw))
    """
    B = w.batch if batch is None else batch
    rng = _rng(w.seed, t)
    out = {}
    if w.conv:
        m = rng.standard_normal((B, w.channels), dtype=np.float32)
        if w.qkv_bf16:
            out["mixed_bits"], out["mixed"] = bf16_round(m)
        else:
            out["mixed"] = m
    else:
        H = w.num_heads
        q = rng.standard_normal((B, H, w.dk), dtype=np.float32) * np.float32(w.qk_mult)
        k = rng.standard_normal((B, H, w.dk), dtype=np.float32) * np.float32(w.qk_mult)
        v = rng.standard_normal((B, H, w.dv), dtype=np.float32)
        for name, arr in (("q", q), ("k", k), ("v", v)):
            if w.qkv_bf16:
                out[name + "_bits"], out[name] = bf16_round(arr)
            else:
                out[name] = arr
    lam, beta, a_raw, b_raw = _gates(rng, w, B)
    if w.raw_value:
        beta = np.ones_like(beta)
    out.update(lam=lam, beta=beta, a_raw=a_raw, b_raw=b_raw)
    if w.kda_full:
        out["f"] = (a_raw - np.float32(3)).astype(np.float32)
        out["out_gate"] = rng.standard_normal((B, w.num_heads, w.dv), dtype=np.float32)
    return out


def kda_gate_params(w: Workload) -> dict:
    """Per-head KDA gate and epilogue parameters (fp32), drawn once per workload."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, 2 << 20])))
    return {
        "a_log": np.log(rng.uniform(1.0, 16.0, size=w.num_heads)).astype(np.float32),
        "dt_bias": (-4.0 + 0.5 * rng.standard_normal((w.num_heads, w.dlam))).astype(np.float32),
        "out_norm_w": (1.0 + 0.1 * rng.standard_normal(w.dv)).astype(np.float32),
        "lower_bound": -5.0,
    }


def conv_weights(w: Workload) -> np.ndarray:
    """Conv weights [channels, 4] fp32, N(0,1) * conv_w_std."""
    rng = _rng(w.seed, 1 << 20)
    return (rng.standard_normal((w.channels, 4), dtype=np.float32) * np.float32(w.conv_w_std))


def identity_slots(batch: int) -> np.ndarray:
    return np.arange(batch, dtype=np.int32)
