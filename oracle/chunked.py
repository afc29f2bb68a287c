"""Chunkwise (prefill-style) forms of the same recurrences, numpy fp64.

TEST INFRASTRUCTURE: used only to pin the C recurrence in ``gdn_oracle.c``
against an independent algorithm that reaches the same result by a different
route (block matrix products and a unit-lower-triangular solve instead of a
token-by-token scan).

State convention: S[dk, dv], readout o = S^T q, row scaling by the decay.

Sources:
  * ``gla_chunked`` -- "线性注意力与混合架构的推理" (inference handbook), section
    "同一个计算的两种写法": inside a chunk, a causal score matrix with a
    cumulative-decay mask; between chunks only the state is carried.
  * ``delta_chunked_wy`` -- "深度解析线性注意力机制演进与 AI Infra 实现", section
    "Prefill中的Chunk微观并行", sub-section "完整计算顺序" (six steps: prefix sums
    of the log-gates, the two decayed key matrices, the strictly lower
    triangular A and (I+A)^{-1}, the local residuals U and the correction
    directions W, the chunk-end state, the in-chunk readout with M). The page
    stores S as [dv, dk]; everything below is transposed to S[dk, dv].
"""
from __future__ import annotations

import numpy as np


def _chunks(T: int, C: int):
    for s in range(0, T, C):
        yield s, min(s + C, T)


def gla_chunked(q, k, v, log_alpha, C, S0=None):
    """Gated linear attention S_t = alpha_t S_{t-1} + k_t v_t^T, o_t = S_t^T q_t,
    evaluated chunk by chunk.

    q, k: [T, dk]; v: [T, dv]; log_alpha: [T] (scalar decay per step).
    Returns (o [T, dv], S_T [dk, dv]).
    """
    q, k, v, la = (np.asarray(x, dtype=np.float64) for x in (q, k, v, log_alpha))
    T, dk = k.shape
    S = np.zeros((dk, v.shape[1])) if S0 is None else np.array(S0, dtype=np.float64)
    out = np.zeros((T, v.shape[1]))
    for s, e in _chunks(T, C):
        G = np.cumsum(la[s:e])                 # decay accumulated from chunk start, per row
        n = e - s
        i_idx, j_idx = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
        causal = j_idx <= i_idx
        # weight of token j as seen from token i inside the chunk: prod_{j<t<=i} alpha_t
        expo = np.where(causal, G[:, None] - G[None, :], -np.inf)
        scores = (q[s:e] @ k[s:e].T) * np.exp(expo)
        out[s:e] = scores @ v[s:e] + np.exp(G)[:, None] * (q[s:e] @ S)
        S = np.exp(G[-1]) * S + (np.exp(G[-1] - G)[:, None] * k[s:e]).T @ v[s:e]
    return out, S


def delta_chunked_wy(q, k, v, beta, log_gate, C, S0=None):
    """Gated delta rule evaluated with the chunkwise WY/UT algebra.

    Recurrence being reproduced (one token): Sbar = D(g_t) S_{t-1};
    r_t = beta_t (v_t - Sbar^T k_t); S_t = Sbar + k_t r_t^T; o_t = S_t^T q_t.

    q, k: [T, dk]; v: [T, dv]; beta: [T]; log_gate: [T, dk] (per-key log-decay;
    a per-head scalar decay is the same value repeated along dk).
    Returns (o [T, dv], S_T [dk, dv]).
    """
    q, k, v, beta, g = (np.asarray(x, dtype=np.float64) for x in (q, k, v, beta, log_gate))
    T, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    out = np.zeros((T, dv))
    for s, e in _chunks(T, C):
        n = e - s
        Kc, Vc, Qc, bc = k[s:e], v[s:e], q[s:e], beta[s:e]
        # step 1: prefix sums of the log-gates inside the chunk, G[i] = g_1 + ... + g_i
        G = np.cumsum(g[s:e], axis=0)                       # [n, dk]
        # step 2: key decayed from chunk start (K_in), key decayed to chunk end (K_g)
        K_in = Kc * np.exp(G)
        K_g = Kc * np.exp(G[-1][None, :] - G)
        # step 3: A_ij = beta_i k_i^T (k_j * exp(G_i - G_j)) for j < i
        diff = G[:, None, :] - G[None, :, :]                 # [n, n, dk], row i, column j
        strict = (np.arange(n)[None, :] < np.arange(n)[:, None])
        expo = np.where(strict[:, :, None], diff, -np.inf)
        A = bc[:, None] * np.einsum("id,ijd,jd->ij", Kc, np.exp(expo), Kc)
        I_plus_A = np.eye(n) + A
        # step 4: U = (I+A)^{-1} B V, W = (I+A)^{-1} B K_in
        U = np.linalg.solve(I_plus_A, bc[:, None] * Vc)
        W = np.linalg.solve(I_plus_A, bc[:, None] * K_in)
        # step 5: actual residuals E = U - W S0; chunk-end state
        E = U - W @ S
        S_end = np.exp(G[-1])[:, None] * S + K_g.T @ E
        # step 6: readout, M_ij = q_i^T (k_j * exp(G_i - G_j)) for j <= i (diagonal kept)
        lower = (np.arange(n)[None, :] <= np.arange(n)[:, None])
        expo_m = np.where(lower[:, :, None], diff, -np.inf)
        Mq = np.einsum("id,ijd,jd->ij", Qc, np.exp(expo_m), Kc)
        out[s:e] = (Qc * np.exp(G)) @ S + Mq @ E
        S = S_end
    return out, S
