"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Every check here is independent of the oracle's own code path:
  * the scalar worked example printed in the DeltaLog notes (Sec. 2.3),
  * an independent chunkwise algorithm (handbook "同一个计算的两种写法" for
    gated linear attention; the evolution article's WY/UT "完整计算顺序" for
    the gated delta rule),
  * closed forms and invariants from the evolution article (appendix 附2:
    non-expansion of I - beta k k^T, the k-readout blend, orthogonal queries;
    the additive special case S + k v^T),
  * brute force from the full input history for the short convolution,
  * DeltaLog base+log emulation == dense recurrence (Eq. (7) invariant).
A planted-mistake test compiles copies of the oracle with one plausible
mistake each and checks that at least one pin fails for every copy.
"""
import math
import os
import shutil
import tempfile

import numpy as np
import pytest

import oracle
from oracle import chunked

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _unit(x):
    return x / np.linalg.norm(x)


# ----------------------------------------------------------------------------
# pins, each a function of the oracle library so planted mistakes can be run
# ----------------------------------------------------------------------------

def _load_teaching():
    rows = []
    with open(os.path.join(GOLDEN, "deltalog_teaching_example.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([float(x) for x in line.split()])
    return rows


def pin_teaching_dense(lib):
    """Immediate-update column of the teaching table: 7, 6.5, 7.25."""
    rows = _load_teaching()
    for d in (1, 16):
        S = np.zeros((d, d))
        S[0, 0] = 10.0
        e0 = np.zeros(d)
        e0[0] = 1.0
        for step, inc, logical, _base in rows:
            v = inc * e0
            o = oracle.gdn_step(S, e0.copy(), e0.copy(), v, [math.log(0.5)], 1.0, plain=True, lib=lib)
            assert abs(o[0] - logical) < 1e-12, (d, step, o[0], logical)
            assert abs(S[0, 0] - logical) < 1e-12


def pin_teaching_deltalog(lib):
    """Base column of the teaching table (10, 10, 7.25) and the log contents behind the
    representations 10/2+2, 10/4+2/2+3, 10/8+2/4+3/2+4."""
    rows = _load_teaching()
    st = oracle.HeadLog(1, 1, C=2, dlam=1, base=[[10.0]])
    one = np.ones(1)
    ln_half = math.log(0.5)
    for step, inc, logical, base in rows:
        o = oracle.deltalog_step(st, one.copy(), one.copy(), np.array([inc]), [ln_half], 1.0,
                                 plain=True, lib=lib)
        assert abs(o[0] - logical) < 1e-12, (step, o[0], logical)
        assert abs(st.base[0, 0] - base) < 1e-12, (step, st.base[0, 0], base)
        assert abs(st.logical_state()[0, 0] - logical) < 1e-12
        if step == 1:
            assert st.length[0] == 1 and abs(st.ell[0] - ln_half) < 1e-15
            assert st.klog[0, 0] == 1.0 and st.ulog[0, 0] == 2.0 and abs(st.lam[0, 0] - ln_half) < 1e-15
        if step == 2:
            assert st.length[0] == 2 and abs(st.ell[0] - 2 * ln_half) < 1e-15
            assert st.ulog[1, 0] == 3.0 and abs(st.lam[1, 0] - 2 * ln_half) < 1e-15
            # 10/4 + 2/2 + 3: base weight exp(ell)=1/4, entry 0 weight exp(ell-Lam0)=1/2, entry 1 weight 1
            assert abs(math.exp(st.ell[0]) - 0.25) < 1e-15
            assert abs(math.exp(st.ell[0] - st.lam[0, 0]) - 0.5) < 1e-15
            assert st.ell[0] == st.lam[1, 0]
        if step == 3:
            assert st.length[0] == 0 and st.ell[0] == 0.0


def pin_gla_chunked(lib, T=64, dk=16, dv=16, C=16, seed=0):
    """Recurrent (oracle, plain update with beta=1) == chunked gated linear attention."""
    r = _rng(seed)
    q, k = r.standard_normal((T, dk)) / 4, r.standard_normal((T, dk)) / 4
    v = r.standard_normal((T, dv))
    alpha = 1.0 / (1.0 + np.exp(-(r.standard_normal(T) + 3.0)))
    S = np.zeros((dk, dv))
    o_rec = np.stack([oracle.gdn_step(S, q[t].copy(), k[t].copy(), v[t].copy(), [math.log(alpha[t])],
                                      1.0, plain=True, lib=lib) for t in range(T)])
    o_ch, S_ch = chunked.gla_chunked(q, k, v, np.log(alpha), C)
    assert np.max(np.abs(o_rec - o_ch)) <= 1e-12 * np.max(np.abs(o_ch)), np.max(np.abs(o_rec - o_ch))
    assert np.max(np.abs(S - S_ch)) <= 1e-12 * np.max(np.abs(S_ch))


def pin_delta_wy(lib, T=64, dk=16, dv=16, C=16, per_key=False, seed=1):
    """Recurrent gated delta rule (oracle) == WY/UT chunkwise algebra, nonzero S0."""
    r = _rng(seed)
    q = np.stack([_unit(x) for x in r.standard_normal((T, dk))])
    k = np.stack([_unit(x) for x in r.standard_normal((T, dk))])
    v = r.standard_normal((T, dv))
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal(T)))
    if per_key:
        g = -np.log1p(np.exp(-(r.standard_normal((T, dk)) + 3.0)))
    else:
        g = np.repeat(-np.log1p(np.exp(-(r.standard_normal((T, 1)) + 3.0))), dk, axis=1)
    S0 = r.standard_normal((dk, dv))
    S = S0.copy()
    o_rec = []
    for t in range(T):
        lam = g[t] if per_key else g[t, :1]
        o_rec.append(oracle.gdn_step(S, q[t].copy(), k[t].copy(), v[t].copy(), lam, beta[t], lib=lib))
    o_rec = np.stack(o_rec)
    o_ch, S_ch = chunked.delta_chunked_wy(q, k, v, beta, g, C, S0=S0)
    assert np.max(np.abs(o_rec - o_ch)) <= 1e-10 * np.max(np.abs(o_ch)), np.max(np.abs(o_rec - o_ch))
    assert np.max(np.abs(S - S_ch)) <= 1e-10 * np.max(np.abs(S_ch))


def pin_transition_form(lib, dk=7, dv=5, seed=2):
    """One step equals the affine form S_t = (I - beta k k^T) D(lambda) S_{t-1} + beta k v^T
    (the state-transition form of the gated delta rule, with D on the rows)."""
    r = _rng(seed)
    for per_key in (False, True):
        S0 = r.standard_normal((dk, dv))
        q, k, v = r.standard_normal(dk), _unit(r.standard_normal(dk)), r.standard_normal(dv)
        lam = -np.abs(r.standard_normal(dk if per_key else 1)) * 0.3
        beta = 0.7
        S = S0.copy()
        o = oracle.gdn_step(S, q.copy(), k.copy(), v.copy(), lam, beta, lib=lib)
        D = np.diag(np.exp(lam if per_key else np.repeat(lam, dk)))
        S_ref = (np.eye(dk) - beta * np.outer(k, k)) @ D @ S0 + beta * np.outer(k, v)
        assert np.allclose(S, S_ref, rtol=0, atol=1e-13)
        assert np.allclose(o, S_ref.T @ q, rtol=0, atol=1e-13)


def pin_invariants(lib, dk=16, dv=12, seed=3):
    """Non-expansion (v = 0, unit k, 0<=beta<=1, alpha<=1), the k-readout blend
    (1-beta) Sbar^T k + beta v, orthogonal queries read Sbar^T q, and the additive
    special case S_1 = S_0 + k v^T at alpha = beta = 1 with k^T S_0 = 0."""
    r = _rng(seed)
    S = r.standard_normal((dk, dv))
    for t in range(50):
        k = _unit(r.standard_normal(dk))
        lam = [-abs(r.standard_normal()) * 0.1]
        n0 = np.linalg.norm(S)
        oracle.gdn_step(S, k.copy(), k.copy(), np.zeros(dv), lam, float(r.uniform(0, 1)), lib=lib)
        assert np.linalg.norm(S) <= n0 * (1 + 1e-12)
    # k-readout blend and orthogonal query
    S0 = r.standard_normal((dk, dv))
    k = _unit(r.standard_normal(dk))
    v = r.standard_normal(dv)
    lam, beta = [-0.2], 0.35
    Sbar = math.exp(lam[0]) * S0
    S = S0.copy()
    o_k = oracle.gdn_step(S, k.copy(), k.copy(), v.copy(), lam, beta, lib=lib)
    assert np.allclose(o_k, (1 - beta) * (Sbar.T @ k) + beta * v, atol=1e-13, rtol=0)
    qo = r.standard_normal(dk)
    qo -= (qo @ k) * k
    S = S0.copy()
    o_q = oracle.gdn_step(S, qo.copy(), k.copy(), v.copy(), lam, beta, lib=lib)
    assert np.allclose(o_q, Sbar.T @ qo, atol=1e-13, rtol=0)
    # additive special case
    S0 = r.standard_normal((dk, dv))
    S0 -= np.outer(k, k @ S0)  # now k^T S0 = 0
    q = r.standard_normal(dk)
    S = S0.copy()
    o = oracle.gdn_step(S, q.copy(), k.copy(), v.copy(), [0.0], 1.0, lib=lib)
    assert np.allclose(S, S0 + np.outer(k, v), atol=1e-13, rtol=0)
    assert np.allclose(o, (S0 + np.outer(k, v)).T @ q, atol=1e-12, rtol=0)


def pin_conv(lib, nch=6, T=9, seed=4):
    """Causal conv + SiLU through the rolling 3-column state == brute force from the full
    input history (zeros before t=0); identity taps pick x_t and x_{t-3}."""
    r = _rng(seed)
    x = r.standard_normal((T, nch))
    w = r.standard_normal((nch, 4))
    bias = r.standard_normal(nch)
    silu = lambda z: z / (1 + np.exp(-z))
    for wt, bt in ((w, bias), (w, None)):
        cs = np.zeros((nch, 3))
        for t in range(T):
            y = oracle.conv1d_silu(x[t].copy(), cs, wt.copy(), None if bt is None else bt.copy(), lib=lib)
            hist = [x[t - 3 + j] if t - 3 + j >= 0 else np.zeros(nch) for j in range(4)]
            z = sum(hist[j] * wt[:, j] for j in range(4)) + (0 if bt is None else bt)
            assert np.allclose(y, silu(z), atol=1e-14, rtol=0)
    for tap, lag in ((3, 0), (0, 3), (1, 2), (2, 1)):
        we = np.zeros((nch, 4))
        we[:, tap] = 1.0
        cs = np.zeros((nch, 3))
        for t in range(T):
            y = oracle.conv1d_silu(x[t].copy(), cs, we, lib=lib)
            src = x[t - lag] if t - lag >= 0 else np.zeros(nch)
            assert np.allclose(y, silu(src), atol=1e-15, rtol=0)


def pin_l2norm(lib):
    x = np.array([3.0, 4.0])
    y, inv = oracle.l2norm(x, 0.0, lib=lib)
    assert np.allclose(y, [0.6, 0.8], atol=1e-16) and abs(inv - 0.2) < 1e-16
    y, inv = oracle.l2norm(x, 11.0, scale=2.0, lib=lib)  # sqrt(25 + 11) = 6
    assert np.allclose(y, [1.0, 4.0 / 3.0], atol=1e-15) and abs(inv - 1 / 6) < 1e-16
    y, _ = oracle.l2norm(np.zeros(4), 1e-6, lib=lib)
    assert np.all(y == 0.0)


def _batch_cfg(B, H, dk, dv, slots, dlam, C, flags, q_scale=1.0, eps=1e-6):
    return dict(batch=B, num_heads=H, dk=dk, dv=dv, num_slots=slots, dlam=dlam, log_capacity=C,
                flags=flags, q_scale=q_scale, l2_eps=eps)


def pin_deltalog_equals_dense(lib, B=3, H=2, dk=8, dv=6, T=20, seed=5):
    """Base+log emulation (Eq. (7), Algorithm 1, Eq. (6)) == dense recurrence at every step,
    for scalar and per-key decay, delta and plain updates, M in {1,2,3,4,8}; the base equals
    the dense state after every merge."""
    r = _rng(seed)
    for per_key in (False, True):
        for plain in (False, True):
            for M in (1, 2, 3, 4, 8):
                C = M - 1
                dlam = dk if per_key else 1
                flags = oracle.L2NORM | (oracle.PLAIN if plain else 0)
                cfg = _batch_cfg(B, H, dk, dv, B + 1, dlam, C, flags, q_scale=0.5)
                slot = np.array([2, 0, 3], dtype=np.int32)
                sd = oracle.BatchState(B + 1, H, dk, dv, dlam, C)
                sl = oracle.BatchState(B + 1, H, dk, dv, dlam, C)
                init = r.standard_normal(sd.S.shape)
                sd.S[:] = init
                sl.S[:] = init
                for t in range(T):
                    q, k = r.standard_normal((B, H, dk)), r.standard_normal((B, H, dk))
                    v = r.standard_normal((B, H, dv))
                    lam = -np.log1p(np.exp(-(r.standard_normal((B, H, dlam)) + 3)))
                    beta = 1 / (1 + np.exp(-r.standard_normal((B, H))))
                    od = oracle.step_batch(cfg, "dense", sd, slot, q=q, k=k, v=v, lam=lam, beta=beta, lib=lib)
                    ol = oracle.step_batch(cfg, "deltalog", sl, slot, q=q, k=k, v=v, lam=lam, beta=beta, lib=lib)
                    assert np.max(np.abs(od - ol)) <= 1e-12 * max(1.0, np.max(np.abs(od))), (per_key, plain, M, t)
                    assert np.all(sl.len[slot] == (t + 1) % M)
                    if (t + 1) % M == 0:
                        assert np.allclose(sl.S, sd.S, atol=1e-12, rtol=0)
                # untouched slot 1 stays at its initial value
                assert np.array_equal(sd.S[1], init[1]) and np.array_equal(sl.S[1], init[1])


def pin_batch_glue(lib, seed=6):
    """orc_step_batch with the fused conv, L2 norm, q scale and raw gates == the single-head
    primitives driven by hand (channel order [q heads | k heads | v heads], slot indirection,
    padding rows untouched)."""
    r = _rng(seed)
    B, H, dk, dv, slots = 3, 2, 4, 5, 4
    nch = 2 * H * dk + H * dv
    slot = np.array([1, -1, 3], dtype=np.int32)
    cfg = _batch_cfg(B, H, dk, dv, slots, 1, 0,
                     oracle.CONV | oracle.L2NORM | oracle.GATE_RAW, q_scale=0.25, eps=1e-3)
    st = oracle.BatchState(slots, H, dk, dv)
    st.S[:] = r.standard_normal(st.S.shape)
    st.conv[:] = r.standard_normal(st.conv.shape)
    S_ref, conv_ref = st.S.copy(), st.conv.copy()
    w = r.standard_normal((nch, 4))
    mixed = r.standard_normal((B, nch))
    a_raw, b_raw = r.standard_normal((B, H, 1)), r.standard_normal((B, H))
    o_in = np.full((B, H, dv), 7.0)
    o = oracle.step_batch(cfg, "dense", st, slot, mixed=mixed, conv_w=w, lam=a_raw, beta=b_raw,
                          o=o_in.copy(), lib=lib)
    silu = lambda z: z / (1 + np.exp(-z))
    for b in range(B):
        s = slot[b]
        if s < 0:
            assert np.all(o[b] == 7.0)
            continue
        cs = conv_ref[s]
        z = (cs * w[:, :3]).sum(1) + mixed[b] * w[:, 3]
        y = silu(z)
        assert np.allclose(st.conv[s], np.concatenate([cs[:, 1:], mixed[b][:, None]], 1))
        for h in range(H):
            qv = y[h * dk:(h + 1) * dk]
            kv = y[H * dk + h * dk:H * dk + (h + 1) * dk]
            vv = y[2 * H * dk + h * dv:2 * H * dk + (h + 1) * dv]
            qn = 0.25 * qv / math.sqrt(qv @ qv + 1e-3)
            kn = kv / math.sqrt(kv @ kv + 1e-3)
            lam = math.log(1 / (1 + math.exp(-a_raw[b, h, 0])))
            beta = 1 / (1 + math.exp(-b_raw[b, h]))
            S = S_ref[s, h].copy()
            oh = oracle.gdn_step(S, qn, kn, vv.copy(), [lam], beta, lib=lib)
            assert np.allclose(o[b, h], oh, atol=1e-13, rtol=0)
            assert np.allclose(st.S[s, h], S, atol=1e-13, rtol=0)
    assert np.array_equal(st.S[0], S_ref[0]) and np.array_equal(st.S[2], S_ref[2])


def pin_prenorm_log(lib, seed=7):
    """Pre-normalisation key variant: K_log holds the raw key exactly, U_log holds the value
    factor scaled by the key's inverse norm, and outputs still equal the dense recurrence."""
    r = _rng(seed)
    B, H, dk, dv, M = 2, 2, 8, 8, 4
    C = M - 1
    cfg_l = _batch_cfg(B, H, dk, dv, B, 1, C, oracle.L2NORM | oracle.KLOG_PRENORM)
    cfg_d = _batch_cfg(B, H, dk, dv, B, 1, C, oracle.L2NORM)
    sl, sd = oracle.BatchState(B, H, dk, dv, 1, C), oracle.BatchState(B, H, dk, dv, 1, C)
    slot = np.arange(B, dtype=np.int32)
    for t in range(9):
        q, k, v = r.standard_normal((B, H, dk)), r.standard_normal((B, H, dk)), r.standard_normal((B, H, dv))
        lam = -np.log1p(np.exp(-(r.standard_normal((B, H, 1)) + 3)))
        beta = 1 / (1 + np.exp(-r.standard_normal((B, H))))
        n_before = sl.len.copy()
        ol = oracle.step_batch(cfg_l, "deltalog", sl, slot, q=q, k=k, v=v, lam=lam, beta=beta, lib=lib)
        od = oracle.step_batch(cfg_d, "dense", sd, slot, q=q, k=k, v=v, lam=lam, beta=beta, lib=lib)
        assert np.max(np.abs(ol - od)) <= 1e-12 * np.max(np.abs(od))
        for b in range(B):
            for h in range(H):
                n = n_before[b, h]
                if n < C:
                    assert np.array_equal(sl.klog[b, h, n], k[b, h])


def pin_verify_routing(lib, seed=11):
    """Speculative-decoding verify (inference handbook, "推测解码：验证后如何恢复状态") on a
    closed form: with lambda = 0, beta = 1 and the plain update, S_t = S_{t-1} + k_t v_t^T, and
    with orthonormal keys every row is a hand-summed matrix. Checks the row routing: the
    initial state is column num_accepted - 1 (read before that row is overwritten), the
    state after position t lands in column t, padding requests and other rows are untouched,
    o_t = S_t^T q_t."""
    r = _rng(seed)
    S, H, d, T = 10, 1, 8, 3
    pool = r.standard_normal((S, H, d, d))
    init = pool.copy()
    idx = np.array([[5, 2, 7], [-1, -1, -1], [0, 9, 3]], dtype=np.int32)
    na = np.array([2, 1, 3], dtype=np.int32)
    B = idx.shape[0]
    eye = np.eye(d)
    k = np.zeros((B, T, H, d))
    for b in range(B):
        for t in range(T):
            k[b, t, 0] = eye[(t + 2 * b) % d]
    q, v = r.standard_normal((B, T, H, d)), r.standard_normal((B, T, H, d))
    lam, beta = np.zeros((B, T, H, 1)), np.ones((B, T, H))
    cfg = _batch_cfg(B, H, d, d, S, 1, 0, oracle.PLAIN)
    o = oracle.verify_batch(cfg, pool, idx, na, q=q, k=k, v=v, lam=lam, beta=beta, lib=lib)
    for b in (0, 2):
        state = init[idx[b, na[b] - 1], 0].copy()
        for t in range(T):
            state = state + np.outer(k[b, t, 0], v[b, t, 0])
            assert np.max(np.abs(pool[idx[b, t], 0] - state)) <= 1e-12
            assert np.max(np.abs(o[b, t, 0] - state.T @ q[b, t, 0])) <= 1e-12
    assert np.all(o[1] == 0)
    for row in (1, 4, 6, 8):
        assert np.array_equal(pool[row], init[row])


def pin_kda_gate(lib):
    """KDA forget-gate parametrisation (evolution article, "KDA实现逻辑概述"):
    lambda = lower_bound * sigmoid(exp(A_log) (f + dt_bias)). Pinned by closed forms and
    identities, not by retyping it: z = 0 gives lower_bound / 2; sigmoid(z) + sigmoid(-z) = 1
    gives lambda(z) + lambda(-z) = lower_bound; A_log = log 2 equals doubling x; the range is
    (lower_bound, 0) and lambda falls as f grows."""
    lb = -5.0
    for a, dt in ((0.0, -0.5), (1.7, 2.25), (-1.3, 0.0)):
        assert oracle.kda_log_decay(-dt, a, dt, lb, lib) == lb / 2
    r = _rng(12)
    for _ in range(50):
        f, a, dt = r.normal(0, 2), r.uniform(-2, 2), r.normal(0, 1)
        lam = oracle.kda_log_decay(f, a, dt, lb, lib)
        mirror = oracle.kda_log_decay(-f - 2 * dt, a, dt, lb, lib)  # x -> -x
        assert lb < lam < 0 and abs(lam + mirror - lb) <= 1e-12
        assert abs(oracle.kda_log_decay(f, np.log(2.0), dt, lb, lib)
                   - oracle.kda_log_decay(2 * f + dt, 0.0, dt, lb, lib)) <= 1e-12
        assert oracle.kda_log_decay(f + 0.1, a, dt, lb, lib) < lam


def pin_out_norm_gate(lib):
    """KDA output epilogue o <- RMSNorm(o) (.) sigmoid(g): the worked value for o = (3, 4)
    at g = 0 is 1.5/sqrt(12.5) and 2/sqrt(12.5); with the gate open the output has unit
    RMS; it is invariant to scaling o; the weight multiplies channel-wise; flipping the
    gate's sign divides channel j by e^{g_j}."""
    y = oracle.out_norm_gate([3.0, 4.0], [0.0, 0.0], eps=0.0, lib=lib)
    assert np.max(np.abs(y - np.array([1.5, 2.0]) / np.sqrt(12.5))) <= 1e-15
    r = _rng(13)
    o, g, w = r.standard_normal(64), r.standard_normal(64), 1 + 0.1 * r.standard_normal(64)
    open_gate = oracle.out_norm_gate(o, np.full(64, 40.0), eps=0.0, lib=lib)
    assert abs(np.mean(open_gate ** 2) - 1.0) <= 1e-12
    assert np.max(np.abs(oracle.out_norm_gate(7.5 * o, g, eps=0.0, lib=lib)
                         - oracle.out_norm_gate(o, g, eps=0.0, lib=lib))) <= 1e-14
    y1 = oracle.out_norm_gate(o, g, None, 1e-6, lib)
    assert np.max(np.abs(oracle.out_norm_gate(o, g, w, 1e-6, lib) - w * y1)) <= 1e-14
    assert np.max(np.abs(y1 / oracle.out_norm_gate(o, -g, None, 1e-6, lib) - np.exp(g))) <= 1e-12


def pin_kda_batch_glue(lib, seed=14):
    """The batch step with the KDA gate and epilogue flags equals the plain batch step fed
    the gate function's lambda and sigmoid(beta), followed by the epilogue per head."""
    r = _rng(seed)
    B, H, d, M = 2, 2, 8, 3
    slot = np.arange(B, dtype=np.int32)
    a_log, dt = r.uniform(0, 2.7, H), -4 + 0.5 * r.standard_normal((H, d))
    w = 1 + 0.1 * r.standard_normal(d)
    for mode, C in (("dense", 0), ("deltalog", M - 1)):
        cfg_k = _batch_cfg(B, H, d, d, B, d, C, oracle.L2NORM | oracle.GATE_KDA | oracle.OUT_NORM_GATE)
        cfg_p = _batch_cfg(B, H, d, d, B, d, C, oracle.L2NORM)
        sk, sp = oracle.BatchState(B, H, d, d, d, C), oracle.BatchState(B, H, d, d, d, C)
        for t in range(7):
            q, k, v = r.standard_normal((B, H, d)), r.standard_normal((B, H, d)), r.standard_normal((B, H, d))
            f, logit, g = r.standard_normal((B, H, d)), r.standard_normal((B, H)), r.standard_normal((B, H, d))
            ok = oracle.step_batch(cfg_k, mode, sk, slot, q=q, k=k, v=v, lam=f, beta=logit, lib=lib,
                                   a_log=a_log, dt_bias=dt, out_gate=g, out_norm_w=w, lower_bound=-5.0)
            lam = np.array([[[oracle.kda_log_decay(f[b, h, c], a_log[h], dt[h, c], -5.0, lib)
                              for c in range(d)] for h in range(H)] for b in range(B)])
            op = oracle.step_batch(cfg_p, mode, sp, slot, q=q, k=k, v=v, lam=lam,
                                   beta=1 / (1 + np.exp(-logit)), lib=lib)
            for b in range(B):
                for h in range(H):
                    ref = oracle.out_norm_gate(op[b, h], g[b, h], w, 1e-6, lib)
                    assert np.max(np.abs(ok[b, h] - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


def pin_prefill_batch(lib, seed=15):
    """The batched prompt pass equals the independent WY/UT chunked algebra per (request,
    head) from the same initial state, for both decay widths, with ragged prompt lengths
    (rows past a prompt stay zero; padding requests and other pool rows stay untouched)."""
    r = _rng(seed)
    B, H, d, T, S = 3, 2, 8, 23, 5
    slot = np.array([4, -1, 1], dtype=np.int32)
    lens = np.array([23, 9, 11])
    for dlam in (1, d):
        pool = 0.3 * r.standard_normal((S, H, d, d))
        init = pool.copy()
        q, k = r.standard_normal((B, T, H, d)), r.standard_normal((B, T, H, d))
        v = r.standard_normal((B, T, H, d))
        lam = -np.log1p(np.exp(-(r.standard_normal((B, T, H, dlam)) + 3)))
        beta = 1 / (1 + np.exp(-r.standard_normal((B, T, H))))
        cfg = _batch_cfg(B, H, d, d, S, dlam, 0, oracle.L2NORM)
        o = oracle.prefill_batch(cfg, pool, slot, lens, q=q, k=k, v=v, lam=lam, beta=beta, lib=lib)
        for b in (0, 2):
            n = lens[b]
            for h in range(H):
                qn = np.array([x / np.sqrt(x @ x + 1e-6) for x in q[b, :n, h]])  # eps as in the step
                kn = np.array([x / np.sqrt(x @ x + 1e-6) for x in k[b, :n, h]])
                g = np.repeat(lam[b, :n, h], d // dlam, axis=1) if dlam == 1 else lam[b, :n, h]
                oc, Sc = chunked.delta_chunked_wy(qn, kn, v[b, :n, h], beta[b, :n, h], g, C=7,
                                                  S0=init[slot[b], h])
                assert np.max(np.abs(o[b, :n, h] - oc)) <= 1e-10 * max(1.0, np.max(np.abs(oc)))
                assert np.max(np.abs(pool[slot[b], h] - Sc)) <= 1e-10 * max(1.0, np.max(np.abs(Sc)))
            assert np.all(o[b, n:] == 0)
        assert np.all(o[1] == 0)
        for row in (0, 2, 3):
            assert np.array_equal(pool[row], init[row])


def _silu(z):
    return z / (1 + np.exp(-z))


def pin_verify_conv_window(lib, nch=5, T=4, rounds=7, seed=16):
    """Widened conv window of speculative-decoding verify (inference handbook, "推测解码：验证后
    如何恢复状态") against brute force over the accepted history: every round's conv outputs
    are SiLU(w . the last four inputs) of (accepted history, the round's inputs up to t), and
    the window afterwards holds the last T+2 of (history, round). Rounds accept 1..T positions
    (all T once); the first round enters a plain three-column cache with num_accepted = 1."""
    r = _rng(seed)
    w, bias = r.standard_normal((nch, 4)), r.standard_normal(nch)
    hist = [r.standard_normal(nch) for _ in range(3)]
    win = np.zeros((nch, T + 2))
    win[:, :3] = np.stack(hist, axis=1)
    na = 1
    for rd in range(rounds):
        x = r.standard_normal((T, nch))
        y = oracle.verify_conv_window(win, na, x.copy(), w, bias, lib=lib)
        for t in range(T):
            taps = (hist[-3:] + [x[u] for u in range(t + 1)])[-4:]
            z = sum(taps[j] * w[:, j] for j in range(4)) + bias
            assert np.allclose(y[t], _silu(z), atol=1e-14, rtol=0), (rd, t)
        assert np.array_equal(win, np.stack(hist[-2:] + [x[u] for u in range(T)], axis=1)), rd
        na = T if rd == 2 else int(r.integers(1, T + 1))
        hist += [x[u] for u in range(na)]
    for bad in (0, T + 1):
        try:
            oracle.verify_conv_window(win, bad, np.zeros((T, nch)), w, lib=lib)
        except ValueError:
            continue
        raise AssertionError(f"num_accepted {bad} accepted")


def pin_verify_conv_glue(lib, seed=17):
    """verify_batch with mixed_qkv == verify_batch on the q, k, v that brute-force conv outputs
    give, split [q heads | k heads | v heads]; the window row is the request's column-0 index,
    a padding request's window is untouched."""
    r = _rng(seed)
    B, T, H, d, S = 3, 3, 2, 4, 9
    nch = 3 * H * d
    idx = np.array([[4, 0, 7], [-1, -1, -1], [2, 8, 5]], dtype=np.int32)
    na = np.array([2, 1, 3], dtype=np.int32)
    pool = r.standard_normal((S, H, d, d)) * 0.3
    win = r.standard_normal((S, nch, T + 2))
    win0, pool0 = win.copy(), pool.copy()
    mixed = r.standard_normal((B, T, nch))
    w = r.standard_normal((nch, 4))
    lam = np.log(1 / (1 + np.exp(-(r.standard_normal((B, T, H, 1)) + 3))))
    beta = 1 / (1 + np.exp(-r.standard_normal((B, T, H))))
    cfg = _batch_cfg(B, H, d, d, S, 1, 0, oracle.L2NORM, q_scale=0.5)
    o = oracle.verify_batch(cfg, pool, idx, na, lam=lam, beta=beta, lib=lib, mixed=mixed, conv_w=w,
                            conv_window=win)
    qkv = np.zeros((B, T, nch))
    for b in (0, 2):
        seq = list(win0[idx[b, 0]][:, na[b] - 1: na[b] + 2].T) + list(mixed[b])
        for t in range(T):
            qkv[b, t] = _silu(sum(seq[t + j] * w[:, j] for j in range(4)))
    q = qkv[..., : H * d].reshape(B, T, H, d)
    k = qkv[..., H * d: 2 * H * d].reshape(B, T, H, d)
    v = qkv[..., 2 * H * d:].reshape(B, T, H, d)
    o_ref = oracle.verify_batch(cfg, pool0, idx, na, q=q, k=k, v=v, lam=lam, beta=beta, lib=lib)
    assert np.max(np.abs(o - o_ref)) <= 1e-12 and np.max(np.abs(pool - pool0)) <= 1e-12
    for row in range(S):
        if row not in (4, 2):
            assert np.array_equal(win[row], win0[row])


def pin_prefill_conv_glue(lib, seed=19):
    """prefill_batch with mixed_qkv == prefill_batch on the q, k, v that brute-force conv
    outputs give (history: the slot's three-column conv state, then the prompt), masked past
    each prompt length; afterwards each slot's conv state holds the last three inputs of
    (old state, prompt) and a padding request's state is untouched."""
    r = _rng(seed)
    B, T, H, d, S = 4, 7, 2, 4, 6
    nch = 3 * H * d
    slot = np.array([3, -1, 0, 5], dtype=np.int32)
    lens = np.array([7, 7, 2, 0])
    pool = r.standard_normal((S, H, d, d)) * 0.3
    cs = r.standard_normal((S, nch, 3))
    pool0, cs0 = pool.copy(), cs.copy()
    mixed = r.standard_normal((B, T, nch))
    w, cb = r.standard_normal((nch, 4)), r.standard_normal(nch)
    lam = np.log(1 / (1 + np.exp(-(r.standard_normal((B, T, H, 1)) + 3))))
    beta = 1 / (1 + np.exp(-r.standard_normal((B, T, H))))
    cfg = _batch_cfg(B, H, d, d, S, 1, 0, oracle.L2NORM, q_scale=0.5)
    o = oracle.prefill_batch(cfg, pool, slot, lens, lam=lam, beta=beta, lib=lib, mixed=mixed,
                             conv_w=w, conv_b=cb, conv_pool=cs)
    qkv = np.zeros((B, T, nch))
    for b in range(B):
        if slot[b] < 0:
            continue
        seq = list(cs0[slot[b]].T) + list(mixed[b, : lens[b]])
        for t in range(lens[b]):
            qkv[b, t] = _silu(sum(seq[t + j] * w[:, j] for j in range(4)) + cb)
        assert np.array_equal(cs[slot[b]], np.stack(seq[-3:], axis=1)), b
    q = qkv[..., : H * d].reshape(B, T, H, d)
    k = qkv[..., H * d: 2 * H * d].reshape(B, T, H, d)
    v = qkv[..., 2 * H * d:].reshape(B, T, H, d)
    o_ref = oracle.prefill_batch(cfg, pool0, slot, lens, q=q, k=k, v=v, lam=lam, beta=beta, lib=lib)
    assert np.max(np.abs(o - o_ref)) <= 1e-12 and np.max(np.abs(pool - pool0)) <= 1e-12
    for row in (1, 2, 4):
        assert np.array_equal(cs[row], cs0[row])


def pin_prefill_kda_glue(lib, seed=20):
    """prefill_batch with the KDA gate and output epilogue == prefill_batch on the decays the
    pinned kda_log_decay gives and beta = sigmoid(logit), each live row then passed through
    the pinned out_norm_gate; per-key decay, ragged prompts."""
    r = _rng(seed)
    B, T, H, d, S = 3, 5, 2, 4, 4
    slot = np.array([2, 0, 3], dtype=np.int32)
    lens = np.array([5, 3, 1])
    pool = r.standard_normal((S, H, d, d)) * 0.3
    pool0 = pool.copy()
    q, k, v = (r.standard_normal((B, T, H, d)) for _ in range(3))
    f = r.standard_normal((B, T, H, d)) - 3
    logit, g = r.standard_normal((B, T, H)), r.standard_normal((B, T, H, d))
    a_log, dt_bias = np.log(r.uniform(1, 16, H)), -4 + 0.5 * r.standard_normal((H, d))
    w = 1 + 0.1 * r.standard_normal(d)
    kda = dict(a_log=a_log, dt_bias=dt_bias, out_norm_w=w, lower_bound=-5.0)
    cfg = _batch_cfg(B, H, d, d, S, d, 0, oracle.L2NORM | oracle.GATE_KDA | oracle.OUT_NORM_GATE)
    o = oracle.prefill_batch(cfg, pool, slot, lens, q=q, k=k, v=v, lam=f, beta=logit, lib=lib,
                             out_gate=g, **kda)
    lam = np.zeros_like(f)
    for b, t, h, c in np.ndindex(f.shape):
        lam[b, t, h, c] = oracle.kda_log_decay(f[b, t, h, c], a_log[h], dt_bias[h, c], -5.0, lib=lib)
    cfg_plain = _batch_cfg(B, H, d, d, S, d, 0, oracle.L2NORM)
    o_plain = oracle.prefill_batch(cfg_plain, pool0, slot, lens, q=q, k=k, v=v, lam=lam,
                                   beta=1 / (1 + np.exp(-logit)), lib=lib)
    assert np.max(np.abs(pool - pool0)) <= 1e-12
    for b in range(B):
        for t in range(T):
            for h in range(H):
                want = (oracle.out_norm_gate(o_plain[b, t, h], g[b, t, h], w, lib=lib) if t < lens[b]
                        else np.zeros(d))
                assert np.max(np.abs(o[b, t, h] - want)) <= 1e-12, (b, t, h)


PINS = [pin_teaching_dense, pin_teaching_deltalog, pin_gla_chunked, pin_delta_wy,
        lambda lib: pin_delta_wy(lib, per_key=True), lambda lib: pin_delta_wy(lib, T=50, dk=8, dv=12, C=16),
        pin_transition_form, pin_invariants, pin_conv, pin_l2norm, pin_deltalog_equals_dense,
        pin_batch_glue, pin_prenorm_log, pin_verify_routing, pin_kda_gate, pin_out_norm_gate,
        pin_kda_batch_glue, pin_prefill_batch, pin_verify_conv_window, pin_verify_conv_glue,
        pin_prefill_conv_glue, pin_prefill_kda_glue]


# ----------------------------------------------------------------------------
# tests
# ----------------------------------------------------------------------------

def test_teaching_example_dense(oracle_lib):
    pin_teaching_dense(oracle_lib)


def test_teaching_example_deltalog(oracle_lib):
    pin_teaching_deltalog(oracle_lib)


@pytest.mark.parametrize("C", [16, 24, 64])
def test_gla_recurrent_equals_chunked(oracle_lib, C):
    pin_gla_chunked(oracle_lib, C=C)


@pytest.mark.parametrize("per_key", [False, True])
@pytest.mark.parametrize("shape", [(64, 16, 16, 16), (50, 8, 12, 16), (40, 12, 8, 7)])
def test_delta_rule_recurrent_equals_wy_chunked(oracle_lib, per_key, shape):
    T, dk, dv, C = shape
    pin_delta_wy(oracle_lib, T=T, dk=dk, dv=dv, C=C, per_key=per_key)


def test_transition_form(oracle_lib):
    pin_transition_form(oracle_lib)


def test_invariants(oracle_lib):
    pin_invariants(oracle_lib)


def test_spectral_norm_of_transition():
    """||I - beta k k^T||_2 <= 1 for unit k and 0 <= beta <= 1 (appendix 附2)."""
    r = _rng(8)
    for _ in range(100):
        k = _unit(r.standard_normal(16))
        beta = r.uniform(0, 1)
        assert np.linalg.norm(np.eye(16) - beta * np.outer(k, k), 2) <= 1 + 1e-12


def test_closure_identity():
    """D(lambda) D(ell) = D(ell + lambda) for diagonal decays (DeltaLog notes Sec. 2.2)."""
    r = _rng(9)
    lam, ell = -np.abs(r.standard_normal(128)), -np.abs(r.standard_normal(128)) * 5
    lhs = np.diag(np.exp(lam)) @ np.diag(np.exp(ell))
    rhs = np.diag(np.exp(ell + lam))
    assert np.max(np.abs(lhs - rhs) / np.maximum(np.abs(rhs), 1e-300)) <= 1e-14  # a few ulp plus argument rounding


def test_conv(oracle_lib):
    pin_conv(oracle_lib)


def test_l2norm(oracle_lib):
    pin_l2norm(oracle_lib)


def test_deltalog_equals_dense(oracle_lib):
    pin_deltalog_equals_dense(oracle_lib)


def test_batch_glue(oracle_lib):
    pin_batch_glue(oracle_lib)


def test_prenorm_log(oracle_lib):
    pin_prenorm_log(oracle_lib)


def test_verify_routing(oracle_lib):
    pin_verify_routing(oracle_lib)


def test_prefill_batch(oracle_lib):
    pin_prefill_batch(oracle_lib)


def test_verify_conv_window(oracle_lib):
    pin_verify_conv_window(oracle_lib)
    pin_verify_conv_window(oracle_lib, T=1, seed=18)


def test_verify_conv_glue(oracle_lib):
    pin_verify_conv_glue(oracle_lib)


def test_prefill_conv_glue(oracle_lib):
    pin_prefill_conv_glue(oracle_lib)


def test_prefill_kda_glue(oracle_lib):
    pin_prefill_kda_glue(oracle_lib)


def test_kda_gate(oracle_lib):
    pin_kda_gate(oracle_lib)


def test_out_norm_gate(oracle_lib):
    pin_out_norm_gate(oracle_lib)


def test_kda_batch_glue(oracle_lib):
    pin_kda_batch_glue(oracle_lib)


def test_batch_errors(oracle_lib):
    st = oracle.BatchState(2, 1, 4, 4, 1, 2)
    z = np.zeros((1, 1, 4))
    cfg = _batch_cfg(1, 1, 4, 4, 2, 1, 2, 0)
    with pytest.raises(ValueError, match="slot"):
        oracle.step_batch(cfg, "dense", st, np.array([2], np.int32), q=z, k=z, v=z,
                          lam=np.zeros((1, 1, 1)), beta=np.zeros((1, 1)), lib=oracle_lib)
    st.len[0, 0] = 3  # above C = 2
    with pytest.raises(ValueError, match="log length"):
        oracle.step_batch(cfg, "deltalog", st, np.array([0], np.int32), q=z, k=z, v=z,
                          lam=np.zeros((1, 1, 1)), beta=np.zeros((1, 1)), lib=oracle_lib)


# Each planted mistake: (description, exact source text, replacement).
MUTANTS = [
    ("correction read before the decay",
     "  for (int j = 0; j < dv; ++j) {\n    double vhat = 0.0;\n    for (int d = 0; d < dk; ++d) vhat += S[(size_t)d * dv + j] * k[d];",
     "  for (int j = 0; j < dv; ++j) {\n    double vhat = 0.0;\n    for (int d = 0; d < dk; ++d) vhat += S[(size_t)d * dv + j] * k[d] / exp(lam[dlam == 1 ? 0 : d]);"),
    ("sign of the delta correction",
     "b[j] = plain ? beta * v[j] : beta * (v[j] - vhat);\n  }\n  for (int d = 0; d < dk; ++d)\n    for (int j = 0; j < dv; ++j) S[(size_t)d * dv + j] += k[d] * b[j];",
     "b[j] = plain ? beta * v[j] : beta * (v[j] + vhat);\n  }\n  for (int d = 0; d < dk; ++d)\n    for (int j = 0; j < dv; ++j) S[(size_t)d * dv + j] += k[d] * b[j];"),
    ("readout before the write",
     "    for (int d = 0; d < dk; ++d) acc += S[(size_t)d * dv + j] * q[d];\n    o[j] = acc;",
     "    for (int d = 0; d < dk; ++d) acc += (S[(size_t)d * dv + j] - k[d] * b[j]) * q[d];\n    o[j] = acc;"),
    ("decay on value columns instead of key rows",
     "    double a = exp(lam[dlam == 1 ? 0 : d]);\n    for (int j = 0; j < dv; ++j) S[(size_t)d * dv + j] *= a;",
     "    for (int j = 0; j < dv; ++j) S[(size_t)d * dv + j] *= exp(lam[dlam == 1 ? 0 : (j % dlam)]);"),
    ("conv taps reversed",
     "acc += cs[c * 3 + j] * w[c * CONV_K + j];",
     "acc += cs[c * 3 + j] * w[c * CONV_K + 2 - j];"),
    ("conv state not shifted",
     "    cs[c * 3 + 0] = cs[c * 3 + 1];\n",
     ""),
    ("L2 norm without the square root",
     "double inv = 1.0 / sqrt(ss + eps);",
     "double inv = 1.0 / (ss + eps);"),
    ("log entry weight sign flipped",
     "acc += exp(ed - lamid) * Klog",
     "acc += exp(lamid - ed) * Klog"),
    ("append stores the old cumulative decay",
     "for (int e = 0; e < dlam; ++e) Lam[(size_t)n * dlam + e] = ellp[e];",
     "for (int e = 0; e < dlam; ++e) Lam[(size_t)n * dlam + e] = ell[e];"),
    ("merge drops the current update",
     "Sbar[(size_t)d * dv + j] = P[(size_t)d * dv + j] + k[d] * b[j];",
     "Sbar[(size_t)d * dv + j] = P[(size_t)d * dv + j];"),
    ("merge keeps the cumulative decay",
     "    for (int e = 0; e < dlam; ++e) ell[e] = 0.0;\n",
     ""),
    ("append decision off by one",
     "  if (n < C) {\n    for (int d = 0; d < dk; ++d) Klog",
     "  if (n + 1 < C) {\n    for (int d = 0; d < dk; ++d) Klog"),
    ("k head offset uses the q block",
     "kr = yb + (size_t)H * dk + (size_t)h * dk;",
     "kr = yb + (size_t)h * dk;"),
    ("q scale dropped",
     "orc_l2norm(dk, qr, cfg->l2_eps, cfg->q_scale, qh);",
     "orc_l2norm(dk, qr, cfg->l2_eps, 1.0, qh);"),
    ("raw decay gate uses sigmoid instead of logsigmoid",
     "lh[e] = orc_log_sigmoid(lr[e]);",
     "lh[e] = orc_sigmoid(lr[e]);"),
    ("KDA gate: A_log not exponentiated",
     "const double z = exp(a_log) * x;",
     "const double z = a_log * x;"),
    ("KDA gate: dt_bias subtracted",
     "const double x = f + dt_bias;",
     "const double x = f - dt_bias;"),
    ("output RMSNorm over the sum instead of the mean",
     "const double inv = 1.0 / sqrt(ss / dv + eps);",
     "const double inv = 1.0 / sqrt(ss + eps);"),
    ("output gate sign flipped",
     "y[j] = o[j] * inv * (w ? w[j] : 1.0) * orc_sigmoid(g[j]);",
     "y[j] = o[j] * inv * (w ? w[j] : 1.0) * orc_sigmoid(-g[j]);"),
    ("verify conv window read from column 0",
     "const int off = na - 1;",
     "const int off = 0;"),
    ("verify conv window keeps the oldest inputs",
     "+ (T + CONV_K - 1 - W) + i];",
     "+ i];"),
    ("verify conv window not rewritten",
     "for (int i = 0; i < W; ++i) win[",
     "for (int i = 0; i < W && 0; ++i) win["),
    ("epilogue not applied in the batch step",
     "      if (fl & ORC_OUT_NORM_GATE)\n        orc_out_norm_gate(",
     "      if (0)\n        orc_out_norm_gate("),
]


@pytest.mark.parametrize("desc,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(desc, old, new):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")).read()
    assert src.count(old) == 1, f"mutation anchor not found exactly once: {desc}"
    tmp = tempfile.mkdtemp(prefix="orc_mut_")
    try:
        mpath = os.path.join(tmp, "gdn_oracle_mut.c")
        with open(mpath, "w") as f:
            f.write(src.replace(old, new))
        lib = oracle.load(oracle.build(force=True, src=mpath, out_path=os.path.join(tmp, "libmut.so")))
        failures = []
        for pin in PINS:
            try:
                pin(lib)
            except (AssertionError, ValueError):
                failures.append(getattr(pin, "__name__", "pin"))
        assert failures, f"no pin caught the planted mistake: {desc}"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
