"""fp64 CPU oracle for the batched Gated-DeltaNet decode step.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg import this package. The CUDA product
path never imports, links or calls it, and this package never touches the CUDA
library.

Contents:
  * ``gdn_oracle.c`` -- the recurrence in plain C, fp64, OpenMP over
    (request, head): short conv + SiLU, L2 normalisation, the dense gated
    delta-rule step and the DeltaLog base+log emulation. Built with gcc by
    :func:`build`, loaded with ctypes.
  * ``verify_batch`` -- speculative-decoding verify: T positions per request
    through the dense step, one pool row per position (composition of the
    pinned dense step with the row routing of the inference handbook); with
    a fused conv, the widened conv window (``orc_verify_conv_window``).
  * ``prefill_batch`` -- the prompt of every request through the dense step,
    token by token, masked past each prompt length.
  * ``chunked.py``   -- numpy fp64 chunkwise forms (gated linear attention
    with a decay mask; the WY/UT form of the gated delta rule) used only to
    pin the recurrence against an independent algorithm.

Parity: every function here is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_pins.py`` (worked example printed on the pages, closed
forms, invariants, an independent chunked algorithm, brute force on tiny
inputs).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libgdn_oracle.so")

# Flags understood by orc_step_batch (oracle-local values).
CONV = 1
L2NORM = 2
PLAIN = 4
GATE_RAW = 8
KLOG_PRENORM = 16
GATE_KDA = 32
OUT_NORM_GATE = 64

ERRORS = {0: "ok", 1: "bad argument", 2: "slot out of range", 3: "log length out of range"}


class OrcCfg(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("dk", ctypes.c_int32),
        ("dv", ctypes.c_int32),
        ("num_slots", ctypes.c_int32),
        ("dlam", ctypes.c_int32),
        ("log_capacity", ctypes.c_int32),
        ("flags", ctypes.c_uint32),
        ("q_scale", ctypes.c_double),
        ("l2_eps", ctypes.c_double),
    ]


_lock = threading.Lock()
_lib = None


class OrcKda(ctypes.Structure):
    _fields_ = [("a_log", ctypes.POINTER(ctypes.c_double)), ("dt_bias", ctypes.POINTER(ctypes.c_double)),
                ("out_gate", ctypes.POINTER(ctypes.c_double)), ("out_norm_w", ctypes.POINTER(ctypes.c_double)),
                ("lower_bound", ctypes.c_double), ("out_eps", ctypes.c_double)]


def build(force: bool = False, src: str | None = None, out_path: str | None = None) -> str:
    """Compile gdn_oracle.c with gcc (-O2 -fopenmp, no fast-math); returns the library path.

    ``src``/``out_path`` let a test compile a copy of the source with a planted
    mistake, to show that the pins catch it.
    """
    src = src or _SRC
    path = out_path or _LIB_PATH
    if not force and os.path.exists(path) and os.path.getmtime(path) >= os.path.getmtime(src):
        return path
    os.makedirs(os.path.dirname(path), exist_ok=True)
    tmp = path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, path)
    return path


def _declare(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int32)
    lib.orc_num_threads.restype = ctypes.c_int
    lib.orc_conv1d_silu.argtypes = [ctypes.c_int, dp, dp, dp, dp, dp]
    lib.orc_conv1d_silu.restype = None
    lib.orc_l2norm.argtypes = [ctypes.c_int, dp, ctypes.c_double, ctypes.c_double, dp]
    lib.orc_l2norm.restype = ctypes.c_double
    lib.orc_gdn_step.argtypes = [ctypes.c_int, ctypes.c_int, dp, dp, dp, dp, dp, ctypes.c_int,
                                 ctypes.c_double, ctypes.c_int, dp]
    lib.orc_gdn_step.restype = None
    lib.orc_deltalog_step.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      dp, dp, dp, dp, dp, ip, dp, dp, dp, dp, ctypes.c_double,
                                      ctypes.c_int, dp, ctypes.c_double, dp]
    lib.orc_deltalog_step.restype = ctypes.c_int
    lib.orc_step_batch.argtypes = [ctypes.POINTER(OrcCfg), ctypes.c_int, ip] + [dp] * 3 + \
        [dp] * 4 + [dp, dp] + [dp] * 5 + [ip, dp]
    lib.orc_step_batch.restype = ctypes.c_int
    lib.orc_step_batch_ex.argtypes = [ctypes.POINTER(OrcCfg), ctypes.c_int, ip] + [dp] * 3 + \
        [dp] * 4 + [dp, dp] + [dp] * 5 + [ip, ctypes.POINTER(OrcKda), dp]
    lib.orc_step_batch_ex.restype = ctypes.c_int
    lib.orc_kda_log_decay.argtypes = [ctypes.c_double] * 4
    lib.orc_kda_log_decay.restype = ctypes.c_double
    lib.orc_out_norm_gate.argtypes = [ctypes.c_int, dp, dp, dp, ctypes.c_double, dp]
    lib.orc_out_norm_gate.restype = None
    lib.orc_verify_conv_window.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, dp, dp, dp, dp, dp]
    lib.orc_verify_conv_window.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
        return _lib


def _f64(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.dtype == np.float64 and a.flags.c_contiguous, \
        "oracle arrays must be C-contiguous float64"
    return a


def _ptr(a, ctype=ctypes.c_double):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def num_threads(lib=None) -> int:
    return (lib or load()).orc_num_threads()


def conv1d_silu(x, conv_state, w, bias=None, lib=None):
    """One token of the width-4 causal conv + SiLU; ``conv_state`` [nch,3] is updated."""
    lib = lib or load()
    x, conv_state, w, bias = map(_f64, (x, conv_state, w, bias))
    y = np.empty_like(x)
    lib.orc_conv1d_silu(x.size, _ptr(x), _ptr(conv_state), _ptr(w), _ptr(bias), _ptr(y))
    return y


def l2norm(x, eps, scale=1.0, lib=None):
    lib = lib or load()
    x = _f64(np.ascontiguousarray(x, dtype=np.float64))
    y = np.empty_like(x)
    inv = lib.orc_l2norm(x.size, _ptr(x), float(eps), float(scale), _ptr(y))
    return y, inv


def gdn_step(S, q, k, v, lam, beta, plain=False, lib=None):
    """One dense step on a single head; ``S`` [dk,dv] float64 is updated, returns o [dv]."""
    lib = lib or load()
    S, q, k, v, lam = map(_f64, (S, q, k, v, np.ascontiguousarray(lam, dtype=np.float64)))
    dk, dv = S.shape
    o = np.empty(dv)
    lib.orc_gdn_step(dk, dv, _ptr(S), _ptr(q), _ptr(k), _ptr(v), _ptr(lam), lam.size,
                     float(beta), int(plain), _ptr(o))
    return o


class HeadLog:
    """DeltaLog physical state of one head (fp64): base, ell, K/U/Lambda logs, length."""

    def __init__(self, dk, dv, C, dlam, base=None):
        self.base = np.zeros((dk, dv)) if base is None else np.array(base, dtype=np.float64)
        self.ell = np.zeros(dlam)
        self.klog = np.zeros((max(C, 1), dk))
        self.ulog = np.zeros((max(C, 1), dv))
        self.lam = np.zeros((max(C, 1), dlam))
        self.length = np.zeros(1, dtype=np.int32)
        self.C, self.dlam = C, dlam

    def logical_state(self):
        """Eq. (7) of the DeltaLog notes, written out."""
        e = self.ell if self.dlam > 1 else np.full(self.base.shape[0], self.ell[0])
        S = np.exp(e)[:, None] * self.base
        for i in range(int(self.length[0])):
            li = self.lam[i] if self.dlam > 1 else np.full(self.base.shape[0], self.lam[i, 0])
            S = S + (np.exp(e - li) * self.klog[i])[:, None] * self.ulog[i][None, :]
        return S


def deltalog_step(st: HeadLog, q, k, v, lam, beta, plain=False, a=None, bscale=1.0, lib=None):
    """One DeltaLog step (append if L < C on entry, else merge) on a single head."""
    lib = lib or load()
    q, k, v = map(_f64, (q, k, v))
    lam = _f64(np.ascontiguousarray(lam, dtype=np.float64))
    a = k if a is None else _f64(a)
    dk, dv = st.base.shape
    o = np.empty(dv)
    rc = lib.orc_deltalog_step(dk, dv, st.dlam, st.C, _ptr(st.base), _ptr(st.ell), _ptr(st.klog),
                               _ptr(st.ulog), _ptr(st.lam), _ptr(st.length, ctypes.c_int32),
                               _ptr(q), _ptr(k), _ptr(v), _ptr(lam), float(beta), int(plain),
                               _ptr(a), float(bscale), _ptr(o))
    if rc != 0:
        raise ValueError(f"oracle deltalog_step: {ERRORS.get(rc, rc)}")
    return o


class BatchState:
    """Slot-indexed pools (fp64) mirroring the GPU layout, for whole-batch steps."""

    def __init__(self, num_slots, H, dk, dv, dlam=1, C=0, nch=None):
        self.S = np.zeros((num_slots, H, dk, dv))
        self.ell = np.zeros((num_slots, H, dlam))
        c = max(C, 1)
        self.klog = np.zeros((num_slots, H, c, dk))
        self.ulog = np.zeros((num_slots, H, c, dv))
        self.lamlog = np.zeros((num_slots, H, c, dlam))
        self.len = np.zeros((num_slots, H), dtype=np.int32)
        nch = nch if nch is not None else 2 * H * dk + H * dv
        self.conv = np.zeros((num_slots, nch, 3))


def kda_log_decay(f, a_log, dt_bias, lower_bound, lib=None) -> float:
    """KDA forget-gate parametrisation for one channel (see gdn_oracle.c)."""
    lib = lib or load()
    return lib.orc_kda_log_decay(float(f), float(a_log), float(dt_bias), float(lower_bound))


def out_norm_gate(o, g, w=None, eps=1e-6, lib=None):
    """KDA output epilogue for one head: RMSNorm over dv, weight w, output gate sigmoid(g)."""
    lib = lib or load()
    o, g = (_f64(np.ascontiguousarray(a, dtype=np.float64)) for a in (o, g))
    w = None if w is None else _f64(np.ascontiguousarray(w, dtype=np.float64))
    y = np.empty_like(o)
    lib.orc_out_norm_gate(o.size, _ptr(o), _ptr(g), _ptr(w), float(eps), _ptr(y))
    return y


def step_batch(cfg: dict, mode: str, st: BatchState, slot, *, q=None, k=None, v=None,
               mixed=None, conv_w=None, conv_b=None, lam=None, beta=None, o=None, lib=None,
               a_log=None, dt_bias=None, out_gate=None, out_norm_w=None, lower_bound=-5.0,
               out_eps=1e-6):
    """One decode step for a whole batch. ``mode`` is 'dense' or 'deltalog'.

    ``cfg`` keys: batch, num_heads, dk, dv, num_slots, dlam, log_capacity, flags,
    q_scale, l2_eps. Inputs are float64 arrays in the layouts documented in
    gdn_oracle.c; returns o [B,H,dv] (rows of padding requests stay as given).
    """
    lib = lib or load()
    c = OrcCfg(cfg["batch"], cfg["num_heads"], cfg["dk"], cfg["dv"], cfg["num_slots"],
               cfg.get("dlam", 1), cfg.get("log_capacity", 0), cfg.get("flags", 0),
               cfg.get("q_scale", 1.0), cfg.get("l2_eps", 1e-6))
    slot = np.ascontiguousarray(slot, dtype=np.int32)
    if o is None:
        o = np.zeros((c.batch, c.num_heads, c.dv))
    q, k, v, mixed, conv_w, conv_b, lam, beta = map(
        lambda a: None if a is None else _f64(np.ascontiguousarray(a, dtype=np.float64)),
        (q, k, v, mixed, conv_w, conv_b, lam, beta))
    a_log, dt_bias, out_gate, out_norm_w = map(
        lambda a: None if a is None else _f64(np.ascontiguousarray(a, dtype=np.float64)),
        (a_log, dt_bias, out_gate, out_norm_w))
    kda = OrcKda(_ptr(a_log), _ptr(dt_bias), _ptr(out_gate), _ptr(out_norm_w), float(lower_bound),
                 float(out_eps))
    rc = lib.orc_step_batch_ex(ctypes.byref(c), {"dense": 0, "deltalog": 1}[mode],
                               _ptr(slot, ctypes.c_int32), _ptr(q), _ptr(k), _ptr(v), _ptr(mixed),
                               _ptr(conv_w), _ptr(conv_b), _ptr(st.conv), _ptr(lam), _ptr(beta),
                               _ptr(st.S), _ptr(st.ell), _ptr(st.klog), _ptr(st.ulog),
                               _ptr(st.lamlog), _ptr(st.len, ctypes.c_int32), ctypes.byref(kda), _ptr(o))
    if rc != 0:
        raise ValueError(f"oracle step_batch: {ERRORS.get(rc, rc)}")
    return o


def verify_conv_window(win, num_accepted, x, w, bias=None, lib=None):
    """One request's widened conv window through a verify round (inference handbook,
    "推测解码：验证后如何恢复状态"): ``win`` [nch, T+2] (the last T+2 pre-conv inputs,
    column 0 oldest) is read at offset num_accepted - 1 and updated in place; ``x``
    [T, nch] are the round's pre-conv inputs. Returns the SiLU(conv) outputs [T, nch]."""
    lib = lib or load()
    win, x, w, bias = map(_f64, (win, x, w, bias))
    T, nch = x.shape
    assert win.shape == (nch, T + 2)
    y = np.empty_like(x)
    rc = lib.orc_verify_conv_window(nch, T, int(num_accepted), _ptr(win), _ptr(x), _ptr(w), _ptr(bias), _ptr(y))
    if rc != 0:
        raise ValueError(f"oracle verify_conv_window: {ERRORS.get(rc, rc)}")
    return y


def verify_batch(cfg: dict, pool, state_indices, num_accepted, *, q=None, k=None, v=None, lam, beta,
                 lib=None, out_gate=None, mixed=None, conv_w=None, conv_b=None, conv_window=None, **kda):
    """Speculative-decoding verify, written from the inference handbook's passage
    "推测解码：验证后如何恢复状态": a request feeds T positions (the last sampled token,
    then the drafts) through the recurrence; the initial state is the pool row of column
    num_accepted - 1 of its index row, and the state after position t is kept in the row
    of column t. Every initial state is read before any row is written.

    ``pool`` [num_slots, H, dk, dv] float64 is updated in place; ``state_indices`` [B, T]
    (row 0 < 0: padding request, skipped), ``num_accepted`` [B] in [1, T]; q, k [B,T,H,dk],
    v [B,T,H,dv], lam [B,T,H,dlam], beta [B,T,H]. ``cfg`` as for :func:`step_batch`
    (flags L2NORM / PLAIN / GATE_RAW, q_scale, l2_eps). Each position is one dense step of
    :func:`step_batch`; the KDA gate / epilogue inputs (``out_gate`` [B,T,H,dv], and
    ``a_log``, ``dt_bias``, ``out_norm_w``, ``lower_bound``) pass through to it.
    With ``mixed`` [B, T, nch] (channels [q heads | k heads | v heads]), q, k and v are the
    outputs of :func:`verify_conv_window` on the request's window ``conv_window[row]``
    ([num_slots, nch, T+2], updated in place), row = the request's column-0 index.
    Returns o [B, T, H, dv]."""
    idx = np.asarray(state_indices, dtype=np.int64)
    na = np.asarray(num_accepted, dtype=np.int64)
    B, T = idx.shape
    H, dk, dv, dlam = cfg["num_heads"], cfg["dk"], cfg["dv"], cfg.get("dlam", 1)
    live = [b for b in range(B) if idx[b, 0] >= 0]
    if mixed is not None:
        q, k, v = np.zeros((B, T, H, dk)), np.zeros((B, T, H, dk)), np.zeros((B, T, H, dv))
        for b in live:
            y = verify_conv_window(conv_window[idx[b, 0]], na[b], np.ascontiguousarray(mixed[b]),
                                   conv_w, conv_b, lib=lib)
            q[b] = y[:, : H * dk].reshape(T, H, dk)
            k[b] = y[:, H * dk: 2 * H * dk].reshape(T, H, dk)
            v[b] = y[:, 2 * H * dk:].reshape(T, H, dv)
    run = BatchState(B, H, dk, dv, dlam)
    for b in live:
        run.S[b] = pool[idx[b, na[b] - 1]]
    slot = np.array([b if idx[b, 0] >= 0 else -1 for b in range(B)], dtype=np.int32)
    c = dict(cfg, batch=B, num_slots=B, log_capacity=0)
    o = np.zeros((B, T, H, dv))
    for t in range(T):
        o[:, t] = step_batch(c, "dense", run, slot, q=q[:, t], k=k[:, t], v=v[:, t],
                             lam=lam[:, t], beta=beta[:, t], lib=lib,
                             out_gate=None if out_gate is None else out_gate[:, t], **kda)
        for b in live:
            pool[idx[b, t]] = run.S[b]
    return o


def prefill_batch(cfg: dict, pool, slot, seq_lens, *, q=None, k=None, v=None, lam, beta, lib=None,
                  mixed=None, conv_w=None, conv_b=None, conv_pool=None, out_gate=None, **kda):
    """The prompt through the recurrence, token by token: position t of request b is one dense
    step of :func:`step_batch` on its pool row when t < seq_lens[b] (a prefill seeds the state
    a decode continues from; evolution article, "Prefill中的Chunk微观并行", states the same
    result for the chunked form). ``pool`` [num_slots, H, dk, dv] float64 is updated in place;
    q, k [B,T,H,dk], v [B,T,H,dv], lam [B,T,H,dlam], beta [B,T,H]. With ``mixed`` [B,T,nch]
    the step runs the causal conv + SiLU on it instead (flag CONV), through the slot's conv
    state ``conv_pool`` [num_slots, nch, 3] (updated in place: afterwards it holds the last
    three inputs of the prompt). The KDA gate / epilogue inputs (``out_gate`` [B,T,H,dv], and
    ``a_log``, ``dt_bias``, ``out_norm_w``, ``lower_bound``) pass through to each step.
    Returns o [B,T,H,dv] (zero past each prompt)."""
    slot = np.asarray(slot, dtype=np.int32)
    src = q if mixed is None else mixed
    B, T = src.shape[0], src.shape[1]
    H, dk, dv, dlam = cfg["num_heads"], cfg["dk"], cfg["dv"], cfg.get("dlam", 1)
    lens = np.full(B, T) if seq_lens is None else np.asarray(seq_lens)
    st = BatchState(cfg["num_slots"], H, dk, dv, dlam)
    st.S = pool  # the step updates the caller's pool in place
    c = dict(cfg, batch=B, log_capacity=0)
    if mixed is not None:
        st.conv = conv_pool
        c["flags"] = c.get("flags", 0) | CONV
    o = np.zeros((B, T, H, dv))
    for t in range(T):
        live = np.where((lens > t) & (slot >= 0), slot, -1).astype(np.int32)
        if mixed is None:
            tok = dict(q=q[:, t], k=k[:, t], v=v[:, t])
        else:
            tok = dict(mixed=mixed[:, t], conv_w=conv_w, conv_b=conv_b)
        o[:, t] = step_batch(c, "dense", st, live, lam=lam[:, t], beta=beta[:, t], lib=lib,
                             out_gate=None if out_gate is None else out_gate[:, t], **tok, **kda)
    return o
