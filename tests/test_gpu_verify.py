"""GPU parity of the speculative-decoding verify path (gdn_decode_verify) against the fp64
oracle: T positions per request through the dense step, the state after every position in
its own pool row, the initial state taken from the column the acceptance count selects
(inference handbook, "推测解码：验证后如何恢复状态")."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import linear_attention_decode_gdn_gb300 as gdn  # noqa: E402
from linear_attention_decode_gdn_gb300 import workloads as wl  # noqa: E402

from gpu_harness import dev_bf16, dev_f32, dev_i32  # noqa: E402

pytestmark = pytest.mark.gpu

TOL = 1e-4  # the dense bar: the verify path is the dense recurrence


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_attention_decode_gdn_gb300 import build
    build.build()


class Round:
    """One verify call's seeded inputs ([B, T, H, ...]) in both precisions."""

    def __init__(self, B, T, H, D, per_key, bf16, seed, gate_raw=False, raw_value=False, kda=None):
        r = np.random.default_rng(seed)
        dlam = D if per_key else 1
        qkm = D ** -0.5 if raw_value else 1.0
        q = r.standard_normal((B, T, H, D), dtype=np.float32) * np.float32(qkm)
        k = r.standard_normal((B, T, H, D), dtype=np.float32) * np.float32(qkm)
        v = r.standard_normal((B, T, H, D), dtype=np.float32)
        self.bits = {}
        if bf16:
            for n, a in (("q", q), ("k", k), ("v", v)):
                self.bits[n], vals = wl.bf16_round(a)
                a[...] = vals
        a_raw = r.standard_normal((B, T, H, dlam), dtype=np.float32) + np.float32(3)
        b_raw = r.standard_normal((B, T, H), dtype=np.float32)
        self.lam = (-np.log1p(np.exp(-a_raw.astype(np.float64)))).astype(np.float32)
        self.beta = (1 / (1 + np.exp(-b_raw.astype(np.float64)))).astype(np.float32)
        if raw_value:
            self.beta[...] = 1
        self.gate_in = (a_raw, b_raw) if gate_raw else (self.lam, self.beta)
        self.kda = kda
        if kda is not None:  # the KDA gate takes the forget pre-activation and the write logit
            self.gate_in = (a_raw - np.float32(3), b_raw)
            self.out_gate = r.standard_normal((B, T, H, D), dtype=np.float32)
        self.q, self.k, self.v = q, k, v
        self.bf16, self.raw_value = bf16, raw_value

    def device_inputs(self):
        d = {}
        for n in ("q", "k", "v"):
            a = getattr(self, n)
            d[n] = dev_bf16(self.bits[n].reshape(a.shape)) if self.bf16 else dev_f32(a)
        d["log_decay"] = dev_f32(self.gate_in[0])
        d["beta"] = None if self.raw_value else dev_f32(self.gate_in[1])
        if self.kda is not None:
            d.update({n: dev_f32(self.kda[n]) for n in ("a_log", "dt_bias", "out_norm_w")},
                     out_gate=dev_f32(self.out_gate))
        return d

    def oracle_inputs(self):
        f = lambda a: np.ascontiguousarray(a, dtype=np.float64)  # noqa: E731
        d = dict(q=f(self.q), k=f(self.k), v=f(self.v), lam=f(self.gate_in[0]), beta=f(self.gate_in[1]))
        if self.kda is not None:
            d.update(a_log=f(self.kda["a_log"]), dt_bias=f(self.kda["dt_bias"]),
                     out_norm_w=f(self.kda["out_norm_w"]), out_gate=f(self.out_gate),
                     lower_bound=self.kda["lower_bound"])
        return d


def _flags(bf16, gate_raw, raw_value, kda=False):
    f = (gdn.QKV_BF16 if bf16 else 0) | (gdn.GATE_RAW if gate_raw else 0)
    if raw_value:
        f |= gdn.PLAIN_UPDATE | gdn.NO_QK_L2NORM
    if kda:
        f |= gdn.GATE_KDA | gdn.OUT_NORM_GATE
    return f


def _oracle_flags(gate_raw, raw_value, kda=False):
    f = oracle.GATE_RAW if gate_raw else 0
    if kda:
        f |= oracle.GATE_KDA | oracle.OUT_NORM_GATE
    return f | (oracle.PLAIN if raw_value else oracle.L2NORM)


def _rows(B, T, S, seed, pad=()):
    r = np.random.default_rng(seed)
    perm = r.permutation(S)[: B * T].reshape(B, T).astype(np.int32)
    for b in pad:
        perm[b, 0] = -1
    return perm


def _run(D, per_key, T, bf16=True, gate_raw=False, raw_value=False, B=6, H=3, seed=0, pad=(1,),
         na=None, rounds=1, kda=False):
    S = B * T + 5
    dlam = D if per_key else 1
    r = np.random.default_rng(seed + 99)
    pool0 = (r.standard_normal((S, H, D, D)) * 0.1).astype(np.float32)
    pool_dev = dev_f32(pool0)
    pool_ref = pool0.astype(np.float64)
    dims = gdn.make_dims(B, H, D, num_slots=S, decay_per_key=per_key,
                         flags=_flags(bf16, gate_raw, raw_value, kda), q_scale=D ** -0.5)
    cfg = dict(batch=B, num_heads=H, dk=D, dv=D, num_slots=S, dlam=dlam, log_capacity=0,
               flags=_oracle_flags(gate_raw, raw_value, kda), q_scale=D ** -0.5, l2_eps=1e-6)
    params = None
    if kda:
        w = wl.Workload("verify_kda", B, H, D, D, 1, (1,), bf16, False, per_key, seed + 5, kda_full=True)
        params = wl.kda_gate_params(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rng = np.random.default_rng(seed + 7)
    idx = _rows(B, T, S, seed, pad)
    err, ref = 0.0, 0.0
    for rd in range(rounds):
        acc = (np.asarray(na, dtype=np.int32) if na is not None and rd == 0
               else rng.integers(1, T + 1, size=B).astype(np.int32))
        x = Round(B, T, H, D, per_key, bf16, seed + 1000 * rd, gate_raw, raw_value, params)
        o = torch.full((B, T, H, D), 7.0, dtype=torch.float32, device="cuda")
        keep = x.device_inputs()
        gdn.decode_verify(dims, T, gdn.make_inputs(**keep), dev_i32(idx), dev_i32(acc), pool_dev, o, status)
        o_ref = oracle.verify_batch(cfg, pool_ref, idx, acc, **x.oracle_inputs())
        torch.cuda.synchronize()
        live = idx[:, 0] >= 0
        og = o.cpu().numpy().astype(np.float64)
        err = max(err, float(np.max(np.abs(og[live] - o_ref[live]))))
        ref = max(ref, float(np.max(np.abs(o_ref[live]))))
        assert np.all(og[~live] == 7.0)  # padding rows of o untouched
        # the next round starts from the rows this round wrote (the rollback chain)
        idx = np.roll(idx, 1, axis=1) if rd % 2 == 0 else idx
    assert int(status.item()) == 0
    pg = pool_dev.cpu().numpy().astype(np.float64)
    serr = float(np.max(np.abs(pg - pool_ref)))
    sref = float(np.max(np.abs(pool_ref)))
    return err / ref, serr / sref, pg, pool_ref


@pytest.mark.parametrize("D", [16, 64, 128])
@pytest.mark.parametrize("per_key", [False, True])
@pytest.mark.parametrize("T", [1, 3, 4])
def test_verify_matches_oracle(D, per_key, T):
    e_o, e_s, _, _ = _run(D, per_key, T, seed=D + 10 * T + int(per_key))
    assert e_o <= TOL and e_s <= TOL, (e_o, e_s)


def test_verify_fp32_inputs_raw_gates():
    e_o, e_s, _, _ = _run(128, False, 4, bf16=False, gate_raw=True, seed=3)
    assert e_o <= TOL and e_s <= TOL, (e_o, e_s)


def test_verify_raw_value_update():
    """The RWKV6 form (beta NULL = 1, plain update, raw q/k) through the verify path."""
    e_o, e_s, _, _ = _run(128, True, 4, raw_value=True, seed=4)
    assert e_o <= TOL and e_s <= TOL, (e_o, e_s)


def test_verify_kda_gate_and_epilogue():
    """The KDA gate parametrisation and output epilogue through the verify path."""
    for per_key in (True, False):
        e_o, e_s, _, _ = _run(128, per_key, 4, kda=True, seed=8 + int(per_key))
        assert e_o <= TOL and e_s <= TOL, (per_key, e_o, e_s)


def test_verify_rollback_chain():
    """Three rounds: each starts from the row its acceptance count selects among the rows
    the previous round wrote (the initial row is also overwritten in the same call)."""
    e_o, e_s, _, _ = _run(128, False, 4, rounds=3, seed=5, pad=())
    assert e_o <= TOL and e_s <= TOL, (e_o, e_s)


def test_verify_all_accepted_and_first_column():
    """num_accepted = T (start from the last column) and = 1 (start from column 0)."""
    for na in (4, 1):
        e_o, e_s, _, _ = _run(64, False, 4, na=[na] * 6, seed=6 + na, pad=())
        assert e_o <= TOL and e_s <= TOL, (na, e_o, e_s)


def test_verify_one_position_is_the_dense_step():
    """T = 1 with num_accepted = 1 runs exactly the dense kernel's arithmetic."""
    B, H, D = 8, 4, 128
    x = Round(B, 1, H, D, False, True, 21)
    S = B
    r = np.random.default_rng(22)
    pool0 = (r.standard_normal((S, H, D, D)) * 0.1).astype(np.float32)
    dims = gdn.make_dims(B, H, D, num_slots=S, flags=gdn.QKV_BF16)
    pa, pb = dev_f32(pool0), dev_f32(pool0)
    oa = torch.zeros((B, H, D), device="cuda")
    ob = torch.zeros((B, 1, H, D), device="cuda")
    keep = x.device_inputs()
    slot = dev_i32(np.arange(B))
    gdn.decode_dense(dims, gdn.make_inputs(slot=slot, **keep), pa, oa)
    gdn.decode_verify(dims, 1, gdn.make_inputs(**keep), dev_i32(np.arange(B).reshape(B, 1)),
                      dev_i32(np.ones(B)), pb, ob)
    torch.cuda.synchronize()
    assert torch.equal(oa, ob[:, 0]) and torch.equal(pa, pb)


def test_verify_status_and_skips():
    B, H, D, T = 4, 2, 64, 3
    S = B * T
    dims = gdn.make_dims(B, H, D, num_slots=S, flags=gdn.QKV_BF16)
    x = Round(B, T, H, D, False, True, 31)
    pool0 = np.random.default_rng(32).standard_normal((S, H, D, D)).astype(np.float32)
    pool = dev_f32(pool0)
    idx = np.arange(S, dtype=np.int32).reshape(B, T)
    idx[1, 2] = S + 3          # row out of range: request 1 skipped, BAD_SLOT
    na = np.array([1, 1, 0, 2], dtype=np.int32)  # request 2: accepted count out of range, BAD_LEN
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = torch.full((B, T, H, D), 3.0, device="cuda")
    gdn.decode_verify(dims, T, gdn.make_inputs(**x.device_inputs()), dev_i32(idx), dev_i32(na), pool, o, status)
    torch.cuda.synchronize()
    assert int(status.item()) == gdn.STATUS_BAD_SLOT | gdn.STATUS_BAD_LEN
    pg = pool.cpu().numpy()
    for b in (1, 2):
        assert torch.all(o[b] == 3.0)
        for row in idx[b]:
            if 0 <= row < S:
                assert np.array_equal(pg[row], pool0[row])
    for b in (0, 3):
        assert not torch.all(o[b] == 3.0)


def _run_conv(D, T, bf16=True, bias=True, B=5, H=2, rounds=3, seed=40, pad=(2,)):
    """Verify with the fused conv through the widened conv window: ``rounds`` calls in a row,
    each entering with the previous round's acceptance counts (column 0 of every request
    keeps its window row). Returns the output / state relative errors and whether every
    window matches the oracle's bit for bit."""
    r = np.random.default_rng(seed)
    nch = 3 * H * D
    S = B * T + 3
    pool0 = (r.standard_normal((S, H, D, D)) * 0.1).astype(np.float32)
    win0 = r.standard_normal((S, nch, T + 2)).astype(np.float32)
    w = (r.standard_normal((nch, 4)) * 0.5).astype(np.float32)
    cb = (r.standard_normal(nch) * 0.1).astype(np.float32) if bias else None
    if bf16:
        win_bits, win0 = wl.bf16_round(win0)
        win_dev = dev_bf16(win_bits)
    else:
        win_dev = dev_f32(win0)
    pool_dev, pool_ref, win_ref = dev_f32(pool0), pool0.astype(np.float64), win0.astype(np.float64)
    flags = (gdn.QKV_BF16 if bf16 else 0) | gdn.FUSE_CONV
    dims = gdn.make_dims(B, H, D, num_slots=S, flags=flags, q_scale=D ** -0.5)
    cfg = dict(batch=B, num_heads=H, dk=D, dv=D, num_slots=S, dlam=1, log_capacity=0,
               flags=oracle.L2NORM, q_scale=D ** -0.5, l2_eps=1e-6)
    idx = _rows(B, T, S, seed, pad)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    err = ref = 0.0
    na = np.ones(B, dtype=np.int32)
    for rd in range(rounds):
        mixed = r.standard_normal((B, T, nch)).astype(np.float32)
        if bf16:
            mbits, mixed = wl.bf16_round(mixed)
            mixed_dev = dev_bf16(mbits.reshape(mixed.shape))
        else:
            mixed_dev = dev_f32(mixed)
        a_raw = r.standard_normal((B, T, H, 1)).astype(np.float32) + np.float32(3)
        lam = (-np.log1p(np.exp(-a_raw.astype(np.float64)))).astype(np.float32)
        beta = (1 / (1 + np.exp(-r.standard_normal((B, T, H)).astype(np.float64)))).astype(np.float32)
        o = torch.full((B, T, H, D), 7.0, dtype=torch.float32, device="cuda")
        keep = dict(mixed_qkv=mixed_dev, conv_w=dev_f32(w), conv_b=None if cb is None else dev_f32(cb),
                    conv_pool=win_dev, log_decay=dev_f32(lam), beta=dev_f32(beta))
        gdn.decode_verify(dims, T, gdn.make_inputs(**keep), dev_i32(idx), dev_i32(na), pool_dev, o, status)
        f = lambda a: np.ascontiguousarray(a, dtype=np.float64)  # noqa: E731
        o_ref = oracle.verify_batch(cfg, pool_ref, idx, na, lam=f(lam), beta=f(beta), mixed=f(mixed),
                                    conv_w=f(w), conv_b=None if cb is None else f(cb), conv_window=win_ref)
        torch.cuda.synchronize()
        live = idx[:, 0] >= 0
        og = o.cpu().numpy().astype(np.float64)
        err = max(err, float(np.max(np.abs(og[live] - o_ref[live]))))
        ref = max(ref, float(np.max(np.abs(o_ref[live]))))
        assert np.all(og[~live] == 7.0)
        na = r.integers(1, T + 1, size=B).astype(np.int32)
    assert int(status.item()) == 0
    if bf16:
        wg = (win_dev.cpu().view(torch.int16).numpy().astype(np.uint16).astype(np.uint32) << 16).view(np.float32)
    else:
        wg = win_dev.cpu().numpy()
    win_ok = np.array_equal(wg.astype(np.float64), win_ref)
    pg = pool_dev.cpu().numpy().astype(np.float64)
    serr = float(np.max(np.abs(pg - pool_ref))) / float(np.max(np.abs(pool_ref)))
    return err / ref, serr, win_ok


@pytest.mark.parametrize("D,T", [(128, 4), (64, 3), (16, 1), (32, 16)])
def test_verify_conv_window(D, T):
    """Fused conv through the widened window (inference handbook, speculative-decoding
    state recovery): outputs and states at the dense bar, windows bit-exact."""
    e_o, e_s, win_ok = _run_conv(D, T, seed=40 + D + T)
    assert e_o <= TOL and e_s <= TOL and win_ok, (e_o, e_s, win_ok)


def test_verify_conv_window_fp32_no_bias():
    e_o, e_s, win_ok = _run_conv(128, 4, bf16=False, bias=False, seed=77)
    assert e_o <= TOL and e_s <= TOL and win_ok, (e_o, e_s, win_ok)
