"""GPU parity of the chunked prefill (gdn_prefill) against the fp64 oracle's token-by-token
prompt pass (which is pinned against the WY/UT chunked algebra): every position's readout,
the final state in the pool row, ragged prompt lengths, and a decode that continues from
the prefilled state."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import linear_attention_decode_gdn_gb300 as gdn  # noqa: E402
from linear_attention_decode_gdn_gb300 import workloads as wl  # noqa: E402

from gpu_harness import dev_bf16, dev_f32, dev_i32  # noqa: E402

pytestmark = pytest.mark.gpu

TOL = 1e-4  # the dense bar: per token the arithmetic is the dense step's


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_attention_decode_gdn_gb300 import build
    build.build()


def _inputs(B, T, H, D, dlam, bf16, seed, raw_value=False, gate_raw=False):
    r = np.random.default_rng(seed)
    m = np.float32(D ** -0.5 if raw_value else 1.0)
    x = {n: r.standard_normal((B, T, H, D), dtype=np.float32) * (m if n != "v" else np.float32(1))
         for n in ("q", "k", "v")}
    bits = {}
    if bf16:
        for n in x:
            bits[n], x[n] = wl.bf16_round(x[n])
    a_raw = r.standard_normal((B, T, H, dlam), dtype=np.float32) + np.float32(3)
    b_raw = r.standard_normal((B, T, H), dtype=np.float32)
    lam = (-np.log1p(np.exp(-a_raw.astype(np.float64)))).astype(np.float32)
    beta = np.ones_like(b_raw) if raw_value else (1 / (1 + np.exp(-b_raw.astype(np.float64)))).astype(np.float32)
    gin = (a_raw, b_raw) if gate_raw else (lam, beta)
    dev = {n: (dev_bf16(bits[n]) if bf16 else dev_f32(x[n])) for n in x}
    dev["log_decay"] = dev_f32(gin[0])
    dev["beta"] = None if raw_value else dev_f32(gin[1])
    ref = {n: x[n].astype(np.float64) for n in x}
    ref.update(lam=gin[0].astype(np.float64), beta=gin[1].astype(np.float64))
    return dev, ref


def _run(D, per_key, T, lens, bf16=True, raw_value=False, gate_raw=False, H=3, seed=0,
         slot=None, init_scale=0.1):
    B = len(lens)
    slot = np.arange(B, dtype=np.int32)[::-1].copy() if slot is None else np.asarray(slot, np.int32)
    S = int(max(slot.max(), 0)) + 2
    dlam = D if per_key else 1
    flags = (gdn.QKV_BF16 if bf16 else 0) | (gdn.GATE_RAW if gate_raw else 0)
    oflags = oracle.GATE_RAW if gate_raw else 0
    if raw_value:
        flags |= gdn.PLAIN_UPDATE | gdn.NO_QK_L2NORM
        oflags |= oracle.PLAIN
    else:
        oflags |= oracle.L2NORM
    r = np.random.default_rng(seed + 1)
    pool0 = (init_scale * r.standard_normal((S, H, D, D))).astype(np.float32)
    pool = dev_f32(pool0)
    pool_ref = pool0.astype(np.float64)
    dev, ref = _inputs(B, T, H, D, dlam, bf16, seed, raw_value, gate_raw)
    dims = gdn.make_dims(B, H, D, num_slots=S, decay_per_key=per_key, flags=flags, q_scale=D ** -0.5)
    cfg = dict(batch=B, num_heads=H, dk=D, dv=D, num_slots=S, dlam=dlam, log_capacity=0, flags=oflags,
               q_scale=D ** -0.5, l2_eps=1e-6)
    o = torch.full((B, T, H, D), 5.0, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.prefill(dims, T, gdn.make_inputs(slot=dev_i32(slot), **dev), pool, o, seq_lens=dev_i32(lens), status=status)
    o_ref = oracle.prefill_batch(cfg, pool_ref, slot, lens, **ref)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    og = o.cpu().numpy().astype(np.float64)
    err = ref_max = 0.0
    for b in range(B):
        n = lens[b] if slot[b] >= 0 else 0
        err = max(err, float(np.max(np.abs(og[b, :n] - o_ref[b, :n]), initial=0.0)))
        ref_max = max(ref_max, float(np.max(np.abs(o_ref[b, :n]), initial=0.0)))
        assert np.all(og[b, n:] == 5.0)  # positions past the prompt (and padding rows) untouched
    pg = pool.cpu().numpy().astype(np.float64)
    serr = float(np.max(np.abs(pg - pool_ref))) / float(np.max(np.abs(pool_ref)))
    return err / ref_max, serr, pg


@pytest.mark.parametrize("D", [16, 64, 128])
@pytest.mark.parametrize("per_key", [False, True])
def test_prefill_matches_oracle(D, per_key):
    # lengths across the chunk boundaries: 0, 1, 31, 32, 33, 70 (ragged, 3 chunks)
    e_o, e_s, _ = _run(D, per_key, 70, np.array([0, 1, 31, 32, 33, 70]), seed=D + int(per_key))
    assert e_o <= TOL and e_s <= TOL, (e_o, e_s)


def test_prefill_padding_fp32_raw_gates():
    e_o, e_s, _ = _run(128, False, 40, np.array([40, 17, 40, 5]), bf16=False, gate_raw=True,
                       slot=[2, -1, 0, 4], seed=3)
    assert e_o <= TOL and e_s <= TOL, (e_o, e_s)


def test_prefill_raw_value_update():
    """The RWKV6 form: per-key decay, b = v (beta NULL), raw q and k."""
    e_o, e_s, _ = _run(128, True, 64, np.array([64, 40, 3]), raw_value=True, seed=4)
    assert e_o <= TOL and e_s <= TOL, (e_o, e_s)


def test_prefill_per_key_bf16_raw_gates_padding():
    """Per-key decay from raw gates (logsigmoid per channel in the decay scan, sigmoid write
    strength) with bf16 inputs -- the tensor-core kernel for a per-key decay -- across padded
    and permuted slots and a ragged tail chunk."""
    e_o, e_s, _ = _run(128, True, 80, np.array([80, 17, 80, 5]), gate_raw=True, slot=[2, -1, 0, 4], seed=7)
    assert e_o <= TOL and e_s <= TOL, (e_o, e_s)


def test_prefill_long_prompt_per_key_from_zero():
    """A fresh request over a long prompt of many chunks with a per-key decay."""
    e_o, e_s, _ = _run(128, True, 300, np.array([300, 257]), H=4, seed=8, init_scale=0.0)
    assert e_o <= TOL and e_s <= TOL, (e_o, e_s)


def test_prefill_long_prompt_from_zero():
    """A fresh request (zero state) over a long prompt of many chunks."""
    e_o, e_s, _ = _run(128, False, 300, np.array([300, 257]), H=4, seed=5, init_scale=0.0)
    assert e_o <= TOL and e_s <= TOL, (e_o, e_s)


def test_prefill_then_decode():
    """Prefill seeds the state; a dense decode and a DeltaLog cycle continue from it, and
    both match the oracle's token-by-token pass over prompt + generated tokens."""
    w = wl.WORKLOADS["headline"]
    B, H, D, T, M = 8, 4, 128, 45, 4
    lens = np.full(B, T)
    slot = np.arange(B, dtype=np.int32)
    dev, ref = _inputs(B, T, H, D, 1, True, 11)
    cfg = dict(batch=B, num_heads=H, dk=D, dv=D, num_slots=B, dlam=1, log_capacity=0,
               flags=oracle.L2NORM, q_scale=1.0, l2_eps=1e-6)
    pool_ref = np.zeros((B, H, D, D))
    oracle.prefill_batch(cfg, pool_ref, slot, lens, **ref)
    st = oracle.BatchState(B, H, D, D)
    st.S = pool_ref
    dims_d = gdn.make_dims(B, H, D, num_slots=B, flags=gdn.QKV_BF16)
    dims_l = gdn.make_dims(B, H, D, num_slots=B, flags=gdn.QKV_BF16, log_capacity=M - 1)
    pd = gdn.Pools.allocate(dims_d)
    pl = gdn.Pools.allocate(dims_l, deltalog=True)
    o_pf = torch.zeros((B, T, H, D), device="cuda")
    slot_dev = dev_i32(slot)
    for pools in (pd, pl):
        gdn.prefill(dims_d, T, gdn.make_inputs(slot=slot_dev, **dev), pools.state, o_pf)
    gdn.slot_reset(dims_l, slot_dev, B, pl.log())  # a prefilled base starts with an empty log
    o_d = torch.zeros((B, H, D), device="cuda")
    o_l = torch.zeros((B, H, D), device="cuda")
    err_d = err_l = ref_max = 0.0
    for t in range(2 * M):
        x = wl.step_inputs(w, 500 + t, batch=B)
        d = dict(slot=slot_dev, log_decay=dev_f32(x["lam"]), beta=dev_f32(x["beta"]),
                 **{n: dev_bf16(x[n + "_bits"]) for n in ("q", "k", "v")})
        gdn.decode_dense(dims_d, gdn.make_inputs(**d), pd.state, o_d)
        call = gdn.decode_merge if (t + 1) % M == 0 else gdn.decode_append
        call(dims_l, gdn.make_inputs(**d), pl.state, pl.log(), o_l)
        o_ref = oracle.step_batch(cfg, "dense", st, slot, q=x["q"].astype(np.float64), k=x["k"].astype(np.float64),
                                  v=x["v"].astype(np.float64), lam=x["lam"].astype(np.float64),
                                  beta=x["beta"].astype(np.float64))
        torch.cuda.synchronize()
        err_d = max(err_d, float(np.max(np.abs(o_d.cpu().numpy() - o_ref))))
        err_l = max(err_l, float(np.max(np.abs(o_l.cpu().numpy() - o_ref))))
        ref_max = max(ref_max, float(np.max(np.abs(o_ref))))
    assert err_d / ref_max <= TOL, err_d / ref_max
    assert err_l / ref_max <= 5e-3, err_l / ref_max


def test_prefill_status_and_skips():
    B, H, D, T = 3, 2, 64, 10
    dims = gdn.make_dims(B, H, D, num_slots=4, flags=gdn.QKV_BF16)
    dev, _ = _inputs(B, T, H, D, 1, True, 21)
    pool0 = np.random.default_rng(22).standard_normal((4, H, D, D)).astype(np.float32)
    pool = dev_f32(pool0)
    o = torch.full((B, T, H, D), 9.0, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.prefill(dims, T, gdn.make_inputs(slot=dev_i32([0, 7, 2]), **dev), pool, o,
                seq_lens=dev_i32([10, 10, 11]), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == gdn.STATUS_BAD_SLOT | gdn.STATUS_BAD_LEN
    pg = pool.cpu().numpy()
    assert np.array_equal(pg[2], pool0[2]) and np.array_equal(pg[1], pool0[1]) and np.array_equal(pg[3], pool0[3])
    assert not np.array_equal(pg[0], pool0[0])
    assert torch.all(o[1] == 9.0) and torch.all(o[2] == 9.0)


def test_back_to_back_launches_match_oracle():
    """A prefill and 12 decode steps (dense and DeltaLog M=4) queued back to back with no
    host synchronisation between them, each step writing its own output row: every launch
    may start while the previous grid drains (programmatic launch), and the results must
    still equal the oracle's sequential pass."""
    w = wl.WORKLOADS["headline"]
    B, H, D, T, M, steps = 16, 8, 128, 40, 4, 12
    slot = np.arange(B, dtype=np.int32)
    slot_dev = dev_i32(slot)
    dev, ref = _inputs(B, T, H, D, 1, True, 31)
    cfg = dict(batch=B, num_heads=H, dk=D, dv=D, num_slots=B, dlam=1, log_capacity=0,
               flags=oracle.L2NORM, q_scale=1.0, l2_eps=1e-6)
    pool_ref = np.zeros((B, H, D, D))
    o_pf_ref = oracle.prefill_batch(cfg, pool_ref, slot, None, **ref)
    st = oracle.BatchState(B, H, D, D)
    st.S = pool_ref
    xs = [wl.step_inputs(w, 700 + t, batch=B) for t in range(steps)]
    ins = [dict(slot=slot_dev, log_decay=dev_f32(x["lam"]), beta=dev_f32(x["beta"]),
                **{n: dev_bf16(x[n + "_bits"]) for n in ("q", "k", "v")}) for x in xs]
    dims_d = gdn.make_dims(B, H, D, num_slots=B, flags=gdn.QKV_BF16)
    dims_l = gdn.make_dims(B, H, D, num_slots=B, flags=gdn.QKV_BF16, log_capacity=M - 1)
    pd, pl = gdn.Pools.allocate(dims_d), gdn.Pools.allocate(dims_l, deltalog=True)
    o_pf = torch.zeros((2, B, T, H, D), device="cuda")
    o_d = torch.zeros((steps, B, H, D), device="cuda")
    o_l = torch.zeros((steps, B, H, D), device="cuda")
    torch.cuda.synchronize()
    inputs = [gdn.make_inputs(**d) for d in ins]
    gdn.prefill(dims_d, T, gdn.make_inputs(slot=slot_dev, **dev), pd.state, o_pf[0])
    gdn.prefill(dims_d, T, gdn.make_inputs(slot=slot_dev, **dev), pl.state, o_pf[1])
    for t in range(steps):  # queued without synchronisation
        gdn.decode_dense(dims_d, inputs[t], pd.state, o_d[t])
        call = gdn.decode_merge if (t + 1) % M == 0 else gdn.decode_append
        call(dims_l, inputs[t], pl.state, pl.log(), o_l[t])
    torch.cuda.synchronize()
    ref_o = [oracle.step_batch(cfg, "dense", st, slot, q=x["q"].astype(np.float64), k=x["k"].astype(np.float64),
                               v=x["v"].astype(np.float64), lam=x["lam"].astype(np.float64),
                               beta=x["beta"].astype(np.float64)) for x in xs]
    ref_o = np.stack(ref_o)
    scale = float(np.max(np.abs(ref_o)))
    assert float(np.max(np.abs(o_d.cpu().numpy() - ref_o))) / scale <= TOL
    assert float(np.max(np.abs(o_l.cpu().numpy() - ref_o))) / scale <= 5e-3
    for i in range(2):
        assert float(np.max(np.abs(o_pf[i].cpu().numpy() - o_pf_ref))) / float(np.max(np.abs(o_pf_ref))) <= TOL
    S_ref = st.S
    assert float(np.max(np.abs(pd.state.cpu().numpy() - S_ref))) / float(np.max(np.abs(S_ref))) <= TOL
    assert float(np.max(np.abs(pl.state.cpu().numpy() - S_ref))) / float(np.max(np.abs(S_ref))) <= 5e-3


def _run_ext(D, per_key, T, lens, conv=False, kda=False, bias=True, H=2, seed=50, slot=None,
             bf16=True):
    """Prefill with the fused conv (q, k, v from mixed_qkv through the slot's conv state)
    and / or the KDA gate and output epilogue. Returns the output and state relative
    errors, whether the conv states match the oracle's bit for bit, and the pools."""
    B = len(lens)
    slot = np.arange(B, dtype=np.int32)[::-1].copy() if slot is None else np.asarray(slot, np.int32)
    S = int(max(slot.max(), 0)) + 2
    dlam = D if per_key else 1
    nch = 3 * H * D
    r = np.random.default_rng(seed)
    pool0 = (0.1 * r.standard_normal((S, H, D, D))).astype(np.float32)
    flags = (gdn.QKV_BF16 if bf16 else 0) | (gdn.FUSE_CONV if conv else 0)
    oflags = oracle.L2NORM
    dev, ref = {}, {}
    if conv:
        mixed = r.standard_normal((B, T, nch)).astype(np.float32)
        cs0 = r.standard_normal((S, nch, 3)).astype(np.float32)
        if bf16:
            mbits, mixed = wl.bf16_round(mixed)
            cbits, cs0 = wl.bf16_round(cs0)
            dev.update(mixed_qkv=dev_bf16(mbits), conv_pool=dev_bf16(cbits))
        else:
            dev.update(mixed_qkv=dev_f32(mixed), conv_pool=dev_f32(cs0))
        w = (0.5 * r.standard_normal((nch, 4))).astype(np.float32)
        cb = (0.1 * r.standard_normal(nch)).astype(np.float32) if bias else None
        dev.update(conv_w=dev_f32(w), conv_b=None if cb is None else dev_f32(cb))
        cs_ref = cs0.astype(np.float64)
        ref.update(mixed=mixed.astype(np.float64), conv_w=w.astype(np.float64),
                   conv_b=None if cb is None else cb.astype(np.float64), conv_pool=cs_ref)
    else:
        x = {n: r.standard_normal((B, T, H, D)).astype(np.float32) for n in ("q", "k", "v")}
        for n in x:
            bits, x[n] = wl.bf16_round(x[n])
            dev[n] = dev_bf16(bits)
            ref[n] = x[n].astype(np.float64)
    if kda:
        flags |= gdn.GATE_KDA | gdn.OUT_NORM_GATE
        oflags |= oracle.GATE_KDA | oracle.OUT_NORM_GATE
        wk = wl.Workload("prefill_kda", B, H, D, D, 1, (1,), True, False, per_key, seed + 3, kda_full=True)
        kp = wl.kda_gate_params(wk)
        f = (r.standard_normal((B, T, H, dlam)) - 3).astype(np.float32)
        logit = r.standard_normal((B, T, H)).astype(np.float32)
        g = r.standard_normal((B, T, H, D)).astype(np.float32)
        dev.update(log_decay=dev_f32(f), beta=dev_f32(logit), out_gate=dev_f32(g),
                   **{n: dev_f32(kp[n]) for n in ("a_log", "dt_bias", "out_norm_w")})
        ref.update(lam=f.astype(np.float64), beta=logit.astype(np.float64), out_gate=g.astype(np.float64),
                   a_log=kp["a_log"].astype(np.float64), dt_bias=kp["dt_bias"].astype(np.float64),
                   out_norm_w=kp["out_norm_w"].astype(np.float64), lower_bound=kp["lower_bound"])
    else:
        a_raw = r.standard_normal((B, T, H, dlam)) + 3
        lam = (-np.log1p(np.exp(-a_raw))).astype(np.float32)
        beta = (1 / (1 + np.exp(-r.standard_normal((B, T, H))))).astype(np.float32)
        dev.update(log_decay=dev_f32(lam), beta=dev_f32(beta))
        ref.update(lam=lam.astype(np.float64), beta=beta.astype(np.float64))
    dims = gdn.make_dims(B, H, D, num_slots=S, decay_per_key=per_key, flags=flags, q_scale=D ** -0.5)
    cfg = dict(batch=B, num_heads=H, dk=D, dv=D, num_slots=S, dlam=dlam, log_capacity=0, flags=oflags,
               q_scale=D ** -0.5, l2_eps=1e-6)
    pool, pool_ref = dev_f32(pool0), pool0.astype(np.float64)
    o = torch.full((B, T, H, D), 5.0, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.prefill(dims, T, gdn.make_inputs(slot=dev_i32(slot), **dev), pool, o, seq_lens=dev_i32(lens), status=status)
    o_ref = oracle.prefill_batch(cfg, pool_ref, slot, lens, **ref)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    og = o.cpu().numpy().astype(np.float64)
    err = ref_max = 0.0
    for b in range(B):
        n = lens[b] if slot[b] >= 0 else 0
        err = max(err, float(np.max(np.abs(og[b, :n] - o_ref[b, :n]), initial=0.0)))
        ref_max = max(ref_max, float(np.max(np.abs(o_ref[b, :n]), initial=0.0)))
        assert np.all(og[b, n:] == 5.0)
    pg = pool.cpu().numpy().astype(np.float64)
    serr = float(np.max(np.abs(pg - pool_ref))) / float(np.max(np.abs(pool_ref)))
    conv_ok = True
    if conv:
        cp = dev["conv_pool"].cpu()
        cg = ((cp.view(torch.int16).numpy().astype(np.uint16).astype(np.uint32) << 16).view(np.float32)
              if bf16 else cp.numpy())
        conv_ok = np.array_equal(cg.astype(np.float64), cs_ref)
    return err / ref_max, serr, conv_ok, (dims, pool, dev, cfg, pool_ref, ref)


@pytest.mark.parametrize("D,per_key", [(128, False), (64, True), (16, False)])
def test_prefill_fused_conv(D, per_key):
    """q, k, v from the width-4 conv of mixed_qkv; prompts of 0, 1, 2, 33 and 70 positions
    (the conv reaches into the slot's conv state for the first three), a padding request;
    conv states afterwards bit-exact."""
    e_o, e_s, ok, _ = _run_ext(D, per_key, 70, np.array([0, 1, 2, 33, 70, 40]), conv=True,
                               slot=[4, 0, 2, -1, 3, 1], seed=50 + D)
    assert e_o <= TOL and e_s <= TOL and ok, (e_o, e_s, ok)


def test_prefill_fused_conv_fp32_no_bias():
    e_o, e_s, ok, _ = _run_ext(128, False, 40, np.array([40, 3, 17]), conv=True, bias=False, bf16=False, seed=61)
    assert e_o <= TOL and e_s <= TOL and ok, (e_o, e_s, ok)


def test_prefill_kda_gate_and_epilogue():
    """The KDA gate parametrisation and output epilogue, per-key and per-head decay."""
    for per_key in (True, False):
        e_o, e_s, _, _ = _run_ext(128, per_key, 70, np.array([70, 33, 1, 0]), kda=True, seed=62 + int(per_key))
        assert e_o <= TOL and e_s <= TOL, (per_key, e_o, e_s)


def test_prefill_conv_then_fused_conv_decode():
    """The small hybrid-layer form end to end: a fused-conv prefill leaves the state and the
    conv state a fused-conv dense decode continues from (matches the oracle's pass over the
    prompt and four generated tokens)."""
    e_o, e_s, ok, (dims, pool, dev, cfg, pool_ref, ref) = _run_ext(
        128, False, 50, np.array([50, 37, 2, 50]), conv=True, slot=[0, 1, 2, 3], seed=70)
    assert e_o <= TOL and e_s <= TOL and ok, (e_o, e_s, ok)
    B, H, D = 4, 2, 128
    nch = 3 * H * D
    st = oracle.BatchState(cfg["num_slots"], H, D, D)
    st.S, st.conv = pool_ref, ref["conv_pool"]
    cfg_d = dict(cfg, batch=B, flags=cfg["flags"] | oracle.CONV)
    slot = np.arange(B, dtype=np.int32)
    r = np.random.default_rng(71)
    o = torch.zeros((B, H, D), device="cuda")
    err = ref_max = 0.0
    for t in range(4):
        bits, mixed = wl.bf16_round(r.standard_normal((B, nch)).astype(np.float32))
        lam = (-np.log1p(np.exp(-(r.standard_normal((B, H, 1)) + 3)))).astype(np.float32)
        beta = (1 / (1 + np.exp(-r.standard_normal((B, H))))).astype(np.float32)
        ins = gdn.make_inputs(mixed_qkv=dev_bf16(bits), conv_w=dev["conv_w"], conv_b=dev["conv_b"],
                              conv_pool=dev["conv_pool"], log_decay=dev_f32(lam), beta=dev_f32(beta),
                              slot=dev_i32(slot))
        gdn.decode_dense(dims, ins, pool, o)
        o_ref = oracle.step_batch(cfg_d, "dense", st, slot, mixed=mixed.astype(np.float64),
                                  conv_w=ref["conv_w"], conv_b=ref["conv_b"], lam=lam.astype(np.float64),
                                  beta=beta.astype(np.float64))
        torch.cuda.synchronize()
        err = max(err, float(np.max(np.abs(o.cpu().numpy() - o_ref))))
        ref_max = max(ref_max, float(np.max(np.abs(o_ref))))
    assert err / ref_max <= TOL, err / ref_max


@pytest.mark.parametrize("lam_mean", [-6.0, -4.5])
def test_prefill_strong_per_key_decay(lam_mean):
    """Per-key decay strong enough that a 16-token sub-block spans more than e^80 (mean -6:
    the exact per-term pair factors) or close to it (mean -4.5: the reference-point split),
    and a prompt whose chunks alternate between mild and strong decay (both paths in one
    call); outputs and states at the dense bar."""
    B, T, H, D = 3, 96, 2, 128
    lens = np.array([96, 70, 33])
    dev, ref = _inputs(B, T, H, D, D, True, 90)
    r = np.random.default_rng(91)
    lam = (lam_mean + 0.5 * r.standard_normal((B, T, H, D))).astype(np.float32)
    lam = np.minimum(lam, np.float32(0))
    mixed = lam.copy()
    mixed[:, 32:64] = (-0.05 * r.random((B, 32, H, D))).astype(np.float32)  # chunk 1 mild
    for lm in (lam, mixed):
        dev["log_decay"] = dev_f32(lm)
        ref["lam"] = lm.astype(np.float64)
        slot = np.arange(B, dtype=np.int32)
        pool0 = (0.1 * r.standard_normal((B, H, D, D))).astype(np.float32)
        pool, pool_ref = dev_f32(pool0), pool0.astype(np.float64)
        dims = gdn.make_dims(B, H, D, num_slots=B, decay_per_key=True, flags=gdn.QKV_BF16, q_scale=D ** -0.5)
        cfg = dict(batch=B, num_heads=H, dk=D, dv=D, num_slots=B, dlam=D, log_capacity=0,
                   flags=oracle.L2NORM, q_scale=D ** -0.5, l2_eps=1e-6)
        o = torch.zeros((B, T, H, D), device="cuda")
        gdn.prefill(dims, T, gdn.make_inputs(slot=dev_i32(slot), **dev), pool, o, seq_lens=dev_i32(lens))
        o_ref = oracle.prefill_batch(cfg, pool_ref, slot, lens, **ref)
        torch.cuda.synchronize()
        og = o.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(og))
        err = max(float(np.max(np.abs(og[b, :lens[b]] - o_ref[b, :lens[b]]))) for b in range(B))
        scale = max(float(np.max(np.abs(o_ref[b, :lens[b]]))) for b in range(B))
        pg = pool.cpu().numpy().astype(np.float64)
        serr = float(np.max(np.abs(pg - pool_ref))) / float(np.max(np.abs(pool_ref)))
        assert err / scale <= TOL and serr <= TOL, (lam_mean, err / scale, serr)


def test_prefill_raw_value_update_per_head_decay():
    """b = beta v (beta NULL: 1), raw q and k, with a per-head decay: the head-size-128 path
    of this shape takes the tensor-core kernel, whose plain form skips the substitution."""
    e_o, e_s, _ = _run(128, False, 64, np.array([64, 40, 3]), raw_value=True, seed=6)
    assert e_o <= TOL and e_s <= TOL, (e_o, e_s)


@pytest.mark.parametrize("lam_mean", [-6.0, -0.02])
def test_prefill_strong_and_weak_per_head_decay(lam_mean):
    """Per-head decay of mean -6 per token (e^gamma underflows inside a chunk: the decayed
    key and query factors reach zero while the pair ratios e^{gamma_t - gamma_s} and the
    Khat factors stay exact) and nearly no decay (the state grows over a long prompt);
    outputs and states at the dense bar, across four chunks and a ragged tail."""
    B, T, H, D = 3, 120, 2, 128
    lens = np.array([120, 97, 33])
    dev, ref = _inputs(B, T, H, D, 1, True, 95)
    r = np.random.default_rng(96)
    lam = np.minimum(lam_mean + 0.5 * abs(lam_mean) * r.standard_normal((B, T, H, 1)), 0).astype(np.float32)
    dev["log_decay"] = dev_f32(lam)
    ref["lam"] = lam.astype(np.float64)
    slot = np.arange(B, dtype=np.int32)
    pool0 = (0.1 * r.standard_normal((B, H, D, D))).astype(np.float32)
    pool, pool_ref = dev_f32(pool0), pool0.astype(np.float64)
    dims = gdn.make_dims(B, H, D, num_slots=B, flags=gdn.QKV_BF16, q_scale=D ** -0.5)
    cfg = dict(batch=B, num_heads=H, dk=D, dv=D, num_slots=B, dlam=1, log_capacity=0,
               flags=oracle.L2NORM, q_scale=D ** -0.5, l2_eps=1e-6)
    o = torch.zeros((B, T, H, D), device="cuda")
    gdn.prefill(dims, T, gdn.make_inputs(slot=dev_i32(slot), **dev), pool, o, seq_lens=dev_i32(lens))
    o_ref = oracle.prefill_batch(cfg, pool_ref, slot, lens, **ref)
    torch.cuda.synchronize()
    og = o.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(og))
    err = max(float(np.max(np.abs(og[b, :lens[b]] - o_ref[b, :lens[b]]))) for b in range(B))
    scale = max(float(np.max(np.abs(o_ref[b, :lens[b]]))) for b in range(B))
    pg = pool.cpu().numpy().astype(np.float64)
    serr = float(np.max(np.abs(pg - pool_ref))) / float(np.max(np.abs(pool_ref)))
    assert err / scale <= TOL and serr <= TOL, (lam_mean, err / scale, serr)


def test_prefill_fused_conv_tensor_core_ragged_chunks_no_bias():
    """The fused conv on the 128-wide tensor-core prefill: three heads (the q, k and v thirds
    of mixed_qkv at every head offset), prompts that end inside the conv state's reach (1, 3),
    at and around chunk edges (31, 32, 35, 64) and over several chunks (97, 200), no bias;
    request 0 is live (its copies start before the first row of the tensor); conv states
    bit-exact afterwards."""
    e_o, e_s, ok, _ = _run_ext(128, False, 200, np.array([200, 3, 1, 31, 32, 35, 97, 64]), conv=True,
                               bias=False, H=3, slot=[0, 5, 2, 7, 1, 3, 6, 4], seed=81)
    assert e_o <= TOL and e_s <= TOL and ok, (e_o, e_s, ok)


def _sampled_full_shape(name, T, pairs, seed):
    """gdn_prefill over a workload's whole batch (B requests x H heads, the grid the bench times),
    from a zero state, checked against the oracle on sampled (request, head) pairs: every
    position's output and the final state (and conv state) of each sampled head. Inputs as the
    bench draws them: N(0,1) bf16 q/k/v (or mixed_qkv through the workload's conv weights),
    alpha = sigmoid(N(0,1) + 3), beta = sigmoid(N(0,1)); the KDA workload takes its raw gate
    f = N(0,1) and write logit, and N(0,1) output gates."""
    w = wl.WORKLOADS[name]
    B, H, D, dlam = w.batch, w.num_heads, w.dk, w.dlam
    r = np.random.default_rng(seed)
    flags, oflags = gdn.QKV_BF16, oracle.L2NORM
    dev, smp = {}, [dict() for _ in pairs]
    chans = [np.concatenate([np.arange(t * H * D + h * D, t * H * D + (h + 1) * D) for t in range(3)])
             for _, h in pairs]
    if w.conv:
        flags |= gdn.FUSE_CONV
        bits, a = wl.bf16_round(r.standard_normal((B, T, w.channels), dtype=np.float32))
        dev["mixed_qkv"] = dev_bf16(bits)
        del bits
        cw = wl.conv_weights(w)
        dev["conv_w"] = dev_f32(cw)
        dev["conv_pool"] = torch.zeros((B, w.channels, 3), dtype=torch.bfloat16, device="cuda")
        for i, (b, h) in enumerate(pairs):
            smp[i].update(mixed=a[b:b + 1][:, :, chans[i]].astype(np.float64), conv_w=cw[chans[i]].astype(np.float64),
                          conv_b=None, conv_pool=np.zeros((1, 3 * D, 3)))
        del a
    else:
        for n in ("q", "k", "v"):
            bits, a = wl.bf16_round(r.standard_normal((B, T, H, D), dtype=np.float32))
            dev[n] = dev_bf16(bits)
            for i, (b, h) in enumerate(pairs):
                smp[i][n] = a[b:b + 1, :, h:h + 1].astype(np.float64)
            del bits, a
    a_raw = r.standard_normal((B, T, H, dlam), dtype=np.float32) + np.float32(3)
    b_raw = r.standard_normal((B, T, H), dtype=np.float32)
    if w.kda_full:
        flags |= gdn.GATE_KDA | gdn.OUT_NORM_GATE
        oflags |= oracle.GATE_KDA | oracle.OUT_NORM_GATE
        kp = wl.kda_gate_params(w)
        lam, beta = a_raw - np.float32(3), b_raw
        g = r.standard_normal((B, T, H, D), dtype=np.float32)
        dev.update(out_gate=dev_f32(g), **{n: dev_f32(kp[n]) for n in ("a_log", "dt_bias", "out_norm_w")})
        for i, (b, h) in enumerate(pairs):
            smp[i].update(out_gate=g[b:b + 1, :, h:h + 1].astype(np.float64),
                          a_log=kp["a_log"][h:h + 1].astype(np.float64),
                          dt_bias=kp["dt_bias"][h:h + 1].astype(np.float64),
                          out_norm_w=kp["out_norm_w"].astype(np.float64), lower_bound=kp["lower_bound"])
        del g
    else:
        lam = (-np.log1p(np.exp(-a_raw.astype(np.float64)))).astype(np.float32)
        beta = (1 / (1 + np.exp(-b_raw.astype(np.float64)))).astype(np.float32)
    dev.update(log_decay=dev_f32(lam), beta=dev_f32(beta))
    for i, (b, h) in enumerate(pairs):
        smp[i].update(lam=lam[b:b + 1, :, h:h + 1].astype(np.float64), beta=beta[b:b + 1, :, h:h + 1].astype(np.float64))
    del lam, beta, a_raw, b_raw
    dims = gdn.make_dims(B, H, D, num_slots=B, decay_per_key=w.decay_per_key, flags=flags, q_scale=D ** -0.5)
    pool = torch.zeros((B, H, D, D), dtype=torch.float32, device="cuda")
    o = torch.full((B, T, H, D), 5.0, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.prefill(dims, T, gdn.make_inputs(slot=dev_i32(np.arange(B)), **dev), pool, o, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    cfg = dict(batch=1, num_heads=1, dk=D, dv=D, num_slots=1, dlam=dlam, log_capacity=0, flags=oflags,
               q_scale=D ** -0.5, l2_eps=1e-6)
    for i, (b, h) in enumerate(pairs):
        pool_ref = np.zeros((1, 1, D, D))
        o_ref = oracle.prefill_batch(cfg, pool_ref, np.zeros(1, np.int32), np.array([T]), **smp[i])
        og = o[b, :, h].cpu().numpy().astype(np.float64)
        e_o = float(np.max(np.abs(og - o_ref[0, :, 0]))) / float(np.max(np.abs(o_ref[0, :, 0])))
        sg = pool[b, h].cpu().numpy().astype(np.float64)
        e_s = float(np.max(np.abs(sg - pool_ref[0, 0]))) / float(np.max(np.abs(pool_ref[0, 0])))
        assert e_o <= TOL and e_s <= TOL, (name, b, h, e_o, e_s)
        if w.conv:
            cp = dev["conv_pool"][b][torch.from_numpy(chans[i]).cuda()].cpu()
            cg = (cp.view(torch.int16).numpy().astype(np.uint16).astype(np.uint32) << 16).view(np.float32)
            assert np.array_equal(cg.astype(np.float64), smp[i]["conv_pool"][0]), (name, b, h)


def test_prefill_headline_full_batch_sampled():
    """The headline prefill (B=128, H=32, T=256: the tensor-core kernel for a per-head decay)."""
    _sampled_full_shape("headline", 256, [(0, 0), (127, 31), (5, 17), (64, 3), (99, 26)], seed=91)


def test_prefill_small_conv_full_batch_sampled():
    """The fused-conv prefill at its workload's full batch (B=64, H=16, T=256)."""
    _sampled_full_shape("small_conv", 256, [(0, 0), (63, 15), (17, 8), (40, 1)], seed=92)


def test_prefill_kda_full_full_batch_sampled():
    """The per-key tensor-core prefill with the KDA gate and epilogue at its workload's full
    batch (B=256, H=32), prompts of 128 positions."""
    _sampled_full_shape("kda_full", 128, [(0, 0), (255, 31), (128, 16), (77, 9)], seed=93)
