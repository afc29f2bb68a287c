"""GPU parity of the decode steps on the other head shapes, through the C ABI, against the fp64
oracle: heads split along dv over a cluster of two CTAs (GDN_SPLIT_DV; the DeltaLog notes'
Sec. 2.6 / Fig. 5 slicing, one writer per slice), and key / value head sizes that differ
(dk = 128 / dv = 64, dk = 64 / dv = 128). Same bars as the square unsplit path: 1e-4 dense,
5e-3 append-merge with bf16 keys, 1e-4 with exact key factors."""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import linear_attention_decode_gdn_gb300 as gdn  # noqa: E402
from linear_attention_decode_gdn_gb300 import workloads as wl  # noqa: E402

from gpu_harness import Lockstep, Variant, dev_bf16, dev_f32, dev_i32  # noqa: E402

pytestmark = pytest.mark.gpu

DENSE_TOL = 1e-4
LOG_TOL = 5e-3
SPLIT = gdn.SPLIT_DV


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_attention_decode_gdn_gb300 import build
    build.build()


def _check(ls: Lockstep, exact=()):
    ls.compare_states()
    report = []
    for v in ls.variants:
        tol = DENSE_TOL if (v.mode == "dense" or v.name in exact) else LOG_TOL
        report.append(f"{v.name}: out {v.rel_err:.3e} state {v.state_rel_err:.3e}")
        assert ls.status(v) == 0, f"{v.name}: status {ls.status(v)}"
        assert v.rel_err <= tol, report
        if not math.isnan(v.state_err):
            assert v.state_rel_err <= tol, report
    print("; ".join(report))
    return report


def _custom(name, B, H, dk, dv, steps, bf16=True, conv=False, per_key=False, qk_mult=1.0, seed=77):
    return wl.Workload(name, B, H, dk, dv, steps, (1,), bf16, conv, per_key, seed, qk_mult=qk_mult)


# ---------------------------------------------------------------- split along dv

def test_split_dv_headline():
    w = wl.WORKLOADS["headline"]
    _check(Lockstep(w, [Variant("dense", extra_flags=SPLIT, name="dense/split"),
                        Variant("deltalog", 8, extra_flags=SPLIT, name="M=8/split"),
                        Variant("deltalog", 8, "step", extra_flags=SPLIT, name="M=8/step/split"),
                        Variant("deltalog", 8, extra_flags=SPLIT | gdn.KLOG_PRENORM, name="M=8/prenorm/split")]).run(),
           exact=("M=8/prenorm/split",))


def test_split_dv_small_conv():
    """The fused conv: slice 0 shifts the q / k cache rows after the cluster barrier, every
    slice the v rows of its columns."""
    w = wl.WORKLOADS["small_conv"]
    _check(Lockstep(w, [Variant("dense", extra_flags=SPLIT, name="dense/split"),
                        Variant("deltalog", 8, extra_flags=SPLIT, name="M=8/split")]).run())


def test_split_dv_kda_and_rwkv6():
    _check(Lockstep(wl.WORKLOADS["kda"], [Variant("deltalog", 8, extra_flags=SPLIT, name="M=8/split")],
                    batch=64).run())
    w = wl.WORKLOADS["rwkv6"]
    ls = Lockstep(w, [Variant("deltalog", 4, extra_flags=SPLIT, name="M=4/split"),
                      Variant("deltalog", 4, "step", extra_flags=SPLIT, name="M=4/step/split")], batch=64).run()
    rep = _check(ls)
    for v in ls.variants:  # exact logged factors: the dense bar
        assert v.rel_err <= DENSE_TOL and v.state_rel_err <= DENSE_TOL, rep


@pytest.mark.parametrize("per_key", [False, True])
def test_split_dv_head64_ragged_batch_and_slots(per_key):
    w = _custom("s64", 5, 3, 64, 64, 24, per_key=per_key, seed=140 + int(per_key))
    slot = np.array([6, -1, 0, 3, 5], dtype=np.int32)
    ls = Lockstep(w, [Variant("dense", extra_flags=SPLIT, name="dense/split"),
                      Variant("deltalog", 3, extra_flags=SPLIT, name="M=3/split"),
                      Variant("deltalog", 5, "step", extra_flags=SPLIT, name="M=5/step/split")],
                  slot=slot, num_slots=8, q_scale=64 ** -0.5).run()
    _check(ls)
    for v in ls.variants:  # padding row untouched; unused slots untouched
        assert torch.all(v.o[1] == 0)
        for s in (1, 2, 4, 7):
            assert torch.all(v.pools.state[s] == 0)


def test_split_dv_matches_unsplit_and_is_deterministic():
    """Split and unsplit agree up to the order of the column sums; the split path is bitwise
    reproducible; the metadata slice 0 commits (L, ell, Lambda and the bf16 key log) is bitwise
    the unsplit path's."""
    w = _custom("sdet", 32, 8, 128, 128, 9, seed=16)
    runs = [Lockstep(w, [Variant("deltalog", 4, extra_flags=SPLIT, name="M=4/split"),
                         Variant("deltalog", 4, name="M=4"),
                         Variant("dense", extra_flags=SPLIT, name="dense/split"), Variant("dense")],
                     keep_outputs=True).run() for _ in range(2)]
    a, b = runs
    for va, vb in zip(a.variants, b.variants):
        for oa, ob in zip(va.outputs, vb.outputs):
            assert np.array_equal(oa, ob), va.name
        assert torch.equal(va.pools.state, vb.pools.state), va.name
    split, plain = a.variants[0], a.variants[1]
    for name in ("length", "ell", "lam_log", "k_log"):
        assert torch.equal(getattr(split.pools, name), getattr(plain.pools, name)), name
    scale = max(float(np.max(np.abs(o))) for o in plain.outputs)
    for os_, op in zip(split.outputs, plain.outputs):
        assert float(np.max(np.abs(os_ - op))) <= 1e-6 * scale
    us, up = split.pools.u_log.float(), plain.pools.u_log.float()
    assert float((us - up).abs().max()) <= 1e-6 * max(1e-30, float(up.abs().max()))


def test_split_dv_m1_merge_is_bitwise_split_dense():
    w = _custom("sm1", 16, 8, 128, 128, 12, seed=15)
    ls = Lockstep(w, [Variant("dense", extra_flags=SPLIT, name="dense/split"),
                      Variant("deltalog", 1, extra_flags=SPLIT, name="M=1/split")], keep_outputs=True).run()
    a, b = ls.variants
    for oa, ob in zip(a.outputs, b.outputs):
        assert np.array_equal(oa, ob)
    assert torch.equal(a.pools.state, b.pools.state)


def test_split_dv_status_and_timeout():
    """A bad slot and a full log are skipped by both slices with one status bit each; the
    test-only starved wait runs out in both slices, the call reports the timeout and writes
    nothing (output, state, log, conv cache); the context survives."""
    B, H, D, C = 2, 2, 128, 3
    flags = SPLIT | gdn.FUSE_CONV | gdn.QKV_BF16
    dims = gdn.make_dims(B, H, D, num_slots=4, log_capacity=C, flags=flags)
    pools = gdn.Pools.allocate(dims, conv=True, deltalog=True)
    ch = 3 * H * D
    pools.conv.copy_(torch.randn(pools.conv.shape, device="cuda").to(torch.bfloat16))
    pools.state.normal_()
    gates = dict(mixed_qkv=torch.randn((B, ch), device="cuda").to(torch.bfloat16),
                 conv_w=torch.randn((ch, 4), device="cuda") * 0.5,
                 log_decay=-torch.rand((B, H), device="cuda") * 0.1, beta=torch.rand((B, H), device="cuda"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = torch.full((B, H, D), 9.0, device="cuda")
    # bad slot + padding
    gdn.decode_dense(dims, gdn.make_inputs(conv_pool=pools.conv, slot=dev_i32([-1, 4]), **gates), pools.state, o,
                     status)
    torch.cuda.synchronize()
    assert status.item() == gdn.STATUS_BAD_SLOT and torch.all(o == 9.0)
    # full log on one slot-head: that head is skipped, the rest appends
    status.zero_()
    pools.length[1, 0] = C
    snap = {n: getattr(pools, n).clone() for n in ("state", "conv", "k_log", "u_log", "lam_log", "ell", "length")}
    gdn.decode_append(dims, gdn.make_inputs(conv_pool=pools.conv, slot=dev_i32([0, 1]), **gates), pools.state,
                      pools.log(), o, status)
    torch.cuda.synchronize()
    assert status.item() == gdn.STATUS_LOG_FULL
    assert torch.all(o[1, 0] == 9.0) and not torch.any(o[0] == 9.0) and not torch.any(o[1, 1] == 9.0)
    assert pools.length[1, 0].item() == C and pools.length[0, 0].item() == 1 and pools.length[1, 1].item() == 1
    # starved wait in both slices: nothing written
    status.zero_()
    o.fill_(9.0)
    snap = {n: getattr(pools, n).clone() for n in ("state", "conv", "k_log", "u_log", "lam_log", "ell", "length")}
    starve = gdn.make_dims(B, H, D, num_slots=4, log_capacity=C, flags=flags | gdn.TEST_STARVE_WAIT)
    gdn.decode_merge(starve, gdn.make_inputs(conv_pool=pools.conv, slot=dev_i32([0, 1]), **gates), pools.state,
                     pools.log(), o, status)
    torch.cuda.synchronize()
    assert status.item() == gdn.STATUS_TIMEOUT and torch.all(o == 9.0)
    for n, t in snap.items():
        assert torch.equal(getattr(pools, n), t), n
    status.zero_()
    gdn.decode_merge(dims, gdn.make_inputs(conv_pool=pools.conv, slot=dev_i32([0, 1]), **gates), pools.state,
                     pools.log(), o, status)
    torch.cuda.synchronize()
    assert status.item() == 0 and not torch.any(o == 9.0) and torch.all(pools.length == 0)


# ---------------------------------------------------------------- dk != dv

@pytest.mark.parametrize("dk,dv", [(128, 64), (64, 128)])
@pytest.mark.parametrize("per_key", [False, True])
def test_nonsquare_heads(dk, dv, per_key):
    w = _custom(f"ns{dk}x{dv}", 5, 3, dk, dv, 24, per_key=per_key, seed=dk + dv + int(per_key))
    slot = np.array([6, -1, 0, 3, 5], dtype=np.int32)
    ls = Lockstep(w, [Variant("dense"), Variant("deltalog", 3), Variant("deltalog", 5, "step"),
                      Variant("deltalog", 4, extra_flags=gdn.KLOG_PRENORM, name="M=4/prenorm")],
                  slot=slot, num_slots=8, q_scale=dk ** -0.5).run()
    _check(ls, exact=("M=4/prenorm",))
    for v in ls.variants:
        assert torch.all(v.o[1] == 0)


@pytest.mark.parametrize("dk,dv", [(128, 64), (64, 128)])
def test_nonsquare_heads_fused_conv_fp32_raw_gates(dk, dv):
    """Channel order [q heads (H dk) | k heads (H dk) | v heads (H dv)] through the fused conv."""
    w = _custom(f"nsc{dk}x{dv}", 3, 2, dk, dv, 20, bf16=False, conv=True, seed=400 + dk)
    _check(Lockstep(w, [Variant("dense"), Variant("deltalog", 4)], gate_raw=True).run())


def test_nonsquare_log_bytes_and_reset():
    """The log sizes of a dk x dv head, and gdn_slot_reset clearing a dk x dv state row."""
    dims = gdn.make_dims(2, 3, 128, 64, num_slots=4, log_capacity=5, flags=gdn.FUSE_CONV | gdn.QKV_BF16)
    s = gdn.log_bytes(dims)
    assert s["k_log"] == 4 * 3 * 5 * 128 * 2 and s["u_log"] == 4 * 3 * 5 * 64 * 4
    pools = gdn.Pools.allocate(dims, conv=True, deltalog=True)
    for t in (pools.state, pools.ell, pools.u_log):
        t.fill_(1)
    pools.conv.fill_(1)
    pools.length.fill_(2)
    gdn.slot_reset(dims, dev_i32([2, -1]), 2, pools.log(), pools.conv, pools.state)
    torch.cuda.synchronize()
    assert torch.all(pools.state[2] == 0) and torch.all(pools.state[1] == 1)
    assert torch.all(pools.conv[2] == 0) and torch.all(pools.conv[0] == 1)
    assert torch.all(pools.length[2] == 0) and torch.all(pools.ell[2] == 0) and torch.all(pools.length[0] == 2)
