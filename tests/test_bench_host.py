"""Host-side plumbing of bench.py that needs no GPU: the extra prefill legs (each workload's
flags and prompt length reach the leg, a failing leg is reported and does not end the run)."""
import argparse

import bench
import linear_attention_decode_gdn_gb300 as gdn


def test_prefill_configs_pass_flags_and_lengths_and_contain_failures():
    calls = []

    def leg(a, w, flags, dev, stream, g):
        calls.append((w.name, a.prefill, a.steps, flags))
        if w.name == "kda_full":
            raise RuntimeError("leg failed")
        return {"ms_per_call": 1.0, "launches": 5}

    args = argparse.Namespace(prefill=256, steps=20, warmup=5, workload="headline")
    legs, launches = bench.run_prefill_configs(args, None, None, gdn, runner=leg)
    assert list(legs) == [f"{n}/T{t}" for n, t in bench.PREFILL_CONFIGS] == ["small_conv/T256", "kda_full/T128"]
    assert launches == 5 and legs["small_conv/T256"]["launches"] == 5
    assert legs["kda_full/T128"]["unavailable"] == "RuntimeError: leg failed"
    assert all(legs[k]["workload"].startswith(k.split("/")[0] + ": ") for k in legs)
    # the conv leg sees the fused conv on bf16 mixed_qkv; the KDA leg its gate and epilogue
    assert calls[0] == ("small_conv", 256, 20, gdn.QKV_BF16 | gdn.FUSE_CONV)
    name, T, steps, flags = calls[1]
    assert (name, T, steps) == ("kda_full", 128, 20)
    assert flags & gdn.GATE_KDA and flags & gdn.OUT_NORM_GATE and flags & gdn.QKV_BF16
    assert not flags & gdn.FUSE_CONV
    assert args.prefill == 256  # the caller's arguments are left as they were


def test_prefill_configs_take_the_tensor_core_kernels():
    """Both extra legs are shapes the tensor-core prefill kernels take (128-wide heads, bf16)."""
    from linear_attention_decode_gdn_gb300 import workloads as wl
    for name, T in bench.PREFILL_CONFIGS:
        w = wl.WORKLOADS[name]
        flags = bench.decode_flags(gdn, w)
        pflags = flags & (gdn.QKV_BF16 | gdn.NO_QK_L2NORM | gdn.PLAIN_UPDATE | gdn.FUSE_CONV)
        if w.kda_full:
            pflags |= gdn.GATE_KDA | gdn.OUT_NORM_GATE
        assert bench.prefill_on_tensor_cores(w.dk, w.decay_per_key, pflags, gdn, w.batch, T), name
