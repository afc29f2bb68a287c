"""The benchmark's algorithmic byte model (bench.head_bytes_rw) against the traffic model of the
DeltaLog reading notes (Sec. 2.5, "流量模型：节省写回，付出重放"): per decode step, dense moves
T_common + 2 C_state and a DeltaLog cycle of M steps moves, on average,
T_common + C_state + C_state / M + ((M-1)/M + (M-1)/2) C_entry + 2 C_decay. The per-launch
model is summed over one cycle and compared with that closed form; the only extra term is the
log length L (4 bytes read and 4 written per head), an index the notes leave out of their
model. Also pinned: the headline figures the notes' Fig. 8 discussion is about."""
import pytest

import bench
from linear_attention_decode_gdn_gb300 import workloads as wl


def _closed_form(w, M, klb=2, ulb=4):
    D, dlam = w.dk, w.dlam
    r, wr = bench.head_bytes_rw("dense", 0, w, klb, w.conv, ulb)
    state = 4 * D * D
    common = r + wr - 2 * state                   # T_common per head
    entry = klb * D + ulb * D + 4 * dlam          # C_entry per head
    decay = 4 * dlam                              # C_decay per head
    dense = common + 2 * state
    delta = common + state + state / M + ((M - 1) / M + (M - 1) / 2) * entry + 2 * decay
    return dense, delta


def _cycle_average(w, M, klb=2, ulb=4):
    launches = [bench.head_bytes_rw("append", n, w, klb, w.conv, ulb) for n in range(M - 1)]
    launches.append(bench.head_bytes_rw("merge", M - 1, w, klb, w.conv, ulb))
    return sum(r + wr for r, wr in launches) / M


@pytest.mark.parametrize("name", ["tiny", "small_conv", "headline", "high_concurrency", "kda", "kda_full"])
@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
def test_cycle_average_equals_the_notes_model(name, M):
    w = wl.WORKLOADS[name]
    dense, delta = _closed_form(w, M)
    assert sum(bench.head_bytes_rw("dense", 0, w, 2, w.conv, 4)) == dense
    assert _cycle_average(w, M) == pytest.approx(delta + 8, rel=1e-12, abs=1e-9)


def test_rwkv6_bf16_value_log():
    w = wl.WORKLOADS["rwkv6"]
    for M in (2, 4):
        _, delta = _closed_form(w, M, ulb=2)
        assert _cycle_average(w, M, ulb=2) == pytest.approx(delta + 8, rel=1e-12)


def test_headline_figures():
    """B=128, H=32, dk=dv=128, bf16 q/k/v, M=8: dense 517.0 MiB per step, the DeltaLog cycle
    306.3 MiB per step (1.69x less traffic, 7.0x fewer writes); per launch, append with L=0
    264.1 MiB, with L=6 282.2 MiB, merge with L=7 538.2 MiB. The read of a dense step, 259.0
    MiB, is the notes' measured 0.253 GiB (Fig. 8); their measured writes fall below the model
    because dirty lines stay in L2 when a kernel ends."""
    w = wl.WORKLOADS["headline"]
    heads, MiB = 128 * 32, 2.0 ** 20
    dr, dw = (x * heads / MiB for x in bench.head_bytes_rw("dense", 0, w))
    assert round(dr + dw, 1) == 517.0 and round(dr, 1) == 259.0
    launches = [bench.head_bytes_rw("append", n, w) for n in range(7)] + [bench.head_bytes_rw("merge", 7, w)]
    step_r = sum(r for r, _ in launches) * heads / 8 / MiB
    step_w = sum(x for _, x in launches) * heads / 8 / MiB
    assert round(step_r + step_w, 1) == 306.3
    assert round((dr + dw) / (step_r + step_w), 2) == 1.69 and round(dw / step_w, 1) == 7.0
    per = {k: sum(bench.head_bytes_rw(m, n, w)) * heads / MiB
           for k, (m, n) in {"a0": ("append", 0), "a6": ("append", 6), "m7": ("merge", 7)}.items()}
    assert (round(per["a0"], 1), round(per["a6"], 1), round(per["m7"], 1)) == (264.1, 282.2, 538.2)


def test_measured_traffic_parser_and_reductions(tmp_path):
    """The bench reads per-launch ncu bytes of one whole cycle only when they were taken on
    the current kernel sources, and forms the per-decode-step view from them: the cycle's
    reads and writes over M against one dense launch."""
    src = bench.kernel_source_hash()
    M = 4
    lines = ["# header", ""]
    for n in range(M - 1):
        lines.append(f"kernel=append L={n} M={M} workload=headline src={src} read={100 + n} write=2")
    lines.append(f"kernel=merge L={M - 1} M={M} workload=headline src={src} read=110 write=90")
    lines.append(f"kernel=dense L=0 M={M} workload=headline src={src} read=95 write=88")
    p = tmp_path / "t.txt"
    p.write_text("\n".join(lines) + "\n")
    meas = bench.measured_traffic("headline", M, path=str(p))
    assert meas[("append", 2)] == (102.0, 2.0) and meas[("dense", 0)] == (95.0, 88.0)
    s = bench.measured_summary(meas, M)
    cyc_r, cyc_w = 100 + 101 + 102 + 110, 2 * 3 + 90
    assert s["per_decode_step"]["deltalog_M4"] == {"read": cyc_r / M, "write": cyc_w / M}
    assert s["write_reduction"] == pytest.approx(88 / (cyc_w / M))
    assert s["total_reduction"] == pytest.approx((95 + 88) / ((cyc_r + cyc_w) / M))
    assert set(s["per_launch"]) == {"append_L0", "append_L2", "merge_L3", "dense"}
    # another source hash, another workload, a missing phase: no measured figures
    p.write_text("\n".join(lines).replace(src, "0" * 16) + "\n")
    assert bench.measured_traffic("headline", M, path=str(p)) is None
    p.write_text("\n".join(lines[:-1]) + "\n")
    assert bench.measured_traffic("headline", M, path=str(p)) is None
    assert bench.measured_traffic("kda", M, path=str(p)) is None


def test_cycle_bytes_per_head_is_the_sum_of_its_launches():
    w = wl.WORKLOADS["headline"]
    assert bench.cycle_bytes_per_head(w, 1, 2, 4) == bench.head_bytes("dense", 0, w)
    for M in (2, 4, 8, 16):
        cyc = sum(bench.head_bytes("append", n, w) for n in range(M - 1)) + bench.head_bytes("merge", M - 1, w)
        assert bench.cycle_bytes_per_head(w, M, 2, 4) == cyc
