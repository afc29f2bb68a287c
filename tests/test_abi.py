"""Host-side checks of the C-ABI library (no GPU needed, no compute launched).

* the library loads and exports every function include/gdn.h declares;
* gdn_log_bytes reproduces the DeltaLog notes' capacity table (Sec. 2.5);
* argument validation rejects bad calls before anything is launched.
Only invalid arguments are passed: every call here returns from validation.
"""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")

MiB = 1 << 20


@pytest.fixture(scope="module")
def gdn():
    from linear_attention_decode_gdn_gb300 import build
    build.build()
    import linear_attention_decode_gdn_gb300 as g
    return g


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(gdn_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("gdn_conv_l2norm", "gdn_decode_dense", "gdn_decode_append", "gdn_decode_merge"):
        assert required in names
    from linear_attention_decode_gdn_gb300 import _abi
    assert sorted(_abi.EXPORTS) == names


def test_library_exports_every_declared_symbol(gdn):
    lib = gdn._abi.load()
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", gdn._abi.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (gdn_\w+)", out))
    assert set(declared_functions()) <= exported
    assert lib.gdn_version() == 2


def test_strerror(gdn):
    lib = gdn._abi.load()
    for code in range(4):
        assert lib.gdn_strerror(code)
    assert lib.gdn_strerror(99) == b"unknown error code"


@pytest.mark.parametrize("per_key,M,bf16_u,C_entry_bytes,expected_mib,frac", [
    (False, 8, False, 2 * 128 + 4 * 128 + 4, 21.125, 0.0825),      # GDN row of the capacity table
    (True, 4, False, 2 * 128 + 4 * 128 + 4 * 128, 17.0, 0.0664),   # KDA row
    (True, 4, True, 2 * 128 + 2 * 128 + 4 * 128, 14.0, 0.0547),    # RWKV6 row (bf16 U log)
])
def test_log_bytes_matches_capacity_table(gdn, per_key, M, bf16_u, C_entry_bytes, expected_mib, frac):
    d = gdn.make_dims(128, 32, 128, num_slots=128, decay_per_key=per_key, log_capacity=M - 1,
                      flags=gdn.ULOG_BF16 if bf16_u else 0)
    s = gdn.log_bytes(d)
    assert s["residency"] == expected_mib * MiB
    B, H = 128, 32
    dlam = 128 if per_key else 1
    assert s["residency"] == (M - 1) * B * H * C_entry_bytes + 4 * B * H * dlam
    assert s["total"] == s["residency"] + 4 * B * H
    assert s["residency"] / (4 * B * H * 128 * 128) == pytest.approx(frac, abs=5e-4)


def test_log_bytes_fp32_keys(gdn):
    d = gdn.make_dims(2, 3, 64, num_slots=5, log_capacity=4, flags=gdn.KLOG_FP32)
    s = gdn.log_bytes(d)
    assert s["k_log"] == 5 * 3 * 4 * 64 * 4 and s["u_log"] == 5 * 3 * 4 * 64 * 4
    assert s["lam_log"] == 5 * 3 * 4 * 4 and s["ell"] == 5 * 3 * 4 and s["len"] == 5 * 3 * 4


def _expect(gdn, fn, code):
    with pytest.raises(gdn.GDNError) as ei:
        fn()
    assert ei.value.code == code, str(ei.value)


def test_validation_rejects_before_launch(gdn):
    from linear_attention_decode_gdn_gb300 import _abi
    lib = _abi.load()
    # NULL dims
    assert lib.gdn_decode_dense(None, None, None, None, None, None) == _abi.GDN_ERR_INVALID_ARG
    assert b"dims" in lib.gdn_last_error()
    fake = 1 << 20  # never dereferenced: every call below fails validation first
    ok_in = gdn.make_inputs(q=fake, k=fake, v=fake, log_decay=fake, beta=fake, slot=fake)
    # unsupported head sizes (the decode steps build square heads of 16..128, 128 x 64 and
    # 64 x 128; splitting along dv needs a square head of 64 or 128 and no KDA gate / epilogue)
    for dk, dv in ((48, 48), (128, 32), (32, 128), (256, 256)):
        d = gdn.make_dims(1, 1, dk, dv)
        _expect(gdn, lambda: gdn.decode_dense(d, ok_in, fake, fake, stream=0), _abi.GDN_ERR_UNSUPPORTED)
    for dk, dv, extra in ((32, 32, 0), (128, 64, 0), (128, 128, gdn.GATE_KDA), (128, 128, gdn.OUT_NORM_GATE)):
        d = gdn.make_dims(1, 1, dk, dv, flags=gdn.SPLIT_DV | extra)
        _expect(gdn, lambda: gdn.decode_dense(d, ok_in, fake, fake, stream=0), _abi.GDN_ERR_UNSUPPORTED)
    # the input stage, verify and prefill: square heads only, never split
    for d in (gdn.make_dims(1, 1, 128, 64), gdn.make_dims(1, 1, 128, flags=gdn.SPLIT_DV)):
        _expect(gdn, lambda: gdn.prefill(d, 4, ok_in, fake, fake, stream=0), _abi.GDN_ERR_UNSUPPORTED)
        _expect(gdn, lambda: gdn.decode_verify(d, 2, ok_in, fake, fake, fake, fake, stream=0),
                _abi.GDN_ERR_UNSUPPORTED)
    d = gdn.make_dims(1, 1, 128)
    # missing inputs
    _expect(gdn, lambda: gdn.decode_dense(d, gdn.make_inputs(q=fake, k=fake, log_decay=fake, beta=fake,
                                                              slot=fake), fake, fake, stream=0),
            _abi.GDN_ERR_INVALID_ARG)
    # misaligned pointers
    bad_in = gdn.make_inputs(q=fake + 8, k=fake, v=fake, log_decay=fake, beta=fake, slot=fake)
    _expect(gdn, lambda: gdn.decode_dense(d, bad_in, fake, fake, stream=0), _abi.GDN_ERR_UNSUPPORTED)
    _expect(gdn, lambda: gdn.decode_dense(d, ok_in, fake + 4, fake, stream=0), _abi.GDN_ERR_UNSUPPORTED)
    # unknown flags, bad decay mode, negative sizes
    for dd in (gdn.make_dims(1, 1, 128, flags=1 << 20), gdn.make_dims(-1, 1, 128),
               gdn.make_dims(1, 0, 128)):
        _expect(gdn, lambda: gdn.decode_dense(dd, ok_in, fake, fake, stream=0), _abi.GDN_ERR_INVALID_ARG)
    d2 = gdn.make_dims(1, 1, 128)
    d2.decay_per_key = 2
    _expect(gdn, lambda: gdn.decode_dense(d2, ok_in, fake, fake, stream=0), _abi.GDN_ERR_INVALID_ARG)
    # DeltaLog calls: log required; append needs C >= 1; C <= 63; log pointers when C > 0
    dl = gdn.make_dims(1, 1, 128, log_capacity=7)
    log_ok = gdn.make_log(fake, fake, fake, fake, fake)
    _expect(gdn, lambda: lib_call(lib, "gdn_decode_append", dl, ok_in, fake, None, fake),
            _abi.GDN_ERR_INVALID_ARG)
    _expect(gdn, lambda: gdn.decode_append(gdn.make_dims(1, 1, 128, log_capacity=0), ok_in, fake,
                                           log_ok, fake, stream=0), _abi.GDN_ERR_INVALID_ARG)
    _expect(gdn, lambda: gdn.decode_merge(gdn.make_dims(1, 1, 128, log_capacity=64), ok_in, fake,
                                          log_ok, fake, stream=0), _abi.GDN_ERR_UNSUPPORTED)
    _expect(gdn, lambda: gdn.decode_merge(dl, ok_in, fake, gdn.make_log(None, fake, fake, fake, fake),
                                          fake, stream=0), _abi.GDN_ERR_INVALID_ARG)
    # flag combinations
    _expect(gdn, lambda: gdn.decode_merge(
        gdn.make_dims(1, 1, 128, log_capacity=7, flags=gdn.KLOG_PRENORM | gdn.FUSE_CONV), ok_in,
        fake, log_ok, fake, stream=0), _abi.GDN_ERR_UNSUPPORTED)
    _expect(gdn, lambda: gdn.conv_l2norm(gdn.make_dims(1, 1, 128), ok_in, fake, fake, fake, stream=0),
            _abi.GDN_ERR_INVALID_ARG)
    _expect(gdn, lambda: gdn.slot_reset(gdn.make_dims(1, 1, 128), None, -1, stream=0),
            _abi.GDN_ERR_INVALID_ARG)
    # batch == 0 is a no-op that launches nothing
    gdn.decode_dense(gdn.make_dims(0, 1, 128, num_slots=1), ok_in, fake, fake, stream=0)


def lib_call(lib, name, dims, inputs, pool, log, o):
    from linear_attention_decode_gdn_gb300 import _abi
    rc = getattr(lib, name)(ctypes.byref(dims), ctypes.byref(inputs), pool,
                            None if log is None else ctypes.byref(log), o, None, None)
    _abi.check(rc, name)


def test_verify_validation_rejects_before_launch(gdn):
    from linear_attention_decode_gdn_gb300 import _abi
    fake = 1 << 20  # never dereferenced: every call below fails validation first
    ins = gdn.make_inputs(q=fake, k=fake, v=fake, log_decay=fake)
    d = gdn.make_dims(2, 2, 64, num_slots=8)
    for T in (0, 17):
        _expect(gdn, lambda: gdn.decode_verify(d, T, ins, fake, fake, fake, fake, stream=0),
                _abi.GDN_ERR_UNSUPPORTED)
    for flag in (gdn.KLOG_FP32, gdn.ULOG_BF16, gdn.KLOG_PRENORM):
        dd = gdn.make_dims(2, 2, 64, num_slots=8, flags=flag)
        _expect(gdn, lambda: gdn.decode_verify(dd, 4, ins, fake, fake, fake, fake, stream=0),
                _abi.GDN_ERR_UNSUPPORTED)
    # the fused conv needs mixed_qkv, conv_w and the window pool, 16-byte aligned
    dc = gdn.make_dims(2, 2, 64, num_slots=8, flags=gdn.FUSE_CONV | gdn.QKV_BF16)
    _expect(gdn, lambda: gdn.decode_verify(dc, 4, ins, fake, fake, fake, fake, stream=0),
            _abi.GDN_ERR_INVALID_ARG)
    cins = gdn.make_inputs(mixed_qkv=fake + 2, conv_w=fake, conv_pool=fake, log_decay=fake)
    _expect(gdn, lambda: gdn.decode_verify(dc, 4, cins, fake, fake, fake, fake, stream=0),
            _abi.GDN_ERR_UNSUPPORTED)
    _expect(gdn, lambda: gdn.decode_verify(d, 4, ins, None, fake, fake, fake, stream=0), _abi.GDN_ERR_INVALID_ARG)
    _expect(gdn, lambda: gdn.decode_verify(d, 4, gdn.make_inputs(q=fake, k=fake, v=fake), fake, fake, fake,
                                           fake, stream=0), _abi.GDN_ERR_INVALID_ARG)
    _expect(gdn, lambda: gdn.decode_verify(d, 4, ins, fake, fake, fake + 4, fake, stream=0),
            _abi.GDN_ERR_UNSUPPORTED)
    # an empty batch is a no-op
    gdn.decode_verify(gdn.make_dims(0, 2, 64, num_slots=8), 4, ins, fake, fake, fake, fake, stream=0)


def test_prefill_validation_rejects_before_launch(gdn):
    from linear_attention_decode_gdn_gb300 import _abi
    fake = 1 << 20  # never dereferenced: every call below fails validation first
    ok = gdn.make_inputs(q=fake, k=fake, v=fake, log_decay=fake, slot=fake)
    d = gdn.make_dims(2, 2, 64, num_slots=8)
    _expect(gdn, lambda: gdn.prefill(d, -1, ok, fake, fake, stream=0), _abi.GDN_ERR_INVALID_ARG)
    for flag in (gdn.KLOG_FP32, gdn.ULOG_BF16, gdn.KLOG_PRENORM):
        dd = gdn.make_dims(2, 2, 64, num_slots=8, flags=flag)
        _expect(gdn, lambda: gdn.prefill(dd, 8, ok, fake, fake, stream=0), _abi.GDN_ERR_UNSUPPORTED)
    # required inputs: slot, log_decay, and q/k/v or (with the fused conv) mixed_qkv, conv_w, conv_pool
    _expect(gdn, lambda: gdn.prefill(d, 8, gdn.make_inputs(q=fake, k=fake, v=fake, log_decay=fake), fake, fake,
                                     stream=0), _abi.GDN_ERR_INVALID_ARG)
    _expect(gdn, lambda: gdn.prefill(d, 8, gdn.make_inputs(q=fake, k=fake, log_decay=fake, slot=fake), fake, fake,
                                     stream=0), _abi.GDN_ERR_INVALID_ARG)
    dc = gdn.make_dims(2, 2, 64, num_slots=8, flags=gdn.FUSE_CONV | gdn.QKV_BF16)
    _expect(gdn, lambda: gdn.prefill(dc, 8, ok, fake, fake, stream=0), _abi.GDN_ERR_INVALID_ARG)
    mis = gdn.make_inputs(mixed_qkv=fake + 2, conv_w=fake, conv_pool=fake, log_decay=fake, slot=fake)
    _expect(gdn, lambda: gdn.prefill(dc, 8, mis, fake, fake, stream=0), _abi.GDN_ERR_UNSUPPORTED)
    # the KDA gate needs A_log and dt_bias; the output epilogue needs the gate logits
    dk = gdn.make_dims(2, 2, 64, num_slots=8, flags=gdn.GATE_KDA)
    _expect(gdn, lambda: gdn.prefill(dk, 8, ok, fake, fake, stream=0), _abi.GDN_ERR_INVALID_ARG)
    de = gdn.make_dims(2, 2, 64, num_slots=8, flags=gdn.OUT_NORM_GATE)
    _expect(gdn, lambda: gdn.prefill(de, 8, ok, fake, fake, stream=0), _abi.GDN_ERR_INVALID_ARG)
    # pools: present and 16-byte aligned
    _expect(gdn, lambda: gdn.prefill(d, 8, ok, None, fake, stream=0), _abi.GDN_ERR_INVALID_ARG)
    _expect(gdn, lambda: gdn.prefill(d, 8, ok, fake + 4, fake, stream=0), _abi.GDN_ERR_UNSUPPORTED)
    # head sizes other than 16/32/64/128 are not built
    _expect(gdn, lambda: gdn.prefill(gdn.make_dims(2, 2, 96, num_slots=8), 8, ok, fake, fake, stream=0),
            _abi.GDN_ERR_UNSUPPORTED)
    # an empty batch or an empty prompt is a no-op
    gdn.prefill(gdn.make_dims(0, 2, 64, num_slots=8), 8, ok, fake, fake, stream=0)
    gdn.prefill(d, 0, ok, fake, fake, stream=0)


def test_pools_shapes(gdn):
    """Pools.allocate sizes every pool as include/gdn.h documents it (device-independent)."""
    import torch
    d = gdn.make_dims(3, 2, 16, num_slots=5, flags=gdn.QKV_BF16, log_capacity=3, decay_per_key=True)
    p = gdn.Pools.allocate(d, device="cpu", conv=True, deltalog=True)
    assert tuple(p.state.shape) == (5, 2, 16, 16) and p.state.dtype == torch.float32
    assert tuple(p.conv.shape) == (5, 3 * 2 * 16, 3) and p.conv.dtype == torch.bfloat16
    assert tuple(p.k_log.shape) == (5, 2, 3, 16) and p.k_log.dtype == torch.bfloat16
    assert tuple(p.u_log.shape) == (5, 2, 3, 16) and p.u_log.dtype == torch.float32
    assert tuple(p.lam_log.shape) == (5, 2, 3, 16) and tuple(p.ell.shape) == (5, 2, 16)
    assert tuple(p.length.shape) == (5, 2) and p.length.dtype == torch.int32
    v = gdn.Pools.allocate(gdn.make_dims(3, 2, 16, num_slots=5), device="cpu", conv=True, verify_tokens=4)
    assert tuple(v.conv.shape) == (5, 96, 6) and v.conv.dtype == torch.float32
    r = gdn.Pools.allocate(gdn.make_dims(3, 2, 16, num_slots=5, flags=gdn.ULOG_BF16 | gdn.KLOG_FP32,
                                         log_capacity=2), device="cpu", deltalog=True)
    assert r.u_log.dtype == torch.bfloat16 and r.k_log.dtype == torch.float32


def test_binding_constants_match_the_header():
    """Every return code, status bit and flag #defined in include/gdn.h has the same value in
    the Python binding (the binding copies them; this catches drift)."""
    from linear_attention_decode_gdn_gb300 import _abi
    text = open(HEADER).read()
    defs = {}
    for name, expr in re.findall(r"^#define (GDN_\w+) ([^/\n]+)", text, flags=re.M):
        expr = expr.strip()
        m = re.fullmatch(r"\(1u << (\d+)\)", expr)
        if m:
            defs[name] = 1 << int(m.group(1))
        elif re.fullmatch(r"(0x[0-9a-fA-F]+|\d+)u?", expr):
            defs[name] = int(expr.rstrip("u"), 0)
    assert len(defs) >= 20, sorted(defs)
    for name, value in defs.items():
        if name in ("GDN_H", "GDN_API_VERSION"):
            continue
        py = name[len("GDN_"):]
        assert hasattr(_abi, py) or hasattr(_abi, name), name
        assert getattr(_abi, py, getattr(_abi, name, None)) == value, (name, value)
