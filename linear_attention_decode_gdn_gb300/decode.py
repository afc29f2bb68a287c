"""Python entry points with the C-ABI's names, taking torch tensors.

Each function only gathers device pointers, the current CUDA stream and the
``gdn_dims`` description, then calls the matching ``gdn_*`` function of
libgdn; the arithmetic runs in the CUDA kernels. PyTorch supplies device memory
and streams; :class:`Pools` allocates the slot-indexed state, conv and log
pools with it.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

from . import _abi
from ._abi import Dims, Inputs, Log, LogSizes, check


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def make_dims(batch, num_heads, dk, dv=None, num_slots=None, *, decay_per_key=False,
              log_capacity=0, flags=0, q_scale=1.0, l2_eps=1e-6, gate_lower_bound=-5.0,
              out_eps=1e-6) -> Dims:
    dv = dk if dv is None else dv
    num_slots = batch if num_slots is None else num_slots
    return Dims(batch, num_heads, dk, dv, num_slots, int(bool(decay_per_key)), log_capacity, flags,
                q_scale, l2_eps, gate_lower_bound, out_eps)


def make_inputs(*, q=None, k=None, v=None, mixed_qkv=None, conv_w=None, conv_b=None,
                conv_pool=None, log_decay=None, beta=None, slot=None, a_log=None, dt_bias=None,
                out_gate=None, out_norm_w=None) -> Inputs:
    inputs = Inputs(_ptr(q), _ptr(k), _ptr(v), _ptr(mixed_qkv), _ptr(conv_w), _ptr(conv_b),
                    _ptr(conv_pool), _ptr(log_decay), _ptr(beta), _ptr(slot), _ptr(a_log),
                    _ptr(dt_bias), _ptr(out_gate), _ptr(out_norm_w))
    # the struct keeps the tensors alive for as long as it holds their addresses
    inputs._keep = (q, k, v, mixed_qkv, conv_w, conv_b, conv_pool, log_decay, beta, slot, a_log,
                    dt_bias, out_gate, out_norm_w)
    return inputs


def make_log(k_log=None, u_log=None, lam_log=None, ell=None, length=None) -> Log:
    log = Log(_ptr(k_log), _ptr(u_log), _ptr(lam_log), _ptr(ell), _ptr(length))
    log._keep = (k_log, u_log, lam_log, ell, length)
    return log


def conv_l2norm(dims: Dims, inputs: Inputs, q_out, k_out, v_out, status=None, stream=None):
    lib = _abi.load()
    check(lib.gdn_conv_l2norm(ctypes.byref(dims), ctypes.byref(inputs), _ptr(q_out), _ptr(k_out),
                              _ptr(v_out), _ptr(status), _stream(stream)), "gdn_conv_l2norm")


def decode_dense(dims: Dims, inputs: Inputs, state_pool, o, status=None, stream=None):
    lib = _abi.load()
    check(lib.gdn_decode_dense(ctypes.byref(dims), ctypes.byref(inputs), _ptr(state_pool), _ptr(o),
                               _ptr(status), _stream(stream)), "gdn_decode_dense")


def _log_call(name, dims, inputs, base_pool, log, o, status, stream):
    lib = _abi.load()
    fn = getattr(lib, name)
    check(fn(ctypes.byref(dims), ctypes.byref(inputs), _ptr(base_pool), ctypes.byref(log), _ptr(o),
             _ptr(status), _stream(stream)), name)


def decode_append(dims, inputs, base_pool, log, o, status=None, stream=None):
    _log_call("gdn_decode_append", dims, inputs, base_pool, log, o, status, stream)


def decode_merge(dims, inputs, base_pool, log, o, status=None, stream=None):
    _log_call("gdn_decode_merge", dims, inputs, base_pool, log, o, status, stream)


def decode_step(dims, inputs, base_pool, log, o, status=None, stream=None):
    _log_call("gdn_decode_step", dims, inputs, base_pool, log, o, status, stream)


def decode_verify(dims: Dims, num_tokens: int, inputs: Inputs, state_indices, num_accepted, state_pool, o,
                  status=None, stream=None):
    """Speculative-decoding verify: num_tokens positions per request through the dense
    step; the state after position t goes to pool row state_indices[b, t]; the initial
    state is row state_indices[b, num_accepted[b] - 1]. Inputs [B, T, H, d], o [B, T, H, dv]."""
    lib = _abi.load()
    check(lib.gdn_decode_verify(ctypes.byref(dims), int(num_tokens), ctypes.byref(inputs), _ptr(state_indices),
                                _ptr(num_accepted), _ptr(state_pool), _ptr(o), _ptr(status), _stream(stream)),
          "gdn_decode_verify")


def prefill(dims: Dims, num_tokens: int, inputs: Inputs, state_pool, o, seq_lens=None, status=None,
            stream=None):
    """Chunked prefill: the prompt positions [B, T, H, d] through the recurrence from each
    request's pool row; the final state is written back there. o [B, T, H, dv]."""
    lib = _abi.load()
    check(lib.gdn_prefill(ctypes.byref(dims), int(num_tokens), ctypes.byref(inputs), _ptr(seq_lens),
                          _ptr(state_pool), _ptr(o), _ptr(status), _stream(stream)), "gdn_prefill")


def log_bytes(dims: Dims) -> dict:
    lib = _abi.load()
    out = LogSizes()
    check(lib.gdn_log_bytes(ctypes.byref(dims), ctypes.byref(out)), "gdn_log_bytes")
    return {name: getattr(out, name) for name, _ in LogSizes._fields_}


def slot_reset(dims: Dims, slots, n: int, log: Log | None = None, conv_pool=None, state_pool=None,
               status=None, stream=None):
    lib = _abi.load()
    check(lib.gdn_slot_reset(ctypes.byref(dims), ctypes.byref(log) if log is not None else None,
                             _ptr(conv_pool), _ptr(state_pool), _ptr(slots), int(n), _ptr(status),
                             _stream(stream)), "gdn_slot_reset")


@dataclass
class Pools:
    """Slot-indexed device pools for one layer (allocated with torch, zero-filled)."""
    state: object
    conv: object | None
    k_log: object | None
    u_log: object | None
    lam_log: object | None
    ell: object | None
    length: object | None

    @classmethod
    def allocate(cls, dims: Dims, device="cuda", conv=False, deltalog=False, verify_tokens=None):
        """conv: the conv cache [slots][channels][3] (decode, prefill); with verify_tokens = T
        instead the widened window [slots][channels][T + 2] of gdn_decode_verify."""
        import torch
        S, H, dk, dv = dims.num_slots, dims.num_heads, dims.dk, dims.dv
        dlam = dk if dims.decay_per_key else 1
        C = dims.log_capacity
        state = torch.zeros((S, H, dk, dv), dtype=torch.float32, device=device)
        conv_pool = None
        if conv:
            ch = 2 * H * dk + H * dv
            cdt = torch.bfloat16 if dims.flags & _abi.QKV_BF16 else torch.float32
            width = 3 if verify_tokens is None else int(verify_tokens) + 2
            conv_pool = torch.zeros((S, ch, width), dtype=cdt, device=device)
        k_log = u_log = lam_log = ell = length = None
        if deltalog:
            kdt = torch.float32 if dims.flags & _abi.KLOG_FP32 else torch.bfloat16
            c = max(C, 1)
            k_log = torch.zeros((S, H, c, dk), dtype=kdt, device=device)
            udt = torch.bfloat16 if dims.flags & _abi.ULOG_BF16 else torch.float32
            u_log = torch.zeros((S, H, c, dv), dtype=udt, device=device)
            lam_log = torch.zeros((S, H, c, dlam), dtype=torch.float32, device=device)
            ell = torch.zeros((S, H, dlam), dtype=torch.float32, device=device)
            length = torch.zeros((S, H), dtype=torch.int32, device=device)
        return cls(state, conv_pool, k_log, u_log, lam_log, ell, length)

    def log(self) -> Log:
        return make_log(self.k_log, self.u_log, self.lam_log, self.ell, self.length)
