"""ctypes view of include/gdn.h: structs, constants and the loaded library.

Argument marshalling only; every step of the decode path runs in libgdn's
kernels. The library is loaded lazily from ``_build/libgdn.so`` next to this
file; if it is missing, the first call raises instead of falling back to
anything else.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libgdn.so")

# return codes
GDN_OK = 0
GDN_ERR_INVALID_ARG = 1
GDN_ERR_UNSUPPORTED = 2
GDN_ERR_CUDA = 3

# device status bits
STATUS_BAD_SLOT = 0x1
STATUS_LOG_FULL = 0x2
STATUS_BAD_LEN = 0x4
STATUS_TIMEOUT = 0x8

# flags
QKV_BF16 = 1 << 0
FUSE_CONV = 1 << 1
NO_QK_L2NORM = 1 << 2
GATE_RAW = 1 << 3
PLAIN_UPDATE = 1 << 4
KLOG_FP32 = 1 << 5
KLOG_PRENORM = 1 << 6
ULOG_BF16 = 1 << 7
GATE_KDA = 1 << 8
OUT_NORM_GATE = 1 << 9
SPLIT_DV = 1 << 10
TEST_STARVE_WAIT = 1 << 31

# every symbol include/gdn.h declares
EXPORTS = ("gdn_version", "gdn_strerror", "gdn_last_error", "gdn_conv_l2norm", "gdn_decode_dense",
           "gdn_decode_append", "gdn_decode_merge", "gdn_decode_step", "gdn_decode_verify",
           "gdn_prefill", "gdn_log_bytes", "gdn_slot_reset")


class Dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_heads", ctypes.c_int32), ("dk", ctypes.c_int32),
                ("dv", ctypes.c_int32), ("num_slots", ctypes.c_int32),
                ("decay_per_key", ctypes.c_int32), ("log_capacity", ctypes.c_int32),
                ("flags", ctypes.c_uint32), ("q_scale", ctypes.c_float), ("l2_eps", ctypes.c_float),
                ("gate_lower_bound", ctypes.c_float), ("out_eps", ctypes.c_float)]


class Inputs(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("mixed_qkv", ctypes.c_void_p), ("conv_w", ctypes.c_void_p),
                ("conv_b", ctypes.c_void_p), ("conv_pool", ctypes.c_void_p),
                ("log_decay", ctypes.c_void_p), ("beta", ctypes.c_void_p), ("slot", ctypes.c_void_p),
                ("a_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p), ("out_gate", ctypes.c_void_p),
                ("out_norm_w", ctypes.c_void_p)]


class Log(ctypes.Structure):
    _fields_ = [("k_log", ctypes.c_void_p), ("u_log", ctypes.c_void_p), ("lam_log", ctypes.c_void_p),
                ("ell", ctypes.c_void_p), ("len", ctypes.c_void_p)]


class LogSizes(ctypes.Structure):
    _fields_ = [("k_log", ctypes.c_size_t), ("u_log", ctypes.c_size_t), ("lam_log", ctypes.c_size_t),
                ("ell", ctypes.c_size_t), ("len", ctypes.c_size_t), ("residency", ctypes.c_size_t),
                ("total", ctypes.c_size_t)]


_lock = threading.Lock()
_lib = None


def _declare(lib):
    P = ctypes.POINTER
    vp = ctypes.c_void_p
    lib.gdn_version.restype = ctypes.c_int
    lib.gdn_version.argtypes = []
    lib.gdn_strerror.restype = ctypes.c_char_p
    lib.gdn_strerror.argtypes = [ctypes.c_int]
    lib.gdn_last_error.restype = ctypes.c_char_p
    lib.gdn_last_error.argtypes = []
    lib.gdn_conv_l2norm.restype = ctypes.c_int
    lib.gdn_conv_l2norm.argtypes = [P(Dims), P(Inputs), vp, vp, vp, vp, vp]
    lib.gdn_decode_dense.restype = ctypes.c_int
    lib.gdn_decode_dense.argtypes = [P(Dims), P(Inputs), vp, vp, vp, vp]
    for name in ("gdn_decode_append", "gdn_decode_merge", "gdn_decode_step"):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int
        fn.argtypes = [P(Dims), P(Inputs), vp, P(Log), vp, vp, vp]
    lib.gdn_decode_verify.restype = ctypes.c_int
    lib.gdn_decode_verify.argtypes = [P(Dims), ctypes.c_int32, P(Inputs), vp, vp, vp, vp, vp, vp]
    lib.gdn_prefill.restype = ctypes.c_int
    lib.gdn_prefill.argtypes = [P(Dims), ctypes.c_int32, P(Inputs), vp, vp, vp, vp, vp]
    lib.gdn_log_bytes.restype = ctypes.c_int
    lib.gdn_log_bytes.argtypes = [P(Dims), P(LogSizes)]
    lib.gdn_slot_reset.restype = ctypes.c_int
    lib.gdn_slot_reset.argtypes = [P(Dims), P(Log), vp, vp, vp, ctypes.c_int32, vp, vp]
    return lib


def load(path: str | None = None):
    """Returns the loaded libgdn (raises RuntimeError if it was not built)."""
    global _lib
    with _lock:
        if _lib is None or path is not None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(
                    f"libgdn is not built ({p} missing); run "
                    "`python -m linear_attention_decode_gdn_gb300.build` (needs nvcc)")
            lib = _declare(ctypes.CDLL(p))
            if path is not None:
                return lib
            _lib = lib
        return _lib


class GDNError(RuntimeError):
    def __init__(self, code: int, where: str, message: str):
        self.code = code
        super().__init__(f"{where}: error {code} ({message})")


def check(rc: int, where: str) -> None:
    if rc != GDN_OK:
        lib = load()
        msg = lib.gdn_last_error().decode() or lib.gdn_strerror(rc).decode()
        raise GDNError(rc, where, msg)
