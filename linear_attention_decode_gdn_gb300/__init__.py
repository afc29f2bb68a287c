"""GB300-native batched Gated-DeltaNet decode (dense and DeltaLog append-merge).

The compute runs in libgdn (``csrc/``, hand-written sm_103a CUDA kernels
behind the C ABI in ``include/gdn.h``). This package adds a ctypes binding with
the same names (``decode``), a build script (``build``) and seeded synthetic
workloads (``workloads``). Importing the package does not load the library; the
first call does, and raises if it has not been built.
"""
from . import _abi  # noqa: F401
from ._abi import (FUSE_CONV, GATE_RAW, KLOG_FP32, KLOG_PRENORM, NO_QK_L2NORM,  # noqa: F401
                   PLAIN_UPDATE, QKV_BF16, STATUS_BAD_LEN, STATUS_BAD_SLOT, STATUS_LOG_FULL,
                   STATUS_TIMEOUT, TEST_STARVE_WAIT, ULOG_BF16, GATE_KDA, OUT_NORM_GATE, SPLIT_DV, GDNError)
from .decode import (Pools, conv_l2norm, decode_append, decode_dense, decode_merge,  # noqa: F401
                     decode_step, decode_verify, log_bytes, make_dims, make_inputs, make_log, prefill,
                     slot_reset)
