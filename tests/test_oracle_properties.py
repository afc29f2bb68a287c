"""Property-based runs of the oracle's pins (CPU): the pins of test_oracle_pins.py with shapes,
lengths and seeds drawn by hypothesis instead of fixed, so an index or boundary mistake that
one fixed shape happens to hide still fails somewhere. Each property is one of the pins'
reference computations: the DeltaLog emulation against the dense recurrence (DeltaLog notes,
Eq. (7), Algorithm 1, Eq. (6)); the recurrence against the WY/UT chunked form (evolution
article, "完整计算顺序"); the widened verify conv window against brute force over the
accepted history (inference handbook, "推测解码：验证后如何恢复状态")."""
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import test_oracle_pins as pins  # noqa: E402

SETTINGS = dict(max_examples=60, deadline=None, derandomize=True)


@settings(**SETTINGS)
@given(dk=st.integers(1, 9), dv=st.integers(1, 9), T=st.integers(1, 17), seed=st.integers(0, 2 ** 16))
def test_deltalog_emulation_equals_dense(oracle_lib, dk, dv, T, seed):
    pins.pin_deltalog_equals_dense(oracle_lib, B=3, H=2, dk=dk, dv=dv, T=T, seed=seed)


@settings(**SETTINGS)
@given(T=st.integers(1, 50), dk=st.integers(2, 12), dv=st.integers(2, 12), C=st.sampled_from([4, 8, 16]),
       per_key=st.booleans(), seed=st.integers(0, 2 ** 16))
def test_recurrence_equals_wy_chunked(oracle_lib, T, dk, dv, C, per_key, seed):
    pins.pin_delta_wy(oracle_lib, T=T, dk=dk, dv=dv, C=C, per_key=per_key, seed=seed)


@settings(**SETTINGS)
@given(nch=st.integers(1, 7), T=st.integers(1, 6), rounds=st.integers(1, 8), seed=st.integers(0, 2 ** 16))
def test_verify_conv_window_against_brute_force(oracle_lib, nch, T, rounds, seed):
    pins.pin_verify_conv_window(oracle_lib, nch=nch, T=T, rounds=rounds, seed=seed)
