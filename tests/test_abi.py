"""The C-ABI library loads and exports every symbol include/moe.h declares (CPU).

No compute call is made; only argument validation that the library performs
on the host before touching a device.
"""
import ctypes
import os
import re

import pytest

import int4_routed_expert_decode_gb300 as moe
from int4_routed_expert_decode_gb300 import build as moe_build


@pytest.fixture(scope="module")
def L():
    moe_build.build()
    return moe.lib()


def _declared(root):
    text = open(os.path.join(root, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L, root):
    names = _declared(root)
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(moe.EXPORTS)


def test_status_strings(L):
    assert moe.moe_status_string(0) == "ok"
    assert "slot" in moe.moe_status_string(moe.MOE_ERR_SLOT)
    assert "unknown" in moe.moe_status_string(12345)


@pytest.mark.parametrize("args,status", [
    ((0, 1, 256, 64, 64, 32), moe.MOE_ERR_UNSUPPORTED),     # E = 0
    ((16, 17, 256, 64, 64, 32), moe.MOE_ERR_INVALID_ARG),   # k > E
    ((16, 2, 300, 64, 64, 32), moe.MOE_ERR_UNSUPPORTED),    # hidden not a multiple of 256
    ((16, 2, 768, 64, 64, 32), moe.MOE_ERR_UNSUPPORTED),    # hidden / 256 not a power of two
    ((16, 2, 3072, 64, 64, 32), moe.MOE_ERR_UNSUPPORTED),   # the same
    ((16, 2, 256, 64, 64, 48), moe.MOE_ERR_UNSUPPORTED),    # group
    ((16, 2, 256, 80, 64, 32), moe.MOE_ERR_UNSUPPORTED),    # inter not a multiple of group
    ((2048, 8, 2048, 512, 512, 64), moe.MOE_ERR_UNSUPPORTED),  # E too large
])
def test_create_rejects_bad_sizes(L, args, status):
    out = ctypes.c_void_p()
    assert L.moe_create(*args, ctypes.byref(out)) == status
    assert out.value is None
    assert moe.moe_last_error(None)


def test_null_context_is_an_error_not_a_crash(L):
    assert L.moe_reserve(None, 4) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_forward(None, None, 1, None, None, None, None, None, None, None) == \
        moe.MOE_ERR_INVALID_ARG
    assert L.moe_get_status(None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_set_path(None, 0) == moe.MOE_ERR_INVALID_ARG
    L.moe_destroy(None)
    assert L.moe_expert_blob_bytes(None) == 0


def test_python_binding_names_match_c(L):
    for n in moe.EXPORTS:
        assert callable(getattr(moe, n)), n


@pytest.mark.parametrize("hidden", [768, 1280, 1536, 3072])
def test_static_routing_rejects_uninstantiated_hidden_up_front(L, hidden):
    """hidden sizes that no router kernel is built for are refused before any
    device call, with MOE_ERR_UNSUPPORTED (nothing is launched)."""
    rc = L.moe_route_static(None, 1, None, None, None, 16, 2, hidden, None, None, None, None)
    assert rc == moe.MOE_ERR_UNSUPPORTED
    assert "hidden" in moe.moe_last_error(None)


def test_stack_calls_reject_null_arguments(L):
    out = ctypes.c_void_p()
    assert L.moe_stack_create(None, 2, None, ctypes.c_float(1e-6), ctypes.byref(out)) == \
        moe.MOE_ERR_INVALID_ARG
    assert "layers" in moe.moe_last_error(None)
    assert L.moe_stack_create(None, 0, None, ctypes.c_float(1e-6), None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_stack_forward(None, None, None, None, None, None, None, None, None) == \
        moe.MOE_ERR_INVALID_ARG
    assert L.moe_stack_get_status(None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_stack_set_test_flags(None, 0) == moe.MOE_ERR_INVALID_ARG
    L.moe_stack_destroy(None)


def test_pool_calls_reject_null_arguments(L):
    assert L.moe_pool_enable(None, 4) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_pool_stats(None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_pool_table(None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_router_check_stats(None, None, None) == moe.MOE_ERR_INVALID_ARG


def test_gdn_recurrence_checks_arguments_before_any_launch(L):
    """Sizes and pointers are checked on the host (no GPU needed): empty calls
    succeed without touching anything; bad sizes are refused."""
    import int4_routed_expert_decode_gb300 as moe
    assert L.moe_gdn_recurrence(None, None, None, None, None, None, None,
                                0, 1, 2, 4, 128, 8, None) == moe.MOE_OK
    assert L.moe_gdn_recurrence(None, None, None, None, None, None, None,
                                1, 0, 2, 4, 128, 8, None) == moe.MOE_OK
    assert L.moe_gdn_recurrence(None, None, None, None, None, None, None,
                                1, 1, 3, 4, 128, 8, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_gdn_recurrence(None, None, None, None, None, None, None,
                                1, 1, 2, 4, 96, 8, None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_gdn_recurrence(None, None, None, None, None, None, None,
                                1, 1, 2, 4, 128, 8, None) == moe.MOE_ERR_INVALID_ARG
    assert b"NULL" in L.moe_last_error(None)


def test_create_quant_checks_bits_before_any_device_call(L):
    import int4_routed_expert_decode_gb300 as moe
    out = ctypes.c_void_p()
    for bits in (0, 2, 3, 5, 16):
        assert L.moe_create_quant(16, 2, 256, 64, 64, 32, bits, ctypes.byref(out)) == \
            moe.MOE_ERR_UNSUPPORTED
        assert b"bits" in L.moe_last_error(None)
