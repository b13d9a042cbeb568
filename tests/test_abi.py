"""The C-ABI library loads and exports every entry point include/*.h declares (CPU only).

No compute call is made: the library is loaded and its symbols are resolved.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(h2o_\w+)\s*\(", src))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from h2o_heavy_hitter_gb300 import _build
    path = _build.build()
    return ctypes.CDLL(str(path))


def test_header_declares_entry_points():
    names = _declared()
    for n in ("h2o_create", "h2o_prefill", "h2o_decode_step", "h2o_cache_positions",
              "h2o_destroy", "h2o_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_last_error_is_callable_without_gpu(lib):
    lib.h2o_last_error.restype = ctypes.c_char_p
    assert lib.h2o_last_error() == b""


def test_null_context_calls_fail_cleanly_without_gpu(lib):
    """Argument checks run before any CUDA call."""
    lib.h2o_cache_dims.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    assert lib.h2o_cache_dims(None, None, None) == -1
    lib.h2o_create.argtypes = [ctypes.c_int] * 6 + [ctypes.c_void_p]
    out = ctypes.c_void_p()
    assert lib.h2o_create(1, 1, 1, 96, 1, 1, ctypes.byref(out)) == -1
    assert out.value is None


def test_misaligned_prompt_buffers_are_rejected_without_gpu(lib):
    """TMA needs 16-byte aligned prompt tensors and outputs; the check runs
    before any CUDA call (the addresses are never dereferenced)."""
    lib.h2o_last_error.restype = ctypes.c_char_p
    for fn, n_tail in ((lib.h2o_prefill_attention, 2), (lib.h2o_prefill_attention_noalloc, 3)):
        fn.restype = ctypes.c_int
        fn.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + [ctypes.c_void_p] * n_tail
    good, bad = 0x10000, 0x10004
    assert lib.h2o_prefill_attention(good, good, good, 2, 256, 128, bad, good) == -1
    assert b"16-byte aligned" in lib.h2o_last_error()
    assert lib.h2o_prefill_attention_noalloc(bad, good, good, 2, 256, 128, good, good, None) == -1
    assert b"16-byte aligned" in lib.h2o_last_error()


def test_new_entry_points_check_arguments_without_gpu(lib):
    """Argument checks of the ragged prefill, the multi-step decode, the ring
    layout and the failure probe run before any CUDA call."""
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.h2o_last_error.restype = ctypes.c_char_p
    lib.h2o_prefill_ragged.argtypes = [P, I, P, P, P, I, P, P]
    assert lib.h2o_prefill_ragged(None, 0, None, None, None, 16, None, None) == -1
    assert b"null lens" in lib.h2o_last_error()
    fake = 0x10000  # never dereferenced: the context check fails first
    assert lib.h2o_prefill_ragged(None, 0, fake, fake, fake, 16, fake, fake) == -1
    assert b"null context" in lib.h2o_last_error()
    lib.h2o_decode_steps.argtypes = [P, I, I, P, P, P, P, P]
    assert lib.h2o_decode_steps(None, 0, 4, None, None, None, None, None) == -1
    lib.h2o_test_wait_limit.argtypes = [P]
    assert lib.h2o_test_wait_limit(None) == -1
    lib.h2o_create_ex.argtypes = [I] * 7 + [ctypes.POINTER(P)]
    out = P()
    ring = 0x100
    assert lib.h2o_create_ex(1, 1, 1, 64, 4, 0, ring, ctypes.byref(out)) == -1  # no window
    assert b"H2O_LAYOUT_RING" in lib.h2o_last_error()
    assert lib.h2o_create_ex(1, 1, 1, 64, 4, 4, 1 | ring, ctypes.byref(out)) == -1  # FP8 + ring
    assert lib.h2o_create_ex(1, 1, 1, 64, 4, 4, 7, ctypes.byref(out)) == -1  # unknown format
    assert out.value is None


def test_state_and_fault_entry_points_check_arguments_without_gpu(lib):
    """h2o_reset, the allocation-failure hook and the device-state reset run
    their argument checks (or touch only host state) without any CUDA call."""
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.h2o_last_error.restype = ctypes.c_char_p
    lib.h2o_reset.argtypes = [P, I]
    assert lib.h2o_reset(None, 0) == -1 and b"null context" in lib.h2o_last_error()
    lib.h2o_test_fail_allocations.argtypes = [I]
    assert lib.h2o_test_fail_allocations(-1) == -1
    assert lib.h2o_test_fail_allocations(0) == 0
    lib.h2o_forget_device_state.restype = None
    lib.h2o_forget_device_state()
