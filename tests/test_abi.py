"""CPU-side checks of the C-ABI library: it builds for sm_103a, loads, exports
every entry point declared in include/pagedattn.h, and rejects bad arguments
on the host before any CUDA work (no GPU needed)."""
import ctypes

import pytest

from paged_gqa_decode_02_gb300 import build as pbuild
from paged_gqa_decode_02_gb300 import binding as B


@pytest.fixture(scope="module")
def lib():
    pbuild.build()
    return B.lib()


def test_header_declares_the_four_core_calls():
    syms = B.header_symbols()
    for s in ("pa_create_pool", "pa_append_kv", "pa_decode", "pa_destroy"):
        assert s in syms


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(B.LIB_PATH)
    missing = [s for s in B.header_symbols() if not hasattr(raw, s)]
    assert not missing, missing


def test_status_strings(lib):
    for code in range(7):
        assert lib.pa_status_string(code)
    assert lib.pa_status_string(99) == b"unknown status"


def test_create_pool_rejects_bad_descriptors_without_a_gpu(lib):
    h = ctypes.c_void_p()
    bad = [dict(num_blocks=0), dict(num_kv_heads=0), dict(block_size=8), dict(head_dim=96),
           dict(kv_dtype=7), dict(device=-1)]
    for over in bad:
        kw = dict(num_blocks=4, block_size=16, num_kv_heads=2, head_dim=64, kv_dtype=0, device=0)
        kw.update(over)
        d = B.pa_pool_desc(**kw)
        st = lib.pa_create_pool(ctypes.byref(d), ctypes.byref(h))
        assert st in (1, 2), (over, st)
        assert h.value is None
        assert lib.pa_last_error()
    assert lib.pa_create_pool(None, ctypes.byref(h)) == 1


def test_null_pool_arguments(lib):
    assert lib.pa_decode(None, None, None, None, 1, 4, 1, 1.0, None, None, 0, 0, None) == 1
    assert lib.pa_append_kv(None, None, None, None, None, None, 1, 1, 0, None) == 1
    assert lib.pa_decode_workspace_bytes(None, 1, 4, 0) == 0
    assert lib.pa_destroy(None) == 0
    assert lib.pa_pool_set_unit_cost(None, 0) == 1
    assert lib.pa_decode_multi(None, None, None, None, 1, 2, 4, 1, 1.0, None, None, 0, 0, None) == 1
    assert lib.pa_decode_multi_workspace_bytes(None, 1, 2, 4, 0) == 0
    f = ctypes.c_uint32()
    assert lib.pa_get_device_error(None, None, ctypes.byref(f)) == 1
    i = (ctypes.c_int32 * 1)(0)
    assert lib.pa_copy_blocks(None, i, i, 1, None) == 1
    assert lib.pa_swap_blocks(None, i, 1, i, i, 1, 0, None) == 1
    assert lib.pa_pool_block_bytes(None) == 0
    assert lib.pa_selftest_wait_timeout(0, 0, ctypes.byref(f)) == 1  # refused before any launch
    assert lib.pa_selftest_wait_timeout(0, 1000, None) == 1
    # the calibration read refuses null, misaligned or ragged arguments before any launch
    assert lib.pa_stream_read(None, 16, ctypes.byref(f), None) == 1
    assert lib.pa_stream_read(ctypes.c_void_p(16), 16, None, None) == 1
    assert lib.pa_stream_read(ctypes.c_void_p(8), 16, ctypes.byref(f), None) == 1
    assert lib.pa_stream_read(ctypes.c_void_p(16), 24, ctypes.byref(f), None) == 1


def test_null_block_manager_arguments(lib):
    i = (ctypes.c_int32 * 4)()
    n = ctypes.c_int32()
    assert lib.pa_bm_create(0, 16, 1, ctypes.byref(ctypes.c_void_p())) == 1
    assert lib.pa_bm_create(4, 16, 1, None) == 1
    assert lib.pa_bm_destroy(None) == 0
    assert lib.pa_bm_add_sequence(None, 1, None, 0, None) == 1
    assert lib.pa_bm_fork(None, 1, 2) == 1
    assert lib.pa_bm_append_tokens(None, 1, None, 1, i, i, 1, ctypes.byref(n)) == 1
    assert lib.pa_bm_free_sequence(None, 1) == 1
    assert lib.pa_bm_block_table(None, 1, i, 4, None, None) == 1
    assert lib.pa_bm_num_free_blocks(None) == 0 and lib.pa_bm_ref_count(None, 0) == -1
    assert lib.pa_bm_set_cpu_blocks(None, 4) == 1 and lib.pa_bm_num_free_cpu_blocks(None) == 0
    assert lib.pa_bm_swap_out(None, 1, i, i, 4, ctypes.byref(n)) == 1
    assert lib.pa_bm_swap_in(None, 1, i, i, 4, ctypes.byref(n)) == 1
    assert lib.pa_bm_swapped_slots(None, 1, i, 4, ctypes.byref(n)) == 1
