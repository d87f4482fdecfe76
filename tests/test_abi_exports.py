"""The C-ABI library builds, loads without a GPU, and exports every entry
point include/pagedkv.h declares (no compute calls here)."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "pagedkv.h")).read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char \*)\s*(pa_\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("pa_kv_append_rope", "pa_decode_attention", "pa_decode_workspace_size", "pa_free"):
        assert n in names


def test_library_exports_every_declared_symbol():
    import paged_kv_cache_205_gb300 as pk
    lib = pk.library()
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing
    assert pk.pa_error_string(-4).startswith("workspace")


def test_host_validation_without_a_device():
    """Argument checks run before any CUDA call: bad sizes and layers are
    refused with their codes even on a machine without a GPU."""
    import ctypes
    import paged_kv_cache_205_gb300 as pk
    lib = pk.library()
    P = ctypes.c_void_p
    z = P(0)
    assert lib.pa_decode_attention(z, z, z, 1, z, 2, 4, z, 3, 2, 0.125, z, 0, z, z) == -3
    assert lib.pa_decode_attention(z, z, z, 1, z, 2, 4, z, -1, 0, 0.125, z, 0, z, z) == -2
    assert lib.pa_decode_attention(z, z, z, 1, z, 2, 4, z, 0, 0, 0.125, z, 0, z, z) == 0
    assert lib.pa_decode_attention(z, z, z, 1, z, 2, 4, z, 3, 0, 0.125, z, 0, z, z) == -1
    assert lib.pa_kv_append_rope(z, z, z, z, 8, z, 1, 4, z, 2, 1, z, z, z, z) == -3
    assert lib.pa_kv_append_rope(z, z, z, z, 8, z, 1, 4, z, 2, 0, z, z, z, z) == -1
    assert lib.pa_free(z, 0, z, 1, 4, z, z, z, 8, z, z) == 0
    assert lib.pa_free(z, 2, z, 1, 4, z, z, z, 8, z, z) == -1
    assert lib.pa_decode_set_grid_limit(-1) == -2
    assert lib.pa_decode_set_grid_limit(0) == 0
    # the bounded-wait test hook: a stage >= -1 and a limit of 1 us .. 1 s
    assert lib.pa_decode_set_test_fault(-2, 0) == -2
    assert lib.pa_decode_set_test_fault(0, 10) == -2
    assert lib.pa_decode_set_test_fault(0, 2_000_000_000) == -2
    assert lib.pa_decode_set_test_fault(0, 50_000) == 0
    assert lib.pa_decode_set_test_fault(-1, 0) == 0
    # the prefill kernel's bounded-wait hook: a chunk >= -1 and a limit of 1 us .. 1 s
    assert lib.pa_prefill_set_test_fault(-2, 0) == -2
    assert lib.pa_prefill_set_test_fault(0, 10) == -2
    assert lib.pa_prefill_set_test_fault(0, 2_000_000_000) == -2
    assert lib.pa_prefill_set_test_fault(0, 50_000) == 0
    assert lib.pa_prefill_set_test_fault(-1, 0) == 0
    # the speculative-plan test hook: modes 0 and 1 only
    assert lib.pa_decode_set_test_plan(2) == -2 and lib.pa_decode_set_test_plan(-1) == -2
    assert lib.pa_decode_set_test_plan(1) == 0 and lib.pa_decode_set_test_plan(0) == 0


def test_decode_path_switch_without_a_device():
    """The kernel choice: only the three path values are accepted; 8-token
    pages take the split kernel unless the per-head kernel is forced; the
    per-sequence kernel takes 16-token pages only (8 and 32 fall back to the
    split kernel), the per-head kernel 8, 16 or 32; a forced path is
    reported as is; a bad count or page size is refused."""
    import paged_kv_cache_205_gb300 as pk
    lib = pk.library()
    assert lib.pa_decode_set_path(4) == -2 and lib.pa_decode_set_path(-1) == -2
    try:
        assert lib.pa_decode_kernel_for(-1, 16) == -2
        assert lib.pa_decode_kernel_for(4, 12) == -2
        assert lib.pa_decode_kernel_for(4, 8) == pk.PA_DECODE_SPLIT
        assert lib.pa_decode_set_path(pk.PA_DECODE_SPLIT) == 0
        assert lib.pa_decode_kernel_for(4, 16) == pk.PA_DECODE_SPLIT
        assert lib.pa_decode_kernel_for(4, 32) == pk.PA_DECODE_SPLIT
        assert lib.pa_decode_set_path(pk.PA_DECODE_CLUSTER) == 0
        assert lib.pa_decode_kernel_for(4, 16) == pk.PA_DECODE_CLUSTER
        assert lib.pa_decode_kernel_for(4, 32) == pk.PA_DECODE_CLUSTER
        assert lib.pa_decode_kernel_for(4, 8) == pk.PA_DECODE_CLUSTER
        assert lib.pa_decode_set_path(pk.PA_DECODE_SEQ) == 0
        assert lib.pa_decode_kernel_for(4, 16) == pk.PA_DECODE_SEQ
        assert lib.pa_decode_kernel_for(4, 32) == pk.PA_DECODE_SPLIT
        assert lib.pa_decode_kernel_for(4, 8) == pk.PA_DECODE_SPLIT
    finally:
        assert lib.pa_decode_set_path(pk.PA_DECODE_AUTO) == 0


def test_length_aware_choice_without_a_device():
    """pa_decode_kernel_for_lengths checks its arguments before it asks for a
    device: a negative count, a null length array with sequences, or a page
    size other than 8, 16 or 32 is refused; an empty batch and 8-token pages
    take the split-context kernel whatever the lengths."""
    import ctypes
    import paged_kv_cache_205_gb300 as pk
    lib = pk.library()
    z = ctypes.c_void_p(0)
    lens = (ctypes.c_int32 * 3)(5, 700, 3000)
    assert lib.pa_decode_kernel_for_lengths(z, -1, 16) == -2
    assert lib.pa_decode_kernel_for_lengths(z, 3, 16) == -2
    assert lib.pa_decode_kernel_for_lengths(lens, 3, 12) == -2
    assert lib.pa_decode_kernel_for_lengths(lens, 3, 64) == -2
    assert lib.pa_decode_kernel_for_lengths(z, 0, 16) == pk.PA_DECODE_SPLIT
    assert lib.pa_decode_kernel_for_lengths(lens, 3, 8) == pk.PA_DECODE_SPLIT
    assert pk.pa_decode_kernel_for_lengths([], 32) == pk.PA_DECODE_SPLIT
    with pytest.raises(pk.PagedKVError):
        pk.pa_decode_kernel_for_lengths([1, 2], 24)


def test_page_size_entry_points_refuse_other_sizes():
    """Only 8-, 16- and 32-token pages are built; anything else is refused
    before any CUDA call."""
    import ctypes
    import paged_kv_cache_205_gb300 as pk
    lib = pk.library()
    z = ctypes.c_void_p(0)
    assert lib.pa_decode_attention_bt(z, z, z, 4, 12, z, 1, 4, z, 1, 0, 0.125, z, 0, z, z) == -2
    assert lib.pa_kv_append_rope_bt(z, z, z, z, 4, 64, z, 1, 4, z, 1, 0, z, z, z, z) == -2
    assert lib.pa_free_bt(z, 1, 4, z, 1, 4, z, z, z, 4, z, z) == -2
    assert lib.pa_decode_workspace_size_bt(4, 4, 24) == 0
    assert pk.pa_decode_workspace_size(4, 4, 8) > 0
