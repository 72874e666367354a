"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every entry point
that include/mla.h declares, sizes workspaces, and rejects bad arguments before any launch."""
import ctypes
import os
import re

import pytest

import mla_latent_kv_75_b300 as mla
import mla_inputs as mi

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "mla.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_expected_entry_points():
    names = declared_functions()
    for n in ("mla_append_cache", "mla_project_q", "mla_decode_absorbed", "mla_prefill",
              "mla_decode_workspace_size", "mla_prefill_workspace_size",
              "mla_project_q_workspace_size", "mla_get_device_status", "mla_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = mla.lib()
    for n in declared_functions():
        assert hasattr(lib, n), n


def v2_dims(dtype=mla.MLA_BF16, **kw):
    d = mi.V2
    return mla.make_dims(d.d, d.n_h, d.d_hc, d.d_hr, d.d_c, d.d_cq, dtype, **kw)


def test_workspace_queries_are_host_only_and_monotone():
    d = v2_dims()
    a = mla.mla_decode_workspace_size(d, 16, 4096)
    b = mla.mla_decode_workspace_size(d, 128, 8193)
    assert 0 < a < b
    assert mla.mla_prefill_workspace_size(d, 8192, 2, 4096) > 0
    assert mla.mla_project_q_workspace_size(d, 16) > 0
    assert mla.mla_decode_workspace_size(d, 0, 0) >= 0


def test_status_strings():
    assert mla.mla_status_string(0) == "ok"
    for code in range(1, 9):
        assert mla.mla_status_string(code) not in ("ok", "unknown status")


@pytest.mark.parametrize("field,value,code", [
    ("n_h", 0, 1), ("d_hr", 63, 2), ("dtype", 7, 1), ("rope_base", 0.0, 1), ("d_c", -2, 1)])
def test_bad_dims_rejected(field, value, code):
    d = v2_dims()
    setattr(d, field, value)
    out = ctypes.c_size_t(0)
    st = mla.raw_status("mla_decode_workspace_size", ctypes.byref(d), 4, 128, ctypes.byref(out))
    assert st == code


def test_null_and_misaligned_pointers_rejected_without_launch():
    d = v2_dims()
    w = mla.MlaWeights()
    cache = mla.MlaCache(0x10000, 0x20000, 100)
    # null h
    st = mla.raw_status("mla_append_cache", ctypes.byref(d), ctypes.byref(w), None, 0x100, 0x200,
                        4, ctypes.byref(cache), None)
    assert st == mla.MLAError(1, "").status
    # misaligned h
    st = mla.raw_status("mla_append_cache", ctypes.byref(d), ctypes.byref(w), 0x1002, 0x100, 0x200,
                        4, ctypes.byref(cache), None)
    assert st == 4
    # aligned h but missing weights -> invalid argument
    st = mla.raw_status("mla_append_cache", ctypes.byref(d), ctypes.byref(w), 0x1000, 0x100, 0x200,
                        4, ctypes.byref(cache), None)
    assert st == 1
    # workspace too small for decode
    w2 = mla.MlaWeights(None, None, None, None, None, 0x3000, 0x4000)
    st = mla.raw_status("mla_decode_absorbed", ctypes.byref(d), ctypes.byref(w2), 0x5000, 0x6000,
                        ctypes.byref(cache), 0x7000, 2, 64, 0x8000, 16, 0x9000, None)
    assert st == 7
    # negative sizes
    st = mla.raw_status("mla_prefill", ctypes.byref(d), ctypes.byref(w), 0x1000, 0x100, -1, 4, 4,
                        ctypes.byref(cache), 0x8000, 1 << 30, 0x9000, None)
    assert st == 1


def test_zero_sized_calls_are_no_ops():
    d = v2_dims()
    w = mla.MlaWeights()
    cache = mla.MlaCache(None, None, 0)
    assert mla.raw_status("mla_append_cache", ctypes.byref(d), ctypes.byref(w), None, None, None,
                          0, ctypes.byref(cache), None) == 0
    assert mla.raw_status("mla_decode_absorbed", ctypes.byref(d), ctypes.byref(w), None, None,
                          ctypes.byref(cache), None, 0, 0, None, 0, None, None) == 0


def test_wait_timeout_hook_checks_its_limit_on_the_host():
    assert mla.raw_status("mla_debug_arm_wait_timeout", ctypes.c_int64(0)) == 1
    assert mla.raw_status("mla_debug_arm_wait_timeout", ctypes.c_int64(3_000_000_000)) == 1


def test_sparse_entry_points_validate_on_the_host():
    """Argument checks of the top-k selection and the sparse decode happen before any launch:
    k out of range, a score stride below max_len, misaligned scores, B = 0 as a no-op."""
    d = v2_dims()
    w = mla.MlaWeights()
    cache = mla.MlaCache(None, None, 0)
    sel = mla.raw_status
    # k < 1 and k above 2^20
    assert sel("mla_select_topk", 0x1000, ctypes.c_int64(64), 0x2000, 1, 64, 0, 0x3000, 0x4000,
               None) == 1
    assert sel("mla_select_topk", 0x1000, ctypes.c_int64(64), 0x2000, 1, 64, (1 << 20) + 1,
               0x3000, 0x4000, None) == 1
    # stride below max_len
    assert sel("mla_select_topk", 0x1000, ctypes.c_int64(32), 0x2000, 1, 64, 8, 0x3000, 0x4000,
               None) == 1
    # scores not 4-byte aligned
    assert sel("mla_select_topk", 0x1002, ctypes.c_int64(64), 0x2000, 1, 64, 8, 0x3000, 0x4000,
               None) == 4
    # nothing to do
    assert sel("mla_select_topk", None, ctypes.c_int64(0), None, 0, 0, 8, None, None, None) == 0
    assert sel("mla_decode_absorbed_sparse", ctypes.byref(d), ctypes.byref(w), None, None,
               ctypes.byref(cache), None, 0, 0, None, ctypes.c_int64(0), 8, None, 0, None,
               None) == 0
    assert sel("mla_decode_absorbed_sparse", ctypes.byref(d), ctypes.byref(w), None, None,
               ctypes.byref(cache), None, 1, 0, None, ctypes.c_int64(0), 0, None, 0, None,
               None) == 1
    # workspace: grows with B and k, and holds at least the packed rows
    a = mla.mla_decode_sparse_workspace_size(d, 16, 2048)
    b = mla.mla_decode_sparse_workspace_size(d, 16, 4096)
    assert 16 * 2048 * 1152 < a < b


def test_every_kernel_id_has_a_trace_name():
    """The launch-trace names cover every kernel id the library records, and only those."""
    names = [mla.mla_kernel_name(i) for i in range(64)]
    known = [n for n in names if n != "unknown"]
    assert known == names[:len(known)], "ids are contiguous from 0"
    assert len(set(known)) == len(known), "names are unique"
    for n in ("down", "q_absorb", "decode_attn", "unabsorb", "topk_select", "gather_rows",
              "prefill_attn", "out_proj"):
        assert n in known
    assert mla.mla_kernel_name(-1) == "unknown"
