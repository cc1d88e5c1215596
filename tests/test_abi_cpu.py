"""The C-ABI library loads and exports every entry point include/gdn.h declares;
host-side argument checks answer without touching a GPU."""
import ctypes
import os
import re

import pytest

import hybrid_linear_attention_gdn_gb300 as gdn
from hybrid_linear_attention_gdn_gb300 import _build, binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "gdn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return gdn.load()


def test_header_declares_the_hot_path_calls():
    names = _declared_functions()
    for must in ["gdn_decode_step", "gdn_spec_verify", "gdn_spec_commit", "gdn_chunk_prefill",
                 "gdn_chunk_prefill_workspace_size", "gdn_slot_copy", "gdn_slot_zero"]:
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
    assert set(_declared_functions()) == set(binding.EXPORTS)


def test_status_strings(lib):
    assert lib.gdn_status_string(0) == b"GDN_OK"
    assert lib.gdn_status_string(1) == b"GDN_ERR_INVALID_ARG"
    assert lib.gdn_status_string(2) == b"GDN_ERR_UNSUPPORTED"
    assert lib.gdn_status_string(3) == b"GDN_ERR_CUDA"
    assert lib.gdn_status_string(99) == b"GDN_UNKNOWN_STATUS"


def _dims(**kw):
    d = dict(hk=16, hv=32, dk=128, dv=128, conv_width=4, act_dtype=1, conv_dtype=1)
    d.update(kw)
    return binding.CDims(**d)


def test_workspace_size_is_host_only(lib):
    d = _dims()
    n = lib.gdn_chunk_prefill_workspace_size(ctypes.byref(d), 4, 32768)
    # q^, k^ [T][16][128], v [T][32][128], g and beta [T][32], fp32, 256-aligned parts
    assert n == 4 * 32768 * (2 * 16 * 128 + 32 * 128 + 2 * 32)
    assert lib.gdn_chunk_prefill_workspace_size(ctypes.byref(d), 4, 0) == 0
    bad = _dims(dk=48)
    assert lib.gdn_chunk_prefill_workspace_size(ctypes.byref(bad), 4, 10) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(hv=30), binding.ERR_INVALID_ARG),       # hv not a multiple of hk
    (dict(hk=0), binding.ERR_INVALID_ARG),
    (dict(act_dtype=7), binding.ERR_INVALID_ARG),
    (dict(dk=32), binding.ERR_UNSUPPORTED),
    (dict(dv=512), binding.ERR_UNSUPPORTED),
    (dict(conv_width=9), binding.ERR_UNSUPPORTED),
    (dict(act_dtype=0, conv_dtype=1), binding.ERR_UNSUPPORTED),  # f32 in, bf16 history
])
def test_dims_rejected_before_any_launch(lib, kw, status):
    d = _dims(**kw)
    pool = binding.CPool(None, None, 0)
    p = binding.CParams(None, None, None)
    n0 = lib.gdn_launch_count(binding.K_DECODE)
    st = lib.gdn_decode_step(ctypes.byref(d), pool, ctypes.byref(p), None, 4, None, None, None,
                             None, None, None)
    assert st == status
    assert lib.gdn_slot_zero(ctypes.byref(d), pool, None, 3, None, None) == status
    assert lib.gdn_launch_count(binding.K_DECODE) == n0


def test_null_and_negative_arguments(lib):
    d = _dims()
    pool = binding.CPool(None, None, 0)
    p = binding.CParams(None, None, None)
    assert lib.gdn_decode_step(None, pool, ctypes.byref(p), None, 1, None, None, None, None,
                               None, None) == binding.ERR_INVALID_ARG
    assert lib.gdn_decode_step(ctypes.byref(d), pool, ctypes.byref(p), None, -1, None, None,
                               None, None, None, None) == binding.ERR_INVALID_ARG
    # batch 0 is a no-op and launches nothing
    assert lib.gdn_decode_step(ctypes.byref(d), pool, ctypes.byref(p), None, 0, None, None, None,
                               None, None, None) == binding.OK
    # a pool with slots but no memory
    pool2 = binding.CPool(None, None, 4)
    assert lib.gdn_slot_zero(ctypes.byref(d), pool2, None, 1, None, None) == binding.ERR_INVALID_ARG
    # misaligned state pointer
    pool3 = binding.CPool(0x1004, 0x2000, 4)
    assert lib.gdn_slot_copy(ctypes.byref(d), pool3, pool3, 0x100, 0x200, 1, None,
                             None) == binding.ERR_INVALID_ARG
    # verify: T out of range
    assert lib.gdn_spec_verify(ctypes.byref(d), pool, pool, ctypes.byref(p), None, None, 1, 0,
                               None, None, None, None, None, None) == binding.ERR_INVALID_ARG
    assert lib.gdn_spec_verify(ctypes.byref(d), pool, pool, ctypes.byref(p), None, None, 1, 17,
                               None, None, None, None, None, None) == binding.ERR_UNSUPPORTED
    # prefill: checkpoint block must be a multiple of the 64-token chunk
    assert lib.gdn_chunk_prefill(ctypes.byref(d), pool, pool, ctypes.byref(p), None, None, None,
                                 1, 10, None, 0, 100, None, None, None, None, None, 0, None,
                                 None) == binding.ERR_INVALID_ARG
    assert lib.gdn_chunk_prefill(ctypes.byref(d), pool, pool, ctypes.byref(p), None, None, None,
                                 0, 0, None, 0, 256, None, None, None, None, None, 0, None,
                                 None) == binding.OK


def test_state_record_and_index_commit_arguments(lib):
    d = _dims()
    # SSM fp32 [32][128][128] + conv history bf16 [3][2*16*128 + 32*128]
    rec = 32 * 128 * 128 * 4 + 3 * (2 * 16 * 128 + 32 * 128) * 2
    assert lib.gdn_state_record_bytes(ctypes.byref(d)) == rec
    assert lib.gdn_state_record_bytes(ctypes.byref(_dims(dk=48))) == 0
    assert lib.gdn_state_record_bytes(None) == 0
    pool = binding.CPool(0x10000, 0x20000, 4)
    n0 = lib.gdn_launch_count(binding.K_STATE_PACK)
    # staging one byte short of one record, misaligned, or absent
    assert lib.gdn_state_pack(ctypes.byref(d), pool, 0x100, 1, 0x40000, rec - 1, None,
                              None) == binding.ERR_INVALID_ARG
    assert lib.gdn_state_unpack(ctypes.byref(d), 0x40008, 4 * rec, pool, 0x100, 1, None,
                                None) == binding.ERR_INVALID_ARG
    assert lib.gdn_state_pack(ctypes.byref(d), pool, 0x100, 1, None, 4 * rec, None,
                              None) == binding.ERR_INVALID_ARG
    assert lib.gdn_state_pack(ctypes.byref(d), pool, 0x100, -1, 0x40000, 4 * rec, None,
                              None) == binding.ERR_INVALID_ARG
    assert lib.gdn_state_unpack(ctypes.byref(d), 0x40000, 0, pool, None, 0, None,
                                None) == binding.OK
    assert lib.gdn_launch_count(binding.K_STATE_PACK) == n0
    n0 = lib.gdn_launch_count(binding.K_COMMIT_INDEX)
    assert lib.gdn_spec_commit_index(0x100, 0x200, 0x300, 0x400, 4, 0, None,
                                     None) == binding.ERR_INVALID_ARG
    assert lib.gdn_spec_commit_index(None, 0x200, 0x300, 0x400, 4, 2, None,
                                     None) == binding.ERR_INVALID_ARG
    assert lib.gdn_spec_commit_index(None, None, None, None, 0, 2, None, None) == binding.OK
    assert lib.gdn_launch_count(binding.K_COMMIT_INDEX) == n0


def test_mixed_step_arguments(lib):
    d = _dims()
    pool = binding.CPool(0x10000, 0x20000, 4)
    p = binding.CParams(0x1000, 0x2000, 0x3000)
    args = lambda n_seq, n_dec, total, blk=256: (  # noqa: E731
        ctypes.byref(d), pool, pool, ctypes.byref(p), 0x100, 0x200, 0x300, n_seq, n_dec, total,
        None, 0, blk, 0x400, 0x500, 0x600, 0x700, 0x800, 1 << 30, None, None)
    n_dec0 = lib.gdn_launch_count(binding.K_DECODE)
    n_pre0 = lib.gdn_launch_count(binding.K_PREFILL)
    assert lib.gdn_mixed_step(*args(2, 3, 10)) == binding.ERR_INVALID_ARG   # n_decode > n_seq
    assert lib.gdn_mixed_step(*args(4, 3, 2)) == binding.ERR_INVALID_ARG    # n_decode > tokens
    assert lib.gdn_mixed_step(*args(4, -1, 10)) == binding.ERR_INVALID_ARG
    # the prefill half is checked before the decode half launches
    assert lib.gdn_mixed_step(*args(4, 2, 10, blk=100)) == binding.ERR_INVALID_ARG
    assert lib.gdn_mixed_step(*args(0, 0, 0)) == binding.OK
    assert lib.gdn_launch_count(binding.K_DECODE) == n_dec0
    assert lib.gdn_launch_count(binding.K_PREFILL) == n_pre0


def test_kda_prefill_arguments(lib):
    d = _dims()
    pool = binding.CPool(0x10000, 0x20000, 4)
    p = binding.CParams(0x1000, 0x2000, 0x3000)
    args = lambda n_seq, total, blk=256, params=p, slots=0x100: (  # noqa: E731
        ctypes.byref(d), pool, pool, ctypes.byref(params) if params else None, slots, 0x200, 0x300, n_seq,
        total, None, 0, blk, 0x400, 0x500, 0x600, 0x700, None, None)
    n0 = lib.gdn_launch_count(binding.K_KDA_PREFILL)
    assert lib.gdn_kda_prefill(*args(2, 10, blk=100)) == binding.ERR_INVALID_ARG  # block not a multiple of 64
    assert lib.gdn_kda_prefill(*args(2, 10, blk=0)) == binding.ERR_INVALID_ARG
    assert lib.gdn_kda_prefill(*args(-1, 10)) == binding.ERR_INVALID_ARG
    assert lib.gdn_kda_prefill(*args(2, -1)) == binding.ERR_INVALID_ARG
    assert lib.gdn_kda_prefill(*args(70000, 10)) == binding.ERR_UNSUPPORTED
    assert lib.gdn_kda_prefill(*args(2, 10, params=None)) == binding.ERR_INVALID_ARG
    assert lib.gdn_kda_prefill(*args(2, 10, slots=None)) == binding.ERR_INVALID_ARG
    assert lib.gdn_kda_prefill(*args(0, 0)) == binding.OK
    assert lib.gdn_launch_count(binding.K_KDA_PREFILL) == n0


def test_gated_rmsnorm_arguments(lib):
    d = _dims()
    n0 = lib.gdn_launch_count(binding.K_GATED_RMSNORM)
    call = lambda n, eps, o=0x100, z=0x200, w=0x300, y=0x400: lib.gdn_gated_rmsnorm(  # noqa: E731
        ctypes.byref(d), o, z, w, eps, n, y, None)
    assert call(-1, 1e-6) == binding.ERR_INVALID_ARG
    assert call(4, -1.0) == binding.ERR_INVALID_ARG
    assert call(4, float("nan")) == binding.ERR_INVALID_ARG
    assert call(4, 1e-6, w=None) == binding.ERR_INVALID_ARG
    assert call(0, 1e-6) == binding.OK
    assert lib.gdn_gated_rmsnorm(None, 0x100, 0x200, 0x300, 1e-6, 4, 0x400, None) == binding.ERR_INVALID_ARG
    assert lib.gdn_launch_count(binding.K_GATED_RMSNORM) == n0


def test_selftest_needs_an_error_word(lib):
    assert lib.gdn_selftest_wait_timeout(None, None) == binding.ERR_INVALID_ARG


def test_launch_counters(lib):
    lib.gdn_launch_count_reset()
    assert all(lib.gdn_launch_count(k) == 0 for k in range(binding.K_COUNT))
    assert lib.gdn_launch_count(-1) == 0 and lib.gdn_launch_count(99) == 0


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "library_path", lambda: str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="libgdn.so not found"):
        binding.load()


def test_normal_library_has_no_bounds_checks(lib):
    """The bounds words and their positive control belong to the checked build
    (libgdn_debug.so); the normal library answers GDN_ERR_UNSUPPORTED from the
    host, launching nothing."""
    count = ctypes.c_uint32(7)
    assert lib.gdn_debug_bounds_take(ctypes.byref(count), None, 0, None, None) == binding.ERR_UNSUPPORTED
    assert lib.gdn_selftest_bounds(None) == binding.ERR_UNSUPPORTED


def test_checked_library_is_selected_by_the_environment(monkeypatch):
    monkeypatch.setenv("GDN_DEBUG_BOUNDS", "1")
    assert binding.library_path() == _build.LIB_DEBUG
    monkeypatch.setenv("GDN_DEBUG_BOUNDS", "0")
    assert binding.library_path() == _build.LIB
