"""Thin ctypes binding over libgdn.so (argument marshalling only).

Each function has the name of the C entry point it wraps, minus the ``gdn_``
prefix, takes torch tensors, passes their ``data_ptr()`` and the current CUDA
stream, and raises :class:`GdnError` on a non-OK status.  All arithmetic runs
in the library's kernels; there is no fallback: if the library is missing the
first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

from . import _build

F32, BF16 = 0, 1
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_SCRATCH_LIMIT = 0, 1, 2, 3, 4
DEV_ERR_SLOT_OOB, DEV_ERR_TIMEOUT, DEV_ERR_SEQLENS = 1, 2, 4
(K_DECODE, K_SPEC_VERIFY, K_SLOT_COPY, K_SLOT_ZERO, K_SPEC_COMMIT, K_PREFILL, K_COMMIT_INDEX,
 K_STATE_PACK, K_GATED_RMSNORM, K_KDA_DECODE, K_KDA_VERIFY, K_KDA_PREFILL, K_MIXED) = range(13)
K_COUNT = 13

_DT_CODE = {torch.float32: F32, torch.bfloat16: BF16}

_lock = threading.Lock()
_lib = None


class GdnError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: {msg} ({status})")
        self.status = status


class CDims(ctypes.Structure):
    _fields_ = [("hk", ctypes.c_int32), ("hv", ctypes.c_int32), ("dk", ctypes.c_int32),
                ("dv", ctypes.c_int32), ("conv_width", ctypes.c_int32),
                ("act_dtype", ctypes.c_int32), ("conv_dtype", ctypes.c_int32)]


class CPool(ctypes.Structure):
    _fields_ = [("ssm", ctypes.c_void_p), ("conv", ctypes.c_void_p),
                ("num_slots", ctypes.c_int32)]


class CParams(ctypes.Structure):
    _fields_ = [("conv_w", ctypes.c_void_p), ("A_log", ctypes.c_void_p),
                ("dt_bias", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_PD = ctypes.POINTER(CDims)
_PP = ctypes.POINTER(CParams)

EXPORTS = {
    "gdn_decode_step": ([_PD, CPool, _PP, _P, _I32, _P, _P, _P, _P, _P, _P], _I32),
    "gdn_kda_decode_step": ([_PD, CPool, _PP, _P, _I32, _P, _P, _P, _P, _P, _P], _I32),
    "gdn_kda_spec_verify": ([_PD, CPool, CPool, _PP, _P, _P, _I32, _I32, _P, _P, _P, _P, _P, _P], _I32),
    "gdn_spec_verify": ([_PD, CPool, CPool, _PP, _P, _P, _I32, _I32, _P, _P, _P, _P, _P, _P], _I32),
    "gdn_spec_commit": ([_PD, CPool, CPool, _P, _P, _P, _I32, _I32, _P, _P], _I32),
    "gdn_kda_prefill": ([_PD, CPool, CPool, _PP, _P, _P, _P, _I32, _I64, _P, _I32, _I32, _P, _P, _P,
                         _P, _P, _P], _I32),
    "gdn_chunk_prefill_workspace_size": ([_PD, _I32, _I64], ctypes.c_size_t),
    "gdn_chunk_prefill": ([_PD, CPool, CPool, _PP, _P, _P, _P, _I32, _I64, _P, _I32, _I32,
                           _P, _P, _P, _P, _P, ctypes.c_size_t, _P, _P], _I32),
    "gdn_chunk_prefill_gated": ([_PD, CPool, CPool, _PP, _P, _P, _P, _I32, _I64, _P, _I32, _I32,
                                 _P, _P, _P, _P, _P, ctypes.c_float, _P, _P, ctypes.c_size_t, _P, _P], _I32),
    "gdn_chunk_prefill_noalloc": ([_PD, CPool, CPool, _PP, _P, _P, _P, _I32, _I64, _P, _I32,
                                   _I32, _P, _P, _P, _P, _P, _P], _I32),
    "gdn_mixed_step": ([_PD, CPool, CPool, _PP, _P, _P, _P, _I32, _I32, _I64, _P, _I32, _I32, _P, _P,
                        _P, _P, _P, ctypes.c_size_t, _P, _P], _I32),
    "gdn_slot_copy": ([_PD, CPool, CPool, _P, _P, _I32, _P, _P], _I32),
    "gdn_slot_zero": ([_PD, CPool, _P, _I32, _P, _P], _I32),
    "gdn_spec_commit_index": ([_P, _P, _P, _P, _I32, _I32, _P, _P], _I32),
    "gdn_state_record_bytes": ([_PD], ctypes.c_size_t),
    "gdn_state_pack": ([_PD, CPool, _P, _I32, _P, ctypes.c_size_t, _P, _P], _I32),
    "gdn_state_unpack": ([_PD, _P, ctypes.c_size_t, CPool, _P, _I32, _P, _P], _I32),
    "gdn_gated_rmsnorm": ([_PD, _P, _P, _P, ctypes.c_float, _I64, _P, _P], _I32),
    "gdn_selftest_wait_timeout": ([_P, _P], _I32),
    "gdn_status_string": ([_I32], ctypes.c_char_p),
    "gdn_launch_count": ([_I32], ctypes.c_uint64),
    "gdn_launch_count_reset": ([], None),
    "gdn_selftest_bounds": ([_P], _I32),
    "gdn_debug_bounds_take": ([ctypes.POINTER(ctypes.c_uint32), ctypes.c_char_p, ctypes.c_size_t,
                               ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)], _I32),
}


def debug_bounds() -> bool:
    """GDN_DEBUG_BOUNDS=1 selects the bounds-checked library, libgdn_debug.so."""
    return os.environ.get("GDN_DEBUG_BOUNDS") == "1"


def library_path() -> str:
    return _build.LIB_DEBUG if debug_bounds() else _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libgdn.so (optionally building it first).  Raises if absent."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if build_if_missing:
                _build.build(debug_bounds=debug_bounds())
            if not os.path.exists(path):
                raise RuntimeError(
                    f"libgdn.so not found at {path}: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            lib = ctypes.CDLL(path)
            for name, (argtypes, restype) in EXPORTS.items():
                fn = getattr(lib, name)
                fn.argtypes = argtypes
                fn.restype = restype
            _lib = lib
    return _lib


class BoundsError(RuntimeError):
    """A kernel of the bounds-checked library indexed outside a buffer."""


def debug_bounds_take():
    """Bounds-checked library only: wait for the device, read and clear the
    kernels' bounds words.  None when no check failed since the last call,
    else (count, "file:line kind", index, limit)."""
    count, idx, lim = ctypes.c_uint32(0), ctypes.c_int64(0), ctypes.c_int64(0)
    where = ctypes.create_string_buffer(256)
    st = load().gdn_debug_bounds_take(ctypes.byref(count), where, 256, ctypes.byref(idx), ctypes.byref(lim))
    if st != OK:
        raise GdnError("gdn_debug_bounds_take", st, load().gdn_status_string(st).decode())
    if count.value == 0:
        return None
    return count.value, where.value.decode(), idx.value, lim.value


def _check(fn: str, status: int):
    if status != OK:
        msg = load().gdn_status_string(status).decode()
        raise GdnError(fn, status, msg)
    # the checked library: every call is followed by a read of the bounds
    # words (not while a CUDA graph is being captured)
    if debug_bounds() and not torch.cuda.is_current_stream_capturing():
        bad = debug_bounds_take()
        if bad is not None:
            raise BoundsError(f"{fn}: {bad[0]} index check(s) failed, first at {bad[1]}: "
                              f"index {bad[2]} of {bad[3]}")


def _ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


# ---------------------------------------------------------------- structures

@dataclass(frozen=True)
class Dims:
    hk: int
    hv: int
    dk: int
    dv: int
    conv_width: int
    act_dtype: torch.dtype
    conv_dtype: torch.dtype

    @staticmethod
    def of(shape) -> "Dims":
        """From any object with hk, hv, dk, dv, w, act_dtype, conv_dtype."""
        return Dims(shape.hk, shape.hv, shape.dk, shape.dv, shape.w, shape.act_dtype,
                    shape.conv_dtype)

    @property
    def channels(self) -> int:
        return 2 * self.hk * self.dk + self.hv * self.dv

    def c(self) -> CDims:
        key = (self.hk, self.hv, self.dk, self.dv, self.conv_width, self.act_dtype, self.conv_dtype)
        cached = self.__dict__.get("_c")
        if cached is None or cached[0] != key:
            cached = (key, CDims(self.hk, self.hv, self.dk, self.dv, self.conv_width,
                                 _DT_CODE[self.act_dtype], _DT_CODE[self.conv_dtype]))
            self.__dict__["_c"] = cached
        return cached[1]


@dataclass
class StatePool:
    """Device pool: ssm [N][HV][DV][DK] fp32, conv [N][W-1][C]."""

    ssm: torch.Tensor
    conv: torch.Tensor

    @property
    def num_slots(self) -> int:
        return self.ssm.shape[0]

    def c(self) -> CPool:
        key = (self.ssm.data_ptr(), self.conv.data_ptr(), self.ssm.shape[0])
        cached = self.__dict__.get("_c")
        if cached is None or cached[0] != key:
            cached = (key, CPool(*key))
            self.__dict__["_c"] = cached
        return cached[1]

    @staticmethod
    def empty(dims: Dims, num_slots: int, device="cuda") -> "StatePool":
        ssm = torch.empty((num_slots, dims.hv, dims.dv, dims.dk), dtype=torch.float32, device=device)
        conv = torch.empty((num_slots, dims.conv_width - 1, dims.channels), dtype=dims.conv_dtype,
                           device=device)
        return StatePool(ssm, conv)


@dataclass
class LayerParams:
    conv_w: torch.Tensor   # [C][W] fp32
    A_log: torch.Tensor    # [HV] fp32
    dt_bias: torch.Tensor  # [HV] fp32

    def c(self) -> CParams:
        key = (self.conv_w.data_ptr(), self.A_log.data_ptr(), self.dt_bias.data_ptr())
        cached = self.__dict__.get("_c")
        if cached is None or cached[0] != key:
            cached = (key, CParams(*key))
            self.__dict__["_c"] = cached
        return cached[1]


# ---------------------------------------------------------------- entry points

def decode_step(dims: Dims, pool: StatePool, params: LayerParams, slot_ids, qkv, a, b, out,
                dev_err=None, stream=None):
    L = load()
    cd, cp = dims.c(), params.c()
    st = L.gdn_decode_step(ctypes.byref(cd), pool.c(), ctypes.byref(cp), _ptr(slot_ids),
                           int(slot_ids.shape[0]), _ptr(qkv), _ptr(a), _ptr(b), _ptr(out),
                           _ptr(dev_err), _stream(stream))
    _check("gdn_decode_step", st)


def kda_decode_step(dims: Dims, pool: StatePool, params: LayerParams, slot_ids, qkv, a, b, out,
                    dev_err=None, stream=None):
    """KDA decode: the gated delta rule with one decay per key channel; a is
    [B][hv][dk] gate logits and params.dt_bias [hv][dk]."""
    L = load()
    cd, cp = dims.c(), params.c()
    st = L.gdn_kda_decode_step(ctypes.byref(cd), pool.c(), ctypes.byref(cp), _ptr(slot_ids),
                               int(slot_ids.shape[0]), _ptr(qkv), _ptr(a), _ptr(b), _ptr(out),
                               _ptr(dev_err), _stream(stream))
    _check("gdn_kda_decode_step", st)


def kda_spec_verify(dims: Dims, work: StatePool, spec: StatePool, params: LayerParams, slot_ids,
                    spec_ids, qkv, a, b, out, dev_err=None, stream=None):
    """KDA speculative verify; a is [B][T][hv][dk], params.dt_bias [hv][dk]."""
    L = load()
    B, T = spec_ids.shape
    cd, cp = dims.c(), params.c()
    st = L.gdn_kda_spec_verify(ctypes.byref(cd), work.c(), spec.c(), ctypes.byref(cp), _ptr(slot_ids),
                               _ptr(spec_ids), int(B), int(T), _ptr(qkv), _ptr(a), _ptr(b), _ptr(out),
                               _ptr(dev_err), _stream(stream))
    _check("gdn_kda_spec_verify", st)


def spec_verify(dims: Dims, work: StatePool, spec: StatePool, params: LayerParams, slot_ids,
                spec_ids, qkv, a, b, out, dev_err=None, stream=None):
    L = load()
    B, T = spec_ids.shape
    cd, cp = dims.c(), params.c()
    st = L.gdn_spec_verify(ctypes.byref(cd), work.c(), spec.c(), ctypes.byref(cp),
                           _ptr(slot_ids), _ptr(spec_ids), int(B), int(T), _ptr(qkv), _ptr(a),
                           _ptr(b), _ptr(out), _ptr(dev_err), _stream(stream))
    _check("gdn_spec_verify", st)


def spec_commit(dims: Dims, spec: StatePool, work: StatePool, spec_ids, accept_len, slot_ids,
                dev_err=None, stream=None):
    L = load()
    B, T = spec_ids.shape
    cd = dims.c()
    st = L.gdn_spec_commit(ctypes.byref(cd), spec.c(), work.c(), _ptr(spec_ids),
                           _ptr(accept_len), _ptr(slot_ids), int(B), int(T), _ptr(dev_err),
                           _stream(stream))
    _check("gdn_spec_commit", st)


def chunk_prefill_workspace_size(dims: Dims, n_seq: int, total_tokens: int) -> int:
    cd = dims.c()
    return int(load().gdn_chunk_prefill_workspace_size(ctypes.byref(cd), int(n_seq),
                                                        int(total_tokens)))


def chunk_prefill(dims: Dims, pool: StatePool, ckpt: StatePool, params: LayerParams, slot_ids,
                  cu_seqlens, start_pos, total_tokens: int, ckpt_ids, ckpt_block: int, qkv, a, b,
                  out, workspace, dev_err=None, stream=None):
    L = load()
    n_seq = int(slot_ids.shape[0])
    max_ckpt = int(ckpt_ids.shape[1]) if ckpt_ids is not None and ckpt_ids.dim() == 2 else 0
    cd, cp = dims.c(), params.c()
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = L.gdn_chunk_prefill(ctypes.byref(cd), pool.c(), ckpt.c(), ctypes.byref(cp),
                             _ptr(slot_ids), _ptr(cu_seqlens), _ptr(start_pos), n_seq,
                             int(total_tokens), _ptr(ckpt_ids), max_ckpt, int(ckpt_block),
                             _ptr(qkv), _ptr(a), _ptr(b), _ptr(out), _ptr(workspace), ws_bytes,
                             _ptr(dev_err), _stream(stream))
    _check("gdn_chunk_prefill", st)


def chunk_prefill_gated(dims: Dims, pool: StatePool, ckpt: StatePool, params: LayerParams, slot_ids,
                        cu_seqlens, start_pos, total_tokens: int, ckpt_ids, ckpt_block: int, qkv, a, b,
                        z, weight, eps: float, y, workspace, dev_err=None, stream=None):
    """chunk_prefill whose output is the gated RMS norm of the readout."""
    L = load()
    n_seq = int(slot_ids.shape[0])
    max_ckpt = int(ckpt_ids.shape[1]) if ckpt_ids is not None and ckpt_ids.dim() == 2 else 0
    cd, cp = dims.c(), params.c()
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = L.gdn_chunk_prefill_gated(ctypes.byref(cd), pool.c(), ckpt.c(), ctypes.byref(cp),
                                   _ptr(slot_ids), _ptr(cu_seqlens), _ptr(start_pos), n_seq,
                                   int(total_tokens), _ptr(ckpt_ids), max_ckpt, int(ckpt_block),
                                   _ptr(qkv), _ptr(a), _ptr(b), _ptr(z), _ptr(weight), float(eps), _ptr(y),
                                   _ptr(workspace), ws_bytes, _ptr(dev_err), _stream(stream))
    _check("gdn_chunk_prefill_gated", st)


def kda_prefill(dims: Dims, pool: StatePool, ckpt: StatePool, params: LayerParams, slot_ids, cu_seqlens,
                start_pos, total_tokens: int, ckpt_ids, ckpt_block: int, qkv, a, b, out, dev_err=None,
                stream=None):
    """KDA prefill: chunk_prefill's contract with per-key-channel gate logits
    a [total][hv][dk] and dt_bias [hv][dk]; it needs no workspace.  dk 128
    with dv <= 128 (dv % 4 == 0) runs the 16-token window form on the tensor
    cores, other shapes (or GDN_KDA_PREFILL_PATH=recurrent) the token
    recurrence; both keep fp32 accuracy."""
    L = load()
    n_seq = int(slot_ids.shape[0])
    max_ckpt = int(ckpt_ids.shape[1]) if ckpt_ids is not None and ckpt_ids.dim() == 2 else 0
    cd, cp = dims.c(), params.c()
    st = L.gdn_kda_prefill(ctypes.byref(cd), pool.c(), ckpt.c(), ctypes.byref(cp), _ptr(slot_ids),
                           _ptr(cu_seqlens), _ptr(start_pos), n_seq, int(total_tokens), _ptr(ckpt_ids),
                           max_ckpt, int(ckpt_block), _ptr(qkv), _ptr(a), _ptr(b), _ptr(out), _ptr(dev_err),
                           _stream(stream))
    _check("gdn_kda_prefill", st)


def selftest_wait_timeout(dev_err, stream=None):
    """Run the device-side failure-path self-test: a bounded wait that nothing
    satisfies expires after the library's wait limit and sets DEV_ERR_TIMEOUT
    in dev_err (an int32 device tensor)."""
    _check("gdn_selftest_wait_timeout", load().gdn_selftest_wait_timeout(_ptr(dev_err), _stream(stream)))


def selftest_bounds(stream=None):
    """Bounds-checked library only: launch the checks' positive control (three
    requests that must fail their checks, none of which can leave real
    memory).  The bounds words are left for debug_bounds_take()."""
    st = load().gdn_selftest_bounds(_stream(stream))
    if st != OK:
        raise GdnError("gdn_selftest_bounds", st, load().gdn_status_string(st).decode())


NOALLOC_SCRATCH_BYTES = 64 << 20


def chunk_prefill_noalloc(dims: Dims, pool: StatePool, ckpt: StatePool, params: LayerParams,
                          slot_ids, cu_seqlens, start_pos, total_tokens: int, ckpt_ids,
                          ckpt_block: int, qkv, a, b, out, dev_err=None, stream=None):
    """The same prefill as chunk_prefill, for callers that cannot allocate a
    device workspace (a host framework that owns all device memory and passes
    only input/output pointers, or a runtime that reserved its whole budget at
    start-up): it works in the library's built-in 64 MiB scratch buffer.
    Raises GdnError (ERR_SCRATCH_LIMIT) when a call needs more than that."""
    L = load()
    n_seq = int(slot_ids.shape[0])
    max_ckpt = int(ckpt_ids.shape[1]) if ckpt_ids is not None and ckpt_ids.dim() == 2 else 0
    cd, cp = dims.c(), params.c()
    st = L.gdn_chunk_prefill_noalloc(ctypes.byref(cd), pool.c(), ckpt.c(), ctypes.byref(cp),
                                     _ptr(slot_ids), _ptr(cu_seqlens), _ptr(start_pos), n_seq,
                                     int(total_tokens), _ptr(ckpt_ids), max_ckpt, int(ckpt_block),
                                     _ptr(qkv), _ptr(a), _ptr(b), _ptr(out), _ptr(dev_err),
                                     _stream(stream))
    _check("gdn_chunk_prefill_noalloc", st)


def mixed_step(dims: Dims, pool: StatePool, ckpt: StatePool, params: LayerParams, slot_ids,
               cu_seqlens, start_pos, total_tokens: int, n_decode: int, ckpt_ids, ckpt_block: int,
               qkv, a, b, out, workspace, dev_err=None, stream=None):
    """Decode-first mixed batch: sequences 0 .. n_decode-1 are single-token
    decode requests on rows 0 .. n_decode-1, the rest chunked-prefill
    continuations at their cu_seqlens offsets."""
    L = load()
    n_seq = int(slot_ids.shape[0])
    max_ckpt = int(ckpt_ids.shape[1]) if ckpt_ids is not None and ckpt_ids.dim() == 2 else 0
    cd, cp = dims.c(), params.c()
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = L.gdn_mixed_step(ctypes.byref(cd), pool.c(), ckpt.c(), ctypes.byref(cp), _ptr(slot_ids),
                          _ptr(cu_seqlens), _ptr(start_pos), n_seq, int(n_decode), int(total_tokens),
                          _ptr(ckpt_ids), max_ckpt, int(ckpt_block), _ptr(qkv), _ptr(a), _ptr(b),
                          _ptr(out), _ptr(workspace), ws_bytes, _ptr(dev_err), _stream(stream))
    _check("gdn_mixed_step", st)


def slot_copy(dims: Dims, src: StatePool, dst: StatePool, src_ids, dst_ids, dev_err=None,
              stream=None):
    L = load()
    cd = dims.c()
    st = L.gdn_slot_copy(ctypes.byref(cd), src.c(), dst.c(), _ptr(src_ids), _ptr(dst_ids),
                         int(src_ids.shape[0]), _ptr(dev_err), _stream(stream))
    _check("gdn_slot_copy", st)


def slot_zero(dims: Dims, pool: StatePool, ids, dev_err=None, stream=None):
    L = load()
    cd = dims.c()
    st = L.gdn_slot_zero(ctypes.byref(cd), pool.c(), _ptr(ids), int(ids.shape[0]), _ptr(dev_err),
                         _stream(stream))
    _check("gdn_slot_zero", st)


def spec_commit_index(spec_ids, accept_len, slot_ids, freed_ids, dev_err=None, stream=None):
    """Adopt the accepted snapshot by index: slot_ids is updated in place and
    freed_ids [B][T] receives the slots the caller returns to its allocator."""
    L = load()
    B, T = spec_ids.shape
    st = L.gdn_spec_commit_index(_ptr(spec_ids), _ptr(accept_len), _ptr(slot_ids),
                                 _ptr(freed_ids), int(B), int(T), _ptr(dev_err),
                                 _stream(stream))
    _check("gdn_spec_commit_index", st)


def state_record_bytes(dims: Dims) -> int:
    cd = dims.c()
    return int(load().gdn_state_record_bytes(ctypes.byref(cd)))


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def state_pack(dims: Dims, pool: StatePool, ids, staging, dev_err=None, stream=None):
    """Records of slots ids[i] into the byte buffer ``staging``."""
    L = load()
    cd = dims.c()
    st = L.gdn_state_pack(ctypes.byref(cd), pool.c(), _ptr(ids), int(ids.shape[0]),
                          _ptr(staging), _nbytes(staging), _ptr(dev_err), _stream(stream))
    _check("gdn_state_pack", st)


def state_unpack(dims: Dims, staging, pool: StatePool, ids, dev_err=None, stream=None):
    """Record i of ``staging`` into slot ids[i]."""
    L = load()
    cd = dims.c()
    st = L.gdn_state_unpack(ctypes.byref(cd), _ptr(staging), _nbytes(staging), pool.c(),
                            _ptr(ids), int(ids.shape[0]), _ptr(dev_err), _stream(stream))
    _check("gdn_state_unpack", st)


def gated_rmsnorm(dims: Dims, o, z, weight, eps: float = 1e-6, y=None, stream=None):
    """Readout epilogue y = o / sqrt(mean(o^2) + eps) * weight * silu(z) per
    (token, V head) row; o, z [n_tok][hv][dv] in the activation dtype, weight
    [dv] fp32.  y defaults to o (in place).  Returns y."""
    L = load()
    if y is None:
        y = o
    cd = dims.c()
    st = L.gdn_gated_rmsnorm(ctypes.byref(cd), _ptr(o), _ptr(z), _ptr(weight), float(eps),
                             int(o.shape[0]), _ptr(y), _stream(stream))
    _check("gdn_gated_rmsnorm", st)
    return y


def launch_count(kernel: int) -> int:
    return int(load().gdn_launch_count(int(kernel)))


def launch_counts() -> list[int]:
    return [launch_count(k) for k in range(K_COUNT)]


def launch_count_reset():
    load().gdn_launch_count_reset()
