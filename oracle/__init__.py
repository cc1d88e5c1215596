"""Double-precision CPU oracle for the Gated DeltaNet slot-pool step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
library never links or calls it, and it shares no code with the CUDA sources.

The arithmetic lives in ``gdn_oracle.c`` (plain C, double precision); this
module builds it with gcc on first use and marshals numpy float64 arrays.
Every function mirrors one step of the hot path:

* :func:`decode_step`   - conv1d update + SiLU + L2 norm + gates + gated delta
  rule + readout for one token per request (TokenSpeed slot lifecycle:
  the working slot is updated in place every decode step).
* :func:`spec_verify` / :func:`spec_commit` - per-draft-step snapshots into
  the spec cache, then commit of the accepted snapshot ("Scheduler dual",
  speculative decoding support).
* :func:`prefill` - token-by-token prefill with block-aligned checkpoints
  ("Ciclo de vida de slots": checkpoint slots published at block-aligned
  prefix boundaries).  :func:`prefill_chunked` evaluates the same recurrence
  in the chunkwise WY/UT form and exists only to cross-check the algebra.
* :func:`slot_copy` / :func:`slot_zero` - copy-on-write and explicit zeroing
  ("Riesgo de correctitud: estado obsoleto").
* :func:`commit_index`, :func:`state_pack` / :func:`state_unpack`,
  :func:`gated_rmsnorm` - the index-update commit, state records for a
  transfer, and the readout epilogue.
* :func:`kda_decode_step`, :func:`kda_spec_verify`, :func:`kda_prefill` - the
  same steps with one decay per key channel (KDA).  :func:`kda_prefill_chunked`
  evaluates the KDA prefill in windows (the algebra of the GPU's chunked form)
  and exists only to cross-check that algebra.

Parity pins for each function are in ``tests/test_oracle_pins.py``.  The
numeric conventions the pages leave open (state orientation, the dk^-1/2 query
scale, eps = 1e-6, channel order, the GQA map h -> h // (HV/HK)) are readings,
not pinned by the pages; those parts are marked "parity unpinned" there.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# a mutated copy of the source (tests/test_oracle_mutations.py) builds elsewhere
_SRC = os.environ.get("GDN_ORACLE_SRC", os.path.join(_HERE, "gdn_oracle.c"))
_OUT_DIR = os.environ.get("GDN_ORACLE_BUILD_DIR", os.path.join(_HERE, "_build"))
_SO = os.path.join(_OUT_DIR, "liborc_gdn.so")
_lock = threading.Lock()
_lib = None

ERR_SLOT_OOB = 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (double precision, OpenMP over requests)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


class _Dims(ctypes.Structure):
    _fields_ = [("hk", ctypes.c_int32), ("hv", ctypes.c_int32),
                ("dk", ctypes.c_int32), ("dv", ctypes.c_int32),
                ("w", ctypes.c_int32)]


class _Pool(ctypes.Structure):
    _fields_ = [("ssm", ctypes.c_void_p), ("conv", ctypes.c_void_p),
                ("num_slots", ctypes.c_int32)]


class _Params(ctypes.Structure):
    _fields_ = [("conv_w", ctypes.c_void_p), ("A_log", ctypes.c_void_p),
                ("dt_bias", ctypes.c_void_p)]


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            d = ctypes.c_double
            _lib.orc_silu.restype = d
            _lib.orc_silu.argtypes = [d]
            _lib.orc_softplus.restype = d
            _lib.orc_softplus.argtypes = [d]
            _lib.orc_sigmoid.restype = d
            _lib.orc_sigmoid.argtypes = [d]
            _lib.orc_gate_g.restype = d
            _lib.orc_gate_g.argtypes = [d, d, d]
            _lib.orc_num_threads.restype = ctypes.c_int
    return _lib


@dataclass(frozen=True)
class Dims:
    hk: int
    hv: int
    dk: int
    dv: int
    w: int = 4

    @property
    def channels(self) -> int:
        return 2 * self.hk * self.dk + self.hv * self.dv

    def c(self) -> _Dims:
        return _Dims(self.hk, self.hv, self.dk, self.dv, self.w)


def _f64(x) -> np.ndarray:
    a = np.ascontiguousarray(x, dtype=np.float64)
    return a


def _i32(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.int32)


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


class Pool:
    """A host pool in double precision: ssm [N][HV][DV][DK], conv [N][W-1][C]."""

    def __init__(self, ssm: np.ndarray, conv: np.ndarray):
        self.ssm = _f64(ssm)
        self.conv = _f64(conv)
        assert self.ssm.shape[0] == self.conv.shape[0]

    @property
    def num_slots(self) -> int:
        return self.ssm.shape[0]

    def c(self) -> _Pool:
        return _Pool(self.ssm.ctypes.data, self.conv.ctypes.data, self.num_slots)

    def copy(self) -> "Pool":
        return Pool(self.ssm.copy(), self.conv.copy())


class Params:
    def __init__(self, conv_w, A_log, dt_bias):
        self.conv_w = _f64(conv_w)
        self.A_log = _f64(A_log)
        self.dt_bias = _f64(dt_bias)

    def c(self) -> _Params:
        return _Params(self.conv_w.ctypes.data, self.A_log.ctypes.data,
                       self.dt_bias.ctypes.data)


def _heads(heads):
    if heads is None:
        return 0, -1
    return int(heads[0]), int(heads[1])


def decode_step(dims: Dims, pool: Pool, params: Params, slot_ids, qkv, a, b,
                heads=None):
    """One decode token per request, in place on ``pool``.  Returns (out, err)."""
    L = lib()
    slot_ids = _i32(slot_ids)
    B = slot_ids.shape[0]
    qkv, a, b = _f64(qkv), _f64(a), _f64(b)
    assert qkv.shape == (B, dims.channels) and a.shape == (B, dims.hv) == b.shape
    out = np.zeros((B, dims.hv, dims.dv), np.float64)
    err = ctypes.c_uint32(0)
    h0, h1 = _heads(heads)
    cd, cpa = dims.c(), params.c()
    rc = L.orc_decode_step(ctypes.byref(cd), pool.c(), ctypes.byref(cpa),
                           _ptr(slot_ids), ctypes.c_int32(B), _ptr(qkv), _ptr(a),
                           _ptr(b), _ptr(out), ctypes.byref(err),
                           ctypes.c_int32(h0), ctypes.c_int32(h1))
    assert rc == 0
    return out, err.value


def slot_copy(dims: Dims, src: Pool, dst: Pool, src_ids, dst_ids):
    L = lib()
    src_ids, dst_ids = _i32(src_ids), _i32(dst_ids)
    err = ctypes.c_uint32(0)
    cd = dims.c()
    rc = L.orc_slot_copy(ctypes.byref(cd), src.c(), dst.c(), _ptr(src_ids),
                         _ptr(dst_ids), ctypes.c_int32(src_ids.shape[0]),
                         ctypes.byref(err))
    assert rc == 0
    return err.value


def slot_zero(dims: Dims, pool: Pool, ids):
    L = lib()
    ids = _i32(ids)
    err = ctypes.c_uint32(0)
    cd = dims.c()
    rc = L.orc_slot_zero(ctypes.byref(cd), pool.c(), _ptr(ids),
                         ctypes.c_int32(ids.shape[0]), ctypes.byref(err))
    assert rc == 0
    return err.value


def spec_verify(dims: Dims, work: Pool, spec: Pool, params: Params, slot_ids,
                spec_ids, qkv, a, b):
    """Draft tokens qkv [B][T][C]; returns (out [B][T][HV][DV], err)."""
    L = lib()
    slot_ids, spec_ids = _i32(slot_ids), _i32(spec_ids)
    B, T = spec_ids.shape
    qkv, a, b = _f64(qkv), _f64(a), _f64(b)
    assert qkv.shape == (B, T, dims.channels)
    out = np.zeros((B, T, dims.hv, dims.dv), np.float64)
    err = ctypes.c_uint32(0)
    cd, cpa = dims.c(), params.c()
    rc = L.orc_spec_verify(ctypes.byref(cd), work.c(), spec.c(), ctypes.byref(cpa),
                           _ptr(slot_ids), _ptr(spec_ids), ctypes.c_int32(B),
                           ctypes.c_int32(T), _ptr(qkv), _ptr(a), _ptr(b),
                           _ptr(out), ctypes.byref(err))
    assert rc == 0
    return out, err.value


def spec_commit(dims: Dims, spec: Pool, work: Pool, spec_ids, accept_len, slot_ids):
    L = lib()
    spec_ids, accept_len, slot_ids = _i32(spec_ids), _i32(accept_len), _i32(slot_ids)
    B, T = spec_ids.shape
    err = ctypes.c_uint32(0)
    cd = dims.c()
    rc = L.orc_spec_commit(ctypes.byref(cd), spec.c(), work.c(), _ptr(spec_ids),
                           _ptr(accept_len), _ptr(slot_ids), ctypes.c_int32(B),
                           ctypes.c_int32(T), ctypes.byref(err))
    assert rc == 0
    return err.value


def commit_index(spec_ids, accept_len, slot_ids):
    """Index-update commit; returns (new slot_ids [B], freed [B][T], err)."""
    L = lib()
    spec_ids, accept_len = _i32(spec_ids), _i32(accept_len)
    B, T = spec_ids.shape
    slots = _i32(slot_ids).copy()
    freed = np.zeros((B, T), np.int32)
    err = ctypes.c_uint32(0)
    rc = L.orc_commit_index(_ptr(spec_ids), _ptr(accept_len), _ptr(slots), _ptr(freed),
                            ctypes.c_int32(B), ctypes.c_int32(T), ctypes.byref(err))
    assert rc == 0
    return slots, freed, err.value


def state_pack(dims: Dims, pool: Pool, ids):
    """Returns (ssm records [n][HV][DV][DK], conv records [n][W-1][C], err)."""
    L = lib()
    ids = _i32(ids)
    n = ids.shape[0]
    st_ssm = np.zeros((n, dims.hv, dims.dv, dims.dk), np.float64)
    st_conv = np.zeros((n, dims.w - 1, dims.channels), np.float64)
    err = ctypes.c_uint32(0)
    cd = dims.c()
    rc = L.orc_state_pack(ctypes.byref(cd), pool.c(), _ptr(ids), ctypes.c_int32(n), _ptr(st_ssm),
                          _ptr(st_conv), ctypes.byref(err))
    assert rc == 0
    return st_ssm, st_conv, err.value


def state_unpack(dims: Dims, st_ssm, st_conv, pool: Pool, ids):
    L = lib()
    ids = _i32(ids)
    st_ssm, st_conv = _f64(st_ssm), _f64(st_conv)
    err = ctypes.c_uint32(0)
    cd = dims.c()
    rc = L.orc_state_unpack(ctypes.byref(cd), _ptr(st_ssm), _ptr(st_conv), pool.c(), _ptr(ids),
                            ctypes.c_int32(ids.shape[0]), ctypes.byref(err))
    assert rc == 0
    return err.value


def kda_decode_step(dims: Dims, pool: Pool, params: Params, slot_ids, qkv, a, b):
    """KDA decode (per-key-channel decay): as decode_step, with a [B][hv][dk]
    gate logits and params.dt_bias [hv][dk].  In place on ``pool``.  Returns
    (out, err)."""
    L = lib()
    slot_ids = _i32(slot_ids)
    B = slot_ids.shape[0]
    qkv, a, b = _f64(qkv), _f64(a), _f64(b)
    assert qkv.shape == (B, dims.channels) and a.shape == (B, dims.hv, dims.dk)
    assert b.shape == (B, dims.hv) and params.dt_bias.shape == (dims.hv, dims.dk)
    out = np.zeros((B, dims.hv, dims.dv), np.float64)
    err = ctypes.c_uint32(0)
    cd, cpa = dims.c(), params.c()
    rc = L.orc_kda_decode_step(ctypes.byref(cd), pool.c(), ctypes.byref(cpa), _ptr(slot_ids),
                               ctypes.c_int32(B), _ptr(qkv), _ptr(a), _ptr(b), _ptr(out),
                               ctypes.byref(err))
    assert rc == 0
    return out, err.value


def kda_spec_verify(dims: Dims, work: Pool, spec: Pool, params: Params, slot_ids, spec_ids, qkv, a, b):
    """KDA verify: T draft tokens per request from the working slot (only
    read), the state after draft t into spec slot spec_ids[r][t]; a
    [B][T][hv][dk].  Returns (out [B][T][hv][dv], err)."""
    L = lib()
    slot_ids, spec_ids = _i32(slot_ids), _i32(spec_ids)
    B, T = spec_ids.shape
    qkv, a, b = _f64(qkv), _f64(a), _f64(b)
    assert qkv.shape == (B, T, dims.channels) and a.shape == (B, T, dims.hv, dims.dk)
    out = np.zeros((B, T, dims.hv, dims.dv), np.float64)
    err = ctypes.c_uint32(0)
    cd, cpa = dims.c(), params.c()
    rc = L.orc_kda_spec_verify(ctypes.byref(cd), work.c(), spec.c(), ctypes.byref(cpa), _ptr(slot_ids),
                               _ptr(spec_ids), ctypes.c_int32(B), ctypes.c_int32(T), _ptr(qkv), _ptr(a),
                               _ptr(b), _ptr(out), ctypes.byref(err))
    assert rc == 0
    return out, err.value


def kda_prefill(dims: Dims, pool: Pool, ckpt: Pool, params: Params, slot_ids, cu_seqlens, start_pos,
                ckpt_ids, ckpt_block, qkv, a, b):
    """Token-by-token KDA prefill (the prefill contract, KDA steps); a is
    [Ttot][hv][dk], params.dt_bias [hv][dk].  Returns (out, err)."""
    L = lib()
    slot_ids = _i32(slot_ids)
    cu = _i32(cu_seqlens)
    sp = np.ascontiguousarray(start_pos, dtype=np.int64)
    ck = _i32(ckpt_ids)
    if ck.ndim == 1:
        ck = ck.reshape(slot_ids.shape[0], -1)
    qkv, a, b = _f64(qkv), _f64(a), _f64(b)
    ttot = int(cu[-1])
    assert qkv.shape == (ttot, dims.channels) and a.shape == (ttot, dims.hv, dims.dk)
    out = np.zeros((ttot, dims.hv, dims.dv), np.float64)
    err = ctypes.c_uint32(0)
    cd, cpa = dims.c(), params.c()
    rc = L.orc_kda_prefill(ctypes.byref(cd), pool.c(), ckpt.c(), ctypes.byref(cpa), _ptr(slot_ids), _ptr(cu),
                           _ptr(sp), ctypes.c_int32(slot_ids.shape[0]), _ptr(ck), ctypes.c_int32(ck.shape[1]),
                           ctypes.c_int32(ckpt_block), _ptr(qkv), _ptr(a), _ptr(b), _ptr(out),
                           ctypes.byref(err))
    assert rc == 0
    return out, err.value


def kda_prefill_chunked(dims: Dims, pool: Pool, ckpt: Pool, params: Params, slot_ids, cu_seqlens, start_pos,
                        ckpt_ids, ckpt_block, chunk, qkv, a, b):
    """The KDA prefill evaluated in windows of `chunk` tokens (the window form:
    A', M, T from per-channel cumulative log decays); cross-check only.
    Returns (out, err)."""
    L = lib()
    slot_ids = _i32(slot_ids)
    cu = _i32(cu_seqlens)
    sp = np.ascontiguousarray(start_pos, dtype=np.int64)
    ck = _i32(ckpt_ids)
    if ck.ndim == 1:
        ck = ck.reshape(slot_ids.shape[0], -1)
    qkv, a, b = _f64(qkv), _f64(a), _f64(b)
    ttot = int(cu[-1])
    assert qkv.shape == (ttot, dims.channels) and a.shape == (ttot, dims.hv, dims.dk)
    out = np.zeros((ttot, dims.hv, dims.dv), np.float64)
    err = ctypes.c_uint32(0)
    cd, cpa = dims.c(), params.c()
    rc = L.orc_kda_prefill_chunked(ctypes.byref(cd), pool.c(), ckpt.c(), ctypes.byref(cpa), _ptr(slot_ids),
                                   _ptr(cu), _ptr(sp), ctypes.c_int32(slot_ids.shape[0]), _ptr(ck),
                                   ctypes.c_int32(ck.shape[1]), ctypes.c_int32(ckpt_block), ctypes.c_int32(chunk),
                                   _ptr(qkv), _ptr(a), _ptr(b), _ptr(out), ctypes.byref(err))
    assert rc == 0
    return out, err.value


def gated_rmsnorm(dims: Dims, o, z, w, eps=1e-6):
    """Readout epilogue y = o / sqrt(mean(o^2) + eps) * w * silu(z) per
    (token, V head) row; o, z [n_tok][hv][dv], w [dv].  Returns y."""
    L = lib()
    o, z, w = _f64(o), _f64(z), _f64(w)
    assert o.shape == z.shape and o.shape[1:] == (dims.hv, dims.dv) and w.shape == (dims.dv,)
    y = np.zeros_like(o)
    cd = dims.c()
    rc = L.orc_gated_rmsnorm(ctypes.byref(cd), _ptr(o), _ptr(z), _ptr(w), ctypes.c_double(eps),
                             ctypes.c_int64(o.shape[0]), _ptr(y))
    assert rc == 0
    return y


def _prefill_common(dims, slot_ids, cu_seqlens, start_pos, ckpt_ids, qkv, a, b):
    slot_ids = _i32(slot_ids)
    cu = _i32(cu_seqlens)
    sp = np.ascontiguousarray(start_pos, dtype=np.int64)
    ck = _i32(ckpt_ids)
    if ck.ndim == 1:
        ck = ck.reshape(slot_ids.shape[0], -1)
    qkv, a, b = _f64(qkv), _f64(a), _f64(b)
    ttot = int(cu[-1])
    assert qkv.shape == (ttot, dims.channels) and a.shape == (ttot, dims.hv)
    out = np.zeros((ttot, dims.hv, dims.dv), np.float64)
    return slot_ids, cu, sp, ck, qkv, a, b, out


def prefill(dims: Dims, pool: Pool, ckpt: Pool, params: Params, slot_ids,
            cu_seqlens, start_pos, ckpt_ids, ckpt_block, qkv, a, b, heads=None):
    """Token-by-token prefill (the plain definition).  Returns (out, err)."""
    L = lib()
    slot_ids, cu, sp, ck, qkv, a, b, out = _prefill_common(
        dims, slot_ids, cu_seqlens, start_pos, ckpt_ids, qkv, a, b)
    err = ctypes.c_uint32(0)
    h0, h1 = _heads(heads)
    cd, cpa = dims.c(), params.c()
    rc = L.orc_prefill(ctypes.byref(cd), pool.c(), ckpt.c(), ctypes.byref(cpa),
                       _ptr(slot_ids), _ptr(cu), _ptr(sp),
                       ctypes.c_int32(slot_ids.shape[0]), _ptr(ck),
                       ctypes.c_int32(ck.shape[1]), ctypes.c_int32(ckpt_block),
                       _ptr(qkv), _ptr(a), _ptr(b), _ptr(out), ctypes.byref(err),
                       ctypes.c_int32(h0), ctypes.c_int32(h1))
    assert rc == 0
    return out, err.value


def prefill_chunked(dims: Dims, pool: Pool, ckpt: Pool, params: Params, slot_ids,
                    cu_seqlens, start_pos, ckpt_ids, ckpt_block, chunk, qkv, a, b):
    """Chunkwise WY/UT evaluation of the same prefill (cross-check only)."""
    L = lib()
    slot_ids, cu, sp, ck, qkv, a, b, out = _prefill_common(
        dims, slot_ids, cu_seqlens, start_pos, ckpt_ids, qkv, a, b)
    err = ctypes.c_uint32(0)
    cd, cpa = dims.c(), params.c()
    rc = L.orc_prefill_chunked(ctypes.byref(cd), pool.c(), ckpt.c(), ctypes.byref(cpa),
                               _ptr(slot_ids), _ptr(cu), _ptr(sp),
                               ctypes.c_int32(slot_ids.shape[0]), _ptr(ck),
                               ctypes.c_int32(ck.shape[1]), ctypes.c_int32(ckpt_block),
                               ctypes.c_int32(chunk), _ptr(qkv), _ptr(a), _ptr(b),
                               _ptr(out), ctypes.byref(err))
    assert rc == 0
    return out, err.value


def delta_core(St, k, v, q, alpha, beta):
    """Single-head gated delta rule on a copy of St [dv][dk]; returns (St', o)."""
    L = lib()
    St = _f64(St).copy()
    dv, dk = St.shape
    k, v, q = _f64(k), _f64(v), _f64(q)
    o = np.zeros(dv, np.float64)
    L.orc_delta_core(ctypes.c_int32(dk), ctypes.c_int32(dv), _ptr(St), _ptr(k),
                     _ptr(v), _ptr(q), ctypes.c_double(alpha), ctypes.c_double(beta),
                     _ptr(o))
    return St, o


def l2norm(x, scale=1.0):
    L = lib()
    x = _f64(x)
    out = np.zeros_like(x)
    L.orc_l2norm(ctypes.c_int32(x.shape[0]), _ptr(x), ctypes.c_double(scale), _ptr(out))
    return out


def conv_silu(dims: Dims, hist, x, conv_w):
    L = lib()
    hist, x, conv_w = _f64(hist), _f64(x), _f64(conv_w)
    y = np.zeros(dims.channels, np.float64)
    cd = dims.c()
    L.orc_conv_silu(ctypes.byref(cd), _ptr(hist), _ptr(x), _ptr(conv_w), _ptr(y))
    return y


def silu(y: float) -> float:
    return lib().orc_silu(float(y))


def softplus(x: float) -> float:
    return lib().orc_softplus(float(x))


def sigmoid(x: float) -> float:
    return lib().orc_sigmoid(float(x))


def gate_g(A_log: float, dt_bias: float, a: float) -> float:
    return lib().orc_gate_g(float(A_log), float(dt_bias), float(a))


def num_threads() -> int:
    return int(lib().orc_num_threads())
