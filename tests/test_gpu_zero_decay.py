"""Tokens whose decay is exactly 0 (gate logit a = +inf, so g = -inf and
alpha = 0) inside the chunked prefills, against the oracle's token-by-token
recurrence.

At such a token the state is wiped before the delta-rule update, so every
output and state after it depends on the tokens from it on only.  The chunked
forms build decays from differences of cumulative log decays; these tests
place zero-decay tokens at a sequence's first token, inside a chunk, on both
sides of a chunk boundary, in runs of two, and (KDA) on single key channels,
on the tensor-core GDN prefill, the fp32 GDN prefill and the KDA window
prefill.  The decode kernels' zero-decay closed forms are in test_gpu_decode."""
import numpy as np
import pytest
import torch

import hybrid_linear_attention_gdn_gb300 as gdn
import oracle
from hybrid_linear_attention_gdn_gb300 import LayerParams, StatePool, synth
from helpers import (PREFILL_TOL, Setup, assert_out_close, conv_bits_equal, max_rel_l2, prefill_row_tol,
                     prefill_state_tol, prefill_tol, to_np)

pytestmark = pytest.mark.gpu

# sequence-relative tokens given a = +inf: the first token, inside the first
# 64-token chunk, both sides of the chunk boundary at 64 (start 0), a run of two
ZERO_TOKENS = [0, 17, 63, 64, 100, 101, 190]


def _ck_pool(st, n):
    p = StatePool.empty(st.dims, n, "cuda")
    p.ssm.fill_(-5.0)
    p.conv.fill_(9.0)
    return p


def _ock_pool(shape, n):
    return oracle.Pool(np.full((n, shape.hv, shape.dv, shape.dk), -5.0),
                       np.full((n, shape.w - 1, shape.channels), 9.0))


def _layout(lens, starts, blk, gen, n_slots):
    n = len(lens)
    ids = synth.slot_ids(n_slots, n, gen)
    max_ck = max(1, max((s + L) // blk - s // blk for s, L in zip(starts, lens)))
    n_ck = n * max_ck + 2
    ck_ids = synth.slot_ids(n_ck, n * max_ck, gen).reshape(n, max_ck)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    sp = torch.tensor(starts, dtype=torch.int64)
    return ids, ck_ids, n_ck, cu, sp


def _zero_rows(lens, cu):
    rows = []
    for i, L in enumerate(lens):
        rows += [int(cu[i]) + t for t in ZERO_TOKENS if t < L]
    return rows


def _check(st, shape, ids, ck, ock, n_ck, out, o_ref, tol, row_tol, stol):
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    assert_out_close(out, o_ref, shape.dv, tol, row_floor_rms=True, row_tol=row_tol)
    used = ids.tolist()
    assert torch.isfinite(st.pool.ssm[used]).all()
    assert max_rel_l2(to_np(st.pool.ssm[used]), st.opool.ssm[used], shape.dv * shape.dk) <= stol
    assert conv_bits_equal(st.pool.conv[used], st.opool.conv[used])
    written = [i for i in range(n_ck) if not np.all(ock.ssm[i] == -5.0)]
    assert written
    assert max_rel_l2(to_np(ck.ssm[written]), ock.ssm[written], shape.dv * shape.dk) <= stol


@pytest.mark.parametrize("path", ["tc", "bf16", "cuda"])
def test_gdn_prefill_zero_decay_tokens(cuda, monkeypatch, path):
    """Half of the V heads see a = +inf at the chosen tokens; path "cuda"
    forces the fp32 prefill, "bf16" the bf16-operand tensor-core prefill."""
    if path != "tc":
        monkeypatch.setenv("GDN_PREFILL_PATH", path)
    shape = synth.QWEN
    lens, starts, blk = [200, 130], [0, 37], 64
    st = Setup(shape, seed=150, num_slots=6)
    ids, ck_ids, n_ck, cu, sp = _layout(lens, starts, blk, st.gen, 6)
    total = int(cu[-1])
    qkv, a, b = st.tokens((total,))
    a[_zero_rows(lens, cu), ::2] = float("inf")
    ck = _ck_pool(st, n_ck)
    out = torch.full((total, shape.hv, shape.dv), 3.0, dtype=shape.act_dtype, device="cuda")
    nbytes = gdn.chunk_prefill_workspace_size(st.dims, len(lens), total)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device="cuda")
    gdn.chunk_prefill(st.dims, st.pool, ck, st.params, ids.cuda(), cu.cuda(), sp.cuda(), total, ck_ids.cuda(),
                      blk, qkv.cuda(), a.cuda(), b.cuda(), out, ws)
    ock = _ock_pool(shape, n_ck)
    o_ref, err = oracle.prefill(st.od, st.opool, ock, st.oparams, ids.numpy(), cu.numpy(), sp.numpy(),
                                ck_ids.numpy(), blk, to_np(qkv), to_np(a), to_np(b))
    assert err == 0
    _check(st, shape, ids, ck, ock, n_ck, out, o_ref, prefill_tol(shape, path), prefill_row_tol(shape, path),
           prefill_state_tol(shape, path))


@pytest.mark.parametrize("path", ["tc", "window"])
def test_kda_prefill_zero_decay_channels(cuda, monkeypatch, path):
    """KDA: every third key channel of every V head sees a = +inf at the
    chosen tokens (the 64-token chunk form on the tensor cores, and the
    16-token window form; the second sequence starts off a chunk and a
    window boundary)."""
    if path == "window":
        monkeypatch.setenv("GDN_KDA_PREFILL_PATH", "window")
    shape = synth.QWEN
    lens, starts, blk = [200, 130], [0, 37], 64
    st = Setup(shape, seed=151, num_slots=6)
    g = synth.generator(152)
    dt = synth.normal((shape.hv, shape.dk), 0.5, g)
    params = LayerParams(st.params.conv_w, st.params.A_log, dt.cuda())
    oparams = oracle.Params(st.oparams.conv_w, st.oparams.A_log, dt.double().numpy())
    ids, ck_ids, n_ck, cu, sp = _layout(lens, starts, blk, st.gen, 6)
    total = int(cu[-1])
    qkv, _, b = st.tokens((total,))
    a = synth.normal((total, shape.hv, shape.dk), 1.0, st.gen, shape.act_dtype)
    a[_zero_rows(lens, cu), :, ::3] = float("inf")
    ck = _ck_pool(st, n_ck)
    out = torch.full((total, shape.hv, shape.dv), 3.0, dtype=shape.act_dtype, device="cuda")
    gdn.kda_prefill(st.dims, st.pool, ck, params, ids.cuda(), cu.cuda(), sp.cuda(), total, ck_ids.cuda(), blk,
                    qkv.cuda(), a.cuda(), b.cuda(), out)
    ock = _ock_pool(shape, n_ck)
    o_ref, err = oracle.kda_prefill(st.od, st.opool, ock, oparams, ids.numpy(), cu.numpy(), sp.numpy(),
                                    ck_ids.numpy(), blk, to_np(qkv), to_np(a), to_np(b))
    assert err == 0
    _check(st, shape, ids, ck, ock, n_ck, out, o_ref, PREFILL_TOL, None, PREFILL_TOL)


# A NaN gate logit (a corrupt input) makes alpha NaN: in the token recurrence
# the state of that head is NaN from that token on, and so is every later
# output.  The chunked forms floor log decays with a comparison that lets NaN
# through, so they poison the same state and outputs instead of hiding the
# NaN as a zero decay.  Within the chunk (GDN) or window (KDA) that holds the
# NaN token, the chunked forms may also return NaN for the tokens before it
# (their products multiply the NaN rows by masked zeros); every other output
# matches the recurrence.
NAN_SEQ_TOKEN = 90  # inside the second 64-token chunk of a sequence starting at 0
NAN_HEAD = 5


def _check_nan(st, shape, lens, cu, ids, ck, ock, ck_ids, out, o_ref, first_clean, tol, stol):
    torch.cuda.synchronize()
    x = out.float().cpu().numpy()
    t_nan = int(cu[0]) + NAN_SEQ_TOKEN
    s0 = int(ids[0])
    # the oracle: NaN from the token on, in that head only
    assert np.isnan(o_ref[t_nan:int(cu[1]), NAN_HEAD]).all()
    assert np.isfinite(o_ref[:t_nan, NAN_HEAD]).all()
    assert np.isnan(st.opool.ssm[s0, NAN_HEAD]).all()
    # the GPU: the same outputs and state are non-finite
    assert not np.isfinite(x[t_nan:int(cu[1]), NAN_HEAD]).any()
    assert not torch.isfinite(st.pool.ssm[s0, NAN_HEAD]).any()
    # everything else is finite and matches: other heads, the other sequence,
    # and the NaN head before the chunk or window that holds the NaN token
    mask = np.ones(x.shape[:2], bool)
    mask[int(cu[0]) + first_clean:int(cu[1]), NAN_HEAD] = False
    assert np.isfinite(x[mask]).all()
    rows_x = x[mask].reshape(-1, shape.dv)
    rows_r = o_ref[mask].reshape(-1, shape.dv)
    err = np.linalg.norm(rows_x - rows_r) / np.linalg.norm(rows_r)
    assert err <= tol, err
    ok_heads = [h for h in range(shape.hv) if h != NAN_HEAD]
    used = ids.tolist()
    assert max_rel_l2(to_np(st.pool.ssm[used][:, ok_heads]), st.opool.ssm[used][:, ok_heads],
                      shape.dv * shape.dk) <= stol
    assert max_rel_l2(to_np(st.pool.ssm[used[1]]), st.opool.ssm[used[1]], shape.dv * shape.dk) <= stol
    # checkpoints of the NaN head: finite before the NaN token, NaN after
    for j, cid in enumerate(ck_ids[0].tolist()):
        end = (j + 1) * 64
        if end > lens[0]:
            break
        if end <= NAN_SEQ_TOKEN:
            assert torch.isfinite(ck.ssm[cid, NAN_HEAD]).all()
        else:
            assert not torch.isfinite(ck.ssm[cid, NAN_HEAD]).any()
            assert np.isnan(ock.ssm[cid, NAN_HEAD]).all()


@pytest.mark.parametrize("path", ["tc", "bf16", "cuda"])
def test_gdn_prefill_nan_gate_poisons_like_the_recurrence(cuda, monkeypatch, path):
    if path != "tc":
        monkeypatch.setenv("GDN_PREFILL_PATH", path)
    shape = synth.QWEN
    lens, starts, blk = [200, 130], [0, 37], 64
    st = Setup(shape, seed=153, num_slots=6)
    ids, ck_ids, n_ck, cu, sp = _layout(lens, starts, blk, st.gen, 6)
    total = int(cu[-1])
    qkv, a, b = st.tokens((total,))
    a[int(cu[0]) + NAN_SEQ_TOKEN, NAN_HEAD] = float("nan")
    ck = _ck_pool(st, n_ck)
    out = torch.full((total, shape.hv, shape.dv), 3.0, dtype=shape.act_dtype, device="cuda")
    nbytes = gdn.chunk_prefill_workspace_size(st.dims, len(lens), total)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device="cuda")
    gdn.chunk_prefill(st.dims, st.pool, ck, st.params, ids.cuda(), cu.cuda(), sp.cuda(), total, ck_ids.cuda(),
                      blk, qkv.cuda(), a.cuda(), b.cuda(), out, ws)
    ock = _ock_pool(shape, n_ck)
    o_ref, err = oracle.prefill(st.od, st.opool, ock, st.oparams, ids.numpy(), cu.numpy(), sp.numpy(),
                                ck_ids.numpy(), blk, to_np(qkv), to_np(a), to_np(b))
    assert err == 0
    _check_nan(st, shape, lens, cu, ids, ck, ock, ck_ids, out, o_ref, 64, prefill_tol(shape, path),
               prefill_state_tol(shape, path))


@pytest.mark.parametrize("path", ["tc", "window"])
def test_kda_prefill_nan_gate_poisons_like_the_recurrence(cuda, monkeypatch, path):
    if path == "window":
        monkeypatch.setenv("GDN_KDA_PREFILL_PATH", "window")
    shape = synth.QWEN
    lens, starts, blk = [200, 130], [0, 37], 64
    st = Setup(shape, seed=154, num_slots=6)
    g = synth.generator(155)
    dt = synth.normal((shape.hv, shape.dk), 0.5, g)
    params = LayerParams(st.params.conv_w, st.params.A_log, dt.cuda())
    oparams = oracle.Params(st.oparams.conv_w, st.oparams.A_log, dt.double().numpy())
    ids, ck_ids, n_ck, cu, sp = _layout(lens, starts, blk, st.gen, 6)
    total = int(cu[-1])
    qkv, _, b = st.tokens((total,))
    a = synth.normal((total, shape.hv, shape.dk), 1.0, st.gen, shape.act_dtype)
    a[int(cu[0]) + NAN_SEQ_TOKEN, NAN_HEAD, 7] = float("nan")  # one key channel
    ck = _ck_pool(st, n_ck)
    out = torch.full((total, shape.hv, shape.dv), 3.0, dtype=shape.act_dtype, device="cuda")
    gdn.kda_prefill(st.dims, st.pool, ck, params, ids.cuda(), cu.cuda(), sp.cuda(), total, ck_ids.cuda(), blk,
                    qkv.cuda(), a.cuda(), b.cuda(), out)
    ock = _ock_pool(shape, n_ck)
    o_ref, err = oracle.kda_prefill(st.od, st.opool, ock, oparams, ids.numpy(), cu.numpy(), sp.numpy(),
                                    ck_ids.numpy(), blk, to_np(qkv), to_np(a), to_np(b))
    assert err == 0
    # the NaN token's 64-token chunk starts at 64, its 16-token window at 80
    _check_nan(st, shape, lens, cu, ids, ck, ock, ck_ids, out, o_ref, 64 if path == "tc" else 80, PREFILL_TOL,
               PREFILL_TOL)
