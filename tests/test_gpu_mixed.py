"""GPU mixed batches (decode-first: single-token decode requests, then chunked
prefill continuations from arbitrary positions) against the oracle's decode
step and token-by-token prefill, and bit-exact against the same rows sent
through gdn_decode_step and gdn_chunk_prefill separately."""
import numpy as np
import pytest
import torch

import hybrid_linear_attention_gdn_gb300 as gdn
import oracle
from hybrid_linear_attention_gdn_gb300 import StatePool, synth
from helpers import (STATE_TOL_1, Setup, assert_out_close, conv_bits_equal, max_rel_l2, out_tol,
                     prefill_row_tol, prefill_state_tol, prefill_tol, to_np)

pytestmark = pytest.mark.gpu

BLK = 256


def _batch(st: Setup, n_dec, lens, starts, n_slots):
    """Ids, cu_seqlens (decode rows first), start positions, checkpoint ids and
    tokens of one decode-first mixed batch."""
    n = n_dec + len(lens)
    ids = synth.slot_ids(n_slots, n, st.gen)
    seq_lens = [1] * n_dec + list(lens)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(seq_lens)]), dtype=torch.int32)
    sp = torch.tensor([0] * n_dec + list(starts), dtype=torch.int64)
    max_ck = max(1, max(((s + L) // BLK - s // BLK for s, L in zip(starts, lens)), default=1))
    ck_ids = torch.full((n, max_ck), -1, dtype=torch.int32)
    n_ck = len(lens) * max_ck + 2
    if lens:
        ck_ids[n_dec:] = synth.slot_ids(n_ck, len(lens) * max_ck, st.gen).reshape(len(lens), max_ck)
    qkv, a, b = st.tokens((int(cu[-1]),))
    return ids, cu, sp, ck_ids, n_ck, qkv, a, b


def _ck_pool(st, n):
    p = StatePool.empty(st.dims, n, "cuda")
    p.ssm.fill_(-5.0)
    p.conv.fill_(9.0)
    return p


def _workspace(dims, n_seq, total):
    nbytes = gdn.chunk_prefill_workspace_size(dims, n_seq, total)
    return torch.empty(max(nbytes, 1), dtype=torch.uint8, device="cuda")


CASES = [
    # (shape, decode requests, continuation lengths, their start positions)
    (synth.QWEN, 6, [200, 1, 70, 129], [200, 77, 4101, 63]),
    (synth.QWEN, 16, [], []),
    (synth.QWEN, 0, [300, 9], [512, 1001]),
    (synth.TINY, 3, [37, 130, 1], [5, 64, 300]),
    # the benchmark's batch: 64 decode requests + 4 continuations of 256 tokens
    (synth.QWEN, 64, [256] * 4, [1000, 3077, 517, 8191]),
]
IDS = ["qwen_6_decode_4_continuations", "qwen_decode_only", "qwen_prefill_only", "tiny_mixed",
       "qwen_64_decode_4x256_bench_batch"]


@pytest.mark.parametrize("shape,n_dec,lens,starts", CASES, ids=IDS)
def test_mixed_step_vs_oracle(cuda, shape, n_dec, lens, starts):
    n_slots = 16 if shape is synth.TINY else max(24, n_dec + len(lens) + 4)
    st = Setup(shape, seed=50, num_slots=n_slots)
    ids, cu, sp, ck_ids, n_ck, qkv, a, b = _batch(st, n_dec, lens, starts, n_slots)
    n, total = ids.shape[0], int(cu[-1])
    ck = _ck_pool(st, n_ck)
    out = torch.full((total, shape.hv, shape.dv), 3.0, dtype=shape.act_dtype, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.mixed_step(st.dims, st.pool, ck, st.params, ids.cuda(), cu.cuda(), sp.cuda(), total, n_dec,
                   ck_ids.cuda(), BLK, qkv.cuda(), a.cuda(), b.cuda(), out, _workspace(st.dims, n, total),
                   err)
    # the oracle: decode steps for the first rows, token-by-token prefill for the rest
    ock = oracle.Pool(np.full((n_ck, shape.hv, shape.dv, shape.dk), -5.0),
                      np.full((n_ck, shape.w - 1, shape.channels), 9.0))
    o_dec = o_pre = None
    if n_dec:
        o_dec, e1 = oracle.decode_step(st.od, st.opool, st.oparams, ids[:n_dec].numpy(),
                                       to_np(qkv[:n_dec]), to_np(a[:n_dec]), to_np(b[:n_dec]))
        assert e1 == 0
    if lens:
        o_pre, e2 = oracle.prefill(st.od, st.opool, ock, st.oparams, ids[n_dec:].numpy(),
                                   (cu[n_dec:] - n_dec).numpy(), sp[n_dec:].numpy(),
                                   ck_ids[n_dec:].numpy(), BLK, to_np(qkv[n_dec:]), to_np(a[n_dec:]),
                                   to_np(b[n_dec:]))
        assert e2 == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    if n_dec:
        assert_out_close(out[:n_dec], o_dec, shape.dv, out_tol(shape))
        dec = ids[:n_dec].tolist()
        assert max_rel_l2(to_np(st.pool.ssm[dec]), st.opool.ssm[dec], shape.dv * shape.dk) <= STATE_TOL_1
        assert conv_bits_equal(st.pool.conv[dec], st.opool.conv[dec])
    if lens:
        assert_out_close(out[n_dec:], o_pre, shape.dv, prefill_tol(shape), row_floor_rms=True,
                         row_tol=prefill_row_tol(shape))
        pre = ids[n_dec:].tolist()
        stol = prefill_state_tol(shape)
        assert max_rel_l2(to_np(st.pool.ssm[pre]), st.opool.ssm[pre], shape.dv * shape.dk) <= stol
        assert conv_bits_equal(st.pool.conv[pre], st.opool.conv[pre])
        written = [i for i in range(n_ck) if not np.all(ock.ssm[i] == -5.0)]
        assert len(written) == sum((s + L) // BLK - s // BLK for s, L in zip(starts, lens))
        if written:
            assert max_rel_l2(to_np(ck.ssm[written]), ock.ssm[written], shape.dv * shape.dk) <= stol
        assert conv_bits_equal(ck.conv, ock.conv)
    # untouched slots keep their values
    rest = [s for s in range(n_slots) if s not in ids.tolist()]
    assert torch.equal(st.pool.ssm[rest].cpu(), torch.from_numpy(st.opool.ssm[rest]).float())


def _one_launch(shape, n_dec, lens):
    """Whether the mixed step is one launch for this batch (both halves on
    their fast paths: the Qwen3.5 shape, the decode step's TMA-fed kernel from
    3 requests up, continuations present)."""
    return shape is synth.QWEN and n_dec >= 3 and len(lens) > 0


@pytest.mark.parametrize("form", ["one_launch", "split"])
@pytest.mark.parametrize("shape,n_dec,lens,starts", CASES, ids=IDS)
def test_mixed_step_equals_separate_calls(cuda, monkeypatch, form, shape, n_dec, lens, starts):
    """Bit for bit the decode step on the decode rows and the chunked prefill on
    the rest, called one after the other: as one launch where the batch allows
    it, and as separate launches (GDN_MIXED=split)."""
    if form == "split":
        monkeypatch.setenv("GDN_MIXED", "split")
    fused = form == "one_launch" and _one_launch(shape, n_dec, lens)
    n_slots = 16 if shape is synth.TINY else max(24, n_dec + len(lens) + 4)
    st = Setup(shape, seed=51, num_slots=n_slots)
    ids, cu, sp, ck_ids, n_ck, qkv, a, b = _batch(st, n_dec, lens, starts, n_slots)
    n, total = ids.shape[0], int(cu[-1])
    q, av, bv = qkv.cuda(), a.cuda(), b.cuda()
    pool2 = StatePool(st.pool.ssm.clone(), st.pool.conv.clone())
    ck1, ck2 = _ck_pool(st, n_ck), _ck_pool(st, n_ck)
    out1 = torch.zeros((total, shape.hv, shape.dv), dtype=shape.act_dtype, device="cuda")
    out2 = torch.zeros_like(out1)
    ws = _workspace(st.dims, n, total)
    n_dec0, n_mix0 = gdn.launch_count(gdn.K_DECODE), gdn.launch_count(gdn.K_MIXED)
    gdn.mixed_step(st.dims, st.pool, ck1, st.params, ids.cuda(), cu.cuda(), sp.cuda(), total, n_dec,
                   ck_ids.cuda(), BLK, q, av, bv, out1, ws)
    assert gdn.launch_count(gdn.K_MIXED) == n_mix0 + (1 if fused else 0)
    assert gdn.launch_count(gdn.K_DECODE) == n_dec0 + (1 if n_dec and not fused else 0)
    if fused:  # the work queue is left zero in the workspace
        assert not torch.any(ws[:8 * (2 + len(lens))])
    if n_dec:
        gdn.decode_step(st.dims, pool2, st.params, ids[:n_dec].cuda(), q[:n_dec], av[:n_dec], bv[:n_dec],
                        out2[:n_dec])
    if lens:
        gdn.chunk_prefill(st.dims, pool2, ck2, st.params, ids[n_dec:].cuda(), (cu[n_dec:] - n_dec).cuda(),
                          sp[n_dec:].cuda(), total - n_dec, ck_ids[n_dec:].cuda(), BLK, q[n_dec:],
                          av[n_dec:], bv[n_dec:], out2[n_dec:], ws)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2)
    assert torch.equal(st.pool.ssm, pool2.ssm) and torch.equal(st.pool.conv, pool2.conv)
    assert torch.equal(ck1.ssm, ck2.ssm) and torch.equal(ck1.conv, ck2.conv)


def test_mixed_step_bad_arguments(cuda):
    st = Setup(synth.TINY, seed=52)
    ids = torch.tensor([0, 1, 2], dtype=torch.int32, device="cuda")
    cu = torch.tensor([0, 1, 2, 5], dtype=torch.int32, device="cuda")
    sp = torch.zeros(3, dtype=torch.int64, device="cuda")
    qkv, a, b = (t.cuda() for t in st.tokens((5,)))
    out = torch.empty((5, 4, 16), dtype=torch.float32, device="cuda")
    ck = _ck_pool(st, 2)
    ws = _workspace(st.dims, 3, 5)
    with pytest.raises(gdn.GdnError) as e:
        gdn.mixed_step(st.dims, st.pool, ck, st.params, ids, cu, sp, 5, 4, None, BLK, qkv, a, b, out, ws)
    assert e.value.status == gdn.binding.ERR_INVALID_ARG


def test_mixed_one_launch_with_padding_and_bad_ids_matches_split(cuda, monkeypatch):
    """Padding (-1) and out-of-range ids among the decode requests and the
    continuations: the one-launch step writes the same bits (zero rows for the
    skipped requests, untouched slots) and the same error bits as the
    separate launches."""
    shape = synth.QWEN
    n_slots = 24
    st = Setup(shape, seed=53, num_slots=n_slots)
    n_dec, lens, starts = 8, [70, 129, 40], [63, 4100, 7]
    ids, cu, sp, ck_ids, n_ck, qkv, a, b = _batch(st, n_dec, lens, starts, n_slots)
    ids[2], ids[5], ids[n_dec + 1] = -1, n_slots + 3, -1
    n, total = ids.shape[0], int(cu[-1])
    q, av, bv = qkv.cuda(), a.cuda(), b.cuda()
    res = []
    for form in ("one_launch", "split"):
        if form == "split":
            monkeypatch.setenv("GDN_MIXED", "split")
        pool = StatePool(st.pool.ssm.clone(), st.pool.conv.clone())
        ck = _ck_pool(st, n_ck)
        out = torch.full((total, shape.hv, shape.dv), 3.0, dtype=shape.act_dtype, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        n_mix0 = gdn.launch_count(gdn.K_MIXED)
        gdn.mixed_step(st.dims, pool, ck, st.params, ids.cuda(), cu.cuda(), sp.cuda(), total, n_dec,
                       ck_ids.cuda(), BLK, q, av, bv, out, _workspace(st.dims, n, total), err)
        torch.cuda.synchronize()
        assert gdn.launch_count(gdn.K_MIXED) == n_mix0 + (1 if form == "one_launch" else 0)
        res.append((out, pool, ck, err))
    (o1, p1, c1, e1), (o2, p2, c2, e2) = res
    assert int(e1.item()) == int(e2.item()) == gdn.DEV_ERR_SLOT_OOB
    assert torch.equal(o1, o2)
    assert torch.equal(p1.ssm, p2.ssm) and torch.equal(p1.conv, p2.conv)
    assert torch.equal(c1.ssm, c2.ssm) and torch.equal(c1.conv, c2.conv)
    assert torch.all(o1[2] == 0) and torch.all(o1[5] == 0)


def test_mixed_one_launch_replayed_from_a_cuda_graph(cuda):
    """The one-launch step captured in a CUDA graph and replayed twice gives the
    bits of two eager calls: its work queue starts afresh on every replay
    (the launch leaves it zero)."""
    shape = synth.QWEN
    n_slots = 24
    st = Setup(shape, seed=54, num_slots=n_slots)
    n_dec, lens, starts = 6, [100, 64], [30, 512]
    ids, cu, sp, ck_ids, n_ck, qkv, a, b = _batch(st, n_dec, lens, starts, n_slots)
    n, total = ids.shape[0], int(cu[-1])
    args = (ids.cuda(), cu.cuda(), sp.cuda(), total, n_dec, ck_ids.cuda(), BLK, qkv.cuda(), a.cuda(), b.cuda())
    ws = _workspace(st.dims, n, total)
    eager = StatePool(st.pool.ssm.clone(), st.pool.conv.clone())
    ck_e = _ck_pool(st, n_ck)
    out_e = torch.zeros((total, shape.hv, shape.dv), dtype=shape.act_dtype, device="cuda")
    for _ in range(2):
        gdn.mixed_step(st.dims, eager, ck_e, st.params, *args, out_e, ws)
    graph = StatePool(st.pool.ssm.clone(), st.pool.conv.clone())
    ck_g = _ck_pool(st, n_ck)
    out_g = torch.zeros_like(out_e)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            gdn.mixed_step(st.dims, graph, ck_g, st.params, *args, out_g, ws)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_g, out_e)
    assert torch.equal(graph.ssm, eager.ssm) and torch.equal(graph.conv, eager.conv)
    assert torch.equal(ck_g.ssm, ck_e.ssm) and torch.equal(ck_g.conv, ck_e.conv)
    assert not torch.any(ws[:8 * (2 + len(lens))])
