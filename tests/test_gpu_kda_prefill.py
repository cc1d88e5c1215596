"""GPU KDA prefill (the chunked form, and the token recurrence) against the oracle's token-by-token
KDA prefill: outputs, final states, checkpoint states and conv histories on
packed sequences from arbitrary start positions; uniform gates land on the
GDN prefill; a prefill continued by KDA decode steps; resuming from a copied
checkpoint is bit exact; padding and bad ids; the full 4 x 8192 workload on
its causal prefix."""
import numpy as np
import pytest
import torch

import hybrid_linear_attention_gdn_gb300 as gdn
import oracle
from hybrid_linear_attention_gdn_gb300 import LayerParams, StatePool, synth
from helpers import (PREFILL_TOL, STATE_TOL_64, Setup, assert_out_close, conv_bits_equal, max_rel_l2, out_tol,
                     to_np)

pytestmark = pytest.mark.gpu


def _kda_params(st: Setup, seed):
    g = synth.generator(seed)
    dt = synth.normal((st.shape.hv, st.shape.dk), 0.5, g)
    return (LayerParams(st.params.conv_w, st.params.A_log, dt.cuda()),
            oracle.Params(st.oparams.conv_w, st.oparams.A_log, dt.double().numpy()))


def _gates(st: Setup, n_tok):
    return synth.normal((n_tok, st.shape.hv, st.shape.dk), 1.0, st.gen, st.shape.act_dtype)


def _ck_pool(st, n):
    p = StatePool.empty(st.dims, n, "cuda")
    p.ssm.fill_(-5.0)
    p.conv.fill_(9.0)
    return p


def _ock_pool(shape, n):
    return oracle.Pool(np.full((n, shape.hv, shape.dv, shape.dk), -5.0),
                       np.full((n, shape.w - 1, shape.channels), 9.0))


def _run(st, ck, params, ids, lens, starts, ck_ids, blk, qkv, a, b, err=None):
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    sp = torch.tensor(starts, dtype=torch.int64)
    total = int(cu[-1])
    out = torch.full((total, st.shape.hv, st.shape.dv), 3.0, dtype=st.shape.act_dtype, device="cuda")
    gdn.kda_prefill(st.dims, st.pool, ck, params, ids.cuda(), cu.cuda(), sp.cuda(), total, ck_ids.cuda(), blk,
                    qkv.cuda(), a.cuda(), b.cuda(), out, err)
    return out, cu, sp


def _n_ck(starts, lens, blk):
    return [(s + L) // blk - s // blk for s, L in zip(starts, lens)]


@pytest.mark.parametrize("shape,lens,starts,blk,path", [
    (synth.TINY, [1, 37, 130, 300, 0], [0, 64, 100, 256, 5], 64, "chunked"),
    (synth.QWEN, [70, 200, 513], [0, 128, 0], 256, "recurrent"),
    (synth.QWEN.replace(hk=2, hv=8, dk=64, dv=64), [129, 64, 3], [0, 192, 61], 64, "chunked"),
    (synth.QWEN.replace(act="f32", conv="f32", hk=4, hv=8), [100, 17], [30, 0], 64, "recurrent"),
    (synth.QWEN, [200, 1, 70, 129], [200, 77, 4101, 63], 256, "recurrent"),
    (synth.QWEN, [70, 200, 513], [0, 128, 0], 256, "chunked"),
    (synth.QWEN.replace(act="f32", conv="f32", hk=4, hv=8), [100, 17], [30, 0], 64, "chunked"),
    (synth.QWEN, [200, 1, 70, 129], [200, 77, 4101, 63], 256, "chunked"),
    (synth.QWEN.replace(conv="f32", dv=96), [33, 300], [5, 64], 64, "chunked"),
    # v rows of 200 bytes: the staging falls back to element copies
    (synth.QWEN.replace(dv=100), [45, 130], [9, 0], 64, "chunked"),
    (synth.QWEN, [70, 200, 513], [0, 128, 0], 256, "window"),
    (synth.QWEN, [200, 1, 70, 129], [200, 77, 4101, 63], 256, "window"),
    # one sequence of 24 chunks, with checkpoints every 64 tokens
    (synth.QWEN, [1500], [7], 64, "chunked"),
], ids=["tiny", "qwen_recurrent", "dk64_g4", "f32_recurrent", "qwen_unaligned_continuations_recurrent", "qwen",
        "f32", "qwen_unaligned_continuations", "dv96_f32conv", "dv100_element_staging", "qwen_window",
        "qwen_unaligned_continuations_window", "qwen_1500_every_chunk_checkpointed"])
def test_kda_prefill_vs_oracle(cuda, monkeypatch, shape, lens, starts, blk, path):
    """path "recurrent" forces the token recurrence and "window" the 16-token
    window form (the library reads GDN_KDA_PREFILL_PATH on every call);
    "chunked" is the default, which takes the 64-token chunk form on the
    tensor cores where it applies (dk = dv = 128, bf16: the qwen cases), the
    window form for the other shapes with dk 128 and dv <= 128, and the
    recurrence elsewhere (the tiny and dk 64 cases)."""
    if path in ("recurrent", "window"):
        monkeypatch.setenv("GDN_KDA_PREFILL_PATH", path)
    n = len(lens)
    n_slots = 8 if shape.dk == 16 else 12
    st = Setup(shape, seed=140, num_slots=n_slots)
    params, oparams = _kda_params(st, 141)
    ids = synth.slot_ids(n_slots, n, st.gen)
    max_ck = max(1, max(_n_ck(starts, lens, blk)))
    n_ck = n * max_ck + 2
    ck_ids = synth.slot_ids(n_ck, n * max_ck, st.gen).reshape(n, max_ck)
    ck = _ck_pool(st, n_ck)
    total = int(sum(lens))
    qkv, _, b = st.tokens((total,))
    a = _gates(st, total)
    n0 = gdn.launch_count(gdn.K_KDA_PREFILL)
    out, cu, sp = _run(st, ck, params, ids, lens, starts, ck_ids, blk, qkv, a, b)
    ock = _ock_pool(shape, n_ck)
    o_ref, err = oracle.kda_prefill(st.od, st.opool, ock, oparams, ids.numpy(), cu.numpy(), sp.numpy(),
                                    ck_ids.numpy(), blk, to_np(qkv), to_np(a), to_np(b))
    torch.cuda.synchronize()
    assert err == 0 and gdn.launch_count(gdn.K_KDA_PREFILL) == n0 + 1
    assert_out_close(out, o_ref, shape.dv, PREFILL_TOL, row_floor_rms=True)
    used = ids.tolist()
    assert max_rel_l2(to_np(st.pool.ssm[used]), st.opool.ssm[used], shape.dv * shape.dk) <= PREFILL_TOL
    assert conv_bits_equal(st.pool.conv[used], st.opool.conv[used])
    written = [i for i in range(n_ck) if not np.all(ock.ssm[i] == -5.0)]
    assert len(written) == sum(_n_ck(starts, lens, blk))
    assert max_rel_l2(to_np(ck.ssm[written]), ock.ssm[written], shape.dv * shape.dk) <= PREFILL_TOL
    assert conv_bits_equal(ck.conv, ock.conv)
    assert torch.all(ck.ssm[[i for i in range(n_ck) if i not in written]] == -5.0)


def test_kda_prefill_uniform_gates_is_the_gdn_prefill(cuda):
    """Every key channel given its head's gate logit and bias: the KDA prefill
    lands on the oracle's GDN prefill."""
    shape = synth.QWEN
    st = Setup(shape, seed=142, num_slots=6)
    lens, starts, blk = [300, 65], [0, 200], 64
    ids = torch.tensor([4, 1], dtype=torch.int32)
    max_ck = max(_n_ck(starts, lens, blk))
    ck_ids = torch.arange(2 * max_ck, dtype=torch.int32).reshape(2, max_ck)
    ck = _ck_pool(st, 2 * max_ck)
    total = sum(lens)
    qkv, a, b = st.tokens((total,))
    a_kda = a[:, :, None].expand(total, shape.hv, shape.dk).contiguous()
    dt = st.params.dt_bias[:, None].expand(shape.hv, shape.dk).contiguous()
    params = LayerParams(st.params.conv_w, st.params.A_log, dt)
    out, cu, sp = _run(st, ck, params, ids, lens, starts, ck_ids, blk, qkv, a_kda, b)
    ock = _ock_pool(shape, 2 * max_ck)
    o_ref, err = oracle.prefill(st.od, st.opool, ock, st.oparams, ids.numpy(), cu.numpy(), sp.numpy(),
                                ck_ids.numpy(), blk, to_np(qkv), to_np(a), to_np(b))
    torch.cuda.synchronize()
    assert err == 0
    assert_out_close(out, o_ref, shape.dv, PREFILL_TOL, row_floor_rms=True)
    assert max_rel_l2(to_np(st.pool.ssm[[4, 1]]), st.opool.ssm[[4, 1]], shape.dv * shape.dk) <= PREFILL_TOL
    assert max_rel_l2(to_np(ck.ssm), ock.ssm, shape.dv * shape.dk) <= PREFILL_TOL
    assert conv_bits_equal(ck.conv, ock.conv)


def test_kda_prefill_then_decode_steps(cuda):
    """A prefill continued by 8 KDA decode steps on the working slots, against
    the oracle doing the same."""
    shape = synth.QWEN
    st = Setup(shape, seed=143, num_slots=10)
    params, oparams = _kda_params(st, 144)
    lens, starts, blk = [97, 256, 5], [0, 0, 11], 256
    ids = torch.tensor([7, 2, 9], dtype=torch.int32)
    ck_ids = torch.tensor([[0], [1], [2]], dtype=torch.int32)
    ck = _ck_pool(st, 3)
    total = sum(lens)
    qkv, _, b = st.tokens((total,))
    a = _gates(st, total)
    _, cu, sp = _run(st, ck, params, ids, lens, starts, ck_ids, blk, qkv, a, b)
    ock = _ock_pool(shape, 3)
    oracle.kda_prefill(st.od, st.opool, ock, oparams, ids.numpy(), cu.numpy(), sp.numpy(), ck_ids.numpy(), blk,
                       to_np(qkv), to_np(a), to_np(b))
    out = torch.empty((3, shape.hv, shape.dv), dtype=shape.act_dtype, device="cuda")
    for _ in range(8):
        dq, _, db = st.tokens((3,))
        da = _gates(st, 3)
        gdn.kda_decode_step(st.dims, st.pool, params, ids.cuda(), dq.cuda(), da.cuda(), db.cuda(), out)
        o_ref, _ = oracle.kda_decode_step(st.od, st.opool, oparams, ids.numpy(), to_np(dq), to_np(da), to_np(db))
    torch.cuda.synchronize()
    assert_out_close(out, o_ref, shape.dv, out_tol(shape))
    used = ids.tolist()
    assert max_rel_l2(to_np(st.pool.ssm[used]), st.opool.ssm[used], shape.dv * shape.dk) <= PREFILL_TOL
    assert conv_bits_equal(st.pool.conv[used], st.opool.conv[used])


def test_kda_prefill_resume_from_checkpoint_bit_exact(cuda):
    """A sequence resumed at token 1024 from a copied checkpoint reaches the
    from-scratch outputs, state and checkpoints bit for bit (the recurrence is
    the same token by token)."""
    shape = synth.QWEN
    st = Setup(shape, seed=145, num_slots=4)
    params, _ = _kda_params(st, 146)
    ck = _ck_pool(st, 16)
    qkv, _, b = st.tokens((2048,))
    a = _gates(st, 2048)
    ck_ids = torch.arange(8, dtype=torch.int32).reshape(1, 8)
    out_full, _, _ = _run(st, ck, params, torch.tensor([0], dtype=torch.int32), [2048], [0], ck_ids, 256,
                          qkv, a, b)
    gdn.slot_copy(st.dims, ck, st.pool, torch.tensor([3], dtype=torch.int32, device="cuda"),
                  torch.tensor([2], dtype=torch.int32, device="cuda"))
    ck_ids2 = torch.arange(8, 12, dtype=torch.int32).reshape(1, 4)
    out_res, _, _ = _run(st, ck, params, torch.tensor([2], dtype=torch.int32), [1024], [1024], ck_ids2, 256,
                         qkv[1024:], a[1024:], b[1024:])
    torch.cuda.synchronize()
    assert torch.equal(out_res, out_full[1024:])
    assert torch.equal(st.pool.ssm[2].view(torch.int32), st.pool.ssm[0].view(torch.int32))
    assert torch.equal(st.pool.conv[2], st.pool.conv[0])
    assert torch.equal(ck.ssm[8:12].view(torch.int32), ck.ssm[4:8].view(torch.int32))
    assert torch.equal(ck.conv[8:12], ck.conv[4:8])


def test_kda_prefill_padding_bad_ids_and_empty(cuda):
    shape = synth.QWEN
    st = Setup(shape, seed=147, num_slots=6)
    params, oparams = _kda_params(st, 148)
    lens, starts, blk = [40, 70, 33], [0, 0, 0], 64
    ids = torch.tensor([3, -1, 6], dtype=torch.int32)  # padding, out of range
    ck_ids = torch.tensor([[0], [1], [2]], dtype=torch.int32)
    ck = _ck_pool(st, 3)
    qkv, _, b = st.tokens((143,))
    a = _gates(st, 143)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ssm0 = st.pool.ssm.clone()
    out, cu, sp = _run(st, ck, params, ids, lens, starts, ck_ids, blk, qkv, a, b, err)
    ock = _ock_pool(shape, 3)
    o_ref, e = oracle.kda_prefill(st.od, st.opool, ock, oparams, ids.numpy(), cu.numpy(), sp.numpy(),
                                  ck_ids.numpy(), blk, to_np(qkv), to_np(a), to_np(b))
    torch.cuda.synchronize()
    assert int(err.item()) == e == gdn.DEV_ERR_SLOT_OOB
    assert torch.all(out[40:] == 0)
    assert_out_close(out[:40], o_ref[:40], shape.dv, PREFILL_TOL, row_floor_rms=True)
    others = [0, 1, 2, 4, 5]
    assert torch.equal(st.pool.ssm[others], ssm0[others])
    assert torch.all(ck.ssm == -5.0)  # the one boundary (seq 1, token 64) belongs to a padding row
    # nothing to do: no launch
    n0 = gdn.launch_count(gdn.K_KDA_PREFILL)
    e0 = torch.empty((0,), dtype=torch.int32, device="cuda")
    gdn.kda_prefill(st.dims, st.pool, ck, params, e0, torch.zeros(1, dtype=torch.int32, device="cuda"),
                    torch.empty((0,), dtype=torch.int64, device="cuda"), 0, None, 64, e0, e0, e0, e0)
    assert gdn.launch_count(gdn.K_KDA_PREFILL) == n0
    with pytest.raises(gdn.GdnError):
        _run(st, ck, params, ids, lens, starts, ck_ids, 100, qkv, a, b)  # block not a multiple of 64


def test_kda_prefill_four_by_8192_causal_prefix(cuda):
    """The full 4 x 8192-token workload (checkpoints every 256) in the launch
    shape the benchmark times.  The recurrence is causal, so the outputs of each
    sequence's first 1024 tokens and its first four checkpoints are those of the
    oracle run on that prefix alone; every later checkpoint is written and
    finite."""
    shape = synth.QWEN
    st = Setup(shape, seed=149, num_slots=8)
    params, oparams = _kda_params(st, 150)
    S, pre, blk = 8192, 1024, 256
    ids = torch.tensor([5, 1, 6, 2], dtype=torch.int32)
    ck_ids = torch.arange(128, dtype=torch.int32).reshape(4, 32)
    ck = _ck_pool(st, 128)
    qkv, _, b = st.tokens((4 * S,))
    a = _gates(st, 4 * S)
    ssm0, conv0 = st.opool.ssm.copy(), st.opool.conv.copy()
    out, _, _ = _run(st, ck, params, ids, [S] * 4, [0] * 4, ck_ids, blk, qkv, a, b)
    torch.cuda.synchronize()
    for n in range(4):
        t0 = S * n
        opool = oracle.Pool(ssm0[[int(ids[n])]].copy(), conv0[[int(ids[n])]].copy())
        ock = _ock_pool(shape, 4)
        o_ref, err = oracle.kda_prefill(st.od, opool, ock, oparams, [0], [0, pre], [0],
                                        np.arange(4, dtype=np.int32).reshape(1, 4), blk,
                                        to_np(qkv[t0:t0 + pre]), to_np(a[t0:t0 + pre]), to_np(b[t0:t0 + pre]))
        assert err == 0
        assert_out_close(out[t0:t0 + pre], o_ref, shape.dv, PREFILL_TOL, row_floor_rms=True)
        cks = ck_ids[n].tolist()
        assert max_rel_l2(to_np(ck.ssm[cks[:4]]), ock.ssm, shape.dv * shape.dk) <= PREFILL_TOL
        assert conv_bits_equal(ck.conv[cks[:4]], ock.conv)
        later = ck.ssm[cks[4:]]
        assert torch.all(torch.isfinite(later)) and not torch.any(torch.all(later.flatten(1) == -5.0, dim=1))
