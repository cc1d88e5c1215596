"""GPU KDA (per-key-channel decay) against the oracle: the decode step on the
Qwen3.5-shaped layer at several batches, other shapes, 32 chained steps,
padding, uniform gates reducing to the GDN step; the speculative verify with
its snapshots, and verify in the working pool followed by the index commit."""
import numpy as np
import pytest
import torch

import hybrid_linear_attention_gdn_gb300 as gdn
import oracle
from hybrid_linear_attention_gdn_gb300 import LayerParams, synth
from helpers import (STATE_TOL_1, STATE_TOL_64, Setup, state_tol, assert_out_close, conv_bits_equal, max_rel_l2,
                     out_tol, to_np)

pytestmark = pytest.mark.gpu


def _kda_params(st: Setup, seed):
    """The layer's conv weights and A_log with a per-channel dt_bias [hv][dk]."""
    g = synth.generator(seed)
    dt = synth.normal((st.shape.hv, st.shape.dk), 0.5, g)
    params = LayerParams(st.params.conv_w, st.params.A_log, dt.cuda())
    oparams = oracle.Params(st.oparams.conv_w, st.oparams.A_log, dt.double().numpy())
    return params, oparams


def _gates(st: Setup, lead):
    """Per-channel gate logits [*lead][hv][dk] in the activation dtype."""
    return synth.normal(lead + (st.shape.hv, st.shape.dk), 1.0, st.gen, st.shape.act_dtype)


@pytest.mark.parametrize("shape,B", [
    (synth.QWEN, 64), (synth.QWEN, 16), (synth.QWEN, 1), (synth.TINY, 5),
    (synth.QWEN.replace(hk=2, hv=8, dk=64, dv=64), 7),
    (synth.QWEN.replace(act="f32", conv="f32", hk=4, hv=8), 9),
], ids=["qwen_b64", "qwen_b16", "qwen_b1", "tiny_f32", "dk64_g4", "f32_b9"])
def test_kda_decode_vs_oracle(cuda, shape, B):
    n_slots = 8 if shape is synth.TINY else 80
    st = Setup(shape, seed=80 + B, num_slots=n_slots)
    params, oparams = _kda_params(st, 81)
    ids = synth.slot_ids(n_slots, B, st.gen)
    qkv, _, b = st.tokens((B,))
    a = _gates(st, (B,))
    out = torch.empty((B, shape.hv, shape.dv), dtype=shape.act_dtype, device="cuda")
    n0 = gdn.launch_count(gdn.K_KDA_DECODE)
    gdn.kda_decode_step(st.dims, st.pool, params, ids.cuda(), qkv.cuda(), a.cuda(), b.cuda(), out)
    o_ref, err = oracle.kda_decode_step(st.od, st.opool, oparams, ids.numpy(), to_np(qkv), to_np(a),
                                        to_np(b))
    torch.cuda.synchronize()
    assert err == 0 and gdn.launch_count(gdn.K_KDA_DECODE) == n0 + 1
    assert_out_close(out, o_ref, shape.dv, out_tol(shape))
    used = ids.tolist()
    assert max_rel_l2(to_np(st.pool.ssm[used]), st.opool.ssm[used], shape.dv * shape.dk) <= STATE_TOL_1
    assert conv_bits_equal(st.pool.conv, st.opool.conv)
    rest = [s for s in range(n_slots) if s not in used]
    assert torch.equal(st.pool.ssm[rest].cpu(), torch.from_numpy(st.opool.ssm[rest]).float())


def test_kda_32_chained_steps(cuda):
    shape = synth.QWEN
    st = Setup(shape, seed=82, num_slots=24)
    params, oparams = _kda_params(st, 83)
    B = 12
    ids = synth.slot_ids(24, B, st.gen)
    out = torch.empty((B, shape.hv, shape.dv), dtype=shape.act_dtype, device="cuda")
    for _ in range(32):
        qkv, _, b = st.tokens((B,))
        a = _gates(st, (B,))
        gdn.kda_decode_step(st.dims, st.pool, params, ids.cuda(), qkv.cuda(), a.cuda(), b.cuda(), out)
        o_ref, _ = oracle.kda_decode_step(st.od, st.opool, oparams, ids.numpy(), to_np(qkv), to_np(a),
                                          to_np(b))
    torch.cuda.synchronize()
    assert_out_close(out, o_ref, shape.dv, out_tol(shape))
    used = ids.tolist()
    assert max_rel_l2(to_np(st.pool.ssm[used]), st.opool.ssm[used], shape.dv * shape.dk) <= STATE_TOL_64
    assert conv_bits_equal(st.pool.conv[used], st.opool.conv[used])


def test_kda_uniform_gates_is_the_gdn_step(cuda):
    """Every channel of a head given the head's gate logit and bias: the KDA
    kernel lands on the oracle's GDN step."""
    shape = synth.QWEN
    st = Setup(shape, seed=84, num_slots=40)
    B = 32
    ids = synth.slot_ids(40, B, st.gen)
    qkv, a, b = st.tokens((B,))
    a_kda = a[:, :, None].expand(B, shape.hv, shape.dk).contiguous()
    dt = st.params.dt_bias[:, None].expand(shape.hv, shape.dk).contiguous()
    params = LayerParams(st.params.conv_w, st.params.A_log, dt)
    out = torch.empty((B, shape.hv, shape.dv), dtype=shape.act_dtype, device="cuda")
    gdn.kda_decode_step(st.dims, st.pool, params, ids.cuda(), qkv.cuda(), a_kda.cuda(), b.cuda(), out)
    o_ref, _ = oracle.decode_step(st.od, st.opool, st.oparams, ids.numpy(), to_np(qkv), to_np(a), to_np(b))
    torch.cuda.synchronize()
    assert_out_close(out, o_ref, shape.dv, out_tol(shape))
    used = ids.tolist()
    assert max_rel_l2(to_np(st.pool.ssm[used]), st.opool.ssm[used], shape.dv * shape.dk) <= STATE_TOL_1


def test_kda_padding_and_bad_ids(cuda):
    shape = synth.QWEN
    st = Setup(shape, seed=85, num_slots=10)
    params, oparams = _kda_params(st, 86)
    ids = torch.tensor([3, -1, 10, 7], dtype=torch.int32)
    qkv, _, b = st.tokens((4,))
    a = _gates(st, (4,))
    out = torch.full((4, shape.hv, shape.dv), 9.0, dtype=shape.act_dtype, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.kda_decode_step(st.dims, st.pool, params, ids.cuda(), qkv.cuda(), a.cuda(), b.cuda(), out, err)
    o_ref, e = oracle.kda_decode_step(st.od, st.opool, oparams, ids.numpy(), to_np(qkv), to_np(a), to_np(b))
    torch.cuda.synchronize()
    assert int(err.item()) == e == gdn.DEV_ERR_SLOT_OOB
    assert torch.all(out[1:3] == 0)
    assert_out_close(out[[0, 3]], o_ref[[0, 3]], shape.dv, out_tol(shape))
    assert max_rel_l2(to_np(st.pool.ssm), st.opool.ssm, shape.dv * shape.dk) <= STATE_TOL_1


@pytest.mark.parametrize("shape,B,T,path", [
    (synth.QWEN, 16, 8, "auto"), (synth.QWEN, 3, 16, "auto"), (synth.TINY, 2, 5, "auto"),
    (synth.QWEN.replace(act="f32", conv="f32", hk=4, hv=8), 5, 4, "auto"),
    (synth.QWEN, 32, 8, "auto"),
    (synth.QWEN, 3, 16, "tma"), (synth.QWEN, 7, 5, "tma"),
    (synth.QWEN.replace(act="f32", conv="f32", hk=4, hv=8), 5, 4, "tma"),
    (synth.QWEN.replace(conv="f32"), 4, 8, "tma"),
], ids=["qwen_b16_t8", "qwen_b3_t16", "tiny", "f32_b5_t4", "qwen_b32_t8_persistent", "qwen_b3_t16_tma",
        "qwen_b7_t5_tma", "f32_b5_t4_tma", "bf16_f32conv_b4_t8_tma"])
def test_kda_verify_vs_oracle(cuda, monkeypatch, shape, B, T, path):
    """path "tma" forces the persistent TMA-fed verify kernel (the library reads
    GDN_DECODE_PATH on every call); batch 32 of the Qwen layer takes it by
    itself (1024 (request, V head) items, at least 6 per SM)."""
    if path == "tma":
        monkeypatch.setenv("GDN_DECODE_PATH", "tma")
    n_work = 8 if shape is synth.TINY else 40
    st = Setup(shape, seed=90 + B, num_slots=n_work)
    params, oparams = _kda_params(st, 91)
    ids = synth.slot_ids(n_work, B, st.gen)
    n_spec = B * T + 2
    spec = gdn.StatePool.empty(st.dims, n_spec, "cuda")
    spec.ssm.fill_(12345.5)
    spec.conv.fill_(-77.0)
    spec_ids = synth.slot_ids(n_spec, B * T, st.gen).reshape(B, T)
    qkv, _, b = st.tokens((B, T))
    a = _gates(st, (B, T))
    before = st.pool.ssm.clone(), st.pool.conv.clone()
    out = torch.empty((B, T, shape.hv, shape.dv), dtype=shape.act_dtype, device="cuda")
    n0 = gdn.launch_count(gdn.K_KDA_VERIFY)
    gdn.kda_spec_verify(st.dims, st.pool, spec, params, ids.cuda(), spec_ids.cuda(), qkv.cuda(), a.cuda(),
                        b.cuda(), out)
    ospec = oracle.Pool(np.full((n_spec, shape.hv, shape.dv, shape.dk), 12345.5),
                        np.full((n_spec, shape.w - 1, shape.channels), -77.0))
    o_ref, err = oracle.kda_spec_verify(st.od, st.opool, ospec, oparams, ids.numpy(), spec_ids.numpy(),
                                        to_np(qkv), to_np(a), to_np(b))
    torch.cuda.synchronize()
    assert err == 0 and gdn.launch_count(gdn.K_KDA_VERIFY) == n0 + 1
    assert torch.equal(st.pool.ssm, before[0]) and torch.equal(st.pool.conv, before[1])
    assert_out_close(out, o_ref, shape.dv, out_tol(shape))
    sids = spec_ids.flatten().tolist()
    for t in range(T):  # snapshot t: the state after t + 1 steps
        st_ids = spec_ids[:, t].tolist()
        assert max_rel_l2(to_np(spec.ssm[st_ids]), ospec.ssm[st_ids], shape.dv * shape.dk) <= state_tol(t + 1), t
    assert conv_bits_equal(spec.conv[sids], ospec.conv[sids])
    unused = [s for s in range(n_spec) if s not in sids]
    assert torch.all(spec.ssm[unused] == 12345.5)


def test_kda_verify_in_place_then_commit_index(cuda):
    """Snapshots in the working pool, then the index commit: each request lands
    on the state of its first L KDA decode steps."""
    shape = synth.QWEN
    B, T = 8, 6
    n_slots = B * (T + 1) + 4
    st = Setup(shape, seed=92, num_slots=n_slots)
    params, oparams = _kda_params(st, 93)
    perm = synth.slot_ids(n_slots, B * (T + 1), st.gen)
    ids, spec_ids = perm[:B].clone(), perm[B:].reshape(B, T).clone()
    qkv, _, b = st.tokens((B, T))
    a = _gates(st, (B, T))
    before = st.pool.ssm.clone(), st.pool.conv.clone()
    out = torch.empty((B, T, shape.hv, shape.dv), dtype=shape.act_dtype, device="cuda")
    gdn.kda_spec_verify(st.dims, st.pool, st.pool, params, ids.cuda(), spec_ids.cuda(), qkv.cuda(), a.cuda(),
                        b.cuda(), out)
    L = synth.accept_lengths(B, T, st.gen)
    L[1] = 0
    d_slots = ids.cuda()
    freed = torch.empty((B, T), dtype=torch.int32, device="cuda")
    gdn.spec_commit_index(spec_ids.cuda(), L.cuda(), d_slots, freed)
    ref = oracle.Pool(to_np(before[0]), to_np(before[1]))
    for r in range(B):
        for t in range(int(L[r])):
            oracle.kda_decode_step(st.od, ref, oparams, ids[r:r + 1].numpy(), to_np(qkv[r:r + 1, t]),
                                   to_np(a[r:r + 1, t]), to_np(b[r:r + 1, t]))
    torch.cuda.synchronize()
    new = d_slots.cpu().tolist()
    for r in range(B):
        assert max_rel_l2(to_np(st.pool.ssm[new[r]]), ref.ssm[int(ids[r])],
                          shape.dv * shape.dk) <= state_tol(int(L[r]))
    assert conv_bits_equal(st.pool.conv[new], ref.conv[ids.tolist()])
