"""GPU speculative verify (per-draft-step snapshots into the spec cache) and
commit of the accepted snapshot, against the oracle."""
import numpy as np
import pytest
import torch

import hybrid_linear_attention_gdn_gb300 as gdn
import oracle
from hybrid_linear_attention_gdn_gb300 import StatePool, synth
from helpers import (assert_out_close, Setup, assert_pool_bits_equal, conv_bits_equal, max_rel_l2, out_tol,
                     state_tol, to_np)

pytestmark = pytest.mark.gpu


def _spec_pool(st: Setup, n):
    """A spec cache filled with a sentinel pattern (stale data)."""
    s = StatePool.empty(st.dims, n, "cuda")
    s.ssm.fill_(12345.5)
    s.conv.fill_(-77.0)
    return s


@pytest.mark.parametrize("shape,B,T,path", [
    (synth.TINY, 2, 5, None),
    (synth.QWEN, 16, 8, None),
    (synth.QWEN, 16, 8, "tma"),
    (synth.QWEN, 32, 8, None),
    (synth.QWEN, 32, 8, "rows"),
    (synth.QWEN, 3, 4, "tma"),
    (synth.QWEN, 24, 16, None),
    (synth.QWEN, 24, 16, "tma"),
    (synth.QWEN.replace(act="f32", conv="f32", hk=4, hv=8), 5, 6, None),
    (synth.QWEN.replace(hk=2, hv=8, dk=64, dv=64), 3, 3, None),
    (synth.QWEN, 64, 8, None),
], ids=["tiny", "qwen_b16_t8", "qwen_b16_t8_persistent", "qwen_b32_t8", "qwen_b32_t8_per_head",
        "qwen_b3_t4_persistent", "qwen_b24_t16", "qwen_b24_t16_persistent", "f32_b5_t6", "dk64_g4",
        "qwen_b64_t8"])
def test_verify_then_commit(cuda, monkeypatch, shape, B, T, path):
    """path: None = the library's own choice (per-head kernel below six
    (request, V head) items per SM, the persistent TMA-fed kernel above);
    "tma" / "rows" force one (GDN_DECODE_PATH, read on every call)."""
    if path:
        monkeypatch.setenv("GDN_DECODE_PATH", path)
    n_work = 8 if shape is synth.TINY else max(48, B + 8)
    st = Setup(shape, seed=30, num_slots=n_work)
    ids = synth.slot_ids(n_work, B, st.gen)
    spec = _spec_pool(st, B * T + 3)
    spec_ids = synth.slot_ids(B * T + 3, B * T, st.gen).reshape(B, T)
    qkv, a, b = st.tokens((B, T))
    work_before = st.pool.ssm.clone(), st.pool.conv.clone()
    out = torch.empty((B, T, shape.hv, shape.dv), dtype=shape.act_dtype, device="cuda")
    gdn.spec_verify(st.dims, st.pool, spec, st.params, ids.cuda(), spec_ids.cuda(), qkv.cuda(),
                    a.cuda(), b.cuda(), out)
    ospec = oracle.Pool(np.full((B * T + 3, shape.hv, shape.dv, shape.dk), 12345.5),
                        np.full((B * T + 3, shape.w - 1, shape.channels), -77.0))
    o_ref, err = oracle.spec_verify(st.od, st.opool, ospec, st.oparams, ids.numpy(),
                                    spec_ids.numpy(), to_np(qkv), to_np(a), to_np(b))
    torch.cuda.synchronize()
    assert err == 0
    # the working slots are only read
    assert torch.equal(st.pool.ssm, work_before[0]) and torch.equal(st.pool.conv, work_before[1])
    assert_out_close(out, o_ref, shape.dv, out_tol(shape))
    sids = spec_ids.flatten().tolist()
    # snapshot t holds the state after t + 1 steps: snapshot 0 is one step
    # from the working state (the one-step bound), the others at most T <= 64
    for t in range(T):
        st_ids = spec_ids[:, t].tolist()
        assert max_rel_l2(to_np(spec.ssm[st_ids]), ospec.ssm[st_ids], shape.dv * shape.dk) <= state_tol(t + 1), t
    assert conv_bits_equal(spec.conv[sids], ospec.conv[sids])
    # unused spec slots keep their sentinel bytes
    unused = [s for s in range(B * T + 3) if s not in sids]
    assert torch.all(spec.ssm[unused] == 12345.5) and torch.all(spec.conv[unused] == -77.0)

    # commit: accepted length uniform in 1..T (plus one explicit 0)
    L = synth.accept_lengths(B, T, st.gen)
    L[0] = 0
    spec_snapshot = StatePool(spec.ssm.clone(), spec.conv.clone())
    gdn.spec_commit(st.dims, spec, st.pool, spec_ids.cuda(), L.cuda(), ids.cuda())
    # the oracle commit is a bit copy; apply it to the GPU's own snapshots
    exp = oracle.Pool(to_np(work_before[0]), to_np(work_before[1]))
    oracle.spec_commit(st.od, oracle.Pool(to_np(spec_snapshot.ssm), to_np(spec_snapshot.conv)),
                       exp, spec_ids.numpy(), L.numpy(), ids.numpy())
    torch.cuda.synchronize()
    assert_pool_bits_equal(st.pool, exp)
    # and against the oracle's own L decode steps (state within tolerance)
    ref = oracle.Pool(to_np(work_before[0]), to_np(work_before[1]))
    for r in range(B):
        for t in range(int(L[r])):
            oracle.decode_step(st.od, ref, st.oparams, ids[r:r + 1].numpy(), to_np(qkv[r:r + 1, t]),
                               to_np(a[r:r + 1, t]), to_np(b[r:r + 1, t]))
    for r in range(B):
        s_ = int(ids[r])
        assert max_rel_l2(to_np(st.pool.ssm[s_]), ref.ssm[s_], shape.dv * shape.dk) <= state_tol(int(L[r]))
    used = ids.tolist()
    assert conv_bits_equal(st.pool.conv[used], ref.conv[used])


def test_verify_bad_ids(cuda):
    shape = synth.QWEN
    st = Setup(shape, seed=31, num_slots=10)
    B, T = 3, 2
    ids = torch.tensor([4, -1, 10], dtype=torch.int32)
    spec = _spec_pool(st, 6)
    spec_ids = torch.tensor([[0, -1], [1, 2], [3, 9]], dtype=torch.int32)
    qkv, a, b = st.tokens((B, T))
    out = torch.empty((B, T, 32, 128), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.spec_verify(st.dims, st.pool, spec, st.params, ids.cuda(), spec_ids.cuda(), qkv.cuda(),
                    a.cuda(), b.cuda(), out, err)
    torch.cuda.synchronize()
    assert int(err.item()) == gdn.DEV_ERR_SLOT_OOB
    assert torch.all(out[1:] == 0)
    # request 0 wrote snapshot 0 only; slots 1..5 untouched
    assert not torch.all(spec.ssm[0] == 12345.5)
    assert torch.all(spec.ssm[1:] == 12345.5)
    L = torch.tensor([2, 1, 1], dtype=torch.int32)  # L=2 for request 0 reads spec_ids[0][1] = -1
    gdn.spec_commit(st.dims, spec, st.pool, spec_ids.cuda(), L.cuda(), ids.cuda(), err)
    L_bad = torch.tensor([5, 0, 0], dtype=torch.int32)
    err2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    before = st.pool.ssm.clone()
    gdn.spec_commit(st.dims, spec, st.pool, spec_ids.cuda(), L_bad.cuda(), ids.cuda(), err2)
    torch.cuda.synchronize()
    assert int(err2.item()) == gdn.DEV_ERR_SLOT_OOB
    assert torch.equal(st.pool.ssm, before)
