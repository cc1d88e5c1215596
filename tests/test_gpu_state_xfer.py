"""GPU index-update commit and state pack / unpack: bit-exact against the
oracle, plus verify-into-the-working-pool followed by the index commit, which
must leave each request on the state of its L accepted decode steps."""
import numpy as np
import pytest
import torch

import hybrid_linear_attention_gdn_gb300 as gdn
import oracle
from hybrid_linear_attention_gdn_gb300 import synth
from helpers import Setup, assert_pool_bits_equal, conv_bits_equal, max_rel_l2, state_tol, to_np

pytestmark = pytest.mark.gpu


def _commit_case(B, T, gen, n_slots):
    """Distinct slot ids, some padded spec entries, accept lengths over the
    whole range including invalid ones."""
    perm = synth.slot_ids(n_slots, B * (T + 1), gen)
    slots = perm[:B].clone()
    spec = perm[B:].reshape(B, T).clone()
    L = synth.accept_lengths(B, T, gen)
    # every fifth request: accept nothing; every seventh: a padded snapshot
    # that is accepted (an error); every eleventh: a length out of range
    for r in range(B):
        if r % 5 == 0:
            L[r] = 0
        if r % 7 == 3:
            spec[r, int(L[r]) - 1 if L[r] > 0 else 0] = -1
        if r % 11 == 6:
            L[r] = T + 1 if r % 2 else -2
        if r % 13 == 9 and 0 <= L[r] < T:
            spec[r, T - 1] = -1  # padding that is not accepted passes through
    return slots, spec, L


@pytest.mark.parametrize("B,T", [(1, 1), (5, 3), (300, 8), (129, 16)])
def test_commit_index_bit_exact(cuda, B, T):
    gen = synth.generator(40 + B)
    slots, spec, L = _commit_case(B, T, gen, B * (T + 1) + 7)
    ref_slots, ref_freed, ref_err = oracle.commit_index(spec.numpy(), L.numpy(), slots.numpy())
    d_slots = slots.cuda()
    d_freed = torch.full((B, T), 777, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    n0 = gdn.launch_count(gdn.K_COMMIT_INDEX)
    gdn.spec_commit_index(spec.cuda(), L.cuda(), d_slots, d_freed, err)
    torch.cuda.synchronize()
    assert gdn.launch_count(gdn.K_COMMIT_INDEX) == n0 + 1
    assert np.array_equal(d_slots.cpu().numpy(), ref_slots)
    assert np.array_equal(d_freed.cpu().numpy(), ref_freed)
    assert int(err.item()) == ref_err
    assert (ref_err != 0) == any(r % 7 == 3 or r % 11 == 6 for r in range(B) if L[r] != 0)


def test_commit_index_empty_batch(cuda):
    e = torch.empty((0, 4), dtype=torch.int32, device="cuda")
    n0 = gdn.launch_count(gdn.K_COMMIT_INDEX)
    gdn.spec_commit_index(e, e[:, 0], e[:, 0], e)
    assert gdn.launch_count(gdn.K_COMMIT_INDEX) == n0


@pytest.mark.parametrize("B,T,path", [(16, 8, None), (24, 4, "tma"), (5, 6, "rows")],
                         ids=["b16_t8", "b24_t4_persistent", "b5_t6_per_head"])
def test_verify_in_place_then_commit_index(cuda, monkeypatch, B, T, path):
    """The snapshots live in the working pool itself: after the index commit
    each request's slot holds the state of its first L draft tokens, the old
    working slot is untouched, and the freed list names every other slot."""
    if path:
        monkeypatch.setenv("GDN_DECODE_PATH", path)
    shape = synth.QWEN
    n_slots = B * (T + 1) + 6
    st = Setup(shape, seed=41, num_slots=n_slots)
    perm = synth.slot_ids(n_slots, B * (T + 1), st.gen)
    ids = perm[:B].clone()
    spec_ids = perm[B:].reshape(B, T).clone()
    qkv, a, b = st.tokens((B, T))
    before = st.pool.ssm.clone(), st.pool.conv.clone()
    out = torch.empty((B, T, shape.hv, shape.dv), dtype=shape.act_dtype, device="cuda")
    gdn.spec_verify(st.dims, st.pool, st.pool, st.params, ids.cuda(), spec_ids.cuda(),
                    qkv.cuda(), a.cuda(), b.cuda(), out)
    L = synth.accept_lengths(B, T, st.gen)
    L[0] = 0
    d_slots = ids.cuda()
    freed = torch.empty((B, T), dtype=torch.int32, device="cuda")
    gdn.spec_commit_index(spec_ids.cuda(), L.cuda(), d_slots, freed)
    ref_slots, ref_freed, ref_err = oracle.commit_index(spec_ids.numpy(), L.numpy(), ids.numpy())
    torch.cuda.synchronize()
    assert ref_err == 0
    assert np.array_equal(d_slots.cpu().numpy(), ref_slots)
    assert np.array_equal(freed.cpu().numpy(), ref_freed)
    # the pre-draft working slots were only read
    old = ids.long()
    assert torch.equal(st.pool.ssm[old], before[0][old])
    assert torch.equal(st.pool.conv[old], before[1][old])
    # the adopted slots hold the oracle's L decode steps from the old state
    ref = oracle.Pool(to_np(before[0]), to_np(before[1]))
    for r in range(B):
        for t in range(int(L[r])):
            oracle.decode_step(st.od, ref, st.oparams, ids[r:r + 1].numpy(),
                               to_np(qkv[r:r + 1, t]), to_np(a[r:r + 1, t]), to_np(b[r:r + 1, t]))
    new = ref_slots.tolist()
    for r in range(B):
        assert max_rel_l2(to_np(st.pool.ssm[new[r]]), ref.ssm[int(ids[r])],
                          shape.dv * shape.dk) <= state_tol(int(L[r]))
    assert conv_bits_equal(st.pool.conv[new], ref.conv[ids.tolist()])
    # every slot the request held is either its new working slot or freed
    held = torch.cat([ids[:, None], spec_ids], 1)
    got = torch.cat([torch.from_numpy(ref_slots)[:, None], freed.cpu()], 1)
    assert torch.equal(held.sort(1).values, got.sort(1).values)


def _records(staging: torch.Tensor, dims: gdn.Dims, shape, n):
    """Split packed records into their SSM and conv halves (bit views)."""
    rec = gdn.state_record_bytes(dims)
    raw = staging.cpu()[: n * rec].view(n, rec)
    ssm_b = shape.hv * shape.dv * shape.dk * 4
    ssm = raw[:, :ssm_b].contiguous().view(torch.int32)
    conv = raw[:, ssm_b:].contiguous()
    conv = conv.view(torch.int16 if shape.conv_dtype == torch.bfloat16 else torch.int32)
    return ssm.reshape(n, -1), conv.reshape(n, -1)


def _bits(ref: np.ndarray, dtype) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(ref)).to(dtype)
    iv = torch.int16 if dtype == torch.bfloat16 else torch.int32
    return t.view(iv).reshape(ref.shape[0], -1)


@pytest.mark.parametrize("shape", [synth.TINY, synth.QWEN], ids=["tiny", "qwen"])
def test_pack_then_unpack_bit_exact(cuda, shape):
    n_slots = 12 if shape is synth.TINY else 40
    src = Setup(shape, seed=42, num_slots=n_slots)
    dst = Setup(shape, seed=43, num_slots=n_slots)
    ids = synth.slot_ids(n_slots, 9, src.gen)
    ids = torch.cat([ids[:4], torch.tensor([-1], dtype=torch.int32), ids[4:],
                     torch.tensor([n_slots + 3], dtype=torch.int32)])
    n = ids.shape[0]
    rec = gdn.state_record_bytes(src.dims)
    assert rec == (shape.hv * shape.dv * shape.dk * 4
                   + (shape.w - 1) * shape.channels * shape.conv_dtype.itemsize)
    staging = torch.full((n * rec + 64,), 0xAB, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    n0 = gdn.launch_count(gdn.K_STATE_PACK)
    gdn.state_pack(src.dims, src.pool, ids.cuda(), staging, err)
    r_ssm, r_conv, r_err = oracle.state_pack(src.od, src.opool, ids.numpy())
    torch.cuda.synchronize()
    assert int(err.item()) == r_err == gdn.DEV_ERR_SLOT_OOB
    g_ssm, g_conv = _records(staging, src.dims, shape, n)
    assert torch.equal(g_ssm, _bits(r_ssm, torch.float32))
    assert torch.equal(g_conv, _bits(r_conv, shape.conv_dtype))
    assert torch.all(staging[n * rec:].cpu() == 0xAB)  # nothing past the last record
    assert_pool_bits_equal(src.pool, src.opool)  # the source is only read

    # unpack into another pool at other ids (with a skip and an out-of-range id)
    dids = synth.slot_ids(n_slots, n, dst.gen)
    dids[4] = -1
    dids[n - 1] = -5 if shape is synth.TINY else n_slots
    err2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.state_unpack(dst.dims, staging, dst.pool, dids.cuda(), err2)
    u_err = oracle.state_unpack(dst.od, r_ssm, r_conv, dst.opool, dids.numpy())
    torch.cuda.synchronize()
    assert gdn.launch_count(gdn.K_STATE_PACK) == n0 + 2
    assert int(err2.item()) == u_err
    assert u_err == gdn.DEV_ERR_SLOT_OOB
    assert_pool_bits_equal(dst.pool, dst.opool)
    # round trip: the moved slots now equal their sources bit for bit
    for i in range(n):
        s, d = int(ids[i]), int(dids[i])
        if 0 <= s < n_slots and 0 <= d < n_slots:
            assert torch.equal(dst.pool.ssm[d], src.pool.ssm[s])
            assert torch.equal(dst.pool.conv[d], src.pool.conv[s])


def test_pack_rejects_short_staging(cuda):
    st = Setup(synth.TINY, seed=44)
    ids = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    rec = gdn.state_record_bytes(st.dims)
    short = torch.zeros(2 * rec - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(gdn.GdnError) as e:
        gdn.state_pack(st.dims, st.pool, ids, short)
    assert e.value.status == gdn.binding.ERR_INVALID_ARG
    with pytest.raises(gdn.GdnError):
        gdn.state_unpack(st.dims, short, st.pool, ids)
