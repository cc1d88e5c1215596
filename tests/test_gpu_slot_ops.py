"""GPU slot copy-on-write and zeroing: bit-exact against the oracle, with
canary slots that must stay untouched."""
import pytest
import torch

import hybrid_linear_attention_gdn_gb300 as gdn
import oracle
from hybrid_linear_attention_gdn_gb300 import StatePool, synth
from helpers import Setup, assert_pool_bits_equal, oracle_pool_of

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [synth.TINY, synth.QWEN], ids=["tiny", "qwen"])
def test_copy_between_pools_bit_exact(cuda, shape):
    n_slots = 8 if shape is synth.TINY else 24
    work = Setup(shape, seed=20, num_slots=n_slots)
    ck = Setup(shape, seed=21, num_slots=n_slots)
    src = torch.tensor([1, 4, -1, 2, 6, 3], dtype=torch.int32)
    dst = torch.tensor([6, 0, 3, n_slots, 2, -1], dtype=torch.int32)
    err_dev = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.slot_copy(work.dims, ck.pool, work.pool, src.cuda(), dst.cuda(), err_dev)
    err = oracle.slot_copy(work.od, ck.opool, work.opool, src.numpy(), dst.numpy())
    torch.cuda.synchronize()
    assert err == oracle.ERR_SLOT_OOB and int(err_dev.item()) == gdn.DEV_ERR_SLOT_OOB
    assert_pool_bits_equal(work.pool, work.opool)
    assert_pool_bits_equal(ck.pool, ck.opool)  # the source pool is untouched


def test_copy_within_one_pool_64_pairs(cuda):
    """Copy-on-write inside one 512-slot pool: 64 random disjoint pairs."""
    shape = synth.QWEN
    st = Setup(shape, seed=22, num_slots=160)
    perm = synth.slot_ids(160, 128, st.gen)
    src, dst = perm[:64], perm[64:]
    gdn.slot_copy(st.dims, st.pool, st.pool, src.cuda(), dst.cuda())
    oracle.slot_copy(st.od, st.opool, st.opool, src.numpy(), dst.numpy())
    torch.cuda.synchronize()
    assert_pool_bits_equal(st.pool, st.opool)


@pytest.mark.parametrize("shape", [synth.TINY, synth.QWEN], ids=["tiny", "qwen"])
def test_zero(cuda, shape):
    n_slots = 8 if shape is synth.TINY else 80
    st = Setup(shape, seed=23, num_slots=n_slots)
    ids = synth.slot_ids(n_slots, min(64, n_slots - 2), st.gen)
    ids = torch.cat([ids, torch.tensor([-1, n_slots + 5], dtype=torch.int32)])
    err_dev = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.slot_zero(st.dims, st.pool, ids.cuda(), err_dev)
    err = oracle.slot_zero(st.od, st.opool, ids.numpy())
    torch.cuda.synchronize()
    assert err == oracle.ERR_SLOT_OOB and int(err_dev.item()) == gdn.DEV_ERR_SLOT_OOB
    assert_pool_bits_equal(st.pool, st.opool)
    z = ids[ids >= 0]
    z = z[z < n_slots].long()
    # +0.0, not -0.0
    assert torch.all(st.pool.ssm[z].view(torch.int32) == 0)


def test_zero_count_and_empty(cuda):
    st = Setup(synth.TINY, seed=24)
    n0 = gdn.launch_count(gdn.binding.K_SLOT_ZERO)
    gdn.slot_zero(st.dims, st.pool, torch.empty(0, dtype=torch.int32, device="cuda"))
    gdn.slot_zero(st.dims, st.pool, torch.tensor([3], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert gdn.launch_count(gdn.binding.K_SLOT_ZERO) == n0 + 1
    assert torch.all(st.pool.ssm[3] == 0) and torch.all(st.pool.conv[3] == 0)


def test_invalid_arguments_raise(cuda):
    st = Setup(synth.TINY, seed=25)
    misaligned = StatePool(st.pool.ssm.view(-1)[1:].view(-1, 1), st.pool.conv)  # 4-byte offset
    one = torch.tensor([1], dtype=torch.int32, device="cuda")
    with pytest.raises(gdn.GdnError) as e:
        gdn.slot_copy(st.dims, misaligned, st.pool, one, one)
    assert e.value.status == gdn.binding.ERR_INVALID_ARG
    odd = gdn.Dims(2, 3, 16, 16, 4, torch.float32, torch.float32)  # hv not a multiple of hk
    with pytest.raises(gdn.GdnError):
        gdn.slot_zero(odd, st.pool, one)
    big = gdn.Dims(2, 4, 32, 16, 4, torch.float32, torch.float32)  # dk=32 is not compiled in
    with pytest.raises(gdn.GdnError) as e:
        gdn.slot_zero(big, st.pool, one)
    assert e.value.status == gdn.binding.ERR_UNSUPPORTED
