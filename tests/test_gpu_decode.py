"""GPU parity for gdn_decode_step (fused conv1d update + SiLU + L2 norm + gates
+ gated delta rule + readout) against the double-precision oracle."""
import numpy as np
import pytest
import torch

import hybrid_linear_attention_gdn_gb300 as gdn
import oracle
from hybrid_linear_attention_gdn_gb300 import synth
from helpers import (assert_out_close, STATE_TOL_1, STATE_TOL_64, Setup, assert_pool_bits_equal, conv_bits_equal,
                     max_rel_l2, out_tol, to_np)

pytestmark = pytest.mark.gpu


def _step(st: Setup, ids: torch.Tensor, qkv, a, b, dev_err=None):
    dev = st.device
    B = ids.shape[0]
    out = torch.full((B, st.shape.hv, st.shape.dv), 7.0, dtype=st.shape.act_dtype, device=dev)
    gdn.decode_step(st.dims, st.pool, st.params, ids.to(dev), qkv.to(dev), a.to(dev), b.to(dev),
                    out, dev_err)
    o_ref, err = oracle.decode_step(st.od, st.opool, st.oparams, ids.numpy(), to_np(qkv),
                                    to_np(a), to_np(b))
    torch.cuda.synchronize()
    return out, o_ref, err


def _check_state(st: Setup, slots, tol):
    slots = [int(s) for s in slots]
    g = to_np(st.pool.ssm[slots])
    r = st.opool.ssm[slots]
    assert max_rel_l2(g, r, st.shape.dv * st.shape.dk) <= tol
    assert conv_bits_equal(st.pool.conv[slots], st.opool.conv[slots])


def test_tiny_eight_steps(cuda):
    """Tiny layer: batch 2, 8 consecutive decode steps on random distinct slots."""
    st = Setup(synth.TINY, seed=0)
    ids = synth.slot_ids(8, 2, st.gen)
    untouched = [s for s in range(8) if s not in ids.tolist()]
    before = st.pool.ssm[untouched].clone(), st.pool.conv[untouched].clone()
    for step in range(8):
        qkv, a, b = st.tokens((2,))
        out, o_ref, err = _step(st, ids, qkv, a, b)
        assert err == 0
        assert_out_close(out, o_ref, st.shape.dv, out_tol(st.shape))
        _check_state(st, ids.tolist(), STATE_TOL_1 if step == 0 else STATE_TOL_64)
    assert torch.equal(st.pool.ssm[untouched], before[0])
    assert torch.equal(st.pool.conv[untouched], before[1])


@pytest.mark.parametrize("B", [1, 3, 8, 16, 64, 128, 256])
def test_qwen_one_step(cuda, B):
    """Qwen3.5-shaped layer (16 QK / 32 V heads, dk=dv=128, bf16), batches from
    far below one work item per SM to many per SM (the benchmark's sweep)."""
    n_slots = max(80, B + 16)
    st = Setup(synth.QWEN, seed=1, num_slots=n_slots)
    ids = synth.slot_ids(n_slots, B, st.gen)
    untouched = [s for s in range(n_slots) if s not in ids.tolist()][:8]
    before = st.pool.ssm[untouched].clone()
    qkv, a, b = st.tokens((B,))
    out, o_ref, err = _step(st, ids, qkv, a, b)
    assert err == 0
    assert_out_close(out, o_ref, 128, out_tol(st.shape))
    _check_state(st, ids.tolist(), STATE_TOL_1)
    assert torch.equal(st.pool.ssm[untouched], before)


@pytest.mark.parametrize("path,B", [("rows", 3), ("rows", 64), ("tma", 1), ("tma", 2)])
def test_qwen_one_step_forced_kernel(cuda, monkeypatch, path, B):
    """Each decode kernel at the Qwen3.5 shape where the library would pick
    the other (per-head below a quarter item per SM, TMA-fed above)."""
    monkeypatch.setenv("GDN_DECODE_PATH", path)
    st = Setup(synth.QWEN, seed=11, num_slots=80)
    ids = synth.slot_ids(80, B, st.gen)
    n0 = gdn.launch_count(gdn.K_DECODE)
    qkv, a, b = st.tokens((B,))
    out, o_ref, err = _step(st, ids, qkv, a, b)
    assert err == 0
    assert gdn.launch_count(gdn.K_DECODE) == n0 + 1
    assert_out_close(out, o_ref, 128, out_tol(st.shape))
    _check_state(st, ids.tolist(), STATE_TOL_1)


@pytest.mark.parametrize("B", [8, 32])
def test_qwen_64_steps(cuda, B):
    st = Setup(synth.QWEN, seed=2, num_slots=40)
    ids = synth.slot_ids(40, B, st.gen)
    for step in range(64):
        qkv, a, b = st.tokens((B,))
        out, o_ref, err = _step(st, ids, qkv, a, b)
        assert err == 0
        assert_out_close(out, o_ref, 128, out_tol(st.shape))
    _check_state(st, ids.tolist(), STATE_TOL_64)


def test_padding_and_out_of_range_ids(cuda):
    st = Setup(synth.QWEN, seed=3, num_slots=12)
    ids = torch.tensor([5, -1, 12, 3, -7], dtype=torch.int32)
    err_dev = torch.zeros(1, dtype=torch.int32, device="cuda")
    qkv, a, b = st.tokens((5,))
    before = st.pool.ssm.clone(), st.pool.conv.clone()
    out, o_ref, err = _step(st, ids, qkv, a, b, dev_err=err_dev)
    assert err == oracle.ERR_SLOT_OOB
    assert int(err_dev.item()) == gdn.DEV_ERR_SLOT_OOB
    o = to_np(out)
    assert np.all(o[[1, 2, 4]] == 0)
    assert_out_close(out, o_ref, 128, out_tol(st.shape))
    others = [s for s in range(12) if s not in (5, 3)]
    assert torch.equal(st.pool.ssm[others], before[0][others])
    assert torch.equal(st.pool.conv[others], before[1][others])
    _check_state(st, [5, 3], STATE_TOL_1)


@pytest.mark.parametrize("shape,B", [
    (synth.QWEN, 20),
    (synth.QWEN.replace(act="f32", conv="f32", hk=4, hv=8), 40),
    (synth.QWEN.replace(conv="f32", hk=4, hv=16, dv=64), 40),
], ids=["qwen_b20", "f32_g2", "bf16_f32hist_g4_dv64"])
def test_persistent_path_with_padding(cuda, shape, B):
    """Batches with at least one (request, QK head) item per SM run the
    persistent TMA-fed kernel; padding and out-of-range ids inside it."""
    n_slots = B + 6
    st = Setup(shape, seed=10, num_slots=n_slots)
    ids = synth.slot_ids(n_slots, B, st.gen)
    ids[3] = -1
    ids[B - 2] = n_slots + 3
    err_dev = torch.zeros(1, dtype=torch.int32, device="cuda")
    before = st.pool.ssm.clone(), st.pool.conv.clone()
    for step in range(3):
        qkv, a, b = st.tokens((B,))
        out, o_ref, err = _step(st, ids, qkv, a, b, dev_err=err_dev)
        assert err == oracle.ERR_SLOT_OOB
        assert int(err_dev.item()) == gdn.DEV_ERR_SLOT_OOB
        assert torch.all(out[3] == 0) and torch.all(out[B - 2] == 0)
        assert_out_close(out, o_ref, shape.dv, out_tol(shape))
    valid = [int(s) for s in ids.tolist() if 0 <= s < n_slots]
    others = [s for s in range(n_slots) if s not in valid]
    assert torch.equal(st.pool.ssm[others], before[0][others])
    assert torch.equal(st.pool.conv[others], before[1][others])
    _check_state(st, valid, STATE_TOL_64)


def test_batch_zero_is_noop(cuda):
    st = Setup(synth.TINY, seed=4)
    before = st.pool.ssm.clone()
    n0 = gdn.launch_count(gdn.binding.K_DECODE)
    e = torch.empty(0, device="cuda")
    gdn.decode_step(st.dims, st.pool, st.params, torch.empty(0, dtype=torch.int32, device="cuda"),
                    e, e, e, e)
    torch.cuda.synchronize()
    assert gdn.launch_count(gdn.binding.K_DECODE) == n0
    assert torch.equal(st.pool.ssm, before)


def test_deterministic_and_counted(cuda):
    st = Setup(synth.QWEN, seed=5, num_slots=20)
    ids = synth.slot_ids(20, 16, st.gen).cuda()
    qkv, a, b = (t.cuda() for t in st.tokens((16,)))
    ssm0, conv0 = st.pool.ssm.clone(), st.pool.conv.clone()
    outs = []
    n0 = gdn.launch_count(gdn.binding.K_DECODE)
    for _ in range(2):
        st.pool.ssm.copy_(ssm0)
        st.pool.conv.copy_(conv0)
        out = torch.empty((16, 32, 128), dtype=torch.bfloat16, device="cuda")
        gdn.decode_step(st.dims, st.pool, st.params, ids, qkv, a, b, out)
        outs.append((out.clone(), st.pool.ssm.clone()))
    torch.cuda.synchronize()
    assert gdn.launch_count(gdn.binding.K_DECODE) == n0 + 2
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1].view(torch.int32), outs[1][1].view(torch.int32))


def test_identity_gates_keep_state_bitwise(cuda):
    """A_log = -inf and b = -inf give alpha = 1, beta = 0: the fp32 state is
    bitwise unchanged and the conv history shifts by one raw input."""
    st = Setup(synth.QWEN, seed=6, num_slots=10)
    st.params.A_log.fill_(-float("inf"))
    st.oparams.A_log[:] = -np.inf
    ids = torch.tensor([2, 7], dtype=torch.int32)
    qkv, a, _ = st.tokens((2,))
    b = torch.full((2, 32), -float("inf"), dtype=torch.bfloat16)
    before = st.pool.ssm.clone()
    out, o_ref, _ = _step(st, ids, qkv, a, b)
    assert torch.equal(st.pool.ssm.view(torch.int32), before.view(torch.int32))
    assert_out_close(out, o_ref, 128, out_tol(st.shape))
    assert conv_bits_equal(st.pool.conv[[2, 7]], st.opool.conv[[2, 7]])


def test_forget_gate_writes_outer_product(cuda):
    """a = +inf (alpha = 0) and b = +inf (beta = 1): S^T becomes v k^T."""
    st = Setup(synth.QWEN, seed=7, num_slots=6)
    ids = torch.tensor([1, 4, 0], dtype=torch.int32)
    qkv, _, _ = st.tokens((3,))
    a = torch.full((3, 32), float("inf"), dtype=torch.bfloat16)
    b = torch.full((3, 32), float("inf"), dtype=torch.bfloat16)
    out, o_ref, _ = _step(st, ids, qkv, a, b)
    _check_state(st, [1, 4, 0], STATE_TOL_1)
    assert_out_close(out, o_ref, 128, out_tol(st.shape))


def test_f32_activations_with_f32_history(cuda):
    shape = synth.QWEN.replace(act="f32", conv="f32", hk=4, hv=8)
    st = Setup(shape, seed=8, num_slots=16)
    ids = synth.slot_ids(16, 5, st.gen)
    for _ in range(3):
        qkv, a, b = st.tokens((5,))
        out, o_ref, err = _step(st, ids, qkv, a, b)
        assert_out_close(out, o_ref, 128, 1e-4)
    _check_state(st, ids.tolist(), STATE_TOL_64)


@pytest.mark.parametrize("B", [1, 5, 24])
def test_per_head_kernel_for_wide_groups(cuda, B):
    """G * dv = 512 rows per QK head is beyond the TMA-fed kernel's item size,
    so these shapes run the per-head kernel (row parts in one cluster)."""
    shape = synth.QWEN.replace(hk=2, hv=8)
    st = Setup(shape, seed=11, num_slots=B + 4)
    ids = synth.slot_ids(B + 4, B, st.gen)
    for _ in range(3):
        qkv, a, b = st.tokens((B,))
        out, o_ref, err = _step(st, ids, qkv, a, b)
        assert err == 0
        assert_out_close(out, o_ref, 128, out_tol(shape))
    _check_state(st, ids.tolist(), STATE_TOL_64)


def test_bf16_activations_with_f32_history_and_dk64(cuda):
    shape = synth.QWEN.replace(conv="f32", hk=2, hv=8, dk=64, dv=96)
    st = Setup(shape, seed=9, num_slots=16)
    ids = synth.slot_ids(16, 7, st.gen)
    for _ in range(3):
        qkv, a, b = st.tokens((7,))
        out, o_ref, err = _step(st, ids, qkv, a, b)
        assert_out_close(out, o_ref, 96, out_tol(shape))
    _check_state(st, ids.tolist(), STATE_TOL_64)
