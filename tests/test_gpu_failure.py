"""Device-side failure path without a fault: a bounded wait that nothing
satisfies expires with GDN_DEV_ERR_TIMEOUT in the caller's error word, the
kernel returns, and the context stays usable for the next call."""
import time

import pytest
import torch

import hybrid_linear_attention_gdn_gb300 as gdn
import oracle
from hybrid_linear_attention_gdn_gb300 import synth
from helpers import STATE_TOL_1, Setup, assert_out_close, max_rel_l2, out_tol, to_np

pytestmark = pytest.mark.gpu


def test_bounded_wait_expires_with_a_status_and_the_context_stays_usable(cuda):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.monotonic()
    gdn.selftest_wait_timeout(err)
    torch.cuda.synchronize()
    waited = time.monotonic() - t0
    assert int(err.item()) == gdn.DEV_ERR_TIMEOUT
    assert 0.5 < waited < 60  # the library's wait limit is one second
    # the next call on the same context runs and is correct
    shape = synth.QWEN
    st = Setup(shape, seed=160, num_slots=20)
    B = 16
    ids = synth.slot_ids(20, B, st.gen)
    qkv, a, b = st.tokens((B,))
    out = torch.empty((B, shape.hv, shape.dv), dtype=shape.act_dtype, device="cuda")
    err2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.decode_step(st.dims, st.pool, st.params, ids.cuda(), qkv.cuda(), a.cuda(), b.cuda(), out, err2)
    o_ref, e = oracle.decode_step(st.od, st.opool, st.oparams, ids.numpy(), to_np(qkv), to_np(a), to_np(b))
    torch.cuda.synchronize()
    assert int(err2.item()) == 0 and e == 0
    assert_out_close(out, o_ref, shape.dv, out_tol(shape))
    used = ids.tolist()
    assert max_rel_l2(to_np(st.pool.ssm[used]), st.opool.ssm[used], shape.dv * shape.dk) <= STATE_TOL_1
