"""gdn_chunk_prefill_noalloc against gdn_chunk_prefill.

The no-allocation entry point runs the same chunked prefill but keeps its
intermediates in the library's built-in static scratch buffer (64 MiB per GPU)
instead of a workspace the caller allocates.  It is there for callers that
cannot allocate device memory when they prefill: code hosted by a framework
that owns all device memory and hands it only input and output pointers, or a
runtime that reserved its whole memory budget at start-up.

Both calls go through the C ABI.  This file is named so that pytest collects it
last; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import hybrid_linear_attention_gdn_gb300 as gdn
from hybrid_linear_attention_gdn_gb300 import StatePool, binding, synth
from helpers import Setup

pytestmark = pytest.mark.gpu


def _ck_pool(st, n):
    p = StatePool.empty(st.dims, n, "cuda")
    p.ssm.fill_(-5.0)
    p.conv.fill_(9.0)
    return p


def _args(lens, starts):
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    sp = torch.tensor(starts, dtype=torch.int64, device="cuda")
    return cu, sp, int(sum(lens))


def test_noalloc_matches_workspace_prefill_on_two_calls(cuda):
    """Two prefill calls in a row (the second continues the same sequences, so
    it finds the first call's leftovers in the shared scratch): outputs, final
    states and checkpoints match the workspace entry point's."""
    shape = synth.QWEN
    ref = Setup(shape, seed=50, num_slots=6)    # regular entry point
    noa = Setup(shape, seed=50, num_slots=6)    # no-allocation entry point
    ck_ref, ck_noa = _ck_pool(ref, 24), _ck_pool(noa, 24)
    ids = torch.tensor([4, 0, 2], dtype=torch.int32, device="cuda")
    ck_ids = torch.arange(24, dtype=torch.int32, device="cuda").reshape(3, 8)
    calls = [([300, 700, 64], [0, 128, 0]), ([200, 100, 900], [300, 828, 64])]
    n0 = binding.launch_count(binding.K_PREFILL)
    for lens, starts in calls:
        cu, sp, total = _args(lens, starts)
        qkv, a, b = (t.cuda() for t in ref.tokens((total,)))
        out_ref = torch.empty((total, 32, 128), dtype=torch.bfloat16, device="cuda")
        out_noa = torch.empty_like(out_ref)
        ws = torch.empty(gdn.chunk_prefill_workspace_size(ref.dims, 3, total), dtype=torch.uint8,
                         device="cuda")
        gdn.chunk_prefill(ref.dims, ref.pool, ck_ref, ref.params, ids, cu, sp, total, ck_ids, 256,
                          qkv, a, b, out_ref, ws)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        gdn.chunk_prefill_noalloc(noa.dims, noa.pool, ck_noa, noa.params, ids, cu, sp, total, ck_ids,
                                  256, qkv, a, b, out_noa, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        # the same deterministic kernels on the same inputs: bit for bit
        assert torch.equal(out_noa.view(torch.int16), out_ref.view(torch.int16))
        assert torch.equal(noa.pool.ssm.view(torch.int32), ref.pool.ssm.view(torch.int32))
        assert torch.equal(noa.pool.conv.view(torch.int16), ref.pool.conv.view(torch.int16))
        assert torch.equal(ck_noa.ssm.view(torch.int32), ck_ref.ssm.view(torch.int32))
        assert torch.equal(ck_noa.conv.view(torch.int16), ck_ref.conv.view(torch.int16))
    assert binding.launch_count(binding.K_PREFILL) == n0 + 4


def test_noalloc_rejects_a_call_beyond_the_scratch(cuda):
    shape = synth.QWEN
    st = Setup(shape, seed=51, num_slots=2)
    total = 2100  # 2100 x 33,024 bytes of intermediates > 64 MiB
    assert gdn.chunk_prefill_workspace_size(st.dims, 1, total) > binding.NOALLOC_SCRATCH_BYTES
    cu, sp, _ = _args([total], [0])
    qkv, a, b = (t.cuda() for t in st.tokens((total,)))
    out = torch.empty((total, 32, 128), dtype=torch.bfloat16, device="cuda")
    ck = _ck_pool(st, 1)
    before = st.pool.ssm.clone()
    n0 = binding.launch_count(binding.K_PREFILL)
    with pytest.raises(gdn.GdnError) as e:
        gdn.chunk_prefill_noalloc(st.dims, st.pool, ck, st.params,
                                  torch.tensor([1], dtype=torch.int32, device="cuda"), cu, sp,
                                  total, torch.full((1, 8), -1, dtype=torch.int32, device="cuda"),
                                  256, qkv, a, b, out)
    assert e.value.status == binding.ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert binding.launch_count(binding.K_PREFILL) == n0
    assert torch.equal(st.pool.ssm, before)
