"""GPU readout epilogue (gated RMS norm) against the oracle: on random rows of
every supported width and on the real readout of a decode step, in place and
out of place."""
import numpy as np
import pytest
import torch

import hybrid_linear_attention_gdn_gb300 as gdn
import oracle
from hybrid_linear_attention_gdn_gb300 import synth
from helpers import Setup, assert_out_close, odims, out_tol, to_np

pytestmark = pytest.mark.gpu


def _rows(shape, n_tok, seed):
    g = synth.generator(seed)
    o = synth.normal((n_tok, shape.hv, shape.dv), 0.7, g, shape.act_dtype)
    z = synth.normal((n_tok, shape.hv, shape.dv), 1.5, g, shape.act_dtype)
    w = 1.0 + synth.normal((shape.dv,), 0.2, g)
    return o, z, w


@pytest.mark.parametrize("form", ["stream", "rows"])
@pytest.mark.parametrize("shape,n_tok", [
    (synth.QWEN, 64), (synth.QWEN, 3), (synth.TINY, 37),
    (synth.QWEN.replace(hk=2, hv=8, dk=64, dv=64), 11),
    (synth.QWEN.replace(act="f32", conv="f32", hk=1, hv=5), 7),
    (synth.QWEN.replace(act="f32", conv="f32", hk=4, hv=8, dv=200), 5),
], ids=["qwen_b64", "qwen_3", "tiny_f32_dv16", "dv64", "f32_dv128_ragged", "f32_dv200_ragged"])
def test_gated_rmsnorm_vs_oracle(cuda, monkeypatch, form, shape, n_tok):
    """Both forms (the streamed one takes rows of 64 to 512 bytes; dv 200 in
    fp32 goes to the general one either way), rows not a whole number of the
    streamed form's groups included."""
    monkeypatch.setenv("GDN_EPILOGUE", form)
    o, z, w = _rows(shape, n_tok, 60 + n_tok)
    od = odims(shape)
    ref = oracle.gated_rmsnorm(od, to_np(o), to_np(z), w.double().numpy(), eps=1e-6)
    o_d, z_d, w_d = o.cuda(), z.cuda(), w.cuda()
    y = torch.full_like(o_d, 5.0)
    n0 = gdn.launch_count(gdn.K_GATED_RMSNORM)
    gdn.gated_rmsnorm(gdn.Dims.of(shape), o_d, z_d, w_d, 1e-6, y)
    torch.cuda.synchronize()
    assert gdn.launch_count(gdn.K_GATED_RMSNORM) == n0 + 1
    assert torch.equal(o_d.cpu(), o)  # out of place: o untouched
    assert_out_close(y, ref, shape.dv, out_tol(shape))
    # in place gives the same bits
    gdn.gated_rmsnorm(gdn.Dims.of(shape), o_d, z_d, w_d, 1e-6)
    torch.cuda.synchronize()
    assert torch.equal(o_d, y)


def test_decode_readout_then_epilogue(cuda):
    """The epilogue on a decode step's own output, both against the oracle's
    decode step followed by the oracle's epilogue."""
    shape = synth.QWEN
    st = Setup(shape, seed=61, num_slots=80)
    B = 64
    ids = synth.slot_ids(80, B, st.gen)
    qkv, a, b = st.tokens((B,))
    out = torch.empty((B, shape.hv, shape.dv), dtype=shape.act_dtype, device="cuda")
    gdn.decode_step(st.dims, st.pool, st.params, ids.cuda(), qkv.cuda(), a.cuda(), b.cuda(), out)
    _, z, w = _rows(shape, B, 62)
    gdn.gated_rmsnorm(st.dims, out, z.cuda(), w.cuda(), 1e-6)
    o_ref, err = oracle.decode_step(st.od, st.opool, st.oparams, ids.numpy(), to_np(qkv), to_np(a),
                                    to_np(b))
    assert err == 0
    y_ref = oracle.gated_rmsnorm(st.od, o_ref, to_np(z), w.double().numpy(), eps=1e-6)
    torch.cuda.synchronize()
    # the decode output is rounded to bf16 before the norm: that rounding
    # (about 2^-9 per element, an error the size of the stated bound) passes
    # through the scale-free norm on top of each call's own error
    assert_out_close(out, y_ref, shape.dv, 2 * out_tol(shape))


def test_gated_rmsnorm_zero_rows_and_empty(cuda):
    shape = synth.QWEN
    o, z, w = _rows(shape, 4, 63)
    o[1] = 0.0
    o_d = o.cuda()
    gdn.gated_rmsnorm(gdn.Dims.of(shape), o_d, z.cuda(), w.cuda(), 1e-6)
    torch.cuda.synchronize()
    assert torch.all(o_d[1] == 0) and torch.all(torch.isfinite(o_d.float()))
    n0 = gdn.launch_count(gdn.K_GATED_RMSNORM)
    e = torch.empty((0, shape.hv, shape.dv), dtype=shape.act_dtype, device="cuda")
    gdn.gated_rmsnorm(gdn.Dims.of(shape), e, e, w.cuda(), 1e-6)
    assert gdn.launch_count(gdn.K_GATED_RMSNORM) == n0
    with pytest.raises(gdn.GdnError):
        gdn.gated_rmsnorm(gdn.Dims.of(shape), o_d, z.cuda(), w.cuda(), -1.0)


def test_gated_rmsnorm_32768_tokens_sampled_rows(cuda):
    """The benchmark's launch: 32768 tokens x 32 heads in place; 4096 sampled
    (token, head) rows against the oracle (the norm is per row)."""
    shape = synth.QWEN
    n_tok = 32768
    o, z, w = _rows(shape, n_tok, 64)
    o_d = o.cuda()
    gdn.gated_rmsnorm(gdn.Dims.of(shape), o_d, z.cuda(), w.cuda(), 1e-6)
    torch.cuda.synchronize()
    g = synth.generator(65)
    tok = torch.randint(0, n_tok, (4096,), generator=g)
    head = torch.randint(0, shape.hv, (4096,), generator=g)
    one = odims(shape.replace(hk=1, hv=1))
    ref = oracle.gated_rmsnorm(one, to_np(o[tok, head])[:, None, :], to_np(z[tok, head])[:, None, :],
                               w.double().numpy(), eps=1e-6)
    got = o_d.cpu()[tok, head][:, None, :]
    assert_out_close(got, ref, shape.dv, out_tol(shape))


def _prefill_case(st, lens, starts, blk, seed, n_slots=12):
    n = len(lens)
    ids = synth.slot_ids(n_slots, n, st.gen)
    max_ck = max(1, max((s + L) // blk - s // blk for s, L in zip(starts, lens)))
    ck_ids = torch.arange(n * max_ck, dtype=torch.int32).reshape(n, max_ck)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    sp = torch.tensor(starts, dtype=torch.int64)
    total = int(cu[-1])
    qkv, a, b = st.tokens((total,))
    _, z, w = _rows(st.shape, total, seed)
    return ids, ck_ids, n * max_ck, cu, sp, total, qkv, a, b, z, w


@pytest.mark.parametrize("path", ["tc", "cuda"])
def test_prefill_gated_vs_oracle_and_plain_prefill(cuda, monkeypatch, path):
    """gdn_chunk_prefill_gated: y against the oracle's token-by-token prefill
    followed by the oracle's gated RMS norm; state, checkpoints and conv
    histories bit for bit those of gdn_chunk_prefill.  path "tc": the tf32
    tensor-core prefill with the epilogue fused into its output; "cuda": the
    fp32 prefill, then the standalone epilogue in place (bit for bit the two
    calls)."""
    from hybrid_linear_attention_gdn_gb300 import StatePool
    from helpers import PREFILL_TOL, conv_bits_equal, max_rel_l2, prefill_state_tol
    if path == "cuda":
        monkeypatch.setenv("GDN_PREFILL_PATH", "cuda")
    shape = synth.QWEN
    lens, starts, blk = [200, 70, 513], [0, 37, 256], 256
    st = Setup(shape, seed=63, num_slots=12)
    twin = Setup(shape, seed=63, num_slots=12)  # the same pool, for the plain prefill
    ids, ck_ids, n_ck, cu, sp, total, qkv, a, b, z, w = _prefill_case(st, lens, starts, blk, 64)
    ck, ck2 = (StatePool.empty(st.dims, n_ck, "cuda") for _ in range(2))
    ck.ssm.fill_(-5.0); ck.conv.fill_(9.0); ck2.ssm.fill_(-5.0); ck2.conv.fill_(9.0)
    nbytes = gdn.chunk_prefill_workspace_size(st.dims, len(lens), total)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device="cuda")
    y = torch.full((total, shape.hv, shape.dv), 3.0, dtype=shape.act_dtype, device="cuda")
    o = torch.full_like(y, 3.0)
    z_d, w_d = z.cuda(), w.cuda()
    gdn.chunk_prefill_gated(st.dims, st.pool, ck, st.params, ids.cuda(), cu.cuda(), sp.cuda(), total,
                            ck_ids.cuda(), blk, qkv.cuda(), a.cuda(), b.cuda(), z_d, w_d, 1e-6, y, ws)
    gdn.chunk_prefill(twin.dims, twin.pool, ck2, twin.params, ids.cuda(), cu.cuda(), sp.cuda(), total,
                      ck_ids.cuda(), blk, qkv.cuda(), a.cuda(), b.cuda(), o, ws)
    ock = oracle.Pool(np.full((n_ck, shape.hv, shape.dv, shape.dk), -5.0),
                      np.full((n_ck, shape.w - 1, shape.channels), 9.0))
    o_ref, err = oracle.prefill(st.od, st.opool, ock, st.oparams, ids.numpy(), cu.numpy(), sp.numpy(),
                                ck_ids.numpy(), blk, to_np(qkv), to_np(a), to_np(b))
    assert err == 0
    y_ref = oracle.gated_rmsnorm(st.od, o_ref, to_np(z), w.double().numpy(), eps=1e-6)
    torch.cuda.synchronize()
    # The norm maps every readout row to unit RMS, so the readout's error,
    # absolute in scale (tf32 operands), becomes relative on rows whose
    # readout is small: each y row's excess is weighted by its readout row's
    # norm over the RMS row norm (at most 1), the prefill's own row floor
    # carried through the norm.  The fused epilogue normalises the fp32
    # readout (the stated bound); the separate one reads the readout rounded
    # to bf16 (up to 2^-8 of a row) and adds its own arithmetic.
    on = np.linalg.norm(o_ref.reshape(-1, shape.dv), axis=1)
    weight = np.minimum(1.0, on / np.sqrt(np.mean(on ** 2)))
    tol = PREFILL_TOL if path == "tc" else 2 * PREFILL_TOL
    assert_out_close(y, y_ref, shape.dv, tol, row_tol=tol + (0.0 if path == "tc" else 2.0 ** -8),
                     row_weight=weight)
    assert torch.equal(st.pool.ssm.view(torch.int32), twin.pool.ssm.view(torch.int32))
    assert torch.equal(st.pool.conv.view(torch.int16), twin.pool.conv.view(torch.int16))
    assert torch.equal(ck.ssm.view(torch.int32), ck2.ssm.view(torch.int32))
    assert torch.equal(ck.conv.view(torch.int16), ck2.conv.view(torch.int16))
    used = ids.tolist()
    assert max_rel_l2(to_np(st.pool.ssm[used]), st.opool.ssm[used], shape.dv * shape.dk) <= \
        prefill_state_tol(shape, path)
    assert conv_bits_equal(st.pool.conv[used], st.opool.conv[used])
    if path == "cuda":
        gdn.gated_rmsnorm(st.dims, o, z_d, w_d, 1e-6)
        torch.cuda.synchronize()
        assert torch.equal(o.view(torch.int16), y.view(torch.int16))
