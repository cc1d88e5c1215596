"""Where the tensor-core prefill's tolerances come from (CPU only).

The workload fixes the intra-chunk WY/UT contractions of the chunked prefill
as bf16 products with fp32 accumulation.  This model evaluates the chunk form
(the Gated DeltaNet chunkwise WY/UT form, Yang et al., NeurIPS 2024, with the
gated decay) in float64 twice on the workload's distributions: exactly, and
with every contraction operand rounded to bf16 (q^, k^, v, T, S, the decayed
K S^T, the masked Q K^T, Delta) and the output rounded to bf16.  The gap between
the two is the error that bf16 operands alone cause; the GPU bounds in
tests/helpers.py sit above it:

  output tensor relative L2      model ~4.0e-3   bound PREFILL_TC_TOL (5e-3)
  worst RMS-floored output row    model ~1.1e-2   bound PREFILL_TC_ROW_TOL (1.5e-2)
  worst state / checkpoint matrix model ~5.8e-3   bound PREFILL_TC_STATE_TOL (1e-2)

(model figures: 12 V heads x 4096 tokens, 192 checkpoint matrices).  This test
runs a smaller case and checks that the model stays under the bounds with
margin, and that with no rounding it reproduces the exact form.
"""
import numpy as np
import torch

from hybrid_linear_attention_gdn_gb300 import synth
from helpers import PREFILL_TC_ROW_TOL, PREFILL_TC_STATE_TOL, PREFILL_TC_TOL


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x)).float().bfloat16().double().numpy()


def _features(shape, seed, n_tok):
    g = synth.generator(seed)
    conv_w, A_log, _ = synth.params(shape, g)
    ssm, conv = synth.pool(shape, g, 1)
    qkv, a, b = synth.tokens(shape, g, (n_tok,))
    x = np.concatenate([conv[0].double().numpy(), qkv.double().numpy()], 0)
    w = conv_w.double().numpy()
    W = shape.w

    def conv_silu(c0, n):
        y = sum(w[c0:c0 + n, j][None, :] * x[j:j + n_tok, c0:c0 + n] for j in range(W))
        return y / (1.0 + np.exp(-y))

    return conv_silu, A_log.double().numpy(), a.double().numpy(), b.double().numpy(), ssm[0].double().numpy()


def _chunk_form(q, k, v, g, beta, S, rounded, ckpt_every=256, C=64):
    """Chunk form over one V head; S is S^T [dv][dk].  Returns (out, checkpoints)."""
    r = _bf16 if rounded else (lambda m: m)
    q, k, v = r(q), r(k), r(v)
    n_tok = q.shape[0]
    out = np.zeros_like(v)
    cks = []
    for c0 in range(0, n_tok, C):
        sl = slice(c0, min(n_tok, c0 + C))
        n = sl.stop - sl.start
        K, Q, V, be = k[sl], q[sl], v[sl], beta[sl]
        bcum = np.cumsum(g[sl])
        diff = bcum[:, None] - bcum[None, :]
        low = np.tril(np.ones((n, n)), -1) > 0
        gam = np.where(low | np.eye(n, dtype=bool), np.exp(np.where(low | np.eye(n, dtype=bool), diff, 0.0)), 0.0)
        A = be[:, None] * (K @ K.T) * gam * low
        X = np.linalg.inv(np.eye(n) + A)
        T = X * be[None, :]
        # Delta = T V - T (diag(e^b) K S^T): the state-dependent operand is
        # formed before T is known (K S^T from the bf16 state image, scaled
        # by e^b and rounded), both products accumulate in fp32
        Sb = r(S)
        E = r(np.exp(bcum)[:, None] * (K @ Sb.T))
        D = r(T) @ V - r(T) @ E
        QK = (Q @ K.T) * gam
        out[sl] = np.exp(bcum)[:, None] * (Q @ Sb.T) + r(QK) @ r(D)
        S = np.exp(bcum[-1]) * S + r(D * np.exp(bcum[-1] - bcum)[:, None]).T @ K
        if (c0 + n) % ckpt_every == 0:
            cks.append(S.copy())
    return (r(out), cks)


def test_bf16_operand_error_model_sits_under_the_bounds():
    shape = synth.QWEN
    n_tok = 1024
    conv_silu, A_log, a, b, S0 = _features(shape, 40, n_tok)
    d_out = n_out = 0.0
    rows_err, rows_ref, st_err = [], [], []
    for h in (0, 7, 13, 20, 26, 31):
        hq = h // (shape.hv // shape.hk)
        q = conv_silu(hq * 128, 128)
        k = conv_silu(shape.hk * 128 + hq * 128, 128)
        v = conv_silu(2 * shape.hk * 128 + h * 128, 128)
        q = q / np.sqrt((q * q).sum(1, keepdims=True) + 1e-6) / np.sqrt(128.0)
        k = k / np.sqrt((k * k).sum(1, keepdims=True) + 1e-6)
        g = -np.exp(A_log[h]) * np.log1p(np.exp(a[:, h]))
        beta = 1.0 / (1.0 + np.exp(-b[:, h]))
        o_x, ck_x = _chunk_form(q, k, v, g, beta, S0[h].copy(), False)
        o_r, ck_r = _chunk_form(q, k, v, g, beta, S0[h].copy(), True)
        d_out += np.sum((o_r - o_x) ** 2)
        n_out += np.sum(o_x ** 2)
        rows_err.append(np.linalg.norm(o_r - o_x, axis=1))
        rows_ref.append(np.linalg.norm(o_x, axis=1))
        st_err += [np.linalg.norm(s1 - s0) / np.linalg.norm(s0) for s1, s0 in zip(ck_r, ck_x)]
    whole = np.sqrt(d_out / n_out)
    re, rr = np.concatenate(rows_err), np.concatenate(rows_ref)
    worst_row = float((re / np.maximum(rr, np.sqrt(np.mean(rr ** 2)))).max())
    worst_state = max(st_err)
    # the model is well above the output rounding alone and well below the bounds
    assert 3e-3 < whole < 0.9 * PREFILL_TC_TOL, whole
    assert worst_row < 0.9 * PREFILL_TC_ROW_TOL, worst_row
    assert 2e-3 < worst_state < 0.9 * PREFILL_TC_STATE_TOL, worst_state


def test_model_without_rounding_is_the_exact_form():
    """No rounding: the model's chunk form equals the token-by-token recurrence."""
    rng = np.random.default_rng(0)
    n, dk, dv = 150, 8, 6
    k = rng.standard_normal((n, dk))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    q = rng.standard_normal((n, dk)) / np.sqrt(dk)
    v = rng.standard_normal((n, dv))
    g = -rng.uniform(0.0, 2.0, n)
    beta = rng.uniform(0.0, 1.0, n)
    S0 = rng.standard_normal((dv, dk))
    out, cks = _chunk_form(q, k, v, g, beta, S0.copy(), False, ckpt_every=64, C=16)
    S = S0.copy()
    ref, ref_ck = np.zeros((n, dv)), []
    for t in range(n):
        al = np.exp(g[t])
        u = v[t] - al * S @ k[t]
        S = al * S + beta[t] * np.outer(u, k[t])
        ref[t] = S @ q[t]
        if (t + 1) % 64 == 0:
            ref_ck.append(S.copy())
    assert np.allclose(out, ref, rtol=0, atol=1e-12)
    assert len(cks) == len(ref_ck) == 2
    for a_, b_ in zip(cks, ref_ck):
        assert np.allclose(a_, b_, rtol=0, atol=1e-12)
