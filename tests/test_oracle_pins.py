"""Pins for the CPU oracle: checks against closed forms, hand-worked values,
invariants and an independent algebraic form, so that a dropped term, a wrong
sign or index, or a transposed operand in the oracle fails one of them.

No GPU is needed; the CUDA library is not involved.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from hybrid_linear_attention_gdn_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
EPS = 1e-6


def _read_golden(name):
    vals = {}
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            try:
                rows.append([float(x) for x in parts])
            except ValueError:
                vals[parts[0]] = np.array([float(x) for x in parts[1:]])
    return vals, rows


def _dims(shape):
    return oracle.Dims(shape.hk, shape.hv, shape.dk, shape.dv, shape.w)


def _tiny_setup(seed=0, shape=synth.TINY):
    g = synth.generator(seed)
    conv_w, A_log, dt_bias = synth.params(shape, g)
    ssm, conv = synth.pool(shape, g)
    pool = oracle.Pool(ssm.double().numpy(), conv.double().numpy())
    params = oracle.Params(conv_w.double().numpy(), A_log.double().numpy(),
                           dt_bias.double().numpy())
    return g, pool, params


# ---------------------------------------------------------------- delta rule

def test_golden_delta_rule_2x2():
    v, _ = _read_golden("delta_rule_2x2.txt")
    S = v["S"].reshape(2, 2)
    St, o = oracle.delta_core(S.T, v["k"], v["v"], v["q"], v["alpha"][0], v["beta"][0])
    np.testing.assert_allclose(St.T, v["S_new"].reshape(2, 2), rtol=0, atol=1e-15)
    np.testing.assert_allclose(o, v["o"], rtol=0, atol=1e-15)


def test_delta_core_identity_when_beta0_alpha1():
    rng = np.random.default_rng(1)
    St = rng.standard_normal((16, 16))
    k, v, q = rng.standard_normal((3, 16))
    St2, o = oracle.delta_core(St, k, v, q, 1.0, 0.0)
    assert np.array_equal(St2, St)
    np.testing.assert_allclose(o, St @ q, rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("alpha", [1.0, 0.7, 0.01, 0.0])
def test_delta_core_retrieves_v_for_unit_key(alpha):
    """beta = 1, |k| = 1: the updated state maps k to v exactly, for any alpha."""
    rng = np.random.default_rng(2)
    St = rng.standard_normal((24, 16))
    k = rng.standard_normal(16)
    k /= np.linalg.norm(k)
    v, q = rng.standard_normal(24), rng.standard_normal(16)
    St2, _ = oracle.delta_core(St, k, v, q, alpha, 1.0)
    np.testing.assert_allclose(St2 @ k, v, rtol=0, atol=1e-12)


def test_delta_core_forget_all():
    """alpha = 0, beta = 1: S = k v^T, o = (k.q) v."""
    rng = np.random.default_rng(3)
    St = rng.standard_normal((8, 16))
    k, q = rng.standard_normal((2, 16))
    v = rng.standard_normal(8)
    St2, o = oracle.delta_core(St, k, v, q, 0.0, 1.0)
    np.testing.assert_allclose(St2, np.outer(v, k), rtol=0, atol=1e-14)
    np.testing.assert_allclose(o, (k @ q) * v, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("seed", range(4))
def test_delta_core_matches_matrix_form(seed):
    """Brute force: alpha (I - beta k k^T) S + beta k v^T, o = S^T q, with
    explicit dk x dk matrices, against the oracle's rank-1 update."""
    rng = np.random.default_rng(10 + seed)
    dk, dv = 12, 9
    S = rng.standard_normal((dk, dv))
    k, q = rng.standard_normal((2, dk))
    v = rng.standard_normal(dv)
    alpha, beta = rng.uniform(0, 1, 2)
    S_ref = alpha * (np.eye(dk) - beta * np.outer(k, k)) @ S + beta * np.outer(k, v)
    St2, o = oracle.delta_core(S.T, k, v, q, alpha, beta)
    np.testing.assert_allclose(St2.T, S_ref, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(o, S_ref.T @ q, rtol=1e-13, atol=1e-13)


def test_readout_linear_in_q():
    rng = np.random.default_rng(4)
    St = rng.standard_normal((16, 16))
    k, v, q1, q2 = rng.standard_normal((4, 16))
    _, o1 = oracle.delta_core(St, k, v, q1, 0.8, 0.3)
    _, o2 = oracle.delta_core(St, k, v, q2, 0.8, 0.3)
    _, o12 = oracle.delta_core(St, k, v, q1 + 2 * q2, 0.8, 0.3)
    np.testing.assert_allclose(o12, o1 + 2 * o2, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------ gates / activations

def test_golden_gates():
    _, rows = _read_golden("gates.txt")
    for A_log, a, dtb, b, g_ref, alpha_ref, beta_ref in rows:
        g = oracle.gate_g(A_log, dtb, a)
        assert g == pytest.approx(g_ref, rel=1e-14, abs=1e-15)
        assert math.exp(g) == pytest.approx(alpha_ref, rel=1e-14)
        assert oracle.sigmoid(b) == pytest.approx(beta_ref, rel=1e-14)


def test_activation_invariants():
    for x in [-30.0, -3.5, -1.0, -1e-3, 0.0, 0.25, 2.0, 17.0]:
        assert oracle.sigmoid(x) + oracle.sigmoid(-x) == pytest.approx(1.0, abs=1e-15)
        assert oracle.softplus(x) - oracle.softplus(-x) == pytest.approx(x, abs=1e-12)
        assert oracle.silu(x) - oracle.silu(-x) == pytest.approx(x, abs=1e-12)
        assert oracle.silu(x) == pytest.approx(x * oracle.sigmoid(x), rel=1e-15, abs=1e-300)
    assert oracle.sigmoid(0.0) == 0.5
    assert oracle.softplus(0.0) == pytest.approx(math.log(2.0), rel=1e-15)
    assert oracle.sigmoid(-math.inf) == 0.0 and oracle.sigmoid(math.inf) == 1.0


def test_gate_sign_and_ranges():
    rng = np.random.default_rng(5)
    for _ in range(200):
        A_log, a, b = rng.uniform(-5, 5), rng.standard_normal() * 4, rng.standard_normal() * 4
        g = oracle.gate_g(A_log, 0.0, a)
        assert g <= 0.0
        assert 0.0 < oracle.sigmoid(b) < 1.0


def test_l2norm_closed_form():
    rng = np.random.default_rng(6)
    for n, scale in [(16, 1.0), (128, 1.0), (128, 128 ** -0.5), (3, 2.0)]:
        x = rng.standard_normal(n) * rng.uniform(0.01, 10)
        y = oracle.l2norm(x, scale)
        ss = float(x @ x)
        assert float(y @ y) == pytest.approx(scale ** 2 * (1 - EPS / (ss + EPS)), rel=1e-13)
        # same direction
        np.testing.assert_allclose(y * np.linalg.norm(x), x * np.linalg.norm(y), rtol=1e-12, atol=1e-14)
    v, _ = _read_golden("delta_rule_2x2.txt")  # reuse: [3,4] hand case below
    y = oracle.l2norm(np.array([3.0, 4.0]), 1.0)
    np.testing.assert_allclose(y, np.array([3.0, 4.0]) / math.sqrt(25 + EPS), rtol=1e-15)


def test_conv_orientation():
    """Weight index W-1 multiplies the newest input; index 0 the oldest."""
    shape = synth.TINY
    d = _dims(shape)
    C, W = d.channels, d.w
    rng = np.random.default_rng(7)
    hist = rng.standard_normal((W - 1, C))
    x = rng.standard_normal(C)
    w_new = np.zeros((C, W)); w_new[:, W - 1] = 1.0
    w_old = np.zeros((C, W)); w_old[:, 0] = 1.0
    y_new = oracle.conv_silu(d, hist, x, w_new)
    y_old = oracle.conv_silu(d, hist, x, w_old)
    sig = lambda z: 1.0 / (1.0 + np.exp(-z))
    np.testing.assert_allclose(y_new, x * sig(x), rtol=1e-14)
    np.testing.assert_allclose(y_old, hist[0] * sig(hist[0]), rtol=1e-14)
    # linear in the weights before the SiLU: a two-tap filter sums its taps
    w2 = w_new + 0.5 * w_old
    pre = x + 0.5 * hist[0]
    np.testing.assert_allclose(oracle.conv_silu(d, hist, x, w2), pre * sig(pre), rtol=1e-13)


# ----------------------------------------------------------- full decode step

def test_decode_identity_gates_leave_state():
    """A_log = -inf (g = -0, alpha = 1) and b = -inf (beta = 0): the SSM state is
    bitwise unchanged; the conv history still shifts by one raw input."""
    shape = synth.TINY
    d = _dims(shape)
    g, pool, params = _tiny_setup(0)
    params = oracle.Params(params.conv_w, np.full(d.hv, -np.inf), params.dt_bias)
    ids = np.array([3, 6], np.int32)
    qkv, a, _ = synth.tokens(shape, g, (2,))
    b = np.full((2, d.hv), -np.inf)
    before = pool.copy()
    out, err = oracle.decode_step(d, pool, params, ids, qkv.double().numpy(), a.double().numpy(), b)
    assert err == 0
    assert np.array_equal(pool.ssm, before.ssm)
    for r, s in enumerate(ids):
        np.testing.assert_array_equal(pool.conv[s, :-1], before.conv[s, 1:])
        np.testing.assert_array_equal(pool.conv[s, -1], qkv[r].double().numpy())
    assert np.all(np.isfinite(out))


def test_decode_retrieval_closed_form():
    """beta = 1 (b = +inf): S_new^T k_hat = v (1 - delta) + alpha S^T k_hat delta,
    delta = eps / (|k|^2 + eps), with k the conv+SiLU output of the QK head."""
    shape = synth.TINY
    d = _dims(shape)
    g, pool, params = _tiny_setup(1)
    ids = np.array([5], np.int32)
    qkv, a, _ = synth.tokens(shape, g, (1,))
    qkv, a = qkv.double().numpy(), a.double().numpy()
    b = np.full((1, d.hv), np.inf)
    s = ids[0]
    y = oracle.conv_silu(d, pool.conv[s], qkv[0], params.conv_w)
    S_before = pool.ssm[s].copy()
    oracle.decode_step(d, pool, params, ids, qkv, a, b)
    G = d.hv // d.hk
    for h in range(d.hv):
        hq = h // G
        kraw = y[d.hk * d.dk + hq * d.dk: d.hk * d.dk + (hq + 1) * d.dk]
        kh = kraw / math.sqrt(kraw @ kraw + EPS)
        delta = EPS / (kraw @ kraw + EPS)
        vv = y[2 * d.hk * d.dk + h * d.dv: 2 * d.hk * d.dk + (h + 1) * d.dv]
        alpha = math.exp(oracle.gate_g(params.A_log[h], 0.0, a[0, h]))
        lhs = pool.ssm[s, h] @ kh
        rhs = vv * (1 - delta) + alpha * (S_before[h] @ kh) * delta
        np.testing.assert_allclose(lhs, rhs, rtol=1e-11, atol=1e-12)


def test_decode_forget_gate():
    """a = +inf: g = -inf, alpha = 0; b = +inf: beta = 1 -> S^T = v k_hat^T."""
    shape = synth.TINY
    d = _dims(shape)
    g, pool, params = _tiny_setup(2)
    ids = np.array([0, 7], np.int32)
    qkv, _, _ = synth.tokens(shape, g, (2,))
    qkv = qkv.double().numpy()
    a = np.full((2, d.hv), np.inf)
    b = np.full((2, d.hv), np.inf)
    ys = [oracle.conv_silu(d, pool.conv[s], qkv[r], params.conv_w) for r, s in enumerate(ids)]
    out, _ = oracle.decode_step(d, pool, params, ids, qkv, a, b)
    G = d.hv // d.hk
    for r, s in enumerate(ids):
        y = ys[r]
        for h in range(d.hv):
            hq = h // G
            kh = oracle.l2norm(y[d.hk * d.dk + hq * d.dk:][:d.dk])
            qh = oracle.l2norm(y[hq * d.dk:][:d.dk], d.dk ** -0.5)
            vv = y[2 * d.hk * d.dk + h * d.dv:][:d.dv]
            np.testing.assert_allclose(pool.ssm[s, h], np.outer(vv, kh), rtol=1e-13, atol=1e-15)
            np.testing.assert_allclose(out[r, h], (kh @ qh) * vv, rtol=1e-12, atol=1e-14)


def test_gqa_map_repeat_interleave():
    """V head h reads QK head h // (HV/HK): perturbing QK head 1's q/k channels
    changes V heads 2, 3 only."""
    shape = synth.TINY
    d = _dims(shape)
    g, pool, params = _tiny_setup(3)
    ids = np.array([1], np.int32)
    qkv, a, b = (t.double().numpy() for t in synth.tokens(shape, g, (1,)))
    o1, _ = oracle.decode_step(d, pool.copy(), params, ids, qkv, a, b)
    qkv2 = qkv.copy()
    qkv2[0, 1 * d.dk:2 * d.dk] += 0.5                         # q of QK head 1
    qkv2[0, (d.hk + 1) * d.dk:(d.hk + 2) * d.dk] -= 0.25      # k of QK head 1
    o2, _ = oracle.decode_step(d, pool.copy(), params, ids, qkv2, a, b)
    np.testing.assert_array_equal(o1[0, :2], o2[0, :2])
    assert np.abs(o1[0, 2:] - o2[0, 2:]).min() > 0


def test_decode_padding_and_oob():
    shape = synth.TINY
    d = _dims(shape)
    g, pool, params = _tiny_setup(4)
    qkv, a, b = (t.double().numpy() for t in synth.tokens(shape, g, (3,)))
    before = pool.copy()
    out, err = oracle.decode_step(d, pool, params, np.array([-1, 8, 2], np.int32), qkv, a, b)
    assert err == oracle.ERR_SLOT_OOB
    assert np.all(out[:2] == 0)
    changed = [s for s in range(8) if not np.array_equal(pool.ssm[s], before.ssm[s])]
    assert changed == [2]
    _, err = oracle.decode_step(d, pool, params, np.array([-1, -1, -1], np.int32), qkv, a, b)
    assert err == 0


# -------------------------------------------------------------- slot ops

def test_slot_copy_zero_canary():
    shape = synth.TINY
    d = _dims(shape)
    _, pool, _ = _tiny_setup(5)
    _, other, _ = _tiny_setup(6)
    before, other_before = pool.copy(), other.copy()
    err = oracle.slot_copy(d, other, pool, [1, 4, -1, 2], [6, 0, 3, 9])
    assert err == oracle.ERR_SLOT_OOB
    np.testing.assert_array_equal(pool.ssm[6], other_before.ssm[1])
    np.testing.assert_array_equal(pool.conv[0], other_before.conv[4])
    for s in [1, 2, 3, 4, 5, 7]:
        np.testing.assert_array_equal(pool.ssm[s], before.ssm[s])
        np.testing.assert_array_equal(pool.conv[s], before.conv[s])
    np.testing.assert_array_equal(other.ssm, other_before.ssm)
    err = oracle.slot_zero(d, pool, [2, -1, 8, 5])
    assert err == oracle.ERR_SLOT_OOB
    assert np.all(pool.ssm[[2, 5]] == 0) and np.all(pool.conv[[2, 5]] == 0)
    np.testing.assert_array_equal(pool.ssm[3], before.ssm[3])


# ---------------------------------------------------- speculative verify

def test_verify_then_commit_equals_L_decode_steps():
    shape = synth.TINY
    d = _dims(shape)
    g, pool, params = _tiny_setup(7)
    B, T = 2, 5
    ids = np.array([2, 5], np.int32)
    spec = oracle.Pool(np.full((B * T, d.hv, d.dv, d.dk), 7.25),
                       np.full((B * T, d.w - 1, d.channels), -3.5))
    spec_ids = np.arange(B * T, dtype=np.int32).reshape(B, T)
    qkv, a, b = (t.double().numpy() for t in synth.tokens(shape, g, (B, T)))
    work_before = pool.copy()
    out, err = oracle.spec_verify(d, pool, spec, params, ids, spec_ids, qkv, a, b)
    assert err == 0
    assert np.array_equal(pool.ssm, work_before.ssm) and np.array_equal(pool.conv, work_before.conv)
    for L in range(0, T + 1):
        ref = work_before.copy()
        outs = []
        for t in range(L):
            o, _ = oracle.decode_step(d, ref, params, ids, qkv[:, t], a[:, t], b[:, t])
            outs.append(o)
        for t in range(L):
            np.testing.assert_array_equal(out[:, t], outs[t])
        work = work_before.copy()
        err = oracle.spec_commit(d, spec, work, spec_ids, np.full(B, L, np.int32), ids)
        assert err == 0
        np.testing.assert_array_equal(work.ssm, ref.ssm)
        np.testing.assert_array_equal(work.conv, ref.conv)


def test_commit_index_hand_worked():
    """Index-update commit, each case worked by hand: rollback (L = 0), a
    middle draft, the last draft, an accepted snapshot that was never written
    (-1) and an accept length beyond T."""
    spec_ids = np.array([[5, 6, 7], [8, 9, 10], [11, 12, 13], [14, -1, 15], [16, 17, 18]], np.int32)
    L = np.array([0, 2, 3, 2, 4], np.int32)
    slots, freed, err = oracle.commit_index(spec_ids, L, [1, 2, 3, 4, 0])
    assert err == oracle.ERR_SLOT_OOB
    np.testing.assert_array_equal(slots, [1, 9, 13, 4, 0])
    np.testing.assert_array_equal(freed, [[5, 6, 7], [2, 8, 10], [3, 11, 12], [-1, -1, -1], [-1, -1, -1]])


def test_commit_index_equals_copy_commit():
    """Adopting the accepted snapshot by index leaves the same state under the
    request's slot as the copying commit, and every slot that held a draft or
    the old working state is either the new working slot or freed, once."""
    shape = synth.TINY
    d = _dims(shape)
    g, pool, params = _tiny_setup(12)
    B, T = 2, 3
    ids = np.array([0, 1], np.int32)
    spec_ids = np.array([[2, 3, 4], [5, 6, 7]], np.int32)  # snapshots in the working pool
    qkv, a, b = (t.double().numpy() for t in synth.tokens(shape, g, (B, T)))
    _, err = oracle.spec_verify(d, pool, pool, params, ids, spec_ids, qkv, a, b)
    assert err == 0
    for L in range(T + 1):
        Ls = np.array([L, T - L], np.int32)
        copied = pool.copy()
        assert oracle.spec_commit(d, copied, copied, spec_ids, Ls, ids) == 0
        slots, freed, err = oracle.commit_index(spec_ids, Ls, ids)
        assert err == 0
        for r in range(B):
            np.testing.assert_array_equal(pool.ssm[slots[r]], copied.ssm[ids[r]])
            np.testing.assert_array_equal(pool.conv[slots[r]], copied.conv[ids[r]])
            assert sorted([slots[r], *freed[r]]) == sorted([ids[r], *spec_ids[r]])


def test_state_pack_unpack():
    """Pack gathers slots into records (zero record for -1 and, with the
    error bit, for an id outside the pool); unpacking the records into other
    slots is the slot copy."""
    shape = synth.TINY
    d = _dims(shape)
    _, pool, _ = _tiny_setup(13)
    ids = [3, -1, 6, 9, 0]
    st_ssm, st_conv, err = oracle.state_pack(d, pool, ids)
    assert err == oracle.ERR_SLOT_OOB
    for i, s in enumerate(ids):
        if 0 <= s < 8:
            np.testing.assert_array_equal(st_ssm[i], pool.ssm[s])
            np.testing.assert_array_equal(st_conv[i], pool.conv[s])
        else:
            assert np.all(st_ssm[i] == 0) and np.all(st_conv[i] == 0)
    _, dst, _ = _tiny_setup(14)
    expect = dst.copy()
    err = oracle.state_unpack(d, st_ssm, st_conv, dst, [7, 2, 1, -1, 12])
    assert err == oracle.ERR_SLOT_OOB
    assert oracle.slot_copy(d, pool, expect, [3, 6], [7, 1]) == 0
    expect.ssm[2] = 0.0  # record 1 is the zero record of id -1
    expect.conv[2] = 0.0
    np.testing.assert_array_equal(dst.ssm, expect.ssm)
    np.testing.assert_array_equal(dst.conv, expect.conv)
    # padding alone is not an error; an id outside the pool alone is, either way
    assert oracle.state_pack(d, pool, [-1, 2, -1])[2] == 0
    assert oracle.state_pack(d, pool, [2, 8])[2] == oracle.ERR_SLOT_OOB
    assert oracle.state_unpack(d, st_ssm[:2], st_conv[:2], dst, [-1, 4]) == 0
    assert oracle.state_unpack(d, st_ssm[:1], st_conv[:1], dst, [-3]) == oracle.ERR_SLOT_OOB


# ----------------------------------------------------------------- prefill

def _prefill_inputs(shape, seed, lens, starts):
    g = synth.generator(seed)
    conv_w, A_log, dt_bias = synth.params(shape, g)
    params = oracle.Params(conv_w.double().numpy(), A_log.double().numpy(), dt_bias.double().numpy())
    ssm, conv = synth.pool(shape, g)
    pool = oracle.Pool(ssm.double().numpy(), conv.double().numpy())
    ttot = int(sum(lens))
    qkv, a, b = (t.double().numpy() for t in synth.tokens(shape, g, (ttot,)))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return pool, params, cu, np.array(starts, np.int64), qkv, a, b


@pytest.mark.parametrize("chunk", [1, 4, 16, 64])
def test_chunked_form_equals_recurrence(chunk):
    shape = synth.TINY
    d = _dims(shape)
    lens, starts = [1, 37, 130, 300], [0, 64, 96, 256]
    ckb = 64
    pool, params, cu, sp, qkv, a, b = _prefill_inputs(shape, 11, lens, starts)
    ids = np.array([0, 3, 5, 6], np.int32)
    maxc = 6
    ck_ids = np.full((4, maxc), -1, np.int32)
    nxt = 0
    for n in range(4):
        for j in range(maxc):
            ck_ids[n, j] = nxt % 16
            nxt += 1
    mk = lambda: oracle.Pool(np.zeros((16, d.hv, d.dv, d.dk)), np.zeros((16, d.w - 1, d.channels)))
    p1, c1 = pool.copy(), mk()
    o1, e1 = oracle.prefill(d, p1, c1, params, ids, cu, sp, ck_ids, ckb, qkv, a, b)
    p2, c2 = pool.copy(), mk()
    o2, e2 = oracle.prefill_chunked(d, p2, c2, params, ids, cu, sp, ck_ids, ckb, chunk, qkv, a, b)
    assert e1 == e2 == 0
    scale = np.abs(o1).max()
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-10 * scale)
    np.testing.assert_allclose(p2.ssm, p1.ssm, rtol=0, atol=1e-10 * np.abs(p1.ssm).max())
    np.testing.assert_array_equal(p2.conv, p1.conv)
    np.testing.assert_allclose(c2.ssm, c1.ssm, rtol=0, atol=1e-10 * max(1.0, np.abs(c1.ssm).max()))
    np.testing.assert_array_equal(c2.conv, c1.conv)
    assert np.abs(c1.ssm).max() > 0  # some checkpoints were written


def test_prefill_equals_decode_steps_and_checkpoints():
    shape = synth.TINY
    d = _dims(shape)
    lens, starts = [200], [0]
    pool, params, cu, sp, qkv, a, b = _prefill_inputs(shape, 12, lens, starts)
    ids = np.array([4], np.int32)
    ck = oracle.Pool(np.zeros((4, d.hv, d.dv, d.dk)), np.zeros((4, d.w - 1, d.channels)))
    ref = pool.copy()
    p1 = pool.copy()
    o1, _ = oracle.prefill(d, p1, ck, params, ids, cu, sp, np.array([[2, 0, 3]], np.int32), 64, qkv, a, b)
    snaps = {}
    for t in range(200):
        o, _ = oracle.decode_step(d, ref, params, ids, qkv[t:t + 1], a[t:t + 1], b[t:t + 1])
        np.testing.assert_array_equal(o1[t], o[0])
        if (t + 1) % 64 == 0:
            snaps[(t + 1) // 64] = (ref.ssm[4].copy(), ref.conv[4].copy())
    np.testing.assert_array_equal(p1.ssm, ref.ssm)
    for blk, slot in [(1, 2), (2, 0), (3, 3)]:
        np.testing.assert_array_equal(ck.ssm[slot], snaps[blk][0])
        np.testing.assert_array_equal(ck.conv[slot], snaps[blk][1])
    # the checkpoint's conv history is the last W-1 raw inputs before the boundary
    np.testing.assert_array_equal(ck.conv[0], qkv[128 - (d.w - 1):128])


def test_prefill_resume_from_checkpoint():
    shape = synth.TINY
    d = _dims(shape)
    pool, params, cu, sp, qkv, a, b = _prefill_inputs(shape, 13, [512], [0])
    ck = oracle.Pool(np.zeros((8, d.hv, d.dv, d.dk)), np.zeros((8, d.w - 1, d.channels)))
    full = pool.copy()
    o_full, _ = oracle.prefill(d, full, ck, params, [1], cu, sp,
                               np.array([[0, 1, 2, 3]], np.int32), 128, qkv, a, b)
    # resume: copy the checkpoint at 256 (index 1) into a fresh slot, prefill the rest
    res = pool.copy()
    oracle.slot_copy(d, ck, res, [1], [6])
    ck2 = oracle.Pool(np.zeros((8, d.hv, d.dv, d.dk)), np.zeros((8, d.w - 1, d.channels)))
    o_res, _ = oracle.prefill(d, res, ck2, params, [6], np.array([0, 256], np.int32),
                              np.array([256], np.int64), np.array([[4, 5]], np.int32), 128,
                              qkv[256:], a[256:], b[256:])
    np.testing.assert_array_equal(o_res, o_full[256:])
    np.testing.assert_array_equal(res.ssm[6], full.ssm[1])
    np.testing.assert_array_equal(res.conv[6], full.conv[1])
    np.testing.assert_array_equal(ck2.ssm[4], ck.ssm[2])
    np.testing.assert_array_equal(ck2.ssm[5], ck.ssm[3])


def test_prefill_padding_and_oob():
    shape = synth.TINY
    d = _dims(shape)
    pool, params, cu, sp, qkv, a, b = _prefill_inputs(shape, 14, [10, 70], [0, 0])
    ck = oracle.Pool(np.zeros((2, d.hv, d.dv, d.dk)), np.zeros((2, d.w - 1, d.channels)))
    before = pool.copy()
    out, err = oracle.prefill(d, pool, ck, params, [-1, 2], cu, sp,
                              np.array([[0], [5]], np.int32), 64, qkv, a, b)
    assert err == oracle.ERR_SLOT_OOB      # checkpoint id 5 is outside the 2-slot pool
    assert np.all(out[:10] == 0) and np.any(out[10:] != 0)
    assert np.array_equal(pool.ssm[[0, 1, 3]], before.ssm[[0, 1, 3]])
    assert np.all(ck.ssm == 0)


@pytest.mark.parametrize("kda", [False, True])
def test_prefill_zero_decay_first_token_forgets_the_initial_state(kda):
    """a = +inf at each sequence's first token (every key channel, for KDA) of
    the even V heads: g = -inf, alpha = 0, so the state is wiped before the
    first update and those heads' outputs, final states and checkpoints do not
    depend on the initial SSM state; the odd heads' outputs (finite gates) do."""
    shape = synth.TINY
    d = _dims(shape)
    lens, starts, blk = [70, 33], [0, 50], 32
    pool, params, cu, sp, qkv, a, b = _prefill_inputs(shape, 16, lens, starts)
    if kda:
        g = synth.generator(17)
        params = oracle.Params(params.conv_w, params.A_log, synth.normal((d.hv, d.dk), 0.5, g).double().numpy())
        a = synth.normal((int(cu[-1]), d.hv, d.dk), 1.0, g).double().numpy()
    a[cu[:-1], ::2] = np.inf
    ids = np.array([3, 6], np.int32)
    ck_ids = np.array([[0, 1, 2], [3, 4, 5]], np.int32)
    run = oracle.kda_prefill if kda else oracle.prefill
    res = []
    for ssm_seed in (0, 1):
        p = pool.copy()
        p.ssm[ids] = np.random.default_rng(ssm_seed).standard_normal(p.ssm[ids].shape)
        ck = oracle.Pool(np.zeros((6, d.hv, d.dv, d.dk)), np.zeros((6, d.w - 1, d.channels)))
        out, err = run(d, p, ck, params, ids, cu, sp, ck_ids, blk, qkv, a, b)
        assert err == 0 and np.isfinite(out).all()
        res.append((out, p.ssm[ids], ck.ssm))
    (o1, s1, c1), (o2, s2, c2) = res
    np.testing.assert_array_equal(o2[:, ::2], o1[:, ::2])
    np.testing.assert_array_equal(s2[:, ::2], s1[:, ::2])
    np.testing.assert_array_equal(c2[:, ::2], c1[:, ::2])
    # (the odd heads' early outputs; their strong decays leave no trace of the
    # initial state in the final fp64 state)
    assert np.abs(o2[:, 1::2] - o1[:, 1::2]).max() > 1e-3


# ---- readout epilogue: gated RMS norm ------------------------------------

def test_gated_rmsnorm_hand_worked():
    """dv = 2, o = (3, 4): mean(o^2) = 12.5, so with eps = 0 the normalised row
    is (3, 4) / sqrt(12.5) = (1.2, 1.6) / sqrt(2); w = (1, 2) and z = 40
    (silu(40) = 40 to 1e-15) give (48/sqrt(2), 128/sqrt(2))."""
    d = oracle.Dims(1, 1, 2, 2)
    y = oracle.gated_rmsnorm(d, np.array([[[3.0, 4.0]]]), np.full((1, 1, 2), 40.0),
                             np.array([1.0, 2.0]), eps=0.0)
    assert np.allclose(y[0, 0], [48.0 / math.sqrt(2.0), 128.0 / math.sqrt(2.0)], rtol=1e-14, atol=0)


def test_gated_rmsnorm_constant_row_and_gate():
    """A constant row c normalises to sign(c) (mean, not sum, of squares), and
    the gate is silu(z) = z sigmoid(z), not sigmoid(z)."""
    d = oracle.Dims(2, 4, 16, 16)
    o = np.full((1, 4, 16), -0.37)
    w = np.ones(16)
    y = oracle.gated_rmsnorm(d, o, np.full((1, 4, 16), 40.0), w, eps=0.0)
    assert np.allclose(y, -40.0, rtol=1e-14, atol=0)
    z2 = np.full((1, 4, 16), 2.0)
    y2 = oracle.gated_rmsnorm(d, o, z2, w, eps=0.0)
    assert np.allclose(y2, -2.0 / (1.0 + math.exp(-2.0)), rtol=1e-14, atol=0)
    # eps enters as mean(o^2) + eps
    y3 = oracle.gated_rmsnorm(d, o, np.full((1, 4, 16), 40.0), w, eps=0.37 ** 2 * 3)
    assert np.allclose(y3, -40.0 / 2.0, rtol=1e-14, atol=0)


def test_gated_rmsnorm_per_row_invariants():
    """eps = 0: each (token, head) row of y / (w silu(z)) has RMS 1 whatever the
    rows' scales; y is odd and scale-free in o; w indexes dv; z = 0 gives 0; a
    zero row with eps > 0 gives zeros."""
    rng = np.random.default_rng(3)
    d = oracle.Dims(2, 4, 16, 8)
    o = rng.standard_normal((5, 4, 8)) * rng.uniform(0.01, 100.0, (5, 4, 1))
    z = rng.standard_normal((5, 4, 8)) + 3.0
    w = rng.uniform(0.5, 2.0, 8)
    y = oracle.gated_rmsnorm(d, o, z, w, eps=0.0)
    silu = z / (1.0 + np.exp(-z))
    g = y / (w * silu)
    assert np.allclose(np.sqrt(np.mean(g ** 2, axis=2)), 1.0, rtol=1e-13)
    assert np.allclose(g * np.sqrt(np.mean(o ** 2, axis=2, keepdims=True)), o, rtol=1e-12)
    assert np.allclose(oracle.gated_rmsnorm(d, -7.5 * o, z, w, eps=0.0), -y, rtol=1e-13)
    onehot = np.zeros(8)
    onehot[5] = 1.0
    y1 = oracle.gated_rmsnorm(d, o, z, onehot, eps=0.0)
    assert np.all(y1[:, :, [0, 1, 2, 3, 4, 6, 7]] == 0.0) and np.all(y1[:, :, 5] != 0.0)
    assert np.all(oracle.gated_rmsnorm(d, o, np.zeros_like(z), w) == 0.0)
    o0 = o.copy()
    o0[2, 1] = 0.0
    y0 = oracle.gated_rmsnorm(d, o0, z, w, eps=1e-6)
    assert np.all(y0[2, 1] == 0.0) and np.all(np.isfinite(y0))


# ---- KDA: per-key-channel decay --------------------------------------------

def _kda_inputs(seed, shape=synth.TINY):
    g, pool, params = _tiny_setup(seed, shape)
    qkv, a, b = synth.tokens(shape, g, (3,))
    return g, pool, params, qkv.double().numpy(), a.double().numpy(), b.double().numpy()


def test_kda_with_uniform_gates_is_gdn():
    """Every key channel of a head given the head's own gate logit and bias:
    the per-channel decay is the scalar one, and KDA is the GDN step."""
    shape = synth.TINY
    d = _dims(shape)
    _, pool, params, qkv, a, b = _kda_inputs(70)
    ids = np.array([6, 1, 3], np.int32)
    pool2 = pool.copy()
    a_kda = np.repeat(a[:, :, None], d.dk, axis=2)
    p_kda = oracle.Params(params.conv_w, params.A_log,
                          np.repeat(params.dt_bias[:, None], d.dk, axis=1) + 0.0)
    o1, e1 = oracle.decode_step(d, pool, params, ids, qkv, a, b)
    o2, e2 = oracle.kda_decode_step(d, pool2, p_kda, ids, qkv, a_kda, b)
    assert e1 == e2 == 0
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(pool2.ssm, pool.ssm, rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(pool2.conv, pool.conv)


def test_kda_per_channel_forgetting():
    """A_log = 0, beta = 0 (b = -inf): a channel whose logit is +1e30 decays
    to 0 (alpha = exp(-softplus(1e30)) = 0), one at -1e30 keeps its value
    (alpha = 1); the readout is the kept columns times q_hat."""
    shape = synth.TINY
    d = _dims(shape)
    _, pool, params, qkv, _, _ = _kda_inputs(71)
    ids = np.array([2], np.int32)
    p0 = oracle.Params(params.conv_w, np.zeros(d.hv), np.zeros((d.hv, d.dk)))
    keep = (np.arange(d.dk) % 3) != 0
    a = np.where(keep, -1e30, 1e30)[None, None, :].repeat(d.hv, axis=1)
    b = np.full((1, d.hv), -np.inf)
    S0 = pool.ssm[2].copy()
    y = oracle.conv_silu(d, pool.conv[2], qkv[0], params.conv_w)
    o, err = oracle.kda_decode_step(d, pool, p0, ids, qkv[:1], a, b)
    assert err == 0
    np.testing.assert_array_equal(pool.ssm[2][:, :, ~keep], 0.0)
    np.testing.assert_array_equal(pool.ssm[2][:, :, keep], S0[:, :, keep])
    G = d.hv // d.hk
    for h in range(d.hv):
        qraw = y[(h // G) * d.dk:(h // G + 1) * d.dk]
        qh = qraw / math.sqrt(qraw @ qraw + EPS) / math.sqrt(d.dk)
        np.testing.assert_allclose(o[0, h], S0[h][:, keep] @ qh[keep], rtol=1e-12, atol=1e-14)


def test_kda_retrieval_for_any_channel_decay():
    """beta = 1: S_new^T k_hat = v (1 - delta) + delta S^T (alpha . k_hat),
    delta = eps / (|k|^2 + eps), whatever the per-channel alpha."""
    shape = synth.TINY
    d = _dims(shape)
    g, pool, params, qkv, _, _ = _kda_inputs(72)
    ids = np.array([4], np.int32)
    dt = synth.normal((d.hv, d.dk), 1.0, g).double().numpy()
    pk = oracle.Params(params.conv_w, params.A_log, dt)
    a = synth.normal((1, d.hv, d.dk), 1.5, g).double().numpy()
    b = np.full((1, d.hv), np.inf)
    S0 = pool.ssm[4].copy()
    y = oracle.conv_silu(d, pool.conv[4], qkv[0], params.conv_w)
    oracle.kda_decode_step(d, pool, pk, ids, qkv[:1], a, b)
    G = d.hv // d.hk
    for h in range(d.hv):
        hq = h // G
        kraw = y[d.hk * d.dk + hq * d.dk: d.hk * d.dk + (hq + 1) * d.dk]
        kh = kraw / math.sqrt(kraw @ kraw + EPS)
        delta = EPS / (kraw @ kraw + EPS)
        vv = y[2 * d.hk * d.dk + h * d.dv: 2 * d.hk * d.dk + (h + 1) * d.dv]
        alpha = np.exp([oracle.gate_g(pk.A_log[h], dt[h, c], a[0, h, c]) for c in range(d.dk)])
        assert np.ptp(alpha) > 0.1  # the decays really differ by channel
        np.testing.assert_allclose(pool.ssm[4, h] @ kh, vv * (1 - delta) + delta * (S0[h] @ (alpha * kh)),
                                   rtol=1e-11, atol=1e-12)


def test_kda_verify_then_commit_equals_L_kda_decode_steps():
    """KDA verify leaves the working slot alone; committing draft L gives the
    state of L KDA decode steps, and the first L outputs are theirs."""
    shape = synth.TINY
    d = _dims(shape)
    g, pool, params = _tiny_setup(73)
    pk = oracle.Params(params.conv_w, params.A_log, synth.normal((d.hv, d.dk), 0.5, g).double().numpy())
    B, T = 2, 4
    ids = np.array([1, 6], np.int32)
    spec = oracle.Pool(np.full((B * T, d.hv, d.dv, d.dk), 7.25), np.full((B * T, d.w - 1, d.channels), -3.5))
    spec_ids = np.arange(B * T, dtype=np.int32).reshape(B, T)
    qkv, _, b = (t.double().numpy() for t in synth.tokens(shape, g, (B, T)))
    a = synth.normal((B, T, d.hv, d.dk), 1.2, g).double().numpy()
    before = pool.copy()
    out, err = oracle.kda_spec_verify(d, pool, spec, pk, ids, spec_ids, qkv, a, b)
    assert err == 0
    assert np.array_equal(pool.ssm, before.ssm) and np.array_equal(pool.conv, before.conv)
    for L in range(0, T + 1):
        ref = before.copy()
        for t in range(L):
            o, _ = oracle.kda_decode_step(d, ref, pk, ids, qkv[:, t], a[:, t], b[:, t])
            np.testing.assert_array_equal(out[:, t], o)
        work = before.copy()
        assert oracle.spec_commit(d, spec, work, spec_ids, np.full(B, L, np.int32), ids) == 0
        np.testing.assert_array_equal(work.ssm, ref.ssm)
        np.testing.assert_array_equal(work.conv, ref.conv)


def test_kda_verify_with_uniform_gates_is_gdn_verify():
    shape = synth.TINY
    d = _dims(shape)
    g, pool, params = _tiny_setup(74)
    B, T = 3, 3
    ids = np.array([0, 4, 7], np.int32)
    mk = lambda: oracle.Pool(np.zeros((B * T, d.hv, d.dv, d.dk)), np.zeros((B * T, d.w - 1, d.channels)))  # noqa: E731
    s1, s2 = mk(), mk()
    spec_ids = np.arange(B * T, dtype=np.int32).reshape(B, T)
    qkv, a, b = (t.double().numpy() for t in synth.tokens(shape, g, (B, T)))
    pk = oracle.Params(params.conv_w, params.A_log, np.repeat(params.dt_bias[:, None], d.dk, axis=1) + 0.0)
    o1, _ = oracle.spec_verify(d, pool, s1, params, ids, spec_ids, qkv, a, b)
    o2, _ = oracle.kda_spec_verify(d, pool, s2, pk, ids, spec_ids, qkv, np.repeat(a[..., None], d.dk, axis=3), b)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(s2.ssm, s1.ssm, rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(s2.conv, s1.conv)


def test_kda_prefill_equals_kda_decode_steps_and_checkpoints():
    """KDA prefill of two sequences (one resumed mid-block) = their tokens as
    KDA decode steps; each checkpoint holds the state after its block boundary."""
    shape = synth.TINY
    d = _dims(shape)
    g, pool, params = _tiny_setup(75)
    pk = oracle.Params(params.conv_w, params.A_log, synth.normal((d.hv, d.dk), 0.5, g).double().numpy())
    lens, starts, blk = [70, 33], [0, 50], 32
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    ids = np.array([3, 6], np.int32)
    qkv, _, b = (t.double().numpy() for t in synth.tokens(shape, g, (int(cu[-1]),)))
    a = synth.normal((int(cu[-1]), d.hv, d.dk), 1.0, g).double().numpy()
    ck = oracle.Pool(np.full((6, d.hv, d.dv, d.dk), -9.0), np.full((6, d.w - 1, d.channels), 4.0))
    ck_ids = np.array([[0, 1, 2], [3, 4, 5]], np.int32)
    ref = pool.copy()
    out, err = oracle.kda_prefill(d, pool, ck, pk, ids, cu, starts, ck_ids, blk, qkv, a, b)
    assert err == 0
    expect_ck = {}
    for n in range(2):
        for i in range(cu[n], cu[n + 1]):
            o, _ = oracle.kda_decode_step(d, ref, pk, ids[n:n + 1], qkv[i:i + 1], a[i:i + 1], b[i:i + 1])
            np.testing.assert_array_equal(out[i], o[0])
            P = starts[n] + (i - cu[n]) + 1
            if P % blk == 0:
                expect_ck[int(ck_ids[n][P // blk - starts[n] // blk - 1])] = (ref.ssm[ids[n]].copy(),
                                                                            ref.conv[ids[n]].copy())
    np.testing.assert_array_equal(pool.ssm, ref.ssm)
    np.testing.assert_array_equal(pool.conv, ref.conv)
    # sequence 0: boundaries 32, 64; sequence 1 (50 .. 83): 64
    assert sorted(expect_ck) == [0, 1, 3]
    for cid, (s_, c_) in expect_ck.items():
        np.testing.assert_array_equal(ck.ssm[cid], s_)
        np.testing.assert_array_equal(ck.conv[cid], c_)
    assert np.all(ck.ssm[[2, 4, 5]] == -9.0)


@pytest.mark.parametrize("chunk", [1, 4, 16, 32, 64])
@pytest.mark.parametrize("strong_decay", [False, True])
def test_kda_window_form_equals_token_recurrence(chunk, strong_decay):
    """The KDA prefill in windows of `chunk` tokens (A', M, T from per-channel
    cumulative log decays; the algebra of the GPU's chunked form) equals the
    token-by-token KDA prefill: outputs, final states, conv histories and
    checkpoints, from aligned and unaligned starts, in double precision.  With
    strong decays (A_log = ln 16) many decay factors underflow to zero."""
    shape = synth.TINY
    d = _dims(shape)
    g, pool, params = _tiny_setup(90 + chunk)
    A_log = np.full(d.hv, math.log(16.0)) if strong_decay else params.A_log
    pk = oracle.Params(params.conv_w, A_log, synth.normal((d.hv, d.dk), 0.5, g).double().numpy())
    # checkpoint blocks of 32 tokens (64 for the 64-token chunks: a block
    # boundary is always a chunk boundary)
    lens, starts, blk = [70, 45, 9], [0, 50, 3], max(32, chunk)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    ids = np.array([3, 6, 1], np.int32)
    qkv, _, b = (t.double().numpy() for t in synth.tokens(shape, g, (int(cu[-1]),)))
    a = synth.normal((int(cu[-1]), d.hv, d.dk), 1.0, g).double().numpy()
    ck_ids = np.array([[0, 1, 2], [3, 4, 5], [6, 7, 8]], np.int32)
    ck1 = oracle.Pool(np.full((9, d.hv, d.dv, d.dk), -9.0), np.full((9, d.w - 1, d.channels), 4.0))
    ck2 = oracle.Pool(ck1.ssm.copy(), ck1.conv.copy())
    pool2 = pool.copy()
    o1, e1 = oracle.kda_prefill(d, pool, ck1, pk, ids, cu, starts, ck_ids, blk, qkv, a, b)
    o2, e2 = oracle.kda_prefill_chunked(d, pool2, ck2, pk, ids, cu, starts, ck_ids, blk, chunk, qkv, a, b)
    assert e1 == e2 == 0
    np.testing.assert_allclose(o2, o1, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(pool2.ssm, pool.ssm, rtol=1e-10, atol=1e-12)
    np.testing.assert_array_equal(pool2.conv, pool.conv)
    np.testing.assert_allclose(ck2.ssm, ck1.ssm, rtol=1e-10, atol=1e-12)
    np.testing.assert_array_equal(ck2.conv, ck1.conv)
    written = [0, 1, 3] if blk == 32 else [0, 3]  # the boundaries 32, 64 (seq 0) and 64 (seq 1)
    assert not np.any([np.all(ck1.ssm[i] == -9.0) for i in written])
