"""The algebra of the KDA 64-token chunk on the tensor cores, in float64 on
the CPU: A'[t][j] = sum_c k_tc k_jc e^{lb_tc - lb_jc} and M (the same with q_t)
taken as the kernel takes them -- 8-token blocks, running products of alpha
within a block (fl8 from its first token, fr8 to its last), block factors as
exponentials of sums of block totals, the 28 off-diagonal block pairs in three
levels of one product each (reference blocks 4; 2 and 6; the row block), the
diagonal blocks by running products down each row -- equal the definition,
and K~, K- from the block factors equal k e^{lb}, k e^{lb_63 - lb}.  Gates
drawn strong enough that many factors underflow (-exp(A_log) softplus with
exp(A_log) up to 16), plus floored tokens (log decay -128)."""
import numpy as np
import pytest

C, D = 64, 128


def _case(seed, eA=None):
    rng = np.random.default_rng(seed)
    eA = np.exp(rng.uniform(0, np.log(16))) if eA is None else eA
    g = -eA * np.log1p(np.exp(rng.normal(0, 1.1, (C, D))))
    g[rng.integers(0, C, 3), rng.integers(0, D, 3)] = -np.inf
    g = np.maximum(g, -128.0)
    k = rng.normal(size=(C, D))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    q = rng.normal(size=(C, D))
    q /= np.linalg.norm(q, axis=1, keepdims=True) * np.sqrt(D)
    return g, k, q


def _direct(g, k, q):
    lb = np.cumsum(g, axis=0)
    A = np.zeros((C, C))
    M = np.zeros((C, C))
    for t in range(C):
        for j in range(t + 1):
            f = np.exp(lb[t] - lb[j])
            M[t, j] = (q[t] * k[j] * f).sum()
            if j < t:
                A[t, j] = (k[t] * k[j] * f).sum()
    return lb, A, M


def _blocked(g, k, q, drop_level2_row_factor=False):
    al = np.exp(g)
    fl = np.ones((C, D))
    fr = np.ones((C, D))
    for B in range(8):
        b, e = 8 * B, 8 * B + 7
        for t in range(b + 1, e + 1):
            fl[t] = fl[t - 1] * al[t]
        for t in range(e - 1, b - 1, -1):
            fr[t] = fr[t + 1] * al[t + 1]
    G = np.array([g[8 * B:8 * B + 8].sum(0) for B in range(8)])   # block totals
    f = np.array([g[8 * B] for B in range(8)])                    # first-token log decays
    Lk, Lq, Rk = k * fl, q * fl, k * fr
    A = np.zeros((C, C))
    M = np.zeros((C, C))
    blk = lambda X, I: X[8 * I:8 * I + 8]
    levels = ([(I, J, 4) for I in range(4, 8) for J in range(4)] +
              [(I, J, 2) for I in (2, 3) for J in (0, 1)] + [(I, J, 6) for I in (6, 7) for J in (4, 5)] +
              [(I, I - 1, I) for I in (1, 3, 5, 7)])
    assert sorted((I, J) for I, J, _ in levels) == [(I, J) for I in range(8) for J in range(I)]
    for I, J, R in levels:
        assert J < R <= I
        # row factor e^{lb_b(I) - lb_b(R)}, column factor e^{lb_b(R) - lb_e(J)}
        if R == 4:
            FA, FB = np.exp(G[4:I].sum(0) - f[4] + f[I]), np.exp(G[J + 1:4].sum(0) + f[4])
        elif R in (2, 6):
            FA = np.exp(G[I - 1] - f[I - 1] + f[I]) if I % 2 and not drop_level2_row_factor else np.ones(D)
            FB = np.exp(G[J + 1:R].sum(0) + f[R])
        else:
            FA, FB = np.ones(D), np.exp(f[I])
        A[8 * I:8 * I + 8, 8 * J:8 * J + 8] = (blk(Lk, I) * FA) @ (blk(Rk, J) * FB).T
        M[8 * I:8 * I + 8, 8 * J:8 * J + 8] = (blk(Lq, I) * FA) @ (blk(Rk, J) * FB).T
    for I in range(8):  # diagonal blocks: running products down each row
        for t in range(8):
            p = np.ones(D)
            for j in range(t, -1, -1):
                if j < t:
                    p = p * al[8 * I + j + 1]
                M[8 * I + t, 8 * I + j] = (q[8 * I + t] * k[8 * I + j] * p).sum()
                if j < t:
                    A[8 * I + t, 8 * I + j] = (k[8 * I + t] * k[8 * I + j] * p).sum()
    Eb = np.array([np.exp(G[:I].sum(0) + f[I]) for I in range(8)])
    Ee = np.array([np.exp(G[I + 1:].sum(0)) for I in range(8)])
    Kt = np.array([k[t] * fl[t] * Eb[t // 8] for t in range(C)])
    Km = np.array([k[t] * fr[t] * Ee[t // 8] for t in range(C)])
    return A, M, Kt, Km, np.exp(G.sum(0))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_blocked_factors_equal_the_definition(seed):
    g, k, q = _case(seed)
    lb, A, M = _direct(g, k, q)
    A2, M2, Kt, Km, alast = _blocked(g, k, q)
    np.testing.assert_allclose(A2, A, rtol=0, atol=1e-13)
    np.testing.assert_allclose(M2, M, rtol=0, atol=1e-13)
    np.testing.assert_allclose(Kt, k * np.exp(lb), rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(Km, k * np.exp(lb[-1] - lb), rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(alast, np.exp(lb[-1]), rtol=1e-12, atol=1e-300)
    # every factor the blocked form multiplies by is at most 1 (no overflow)
    assert np.all(np.exp(g) <= 1.0)


def test_a_dropped_factor_fails():
    """A plausible mistake (the level-2 row factor of odd row blocks left out)
    is caught, with decays weak enough that the factor matters."""
    g, k, q = _case(3, eA=0.2)
    _, A, M = _direct(g, k, q)
    A2, M2, *_ = _blocked(g, k, q, drop_level2_row_factor=True)
    assert np.abs(A2 - A).max() > 1e-3 and np.abs(M2 - M).max() > 1e-4
    A3, M3, *_ = _blocked(g, k, q)
    np.testing.assert_allclose(A3, A, rtol=0, atol=1e-13)
