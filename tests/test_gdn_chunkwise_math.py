"""The algebra behind the chunkwise Log-Linear Gated DeltaNet forward, checked
in fp64 numpy against the oracle (no GPU, no code shared with the kernels).

The kernels (csrc/gdn_chunk.cu) rest on three facts about the reading of
"Log-Linear Attention" §3 that the oracle implements (every Fenwick bucket
keeps its own Gated DeltaNet state; all states take each token's transition
A_r = exp(g_r) (I - beta_r k_r k_r^T); the read-out weights buckets by lambda):

  1. the product of a chunk's undecayed factors has the compact form
         (I - b_{n-1} k k^T) ... (I - b_0 k k^T) = I - K^T T K,
         T = (I + strict_lower(diag(b) K K^T))^{-1} diag(b);
  2. column s of K^T T is (product of the factors after s) b_s k_s, which
     gives the chunk's own state K^T T diag(exp(gam_end - gam)) V and, over a
     sub-range of columns, the states of the low-bit buckets of a ragged end;
  3. the decay is a scalar and factors out of every product, so a chunk
     reads out a state S through q~ = diag(exp(gam)) (Q - lower(Q K^T) T K),
     transitions it as exp(gam_end) (S - K^T (T K) S), and its intra-chunk
     output is (lambda by level x decay x lower(Q K^T) T) V.

Here the whole chunkwise evaluation is written out with those formulas and
compared with the oracle's pair form and with its decode states.
"""

import numpy as np
import pytest

import oracle
from test_oracle_gdn import gdn_inputs, rel

C = 64


def compact_T(K, b):
    n = K.shape[0]
    A = np.tril(b[:, None] * (K @ K.T), -1)
    return np.linalg.solve(np.eye(n) + A, np.diag(b))


def level(t, s):
    return int(t ^ s).bit_length()


def chunkwise(q, k, v, g, beta, lam, Ls=None):
    """One (batch, head): outputs [T, dv] and, with Ls, the final state in the
    decode layout [Ls, dk, dv] (slot j = level j + 1, dead slots zero)."""
    T, dk = q.shape
    dv = v.shape[1]
    N = -(-T // C)
    out = np.zeros((T, dv))
    S = {}  # chunk-level slot m (level 7 + m) -> state at the current chunk start
    low = {}
    for i in range(N):
        sl = slice(i * C, min(T, (i + 1) * C))
        n = sl.stop - sl.start
        Q, K, V, b, Lm = q[sl], k[sl], v[sl], beta[sl], lam[sl]
        gam = np.cumsum(g[sl])
        Tm = compact_T(K, b)
        QK = np.tril(Q @ K.T)
        Cm = QK @ Tm
        a_idx = np.arange(n)
        lev = np.array([[level(a, s) for s in range(n)] for a in range(n)])
        Wgt = np.where(a_idx[:, None] >= a_idx[None, :],
                       np.take_along_axis(Lm, np.minimum(lev, Lm.shape[1] - 1), axis=1)
                       * np.exp(gam[:, None] - gam[None, :]), 0.0)
        o = (Wgt * Cm) @ V
        Qt = np.exp(gam)[:, None] * (Q - Cm @ K)
        for m, St in S.items():
            o += Lm[:, 7 + m][:, None] * (Qt @ St)
        out[sl] = o
        W = Tm @ K
        for m in S:
            S[m] = np.exp(gam[-1]) * (S[m] - K.T @ (W @ S[m]))
        Tp = Tm * np.exp(gam[-1] - gam)[None, :]
        if n == C:
            m0 = ((i + 1) & -(i + 1)).bit_length() - 1
            new = K.T @ (Tp @ V)
            for m in range(m0):
                new = new + S.pop(m)
            S[m0] = new
        else:
            for j in range(6):
                if (n >> j) & 1:
                    hi = n - (n & ((1 << j) - 1))
                    lo = hi - (1 << j)
                    low[j] = K.T @ (Tp[:, lo:hi] @ V[lo:hi])
    if Ls is None:
        return out
    state = np.zeros((Ls, dk, dv))
    nfull = T // C
    for m, St in S.items():
        if (nfull >> m) & 1:
            state[6 + m] = St
    for j, St in low.items():
        state[j] = St
    return out, state


def test_compact_product_identity():
    rng = np.random.default_rng(3)
    for n, d in ((1, 4), (5, 8), (64, 32), (64, 64)):
        K = rng.standard_normal((n, d))
        K /= np.linalg.norm(K, axis=1, keepdims=True)
        b = rng.uniform(0.0, 1.0, n)
        P = np.eye(d)
        for r in range(n):
            P = (np.eye(d) - b[r] * np.outer(K[r], K[r])) @ P
        assert rel(np.eye(d) - K.T @ compact_T(K, b) @ K, P) < 1e-12


def test_columns_of_KT_T_are_the_later_products():
    rng = np.random.default_rng(4)
    n, d = 37, 16
    K = rng.standard_normal((n, d))
    K /= np.linalg.norm(K, axis=1, keepdims=True)
    b = rng.uniform(0.0, 1.0, n)
    KT_T = K.T @ compact_T(K, b)
    for s in range(n):
        x = b[s] * K[s]
        for r in range(s + 1, n):
            x = x - b[r] * K[r] * (K[r] @ x)
        assert np.abs(KT_T[:, s] - x).max() < 1e-12


@pytest.mark.parametrize("T,dk,dv,seed", [(64, 8, 4, 1), (100, 16, 8, 2), (333, 16, 16, 3), (512, 8, 8, 4),
                                          (1000, 8, 4, 5)])
def test_chunkwise_evaluation_matches_the_pair_form(T, dk, dv, seed):
    q, k, v, g, beta, lam = gdn_inputs(1, 1, T, dk, dv, seed)
    ref = oracle.gdn_naive(q, k, v, g, beta, lam)[0, 0]
    got = chunkwise(q[0, 0], k[0, 0], v[0, 0], g[0, 0], beta[0, 0], lam[0, 0])
    assert rel(got, ref) < 1e-11


@pytest.mark.parametrize("T", [45, 128, 200, 448, 513])
def test_chunkwise_final_state_matches_the_decode_states(T):
    dk, dv = 8, 4
    q, k, v, g, beta, lam = gdn_inputs(1, 1, T, dk, dv, 20 + T)
    Ls = T.bit_length() + 1
    _, state = chunkwise(q[0, 0], k[0, 0], v[0, 0], g[0, 0], beta[0, 0], lam[0, 0], Ls)
    S = np.zeros((1, 1, Ls, dk, dv))
    for t in range(T):
        lt = np.zeros((1, 1, Ls + 1))
        lt[..., :lam.shape[-1]] = lam[:, :, t]
        oracle.gdn_decode_step(S, q[:, :, t], k[:, :, t], v[:, :, t], g[:, :, t], beta[:, :, t], lt, [t])
    live = [j for j in range(Ls) if (T >> j) & 1]
    assert rel(state[live], S[0, 0, live]) < 1e-11
    assert not state[[j for j in range(Ls) if j not in live]].any()
