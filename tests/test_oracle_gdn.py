"""Pins of the fp64 oracle's Log-Linear Gated DeltaNet.

"Log-Linear Attention" §3 names Log-Linear Gated DeltaNet and says it keeps
the base model's structure under the hierarchical (Fenwick) mask, without a
formula.  The reading implemented by the oracle: every Fenwick bucket keeps its
own Gated DeltaNet state, all states take every token's transition
A_r = alpha_r (I - beta_r k_r k_r^T), and the read-out weights the buckets by
lambda.  The pins tie that reading to facts that do not depend on the oracle:

  - the pair form and the recurrent form agree (two derivations);
  - lambda = 1 gives Gated DeltaNet itself (one state, the base recurrence);
  - mutually orthogonal keys turn every transition into the scalar decay, so
    the result is Log-Linear Mamba-2 (the pinned `naive`) with values beta v;
  - one-dimensional keys (k = +-1) make A_r the scalar alpha_r (1 - beta_r),
    checked against a closed form written out for T = 3;
  - the output is linear in lambda and vanishes with beta;
  - replaying the decode step from the empty state reproduces the pair form.
"""

import math

import numpy as np
import pytest

import oracle


def gdn_inputs(B, H, T, dk, dv, seed, L=None):
    rng = np.random.default_rng(seed)
    L = oracle.num_levels(T) if L is None else L
    q = rng.standard_normal((B, H, T, dk)) / math.sqrt(dk)
    k = rng.standard_normal((B, H, T, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, H, T, dv))
    g = -np.log1p(np.exp(rng.standard_normal((B, H, T)) - 2.0))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, H, T))))
    lam = np.log1p(np.exp(0.54 + 0.3 * rng.standard_normal((B, H, T, L))))
    return q, k, v, g, beta, lam


def rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


@pytest.mark.parametrize("B,H,T,dk,dv", [(1, 1, 1, 3, 2), (1, 2, 13, 4, 3), (2, 1, 64, 8, 5),
                                         (1, 1, 100, 16, 16)])
def test_pair_form_equals_recurrent_form(B, H, T, dk, dv):
    x = gdn_inputs(B, H, T, dk, dv, seed=T + dk)
    assert rel(oracle.gdn_fenwick(*x), oracle.gdn_naive(*x)) < 1e-12


def test_lambda_one_is_gated_deltanet():
    q, k, v, g, beta, lam = gdn_inputs(1, 2, 40, 6, 5, seed=1)
    ones = np.ones_like(lam)
    base = oracle.gdn_base(q, k, v, g, beta)
    assert rel(oracle.gdn_naive(q, k, v, g, beta, ones), base) < 1e-12
    assert rel(oracle.gdn_fenwick(q, k, v, g, beta, ones), base) < 1e-12


def test_orthogonal_keys_reduce_to_log_linear_mamba2():
    B, H, T, dk, dv = 1, 2, 12, 16, 5
    q, k, v, g, beta, lam = gdn_inputs(B, H, T, dk, dv, seed=2)
    rng = np.random.default_rng(3)
    for b in range(B):
        for h in range(H):
            Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
            k[b, h] = Qm[:T]  # T orthonormal rows
    got = oracle.gdn_naive(q, k, v, g, beta, lam)
    want = oracle.naive(q, k, beta[..., None] * v, g, lam)
    assert rel(got, want) < 1e-12


def test_one_dimensional_closed_form_T3():
    # dk = dv = 1, k = +-1: A_r = alpha_r (1 - beta_r), levels (t,s): (1,0)->1,
    # (2,0)->2, (2,1)->2
    q = np.array([0.7, -1.3, 0.4]).reshape(1, 1, 3, 1)
    k = np.array([1.0, -1.0, 1.0]).reshape(1, 1, 3, 1)
    v = np.array([2.0, 0.5, -1.5]).reshape(1, 1, 3, 1)
    g = np.array([-0.1, -0.3, -0.2]).reshape(1, 1, 3)
    beta = np.array([0.6, 0.25, 0.9]).reshape(1, 1, 3)
    lam = np.array([[1.1, 0.8, 0.5], [0.9, 1.3, 0.7], [1.2, 0.6, 1.4]]).reshape(1, 1, 3, 3)
    a = np.exp(g[0, 0]) * (1.0 - beta[0, 0])
    bkv = beta[0, 0] * k[0, 0, :, 0] * v[0, 0, :, 0]
    qq = q[0, 0, :, 0]
    L = lam[0, 0]
    want = np.array([
        L[0, 0] * bkv[0] * qq[0],
        L[1, 0] * bkv[1] * qq[1] + L[1, 1] * bkv[0] * a[1] * qq[1],
        L[2, 0] * bkv[2] * qq[2] + L[2, 2] * (bkv[1] * a[2] + bkv[0] * a[1] * a[2]) * qq[2],
    ])
    for fn in (oracle.gdn_naive, oracle.gdn_fenwick):
        got = fn(q, k, v, g, beta, lam)[0, 0, :, 0]
        assert np.allclose(got, want, rtol=1e-14, atol=1e-15), (fn.__name__, got, want)


def test_linear_in_lambda_and_zero_beta():
    q, k, v, g, beta, lam = gdn_inputs(1, 1, 20, 4, 3, seed=4)
    full = oracle.gdn_naive(q, k, v, g, beta, lam)
    parts = 0.0
    for l in range(lam.shape[-1]):
        e = np.zeros_like(lam)
        e[..., l] = lam[..., l]
        parts = parts + oracle.gdn_naive(q, k, v, g, beta, e)
    assert rel(parts, full) < 1e-12
    assert np.max(np.abs(oracle.gdn_fenwick(q, k, v, g, np.zeros_like(beta), lam))) == 0.0


def test_decode_replay_reproduces_pair_form():
    B, H, T, dk, dv = 2, 2, 37, 5, 4
    q, k, v, g, beta, lam = gdn_inputs(B, H, T, dk, dv, seed=5)
    want = oracle.gdn_naive(q, k, v, g, beta, lam)
    Ls = T.bit_length()
    S = np.zeros((B, H, Ls, dk, dv))
    lam_w = np.zeros((B, H, T, Ls + 1))
    lam_w[..., :lam.shape[-1]] = lam
    for t in range(T):
        o = oracle.gdn_decode_step(S, q[:, :, t], k[:, :, t], v[:, :, t], g[:, :, t], beta[:, :, t],
                                   lam_w[:, :, t], np.full(B, t))
        assert rel(o, want[:, :, t]) < 1e-12, t
