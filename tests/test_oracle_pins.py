"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics,
not against the oracle itself.

Page "Log-Linear Attention" (gist.science 2506.04761), technical summary:
  §2.2  the output is sum_l lambda_t^(l) q_t^T S_t^(l), the prefix [0,t) split
        into <= L disjoint Fenwick buckets;
  §2.3  decoding is recurrent with O(log T) states;
  §3    the Mamba-2 instance with a scalar gate.
Page "Adaptive memory decay for Log-Linear Attention", §LambdaMLPSoftplus:
  softplus(0.54) is about 1.0 (the lambda initialisation the workloads centre on).

The backward (no formula on the pages) is pinned to the forward double sum by
central finite differences, and by identities of that sum: it is linear in each
of q, k, v and lambda (so, by Euler's theorem, <x, dx> equals the loss for each),
dq is the forward with (q, k, v) -> (dout, v, k), and the loss depends on G only
through differences, so dg_0 = sum_u dG_u = 0.

Each test below would fail on a plausible slip in the oracle: a wrong level
index (bucket tests, hand table), an exclusive instead of inclusive gate sum or
a sign error in the decay (hand-expanded T=3 case, SSD reduction), a dropped
diagonal or level term (lambda = e_l tests), a transposed state (decode replay
and closed-form state against the double sum).
"""

import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_inputs(B, H, T, dk, dv, seed, g_scale=1.0, L=None):
    rng = np.random.default_rng(seed)
    L = oracle.num_levels(T) if L is None else L
    q = rng.standard_normal((B, H, T, dk)) / math.sqrt(dk)
    k = rng.standard_normal((B, H, T, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, H, T, dv))
    g = -np.log1p(np.exp(rng.standard_normal((B, H, T)))) * g_scale
    lam = np.log1p(np.exp(0.54 + 0.3 * rng.standard_normal((B, H, T, L))))
    return q, k, v, g, lam


def fenwick_buckets(t):
    """Buckets of [0,t) by peeling the lowest set bit of the Fenwick index:
    j = t, t - lowbit(t), ...; bucket [j - lowbit(j), j) has lowbit(j) keys.
    Returns a list of (first, end, size)."""
    out = []
    j = t
    while j > 0:
        low = j & -j
        out.append((j - low, j, low))
        j -= low
    return out


def relerr(a, b):
    return np.max(np.abs(a - b)) / max(1.0, np.max(np.abs(b)))


# ---------------------------------------------------------------- levels

def test_level_table_T8_golden():
    rows = {}
    with open(os.path.join(GOLDEN, "fenwick_levels_T8.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            t, rest = line.split(":")
            rows[int(t)] = [int(x) for x in rest.split()]
    assert sorted(rows) == list(range(8))
    for t, levels in rows.items():
        assert [oracle.level(t, s) for s in range(t + 1)] == levels


@pytest.mark.parametrize("T", list(range(1, 17)))
def test_levels_are_fenwick_buckets(T):
    for t in range(T):
        buckets = fenwick_buckets(t)
        # the buckets partition [0, t), finer near t, at most L-1 of them
        covered = sorted(s for a, b, _ in buckets for s in range(a, b))
        assert covered == list(range(t))
        assert len(buckets) == bin(t).count("1")
        assert len(buckets) <= oracle.num_levels(T) - 1
        sizes = [n for _, _, n in buckets]
        assert sizes == sorted(sizes)
        for a, b, n in buckets:
            lev = n.bit_length()  # 2^(l-1) keys <-> level l
            for s in range(a, b):
                assert oracle.level(t, s) == lev
        assert oracle.level(t, t) == 0


def test_num_levels_of_the_workloads():
    assert [oracle.num_levels(T) for T in (256, 2048, 8192, 32768, 65536)] == \
        [9, 12, 14, 16, 17]
    assert oracle.num_levels(1) == 1


# ---------------------------------------------------------- hand expansion

def test_hand_expanded_T3():
    """o_2 written out by hand from the definition: keys 0 and 1 form the
    level-2 bucket of query 2; key 2 is the diagonal.  G is the inclusive
    running sum, so key 1 decays by exp(g_2) and key 0 by exp(g_1 + g_2)."""
    q, k, v, g, lam = rand_inputs(1, 1, 3, 4, 5, seed=11, L=3)
    q0, k0, v0, g0, l0 = q[0, 0], k[0, 0], v[0, 0], g[0, 0], lam[0, 0]
    o = oracle.naive(q, k, v, g, lam)[0, 0]
    o0 = l0[0, 0] * (q0[0] @ k0[0]) * v0[0]
    o1 = l0[1, 0] * (q0[1] @ k0[1]) * v0[1] + \
        l0[1, 1] * math.exp(g0[1]) * (q0[1] @ k0[0]) * v0[0]
    o2 = l0[2, 0] * (q0[2] @ k0[2]) * v0[2] + l0[2, 2] * (
        math.exp(g0[1] + g0[2]) * (q0[2] @ k0[0]) * v0[0] +
        math.exp(g0[2]) * (q0[2] @ k0[1]) * v0[1])
    np.testing.assert_allclose(o[0], o0, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(o[1], o1, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(o[2], o2, rtol=1e-13, atol=1e-15)
    # lambda entries at levels with no bucket are ignored
    lam2 = lam.copy()
    lam2[0, 0, 2, 1] = 1e6
    lam2[0, 0, 1, 2] = -7.0
    np.testing.assert_allclose(oracle.naive(q, k, v, g, lam2)[0, 0], o, rtol=1e-14)


# ------------------------------------------------ two independent derivations

@pytest.mark.parametrize("B,H,T,dk,dv", [(1, 1, 1, 4, 4), (2, 3, 64, 8, 8), (1, 2, 100, 5, 7),
                                         (1, 1, 257, 6, 3), (1, 1, 512, 4, 4)])
def test_naive_equals_fenwick_recurrence(B, H, T, dk, dv):
    q, k, v, g, lam = rand_inputs(B, H, T, dk, dv, seed=T)
    a = oracle.naive(q, k, v, g, lam)
    b, live = oracle.fenwick(q, k, v, g, lam, return_live_counts=True)
    assert relerr(b, a) <= 1e-10
    # the recurrent form touches popcount(t) <= bit_length(t) states (§2.3)
    for t in range(T):
        assert (live[..., t] == bin(t).count("1")).all()
        assert bin(t).count("1") <= max(t, 0).bit_length()


def test_naive_equals_fenwick_slow_decay():
    q, k, v, g, lam = rand_inputs(1, 2, 300, 8, 8, seed=3, g_scale=0.01)
    assert relerr(oracle.fenwick(q, k, v, g, lam), oracle.naive(q, k, v, g, lam)) <= 1e-10


# ------------------------------------------------------------- reductions

def test_lambda_one_is_gated_linear_attention():
    """Every lambda = 1: the Fenwick levels merge back into the single-state
    Mamba-2 scan S_t = e^{g_t} S_{t-1} + k_t v_t^T, o_t = S_t^T q_t."""
    q, k, v, g, lam = rand_inputs(2, 2, 200, 6, 5, seed=5)
    ones = np.ones_like(lam)
    ref = oracle.ssd(q, k, v, g)
    assert relerr(oracle.naive(q, k, v, g, ones), ref) <= 1e-10
    assert relerr(oracle.fenwick(q, k, v, g, ones), ref) <= 1e-10


def test_no_decay_lambda_one_is_causal_linear_attention():
    q, k, v, g, lam = rand_inputs(1, 1, 50, 7, 6, seed=6)
    zeros = np.zeros_like(g)
    ones = np.ones_like(lam)
    Q, K, V = q[0, 0], k[0, 0], v[0, 0]
    ref = np.tril(Q @ K.T) @ V
    assert relerr(oracle.naive(q, k, v, zeros, ones)[0, 0], ref) <= 1e-12
    assert relerr(oracle.fenwick(q, k, v, zeros, ones)[0, 0], ref) <= 1e-12
    assert relerr(oracle.ssd(q, k, v, zeros)[0, 0], ref) <= 1e-12


def test_level0_only_is_the_diagonal():
    q, k, v, g, lam = rand_inputs(1, 2, 40, 6, 4, seed=7)
    lam0 = np.zeros_like(lam)
    lam0[..., 0] = lam[..., 0]
    ref = lam[..., 0:1] * np.sum(q * k, axis=-1, keepdims=True) * v
    assert relerr(oracle.naive(q, k, v, g, lam0), ref) <= 1e-13
    assert relerr(oracle.fenwick(q, k, v, g, lam0), ref) <= 1e-13


@pytest.mark.parametrize("lev", [1, 2, 3, 4, 5])
def test_single_level_is_its_bucket_sum(lev):
    """lambda = e_l: the output is the decayed sum over the level-l Fenwick
    bucket of [0,t), the bucket taken from lowest-bit peeling."""
    T = 40
    q, k, v, g, lam = rand_inputs(1, 1, T, 5, 3, seed=8 + lev)
    e = np.zeros_like(lam)
    e[..., lev] = 1.0
    G = np.cumsum(g[0, 0])
    ref = np.zeros((T, 3))
    for t in range(T):
        for a, b, n in fenwick_buckets(t):
            if n.bit_length() != lev:
                continue
            for s in range(a, b):
                ref[t] += math.exp(G[t] - G[s]) * (q[0, 0, t] @ k[0, 0, s]) * v[0, 0, s]
    assert relerr(oracle.naive(q, k, v, g, e)[0, 0], ref) <= 1e-12
    assert relerr(oracle.fenwick(q, k, v, g, e)[0, 0], ref) <= 1e-12


def test_linear_in_lambda():
    q, k, v, g, lam = rand_inputs(1, 2, 64, 4, 4, seed=9)
    L = lam.shape[-1]
    total = np.zeros_like(oracle.naive(q, k, v, g, lam))
    for lev in range(L):
        part = np.zeros_like(lam)
        part[..., lev] = lam[..., lev]
        total += oracle.naive(q, k, v, g, part)
    assert relerr(total, oracle.naive(q, k, v, g, lam)) <= 1e-12


# ------------------------------------------------------------------ decode

def test_decode_replay_reproduces_the_double_sum():
    B, H, T, dk, dv = 2, 2, 70, 6, 5
    q, k, v, g, lam = rand_inputs(B, H, T, dk, dv, seed=12)
    Ls = (T).bit_length()  # room for the carry after the last token
    L = lam.shape[-1]
    ref = oracle.naive(q, k, v, g, lam)
    S = np.zeros((B, H, Ls, dk, dv))
    d = np.zeros((B, H, Ls))
    for t in range(T):
        lam_t = np.zeros((B, H, Ls + 1))
        lam_t[..., :L] = lam[:, :, t]
        o = oracle.decode_step(S, d, q[:, :, t], k[:, :, t], v[:, :, t], g[:, :, t], lam_t,
                               np.full(B, t))
        assert relerr(o, ref[:, :, t]) <= 1e-10
    # after T tokens the lazily decayed state equals the bucket states of [0,T)
    S_cf, d_cf = oracle.state_closed_form(k, v, g, np.full(B, T), Ls)
    live = np.array([(T >> i) & 1 for i in range(Ls)], bool)
    true_state = np.exp(d)[..., None, None] * S
    assert relerr(true_state[:, :, live], S_cf[:, :, live]) <= 1e-10
    assert np.all(S_cf[:, :, ~live] == 0)


def test_decode_from_closed_form_state_mid_sequence():
    """Start decode at a position p taken from the closed-form state and
    check the next outputs against the double sum."""
    B, H, T, dk, dv = 3, 1, 90, 4, 4
    q, k, v, g, lam = rand_inputs(B, H, T, dk, dv, seed=13)
    ref = oracle.naive(q, k, v, g, lam)
    L = lam.shape[-1]
    Ls = T.bit_length()
    pos = np.array([37, 64, 81])
    S, d = oracle.state_closed_form(k, v, g, pos, Ls)
    for step in range(T - 81):
        p = pos + step
        lam_t = np.zeros((B, H, Ls + 1))
        bidx = np.arange(B)
        lam_t[..., :L] = lam[bidx, :, p]
        o = oracle.decode_step(S, d, q[bidx, :, p], k[bidx, :, p], v[bidx, :, p],
                               g[bidx, :, p], lam_t, p)
        assert relerr(o, ref[bidx, :, p]) <= 1e-10


def test_decode_rejects_a_state_without_room():
    S = np.zeros((1, 1, 3, 2, 2))
    d = np.zeros((1, 1, 3))
    z = np.zeros((1, 1, 2))
    with pytest.raises(RuntimeError):  # bit_length(7 + 1) = 4 > 3 slots
        oracle.decode_step(S, d, z, z, z, np.zeros((1, 1)), np.zeros((1, 1, 4)), [7])


# ------------------------------------------------------- lambda's centre

def test_softplus_centre_is_one():
    """Page "Adaptive memory decay for Log-Linear Attention": the bias 0.54
    makes softplus start near 1.0."""
    assert abs(math.log1p(math.exp(0.54)) - 0.99916) < 5e-6


def test_naive_rows_equal_full_double_sum():
    q, k, v, g, lam = rand_inputs(1, 1, 130, 6, 5, seed=21)
    full = oracle.naive(q, k, v, g, lam)[0, 0]
    rows = [0, 1, 63, 64, 65, 127, 129]
    part = oracle.naive_rows(q[0, 0], k[0, 0], v[0, 0], g[0, 0], lam[0, 0], rows)
    np.testing.assert_array_equal(part, full[rows])


# ------------------------------------------------------ lambda producer

def mlp_inputs(N, Dd, L, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((N, Dd)), rng.standard_normal((Dd, 2 * L)) / math.sqrt(Dd),
            rng.standard_normal((2 * L, L)) / math.sqrt(2 * L), rng.standard_normal(L))


def inv_softplus(y):
    return y + np.log(-np.expm1(-y))


def test_lambda_mlp_initialisation_is_one():
    """Page "Adaptive memory decay for Log-Linear Attention": W2 = 0 and
    b = 0.54 make every weight softplus(0.54), about 1.0."""
    d, W1, _, _ = mlp_inputs(50, 16, 9, seed=1)
    lam = oracle.lambda_mlp(d, W1, np.zeros((18, 9)), np.full(9, 0.54))
    np.testing.assert_allclose(lam, 0.99916, atol=5e-6)


def test_lambda_mlp_layers_are_linear_in_d():
    """No activation between the two layers: the pre-activation is linear in d."""
    d1, W1, W2, b = mlp_inputs(40, 12, 7, seed=2)
    d2 = mlp_inputs(40, 12, 7, seed=3)[0]
    pre = lambda d: inv_softplus(oracle.lambda_mlp(d, W1, W2, b)) - b
    np.testing.assert_allclose(pre(d1 + d2), pre(d1) + pre(d2), rtol=1e-9, atol=1e-9)
    np.testing.assert_allclose(pre(3.0 * d1), 3.0 * pre(d1), rtol=1e-9, atol=1e-9)


def test_lambda_mlp_softplus_identities():
    """softplus(z) - softplus(-z) = z, positivity, and the tails z and e^z."""
    d, W1, W2, b = mlp_inputs(30, 8, 5, seed=4)
    plus = oracle.lambda_mlp(d, W1, W2, b)
    minus = oracle.lambda_mlp(d, W1, -W2, -b)
    z = (d @ W1) @ W2 + b
    np.testing.assert_allclose(plus - minus, z, rtol=1e-10, atol=1e-12)
    assert (plus > 0).all()
    big = oracle.lambda_mlp(d, W1, W2, b + 60.0)
    np.testing.assert_allclose(big, z + 60.0, rtol=1e-12)
    small = oracle.lambda_mlp(d, W1, W2, b - 60.0)
    np.testing.assert_allclose(small, np.exp(z - 60.0), rtol=1e-9)


def loss_of(q, k, v, g, lam, dout):
    return float(np.sum(dout * oracle.naive(q, k, v, g, lam)))


def test_backward_matches_finite_differences():
    q, k, v, g, lam = rand_inputs(1, 2, 7, 3, 2, seed=41)
    dout = np.random.default_rng(42).standard_normal(v.shape)
    grads = oracle.backward(q, k, v, g, lam, dout)
    args = [q, k, v, g, lam]
    h = 1e-6
    for which, grad in zip((0, 1, 2, 3, 4), (grads[0], grads[1], grads[2], grads[3], grads[4])):
        x = args[which]
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            saved = x[idx]
            x[idx] = saved + h
            up = loss_of(*args, dout)
            x[idx] = saved - h
            dn = loss_of(*args, dout)
            x[idx] = saved
            num[idx] = (up - dn) / (2 * h)
        assert np.max(np.abs(num - grad)) < 1e-7 * max(1.0, np.max(np.abs(grad))), which


def test_backward_dq_is_the_forward_with_swapped_roles():
    q, k, v, g, lam = rand_inputs(2, 1, 40, 5, 6, seed=43)
    dout = np.random.default_rng(44).standard_normal(v.shape)
    dq = oracle.backward(q, k, v, g, lam, dout)[0]
    assert relerr(dq, oracle.naive(dout, v, k, g, lam)) < 1e-12


def test_backward_euler_identities_and_gate_shift():
    q, k, v, g, lam = rand_inputs(1, 3, 33, 4, 5, seed=45, g_scale=0.3)
    dout = np.random.default_rng(46).standard_normal(v.shape)
    dq, dk, dv, dg, dlam = oracle.backward(q, k, v, g, lam, dout)
    loss = np.sum(dout * oracle.naive(q, k, v, g, lam), axis=(2, 3))
    for x, dx in ((q, dq), (k, dk), (v, dv), (lam, dlam)):
        assert np.allclose(np.sum(x * dx, axis=(2, 3)), loss, rtol=1e-11, atol=1e-11)
    # the loss sees G only through differences: the total gate gradient vanishes
    assert np.max(np.abs(dg[:, :, 0])) < 1e-11 * max(1.0, np.max(np.abs(dg)))


def test_backward_rows_equal_the_full_backward():
    q, k, v, g, lam = rand_inputs(1, 1, 45, 4, 3, seed=47)
    dout = np.random.default_rng(48).standard_normal(v.shape)
    dq, dk, dv, dg, dlam = oracle.backward(q, k, v, g, lam, dout)
    rows = [0, 7, 31, 44]
    rq, rl, rk, rv = oracle.backward_rows(q[0, 0], k[0, 0], v[0, 0], g[0, 0], lam[0, 0], dout[0, 0],
                                          rows, rows)
    for got, full in ((rq, dq), (rl, dlam), (rk, dk), (rv, dv)):
        assert relerr(got, full[0, 0, rows]) < 1e-13
