"""Pins of the sampling-mode verify oracle (oracle/sampling.py), on CPU.

Brute force for the categorical draw, the greedy limit T -> 0 against the
greedy verify, exact special cases (q = p accepts everything, disjoint
supports reject and draw from p), and Monte Carlo checks of the properties
that make the rule lossless: each emitted token follows the target's
distribution given the tokens before it, and the acceptance rates match
their closed forms.  Monte Carlo bounds are 4.5 standard deviations on a
fixed seed.
"""
import numpy as np

import oracle as O
from oracle import sampling as S


def rng(seed):
    return np.random.default_rng(seed)


def test_inverse_cdf_brute_force_on_a_uniform_grid():
    w = np.array([0.0, 3.0, 1.0, 0.0, 4.0, 2.0])
    N = 10_000
    a = (np.arange(N) + 0.5) / N
    k = S.sample_inverse_cdf(np.broadcast_to(w, (N, w.size)), a)
    counts = np.bincount(k, minlength=w.size)
    expect = N * w / w.sum()
    assert np.all(np.abs(counts - expect) <= 1)
    assert counts[0] == 0 and counts[3] == 0          # zero weight: never drawn
    assert S.sample_inverse_cdf(w, 0.0) == 1          # a = 0: first positive weight
    assert S.sample_inverse_cdf(w, np.nextafter(1.0, 0.0)) == 5


def test_softmax_t_closed_form():
    z = np.array([0.0, np.log(3.0)])
    assert np.allclose(S.softmax_t(z, 1.0), [0.25, 0.75])
    assert np.allclose(S.softmax_t(z, 0.5), [0.1, 0.9])   # 1 : 9 at T = 1/2
    assert np.allclose(S.softmax_t(z + 1e4, 1.0), [0.25, 0.75])


def test_greedy_limit():
    """As T -> 0 both distributions become one-hot at the argmax: the
    drafts are the drafter's argmax and the verify is the greedy one."""
    g = rng(1)
    b, B, V, T = 64, 8, 50, 1e-4
    zd = g.normal(size=(b, B - 1, V))
    zt = g.normal(size=(b, B, V))
    # make the target agree with the drafter on a random prefix
    for r in range(b):
        m = g.integers(0, B)
        for i in range(min(m, B - 1)):
            zt[r, i, np.argmax(zd[r, i])] += 10.0
    d = S.draft_sample(zd, T, g.random((b, B - 1)))
    assert np.array_equal(d, np.argmax(zd, axis=-1))
    n, out = S.verify_sampling(d, zd, zt, T, g.random((b, B - 1)), g.random((b, B)))
    tgt = np.argmax(zt, axis=-1)
    for r in range(b):
        ng, em = O.verify_greedy(d[r], tgt[r])
        assert n[r] == ng
        assert list(out[r, :ng + 1]) == em
        assert np.all(out[r, ng + 1:] == -1)


def test_identical_distributions_accept_every_draft():
    g = rng(2)
    b, B, V, T = 32, 6, 20, 0.7
    zt = g.normal(size=(b, B, V))
    zd = zt[:, :B - 1].copy()
    d = S.draft_sample(zd, T, g.random((b, B - 1)))
    w = g.random((b, B))
    n, out = S.verify_sampling(d, zd, zt, T, g.random((b, B - 1)), w)
    assert np.all(n == B - 1)
    assert np.array_equal(out[:, :B - 1], d)
    bonus = S.sample_inverse_cdf(S.softmax_t(zt[:, B - 1], T), w[:, B - 1])
    assert np.array_equal(out[:, B - 1], bonus)


def test_disjoint_supports_reject_first_and_draw_from_target():
    g = rng(3)
    b, B, V, T = 32, 4, 8, 1.0
    zd = np.full((b, B - 1, V), -1e4)
    zd[:, :, :3] = g.normal(size=(b, B - 1, 3))       # drafter: tokens 0..2
    zt = np.full((b, B, V), -1e4)
    zt[:, :, 4:] = g.normal(size=(b, B, 4))           # target: tokens 4..7
    d = S.draft_sample(zd, T, g.random((b, B - 1)))
    w = g.random((b, B))
    n, out = S.verify_sampling(d, zd, zt, T, g.random((b, B - 1)), w)
    assert np.all(n == 0)
    first = S.sample_inverse_cdf(S.softmax_t(zt[:, 0], T), w[:, 0])
    assert np.array_equal(out[:, 0], first)
    assert np.all(out[:, 1:] == -1)


def mc_bound(p, N, k=4.5):
    return k * np.sqrt(np.maximum(p * (1 - p), 1e-12) / N) + 1e-9


def test_first_emitted_token_follows_the_target():
    """One draft (B = 2): whatever the drafter's q, the first emitted token
    (accepted draft or residual draw) is distributed as p_1, and the draft
    is accepted with probability sum_x min(p_1(x), q_1(x))."""
    g = rng(4)
    V, N, T = 6, 100_000, 0.8
    zd1 = g.normal(size=V) * 1.5
    zt1 = g.normal(size=V) * 1.5
    zt2 = g.normal(size=V)
    zd = np.broadcast_to(zd1, (N, 1, V))
    zt = np.broadcast_to(np.stack([zt1, zt2]), (N, 2, V))
    d = S.draft_sample(zd, T, g.random((N, 1)))
    n, out = S.verify_sampling(d, zd, zt, T, g.random((N, 1)), g.random((N, 2)))
    p1 = S.softmax_t(zt1, T)
    q1 = S.softmax_t(zd1, T)
    freq = np.bincount(out[:, 0], minlength=V) / N
    assert np.all(np.abs(freq - p1) < mc_bound(p1, N))
    acc = float(np.mean(n == 1))
    overlap = float(np.minimum(p1, q1).sum())
    assert abs(acc - overlap) < mc_bound(overlap, N)
    # drafts themselves follow q_1
    dfreq = np.bincount(d[:, 0], minlength=V) / N
    assert np.all(np.abs(dfreq - q1) < mc_bound(q1, N))
    # after an accepted draft the bonus token follows p_2
    p2 = S.softmax_t(zt2, T)
    sel = n == 1
    bfreq = np.bincount(out[sel, 1], minlength=V) / sel.sum()
    assert np.all(np.abs(bfreq - p2) < mc_bound(p2, sel.sum()))


def test_second_token_follows_the_target_given_the_first():
    """B = 3 with a causal target: p_2 depends on the first drafted token.
    Given that the first draft x was accepted, the second emitted token
    (the accepted second draft, or the residual draw at position 2) is
    distributed as p_2(. | x)."""
    g = rng(5)
    V, N, T = 4, 120_000, 1.0
    zd = np.broadcast_to(g.normal(size=(2, V)) * 1.2, (N, 2, V))
    zt1 = g.normal(size=V) * 1.2
    table = g.normal(size=(V, V)) * 1.2               # y_2 = table[d_1]
    d = S.draft_sample(zd, T, g.random((N, 2)))
    zt = np.empty((N, 3, V))
    zt[:, 0] = zt1
    zt[:, 1] = table[d[:, 0]]
    zt[:, 2] = 0.0
    n, out = S.verify_sampling(d, zd, zt, T, g.random((N, 2)), g.random((N, 3)))
    p1 = S.softmax_t(zt1, T)
    freq1 = np.bincount(out[:, 0], minlength=V) / N
    assert np.all(np.abs(freq1 - p1) < mc_bound(p1, N))
    for x in range(V):
        sel = (n >= 1) & (out[:, 0] == x)
        m = int(sel.sum())
        if m < 2000:
            continue
        p2 = S.softmax_t(table[x], T)
        f2 = np.bincount(out[sel, 1], minlength=V) / m
        assert np.all(np.abs(f2 - p2) < mc_bound(p2, m)), x


def test_accepted_length_with_independent_positions():
    """When p_j and q_j do not depend on the prefix, position i is reached
    with probability prod_{j <= i} sum_x min(p_j(x), q_j(x))."""
    g = rng(6)
    V, B, N, T = 5, 5, 100_000, 0.9
    zd1 = g.normal(size=(B - 1, V))
    zt1 = np.concatenate([zd1 + 0.6 * g.normal(size=(B - 1, V)), g.normal(size=(1, V))])
    zd = np.broadcast_to(zd1, (N, B - 1, V))
    zt = np.broadcast_to(zt1, (N, B, V))
    d = S.draft_sample(zd, T, g.random((N, B - 1)))
    n, out = S.verify_sampling(d, zd, zt, T, g.random((N, B - 1)), g.random((N, B)))
    ov = np.minimum(S.softmax_t(zt1[:B - 1], T), S.softmax_t(zd1, T)).sum(axis=-1)
    for i in range(1, B):
        expect = float(np.prod(ov[:i]))
        got = float(np.mean(n >= i))
        assert abs(got - expect) < mc_bound(expect, N), i
    # bookkeeping: n + 1 tokens, then -1
    cnt = (out >= 0).sum(axis=1)
    assert np.array_equal(cnt, n + 1)
