"""Host-side accounting of bench.py (no GPU): per-position acceptance from a
histogram, and the algorithmic bytes of the batch-1 step."""
import numpy as np

import bench
import workload as W


def test_acceptance_profile_of_an_exact_geometric_histogram():
    # p = 1/2, B = 4: P(n=0..3) = 1/2, 1/4, 1/8, 1/8 (n = 3 absorbs the tail)
    prof = bench.acceptance_profile([4, 2, 1, 1], np.full(3, 0.5))
    assert prof["samples"] == 8
    assert prof["p_accept_at_position"] == [0.5, 0.25, 0.125]
    assert prof["expected_p_accept_at_position"] == [0.5, 0.25, 0.125]
    assert prof["mean_accepted_drafts"] == (2 + 2 + 3) / 8


def test_acceptance_profile_mixes_requests():
    prof = bench.acceptance_profile([1, 0, 1], [0.2, 0.6])
    assert prof["p_accept_at_position"] == [0.5, 0.5]
    assert prof["expected_p_accept_at_position"] == [0.4, 0.2]


def test_acceptance_profile_matches_geometric_draws():
    p, B, n = 0.85, 16, 200_000
    rng = np.random.default_rng(5)
    agree = rng.random((n, B - 1)) < p
    accepted = np.where(agree.all(axis=1), B - 1, np.argmin(agree, axis=1))
    prof = bench.acceptance_profile(np.bincount(accepted, minlength=B), [p])
    i = np.arange(1, B)
    sigma = np.sqrt(p ** i * (1 - p ** i) / n)
    assert np.all(np.abs(np.array(prof["p_accept_at_position"]) - p ** i) < 3 * sigma + 1e-4)
    # E[n] = sum_{i=1}^{B-1} p^i
    assert abs(prof["mean_accepted_drafts"] - (p ** i).sum()) < 0.02


def test_step_bytes_of_the_batch1_step():
    """Weights once (fuse 83.9 M, 5 layers x 192.9 M, LM head 622.3 M
    parameters, bf16) plus the context K/V read once per layer."""
    wl = W.get_workload("qwen3_8b_b1")
    d = wl.draft
    ctx, new = W.ctx_lengths(wl), W.new_row_counts(wl)
    b = bench.step_bytes(wl, ctx, new)
    fuse = 4096 * 5 * 4096
    layer = (4096 * (4096 + 2 * 1024) + 4096 * 4096 + 3 * 12288 * 4096)
    lm = 151936 * 4096
    kv = 5 * 2 * 8 * 128 * (2048 + 16)
    approx = 2 * (fuse + 5 * layer + lm + kv)
    assert d.n_layers == 5 and d.hidden == 4096
    assert abs(b - approx) / approx < 1e-3
    assert abs(b - 3.385e9) / 3.385e9 < 1e-3
