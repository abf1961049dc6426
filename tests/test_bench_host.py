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


def test_phase_roofline_reduces_to_hbm_at_batch_1_and_is_mixed_at_batch_32():
    hbm, tc = 6689.5, 1693.4
    for name, bound in (("qwen3_8b_b1", "hbm"), ("qwen3_8b_b32_paged", "tensor")):
        wl = W.get_workload(name)
        ctx, new = W.ctx_lengths(wl), W.new_row_counts(wl)
        ph = bench.phase_roofline(wl, ctx, new, "bf16", hbm, tc)
        hbm_ms = bench.step_bytes(wl, ctx, new) / (hbm * 1e9) * 1e3
        flop_ms = bench.step_flops(wl, ctx, new) / (tc * 1e12) * 1e3
        assert ph["gemm_bound"] == bound
        assert abs(ph["t_min_ms"] - (ph["attention_ms"] + ph["gemm_ms"])) < 1e-12
        # never below either whole-step bound, never above their sum
        assert ph["t_min_ms"] >= max(hbm_ms, flop_ms) - 1e-9
        assert ph["t_min_ms"] <= hbm_ms + flop_ms + 1e-9
        if bound == "hbm":
            assert abs(ph["t_min_ms"] - hbm_ms) < 1e-9
    # batch 32: ~1.48 ms (attention ~0.47 ms at HBM speed, the 512-row GEMMs
    # ~1.0 ms at the sustained tensor rate)
    wl = W.get_workload("qwen3_8b_b32_paged")
    ph = bench.phase_roofline(wl, W.ctx_lengths(wl), W.new_row_counts(wl), "bf16", hbm, tc)
    assert 1.3 < ph["t_min_ms"] < 1.6
