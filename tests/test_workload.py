"""Host logic of the seeded input generators (workload/), on CPU: they feed
both the CUDA path and the oracle, so their definitions are pinned here."""
import numpy as np
import torch

import workload as W
from workload import gen as G
from workload.shapes import tiny_workload


def test_streams_are_deterministic_and_distinct():
    a = W.rng_for(3, 7).standard_normal(5)
    b = W.rng_for(3, 7).standard_normal(5)
    c = W.rng_for(3, 8).standard_normal(5)
    d = W.rng_for(4, 7).standard_normal(5)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, c) and not np.array_equal(a, d)
    x = W.normal_bf16((300, 70), 0.02, 5, 11)
    assert np.array_equal(x, W.normal_bf16((300, 70), 0.02, 5, 11))
    assert x.dtype == np.uint16


def test_bf16_rounding_matches_torch():
    g = np.random.default_rng(0)
    x = np.concatenate([g.normal(size=10000) * s for s in (1e-30, 1e-3, 1.0, 1e20)])
    x = np.concatenate([x, [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8]]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(W.bf16_bits(x), ref)


def test_normal_samples_have_the_requested_scale():
    x = W.normal_bf16((512, 512), 0.02, 9, 3)
    f = (x.astype(np.uint32) << 16).view(np.float32)
    assert abs(float(f.std()) - 0.02) < 0.02 * 0.01
    assert abs(float(f.mean())) < 0.02 * 0.01


def test_page_table_is_a_permutation_of_the_pool():
    lengths = np.array([0, 1, 16, 17, 100])
    for shuffle in (False, True):
        table, total = W.page_table(lengths, 16, 3, shuffle=shuffle, spare_pages=1)
        need = (lengths + 15) // 16 + 1
        assert total == need.sum()
        assert table.shape == (5, need.max())
        used = np.concatenate([table[b, :need[b]] for b in range(5)])
        assert np.array_equal(np.sort(used), np.arange(total))
        for b in range(5):
            assert np.all(table[b, need[b]:] == -1)
        if not shuffle:
            assert np.array_equal(used, np.arange(total))


def test_lengths_and_pending_rows_stay_in_range():
    wl = tiny_workload("gen", wid=41, block=16, batch=500, ctx_len_range=(3, 70),
                       agree_p_range=(0.5, 0.95))
    c = W.ctx_lengths(wl)
    assert c.min() >= 3 and c.max() <= 70
    p = W.agreement_probs(wl)
    assert p.min() >= 0.5 and p.max() <= 0.95
    n = W.new_row_counts(wl)
    assert n.min() >= 1 and n.max() <= 16
    # n_b - 1 is a geometric count truncated at B - 1: mean close to the
    # truncated closed form sum_{k=1}^{15} p^k, averaged over requests
    expect = np.mean([sum(q ** k for k in range(1, 16)) for q in p])
    assert abs(float(np.mean(n - 1)) - expect) < 0.35
    fixed = tiny_workload("gen2", wid=42, batch=4, ctx_len=9, new_rows=3)
    assert np.all(W.ctx_lengths(fixed) == 9) and np.all(W.new_row_counts(fixed) == 3)


def test_agreement_threshold():
    assert W.agree_threshold(0.0) == 0
    assert W.agree_threshold(1.0) == 1 << 53
    assert W.agree_threshold(0.5) == 1 << 52
    assert W.agree_threshold(0.85) == int(0.85 * 2 ** 53)
    assert W.agree_threshold(-1.0) == 0 and W.agree_threshold(2.0) == 1 << 53


def test_splitmix64_published_sequence():
    """The synthetic target's counter-based generator is splitmix64's output
    function: from state 0, the generator's published first outputs."""
    gold = 0x9E3779B97F4A7C15
    z = np.array([(k * gold) % (1 << 64) for k in range(4)], dtype=np.uint64)
    with np.errstate(over="ignore"):
        out = [int(v) for v in G.splitmix64_np(z)]
    assert out == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F,
                   0xF88BB8A8724C81EC]


def test_jittered_gains_replace_only_the_norm_gains():
    d = tiny_workload("gains", wid=5, conv_width=3).draft
    w = W.draft_weights(d, 5)
    j = W.jittered_gains(w, 5)
    j2 = W.jittered_gains(w, 5)
    for k in w:
        if k in W.GAIN_KEYS:
            assert j[k].shape == w[k].shape and j[k].dtype == np.uint16
            assert np.array_equal(j[k], j2[k])                      # seeded
            g = (j[k].astype(np.uint32) << 16).view(np.float32)
            assert 0.5 < g.mean() < 1.5 and g.std() > 0.1           # not ones
        else:
            assert j[k] is w[k]
    gains = [j[k].ravel()[:64] for k in W.GAIN_KEYS if k in j]
    assert len({g.tobytes() for g in gains}) == len(gains)          # distinct per tensor
