"""Pins of the CPU oracle against what the mathematics and the pages fix.

Each test targets a plausible mistake (a dropped term, a wrong sign or index,
a transposed operand, an off-by-one in the verify bookkeeping) so that it
fails one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as TF

import oracle as O
import workload as W
from tests.helpers import build_models, tiny_draft, tiny_target

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def rnd(*shape, seed=0, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# --------------------------------------------------------------------------
# storage decode
# --------------------------------------------------------------------------
def test_bf16_decode_exact_values():
    bits = np.array([0x3F80, 0xBF80, 0x4000, 0x3E80, 0x0000, 0x4049], np.uint16)
    want = [1.0, -1.0, 2.0, 0.25, 0.0, 3.140625]
    assert O.bf16_to_f64(bits).tolist() == want


def test_bf16_roundtrip_of_generator_bits():
    x = np.float32([1.0, 1.00390625, 1.00390625 + 2 ** -20, 1.01171875, -3.5, 1e-3])
    y = O.bf16_to_f64(W.bf16_bits(x))
    # bf16 spacing at 1 is 2^-7: 1 + 2^-8 is a tie -> even (1.0); just above
    # the tie rounds up; 1 + 3*2^-8 is a tie between odd and even -> up
    assert y[:5].tolist() == [1.0, 1.0, 1.0078125, 1.015625, -3.5]
    assert abs(y[5] - 1e-3) / 1e-3 < 2 ** -8


# --------------------------------------------------------------------------
# RMSNorm
# --------------------------------------------------------------------------
def test_rmsnorm_closed_form():
    y = O.rmsnorm(np.array([3.0, 4.0]), np.ones(2), 0.0)
    r = math.sqrt((9 + 16) / 2)
    assert np.allclose(y, [3 / r, 4 / r], rtol=0, atol=1e-15)
    c = -2.5
    y = O.rmsnorm(np.full(7, c), np.full(7, 3.0), 1e-6)
    assert np.allclose(y, 3.0 * c / math.sqrt(c * c + 1e-6), atol=1e-14)


def test_rmsnorm_matches_torch():
    x = rnd(5, 33, seed=1)
    g = rnd(33, seed=2)
    want = TF.rms_norm(torch.from_numpy(x), (33,), torch.from_numpy(g), eps=1e-6)
    assert np.allclose(O.rmsnorm(x, g, 1e-6), want.numpy(), rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------
# RoPE
# --------------------------------------------------------------------------
def test_rope_golden_d2():
    cases = json.load(open(os.path.join(GOLD, "rope_rotation.json")))["cases"]
    for c in cases:
        got = O.rope(np.array(c["x"]), np.array(c["pos"]), 1e4)
        assert np.allclose(got, c["out"], atol=1e-14), c


def test_rope_pairs_and_frequencies_as_complex_rotation():
    d, base = 8, 1e4
    x = rnd(d, seed=3)
    p = 7.0
    got = O.rope(x, np.array(p), base)
    for i in range(d // 2):
        z = complex(x[i], x[i + d // 2]) * complex(math.cos(p * base ** (-2 * i / d)),
                                                   math.sin(p * base ** (-2 * i / d)))
        assert abs(got[i] - z.real) < 1e-13 and abs(got[i + d // 2] - z.imag) < 1e-13


def test_rope_relative_position_property():
    d = 16
    q, k = rnd(d, seed=4), rnd(d, seed=5)
    a = O.rope(q, np.array(11.0), 1e6) @ O.rope(k, np.array(4.0), 1e6)
    b = O.rope(q, np.array(1011.0), 1e6) @ O.rope(k, np.array(1004.0), 1e6)
    assert abs(a - b) < 1e-11
    assert np.allclose(O.rope(q, np.array(0.0), 1e6), q)


# --------------------------------------------------------------------------
# linear / SwiGLU / attention against independent routines
# --------------------------------------------------------------------------
def test_linear_matches_torch_nonsquare():
    x, w = rnd(3, 5, seed=6), rnd(7, 5, seed=7)
    want = TF.linear(torch.from_numpy(x), torch.from_numpy(w)).numpy()
    assert np.allclose(O.linear(x, w), want, atol=1e-13)


def test_silu_matches_torch_and_limits():
    x = np.linspace(-30, 30, 121)
    assert np.allclose(O.silu(x), TF.silu(torch.from_numpy(x)).numpy(), atol=1e-13)
    assert O.silu(np.array(0.0)) == 0.0


def test_swiglu_scalar_special_case():
    m = tiny_target(hidden=1, mlp=1, hq=1, hkv=1, d=2)
    a, b, c = 1.5, -0.75, 2.0
    ws = O.LayerStack.__new__(O.LayerStack)
    ws.shape = m
    ws.d = {"w_gate_up": np.array([[[a], [b]]]), "w_down": np.array([[[c]]])}
    for x in (0.3, -1.2, 2.0):
        got = ws.mlp(np.array([[x]]), 0)[0, 0]
        want = c * (a * x / (1 + math.exp(-a * x))) * (b * x)
        assert abs(got - want) < 1e-14


@pytest.mark.parametrize("hq,hkv", [(4, 4), (4, 2), (8, 1)])
def test_gqa_attention_matches_torch_sdpa(hq, hkv):
    nq, nk, d = 5, 9, 16
    q, k, v = rnd(nq, hq, d, seed=8), rnd(nk, hkv, d, seed=9), rnd(nk, hkv, d, seed=10)
    got = O.gqa_attention(q, k, v)
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]
    tk = torch.from_numpy(k).permute(1, 0, 2)[None].repeat_interleave(hq // hkv, dim=1)
    tv = torch.from_numpy(v).permute(1, 0, 2)[None].repeat_interleave(hq // hkv, dim=1)
    want = TF.scaled_dot_product_attention(tq, tk, tv)[0].permute(1, 0, 2).numpy()
    assert np.allclose(got, want, atol=1e-12)


def test_causal_mask_matches_torch_sdpa():
    n, h, d = 6, 2, 8
    q, k, v = rnd(n, h, d, seed=11), rnd(n, h, d, seed=12), rnd(n, h, d, seed=13)
    allowed = np.tril(np.ones((n, n), bool))
    got = O.gqa_attention(q, k, v, allowed)
    t = lambda a: torch.from_numpy(a).permute(1, 0, 2)[None]
    want = TF.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=True)[0]
    assert np.allclose(got, want.permute(1, 0, 2).numpy(), atol=1e-12)


def test_attention_single_key_and_equal_scores():
    v = rnd(1, 1, 4, seed=14)
    out = O.gqa_attention(rnd(3, 1, 4, seed=15), rnd(1, 1, 4, seed=16), v)
    assert np.allclose(out, v[0, 0])
    k = np.zeros((5, 1, 4))
    v = rnd(5, 1, 4, seed=17)
    out = O.gqa_attention(rnd(2, 1, 4, seed=18), k, v)
    assert np.allclose(out[0, 0], v[:, 0].mean(0))


# --------------------------------------------------------------------------
# DFlash-2 block conv
# --------------------------------------------------------------------------
def test_dwconv_reductions_and_locality():
    B, H = 6, 5
    x = rnd(B, H, seed=19)
    assert np.all(O.dwconv_block(x, np.zeros((H, 3))) == 0)
    w = np.zeros((H, 3))
    w[:, 1] = np.arange(H) * 0.1
    assert np.allclose(O.dwconv_block(x, w), x * w[:, 1])
    one = np.zeros((B, H))
    one[3, 2] = 1.0
    y = O.dwconv_block(one, rnd(H, 3, seed=20))
    nz = {tuple(i) for i in np.argwhere(y != 0)}
    assert nz <= {(2, 2), (3, 2), (4, 2)} and len(nz) == 3
    # edge: zero padding at the first position
    wl = np.zeros((H, 3))
    wl[:, 0] = 1.0     # y_p = x_{p-1}
    y = O.dwconv_block(x, wl)
    assert np.all(y[0] == 0) and np.allclose(y[1:], x[:-1])


# --------------------------------------------------------------------------
# Verify
# --------------------------------------------------------------------------
def test_verify_golden_cases():
    cases = json.load(open(os.path.join(GOLD, "verify_cases.json")))["cases"]
    for c in cases:
        n, em = O.verify_greedy(c["draft"], c["target"])
        assert n == c["n"] and em == c["emitted"], c


@pytest.mark.parametrize("B", [1, 2, 4, 8])
def test_verify_brute_force_all_patterns(B):
    import itertools
    for pattern in itertools.product([0, 1], repeat=B - 1):
        d = list(range(10, 10 + B - 1))
        t = [d[i] if pattern[i] else d[i] + 100 for i in range(B - 1)] + [999]
        n, em = O.verify_greedy(d, t)
        # definition: largest j with d_i == t_i for all i <= j
        want = max(j for j in range(B) if all(pattern[:j]))
        assert n == want
        assert 0 <= n <= B - 1 and len(em) == n + 1 and em[-1] == t[n]
        assert em[:n] == d[:n]


def test_verify_batch_bookkeeping():
    d = np.array([[5, 7, 9], [1, 2, 3]])
    t = np.array([[5, 7, 2, 4], [1, 2, 3, 8]])
    r = O.verify_batch(d, t, tgt_len=[100, 50], anchor_pos=[100, 50])
    assert r["n_accept"].tolist() == [2, 3]
    assert r["out_tokens"].tolist() == [[5, 7, 2, -1], [1, 2, 3, 8]]
    assert r["tgt_len"].tolist() == [103, 54]
    assert r["ctx_pending"].tolist() == [3, 4]
    assert r["anchor"].tolist() == [2, 8]
    assert r["anchor_pos"].tolist() == [103, 54]
    # the anchor (position 100 / 50) and the accepted drafts become context
    assert r["ctx_pos"].tolist() == [[100, 101, 102, -1], [50, 51, 52, 53]]


def test_synthetic_acceptance_closed_form():
    """E[n] = sum_{k=1}^{B-1} p^k and P(n = B-1) = p^(B-1) for the geometric
    agreement generator (block 16, p = 0.85)."""
    B, p, V, steps = 16, 0.85, 151936, 4000
    draft = W.uniform_tokens(steps * (B - 1), V, 99, 1).reshape(steps, B - 1)
    t = W.synth_target_ids(draft, p, V, seed=1234, step=0)
    ns = np.array([O.verify_greedy(draft[i], t[i])[0] for i in range(steps)])
    mean = sum(p ** k for k in range(1, B))
    assert abs(mean - p * (1 - p ** (B - 1)) / (1 - p)) < 1e-12   # 5.17166
    var = np.var(ns)
    assert abs(ns.mean() - mean) < 4 * math.sqrt(var / steps)
    pfull = p ** (B - 1)
    assert abs((ns == B - 1).mean() - pfull) < 4 * math.sqrt(pfull * (1 - pfull) / steps)


# --------------------------------------------------------------------------
# Draft step invariants
# --------------------------------------------------------------------------
def _draft_setup(conv_width=0, block=4, ctx_len=10, wid=41):
    ts = tiny_target()
    ds = tiny_draft(block=block, conv_width=conv_width)
    shared, tw, dw = build_models(wid, ts, ds)
    dws = O.LayerStack(ds, dw, shared)
    taps = O.bf16_to_f64(W.taps_bf16(ctx_len, ds, wid))
    c = O.ctx_fuse(ds, dws, taps)
    return ds, dws, c


def _ctx_lists(ds, dws, c, pos):
    ks, vs = [], []
    for l in range(ds.n_layers):
        k, v = O.ctx_kv(ds, dws, l, c, pos)
        ks.append(k)
        vs.append(v)
    return ks, vs


def test_incremental_append_equals_one_shot():
    ds, dws, c = _draft_setup(ctx_len=23)
    one = O.DraftContext(ds, 40)
    one.append(ds, dws, c, np.arange(23))
    inc = O.DraftContext(ds, 40, perm=np.random.default_rng(1).permutation(3))
    for lo, hi in [(0, 7), (7, 8), (8, 23)]:
        inc.append(ds, dws, c[lo:hi], np.arange(lo, hi))
    for l in range(ds.n_layers):
        a, b = one.read(l, 23), inc.read(l, 23)
        # equal up to BLAS blocking of the row batch (fp64 rounding only)
        assert np.allclose(a[0], b[0], rtol=0, atol=1e-12)
        assert np.allclose(a[1], b[1], rtol=0, atol=1e-12)


def test_block_output_invariant_to_context_storage_order():
    ds, dws, c = _draft_setup(ctx_len=37)
    outs = []
    for perm in (None, np.random.default_rng(5).permutation(3),
                 np.random.default_rng(6).permutation(3)):
        ctx = O.DraftContext(ds, 48, page=16, perm=perm)
        ctx.append(ds, dws, c, np.arange(37))
        ks = [ctx.read(l, 37)[0] for l in range(ds.n_layers)]
        vs = [ctx.read(l, 37)[1] for l in range(ds.n_layers)]
        outs.append(O.draft_block(ds, dws, 17, 37, ks, vs)[1])
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_block_shift_invariance_of_positions():
    """RoPE makes scores depend on position differences only: shifting every
    context position and the anchor position by the same amount leaves the
    logits unchanged.  Fails if context keys and block rows use different
    position conventions."""
    ds, dws, c = _draft_setup(ctx_len=12)
    a = O.draft_block(ds, dws, 3, 12, *_ctx_lists(ds, dws, c, np.arange(12)))[1]
    b = O.draft_block(ds, dws, 3, 512, *_ctx_lists(ds, dws, c, np.arange(500, 512)))[1]
    assert np.allclose(a, b, atol=1e-9)
    # a wrong anchor position (off by one) must change the logits
    d = O.draft_block(ds, dws, 3, 13, *_ctx_lists(ds, dws, c, np.arange(12)))[1]
    assert not np.allclose(a, d, atol=1e-6)


def test_block_is_non_causal():
    ds, dws, c = _draft_setup(ctx_len=9)
    ks, vs = _ctx_lists(ds, dws, c, np.arange(9))
    x0 = np.empty((ds.block, ds.hidden))
    x0[0] = dws.embed[5]
    x0[1:] = dws["mask_embed"]
    x1 = x0.copy()
    x1[-1] += 0.5 * rnd(ds.hidden, seed=21)
    _, la, ha = O.draft_block(ds, dws, 5, 9, ks, vs, x0=x0, return_hidden=True)
    _, lb, hb = O.draft_block(ds, dws, 5, 9, ks, vs, x0=x1, return_hidden=True)
    assert np.abs(ha[0] - hb[0]).max() > 1e-6      # last row reaches the first
    _, _, ca = O.draft_block(ds, dws, 5, 9, ks, vs, x0=x0, causal=True, return_hidden=True)
    _, _, cb = O.draft_block(ds, dws, 5, 9, ks, vs, x0=x1, causal=True, return_hidden=True)
    assert np.array_equal(ca[0], cb[0])             # a causal variant would not


def test_block_empty_context_is_plain_self_attention():
    ds, dws, c = _draft_setup(ctx_len=1)
    empty = [np.zeros((0, ds.n_kv_heads, ds.head_dim))] * ds.n_layers
    d, lg = O.draft_block(ds, dws, 9, 0, empty, empty)
    assert lg.shape == (ds.block, ds.vocab) and np.all(np.isfinite(lg))
    assert d.shape == (ds.block - 1,)


def test_conv_zero_weights_reduce_to_dflash():
    ds, dws, c = _draft_setup(conv_width=3)
    ks, vs = _ctx_lists(ds, dws, c, np.arange(10))
    with_conv = O.draft_block(ds, dws, 4, 10, ks, vs)[1]
    saved = dws.d["conv"].copy()
    dws.d["conv"][:] = 0.0
    zero = O.draft_block(ds, dws, 4, 10, ks, vs)[1]
    dws.d["conv"] = saved
    plain = tiny_draft(conv_width=0)
    ref = O.draft_block(plain, dws, 4, 10, ks, vs)[1]
    assert np.array_equal(zero, ref)
    assert not np.allclose(with_conv, ref)


def test_draft_argmax_lowest_index_on_ties():
    assert O.argmax_lowest(np.array([[1.0, 3.0, 3.0, 2.0]])).tolist() == [1]


# --------------------------------------------------------------------------
# Losslessness: speculative greedy == autoregressive greedy
# --------------------------------------------------------------------------
def _tiny_pair(wid, block=4):
    ts = tiny_target()
    ds = tiny_draft(block=block, n_taps=2)
    shared, tw, dw = build_models(wid, ts, ds, std=0.02, target_std=0.15)
    return (ts, O.LayerStack(ts, tw, shared), ds, O.LayerStack(ds, dw, shared))


@pytest.mark.parametrize("wid", [51, 52])
def test_spec_equals_ar_random_drafter(wid):
    ts, tws, ds, dws = _tiny_pair(wid)
    prompt = W.uniform_tokens(9, ts.vocab, wid, 3)
    ar = O.ar_generate(ts, tws, prompt, 24)
    sp = O.spec_generate(ts, tws, ds, dws, (0, 2), prompt, 24)
    assert sp == ar


def test_spec_equals_ar_adversarial_and_cheating_drafters():
    ts, tws, ds, dws = _tiny_pair(53, block=6)
    prompt = W.uniform_tokens(7, ts.vocab, 53, 3)
    ar = O.ar_generate(ts, tws, prompt, 40)
    P = len(prompt)
    # all drafts wrong: n = 0 on every iteration
    stats = []
    def wrong(anchor, L, ctx):
        return [(ar[j] + 1) % ts.vocab if j < len(ar) else 0
                for j in range(L - P + 1, L - P + ds.block)]

    sp = O.spec_generate(ts, tws, ds, dws, (1, 2), prompt, 40, drafter=wrong, stats=stats)
    assert sp == ar and set(stats) == {0}
    # the target's own tokens with seeded corruptions: exercises every n
    g = np.random.default_rng(7)
    stats = []

    def cheat(anchor, L, ctx):
        out = []
        for i in range(ds.block - 1):
            j = L - P + 1 + i
            tok = ar[j] if j < len(ar) else 0
            if g.random() < 0.12:
                tok = (tok + 1) % ts.vocab
            out.append(tok)
        return out

    for _ in range(3):
        sp = O.spec_generate(ts, tws, ds, dws, (1, 2), prompt, 40, drafter=cheat, stats=stats)
        assert sp == ar
    assert all(0 <= n <= ds.block - 1 for n in stats)
    assert len(set(stats)) >= 4 and max(stats) == ds.block - 1


def test_block_size_one_reduces_to_ar():
    ts, tws, ds, dws = _tiny_pair(54, block=1)
    prompt = W.uniform_tokens(5, ts.vocab, 54, 3)
    stats = []
    sp = O.spec_generate(ts, tws, ds, dws, (0, 1), prompt, 12, stats=stats)
    assert sp == O.ar_generate(ts, tws, prompt, 12)
    assert set(stats) == {0} and len(stats) == 11
