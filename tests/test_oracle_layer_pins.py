"""Pins of the oracle's composed layer stacks: the drafter's block pass and
the target's causal row.

Pages: "DFlash: how block diffusion boosts NVIDIA Blackwell throughput",
section "Block diffusion architecture" (a small drafter run once over the
block, the target's LM head shared); "DFlash-2: z-lab boosts speculative
decoding throughput", section "Architecture upgrade details" (a local
convolution between attention and MLP).  The layer itself is read as a
Qwen3-shaped pre-norm decoder layer: x += W_o attn(norm_in(x)); x +=
MLP(norm_post(x)); logits = LM_head(norm_final(x)).

The building blocks are pinned elsewhere; these checks pin how they are
composed, through special cases whose results PyTorch CPU routines
(``rms_norm``, ``linear``, ``silu``, ``conv1d``) compute directly:
- with the attention output and MLP down projections zero, every layer is
  the identity on the residual stream, so the logits are the LM head of the
  final-normed input rows (the context cannot matter);
- when every key carries the same V (identical block rows, no context; or a
  target token at position 0, which sees only itself), the softmax weights
  sum to one and attention returns that V whatever the scores, so one layer
  is a plain composition of norms and linear maps;
- with both projections zero and a width-3 kernel, a DFlash-2 layer adds
  the depthwise convolution of its input rows.
The last tests plant one plausible mistake at a time in source copies of
the oracle's functions and require every copy to fail at least one check.
"""
import inspect
import textwrap

import numpy as np
import torch
import torch.nn.functional as TF

import oracle as O
import oracle.dflash_oracle as OD
from tests.helpers import build_models, tiny_draft, tiny_target

WID = 73


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64))


def _close(a, b):
    return np.allclose(np.asarray(a), np.asarray(b), rtol=1e-10, atol=1e-12)


def _norm(x, g, eps):
    return TF.rms_norm(_t(x), (x.shape[-1],), _t(g), eps=eps)


def _split_v(m, wqkv_l):
    # rows of the fused projection: Q (q_dim), K (kv_dim), V (kv_dim)
    return wqkv_l[m.q_dim + m.kv_dim:m.q_dim + 2 * m.kv_dim]


def _attn_of_equal_values(m, x, S, l):
    """Attention output when every key's V is the V of rows x: each query
    head h returns V of KV head h // G."""
    a = _norm(x, S["in_norm"][l], m.rms_eps)
    v = TF.linear(a, _t(_split_v(m, S["wqkv"][l]))).reshape(x.shape[0], m.n_kv_heads, m.head_dim)
    G = m.n_q_heads // m.n_kv_heads
    o = v.repeat_interleave(G, dim=1).reshape(x.shape[0], m.q_dim)
    return TF.linear(o, _t(S["wo"][l]))


def _mlp_of(m, x, S, l):
    n = _norm(x, S["post_norm"][l], m.rms_eps)
    gu = S["w_gate_up"][l]
    F = m.mlp
    h = TF.silu(TF.linear(n, _t(gu[:F]))) * TF.linear(n, _t(gu[F:]))
    return TF.linear(h, _t(S["w_down"][l]))


def _head(m, x, S):
    return TF.linear(_norm(x, S["final_norm"], m.rms_eps), _t(S.lm_head))


def _distinct_gains(S, seed):
    """Norm gains are generated as ones; give every norm its own gains so
    that reading the wrong gain vector shows."""
    rng = np.random.default_rng(seed)
    for k in ("in_norm", "post_norm", "final_norm", "q_norm", "k_norm"):
        if k in S.d:
            S.d[k] = 0.5 + rng.random(S.d[k].shape)
    return S


def _draft_models(stack_cls, layers, conv_width=0, block=4):
    ds = tiny_draft(layers=layers, conv_width=conv_width, block=block)
    shared, _, dw = build_models(WID, tiny_target(), ds)
    return ds, _distinct_gains(stack_cls(ds, dw, shared), 10 * layers + conv_width)


# --------------------------------------------------------------------------
# check suites (each returns the names of the checks that failed)
# --------------------------------------------------------------------------
def draft_failures(draft, stack_cls=O.LayerStack):
    bad = []
    rng = np.random.default_rng(3)

    # zero branches: the residual stream keeps the embedded rows, whatever
    # the context holds
    ds, S = _draft_models(stack_cls, layers=2)
    S.d["wo"][:] = 0.0
    S.d["w_down"][:] = 0.0
    ck = [rng.standard_normal((5, ds.n_kv_heads, ds.head_dim)) for _ in range(ds.n_layers)]
    cv = [rng.standard_normal((5, ds.n_kv_heads, ds.head_dim)) for _ in range(ds.n_layers)]
    _, logits, xf = draft(ds, S, 7, 5, ck, cv, return_hidden=True)
    x0 = np.stack([S.embed[7]] + [S["mask_embed"]] * (ds.block - 1))
    if not np.array_equal(xf, x0):
        bad.append("zero branches: residual stream")
    if not _close(logits, _head(ds, x0, S).numpy()):
        bad.append("zero branches: logits")

    # one layer, equal values (identical rows, empty context), MLP off
    ds, S = _draft_models(stack_cls, layers=1)
    S.d["w_down"][:] = 0.0
    x0 = np.tile(S.embed[11], (ds.block, 1))
    empty = [np.zeros((0, ds.n_kv_heads, ds.head_dim))]
    _, _, xf = draft(ds, S, 11, 3, empty, empty, x0=x0, return_hidden=True)
    if not _close(xf, (_t(x0) + _attn_of_equal_values(ds, x0, S, 0)).numpy()):
        bad.append("attention branch")

    # one layer, attention output off: the MLP on the post-norm rows
    ds, S = _draft_models(stack_cls, layers=1)
    S.d["wo"][:] = 0.0
    x0 = rng.standard_normal((ds.block, ds.hidden))
    _, _, xf = draft(ds, S, 2, 9, empty, empty, x0=x0, return_hidden=True)
    if not _close(xf, (_t(x0) + _mlp_of(ds, x0, S, 0)).numpy()):
        bad.append("MLP branch")

    # one full layer, equal values: the MLP reads the post-attention stream
    ds, S = _draft_models(stack_cls, layers=1)
    x0 = np.tile(S.embed[4], (ds.block, 1))
    _, logits, xf = draft(ds, S, 4, 0, empty, empty, x0=x0, return_hidden=True)
    x1 = _t(x0) + _attn_of_equal_values(ds, x0, S, 0)
    x2 = x1 + _mlp_of(ds, x1.numpy(), S, 0)
    if not _close(xf, x2.numpy()) or not _close(logits, _head(ds, x2.numpy(), S).numpy()):
        bad.append("full layer")

    # DFlash-2: with both projections zero the layer adds the depthwise
    # convolution of its rows (zero padded at the block edges)
    ds, S = _draft_models(stack_cls, layers=1, conv_width=3)
    S.d["wo"][:] = 0.0
    S.d["w_down"][:] = 0.0
    x0 = rng.standard_normal((ds.block, ds.hidden))
    _, _, xf = draft(ds, S, 1, 2, empty, empty, x0=x0, return_hidden=True)
    w = S["conv"][0]                                        # [H][width]
    y = TF.conv1d(_t(x0).T[None], _t(w)[:, None, :], padding=(w.shape[1] - 1) // 2,
                  groups=ds.hidden)[0].T
    if not _close(xf, (_t(x0) + y).numpy()):
        bad.append("conv branch")
    return bad


def target_failures(row, stack_cls=O.LayerStack):
    bad = []
    # zero branches over two layers: taps and logits of the embedded token
    ts = tiny_target(layers=2)
    shared, tw, _ = build_models(WID, ts, tiny_draft())
    S = _distinct_gains(stack_cls(ts, tw, shared), 1)
    S.d["wo"][:] = 0.0
    S.d["w_down"][:] = 0.0
    cache = O.TargetCache(ts, 4)
    row(ts, S, 13, 0, cache, taps=())
    logits, taps = row(ts, S, 29, 1, cache, taps=(0, 1))
    e = S.embed[29]
    if not (np.array_equal(taps[0], e) and np.array_equal(taps[1], e)):
        bad.append("zero branches: taps")
    if not _close(logits, _head(ts, e[None], S).numpy()[0]):
        bad.append("zero branches: logits")

    # one full layer at position 0: the token attends to itself only
    ts = tiny_target(layers=1)
    shared, tw, _ = build_models(WID + 1, ts, tiny_draft())
    S = _distinct_gains(stack_cls(ts, tw, shared), 2)
    cache = O.TargetCache(ts, 2)
    logits, taps = row(ts, S, 17, 0, cache, taps=(0,))
    x0 = S.embed[17][None]
    x1 = _t(x0) + _attn_of_equal_values(ts, x0, S, 0)
    x2 = x1 + _mlp_of(ts, x1.numpy(), S, 0)
    if not _close(taps[0], x2.numpy()[0]):
        bad.append("full layer: tap")
    if not _close(logits, _head(ts, x2.numpy(), S).numpy()[0]):
        bad.append("full layer: logits")
    return bad


def test_draft_block_composition_pins():
    assert draft_failures(O.draft_block) == []


def test_target_row_composition_pins():
    assert target_failures(O.target_row) == []


# --------------------------------------------------------------------------
# planted mistakes: each source copy must fail at least one check
# --------------------------------------------------------------------------
def _mutant(fn, old, new):
    src = textwrap.dedent(inspect.getsource(fn))
    assert src.count(old) == 1, old
    ns = dict(vars(OD))
    exec(compile(src.replace(old, new), f"<{fn.__name__} with a planted mistake>", "exec"), ns)
    return ns[fn.__name__]


def _stack_with(method, old, new):
    return type("PlantedStack", (O.LayerStack,),
                {method: _mutant(getattr(O.LayerStack, method), old, new)})


DRAFT_PLANTS = {
    "attention residual dropped": ('x = x + linear(o, dw["wo"][l])', 'x = linear(o, dw["wo"][l])'),
    "MLP input not normed": ('dw.mlp(rmsnorm(x, dw["post_norm"][l], m.rms_eps), l)', "dw.mlp(x, l)"),
    "MLP norm takes the input gains": ('dw["post_norm"][l]', 'dw["in_norm"][l]'),
    "attention norm takes the MLP gains": ('dw["in_norm"][l]', 'dw["post_norm"][l]'),
    "final norm dropped": ('hf = rmsnorm(x, dw["final_norm"], m.rms_eps)', "hf = x"),
    "attention input not normed": ('a = rmsnorm(x, dw["in_norm"][l], m.rms_eps)', "a = x"),
    "conv replaces the stream": ('x = x + dwconv_block(x, dw["conv"][l])', 'x = dwconv_block(x, dw["conv"][l])'),
    "mask rows embed the anchor": ('x[1:] = dw["mask_embed"]', "x[1:] = dw.embed[anchor]"),
}
STACK_PLANTS = {
    "gate and up swapped": ("mlp", "silu(linear(x, wgu[:F])) * linear(x, wgu[F:])",
                            "linear(x, wgu[:F]) * silu(linear(x, wgu[F:]))"),
    "V rows taken from K": ("qkv_split", "w[m.q_dim + m.kv_dim:])", "w[m.q_dim:m.q_dim + m.kv_dim])"),
}
TARGET_PLANTS = {
    "attention residual dropped": ('x = x + linear(o.reshape(1, m.q_dim), tw["wo"][l])[0]',
                                   'x = linear(o.reshape(1, m.q_dim), tw["wo"][l])[0]'),
    "MLP input not normed": ('tw.mlp(rmsnorm(x[None], tw["post_norm"][l], m.rms_eps), l)', "tw.mlp(x[None], l)"),
    "MLP norm takes the input gains": ('tw["post_norm"][l]', 'tw["in_norm"][l]'),
    "final norm dropped": ('linear(rmsnorm(x[None], tw["final_norm"], m.rms_eps), tw.lm_head)',
                           "linear(x[None], tw.lm_head)"),
    "tap is the normed layer input": ("tapped[l] = x.copy()", "tapped[l] = a[0].copy()"),
}


def test_planted_draft_mistakes_fail_a_pin():
    for name, (old, new) in DRAFT_PLANTS.items():
        assert draft_failures(_mutant(O.draft_block, old, new)), name
    for name, (method, old, new) in STACK_PLANTS.items():
        assert draft_failures(O.draft_block, _stack_with(method, old, new)), name


def test_planted_target_mistakes_fail_a_pin():
    for name, (old, new) in TARGET_PLANTS.items():
        assert target_failures(_mutant(O.target_row, old, new)), name
    for name, (method, old, new) in STACK_PLANTS.items():
        assert target_failures(O.target_row, _stack_with(method, old, new)), name
