"""fp64 NumPy oracle: context fuse, K/V injection, non-causal block draft,
greedy verify, causal target forward and the speculative / autoregressive
generation loops.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source passages (cited by page title and section):
  [P1] "DFlash: how block diffusion boosts NVIDIA Blackwell throughput"
       (dothoosh.com), sections "Block diffusion architecture" and
       "Real-world integration".
  [P2] "DFlash-2: z-lab boosts speculative decoding throughput..."
       (dothoosh.com), sections "DFlash-2 mechanisms" and "Architecture
       upgrade details".
  [P3] "NVIDIA tests DFlash to cut LLM inference bottlenecks"
       (stechtimes.com), section "DFlash moves drafting to parallel compute".

Readings of points the pages leave open:
  R1 pre-norm RMSNorm decoder layers, SwiGLU MLP, GQA with per-head q/k
     RMSNorm before rotate-half RoPE (Qwen3-shaped);
  R2 a tap is the residual-stream output of a 0-indexed target layer;
  R3 fuse = concat taps in listed order -> linear (no bias) -> RMSNorm;
  R4 context K/V use each draft layer's own W_k, W_v on the fused feature
     (no per-layer input norm), k-norm and RoPE at the context position;
  R5 block inputs: embedding of the anchor, then one learned mask vector;
  R6 block position i sits at absolute position anchor_pos + i;
  R7 block rows attend, unmasked, to every context key and every block key;
  R8 DFlash-2 conv: x += depthwise width-w conv over block positions,
     zero padded, after the attention residual add, in every layer;
  R9 block rows 1..B-1 give the B-1 drafted tokens (argmax, lowest index on
     ties); the anchor row's logits are unused;
  R10 verify: longest prefix of drafts equal to the target's argmax, then the
     target's own token; the target cache keeps positions up to L+n.
"""
import math

import numpy as np

F64 = np.float64


# ---------------------------------------------------------------------------
# Storage decode
# ---------------------------------------------------------------------------
def bf16_to_f64(u16) -> np.ndarray:
    """bfloat16 bit patterns -> float64 (exact)."""
    u = np.ascontiguousarray(u16, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(F64)


# ---------------------------------------------------------------------------
# Building blocks (R1)
# ---------------------------------------------------------------------------
def rmsnorm(x, g, eps):
    """x * g / sqrt(mean(x^2) + eps) over the last axis."""
    x = np.asarray(x, dtype=F64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(g, dtype=F64)


def rope(x, pos, base):
    """Rotate-half rotary embedding.  Pair (x_i, x_{i+d/2}) is rotated by the
    angle pos * base^(-2i/d), i = 0 .. d/2-1.  ``pos`` broadcasts against
    x.shape[:-1]."""
    x = np.asarray(x, dtype=F64)
    d = x.shape[-1]
    half = d // 2
    inv_freq = np.power(F64(base), -np.arange(half, dtype=F64) * 2.0 / d)
    ang = np.asarray(pos, dtype=F64)[..., None] * inv_freq
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x):
    x = np.asarray(x, dtype=F64)
    return x / (1.0 + np.exp(-x))


def linear(x, w):
    """y = x W^T with W stored [out][in]."""
    return np.asarray(x, dtype=F64) @ np.asarray(w, dtype=F64).T


def softmax_attend(q, k, v, scale, allowed=None):
    """One query vector q [d] over keys k [n][d], values v [n][d]:
    softmax(scale * k q) v, restricted to ``allowed`` (bool [n]) if given."""
    s = (k @ q) * scale
    if allowed is not None:
        s = np.where(allowed, s, -np.inf)
    m = np.max(s)
    p = np.exp(s - m)
    p = p / np.sum(p)
    return p @ v


def gqa_attention(q, k, v, allowed=None):
    """q [nq][hq][d]; k, v [nk][hkv][d]; query head h reads KV head
    h // (hq / hkv) (grouped-query attention); scale 1/sqrt(d).
    ``allowed`` [nq][nk] bool or None (no mask)."""
    nq, hq, d = q.shape
    hkv = k.shape[1]
    grp = hq // hkv
    scale = 1.0 / math.sqrt(d)
    out = np.empty((nq, hq, d), dtype=F64)
    for i in range(nq):
        for h in range(hq):
            g = h // grp
            out[i, h] = softmax_attend(q[i, h], k[:, g], v[:, g], scale,
                                       None if allowed is None else allowed[i])
    return out


def dwconv_block(x, w):
    """Depthwise conv over block positions: y_p = sum_j w[:, j] x_{p+j-c},
    c = (width-1)/2, zero padded at the block edges.  x [B][H], w [H][width]."""
    x = np.asarray(x, dtype=F64)
    w = np.asarray(w, dtype=F64)
    B, H = x.shape
    width = w.shape[1]
    c = (width - 1) // 2
    y = np.zeros_like(x)
    for p in range(B):
        for j in range(width):
            src = p + j - c
            if 0 <= src < B:
                y[p] += w[:, j] * x[src]
    return y


def argmax_lowest(logits):
    """Index of the maximum along the last axis; the lowest index wins ties."""
    return np.argmax(np.asarray(logits), axis=-1)


# ---------------------------------------------------------------------------
# Weights
# ---------------------------------------------------------------------------
class LayerStack:
    """Decoded fp64 weights of a decoder-layer stack plus its extras."""

    def __init__(self, shape, w: dict, shared: dict):
        self.shape = shape
        self.d = {k: bf16_to_f64(v) for k, v in w.items()}
        self.embed = bf16_to_f64(shared["embed"])
        self.lm_head = bf16_to_f64(shared["lm_head"])

    def __getitem__(self, k):
        return self.d[k]

    def qkv_split(self, l):
        m = self.shape
        w = self.d["wqkv"][l]
        return (w[:m.q_dim], w[m.q_dim:m.q_dim + m.kv_dim],
                w[m.q_dim + m.kv_dim:])

    def mlp(self, x, l):
        F = self.shape.mlp
        wgu = self.d["w_gate_up"][l]
        return linear(silu(linear(x, wgu[:F])) * linear(x, wgu[F:]),
                      self.d["w_down"][l])


def _qk_heads(m, ws, l, a, pos):
    """Project rows a [n][H] to rotated q [n][hq][d], k, v [n][hkv][d]."""
    wq, wk, wv = ws.qkv_split(l)
    n = a.shape[0]
    q = linear(a, wq).reshape(n, m.n_q_heads, m.head_dim)
    k = linear(a, wk).reshape(n, m.n_kv_heads, m.head_dim)
    v = linear(a, wv).reshape(n, m.n_kv_heads, m.head_dim)
    if m.qk_norm:
        q = rmsnorm(q, ws["q_norm"][l], m.rms_eps)
        k = rmsnorm(k, ws["k_norm"][l], m.rms_eps)
    pos = np.asarray(pos, dtype=F64)
    q = rope(q, pos[:, None], m.rope_base)
    k = rope(k, pos[:, None], m.rope_base)
    return q, k, v


# ---------------------------------------------------------------------------
# Draft side: fuse (a1), K/V injection (a2), block draft (a3, a4)
# ---------------------------------------------------------------------------
def ctx_fuse(dshape, dw: LayerStack, taps):
    """c_t = RMSNorm_fc(W_fc [h^{l1}_t; ...; h^{lk}_t])  ([P1] "Block
    diffusion architecture": target hidden states from several layers fused
    into one dense context feature; reading R3)."""
    y = linear(taps, dw["fc"])
    if dshape.fc_norm:
        y = rmsnorm(y, dw["fc_norm"], dshape.rms_eps)
    return y


def ctx_kv(dshape, dw: LayerStack, l, c, pos):
    """K/V of context rows c [T][H] for draft layer l at positions pos [T]
    ([P1] "Block diffusion architecture": the feature enters the K and V
    projections of every draft layer; reading R4)."""
    m = dshape
    _, wk, wv = dw.qkv_split(l)
    T = c.shape[0]
    k = linear(c, wk).reshape(T, m.n_kv_heads, m.head_dim)
    v = linear(c, wv).reshape(T, m.n_kv_heads, m.head_dim)
    if m.qk_norm:
        k = rmsnorm(k, dw["k_norm"][l], m.rms_eps)
    k = rope(k, np.asarray(pos, dtype=F64)[:, None], m.rope_base)
    return k, v


class DraftContext:
    """Draft KV cache of one request: the projected context K/V per layer,
    kept across iterations ([P1] "Block diffusion architecture").  Stored in
    pages of ``page`` positions placed at arbitrary physical slots; reads go
    through the page table in logical order."""

    def __init__(self, dshape, capacity, page=16, perm=None):
        m = dshape
        self.m = m
        self.page = page
        npages = (capacity + page - 1) // page
        self.table = (np.arange(npages) if perm is None
                      else np.asarray(perm)[:npages])
        slots = int(np.max(self.table)) + 1 if npages else 0
        self.k = np.zeros((m.n_layers, slots, page, m.n_kv_heads, m.head_dim))
        self.v = np.zeros_like(self.k)
        self.length = 0

    def write(self, l, pos, k, v):
        for t, p in enumerate(np.asarray(pos)):
            pg, off = self.table[p // self.page], p % self.page
            self.k[l, pg, off] = k[t]
            self.v[l, pg, off] = v[t]

    def read(self, l, n):
        idx = np.arange(n)
        pg = self.table[idx // self.page]
        off = idx % self.page
        return self.k[l, pg, off], self.v[l, pg, off]

    def append(self, dshape, dw, c, pos):
        for l in range(dshape.n_layers):
            k, v = ctx_kv(dshape, dw, l, c, pos)
            self.write(l, pos, k, v)
        self.length = max(self.length, int(np.max(pos)) + 1)


def draft_block(dshape, dw: LayerStack, anchor, anchor_pos, ctx_k, ctx_v,
                x0=None, causal=False, return_hidden=False):
    """One non-causal pass of the drafter over [anchor, mask x (B-1)].

    ctx_k / ctx_v: per layer, the context keys/values [L][hkv][d] in logical
    order.  Returns (drafts [B-1], logits [B][V][, final residual [B][H]]).
    ([P1] "Block diffusion architecture": one parallel pass over the block;
    [P2] "DFlash-2 mechanisms": non-causal drafter; [P2] "Architecture
    upgrade details": local convolution between attention and MLP; [P3]
    "DFlash moves drafting to parallel compute": a block of masked future
    tokens in one forward pass.)  ``causal`` exists only for the negative
    test of non-causality.
    """
    m = dshape
    B = m.block
    if x0 is None:
        x = np.empty((B, m.hidden), dtype=F64)
        x[0] = dw.embed[anchor]
        x[1:] = dw["mask_embed"]
    else:
        x = np.array(x0, dtype=F64)
    pos = anchor_pos + np.arange(B)
    for l in range(m.n_layers):
        a = rmsnorm(x, dw["in_norm"][l], m.rms_eps)
        q, k, v = _qk_heads(m, dw, l, a, pos)
        K = np.concatenate([ctx_k[l], k], axis=0)
        V = np.concatenate([ctx_v[l], v], axis=0)
        allowed = None
        if causal:
            nctx = ctx_k[l].shape[0]
            allowed = np.arange(nctx + B)[None, :] <= (nctx + np.arange(B))[:, None]
        o = gqa_attention(q, K, V, allowed).reshape(B, m.q_dim)
        x = x + linear(o, dw["wo"][l])
        if m.conv_width:
            x = x + dwconv_block(x, dw["conv"][l])
        x = x + dw.mlp(rmsnorm(x, dw["post_norm"][l], m.rms_eps), l)
    hf = rmsnorm(x, dw["final_norm"], m.rms_eps)
    logits = linear(hf, dw.lm_head)
    drafts = argmax_lowest(logits[1:])
    if return_hidden:
        return drafts, logits, x
    return drafts, logits


# ---------------------------------------------------------------------------
# Verify (a5)
# ---------------------------------------------------------------------------
def verify_greedy(draft, target):
    """Temperature-0 verification of one request.  draft = d_1..d_{B-1},
    target = t_1..t_B (t_j is the target's argmax for the token at block
    position j).  Accept the longest prefix with d_i == t_i, then emit the
    target's own token t_{n+1} ([P1] "Introduction": lossless; [P3]
    "DFlash moves drafting to parallel compute": the target verifies).
    Returns (n, emitted list of n+1 tokens)."""
    draft = list(draft)
    target = list(target)
    n = 0
    while n < len(draft) and draft[n] == target[n]:
        n += 1
    return n, draft[:n] + [target[n]]


def verify_batch(draft, target, tgt_len, anchor_pos):
    """Batched form with the bookkeeping the hot path needs: out_tokens
    [b][B] (-1 padded), n [b], new target length, pending context rows n+1,
    their positions ctx_pos [b][B] (the anchor's and the accepted drafts':
    anchor_pos + j for j <= n, then -1; the rows spec_generate appends to
    the draft context), new anchor token and position."""
    draft = np.asarray(draft)
    target = np.asarray(target)
    b, B = target.shape
    out = np.full((b, B), -1, dtype=np.int32)
    n = np.zeros(b, dtype=np.int32)
    for r in range(b):
        nr, em = verify_greedy(draft[r], target[r])
        n[r] = nr
        out[r, :len(em)] = em
    tgt_len = np.asarray(tgt_len, dtype=np.int64)
    anchor_pos = np.asarray(anchor_pos, dtype=np.int64)
    new_anchor = target[np.arange(b), n]
    j = np.arange(B)[None, :]
    ctx_pos = np.where(j <= n[:, None], anchor_pos[:, None] + j, -1)
    return dict(out_tokens=out, n_accept=n,
                tgt_len=(tgt_len + n + 1).astype(np.int32),
                ctx_pending=(n + 1).astype(np.int32),
                ctx_pos=ctx_pos.astype(np.int32),
                anchor=new_anchor.astype(np.int32),
                anchor_pos=(anchor_pos + n + 1).astype(np.int32))


# ---------------------------------------------------------------------------
# Target side (a6): causal forward, one row at a time
# ---------------------------------------------------------------------------
class TargetCache:
    def __init__(self, m, capacity):
        self.k = np.zeros((m.n_layers, capacity, m.n_kv_heads, m.head_dim))
        self.v = np.zeros_like(self.k)
        self.length = 0


def target_row(m, tw: LayerStack, tok, pos, cache: TargetCache, taps=()):
    """Causal forward of one token at position pos; its K/V are written to
    the cache at pos and it attends to positions 0..pos.  Returns (logits
    [V], {layer: residual output [H]} for the tapped layers)."""
    x = tw.embed[tok].copy()
    tapped = {}
    for l in range(m.n_layers):
        a = rmsnorm(x[None], tw["in_norm"][l], m.rms_eps)
        q, k, v = _qk_heads(m, tw, l, a, np.array([pos]))
        cache.k[l, pos] = k[0]
        cache.v[l, pos] = v[0]
        o = gqa_attention(q, cache.k[l, :pos + 1], cache.v[l, :pos + 1])
        x = x + linear(o.reshape(1, m.q_dim), tw["wo"][l])[0]
        x = x + tw.mlp(rmsnorm(x[None], tw["post_norm"][l], m.rms_eps), l)[0]
        if l in taps:
            tapped[l] = x.copy()
    cache.length = max(cache.length, pos + 1)
    logits = linear(rmsnorm(x[None], tw["final_norm"], m.rms_eps), tw.lm_head)[0]
    return logits, tapped


def target_rows(m, tw, toks, pos0, cache, taps=()):
    """Rows processed in order, each exactly as target_row does."""
    logits, hs = [], []
    for i, t in enumerate(toks):
        lg, tp = target_row(m, tw, int(t), pos0 + i, cache, taps)
        logits.append(lg)
        hs.append(np.concatenate([tp[l] for l in taps]) if taps else None)
    return np.array(logits), (np.array(hs) if taps else None)


def ar_generate(m, tw, prompt, n_tokens):
    """Autoregressive greedy decoding: the reference result for losslessness."""
    cache = TargetCache(m, len(prompt) + n_tokens + 1)
    logits, _ = target_rows(m, tw, prompt, 0, cache)
    out = [int(argmax_lowest(logits[-1]))]
    pos = len(prompt)
    while len(out) < n_tokens:
        lg, _ = target_row(m, tw, out[-1], pos, cache)
        out.append(int(argmax_lowest(lg)))
        pos += 1
    return out


def spec_generate(tm, tw, dshape, dw, taps, prompt, n_tokens, drafter=None,
                  stats=None):
    """Greedy speculative decoding with the block drafter.

    Prefill: target over the prompt; its argmax at the last position is the
    first anchor; the prompt's tapped states become context rows 0..P-1.
    Each iteration: draft B-1 tokens from the anchor at position L; the
    target runs causally over [anchor, d_1..d_{B-1}] at L..L+B-1; accept n;
    emit d_1..d_n, t_{n+1}; the target cache keeps L..L+n; rows L..L+n are
    fused and appended to the draft context; the anchor becomes t_{n+1} at
    L+n+1.  ``drafter(anchor, L, ctx) -> drafts`` overrides the drafter (for
    adversarial tests)."""
    B = dshape.block
    P = len(prompt)
    cap = P + n_tokens + B + 1
    cache = TargetCache(tm, cap)
    ctx = DraftContext(dshape, cap)
    logits, h = target_rows(tm, tw, prompt, 0, cache, taps)
    anchor = int(argmax_lowest(logits[-1]))
    out = [anchor]
    ctx.append(dshape, dw, ctx_fuse(dshape, dw, h), np.arange(P))
    L = P
    while len(out) < n_tokens:
        if drafter is None:
            ks = [ctx.read(l, L)[0] for l in range(dshape.n_layers)]
            vs = [ctx.read(l, L)[1] for l in range(dshape.n_layers)]
            d, _ = draft_block(dshape, dw, anchor, L, ks, vs)
        else:
            d = np.asarray(drafter(anchor, L, ctx), dtype=np.int64)
        lg, h = target_rows(tm, tw, [anchor, *[int(t) for t in d]], L, cache, taps)
        t = argmax_lowest(lg)
        n, emitted = verify_greedy(d, t)
        if stats is not None:
            stats.append(n)
        # target cache keeps L..L+n (entries beyond are overwritten later)
        cache.length = L + n + 1
        ctx.append(dshape, dw, ctx_fuse(dshape, dw, h[:n + 1]),
                   L + np.arange(n + 1))
        out.extend(int(e) for e in emitted)
        anchor = int(emitted[-1])
        L = L + n + 1
    return out[:n_tokens]


__all__ = [
    "F64", "bf16_to_f64", "rmsnorm", "rope", "silu", "linear",
    "softmax_attend", "gqa_attention", "dwconv_block", "argmax_lowest",
    "LayerStack", "ctx_fuse", "ctx_kv", "DraftContext", "draft_block",
    "verify_greedy", "verify_batch", "TargetCache", "target_row",
    "target_rows", "ar_generate", "spec_generate",
]
