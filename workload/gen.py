"""Seeded generators: weights, tapped hidden states, context K/V, page tables,
request lengths and the synthetic stand-in for the target's verify tokens.

Nothing here computes any part of the drafting or verification method; the
oracle and the CUDA path both receive these arrays as inputs.
"""
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from .shapes import DraftShape, ModelShape, Workload

SEED_SALT = 20261202
CHUNK = 1 << 22

# Stable small integers naming each generated tensor (part of the seed).
TENSOR_IDS = {
    "embed": 1, "lm_head": 2, "mask_embed": 3, "fc": 4, "fc_norm": 5,
    "final_norm": 6,
    "in_norm": 10, "wqkv": 11, "q_norm": 12, "k_norm": 13, "wo": 14,
    "post_norm": 15, "w_gate_up": 16, "w_down": 17, "conv": 18,
    "taps": 200, "ctx_k": 201, "ctx_v": 202, "anchor": 203, "prompt": 204,
    "ctx_len": 205, "agree_p": 206, "page_perm": 207, "prev_accept": 208,
    "synth_seed": 209, "block_x": 210, "gain_jitter": 220,
}
TARGET_OFFSET = 100   # target-model tensors use TENSOR_IDS[name] + 100


def rng_for(wid: int, tid: int, *sub: int) -> np.random.Generator:
    ss = np.random.SeedSequence([int(wid), int(tid), *[int(s) for s in sub],
                                 SEED_SALT])
    return np.random.Generator(np.random.PCG64(ss))


def bf16_bits(x) -> np.ndarray:
    """float32 -> bfloat16 bit pattern, round to nearest even (finite input)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))) \
        >> np.uint32(16)
    return r.astype(np.uint16)


_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        n = max(1, min(32, len(os.sched_getaffinity(0))))
        _POOL = ThreadPoolExecutor(max_workers=n)
    return _POOL


def normal_bf16(shape, std: float, wid: int, tid: int, sub: int = 0) -> np.ndarray:
    """N(0, std^2) samples stored as bf16 bits; chunked so any thread count
    gives the same bits."""
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape)) if shape else 1
    out = np.empty(n, dtype=np.uint16)
    nchunks = max(1, (n + CHUNK - 1) // CHUNK)

    def work(c):
        lo = c * CHUNK
        hi = min(n, lo + CHUNK)
        g = rng_for(wid, tid, sub, c)
        x = g.standard_normal(hi - lo, dtype=np.float32)
        x *= np.float32(std)
        out[lo:hi] = bf16_bits(x)

    if nchunks == 1:
        work(0)
    else:
        list(_pool().map(work, range(nchunks)))
    return out.reshape(shape)


def ones_bf16(shape) -> np.ndarray:
    return np.full(shape, 0x3F80, dtype=np.uint16)


def uniform_tokens(n, vocab: int, wid: int, tid: int, sub: int = 0) -> np.ndarray:
    g = rng_for(wid, tid, sub)
    return g.integers(0, vocab, size=n, dtype=np.int64).astype(np.int32)


def _layer_weights(m: ModelShape, wid: int, off: int, std: float = 0.02):
    L, H, F, d = m.n_layers, m.hidden, m.mlp, m.head_dim
    t = lambda k: TENSOR_IDS[k] + off
    return {
        "in_norm": ones_bf16((L, H)),
        "wqkv": normal_bf16((L, m.qkv_rows, H), std, wid, t("wqkv")),
        "q_norm": ones_bf16((L, d)),
        "k_norm": ones_bf16((L, d)),
        "wo": normal_bf16((L, H, m.q_dim), std, wid, t("wo")),
        "post_norm": ones_bf16((L, H)),
        # gate rows [0, F), up rows [F, 2F) of each layer
        "w_gate_up": normal_bf16((L, 2 * F, H), std, wid, t("w_gate_up")),
        "w_down": normal_bf16((L, H, F), std, wid, t("w_down")),
    }


def shared_weights(m: ModelShape, wid: int, std: float = 0.02):
    """Token embedding and LM head shared by the target and the drafter."""
    return {
        "embed": normal_bf16((m.vocab, m.hidden), std, wid, TENSOR_IDS["embed"]),
        "lm_head": normal_bf16((m.vocab, m.hidden), std, wid,
                               TENSOR_IDS["lm_head"]),
    }


def draft_weights(d: DraftShape, wid: int, std: float = 0.02,
                  conv_std: float = 0.1):
    w = _layer_weights(d, wid, 0, std)
    H = d.hidden
    w["fc"] = normal_bf16((H, d.n_taps * H), std, wid, TENSOR_IDS["fc"])
    w["fc_norm"] = ones_bf16((H,))
    w["final_norm"] = ones_bf16((H,))
    w["mask_embed"] = normal_bf16((H,), std, wid, TENSOR_IDS["mask_embed"])
    if d.conv_width:
        w["conv"] = normal_bf16((d.n_layers, H, d.conv_width), conv_std, wid,
                                TENSOR_IDS["conv"])
    return w


GAIN_KEYS = ("in_norm", "post_norm", "q_norm", "k_norm", "final_norm", "fc_norm")


def jittered_gains(weights: dict, wid: int, std: float = 0.25) -> dict:
    """A copy of a weight dict whose RMSNorm gains are bf16(1 + std*N(0, 1))
    instead of ones, every gain tensor from its own stream: with distinct
    gains, reading the wrong gain vector changes the result."""
    out = dict(weights)
    for i, k in enumerate(GAIN_KEYS):
        if k in weights:
            g = rng_for(wid, TENSOR_IDS["gain_jitter"] + i)
            x = np.float32(1.0) + np.float32(std) * g.standard_normal(weights[k].shape,
                                                                      dtype=np.float32)
            out[k] = bf16_bits(x)
    return out


def target_weights(m: ModelShape, wid: int, std: float = 0.02):
    w = _layer_weights(m, wid, TARGET_OFFSET, std)
    w["final_norm"] = ones_bf16((m.hidden,))
    return w


def taps_bf16(rows: int, d: DraftShape, wid: int, sub: int = 0) -> np.ndarray:
    """Hidden states of the tapped target layers, N(0,1)/sqrt(H), [rows][k*H]."""
    return normal_bf16((rows, d.n_taps * d.hidden), 1.0 / math.sqrt(d.hidden),
                       wid, TENSOR_IDS["taps"], sub)


def context_kv_bf16(d: DraftShape, wid: int, layer: int, req: int, length: int,
                    kind: str) -> np.ndarray:
    """Already-projected context K or V of one request and layer, N(0,1),
    logical order [length][n_kv_heads][head_dim]."""
    tid = TENSOR_IDS["ctx_k" if kind == "k" else "ctx_v"]
    return normal_bf16((length, d.n_kv_heads, d.head_dim), 1.0, wid, tid,
                       layer * 65536 + req)


def ctx_lengths(w: Workload) -> np.ndarray:
    if w.ctx_len is not None:
        return np.full(w.batch, w.ctx_len, dtype=np.int32)
    lo, hi = w.ctx_len_range
    g = rng_for(w.wid, TENSOR_IDS["ctx_len"])
    return g.integers(lo, hi + 1, size=w.batch, dtype=np.int64).astype(np.int32)


def agreement_probs(w: Workload) -> np.ndarray:
    if w.agree_p is not None:
        return np.full(w.batch, w.agree_p, dtype=np.float64)
    lo, hi = w.agree_p_range
    g = rng_for(w.wid, TENSOR_IDS["agree_p"])
    return g.uniform(lo, hi, size=w.batch)


def new_row_counts(w: Workload) -> np.ndarray:
    """Context rows appended per request this step: fixed, or n_b + 1 with
    n_b a truncated geometric draw (successes before the first failure at
    agreement probability p_b, at most B-1)."""
    if w.new_rows is not None:
        return np.full(w.batch, w.new_rows, dtype=np.int32)
    p = agreement_probs(w)
    g = rng_for(w.wid, TENSOR_IDS["prev_accept"])
    n = g.geometric(1.0 - p) - 1
    n = np.minimum(n, w.draft.block - 1)
    return (n + 1).astype(np.int32)


def page_table(lengths, page_size: int, wid: int, shuffle: bool = True,
               spare_pages: int = 0):
    """Pages covering ``lengths[b]`` positions per request; physical page ids
    are a seeded permutation of the pool.  Returns (table[b][max_pages] int32
    with -1 padding, n_pages_total)."""
    lengths = np.asarray(lengths, dtype=np.int64)
    need = (lengths + page_size - 1) // page_size + spare_pages
    total = int(need.sum())
    ids = np.arange(total, dtype=np.int64)
    if shuffle:
        ids = rng_for(wid, TENSOR_IDS["page_perm"]).permutation(total)
    maxp = int(need.max()) if len(need) else 0
    table = np.full((len(lengths), max(1, maxp)), -1, dtype=np.int32)
    o = 0
    for b, k in enumerate(need):
        table[b, :k] = ids[o:o + k]
        o += int(k)
    return table, total


# ---------------------------------------------------------------------------
# Synthetic target tokens (stand-in for a target model's verify pass).
# Counter-based: splitmix64's output function (Steele, Lea and Flood, 2014)
# applied to a key built from (seed, step, request, position, stream).
# ---------------------------------------------------------------------------
_M64 = (1 << 64) - 1
_GOLD = 0x9E3779B97F4A7C15
_MIX1 = 0xBF58476D1CE4E5B9
_MIX2 = 0x94D049BB133111EB
_KEYMUL = 0x100000001B3  # FNV-1a 64-bit prime, used only to spread the key


def splitmix64_np(z: np.ndarray) -> np.ndarray:
    z = (z + np.uint64(_GOLD)).astype(np.uint64)
    z = (z ^ (z >> np.uint64(30))) * np.uint64(_MIX1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(_MIX2)
    return z ^ (z >> np.uint64(31))


def synth_key_np(seed, step, req, pos, stream) -> np.ndarray:
    with np.errstate(over="ignore"):
        k = np.uint64(seed)
        for part in (step, req, pos, stream):
            k = k * np.uint64(_KEYMUL) + np.asarray(part, dtype=np.uint64)
        return k.astype(np.uint64)


def agree_threshold(p: float) -> int:
    """Integer acceptance threshold on the top 53 bits of a hash."""
    return int(math.floor(min(max(p, 0.0), 1.0) * (1 << 53)))


def synth_target_ids(draft: np.ndarray, p, vocab: int, seed: int, step: int) -> np.ndarray:
    """t[b][i] for i = 1..B-1 equals draft[b][i-1] with probability p_b, else
    a uniform token different from it; t[b][B] is uniform.  Exactly the rule
    the CUDA stand-in kernel applies (same integer arithmetic)."""
    draft = np.asarray(draft, dtype=np.int64)
    b, bm1 = draft.shape
    p = np.broadcast_to(np.asarray(p, dtype=np.float64), (b,))
    thr = np.array([agree_threshold(x) for x in p], dtype=np.uint64)
    out = np.empty((b, bm1 + 1), dtype=np.int32)
    with np.errstate(over="ignore"):
        r = np.arange(b, dtype=np.uint64)[:, None]
        i = np.arange(bm1 + 1, dtype=np.uint64)[None, :]
        h0 = splitmix64_np(synth_key_np(seed, step, r, i, 0))
        h1 = splitmix64_np(synth_key_np(seed, step, r, i, 1))
        ok = (h0 >> np.uint64(11)) < thr[:, None]
        alt_off = (h1 % np.uint64(vocab - 1)).astype(np.int64) + 1
        full = (h1 % np.uint64(vocab)).astype(np.int64)
    d_ext = np.concatenate([draft, np.zeros((b, 1), np.int64)], axis=1)
    t = np.where(ok, d_ext, (d_ext + alt_off) % vocab)
    t[:, bm1] = full[:, bm1]
    out[:] = t
    return out
