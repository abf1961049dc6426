"""fp64 NumPy oracle for speculative verification at temperature T > 0.

TEST INFRASTRUCTURE ONLY (see the package docstring).

[P1] "DFlash: how block diffusion boosts NVIDIA Blackwell throughput"
(dothoosh.com) reports speedups in sampling mode as well as greedy mode
(section "Real-world integration", reasoning-model use case) and calls the
method lossless (introduction), but states no acceptance rule for sampling.
The reading taken here is the standard lossless rule of speculative sampling
(Leviathan, Kalman and Matias 2023; Chen et al. 2023), applied position by
position to a block draft:

  q_i = softmax(z_i / T) over the vocabulary: the drafter's distribution for
        block position i, from its logits z_i (block row i), i = 1..B-1;
  p_j = softmax(y_j / T): the target's distribution for the token at block
        position j, from its logits y_j (row j-1 of the target's causal pass
        over [anchor, d_1..d_{B-1}]), j = 1..B;
  draft d_i ~ q_i, drawn independently per position (the block pass gives
        every q_i at once, none conditioned on the other drafts);
  for i = 1, 2, ...: accept d_i when u_i * q_i(d_i) < p_i(d_i), i.e. with
        probability min(1, p_i(d_i) / q_i(d_i)); at the first rejection emit
        a token drawn from max(0, p_i - q_i) (normalised) and stop; when all
        B-1 drafts are accepted, emit a bonus token drawn from p_B.

Each emitted token then has exactly the target's distribution given the
tokens before it.  The argument is the single-step one: d_i is drawn from q_i
independently of the target's randomness, and p_i is conditioned on the
accepted prefix d_1..d_{i-1}.  So a block draft is as lossless as a
sequential one.

All randomness is passed in: one uniform in [0, 1) per draw.  A categorical
draw takes the smallest index k with a * S < C_k, where C_k is the running
sum of the (unnormalised) weights and S their total: the inverse of the
cumulative distribution, so index k has probability w_k / S exactly.
"""
import numpy as np

F64 = np.float64


def softmax_t(logits, T):
    """softmax(logits / T) along the last axis, in fp64 (max subtracted)."""
    z = np.asarray(logits, dtype=F64) / F64(T)
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def sample_inverse_cdf(weights, a):
    """Categorical draw from non-negative weights (last axis, need not sum to
    1) with uniforms a in [0, 1): the smallest k with a * S < C_k."""
    w = np.asarray(weights, dtype=F64)
    c = np.cumsum(w, axis=-1)
    s = c[..., -1:]
    a = np.asarray(a, dtype=F64)[..., None]
    k = np.sum(c <= a * s, axis=-1)  # number of prefixes not yet past a * S
    return np.minimum(k, w.shape[-1] - 1).astype(np.int64)


def draft_sample(draft_logits, T, a):
    """d_i ~ q_i for every request and block row 1..B-1.
    draft_logits: [b][B-1][V] (rows 1..B-1 of the block); a: [b][B-1]."""
    return sample_inverse_cdf(softmax_t(draft_logits, T), a)


def verify_sampling(draft, draft_logits, target_logits, T, u, w):
    """Speculative verification at temperature T for a batch of requests.

    draft:         [b][B-1] drafted tokens d_1..d_{B-1};
    draft_logits:  [b][B-1][V] drafter logits of block rows 1..B-1 (q);
    target_logits: [b][B][V] target logits for block positions 1..B (p);
    u:             [b][B-1] acceptance uniforms; w: [b][B] uniforms of the
                   residual draw at each position (w[:, B-1]: the bonus).
    Returns n [b] (accepted drafts) and out_tokens [b][B] (n + 1 emitted
    tokens, then -1), the same bookkeeping as the greedy verify."""
    draft = np.asarray(draft, dtype=np.int64)
    b, Bm1 = draft.shape
    B = Bm1 + 1
    q = softmax_t(draft_logits, T)
    p = softmax_t(target_logits, T)
    u = np.asarray(u, dtype=F64)
    w = np.asarray(w, dtype=F64)
    n = np.zeros(b, dtype=np.int32)
    out = np.full((b, B), -1, dtype=np.int64)
    for r in range(b):
        i = 0
        while i < Bm1:
            d = draft[r, i]
            if u[r, i] * q[r, i, d] < p[r, i, d]:
                out[r, i] = d
                i += 1
                continue
            resid = np.maximum(p[r, i] - q[r, i], 0.0)
            out[r, i] = sample_inverse_cdf(resid, w[r, i])
            break
        if i == Bm1:
            out[r, Bm1] = sample_inverse_cdf(p[r, Bm1], w[r, Bm1])
        n[r] = i
    return n, out.astype(np.int32)


__all__ = ["softmax_t", "sample_inverse_cdf", "draft_sample", "verify_sampling"]
