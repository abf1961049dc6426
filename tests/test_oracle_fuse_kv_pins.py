"""Pins of the oracle's context fuse and context K/V injection.

The fuse ("DFlash: how block diffusion boosts NVIDIA Blackwell throughput",
section "Block diffusion architecture": hidden states of several target
layers fused into one dense context feature) is read as concat -> linear ->
RMSNorm; the injection (same section: the feature enters the K and V
projections of every draft layer and stays in the draft KV cache) as each
draft layer's own W_k, W_v on the feature, k-norm and RoPE on K only, no
input norm on the feature.

Every check compares against something other than the oracle's own
arithmetic: direct indexing of the stored weights (one-hot inputs), PyTorch's
linear / rms_norm, complex rotation, and norm invariants.  The last test
plants plausible mistakes in copies of the two functions and requires each
copy to fail at least one check.
"""
import cmath
import math

import numpy as np
import torch
import torch.nn.functional as TF

import oracle as O
import workload as W
from tests.helpers import build_models, tiny_draft, tiny_target

WID = 57


def _models():
    ds = tiny_draft(hidden=64, hq=4, hkv=2, d=16, n_taps=3, layers=2)
    shared, _, dw = build_models(WID, tiny_target(hidden=64), ds)
    return ds, O.LayerStack(ds, dw, shared)


def _rng(seed):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------
# check suites (each returns the names of the checks that failed)
# --------------------------------------------------------------------------
def fuse_failures(fuse):
    ds, dws = _models()
    H, K = ds.hidden, ds.n_taps * ds.hidden
    bad = []

    # one-hot tap rows: W_fc e_j is column j of the stored weight; with the
    # norm the row is torch's rms_norm of that column
    g = 0.5 + _rng(1).random(H)
    dws.d["fc_norm"] = g.copy()
    cols = [0, 5, H + 3, K - 1]
    x = np.zeros((len(cols), K))
    for i, j in enumerate(cols):
        x[i, j] = 1.0
    got = fuse(ds, dws, x)
    for i, j in enumerate(cols):
        col = torch.from_numpy(dws["fc"][:, j].copy())
        want = TF.rms_norm(col, (H,), torch.from_numpy(g), eps=ds.rms_eps).numpy()
        if not np.allclose(got[i], want, rtol=1e-12, atol=1e-12):
            bad.append(f"one-hot column {j}")

    # identity blocks: W_fc = [0 .. I .. 0] selects tap slot s, so the
    # feature is the RMS-normalised tap of that slot, times the gains
    taps = _rng(2).standard_normal((5, K)) * 0.3
    for s in range(ds.n_taps):
        wfc = np.zeros((H, K))
        wfc[:, s * H:(s + 1) * H] = np.eye(H)
        dws.d["fc"] = wfc
        dws.d["fc_norm"] = np.full(H, 2.0)
        got = fuse(ds, dws, taps)
        h = taps[:, s * H:(s + 1) * H]
        want = 2.0 * h / np.sqrt(np.mean(h * h, axis=1, keepdims=True) + ds.rms_eps)
        if not np.allclose(got, want, rtol=1e-12, atol=1e-12):
            bad.append(f"identity slot {s}")

    # random weights and taps against torch (linear, then rms_norm)
    ds, dws = _models()
    taps = O.bf16_to_f64(W.taps_bf16(7, ds, WID))
    want = TF.rms_norm(TF.linear(torch.from_numpy(taps), torch.from_numpy(dws["fc"])),
                       (H,), torch.from_numpy(dws["fc_norm"]), eps=ds.rms_eps).numpy()
    if not np.allclose(fuse(ds, dws, taps), want, rtol=1e-10, atol=1e-12):
        bad.append("torch linear + rms_norm")

    # gains 1: every feature row has mean square m / (m + eps), m the mean
    # square of the pre-norm row (RMS ~ 1 for any input scale)
    dws.d["fc_norm"] = np.ones(H)
    for scale in (1e-2, 1.0, 37.0):
        c = fuse(ds, dws, taps * scale)
        pre = TF.linear(torch.from_numpy(taps * scale), torch.from_numpy(dws["fc"])).numpy()
        m = np.mean(pre * pre, axis=1)
        if not np.allclose(np.mean(c * c, axis=1), m / (m + ds.rms_eps), rtol=1e-10):
            bad.append(f"unit RMS at scale {scale}")
    return bad


def kv_failures(ctx_kv):
    ds, dws = _models()
    H, d, hkv = ds.hidden, ds.head_dim, ds.n_kv_heads
    qd, kvd = ds.q_dim, ds.kv_dim
    bad = []
    for l in range(ds.n_layers):
        wqkv = dws["wqkv"][l]          # [q rows | k rows | v rows][H]
        # non-unit k-norm gains, so that the gains' place relative to RoPE shows
        dws.d["k_norm"][l] = 0.5 + _rng(30 + l).random(d)
        kn = dws["k_norm"][l]
        # one-hot feature e_j at position 0: V is column j of the V rows;
        # K is the per-head rms_norm of column j of the K rows (no rotation
        # at position 0)
        for j in (0, 17, H - 1):
            c = np.zeros((1, H))
            c[0, j] = 1.0
            k, v = ctx_kv(ds, dws, l, c, np.array([0]))
            if not np.allclose(v.reshape(kvd), wqkv[qd + kvd:, j], rtol=0, atol=1e-15):
                bad.append(f"layer {l} V one-hot {j}")
            kcol = torch.from_numpy(wqkv[qd:qd + kvd, j].reshape(hkv, d).copy())
            want = TF.rms_norm(kcol, (d,), torch.from_numpy(kn), eps=ds.rms_eps).numpy()
            if not np.allclose(k.reshape(hkv, d), want, rtol=1e-12, atol=1e-12):
                bad.append(f"layer {l} K one-hot {j}")

        # rows at arbitrary positions: K is K(0) rotated pairwise (i, i+d/2)
        # by pos * base^(-2i/d), as a complex product; V does not move
        c = _rng(10 + l).standard_normal((4, H)) * 0.5
        pos = np.array([0, 1, 250, 4097])
        k, v = ctx_kv(ds, dws, l, c, pos)
        k0, v0 = ctx_kv(ds, dws, l, c, np.zeros(4, dtype=np.int64))
        if not np.array_equal(v, v0):
            bad.append(f"layer {l} V depends on position")
        vt = TF.linear(torch.from_numpy(c), torch.from_numpy(wqkv[qd + kvd:])).numpy()
        if not np.allclose(v.reshape(4, kvd), vt, rtol=1e-12, atol=1e-13):
            bad.append(f"layer {l} V against torch")
        for t in range(4):
            for h in range(hkv):
                for i in range(d // 2):
                    z0 = complex(k0[t, h, i], k0[t, h, i + d // 2])
                    ang = pos[t] * ds.rope_base ** (-2.0 * i / d)
                    z = z0 * cmath.exp(1j * ang)
                    if abs(complex(k[t, h, i], k[t, h, i + d // 2]) - z) > 1e-12:
                        bad.append(f"layer {l} K rotation row {t}")
                        break

        # k-norm with unit gains: every head of K has squared norm
        # d * m / (m + eps) (RoPE is a rotation), m the head's pre-norm mean square
        saved = dws.d["k_norm"][l].copy()
        dws.d["k_norm"][l] = np.ones(d)
        k, _ = ctx_kv(ds, dws, l, c * 3.0, pos)
        pre = TF.linear(torch.from_numpy(c * 3.0),
                        torch.from_numpy(wqkv[qd:qd + kvd])).numpy().reshape(4, hkv, d)
        m = np.mean(pre * pre, axis=-1)
        if not np.allclose(np.sum(k * k, axis=-1), d * m / (m + ds.rms_eps), rtol=1e-10):
            bad.append(f"layer {l} K head norm")
        dws.d["k_norm"][l] = saved

        # no input norm on the feature: V is linear in c, K is scale-free
        # (inputs large enough that eps moves K by < 1e-8 relative)
        k1, v1 = ctx_kv(ds, dws, l, c * 100.0, pos)
        k3, v3 = ctx_kv(ds, dws, l, c * 300.0, pos)
        if not np.allclose(v3, 3.0 * v1, rtol=1e-12, atol=1e-12):
            bad.append(f"layer {l} V not linear in the feature")
        if not np.allclose(k3, k1, rtol=1e-7, atol=1e-9):
            bad.append(f"layer {l} K not scale-free")
    return bad


# --------------------------------------------------------------------------
# the oracle passes
# --------------------------------------------------------------------------
def test_ctx_fuse_pins():
    assert fuse_failures(O.ctx_fuse) == []


def test_ctx_kv_pins():
    assert kv_failures(O.ctx_kv) == []


# --------------------------------------------------------------------------
# planted mistakes fail
# --------------------------------------------------------------------------
def _fuse_no_norm(ds, dw, taps):
    return O.linear(taps, dw["fc"])


def _fuse_norm_first(ds, dw, taps):
    x = np.asarray(taps, dtype=np.float64)
    x = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + ds.rms_eps)
    return O.linear(x, dw["fc"]) * dw["fc_norm"]


def _fuse_no_gain(ds, dw, taps):
    y = O.linear(taps, dw["fc"])
    return O.rmsnorm(y, np.ones(y.shape[-1]), ds.rms_eps)


def _fuse_slots_swapped(ds, dw, taps):
    H = ds.hidden
    t = np.asarray(taps, dtype=np.float64)
    t = np.concatenate([t[:, H:2 * H], t[:, :H], t[:, 2 * H:]], axis=1)
    return O.ctx_fuse(ds, dw, t)


def _kv_variant(kind):
    def fn(ds, dw, l, c, pos):
        m = ds
        wq, wk, wv = dw.qkv_split(l)
        if kind == "k_from_q_rows":
            wk = wq[:m.kv_dim]
        if kind == "kv_swapped":
            wk, wv = wv, wk
        if kind == "input_norm":
            c = O.rmsnorm(c, np.ones(c.shape[-1]), m.rms_eps)
        T = c.shape[0]
        k = O.linear(c, wk).reshape(T, m.n_kv_heads, m.head_dim)
        v = O.linear(c, wv).reshape(T, m.n_kv_heads, m.head_dim)
        if kind != "no_k_norm":
            k = O.rmsnorm(k, dw["k_norm"][l], m.rms_eps)
        if kind == "v_norm":
            v = O.rmsnorm(v, dw["k_norm"][l], m.rms_eps)
        p = np.asarray(pos, dtype=np.float64)
        if kind == "pos_plus_one":
            p = p + 1
        if kind == "norm_after_rope":
            k = O.linear(c, wk).reshape(T, m.n_kv_heads, m.head_dim)
            k = O.rope(k, p[:, None], m.rope_base)
            k = O.rmsnorm(k, dw["k_norm"][l], m.rms_eps)
        else:
            k = O.rope(k, p[:, None], m.rope_base)
        if kind == "v_rotated":
            v = O.rope(v, p[:, None], m.rope_base)
        if kind == "layer0":
            return O.ctx_kv(ds, dw, 0, c, pos)
        return k, v
    return fn


def test_planted_fuse_mistakes_fail_a_pin():
    for fn in (_fuse_no_norm, _fuse_norm_first, _fuse_no_gain, _fuse_slots_swapped):
        assert fuse_failures(fn), fn.__name__


def test_planted_kv_mistakes_fail_a_pin():
    for kind in ("k_from_q_rows", "kv_swapped", "input_norm", "no_k_norm", "v_norm",
                 "pos_plus_one", "norm_after_rope", "v_rotated", "layer0"):
        assert kv_failures(_kv_variant(kind)), kind
    assert kv_failures(_kv_variant("none")) == []
