"""End-to-end greedy speculative decoding on the GPU (causal target path).

Losslessness: GPU speculative output == GPU autoregressive output, token for
token (the target path is batch invariant).  Against the oracle: target
logits within 0.05 and tapped states within 2e-2 (relative row norm); tokens
equal up to the first position where the oracle's top-1/top-2 gap is <= 0.1.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workload as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_diffusion_speculative_fuse_gb300 import _build, binding
    _build.build()
    binding.load()


def models(wl, target_std=0.02, distinct_gains=False):
    from block_diffusion_speculative_fuse_gb300.device import DeviceModel
    ts, ds = wl.target, wl.draft
    shared = W.shared_weights(ts, wl.wid, std=target_std)
    tw = W.target_weights(ts, wl.wid, std=target_std)
    dw = W.draft_weights(ds, wl.wid)
    if distinct_gains:
        tw = W.jittered_gains(tw, wl.wid + 1)
        dw = W.jittered_gains(dw, wl.wid + 2)
    tm = DeviceModel(ts, tw, shared, draft=False)
    dm = DeviceModel(ds, dw, {k: tm.t[k] for k in ("embed", "lm_head")}, draft=True)
    return shared, tw, dw, tm, dm


@pytest.mark.parametrize("distinct_gains", [False, True])
def test_target_forward_parity_and_taps_tiny(distinct_gains):
    """distinct_gains: every RMSNorm of the target with its own non-unit
    gains (a kernel reading the wrong gain vector fails)."""
    from block_diffusion_speculative_fuse_gb300.device import i32
    from block_diffusion_speculative_fuse_gb300.generate import TargetRunner
    wl = W.get_workload("tiny_e2e")
    shared, tw, dw, tm, dm = models(wl, target_std=0.05, distinct_gains=distinct_gains)
    P = 40
    prompt = W.uniform_tokens(P, wl.target.vocab, wl.wid, W.TENSOR_IDS["prompt"])
    run = TargetRunner(tm, 1, 128, P, wl.tap_layers)
    logits = torch.zeros((P, wl.target.vocab), dtype=torch.float32, device="cuda")
    out, taps = run.forward(i32(prompt[None]), i32([0]), P, want_taps=True, logits=logits)
    torch.cuda.synchronize()
    tws = O.LayerStack(wl.target, tw, shared)
    cache = O.TargetCache(wl.target, 128)
    lref, href = O.target_rows(wl.target, tws, prompt, 0, cache, wl.tap_layers)
    lg = logits.cpu().numpy()
    assert np.abs(lg - lref).max() <= 0.05
    hg = taps.float().cpu().numpy()
    err = np.max(np.linalg.norm(hg - href, axis=1) / np.linalg.norm(href, axis=1))
    assert err <= 2e-2, err
    top = np.sort(lref, axis=-1)
    sure = (top[:, -1] - top[:, -2]) > 0.1
    assert np.array_equal(out.cpu().numpy()[0][sure], np.argmax(lref, -1)[sure])


def test_tiny_e2e_spec_equals_ar_and_oracle():
    """tiny_e2e: 4-layer H=256 target, 2-layer B=8 drafter, prompt 64,
    generate 128, batch 1."""
    from block_diffusion_speculative_fuse_gb300.generate import SpecDecoder, TargetRunner, \
        ar_generate
    wl = W.get_workload("tiny_e2e")
    shared, tw, dw, tm, dm = models(wl, target_std=0.05)
    P, N = wl.prompt_len, wl.gen_tokens
    prompt = W.uniform_tokens(P, wl.target.vocab, wl.wid, W.TENSOR_IDS["prompt"])[None]
    ar = ar_generate(TargetRunner(tm, 1, P + N + 1, P), prompt, N)
    sd = SpecDecoder(tm, dm, wl.tap_layers, 1, P + N)
    sp = sd.generate(prompt, N)
    assert np.array_equal(sp, ar), "speculative output differs from autoregressive output"
    assert all(0 <= n <= wl.draft.block - 1 for n in sd.stats)
    # oracle with teacher forcing on the GPU's own sequence: at every position
    # whose oracle top-1/top-2 gap exceeds 0.1 the GPU token is the argmax
    tws = O.LayerStack(wl.target, tw, shared)
    cache = O.TargetCache(wl.target, P + N + 1)
    seq = np.concatenate([prompt[0], ar[0, :-1]])
    lg, _ = O.target_rows(wl.target, tws, seq, 0, cache)
    lg = lg[P - 1:]
    top = np.sort(lg, axis=-1)
    sure = (top[:, -1] - top[:, -2]) > 0.1
    assert sure.sum() >= N // 5, "too few unambiguous positions to compare"
    assert np.array_equal(ar[0][sure], np.argmax(lg, -1)[sure])


def test_tiny_e2e_at_configured_init_spec_equals_ar_and_oracle():
    """tiny_e2e with the target drawn from N(0, 0.02), as the workload states.
    GPU speculative == GPU autoregressive for the whole run; against the
    oracle under teacher forcing every logit is within 0.05 and the token
    agrees wherever the oracle's top-1/top-2 gap exceeds 0.1 (at this init
    the logits are small, so few positions have such a gap; the 0.05-std
    test above checks the token rule on many more)."""
    from block_diffusion_speculative_fuse_gb300.device import i32
    from block_diffusion_speculative_fuse_gb300.generate import SpecDecoder, TargetRunner, \
        ar_generate
    wl = W.get_workload("tiny_e2e")
    shared, tw, dw, tm, dm = models(wl, target_std=0.02)
    P, N = wl.prompt_len, wl.gen_tokens
    prompt = W.uniform_tokens(P, wl.target.vocab, wl.wid, W.TENSOR_IDS["prompt"])[None]
    ar = ar_generate(TargetRunner(tm, 1, P + N + 1, P), prompt, N)
    sd = SpecDecoder(tm, dm, wl.tap_layers, 1, P + N)
    assert np.array_equal(sd.generate(prompt, N), ar)
    seq = np.concatenate([prompt[0], ar[0, :-1]])
    run = TargetRunner(tm, 1, len(seq) + 1, len(seq))
    logits = torch.zeros((len(seq), wl.target.vocab), dtype=torch.float32, device="cuda")
    run.forward(i32(seq[None]), i32([0]), len(seq), logits=logits)
    torch.cuda.synchronize()
    tws = O.LayerStack(wl.target, tw, shared)
    lref, _ = O.target_rows(wl.target, tws, seq, 0, O.TargetCache(wl.target, len(seq) + 1))
    assert np.abs(logits.cpu().numpy() - lref).max() <= 0.05
    lg = lref[P - 1:]
    top = np.sort(lg, axis=-1)
    sure = (top[:, -1] - top[:, -2]) > 0.1
    assert np.array_equal(ar[0][sure], np.argmax(lg, -1)[sure])


@pytest.mark.parametrize("block", [1, 4])
def test_spec_equals_ar_other_block_sizes(block):
    from dataclasses import replace
    from block_diffusion_speculative_fuse_gb300.generate import SpecDecoder, TargetRunner, \
        ar_generate
    wl = W.get_workload("tiny_e2e")
    wl = replace(wl, draft=replace(wl.draft, block=block))
    shared, tw, dw, tm, dm = models(wl, target_std=0.05)
    prompt = W.uniform_tokens(2 * 24, wl.target.vocab, 3, 3).reshape(2, 24)
    ar = ar_generate(TargetRunner(tm, 2, 24 + 40 + 1, 24), prompt, 40)
    sd = SpecDecoder(tm, dm, wl.tap_layers, 2, 24 + 40)
    assert np.array_equal(sd.generate(prompt, 40), ar)


def test_target_forward_rows_independent_of_batch():
    """Batch invariance of the target path across the row-scale code paths:
    3 requests x 16 rows in one call (48 rows per GEMM tile: one thread per
    row for the deferred RMSNorm scale) give bit-identical logits to each
    request alone (16 rows: one warp per row)."""
    from block_diffusion_speculative_fuse_gb300.device import i32
    from block_diffusion_speculative_fuse_gb300.generate import TargetRunner
    wl = W.get_workload("tiny_e2e")
    shared, tw, dw, tm, dm = models(wl, target_std=0.05)
    V, n, b = wl.target.vocab, 16, 3
    toks = W.uniform_tokens(b * n, V, wl.wid, W.TENSOR_IDS["prompt"], 7).reshape(b, n)
    run3 = TargetRunner(tm, b, 64, n)
    l3 = torch.zeros((b * n, V), dtype=torch.float32, device="cuda")
    out3, _ = run3.forward(i32(toks), i32([0] * b), n, logits=l3)
    for r in range(b):
        run1 = TargetRunner(tm, 1, 64, n)
        l1 = torch.zeros((n, V), dtype=torch.float32, device="cuda")
        out1, _ = run1.forward(i32(toks[r:r + 1]), i32([0]), n, logits=l1)
        torch.cuda.synchronize()
        assert torch.equal(l1, l3[r * n:(r + 1) * n]), r
        assert torch.equal(out1[0], out3[r])


@pytest.mark.parametrize("attn_tc", ["0", "1"])
def test_spec_equals_ar_either_target_attention(attn_tc, monkeypatch):
    """Both target attention kernels (tcgen05 query tiles with fixed key
    splits, and the mma.sync fallback; chosen at model creation) keep the
    target batch invariant: speculative == autoregressive, and one block
    verify gives the logits of one-token decode bit for bit."""
    from block_diffusion_speculative_fuse_gb300.device import i32
    from block_diffusion_speculative_fuse_gb300.generate import SpecDecoder, TargetRunner, \
        ar_generate
    monkeypatch.setenv("DFLASH_ATTN_TC", attn_tc)
    wl = W.get_workload("tiny_e2e")
    shared, tw, dw, tm, dm = models(wl, target_std=0.05)
    prompt = W.uniform_tokens(2 * 40, wl.target.vocab, 8, 8).reshape(2, 40)
    ar = ar_generate(TargetRunner(tm, 2, 40 + 48 + 1, 40), prompt, 48)
    sd = SpecDecoder(tm, dm, wl.tap_layers, 2, 40 + 48)
    assert np.array_equal(sd.generate(prompt, 48), ar)
    # 8 rows at once vs one at a time, after a 40-token prefill
    V, n = wl.target.vocab, 8
    toks = W.uniform_tokens(n, V, 9, 9)
    blk = TargetRunner(tm, 1, 64, 40)
    blk.forward(i32(prompt[:1]), i32([0]), 40)
    lb = torch.zeros((n, V), dtype=torch.float32, device="cuda")
    blk.forward(i32(toks[None]), i32([40]), n, logits=lb)
    one = TargetRunner(tm, 1, 64, 40)
    one.forward(i32(prompt[:1]), i32([0]), 40)
    for i in range(n):
        l1 = torch.zeros((1, V), dtype=torch.float32, device="cuda")
        one.forward(i32(toks[None, i:i + 1]), i32([40 + i]), 1, logits=l1)
        torch.cuda.synchronize()
        assert torch.equal(l1[0], lb[i]), i
