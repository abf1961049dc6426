"""GPU path vs the CPU oracle on the same seeded inputs, through the C ABI.

Tolerances (floating point, bf16 GPU vs fp64 oracle): max |d logit| <= 0.05,
max over rows of ||h_gpu - h||_2 / ||h||_2 <= 2e-2, argmax tokens equal
wherever the oracle's top-1/top-2 logit gap exceeds 0.1.  Integer work
(verify, acceptance, compaction) is compared bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workload as W
from workload.shapes import tiny_workload

pytestmark = pytest.mark.gpu

LOGIT_TOL = 0.05
HIDDEN_RTOL = 2e-2
GAP = 0.1


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_diffusion_speculative_fuse_gb300 import _build, binding
    _build.build()
    binding.load()


def B_():
    from block_diffusion_speculative_fuse_gb300 import binding
    return binding


def rel_rows(a, b):
    num = np.linalg.norm(a - b, axis=-1)
    den = np.linalg.norm(b, axis=-1)
    return float(np.max(num / den))


# --------------------------------------------------------------------- verify
def test_verify_bitexact_random_and_all_n():
    B = B_()
    rng = np.random.default_rng(0)
    for Bs in (1, 2, 8, 16, 32):
        n_req = 20000
        V = 50
        draft = rng.integers(0, V, size=(n_req, max(1, Bs - 1))).astype(np.int32)
        # force every acceptance length: copy a prefix of length k, then break
        target = rng.integers(0, V, size=(n_req, Bs)).astype(np.int32)
        k = rng.integers(0, Bs, size=n_req)
        for r in range(n_req):
            target[r, :k[r]] = draft[r, :k[r]]
            if k[r] < Bs - 1:
                target[r, k[r]] = (draft[r, k[r]] + 1) % V
        tl = rng.integers(0, 10000, size=n_req).astype(np.int32)
        ap = rng.integers(0, 10000, size=n_req).astype(np.int32)
        dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
        d_d, d_t, d_tl, d_ap = dev(draft), dev(target), dev(tl), dev(ap)
        out = torch.full((n_req, Bs), 7, dtype=torch.int32, device="cuda")
        n = torch.zeros(n_req, dtype=torch.int32, device="cuda")
        tlo, cp, ao, apo = (torch.zeros(n_req, dtype=torch.int32, device="cuda") for _ in range(4))
        cpos = torch.full((n_req, Bs), 7, dtype=torch.int32, device="cuda")
        B.dflash_verify_greedy(d_d if Bs > 1 else None, d_t, n_req, Bs, out, n, d_tl, tlo, cp,
                               ao, d_ap, apo, ctx_pos=cpos)
        torch.cuda.synchronize()
        ref = O.verify_batch(draft[:, :Bs - 1], target, tl, ap)
        assert np.array_equal(n.cpu().numpy(), ref["n_accept"])
        assert np.array_equal(out.cpu().numpy(), ref["out_tokens"])
        assert np.array_equal(tlo.cpu().numpy(), ref["tgt_len"])
        assert np.array_equal(cp.cpu().numpy(), ref["ctx_pending"])
        assert np.array_equal(ao.cpu().numpy(), ref["anchor"])
        assert np.array_equal(apo.cpu().numpy(), ref["anchor_pos"])
        assert np.array_equal(cpos.cpu().numpy(), ref["ctx_pos"])
        assert set(np.unique(ref["n_accept"])) == set(range(Bs))


def test_verify_in_place_aliasing():
    B = B_()
    draft = torch.tensor([[1, 2, 3]], dtype=torch.int32, device="cuda")
    target = torch.tensor([[1, 2, 9, 4]], dtype=torch.int32, device="cuda")
    ln = torch.tensor([100], dtype=torch.int32, device="cuda")
    ap = torch.tensor([100], dtype=torch.int32, device="cuda")
    B.dflash_verify_greedy(draft, target, 1, 4, None, None, ln, ln, None, None, ap, ap)
    torch.cuda.synchronize()
    assert ln.item() == 103 and ap.item() == 103


def test_synth_target_matches_generator_definition():
    B = B_()
    rng = np.random.default_rng(1)
    b, Bs, V = 32, 16, 151936
    draft = rng.integers(0, V, size=(b, Bs - 1)).astype(np.int32)
    p = rng.uniform(0.6, 0.95, size=b)
    thr = np.array([W.agree_threshold(x) for x in p], dtype=np.uint64)
    step = torch.tensor([5], dtype=torch.int64, device="cuda")
    out = torch.zeros((b, Bs), dtype=torch.int32, device="cuda")
    B.dflash_synth_target(torch.from_numpy(draft).cuda(), b, Bs,
                          torch.from_numpy(thr.view(np.int64)).cuda(), V, 77, step, 1, out)
    torch.cuda.synchronize()
    want = W.synth_target_ids(draft, p, V, seed=77, step=5)
    assert np.array_equal(out.cpu().numpy(), want)
    assert step.item() == 6


# ------------------------------------------------------------ GEMM (fuse)
@pytest.mark.parametrize("T,H,k,fc_norm", [(16, 256, 3, False), (5, 512, 2, True),
                                           (37, 256, 5, False), (130, 256, 2, True),
                                           (300, 384, 2, False)])
def test_ctx_fuse_parity(T, H, k, fc_norm):
    from block_diffusion_speculative_fuse_gb300.device import DeviceModel, to_device_u16
    B = B_()
    wl = tiny_workload("fuse", wid=700 + T, hidden=H, n_q_heads=H // 64, n_kv_heads=H // 128,
                       head_dim=64, mlp=256, vocab=256, n_taps=k, fc_norm=fc_norm)
    d = wl.draft
    w = W.draft_weights(d, wl.wid)
    sh = W.shared_weights(d, wl.wid)
    m = DeviceModel(d, w, sh, draft=True)
    taps = W.taps_bf16(T, d, wl.wid)
    ctx = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    ws = m.workspace(d.block, T, 1, 16)
    B.dflash_ctx_fuse(m.handle, to_device_u16(taps), T, ctx, ws)
    torch.cuda.synchronize()
    assert B.dflash_get_status(ws)[0] == 0
    got = ctx.float().cpu().numpy()
    want = O.ctx_fuse(d, O.LayerStack(d, w, sh), O.bf16_to_f64(taps))
    assert rel_rows(got, want) < 8e-3, rel_rows(got, want)


# ---------------------------------------------------------- K/V injection
def test_kv_append_parity_paged_and_shuffled():
    from block_diffusion_speculative_fuse_gb300.device import DeviceModel, PagedKV, i32, \
        to_device_u16
    B = B_()
    wl = tiny_workload("kv", wid=720, hidden=256, n_layers=3, n_q_heads=4, n_kv_heads=2,
                       head_dim=64, mlp=256, vocab=256)
    d = wl.draft
    w, sh = W.draft_weights(d, wl.wid), W.shared_weights(d, wl.wid)
    m = DeviceModel(d, w, sh, draft=True)
    lengths = [45, 17, 64]
    table, npg = W.page_table(lengths, 16, wl.wid, shuffle=True)
    kv = PagedKV(d, table, npg)
    T = sum(lengths)
    req = np.repeat(np.arange(3), lengths).astype(np.int32)
    pos = np.concatenate([np.arange(n) for n in lengths]).astype(np.int32)
    pos_in = pos.copy()
    pos_in[5] = -1  # skipped row
    c = W.normal_bf16((T, d.hidden), 1.0, wl.wid, 999)
    ws = m.workspace(d.block, T, 3, 64)
    B.dflash_kv_append(m.handle, to_device_u16(c), i32(req), i32(pos_in), T, kv.struct, ws)
    torch.cuda.synchronize()
    assert B.dflash_get_status(ws)[0] == 0
    dws = O.LayerStack(d, w, sh)
    cf = O.bf16_to_f64(c)
    for l in range(d.n_layers):
        o = 0
        for r, n in enumerate(lengths):
            k_ref, v_ref = O.ctx_kv(d, dws, l, cf[o:o + n], np.arange(n))
            kg, vg = kv.read_logical(l, r, n)
            kg, vg = kg.cpu().numpy(), vg.cpu().numpy()
            rows = [i for i in range(n) if not (r == 0 and i == 5)]
            assert rel_rows(kg[rows].reshape(len(rows), -1), k_ref[rows].reshape(len(rows), -1)) < 1e-2
            assert rel_rows(vg[rows].reshape(len(rows), -1), v_ref[rows].reshape(len(rows), -1)) < 1e-2
            o += n
    # the skipped row stays zero
    kg, _ = kv.read_logical(0, 0, 6)
    assert float(kg[5].abs().max()) == 0.0


# -------------------------------------------------------------- draft block
def draft_reference(st, d, dws, r, c_rows, o):
    h = st.host
    C, T = int(st.ctx_before[r]), int(st.new_rows[r])
    ks, vs = [], []
    for l in range(d.n_layers):
        kn, vn = O.ctx_kv(d, dws, l, c_rows[o:o + T], np.arange(C, C + T))
        if C:
            ks.append(np.concatenate([O.bf16_to_f64(h["ctx_k"][(l, r)]), kn]))
            vs.append(np.concatenate([O.bf16_to_f64(h["ctx_v"][(l, r)]), vn]))
        else:
            ks.append(kn)
            vs.append(vn)
    return O.draft_block(d, dws, int(h["anchor"][r]), C + T, ks, vs, return_hidden=True)


def check_draft_step(wl, weights=None):
    from block_diffusion_speculative_fuse_gb300.session import DraftStep
    st = DraftStep(wl, keep_host=True, weights=weights)
    d = wl.draft
    rows = st.batch * st.B
    logits = torch.zeros((rows, d.vocab), dtype=torch.float32, device="cuda")
    hidden = torch.zeros((rows, d.hidden), dtype=torch.float32, device="cuda")
    st.fuse()
    st.draft_block(logits=logits, hidden=hidden)
    torch.cuda.synchronize()
    status, site = st.status()
    assert status == 0, (status, site)
    h = st.host
    dws = O.LayerStack(d, h["weights"], h["shared"])
    c_rows = O.ctx_fuse(d, dws, O.bf16_to_f64(h["taps"]))
    lg = logits.cpu().numpy()
    hd = hidden.cpu().numpy()
    dr_gpu = st.draft.cpu().numpy()
    o = 0
    worst = 0.0
    for r in range(st.batch):
        dr, lref, href = draft_reference(st, d, dws, r, c_rows, o)
        o += int(st.new_rows[r])
        sl = slice(r * st.B, (r + 1) * st.B)
        err = np.abs(lg[sl] - lref).max()
        worst = max(worst, err)
        assert err <= LOGIT_TOL, f"request {r}: max |dlogit| {err}"
        assert rel_rows(hd[sl], href) <= HIDDEN_RTOL
        top = np.sort(lref[1:], axis=-1)
        sure = (top[:, -1] - top[:, -2]) > GAP
        assert np.array_equal(dr_gpu[r][sure], dr[sure])
    return st, worst


@pytest.mark.parametrize("kw", [
    dict(hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, block=8, batch=2),
    dict(hidden=256, n_q_heads=4, n_kv_heads=4, head_dim=64, block=8, batch=1),
    dict(hidden=512, n_q_heads=8, n_kv_heads=2, head_dim=64, block=16, batch=3),
    dict(hidden=512, n_q_heads=4, n_kv_heads=1, head_dim=128, block=16, batch=2),
    dict(hidden=512, n_q_heads=8, n_kv_heads=1, head_dim=64, block=4, batch=5),
    dict(hidden=256, n_q_heads=2, n_kv_heads=1, head_dim=128, block=16, batch=2, conv_width=3),
])
def test_draft_block_parity_small(kw):
    wl = tiny_workload("draft", wid=750 + kw["hidden"] + kw["batch"] + kw["block"], mlp=512,
                       vocab=2048, n_layers=2, n_taps=3, ctx_len_range=(1, 300), **kw)
    check_draft_step(wl)


@pytest.mark.parametrize("kw", [
    dict(hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, block=8, batch=3),
    dict(hidden=512, n_q_heads=4, n_kv_heads=1, head_dim=128, block=16, batch=2, conv_width=3),
    dict(hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=128, block=16, batch=16),
])
def test_draft_block_parity_distinct_norm_gains(kw):
    """Every RMSNorm (fuse, attention input, q/k, MLP input, final) with its
    own non-unit gains, so that a kernel reading the wrong gain vector (or
    none) fails.  The last case has 256 block rows: 128-row GEMM tiles and
    one-term activations past the first two layers."""
    wid = 900 + kw["hidden"] + kw["batch"]
    wl = tiny_workload("gains", wid=wid, mlp=256, vocab=1024, n_layers=3, n_taps=3,
                       ctx_len_range=(1, 400), **kw)
    check_draft_step(wl, weights=W.jittered_gains(W.draft_weights(wl.draft, wid), wid))


def test_draft_block_long_context_many_splits():
    wl = tiny_workload("long", wid=790, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=128,
                       mlp=256, vocab=1024, block=16, batch=2, ctx_len_range=(3000, 5000))
    check_draft_step(wl)


def test_draft_step_verify_and_status_clean():
    from block_diffusion_speculative_fuse_gb300.session import DraftStep
    wl = tiny_workload("sv", wid=795, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
                       mlp=256, vocab=1024, block=16, batch=4)
    st = DraftStep(wl)
    for _ in range(3):
        st.step()
    torch.cuda.synchronize()
    assert st.status()[0] == 0
    ref = O.verify_batch(st.draft.cpu().numpy(), st.target.cpu().numpy(),
                         st.tgt_len_in.cpu().numpy(), st.anchor_pos.cpu().numpy())
    assert np.array_equal(ref["out_tokens"], st.out_tokens.cpu().numpy())
    assert np.array_equal(ref["anchor_pos"], st.anchor_pos_out.cpu().numpy())
    assert st.step_counter.item() == 3


def test_draft_block_parity_wide_batch():
    """256 block rows (+ ragged context rows): the BN=256 GEMM path with
    several activation-row tiles, ragged paged attention."""
    wl = tiny_workload("wide", wid=796, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=128,
                       mlp=256, vocab=1024, block=16, batch=16, ctx_len_range=(16, 700))
    check_draft_step(wl)


def test_draft_block_parity_mma_sync_attention(monkeypatch):
    """The drafter on the mma.sync attention kernel (DFLASH_ATTN_TC=0, read at
    model creation) still matches the oracle."""
    monkeypatch.setenv("DFLASH_ATTN_TC", "0")
    wl = tiny_workload("mmasync", wid=797, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=128,
                       mlp=256, vocab=1024, block=16, batch=3, ctx_len_range=(1, 900))
    check_draft_step(wl)


def test_draft_block_parity_wide_query_tile_fallback():
    """block 32 x 8 query heads per KV head = 256 query rows per KV head: more
    than one tcgen05 tile, so the drafter takes the mma.sync kernel."""
    wl = tiny_workload("wideq", wid=798, hidden=512, n_q_heads=8, n_kv_heads=1, head_dim=64,
                       mlp=256, vocab=1024, block=32, batch=2, ctx_len_range=(10, 400))
    check_draft_step(wl)


@pytest.mark.parametrize("d,wid", [(64, 799), (128, 800)])
def test_draft_block_parity_single_softmax_state(d, wid):
    """8 query heads per KV head x block 16 = 128 query rows per KV head, so
    the tcgen05 attention runs one softmax state over all four warps instead
    of two warp pairs."""
    wl = tiny_workload("single", wid=wid, hidden=8 * d, n_q_heads=8, n_kv_heads=1, head_dim=d,
                       mlp=256, vocab=1024, block=16, batch=2, ctx_len_range=(5, 700))
    check_draft_step(wl)
