"""E4M3 (fp8) drafter context cache on the GPU against the oracle's codec and
draft pass (oracle/fp8.py, oracle.draft_block).

"DFlash-2: z-lab boosts speculative decoding throughput..." (section on the
cost of precision) compares an 8-bit KV cache with a 16-bit one.  Here the
context K/V are stored as E4M3 codes with one fp32 scale per (position, KV
head) vector, scale = amax / 448 of the vector's bf16 values; the block's own
K/V stay bf16.

Codes and scales are compared bit for bit: both sides take the scale
amax / 448 in fp32 and decide each code from the fp32 quotient value / scale
(round to nearest, ties to the even mantissa).  Draft logits: against the
oracle's draft pass over the decoded (quantize, then decode) context K/V,
within the bf16 parity tolerance 0.05.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workload as W
from oracle import fp8 as F
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
    return float(np.max(np.linalg.norm(a - b, axis=-1) / np.linalg.norm(b, axis=-1)))


def check_codes(codes, scales, x):
    """GPU codes [..., d] and scales [...] of the vectors x (fp64 values of
    bf16) against the oracle's quantizer, bit for bit."""
    rc, rs = F.quantize_kv(x)
    assert scales.dtype == np.float32
    assert np.array_equal(scales, rs), "scales differ"
    bad = np.argwhere(codes != rc)
    assert len(bad) == 0, f"{len(bad)} codes differ, first at {bad[:4].tolist()}"


def bf16_vectors(g, shape, d):
    """Random bf16 vectors over a wide range of magnitudes (per vector
    2^U(-30, 20)), as uint16 bits and fp64 values."""
    x = g.standard_normal(shape + (d,)) * np.exp2(g.uniform(-30, 20, size=shape + (1,)))
    bits = (np.asarray(x, dtype=np.float32).view(np.uint32) + 0x8000) >> 16
    bits = bits.astype(np.uint16)
    return bits, O.bf16_to_f64(bits)


def draft_model(wid, **kw):
    from block_diffusion_speculative_fuse_gb300.device import DeviceModel
    wl = tiny_workload("fp8", wid=wid, **kw)
    d = wl.draft
    w, sh = W.draft_weights(d, wl.wid), W.shared_weights(d, wl.wid)
    return wl, d, w, sh, DeviceModel(d, w, sh, draft=True)


# ------------------------------------------------------------------ codec
@pytest.mark.parametrize("d", [64, 128])
def test_kv_quantize_matches_oracle_codec(d):
    from block_diffusion_speculative_fuse_gb300.device import PagedKV
    B = B_()
    wl, ds, _, _, m = draft_model(900 + d, hidden=256, n_layers=2, n_q_heads=256 // d,
                                  n_kv_heads=2, head_dim=d, mlp=256, vocab=256)
    n_pages = 23
    table = np.arange(n_pages, dtype=np.int32)[None]
    kv = PagedKV(ds, table, n_pages)
    g = np.random.default_rng(d)
    bits, x = bf16_vectors(g, tuple(kv.pool.shape[:-1]), d)
    # special vectors: all zero, one nonzero, exact E4M3 ties (scale 1: the
    # largest element is 448, odd integers in [16, 32) lie halfway between
    # codes), and the smallest magnitudes of the subnormal range
    special = np.zeros((4, d))
    special[1, 7] = -3.25
    special[2, :16] = [448, 17, 19, 21, -23, 25, 27, 29, 31, 9, -11, 13, 15, 5, 7, 0.5]
    special[3, 0] = 448
    special[3, 1:9] = [2.0 ** -10, 3 * 2.0 ** -11, 2.0 ** -9, -(2.0 ** -10), 2.0 ** -8, 0, 7 * 2.0 ** -12,
                       3 * 2.0 ** -10]
    sb = (special.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(O.bf16_to_f64(sb), special)  # every special value is a bf16
    flat_bits, flat_x = bits.reshape(-1, d), x.reshape(-1, d)
    flat_bits[:4], flat_x[:4] = sb, special
    kv.pool.copy_(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16))
    q = kv.quantized(m)
    torch.cuda.synchronize()
    codes = q.pool.cpu().numpy()
    scales = q.scales.cpu().numpy()
    check_codes(codes, scales, x)
    # the tie vector rounds to even mantissas: 17 -> 16, 19 -> 20, ... (9..15 exact)
    c0 = codes.reshape(-1, d)[2, :16]
    assert list(F.e4m3_decode(c0)) == [448, 16, 20, 20, -24, 24, 28, 28, 32, 9, -11, 13, 15, 5, 7, 0.5]
    assert np.all(codes.reshape(-1, d)[0] == 0) and scales.reshape(-1)[0] == 1.0


def test_kv_quantize_rejects_bad_arguments():
    from block_diffusion_speculative_fuse_gb300.device import PagedKV
    B = B_()
    wl, ds, _, _, m = draft_model(905, hidden=256, n_layers=1, n_q_heads=4, n_kv_heads=2,
                                  head_dim=64, mlp=256, vocab=256)
    table = np.arange(4, dtype=np.int32)[None]
    src = PagedKV(ds, table, 4)
    dst = PagedKV(ds, table, 4, dtype="e4m3")
    with pytest.raises(B.DflashError):
        B.dflash_kv_quantize(m.handle, dst.struct, src.struct)      # wrong direction
    other = PagedKV(ds, np.arange(3, dtype=np.int32)[None], 3, dtype="e4m3")
    with pytest.raises(B.DflashError):
        B.dflash_kv_quantize(m.handle, src.struct, other.struct)    # page counts differ


# ---------------------------------------------------------- K/V injection
def test_kv_append_into_e4m3_cache():
    """The same rows appended to a bf16 cache and to an E4M3 cache: the E4M3
    codes and scales are the oracle's quantization of the bf16 cache's
    values; a skipped row (position -1) is not written."""
    from block_diffusion_speculative_fuse_gb300.device import PagedKV, i32, to_device_u16
    B = B_()
    wl, d, w, sh, m = draft_model(910, hidden=512, n_layers=3, n_q_heads=4, n_kv_heads=2,
                                  head_dim=128, mlp=256, vocab=256)
    lengths = [45, 17, 64]
    table, npg = W.page_table(lengths, 16, wl.wid, shuffle=True)
    kv16 = PagedKV(d, table, npg)
    kv8 = PagedKV(d, table, npg, dtype="e4m3")
    T = sum(lengths)
    req = np.repeat(np.arange(3), lengths).astype(np.int32)
    pos = np.concatenate([np.arange(n) for n in lengths]).astype(np.int32)
    pos[5] = -1
    c = to_device_u16(W.normal_bf16((T, d.hidden), 1.0, wl.wid, 999))
    ws = m.workspace(d.block, T, 3, 64)
    for kv in (kv16, kv8):
        B.dflash_kv_append(m.handle, c, i32(req), i32(pos), T, kv.struct, ws)
    torch.cuda.synchronize()
    assert B.dflash_get_status(ws)[0] == 0
    for l in range(d.n_layers):
        for r, n in enumerate(lengths):
            k, v = kv16.read_logical(l, r, n)
            x = np.stack([k.cpu().numpy(), v.cpu().numpy()], axis=1).astype(np.float64)
            codes, scales = kv8.read_codes(l, r, n)
            rows = [i for i in range(n) if not (r == 0 and i == 5)]
            check_codes(codes[rows], scales[rows], x[rows])
    codes, scales = kv8.read_codes(0, 0, 6)
    assert np.all(codes[5] == 0) and np.all(scales[5] == 0)


# -------------------------------------------------------------- draft block
def oracle_request_fp8(st, d, dws, c_rows, r):
    """The oracle's draft pass of request r over decoded E4M3 context K/V
    (the cached context and the rows appended this step)."""
    h = st.host
    offs = np.concatenate([[0], np.cumsum(st.new_rows)])
    C, T = int(st.ctx_before[r]), int(st.new_rows[r])
    ks, vs = [], []
    for l in range(d.n_layers):
        kn, vn = O.ctx_kv(d, dws, l, c_rows[offs[r]:offs[r] + T], np.arange(C, C + T))
        k = np.concatenate([O.bf16_to_f64(h["ctx_k"][(l, r)]), kn]) if C else kn
        v = np.concatenate([O.bf16_to_f64(h["ctx_v"][(l, r)]), vn]) if C else vn
        ks.append(F.kv_roundtrip(k))
        vs.append(F.kv_roundtrip(v))
    return O.draft_block(d, dws, int(h["anchor"][r]), C + T, ks, vs, return_hidden=True)


def check_fp8_step(wl, requests=None, graph=False):
    """Draft step with an E4M3 context cache vs the oracle; returns the
    E4M3-vs-bf16 drafts' prefix agreement per request."""
    from block_diffusion_speculative_fuse_gb300.session import DraftStep
    d = wl.draft
    st = DraftStep(wl, keep_host=True, kv_dtype="e4m3")
    assert st.kv.dtype == "e4m3"
    rows = st.batch * st.B
    logits = torch.zeros((rows, d.vocab), dtype=torch.float32, device="cuda")
    hidden = torch.zeros((rows, d.hidden), dtype=torch.float32, device="cuda")
    if graph:
        stream = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            st.fuse(stream)
            st.draft_block(logits=logits, hidden=hidden, stream=stream)
        with torch.cuda.stream(stream):
            g.replay()
    else:
        st.fuse()
        st.draft_block(logits=logits, hidden=hidden)
    torch.cuda.synchronize()
    assert st.status()[0] == 0, st.status()
    h = st.host
    dws = O.LayerStack(d, h["weights"], h["shared"])
    taps = O.bf16_to_f64(h["taps"])
    offs = np.concatenate([[0], np.cumsum(st.new_rows)])
    requests = list(range(st.batch)) if requests is None else requests
    c_rows = np.zeros((taps.shape[0], d.hidden))
    for r in requests:
        c_rows[offs[r]:offs[r + 1]] = O.ctx_fuse(d, dws, taps[offs[r]:offs[r + 1]])
    lg_all = logits.cpu().numpy()
    hd_all = hidden.cpu().numpy()
    drafts = st.draft.cpu().numpy()
    worst = 0.0
    for r in requests:
        dr, lref, href = oracle_request_fp8(st, d, dws, c_rows, r)
        sl = slice(r * st.B, (r + 1) * st.B)
        err = float(np.abs(lg_all[sl] - lref).max())
        worst = max(worst, err)
        assert err <= LOGIT_TOL, f"request {r}: max |dlogit| {err}"
        assert rel_rows(hd_all[sl], href) <= HIDDEN_RTOL
        top = np.sort(lref[1:], axis=-1)
        sure = (top[:, -1] - top[:, -2]) > GAP
        assert np.array_equal(drafts[r][sure], dr[sure])
    # the same step over a bf16 cache: how far the E4M3 drafts follow it
    st16 = DraftStep(wl, model=st.model)
    st16.fuse()
    st16.draft_block()
    torch.cuda.synchronize()
    d16 = st16.draft.cpu().numpy()
    same = drafts == d16
    prefix = np.where(same.all(1), same.shape[1], np.argmin(same, axis=1))
    print(f"\n{wl.name}: max |dlogit| vs oracle {worst:.4f}; E4M3 drafts equal to bf16 "
          f"drafts {same.mean():.3f}, mean matching prefix {prefix.mean():.2f} of {same.shape[1]}")
    return prefix


@pytest.mark.parametrize("kw", [
    dict(hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, block=8, batch=2),
    dict(hidden=512, n_q_heads=4, n_kv_heads=1, head_dim=128, block=16, batch=2),
    dict(hidden=512, n_q_heads=8, n_kv_heads=1, head_dim=64, block=16, batch=3),
    dict(hidden=256, n_q_heads=2, n_kv_heads=1, head_dim=128, block=16, batch=2, conv_width=3),
])
def test_draft_block_e4m3_cache_parity_small(kw):
    wl = tiny_workload("fp8draft", wid=920 + kw["hidden"] + kw["batch"] + kw["block"], mlp=512,
                       vocab=2048, n_layers=2, n_taps=3, ctx_len_range=(1, 300), **kw)
    check_fp8_step(wl)


def test_draft_block_e4m3_cache_long_context_many_splits():
    wl = tiny_workload("fp8long", wid=930, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=128,
                       mlp=256, vocab=1024, block=16, batch=2, ctx_len_range=(3000, 5000))
    check_fp8_step(wl)


def test_draft_block_e4m3_cache_rejected_where_unsupported(monkeypatch):
    """E4M3 caches run on the tcgen05 attention only: a drafter created on
    the mma.sync kernel refuses them (unsupported), before any launch."""
    from block_diffusion_speculative_fuse_gb300.session import DraftStep
    monkeypatch.setenv("DFLASH_ATTN_TC", "0")
    wl = tiny_workload("fp8no", wid=935, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
                       mlp=256, vocab=1024, block=8, batch=1, ctx_len_range=(20, 40))
    st = DraftStep(wl, kv_dtype="e4m3")
    B = B_()
    with pytest.raises(B.DflashError) as e:
        st.draft_block()
    assert e.value.code == -2


def test_dflash2_b16_e4m3_cache_sampled_requests():
    """DFlash-2-shaped drafter (8 layers, H=2048, width-3 conv), batch 16,
    16384-token contexts, with an E4M3 context cache, in a CUDA graph:
    requests 0 and 15 against the oracle."""
    check_fp8_step(W.get_workload("dflash2_b16"), requests=[0, 15], graph=True)
