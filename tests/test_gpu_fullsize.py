"""Parity at the measured sizes, in the launch configuration bench.py times
(the step captured in a CUDA graph and replayed).

qwen3_8b_b1: the whole step against the oracle (every logit of the block,
the final hidden rows, the drafts, the verify outputs).
qwen3_8b_b32_paged and dflash2_b16: sampled requests (the first, the last,
and one from the middle of the batch: for the ragged batch the request with
the longest context, whose keys span the most splits) against the oracle,
which computes a request's block independently.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workload as W

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


def rel_rows(a, b):
    return float(np.max(np.linalg.norm(a - b, axis=-1) / np.linalg.norm(b, axis=-1)))


def run_graph_step(st, logits, hidden):
    """fuse + draft (logits/hidden dumped) captured in a graph, replayed twice."""
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        st.fuse(stream)
        st.draft_block(logits=logits, hidden=hidden, stream=stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        st.fuse(stream)
        st.draft_block(logits=logits, hidden=hidden, stream=stream)
        st.synth_and_verify(stream)
    with torch.cuda.stream(stream):
        g.replay()
        g.replay()
    torch.cuda.synchronize()


def oracle_request(st, d, dws, c_rows, r):
    h = st.host
    offs = np.concatenate([[0], np.cumsum(st.new_rows)])
    C, T = int(st.ctx_before[r]), int(st.new_rows[r])
    ks, vs = [], []
    for l in range(d.n_layers):
        kn, vn = O.ctx_kv(d, dws, l, c_rows[offs[r]:offs[r] + T], np.arange(C, C + T))
        ks.append(np.concatenate([O.bf16_to_f64(h["ctx_k"][(l, r)]), kn]) if C else kn)
        vs.append(np.concatenate([O.bf16_to_f64(h["ctx_v"][(l, r)]), vn]) if C else vn)
    return O.draft_block(d, dws, int(h["anchor"][r]), C + T, ks, vs, return_hidden=True)


def check_requests(name, requests, longest=False):
    from block_diffusion_speculative_fuse_gb300.session import DraftStep
    wl = W.get_workload(name)
    d = wl.draft
    st = DraftStep(wl, keep_host=True)
    if longest:
        requests = sorted(set(requests) | {int(np.argmax(st.anchor_pos_np))})
    rows = st.batch * st.B
    logits = torch.zeros((rows, d.vocab), dtype=torch.float32, device="cuda")
    hidden = torch.zeros((rows, d.hidden), dtype=torch.float32, device="cuda")
    run_graph_step(st, logits, hidden)
    assert st.status()[0] == 0
    h = st.host
    dws = O.LayerStack(d, h["weights"], h["shared"])
    taps = O.bf16_to_f64(h["taps"])
    # context feature rows of the sampled requests only
    offs = np.concatenate([[0], np.cumsum(st.new_rows)])
    c_rows = np.zeros((taps.shape[0], d.hidden))
    for r in requests:
        c_rows[offs[r]:offs[r + 1]] = O.ctx_fuse(d, dws, taps[offs[r]:offs[r + 1]])
    drafts = st.draft.cpu().numpy()
    for r in requests:
        dr, lref, href = oracle_request(st, d, dws, c_rows, r)
        sl = slice(r * st.B, (r + 1) * st.B)
        lg = logits[sl].cpu().numpy()
        hd = hidden[sl].cpu().numpy()
        err = float(np.abs(lg - lref).max())
        assert err <= LOGIT_TOL, f"{name} request {r}: max |dlogit| {err}"
        assert rel_rows(hd, href) <= HIDDEN_RTOL
        top = np.sort(lref[1:], axis=-1)
        sure = (top[:, -1] - top[:, -2]) > GAP
        assert np.array_equal(drafts[r][sure], dr[sure])
    ver = O.verify_batch(drafts, st.target.cpu().numpy(), st.tgt_len_in.cpu().numpy(),
                         st.anchor_pos.cpu().numpy())
    assert np.array_equal(ver["out_tokens"], st.out_tokens.cpu().numpy())
    assert np.array_equal(ver["n_accept"], st.n_accept.cpu().numpy())
    assert np.array_equal(ver["anchor_pos"], st.anchor_pos_out.cpu().numpy())
    # the exact step the benchmark replays (no logits/hidden dump) drafts the
    # same tokens bit for bit
    st.draft.zero_()
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        st.step(stream)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    assert st.status()[0] == 0
    assert np.array_equal(st.draft.cpu().numpy(), drafts)


def test_qwen3_8b_b1_full_step():
    check_requests("qwen3_8b_b1", [0])


def test_qwen3_8b_b32_paged_sampled_requests():
    check_requests("qwen3_8b_b32_paged", [0, 31], longest=True)


def test_dflash2_b16_sampled_requests():
    check_requests("dflash2_b16", [0, 7, 15])
