"""Device-side failure reporting and run-to-run determinism, through the C ABI.

Nothing here faults or hangs the GPU: an out-of-range page id is caught by
the kernels' own checks (the page is skipped or read as zeros and
DFLASH_ERR_CAPACITY is recorded), and the timeout case is a bounded wait of a
few milliseconds on a barrier that nothing arrives at, which records
DFLASH_ERR_TIMEOUT and returns.  After each, the same CUDA context runs a
clean step again.
"""
import pytest
import torch

from workload.shapes import tiny_workload

pytestmark = pytest.mark.gpu

CAPACITY, TIMEOUT = -3, -5
SELFTEST_SITE = 901
PAGE_SITES = {101, 201, 301}  # K/V append epilogue, mma.sync attention, tcgen05 attention


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


def header_ws():
    ws = torch.empty(64 * 1024, dtype=torch.uint8, device="cuda")
    B_().dflash_workspace_init(ws)
    return ws


# ------------------------------------------------------------- bounded wait
def test_bounded_wait_returns_when_the_barrier_completes():
    B = B_()
    ws = header_ws()
    waited = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    B.dflash_selftest_wait(True, 5_000_000, ws, waited)
    assert B.dflash_get_status(ws) == (0, 0)
    assert 0 <= int(waited.item()) < 5_000_000


@pytest.mark.parametrize("limit_ns", [2_000_000, 20_000_000])
def test_bounded_wait_times_out_and_reports_status(limit_ns):
    B = B_()
    ws = header_ws()
    waited = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    B.dflash_selftest_wait(False, limit_ns, ws, waited)
    assert B.dflash_get_status(ws) == (TIMEOUT, SELFTEST_SITE)
    w = int(waited.item())
    # the wait gave up after the limit, not long after it (one polling round)
    assert limit_ns <= w < limit_ns + 50_000_000, w
    # the first error sticks until the workspace is re-initialised
    B.dflash_selftest_wait(True, 1_000_000, ws, waited)
    assert B.dflash_get_status(ws) == (TIMEOUT, SELFTEST_SITE)
    B.dflash_workspace_init(ws)
    assert B.dflash_get_status(ws) == (0, 0)
    # the context is still usable
    B.dflash_selftest_wait(True, 1_000_000, ws, waited)
    assert B.dflash_get_status(ws) == (0, 0)


@pytest.mark.parametrize("limit_ns", [0, -1, 1_000_000_001])
def test_bounded_wait_rejects_limits_out_of_range(limit_ns):
    B = B_()
    ws = header_ws()
    with pytest.raises(B.DflashError) as e:
        B.dflash_selftest_wait(False, limit_ns, ws)
    assert e.value.code == -1
    assert B.dflash_get_status(ws) == (0, 0)


# ------------------------------------------------- page table out of range
def run_draft(st, logits):
    st.fuse()
    st.draft_block(logits=logits)
    torch.cuda.synchronize()
    return st.status()


@pytest.mark.parametrize("tc", ["1", "0"])
def test_bad_page_id_reports_capacity_and_recovers(tc, monkeypatch):
    """A context page id past the pool (and one negative) in the page table:
    the step records DFLASH_ERR_CAPACITY at a page-checking site instead of
    reading or writing outside the pool; with the table repaired and the
    status cleared, the next step gives the clean step's logits bit for bit."""
    from block_diffusion_speculative_fuse_gb300.session import DraftStep
    monkeypatch.setenv("DFLASH_ATTN_TC", tc)  # read at model creation
    wl = tiny_workload("badpage", wid=810, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=128,
                       mlp=256, vocab=1024, block=16, batch=3, ctx_len_range=(20, 600))
    st = DraftStep(wl)
    rows = st.batch * st.B
    clean = torch.zeros((rows, wl.draft.vocab), dtype=torch.float32, device="cuda")
    assert run_draft(st, clean) == (0, 0)
    good = st.kv.table.clone()
    st.kv.table[0, 0] = st.kv.n_pages
    st.kv.table[2, 0] = -7
    bad = torch.zeros_like(clean)
    status, site = run_draft(st, bad)
    assert status == CAPACITY and site in PAGE_SITES, (status, site)
    st.kv.table.copy_(good)
    B_().dflash_workspace_init(st.ws)
    again = torch.zeros_like(clean)
    assert run_draft(st, again) == (0, 0)
    assert torch.equal(again, clean)


def test_bad_request_index_reports_capacity_and_recovers():
    """Pending context rows whose request index lies outside the page table
    (one past its last row, and a negative one): the K/V routing records
    DFLASH_ERR_CAPACITY at site 102 and skips those rows instead of reading
    the page table out of bounds.  A batch larger than the table is refused
    before any launch.  With the indices repaired and the status cleared, the
    next step gives the clean step's logits bit for bit."""
    from block_diffusion_speculative_fuse_gb300.session import DraftStep
    wl = tiny_workload("badreq", wid=814, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=128,
                       mlp=256, vocab=1024, block=16, batch=3, ctx_len_range=(20, 300))
    st = DraftStep(wl)
    rows = st.batch * st.B
    clean = torch.zeros((rows, wl.draft.vocab), dtype=torch.float32, device="cuda")
    assert run_draft(st, clean) == (0, 0)
    good = st.pending_req.clone()
    st.pending_req[0] = st.kv.table.shape[0]
    st.pending_req[-1] = -2
    bad = torch.zeros_like(clean)
    assert run_draft(st, bad) == (CAPACITY, 102)
    st.pending_req.copy_(good)
    B_().dflash_workspace_init(st.ws)
    # more requests than the page table has rows: rejected on the host
    B = B_()
    big = torch.zeros(st.batch + 1, dtype=torch.int32, device="cuda")
    draft = torch.zeros((st.batch + 1, st.B - 1), dtype=torch.int32, device="cuda")
    with pytest.raises(B.DflashError) as e:
        B.dflash_draft_block(st.model.handle, big, big, st.batch + 1, st.kv.struct, None, None,
                             None, 0, draft, None, None, st.ws)
    assert e.value.code == CAPACITY
    assert B.dflash_get_status(st.ws) == (0, 0)
    again = torch.zeros_like(clean)
    assert run_draft(st, again) == (0, 0)
    assert torch.equal(again, clean)


# -------------------------------------------------------------- determinism
@pytest.mark.parametrize("kw", [
    # long contexts: several key splits per request, merged in split order
    dict(wid=811, hidden=512, n_q_heads=8, n_kv_heads=2, head_dim=64, block=16, batch=4,
         ctx_len_range=(2000, 5000)),
    # 256 block rows, DFlash-2 block convolution
    dict(wid=812, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=128, block=16, batch=16,
         conv_width=3, ctx_len_range=(16, 700)),
])
def test_same_step_twice_is_bitwise_identical(kw):
    """Split-K partials and attention splits are combined in a fixed order,
    so the same inputs give the same logits, hidden states and tokens."""
    from block_diffusion_speculative_fuse_gb300.session import DraftStep
    wl = tiny_workload("determinism", mlp=512, vocab=2048, n_layers=2, **kw)
    st = DraftStep(wl)
    rows = st.batch * st.B
    outs = []
    for _ in range(2):
        lg = torch.zeros((rows, wl.draft.vocab), dtype=torch.float32, device="cuda")
        hd = torch.zeros((rows, wl.draft.hidden), dtype=torch.float32, device="cuda")
        st.fuse()
        st.draft_block(logits=lg, hidden=hd)
        st.synth_and_verify(advance=False)
        torch.cuda.synchronize()
        assert st.status() == (0, 0)
        outs.append((lg, hd, st.draft.clone(), st.out_tokens.clone(), st.n_accept.clone()))
    for a, b in zip(*outs):
        assert torch.equal(a, b)
