"""Sampling-mode verify (temperature T > 0) and draft sampling on the GPU
against the oracle (oracle/sampling.py), at the Qwen3-8B drafter's vocabulary
(151936) and block 16, batch 1 and 32.

The reading of the rule is the standard lossless speculative-sampling rule per
block position ("DFlash: how block diffusion boosts NVIDIA Blackwell
throughput", section "Real-world integration": sampling-mode results;
introduction: lossless).  The GPU forms the exponentials in fp32 and every sum
in fp64, the oracle everything in fp64, so a decision may differ only when
its uniform lies within a relative EPS of the decision's boundary: such cases
are recognised from the oracle's own fp64 quantities, counted and reported;
any other difference fails.

Coverage by construction: requests whose target logits equal the drafter's
(q = p: every draft is accepted and the bonus is drawn from p_B), requests
with unrelated target logits (early rejections and residual draws), and
requests in between.
"""
import numpy as np
import pytest
import torch

from oracle import sampling as S

pytestmark = pytest.mark.gpu

V, B = 151936, 16
EPS = 1e-5


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


def logits_case(batch, seed):
    """Drafter logits [batch][B][V] (row 0 unused) and target logits
    [batch][B][V]; request r mixes the target as y = z + c_r * noise."""
    g = np.random.default_rng(seed)
    z = (g.standard_normal((batch, B, V)) * 1.3).astype(np.float32)
    noise = (g.standard_normal((batch, B, V)) * 1.3).astype(np.float32)
    c = np.linspace(0.0, 3.0, batch) if batch > 1 else np.array([0.4])
    y = np.empty_like(z)
    y[:, :B - 1] = z[:, 1:] + c[:, None, None] * noise[:, :B - 1]   # p_j vs q_j for j < B
    y[:, B - 1] = noise[:, B - 1] + z[:, B - 1]
    return z, y, g


def valid_draw(weights, a, k, eps=EPS):
    """k is an inverse-CDF draw of a from the weights, up to eps*S."""
    c = np.cumsum(np.asarray(weights, dtype=np.float64))
    s = c[-1]
    lo = c[k - 1] if k > 0 else 0.0
    return lo - eps * s <= a * s < c[k] + eps * s


def run_sample_rows(z, T, a):
    B_mod = B_()
    batch = z.shape[0]
    zt = torch.from_numpy(z).cuda()
    at = torch.from_numpy(a).cuda()
    out = torch.zeros((batch, B - 1), dtype=torch.int32, device="cuda")
    ws = torch.zeros(64 * 1024 + 16 * batch * B + 256, dtype=torch.uint8, device="cuda")
    B_mod.dflash_workspace_init(ws)
    B_mod.dflash_sample_rows(zt, batch, B, 1, V, T, at, out, ws)
    torch.cuda.synchronize()
    assert B_mod.dflash_get_status(ws) == (0, 0)
    return out.cpu().numpy()


@pytest.mark.parametrize("batch,T,seed", [(1, 0.7, 11), (32, 1.0, 12), (32, 0.7, 13)])
def test_draft_sampling_and_verify_match_oracle(batch, T, seed):
    B_mod = B_()
    z, y, g = logits_case(batch, seed)
    if batch > 1:
        y[0, :B - 1] = z[0, 1:]            # q = p: all drafts accepted, bonus draw
    a = g.random((batch, B - 1))
    u = g.random((batch, B - 1))
    w = g.random((batch, B))

    # ---- draft sampling: d_i ~ q_i
    d_gpu = run_sample_rows(z, T, a)
    d_ref = S.draft_sample(z[:, 1:], T, a)
    q = S.softmax_t(z[:, 1:], T)
    near = 0
    for r, i in zip(*np.nonzero(d_gpu != d_ref)):
        assert valid_draw(q[r, i], a[r, i], d_gpu[r, i]), (r, i, d_gpu[r, i], d_ref[r, i])
        near += 1
    assert near <= max(1, d_gpu.size // 100)

    # ---- verify at temperature T, on the GPU's drafts
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    out = torch.zeros((batch, B), dtype=torch.int32, device="cuda")
    n = torch.zeros(batch, dtype=torch.int32, device="cuda")
    anchor = torch.zeros(batch, dtype=torch.int32, device="cuda")
    ws = torch.zeros(B_mod.dflash_sampling_workspace_bytes(batch, B), dtype=torch.uint8,
                     device="cuda")
    B_mod.dflash_workspace_init(ws)
    B_mod.dflash_verify_sampling(dev(d_gpu.astype(np.int32)), dev(z), dev(y), batch, B, V, T,
                                 dev(u), dev(w), out, n, None, None, None, anchor, None, None, ws)
    torch.cuda.synchronize()
    assert B_mod.dflash_get_status(ws) == (0, 0)
    n_gpu, out_gpu = n.cpu().numpy(), out.cpu().numpy()
    n_ref, out_ref = S.verify_sampling(d_gpu, z[:, 1:], y, T, u, w)
    p = S.softmax_t(y, T)
    near_v = 0
    for r in range(batch):
        assert 0 <= n_gpu[r] <= B - 1
        assert np.all(out_gpu[r, n_gpu[r] + 1:] == -1)
        assert anchor.cpu().numpy()[r] == out_gpu[r, n_gpu[r]]
        if n_gpu[r] != n_ref[r]:
            # the first differing decision is an accept test within EPS
            i = min(n_gpu[r], n_ref[r])
            dd = d_gpu[r, i]
            lhs, rhs = u[r, i] * q[r, i, dd], p[r, i, dd]
            assert abs(lhs - rhs) <= EPS * max(lhs, rhs), (r, i, lhs, rhs)
            near_v += 1
            continue
        k = n_ref[r]
        assert np.array_equal(out_gpu[r, :k], out_ref[r, :k])
        if out_gpu[r, k] != out_ref[r, k]:
            wts = np.maximum(p[r, k] - q[r, k], 0.0) if k < B - 1 else p[r, B - 1]
            assert valid_draw(wts, w[r, k], out_gpu[r, k]), (r, k)
            near_v += 1
    assert near_v <= max(1, batch // 16)
    if batch > 1:
        assert n_gpu[0] == B - 1                       # q = p accepts every draft
        assert (n_gpu < B - 1).any()                   # and some requests reject
    print(f"batch {batch} T {T}: n = {n_gpu.tolist()}, near-boundary cases: "
          f"draft {near}, verify {near_v}")


def test_sampling_rejects_bad_arguments():
    B_mod = B_()
    ws = torch.zeros(B_mod.dflash_sampling_workspace_bytes(2, B), dtype=torch.uint8, device="cuda")
    x = torch.zeros((2, B, 256), dtype=torch.float32, device="cuda")
    d = torch.zeros((2, B - 1), dtype=torch.int32, device="cuda")
    u = torch.zeros((2, B), dtype=torch.float64, device="cuda")
    out = torch.zeros((2, B), dtype=torch.int32, device="cuda")
    for T in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(B_mod.DflashError) as e:
            B_mod.dflash_verify_sampling(d, x, x, 2, B, 256, T, u, u, out, None, None, None, None,
                                         None, None, None, ws)
        assert e.value.code == -1
    small = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(B_mod.DflashError) as e:
        B_mod.dflash_verify_sampling(d, x, x, 2, B, 256, 1.0, u, u, out, None, None, None, None,
                                     None, None, None, small)
    assert e.value.code == -3


def test_sampling_small_temperature_is_greedy():
    """T -> 0: draft sampling gives the drafter's argmax and the verify gives
    the greedy verify's n and tokens (on a small vocabulary)."""
    B_mod = B_()
    g = np.random.default_rng(5)
    batch, Vs, T = 8, 512, 1e-3
    z = g.standard_normal((batch, B, Vs)).astype(np.float32)
    y = g.standard_normal((batch, B, Vs)).astype(np.float32)
    dz = np.argmax(z[:, 1:], -1)
    for r in range(batch):
        for i in range(min(r, B - 1)):          # request r agrees on its first r positions
            y[r, i, dz[r, i]] = 10.0
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    a = g.random((batch, B - 1))
    out = torch.zeros((batch, B - 1), dtype=torch.int32, device="cuda")
    ws = torch.zeros(B_mod.dflash_sampling_workspace_bytes(batch, B), dtype=torch.uint8,
                     device="cuda")
    B_mod.dflash_workspace_init(ws)
    B_mod.dflash_sample_rows(dev(z), batch, B, 1, Vs, T, dev(a), out, ws)
    d = out.cpu().numpy()
    assert np.array_equal(d, dz)
    o = torch.zeros((batch, B), dtype=torch.int32, device="cuda")
    n = torch.zeros(batch, dtype=torch.int32, device="cuda")
    B_mod.dflash_verify_sampling(out, dev(z), dev(y), batch, B, Vs, T, dev(g.random((batch, B - 1))),
                                 dev(g.random((batch, B))), o, n, None, None, None, None, None,
                                 None, ws)
    torch.cuda.synchronize()
    import oracle as O
    tgt = np.argmax(y, -1)
    for r in range(batch):
        ng, em = O.verify_greedy(d[r], tgt[r])
        assert n.cpu().numpy()[r] == ng
        assert list(o.cpu().numpy()[r, :ng + 1]) == em
