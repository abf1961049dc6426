"""dflash_ctx_fuse_noalloc: the context fuse for callers that cannot allocate
device memory (its scratch is a fixed array inside the library).  Its output
must match dflash_ctx_fuse with a caller workspace, call after call.

Kept in a file that pytest collects last, so a run that stops at the first
failure has run every other test first."""
import numpy as np
import pytest
import torch

import workload as W
from workload.shapes import tiny_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_diffusion_speculative_fuse_gb300 import _build, binding
    _build.build()
    binding.load()


def rel_rows(a, b):
    return float(np.max(np.linalg.norm(a - b, axis=-1) / np.linalg.norm(b, axis=-1)))


@pytest.mark.parametrize("T,H,k", [(16, 512, 3), (37, 256, 5)])
def test_noalloc_fuse_matches_workspace_fuse_twice(T, H, k):
    from block_diffusion_speculative_fuse_gb300 import binding as B
    from block_diffusion_speculative_fuse_gb300.device import DeviceModel, to_device_u16
    wl = tiny_workload("noalloc", wid=880 + T, hidden=H, n_q_heads=H // 64,
                       n_kv_heads=H // 128, head_dim=64, mlp=256, vocab=256, n_taps=k)
    d = wl.draft
    m = DeviceModel(d, W.draft_weights(d, wl.wid), W.shared_weights(d, wl.wid), draft=True)
    ref = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    ws = m.workspace(d.block, T, 1, 16)
    taps1 = to_device_u16(W.taps_bf16(T, d, wl.wid))
    taps2 = to_device_u16(W.taps_bf16(T, d, wl.wid, sub=1))
    for taps in (taps1, taps2):
        B.dflash_ctx_fuse(m.handle, taps, T, ref, ws)
        out = torch.full((T, H), 7.0, dtype=torch.bfloat16, device="cuda")
        B.dflash_ctx_fuse_noalloc(m.handle, taps, T, out)
        torch.cuda.synchronize()
        a, b = out.float().cpu().numpy(), ref.float().cpu().numpy()
        assert rel_rows(a, b) < 8e-3
        assert np.array_equal(a, b)  # same kernels, same order: identical bits


def test_noalloc_rejects_oversize():
    from block_diffusion_speculative_fuse_gb300 import binding as B
    from block_diffusion_speculative_fuse_gb300.device import DeviceModel
    wl = tiny_workload("noalloc_big", wid=899, hidden=512, n_q_heads=8, n_kv_heads=4,
                       head_dim=64, mlp=256, vocab=256, n_taps=2)
    d = wl.draft
    m = DeviceModel(d, W.draft_weights(d, wl.wid), W.shared_weights(d, wl.wid), draft=True)
    T = 4096  # 4096 rows x 512 x 4 B = 8 MiB of fp32 rows > the 4 MiB array
    taps = torch.zeros((T, d.n_taps * d.hidden), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((T, d.hidden), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.DflashError) as e:
        B.dflash_ctx_fuse_noalloc(m.handle, taps, T, out)
    assert e.value.code == -3


def test_noalloc_capacity_edge():
    """The largest T that fits the 4 MiB array works and matches the workspace
    fuse; one row more is rejected before anything runs, and the array still
    gives correct results afterwards."""
    from block_diffusion_speculative_fuse_gb300 import binding as B
    from block_diffusion_speculative_fuse_gb300.device import DeviceModel, to_device_u16
    H = 512
    wl = tiny_workload("noalloc_edge", wid=897, hidden=H, n_q_heads=8, n_kv_heads=4,
                       head_dim=64, mlp=256, vocab=256, n_taps=2)
    d = wl.draft
    m = DeviceModel(d, W.draft_weights(d, wl.wid), W.shared_weights(d, wl.wid), draft=True)
    t_max = ((4 << 20) - (64 << 10)) // (H * 4)   # 2016 rows
    taps = to_device_u16(W.taps_bf16(t_max + 1, d, wl.wid))
    ref = torch.zeros((t_max, H), dtype=torch.bfloat16, device="cuda")
    ws = m.workspace(d.block, t_max, 1, 16)
    B.dflash_ctx_fuse(m.handle, taps, t_max, ref, ws)
    out = torch.zeros((t_max + 1, H), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.DflashError) as e:
        B.dflash_ctx_fuse_noalloc(m.handle, taps, t_max + 1, out)
    assert e.value.code == -3
    B.dflash_ctx_fuse_noalloc(m.handle, taps, t_max, out)
    torch.cuda.synchronize()
    assert np.array_equal(out[:t_max].float().cpu().numpy(), ref.float().cpu().numpy())
    assert not out[t_max].float().abs().sum().item()  # the row past T is untouched
