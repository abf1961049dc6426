"""The opt-in persistent layer-stack kernel (DFLASH_PERSISTENT=1) against the
oracle, the same checks as the per-GEMM path.  The variable is read when a
model is created, so it is set around model creation only."""
import os

import pytest
import torch

from workload.shapes import tiny_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_diffusion_speculative_fuse_gb300 import _build, binding
    _build.build()
    binding.load()


@pytest.fixture()
def persistent_env():
    old = os.environ.get("DFLASH_PERSISTENT")
    os.environ["DFLASH_PERSISTENT"] = "1"
    yield
    if old is None:
        del os.environ["DFLASH_PERSISTENT"]
    else:
        os.environ["DFLASH_PERSISTENT"] = old


@pytest.mark.parametrize("kw", [
    dict(hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, block=8, batch=2, n_layers=2),
    dict(hidden=512, n_q_heads=4, n_kv_heads=1, head_dim=128, block=16, batch=1, n_layers=3),
    dict(hidden=256, n_q_heads=2, n_kv_heads=1, head_dim=128, block=16, batch=1, n_layers=2,
         conv_width=3),
])
def test_persistent_stack_parity(kw, persistent_env):
    from tests.test_gpu_parity import check_draft_step
    wl = tiny_workload("persist", wid=850 + kw["hidden"] + kw["block"], mlp=512, vocab=2048,
                       n_taps=3, ctx_len_range=(30, 400), **kw)
    st, worst = check_draft_step(wl)
    assert st.status()[0] == 0
