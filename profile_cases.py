"""Small, self-contained launch cases for profiling single kernels with ncu.

    python profile_cases.py lm_head
    python profile_cases.py step [--config NAME]

lm_head: the shared LM head + argmax of the Qwen3-8B-shaped drafter
(151936 x 4096 bf16 weights, 16 rows), launched a few times, ~1.7 GB on the
device.  step: a few eager draft steps of a workload (default qwen3_8b_b1).
"""
import argparse
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workload as W  # noqa: E402

from block_diffusion_speculative_fuse_gb300 import _build, binding as B  # noqa: E402
from block_diffusion_speculative_fuse_gb300.device import DeviceModel, to_device_u16  # noqa: E402


def lm_head(iters=3, rows=16):
    from dataclasses import replace
    d = replace(W.get_workload("qwen3_8b_b1").draft, n_layers=1, mlp=128, n_taps=1)
    wid = 2
    lm = to_device_u16(W.normal_bf16((d.vocab, d.hidden), 0.02, wid, W.TENSOR_IDS["lm_head"]))
    w = W.draft_weights(d, wid)
    m = DeviceModel(d, w, {"embed": lm, "lm_head": lm}, draft=True)
    x = torch.randn((rows, d.hidden), device="cuda").to(torch.bfloat16)
    out = torch.zeros(rows, dtype=torch.int32, device="cuda")
    ws = m.workspace(rows, 16, 1, 64)
    for _ in range(iters):
        B.dflash_lm_head_argmax(m.handle, x, rows, out, None, ws)
    torch.cuda.synchronize()
    print("lm_head ok", out[:4].tolist())


def step(config="qwen3_8b_b1", iters=3):
    from block_diffusion_speculative_fuse_gb300.session import DraftStep
    st = DraftStep(W.get_workload(config))
    for _ in range(iters):
        st.step()
    torch.cuda.synchronize()
    assert st.status()[0] == 0
    print("step ok", st.n_accept.tolist()[:4])


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["lm_head", "step"])
    ap.add_argument("--config", default="qwen3_8b_b1")
    ap.add_argument("--iters", type=int, default=3)
    a = ap.parse_args()
    _build.build()
    B.load()
    if a.case == "lm_head":
        lm_head(a.iters)
    else:
        step(a.config, a.iters)


if __name__ == "__main__":
    main()
