"""Small, self-contained launch cases for profiling kernels with ncu.

    python profile_cases.py lm_head [--rows 16]
    python profile_cases.py step [--config NAME] [--kv bf16|e4m3] [--batch N]
    python profile_cases.py target [--iters 2]
    python profile_cases.py sampling

lm_head: the shared LM head + argmax of the Qwen3-8B-shaped drafter
(151936 x 4096 bf16 weights, `rows` rows), launched a few times, ~1.7 GB on
the device.  step: a few eager draft steps of a workload (default
qwen3_8b_b1; --kv e4m3: E4M3 context cache; --batch: fewer requests; --ctx: context
length).  target: block-verify passes of the end-to-end workload's
8-layer H=4096 target (batch 8 x 16 rows, context 1024), ~5 GB.  sampling:
draft sampling and the temperature-1 verify at batch 32, block 16, vocab
151936 (random logits, ~0.7 GB).
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


def step(config="qwen3_8b_b1", iters=3, kv="bf16", batch=None, ctx=None):
    from dataclasses import replace
    from block_diffusion_speculative_fuse_gb300.session import DraftStep
    wl = W.get_workload(config)
    if batch is not None:
        wl = replace(wl, batch=batch)
    if ctx is not None:
        wl = replace(wl, ctx_len=ctx)
    st = DraftStep(wl, kv_dtype=kv)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()  # the bf16 staging of an E4M3 cache
    for _ in range(iters):
        st.step()
    torch.cuda.synchronize()
    assert st.status()[0] == 0
    print("step ok", st.n_accept.tolist()[:4])


def target(iters=2, batch=8, ctx=1024, n=16):
    from block_diffusion_speculative_fuse_gb300.device import i32
    from block_diffusion_speculative_fuse_gb300.generate import TargetRunner
    wl = W.get_workload("e2e_8layer")
    ts = wl.target
    m = DeviceModel(ts, W.target_weights(ts, wl.wid), W.shared_weights(ts, wl.wid), draft=False)
    run = TargetRunner(m, batch, ctx + n + 1, n, wl.tap_layers)
    toks = i32(W.uniform_tokens(batch * n, ts.vocab, wl.wid, 99).reshape(batch, n))
    pos = i32(np.full(batch, ctx))
    for _ in range(iters):
        out, _ = run.forward(toks, pos, n, want_taps=True)
    torch.cuda.synchronize()
    print("target ok", out[0, :4].tolist())


def sampling(iters=2, batch=32, block=16, vocab=151936):
    g = np.random.default_rng(3)
    z = torch.from_numpy((g.standard_normal((batch, block, vocab)) * 1.3).astype(np.float32)).cuda()
    y = torch.from_numpy((g.standard_normal((batch, block, vocab)) * 1.3).astype(np.float32)).cuda()
    a = torch.from_numpy(g.random((batch, block))).cuda()
    d = torch.zeros((batch, block - 1), dtype=torch.int32, device="cuda")
    out = torch.zeros((batch, block), dtype=torch.int32, device="cuda")
    ws = torch.zeros(B.dflash_sampling_workspace_bytes(batch, block), dtype=torch.uint8,
                     device="cuda")
    B.dflash_workspace_init(ws)
    for _ in range(iters):
        B.dflash_sample_rows(z, batch, block, 1, vocab, 1.0, a, d, ws)
        B.dflash_verify_sampling(d, z, y, batch, block, vocab, 1.0, a, a, out, None, None, None,
                                 None, None, None, None, ws)
    torch.cuda.synchronize()
    assert B.dflash_get_status(ws)[0] == 0
    print("sampling ok", out[0, :4].tolist())


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["lm_head", "step", "target", "sampling"])
    ap.add_argument("--config", default="qwen3_8b_b1")
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--rows", type=int, default=16)
    ap.add_argument("--kv", default="bf16", choices=["bf16", "e4m3"])
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--ctx", type=int, default=None, help="context length per request")
    a = ap.parse_args()
    _build.build()
    B.load()
    if a.case == "lm_head":
        lm_head(a.iters, a.rows)
    elif a.case == "target":
        target(a.iters)
    elif a.case == "sampling":
        sampling(a.iters)
    else:
        step(a.config, a.iters, a.kv, a.batch, a.ctx)


if __name__ == "__main__":
    main()
