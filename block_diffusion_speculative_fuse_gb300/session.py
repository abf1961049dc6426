"""One draft step of a synthetic workload, resident on the device.

A step is: fuse the new context rows' tapped hidden states (dflash_ctx_fuse),
draft the block while appending those rows to the paged draft cache in the
same weight pass (dflash_draft_block with pending rows), produce the stand-in
target tokens (dflash_synth_target) and verify greedily
(dflash_verify_greedy).  The step reads its inputs and writes its outputs in
separate buffers, so it can be replayed (and captured in a CUDA graph)
without changing the work it does.
"""
import numpy as np
import torch

import workload as W

from . import binding as B
from .device import DeviceModel, PagedKV, i32, to_device_u16


class DraftStep:
    def __init__(self, wl, device="cuda", keep_host=False, model=None, weights=None,
                 shared=None, kv_dtype="bf16"):
        self.wl = wl
        d = wl.draft
        self.shape = d
        self.device = device
        self.batch = b = wl.batch
        self.B = d.block
        wid = wl.wid
        if model is None:
            weights = weights if weights is not None else W.draft_weights(d, wid)
            shared = shared if shared is not None else W.shared_weights(d, wid)
            model = DeviceModel(d, weights, shared, draft=True, device=device)
        self.model = model
        self.host = {"weights": weights, "shared": shared} if keep_host else {}

        self.ctx_before = W.ctx_lengths(wl)                 # C_b (already cached)
        self.new_rows = W.new_row_counts(wl)                # T_b appended this step
        self.anchor_pos_np = (self.ctx_before + self.new_rows).astype(np.int32)
        self.T = int(self.new_rows.sum())
        table, n_pages = W.page_table(self.anchor_pos_np, wl.page_size, wid,
                                      shuffle=wl.shuffle_pages)
        self.kv = PagedKV(d, table, n_pages, wl.page_size, device)
        ctx_k, ctx_v = {}, {}
        for l in range(d.n_layers):
            for r in range(b):
                n = int(self.ctx_before[r])
                if n == 0:
                    continue
                k = W.context_kv_bf16(d, wid, l, r, n, "k")
                v = W.context_kv_bf16(d, wid, l, r, n, "v")
                self.kv.fill_logical(l, r, k, v)
                if keep_host:
                    ctx_k[(l, r)] = k
                    ctx_v[(l, r)] = v
        if kv_dtype == "e4m3":
            # the synthetic context is laid out in bf16, then converted on the device
            self.kv = self.kv.quantized(model)
        elif kv_dtype != "bf16":
            raise ValueError(f"unknown cache dtype {kv_dtype!r}")
        taps = W.taps_bf16(self.T, d, wid)
        req = np.repeat(np.arange(b, dtype=np.int32), self.new_rows)
        pos = np.concatenate([np.arange(c, c + t, dtype=np.int32)
                              for c, t in zip(self.ctx_before, self.new_rows)])
        anchor = W.uniform_tokens(b, d.vocab, wid, W.TENSOR_IDS["anchor"])
        p = W.agreement_probs(wl)
        thr = np.array([W.agree_threshold(x) for x in p], dtype=np.uint64)
        if keep_host:
            self.host.update(ctx_k=ctx_k, ctx_v=ctx_v, taps=taps, req=req, pos=pos,
                             anchor=anchor, p=p)

        dev = device
        self.taps = to_device_u16(taps, dev)
        self.pending_req = i32(req, dev)
        self.pending_pos = i32(pos, dev)
        self.anchor = i32(anchor, dev)
        self.anchor_pos = i32(self.anchor_pos_np, dev)
        self.threshold = torch.from_numpy(thr.view(np.int64)).to(dev)
        self.synth_seed = int(W.rng_for(wid, W.TENSOR_IDS["synth_seed"]).integers(0, 2**62))
        self.step_counter = torch.zeros(1, dtype=torch.int64, device=dev)
        H = d.hidden
        self.ctx = torch.empty((max(1, self.T), H), dtype=torch.bfloat16, device=dev)
        self.draft = torch.zeros((b, max(1, self.B - 1)), dtype=torch.int32, device=dev)
        self.target = torch.zeros((b, self.B), dtype=torch.int32, device=dev)
        self.out_tokens = torch.zeros((b, self.B), dtype=torch.int32, device=dev)
        self.n_accept = torch.zeros(b, dtype=torch.int32, device=dev)
        self.tgt_len_in = self.anchor_pos.clone()
        self.tgt_len_out = torch.zeros(b, dtype=torch.int32, device=dev)
        self.ctx_pending = torch.zeros(b, dtype=torch.int32, device=dev)
        self.anchor_out = torch.zeros(b, dtype=torch.int32, device=dev)
        self.anchor_pos_out = torch.zeros(b, dtype=torch.int32, device=dev)
        max_ctx = int(self.kv.table_np.shape[1] * wl.page_size)
        self.ws = model.workspace(b * self.B, max(1, self.T), b, max_ctx, dev)

    # ------------------------------------------------------------------
    def fuse(self, stream=None):
        if self.T:
            B.dflash_ctx_fuse(self.model.handle, self.taps, self.T, self.ctx, self.ws, stream)

    def draft_block(self, logits=None, hidden=None, stream=None, append=True):
        T = self.T if append else 0
        B.dflash_draft_block(self.model.handle, self.anchor, self.anchor_pos, self.batch,
                             self.kv.struct, self.ctx if T else None,
                             self.pending_req if T else None,
                             self.pending_pos if T else None, T, self.draft, logits, hidden,
                             self.ws, stream)

    def synth_and_verify(self, stream=None, advance=True):
        B.dflash_synth_target(self.draft, self.batch, self.B, self.threshold,
                              self.shape.vocab, self.synth_seed, self.step_counter,
                              1 if advance else 0, self.target, stream)
        B.dflash_verify_greedy(self.draft, self.target, self.batch, self.B, self.out_tokens,
                               self.n_accept, self.tgt_len_in, self.tgt_len_out,
                               self.ctx_pending, self.anchor_out, self.anchor_pos,
                               self.anchor_pos_out, stream)

    def step(self, stream=None):
        """One full step of the hot path (fuse, append + draft, target stand-in, verify)."""
        self.fuse(stream)
        self.draft_block(stream=stream)
        self.synth_and_verify(stream)

    def status(self):
        return B.dflash_get_status(self.ws)
