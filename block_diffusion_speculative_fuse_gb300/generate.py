"""Greedy speculative decoding and plain autoregressive decoding on the GPU,
driven from the host through the C ABI (the end-to-end loop of the method).

Speculative iteration (lossless at temperature 0):
  1. dflash_draft_block drafts B-1 tokens from the anchor at position L; the
     pending context rows of the previous verify (anchor + accepted drafts)
     are appended to the draft cache in the same weight pass;
  2. dflash_target_forward runs the target causally over [anchor, drafts] at
     L..L+B-1, writing its K/V and tapping hidden states;
  3. dflash_verify_greedy accepts n, emits t_1..t_{n+1}, advances lengths;
  4. dflash_ctx_fuse turns the tapped states of the B rows into context rows;
     only rows 0..n become pending rows for the next draft (the verify
     kernel writes their positions; the others get -1 and are skipped).
The loop state (anchors, positions, pending rows, emitted counts, emitted
tokens) stays on the device; each iteration reads back only the emitted
count per request (batch int32) for the stop test.  The target cache needs
no explicit rollback: positions past L+n are rewritten before any row at or
after them attends to them.  Fusing only the accepted rows would not save
weight bytes: the fuse GEMM streams its weights once for any row count up to
a few hundred.
"""
import numpy as np
import torch

from . import binding as B
from .device import DeviceModel, PagedKV, i32


def _sequential_table(batch, positions, page):
    pages_per = (positions + page - 1) // page
    table = np.arange(batch * pages_per, dtype=np.int32).reshape(batch, pages_per)
    return table, batch * pages_per


class TargetRunner:
    def __init__(self, target: DeviceModel, batch: int, max_len: int, max_rows_per_req: int,
                 tap_layers=(), device="cuda"):
        self.m = target
        self.shape = target.shape
        self.batch = batch
        table, npg = _sequential_table(batch, max_len, 16)
        self.kv = PagedKV(self.shape, table, npg, 16, device)
        # host array: the library reads the layer list on the host
        self.taps_ids = torch.tensor(list(tap_layers), dtype=torch.int32) if len(tap_layers) else None
        self.n_taps = len(tap_layers)
        self.max_len = max_len
        self.device = device
        self._ws = {}

    def workspace(self, n):
        """Workspace for calls with n rows per request (allocated once per n)."""
        if n not in self._ws:
            self._ws[n] = self.m.workspace(self.batch * n, 0, self.batch, self.max_len,
                                           self.device)
        return self._ws[n]

    def forward(self, tokens: torch.Tensor, pos0: torch.Tensor, n: int, want_taps=False,
                logits=None):
        b = self.batch
        out = torch.empty((b, n), dtype=torch.int32, device=self.device)
        taps = None
        if want_taps and self.n_taps:
            taps = torch.empty((b * n, self.n_taps * self.shape.hidden), dtype=torch.bfloat16,
                               device=self.device)
        B.dflash_target_forward(self.m.handle, tokens, pos0, b, n, self.kv.struct,
                                self.taps_ids if taps is not None else None,
                                self.n_taps if taps is not None else 0, taps, out, logits,
                                self.workspace(n))
        return out, taps


def ar_generate(runner: TargetRunner, prompts: np.ndarray, n_tokens: int):
    """Greedy autoregressive decoding, one target forward per token."""
    b, P = prompts.shape
    dev = runner.device
    out, _ = runner.forward(i32(prompts, dev), i32(np.zeros(b), dev), P)
    tok = out[:, P - 1:P].contiguous()
    res = [tok]
    pos = torch.full((b,), P, dtype=torch.int32, device=dev)
    for _ in range(n_tokens - 1):
        tok, _ = runner.forward(tok, pos, 1)
        res.append(tok)
        pos += 1
    return torch.cat(res, dim=1).cpu().numpy()


class SpecDecoder:
    def __init__(self, target: DeviceModel, drafter: DeviceModel, tap_layers, batch: int,
                 max_len: int, device="cuda"):
        d = drafter.shape
        self.d = d
        self.B = d.block
        self.batch = batch
        self.drafter = drafter
        self.target = TargetRunner(target, batch, max_len + d.block + 1,
                                   max(d.block, 1), tap_layers, device)
        table, npg = _sequential_table(batch, max_len + d.block + 1, 16)
        self.dkv = PagedKV(d, table, npg, 16, device)
        self.max_len = max_len
        self.device = device
        self.ws_d = drafter.workspace(batch * d.block, max(batch * d.block, batch * max_len),
                                      batch, max_len + d.block + 1, device)
        self.stats = []

    def generate(self, prompts: np.ndarray, n_tokens: int):
        b, P = prompts.shape
        dev = self.device
        d = self.d
        Bk = self.B
        # prefill: target over the prompt, its taps become context rows 0..P-1
        out, taps = self.target.forward(i32(prompts, dev), i32(np.zeros(b), dev), P,
                                        want_taps=True)
        anchor = out[:, P - 1].contiguous()
        ctx = torch.empty((b * P, d.hidden), dtype=torch.bfloat16, device=dev)
        B.dflash_ctx_fuse(self.drafter.handle, taps, b * P, ctx, self.ws_d)
        req = i32(np.repeat(np.arange(b), P), dev)
        pos = i32(np.tile(np.arange(P), b), dev)
        B.dflash_kv_append(self.drafter.handle, ctx, req, pos, b * P, self.dkv.struct, self.ws_d)
        first = anchor.clone()
        max_iters = n_tokens  # at least one token per request per iteration
        history = torch.full((max_iters, b, Bk), -1, dtype=torch.int32, device=dev)
        draft = torch.zeros((b, max(1, Bk - 1)), dtype=torch.int32, device=dev)
        n_acc = torch.zeros(b, dtype=torch.int32, device=dev)
        emitted = torch.ones(b, dtype=torch.int32, device=dev)  # the prefill's token
        anchor_pos = torch.full((b,), P, dtype=torch.int32, device=dev)
        anchor_pos_next = torch.zeros(b, dtype=torch.int32, device=dev)
        anchor_next = torch.zeros(b, dtype=torch.int32, device=dev)
        pend_ctx = torch.empty((b * Bk, d.hidden), dtype=torch.bfloat16, device=dev)
        pend_req = i32(np.repeat(np.arange(b), Bk), dev)
        pend_pos = torch.full((b, Bk), -1, dtype=torch.int32, device=dev)
        rows = torch.empty((b, Bk), dtype=torch.int32, device=dev)
        counts = torch.empty(b, dtype=torch.int32, device="cpu").pin_memory()
        T = 0
        it = 0
        while it < max_iters:
            B.dflash_draft_block(self.drafter.handle, anchor, anchor_pos, b, self.dkv.struct,
                                 pend_ctx if T else None, pend_req if T else None,
                                 pend_pos if T else None, T, draft, None, None, self.ws_d)
            rows[:, 0] = anchor
            if Bk > 1:
                rows[:, 1:] = draft[:, :Bk - 1]
            t, taps = self.target.forward(rows, anchor_pos, Bk, want_taps=True)
            B.dflash_verify_greedy(draft if Bk > 1 else None, t, b, Bk, history[it], n_acc,
                                   emitted, emitted, None, anchor_next, anchor_pos,
                                   anchor_pos_next, ctx_pos=pend_pos)
            B.dflash_ctx_fuse(self.drafter.handle, taps, b * Bk, pend_ctx, self.ws_d)
            T = b * Bk
            anchor, anchor_next = anchor_next, anchor
            anchor_pos, anchor_pos_next = anchor_pos_next, anchor_pos
            it += 1
            counts.copy_(emitted)  # the stop test: one D2H of batch int32
            if int(counts.min()) >= n_tokens:
                break
        hist = history[:it].cpu().numpy()
        first = first.cpu().numpy()
        result = []
        for r in range(b):
            em = hist[:, r, :]
            toks = [int(first[r])] + [int(x) for x in em[em >= 0]]
            self.stats.extend(int((row >= 0).sum()) - 1 for row in em)
            result.append(toks[:n_tokens])
        return np.array(result, dtype=np.int32)
