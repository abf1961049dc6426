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
     only rows 0..n become pending rows for the next draft (others get
     position -1 and are skipped).
The target cache needs no explicit rollback: positions past L+n are
rewritten before any row at or after them attends to them.
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
        L = np.full(b, P, dtype=np.int64)
        result = [[int(t)] for t in anchor.cpu().numpy()]
        draft = torch.zeros((b, max(1, Bk - 1)), dtype=torch.int32, device=dev)
        out_tok = torch.zeros((b, Bk), dtype=torch.int32, device=dev)
        n_acc = torch.zeros(b, dtype=torch.int32, device=dev)
        anchor_pos = i32(L, dev)
        anchor_pos_out = torch.zeros(b, dtype=torch.int32, device=dev)
        anchor_out = torch.zeros(b, dtype=torch.int32, device=dev)
        pend_ctx = torch.empty((b * Bk, d.hidden), dtype=torch.bfloat16, device=dev)
        pend_req = i32(np.repeat(np.arange(b), Bk), dev)
        T = 0
        pend_pos = None
        while min(len(r) for r in result) < n_tokens:
            B.dflash_draft_block(self.drafter.handle, anchor, anchor_pos, b, self.dkv.struct,
                                 pend_ctx if T else None, pend_req if T else None,
                                 pend_pos if T else None, T, draft, None, None, self.ws_d)
            rows = torch.cat([anchor.view(b, 1), draft[:, :Bk - 1]], dim=1).contiguous()
            t, taps = self.target.forward(rows, anchor_pos, Bk, want_taps=True)
            B.dflash_verify_greedy(draft if Bk > 1 else None, t, b, Bk, out_tok, n_acc, None,
                                   None, None, anchor_out, anchor_pos, anchor_pos_out)
            B.dflash_ctx_fuse(self.drafter.handle, taps, b * Bk, pend_ctx, self.ws_d)
            n_np = n_acc.cpu().numpy()
            toks = out_tok.cpu().numpy()
            self.stats.extend(int(x) for x in n_np)
            pp = np.full((b, Bk), -1, dtype=np.int32)
            for r in range(b):
                k = int(n_np[r]) + 1
                result[r].extend(int(x) for x in toks[r, :k])
                pp[r, :k] = L[r] + np.arange(k)
                L[r] += k
            pend_pos = i32(pp.reshape(-1), dev)
            T = b * Bk
            anchor = anchor_out.clone()
            anchor_pos = anchor_pos_out.clone()
        return np.array([r[:n_tokens] for r in result], dtype=np.int32)
