"""ctypes binding of the C ABI in include/dflash.h.

Argument marshalling only: every function forwards device pointers (taken
from torch tensors) and sizes to the library of the same name and raises
``DflashError`` on a non-zero return code.  There is no fallback: if the
shared library is missing, loading fails loudly.
"""
import ctypes
import os

import torch

from . import _build

_LIB = None


class DflashError(RuntimeError):
    def __init__(self, fn, code, cuda_code=0):
        msg = f"{fn}: {code} ({strerror(code)})"
        if cuda_code:
            msg += f", CUDA error {cuda_code}"
        super().__init__(msg)
        self.code = code


class DflashConfig(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("mlp", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("block", ctypes.c_int32),
                ("n_taps", ctypes.c_int32), ("conv_width", ctypes.c_int32),
                ("qk_norm", ctypes.c_int32), ("fc_norm", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("rms_eps", ctypes.c_float),
                ("rope_base", ctypes.c_float), ("kv_terms", ctypes.c_int32)]


WEIGHT_FIELDS = ["embed", "lm_head", "final_norm", "in_norm", "wqkv", "q_norm",
                 "k_norm", "wo", "post_norm", "w_gate_up", "w_down", "conv", "fc",
                 "fc_norm", "mask_embed"]


class DflashWeights(ctypes.Structure):
    _fields_ = [(f, ctypes.c_void_p) for f in WEIGHT_FIELDS]


class DflashKV(ctypes.Structure):
    _fields_ = [("pool", ctypes.c_void_p), ("page_table", ctypes.c_void_p),
                ("n_pages", ctypes.c_int32), ("max_pages", ctypes.c_int32),
                ("n_rows", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("scales", ctypes.c_void_p)]


EXPORTS = {
    # name: (restype, argtypes)
    "dflash_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "dflash_last_cuda_error": (ctypes.c_int, []),
    "dflash_model_create": (ctypes.c_int, [ctypes.POINTER(DflashConfig),
                                           ctypes.POINTER(DflashWeights),
                                           ctypes.POINTER(ctypes.c_void_p)]),
    "dflash_model_destroy": (ctypes.c_int, [ctypes.c_void_p]),
    "dflash_selftest_wait": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "dflash_workspace_bytes": (ctypes.c_size_t, [ctypes.c_void_p, ctypes.c_int32,
                                                 ctypes.c_int32, ctypes.c_int32,
                                                 ctypes.c_int32]),
    "dflash_workspace_init": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t,
                                             ctypes.c_void_p]),
    "dflash_get_status": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32),
                                         ctypes.POINTER(ctypes.c_int32), ctypes.c_void_p]),
    "dflash_ctx_fuse": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                       ctypes.c_void_p]),
    "dflash_kv_append": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_int32,
                                        ctypes.POINTER(DflashKV), ctypes.c_void_p,
                                        ctypes.c_size_t, ctypes.c_void_p]),
    "dflash_draft_block": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_int32, ctypes.POINTER(DflashKV),
                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                          ctypes.c_void_p]),
    "dflash_verify_greedy": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                            ctypes.c_int32] + [ctypes.c_void_p] * 9 +
                             [ctypes.c_void_p]),
    "dflash_kv_quantize": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_void_p]),
    "dflash_sampling_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int32, ctypes.c_int32]),
    "dflash_verify_sampling": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                              ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p] +
                               [ctypes.c_void_p] * 9 + [ctypes.c_void_p, ctypes.c_size_t,
                                                        ctypes.c_void_p]),
    "dflash_sample_rows": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                          ctypes.c_int32, ctypes.c_int32, ctypes.c_double,
                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_size_t, ctypes.c_void_p]),
    "dflash_target_forward": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_int32, ctypes.c_int32,
                                             ctypes.POINTER(DflashKV), ctypes.c_void_p,
                                             ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                             ctypes.c_void_p]),
    "dflash_kernel_launches": (ctypes.c_uint64, []),
    "dflash_ctx_fuse_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                               ctypes.c_void_p, ctypes.c_void_p]),
    "dflash_lm_head_argmax": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_size_t, ctypes.c_void_p]),
    "dflash_synth_target": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                           ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint64,
                                           ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                           ctypes.c_void_p]),
}


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Load the shared library (raises if it is not built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = lib_path()
    if not os.path.exists(path):
        if build_if_missing:
            _build.build()
        else:
            raise RuntimeError(f"CUDA library not built: {path} (run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    for name, (res, args) in EXPORTS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def strerror(code: int) -> str:
    try:
        return load().dflash_strerror(int(code)).decode()
    except Exception:  # library not loadable: still format the message
        return "?"


def _check(name, rc):
    if rc != 0:
        raise DflashError(name, rc, load().dflash_last_cuda_error())
    return rc


def ptr(t):
    """Device (or host) address of a tensor, None for None."""
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def stream_handle(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


# ----------------------------------------------------------------- the ABI
def dflash_model_create(cfg: DflashConfig, w: DflashWeights):
    h = ctypes.c_void_p()
    _check("dflash_model_create", load().dflash_model_create(ctypes.byref(cfg), ctypes.byref(w),
                                                             ctypes.byref(h)))
    return h


def dflash_model_destroy(h):
    return _check("dflash_model_destroy", load().dflash_model_destroy(h))


def dflash_workspace_bytes(h, max_block_rows, max_ctx_rows, max_batch, max_ctx_len) -> int:
    n = load().dflash_workspace_bytes(h, max_block_rows, max_ctx_rows, max_batch, max_ctx_len)
    if n == 0:
        raise DflashError("dflash_workspace_bytes", -1)
    return int(n)


def dflash_workspace_init(ws, stream=None):
    return _check("dflash_workspace_init",
                  load().dflash_workspace_init(ptr(ws), ws.numel() * ws.element_size(),
                                               stream_handle(stream)))


def dflash_get_status(ws, stream=None):
    st = ctypes.c_int32()
    site = ctypes.c_int32()
    _check("dflash_get_status", load().dflash_get_status(ptr(ws), ctypes.byref(st),
                                                         ctypes.byref(site),
                                                         stream_handle(stream)))
    return st.value, site.value


def dflash_selftest_wait(arrive, limit_ns, ws, waited_ns=None, stream=None):
    return _check("dflash_selftest_wait", load().dflash_selftest_wait(
        1 if arrive else 0, int(limit_ns), ptr(waited_ns), ptr(ws),
        ws.numel() * ws.element_size(), stream_handle(stream)))


def dflash_ctx_fuse(h, taps, T, ctx, ws, stream=None):
    return _check("dflash_ctx_fuse", load().dflash_ctx_fuse(
        h, ptr(taps), T, ptr(ctx), ptr(ws), ws.numel() * ws.element_size(),
        stream_handle(stream)))


def dflash_kv_append(h, ctx, row_req, row_pos, T, kv: DflashKV, ws, stream=None):
    return _check("dflash_kv_append", load().dflash_kv_append(
        h, ptr(ctx), ptr(row_req), ptr(row_pos), T, ctypes.byref(kv), ptr(ws),
        ws.numel() * ws.element_size(), stream_handle(stream)))


def dflash_draft_block(h, anchor, anchor_pos, batch, kv: DflashKV, pending_ctx, pending_req,
                       pending_pos, T, draft, logits, hidden, ws, stream=None):
    return _check("dflash_draft_block", load().dflash_draft_block(
        h, ptr(anchor), ptr(anchor_pos), batch, ctypes.byref(kv), ptr(pending_ctx),
        ptr(pending_req), ptr(pending_pos), T, ptr(draft), ptr(logits), ptr(hidden), ptr(ws),
        ws.numel() * ws.element_size(), stream_handle(stream)))


def dflash_kv_quantize(h, src: DflashKV, dst: DflashKV, stream=None):
    return _check("dflash_kv_quantize", load().dflash_kv_quantize(
        h, ctypes.byref(src), ctypes.byref(dst), stream_handle(stream)))


def dflash_sampling_workspace_bytes(batch, B):
    return int(load().dflash_sampling_workspace_bytes(batch, B))


def dflash_verify_sampling(draft, draft_logits, target_logits, batch, B, vocab, temperature, u, w,
                           out_tokens, n_accept, tgt_len_in, tgt_len_out, ctx_pending, anchor_out,
                           anchor_pos_in, anchor_pos_out, ws, stream=None, ctx_pos=None):
    return _check("dflash_verify_sampling", load().dflash_verify_sampling(
        ptr(draft), ptr(draft_logits), ptr(target_logits), batch, B, vocab, float(temperature),
        ptr(u), ptr(w), ptr(out_tokens), ptr(n_accept), ptr(tgt_len_in), ptr(tgt_len_out),
        ptr(ctx_pending), ptr(anchor_out), ptr(anchor_pos_in), ptr(anchor_pos_out), ptr(ctx_pos),
        ptr(ws), ws.numel() * ws.element_size(), stream_handle(stream)))


def dflash_sample_rows(logits, n_blocks, block, skip_first, vocab, temperature, a, out, ws,
                       stream=None):
    return _check("dflash_sample_rows", load().dflash_sample_rows(
        ptr(logits), n_blocks, block, skip_first, vocab, float(temperature), ptr(a), ptr(out),
        ptr(ws), ws.numel() * ws.element_size(), stream_handle(stream)))


def dflash_verify_greedy(draft, target, batch, B, out_tokens, n_accept, tgt_len_in,
                         tgt_len_out, ctx_pending, anchor_out, anchor_pos_in, anchor_pos_out,
                         stream=None, ctx_pos=None):
    return _check("dflash_verify_greedy", load().dflash_verify_greedy(
        ptr(draft), ptr(target), batch, B, ptr(out_tokens), ptr(n_accept), ptr(tgt_len_in),
        ptr(tgt_len_out), ptr(ctx_pending), ptr(anchor_out), ptr(anchor_pos_in),
        ptr(anchor_pos_out), ptr(ctx_pos), stream_handle(stream)))


def dflash_target_forward(h, tokens, pos0, batch, n, kv: DflashKV, tap_layers, n_taps, taps,
                          argmax, logits, ws, stream=None):
    return _check("dflash_target_forward", load().dflash_target_forward(
        h, ptr(tokens), ptr(pos0), batch, n, ctypes.byref(kv), ptr(tap_layers), n_taps,
        ptr(taps), ptr(argmax), ptr(logits), ptr(ws), ws.numel() * ws.element_size(),
        stream_handle(stream)))


def dflash_synth_target(draft, batch, B, threshold, vocab, seed, step, advance, target,
                        stream=None):
    return _check("dflash_synth_target", load().dflash_synth_target(
        ptr(draft), batch, B, ptr(threshold), vocab, ctypes.c_uint64(seed), ptr(step),
        int(advance), ptr(target), stream_handle(stream)))


def dflash_lm_head_argmax(h, x, rows, argmax, logits, ws, stream=None):
    return _check("dflash_lm_head_argmax", load().dflash_lm_head_argmax(
        h, ptr(x), rows, ptr(argmax), ptr(logits), ptr(ws), ws.numel() * ws.element_size(),
        stream_handle(stream)))


def dflash_kernel_launches() -> int:
    return int(load().dflash_kernel_launches())


def dflash_ctx_fuse_noalloc(h, taps, T, ctx, stream=None):
    """dflash_ctx_fuse without a workspace, for callers that cannot allocate
    device memory; its scratch is a fixed array inside the library."""
    return _check("dflash_ctx_fuse_noalloc", load().dflash_ctx_fuse_noalloc(
        h, ptr(taps), T, ptr(ctx), stream_handle(stream)))
