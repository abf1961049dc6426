"""Host-side checks of the C-ABI library (no GPU needed): it loads, exports
every symbol the header declares, and rejects bad arguments before launching
anything."""
import ctypes
import os
import re

import pytest

from block_diffusion_speculative_fuse_gb300 import _build, binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return B.load()


def header_symbols():
    src = open(os.path.join(ROOT, "include", "dflash.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary_calls():
    syms = header_symbols()
    for s in ("dflash_ctx_fuse", "dflash_kv_append", "dflash_draft_block",
              "dflash_verify_greedy"):
        assert s in syms


def test_library_exports_every_declared_symbol(lib):
    for s in header_symbols():
        assert hasattr(lib, s), s
        assert s in B.EXPORTS, f"binding misses {s}"


def test_strerror_codes(lib):
    assert B.strerror(0) == "ok"
    assert "invalid" in B.strerror(-1)
    assert "capacity" in B.strerror(-3)
    assert B.strerror(-99) == "unknown error"


def test_model_create_rejects_bad_args(lib):
    h = ctypes.c_void_p()
    assert lib.dflash_model_create(None, None, ctypes.byref(h)) == -1
    cfg = B.DflashConfig(n_layers=1, hidden=100, n_q_heads=4, n_kv_heads=2, head_dim=64,
                         mlp=256, vocab=1024, block=8, n_taps=2, conv_width=0, qk_norm=1,
                         fc_norm=1, page_size=16, rms_eps=1e-6, rope_base=1e4)
    w = B.DflashWeights()
    assert lib.dflash_model_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == -2
    cfg.hidden = 256
    cfg.head_dim = 96
    assert lib.dflash_model_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == -2
    cfg.head_dim = 64
    cfg.block = 33
    assert lib.dflash_model_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == -2
    cfg.block = 8
    cfg.conv_width = 2
    assert lib.dflash_model_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == -2
    cfg.conv_width = 0
    # valid shape, missing weight pointers
    assert lib.dflash_model_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == -1
    w.embed = 0x1001  # misaligned
    assert lib.dflash_model_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == -1


def test_verify_rejects_bad_sizes(lib):
    f = lib.dflash_verify_greedy
    dummy = ctypes.c_void_p(0x1000)
    assert f(dummy, dummy, 0, 16, *([None] * 9), None) == -1      # batch 0
    assert f(dummy, dummy, 1, 0, *([None] * 9), None) == -1       # B 0
    assert f(dummy, dummy, 1, 33, *([None] * 9), None) == -1      # B > 32
    assert f(None, dummy, 1, 4, *([None] * 9), None) == -1        # drafts missing
    # an output length without its input
    args = [None] * 9
    args[3] = dummy
    assert f(dummy, dummy, 1, 4, *args, None) == -1
    # pending positions without the anchor positions they are built from
    args = [None] * 9
    args[8] = dummy
    assert f(dummy, dummy, 1, 4, *args, None) == -1


def test_synth_target_rejects_bad_sizes(lib):
    f = lib.dflash_synth_target
    d = ctypes.c_void_p(0x1000)
    assert f(d, 64, 32, d, 100, 1, d, 1, d, None) == -1          # batch*B > 1024
    assert f(d, 1, 4, d, 1, 1, d, 1, d, None) == -1               # vocab < 2
    assert f(d, 1, 4, None, 100, 1, d, 1, d, None) == -1          # no thresholds


def test_workspace_init_rejects_misaligned(lib):
    assert lib.dflash_workspace_init(ctypes.c_void_p(0x1004), 1 << 20, None) == -1
    assert lib.dflash_workspace_init(ctypes.c_void_p(0x1000), 16, None) == -1


def test_compute_calls_reject_null_handle(lib):
    d = ctypes.c_void_p(0x1000)
    assert lib.dflash_ctx_fuse(None, d, 4, d, d, 1 << 20, None) == -1
    kv = B.DflashKV()
    assert lib.dflash_kv_append(None, d, d, d, 4, ctypes.byref(kv), d, 1 << 20, None) == -1
    assert lib.dflash_draft_block(None, d, d, 1, ctypes.byref(kv), None, None, None, 0, d,
                                  None, None, d, 1 << 20, None) == -1
    assert lib.dflash_target_forward(None, d, d, 1, 1, ctypes.byref(kv), None, 0, None, d,
                                     None, d, 1 << 20, None) == -1
    assert lib.dflash_workspace_bytes(None, 16, 16, 1, 128) == 0


def test_selftest_wait_rejects_bad_args_before_launch(lib):
    ws = ctypes.c_void_p(1 << 20)  # never dereferenced: every call below fails its checks
    assert lib.dflash_selftest_wait(0, 1000, None, None, 1 << 16, None) == -1
    assert lib.dflash_selftest_wait(0, 1000, None, ws, 1024, None) == -1
    assert lib.dflash_selftest_wait(0, 0, None, ws, 1 << 16, None) == -1
    assert lib.dflash_selftest_wait(0, 10**9 + 1, None, ws, 1 << 16, None) == -1
    assert lib.dflash_selftest_wait(0, 1000, ctypes.c_void_p(4), ws, 1 << 16, None) == -1


def test_sampling_calls_reject_bad_args_before_launch(lib):
    d = ctypes.c_void_p(0x1000)
    ws = ctypes.c_void_p(1 << 20)  # never dereferenced: every call below fails its checks
    need = lib.dflash_sampling_workspace_bytes(2, 16)
    assert need == 64 * 1024 + ((2 * 31 * 16 + 255) // 256) * 256
    assert lib.dflash_sampling_workspace_bytes(0, 16) == 0
    f = lib.dflash_verify_sampling
    ok = [d, d, d, 2, 16, 1000, 0.7, d, d] + [d] + [None] * 8
    assert f(*ok[:6], 0.0, *ok[7:], ws, need, None) == -1          # T = 0
    assert f(*ok[:6], float("nan"), *ok[7:], ws, need, None) == -1
    assert f(*ok[:3], 2, 33, *ok[5:], ws, need, None) == -1        # B > 32
    assert f(None, *ok[1:], ws, need, None) == -1                  # drafts missing (B > 1)
    assert f(*ok[:9], None, *ok[10:], ws, need, None) == -1        # out_tokens missing
    assert f(*ok, ctypes.c_void_p((1 << 20) + 8), need, None) == -1  # misaligned workspace
    assert f(*ok, ws, need - 1, None) == -3                        # workspace too small
    g = lib.dflash_sample_rows
    assert g(d, 2, 16, 2, 1000, 0.7, d, d, ws, need, None) == -1   # skip_first not 0/1
    assert g(d, 2, 1, 1, 1000, 0.7, d, d, ws, need, None) == -1    # no used rows
    assert g(d, 2, 16, 1, 1000, -1.0, d, d, ws, need, None) == -1  # T < 0
    assert g(d, 2, 16, 1, 1000, 0.7, d, d, ws, 1024, None) == -3   # workspace too small
