"""Shared test fixtures: tiny models built from the seeded generators."""
import numpy as np

import workload as W
from workload.shapes import DraftShape, ModelShape, tiny_workload


def tiny_target(vocab=211, hidden=64, layers=3, hq=4, hkv=2, d=16, mlp=96,
                rope_base=1e4):
    return ModelShape(n_layers=layers, hidden=hidden, n_q_heads=hq,
                      n_kv_heads=hkv, head_dim=d, mlp=mlp, vocab=vocab,
                      rms_eps=1e-6, rope_base=rope_base)


def tiny_draft(vocab=211, hidden=64, layers=2, hq=4, hkv=2, d=16, mlp=96,
               block=4, n_taps=2, conv_width=0, rope_base=1e4, qk_norm=True):
    return DraftShape(n_layers=layers, hidden=hidden, n_q_heads=hq,
                      n_kv_heads=hkv, head_dim=d, mlp=mlp, vocab=vocab,
                      rms_eps=1e-6, rope_base=rope_base, qk_norm=qk_norm,
                      block=block, n_taps=n_taps, conv_width=conv_width)


def build_models(wid, tshape, dshape, std=0.02, target_std=None):
    """Returns (shared, target weights, draft weights) as bf16-bit dicts."""
    shared = W.shared_weights(tshape, wid, std=target_std or std)
    tw = W.target_weights(tshape, wid, std=target_std or std)
    dw = W.draft_weights(dshape, wid, std=std)
    return shared, tw, dw
