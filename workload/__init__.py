"""Seeded synthetic inputs for DFlash-style block-diffusion drafting.

This package is the only code shared by the CPU oracle (``oracle/``) and the
CUDA path (``block_diffusion_speculative_fuse_gb300``).  It draws random
numbers and lays them out; it holds none of the method's arithmetic (no
norm, projection, attention, argmax or acceptance rule).

Every tensor is a pure function of (workload id, tensor id, chunk index):
NumPy ``PCG64(SeedSequence([workload, tensor, chunk, 20261202]))``.
Floating-point tensors are produced in float32 and stored as bfloat16 bit
patterns (``uint16``, round-to-nearest-even), so both sides see the same bits.
"""
from .shapes import (ModelShape, DraftShape, Workload, WORKLOADS, get_workload,
                     tiny_workload)
from .gen import (bf16_bits, normal_bf16, ones_bf16, uniform_tokens, rng_for,
                  draft_weights, target_weights, shared_weights, taps_bf16,
                  context_kv_bf16, page_table, ctx_lengths, agreement_probs,
                  synth_target_ids, new_row_counts, agree_threshold, TENSOR_IDS,
                  jittered_gains, GAIN_KEYS)

__all__ = [
    "ModelShape", "DraftShape", "Workload", "WORKLOADS", "get_workload",
    "jittered_gains", "GAIN_KEYS",
    "tiny_workload", "bf16_bits", "normal_bf16", "ones_bf16", "uniform_tokens",
    "rng_for", "draft_weights", "target_weights", "shared_weights",
    "taps_bf16", "context_kv_bf16", "page_table", "ctx_lengths",
    "agreement_probs", "synth_target_ids", "new_row_counts", "agree_threshold", "TENSOR_IDS",
]
