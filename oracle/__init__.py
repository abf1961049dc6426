"""CPU oracle for DFlash-style block-diffusion drafting and greedy verification.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
anything in this package.  The product (the CUDA library and its Python
binding) never calls it and has no CPU fallback.

Plain NumPy in float64, written from the method's description, sharing no code
with the CUDA path (only the seeded generators in ``workload/`` feed both).

Pins (tests/test_oracle_pins.py): every building block is checked against
closed forms, textbook special cases, an independent library routine (PyTorch
CPU ``rms_norm``, ``scaled_dot_product_attention``, ``linear``, ``silu``) or
brute force; the composed draft step is pinned by invariants (non-causality,
context-order invariance, RoPE shift invariance, incremental == one-shot
context projection, DFlash-2 conv reductions) and the speculative loop by
token identity with autoregressive greedy decoding; the composition of the
layer stacks (tests/test_oracle_layer_pins.py) by special cases with closed
forms: zero output/down projections (identity layers), equal values
(attention returns V whatever the scores) and the DFlash-2 convolution
against PyTorch's conv1d, with planted mistakes that must fail.  A full
random-init step has no external reference value (no trained model, no
printed example); the pins above vouch for every piece of it.

``oracle.sampling`` holds the sampling-mode (temperature > 0) verify: the
standard speculative-sampling acceptance rule applied to a block draft,
pinned by brute force, its greedy limit, exact special cases and Monte Carlo
checks of losslessness (tests/test_oracle_sampling.py).

``oracle.fp8`` holds the E4M3 codec and per-(position, head) scaling for an
fp8 context K/V cache and the study of its effect on the draft logits,
pinned against the format's table and PyTorch's float8 cast
(tests/test_oracle_fp8.py).
"""
from .dflash_oracle import *  # noqa: F401,F403
from . import fp8, sampling  # noqa: F401,E402
