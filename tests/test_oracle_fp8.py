"""Pins of the fp8 (E4M3) context-K/V oracle (oracle/fp8.py), on CPU.

The codec is checked against the format's table of special values, against
PyTorch's own float8_e4m3fn cast (an independent implementation, compared
where PyTorch does not turn large values into NaN), for round trips of every
code and for ties and saturation.  The K/V scaling is checked against its
error bound.  A slow test measures what fp8 storage of the context does to
the draft logits of the Qwen3-8B-shaped and the DFlash-2 workloads.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workload as W
from oracle import fp8 as F


def test_special_codes():
    dec = F.e4m3_decode
    assert dec(0x00) == 0.0 and np.signbit(dec(0x80))
    assert dec(0x01) == 2.0 ** -9                 # smallest subnormal
    assert dec(0x07) == 7 * 2.0 ** -9             # largest subnormal
    assert dec(0x08) == 2.0 ** -6                 # smallest normal
    assert dec(0x38) == 1.0                       # exponent field 7 = bias
    assert dec(0x7E) == 448.0 and dec(0xFE) == -448.0
    assert np.isnan(dec(0x7F)) and np.isnan(dec(0xFF))
    assert dec(0x78) == 256.0                     # exponent field 15 is a normal binade
    vals = dec(np.arange(256))
    assert np.isfinite(vals).sum() == 254


def test_every_code_round_trips():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    assert np.array_equal(F.e4m3_encode(F.e4m3_decode(codes)), codes)


def test_matches_torch_float8_cast():
    g = np.random.default_rng(0)
    x = np.concatenate([g.normal(size=20000) * s for s in (1e-3, 0.05, 1.0, 30.0, 150.0)])
    x = np.concatenate([x, F.e4m3_decode(np.arange(0x7F)) * 1.0000001,
                        (F.e4m3_decode(np.arange(1, 0x7E)) + F.e4m3_decode(np.arange(2, 0x7F))) / 2])
    x = x[np.abs(x) < 464.0].astype(np.float32)   # torch gives NaN from 464 on
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = F.e4m3_decode(F.e4m3_encode(x.astype(np.float64)))
    assert np.array_equal(got, ref)


def test_ties_go_to_the_even_mantissa_and_large_values_saturate():
    enc = F.e4m3_encode
    assert enc(1.0625) == 0x38      # between 1.0 (m=0) and 1.125 (m=1): even
    assert enc(1.1875) == 0x3A      # between 1.125 (m=1) and 1.25 (m=2): even
    assert enc(2.0 ** -10) == 0x00  # half the smallest subnormal: to zero
    assert enc(1.5 * 2.0 ** -9) == 0x02
    assert enc(460.0) == 0x7E and enc(1e9) == 0x7E and enc(-1e9) == 0xFE
    assert enc(np.nan) == 0x7F


def test_quantize_kv_matches_torch_fp32_quotient_and_cast():
    """quantize_kv on bf16 vectors against PyTorch: fp32 scale amax/448,
    fp32 division, float8_e4m3fn cast (round to nearest even).  Vectors of
    small integers times a power of two make 448 * value / amax land exactly
    on E4M3 midpoints often, where an fp64 quotient would decide otherwise."""
    g = np.random.default_rng(3)
    ints = g.integers(-255, 256, size=(4000, 64)).astype(np.float64)
    ints[:, 0] = g.choice([255.0, 224.0, 192.0, 160.0, 96.0, 7.0], size=4000)
    x = ints * np.exp2(g.integers(-20, 10, size=(4000, 1)))
    x = np.concatenate([x, g.normal(size=(4000, 64)) * np.exp2(g.uniform(-20, 10, (4000, 1)))])
    x = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()  # bf16 values
    codes, scale = F.quantize_kv(x)
    xt = torch.from_numpy(x).to(torch.float32)
    amax = xt.abs().amax(-1)
    st = torch.where(amax > 0, (amax.double() / 448.0).float(), torch.ones_like(amax))
    assert np.array_equal(scale, st.numpy())
    q = xt / st[:, None]
    assert float(q.abs().max()) < 464.0            # inside torch's finite range
    ref = q.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)
    # the exact quotient decides differently from the fp32 one in many places
    exact = F.e4m3_encode(x / scale.astype(np.float64)[:, None])
    assert int((exact != codes).sum()) > 100


def test_kv_scaling_error_bound():
    """Per (position, head) scale amax/448: every element is within half a
    3-bit-mantissa step of its value (relative 2^-4) or, below the normal
    range, within half the subnormal step times the scale."""
    g = np.random.default_rng(1)
    x = g.normal(size=(300, 8, 128)) * g.uniform(0.01, 10, size=(300, 8, 1))
    x[5, 3] = 0.0
    codes, scale = F.quantize_kv(x)
    y = F.dequantize_kv(codes, scale)
    assert codes.dtype == np.uint8 and scale.dtype == np.float32
    assert np.all(np.max(np.abs(F.e4m3_decode(codes)), axis=-1)[np.any(x != 0, axis=-1)] == 448.0)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, scale.astype(np.float64)[..., None] * 2.0 ** -10)
    assert np.all(np.abs(y - x) <= bound * (1 + 1e-6))
    assert np.all(y[5, 3] == 0.0) and scale[5, 3] == 1.0


def fp8_study(name, req=0):
    """Draft logits of one request of a workload with the context K/V in bf16
    and in fp8; returns (max |dlogit|, rms, logit std, top-1 agreement,
    rows)."""
    wl = W.get_workload(name)
    d = wl.draft
    wid = wl.wid
    dws = O.LayerStack(d, W.draft_weights(d, wid), W.shared_weights(d, wid))
    C = int(W.ctx_lengths(wl)[req])
    new = W.new_row_counts(wl)
    T, o = int(new[req]), int(new[:req].sum())
    taps = W.taps_bf16(int(new.sum()), d, wid)[o:o + T]
    c_rows = O.ctx_fuse(d, dws, O.bf16_to_f64(taps))
    ks, vs = [], []
    for l in range(d.n_layers):
        kn, vn = O.ctx_kv(d, dws, l, c_rows, np.arange(C, C + T))
        ks.append(np.concatenate([O.bf16_to_f64(W.context_kv_bf16(d, wid, l, req, C, "k")), kn]))
        vs.append(np.concatenate([O.bf16_to_f64(W.context_kv_bf16(d, wid, l, req, C, "v")), vn]))
    anchor = int(W.uniform_tokens(wl.batch, d.vocab, wid, W.TENSOR_IDS["anchor"])[req])
    ref, q8 = F.kv_study(d, dws, anchor, C + T, ks, vs, O.draft_block)
    assert np.all(np.isfinite(q8))
    diff = np.abs(q8 - ref)[1:]
    agree = float(np.mean(np.argmax(q8[1:], -1) == np.argmax(ref[1:], -1)))
    return float(diff.max()), float(np.sqrt((diff ** 2).mean())), float(ref[1:].std()), agree, \
        diff.shape[0]


@pytest.mark.slow
@pytest.mark.parametrize("name", ["qwen3_8b_b1", "dflash2_b16"])
def test_fp8_context_study(name):
    """Draft logits with the context K/V in bf16 and in fp8 for the first
    request of the Qwen3-8B-shaped batch-1 and the DFlash-2 workloads.
    Prints the measured change; asserts only that the fp8 cache perturbs the
    logits (it is a lossy format) and keeps every logit finite."""
    mx, rms, std, agree, rows = fp8_study(name)
    print(f"\nfp8 context K/V, {name}: max|dlogit| {mx:.4f}, rms {rms:.5f}, "
          f"logit std {std:.3f}, top-1 agreement {agree:.3f} over {rows} rows")
    assert mx > 0.0
