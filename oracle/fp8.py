"""fp8 (E4M3) storage of the draft context K/V: codec and the accuracy study.

TEST INFRASTRUCTURE ONLY (see the package docstring).

"DFlash-2: z-lab boosts speculative decoding throughput..." (dothoosh.com),
section on the cost of precision, reports that an 8-bit KV cache lowered
DFlash-2's acceptance against a 16-bit one.  This module lets the same
trade-off be measured for an fp8 context cache: the K/V rows are stored as
E4M3 codes with one fp32 scale per (position, KV head) and decoded before
attention; the block's own K/V stay in full precision.

E4M3, written from the format's definition: sign bit, 4 exponent bits (bias
7), 3 mantissa bits; exponent field 0 holds the subnormals m * 2^-9; code
S.1111.111 is NaN and there are no infinities, so the largest finite
magnitude is 1.75 * 2^8 = 448.  Encoding rounds to the nearest code, ties to
the even mantissa, and saturates finite values beyond 448 to +-448.

Reading: the scale of a (position, head) vector of d values is amax / 448,
so its largest element maps to the top code (an all-zero vector keeps scale
1).  The pages name no scaling granularity; per (position, head) is the
plainest choice that needs no calibration data.  Nor do they fix the
precision of value / scale: the quotient is taken in fp32, the precision a
GPU kernel forms it in, so that both decide each code from the same number.
"""
import numpy as np

F64 = np.float64
E4M3_MAX = 448.0


def e4m3_decode(codes):
    """Value of each 8-bit code (NaN for the two NaN codes)."""
    c = np.asarray(codes, dtype=np.int64) & 0xFF
    s = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * 2.0 ** (e.astype(F64) - 7))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return s * val


_CODES = np.arange(256)
_VALS = e4m3_decode(_CODES)
_FINITE_POS = np.array([c for c in range(128) if np.isfinite(_VALS[c])])  # 0x00 .. 0x7E


def e4m3_encode(x):
    """Nearest E4M3 code of each value: ties to the even mantissa, finite
    values beyond 448 saturate, NaN maps to 0x7F.  Plain search over the 127
    non-negative finite codes (their values increase with the code)."""
    x = np.asarray(x, dtype=F64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    vals = _VALS[_FINITE_POS]
    hi = np.clip(np.searchsorted(vals, a, side="left"), 0, len(vals) - 1)
    lo = np.clip(hi - 1, 0, len(vals) - 1)
    d_lo = np.abs(a - vals[lo])
    d_hi = np.abs(vals[hi] - a)
    code_lo, code_hi = _FINITE_POS[lo], _FINITE_POS[hi]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (code_hi % 2 == 0) & (code_lo % 2 == 1))
    code = np.where(pick_hi, code_hi, code_lo)
    code = np.where(np.signbit(x), code | 0x80, code)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def quantize_kv(x):
    """x: [..., d] K or V vectors.  Returns (codes uint8 [..., d], scale
    fp32 [...]) with scale = amax / 448 per vector (1 for a zero vector).

    The code is decided from the quotient value / scale formed in fp32 (the
    values and the scale are fp32 numbers; the division is rounded to
    nearest), then rounded to E4M3.  With bf16 inputs 448 * value / amax is
    often exactly halfway between two codes, and the rounded fp32 scale moves
    the exact quotient just off that midpoint in either direction; deciding
    from the fp32 quotient makes every such case a tie, resolved to the even
    mantissa."""
    x = np.asarray(x, dtype=F64)
    amax = np.max(np.abs(x), axis=-1)
    scale = np.where(amax > 0, amax / E4M3_MAX, 1.0).astype(np.float32)
    q = np.asarray(x, dtype=np.float32) / scale[..., None]
    codes = e4m3_encode(q.astype(F64))
    return codes, scale


def dequantize_kv(codes, scale):
    return e4m3_decode(codes) * np.asarray(scale, dtype=F64)[..., None]


def kv_roundtrip(x):
    """K/V as an fp8 context cache returns them: quantize, then decode."""
    return dequantize_kv(*quantize_kv(x))


def kv_study(dshape, dw, anchor, L, ctx_k, ctx_v, draft_block):
    """Draft logits with the context K/V as given and with the same K/V
    stored as fp8.  ``draft_block`` is the oracle's block pass
    (``oracle.draft_block``); ctx_k / ctx_v: per layer [L][hkv][d].
    Returns (logits_ref, logits_fp8), each [B][V]."""
    _, ref = draft_block(dshape, dw, anchor, L, ctx_k, ctx_v)
    qk = [kv_roundtrip(k) for k in ctx_k]
    qv = [kv_roundtrip(v) for v in ctx_v]
    _, q8 = draft_block(dshape, dw, anchor, L, qk, qv)
    return ref, q8


__all__ = ["E4M3_MAX", "e4m3_decode", "e4m3_encode", "quantize_kv", "dequantize_kv",
           "kv_roundtrip", "kv_study"]
