"""FP8 latent-cache decoding, written from the published format definitions.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Format facts used:
  * "DeepSeek-R1" model record, engine kernel constraint (2): latents are
    stored as float8_e4m3 with one float8_e8m0 scale per 32 e4m3 values,
    inlined in each token's row.
  * "DeepSeek R1 Architecture & Deployment Guide", section 4: E4M3 max
    normal = 448.0.
  * OCP 8-bit floating point specification, E4M3 ("fn" flavour): 1 sign bit,
    4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 encodes
    subnormals m/8 * 2^-6; no infinities; S.1111.111 is NaN.
  * OCP Microscaling (MX) specification, E8M0 scale: an unsigned 8-bit
    exponent with bias 127, value 2^(e-127); 0xFF is NaN.

Row layout (the reading taken for the 594-byte row): bytes [0, 576) are the
e4m3 codes of the 576 values (512 latent, then 64 RoPE), bytes [576, 594) are
18 e8m0 scales, scale k covering values [32k, 32k+32).

The V4.1 row (same record, same constraint (2)): 528 bytes per token, 512
e4m3 codes "over all 512 dims", the 64 RoPE dims quantized too, then 16 e8m0
scales, one per 32 codes.  Reading taken: its 512 values are 448 latent
values followed by the 64 RoPE values (the same order as the 576-value row),
scale k covering values [32k, 32k+32).  On this path's 576-value row the
V4.1 latent occupies dims [0, 448); dims [448, 512) are zero.
"""
from __future__ import annotations

import numpy as np

ROW_VALUES = 576
SCALE_GROUP = 32
NUM_SCALES = ROW_VALUES // SCALE_GROUP
ROW_BYTES = ROW_VALUES + NUM_SCALES

V41_VALUES = 512                          # 448 latent + 64 RoPE
V41_LATENT = 448
V41_NUM_SCALES = V41_VALUES // SCALE_GROUP  # 16
V41_ROW_BYTES = V41_VALUES + V41_NUM_SCALES  # 528


def e4m3fn_to_float64(codes: np.ndarray) -> np.ndarray:
    """Decode OCP E4M3FN bytes to float64 by their bit fields."""
    b = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where((b & 0x80) != 0, -1.0, 1.0)
    exp = (b >> 3) & 0xF
    man = (b & 0x7).astype(np.float64)
    normal = sign * (1.0 + man / 8.0) * np.exp2(exp - 7)
    subnormal = sign * (man / 8.0) * 2.0 ** -6
    val = np.where(exp == 0, subnormal, normal)
    return np.where((exp == 0xF) & ((b & 0x7) == 0x7), np.nan, val)


def e8m0_to_float64(codes: np.ndarray) -> np.ndarray:
    """Decode OCP MX E8M0 scale bytes: 2^(e-127), 0xFF -> NaN."""
    e = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    return np.where(e == 0xFF, np.nan, np.exp2(e - 127).astype(np.float64))


def dequant_rows(raw: np.ndarray) -> np.ndarray:
    """[..., 594] uint8 rows -> [..., 576] float64 values.

    value[k] = e4m3(byte[k]) * e8m0(byte[576 + k // 32]).
    """
    raw = np.asarray(raw, dtype=np.uint8)
    assert raw.shape[-1] == ROW_BYTES, raw.shape
    vals = e4m3fn_to_float64(raw[..., :ROW_VALUES])
    scales = e8m0_to_float64(raw[..., ROW_VALUES:])
    return vals * np.repeat(scales, SCALE_GROUP, axis=-1)


def dequant_rows_v41(raw: np.ndarray) -> np.ndarray:
    """[..., 528] uint8 V4.1 rows -> [..., 576] float64 values on this path's
    row: dims [0, 448) are the V4.1 latent, [448, 512) zero, [512, 576) the
    RoPE values.  value[k] = e4m3(byte[k]) * e8m0(byte[512 + k // 32])."""
    raw = np.asarray(raw, dtype=np.uint8)
    assert raw.shape[-1] == V41_ROW_BYTES, raw.shape
    vals = e4m3fn_to_float64(raw[..., :V41_VALUES])
    scales = e8m0_to_float64(raw[..., V41_VALUES:])
    v = vals * np.repeat(scales, SCALE_GROUP, axis=-1)
    out = np.zeros(raw.shape[:-1] + (ROW_VALUES,), dtype=np.float64)
    out[..., :V41_LATENT] = v[..., :V41_LATENT]
    out[..., ROW_VALUES - (V41_VALUES - V41_LATENT):] = v[..., V41_LATENT:]
    return out



# ---------------------------------------------------------------------------
# Encoding: the query side of a block-scaled FP8 score product.
#
# Reading taken (the record's constraint (2) fixes the cache's codes and
# scales, not the query's): the query is quantised like a cache row, e4m3
# codes with one e8m0 scale per 32 values, the scale being the smallest power
# of two that brings the group's largest magnitude to at most 448 (the e4m3
# maximum normal, architecture guide section 4), codes rounded to nearest with
# ties to even.  One such term keeps four significant bits of each value; the
# residual q - deq(hi), quantised the same way, gives a second term, and the
# two together carry about as many bits as the bf16 query does.

def float64_to_e4m3fn(x: np.ndarray) -> np.ndarray:
    """Encode float64 values with |x| <= 448 as OCP E4M3FN bytes, rounding to
    nearest, ties to even (the encoding's own grid: spacing 2^(e-3) in the
    binade [2^e, 2^(e+1)) for e >= -6, spacing 2^-9 below 2^-6)."""
    x = np.asarray(x, dtype=np.float64)
    assert np.all(np.isfinite(x)) and np.all(np.abs(x) <= 448.0), "outside the e4m3 range"
    a = np.abs(x)
    _, ex = np.frexp(a)                             # a = m 2^ex, m in [0.5, 1)
    e = np.maximum(ex.astype(np.int64) - 1, -6)     # binade exponent, floored at the subnormal range
    quantum = np.exp2((e - 3).astype(np.float64))
    n = np.rint(a / quantum)                        # numpy rounds half to even
    v = n * quantum                                 # the rounded magnitude, exact
    _, vex = np.frexp(v)
    normal = v >= 2.0 ** -6
    exp_field = np.where(normal, vex.astype(np.int64) - 1 + 7, 0)
    man_field = np.where(normal, v / np.exp2((exp_field - 7).astype(np.float64)) * 8 - 8, v / 2.0 ** -9)
    code = (exp_field << 3) | man_field.astype(np.int64)
    return (code | (np.signbit(x).astype(np.int64) << 7)).astype(np.uint8)


def block_scale_exponent(amax: np.ndarray) -> np.ndarray:
    """Smallest integer k with amax <= 448 * 2^k (k = 0 for an all-zero group).
    With amax = m 2^E, m in [0.5, 1): 448 * 2^k = 0.875 * 2^(k+9), so k = E - 9
    when m <= 0.875 and E - 8 otherwise, with no rounding anywhere."""
    amax = np.asarray(amax, dtype=np.float64)
    m, ex = np.frexp(amax)
    k = np.where(m <= 0.875, ex - 9, ex - 8).astype(np.int64)
    return np.where(amax == 0, 0, k)


def quantise_blocks(x: np.ndarray, group: int = SCALE_GROUP):
    """[..., n] float64 -> (e4m3 codes [..., n], e8m0 scale codes [..., n/group]).
    Group g's scale is 2^k with k = block_scale_exponent(max |x| over the group);
    its codes are e4m3(x / 2^k)."""
    x = np.asarray(x, dtype=np.float64)
    assert x.shape[-1] % group == 0
    g = x.reshape(x.shape[:-1] + (x.shape[-1] // group, group))
    k = block_scale_exponent(np.abs(g).max(axis=-1))
    assert np.all((k >= -127) & (k <= 127)), "scale outside e8m0"
    codes = float64_to_e4m3fn(g / np.exp2(k.astype(np.float64))[..., None])
    return codes.reshape(x.shape), (k + 127).astype(np.uint8)


def dequant_blocks(codes: np.ndarray, scales: np.ndarray, group: int = SCALE_GROUP) -> np.ndarray:
    """The inverse map: value[k] = e4m3(codes[k]) * e8m0(scales[k // group])."""
    return e4m3fn_to_float64(codes) * np.repeat(e8m0_to_float64(scales), group, axis=-1)


def split_e4m3_terms(x: np.ndarray, group: int = SCALE_GROUP):
    """x ~ hi + lo: hi = quantise_blocks(x), lo = quantise_blocks(x - deq(hi)).
    Returns ((hi codes, hi scales), (lo codes, lo scales))."""
    x = np.asarray(x, dtype=np.float64)
    hi = quantise_blocks(x, group)
    lo = quantise_blocks(x - dequant_blocks(*hi, group=group), group)
    return hi, lo
