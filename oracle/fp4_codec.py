"""FP4 latent-cache decoding, written from the published format definitions.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Format facts used:
  * "DeepSeek-R1" model record, engine kernel constraint (2): the decode
    kernel takes FP8 or FP4 latents with per-token inlined scales; the FP8
    row carries one float8_e8m0 scale per 32 values, and the FP4 variant is
    288 bytes per token for a row of 512 values.
  * OCP Microscaling (MX) specification, FP4 E2M1: 1 sign bit, 2 exponent
    bits with bias 1, 1 mantissa bit; exponent field 0 encodes the
    subnormal m * 0.5; no infinities and no NaN.
  * OCP MX specification, E8M0 scale: 2^(e-127), 0xFF is NaN.

Reading taken for the row (the record gives only its size): every value is
an e2m1 code, two codes per byte with value 2i in the low nibble of byte i,
followed by one e8m0 scale per 16 values.  That is 256 + 32 = 288 bytes for
512 values, the record's figure, and 288 + 36 = 324 bytes for the 576-value
row (512 latent, then 64 RoPE) decoded here: bytes [0, 288) hold the codes,
bytes [288, 324) the 36 scales, scale k covering values [16k, 16k+16).

The record's own 288-byte row (the V4.1 geometry, 512 values) is read the
same way: bytes [0, 256) hold the 512 codes, bytes [256, 288) the 32 scales,
and its 512 values are 448 latent values followed by the 64 RoPE values, as
for the 528-byte FP8 row; on the 576-value row the latent fills dims
[0, 448) and dims [448, 512) are zero.
"""
from __future__ import annotations

import numpy as np

from .fp8_codec import e8m0_to_float64

ROW_VALUES = 576
SCALE_GROUP = 16
NUM_SCALES = ROW_VALUES // SCALE_GROUP        # 36
CODE_BYTES = ROW_VALUES // 2                  # 288
ROW_BYTES = CODE_BYTES + NUM_SCALES           # 324

V41_VALUES = 512                              # 448 latent + 64 RoPE
V41_LATENT = 448
V41_CODE_BYTES = V41_VALUES // 2              # 256
V41_ROW_BYTES = V41_CODE_BYTES + V41_VALUES // SCALE_GROUP   # 288


def e2m1_to_float64(codes: np.ndarray) -> np.ndarray:
    """Decode 4-bit OCP E2M1 codes (0..15) to float64 by their bit fields."""
    c = np.asarray(codes, dtype=np.int64)
    assert np.all((c >= 0) & (c < 16))
    sign = np.where((c & 0x8) != 0, -1.0, 1.0)
    exp = (c >> 1) & 0x3
    man = (c & 0x1).astype(np.float64)
    normal = sign * (1.0 + man / 2.0) * np.exp2(exp - 1)
    subnormal = sign * man * 0.5
    return np.where(exp == 0, subnormal, normal)


def unpack_codes(code_bytes: np.ndarray) -> np.ndarray:
    """[..., n] bytes -> [..., 2n] 4-bit codes: value 2i from the low nibble
    of byte i, value 2i+1 from its high nibble."""
    b = np.asarray(code_bytes, dtype=np.uint8)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = b & 0x0F
    out[..., 1::2] = b >> 4
    return out


def dequant_rows(raw: np.ndarray) -> np.ndarray:
    """[..., 324] uint8 rows -> [..., 576] float64 values.

    value[k] = e2m1(code k) * e8m0(byte[288 + k // 16]).
    """
    raw = np.asarray(raw, dtype=np.uint8)
    assert raw.shape[-1] == ROW_BYTES, raw.shape
    vals = e2m1_to_float64(unpack_codes(raw[..., :CODE_BYTES]))
    scales = e8m0_to_float64(raw[..., CODE_BYTES:])
    return vals * np.repeat(scales, SCALE_GROUP, axis=-1)


def dequant_rows_v41(raw: np.ndarray) -> np.ndarray:
    """[..., 288] uint8 V4.1 rows -> [..., 576] float64 values on this path's
    row: dims [0, 448) the V4.1 latent, [448, 512) zero, [512, 576) the RoPE
    values.  value[k] = e2m1(code k) * e8m0(byte[256 + k // 16])."""
    raw = np.asarray(raw, dtype=np.uint8)
    assert raw.shape[-1] == V41_ROW_BYTES, raw.shape
    vals = e2m1_to_float64(unpack_codes(raw[..., :V41_CODE_BYTES]))
    scales = e8m0_to_float64(raw[..., V41_CODE_BYTES:])
    v = vals * np.repeat(scales, SCALE_GROUP, axis=-1)
    out = np.zeros(raw.shape[:-1] + (ROW_VALUES,), dtype=np.float64)
    out[..., :V41_LATENT] = v[..., :V41_LATENT]
    out[..., ROW_VALUES - (V41_VALUES - V41_LATENT):] = v[..., V41_LATENT:]
    return out

