"""Pins of the oracle's e4m3 encoder and block quantiser (the query side of a
block-scaled FP8 score product).

Against torch's float8_e4m3fn cast (an independent library routine), the
decoder it inverts, a brute-force search for the block scale, the format's
rounding-error bound, and the attention oracle's LSE on workload-shaped
inputs.  The last test plants plausible mistakes in copies and checks that
each is caught.
"""
import math

import numpy as np
import pytest
import torch

from oracle import fp8_codec, mla_oracle
from mla_latent_kv_05_gb300 import inputs as gen


def _torch_e4m3(x):
    # the values are float32-exact, so torch's float32 -> e4m3 step sees them unrounded
    return torch.from_numpy(np.asarray(x, dtype=np.float64)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _finite_values():
    codes = np.arange(256, dtype=np.uint8)
    v = fp8_codec.e4m3fn_to_float64(codes)
    return codes[~np.isnan(v)], v[~np.isnan(v)]


def _encoder_cases():
    rng = np.random.default_rng(21)
    spread = rng.standard_normal(100_000) * np.exp2(rng.integers(-14, 9, 100_000))
    _, v = _finite_values()
    pos = np.unique(v[v >= 0])
    ties = (pos[1:] + pos[:-1]) / 2                       # every midpoint of adjacent values
    near = np.concatenate([np.nextafter(ties, 0), np.nextafter(ties, 1000)])
    x = np.concatenate([spread, ties, -ties, near, -near, v]).astype(np.float32).astype(np.float64)
    return x[np.abs(x) <= 448.0]


def _encoder_pins_ok(encode) -> bool:
    x = _encoder_cases()
    if not np.array_equal(encode(x), _torch_e4m3(x)):
        return False
    codes, v = _finite_values()
    return np.array_equal(encode(v), codes)


def test_encoder_matches_torch_cast_including_ties_and_subnormals():
    x = _encoder_cases()
    assert np.any(np.abs(x) < 2.0 ** -6) and np.any(np.abs(x) > 240)
    assert np.array_equal(fp8_codec.float64_to_e4m3fn(x), _torch_e4m3(x))


def test_encoder_inverts_the_decoder_on_every_finite_code():
    codes, v = _finite_values()
    assert len(codes) == 254
    assert np.array_equal(fp8_codec.float64_to_e4m3fn(v), codes)    # +0 and -0 included


def test_ties_go_to_the_even_code():
    # 1.0625 lies halfway between 1.0 (mantissa 000) and 1.125 (001);
    # 1.1875 halfway between 1.125 (001) and 1.25 (010)
    enc = fp8_codec.float64_to_e4m3fn(np.array([1.0625, 1.1875, -1.0625, 2.0 ** -10, 3 * 2.0 ** -10]))
    assert list(enc) == [0x38, 0x3A, 0xB8, 0x00, 0x02]


def _brute_scale_exponent(amax):
    if amax == 0:
        return 0
    k = -140
    while amax > 448.0 * math.ldexp(1.0, k):
        k += 1
    return k


def test_block_scale_is_the_smallest_power_of_two_that_fits():
    rng = np.random.default_rng(3)
    amax = np.concatenate([
        np.abs(rng.standard_normal(2000)) * np.exp2(rng.integers(-60, 60, 2000)),
        448.0 * np.exp2(np.arange(-20, 21.0)),                    # exactly on a boundary
        np.nextafter(448.0 * np.exp2(np.arange(-20, 21.0)), np.inf),
        np.nextafter(448.0 * np.exp2(np.arange(-20, 21.0)), 0),
        [0.0, 7 * 2.0 ** -9, 448.0, 449.0, 1.0]])
    got = fp8_codec.block_scale_exponent(amax)
    assert [int(k) for k in got] == [_brute_scale_exponent(float(a)) for a in amax]


def test_block_quantise_error_bound_and_idempotence():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((64, 576)) * np.exp2(rng.integers(-8, 8, (64, 1)))
    x[3, 32:64] = 0.0                                              # an all-zero group
    codes, scales = fp8_codec.quantise_blocks(x)
    assert codes.shape == x.shape and scales.shape == (64, 18)
    assert np.all(scales[3, 1] == 127) and np.all(codes[3, 32:64] == 0)
    d = fp8_codec.dequant_blocks(codes, scales)
    s = np.repeat(fp8_codec.e8m0_to_float64(scales), 32, axis=-1)
    # half a spacing: 2^-4 relative in the normal range, 2^-10 * s below it
    assert np.all(np.abs(x - d) <= np.maximum(np.abs(x) * 2.0 ** -4, s * 2.0 ** -10))
    # every group's largest code reaches past half the range: the scale is tight
    g = np.abs(d.reshape(64, 18, 32)).max(-1) / fp8_codec.e8m0_to_float64(scales)
    nonzero = g > 0
    assert np.all(g[nonzero] >= 224.0) and np.all(g <= 448.0)
    c2, s2 = fp8_codec.quantise_blocks(d)
    assert np.array_equal(fp8_codec.dequant_blocks(c2, s2), d)


def _workload_query(kv="fp8", seed=3):
    inp = gen.make_inputs(2, 1, [700, 300], kv_dtype=kv, seed=seed)
    rows = mla_oracle.cache_rows(inp.kv_cache.to(torch.float64).numpy() if kv == "bf16" else inp.kv_cache.numpy(), kv)
    return inp, rows


def _split_pins_ok(split) -> bool:
    """Candidate split x -> ((hi codes, scales), (lo codes, scales))."""
    inp, _ = _workload_query()
    q = torch.cat([inp.q_absorbed, inp.q_rope], -1).to(torch.float64).numpy()
    hi, lo = split(q)
    h, l = fp8_codec.dequant_blocks(*hi), fp8_codec.dequant_blocks(*lo)
    if not np.array_equal(h, fp8_codec.dequant_blocks(*fp8_codec.quantise_blocks(q))):
        return False
    r = q - h
    sl = np.repeat(fp8_codec.e8m0_to_float64(lo[1]), 32, axis=-1)
    if not np.all(np.abs(r - l) <= np.maximum(np.abs(r) * 2.0 ** -4, sl * 2.0 ** -10)):
        return False
    # a bf16 query has 8 significant bits: two 4-bit terms hold nearly all of it
    return float(np.mean(h + l == q)) > 0.999


def test_two_term_split_holds_the_bf16_query():
    assert _split_pins_ok(fp8_codec.split_e4m3_terms)


def test_one_term_moves_the_lse_two_terms_do_not():
    """The reading behind a block-scaled score product: one e4m3 term of the
    query moves the LSE far past the 1e-3 bound; two terms stay far inside."""
    for kv in ("bf16", "fp8"):
        inp, rows = _workload_query(kv)
        qa = inp.q_absorbed.to(torch.float64).numpy()
        qr = inp.q_rope.to(torch.float64).numpy()
        bt, sl = inp.block_table.numpy(), inp.seq_lens.numpy()
        _, lse = mla_oracle.mla_decode(qa, qr, rows, bt, sl, inp.scale)
        _, lse1 = mla_oracle.mla_decode(*mla_oracle.query_as_e4m3_terms(qa, qr, terms=1), rows, bt, sl, inp.scale)
        _, lse2 = mla_oracle.mla_decode(*mla_oracle.query_as_e4m3_terms(qa, qr, terms=2), rows, bt, sl, inp.scale)
        assert np.abs(lse1 - lse).max() > 1e-2, kv        # ten times the bound
        assert np.abs(lse2 - lse).max() < 1e-5, kv


def test_planted_mistakes_in_the_encoder_and_split_are_caught():
    good = fp8_codec.float64_to_e4m3fn
    assert _encoder_pins_ok(good)

    def ties_away_from_zero(x):
        x = np.asarray(x, dtype=np.float64)
        a = np.abs(x)
        _, ex = np.frexp(a)
        q = np.exp2(np.maximum(ex - 1, -6) - 3.0)
        return good(np.sign(x) * np.minimum(np.floor(a / q + 0.5) * q, 448.0))

    def truncating(x):
        x = np.asarray(x, dtype=np.float64)
        a = np.abs(x)
        _, ex = np.frexp(a)
        q = np.exp2(np.maximum(ex - 1, -6) - 3.0)
        return good(np.sign(x) * np.floor(a / q) * q)

    def no_subnormals(x):
        x = np.asarray(x, dtype=np.float64)
        return good(np.where(np.abs(x) < 2.0 ** -6, 0.0 * x, x))

    for bad in (ties_away_from_zero, truncating, no_subnormals):
        assert not _encoder_pins_ok(bad), bad.__name__

    assert _split_pins_ok(fp8_codec.split_e4m3_terms)

    def residual_sign_flipped(x):
        hi = fp8_codec.quantise_blocks(x)
        return hi, fp8_codec.quantise_blocks(fp8_codec.dequant_blocks(*hi) - x)

    def scale_one_step_large(x):
        g = x.reshape(x.shape[:-1] + (-1, 32))
        k = fp8_codec.block_scale_exponent(np.abs(g).max(-1)) + 1
        c = fp8_codec.float64_to_e4m3fn(g / np.exp2(k.astype(np.float64))[..., None]).reshape(x.shape)
        hi = (c, (k + 127).astype(np.uint8))
        return hi, fp8_codec.quantise_blocks(x - fp8_codec.dequant_blocks(*hi))

    def hi_only(x):
        hi = fp8_codec.quantise_blocks(x)
        return hi, (np.zeros_like(hi[0]), hi[1])

    for bad in (residual_sign_flipped, scale_one_step_large, hi_only):
        assert not _split_pins_ok(bad), bad.__name__

    # a scale one step too small overflows the e4m3 range: the quantiser refuses
    orig = fp8_codec.block_scale_exponent
    try:
        fp8_codec.block_scale_exponent = lambda amax: orig(amax) - 1
        with pytest.raises(AssertionError):
            fp8_codec.quantise_blocks(np.full((1, 32), 300.0))
    finally:
        fp8_codec.block_scale_exponent = orig
