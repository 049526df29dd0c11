"""Pins of the float64 oracle against things other than itself.

Closed forms printed on the pages, torch's float8 casts, torch's float64
scaled-dot-product attention, the matrix-absorption identity (two independent
computations), brute-force special cases and invariants.  The last test
plants plausible mistakes in copies of the oracle and checks that each is
caught by at least one pin.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import closed_forms as cf
from oracle import fp4_codec, fp8_codec, mla_oracle
from mla_latent_kv_05_gb300 import inputs as gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.txt")


def _golden():
    out = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, value, tol, _where = [x.strip() for x in line.split("|", 3)]
        out[name] = (float(value), float(tol))
    return out


def test_closed_forms_match_printed_values():
    g = _golden()
    computed = {
        "mla_elems_per_token_layer": cf.mla_elems_per_token_layer(),
        "mla_bytes_per_token_61_layers_bf16": cf.mla_bytes_per_token(),
        "mla_kib_per_token_61_layers_bf16": cf.mla_bytes_per_token() / 1024,
        "mla_cache_gb_128k_bf16": cf.mla_cache_bytes() / 1e9,
        "mha_cache_gb_128k_bf16": cf.mha_cache_bytes() / 1e9,
        "mla_reduction_vs_mha_percent": 100 * cf.mla_reduction_vs_mha(),
        "mha_elems_per_token_layer": cf.mha_elems_per_token_layer(),
        "e4m3_max_normal": float(np.nanmax(fp8_codec.e4m3fn_to_float64(np.arange(256, dtype=np.uint8)))),
        "fp8_scales_per_row_group": fp8_codec.SCALE_GROUP,
        "page_block_size": cf.PAGE_SIZE,
        "fp4_row_bytes_512_values": cf.fp4_row_bytes(512),
    }
    assert set(computed) == set(g)
    for k, (v, tol) in g.items():
        assert abs(computed[k] - v) <= tol + 1e-12, (k, computed[k], v)
    # exact integers behind the printed figures
    assert cf.mla_cache_bytes() == 9_210_691_584
    assert cf.mha_cache_bytes() == 523_986_010_112
    assert cf.fp8_row_bytes() == 594 and cf.fp8_page_bytes() == 38_016
    assert cf.fp4_row_bytes() == fp4_codec.ROW_BYTES == 324 and cf.fp4_page_bytes() == 20_736


def test_e4m3_table_matches_torch_cast():
    codes = np.arange(256, dtype=np.uint8)
    mine = fp8_codec.e4m3fn_to_float64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])
    assert np.isnan(mine).sum() == 2           # 0x7F and 0xFF only
    assert mine[0x7E] == 448.0 and mine[0xFE] == -448.0
    assert mine[0x01] == 2.0 ** -9             # smallest subnormal


def test_e8m0_matches_torch_cast():
    codes = np.arange(256, dtype=np.uint8)
    mine = fp8_codec.e8m0_to_float64(codes)
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("torch has no float8_e8m0fnu")
    ref = torch.from_numpy(codes).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])


def test_fp8_row_dequant_layout_against_torch():
    inp = gen.make_inputs(2, 1, [70, 5], kv_dtype="fp8", seed=3)
    raw = inp.kv_cache
    mine = fp8_codec.dequant_rows(raw.numpy())
    v = raw[..., :576].contiguous().view(torch.float8_e4m3fn).to(torch.float64)
    s = raw[..., 576:].contiguous().view(torch.float8_e8m0fnu).to(torch.float64)
    ref = (v * s.repeat_interleave(32, dim=-1)).numpy()
    assert np.array_equal(mine, ref)
    # every dequantised value is exactly representable in bf16
    as_bf16 = torch.from_numpy(mine).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(as_bf16, mine)


def _fp8_pins_ok(decode) -> bool:
    """The 594-byte row against torch's float8 casts, for a candidate decoder."""
    raw = gen.make_inputs(2, 1, [70, 5], kv_dtype="fp8", seed=3).kv_cache
    v = raw[..., :576].contiguous().view(torch.float8_e4m3fn).to(torch.float64)
    s = fp8_codec.e8m0_to_float64(raw[..., 576:].numpy())      # pinned against torch's e8m0 cast above
    ref = v.numpy() * np.repeat(s, 32, axis=-1)
    return np.array_equal(decode(raw.numpy()), ref)


def test_fp8_pins_catch_planted_mistakes():
    good = fp8_codec.dequant_rows
    assert _fp8_pins_ok(good)

    def scales_one_byte_late(raw):
        raw = np.asarray(raw).copy()
        raw[..., 576:] = np.roll(raw[..., 576:], 1, axis=-1)
        return good(raw)

    def scale_per_16(raw):
        raw = np.asarray(raw)
        vals = fp8_codec.e4m3fn_to_float64(raw[..., :576])
        sc = fp8_codec.e8m0_to_float64(raw[..., 576:])
        return vals * sc[..., (np.arange(576) // 16) % 18]

    def e8m0_bias_126(raw):
        return good(raw) * 2.0

    def rope_unscaled(raw):
        out = good(raw)
        out[..., 512:] = fp8_codec.e4m3fn_to_float64(np.asarray(raw)[..., 512:576])
        return out

    for bad in (scales_one_byte_late, scale_per_16, e8m0_bias_126, rope_unscaled):
        assert not _fp8_pins_ok(bad), bad.__name__


def test_v41_row_is_the_printed_528_bytes():
    # "DeepSeek-R1" record, constraint (2): 512 e4m3 values plus 16 e8m0
    # scales, one per 32 values, make the 528-byte V4.1 row
    assert cf.fp8_row_bytes(512) == 528 == fp8_codec.V41_ROW_BYTES
    assert fp8_codec.V41_NUM_SCALES == 16 and fp8_codec.V41_LATENT + 64 == fp8_codec.V41_VALUES


def test_v41_row_layout_by_hand():
    # codes all 1.0 (0x38), scale of group k = 2^(k - 7): value k of the V4.1
    # row is 2^(k//32 - 7); latent values land in dims [0, 448), the RoPE
    # values (the row's last 64) in dims [512, 576), and dims [448, 512) are 0
    row = np.zeros(528, dtype=np.uint8)
    row[:512] = 0x38
    row[512:] = 120 + np.arange(16)
    got = fp8_codec.dequant_rows_v41(row)
    want = np.zeros(576)
    v = 2.0 ** (np.arange(512) // 32 - 7)
    want[:448] = v[:448]
    want[512:] = v[448:]
    assert np.array_equal(got, want)
    assert got[447] == 2.0 ** 6 and got[448] == 0 and got[511] == 0 and got[512] == 2.0 ** 7 and got[575] == 2.0 ** 8


def test_v41_rows_equal_the_594_byte_rows_they_embed_in():
    # a V4.1 row and the 594-byte row with the same latent and RoPE values
    # (zero codes for dims 448..511) decode to the same 576 values
    inp = gen.make_inputs(2, 1, [70, 5], kv_dtype="fp8v41", seed=5)
    raw = inp.kv_cache.numpy()
    wide = np.zeros(raw.shape[:-1] + (594,), dtype=np.uint8)
    wide[..., :448] = raw[..., :448]
    wide[..., 512:576] = raw[..., 448:512]
    wide[..., 576:590] = raw[..., 512:526]          # scales of latent groups 0..13
    wide[..., 590:592] = 127                         # groups 14, 15: zero codes, any scale
    wide[..., 592:594] = raw[..., 526:528]          # scales of the RoPE groups
    assert np.array_equal(fp8_codec.dequant_rows_v41(raw), fp8_codec.dequant_rows(wide))
    # and against torch's own casts of the same bytes
    v = torch.from_numpy(raw[..., :512].copy()).view(torch.float8_e4m3fn).to(torch.float64)
    sc = torch.from_numpy(raw[..., 512:].copy()).view(torch.float8_e8m0fnu).to(torch.float64)
    vals = (v * sc.repeat_interleave(32, dim=-1)).numpy()
    got = fp8_codec.dequant_rows_v41(raw)
    assert np.array_equal(got[..., :448], vals[..., :448]) and np.array_equal(got[..., 512:], vals[..., 448:])
    assert not got[..., 448:512].any()


def test_fp4_v41_row_is_the_printed_288_bytes():
    # the record's FP4 variant: 288 bytes per token for the 512-value row
    assert cf.fp4_row_bytes(512) == 288 == fp4_codec.V41_ROW_BYTES


def test_fp4_v41_row_layout_by_hand():
    # code bytes 0x22 (both nibbles 1.0), scale of group k (16 values) =
    # 2^(k - 10): value k of the row is 2^(k//16 - 10); latent values in dims
    # [0, 448), RoPE values (the row's last 64) in [512, 576), zeros between
    row = np.zeros(288, dtype=np.uint8)
    row[:256] = 0x22
    row[256:] = 117 + np.arange(32)
    got = fp4_codec.dequant_rows_v41(row)
    v = 2.0 ** (np.arange(512) // 16 - 10)
    want = np.zeros(576)
    want[:448] = v[:448]
    want[512:] = v[448:]
    assert np.array_equal(got, want)
    assert got[447] == 2.0 ** 17 and not got[448:512].any() and got[512] == 2.0 ** 18 and got[575] == 2.0 ** 21


def test_fp4_v41_rows_equal_the_324_byte_rows_they_embed_in():
    inp = gen.make_inputs(2, 1, [70, 5], kv_dtype="fp4v41", seed=6)
    raw = inp.kv_cache.numpy()
    wide = np.zeros(raw.shape[:-1] + (324,), dtype=np.uint8)
    wide[..., :224] = raw[..., :224]                 # latent codes (values 0..447)
    wide[..., 256:288] = raw[..., 224:256]           # RoPE codes (values 512..575)
    wide[..., 288:316] = raw[..., 256:284]           # latent scales (groups 0..27)
    wide[..., 316:320] = 127                         # groups 28..31: zero codes, any scale
    wide[..., 320:324] = raw[..., 284:288]           # RoPE scales
    assert np.array_equal(fp4_codec.dequant_rows_v41(raw), fp4_codec.dequant_rows(wide))


def _v41_fp8_pins_ok(decode) -> bool:
    """The 528-byte row's hand-built pin and its 594-byte embedding, for a
    candidate decoder [..., 528] -> [..., 576]."""
    row = np.zeros(528, dtype=np.uint8)
    row[:512] = 0x38
    row[512:] = 120 + np.arange(16)
    v = 2.0 ** (np.arange(512) // 32 - 7)
    want = np.zeros(576)
    want[:448], want[512:] = v[:448], v[448:]
    if not np.array_equal(decode(row), want):
        return False
    raw = gen.make_inputs(2, 1, [70, 5], kv_dtype="fp8v41", seed=5).kv_cache.numpy()
    wide = np.zeros(raw.shape[:-1] + (594,), dtype=np.uint8)
    wide[..., :448], wide[..., 512:576] = raw[..., :448], raw[..., 448:512]
    wide[..., 576:590], wide[..., 590:592], wide[..., 592:594] = raw[..., 512:526], 127, raw[..., 526:528]
    return np.array_equal(decode(raw), fp8_codec.dequant_rows(wide))


def test_v41_pins_catch_planted_mistakes():
    good = fp8_codec.dequant_rows_v41
    assert _v41_fp8_pins_ok(good)

    def scales_one_group_late(raw):
        raw = np.asarray(raw).copy()
        raw[..., 512:] = np.roll(raw[..., 512:], 1, axis=-1)
        return good(raw)

    def rope_in_the_padding(raw):
        out = good(raw)
        fixed = out.copy()
        fixed[..., 448:512], fixed[..., 512:] = out[..., 512:], 0
        return fixed

    def padding_not_zero(raw):
        out = good(raw)
        out[..., 448:512] = out[..., 512:]
        return out

    for bad in (scales_one_group_late, rope_in_the_padding, padding_not_zero):
        assert not _v41_fp8_pins_ok(bad), bad.__name__


def _v41_fp4_pins_ok(decode) -> bool:
    """The 288-byte row's hand-built pin and its 324-byte embedding, for a
    candidate decoder [..., 288] -> [..., 576]."""
    row = np.zeros(288, dtype=np.uint8)
    row[:256] = 0x22
    row[256:] = 117 + np.arange(32)
    v = 2.0 ** (np.arange(512) // 16 - 10)
    want = np.zeros(576)
    want[:448], want[512:] = v[:448], v[448:]
    if not np.array_equal(decode(row), want):
        return False
    raw = gen.make_inputs(2, 1, [70, 5], kv_dtype="fp4v41", seed=6).kv_cache.numpy()
    wide = np.zeros(raw.shape[:-1] + (324,), dtype=np.uint8)
    wide[..., :224], wide[..., 256:288] = raw[..., :224], raw[..., 224:256]
    wide[..., 288:316], wide[..., 316:320], wide[..., 320:324] = raw[..., 256:284], 127, raw[..., 284:288]
    return np.array_equal(decode(raw), fp4_codec.dequant_rows(wide))


def test_fp4_v41_pins_catch_planted_mistakes():
    good = fp4_codec.dequant_rows_v41
    assert _v41_fp4_pins_ok(good)

    def scales_one_group_late(raw):
        raw = np.asarray(raw).copy()
        raw[..., 256:] = np.roll(raw[..., 256:], 1, axis=-1)
        return good(raw)

    def rope_in_the_padding(raw):
        out = good(raw)
        fixed = out.copy()
        fixed[..., 448:512], fixed[..., 512:] = out[..., 512:], 0
        return fixed

    def nibbles_swapped(raw):
        raw = np.asarray(raw).copy()
        raw[..., :256] = ((raw[..., :256] & 0x0F) << 4) | (raw[..., :256] >> 4)
        return good(raw)

    for bad in (scales_one_group_late, rope_in_the_padding, nibbles_swapped):
        assert not _v41_fp4_pins_ok(bad), bad.__name__


def test_e2m1_table_is_the_ocp_value_set():
    # OCP MX FP4 E2M1: the eight magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 in
    # code order, the sign bit negating them; no NaN or infinity
    v = fp4_codec.e2m1_to_float64(np.arange(16))
    assert list(v[:8]) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert np.array_equal(v[8:], -v[:8])
    assert np.signbit(v[8]) and not np.signbit(v[0])
    assert np.all(np.isfinite(v))


def test_fp4_row_layout_by_hand():
    row = np.zeros(324, dtype=np.uint8)
    row[0] = 0x21          # value 0: code 1 (0.5), value 1: code 2 (1.0)
    row[7] = 0xF7          # value 14: code 7 (6), value 15: code 15 (-6)
    row[8] = 0x3B          # value 16: code 11 (-1.5), value 17: code 3 (1.5)
    row[287] = 0x5C        # value 574: code 12 (-2), value 575: code 5 (3)
    row[288] = 127         # scale of values 0..15: 1
    row[289] = 130         # values 16..31: 8
    row[323] = 125         # values 560..575: 1/4
    v = fp4_codec.dequant_rows(row)
    assert v.shape == (576,)
    assert (v[0], v[1], v[14], v[15]) == (0.5, 1.0, 6.0, -6.0)
    assert (v[16], v[17]) == (-12.0, 12.0)
    assert (v[574], v[575]) == (-0.5, 0.75)
    assert np.count_nonzero(v) == 8


def test_fp4_value_k_takes_scale_k_div_16():
    # every code 2 (= 1.0), so each value is its scale: 2^(byte - 127)
    inp = gen.make_inputs(1, 1, [64], kv_dtype="fp4", seed=9)
    raw = inp.kv_cache.numpy().copy()
    raw[..., :288] = 0x22
    v = fp4_codec.dequant_rows(raw)
    sc = raw[..., 288:].astype(np.int64)
    for k in (0, 15, 16, 31, 100, 511, 512, 575):
        assert np.array_equal(v[..., k], np.exp2(sc[..., k // 16] - 127.0)), k


def _fp4_pins_ok(decode) -> bool:
    """The by-hand 324-byte row and the per-16 scale rule, for a candidate
    decoder [..., 324] -> [..., 576]."""
    row = np.zeros(324, dtype=np.uint8)
    row[0], row[7], row[8], row[287] = 0x21, 0xF7, 0x3B, 0x5C
    row[288], row[289], row[323] = 127, 130, 125
    v = decode(row)
    if not ((v[0], v[1], v[14], v[15], v[16], v[17], v[574], v[575]) ==
            (0.5, 1.0, 6.0, -6.0, -12.0, 12.0, -0.5, 0.75) and np.count_nonzero(v) == 8):
        return False
    raw = gen.make_inputs(1, 1, [64], kv_dtype="fp4", seed=9).kv_cache.numpy().copy()
    raw[..., :288] = 0x22
    v = decode(raw)
    sc = raw[..., 288:].astype(np.int64)
    return all(np.array_equal(v[..., k], np.exp2(sc[..., k // 16] - 127.0)) for k in range(576))


def test_fp4_pins_catch_planted_mistakes():
    good = fp4_codec.dequant_rows
    assert _fp4_pins_ok(good)

    def nibbles_swapped(raw):
        raw = np.asarray(raw).copy()
        raw[..., :288] = ((raw[..., :288] & 0x0F) << 4) | (raw[..., :288] >> 4)
        return good(raw)

    def one_scale_per_32(raw):
        raw = np.asarray(raw).copy()
        raw[..., 288:] = np.repeat(raw[..., 288:306], 2, axis=-1)
        return good(raw)

    def scales_one_byte_late(raw):
        raw = np.asarray(raw).copy()
        raw[..., 288:] = np.roll(raw[..., 288:], 1, axis=-1)
        return good(raw)

    def sign_dropped(raw):
        return np.abs(good(raw))

    for bad in (nibbles_swapped, one_scale_per_32, scales_one_byte_late, sign_dropped):
        assert not _fp4_pins_ok(bad), bad.__name__


def test_fp4_generated_rows_are_bf16_exact():
    inp = gen.make_inputs(2, 1, [70, 5], kv_dtype="fp4", seed=3)
    assert inp.kv_cache.shape[-1] == 324
    v = fp4_codec.dequant_rows(inp.kv_cache.numpy())
    as_bf16 = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(as_bf16, v)
    # both nibbles carry all sixteen codes somewhere
    codes = fp4_codec.unpack_codes(inp.kv_cache.numpy()[..., :288])
    assert set(np.unique(codes[..., 0::2])) == set(range(16)) == set(np.unique(codes[..., 1::2]))


def _f64(t):
    return t.to(torch.float64).numpy()


def _sdpa_reference(q_abs, q_rope, rows, scale):
    """torch's float64 SDPA on the gathered dense keys; lse by torch.logsumexp."""
    q = torch.cat([torch.from_numpy(q_abs), torch.from_numpy(q_rope)], -1)[None, :, None, :]  # [1, H, 1, 576]
    k = torch.from_numpy(rows)[None, None, :, :].expand(1, q.shape[1], -1, -1)
    v = torch.from_numpy(rows[:, :512])[None, None, :, :].expand(1, q.shape[1], -1, -1)
    out = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=scale)
    lse = torch.logsumexp(scale * (q @ k.transpose(-1, -2)), dim=-1)
    return out[0, :, 0].numpy(), lse[0, :, 0].numpy()


def _gathered(inp, b, i=0):
    rows = mla_oracle.cache_rows(_f64(inp.kv_cache) if inp.kv_dtype == "bf16" else inp.kv_cache.numpy(), inp.kv_dtype)
    n = max(mla_oracle.visible_len(int(inp.seq_lens[b]), inp.sq, i), 0)
    return mla_oracle.gather_rows(rows, inp.block_table[b].numpy(), n)


@pytest.mark.parametrize("seq,kv", [([256], "bf16"), ([1, 63, 64, 65, 200], "bf16"), ([130, 7], "fp8"),
                                    ([130, 7], "fp4")])
def test_attend_matches_torch_sdpa(seq, kv):
    inp = gen.make_inputs(len(seq), 1, seq, kv_dtype=kv, seed=11)
    for b in range(len(seq)):
        g = _gathered(inp, b)
        out, lse = mla_oracle.attend_latent(_f64(inp.q_absorbed[b, 0]), _f64(inp.q_rope[b, 0]), g, inp.scale)
        ro, rl = _sdpa_reference(_f64(inp.q_absorbed[b, 0]), _f64(inp.q_rope[b, 0]), g, inp.scale)
        np.testing.assert_allclose(out, ro, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(lse, rl, rtol=1e-12, atol=1e-12)


def test_workload1_matches_sdpa():
    inp = gen.make_workload(1)
    assert inp.num_pages == 8 and inp.max_pages == 4 and int(inp.seq_lens[0]) == 256
    rows = mla_oracle.cache_rows(_f64(inp.kv_cache), "bf16")
    out, lse = mla_oracle.mla_decode(_f64(inp.q_absorbed), _f64(inp.q_rope), rows,
                                     inp.block_table.numpy(), inp.seq_lens.numpy(), inp.scale)
    ro, rl = _sdpa_reference(_f64(inp.q_absorbed[0, 0]), _f64(inp.q_rope[0, 0]), _gathered(inp, 0), inp.scale)
    np.testing.assert_allclose(out[0, 0], ro, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], rl, rtol=1e-12)


def test_absorption_identity():
    """Un-absorbed attention with explicit W^UK / W^UV equals the absorbed
    latent form followed by W^UV (architecture guide, section 1.1)."""
    rng = np.random.default_rng(5)
    H, d_h, n = 16, 128, 97
    w_uk = rng.standard_normal((H, d_h, 512)) / math.sqrt(512)
    w_uv = rng.standard_normal((H, d_h, 512)) / math.sqrt(512)
    q_nope = rng.standard_normal((H, d_h))
    q_rope = rng.standard_normal((H, 64))
    c_kv = rng.standard_normal((n, 512))
    k_r = rng.standard_normal((n, 64))
    scale = 1 / math.sqrt(192)
    o_ref, lse_ref = mla_oracle.attend_unabsorbed(q_nope, q_rope, c_kv, k_r, w_uk, w_uv, scale)
    q_abs = mla_oracle.absorb_query(q_nope, w_uk)
    out_lat, lse = mla_oracle.attend_latent(q_abs, q_rope, np.concatenate([c_kv, k_r], 1), scale)
    o = mla_oracle.up_project_output(out_lat, w_uv)
    np.testing.assert_allclose(o, o_ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12)


def _absorption_ok(attend_unabsorbed, up_project) -> bool:
    """The absorption identity for candidate un-absorbed attention and
    up-projection, against the SDPA-pinned latent form."""
    rng = np.random.default_rng(15)
    H, d_h, n = 8, 128, 61
    w_uk = rng.standard_normal((H, d_h, 512)) / math.sqrt(512)
    w_uv = rng.standard_normal((H, d_h, 512)) / math.sqrt(512)
    q_nope, q_rope = rng.standard_normal((H, d_h)), rng.standard_normal((H, 64))
    c_kv, k_r = rng.standard_normal((n, 512)), rng.standard_normal((n, 64))
    scale = 1 / math.sqrt(192)
    try:
        o_ref, lse_ref = attend_unabsorbed(q_nope, q_rope, c_kv, k_r, w_uk, w_uv, scale)
        out_lat, lse = mla_oracle.attend_latent(mla_oracle.absorb_query(q_nope, w_uk), q_rope,
                                                np.concatenate([c_kv, k_r], 1), scale)
        o = up_project(out_lat, w_uv)
    except (ValueError, IndexError):
        return False
    return bool(np.allclose(o, o_ref, rtol=1e-10, atol=1e-12) and np.allclose(lse, lse_ref, rtol=1e-12))


def test_absorption_pins_catch_planted_mistakes():
    good_attend, good_up = mla_oracle.attend_unabsorbed, mla_oracle.up_project_output
    assert _absorption_ok(good_attend, good_up)

    def values_through_w_uk(q_nope, q_rope, c_kv, k_r, w_uk, w_uv, scale):
        return good_attend(q_nope, q_rope, c_kv, k_r, w_uk, w_uk, scale)

    def rope_dropped(q_nope, q_rope, c_kv, k_r, w_uk, w_uv, scale):
        return good_attend(q_nope, np.zeros_like(q_rope), c_kv, k_r, w_uk, w_uv, scale)

    def heads_shifted(q_nope, q_rope, c_kv, k_r, w_uk, w_uv, scale):
        return good_attend(q_nope, q_rope, c_kv, k_r, w_uk, np.roll(w_uv, 1, axis=0), scale)

    for bad in (values_through_w_uk, rope_dropped, heads_shifted):
        assert not _absorption_ok(bad, good_up), bad.__name__

    def up_transposed(out_lat, w_uv):
        return np.einsum("hck,hc->hk", w_uv.transpose(0, 2, 1), out_lat[:, :128])

    def up_first_head_only(out_lat, w_uv):
        return np.einsum("kc,hc->hk", w_uv[0], out_lat)

    for bad in (up_transposed, up_first_head_only):
        assert not _absorption_ok(good_attend, bad), bad.__name__


def test_single_token_is_exact_row():
    rng = np.random.default_rng(1)
    row = rng.standard_normal((1, 576))
    qa, qr = rng.standard_normal((128, 512)), rng.standard_normal((128, 64))
    out, lse = mla_oracle.attend_latent(qa, qr, row, 0.1)
    assert np.array_equal(out, np.broadcast_to(row[0, :512], (128, 512)))
    np.testing.assert_allclose(lse, 0.1 * (qa @ row[0, :512] + qr @ row[0, 512:]), rtol=1e-13)


def test_identical_rows_mean_and_log_n():
    rng = np.random.default_rng(2)
    row = rng.standard_normal(576)
    n = 37
    rows = np.tile(row, (n, 1))
    qa, qr = rng.standard_normal((128, 512)), rng.standard_normal((128, 64))
    out, lse = mla_oracle.attend_latent(qa, qr, rows, 0.05)
    np.testing.assert_allclose(out, np.broadcast_to(row[:512], (128, 512)), rtol=1e-13, atol=1e-14)
    s = 0.05 * (qa @ row[:512] + qr @ row[512:])
    np.testing.assert_allclose(lse, s + math.log(n), rtol=1e-13)


def test_dominant_score_selects_row():
    rng = np.random.default_rng(3)
    rows = rng.standard_normal((20, 576)) * 0.01
    qa = np.zeros((1, 512)); qr = np.zeros((1, 64))
    qa[0, 7] = 1.0
    rows[13, 7] = 50.0
    out, _ = mla_oracle.attend_latent(qa, qr, rows, 1.0)
    np.testing.assert_allclose(out[0], rows[13, :512], atol=1e-15 * 1e6)


def test_page_permutation_invariance_and_unused_slots():
    inp = gen.make_inputs(3, 1, [100, 64, 129], seed=8, physical_pages=9)
    rows = mla_oracle.cache_rows(_f64(inp.kv_cache), "bf16")
    qa, qr = _f64(inp.q_absorbed), _f64(inp.q_rope)
    bt, sl = inp.block_table.numpy(), inp.seq_lens.numpy()
    out, lse = mla_oracle.mla_decode(qa, qr, rows, bt, sl, inp.scale)
    perm = np.random.default_rng(0).permutation(rows.shape[0])
    inv = np.argsort(perm)
    rows2 = rows[perm].copy()
    bt2 = np.where(bt >= 0, inv[np.maximum(bt, 0)], -1)
    # slots past the visible length hold garbage, which must not matter
    for b, s in enumerate(sl):
        if s % 64:
            rows2[bt2[b, s // 64], s % 64:] = np.nan
    out2, lse2 = mla_oracle.mla_decode(qa, qr, rows2, bt2, sl, inp.scale)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(lse, lse2)


def test_split_merge_equals_unsplit():
    rng = np.random.default_rng(4)
    rows = rng.standard_normal((300, 576))
    qa, qr = rng.standard_normal((128, 512)), rng.standard_normal((128, 64))
    full, lse_full = mla_oracle.attend_latent(qa, qr, rows, 0.07)
    for cuts in ([0, 150, 300], [0, 1, 64, 65, 299, 300], [0, 299, 300]):
        parts = [mla_oracle.attend_latent(qa, qr, rows[a:b], 0.07) for a, b in zip(cuts[:-1], cuts[1:])]
        o, l = mla_oracle.merge_partials(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
        np.testing.assert_allclose(o, full, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(l, lse_full, rtol=1e-13)
    # an empty part (lse = -inf) contributes nothing
    e = mla_oracle.attend_latent(qa, qr, rows[:0], 0.07)
    o, l = mla_oracle.merge_partials(np.stack([full, e[0]]), np.stack([lse_full, e[1]]))
    np.testing.assert_allclose(o, full, rtol=1e-13)


def _merge_pins_ok(merge) -> bool:
    """Split + merge reproduces the unsplit attention, and an all-empty row
    merges to 0 and -inf, for a candidate merge (outs [k,H,D], lses [k,H])."""
    rng = np.random.default_rng(4)
    rows = rng.standard_normal((300, 576))
    qa, qr = rng.standard_normal((16, 512)), rng.standard_normal((16, 64))
    full, lse_full = mla_oracle.attend_latent(qa, qr, rows, 0.07)
    cuts = [0, 1, 64, 65, 299, 300]
    parts = [mla_oracle.attend_latent(qa, qr, rows[a:b], 0.07) for a, b in zip(cuts[:-1], cuts[1:])]
    with np.errstate(all="ignore"):
        o, l = merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
        if not (np.allclose(o, full, rtol=1e-10, atol=1e-12) and np.allclose(l, lse_full, rtol=1e-12)):
            return False
        e = mla_oracle.attend_latent(qa, qr, rows[:0], 0.07)
        o, l = merge(np.stack([e[0], e[0]]), np.stack([e[1], e[1]]))
    return bool(np.all(o == 0) and np.all(np.isneginf(l)))


def test_merge_pins_catch_planted_mistakes():
    good = mla_oracle.merge_partials
    assert _merge_pins_ok(good)

    def base2_lse(outs, lses):
        o, l = good(outs, lses)
        return o, np.logaddexp2.reduce(np.asarray(lses), axis=0)

    def plain_average(outs, lses):
        o, l = good(outs, lses)
        return np.mean(np.asarray(outs), axis=0), l

    def weights_not_normalised(outs, lses):
        lses = np.asarray(lses)
        return np.einsum("kh,khd->hd", np.exp(lses), np.asarray(outs)), np.logaddexp.reduce(lses, axis=0)

    def empty_row_nan(outs, lses):
        lses = np.asarray(lses)
        L = np.logaddexp.reduce(lses, axis=0)
        return np.einsum("kh,khd->hd", np.exp(lses - L), np.asarray(outs)), L

    for bad in (base2_lse, plain_average, weights_not_normalised, empty_row_nan):
        assert not _merge_pins_ok(bad), bad.__name__


def test_causal_two_token_query():
    inp = gen.make_inputs(2, 2, [65, 1], seed=9)
    rows = mla_oracle.cache_rows(_f64(inp.kv_cache), "bf16")
    qa, qr = _f64(inp.q_absorbed), _f64(inp.q_rope)
    out, lse = mla_oracle.mla_decode(qa, qr, rows, inp.block_table.numpy(), inp.seq_lens.numpy(), inp.scale)
    for b, s in enumerate([65, 1]):
        for i, n in enumerate([s - 1, s]):
            g = mla_oracle.gather_rows(rows, inp.block_table[b].numpy(), n)
            if n == 0:
                assert np.all(out[b, i] == 0) and np.all(lse[b, i] == -np.inf)
                continue
            ro, rl = _sdpa_reference(qa[b, i], qr[b, i], g, inp.scale)
            np.testing.assert_allclose(out[b, i], ro, rtol=1e-11, atol=1e-12)
            np.testing.assert_allclose(lse[b, i], rl, rtol=1e-12)


def _causal_pin_ok() -> bool:
    """Sq = 2 and 3 query blocks: query i sees seq_len - (Sq-1-i) tokens,
    counted here by hand, each row checked against torch's SDPA."""
    for sq, lens in ((2, [65, 1]), (3, [130, 2])):
        inp = gen.make_inputs(2, sq, lens, seed=9)
        rows = mla_oracle.cache_rows(_f64(inp.kv_cache), "bf16")
        qa, qr = _f64(inp.q_absorbed), _f64(inp.q_rope)
        out, lse = mla_oracle.mla_decode(qa, qr, rows, inp.block_table.numpy(), inp.seq_lens.numpy(), inp.scale)
        for b, s in enumerate(lens):
            for i in range(sq):
                n = max(s - (sq - 1 - i), 0)
                if n == 0:
                    if not (np.all(out[b, i] == 0) and np.all(lse[b, i] == -np.inf)):
                        return False
                    continue
                g = mla_oracle.gather_rows(rows, inp.block_table[b].numpy(), n)
                ro, rl = _sdpa_reference(qa[b, i], qr[b, i], g, inp.scale)
                if not (np.allclose(out[b, i], ro, rtol=1e-11, atol=1e-12) and np.allclose(lse[b, i], rl, rtol=1e-12)):
                    return False
    return True


def test_causal_pin_catches_planted_mistakes(monkeypatch):
    assert _causal_pin_ok()
    for bad in (lambda s, sq, i: int(s) - (int(sq) - int(i)),      # one token short everywhere
                lambda s, sq, i: int(s) - int(i),                   # the query order reversed
                lambda s, sq, i: int(s)):                           # no causal rule
        monkeypatch.setattr(mla_oracle, "visible_len", bad)
        assert not _causal_pin_ok()
    monkeypatch.undo()
    assert _causal_pin_ok()


def _pin_suite(attend):
    """Run the attention pins against a candidate implementation; return the
    number of pins that fail."""
    fails = 0
    rng = np.random.default_rng(12)
    rows = rng.standard_normal((70, 576))
    qa, qr = rng.standard_normal((8, 512)), rng.standard_normal((8, 64))
    try:
        o, l = attend(qa, qr, rows, 0.07)
        ro, rl = _sdpa_reference(qa, qr, rows, 0.07)
        if not (np.allclose(o, ro, rtol=1e-10) and np.allclose(l, rl, rtol=1e-10)):
            fails += 1
    except Exception:
        fails += 1
    o, l = attend(qa, qr, rows[:1], 0.07)
    if not np.allclose(o, np.broadcast_to(rows[0, :512], o.shape)):
        fails += 1
    return fails


def test_planted_mistakes_are_caught():
    good = mla_oracle.attend_latent

    def no_rope(qa, qr, rows, sc):
        return good(qa, np.zeros_like(qr), rows, sc)

    def scale_outside(qa, qr, rows, sc):
        o, l = good(qa, qr, rows, 1.0)
        return o, l * sc

    def v_includes_rope_slice(qa, qr, rows, sc):
        shifted = np.concatenate([rows[:, 64:], rows[:, :64]], 1)
        o, l = good(qa, qr, rows, sc)
        o2, _ = good(qa, qr, shifted, sc)
        return o2, l

    def off_by_one_len(qa, qr, rows, sc):
        return good(qa, qr, rows[:-1] if rows.shape[0] > 1 else rows, sc)

    assert _pin_suite(good) == 0
    for bad in (no_rope, scale_outside, v_includes_rope_slice, off_by_one_len):
        assert _pin_suite(bad) >= 1, bad.__name__

    # a wrong page or slot index is caught by the marker pin
    def bad_gather(rows, btr, n):
        j = np.arange(int(n))
        return rows[np.asarray(btr)[j // rows.shape[1]], (j + 1) % rows.shape[1]]

    assert _marker_gather_ok(mla_oracle.gather_rows)
    assert not _marker_gather_ok(bad_gather)


def _marker_gather_ok(gather):
    """Fill every physical slot with the token index the block table says it
    holds (and -1 in unused slots); gathering must return 0, 1, ..., n-1."""
    inp = gen.make_inputs(3, 1, [100, 64, 129], seed=8, physical_pages=9)
    bt, sl = inp.block_table.numpy(), inp.seq_lens.numpy()
    rows = np.full((inp.num_pages, 64, 576), -1.0)
    for b, s in enumerate(sl):
        for j in range(s):
            rows[bt[b, j // 64], j % 64, :] = j
    for b, s in enumerate(sl):
        g = gather(rows, bt[b], s)
        if not np.array_equal(g[:, 0], np.arange(s)) or not np.all(g == g[:, :1]):
            return False
    return True


def test_gather_by_markers():
    assert _marker_gather_ok(mla_oracle.gather_rows)


# ----------------------------------------------------------------- sparse top-k
def _context_slots(bt_row, n, page=64):
    """Cache slots of the first n tokens of a row (block-table order)."""
    j = np.arange(n)
    return np.asarray(bt_row, dtype=np.int64)[j // page] * page + j % page


def test_sparse_listing_the_visible_context_equals_dense_decode():
    # Listing exactly the tokens a dense query sees (any order, -1 padded)
    # must reproduce the dense decode, which is pinned to torch's SDPA above.
    inp = gen.make_inputs(3, 2, [70, 1, 200], seed=21)
    rows = mla_oracle.cache_rows(_f64(inp.kv_cache), "bf16")
    qa, qr = _f64(inp.q_absorbed), _f64(inp.q_rope)
    bt, sl = inp.block_table.numpy(), inp.seq_lens.numpy()
    out, lse = mla_oracle.mla_decode(qa, qr, rows, bt, sl, inp.scale)
    topk = 256
    slots = np.full((3, 2, topk), -1, dtype=np.int64)
    rng = np.random.default_rng(5)
    for b in range(3):
        for i in range(2):
            n = max(int(sl[b]) - (2 - 1 - i), 0)
            s = _context_slots(bt[b], n)
            slots[b, i, :n] = s
            slots[b, i] = rng.permutation(slots[b, i])
    out2, lse2 = mla_oracle.mla_decode_sparse(qa, qr, rows, slots, inp.scale)
    fin = np.isfinite(lse)
    np.testing.assert_allclose(out2, out, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(lse2[fin], lse[fin], rtol=1e-13)
    assert np.all(np.isneginf(lse2[~fin])) and np.all(out2[~fin] == 0)


def test_sparse_order_padding_and_split_invariance():
    inp = gen.make_sparse_inputs(2, 1, [500, 130], 96, seed=22, pad_middle=True)
    d = inp.dense
    rows = mla_oracle.cache_rows(_f64(d.kv_cache), "bf16")
    qa, qr = _f64(d.q_absorbed), _f64(d.q_rope)
    slots = inp.token_slots.numpy()
    out, lse = mla_oracle.mla_decode_sparse(qa, qr, rows, slots, d.scale)
    rng = np.random.default_rng(6)
    perm = np.stack([[rng.permutation(slots[b, 0])] for b in range(2)])
    out2, lse2 = mla_oracle.mla_decode_sparse(qa, qr, rows, perm, d.scale)
    np.testing.assert_allclose(out2, out, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse2, lse, rtol=1e-14)
    # two halves of the list merged by the LSE rule equal the whole list
    for b in range(2):
        h = slots.shape[-1] // 2
        parts = [mla_oracle.mla_decode_sparse(qa[b:b + 1], qr[b:b + 1], rows, slots[b:b + 1, :, a:e], d.scale)
                 for a, e in ((0, h), (h, slots.shape[-1]))]
        o, l = mla_oracle.merge_partials(np.stack([p[0][0, 0] for p in parts]), np.stack([p[1][0, 0] for p in parts]))
        np.testing.assert_allclose(o, out[b, 0], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(l, lse[b, 0], rtol=1e-13)


def test_sparse_duplicates_count_twice_and_minus_one_is_skipped():
    # Two tokens A, B; the list [A, -1, A, B] gives weights 2 e^sA : e^sB.
    rng = np.random.default_rng(7)
    rows = rng.standard_normal((1, 64, 576))
    qa, qr = rng.standard_normal((1, 1, 2, 512)), rng.standard_normal((1, 1, 2, 64))
    A, B, scale = 5, 17, 0.05
    out, lse = mla_oracle.mla_decode_sparse(qa, qr, rows, np.array([[[A, -1, A, B]]]), scale)
    for h in range(2):
        sa = scale * (qa[0, 0, h] @ rows[0, A, :512] + qr[0, 0, h] @ rows[0, A, 512:])
        sb = scale * (qa[0, 0, h] @ rows[0, B, :512] + qr[0, 0, h] @ rows[0, B, 512:])
        z = 2 * math.exp(sa) + math.exp(sb)
        want = (2 * math.exp(sa) * rows[0, A, :512] + math.exp(sb) * rows[0, B, :512]) / z
        np.testing.assert_allclose(out[0, 0, h], want, rtol=1e-12, atol=1e-14)
        assert abs(lse[0, 0, h] - math.log(z)) < 1e-12
    out, lse = mla_oracle.mla_decode_sparse(qa, qr, rows, np.full((1, 1, 8), -1), scale)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def _sparse_marker_gather_ok(gather):
    """Fill every cache slot with its own slot number; gathering a list must
    return exactly the listed slots, in order, without the -1 entries."""
    rows = np.arange(5 * 64, dtype=np.float64).reshape(5, 64, 1) * np.ones((1, 1, 576))
    rng = np.random.default_rng(8)
    for _ in range(20):
        lst = rng.integers(0, 5 * 64, size=37)
        lst[rng.integers(0, 37, size=5)] = -1
        g = gather(rows, lst)
        want = lst[lst >= 0]
        if g.shape[0] != want.size or not np.array_equal(g[:, 0], want) or not np.all(g == g[:, :1]):
            return False
    return True


def test_sparse_gather_by_markers_catches_planted_mistakes():
    assert _sparse_marker_gather_ok(mla_oracle.sparse_gather_rows)

    def keeps_minus_one(rows, slots):        # -1 read as the last slot
        return rows.reshape(-1, rows.shape[-1])[np.asarray(slots, dtype=np.int64)]

    def sorted_slots(rows, slots):           # order lost (harmless for attention, caught here)
        s = np.sort(np.asarray(slots, dtype=np.int64))
        return rows.reshape(-1, rows.shape[-1])[s[s >= 0]]

    def page_major_swap(rows, slots):        # slot read as offset * pages + page
        s = np.asarray(slots, dtype=np.int64)
        s = s[s >= 0]
        return rows[s % rows.shape[0], s // rows.shape[0]]

    for bad in (keeps_minus_one, sorted_slots, page_major_swap):
        assert not _sparse_marker_gather_ok(bad), bad.__name__
