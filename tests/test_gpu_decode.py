"""GPU parity of the CUDA decode path (through the C ABI) against the float64
oracle, on small seeded problems that span several tiles, ragged tails,
split-KV, multi-token causal queries and the degenerate cases.

Bounds: max|out - ref| <= 1e-2 * max|ref| and max|lse - ref| <= 1e-3;
bit-exact where the result is a copy (one visible token).
"""
import math

import numpy as np
import pytest
import torch

from mla_latent_kv_05_gb300 import binding
from mla_latent_kv_05_gb300 import inputs as gen
from oracle import fp4_codec, mla_oracle

pytestmark = pytest.mark.gpu

OUT_RTOL = 1e-2
LSE_ATOL = 1e-3


def to_dev(inp, dev="cuda"):
    return dict(q=inp.q_absorbed.to(dev), qr=inp.q_rope.to(dev), kv=inp.kv_cache.to(dev),
                bt=inp.block_table.to(dev), sl=inp.seq_lens.to(dev))


def run_gpu(inp, d=None):
    d = d or to_dev(inp)
    ws = binding.alloc_workspace(inp.batch, inp.sq)
    fn = {"bf16": binding.mla_decode_bf16, "fp8": binding.mla_decode_fp8, "fp4": binding.mla_decode_fp4,
          "fp8v41": binding.mla_decode_fp8_v41, "fp4v41": binding.mla_decode_fp4_v41}[inp.kv_dtype]
    out, lse = fn(d["q"], d["qr"], d["kv"], d["bt"], d["sl"], inp.scale, workspace=ws)
    st = binding.mla_get_status(ws)
    return out, lse, st


def oracle(inp, query_rows=None):
    raw = inp.kv_cache.double().numpy() if inp.kv_dtype == "bf16" else inp.kv_cache.numpy()
    rows = mla_oracle.cache_rows(raw, inp.kv_dtype)
    return mla_oracle.mla_decode(inp.q_absorbed.double().numpy(), inp.q_rope.double().numpy(), rows,
                                 inp.block_table.numpy(), inp.seq_lens.numpy(), inp.scale, query_rows)


def assert_close(out, lse, ref_out, ref_lse, query_rows=None):
    got = out.double().cpu().numpy()
    gl = lse.double().cpu().numpy()
    if query_rows is None:
        query_rows = [(b, i) for b in range(got.shape[0]) for i in range(got.shape[1])]
    for b, i in query_rows:
        r, rl = ref_out[b, i], ref_lse[b, i]
        if np.all(np.isneginf(rl)):
            assert np.all(got[b, i] == 0), (b, i)
            assert np.all(np.isneginf(gl[b, i])), (b, i)
            continue
        err = np.abs(got[b, i] - r).max()
        bound = OUT_RTOL * np.abs(r).max()
        assert err <= bound, f"row ({b},{i}): max|dout| {err:.3e} > {bound:.3e}"
        lerr = np.abs(gl[b, i] - rl).max()
        assert lerr <= LSE_ATOL, f"row ({b},{i}): max|dlse| {lerr:.3e}"


def test_workload1_oracle_sized(cuda_device):
    inp = gen.make_workload(1)
    out, lse, st = run_gpu(inp)
    assert st == 0
    assert_close(out, lse, *oracle(inp))


@pytest.mark.parametrize("lens", [
    [1, 2, 63, 64, 65, 127, 128, 129],
    [95, 96, 97, 191, 192, 193, 288],   # the 96-token score-tile edges
    [1000, 4097, 3, 700],
    [5000],
])
def test_ragged_lengths(cuda_device, lens):
    inp = gen.make_inputs(len(lens), 1, lens, seed=sum(lens))
    out, lse, st = run_gpu(inp)
    assert st == 0
    assert_close(out, lse, *oracle(inp))


@pytest.mark.parametrize("sq,lens", [(2, [1, 2, 64, 65, 300]), (2, [129, 4096]), (3, [3, 64, 200]), (4, [70])])
def test_multi_token_causal(cuda_device, sq, lens):
    inp = gen.make_inputs(len(lens), sq, lens, seed=17 + sq)
    out, lse, st = run_gpu(inp)
    assert st == 0
    assert_close(out, lse, *oracle(inp))


def test_empty_rows(cuda_device):
    inp = gen.make_inputs(4, 1, [0, 70, 0, 1], seed=3, physical_pages=4)
    out, lse, st = run_gpu(inp)
    assert st == 0
    assert_close(out, lse, *oracle(inp))


def test_empty_rows_with_multi_token_queries(cuda_device):
    # rows with no token are written by the planner for every query index;
    # a one-token row leaves its first query with nothing to see
    inp = gen.make_inputs(3, 2, [0, 1, 130], seed=4)
    out, lse, st = run_gpu(inp)
    assert st == 0
    assert_close(out, lse, *oracle(inp))


@pytest.mark.parametrize("sq,lens", [(1, [1, 70, 0, 130]), (2, [3, 65])])
def test_wide_block_table_leaves_pairs_without_pages(cuda_device, sq, lens):
    # a block table far wider than the rows: the call gets many CTA pairs
    # (one per 8 pages it could hold) for a few pages, so most pair ranges
    # are empty, and the rows that do have pages may be split between pairs
    inp = gen.make_inputs(len(lens), sq, lens, seed=41 + sq, max_pages=96)
    out, lse, st = run_gpu(inp)
    assert st == 0
    assert_close(out, lse, *oracle(inp))


@pytest.mark.parametrize("sq,lens", [(1, [20000]), (2, [9000, 40])])
def test_rows_split_over_many_pairs(cuda_device, sq, lens):
    # one long row cut into dozens of parts (40 for the 20000-token row, so
    # the merge kernel takes their lse values in two groups of up to 32)
    inp = gen.make_inputs(len(lens), sq, lens, seed=31 + sq)
    out, lse, st = run_gpu(inp)
    assert st == 0
    assert_close(out, lse, *oracle(inp))


def test_large_batch_plans_from_global_memory(cuda_device):
    # 3000 rows (more than the planner mirrors in shared memory, so it
    # searches its global arrays; three rows per planner thread), short
    # random lengths with some empty rows.  Sampled rows are checked against
    # the oracle (on just their pages), every empty row for out = 0 and
    # lse = -inf.
    rng = np.random.default_rng(71)
    lens = rng.integers(0, 300, size=3000)
    lens[rng.choice(3000, 40, replace=False)] = 0
    inp = gen.make_inputs(3000, 1, lens.tolist(), seed=71)
    out, lse, st = run_gpu(inp)
    assert st == 0
    sample = np.array(sorted(set(rng.choice(3000, 48, replace=False).tolist()) | {0, 1, 2997, 2998, 2999}))
    bt = inp.block_table.numpy()[sample]
    used = np.unique(bt[bt >= 0])
    remap = {int(p): k for k, p in enumerate(used)}
    bt_sub = np.vectorize(lambda p: remap.get(int(p), -1))(bt).astype(np.int64)
    rows = mla_oracle.cache_rows(inp.kv_cache[torch.as_tensor(used)].double().numpy(), "bf16")
    ref_out, ref_lse = mla_oracle.mla_decode(inp.q_absorbed[sample].double().numpy(),
                                             inp.q_rope[sample].double().numpy(), rows, bt_sub,
                                             lens[sample], inp.scale)
    assert_close(out[torch.as_tensor(sample)], lse[torch.as_tensor(sample)], ref_out, ref_lse)
    empty = torch.as_tensor(np.nonzero(lens == 0)[0])
    assert torch.all(out[empty].float() == 0)
    assert torch.all(torch.isneginf(lse[empty]))


def test_lengths_written_just_before_the_call_are_used(cuda_device):
    # The planner is launched as a programmatic dependent of whatever precedes
    # it on the stream: lengths that a device kernel writes immediately before
    # the call (here the reversed list, capped at 1000) must be the ones it
    # plans with, and a second call with the original lengths must not see
    # stale plan state from the first.  Every row's block table covers both.
    lens = [300, 1, 0, 2000, 777, 64, 65, 1500]
    new = [min(x, 1000) for x in lens[::-1]]
    alloc = [max(a, b) for a, b in zip(lens, new)]
    inp = gen.make_inputs(len(lens), 1, alloc, seed=61)
    d = to_dev(inp)
    ws = binding.alloc_workspace(inp.batch, inp.sq)
    orig = torch.tensor(lens, dtype=torch.int32, device="cuda")
    sl = torch.minimum(orig.flip(0), torch.full_like(orig, 1000))   # device kernels on the call's stream
    raw = inp.kv_cache.double().numpy()
    rows = mla_oracle.cache_rows(raw, "bf16")

    def ref(lengths):
        return mla_oracle.mla_decode(inp.q_absorbed.double().numpy(), inp.q_rope.double().numpy(), rows,
                                     inp.block_table.numpy(), np.array(lengths, dtype=np.int64), inp.scale)

    out, lse = binding.mla_decode_bf16(d["q"], d["qr"], d["kv"], d["bt"], sl, inp.scale, workspace=ws)
    assert binding.mla_get_status(ws) == 0
    assert_close(out, lse, *ref(new))
    out2, lse2 = binding.mla_decode_bf16(d["q"], d["qr"], d["kv"], d["bt"], orig, inp.scale, workspace=ws)
    assert binding.mla_get_status(ws) == 0
    assert_close(out2, lse2, *ref(lens))


def test_single_token_is_bit_exact_copy(cuda_device):
    lens = [1] * 6
    inp = gen.make_inputs(6, 1, lens, seed=21)
    out, lse, st = run_gpu(inp)
    assert st == 0
    for b in range(6):
        page = int(inp.block_table[b, 0])
        row = inp.kv_cache[page, 0, :512]
        assert torch.equal(out[b, 0].cpu(), row.expand(128, 512)), b
    ref_out, ref_lse = oracle(inp)
    assert np.abs(lse.double().cpu().numpy() - ref_lse).max() <= LSE_ATOL


def test_unused_slots_hold_nan(cuda_device):
    lens = [70, 130, 1]
    inp = gen.make_inputs(3, 1, lens, seed=5)
    ref = oracle(inp)
    for b, s in enumerate(lens):
        page = int(inp.block_table[b, (s - 1) // 64])
        inp.kv_cache[page, s % 64 if s % 64 else 64:, :] = float("nan")
    out, lse, st = run_gpu(inp)
    assert st == 0
    assert torch.isfinite(out.float()).all()
    assert_close(out, lse, *ref)


def test_page_permutation_gives_identical_bits(cuda_device):
    lens = [300, 77]
    inp = gen.make_inputs(2, 1, lens, seed=9, physical_pages=12)
    out1, lse1, _ = run_gpu(inp)
    perm = torch.randperm(inp.num_pages, generator=torch.Generator().manual_seed(1))
    inv = torch.argsort(perm)
    kv2 = inp.kv_cache[perm].contiguous()
    bt2 = torch.where(inp.block_table >= 0, inv[inp.block_table.clamp(min=0).long()].int(), inp.block_table)
    inp2 = gen.DecodeInputs(inp.q_absorbed, inp.q_rope, kv2, bt2, inp.seq_lens, inp.scale, "bf16")
    out2, lse2, _ = run_gpu(inp2)
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


def test_growing_scores_exercise_rescale(cuda_device):
    """Scores that rise along the sequence make the reference max move by
    more than the lazy-rescale threshold many times."""
    n = 2000
    inp = gen.make_inputs(1, 1, [n], seed=2)
    pages = inp.block_table[0, : (n + 63) // 64]
    for j in range(n):
        inp.kv_cache[pages[j // 64], j % 64, 0] = j * 0.02
    inp.q_absorbed[..., 0] = torch.linspace(1, 120, 128).to(torch.bfloat16)
    out, lse, st = run_gpu(inp)
    assert st == 0
    assert_close(out, lse, *oracle(inp))


def test_bad_page_and_bad_length_set_status(cuda_device):
    inp = gen.make_inputs(2, 1, [100, 64], seed=4)
    inp.block_table[0, 1] = inp.num_pages + 7
    _, _, st = run_gpu(inp)
    assert st == -5
    inp = gen.make_inputs(2, 1, [100, 64], seed=4)
    inp.seq_lens[1] = inp.max_pages * 64 + 1
    _, _, st = run_gpu(inp)
    assert st == -7


def test_workspace_too_small_is_rejected(cuda_device):
    inp = gen.make_inputs(1, 1, [64], seed=4)
    d = to_dev(inp)
    ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.MLAError) as e:
        binding.mla_decode_bf16(d["q"], d["qr"], d["kv"], d["bt"], d["sl"], inp.scale, workspace=ws)
    assert e.value.code == -3


def test_combine_splits_matches_oracle_merge(cuda_device):
    rng = np.random.default_rng(0)
    counts = [1, 3, 0, 2]
    n = sum(counts)
    po = rng.standard_normal((n, 128, 512)).astype(np.float32)
    pl = (rng.standard_normal((n, 128)) * 3).astype(np.float32)
    pl[1, :5] = -np.inf
    indptr = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    out, lse = binding.mla_combine_splits(torch.from_numpy(po).cuda(), torch.from_numpy(pl).cuda(),
                                          torch.from_numpy(indptr).cuda())
    torch.cuda.synchronize()
    for r in range(len(counts)):
        a, b = indptr[r], indptr[r + 1]
        ro, rl = mla_oracle.merge_partials(po[a:b].astype(np.float64), pl[a:b].astype(np.float64))
        if b == a:
            assert torch.all(out[r] == 0) and torch.all(torch.isneginf(lse[r]))
            continue
        np.testing.assert_allclose(out[r].double().cpu().numpy(), ro, atol=1e-2 * np.abs(ro).max())
        np.testing.assert_allclose(lse[r].double().cpu().numpy(), rl, atol=1e-5)


# ----------------------------------------------------------------- FP8 cache
def _dequant_bf16(raw: torch.Tensor) -> torch.Tensor:
    """Oracle dequantisation of [..., 594] rows, cast to bf16 (exact)."""
    from oracle import fp8_codec
    return torch.from_numpy(fp8_codec.dequant_rows(raw.numpy())).to(torch.bfloat16)


def test_fp8_single_token_is_bit_exact_dequant(cuda_device):
    inp = gen.make_inputs(8, 1, [1] * 8, kv_dtype="fp8", seed=31)
    # a wide range of e8m0 exponents (kept where every product is a finite,
    # normal bf16 number, so the MMA's copy is exact) and the e4m3 extremes
    scales = [10, 11, 100, 120, 127, 130, 142, 143, 150, 200]
    for b in range(8):
        page = int(inp.block_table[b, 0])
        row = inp.kv_cache[page, 0]
        row[576:] = torch.tensor([scales[(b + k) % len(scales)] for k in range(18)], dtype=torch.uint8)
        row[:8] = torch.tensor([0x00, 0x80, 0x01, 0x81, 0x7E, 0xFE, 0x08, 0x77], dtype=torch.uint8)
    out, lse, st = run_gpu(inp)
    assert st == 0
    for b in range(8):
        page = int(inp.block_table[b, 0])
        want = _dequant_bf16(inp.kv_cache[page, 0])[:512]
        got = out[b, 0].cpu()
        # value-exact (the sign of a zero is not kept through the P.V sum,
        # where masked tokens add +0 to 1 * -0)
        assert torch.equal(got, want.expand(128, 512)), b


def test_fp8_every_token_position_is_bit_exact_dequant(cuda_device):
    # Batch row b attends to token b of its page and to nothing else: only
    # the first RoPE dimension of the query is set, and token b's first RoPE
    # value is +448 against -448 for every other token, so every other
    # weight is exp(-4000) = 0 and out = token b's dequantised latent,
    # exactly.  All 64 positions of a page are covered, which includes the
    # rows each SM of the pair dequantises.
    n = 64
    inp = gen.make_inputs(n, 1, [n] * n, kv_dtype="fp8", seed=33)
    inp.q_absorbed.zero_()
    inp.q_rope.zero_()
    inp.q_rope[..., 0] = 64.0
    for b in range(n):
        page = int(inp.block_table[b, 0])
        rows = inp.kv_cache[page]
        rows[:, 512:576] = 0                 # RoPE codes: zero ...
        rows[:, 576 + 16] = 127              # ... with scale 1 on the first RoPE group
        rows[:, 512] = 0xFE                  # -448 for every token
        rows[b, 512] = 0x7E                  # +448 for token b
        rows[b, :8] = torch.tensor([0x00, 0x80, 0x01, 0x81, 0x7E, 0xFE, 0x08, 0x77], dtype=torch.uint8)
    out, lse, st = run_gpu(inp)
    assert st == 0
    for b in range(n):
        page = int(inp.block_table[b, 0])
        want = _dequant_bf16(inp.kv_cache[page, b])[:512]
        got = out[b, 0].cpu()
        assert torch.equal(got, want.expand(128, 512)), b   # value-exact (-0 == +0)


@pytest.mark.parametrize("lens", [[1, 63, 64, 65, 200], [3000, 17]])
def test_fp8_ragged(cuda_device, lens):
    inp = gen.make_inputs(len(lens), 1, lens, kv_dtype="fp8", seed=7 + len(lens))
    out, lse, st = run_gpu(inp)
    assert st == 0
    assert_close(out, lse, *oracle(inp))


def test_fp8_causal_and_unused_nan_codes(cuda_device):
    lens = [70, 130]
    inp = gen.make_inputs(2, 2, lens, kv_dtype="fp8", seed=12)
    ref = oracle(inp)
    for b, s in enumerate(lens):
        page = int(inp.block_table[b, (s - 1) // 64])
        inp.kv_cache[page, s % 64:, :] = 0x7F          # NaN codes past the visible length
    out, lse, st = run_gpu(inp)
    assert st == 0
    assert torch.isfinite(out.float()).all()
    assert_close(out, lse, *ref)


def test_fp8_query_beyond_f16_range_takes_the_exact_pass(cuda_device):
    # The FP8 path computes with f16 operands when every scale exponent lies
    # in [113, 134] and every query value fits f16; otherwise an exact pass
    # with bf16 operands recomputes the call.  One query value of 1e5 (past
    # the f16 maximum 65504) forces that pass.  Latent dimension 7 of every
    # cached token is zero, so the scores keep their usual size and the
    # result must still match the oracle (in f16 the product would be
    # inf * 0 = NaN).
    inp = gen.make_inputs(3, 1, [200, 64, 1], kv_dtype="fp8", seed=41)
    inp.kv_cache[:, :, 7] = 0
    inp.q_absorbed[1, 0, 5, 7] = 1.0e5
    out, lse, st = run_gpu(inp)
    assert st == 0
    assert torch.isfinite(out.float()).all()
    assert_close(out, lse, *oracle(inp))


# ----------------------------------------------------------------- FP8 cache, V4.1 528-byte rows
def _dequant_v41_bf16(raw: torch.Tensor) -> torch.Tensor:
    """Oracle dequantisation of [..., 528] rows onto the 576-value row, cast
    to bf16 (exact)."""
    from oracle import fp8_codec
    return torch.from_numpy(fp8_codec.dequant_rows_v41(raw.numpy())).to(torch.bfloat16)


def test_fp8v41_single_token_is_bit_exact_dequant(cuda_device):
    # scale bytes far outside the f16-exact range: the exact bf16 pass
    inp = gen.make_inputs(8, 1, [1] * 8, kv_dtype="fp8v41", seed=32)
    scales = [10, 11, 100, 120, 127, 130, 142, 143, 150, 200]
    for b in range(8):
        page = int(inp.block_table[b, 0])
        row = inp.kv_cache[page, 0]
        row[512:] = torch.tensor([scales[(b + k) % len(scales)] for k in range(16)], dtype=torch.uint8)
        row[:8] = torch.tensor([0x00, 0x80, 0x01, 0x81, 0x7E, 0xFE, 0x08, 0x77], dtype=torch.uint8)
        row[440:448] = torch.tensor([0x7E, 0xFE, 0x01, 0x81, 0x38, 0xB8, 0x08, 0x77], dtype=torch.uint8)
    inp.q_absorbed[..., 448:] = float("nan")    # ignored: those latent dims are zero
    out, lse, st = run_gpu(inp)
    assert st == 0
    for b in range(8):
        page = int(inp.block_table[b, 0])
        want = _dequant_v41_bf16(inp.kv_cache[page, 0])[:512]
        assert not want[448:].float().any()
        got = out[b, 0].cpu()
        assert torch.equal(got, want.expand(128, 512)), b   # value-exact (-0 == +0)


def test_fp8v41_every_token_position_is_bit_exact_dequant(cuda_device):
    # as for the 594-byte row: only the first RoPE dimension of the query is
    # set, and token b's first RoPE value (byte 448 of the V4.1 row, scale
    # byte 526) is +448 against -448 for every other token; the default
    # scales (120..130) take the f16-operand pass
    n = 64
    inp = gen.make_inputs(n, 1, [n] * n, kv_dtype="fp8v41", seed=34)
    inp.q_absorbed.zero_()
    inp.q_rope.zero_()
    inp.q_rope[..., 0] = 64.0
    for b in range(n):
        page = int(inp.block_table[b, 0])
        rows = inp.kv_cache[page]
        rows[:, 448:512] = 0                 # RoPE codes: zero ...
        rows[:, 512 + 14] = 127              # ... with scale 1 on the first RoPE group
        rows[:, 448] = 0xFE                  # -448 for every token
        rows[b, 448] = 0x7E                  # +448 for token b
        rows[b, :8] = torch.tensor([0x00, 0x80, 0x01, 0x81, 0x7E, 0xFE, 0x08, 0x77], dtype=torch.uint8)
    out, lse, st = run_gpu(inp)
    assert st == 0
    for b in range(n):
        page = int(inp.block_table[b, 0])
        want = _dequant_v41_bf16(inp.kv_cache[page, b])[:512]
        got = out[b, 0].cpu()
        assert torch.equal(got, want.expand(128, 512)), b


@pytest.mark.parametrize("sq,lens", [(1, [1, 63, 64, 65, 200]), (1, [3000, 17]), (2, [70, 130, 1])])
def test_fp8v41_ragged_and_causal(cuda_device, sq, lens):
    inp = gen.make_inputs(len(lens), sq, lens, kv_dtype="fp8v41", seed=9 + len(lens) + sq)
    ref = oracle(inp)
    inp.q_absorbed[..., 448:] = float("nan")    # ignored: the oracle saw them as they were (finite)
    out, lse, st = run_gpu(inp)
    assert st == 0
    assert_close(out, lse, *ref)
    assert not out[..., 448:].float().any()


def test_fp8_bad_page_sets_status(cuda_device):
    inp = gen.make_inputs(2, 1, [100, 64], kv_dtype="fp8", seed=4)
    inp.block_table[1, 0] = -3
    _, _, st = run_gpu(inp)
    assert st == -5


def _dequant4_bf16(raw):
    return torch.from_numpy(fp4_codec.dequant_rows(raw.numpy())).to(torch.bfloat16)


# FP4 rows: 288 code bytes (two e2m1 per byte, value 2k in the low nibble),
# then 36 e8m0 scales, one per 16 values.

def test_fp4_every_token_position_is_bit_exact_dequant(cuda_device):
    # As for FP8: batch row b attends to token b of its page alone (only the
    # first RoPE dimension of the query is set; token b's first RoPE value is
    # +6 * 2^4 against -6 * 2^4 for every other token, so every other weight
    # is exp(-16 * 192 / sqrt(192)) ~ 1e-96 = 0 in fp32), and out = token b's
    # dequantised latent row exactly.  Token b's first code bytes cover all
    # sixteen e2m1 codes in both nibbles, and its scales span a wide range
    # (kept where every value is a normal bf16 number, so the MMA's copy is
    # exact).
    n = 64
    inp = gen.make_inputs(n, 1, [n] * n, kv_dtype="fp4", seed=35)
    inp.q_absorbed.zero_()
    inp.q_rope.zero_()
    inp.q_rope[..., 0] = 16.0
    scales = [2, 10, 100, 119, 127, 128, 135, 150, 200, 252]
    for b in range(n):
        page = int(inp.block_table[b, 0])
        rows = inp.kv_cache[page]
        rows[:, 256:288] = 0                     # RoPE codes (values 512..575): zero ...
        rows[:, 288 + 32] = 131                  # ... scale 2^4 on values 512..527
        rows[:, 256] = 0x0F                      # value 512 = -6 * 2^4 for every token ...
        rows[b, 256] = 0x07                      # ... and +6 * 2^4 for token b
        rows[b, :16] = torch.tensor([0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE,
                                     0x01, 0x23, 0x45, 0x67, 0x89, 0xAB, 0xCD, 0xEF], dtype=torch.uint8)
        rows[b, 288:288 + 32] = torch.tensor([scales[(b + k) % len(scales)] for k in range(32)], dtype=torch.uint8)
    out, lse, st = run_gpu(inp)
    assert st == 0
    for b in range(n):
        page = int(inp.block_table[b, 0])
        want = _dequant4_bf16(inp.kv_cache[page, b])[:512]
        got = out[b, 0].cpu()
        assert torch.equal(got, want.expand(128, 512)), b   # value-exact (-0 == +0)


@pytest.mark.parametrize("lens", [[1, 63, 64, 65, 200], [3000, 17]])
def test_fp4_ragged(cuda_device, lens):
    inp = gen.make_inputs(len(lens), 1, lens, kv_dtype="fp4", seed=17 + len(lens))
    out, lse, st = run_gpu(inp)
    assert st == 0
    assert_close(out, lse, *oracle(inp))


def test_fp4_causal_split_rows(cuda_device):
    inp = gen.make_inputs(3, 2, [70, 5000, 130], kv_dtype="fp4", seed=18)
    out, lse, st = run_gpu(inp)
    assert st == 0
    assert_close(out, lse, *oracle(inp))


@pytest.mark.parametrize("scale_byte", [112, 140, 141])
def test_fp4_scale_at_the_f16_range_edges(cuda_device, scale_byte):
    # the f16-operand pass takes scale bytes in [113, 140]; 112 and 141 make
    # the exact bf16-operand pass recompute the call, and all three must
    # match the oracle.  The edge scale sits on latent values 48..63 of one
    # token (up to 6 * 2^14 there), and the query is zero on those
    # dimensions, so they reach the output but not the scores (scores in the
    # thousands would put fp32 accumulation error above the lse bound).
    inp = gen.make_inputs(2, 1, [150, 64], kv_dtype="fp4", seed=19)
    page = int(inp.block_table[0, 1])
    inp.kv_cache[page, 5, 288 + 3] = scale_byte
    inp.q_absorbed[0, :, :, 48:64] = 0
    out, lse, st = run_gpu(inp)
    assert st == 0
    assert torch.isfinite(out.float()).all()
    assert_close(out, lse, *oracle(inp))


# FP4 V4.1 rows: 256 code bytes (512 values: 448 latent, then 64 RoPE), then
# 32 e8m0 scales, one per 16 values.

def test_fp4v41_every_token_position_is_bit_exact_dequant(cuda_device):
    # as for the 324-byte row: token b's first RoPE value (code byte 224, low
    # nibble; scale byte 256 + 28) is +6 * 2^4 against -6 * 2^4 elsewhere;
    # token b's first code bytes cover all sixteen codes in both nibbles and
    # its scales span a wide range (the exact bf16 pass)
    n = 64
    inp = gen.make_inputs(n, 1, [n] * n, kv_dtype="fp4v41", seed=36)
    inp.q_absorbed.zero_()
    inp.q_absorbed[..., 448:] = float("nan")   # ignored
    inp.q_rope.zero_()
    inp.q_rope[..., 0] = 16.0
    scales = [2, 10, 100, 119, 127, 128, 135, 150, 200, 252]
    for b in range(n):
        page = int(inp.block_table[b, 0])
        rows = inp.kv_cache[page]
        rows[:, 224:256] = 0                     # RoPE codes (values 448..511): zero ...
        rows[:, 256 + 28] = 131                  # ... scale 2^4 on values 448..463
        rows[:, 224] = 0x0F                      # RoPE value 0 = -6 * 2^4 for every token ...
        rows[b, 224] = 0x07                      # ... and +6 * 2^4 for token b
        rows[b, :16] = torch.tensor([0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE,
                                     0x01, 0x23, 0x45, 0x67, 0x89, 0xAB, 0xCD, 0xEF], dtype=torch.uint8)
        rows[b, 256:256 + 28] = torch.tensor([scales[(b + k) % len(scales)] for k in range(28)], dtype=torch.uint8)
    out, lse, st = run_gpu(inp)
    assert st == 0
    for b in range(n):
        page = int(inp.block_table[b, 0])
        want = torch.from_numpy(fp4_codec.dequant_rows_v41(inp.kv_cache[page, b].numpy())).to(torch.bfloat16)[:512]
        got = out[b, 0].cpu()
        assert torch.equal(got, want.expand(128, 512)), b


@pytest.mark.parametrize("sq,lens", [(1, [1, 63, 64, 65, 200]), (1, [3000, 17]), (2, [70, 5000, 130])])
def test_fp4v41_ragged_and_causal(cuda_device, sq, lens):
    inp = gen.make_inputs(len(lens), sq, lens, kv_dtype="fp4v41", seed=27 + len(lens) + sq)
    ref = oracle(inp)
    inp.q_absorbed[..., 448:] = float("nan")
    out, lse, st = run_gpu(inp)
    assert st == 0
    assert_close(out, lse, *ref)
    assert not out[..., 448:].float().any()


@pytest.mark.parametrize("kv", ["fp8v41", "fp4v41"])
def test_v41_bad_page_sets_status(cuda_device, kv):
    inp = gen.make_inputs(2, 1, [100, 64], kv_dtype=kv, seed=7)
    inp.block_table[1, 0] = -3
    _, _, st = run_gpu(inp)
    assert st == -5


def test_fp4_bad_page_sets_status(cuda_device):
    inp = gen.make_inputs(2, 1, [100, 64], kv_dtype="fp4", seed=5)
    inp.block_table[1, 0] = -3
    _, _, st = run_gpu(inp)
    assert st == -5
