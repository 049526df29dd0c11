"""GPU parity of the sparse top-k decode (through the C ABI) against the
float64 oracle: random slot lists drawn from each row's context, -1 padding
at the end and in the middle, duplicates, a list that names the whole
context (equal to the dense decode), empty rows, single tokens (bit-exact
copies) and bad entries.

Bounds: max|out - ref| <= 1e-2 * max|ref| and max|lse - ref| <= 1e-3.
"""
import numpy as np
import pytest
import torch

from mla_latent_kv_05_gb300 import binding
from mla_latent_kv_05_gb300 import inputs as gen
from oracle import mla_oracle

pytestmark = pytest.mark.gpu

OUT_RTOL = 1e-2
LSE_ATOL = 1e-3


def run_sparse(inp, slots=None):
    d = inp.dense
    slots = inp.token_slots if slots is None else slots
    ws = binding.alloc_workspace_sparse(d.batch, d.sq, slots.shape[2])
    out, lse = binding.mla_decode_sparse_bf16(d.q_absorbed.cuda(), d.q_rope.cuda(), d.kv_cache.cuda(),
                                              slots.cuda(), d.scale, workspace=ws)
    return out, lse, binding.mla_get_status(ws)


def oracle_sparse(inp, slots=None):
    d = inp.dense
    slots = inp.token_slots if slots is None else slots
    rows = mla_oracle.cache_rows(d.kv_cache.double().numpy(), "bf16")
    return mla_oracle.mla_decode_sparse(d.q_absorbed.double().numpy(), d.q_rope.double().numpy(), rows,
                                        slots.numpy(), d.scale)


def assert_close(out, lse, ref_out, ref_lse):
    got = out.double().cpu().numpy()
    gl = lse.double().cpu().numpy()
    B, Sq = got.shape[:2]
    for b in range(B):
        for i in range(Sq):
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


@pytest.mark.parametrize("lens,sq,topk,pad", [
    ([700, 130, 64, 3000], 2, 256, True),
    ([5000, 40], 1, 2048, False),
    ([300, 301, 95], 1, 100, True),
    ([64] * 6, 3, 64, False),
])
def test_sparse_matches_oracle(cuda_device, lens, sq, topk, pad):
    inp = gen.make_sparse_inputs(len(lens), sq, lens, topk, seed=50 + topk + len(lens), pad_middle=pad)
    out, lse, st = run_sparse(inp)
    assert st == 0
    assert_close(out, lse, *oracle_sparse(inp))


def test_sparse_listing_the_context_equals_dense_decode(cuda_device):
    d = gen.make_inputs(3, 1, [1000, 77, 2048], seed=61)
    topk = 2048
    slots = torch.full((3, 1, topk), -1, dtype=torch.int32)
    bt = d.block_table.to(torch.int64)
    for b in range(3):
        n = int(d.seq_lens[b])
        j = torch.arange(n)
        slots[b, 0, :n] = (bt[b, j // 64] * 64 + j % 64).to(torch.int32)
    inp = gen.SparseInputs(dense=d, token_slots=slots, topk=topk)
    out, lse, st = run_sparse(inp)
    assert st == 0
    dense_out, dense_lse = binding.mla_decode_bf16(d.q_absorbed.cuda(), d.q_rope.cuda(), d.kv_cache.cuda(),
                                                   d.block_table.cuda(), d.seq_lens.cuda(), d.scale)
    assert_close(out, lse, *oracle_sparse(inp))
    # the two paths differ only in summation order
    assert torch.allclose(out.float(), dense_out.float(), rtol=2e-2, atol=2e-2)
    assert torch.allclose(lse, dense_lse, atol=1e-3)


def test_sparse_duplicates_empty_rows_and_single_tokens(cuda_device):
    d = gen.make_inputs(4, 1, [200, 200, 200, 200], seed=62)
    topk = 96
    slots = torch.full((4, 1, topk), -1, dtype=torch.int32)
    p0 = int(d.block_table[0, 0]) * 64
    slots[0, 0, :6] = torch.tensor([p0 + 3, p0 + 3, p0 + 9, -1, p0 + 3, p0 + 40])   # duplicates
    # row 1: no token at all
    slots[2, 0, 57] = p0 + 11                                                       # one token, mid-list
    slots[3, 0, :] = torch.arange(topk, dtype=torch.int32) + 64                    # two whole pages' slots
    inp = gen.SparseInputs(dense=d, token_slots=slots, topk=topk)
    out, lse, st = run_sparse(inp)
    assert st == 0
    ref_out, ref_lse = oracle_sparse(inp)
    assert_close(out, lse, ref_out, ref_lse)
    # a single listed token is an exact copy of its latent row
    row = d.kv_cache.view(-1, 576)[p0 + 11, :512]
    assert torch.equal(out[2, 0].cpu(), row.expand(128, 512))


def test_sparse_bad_entries_set_status_and_are_skipped(cuda_device):
    inp = gen.make_sparse_inputs(2, 1, [500, 300], 128, seed=63)
    slots = inp.token_slots.clone()
    n_slots = inp.dense.num_pages * 64
    slots[0, 0, 5] = n_slots + 7
    slots[1, 0, 0] = -5
    out, lse, st = run_sparse(inp, slots)
    assert st == -8
    cleaned = torch.where((slots >= 0) & (slots < n_slots), slots, torch.full_like(slots, -1))
    assert_close(out, lse, *oracle_sparse(inp, cleaned))
