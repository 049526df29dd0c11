"""The seeded input generator: determinism and the structure of the workloads."""
import torch

from mla_latent_kv_05_gb300 import inputs as gen


def test_same_seed_same_inputs():
    a = gen.make_inputs(3, 2, [5, 64, 130], seed=4)
    b = gen.make_inputs(3, 2, [5, 64, 130], seed=4)
    for x, y in [(a.q_absorbed, b.q_absorbed), (a.q_rope, b.q_rope), (a.kv_cache, b.kv_cache),
                 (a.block_table, b.block_table), (a.seq_lens, b.seq_lens)]:
        assert torch.equal(x, y)
    c = gen.make_inputs(3, 2, [5, 64, 130], seed=5)
    assert not torch.equal(a.kv_cache, c.kv_cache)


def test_block_table_is_a_slice_of_a_permutation():
    inp = gen.make_inputs(4, 1, [1, 64, 65, 0], seed=2, physical_pages=10)
    bt = inp.block_table
    used = []
    for b, s in enumerate(inp.seq_lens.tolist()):
        n = (s + 63) // 64
        used += bt[b, :n].tolist()
        assert torch.all(bt[b, n:] == -1)
    assert len(set(used)) == len(used) == 4
    assert all(0 <= p < inp.num_pages for p in used)


def test_workload_shapes():
    seq3 = gen.workload_seq_lens(3)
    assert len(seq3) == 64 and min(seq3) >= 1 and max(seq3) <= 32768
    assert seq3 == gen.workload_seq_lens(3)
    assert gen.workload_seq_lens(5) == [131072] * 4
    w1 = gen.make_workload(1)
    assert w1.kv_cache.shape == (8, 64, 576) and w1.kv_cache.dtype == torch.bfloat16
    assert w1.q_absorbed.shape == (1, 1, 128, 512) and w1.q_rope.shape == (1, 1, 128, 64)


def test_fp8_scale_bytes_in_range():
    inp = gen.make_inputs(2, 1, [100, 3], kv_dtype="fp8", seed=1)
    assert inp.kv_cache.shape[-1] == 594 and inp.kv_cache.dtype == torch.uint8
    sc = inp.kv_cache[..., 576:]
    assert int(sc.min()) >= 120 and int(sc.max()) <= 130
    vals = inp.kv_cache[..., :576].contiguous().view(torch.float8_e4m3fn).float()
    assert torch.isfinite(vals).all()


def test_counts_workload2():
    c = gen.workload_counts(gen.make_inputs(32, 1, [4096] * 32, seed=0, num_heads=128))
    assert c["kv_tokens"] == 32 * 4096
    assert c["flops"] == 32 * 4096 * 2 * 128 * (576 + 512)


def test_fp4_cache_bytes_and_scales():
    a = gen.make_inputs(2, 1, [100, 3], kv_dtype="fp4", seed=1)
    b = gen.make_inputs(2, 1, [100, 3], kv_dtype="fp4", seed=1)
    assert torch.equal(a.kv_cache, b.kv_cache)
    assert a.kv_cache.shape == (3, 64, 324) and a.kv_cache.dtype == torch.uint8
    sc = a.kv_cache[..., 288:]
    assert int(sc.min()) >= 120 and int(sc.max()) <= 130
    # both nibbles of the code bytes take all sixteen values
    codes = a.kv_cache[..., :288]
    assert set((codes & 0xF).unique().tolist()) == set(range(16)) == set((codes >> 4).unique().tolist())


def test_counts_per_cache_format():
    # the algorithmic KV bytes per token: 1152 (bf16), 594 (fp8), 324 (fp4)
    for kv, row in (("bf16", 1152), ("fp8", 594), ("fp4", 324)):
        c = gen.workload_counts(gen.make_inputs(2, 1, [100, 28], kv_dtype=kv, seed=0))
        assert c["kv_bytes"] == 128 * row, kv
    assert gen.WORKLOADS[7]["kv_dtype"] == "fp4"
    assert gen.WORKLOADS[7]["batch"] == gen.WORKLOADS[4]["batch"] and gen.WORKLOADS[7]["seq"] == gen.WORKLOADS[4]["seq"]


def test_v41_caches_bytes_scales_and_counts():
    a = gen.make_inputs(2, 1, [100, 3], kv_dtype="fp8v41", seed=1)
    assert a.kv_cache.shape == (3, 64, 528) and a.kv_cache.dtype == torch.uint8
    sc = a.kv_cache[..., 512:]
    assert int(sc.min()) >= 120 and int(sc.max()) <= 130
    assert torch.isfinite(a.kv_cache[..., :512].contiguous().view(torch.float8_e4m3fn).float()).all()
    b = gen.make_inputs(2, 1, [100, 3], kv_dtype="fp4v41", seed=1)
    assert b.kv_cache.shape == (3, 64, 288)
    assert int(b.kv_cache[..., 256:].min()) >= 120 and int(b.kv_cache[..., 256:].max()) <= 130
    # the V4.1 rows' FLOPs are counted on their own 448-value latent
    for kv, row in (("fp8v41", 528), ("fp4v41", 288)):
        c = gen.workload_counts(gen.make_inputs(2, 1, [100, 28], kv_dtype=kv, seed=0))
        assert c["kv_bytes"] == 128 * row
        assert c["flops"] == 128 * 2 * 128 * ((448 + 64) + 448)
    for w in (8, 9):
        assert gen.WORKLOADS[w]["batch"] == 128 and gen.WORKLOADS[w]["seq"] == 8192


def test_workload3_lengths_are_the_seeded_uniform_draw():
    lens = gen.workload_seq_lens(3)
    assert lens == gen.workload_seq_lens(3) and len(lens) == 64
    assert min(lens) >= 1 and max(lens) <= 32768
    assert 8000 < sum(lens) / 64 < 24000                       # a U[1, 32768] mean, loosely
    assert gen.workload_seq_lens(2) == [4096] * 32


def test_sparse_lists_name_distinct_visible_slots():
    sp = gen.make_sparse_inputs(3, 2, [300, 5, 0], 64, seed=2, pad_middle=True)
    bt = sp.dense.block_table
    for b, ctx in enumerate([300, 5, 0]):
        for i in range(2):
            vis = max(ctx - (1 - i), 0)
            lst = [int(x) for x in sp.token_slots[b, i] if int(x) >= 0]
            assert len(lst) == len(set(lst)) <= min(vis, 64)
            allowed = {int(bt[b, t // 64]) * 64 + t % 64 for t in range(vis)}
            assert set(lst) <= allowed
            if not sp.token_slots.shape[2] > vis:
                continue
            assert (sp.token_slots[b, i] == -1).sum() >= 64 - vis
    c = gen.sparse_counts(sp)
    assert c["kv_tokens"] == int((sp.token_slots >= 0).sum())
