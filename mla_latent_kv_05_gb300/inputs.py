"""Seeded synthetic inputs for MLA decode over a paged latent KV cache.

This module is the one piece shared by the float64 oracle tests and the CUDA
path: it only draws random numbers and builds page tables. It holds none of the
attention arithmetic. The FP8 cache is produced by rounding N(0,1) draws to
e4m3 with torch's own cast and drawing the e8m0 scale bytes independently; the
FP4 cache is uniform random bytes (two e2m1 codes each) and uniform scale
bytes.  The decoding of those bytes is done separately by each side.

Shapes follow the model records on the pages (DeepSeek-R1 / V3.2 records:
kv_lora_rank 512; architecture guide section 1.1: 512 latent + 64 decoupled
RoPE values per cached token, 128 heads; page-block size 64 from the serving
constraints paragraph of the R1 record).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

NUM_HEADS = 128
D_LATENT = 512
D_ROPE = 64
ROW_ELEMS = D_LATENT + D_ROPE          # 576 values per token per layer
PAGE_SIZE = 64
FP8_SCALE_GROUP = 32
FP8_NUM_SCALES = ROW_ELEMS // FP8_SCALE_GROUP   # 18
FP8_ROW_BYTES = ROW_ELEMS + FP8_NUM_SCALES      # 594
FP4_SCALE_GROUP = 16
FP4_NUM_SCALES = ROW_ELEMS // FP4_SCALE_GROUP   # 36
FP4_ROW_BYTES = ROW_ELEMS // 2 + FP4_NUM_SCALES # 324
V41_VALUES = 512                                # V4.1 row: 448 latent + 64 RoPE values
V41_NUM_SCALES = V41_VALUES // FP8_SCALE_GROUP  # 16
V41_ROW_BYTES = V41_VALUES + V41_NUM_SCALES     # 528
V41_FP4_ROW_BYTES = V41_VALUES // 2 + V41_VALUES // FP4_SCALE_GROUP   # 288
DEFAULT_SCALE = 1.0 / math.sqrt(128 + 64)       # 1/sqrt(d_h + d_h^R)


def row_bytes_of(kv_dtype: str) -> int:
    """Bytes of one cached token row in each cache format."""
    return {"bf16": ROW_ELEMS * 2, "fp8": FP8_ROW_BYTES, "fp4": FP4_ROW_BYTES, "fp8v41": V41_ROW_BYTES,
            "fp4v41": V41_FP4_ROW_BYTES}[kv_dtype]


@dataclass
class DecodeInputs:
    """One decode call's inputs, on the host (CPU tensors)."""
    q_absorbed: torch.Tensor   # [B, Sq, H, 512] bf16
    q_rope: torch.Tensor       # [B, Sq, H, 64] bf16
    kv_cache: torch.Tensor     # bf16 [P, 64, 576]; uint8 [P, 64, 594] (fp8), [P, 64, 528] (fp8v41),
                               # [P, 64, 324] (fp4) or [P, 64, 288] (fp4v41)
    block_table: torch.Tensor  # int32 [B, max_pages], -1 where unused
    seq_lens: torch.Tensor     # int32 [B]
    scale: float
    kv_dtype: str              # "bf16", "fp8", "fp8v41", "fp4" or "fp4v41"
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.q_absorbed.shape[0])

    @property
    def sq(self) -> int:
        return int(self.q_absorbed.shape[1])

    @property
    def num_pages(self) -> int:
        return int(self.kv_cache.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])


# The dense workloads: name -> parameters.  seq is either an int (uniform) or
# ("uniform", lo, hi) for lengths drawn from the seed.
WORKLOADS = {
    1: dict(name="oracle-sized B1 seq256 bf16", batch=1, sq=1, seq=256,
            kv_dtype="bf16", physical_pages=8),
    2: dict(name="uniform B32 seq4096 bf16", batch=32, sq=1, seq=4096,
            kv_dtype="bf16"),
    3: dict(name="ragged B64 seq U[1,32768] bf16", batch=64, sq=1,
            seq=("uniform", 1, 32768), kv_dtype="bf16"),
    4: dict(name="fp8 B128 seq8192", batch=128, sq=1, seq=8192,
            kv_dtype="fp8"),
    5: dict(name="B4 Sq2 causal seq131072 bf16", batch=4, sq=2, seq=131072,
            kv_dtype="bf16"),
    7: dict(name="fp4 B128 seq8192", batch=128, sq=1, seq=8192,
            kv_dtype="fp4"),
    8: dict(name="fp8 V4.1 row B128 seq8192", batch=128, sq=1, seq=8192,
            kv_dtype="fp8v41"),
    9: dict(name="fp4 V4.1 row B128 seq8192", batch=128, sq=1, seq=8192,
            kv_dtype="fp4v41"),
}


def seed_for(workload: int) -> int:
    return 1000 + int(workload)


def _randn_bf16(gen: torch.Generator, shape, chunk_elems: int = 1 << 24) -> torch.Tensor:
    """N(0,1) rounded to bf16, drawn in fixed chunks along dim 0 so peak host
    memory stays bounded; the chunking is part of the recipe (deterministic)."""
    out = torch.empty(shape, dtype=torch.bfloat16)
    flat = out.view(shape[0], -1)
    per_row = flat.shape[1]
    rows_per_chunk = max(1, chunk_elems // max(per_row, 1))
    for r0 in range(0, shape[0], rows_per_chunk):
        r1 = min(shape[0], r0 + rows_per_chunk)
        flat[r0:r1] = torch.randn((r1 - r0, per_row), generator=gen).to(torch.bfloat16)
    return out


def _fp8_cache(gen: torch.Generator, num_pages: int, page_size: int) -> torch.Tensor:
    """[P, page, 594] uint8: 576 e4m3 bytes (N(0,1) rounded by torch's cast)
    followed by 18 e8m0 exponent bytes drawn uniformly from [120, 130]."""
    out = torch.empty((num_pages, page_size, FP8_ROW_BYTES), dtype=torch.uint8)
    step = 512
    for p0 in range(0, num_pages, step):
        p1 = min(num_pages, p0 + step)
        vals = torch.randn((p1 - p0, page_size, ROW_ELEMS), generator=gen)
        out[p0:p1, :, :ROW_ELEMS] = vals.to(torch.float8_e4m3fn).view(torch.uint8)
        out[p0:p1, :, ROW_ELEMS:] = torch.randint(
            120, 131, (p1 - p0, page_size, FP8_NUM_SCALES), generator=gen,
            dtype=torch.int64).to(torch.uint8)
    return out


def _fp8v41_cache(gen: torch.Generator, num_pages: int, page_size: int) -> torch.Tensor:
    """[P, page, 528] uint8 V4.1 rows: 512 e4m3 bytes (N(0,1) rounded by
    torch's cast; 448 latent then 64 RoPE values) followed by 16 e8m0
    exponent bytes drawn uniformly from [120, 130]."""
    out = torch.empty((num_pages, page_size, V41_ROW_BYTES), dtype=torch.uint8)
    step = 512
    for p0 in range(0, num_pages, step):
        p1 = min(num_pages, p0 + step)
        vals = torch.randn((p1 - p0, page_size, V41_VALUES), generator=gen)
        out[p0:p1, :, :V41_VALUES] = vals.to(torch.float8_e4m3fn).view(torch.uint8)
        out[p0:p1, :, V41_VALUES:] = torch.randint(
            120, 131, (p1 - p0, page_size, V41_NUM_SCALES), generator=gen,
            dtype=torch.int64).to(torch.uint8)
    return out


def _fp4v41_cache(gen: torch.Generator, num_pages: int, page_size: int) -> torch.Tensor:
    """[P, page, 288] uint8 V4.1 FP4 rows: 256 uniform random bytes (512
    e2m1 codes, two per byte; 448 latent then 64 RoPE values) followed by 32
    e8m0 exponent bytes drawn uniformly from [120, 130]."""
    out = torch.empty((num_pages, page_size, V41_FP4_ROW_BYTES), dtype=torch.uint8)
    step = 1024
    nc = V41_VALUES // 2
    for p0 in range(0, num_pages, step):
        p1 = min(num_pages, p0 + step)
        out[p0:p1, :, :nc] = torch.randint(0, 256, (p1 - p0, page_size, nc), generator=gen,
                                           dtype=torch.int64).to(torch.uint8)
        out[p0:p1, :, nc:] = torch.randint(120, 131, (p1 - p0, page_size, V41_VALUES // FP4_SCALE_GROUP),
                                           generator=gen, dtype=torch.int64).to(torch.uint8)
    return out


def _fp4_cache(gen: torch.Generator, num_pages: int, page_size: int,
               scale_lo: int = 120, scale_hi: int = 130) -> torch.Tensor:
    """[P, page, 324] uint8: 288 uniform random bytes (576 e2m1 codes, two per
    byte) followed by 36 e8m0 exponent bytes drawn uniformly from
    [scale_lo, scale_hi]."""
    out = torch.empty((num_pages, page_size, FP4_ROW_BYTES), dtype=torch.uint8)
    step = 1024
    nc = ROW_ELEMS // 2
    for p0 in range(0, num_pages, step):
        p1 = min(num_pages, p0 + step)
        out[p0:p1, :, :nc] = torch.randint(0, 256, (p1 - p0, page_size, nc), generator=gen,
                                           dtype=torch.int64).to(torch.uint8)
        out[p0:p1, :, nc:] = torch.randint(scale_lo, scale_hi + 1, (p1 - p0, page_size, FP4_NUM_SCALES),
                                           generator=gen, dtype=torch.int64).to(torch.uint8)
    return out


def make_inputs(batch: int, sq: int, seq_lens, kv_dtype: str = "bf16",
                seed: int = 0, physical_pages: int | None = None,
                max_pages: int | None = None, scale: float = DEFAULT_SCALE,
                page_size: int = PAGE_SIZE, num_heads: int = NUM_HEADS,
                name: str = "") -> DecodeInputs:
    """Build one seeded decode problem.

    seq_lens: list/tensor of B ints.  Pages: each row b needs ceil(len/64)
    pages; the physical page pool is a seeded permutation of all pages
    (plus any extra physical pages requested), sliced row by row into the
    block table; unused block-table entries are -1.
    """
    gen = torch.Generator().manual_seed(int(seed))
    seq = torch.as_tensor(seq_lens, dtype=torch.int64).reshape(-1)
    assert seq.numel() == batch
    need = [(int(s) + page_size - 1) // page_size if int(s) > 0 else 0 for s in seq]
    total_needed = sum(need)
    n_phys = max(total_needed, int(physical_pages or 0), 1)
    mp = max(max(need) if need else 0, int(max_pages or 0), 1)
    perm = torch.randperm(n_phys, generator=gen)
    block_table = torch.full((batch, mp), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(need):
        if n:
            block_table[b, :n] = perm[off:off + n].to(torch.int32)
            off += n
    q_abs = _randn_bf16(gen, (batch, sq, num_heads, D_LATENT))
    q_rope = _randn_bf16(gen, (batch, sq, num_heads, D_ROPE))
    if kv_dtype == "bf16":
        cache = _randn_bf16(gen, (n_phys, page_size, ROW_ELEMS))
    elif kv_dtype == "fp8":
        cache = _fp8_cache(gen, n_phys, page_size)
    elif kv_dtype == "fp4":
        cache = _fp4_cache(gen, n_phys, page_size)
    elif kv_dtype == "fp8v41":
        cache = _fp8v41_cache(gen, n_phys, page_size)
    elif kv_dtype == "fp4v41":
        cache = _fp4v41_cache(gen, n_phys, page_size)
    else:
        raise ValueError(kv_dtype)
    return DecodeInputs(q_absorbed=q_abs, q_rope=q_rope, kv_cache=cache,
                        block_table=block_table,
                        seq_lens=seq.to(torch.int32), scale=float(scale),
                        kv_dtype=kv_dtype, name=name)


def workload_seq_lens(workload: int) -> list[int]:
    w = WORKLOADS[workload]
    if isinstance(w["seq"], tuple):
        _, lo, hi = w["seq"]
        gen = torch.Generator().manual_seed(seed_for(workload) * 7919)
        return torch.randint(lo, hi + 1, (w["batch"],), generator=gen).tolist()
    return [int(w["seq"])] * w["batch"]


def make_workload(workload: int) -> DecodeInputs:
    """The seeded inputs of one of the dense workloads (seed = 1000 + index)."""
    w = WORKLOADS[workload]
    return make_inputs(w["batch"], w["sq"], workload_seq_lens(workload),
                       kv_dtype=w["kv_dtype"], seed=seed_for(workload),
                       physical_pages=w.get("physical_pages"),
                       name=w["name"])


def workload_counts(inp: DecodeInputs) -> dict:
    """Units of work of a problem, for throughput and roofline accounting:
    visible (query, token) pairs, distinct KV rows read, and the algorithmic
    byte and FLOP counts (bytes: each visible KV row once per batch row, q,
    out, lse, used block-table entries and seq_lens)."""
    seq = [int(s) for s in inp.seq_lens.tolist()]
    sq = inp.sq
    H = int(inp.q_absorbed.shape[2])
    row_bytes = row_bytes_of(inp.kv_dtype)
    kv_tokens = sum(max(s, 0) for s in seq)
    pairs = 0
    for s in seq:
        for i in range(sq):
            pairs += max(s - (sq - 1 - i), 0)
    used_pages = sum((max(s, 0) + PAGE_SIZE - 1) // PAGE_SIZE for s in seq)
    q_bytes = inp.batch * sq * H * (D_LATENT + D_ROPE) * 2
    out_bytes = inp.batch * sq * H * D_LATENT * 2
    lse_bytes = inp.batch * sq * H * 4
    bytes_ = kv_tokens * row_bytes + q_bytes + out_bytes + lse_bytes + used_pages * 4 + inp.batch * 4
    # the V4.1 row carries a 448-value latent: the method's work is scores
    # over 448 + 64 values and P.V over 448 (this path pads both to 512)
    latent = V41_VALUES - D_ROPE if inp.kv_dtype in ("fp8v41", "fp4v41") else D_LATENT
    flops = pairs * 2 * H * ((latent + D_ROPE) + latent)
    return dict(kv_tokens=kv_tokens, query_token_pairs=pairs, bytes=bytes_,
                flops=flops, kv_bytes=kv_tokens * row_bytes)


# --------------------------------------------------------------------------
# Sparse top-k decode inputs (DeepSeek-V3.2 record: index_topk 2048).  The
# indexer's output is stood in for by seeded random picks: each query row
# (b, i) gets up to topk distinct tokens drawn uniformly from the tokens
# visible to it in its own context (the first seq_len - (Sq-1-i) tokens of
# row b), given as physical cache slots (page * 64 + offset, read off the
# block table) in a random order, padded with -1 when fewer than topk are
# visible.
# --------------------------------------------------------------------------

@dataclass
class SparseInputs:
    dense: DecodeInputs          # cache, queries, context block table and lengths
    token_slots: torch.Tensor    # int32 [B, Sq, topk]: cache slot or -1
    topk: int
    name: str = ""

    @property
    def batch(self) -> int:
        return self.dense.batch

    @property
    def sq(self) -> int:
        return self.dense.sq


def make_sparse_inputs(batch: int, sq: int, context_lens, topk: int, kv_dtype: str = "bf16",
                       seed: int = 0, pad_middle: bool = False, name: str = "") -> SparseInputs:
    """Seeded sparse decode problem.  pad_middle: also scatter a few -1
    entries inside the list (a stress case for the masking)."""
    dense = make_inputs(batch, sq, context_lens, kv_dtype=kv_dtype, seed=seed)
    gen = torch.Generator().manual_seed(int(seed) * 31 + 7)
    slots = torch.full((batch, sq, topk), -1, dtype=torch.int32)
    bt = dense.block_table.to(torch.int64)
    for b in range(batch):
        for i in range(sq):
            vis = int(dense.seq_lens[b]) - (sq - 1 - i)
            if vis <= 0:
                continue
            n = min(vis, topk)
            pos = torch.randperm(vis, generator=gen)[:n]
            s = bt[b, pos // PAGE_SIZE] * PAGE_SIZE + pos % PAGE_SIZE
            slots[b, i, :n] = s.to(torch.int32)
            if pad_middle and n > 4:
                holes = torch.randperm(n, generator=gen)[: max(1, n // 16)]
                slots[b, i, holes] = -1
            slots[b, i] = slots[b, i, torch.randperm(topk, generator=gen)]
    return SparseInputs(dense=dense, token_slots=slots, topk=int(topk), name=name)


SPARSE_WORKLOADS = {
    6: dict(name="sparse top-2048 B64 Sq1 over 32K contexts bf16", batch=64, sq=1, context=32768,
            topk=2048, kv_dtype="bf16"),
}


def make_sparse_workload(workload: int) -> SparseInputs:
    w = SPARSE_WORKLOADS[workload]
    return make_sparse_inputs(w["batch"], w["sq"], [w["context"]] * w["batch"], w["topk"],
                              kv_dtype=w["kv_dtype"], seed=seed_for(workload), name=w["name"])


def sparse_counts(inp: SparseInputs) -> dict:
    """Units of work of a sparse problem: listed tokens (query, token pairs),
    algorithmic bytes (each listed cache row once, q, out, lse, the slot
    lists) and FLOPs."""
    d = inp.dense
    H = int(d.q_absorbed.shape[2])
    row_bytes = row_bytes_of(d.kv_dtype)
    pairs = int((inp.token_slots >= 0).sum())
    rows = inp.batch * inp.sq
    bytes_ = (pairs * row_bytes + rows * H * (D_LATENT + D_ROPE) * 2 + rows * H * D_LATENT * 2 + rows * H * 4
              + inp.token_slots.numel() * 4)
    flops = pairs * 2 * H * (ROW_ELEMS + D_LATENT)
    return dict(kv_tokens=pairs, query_token_pairs=pairs, bytes=bytes_, flops=flops, kv_bytes=pairs * row_bytes)
