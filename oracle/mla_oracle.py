"""Float64 MLA decode attention over a paged latent cache: the plain definition.

TEST INFRASTRUCTURE ONLY (see the package docstring).

What is computed ("DeepSeek R1 Architecture & Deployment Guide", section 1.1,
matrix absorption and decoupled RoPE):

  Each cached token j holds the row R_j = [c_j^KV (512) | k_j^R (64)].  The
  key up-projection W_i^UK is folded into the query, so head i's score is
      s_ij = scale * ( q_i^absorbed . c_j^KV  +  q_i^rope . k_j^R )
  and the value up-projection W_i^UV is folded into the output projection, so
  the attention output stays in the 512-d latent space:
      out_i = sum_j softmax_j(s_ij) c_j^KV,     lse_i = ln sum_j exp(s_ij).

Readings where the pages are silent (listed again in the design notes):
  * scale is a parameter (1/sqrt(128+64) in the workloads), applied inside the
    exponent and inside the LSE (natural log);
  * V is c^KV only; k^R takes part in the scores alone;
  * rows arrive already rotated: nothing here applies RoPE;
  * query i of Sq sees the first seq_len - (Sq - 1 - i) tokens;
  * a row with no visible token gives out = 0 and lse = -inf;
  * cache page p, slot t holds token p_index*64 + t of the row whose block
    table lists p at p_index (page-block size 64, "DeepSeek-R1" record,
    engine kernel constraint (1)); tokens past the visible length are never
    read, whatever a partly used page holds.

The un-absorbed form (section 1: k^C = W^UK c^KV, v^C = W^UV c^KV per head,
then ordinary attention) is written separately so the absorption identity
can be checked between two independent computations.
"""
from __future__ import annotations

import numpy as np

from .fp8_codec import dequant_blocks, dequant_rows, dequant_rows_v41, split_e4m3_terms
from . import fp4_codec

D_LATENT = 512
D_ROPE = 64
ROW = D_LATENT + D_ROPE


def visible_len(seq_len: int, sq: int, i: int) -> int:
    """Tokens visible to query i of an Sq-token speculative query block."""
    return int(seq_len) - (int(sq) - 1 - int(i))


def cache_rows(kv_cache: np.ndarray, kv_dtype: str) -> np.ndarray:
    """The cache as float64 rows [P, page, 576]: bf16 caches arrive already
    widened to float64 by the caller; FP8 (594- and 528-byte rows) and FP4
    (324- and 288-byte rows) caches are decoded here."""
    if kv_dtype == "fp8":
        return dequant_rows(kv_cache)
    if kv_dtype == "fp8v41":
        return dequant_rows_v41(kv_cache)
    if kv_dtype == "fp4":
        return fp4_codec.dequant_rows(kv_cache)
    if kv_dtype == "fp4v41":
        return fp4_codec.dequant_rows_v41(kv_cache)
    arr = np.asarray(kv_cache, dtype=np.float64)
    assert arr.shape[-1] == ROW
    return arr


def gather_rows(rows: np.ndarray, block_table_row: np.ndarray, n: int) -> np.ndarray:
    """Token j of the row lives at page block_table_row[j // page], slot
    j % page.  Returns [n, 576]."""
    page = rows.shape[1]
    j = np.arange(int(n))
    pages = np.asarray(block_table_row, dtype=np.int64)[j // page]
    return rows[pages, j % page]


def attend_latent(q_abs: np.ndarray, q_rope: np.ndarray, rows: np.ndarray,
                  scale: float):
    """Absorbed-form attention of H query heads over n gathered rows.

    q_abs [H, 512], q_rope [H, 64], rows [n, 576] -> out [H, 512], lse [H].
    """
    q_abs = np.asarray(q_abs, dtype=np.float64)
    q_rope = np.asarray(q_rope, dtype=np.float64)
    H = q_abs.shape[0]
    n = rows.shape[0]
    if n <= 0:
        return np.zeros((H, D_LATENT)), np.full(H, -np.inf)
    c_kv = rows[:, :D_LATENT]
    k_r = rows[:, D_LATENT:]
    s = scale * (q_abs @ c_kv.T + q_rope @ k_r.T)          # [H, n]
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    lse = m[:, 0] + np.log(l[:, 0])
    p = e / l
    return p @ c_kv, lse


def mla_decode(q_abs: np.ndarray, q_rope: np.ndarray, rows: np.ndarray,
               block_table: np.ndarray, seq_lens: np.ndarray, scale: float,
               query_rows=None):
    """Decode for a batch.

    q_abs [B, Sq, H, 512], q_rope [B, Sq, H, 64] (float64), rows: the cache as
    float64 [P, page, 576] (see cache_rows), block_table [B, max_pages],
    seq_lens [B].  query_rows: optional iterable of (b, i) to compute; the
    others are left NaN.  Returns out [B, Sq, H, 512], lse [B, Sq, H].
    """
    B, Sq, H, _ = q_abs.shape
    out = np.full((B, Sq, H, D_LATENT), np.nan)
    lse = np.full((B, Sq, H), np.nan)
    todo = query_rows if query_rows is not None else [
        (b, i) for b in range(B) for i in range(Sq)]
    for b, i in todo:
        n = max(visible_len(seq_lens[b], Sq, i), 0)
        g = gather_rows(rows, block_table[b], n)
        out[b, i], lse[b, i] = attend_latent(q_abs[b, i], q_rope[b, i], g, scale)
    return out, lse


def query_as_e4m3_terms(q_abs: np.ndarray, q_rope: np.ndarray, terms: int = 2):
    """The query a block-scaled FP8 score product would see.

    Each head's 576-value row [q_abs | q_rope] is split into e4m3 terms with
    one e8m0 scale per 32 values (fp8_codec.split_e4m3_terms: the scale
    groups are the cache row's, so group k of the query meets group k of
    the key).  terms=1 keeps the first term alone, terms=2 their sum.
    Returns the float64 value, split back into its 512 and 64 parts; decoding
    with it is mla_decode / attend_latent on these arrays.
    """
    q = np.concatenate([np.asarray(q_abs, dtype=np.float64), np.asarray(q_rope, dtype=np.float64)], axis=-1)
    hi, lo = split_e4m3_terms(q)
    v = dequant_blocks(*hi) + (dequant_blocks(*lo) if terms == 2 else 0.0)
    return v[..., :D_LATENT], v[..., D_LATENT:]


def merge_partials(outs: np.ndarray, lses: np.ndarray):
    """Combine attention over disjoint key sets from per-part normalised
    outputs and LSEs: L = ln sum_s e^{lse_s}, out = sum_s e^{lse_s - L} out_s.

    outs [k, H, D], lses [k, H] -> out [H, D], lse [H].
    """
    lses = np.asarray(lses, dtype=np.float64)
    L = np.logaddexp.reduce(lses, axis=0)
    finite = np.isfinite(L)
    w = np.where(finite[None, :], np.exp(lses - np.where(finite, L, 0.0)[None, :]), 0.0)
    out = np.einsum("kh,khd->hd", w, np.asarray(outs, dtype=np.float64))
    return out, L


def absorb_query(q_nope: np.ndarray, w_uk: np.ndarray) -> np.ndarray:
    """q_i^absorbed = (W_i^UK)^T q_i for W_i^UK in R^{d_h x d_c}.
    q_nope [H, d_h], w_uk [H, d_h, d_c] -> [H, d_c]."""
    return np.einsum("hkc,hk->hc", w_uk, q_nope)


def attend_unabsorbed(q_nope: np.ndarray, q_rope: np.ndarray, c_kv: np.ndarray,
                      k_rope: np.ndarray, w_uk: np.ndarray, w_uv: np.ndarray,
                      scale: float):
    """Ordinary per-head attention with explicit up-projected keys and values.

    k_{j,i} = W_i^UK c_j, v_{j,i} = W_i^UV c_j; head i scores
    s_ij = scale * (q_i . k_{j,i} + q_i^rope . k_j^R); output o_i = sum_j p_ij v_{j,i}.
    q_nope [H, d_h], q_rope [H, 64], c_kv [n, 512], k_rope [n, 64],
    w_uk, w_uv [H, d_h, 512].  Returns o [H, d_h], lse [H].
    """
    H, d_h = q_nope.shape
    o = np.zeros((H, d_h))
    lse = np.zeros(H)
    for h in range(H):
        k = c_kv @ w_uk[h].T            # [n, d_h]
        v = c_kv @ w_uv[h].T            # [n, d_h]
        s = scale * (k @ q_nope[h] + k_rope @ q_rope[h])
        m = s.max()
        e = np.exp(s - m)
        l = e.sum()
        lse[h] = m + np.log(l)
        o[h] = (e / l) @ v
    return o, lse


def up_project_output(out_latent: np.ndarray, w_uv: np.ndarray) -> np.ndarray:
    """Apply W_i^UV to the latent output of each head: [H, 512] -> [H, d_h]."""
    return np.einsum("hkc,hc->hk", w_uv, out_latent)


# --------------------------------------------------------------------------
# Sparse top-k decode ("DeepSeek-V3.2" record: the sparse attention indexer,
# config index_topk 2048 -- a lightweight selector picks a candidate set of
# cached tokens and attention runs over that set instead of the whole
# context; the latent rows are cached per token as before).
#
# Readings where the record is silent (listed again in the design notes):
#   * the selector's output reaches the attention as, per query row, a list
#     of topk physical cache slots, slot = page * page_size + offset into the
#     paged cache; -1 means "no token" (fewer candidates than topk);
#   * attention runs over the listed tokens as given: no further causal
#     mask, and a slot listed twice counts twice;
#   * scale, LSE and the empty-row convention are those of the dense decode.
# --------------------------------------------------------------------------

def sparse_gather_rows(rows: np.ndarray, slots: np.ndarray) -> np.ndarray:
    """The rows of the listed cache slots, in list order, skipping -1.
    rows [P, page, 576]; slots [topk] int -> [n, 576]."""
    flat = rows.reshape(-1, rows.shape[-1])
    s = np.asarray(slots, dtype=np.int64)
    s = s[s >= 0]
    assert np.all(s < flat.shape[0]), "slot past the cache"
    return flat[s]


def mla_decode_sparse(q_abs: np.ndarray, q_rope: np.ndarray, rows: np.ndarray,
                      token_slots: np.ndarray, scale: float, query_rows=None):
    """Sparse decode: query row (b, i) attends over the cache slots
    token_slots[b, i, :] (see the readings above).

    q_abs [B, Sq, H, 512], q_rope [B, Sq, H, 64], rows [P, page, 576] as in
    cache_rows, token_slots [B, Sq, topk].  Returns out [B, Sq, H, 512],
    lse [B, Sq, H] (rows not in query_rows are left NaN).
    """
    B, Sq, H, _ = q_abs.shape
    out = np.full((B, Sq, H, D_LATENT), np.nan)
    lse = np.full((B, Sq, H), np.nan)
    todo = query_rows if query_rows is not None else [
        (b, i) for b in range(B) for i in range(Sq)]
    for b, i in todo:
        g = sparse_gather_rows(rows, token_slots[b, i])
        out[b, i], lse[b, i] = attend_latent(q_abs[b, i], q_rope[b, i], g, scale)
    return out, lse
