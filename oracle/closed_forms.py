"""Cache-size arithmetic stated on the pages, written out.

TEST INFRASTRUCTURE ONLY (see the package docstring).

  * "DeepSeek R1 Architecture & Deployment Guide", section 1: MHA cache for
    one 128K sequence = 2 (K and V) x 61 layers x 128 heads x 128 d_h x
    131,072 tokens x 2 bytes.
  * same guide, section 1.1: MLA cache row = concat(c_KV, k_R) = 512 + 64 =
    576 elements per token per layer; reduction vs MHA = 1 - 576/32,768; a
    128K bf16 sequence over 61 layers = 61 x 576 x 131,072 x 2 bytes.
  * "DeepSeek-R1" and "DeepSeek-V3.2" model records: 61 x 576 x 2 =
    70,272 B/token (68.6 KiB).
  * FP8 row used by this library: 576 e4m3 bytes + 18 e8m0 bytes; a page of
    64 tokens (page-block size 64, R1 record constraint (1)).
"""
from __future__ import annotations

LAYERS = 61
HEADS = 128
D_HEAD = 128
D_LATENT = 512
D_ROPE = 64
CONTEXT_128K = 131072
PAGE_SIZE = 64


def mla_elems_per_token_layer(d_latent: int = D_LATENT, d_rope: int = D_ROPE) -> int:
    return d_latent + d_rope


def mla_bytes_per_token(layers: int = LAYERS, bytes_per_elem: int = 2) -> int:
    return layers * mla_elems_per_token_layer() * bytes_per_elem


def mla_cache_bytes(seq: int = CONTEXT_128K, layers: int = LAYERS,
                    bytes_per_elem: int = 2) -> int:
    return layers * mla_elems_per_token_layer() * seq * bytes_per_elem


def mha_elems_per_token_layer(heads: int = HEADS, d_head: int = D_HEAD) -> int:
    return 2 * heads * d_head


def mha_cache_bytes(seq: int = CONTEXT_128K, layers: int = LAYERS,
                    heads: int = HEADS, d_head: int = D_HEAD,
                    bytes_per_elem: int = 2) -> int:
    return 2 * layers * heads * d_head * seq * bytes_per_elem


def mla_reduction_vs_mha() -> float:
    return 1.0 - mla_elems_per_token_layer() / mha_elems_per_token_layer()


def fp8_row_bytes(values: int = D_LATENT + D_ROPE, group: int = 32) -> int:
    return values + values // group


def fp8_page_bytes(page_size: int = PAGE_SIZE) -> int:
    return page_size * fp8_row_bytes()


def fp4_row_bytes(values: int = D_LATENT + D_ROPE, group: int = 16) -> int:
    """e2m1 codes, two per byte, plus one e8m0 byte per `group` values (the
    reading taken for the FP4 row): 288 for the record's 512-value row."""
    return values // 2 + values // group


def fp4_page_bytes(page_size: int = PAGE_SIZE) -> int:
    return page_size * fp4_row_bytes()
