"""Float64 CPU oracle for MLA decode over a paged compressed-latent KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports, links or runs this
package: only the tests, the smoke check and the benchmark's CPU-baseline arm
use it.  It shares no code with the CUDA path (no kernels, headers, tables or
helpers); the only module both sides use is the seeded input generator, which
holds no attention arithmetic.

Sources (web pages, cited by title and section):
  * "DeepSeek R1 Architecture & Deployment Guide", section 1 (MHA cache size),
    section 1.1 (matrix absorption, decoupled RoPE, 576-element cache row,
    98.24 % reduction, 9.21 GB at 128K), section 4 (e4m3 max normal 448).
  * "DeepSeek-R1" model record: 61 x 576 x 2 = 70,272 B/token; engine kernel
    constraints (1) page-block size 64 and (2) e4m3 latents with one e8m0
    scale per 32 values inlined in each token row, and an FP4 variant of
    288 B per 512-value row.
  * "DeepSeek-V3.2" model record: the same cache figures.

Modules:
  fp8_codec     e4m3 (OCP E4M3FN) and e8m0 decoders, FP8 row dequantisation;
                the e4m3 encoder and per-32 block quantiser of a query
  fp4_codec     e2m1 (OCP MX FP4) decoder, FP4 row dequantisation
  mla_oracle    absorbed and un-absorbed attention, paged gather, LSE merge,
                the query as two e4m3 terms
  closed_forms  the pages' cache-size arithmetic

Every function here is pinned by a CPU test against something other than
itself (closed forms printed on the pages, torch's float8 casts, torch's
scaled-dot-product attention in float64, the absorption identity, brute-force
special cases and invariants).  No function is "parity unpinned".
"""
from . import closed_forms, fp4_codec, fp8_codec, mla_oracle  # noqa: F401
