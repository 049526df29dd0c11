// Shared constants, the workspace layout of the split-KV plan, and bounded
// waits for the MLA decode kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

#include "mla_decode.h"
#include "ptx.cuh"

namespace mla {

constexpr int kHeads = 128;
constexpr int kDc = 512;            // latent c_KV
constexpr int kDr = 64;             // decoupled RoPE key
constexpr int kRow = kDc + kDr;     // 576 values per cached token
constexpr int kPage = 64;           // tokens per page (= tokens per KV tile)
constexpr int kFp8Row = kRow + kRow / 32;   // 594 bytes
constexpr int kFp4Codes = kRow / 2;         // FP4 row: 288 bytes of e2m1 codes (two per byte) ...
constexpr int kFp4Row = kFp4Codes + kRow / 16;   // ... then 36 e8m0 scales (one per 16 values): 324 bytes
// FP8 V4.1 row: 512 e4m3 codes (448 latent, then the 64 RoPE values) and 16
// e8m0 scales (one per 32 codes): 528 bytes.  On the 576-value row the V4.1
// latent fills dims [0, 448) and dims [448, 512) are zero.
constexpr int kV41Values = 512;
constexpr int kV41Latent = 448;
constexpr int kV41Row = kV41Values + kV41Values / 32;   // 528 bytes
// FP4 V4.1 row: 512 e2m1 codes (two per byte), then 32 e8m0 scales (one per
// 16 values): 288 bytes, the same value order.
constexpr int kV41Fp4Row = kV41Values / 2 + kV41Values / 16;   // 288 bytes
constexpr int kMaxSq = 4;
constexpr int kMaxRows = 1 << 16;   // batch * Sq handled by the planner

// Plan header at workspace offset 0.
struct PlanHeader {
  int status;            // first device-side problem seen (0 = none)
  int n_tiles;           // total KV tiles over the batch (longest query)
  int chunk;             // mean pages per pair (information only; the ranges are pair_lo)
  int slots_per_query;   // partial slots of one query index
  int n_empty;           // rows with no token (written by the planner)
  int pairs_per_group;   // pairs that serve one query index
  int abort_flag;        // set by the first wait that times out; all waits then give up
  int fp8_range;         // FP8/FP4 f16 pass: an input lies outside the f16-exact range (the exact pass recomputes)
  int pad[8];
};

// Offsets (bytes) of the plan arrays and split partials inside the workspace.
struct WsLayout {
  size_t lens, tile_start, row_cost, pair_lo, pair_rank, pair_b0, first_pair, slot_base, n_parts, empty_rows;
  size_t part_lse, part_out;
  size_t sp_lens, sp_slots;   // sparse decode: listed tokens per row, compacted slot lists [rows, topk]
  size_t total;
  int max_slots;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// topk > 0: the sparse decode's extra arrays (its rows are batch * sq query
// rows, planned as a batch of that many rows with one query each)
__host__ __device__ inline WsLayout ws_layout(int batch, int sq, int pairs, int topk = 0) {
  WsLayout L;
  const int pg = pairs / sq > 0 ? pairs / sq : 1;
  // every pair boundary splits at most one row: slots per query <= 2*(pg-1)
  L.max_slots = sq * 2 * pg;
  size_t o = align256(sizeof(PlanHeader));
  L.lens = o;        o = align256(o + sizeof(int) * batch);
  L.tile_start = o;  o = align256(o + sizeof(int) * (batch + 1));
  L.row_cost = o;    o = align256(o + sizeof(int) * (batch + 1));
  L.pair_lo = o;     o = align256(o + sizeof(int) * (pg + 1));
  L.pair_rank = o;   o = align256(o + sizeof(int) * (pg + 1));
  L.pair_b0 = o;     o = align256(o + sizeof(int) * (pg + 1));
  L.first_pair = o;  o = align256(o + sizeof(int) * batch);
  L.slot_base = o;   o = align256(o + sizeof(int) * batch);
  L.n_parts = o;     o = align256(o + sizeof(int) * batch);
  L.empty_rows = o;  o = align256(o + sizeof(int) * batch);
  L.part_lse = o;    o = align256(o + sizeof(float) * static_cast<size_t>(L.max_slots) * kHeads);
  L.part_out = o;    o = align256(o + 2 * static_cast<size_t>(L.max_slots) * kHeads * kDc);   // bf16 partials
  L.sp_lens = o;     o = align256(o + (topk > 0 ? sizeof(int) * batch : 0));
  L.sp_slots = o;    o = align256(o + (topk > 0 ? sizeof(int) * static_cast<size_t>(batch) * topk : 0));
  L.total = o;
  return L;
}

// Launch `kern` and return this launch's own error.  (A <<<>>> launch is
// checked through cudaGetLastError, which would also return, and clear, an
// earlier error of the caller's.)
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Record the first problem seen (never overwrites an earlier one).
__device__ __forceinline__ void set_status(int* status, int code) {
  atomicCAS(status, 0, code);
}

__device__ __forceinline__ int read_status(const int* status) {
  return *reinterpret_cast<const volatile int*>(status);
}

#ifndef MLA_WAIT_TIMEOUT_NS
#define MLA_WAIT_TIMEOUT_NS 2000000000ull   // 2 s: far beyond any legal wait
#endif

// Bounded mbarrier wait.  Returns false (after recording MLA_STATUS_TIMEOUT)
// if the phase did not complete within the time limit, or if another thread
// of the grid already gave up; the caller then leaves its loop.
// `hdr` is the plan header in global memory.
template <bool kCluster>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, PlanHeader* hdr) {
  auto poll = [&]() {
    return kCluster ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity);
  };
  if (poll()) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t n = 1;; ++n) {
    if (poll()) return true;
    if ((n & 255u) == 0) {
      if (read_status(&hdr->abort_flag) != 0) return false;
      if (ptx::globaltimer() - t0 > MLA_WAIT_TIMEOUT_NS) {
        set_status(&hdr->status, MLA_STATUS_TIMEOUT);
        atomicExch(&hdr->abort_flag, 1);
        return false;
      }
    }
  }
}

// Time limit of the teardown drains below.  It does not follow
// MLA_WAIT_TIMEOUT_NS: a drain waits for copies and MMAs that were already
// issued and complete on their own, whatever happened to the pipeline.
constexpr uint64_t kDrainTimeoutNs = 200000000ull;   // 200 ms

// Wait until the phase with `parity` of a barrier has completed, i.e. until
// the copies or MMAs counted on it have landed, ignoring the abort flag.
// Gives up (recording MLA_STATUS_TIMEOUT) only after kDrainTimeoutNs.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, PlanHeader* hdr) {
  if (ptx::mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > kDrainTimeoutNs) {
      set_status(&hdr->status, MLA_STATUS_TIMEOUT);
      return;
    }
  }
}

// Spin for `ns` nanoseconds (the abort path's grace for stores another CTA
// of the cluster issued into this one's shared memory and cannot track).
__device__ __forceinline__ void spin_ns(uint64_t ns) {
  const uint64_t t0 = ptx::globaltimer();
  while (ptx::globaltimer() - t0 < ns) {
  }
}

// Warp-uniform bounded wait: every lane polls (so every lane acquires the
// phase), and the warp leaves together if any lane gave up.
template <bool kCluster>
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, PlanHeader* hdr) {
  const bool ok = wait_bounded<kCluster>(bar, parity, hdr);
  return __all_sync(0xffffffffu, ok);
}

}  // namespace mla
