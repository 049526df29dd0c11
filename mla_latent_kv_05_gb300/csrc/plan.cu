// Split-KV planner: turns seq_lens (on the device, no host sync) into an even
// partition of KV tiles over the persistent CTA pairs and the partial-output
// slots of rows that end up split.  One CTA of 128 to 1024 threads; the arrays it
// searches are mirrored in shared memory, because a chain of dependent
// global reads would sit on the call's critical path (the attention kernel
// waits for this grid).
//
// Partition: every batch row b has n_b = ceil(seq_len_b / 64) pages.  The
// rows' pages are laid end to end (prefix sums tile_start) and cut into one
// contiguous range per pair of a query group, [pair_lo[p], pair_lo[p+1]).
// The cut balances cost, not pages: a pair's cost is its pages plus a fixed
// cost for every row segment it starts (query load, output write, pipeline
// refill), so a pair that crosses more row starts gets fewer pages.  Each
// query index i < Sq has its own group of pairs with the identical
// partition, so the groups read the same pages at about the same time and
// share them in L2.  A row covered by one pair is written straight to `out`;
// a row covered by k > 1 pairs gets k partial slots (per query index),
// which the merge kernel combines.  The planner writes the rows that have no
// token (out = 0, lse = -inf), which neither kernel visits.
#include <cuda_bf16.h>

#include "common.cuh"

namespace mla {

namespace {

// Cost of starting a row segment, in pages.  Tuned on GB300 by timing the
// attention kernel over 3..24: 8..12 are best on the ragged, uniform and
// long causal workloads alike (a segment start costs a query load, a
// pipeline refill and an output drain, about 10 us against 1.2 us per page).
constexpr int kSegCost = 10;

__device__ int block_exclusive_scan(int v, int* smem_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) smem_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < static_cast<int>(blockDim.x >> 5)) ? smem_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    smem_warp[lane] = w;   // inclusive scan of warp totals
  }
  __syncthreads();
  const int warp_excl = warp > 0 ? smem_warp[warp - 1] : 0;
  *total = smem_warp[(blockDim.x >> 5) - 1];
  __syncthreads();
  return warp_excl + x - v;
}

// Exclusive block scan of two non-negative counts at once (one round of
// barriers): a and b are packed into one 64-bit word, a in the high half.
// Both sums stay below 2^31, as the planner's int totals already require, so
// b never carries into a.
__device__ void block_exclusive_scan2(int a, int b, unsigned long long* smem_warp, int* ex_a, int* ex_b, int* tot_a,
                                      int* tot_b) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned long long v = (static_cast<unsigned long long>(static_cast<unsigned>(a)) << 32) |
                               static_cast<unsigned>(b);
  unsigned long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) smem_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    unsigned long long w = (lane < static_cast<int>(blockDim.x >> 5)) ? smem_warp[lane] : 0ull;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    smem_warp[lane] = w;   // inclusive scan of warp totals
  }
  __syncthreads();
  const unsigned long long ex = (warp > 0 ? smem_warp[warp - 1] : 0ull) + x - v;
  const unsigned long long tot = smem_warp[(blockDim.x >> 5) - 1];
  *ex_a = static_cast<int>(ex >> 32);
  *ex_b = static_cast<int>(ex & 0xFFFFFFFFull);
  *tot_a = static_cast<int>(tot >> 32);
  *tot_b = static_cast<int>(tot & 0xFFFFFFFFull);
  __syncthreads();
}

// Rows whose planner arrays (tile starts and costs) are kept in shared
// memory while the planner searches them; larger batches search the global
// copies instead (the same result, with longer dependent reads).
constexpr int kPlanSmemRows = 2048;   // 4 mirrors of [batch + 1] ints: 32 KiB, under the 48 KiB default

__global__ void __launch_bounds__(1024) plan_kernel(const int32_t* __restrict__ seq_lens, int batch, int sq,
                                                    int max_pages, int pairs_per_group,
                                                    uint8_t* __restrict__ ws, WsLayout L,
                                                    __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
  __shared__ int s_warp[32];
  __shared__ unsigned long long s_warp2[32];
  __shared__ int s_chunk;
  // dynamic: pair_lo and pair_rank mirrors [ppg + 1] each, then (batch <=
  // kPlanSmemRows) tile_start and row_cost mirrors [batch + 1] each and the
  // rows' clamped lengths and part counts [batch] each
  extern __shared__ int s_dyn[];
  PlanHeader* hdr = reinterpret_cast<PlanHeader*>(ws);
  int* lens = reinterpret_cast<int*>(ws + L.lens);
  int* tile_start = reinterpret_cast<int*>(ws + L.tile_start);
  int* pair_lo = reinterpret_cast<int*>(ws + L.pair_lo);
  int* pair_rank = reinterpret_cast<int*>(ws + L.pair_rank);
  int* pair_b0 = reinterpret_cast<int*>(ws + L.pair_b0);
  int* first_pair = reinterpret_cast<int*>(ws + L.first_pair);
  int* slot_base = reinterpret_cast<int*>(ws + L.slot_base);
  int* n_parts = reinterpret_cast<int*>(ws + L.n_parts);
  int* empty_rows = reinterpret_cast<int*>(ws + L.empty_rows);
  const int ppg = pairs_per_group;
  int* s_lo = s_dyn;
  int* s_rank = s_dyn + (ppg + 1);
  const bool rows_in_smem = batch <= kPlanSmemRows;
  int* r_ts = rows_in_smem ? s_dyn + 2 * (ppg + 1) : tile_start;
  int* r_cost = rows_in_smem ? r_ts + (batch + 1) : reinterpret_cast<int*>(ws + L.row_cost);
  int* r_len = rows_in_smem ? r_cost + (batch + 1) : lens;
  int* r_parts = rows_in_smem ? r_len + batch : n_parts;

  const int tid = threadIdx.x;
  // This grid is a programmatic dependent of whatever precedes it in the
  // stream (seq_lens may come from it, and the previous call's merge kernel
  // reads the plan arrays): nothing is read or written before the wait.
  ptx::grid_dep_wait();
  // the attention kernel may begin its prologue now; it reads the plan only
  // after this grid has completed (griddepcontrol.wait)
  ptx::grid_dep_launch();
  const int per = (batch + blockDim.x - 1) / blockDim.x;
  const int lo = min(batch, tid * per), hi = min(batch, lo + per);
  const int max_len = max_pages * kPage;

  // pass 1: clamp lengths, tiles per row, prefix sums
  int local = 0, local_ne = 0;
  for (int b = lo; b < hi; ++b) {
    int s = seq_lens[b];
    if (s < 0 || s > max_len) {
      set_status(&hdr->status, MLA_STATUS_BAD_SEQ_LEN);
      s = s < 0 ? 0 : max_len;
    }
    lens[b] = s;
    r_len[b] = s;
    local += (s + kPage - 1) / kPage;
    local_ne += s > 0 ? 1 : 0;
  }
  // Row costs for the partition: a row with pages costs its pages plus
  // kSegCost pages' worth for its segment start (query load, output write,
  // pipeline refill).
  int total = 0, ne_total = 0, excl = 0, ne_excl = 0;
  block_exclusive_scan2(local, local_ne, s_warp2, &excl, &ne_excl, &total, &ne_total);
  for (int b = lo; b < hi; ++b) {
    const int n = (r_len[b] + kPage - 1) / kPage;
    r_ts[b] = excl;
    if (rows_in_smem) tile_start[b] = excl;
    r_cost[b] = excl + kSegCost * ne_excl;
    excl += n;
    ne_excl += n > 0 ? 1 : 0;
  }
  if (tid == 0) {
    r_ts[batch] = total;
    tile_start[batch] = total;
    r_cost[batch] = total + kSegCost * ne_total;
    s_chunk = total > 0 ? (total + ppg - 1) / ppg : 1;
  }
  __syncthreads();
  const int chunk = s_chunk;

  // Pair p starts where the cumulative cost reaches p/ppg of the total: in
  // the row whose cost range holds that point, past the row's start cost.
  // pair_b0[p]: the row holding the pair's first page (the last row whose
  // pages start at or before it), where the attention kernel begins walking.
  const long long cost_total = static_cast<long long>(total) + static_cast<long long>(kSegCost) * ne_total;
  for (int pp = tid; pp <= ppg; pp += blockDim.x) {
    int x = pp == 0 ? 0 : total;
    if (pp > 0 && pp < ppg) {
      const long long target = cost_total * pp / ppg;
      int l = 0, r = batch - 1;            // largest row with row_cost <= target
      while (l < r) {
        const int mid = (l + r + 1) >> 1;
        if (r_cost[mid] <= target) l = mid; else r = mid - 1;
      }
      const int n = r_ts[l + 1] - r_ts[l];
      const long long off = target - r_cost[l] - (n > 0 ? kSegCost : 0);
      x = r_ts[l] + static_cast<int>(off < 0 ? 0 : (off > n ? n : off));
    }
    s_lo[pp] = x;
    pair_lo[pp] = x;
    if (pp < ppg) {
      int l = 0, r = batch - 1;            // largest row with tile_start <= x
      while (l < r) {
        const int mid = (l + r + 1) >> 1;
        if (r_ts[mid] <= x) l = mid; else r = mid - 1;
      }
      pair_b0[pp] = l;
    }
  }
  __syncthreads();
  // pair_rank[p]: pairs before p that have pages.  A pair range can be empty
  // (its cost share falls inside a row's start cost); a split row's parts
  // are the non-empty pairs over it, numbered by rank.
  if (tid < 32) {
    int carry = 0;
    for (int base = 0; base <= ppg; base += 32) {
      const int pp = base + tid;
      const int ne = pp < ppg && s_lo[pp + 1] > s_lo[pp] ? 1 : 0;
      int x = ne;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (tid >= o) x += y;
      }
      if (pp <= ppg) {
        s_rank[pp] = carry + x - ne;
        pair_rank[pp] = carry + x - ne;
      }
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
  }
  __syncthreads();
  // the pair whose page range [pair_lo[p], pair_lo[p+1]) holds page t
  auto pair_of = [&](int t) {
    int l = 0, r = ppg - 1;
    while (l < r) {
      const int mid = (l + r + 1) >> 1;
      if (s_lo[mid] <= t) l = mid; else r = mid - 1;
    }
    return l;
  };

  // pass 2: pairs covering each row; slots for rows that are split
  local = 0;
  int local_empty = 0;
  for (int b = lo; b < hi; ++b) {
    const int n = (r_len[b] + kPage - 1) / kPage;
    int parts = 0, fp = 0;
    if (n > 0) {
      const int t0 = r_ts[b];
      fp = pair_of(t0);
      parts = s_rank[pair_of(t0 + n - 1) + 1] - s_rank[fp];
    }
    first_pair[b] = fp;
    n_parts[b] = parts;
    r_parts[b] = parts;
    local += parts > 1 ? parts : 0;
    local_empty += parts == 0 ? 1 : 0;
  }
  int slots_total = 0, empty_total = 0, slot_excl = 0, empty_excl = 0;
  block_exclusive_scan2(local, local_empty, s_warp2, &slot_excl, &empty_excl, &slots_total, &empty_total);
  for (int b = lo; b < hi; ++b) {
    const int parts = r_parts[b];
    slot_base[b] = parts > 1 ? slot_excl : -1;
    if (parts > 1) slot_excl += parts;
    if (parts == 0) empty_rows[empty_excl++] = b;
  }
  if (tid == 0) {
    hdr->n_tiles = total;
    hdr->chunk = chunk;
    hdr->slots_per_query = slots_total;
    hdr->n_empty = empty_total;
    hdr->pairs_per_group = ppg;
    hdr->abort_flag = 0;
    hdr->fp8_range = 0;
  }
  // Rows with no token: out = 0, lse = -inf for every query index (the
  // attention kernel has no page of theirs to visit).
  __syncthreads();
  constexpr int kRowVec = kHeads * kDc * 2 / 16;   // 16-byte stores per output row
  for (int k = 0; k < empty_total; ++k) {
    const int b = empty_rows[k];
    for (int i = 0; i < sq; ++i) {
      const size_t row = static_cast<size_t>(b) * sq + i;
      uint4* dst = reinterpret_cast<uint4*>(out + row * kHeads * kDc);
      for (int e = tid; e < kRowVec; e += blockDim.x) dst[e] = make_uint4(0, 0, 0, 0);
      if (tid < kHeads) lse[row * kHeads + tid] = -INFINITY;
    }
  }
}

// Sparse decode: one CTA per query row compacts the row's listed cache slots
// (list order kept, -1 entries dropped) into the workspace and counts them;
// the planner then treats the count as the row's length.  An entry outside
// [-1, num_slots) is dropped too and recorded as MLA_STATUS_BAD_INDEX.
__global__ void __launch_bounds__(256) sparse_prep_kernel(const int32_t* __restrict__ token_slots, int topk,
                                                          int num_slots, uint8_t* __restrict__ ws, WsLayout L) {
  __shared__ int s_warp[32];
  PlanHeader* hdr = reinterpret_cast<PlanHeader*>(ws);
  const int row = blockIdx.x;
  const int32_t* src = token_slots + static_cast<size_t>(row) * topk;
  int* dst = reinterpret_cast<int*>(ws + L.sp_slots) + static_cast<size_t>(row) * topk;
  int base = 0;
  for (int c0 = 0; c0 < topk; c0 += blockDim.x) {
    const int k = c0 + static_cast<int>(threadIdx.x);
    const int v = k < topk ? src[k] : -1;
    const bool ok = v >= 0 && v < num_slots;
    if (k < topk && !ok && v != -1) set_status(&hdr->status, MLA_STATUS_BAD_INDEX);
    int total = 0;
    const int pos = block_exclusive_scan(ok ? 1 : 0, s_warp, &total);
    if (ok) dst[base + pos] = v;
    base += total;
  }
  if (threadIdx.x == 0) reinterpret_cast<int*>(ws + L.sp_lens)[row] = base;
}

}  // namespace

cudaError_t launch_sparse_prep(const int32_t* token_slots, int rows, int topk, int num_slots, void* ws,
                               const WsLayout& L, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  return launch_kernel(sparse_prep_kernel, dim3(rows), dim3(256), 0, stream, token_slots, topk, num_slots,
                       static_cast<uint8_t*>(ws), L);
}

cudaError_t launch_plan(const int32_t* seq_lens, int batch, int sq, int max_pages, int pairs_per_group,
                        void* ws, const WsLayout& L, __nv_bfloat16* out, float* lse, cudaStream_t stream) {
  const size_t smem = sizeof(int) * (2 * static_cast<size_t>(pairs_per_group + 1) +
                                     (batch <= kPlanSmemRows ? 4 * static_cast<size_t>(batch + 1) : 0));
  // one thread per row (or pair boundary), at least four warps: a small
  // batch synchronises fewer warps at each of the planner's block barriers
  const int want = batch > pairs_per_group + 1 ? batch : pairs_per_group + 1;
  const int threads = want >= 1024 ? 1024 : (want <= 128 ? 128 : (want + 31) / 32 * 32);
  // a programmatic dependent of the previous kernel in the stream: its launch
  // overlaps that kernel's tail, and it waits for it before reading anything
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, plan_kernel, seq_lens, batch, sq, max_pages, pairs_per_group,
                            static_cast<uint8_t*>(ws), L, out, lse);
}

}  // namespace mla
