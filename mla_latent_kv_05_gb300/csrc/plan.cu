// Split-KV planner: turns seq_lens (on the device, no host sync) into an even
// partition of KV tiles over the persistent CTA pairs, the partial-output
// slots of rows that end up split, and the list of rows the merge kernel
// writes.  One CTA of 1024 threads.
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
// a row covered by k > 1 pairs gets k partial slots (per query index) and a
// merge entry.
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

__global__ void __launch_bounds__(1024) plan_kernel(const int32_t* __restrict__ seq_lens, int batch, int sq,
                                                    int max_pages, int pairs_per_group,
                                                    uint8_t* __restrict__ ws, WsLayout L) {
  __shared__ int s_warp[32];
  __shared__ int s_chunk;
  PlanHeader* hdr = reinterpret_cast<PlanHeader*>(ws);
  int* lens = reinterpret_cast<int*>(ws + L.lens);
  int* tile_start = reinterpret_cast<int*>(ws + L.tile_start);
  int* row_cost = reinterpret_cast<int*>(ws + L.row_cost);
  int* pair_lo = reinterpret_cast<int*>(ws + L.pair_lo);
  int* pair_rank = reinterpret_cast<int*>(ws + L.pair_rank);
  int* first_pair = reinterpret_cast<int*>(ws + L.first_pair);
  int* slot_base = reinterpret_cast<int*>(ws + L.slot_base);
  int* comb_row = reinterpret_cast<int*>(ws + L.comb_row);
  int* comb_start = reinterpret_cast<int*>(ws + L.comb_start);
  int* comb_count = reinterpret_cast<int*>(ws + L.comb_count);

  const int tid = threadIdx.x;
  // the attention kernel may begin its prologue now; it reads the plan only
  // after this grid has completed (griddepcontrol.wait)
  ptx::grid_dep_launch();
  const int per = (batch + blockDim.x - 1) / blockDim.x;
  const int lo = min(batch, tid * per), hi = min(batch, lo + per);
  const int max_len = max_pages * kPage;

  // pass 1: clamp lengths, tiles per row, prefix sums
  int local = 0;
  for (int b = lo; b < hi; ++b) {
    int s = seq_lens[b];
    if (s < 0 || s > max_len) {
      set_status(&hdr->status, MLA_STATUS_BAD_SEQ_LEN);
      s = s < 0 ? 0 : max_len;
    }
    lens[b] = s;
    local += (s + kPage - 1) / kPage;
  }
  int total = 0;
  int excl = block_exclusive_scan(local, s_warp, &total);
  for (int b = lo; b < hi; ++b) {
    tile_start[b] = excl;
    excl += (lens[b] + kPage - 1) / kPage;
  }
  // Row costs for the partition: a row with pages costs its pages plus
  // kSegCost pages' worth for its segment start (query load, output write,
  // pipeline refill).
  int local_ne = 0;
  for (int b = lo; b < hi; ++b) local_ne += lens[b] > 0 ? 1 : 0;
  int ne_total = 0;
  int ne_excl = block_exclusive_scan(local_ne, s_warp, &ne_total);
  for (int b = lo; b < hi; ++b) {
    row_cost[b] = tile_start[b] + kSegCost * ne_excl;
    ne_excl += lens[b] > 0 ? 1 : 0;
  }
  if (tid == 0) {
    tile_start[batch] = total;
    row_cost[batch] = total + kSegCost * ne_total;
    s_chunk = total > 0 ? (total + pairs_per_group - 1) / pairs_per_group : 1;
  }
  __syncthreads();
  const int chunk = s_chunk;

  // Pair p starts where the cumulative cost reaches p/ppg of the total: in
  // the row whose cost range holds that point, past the row's start cost.
  const long long cost_total = static_cast<long long>(total) + static_cast<long long>(kSegCost) * ne_total;
  for (int pp = tid; pp <= pairs_per_group; pp += blockDim.x) {
    int x = pp == 0 ? 0 : total;
    if (pp > 0 && pp < pairs_per_group) {
      const long long target = cost_total * pp / pairs_per_group;
      int l = 0, r = batch - 1;            // largest row with row_cost <= target
      while (l < r) {
        const int mid = (l + r + 1) >> 1;
        if (row_cost[mid] <= target) l = mid; else r = mid - 1;
      }
      const int n = tile_start[l + 1] - tile_start[l];
      const long long off = target - row_cost[l] - (n > 0 ? kSegCost : 0);
      x = tile_start[l] + static_cast<int>(off < 0 ? 0 : (off > n ? n : off));
    }
    pair_lo[pp] = x;
  }
  __syncthreads();
  // pair_rank[p]: pairs before p that have pages.  A pair range can be empty
  // (its cost share falls inside a row's start cost); a split row's parts
  // are the non-empty pairs over it, numbered by rank.
  if (tid < 32) {
    int carry = 0;
    for (int base = 0; base <= pairs_per_group; base += 32) {
      const int pp = base + tid;
      const int ne = pp < pairs_per_group && pair_lo[pp + 1] > pair_lo[pp] ? 1 : 0;
      int x = ne;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (tid >= o) x += y;
      }
      if (pp <= pairs_per_group) pair_rank[pp] = carry + x - ne;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
  }
  __syncthreads();
  // the pair whose page range [pair_lo[p], pair_lo[p+1]) holds page t
  auto pair_of = [&](int t) {
    int l = 0, r = pairs_per_group - 1;
    while (l < r) {
      const int mid = (l + r + 1) >> 1;
      if (pair_lo[mid] <= t) l = mid; else r = mid - 1;
    }
    return l;
  };

  // pass 2: pairs covering each row; slots for rows that are split
  local = 0;
  int local_comb = 0;
  for (int b = lo; b < hi; ++b) {
    const int n = (lens[b] + kPage - 1) / kPage;
    int parts = 0, fp = 0;
    if (n > 0) {
      fp = pair_of(tile_start[b]);
      parts = pair_rank[pair_of(tile_start[b] + n - 1) + 1] - pair_rank[fp];
    }
    first_pair[b] = fp;
    local += parts > 1 ? parts : 0;
    local_comb += (parts != 1) ? 1 : 0;
  }
  int slots_total = 0;
  int slot_excl = block_exclusive_scan(local, s_warp, &slots_total);
  int comb_total = 0;
  int comb_excl = block_exclusive_scan(local_comb, s_warp, &comb_total);
  for (int b = lo; b < hi; ++b) {
    const int n = (lens[b] + kPage - 1) / kPage;
    int parts = 0;
    if (n > 0) parts = pair_rank[pair_of(tile_start[b] + n - 1) + 1] - pair_rank[first_pair[b]];
    slot_base[b] = parts > 1 ? slot_excl : -1;
    if (parts != 1) {
      for (int i = 0; i < sq; ++i) {
        const int k = comb_excl * sq + i;
        comb_row[k] = b * sq + i;
        comb_start[k] = parts > 1 ? i * slots_total + slot_excl : 0;
        comb_count[k] = parts > 1 ? parts : 0;
      }
      ++comb_excl;
    }
    if (parts > 1) slot_excl += parts;
  }
  if (tid == 0) {
    hdr->n_tiles = total;
    hdr->chunk = chunk;
    hdr->slots_per_query = slots_total;
    hdr->n_comb = comb_total * sq;
    hdr->pairs_per_group = pairs_per_group;
    hdr->abort_flag = 0;
    hdr->fp8_range = 0;
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
  sparse_prep_kernel<<<rows, 256, 0, stream>>>(token_slots, topk, num_slots, static_cast<uint8_t*>(ws), L);
  return cudaGetLastError();
}

cudaError_t launch_plan(const int32_t* seq_lens, int batch, int sq, int max_pages, int pairs_per_group,
                        void* ws, const WsLayout& L, cudaStream_t stream) {
  plan_kernel<<<1, 1024, 0, stream>>>(seq_lens, batch, sq, max_pages, pairs_per_group,
                                      static_cast<uint8_t*>(ws), L);
  return cudaGetLastError();
}

}  // namespace mla
