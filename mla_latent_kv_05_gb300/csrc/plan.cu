// Split-KV planner: turns seq_lens (on the device, no host sync) into an even
// partition of KV tiles over the persistent CTA pairs, the partial-output
// slots of rows that end up split, and the list of rows the merge kernel
// writes.  One CTA of 1024 threads.
//
// Partition: every batch row b has n_b = ceil(seq_len_b / 64) tiles (one tile
// = one page).  The rows' tiles are laid end to end (prefix sums tile_start)
// and cut into pieces of `chunk` = ceil(total / pairs_per_group) tiles; pair
// p of a query group takes tiles [p*chunk, (p+1)*chunk).  Each query index
// i < Sq has its own group of pairs with the identical partition, so the
// groups read the same pages at about the same time and share them in L2.
// A row covered by one pair is written straight to `out`; a row covered by
// k > 1 pairs gets k partial slots (per query index) and a merge entry.
#include "common.cuh"

namespace mla {

namespace {

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
  if (tid == 0) {
    tile_start[batch] = total;
    s_chunk = total > 0 ? (total + pairs_per_group - 1) / pairs_per_group : 1;
  }
  __syncthreads();
  const int chunk = s_chunk;

  // pass 2: pairs covering each row; slots for rows that are split
  local = 0;
  int local_comb = 0;
  for (int b = lo; b < hi; ++b) {
    const int n = (lens[b] + kPage - 1) / kPage;
    int parts = 0, fp = 0;
    if (n > 0) {
      fp = tile_start[b] / chunk;
      parts = (tile_start[b] + n - 1) / chunk - fp + 1;
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
    if (n > 0) parts = (tile_start[b] + n - 1) / chunk - first_pair[b] + 1;
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
  }
}

}  // namespace

cudaError_t launch_plan(const int32_t* seq_lens, int batch, int sq, int max_pages, int pairs_per_group,
                        void* ws, const WsLayout& L, cudaStream_t stream) {
  plan_kernel<<<1, 1024, 0, stream>>>(seq_lens, batch, sq, max_pages, pairs_per_group,
                                      static_cast<uint8_t*>(ws), L);
  return cudaGetLastError();
}

}  // namespace mla
