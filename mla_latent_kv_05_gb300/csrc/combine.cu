// Split-KV merge of caller-made parts (the public mla_combine_splits; the
// decode calls merge their own splits inside the attention kernel).
// Attention over disjoint token sets combines exactly from each part's
// normalised output and LSE:
//     L = ln sum_s exp(lse_s),   out = sum_s exp(lse_s - L) * out_s.
// One warp per (output row, head), 16 values per lane, fp32 partials in,
// bf16 out.
#include <cuda_bf16.h>

#include "common.cuh"

namespace mla {

namespace {

// Eight consecutive values of a partial row, as fp32: element offset e
// (a multiple of 8), 16-byte loads that bypass L1 (each partial is read once).
__device__ __forceinline__ void load8(const float* src, int e, float* x) {
  const float4 a = __ldcs(reinterpret_cast<const float4*>(src + e));
  const float4 b = __ldcs(reinterpret_cast<const float4*>(src + e + 4));
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// grid (rows, 128 / 8): one warp per (row, head); lane holds values
// [8 lane, 8 lane + 8) and [256 + 8 lane, 256 + 8 lane + 8).  Each lane reads
// one part's lse (parts beyond 32 loop); the weights reach the other lanes by
// shuffles, and the parts' values are loaded four parts at a time so their
// loads overlap.  Row r merges parts [indptr[r], indptr[r+1]).
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ part_out,
                                                      const float* __restrict__ part_lse,
                                                      const int32_t* __restrict__ indptr,
                                                      __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
  const int row = blockIdx.x;
  const int start = indptr[row];
  const int count = indptr[row + 1] - start;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * 8 + warp;
  float L = -INFINITY;
  for (int s = lane; s < count; s += 32) L = fmaxf(L, part_lse[static_cast<size_t>(start + s) * kHeads + h]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L = fmaxf(L, __shfl_xor_sync(0xffffffffu, L, o));
  float acc[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) acc[e] = 0.f;
  float sum = 0.f;
  if (L != -INFINITY) {
    for (int s0 = 0; s0 < count; s0 += 32) {
      // this lane's part weight for parts s0 .. s0 + 31
      const int sl = s0 + lane;
      const float v = sl < count ? part_lse[static_cast<size_t>(start + sl) * kHeads + h] : -INFINITY;
      const float wl = v == -INFINITY ? 0.f : __expf(v - L);
      const int n = min(32, count - s0);
      for (int j0 = 0; j0 < n; j0 += 4) {
        float x[4][16], wgt[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          wgt[u] = __shfl_sync(0xffffffffu, wl, (j0 + u) & 31);
          if (j0 + u < n) {
            const float* src = part_out + (static_cast<size_t>(start + s0 + j0 + u) * kHeads + h) * kDc;
            load8(src, 8 * lane, x[u]);
            load8(src, 256 + 8 * lane, x[u] + 8);
          } else {
            wgt[u] = 0.f;
#pragma unroll
            for (int e = 0; e < 16; ++e) x[u][e] = 0.f;
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          sum += wgt[u];
#pragma unroll
          for (int e = 0; e < 16; ++e) acc[e] += wgt[u] * x[u][e];
        }
      }
    }
  }
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  __nv_bfloat16* dst = out + (static_cast<size_t>(row) * kHeads + h) * kDc;
  uint32_t o[8];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      __nv_bfloat162 b = __floats2bfloat162_rn(acc[8 * half + 2 * q] * inv, acc[8 * half + 2 * q + 1] * inv);
      o[q] = *reinterpret_cast<uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(dst + 256 * half + 8 * lane) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (lane == 0) lse[static_cast<size_t>(row) * kHeads + h] = sum > 0.f ? L + logf(sum) : -INFINITY;
}

}  // namespace

// Public merge: parts of row r are [indptr[r], indptr[r+1]).
cudaError_t launch_combine_indptr(const float* part_out, const float* part_lse, const int32_t* indptr, int rows,
                                  __nv_bfloat16* out, float* lse, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  return launch_kernel(combine_kernel, dim3(rows, kHeads / 8), dim3(256), 0, stream, part_out, part_lse, indptr, out,
                       lse);
}

}  // namespace mla
