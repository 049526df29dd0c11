// Split-KV merge.  Attention over disjoint token sets combines exactly from
// each part's normalised output and LSE:
//     L = ln sum_s exp(lse_s),   out = sum_s exp(lse_s - L) * out_s.
// One warp per (output row, head), 16 values per lane, bf16 out.  The
// decode plan's partials are bf16 (each part already normalised, so its
// rounding adds at most 2^-9 relative to the merge); the public entry point
// merges fp32 partials.
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
__device__ __forceinline__ void load8(const __nv_bfloat16* src, int e, float* x) {
  const uint4 v = __ldcs(reinterpret_cast<const uint4*>(src + e));
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
    x[2 * k] = f.x;
    x[2 * k + 1] = f.y;
  }
}

// grid (rows, 128 / 8): one warp per (row, head); lane holds values
// [8 lane, 8 lane + 8) and [256 + 8 lane, 256 + 8 lane + 8).  Each lane reads
// one part's lse (parts beyond 32 loop); the weights reach the other lanes by
// shuffles, and the parts' values are loaded four parts at a time so their
// loads overlap.
template <typename TP>
__global__ void __launch_bounds__(256) combine_kernel(const TP* __restrict__ part_out,
                                                      const float* __restrict__ part_lse,
                                                      const int32_t* __restrict__ row_start,
                                                      const int32_t* __restrict__ row_count,
                                                      const int32_t* __restrict__ row_index,
                                                      const int32_t* __restrict__ n_rows_dev, int n_rows,
                                                      __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
  // launched as a programmatic dependent of the attention kernel: its
  // partials are read only after that grid has completed
  ptx::grid_dep_wait();
  const int k = blockIdx.x;
  const int rows = n_rows_dev ? *n_rows_dev : n_rows;
  if (k >= rows) return;
  const int start = row_start[k];
  const int count = row_count ? row_count[k] : row_start[k + 1] - start;   // null: row_start is an indptr
  const int row = row_index ? row_index[k] : k;
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
            const TP* src = part_out + (static_cast<size_t>(start + s0 + j0 + u) * kHeads + h) * kDc;
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

// Merge of the decode plan's split rows (row list and count on the device).
cudaError_t launch_combine_plan(const void* ws, const WsLayout& Lw, int max_rows, __nv_bfloat16* out, float* lse,
                                bool pdl, cudaStream_t stream) {
  const uint8_t* w = static_cast<const uint8_t*>(ws);
  if (max_rows <= 0) return cudaSuccess;
  // programmatic dependent launch: the kernel's launch overlaps the tail of
  // the attention kernel; griddepcontrol.wait orders its reads after it
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(max_rows, kHeads / 8, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel<__nv_bfloat16>, reinterpret_cast<const __nv_bfloat16*>(w + Lw.part_out),
                            reinterpret_cast<const float*>(w + Lw.part_lse),
                            reinterpret_cast<const int32_t*>(w + Lw.comb_start),
                            reinterpret_cast<const int32_t*>(w + Lw.comb_count),
                            reinterpret_cast<const int32_t*>(w + Lw.comb_row),
                            reinterpret_cast<const int32_t*>(w + offsetof(PlanHeader, n_comb)), 0, out, lse);
}

// Public merge: parts of row r are [indptr[r], indptr[r+1]).
cudaError_t launch_combine_indptr(const float* part_out, const float* part_lse, const int32_t* indptr, int rows,
                                  __nv_bfloat16* out, float* lse, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  combine_kernel<float><<<dim3(rows, kHeads / 8), 256, 0, stream>>>(part_out, part_lse, indptr, nullptr, nullptr, nullptr,
                                                                    rows, out, lse);
  return cudaGetLastError();
}

}  // namespace mla
