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

__device__ __forceinline__ void load4(const float* src, int i, float* x) {
  const float4 v = __ldcs(reinterpret_cast<const float4*>(src) + i);
  x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* src, int i, float* x) {
  const uint2 v = __ldcs(reinterpret_cast<const uint2*>(src) + i);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
  x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
}

// grid (rows, 128 / 8): one warp per (row, head); lane holds values
// 4(32q + lane) .. +3 for q = 0..3.
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
  // each lane reads one part's lse (parts beyond 32 loop), then a warp max / sum
  float L = -INFINITY;
  for (int s = lane; s < count; s += 32) L = fmaxf(L, part_lse[static_cast<size_t>(start + s) * kHeads + h]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L = fmaxf(L, __shfl_xor_sync(0xffffffffu, L, o));
  float acc[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) acc[e] = 0.f;
  float sum = 0.f;
  if (L != -INFINITY) {
    for (int s = 0; s < count; ++s) {
      const float v = part_lse[static_cast<size_t>(start + s) * kHeads + h];
      const float wgt = v == -INFINITY ? 0.f : __expf(v - L);
      sum += wgt;
      const TP* src = part_out + (static_cast<size_t>(start + s) * kHeads + h) * kDc;
      float x[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) load4(src, q * 32 + lane, x + 4 * q);
#pragma unroll
      for (int e = 0; e < 16; ++e) acc[e] += wgt * x[e];
    }
  }
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  __nv_bfloat16* dst = out + (static_cast<size_t>(row) * kHeads + h) * kDc;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    __nv_bfloat162 a = __floats2bfloat162_rn(acc[4 * q] * inv, acc[4 * q + 1] * inv);
    __nv_bfloat162 b = __floats2bfloat162_rn(acc[4 * q + 2] * inv, acc[4 * q + 3] * inv);
    uint2 v;
    v.x = *reinterpret_cast<uint32_t*>(&a);
    v.y = *reinterpret_cast<uint32_t*>(&b);
    reinterpret_cast<uint2*>(dst)[q * 32 + lane] = v;
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
