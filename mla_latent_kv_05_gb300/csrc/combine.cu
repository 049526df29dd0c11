// Split-KV merge.  Attention over disjoint token sets combines exactly from
// each part's normalised output and LSE:
//     L = ln sum_s exp(lse_s),   out = sum_s exp(lse_s - L) * out_s.
// Two kernels: the decode calls' merge of their own split rows (bf16
// partials, from the plan), and the public mla_combine_splits (fp32
// partials, caller's indptr).  One warp per (output row, head), bf16 out.
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

// The decode's split rows, launched as a programmatic dependent of the
// attention kernel (its partials are read only after that grid completed):
// grid (B*Sq, 128/8), one warp per (row, head), lane = 16 latent columns
// (one 32-byte sector).  Row k = b*Sq + i merges its bf16 partials at slots
// [i*spq + slot_base[b], + n_parts[b]) when the planner split it
// (n_parts[b] > 1); other rows were written by the attention kernel (one
// part) or the planner (no token).  Four parts' loads are in flight at a
// time; the parts are summed in slot order.
__global__ void __launch_bounds__(256) combine_plan_kernel(const uint8_t* __restrict__ ws, WsLayout Lw, int sq,
                                                           __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
  // The plan (part counts and slot bases) was written by the planner, which
  // completed before the attention kernel let this grid launch, so it is read
  // before the wait; the partials and their lse only after it.
  const int k = blockIdx.x;
  const int b = k / sq, i = k - b * sq;
  const int parts = __ldcg(reinterpret_cast<const int*>(ws + Lw.n_parts) + b);
  const int base = __ldcg(reinterpret_cast<const int*>(ws + Lw.slot_base) + b);
  const int spq = __ldcg(&reinterpret_cast<const PlanHeader*>(ws)->slots_per_query);
  ptx::grid_dep_wait();
  // the next call's planner may begin launching (it waits for this grid
  // before it reads or writes anything)
  ptx::grid_dep_launch();
  if (parts <= 1) return;
  const int start = i * spq + base;
  const float* part_lse = reinterpret_cast<const float*>(ws + Lw.part_lse);
  const __nv_bfloat16* part_out = reinterpret_cast<const __nv_bfloat16*>(ws + Lw.part_out);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * 8 + warp;
  float acc[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) acc[e] = 0.f;
  float sum = 0.f, L = -INFINITY;
  // Parts in groups of 32 (one lse per lane); within a group the partial
  // rows are read four at a time, and the first four are requested together
  // with the group's lse values.  Each group's weights are taken against the
  // running maximum, and earlier groups are rescaled when it grows.
  for (int s0 = 0; s0 < parts; s0 += 32) {
    const int n = min(32, parts - s0);
    const int sl = s0 + lane;
    const float v = sl < parts ? __ldcg(part_lse + static_cast<size_t>(start + sl) * kHeads + h) : -INFINITY;
    uint32_t x[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (u < n) ptx::ld_global_cg_v8(part_out + (static_cast<size_t>(start + s0 + u) * kHeads + h) * kDc + 16 * lane, x[u]);
    float gm = v;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, o));
    const float Ln = fmaxf(L, gm);
    if (Ln != -INFINITY && L != Ln && L != -INFINITY) {
      const float r = __expf(L - Ln);
      sum *= r;
#pragma unroll
      for (int e = 0; e < 16; ++e) acc[e] *= r;
    }
    L = Ln;
    const float wl = (v == -INFINITY || L == -INFINITY) ? 0.f : __expf(v - L);
    for (int j0 = 0; j0 < n; j0 += 4) {
      if (j0 > 0) {
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (j0 + u < n)
            ptx::ld_global_cg_v8(part_out + (static_cast<size_t>(start + s0 + j0 + u) * kHeads + h) * kDc + 16 * lane, x[u]);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float wg = __shfl_sync(0xffffffffu, wl, (j0 + u) & 31);
        if (j0 + u < n) {
          sum += wg;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x[u][e]));
            acc[2 * e] = fmaf(wg, f.x, acc[2 * e]);
            acc[2 * e + 1] = fmaf(wg, f.y, acc[2 * e + 1]);
          }
        }
      }
    }
  }
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  uint32_t o[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    __nv_bfloat162 bb = __floats2bfloat162_rn(acc[2 * e] * inv, acc[2 * e + 1] * inv);
    o[e] = *reinterpret_cast<uint32_t*>(&bb);
  }
  ptx::st_global_v8(out + (static_cast<size_t>(k) * kHeads + h) * kDc + 16 * lane, o);
  if (lane == 0) lse[static_cast<size_t>(k) * kHeads + h] = sum > 0.f ? L + logf(sum) : -INFINITY;
}

}  // namespace

cudaError_t launch_combine_plan(const void* ws, const WsLayout& Lw, int batch, int sq, __nv_bfloat16* out, float* lse,
                                bool pdl, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(batch * sq, kHeads / 8, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_plan_kernel, static_cast<const uint8_t*>(ws), Lw, sq, out, lse);
}

// Public merge: parts of row r are [indptr[r], indptr[r+1]).
cudaError_t launch_combine_indptr(const float* part_out, const float* part_lse, const int32_t* indptr, int rows,
                                  __nv_bfloat16* out, float* lse, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  return launch_kernel(combine_kernel, dim3(rows, kHeads / 8), dim3(256), 0, stream, part_out, part_lse, indptr, out,
                       lse);
}

}  // namespace mla
