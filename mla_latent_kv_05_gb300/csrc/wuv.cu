// Up-projection of the latent attention output through W^UV.
//
// What it computes ("DeepSeek R1 Architecture & Deployment Guide", section
// 1.1, matrix absorption): the value up-projection W_h^UV (d_v x 512 per
// head) is folded out of the attention, which therefore returns the latent
// output o_h (512 values per head); the head's output in the value space is
//     v_h = W_h^UV o_h                                  (d_v = 128 values).
// For a batch of R query rows this is one GEMM per head:
//     V_h[R x d_v] = O_h[R x 512] . (W_h^UV)^T,
// a batched GEMM with M = R rows, N = d_v, K = 512.
//
// One CTA per (head, 128 query rows): tcgen05.mma kind::f16, M = 128,
// N = 128, K = 512 as 32 K-steps, both operands K-major in shared memory,
// staged by TMA in K-blocks of 64 (16 KiB of O and 16 KiB of W per block,
// 128B swizzle) through a four-block ring; the fp32 accumulator (128 TMEM
// columns) is converted to bf16 by four warps (thread = query row).  Rows
// past R are read as zeros (out-of-range TMA box) and not written.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace mla {

namespace {

constexpr int kDv = 128;                 // value head dimension (W^UV rows per head)
constexpr int kKBlock = 64;              // K values per staged block (128 B rows)
constexpr int kStages = 4;
constexpr uint32_t kBlockBytes = 128u * kKBlock * 2;     // 16 KiB: 128 rows x 128 B
constexpr uint32_t kStageBytes = 2 * kBlockBytes;        // O block + W block
constexpr uint32_t kOffBar = kStages * kStageBytes;      // 128 KiB
constexpr uint32_t kSmem = kOffBar + 256;
constexpr uint32_t kIdesc = ptx::idesc_bf16(128, kDv, 0, 0);

__global__ void __launch_bounds__(128, 1) wuv_kernel(const __grid_constant__ CUtensorMap tmap_o,
                                                     const __grid_constant__ CUtensorMap tmap_w, int rows,
                                                     __nv_bfloat16* __restrict__ out, PlanHeader* hdr) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = ptx::smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x, row0 = blockIdx.y * 128;
  auto FULL = [&](int s) { return sbase + kOffBar + 8u * s; };
  auto EMPTY = [&](int s) { return sbase + kOffBar + 8u * (kStages + s); };
  const uint32_t DONE = sbase + kOffBar + 8u * (2 * kStages);
  const uint32_t tmem_slot = sbase + kOffBar + 8u * (2 * kStages + 1);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) { ptx::mbar_init(FULL(s), 1); ptx::mbar_init(EMPTY(s), 1); }
    ptx::mbar_init(DONE, 1);
    ptx::fence_barrier_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(tmem_slot, kDv);
    ptx::tmem_relinquish();
  }
  if (threadIdx.x == 32) { ptx::prefetch_tmap(&tmap_o); ptx::prefetch_tmap(&tmap_w); }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffBar + 8u * (2 * kStages + 1));
  const bool aligned = (sbase & 1023u) == 0;
  if (threadIdx.x == 0 && !aligned) set_status(&hdr->status, MLA_ERR_UNSUPPORTED);
  constexpr int kBlocks = kDc / kKBlock;   // 8
  bool ok = aligned;

  if (ok && warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol = ptx::policy_evict_first();
      for (int kb = 0; kb < kBlocks && ok; ++kb) {
        const int s = kb % kStages;
        const uint32_t ph = (kb / kStages) & 1u;
        if (!wait_bounded<false>(EMPTY(s), ph ^ 1u, hdr)) { ok = false; break; }
        ptx::mbar_arrive_expect_tx(FULL(s), kStageBytes);
        const uint32_t st = sbase + static_cast<uint32_t>(s) * kStageBytes;
        ptx::tma_load_3d(st, &tmap_o, FULL(s), kb * kKBlock, h, row0, pol);              // O_h rows
        ptx::tma_load_3d(st + kBlockBytes, &tmap_w, FULL(s), kb * kKBlock, 0, h, pol);   // W_h rows
      }
    }
  } else if (ok && warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    for (int kb = 0; kb < kBlocks && ok; ++kb) {
      const int s = kb % kStages;
      const uint32_t ph = (kb / kStages) & 1u;
      if (!wait_warp<false>(FULL(s), ph, hdr)) { ok = false; break; }
      ptx::tc_fence_after();
      if (lane == 0) {
        const uint32_t st = sbase + static_cast<uint32_t>(s) * kStageBytes;
        const uint64_t da = ptx::sdesc_sw128(st, 16, 1024);
        const uint64_t db = ptx::sdesc_sw128(st + kBlockBytes, 16, 1024);
#pragma unroll
        for (int k = 0; k < kKBlock / 16; ++k)
          ptx::mma_ss(tmem, da + static_cast<uint64_t>((k * 32) >> 4), db + static_cast<uint64_t>((k * 32) >> 4),
                      kIdesc, (kb > 0 || k > 0) ? 1u : 0u);
        ptx::mma_commit(EMPTY(s));
        if (kb == kBlocks - 1) ptx::mma_commit(DONE);
      }
      __syncwarp();
    }
  }
  __syncwarp();

  // ------------------------------------------------------------ epilogue (all four warps)
  ok = __syncthreads_and(ok ? 1 : 0) != 0;
  if (ok && wait_warp<false>(DONE, 0, hdr)) {
    ptx::tc_fence_after();
    const int r = row0 + warp * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
#pragma unroll 1
    for (int c = 0; c < kDv / 32; ++c) {
      uint32_t v[32];
      ptx::tmem_ld32(tmem + lane_base + 32u * c, v);
      ptx::tmem_wait_ld();
      if (r < rows) {
        uint32_t o[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          __nv_bfloat162 b = __floats2bfloat162_rn(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
          o[e] = *reinterpret_cast<uint32_t*>(&b);
        }
        __nv_bfloat16* dst = out + (static_cast<size_t>(r) * kHeads + h) * kDv + 32 * c;
        ptx::st_global_v8(dst, o);
        ptx::st_global_v8(dst + 16, o + 8);
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kDv);
  }
}

}  // namespace

// o: [rows, 128, 512] bf16 (the decode's latent output); w: [128, 128, 512]
// bf16 (W^UV per head, rows = value dims); out: [rows, 128, 128] bf16.
cudaError_t launch_wuv(PFN_cuTensorMapEncodeTiled_v12000 encode, const void* o, const void* w, int rows,
                       void* out, void* hdr, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  CUtensorMap tm_o, tm_w;
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kDc), static_cast<cuuint64_t>(kHeads), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(kDc) * 2, static_cast<cuuint64_t>(kHeads) * kDc * 2};
    cuuint32_t box[3] = {kKBlock, 1, 128};
    cuuint32_t es[3] = {1, 1, 1};
    if (encode(&tm_o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(o), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kDc), static_cast<cuuint64_t>(kDv), static_cast<cuuint64_t>(kHeads)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(kDc) * 2, static_cast<cuuint64_t>(kDv) * kDc * 2};
    cuuint32_t box[3] = {kKBlock, kDv, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (encode(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(w), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(wuv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  return launch_kernel(wuv_kernel, dim3(kHeads, (rows + 127) / 128), dim3(128), kSmem, stream, tm_o, tm_w, rows,
                       static_cast<__nv_bfloat16*>(out), static_cast<PlanHeader*>(hdr));
}

}  // namespace mla
