// Parameters and host launchers of the MLA decode kernels.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "common.cuh"

namespace mla {

struct DecodeParams {
  const __nv_bfloat16* q_abs;    // [B, Sq, 128, 512]
  const __nv_bfloat16* q_rope;   // [B, Sq, 128, 64]
  const uint8_t* kv_quant;       // FP8 cache [P, 64, 594] or FP4 cache [P, 64, 324] (modes 1, 2, 4)
  const uint8_t* kv_bf16;        // bf16 cache [P, 64, 576] (read by address in the sparse mode)
  const int32_t* block_table;    // [B, max_pages]
  int batch, sq, num_pages, max_pages;
  int pairs_per_group;           // CTA pairs that serve one query index (the planner's partition)
  float scale_log2;              // softmax scale * log2(e)
  int fp8_fallback;              // FP8/FP4 exact pass: run only if the f16 pass flagged its inputs
  const int32_t* sp_slots;       // sparse decode: compacted slot lists [rows, topk] (workspace)
  int topk;
  __nv_bfloat16* out;            // [B, Sq, 128, 512]
  float* lse;                    // [B, Sq, 128]
  uint8_t* ws;
  WsLayout L;
};

// out / lse: the rows with no token are written here (out = 0, lse = -inf).
cudaError_t launch_plan(const int32_t* seq_lens, int batch, int sq, int max_pages, int pairs_per_group,
                        void* ws, const WsLayout& L, __nv_bfloat16* out, float* lse, cudaStream_t stream);
// Sparse decode: compact each query row's listed slots into the workspace.
cudaError_t launch_sparse_prep(const int32_t* token_slots, int rows, int topk, int num_slots, void* ws,
                               const WsLayout& L, cudaStream_t stream);
// TMA descriptors of the bf16 cache (4-D: 64 columns, 8 rows, 9 chunks, row
// groups).  The score SM loads chunks 0..4 (k) and 5..8 (kb) of a half page,
// or of a whole page when a tile's two adjacent slots are the two halves of
// one page (k8, kb8); the value SM loads the eight latent chunks of a half
// page (v).
struct CacheMaps {
  CUtensorMap k, k8, kb, kb8, v;
};

// pdl: launch as a programmatic dependent of the planner (the kernel waits on
// griddepcontrol before reading the plan)
cudaError_t launch_decode_bf16(const CacheMaps& maps, const DecodeParams& p, int n_pairs, bool pdl,
                               cudaStream_t stream);
cudaError_t launch_decode_fp8(const DecodeParams& p, int n_pairs, bool pdl, cudaStream_t stream);
cudaError_t launch_decode_fp4(const DecodeParams& p, int n_pairs, bool pdl, cudaStream_t stream);
cudaError_t launch_decode_fp8_v41(const DecodeParams& p, int n_pairs, bool pdl, cudaStream_t stream);
cudaError_t launch_decode_fp4_v41(const DecodeParams& p, int n_pairs, bool pdl, cudaStream_t stream);
// Sparse decode over the bf16 cache (p.kv_bf16, p.sp_slots; rows planned
// with one query each).
cudaError_t launch_decode_sparse(const DecodeParams& p, int n_pairs, bool pdl, cudaStream_t stream);
int decode_max_pairs();
// W^UV up-projection of latent outputs (see wuv.cu).
cudaError_t launch_wuv(PFN_cuTensorMapEncodeTiled_v12000 encode, const void* o, const void* w, int rows, void* out,
                       void* hdr, cudaStream_t stream);
cudaError_t launch_combine_plan(const void* ws, const WsLayout& Lw, int batch, int sq, __nv_bfloat16* out, float* lse,
                                bool pdl, cudaStream_t stream);
cudaError_t launch_combine_indptr(const float* part_out, const float* part_lse, const int32_t* indptr, int rows,
                                  __nv_bfloat16* out, float* lse, cudaStream_t stream);

}  // namespace mla
