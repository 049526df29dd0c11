// C ABI of the MLA decode library: argument validation, workspace sizing,
// tensor-map creation and the launch sequence (planner -> paired decode
// kernel -> split merge), all on the caller's stream.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "decode.cuh"

namespace {

using namespace mla;

thread_local cudaEvent_t g_prof_before = nullptr, g_prof_after = nullptr;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// The bf16 cache viewed as a 4-D tensor: (64 columns, 8 rows, 9 column
// chunks, num_pages*8 row groups) with strides 1152 B (row), 128 B (chunk)
// and 9216 B (row group).  A box of 64 x 8 x `chunks` x 4 is one half page
// (32 tokens), written to shared memory as 8-row x 128-byte swizzle atoms in
// (row group, chunk, row) order, so consecutive half-page slots form one
// K-major operand with a constant row-group stride.
// `groups` row groups per box: 4 for a half page, 8 for a whole page.
int make_cache_tmap(CUtensorMap* m, const void* cache, int num_pages, unsigned chunks, unsigned groups = 4) {
  auto fn = encode_fn();
  if (!fn) return MLA_ERR_CUDA;
  cuuint64_t dims[4] = {64, 8, static_cast<cuuint64_t>(kRow / 64), static_cast<cuuint64_t>(num_pages) * (kPage / 8)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(kRow) * 2, 128, static_cast<cuuint64_t>(kRow) * 2 * 8};
  cuuint32_t box[4] = {64, 8, chunks, groups};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(cache), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_CUDA;
}

int validate_common(const void* q_absorbed, const void* q_rope, const void* kv_cache, const int32_t* block_table,
                    const int32_t* seq_lens, int batch, int sq, int num_heads, int num_pages, int page_size,
                    int max_pages, float scale, const void* out, const float* lse, const void* workspace) {
  if (!q_absorbed || !q_rope || !kv_cache || !block_table || !seq_lens || !out || !lse || !workspace)
    return MLA_ERR_INVALID_ARG;
  if (batch < 0 || sq <= 0 || num_pages <= 0 || max_pages <= 0 || !std::isfinite(scale) || !(scale > 0.f))
    return MLA_ERR_INVALID_ARG;
  if (num_heads != kHeads || page_size != kPage || sq > kMaxSq) return MLA_ERR_UNSUPPORTED;
  if (static_cast<long long>(batch) * sq > kMaxRows) return MLA_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_pages) * kPage >= INT_MAX / 2 ||
      static_cast<long long>(max_pages) * kPage >= INT_MAX / 2)
    return MLA_ERR_UNSUPPORTED;
  if (!aligned(q_absorbed, 16) || !aligned(q_rope, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) ||
      !aligned(lse, 4) || !aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(workspace, 256))
    return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}

enum class CacheKind { kBf16, kFp8, kFp4, kFp8V41, kFp4V41 };

// CTA pairs a query index gets: all resident pairs, but no more than one per
// kPagesPerPair pages the call can hold (batch * max_pages, known on the host
// without reading seq_lens).  A small decode then runs on a few pairs, and a
// row of a few pages is not split (no partial write, nothing to merge).  The
// workspace stays sized for all resident pairs.
constexpr long long kPagesPerPair = 8;
int pairs_for(int max_pairs, long long page_bound) {
  const long long want = (page_bound + kPagesPerPair - 1) / kPagesPerPair;
  return static_cast<int>(want < 1 ? 1 : (want < max_pairs ? want : max_pairs));
}

int run_decode(CacheKind kind, const uint16_t* q_absorbed, const uint16_t* q_rope, const void* kv_cache,
               const int32_t* block_table, const int32_t* seq_lens, int batch, int sq, int num_heads, int num_pages,
               int page_size, int max_pages, float softmax_scale, uint16_t* out, float* lse, void* workspace,
               size_t workspace_bytes, void* stream_ptr) {
  int st = validate_common(q_absorbed, q_rope, kv_cache, block_table, seq_lens, batch, sq, num_heads, num_pages,
                           page_size, max_pages, softmax_scale, out, lse, workspace);
  if (st != MLA_OK) return st;
  if (batch == 0) return MLA_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const int pairs = decode_max_pairs();
  if (pairs <= 0) return MLA_ERR_CUDA;
  const int ppg = pairs_for(pairs / sq > 0 ? pairs / sq : 1, static_cast<long long>(batch) * max_pages);
  const WsLayout L = ws_layout(batch, sq, pairs);
  if (workspace_bytes < L.total) return MLA_ERR_WORKSPACE;

  // half and whole pages of chunks 0..4 and 5..8 (score SM), half pages of
  // the 8 latent chunks (value SM)
  CacheMaps maps;
  const bool quant = kind != CacheKind::kBf16;
  if (!quant) {
    st = make_cache_tmap(&maps.k, kv_cache, num_pages, 5);
    if (st == MLA_OK) st = make_cache_tmap(&maps.k8, kv_cache, num_pages, 5, 8);
    if (st == MLA_OK) st = make_cache_tmap(&maps.kb, kv_cache, num_pages, 4);
    if (st == MLA_OK) st = make_cache_tmap(&maps.kb8, kv_cache, num_pages, 4, 8);
    if (st == MLA_OK) st = make_cache_tmap(&maps.v, kv_cache, num_pages, 8);
    if (st != MLA_OK) return st;
  }

  if (launch_plan(seq_lens, batch, sq, max_pages, ppg, workspace, L, reinterpret_cast<__nv_bfloat16*>(out), lse,
                  stream) != cudaSuccess)
    return MLA_ERR_CUDA;
  DecodeParams p;
  p.q_abs = reinterpret_cast<const __nv_bfloat16*>(q_absorbed);
  p.q_rope = reinterpret_cast<const __nv_bfloat16*>(q_rope);
  p.kv_quant = quant ? static_cast<const uint8_t*>(kv_cache) : nullptr;
  p.kv_bf16 = quant ? nullptr : static_cast<const uint8_t*>(kv_cache);
  p.sp_slots = nullptr;
  p.topk = 0;
  p.block_table = block_table;
  p.batch = batch;
  p.sq = sq;
  p.pairs_per_group = ppg;
  p.num_pages = num_pages;
  p.max_pages = max_pages;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.fp8_fallback = 0;
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.ws = static_cast<uint8_t*>(workspace);
  p.L = L;
  // The three kernels are chained with programmatic dependent launch, so the
  // attention kernel's prologue overlaps the planner and the merge kernel's
  // launch overlaps the attention kernel's tail.  A call with the profiling
  // hook set records its events around the attention kernel and launches the
  // kernels without that overlap, so that the events bracket it alone.
  cudaEvent_t ev0 = g_prof_before, ev1 = g_prof_after;
  g_prof_before = g_prof_after = nullptr;
  const bool pdl = ev0 == nullptr;
  if (ev0 && cudaEventRecord(ev0, stream) != cudaSuccess) return MLA_ERR_CUDA;
  cudaError_t le;
  if (kind == CacheKind::kFp8) le = launch_decode_fp8(p, ppg * sq, pdl, stream);
  else if (kind == CacheKind::kFp4) le = launch_decode_fp4(p, ppg * sq, pdl, stream);
  else if (kind == CacheKind::kFp8V41) le = launch_decode_fp8_v41(p, ppg * sq, pdl, stream);
  else if (kind == CacheKind::kFp4V41) le = launch_decode_fp4_v41(p, ppg * sq, pdl, stream);
  else le = launch_decode_bf16(maps, p, ppg * sq, pdl, stream);
  if (le != cudaSuccess) return MLA_ERR_CUDA;
  if (ev1 && cudaEventRecord(ev1, stream) != cudaSuccess) return MLA_ERR_CUDA;
  if (launch_combine_plan(workspace, L, batch, sq, p.out, lse, pdl, stream) != cudaSuccess) return MLA_ERR_CUDA;
  return MLA_OK;
}

// Library-owned scratch of mla_decode_bf16_noalloc: the plan header, the
// split-KV plan and the fp32 partial outputs, for callers that cannot hand
// the library device memory.  40 MiB holds the partials of 76 CTA pairs (the
// 152 SMs of a GB300: 152 slots x 128 heads x 512 bf16 = 19 MiB) plus the
// plan of up to kStaticMaxRows query rows, with room to spare.  One copy per
// device, shared by every call on that device.
constexpr size_t kStaticScratchBytes = size_t{40} << 20;
constexpr int kStaticMaxRows = 8192;
constexpr int kStaticMaxDevices = 64;
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

std::mutex g_static_mu;
void* g_static_ptr[kStaticMaxDevices] = {};

// Device address of this device's copy of the scratch, looked up once per
// device (with that device current) and cached.
int static_scratch(void** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  if (dev < 0 || dev >= kStaticMaxDevices) return MLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
    g_static_ptr[dev] = p;
  }
  *ptr = g_static_ptr[dev];
  return MLA_OK;
}

constexpr int kMaxTopk = 16384;

// Sparse top-k decode: compact the slot lists, plan the B*Sq query rows as a
// batch of rows with one query each, gather-attend, merge.
int run_sparse(const uint16_t* q_absorbed, const uint16_t* q_rope, const void* kv_cache, const int32_t* token_slots,
               int batch, int sq, int topk, int num_heads, int num_pages, int page_size, float softmax_scale,
               uint16_t* out, float* lse, void* workspace, size_t workspace_bytes, void* stream_ptr) {
  if (!q_absorbed || !q_rope || !kv_cache || !token_slots || !out || !lse || !workspace) return MLA_ERR_INVALID_ARG;
  if (batch < 0 || sq <= 0 || topk <= 0 || num_pages <= 0 || !std::isfinite(softmax_scale) || !(softmax_scale > 0.f))
    return MLA_ERR_INVALID_ARG;
  if (num_heads != kHeads || page_size != kPage || topk > kMaxTopk) return MLA_ERR_UNSUPPORTED;
  if (static_cast<long long>(batch) * sq > kMaxRows) return MLA_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_pages) * kPage >= INT_MAX / 2) return MLA_ERR_UNSUPPORTED;
  if (!aligned(q_absorbed, 16) || !aligned(q_rope, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) ||
      !aligned(lse, 4) || !aligned(token_slots, 4) || !aligned(workspace, 256))
    return MLA_ERR_INVALID_ARG;
  if (batch == 0) return MLA_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const int pairs = decode_max_pairs();
  if (pairs <= 0) return MLA_ERR_CUDA;
  const int rows = batch * sq;
  const WsLayout L = ws_layout(rows, 1, pairs, topk);
  if (workspace_bytes < L.total) return MLA_ERR_WORKSPACE;
  const int max_pages = (topk + kPage - 1) / kPage;
  const int ppg = pairs_for(pairs, static_cast<long long>(rows) * max_pages);
  if (launch_sparse_prep(token_slots, rows, topk, num_pages * kPage, workspace, L, stream) != cudaSuccess)
    return MLA_ERR_CUDA;
  const int32_t* counts = reinterpret_cast<const int32_t*>(static_cast<const uint8_t*>(workspace) + L.sp_lens);
  if (launch_plan(counts, rows, 1, max_pages, ppg, workspace, L, reinterpret_cast<__nv_bfloat16*>(out), lse,
                  stream) != cudaSuccess)
    return MLA_ERR_CUDA;
  DecodeParams p;
  memset(&p, 0, sizeof(p));
  p.q_abs = reinterpret_cast<const __nv_bfloat16*>(q_absorbed);
  p.q_rope = reinterpret_cast<const __nv_bfloat16*>(q_rope);
  p.kv_bf16 = static_cast<const uint8_t*>(kv_cache);
  p.block_table = nullptr;
  p.batch = rows;
  p.sq = 1;
  p.pairs_per_group = ppg;
  p.num_pages = num_pages;
  p.max_pages = max_pages;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.sp_slots = reinterpret_cast<const int32_t*>(static_cast<const uint8_t*>(workspace) + L.sp_slots);
  p.topk = topk;
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.ws = static_cast<uint8_t*>(workspace);
  p.L = L;
  cudaEvent_t ev0 = g_prof_before, ev1 = g_prof_after;
  g_prof_before = g_prof_after = nullptr;
  const bool pdl = ev0 == nullptr;
  if (ev0 && cudaEventRecord(ev0, stream) != cudaSuccess) return MLA_ERR_CUDA;
  if (launch_decode_sparse(p, ppg, pdl, stream) != cudaSuccess) return MLA_ERR_CUDA;
  if (ev1 && cudaEventRecord(ev1, stream) != cudaSuccess) return MLA_ERR_CUDA;
  if (launch_combine_plan(workspace, L, rows, 1, p.out, lse, pdl, stream) != cudaSuccess) return MLA_ERR_CUDA;
  return MLA_OK;
}

}  // namespace

// Only the C ABI below is exported (the library is built with hidden
// visibility), so a process may load several copies without their internals
// binding to each other.
#pragma GCC visibility push(default)
extern "C" {

int mla_up_project_wuv(const uint16_t* latent, const uint16_t* w_uv, int rows, int num_heads, int d_v,
                       uint16_t* out, void* workspace, size_t workspace_bytes, void* stream) {
  if (!latent || !w_uv || !out || !workspace || rows < 0) return MLA_ERR_INVALID_ARG;
  if (num_heads != kHeads || d_v != 128) return MLA_ERR_UNSUPPORTED;
  if (rows > kMaxRows) return MLA_ERR_UNSUPPORTED;
  if (!aligned(latent, 16) || !aligned(w_uv, 16) || !aligned(out, 16) || !aligned(workspace, 256))
    return MLA_ERR_INVALID_ARG;
  if (workspace_bytes < sizeof(PlanHeader)) return MLA_ERR_WORKSPACE;
  if (rows == 0) return MLA_OK;
  auto fn = encode_fn();
  if (!fn) return MLA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(static_cast<uint8_t*>(workspace) + offsetof(PlanHeader, abort_flag), 0, sizeof(int), st) !=
      cudaSuccess)
    return MLA_ERR_CUDA;
  return launch_wuv(fn, latent, w_uv, rows, out, workspace, st) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_workspace_size_sparse(int batch, int sq, int topk, int num_heads, int page_size, size_t* bytes) {
  if (!bytes || batch < 0 || sq <= 0 || topk <= 0) return MLA_ERR_INVALID_ARG;
  if (num_heads != kHeads || page_size != kPage || topk > kMaxTopk) return MLA_ERR_UNSUPPORTED;
  if (static_cast<long long>(batch) * sq > kMaxRows) return MLA_ERR_UNSUPPORTED;
  const int pairs = decode_max_pairs();
  if (pairs <= 0) return MLA_ERR_CUDA;
  *bytes = ws_layout(batch > 0 ? batch * sq : 1, 1, pairs, topk).total;
  return MLA_OK;
}

int mla_decode_sparse_bf16(const uint16_t* q_absorbed, const uint16_t* q_rope, const uint16_t* kv_cache,
                           const int32_t* token_slots, int batch, int sq, int topk, int num_heads, int num_pages,
                           int page_size, float softmax_scale, uint16_t* out, float* lse, void* workspace,
                           size_t workspace_bytes, void* stream) {
  return run_sparse(q_absorbed, q_rope, kv_cache, token_slots, batch, sq, topk, num_heads, num_pages, page_size,
                    softmax_scale, out, lse, workspace, workspace_bytes, stream);
}

int mla_workspace_size(int batch, int sq, int num_heads, int page_size, size_t* bytes) {
  if (!bytes || batch < 0 || sq <= 0) return MLA_ERR_INVALID_ARG;
  if (num_heads != kHeads || page_size != kPage || sq > kMaxSq) return MLA_ERR_UNSUPPORTED;
  if (static_cast<long long>(batch) * sq > kMaxRows) return MLA_ERR_UNSUPPORTED;
  const int pairs = decode_max_pairs();
  if (pairs <= 0) return MLA_ERR_CUDA;
  *bytes = ws_layout(batch > 0 ? batch : 1, sq, pairs).total;
  return MLA_OK;
}

int mla_decode_bf16(const uint16_t* q_absorbed, const uint16_t* q_rope, const uint16_t* kv_cache,
                    const int32_t* block_table, const int32_t* seq_lens, int batch, int sq, int num_heads,
                    int num_pages, int page_size, int max_pages, float softmax_scale, uint16_t* out, float* lse,
                    void* workspace, size_t workspace_bytes, void* stream) {
  return run_decode(CacheKind::kBf16, q_absorbed, q_rope, kv_cache, block_table, seq_lens, batch, sq, num_heads,
                    num_pages, page_size, max_pages, softmax_scale, out, lse, workspace, workspace_bytes, stream);
}

int mla_decode_bf16_noalloc(const uint16_t* q_absorbed, const uint16_t* q_rope, const uint16_t* kv_cache,
                            const int32_t* block_table, const int32_t* seq_lens, int batch, int sq, int num_heads,
                            int num_pages, int page_size, int max_pages, float softmax_scale, uint16_t* out,
                            float* lse, int* device_status, void* stream) {
  void* scratch = nullptr;
  int st = static_scratch(&scratch);
  if (st != MLA_OK) return st;
  st = validate_common(q_absorbed, q_rope, kv_cache, block_table, seq_lens, batch, sq, num_heads, num_pages,
                       page_size, max_pages, softmax_scale, out, lse, scratch);
  if (st != MLA_OK) return st;
  if (device_status && !aligned(device_status, 4)) return MLA_ERR_INVALID_ARG;
  if (static_cast<long long>(batch) * sq > kStaticMaxRows) return MLA_ERR_WORKSPACE;
  const int pairs = decode_max_pairs();
  if (pairs <= 0) return MLA_ERR_CUDA;
  if (ws_layout(batch, sq, pairs).total > kStaticScratchBytes) return MLA_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the status word and the abort flag must start at zero for this call
  if (cudaMemsetAsync(scratch, 0, sizeof(PlanHeader), s) != cudaSuccess) return MLA_ERR_CUDA;
  st = run_decode(CacheKind::kBf16, q_absorbed, q_rope, kv_cache, block_table, seq_lens, batch, sq, num_heads,
                  num_pages, page_size, max_pages, softmax_scale, out, lse, scratch, kStaticScratchBytes, stream);
  if (st != MLA_OK) return st;
  if (device_status &&
      cudaMemcpyAsync(device_status, scratch, sizeof(int), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

int mla_decode_fp8(const uint16_t* q_absorbed, const uint16_t* q_rope, const uint8_t* kv_cache,
                   const int32_t* block_table, const int32_t* seq_lens, int batch, int sq, int num_heads,
                   int num_pages, int page_size, int max_pages, float softmax_scale, uint16_t* out, float* lse,
                   void* workspace, size_t workspace_bytes, void* stream) {
  return run_decode(CacheKind::kFp8, q_absorbed, q_rope, kv_cache, block_table, seq_lens, batch, sq, num_heads,
                    num_pages, page_size, max_pages, softmax_scale, out, lse, workspace, workspace_bytes, stream);
}

int mla_decode_fp4(const uint16_t* q_absorbed, const uint16_t* q_rope, const uint8_t* kv_cache,
                   const int32_t* block_table, const int32_t* seq_lens, int batch, int sq, int num_heads,
                   int num_pages, int page_size, int max_pages, float softmax_scale, uint16_t* out, float* lse,
                   void* workspace, size_t workspace_bytes, void* stream) {
  return run_decode(CacheKind::kFp4, q_absorbed, q_rope, kv_cache, block_table, seq_lens, batch, sq, num_heads,
                    num_pages, page_size, max_pages, softmax_scale, out, lse, workspace, workspace_bytes, stream);
}

int mla_decode_fp8_v41(const uint16_t* q_absorbed, const uint16_t* q_rope, const uint8_t* kv_cache,
                       const int32_t* block_table, const int32_t* seq_lens, int batch, int sq, int num_heads,
                       int num_pages, int page_size, int max_pages, float softmax_scale, uint16_t* out, float* lse,
                       void* workspace, size_t workspace_bytes, void* stream) {
  return run_decode(CacheKind::kFp8V41, q_absorbed, q_rope, kv_cache, block_table, seq_lens, batch, sq, num_heads,
                    num_pages, page_size, max_pages, softmax_scale, out, lse, workspace, workspace_bytes, stream);
}

int mla_decode_fp4_v41(const uint16_t* q_absorbed, const uint16_t* q_rope, const uint8_t* kv_cache,
                       const int32_t* block_table, const int32_t* seq_lens, int batch, int sq, int num_heads,
                       int num_pages, int page_size, int max_pages, float softmax_scale, uint16_t* out, float* lse,
                       void* workspace, size_t workspace_bytes, void* stream) {
  return run_decode(CacheKind::kFp4V41, q_absorbed, q_rope, kv_cache, block_table, seq_lens, batch, sq, num_heads,
                    num_pages, page_size, max_pages, softmax_scale, out, lse, workspace, workspace_bytes, stream);
}

int mla_combine_splits(const float* partial_out, const float* partial_lse, const int32_t* split_indptr, int rows,
                       int num_heads, uint16_t* out, float* lse, void* stream) {
  if (rows < 0 || !split_indptr || !out || !lse) return MLA_ERR_INVALID_ARG;
  if (num_heads != kHeads) return MLA_ERR_UNSUPPORTED;
  if (rows == 0) return MLA_OK;
  if (!partial_out || !partial_lse) return MLA_ERR_INVALID_ARG;
  if (!aligned(partial_out, 16) || !aligned(out, 8)) return MLA_ERR_INVALID_ARG;
  if (launch_combine_indptr(partial_out, partial_lse, split_indptr, rows, reinterpret_cast<__nv_bfloat16*>(out), lse,
                            static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

int mla_profile_next_decode(void* before, void* after) {
  if ((before == nullptr) != (after == nullptr)) return MLA_ERR_INVALID_ARG;
  g_prof_before = static_cast<cudaEvent_t>(before);
  g_prof_after = static_cast<cudaEvent_t>(after);
  return MLA_OK;
}

int mla_get_status(void* workspace, void* stream) {
  if (!workspace) return MLA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MLA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MLA_ERR_CUDA;
  if (v != 0 && cudaMemset(workspace, 0, sizeof(int)) != cudaSuccess) return MLA_ERR_CUDA;
  return v;
}

const char* mla_status_string(int code) {
  switch (code) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_STATUS_BAD_PAGE: return "MLA_STATUS_BAD_PAGE";
    case MLA_STATUS_TIMEOUT: return "MLA_STATUS_TIMEOUT";
    case MLA_STATUS_BAD_SEQ_LEN: return "MLA_STATUS_BAD_SEQ_LEN";
    case MLA_STATUS_BAD_INDEX: return "MLA_STATUS_BAD_INDEX";
    default: return "MLA_UNKNOWN_STATUS";
  }
}

}  // extern "C"
#pragma GCC visibility pop
