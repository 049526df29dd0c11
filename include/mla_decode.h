/*
 * mla_decode.h -- C ABI of the GB300 (sm_103a) MLA decode library.
 *
 * Multi-Head Latent Attention decode over a paged compressed-latent KV cache
 * ("DeepSeek R1 Architecture & Deployment Guide", section 1.1, matrix
 * absorption and decoupled RoPE).  Each cached token is one row
 * [c_KV (512) | k_R (64)] = 576 values.  The 128 query heads arrive absorbed:
 * q_absorbed = (W^UK)^T q (512 values) and q_rope (64 values, already
 * rotated).  For every query row and head h the library computes
 *
 *     s_j   = scale * (q_absorbed[h] . c_KV_j + q_rope[h] . k_R_j)
 *     out[h]= sum_j softmax_j(s) * c_KV_j            (512 values, latent space)
 *     lse[h]= ln sum_j exp(s_j)                      (natural log, scale included)
 *
 * V is the latent c_KV itself (W^UV is folded into the output projection,
 * same section); k_R enters the scores only.
 *
 * Layouts (all row-major, contiguous, device memory unless stated):
 *   q_absorbed  [B, Sq, 128, 512] bf16      q_rope [B, Sq, 128, 64] bf16
 *   kv_cache    bf16: [num_pages, 64, 576]  (1152 B per token)
 *               fp8 : [num_pages, 64, 594] bytes: 576 e4m3 codes then 18
 *                     e8m0 scales, scale k covering values [32k, 32k+32)
 *                     (inlined per-token scales, "DeepSeek-R1" model record,
 *                     engine kernel constraint (2); 16-byte aligned base)
 *   block_table [B, max_pages] int32: page p_index of row b; token t of row
 *               b is page block_table[b][t/64], slot t%64 (page-block size
 *               64, same record, constraint (1)).  Entries past
 *               ceil(seq_len/64) are never read.
 *   seq_lens    [B] int32, 0 <= seq_len <= max_pages*64.
 *   out         [B, Sq, 128, 512] bf16      lse [B, Sq, 128] fp32
 *
 * softmax_scale must be finite and > 0.
 *
 * Speculative multi-token queries (Multi-Token Prediction, guide section 4):
 * query i of Sq sees the first seq_len - (Sq-1-i) tokens.  A query row that
 * sees no token gets out = 0 and lse = -inf.
 *
 * Ownership: the caller owns every buffer; the library never allocates,
 * frees or synchronises inside the decode calls.  All work is queued on
 * `stream` (a cudaStream_t passed as void*; NULL = legacy default stream).
 * Tokens past seq_len inside a row's last page are ignored whatever they
 * hold (including NaN).
 *
 * Stream order: the decode calls' kernels are chained with programmatic
 * dependent launch.  The first one (the planner) is launched as a
 * programmatic dependent of whatever precedes it on `stream` and waits for
 * it before reading any input, so inputs written by earlier work on the
 * stream are always seen.  The last one (the merge) lets a programmatic
 * dependent that follows it begin launching early; such a kernel must wait
 * for its predecessor (griddepcontrol.wait) before reading out or lse, as
 * programmatic dependent launch requires of any kernel.
 *
 * Threads and devices: every call works on the calling thread's current
 * CUDA device.  The first call on a device sets the kernels' shared-memory
 * limits and caches the number of resident CTA pairs in process-wide
 * variables that take no lock, so make the first call on each device from
 * one thread; later calls may come from any thread, each with its own
 * stream and workspace (mla_profile_next_decode is per thread).
 *
 * Errors: host-side validation failures return a negative mla_status before
 * anything is launched.  Launch failures return MLA_ERR_CUDA.  Problems only
 * the device can see (a block-table entry outside [0, num_pages), a
 * seq_len outside [0, max_pages*64], an internal wait that timed out) are
 * recorded in a status word inside the workspace, read by mla_get_status.
 * A bad page is never read: its rows are taken as zeros.
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = -1,   /* null pointer, negative size, bad alignment  */
  MLA_ERR_UNSUPPORTED = -2,   /* num_heads != 128, page_size != 64, Sq > 4   */
  MLA_ERR_WORKSPACE = -3,     /* workspace too small                          */
  MLA_ERR_CUDA = -4,          /* a CUDA runtime call failed                   */
  MLA_STATUS_BAD_PAGE = -5,   /* device: block-table entry out of range       */
  MLA_STATUS_TIMEOUT = -6,    /* device: a pipeline wait gave up              */
  MLA_STATUS_BAD_SEQ_LEN = -7, /* device: seq_len outside [0, max_pages*64]   */
  MLA_STATUS_BAD_INDEX = -8    /* device: sparse token slot outside [-1, num_pages*64) */
} mla_status;

/* Bytes of device workspace a decode call with these sizes needs on the
 * current device (the split-KV plan, per-split partial outputs and the
 * status word).  Returns MLA_OK and writes *bytes, or a negative status.
 * The size does not depend on max_pages (the partials are bounded by the
 * number of CTA pairs, not by the context length), so that argument is not
 * taken; a status return keeps size and error apart. */
int mla_workspace_size(int batch, int sq, int num_heads, int page_size, size_t* bytes);

/* MLA decode over a bf16 latent cache (guide section 1.1; see top of file).
 * Queues three kernels: the split-KV planner, the paired tcgen05 decode
 * kernel, and the merge of the rows it split (the rule of
 * mla_combine_splits).  workspace: device memory of at least
 * mla_workspace_size(...) bytes, 256-byte aligned, not shared with a call
 * that may run concurrently.  Returns MLA_OK or a negative mla_status. */
int mla_decode_bf16(const uint16_t* q_absorbed, const uint16_t* q_rope,
                    const uint16_t* kv_cache, const int32_t* block_table,
                    const int32_t* seq_lens, int batch, int sq, int num_heads,
                    int num_pages, int page_size, int max_pages,
                    float softmax_scale, uint16_t* out, float* lse,
                    void* workspace, size_t workspace_bytes, void* stream);

/* mla_decode_bf16 without a caller workspace.  The method has no
 * counterpart to this call: it exists for callers that cannot hand the
 * library device memory, such as a host that has already given (almost) all
 * of HBM to its KV-cache pool, a loop that must not block in
 * cudaMalloc/cudaFree (both may synchronise the device), or a foreign runtime
 * that gives its plug-ins no device allocator.  The call itself allocates
 * nothing: its scratch is one 40 MiB array that the library owns as a static
 * device variable (one copy per device).
 *
 * Set-up: the first call on each device, with that device current, looks up
 * the array's address (cudaGetSymbolAddress) and caches it; make that first
 * call before any stream capture begins.  A failed look-up returns
 * MLA_ERR_CUDA and is retried by the next call.
 *
 * Limit: batch * sq <= 8192 query rows, and the call's split-KV plan and
 * partial outputs must fit the 40 MiB array.  They take about 20 MiB on a
 * GB300 (76 resident CTA pairs on 152 SMs) whatever the batch, and grow
 * with the number of resident pairs of the device.  A request beyond either
 * bound returns MLA_ERR_WORKSPACE before anything is queued.
 *
 * Concurrency: every call on one device shares the one scratch array.  Calls
 * queued on the same stream are ordered and safe; calls whose work can
 * overlap in time (other streams, other host threads) race on it and give
 * undefined results.
 *
 * device_status: NULL, or 4 bytes of device memory, which receive this
 * call's device status (MLA_OK or an MLA_STATUS_* code, as mla_get_status
 * would report it) once the call's work has run on `stream`.  The status
 * word is cleared at the start of every call.
 * All other arguments, layouts and results are those of mla_decode_bf16. */
int mla_decode_bf16_noalloc(const uint16_t* q_absorbed, const uint16_t* q_rope,
                            const uint16_t* kv_cache, const int32_t* block_table,
                            const int32_t* seq_lens, int batch, int sq,
                            int num_heads, int num_pages, int page_size,
                            int max_pages, float softmax_scale, uint16_t* out,
                            float* lse, int* device_status, void* stream);

/* Same over the FP8 cache: each 594-byte row is dequantised as
 * v[k] = e4m3(byte[k]) * 2^(byte[576 + k/32] - 127) ("DeepSeek-R1" model
 * record, engine kernel constraint (2): e4m3 values, one e8m0 scale per 32)
 * and then attended as the bf16 path does.  The dequantised values are exact
 * in bf16; when every scale exponent of the call lies in [113, 134] and every
 * query value fits f16 they are exact in f16 too, and the MMAs take f16
 * operands (the query and the softmax weights rounded to f16 instead of
 * bf16); otherwise a second pass recomputes the call with bf16 operands.
 * kv_cache must be 16-byte aligned. */
int mla_decode_fp8(const uint16_t* q_absorbed, const uint16_t* q_rope,
                   const uint8_t* kv_cache, const int32_t* block_table,
                   const int32_t* seq_lens, int batch, int sq, int num_heads,
                   int num_pages, int page_size, int max_pages,
                   float softmax_scale, uint16_t* out, float* lse,
                   void* workspace, size_t workspace_bytes, void* stream);

/* Same over an FP4 cache [num_pages, 64, 324] (uint8).  The "DeepSeek-R1"
 * model record (engine kernel constraint (2)) gives only the size of the
 * FP4 variant, 288 bytes per token for a 512-value row; the reading taken
 * is e2m1 codes for every value (two per byte, value 2k in the low nibble
 * of byte k) followed by one e8m0 scale per 16 values, which is 256 + 32 =
 * 288 bytes for 512 values and 288 + 36 = 324 bytes for this 576-value row:
 *   v[k] = e2m1(nibble k) * 2^(byte[288 + k/16] - 127),
 * e2m1 = OCP MX FP4: sign, 2 exponent bits (bias 1), 1 mantissa bit.
 * The values are exact in bf16 for scale bytes in [0, 252] (255 is NaN;
 * 253 and 254 overflow).  As for FP8, when every scale byte of the call
 * lies in [113, 140] and every query value fits f16 the values are exact in
 * f16 too and the MMAs take f16 operands; otherwise a second pass
 * recomputes the call with bf16 operands.  kv_cache must be 16-byte
 * aligned.  Arguments, layouts,
 * results and errors are otherwise those of mla_decode_bf16. */
int mla_decode_fp4(const uint16_t* q_absorbed, const uint16_t* q_rope,
                   const uint8_t* kv_cache, const int32_t* block_table,
                   const int32_t* seq_lens, int batch, int sq, int num_heads,
                   int num_pages, int page_size, int max_pages,
                   float softmax_scale, uint16_t* out, float* lse,
                   void* workspace, size_t workspace_bytes, void* stream);

/* Same over an FP8 cache in the V4.1 row layout [num_pages, 64, 528]
 * (uint8; "DeepSeek-R1" model record, engine kernel constraint (2): 512
 * e4m3 values over all 512 dims, the 64 RoPE dims quantised too, then 16
 * e8m0 scales, one per 32 values).  Reading taken: the 512 values are 448
 * latent values followed by the 64 RoPE values:
 *   v[k] = e4m3(byte[k]) * 2^(byte[512 + k/32] - 127),
 * latent = v[0..447], RoPE key = v[448..511].  The call runs on the
 * 512-value latent layout of the other entry points with latent dims
 * [448, 512) taken as zero: q_absorbed keeps its [.., 512] shape and its
 * dims 448..511 are ignored (read as zero, whatever they hold), and out
 * dims 448..511 are written as 0.  Exactness, the f16-operand pass and its
 * fallback are those of mla_decode_fp8; kv_cache must be 16-byte aligned.
 * Arguments, layouts, results and errors are otherwise those of
 * mla_decode_bf16. */
int mla_decode_fp8_v41(const uint16_t* q_absorbed, const uint16_t* q_rope,
                       const uint8_t* kv_cache, const int32_t* block_table,
                       const int32_t* seq_lens, int batch, int sq, int num_heads,
                       int num_pages, int page_size, int max_pages,
                       float softmax_scale, uint16_t* out, float* lse,
                       void* workspace, size_t workspace_bytes, void* stream);

/* Same over an FP4 cache in the record's own 288-byte row [num_pages, 64,
 * 288] (uint8; the FP4 variant of the V4.1 row, 512 values): 256 bytes of
 * e2m1 codes (two per byte, value 2k in the low nibble of byte k), then 32
 * e8m0 scales, one per 16 values:
 *   v[k] = e2m1(nibble k) * 2^(byte[256 + k/16] - 127),
 * latent = v[0..447], RoPE key = v[448..511], as for mla_decode_fp8_v41
 * (query dims 448..511 ignored, output dims 448..511 written as 0).
 * Exactness and the f16-operand pass are those of mla_decode_fp4;
 * kv_cache must be 16-byte aligned. */
int mla_decode_fp4_v41(const uint16_t* q_absorbed, const uint16_t* q_rope,
                       const uint8_t* kv_cache, const int32_t* block_table,
                       const int32_t* seq_lens, int batch, int sq, int num_heads,
                       int num_pages, int page_size, int max_pages,
                       float softmax_scale, uint16_t* out, float* lse,
                       void* workspace, size_t workspace_bytes, void* stream);

/* Sparse top-k decode ("DeepSeek-V3.2" model record: the sparse attention
 * indexer, index_topk 2048, selects the candidate tokens each query attends
 * over; the latent rows stay cached per token).  Query row (b, i) attends
 * over the tokens listed in token_slots[b][i][0..topk): each entry is a
 * physical cache slot, page * 64 + offset into kv_cache (bf16
 * [num_pages, 64, 576]), or -1 for "no token".  No other mask applies; a
 * slot listed twice counts twice.  The scores, softmax, out and lse are
 * those of mla_decode_bf16.  A row with no listed token gets out = 0 and
 * lse = -inf.  An entry outside [-1, num_pages*64) is skipped and sets
 * MLA_STATUS_BAD_INDEX.
 * token_slots: int32 [batch, sq, topk], device; 1 <= topk <= 16384.
 * workspace: mla_workspace_size_sparse(...) bytes, 256-byte aligned. */
int mla_workspace_size_sparse(int batch, int sq, int topk, int num_heads, int page_size, size_t* bytes);
int mla_decode_sparse_bf16(const uint16_t* q_absorbed, const uint16_t* q_rope,
                           const uint16_t* kv_cache, const int32_t* token_slots,
                           int batch, int sq, int topk, int num_heads,
                           int num_pages, int page_size, float softmax_scale,
                           uint16_t* out, float* lse, void* workspace,
                           size_t workspace_bytes, void* stream);

/* Up-projection of latent attention outputs through W^UV ("DeepSeek R1
 * Architecture & Deployment Guide", section 1.1: the value up-projection is
 * folded out of the attention, which returns the 512-value latent output
 * per head): out[r][h][:] = W_uv[h] . latent[r][h][:], i.e. per head the GEMM
 * [rows x 512] . [512 x d_v].  latent [rows, 128, 512] bf16 (the decode's
 * out), w_uv [128, d_v, 512] bf16, out [rows, 128, d_v] bf16 (fp32
 * accumulation, rounded to nearest).  num_heads must be 128 and d_v 128.
 * workspace: at least 256 bytes, 256-byte aligned; it receives the status
 * word (read with mla_get_status; the decode's workspace may be reused). */
int mla_up_project_wuv(const uint16_t* latent, const uint16_t* w_uv, int rows, int num_heads, int d_v,
                       uint16_t* out, void* workspace, size_t workspace_bytes, void* stream);

/* Merge split-KV partial results (attention over disjoint token sets):
 *   L = ln sum_s exp(lse_s),  out = sum_s exp(lse_s - L) * partial_out_s,
 *   lse = L.
 * Source: the 128K-token contexts of "DeepSeek R1 Architecture & Deployment
 * Guide", section 1.1, are far more than one SM pair can stream in time, so
 * a long row is cut into parts whose softmax results are combined exactly
 * by this log-sum-exp rule (the decode calls run it on their own splits;
 * this entry point merges parts a caller produced).
 * partial_out [n_parts, num_heads, 512] fp32 (each part already normalised
 * by its own softmax sum), partial_lse [n_parts, num_heads] fp32,
 * split_indptr [rows+1] int32: row r merges parts [indptr[r], indptr[r+1]).
 * The call has no n_parts argument and reads the parts split_indptr names
 * without a bound: it must start at 0, never decrease and end at most at
 * n_parts (device memory, so the host cannot check it).
 * A row with no part (or whose parts all have lse = -inf) gets out = 0,
 * lse = -inf.  out [rows, num_heads, 512] bf16, lse [rows, num_heads] fp32.
 * num_heads must be 128. */
int mla_combine_splits(const float* partial_out, const float* partial_lse,
                       const int32_t* split_indptr, int rows, int num_heads,
                       uint16_t* out, float* lse, void* stream);

/* Synchronises `stream`, then returns the device status word recorded in
 * `workspace` by the calls queued before (MLA_OK or an MLA_STATUS_* code)
 * and clears it.  Returns MLA_ERR_CUDA if the stream reported an error. */
int mla_get_status(void* workspace, void* stream);

/* Profiling hook: when both events are non-NULL, the next decode call on this
 * host thread records `before` on its stream just before the attention
 * kernel and `after` just after it (planner and merge excluded), then clears
 * the hook.  The events are cudaEvent_t handles passed as void*.  Used to time
 * the attention kernel alone; it changes nothing else. */
int mla_profile_next_decode(void* before, void* after);

/* Static string naming a status code. */
const char* mla_status_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H_ */
