// Paired tcgen05 MLA decode kernel for sm_103a.
//
// What it computes ("DeepSeek R1 Architecture & Deployment Guide", section
// 1.1): for one query row (128 absorbed heads) over a row's paged latent
// cache, s = scale * Q[128 x 576] . K^T with K the gathered rows
// [c_KV | k_R]; P = online softmax(s); O[128 x 512] = P . V with V = c_KV
// (the first 512 columns of the same rows); out = O / l, lse = m + ln l.
//
// Why a CTA pair.  O for 128 heads x 512 latent columns in fp32 is exactly
// the 512-column x 128-lane tensor memory of one SM, so S cannot live beside
// it.  Each 2-CTA cluster splits the work by role, not by data, and no FLOP
// is computed twice:
//   rank 1 ("score SM"): Q [128 x 576] bf16 resident in TMEM (288 columns);
//       per 64-token page S = Q . K^T (36 tcgen05.mma, M=128, N=64, A from
//       TMEM) into one of two 64-column S buffers; eight softmax warps in two
//       groups (columns 0..31 and 32..63 of each head row; both take the row
//       max over all 64 columns, so their reference maxima agree without an
//       exchange) round P to bf16 and send it with st.async into rank 0's
//       shared memory in the 128B-swizzled K-major layout its MMA reads; the
//       bytes are counted on rank 0's barrier, so no thread waits for them.
//   rank 0 ("value SM"): O [128 x 512] fp32 in all 512 TMEM columns;
//       O += P . V with P from shared memory and V read from the page tile as
//       an MN-major operand (two M=128, N=256, K=16 MMAs per 16 tokens); its
//       epilogue warps rescale O when rank 1 moves a head's reference max and
//       write out = O / l (or an fp32 split partial).
// Page loads.  One TMA operation per page per rank: the bf16 cache is
// described as a 3-D tensor (64 columns, rows, 9 column chunks) with row
// stride 1152 B and chunk stride 128 B, so a single box of 64 x 64 x 9 (rank
// 1, 72 KiB) or 64 x 64 x 8 (rank 0, 64 KiB) lands as nine (eight) 128B-
// swizzled chunks of 64 rows -- exactly the operand layout -- in one copy.
// An SM's copy engine streams far more bytes per second in large operations
// than in 8 KiB boxes, so whole-page copies are what lets 152 SMs reach HBM
// speed.  Both ranks read every page; the second read is an L2 hit.  The FP8
// cache is bulk-copied as raw half pages and dequantised by four warps into
// the same layouts.
//
// Lazy rescaling: rank 1 keeps a per-head reference max m_ref (raw score
// units) and moves it only when a page's max exceeds it by more than 8 in
// log2 units, so P <= 256 and O is rescaled only on those rare pages.
//
// Every wait is bounded (wait_bounded / wait_warp); a timeout records
// MLA_STATUS_TIMEOUT and raises an abort flag so every role leaves its loop
// and the kernel ends through the normal teardown.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstring>

#include "decode.cuh"

namespace mla {

namespace dk {

constexpr uint32_t kChunkBytes = 64 * 128;            // 64 rows x 64 bf16, 128B swizzle
constexpr uint32_t kVPageBytes = 8 * kChunkBytes;     // latent c_KV part of one page (64 KiB)
constexpr uint32_t kPSlotBytes = 128 * 128;           // P of one page: 128 heads x 64 tokens bf16
constexpr int kPSlots = 2;
constexpr int kMailSlots = 2;
constexpr uint32_t kRawBytes = 32 * kFp8Row;          // half a page of FP8 rows: 19,008 B
constexpr int kMaxStages = 3, kMaxRaw = 4;

// Shared-memory plans (bytes).  The small common region (alpha, 1/l, flags,
// barriers) sits at the same offset in both ranks so remote stores and
// arrivals can address it.
//   bf16: rank 1 = 3 K pages of 72 KiB (chunks 0..8 contiguous);
//         rank 0 = 3 V pages of 64 KiB + 2 P slots.
//   FP8:  rank 1 = 2 bf16 K pages (latent chunks at stage*64K, RoPE chunk in
//         a separate ring) + 4 raw half pages; rank 0 = 2 V pages + 2 P slots
//         + 3 raw half pages.
template <int kMode> struct Cfg;
template <> struct Cfg<0> {
  static constexpr int kStages = 3;
  static constexpr int kRaw1 = 0, kRaw0 = 0;
  static constexpr uint32_t kKStageBytes = 9 * kChunkBytes;
  static constexpr uint32_t kOffRope = 0;                           // unused: RoPE chunk is chunk 8 of the stage
  static constexpr uint32_t kOffP = kStages * kVPageBytes;
  static constexpr uint32_t kOffRaw1 = 0, kOffRaw0 = 0;
  static constexpr uint32_t kOffMisc = kOffP + kPSlots * kPSlotBytes;
  static constexpr int kThreads = 384;
  __device__ static uint32_t k_chunk(int stage, int c) { return stage * kKStageBytes + c * kChunkBytes; }
};
template <> struct Cfg<1> {
  static constexpr int kStages = 2;
  static constexpr int kRaw1 = 4, kRaw0 = 3;
  static constexpr uint32_t kKStageBytes = kVPageBytes;
  static constexpr uint32_t kOffRope = kStages * kVPageBytes;       // rank 1: RoPE chunk ring
  static constexpr uint32_t kOffP = kStages * kVPageBytes;          // rank 0: P slots
  static constexpr uint32_t kOffRaw1 = kOffRope + kStages * kChunkBytes;
  static constexpr uint32_t kOffRaw0 = kOffP + kPSlots * kPSlotBytes;
  static constexpr uint32_t kOffMisc = kOffRaw1 + kRaw1 * kRawBytes;
  static constexpr int kThreads = 512;
  __device__ static uint32_t k_chunk(int stage, int c) {
    return c < 8 ? stage * kVPageBytes + c * kChunkBytes : kOffRope + stage * kChunkBytes;
  }
};
constexpr uint32_t kMiscAlpha = 0;       // rank 0: fp32 alpha [2][128]
constexpr uint32_t kMiscLPart = 0;       // rank 1 (same bytes): group-1 partial softmax sums [128]
constexpr uint32_t kMiscMail = 1024;     // rank 0: fp32 1/l [2][128]
constexpr uint32_t kMiscReq = 2048;      // rank 0: P slot of a rescale request
constexpr uint32_t kMiscRawFlag = 2064;  // per raw stage: 1 = write zeros (bad page)
constexpr uint32_t kMiscBar = 2080;
enum Bar {
  FULL = 0, EMPTY = FULL + kMaxStages,
  PFULL = EMPTY + kMaxStages, PEMPTY = PFULL + kPSlots,
  SFULL = PEMPTY + kPSlots, SEMPTY = SFULL + 2,
  QREADY = SEMPTY + 2, REQ, CORR, OFULL, OEMPTY, LSUM,
  MBFULL, MBEMPTY = MBFULL + kMailSlots,
  RAWFULL = MBEMPTY + kMailSlots, RAWEMPTY = RAWFULL + kMaxRaw,
  NBAR = RAWEMPTY + kMaxRaw
};
constexpr uint32_t kMiscTmem = kMiscBar + NBAR * 8;
constexpr uint32_t kMiscBytes = kMiscTmem + 16;
template <int kMode> constexpr uint32_t smem_bytes() { return Cfg<kMode>::kOffMisc + kMiscBytes; }
static_assert(smem_bytes<0>() <= 232448 && smem_bytes<1>() <= 232448, "shared memory budget");
static_assert(3 * 9 * kChunkBytes <= Cfg<0>::kOffMisc, "rank 1 plan (bf16)");
static_assert(Cfg<1>::kOffRaw0 + Cfg<1>::kRaw0 * kRawBytes <= Cfg<1>::kOffMisc, "rank 0 plan (fp8)");

// TMEM columns.
constexpr uint32_t kQCol = 0;      // rank 1: Q, 288 columns (2 bf16 per column)
constexpr uint32_t kSCol = 320;    // rank 1: two S buffers of 64 columns
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kIdescS = ptx::idesc_bf16(128, 64, 0, 0);    // A = Q (TMEM, K-major), B = K (K-major)
constexpr uint32_t kIdescPV = ptx::idesc_bf16(128, 256, 0, 1);  // A = P (K-major), B = V (MN-major)

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units: P <= 2^8

struct Segment {
  int b;          // batch row
  int t0, t1;     // row-local page range [t0, t1)
};

// Walks the segments of one pair: the pair's page range [lo, hi) cut at row
// boundaries.  Every role of both ranks walks the same sequence.
struct SegWalker {
  const int* tile_start;
  int batch, b, lo, hi;
  __device__ void init(const int* ts, int nb, int lo_, int hi_) {
    tile_start = ts; batch = nb; lo = lo_; hi = hi_;
    b = 0;
    if (lo >= hi) { b = nb; return; }
    int l = 0, r = nb - 1;            // largest b with ts[b] <= lo
    while (l < r) {
      const int mid = (l + r + 1) >> 1;
      if (__ldg(ts + mid) <= lo) l = mid; else r = mid - 1;
    }
    b = l;
  }
  __device__ bool next(Segment& s) {
    while (b < batch) {
      const int a = __ldg(tile_start + b), e = __ldg(tile_start + b + 1);
      if (a >= hi) { b = batch; return false; }
      const int cb = b++;
      if (e > a) {
        s.b = cb;
        s.t0 = max(lo, a) - a;
        s.t1 = min(hi, e) - a;
        if (s.t1 > s.t0) return true;
      }
    }
    return false;
  }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 32 e4m3 codes (8 words, lowest byte first) with their e8m0 scale byte ->
// 16 bf16x2 words.  e4m3 -> f16 is exact in hardware, the product with the
// power-of-two scale is exact in fp32 (no flush), and the result has at most
// 4 significant bits, so the bf16 rounding is exact too.  NaN codes and the
// NaN scale (0xFF) give NaN, as in the format definitions.
__device__ __forceinline__ void dequant32(const uint32_t* wd, uint32_t e, uint32_t* o) {
  const float sc = __uint_as_float(e == 0 ? 0x00400000u : (e == 255 ? 0x7FC00000u : (e << 23)));
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t h01, h23;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h01) : "h"(static_cast<unsigned short>(wd[i] & 0xFFFFu)));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h23) : "h"(static_cast<unsigned short>(wd[i] >> 16)));
    const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
    const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
    o[2 * i] = pack_bf16x2(f01.x * sc, f01.y * sc);
    o[2 * i + 1] = pack_bf16x2(f23.x * sc, f23.y * sc);
  }
}

// Dequantise value group g (32 values) of raw FP8 row `row` (2-byte aligned
// in shared memory) into 16 bf16x2 words.  The 32 codes are read as nine
// aligned words and funnel-shifted by the row's misalignment (0 or 2 bytes).
__device__ __forceinline__ void dequant_group(const uint8_t* row, int g, uint32_t* o) {
  const uint8_t* src = row + 32 * g;
  const uintptr_t a = reinterpret_cast<uintptr_t>(src);
  const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~static_cast<uintptr_t>(3));
  const uint32_t sh = static_cast<uint32_t>(a & 3u) * 8u;
  uint32_t u[9], wd[8];
#pragma unroll
  for (int i = 0; i < 9; ++i) u[i] = w[i];
#pragma unroll
  for (int i = 0; i < 8; ++i) wd[i] = __funnelshift_r(u[i], u[i + 1], sh);
  dequant32(wd, row[kRow + g], o);
}

// Store 16 bf16x2 words (32 values of value group g) into row `r` of a
// 128B-swizzled chunk whose 128-byte rows hold 64 values (two groups).
__device__ __forceinline__ void store_group(uint8_t* chunk, int r, int g, const uint32_t* o) {
  uint8_t* dst = chunk + r * 128;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int piece = ((g & 1) * 4 + j) ^ (r & 7);
    *reinterpret_cast<uint4*>(dst + piece * 16) = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
  }
}

}  // namespace dk

template <int kMode>   // 0: bf16 cache via TMA, 1: FP8 cache via bulk copies + dequant
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(dk::Cfg<kMode>::kThreads, 1)
mla_decode_pair_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                       const DecodeParams p) {
  using namespace dk;
  using C = Cfg<kMode>;
  constexpr int kStages = C::kStages;
  constexpr uint32_t kOffAlpha = C::kOffMisc + kMiscAlpha;
  constexpr uint32_t kOffMail = C::kOffMisc + kMiscMail;
  constexpr uint32_t kOffReq = C::kOffMisc + kMiscReq;
  constexpr uint32_t kOffRawFlag = C::kOffMisc + kMiscRawFlag;
  constexpr uint32_t kOffBar = C::kOffMisc + kMiscBar;
  constexpr uint32_t kOffTmemPtr = C::kOffMisc + kMiscTmem;

  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t rank = ptx::cluster_ctarank();
  const uint32_t pair = ptx::cluster_id_x();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  PlanHeader* hdr = reinterpret_cast<PlanHeader*>(p.ws);
  const int* lens = reinterpret_cast<const int*>(p.ws + p.L.lens);
  const int* tile_start = reinterpret_cast<const int*>(p.ws + p.L.tile_start);
  const int* first_pair = reinterpret_cast<const int*>(p.ws + p.L.first_pair);
  const int* slot_base = reinterpret_cast<const int*>(p.ws + p.L.slot_base);
  float* part_lse = reinterpret_cast<float*>(p.ws + p.L.part_lse);
  float* part_out = reinterpret_cast<float*>(p.ws + p.L.part_out);
  auto BAR = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * static_cast<uint32_t>(i); };

  const bool smem_ok = (sbase & 1023u) == 0;
  if (threadIdx.x == 0) {
    if (!smem_ok) set_status(&hdr->status, MLA_ERR_UNSUPPORTED);
    for (int s = 0; s < kMaxStages; ++s) {
      ptx::mbar_init(BAR(FULL + s), kMode == 0 ? 1u : 4u);   // TMA bytes, or the 4 dequant warps
      ptx::mbar_init(BAR(EMPTY + s), 1);
    }
    for (int s = 0; s < kPSlots; ++s) { ptx::mbar_init(BAR(PFULL + s), 256); ptx::mbar_init(BAR(PEMPTY + s), 1); }
    for (int s = 0; s < 2; ++s) { ptx::mbar_init(BAR(SFULL + s), 1); ptx::mbar_init(BAR(SEMPTY + s), 256); }
    ptx::mbar_init(BAR(QREADY), 128);
    ptx::mbar_init(BAR(REQ), 2);
    ptx::mbar_init(BAR(CORR), 4);
    ptx::mbar_init(BAR(OFULL), 1);
    ptx::mbar_init(BAR(OEMPTY), 128);
    ptx::mbar_init(BAR(LSUM), 128);
    for (int s = 0; s < kMailSlots; ++s) { ptx::mbar_init(BAR(MBFULL + s), 128); ptx::mbar_init(BAR(MBEMPTY + s), 4); }
    for (int s = 0; s < kMaxRaw; ++s) { ptx::mbar_init(BAR(RAWFULL + s), 1); ptx::mbar_init(BAR(RAWEMPTY + s), 4); }
    ptx::fence_barrier_init();
  }
  if (warp == 2) {
    ptx::tmem_alloc(sbase + kOffTmemPtr, kTmemCols);
    ptx::tmem_relinquish();
  }
  if (kMode == 0 && warp == 0 && lane == 0) ptx::prefetch_tmap(rank == 1 ? &tmap_k : &tmap_v);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  ptx::cluster_sync();   // barriers of both ranks initialised before any remote arrive
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffTmemPtr);

  const int ppg = hdr->pairs_per_group;
  const int group = static_cast<int>(pair) / ppg;     // query index i served by this pair
  const int pl = static_cast<int>(pair) % ppg;
  const int chunk = hdr->chunk;
  const int n_tiles = hdr->n_tiles;
  const int spq = hdr->slots_per_query;
  const int lo = min(pl * chunk, n_tiles), hi = min(lo + chunk, n_tiles);
  const int sq = p.sq;
  const bool active = smem_ok && group < sq;

  if (active && warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = ptx::policy_evict_normal();
      SegWalker w; w.init(tile_start, p.batch, lo, hi);
      Segment sg;
      int stage = 0; uint32_t phase = 0;
      int rs = 0; uint32_t rphase = 0;
      const int n_raw = rank == 1 ? C::kRaw1 : C::kRaw0;
      const uint32_t raw_off = rank == 1 ? C::kOffRaw1 : C::kOffRaw0;
      volatile uint32_t* raw_flag = reinterpret_cast<volatile uint32_t*>(smem + kOffRawFlag);
      bool ok = true;
      while (ok && w.next(sg)) {
        for (int t = sg.t0; t < sg.t1 && ok; ++t) {
          int page = __ldg(p.block_table + static_cast<size_t>(sg.b) * p.max_pages + t);
          const bool bad = page < 0 || page >= p.num_pages;
          if (bad) set_status(&hdr->status, MLA_STATUS_BAD_PAGE);
          if constexpr (kMode == 0) {
            // one copy per page: rank 1 all nine chunks (72 KiB), rank 0 the
            // eight latent chunks (64 KiB); a bad page is read fully outside
            // the tensor, which fills zeros
            if (!wait_bounded<true>(BAR(EMPTY + stage), phase ^ 1u, hdr)) { ok = false; break; }
            const int y = (bad ? p.num_pages : page) * kPage;
            if (rank == 1) {
              ptx::mbar_arrive_expect_tx(BAR(FULL + stage), 9u * kChunkBytes);
              ptx::tma_load_3d(sbase + C::k_chunk(stage, 0), &tmap_k, BAR(FULL + stage), 0, y, 0, pol);
            } else {
              ptx::mbar_arrive_expect_tx(BAR(FULL + stage), kVPageBytes);
              ptx::tma_load_3d(sbase + static_cast<uint32_t>(stage) * kVPageBytes, &tmap_v, BAR(FULL + stage),
                               0, y, 0, pol);
            }
            if (++stage == kStages) { stage = 0; phase ^= 1u; }
          } else {
            // two raw half pages; a bad page is never read (dequant writes zeros)
            for (int half = 0; half < 2; ++half) {
              if (!wait_bounded<true>(BAR(RAWEMPTY + rs), rphase ^ 1u, hdr)) { ok = false; break; }
              raw_flag[rs] = bad ? 1u : 0u;
              if (bad) {
                ptx::mbar_arrive(BAR(RAWFULL + rs));
              } else {
                ptx::mbar_arrive_expect_tx(BAR(RAWFULL + rs), kRawBytes);
                const uint8_t* src = p.kv_fp8 + static_cast<size_t>(page) * (kPage * kFp8Row) + half * kRawBytes;
                ptx::bulk_load(sbase + raw_off + static_cast<uint32_t>(rs) * kRawBytes, src, kRawBytes,
                               BAR(RAWFULL + rs), pol);
              }
              if (++rs == n_raw) { rs = 0; rphase ^= 1u; }
            }
          }
        }
      }
    }
  } else if (kMode == 1 && active && warp >= 12) {
    // ------------------------------------------------------------ FP8 dequant (warps 12..15)
    // raw half page -> bf16 operand rows [32*half, 32*half+32) of the page.
    // Warp wq handles tokens of parity (wq & 1) (so the row's 2-byte
    // misalignment is warp-uniform) and half of the 32-value groups (9 of 18
    // on rank 1, 8 of the 16 latent groups on rank 0).
    const int wq = warp - 12;
    const int parity = wq & 1;
    const int G = rank == 1 ? 9 : 8;
    const int g0 = (wq >> 1) * G;
    const int n_tasks = 16 * G;
    const int n_raw = rank == 1 ? C::kRaw1 : C::kRaw0;
    const uint32_t raw_off = rank == 1 ? C::kOffRaw1 : C::kOffRaw0;
    const volatile uint32_t* raw_flag = reinterpret_cast<const volatile uint32_t*>(smem + kOffRawFlag);
    SegWalker w; w.init(tile_start, p.batch, lo, hi);
    Segment sg;
    int stage = 0; uint32_t phase = 0;
    int rs = 0; uint32_t rphase = 0;
    bool ok = true;
    while (ok && w.next(sg)) {
      for (int t = sg.t0; t < sg.t1 && ok; ++t) {
        if (!wait_warp<true>(BAR(EMPTY + stage), phase ^ 1u, hdr)) { ok = false; break; }
        for (int half = 0; half < 2; ++half) {
          if (!wait_warp<false>(BAR(RAWFULL + rs), rphase, hdr)) { ok = false; break; }
          const bool zero = raw_flag[rs] != 0;
          const uint8_t* raw = smem + raw_off + static_cast<uint32_t>(rs) * kRawBytes;
          for (int task = lane; task < n_tasks; task += 32) {
            const int tok = 2 * (task / G) + parity;          // token within the half page
            const int g = g0 + task % G;                       // 32-value group
            uint32_t o[16];
            if (!zero) {
              dequant_group(raw + tok * kFp8Row, g, o);
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i) o[i] = 0u;
            }
            store_group(smem + C::k_chunk(stage, g >> 1), 32 * half + tok, g, o);
          }
          ptx::fence_proxy_async_cta();      // generic smem writes -> visible to the MMA (async proxy)
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(BAR(RAWEMPTY + rs));
          if (++rs == n_raw) { rs = 0; rphase ^= 1u; }
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(BAR(FULL + stage));
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
    }
  } else if (active && warp == 1 && rank == 1) {
    // ------------------------------------------------------------ S = Q K^T issuer
    SegWalker w; w.init(tile_start, p.batch, lo, hi);
    Segment sg;
    int stage = 0; uint32_t phase = 0;
    int sb = 0; uint32_t sphase = 0;
    uint32_t qphase = 0;
    bool ok = true;
    while (ok && w.next(sg)) {
      if (!wait_warp<false>(BAR(QREADY), qphase, hdr)) break;
      qphase ^= 1u;
      for (int t = sg.t0; t < sg.t1 && ok; ++t) {
        if (!wait_warp<false>(BAR(FULL + stage), phase, hdr) ||
            !wait_warp<false>(BAR(SEMPTY + sb), sphase ^ 1u, hdr)) { ok = false; break; }
        ptx::tc_fence_after();
        if (lane == 0) {
          // descriptors built once per page; each of the 36 MMAs then costs an
          // add and the issue (the start address is the descriptor's low field)
          const uint32_t d = tmem + kSCol + 64u * sb;
          const uint64_t lat0 = ptx::sdesc_sw128(sbase + C::k_chunk(stage, 0), 16, 1024);
          const uint64_t rope0 = ptx::sdesc_sw128(sbase + C::k_chunk(stage, 8), 16, 1024);
#pragma unroll
          for (int k = 0; k < kRow / 16; ++k) {
            const int c = k >> 2, kk = k & 3;
            const uint64_t bdesc = c < 8 ? lat0 + static_cast<uint64_t>((c * kChunkBytes + kk * 32) >> 4)
                                         : rope0 + static_cast<uint64_t>((kk * 32) >> 4);
            ptx::mma_ts(d, tmem + kQCol + 8u * k, bdesc, kIdescS, k > 0 ? 1u : 0u);
          }
          ptx::mma_commit(BAR(EMPTY + stage));
          ptx::mma_commit(BAR(SFULL + sb));
        }
        __syncwarp();
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
        if (++sb == 2) { sb = 0; sphase ^= 1u; }
      }
    }
  } else if (active && warp == 1 && rank == 0) {
    // ------------------------------------------------------------ O += P V issuer
    SegWalker w; w.init(tile_start, p.batch, lo, hi);
    Segment sg;
    int stage = 0; uint32_t phase = 0;
    int ps = 0; uint32_t pphase = 0;
    uint32_t corr_phase = 0, oe_phase = 0;
    bool first_seg = true, ok = true;
    volatile uint32_t* req_slot = reinterpret_cast<volatile uint32_t*>(smem + kOffReq);
    const volatile float* alpha_buf = reinterpret_cast<const volatile float*>(smem + kOffAlpha);
    while (ok && w.next(sg)) {
      const int len_i = lens[sg.b] - (sq - 1 - group);
      for (int t = sg.t0; t < sg.t1 && ok; ++t) {
        if (!wait_warp<false>(BAR(FULL + stage), phase, hdr) ||
            !wait_warp<true>(BAR(PFULL + ps), pphase, hdr)) { ok = false; break; }
        ptx::fence_proxy_async_cta();
        // did rank 1 move its reference max for any head of this page?
        bool moved = false;
#pragma unroll
        for (int i = 0; i < 4; ++i) moved |= alpha_buf[ps * 128 + lane * 4 + i] != 1.f;
        if (__any_sync(0xffffffffu, moved)) {
          // drain prior MMAs, then let the epilogue warps rescale O
          if (lane == 0) {
            *req_slot = static_cast<uint32_t>(ps);
            ptx::mma_commit(BAR(REQ));
            ptx::mbar_arrive(BAR(REQ));
          }
          __syncwarp();
          if (!wait_warp<false>(BAR(CORR), corr_phase, hdr)) { ok = false; break; }
          corr_phase ^= 1u;
        }
        if (t == sg.t0 && !first_seg) {
          if (!wait_warp<false>(BAR(OEMPTY), oe_phase, hdr)) { ok = false; break; }
          oe_phase ^= 1u;
        }
        const uint32_t vpage = static_cast<uint32_t>(stage) * kVPageBytes;
        const int valid = len_i - t * kPage;   // rows of this page visible to the query
        if (valid < kPage) {
          // rows past the visible length get P = 0; make their V finite too
          const int v0 = valid > 0 ? valid : 0;
          uint4* base = reinterpret_cast<uint4*>(smem + vpage);
          const int n16 = (kPage - v0) * 8;     // 16-byte pieces per chunk
          for (int c = 0; c < 8; ++c)
            for (int i = lane; i < n16; i += 32)
              base[(c * kChunkBytes + v0 * 128) / 16 + i] = make_uint4(0, 0, 0, 0);
          ptx::fence_proxy_async_cta();
          __syncwarp();
        }
        ptx::tc_fence_after();
        if (lane == 0) {
          const uint32_t pbase = sbase + C::kOffP + static_cast<uint32_t>(ps) * kPSlotBytes;
          const uint32_t vbase = sbase + vpage;
#pragma unroll
          for (int k = 0; k < kPage / 16; ++k) {
            const uint64_t adesc = ptx::sdesc_sw128(pbase + k * 32, 16, 1024);
#pragma unroll
            for (int n = 0; n < 2; ++n) {
              const uint64_t bdesc = ptx::sdesc_sw128(vbase + n * 4 * kChunkBytes + k * 2048, kChunkBytes, 1024);
              ptx::mma_ss(tmem + 256u * n, adesc, bdesc, kIdescPV, (t > sg.t0 || k > 0) ? 1u : 0u);
            }
          }
          ptx::mma_commit(BAR(EMPTY + stage));
          ptx::mma_commit_mc(BAR(PEMPTY + ps), static_cast<uint16_t>(1u << 1));
          if (t == sg.t1 - 1) ptx::mma_commit(BAR(OFULL));
        }
        __syncwarp();
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
        if (++ps == kPSlots) { ps = 0; pphase ^= 1u; }
      }
      first_seg = false;
    }
  } else if (active && warp >= 4 && warp < 12 && rank == 1) {
    // ------------------------------------------------------------ softmax (thread = head)
    // Group 0 (warps 4..7) turns columns 0..31 of each page's S into P, group
    // 1 (warps 8..11) columns 32..63.  Both take the row max over all 64
    // columns, so their reference maxima and rescale factors agree without an
    // exchange; the two partial sums meet once per segment (LSUM barrier).
    const int grp = (warp - 4) >> 2;
    const int h = (threadIdx.x - 128) & 127;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    volatile float* l_part = reinterpret_cast<volatile float*>(smem + C::kOffMisc + kMiscLPart);
    SegWalker w; w.init(tile_start, p.batch, lo, hi);
    Segment sg;
    int sb = 0; uint32_t sphase = 0;
    int ps = 0; uint32_t pphase = 0;
    int ms = 0; uint32_t mphase = 0;
    uint32_t lsum_phase = 0;
    bool ok = true;
    const float c = p.scale_log2;
    while (ok && w.next(sg)) {
      const int row = sg.b * sq + group;
      const int len_i = lens[sg.b] - (sq - 1 - group);
      if (grp == 0) {
        // Q row h -> TMEM lane h, columns [0, 288): two bf16 per column, K order
        const uint4* qa = reinterpret_cast<const uint4*>(p.q_abs + (static_cast<size_t>(row) * kHeads + h) * kDc);
        const uint4* qr = reinterpret_cast<const uint4*>(p.q_rope + (static_cast<size_t>(row) * kHeads + h) * kDr);
#pragma unroll 1
        for (int c3 = 0; c3 < 3; ++c3) {          // three chunks of 32 columns per round trip
          uint4 x[24];
#pragma unroll
          for (int v = 0; v < 24; ++v) {
            const int cc = c3 * 3 + v / 8;
            x[v] = __ldg((cc < 8 ? qa + cc * 8 : qr) + (v & 7));
          }
#pragma unroll
          for (int j = 0; j < 3; ++j) {
            uint32_t r[32];
#pragma unroll
            for (int v = 0; v < 8; ++v) {
              r[4 * v] = x[8 * j + v].x; r[4 * v + 1] = x[8 * j + v].y;
              r[4 * v + 2] = x[8 * j + v].z; r[4 * v + 3] = x[8 * j + v].w;
            }
            ptx::tmem_st32(tmem + lane_base + kQCol + 32u * (c3 * 3 + j), r);
          }
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(BAR(QREADY));
      }
      float m_ref = -INFINITY, l = 0.f;
      for (int t = sg.t0; t < sg.t1; ++t) {
        if (!wait_warp<false>(BAR(SFULL + sb), sphase, hdr)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t sadr = tmem + lane_base + kSCol + 64u * sb;
        uint32_t mine[32], other[32];
        ptx::tmem_ld32(sadr + 32u * grp, mine);
        ptx::tmem_ld32(sadr + 32u * (grp ^ 1), other);
        ptx::tmem_wait_ld();
        ptx::tc_fence_before();
        ptx::mbar_arrive(BAR(SEMPTY + sb));
        const int valid = len_i - t * kPage;          // columns of this page visible to the query
        const int c_mine = 32 * grp, c_other = 32 * (grp ^ 1);
        // row max of the masked raw scores.  m_ref stays in raw score units and
        // P = exp2((s - m_ref) * c), so the max element gets exactly exp2(0) = 1
        // whatever the magnitude of the scores (scale c > 0).
        float mx = -INFINITY;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          if (c_mine + e < valid) mx = fmaxf(mx, __uint_as_float(mine[e]));
          if (c_other + e < valid) mx = fmaxf(mx, __uint_as_float(other[e]));
        }
        float alpha = 1.f;
        if (t == sg.t0) {
          m_ref = mx;
        } else if ((mx - m_ref) * c > kRescaleThreshold) {
          alpha = fast_exp2((m_ref - mx) * c);
          l *= alpha;
          m_ref = mx;
        }
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int col = c_mine + 2 * e;
          const float p0 = col < valid ? fast_exp2((__uint_as_float(mine[2 * e]) - m_ref) * c) : 0.f;
          const float p1 = col + 1 < valid ? fast_exp2((__uint_as_float(mine[2 * e + 1]) - m_ref) * c) : 0.f;
          pk[e] = pack_bf16x2(p0, p1);
          l += p0 + p1;
        }
        if (m_ref == -INFINITY) l = 0.f;     // nothing visible yet (every p was 0)
        if (!wait_warp<true>(BAR(PEMPTY + ps), pphase ^ 1u, hdr)) { ok = false; break; }
        // This group's half of P row h (64 B, swizzled) -- and, from group 0,
        // alpha_h -- go to rank 0 as st.async bytes counted on its PFULL
        // barrier: nobody waits for them here.
        const uint32_t pfull = ptx::mapa(BAR(PFULL + ps), 0);
        ptx::mbar_arrive_expect_tx_remote(pfull, grp == 0 ? 4u * 16u + 4u : 4u * 16u);
        const uint32_t prow = ptx::mapa(sbase + C::kOffP + static_cast<uint32_t>(ps) * kPSlotBytes + h * 128u, 0);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          ptx::st_async_v4(prow + (((4 * grp + j) ^ (h & 7)) << 4), pk[4 * j], pk[4 * j + 1], pk[4 * j + 2],
                           pk[4 * j + 3], pfull);
        if (grp == 0)
          ptx::st_async_b32(ptx::mapa(sbase + kOffAlpha + ps * 512u + h * 4u, 0), __float_as_uint(alpha), pfull);
        if (++sb == 2) { sb = 0; sphase ^= 1u; }
        if (++ps == kPSlots) { ps = 0; pphase ^= 1u; }
      }
      if (!ok) break;
      if (grp == 1) {
        // hand group 1's partial sum to group 0 (read before group 0 loads the
        // next segment's Q, so group 1 cannot overwrite it early)
        l_part[h] = l;
        ptx::mbar_arrive(BAR(LSUM));
      } else {
        if (!wait_warp<false>(BAR(LSUM), lsum_phase, hdr)) { ok = false; break; }
        l += l_part[h];
        const bool split = slot_base[sg.b] >= 0;
        const int slot = split ? group * spq + slot_base[sg.b] + (pl - first_pair[sg.b]) : -1;
        const float lse_v = l > 0.f ? (m_ref * c + log2f(l)) * kLn2 : -INFINITY;
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        if (split) part_lse[static_cast<size_t>(slot) * kHeads + h] = lse_v;
        else p.lse[static_cast<size_t>(row) * kHeads + h] = lse_v;
        if (!wait_warp<true>(BAR(MBEMPTY + ms), mphase ^ 1u, hdr)) { ok = false; break; }
        const uint32_t mbfull = ptx::mapa(BAR(MBFULL + ms), 0);
        ptx::mbar_arrive_expect_tx_remote(mbfull, 4u);
        ptx::st_async_b32(ptx::mapa(sbase + kOffMail + ms * 512u + h * 4u, 0), __float_as_uint(inv_l), mbfull);
        if (++ms == kMailSlots) { ms = 0; mphase ^= 1u; }
      }
      lsum_phase ^= 1u;
    }
    // the last remote arrivals from rank 0 must land before this CTA exits
    if (ok && grp == 0) {
      for (int s = 0; s < kPSlots && ok; ++s) {
        ok = wait_warp<true>(BAR(PEMPTY + ps), pphase ^ 1u, hdr);
        if (++ps == kPSlots) { ps = 0; pphase ^= 1u; }
      }
      for (int s = 0; s < kMailSlots && ok; ++s) {
        ok = wait_warp<true>(BAR(MBEMPTY + ms), mphase ^ 1u, hdr);
        if (++ms == kMailSlots) { ms = 0; mphase ^= 1u; }
      }
    }
  } else if (active && warp >= 4 && warp < 8 && rank == 0) {
    // ------------------------------------------------------------ rescale + epilogue
    const int h = threadIdx.x - 128;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    SegWalker w; w.init(tile_start, p.batch, lo, hi);
    Segment sg;
    uint32_t req_phase = 0, of_phase = 0;
    int ms = 0; uint32_t mphase = 0;
    bool ok = true;
    volatile uint32_t* req_slot = reinterpret_cast<volatile uint32_t*>(smem + kOffReq);
    const volatile float* alpha_buf = reinterpret_cast<const volatile float*>(smem + kOffAlpha);
    const volatile float* mail = reinterpret_cast<const volatile float*>(smem + kOffMail);
    while (ok && w.next(sg)) {
      const int row = sg.b * sq + group;
      // serve rescale requests until the segment's last P.V completes
      const uint64_t t0 = ptx::globaltimer();
      uint32_t spins = 0;
      while (true) {
        // Poll warp-uniformly; once a phase is seen complete it stays complete
        // until this warp answers, so every lane's own try_wait then succeeds
        // (and acquires).
        if (__any_sync(0xffffffffu, ptx::mbar_try_wait(BAR(REQ), req_phase))) {
          while (!ptx::mbar_try_wait(BAR(REQ), req_phase)) {}
          req_phase ^= 1u;
          ptx::tc_fence_after();
          const float a = alpha_buf[*req_slot * 128 + h];
          if (__any_sync(0xffffffffu, a != 1.f)) {
#pragma unroll 1
            for (int cc = 0; cc < 16; ++cc) {
              uint32_t r[32];
              ptx::tmem_ld32(tmem + lane_base + 32u * cc, r);
              ptx::tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * a);
              ptx::tmem_st32(tmem + lane_base + 32u * cc, r);
            }
            ptx::tmem_wait_st();
          }
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(BAR(CORR));
          continue;
        }
        if (__any_sync(0xffffffffu, ptx::mbar_try_wait(BAR(OFULL), of_phase))) {
          while (!ptx::mbar_try_wait(BAR(OFULL), of_phase)) {}
          of_phase ^= 1u;
          break;
        }
        if ((++spins & 255u) == 0) {
          bool give_up = read_status(&hdr->abort_flag) != 0;
          if (!give_up && ptx::globaltimer() - t0 > MLA_WAIT_TIMEOUT_NS) {
            set_status(&hdr->status, MLA_STATUS_TIMEOUT);
            atomicExch(&hdr->abort_flag, 1);
            give_up = true;
          }
          if (__any_sync(0xffffffffu, give_up)) { ok = false; break; }
        }
      }
      if (!ok) break;
      ptx::tc_fence_after();
      if (!wait_warp<true>(BAR(MBFULL + ms), mphase, hdr)) { ok = false; break; }
      const float inv_l = mail[ms * 128 + h];
      const bool split = slot_base[sg.b] >= 0;
      if (split) {
        const int slot = group * spq + slot_base[sg.b] + (pl - first_pair[sg.b]);
        float4* dst = reinterpret_cast<float4*>(part_out + (static_cast<size_t>(slot) * kHeads + h) * kDc);
#pragma unroll 1
        for (int cc = 0; cc < 16; ++cc) {
          uint32_t r[32];
          ptx::tmem_ld32(tmem + lane_base + 32u * cc, r);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[cc * 8 + v] = make_float4(__uint_as_float(r[4 * v]) * inv_l, __uint_as_float(r[4 * v + 1]) * inv_l,
                                          __uint_as_float(r[4 * v + 2]) * inv_l, __uint_as_float(r[4 * v + 3]) * inv_l);
        }
      } else {
        uint4* dst = reinterpret_cast<uint4*>(p.out + (static_cast<size_t>(row) * kHeads + h) * kDc);
#pragma unroll 1
        for (int cc = 0; cc < 16; ++cc) {
          uint32_t r[32];
          ptx::tmem_ld32(tmem + lane_base + 32u * cc, r);
          ptx::tmem_wait_ld();
          uint32_t o[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) o[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * inv_l, __uint_as_float(r[2 * e + 1]) * inv_l);
#pragma unroll
          for (int v = 0; v < 4; ++v) dst[cc * 4 + v] = make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(BAR(OEMPTY));
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_remote(ptx::mapa(BAR(MBEMPTY + ms), 1));
      if (++ms == kMailSlots) { ms = 0; mphase ^= 1u; }
    }
  }

  // ------------------------------------------------------------ teardown
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();
  if (warp == 2) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// Host-side launcher.  kMode 0: bf16 cache through the two 3-D tensor maps
// (whole-page boxes: nine chunks for rank 1, eight for rank 0); 1: FP8 cache
// (p.kv_fp8; tensor maps unused).
template <int kMode>
cudaError_t launch_decode_mode(const CUtensorMap& tmap_k, const CUtensorMap& tmap_v, const DecodeParams& p,
                               int n_pairs, cudaStream_t stream) {
  auto kern = mla_decode_pair_kernel<kMode>;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dk::smem_bytes<kMode>());
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * n_pairs, 1, 1);
  cfg.blockDim = dim3(dk::Cfg<kMode>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = dk::smem_bytes<kMode>();
  cfg.stream = stream;
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, kern, tmap_k, tmap_v, p);
}

cudaError_t launch_decode_bf16(const CUtensorMap& tmap_k, const CUtensorMap& tmap_v, const DecodeParams& p,
                               int n_pairs, cudaStream_t stream) {
  return launch_decode_mode<0>(tmap_k, tmap_v, p, n_pairs, stream);
}

cudaError_t launch_decode_fp8(const DecodeParams& p, int n_pairs, cudaStream_t stream) {
  CUtensorMap unused;
  memset(&unused, 0, sizeof(unused));
  return launch_decode_mode<1>(unused, unused, p, n_pairs, stream);
}

int decode_max_pairs() {
  // clusters of two CTAs that can be resident at once (one CTA per SM)
  static int cached_device = -1, cached = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cached_device == dev) return cached;
  auto kern = mla_decode_pair_kernel<0>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dk::smem_bytes<0>()) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(dk::Cfg<0>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = dk::smem_bytes<0>();
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2; attr[0].val.clusterDim.y = 1; attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    n = sms / 2;
  }
  cached_device = dev;
  cached = n;
  return n;
}

}  // namespace mla
