// Paired tcgen05 MLA decode kernel for sm_103a.
//
// What it computes ("DeepSeek R1 Architecture & Deployment Guide", section
// 1.1): for one query row (128 absorbed heads) over a row's paged latent
// cache, s = scale * Q[128 x 576] . K^T with K the gathered rows
// [c_KV | k_R]; P = online softmax(s); O[128 x 512] = P . V with V = c_KV
// (the first 512 columns of the same rows); out = O / l, lse = m + ln l.
//
// Why a CTA pair.  O for 128 heads x 512 latent columns in fp32 is exactly
// the 512 x 128-lane tensor memory of one SM, so S cannot live beside it.
// Each 2-CTA cluster therefore splits the work by role, not by data:
//   rank 1 ("score SM"):  Q [128 x 576] bf16 resident in TMEM (288 columns),
//       S = Q . K^T with A read from TMEM (kind::f16, M=128, N=64, K=576),
//       double-buffered S in TMEM, online softmax in 4 warps (thread = head
//       row, so row max / row sum need no cross-thread reduction), P rounded
//       to bf16 and sent with st.async straight into rank 0's shared memory
//       in the 128B-swizzled K-major layout the MMA reads (the bytes are
//       counted on rank 0's barrier, so no thread waits for the transfer);
//   rank 0 ("value SM"):  O [128 x 512] fp32 in all of its TMEM,
//       O += P . V with P from shared memory (K-major) and V read from the
//       page tile as an MN-major operand (two M=128, N=256, K=16 MMAs per
//       16 tokens), rescales O when rank 1 moves its reference max, and runs
//       the epilogue (O / l -> bf16 out, or fp32 split partial).
// Both ranks stream the same pages through a 3-stage TMA ring (one stage =
// one 64-token page: 8 chunks of 64 columns x 64 rows with 128B swizzle,
// plus the 64 RoPE columns on rank 1); the second read of a page is an L2
// hit.  No FLOP is computed twice: rank 1 does 2*128*576 and rank 0
// 2*128*512 FLOP per (query, token).
//
// Lazy rescaling: rank 1 keeps a per-head reference max m_ref (log2 units)
// and only moves it when a tile's max exceeds it by more than 8, so P <= 256
// in bf16 and O is rescaled (TMEM load/multiply/store by rank 0's epilogue
// warps) only on those rare tiles.
//
// Every wait is bounded (wait_bounded); a timeout sets the status word and an
// abort flag so all waits of the grid give up and the kernel exits cleanly.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstring>

#include "decode.cuh"

namespace mla {

namespace dk {

constexpr uint32_t kChunkBytes = 64 * 128;            // 64 rows x 64 bf16, 128B swizzle
constexpr uint32_t kStageBytes = 8 * kChunkBytes;     // latent c_KV part of one page
constexpr uint32_t kPSlotBytes = 128 * 128;           // P tile: 128 heads x 64 tokens bf16
constexpr int kPSlots = 2;
constexpr int kMailSlots = 2;
constexpr uint32_t kRawBytes = 32 * kFp8Row;          // half a page of FP8 rows: 19,008 B
constexpr int kMaxRaw = 4;

// Shared-memory plans.  The operand ring holds bf16 page tiles in the
// 128B-swizzled layout the MMAs read (latent chunks at stage*64K + c*8K);
// behind it rank 1 keeps the RoPE chunk of each stage and rank 0 its P slots.
// The FP8 plan adds a ring of raw half pages per rank.  Both ranks put the
// small shared region (alpha, 1/l, flags, barriers) at the same offset so
// remote stores and arrivals can address it by offset.
template <int kMode> struct Cfg;
template <> struct Cfg<0> {            // bf16 cache: 2-D TMA tiles
  static constexpr int kStages = 3;
  static constexpr int kRawStages1 = 0, kRawStages0 = 0;
  static constexpr uint32_t kOffAux = kStages * kStageBytes;
  static constexpr uint32_t kOffRaw1 = 0, kOffRaw0 = 0;
  static constexpr uint32_t kOffMisc = kOffAux + kPSlots * kPSlotBytes;
  static constexpr int kThreads = 256;
};
template <> struct Cfg<1> {            // FP8 cache: 1-D bulk copies + dequant warps 8..11
  static constexpr int kStages = 2;
  static constexpr int kRawStages1 = 4, kRawStages0 = 3;
  static constexpr uint32_t kOffAux = kStages * kStageBytes;
  static constexpr uint32_t kOffRaw1 = kOffAux + kStages * kChunkBytes;   // after the RoPE ring
  static constexpr uint32_t kOffRaw0 = kOffAux + kPSlots * kPSlotBytes;   // after the P ring
  static constexpr uint32_t kOffMisc = kOffRaw1 + kRawStages1 * kRawBytes;
  static constexpr int kThreads = 384;
};
constexpr uint32_t kMiscAlpha = 0;       // rank 0: fp32 alpha [2][128]
constexpr uint32_t kMiscMail = 1024;     // rank 0: fp32 1/l [2][128]
constexpr uint32_t kMiscReq = 2048;      // rank 0: P slot of a rescale request
constexpr uint32_t kMiscRawBad = 2064;   // per raw stage: 1 if its page id was out of range
constexpr uint32_t kMiscBar = 2080;
enum Bar {
  FULL = 0, EMPTY = FULL + 3,
  PFULL = EMPTY + 3, PEMPTY = PFULL + kPSlots,
  SFULL = PEMPTY + kPSlots, SEMPTY = SFULL + 2,
  QREADY = SEMPTY + 2, REQ, CORR, OFULL, OEMPTY,
  MBFULL, MBEMPTY = MBFULL + kMailSlots,
  RAWFULL = MBEMPTY + kMailSlots, RAWEMPTY = RAWFULL + kMaxRaw,
  NBAR = RAWEMPTY + kMaxRaw
};
constexpr uint32_t kMiscTmem = kMiscBar + NBAR * 8;
constexpr uint32_t kMiscBytes = kMiscTmem + 16;
template <int kMode> constexpr uint32_t smem_bytes() { return Cfg<kMode>::kOffMisc + kMiscBytes; }
static_assert(smem_bytes<0>() <= 232448 && smem_bytes<1>() <= 232448, "shared memory budget");
static_assert(Cfg<1>::kOffRaw0 + Cfg<1>::kRawStages0 * kRawBytes <= Cfg<1>::kOffMisc, "rank 0 raw ring");

// TMEM columns.
constexpr uint32_t kQCol = 0;      // rank 1: Q, 288 columns (2 bf16 per column)
constexpr uint32_t kSCol = 320;    // rank 1: two S buffers of 64 columns
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kIdescS = ptx::idesc_bf16(128, 64, 0, 0);    // A=Q (TMEM, K-major), B=K (K-major)
constexpr uint32_t kIdescPV = ptx::idesc_bf16(128, 256, 0, 1);  // A=P (K-major), B=V (MN-major)

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units: P <= 2^8

struct Segment {
  int b;          // batch row
  int t0, t1;     // row-local tile range [t0, t1)
  int n_row;      // tiles of the whole row
};

// Walks the segments of one pair: the pair's tile range [lo, hi) cut at
// row boundaries.  Every role of both ranks walks the same sequence.
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
        s.n_row = e - a;
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

}  // namespace dk

template <int kMode>   // 0: bf16 cache via TMA, 1: FP8 cache via bulk copies + dequant
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(dk::Cfg<kMode>::kThreads, 1)
mla_decode_pair_kernel(const __grid_constant__ CUtensorMap tmap, const DecodeParams p) {
  using namespace dk;
  using C = Cfg<kMode>;
  constexpr int kStages = C::kStages;
  constexpr uint32_t kOffAux = C::kOffAux;
  constexpr uint32_t kOffAlpha = C::kOffMisc + kMiscAlpha;
  constexpr uint32_t kOffMail = C::kOffMisc + kMiscMail;
  constexpr uint32_t kOffFlag = C::kOffMisc + kMiscReq;
  constexpr uint32_t kOffRawBad = C::kOffMisc + kMiscRawBad;
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
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(BAR(FULL + s), kMode == 0 ? 1 : 4);   // TMA bytes, or the 4 dequant warps
      ptx::mbar_init(BAR(EMPTY + s), 1);
    }
    for (int s = 0; s < kMaxRaw; ++s) { ptx::mbar_init(BAR(RAWFULL + s), 1); ptx::mbar_init(BAR(RAWEMPTY + s), 4); }
    for (int s = 0; s < kPSlots; ++s) { ptx::mbar_init(BAR(PFULL + s), 128); ptx::mbar_init(BAR(PEMPTY + s), 1); }
    for (int s = 0; s < 2; ++s) { ptx::mbar_init(BAR(SFULL + s), 1); ptx::mbar_init(BAR(SEMPTY + s), 128); }
    ptx::mbar_init(BAR(QREADY), 128);
    ptx::mbar_init(BAR(REQ), 2);
    ptx::mbar_init(BAR(CORR), 4);
    ptx::mbar_init(BAR(OFULL), 1);
    ptx::mbar_init(BAR(OEMPTY), 128);
    for (int s = 0; s < kMailSlots; ++s) { ptx::mbar_init(BAR(MBFULL + s), 128); ptx::mbar_init(BAR(MBEMPTY + s), 4); }
    ptx::fence_barrier_init();
  }
  if (warp == 2) {
    ptx::tmem_alloc(sbase + kOffTmemPtr, kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) ptx::prefetch_tmap(&tmap);
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
      const int n_raw = rank == 1 ? C::kRawStages1 : C::kRawStages0;
      const uint32_t raw_off = rank == 1 ? C::kOffRaw1 : C::kOffRaw0;
      volatile uint32_t* raw_bad = reinterpret_cast<volatile uint32_t*>(smem + kOffRawBad);
      bool ok = true;
      while (ok && w.next(sg)) {
        for (int t = sg.t0; t < sg.t1; ++t) {
          int page = __ldg(p.block_table + static_cast<size_t>(sg.b) * p.max_pages + t);
          const bool bad = page < 0 || page >= p.num_pages;
          if (bad) set_status(&hdr->status, MLA_STATUS_BAD_PAGE);
          if constexpr (kMode == 0) {
            if (bad) page = p.num_pages;   // fully outside the tensor: TMA fills zeros
            if (!wait_bounded<true>(BAR(EMPTY + stage), phase ^ 1u, hdr)) { ok = false; break; }
            const uint32_t bytes = (rank == 1 ? 9u : 8u) * kChunkBytes;
            ptx::mbar_arrive_expect_tx(BAR(FULL + stage), bytes);
            const int y = page * kPage;
            const uint32_t dst = sbase + static_cast<uint32_t>(stage) * kStageBytes;
#pragma unroll
            for (int c = 0; c < 8; ++c)
              ptx::tma_load_2d(dst + c * kChunkBytes, &tmap, BAR(FULL + stage), c * 64, y, pol);
            if (rank == 1)
              ptx::tma_load_2d(sbase + kOffAux + stage * kChunkBytes, &tmap, BAR(FULL + stage), 512, y, pol);
            if (++stage == kStages) { stage = 0; phase ^= 1u; }
          } else {
            // two half pages of raw FP8 rows; a bad page is never read (zeros)
            for (int half = 0; half < 2; ++half) {
              if (!wait_bounded<true>(BAR(RAWEMPTY + rs), rphase ^ 1u, hdr)) { ok = false; break; }
              raw_bad[rs] = bad ? 1u : 0u;
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
            if (!ok) break;
          }
        }
      }
    }
  } else if (kMode == 1 && active && warp >= 8) {
    // ------------------------------------------------------------ FP8 dequant (warps 8..11)
    // raw half page -> bf16 operand tile rows [32*half, 32*half+32).  Warp
    // wq handles tokens of parity (wq & 1) and half of the 32-value groups
    // (9 of 18 on rank 1, 8 of the 16 latent groups on rank 0).
    const int wq = warp - 8;
    const int parity = wq & 1;
    const int G = rank == 1 ? 9 : 8;
    const int g0 = (wq >> 1) * G;
    const int n_tasks = 16 * G;
    const int n_raw = rank == 1 ? C::kRawStages1 : C::kRawStages0;
    const uint32_t raw_off = rank == 1 ? C::kOffRaw1 : C::kOffRaw0;
    const volatile uint32_t* raw_bad = reinterpret_cast<const volatile uint32_t*>(smem + kOffRawBad);
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
          const bool bad = raw_bad[rs] != 0;
          const uint8_t* raw = smem + raw_off + static_cast<uint32_t>(rs) * kRawBytes;
          for (int task = lane; task < n_tasks; task += 32) {
            const int tok = 2 * (task / G) + parity;          // token within the half page
            const int g = g0 + task % G;                       // 32-value group
            const int tp = 32 * half + tok;                    // row within the page tile
            uint32_t o[16];
            if (!bad) {
              const uint8_t* src = raw + tok * kFp8Row + 32 * g;
              uint32_t wd[8];
              if (parity == 0) {
#pragma unroll
                for (int i = 0; i < 8; ++i) wd[i] = reinterpret_cast<const uint32_t*>(src)[i];
              } else {
                const uint32_t* a = reinterpret_cast<const uint32_t*>(src - 2);
                uint32_t u[9];
#pragma unroll
                for (int i = 0; i < 9; ++i) u[i] = a[i];
#pragma unroll
                for (int i = 0; i < 8; ++i) wd[i] = __funnelshift_r(u[i], u[i + 1], 16);
              }
              dequant32(wd, raw[tok * kFp8Row + kRow + g], o);
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i) o[i] = 0u;
            }
            const int c = g >> 1;
            uint8_t* dst = smem + (c < 8 ? static_cast<uint32_t>(stage) * kStageBytes + c * kChunkBytes
                                         : kOffAux + static_cast<uint32_t>(stage) * kChunkBytes) + tp * 128;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int piece = ((g & 1) * 4 + j) ^ (tp & 7);
              *reinterpret_cast<uint4*>(dst + piece * 16) = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
            }
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
          const uint32_t d = tmem + kSCol + 64u * sb;
          const uint32_t kbase = sbase + static_cast<uint32_t>(stage) * kStageBytes;
          const uint32_t rbase = sbase + kOffAux + static_cast<uint32_t>(stage) * kChunkBytes;
#pragma unroll 4
          for (int k = 0; k < kRow / 16; ++k) {
            const int c = k >> 2, kk = k & 3;
            const uint32_t baddr = (c < 8 ? kbase + c * kChunkBytes : rbase) + kk * 32;
            const uint64_t bdesc = ptx::sdesc_sw128(baddr, 16, 1024);
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
    volatile uint32_t* req_slot = reinterpret_cast<volatile uint32_t*>(smem + kOffFlag);
    const volatile float* alpha_buf = reinterpret_cast<const volatile float*>(smem + kOffAlpha);
    while (ok && w.next(sg)) {
      const int len_i = lens[sg.b] - (sq - 1 - group);
      for (int t = sg.t0; t < sg.t1 && ok; ++t) {
        if (!wait_warp<false>(BAR(FULL + stage), phase, hdr) ||
            !wait_warp<true>(BAR(PFULL + ps), pphase, hdr)) { ok = false; break; }
        ptx::fence_proxy_async_cta();
        // did rank 1 move its reference max for any head of this tile?
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
        const int valid = len_i - t * kPage;   // rows of this page visible to the query
        if (valid < kPage) {
          // rows past the visible length get P = 0; make their V finite too
          const int v0 = valid > 0 ? valid : 0;
          uint4* base = reinterpret_cast<uint4*>(smem + static_cast<uint32_t>(stage) * kStageBytes);
          const int n16 = (kPage - v0) * 8;     // 16-byte pieces per chunk
          for (int c = 0; c < 8; ++c)
            for (int i = lane; i < n16; i += 32)
              base[(c * kChunkBytes + v0 * 128) / 16 + i] = make_uint4(0, 0, 0, 0);
          ptx::fence_proxy_async_cta();
          __syncwarp();
        }
        ptx::tc_fence_after();
        if (lane == 0) {
          const uint32_t pbase = sbase + kOffAux + static_cast<uint32_t>(ps) * kPSlotBytes;
          const uint32_t vbase = sbase + static_cast<uint32_t>(stage) * kStageBytes;
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
  } else if (active && warp >= 4 && rank == 1) {
    // ------------------------------------------------------------ softmax (thread = head)
    const int h = threadIdx.x - 128;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    SegWalker w; w.init(tile_start, p.batch, lo, hi);
    Segment sg;
    int sb = 0; uint32_t sphase = 0;
    int ps = 0; uint32_t pphase = 0;
    int ms = 0; uint32_t mphase = 0;
    bool ok = true;
    const float c = p.scale_log2;
    while (ok && w.next(sg)) {
      const int row = sg.b * sq + group;
      const int len_i = lens[sg.b] - (sq - 1 - group);
      // Q row h -> TMEM lane h, columns [0, 288): two bf16 per column, K order.
      {
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
        uint32_t r[64];
        ptx::tmem_ld32(tmem + lane_base + kSCol + 64u * sb, r);
        ptx::tmem_ld32(tmem + lane_base + kSCol + 64u * sb + 32u, r + 32);
        ptx::tmem_wait_ld();
        ptx::tc_fence_before();
        ptx::mbar_arrive(BAR(SEMPTY + sb));
        const int valid = len_i - t * kPage;
        float mx = -INFINITY;
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          const float x = e < valid ? __uint_as_float(r[e]) * c : -INFINITY;
          r[e] = __float_as_uint(x);
          mx = fmaxf(mx, x);
        }
        float alpha = 1.f;
        if (t == sg.t0) {
          m_ref = mx;
        } else if (mx > m_ref + kRescaleThreshold) {
          alpha = exp2f(m_ref - mx);
          l *= alpha;
          m_ref = mx;
        }
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float x0 = __uint_as_float(r[2 * e]), x1 = __uint_as_float(r[2 * e + 1]);
          const float p0 = x0 == -INFINITY ? 0.f : exp2f(x0 - m_ref);
          const float p1 = x1 == -INFINITY ? 0.f : exp2f(x1 - m_ref);
          pk[e] = pack_bf16x2(p0, p1);
          l += p0 + p1;
        }
        if (!wait_warp<true>(BAR(PEMPTY + ps), pphase ^ 1u, hdr)) { ok = false; break; }
        // P row h (128 B, swizzled) and alpha_h go to rank 0 as st.async
        // bytes counted on its PFULL barrier: nobody waits for them here.
        const uint32_t pfull = ptx::mapa(BAR(PFULL + ps), 0);
        ptx::mbar_arrive_expect_tx_remote(pfull, 8u * 16u + 4u);
        const uint32_t prow = ptx::mapa(sbase + kOffAux + static_cast<uint32_t>(ps) * kPSlotBytes + h * 128u, 0);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          ptx::st_async_v4(prow + ((j ^ (h & 7)) << 4), pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3],
                           pfull);
        ptx::st_async_b32(ptx::mapa(sbase + kOffAlpha + ps * 512u + h * 4u, 0), __float_as_uint(alpha), pfull);
        if (++sb == 2) { sb = 0; sphase ^= 1u; }
        if (++ps == kPSlots) { ps = 0; pphase ^= 1u; }
      }
      if (!ok) break;
      const bool split = slot_base[sg.b] >= 0;
      const int slot = split ? group * spq + slot_base[sg.b] + (pl - first_pair[sg.b]) : -1;
      const float lse_v = l > 0.f ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      if (split) part_lse[static_cast<size_t>(slot) * kHeads + h] = lse_v;
      else p.lse[static_cast<size_t>(row) * kHeads + h] = lse_v;
      if (!wait_warp<true>(BAR(MBEMPTY + ms), mphase ^ 1u, hdr)) { ok = false; break; }
      const uint32_t mbfull = ptx::mapa(BAR(MBFULL + ms), 0);
      ptx::mbar_arrive_expect_tx_remote(mbfull, 4u);
      ptx::st_async_b32(ptx::mapa(sbase + kOffMail + ms * 512u + h * 4u, 0), __float_as_uint(inv_l), mbfull);
      if (++ms == kMailSlots) { ms = 0; mphase ^= 1u; }
    }
    // the last remote arrivals from rank 0 must land before this CTA exits
    if (ok) {
      for (int s = 0; s < kPSlots && ok; ++s) {
        ok = wait_warp<true>(BAR(PEMPTY + ps), pphase ^ 1u, hdr);
        if (++ps == kPSlots) { ps = 0; pphase ^= 1u; }
      }
      for (int s = 0; s < kMailSlots && ok; ++s) {
        ok = wait_warp<true>(BAR(MBEMPTY + ms), mphase ^ 1u, hdr);
        if (++ms == kMailSlots) { ms = 0; mphase ^= 1u; }
      }
    }
  } else if (active && warp >= 4 && rank == 0) {
    // ------------------------------------------------------------ rescale + epilogue
    const int h = threadIdx.x - 128;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    SegWalker w; w.init(tile_start, p.batch, lo, hi);
    Segment sg;
    uint32_t req_phase = 0, of_phase = 0;
    int ms = 0; uint32_t mphase = 0;
    bool ok = true;
    volatile uint32_t* req_slot = reinterpret_cast<volatile uint32_t*>(smem + kOffFlag);
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
          for (int e = 0; e < 16; ++e) {
            __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(r[2 * e]) * inv_l,
                                                     __uint_as_float(r[2 * e + 1]) * inv_l);
            o[e] = *reinterpret_cast<uint32_t*>(&v);
          }
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

// Host-side launcher.  kMode 0: bf16 cache through `tmap`; 1: FP8 cache
// (p.kv_fp8; `tmap` unused).
template <int kMode>
cudaError_t launch_decode_mode(const CUtensorMap& tmap, const DecodeParams& p, int n_pairs, cudaStream_t stream) {
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
  return cudaLaunchKernelEx(&cfg, kern, tmap, p);
}

cudaError_t launch_decode_bf16(const CUtensorMap& tmap, const DecodeParams& p, int n_pairs, cudaStream_t stream) {
  return launch_decode_mode<0>(tmap, p, n_pairs, stream);
}

cudaError_t launch_decode_fp8(const DecodeParams& p, int n_pairs, cudaStream_t stream) {
  CUtensorMap unused;
  memset(&unused, 0, sizeof(unused));
  return launch_decode_mode<1>(unused, p, n_pairs, stream);
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
  cfg.blockDim = dim3(256, 1, 1);
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
