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
//       per tile of N tokens S = Q . K^T (36 tcgen05.mma, M=128, A from TMEM)
//       into one of two N-column S buffers (three for the quantised caches);
//       eight softmax warps in two groups
//       (each turns half of the tile's columns into P, both take the row max
//       over all N columns, so their reference maxima agree without an
//       exchange) round P to bf16 and send it with st.async into rank 0's
//       shared memory in the 128B-swizzled K-major layout its MMA reads; the
//       bytes are counted on rank 0's barrier, so no thread waits for them.
//   rank 0 ("value SM"): O [128 x 512] fp32 in all 512 TMEM columns;
//       O += P . V with P from shared memory and V read as an MN-major operand
//       (two M=128, N=256, K=16 MMAs per 16 tokens); its epilogue warps
//       rescale O when rank 1 moves a head's reference max and write
//       out = O / l (or, for a row split over several pairs, the bf16
//       partial that the merge kernel combines).
//
// Tiles of 96 tokens.  A tcgen05.mma with N <= 96 costs about as much as one
// with N = 64, so the score SM works on 96-token tiles (three half pages).
// The cache is described to TMA as a 4-D tensor (64 columns, 8 rows, 9
// column chunks, 8-row groups) with strides 1152 B (row), 128 B (chunk) and
// 9216 B (row group); a box of 4 row groups is a half page and lands as
// 8-row x 128-byte swizzle atoms ordered (row group, chunk, row).  A score
// SM tile buffer holds two blocks: chunks 0..4 (A part) and chunks 5..8 (B
// part) of its three half pages.  In each block consecutive slots continue
// each other's row-group sequence at a constant stride (5 KiB, 4 KiB), so a
// block is one 96-row K-major operand, whatever pages the slots came from.
// S consumes the A part first and releases it, so the next tile's A part
// loads while S reads the B part.  Each SM's TMA loads land only in its own
// shared memory.  Each TMA operation costs the issuing SM about 225 ns, so
// the score SM loads two adjacent slots that hold the halves of one page with
// one whole-page box (two operations per part and tile instead of three).
// The value SM keeps half-page V slots (atoms at 1 KiB per chunk, 8 KiB per
// row group), read as MN-major operands 16 tokens at a time.  Both ranks
// read every half page; the second read is an L2 hit.
//
// The FP8 cache is bulk-copied as raw half pages by both SMs, and each SM
// dequantises what its own MMAs read (score SM: all nine chunks into the
// nine-chunk K layout; value SM: the eight latent chunks into V slots), in
// 64-token tiles (the raw buffers take the shared memory of a third slot).
// The FP4 cache and the V4.1 rows (528-byte FP8, 288-byte FP4) use the same
// roles, layouts and tiles with their own raw copies and decoders.
// Moving dequantised rows between the two SMs would cost more than the
// second dequant: traffic inside a cluster runs at about 42 GB/s per pair.
//
// Sparse top-k decode (mode 3) is the bf16 kernel with the copies done by
// three warps per SM that gather listed cache rows with 16-byte cp.async
// into the same layouts (TMA cannot gather 1152-byte rows into the swizzled
// operand layout at a useful rate).
//
// Lazy rescaling: rank 1 keeps a per-head reference max m_ref (raw score
// units) and moves it only when a tile's max exceeds it by more than 16 in
// log2 units, so P <= 2^16 and O is rescaled only on those tiles; the
// epilogue warps on rank 0 (eight for bf16, four for FP8) do the rescale.
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

constexpr uint32_t kAtom = 1024;                        // 8 rows x 128 B, 128B swizzle
constexpr uint32_t kKSlot = 4 * 9 * kAtom;             // half page, nine chunks (36 KiB)
constexpr uint32_t kKGroup = 9 * kAtom;                // row-group stride of a K slot
constexpr uint32_t kKA = 4 * 5 * kAtom;                // bf16 score SM: half page, chunks 0..4 (20 KiB)
constexpr uint32_t kKB = 4 * 4 * kAtom;                // bf16 score SM: half page, chunks 5..8 (16 KiB)
constexpr uint32_t kVSlot = 4 * 8 * kAtom;             // half page, eight latent chunks (32 KiB)
constexpr uint32_t kVGroup = 8 * kAtom;                // row-group stride of a V slot
constexpr uint32_t kPChunk = 128 * 128;                // 64 tokens of P for 128 heads (16 KiB)
constexpr int kMaxPSlots = 3;  // P slots on the value SM (per mode: Cfg::kPSlots)
constexpr int kMaxSBufs = 3;   // S buffers in TMEM (per mode: Cfg::kSBufs)
constexpr int kMailSlots = 2;
constexpr int kHalf = kPage / 2;                        // tokens per half page
constexpr uint32_t kRawBytes = kHalf * kFp8Row;         // raw FP8 half page: 19,008 B
constexpr int kMaxVSlots = 5, kMaxRaw = 4;

// Shared-memory plans (bytes).  The small common region (alpha, 1/l, flags,
// barriers) sits at the same offset in both ranks so remote stores and
// arrivals can address it.
//   bf16: rank 1 = 6 K slots (two 3-slot tiles); rank 0 = 5 V slots + 2 P
//         slots of two chunks (96 tokens).
//   FP8:  each SM bulk-loads every raw half page (the second read is an L2
//         hit) and dequantises what its own MMAs read: rank 1 = 4 K slots
//         (two 2-slot tiles) + 4 raw half pages; rank 0 = 4 V slots + 3
//         one-chunk P slots + 2 raw half pages.  Moving dequantised rows
//         between the two SMs instead would cost more: shared-to-shared
//         traffic inside a cluster runs at about 42 GB/s per pair on GB300.
template <int kMode> struct Cfg;
template <> struct Cfg<0> {
  static constexpr int kTileHalves = 3;
  static constexpr int kSBufs = 2;             // 2 x 96 columns of S beside Q's 288 + 32 spare
  static constexpr int kVSlots = 5;
  static constexpr int kPSlots = 2;
  static constexpr uint32_t kPSlotBytes = 2 * kPChunk;
  static constexpr uint32_t kOffP = kVSlots * kVSlot;
  static constexpr int kRaw0 = 0, kRaw1 = 0;
  static constexpr uint32_t kOffRaw0 = 0, kOffRaw1 = 0;
  static constexpr uint32_t kEnd1 = 2 * kTileHalves * kKSlot;
  static constexpr uint32_t kEnd0 = kOffP + kPSlots * kPSlotBytes;
  static constexpr uint32_t kOffMisc = kEnd1 > kEnd0 ? kEnd1 : kEnd0;
  static constexpr int kThreads = 384;
  static constexpr int kSmGroups = 2;          // softmax warp groups (4 warps each)
  static constexpr int kDqWarps1 = 0, kDqWarps0 = 0;
  static constexpr int kEpWarps = 8;           // epilogue warps on rank 0 (256 columns each)
};
// FP8 modes: 1 = exact bf16 operands; 2 = f16 operands (same layout)
template <> struct Cfg<1> {
  static constexpr int kTileHalves = 2;
  static constexpr int kSBufs = 3;             // 3 x 64 columns: S runs a tile further ahead of the softmax
  static constexpr int kVSlots = 4;
  static constexpr int kPSlots = 3;            // and P a tile further ahead of P.V
  static constexpr uint32_t kPSlotBytes = kPChunk;
  static constexpr uint32_t kOffP = kVSlots * kVSlot;                       // rank 0
  static constexpr int kRaw0 = 2, kRaw1 = 4;
  static constexpr uint32_t kOffRaw0 = kOffP + kPSlots * kPSlotBytes;       // rank 0
  static constexpr uint32_t kOffRaw1 = 2 * kTileHalves * kKSlot;            // rank 1: after the K slots
  static constexpr uint32_t kEnd1 = kOffRaw1 + kRaw1 * kRawBytes;
  static constexpr uint32_t kEnd0 = kOffRaw0 + kRaw0 * kRawBytes;
  static constexpr uint32_t kOffMisc = ((kEnd1 > kEnd0 ? kEnd1 : kEnd0) + 1023) & ~1023u;
  static constexpr int kThreads = 512;
  static constexpr int kSmGroups = 1;          // 64-token tiles: one group of 4 warps takes all columns
  static constexpr int kDqWarps1 = 9;          // rank 1: warps 8..15 and 2, one value-group pair of 18 each
  static constexpr int kDqWarps0 = 8;          // rank 0: warps 8..15, one latent value-group pair of 16 each
  static constexpr int kEpWarps = 4;           // rank 0: four epilogue warps (512 columns each)
};
template <> struct Cfg<2> : Cfg<1> {};
// FP4 cache: the FP8 roles and layout, smaller raw copies; 4 = bf16
// operands (exact), 5 = f16 operands
template <> struct Cfg<4> : Cfg<1> {};
template <> struct Cfg<5> : Cfg<1> {};
// FP8 V4.1 cache (528-byte rows): the FP8 roles and layout; 6 = bf16
// operands (exact), 7 = f16 operands
template <> struct Cfg<6> : Cfg<1> {};
template <> struct Cfg<7> : Cfg<1> {};
// FP4 V4.1 cache (288-byte rows): 8 = bf16 operands (exact), 9 = f16 operands
template <> struct Cfg<8> : Cfg<1> {};
template <> struct Cfg<9> : Cfg<1> {};
// sparse decode over the bf16 cache: the bf16 plan, K and V gathered by rows
template <> struct Cfg<3> : Cfg<0> {};
constexpr int kGatherWarps = 3;          // sparse: warps 0, 2, 3 of each rank copy one half page of a tile each
constexpr uint32_t kMiscAlpha = 0;       // rank 0: fp32 alpha [kMaxPSlots][128]
constexpr uint32_t kMiscLPart = 0;       // rank 1 (same bytes): group-1 partial softmax sums [128]
constexpr uint32_t kMiscMail = 512 * kMaxPSlots;   // rank 0: fp32 1/l [2][128]
constexpr uint32_t kMiscReq = kMiscMail + 1024;    // rank 0: P slot of a rescale request
constexpr uint32_t kMiscRawFlag = kMiscReq + 16;   // per raw stage: 1 = write zeros (bad page)
constexpr uint32_t kMiscBar = kMiscRawFlag + 4 * kMaxRaw;
enum Bar {
  KFULL = 0, KEMPTY = KFULL + 2,
  KFULLB = KEMPTY + 2, KEMPTYB = KFULLB + 2,   // bf16 score SM: the chunk 5..8 part of a tile
  VFULL = KEMPTYB + 2, VEMPTY = VFULL + kMaxVSlots,
  PFULL = VEMPTY + kMaxVSlots, PEMPTY = PFULL + kMaxPSlots,
  SFULL = PEMPTY + kMaxPSlots, SEMPTY = SFULL + kMaxSBufs,
  QREADY = SEMPTY + kMaxSBufs, REQ, CORR, OFULL, OEMPTY, LSUM,
  MBFULL, MBEMPTY = MBFULL + kMailSlots,
  RAWFULL = MBEMPTY + kMailSlots, RAWEMPTY = RAWFULL + kMaxRaw,
  DRAIN = RAWEMPTY + kMaxRaw,   // the MMA issuer's last commit, waited for at teardown
  NBAR
};
constexpr uint32_t kMiscTmem = kMiscBar + NBAR * 8;
constexpr uint32_t kMiscBytes = kMiscTmem + 16;
template <int kMode> constexpr uint32_t smem_bytes() { return Cfg<kMode>::kOffMisc + kMiscBytes; }
static_assert(smem_bytes<0>() <= 232448 && smem_bytes<1>() <= 232448, "shared memory budget");
static_assert(Cfg<0>::kVSlots <= kMaxVSlots && Cfg<1>::kVSlots <= kMaxVSlots, "V slot barriers");
static_assert(Cfg<1>::kRaw1 <= kMaxRaw && Cfg<1>::kRaw0 <= kMaxRaw, "raw barriers");
static_assert(Cfg<1>::kOffMisc % 1024 == 0 && Cfg<1>::kOffRaw0 % 16 == 0 && Cfg<1>::kOffRaw1 % 16 == 0,
              "slot alignment");
static_assert(Cfg<0>::kOffMisc % 1024 == 0, "slot alignment");

// TMEM columns.
constexpr uint32_t kQCol = 0;      // rank 1: Q, 288 columns (2 bf16 per column)
constexpr uint32_t kSCol = 320;    // rank 1: Cfg::kSBufs S buffers of N columns (up to column 512)
constexpr uint32_t kTmemCols = 512;

// Modes: 0 bf16 cache (TMA), 3 sparse over the bf16 cache; quantised caches
// (raw rings + dequant warps), exact bf16 operands / f16 operands: FP8
// 594-byte row 1 / 2, FP4 324-byte row 4 / 5, FP8 528-byte V4.1 row 6 / 7,
// FP4 288-byte V4.1 row 8 / 9.
template <int kMode> constexpr bool kModeF16 = kMode == 2 || kMode == 5 || kMode == 7 || kMode == 9;
template <int kMode> constexpr bool kModeQuant = kMode == 1 || kMode == 2 || (kMode >= 4 && kMode <= 9);
template <int kMode> constexpr bool kModeFp4 = kMode == 4 || kMode == 5 || kMode == 8 || kMode == 9;
template <int kMode> constexpr bool kModeV41 = kMode >= 6 && kMode <= 9;

// P.V: A = P (K-major), B = V (MN-major); bf16, or f16 in the f16 modes
template <int kMode>
constexpr uint32_t kIdescPV = kModeF16<kMode> ? ptx::idesc_f16(128, 256, 0, 1) : ptx::idesc_bf16(128, 256, 0, 1);

constexpr float kLn2 = 0.69314718055994530942f;
// log2 units: P <= 2^16 (exact in relative terms; O stays far from fp32
// overflow).  The FP8 f16 mode keeps P <= 2^15, inside the f16 range.
template <int kMode>
constexpr float kRescaleThreshold = kModeF16<kMode> ? 15.0f : 16.0f;

// FP8 f16 mode: a scale exponent e in [113, 134] makes every e4m3 code times
// 2^(e-127) an exact f16 number (largest 448 * 2^7 = 57344 < 65504; smallest
// step 2^-9 * 2^-14 = 2^-23, above the f16 subnormal step 2^-24), and keeps
// the f16 scale itself normal.
constexpr uint32_t kF16ScaleLo = 113, kF16ScaleHi = 134;
constexpr float kF16Max = 65504.0f;

struct Segment {
  int b;          // batch row
  int t0, t1;     // row-local page range [t0, t1)
};

// Walks the segments of one pair: the pair's page range [lo, hi) cut at row
// boundaries.  Every role of both ranks walks the same sequence; inside a
// segment the half pages [2*t0, 2*t1) are taken kTileHalves at a time.
struct SegWalker {
  const int* tile_start;
  int batch, b, lo, hi;
  // b0: the row holding page lo (the planner's pair_b0)
  __device__ void init(const int* ts, int nb, int lo_, int hi_, int b0) {
    tile_start = ts; batch = nb; lo = lo_; hi = hi_;
    b = lo >= hi ? nb : b0;
  }
  __device__ bool next(Segment& s) {
    while (b < batch) {
      const int a = __ldg(tile_start + b), e = __ldg(tile_start + b + 1);
      if (a >= hi) { b = batch; return false; }
      const int cb = b++;
      if (e >= hi) b = batch;   // this segment reaches the end of the range: no read for the next call
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

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (x0, x1) <- ((x0 - m) * c, (x1 - m) * c) with packed fp32x2 arithmetic.
// The subtraction comes first, so x == m gives exactly 0 however large the
// magnitudes are.
__device__ __forceinline__ void sub_scale2(float& x0, float& x1, float neg_m, float c) {
  const float2 v = __fmul2_rn(__fadd2_rn(make_float2(x0, x1), make_float2(neg_m, neg_m)), make_float2(c, c));
  x0 = v.x;
  x1 = v.y;
}

// (a0, a1) += (b0, b1), packed.
__device__ __forceinline__ void add2(float& a0, float& a1, float b0, float b1) {
  const float2 v = __fadd2_rn(make_float2(a0, a1), make_float2(b0, b1));
  a0 = v.x;
  a1 = v.y;
}

// 32 e4m3 codes (8 words, lowest byte first) with their e8m0 scale byte ->
// 16 bf16x2 words.  e4m3 -> f16 is exact in hardware and the product with
// the power-of-two scale is exact in fp32 (no flush).  The product has at
// most 4 significant bits, and for scale exponents e >= 3 its smallest bit is
// at least 2^-133, the last bit of a bf16 subnormal, so the bf16 value is the
// fp32 value's upper 16 bits: a byte permute, not a rounding conversion.
// Below that (results under 2^-133) the rounding conversion is used.  NaN
// codes and the NaN scale (0xFF) give NaN, as in the format definitions.
__device__ __forceinline__ void dequant32(const uint32_t* wd, uint32_t e, uint32_t* o) {
  const float sc = __uint_as_float(e == 0 ? 0x00400000u : (e == 255 ? 0x7FC00000u : (e << 23)));
  const bool trunc_exact = e >= 3;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t h01, h23;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h01) : "h"(static_cast<unsigned short>(wd[i] & 0xFFFFu)));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h23) : "h"(static_cast<unsigned short>(wd[i] >> 16)));
    const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
    const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
    const float a = f01.x * sc, b = f01.y * sc, c = f23.x * sc, d = f23.y * sc;
    if (trunc_exact) {
      o[2 * i] = __byte_perm(__float_as_uint(a), __float_as_uint(b), 0x7632);
      o[2 * i + 1] = __byte_perm(__float_as_uint(c), __float_as_uint(d), 0x7632);
    } else {
      o[2 * i] = pack_bf16x2(a, b);
      o[2 * i + 1] = pack_bf16x2(c, d);
    }
  }
}

// FP8 f16 mode: 32 e4m3 codes with their e8m0 scale byte -> 16 f16x2 words,
// each the exact hardware e4m3 -> f16 conversion times the f16 scale 2^(e-127)
// (a packed f16 multiply, exact for e in [kF16ScaleLo, kF16ScaleHi], where no
// product leaves the f16 range).  Returns false (and writes nothing useful)
// for a scale outside that range.
__device__ __forceinline__ bool dequant32_f16(const uint32_t* wd, uint32_t e, uint32_t* o) {
  const bool in_range = e >= kF16ScaleLo && e <= kF16ScaleHi;
  const uint32_t sh = ((e - 112u) & 31u) << 10;
  const uint32_t sc = sh | (sh << 16);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t h01, h23;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h01) : "h"(static_cast<unsigned short>(wd[i] & 0xFFFFu)));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h23) : "h"(static_cast<unsigned short>(wd[i] >> 16)));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[2 * i]) : "r"(h01), "r"(sc));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[2 * i + 1]) : "r"(h23), "r"(sc));
  }
  return in_range;
}

// Dequantise value group g (32 values) of raw FP8 row `row` (2-byte aligned
// in shared memory) into 16 bf16x2 words.  The 32 codes are read as nine
// aligned words and funnel-shifted by the row's misalignment (0 or 2 bytes).
// The group's e8m0 scale is byte kScales + g (576 for the 594-byte row, 512
// for the 528-byte V4.1 row).
template <bool kF16 = false, int kScales = kRow>
__device__ __forceinline__ bool dequant_group(const uint8_t* row, int g, uint32_t* o) {
  const uint8_t* src = row + 32 * g;
  uint32_t wd[8];
  if constexpr (kScales == kV41Values) {
    // 528-byte rows start on 16-byte boundaries: two 16-byte loads
    const uint4 lo = *reinterpret_cast<const uint4*>(src), hi = *reinterpret_cast<const uint4*>(src + 16);
    wd[0] = lo.x; wd[1] = lo.y; wd[2] = lo.z; wd[3] = lo.w;
    wd[4] = hi.x; wd[5] = hi.y; wd[6] = hi.z; wd[7] = hi.w;
  } else {
    const uintptr_t a = reinterpret_cast<uintptr_t>(src);
    const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~static_cast<uintptr_t>(3));
    const uint32_t sh = static_cast<uint32_t>(a & 3u) * 8u;
    uint32_t u[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) u[i] = w[i];
#pragma unroll
    for (int i = 0; i < 8; ++i) wd[i] = __funnelshift_r(u[i], u[i + 1], sh);
  }
  if constexpr (kF16) {
    return dequant32_f16(wd, row[kScales + g], o);
  } else {
    dequant32(wd, row[kScales + g], o);
    return true;
  }
}

// FP4 row: value group g (32 values) -> 16 bf16x2 words.  Codes are two
// e2m1 per byte, value 2k in the low nibble of byte k, so the group is the
// 16 bytes at 16g (word-aligned: rows are 324 bytes); its two e8m0 scales
// (values 32g..32g+15, then the next 16) are bytes kFp4Codes + 2g and + 1.
// e2m1 -> f16 is exact in hardware (the low nibble becomes the low half),
// the product with the power-of-two scale is exact in fp32, and with at most
// two significant bits and a smallest bit of at least 2^-128 (> 2^-133, the
// last bit of a bf16 subnormal) the bf16 value is the fp32 value's upper 16
// bits.  Scale bytes up to 252 keep every product finite; 0xFF gives NaN.
__device__ __forceinline__ float e8m0_f32(uint32_t e) {
  return __uint_as_float(e == 0 ? 0x00400000u : (e == 255 ? 0x7FC00000u : (e << 23)));
}

// kScales: the first scale byte (288 for the 324-byte row, 256 for the
// 288-byte V4.1 row).
template <int kScales = kFp4Codes>
__device__ __forceinline__ void dequant_group_fp4(const uint8_t* row, int g, uint32_t* o) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(row + 16 * g);
  const uint32_t sc = *reinterpret_cast<const uint16_t*>(row + kScales + 2 * g);
  const float s0 = e8m0_f32(sc & 0xFFu), s1 = e8m0_f32(sc >> 8);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t c = w[i];
    const float s = i < 2 ? s0 : s1;
    uint32_t h[4];
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3]) : "r"(c));
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[k]));
      o[4 * i + k] = __byte_perm(__float_as_uint(f.x * s), __float_as_uint(f.y * s), 0x7632);
    }
  }
}

// FP4 f16 mode: the same group as 16 f16x2 words, each the exact hardware
// e2m1 -> f16 conversion times the f16 scale 2^(e-127) (a packed f16
// multiply).  Exact for both scale bytes in [kFp4F16ScaleLo, kFp4F16ScaleHi]:
// the largest product 6 * 2^13 = 49152 fits f16, every product is a
// multiple of 2^-15, above the f16 subnormal step, and the scale itself is a
// normal f16 number.  Returns false for a scale outside that range.
constexpr uint32_t kFp4F16ScaleLo = 113, kFp4F16ScaleHi = 140;

template <int kScales = kFp4Codes>
__device__ __forceinline__ bool dequant_group_fp4_f16(const uint8_t* row, int g, uint32_t* o) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(row + 16 * g);
  const uint32_t sc = *reinterpret_cast<const uint16_t*>(row + kScales + 2 * g);
  const uint32_t e0 = sc & 0xFFu, e1 = sc >> 8;
  const bool in_range = e0 >= kFp4F16ScaleLo && e0 <= kFp4F16ScaleHi && e1 >= kFp4F16ScaleLo && e1 <= kFp4F16ScaleHi;
  const uint32_t f0 = ((e0 - 112u) & 31u) << 10, f1 = ((e1 - 112u) & 31u) << 10;
  const uint32_t s0 = f0 | (f0 << 16), s1 = f1 | (f1 << 16);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t c = w[i];
    const uint32_t s = i < 2 ? s0 : s1;
    uint32_t h[4];
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3]) : "r"(c));
#pragma unroll
    for (int k = 0; k < 4; ++k) asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[4 * i + k]) : "r"(h[k]), "r"(s));
  }
  return in_range;
}

// Store 16 bf16x2 words (32 values of value group g) as token r of a
// half-page slot whose 8-row atoms are `group_stride` bytes apart per row
// group (chunk c = g/2 at c KiB inside the group, 128-byte rows, 128B
// swizzle: 16-byte piece j of row r sits at piece j ^ (r % 8)).
__device__ __forceinline__ void store_group(uint8_t* slot, uint32_t group_stride, int r, int g, const uint32_t* o) {
  uint8_t* dst = slot + (r >> 3) * group_stride + (g >> 1) * kAtom + (r & 7) * 128;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int piece = ((g & 1) * 4 + j) ^ (r & 7);
    *reinterpret_cast<uint4*>(dst + piece * 16) = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
  }
}

// Load 32-column chunks [C0, C1) of one head's query row (chunk c < 8: the
// absorbed query at byte 128c, chunk 8: the RoPE query) with 32-byte loads
// and store them into the TMEM lane row at column 32c (two bf16 per column).
// Two chunks per round trip.
// bf16x2 word -> f16x2 word (round to nearest); qmax tracks the largest
// magnitude seen, so that values past the f16 range can be detected.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w, float& qmax) {
  const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xFFFF0000u);
  qmax = max3(qmax, fabsf(lo), fabsf(hi));
  return pack_f16x2(lo, hi);
}

// With kF16 (FP8 f16 mode) the query is stored as f16, and qmax returns its
// largest magnitude.
// kZero >= 0: that chunk is stored as zeros instead (the V4.1 row's latent
// dims 448..511, which meet zero keys; a non-finite query value there would
// otherwise turn its zero products into NaN).
template <int C0, int C1, bool kF16 = false, int kZero = -1>
__device__ __forceinline__ void load_q_chunks(const uint8_t* qa, const uint8_t* qr, uint32_t taddr, float& qmax) {
  if constexpr (kF16) {
    // one chunk per round trip: the conversion needs the registers
#pragma unroll 1
    for (int c = C0; c < C1; ++c) {
      uint32_t r0[32];
      if (c == kZero) {
#pragma unroll
        for (int i = 0; i < 32; ++i) r0[i] = 0u;
      } else {
#pragma unroll
        for (int v = 0; v < 4; ++v) ptx::ld_global_nc_v8((c < 8 ? qa + c * 128 : qr) + 32 * v, r0 + 8 * v);
#pragma unroll
        for (int i = 0; i < 32; ++i) r0[i] = bf16x2_to_f16x2(r0[i], qmax);
      }
      ptx::tmem_st32(taddr + 32u * c, r0);
    }
  } else {
#pragma unroll 1
  for (int c = C0; c < C1; c += 2) {
    uint32_t r0[32], r1[32];
    const bool two = c + 1 < C1;
#pragma unroll
    for (int v = 0; v < 4; ++v) ptx::ld_global_nc_v8((c < 8 ? qa + c * 128 : qr) + 32 * v, r0 + 8 * v);
    if (two) {
#pragma unroll
      for (int v = 0; v < 4; ++v) ptx::ld_global_nc_v8((c + 1 < 8 ? qa + (c + 1) * 128 : qr) + 32 * v, r1 + 8 * v);
    }
    if (c == kZero) {
#pragma unroll
      for (int i = 0; i < 32; ++i) r0[i] = 0u;
    }
    if (c + 1 == kZero) {
#pragma unroll
      for (int i = 0; i < 32; ++i) r1[i] = 0u;
    }
    ptx::tmem_st32(taddr + 32u * c, r0);
    if (two) ptx::tmem_st32(taddr + 32u * (c + 1), r1);
  }
  }
}

// Load 32-column chunks [c0, c1) of one head's query row into TMEM, one
// chunk per round trip.  The bf16 segment start uses this rolled form: it
// keeps the softmax role's code small, which measured faster than issuing
// two chunks per round trip from unrolled code.
__device__ __forceinline__ void load_q_rolled(const uint8_t* qa, const uint8_t* qr, uint32_t taddr, int c0, int c1) {
#pragma unroll 1
  for (int c = c0; c < c1; ++c) {
    uint32_t r0[32];
    const uint8_t* src = c < 8 ? qa + c * 128 : qr;
#pragma unroll
    for (int v = 0; v < 4; ++v) ptx::ld_global_nc_v8(src + 32 * v, r0 + 8 * v);
    ptx::tmem_st32(taddr + 32u * c, r0);
  }
}

}  // namespace dk

// kMode 0: bf16 cache via TMA; 1: FP8 cache via bulk copies + dequant to
// bf16 operands; 2: FP8 cache with f16 operands (flags inputs outside the
// f16-exact range, which mode 1 then recomputes); 3: sparse top-k decode
// over the bf16 cache (rows gathered by listed slot with 16-byte cp.async);
// 4 / 5: the FP4 cache as 1 / 2; 6 / 7: the 528-byte V4.1 FP8 rows as 1 / 2;
// 8 / 9: the 288-byte V4.1 FP4 rows as 1 / 2
template <int kMode>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(dk::Cfg<kMode>::kThreads, 1)
mla_decode_pair_kernel(const __grid_constant__ CacheMaps maps, const DecodeParams p) {
  using namespace dk;
  using C = Cfg<kMode>;
  constexpr int TH = C::kTileHalves;            // half pages per tile
  constexpr int kN = TH * kHalf;                // tokens per tile (S columns)
  constexpr int kSG = C::kSmGroups;             // softmax warp groups
  constexpr int kHC = kN / kSG;                 // S columns per softmax group
  constexpr int kVSlots = C::kVSlots;
  static_assert(C::kSBufs <= kMaxSBufs && kSCol + C::kSBufs * kN <= 512, "S buffers fit in TMEM");
  static_assert(C::kPSlots <= kMaxPSlots, "P slots and their alpha rows");
  constexpr bool kQuant = kModeQuant<kMode>;   // FP8 or FP4 cache (raw rings, dequant warps)
  constexpr bool kFp4 = kModeFp4<kMode>;
  constexpr bool kV41 = kModeV41<kMode>;         // V4.1 row: 448 latent values, latent dims 448..511 zero
  // a quantised row and the half page the producer copies (its ring slots
  // are sized for the larger FP8 half page)
  constexpr uint32_t kQRow = kFp4 ? (kV41 ? kV41Fp4Row : kFp4Row) : (kV41 ? kV41Row : kFp8Row);
  constexpr uint32_t kQRaw = kHalf * kQRow;
  constexpr bool kF16 = kModeF16<kMode>;          // FP8 or FP4 with f16 operands
  constexpr uint32_t kIdescS =                    // A = Q (TMEM), B = K (K-major)
      kF16 ? ptx::idesc_f16(128, kN, 0, 0) : ptx::idesc_bf16(128, kN, 0, 0);
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
  __nv_bfloat16* part_out = reinterpret_cast<__nv_bfloat16*>(p.ws + p.L.part_out);
  const int* n_parts = reinterpret_cast<const int*>(p.ws + p.L.n_parts);
  auto BAR = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * static_cast<uint32_t>(i); };
  // physical page of row-local half page hp of batch row b (or -1 if out of range)
  auto half_page = [&](int b, int hp) -> int {
    const int page = __ldg(p.block_table + static_cast<size_t>(b) * p.max_pages + (hp >> 1));
    return (page < 0 || page >= p.num_pages) ? -1 : page;
  };

  const bool smem_ok = (sbase & 1023u) == 0;
  if (threadIdx.x == 0) {
    // FP8: this SM's dequant warps
    const uint32_t dq = static_cast<uint32_t>(rank == 1 ? C::kDqWarps1 : C::kDqWarps0);
    constexpr uint32_t kEp = static_cast<uint32_t>(C::kEpWarps);
    // K tiles: the TMA bytes (bf16) or the dequant warps (FP8)
    // sparse: each gather thread arrives once per tile (cp.async noinc)
    constexpr uint32_t kGatherThreads = 32u * kGatherWarps;
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(BAR(KFULL + s), kQuant ? dq : (kMode == 3 ? kGatherThreads : 1u));
      ptx::mbar_init(BAR(KEMPTY + s), 1);
      ptx::mbar_init(BAR(KFULLB + s), kMode == 3 ? kGatherThreads : 1u);
      ptx::mbar_init(BAR(KEMPTYB + s), 1);
    }
    // V slots: the TMA bytes (bf16) or the dequant warps (FP8)
    for (int s = 0; s < kMaxVSlots; ++s) {
      ptx::mbar_init(BAR(VFULL + s), kQuant ? dq : (kMode == 3 ? 32u : 1u));   // sparse: one warp per half page
      ptx::mbar_init(BAR(VEMPTY + s), 1);
    }
    for (int s = 0; s < kMaxPSlots; ++s) { ptx::mbar_init(BAR(PFULL + s), 128 * kSG); ptx::mbar_init(BAR(PEMPTY + s), 1); }
    for (int s = 0; s < kMaxSBufs; ++s) { ptx::mbar_init(BAR(SFULL + s), 1); ptx::mbar_init(BAR(SEMPTY + s), 128 * kSG); }
    ptx::mbar_init(BAR(QREADY), 128 * kSG);
    ptx::mbar_init(BAR(REQ), 2);
    ptx::mbar_init(BAR(CORR), kEp);
    ptx::mbar_init(BAR(OFULL), 1);
    ptx::mbar_init(BAR(OEMPTY), 32 * kEp);
    ptx::mbar_init(BAR(LSUM), 128);
    for (int s = 0; s < kMailSlots; ++s) { ptx::mbar_init(BAR(MBFULL + s), 128); ptx::mbar_init(BAR(MBEMPTY + s), kEp); }
    for (int s = 0; s < kMaxRaw; ++s) {
      ptx::mbar_init(BAR(RAWFULL + s), 1);
      ptx::mbar_init(BAR(RAWEMPTY + s), kQuant ? dq : 1u);
    }
    ptx::mbar_init(BAR(DRAIN), 1);
    ptx::fence_barrier_init();
  }
  if (warp == 2) {
    ptx::tmem_alloc(sbase + kOffTmemPtr, kTmemCols);
    ptx::tmem_relinquish();
  }
  if (kMode == 0 && warp == 0 && lane == 0) {
    if (rank == 1) {
      ptx::prefetch_tmap(&maps.k);
      ptx::prefetch_tmap(&maps.k8);
      ptx::prefetch_tmap(&maps.kb);
      ptx::prefetch_tmap(&maps.kb8);
    } else {
      ptx::prefetch_tmap(&maps.v);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  ptx::cluster_sync();   // barriers of both ranks initialised before any remote arrive
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffTmemPtr);
  // Everything above overlaps the planner when this grid is its programmatic
  // dependent; the plan is read only after the planner grid has completed.
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();   // the merge kernel may begin launching
  if (threadIdx.x == 0 && !smem_ok) set_status(&hdr->status, MLA_ERR_UNSUPPORTED);

  const int ppg = p.pairs_per_group;
  const int group = static_cast<int>(pair) / ppg;     // query index i served by this pair
  const int pl = static_cast<int>(pair) % ppg;
  const int spq = hdr->slots_per_query;
  const int* pair_lo = reinterpret_cast<const int*>(p.ws + p.L.pair_lo);
  const int* pair_rank = reinterpret_cast<const int*>(p.ws + p.L.pair_rank);   // non-empty pairs before p
  const int lo = pair_lo[pl], hi = pair_lo[pl + 1];     // this pair's page range (cost-balanced by the planner)
  const int b0 = reinterpret_cast<const int*>(p.ws + p.L.pair_b0)[pl];   // the row holding page lo

  const int sq = p.sq;
  // the exact FP8 pass after an f16 pass runs only if that pass flagged an
  // input outside the f16-exact range
  const bool active = smem_ok && group < sq && !(p.fp8_fallback && hdr->fp8_range == 0);

  if (kMode == 3 && active && (warp == 0 || warp == 2 || warp == 3)) {
    // ------------------------------------------------------------ sparse gather (both ranks)
    // Warp gw copies half page gw of every tile: the row-local tokens
    // [32 (h0 + gw), +32) of the segment's row, whose cache slots come from
    // the compacted list.  One cache row is 1152 contiguous bytes; the lanes
    // copy consecutive 16-byte pieces of it (coalesced), each into its
    // 128B-swizzled place: rank 1 the A part (chunks 0..4) and B part
    // (chunks 5..8) blocks of the K tile buffer, rank 0 the eight latent
    // chunks of a V slot.  Completion is counted per thread with
    // cp.async.mbarrier.arrive.noinc; the MMA issuers fence the generic and
    // async proxies after their waits.  Tokens past the row's count are not
    // copied (the softmax masks them; the value SM zeroes their V rows).
    const int gw = warp == 0 ? 0 : warp - 1;
    SegWalker w; w.init(tile_start, p.batch, lo, hi, b0);
    Segment sg;
    int kb = 0; uint32_t kphase = 0;      // rank 1: K tile buffer
    int vs = 0; uint32_t vphase = 0;      // rank 0: V ring head
    bool ok = true;
    while (ok && w.next(sg)) {
      const int len = lens[sg.b];
      const int32_t* slots = p.sp_slots + static_cast<size_t>(sg.b) * p.topk;
      const int hp_end = 2 * sg.t1;
      for (int h0 = 2 * sg.t0; h0 < hp_end && ok; h0 += TH) {
        const int nh = min(TH, hp_end - h0);
        const int r0 = (h0 + gw) * kHalf;                       // row-local index of this warp's first token
        const int n_rows = gw < nh ? max(0, min(kHalf, len - r0)) : 0;
        const int my_slot = lane < n_rows ? __ldg(slots + r0 + lane) : 0;
        const int c = lane >> 3, q = lane & 7;                  // chunk (of four) and 16-byte piece of a lane
        if (rank == 1) {
          // A part: chunks 0..3 of a row are 32 pieces, lane L taking piece
          // L (chunk L/8, piece L%8) of every row; chunk 4 of four rows at a
          // time are 32 pieces, lane L taking piece L%8 of row L/8 of the
          // four.  B part: chunks 5..8, lane L taking piece L of every row.
          const uint32_t tbase = sbase + static_cast<uint32_t>(kb) * (TH * kKSlot) +
                                 static_cast<uint32_t>(gw) * (4 * 5 * kAtom);     // row group 4 gw
          if (!wait_warp<false>(BAR(KEMPTY + kb), kphase ^ 1u, hdr)) { ok = false; break; }
          const uint8_t* asrc = p.kv_bf16 + lane * 16;
#pragma unroll 4
          for (int i = 0; i < n_rows; ++i) {
            const int slot = __shfl_sync(0xffffffffu, my_slot, i);
            ptx::cp_async_16(tbase + static_cast<uint32_t>(i >> 3) * (5 * kAtom) + c * kAtom + (i & 7) * 128 +
                                 ((q ^ (i & 7)) << 4),
                             asrc + static_cast<size_t>(slot) * (kRow * 2));
          }
          const uint8_t* a4src = p.kv_bf16 + 4 * 128 + q * 16;
#pragma unroll 2
          for (int g = 0; 4 * g < n_rows; ++g) {
            const int row = 4 * g + c;                          // c = lane / 8 < 4
            const int slot = __shfl_sync(0xffffffffu, my_slot, row);
            if (row < n_rows)
              ptx::cp_async_16(tbase + static_cast<uint32_t>(row >> 3) * (5 * kAtom) + 4 * kAtom + (row & 7) * 128 +
                                   ((q ^ (row & 7)) << 4),
                               a4src + static_cast<size_t>(slot) * (kRow * 2));
          }
          ptx::cp_async_arrive_noinc(BAR(KFULL + kb));
          if (!wait_warp<false>(BAR(KEMPTYB + kb), kphase ^ 1u, hdr)) { ok = false; break; }
          const uint32_t bbase = sbase + static_cast<uint32_t>(kb) * (TH * kKSlot) + static_cast<uint32_t>(TH) * kKA +
                                 static_cast<uint32_t>(gw) * (4 * 4 * kAtom) + c * kAtom;
          const uint8_t* bsrc = p.kv_bf16 + (5 + c) * 128 + q * 16;
#pragma unroll 4
          for (int i = 0; i < n_rows; ++i) {
            const int slot = __shfl_sync(0xffffffffu, my_slot, i);
            ptx::cp_async_16(bbase + static_cast<uint32_t>(i >> 3) * (4 * kAtom) + (i & 7) * 128 + ((q ^ (i & 7)) << 4),
                             bsrc + static_cast<size_t>(slot) * (kRow * 2));
          }
          ptx::cp_async_arrive_noinc(BAR(KFULLB + kb));
          kb ^= 1;
          if (kb == 0) kphase ^= 1u;
        } else {
          if (gw < nh) {
            int v = vs + gw;
            uint32_t vp = vphase;
            if (v >= kVSlots) { v -= kVSlots; vp ^= 1u; }
            if (!wait_warp<false>(BAR(VEMPTY + v), vp ^ 1u, hdr)) { ok = false; break; }
            const uint32_t vbase = sbase + static_cast<uint32_t>(v) * kVSlot + c * kAtom;
            const uint8_t* vsrc = p.kv_bf16 + lane * 16;
#pragma unroll 4
            for (int i = 0; i < n_rows; ++i) {
              const int slot = __shfl_sync(0xffffffffu, my_slot, i);
              const uint8_t* src = vsrc + static_cast<size_t>(slot) * (kRow * 2);
              const uint32_t dst = vbase + static_cast<uint32_t>(i >> 3) * kVGroup + (i & 7) * 128 + ((q ^ (i & 7)) << 4);
              ptx::cp_async_16(dst, src);
              ptx::cp_async_16(dst + 4 * kAtom, src + 512);
            }
            ptx::cp_async_arrive_noinc(BAR(VFULL + v));
          }
          vs += nh;
          if (vs >= kVSlots) { vs -= kVSlots; vphase ^= 1u; }
        }
      }
    }
    ptx::cp_async_wait_all();   // (after an abort) no copy of this thread may land after the CTA left
  } else if (kMode != 3 && active && warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = ptx::policy_evict_normal();
      SegWalker w; w.init(tile_start, p.batch, lo, hi, b0);
      Segment sg;
      int kb = 0; uint32_t kphase = 0;      // rank 1: K tile buffer
      int vs = 0; uint32_t vphase = 0;      // rank 0: V slot
      int rs = 0; uint32_t rphase = 0;      // FP8: raw ring
      const int n_raw = rank == 1 ? C::kRaw1 : C::kRaw0;
      const uint32_t raw_off = rank == 1 ? C::kOffRaw1 : C::kOffRaw0;
      volatile uint32_t* raw_flag = reinterpret_cast<volatile uint32_t*>(smem + kOffRawFlag);
      // Full barriers this thread armed for copies (bit i: ring slot i, see
      // full_bar below) and the phase parity of each one's last arming: at
      // the end every such phase is waited for, so that no copy lands after
      // the CTA has left (which matters only when a wait gave up).
      uint32_t armed = 0, armed_par = 0;
      auto arm = [&](int bit, uint32_t phase) {
        armed |= 1u << bit;
        armed_par = (armed_par & ~(1u << bit)) | (phase << bit);
      };
      auto full_bar = [&](int bit) -> uint32_t {
        if (kMode != 0) return BAR(RAWFULL + bit);
        if (rank == 0) return BAR(VFULL + bit);
        return bit < 2 ? BAR(KFULL + bit) : BAR(KFULLB + bit - 2);
      };
      bool ok = true;
      while (ok && w.next(sg)) {
        const int hp_end = 2 * sg.t1;
        // Block-table entries are read one tile ahead, so their global-memory
        // latency overlaps the previous tile's waits and copies instead of
        // sitting between the copies (the copies' memory clobbers keep the
        // compiler from hoisting the reads on its own).
        int next_pages[TH];
#pragma unroll
        for (int j = 0; j < TH; ++j) next_pages[j] = 2 * sg.t0 + j < hp_end ? half_page(sg.b, 2 * sg.t0 + j) : 0;
        for (int h0 = 2 * sg.t0; h0 < hp_end && ok; h0 += TH) {
          const int nh = min(TH, hp_end - h0);
          int pages[TH];
#pragma unroll
          for (int j = 0; j < TH; ++j) {
            pages[j] = next_pages[j];
            next_pages[j] = h0 + TH + j < hp_end ? half_page(sg.b, h0 + TH + j) : 0;
          }
          if constexpr (kMode == 0) {
            // a bad page is read fully outside the tensor, which fills zeros
            if (rank == 1) {
              // A tile buffer holds the tile's chunks 0..4 (A part) and
              // chunks 5..8 (B part) of every half page in two blocks.  S
              // consumes the A part first, so the next tile's A part is
              // refilled while S still reads the B part.  Two adjacent slots
              // that hold the two halves of one page take one whole-page box
              // (8 row groups land as the two slots' row groups 0..7), so a
              // 96-token tile costs two TMA operations per part, not three:
              // each operation costs the issuing SM's TMA unit a roughly
              // fixed time, whatever its size.
              const uint32_t tbase = sbase + static_cast<uint32_t>(kb) * (TH * kKSlot);
              int wq[TH];
#pragma unroll
              for (int j = 0; j < TH; ++j) {
                const int page = pages[j];
                if (j < nh && page < 0) set_status(&hdr->status, MLA_STATUS_BAD_PAGE);
                wq[j] = (page < 0 ? p.num_pages : page) * 8 + ((h0 + j) & 1) * 4;
              }
              if (!wait_bounded<true>(BAR(KEMPTY + kb), kphase ^ 1u, hdr)) { ok = false; break; }
              ptx::mbar_arrive_expect_tx(BAR(KFULL + kb), static_cast<uint32_t>(nh) * kKA);
              arm(kb, kphase);
#pragma unroll
              for (int j = 0; j < TH; ++j) {
                if (j >= nh) break;
                const bool whole = ((h0 + j) & 1) == 0 && j + 1 < nh;
                if (j > 0 && ((h0 + j) & 1) == 1) continue;   // second half, loaded with the first
                ptx::tma_load_4d(tbase + static_cast<uint32_t>(j) * kKA, whole ? &maps.k8 : &maps.k, BAR(KFULL + kb),
                                 0, 0, 0, wq[j], pol);
              }
              if (!wait_bounded<true>(BAR(KEMPTYB + kb), kphase ^ 1u, hdr)) { ok = false; break; }
              ptx::mbar_arrive_expect_tx(BAR(KFULLB + kb), static_cast<uint32_t>(nh) * kKB);
              arm(2 + kb, kphase);
#pragma unroll
              for (int j = 0; j < TH; ++j) {
                if (j >= nh) break;
                const bool whole = ((h0 + j) & 1) == 0 && j + 1 < nh;
                if (j > 0 && ((h0 + j) & 1) == 1) continue;
                ptx::tma_load_4d(tbase + static_cast<uint32_t>(TH) * kKA + static_cast<uint32_t>(j) * kKB,
                                 whole ? &maps.kb8 : &maps.kb, BAR(KFULLB + kb), 0, 0, 5, wq[j], pol);
              }
              kb ^= 1;
              if (kb == 0) kphase ^= 1u;
            } else {
#pragma unroll
              for (int j = 0; j < TH; ++j) {
                if (j >= nh) break;
                if (!wait_bounded<true>(BAR(VEMPTY + vs), vphase ^ 1u, hdr)) { ok = false; break; }
                const int hp = h0 + j, page = pages[j];
                const int wq = (page < 0 ? p.num_pages : page) * 8 + (hp & 1) * 4;
                ptx::mbar_arrive_expect_tx(BAR(VFULL + vs), kVSlot);
                arm(vs, vphase);
                ptx::tma_load_4d(sbase + static_cast<uint32_t>(vs) * kVSlot, &maps.v, BAR(VFULL + vs), 0, 0, 0, wq,
                                 pol);
                if (++vs == kVSlots) { vs = 0; vphase ^= 1u; }
              }
            }
          } else {
            // raw half pages; a bad page is never read (dequant writes zeros)
#pragma unroll
            for (int j = 0; j < TH; ++j) {
              if (j >= nh) break;
              if (!wait_bounded<true>(BAR(RAWEMPTY + rs), rphase ^ 1u, hdr)) { ok = false; break; }
              const int hp = h0 + j, page = pages[j];
              if (page < 0) set_status(&hdr->status, MLA_STATUS_BAD_PAGE);
              raw_flag[rs] = page < 0 ? 1u : 0u;
              arm(rs, rphase);
              if (page < 0) {
                ptx::mbar_arrive(BAR(RAWFULL + rs));
              } else {
                ptx::mbar_arrive_expect_tx(BAR(RAWFULL + rs), kQRaw);
                const uint8_t* src = p.kv_quant + static_cast<size_t>(page) * (kPage * kQRow) + (hp & 1) * kQRaw;
                ptx::bulk_load(sbase + raw_off + static_cast<uint32_t>(rs) * kRawBytes, src, kQRaw,
                               BAR(RAWFULL + rs), pol);
              }
              if (++rs == n_raw) { rs = 0; rphase ^= 1u; }
            }
          }
          if (rank == 1 && h0 + TH >= hp_end) {
            // The segment's last tile is on its way: bring the next segment's
            // query rows (128 KiB absorbed + 16 KiB RoPE, each contiguous)
            // into L2, so the softmax warps' Q load a few tiles later hits L2.
            SegWalker w2 = w;
            Segment nx;
            if (w2.next(nx)) {
              const size_t qrow = static_cast<size_t>(nx.b) * sq + group;
              const uint8_t* qa = reinterpret_cast<const uint8_t*>(p.q_abs + qrow * kHeads * kDc);
              const uint8_t* qr = reinterpret_cast<const uint8_t*>(p.q_rope + qrow * kHeads * kDr);
#pragma unroll
              for (int k = 0; k < 4; ++k) ptx::prefetch_l2_bulk(qa + k * 32768, 32768);
              ptx::prefetch_l2_bulk(qr, kHeads * kDr * 2);
            }
          }
        }
      }
#pragma unroll 1
      for (int i = 0; i < 8; ++i)
        if ((armed >> i) & 1u) wait_drain(full_bar(i), (armed_par >> i) & 1u, hdr);
    }
  } else if (kQuant && active && (warp >= 8 || (warp == 2 && rank == 1))) {
    // ------------------------------------------------------------ FP8 dequant
    // raw half page -> rank 1: K slot (all 18 value groups, nine-chunk
    // layout); rank 0: V slot (the 16 latent groups).  Warp wq takes value
    // groups 2wq and 2wq+1; lane = (token lane % 16 and the same token + 16,
    // group 2wq + lane / 16): two independent chains per lane, and each
    // 8-lane phase of a 16-byte store hits eight different swizzled rows.
    const int wq = warp == 2 ? 8 : warp - 8;
    const int t = lane & 15, g = 2 * wq + (lane >> 4);
    const volatile uint32_t* raw_flag = reinterpret_cast<const volatile uint32_t*>(smem + kOffRawFlag);
    const uint32_t raw_off = rank == 1 ? C::kOffRaw1 : C::kOffRaw0;
    const int n_raw = rank == 1 ? C::kRaw1 : C::kRaw0;
    SegWalker w; w.init(tile_start, p.batch, lo, hi, b0);
    Segment sg;
    int kb = 0; uint32_t kphase = 0;      // rank 1: K tile buffer
    int vs = 0; uint32_t vphase = 0;      // rank 0: V slot
    int rs = 0; uint32_t rphase = 0;
    bool ok = true, range_flagged = false;
    while (ok && w.next(sg)) {
      const int hp_end = 2 * sg.t1;
      for (int h0 = 2 * sg.t0; h0 < hp_end && ok; h0 += TH) {
        const int nh = min(TH, hp_end - h0);
        // rank 1: the tile's slots are free once S of the tile two back is done
        if (rank == 1 && !wait_warp<false>(BAR(KEMPTY + kb), kphase ^ 1u, hdr)) { ok = false; break; }
        for (int j = 0; j < nh; ++j) {
          // rank 0: the V slot is free once its P.V is done
          if (rank == 0 && !wait_warp<false>(BAR(VEMPTY + vs), vphase ^ 1u, hdr)) { ok = false; break; }
          if (!wait_warp<false>(BAR(RAWFULL + rs), rphase, hdr)) { ok = false; break; }
          uint32_t o0[16], o1[16];
          if (raw_flag[rs] == 0) {
            const uint8_t* row = smem + raw_off + static_cast<uint32_t>(rs) * kRawBytes + t * kQRow;
            bool r0 = true, r1 = true;
            if constexpr (kV41) {
              // V4.1 row: its groups 0..13 are the latent (dims 0..447), its
              // groups 14 and 15 the RoPE values (this row's groups 16, 17);
              // this row's groups 14 and 15 (dims 448..511) are zero
              const int sg = g < 14 ? g : g - 2;
              if (g == 14 || g == 15) {
#pragma unroll
                for (int e = 0; e < 16; ++e) { o0[e] = 0u; o1[e] = 0u; }
              } else if constexpr (kFp4 && kF16) {
                r0 = dequant_group_fp4_f16<kV41Values / 2>(row, sg, o0);
                r1 = dequant_group_fp4_f16<kV41Values / 2>(row + 16 * kQRow, sg, o1);
              } else if constexpr (kFp4) {
                dequant_group_fp4<kV41Values / 2>(row, sg, o0);
                dequant_group_fp4<kV41Values / 2>(row + 16 * kQRow, sg, o1);
              } else {
                r0 = dequant_group<kF16, kV41Values>(row, sg, o0);
                r1 = dequant_group<kF16, kV41Values>(row + 16 * kQRow, sg, o1);
              }
            } else if constexpr (kFp4 && kF16) {
              r0 = dequant_group_fp4_f16(row, g, o0);
              r1 = dequant_group_fp4_f16(row + 16 * kQRow, g, o1);
            } else if constexpr (kFp4) {
              dequant_group_fp4(row, g, o0);
              dequant_group_fp4(row + 16 * kQRow, g, o1);
            } else {
              r0 = dequant_group<kF16>(row, g, o0);
              r1 = dequant_group<kF16>(row + 16 * kQRow, g, o1);
            }
            if (kF16 && !range_flagged && __any_sync(0xffffffffu, !(r0 && r1))) {
              if (lane == 0) atomicExch(&hdr->fp8_range, 1);
              range_flagged = true;
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) { o0[e] = 0u; o1[e] = 0u; }
          }
          if (rank == 1) {
            uint8_t* slot = smem + static_cast<uint32_t>(kb * TH + j) * kKSlot;
            store_group(slot, kKGroup, t, g, o0);
            store_group(slot, kKGroup, t + 16, g, o1);
          } else {
            uint8_t* slot = smem + static_cast<uint32_t>(vs) * kVSlot;
            store_group(slot, kVGroup, t, g, o0);
            store_group(slot, kVGroup, t + 16, g, o1);
          }
          ptx::fence_proxy_async_cta();      // generic smem writes -> visible to the MMA
          __syncwarp();
          if (lane == 0) {
            ptx::mbar_arrive(BAR(RAWEMPTY + rs));
            if (rank == 0) ptx::mbar_arrive(BAR(VFULL + vs));
          }
          if (++rs == n_raw) { rs = 0; rphase ^= 1u; }
          if (rank == 0 && ++vs == kVSlots) { vs = 0; vphase ^= 1u; }
        }
        if (!ok) break;
        __syncwarp();
        if (rank == 1 && lane == 0) ptx::mbar_arrive(BAR(KFULL + kb));
        kb ^= 1;
        if (kb == 0) kphase ^= 1u;
      }
    }
  } else if (active && warp == 1 && rank == 1) {
    // ------------------------------------------------------------ S = Q K^T issuer
    // One tile = TH adjacent half-page slots = one kN-row K-major operand;
    // K-step k reads chunk k/4 at byte 32*(k%4) inside the 8-row atoms.
    SegWalker w; w.init(tile_start, p.batch, lo, hi, b0);
    Segment sg;
    int kb = 0; uint32_t kphase = 0;
    int sb = 0; uint32_t sphase = 0;
    uint32_t qphase = 0;
    bool ok = true, issued = false;
#ifdef MLA_TEST_STALL_WAIT
    // Test builds only: a wait on a barrier that nothing arrives on before
    // the end of the kernel, so that the wait limit (MLA_WAIT_TIMEOUT_NS) runs
    // out and every role leaves through the abort path.
    ok = wait_warp<false>(BAR(DRAIN), 0u, hdr);
#endif
    while (ok && w.next(sg)) {
      if (!wait_warp<false>(BAR(QREADY), qphase, hdr)) break;
      issued = true;
      qphase ^= 1u;
      const int hp_end = 2 * sg.t1;
      for (int h0 = 2 * sg.t0; h0 < hp_end && ok; h0 += TH) {
        if (!wait_warp<false>(BAR(KFULL + kb), kphase, hdr) ||
            !wait_warp<false>(BAR(SEMPTY + sb), sphase ^ 1u, hdr)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t d = tmem + kSCol + static_cast<uint32_t>(kN * sb);
        if constexpr (kMode == 0 || kMode == 3) {
          if constexpr (kMode == 3) ptx::fence_proxy_async_cta();   // rows written by cp.async
          // A part (K-steps 0..19, chunks 0..4, 5 KiB per row group), then
          // B part (K-steps 20..35, chunks 5..8, 4 KiB per row group); the
          // A part's slots are released as soon as its MMAs are done
          const uint32_t tbase = sbase + static_cast<uint32_t>(kb) * (TH * kKSlot);
          if (lane == 0) {
            const uint64_t da = ptx::sdesc_sw128(tbase, 16, 5 * kAtom);
#pragma unroll
            for (int k = 0; k < 20; ++k)
              ptx::mma_ts(d, tmem + kQCol + 8u * k, da + static_cast<uint64_t>(((k >> 2) * kAtom + (k & 3) * 32) >> 4),
                          kIdescS, k > 0 ? 1u : 0u);
            ptx::mma_commit(BAR(KEMPTY + kb));
          }
          __syncwarp();
          if (!wait_warp<false>(BAR(KFULLB + kb), kphase, hdr)) { ok = false; break; }
          ptx::tc_fence_after();
          if constexpr (kMode == 3) ptx::fence_proxy_async_cta();
          if (lane == 0) {
            const uint64_t db = ptx::sdesc_sw128(tbase + static_cast<uint32_t>(TH) * kKA, 16, 4 * kAtom);
#pragma unroll
            for (int k = 20; k < kRow / 16; ++k)
              ptx::mma_ts(d, tmem + kQCol + 8u * k,
                          db + static_cast<uint64_t>((((k >> 2) - 5) * kAtom + (k & 3) * 32) >> 4), kIdescS, 1u);
            ptx::mma_commit(BAR(KEMPTYB + kb));
            ptx::mma_commit(BAR(SFULL + sb));
          }
        } else if (lane == 0) {
          // FP8: nine chunks per row group in one slot run (the RoPE chunk is
          // the ninth, 8 KiB into each row group)
          const uint64_t desc0 = ptx::sdesc_sw128(sbase + static_cast<uint32_t>(kb * TH) * kKSlot, 16, kKGroup);
          const uint64_t rope0 = desc0 + static_cast<uint64_t>((8 * kAtom) >> 4);
#pragma unroll
          for (int k = 0; k < kRow / 16; ++k) {
            const uint64_t bdesc = k < 32 ? desc0 + static_cast<uint64_t>(((k >> 2) * kAtom + (k & 3) * 32) >> 4)
                                          : rope0 + static_cast<uint64_t>(((k & 3) * 32) >> 4);
            ptx::mma_ts(d, tmem + kQCol + 8u * k, bdesc, kIdescS, k > 0 ? 1u : 0u);
          }
          ptx::mma_commit(BAR(KEMPTY + kb));
          ptx::mma_commit(BAR(SFULL + sb));
        }
        __syncwarp();
        kb ^= 1;
        if (kb == 0) kphase ^= 1u;
        if (++sb == C::kSBufs) { sb = 0; sphase ^= 1u; }
      }
    }
    // every MMA this thread issued completes before the CTA may leave
    if (issued && lane == 0) {
      ptx::mma_commit(BAR(DRAIN));
      wait_drain(BAR(DRAIN), 0u, hdr);
    }
    __syncwarp();
  } else if (active && warp == 1 && rank == 0) {
    // ------------------------------------------------------------ O += P V issuer
    // Per half page of the tile: two K-steps of 16 tokens (two row groups of
    // the V slot each), two N=256 halves of the latent columns per step.
    SegWalker w; w.init(tile_start, p.batch, lo, hi, b0);
    Segment sg;
    int vs = 0; uint32_t vphase = 0;
    int ps = 0; uint32_t pphase = 0;
    uint32_t corr_phase = 0, oe_phase = 0;
    bool first_seg = true, ok = true, issued = false;
    volatile uint32_t* req_slot = reinterpret_cast<volatile uint32_t*>(smem + kOffReq);
    const volatile float* alpha_buf = reinterpret_cast<const volatile float*>(smem + kOffAlpha);
    while (ok && w.next(sg)) {
      issued = true;
      const int len_i = lens[sg.b] - (sq - 1 - group);
      const int hp_end = 2 * sg.t1;
      for (int h0 = 2 * sg.t0; h0 < hp_end && ok; h0 += TH) {
        const int nh = min(TH, hp_end - h0);
        if (!wait_warp<true>(BAR(PFULL + ps), pphase, hdr)) { ok = false; break; }
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
        if (h0 == 2 * sg.t0 && !first_seg) {
          if (!wait_warp<false>(BAR(OEMPTY), oe_phase, hdr)) { ok = false; break; }
          oe_phase ^= 1u;
        }
        const uint32_t pbase = sbase + C::kOffP + static_cast<uint32_t>(ps) * C::kPSlotBytes;
        for (int j = 0; j < nh; ++j) {
          if (!wait_warp<false>(BAR(VFULL + vs), vphase, hdr)) { ok = false; break; }
          if constexpr (kMode == 3) ptx::fence_proxy_async_cta();   // rows written by cp.async
          const int valid = len_i - (h0 + j) * kHalf;   // tokens of this half page visible to the query
          if (valid < kHalf) {
            // rows past the visible length get P = 0; make their V finite too
            const int v0 = valid > 0 ? valid : 0;
            uint8_t* slot = smem + static_cast<uint32_t>(vs) * kVSlot;
            for (int i = lane; i < (kHalf - v0) * 8 * 8; i += 32) {   // rows x chunks x 16-byte pieces
              const int r = v0 + i / 64, c = (i / 8) & 7, q = i & 7;
              *reinterpret_cast<uint4*>(slot + (r >> 3) * kVGroup + c * kAtom + (r & 7) * 128 + q * 16) =
                  make_uint4(0, 0, 0, 0);
            }
            ptx::fence_proxy_async_cta();
            __syncwarp();
          }
          ptx::tc_fence_after();
          if (lane == 0) {
            const uint32_t vbase = sbase + static_cast<uint32_t>(vs) * kVSlot;
#pragma unroll
            for (int s = 0; s < 2; ++s) {
              const int k = 2 * j + s;                   // K-step of the tile
              const uint64_t adesc = ptx::sdesc_sw128(pbase + (k >> 2) * kPChunk + (k & 3) * 32, 16, 1024);
#pragma unroll
              for (int n = 0; n < 2; ++n) {
                const uint64_t bdesc =
                    ptx::sdesc_sw128(vbase + static_cast<uint32_t>(s * 2) * kVGroup + n * 4 * kAtom, kAtom, kVGroup);
                ptx::mma_ss(tmem + 256u * n, adesc, bdesc, kIdescPV<kMode>, (h0 > 2 * sg.t0 || k > 0) ? 1u : 0u);
              }
            }
            ptx::mma_commit(BAR(VEMPTY + vs));
          }
          __syncwarp();
          if (++vs == kVSlots) { vs = 0; vphase ^= 1u; }
        }
        if (!ok) break;
        if (lane == 0) {
          ptx::mma_commit_mc(BAR(PEMPTY + ps), static_cast<uint16_t>(1u << 1));
          if (h0 + TH >= hp_end) ptx::mma_commit(BAR(OFULL));
        }
        __syncwarp();
        if (++ps == C::kPSlots) { ps = 0; pphase ^= 1u; }
      }
      first_seg = false;
    }
    // every MMA (and the commits to rank 1) this thread issued completes
    // before the CTA may leave
    if (issued && lane == 0) {
      ptx::mma_commit(BAR(DRAIN));
      wait_drain(BAR(DRAIN), 0u, hdr);
    }
    __syncwarp();
  } else if (active && warp >= 4 && warp < 4 + 4 * kSG && rank == 1) {
    // ------------------------------------------------------------ softmax (thread = head)
    // bf16 (two groups): group 0 (warps 4..7) turns columns [0, kHC) of each
    // tile's S into P, group 1 (warps 8..11) columns [kHC, kN).  Both take the
    // row max over all kN columns, so their reference maxima and rescale
    // factors agree without an exchange; the two partial sums meet once per
    // segment (LSUM barrier).  FP8 (one group): warps 4..7 take all columns.
    const int grp = (warp - 4) >> 2;
    const int h = (threadIdx.x - 128) & 127;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    volatile float* l_part = reinterpret_cast<volatile float*>(smem + C::kOffMisc + kMiscLPart);
    SegWalker w; w.init(tile_start, p.batch, lo, hi, b0);
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
      {
        // Q row h -> TMEM lane h, columns [0, 288): two bf16 per column, K
        // order, 32 columns (128 B of the row) per chunk.  With two groups,
        // group 0 loads chunks 0..4 and group 1 chunks 5..8; each reaches
        // this point only after the previous segment's last S (which reads
        // Q) has completed.
        const uint8_t* qa = reinterpret_cast<const uint8_t*>(p.q_abs + (static_cast<size_t>(row) * kHeads + h) * kDc);
        const uint8_t* qr = reinterpret_cast<const uint8_t*>(p.q_rope + (static_cast<size_t>(row) * kHeads + h) * kDr);
        const uint32_t qaddr = tmem + lane_base + kQCol;
        float qmax = 0.f;
        if (kSG == 1) load_q_chunks<0, 9, kF16, kV41 ? 7 : -1>(qa, qr, qaddr, qmax);
        else load_q_rolled(qa, qr, qaddr, grp == 0 ? 0 : 5, grp == 0 ? 5 : 9);
        if (kF16 && __any_sync(0xffffffffu, qmax > kF16Max) && lane == 0) atomicExch(&hdr->fp8_range, 1);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(BAR(QREADY));
      }
      float m_ref = -INFINITY, l = 0.f;
      const int hp_end = 2 * sg.t1;
      for (int h0 = 2 * sg.t0; h0 < hp_end; h0 += TH) {
        if (!wait_warp<false>(BAR(SFULL + sb), sphase, hdr)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t sadr = tmem + lane_base + kSCol + static_cast<uint32_t>(kN * sb);
        const int c_mine = kHC * grp, c_other = kHC * (grp ^ 1);
        uint32_t mine[kHC], other[kSG == 2 ? kHC : 1];
#pragma unroll
        for (int j = 0; j < kHC / 16; ++j) {
          ptx::tmem_ld16(sadr + c_mine + 16 * j, mine + 16 * j);
          if constexpr (kSG == 2) ptx::tmem_ld16(sadr + c_other + 16 * j, other + 16 * j);
        }
        ptx::tmem_wait_ld();
        ptx::tc_fence_before();
        ptx::mbar_arrive(BAR(SEMPTY + sb));
        // columns of this tile visible to the query: within the row's length
        // and within the half pages this tile loaded (the segment may end
        // before the row does; slots past it hold stale data)
        const int valid = min(len_i - h0 * kHalf, min(TH, hp_end - h0) * kHalf);
        // row max of the masked raw scores.  m_ref stays in raw score units and
        // P = exp2((s - m_ref) * c), so the max element gets exactly exp2(0) = 1
        // whatever the magnitude of the scores (scale c > 0).
        const bool full = valid >= kN;                 // the same for every head of the tile
        float mx = -INFINITY;
        if (full) {
          if constexpr (kSG == 2) {
#pragma unroll
            for (int e = 0; e < kHC; ++e) mx = max3(mx, __uint_as_float(mine[e]), __uint_as_float(other[e]));
          } else {
#pragma unroll
            for (int e = 0; e < kHC; e += 2) mx = max3(mx, __uint_as_float(mine[e]), __uint_as_float(mine[e + 1]));
          }
        } else {
#pragma unroll
          for (int e = 0; e < kHC; ++e) {
            if (c_mine + e < valid) mx = fmaxf(mx, __uint_as_float(mine[e]));
            if constexpr (kSG == 2)
              if (c_other + e < valid) mx = fmaxf(mx, __uint_as_float(other[e]));
          }
        }
        float alpha = 1.f;
        if (h0 == 2 * sg.t0) {
          m_ref = mx;
        } else if ((mx - m_ref) * c > kRescaleThreshold<kMode>) {
          alpha = fast_exp2((m_ref - mx) * c);
          l *= alpha;
          m_ref = mx;
        }
        uint32_t pk[kHC / 2];
        float la = 0.f, lb = 0.f;
        if (full) {
#pragma unroll
          for (int e = 0; e < kHC / 2; ++e) {
            float x0 = __uint_as_float(mine[2 * e]), x1 = __uint_as_float(mine[2 * e + 1]);
            sub_scale2(x0, x1, -m_ref, c);
            const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
            pk[e] = kF16 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
            add2(la, lb, p0, p1);
          }
        } else {
#pragma unroll
          for (int e = 0; e < kHC / 2; ++e) {
            const int col = c_mine + 2 * e;
            const float p0 = col < valid ? fast_exp2((__uint_as_float(mine[2 * e]) - m_ref) * c) : 0.f;
            const float p1 = col + 1 < valid ? fast_exp2((__uint_as_float(mine[2 * e + 1]) - m_ref) * c) : 0.f;
            pk[e] = kF16 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
            la += p0;
            lb += p1;
          }
        }
        l += la + lb;
        if (m_ref == -INFINITY) l = 0.f;     // nothing visible yet (every p was 0)
        if (!wait_warp<true>(BAR(PEMPTY + ps), pphase ^ 1u, hdr)) { ok = false; break; }
        // This group's columns of P row h (kHC/8 pieces of 16 B: piece q holds
        // tokens 8q..8q+7, in chunk q/8 at swizzled position (q%8) ^ (h%8)) --
        // and, from group 0, alpha_h -- go to rank 0 as st.async bytes counted
        // on its PFULL barrier: nobody waits for them here.
        // alpha of heads 4i..4i+3 gathered into lane i (< 8) of each group-0
        // warp, sent as one 16-byte store per lane
        float a4[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) a4[k] = __shfl_sync(0xffffffffu, alpha, ((lane & 7) << 2) + k);
        const bool sends_alpha = grp == 0 && lane < 8;
        const uint32_t pfull = ptx::mapa(BAR(PFULL + ps), 0);
        ptx::mbar_arrive_expect_tx_remote(pfull, 2u * kHC + (sends_alpha ? 16u : 0u));
        const uint32_t prow = ptx::mapa(sbase + C::kOffP + static_cast<uint32_t>(ps) * C::kPSlotBytes + h * 128u, 0);
#pragma unroll
        for (int j = 0; j < kHC / 8; ++j) {
          const int q = grp * (kHC / 8) + j;
          ptx::st_async_v4(prow + static_cast<uint32_t>(q >> 3) * kPChunk + ((static_cast<uint32_t>(q & 7) ^ (h & 7)) << 4),
                           pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3], pfull);
        }
        if (sends_alpha)
          ptx::st_async_v4(ptx::mapa(sbase + kOffAlpha + ps * 512u + (h + 3 * lane) * 4u, 0), __float_as_uint(a4[0]),
                           __float_as_uint(a4[1]), __float_as_uint(a4[2]), __float_as_uint(a4[3]), pfull);
        if (++sb == C::kSBufs) { sb = 0; sphase ^= 1u; }
        if (++ps == C::kPSlots) { ps = 0; pphase ^= 1u; }
      }
      if (!ok) break;
      if (kSG == 2 && grp == 1) {
        // hand group 1's partial sum to group 0 (read before group 0 loads the
        // next segment's Q, so group 1 cannot overwrite it early)
        l_part[h] = l;
        ptx::mbar_arrive(BAR(LSUM));
      } else {
        if constexpr (kSG == 2) {
          if (!wait_warp<false>(BAR(LSUM), lsum_phase, hdr)) { ok = false; break; }
          l += l_part[h];
        }
        const bool split = slot_base[sg.b] >= 0;
        const int slot = split ? group * spq + slot_base[sg.b] + (pair_rank[pl] - pair_rank[first_pair[sg.b]]) : -1;
        const float lse_v = l > 0.f ? (m_ref * c + log2f(l)) * kLn2 : -INFINITY;
        const float inv_l = l > 0.f ? __frcp_rn(l) : 0.f;   // correctly rounded, as 1/l
        if (split) {
          part_lse[static_cast<size_t>(slot) * kHeads + h] = lse_v;
        } else {
          p.lse[static_cast<size_t>(row) * kHeads + h] = lse_v;
        }
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
      for (int s = 0; s < C::kPSlots && ok; ++s) {
        ok = wait_warp<true>(BAR(PEMPTY + ps), pphase ^ 1u, hdr);
        if (++ps == C::kPSlots) { ps = 0; pphase ^= 1u; }
      }
      for (int s = 0; s < kMailSlots && ok; ++s) {
        ok = wait_warp<true>(BAR(MBEMPTY + ms), mphase ^ 1u, hdr);
        if (++ms == kMailSlots) { ms = 0; mphase ^= 1u; }
      }
    }
  } else if (active && warp >= 4 && warp < 4 + C::kEpWarps && rank == 0) {
    // ------------------------------------------------------------ rescale + epilogue
    // bf16: eight warps, warps 4..7 take latent columns [0, 256) of head rows
    // 0..127, warps 8..11 columns [256, 512).  FP8: warps 4..7 take all 512.
    constexpr int kEpChunks = 16 / (C::kEpWarps / 4);   // 32-column chunks per warp
    const int h = (threadIdx.x - 128) & 127;
    const int c0 = kEpChunks * ((warp - 4) >> 2);     // first 32-column chunk of this warp
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    SegWalker w; w.init(tile_start, p.batch, lo, hi, b0);
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
            for (int cc = c0; cc < c0 + kEpChunks; ++cc) {
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
      const int parts = n_parts[sg.b];
      const int slot0 = parts > 1 ? group * spq + slot_base[sg.b] : 0;        // the row's first partial slot
      const int mine = parts > 1 ? pair_rank[pl] - pair_rank[first_pair[sg.b]] : 0;
      {
        // out = bf16(O / l): into the output row, or (split rows) into the
        // row's partial slot (number `mine` of the row's parts), which the
        // merge kernel combines
        __nv_bfloat16* dst = parts > 1 ? part_out + (static_cast<size_t>(slot0 + mine) * kHeads + h) * kDc
                                       : p.out + (static_cast<size_t>(row) * kHeads + h) * kDc;
        // two chunks per tensor-memory wait where the registers allow (bf16)
        constexpr int kEpBatch = C::kThreads <= 384 ? 2 : 1;
#pragma unroll 1
        for (int cc = c0; cc < c0 + kEpChunks; cc += kEpBatch) {
          uint32_t r[kEpBatch][32];
#pragma unroll
          for (int k = 0; k < kEpBatch; ++k) ptx::tmem_ld32(tmem + lane_base + 32u * (cc + k), r[k]);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < kEpBatch; ++k) {
            uint32_t o[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              o[e] = pack_bf16x2(__uint_as_float(r[k][2 * e]) * inv_l, __uint_as_float(r[k][2 * e + 1]) * inv_l);
            ptx::st_global_v8(dst + (cc + k) * 32, o);          // whole 32-byte sectors
            ptx::st_global_v8(dst + (cc + k) * 32 + 16, o + 8);
          }
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
  // After a wait gave up, the partner CTA's st.async stores into this CTA's
  // shared memory may still be in flight, and nothing counts them any more:
  // give them time to land (they take about a microsecond) before the
  // cluster may leave.  Copies and MMAs this CTA issued were drained above.
  if (read_status(&hdr->abort_flag) != 0) spin_ns(20000);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();
  if (warp == 2) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

namespace {

// Host-side launcher.  kMode 0: bf16 cache through the 4-D tensor maps
// (half- and whole-page boxes of chunks 0..4 and 5..8 for rank 1, half-page
// boxes of the eight latent chunks for rank 0); 1 and 2: FP8 cache, 4 and 5:
// FP4 cache, 6 and 7: FP8 V4.1 rows, 8 and 9: FP4 V4.1 rows (p.kv_quant;
// tensor maps unused; 2, 5, 7 and 9 take f16 operands, 1, 4, 6 and 8
// bf16); 3: sparse gather from the bf16 cache.  It lives in an
// unnamed namespace so that its per-device static is this library's own:
// a function-local static of a template with external linkage is one
// object per process, shared by every loaded copy of the library.
template <int kMode>
cudaError_t launch_decode_mode(const CacheMaps& maps, const DecodeParams& p, int n_pairs, bool pdl,
                               cudaStream_t stream) {
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
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, maps, p);
}

}  // namespace

cudaError_t launch_decode_bf16(const CacheMaps& maps, const DecodeParams& p, int n_pairs, bool pdl,
                               cudaStream_t stream) {
  return launch_decode_mode<0>(maps, p, n_pairs, pdl, stream);
}

cudaError_t launch_decode_fp8(const DecodeParams& p, int n_pairs, bool pdl, cudaStream_t stream) {
  CacheMaps unused;
  memset(&unused, 0, sizeof(unused));
  // the f16-operand pass, then the exact bf16-operand pass, which returns at
  // once unless the first pass flagged an input outside the f16-exact range
  DecodeParams q = p;
  q.fp8_fallback = 0;
  cudaError_t e = launch_decode_mode<2>(unused, q, n_pairs, pdl, stream);
  if (e != cudaSuccess) return e;
  q.fp8_fallback = 1;
  return launch_decode_mode<1>(unused, q, n_pairs, pdl, stream);
}

cudaError_t launch_decode_fp4(const DecodeParams& p, int n_pairs, bool pdl, cudaStream_t stream) {
  CacheMaps unused;
  memset(&unused, 0, sizeof(unused));
  // as for FP8: the f16-operand pass, then the exact bf16-operand pass,
  // which returns at once unless the first pass flagged an input
  DecodeParams q = p;
  q.fp8_fallback = 0;
  cudaError_t e = launch_decode_mode<5>(unused, q, n_pairs, pdl, stream);
  if (e != cudaSuccess) return e;
  q.fp8_fallback = 1;
  return launch_decode_mode<4>(unused, q, n_pairs, pdl, stream);
}

cudaError_t launch_decode_fp8_v41(const DecodeParams& p, int n_pairs, bool pdl, cudaStream_t stream) {
  CacheMaps unused;
  memset(&unused, 0, sizeof(unused));
  // as for FP8: the f16-operand pass, then the exact bf16-operand pass,
  // which returns at once unless the first pass flagged an input
  DecodeParams q = p;
  q.fp8_fallback = 0;
  cudaError_t e = launch_decode_mode<7>(unused, q, n_pairs, pdl, stream);
  if (e != cudaSuccess) return e;
  q.fp8_fallback = 1;
  return launch_decode_mode<6>(unused, q, n_pairs, pdl, stream);
}

cudaError_t launch_decode_fp4_v41(const DecodeParams& p, int n_pairs, bool pdl, cudaStream_t stream) {
  CacheMaps unused;
  memset(&unused, 0, sizeof(unused));
  DecodeParams q = p;
  q.fp8_fallback = 0;
  cudaError_t e = launch_decode_mode<9>(unused, q, n_pairs, pdl, stream);
  if (e != cudaSuccess) return e;
  q.fp8_fallback = 1;
  return launch_decode_mode<8>(unused, q, n_pairs, pdl, stream);
}

cudaError_t launch_decode_sparse(const DecodeParams& p, int n_pairs, bool pdl, cudaStream_t stream) {
  CacheMaps unused;
  memset(&unused, 0, sizeof(unused));
  return launch_decode_mode<3>(unused, p, n_pairs, pdl, stream);
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
