// Split kernel of sparse MLA decode for sm_103a.
//
// One CTA handles one (query b, group of NH heads, split s of the top-k list).  For
// each tile of 128 index slots it
//   1. gathers the selected 584-byte rows once for all NH heads ("The Moment of
//      Compilation: When a Triton Kernel Meets Its Constraints", section "The
//      Context: A Kernel Optimization Campaign": one KV read shared by all heads),
//   2. dequantises the FP8 e4m3 nope part with its per-64-column UE8M0 scales into an
//      f16 tile ("The Power-of-Two Trap: Debugging a Triton MMA Kernel on Blackwell
//      GPUs", section "3. The Scale Indexing Complication") next to the rope,
//   3. computes S^T = K_tile . Q^T on the tensor cores (tcgen05.mma, M = 128 tokens,
//      N = NH heads, K = 512) into tensor memory,
//   4. runs the online softmax of the tile,
//   5. accumulates O^T += V_tile^T . P^T on the tensor cores (4 blocks of M = 128
//      value columns, N = NH, K = 128 tokens) in tensor memory,
// and finally writes the normalised partial O and its log-sum-exp for the split
// (the split-K scheme of "The 80KB Mystery: Resolving Contradictory Evidence in
// Triton Kernel Optimization", section "The Context: Optimizing Attention on
// Blackwell").
//
// Design (sm_103a).  Tokens are the MMA's M dimension, so every MMA is a full
// 128-row tcgen05 instruction even with 16 heads.  The nope operands are f16 (fp32
// accumulation): e4m3 -> f16 is one conversion and the power-of-two group scale
// one f16x2 multiply, with no integer work per element, and the attention weights
// P keep 11 significant bits.  Nope values must lie in the f16 range (the kernel
// reports SMLA_ERR_RANGE otherwise).  The rope columns stay bf16 and are multiplied
// by bf16 q into the same fp32 accumulator.  One tile in shared memory
// serves as K (K-major view) for the scores and as V^T (MN-major view) for the
// output.  The 448-wide value product runs as four 128-row blocks; the 4th block
// pairs value columns 384..447 with a constant block whose first column is 1, so
// output row 448 of that block is sum_t P[t], the softmax denominator, accumulated
// and rescaled by the tensor core together with O.
//
// Warp roles (512 threads):
//   warp 0       allocates tensor memory and issues every tcgen05.mma (one lane)
//   warps 4..7   softmax and epilogue; thread t owns TMEM lane t (token t of the
//                tile for S^T, value row t of each block for O^T)
//   warps 8..15  loaders: read the next tile's rows into registers while the
//                current tile computes, then dequantise into shared memory as
//                soon as the tensor core has released each half of the tile
//   warps 1..3   idle
// Pipeline per tile i: loaders fill half A (columns 0..255) and half B (256..511)
// -> QK(i) -> softmax(i) -> PV(i) blocks 0,1 release half A -> PV(i) blocks 2,3
// release half B.  All waits are bounded; on timeout the CTA records
// SMLA_ERR_TIMEOUT in the device status word and leaves through the epilogue.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../include/smla.h"
#include "smla_internal.h"
#include "smla_ptx.cuh"

namespace smla {

__device__ int g_smla_status = 0;

namespace {

constexpr int kTile = 128;                      // tokens per tile (MMA M)
constexpr int kChunkBytes = kTile * 128;        // one 64-column f16 slab of the tile
constexpr int kThreads = 512;
constexpr int kLoaderWarp0 = 8;
constexpr int kLoaderWarps = 8;
constexpr int kSoftWarp0 = 4;
constexpr long long kWaitLimit = 2000000000LL;  // ~1 s of SM clocks
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLazyMax = 8.0f;                // log2 headroom before the max is raised
constexpr int kRowWords = 73;                   // 584 bytes = 73 x 8

enum Bar : int { B_Q = 0, B_FULLA, B_FULLB, B_FREEA, B_FREEB, B_SFULL, B_PFULL, B_ODONE, B_COUNT };

template <int NH>
struct Cfg {
  static constexpr int kQOff = 8 * kChunkBytes;
  static constexpr int kQChunk = NH * 128;
  static constexpr int kPOff = kQOff + 8 * kQChunk;
  static constexpr int kPRow = 2 * NH;
  static constexpr int kPBytes = kTile * kPRow;
  static constexpr int kOnesOff = kPOff + ((kPBytes + 1023) / 1024) * 1024;  // 2 KB, 1024-aligned
  static constexpr int kMiscOff = kOnesOff + 2048;
  static constexpr int kRedOff = kMiscOff;                 // float [4][NH]
  static constexpr int kMOff = kRedOff + 4 * NH * 4;       // float [2][NH] running max (log2)
  static constexpr int kLOff = kMOff + 2 * NH * 4;         // float [NH] final denominators
  static constexpr int kBarOff = kLOff + NH * 4;           // uint64 [B_COUNT]
  static constexpr int kTaddrOff = kBarOff + 8 * B_COUNT;  // uint32
  static constexpr int kAbortOff = kTaddrOff + 4;          // int
  static constexpr int kSmemBytes = kAbortOff + 4 + 1024;  // + alignment slack
  // S^T (NH columns), O^T (4 x NH), per-thread fp32 softmax sums (NH)
  static constexpr uint32_t kTmemCols = 6 * NH <= 64 ? 64 : 6 * NH <= 128 ? 128
                                      : 6 * NH <= 256 ? 256 : 512;
  static constexpr uint32_t kPSwz = NH == 64 ? SWZ_128B : NH == 32 ? SWZ_64B : SWZ_32B;
};

__device__ __forceinline__ void record_status(int code) { atomicCAS(&g_smla_status, 0, code); }

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_shared_v2(uint32_t addr, uint2 v) {
  asm volatile("st.shared.v2.u32 [%0], {%1,%2};" ::"r"(addr), "r"(v.x), "r"(v.y) : "memory");
}
__device__ __forceinline__ uint2 ldg_nc_u2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p));
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}
// Barrier among the 128 softmax threads (id 1); returns true if any thread passed true.
__device__ __forceinline__ bool softmax_bar_or(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred a, b;\n\tsetp.ne.u32 a, %1, 0;\n\t"
      "bar.red.or.pred b, 1, 128, a;\n\tselp.u32 %0, 1, 0, b;\n\t}\n"
      : "=r"(r)
      : "r"(p ? 1u : 0u)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void softmax_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// 2^x on the SFU (ex2.approx, relative error ~2^-22; subnormal results flush to 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// UE8M0 byte -> fp32 2^(e-127) (e = 0 is the fp32 subnormal 2^-127, 0xFF is NaN).
__device__ __forceinline__ float ue8m0_to_f32(uint32_t e) {
  const uint32_t bits = e == 0u ? 0x00400000u : (e == 255u ? 0x7fffffffu : (e << 23));
  return __uint_as_float(bits);
}

// f16 2^(s - 127) in both halves: normal for s in [113, 142], subnormal for
// [103, 112], 0 below (such values are below the f16 range).
__device__ __forceinline__ uint32_t f16_pow2x2(uint32_t s) {
  const uint32_t bits = (s >= 113u && s <= 142u) ? ((s - 112u) << 10)
                        : ((s >= 103u && s < 113u) ? (1u << (s - 103u)) : 0u);
  return bits | (bits << 16);
}
// Two e4m3 bytes -> f16x2 of value * 2^(s - 127): e4m3 -> f16 is exact and the
// product by a power of two is exact while it stays a normal f16.
__device__ __forceinline__ uint32_t dq_pair_f16(uint32_t two, uint32_t m2) {
  uint32_t h2;
  const uint16_t in = static_cast<uint16_t>(two);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h2), "r"(m2));
  return r;
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ bool f16x2_has_inf_or_nan(uint32_t v) {
  return ((v & 0x7c00u) == 0x7c00u) || ((v & 0x7c000000u) == 0x7c000000u);
}
// 8 e4m3 bytes with scale byte s -> 8 f16.  |e4m3| <= 448, so s <= 134 can never
// leave the f16 range; larger scales take a checked path that reports values
// beyond it (SMLA_ERR_RANGE).
__device__ __forceinline__ uint4 dequant8_f16(uint2 w, uint32_t s) {
  uint4 r;
  if (s <= 134u) {
    const uint32_t m = f16_pow2x2(s);
    r.x = dq_pair_f16(w.x & 0xffffu, m);
    r.y = dq_pair_f16(w.x >> 16, m);
    r.z = dq_pair_f16(w.y & 0xffffu, m);
    r.w = dq_pair_f16(w.y >> 16, m);
    return r;
  }
  const float sc = ue8m0_to_f32(s);
  const uint32_t in[4] = {w.x & 0xffffu, w.x >> 16, w.y & 0xffffu, w.y >> 16};
  uint32_t o[4];
  bool bad = false;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t h2;
    const uint16_t v = static_cast<uint16_t>(in[i]);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
    o[i] = pack_f16x2(f.x * sc, f.y * sc);
    bad |= f16x2_has_inf_or_nan(o[i]);
  }
  if (bad) record_status(SMLA_ERR_RANGE);
  r.x = o[0];
  r.y = o[1];
  r.z = o[2];
  r.w = o[3];
  return r;
}
// Four bf16 (rope) -> four f16 (exact for magnitudes in [2^-14, 65504]).
__device__ __forceinline__ uint2 bf16x4_to_f16x4(uint2 v) {
  return make_uint2(pack_f16x2(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u)),
                    pack_f16x2(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u)));
}


// Bounded mbarrier wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_f) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_f) return false;
    if (clock64() - t0 > kWaitLimit) {
      *abort_f = 1;
      record_status(SMLA_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

struct Split {
  int t_begin, t_end, ntiles;
};
__device__ __forceinline__ Split split_range(int topk, int S, int s) {
  const int G = (topk + 15) >> 4;
  const int g0 = static_cast<int>((static_cast<int64_t>(s) * G) / S);
  const int g1 = static_cast<int>((static_cast<int64_t>(s + 1) * G) / S);
  Split r;
  r.t_begin = min(16 * g0, topk);
  r.t_end = min(16 * g1, topk);
  r.ntiles = (r.t_end - r.t_begin + kTile - 1) / kTile;
  return r;
}

// Row id of tile slot `pos`, or -1 if the slot is masked, past the split or out of
// range (the latter is also reported).
__device__ __forceinline__ int64_t slot_row(const int32_t* idx_row, int pos, int t_end,
                                            int64_t num_rows, bool report) {
  if (pos >= t_end) return -1;
  const int idx = __ldg(idx_row + pos);
  if (idx < 0) return -1;
  if (static_cast<int64_t>(idx) >= num_rows) {
    if (report) record_status(SMLA_ERR_INDEX_RANGE);
    return -1;
  }
  return idx;
}

// ---------------------------------------------------------------------------
// Loader: 8 warps, each owns 16 rows of the tile as 4 groups of 4 rows, 8 lanes per
// row, so every load instruction reads 128 contiguous bytes of 4 rows.  A row
// starting at byte address a (8-byte aligned) is read as 16-byte chunks from
// a & ~15: lane q reads chunks q + 8j, j = 0..4 (37 chunks; the last is read as 8
// bytes when the row is 16-byte aligned, so nothing past the row is touched).
// With s = 1 for rows that start 8 bytes into a chunk, chunk c holds row words
// 2c - s and 2c + 1 - s.  Word w < 56: nope columns 8w..8w+7 (scale group w / 8);
// w = 56: the 7 scales and the pad; w = 57..72: rope.  Half A of the tile = words
// 0..31, half B = words 32..72.
// ---------------------------------------------------------------------------
constexpr int kSlots = 5;

struct RowRegs {
  uint4 c[kSlots];
  uint32_t s8a, s8b;   // row alignment shift seen by the half-A / half-B slots
};

__device__ __forceinline__ uint4 ldg_nc_u4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Loads slots [J0, J1) of a row (half A = slots 0, 1; half B = slots 2..4).
template <int J0, int J1>
__device__ __forceinline__ void load_row(RowRegs& R, const uint8_t* row, int q) {
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  if (row == nullptr) {
#pragma unroll
    for (int j = J0; j < J1; ++j) R.c[j] = z;
    if (J0 == 0) R.s8a = 0; else R.s8b = 0;
    return;
  }
  const uintptr_t a = reinterpret_cast<uintptr_t>(row);
  const uint8_t* base = reinterpret_cast<const uint8_t*>(a & ~static_cast<uintptr_t>(15));
  const uint32_t s8 = static_cast<uint32_t>((a >> 3) & 1);
  if (J0 == 0) R.s8a = s8; else R.s8b = s8;
#pragma unroll
  for (int j = J0; j < J1; ++j) {
    const int c = q + 8 * j;
    if (c < 36) {
      R.c[j] = ldg_nc_u4(base + 16 * c);
    } else if (c == 36) {
      if (s8) {
        R.c[j] = ldg_nc_u4(base + 16 * c);
      } else {
        const uint2 v = ldg_nc_u2(base + 16 * c);
        R.c[j] = make_uint4(v.x, v.y, 0u, 0u);
      }
    } else {
      R.c[j] = z;
    }
  }
}

struct Scales {
  uint32_t lo, hi;  // scale bytes of groups 0..3 and 4..6 (byte 7 = pad)
};

// Slow path: one word of any scale byte (also masked rows, whose bytes are 0).
__device__ __forceinline__ void nope_store(uint32_t tile, uint32_t r, int w, uint32_t x, uint32_t y,
                                           const Scales& sc) {
  const int g = w >> 3;
  const uint32_t sb = g < 4 ? (sc.lo >> (8 * g)) & 0xffu : (sc.hi >> (8 * (g - 4))) & 0xffu;
  st_shared_v4(tile + g * kChunkBytes + swz_offset(r, w & 7, 128), dequant8_f16(make_uint2(x, y), sb));
}
// Rope words stay bf16 (the rope slab is multiplied by bf16 q on the tensor core).
__device__ __forceinline__ void rope_store(uint32_t tile, uint32_t r, int w, uint32_t x, uint32_t y) {
  const uint32_t rr = static_cast<uint32_t>(w - 57);   // rope columns 4rr..4rr+3
  st_shared_v2(tile + 7 * kChunkBytes + swz_offset(r, rr >> 1, 128) + (rr & 1) * 8,
               make_uint2(x, y));
}
__device__ __forceinline__ void any_store(uint32_t tile, uint32_t r, int w, uint32_t x, uint32_t y,
                                          const Scales& sc) {
  if (w < 56) nope_store(tile, r, w, x, y, sc);
  else if (w >= 57 && w < kRowWords) rope_store(tile, r, w, x, y);
}

// True if the 7 scale bytes all lie in [113, 134]: then 2^(s - 127) is a normal f16
// and no value can leave the f16 range, so the fast path is exact.  Bytes are
// checked two at a time in 16-bit lanes: +121 carries into bit 8 iff a byte > 134,
// +143 carries iff a byte >= 113.
__device__ __forceinline__ bool scales_fast(uint32_t lo, uint32_t hi) {
  const uint32_t e0 = lo & 0x00ff00ffu, o0 = (lo >> 8) & 0x00ff00ffu;
  const uint32_t e1 = hi & 0x00ff00ffu, o1 = (hi >> 8) & 0x000000ffu;   // pad byte excluded
  const uint32_t over = ((e0 + 0x00790079u) | (o0 + 0x00790079u) | (e1 + 0x00790079u) |
                         (o1 + 0x00000079u)) & 0x01000100u;
  const uint32_t ge = (e0 + 0x008f008fu) & (o0 + 0x008f008fu) & (e1 + 0x008f008fu) &
                      ((o1 + 0x0000008fu) | 0x01000000u);
  return over == 0u && (ge & 0x01000100u) == 0x01000100u;
}
// f16x2 multiplier 2^(s - 127) from byte k of t = s - 112 (bytewise), s in [113, 134]:
// byte k goes to bits 8..15 of both halves, then << 2 puts it in the exponent field.
template <int K>
__device__ __forceinline__ uint32_t mult_from(uint32_t t) {
  constexpr uint32_t kSel = (K << 12) | 0x0400u | (K << 4) | 0x4u;
  uint32_t r;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(r) : "r"(t), "n"(kSel));
  return r << 2;
}
__device__ __forceinline__ uint4 dq8_fast(uint32_t x, uint32_t y, uint32_t m) {
  uint4 v;
  v.x = dq_pair_f16(x & 0xffffu, m);
  v.y = dq_pair_f16(x >> 16, m);
  v.z = dq_pair_f16(y & 0xffffu, m);
  v.w = dq_pair_f16(y >> 16, m);
  return v;
}
__device__ __forceinline__ void sts128_off(uint32_t addr, int off, uint4 v) {
  st_shared_v4(addr + static_cast<uint32_t>(off), v);
}

// Stores half A (half == 0) or half B (half == 1) of one row into the f16 tile.
//
// Lane q of a row holds chunks q + 8j.  With d = 2q - s (s = alignment shift), its
// words are w = d + h + 16j (h = 0: low 8 bytes of the chunk, h = 1: high), so
// for each h the column group is 2j + ((d + h) >> 3) and the 16-byte unit within
// the 128-byte row is (d + h) & 7: one address base per h, plus 32 KB per j.  The
// only irregular word is lane 0 of a row with s = 1, whose (j = 0, h = 0) slot is
// the previous row's tail; it takes word 31 from chunk 16 instead.
__device__ __forceinline__ void store_half(uint32_t tile, const RowRegs& R, uint32_t r, int q,
                                           int lane, int half) {
  // Half A of a tile is converted while slots 2..4 already hold the same tile (they
  // were refilled after the previous tile's half B), so s8a == s8b then.
  const int s8 = static_cast<int>(half == 0 ? R.s8a : R.s8b);
  // the scale word (w = 56) is in chunk 28 = slot 3 of lane 4 of this row
  const uint32_t cand_lo = s8 ? R.c[3].z : R.c[3].x;
  const uint32_t cand_hi = s8 ? R.c[3].w : R.c[3].y;
  const int src = (lane & ~7) | 4;
  Scales sc;
  sc.lo = __shfl_sync(0xffffffffu, cand_lo, src);
  sc.hi = __shfl_sync(0xffffffffu, cand_hi, src);
  const bool masked = (sc.lo | (sc.hi & 0x00ffffffu)) == 0u;   // a zero-filled row
  const int d = 2 * q - s8;
  if (masked || scales_fast(sc.lo, sc.hi)) {
    const uint32_t tlo = masked ? 0u : sc.lo - 0x70707070u;
    const uint32_t thi = masked ? 0u : sc.hi - 0x00707070u;
    const uint32_t rowbase = tile + r * 128u, rx = r & 7u;
    const int b0 = d >> 3, b1 = (d + 1) >> 3;                     // -1, 0 or 1
    const uint32_t base0 = rowbase + static_cast<uint32_t>(b0 * kChunkBytes) +
                           ((static_cast<uint32_t>(d & 7) ^ rx) << 4);
    const uint32_t base1 = rowbase + static_cast<uint32_t>(b1 * kChunkBytes) +
                           ((static_cast<uint32_t>((d + 1) & 7) ^ rx) << 4);
    if (half == 0) {
      const uint32_t m0 = mult_from<0>(tlo), m1 = mult_from<1>(tlo);
      const uint32_t m2 = mult_from<2>(tlo), m3 = mult_from<3>(tlo);
      const bool tail = d < 0;                                      // lane 0, s = 1
      // j = 0
      {
        const uint32_t x = tail ? R.c[2].x : R.c[0].x, y = tail ? R.c[2].y : R.c[0].y;
        const uint32_t m = tail ? m3 : (b0 ? m1 : m0);
        sts128_off(base0, tail ? 4 * kChunkBytes : 0, dq8_fast(x, y, m));
        sts128_off(base1, 0, dq8_fast(R.c[0].z, R.c[0].w, b1 ? m1 : m0));
      }
      // j = 1
      sts128_off(base0, 2 * kChunkBytes, dq8_fast(R.c[1].x, R.c[1].y, b0 < 0 ? m1 : (b0 ? m3 : m2)));
      sts128_off(base1, 2 * kChunkBytes, dq8_fast(R.c[1].z, R.c[1].w, b1 ? m3 : m2));
    } else {
      const uint32_t m4 = mult_from<0>(thi), m5 = mult_from<1>(thi), m6 = mult_from<2>(thi);
      const uint32_t m3 = mult_from<3>(tlo);
      // j = 2: words 31..47 (word 31, the tail lane's, belongs to half A)
      if (d >= 0) sts128_off(base0, 4 * kChunkBytes, dq8_fast(R.c[2].x, R.c[2].y, b0 ? m5 : m4));
      sts128_off(base1, 4 * kChunkBytes, dq8_fast(R.c[2].z, R.c[2].w, b1 ? m5 : m4));
      // j = 3: words 47..63: nope while group 2j + b <= 6, then the scale word, then rope
      {
        const int w0 = d + 48, w1 = d + 49;
        if (w0 < 56) sts128_off(base0, 6 * kChunkBytes, dq8_fast(R.c[3].x, R.c[3].y, b0 < 0 ? m5 : m6));
        else if (w0 >= 57) rope_store(tile, r, w0, R.c[3].x, R.c[3].y);
        if (w1 < 56) sts128_off(base1, 6 * kChunkBytes, dq8_fast(R.c[3].z, R.c[3].w, m6));
        else if (w1 >= 57) rope_store(tile, r, w1, R.c[3].z, R.c[3].w);
      }
      // j = 4: rope words 63..73
      if (q <= 4) {
        const int w0 = d + 64;
        rope_store(tile, r, w0, R.c[4].x, R.c[4].y);
        if (w0 + 1 < kRowWords) rope_store(tile, r, w0 + 1, R.c[4].z, R.c[4].w);
      }
      (void)m3;
    }
    return;
  }
  // Slow path: a scale byte outside [113, 134] somewhere in the row.
  if (half == 0) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {          // chunks 0..15: words -1..31
      const int w0 = 2 * (q + 8 * j) - s8;
      if (w0 >= 0) nope_store(tile, r, w0, R.c[j].x, R.c[j].y, sc);
      nope_store(tile, r, w0 + 1, R.c[j].z, R.c[j].w, sc);
    }
    if (q == 0 && s8) nope_store(tile, r, 31, R.c[2].x, R.c[2].y, sc);   // chunk 16, low word
  } else {
    {                                      // chunks 16..23: words 31..47
      const int w0 = 2 * (q + 16) - s8;
      if (w0 >= 32) nope_store(tile, r, w0, R.c[2].x, R.c[2].y, sc);
      nope_store(tile, r, w0 + 1, R.c[2].z, R.c[2].w, sc);
    }
    {                                      // chunks 24..31: words 47..63
      const int w0 = 2 * (q + 24) - s8;
      any_store(tile, r, w0, R.c[3].x, R.c[3].y, sc);
      any_store(tile, r, w0 + 1, R.c[3].z, R.c[3].w, sc);
    }
    if (q <= 4) {                          // chunks 32..36: rope words 63..73
      const int w0 = 2 * (q + 32) - s8;
      rope_store(tile, r, w0, R.c[4].x, R.c[4].y);
      if (w0 + 1 < kRowWords) rope_store(tile, r, w0 + 1, R.c[4].z, R.c[4].w);
    }
  }
}

template <int NH>
__global__ void __launch_bounds__(kThreads, 1)
    split_kernel(const uint16_t* __restrict__ q, const uint8_t* __restrict__ kv,
                 const int32_t* __restrict__ indices, float* __restrict__ o_part,
                 float* __restrict__ lse_part, int H, int topk, int S, int64_t num_rows,
                 int64_t stride, float scale_log2) {
  using C = Cfg<NH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int s = blockIdx.x, h0 = blockIdx.y * NH, b = blockIdx.z;
  const Split sp = split_range(topk, S, s);
  const int32_t* idx_row = indices + static_cast<int64_t>(b) * topk;

  float* red = reinterpret_cast<float*>(smem + C::kRedOff);
  float* mbuf = reinterpret_cast<float*>(smem + C::kMOff);
  float* lfin = reinterpret_cast<float*>(smem + C::kLOff);
  const uint32_t bars = sbase + C::kBarOff;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  volatile uint32_t* taddr_s = reinterpret_cast<volatile uint32_t*>(smem + C::kTaddrOff);
  volatile int* abort_f = reinterpret_cast<volatile int*>(smem + C::kAbortOff);

  if (tid == 0) {
    mbar_init(bar(B_Q), kLoaderWarps);
    mbar_init(bar(B_FULLA), kLoaderWarps);
    mbar_init(bar(B_FULLB), kLoaderWarps);
    mbar_init(bar(B_FREEA), 1);
    mbar_init(bar(B_FREEB), 1);
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_PFULL), 4);
    mbar_init(bar(B_ODONE), 1);
    *abort_f = 0;
    fence_mbar_init();
  }
  if (tid < 2 * NH) mbuf[tid] = -INFINITY;
  if (warp == 0) {
    tmem_alloc(sbase + C::kTaddrOff, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *taddr_s;
  const uint32_t tS = tmem;        // S^T: columns [0, NH)
  const uint32_t tO = tmem + NH;   // O^T block mb: columns [NH + mb*NH, NH + (mb+1)*NH)
  const uint32_t tL = tmem + 5 * NH;  // this thread's partial sum_t P[t, h] in fp32

  // Registers: warpgroup 0 (MMA issuer + idle warps) gives up registers so that the
  // softmax and loader warpgroups can hold a tile of raw rows and a row of scores.
  // Each role runs entirely inside its own branch (no join before the end).
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 56;" ::: "memory");
    // ===================== MMA issuer =====================
    if (warp == 0 && lane == 0 && sp.ntiles > 0) {
      constexpr uint32_t kIdescQK = idesc_f16(128, NH, false, false);
      constexpr uint32_t kIdescQKRope = idesc_bf16(128, NH, false, false);
      constexpr uint32_t kIdescPV = idesc_f16(128, NH, true, true);
      bool ok = wait_or_abort(bar(B_Q), 0, abort_f);
      // Base descriptors; moving a start address by X bytes adds X >> 4 to the low
      // field (addresses stay below 256 KB, so the 14-bit field never carries).
      const uint64_t dK = smem_desc(sbase, 16, 1024, SWZ_128B);
      const uint64_t dQ = smem_desc(sbase + C::kQOff, 16, 1024, SWZ_128B);
      const uint64_t dV = smem_desc(sbase, kChunkBytes, 1024, SWZ_128B);
      // block 3 pairs columns 384..447 with the constant block: leading offset
      // (ones - a_start) shrinks by 2048 bytes per K step
      const uint64_t dV3 = smem_desc(sbase + 6 * kChunkBytes, C::kOnesOff - 6 * kChunkBytes, 1024,
                                     SWZ_128B);
      const uint64_t dP = smem_desc(sbase + C::kPOff, 8 * C::kPRow, 8 * C::kPRow, C::kPSwz);
      for (int it = 0; it < sp.ntiles && ok; ++it) {
        const uint32_t par = it & 1;
        ok = wait_or_abort(bar(B_FULLA), par, abort_f);
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int j = 0; j < 8; ++j) {
          if (j == 4) {
            ok = wait_or_abort(bar(B_FULLB), par, abort_f);
            if (!ok) break;
            tc_fence_after();
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            mma_f16_ss(tS, dK + static_cast<uint64_t>((j * kChunkBytes + k * 32) >> 4),
                       dQ + static_cast<uint64_t>((j * C::kQChunk + k * 32) >> 4),
                       j == 7 ? kIdescQKRope : kIdescQK, (j | k) != 0);
          }
        }
        if (!ok) break;
        mma_commit(bar(B_SFULL));
        ok = wait_or_abort(bar(B_PFULL), par, abort_f);
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint64_t a = mb < 3
                ? dV + static_cast<uint64_t>((2 * mb * kChunkBytes + ks * 2048) >> 4)
                : dV3 + static_cast<uint64_t>(ks * 128) - (static_cast<uint64_t>(ks * 128) << 16);
            mma_f16_ss(tO + mb * NH, a, dP + static_cast<uint64_t>((ks * 16 * C::kPRow) >> 4),
                        kIdescPV, (it > 0 || ks > 0) ? 1u : 0u);
          }
          if (mb == 1) mma_commit(bar(B_FREEA));
        }
        mma_commit(bar(B_FREEB));
      }
      mma_commit(bar(B_ODONE));
    }
  } else if (warp >= kLoaderWarp0) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 144;" ::: "memory");
    // ===================== loaders =====================
    const int lw = warp - kLoaderWarp0;          // 0..7
    const int lt = tid - kLoaderWarp0 * 32;      // 0..255
    const uint32_t tile = sbase;
    // Q rows h0..h0+NH-1 -> 8 K-major SW128 slabs; the constant ones block.
    bool q_bad = false;
    for (int u = lt; u < NH * 64; u += kLoaderWarps * 32) {
      const int r = u >> 6, cu = u & 63;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(
          q + (static_cast<int64_t>(b) * H + h0 + r) * kQkDim + cu * 8));
      uint4 o = v;                       // the rope columns (slab 7) stay bf16
      if (cu < 56) {
        const uint2 lo = bf16x4_to_f16x4(make_uint2(v.x, v.y));
        const uint2 hi = bf16x4_to_f16x4(make_uint2(v.z, v.w));
        q_bad |= f16x2_has_inf_or_nan(lo.x) | f16x2_has_inf_or_nan(lo.y) |
                 f16x2_has_inf_or_nan(hi.x) | f16x2_has_inf_or_nan(hi.y);
        o = make_uint4(lo.x, lo.y, hi.x, hi.y);
      }
      st_shared_v4(sbase + C::kQOff + (cu >> 3) * C::kQChunk + swz_offset(r, cu & 7, 128), o);
    }
    if (q_bad) record_status(SMLA_ERR_RANGE);
    if (lt < 128) {   // 16 rows x 8 units of 16 B
      const uint32_t r = lt >> 3, unit = lt & 7;
      const uint4 v = make_uint4(unit == 0 ? 0x3C00u : 0u, 0u, 0u, 0u);   // f16 1.0
      st_shared_v4(sbase + C::kOnesOff + (r >> 3) * 1024 + swz_offset(r & 7, unit, 128), v);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(B_Q));

    const int q8 = lane & 7;                     // chunk lane within the row
    const int rsub = lane >> 3;                  // row within a group of 4
    RowRegs R[4];
    int rows_next[4];
    auto load_idx = [&](int it, int* out) {
#pragma unroll
      for (int g = 0; g < 4; ++g)
        out[g] = static_cast<int>(slot_row(idx_row, sp.t_begin + it * kTile + lw * 16 + 4 * g + rsub,
                                           sp.t_end, num_rows, q8 == 0));
    };
    // Half A (slots 0, 1) and half B (slots 2..4) of the staged rows are refilled
    // separately, each right after it has been converted, so the loads for the
    // next tile are in flight for a whole tile period.
    auto fetch_a = [&](const int* rows) {
#pragma unroll
      for (int g = 0; g < 4; ++g)
        load_row<0, 2>(R[g], rows[g] >= 0 ? kv + static_cast<int64_t>(rows[g]) * stride : nullptr, q8);
    };
    auto fetch_b = [&](const int* rows) {
#pragma unroll
      for (int g = 0; g < 4; ++g)
        load_row<2, kSlots>(R[g], rows[g] >= 0 ? kv + static_cast<int64_t>(rows[g]) * stride : nullptr,
                            q8);
    };
    if (sp.ntiles > 0) {
      int rows0[4];
      load_idx(0, rows0);
      fetch_a(rows0);
      fetch_b(rows0);
      if (sp.ntiles > 1) load_idx(1, rows_next);
    }
    for (int it = 0; it < sp.ntiles; ++it) {
      const uint32_t pprev = (it - 1) & 1;
      if (it > 0 && !__all_sync(0xffffffffu, wait_or_abort(bar(B_FREEA), pprev, abort_f))) break;
#pragma unroll
      for (int g = 0; g < 4; ++g) store_half(tile, R[g], lw * 16 + 4 * g + rsub, q8, lane, 0);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_FULLA));
      if (it + 1 < sp.ntiles) fetch_a(rows_next);
      if (it > 0 && !__all_sync(0xffffffffu, wait_or_abort(bar(B_FREEB), pprev, abort_f))) break;
#pragma unroll
      for (int g = 0; g < 4; ++g) store_half(tile, R[g], lw * 16 + 4 * g + rsub, q8, lane, 1);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_FULLB));
      if (it + 1 < sp.ntiles) {
        fetch_b(rows_next);
        if (it + 2 < sp.ntiles) load_idx(it + 2, rows_next);
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 168;" ::: "memory");
    // ===================== softmax + epilogue =====================
    const int st = tid - kSoftWarp0 * 32;        // 0..127 = TMEM lane
    const int sw = warp - kSoftWarp0;            // 0..3 = lane quarter
    const uint32_t lane_base = static_cast<uint32_t>(sw * 32) << 16;
    int cur = 0;                                 // which half of mbuf holds the running max
    bool ok = true;
    // validity of this thread's token, read one tile ahead of its use
    bool valid_next = sp.ntiles > 0 &&
        slot_row(idx_row, sp.t_begin + st, sp.t_end, num_rows, false) >= 0;
    for (int it = 0; it < sp.ntiles; ++it) {
      const bool valid = valid_next;
      if (it + 1 < sp.ntiles)
        valid_next = slot_row(idx_row, sp.t_begin + (it + 1) * kTile + st, sp.t_end, num_rows,
                              false) >= 0;
      ok = wait_or_abort(bar(B_SFULL), it & 1, abort_f);
      if (softmax_bar_or(!ok)) {   // leave together
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[NH];
#pragma unroll
      for (int c = 0; c < NH / 16; ++c) tmem_ld16(tS + lane_base + 16 * c, sv + 16 * c);
      tmem_wait_ld();
      const float* m_old = mbuf + cur * NH;
      float ex = -INFINITY;
#pragma unroll
      for (int h4 = 0; h4 < NH / 4; ++h4) {
        const float4 mo = reinterpret_cast<const float4*>(m_old)[h4];
        const float mv[4] = {mo.x, mo.y, mo.z, mo.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int h = 4 * h4 + i;
          sv[h] = valid ? sv[h] * scale_log2 : -INFINITY;
          ex = fmaxf(ex, sv[h] - mv[i]);   // -inf - m and NaN-free: sv = -inf only if invalid
        }
      }
      if (!valid) ex = -INFINITY;
      if (softmax_bar_or(ex > kLazyMax)) {
        // Raise the running max to the exact tile max and rescale O (and with it
        // the denominator row) by 2^(m_old - m_new).
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          const float m = warp_max(sv[h]);
          if (lane == (h & 31)) red[sw * NH + h] = m;
        }
        softmax_bar();
        float* m_new = mbuf + (cur ^ 1) * NH;
        if (st < NH) {
          const float mt = fmaxf(fmaxf(red[st], red[NH + st]), fmaxf(red[2 * NH + st], red[3 * NH + st]));
          m_new[st] = fmaxf(m_old[st], mt);
        }
        softmax_bar();
        if (it > 0) {
          // 4 O^T blocks, then the fp32 partial sums (block 4 = tL)
#pragma unroll 1
          for (int mb = 0; mb < 5; ++mb) {
#pragma unroll
            for (int c = 0; c < NH / 16; ++c) {
              float o[16];
              tmem_ld16(tO + lane_base + mb * NH + 16 * c, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int h = 16 * c + i;
                const float mn = m_new[h];
                o[i] *= (mn == -INFINITY) ? 1.f : exp2f(m_old[h] - mn);
              }
              tmem_st16(tO + lane_base + mb * NH + 16 * c, o);
            }
          }
          tmem_wait_st();
        }
        cur ^= 1;
      }
      const float* m = mbuf + cur * NH;
#pragma unroll
      for (int h4 = 0; h4 < NH / 4; ++h4) {
        const float4 mo = reinterpret_cast<const float4*>(m)[h4];
        const float mv[4] = {mo.x, mo.y, mo.z, mo.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int h = 4 * h4 + i;
          // sv = -inf (masked) gives 0; m = -inf only while every score so far is
          // masked, and then sv is -inf too
          sv[h] = (sv[h] == -INFINITY) ? 0.f : fast_exp2(sv[h] - mv[i]);
        }
      }
#pragma unroll
      for (int u = 0; u < NH / 8; ++u) {
        uint4 v;
        v.x = pack_f16x2(sv[8 * u + 0], sv[8 * u + 1]);
        v.y = pack_f16x2(sv[8 * u + 2], sv[8 * u + 3]);
        v.z = pack_f16x2(sv[8 * u + 4], sv[8 * u + 5]);
        v.w = pack_f16x2(sv[8 * u + 6], sv[8 * u + 7]);
        st_shared_v4(sbase + C::kPOff + swz_offset(st, u, C::kPRow), v);
      }
      // unrounded sums for the log-sum-exp
#pragma unroll
      for (int c = 0; c < NH / 16; ++c) {
        float lp[16];
        if (it > 0) {
          tmem_ld16(tL + lane_base + 16 * c, lp);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) lp[i] += sv[16 * c + i];
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) lp[i] = sv[16 * c + i];
        }
        tmem_st16(tL + lane_base + 16 * c, lp);
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PFULL));
    }
    // ---- epilogue ----
    const bool have_o = !softmax_bar_or(
        !(sp.ntiles > 0 && ok && wait_or_abort(bar(B_ODONE), 0, abort_f)));
    if (have_o) tc_fence_after();
    if (have_o && sw == 2) {
      // row 448 of block 3 (TMEM lane 64, lane 0 of this warp) = sum_t P[t] per head
#pragma unroll
      for (int c = 0; c < NH / 16; ++c) {
        float o[16];
        tmem_ld16(tO + lane_base + 3 * NH + 16 * c, o);
        tmem_wait_ld();
        if (lane == 0) {
#pragma unroll
          for (int i = 0; i < 16; ++i) lfin[16 * c + i] = o[i];
        }
      }
    } else if (!have_o && st < NH) {
      lfin[st] = 0.f;
    }
    // sum the per-thread fp32 partials over the 128 threads for the LSE
    if (have_o) {
#pragma unroll
      for (int c = 0; c < NH / 16; ++c) {
        float lp[16];
        tmem_ld16(tL + lane_base + 16 * c, lp);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float v = lp[i];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == ((16 * c + i) & 31)) red[sw * NH + 16 * c + i] = v;
        }
      }
    }
    softmax_bar();
    const float* m = mbuf + cur * NH;
    if (st < NH) {
      const float lt = have_o ? (red[st] + red[NH + st]) + (red[2 * NH + st] + red[3 * NH + st]) : 0.f;
      const float lse = lt > 0.f ? (m[st] + log2f(lt)) * kLn2 : -INFINITY;
      lse_part[(static_cast<int64_t>(b) * H + h0 + st) * S + s] = lse;
    }
#pragma unroll 1
    for (int mb = 0; mb < 4; ++mb) {
      const int d = mb * 128 + st;
#pragma unroll
      for (int c = 0; c < NH / 16; ++c) {
        float o[16];
        if (have_o) {
          tmem_ld16(tO + lane_base + mb * NH + 16 * c, o);
          tmem_wait_ld();
        }
        if (d < kNope) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int h = 16 * c + i;
            const float lt = lfin[h];
            const float val = (have_o && lt > 0.f) ? o[i] / lt : 0.f;
            o_part[((static_cast<int64_t>(b) * H + h0 + h) * S + s) * kNope + d] = val;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int NH>
cudaError_t launch_split_t(const void* q, const void* kv, const int32_t* indices, float* o_part,
                           float* lse_part, int B, int H, int topk, int S, int64_t num_rows,
                           int64_t stride, float softmax_scale, cudaStream_t stream) {
  using C = Cfg<NH>;
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(split_kernel<NH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const dim3 grid(S, H / NH, B);
  const float scale_log2 = softmax_scale * 1.4426950408889634f;
  split_kernel<NH><<<grid, kThreads, C::kSmemBytes, stream>>>(
      static_cast<const uint16_t*>(q), static_cast<const uint8_t*>(kv), indices, o_part, lse_part,
      H, topk, S, num_rows, stride, scale_log2);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_split(const void* q, const void* kv, const int32_t* indices, float* o_part,
                         float* lse_part, int B, int H, int topk, int S, int64_t num_rows,
                         int64_t stride, float softmax_scale, cudaStream_t stream) {
  switch (H) {
    case 16:
      return launch_split_t<16>(q, kv, indices, o_part, lse_part, B, H, topk, S, num_rows, stride,
                                softmax_scale, stream);
    case 32:
      return launch_split_t<32>(q, kv, indices, o_part, lse_part, B, H, topk, S, num_rows, stride,
                                softmax_scale, stream);
    default:  // 64 and 128 (two head groups of 64)
      return launch_split_t<64>(q, kv, indices, o_part, lse_part, B, H, topk, S, num_rows, stride,
                                softmax_scale, stream);
  }
}

cudaError_t read_device_status(int32_t* status, bool clear) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_smla_status, sizeof(int));
  if (e != cudaSuccess) return e;
  *status = v;
  if (clear) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_smla_status, &zero, sizeof(int));
  }
  return e;
}

}  // namespace smla
