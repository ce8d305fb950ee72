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
// Blackwell").  Launched as thread-block clusters of the S splits of a (query, head
// group), the CTAs then also merge the splits (the combine step) after a cluster
// barrier, each for a slice of the heads, and write the final out and lse.
//
// Design (sm_103a).  Tokens are the MMA's M dimension, so every MMA is a full
// 128-row tcgen05 instruction even with 16 heads.  The nope operands are f16 (fp32
// accumulation): e4m3 -> f16 is one conversion and the power-of-two group scale
// one f16x2 multiply, and the attention weights P keep 11 significant bits.  Nope
// values must lie in the f16 range (the kernel reports SMLA_ERR_RANGE otherwise).
// The rope columns stay bf16 and are multiplied by bf16 q into the same fp32
// accumulator.  One tile in shared memory serves as K (K-major view) for the scores
// and as V^T (MN-major view) for the output.  The 448-wide value product runs as
// four 128-row blocks; the 4th block pairs value columns 384..447 with a constant
// block whose first column is 1, so output row 448 of that block is sum_t P[t], the
// softmax denominator, accumulated and rescaled by the tensor core together with O.
//
// Warp roles (640 threads):
//   warp 0       allocates tensor memory and issues every tcgen05.mma (one lane)
//   warps 1..3   idle
//   warps 4..19  16 workers.  Each owns 8 rows of the tile for loading and
//                dequantising, and 32 tokens x NH/4 heads of the tile's scores for
//                the softmax (TMEM lane quarter = warp % 4).
// The tile is released in the order the value product finishes with it, and
// refilled in the same order: the rope slab as soon as the scores are computed,
// then the slab pairs (0,1), (2,3), (4,5) and slab 6 as the four value blocks
// complete.  The score MMAs of the next tile start on each part as soon as it is
// written, so the tensor pipe stays busy while the workers convert.  The rows of
// the tile after next are read into registers right after each part is converted.
// All waits are bounded; on timeout the CTA records SMLA_ERR_TIMEOUT in the device
// status word and leaves through the epilogue.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "../../include/smla.h"
#include "smla_internal.h"
#include "smla_ptx.cuh"

namespace smla {

__device__ int g_smla_status = 0;

namespace {

constexpr int kTile = 128;                      // tokens per tile (MMA M)
constexpr int kSlabBytes = kTile * 128;         // one 64-column 16-bit slab of the tile
constexpr int kWorkerWarp0 = 4;
constexpr int kWorkerWarps = 16;
constexpr int kWorkers = kWorkerWarps * 32;     // 512
constexpr int kThreads = (kWorkerWarp0 + kWorkerWarps) * 32;   // 640
// Register split (setmaxnreg): the kernel is launched with kLaunchRegs per thread
// (65536 / 640 rounded down to a multiple of 8); warpgroup 0 gives registers back
// and the four worker warpgroups take them.
constexpr int kLaunchRegs = 96;
constexpr long long kWaitLimit = 2000000000LL;  // ~1 s of SM clocks
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLazyMax = 8.0f;                // log2 headroom before the max is raised
constexpr int kMaxCluster = 8;                  // splits merged on chip (portable cluster size)
enum : int { kSplitOnly = 0, kMergeL2 = 1 };

// mbarriers.  FR: rope slab written; F0..F3: slab pairs (0,1), (2,3), (4,5) and slab
// 6 written; E0..E3: value block 0..3 done (its slabs may be overwritten); SFULL:
// scores in TMEM; PFULL: P in shared memory; ODONE: all value products done; QRAW:
// the bf16 q rows copied into the (not yet used) tile area.
enum Bar : int {
  B_FR = 0, B_F0, B_F1, B_F2, B_F3, B_E0, B_E1, B_E2, B_E3, B_SFULL, B_PFULL, B_ODONE, B_QRAW,
  B_COUNT
};

template <int NH>
struct Cfg {
  static constexpr int kHW = NH / 4;                      // heads per worker in the softmax
  static constexpr int kQOff = 8 * kSlabBytes;
  static constexpr int kQChunk = NH * 128;
  static constexpr int kPOff = kQOff + 8 * kQChunk;
  static constexpr int kPRow = 2 * NH;
  static constexpr int kPBytes = kTile * kPRow;
  static constexpr int kOnesOff = kPOff + ((kPBytes + 1023) / 1024) * 1024;  // 2 KB, 1024-aligned
  static constexpr int kMiscOff = kOnesOff + 2048;
  static constexpr int kRedOff = kMiscOff;                 // float [4][NH]
  static constexpr int kMOff = kRedOff + 4 * NH * 4;       // float [2][NH] running max (log2)
  static constexpr int kLOff = kMOff + 2 * NH * 4;         // float [NH] denominators
  static constexpr int kBarOff = kLOff + NH * 4;           // uint64 [B_COUNT]
  static constexpr int kTaddrOff = kBarOff + 8 * B_COUNT;  // uint32
  static constexpr int kAbortOff = kTaddrOff + 4;          // int
  static constexpr int kSmemBytes = kAbortOff + 4 + 1024;  // + alignment slack
  // S^T (NH columns) and O^T (4 x NH)
  static constexpr uint32_t kTmemCols = 5 * NH <= 64 ? 64 : 5 * NH <= 128 ? 128
                                      : 5 * NH <= 256 ? 256 : 512;
  static constexpr uint32_t kPSwz = NH == 64 ? SWZ_128B : NH == 32 ? SWZ_64B : SWZ_32B;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  // registers per thread of warpgroup 0 (MMA issuer) and of the workers
  static constexpr int kRegsWg0 = NH == 16 ? 40 : 32;
  static constexpr int kRegsWorker = NH == 16 ? 104 : 112;
  static_assert(kRegsWg0 * 128 + kRegsWorker * kWorkers <= kLaunchRegs * kThreads,
                "register split exceeds the launch allocation");
};

__device__ __forceinline__ void record_status(int code) { atomicCAS(&g_smla_status, 0, code); }

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ void st_shared_v2(uint32_t addr, uint2 v) {
  asm volatile("st.shared.v2.u32 [%0], {%1,%2};" ::"r"(addr), "r"(v.x), "r"(v.y) : "memory");
}
__device__ __forceinline__ uint4 ldg_nc_u4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
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
// Barrier among the 512 worker threads (id 1); returns true if any thread passed true.
__device__ __forceinline__ bool workers_bar_or(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred a, b;\n\tsetp.ne.u32 a, %1, 0;\n\t"
      "bar.red.or.pred b, 1, 512, a;\n\tselp.u32 %0, 1, 0, b;\n\t}\n"
      : "=r"(r)
      : "r"(p ? 1u : 0u)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void workers_bar() { asm volatile("bar.sync 1, 512;" ::: "memory"); }
// Barrier among the 512 workers; returns true if every thread passed true.
__device__ __forceinline__ bool workers_bar_and(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred a, b;\n\tsetp.ne.u32 a, %1, 0;\n\t"
      "bar.red.and.pred b, 1, 512, a;\n\tselp.u32 %0, 1, 0, b;\n\t}\n"
      : "=r"(r)
      : "r"(p ? 1u : 0u)
      : "memory");
  return r != 0;
}

// Barrier over every thread of every CTA of the thread-block cluster, ordering their
// memory accesses (release before, acquire after).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// 2^x on the SFU (ex2.approx, relative error ~2^-22; subnormal results flush to 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// TMEM loads/stores of N consecutive 32-bit columns, 32 lanes (32x32b shape): thread
// i of the warp holds lane (warp quarter * 32 + i).
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float* v) {
  static_assert(N == 4 || N == 8 || N == 16, "width");
  if constexpr (N == 16) {
    tmem_ld16(taddr, v);
  } else if constexpr (N == 8) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
  } else {
    uint32_t r[4];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr)
                 : "memory");
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
  }
}
template <int N>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const float* v) {
  static_assert(N == 4 || N == 8 || N == 16, "width");
  if constexpr (N == 16) {
    tmem_st16(taddr, v);
  } else if constexpr (N == 8) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(
                     taddr),
                 "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
                 "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
                 "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                 "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
                 : "memory");
  } else {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr),
                 "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
                 "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3]))
                 : "memory");
  }
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
// 8 e4m3 bytes with scale byte s -> 8 f16, any s.  |e4m3| <= 448, so s <= 134 can
// never leave the f16 range; larger scales take a checked path that reports values
// beyond it (SMLA_ERR_RANGE).
__device__ __forceinline__ uint4 dequant8_f16(uint32_t x, uint32_t y, uint32_t s) {
  uint4 r;
  if (s <= 134u) {
    const uint32_t m = f16_pow2x2(s);
    r.x = dq_pair_f16(x & 0xffffu, m);
    r.y = dq_pair_f16(x >> 16, m);
    r.z = dq_pair_f16(y & 0xffffu, m);
    r.w = dq_pair_f16(y >> 16, m);
    return r;
  }
  const float sc = ue8m0_to_f32(s);
  const uint32_t in[4] = {x & 0xffffu, x >> 16, y & 0xffffu, y >> 16};
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
// 8 e4m3 bytes times the f16x2 power of two m (fast path: exact, in range).
__device__ __forceinline__ uint4 dq8_fast(uint32_t x, uint32_t y, uint32_t m) {
  uint4 v;
  v.x = dq_pair_f16(x & 0xffffu, m);
  v.y = dq_pair_f16(x >> 16, m);
  v.z = dq_pair_f16(y & 0xffffu, m);
  v.w = dq_pair_f16(y >> 16, m);
  return v;
}
// Four bf16 (q nope) -> four f16 (exact for magnitudes in [2^-14, 65504]).
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

// Wait of all 512 workers on an mbarrier phase: one thread polls it (bounded), the
// others sleep on a named barrier, so the waiting warps take no issue slots and no
// shared-memory bandwidth from the tensor core.  Every thread gets the same verdict.
__device__ __forceinline__ bool workers_wait(uint32_t bar, uint32_t parity, volatile int* abort_f,
                                             bool poller) {
  bool ok = true;
  if (poller) ok = wait_or_abort(bar, parity, abort_f);
  __syncwarp();
  return workers_bar_and(ok);
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

// Index of slot `pos` as stored (-1 past the split).  Loaded a tile ahead of its
// use; nothing waits for it until then.
__device__ __forceinline__ int raw_idx(const int32_t* idx_row, int pos, int t_end) {
  return pos < t_end ? __ldg(idx_row + pos) : -1;
}
// A stored index names a row (out-of-range ones are masked and reported).
__device__ __forceinline__ bool idx_ok(int idx, int64_t num_rows, bool report) {
  if (idx < 0) return false;
  if (static_cast<int64_t>(idx) >= num_rows) {
    if (report) record_status(SMLA_ERR_INDEX_RANGE);
    return false;
  }
  return true;
}

// ---------------------------------------------------------------------------
// Row loading.  A row starting at byte address a (8-byte aligned) is read as 16-byte
// chunks from a & ~15; s = (a >> 3) & 1 is its shift in that grid.  8 lanes share a
// row, lane q reading chunks q + 8j into register slot j (j = 0..4; 37 chunks, the
// last read as 8 bytes when s = 0, so nothing past the row is touched).  Chunk c
// holds row words 2c - s and 2c + 1 - s (a word = 8 bytes).  Word w < 56: nope
// columns 8w..8w+7 (scale group w / 8); w = 56: the 7 scales and the pad; w =
// 57..72: rope.
//
// Lane layout within a warp (4 rows): lane = qq + 4*rowbit + 8*qhi + 16*pairsel,
// q = qq + 4*qhi, row = 2*pairsel + rowbit.  A 16-byte shared store is served in
// four phases of 8 consecutive lanes; each phase then holds 4 lanes of an even row
// and 4 lanes of the odd row after it.
//
// Dequantising word pair j (words 16j..16j+15 = slabs 2j and 2j+1): lane q stores
// its even word 16j + 2q (unit 2q & 7 of slab 2j + q/4) and one odd word: 16j + 2q
// + 1 if s = 0, else 16j + 2q - 1 (16j + 15, from slot j + 1, for q = 0).  Units
// are XOR-swizzled with row & 7, so in every phase the 8 stores hit 8 distinct
// 16-byte units: the even row's even words and the odd row's even words land on
// units of opposite parity, and likewise for odd words.
// ---------------------------------------------------------------------------
constexpr int kSlots = 5;

template <int J>
__device__ __forceinline__ uint4 load_slot(const uint8_t* base, int q, bool s) {
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  if (base == nullptr) return z;
  const int c = q + 8 * J;
  if (J < 4 || c < 36) return ldg_nc_u4(base + 16 * c);
  if (c == 36) {
    if (s) return ldg_nc_u4(base + 16 * c);
    const uint2 v = ldg_nc_u2(base + 16 * c);
    return make_uint4(v.x, v.y, 0u, 0u);
  }
  return z;
}

// prmt selector that puts byte k of the first operand in bits 8..15 of both halves
// (the other bytes come from the zero second operand).
__device__ __forceinline__ uint32_t byte_sel(uint32_t k) { return (k << 12) | 0x0400u | (k << 4) | 4u; }
__device__ __forceinline__ uint32_t prmt0(uint32_t a, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(r) : "r"(a), "r"(sel));
  return r;
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
__device__ __forceinline__ uint32_t scale_byte(uint32_t lo, uint32_t hi, int g) {
  return ((g < 4 ? lo : hi) >> (8 * (g & 3))) & 0xffu;
}

// Per-row values for dequantising one tile's row.
struct RowPrep {
  uint32_t lo, hi;          // raw scale words (bytes 0..6 = scales, 7 = pad)
  uint32_t tlo, thi;        // (scale - 112) << 2 per byte, 0 for a zero-filled row
  uint32_t sel_o0, sel_o1;  // byte selectors of the odd word's group (pairs 0,2 / 1,3)
  uint32_t base_o;          // shared address of the odd word of pair 0
};

// MODE kSplitOnly: writes the split's normalised partial O and lse (o_part, lse_part).
// MODE kMergeL2: launched as clusters of the S splits of one (query, head group); each
//   split writes its partials as above, then after a cluster barrier each CTA merges
//   a slice of the heads from the (L2-resident) partials of all the splits and writes
//   the final bf16 out and lse: the split-K combine without a second launch.
template <int NH, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    split_kernel(const uint16_t* __restrict__ q, const uint8_t* __restrict__ kv,
                 const int32_t* __restrict__ indices, float* __restrict__ o_part,
                 float* __restrict__ lse_part, __nv_bfloat16* __restrict__ out,
                 float* __restrict__ lse_out, int H, int topk, int S, int64_t num_rows,
                 int64_t stride, float scale_log2) {
  using C = Cfg<NH>;
  constexpr int HW = C::kHW;
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
    for (int i = B_FR; i <= B_F3; ++i) mbar_init(bar(i), kWorkerWarps);
    for (int i = B_E0; i <= B_E3; ++i) mbar_init(bar(i), 1);
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_PFULL), kWorkerWarps);
    mbar_init(bar(B_ODONE), 1);
    mbar_init(bar(B_QRAW), 1);
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
  // Nothing above touches global memory: under programmatic launch the previous
  // kernel in the stream may run until here.
  grid_dep_wait();
  grid_dep_launch();
  const uint32_t tS = tmem;        // S^T: columns [0, NH)
  const uint32_t tO = tmem + NH;   // O^T block mb: columns [NH + mb*NH, NH + (mb+1)*NH)

  if (warp < kWorkerWarp0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::kRegsWg0) : "memory");
    // ===================== MMA issuer =====================
    if (warp == 0 && lane == 0 && sp.ntiles > 0) {
      // The bf16 q rows h0..h0+NH-1 (contiguous, NH KB) into the still unused tile
      // area, where the workers convert them into the Q operand.
      {
        const uint8_t* src =
            reinterpret_cast<const uint8_t*>(q + (static_cast<int64_t>(b) * H + h0) * kQkDim);
        mbar_arrive_expect_tx(bar(B_QRAW), NH * 1024);
#pragma unroll
        for (int k = 0; k < NH / 16; ++k)
          bulk_g2s(sbase + k * 16384, src + k * 16384, 16384, bar(B_QRAW));
      }
      constexpr uint32_t kIdescQK = idesc_f16(128, NH, false, false);
      constexpr uint32_t kIdescQKRope = idesc_bf16(128, NH, false, false);
      constexpr uint32_t kIdescPV = idesc_f16(128, NH, true, true);
      // Descriptors as 32-bit halves: moving a start address by X bytes adds X >> 4 to
      // the low half (addresses stay below 256 KB, so the 14-bit field never
      // carries); the high halves (stride, swizzle) are fixed.
      const uint64_t dK = smem_desc(sbase, 16, 1024, SWZ_128B);
      const uint64_t dQ = smem_desc(sbase + C::kQOff, 16, 1024, SWZ_128B);
      const uint64_t dV = smem_desc(sbase, kSlabBytes, 1024, SWZ_128B);
      // block 3 pairs columns 384..447 with the constant block: leading offset
      // (ones - a_start) shrinks by 2048 bytes per K step
      const uint64_t dV3 = smem_desc(sbase + 6 * kSlabBytes, C::kOnesOff - 6 * kSlabBytes, 1024,
                                     SWZ_128B);
      const uint64_t dP = smem_desc(sbase + C::kPOff, 8 * C::kPRow, 8 * C::kPRow, C::kPSwz);
      const uint32_t hi = static_cast<uint32_t>(dK >> 32);   // same for dQ, dV, dV3
      const uint32_t hiP = static_cast<uint32_t>(dP >> 32);
      uint32_t lK = static_cast<uint32_t>(dK), lQ = static_cast<uint32_t>(dQ);
      uint32_t lV = static_cast<uint32_t>(dV), lV3 = static_cast<uint32_t>(dV3);
      uint32_t lP = static_cast<uint32_t>(dP);
      // Makes the bases opaque, so each MMA's operands are one add at the point of
      // use rather than values computed ahead (the issuer runs on few registers).
      auto opaque = [&]() { asm volatile("" : "+r"(lK), "+r"(lQ), "+r"(lV), "+r"(lV3), "+r"(lP)); };
      auto qk_slab = [&](int j, uint32_t idesc, bool first) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_f16_ss_hl(tS, lK + static_cast<uint32_t>((j * kSlabBytes + k * 32) >> 4), hi,
                        lQ + static_cast<uint32_t>((j * C::kQChunk + k * 32) >> 4), hi, idesc,
                        (first && k == 0) ? 0u : 1u);
      };
      auto wait = [&](int i, uint32_t par) {
        const bool r = wait_or_abort(bar(i), par, abort_f);
        tc_fence_after();
        opaque();
        return r;
      };
      bool ok = true;
      for (int it = 0; it < sp.ntiles; ++it) {
        const uint32_t par = it & 1;
        // scores: rope slab first (written earliest), then the nope parts in order
        if (!(ok = wait(B_FR, par))) break;
        qk_slab(7, kIdescQKRope, true);
        if (!(ok = wait(B_F0, par))) break;
        qk_slab(0, kIdescQK, false);
        qk_slab(1, kIdescQK, false);
        if (!(ok = wait(B_F1, par))) break;
        qk_slab(2, kIdescQK, false);
        qk_slab(3, kIdescQK, false);
        if (!(ok = wait(B_F2, par))) break;
        qk_slab(4, kIdescQK, false);
        qk_slab(5, kIdescQK, false);
        if (!(ok = wait(B_F3, par))) break;
        qk_slab(6, kIdescQK, false);
        mma_commit(bar(B_SFULL));
        if (!(ok = wait(B_PFULL, par))) break;
        const uint32_t acc0 = it > 0 ? 1u : 0u;
#pragma unroll
        for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t a = mb < 3
                ? lV + static_cast<uint32_t>((2 * mb * kSlabBytes + ks * 2048) >> 4)
                : lV3 + static_cast<uint32_t>(ks * 128) - (static_cast<uint32_t>(ks * 128) << 16);
            mma_f16_ss_hl(tO + mb * NH, a, hi,
                          lP + static_cast<uint32_t>((ks * 16 * C::kPRow) >> 4), hiP, kIdescPV,
                          ks > 0 ? 1u : acc0);
          }
          mma_commit(bar(B_E0 + mb));
          opaque();
        }
      }
      mma_commit(bar(B_ODONE));
      // Let the tensor pipe drain before the final barrier (tensor memory is freed
      // after it), also when the workers left early.
      if (!ok) mbar_wait(bar(B_ODONE), 0, kWaitLimit);
    }
    __syncwarp();
    // the cluster barrier of the merging epilogue, in step with the workers
    if constexpr (MODE == kMergeL2) cluster_sync();
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::kRegsWorker) : "memory");
    // ===================== workers =====================
    const int wt = tid - kWorkerWarp0 * 32;      // 0..511
    const int wk = wt >> 5;                      // 0..15
    // loader lanes
    const int q8 = (lane & 3) + 4 * ((lane >> 3) & 1);   // chunk lane within the row
    const int rsub = 2 * (lane >> 4) + ((lane >> 2) & 1);
    const int scale_src = (lane & 0x14) | 8;     // lane with q8 = 4 of the same row
    const bool lane_q0 = q8 == 0;
    const bool flip_lane = q8 == 0 || q8 == 4;
    // Shared addresses of this lane's words in row r: the even word of pair 0, and
    // the odd word of pair 0 for shift 0 / shift 1 (recomputed when needed: cheap).
    const uint32_t w1 = (q8 == 0 ? 8u : static_cast<uint32_t>(q8)) * 2u - 1u;   // 1..15
    auto rowb = [&](int g) { return sbase + static_cast<uint32_t>(8 * wk + 4 * g + rsub) * 128u; };
    auto rxor = [&](int g) { return static_cast<uint32_t>((4 * g + rsub) & 7); };
    auto base_e = [&](int g) {
      return rowb(g) + (q8 >> 2) * kSlabBytes + ((((2u * q8) & 7u) ^ rxor(g)) << 4);
    };
    auto base_o = [&](int g, bool sh) {
      return sh ? rowb(g) + (w1 >> 3) * kSlabBytes + (((w1 & 7u) ^ rxor(g)) << 4)
                : rowb(g) + (q8 >> 2) * kSlabBytes + ((((2u * q8 + 1u) & 7u) ^ rxor(g)) << 4);
    };
    int rr[2];
    rr[0] = 8 * wk + rsub;
    rr[1] = rr[0] + 4;
    // softmax lanes: TMEM lane quarter qd, heads [hq*HW, hq*HW + HW)
    const int qd = warp & 3;
    const int hq = wk >> 2;
    const int r_s = 32 * qd + lane;              // token row of this thread's scores
    const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;

    uint4 c[2][kSlots];
    bool s_cur[2] = {false, false};
    int nraw[2] = {-1, -1};                      // stored indices of the next tile's rows
    int vraw = -1;                               // stored index of this thread's score row
    const bool poller = wt == 0;
    bool ok = sp.ntiles > 0;
    int cur = 0;                                 // which half of mbuf holds the running max

    if (ok) {
      // ---- prologue: indices, the first tile's rows, Q ----
      int i0[2];
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        i0[g] = raw_idx(idx_row, sp.t_begin + rr[g], sp.t_end);
        nraw[g] = sp.ntiles > 1 ? raw_idx(idx_row, sp.t_begin + kTile + rr[g], sp.t_end) : -1;
      }
      vraw = raw_idx(idx_row, sp.t_begin + r_s, sp.t_end);
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const uint8_t* row = idx_ok(i0[g], num_rows, lane_q0)
                                 ? kv + static_cast<int64_t>(i0[g]) * stride : nullptr;
        const uint8_t* base = reinterpret_cast<const uint8_t*>(
            reinterpret_cast<uintptr_t>(row) & ~static_cast<uintptr_t>(15));
        const bool sh = ((reinterpret_cast<uintptr_t>(row) >> 3) & 1) != 0;
        s_cur[g] = sh;
        c[g][0] = load_slot<0>(base, q8, sh);
        c[g][1] = load_slot<1>(base, q8, sh);
        c[g][2] = load_slot<2>(base, q8, sh);
        c[g][3] = load_slot<3>(base, q8, sh);
        c[g][4] = load_slot<4>(base, q8, sh);
      }
      // Q rows h0..h0+NH-1 (bf16, copied into the tile area) -> 8 K-major SW128 slabs,
      // nope as f16, rope as bf16
      ok = workers_wait(bar(B_QRAW), 0, abort_f, poller);
      if (ok) {
        constexpr int kQPer = NH * 64 / kWorkers;
        bool q_bad = false;
#pragma unroll
        for (int k = 0; k < kQPer; ++k) {
          const int u = wt + k * kWorkers, r = u >> 6, cu = u & 63;
          uint4 o = ld_shared_v4(sbase + r * 1024 + cu * 16);
          if (cu < 56) {
            const uint2 lo = bf16x4_to_f16x4(make_uint2(o.x, o.y));
            const uint2 hi = bf16x4_to_f16x4(make_uint2(o.z, o.w));
            q_bad |= f16x2_has_inf_or_nan(lo.x) | f16x2_has_inf_or_nan(lo.y) |
                     f16x2_has_inf_or_nan(hi.x) | f16x2_has_inf_or_nan(hi.y);
            o = make_uint4(lo.x, lo.y, hi.x, hi.y);
          }
          st_shared_v4(sbase + C::kQOff + (cu >> 3) * C::kQChunk + swz_offset(r, cu & 7, 128), o);
        }
        if (q_bad) record_status(SMLA_ERR_RANGE);
        if (wt < 128) {   // the constant block: 16 rows x 8 units of 16 B
          const uint32_t r = wt >> 3, unit = wt & 7;
          const uint4 v = make_uint4(unit == 0 ? 0x3C00u : 0u, 0u, 0u, 0u);   // f16 1.0
          st_shared_v4(sbase + C::kOnesOff + (r >> 3) * 1024 + swz_offset(r & 7, unit, 128), v);
        }
      }
      workers_bar();   // the staged q is consumed before the tile area is written
    }

    for (int it = 0; ok && it < sp.ntiles; ++it) {
      const bool has_next = it + 1 < sp.ntiles;
      // ---- rows of the next tile (fetched while this one is converted) ----
      const uint8_t* nbase[2];
      bool ns[2];
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const uint8_t* row = (has_next && idx_ok(nraw[g], num_rows, lane_q0))
                                 ? kv + static_cast<int64_t>(nraw[g]) * stride : nullptr;
        nbase[g] = reinterpret_cast<const uint8_t*>(reinterpret_cast<uintptr_t>(row) &
                                                    ~static_cast<uintptr_t>(15));
        ns[g] = ((reinterpret_cast<uintptr_t>(row) >> 3) & 1) != 0;
        nraw[g] = it + 2 < sp.ntiles
                      ? raw_idx(idx_row, sp.t_begin + (it + 2) * kTile + rr[g], sp.t_end)
                      : -1;
      }
      // ---- per-row scale words of this tile ----
      RowPrep rp[2];
      bool fast = true;
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const bool sh = s_cur[g];
        // the scale word (w = 56) is the even word of chunk 28 (slot 3, q8 = 4)
        const uint32_t cand_lo = sh ? c[g][3].z : c[g][3].x;
        const uint32_t cand_hi = sh ? c[g][3].w : c[g][3].y;
        const uint32_t lo = __shfl_sync(0xffffffffu, cand_lo, scale_src);
        const uint32_t hi = __shfl_sync(0xffffffffu, cand_hi, scale_src);
        const bool masked = (lo | (hi & 0x00ffffffu)) == 0u;   // a zero-filled row
        fast &= masked || scales_fast(lo, hi);
        rp[g].lo = lo;
        rp[g].hi = hi;
        rp[g].tlo = masked ? 0u : (lo - 0x70707070u) << 2;
        rp[g].thi = masked ? 0u : (hi - 0x00707070u) << 2;
        const uint32_t kf = (sh && flip_lane) ? 1u : 0u;
        rp[g].sel_o0 = byte_sel(((q8 >> 2) ^ kf));
        rp[g].sel_o1 = byte_sel(((2 + (q8 >> 2)) ^ kf));
        rp[g].base_o = base_o(g, sh);
      }
      fast = __all_sync(0xffffffffu, fast);
      // ---- rope slab (free: the previous tile's scores are complete) ----
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const int sh = s_cur[g] ? 1 : 0;
        const int w3 = 48 + 2 * q8 - sh, w4 = 64 + 2 * q8 - sh;
        const uint32_t rx = rxor(g), rb = rowb(g) + 7 * kSlabBytes;
        auto put = [&](int w, uint32_t x, uint32_t y) {
          if (w >= 57 && w <= 72) {
            const uint32_t k = static_cast<uint32_t>(w - 57);
            st_shared_v2(rb + ((((k >> 1) ^ rx) << 4) | ((k & 1u) << 3)),
                         make_uint2(x, y));
          }
        };
        put(w3, c[g][3].x, c[g][3].y);
        put(w3 + 1, c[g][3].z, c[g][3].w);
        put(w4, c[g][4].x, c[g][4].y);
        put(w4 + 1, c[g][4].z, c[g][4].w);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_FR));
      if (has_next) {
        c[0][4] = load_slot<4>(nbase[0], q8, ns[0]);
        c[1][4] = load_slot<4>(nbase[1], q8, ns[1]);
      }
      // ---- nope: slab pairs 0..2, then slab 6, each once its value block is done ----
      auto convert_pair = [&](auto jc) {
        constexpr int J = decltype(jc)::value;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          const bool sh = s_cur[g];
          const uint4 cj = c[g][J];
          const uint32_t ex = sh ? cj.z : cj.x, ey = sh ? cj.w : cj.y;
          const uint32_t ax = lane_q0 ? c[g][J + 1].x : cj.x;
          const uint32_t ay = lane_q0 ? c[g][J + 1].y : cj.y;
          const uint32_t ox = sh ? ax : cj.z, oy = sh ? ay : cj.w;
          const uint32_t ae = base_e(g) + 2 * J * kSlabBytes;
          const uint32_t ao = rp[g].base_o + 2 * J * kSlabBytes;
          if (fast) {
            const uint32_t src = J < 2 ? rp[g].tlo : rp[g].thi;
            const uint32_t me = prmt0(src, byte_sel(2 * (J & 1) + (q8 >> 2)));
            const uint32_t mo = prmt0(src, (J & 1) ? rp[g].sel_o1 : rp[g].sel_o0);
            st_shared_v4(ae, dq8_fast(ex, ey, me));
            st_shared_v4(ao, dq8_fast(ox, oy, mo));
          } else {
            const int ge = 2 * J + (q8 >> 2);
            const int go = 2 * J + (sh ? (lane_q0 ? 1 : ((2 * q8 - 1) >> 3)) : (q8 >> 2));
            st_shared_v4(ae, dequant8_f16(ex, ey, scale_byte(rp[g].lo, rp[g].hi, ge)));
            st_shared_v4(ao, dequant8_f16(ox, oy, scale_byte(rp[g].lo, rp[g].hi, go)));
          }
        }
      };
      auto convert_slab6 = [&]() {
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          const bool sh = s_cur[g];
          const uint4 cj = c[g][3];
          const uint32_t ex = sh ? cj.z : cj.x, ey = sh ? cj.w : cj.y;
          const uint32_t ox = sh ? cj.x : cj.z, oy = sh ? cj.y : cj.w;
          const bool do_e = q8 < 4;
          const bool do_o = sh ? (q8 >= 1 && q8 <= 4) : (q8 < 4);
          const uint32_t ae = base_e(g) + 6 * kSlabBytes;
          const uint32_t ao = rp[g].base_o + 6 * kSlabBytes;
          if (fast) {
            const uint32_t m = prmt0(rp[g].thi, byte_sel(2));
            if (do_e) st_shared_v4(ae, dq8_fast(ex, ey, m));
            if (do_o) st_shared_v4(ao, dq8_fast(ox, oy, m));
          } else {
            const uint32_t sb = scale_byte(rp[g].lo, rp[g].hi, 6);
            if (do_e) st_shared_v4(ae, dequant8_f16(ex, ey, sb));
            if (do_o) st_shared_v4(ao, dequant8_f16(ox, oy, sb));
          }
        }
      };
      auto release = [&](int fb) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(fb));
      };
      // the value block that last read slabs of this part is done (no wait on tile 0)
      auto free_wait = [&](int eb) {
        return it == 0 || workers_wait(bar(eb), (it - 1) & 1, abort_f, poller);
      };
      if (!(ok = free_wait(B_E0))) break;
      convert_pair(std::integral_constant<int, 0>{});
      release(B_F0);
      if (has_next) {
        c[0][0] = load_slot<0>(nbase[0], q8, ns[0]);
        c[1][0] = load_slot<0>(nbase[1], q8, ns[1]);
      }
      if (!(ok = free_wait(B_E1))) break;
      convert_pair(std::integral_constant<int, 1>{});
      release(B_F1);
      if (has_next) {
        c[0][1] = load_slot<1>(nbase[0], q8, ns[0]);
        c[1][1] = load_slot<1>(nbase[1], q8, ns[1]);
      }
      if (!(ok = free_wait(B_E2))) break;
      convert_pair(std::integral_constant<int, 2>{});
      release(B_F2);
      if (has_next) {
        c[0][2] = load_slot<2>(nbase[0], q8, ns[0]);
        c[1][2] = load_slot<2>(nbase[1], q8, ns[1]);
      }
      if (!(ok = free_wait(B_E3))) break;
      convert_slab6();
      release(B_F3);
      if (has_next) {
        c[0][3] = load_slot<3>(nbase[0], q8, ns[0]);
        c[1][3] = load_slot<3>(nbase[1], q8, ns[1]);
      }
      s_cur[0] = ns[0];
      s_cur[1] = ns[1];

      // ---- softmax of this tile ----
      const bool valid = idx_ok(vraw, num_rows, false);
      vraw = has_next ? raw_idx(idx_row, sp.t_begin + (it + 1) * kTile + r_s, sp.t_end) : -1;
      if (!(ok = workers_wait(bar(B_SFULL), it & 1, abort_f, poller))) break;
      tc_fence_after();
      float sv[HW];
      float ex = -INFINITY;
      tmem_ld<HW>(tS + lane_base + hq * HW, sv);
      tmem_wait_ld();
      {
        const float* m_old = mbuf + cur * NH + hq * HW;
#pragma unroll
        for (int i = 0; i < HW; ++i) {
          sv[i] = valid ? sv[i] * scale_log2 : -INFINITY;
          ex = fmaxf(ex, sv[i] - m_old[i]);   // NaN (-inf - -inf) is ignored by fmaxf
        }
        if (!valid) ex = -INFINITY;
      }
      // One barrier in the common case: no score passed the running max by more
      // than the headroom.
      if (workers_bar_or(ex > kLazyMax)) {
        // Raise the running max to the exact tile max and rescale O (and with it
        // the denominator row) by 2^(m_old - m_new).
#pragma unroll
        for (int i = 0; i < HW; ++i) {
          const float m = warp_max(sv[i]);
          if (lane == i) red[qd * NH + hq * HW + i] = m;
        }
        workers_bar();
        const float* m_old = mbuf + cur * NH;
        float* m_new = mbuf + (cur ^ 1) * NH;
        if (wt < NH) {
          const float mt = fmaxf(fmaxf(red[wt], red[NH + wt]), fmaxf(red[2 * NH + wt], red[3 * NH + wt]));
          m_new[wt] = fmaxf(m_old[wt], mt);
        }
        workers_bar();
        if (it > 0) {
          float f[HW];
#pragma unroll
          for (int i = 0; i < HW; ++i) {
            const float mn = m_new[hq * HW + i];
            f[i] = (mn == -INFINITY) ? 1.f : exp2f(m_old[hq * HW + i] - mn);
          }
#pragma unroll 1
          for (int mb = 0; mb < 4; ++mb) {
            float o[HW];
            tmem_ld<HW>(tO + lane_base + mb * NH + hq * HW, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < HW; ++i) o[i] *= f[i];
            tmem_st<HW>(tO + lane_base + mb * NH + hq * HW, o);
          }
          tmem_wait_st();
        }
        cur ^= 1;
      }
      {
        const float* m = mbuf + cur * NH + hq * HW;
#pragma unroll
        for (int i = 0; i < HW; ++i)
          // sv = -inf (masked) gives 0; m = -inf only while every score so far is
          // masked, and then sv is -inf too
          sv[i] = (sv[i] == -INFINITY) ? 0.f : fast_exp2(sv[i] - m[i]);
        const uint32_t prow = sbase + C::kPOff;
        if constexpr (HW == 16) {
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            uint4 v;
            v.x = pack_f16x2(sv[8 * u + 0], sv[8 * u + 1]);
            v.y = pack_f16x2(sv[8 * u + 2], sv[8 * u + 3]);
            v.z = pack_f16x2(sv[8 * u + 4], sv[8 * u + 5]);
            v.w = pack_f16x2(sv[8 * u + 6], sv[8 * u + 7]);
            st_shared_v4(prow + swz_offset(r_s, 2 * hq + u, C::kPRow), v);
          }
        } else if constexpr (HW == 8) {
          uint4 v;
          v.x = pack_f16x2(sv[0], sv[1]);
          v.y = pack_f16x2(sv[2], sv[3]);
          v.z = pack_f16x2(sv[4], sv[5]);
          v.w = pack_f16x2(sv[6], sv[7]);
          st_shared_v4(prow + swz_offset(r_s, hq, C::kPRow), v);
        } else {
          const uint2 v = make_uint2(pack_f16x2(sv[0], sv[1]), pack_f16x2(sv[2], sv[3]));
          st_shared_v2(prow + swz_offset(r_s, hq >> 1, C::kPRow) + (hq & 1) * 8, v);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PFULL));
    }

    // ===================== epilogue =====================
    // ok is the same in every worker here (all its changes came from uniform waits)
    const bool have_o = ok && workers_wait(bar(B_ODONE), 0, abort_f, poller);
    if (have_o) tc_fence_after();
    if (qd == 2) {
      // row 448 of block 3 (TMEM lane 64: lane 0 of quarter 2) = sum_t P[t] per head
      float o[HW];
      if (have_o) {
        tmem_ld<HW>(tO + lane_base + 3 * NH + hq * HW, o);
        tmem_wait_ld();
      }
      if (lane == 0) {
#pragma unroll
        for (int i = 0; i < HW; ++i) lfin[hq * HW + i] = have_o ? o[i] : 0.f;
      }
    }
    workers_bar();
    {
    if (wt < NH) {
      const float lt = lfin[wt];
      const float lse = lt > 0.f ? (mbuf[cur * NH + wt] + log2f(lt)) * kLn2 : -INFINITY;
      lse_part[(static_cast<int64_t>(b) * H + h0 + wt) * S + s] = lse;
      red[wt] = lt > 0.f ? 1.0f / lt : 0.f;
    }
    workers_bar();
    {
      // warp (block mb, quarter qd) writes value rows 128 mb + 32 qd + lane
      const int mb = wk >> 2;
      const int d = mb * 128 + qd * 32 + lane;
      const int64_t hstride = static_cast<int64_t>(S) * kNope;
      float* dst = o_part + ((static_cast<int64_t>(b) * H + h0) * S + s) * kNope + d;
#pragma unroll
      for (int cc = 0; cc < NH / 16; ++cc) {
        float o[16];
        if (have_o) {
          tmem_ld16(tO + lane_base + mb * NH + 16 * cc, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] = 0.f;
        }
        if (d < kNope) {
#pragma unroll
          for (int i = 0; i < 16; ++i) dst[(16 * cc + i) * hstride] = o[i] * red[16 * cc + i];
        }
      }
    }
    if constexpr (MODE == kMergeL2) {
      cluster_sync();   // every split of this (query, head group) has written its partials
      // this CTA merges heads [h_lo, h_hi): weights exp(lse_s - lse) per head first
      const int h_lo = s * NH / S, h_hi = (s + 1) * NH / S, nh = h_hi - h_lo;
      float* wgt = reinterpret_cast<float*>(smem);   // [nh][kMaxCluster] (tile area is free)
      float* fin = wgt + NH * kMaxCluster;            // [nh] final lse (natural log)
      if (wt < nh) {
        const float* lp = lse_part + (static_cast<int64_t>(b) * H + h0 + h_lo + wt) * S;
        float x[kMaxCluster];
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r) x[r] = r < S ? lp[r] : -INFINITY;
        float M = -INFINITY;
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r) M = fmaxf(M, x[r]);
        float sum = 0.f;
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r) {
          const float e = (M == -INFINITY || x[r] == -INFINITY) ? 0.f : __expf(x[r] - M);
          x[r] = e;
          sum += e;
        }
        const float inv = sum > 0.f ? 1.f / sum : 0.f;
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r) wgt[wt * kMaxCluster + r] = x[r] * inv;
        fin[wt] = sum > 0.f ? M + logf(sum) : -INFINITY;
      }
      workers_bar();
      const int units = nh * (kNope / 4);
      for (int u = wt; u < units; u += kWorkers) {
        const int hl = u / (kNope / 4), d4 = u % (kNope / 4);
        const float4* src = reinterpret_cast<const float4*>(
            o_part + ((static_cast<int64_t>(b) * H + h0 + h_lo + hl) * S) * kNope) + d4;
        float4 v[kMaxCluster];
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r)
          if (r < S) v[r] = __ldcg(src + r * (kNope / 4));
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r) {
          if (r < S) {
            const float ws = wgt[hl * kMaxCluster + r];
            acc.x = fmaf(ws, v[r].x, acc.x);
            acc.y = fmaf(ws, v[r].y, acc.y);
            acc.z = fmaf(ws, v[r].z, acc.z);
            acc.w = fmaf(ws, v[r].w, acc.w);
          }
        }
        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 pk;
        pk.x = *reinterpret_cast<const uint32_t*>(&lo);
        pk.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(out + (static_cast<int64_t>(b) * H + h0 + h_lo + hl) * kNope +
                                  4 * d4) = pk;
      }
      if (wt < nh) lse_out[static_cast<int64_t>(b) * H + h0 + h_lo + wt] = fin[wt];
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

// Once per device and kernel: shared-memory size and the register check (the
// setmaxnreg split assumes the launch allocation; a build that differs is refused,
// since its register increase would never be granted).
template <int NH, int MODE>
cudaError_t configure(int dev) {
  static int configured_device = -1;
  if (configured_device == dev) return cudaSuccess;
  using C = Cfg<NH>;
  cudaError_t e = cudaFuncSetAttribute(split_kernel<NH, MODE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, split_kernel<NH, MODE>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidKernelImage;
  configured_device = dev;
  return cudaSuccess;
}

template <int NH>
cudaError_t launch_split_t(const void* q, const void* kv, const int32_t* indices, float* o_part,
                           float* lse_part, int B, int H, int topk, int S, int64_t num_rows,
                           int64_t stride, float softmax_scale, cudaStream_t stream) {
  using C = Cfg<NH>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = configure<NH, kSplitOnly>(dev);
  if (e != cudaSuccess) return e;
  const dim3 grid(S, H / NH, B);
  const float scale_log2 = softmax_scale * 1.4426950408889634f;
  return launch_programmatic(split_kernel<NH, kSplitOnly>, grid, dim3(kThreads), C::kSmemBytes,
                             stream, static_cast<const uint16_t*>(q),
                             static_cast<const uint8_t*>(kv), indices, o_part, lse_part,
                             static_cast<__nv_bfloat16*>(nullptr), static_cast<float*>(nullptr), H,
                             topk, S, num_rows, stride, scale_log2);
}

constexpr int kMaxClusterSplits = kMaxCluster;

// Whether a cluster of S split CTAs fits on the device: asked once per (device, S).
template <int NH, int MODE>
cudaError_t cluster_fits(int dev, int S, bool* fits) {
  static int asked_device[kMaxClusterSplits + 1] = {-1, -1, -1, -1, -1, -1, -1, -1, -1};
  static bool answer[kMaxClusterSplits + 1] = {};
  if (S < 1 || S > kMaxClusterSplits) {
    *fits = false;
    return cudaSuccess;
  }
  if (asked_device[S] != dev) {
    cudaError_t e = configure<NH, MODE>(dev);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg<NH>::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, split_kernel<NH, MODE>, &cfg);
    if (e != cudaSuccess) return e;
    answer[S] = n > 0;
    asked_device[S] = dev;
  }
  *fits = answer[S];
  return cudaSuccess;
}

template <int NH, int MODE>
cudaError_t launch_fused_t(const void* q, const void* kv, const int32_t* indices, float* o_part,
                           float* lse_part, void* out, float* lse, int B, int H, int topk, int S,
                           int64_t num_rows, int64_t stride, float softmax_scale,
                           cudaStream_t stream) {
  using C = Cfg<NH>;
  if (S < 1 || S > kMaxClusterSplits) return cudaErrorNotSupported;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = configure<NH, MODE>(dev);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S, H / NH, B);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  bool fits = false;
  e = cluster_fits<NH, MODE>(dev, S, &fits);
  if (e != cudaSuccess) return e;
  if (!fits) return cudaErrorNotSupported;
  const float scale_log2 = softmax_scale * 1.4426950408889634f;
  return cudaLaunchKernelEx(&cfg, split_kernel<NH, MODE>, static_cast<const uint16_t*>(q),
                            static_cast<const uint8_t*>(kv), indices, o_part, lse_part,
                            static_cast<__nv_bfloat16*>(out), lse, H, topk, S, num_rows, stride,
                            scale_log2);
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

cudaError_t launch_decode_fused(const void* q, const void* kv, const int32_t* indices,
                                float* o_part, float* lse_part, void* out, float* lse, int B,
                                int H, int topk, int S, int64_t num_rows, int64_t stride,
                                float softmax_scale, cudaStream_t stream) {
  switch (H) {
    case 16:
      return launch_fused_t<16, kMergeL2>(q, kv, indices, o_part, lse_part, out, lse, B, H, topk,
                                          S, num_rows, stride, softmax_scale, stream);
    case 32:
      return launch_fused_t<32, kMergeL2>(q, kv, indices, o_part, lse_part, out, lse, B, H, topk,
                                          S, num_rows, stride, softmax_scale, stream);
    default:
      return launch_fused_t<64, kMergeL2>(q, kv, indices, o_part, lse_part, out, lse, B, H, topk,
                                          S, num_rows, stride, softmax_scale, stream);
  }
}

cudaError_t fused_supported(int H, int S, bool* supported) {
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  switch (H) {
    case 16: return cluster_fits<16, kMergeL2>(dev, S, supported);
    case 32: return cluster_fits<32, kMergeL2>(dev, S, supported);
    default: return cluster_fits<64, kMergeL2>(dev, S, supported);
  }
}

cudaError_t status_word_address(int** ptr) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(ptr), g_smla_status);
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
