// Split kernel of sparse MLA decode for sm_103a.
//
// One CTA handles one (query b, group of NH heads, split s of the top-k list).  For
// each block of 64 index slots it
//   1. gathers the selected 584-byte rows once for all NH heads ("The Moment of
//      Compilation: When a Triton Kernel Meets Its Constraints", section "The
//      Context: A Kernel Optimization Campaign": one KV read shared by all heads),
//   2. dequantises the FP8 e4m3 nope part with its per-64-column UE8M0 scales into
//      f16 ("The Power-of-Two Trap: Debugging a Triton MMA Kernel on Blackwell GPUs",
//      section "3. The Scale Indexing Complication"), next to the rope part,
//   3. computes the scores of the block on the tensor cores (tcgen05.mma) into tensor
//      memory,
//   4. runs the online softmax of the block,
//   5. accumulates O^T += V^T . P^T on the tensor cores (value columns as the MMA's
//      M dimension, heads as N, tokens as K) in tensor memory,
// and finally writes the normalised partial O and its log-sum-exp for the split (the
// split-K scheme of "The 80KB Mystery: Resolving Contradictory Evidence in Triton
// Kernel Optimization", section "The Context: Optimizing Attention on Blackwell").
// Launched as thread-block clusters of the S splits of a (query, head group), the
// CTAs keep their partials in shared memory and, after a cluster barrier, each merges
// a slice of the heads from the other splits' shared memory and writes the final out
// and lse.
//
// Stacked blocks.  A block of 64 tokens is held as a 128-row f16 operand: row t
// (< 64) holds token t's columns 0..255, row 64 + t its columns 256..511 (nope
// 256..447 and the rope), so every tcgen05.mma has M = 128 although a block has 64
// tokens.  The query is stacked the same way (head h's columns 0..255, then again
// its columns 256..511); each half of a score is a partial dot product, and the
// softmax threads holding the two halves add them (trading them through shared
// memory; the two halves sit in different warps, since a tensor-memory load takes one
// column address per warp).
//   - 16 / 32 heads (Q in shared memory): S^T = K_stacked . Q_stacked^T, tokens as
//     the MMA's M, N = 2 NH.  A softmax thread owns one token half for all heads.
//   - 64 heads (Q in tensor memory): S = Q_stacked . K_stacked^T with the stacked
//     query (2 NH = 128 rows) as the A operand in tensor memory, so shared memory is
//     not re-read for Q every block.  A softmax thread owns one head half for the
//     block's tokens; the running max of a head lives in a register.
// The value product reads the same bytes: value columns 0..127 are slabs 0-1 of rows
// 0..63, 128..255 slabs 2-3, 256..383 slabs 0-1 of rows 64..127, and 384..447 slab 2
// of rows 64..127 paired with a constant block whose first column is 1, so output
// row 448 is sum_t P[t], the softmax denominator, accumulated and rescaled by the
// tensor core together with O.
//
// Pipeline.  Two block buffers: while the tensor core and the softmax work on one
// block, a set of converter warps fills the other.  With 64 heads the rows are
// gathered by TMA tile::gather4 copies into a staging ring of half blocks, a few
// half blocks ahead of the converters; with 16 / 32 heads the converters load them
// through L1 themselves, a block ahead.  All operands are f16 (fp32 accumulation):
// e4m3 -> f16 is one conversion and the power-of-two group scale one f16x2
// multiply; q and the rope are converted from bf16 (values beyond the f16 range are
// reported as SMLA_ERR_RANGE).  The running max is raised lazily (headroom 2^15).
//
// Warp roles (768 threads, one CTA per SM, 155-222 KiB of shared memory):
//   warps 0..3    softmax: one thread per tensor-memory lane; they also convert q
//   warps 4..19   16 converters in two sets of 8 (even / odd blocks): each warp
//                 takes 8 rows of its set's block as 8-byte words (8 lanes per row)
//                 out of the staging ring or from the cache, dequantises them into
//                 the buffer, and writes the epilogue
//   warp 20       allocates tensor memory, copies q in, and issues the score MMAs
//                 (one lane); with Q in tensor memory it also issues the value
//                 products, in readiness order
//   warp 21       with Q in shared memory: issues the value-product MMAs (one lane)
//   warp 22       with 64 heads: gathers the rows (tensor copies)
//   others        idle (their registers go to the other roles)
// Every wait is bounded; on timeout the CTA records SMLA_ERR_TIMEOUT in the device
// status word and leaves through the epilogue.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "../../include/smla.h"
#include "smla_internal.h"
#include "smla_ptx.cuh"

namespace smla {

__device__ int g_smla_status = 0;

// Test hook (smla_test_inject_fault): block index at which converter warp 0 of every
// CTA withholds its "block filled" arrival, or -1.
std::atomic<int> g_fault_block{-1};

namespace {

constexpr int kBlk = 64;                        // tokens per block
constexpr int kSlab = 128 * 128;                // one 64-column f16 slab of 128 rows
constexpr int kBuf = 4 * kSlab;                 // one stacked block
constexpr int kSoftWarps = 4;
constexpr int kConvWarp0 = 4;
constexpr int kConvWarps = 16;
constexpr int kConv = kConvWarps * 32;          // 512
constexpr int kMmaWarp = 20;
constexpr int kTmaWarp = 22;                    // issues the row gathers (tensor copies)
constexpr int kThreads = 24 * 32;               // 768
// Register split (setmaxnreg): launched with kLaunchRegs per thread (65536 / 768
// rounded down to a multiple of 8); the MMA warpgroup gives registers back, the
// softmax and converter warpgroups take them.
constexpr int kLaunchRegs = 80;
constexpr int kRegsSoft = 88;
constexpr int kRegsConv = 88;
constexpr int kRegsMma = 40;
static_assert(kRegsSoft * 128 + kRegsConv * kConv + kRegsMma * 128 <= kLaunchRegs * kThreads,
              "register split exceeds the launch allocation");
// Bounded waits, in units of 1024 SM clocks: ~1 s, and ~10 ms with the test hook on.
constexpr uint32_t kWaitLimitK = 2000000u;
constexpr uint32_t kFaultWaitLimitK = 20000u;
constexpr float kLn2 = 0.69314718055994530942f;
// log2 headroom before the running max is raised: P = 2^(s - m) <= 2^15 stays inside
// the f16 range (65504) with its full 11-bit precision, and a rescale (which waits for
// the previous value product) happens only when a score passes the max by 2^15
constexpr float kLazyMax = 15.0f;
constexpr int kMaxCluster = 8;                  // splits merged on chip (portable cluster size)
// Row gather by tensor copies (64 heads).  The rows of half a block (32
// slots) land in one stage of a ring, as 592-byte windows (74 words of 8 bytes: the row
// and 8 bytes before or after it), four rows per copy; the four windows of a copy land
// back to back in a 2432-byte group (a multiple of 128 bytes).  The rows are split by
// the parity of their 16-byte alignment, so a half block takes at most 9 groups.
constexpr int kHalfRows = 32;
constexpr int kWinWords = 74;
constexpr int kWin = kWinWords * 8;             // 592
constexpr int kGrp = 2432;
constexpr int kMaxGroups = 9;
constexpr int kStageBytes = kMaxGroups * kGrp;  // 21888
constexpr int kStages = 3;
constexpr uint32_t kNoRow = 0xffffu;            // window offset of a masked slot
enum : int { kSplitOnly = 0, kMergeCluster = 1 };

// Named barriers (id 0 is __syncthreads).
enum : int { kBarSoft = 1, kBarConv = 2, kBarEpi = 3, kBarPair0 = 4, kBarPair1 = 5 };

// mbarriers.  FULL0..2: block buffer filled (one arrival per converter warp of the
// set that fills it); EMPTY0..2: value product of the block in that buffer done
// (buffer and, with one P buffer, P free);
// SFULL0/1: scores in tensor-memory buffer 0/1 (one buffer, SFULL0, with Q in tensor
// memory); SEMPTY0/1: softmax has read them; PFULL0/1: P buffer 0/1 written (one
// buffer, PFULL0, with Q in shared memory); ODONE: all value products done (and with
// them all scores); QDONE: the score MMAs done (drain on abort); QRAW: the bf16 q
// rows copied into buffer 1 (Q in shared memory); QREADY: the stacked f16 Q and the
// constant block written.  Rows gathered by tensor copies: RAWFULL0..3: the rows of the
// next half block that converter group g (set g / 2, half g % 2) takes have landed in
// their stage (one barrier per group, so each is waited in order by one group only);
// RAWEMPTY0..2: the converters have taken the rows out of stage 0..2.
enum Bar : int {
  B_FULL0 = 0, B_FULL1, B_FULL2, B_EMPTY0, B_EMPTY1, B_EMPTY2, B_SFULL0, B_SFULL1,
  B_SEMPTY0, B_SEMPTY1,
  B_PFULL0, B_PFULL1, B_ODONE, B_QDONE, B_QRAW, B_QREADY, B_RAWFULL0, B_RAWFULL1, B_RAWFULL2,
  B_RAWFULL3, B_RAWEMPTY0, B_RAWEMPTY1, B_RAWEMPTY2, B_COUNT
};

// The tensor maps of one launch.  Rows are gathered through `even` and `odd`: rows are
// 8-byte aligned and a tensor copy must start on a 16-byte boundary.  With a row stride
// that is a multiple of 16 every row starts on one and `even` maps them all (x = 0: the
// row and 8 zero-filled bytes past its 73 words).  Otherwise every other row starts 8
// bytes past a boundary: `even` then maps row pairs (row 2k at x = 0), `odd` the row
// pairs shifted by stride - 8 bytes (row 2k + 1 at byte 8 of its window), and split is
// 1.  `q` maps q as [B H rows][512 bf16] in boxes of 64 columns x NH rows, 128-byte
// swizzled (16-byte unit u of row r lands at unit u ^ (r % 8) of its 128-byte row).
struct RowMaps {   // (aligned as CUtensorMap requires)
  CUtensorMap even;
  CUtensorMap odd;
  CUtensorMap q;
  int split;
};

template <int NH>
struct Cfg {
  // Q in tensor memory (the score MMA's A operand, scores transposed: heads as M) for
  // 64 heads, where 2 NH = 128 stacked query rows fill the MMA's M; Q in shared
  // memory (tokens as M) for fewer heads.
  static constexpr bool kTS = NH == 64;
  // rows gathered by tensor copies into a staging ring, else by the converters' loads
  // through L1.  Measured: with 64 heads the tensor copies are faster (the loads
  // congest the load/store path the softmax warps use); with 16 heads, where the
  // gather rate bounds the kernel, the loads of all 16 converter warps are (the
  // tensor-copy unit moves ~13.5 bytes per clock per SM on these rows).
  static constexpr bool kTmaRows = NH == 64;
  static constexpr int kHalf = NH / 2;                     // heads per softmax thread (SS)
  static constexpr int kQSlab = 2 * NH * 128;              // stacked Q: 2 NH rows x 128 B
  // Two block buffers.  With kTmaRows the rows are gathered by tensor copies into a
  // staging ring, so L1 is not involved and the carve-out may leave it small;
  // otherwise the converters load the rows through L1, which above ~195 KB of shared
  // memory the carve-out leaves too small for them (measured slower).
  static constexpr int kNBuf = 2;
  // the buffer that holds the bf16 q rows until the softmax warps have converted them
  static constexpr int kQRawBuf = 1;
  static constexpr int kQOff = kNBuf * kBuf;
  // P: SS [64 tokens][NH] (MN-major B operand); TS [NH heads][64 tokens] (K-major B
  // operand, 128-byte rows).  One buffer, free again once the block's value product
  // is done.
  static constexpr int kPOff = kTS ? kNBuf * kBuf : kQOff + 4 * kQSlab;
  static constexpr int kPRow = 2 * NH;                     // bytes of one P row (SS: token)
  static constexpr int kPBytes = kBlk * kPRow;
  static constexpr int kPStride = ((kPBytes + 1023) / 1024) * 1024;
  // (a second P buffer measured no faster with 16 heads; with 64 heads the staging
  // ring takes the room)
  static constexpr int kPBufs = 1;
  static constexpr int kXOff = kPOff + kPBufs * kPStride;
  // SS: score halves traded, and the block-max transpose (NH heads x 65 floats);
  // TS: 32 partial scores per thread (128 rows of 128 bytes)
  static constexpr int kXBytes = kTS ? 128 * 128 : NH * 65 * 4;
  static constexpr int kOnesOff = kXOff + ((kXBytes + 1023) / 1024) * 1024;  // 2 KB
  static constexpr int kMOff = kOnesOff + 2048;            // float [2][NH] running max (log2)
  static constexpr int kLOff = kMOff + 2 * NH * 4;         // float [NH] denominators
  static constexpr int kRinvOff = kLOff + NH * 4;          // float [NH] 1 / denominators
  static constexpr int kMxOff = kRinvOff + NH * 4;         // float [128] block maxima (TS)
  static constexpr int kAlphaOff = kMxOff + 128 * 4;       // float [NH] rescale factors (TS)
  static constexpr int kBarOff = kAlphaOff + NH * 4;       // uint64 [B_COUNT]
  static constexpr int kTaddrOff = kBarOff + 8 * B_COUNT;  // uint32
  static constexpr int kAbortOff = kTaddrOff + 4;          // int
  // tensor-copy gather: the staging ring, the window offset of each slot's row per
  // stage, and the map rows in gather order
  static constexpr int kStageOff = ((kAbortOff + 4 + 1023) / 1024) * 1024;
  static constexpr int kTabOff = kStageOff + (kTmaRows ? kStages * kStageBytes : 0);  // u16 [3][32]
  static constexpr int kListOff = kTabOff + (kTmaRows ? kStages * 2 * kHalfRows : 0);  // int [36]
  // the indices of the next four half blocks (int [4][32])
  static constexpr int kIdxOff = kListOff + (kTmaRows ? 4 * (kHalfRows + 4) : 0);
  static constexpr int kSmemBytes = kIdxOff + (kTmaRows ? 4 * 4 * kHalfRows : 0) + 1024;  // + slack
  // TS: Q (128 columns), S (128: stacked heads x tokens), O^T (4 x NH); SS: S^T (two
  // buffers of 2 NH columns) and O^T (4 x NH)
  static constexpr uint32_t kTmemCols = kTS ? 512 : 8 * NH <= 128 ? 128 : 8 * NH <= 256 ? 256 : 512;
  static constexpr uint32_t kTQ = 0, kTS_S = kTS ? 128 : 0, kTO = kTS ? 256 : 4 * NH;
  static constexpr uint32_t kPSwz = NH == 64 ? SWZ_128B : NH == 32 ? SWZ_64B : SWZ_32B;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(kTS || NH * 64 <= kBuf / 2, "the staged q rows fit in a block buffer");
  static_assert(!kTS || 4 * NH + 256 <= 512, "tensor memory");
};

__device__ __forceinline__ void record_status(int code) { atomicCAS(&g_smla_status, 0, code); }

#ifdef SMLA_DEBUG
// Debug build: every computed shared-memory address of the explicit shared loads and
// stores is checked against this CTA's dynamic shared-memory window, and every
// gathered row's byte range against the cache; a violation records
// SMLA_ERR_INTERNAL in the device status word and the access is skipped (no trap).
extern __shared__ uint8_t smla_dbg_dynamic_smem[];
__device__ __forceinline__ bool smem_access_ok(uint32_t addr, uint32_t bytes) {
  uint32_t size;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(size));
  const uint32_t lo = smem_u32(smla_dbg_dynamic_smem);
  const bool ok = addr >= lo && addr + bytes <= lo + size;
  if (!ok) record_status(SMLA_ERR_INTERNAL);
  return ok;
}
#define SMLA_SMEM_OK(addr, bytes) smem_access_ok((addr), (bytes))
#else
#define SMLA_SMEM_OK(addr, bytes) true
#endif

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  if (!SMLA_SMEM_OK(addr, 16)) return;
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  if (!SMLA_SMEM_OK(addr, 16)) return make_uint4(0u, 0u, 0u, 0u);
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ uint2 ld_shared_v2(uint32_t addr) {
  uint2 v;
  if (!SMLA_SMEM_OK(addr, 8)) return make_uint2(0u, 0u);
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_shared_v2(uint32_t addr, uint2 v) {
  if (!SMLA_SMEM_OK(addr, 8)) return;
  asm volatile("st.shared.v2.u32 [%0], {%1,%2};" ::"r"(addr), "r"(v.x), "r"(v.y) : "memory");
}
__device__ __forceinline__ uint2 ldg_nc_u2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p));
  return v;
}
// Named-barrier helpers: `count` threads meet at barrier `id`.
__device__ __forceinline__ void bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Returns true if any of the threads passed true.
__device__ __forceinline__ bool bar_or(int id, int count, bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred a, b;\n\tsetp.ne.u32 a, %1, 0;\n\t"
      "bar.red.or.pred b, %2, %3, a;\n\tselp.u32 %0, 1, 0, b;\n\t}\n"
      : "=r"(r)
      : "r"(p ? 1u : 0u), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}
// Returns true if every thread passed true.
__device__ __forceinline__ bool bar_and(int id, int count, bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred a, b;\n\tsetp.ne.u32 a, %1, 0;\n\t"
      "bar.red.and.pred b, %2, %3, a;\n\tselp.u32 %0, 1, 0, b;\n\t}\n"
      : "=r"(r)
      : "r"(p ? 1u : 0u), "r"(id), "r"(count)
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
  static_assert(N == 8 || N == 16, "width");
  if constexpr (N == 16) {
    tmem_ld16(taddr, v);
  } else {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
  }
}
template <int N>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const float* v) {
  static_assert(N == 8 || N == 16, "width");
  if constexpr (N == 16) {
    tmem_st16(taddr, v);
  } else {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(
                     taddr),
                 "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
                 "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
                 "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                 "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
                 : "memory");
  }
}
// N columns in chunks of 8 or 16.
template <int N>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, float* v) {
  if constexpr (N % 16 == 0) {
#pragma unroll
    for (int k = 0; k < N / 16; ++k) tmem_ld<16>(taddr + 16 * k, v + 16 * k);
  } else {
    static_assert(N == 8, "width");
    tmem_ld<8>(taddr, v);
  }
}

// UE8M0 byte -> fp32 2^(e-127) (e = 0 is the fp32 subnormal 2^-127, 0xFF is NaN).
__device__ __forceinline__ float ue8m0_to_f32(uint32_t e) {
  const uint32_t bits = e == 0u ? 0x00400000u : (e == 255u ? 0x7fffffffu : (e << 23));
  return __uint_as_float(bits);
}

// Two e4m3 bytes -> f16x2 of value * m2 (m2 = f16x2 2^(s - 127)): e4m3 -> f16 is
// exact and the product by a power of two is exact while it stays in the f16 range.
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
// 8 e4m3 bytes times the f16x2 power of two m (fast path: exact, in range).
__device__ __forceinline__ uint4 dq8_fast(uint32_t x, uint32_t y, uint32_t m) {
  uint4 v;
  v.x = dq_pair_f16(x & 0xffffu, m);
  v.y = dq_pair_f16(x >> 16, m);
  v.z = dq_pair_f16(y & 0xffffu, m);
  v.w = dq_pair_f16(y >> 16, m);
  return v;
}
// 8 e4m3 bytes with scale byte s -> 8 f16, any s: the product is formed in fp32 and
// rounded to f16 (subnormal results are rounded, not flushed); values beyond the f16
// range become inf and are reported (SMLA_ERR_RANGE).  Out of line: it serves only
// rows with unusual scale bytes, and keeping it out of the converters' loop keeps
// that loop small in the instruction cache.
__device__ __noinline__ uint4 dequant8_checked(uint32_t x, uint32_t y, uint32_t s) {
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
  return make_uint4(o[0], o[1], o[2], o[3]);
}
// Two bf16 (one 32-bit word) -> f16x2 (exact for magnitudes in [2^-14, 65504];
// smaller ones round to f16 subnormals, larger ones become inf).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  return pack_f16x2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

// Bounded mbarrier wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_f,
                                              uint32_t limit_k) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_f) return false;
    if (clock64() - t0 > (static_cast<long long>(limit_k) << 10)) {
      *abort_f = 1;
      record_status(SMLA_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}
// Wait of a group of warps that meet at named barrier `id`: one thread polls the
// mbarrier (bounded), the others sleep on the named barrier, and every thread gets
// the same verdict.
__device__ __forceinline__ bool group_wait(uint32_t bar, uint32_t parity, volatile int* abort_f,
                                           uint32_t limit, bool poller, int id, int count) {
  bool ok = true;
  if (poller) ok = wait_or_abort(bar, parity, abort_f, limit);
  __syncwarp();
  return bar_and(id, count, ok);
}
// Wait of one warp: lane 0 polls, the warp shares its verdict.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_f,
                                          uint32_t limit) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = wait_or_abort(bar, parity, abort_f, limit);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

struct Split {
  int t_begin, t_end, nblocks;
};
__device__ __forceinline__ Split split_range(int topk, int S, int s) {
  const int G = (topk + 15) >> 4;
  const int g0 = static_cast<int>((static_cast<int64_t>(s) * G) / S);
  const int g1 = static_cast<int>((static_cast<int64_t>(s + 1) * G) / S);
  Split r;
  r.t_begin = min(16 * g0, topk);
  r.t_end = min(16 * g1, topk);
  r.nblocks = (r.t_end - r.t_begin + kBlk - 1) / kBlk;
  return r;
}

// Index of slot `pos` as stored (-1 past the split).
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
// Row words.  A row is 73 words of 8 bytes (rows are 8-byte aligned): word w < 56
// holds nope columns 8w..8w+7 (scale group w / 8), word 56 the 7 scales and the pad,
// words 57..72 the rope.  8 lanes share a row (lane = 8 * row + q); lane q reads words
// q + 8k of the row (gathered, or from the cache) into register slot k (k = 0..8, and
// k = 9 for word 72 on lane 0), so slot k < 7 of every lane is a nope word of group k, slot 7 is the scale
// word (lane 0) or rope word 56 + q, slot 8 rope word 64 + q.  A 16-byte shared store
// of slot k by a warp is served in four phases of 8 consecutive lanes, i.e. one row
// each, whose 8 words fill the 8 distinct 16-byte units of their 128-byte row: no bank
// conflicts.
// ---------------------------------------------------------------------------
constexpr int kSlots = 10;

__device__ __forceinline__ uint2 load_word(const uint8_t* row, int w) {
  return row == nullptr ? make_uint2(0u, 0u) : ldg_nc_u2(row + 8 * w);
}

// prmt selecting byte g of the pair (a, b) into bits 8..15 of both halves, with byte
// 7 of the pair (zero by construction) elsewhere.
__device__ __forceinline__ uint32_t prmt2(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
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

// MODE kSplitOnly: writes the split's normalised partial O and lse (o_part, lse_part).
// MODE kMergeCluster: launched as clusters of the S splits of one (query, head group);
//   each split keeps its partial in shared memory, then after a cluster barrier each
//   CTA merges a slice of the heads from all the splits' shared memory (distributed
//   shared memory) and writes the final bf16 out and lse: the split-K combine without
//   a second launch and without partials in global memory.
template <int NH, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    split_kernel(const uint16_t* __restrict__ q, const uint8_t* __restrict__ kv,
                 const __grid_constant__ RowMaps rows, const int32_t* __restrict__ indices,
                 float* __restrict__ o_part, float* __restrict__ lse_part,
                 __nv_bfloat16* __restrict__ out, float* __restrict__ lse_out, int H, int topk,
                 int S, int64_t num_rows, int64_t stride, float scale_log2, int fault_block) {
  using C = Cfg<NH>;
  constexpr int HH = C::kHalf;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int s = blockIdx.x, h0 = blockIdx.y * NH, b = blockIdx.z;
  const Split sp = split_range(topk, S, s);
  const int nb = sp.nblocks;
  const int32_t* idx_row = indices + static_cast<int64_t>(b) * topk;
  const uint32_t limit = fault_block >= 0 ? kFaultWaitLimitK : kWaitLimitK;

  float* mbuf = reinterpret_cast<float*>(smem + C::kMOff);
  float* lfin = reinterpret_cast<float*>(smem + C::kLOff);
  float* rinv = reinterpret_cast<float*>(smem + C::kRinvOff);
  const uint32_t bars = sbase + C::kBarOff;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  volatile uint32_t* taddr_s = reinterpret_cast<volatile uint32_t*>(smem + C::kTaddrOff);
  volatile int* abort_f = reinterpret_cast<volatile int*>(smem + C::kAbortOff);

  if (tid == 0) {
    // one set of converter warps (8) fills each block
    for (int i = B_FULL0; i <= B_FULL2; ++i) mbar_init(bar(i), kConvWarps / 2);
    for (int i = B_EMPTY0; i <= B_SFULL1; ++i) mbar_init(bar(i), 1);
    mbar_init(bar(B_SEMPTY0), kSoftWarps);
    mbar_init(bar(B_SEMPTY1), kSoftWarps);
    mbar_init(bar(B_PFULL0), kSoftWarps);
    mbar_init(bar(B_PFULL1), kSoftWarps);
    mbar_init(bar(B_ODONE), 1);
    mbar_init(bar(B_QDONE), 1);
    mbar_init(bar(B_QRAW), 1);
    mbar_init(bar(B_QREADY), kSoftWarps);
    for (int i = B_RAWFULL0; i <= B_RAWFULL3; ++i) mbar_init(bar(i), 1);
    for (int i = B_RAWEMPTY0; i <= B_RAWEMPTY2; ++i) mbar_init(bar(i), kConvWarps / 4);
    *abort_f = 0;
    fence_mbar_init();
  }
  if (tid < 2 * NH) mbuf[tid] = -INFINITY;
  if (warp == kMmaWarp) {
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
  // SS: S^T buffer u at columns [2 NH u, 2 NH (u + 1)), O^T block mb at 4 NH + mb NH;
  // TS: Q at 0..127, S at 128..255, O^T block mb at 256 + mb NH
  const uint32_t tQ = tmem + C::kTQ;
  const uint32_t tS = tmem + C::kTS_S;
  const uint32_t tO = tmem + C::kTO;

  if (warp >= kMmaWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsMma) : "memory");
    // ===================== MMA issuer =====================
    // Q in shared memory: warp kMmaWarp issues the score MMAs, warp kMmaWarp + 1 the
    // value products, each waiting (suspending) on its own barriers only.  Q in tensor
    // memory (one scores buffer): warp kMmaWarp issues both in readiness order, which
    // measured faster there (two issuers interleave a block's value product with the
    // next block's scores in the tensor pipe and delay both).
    constexpr bool kTwoIssuers = !C::kTS;
    const bool qk_issuer = warp == kMmaWarp, pv_issuer = kTwoIssuers && warp == kMmaWarp + 1;
    if ((qk_issuer || pv_issuer) && lane == 0 && nb > 0) {
      // The bf16 q rows h0..h0+NH-1 (NH KB) into block buffer kQRawBuf, where the
      // softmax warps convert them into the stacked Q operand: SS as they are
      // (contiguous rows), TS as 8 swizzled boxes of 64 columns (box c at c NH 128
      // bytes).
      if (qk_issuer) {
        mbar_arrive_expect_tx(bar(B_QRAW), NH * 1024);
        if constexpr (C::kTS) {
#pragma unroll
          for (int c = 0; c < 8; ++c)
            tma_load_2d(sbase + C::kQRawBuf * kBuf + c * NH * 128, &rows.q, 64 * c, b * H + h0,
                        bar(B_QRAW));
        } else {
          const uint8_t* src =
              reinterpret_cast<const uint8_t*>(q + (static_cast<int64_t>(b) * H + h0) * kQkDim);
#pragma unroll
          for (int k = 0; k < NH / 16; ++k)
            bulk_g2s(sbase + C::kQRawBuf * kBuf + k * 16384, src + k * 16384, 16384, bar(B_QRAW));
        }
      }
      // SS: S^T (tokens x stacked heads) = stacked K . stacked Q^T, both from shared
      // memory; TS: S (stacked heads x stacked tokens) = Q (tensor memory) . K^T.
      // PV: O^T += V^T . P with V^T the MN-major view of the block; P is MN-major
      // ([token][head]) in SS, K-major ([head][token]) in TS.
      constexpr uint32_t kIdescQK = idesc_f16(128, C::kTS ? 128 : 2 * NH, false, false);
      constexpr uint32_t kIdescPV = idesc_f16(128, NH, true, !C::kTS);
      // Descriptors as 32-bit halves: moving a start address by X bytes adds X >> 4 to
      // the low half (addresses stay below 256 KB, so the 14-bit field never
      // carries); the high halves (stride, swizzle) are fixed.
      // Every A/B operand here shares one high half (stride 1024, 128-byte swizzle); the
      // low halves differ from lK (start sbase, leading offset 16) by constants: the
      // start field (bits 0-13) by the byte offset >> 4, the leading-offset field
      // (bits 16-29) by the change of the leading offset >> 4.
      const uint64_t dK = smem_desc(sbase, 16, 1024, SWZ_128B);
      const uint64_t dP = C::kTS ? smem_desc(sbase + C::kPOff, 16, 1024, SWZ_128B)
                                 : smem_desc(sbase + C::kPOff, 8 * C::kPRow, 8 * C::kPRow, C::kPSwz);
      const uint32_t hi = static_cast<uint32_t>(dK >> 32);
      const uint32_t hiP = static_cast<uint32_t>(dP >> 32);
      uint32_t lK = static_cast<uint32_t>(dK), lP = static_cast<uint32_t>(dP);
      constexpr uint32_t kLbo16 = 16 >> 4;
      auto lo_of = [](uint32_t start_off, uint32_t lbo) {
        return (start_off >> 4) + (((lbo >> 4) - kLbo16) << 16);
      };
      // value block 3 pairs columns 384..447 (slab 2, rows 64..127) with the constant
      // block: leading offset (ones - a_start) shrinks by 2048 bytes per K step
      constexpr uint32_t kV3 = 2 * kSlab + 64 * 128;
      // Makes the bases opaque, so each MMA's operands are one add at the point of
      // use rather than values computed ahead (the issuer runs on few registers).
      auto opaque = [&]() { asm volatile("" : "+r"(lK), "+r"(lP)); };
      auto wait = [&](int i, uint32_t par) {
        const bool r = wait_or_abort(bar(i), par, abort_f, limit);
        tc_fence_after();
        opaque();
        return r;
      };
      bool ok = true;
      auto qk = [&](int i) {
        const int u = i & 1;                 // scores buffer (SS)
        const int kb = i % C::kNBuf;         // block buffer
        const uint32_t aK = lK + static_cast<uint32_t>((kb * kBuf) >> 4);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if constexpr (C::kTS)   // K step 16: 8 columns of Q, 32 bytes of the slab
              mma_f16_ts_hl(tS, tQ + static_cast<uint32_t>(8 * (4 * j + k)),
                            aK + static_cast<uint32_t>((j * kSlab + k * 32) >> 4), hi,
                            kIdescQK, (j | k) != 0 ? 1u : 0u);
            else
              mma_f16_ss_hl(tS + u * 2 * NH, aK + static_cast<uint32_t>((j * kSlab + k * 32) >> 4),
                            hi, lK + lo_of(C::kQOff + j * C::kQSlab + k * 32, 16), hi,
                            kIdescQK, (j | k) != 0 ? 1u : 0u);
          }
        }
        mma_commit(bar(B_SFULL0 + (C::kTS ? 0 : u)));
        opaque();
        return true;
      };
      auto pv = [&](int i) {
        const int kb = i % C::kNBuf;                     // block buffer
        const int pb = C::kPBufs == 2 ? (i & 1) : 0;     // P buffer
        const uint32_t acc0 = i > 0 ? 1u : 0u;
#pragma unroll
        for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            uint32_t a;
            if (mb < 3) {
              a = lK + lo_of(kb * kBuf + (mb & 1) * 2 * kSlab + (mb >> 1) * 64 * 128 + ks * 2048,
                             kSlab);
            } else {
              const uint32_t st = kb * kBuf + kV3 + ks * 2048;
              a = lK + lo_of(st, C::kOnesOff - st);
            }
            // K step of 16 tokens: SS 16 P rows down, TS 32 bytes along each P row
            const uint32_t bP = C::kTS ? static_cast<uint32_t>((pb * C::kPStride + ks * 32) >> 4)
                                       : static_cast<uint32_t>((ks * 16 * C::kPRow) >> 4);
            mma_f16_ss_hl(tO + mb * NH, a, hi, lP + bP, hiP, kIdescPV, ks > 0 ? 1u : acc0);
          }
        }
        mma_commit(bar(B_EMPTY0 + kb));
        opaque();
        return true;
      };
      if (!kTwoIssuers) {
        // Issue order decided by readiness: the value product of block np (its P
        // written) or the scores of block nq (its buffer filled, the scores buffer
        // read by the softmax of block nq - 1; at most one block ahead of the value
        // products), the value product first when both are ready (it frees a block
        // buffer for the converters; measured slightly faster).  Each barrier is
        // tested without suspending (test_wait), so a late converter set or a late
        // softmax holds up only its own block.
        ok = wait(B_QREADY, 0);
        int nq = 0, np = 0;
        long long t_idle = clock64();
#pragma unroll 1
        while (ok && np < nb) {
          if (np < nq && (C::kPBufs == 2 ? mbar_test_wait(bar(B_PFULL0 + (np & 1)), (np >> 1) & 1)
                                         : mbar_test_wait(bar(B_PFULL0), np & 1))) {
            tc_fence_after();
            opaque();
            ok = pv(np);
            ++np;
            t_idle = clock64();
          } else if (nq < nb && nq <= np + 1 &&
                     mbar_test_wait(bar(B_FULL0 + nq % C::kNBuf), (nq / C::kNBuf) & 1) &&
                     (nq < 1 || mbar_test_wait(bar(B_SEMPTY0), (nq - 1) & 1))) {
            tc_fence_after();
            opaque();
            ok = qk(nq);
            ++nq;
            t_idle = clock64();
          } else if (*abort_f) {
            ok = false;
          } else if (clock64() - t_idle > (static_cast<long long>(limit) << 10)) {
            *abort_f = 1;
            record_status(SMLA_ERR_TIMEOUT);
            ok = false;
          }
        }
        mma_commit(bar(B_ODONE));
        // Let the tensor pipe drain before the final barrier (tensor memory is freed
        // after it), also when another role left early.
        if (!ok) mbar_wait(bar(B_ODONE), 0, static_cast<long long>(kWaitLimitK) << 10);
      } else       if (qk_issuer) {
        // scores of block i: its buffer filled, and its scores buffer read by the
        // softmax (TS: one buffer, block i - 1; SS: two, block i - 2)
        ok = wait(B_QREADY, 0);
#pragma unroll 1
        for (int i = 0; ok && i < nb; ++i) {
          ok = wait(B_FULL0 + i % C::kNBuf, (i / C::kNBuf) & 1);
          if (ok && C::kTS && i >= 1) ok = wait(B_SEMPTY0, (i - 1) & 1);
          if (ok && !C::kTS && i >= 2) ok = wait(B_SEMPTY0 + (i & 1), ((i >> 1) - 1) & 1);
          if (ok) ok = qk(i);
        }
        mma_commit(bar(B_QDONE));
        // let the score MMAs drain before tensor memory is freed, also when another
        // role left early
        if (!ok) mbar_wait(bar(B_QDONE), 0, static_cast<long long>(kWaitLimitK) << 10);
      } else {
        // value product of block i: its P written (every earlier value product of the
        // same accumulator was issued before by this thread)
#pragma unroll 1
        for (int i = 0; ok && i < nb; ++i) {
          ok = C::kPBufs == 2 ? wait(B_PFULL0 + (i & 1), (i >> 1) & 1) : wait(B_PFULL0, i & 1);
          if (ok) ok = pv(i);
        }
        mma_commit(bar(B_ODONE));
        if (!ok) mbar_wait(bar(B_ODONE), 0, static_cast<long long>(kWaitLimitK) << 10);
      }
    }
    if (C::kTmaRows && warp == kTmaWarp && nb > 0) {
      // ===================== row gather =====================
      // Half block h (slots 32h .. 32h + 31 of the split) into stage h % kStages, once
      // the converters have taken half block h - kStages out of it.  Lane l handles
      // slot l: the valid rows are ordered even-map rows first, then odd-map rows, each
      // run padded to a multiple of 4 with a copy of its first row, and lane g issues
      // the copy of rows 4g..4g+3.  A masked slot (index -1, past the split, or out of
      // range: reported) is not gathered; its window offset is kNoRow.  Converter
      // group 2 (h / 2 % 2) + h % 2 takes half block h.
      if (lane == 0) {
        prefetch_tensormap(&rows.even);
        prefetch_tensormap(&rows.odd);
      }
      uint16_t* tab = reinterpret_cast<uint16_t*>(smem + C::kTabOff);
      int* list = reinterpret_cast<int*>(smem + C::kListOff);
      const uint32_t stage0 = sbase + C::kStageOff;
      const uint32_t lt = (1u << lane) - 1u;
      const bool split = rows.split != 0;
      const int nh = 2 * nb;
      // The indices of the next four half blocks are in flight, copied asynchronously
      // into a ring of four 32-slot rows (a load's latency is longer than a half
      // block's turn when its stage is free).
      int* iring = reinterpret_cast<int*>(smem + C::kIdxOff);
      auto fetch = [&](int hx) {   // one commit group per half block, empty past the end
        if (hx < nh) {
          const int pos = sp.t_begin + hx * kHalfRows + lane;
          cp_async4(smem_u32(iring + (hx & 3) * kHalfRows + lane),
                    idx_row + (pos < sp.t_end ? pos : sp.t_begin), pos < sp.t_end ? 4u : 0u);
        }
        cp_async_commit();
      };
      fetch(0);
      fetch(1);
      fetch(2);
      fetch(3);
      int issued = 0;
#pragma unroll 1
      for (int h = 0; h < nh; ++h) {
        const int st = h % kStages;
        cp_async_wait<3>();   // half block h's indices have landed
        const int pos = sp.t_begin + h * kHalfRows + lane;
        const int r = pos < sp.t_end ? iring[(h & 3) * kHalfRows + lane] : -1;
        const bool v = idx_ok(r, num_rows, true);
        const bool o = split && (r & 1);
        const uint32_t e = __ballot_sync(0xffffffffu, v && !o);
        const uint32_t d = __ballot_sync(0xffffffffu, v && o);
        fetch(h + 4);         // (r is in use above: its ring row may be refilled)
        const int ne = __popc(e), nep = (ne + 3) & ~3;
        const int no = __popc(d), nop = (no + 3) & ~3;
        const int p = !v ? -1 : o ? nep + __popc(d & lt) : __popc(e & lt);
        const int m = split ? r >> 1 : r;   // map row
        if (h >= kStages && !warp_wait(bar(B_RAWEMPTY0 + st), (h / kStages - 1) & 1, abort_f, limit))
          break;
        tab[st * kHalfRows + lane] =
            p < 0 ? static_cast<uint16_t>(kNoRow)
                  : static_cast<uint16_t>((p >> 2) * kGrp + (p & 3) * kWin + (o ? 8 : 0));
        if (p >= 0) list[p] = m;
        __syncwarp();
        if (lane < nep - ne) list[ne + lane] = list[0];
        if (lane < nop - no) list[nep + no + lane] = list[nep];
        __syncwarp();
        const int ng = (nep + nop) >> 2;
        const uint32_t full = bar(B_RAWFULL0 + 2 * ((h >> 1) & 1) + (h & 1));
        if (lane == 0) mbar_arrive_expect_tx(full, static_cast<uint32_t>(ng * 4 * kWin));
        __syncwarp();
        if (lane < ng) {
          const bool odd_map = 4 * lane >= nep;
          int g[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            g[k] = list[4 * lane + k];
#ifdef SMLA_DEBUG
            // the map row lies inside its map (a row out of range is not copied:
            // row 0 stands in, so the byte count stays right)
            const int64_t extent = !split ? num_rows : odd_map ? num_rows / 2 : (num_rows + 1) / 2;
            if (g[k] < 0 || g[k] >= extent) {
              record_status(SMLA_ERR_INTERNAL);
              g[k] = 0;
            }
#endif
          }
          tma_gather4(stage0 + static_cast<uint32_t>(st * kStageBytes + lane * kGrp),
                      odd_map ? &rows.odd : &rows.even, 0, g[0], g[1], g[2], g[3], full);
        }
        __syncwarp();
        issued = h + 1;
      }
      cp_async_wait<0>();   // no copy into the ring is left in flight
      // Every copy has landed before the CTA can leave.  The halves before the last
      // kStages were taken by the converters (their stages were reused), so only the
      // last kStages can still be in flight; each is the latest phase of its group's
      // barrier.
      if (lane == 0) {
        for (int h = max(0, issued - kStages); h < issued; ++h)
          mbar_wait(bar(B_RAWFULL0 + 2 * ((h >> 1) & 1) + (h & 1)), (h >> 2) & 1,
                    static_cast<long long>(kWaitLimitK) << 10);
      }
      __syncwarp();
    }
    // the copy of q has landed before the CTA can leave
    if (qk_issuer && lane == 0 && nb > 0)
      mbar_wait(bar(B_QRAW), 0, static_cast<long long>(limit) << 10);
    __syncwarp();
    // the two cluster barriers of the merging epilogue, in step with the other roles
    if constexpr (MODE == kMergeCluster) {
      cluster_sync();
      cluster_sync();
    }
  } else if (warp < kSoftWarps) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoft) : "memory");
    if constexpr (C::kTS) {
    // ===================== softmax, Q in tensor memory (64 heads) =====================
    // Thread tid owns tensor-memory lane tid: head h = tid % 64 and the half of the
    // q/k columns (tid / 64) whose partial scores that lane accumulates.  The two
    // threads of a head trade the partial scores of each other's tokens through X and
    // each finishes 32 tokens of the block: thread (h, 0) tokens 0..31, (h, 1) 32..63.
    // The running max of head h lives in a register of both threads.
    const int h = tid & 63, half = tid >> 6;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const int partner = tid ^ 64;
    const bool poller = tid == 0;
    bool ok = nb > 0;
    if (ok) {
      // ---- q row h, columns 256 half .. +255 (bf16) -> f16 pairs in columns 0..127 of
      // this lane: the stacked Q operand; then the constant block of the value product.
      // Phase ph reads box 4 half + ph (64 columns): unit u of row h at u ^ (h % 8).
      ok = group_wait(bar(B_QRAW), 0, abort_f, limit, poller, kBarSoft, 128);
      bool q_bad = false;
      const uint32_t qrow = sbase + C::kQRawBuf * kBuf + static_cast<uint32_t>(h) * 128;
      const uint32_t qsw = static_cast<uint32_t>(h & 7);
#pragma unroll 1
      for (int ph = 0; ok && ph < 4; ++ph) {
        const uint32_t box = qrow + static_cast<uint32_t>((4 * half + ph) * NH * 128);
        float f[32];   // column 32 ph + j: elements 2j, 2j + 1 of the box row (f16 pair)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 c4 = ld_shared_v4(box + ((static_cast<uint32_t>(k) ^ qsw) << 4));
          const uint32_t w[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t hv = bf16x2_to_f16x2(w[j]);
            q_bad |= f16x2_has_inf_or_nan(hv);
            f[4 * k + j] = __uint_as_float(hv);
          }
        }
        tmem_st16(tQ + lane_base + 32 * ph, f);
        tmem_st16(tQ + lane_base + 32 * ph + 16, f + 16);
      }
      tmem_wait_st();
      if (q_bad) record_status(SMLA_ERR_RANGE);
      {   // the constant block: 16 rows x 8 units of 16 B, column 0 = f16 1.0
        const uint32_t r = tid >> 3, unit = tid & 7;
        st_shared_v4(sbase + C::kOnesOff + (r >> 3) * 1024 + swz_offset(r & 7, unit, 128),
                     make_uint4(unit == 0 ? 0x3C00u : 0u, 0u, 0u, 0u));
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_QREADY));
    }
    const int pair_bar = kBarPair0 + (warp & 1);   // warps w and w + 2 hold the two halves
    const int tok0 = 32 * half;
    // score columns: half 0 holds tokens 0..63 at 0..63, half 1 at 64..127; each
    // thread keeps its own tokens and sends the partner's
    const uint32_t send_col = half ? 64u : 32u, keep_col = half ? 96u : 0u;
    // X row r (128 bytes) receives the 32 partial scores for thread r, 16-byte units
    // XOR-swizzled with r so that 8 consecutive rows use 8 distinct bank groups
    const uint32_t xw = sbase + C::kXOff + static_cast<uint32_t>(partner) * 128;
    const uint32_t xr = sbase + C::kXOff + static_cast<uint32_t>(tid) * 128;
    const uint32_t xsw = static_cast<uint32_t>(partner & 7), xsr = static_cast<uint32_t>(tid & 7);
    float* mx = reinterpret_cast<float*>(smem + C::kMxOff);
    float* alph = reinterpret_cast<float*>(smem + C::kAlphaOff);
    float m_run = 0.f;     // running max of head h (log2 units), once have_m
    bool have_m = false;   // a valid token has been seen (every head gets it at once)
    int vraw = ok ? raw_idx(idx_row, sp.t_begin + tok0 + lane, sp.t_end) : -1;
    for (int i = 0; ok && i < nb; ++i) {
      // validity of this thread's 32 tokens: lane j tests token tok0 + j
      const uint32_t vm = __ballot_sync(0xffffffffu, idx_ok(vraw, num_rows, false));
      vraw = i + 1 < nb ? raw_idx(idx_row, sp.t_begin + (i + 1) * kBlk + tok0 + lane, sp.t_end)
                        : -1;
      bool wok = warp_wait(bar(B_SFULL0), i & 1, abort_f, limit);
      float sv[32];
      if (wok) {
        tc_fence_after();
        float x[32];
        tmem_ld16(tS + lane_base + send_col, x);
        tmem_ld16(tS + lane_base + send_col + 16, x + 16);
        tmem_ld16(tS + lane_base + keep_col, sv);
        tmem_ld16(tS + lane_base + keep_col + 16, sv + 16);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_SEMPTY0));   // the scores may be rewritten
#pragma unroll
        for (int k = 0; k < 8; ++k)
          st_shared_v4(xw + ((static_cast<uint32_t>(k) ^ xsw) << 4),
                       make_uint4(__float_as_uint(x[4 * k]), __float_as_uint(x[4 * k + 1]),
                                  __float_as_uint(x[4 * k + 2]), __float_as_uint(x[4 * k + 3])));
      }
      wok = bar_and(pair_bar, 64, wok);   // both threads of every head have written X
      // t = score * scale (log2 units) - running max (0 until the first valid token);
      // masked tokens -inf.  ex: max of t over this thread's tokens; bm: the same before
      // the running max is subtracted.
      float ex = -INFINITY, bm = -INFINITY;
      if (wok) {
        const float base = have_m ? m_run : 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 v = ld_shared_v4(xr + ((static_cast<uint32_t>(k) ^ xsr) << 4));
          sv[4 * k] = fmaf(sv[4 * k] + __uint_as_float(v.x), scale_log2, -base);
          sv[4 * k + 1] = fmaf(sv[4 * k + 1] + __uint_as_float(v.y), scale_log2, -base);
          sv[4 * k + 2] = fmaf(sv[4 * k + 2] + __uint_as_float(v.z), scale_log2, -base);
          sv[4 * k + 3] = fmaf(sv[4 * k + 3] + __uint_as_float(v.w), scale_log2, -base);
        }
        if (vm != 0xffffffffu) {   // (warp-uniform: the tokens are the warp's)
#pragma unroll
          for (int t = 0; t < 32; ++t)
            if (!((vm >> t) & 1u)) sv[t] = -INFINITY;
        }
        float e4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int t = 0; t < 32; ++t) e4[t & 3] = fmaxf(e4[t & 3], sv[t]);
        ex = fmaxf(fmaxf(e4[0], e4[1]), fmaxf(e4[2], e4[3]));
        bm = ex + base;
        if (!have_m && vm != 0u) ex = INFINITY;   // the first valid token sets the max
      }
      // One barrier in the common case: no score passed the running max by more than
      // the headroom.
      if (bar_or(kBarSoft, 128, !wok || ex > kLazyMax)) {
        if (!(ok = bar_and(kBarSoft, 128, wok))) break;   // a wait ran out: leave together
        // the new running max of head h: the old one and both threads' block maxima
        // (finite: a valid token of this block or an earlier one exists)
        mx[tid] = bm;
        bar_sync(kBarSoft, 128);
        const float m_new = fmaxf(have_m ? m_run : -INFINITY, fmaxf(bm, mx[partner]));
        if (have_m) {
          // rescale O (and with it the denominator row) by 2^(m_old - m_new), once the
          // value product of block i - 1 has finished
          if (tid < NH) alph[tid] = exp2f(m_run - m_new);
          if (!(ok = group_wait(bar(B_EMPTY0 + (i - 1) % C::kNBuf), ((i - 1) / C::kNBuf) & 1, abort_f,
                                limit, poller, kBarSoft, 128)))
            break;
          tc_fence_after();
#pragma unroll 1
          for (int hc = 0; hc < NH; hc += 8) {
            float f[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) f[k] = alph[hc + k];
#pragma unroll 1
            for (int mb = 0; mb < 4; ++mb) {
              float o[8];
              tmem_ld<8>(tO + lane_base + mb * NH + hc, o);
              tmem_wait_ld();
#pragma unroll
              for (int k = 0; k < 8; ++k) o[k] *= f[k];
              tmem_st<8>(tO + lane_base + mb * NH + hc, o);
            }
          }
          tmem_wait_st();
        }
        const float d = m_new - (have_m ? m_run : 0.f);
#pragma unroll
        for (int t = 0; t < 32; ++t) sv[t] -= d;
        m_run = m_new;
        have_m = true;
      }
#pragma unroll
      for (int t = 0; t < 32; ++t) sv[t] = fast_exp2(sv[t]);   // 2^-inf = 0 (masked)
      // P buffer pb is free once the value product that last read it (block i - kPBufs)
      // has finished
      const int pb = C::kPBufs == 2 ? (i & 1) : 0;
      const int pj = i - C::kPBufs;
      if (pj < 0 || warp_wait(bar(B_EMPTY0 + pj % C::kNBuf), (pj / C::kNBuf) & 1, abort_f, limit)) {
        // row h of P (128 bytes: tokens 0..63), 16-byte units XOR-swizzled with h & 7
        const uint32_t prow = sbase + C::kPOff + pb * C::kPStride +
                              static_cast<uint32_t>((h >> 3) * 1024 + (h & 7) * 128);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint4 v;
          v.x = pack_f16x2(sv[8 * k + 0], sv[8 * k + 1]);
          v.y = pack_f16x2(sv[8 * k + 2], sv[8 * k + 3]);
          v.z = pack_f16x2(sv[8 * k + 4], sv[8 * k + 5]);
          v.w = pack_f16x2(sv[8 * k + 6], sv[8 * k + 7]);
          st_shared_v4(prow + ((static_cast<uint32_t>(4 * half + k) ^ static_cast<uint32_t>(h & 7)) << 4), v);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_PFULL0 + pb));
      }
    }
    // the final running max into mbuf[0, NH) for the epilogue
    if (tid < NH) mbuf[tid] = have_m ? m_run : 0.f;
    } else {
    // ===================== softmax (and q conversion) =====================
    const int t = tid & (kBlk - 1);          // token of the block (tensor-memory lane tid)
    const bool upper = tid >= kBlk;          // this lane holds the columns 256..511 half
    const int keep0 = upper ? HH : 0;        // heads this thread finishes
    const int send0 = upper ? 0 : HH;        // heads it hands to the other half's thread
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t scol = upper ? NH : 0;
    const bool poller = tid == 0;
    // score halves traded through X: row t, 16-byte chunks XOR-swizzled with t
    const uint32_t xrow = sbase + C::kXOff + static_cast<uint32_t>(t * NH * 4);
    const uint32_t xsw = static_cast<uint32_t>(t & (NH / 4 < 8 ? NH / 4 - 1 : 7));
    bool ok = nb > 0;
    int cur = 0;
    bool have_m = false;   // the running max is set (a valid token has been seen)
    if (ok) {
      // ---- q: bf16 rows staged in buffer 1 -> stacked f16 Q operand; constant block
      ok = group_wait(bar(B_QRAW), 0, abort_f, limit, poller, kBarSoft, 128);
      if (ok) {
        bool q_bad = false;
#pragma unroll 4
        for (int k = 0; k < NH * 64 / 128; ++k) {
          const int ui = tid + 128 * k, h = ui >> 6, u = ui & 63;
          const uint4 v = ld_shared_v4(sbase + C::kQRawBuf * kBuf + ui * 16);
          const uint4 o = make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y),
                                     bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
          q_bad |= f16x2_has_inf_or_nan(o.x) | f16x2_has_inf_or_nan(o.y) |
                   f16x2_has_inf_or_nan(o.z) | f16x2_has_inf_or_nan(o.w);
          // column 8u..8u+7: half u / 32, slab (u / 8) % 4, unit u % 8; row h + NH half
          const int n = h + NH * (u >> 5);
          st_shared_v4(sbase + C::kQOff + ((u >> 3) & 3) * C::kQSlab + n * 128 +
                           (((u & 7) ^ (n & 7)) << 4),
                       o);
        }
        if (q_bad) record_status(SMLA_ERR_RANGE);
        {   // the constant block: 16 rows x 8 units of 16 B, column 0 = f16 1.0
          const uint32_t r = tid >> 3, unit = tid & 7;
          st_shared_v4(sbase + C::kOnesOff + (r >> 3) * 1024 + swz_offset(r & 7, unit, 128),
                       make_uint4(unit == 0 ? 0x3C00u : 0u, 0u, 0u, 0u));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_QREADY));
      }
    }
    // Each warp waits for its scores and for the P buffer on its own; warps w and w ^ 2
    // (the two halves of the same tokens) meet at a 64-thread barrier to trade their
    // halves, and all four meet once per block for the lazy-max vote.  Every warp
    // executes the same sequence of named barriers whatever its verdicts, and a failed
    // wait makes the vote fire, where the verdict is made uniform and the loop left.
    const int pair_bar = kBarPair0 + (warp & 1);
    int vraw = ok ? raw_idx(idx_row, sp.t_begin + t, sp.t_end) : -1;
    for (int i = 0; ok && i < nb; ++i) {
      const int u = i & 1;
      const bool valid = idx_ok(vraw, num_rows, false);
      vraw = i + 1 < nb ? raw_idx(idx_row, sp.t_begin + (i + 1) * kBlk + t, sp.t_end) : -1;
      bool wok = warp_wait(bar(B_SFULL0 + u), (i >> 1) & 1, abort_f, limit);
      const uint32_t scols = tS + lane_base + u * 2 * NH + scol;
      float sv[HH];
      if (wok) {
        tc_fence_after();
        // the half handed over first (8 columns at a time), then the half kept
#pragma unroll
        for (int c8 = 0; c8 < HH; c8 += 8) {
          float x[8];
          tmem_ld<8>(scols + send0 + c8, x);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 2; ++k)
            st_shared_v4(xrow + ((static_cast<uint32_t>((send0 + c8) / 4 + k) ^ xsw) << 4),
                         make_uint4(__float_as_uint(x[4 * k]), __float_as_uint(x[4 * k + 1]),
                                    __float_as_uint(x[4 * k + 2]), __float_as_uint(x[4 * k + 3])));
        }
        tmem_ld_n<HH>(scols + keep0, sv);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_SEMPTY0 + u));   // scores buffer u may be rewritten
      }
      wok = bar_and(pair_bar, 64, wok);                   // both halves of the tokens are in X
      // t = score * scale (log2 units) - running max (0 until the first valid token
      // sets the max: every head gets its first finite max at that same block);
      // masked tokens -inf
      float ex = -INFINITY;
      if (wok) {
        const float* m_old = mbuf + cur * NH + keep0;
#pragma unroll
        for (int k = 0; k < HH / 4; ++k) {
          const uint4 v = ld_shared_v4(xrow + ((static_cast<uint32_t>(keep0 / 4 + k) ^ xsw) << 4));
          float4 m4 = *reinterpret_cast<const float4*>(m_old + 4 * k);
          if (!have_m) m4 = make_float4(0.f, 0.f, 0.f, 0.f);
          sv[4 * k] = fmaf(sv[4 * k] + __uint_as_float(v.x), scale_log2, -m4.x);
          sv[4 * k + 1] = fmaf(sv[4 * k + 1] + __uint_as_float(v.y), scale_log2, -m4.y);
          sv[4 * k + 2] = fmaf(sv[4 * k + 2] + __uint_as_float(v.z), scale_log2, -m4.z);
          sv[4 * k + 3] = fmaf(sv[4 * k + 3] + __uint_as_float(v.w), scale_log2, -m4.w);
        }
        if (valid) {
          float e4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int h = 0; h < HH; ++h) e4[h & 3] = fmaxf(e4[h & 3], sv[h]);
          ex = fmaxf(fmaxf(e4[0], e4[1]), fmaxf(e4[2], e4[3]));
          if (!have_m) ex = INFINITY;   // the first valid token sets the running max
        } else {
#pragma unroll
          for (int h = 0; h < HH; ++h) sv[h] = -INFINITY;
        }
      }
      // One barrier in the common case: no score passed the running max by more than
      // the headroom.  (It also ends every thread's reads of X for this block.)
      if (bar_or(kBarSoft, 128, !wok || ex > kLazyMax)) {
        if (!(ok = bar_and(kBarSoft, 128, wok))) break;   // a wait ran out: leave together
        // Raise the running max to the exact block max; rescale O (and with it the
        // denominator row) by 2^(m_old - m_new).  Warps 0-1 hold heads [0, NH/2),
        // warps 2-3 heads [NH/2, NH), 32 tokens each.
        const float* m_old = mbuf + cur * NH;
        float* m_new = mbuf + (cur ^ 1) * NH;
        // block max per head through X (free again: every thread has read its half),
        // transposed with a skew of 65 floats per head so both the writes (one head,
        // consecutive tokens) and the reads (consecutive heads) are conflict-free
        float* xt = reinterpret_cast<float*>(smem + C::kXOff);
#pragma unroll
        for (int h = 0; h < HH; ++h)
          xt[(keep0 + h) * 65 + t] = have_m ? sv[h] + m_old[keep0 + h] : sv[h];
        bar_sync(kBarSoft, 128);
        if (tid < NH) {
          float m = -INFINITY;
#pragma unroll 8
          for (int tk = 0; tk < kBlk; ++tk) m = fmaxf(m, xt[tid * 65 + tk]);
          m_new[tid] = fmaxf(m_old[tid], m);
        }
        bar_sync(kBarSoft, 128);
        if (have_m) {
          // O holds the value products up to block i - 1: let the last one finish
          if (!(ok = group_wait(bar(B_EMPTY0 + (i - 1) % C::kNBuf), ((i - 1) / C::kNBuf) & 1, abort_f,
                                limit, poller, kBarSoft, 128)))
            break;
          tc_fence_after();
#pragma unroll 1
          for (int hc = 0; hc < NH; hc += 8) {
            float f[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) f[k] = exp2f(m_old[hc + k] - m_new[hc + k]);
#pragma unroll 1
            for (int mb = 0; mb < 4; ++mb) {
              float o[8];
              tmem_ld<8>(tO + lane_base + mb * NH + hc, o);
              tmem_wait_ld();
#pragma unroll
              for (int k = 0; k < 8; ++k) o[k] *= f[k];
              tmem_st<8>(tO + lane_base + mb * NH + hc, o);
            }
          }
          tmem_wait_st();
        }
        // re-base t on the new max
#pragma unroll
        for (int h = 0; h < HH; ++h)
          sv[h] = sv[h] + ((have_m ? m_old[keep0 + h] : 0.f) - m_new[keep0 + h]);
        have_m = true;
        cur ^= 1;
      }
#pragma unroll
      for (int h = 0; h < HH; ++h) sv[h] = fast_exp2(sv[h]);   // 2^-inf = 0 (masked)
      // P is single-buffered: the value product of block i - 1 must have read it.  A
      // warp whose wait runs out skips its part of P; the abort flag it set makes the
      // next block's vote fire (or the MMA warp give up on this block's P).
      if (i == 0 || warp_wait(bar(B_EMPTY0 + (i - 1) % C::kNBuf), ((i - 1) / C::kNBuf) & 1, abort_f,
                              limit)) {
        const uint32_t prow = sbase + C::kPOff;   // row t: token-major, heads contiguous
#pragma unroll
        for (int k = 0; k < HH / 8; ++k) {
          uint4 v;
          v.x = pack_f16x2(sv[8 * k + 0], sv[8 * k + 1]);
          v.y = pack_f16x2(sv[8 * k + 2], sv[8 * k + 3]);
          v.z = pack_f16x2(sv[8 * k + 4], sv[8 * k + 5]);
          v.w = pack_f16x2(sv[8 * k + 6], sv[8 * k + 7]);
          st_shared_v4(prow + swz_offset(t, keep0 / 8 + k, C::kPRow), v);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_PFULL0));
      }
    }
    // the final running max into mbuf[0, NH) for the epilogue
    bar_sync(kBarSoft, 128);
    if (cur == 1 && tid < NH) mbuf[tid] = mbuf[NH + tid];
    }
    bar_sync(kBarEpi, kSoftWarps * 32 + kConv);
    // the two cluster barriers of the merging epilogue, in step with the other roles
    if constexpr (MODE == kMergeCluster) {
      cluster_sync();
      cluster_sync();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsConv) : "memory");
    // ===================== converters =====================
    // Two sets of 8 warps: set 0 fills buffer 0 with the even blocks, set 1 buffer 1
    // with the odd blocks.  A warp converts 8 rows of its block (two quads of 4 rows, 8
    // lanes per row) from registers, then fetches the same rows of its next block (two
    // blocks on) into registers, so each warp holds one block ahead:
    //   kTmaRows (64 heads): out of the staging ring (gathered by tensor copies),
    //   which frees the stage for another gather; warps 0-3 of a set (group 2 set)
    //   take the first half of each block, warps 4-7 (group 2 set + 1) the second;
    //   otherwise (16 and 32 heads): by its own loads from the cache.
    const int cw = warp - kConvWarp0;            // 0..15
    const int wt = tid - kConvWarp0 * 32;        // 0..511
    const int set = cw >> 3;
    const int q8 = lane & 7;                     // word lane within the row
    const int rb0 = 8 * (cw & 7) + (lane >> 3);  // row of quad 0 (quad 1: + 4)
    const int row_lane0 = lane & ~7;             // lane q = 0 of this row (holds the scales)
    uint2 c[2][kSlots];                          // [quad][slot]
    bool ok = set < nb;
    const int hq = (cw >> 2) & 1;                // half of the block this warp takes
    const uint16_t* tab = reinterpret_cast<const uint16_t*>(smem + C::kTabOff);
    // kTmaRows: block i's rows from its stage into c (a masked slot reads as
    // zeros)
    auto take_rows = [&](int i) -> bool {
      const int h = 2 * i + hq, st = h % kStages;
      if (!warp_wait(bar(B_RAWFULL0 + 2 * set + hq), (i >> 1) & 1, abort_f, limit)) return false;
      const uint32_t stage = sbase + C::kStageOff + static_cast<uint32_t>(st * kStageBytes);
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const uint32_t off = tab[st * kHalfRows + rb0 - kHalfRows * hq + 4 * g];
        const uint32_t a = stage + off + 8u * static_cast<uint32_t>(q8);
        const bool has = off != kNoRow;
#pragma unroll
        for (int k = 0; k < 9; ++k) c[g][k] = has ? ld_shared_v2(a + 64u * k) : make_uint2(0u, 0u);
        c[g][9] = has && q8 == 0 ? ld_shared_v2(a + 576u) : make_uint2(0u, 0u);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_RAWEMPTY0 + st));
      return true;
    };
    // otherwise: rows loaded from the cache
    int nraw[2] = {-1, -1};                      // stored indices of the rows, 2 blocks ahead
    auto row_of = [&](int raw, bool report) -> const uint8_t* {
      if (!idx_ok(raw, num_rows, report)) return nullptr;
#ifdef SMLA_DEBUG
      // the row's 584 bytes lie inside the cache
      if (static_cast<int64_t>(raw) * stride + kRowBytes > num_rows * stride) {
        record_status(SMLA_ERR_INTERNAL);
        return nullptr;
      }
#endif
      return kv + static_cast<int64_t>(raw) * stride;
    };
    auto load_rows = [&](int i) {   // rows of block i (nraw) into c; indices of block i + 2
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const uint8_t* row = row_of(i < nb ? nraw[g] : -1, q8 == 0);
#pragma unroll
        for (int k = 0; k < 9; ++k) c[g][k] = load_word(row, q8 + 8 * k);
        c[g][9] = load_word(q8 == 0 ? row : nullptr, 72);
        nraw[g] = raw_idx(idx_row, sp.t_begin + (i + 2) * kBlk + rb0 + 4 * g, sp.t_end);
      }
    };
    if (C::kTmaRows && ok) {
      ok = take_rows(set);
    } else if (ok) {
#pragma unroll
      for (int g = 0; g < 2; ++g)
        nraw[g] = raw_idx(idx_row, sp.t_begin + set * kBlk + rb0 + 4 * g, sp.t_end);
      // Every CTA starts at once: block 0's rows are requested alone first, so they
      // are not interleaved with block 1's in the memory queues; set 1 issues its
      // first loads once block 0 is converted.
      if (set == 1) ok = warp_wait(bar(B_FULL0), 0, abort_f, limit);
      if (ok) load_rows(set);
    }
    // Word q + 8k (k < 7) of row r lands in slab k & 3, row r + 64 (k >> 2), 16-byte
    // unit q (XOR-swizzled with the row): this lane's base plus a compile-time offset.
    const uint32_t rx0 = static_cast<uint32_t>(rb0 & 7);
    // Converts quad g (runtime 0 or 1) of block i from d (its register slots).  One
    // copy of this code serves both quads, and the checked path of unusual scale
    // bytes is a call, so the converters' loop stays small in the instruction cache.
    auto convert = [&](const uint2 (&d)[kSlots], int g, int i) {
      const uint32_t rx = rx0 ^ (4u * g);
      const uint32_t rowq = static_cast<uint32_t>(rb0 + 4 * g) * 128;
      const uint32_t buf = sbase + (i % C::kNBuf) * kBuf;
      // scale word of this lane's row (word 56: slot 7 of lane q = 0)
      const uint32_t lo = __shfl_sync(0xffffffffu, d[7].x, row_lane0);
      const uint32_t hi = __shfl_sync(0xffffffffu, d[7].y, row_lane0);
      const bool masked = (lo | (hi & 0x00ffffffu)) == 0u;   // a zero-filled row
      const bool fast = __all_sync(0xffffffffu, masked || scales_fast(lo, hi));
      // f16 exponent field (s - 112) << 2 of each group's scale; byte 7 stays zero
      const uint32_t tlo = masked ? 0u : (lo - 0x70707070u) << 2;
      const uint32_t thi = masked ? 0u : ((hi & 0x00ffffffu) - 0x00707070u) << 2;
      const uint32_t an = buf + rowq + ((static_cast<uint32_t>(q8) ^ rx) << 4);
      // FAST: every scale byte of the warp's rows in [113, 134] (exact f16x2 multiply);
      // otherwise the checked fp32 path, out of line.  One branch per quad.
      if (fast) {
#pragma unroll
        for (int k = 0; k < 7; ++k) {
          // prmt: scale byte k of (tlo, thi) into bits 8..15 and 24..31, zero elsewhere
          const uint32_t m = prmt2(tlo, thi, 0x0707u + 0x1010u * k);
          st_shared_v4(an + (k & 3) * kSlab + (k >> 2) * 64 * 128, dq8_fast(d[k].x, d[k].y, m));
        }
      } else {
#pragma unroll
        for (int k = 0; k < 7; ++k) {
          const uint32_t sb = ((k < 4 ? lo : hi) >> (8 * (k & 3))) & 0xffu;
          st_shared_v4(an + (k & 3) * kSlab + (k >> 2) * 64 * 128, dequant8_checked(d[k].x, d[k].y, sb));
        }
      }
      // rope: word 56 + q (slot 7, q >= 1), 64 + q (slot 8), 72 (slot 9, q = 0) is
      // rope word r = w - 57: f16 8 bytes at unit r / 2, half r % 2 of the rope row
      // (range: a bf16 magnitude >= 0x4780 = 65536, or inf / NaN, is beyond the f16
      // range; one 16-bit SIMD max of the magnitudes, tested once)
      uint32_t mag = 0u;
      const uint32_t rope_base = buf + 3 * kSlab + 64 * 128 + rowq;
      auto rope = [&](int r, uint2 v2) {
        mag = __vmaxu2(mag, __vmaxu2(v2.x & 0x7fff7fffu, v2.y & 0x7fff7fffu));
        const uint2 v = make_uint2(bf16x2_to_f16x2(v2.x), bf16x2_to_f16x2(v2.y));
        st_shared_v2(rope_base + (((static_cast<uint32_t>(r) >> 1) ^ rx) << 4) + (r & 1) * 8, v);
      };
      if (q8 >= 1) rope(q8 - 1, d[7]);
      rope(q8 + 7, d[8]);
      if (q8 == 0) rope(15, d[9]);
      if (__vcmpgeu2(mag, 0x47804780u) != 0u) record_status(SMLA_ERR_RANGE);
    };
    for (int i = set; ok && i < nb; i += 2) {
      const int u = i % C::kNBuf;
      // buffer u is free once the value product of block i - kNBuf is done; buffer
      // kQRawBuf first holds the staged q rows until the softmax warps have converted
      // them
      if (i >= C::kNBuf)
        ok = warp_wait(bar(B_EMPTY0 + u), ((i / C::kNBuf) - 1) & 1, abort_f, limit);
      else if (i == C::kQRawBuf)
        ok = warp_wait(bar(B_QREADY), 0, abort_f, limit);
      if (!ok) break;
      convert(c[0], 0, i);
      convert(c[1], 1, i);
      fence_proxy_async_smem();
      __syncwarp();
      // (the test hook withholds one warp's arrival, so the MMA warp's wait runs out)
      if (lane == 0 && !(i == fault_block && (cw & 7) == 0)) mbar_arrive(bar(B_FULL0 + u));
      if (i + 2 < nb) {
        if constexpr (C::kTmaRows)
          ok = take_rows(i + 2);
        else
          load_rows(i + 2);
      }
    }

    // ===================== epilogue =====================
    const bool have_o = nb > 0 && group_wait(bar(B_ODONE), 0, abort_f, limit, wt == 0, kBarConv,
                                             kConv);
    if (have_o) tc_fence_after();
    bar_sync(kBarEpi, kSoftWarps * 32 + kConv);   // the softmax's final max is in mbuf
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    // Clustered launch: the block buffers (free once every MMA is done) hold this
    // split's partial o_s [NH][448] (not yet divided by the denominators), its lse_s
    // [NH] and 1/denominator rinv_s [NH], which the other splits of the cluster read,
    // and the merge weights of the heads this CTA merges.
    float* o_s = reinterpret_cast<float*>(smem);
    float* lse_s = o_s + NH * kNope;
    float* rinv_s = lse_s + NH;
    float* wgt = rinv_s + NH;                // [NH][kMaxCluster]
    float* fin = wgt + NH * kMaxCluster;     // [NH] final lse (natural log)
    const uint32_t o_s_addr = sbase, lse_s_addr = sbase + 4u * NH * kNope,
                   rinv_s_addr = lse_s_addr + 4u * NH;
    // Warp (value block mb, quarter qd) holds O^T rows 128 mb + 32 qd + lane: value
    // column d, all NH heads, in one batch of tensor-memory loads.  Row 448 (block 3,
    // quarter 2, lane 0) is sum_t P[t], the denominators.
    const int mb = cw >> 2;
    const int d = mb * 128 + (warp & 3) * 32 + lane;
    float o[NH];
    if (have_o) {
#pragma unroll
      for (int cc = 0; cc < NH / 16; ++cc) tmem_ld16(tO + lane_base + mb * NH + 16 * cc, o + 16 * cc);
      tmem_wait_ld();
    } else {
#pragma unroll
      for (int k = 0; k < NH; ++k) o[k] = 0.f;
    }
    if (d == kNope) {
#pragma unroll
      for (int k = 0; k < NH; ++k) lfin[k] = o[k];
    }
    if constexpr (MODE == kMergeCluster) {
      if (d < kNope) {
#pragma unroll
        for (int k = 0; k < NH; ++k) o_s[k * kNope + d] = o[k];
      }
    }
    bar_sync(kBarConv, kConv);
    if (wt < NH) {
      const float lt = lfin[wt];
      const float lse = lt > 0.f ? (mbuf[wt] + log2f(lt)) * kLn2 : -INFINITY;
      const float ri = lt > 0.f ? 1.0f / lt : 0.f;
      if constexpr (MODE == kMergeCluster) {   // read by the other splits of the cluster
        lse_s[wt] = lse;
        rinv_s[wt] = ri;
      } else {
        lse_part[(static_cast<int64_t>(b) * H + h0 + wt) * S + s] = lse;
        rinv[wt] = ri;
      }
    }
    if constexpr (MODE != kMergeCluster) {
      bar_sync(kBarConv, kConv);
      if (d < kNope) {
        const int64_t hstride = static_cast<int64_t>(S) * kNope;
        float* dst = o_part + ((static_cast<int64_t>(b) * H + h0) * S + s) * kNope + d;
#pragma unroll
        for (int k = 0; k < NH; ++k) dst[k * hstride] = o[k] * rinv[k];
      }
    }
    if constexpr (MODE == kMergeCluster) {
      cluster_sync();   // every split of this (query, head group) holds its partial
      // This CTA merges heads [h_lo, h_hi), reading the other splits' partials from
      // their shared memory (split r is cluster rank r): weights exp(lse_r - lse) / l_r.
      const int h_lo = s * NH / S, h_hi = (s + 1) * NH / S, nh = h_hi - h_lo;
      if (wt < nh) {
        float x[kMaxCluster], ri[kMaxCluster];
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r) {
          const uint32_t off = 4u * static_cast<uint32_t>(h_lo + wt);
          x[r] = r < S ? ld_dsmem_f32(dsmem_addr(lse_s_addr + off, static_cast<uint32_t>(r)))
                       : -INFINITY;
          ri[r] = r < S ? ld_dsmem_f32(dsmem_addr(rinv_s_addr + off, static_cast<uint32_t>(r))) : 0.f;
        }
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
        for (int r = 0; r < kMaxCluster; ++r) wgt[wt * kMaxCluster + r] = x[r] * inv * ri[r];
        fin[wt] = sum > 0.f ? M + logf(sum) : -INFINITY;
      }
      bar_sync(kBarConv, kConv);
      const int units = nh * (kNope / 4);
      // two units of 4 value columns per thread and round, so that 2 S loads from the
      // other CTAs' shared memory are in flight together
      for (int u0 = wt; u0 < units; u0 += 2 * kConv) {
        bool act[2];
        int hl[2], d4[2];
        uint32_t src[2];
        float4 acc[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int uu = u0 + j * kConv;
          act[j] = uu < units;
          hl[j] = act[j] ? uu / (kNope / 4) : 0;
          d4[j] = act[j] ? uu % (kNope / 4) : 0;
          src[j] = o_s_addr + 4u * static_cast<uint32_t>((h_lo + hl[j]) * kNope + 4 * d4[j]);
          acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int r0 = 0; r0 < kMaxCluster; r0 += 4) {
          float4 v[2][4];
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int r = 0; r < 4; ++r)
              if (act[j] && r0 + r < S) v[j][r] = ld_dsmem_v4(dsmem_addr(src[j], static_cast<uint32_t>(r0 + r)));
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              if (act[j] && r0 + r < S) {
                const float ws = wgt[hl[j] * kMaxCluster + r0 + r];
                acc[j].x = fmaf(ws, v[j][r].x, acc[j].x);
                acc[j].y = fmaf(ws, v[j][r].y, acc[j].y);
                acc[j].z = fmaf(ws, v[j][r].z, acc[j].z);
                acc[j].w = fmaf(ws, v[j][r].w, acc[j].w);
              }
            }
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          if (!act[j]) continue;
          const __nv_bfloat162 lo = __floats2bfloat162_rn(acc[j].x, acc[j].y);
          const __nv_bfloat162 hi = __floats2bfloat162_rn(acc[j].z, acc[j].w);
          uint2 pk;
          pk.x = *reinterpret_cast<const uint32_t*>(&lo);
          pk.y = *reinterpret_cast<const uint32_t*>(&hi);
          *reinterpret_cast<uint2*>(out + (static_cast<int64_t>(b) * H + h0 + h_lo + hl[j]) * kNope +
                                    4 * d4[j]) = pk;
        }
      }
      if (wt < nh) lse_out[static_cast<int64_t>(b) * H + h0 + h_lo + wt] = fin[wt];
      cluster_sync();   // the other splits have finished reading this CTA's shared memory
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Once per (device, kernel): shared-memory size and the register check (the
// setmaxnreg split assumes the launch allocation; a build that differs is refused,
// since its register increase would never be granted).  Thread-safe.
constexpr int kMaxDevices = 64;
std::mutex g_cfg_mu;

template <int NH, int MODE>
cudaError_t configure(int dev) {
  static bool configured[kMaxDevices] = {};
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_cfg_mu);
  if (configured[dev]) return cudaSuccess;
  using C = Cfg<NH>;
  cudaError_t e = cudaFuncSetAttribute(split_kernel<NH, MODE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, split_kernel<NH, MODE>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidKernelImage;
  configured[dev] = true;
  return cudaSuccess;
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime (the
// library does not link against the driver library).
using EncodeTiledFn = decltype(&cuTensorMapEncodeTiled);
EncodeTiledFn encode_tiled() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult found = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &found) != cudaSuccess ||
        found != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// The tensor maps of a launch: the gather maps of a cache of num_rows (>= 1) rows,
// `stride` bytes apart (a multiple of 8, >= 584), starting at the 16-byte aligned kv
// (elements of 8 bytes, boxes of one 74-word window), and the map of the 16-byte
// aligned q [q_rows][512] bf16 (boxes of 64 columns x nh rows, 128-byte swizzle).
cudaError_t row_maps(const void* kv, int64_t num_rows, int64_t stride, const void* q,
                     int64_t q_rows, int nh, RowMaps* m) {
  const EncodeTiledFn encode = encode_tiled();
  if (encode == nullptr) return cudaErrorNotSupported;
  std::memset(static_cast<void*>(m), 0, sizeof(RowMaps));
  const bool split = (stride % 16) != 0;
  const cuuint64_t pitch[1] = {static_cast<cuuint64_t>(split ? 2 * stride : stride)};
  const cuuint32_t box[2] = {kWinWords, 1};
  const cuuint32_t step[2] = {1, 1};
  auto make = [&](CUtensorMap* map, const uint8_t* base, cuuint64_t words, cuuint64_t rows_) {
    const cuuint64_t dim[2] = {words, rows_};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<uint8_t*>(base), dim, pitch,
                  box, step, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  };
  const uint8_t* base = static_cast<const uint8_t*>(kv);
  // indices are int32: rows at or past 2^31 are never gathered, so the maps stop there
  if (num_rows > (int64_t{1} << 31)) num_rows = int64_t{1} << 31;
  // even: the row's 73 words (the window's last word lies past the extent: zero-filled)
  if (make(&m->even, base, kRowBytes / 8, split ? (num_rows + 1) / 2 : num_rows) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (split && num_rows >= 2) {
    // odd: the window of row 2k + 1 starts 8 bytes before the row and ends with it
    if (make(&m->odd, base + stride - 8, kWinWords, num_rows / 2) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  } else {
    m->odd = m->even;
  }
  m->split = split ? 1 : 0;
  const cuuint64_t qdim[2] = {static_cast<cuuint64_t>(kQkDim), static_cast<cuuint64_t>(q_rows)};
  const cuuint64_t qpitch[1] = {static_cast<cuuint64_t>(kQkDim * 2)};
  const cuuint32_t qbox[2] = {64, static_cast<cuuint32_t>(nh)};
  if (encode(&m->q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q), qdim, qpitch, qbox,
             step, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
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
  RowMaps maps;   // (read only by the kernels that gather by tensor copies)
  std::memset(static_cast<void*>(&maps), 0, sizeof(RowMaps));
  if (C::kTmaRows) {
    e = row_maps(kv, num_rows, stride, q, static_cast<int64_t>(B) * H, NH, &maps);
    if (e != cudaSuccess) return e;
  }
  const dim3 grid(S, H / NH, B);
  const float scale_log2 = softmax_scale * 1.4426950408889634f;
  return launch_programmatic(split_kernel<NH, kSplitOnly>, grid, dim3(kThreads), C::kSmemBytes,
                             stream, static_cast<const uint16_t*>(q),
                             static_cast<const uint8_t*>(kv), maps, indices, o_part, lse_part,
                             static_cast<__nv_bfloat16*>(nullptr), static_cast<float*>(nullptr), H,
                             topk, S, num_rows, stride, scale_log2,
                             g_fault_block.load(std::memory_order_relaxed));
}

// How many clusters of S split CTAs the device holds at once (0: such a cluster does
// not fit, or S > 8): asked once per (device, S).
template <int NH, int MODE>
cudaError_t cluster_count(int dev, int S, int* clusters) {
  static int answer[kMaxDevices][kMaxCluster + 1] = {};   // 0 unknown, else count + 1
  if (S < 1 || S > kMaxCluster) {
    *clusters = 0;
    return cudaSuccess;
  }
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaError_t e = configure<NH, MODE>(dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_cfg_mu);
  if (answer[dev][S] == 0) {
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
    answer[dev][S] = (n > 0 ? n : 0) + 1;
  }
  *clusters = answer[dev][S] - 1;
  return cudaSuccess;
}

template <int NH, int MODE>
cudaError_t cluster_fits(int dev, int S, bool* fits) {
  int n = 0;
  const cudaError_t e = cluster_count<NH, MODE>(dev, S, &n);
  *fits = n > 0;
  return e;
}

template <int NH, int MODE>
cudaError_t launch_fused_t(const void* q, const void* kv, const int32_t* indices, float* o_part,
                           float* lse_part, void* out, float* lse, int B, int H, int topk, int S,
                           int64_t num_rows, int64_t stride, float softmax_scale,
                           cudaStream_t stream) {
  using C = Cfg<NH>;
  if (S < 1 || S > kMaxCluster) return cudaErrorNotSupported;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  bool fits = false;
  e = cluster_fits<NH, MODE>(dev, S, &fits);
  if (e != cudaSuccess) return e;
  if (!fits) return cudaErrorNotSupported;
  RowMaps maps;   // (read only by the kernels that gather by tensor copies)
  std::memset(static_cast<void*>(&maps), 0, sizeof(RowMaps));
  if (C::kTmaRows) {
    e = row_maps(kv, num_rows, stride, q, static_cast<int64_t>(B) * H, NH, &maps);
    if (e != cudaSuccess) return e;
  }
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
  const float scale_log2 = softmax_scale * 1.4426950408889634f;
  return cudaLaunchKernelEx(&cfg, split_kernel<NH, MODE>, static_cast<const uint16_t*>(q),
                            static_cast<const uint8_t*>(kv), maps, indices, o_part, lse_part,
                            static_cast<__nv_bfloat16*>(out), lse, H, topk, S, num_rows, stride,
                            scale_log2, g_fault_block.load(std::memory_order_relaxed));
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
      return launch_fused_t<16, kMergeCluster>(q, kv, indices, o_part, lse_part, out, lse, B, H, topk,
                                          S, num_rows, stride, softmax_scale, stream);
    case 32:
      return launch_fused_t<32, kMergeCluster>(q, kv, indices, o_part, lse_part, out, lse, B, H, topk,
                                          S, num_rows, stride, softmax_scale, stream);
    default:
      return launch_fused_t<64, kMergeCluster>(q, kv, indices, o_part, lse_part, out, lse, B, H, topk,
                                          S, num_rows, stride, softmax_scale, stream);
  }
}

cudaError_t fused_clusters(int H, int S, int* clusters) {
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  switch (H) {
    case 16: return cluster_count<16, kMergeCluster>(dev, S, clusters);
    case 32: return cluster_count<32, kMergeCluster>(dev, S, clusters);
    default: return cluster_count<64, kMergeCluster>(dev, S, clusters);
  }
}

void set_fault_block(int block) { g_fault_block.store(block, std::memory_order_relaxed); }

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
