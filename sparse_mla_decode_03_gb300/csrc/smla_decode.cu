// Split kernel of sparse MLA decode for sm_103a.
//
// One CTA handles one (query b, group of NH heads, split s of the top-k list).  For
// each tile of 128 index slots it
//   1. gathers the selected 584-byte rows once for all NH heads ("The Moment of
//      Compilation: When a Triton Kernel Meets Its Constraints", section "The
//      Context: A Kernel Optimization Campaign": one KV read shared by all heads),
//   2. dequantises the FP8 e4m3 nope part with its per-64-column UE8M0 scales into a
//      bf16 tile ("The Power-of-Two Trap: Debugging a Triton MMA Kernel on Blackwell
//      GPUs", section "3. The Scale Indexing Complication"), next to the bf16 rope,
//   3. computes S^T = K_tile . Q^T on the tensor cores (tcgen05.mma, M = 128 tokens,
//      N = NH heads, K = 512) into tensor memory,
//   4. runs the online softmax over the tile (running max / sum per head),
//   5. accumulates O^T += V_tile^T . P^T on the tensor cores (M = 128 value columns per
//      block, 4 blocks, N = NH, K = 128 tokens) in tensor memory,
// and finally writes the normalised partial O and its log-sum-exp for the split
// (the split-K scheme of "The 80KB Mystery: Resolving Contradictory Evidence in
// Triton Kernel Optimization", section "The Context: Optimizing Attention on
// Blackwell").
//
// Tokens are the MMA's M dimension so that every MMA is a full 128-row tcgen05
// instruction even with 16 heads.  The same bf16 tile serves as K (K-major view) for
// the scores and as V^T (MN-major view) for the output; its 4th 128-column block
// holds dims 384..511 whose last 64 (the rope) produce output rows that are never
// stored, so the 448-wide value product needs no separate padding.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../include/smla.h"
#include "smla_internal.h"
#include "smla_ptx.cuh"

namespace smla {

__device__ int g_smla_status = 0;

namespace {

constexpr int kTile = 128;                    // tokens per tile (MMA M)
constexpr int kChunkBytes = kTile * 128;      // one 64-column bf16 slab of the tile
constexpr int kThreads = 128;
constexpr long long kWaitLimit = 2000000000LL;  // ~1 s of SM clocks
constexpr float kLn2 = 0.69314718055994530942f;

template <int NH>
struct Cfg {
  static constexpr int kQOff = 8 * kChunkBytes;
  static constexpr int kQChunk = NH * 128;
  static constexpr int kPOff = kQOff + 8 * kQChunk;
  static constexpr int kPRow = 2 * NH;
  static constexpr int kPBytes = kTile * kPRow;
  static constexpr int kMiscOff = kPOff + ((kPBytes + 1023) / 1024) * 1024;
  static constexpr int kRedOff = kMiscOff;                 // float [4][NH]
  static constexpr int kMOff = kRedOff + 4 * NH * 4;       // float [2][NH] running max
  static constexpr int kValidOff = kMOff + 2 * NH * 4;     // uint8 [128]
  static constexpr int kBarOff = kValidOff + 128;          // uint64
  static constexpr int kTaddrOff = kBarOff + 8;            // uint32
  static constexpr int kFlagOff = kTaddrOff + 4;           // int
  static constexpr int kSmemBytes = kFlagOff + 4 + 1024;   // + alignment slack
  static constexpr uint32_t kTmemCols =
      5 * NH <= 32 ? 32 : 5 * NH <= 64 ? 64 : 5 * NH <= 128 ? 128 : 5 * NH <= 256 ? 256 : 512;
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

__device__ __forceinline__ uint2 ldg_nc_u2(const uint2* p) {
  uint2 v;
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// UE8M0 byte -> fp32 2^(e-127) (e = 0 is the fp32 subnormal 2^-127, 0xFF is NaN).
__device__ __forceinline__ float ue8m0_to_f32(uint32_t e) {
  const uint32_t bits = e == 0u ? 0x00400000u : (e == 255u ? 0x7fffffffu : (e << 23));
  return __uint_as_float(bits);
}

// Two e4m3 bytes (low byte = first element) -> bf16x2 of value * scale.
__device__ __forceinline__ uint32_t dequant_pair(uint32_t two, float scale) {
  uint32_t h2;
  const uint16_t in = static_cast<uint16_t>(two);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  const __half2 hh = *reinterpret_cast<const __half2*>(&h2);
  const float2 f = __half22float2(hh);
  const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale, f.y * scale);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// 8 e4m3 bytes -> 8 bf16 (16 bytes).
__device__ __forceinline__ uint4 dequant8(uint2 w, float scale) {
  uint4 r;
  r.x = dequant_pair(w.x & 0xffffu, scale);
  r.y = dequant_pair(w.x >> 16, scale);
  r.z = dequant_pair(w.y & 0xffffu, scale);
  r.w = dequant_pair(w.y >> 16, scale);
  return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// Gathers and dequantises the 32 tile rows owned by this warp.  A row is 73 8-byte
// words: words 0..55 nope, word 56 the 7 scales + pad, words 57..72 rope.  Lane l
// loads words l, 32 + l and (l < 9) 64 + l, so each row is read with coalesced
// 8-byte loads.  Rows that are masked, beyond the split or out of range are written
// as zeros.
template <int NH>
__device__ __forceinline__ void gather_rows(uint32_t sbase, uint8_t* vflag, const uint8_t* kv,
                                            const int32_t* idx_row, int tile0, int t_end,
                                            int64_t num_rows, int64_t stride, int warp,
                                            int lane) {
  constexpr int kBatch = 4;
  const uint2 zero = make_uint2(0u, 0u);
#pragma unroll 1
  for (int i0 = 0; i0 < 32; i0 += kBatch) {
    uint2 wa[kBatch], wb[kBatch], wc[kBatch];
    bool val[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int r = warp * 32 + i0 + j;
      const int pos = tile0 + r;
      int idx = -1;
      if (pos < t_end) idx = __ldg(idx_row + pos);
      bool v = idx >= 0;
      if (v && static_cast<int64_t>(idx) >= num_rows) {
        v = false;
        if (lane == 0) record_status(SMLA_ERR_INDEX_RANGE);
      }
      val[j] = v;
      const uint2* row =
          reinterpret_cast<const uint2*>(kv + (v ? static_cast<int64_t>(idx) * stride : 0));
      wa[j] = v ? ldg_nc_u2(row + lane) : zero;
      wb[j] = v ? ldg_nc_u2(row + 32 + lane) : zero;
      wc[j] = (v && lane < 9) ? ldg_nc_u2(row + 64 + lane) : zero;
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const uint32_t r = static_cast<uint32_t>(warp * 32 + i0 + j);
      const uint32_t sc_lo = __shfl_sync(0xffffffffu, wb[j].x, 24);
      const uint32_t sc_hi = __shfl_sync(0xffffffffu, wb[j].y, 24);
      // word `lane`: columns 8*lane.., group lane/8 (0..3)
      const float fa = ue8m0_to_f32((sc_lo >> (8 * (lane >> 3))) & 0xffu);
      st_shared_v4(sbase + (lane >> 3) * kChunkBytes + swz_offset(r, lane & 7, 128),
                   dequant8(wa[j], fa));
      if (lane < 24) {
        // word 32 + lane: group 4 + lane/8 (4..6) = byte lane/8 of the high scale word
        const float fb = ue8m0_to_f32((sc_hi >> (8 * (lane >> 3))) & 0xffu);
        st_shared_v4(sbase + (4 + (lane >> 3)) * kChunkBytes + swz_offset(r, lane & 7, 128),
                     dequant8(wb[j], fb));
      } else if (lane >= 25) {
        const uint32_t rr = lane - 25;  // rope word 0..6: rope columns 4rr..4rr+3
        st_shared_v2(sbase + 7 * kChunkBytes + swz_offset(r, rr >> 1, 128) + (rr & 1) * 8, wb[j]);
      }
      if (lane < 9) {
        const uint32_t rr = 7 + lane;  // rope word 7..15
        st_shared_v2(sbase + 7 * kChunkBytes + swz_offset(r, rr >> 1, 128) + (rr & 1) * 8, wc[j]);
      }
      if (lane == 0) vflag[r] = val[j] ? 1 : 0;
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

  const int G = (topk + 15) >> 4;
  const int g0 = static_cast<int>((static_cast<int64_t>(s) * G) / S);
  const int g1 = static_cast<int>((static_cast<int64_t>(s + 1) * G) / S);
  const int t_begin = min(16 * g0, topk), t_end = min(16 * g1, topk);
  const int ntiles = (t_end - t_begin + kTile - 1) / kTile;

  float* red = reinterpret_cast<float*>(smem + C::kRedOff);
  float* mbuf = reinterpret_cast<float*>(smem + C::kMOff);
  uint8_t* vflag = smem + C::kValidOff;
  const uint32_t bar = sbase + C::kBarOff;
  volatile uint32_t* taddr_s = reinterpret_cast<volatile uint32_t*>(smem + C::kTaddrOff);

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (tid < NH) mbuf[tid] = -INFINITY;
  if (warp == 0) {
    tmem_alloc(sbase + C::kTaddrOff, C::kTmemCols);
    tmem_relinquish();
  }
  // Q rows h0..h0+NH-1 of query b -> 8 K-major SW128 slabs of 64 columns.
  for (int u = tid; u < NH * 64; u += kThreads) {
    const int r = u >> 6, cu = u & 63;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(
        q + (static_cast<int64_t>(b) * H + h0 + r) * kQkDim + cu * 8));
    st_shared_v4(sbase + C::kQOff + (cu >> 3) * C::kQChunk + swz_offset(r, cu & 7, 128), v);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *taddr_s;
  const uint32_t tS = tmem;        // S^T: columns [0, NH)
  const uint32_t tO = tmem + NH;   // O^T block mb: columns [NH + mb*NH, NH + (mb+1)*NH)
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;

  constexpr uint32_t kIdescQK = idesc_bf16(128, NH, false, false);
  constexpr uint32_t kIdescPV = idesc_bf16(128, NH, true, true);

  float l[NH];
#pragma unroll
  for (int h = 0; h < NH; ++h) l[h] = 0.f;

  uint32_t phase = 0;
  bool failed = false;
  const int32_t* idx_row = indices + static_cast<int64_t>(b) * topk;

  for (int it = 0; it < ntiles; ++it) {
    const int tile0 = t_begin + it * kTile;
    gather_rows<NH>(sbase, vflag, kv, idx_row, tile0, t_end, num_rows, stride, warp, lane);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- S^T = K . Q^T  (M = 128 tokens, N = NH, K = 512 in 32 steps) ----
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t a = smem_desc(sbase + j * kChunkBytes + k * 32, 16, 1024, SWZ_128B);
          const uint64_t bq =
              smem_desc(sbase + C::kQOff + j * C::kQChunk + k * 32, 16, 1024, SWZ_128B);
          mma_bf16_ss(tS, a, bq, kIdescQK, (j | k) != 0);
        }
      }
      mma_commit(bar);
    }
    bool ok = mbar_wait(bar, phase, kWaitLimit);
    phase ^= 1u;
    tc_fence_after();

    float sv[NH];
#pragma unroll
    for (int c = 0; c < NH / 16; ++c) tmem_ld16(tS + lane_base + 16 * c, sv + 16 * c);
    tmem_wait_ld();

    // ---- online softmax (log2 domain) ----
    const bool valid = vflag[tid] != 0;
#pragma unroll
    for (int h = 0; h < NH; ++h) sv[h] = valid ? sv[h] * scale_log2 : -INFINITY;
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      const float m = warp_max(sv[h]);
      if (lane == (h & 31)) red[warp * NH + h] = m;
    }
    __syncthreads();
    const float* m_old = mbuf + (it & 1) * NH;
    float* m_new_s = mbuf + ((it + 1) & 1) * NH;
    bool rescale = false;
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      const float mt = fmaxf(fmaxf(red[h], red[NH + h]), fmaxf(red[2 * NH + h], red[3 * NH + h]));
      const float mo = m_old[h];
      const float mn = fmaxf(mo, mt);
      const float alpha = (mn == -INFINITY) ? 1.f : exp2f(mo - mn);
      rescale |= alpha != 1.f;
      const float p = (sv[h] == -INFINITY) ? 0.f : exp2f(sv[h] - mn);
      l[h] = l[h] * alpha + p;
      sv[h] = p;
      if (tid == h) m_new_s[h] = mn;
    }
    // P^T row `tid` (NH bf16), MN-major with rows of 2*NH bytes
#pragma unroll
    for (int u = 0; u < NH / 8; ++u) {
      uint4 v;
      v.x = pack_bf16x2(sv[8 * u + 0], sv[8 * u + 1]);
      v.y = pack_bf16x2(sv[8 * u + 2], sv[8 * u + 3]);
      v.z = pack_bf16x2(sv[8 * u + 4], sv[8 * u + 5]);
      v.w = pack_bf16x2(sv[8 * u + 6], sv[8 * u + 7]);
      st_shared_v4(sbase + C::kPOff + swz_offset(tid, u, C::kPRow), v);
    }
    __syncthreads();  // m_new_s complete
    if (rescale && it > 0) {
#pragma unroll 1
      for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
        for (int c = 0; c < NH / 16; ++c) {
          float o[16];
          tmem_ld16(tO + lane_base + mb * NH + 16 * c, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int h = 16 * c + i;
            const float mn = m_new_s[h];
            o[i] *= (mn == -INFINITY) ? 1.f : exp2f(m_old[h] - mn);
          }
          tmem_st16(tO + lane_base + mb * NH + 16 * c, o);
        }
      }
      tmem_wait_st();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- O^T += V^T . P^T  (4 blocks of M = 128 columns, N = NH, K = 128 tokens) ----
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t a =
              smem_desc(sbase + (2 * mb) * kChunkBytes + ks * 2048, kChunkBytes, 1024, SWZ_128B);
          // N = NH is a single swizzle atom wide, so the leading offset is unused;
          // it is set equal to the stride offset to keep every address in bounds.
          const uint64_t bp = smem_desc(sbase + C::kPOff + ks * 16 * C::kPRow, 8 * C::kPRow,
                                        8 * C::kPRow, C::kPSwz);
          mma_bf16_ss(tO + mb * NH, a, bp, kIdescPV, (it > 0 || ks > 0) ? 1u : 0u);
        }
      }
      mma_commit(bar);
    }
    ok = mbar_wait(bar, phase, kWaitLimit) && ok;
    phase ^= 1u;
    tc_fence_after();
    if (__syncthreads_or(!ok)) {
      failed = true;
      if (tid == 0) record_status(SMLA_ERR_TIMEOUT);
      break;
    }
  }

  // ---- epilogue: l over the 128 threads, lse, normalised O ----
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    float v = l[h];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == (h & 31)) red[warp * NH + h] = v;
  }
  __syncthreads();
  const float* m_fin = mbuf + (ntiles & 1) * NH;
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    const float lt = red[h] + red[NH + h] + red[2 * NH + h] + red[3 * NH + h];
    l[h] = (lt > 0.f && !failed) ? 1.f / lt : 0.f;
    if (tid == h) {
      const float lse = (lt > 0.f && !failed) ? (m_fin[h] + log2f(lt)) * kLn2 : -INFINITY;
      lse_part[(static_cast<int64_t>(b) * H + h0 + h) * S + s] = lse;
    }
  }
  const bool have_o = ntiles > 0 && !failed;
#pragma unroll 1
  for (int mb = 0; mb < 4; ++mb) {
    const int d = mb * 128 + tid;
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
          const float val = (have_o && l[h] > 0.f) ? o[i] * l[h] : 0.f;
          o_part[((static_cast<int64_t>(b) * H + h0 + h) * S + s) * kNope + d] = val;
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
