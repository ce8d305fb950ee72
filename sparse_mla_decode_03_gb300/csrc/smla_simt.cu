// Per-head SIMT sparse MLA decode: the kind of kernel the tensor-core path replaces,
// kept as a same-device reference point.  "The Moment of Compilation: When a Triton
// Kernel Meets Its Constraints", sections "The Context: A Kernel Optimization
// Campaign" and "The Assumption That Broke", describe the production kernel before
// the MMA rewrite: one program per head, element-wise fp32 arithmetic, and every
// head re-reading the selected KV rows.
//
// One CTA per (query b, head h), 4 warps.  Warp w takes the index slots w, w+4, ...;
// for each valid row its 32 lanes dequantise their share of the 448 nope columns
// (4-byte words, scale byte per 64-column group) and of the 64 rope columns, the
// score is a warp sum, and the warp keeps its own online-softmax state (running max,
// sum, and 14 of the 448 output columns per lane).  The four warps merge at the end.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../include/smla.h"
#include "smla_internal.h"

namespace smla {
namespace {

constexpr int kSimtWarps = 4;
constexpr int kNopeWords = kNope / 4;                 // 112 words of 4 e4m3 bytes
constexpr int kWordsPerLane = (kNopeWords + 31) / 32;  // 4 (lanes 16..31 use 3)

__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
  uint32_t h2;
  const uint16_t in = static_cast<uint16_t>(byte);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xffffu)));
}
// UE8M0 byte -> 2^(e-127) (e = 0 is 2^-127, a subnormal fp32; 0xFF is NaN).
__device__ __forceinline__ float ue8m0(uint32_t e) {
  const uint32_t bits = e == 0u ? 0x00400000u : (e == 255u ? 0x7fffffffu : (e << 23));
  return __uint_as_float(bits);
}

__global__ void __launch_bounds__(kSimtWarps * 32)
    simt_kernel(const uint16_t* __restrict__ q, const uint8_t* __restrict__ kv,
                const int32_t* __restrict__ indices, __nv_bfloat16* __restrict__ out,
                float* __restrict__ lse, int* __restrict__ status, int H, int topk,
                int64_t num_rows, int64_t stride, float scale) {
  __shared__ float qs[kQkDim];
  __shared__ float wm[kSimtWarps], wl[kSimtWarps];
  __shared__ float wacc[kSimtWarps][kNope];
  const int h = blockIdx.x, b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint16_t* qrow = q + (static_cast<int64_t>(b) * H + h) * kQkDim;
  for (int c = threadIdx.x; c < kQkDim; c += blockDim.x)
    qs[c] = __uint_as_float(static_cast<uint32_t>(qrow[c]) << 16);
  __syncthreads();

  float m = -INFINITY, l = 0.f;
  float acc[kWordsPerLane * 4];
#pragma unroll
  for (int i = 0; i < kWordsPerLane * 4; ++i) acc[i] = 0.f;
  const int32_t* idx_row = indices + static_cast<int64_t>(b) * topk;
  for (int t = warp; t < topk; t += kSimtWarps) {
    const int idx = __ldg(idx_row + t);
    if (idx < 0) continue;
    if (static_cast<int64_t>(idx) >= num_rows) {
      if (lane == 0) atomicCAS(status, 0, SMLA_ERR_INDEX_RANGE);
      continue;
    }
    const uint8_t* row = kv + static_cast<int64_t>(idx) * stride;
    float v[kWordsPerLane * 4];
    float dot = 0.f;
#pragma unroll
    for (int j = 0; j < kWordsPerLane; ++j) {
      const int w = lane + 32 * j;
      if (w < kNopeWords) {
        const uint32_t word = __ldg(reinterpret_cast<const uint32_t*>(row) + w);
        const float sc = ue8m0(__ldg(row + kNope + (4 * w) / 64));
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v[4 * j + e] = e4m3_to_f32((word >> (8 * e)) & 0xffu) * sc;
          dot = fmaf(qs[4 * w + e], v[4 * j + e], dot);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) v[4 * j + e] = 0.f;
      }
    }
    // rope: 64 bf16 at byte 456, two per lane
    const uint32_t rw = __ldg(reinterpret_cast<const uint32_t*>(row + 456) + lane);
    dot = fmaf(qs[kNope + 2 * lane], __uint_as_float(rw << 16), dot);
    dot = fmaf(qs[kNope + 2 * lane + 1], __uint_as_float(rw & 0xffff0000u), dot);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    const float s = dot * scale;
    const float m_new = fmaxf(m, s);
    const float f = expf(m - m_new);   // 0 on the first valid row (m = -inf)
    const float p = expf(s - m_new);
    l = l * f + p;
#pragma unroll
    for (int i = 0; i < kWordsPerLane * 4; ++i) acc[i] = acc[i] * f + p * v[i];
    m = m_new;
  }
  // merge the four warps
  if (lane == 0) {
    wm[warp] = m;
    wl[warp] = l;
  }
#pragma unroll
  for (int j = 0; j < kWordsPerLane; ++j) {
    const int w = lane + 32 * j;
    if (w < kNopeWords) {
#pragma unroll
      for (int e = 0; e < 4; ++e) wacc[warp][4 * w + e] = acc[4 * j + e];
    }
  }
  __syncthreads();
  float M = -INFINITY;
#pragma unroll
  for (int i = 0; i < kSimtWarps; ++i) M = fmaxf(M, wm[i]);
  float L = 0.f, fw[kSimtWarps];
#pragma unroll
  for (int i = 0; i < kSimtWarps; ++i) {
    fw[i] = (wm[i] == -INFINITY) ? 0.f : expf(wm[i] - M);
    L += wl[i] * fw[i];
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  __nv_bfloat16* orow = out + (static_cast<int64_t>(b) * H + h) * kNope;
  for (int c = threadIdx.x; c < kNope; c += blockDim.x) {
    float o = 0.f;
#pragma unroll
    for (int i = 0; i < kSimtWarps; ++i) o += wacc[i][c] * fw[i];
    orow[c] = __float2bfloat16_rn(o * inv);
  }
  if (threadIdx.x == 0) lse[static_cast<int64_t>(b) * H + h] = L > 0.f ? M + logf(L) : -INFINITY;
}

}  // namespace

cudaError_t launch_simt(const void* q, const void* kv, const int32_t* indices, void* out,
                        float* lse, int B, int H, int topk, int64_t num_rows, int64_t stride,
                        float softmax_scale, cudaStream_t stream) {
  int* status = nullptr;
  const cudaError_t e = status_word_address(&status);
  if (e != cudaSuccess) return e;
  simt_kernel<<<dim3(H, B), kSimtWarps * 32, 0, stream>>>(
      static_cast<const uint16_t*>(q), static_cast<const uint8_t*>(kv), indices,
      static_cast<__nv_bfloat16*>(out), lse, status, H, topk, num_rows, stride, softmax_scale);
  return cudaGetLastError();
}

}  // namespace smla
