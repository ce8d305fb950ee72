// Combine kernel: merges the split-K partials of sparse MLA decode ("The 80KB
// Mystery: Resolving Contradictory Evidence in Triton Kernel Optimization", section
// "The Context: Optimizing Attention on Blackwell": the top-k is split across CTAs,
// so each (query, head) ends with one partial per split).
//
//   lse = ln sum_s exp(lse_s)          out = sum_s exp(lse_s - lse) * o_s   -> bf16
//
// One warp per (query, head): the split LSEs are reduced with warp shuffles, then
// each lane accumulates 14 of the 448 output columns (7 float2) over the splits.
#include <cuda_bf16.h>

#include "smla_internal.h"

namespace smla {
namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32)
    combine_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part, int BH,
                   int S, __nv_bfloat162* __restrict__ out, float* __restrict__ lse) {
  const int pair = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (pair >= BH) return;
  const float* lp = lse_part + static_cast<int64_t>(pair) * S;

  float m = -INFINITY;
  for (int s = lane; s < S; s += 32) m = fmaxf(m, lp[s]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));

  float sum = 0.f;
  if (m != -INFINITY) {
    for (int s = lane; s < S; s += 32) {
      const float x = lp[s];
      sum += (x == -INFINITY) ? 0.f : expf(x - m);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);

  float2 acc[7];
#pragma unroll
  for (int i = 0; i < 7; ++i) acc[i] = make_float2(0.f, 0.f);
  if (sum > 0.f) {
    const float inv = 1.f / sum;
    const float2* op = reinterpret_cast<const float2*>(o_part + static_cast<int64_t>(pair) * S * 448);
    for (int s = 0; s < S; ++s) {
      const float x = lp[s];
      if (x == -INFINITY) continue;  // same decision in every lane
      const float w = expf(x - m) * inv;
#pragma unroll
      for (int i = 0; i < 7; ++i) {
        const float2 v = __ldg(op + s * 224 + lane + 32 * i);
        acc[i].x = fmaf(w, v.x, acc[i].x);
        acc[i].y = fmaf(w, v.y, acc[i].y);
      }
    }
  }
  __nv_bfloat162* orow = out + static_cast<int64_t>(pair) * 224;
#pragma unroll
  for (int i = 0; i < 7; ++i) orow[lane + 32 * i] = __floats2bfloat162_rn(acc[i].x, acc[i].y);
  if (lane == 0) lse[pair] = (sum > 0.f) ? m + logf(sum) : -INFINITY;
}

}  // namespace

cudaError_t launch_combine(const float* o_part, const float* lse_part, int B, int H, int S,
                           void* out, float* lse, cudaStream_t stream) {
  const int BH = B * H;
  const int blocks = (BH + kWarps - 1) / kWarps;
  combine_kernel<<<blocks, kWarps * 32, 0, stream>>>(
      o_part, lse_part, BH, S, static_cast<__nv_bfloat162*>(out), lse);
  return cudaGetLastError();
}

}  // namespace smla
