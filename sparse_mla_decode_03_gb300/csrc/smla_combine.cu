// Combine kernel: merges the split-K partials of sparse MLA decode ("The 80KB
// Mystery: Resolving Contradictory Evidence in Triton Kernel Optimization", section
// "The Context: Optimizing Attention on Blackwell": the top-k is split across CTAs,
// so each (query, head) ends with one partial per split).
//
//   lse = ln sum_s exp(lse_s)          out = sum_s exp(lse_s - lse) * o_s   -> bf16
//
// Blocks of 224 threads, one output column pair per thread.  With up to 8 splits a
// block combines several (query, head) pairs and every thread loads all their split
// LSEs and column pairs in one round, so the whole combine is one wave of loads;
// with more splits one block per pair computes the split weights exp(lse_s - lse)
// once into shared memory and reads the column pairs four splits at a time.
#include <cuda_bf16.h>

#include "smla_internal.h"
#include "smla_ptx.cuh"

namespace smla {
namespace {

constexpr int kThreads = 224;                 // 448 columns as float2
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int i = 1; i < kWarps; ++i) r = fmaxf(r, red[i]);
  __syncthreads();
  return r;
}
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int i = 1; i < kWarps; ++i) r += red[i];
  __syncthreads();
  return r;
}

// Up to SMAX splits: each block combines P (query, head) pairs, every thread one
// column pair of each, with all split LSEs and column pairs loaded in one round.
template <int SMAX, int P>
__global__ void __launch_bounds__(kThreads)
    combine_few_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                       int BH, int S, __nv_bfloat162* __restrict__ out, float* __restrict__ lse) {
  const int t = threadIdx.x;
  grid_dep_wait();   // the partials come from the previous kernel in the stream
  grid_dep_launch();
  float l[P][SMAX];
  float2 v[P][SMAX];
#pragma unroll
  for (int p = 0; p < P; ++p) {
    const int64_t pair = static_cast<int64_t>(blockIdx.x) * P + p;
    const float2* op = reinterpret_cast<const float2*>(o_part) + pair * S * 224 + t;
#pragma unroll
    for (int k = 0; k < SMAX; ++k) {
      if (pair < BH && k < S) {
        l[p][k] = __ldg(lse_part + pair * S + k);
        v[p][k] = __ldg(op + k * 224);
      }
    }
  }
#pragma unroll
  for (int p = 0; p < P; ++p) {
    const int64_t pair = static_cast<int64_t>(blockIdx.x) * P + p;
    if (pair >= BH) break;
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < SMAX; ++k)
      if (k < S) m = fmaxf(m, l[p][k]);
    float sum = 0.f;
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < SMAX; ++k) {
      if (k < S) {
        const float e = (m == -INFINITY || l[p][k] == -INFINITY) ? 0.f : expf(l[p][k] - m);
        sum += e;
        acc.x = fmaf(e, v[p][k].x, acc.x);
        acc.y = fmaf(e, v[p][k].y, acc.y);
      }
    }
    const float inv = sum > 0.f ? 1.f / sum : 0.f;
    out[pair * 224 + t] = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    if (t == 0) lse[pair] = (sum > 0.f) ? m + logf(sum) : -INFINITY;
  }
}

// Any number of splits: one block per (query, head); the split weights go to shared
// memory first.
__global__ void __launch_bounds__(kThreads)
    combine_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part, int S,
                   __nv_bfloat162* __restrict__ out, float* __restrict__ lse) {
  __shared__ float w[kMaxCombineSplits];
  __shared__ float red[kWarps];
  const int pair = blockIdx.x;
  const int t = threadIdx.x;
  const float* lp = lse_part + static_cast<int64_t>(pair) * S;
  const float2* op = reinterpret_cast<const float2*>(o_part) + static_cast<int64_t>(pair) * S * 224 + t;
  grid_dep_wait();   // the partials come from the previous kernel in the stream
  grid_dep_launch();

  float m = -INFINITY;
  for (int s = t; s < S; s += kThreads) m = fmaxf(m, lp[s]);
  m = block_max(m, red);
  float part = 0.f;
  for (int s = t; s < S; s += kThreads) {
    const float x = lp[s];
    const float e = (m == -INFINITY || x == -INFINITY) ? 0.f : expf(x - m);
    w[s] = e;
    part += e;
  }
  const float sum = block_sum(part, red);   // also orders the w[] writes before the reads
  const float inv = sum > 0.f ? 1.f / sum : 0.f;

  float2 acc = make_float2(0.f, 0.f);
  int s = 0;
  for (; s + 4 <= S; s += 4) {
    float2 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = __ldg(op + (s + k) * 224);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float ws = w[s + k] * inv;
      acc.x = fmaf(ws, v[k].x, acc.x);
      acc.y = fmaf(ws, v[k].y, acc.y);
    }
  }
  for (; s < S; ++s) {
    const float2 v = __ldg(op + s * 224);
    const float ws = w[s] * inv;
    acc.x = fmaf(ws, v.x, acc.x);
    acc.y = fmaf(ws, v.y, acc.y);
  }
  out[static_cast<int64_t>(pair) * 224 + t] = __floats2bfloat162_rn(acc.x, acc.y);
  if (t == 0) lse[pair] = (sum > 0.f) ? m + logf(sum) : -INFINITY;
}

}  // namespace

cudaError_t launch_combine(const float* o_part, const float* lse_part, int B, int H, int S,
                           void* out, float* lse, cudaStream_t stream) {
  const int BH = B * H;
  if (BH == 0) return cudaSuccess;
  auto* o = static_cast<__nv_bfloat162*>(out);
  const dim3 blk(kThreads);
  if (S <= 2)
    return launch_programmatic(combine_few_kernel<2, 16>, dim3((BH + 15) / 16), blk, 0, stream,
                               o_part, lse_part, BH, S, o, lse);
  if (S <= 4)
    return launch_programmatic(combine_few_kernel<4, 8>, dim3((BH + 7) / 8), blk, 0, stream,
                               o_part, lse_part, BH, S, o, lse);
  if (S <= 8)
    return launch_programmatic(combine_few_kernel<8, 4>, dim3((BH + 3) / 4), blk, 0, stream,
                               o_part, lse_part, BH, S, o, lse);
  return launch_programmatic(combine_kernel, dim3(BH), blk, 0, stream, o_part, lse_part, S, o, lse);
}

}  // namespace smla
