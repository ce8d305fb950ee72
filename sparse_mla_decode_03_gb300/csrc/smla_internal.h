// Host-side interface between the C ABI layer (smla_api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/smla.h"

namespace smla {

constexpr int kQkDim = 512;     // q / k width: 448 nope + 64 rope
constexpr int kNope = 448;      // value / output width
constexpr int kRowBytes = 584;  // packed KV row
constexpr int kMaxSplits = 256;
constexpr int kMaxCombineSplits = 1024;

// Launches `kernel` with programmatic stream serialization: the grid may be scheduled
// while the previous kernel in the stream finishes.  Every kernel launched this way
// calls grid_dep_wait before its first global-memory access.
template <typename... KArgs, typename... Args>
cudaError_t launch_programmatic(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Launches the split kernel: grid (S, H / heads_per_cta, B), 640 threads.
cudaError_t launch_split(const void* q, const void* kv, const int32_t* indices, float* o_part,
                         float* lse_part, int B, int H, int topk, int S, int64_t num_rows,
                         int64_t stride, float softmax_scale, cudaStream_t stream);

// Launches the split kernel as clusters of the S splits of each (query, head group):
// the splits write o_part / lse_part, then (after a cluster barrier) each CTA merges
// a slice of the heads from them and writes the final out / lse.  Returns
// cudaErrorNotSupported (nothing launched) when S > 8 or such a cluster does not fit
// on the device; the caller then uses split + combine.
cudaError_t launch_decode_fused(const void* q, const void* kv, const int32_t* indices,
                                float* o_part, float* lse_part, void* out, float* lse, int B,
                                int H, int topk, int S, int64_t num_rows, int64_t stride,
                                float softmax_scale, cudaStream_t stream);

// How many clusters of S splits of H heads the current device holds at once for
// launch_decode_fused (0: it cannot run them).
cudaError_t fused_clusters(int H, int S, int* clusters);

// Launches the combine kernel over B * H (batch, head) pairs.
cudaError_t launch_combine(const float* o_part, const float* lse_part, int B, int H, int S,
                           void* out, float* lse, cudaStream_t stream);

// Launches the per-head SIMT decode (one CTA per (query, head), fp32 arithmetic).
cudaError_t launch_simt(const void* q, const void* kv, const int32_t* indices, void* out,
                        float* lse, int B, int H, int topk, int64_t num_rows, int64_t stride,
                        float softmax_scale, cudaStream_t stream);

// Translates logical positions of a paged cache into pool rows (-1 = masked).
cudaError_t launch_paged_rows(const int32_t* indices, const int32_t* block_table, int B, int topk,
                              int max_pages, int page_size, int64_t num_rows, int32_t* rows,
                              cudaStream_t stream);

// SMLA_OK if the current device is a compute capability 10.3 GPU, else an
// smla_status (SMLA_ERR_UNSUPPORTED_DEVICE or SMLA_ERR_CUDA).
int check_device();

// The launch form of a decode step with S splits on the current device: *fused is
// true when the clustered launch (splits merged on chip) is modelled faster than
// split + combine and fits.  Returns an smla_status.
int plan_mode(const smla_params* p, int S, bool* fused);

// One whole decode step (sparse_mla_decode after argument checks): S splits, the
// split partials in `workspace` (laid out as smla_workspace_size describes), in the
// form plan_mode chooses.  Returns an smla_status.
int launch_step(const void* q, const void* kv_cache, const int32_t* indices, void* out,
                float* lse, const smla_params* p, int S, void* workspace, cudaStream_t stream);

// Test hook of smla_test_inject_fault: block index at which one converter warp of
// every CTA of later decode launches withholds its "block filled" arrival (-1: off).
void set_fault_block(int block);

// Device address of the status word (kernels in other translation units record
// their errors through it; device variables are not shared across them).
cudaError_t status_word_address(int** ptr);

// Device status word (first error wins).
cudaError_t read_device_status(int32_t* status, bool clear);

}  // namespace smla
