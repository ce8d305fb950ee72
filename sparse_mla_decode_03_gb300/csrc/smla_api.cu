// C ABI of libsmla.so: argument validation, split planning and kernel launches.
// Declarations and their documentation are in include/smla.h.
#include <cmath>
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>

#include "../../include/smla.h"
#include "smla_internal.h"

namespace {

using smla::kMaxCombineSplits;
using smla::kMaxSplits;

constexpr int kMaxDevices = 64;
// 0 = not queried yet, -1 = unsupported device, else the SM count.  Written at most
// once per device with the same value by whichever host thread gets there first.
std::atomic<int> g_sm_count[kMaxDevices];

// SM count of the current device, or an error status if it is not sm_103.
int current_device_sms(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SMLA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SMLA_ERR_UNSUPPORTED_DEVICE;
  int v = g_sm_count[dev].load(std::memory_order_acquire);
  if (v == 0) {
    int major = 0, minor = 0, n = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return SMLA_ERR_CUDA;
    v = (major == 10 && minor == 3) ? n : -1;
    g_sm_count[dev].store(v, std::memory_order_release);
  }
  if (v < 0) return SMLA_ERR_UNSUPPORTED_DEVICE;
  *sms = v;
  return SMLA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_params(const smla_params* p) {
  if (p == nullptr) return SMLA_ERR_INVALID_ARG;
  if (p->batch < 1 || p->topk < 1 || p->topk > 65536 || p->num_rows < 1 || p->reserved != 0)
    return SMLA_ERR_INVALID_ARG;
  if (p->kv_row_stride < smla::kRowBytes || (p->kv_row_stride % 8) != 0)
    return SMLA_ERR_INVALID_ARG;
  if (!(std::isfinite(p->softmax_scale) && p->softmax_scale > 0.f)) return SMLA_ERR_INVALID_ARG;
  if (p->num_heads != 16 && p->num_heads != 32 && p->num_heads != 64 && p->num_heads != 128)
    return SMLA_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<int64_t>(p->batch) * p->num_heads > (int64_t(1) << 30))
    return SMLA_ERR_UNSUPPORTED_SHAPE;
  if (p->batch > 65535) return SMLA_ERR_UNSUPPORTED_SHAPE;   // grid z of the decode kernels
  return SMLA_OK;
}

int max_splits(const smla_params* p) {
  const int granules = (p->topk + 15) / 16;
  return granules < kMaxSplits ? granules : kMaxSplits;
}

// Step time model, in units of one 64-slot block of a CTA (one CTA per SM is
// resident): waves * (slots of the largest split / 64 + kFixedBlocks) plus the
// merge: kCombineBlocks for a second kernel, kClusterMergeBlocks per split for the
// on-chip merge.  A split's slots count fractionally (a latency-bound split of few
// slots gathers few rows) but at least kMinBlocks.  A wave holds `per_wave` CTAs:
// the SM count for plain launches, (clusters the device holds at once) * S for
// clustered ones, which can be fewer since a cluster's CTAs share one GPC.  The
// constants are GB300 measurements: the prologue (first gathers, q) and epilogue
// of a CTA cost ~2.6 blocks, the combine launch ~0.5 block, the on-chip merge
// ~0.05 block per split of the cluster.
constexpr double kFixedBlocks = 2.6;
constexpr double kCombineBlocks = 0.5;
constexpr double kClusterMergeBlocks = 0.05;
constexpr double kMinBlocks = 0.5;

double step_cost(const smla_params* p, int s, int64_t per_wave, bool fused) {
  const int groups = p->num_heads > 64 ? p->num_heads / 64 : 1;
  const int64_t ctas = static_cast<int64_t>(p->batch) * groups * s;
  const int granules = (p->topk + 15) / 16;
  const int gmax = (granules + s - 1) / s;                // granules of the largest split
  const double blocks = std::max(gmax * 16 / 64.0, kMinBlocks);
  const int64_t waves = (ctas + per_wave - 1) / std::max<int64_t>(per_wave, 1);
  return static_cast<double>(waves) * (blocks + kFixedBlocks) +
         (fused ? kClusterMergeBlocks * s : kCombineBlocks);
}

// Cost of S splits in the cheaper of the two launch forms; *fused tells which.
int mode_cost(const smla_params* p, int s, int sms, double* cost, bool* fused) {
  int clusters = 0;
  if (smla::fused_clusters(p->num_heads, s, &clusters) != cudaSuccess) return SMLA_ERR_CUDA;
  const double plain = step_cost(p, s, sms, false);
  const double clustered = clusters > 0 ? step_cost(p, s, static_cast<int64_t>(clusters) * s, true)
                                        : 1e300;
  *fused = clustered <= plain;
  *cost = std::min(plain, clustered);
  return SMLA_OK;
}

// Plan: the split count of least modelled time, preferring fewer splits on ties.
int plan_splits(const smla_params* p, int sms, int* S) {
  int best = 1;
  double best_cost = 1e300;
  for (int s = 1; s <= max_splits(p); ++s) {
    double c = 0;
    bool f = false;
    const int st = mode_cost(p, s, sms, &c, &f);
    if (st != SMLA_OK) return st;
    if (c < best_cost - 1e-9) {
      best_cost = c;
      best = s;
    }
  }
  *S = best;
  return SMLA_OK;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

namespace smla {

int check_device() {
  int sms = 0;
  return current_device_sms(&sms);
}

// One whole decode step on validated arguments: one launch when the splits of a
// query fit in a thread-block cluster (they merge their partials in the workspace
// inside that launch), split + combine kernels otherwise.
int plan_mode(const smla_params* p, int S, bool* fused) {
  int sms = 0;
  int st = current_device_sms(&sms);
  if (st != SMLA_OK) return st;
  double c = 0;
  return mode_cost(p, S, sms, &c, fused);
}

int launch_step(const void* q, const void* kv_cache, const int32_t* indices, void* out,
                float* lse, const smla_params* p, int S, void* workspace, cudaStream_t s) {
  const size_t bhs = static_cast<size_t>(p->batch) * p->num_heads * S;
  float* o_part = static_cast<float*>(workspace);
  float* lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                             round256(bhs * kNope * sizeof(float)));
  bool fused = false;
  const int st = plan_mode(p, S, &fused);
  if (st != SMLA_OK) return st;
  cudaError_t e = cudaErrorNotSupported;
  if (fused)
    e = launch_decode_fused(q, kv_cache, indices, o_part, lse_part, out, lse, p->batch,
                            p->num_heads, p->topk, S, p->num_rows, p->kv_row_stride,
                            p->softmax_scale, s);
  if (e == cudaSuccess) return SMLA_OK;
  if (e != cudaErrorNotSupported) return SMLA_ERR_CUDA;
  e = launch_split(q, kv_cache, indices, o_part, lse_part, p->batch, p->num_heads, p->topk, S,
                   p->num_rows, p->kv_row_stride, p->softmax_scale, s);
  if (e != cudaSuccess) return SMLA_ERR_CUDA;
  e = launch_combine(o_part, lse_part, p->batch, p->num_heads, S, out, lse, s);
  return e == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

}  // namespace smla

namespace {

void workspace_layout(const smla_params* p, int S, size_t* o_bytes, size_t* total) {
  const size_t bhs = static_cast<size_t>(p->batch) * p->num_heads * S;
  *o_bytes = round256(bhs * smla::kNope * sizeof(float));
  *total = *o_bytes + round256(bhs * sizeof(float));
}

// The split count of a call: the plan for the current device (requested = 0, which
// needs an sm_103 GPU to be current) or the caller's count (pure arithmetic).
int resolve_splits(const smla_params* p, int32_t requested, int* S) {
  if (requested < 0) return SMLA_ERR_INVALID_ARG;
  if (requested > max_splits(p)) return SMLA_ERR_INVALID_ARG;
  if (requested > 0) {
    *S = requested;
    return SMLA_OK;
  }
  int sms = 0;
  const int st = current_device_sms(&sms);
  if (st != SMLA_OK) return st;
  return plan_splits(p, sms, S);
}

int check_tensors(const void* q, const void* kv, const int32_t* idx) {
  if (q == nullptr || kv == nullptr || idx == nullptr) return SMLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(idx, 4)) return SMLA_ERR_INVALID_ARG;
  return SMLA_OK;
}

}  // namespace

extern "C" {

int smla_default_num_splits(const smla_params* p, int32_t* num_splits) {
  int st = check_params(p);
  if (st != SMLA_OK) return st;
  if (num_splits == nullptr) return SMLA_ERR_INVALID_ARG;
  int S = 0;
  st = resolve_splits(p, 0, &S);
  if (st != SMLA_OK) return st;
  *num_splits = S;
  return SMLA_OK;
}

int smla_decode_plan(const smla_params* p, int32_t num_splits, int32_t* splits, int32_t* fused) {
  int st = check_params(p);
  if (st != SMLA_OK) return st;
  if (splits == nullptr || fused == nullptr) return SMLA_ERR_INVALID_ARG;
  int S = 0;
  st = resolve_splits(p, num_splits, &S);
  if (st != SMLA_OK) return st;
  bool f = false;
  st = smla::plan_mode(p, S, &f);
  if (st != SMLA_OK) return st;
  *splits = S;
  *fused = f ? 1 : 0;
  return SMLA_OK;
}

int smla_workspace_size(const smla_params* p, int32_t num_splits, size_t* bytes) {
  int st = check_params(p);
  if (st != SMLA_OK) return st;
  if (bytes == nullptr) return SMLA_ERR_INVALID_ARG;
  int S = 0;
  st = resolve_splits(p, num_splits, &S);
  if (st != SMLA_OK) return st;
  size_t o_bytes = 0, total = 0;
  workspace_layout(p, S, &o_bytes, &total);
  *bytes = total;
  return SMLA_OK;
}

int sparse_mla_decode_split(const void* q, const void* kv_cache, const int32_t* indices,
                            const smla_params* p, int32_t num_splits, float* o_part,
                            float* lse_part, smla_stream_t stream) {
  int st = check_params(p);
  if (st != SMLA_OK) return st;
  st = check_tensors(q, kv_cache, indices);
  if (st != SMLA_OK) return st;
  if (o_part == nullptr || lse_part == nullptr || !aligned(o_part, 16) || !aligned(lse_part, 4))
    return SMLA_ERR_INVALID_ARG;
  if (num_splits < 1 || num_splits > max_splits(p)) return SMLA_ERR_INVALID_ARG;
  int sms = 0;
  st = current_device_sms(&sms);
  if (st != SMLA_OK) return st;
  const cudaError_t e = smla::launch_split(q, kv_cache, indices, o_part, lse_part, p->batch,
                                           p->num_heads, p->topk, num_splits, p->num_rows,
                                           p->kv_row_stride, p->softmax_scale,
                                           reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

int sparse_mla_combine(const float* o_part, const float* lse_part, int32_t batch,
                       int32_t num_heads, int32_t num_splits, void* out, float* lse,
                       smla_stream_t stream) {
  if (o_part == nullptr || lse_part == nullptr || out == nullptr || lse == nullptr)
    return SMLA_ERR_INVALID_ARG;
  if (!aligned(o_part, 8) || !aligned(lse_part, 4) || !aligned(out, 16) || !aligned(lse, 4))
    return SMLA_ERR_INVALID_ARG;
  if (batch < 1 || num_heads < 1 || num_splits < 1 || num_splits > kMaxCombineSplits)
    return SMLA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(batch) * num_heads > (int64_t(1) << 30))
    return SMLA_ERR_UNSUPPORTED_SHAPE;
  int sms = 0;
  const int st = current_device_sms(&sms);
  if (st != SMLA_OK) return st;
  const cudaError_t e = smla::launch_combine(o_part, lse_part, batch, num_heads, num_splits, out,
                                             lse, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

int sparse_mla_decode(const void* q, const void* kv_cache, const int32_t* indices, void* out,
                      float* lse, const smla_params* p, int32_t num_splits, void* workspace,
                      size_t workspace_bytes, smla_stream_t stream) {
  int st = check_params(p);
  if (st != SMLA_OK) return st;
  st = check_tensors(q, kv_cache, indices);
  if (st != SMLA_OK) return st;
  if (out == nullptr || lse == nullptr || !aligned(out, 16) || !aligned(lse, 4))
    return SMLA_ERR_INVALID_ARG;
  int S = 0;
  st = resolve_splits(p, num_splits, &S);
  if (st != SMLA_OK) return st;
  size_t o_bytes = 0, total = 0;
  workspace_layout(p, S, &o_bytes, &total);
  if (workspace == nullptr || !aligned(workspace, 256)) return SMLA_ERR_INVALID_ARG;
  if (workspace_bytes < total) return SMLA_ERR_WORKSPACE_TOO_SMALL;
  int sms = 0;
  st = current_device_sms(&sms);    // an explicit split count skips the plan's check
  if (st != SMLA_OK) return st;
  return smla::launch_step(q, kv_cache, indices, out, lse, p, S, workspace,
                           reinterpret_cast<cudaStream_t>(stream));
}

int smla_paged_workspace_size(const smla_params* p, int32_t num_splits, size_t* bytes) {
  size_t total = 0;
  const int st = smla_workspace_size(p, num_splits, &total);
  if (st != SMLA_OK) return st;
  *bytes = total + round256(static_cast<size_t>(p->batch) * p->topk * sizeof(int32_t));
  return SMLA_OK;
}

int sparse_mla_decode_paged(const void* q, const void* kv_pages, const int32_t* block_table,
                            int32_t max_pages_per_seq, int32_t page_size, const int32_t* indices,
                            void* out, float* lse, const smla_params* p, int32_t num_splits,
                            void* workspace, size_t workspace_bytes, smla_stream_t stream) {
  int st = check_params(p);
  if (st != SMLA_OK) return st;
  st = check_tensors(q, kv_pages, indices);
  if (st != SMLA_OK) return st;
  if (block_table == nullptr || !aligned(block_table, 4) || max_pages_per_seq < 1 || page_size < 1)
    return SMLA_ERR_INVALID_ARG;
  if (out == nullptr || lse == nullptr || !aligned(out, 16) || !aligned(lse, 4))
    return SMLA_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned(workspace, 256)) return SMLA_ERR_INVALID_ARG;
  size_t total = 0, need = 0;
  st = smla_workspace_size(p, num_splits, &total);
  if (st != SMLA_OK) return st;
  st = smla_paged_workspace_size(p, num_splits, &need);
  if (st != SMLA_OK) return st;
  if (workspace_bytes < need) return SMLA_ERR_WORKSPACE_TOO_SMALL;
  int sms = 0;
  st = current_device_sms(&sms);
  if (st != SMLA_OK) return st;
  // the translated rows sit after the decode's own part of the workspace
  int32_t* rows = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + total);
  const cudaError_t e = smla::launch_paged_rows(indices, block_table, p->batch, p->topk,
                                                max_pages_per_seq, page_size, p->num_rows, rows,
                                                reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return SMLA_ERR_CUDA;
  return sparse_mla_decode(q, kv_pages, rows, out, lse, p, num_splits, workspace, total, stream);
}

int sparse_mla_decode_simt(const void* q, const void* kv_cache, const int32_t* indices,
                           void* out, float* lse, const smla_params* p, smla_stream_t stream) {
  int st = check_params(p);
  if (st != SMLA_OK) return st;
  st = check_tensors(q, kv_cache, indices);
  if (st != SMLA_OK) return st;
  if (out == nullptr || lse == nullptr || !aligned(out, 16) || !aligned(lse, 4))
    return SMLA_ERR_INVALID_ARG;
  if (p->batch > 65535) return SMLA_ERR_UNSUPPORTED_SHAPE;
  int sms = 0;
  st = current_device_sms(&sms);
  if (st != SMLA_OK) return st;
  const cudaError_t e = smla::launch_simt(q, kv_cache, indices, out, lse, p->batch, p->num_heads,
                                          p->topk, p->num_rows, p->kv_row_stride,
                                          p->softmax_scale, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

const char* smla_status_string(int status) {
  switch (status) {
    case SMLA_OK: return "SMLA_OK";
    case SMLA_ERR_INVALID_ARG: return "SMLA_ERR_INVALID_ARG: invalid argument";
    case SMLA_ERR_UNSUPPORTED_SHAPE: return "SMLA_ERR_UNSUPPORTED_SHAPE: unsupported shape";
    case SMLA_ERR_WORKSPACE_TOO_SMALL: return "SMLA_ERR_WORKSPACE_TOO_SMALL: workspace too small";
    case SMLA_ERR_UNSUPPORTED_DEVICE:
      return "SMLA_ERR_UNSUPPORTED_DEVICE: needs a compute capability 10.3 GPU";
    case SMLA_ERR_CUDA: return "SMLA_ERR_CUDA: CUDA runtime error";
    case SMLA_ERR_TIMEOUT: return "SMLA_ERR_TIMEOUT: a bounded wait in a kernel ran out";
    case SMLA_ERR_INDEX_RANGE: return "SMLA_ERR_INDEX_RANGE: an index >= num_rows was skipped";
    case SMLA_ERR_RANGE: return "SMLA_ERR_RANGE: a q or KV value exceeds the f16 operand range";
    case SMLA_ERR_SCRATCH_TOO_SMALL:
      return "SMLA_ERR_SCRATCH_TOO_SMALL: split partials exceed the 16 MiB built-in scratch";
    case SMLA_ERR_INTERNAL:
      return "SMLA_ERR_INTERNAL: a debug-build bounds check failed (access skipped)";
    default: return "SMLA: unknown status";
  }
}

int smla_test_inject_fault(int32_t block) {
  if (block < -1) return SMLA_ERR_INVALID_ARG;
  smla::set_fault_block(block);
  return SMLA_OK;
}

int smla_device_status(int32_t* status, int32_t clear) {
  if (status == nullptr) return SMLA_ERR_INVALID_ARG;
  int sms = 0;
  const int st = current_device_sms(&sms);
  if (st != SMLA_OK) return st;
  return smla::read_device_status(status, clear != 0) == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

}  // extern "C"
