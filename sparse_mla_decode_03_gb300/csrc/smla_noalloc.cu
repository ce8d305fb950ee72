// sparse_mla_decode_noalloc: the whole decode step with the split partials kept in a
// fixed scratch array that belongs to the library, for callers
// that cannot allocate device memory.  Declared and documented in include/smla.h.
#include <cstdint>
#include <mutex>

#include "../../include/smla.h"
#include "smla_internal.h"

namespace {

// Built-in scratch for the split partials: fp32 o_part [B, H, S, 448] followed by
// fp32 lse_part [B, H, S], each 256-byte aligned.  Every GPU that loads the library
// holds it until the process exits.
constexpr size_t kScratchBytes = size_t(16) << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;                       // guards g_scratch_ptr
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device.  The host-side name
// g_noalloc_scratch is only a stand-in for the symbol, so the address is looked
// up once per device (with that device current) and cached.
int scratch_address(int dev, void** ptr) {
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return SMLA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *ptr = g_scratch_ptr[dev];
  return SMLA_OK;
}

// Forgets the cached address of a device (after a CUDA error, which may come from a
// reset device whose module, and with it the scratch, was reloaded elsewhere).
void forget_scratch_address(int dev) {
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  g_scratch_ptr[dev] = nullptr;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" int sparse_mla_decode_noalloc(const void* q, const void* kv_cache,
                                         const int32_t* indices, void* out, float* lse,
                                         const smla_params* p, int32_t num_splits,
                                         smla_stream_t stream) {
  // Validates p (and a non-default num_splits) exactly as the other entry points do.
  size_t need = 0;
  int st = smla_workspace_size(p, num_splits, &need);
  if (st != SMLA_OK) return st;
  if (q == nullptr || kv_cache == nullptr || indices == nullptr || out == nullptr ||
      lse == nullptr)
    return SMLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(indices, 4) || !aligned(out, 16) ||
      !aligned(lse, 4))
    return SMLA_ERR_INVALID_ARG;
  int32_t S = num_splits;
  if (S == 0) {
    st = smla_default_num_splits(p, &S);
    if (st != SMLA_OK) return st;
    // the default plan, or the largest split count below it whose partials fit
    while (S > 1 && smla_workspace_size(p, S, &need) == SMLA_OK && need > kScratchBytes) --S;
  }
  st = smla_workspace_size(p, S, &need);
  if (st != SMLA_OK) return st;
  if (need > kScratchBytes) return SMLA_ERR_SCRATCH_TOO_SMALL;
  st = smla::check_device();
  if (st != SMLA_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SMLA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SMLA_ERR_UNSUPPORTED_DEVICE;
  void* scratch = nullptr;
  st = scratch_address(dev, &scratch);
  if (st != SMLA_OK) return st;
  // the same launches as sparse_mla_decode with this split count, the scratch as
  // its workspace
  st = smla::launch_step(q, kv_cache, indices, out, lse, p, S, scratch,
                         reinterpret_cast<cudaStream_t>(stream));
  if (st == SMLA_ERR_CUDA) forget_scratch_address(dev);
  return st;
}
