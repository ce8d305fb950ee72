// Paged KV cache: translation of logical token positions into physical rows of a page
// pool, ahead of the decode kernels.  "The Power-of-Two Trap: Debugging a Triton MMA
// Kernel on Blackwell GPUs", section "Input Knowledge Required", states that the
// model's KV cache is paged; the pages give no layout, so this file takes the usual
// one: a pool of pages of `page_size` consecutive 584-byte rows, and per query a
// block table of page ids, so that logical position t of query b is row
//     block_table[b][t / page_size] * page_size + t % page_size.
#include "../../include/smla.h"
#include "smla_internal.h"

namespace smla {
namespace {

__global__ void paged_rows_kernel(const int32_t* __restrict__ indices,
                                  const int32_t* __restrict__ table, int64_t n, int topk,
                                  int max_pages, int page_size, int64_t num_rows,
                                  int32_t* __restrict__ rows, int* __restrict__ status) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int32_t pos = indices[i];
    int32_t row = -1;
    if (pos >= 0) {
      const int64_t b = i / topk;
      const int32_t page = pos / page_size;
      if (page >= max_pages) {
        atomicCAS(status, 0, SMLA_ERR_INDEX_RANGE);
      } else {
        const int32_t phys = table[b * max_pages + page];
        if (phys >= 0) {
          const int64_t r = static_cast<int64_t>(phys) * page_size + pos % page_size;
          if (r < num_rows && r <= INT32_MAX) {
            row = static_cast<int32_t>(r);
          } else {
            atomicCAS(status, 0, SMLA_ERR_INDEX_RANGE);
          }
        }
      }
    }
    rows[i] = row;
  }
}

}  // namespace

cudaError_t launch_paged_rows(const int32_t* indices, const int32_t* block_table, int B, int topk,
                              int max_pages, int page_size, int64_t num_rows, int32_t* rows,
                              cudaStream_t stream) {
  int* status = nullptr;
  cudaError_t e = status_word_address(&status);
  if (e != cudaSuccess) return e;
  const int64_t n = static_cast<int64_t>(B) * topk;
  const int threads = 256;
  const int64_t blocks64 = (n + threads - 1) / threads;
  const int blocks = static_cast<int>(blocks64 < 4096 ? blocks64 : 4096);
  paged_rows_kernel<<<blocks, threads, 0, stream>>>(indices, block_table, n, topk, max_pages,
                                                     page_size, num_rows, rows, status);
  return cudaGetLastError();
}

}  // namespace smla
