/*
 * smla.h -- C ABI of the GB300 (sm_103a) sparse MLA decode library (libsmla.so).
 *
 * The operation.  Sparse Multi-head Latent Attention decode: for every decode
 * query b and head h, softmax attention over the top-k KV-cache rows selected for
 * that query, all heads sharing one gathered read of the rows ("The Moment of
 * Compilation: When a Triton Kernel Meets Its Constraints", section "The Context:
 * A Kernel Optimization Campaign": one KV read shared by all heads, scores for all
 * heads in one batched matrix product).  Row format ("The Power-of-Two Trap:
 * Debugging a Triton MMA Kernel on Blackwell GPUs", sections "3. The Scale
 * Indexing Complication" and "Input Knowledge Required"), 584 bytes per row:
 *
 *     [0,448)   FP8 e4m3 nope values        k_nope[c] = e4m3(byte c) * 2^(s[c/64]-127)
 *     [448,455) UE8M0 scale of each 64-column group s[0..6]
 *     455       padding byte (never used)
 *     [456,584) 64 bf16 rope values (little endian)
 *
 * With q = bf16 [512] = q_nope[448] | q_rope[64] and scale = softmax_scale:
 *     score[t] = scale * (q_nope . k_nope[t] + q_rope . k_rope[t])
 *     lse      = ln sum_t exp(score[t])
 *     out      = sum_t exp(score[t] - lse) * k_nope[t]          (448 wide)
 * over the valid (>= 0) indices of the query; no valid index gives out = 0 and
 * lse = -inf.  The split-K form ("The 80KB Mystery: Resolving Contradictory
 * Evidence in Triton Kernel Optimization", section "The Context: Optimizing
 * Attention on Blackwell": the top-k is partitioned across CTAs, nsplit) computes
 * the same quantities per split of the index list, and the combine merges them:
 *     lse = ln sum_s exp(lse_s),   out = sum_s exp(lse_s - lse) * out_s.
 *
 * Conventions common to every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library keeps
 *     no pointer after a call returns and allocates no device or host memory.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream).  They do not
 *     synchronise the host and allocate nothing, so they may be captured in a CUDA
 *     graph once the device has been initialised by one eager call.
 *   - The decode and combine kernels are launched with programmatic stream
 *     serialization (programmatic dependent launch): a kernel may be scheduled
 *     while the previous kernel in the stream is still running, and it waits for
 *     that kernel to complete (griddepcontrol.wait) before its first access to
 *     global memory, so stream order holds for every input, output and workspace
 *     byte.  The kernels also allow the next kernel in the stream to be scheduled
 *     early; a caller's kernel launched with the same attribute must wait the same
 *     way before it reads this library's outputs (one launched without it simply
 *     waits for completion).
 *   - Layouts are dense, row-major, with the shapes given.  bf16 means IEEE
 *     bfloat16 bit patterns (uint16).
 *   - Return value: SMLA_OK (0) or a negative smla_status.  Argument errors are
 *     detected on the host before any launch; nothing is launched then.
 *   - Index values >= num_rows violate the contract.  The kernels never read such a
 *     row: they treat it as masked and record SMLA_ERR_INDEX_RANGE in the device
 *     status word (see smla_device_status).
 */
#ifndef SMLA_H_
#define SMLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* smla_stream_t; /* == cudaStream_t */

enum smla_status {
  SMLA_OK = 0,
  SMLA_ERR_INVALID_ARG = -1,        /* null pointer, bad alignment, bad size          */
  SMLA_ERR_UNSUPPORTED_SHAPE = -2,  /* num_heads not in {16, 32, 64, 128}, batch > 65535, ... */
  SMLA_ERR_WORKSPACE_TOO_SMALL = -3,
  SMLA_ERR_UNSUPPORTED_DEVICE = -4, /* current device is not compute capability 10.3 */
  SMLA_ERR_CUDA = -5,               /* a CUDA runtime call or launch failed           */
  SMLA_ERR_TIMEOUT = -6,            /* device status: a bounded wait in a kernel ran out */
  SMLA_ERR_INDEX_RANGE = -7,        /* device status: an index >= num_rows was skipped */
  SMLA_ERR_RANGE = -8,              /* device status: a q or dequantised KV value is
                                       outside the f16 range of the tensor-core operands */
  SMLA_ERR_SCRATCH_TOO_SMALL = -9,  /* sparse_mla_decode_noalloc: the split partials need
                                       more than its built-in 16 MiB scratch */
  SMLA_ERR_INTERNAL = -10,          /* device status, debug build (libsmla_debug.so, built
                                       with SMLA_DEBUG) only: a computed shared-memory
                                       address or gathered row fell outside its buffer;
                                       the access was skipped */
};

/* Problem description shared by the entry points. */
typedef struct smla_params {
  int32_t batch;          /* B: decode queries (one token each), 1 .. 65535            */
  int32_t num_heads;      /* H: query heads, one of 16, 32, 64, 128                    */
  int32_t topk;           /* k: index slots per query, 1 .. 65536                      */
  int32_t reserved;       /* must be 0                                                 */
  int64_t num_rows;       /* rows in kv_cache, >= 1                                    */
  int64_t kv_row_stride;  /* bytes between consecutive rows, >= 584, multiple of 8      */
  float softmax_scale;    /* multiplies q.k (e.g. 1/sqrt(512)), finite and > 0          */
} smla_params;

/* Number of splits the library would use for `p` on the current device (its plan:
 * enough CTAs to fill the device's SMs, splits aligned to 16 index slots).  */
int smla_default_num_splits(const smla_params* p, int32_t* num_splits);

/* Workspace bytes sparse_mla_decode needs with `num_splits` splits (0 = the default
 * plan).  The workspace holds the split partials: fp32 o_part [B, H, S, 448] and
 * fp32 lse_part [B, H, S], each 256-byte aligned. */
int smla_workspace_size(const smla_params* p, int32_t num_splits, size_t* bytes);

/* How sparse_mla_decode runs for `p` with `num_splits` splits (0 = the default plan)
 * on the current device: *splits receives the resolved split count; *fused is 1 when
 * the splits of each (query, head group) run as one thread-block cluster that also
 * merges them (one launch: each split keeps its partial in its shared memory, and
 * after a cluster barrier each CTA merges a slice of the heads, reading the other
 * splits' partials through distributed shared memory), 0 when a separate
 * combine kernel merges them.  Either way this is the split-K scheme of "The 80KB
 * Mystery: Resolving Contradictory Evidence in Triton Kernel Optimization", section
 * "The Context: Optimizing Attention on Blackwell".  Clusters need splits <= 8 and
 * a device with room for such a cluster. */
int smla_decode_plan(const smla_params* p, int32_t num_splits, int32_t* splits, int32_t* fused);

/*
 * One whole decode step: the split-K attention and the merge of its splits, as one
 * clustered launch when smla_decode_plan reports fused, else split + combine kernels
 * (the workspace holds the split partials for the combine kernel; the clustered
 * launch merges on chip and leaves it untouched).  With 64 heads per CTA (H = 64 or
 * 128) the rows and q are read by tensor (TMA) copies whose descriptors are encoded
 * on the host for each call, through the driver's cuTensorMapEncodeTiled (looked up
 * once via the runtime); a driver without it, or a cache or q the encoder rejects,
 * gives SMLA_ERR_CUDA and nothing is launched.
 *   q          bf16  [B, H, 512]  (448 nope | 64 rope), 16-byte aligned
 *   kv_cache   uint8 [num_rows, kv_row_stride], 16-byte aligned, rows as above
 *   indices    int32 [B, topk]    row ids; < 0 = masked slot (shared by all heads)
 *   out        bf16  [B, H, 448]  16-byte aligned
 *   lse        fp32  [B, H]       natural-log LSE of the scaled scores (-inf if empty)
 *   workspace  device scratch of >= smla_workspace_size(p, num_splits) bytes,
 *              256-byte aligned; its contents on entry do not matter
 *   num_splits 0 = default plan, else 1 .. min(256, ceil(topk / 16))
 */
int sparse_mla_decode(const void* q, const void* kv_cache, const int32_t* indices,
                      void* out, float* lse, const smla_params* p, int32_t num_splits,
                      void* workspace, size_t workspace_bytes, smla_stream_t stream);

/*
 * Split kernel alone.  Split s covers index positions [16*g0, min(16*g1, topk)) with
 * G = ceil(topk/16), g0 = s*G/S, g1 = (s+1)*G/S (integer division); a split may be
 * empty.  Writes, per split, the normalised partial attention and its LSE:
 *   o_part   fp32 [B, H, S, 448]   (0 where the split has no valid index)
 *   lse_part fp32 [B, H, S]        (-inf where the split has no valid index)
 * num_splits: 1 .. min(256, ceil(topk / 16)).
 */
int sparse_mla_decode_split(const void* q, const void* kv_cache, const int32_t* indices,
                            const smla_params* p, int32_t num_splits, float* o_part,
                            float* lse_part, smla_stream_t stream);

/*
 * Combine kernel alone: merges S split partials per (b, h) with log-sum-exp weights.
 *   o_part fp32 [B, H, S, 448], lse_part fp32 [B, H, S]  (as written by the split call)
 *   out bf16 [B, H, 448] (16-byte aligned), lse fp32 [B, H]
 * Splits with lse_part = -inf carry no weight; all -inf gives out = 0, lse = -inf.
 * 1 <= S <= 1024.
 */
int sparse_mla_combine(const float* o_part, const float* lse_part, int32_t batch,
                       int32_t num_heads, int32_t num_splits, void* out, float* lse,
                       smla_stream_t stream);

/*
 * The decode step over a paged cache.  "The Power-of-Two Trap: Debugging a Triton MMA
 * Kernel on Blackwell GPUs", section "Input Knowledge Required", says the KV cache is
 * paged but gives no layout; this entry point takes the usual one:
 *   kv_pages    uint8 [num_rows, kv_row_stride]: a pool of pages of page_size
 *               consecutive rows (num_rows = pool rows, params as for
 *               sparse_mla_decode), 16-byte aligned
 *   block_table int32 [B, max_pages_per_seq]: page ids of each query's sequence,
 *               < 0 = unmapped page
 *   indices     int32 [B, topk]: logical token positions in the sequence, < 0 = masked
 * Position t of query b is row block_table[b][t / page_size] * page_size +
 * t % page_size.  Positions on an unmapped page are masked; positions past the table
 * or rows past the pool are masked and reported as SMLA_ERR_INDEX_RANGE in the
 * device status word.  The workspace (smla_paged_workspace_size bytes, 256-byte
 * aligned) also holds the translated rows; a small translation kernel runs first,
 * then the decode as in sparse_mla_decode.  page_size >= 1, max_pages_per_seq >= 1.
 */
int smla_paged_workspace_size(const smla_params* p, int32_t num_splits, size_t* bytes);
int sparse_mla_decode_paged(const void* q, const void* kv_pages, const int32_t* block_table,
                            int32_t max_pages_per_seq, int32_t page_size, const int32_t* indices,
                            void* out, float* lse, const smla_params* p, int32_t num_splits,
                            void* workspace, size_t workspace_bytes, smla_stream_t stream);

/*
 * The same decode step computed the way the pages' production kernel did before the
 * tensor-core rewrite: one CTA per (query, head), element-wise fp32 arithmetic, and
 * every head reading the selected rows again ("The Moment of Compilation: When a
 * Triton Kernel Meets Its Constraints", sections "The Context: A Kernel
 * Optimization Campaign" and "The Assumption That Broke").  It is a same-device
 * reference point for the tensor-core path, not a faster alternative.  Arguments as
 * for sparse_mla_decode (no workspace, no splits); batch <= 65535.
 */
int sparse_mla_decode_simt(const void* q, const void* kv_cache, const int32_t* indices,
                           void* out, float* lse, const smla_params* p, smla_stream_t stream);

/*
 * sparse_mla_decode without a caller-provided workspace.  The pages have no
 * counterpart to this entry point; it exists for callers that cannot allocate
 * device memory: for example code that runs inside another framework's memory
 * pool or a serving loop that must never call cudaMalloc (it can synchronise the
 * device and fail under memory pressure).  Such a caller still owns q, kv_cache,
 * indices, out and lse; only the split partials move into a scratch array that the
 * library itself holds: 16 MiB of device memory in every GPU process that loads the
 * library, kept until the process exits.  The function allocates nothing and calls
 * no cudaMalloc, cudaFree or allocating library routine.
 *   - Same arguments and results as sparse_mla_decode, minus the workspace.
 *   - num_splits = 0 takes the default plan, or the largest smaller split count
 *     whose partials (smla_workspace_size bytes) fit in the scratch; an explicit
 *     num_splits whose partials do not fit, or a problem for which even one split
 *     does not fit (batch * num_heads above about 9300), returns
 *     SMLA_ERR_SCRATCH_TOO_SMALL before anything is launched.
 *   - It runs the same kernels as sparse_mla_decode with the resolved split count
 *     (one clustered launch that also merges the splits, or split + combine).
 *   - The first call on each device looks up the scratch array's device address
 *     (cudaGetSymbolAddress) with that device current and caches it; make that first
 *     call before any stream capture on the device.  The cached address does not
 *     survive cudaDeviceReset: a call that fails with SMLA_ERR_CUDA drops it, and
 *     the next call looks it up again.  The cache is guarded by a mutex.
 *   - All calls in the process share the one scratch array, which keeps the last
 *     call's partials (every partial a call reads is written by the same call, so
 *     nothing needs clearing).  Calls whose kernels overlap on the GPU (several
 *     streams, or several host threads) race on it and must be serialised by the
 *     caller.
 */
int sparse_mla_decode_noalloc(const void* q, const void* kv_cache, const int32_t* indices,
                              void* out, float* lse, const smla_params* p, int32_t num_splits,
                              smla_stream_t stream);

/*
 * Test hook for the failure path of the decode kernels; the pages have no
 * counterpart.  With block >= 0, every later launch of the decode kernels (any
 * device, any thread) runs with one converter warp of every CTA withholding its
 * "block filled" signal for block `block` (64 index slots) of its split, and with
 * its bounded waits shortened to about 10 ms of SM clocks: the tensor-core warp's
 * wait for that block then runs out, the CTA records SMLA_ERR_TIMEOUT in the device
 * status word (smla_device_status), every role leaves through its bounded waits and
 * the epilogue, and the launch completes without a fault; its outputs are undefined.
 * CTAs whose split has no such block are unaffected.  block = -1 switches the hook
 * off.  Returns SMLA_OK, or SMLA_ERR_INVALID_ARG for block < -1.  Not for use in
 * production; calls made while it is on are not thread-safe with respect to it.
 */
int smla_test_inject_fault(int32_t block);

/* Human-readable name of a status code (static string, never NULL). */
const char* smla_status_string(int status);

/* Reads the current device's status word, which kernels set (first error wins) when
 * a bounded wait runs out (SMLA_ERR_TIMEOUT) or an index is out of range
 * (SMLA_ERR_INDEX_RANGE).  Synchronises the device.  clear != 0 resets it to 0. */
int smla_device_status(int32_t* status, int32_t clear);

#ifdef __cplusplus
}
#endif
#endif /* SMLA_H_ */
