// pkv_internal.h -- host-side declarations shared by the translation units of
// libpkv (not part of the public C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// Which decode kernel runs and how the context is partitioned.
struct DecodePlan {
  int kernel;          // 2: wide-group tcgen05 kernel, 1: TMA + tensor-core kernel, 0: CUDA-core kernel
  int P;               // partition size in tokens (multiple of 16)
  int max_parts;       // partitions per sequence the grid covers
  int heads_per_cta;   // query heads served by one CTA
  int gchunks;         // CTAs per KV head (ceil(G / heads_per_cta))
  int stages;          // TMA pipeline depth per warp
  int threads;         // threads per CTA
  size_t smem_bytes;   // dynamic shared memory per CTA
  int part_major;      // tensor-core kernel: the partition is the grid's slowest index
};

// Heads one tensor-core CTA serves (the M = 16 rows of one mma tile).
constexpr int kTcHeads = 16;
// Partitions per sequence the automatic partition size never exceeds.
constexpr int kMaxAutoParts = 64;
// Shared memory a block may opt in to on sm_100-class GPUs (used when no
// device is queried).
constexpr size_t kDefaultSmemOptin = 232448;

// Whether a decode launch on `stream` goes out as a programmatic dependent
// of the kernel before it: only while the stream is being captured into a
// graph, where consecutive steps run back to back and one launch's start-up
// can overlap the previous one's tail.  Launched eagerly (a step at a time,
// synchronised), the attribute bought nothing and cost a little.
inline bool launch_as_dependent(cudaStream_t stream) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  return cudaStreamIsCapturing(stream, &st) == cudaSuccess && st == cudaStreamCaptureStatusActive;
}

bool tc_eligible(pkv_dtype dt, int D, int bs);
// Fills *plan; returns false for sizes no kernel handles.
bool make_plan(int B, int H, int KVH, int D, int bs, int max_blocks, int max_context_len,
               int partition_size, pkv_dtype dt, int num_sms, size_t smem_optin, bool aligned16,
               DecodePlan *plan, bool allow_wide = true, int force_kernel = -1);
// Every host-side check of a decode call except the workspace's, then the
// plan (force_kernel: -1 automatic, else the kernel number of
// DecodePlan::kernel).  *empty: B == 0, nothing to enqueue.
pkv_status decode_check_and_plan(const void *out, const void *q, const void *k_cache,
                                 const void *v_cache, const int32_t *block_tables,
                                 const int32_t *context_lens, int B, int H, int num_kv_heads,
                                 int head_dim, int block_size, int max_blocks, int64_t num_blocks,
                                 pkv_dtype dt, int max_context_len, int partition_size,
                                 bool xpacked, int force_kernel, DecodePlan *plan, int *num_sms,
                                 bool *empty);
size_t workspace_bytes_for(int B, int H, int D, int max_parts);
// Bytes at the start of the workspace that must be zero before a call (the
// work queue and the per-(sequence, head group) counters).
size_t workspace_counter_bytes(int B, int H);

pkv_status launch_write(void *k_cache, void *v_cache, const void *k, const void *v,
                        const int64_t *slot_mapping, int64_t T, int64_t k_stride, int64_t v_stride,
                        int64_t num_blocks, int bs, int KVH, int D, int elem, int *err,
                        cudaStream_t stream);

// Tensor map of a [num_blocks, bs, KVH, D] 16-bit cache: box of 64 elements
// x 1 head x 16 rows x 1 block, 128-byte swizzle (false if unavailable).
bool encode_cache_map(CUtensorMap *map, const void *cache, pkv_dtype dt, long long num_blocks,
                      int bs, int KVH, int D);

// Tensor map of a [rows, H, D] 16-bit tensor: box of 64 elements x 1 head x
// box_rows rows, 128-byte swizzle, zero past the last row.
bool encode_rows_map(CUtensorMap *map, const void *base, pkv_dtype dt, long long rows, int H, int D,
                     int box_rows);

// One-time opt-in to a kernel's dynamic shared memory, per device
// (`configured` is the kernel's own per-device record).
template <typename K>
inline bool allow_smem(K kern, size_t bytes, int *configured) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (dev < 64 && configured[dev] >= (int)bytes) return true;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) !=
      cudaSuccess)
    return false;
  if (dev < 64) configured[dev] = (int)bytes;
  return true;
}

// Persistent varlen prefill: pairs_bound bounds the (sequence, 256-query
// tile) pairs, q_tiles the tiles of one sequence.
pkv_status launch_prefill_tc(void *out, const void *q, const void *k_cache, const void *v_cache,
                             const int32_t *tables, const int32_t *cu_q, const int32_t *lens,
                             int B, long long total_q, int H, int KVH, int D, int bs,
                             int max_blocks, long long num_blocks, float scale, pkv_dtype dt,
                             int q_tiles, int pairs_bound, int *err, cudaStream_t stream);

pkv_status launch_write_xpacked(void *kx, void *vx, const void *k, const void *v,
                                const int64_t *slots, long long ntok, long long k_stride,
                                long long v_stride, long long num_blocks, int KVH, int D,
                                pkv_dtype dt, int *err, cudaStream_t stream);

struct DecodeArgs;
pkv_status launch_decode_xpacked(const DecodeArgs &a, const DecodePlan &plan, pkv_dtype dt,
                                 cudaStream_t stream);
pkv_status launch_decode_simt(const DecodeArgs &a, const DecodePlan &plan, pkv_dtype dt,
                              cudaStream_t stream);
pkv_status launch_decode_tc(const DecodeArgs &a, const DecodePlan &plan, pkv_dtype dt,
                            cudaStream_t stream);
// Wide query groups (16 query heads per KV head, D of 128 or 256): the
// persistent tensor-core decode with tokens as the product's M.
size_t wide_smem_bytes(int D);
pkv_status launch_decode_wide(const DecodeArgs &a, pkv_dtype dt, int num_sms, bool auto_items,
                              cudaStream_t stream);

}  // namespace pkv
