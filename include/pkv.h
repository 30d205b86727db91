/*
 * pkv.h -- C ABI of the paged KV-cache library for one NVIDIA GB300 (sm_103a).
 *
 * Two operations, as the course page "P09 · Paged KV 写入 + decode attention
 * （参考实现）" (kuanzhou.online, nano-vllm-omni drills) defines them in its
 * section 题面速览 and its two shape-trace tables (框架视角 · shape trace):
 *
 *   pkv_write             write_kv: cache[slot // bs, slot % bs] = k[i] (and v),
 *                         in place; a negative slot is a padding token and is
 *                         not written.
 *   pkv_decode_attention  paged decode attention: each sequence's single query
 *                         attends to the first context_lens[b] tokens of its
 *                         paged context, gathered through block_tables[b, :nb]
 *                         with nb = ceil(n / bs); query head h reads KV head
 *                         h // (H / KVH); softmax(q . K^T * scale) . V with the
 *                         softmax in fp32, output in q's dtype.
 * Long contexts are split into partitions whose partial results are merged
 * with a log-sum-exp rescale, the partitioned variant the interview note
 * "PagedAttention kernel: paged KV cache 与 block table"
 * (inference-learning-path.pages.dev), section 深入原理 ("v1 vs v2"),
 * describes; the result equals the unsplit one up to rounding.
 *
 * Common rules
 *   - Every pointer argument except the host-side ones named below is a
 *     DEVICE pointer on the current CUDA device.  The caller owns all memory;
 *     the library allocates nothing on the call path and keeps no pointer
 *     after a call returns.
 *   - All work is enqueued on `stream` (NULL = the legacy default stream);
 *     calls return once the work is enqueued, before it runs.
 *   - Argument errors that need no device data are caught on the host before
 *     anything is enqueued and returned as a status.
 *   - Errors that depend on device data (a slot past the pool, a table entry
 *     outside [0, num_blocks), an over-long context) cannot be seen on the
 *     host: the kernels skip the offending access and OR a PKV_FLAG_* bit into
 *     *err_flags (a device int, may be NULL).  The caller reads it after the
 *     stream has synchronised.  Nothing in the library traps or asserts on
 *     the device.
 *   - Cache layout: K and V are separate tensors
 *     [num_blocks, block_size, num_kv_heads, head_dim], contiguous, one
 *     token's row of num_kv_heads * head_dim elements contiguous.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* The same handle type as cudaStream_t (a CUstream). */
typedef struct CUstream_st *pkv_stream_t;

typedef enum pkv_status {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,   /* a size, pointer, alignment or count is not valid */
  PKV_ERR_UNSUPPORTED = 2,   /* valid, but a shape/dtype this build does not handle */
  PKV_ERR_CUDA = 3,          /* a CUDA runtime call or a kernel launch failed */
  PKV_ERR_WORKSPACE = 4,     /* the workspace is missing or smaller than needed */
  PKV_ERR_OUT_OF_BLOCKS = 5  /* block manager (pkv_block_manager.h): not enough free blocks */
} pkv_status;

typedef enum pkv_dtype {
  PKV_F32 = 0,   /* float32 */
  PKV_BF16 = 1,  /* bfloat16 */
  PKV_F16 = 2    /* float16 */
} pkv_dtype;

/* Bits the kernels OR into *err_flags. */
#define PKV_FLAG_SLOT_OUT_OF_RANGE 0x1   /* pkv_write: slot >= num_blocks * block_size; token skipped */
#define PKV_FLAG_BLOCK_OUT_OF_RANGE 0x2  /* decode: an entry of block_tables[b, :nb] outside
                                            [0, num_blocks); block 0 is read in its place and
                                            that sequence's output is unspecified */
#define PKV_FLAG_CONTEXT_TOO_LONG 0x4    /* decode: context_lens[b] > max_blocks * block_size;
                                            clamped, output of that sequence unspecified */
#define PKV_FLAG_CONTEXT_NEGATIVE 0x8    /* decode: context_lens[b] < 0; treated as 0 */
#define PKV_FLAG_CONTEXT_OVER_HINT 0x10  /* decode: context_lens[b] > max_context_len (the host
                                            hint sized the grid too small); output of that
                                            sequence unspecified */
#define PKV_FLAG_TIMEOUT 0x20            /* a bounded wait for an asynchronous copy ran out
                                            (should never happen); outputs unspecified, and a
                                            decode workspace used by that call must be
                                            zero-filled again before its next use */
#define PKV_FLAG_QUERY_LEN 0x80          /* prefill: a sequence with qlen < 0, qlen > context_lens[b]
                                            or a context longer than the table; skipped, its
                                            output rows unspecified */
#define PKV_FLAG_QUERY_OVER_HINT 0x100   /* prefill: a sequence has more queries than max_q_len;
                                            rows past max_q_len are not computed */
#define PKV_FLAG_APPEND_MISMATCH 0x40    /* pkv_write_decode_attention: a kept slot is not the
                                            slot of position context_lens[b] - 1 through
                                            block_tables (or context_lens[b] == 0); the token
                                            is still written, that sequence's output is
                                            unspecified */

/*
 * pkv_write -- write_kv / reshape_and_cache.
 * Definition: course page "P09 · Paged KV 写入 + decode attention（参考实现）",
 * section 题面速览 ("写: cache[slot // bs, slot % bs] = k[i]") and the
 * write_kv shape trace (keep = slot >= 0; blk = s // bs; off = s % bs;
 * k_cache[blk, off] = k[keep]; same for v; in place, returns nothing).
 *
 *   k_cache, v_cache  [num_blocks, block_size, num_kv_heads, head_dim], dtype dt,
 *                     written in place (only rows named by a kept slot change)
 *   k, v              [num_tokens, num_kv_heads, head_dim]; token i starts at
 *                     element i * k_token_stride (resp. v_token_stride);
 *                     each token's num_kv_heads * head_dim elements contiguous
 *   slot_mapping      [num_tokens] int64: flat slot block * block_size + offset;
 *                     any negative value = padding, skipped silently
 *   err_flags         device int or NULL: PKV_FLAG_SLOT_OUT_OF_RANGE
 * The copy is bit-exact.  Two kept tokens with the same slot in one call
 * race (which one lands is unspecified).  num_tokens == 0 enqueues nothing.
 * Errors: PKV_ERR_INVALID_ARG for a NULL pointer with num_tokens > 0, a
 * non-positive size, or a token stride smaller than one row;
 * PKV_ERR_CUDA if the launch fails.
 */
PKV_API pkv_status pkv_write(void *k_cache, void *v_cache, const void *k, const void *v,
                             const int64_t *slot_mapping, int64_t num_tokens,
                             int64_t k_token_stride, int64_t v_token_stride,
                             int64_t num_blocks, int block_size, int num_kv_heads,
                             int head_dim, pkv_dtype dt, int *err_flags, pkv_stream_t stream);

/*
 * pkv_decode_workspace_size -- bytes of device workspace pkv_decode_attention
 * needs for these sizes (host only, no CUDA call).  partition_size as in
 * pkv_decode_attention (0 = automatic: the size covers every partition size
 * the automatic choice can make).  max_context_len: the longest context the
 * calls will see (0 = max_blocks * block_size).  Returns 0 for invalid sizes.
 *
 * The workspace holds per-partition partial results and one counter per
 * (sequence, head group).  Before its FIRST use it must be zero-filled
 * (e.g. cudaMemset); every call that completes without PKV_FLAG_TIMEOUT
 * leaves the counters at zero again, so the same workspace can be reused by
 * later calls on the same stream without clearing.  A call that raised
 * PKV_FLAG_TIMEOUT may have left a partition uncounted: zero-fill the
 * workspace again before reusing it.  Calls that run concurrently need
 * separate workspaces.
 */
PKV_API size_t pkv_decode_workspace_size(int B, int H, int num_kv_heads, int head_dim,
                                         int block_size, int max_blocks, int max_context_len,
                                         int partition_size);

/*
 * pkv_decode_attention -- paged decode attention (one query per sequence).
 * Definition: course page "P09 · Paged KV 写入 + decode attention（参考实现）",
 * section 题面速览 ("decode 读") and the paged_decode_attention shape trace:
 * n = context_lens[b]; nb = ceil(n / bs); table = block_tables[b, :nb];
 * gather k_cache[table] in table order; keep the first n rows; head h uses
 * KV head h // (H / KVH); fp32 scores times scale, softmax over the n
 * tokens in fp32, weighted sum of V, cast to q's dtype.
 *
 *   out           [B, H, head_dim], dtype dt (written; rows of sequences with
 *                 context_lens[b] == 0 are set to zero).  Device memory, or
 *                 host memory the GPU addresses directly (pinned memory under
 *                 unified addressing; any host memory where the system
 *                 translates host addresses for the GPU): the kernels only
 *                 store to out -- no reads, atomics or TMA -- so the result
 *                 crosses to the host inside the launch and needs no copy
 *                 after it.  Its rows are complete for the host once the
 *                 stream is synchronised.
 *   q             [B, H, head_dim], dtype dt
 *   k_cache, v_cache  [num_blocks, block_size, num_kv_heads, head_dim], dtype dt
 *   block_tables  [B, max_blocks] int32; only the first ceil(n/bs) entries of
 *                 row b are read -- the rest may hold anything (e.g. 99999)
 *   context_lens  [B] int32
 *   scale         multiplies q.K before the softmax (e.g. 1/sqrt(head_dim))
 *   max_context_len  host-side upper bound on context_lens (sizes the grid;
 *                 0 = max_blocks * block_size).  A longer context sets
 *                 PKV_FLAG_CONTEXT_OVER_HINT.
 *   partition_size   tokens per partition of the split-KV path: 0 = choose
 *                 from the sizes and the SM count, else a positive multiple
 *                 of 16 (any other value is PKV_ERR_INVALID_ARG), whatever
 *                 the block size (a partition may end inside a block).  A
 *                 context longer than one partition is processed by several
 *                 CTAs whose (max, sum, weighted-V) partials are merged in the
 *                 workspace with a log-sum-exp rescale.
 *   workspace, workspace_bytes  device scratch of at least
 *                 pkv_decode_workspace_size(...) bytes, 256-byte aligned,
 *                 zero-filled before first use; always required (it holds the
 *                 merge counters even when nothing is split)
 *   err_flags     device int or NULL (PKV_FLAG_BLOCK_OUT_OF_RANGE,
 *                 PKV_FLAG_CONTEXT_*, PKV_FLAG_TIMEOUT)
 * Supported: H % num_kv_heads == 0; head_dim a multiple of 8 in [8, 512] (fp32:
 * a multiple of 4); block_size >= 1; q, out, caches 16-byte aligned.  bf16 /
 * fp16 with head_dim in {64, 128, 192, 256} and block_size a multiple of 16
 * run a tensor-core kernel: groups of exactly 16 query heads per KV head at
 * head_dim 128 or 256 (MQA-like) the wide-group kernel (persistent, one CTA
 * per SM claiming (sequence, KV head, partition) items from a device
 * counter; 5th-generation tensor cores with the KV tile's tokens as the
 * product's M; with partition_size 0 its items may be larger than the
 * plan's partition -- about 1.2 CTA shares of the batch's 128-token tiles,
 * worked out on the device from context_lens -- never smaller, so the
 * workspace the plan sizes always holds them), the others the TMA +
 * mma.sync kernel; every other supported shape runs the CUDA-core kernel.
 * An explicit partition_size is used as given.  The output does not depend
 * on the partitioning beyond fp32 rounding order.
 * Inside a stream capture the tensor-core kernels launch as programmatic
 * dependents of the kernel before them (their start-up overlaps that
 * kernel's end in the graph): they read q, block_tables, context_lens and
 * (fused step) the new rows and slots before waiting for that kernel, and
 * the caches, the workspace and out only after.  So a kernel captured just
 * before them that releases its dependents early (griddepcontrol.
 * launch_dependents) must not write those inputs; this library's kernels
 * never do, and any other kernel is waited for in full.
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_WORKSPACE,
 * PKV_ERR_CUDA.  B == 0 enqueues nothing.
 */
PKV_API pkv_status pkv_decode_attention(void *out, const void *q, const void *k_cache,
                                        const void *v_cache, const int32_t *block_tables,
                                        const int32_t *context_lens, int B, int H,
                                        int num_kv_heads, int head_dim, int block_size,
                                        int max_blocks, int64_t num_blocks, float scale,
                                        pkv_dtype dt, int max_context_len, int partition_size,
                                        void *workspace, size_t workspace_bytes, int *err_flags,
                                        pkv_stream_t stream);

/*
 * pkv_decode_attention_static -- pkv_decode_attention without a workspace
 * argument, for callers that may not allocate device memory: for example an
 * engine plugin whose execute step is forbidden to call cudaMalloc, code that
 * enqueues work while some other component owns the device allocator, or a
 * deployment whose device memory is fixed when the process starts.  The
 * pages have no counterpart: this is a convenience of this library.
 *
 * Arguments, results and errors are those of pkv_decode_attention, minus
 * workspace / workspace_bytes.  The split-KV scratch comes instead from a
 * fixed array of PKV_STATIC_SCRATCH_BYTES bytes inside the library, which
 * every GPU the library runs on keeps until the process exits.
 *   - Sizes whose split-KV scratch would exceed PKV_STATIC_SCRATCH_BYTES are
 *     rejected with PKV_ERR_WORKSPACE before anything is enqueued (pass a
 *     larger partition_size, or use pkv_decode_attention with a workspace).
 *   - Every argument check of pkv_decode_attention, and the size check, is
 *     made before anything is enqueued: a rejected call enqueues nothing.
 *   - No cudaMalloc, cudaFree or other allocating call is made.  The first
 *     call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current, and keeps it for that
 *     device's context (after cudaDeviceReset it is looked up again); make
 *     that first call before any stream capture.
 *   - Each call clears the array's merge counters on `stream` before the
 *     kernel runs.  All calls share the one array: calls whose work overlaps
 *     on the GPU (different streams, or concurrent host threads) race and
 *     give wrong results; serialise them.
 */
#define PKV_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)
PKV_API pkv_status pkv_decode_attention_static(void *out, const void *q, const void *k_cache,
                                               const void *v_cache, const int32_t *block_tables,
                                               const int32_t *context_lens, int B, int H,
                                               int num_kv_heads, int head_dim, int block_size,
                                               int max_blocks, int64_t num_blocks, float scale,
                                               pkv_dtype dt, int max_context_len,
                                               int partition_size, int *err_flags,
                                               pkv_stream_t stream);

/*
 * pkv_decode_attention_with_kernel -- pkv_decode_attention with the kernel
 * named by the caller instead of chosen by the plan, for tests and tuning
 * (the pages have no counterpart: it exists to measure one kernel against
 * another on the same batch).  kernel: -1 = the plan's choice (exactly
 * pkv_decode_attention), 0 = the CUDA-core kernel (any supported shape),
 * 1 = the TMA + mma.sync tensor-core kernel, 2 = the wide-group tcgen05
 * kernel.  A kernel that cannot run the given shape returns
 * PKV_ERR_UNSUPPORTED before anything is enqueued; any other kernel value is
 * PKV_ERR_INVALID_ARG.  Arguments, workspace (sized by
 * pkv_decode_workspace_size, which covers every kernel), results and errors
 * otherwise as in pkv_decode_attention.
 */
PKV_API pkv_status pkv_decode_attention_with_kernel(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, const int32_t *context_lens, int B, int H, int num_kv_heads,
    int head_dim, int block_size, int max_blocks, int64_t num_blocks, float scale, pkv_dtype dt,
    int max_context_len, int partition_size, void *workspace, size_t workspace_bytes,
    int *err_flags, int kernel, pkv_stream_t stream);

/*
 * pkv_write_decode_attention -- one decode step in one launch: pkv_write of
 * each sequence's new token followed by pkv_decode_attention over contexts
 * that already count it.
 * Definition: course page "P09 · Paged KV 写入 + decode attention（参考实现）",
 * section 在系统中的位置 -- each model-runner step first writes the new
 * tokens' K/V into the cache by slot_mapping, then attention reads the
 * history through block_tables; the result is that of the two calls above
 * made one after the other.
 *
 *   k, v          [B, num_kv_heads, head_dim]: the new token of sequence b
 *                 starts at element b * k_token_stride (resp. v_token_stride)
 *   slot_mapping  [B] int64: slot of sequence b's new token; negative = no
 *                 new token (padding), nothing written for b
 *   everything else as in pkv_decode_attention (k_cache, v_cache are
 *   written in place at the kept slots).
 * Precondition (the decode append): a kept slot_mapping[b] is the slot of
 * logical position context_lens[b] - 1 of sequence b,
 *   block_tables[b, (n-1) / bs] * bs + (n-1) % bs,   n = context_lens[b],
 * and no other sequence's context reads that slot.  The kernel checks the
 * first part and raises PKV_FLAG_APPEND_MISMATCH when it does not hold.
 * The launch that reads position n-1 takes the new token's K/V from k/v
 * directly, so it does not wait for its own cache write; one CTA per
 * (sequence, KV head) writes the cache row.  (On the wide-group kernel --
 * see pkv_decode_attention -- the row read at position n-1 is replaced in
 * shared memory by the new token's once the tile has landed; still one
 * launch.)  The
 * cache ends bit-identical to pkv_write's; the output is bit-identical to
 * pkv_write + pkv_decode_attention with the same partition size.
 * Additional requirements: k, v, k_cache, v_cache 16-byte aligned;
 * head_dim * element size a multiple of 16 bytes; k_token_stride and
 * v_token_stride >= num_kv_heads * head_dim and multiples of 16 bytes.
 * Errors: those of pkv_decode_attention; PKV_ERR_INVALID_ARG for a NULL
 * k, v or slot_mapping or a misaligned row.
 */
PKV_API pkv_status pkv_write_decode_attention(
    void *out, const void *q, const void *k, const void *v, int64_t k_token_stride,
    int64_t v_token_stride, const int64_t *slot_mapping, void *k_cache, void *v_cache,
    const int32_t *block_tables, const int32_t *context_lens, int B, int H, int num_kv_heads,
    int head_dim, int block_size, int max_blocks, int64_t num_blocks, float scale, pkv_dtype dt,
    int max_context_len, int partition_size, void *workspace, size_t workspace_bytes,
    int *err_flags, pkv_stream_t stream);

/*
 * pkv_prefill_attention -- paged causal prefill attention: several new query
 * tokens per sequence (varlen), each attending to the context up to itself.
 * Definition: the course page "P09 · Paged KV 写入 + decode attention（参考
 * 实现）" asks how the varlen prefill version is written (section 面试官追问)
 * without giving it; this library's reading is the multi-query form of its
 * decode (section 细节: the decode query is the newest token, already
 * written, and sees the whole context including itself):
 *   qlen = cu_seqlens_q[b+1] - cu_seqlens_q[b] queries of sequence b are the
 *   LAST qlen of its n = context_lens[b] tokens, all already written to the
 *   cache (pkv_write); query i (row cu_seqlens_q[b] + i) sits at position
 *   p = n - qlen + i and attends to tokens 0 .. p; head h uses KV head
 *   h // (H / KVH); fp32 scores times scale, fp32 softmax, output in q's
 *   dtype.  With qlen = 1 it is pkv_decode_attention.
 *
 *   out, q        [total_q, H, head_dim], total_q = cu_seqlens_q[B]
 *   cu_seqlens_q  [B + 1] int32, cu_seqlens_q[0] = 0, non-decreasing
 *   k_cache, v_cache, block_tables, context_lens: as in pkv_decode_attention
 *   max_q_len     host-side upper bound on qlen (sizes the grid; 0 = total_q);
 *                 a longer sequence raises PKV_FLAG_QUERY_OVER_HINT
 *   err_flags     device int or NULL (PKV_FLAG_QUERY_LEN,
 *                 PKV_FLAG_QUERY_OVER_HINT, PKV_FLAG_BLOCK_OUT_OF_RANGE,
 *                 PKV_FLAG_TIMEOUT)
 * Supported: bf16 / fp16, head_dim 64 or 128, block_size a multiple of 16,
 * q, out, caches 16-byte aligned (tensor-core kernel, tcgen05).  No
 * workspace.  Errors: PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA.
 * B == 0 or total_q == 0 enqueues nothing.
 */
PKV_API pkv_status pkv_prefill_attention(void *out, const void *q, const void *k_cache,
                                         const void *v_cache, const int32_t *block_tables,
                                         const int32_t *cu_seqlens_q, const int32_t *context_lens,
                                         int B, int64_t total_q, int H, int num_kv_heads,
                                         int head_dim, int block_size, int max_blocks,
                                         int64_t num_blocks, float scale, pkv_dtype dt,
                                         int max_q_len, int *err_flags, pkv_stream_t stream);

/*
 * The layout experiment: vLLM's packed cache layout, which the interview
 * note "PagedAttention kernel: paged KV cache 与 block table" describes in
 * section 深入原理 (K cache [num_blocks, num_kv_heads, head_size / x,
 * block_size, x] with x = 16 / element size so that loads are aligned
 * 16-byte vectors; V cache [num_blocks, num_kv_heads, head_size,
 * block_size]).  For 16-bit types x = 8:
 *   k_cache_x[blk][kvh][d / 8][off][d % 8],   v_cache_x[blk][kvh][d][off]
 * holding the same values as the token-major caches of pkv_write /
 * pkv_decode_attention.  Only block_size 16, bf16 / fp16.  The library's
 * main path keeps the token-major layout; these two calls exist to measure
 * the difference (one contiguous copy per (block, KV head) instead of
 * head_dim / 64 tiled boxes).
 *
 * pkv_write_xpacked -- pkv_write into the packed layout (same arguments and
 * errors; block_size must be 16, head_dim a multiple of 8, k and the
 * caches 16-byte aligned, token strides multiples of 8 elements).
 * pkv_decode_attention_xpacked -- pkv_decode_attention over packed caches
 * (same arguments, workspace and errors, out in device memory; head_dim 64,
 * 128 or 256; returns PKV_ERR_UNSUPPORTED for other shapes and for fp32).
 */
PKV_API pkv_status pkv_write_xpacked(void *k_cache_x, void *v_cache_x, const void *k, const void *v,
                                     const int64_t *slot_mapping, int64_t num_tokens,
                                     int64_t k_token_stride, int64_t v_token_stride,
                                     int64_t num_blocks, int block_size, int num_kv_heads,
                                     int head_dim, pkv_dtype dt, int *err_flags,
                                     pkv_stream_t stream);
PKV_API pkv_status pkv_decode_attention_xpacked(
    void *out, const void *q, const void *k_cache_x, const void *v_cache_x,
    const int32_t *block_tables, const int32_t *context_lens, int B, int H, int num_kv_heads,
    int head_dim, int block_size, int max_blocks, int64_t num_blocks, float scale, pkv_dtype dt,
    int max_context_len, int partition_size, void *workspace, size_t workspace_bytes,
    int *err_flags, pkv_stream_t stream);

/*
 * pkv_decode_plan -- the partition size and the partitions per sequence that
 * pkv_decode_attention would use for these arguments on a GPU with
 * num_sms SMs (host only, no CUDA call; for tests and tuning; on the
 * wide-group kernel with partition_size 0, the floor of its item size and
 * the most partitions a sequence can have).  Returns the
 * partition size in tokens (>= 16), or 0 for invalid sizes; *kernel is set to
 * 2 for the wide-group tensor-core kernel, 1 for the TMA + mma.sync
 * tensor-core kernel, 0 for the CUDA-core kernel.
 */
PKV_API int pkv_decode_plan(int B, int H, int num_kv_heads, int head_dim, int block_size,
                            int max_blocks, int max_context_len, int partition_size,
                            pkv_dtype dt, int num_sms, int *max_partitions, int *kernel);

/*
 * pkv_hbm_copy -- a plain streaming copy of `bytes` bytes from src to dst
 * (device pointers, 16-byte aligned, bytes a multiple of 16, the ranges
 * not overlapping), enqueued on `stream`.  It is the yardstick the other
 * kernels are measured against: the HBM bandwidth a copy reaches on this
 * GPU (2 * bytes of traffic per call), taken in the same run.  The pages
 * have no counterpart.  Errors: PKV_ERR_INVALID_ARG (alignment, size,
 * overlap, NULL), PKV_ERR_CUDA.  bytes == 0 enqueues nothing.
 */
PKV_API pkv_status pkv_hbm_copy(void *dst, const void *src, size_t bytes, pkv_stream_t stream);

/*
 * pkv_hbm_gather_read -- reads nchunks chunks of chunk_bytes bytes, chunk i
 * starting at base + chunk_index[i] * chunk_stride_bytes (device pointers;
 * base 16-byte aligned, chunk_bytes and chunk_stride_bytes multiples of 16;
 * every chunk inside the caller's buffer -- the indices are not checked),
 * and XORs the 16-byte words read into *sink (a device uint64; the XOR of
 * the two 64-bit halves of every word, folded in, so no read is dead).  The
 * yardstick for the decode kernels' access pattern: the bandwidth reads of
 * randomly placed whole cache blocks reach on this GPU (bytes read =
 * nchunks * chunk_bytes), taken in the same run.  The pages have no
 * counterpart.  Errors: PKV_ERR_INVALID_ARG, PKV_ERR_CUDA.  nchunks == 0 or
 * chunk_bytes == 0 enqueues nothing.
 */
PKV_API pkv_status pkv_hbm_gather_read(const void *base, const int32_t *chunk_index,
                                       int64_t nchunks, int64_t chunk_stride_bytes,
                                       int64_t chunk_bytes, unsigned long long *sink,
                                       pkv_stream_t stream);

/*
 * pkv_hbm_gather_read_pair -- the same reads over two buffers in one launch:
 * every listed chunk of base_a, then every listed chunk of base_b (both
 * 16-byte aligned, both holding every listed chunk), all folded into
 * *sink.  Bytes read = 2 * nchunks * chunk_bytes.  The decode reads a
 * batch's K and V blocks in one launch; so does this yardstick (two
 * launches of half the size each pay their own ramp and tail).  Errors:
 * PKV_ERR_INVALID_ARG (as pkv_hbm_gather_read, or base_b NULL), PKV_ERR_CUDA.
 */
PKV_API pkv_status pkv_hbm_gather_read_pair(const void *base_a, const void *base_b,
                                            const int32_t *chunk_index, int64_t nchunks,
                                            int64_t chunk_stride_bytes, int64_t chunk_bytes,
                                            unsigned long long *sink, pkv_stream_t stream);

/*
 * pkv_fp32_fma_peak -- the CUDA-core yardstick: `blocks` blocks of 256
 * threads, each thread running eight independent fp32 multiply-add chains
 * x <- x * a + b from x = 0 for `iters` steps (fmaf, or with paired != 0 the
 * two-lane fma.rn.f32x2 on four pairs): 2 * 8 * iters flops per thread.
 * Thread 0 of block i stores the sum of its chains in out[i] (device
 * float[blocks]); any other thread stores it only if it equals `never`, so
 * no chain is dead code (pass a value no sum reaches).  With a = b = 1 every
 * chain ends at exactly iters (iters < 2^24), which makes the result
 * checkable.  The fp32 rate the CUDA cores reach in the same run, against
 * which a decode's arithmetic (2 * G * D flops per key and per value row of
 * D elements) is set when choosing tensor cores for a group of G query
 * heads.  The pages have no counterpart.  Errors: PKV_ERR_INVALID_ARG
 * (out NULL or not 4-byte aligned, blocks < 1 or > 2^20, iters < 0),
 * PKV_ERR_CUDA.
 */
PKV_API pkv_status pkv_fp32_fma_peak(float *out, int blocks, int iters, float a, float b,
                                     float never, int paired, pkv_stream_t stream);

/*
 * pkv_copy_async -- enqueues one copy of `bytes` bytes from src to dst on
 * `stream`, between any two memories the GPU addresses (device memory,
 * pinned or pageable host memory; the runtime tells which from the
 * pointers).  It is how a serving loop built on this library moves a step's
 * staged inputs in and its output out around a prepared step call, one
 * call per copy, without a framework's tensor copy in between.  The ranges
 * must not overlap.  Pinned host memory gives an asynchronous copy;
 * pageable host memory is staged by the runtime and may return only once
 * the copy is done.  Errors: PKV_ERR_INVALID_ARG (dst or src NULL with
 * bytes > 0, overlapping ranges), PKV_ERR_CUDA (the runtime refused the
 * copy).  bytes == 0 enqueues nothing.
 */
PKV_API pkv_status pkv_copy_async(void *dst, const void *src, size_t bytes, pkv_stream_t stream);

/* A static, human-readable name for a status code. */
PKV_API const char *pkv_status_string(pkv_status status);

/* Version string of the library build. */
PKV_API const char *pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
