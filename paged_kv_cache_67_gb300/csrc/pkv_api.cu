// pkv_api.cu -- the C ABI declared in include/pkv.h: host-side argument
// checks, the decode plan (kernel choice, partition size, workspace
// layout) and the launches.  Nothing here allocates device memory.
#include <math.h>

#include <algorithm>
#include <string.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

size_t simt_smem_bytes(int D, int GH);
size_t tc_smem_bytes(int D, int stages);


static int round_up(long long x, int m) { return (int)(((x + m - 1) / m) * m); }
static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool tc_eligible(pkv_dtype dt, int D, int bs) {
  return (dt == PKV_BF16 || dt == PKV_F16) && (D == 64 || D == 128 || D == 192 || D == 256) &&
         bs % 16 == 0;
}

// Context capacity the grid must cover: the host hint, else the table width.
static long long context_cap(int bs, int max_blocks, int max_context_len) {
  const long long table = (long long)max_blocks * bs;
  long long cap = max_context_len > 0 ? (long long)max_context_len : table;
  if (cap > table) cap = table;
  return cap < 1 ? 1 : cap;
}

// Smallest partition the automatic choice uses for this capacity: at least
// 64 tokens and at most kMaxAutoParts partitions per sequence.
static int auto_partition_floor(long long cap) {
  const int p = round_up((cap + kMaxAutoParts - 1) / kMaxAutoParts, 16);
  return p < 64 ? 64 : p;
}

// Partial-result slots per (sequence, head) the workspace holds: ceil(cap / P)
// for an explicit partition size P; for the automatic choice the partition
// is never below the floor, so ceil(cap / floor) <= kMaxAutoParts.
static int workspace_parts(long long cap, int partition_size) {
  const long long P = partition_size > 0 ? partition_size : auto_partition_floor(cap);
  const long long parts = (cap + P - 1) / P;
  return parts > 0x7fffffffLL ? 0x7fffffff : (int)parts;
}

static int tc_stages(int D) { return D <= 64 ? 6 : (D <= 128 ? 3 : (D <= 192 ? 2 : 3)); }

bool make_plan(int B, int H, int KVH, int D, int bs, int max_blocks, int max_context_len,
               int partition_size, pkv_dtype dt, int num_sms, size_t smem_optin, bool aligned16,
               DecodePlan *plan, bool allow_wide, int force_kernel) {
  if (B < 0 || H <= 0 || KVH <= 0 || H % KVH != 0 || D <= 0 || D > 512 || bs <= 0 ||
      max_blocks < 0 || partition_size < 0 || partition_size % 16 != 0 || max_context_len < 0)
    return false;
  if (dt != PKV_F32 && dt != PKV_BF16 && dt != PKV_F16) return false;
  const int G = H / KVH;
  DecodePlan p;
  memset(&p, 0, sizeof p);
  p.kernel = (tc_eligible(dt, D, bs) && aligned16 && force_kernel != 0) ? 1 : 0;
  p.heads_per_cta = p.kernel ? kTcHeads : (D <= 256 ? 4 : 2);
  p.gchunks = (G + p.heads_per_cta - 1) / p.heads_per_cta;
  p.threads = 128;
  const long long cap = context_cap(bs, max_blocks, max_context_len);
  if (partition_size > 0) {
    p.P = partition_size;
  } else {
    // About four CTAs per resident CTA slot (two for the tensor-core kernel
    // when the units alone do not fill the slots: fewer, longer CTAs pay
    // the per-CTA start-up and drain fewer times -- on the long-context
    // batch, three seeds, 0.945 of the copy peak at two against 0.916 at
    // four, 0.878-0.912 at 2.5-6): split each (sequence, head group) unit
    // into enough partitions of the capacity, but never below 1024 tokens
    // (each CTA pays a fixed start-up and merge cost) nor below the floor
    // that bounds the partitions per sequence.  With enough units to fill
    // the GPU nothing is split.
    const long long units = (long long)B * KVH * p.gchunks;
    const int per_sm = p.kernel ? (D <= 128 ? 2 : 1) : 4;
    const long long slots = (long long)(num_sms > 0 ? num_sms : 1) * per_sm;
    const long long per_slot = (p.kernel == 1 && units < slots) ? 2 : 4;
    long long parts = units > 0 ? (per_slot * slots + units - 1) / units : 1;
    if (parts < 1) parts = 1;
    int P = round_up((cap + parts - 1) / parts, 16);
    const int floor_p = auto_partition_floor(cap);
    if (P < floor_p) P = floor_p;
    const int min_p = cap < 1024 ? round_up(cap, 16) : 1024;
    if (P < min_p) P = min_p;
    p.P = P;
  }
  const long long mp = (cap + p.P - 1) / p.P;
  if (mp > 0x7fffffffLL) return false;
  p.max_parts = (int)(mp < 1 ? 1 : mp);
  p.stages = p.kernel ? tc_stages(D) : 0;
  p.smem_bytes = p.kernel ? tc_smem_bytes(D, p.stages) : simt_smem_bytes(D, p.heads_per_cta);
  // Launch order of the tensor-core kernel: with fewer units than resident
  // CTA slots every wave holds several partitions of each unit, and
  // launching partitions in order puts the short and empty last ones at the
  // end (long contexts: 64 units on 304 slots, 126.3 against 130.5 us);
  // with more units a unit's partitions launch together (the 8B-shaped
  // batch, 512 units: 114.8 against 118.4 us partition-major).
  {
    const long long units = (long long)B * KVH * p.gchunks;
    const long long slots = (long long)(num_sms > 0 ? num_sms : 1) * (D <= 128 ? 2 : 1);
    p.part_major = p.kernel == 1 && units < slots;
  }
  // Groups of exactly 16 query heads with D = 128 or 256 (MQA-like): the
  // persistent kernel with tokens as the product's M.  The plan's partition
  // is 1024 tokens (never below the automatic floor that keeps the
  // partitions within the workspace); with it the kernel sizes its work
  // items from the batch's lengths (about 1.2 CTA shares of tiles, never
  // smaller than the plan's partition).
  if (allow_wide && force_kernel != 1 && p.kernel == 1 && G == 16 && (D == 128 || D == 256) &&
      wide_smem_bytes(D) <= (smem_optin > 0 ? smem_optin : kDefaultSmemOptin)) {
    p.kernel = 2;
    p.heads_per_cta = 16;
    p.gchunks = 1;
    if (partition_size == 0) {
      int P = 1024;
      const int floor_p = auto_partition_floor(cap);
      if (P < floor_p) P = floor_p;
      if (P > cap) P = round_up(cap, 16);
      p.P = P;
      p.max_parts = (int)((cap + P - 1) / P);
    }
    p.stages = 0;
    p.smem_bytes = wide_smem_bytes(D);
  }
  // a kernel named by the caller (tests and tuning) that cannot run these
  // sizes: no plan
  if (force_kernel >= 0 && p.kernel != force_kernel) return false;
  *plan = p;
  return true;
}

size_t workspace_counter_bytes(int B, int H) { return align256((size_t)B * H * sizeof(int)); }

size_t workspace_bytes_for(int B, int H, int D, int max_parts) {
  const size_t rows = (size_t)B * H;
  size_t bytes = workspace_counter_bytes(B, H);
  if (max_parts > 1)
    bytes += 2 * align256(rows * max_parts * sizeof(float)) +
             rows * max_parts * (size_t)D * sizeof(float);
  return bytes;
}

// SM count and opt-in shared memory per block of the current device (cached).
static bool device_caps(int *sms, size_t *smem_optin) {
  static int counts[64] = {0};
  static int optin[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return false;
  int n = dev < 64 ? counts[dev] : 0, o = dev < 64 ? optin[dev] : 0;
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&o, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return false;
    if (dev < 64) {
      counts[dev] = n;
      optin[dev] = o;
    }
  }
  *sms = n;
  *smem_optin = (size_t)o;
  return n > 0;
}

static int elem_size(pkv_dtype dt) { return dt == PKV_F32 ? 4 : 2; }

}  // namespace pkv

using namespace pkv;

extern "C" {

PKV_API pkv_status pkv_write(void *k_cache, void *v_cache, const void *k, const void *v,
                             const int64_t *slot_mapping, int64_t num_tokens,
                             int64_t k_token_stride, int64_t v_token_stride, int64_t num_blocks,
                             int block_size, int num_kv_heads, int head_dim, pkv_dtype dt,
                             int *err_flags, pkv_stream_t stream) {
  if (num_tokens < 0 || num_blocks < 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return PKV_ERR_INVALID_ARG;
  if (dt != PKV_F32 && dt != PKV_BF16 && dt != PKV_F16) return PKV_ERR_INVALID_ARG;
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  if (k_token_stride < row || v_token_stride < row) return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!k_cache || !v_cache || !k || !v || !slot_mapping) return PKV_ERR_INVALID_ARG;
  return launch_write(k_cache, v_cache, k, v, slot_mapping, num_tokens, k_token_stride,
                      v_token_stride, num_blocks, block_size, num_kv_heads, head_dim,
                      elem_size(dt), err_flags, reinterpret_cast<cudaStream_t>(stream));
}

PKV_API size_t pkv_decode_workspace_size(int B, int H, int num_kv_heads, int head_dim,
                                         int block_size, int max_blocks, int max_context_len,
                                         int partition_size) {
  if (B < 0 || H <= 0 || num_kv_heads <= 0 || H % num_kv_heads != 0 || head_dim <= 0 ||
      head_dim > 512 || block_size <= 0 || max_blocks < 0 || max_context_len < 0 ||
      partition_size < 0 || partition_size % 16 != 0)
    return 0;
  const long long cap = context_cap(block_size, max_blocks, max_context_len);
  const int parts = workspace_parts(cap, partition_size);
  if ((long long)B * H * parts > 0x7fffffffLL) return 0;
  return workspace_bytes_for(B, H, head_dim, parts);
}

PKV_API int pkv_decode_plan(int B, int H, int num_kv_heads, int head_dim, int block_size,
                            int max_blocks, int max_context_len, int partition_size, pkv_dtype dt,
                            int num_sms, int *max_partitions, int *kernel) {
  DecodePlan p;
  if (!make_plan(B, H, num_kv_heads, head_dim, block_size, max_blocks, max_context_len,
                 partition_size, dt, num_sms, kDefaultSmemOptin, true, &p))
    return 0;
  if (max_partitions) *max_partitions = p.max_parts;
  if (kernel) *kernel = p.kernel;
  return p.P;
}

}  // extern "C"

namespace pkv {

// New tokens of a fused write + decode launch (see pkv_write_decode_attention).
struct AppendIn {
  const void *k, *v;
  int64_t k_stride, v_stride;
  const int64_t *slots;
};

// Every host-side check of a decode call that needs no workspace, and the
// plan.  *empty is set when B == 0 (nothing to enqueue).  Used by the
// workspace entry points and by pkv_decode_attention_static, so that a call
// rejected here has enqueued nothing.
pkv_status decode_check_and_plan(const void *out, const void *q, const void *k_cache,
                                 const void *v_cache, const int32_t *block_tables,
                                 const int32_t *context_lens, int B, int H, int num_kv_heads,
                                 int head_dim, int block_size, int max_blocks, int64_t num_blocks,
                                 pkv_dtype dt, int max_context_len, int partition_size,
                                 bool xpacked, int force_kernel, DecodePlan *plan, int *num_sms,
                                 bool *empty) {
  *empty = false;
  if (B < 0 || B > 65535 || H <= 0 || H > 65535 || num_kv_heads <= 0 || H % num_kv_heads != 0 ||
      head_dim <= 0 || block_size <= 0 || max_blocks < 0 || num_blocks < 0 ||
      num_blocks > 0x7fffffffLL || max_context_len < 0 || partition_size < 0 ||
      partition_size % 16 != 0 || force_kernel < -1 || force_kernel > 2)
    return PKV_ERR_INVALID_ARG;
  if (dt != PKV_F32 && dt != PKV_BF16 && dt != PKV_F16) return PKV_ERR_INVALID_ARG;
  if (head_dim > 512) return PKV_ERR_UNSUPPORTED;
  if (B == 0) {
    *empty = true;
    return PKV_OK;
  }
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
    return PKV_ERR_INVALID_ARG;
  const uintptr_t el = (uintptr_t)elem_size(dt);
  const void *ptrs[4] = {out, q, k_cache, v_cache};
  bool aligned16 = true;
  for (const void *p : ptrs) {
    if (reinterpret_cast<uintptr_t>(p) % el) return PKV_ERR_INVALID_ARG;
    aligned16 = aligned16 && (reinterpret_cast<uintptr_t>(p) % 16 == 0);
  }
  if (reinterpret_cast<uintptr_t>(block_tables) % 4 || reinterpret_cast<uintptr_t>(context_lens) % 4)
    return PKV_ERR_INVALID_ARG;

  int sms = 0;
  size_t smem_optin = 0;
  if (!device_caps(&sms, &smem_optin)) return PKV_ERR_CUDA;
  if (!make_plan(B, H, num_kv_heads, head_dim, block_size, max_blocks, max_context_len,
                 partition_size, dt, sms, smem_optin, aligned16, plan, !xpacked, force_kernel)) {
    // valid sizes that the named kernel does not handle
    DecodePlan any;
    if (force_kernel >= 0 && make_plan(B, H, num_kv_heads, head_dim, block_size, max_blocks,
                                       max_context_len, partition_size, dt, sms, smem_optin,
                                       aligned16, &any, !xpacked))
      return PKV_ERR_UNSUPPORTED;
    return PKV_ERR_INVALID_ARG;
  }
  if ((long long)num_kv_heads * plan->gchunks > 65535) return PKV_ERR_UNSUPPORTED;
  if (xpacked && (plan->kernel != 1 || block_size != 16 || head_dim == 192))
    return PKV_ERR_UNSUPPORTED;
  *num_sms = sms;
  return PKV_OK;
}

// pkv_decode_attention, and with `app` the fused append of one new token per
// sequence.
static pkv_status decode_entry(void *out, const void *q, const void *k_cache, const void *v_cache,
                               const int32_t *block_tables, const int32_t *context_lens, int B,
                               int H, int num_kv_heads, int head_dim, int block_size,
                               int max_blocks, int64_t num_blocks, float scale, pkv_dtype dt,
                               int max_context_len, int partition_size, void *workspace,
                               size_t workspace_bytes, int *err_flags, pkv_stream_t stream,
                               const AppendIn *app, bool xpacked = false, int force_kernel = -1) {
  DecodePlan plan;
  int sms = 0;
  bool empty = false;
  const pkv_status chk = decode_check_and_plan(
      out, q, k_cache, v_cache, block_tables, context_lens, B, H, num_kv_heads, head_dim,
      block_size, max_blocks, num_blocks, dt, max_context_len, partition_size, xpacked,
      force_kernel, &plan, &sms, &empty);
  if (chk != PKV_OK || empty) return chk;

  DecodeArgs a;
  memset(&a, 0, sizeof a);
  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.tables = block_tables;
  a.lens = context_lens;
  a.err = err_flags;
  a.num_blocks = num_blocks;
  a.B = B;
  a.H = H;
  a.KVH = num_kv_heads;
  a.D = head_dim;
  a.G = H / num_kv_heads;
  a.bs = block_size;
  a.max_blocks = max_blocks;
  a.heads_per_cta = plan.heads_per_cta;
  a.gchunks = plan.gchunks;
  a.P = plan.P;
  a.max_parts = plan.max_parts;
  a.stages = plan.stages;
  a.part_major = plan.part_major;
  a.scale_log2 = scale * kLog2e;
  if (app) {
    a.new_slots = app->slots;
    a.new_k = app->k;
    a.new_v = app->v;
    a.new_k_stride = app->k_stride;
    a.new_v_stride = app->v_stride;
  }

  const size_t need = workspace_bytes_for(B, H, head_dim, plan.max_parts);
  if (!workspace || workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 256)
    return PKV_ERR_WORKSPACE;
  {
    const size_t rows = (size_t)B * H;
    char *ws = static_cast<char *>(workspace);
    a.ws_cnt = reinterpret_cast<int *>(ws);
    ws += align256(rows * sizeof(int));
    if (plan.max_parts > 1) {
      a.ws_m = reinterpret_cast<float *>(ws);
      ws += align256(rows * plan.max_parts * sizeof(float));
      a.ws_l = reinterpret_cast<float *>(ws);
      ws += align256(rows * plan.max_parts * sizeof(float));
      a.ws_o = reinterpret_cast<float *>(ws);
    }
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (xpacked) return launch_decode_xpacked(a, plan, dt, s);
  if (plan.kernel == 2) return launch_decode_wide(a, dt, sms, partition_size == 0, s);
  return plan.kernel ? launch_decode_tc(a, plan, dt, s) : launch_decode_simt(a, plan, dt, s);
}

}  // namespace pkv

extern "C" {

PKV_API pkv_status pkv_decode_attention(void *out, const void *q, const void *k_cache,
                                        const void *v_cache, const int32_t *block_tables,
                                        const int32_t *context_lens, int B, int H,
                                        int num_kv_heads, int head_dim, int block_size,
                                        int max_blocks, int64_t num_blocks, float scale,
                                        pkv_dtype dt, int max_context_len, int partition_size,
                                        void *workspace, size_t workspace_bytes, int *err_flags,
                                        pkv_stream_t stream) {
  return decode_entry(out, q, k_cache, v_cache, block_tables, context_lens, B, H, num_kv_heads,
                      head_dim, block_size, max_blocks, num_blocks, scale, dt, max_context_len,
                      partition_size, workspace, workspace_bytes, err_flags, stream, nullptr);
}

PKV_API pkv_status pkv_decode_attention_with_kernel(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, const int32_t *context_lens, int B, int H, int num_kv_heads,
    int head_dim, int block_size, int max_blocks, int64_t num_blocks, float scale, pkv_dtype dt,
    int max_context_len, int partition_size, void *workspace, size_t workspace_bytes,
    int *err_flags, int kernel, pkv_stream_t stream) {
  return decode_entry(out, q, k_cache, v_cache, block_tables, context_lens, B, H, num_kv_heads,
                      head_dim, block_size, max_blocks, num_blocks, scale, dt, max_context_len,
                      partition_size, workspace, workspace_bytes, err_flags, stream, nullptr, false,
                      kernel);
}

PKV_API pkv_status pkv_write_decode_attention(
    void *out, const void *q, const void *k, const void *v, int64_t k_token_stride,
    int64_t v_token_stride, const int64_t *slot_mapping, void *k_cache, void *v_cache,
    const int32_t *block_tables, const int32_t *context_lens, int B, int H, int num_kv_heads,
    int head_dim, int block_size, int max_blocks, int64_t num_blocks, float scale, pkv_dtype dt,
    int max_context_len, int partition_size, void *workspace, size_t workspace_bytes,
    int *err_flags, pkv_stream_t stream) {
  if (dt != PKV_F32 && dt != PKV_BF16 && dt != PKV_F16) return PKV_ERR_INVALID_ARG;
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  const int64_t el = elem_size(dt);
  if (num_kv_heads <= 0 || head_dim <= 0 || k_token_stride < row || v_token_stride < row ||
      (k_token_stride * el) % 16 || (v_token_stride * el) % 16 || (head_dim * el) % 16)
    return PKV_ERR_INVALID_ARG;
  // the new rows are copied as 16-byte vectors: inputs and cache rows aligned
  if (B > 0 && (!k || !v || !slot_mapping || reinterpret_cast<uintptr_t>(k) % 16 ||
                reinterpret_cast<uintptr_t>(v) % 16 || reinterpret_cast<uintptr_t>(slot_mapping) % 8 ||
                reinterpret_cast<uintptr_t>(k_cache) % 16 || reinterpret_cast<uintptr_t>(v_cache) % 16))
    return PKV_ERR_INVALID_ARG;
  const AppendIn app{k, v, k_token_stride, v_token_stride, slot_mapping};
  return decode_entry(out, q, k_cache, v_cache, block_tables, context_lens, B, H, num_kv_heads,
                      head_dim, block_size, max_blocks, num_blocks, scale, dt, max_context_len,
                      partition_size, workspace, workspace_bytes, err_flags, stream, &app);
}

PKV_API pkv_status pkv_write_xpacked(void *k_cache_x, void *v_cache_x, const void *k, const void *v,
                                     const int64_t *slot_mapping, int64_t num_tokens,
                                     int64_t k_token_stride, int64_t v_token_stride,
                                     int64_t num_blocks, int block_size, int num_kv_heads,
                                     int head_dim, pkv_dtype dt, int *err_flags,
                                     pkv_stream_t stream) {
  if (num_tokens < 0 || num_blocks < 0 || num_kv_heads <= 0 || head_dim <= 0)
    return PKV_ERR_INVALID_ARG;
  if (dt != PKV_F32 && dt != PKV_BF16 && dt != PKV_F16) return PKV_ERR_INVALID_ARG;
  if (dt == PKV_F32 || block_size != 16 || head_dim % 8 != 0) return PKV_ERR_UNSUPPORTED;
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  if (k_token_stride < row || v_token_stride < row || k_token_stride % 8 || v_token_stride % 8)
    return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!k_cache_x || !v_cache_x || !k || !v || !slot_mapping ||
      reinterpret_cast<uintptr_t>(k) % 16 || reinterpret_cast<uintptr_t>(k_cache_x) % 16)
    return PKV_ERR_INVALID_ARG;
  return launch_write_xpacked(k_cache_x, v_cache_x, k, v, slot_mapping, num_tokens, k_token_stride,
                              v_token_stride, num_blocks, num_kv_heads, head_dim, dt, err_flags,
                              reinterpret_cast<cudaStream_t>(stream));
}

PKV_API pkv_status pkv_decode_attention_xpacked(
    void *out, const void *q, const void *k_cache_x, const void *v_cache_x,
    const int32_t *block_tables, const int32_t *context_lens, int B, int H, int num_kv_heads,
    int head_dim, int block_size, int max_blocks, int64_t num_blocks, float scale, pkv_dtype dt,
    int max_context_len, int partition_size, void *workspace, size_t workspace_bytes,
    int *err_flags, pkv_stream_t stream) {
  return decode_entry(out, q, k_cache_x, v_cache_x, block_tables, context_lens, B, H, num_kv_heads,
                      head_dim, block_size, max_blocks, num_blocks, scale, dt, max_context_len,
                      partition_size, workspace, workspace_bytes, err_flags, stream, nullptr, true);
}

PKV_API pkv_status pkv_prefill_attention(void *out, const void *q, const void *k_cache,
                                         const void *v_cache, const int32_t *block_tables,
                                         const int32_t *cu_seqlens_q, const int32_t *context_lens,
                                         int B, int64_t total_q, int H, int num_kv_heads,
                                         int head_dim, int block_size, int max_blocks,
                                         int64_t num_blocks, float scale, pkv_dtype dt,
                                         int max_q_len, int *err_flags, pkv_stream_t stream) {
  if (B < 0 || B > 65535 || total_q < 0 || total_q > 0x7fffffffLL || H <= 0 || H > 65535 ||
      num_kv_heads <= 0 || H % num_kv_heads != 0 || head_dim <= 0 || block_size <= 0 ||
      max_blocks < 0 || num_blocks < 0 || num_blocks > 0x7fffffffLL || max_q_len < 0)
    return PKV_ERR_INVALID_ARG;
  if (dt != PKV_F32 && dt != PKV_BF16 && dt != PKV_F16) return PKV_ERR_INVALID_ARG;
  if (dt == PKV_F32 || (head_dim != 64 && head_dim != 128) || block_size % 16 != 0)
    return PKV_ERR_UNSUPPORTED;
  if (B == 0 || total_q == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !cu_seqlens_q || !context_lens)
    return PKV_ERR_INVALID_ARG;
  const void *ptrs[4] = {out, q, k_cache, v_cache};
  for (const void *p : ptrs)
    if (reinterpret_cast<uintptr_t>(p) % 16) return PKV_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(block_tables) % 4 || reinterpret_cast<uintptr_t>(cu_seqlens_q) % 4 ||
      reinterpret_cast<uintptr_t>(context_lens) % 4)
    return PKV_ERR_INVALID_ARG;
  const long long mq = max_q_len > 0 ? max_q_len : total_q;
  const long long q_tiles = (mq + 255) / 256;  // 256 queries (two 128-row tiles) per work item
  // (sequence, tile) pairs: sum ceil(qlen / 256) <= total_q / 256 + B; work
  // items are (pair, head) and are counted in 32 bits
  const long long pairs = std::min<long long>((total_q + 255) / 256 + B, (long long)B * q_tiles);
  if (q_tiles > 65535 || pairs * H > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
  return launch_prefill_tc(out, q, k_cache, v_cache, block_tables, cu_seqlens_q, context_lens, B,
                           total_q, H, num_kv_heads, head_dim, block_size, max_blocks, num_blocks,
                           scale, dt, (int)q_tiles, (int)pairs, err_flags,
                           reinterpret_cast<cudaStream_t>(stream));
}

PKV_API pkv_status pkv_copy_async(void *dst, const void *src, size_t bytes, pkv_stream_t stream) {
  if (bytes == 0) return PKV_OK;
  if (!dst || !src) return PKV_ERR_INVALID_ARG;
  const uintptr_t d0 = reinterpret_cast<uintptr_t>(dst), s0 = reinterpret_cast<uintptr_t>(src);
  if (d0 < s0 + bytes && s0 < d0 + bytes) return PKV_ERR_INVALID_ARG;  // overlapping ranges
  const cudaError_t e =
      cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

PKV_API const char *pkv_status_string(pkv_status status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_WORKSPACE: return "workspace missing or too small";
    case PKV_ERR_OUT_OF_BLOCKS: return "not enough free cache blocks";
  }
  return "unknown status";
}

PKV_API const char *pkv_version(void) { return "pkv 0.1 (sm_103a)"; }

}  // extern "C"
