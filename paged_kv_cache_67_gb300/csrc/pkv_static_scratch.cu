// pkv_static_scratch.cu -- pkv_decode_attention_static: paged decode attention
// for callers that cannot allocate device memory.
//
// Some callers are not allowed to call cudaMalloc (or any allocating
// routine) when they run attention: an engine plugin whose execute step must
// not allocate, code that enqueues work while another component owns the
// device allocator, or a deployment whose device memory is fixed and
// accounted for when the process starts.  For them this entry point takes
// the split-KV scratch (partial results and merge counters) from a fixed
// array compiled into the library instead of a caller-provided workspace.
//
// The array below lives for as long as the library is loaded, on every GPU
// the library is used on.  Host code cannot use its name as a device
// address, so the first call on each device looks the address up with
// cudaGetSymbolAddress (with that device current) and keeps it.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = PKV_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_pkv_scratch[kStaticScratchBytes];

void *g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of g_pkv_scratch on the current device (looked up once).
pkv_status scratch_address(void **addr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pkv_scratch) != cudaSuccess || p == nullptr)
      return PKV_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" PKV_API pkv_status pkv_decode_attention_static(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, const int32_t *context_lens, int B, int H, int num_kv_heads,
    int head_dim, int block_size, int max_blocks, int64_t num_blocks, float scale, pkv_dtype dt,
    int max_context_len, int partition_size, int *err_flags, pkv_stream_t stream) {
  if (B < 0 || H <= 0 || num_kv_heads <= 0 || H % num_kv_heads != 0 || head_dim <= 0 ||
      block_size <= 0 || max_blocks < 0 || max_context_len < 0 || partition_size < 0 ||
      partition_size % 16 != 0)
    return PKV_ERR_INVALID_ARG;
  if (B == 0) return PKV_OK;
  void *scratch = nullptr;
  pkv_status st = scratch_address(&scratch);
  if (st != PKV_OK) return st;
  int dev = 0, sms = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return PKV_ERR_CUDA;
  // The same plan pkv_decode_attention will make: how much scratch it needs.
  const void *ptrs[4] = {out, q, k_cache, v_cache};
  bool aligned16 = true;
  for (const void *p : ptrs) aligned16 = aligned16 && (reinterpret_cast<uintptr_t>(p) % 16 == 0);
  pkv::DecodePlan plan;
  if (!pkv::make_plan(B, H, num_kv_heads, head_dim, block_size, max_blocks, max_context_len,
                      partition_size, dt, sms, (size_t)optin, aligned16, &plan))
    return PKV_ERR_INVALID_ARG;
  const size_t need = pkv::workspace_bytes_for(B, H, head_dim, plan.max_parts);
  if (need > kStaticScratchBytes) return PKV_ERR_WORKSPACE;  // beyond the fixed maximum
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The merge counters must start at zero; the array keeps whatever the
  // previous call left, so clear them on this call's stream.
  if (cudaMemsetAsync(scratch, 0, pkv::workspace_counter_bytes(B, H), s) != cudaSuccess)
    return PKV_ERR_CUDA;
  return pkv_decode_attention(out, q, k_cache, v_cache, block_tables, context_lens, B, H,
                              num_kv_heads, head_dim, block_size, max_blocks, num_blocks, scale, dt,
                              max_context_len, partition_size, scratch, kStaticScratchBytes,
                              err_flags, stream);
}
