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
// cudaGetSymbolAddress (with that device current) and keeps it, together
// with the identity of the device's context: after cudaDeviceReset the
// context is new, the module is loaded again and the address is looked up
// again.  Devices past the cache's range look it up on every call.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = PKV_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_pkv_scratch[kStaticScratchBytes];

struct ScratchEntry {
  unsigned long long ctx_id;   // the context the address belongs to (0: none yet)
  void *addr;
};
ScratchEntry g_scratch[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

// Identity of the current context (0 if it cannot be read: then the address
// is looked up on every call).
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static bool tried = false;
  if (!tried) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
    tried = true;
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_pkv_scratch in the current device's context.
pkv_status scratch_address(void **addr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return PKV_ERR_CUDA;
  // the runtime makes the device's context current (and loads the module)
  // when the symbol is looked up; the context's identity is read after that
  void *p = nullptr;
  const unsigned long long id = dev < kMaxDevices ? current_context_id() : 0;
  if (dev < kMaxDevices && id != 0 && g_scratch[dev].ctx_id == id) {
    *addr = g_scratch[dev].addr;
    return PKV_OK;
  }
  if (cudaGetSymbolAddress(&p, g_pkv_scratch) != cudaSuccess || p == nullptr) return PKV_ERR_CUDA;
  if (dev < kMaxDevices) {
    const unsigned long long now = current_context_id();
    g_scratch[dev].ctx_id = now;
    g_scratch[dev].addr = p;
  }
  *addr = p;
  return PKV_OK;
}

}  // namespace

extern "C" PKV_API pkv_status pkv_decode_attention_static(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, const int32_t *context_lens, int B, int H, int num_kv_heads,
    int head_dim, int block_size, int max_blocks, int64_t num_blocks, float scale, pkv_dtype dt,
    int max_context_len, int partition_size, int *err_flags, pkv_stream_t stream) {
  // Every argument check of pkv_decode_attention first, so that a rejected
  // call enqueues nothing (in particular no clearing of the shared array,
  // which another call may still be using on another stream).
  pkv::DecodePlan plan;
  int sms = 0;
  bool empty = false;
  pkv_status st = pkv::decode_check_and_plan(out, q, k_cache, v_cache, block_tables, context_lens,
                                             B, H, num_kv_heads, head_dim, block_size, max_blocks,
                                             num_blocks, dt, max_context_len, partition_size,
                                             false, -1, &plan, &sms, &empty);
  if (st != PKV_OK || empty) return st;
  // The scratch this plan needs (the same plan pkv_decode_attention makes).
  const size_t need = pkv::workspace_bytes_for(B, H, head_dim, plan.max_parts);
  if (need > kStaticScratchBytes) return PKV_ERR_WORKSPACE;  // beyond the fixed maximum
  void *scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != PKV_OK) return st;
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
