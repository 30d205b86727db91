// pkv_write.cu -- write_kv / reshape_and_cache on the GPU.
//
// Definition (course page "P09 · Paged KV 写入 + decode attention（参考实现）",
// section 题面速览 and the write_kv shape trace): for every new token i with
// slot = slot_mapping[i] >= 0, k_cache[slot // bs, slot % bs] = k[i] and the
// same for v; negative slots are padding and are skipped; in place.
//
// With the contiguous [num_blocks, bs, KVH, D] layout the destination row
// cache[slot // bs, slot % bs] is row `slot` of the flattened cache (the
// page's "储物柜墙" identity), so the kernel addresses it as slot * row.
//
// One warp per token: the slot is read once (a broadcast load), the warp
// leaves at once for a padding token, and otherwise its lanes move the row
// in VEC-byte pieces (16 bytes when sizes and pointers allow), with up to
// four k and four v loads in flight per lane before the stores.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

template <int VEC>
struct VecType;
template <> struct VecType<16> { using type = uint4; };
template <> struct VecType<8> { using type = uint2; };
template <> struct VecType<4> { using type = uint32_t; };
template <> struct VecType<2> { using type = uint16_t; };

struct WriteArgs {
  char *kc;
  char *vc;
  const char *k;
  const char *v;
  const int64_t *slots;
  int64_t T;
  int64_t capacity;      // num_blocks * block_size
  int64_t row_vecs;      // vectors per token row
  int64_t k_stride;      // vectors between consecutive tokens of k
  int64_t v_stride;
  int *err;
};

constexpr int kWriteWarps = 4;

template <int VEC>
__global__ void __launch_bounds__(32 * kWriteWarps) pkv_write_kernel(const WriteArgs a) {
  using V = typename VecType<VEC>::type;
  // a kernel launched after this one as its programmatic dependent may start
  // now; it waits for this grid's rows before it reads them (no effect on a
  // plain launch after)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * kWriteWarps + (threadIdx.x >> 5);
  if (t >= a.T) return;
  const int64_t slot = __ldg(a.slots + t);
  if (slot < 0) return;                       // padding token: not written
  if (slot >= a.capacity) {                   // past the pool: report, skip
    if (lane == 0) raise_flag(a.err, PKV_FLAG_SLOT_OUT_OF_RANGE);
    return;
  }
  const V *ks = reinterpret_cast<const V *>(a.k) + t * a.k_stride;
  const V *vs = reinterpret_cast<const V *>(a.v) + t * a.v_stride;
  V *kd = reinterpret_cast<V *>(a.kc) + slot * a.row_vecs;
  V *vd = reinterpret_cast<V *>(a.vc) + slot * a.row_vecs;
  const int64_t n = a.row_vecs;
  int64_t c = lane;
  for (; c + 96 < n; c += 128) {
    V k0 = __ldg(ks + c), k1 = __ldg(ks + c + 32), k2 = __ldg(ks + c + 64), k3 = __ldg(ks + c + 96);
    V v0 = __ldg(vs + c), v1 = __ldg(vs + c + 32), v2 = __ldg(vs + c + 64), v3 = __ldg(vs + c + 96);
    kd[c] = k0; kd[c + 32] = k1; kd[c + 64] = k2; kd[c + 96] = k3;
    vd[c] = v0; vd[c + 32] = v1; vd[c + 64] = v2; vd[c + 96] = v3;
  }
  for (; c < n; c += 32) {
    V k0 = __ldg(ks + c), v0 = __ldg(vs + c);
    kd[c] = k0;
    vd[c] = v0;
  }
}

static int pick_vec(int64_t row_bytes, int64_t ks_bytes, int64_t vs_bytes, const void *const *ptrs,
                    int nptrs, int elem) {
  for (int vec = 16; vec >= 2; vec >>= 1) {
    if (vec < elem) break;
    if (row_bytes % vec || ks_bytes % vec || vs_bytes % vec) continue;
    bool ok = true;
    for (int i = 0; i < nptrs; ++i) ok = ok && (reinterpret_cast<uintptr_t>(ptrs[i]) % vec == 0);
    if (ok) return vec;
  }
  return 0;
}

pkv_status launch_write(void *k_cache, void *v_cache, const void *k, const void *v,
                        const int64_t *slot_mapping, int64_t T, int64_t k_stride, int64_t v_stride,
                        int64_t num_blocks, int bs, int KVH, int D, int elem, int *err,
                        cudaStream_t stream) {
  const int64_t row_bytes = (int64_t)KVH * D * elem;
  const void *ptrs[4] = {k_cache, v_cache, k, v};
  const int vec = pick_vec(row_bytes, k_stride * elem, v_stride * elem, ptrs, 4, elem);
  if (vec == 0) return PKV_ERR_INVALID_ARG;  // element-misaligned pointer
  WriteArgs a;
  a.kc = static_cast<char *>(k_cache);
  a.vc = static_cast<char *>(v_cache);
  a.k = static_cast<const char *>(k);
  a.v = static_cast<const char *>(v);
  a.slots = slot_mapping;
  a.T = T;
  a.capacity = num_blocks * (int64_t)bs;
  a.row_vecs = row_bytes / vec;
  a.k_stride = k_stride * elem / vec;
  a.v_stride = v_stride * elem / vec;
  a.err = err;
  const int64_t blocks = (T + kWriteWarps - 1) / kWriteWarps;
  if (blocks > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
  dim3 grid((unsigned)blocks), block(32 * kWriteWarps);
  switch (vec) {
    case 16: pkv_write_kernel<16><<<grid, block, 0, stream>>>(a); break;
    case 8: pkv_write_kernel<8><<<grid, block, 0, stream>>>(a); break;
    case 4: pkv_write_kernel<4><<<grid, block, 0, stream>>>(a); break;
    default: pkv_write_kernel<2><<<grid, block, 0, stream>>>(a); break;
  }
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
