// pkv_copy.cu -- pkv_hbm_copy: a plain streaming device-to-device copy, the
// yardstick the decode and write kernels are measured against (the HBM
// bandwidth a copy reaches on this GPU, taken in the same run as them).
//
// Every thread moves 16-byte vectors with four loads in flight before the
// stores, over a grid-stride loop; the grid is eight 256-thread blocks per
// SM (a full SM of resident threads).  Loads and stores carry the
// streaming cache hint: each byte is touched once.
#include <algorithm>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

constexpr int kCopyThreads = 256;
constexpr int kCopyBlocksPerSm = 8;

__global__ void __launch_bounds__(kCopyThreads) pkv_copy_kernel(uint4 *__restrict__ dst,
                                                                const uint4 *__restrict__ src,
                                                                int64_t n) {
  const int64_t stride = (int64_t)gridDim.x * kCopyThreads;
  int64_t i = (int64_t)blockIdx.x * kCopyThreads + threadIdx.x;
  for (; i + 3 * stride < n; i += 4 * stride) {
    const uint4 a = __ldcs(src + i), b = __ldcs(src + i + stride);
    const uint4 c = __ldcs(src + i + 2 * stride), d = __ldcs(src + i + 3 * stride);
    __stcs(dst + i, a);
    __stcs(dst + i + stride, b);
    __stcs(dst + i + 2 * stride, c);
    __stcs(dst + i + 3 * stride, d);
  }
  for (; i < n; i += stride) __stcs(dst + i, __ldcs(src + i));
}

}  // namespace pkv

extern "C" PKV_API pkv_status pkv_hbm_copy(void *dst, const void *src, size_t bytes,
                                           pkv_stream_t stream) {
  if (bytes == 0) return PKV_OK;
  if (!dst || !src || bytes % 16 || reinterpret_cast<uintptr_t>(dst) % 16 ||
      reinterpret_cast<uintptr_t>(src) % 16)
    return PKV_ERR_INVALID_ARG;
  const uintptr_t d0 = reinterpret_cast<uintptr_t>(dst), s0 = reinterpret_cast<uintptr_t>(src);
  if (d0 < s0 + bytes && s0 < d0 + bytes) return PKV_ERR_INVALID_ARG;  // overlapping ranges
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return PKV_ERR_CUDA;
  const int64_t n = (int64_t)(bytes / 16);
  const int64_t want = (n + pkv::kCopyThreads - 1) / pkv::kCopyThreads;
  const int blocks = (int)std::min<int64_t>(want, (int64_t)sms * pkv::kCopyBlocksPerSm);
  pkv::pkv_copy_kernel<<<blocks, pkv::kCopyThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4 *>(dst), static_cast<const uint4 *>(src), n);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
