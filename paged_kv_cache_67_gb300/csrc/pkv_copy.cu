// pkv_copy.cu -- the yardsticks the decode and write kernels are measured
// against, taken in the same run as them:
//   pkv_hbm_copy         a plain streaming device-to-device copy (the HBM
//                        bandwidth a copy reaches on this GPU);
//   pkv_hbm_gather_read  reads of whole chunks at listed places (the
//                        bandwidth reads of randomly placed cache blocks
//                        reach -- the decode's own access pattern, without
//                        its arithmetic); pkv_hbm_gather_read_pair reads the
//                        listed chunks of two buffers (K and V) in one launch.
//
// The copy: one 256-thread block per contiguous run of 1024 16-byte
// vectors, each thread with its four loads in flight before its stores (a
// grid of many short blocks: on a GB300, 7.05 TB/s on 1 GiB against 6.72
// for a persistent grid-stride loop and 6.65 for cudaMemcpyAsync).  Loads
// and stores carry the streaming cache hint: each byte is touched once.
//
// The gather: one warp per chunk at a time (chunks taken in list order,
// grid-stride over warps), each lane with eight 16-byte loads in flight;
// the words are folded by XOR into a checksum so that no load is dead.
//
//   pkv_fp32_fma_peak    the fp32 multiply-add rate of the CUDA cores: eight
//                        independent chains per thread (enough, with eight
//                        blocks of 256 threads per SM, to keep every lane's
//                        FMA pipe busy), plain fmaf or paired fma.rn.f32x2.
#include <algorithm>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

constexpr int kCopyThreads = 256;
constexpr int kCopyVecs = 4;   // 16-byte vectors per thread

__global__ void __launch_bounds__(kCopyThreads) pkv_copy_kernel(uint4 *__restrict__ dst,
                                                                const uint4 *__restrict__ src,
                                                                int64_t n) {
  const int64_t base = (int64_t)blockIdx.x * (kCopyVecs * kCopyThreads) + threadIdx.x;
  uint4 r[kCopyVecs];
#pragma unroll
  for (int u = 0; u < kCopyVecs; ++u) {
    const int64_t i = base + u * kCopyThreads;
    if (i < n) r[u] = __ldcs(src + i);
  }
#pragma unroll
  for (int u = 0; u < kCopyVecs; ++u) {
    const int64_t i = base + u * kCopyThreads;
    if (i < n) __stcs(dst + i, r[u]);
  }
}

constexpr int kGatherThreads = 256;
constexpr int kGatherBlocksPerSm = 8;
constexpr int kGatherInFlight = 8;

// Chunk c < nchunks of the list is read from base, chunk nchunks + c (with
// a second base) from base2: one launch over both.
__global__ void __launch_bounds__(kGatherThreads) pkv_gather_read_kernel(
    const uint8_t *__restrict__ base, const uint8_t *__restrict__ base2,
    const int32_t *__restrict__ index, int64_t nchunks, int64_t stride, int64_t vecs,
    unsigned long long *sink) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (kGatherThreads / 32);
  const int64_t total = base2 ? 2 * nchunks : nchunks;
  uint4 acc = make_uint4(0, 0, 0, 0);
  for (int64_t c = (int64_t)blockIdx.x * (kGatherThreads / 32) + (threadIdx.x >> 5); c < total;
       c += warps) {
    const bool second = c >= nchunks;
    const uint4 *src = reinterpret_cast<const uint4 *>((second ? base2 : base) +
                                                       (int64_t)__ldg(index + (second ? c - nchunks : c)) * stride);
    int64_t v = lane;
    for (; v + 32 * (kGatherInFlight - 1) < vecs; v += 32 * kGatherInFlight) {
      uint4 r[kGatherInFlight];
#pragma unroll
      for (int u = 0; u < kGatherInFlight; ++u) r[u] = __ldcs(src + v + 32 * u);
#pragma unroll
      for (int u = 0; u < kGatherInFlight; ++u) {
        acc.x ^= r[u].x; acc.y ^= r[u].y; acc.z ^= r[u].z; acc.w ^= r[u].w;
      }
    }
    for (; v < vecs; v += 32) {
      const uint4 r = __ldcs(src + v);
      acc.x ^= r.x; acc.y ^= r.y; acc.z ^= r.z; acc.w ^= r.w;
    }
  }
  unsigned long long x = ((unsigned long long)acc.y << 32 | acc.x) ^ ((unsigned long long)acc.w << 32 | acc.z);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x ^= __shfl_xor_sync(0xffffffffu, x, o);
  if (lane == 0 && x != 0) atomicXor(sink, x);
}

constexpr int kFmaThreads = 256;
constexpr int kFmaChains = 8;

template <bool kPaired>
__global__ void __launch_bounds__(kFmaThreads) pkv_fma_kernel(float *out, int iters, float a,
                                                             float b, float never) {
  float x[kFmaChains];
#pragma unroll
  for (int k = 0; k < kFmaChains; ++k) x[k] = 0.f;
  if constexpr (kPaired) {
    const float2 a2 = make_float2(a, a), b2 = make_float2(b, b);
    float2 *x2 = reinterpret_cast<float2 *>(x);
    for (int i = 0; i < iters; ++i) {
#pragma unroll
      for (int k = 0; k < kFmaChains / 2; ++k) x2[k] = ffma2(x2[k], a2, b2);
    }
  } else {
    for (int i = 0; i < iters; ++i) {
#pragma unroll
      for (int k = 0; k < kFmaChains; ++k) x[k] = fmaf(x[k], a, b);
    }
  }
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < kFmaChains; ++k) s += x[k];
  if (threadIdx.x == 0 || s == never) out[blockIdx.x] = s;
}

}  // namespace pkv

extern "C" PKV_API pkv_status pkv_fp32_fma_peak(float *out, int blocks, int iters, float a, float b,
                                                float never, int paired, pkv_stream_t stream) {
  if (!out || reinterpret_cast<uintptr_t>(out) % 4 || blocks < 1 || blocks > (1 << 20) || iters < 0)
    return PKV_ERR_INVALID_ARG;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (paired)
    pkv::pkv_fma_kernel<true><<<blocks, pkv::kFmaThreads, 0, st>>>(out, iters, a, b, never);
  else
    pkv::pkv_fma_kernel<false><<<blocks, pkv::kFmaThreads, 0, st>>>(out, iters, a, b, never);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

static pkv_status gather_read(const void *base, const void *base2, const int32_t *chunk_index,
                              int64_t nchunks, int64_t chunk_stride_bytes, int64_t chunk_bytes,
                              unsigned long long *sink, pkv_stream_t stream) {
  if (nchunks < 0 || chunk_stride_bytes < 0 || chunk_bytes < 0) return PKV_ERR_INVALID_ARG;
  if (nchunks == 0 || chunk_bytes == 0) return PKV_OK;
  if (!base || !chunk_index || !sink || chunk_bytes % 16 || chunk_stride_bytes % 16 ||
      reinterpret_cast<uintptr_t>(base) % 16 || reinterpret_cast<uintptr_t>(base2) % 16 ||
      reinterpret_cast<uintptr_t>(chunk_index) % 4 || reinterpret_cast<uintptr_t>(sink) % 8)
    return PKV_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return PKV_ERR_CUDA;
  const int64_t total = base2 ? 2 * nchunks : nchunks;
  const int64_t want = (total + pkv::kGatherThreads / 32 - 1) / (pkv::kGatherThreads / 32);
  const int blocks = (int)std::min<int64_t>(want, (int64_t)sms * pkv::kGatherBlocksPerSm);
  pkv::pkv_gather_read_kernel<<<blocks, pkv::kGatherThreads, 0,
                                reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint8_t *>(base), static_cast<const uint8_t *>(base2), chunk_index, nchunks,
      chunk_stride_bytes, chunk_bytes / 16, sink);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" PKV_API pkv_status pkv_hbm_gather_read(const void *base, const int32_t *chunk_index,
                                                  int64_t nchunks, int64_t chunk_stride_bytes,
                                                  int64_t chunk_bytes, unsigned long long *sink,
                                                  pkv_stream_t stream) {
  return gather_read(base, nullptr, chunk_index, nchunks, chunk_stride_bytes, chunk_bytes, sink,
                     stream);
}

extern "C" PKV_API pkv_status pkv_hbm_gather_read_pair(const void *base_a, const void *base_b,
                                                       const int32_t *chunk_index, int64_t nchunks,
                                                       int64_t chunk_stride_bytes,
                                                       int64_t chunk_bytes,
                                                       unsigned long long *sink,
                                                       pkv_stream_t stream) {
  if (!base_b) return PKV_ERR_INVALID_ARG;
  return gather_read(base_a, base_b, chunk_index, nchunks, chunk_stride_bytes, chunk_bytes, sink,
                     stream);
}

extern "C" PKV_API pkv_status pkv_hbm_copy(void *dst, const void *src, size_t bytes,
                                           pkv_stream_t stream) {
  if (bytes == 0) return PKV_OK;
  if (!dst || !src || bytes % 16 || reinterpret_cast<uintptr_t>(dst) % 16 ||
      reinterpret_cast<uintptr_t>(src) % 16)
    return PKV_ERR_INVALID_ARG;
  const uintptr_t d0 = reinterpret_cast<uintptr_t>(dst), s0 = reinterpret_cast<uintptr_t>(src);
  if (d0 < s0 + bytes && s0 < d0 + bytes) return PKV_ERR_INVALID_ARG;  // overlapping ranges
  const int64_t n = (int64_t)(bytes / 16);
  const int64_t per_block = (int64_t)pkv::kCopyVecs * pkv::kCopyThreads;
  const int64_t blocks = (n + per_block - 1) / per_block;
  if (blocks > 0x7fffffffLL) return PKV_ERR_INVALID_ARG;
  pkv::pkv_copy_kernel<<<(unsigned)blocks, pkv::kCopyThreads, 0,
                         reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4 *>(dst), static_cast<const uint4 *>(src), n);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
