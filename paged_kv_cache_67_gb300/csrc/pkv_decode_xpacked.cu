// pkv_decode_xpacked.cu -- the layout experiment: paged decode attention over
// caches in vLLM's packed layout instead of the token-major one, and the
// write into that layout.
//
// Layout (interview note "PagedAttention kernel: paged KV cache 与 block
// table", section 深入原理: K cache [num_blocks, num_kv_heads, head_size/x,
// block_size, x] with x = 16 / element size, so that loads are 16-byte
// aligned vectors; V cache [num_blocks, num_kv_heads, head_size,
// block_size]):
//   K_x[blk][kvh][d / 8][off][d % 8]     (x = 8 for 16-bit types)
//   V_x[blk][kvh][d][off]
// Only block_size 16 is served: one block is one 16-token chunk, and one
// (block, KV head) of K (or V) is a single contiguous D * 16 * 2-byte run --
// one bulk copy (cp.async.bulk) instead of D/64 tiled boxes.
//
// Shared-memory fragments.  K_x's 16-byte rows are (d/8, token): rows of
// one ldmatrix 8x8 matrix (8 tokens, 8 consecutive d) are consecutive 16-byte
// rows -- conflict-free without a swizzle -- and give the col-major B
// fragment of K^T directly.  V_x's rows are d with 16 tokens (32 bytes): an
// 8x8 matrix of 8 d-rows x 8 tokens, non-transposed, is the col-major B
// fragment of V (two-way bank conflict: 32-byte row stride).
//
// Everything else -- the work decomposition, the online softmax in log2
// units, masking, the partition epilogue and merge -- is the token-major
// tensor-core kernel's (pkv_decode_tc.cu); the operation is the same
// (course page "P09 · Paged KV 写入 + decode attention（参考实现）", section 题面
// 速览 and the paged_decode_attention shape trace), only the bytes move
// differently.
#include <string.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

constexpr int kXChunk = 16;   // tokens per chunk = block size
constexpr int kXWarps = 4;

template <int D>
struct XShape {
  static constexpr int kSteps = D / 16;
  static constexpr int kNTiles = D / 8;
  static constexpr int kRunBytes = D * kXChunk * 2;       // one (block, head) of K or V
  static constexpr int kStageBytes = 2 * kRunBytes;
  static constexpr int kQStride = D + 8;
  static constexpr int kOStride = D + 8;
  static constexpr bool kQInRegs = D <= 128;
};

size_t xpacked_smem_bytes(int D, int stages) {
  return 1024 + (size_t)kXWarps * stages * 2 * D * kXChunk * 2 + (size_t)kTcHeads * (D + 8) * 2 +
         (size_t)kXWarps * stages * 8 + sizeof(float) * (2 * kXWarps * kTcHeads + 2 * kTcHeads) +
         sizeof(int) * (4 + 2 * kTcHeads);
}

// 1-D bulk copy global -> shared, completion counted on `bar`, L2 evict-first.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// One 16-token chunk of one warp (see the token-major kernel's tc_chunk for
// the softmax; only the fragment addresses differ).
template <int D, typename T, typename QFrag>
__device__ __forceinline__ void x_chunk(uint32_t kb, uint32_t vb, int valid, const QFrag &qfrag,
                                        float (&o)[D / 8][4], float &m0, float &m1, float &l0,
                                        float &l1, float scale_log2, int lane) {
  using Sh = XShape<D>;
  using Mma = MmaOp<T>;
  const int mi = lane >> 3, rw = lane & 7;       // ldmatrix: matrix, row within it
  // K: matrix mi = (tokens 8 (mi >> 1) .., d-group 2 kk + (mi & 1)); row = token
  const uint32_t k_lane = kb + (((mi & 1) * kXChunk + rw + 8 * (mi >> 1)) << 4);
  // V: matrix mi = (d 16 dp + 8 (mi >> 1) .., tokens 8 (mi & 1) ..); row = d
  const uint32_t v_lane = vb + (((rw + 8 * (mi >> 1)) * kXChunk + 8 * (mi & 1)) << 1);

  float sacc[2][2][4] = {};
#pragma unroll
  for (int kk = 0; kk < Sh::kSteps; ++kk) {
    uint32_t b0, b1, b2, b3;
    ldsm_x4(k_lane + kk * (2 * kXChunk * 16), b0, b1, b2, b3);
    uint32_t af[4];
    qfrag(kk, af);
    Mma::run(sacc[kk & 1][0], af, b0, b1);
    Mma::run(sacc[kk & 1][1], af, b2, b3);
  }

  float x[2][4];
  if (valid == kXChunk) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) x[nt][e] = (sacc[0][nt][e] + sacc[1][nt][e]) * scale_log2;
  } else {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tok = nt * 8 + (lane & 3) * 2 + (e & 1);
        x[nt][e] = tok < valid ? (sacc[0][nt][e] + sacc[1][nt][e]) * scale_log2 : -INFINITY;
      }
  }
  float mx0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
  float mx1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
  const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
  if (__any_sync(0xffffffffu, (mn0 > m0) || (mn1 > m1))) {
    const float c0 = fast_exp2(m0 - mn0), c1 = fast_exp2(m1 - mn1);
    l0 *= c0;
    l1 *= c1;
#pragma unroll
    for (int nt = 0; nt < Sh::kNTiles; ++nt) {
      o[nt][0] *= c0; o[nt][1] *= c0;
      o[nt][2] *= c1; o[nt][3] *= c1;
    }
    m0 = mn0;
    m1 = mn1;
  }
  uint32_t pa[4];
  pa[0] = Mma::pack(fast_exp2(x[0][0] - m0), fast_exp2(x[0][1] - m0), l0);
  pa[1] = Mma::pack(fast_exp2(x[0][2] - m1), fast_exp2(x[0][3] - m1), l1);
  pa[2] = Mma::pack(fast_exp2(x[1][0] - m0), fast_exp2(x[1][1] - m0), l0);
  pa[3] = Mma::pack(fast_exp2(x[1][2] - m1), fast_exp2(x[1][3] - m1), l1);

  uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
  if (valid < kXChunk) {
    const int tk = (lane & 3) * 2;
    vm0 = (tk < valid ? 0x0000ffffu : 0u) | (tk + 1 < valid ? 0xffff0000u : 0u);
    vm1 = (tk + 8 < valid ? 0x0000ffffu : 0u) | (tk + 9 < valid ? 0xffff0000u : 0u);
  }
#pragma unroll
  for (int dp = 0; dp < Sh::kSteps; ++dp) {
    uint32_t b0, b1, b2, b3;
    ldsm_x4(v_lane + dp * (16 * kXChunk * 2), b0, b1, b2, b3);
    b0 &= vm0; b1 &= vm1; b2 &= vm0; b3 &= vm1;
    Mma::run(o[2 * dp], pa, b0, b1);
    Mma::run(o[2 * dp + 1], pa, b2, b3);
  }
}

template <int D, typename T>
__global__ void __launch_bounds__(32 * kXWarps, 1) pkv_decode_xpacked_kernel(const DecodeArgs a) {
  using Sh = XShape<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = a.stages;
  uint8_t *ring = smem;                                              // [W][S][K run, V run]
  T *sQ = reinterpret_cast<T *>(ring + (size_t)kXWarps * S * Sh::kStageBytes);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sQ + kTcHeads * Sh::kQStride);
  float *s_wm = reinterpret_cast<float *>(bars + kXWarps * S);
  float *s_wl = s_wm + kXWarps * kTcHeads;
  float *s_m = s_wl + kXWarps * kTcHeads;
  float *s_l = s_m + kTcHeads;
  int *s_scratch = reinterpret_cast<int *>(s_l + kTcHeads);

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int b = blockIdx.z, hc = blockIdx.y, part = blockIdx.x;
  const int kvh = hc / a.gchunks, gc = hc - kvh * a.gchunks;
  const int head0 = kvh * a.G + gc * kTcHeads;
  const int nh = min(kTcHeads, a.G - gc * kTcHeads);

  const int n = checked_len(a, b, part == 0 && hc == 0 && tid == 0);
  int nparts = (n + a.P - 1) / a.P;
  if (nparts > (int)gridDim.x) {
    if (part == (int)gridDim.x - 1 && hc == 0 && tid == 0) raise_flag(a.err, PKV_FLAG_CONTEXT_OVER_HINT);
    nparts = gridDim.x;
  }
  if (n == 0) {
    if (part == 0) zero_rows<T>(a, b, head0, nh);
    return;
  }
  if (part >= nparts) return;
  const int t0 = part * a.P;
  const int t1 = min(n, t0 + a.P);
  const int nchunks = (t1 - t0 + kXChunk - 1) / kXChunk;
  const int nch_w = nchunks > w ? (nchunks - w + kXWarps - 1) / kXWarps : 0;

  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[w * S + s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  const uint64_t policy = l2_evict_first_policy();
  const T *kc = reinterpret_cast<const T *>(a.k_cache);
  const T *vc = reinterpret_cast<const T *>(a.v_cache);
  const size_t run = (size_t)D * kXChunk;                // elements of one (block, head) run
  int tbl_batch = -1, my_phys = 0;
  auto phys_of = [&](int i) -> int {  // physical block of this warp's i-th chunk (warp-collective)
    const int batch = i >> 5;
    if (batch != tbl_batch) {
      tbl_batch = batch;
      const int ii = batch * 32 + lane;
      my_phys = 0;
      if (ii < nch_w) my_phys = checked_block(a, b, (t0 + kXChunk * (w + kXWarps * ii)) / kXChunk);
    }
    return __shfl_sync(0xffffffffu, my_phys, i & 31);
  };
  // chunk i = one block: lane 0 posts the bytes, lanes 0 / 1 copy the K / V run
  auto issue = [&](int i, int slot) {
    const int phys = phys_of(i);
    uint8_t *st = ring + (size_t)(w * S + slot) * Sh::kStageBytes;
    uint64_t *bar = &bars[w * S + slot];
    if (lane == 0) mbar_arrive_expect_tx(bar, Sh::kStageBytes);
    __syncwarp();
    const size_t src = ((size_t)phys * a.KVH + kvh) * run;
    if (lane == 0) bulk_load(st, kc + src, Sh::kRunBytes, bar, policy);
    if (lane == 1) bulk_load(st + Sh::kRunBytes, vc + src, Sh::kRunBytes, bar, policy);
  };
  const int npro = min(S, nch_w);
  for (int i = 0; i < npro; ++i) issue(i, i);

  {
    const T *qg = reinterpret_cast<const T *>(a.q) + ((size_t)b * a.H + head0) * D;
    constexpr int VPR = D / 8;
    for (int i = tid; i < kTcHeads * VPR; i += blockDim.x) {
      const int r = i / VPR, c = i - r * VPR;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r < nh) v = __ldg(reinterpret_cast<const uint4 *>(qg + (size_t)r * D) + c);
      *reinterpret_cast<uint4 *>(sQ + r * Sh::kQStride + c * 8) = v;
    }
  }
  __syncthreads();

  const uint32_t q_lane_addr =
      smem_u32(sQ) + (((lane & 7) + ((lane >> 3) & 1) * 8) * Sh::kQStride + (lane >> 4) * 8) * 2;
  uint32_t qf[Sh::kQInRegs ? Sh::kSteps : 1][4];
  if constexpr (Sh::kQInRegs) {
#pragma unroll
    for (int kk = 0; kk < Sh::kSteps; ++kk)
      ldsm_x4(q_lane_addr + kk * 32, qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
  }
  auto qfrag = [&](int kk, uint32_t(&af)[4]) {
    if constexpr (Sh::kQInRegs) {
      af[0] = qf[kk][0]; af[1] = qf[kk][1]; af[2] = qf[kk][2]; af[3] = qf[kk][3];
    } else {
      ldsm_x4(q_lane_addr + kk * 32, af[0], af[1], af[2], af[3]);
    }
  };

  float o[Sh::kNTiles][4];
#pragma unroll
  for (int nt = 0; nt < Sh::kNTiles; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  int slot = 0;
  uint32_t parity = 0;
  int i = 0;
  for (; i < nch_w; ++i) {
    const bool ok = mbar_wait_bounded(&bars[w * S + slot], parity);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) raise_flag(a.err, PKV_FLAG_TIMEOUT);
      break;
    }
    const int valid = min(kXChunk, t1 - (t0 + kXChunk * (w + kXWarps * i)));
    const uint32_t kb = smem_u32(ring + (size_t)(w * S + slot) * Sh::kStageBytes);
    x_chunk<D, T>(kb, kb + Sh::kRunBytes, valid, qfrag, o, m0, m1, l0, l1, a.scale_log2, lane);
    __syncwarp();
    if (i + S < nch_w) issue(i + S, slot);
    if (++slot == S) {
      slot = 0;
      parity ^= 1u;
    }
  }
  if (i < nch_w) {
    for (int j = i; j < min(i + S, nch_w); ++j) {
      mbar_wait_bounded(&bars[w * S + slot], parity);
      if (++slot == S) {
        slot = 0;
        parity ^= 1u;
      }
    }
  }

  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  const int r0 = lane >> 2, r1 = r0 + 8;
  if ((lane & 3) == 0) {
    s_wm[w * kTcHeads + r0] = m0;
    s_wm[w * kTcHeads + r1] = m1;
    s_wl[w * kTcHeads + r0] = l0;
    s_wl[w * kTcHeads + r1] = l1;
  }
  __syncthreads();
  float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
  for (int ww = 0; ww < kXWarps; ++ww) {
    M0 = fmaxf(M0, s_wm[ww * kTcHeads + r0]);
    M1 = fmaxf(M1, s_wm[ww * kTcHeads + r1]);
  }
  const float f0 = fast_exp2(m0 - M0), f1 = fast_exp2(m1 - M1);
  float *sO = reinterpret_cast<float *>(ring);
  if (r0 < nh) {
#pragma unroll
    for (int nt = 0; nt < Sh::kNTiles; ++nt)
      *reinterpret_cast<float2 *>(sO + (w * kTcHeads + r0) * Sh::kOStride + nt * 8 + (lane & 3) * 2) =
          make_float2(o[nt][0] * f0, o[nt][1] * f0);
  }
  if (r1 < nh) {
#pragma unroll
    for (int nt = 0; nt < Sh::kNTiles; ++nt)
      *reinterpret_cast<float2 *>(sO + (w * kTcHeads + r1) * Sh::kOStride + nt * 8 + (lane & 3) * 2) =
          make_float2(o[nt][2] * f1, o[nt][3] * f1);
  }
  if (tid < kTcHeads) {
    float M = -INFINITY;
    for (int ww = 0; ww < kXWarps; ++ww) M = fmaxf(M, s_wm[ww * kTcHeads + tid]);
    float L = 0.f;
    for (int ww = 0; ww < kXWarps; ++ww)
      L += s_wl[ww * kTcHeads + tid] * fast_exp2(s_wm[ww * kTcHeads + tid] - M);
    s_m[tid] = M;
    s_l[tid] = L;
  }
  __syncthreads();
  for (int e = tid; e < nh * D; e += blockDim.x) {
    const int r = e / D, d = e - r * D;
    float acc = 0.f;
#pragma unroll
    for (int ww = 0; ww < kXWarps; ++ww) acc += sO[(ww * kTcHeads + r) * Sh::kOStride + d];
    sO[r * Sh::kOStride + d] = acc;
  }
  __syncthreads();
  finish_partition<T>(a, b, head0, nh, part, nparts, s_m, s_l, sO, Sh::kOStride, s_scratch,
                      a.ws_cnt + (size_t)b * gridDim.y + blockIdx.y, tid, blockDim.x, CtaSync(),
                      false);
}

// Write into the packed layout: one warp per token; K as 16-byte runs of 8
// d-values (contiguous in both layouts), V element by element (token-minor).
template <typename T>
__global__ void pkv_write_xpacked_kernel(T *kx, T *vx, const T *k, const T *v, const int64_t *slots,
                                         long long ntok, long long k_stride, long long v_stride,
                                         long long num_blocks, int KVH, int D, int *err) {
  const long long i = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= ntok) return;
  const long long slot = slots[i];
  if (slot < 0) return;
  if (slot >= num_blocks * kXChunk) {
    if (lane == 0) raise_flag(err, PKV_FLAG_SLOT_OUT_OF_RANGE);
    return;
  }
  const long long blk = slot / kXChunk, off = slot % kXChunk;
  const int vec = D / 8;
  for (int e = lane; e < KVH * vec; e += 32) {  // K: (kvh, d / 8) runs
    const int h = e / vec, dg = e - h * vec;
    const uint4 val = *reinterpret_cast<const uint4 *>(k + i * k_stride + (size_t)h * D + dg * 8);
    *reinterpret_cast<uint4 *>(kx + ((((size_t)blk * KVH + h) * vec + dg) * kXChunk + off) * 8) = val;
  }
  for (int e = lane; e < KVH * D; e += 32) {    // V: (kvh, d) elements
    const int h = e / D, d = e - h * D;
    vx[(((size_t)blk * KVH + h) * D + d) * kXChunk + off] = v[i * v_stride + (size_t)h * D + d];
  }
}

// ---------------------------------------------------------------- host side

template <int D, typename T>
static pkv_status launch_x_t(const DecodeArgs &a, const DecodePlan &plan, cudaStream_t stream) {
  auto kern = pkv_decode_xpacked_kernel<D, T>;
  static int configured[64] = {0};
  const size_t smem = xpacked_smem_bytes(D, plan.stages);
  if (!allow_smem(kern, smem, configured)) return PKV_ERR_CUDA;
  dim3 grid(plan.max_parts, a.KVH * plan.gchunks, a.B);
  kern<<<grid, 32 * kXWarps, smem, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status launch_decode_xpacked(const DecodeArgs &a, const DecodePlan &plan, pkv_dtype dt,
                                 cudaStream_t stream) {
  const bool bf = dt == PKV_BF16;
  switch (a.D) {
    case 64: return bf ? launch_x_t<64, __nv_bfloat16>(a, plan, stream)
                       : launch_x_t<64, __half>(a, plan, stream);
    case 128: return bf ? launch_x_t<128, __nv_bfloat16>(a, plan, stream)
                        : launch_x_t<128, __half>(a, plan, stream);
    case 256: return bf ? launch_x_t<256, __nv_bfloat16>(a, plan, stream)
                        : launch_x_t<256, __half>(a, plan, stream);
  }
  return PKV_ERR_UNSUPPORTED;
}

pkv_status launch_write_xpacked(void *kx, void *vx, const void *k, const void *v,
                                const int64_t *slots, long long ntok, long long k_stride,
                                long long v_stride, long long num_blocks, int KVH, int D,
                                pkv_dtype dt, int *err, cudaStream_t stream) {
  const int warps = 8;
  const long long blocks = (ntok + warps - 1) / warps;
  if (blocks > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
  if (dt == PKV_BF16)
    pkv_write_xpacked_kernel<__nv_bfloat16><<<(unsigned)blocks, 32 * warps, 0, stream>>>(
        static_cast<__nv_bfloat16 *>(kx), static_cast<__nv_bfloat16 *>(vx),
        static_cast<const __nv_bfloat16 *>(k), static_cast<const __nv_bfloat16 *>(v), slots, ntok,
        k_stride, v_stride, num_blocks, KVH, D, err);
  else
    pkv_write_xpacked_kernel<__half><<<(unsigned)blocks, 32 * warps, 0, stream>>>(
        static_cast<__half *>(kx), static_cast<__half *>(vx), static_cast<const __half *>(k),
        static_cast<const __half *>(v), slots, ntok, k_stride, v_stride, num_blocks, KVH, D, err);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
