// pkv_decode_simt.cu -- paged decode attention on the CUDA cores.
//
// Any dtype (fp32, bf16, fp16), any head_dim in [1, 512], any block size.
// It serves fp32 caches (whose tolerance rules out bf16 tensor-core inputs)
// and the shapes the TMA/tensor-core kernel does not take.
//
// Definition (course page "P09 · Paged KV 写入 + decode attention（参考实现）",
// section 题面速览 "decode 读" and the paged_decode_attention shape trace):
// n = context_lens[b]; only block_tables[b, :ceil(n/bs)] is read; logical
// token t is row t % bs of physical block tbl[t / bs]; exactly n tokens;
// query head h uses KV head h / (H / KVH); fp32 scores scaled before an
// fp32 softmax; weighted sum of V; cast to the output dtype.
//
// CTA = (partition, KV head x head chunk, sequence), 4 warps.  The CTA
// stages its window of table entries in shared memory (checked once); each
// warp walks every 4th token of the partition with its lanes spread over
// head_dim (the row loads of several of its tokens in flight at once), keeps
// one online-softmax state (running max m, sum l, weighted
// V sum) per query head in registers -- the online softmax of the interview
// note "PagedAttention kernel: paged KV cache 与 block table", section 代码 --
// and the four warp states are merged at the end.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

constexpr int kSimtWarps = 4;
constexpr int kTableWindow = 256;  // table entries staged per window

template <typename T, int EPL, int GH, bool kAppend>
__global__ void __launch_bounds__(32 * kSimtWarps) pkv_decode_simt_kernel(const DecodeArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const int D = a.D;
  int *s_tbl = reinterpret_cast<int *>(smem_raw);                     // [kTableWindow]
  float *s_wm = reinterpret_cast<float *>(s_tbl + kTableWindow);      // [W][GH]
  float *s_wl = s_wm + kSimtWarps * GH;                               // [W][GH]
  float *s_m = s_wl + kSimtWarps * GH;                                // [GH]
  float *s_l = s_m + GH;                                              // [GH]
  int *s_scratch = reinterpret_cast<int *>(s_l + GH);                 // [1 + 2*GH]
  float *s_wo = reinterpret_cast<float *>(s_scratch + 4 + 2 * GH);    // [W][GH][D]
  float *s_o = s_wo + kSimtWarps * GH * D;                            // [GH][D]

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int b = blockIdx.z, hc = blockIdx.y, part = blockIdx.x;
  const int kvh = hc / a.gchunks, gc = hc - kvh * a.gchunks;
  const int head0 = kvh * a.G + gc * a.heads_per_cta;
  const int nh = min(a.heads_per_cta, a.G - gc * a.heads_per_cta);

  const int n = checked_len(a, b, part == 0 && hc == 0 && tid == 0);
  int nparts = (n + a.P - 1) / a.P;
  if (nparts > (int)gridDim.x) {
    if (part == (int)gridDim.x - 1 && hc == 0 && tid == 0) raise_flag(a.err, PKV_FLAG_CONTEXT_OVER_HINT);
    nparts = gridDim.x;
  }
  // fused append (kAppend): the new token's slot, or -1
  const long long s_new = kAppend ? append_slot(a, b) : -1LL;
  if (n == 0) {
    if (part == 0) {
      zero_rows<T>(a, b, head0, nh);
      if (s_new >= 0 && gc == 0 && w == 0) append_write_row<T>(a, b, kvh, s_new, n, lane);
    }
    return;
  }
  if (part >= nparts) return;
  const int t0 = part * a.P;
  const int t1 = min(n, t0 + a.P);
  const int bs = a.bs;
  // Fused append: one CTA per (sequence, KV head) writes the cache row;
  // every CTA reads position n-1 from the new token's input row instead of
  // the cache, so no read waits for (or races with) that write.
  if (s_new >= 0 && gc == 0 && part == nparts - 1 && w == 0)
    append_write_row<T>(a, b, kvh, s_new, n, lane);
  const int t_new = s_new >= 0 ? n - 1 : -1;

  // Queries of this CTA's heads, scaled into log2 units: s2 = q.k * scale * log2(e).
  const T *qg = reinterpret_cast<const T *>(a.q) + ((size_t)b * a.H + head0) * D;
  float qv[GH][EPL];
#pragma unroll
  for (int r = 0; r < GH; ++r)
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const int d = lane + 32 * e;
      qv[r][e] = (r < nh && d < D) ? to_f32<T>(qg[(size_t)r * D + d]) * a.scale_log2 : 0.f;
    }

  float m[GH], l[GH], acc[GH][EPL];
#pragma unroll
  for (int r = 0; r < GH; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[r][e] = 0.f;
  }

  const T *kc = reinterpret_cast<const T *>(a.k_cache);
  const T *vc = reinterpret_cast<const T *>(a.v_cache);
  const size_t tok_stride = (size_t)a.KVH * D;  // elements between rows of one block
  const int lb_first = t0 / bs, lb_last = (t1 - 1) / bs;

  for (int lbA = lb_first; lbA <= lb_last; lbA += kTableWindow) {
    const int cnt = min(kTableWindow, lb_last - lbA + 1);
    __syncthreads();  // the previous window is no longer read
    for (int i = tid; i < cnt; i += blockDim.x) s_tbl[i] = checked_block(a, b, lbA + i);
    __syncthreads();
    const int ta = max(t0, lbA * bs), tb = min(t1, (lbA + cnt) * bs);
    // kU tokens of the warp per step: every row load of the step is issued
    // before any is used, so the step costs one memory round trip, not kU;
    // the tokens are still taken in the warp's order (same results).  Only
    // for head_dim <= 64 (four registers per token): with more values per
    // lane the extra registers halve the resident CTAs, which cost more than
    // the round trips saved (bf16, head_dim 128: 543 -> 829 us on the
    // 8B-shaped batch at kU = 4).
    constexpr int kU = EPL <= 2 ? 8 : 1;
    for (int tu = ta + w; tu < tb; tu += kSimtWarps * kU) {
      float kx[kU][EPL], vx[kU][EPL];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int t = tu + u * kSimtWarps;
        const T *kp = kc, *vp = vc;
        bool live = t < tb;
        if (live) {
          const int lb = t / bs;
          const int phys = s_tbl[lb - lbA];
          const size_t row = ((size_t)phys * bs + (t - lb * bs)) * tok_stride + (size_t)kvh * D;
          kp = kc + row;
          vp = vc + row;
          if (t == t_new) {
            kp = reinterpret_cast<const T *>(append_src<T>(a, false, b, kvh));
            vp = reinterpret_cast<const T *>(append_src<T>(a, true, b, kvh));
          }
        }
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          const int d = lane + 32 * e;
          kx[u][e] = (live && d < D) ? to_f32<T>(kp[d]) : 0.f;
          vx[u][e] = (live && d < D) ? to_f32<T>(vp[d]) : 0.f;
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        if (tu + u * kSimtWarps >= tb) break;
#pragma unroll
        for (int r = 0; r < GH; ++r) {
          float s = 0.f;
#pragma unroll
          for (int e = 0; e < EPL; ++e) s = fmaf(qv[r][e], kx[u][e], s);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
          const float mn = fmaxf(m[r], s);
          const float corr = fast_exp2(m[r] - mn);
          const float p = fast_exp2(s - mn);
          l[r] = fmaf(l[r], corr, p);
#pragma unroll
          for (int e = 0; e < EPL; ++e) acc[r][e] = fmaf(acc[r][e], corr, p * vx[u][e]);
          m[r] = mn;
        }
      }
    }
  }

  // Merge the four warp states: rescale each to the common max.
#pragma unroll
  for (int r = 0; r < GH; ++r) {
    if (lane == 0) {
      s_wm[w * GH + r] = m[r];
      s_wl[w * GH + r] = l[r];
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const int d = lane + 32 * e;
      if (d < D) s_wo[(w * GH + r) * D + d] = acc[r][e];
    }
  }
  __syncthreads();
  if (tid < nh) {
    float M = -INFINITY;
    for (int ww = 0; ww < kSimtWarps; ++ww) M = fmaxf(M, s_wm[ww * GH + tid]);
    float L = 0.f;
    for (int ww = 0; ww < kSimtWarps; ++ww) L += s_wl[ww * GH + tid] * fast_exp2(s_wm[ww * GH + tid] - M);
    s_m[tid] = M;
    s_l[tid] = L;
  }
  __syncthreads();
  for (int i = tid; i < nh * D; i += blockDim.x) {
    const int r = i / D, d = i - r * D;
    float o = 0.f;
    for (int ww = 0; ww < kSimtWarps; ++ww)
      o += s_wo[(ww * GH + r) * D + d] * fast_exp2(s_wm[ww * GH + r] - s_m[r]);
    s_o[r * D + d] = o;
  }
  __syncthreads();
  finish_partition<T>(a, b, head0, nh, part, nparts, s_m, s_l, s_o, D, s_scratch,
                      a.ws_cnt + (size_t)b * gridDim.y + blockIdx.y, tid, blockDim.x, CtaSync(),
                      false);
}

template <typename T, int EPL, int GH>
static pkv_status launch_simt_t(const DecodeArgs &a, const DecodePlan &plan, cudaStream_t stream) {
  dim3 grid(plan.max_parts, a.KVH * plan.gchunks, a.B);
  if (a.new_slots)
    pkv_decode_simt_kernel<T, EPL, GH, true><<<grid, 32 * kSimtWarps, plan.smem_bytes, stream>>>(a);
  else
    pkv_decode_simt_kernel<T, EPL, GH, false><<<grid, 32 * kSimtWarps, plan.smem_bytes, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

template <typename T>
static pkv_status launch_simt_dt(const DecodeArgs &a, const DecodePlan &plan, cudaStream_t stream) {
  if (a.D <= 32) return launch_simt_t<T, 1, 4>(a, plan, stream);
  if (a.D <= 64) return launch_simt_t<T, 2, 4>(a, plan, stream);
  if (a.D <= 128) return launch_simt_t<T, 4, 4>(a, plan, stream);
  if (a.D <= 256) return launch_simt_t<T, 8, 4>(a, plan, stream);
  return launch_simt_t<T, 16, 2>(a, plan, stream);
}

size_t simt_smem_bytes(int D, int GH) {
  return sizeof(int) * kTableWindow + sizeof(float) * (2 * kSimtWarps * GH + 2 * GH) +
         sizeof(int) * (4 + 2 * GH) + sizeof(float) * ((size_t)kSimtWarps * GH * D + (size_t)GH * D);
}

pkv_status launch_decode_simt(const DecodeArgs &a, const DecodePlan &plan, pkv_dtype dt,
                              cudaStream_t stream) {
  switch (dt) {
    case PKV_F32: return launch_simt_dt<float>(a, plan, stream);
    case PKV_BF16: return launch_simt_dt<__nv_bfloat16>(a, plan, stream);
    case PKV_F16: return launch_simt_dt<__half>(a, plan, stream);
  }
  return PKV_ERR_INVALID_ARG;
}

}  // namespace pkv
