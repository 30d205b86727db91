// pkv_prefill_tc.cu -- paged causal prefill attention (several new query
// tokens per sequence, varlen) for bf16 / fp16 caches on sm_103a, on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// Definition.  The pages only ask how the varlen prefill version would be
// written (course page "P09 · Paged KV 写入 + decode attention（参考实现）",
// section 面试官追问); this library reads it as the multi-query form of the
// decode it defines (same page, section 细节: the decode query is the newest
// token, already written, and sees the whole context including itself):
// sequence b's qlen = cu_seqlens_q[b+1] - cu_seqlens_q[b] queries are the
// last qlen of its n = context_lens[b] tokens (already written to the
// cache); query i sits at position p = n - qlen + i and attends to tokens
// 0 .. p; query head h reads KV head h / (H / KVH); fp32 scores scaled before
// an fp32 softmax; the weighted sum of V rows is cast to the output type.
// The tile-wise online softmax is the block-wise one of the interview note
// "PagedAttention kernel: paged KV cache 与 block table", section 代码.
//
// Work decomposition.  CTA = (query head, 128-query tile, sequence), the
// heaviest tiles (latest queries) first; 6 warps:
//   warp 0     producer: per 128-token KV tile, 32 lanes issue one tiled TMA
//              load each (a 16-token chunk of one 64-column region of K or V
//              of this KV head, 128-byte swizzle) into a 2-stage ring;
//   warp 1     MMA issuer (one thread): S = Q . K^T (M = 128 queries,
//              N = 128 tokens, fp32 in tensor memory), then O += P . V
//              (N = D), S of the next tile issued before P . V of this one;
//   warps 2-5  softmax, one query row per thread (its tensor-memory lane):
//              stage Q, then per tile read S, mask (causal, end of context),
//              update the running max -- the reference max moves only when
//              the row max grows by more than 2^8, and only then is the
//              O row in tensor memory rescaled -- write P = 2^(s - m) as
//              bf16/fp16 into a swizzled shared tile, and finally O / l.
// Every wait on an mbarrier is bounded; on time-out the CTA raises
// PKV_FLAG_TIMEOUT, lets its copies and products land (bounded) and exits.
#include <string.h>

#include <type_traits>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_tcgen05.cuh"

namespace pkv {

constexpr int kPfRows = 128;     // query rows per CTA (MMA M)
constexpr int kPfTile = 128;     // KV tokens per tile
constexpr int kPfStages = 2;     // K/V ring depth
constexpr int kPfWarps = 6;
constexpr int kPfThreads = 32 * kPfWarps;
constexpr int kRegionBytes = 128 * 128;  // 128 rows x 64 elements of 16 bits

struct PrefillArgs {
  void *out;
  const void *q;
  const int32_t *tables;
  const int32_t *cu_q;
  const int32_t *lens;
  int *err;
  long long num_blocks;
  int B, H, KVH, D, G, bs, max_blocks;
  int q_tiles;        // 128-query tiles per sequence the grid covers (gridDim.y)
  float scale_log2;   // scale * log2(e)
};

template <int D>
struct PfShape {
  static constexpr int kRegions = D / 64;
  static constexpr int kTileBytes = kRegions * kRegionBytes;      // one 128-row operand
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQOff + kTileBytes;               // [stage][K, V]
  static constexpr int kPOff = kKVOff + kPfStages * 2 * kTileBytes;
  static constexpr int kBarOff = kPOff + 2 * kRegionBytes;        // P: 128 tokens
  static constexpr int kSmem = kBarOff + 256 + 1024;              // + alignment slack
  static constexpr uint32_t kTmemCols = 256;                      // S: 128, O: D
};

// Tiled 4-D TMA load global -> shared with the default L2 policy (the K/V
// tiles are read again by the other heads of the group and later tiles).
__device__ __forceinline__ void tma_load_4d_keep(void *dst, const CUtensorMap *map, uint64_t *bar,
                                                 int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
      "r"(c3)
      : "memory");
}

template <typename T>
struct PackPair;
template <>
struct PackPair<__nv_bfloat16> {
  // two fp32 -> packed bf16 pair (RNE); also adds the rounded values to sum
  __device__ __forceinline__ static uint32_t run(float lo, float hi, float &sum) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    const float2 f = __bfloat1622float2(v);
    sum += f.x + f.y;
    return *reinterpret_cast<uint32_t *>(&v);
  }
};
template <>
struct PackPair<__half> {
  __device__ __forceinline__ static uint32_t run(float lo, float hi, float &sum) {
    __half2 v = __floats2half2_rn(lo, hi);
    const float2 f = __half22float2(v);
    sum += f.x + f.y;
    return *reinterpret_cast<uint32_t *>(&v);
  }
};

template <int D, typename T>
__global__ void __launch_bounds__(kPfThreads, 1)
    pkv_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const PrefillArgs a) {
  using Sh = PfShape<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + Sh::kBarOff);
  uint64_t *q_full = bars + 0;
  uint64_t *kv_full = bars + 1;    // [2]
  uint64_t *kv_empty = bars + 3;   // [2]
  uint64_t *s_full = bars + 5;
  uint64_t *p_full = bars + 6;
  uint64_t *o_done = bars + 7;
  uint64_t *mma_done = bars + 8;
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 12);
  int *abort_flag = reinterpret_cast<int *>(bars + 13);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.x, b = blockIdx.z;
  const int qt = a.q_tiles - 1 - (int)blockIdx.y;  // latest (heaviest) tiles first

  // ---- the sequence and this CTA's query rows (uniform: before any barrier)
  const int q0 = __ldg(a.cu_q + b), qlen = __ldg(a.cu_q + b + 1) - q0;
  const int n = __ldg(a.lens + b);
  const bool lead = h == 0 && blockIdx.y == 0 && tid == 0;
  if (qlen < 0 || n < qlen || (long long)n > (long long)a.max_blocks * a.bs) {
    if (lead) raise_flag(a.err, PKV_FLAG_QUERY_LEN);
    return;
  }
  if (qlen > a.q_tiles * kPfRows && lead) raise_flag(a.err, PKV_FLAG_QUERY_OVER_HINT);
  const int i0 = qt * kPfRows;
  if (i0 >= qlen) return;
  const int rows = min(kPfRows, qlen - i0);
  const int p_first = n - qlen + i0;               // position of query row 0
  const int p_last = p_first + rows - 1;           // position of the last real row
  const int ntiles = p_last / kPfTile + 1;
  const int kvh = h / a.G;

  if (tid == 0) {
    mbar_init(q_full, 128);
    for (int s = 0; s < kPfStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, 128);
    mbar_init(o_done, 1);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_holder, Sh::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t tmem_s = tmem, tmem_o = tmem + 128;
  constexpr bool bf16 = std::is_same<T, __nv_bfloat16>::value;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const int per_tensor = 8 * Sh::kRegions;       // boxes of K (or V) per tile
    const bool issuer = lane < 2 * per_tensor;
    const bool is_v = lane >= per_tensor;
    const int region = (lane % per_tensor) >> 3, chunk = lane & 7;
    int issued = 0;
    for (int j = 0; j < ntiles; ++j) {
      const int stage = j & 1;
      if (j >= kPfStages) {
        const bool ok = mbar_wait_bounded(&kv_empty[stage], ((j >> 1) - 1) & 1);
        if (!__all_sync(0xffffffffu, ok) || *(volatile int *)abort_flag) {
          if (lane == 0) {
            raise_flag(a.err, PKV_FLAG_TIMEOUT);
            *(volatile int *)abort_flag = 1;
          }
          break;
        }
      }
      const int tok0 = j * kPfTile;
      const int valid_chunks = min(8, (n - tok0 + 15) >> 4);
      if (lane == 0)
        mbar_arrive_expect_tx(&kv_full[stage],
                              (uint32_t)(valid_chunks * 2 * Sh::kRegions * 2048));
      __syncwarp();
      if (issuer && chunk < valid_chunks) {
        const int t = tok0 + 16 * chunk;
        const int lb = t / a.bs;
        int phys = __ldg(a.tables + (size_t)b * a.max_blocks + lb);
        if (phys < 0 || (long long)phys >= a.num_blocks) {
          raise_flag(a.err, PKV_FLAG_BLOCK_OUT_OF_RANGE);
          phys = 0;
        }
        uint8_t *dst = sm + Sh::kKVOff + stage * 2 * Sh::kTileBytes + (is_v ? Sh::kTileBytes : 0) +
                       region * kRegionBytes + chunk * 2048;
        tma_load_4d_keep(dst, is_v ? &tmV : &tmK, &kv_full[stage], region * 64, kvh, t - lb * a.bs,
                         phys);
      }
      ++issued;
    }
    // the last fills land before the CTA can end (bounded)
    for (int j = max(0, issued - kPfStages); j < issued; ++j)
      mbar_wait_bounded(&kv_full[j & 1], (j >> 1) & 1);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = umma_idesc_f16(128, kPfTile, bf16, false);
      const uint32_t idesc_o = umma_idesc_f16(128, D, bf16, true);
      const uint32_t q_base = smem_u32(sm + Sh::kQOff), p_base = smem_u32(sm + Sh::kPOff);
      auto kv_base = [&](int j, bool v) {
        return smem_u32(sm + Sh::kKVOff + (j & 1) * 2 * Sh::kTileBytes + (v ? Sh::kTileBytes : 0));
      };
      auto issue_s = [&](int j) {  // S = Q . K_j^T over D in 16-wide steps
        const uint32_t kb = kv_base(j, false);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * kRegionBytes + (k & 3) * 32;
          umma_f16(tmem_s, umma_desc_sw128(q_base + off, 16, 1024),
                   umma_desc_sw128(kb + off, 16, 1024), idesc_s, k > 0);
        }
        umma_commit(s_full);
      };
      bool ok = mbar_wait_bounded(q_full, 0) && mbar_wait_bounded(&kv_full[0], 0);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      for (int j = 0; ok && j < ntiles; ++j) {
        ok = mbar_wait_bounded(p_full, j & 1) && !*(volatile int *)abort_flag;
        if (!ok) break;
        tc_fence_after();
        if (j + 1 < ntiles) {
          ok = mbar_wait_bounded(&kv_full[(j + 1) & 1], ((j + 1) >> 1) & 1);
          if (!ok) break;
          tc_fence_after();
          issue_s(j + 1);
        }
        const uint32_t vb = kv_base(j, true);
#pragma unroll
        for (int k = 0; k < kPfTile / 16; ++k) {  // O += P_j . V_j over 16-token steps
          const uint32_t poff = (k >> 2) * kRegionBytes + (k & 3) * 32;
          umma_f16(tmem_o, umma_desc_sw128(p_base + poff, 16, 1024),
                   umma_desc_sw128(vb + k * 2048, kRegionBytes, 1024), idesc_o, (j > 0 || k > 0));
        }
        umma_commit(o_done);
        umma_commit(&kv_empty[j & 1]);
      }
      if (!ok) {
        raise_flag(a.err, PKV_FLAG_TIMEOUT);
        *(volatile int *)abort_flag = 1;
      }
      umma_commit(mma_done);  // every product issued above has completed when this arrives
      mbar_wait_bounded(mma_done, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;
    const int r = 32 * quarter + lane;                  // query row = tensor-memory lane
    const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
    const bool real_row = r < rows;
    const int p_row = p_first + (real_row ? r : rows - 1);  // padding rows mirror the last row
    const size_t q_row = (size_t)(q0 + i0 + (real_row ? r : 0)) * a.H + h;

    // stage this row of Q into the swizzled K-major tile
    {
      const uint4 *src = reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(a.q) + q_row * D);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint4 v = real_row ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4 *>(sm + Sh::kQOff + (c >> 3) * kRegionBytes + r * 128 +
                                   (((c & 7) ^ (r & 7)) << 4)) = v;
      }
      fence_proxy_async_shared();
      mbar_arrive(q_full);
    }

    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      ok = mbar_wait_bounded(s_full, j & 1);
      if (!__all_sync(0xffffffffu, ok) || *(volatile int *)abort_flag) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int t0 = j * kPfTile;
      // pass 1: the row max of the scaled scores of tokens t <= p_row
      float mx = -INFINITY;
#pragma unroll
      for (int cc = 0; cc < kPfTile / 32; ++cc) {
        float v[32];
        tmem_ld32(tmem_s + lane_off + 32 * cc, v);
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (t0 + 32 * cc + i <= p_row) mx = fmaxf(mx, v[i] * a.scale_log2);
      }
      // the reference max moves only when the row max exceeds it by 2^8
      const float m_new = (mx > m_used + 8.f) ? mx : m_used;
      const float alpha = fast_exp2(m_used - m_new);  // 0 on the first tile
      const bool rescale = __any_sync(0xffffffffu, m_new != m_used) && j > 0;
      l *= alpha;
      m_used = m_new;

      // P_{j-1} . V_{j-1} must be done: P's tile is rewritten and O is read
      if (j > 0) {
        ok = mbar_wait_bounded(o_done, (j - 1) & 1);
        if (!__all_sync(0xffffffffu, ok)) break;
        tc_fence_after();
        if (rescale) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            float v[32];
            tmem_ld32(tmem_o + lane_off + 32 * c, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= alpha;
            tmem_st32(tmem_o + lane_off + 32 * c, v);
          }
        }
      }
      // the last tile's V rows past the context are zeroed (they may hold
      // anything, and 0 * NaN would poison the product)
      if (t0 + kPfTile > n) {
        ok = mbar_wait_bounded(&kv_full[j & 1], (j >> 1) & 1);
        if (!__all_sync(0xffffffffu, ok)) break;
        if (r >= n - t0) {
          uint8_t *vrow = sm + Sh::kKVOff + (j & 1) * 2 * Sh::kTileBytes + Sh::kTileBytes + r * 128;
#pragma unroll
          for (int g = 0; g < Sh::kRegions; ++g)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4 *>(vrow + g * kRegionBytes + c * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      // pass 2: P = 2^(s - m) (0 past p_row), rounded to the input type, into
      // the swizzled K-major P tile; l sums the rounded weights
#pragma unroll
      for (int cc = 0; cc < kPfTile / 32; ++cc) {
        float v[32];
        tmem_ld32(tmem_s + lane_off + 32 * cc, v);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int t = t0 + 32 * cc + 2 * i;
          const float e0 = t <= p_row ? fast_exp2(v[2 * i] * a.scale_log2 - m_used) : 0.f;
          const float e1 = t + 1 <= p_row ? fast_exp2(v[2 * i + 1] * a.scale_log2 - m_used) : 0.f;
          pk[i] = PackPair<T>::run(e0, e1, l);
        }
        uint8_t *prow = sm + Sh::kPOff + (cc >> 1) * kRegionBytes + r * 128;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          const int chunk = (cc & 1) * 4 + c4;
          *reinterpret_cast<uint4 *>(prow + ((chunk ^ (r & 7)) << 4)) =
              make_uint4(pk[4 * c4], pk[4 * c4 + 1], pk[4 * c4 + 2], pk[4 * c4 + 3]);
        }
      }
      fence_proxy_async_shared();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    if (ok) ok = mbar_wait_bounded(o_done, (ntiles - 1) & 1);
    if (__all_sync(0xffffffffu, ok) && !*(volatile int *)abort_flag) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      T *orow = reinterpret_cast<T *>(a.out) + q_row * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float v[32];
        tmem_ld32(tmem_o + lane_off + 32 * c, v);
        if (real_row) {
          uint32_t pk[16];
          float unused = 0.f;
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[i] = PackPair<T>::run(v[2 * i] * inv_l, v[2 * i + 1] * inv_l, unused);
          uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * c);
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4)
            dst[c4] = make_uint4(pk[4 * c4], pk[4 * c4 + 1], pk[4 * c4 + 2], pk[4 * c4 + 3]);
        }
      }
    } else if (lane == 0) {
      raise_flag(a.err, PKV_FLAG_TIMEOUT);
      *(volatile int *)abort_flag = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, Sh::kTmemCols);
}

// ---------------------------------------------------------------- host side

template <int D, typename T>
static pkv_status launch_prefill_t(const PrefillArgs &a, const CUtensorMap &mk,
                                   const CUtensorMap &mv, cudaStream_t stream) {
  auto kern = pkv_prefill_tc_kernel<D, T>;
  static int configured[64] = {0};
  if (!allow_smem(kern, PfShape<D>::kSmem, configured)) return PKV_ERR_CUDA;
  dim3 grid(a.H, a.q_tiles, a.B);
  kern<<<grid, kPfThreads, PfShape<D>::kSmem, stream>>>(mk, mv, a);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status launch_prefill_tc(void *out, const void *q, const void *k_cache, const void *v_cache,
                             const int32_t *tables, const int32_t *cu_q, const int32_t *lens,
                             int B, int H, int KVH, int D, int bs, int max_blocks,
                             long long num_blocks, float scale, pkv_dtype dt, int q_tiles,
                             int *err, cudaStream_t stream) {
  CUtensorMap mk, mv;
  if (!encode_cache_map(&mk, k_cache, dt, num_blocks, bs, KVH, D) ||
      !encode_cache_map(&mv, v_cache, dt, num_blocks, bs, KVH, D))
    return PKV_ERR_CUDA;
  PrefillArgs a;
  memset(&a, 0, sizeof a);
  a.out = out;
  a.q = q;
  a.tables = tables;
  a.cu_q = cu_q;
  a.lens = lens;
  a.err = err;
  a.num_blocks = num_blocks;
  a.B = B;
  a.H = H;
  a.KVH = KVH;
  a.D = D;
  a.G = H / KVH;
  a.bs = bs;
  a.max_blocks = max_blocks;
  a.q_tiles = q_tiles;
  a.scale_log2 = scale * kLog2e;
  const bool bf = dt == PKV_BF16;
  if (D == 128) return bf ? launch_prefill_t<128, __nv_bfloat16>(a, mk, mv, stream)
                          : launch_prefill_t<128, __half>(a, mk, mv, stream);
  if (D == 64) return bf ? launch_prefill_t<64, __nv_bfloat16>(a, mk, mv, stream)
                         : launch_prefill_t<64, __half>(a, mk, mv, stream);
  return PKV_ERR_UNSUPPORTED;
}

}  // namespace pkv
