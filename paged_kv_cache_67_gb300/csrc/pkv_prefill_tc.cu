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
// Work decomposition.  CTA = (query head, 256 queries, sequence), the
// latest (heaviest) query tiles first; 10 warps:
//   warp 0     producer: per 64-token KV tile, 16 lanes issue one tiled TMA
//              load each (a 16-token chunk of one 64-column region of K or V
//              of this KV head, 128-byte swizzle) into a 3-stage ring;
//   warp 1     MMA issuer (one thread), alternating between the two query
//              tiles: S_g = Q_g . K^T (M = 128, N = 64 tokens, fp32 in tensor
//              memory), then O_g += P_g . V (N = D); the next tile's S_g is
//              issued before this tile's P_g . V, so while one warpgroup
//              works on its scores the tensor core serves the other;
//   warps 2-5, 6-9  two softmax warpgroups, one per 128-query tile, one query
//              row per thread (its tensor-memory lane): stage Q, then per KV
//              tile read S, mask (causal, end of context), update the running
//              max -- the reference max moves only when the row max grows by
//              more than 2^8, and only then is the O row in tensor memory
//              rescaled -- write P = 2^(s - m) as bf16/fp16 into a swizzled
//              shared tile, and finally O / l.
// Every wait on an mbarrier is bounded; on time-out the CTA raises
// PKV_FLAG_TIMEOUT, lets its copies and products land (bounded) and exits.
#include <string.h>

#include <type_traits>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_tcgen05.cuh"

namespace pkv {

constexpr int kPfRows = 128;     // query rows per softmax warpgroup (MMA M)
constexpr int kPfGroups = 2;     // query tiles per CTA, one softmax warpgroup each
constexpr int kPfTile = 128;     // KV tokens per tile
constexpr int kPfStages = 2;     // K/V ring depth
constexpr int kPfWarps = 2 + 4 * kPfGroups;
constexpr int kPfThreads = 32 * kPfWarps;
constexpr int kQRegion = kPfRows * 128;   // 128 query rows x 64 elements of 16 bits
constexpr int kKVRegion = kPfTile * 128;  // 128 token rows x 64 elements

struct PrefillArgs {
  void *out;
  const void *q;
  const int32_t *tables;
  const int32_t *cu_q;
  const int32_t *lens;
  int *err;
  long long num_blocks;
  int B, H, KVH, D, G, bs, max_blocks;
  int q_tiles;        // 256-query tiles per sequence served (from the host's bound on qlen)
  float scale_log2;   // scale * log2(e)
};

template <int D>
struct PfShape {
  static constexpr int kRegions = D / 64;
  static constexpr int kQBytes = kRegions * kQRegion;           // one warpgroup's query tile
  static constexpr int kKVBytes = kRegions * kKVRegion;         // one K (or V) tile
  static constexpr int kQOff = 0;                               // [group]
  static constexpr int kKVOff = kQOff + kPfGroups * kQBytes;    // [stage][K, V]
  static constexpr int kBarOff = kKVOff + kPfStages * 2 * kKVBytes;
  static constexpr int kSmem = kBarOff + 256 + 1024;            // + alignment slack
  // tensor memory, 256 columns per group: S (128 fp32 columns; P, 128
  // tokens as 64 packed columns, is written over its first half once S is
  // read), O (D fp32 columns)
  static constexpr uint32_t kTmemCols = 512;
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

// Blackwell paired fp32 arithmetic and the three-input max.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<unsigned long long *>(&a)), "l"(*reinterpret_cast<unsigned long long *>(&b)),
        "l"(*reinterpret_cast<unsigned long long *>(&c)));
  return *reinterpret_cast<float2 *>(&d);
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<unsigned long long *>(&a)), "l"(*reinterpret_cast<unsigned long long *>(&b)));
  return *reinterpret_cast<float2 *>(&d);
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

template <typename T>
struct PackPair;
template <>
struct PackPair<__nv_bfloat16> {
  // two fp32 -> packed bf16 pair (round to nearest even)
  __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
  }
};
template <>
struct PackPair<__half> {
  __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
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
  uint64_t *k_full = bars + 1;     // [kPfStages]: K and V of a stage arrive and are
  uint64_t *v_full = bars + 3;     // [kPfStages]  released separately, so the next
  uint64_t *k_empty = bars + 5;    // [kPfStages]  keys are fetched as soon as the
  uint64_t *v_empty = bars + 7;    // [kPfStages]  scores that read a slot are done
  uint64_t *s_full = bars + 9;     // [kPfGroups]: S of the group's current tile
  uint64_t *p_full = bars + 11;    // [kPfGroups]: P of the group's current tile
  uint64_t *o_done = bars + 13;    // [kPfGroups]: the group's last P . V done
  uint64_t *mma_done = bars + 15;
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 16);
  int *abort_flag = reinterpret_cast<int *>(bars + 17);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.x;
  constexpr int kCtaRows = kPfGroups * kPfRows;

  // ---- checks of the whole batch, by one warp of one CTA
  auto seq_ok = [&](int bb, int ql) {
    const int nn = __ldg(a.lens + bb);
    return ql >= 0 && nn >= ql && (long long)nn <= (long long)a.max_blocks * a.bs;
  };
  if (h == 0 && blockIdx.y == 0 && warp == 0) {
    int bad = 0, over = 0;
    for (int bb = lane; bb < a.B; bb += 32) {
      const int ql = __ldg(a.cu_q + bb + 1) - __ldg(a.cu_q + bb);
      bad |= !seq_ok(bb, ql);
      over |= ql > a.q_tiles * kCtaRows;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) raise_flag(a.err, PKV_FLAG_QUERY_LEN);
    if (__any_sync(0xffffffffu, over) && lane == 0) raise_flag(a.err, PKV_FLAG_QUERY_OVER_HINT);
  }

  // ---- which (sequence, 256-query tile) this CTA serves: the k-th of the
  // real pairs in the order (tile index descending, then sequence), so the
  // latest (heaviest) tiles start first and no CTA is launched for nothing.
  // Every warp finds it on its own (uniform, before any barrier).
  int b = -1, qt = 0;
  {
    int k = blockIdx.y;
    if (a.B <= 32) {  // one sequence per lane: the query counts stay in registers
      const int ql = lane < a.B ? __ldg(a.cu_q + lane + 1) - __ldg(a.cu_q + lane) : 0;
      for (int t = a.q_tiles - 1; t >= 0; --t) {
        const unsigned m = __ballot_sync(0xffffffffu, ql > t * kCtaRows);
        const int c = __popc(m);
        if (k < c) {
          b = (int)__fns(m, 0, k + 1);  // position of the k-th set bit
          qt = t;
          break;
        }
        k -= c;
      }
    } else {
      for (int t = a.q_tiles - 1; t >= 0 && b < 0; --t) {
        int cnt = 0;
        for (int base = 0; base < a.B; base += 32) {
          const int bb = base + lane;
          const bool has = bb < a.B && __ldg(a.cu_q + bb + 1) - __ldg(a.cu_q + bb) > t * kCtaRows;
          const unsigned m = __ballot_sync(0xffffffffu, has);
          const int c = __popc(m);
          if (k < cnt + c) {
            b = base + (int)__fns(m, 0, k - cnt + 1);
            qt = t;
            break;
          }
          cnt += c;
        }
        if (b < 0) k -= cnt;
      }
    }
  }
  if (b < 0) return;
  const int q0 = __ldg(a.cu_q + b), qlen = __ldg(a.cu_q + b + 1) - q0;
  const int n = __ldg(a.lens + b);
  if (!seq_ok(b, qlen)) return;
  const int i0 = qt * kCtaRows;
  const int rows = min(kCtaRows, qlen - i0);
  const int p_first = n - qlen + i0;               // position of query row 0
  // tiles each warpgroup needs: up to the position of its last real row
  const int rows1 = rows - kPfRows;                // rows of the second tile (may be <= 0)
  const int ntiles0 = (p_first + min(kPfRows, rows) - 1) / kPfTile + 1;
  const int ntiles1 = rows1 > 0 ? (p_first + kPfRows + rows1 - 1) / kPfTile + 1 : 0;
  const int ntiles = max(ntiles0, ntiles1);
  auto tiles_of = [&](int g) { return g == 0 ? ntiles0 : ntiles1; };
  const int kvh = h / a.G;

  if (tid == 0) {
    mbar_init(q_full, 4 * 32 * kPfGroups);
    for (int s = 0; s < kPfStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int g = 0; g < kPfGroups; ++g) {
      mbar_init(&s_full[g], 1);
      mbar_init(&p_full[g], 128);
      mbar_init(&o_done[g], 1);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_holder, Sh::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  constexpr bool bf16 = std::is_same<T, __nv_bfloat16>::value;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // per tile: the K boxes (one per lane) once the keys of tile j-2 are no
    // longer read, then the V boxes once the values of tile j-2 are not
    const int per_tensor = 8 * Sh::kRegions;     // boxes of K (or V) per 128-token tile
    const int region = (lane % per_tensor) >> 3, chunk = lane & 7;
    int issued = 0;
    bool ok = true;
    for (int j = 0; j < ntiles && ok; ++j) {
      const int stage = j % kPfStages;
      const int tok0 = j * kPfTile;
      const int valid_chunks = min(8, (n - tok0 + 15) >> 4);
      const uint32_t bytes = (uint32_t)(valid_chunks * Sh::kRegions * 2048);
      // the tile's table entries: lane c < 8 loads chunk c's, broadcast to the
      // lanes that issue that chunk's boxes (K and V, every region)
      int phys = 0;
      if (lane < valid_chunks) {
        const int lb = (tok0 + 16 * lane) / a.bs;
        phys = __ldg(a.tables + (size_t)b * a.max_blocks + lb);
        if (phys < 0 || (long long)phys >= a.num_blocks) {
          raise_flag(a.err, PKV_FLAG_BLOCK_OUT_OF_RANGE);
          phys = 0;
        }
      }
      phys = __shfl_sync(0xffffffffu, phys, chunk);
      for (int v = 0; v < 2 && ok; ++v) {
        if (j >= kPfStages) {
          const bool got = mbar_wait_bounded(v ? &v_empty[stage] : &k_empty[stage],
                                             (j / kPfStages - 1) & 1);
          if (!__all_sync(0xffffffffu, got) || *(volatile int *)abort_flag) {
            if (lane == 0) {
              raise_flag(a.err, PKV_FLAG_TIMEOUT);
              *(volatile int *)abort_flag = 1;
            }
            ok = false;
            break;
          }
        }
        uint64_t *full = v ? &v_full[stage] : &k_full[stage];
        if (lane == 0) mbar_arrive_expect_tx(full, bytes);
        __syncwarp();
        if (lane < per_tensor && chunk < valid_chunks) {
          const int t = tok0 + 16 * chunk;
          const int lb = t / a.bs;
          uint8_t *dst = sm + Sh::kKVOff + stage * 2 * Sh::kKVBytes + (v ? Sh::kKVBytes : 0) +
                         region * kKVRegion + chunk * 2048;
          tma_load_4d_keep(dst, v ? &tmV : &tmK, full, region * 64, kvh, t - lb * a.bs, phys);
        }
      }
      if (ok) ++issued;
    }
    // the last fills land before the CTA can end (bounded)
    for (int j = max(0, issued - kPfStages); j < issued; ++j) {
      mbar_wait_bounded(&k_full[j % kPfStages], (j / kPfStages) & 1);
      mbar_wait_bounded(&v_full[j % kPfStages], (j / kPfStages) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = umma_idesc_f16(128, kPfTile, bf16, false);
      const uint32_t idesc_o = umma_idesc_f16(128, D, bf16, true);
      auto kv_base = [&](int j, bool v) {
        return smem_u32(sm + Sh::kKVOff + (j % kPfStages) * 2 * Sh::kKVBytes +
                        (v ? Sh::kKVBytes : 0));
      };
      auto issue_s = [&](int g, int j) {  // S_g = Q_g . K_j^T over D in 16-wide steps
        const uint32_t qb = smem_u32(sm + Sh::kQOff + g * Sh::kQBytes), kb = kv_base(j, false);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          umma_f16(tmem + 256 * g, umma_desc_sw128(qb + (k >> 2) * kQRegion + (k & 3) * 32, 16, 1024),
                   umma_desc_sw128(kb + (k >> 2) * kKVRegion + (k & 3) * 32, 16, 1024), idesc_s,
                   k > 0);
        umma_commit(&s_full[g]);
      };
      auto issue_pv = [&](int g, int j) {  // O_g += P_g . V_j, P from tensor memory
        const uint32_t vb = kv_base(j, true);
#pragma unroll
        for (int k = 0; k < kPfTile / 16; ++k)
          umma_f16_tmem_a(tmem + 256 * g + 128, tmem + 256 * g + 8 * k,
                          umma_desc_sw128(vb + k * 2048, kKVRegion, 1024), idesc_o, (j > 0 || k > 0));
      };
      // S of the first tile of both groups; then per tile and group, as soon
      // as P_g(j) arrives: P_g(j) . V_j, then S_g(j+1).  The products of one
      // thread run in issue order, so S_g(j+1) -- written over P_g(j) --
      // starts after P_g(j) . V_j has read it, and the commit that signals
      // S_g(j+1) also covers P_g(j) . V_j (O is final for tile j when the
      // softmax sees S_g(j+1)).  One commit per group and tile, one per
      // released K and V slot; O's completion is signalled once, at the end.
      bool ok = mbar_wait_bounded(q_full, 0) && mbar_wait_bounded(&k_full[0], 0);
      if (ok) {
        tc_fence_after();
        for (int g = 0; g < kPfGroups; ++g)
          if (tiles_of(g) > 0) issue_s(g, 0);
        umma_commit(&k_empty[0]);
      }
      for (int j = 0; ok && j < ntiles; ++j) {
        bool v_ready = false, k_ready = false;
        for (int g = 0; g < kPfGroups && ok; ++g) {
          if (j >= tiles_of(g)) continue;
          ok = mbar_wait_bounded(&p_full[g], j & 1) && !*(volatile int *)abort_flag;
          if (!ok) break;
          if (!v_ready) {
            ok = mbar_wait_bounded(&v_full[j % kPfStages], (j / kPfStages) & 1);
            if (!ok) break;
            v_ready = true;
          }
          tc_fence_after();
          issue_pv(g, j);
          if (j + 1 < tiles_of(g)) {
            if (!k_ready) {
              ok = mbar_wait_bounded(&k_full[(j + 1) % kPfStages], ((j + 1) / kPfStages) & 1);
              if (!ok) break;
              k_ready = true;
            }
            issue_s(g, j + 1);
          } else {
            umma_commit(&o_done[g]);  // the group's last product
          }
        }
        if (!ok) break;
        umma_commit(&v_empty[j % kPfStages]);
        if (j + 1 < ntiles) umma_commit(&k_empty[(j + 1) % kPfStages]);
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
    const int g = (warp - 2) >> 2;                      // warpgroup = query tile
    const int quarter = warp & 3;
    const int r = 32 * quarter + lane;                  // row in the tile = tensor-memory lane
    const int rr = g * kPfRows + r;                     // row in the CTA
    const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
    const uint32_t tmem_o = tmem + 256 * g + 128;
    const bool real_row = rr < rows;
    const int p_row = p_first + (real_row ? rr : rows - 1);  // padding rows mirror the last row
    const size_t q_row = (size_t)(q0 + i0 + (real_row ? rr : 0)) * a.H + h;
    const int my_tiles = tiles_of(g);

    // stage this row of Q into the group's swizzled K-major tile
    {
      const uint4 *src = reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(a.q) + q_row * D);
      uint8_t *qt_base = sm + Sh::kQOff + g * Sh::kQBytes + r * 128;
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint4 v = real_row ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4 *>(qt_base + (c >> 3) * kQRegion + (((c & 7) ^ (r & 7)) << 4)) = v;
      }
      fence_proxy_async_shared();
      mbar_arrive(q_full);
    }

    // scores are kept raw; with scale > 0 the max commutes with the scale
    // and one fused multiply-add per pair gives s * scale * log2(e) - m
    const float sl2 = a.scale_log2;
    const bool pos_scale = sl2 > 0.f;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < my_tiles; ++j) {
      ok = mbar_wait_bounded(&s_full[g], j & 1);
      if (!__all_sync(0xffffffffu, ok) || *(volatile int *)abort_flag) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int t0 = j * kPfTile;
      const uint32_t tmem_sp = tmem + 256 * g + lane_off;  // S, then P over its first half
      // pass 1: row max (scores raw when scale > 0: the max commutes)
      float mx = -INFINITY;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int tb = t0 + 64 * hf;
        float s[64];
        tmem_ld64(tmem_sp + 64 * hf, s);
        if (!pos_scale) {
#pragma unroll
          for (int i = 0; i < 64; ++i) s[i] *= sl2;
        }
        if (tb + 63 > p_row) {
#pragma unroll
          for (int i = 0; i < 64; ++i) s[i] = tb + i <= p_row ? s[i] : -INFINITY;
        }
#pragma unroll
        for (int i = 0; i < 64; i += 2) mx = max3f(mx, s[i], s[i + 1]);
      }
      if (pos_scale) mx *= sl2;
      // the reference max moves only when the row max exceeds it by 2^8
      const float m_new = (mx > m_used + 8.f) ? mx : m_used;
      const float alpha = fast_exp2(m_used - m_new);  // 0 on the first tile
      const bool rescale = __any_sync(0xffffffffu, m_new != m_used) && j > 0;
      l *= alpha;
      m_used = m_new;
      // O is final for tile j-1 here: the commit that signalled S_g(j) also
      // covers P_g(j-1) . V, issued before it
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
      // the tile's V rows past the context are zeroed (they may hold
      // anything, and 0 * NaN would poison the product)
      const bool past_end = t0 + kPfTile > n;
      if (past_end) {
        ok = mbar_wait_bounded(&v_full[j % kPfStages], (j / kPfStages) & 1);
        if (!__all_sync(0xffffffffu, ok)) break;
        if (r >= n - t0) {
          uint8_t *vrow = sm + Sh::kKVOff + (j % kPfStages) * 2 * Sh::kKVBytes + Sh::kKVBytes + r * 128;
#pragma unroll
          for (int rg = 0; rg < Sh::kRegions; ++rg)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4 *>(vrow + rg * kKVRegion + c * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      // pass 2: P = 2^(s * scale * log2(e) - m), rounded to the input type,
      // two tokens per column over S columns already read (P columns
      // 32 hf .. +31 lie below S columns 64 hf read in this or the earlier
      // step); l sums the unrounded weights
      const float mul = pos_scale ? sl2 : 1.f;
      float2 lsum = make_float2(0.f, 0.f);
#pragma unroll 1
      for (int hf = 0; hf < 2; ++hf) {   // 64 tokens at a time: P columns 32 hf .. +31
        const int tb = t0 + 64 * hf;
        float s[64];
        tmem_ld64(tmem_sp + 64 * hf, s);
        if (!pos_scale) {
#pragma unroll
          for (int i = 0; i < 64; ++i) s[i] *= sl2;
        }
        if (tb + 63 > p_row) {
#pragma unroll
          for (int i = 0; i < 64; ++i) s[i] = tb + i <= p_row ? s[i] : -INFINITY;
        }
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float2 x = ffma2(make_float2(s[2 * i], s[2 * i + 1]), make_float2(mul, mul),
                           make_float2(-m_used, -m_used));
          x.x = fast_exp2(x.x);
          x.y = fast_exp2(x.y);
          lsum = fadd2(lsum, x);
          pk[i] = PackPair<T>::pack(x.x, x.y);
        }
        tmem_st32u(tmem_sp + 32 * hf, pk);
      }
      l += lsum.x + lsum.y;
      // the zeroed V rows (generic writes) before the product reads them
      if (past_end) fence_proxy_async_shared();
      tc_fence_before();
      mbar_arrive(&p_full[g]);
    }
    if (ok && my_tiles > 0) ok = mbar_wait_bounded(&o_done[g], 0);
    if (my_tiles > 0 && __all_sync(0xffffffffu, ok) && !*(volatile int *)abort_flag) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      T *orow = reinterpret_cast<T *>(a.out) + q_row * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float v[32];
        tmem_ld32(tmem_o + lane_off + 32 * c, v);
        if (real_row) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[i] = PackPair<T>::pack(v[2 * i] * inv_l, v[2 * i + 1] * inv_l);
          uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * c);
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4)
            dst[c4] = make_uint4(pk[4 * c4], pk[4 * c4 + 1], pk[4 * c4 + 2], pk[4 * c4 + 3]);
        }
      }
    } else if (my_tiles > 0 && lane == 0) {
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
                                   const CUtensorMap &mv, int ctas_per_head, cudaStream_t stream) {
  auto kern = pkv_prefill_tc_kernel<D, T>;
  static int configured[64] = {0};
  if (!allow_smem(kern, PfShape<D>::kSmem, configured)) return PKV_ERR_CUDA;
  dim3 grid(a.H, ctas_per_head, 1);
  kern<<<grid, kPfThreads, PfShape<D>::kSmem, stream>>>(mk, mv, a);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status launch_prefill_tc(void *out, const void *q, const void *k_cache, const void *v_cache,
                             const int32_t *tables, const int32_t *cu_q, const int32_t *lens,
                             int B, int H, int KVH, int D, int bs, int max_blocks,
                             long long num_blocks, float scale, pkv_dtype dt, int q_tiles,
                             int ctas_per_head, int *err, cudaStream_t stream) {
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
  if (D == 128) return bf ? launch_prefill_t<128, __nv_bfloat16>(a, mk, mv, ctas_per_head, stream)
                          : launch_prefill_t<128, __half>(a, mk, mv, ctas_per_head, stream);
  if (D == 64) return bf ? launch_prefill_t<64, __nv_bfloat16>(a, mk, mv, ctas_per_head, stream)
                         : launch_prefill_t<64, __half>(a, mk, mv, ctas_per_head, stream);
  return PKV_ERR_UNSUPPORTED;
}

}  // namespace pkv
