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
// Work decomposition.  A work item is (query head, sequence, 256 queries):
// two 128-query tiles that share every K/V tile.  Items are numbered by
// their KV tile count, most first (a chunk on a long cached prefix is heavy
// even at its first query tile); the grid is persistent (at most one CTA per
// SM) and CTA c takes item c, then the next unclaimed one from a counter in
// device memory, so the tensor memory stays allocated, the next item's
// queries and first K/V tiles load while the current one finishes, and the
// epilogue of one item overlaps the first products of the next.  11 warps:
//   warp 10    scheduler: claims items, publishes each (its geometry
//              worked out once) to the CTA through a two-slot ring as soon
//              as a slot is free, and loads the item's two query tiles (TMA,
//              128-byte swizzle) once the products that read the previous
//              ones are done;
//   warp 0     producer: per item and 128-token KV tile issues the tiled
//              TMA loads of K and of V (16-token chunks of 64-column
//              regions, 128-byte swizzle) into a two-stage ring that runs on
//              across items;
//   warp 1     MMA issuer (one thread): per group g (query tile),
//              S_g = Q_g . K^T (M = 128, N = 128 tokens, fp32 in tensor
//              memory); once the softmax wrote P_g over S_g, O_g += P_g . V
//              (P from tensor memory, N = D), and right behind it the next
//              tile's S_g; the products of one thread run in issue order;
//              group 0 starts its next item while group 1 ends the current
//              one;
//   warps 2-5, 6-9  two softmax warpgroups, one per query tile, one query
//              row per thread (its tensor-memory lane): per KV tile read S,
//              mask (causal, end of context), update the running max -- the
//              reference max moves only when the row max grows by more than
//              2^8, and only then is the O row in tensor memory rescaled --
//              write P = 2^(s - m) as bf16/fp16 over S, and after the item's
//              last tile store O / l.
// Every wait on an mbarrier is bounded; on time-out the CTA raises
// PKV_FLAG_TIMEOUT, lets its copies and products land (bounded) and exits.
#include <string.h>

#include <atomic>
#include <type_traits>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_tcgen05.cuh"

namespace pkv {

constexpr int kPfRows = 128;     // query rows per softmax warpgroup (MMA M)
constexpr int kPfGroups = 2;     // query tiles per item, one softmax warpgroup each
constexpr int kPfTile = 128;     // KV tokens per tile
constexpr int kPfStages = 2;     // K/V ring depth
constexpr int kSchedWarp = 2 + 4 * kPfGroups;  // after producer, MMA and softmax warps
constexpr int kPfWarps = 3 + 4 * kPfGroups;
constexpr int kPfThreads = 32 * kPfWarps;
constexpr int kQRegion = kPfRows * 128;   // 128 query rows x 64 elements of 16 bits
constexpr int kKVRegion = kPfTile * 128;  // 128 token rows x 64 elements
constexpr int kItemReaders = 2 + 4 * kPfGroups;  // producer, MMA thread, one lane per softmax warp
constexpr int kSchedSlots = 1024;         // work counters, one per launch in flight

// Work counters of the persistent launches: slot s holds (next item to claim
// beyond the first gridDim.x, CTAs finished); the last CTA of a launch puts
// both back to zero, so a slot is ready again for the launch after.
__device__ unsigned g_pf_sched[2 * kSchedSlots];

struct PrefillArgs {
  void *out;
  const int32_t *tables;
  const int32_t *cu_q;
  const int32_t *lens;
  int *err;
  unsigned *sched;    // this launch's (next, done) counters
  long long num_blocks;
  int B, H, KVH, D, G, bs, max_blocks;
  int q_tiles;        // 256-query tiles per sequence served (from the host's bound on qlen)
  float scale_log2;   // scale * log2(e)
};

template <int D>
struct PfShape {
  static constexpr int kRegions = D / 64;
  static constexpr int kQBytes = kRegions * kQRegion;           // one group's query tile
  static constexpr int kKVBytes = kRegions * kKVRegion;         // one K (or V) tile
  static constexpr int kQOff = 0;                               // [group]
  static constexpr int kKVOff = kQOff + kPfGroups * kQBytes;    // [stage][K, V]
  static constexpr int kBarOff = kKVOff + kPfStages * 2 * kKVBytes;
  static constexpr int kSmem = kBarOff + 1024 + 1024;           // barriers, item ring, claim table; + alignment slack
  // tensor memory, 256 columns per group: S (128 fp32 columns; P, 128
  // tokens as 64 packed columns, is written over its first half once S is
  // read), O (D fp32 columns)
  static constexpr uint32_t kTmemCols = 512;
};

// Tiled TMA loads global -> shared with the default L2 policy (K/V tiles
// are read again by the other heads of the group and later items).
__device__ __forceinline__ void tma_load_4d_keep(void *dst, const CUtensorMap *map, uint64_t *bar,
                                                 int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
      "r"(c3)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_keep(void *dst, const CUtensorMap *map, uint64_t *bar,
                                                 int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Whether the phase with the given parity has completed (never waits).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// The three-input max (the paired fp32 arithmetic is in pkv_device.cuh).
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

// One work item as every role sees it (published in shared memory by the
// scheduler warp).  kind: 1 work, 0 skipped (a sequence whose lengths are
// invalid), -1 no more items.
struct __align__(16) PfItem {
  int kind, h, b, qt;
  int q0, qlen, n, rows;   // q0: the item's first query row
  int p_first;             // position of the item's query row 0
  int nt[kPfGroups];       // KV tiles each query tile needs (up to its last real row)
  int ntiles;
};
static_assert(sizeof(PfItem) == 48, "three 16-byte words");

__device__ __forceinline__ int nt_of(const PfItem &it, int g) { return g == 0 ? it.nt[0] : it.nt[1]; }

__device__ __forceinline__ bool pf_seq_ok(const PrefillArgs &a, int bb, int ql) {
  const int nn = __ldg(a.lens + bb);
  return ql >= 0 && nn >= ql && (long long)nn <= (long long)a.max_blocks * a.bs;
}

__device__ __forceinline__ PfItem pf_item(const PrefillArgs &a, int kind, int h, int b, int qt) {
  PfItem it;
  memset(&it, 0, sizeof it);
  it.kind = kind;
  it.h = h;
  it.b = b;
  it.qt = qt;
  if (kind != 1) return it;
  it.q0 = __ldg(a.cu_q + b);
  it.qlen = __ldg(a.cu_q + b + 1) - it.q0;
  it.n = __ldg(a.lens + b);
  const int i0 = qt * kPfGroups * kPfRows;
  it.rows = min(kPfGroups * kPfRows, it.qlen - i0);
  it.p_first = it.n - it.qlen + i0;
  const int rows1 = it.rows - kPfRows;            // rows of the second tile (may be <= 0)
  it.nt[0] = (it.p_first + min(kPfRows, it.rows) - 1) / kPfTile + 1;
  it.nt[1] = rows1 > 0 ? (it.p_first + kPfRows + rows1 - 1) / kPfTile + 1 : 0;
  it.ntiles = max(it.nt[0], it.nt[1]);
  it.q0 += i0;
  return it;
}

// The k-th (sequence, 256-query tile) pair in the order (tile index
// descending, then sequence): *b = -1 past the last.  One warp, uniform.
__device__ __forceinline__ void pf_pair(const PrefillArgs &a, int k, int lane, int *b_out,
                                        int *qt_out) {
  constexpr int kCtaRows = kPfGroups * kPfRows;
  int b = -1, qt = 0;
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
  *b_out = b;
  *qt_out = qt;
}

template <int D, typename T>
__global__ void __launch_bounds__(kPfThreads, 1)
    pkv_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                          const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const PrefillArgs a) {
  using Sh = PfShape<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + Sh::kBarOff);
  uint64_t *k_full = bars + 0;      // [kPfStages]: K and V of a stage arrive and are
  uint64_t *v_full = bars + 2;      // [kPfStages]  released separately, so the next
  uint64_t *k_empty = bars + 4;     // [kPfStages]  keys are fetched as soon as the
  uint64_t *v_empty = bars + 6;     // [kPfStages]  scores that read a slot are done
  uint64_t *q_full = bars + 8;      // [kPfGroups]: the group's query tile landed
  uint64_t *q_empty = bars + 10;    // [kPfGroups]: the group's last S of an item done
  uint64_t *s_full = bars + 12;     // [kPfGroups]: S of the group's current tile
  uint64_t *p_full = bars + 14;     // [kPfGroups]: P of the group's current tile
  uint64_t *o_done = bars + 16;     // [kPfGroups]: the group's last P . V of an item done
  uint64_t *item_full = bars + 18;  // [2]: an item published
  uint64_t *item_empty = bars + 20; // [2]: every role has read it
  uint64_t *mma_done = bars + 22;
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 23);
  int *abort_flag = reinterpret_cast<int *>(bars + 24);
  PfItem *items = reinterpret_cast<PfItem *>(bars + 26);  // [2], 16-byte aligned

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (tid == 0) {
    for (int s = 0; s < kPfStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int g = 0; g < kPfGroups; ++g) {
      mbar_init(&q_full[g], 1);
      mbar_init(&q_empty[g], 1);
      mbar_init(&s_full[g], 1);
      mbar_init(&p_full[g], 128);
      mbar_init(&o_done[g], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&item_full[s], 1);
      mbar_init(&item_empty[s], kItemReaders);
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
  constexpr int kCtaRows = kPfGroups * kPfRows;

  auto abort_cta = [&]() {
    raise_flag(a.err, PKV_FLAG_TIMEOUT);
    *(volatile int *)abort_flag = 1;
  };
  auto aborted = [&]() { return *(volatile int *)abort_flag != 0; };

  if (warp == kSchedWarp) {
    // ------------------------------------------------------------ scheduler
    // the pairs there are, and (one CTA) the checks of the whole batch
    int pairs = 0, bad = 0, over = 0;
    for (int bb = lane; bb < a.B; bb += 32) {
      const int ql = __ldg(a.cu_q + bb + 1) - __ldg(a.cu_q + bb);
      if (ql > 0) pairs += min(a.q_tiles, (ql + kCtaRows - 1) / kCtaRows);
      if (blockIdx.x == 0) {
        bad |= !pf_seq_ok(a, bb, ql);
        over |= ql > a.q_tiles * kCtaRows;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) pairs += __shfl_xor_sync(0xffffffffu, pairs, o);
    if (__any_sync(0xffffffffu, bad) && lane == 0) raise_flag(a.err, PKV_FLAG_QUERY_LEN);
    if (__any_sync(0xffffffffu, over) && lane == 0) raise_flag(a.err, PKV_FLAG_QUERY_OVER_HINT);
    const unsigned total = (unsigned)pairs * (unsigned)a.H;
    // The claim order: pairs (sequence, 256-query tile) by their KV tiles,
    // most first (a chunk on a long cached prefix is heavy even at tile 0),
    // then sequence and tile; each pair's heads one after another.  The
    // first item number of each tile-count class comes from a histogram in
    // shared memory (64 classes, 63 tiles and more together); batches with
    // more than 4096 (sequence, tile) slots keep the order of pf_pair.
    auto pair_tiles = [&](int ql, int n, int t) {
      const int i0 = t * kCtaRows;
      const int rows = min(kCtaRows, ql - i0);
      const int p_first = n - ql + i0;
      const int nt0 = (p_first + min(kPfRows, rows) - 1) / kPfTile + 1;
      const int rows1 = rows - kPfRows;
      const int nt1 = rows1 > 0 ? (p_first + kPfRows + rows1 - 1) / kPfTile + 1 : 0;
      return max(nt0, nt1);
    };
    auto pair_class = [&](int bb, int ql, int t) {  // 0 heaviest .. 63 lightest or invalid
      if (!pf_seq_ok(a, bb, ql)) return 63;
      return 63 - min(63, pair_tiles(ql, __ldg(a.lens + bb), t));
    };
    const bool by_work = (long long)a.B * a.q_tiles <= 4096;
    int *s_cls = reinterpret_cast<int *>(sm + Sh::kBarOff + 512);  // [65]
    if (by_work) {
      for (int i = lane; i < 65; i += 32) s_cls[i] = 0;
      __syncwarp();
      for (int bb = lane; bb < a.B; bb += 32) {
        const int ql = __ldg(a.cu_q + bb + 1) - __ldg(a.cu_q + bb);
        const int tl = ql > 0 ? min(a.q_tiles, (ql + kCtaRows - 1) / kCtaRows) : 0;
        for (int t = 0; t < tl; ++t) atomicAdd(&s_cls[pair_class(bb, ql, t)], 1);
      }
      __syncwarp();
      if (lane == 0) {
        int cum = 0;
        for (int c = 0; c < 64; ++c) {
          const int hcount = s_cls[c];
          s_cls[c] = cum;
          cum += hcount;
        }
        s_cls[64] = cum;
      }
      __syncwarp();
    }
    // the pr-th pair of the claim order (warp-uniform)
    auto pair_of = [&](int pr, int *b_out, int *qt_out) {
      if (!by_work) {
        pf_pair(a, pr, lane, b_out, qt_out);
        return;
      }
      const unsigned m0 = __ballot_sync(0xffffffffu, s_cls[lane] <= pr);
      const unsigned m1 = __ballot_sync(0xffffffffu, s_cls[lane + 32] <= pr);
      const int c = m1 ? 63 - __clz(m1) : 31 - __clz(m0);
      int idx = pr - s_cls[c];
      *b_out = -1;
      *qt_out = 0;
      for (int base = 0; base < a.B; base += 32) {
        const int bb = base + lane;
        int cnt = 0, ql = 0, tl = 0;
        if (bb < a.B) {
          ql = __ldg(a.cu_q + bb + 1) - __ldg(a.cu_q + bb);
          tl = ql > 0 ? min(a.q_tiles, (ql + kCtaRows - 1) / kCtaRows) : 0;
          for (int t = 0; t < tl; ++t) cnt += pair_class(bb, ql, t) == c;
        }
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const int chunk = __shfl_sync(0xffffffffu, incl, 31);
        if (idx < chunk) {
          const int src = __ffs(__ballot_sync(0xffffffffu, incl > idx)) - 1;
          int t_hit = 0;
          if (lane == src) {
            int k = idx - (incl - cnt);
            for (int t = 0; t < tl; ++t)
              if (pair_class(bb, ql, t) == c && k-- == 0) {
                t_hit = t;
                break;
              }
          }
          *b_out = base + src;
          *qt_out = __shfl_sync(0xffffffffu, t_hit, src);
          return;
        }
        idx -= chunk;
      }
    };
    // claim items (CTA c starts with item c, then takes the next unclaimed
    // one), publish each to the CTA as soon as a ring slot is free, and load
    // its query tiles once the products that read the previous ones are done
    unsigned w = blockIdx.x;
    int it = 0, ig[kPfGroups] = {0, 0};
    bool ok = true;
    while (true) {
      PfItem item = pf_item(a, -1, 0, -1, 0);
      if (w < total) {
        int bb, qq;
        pair_of((int)(w / (unsigned)a.H), &bb, &qq);
        const int hh = (int)(w % (unsigned)a.H);
        if (bb < 0) {
          item = pf_item(a, 0, hh, bb, qq);
        } else {
          const int ql = __ldg(a.cu_q + bb + 1) - __ldg(a.cu_q + bb);
          item = pf_item(a, pf_seq_ok(a, bb, ql) ? 1 : 0, hh, bb, qq);
        }
      }
      const int slot = it & 1;
      if (it >= 2) {
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&item_empty[slot], ((it >> 1) - 1) & 1));
        if (!ok) break;
      }
      if (lane == 0) {
        items[slot] = item;
        mbar_arrive(&item_full[slot]);
      }
      __syncwarp();
      ++it;
      if (item.kind < 0) break;
      if (item.kind == 1) {
#pragma unroll
        for (int g = 0; g < kPfGroups; ++g) {
          if (!ok || item.nt[g] == 0) continue;
          if (ig[g] > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(&q_empty[g], (ig[g] - 1) & 1)) && !aborted();
            if (!ok) break;
          }
          if (lane == 0) mbar_arrive_expect_tx(&q_full[g], (uint32_t)Sh::kQBytes);
          __syncwarp();
          if (lane < Sh::kRegions)
            tma_load_3d_keep(sm + Sh::kQOff + g * Sh::kQBytes + lane * kQRegion, &tmQ, &q_full[g],
                             64 * lane, item.h, item.q0 + kPfRows * g);
          ++ig[g];
        }
        if (!ok) break;
      }
      unsigned nw = 0;
      if (lane == 0) nw = atomicAdd(a.sched, 1u) + gridDim.x;
      w = __shfl_sync(0xffffffffu, nw, 0);
    }
    if (!ok && lane == 0) abort_cta();
    // the last query tiles land before the CTA can end (bounded)
#pragma unroll
    for (int g = 0; g < kPfGroups; ++g)
      if (ig[g] > 0) mbar_wait_bounded(&q_full[g], (ig[g] - 1) & 1);
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    // per item and 128-token KV tile: the K boxes (one per lane) once the
    // keys two ring tiles back are no longer read, then the V boxes once
    // the values two ring tiles back are not
    const int per_tensor = 8 * Sh::kRegions;     // boxes of K (or V) per 128-token tile
    const int region = (lane % per_tensor) >> 3, chunk = lane & 7;
    int it = 0, k_issued = 0, v_issued = 0;     // items read, ring tiles whose K / V loads were issued
    bool ok = true;
    while (ok) {
      const int slot = it & 1;
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&item_full[slot], (it >> 1) & 1));
      if (!ok) break;
      const PfItem item = items[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[slot]);
      ++it;
      if (item.kind < 0) break;
      const int kvh = item.h / a.G;
      for (int j = 0; j < item.ntiles && ok; ++j) {
        const int ring = k_issued, stage = ring % kPfStages, use = ring / kPfStages;
        const int tok0 = j * kPfTile;
        const int valid_chunks = min(8, (item.n - tok0 + 15) >> 4);
        const uint32_t bytes = (uint32_t)(valid_chunks * Sh::kRegions * 2048);
        // the tile's table entries: lane c < 8 loads chunk c's (in flight
        // during the wait below), broadcast to the lanes that issue that
        // chunk's boxes (K and V, every region)
        int phys = 0;
        if (lane < valid_chunks) phys = __ldg(a.tables + (size_t)item.b * a.max_blocks + (tok0 + 16 * lane) / a.bs);
        for (int v = 0; v < 2 && ok; ++v) {
          if (ring >= kPfStages) {
            ok = __all_sync(0xffffffffu,
                            mbar_wait_bounded(v ? &v_empty[stage] : &k_empty[stage], (use - 1) & 1)) &&
                 !aborted();
            if (!ok) break;
          }
          if (v == 0) {
            if (lane < valid_chunks && (phys < 0 || (long long)phys >= a.num_blocks)) {
              raise_flag(a.err, PKV_FLAG_BLOCK_OUT_OF_RANGE);
              phys = 0;
            }
            phys = __shfl_sync(0xffffffffu, phys, chunk);
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
          if (v) ++v_issued; else ++k_issued;
        }
      }
    }
    if (!ok && lane == 0) abort_cta();
    // the last fills land before the CTA can end (bounded)
    for (int r = max(0, k_issued - kPfStages); r < k_issued; ++r)
      mbar_wait_bounded(&k_full[r % kPfStages], (r / kPfStages) & 1);
    for (int r = max(0, v_issued - kPfStages); r < v_issued; ++r)
      mbar_wait_bounded(&v_full[r % kPfStages], (r / kPfStages) & 1);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = umma_idesc_f16(128, kPfTile, bf16, false);
      const uint32_t idesc_o = umma_idesc_f16(128, D, bf16, true);
      auto kv_base = [&](int ring, bool v) {
        return smem_u32(sm + Sh::kKVOff + (ring % kPfStages) * 2 * Sh::kKVBytes +
                        (v ? Sh::kKVBytes : 0));
      };
      auto issue_s = [&](int g, int ring) {  // S_g = Q_g . K^T over D in 16-wide steps
        const uint32_t qb = smem_u32(sm + Sh::kQOff + g * Sh::kQBytes), kb = kv_base(ring, false);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          umma_f16(tmem + 256 * g, umma_desc_sw128(qb + (k >> 2) * kQRegion + (k & 3) * 32, 16, 1024),
                   umma_desc_sw128(kb + (k >> 2) * kKVRegion + (k & 3) * 32, 16, 1024), idesc_s,
                   k > 0);
        umma_commit(&s_full[g]);
      };
      auto issue_pv = [&](int g, int ring, bool acc) {  // O_g (+)= P_g . V, P from tensor memory
        const uint32_t vb = kv_base(ring, true);
#pragma unroll
        for (int k = 0; k < kPfTile / 16; ++k)
          umma_f16_tmem_a(tmem + 256 * g + 128, tmem + 256 * g + 8 * k,
                          umma_desc_sw128(vb + k * 2048, kKVRegion, 1024), idesc_o, acc || k > 0);
      };
      // Per item: S of the first tile of both groups; then per tile and
      // group, as soon as P_g(j) arrives: P_g(j) . V_j, then S_g(j+1).  The
      // products of one thread run in issue order, so S_g(j+1) -- written
      // over P_g(j) -- starts after P_g(j) . V_j has read it, and the commit
      // that signals S_g(j+1) also covers P_g(j) . V_j (O is final for tile
      // j when the softmax sees S_g(j+1)).  The next item's first product
      // into O (no accumulate) comes after the softmax's first P of that
      // item, which the softmax writes only once it has read the previous O.
      // Group 0 (the earlier query rows) needs no more KV tiles than group
      // 1: once its last product of an item is issued, group 0's first S of
      // the next item is issued as soon as that item, its query tile and its
      // first keys are there, so group 0's softmax starts on the next item
      // while group 1 finishes this one.
      int it = 0, ring0 = 0, ig[kPfGroups] = {0, 0}, tcnt[kPfGroups] = {0, 0};
      PfItem nx;
      bool have_nx = false;   // the next item is read already
      bool early = false;     // ... and group 0's first S of it issued
      bool ok = true;
      while (ok) {
        PfItem item;
        if (have_nx) {
          item = nx;
          have_nx = false;
        } else {
          const int slot = it & 1;
          ok = mbar_wait_bounded(&item_full[slot], (it >> 1) & 1);
          if (!ok) break;
          item = items[slot];
          mbar_arrive(&item_empty[slot]);
          ++it;
        }
        if (item.kind < 0) break;
        if (item.ntiles == 0) continue;
        const bool pre = early;
        early = false;
        ok = mbar_wait_bounded(&k_full[ring0 % kPfStages], (ring0 / kPfStages) & 1);
#pragma unroll
        for (int g = 0; g < kPfGroups; ++g)
          if (ok && item.nt[g] > 0 && !(g == 0 && pre)) ok = mbar_wait_bounded(&q_full[g], ig[g] & 1);
        if (!ok || aborted()) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int g = 0; g < kPfGroups; ++g) {
          if (item.nt[g] == 0 || (g == 0 && pre)) continue;
          issue_s(g, ring0);
          if (item.nt[g] == 1) umma_commit(&q_empty[g]);  // the group's last S of the item
        }
        umma_commit(&k_empty[ring0 % kPfStages]);
        const int ring_next = ring0 + item.ntiles;
        // group 0's first S of the next item, if everything it reads is
        // there (never waits)
        auto try_early = [&]() {
          if (early) return;
          if (!have_nx) {
            const int slot = it & 1;
            if (!mbar_test_wait(&item_full[slot], (it >> 1) & 1)) return;
            nx = items[slot];
            mbar_arrive(&item_empty[slot]);
            ++it;
            have_nx = true;
          }
          if (nx.kind != 1) return;
          if (!mbar_test_wait(&k_full[ring_next % kPfStages], (ring_next / kPfStages) & 1) ||
              !mbar_test_wait(&q_full[0], (ig[0] + 1) & 1))
            return;
          tc_fence_after();
          issue_s(0, ring_next);
          if (nx.nt[0] == 1) umma_commit(&q_empty[0]);
          early = true;
        };
        for (int j = 0; ok && j < item.ntiles; ++j) {
          const int ring = ring0 + j;
          bool v_ready = false, k_ready = false;
#pragma unroll
          for (int g = 0; g < kPfGroups; ++g) {
            if (!ok || j >= item.nt[g]) continue;
            if (g == 1 && j + 1 >= item.nt[0]) {
              // group 0 is done with this item: look for its next one while
              // group 1's P is not there yet
              const unsigned long long t0 = global_timer_ns();
              while (!mbar_test_wait(&p_full[1], tcnt[1] & 1)) {
                try_early();
                if (global_timer_ns() - t0 > kWaitLimitNs) break;
              }
            }
            ok = mbar_wait_bounded(&p_full[g], tcnt[g] & 1);
            ++tcnt[g];
            if (!ok) break;
            if (!v_ready) {
              ok = mbar_wait_bounded(&v_full[ring % kPfStages], (ring / kPfStages) & 1);
              if (!ok) break;
              v_ready = true;
            }
            tc_fence_after();
            issue_pv(g, ring, j > 0);
            // the tile's last P . V: its V slot is free once that has run
            if (g == kPfGroups - 1 || j >= item.nt[g + 1]) umma_commit(&v_empty[ring % kPfStages]);
            if (j + 1 < item.nt[g]) {
              if (!k_ready) {
                ok = mbar_wait_bounded(&k_full[(ring + 1) % kPfStages], ((ring + 1) / kPfStages) & 1);
                if (!ok) break;
                k_ready = true;
              }
              issue_s(g, ring + 1);
              if (j + 2 == item.nt[g]) umma_commit(&q_empty[g]);
            } else {
              umma_commit(&o_done[g]);  // the group's last product of the item
            }
          }
          if (!ok) break;
          if (j + 1 < item.ntiles) umma_commit(&k_empty[(ring + 1) % kPfStages]);
        }
        ring0 = ring_next;
        if (ok && aborted()) ok = false;
#pragma unroll
        for (int g = 0; g < kPfGroups; ++g) ig[g] += item.nt[g] > 0;
      }
      if (!ok) abort_cta();
      umma_commit(mma_done);  // every product issued above has completed when this arrives
      mbar_wait_bounded(mma_done, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int g = (warp - 2) >> 2;                      // warpgroup = query tile
    const int quarter = warp & 3;
    const int r = 32 * quarter + lane;                  // row in the tile = tensor-memory lane
    const int rr = g * kPfRows + r;                     // row in the item
    const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
    const uint32_t tmem_sp = tmem + 256 * g + lane_off; // S, then P over its first half
    const uint32_t tmem_o = tmem + 256 * g + 128 + lane_off;
    // scores are kept raw; with scale > 0 the max commutes with the scale
    // and one fused multiply-add per pair gives s * scale * log2(e) - m
    const float sl2 = a.scale_log2;
    const bool pos_scale = sl2 > 0.f;
    const float mul = pos_scale ? sl2 : 1.f;
    int it = 0, ring0 = 0, ig = 0, tcnt = 0;
    bool ok = true;
    while (true) {
      const int slot = it & 1;
      ok = mbar_wait_bounded(&item_full[slot], (it >> 1) & 1);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      const PfItem item = items[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[slot]);
      ++it;
      if (item.kind < 0) break;
      const int my_tiles = nt_of(item, g);
      if (my_tiles == 0) {
        ring0 += item.ntiles;
        continue;
      }
      const bool real_row = rr < item.rows;
      const int p_row = item.p_first + (real_row ? rr : item.rows - 1);  // padding rows mirror the last row
      const int n = item.n;
      float m_used = -INFINITY, l = 0.f;
      for (int j = 0; j < my_tiles; ++j) {
        ok = mbar_wait_bounded(&s_full[g], tcnt & 1);
        ++tcnt;
        if (!__all_sync(0xffffffffu, ok) || aborted()) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int t0 = j * kPfTile;
        const int ring = ring0 + j;
        // the row's 128 scores in registers: both loads in flight, one wait
        // (scores raw when scale > 0: the max commutes with the scale)
        uint32_t sa[64], sb[64];
        tmem_ld64_nowait(tmem_sp, sa);
        tmem_ld64_nowait(tmem_sp + 64, sb);
        tmem_wait_ld_bind64(sa);
        reg_bind64(sb);
        float sc[128];
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          sc[i] = __uint_as_float(sa[i]);
          sc[64 + i] = __uint_as_float(sb[i]);
        }
        if (!pos_scale) {
#pragma unroll
          for (int i = 0; i < 128; ++i) sc[i] *= sl2;
        }
        if (t0 + kPfTile - 1 > p_row) {
#pragma unroll
          for (int i = 0; i < 128; ++i) sc[i] = t0 + i <= p_row ? sc[i] : -INFINITY;
        }
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < 128; i += 2) mx = max3f(mx, sc[i], sc[i + 1]);
        if (pos_scale) mx *= sl2;
        // the reference max moves only when the row max exceeds it by 2^8
        const float m_new = (mx > m_used + 8.f) ? mx : m_used;
        const float alpha = fast_exp2(m_used - m_new);  // 0 on the first tile
        const bool rescale = __any_sync(0xffffffffu, m_new != m_used) && j > 0;
        l *= alpha;
        m_used = m_new;
        // P = 2^(s * scale * log2(e) - m), rounded to the input type, two
        // tokens per column over the first 64 S columns; l sums the
        // unrounded weights
        float2 lsum = make_float2(0.f, 0.f);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int c = 64 * hf + 2 * i;
            float2 x = ffma2(make_float2(sc[c], sc[c + 1]), make_float2(mul, mul),
                             make_float2(-m_used, -m_used));
            x.x = fast_exp2(x.x);
            x.y = fast_exp2(x.y);
            lsum = fadd2(lsum, x);
            pk[i] = PackPair<T>::pack(x.x, x.y);
          }
          tmem_st32u_nowait(tmem_sp + 32 * hf, pk);
        }
        tmem_wait_st();
        l += lsum.x + lsum.y;
        // O is final for tile j-1 here: the commit that signalled S_g(j) also
        // covers P_g(j-1) . V, issued before it.  The rescale and the zeroed V
        // rows come after P (the scores' registers are free by then) and
        // before the arrive that lets P_g(j) . V_j go.
        if (rescale) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            float v[32];
            tmem_ld32(tmem_o + 32 * c, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= alpha;
            tmem_st32(tmem_o + 32 * c, v);
          }
        }
        // the tile's V rows past the context are zeroed (they may hold
        // anything, and 0 * NaN would poison the product)
        const bool past_end = t0 + kPfTile > n;
        if (past_end) {
          ok = mbar_wait_bounded(&v_full[ring % kPfStages], (ring / kPfStages) & 1);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          if (r >= n - t0) {
            uint8_t *vrow = sm + Sh::kKVOff + (ring % kPfStages) * 2 * Sh::kKVBytes + Sh::kKVBytes + r * 128;
#pragma unroll
            for (int rg = 0; rg < Sh::kRegions; ++rg)
#pragma unroll
              for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4 *>(vrow + rg * kKVRegion + c * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        // the zeroed V rows (generic writes) before the product reads them
        if (past_end) fence_proxy_async_shared();
        tc_fence_before();
        mbar_arrive(&p_full[g]);
      }
      if (!ok) break;
      ok = mbar_wait_bounded(&o_done[g], ig & 1);
      ++ig;
      if (!__all_sync(0xffffffffu, ok) || aborted()) {
        ok = false;
        break;
      }
      tc_fence_after();
      // O / l; the next item's first product into O waits for this group's
      // first P of that item, written after these reads
      const float inv_l = 1.f / l;
      const size_t q_row = (size_t)(item.q0 + (real_row ? rr : 0)) * a.H + item.h;
      T *orow = reinterpret_cast<T *>(a.out) + q_row * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float v[32];
        tmem_ld32(tmem_o + 32 * c, v);
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
      ring0 += item.ntiles;
    }
    if (!ok && lane == 0) abort_cta();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, Sh::kTmemCols);
  if (tid == 0) {
    // the last CTA of the launch puts the work counters back for the next
    // (every claim of this CTA was an atomic whose value it used before the
    // barrier, so it is performed already: no fence, which at the end of a
    // launch can hold a thread for tens of microseconds)
    if (atomicAdd(a.sched + 1, 1u) == gridDim.x - 1) {
      atomicExch(a.sched, 0u);
      atomicExch(a.sched + 1, 0u);
    }
  }
}

// ---------------------------------------------------------------- host side

static int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < 64) cached[dev] = n;
  return n;
}

// This device's work counters (looked up once per device).
static unsigned *sched_counters() {
  static unsigned *cached[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  if (dev < 64 && cached[dev]) return cached[dev];
  unsigned *p = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_pf_sched) != cudaSuccess) return nullptr;
  if (dev < 64) cached[dev] = p;
  return p;
}

template <int D, typename T>
static pkv_status launch_prefill_t(const PrefillArgs &a, const CUtensorMap &mq, const CUtensorMap &mk,
                                   const CUtensorMap &mv, int ctas, cudaStream_t stream) {
  auto kern = pkv_prefill_tc_kernel<D, T>;
  static int configured[64] = {0};
  if (!allow_smem(kern, PfShape<D>::kSmem, configured)) return PKV_ERR_CUDA;
  kern<<<ctas, kPfThreads, PfShape<D>::kSmem, stream>>>(mq, mk, mv, a);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status launch_prefill_tc(void *out, const void *q, const void *k_cache, const void *v_cache,
                             const int32_t *tables, const int32_t *cu_q, const int32_t *lens,
                             int B, long long total_q, int H, int KVH, int D, int bs,
                             int max_blocks, long long num_blocks, float scale, pkv_dtype dt,
                             int q_tiles, int pairs_bound, int *err, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  if (!encode_rows_map(&mq, q, dt, total_q, H, D, kPfRows) ||
      !encode_cache_map(&mk, k_cache, dt, num_blocks, bs, KVH, D) ||
      !encode_cache_map(&mv, v_cache, dt, num_blocks, bs, KVH, D))
    return PKV_ERR_CUDA;
  unsigned *sched = sched_counters();
  if (!sched) return PKV_ERR_CUDA;
  // a counter slot per launch, taken in turn (launches in flight at once on
  // one device must number fewer than kSchedSlots)
  static std::atomic<unsigned> next_slot{0};
  const unsigned slot = next_slot.fetch_add(1u) % kSchedSlots;
  PrefillArgs a;
  memset(&a, 0, sizeof a);
  a.out = out;
  a.tables = tables;
  a.cu_q = cu_q;
  a.lens = lens;
  a.err = err;
  a.sched = sched + 2 * slot;
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
  const int sms = sm_count();
  if (sms <= 0) return PKV_ERR_CUDA;
  // one persistent CTA per SM, never more than the items there can be
  const int ctas = (int)std::min<long long>((long long)pairs_bound * H, sms);
  const bool bf = dt == PKV_BF16;
  if (D == 128) return bf ? launch_prefill_t<128, __nv_bfloat16>(a, mq, mk, mv, ctas, stream)
                          : launch_prefill_t<128, __half>(a, mq, mk, mv, ctas, stream);
  if (D == 64) return bf ? launch_prefill_t<64, __nv_bfloat16>(a, mq, mk, mv, ctas, stream)
                         : launch_prefill_t<64, __half>(a, mq, mk, mv, ctas, stream);
  return PKV_ERR_UNSUPPORTED;
}

}  // namespace pkv
