// pkv_decode_wide.cu -- paged decode attention for wide query groups (16
// query heads per KV head: MQA and wide GQA) with bf16 / fp16 caches on
// sm_103a, on the 5th-generation tensor cores with the roles of the
// operands swapped.
//
// Definition (course page "P09 · Paged KV 写入 + decode attention（参考实现）",
// section 题面速览 "decode 读" and the paged_decode_attention shape trace):
// n = context_lens[b]; only block_tables[b, :ceil(n/bs)] is read; token t is
// row t % bs of physical block tbl[t / bs]; exactly n tokens; query head h
// uses KV head h / (H / KVH); fp32 scores scaled before an fp32 softmax;
// weighted V sum cast to the output dtype.  The block-wise online softmax is
// the one of the interview note "PagedAttention kernel: paged KV cache 与
// block table", section 代码; its partitioned (v2) variant, section 深入原理,
// is the split into work items, merged by log-sum-exp.
//
// Why swapped.  A decode query group is 16 rows at most -- below the
// smallest M of a tensor-core product -- while a KV tile has many tokens.
// So the products run with tokens as M:
//   S^T [128 tokens x 16 heads]  = K_tile [128 x D] . Q_group^T [D x 16]
//   O^T [D x 16 heads]          += V_tile^T [D x 128] . P^T [128 x 16]
// (M = 128 tokens or 128 of the D values, N = 16 heads, accumulators in
// tensor memory); the softmax thread of token lane t holds that token's 16
// head scores, and the per-head max is a reduction over the 128 lanes, done
// only when some score exceeds the running max by more than 2^8.
//
// Work decomposition.  A work item is (sequence, KV head, 16-head chunk,
// partition of P tokens: the plan's partition size, or, when the plan chose
// it, about 1.2 CTA shares of the batch's 128-token tiles, worked out by
// every CTA from the lengths); the grid is persistent (at most one CTA per
// SM) and CTAs claim items from a counter in device memory: every full
// partition first (the latest partitions, which only long contexts have,
// first), then the partial ones by tile count, most first -- long contexts
// spread over SMs early and the last claims are the smallest.  8 warps:
//   warp 6     scheduler: claims items (the next once the producer reaches
//              the current item's last tile), publishes each to the CTA
//              through a two-slot ring, loads the item's 16 query rows (TMA,
//              128-byte swizzle) once the last S^T of the previous item is
//              done;
//   warp 0     producer: the tiled TMA loads of K and V tiles (boxes of up
//              to 128 tokens of one cache block x 64 columns, 128-byte
//              swizzle; block-table entries read four tiles ahead) into one
//              ring of K-or-V slots, in the order K0, K1, V0, K2, V1, ... so
//              keys run a tile ahead of values;
//   warp 1     MMA issuer (one thread): S^T of the item's first two tiles,
//              then per tile, once its P^T is written: O^T += V^T . P^T and
//              the S^T two tiles ahead into the freed score buffer; frees
//              the tensor memory at the end;
//   warp 7     append (fused step, one launch): per item that ends its
//              context, the new token's K and V rows -- written to the cache
//              row by head chunk 0's item, and written over row n - 1 of the
//              last tile's K and V in shared memory once they land, before
//              the MMA thread may read them (so no read waits for the cache
//              write: bit-identical to writing first, then reading);
//   warps 2-5  softmax, thread = token lane: scores from tensor memory,
//              running max and per-lane weight sums per head, P^T written to
//              shared memory; after the item's last tile the per-head sums
//              are reduced and the item is finished -- output rows, or the
//              partition's partials counted by an atomic read at the next
//              item's end, where the last partition of the sequence merges
//              (log-sum-exp).  The CTA's last merge waits for the roles to
//              end and is run by all eight warps: twice the threads, half
//              the rounds of partial loads, on the launch's tail (the whole
//              CTA's: 35.2 -> 34.2 us on the MQA batch, three input sets).
// Launched into a captured graph, the kernel is a programmatic dependent of
// the step before it: a CTA works out its schedule, reads its first item's
// table entries and asks L2 for that item's first two K/V tiles (TMA
// prefetches of the boxes its loads will read) before griddepcontrol.wait;
// K/V loads, cache, workspace and output writes come after.
// Every wait on an mbarrier is bounded; on time-out the CTA raises
// PKV_FLAG_TIMEOUT, lets its copies and products land (bounded) and exits.
#include <string.h>

#include <atomic>
#include <type_traits>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_tcgen05.cuh"

namespace pkv {

constexpr int kWdTile = 128;             // tokens per KV tile (M of S^T)
constexpr int kWdHeads = 16;             // query heads per item (N)
constexpr int kWdWarps = 8;
constexpr int kWdThreads = 32 * kWdWarps;
constexpr int kWdSchedWarp = 6;
constexpr int kWdAppendWarp = 7;
constexpr int kWdReaders = 3 + 4;        // producer, MMA thread, append warp, one lane per softmax warp
constexpr int kWdPatchOff = 1952;        // misc area: the four append counters
constexpr int kWdFinOff = 1968;          // misc area: the CTA's last merge, run by all threads
constexpr int kWdSchedSlots = 1024;      // work counters, one per launch in flight
constexpr int kWdRingBytes = 192 * 1024; // K-or-V slots

// Work counters of the persistent launches: slot s holds (next item to claim
// beyond the first gridDim.x, CTAs finished); the last CTA of a launch puts
// both back to zero, so a slot is ready again for the launch after.
__device__ unsigned g_wd_sched[2 * kWdSchedSlots];

template <int D>
struct WdShape {
  static constexpr int kRegions = D / 64;
  static constexpr int kRegionBytes = kWdTile * 128;            // 128 token rows x 64 elements
  static constexpr int kTileBytes = kRegions * kRegionBytes;    // one K or V tile
  static constexpr int kSlots = kWdRingBytes / kTileBytes;      // 3 at D = 256, 6 at D = 128
  static constexpr int kQRegion = kWdHeads * 128;               // 16 query rows x 64 elements
  static constexpr int kQBytes = kRegions * kQRegion;
  static constexpr int kPRegion = kWdHeads * 128;               // P^T: 16 head rows x 64 tokens
  static constexpr int kPBytes = 2 * kPRegion;                  // one 128-token P^T buffer
  static constexpr int kQOff = kSlots * kTileBytes;
  static constexpr int kPOff = kQOff + kQBytes;                 // [2]
  static constexpr int kOOff = kPOff + 2 * kPBytes;             // [16][D] fp32 (finishing)
  static constexpr int kMiscOff = kOOff + kWdHeads * D * 4;
  static constexpr int kMiscBytes = 2048;   // barriers, item ring, reductions, claim tables,
                                            // append counters
  static constexpr int kSmem = kMiscOff + kMiscBytes + 1024;    // + alignment slack
  // tensor memory: two S^T buffers (16 columns each), O^T (D / 128 blocks
  // of 16 columns)
  static constexpr uint32_t kTmemCols = 64;
  static_assert(kSlots >= 3 && kSlots <= 6, "the ring has three to six slots");
  static_assert(1168 + 3 * 65 * 4 <= kWdPatchOff && kWdPatchOff + 16 <= kWdFinOff &&
                    kWdFinOff + 5 * 4 <= kMiscBytes,
                "shared-memory misc area");
  static_assert(kSmem <= 232448, "shared memory per block");
  static_assert(32 + 16 * (D / 128) <= (int)kTmemCols, "tensor memory");
};

// One work item as every role sees it.  kind: 1 work, -1 no more items.
struct __align__(16) WdItem {
  int kind, b, kvh, hc;    // sequence, KV head, 16-head chunk of its group
  int part, nparts;        // partition and partitions of the sequence
  int t0, t1;              // the partition's tokens
  int n, ntiles;
  int patch_row;           // fused step: row of position n - 1 in the item's last tile
                           // (the item ends the context), else -1
  int pad1;
};
static_assert(sizeof(WdItem) == 48, "three 16-byte words");

struct WdArgs {
  DecodeArgs d;        // shapes, caches, workspace, flags (the merge reads these)
  unsigned *sched;     // this launch's (next, done) counters
  int hchunks;         // 16-head chunks per KV head (G / 16)
  int units;           // B * KVH * hchunks
  int check_append;    // fused step (new_slots given): write each new token, read it at n - 1
  int box_tok;         // tokens per K/V box: 16, 32, 64 or 128, dividing bs and P
  int auto_items;      // the partition size is the plan's own: items may be larger
};

// Whether the phase with the given parity has completed (never waits).
__device__ __forceinline__ bool wd_test_wait(uint64_t *bar, uint32_t parity) {
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

// Monotonic event counters in shared memory, written by one thread with
// release and read with acquire (no phase parity: a waiter can never
// mistake an old event for the one it waits for).
__device__ __forceinline__ void wd_count_store(int *p, int v) {
  asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ int wd_count_load(const int *p) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
// Wait until *p >= v; false after kWaitLimitNs.
__device__ __forceinline__ bool wd_count_wait(const int *p, int v) {
  if (wd_count_load(p) >= v) return true;
  const unsigned long long t0 = global_timer_ns();
  while (wd_count_load(p) < v)
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  return true;
}

// A barrier of the 128 softmax threads on an mbarrier, with the bounded
// wait (a thread that gave up elsewhere cannot leave the others waiting
// forever).
struct WdGroupSync {
  uint64_t *bar;
  int *phase;
  __device__ __forceinline__ void operator()() const {
    mbar_arrive(bar);
    // a short wait: spin on the non-suspending test (bounded)
    const uint32_t par = (uint32_t)(*phase) & 1u;
    if (!wd_test_wait(bar, par)) {
      const unsigned long long t0 = global_timer_ns();
      while (!wd_test_wait(bar, par) && global_timer_ns() - t0 <= kWaitLimitNs) {
      }
    }
    ++*phase;
  }
};

__device__ __forceinline__ void wd_tma_4d(void *dst, const CUtensorMap *map, uint64_t *bar, int c0,
                                          int c1, int c2, int c3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "l"(policy)
      : "memory");
}

// The same 4-D box asked into L2 only (no shared memory, no barrier).
__device__ __forceinline__ void wd_tma_prefetch_4d(const CUtensorMap *map, int c0, int c1, int c2,
                                                   int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}

__device__ __forceinline__ void wd_tma_3d(void *dst, const CUtensorMap *map, uint64_t *bar, int c0,
                                          int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

template <typename T>
__device__ __forceinline__ unsigned short wd_bits(float x);
template <>
__device__ __forceinline__ unsigned short wd_bits<__nv_bfloat16>(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
template <>
__device__ __forceinline__ unsigned short wd_bits<__half>(float x) {
  return __half_as_ushort(__float2half_rn(x));
}

// Order of an item's loads through the ring: K0, K1, V0, K2, V1, K3, V2, ...,
// V(n-1) -- keys a tile ahead of values, so the keys of tile j+2 are fetched
// as soon as the values of tile j-1 are no longer read.
__device__ __forceinline__ int wd_kidx(int j) { return j < 2 ? j : 2 * j - 1; }
__device__ __forceinline__ int wd_vidx(int j, int n) { return j == n - 1 ? 2 * n - 1 : 2 * j + 2; }

// Units u = (sequence, KV head, 16-head chunk): a unit's length (its
// sequence's, checked, clamped to the partitions the launch covers) and its
// work item for a partition, given the length (an empty context is one item
// that writes zero rows).
// A length as loaded, checked: negative counts as empty; beyond the block
// table or the partitions the launch covers it is cut there (CTA 0 flags
// both).
__device__ __forceinline__ int wd_clamp_len(const WdArgs &w, int n) {
  const DecodeArgs &a = w.d;
  const long long cap = min((long long)a.max_blocks * a.bs, (long long)a.max_parts * a.P);
  n = max(n, 0);
  return (long long)n > cap ? (int)cap : n;
}
__device__ __forceinline__ int wd_unit_len(const WdArgs &w, int u) {
  return wd_clamp_len(w, __ldg(w.d.lens + u / (w.d.KVH * w.hchunks)));
}
__device__ __forceinline__ WdItem wd_make_item(const WdArgs &w, int u, int part, int n, int P) {
  const DecodeArgs &a = w.d;
  WdItem it;
  memset(&it, 0, sizeof it);
  it.patch_row = -1;
  it.b = u / (a.KVH * w.hchunks);
  it.kvh = (u / w.hchunks) % a.KVH;
  it.hc = u % w.hchunks;
  it.part = part;
  it.n = n;
  it.nparts = n > 0 ? (n + P - 1) / P : 1;
  it.t0 = part * P;
  it.t1 = min(n, it.t0 + P);
  if (n == 0) {
    it.kind = 2;  // empty context: zero output rows
    return it;
  }
  it.kind = 1;
  it.ntiles = (it.t1 - it.t0 + kWdTile - 1) / kWdTile;
  it.patch_row = (w.check_append && it.t1 == n) ? n - 1 - (it.t0 + (it.ntiles - 1) * kWdTile) : -1;
  return it;
}

// Two fp32 values rounded to nearest even and packed as one pair of T (the
// first in the low half, so at the lower address).
template <typename T>
__device__ __forceinline__ uint32_t wd_pack2(float lo, float hi) {
  if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
  } else {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
  }
}

// The end of one item, by the 128 softmax threads (thread ts, barrier
// `sync`), given per head r: s_m[r] running max (log2 units), the sum of
// 2^(score - s_m[r]) as four partial sums s_lw[w * 16 + r] (one per softmax
// warp, added here by each thread that needs them), s_o[r * D + d] the
// weighted V sum.  One partition:
// the output rows s_o / l.  Otherwise the partials go to the workspace and
// thread 0 counts the partition with an acquire-release atomic whose result
// it reads only later (at the next item's end, where the last partition
// merges): the atomic's round trip is not waited for.  Returns whether a
// count is pending.
template <int D, typename T, typename Sync>
__device__ bool wd_publish(const DecodeArgs &a, int b, int head0, int part, int nparts,
                           const float *s_m, const float *s_lw, const float *s_o, int *counter,
                           int ts, Sync sync, unsigned *prev) {
  T *out = reinterpret_cast<T *>(a.out);
  const size_t row0 = (size_t)b * a.H + head0;
  auto l_of = [&](int r) {
    return (s_lw[r] + s_lw[kWdHeads + r]) + (s_lw[2 * kWdHeads + r] + s_lw[3 * kWdHeads + r]);
  };
  if (nparts == 1) {
    // eight outputs per thread and step: one 16-byte store
    for (int i = ts; i < kWdHeads * D / 8; i += 128) {
      const float4 x0 = *reinterpret_cast<const float4 *>(s_o + 8 * i);
      const float4 x1 = *reinterpret_cast<const float4 *>(s_o + 8 * i + 4);
      const float inv_l = 1.f / l_of(8 * i / D);
      uint4 v;
      v.x = wd_pack2<T>(x0.x * inv_l, x0.y * inv_l);
      v.y = wd_pack2<T>(x0.z * inv_l, x0.w * inv_l);
      v.z = wd_pack2<T>(x1.x * inv_l, x1.y * inv_l);
      v.w = wd_pack2<T>(x1.z * inv_l, x1.w * inv_l);
      *reinterpret_cast<uint4 *>(out + row0 * D + 8 * i) = v;
    }
    return false;
  }
  if (ts < kWdHeads) {
    a.ws_m[(row0 + ts) * a.max_parts + part] = s_m[ts];
    a.ws_l[(row0 + ts) * a.max_parts + part] = l_of(ts);
  }
  for (int i = ts; i < kWdHeads * D / 4; i += 128) {
    const int r = 4 * i / D, d = 4 * i - r * D;
    *reinterpret_cast<float4 *>(a.ws_o + ((row0 + r) * a.max_parts + part) * D + d) =
        *reinterpret_cast<const float4 *>(s_o + 4 * i);
  }
  // the barrier orders the group's writes before thread 0's release
  sync();
  if (ts == 0) {
    unsigned v;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                 : "=r"(v)
                 : "l"(reinterpret_cast<uint64_t>(counter))
                 : "memory");
    *prev = v;
  }
  return true;
}

// The merge of a (sequence, head chunk) whose partitions have all arrived,
// by NT threads (the softmax group, or the whole CTA for its last item)
// of the CTA whose count was the last:  M = max_p m_p,
// L = sum_p l_p 2^(m_p - M),  out = sum_p o_p 2^(m_p - M) / L.  It sits at
// the end of the work, so it is written for latency: warp w of the NT / 32
// takes rows w, w + NT / 32, ... together (their m and l loads in one round
// trip when nparts <= 32) and puts the weights in s_w (16 x nparts floats
// when they fit in w_cap); then each thread takes up to four output vectors
// of four values at a time with eight partitions' loads of each in flight.
// The counter is put back to zero for the next call.
template <int D, typename T, int NT, typename Sync>
__device__ void wd_merge(const DecodeArgs &a, int b, int head0, int nparts, float *s_w, int w_cap,
                         int *s_scratch, int *counter, int ts, Sync sync) {
  T *out = reinterpret_cast<T *>(a.out);
  const size_t row0 = (size_t)b * a.H + head0;
  constexpr int kVecs = kWdHeads * D / 4;   // output vectors of four values
  constexpr int kU = kVecs / NT < 4 ? kVecs / NT : 4;   // vectors per thread and step
  static_assert(kU >= 1 && kVecs % (NT * kU) == 0, "whole steps of the threads");
  // the other partitions' partials: thread 0's count was an acquire-release
  // atomic that saw theirs, the group barrier passes that on, and the loads
  // below go to L2
  const int warp = ts >> 5, lane = ts & 31;
  constexpr int kWarps = NT / 32;
  constexpr int kRows = kWdHeads / kWarps;
  static_assert(kRows * kWarps == kWdHeads, "rows per warp");
  const bool cached = kWdHeads * nparts <= w_cap;
  float *s_M = reinterpret_cast<float *>(s_scratch + 1), *s_invL = s_M + kWdHeads;
  const float *pm[kRows], *pl[kRows];
#pragma unroll
  for (int j = 0; j < kRows; ++j) {
    pm[j] = a.ws_m + (row0 + warp + kWarps * j) * a.max_parts;
    pl[j] = a.ws_l + (row0 + warp + kWarps * j) * a.max_parts;
  }
  auto warp_max = [](float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
  };
  auto warp_sum = [](float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
  };
  float M[kRows], inv_l[kRows];
  if (nparts <= 32) {
    const bool mine = lane < nparts;
    const int pc = min(lane, nparts - 1);   // clamped: the loads are not predicated
    float mv[kRows], lv[kRows];
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      mv[j] = __ldcg(pm[j] + pc);
      lv[j] = __ldcg(pl[j] + pc);
    }
#pragma unroll
    for (int j = 0; j < kRows; ++j) mv[j] = mine ? mv[j] : -INFINITY;
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      M[j] = warp_max(mv[j]);
      const float e = mine ? fast_exp2(mv[j] - M[j]) : 0.f;
      inv_l[j] = 1.f / warp_sum(mine ? lv[j] * e : 0.f);
      if (cached && mine) s_w[(warp + kWarps * j) * nparts + lane] = e * inv_l[j];
    }
  } else {
    float L[kRows];
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      M[j] = -INFINITY;
      L[j] = 0.f;
    }
    for (int p = lane; p < nparts; p += 32) {
#pragma unroll
      for (int j = 0; j < kRows; ++j) M[j] = fmaxf(M[j], __ldcg(pm[j] + p));
    }
#pragma unroll
    for (int j = 0; j < kRows; ++j) M[j] = warp_max(M[j]);
    for (int p = lane; p < nparts; p += 32) {
#pragma unroll
      for (int j = 0; j < kRows; ++j) L[j] += __ldcg(pl[j] + p) * fast_exp2(__ldcg(pm[j] + p) - M[j]);
    }
#pragma unroll
    for (int j = 0; j < kRows; ++j) inv_l[j] = 1.f / warp_sum(L[j]);
    if (cached)
      for (int p = lane; p < nparts; p += 32) {
#pragma unroll
        for (int j = 0; j < kRows; ++j)
          s_w[(warp + kWarps * j) * nparts + p] = fast_exp2(__ldcg(pm[j] + p) - M[j]) * inv_l[j];
      }
  }
  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      s_M[warp + kWarps * j] = M[j];
      s_invL[warp + kWarps * j] = inv_l[j];
    }
  }
  sync();
  for (int i0 = ts; i0 < kVecs; i0 += NT * kU) {
    int r[kU], d[kU];
    const float4 *po[kU];
    float4 acc[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = i0 + NT * u;
      r[u] = 4 * i / D;
      d[u] = 4 * i - r[u] * D;
      po[u] = reinterpret_cast<const float4 *>(a.ws_o + (row0 + r[u]) * a.max_parts * D + d[u]);
      acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (cached) {
      // every load of a step issued before any is used: the partition index
      // is clamped (a repeated load gets weight 0), so no load is predicated
      for (int p0 = 0; p0 < nparts; p0 += 8) {
        float4 v[kU][8];
#pragma unroll
        for (int u = 0; u < kU; ++u)
#pragma unroll
          for (int q = 0; q < 8; ++q) v[u][q] = __ldcg(po[u] + (size_t)min(p0 + q, nparts - 1) * (D / 4));
#pragma unroll
        for (int u = 0; u < kU; ++u)
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float wt = p0 + q < nparts ? s_w[r[u] * nparts + p0 + q] : 0.f;
            acc[u].x += wt * v[u][q].x;
            acc[u].y += wt * v[u][q].y;
            acc[u].z += wt * v[u][q].z;
            acc[u].w += wt * v[u][q].w;
          }
      }
    } else {
      // more partitions than weights fit: each weight from its m
      for (int p = 0; p < nparts; ++p) {
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const float wt = fast_exp2(__ldcg(a.ws_m + (row0 + r[u]) * a.max_parts + p) - s_M[r[u]]) *
                           s_invL[r[u]];
          const float4 v = __ldcg(po[u] + (size_t)p * (D / 4));
          acc[u].x += wt * v.x;
          acc[u].y += wt * v.y;
          acc[u].z += wt * v.z;
          acc[u].w += wt * v.w;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      uint2 o;
      o.x = wd_pack2<T>(acc[u].x, acc[u].y);
      o.y = wd_pack2<T>(acc[u].z, acc[u].w);
      *reinterpret_cast<uint2 *>(out + (row0 + r[u]) * D + d[u]) = o;
    }
  }
  if (ts == 0) *counter = 0;  // every partition has arrived: ready for the next call
}

template <int D, typename T>
__global__ void __launch_bounds__(kWdThreads, 1)
    pkv_decode_wide_kernel(const __grid_constant__ CUtensorMap tmQ,
                           const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const WdArgs w) {
  using Sh = WdShape<D>;
  const DecodeArgs &a = w.d;
  // Launched as a programmatic dependent of the previous kernel on the
  // stream, a CTA reads only inputs (lengths, tables, queries, new rows)
  // and works out its schedule before griddep_wait; every access the
  // previous grid may conflict with (K/V loads, cache, workspace and output
  // writes) comes after it.  All CTAs are resident at once (at most one per
  // SM), so the next launch may be scheduled as soon as they are.
  griddep_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + Sh::kMiscOff);
  uint64_t *slot_full = bars + 0;    // [kSlots]: a K or V tile landed
  uint64_t *slot_empty = bars + 8;   // [kSlots]: the product that read it is done
  uint64_t *prod_done = bars + 14;   // the producer is at an item's last tile
  uint64_t *tmem_done = bars + 15;   // the softmax threads' last tensor-memory access is done
  uint64_t *q_full = bars + 16;      // the item's query rows landed
  uint64_t *q_empty = bars + 17;     // the item's last S^T is done
  uint64_t *s_full = bars + 18;      // [2]: S^T in score buffer b
  uint64_t *p_full = bars + 20;      // [2]: P^T written to buffer b
  uint64_t *p_free = bars + 22;      // [2]: the O^T product that read P^T buffer b is done
  uint64_t *o_done = bars + 24;      // the item's last O^T product is done
  uint64_t *item_full = bars + 25;   // [2]: an item published
  uint64_t *item_empty = bars + 27;  // [2]: every role has read it
  uint64_t *mma_done = bars + 29;
  uint64_t *grp_bar = bars + 30;     // the softmax warps' own barrier (128 arrivals a phase)
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 31);
  int *abort_flag = reinterpret_cast<int *>(tmem_holder + 1);
  WdItem *items = reinterpret_cast<WdItem *>(bars + 32);            // [2] (96 bytes)
  float *s_red = reinterpret_cast<float *>(bars + 44);              // [2][4 warps][16]
  int *s_vote = reinterpret_cast<int *>(s_red + 2 * 4 * kWdHeads);  // [2][4]
  float *s_m = reinterpret_cast<float *>(s_vote + 8);               // [16]
  int *s_scratch = reinterpret_cast<int *>(s_m + 2 * kWdHeads);     // [1 + 2 * 16] (16 floats unused before)
  float *s_o = reinterpret_cast<float *>(sm + Sh::kOOff);           // [16][D]
  // fused step, per item that ends its context (counted in item order):
  // [0] / [1] the producer has issued the last tile's K / V load, [2] / [3]
  // the append warp has written the new token's row over its row n - 1
  int *patch_cnt = reinterpret_cast<int *>(sm + Sh::kMiscOff + kWdPatchOff);
  // the CTA's last item, if it was the last partition of its context: merge
  // it (1 / 0), sequence, first head, partitions, counter index
  int *fin = reinterpret_cast<int *>(sm + Sh::kMiscOff + kWdFinOff);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (tid == 0) {
    for (int s = 0; s < Sh::kSlots; ++s) {
      mbar_init(&slot_full[s], 1);
      mbar_init(&slot_empty[s], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&p_free[i], 1);
      mbar_init(&item_full[i], 1);
      mbar_init(&item_empty[i], kWdReaders);
    }
    mbar_init(o_done, 1);
    mbar_init(mma_done, 1);
    mbar_init(grp_bar, 128);
    mbar_init(prod_done, 1);
    mbar_init(tmem_done, 128);
    for (int i = 0; i < 4; ++i) patch_cnt[i] = 0;
    fin[0] = 0;
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_holder, Sh::kTmemCols);
  // the scheduler's unit lengths (up to 8 x 32 units), in flight across the
  // set-up barrier: not predicated (the index is clamped), so all at once
  constexpr int kRegUnits = 8;
  int unit_raw[kRegUnits];
  if (warp == kWdSchedWarp) {
    const int last = max(w.units - 1, 0), per_seq = a.KVH * w.hchunks;
#pragma unroll
    for (int r = 0; r < kRegUnits; ++r) unit_raw[r] = __ldg(a.lens + min(32 * r + lane, last) / per_seq);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  constexpr bool bf16 = std::is_same<T, __nv_bfloat16>::value;

  auto abort_cta = [&]() {
    raise_flag(a.err, PKV_FLAG_TIMEOUT);
    *(volatile int *)abort_flag = 1;
  };
  auto aborted = [&]() { return *(volatile int *)abort_flag != 0; };

  if (warp == kWdSchedWarp) {
    // ------------------------------------------------------------ scheduler
    // the checks of the whole batch, once, by CTA 0 after its first item is
    // out: lengths, the host's bound on them, and (fused step) each new
    // token's slot against position n - 1
    // (fused step) the new rows of contexts the launch does not reach to
    // their end -- cut by the host's bound or the table -- are written here:
    // no item holds their position n - 1
    auto batch_checks = [&]() {
      const long long reach = (long long)a.max_parts * a.P;
      int over = 0;
      for (int b0 = 0; b0 < a.B; b0 += 32) {
        const int bb = b0 + lane;
        bool cut = false;
        long long slot = -1;
        if (bb < a.B) {
          const int n = checked_len(a, bb, true);
          over |= (long long)n > reach;
          if (w.check_append) {
            slot = __ldg(a.new_slots + bb);
            cut = slot >= 0 && wd_clamp_len(w, __ldg(a.lens + bb)) != max(__ldg(a.lens + bb), 0);
          }
        }
        for (unsigned m = __ballot_sync(0xffffffffu, cut); m; m &= m - 1) {
          const int src = __ffs(m) - 1;
          const int b = b0 + src;
          const long long sl = __shfl_sync(0xffffffffu, slot, src);
          const int n = checked_len(a, b, false);
          for (int kv = 0; kv < a.KVH; ++kv) append_write_row<T>(a, b, kv, sl, n, lane);
        }
      }
      if (__any_sync(0xffffffffu, over) && lane == 0) raise_flag(a.err, PKV_FLAG_CONTEXT_OVER_HINT);
    };
    // The claim order, numbered densely: first every full partition (P
    // tokens) -- round r holds partition maxp - 1 - r of the units long
    // enough, so the latest partitions, only long contexts have them, go
    // first -- then every unit's last, partial partition (or its empty
    // context) by its tile count, most first: the last items claimed are the
    // smallest.  The first item number of each round and of each tile
    // count comes from histograms of the units' lengths in shared memory (up
    // to 64 rounds and 63 tile counts; beyond, units in order).  Up to 256
    // units keep their lengths in the lanes' registers.
    const bool in_regs = w.units <= 32 * kRegUnits;
    int unit_n[kRegUnits];
#pragma unroll
    for (int r = 0; r < kRegUnits; ++r) {
      const int u = 32 * r + lane;
      unit_n[r] = (in_regs && u < w.units) ? wd_clamp_len(w, unit_raw[r]) : -1;
    }
    // The item size P: the plan's partition size, or (the plan's own choice)
    // about 1.2 times each CTA's share of the batch's 128-token tiles,
    // rounded to whole tiles and never below the plan's, so a sequence
    // never has more partitions than the workspace holds.  Measured on
    // log-uniform MQA batches: the best item was 1.18 to 1.21 shares on
    // three seeds; smaller items pay more item starts and merges than they
    // gain in balance, larger ones leave the last CTAs alone.  Every CTA
    // computes the same P from the same lengths.
    int P = a.P;
    if (w.auto_items && in_regs) {
      int tiles = 0;   // this lane's units (<= 8 x 2^24 tiles)
#pragma unroll
      for (int r = 0; r < kRegUnits; ++r) tiles += unit_n[r] > 0 ? (unit_n[r] + kWdTile - 1) / kWdTile : 0;
      // saturated before the sum, which then stays far inside 32 bits: a lane
      // past 2^20 tiles already puts the item size at its 63-tile cap
      tiles = min(tiles, 1 << 20);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tiles += __shfl_xor_sync(0xffffffffu, tiles, o);
      const int c = (int)gridDim.x;
      P = max(P, min((12 * tiles + 5 * c) / (10 * c), 63) * kWdTile);
    }
    const int maxp = a.max_parts;
    const int tmax = (P + kWdTile - 1) / kWdTile;       // tiles of a full partition
    const bool sorted = maxp <= 64 && tmax <= 63;
    auto len_of = [&](int base) -> int {              // unit base + lane's length, -1 past the end
      if (!in_regs) return base + lane < w.units ? wd_unit_len(w, base + lane) : -1;
      int v = -1;
#pragma unroll
      for (int r = 0; r < kRegUnits; ++r) v = (base == 32 * r) ? unit_n[r] : v;
      return v;
    };
    auto full_parts = [&](int n) { return n > 0 ? n / P : 0; };
    // the tile count of a unit's partial item: 1..tmax, 0 for an empty
    // context, -1 for none (the context is whole partitions)
    auto part_tiles = [&](int n) {
      if (n < 0) return -1;
      if (n == 0) return 0;
      const int rem = n % P;
      return rem == 0 ? -1 : (rem + kWdTile - 1) / kWdTile;
    };
    int *s_histA = reinterpret_cast<int *>(sm + Sh::kMiscOff + 1168);  // [65], after s_scratch
    int *s_cumA = s_histA + 65;   // [65] first item number of each round
    int *s_cumB = s_cumA + 65;    // [65] first item number of each tile count
    unsigned total = 0, total_full = 0;
    if (sorted) {
      for (int i = lane; i < 3 * 65; i += 32) s_histA[i] = 0;
      __syncwarp();
      for (int base = 0; base < w.units; base += 32) {
        const int n = len_of(base);
        const int f = full_parts(n);
        if (f > 0) atomicAdd(&s_histA[f - 1], 1);   // units with f full partitions (at f - 1)
        const int t = part_tiles(n);
        if (t >= 0) atomicAdd(&s_cumB[t], 1);       // partial items of t tiles (in place)
      }
      __syncwarp();
      // Prefix sums as warp scans, lane l holding entries l and l + 32 (a
      // serial loop in one lane cost about a microsecond before the first
      // claim).  Inclusive suffix sums first: su(i) = sum over j >= i.
      auto suffix64 = [&](int &x0, int &x1) {
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y0 = __shfl_down_sync(0xffffffffu, x0, o), y1 = __shfl_down_sync(0xffffffffu, x1, o);
          if (lane + o < 32) {
            x0 += y0;
            x1 += y1;
          }
        }
        x0 += __shfl_sync(0xffffffffu, x1, 0);
      };
      auto at64 = [&](int x0, int x1, int i) {   // entry i (0..63) of a lane-distributed pair
        const int a0 = __shfl_sync(0xffffffffu, x0, i & 31), a1 = __shfl_sync(0xffffffffu, x1, i & 31);
        return i < 32 ? a0 : a1;
      };
      // round r (r < maxp) holds the units with at least maxp - r full
      // partitions: su(maxp - r - 1) of the histogram over f - 1
      int u0 = s_histA[lane], u1 = s_histA[lane + 32];
      suffix64(u0, u1);
      const int w0 = at64(u0, u1, max(maxp - lane - 1, 0)), w1 = at64(u0, u1, max(maxp - lane - 33, 0));
      int c0 = lane < maxp ? w0 : 0, c1 = lane + 32 < maxp ? w1 : 0;
      // first item number of each round: the exclusive prefix of the counts
      int e0 = c0, e1 = c1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y0 = __shfl_up_sync(0xffffffffu, e0, o), y1 = __shfl_up_sync(0xffffffffu, e1, o);
        if (lane >= o) {
          e0 += y0;
          e1 += y1;
        }
      }
      const int half = __shfl_sync(0xffffffffu, e0, 31);
      e1 += half;
      total_full = (unsigned)__shfl_sync(0xffffffffu, e1, 31);
      // classes by tile count, most first: first item number of count t =
      // total_full + the partial items with more tiles
      int b0 = s_cumB[lane], b1 = s_cumB[lane + 32];
      int v0 = b0, v1 = b1;
      suffix64(v0, v1);
      total = total_full + (unsigned)__shfl_sync(0xffffffffu, v0, 0);
      __syncwarp();
      s_cumA[lane] = e0 - c0;
      s_cumA[lane + 32] = e1 - c1;
      if (lane == 0) s_cumA[64] = (int)total_full;
      s_cumB[lane] = (int)total_full + v0 - b0;
      s_cumB[lane + 32] = (int)total_full + v1 - b1;
      __syncwarp();
      if (lane == 0 && maxp < 64) s_cumA[maxp] = (int)total_full;
      __syncwarp();
    } else {
      for (int base = 0; base < w.units; base += 32) {
        const int n = len_of(base);
        int np = n < 0 ? 0 : (n > 0 ? (n + P - 1) / P : 1);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) np += __shfl_xor_sync(0xffffffffu, np, o);
        total += (unsigned)np;
      }
    }
    // units in order (no sort): claims rise, so the search resumes
    int chunk_base = 0;
    unsigned chunk_cum = 0;   // items of the units before chunk_base
    unsigned k = blockIdx.x;
    int it = 0, iq = 0;
    bool ok = true;
    while (true) {
      WdItem item;
      memset(&item, 0, sizeof item);
      item.kind = -1;
      if (k < total && sorted) {
        // the idx-th unit (in unit order) satisfying `pred`, made an item
        auto pick = [&](unsigned idx, auto pred, auto part_of) {
          for (int base = 0; base < w.units; base += 32) {
            const int n = len_of(base);
            const unsigned m = __ballot_sync(0xffffffffu, pred(n));
            const unsigned c = (unsigned)__popc(m);
            if (idx < c) {
              const int src = (int)__fns(m, 0, idx + 1);
              const int nn = __shfl_sync(0xffffffffu, n, src);
              item = wd_make_item(w, base + src, part_of(nn), nn, P);
              return;
            }
            idx -= c;
          }
        };
        if (k < total_full) {
          // the round: the last whose first item number is <= k
          const unsigned m0 = __ballot_sync(0xffffffffu, lane < maxp && (unsigned)s_cumA[lane] <= k);
          const unsigned m1 = __ballot_sync(0xffffffffu, lane + 32 < maxp && (unsigned)s_cumA[lane + 32] <= k);
          const int r = m1 ? 63 - __clz(m1) : 31 - __clz(m0);
          const int p = maxp - 1 - r;
          pick(k - (unsigned)s_cumA[r], [&](int n) { return full_parts(n) > p; }, [&](int) { return p; });
        } else {
          // the tile count: the last class whose first item number is <= k
          // (class c holds tile count tmax - c; s_cumB is indexed by count)
          const unsigned m0 = __ballot_sync(0xffffffffu, lane <= tmax && (unsigned)s_cumB[tmax - lane] <= k);
          const unsigned m1 = __ballot_sync(0xffffffffu, lane + 32 <= tmax && (unsigned)s_cumB[tmax - lane - 32] <= k);
          const int c = m1 ? 63 - __clz(m1) : 31 - __clz(m0);
          const int t = tmax - c;
          pick(k - (unsigned)s_cumB[t], [&](int n) { return part_tiles(n) == t; },
               [&](int n) { return n > 0 ? n / P : 0; });
        }
      } else if (k < total) {
        while (true) {
          const int n = len_of(chunk_base);
          const int np = n < 0 ? 0 : (n > 0 ? (n + P - 1) / P : 1);
          int incl = np;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
          }
          const unsigned chunk_total = (unsigned)__shfl_sync(0xffffffffu, incl, 31);
          if (k < chunk_cum + chunk_total) {
            const unsigned hit = __ballot_sync(0xffffffffu, chunk_cum + (unsigned)incl > k);
            const int src = __ffs(hit) - 1;
            const int excl = __shfl_sync(0xffffffffu, incl - np, src);
            const int nn = __shfl_sync(0xffffffffu, n, src);
            item = wd_make_item(w, chunk_base + src, (int)(k - chunk_cum) - excl, nn, P);
            break;
          }
          chunk_cum += chunk_total;
          chunk_base += 32;
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
      if (it == 1 && blockIdx.x == 0) {
        griddep_wait();
        batch_checks();
      }
      if (item.kind < 0) break;
      if (item.kind == 1) {
        // the item's 16 query rows, once the last S^T of the previous is done
        if (iq > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(q_empty, (iq - 1) & 1)) && !aborted();
          if (!ok) break;
        }
        if (lane == 0) mbar_arrive_expect_tx(q_full, (uint32_t)Sh::kQBytes);
        __syncwarp();
        const int head0 = item.kvh * a.G + item.hc * kWdHeads;
        if (lane < Sh::kRegions)
          wd_tma_3d(sm + Sh::kQOff + lane * Sh::kQRegion, &tmQ, q_full, 64 * lane, head0, item.b);
        ++iq;
      }
      // the next item is claimed once the producer is at this one's last
      // tile: a CTA holds one item ahead, not two, which keeps the last items
      // for the CTAs that are free
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(prod_done, (it - 1) & 1)) && !aborted();
      if (!ok) break;
      unsigned nk = 0;
      if (lane == 0) nk = atomicAdd(w.sched, 1u) + gridDim.x;
      k = __shfl_sync(0xffffffffu, nk, 0);
    }
    if (!ok && lane == 0) abort_cta();
    if (iq > 0) mbar_wait_bounded(q_full, (iq - 1) & 1);  // the last query rows land (bounded)
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    // per tile: K into the next ring slot, then V into the one after; a slot
    // is reused once the product that read it is done
    // a tile of one tensor is nch chunks of box_tok tokens (one box each,
    // never across a cache block) times kRegions blocks of 64 values
    const int bt = w.box_tok, nch = kWdTile / bt;
    const int per_tensor = nch * Sh::kRegions;           // boxes per tile (<= 32)
    const int region = (lane % per_tensor) / nch, chunk = lane % nch;
    const uint64_t policy = l2_evict_first_policy();
    if (lane == 0) {
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
    }
    int it = 0, loads = 0, npatch = 0;
    bool ok = true, dep_done = false;
    while (ok) {
      const int slot = it & 1;
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&item_full[slot], (it >> 1) & 1));
      if (!ok) break;
      const WdItem item = items[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[slot]);
      ++it;
      if (item.kind < 0) break;
      if (item.kind != 1) {
        if (lane == 0) mbar_arrive(prod_done);
        continue;
      }
      const int nt = item.ntiles;
      // the physical blocks, read four tiles ahead of their use (a lookup
      // per load would hold each load for a round trip): lane 8 * (j % 4) + c
      // holds the table entry of tokens 16c .. 16c + 15 of tile j; tokens past
      // the context read the last entry inside it; checked where used
      const size_t trow = (size_t)item.b * a.max_blocks;
      auto entry_of = [&](int j) {
        const int t = min(item.t0 + j * kWdTile + 16 * (lane & 7), item.t1 - 1);
        return __ldg(a.tables + trow + t / a.bs);
      };
      int ahead = (lane >> 3) < nt ? entry_of(lane >> 3) : 0;
      if (!dep_done) {  // the previous grid's cache writes land before the first K/V load
        // Before waiting: the first item's first two tiles of K and V are
        // asked into L2 by TMA prefetches of the very boxes the loads will
        // read, so those loads find them there.  A line the previous grid
        // still writes is updated in L2, which the loads after the wait read.
        for (int j = 0; j < min(nt, 2); ++j) {
          const int tok0 = item.t0 + j * kWdTile;
          const int valid_chunks = min(nch, (item.t1 - tok0 + bt - 1) / bt);
          const int phys = __shfl_sync(0xffffffffu, ahead, 8 * j + (bt >> 4) * chunk);
          if (lane < per_tensor && chunk < valid_chunks && phys >= 0 && (long long)phys < a.num_blocks) {
            const int t = tok0 + bt * chunk;
            const int lb = t / a.bs;
            wd_tma_prefetch_4d(&tmK, region * 64, item.kvh, t - lb * a.bs, phys);
            wd_tma_prefetch_4d(&tmV, region * 64, item.kvh, t - lb * a.bs, phys);
          }
        }
        griddep_wait();
        dep_done = true;
      }
      for (int idx = 0; idx < 2 * nt && ok; ++idx) {
        // which tile, K or V
        int j, v;
        if (idx == 2 * nt - 1) {
          j = nt - 1;
          v = 1;
        } else if (idx < 2) {
          j = idx;
          v = 0;
        } else if ((idx & 1) == 0) {
          j = (idx - 2) >> 1;
          v = 1;
        } else {
          j = (idx + 1) >> 1;
          v = 0;
        }
        const int tok0 = item.t0 + j * kWdTile;
        const int valid_chunks = min(nch, (item.t1 - tok0 + bt - 1) / bt);
        const uint32_t bytes = (uint32_t)(valid_chunks * Sh::kRegions * bt * 128);
        int phys = __shfl_sync(0xffffffffu, ahead, 8 * (j & 3) + (bt >> 4) * chunk);
        if (phys < 0 || (long long)phys >= a.num_blocks) {  // outside the pool: flagged, block 0 read
          if (lane < valid_chunks) raise_flag(a.err, PKV_FLAG_BLOCK_OUT_OF_RANGE);
          phys = 0;
        }
        const int s = loads % Sh::kSlots, use = loads / Sh::kSlots;
        if (use > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(&slot_empty[s], (use - 1) & 1)) && !aborted();
          if (!ok) break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&slot_full[s], bytes);
        __syncwarp();
        if (lane < per_tensor && chunk < valid_chunks) {
          const int t = tok0 + bt * chunk;
          const int lb = t / a.bs;
          uint8_t *dst = sm + s * Sh::kTileBytes + region * Sh::kRegionBytes + chunk * bt * 128;
          wd_tma_4d(dst, v ? &tmV : &tmK, &slot_full[s], region * 64, item.kvh, t - lb * a.bs, phys,
                    policy);
        }
        ++loads;
        // the append warp may wait for the last tile's K (V) to land only
        // once it is issued: its slot's earlier phases are complete then
        if (item.patch_row >= 0 && j == nt - 1) {
          __syncwarp();
          if (lane == 0) wd_count_store(patch_cnt + v, npatch + 1);
          if (v) ++npatch;
        }
        // tile j's entries are done with once its values are on the way:
        // the lanes of its group read those of tile j + 4
        if (v && (lane >> 3) == (j & 3) && j + 4 < nt) ahead = entry_of(j + 4);
        // the scheduler may claim the next item once the last tile's loads
        // are next (the claim's latency overlaps them)
        if (idx == max(0, 2 * nt - 3) && lane == 0) mbar_arrive(prod_done);
      }
    }
    if (!ok && lane == 0) abort_cta();
    // the last fills land before the CTA can end (bounded)
    for (int l = max(0, loads - Sh::kSlots); l < loads; ++l)
      mbar_wait_bounded(&slot_full[l % Sh::kSlots], (l / Sh::kSlots) & 1);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = umma_idesc_f16(128, kWdHeads, bf16, false);       // K, Q: K-major
      const uint32_t idesc_o = umma_idesc_f16_mn(128, kWdHeads, bf16, true, false);  // V MN-major
      const uint32_t q_base = smem_u32(sm + Sh::kQOff), p_base = smem_u32(sm + Sh::kPOff);
      int it = 0, loads = 0, st = 0, pt = 0, iq = 0, npk = 0, npv = 0;  // patches waited for
      bool ok = true;
      while (ok) {
        const int slot = it & 1;
        ok = mbar_wait_bounded(&item_full[slot], (it >> 1) & 1);
        if (!ok) break;
        const WdItem item = items[slot];
        mbar_arrive(&item_empty[slot]);
        ++it;
        if (item.kind < 0) break;
        if (item.kind != 1) continue;
        const int L0 = loads;   // the item's loads are L0 + wd_kidx(j) (K), L0 + wd_vidx(j, n) (V)
        ok = mbar_wait_bounded(q_full, iq & 1) && !aborted();
        ++iq;
        if (!ok) break;
        // S^T of tile j into the next score buffer
        auto issue_s = [&](int j) -> bool {
          const int l = L0 + wd_kidx(j), s = l % Sh::kSlots;
          if (!mbar_wait_bounded(&slot_full[s], (l / Sh::kSlots) & 1)) return false;
          // fused step: the last tile's K row n - 1 is the new token's
          if (j == item.ntiles - 1 && item.patch_row >= 0 && !wd_count_wait(patch_cnt + 2, ++npk))
            return false;
          tc_fence_after();
          const int buf = st & 1;
          const uint32_t kb = smem_u32(sm + s * Sh::kTileBytes);
#pragma unroll
          for (int k = 0; k < D / 16; ++k)
            umma_f16(tmem + 16 * buf,
                     umma_desc_sw128(kb + (k >> 2) * Sh::kRegionBytes + (k & 3) * 32, 16, 1024),
                     umma_desc_sw128(q_base + (k >> 2) * Sh::kQRegion + (k & 3) * 32, 16, 1024),
                     idesc_s, k > 0);
          umma_commit(&s_full[buf]);
          umma_commit(&slot_empty[s]);
          ++st;
          if (j == item.ntiles - 1) umma_commit(q_empty);  // the item's last S^T
          return true;
        };
        ok = issue_s(0) && (item.ntiles < 2 || issue_s(1));
        for (int j = 0; ok && j < item.ntiles; ++j) {
          ok = mbar_wait_bounded(&p_full[pt & 1], (pt >> 1) & 1) && !aborted();
          if (!ok) break;
          const int l = L0 + wd_vidx(j, item.ntiles), s = l % Sh::kSlots;
          ok = mbar_wait_bounded(&slot_full[s], (l / Sh::kSlots) & 1);
          if (ok && j == item.ntiles - 1 && item.patch_row >= 0)
            ok = wd_count_wait(patch_cnt + 3, ++npv);  // the new token's V row
          if (!ok) break;
          tc_fence_after();
          // O^T (+)= V^T . P^T, per block of 128 of the D values
          const uint32_t vb = smem_u32(sm + s * Sh::kTileBytes), pb = p_base + (pt & 1) * Sh::kPBytes;
#pragma unroll
          for (int hh = 0; hh < D / 128; ++hh)
#pragma unroll
            for (int k = 0; k < kWdTile / 16; ++k)
              umma_f16(tmem + 32 + 16 * hh,
                       umma_desc_sw128(vb + 2 * hh * Sh::kRegionBytes + k * 2048, Sh::kRegionBytes, 1024),
                       umma_desc_sw128(pb + (k >> 2) * Sh::kPRegion + (k & 3) * 32, 16, 1024),
                       idesc_o, (j > 0 || k > 0));
          umma_commit(&p_free[pt & 1]);
          umma_commit(&slot_empty[s]);
          ++pt;
          if (j + 2 < item.ntiles) ok = issue_s(j + 2);
          if (j == item.ntiles - 1) umma_commit(o_done);
        }
        loads = L0 + 2 * item.ntiles;
      }
      if (!ok) abort_cta();
      umma_commit(mma_done);  // every product issued above has completed when this arrives
      mbar_wait_bounded(mma_done, 0);
    }
    __syncwarp();
    // the tensor memory is freed as soon as no product and no softmax thread
    // uses it any more (the softmax threads' last merge and stores go on)
    mbar_wait_bounded(tmem_done, 0);
    tc_fence_after();
    tmem_dealloc(tmem, Sh::kTmemCols);
  } else if (warp == kWdAppendWarp) {
    // ------------------------------------------------------------ append
    // Fused step only (no items carry a patch row otherwise).  Per item that
    // ends its context: the new token's K and V rows of the item's KV head
    // are loaded; the item of head chunk 0 writes them to the cache row
    // (after the slot checks); once the last tile's K (then V) has landed
    // its row n - 1 is overwritten with the new row in shared memory (so
    // nothing waits for the cache write, and whatever a load read of that
    // row is replaced) and the MMA thread is released.  Empty contexts with
    // a new token are written (and flagged) here too.
    constexpr int kRowVecs = D / 8;        // 16-byte vectors of one head's row (<= 32)
    int it = 0, loads = 0, npatch = 0;
    bool ok = true;
    griddep_wait();  // it writes cache rows
    while (true) {
      const int slot = it & 1;
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&item_full[slot], (it >> 1) & 1));
      if (!ok) break;
      const WdItem item = items[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[slot]);
      ++it;
      if (item.kind < 0) break;
      const long long snew = w.check_append ? append_slot(a, item.b) : -1LL;
      if (item.kind == 2) {  // empty context: no rows read; the token is still written (flagged)
        if (snew >= 0 && item.hc == 0) append_write_row<T>(a, item.b, item.kvh, snew, 0, lane);
        continue;
      }
      if (item.kind != 1) continue;
      const int L0 = loads;
      loads += 2 * item.ntiles;
      if (item.patch_row < 0) continue;
      // Every load the item needs is in flight at once (one round trip, not
      // three): the new token's slot (above), the context's length, the new K and V
      // rows (row b of the new-token inputs exists for every sequence), and
      // for head chunk 0 the table entry of position n - 1 that the cache
      // write is checked against.  The rows are patched into the landed
      // tiles first -- the MMA thread waits for them -- and the cache row is
      // written after (nothing in this launch reads it from the cache).
      // A context cut short by the host's bound never reaches here with its
      // true length (the batch checks write its row).
      const int len_b = __ldg(a.lens + item.b);
      uint4 kv = make_uint4(0, 0, 0, 0), vv = kv;
      if (lane < kRowVecs) {
        kv = __ldg(append_src<T>(a, false, item.b, item.kvh) + lane);
        vv = __ldg(append_src<T>(a, true, item.b, item.kvh) + lane);
      }
      const int phys_last = (item.hc == 0 && lane == 0)
                                ? __ldg(a.tables + (size_t)item.b * a.max_blocks + (item.n - 1) / a.bs)
                                : 0;
      const bool has = snew >= 0 && max(len_b, 0) == item.n;
      const int r = item.patch_row;
      ++npatch;
      // 16-byte column lane & 7 of the 64-value region lane >> 3, row r,
      // 128-byte swizzle (the tile's regions are 1024-byte aligned)
      const uint32_t off = (uint32_t)((lane >> 3) * Sh::kRegionBytes + r * 128 +
                                      (((lane & 7) ^ (r & 7)) << 4));
      for (int v = 0; v < 2 && ok; ++v) {
        const int l = L0 + (v ? wd_vidx(item.ntiles - 1, item.ntiles) : wd_kidx(item.ntiles - 1));
        if (has) {
          // issued (so the slot holds no older load), then landed
          ok = __all_sync(0xffffffffu, wd_count_wait(patch_cnt + v, npatch)) &&
               __all_sync(0xffffffffu,
                          mbar_wait_bounded(&slot_full[l % Sh::kSlots], (l / Sh::kSlots) & 1)) &&
               !aborted();
          if (!ok) break;
          if (lane < kRowVecs)
            st_shared_v4(smem_u32(sm + (l % Sh::kSlots) * Sh::kTileBytes) + off, v ? vv : kv);
          fence_proxy_async_shared();  // the row before the product reads it
          __syncwarp();
        }
        if (lane == 0) wd_count_store(patch_cnt + 2 + v, npatch);
      }
      if (!ok) break;
      if (has && item.hc == 0) {
        int wr = 0;
        if (lane == 0) wr = append_check_entry(a, item.kvh, snew, item.n, phys_last);
        if (__shfl_sync(0xffffffffu, wr, 0) && lane < kRowVecs)
          append_store<T>(a, item.kvh, snew, lane, kv, vv);
      }
    }
    if (!ok && lane == 0) abort_cta();
  } else {
    // ------------------------------------------------------------ softmax
    griddep_wait();  // output rows, partials and counters of the workspace
    const int q4 = warp & 3;                       // tensor-memory lane quarter
    const int t = 32 * q4 + lane;                  // token lane of the tile; D lane of O^T
    const int ts = (warp - 2) * 32 + lane;         // thread of the softmax group
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const float sl2 = a.scale_log2;
    T *out = reinterpret_cast<T *>(a.out);
    int it = 0, loads = 0, tg = 0, io = 0;
    int gphase = 0;   // phases of grp_bar this thread has passed
    const WdGroupSync group_sync{grp_bar, &gphase};
    // a partition count still in flight (thread 0 holds the atomic's result)
    bool pend = false;
    int pend_b = 0, pend_head0 = 0, pend_nparts = 0;
    int *pend_cnt = nullptr;
    unsigned pend_prev = 0;
    // the pending count's result: the last partition merges (the weights go
    // to the P^T buffers, free between items).  Thread 0 posts whether to
    // merge (s_scratch[0]) before the item end's first barrier; settle runs
    // after it.
    auto settle = [&]() {
      if (!pend) return;
      if (s_scratch[0]) {
        wd_merge<D, T, 128>(a, pend_b, pend_head0, pend_nparts, reinterpret_cast<float *>(sm + Sh::kPOff),
                       2 * Sh::kPBytes / 4, s_scratch, pend_cnt, ts, group_sync);
        group_sync();
      }
      pend = false;
    };
    bool ok = true;
    while (true) {
      const int slot = it & 1;
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&item_full[slot], (it >> 1) & 1));
      if (!ok) break;
      const WdItem item = items[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[slot]);
      ++it;
      if (item.kind < 0) break;
      const int head0 = item.kvh * a.G + item.hc * kWdHeads;
      if (item.kind == 2) {  // empty context: zero output rows
        for (int i = ts; i < kWdHeads * D; i += 128)
          out[((size_t)item.b * a.H + head0) * D + i] = from_f32<T>(0.f);
        continue;
      }
      if (item.kind != 1) continue;
      const int L0 = loads;
      float m_used[kWdHeads], l_part[kWdHeads];
#pragma unroll
      for (int h = 0; h < kWdHeads; ++h) {
        m_used[h] = -INFINITY;
        l_part[h] = 0.f;
      }
      for (int j = 0; j < item.ntiles; ++j, ++tg) {
        const int buf = tg & 1;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&s_full[buf], (tg >> 1) & 1)) && !aborted();
        if (!ok) break;
        tc_fence_after();
        float x[kWdHeads];
        tmem_ld16(tmem + lane_off + 16 * buf, x);
        const int tok = item.t0 + j * kWdTile + t;
        const bool valid = tok < item.t1;
        bool need = false;
#pragma unroll
        for (int h = 0; h < kWdHeads; ++h) {
          x[h] = valid ? x[h] * sl2 : -INFINITY;
          need |= x[h] > m_used[h] + 8.f;
        }
        // does any score of the tile pass its head's running max by 2^8?
        // (always on an item's first tile, whose running maxima are -inf: no
        // vote there)
        const int par = tg & 1;
        bool any = true;
        if (j > 0) {
          const int need_w = __any_sync(0xffffffffu, need);
          if (lane == 0) s_vote[par * 4 + (warp - 2)] = need_w;
          group_sync();
          any = s_vote[par * 4] | s_vote[par * 4 + 1] | s_vote[par * 4 + 2] | s_vote[par * 4 + 3];
        }
        if (any) {
          // per-head max of the tile over the 128 token lanes
#pragma unroll
          for (int h = 0; h < kWdHeads; ++h) {
            float v = x[h];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == 0) s_red[(par * 4 + (warp - 2)) * kWdHeads + h] = v;
          }
          group_sync();
          bool moved = false;
          float alpha[kWdHeads];
#pragma unroll
          for (int h = 0; h < kWdHeads; ++h) {
            const float* r = s_red + par * 4 * kWdHeads + h;
            const float tmax = fmaxf(fmaxf(r[0], r[kWdHeads]), fmaxf(r[2 * kWdHeads], r[3 * kWdHeads]));
            const float m_new = tmax > m_used[h] + 8.f ? tmax : m_used[h];
            alpha[h] = fast_exp2(m_used[h] - m_new);
            moved |= m_new != m_used[h];
            l_part[h] *= alpha[h];
            m_used[h] = m_new;
          }
          if (moved && j > 0) {
            // O^T holds tiles 0 .. j-1 once the product of tile j-1 is done
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(&p_free[(tg - 1) & 1], ((tg - 1) >> 1) & 1));
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int hh = 0; hh < D / 128; ++hh) {
              float o[kWdHeads];
              tmem_ld16(tmem + lane_off + 32 + 16 * hh, o);
#pragma unroll
              for (int h = 0; h < kWdHeads; ++h) o[h] *= alpha[h];
              tmem_st16(tmem + lane_off + 32 + 16 * hh, o);
            }
          }
        }
        // P^T buffer: free once the product two tiles back is done
        if (tg >= 2) {
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(&p_free[buf], ((tg - 2) >> 1) & 1));
          if (!ok) break;
        }
        uint8_t *pb = sm + Sh::kPOff + buf * Sh::kPBytes + (t >> 6) * Sh::kPRegion + (t & 7) * 2;
        const int c16 = (t & 63) >> 3;
#pragma unroll
        for (int h = 0; h < kWdHeads; ++h) {
          const float p = fast_exp2(x[h] - m_used[h]);
          l_part[h] += p;
          *reinterpret_cast<unsigned short *>(pb + h * 128 + ((c16 ^ (h & 7)) << 4)) = wd_bits<T>(p);
        }
        // the tile's V rows past the partition are zeroed (they may hold
        // anything, and 0 * NaN would poison the product): in each 64-value
        // region they are one contiguous run of 128-byte rows, written by
        // the 128 threads as consecutive 16-byte vectors (a row per thread
        // put eight lanes of every store on the same banks: ~2 us a tile)
        const int vl = L0 + wd_vidx(j, item.ntiles);
        if (item.t0 + (j + 1) * kWdTile > item.t1) {
          const int vs = vl % Sh::kSlots;
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(&slot_full[vs], (vl / Sh::kSlots) & 1));
          if (!ok) break;
          const int v_rows = item.t1 - (item.t0 + j * kWdTile);   // 1 .. 127
          const int vecs = (kWdTile - v_rows) * 8;                // per region
          uint8_t *vtail = sm + vs * Sh::kTileBytes + v_rows * 128;
#pragma unroll
          for (int r = 0; r < Sh::kRegions; ++r)
            for (int i = ts; i < vecs; i += 128)
              *reinterpret_cast<uint4 *>(vtail + r * Sh::kRegionBytes + i * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_shared();  // P^T and zeroed rows before the product reads them
        tc_fence_before();
        mbar_arrive(&p_full[buf]);
      }
      if (!ok) break;
      loads = L0 + 2 * item.ntiles;
      // the item's end: per-head sums over the 128 lanes, O^T to shared
      // memory, then the output rows or the partition's partials (merged by
      // the sequence's last partition)
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(o_done, io & 1)) && !aborted();
      ++io;
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int h = 0; h < kWdHeads; ++h) {
        float v = l_part[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) s_red[(warp - 2) * kWdHeads + h] = v;
      }
#pragma unroll
      for (int hh = 0; hh < D / 128; ++hh) {
        float o[kWdHeads];
        tmem_ld16(tmem + lane_off + 32 + 16 * hh, o);
#pragma unroll
        for (int h = 0; h < kWdHeads; ++h) s_o[h * D + 128 * hh + t] = o[h];
      }
      if (ts == 0) {
#pragma unroll
        for (int h = 0; h < kWdHeads; ++h) s_m[h] = m_used[h];
        if (pend) s_scratch[0] = pend_prev == (unsigned)(pend_nparts - 1);
      }
      group_sync();
      settle();  // the previous item's merge, if it was the last partition
      int *cnt = a.ws_cnt + (size_t)item.b * (a.KVH * w.hchunks) + item.kvh * w.hchunks + item.hc;
      if (wd_publish<D, T>(a, item.b, head0, item.part, item.nparts, s_m, s_red, s_o, cnt, ts,
                           group_sync, &pend_prev)) {
        pend = true;
        pend_b = item.b;
        pend_head0 = head0;
        pend_nparts = item.nparts;
        pend_cnt = cnt;
      }
      group_sync();  // shared memory free for the next item
    }
    tc_fence_before();
    mbar_arrive(tmem_done);  // no tensor-memory access after this
    // the last item's merge, if it was the last partition, is left to the
    // whole CTA after the barrier below (the other roles are done by then):
    // twice the threads, half the rounds of partial loads
    if (ts == 0) {
      fin[0] = ok && pend && pend_prev == (unsigned)(pend_nparts - 1);
      fin[1] = pend_b;
      fin[2] = pend_head0;
      fin[3] = pend_nparts;
      fin[4] = pend ? (int)(pend_cnt - a.ws_cnt) : 0;
    }
    if (!ok && lane == 0) abort_cta();
  }

  __syncthreads();
  griddep_wait();  // (returned already for the roles that touch global memory)
  if (fin[0])
    wd_merge<D, T, kWdThreads>(a, fin[1], fin[2], fin[3], reinterpret_cast<float *>(sm + Sh::kPOff),
                               2 * Sh::kPBytes / 4, s_scratch, a.ws_cnt + fin[4], tid, CtaSync());
  if (tid == 0) {
    // the last CTA of the launch puts the work counters back for the next
    // (every claim of this CTA was an atomic whose value it used before the
    // barrier, so it is performed already: no fence, which at the end of a
    // launch can hold a thread for tens of microseconds)
    if (atomicAdd(w.sched + 1, 1u) == gridDim.x - 1) {
      atomicExch(w.sched, 0u);
      atomicExch(w.sched + 1, 0u);
    }
  }
}

// ---------------------------------------------------------------- host side

typedef CUresult (*WdEncodeFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                               const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                               const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                               CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static WdEncodeFn wd_encode_fn() {
  static WdEncodeFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<WdEncodeFn>(p);
  }
  return fn;
}

// Tensor map of the [B, H, D] queries: box of 64 elements x 16 heads x 1
// sequence, 128-byte swizzle.
static bool encode_query_group_map(CUtensorMap *map, const void *q, pkv_dtype dt, int B, int H,
                                   int D) {
  WdEncodeFn fn = wd_encode_fn();
  if (!fn) return false;
  const cuuint64_t el = 2;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)B};
  cuuint64_t strides[2] = {D * el, (cuuint64_t)H * D * el};
  cuuint32_t box[3] = {64, (cuuint32_t)kWdHeads, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map,
            dt == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
            const_cast<void *>(q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map of a [num_blocks, bs, KVH, D] cache: box of 64 values x 1 head
// x box_tok tokens x 1 block, 128-byte swizzle (a box lands as box_tok
// consecutive 128-byte rows of one 64-value block of a tile).
static bool encode_wide_cache_map(CUtensorMap *map, const void *cache, pkv_dtype dt,
                                  long long num_blocks, int bs, int KVH, int D, int box_tok) {
  WdEncodeFn fn = wd_encode_fn();
  if (!fn) return false;
  const cuuint64_t el = 2;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)KVH, (cuuint64_t)bs, (cuuint64_t)num_blocks};
  cuuint64_t strides[3] = {D * el, (cuuint64_t)KVH * D * el, (cuuint64_t)bs * KVH * D * el};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)box_tok, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map,
            dt == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
            const_cast<void *>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tokens per K/V box: the largest of 128, 64, 32, 16 dividing both the block
// size and the partition size, so that every box starts on a multiple of it
// (tiles start at multiples of the partition size plus 128) and stays in one
// block.  Fewer, larger boxes: with 16-token (2 KB) boxes the TMA unit's
// per-box cost, not HBM, paced each CTA's loads (a 64 KB tile took ~1.4 us to
// issue; ~0.9 us with 32-token boxes).
static int wd_box_tokens(int bs, int P) {
  for (int bt = kWdTile; bt > 16; bt >>= 1)
    if (bs % bt == 0 && P % bt == 0) return bt;
  return 16;
}

static unsigned *wd_sched_counters() {
  static unsigned *cached[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  if (dev < 64 && cached[dev]) return cached[dev];
  unsigned *p = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_wd_sched) != cudaSuccess) return nullptr;
  if (dev < 64) cached[dev] = p;
  return p;
}

size_t wide_smem_bytes(int D) {
  return D == 256 ? (size_t)WdShape<256>::kSmem : (size_t)WdShape<128>::kSmem;
}

template <int D, typename T>
static pkv_status launch_wide_t(const WdArgs &w, const CUtensorMap &mq, const CUtensorMap &mk,
                                const CUtensorMap &mv, int ctas, cudaStream_t stream) {
  auto kern = pkv_decode_wide_kernel<D, T>;
  static int configured[64] = {0};
  if (!allow_smem(kern, WdShape<D>::kSmem, configured)) return PKV_ERR_CUDA;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kWdThreads);
  cfg.dynamicSmemBytes = WdShape<D>::kSmem;
  cfg.stream = stream;
  // a programmatic dependent of the previous kernel on the stream: its
  // start-up overlaps that kernel's tail (see the kernel's griddep_wait)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = launch_as_dependent(stream) ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, w) != cudaSuccess) return PKV_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status launch_decode_wide(const DecodeArgs &a, pkv_dtype dt, int num_sms, bool auto_items,
                              cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  const int box_tok = wd_box_tokens(a.bs, a.P);
  if (!encode_query_group_map(&mq, a.q, dt, a.B, a.H, a.D) ||
      !encode_wide_cache_map(&mk, a.k_cache, dt, a.num_blocks, a.bs, a.KVH, a.D, box_tok) ||
      !encode_wide_cache_map(&mv, a.v_cache, dt, a.num_blocks, a.bs, a.KVH, a.D, box_tok))
    return PKV_ERR_CUDA;
  unsigned *sched = wd_sched_counters();
  if (!sched) return PKV_ERR_CUDA;
  // a counter slot per launch, taken in turn (launches in flight at once on
  // one device must number fewer than kWdSchedSlots)
  static std::atomic<unsigned> next_slot{0};
  const unsigned slot = next_slot.fetch_add(1u) % kWdSchedSlots;
  WdArgs w;
  memset(&w, 0, sizeof w);
  w.d = a;
  w.sched = sched + 2 * slot;
  w.hchunks = a.G / kWdHeads;
  w.units = a.B * a.KVH * w.hchunks;
  w.check_append = a.new_slots != nullptr;
  w.box_tok = box_tok;
  w.auto_items = auto_items;
  // one persistent CTA per SM, never more than the items there can be
  const long long items = (long long)w.units * a.max_parts;
  const int ctas = (int)std::min<long long>(items, num_sms > 0 ? num_sms : 1);
  const bool bf = dt == PKV_BF16;
  if (a.D == 256) return bf ? launch_wide_t<256, __nv_bfloat16>(w, mq, mk, mv, ctas, stream)
                            : launch_wide_t<256, __half>(w, mq, mk, mv, ctas, stream);
  if (a.D == 128) return bf ? launch_wide_t<128, __nv_bfloat16>(w, mq, mk, mv, ctas, stream)
                            : launch_wide_t<128, __half>(w, mq, mk, mv, ctas, stream);
  return PKV_ERR_UNSUPPORTED;
}

}  // namespace pkv
