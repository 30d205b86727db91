// pkv_device.cuh -- device-side building blocks shared by the decode kernels:
// PTX wrappers (mbarrier, TMA, ldmatrix, mma.sync, ex2), bounded waits, the
// per-launch argument block and the end-of-partition epilogue (direct
// output, or partial results + log-sum-exp merge by the last CTA).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

constexpr float kLog2e = 1.4426950408889634f;
// A wait on an asynchronous copy gives up after this long (the copies take
// microseconds); the kernel then reports PKV_FLAG_TIMEOUT and winds down.
constexpr unsigned long long kWaitLimitNs = 500ull * 1000ull * 1000ull;

// Everything a decode launch needs, passed by value.
struct DecodeArgs {
  void *out;
  const void *q;
  const void *k_cache;   // used by the CUDA-core kernel (the TMA kernel uses tensor maps)
  const void *v_cache;
  const int32_t *tables;
  const int32_t *lens;
  float *ws_m;           // [B][H][max_parts]   running max (log2 units)
  float *ws_l;           // [B][H][max_parts]   sum of weights
  float *ws_o;           // [B][H][max_parts][D] weighted sum of V rows (unnormalised)
  int *ws_cnt;           // [B][heads_chunks]    finished-partition counters
  int *err;
  long long num_blocks;
  int B, H, KVH, D, G, bs, max_blocks;
  int heads_per_cta;     // query heads one CTA serves (<= its kernel's maximum)
  int gchunks;           // ceil(G / heads_per_cta)
  int P;                 // partition size in tokens (multiple of 16)
  int max_parts;         // partitions the grid covers per sequence; workspace stride
  int stages;            // pipeline depth per warp (TMA kernel)
  int part_major;        // TMA kernel: grid (head chunks, B, max_parts), else (max_parts, head chunks, B)
  float scale_log2;      // scale * log2(e): scores are kept in log2 units
  // Fused append (pkv_write_decode_attention); new_slots == nullptr otherwise.
  const int64_t *new_slots;   // [B] slot of sequence b's new token, negative: none
  const void *new_k;          // new token of b at element b * new_k_stride
  const void *new_v;
  long long new_k_stride, new_v_stride;
};

__device__ __forceinline__ void raise_flag(int *err, int bit) {
  if (err) atomicOr(err, bit);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Programmatic dependent launch.  launch_dependents: a grid launched after
// this one with programmatic stream serialization may be scheduled once every
// CTA of this grid has issued it (or exited).  griddep_wait: wait until the
// grids this one depends on have completed and their memory operations are
// visible (returns at once when launched without the attribute).
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Blackwell paired fp32 arithmetic: two lanes of fma / add in one instruction.
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

// 2^x on the SFU (ex2.approx, flush-to-zero); exp2(-inf) = 0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------ mbarrier + TMA

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Wait for the phase with the given parity to complete; false after
// kWaitLimitNs without completion.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// Tiled 4-D TMA load global -> shared, completion counted on `bar`.
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1, int c2, int c3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
      "r"(c3), "l"(policy)
      : "memory");
}

// Tiled 5-D TMA load global -> shared, completion counted on `bar`.
// The same 5-D box asked into L2 only (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_5d(const CUtensorMap *map, int c0, int c1, int c2,
                                                int c3, int c4) {
  asm volatile("cp.async.bulk.prefetch.tensor.5d.L2.global.tile [%0, {%1, %2, %3, %4, %5}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
               : "memory");
}

__device__ __forceinline__ void tma_load_5d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1, int c2, int c3, int c4,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
      "r"(c3), "r"(c4), "l"(policy)
      : "memory");
}

// Tiled 2-D TMA load global -> shared (no cache hint).
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// L2 policy for data read exactly once (K/V rows): evict first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// Orders this thread's generic-proxy shared-memory accesses before later
// asynchronous-proxy (TMA) accesses of the same locations.
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------ ldmatrix + mma.sync

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                              uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <typename T>
struct MmaOp;

template <>
struct MmaOp<__nv_bfloat16> {
  __device__ __forceinline__ static void run(float c[4], const uint32_t a[4], uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  // Two fp32 -> one packed pair (lo in the low half), round to nearest even;
  // also returns the rounded values' sum so weights and their total agree.
  __device__ __forceinline__ static uint32_t pack(float lo, float hi, float &sum) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    float2 f = __bfloat1622float2(v);
    sum += f.x + f.y;
    return *reinterpret_cast<uint32_t *>(&v);
  }
};

template <>
struct MmaOp<__half> {
  __device__ __forceinline__ static void run(float c[4], const uint32_t a[4], uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  __device__ __forceinline__ static uint32_t pack(float lo, float hi, float &sum) {
    __half2 v = __floats2half2_rn(lo, hi);
    float2 f = __half22float2(v);
    sum += f.x + f.y;
    return *reinterpret_cast<uint32_t *>(&v);
  }
};

// --------------------------------------------------------- element access

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <>
__device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}
template <>
__device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }

// ------------------------------------------------------ sequence bookkeeping

// Context length of sequence b after the device-side checks: negative -> 0,
// longer than the table -> clamped.  Flags are raised by partition 0 only.
__device__ __forceinline__ int checked_len(const DecodeArgs &a, int b, bool report) {
  int n = __ldg(a.lens + b);
  if (n < 0) {
    if (report) raise_flag(a.err, PKV_FLAG_CONTEXT_NEGATIVE);
    n = 0;
  }
  const long long cap = (long long)a.max_blocks * a.bs;
  if ((long long)n > cap) {
    if (report) raise_flag(a.err, PKV_FLAG_CONTEXT_TOO_LONG);
    n = (int)cap;
  }
  return n;
}

// Physical block of logical block lb of sequence b; an entry outside
// [0, num_blocks) is reported and replaced by block 0 (always in bounds).
__device__ __forceinline__ int checked_block(const DecodeArgs &a, int b, int lb) {
  const int phys = __ldg(a.tables + (size_t)b * a.max_blocks + lb);
  if (phys < 0 || (long long)phys >= a.num_blocks) {
    raise_flag(a.err, PKV_FLAG_BLOCK_OUT_OF_RANGE);
    return 0;
  }
  return phys;
}

// ----------------------------------------------------------------- epilogue

// Named barrier over the first `nthreads` threads of the CTA (id 1..15).
__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

struct CtaSync {
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

struct NamedSync {
  int id, nthreads;
  __device__ __forceinline__ void operator()() const { named_barrier(id, nthreads); }
};

//
// Called by `nthr` threads (thread index `tid`, synchronised by `sync`) once
// the partition [part*P, ...) of sequence b has been reduced to, for each of
// its nh query heads r:
//   s_m[r]  running max of the log2-unit scores,
//   s_l[r]  sum of 2^(score - s_m[r]),
//   s_o[r*ostride + d]  sum of 2^(score - s_m[r]) * V[d].
// With one partition the output row is s_o / s_l.  Otherwise the partials go
// to the workspace; the group that finishes a (sequence, head group) last --
// counted by `counter` -- merges all partitions:  M = max_p m_p,
// L = sum_p l_p 2^(m_p - M),  out = sum_p o_p 2^(m_p - M) / L, and resets the
// counter to zero.  With `clear_o`, each s_o element is zeroed right after
// the thread that reads it has read it.
template <typename T, typename Sync>
__device__ void finish_partition(const DecodeArgs &a, int b, int head0, int nh, int part,
                                 int nparts, const float *s_m, const float *s_l, float *s_o,
                                 int ostride, int *s_scratch, int *counter, int tid, int nthr,
                                 Sync sync, bool clear_o) {
  const int D = a.D;
  T *out = reinterpret_cast<T *>(a.out);
  if (nparts == 1) {
    for (int i = tid; i < nh * D; i += nthr) {
      const int r = i / D, d = i - r * D;
      const float v = s_o[r * ostride + d] / s_l[r];
      if (clear_o) s_o[r * ostride + d] = 0.f;
      out[((size_t)b * a.H + head0 + r) * D + d] = from_f32<T>(v);
    }
    return;
  }
  const size_t row0 = (size_t)b * a.H + head0;  // first (b, h) row of this group
  for (int r = tid; r < nh; r += nthr) {
    a.ws_m[(row0 + r) * a.max_parts + part] = s_m[r];
    a.ws_l[(row0 + r) * a.max_parts + part] = s_l[r];
  }
  for (int i = tid; i < nh * D; i += nthr) {
    const int r = i / D, d = i - r * D;
    a.ws_o[((row0 + r) * a.max_parts + part) * D + d] = s_o[r * ostride + d];
    if (clear_o) s_o[r * ostride + d] = 0.f;
  }
  // One thread publishes the group's partials and counts the partition with
  // one acquire-release atomic: the barrier orders the group's writes before
  // its release (cumulative), and for the last partition its acquire orders
  // the merge's reads after the other partitions' writes (no separate fences,
  // which can hold a thread for microseconds under load).
  sync();
  if (tid == 0) {
    int prev;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                 : "=r"(prev)
                 : "l"(reinterpret_cast<uint64_t>(counter))
                 : "memory");
    s_scratch[0] = prev == nparts - 1;
  }
  sync();
  if (!s_scratch[0]) return;
  // Last group: per-row max and total, then the merged rows.
  float *s_M = reinterpret_cast<float *>(s_scratch + 1);
  float *s_invL = s_M + nh;
  const int warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
  for (int r = warp; r < nh; r += nwarps) {
    const float *pm = a.ws_m + (row0 + r) * a.max_parts;
    const float *pl = a.ws_l + (row0 + r) * a.max_parts;
    float M = -INFINITY;
    for (int p = lane; p < nparts; p += 32) M = fmaxf(M, __ldcg(pm + p));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    for (int p = lane; p < nparts; p += 32) L += __ldcg(pl + p) * fast_exp2(__ldcg(pm + p) - M);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (lane == 0) {
      s_M[r] = M;
      s_invL[r] = 1.f / L;
    }
  }
  sync();
  for (int i = tid; i < nh * D; i += nthr) {
    const int r = i / D, d = i - r * D;
    const float *pm = a.ws_m + (row0 + r) * a.max_parts;
    const float *po = a.ws_o + (row0 + r) * a.max_parts * D + d;
    const float M = s_M[r];
    float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;  // four independent load chains
    int p = 0;
    for (; p + 3 < nparts; p += 4) {
      acc0 += __ldcg(po + (size_t)p * D) * fast_exp2(__ldcg(pm + p) - M);
      acc1 += __ldcg(po + (size_t)(p + 1) * D) * fast_exp2(__ldcg(pm + p + 1) - M);
      acc2 += __ldcg(po + (size_t)(p + 2) * D) * fast_exp2(__ldcg(pm + p + 2) - M);
      acc3 += __ldcg(po + (size_t)(p + 3) * D) * fast_exp2(__ldcg(pm + p + 3) - M);
    }
    for (; p < nparts; ++p) acc0 += __ldcg(po + (size_t)p * D) * fast_exp2(__ldcg(pm + p) - M);
    out[(row0 + r) * D + d] = from_f32<T>(((acc0 + acc1) + (acc2 + acc3)) * s_invL[r]);
  }
  if (tid == 0) *counter = 0;  // every partition has arrived: ready for the next call
}

// ------------------------------------------------------------ fused append

// Slot of sequence b's new token, or -1 (no append in this launch, or padding).
__device__ __forceinline__ long long append_slot(const DecodeArgs &a, int b) {
  if (!a.new_slots) return -1;
  const long long s = __ldg(a.new_slots + b);
  return s < 0 ? -1 : s;
}

// Row of KV head kvh of sequence b's new token in the k (or v) input.
template <typename T>
__device__ __forceinline__ const uint4 *append_src(const DecodeArgs &a, bool is_v, int b,
                                                   int kvh) {
  const T *base = reinterpret_cast<const T *>(is_v ? a.new_v : a.new_k);
  const long long stride = is_v ? a.new_v_stride : a.new_k_stride;
  return reinterpret_cast<const uint4 *>(base + (size_t)b * stride + (size_t)kvh * a.D);
}

// Checks of the cache half of the append (one thread of the writing CTA of
// (sequence b, KV head kvh)): `slot` must be where the context's position
// n-1 lives -- the physical block the table gives for it, row (n-1) % bs --
// and inside the pool.  Flags are raised for KV head 0 only.  Returns
// whether the row may be written.
// The same check given the table entry of position n - 1 (`phys`, read by
// the caller; ignored when n == 0).
__device__ __forceinline__ bool append_check_entry(const DecodeArgs &a, int kvh, long long slot,
                                                   int n, int phys) {
  bool match = false;
  if (n > 0) {
    const int lb = (n - 1) / a.bs;
    match = (long long)phys * a.bs + (n - 1 - lb * a.bs) == slot;
  }
  if (!match && kvh == 0) raise_flag(a.err, PKV_FLAG_APPEND_MISMATCH);
  const bool in_pool = slot < a.num_blocks * (long long)a.bs;
  if (!in_pool && kvh == 0) raise_flag(a.err, PKV_FLAG_SLOT_OUT_OF_RANGE);
  return in_pool;
}

__device__ __forceinline__ bool append_check(const DecodeArgs &a, int b, int kvh, long long slot,
                                             int n) {
  const int phys = n > 0 ? __ldg(a.tables + (size_t)b * a.max_blocks + (n - 1) / a.bs) : 0;
  return append_check_entry(a, kvh, slot, n, phys);
}

// 16-byte vector j of the K and V rows of KV head kvh at cache row `slot`.
template <typename T>
__device__ __forceinline__ void append_store(const DecodeArgs &a, int kvh, long long slot, int j,
                                             uint4 kv, uint4 vv) {
  const size_t row = ((size_t)slot * a.KVH + kvh) * a.D;
  T *kc = const_cast<T *>(reinterpret_cast<const T *>(a.k_cache)) + row;
  T *vc = const_cast<T *>(reinterpret_cast<const T *>(a.v_cache)) + row;
  reinterpret_cast<uint4 *>(kc)[j] = kv;
  reinterpret_cast<uint4 *>(vc)[j] = vv;
}

// The cache half of the append by one warp: check, then copy the new
// token's K and V rows of KV head kvh to cache row `slot`.
template <typename T>
__device__ void append_write_row(const DecodeArgs &a, int b, int kvh, long long slot, int n,
                                 int lane) {
  int ok = 0;
  if (lane == 0) ok = append_check(a, b, kvh, slot, n);
  if (!__shfl_sync(0xffffffffu, ok, 0)) return;
  const int vecs = a.D * (int)sizeof(T) / 16;  // per row of one head
  const uint4 *ks = append_src<T>(a, false, b, kvh), *vs = append_src<T>(a, true, b, kvh);
  for (int j = lane; j < vecs; j += 32) append_store<T>(a, kvh, slot, j, __ldg(ks + j), __ldg(vs + j));
}

// Zero output rows for an empty context (partition 0 only).
template <typename T>
__device__ void zero_rows(const DecodeArgs &a, int b, int head0, int nh) {
  T *out = reinterpret_cast<T *>(a.out);
  for (int i = threadIdx.x; i < nh * a.D; i += blockDim.x)
    out[((size_t)b * a.H + head0) * a.D + i] = from_f32<T>(0.f);
}

}  // namespace pkv
