// pkv_decode_tc.cu -- paged decode attention for bf16 / fp16 caches on
// sm_103a: TMA-staged K/V chunks, tensor-core (mma.sync m16n8k16) products
// for the query group, fp32 online softmax.
//
// Definition (course page "P09 · Paged KV 写入 + decode attention（参考实现）",
// section 题面速览 "decode 读" and the paged_decode_attention shape trace):
// n = context_lens[b]; only block_tables[b, :ceil(n/bs)] is read; token t is
// row t % bs of physical block tbl[t / bs]; exactly n tokens; query head h
// uses KV head h / (H / KVH) -- the L2 hint's "reshape q to [KVH, group, D]
// instead of copying K": one CTA serves the whole group; fp32 scores scaled
// before an fp32 softmax; weighted V sum cast to the output dtype.  The
// block-wise online softmax is the one of the interview note
// "PagedAttention kernel: paged KV cache 与 block table", section 代码; its
// partitioned (v2) variant, section 深入原理, is the split into work items.
//
// Work decomposition.  CTA = (partition of the context, KV head x chunk of
// <= 16 query heads, sequence); 4 warps; with fewer such units than resident
// CTA slots the partition is the grid's slowest index (first partitions
// launch first).  A partition is split into 16-token chunks (block_size is a
// multiple of 16, so a chunk never spans two physical blocks); warp w takes
// chunks w, w+4, w+8, ...  Each warp has its own ring of `stages`
// shared-memory slots; lanes 0 and 1 fetch a chunk's K and V rows of this KV
// head with one tiled 5-D TMA load each (box 64 elements x 16 rows x D/64
// blocks of 64 elements x 1 head x 1 block, 128-byte swizzle, L2
// evict-first) completing on the slot's mbarrier; the table entries come
// from one coalesced load per 32 chunks, broadcast by shuffle.
//
// Per chunk, per warp (the query group padded to the 16 rows of one tile):
//   S[16 x 16]  = Qgroup[16 x D] . K^T        D/16 mma, K via ldmatrix
//   online softmax on S in fp32 (log2 units), masked past the end
//   O[16 x D]  += P[16 x 16] . V              D/16 mma, V via ldmatrix.trans
// The P fragment is the S accumulator re-packed to bf16/fp16 in registers.
// At the end the 4 warp states are merged in shared memory and the
// partition is finished by finish_partition (direct output, or partials +
// log-sum-exp merge by the last CTA of the sequence).
//
// Launched into a captured graph, the kernel is a programmatic dependent of
// the step before it: a CTA reads its length, slot and table entries and
// asks L2 for its warps' first chunks (TMA prefetches of the boxes the
// first loads read) before griddepcontrol.wait; K/V loads and every write
// come after it.
#include <string.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

constexpr int kChunk = 16;          // tokens per pipeline slot
constexpr int kBoxElems = 64;       // elements per TMA box row (128 bytes)
constexpr int kBoxBytes = kChunk * 128;
constexpr int kTcWarps = 4;         // grid kernel: warps per CTA

template <int D>
struct TcShape {
  static constexpr int kSteps = D / 16;         // k-steps of Q.K^T, 16-wide n-pairs of P.V
  static constexpr int kNTiles = D / 8;         // 8-wide output tiles
  static constexpr int kBoxes = D / kBoxElems;  // TMA boxes per row
  static constexpr int kStageBytes = 2 * kBoxes * kBoxBytes;  // K + V of one chunk
  static constexpr int kQBytes = kBoxes * kBoxBytes;          // 16 query rows (TMA, swizzled)
  static constexpr int kQStride = D + 8;        // grid kernel: padded Q row (elements)
  static constexpr int kOStride = D + 8;        // padded fp32 row for the warp merge
  static constexpr bool kQInRegs = D <= 128;
};

// --------------------------------------------------- one chunk of one warp
//
// kb / vb: shared addresses of the chunk's K and V tiles (kBoxes boxes of 16
// rows x 128 bytes, 128-byte swizzle: 16-byte column c of row r sits at
// r * 128 + ((c ^ (r & 7)) << 4)).  qfrag(kk, af) yields the A fragment of
// the 16 x 16 query tile for k-step kk.  o/m/l: the warp's running state for
// rows lane/4 (m0, l0, o[.][0..1]) and lane/4 + 8 (m1, l1, o[.][2..3]).
template <int D, typename T, typename QFrag>
__device__ __forceinline__ void tc_chunk(uint32_t kb, uint32_t vb, int valid, const QFrag &qfrag,
                                         float (&o)[D / 8][4], float &m0, float &m1, float &l0,
                                         float &l1, float scale_log2, int lane) {
  using Sh = TcShape<D>;
  using Mma = MmaOp<T>;
  const int k_row = (lane & 7) + ((lane >> 4) << 3);        // token row of the K fragment
  const int k_col = (lane >> 3) & 1;                        // +1 column for b1 / b3
  const int v_row = (lane & 7) + (((lane >> 3) & 1) << 3);  // token row of the V fragment
  const int v_col = lane >> 4;                              // +1 column for the 2nd n-tile
  const int sw = lane & 7;                                  // swizzle term (row & 7)

  // ---- S = Q . K^T  (rows: query heads, cols: the chunk's 16 tokens); even
  // and odd k-steps accumulate separately (two shorter dependency chains)
  float sacc[2][2][4] = {};
#pragma unroll
  for (int kk = 0; kk < Sh::kSteps; ++kk) {
    const int col = ((kk & 3) << 1) + k_col;
    const uint32_t addr = kb + (kk >> 2) * kBoxBytes + k_row * 128 + ((col ^ sw) << 4);
    uint32_t b0, b1, b2, b3;
    ldsm_x4(addr, b0, b1, b2, b3);
    uint32_t af[4];
    qfrag(kk, af);
    Mma::run(sacc[kk & 1][0], af, b0, b1);
    Mma::run(sacc[kk & 1][1], af, b2, b3);
  }

  // ---- online softmax in log2 units; tokens past the end are -inf
  float x[2][4];
  if (valid == kChunk) {
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

  // ---- O += P . V ; V rows past the end are zeroed (they may hold NaN/Inf)
  uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
  if (valid < kChunk) {
    const int tk = (lane & 3) * 2;
    vm0 = (tk < valid ? 0x0000ffffu : 0u) | (tk + 1 < valid ? 0xffff0000u : 0u);
    vm1 = (tk + 8 < valid ? 0x0000ffffu : 0u) | (tk + 9 < valid ? 0xffff0000u : 0u);
  }
#pragma unroll
  for (int dp = 0; dp < Sh::kSteps; ++dp) {
    const int col = ((dp & 3) << 1) + v_col;
    const uint32_t addr = vb + (dp >> 2) * kBoxBytes + v_row * 128 + ((col ^ sw) << 4);
    uint32_t b0, b1, b2, b3;
    ldsm_x4_trans(addr, b0, b1, b2, b3);
    b0 &= vm0; b1 &= vm1; b2 &= vm0; b3 &= vm1;
    Mma::run(o[2 * dp], pa, b0, b1);
    Mma::run(o[2 * dp + 1], pa, b2, b3);
  }
}

// ======================================================= grid kernel (4 warps)

size_t tc_smem_bytes(int D, int stages) {
  const size_t stage_bytes = 2 * (size_t)(D / kBoxElems) * kBoxBytes;
  return 1024                                             // alignment slack
         + (size_t)kTcWarps * stages * stage_bytes        // K/V rings
         + (size_t)kTcHeads * (D + 8) * 2                 // Q
         + (size_t)2 * D * 2                              // fused append: new K and V rows
         + (size_t)kTcWarps * stages * 8                  // mbarriers
         + sizeof(float) * (2 * kTcWarps * kTcHeads + 2 * kTcHeads)  // warp m/l, final m/l
         + sizeof(int) * (4 + 2 * kTcHeads);              // epilogue scratch
}

// CTA = (partition, KV head x chunk of <= 16 query heads, sequence); warp w
// takes chunks w, w+4, ... of the partition through its own ring of
// `stages` slots; lane 0 issues the TMA loads; table entries are fetched 32
// at a time by one coalesced load and broadcast by shuffle.
template <int D, typename T, bool kAppend>
__global__ void __launch_bounds__(32 * kTcWarps, 1)
    pkv_decode_tc_kernel(const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const DecodeArgs a) {
  using Sh = TcShape<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = a.stages;
  uint8_t *ring = smem;                                              // [W][S][stage]
  T *sQ = reinterpret_cast<T *>(ring + (size_t)kTcWarps * S * Sh::kStageBytes);
  T *sNew = sQ + kTcHeads * Sh::kQStride;                            // [2][D] new K, V rows
  uint64_t *bars = reinterpret_cast<uint64_t *>(sNew + 2 * D);
  float *s_wm = reinterpret_cast<float *>(bars + kTcWarps * S);     // [W][16]
  float *s_wl = s_wm + kTcWarps * kTcHeads;                         // [W][16]
  float *s_m = s_wl + kTcWarps * kTcHeads;                          // [16]
  float *s_l = s_m + kTcHeads;                                      // [16]
  int *s_scratch = reinterpret_cast<int *>(s_l + kTcHeads);

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  // Launched as a programmatic dependent of the previous kernel on the
  // stream, a CTA reads only inputs (lengths, slots, tables, new rows)
  // before griddep_wait; K/V loads and every write come after it.  The next
  // launch may be scheduled once every CTA of this grid has started.
  griddep_launch_dependents();
  // grid (max_parts, head chunks, B), or with part_major (head chunks, B,
  // max_parts): every unit's first partitions launch first and the short or
  // empty last ones at the end of the launch
  const int hc = a.part_major ? blockIdx.x : blockIdx.y;
  const int b = a.part_major ? blockIdx.y : blockIdx.z;
  const int part = a.part_major ? blockIdx.z : blockIdx.x;
  const int kvh = hc / a.gchunks, gc = hc - kvh * a.gchunks;
  const int head0 = kvh * a.G + gc * kTcHeads;
  const int nh = min(kTcHeads, a.G - gc * kTcHeads);

  // fused append (kAppend): the new token's slot, or -1 -- loaded first, so
  // that its latency overlaps the length's
  const long long s_new = kAppend ? append_slot(a, b) : -1LL;
  const int n = checked_len(a, b, part == 0 && hc == 0 && tid == 0);
  int nparts = (n + a.P - 1) / a.P;
  if (nparts > a.max_parts) {
    if (part == a.max_parts - 1 && hc == 0 && tid == 0) raise_flag(a.err, PKV_FLAG_CONTEXT_OVER_HINT);
    nparts = a.max_parts;
  }
  if (n == 0) {
    if (part == 0) {
      griddep_wait();
      zero_rows<T>(a, b, head0, nh);
      if (s_new >= 0 && gc == 0 && w == 0) append_write_row<T>(a, b, kvh, s_new, n, lane);
    }
    return;
  }
  if (part >= nparts) return;
  const int t0 = part * a.P;
  const int t1 = min(n, t0 + a.P);
  const int nchunks = (t1 - t0 + kChunk - 1) / kChunk;
  const int nch_w = nchunks > w ? (nchunks - w + kTcWarps - 1) / kTcWarps : 0;
  // Fused append: the warp whose chunk holds position n-1 overwrites that
  // row of its shared-memory tile with the new token (so nothing waits for
  // the cache write); in the one CTA per (sequence, KV head) that writes the
  // cache row, the same warp stores it.
  const bool cache_writer = s_new >= 0 && gc == 0 && part == nparts - 1;
  const bool covers_new = s_new >= 0 && n - 1 >= t0 && n - 1 < t1;
  int patch_i = -1, patch_row = 0;
  if (covers_new && ((n - 1 - t0) / kChunk) % kTcWarps == w) {
    patch_i = (n - 1 - t0) / kChunk / kTcWarps;
    patch_row = (n - 1 - t0) % kChunk;
  }

  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[w * S + s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (tid == 0) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  const uint64_t policy = l2_evict_first_policy();
  int tbl_batch = -1, my_phys = 0;
  auto phys_of = [&](int i) -> int {  // physical block of this warp's i-th chunk (warp-collective)
    const int batch = i >> 5;
    if (batch != tbl_batch) {
      tbl_batch = batch;
      const int ii = batch * 32 + lane;
      my_phys = 0;
      if (ii < nch_w) my_phys = checked_block(a, b, (t0 + kChunk * (w + kTcWarps * ii)) / a.bs);
    }
    return __shfl_sync(0xffffffffu, my_phys, i & 31);
  };
  // Fetch chunk i of this warp into `slot` (warp-collective).  Lane 0 posts
  // the byte count; lane 0 issues K's box, lane 1 V's: one box per tensor
  // covers the chunk's 16 rows and all D / 64 blocks of 64 values (the TMA
  // unit's cost is per box: a box per 64 values was the larger part of it).
  const int bs_mask = (a.bs & (a.bs - 1)) == 0 ? a.bs - 1 : -1;
  auto issue = [&](int i, int slot) {
    const int phys = phys_of(i);
    const int tok = t0 + kChunk * (w + kTcWarps * i);
    const int row0 = bs_mask >= 0 ? (tok & bs_mask) : tok % a.bs;
    uint8_t *st = ring + (size_t)(w * S + slot) * Sh::kStageBytes;
    uint64_t *bar = &bars[w * S + slot];
    if (lane == 0) mbar_arrive_expect_tx(bar, Sh::kStageBytes);
    __syncwarp();
    if (lane < 2)
      tma_load_5d(st + lane * Sh::kBoxes * kBoxBytes, lane ? &tmV : &tmK, bar, 0, row0, 0, kvh, phys,
                  policy);
  };
  // The patching warp loads the new rows (and checks the slot) before
  // anything else, so that these loads overlap the first fetches and the
  // query loads ...
  uint4 new_kv = make_uint4(0, 0, 0, 0), new_vv = new_kv;
  int new_ok = 0;
  if (patch_i >= 0) {
    if (lane < D / 8) {
      new_kv = __ldg(append_src<T>(a, false, b, kvh) + lane);
      new_vv = __ldg(append_src<T>(a, true, b, kvh) + lane);
    }
    if (cache_writer && lane == 0) new_ok = append_check(a, b, kvh, s_new, n);
  }
  // The warp's first table entries are read before the wait (the tables are
  // inputs), and its first chunks of K and V asked into L2 by TMA prefetches
  // of the very boxes the loads will read (a line the previous grid still
  // writes is updated in L2, which the loads read); the K/V loads, the cache
  // write and every other write come after the wait.
  const int npro = min(S, nch_w);
  for (int i = 0; i < npro; ++i) {
    const int phys = phys_of(i);
    const int tok = t0 + kChunk * (w + kTcWarps * i);
    const int row0 = bs_mask >= 0 ? (tok & bs_mask) : tok % a.bs;
    if (lane < 2) tma_prefetch_5d(lane ? &tmV : &tmK, 0, row0, 0, kvh, phys);
  }
  griddep_wait();
  // Start the warp's first fetches before staging Q: the copies are in
  // flight while the query tile is loaded.
  for (int i = 0; i < npro; ++i) issue(i, i);

  // Q rows of the group (rows >= nh are zero) into padded shared rows.
  {
    const T *qg = reinterpret_cast<const T *>(a.q) + ((size_t)b * a.H + head0) * D;
    constexpr int VPR = D / 8;  // 16-byte vectors per row
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

  // ... and stages the new rows in shared memory and, in the writing CTA,
  // stores them to the cache row: no registers are held through the main
  // loop, no other warp waits, and whatever a TMA load reads of that row
  // before or after the store is overwritten by the patch.
  if (patch_i >= 0) {
    const int ok = __shfl_sync(0xffffffffu, new_ok, 0);
    if (lane < D / 8) {
      reinterpret_cast<uint4 *>(sNew)[lane] = new_kv;
      reinterpret_cast<uint4 *>(sNew)[D / 8 + lane] = new_vv;
      if (ok) append_store<T>(a, kvh, s_new, lane, new_kv, new_vv);
    }
  }

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
    const int valid = min(kChunk, t1 - (t0 + kChunk * (w + kTcWarps * i)));
    const uint32_t kb = smem_u32(ring + (size_t)(w * S + slot) * Sh::kStageBytes);
    if (i == patch_i) {  // overwrite row patch_row of the tiles with the new token
      if (lane < D / 8) {  // 16-byte column lane&7 of box lane>>3, swizzled
        const uint32_t off = (lane >> 3) * kBoxBytes + patch_row * 128 +
                             (((lane & 7) ^ (patch_row & 7)) << 4);
        st_shared_v4(kb + off, reinterpret_cast<const uint4 *>(sNew)[lane]);
        st_shared_v4(kb + Sh::kBoxes * kBoxBytes + off,
                     reinterpret_cast<const uint4 *>(sNew)[D / 8 + lane]);
      }
      fence_proxy_async_shared();  // the slot is refilled by TMA later
      __syncwarp();
    }
    tc_chunk<D, T>(kb, kb + Sh::kBoxes * kBoxBytes, valid, qfrag, o, m0, m1, l0, l1, a.scale_log2,
                   lane);
    __syncwarp();
    if (i + S < nch_w) issue(i + S, slot);
    if (++slot == S) {
      slot = 0;
      parity ^= 1u;
    }
  }
  if (i < nch_w) {
    // Gave up waiting: let the copies already issued land (bounded) before
    // the shared memory is reused.
    for (int j = i; j < min(i + S, nch_w); ++j) {
      mbar_wait_bounded(&bars[w * S + slot], parity);
      if (++slot == S) {
        slot = 0;
        parity ^= 1u;
      }
    }
  }

  // The context was cut short (PKV_FLAG_CONTEXT_OVER_HINT): position n-1 was
  // not read here, but the cache row is still written.
  if (cache_writer && !covers_new && w == 0) append_write_row<T>(a, b, kvh, s_new, n, lane);

  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  // ---- merge the 4 warp states (the rings are free now)
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
  for (int ww = 0; ww < kTcWarps; ++ww) {
    M0 = fmaxf(M0, s_wm[ww * kTcHeads + r0]);
    M1 = fmaxf(M1, s_wm[ww * kTcHeads + r1]);
  }
  const float f0 = fast_exp2(m0 - M0), f1 = fast_exp2(m1 - M1);  // 0 for a warp without chunks
  float *sO = reinterpret_cast<float *>(ring);                   // [W][16][kOStride]
  if (r0 < nh) {  // rows past the group are padding: never merged
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
    for (int ww = 0; ww < kTcWarps; ++ww) M = fmaxf(M, s_wm[ww * kTcHeads + tid]);
    float L = 0.f;
    for (int ww = 0; ww < kTcWarps; ++ww)
      L += s_wl[ww * kTcHeads + tid] * fast_exp2(s_wm[ww * kTcHeads + tid] - M);
    s_m[tid] = M;
    s_l[tid] = L;
  }
  __syncthreads();
  for (int e = tid; e < nh * D; e += blockDim.x) {
    const int r = e / D, d = e - r * D;
    float acc = 0.f;
#pragma unroll
    for (int ww = 0; ww < kTcWarps; ++ww) acc += sO[(ww * kTcHeads + r) * Sh::kOStride + d];
    sO[r * Sh::kOStride + d] = acc;  // row r of warp 0's slot: read above only by this thread
  }
  __syncthreads();
  finish_partition<T>(a, b, head0, nh, part, nparts, s_m, s_l, sO, Sh::kOStride, s_scratch,
                      a.ws_cnt + (size_t)b * (a.KVH * a.gchunks) + hc, tid, blockDim.x, CtaSync(),
                      false);
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

static CUtensorMapDataType map_type(pkv_dtype dt) {
  return dt == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

// Tensor map of a [num_blocks, bs, KVH, D] cache: dims innermost first, box of
// 64 elements x 1 head x 16 rows x 1 block, 128-byte swizzle.
bool encode_cache_map(CUtensorMap *map, const void *cache, pkv_dtype dt, long long num_blocks,
                             int bs, int KVH, int D) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t el = 2;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)KVH, (cuuint64_t)bs, (cuuint64_t)num_blocks};
  cuuint64_t strides[3] = {D * el, (cuuint64_t)KVH * D * el, (cuuint64_t)bs * KVH * D * el};
  cuuint32_t box[4] = {kBoxElems, 1, kChunk, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, map_type(dt), 4, const_cast<void *>(cache), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map of a [num_blocks, bs, KVH, D] cache seen as 5-D, innermost first:
// 64 values (stride 1), row in the block, block of 64 values (stride 128
// bytes), head, block; box of 64 values x 16 rows x D / 64 blocks x 1 head x
// 1 block, 128-byte swizzle.  A box lands as D / 64 tiles of 16 rows x 128
// bytes, one after another: the layout of one 4-D box per 64 values, in one
// copy.
static bool encode_chunk_map(CUtensorMap *map, const void *cache, pkv_dtype dt,
                             long long num_blocks, int bs, int KVH, int D) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t el = 2;
  cuuint64_t dims[5] = {(cuuint64_t)kBoxElems, (cuuint64_t)bs, (cuuint64_t)(D / kBoxElems),
                        (cuuint64_t)KVH, (cuuint64_t)num_blocks};
  cuuint64_t strides[4] = {(cuuint64_t)KVH * D * el, kBoxElems * el, D * el,
                           (cuuint64_t)bs * KVH * D * el};
  cuuint32_t box[5] = {kBoxElems, kChunk, (cuuint32_t)(D / kBoxElems), 1, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(map, map_type(dt), 5, const_cast<void *>(cache), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map of a [rows, H, D] 16-bit tensor (one row of H heads per token):
// box of 64 elements x 1 head x box_rows rows, 128-byte swizzle; rows past
// the end read as zero.
bool encode_rows_map(CUtensorMap *map, const void *base, pkv_dtype dt, long long rows, int H, int D,
                     int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t el = 2;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[2] = {D * el, (cuuint64_t)H * D * el};
  cuuint32_t box[3] = {kBoxElems, 1, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, map_type(dt), 3, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, typename T, bool kAppend>
static pkv_status launch_tc_k(const DecodeArgs &a, const DecodePlan &plan, const CUtensorMap &mk,
                              const CUtensorMap &mv, cudaStream_t stream) {
  auto kern = pkv_decode_tc_kernel<D, T, kAppend>;
  static int configured[64] = {0};
  if (!allow_smem(kern, plan.smem_bytes, configured)) return PKV_ERR_CUDA;
  DecodeArgs args = a;
  if (plan.max_parts > 65535) args.part_major = 0;  // past the grid's z extent: unit-major
  const dim3 grid = args.part_major ? dim3(a.KVH * plan.gchunks, a.B, plan.max_parts)
                                    : dim3(plan.max_parts, a.KVH * plan.gchunks, a.B);
  // a programmatic dependent of the previous kernel on the stream: its CTAs'
  // start-up overlaps that kernel's last CTAs (see the kernel's griddep_wait)
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = grid;
  cfg.blockDim = dim3(32 * kTcWarps);
  cfg.dynamicSmemBytes = plan.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = launch_as_dependent(stream) ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, kern, mk, mv, args) != cudaSuccess) return PKV_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

template <int D, typename T>
static pkv_status launch_tc_t(const DecodeArgs &a, const DecodePlan &plan, const CUtensorMap &mk,
                              const CUtensorMap &mv, cudaStream_t stream) {
  return a.new_slots ? launch_tc_k<D, T, true>(a, plan, mk, mv, stream)
                     : launch_tc_k<D, T, false>(a, plan, mk, mv, stream);
}

template <typename T>
static pkv_status launch_tc_dt(const DecodeArgs &a, const DecodePlan &plan, const CUtensorMap &mk,
                               const CUtensorMap &mv, cudaStream_t stream) {
  switch (a.D) {
    case 64: return launch_tc_t<64, T>(a, plan, mk, mv, stream);
    case 128: return launch_tc_t<128, T>(a, plan, mk, mv, stream);
    case 192: return launch_tc_t<192, T>(a, plan, mk, mv, stream);
    case 256: return launch_tc_t<256, T>(a, plan, mk, mv, stream);
  }
  return PKV_ERR_UNSUPPORTED;
}

pkv_status launch_decode_tc(const DecodeArgs &a, const DecodePlan &plan, pkv_dtype dt,
                            cudaStream_t stream) {
  CUtensorMap mk, mv;
  if (!encode_chunk_map(&mk, a.k_cache, dt, a.num_blocks, a.bs, a.KVH, a.D) ||
      !encode_chunk_map(&mv, a.v_cache, dt, a.num_blocks, a.bs, a.KVH, a.D))
    return PKV_ERR_CUDA;
  if (dt == PKV_BF16) return launch_tc_dt<__nv_bfloat16>(a, plan, mk, mv, stream);
  if (dt == PKV_F16) return launch_tc_dt<__half>(a, plan, mk, mv, stream);
  return PKV_ERR_UNSUPPORTED;
}

}  // namespace pkv
