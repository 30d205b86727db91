/*
 * pkv_oracle.c -- the oracle for the paged KV-cache write and paged decode
 * attention.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * CPU-baseline leg of the benchmark call it; the library never does.
 *
 * A plain, slow, fp64 CPU restatement of what the two operations compute,
 * written from the course page "P09 · Paged KV 写入 + decode attention
 * （参考实现）" (kuanzhou.online, nano-vllm-omni drills):
 *   - write:  section 题面速览 ("写: cache[slot // bs, slot % bs] = k[i]",
 *             slot -1 is padding) and the write_kv shape trace
 *             (keep = slot >= 0, blk = s // bs, off = s % bs, in-place);
 *   - decode: section 题面速览 ("decode 读") and the paged_decode_attention
 *             shape trace: n = context_lens[b], nb = ceil(n / bs), only
 *             block_tables[b, :nb] is read, gather in table order, keep the
 *             first n rows, query head h reads KV head h // (H / KVH),
 *             scores are scaled BEFORE the softmax, output cast to q.dtype.
 * The interview note "PagedAttention kernel: paged KV cache 与 block table"
 * (inference-learning-path.pages.dev), section 直接答案, states that paging
 * changes only where K/V live, never what attention computes; so the oracle
 * is the plain definition of softmax attention over the gathered rows.
 *
 * Precision: inputs (fp32 / bf16 / fp16) are promoted exactly to double; the
 * dot products, a two-pass max-subtracted softmax and the weighted sum are
 * all in double; the result is rounded ONCE to the output type with
 * round-to-nearest-even.  Nothing is blocked, fused or reordered beyond the
 * definition.  The code shares nothing with the CUDA library.
 *
 * Readings of points the pages leave open (each is listed in the design
 * notes of the repository):
 *   - every negative slot is padding and skipped (the filter is slot >= 0);
 *   - a slot >= num_blocks * bs, a table entry of the used prefix outside
 *     [0, num_blocks), or a context longer than max_blocks * bs is an error
 *     (the PyTorch reference would raise); the oracle returns a code;
 *   - context_len == 0 gives an all-zero output row and reads nothing.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F16 = 2 };

enum {
  ORC_OK = 0,
  ORC_ERR_ARG = -1,
  ORC_ERR_SLOT_RANGE = -2,
  ORC_ERR_BLOCK_RANGE = -3,
  ORC_ERR_CONTEXT = -4,
  ORC_ERR_NOMEM = -5
};

/* ---------------------------------------------------------------- numbers */

/* Exact value of an IEEE binary16 bit pattern. */
static double half_bits_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double x;
  if (e == 0) {
    x = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  } else if (e == 31) {
    x = m ? NAN : INFINITY;
  } else {
    x = ldexp((double)(1024 + m), e - 15 - 10);
  }
  return sign ? -x : x;
}

/* Exact value of a bfloat16 bit pattern: the top half of a binary32. */
static double bf16_bits_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static int elem_bytes(int dtype) {
  return dtype == ORC_F32 ? 4 : 2;
}

static double load_elem(const void *base, int64_t i, int dtype) {
  if (dtype == ORC_F32) return (double)((const float *)base)[i];
  uint16_t bits = ((const uint16_t *)base)[i];
  return dtype == ORC_BF16 ? bf16_bits_to_double(bits) : half_bits_to_double(bits);
}

/*
 * Round x to the nearest value of a binary format with p significand bits
 * (implicit bit included), minimum normal exponent emin and largest finite
 * value maxfinite; ties go to the even significand (IEEE 754
 * roundTiesToEven).  Subnormals keep the fixed quantum 2^(emin - p + 1).
 * One rounding step straight from double, so no double rounding occurs.
 */
static double round_to_format(double x, int p, int emin, double maxfinite) {
  if (x == 0.0 || isnan(x) || isinf(x)) return x;
  int e;
  frexp(x, &e);          /* |x| = f * 2^e with 0.5 <= f < 1: leading bit 2^(e-1) */
  int q = e - p;         /* exponent of one unit in the last place */
  if (q < emin - p + 1) q = emin - p + 1;
  double r = nearbyint(ldexp(x, -q)); /* default rounding mode: ties to even */
  double y = ldexp(r, q);
  if (fabs(y) > maxfinite) y = copysign(INFINITY, x);
  return y;
}

static uint16_t double_to_bf16_bits(double x) {
  if (isnan(x)) return 0x7fc0;
  double y = round_to_format(x, 8, -126, ldexp(255.0, 120)); /* max (2-2^-7)*2^127 */
  float f = (float)y; /* exact: y is a bfloat16 value */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(u >> 16);
}

static uint16_t double_to_half_bits(double x) {
  if (isnan(x)) return 0x7e00;
  double y = round_to_format(x, 11, -14, 65504.0);
  uint16_t sign = signbit(y) ? 0x8000 : 0;
  double a = fabs(y);
  if (a == 0.0) return sign;
  if (isinf(a)) return sign | 0x7c00;
  if (a < ldexp(1.0, -14)) /* subnormal: a = m * 2^-24 */
    return sign | (uint16_t)ldexp(a, 24);
  int e;
  frexp(a, &e);           /* a = f * 2^e, leading bit 2^(e-1) */
  int E = e - 1;
  uint16_t mant = (uint16_t)(ldexp(a, 10 - E) - 1024.0);
  return sign | (uint16_t)((E + 15) << 10) | mant;
}

static void store_elem(void *base, int64_t i, int dtype, double x) {
  if (dtype == ORC_F32) {
    ((float *)base)[i] = (float)round_to_format(x, 24, -126, 3.4028234663852886e38);
  } else if (dtype == ORC_BF16) {
    ((uint16_t *)base)[i] = double_to_bf16_bits(x);
  } else {
    ((uint16_t *)base)[i] = double_to_half_bits(x);
  }
}

/* Round n doubles to the given type (exposed so the rounding is testable). */
int pkv_oracle_round(const double *x, void *out, int64_t n, int dtype) {
  if (dtype < ORC_F32 || dtype > ORC_F16 || n < 0) return ORC_ERR_ARG;
  for (int64_t i = 0; i < n; ++i) store_elem(out, i, dtype, x[i]);
  return ORC_OK;
}

/* Widen n elements of the given type to double, exactly. */
int pkv_oracle_widen(const void *in, double *x, int64_t n, int dtype) {
  if (dtype < ORC_F32 || dtype > ORC_F16 || n < 0) return ORC_ERR_ARG;
  for (int64_t i = 0; i < n; ++i) x[i] = load_elem(in, i, dtype);
  return ORC_OK;
}

/* ------------------------------------------------------------------ write */

/*
 * write_kv: for every new token i in order, skip it when slot_mapping[i] is
 * negative (padding); otherwise copy the bits of k[i] into
 * k_cache[slot // bs, slot % bs] and of v[i] into v_cache[...], in place.
 * Cache layout [num_blocks, block_size, num_kv_heads, head_dim]; k and v are
 * [T, num_kv_heads, head_dim] with consecutive tokens token_stride elements
 * apart.  Returns ORC_ERR_SLOT_RANGE (after the tokens before it are
 * written) when a slot is past the end of the pool.
 */
int pkv_oracle_write(void *k_cache, void *v_cache, const void *k, const void *v,
                     const int64_t *slot_mapping, int64_t num_tokens, int64_t token_stride,
                     int64_t num_blocks, int64_t block_size, int64_t num_kv_heads,
                     int64_t head_dim, int dtype) {
  if (num_tokens < 0 || num_blocks < 0 || block_size <= 0 || num_kv_heads <= 0 ||
      head_dim <= 0 || dtype < ORC_F32 || dtype > ORC_F16)
    return ORC_ERR_ARG;
  const int64_t row_elems = num_kv_heads * head_dim;  /* one token: [KVH, D] */
  const size_t row_bytes = (size_t)row_elems * (size_t)elem_bytes(dtype);
  for (int64_t i = 0; i < num_tokens; ++i) {
    int64_t slot = slot_mapping[i];
    if (slot < 0) continue;                        /* padding token: not written */
    if (slot >= num_blocks * block_size) return ORC_ERR_SLOT_RANGE;
    const int64_t blk = slot / block_size;         /* physical block */
    const int64_t off = slot % block_size;         /* row inside the block */
    const int64_t dst = (blk * block_size + off) * row_elems;
    const int64_t src = i * token_stride;
    memcpy((char *)k_cache + (size_t)dst * elem_bytes(dtype),
           (const char *)k + (size_t)src * elem_bytes(dtype), row_bytes);
    memcpy((char *)v_cache + (size_t)dst * elem_bytes(dtype),
           (const char *)v + (size_t)src * elem_bytes(dtype), row_bytes);
  }
  return ORC_OK;
}

/* ----------------------------------------------------------------- decode */

/*
 * paged decode attention for the sequences b in [b_begin, b_end) and the
 * query heads h in [h_begin, h_end) (the whole batch: [0, B) x [0, H)):
 *   n    = context_lens[b]
 *   nb   = ceil(n / bs); only block_tables[b, 0:nb] is read
 *   for each query head h:  kvh = h / (H / KVH)
 *     logical token t < n lives in physical block tbl[t / bs], row t % bs
 *     s_t   = scale * sum_d q[b,h,d] * K[t,kvh,d]
 *     w_t   = exp(s_t - max_j s_j)
 *     out[b,h,:] = sum_t w_t V[t,kvh,:] / sum_t w_t      (rounded once)
 * q and out are [B, H, D]; block_tables is [B, max_blocks] int32.
 */
int pkv_oracle_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *block_tables, const int32_t *context_lens,
                      int64_t B, int64_t H, int64_t num_kv_heads, int64_t head_dim,
                      int64_t block_size, int64_t max_blocks, int64_t num_blocks,
                      double scale, int dtype, int64_t b_begin, int64_t b_end,
                      int64_t h_begin, int64_t h_end) {
  if (B < 0 || H <= 0 || num_kv_heads <= 0 || H % num_kv_heads != 0 || head_dim <= 0 ||
      block_size <= 0 || max_blocks < 0 || num_blocks < 0 || dtype < ORC_F32 ||
      dtype > ORC_F16 || b_begin < 0 || b_end > B || b_begin > b_end || h_begin < 0 ||
      h_end > H || h_begin > h_end)
    return ORC_ERR_ARG;
  const int64_t KVH = num_kv_heads, D = head_dim, bs = block_size;
  const int64_t group = H / KVH;
  int rc = ORC_OK;

  for (int64_t b = b_begin; b < b_end && rc == ORC_OK; ++b) {
    const int64_t n = context_lens[b];
    if (n < 0) { rc = ORC_ERR_CONTEXT; break; }
    const int64_t nb = (n + bs - 1) / bs;       /* ceil: a partial last block counts */
    if (nb > max_blocks) { rc = ORC_ERR_CONTEXT; break; }
    const int32_t *tbl = block_tables + b * max_blocks;
    for (int64_t j = 0; j < nb; ++j)
      if (tbl[j] < 0 || tbl[j] >= num_blocks) { rc = ORC_ERR_BLOCK_RANGE; break; }
    if (rc != ORC_OK) break;

    double *s = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    if (!s) { rc = ORC_ERR_NOMEM; break; }

    for (int64_t h = h_begin; h < h_end; ++h) {
      const int64_t kvh = h / group;            /* GQA: repeat_interleave order */
      const int64_t qoff = (b * H + h) * D;
      if (n == 0) {                             /* empty context: zero output */
        for (int64_t d = 0; d < D; ++d) store_elem(out, qoff + d, dtype, 0.0);
        continue;
      }
      /* scores over exactly the first n logical tokens, in table order */
      double m = -INFINITY;
      for (int64_t t = 0; t < n; ++t) {
        const int64_t phys = tbl[t / bs];
        const int64_t row = ((phys * bs + t % bs) * KVH + kvh) * D;
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d)
          dot += load_elem(q, qoff + d, dtype) * load_elem(k_cache, row + d, dtype);
        s[t] = scale * dot;                     /* scale before the softmax */
        if (s[t] > m) m = s[t];
      }
      double denom = 0.0;
      for (int64_t t = 0; t < n; ++t) {
        s[t] = exp(s[t] - m);                   /* now the unnormalised weight */
        denom += s[t];
      }
      for (int64_t d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int64_t t = 0; t < n; ++t) {
          const int64_t phys = tbl[t / bs];
          const int64_t row = ((phys * bs + t % bs) * KVH + kvh) * D;
          acc += s[t] * load_elem(v_cache, row + d, dtype);
        }
        store_elem(out, qoff + d, dtype, acc / denom);
      }
    }
    free(s);
  }
  return rc;
}

/*
 * paged prefill attention (several new query tokens per sequence, causal)
 * for the sequences b in [b_begin, b_end).  The pages only ask how the
 * varlen prefill version would be written (course page "P09 · Paged KV 写入
 * + decode attention（参考实现）", section 面试官追问); the reading taken
 * here is the one decode is the one-query case of (same page, section 细节:
 * the decode query is the newest token, already written, and sees the
 * whole context including itself):
 *   qlen = cu_seqlens_q[b+1] - cu_seqlens_q[b] new tokens, the LAST qlen
 *   tokens of a context of n = context_lens[b] tokens (qlen <= n, all
 *   already written to the cache);
 *   query i (row cu_seqlens_q[b] + i of q / out) sits at logical position
 *   p = n - qlen + i and attends to the tokens 0 .. p (causal);
 *   kvh = h / (H / KVH); scores scaled before an exact softmax; rounded once.
 * q and out are [total_q, H, D] with total_q = cu_seqlens_q[B].
 */
int pkv_oracle_prefill(void *out, const void *q, const void *k_cache, const void *v_cache,
                       const int32_t *block_tables, const int32_t *cu_seqlens_q,
                       const int32_t *context_lens, int64_t B, int64_t H, int64_t num_kv_heads,
                       int64_t head_dim, int64_t block_size, int64_t max_blocks,
                       int64_t num_blocks, double scale, int dtype, int64_t b_begin,
                       int64_t b_end) {
  if (B < 0 || H <= 0 || num_kv_heads <= 0 || H % num_kv_heads != 0 || head_dim <= 0 ||
      block_size <= 0 || max_blocks < 0 || num_blocks < 0 || dtype < ORC_F32 ||
      dtype > ORC_F16 || b_begin < 0 || b_end > B || b_begin > b_end || cu_seqlens_q[0] != 0)
    return ORC_ERR_ARG;
  const int64_t KVH = num_kv_heads, D = head_dim, bs = block_size;
  const int64_t heads_per_kv = H / KVH;
  int status = ORC_OK;

  for (int64_t b = b_begin; b < b_end && status == ORC_OK; ++b) {
    const int64_t qlen = (int64_t)cu_seqlens_q[b + 1] - cu_seqlens_q[b];
    const int64_t n = context_lens[b];
    if (qlen < 0 || n < qlen) { status = ORC_ERR_CONTEXT; break; }
    const int64_t nb = (n + bs - 1) / bs;
    if (nb > max_blocks) { status = ORC_ERR_CONTEXT; break; }
    const int32_t *table = block_tables + b * max_blocks;
    for (int64_t j = 0; j < nb; ++j)
      if (table[j] < 0 || table[j] >= num_blocks) { status = ORC_ERR_BLOCK_RANGE; break; }
    if (status != ORC_OK) break;

    double *w = (double *)calloc((size_t)(n > 0 ? n : 1), sizeof(double));
    if (!w) { status = ORC_ERR_NOMEM; break; }

    for (int64_t i = 0; i < qlen; ++i) {
      const int64_t p = n - qlen + i;           /* logical position of query i */
      const int64_t lim = p + 1;                /* causal: tokens 0 .. p, p included */
      const int64_t q_row = cu_seqlens_q[b] + i;
      for (int64_t h = 0; h < H; ++h) {
        const int64_t g = h / heads_per_kv;     /* GQA: repeat_interleave order */
        const int64_t qbase = (q_row * H + h) * D;
        double mx = -INFINITY;
        for (int64_t t = 0; t < lim; ++t) {
          const int64_t krow = ((table[t / bs] * bs + t % bs) * KVH + g) * D;
          double qk = 0.0;
          for (int64_t d = 0; d < D; ++d)
            qk += load_elem(q, qbase + d, dtype) * load_elem(k_cache, krow + d, dtype);
          w[t] = qk * scale;                    /* scaled before the softmax */
          mx = w[t] > mx ? w[t] : mx;
        }
        double total = 0.0;
        for (int64_t t = 0; t < lim; ++t) total += (w[t] = exp(w[t] - mx));
        for (int64_t d = 0; d < D; ++d) {
          double o = 0.0;
          for (int64_t t = 0; t < lim; ++t)
            o += w[t] * load_elem(v_cache, ((table[t / bs] * bs + t % bs) * KVH + g) * D + d, dtype);
          store_elem(out, qbase + d, dtype, o / total);
        }
      }
    }
    free(w);
  }
  return status;
}
