/*
 * kvo_oracle.c -- plain CPU oracle (test infrastructure only; see the header).
 *
 * Every function follows the definition it names in the header, in the
 * order the source pages state it, with no blocking, fusion or reordering.
 */
#include "kvo_oracle.h"

#include <math.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits.  Subnormals are f * 2^-24; normals (1024 + f) * 2^(e - 25). */
double orc_half_to_double(uint16_t bits) {
  int sign = (bits >> 15) & 1;
  int e = (bits >> 10) & 0x1f;
  int f = bits & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24);
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + f), e - 25);
  }
  return sign ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits.
 * Subnormals are f * 2^-133; normals (128 + f) * 2^(e - 134). */
double orc_bf16_to_double(uint16_t bits) {
  int sign = (bits >> 15) & 1;
  int e = (bits >> 7) & 0xff;
  int f = bits & 0x7f;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -133);
  } else if (e == 255) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp((double)(128 + f), e - 134);
  }
  return sign ? -v : v;
}

int64_t orc_row_bytes(int dtype, int64_t n_kv_heads, int64_t head_dim) {
  if (dtype == ORC_F16 || dtype == ORC_BF16) return n_kv_heads * head_dim * 2;
  if (dtype == ORC_Q8_0) {
    if (head_dim % 32) return 0;
    return n_kv_heads * (head_dim / 32) * 34;
  }
  return 0;
}

static uint16_t rd16(const uint8_t *p) {
  return (uint16_t)(p[0] | ((uint16_t)p[1] << 8));
}

void orc_load_head(const uint8_t *row, int dtype, int64_t head_dim,
                   int64_t head, double *out) {
  int64_t d;
  if (dtype == ORC_F16 || dtype == ORC_BF16) {
    const uint8_t *h = row + head * head_dim * 2;
    for (d = 0; d < head_dim; ++d) {
      uint16_t bits = rd16(h + 2 * d);
      out[d] = dtype == ORC_F16 ? orc_half_to_double(bits)
                                : orc_bf16_to_double(bits);
    }
  } else {
    /* q8_0: head `head` owns blocks head*(D/32) .. head*(D/32) + D/32 - 1. */
    int64_t nb = head_dim / 32;
    for (d = 0; d < head_dim; ++d) {
      const uint8_t *blk = row + (head * nb + d / 32) * 34;
      double scale = orc_half_to_double(rd16(blk));
      int8_t q = (int8_t)blk[2 + d % 32];
      out[d] = scale * (double)q;
    }
  }
}

int orc_sub_block_ptrs(const int64_t *block_ids, int64_t n_ids,
                       int64_t blocks_per_chunk, int64_t skip_count,
                       uint64_t base, int64_t row_stride_bytes,
                       int64_t row_bytes, uint64_t *out, int64_t n_out) {
  int64_t i;
  if (blocks_per_chunk < 1 || skip_count < 0 || skip_count >= blocks_per_chunk)
    return -1;
  if (blocks_per_chunk > 1 && row_bytes % blocks_per_chunk != 0) return -1;
  if (n_out < 0 || n_out + skip_count > n_ids * blocks_per_chunk) return -1;
  {
    uint64_t page = (uint64_t)(row_bytes / blocks_per_chunk);
    for (i = 0; i < n_out; ++i) {
      int64_t flat = i + skip_count;
      int64_t k = flat / blocks_per_chunk; /* which block id */
      int64_t j = flat % blocks_per_chunk; /* which sub-block inside it */
      out[i] = base + (uint64_t)block_ids[k] * (uint64_t)row_stride_bytes +
               (uint64_t)j * page;
    }
  }
  return 0;
}

void orc_swap_blocks(const uint64_t *src, const uint64_t *dst,
                     const int64_t *sizes, int64_t n) {
  int64_t i;
  for (i = 0; i < n; ++i)
    memcpy((void *)(uintptr_t)dst[i], (const void *)(uintptr_t)src[i],
           (size_t)sizes[i]);
}

int orc_gather_blocks(const uint8_t *plane, int64_t n_seq,
                      int64_t seq_stride_tokens, int64_t n_kv_heads,
                      int64_t head_dim, int64_t elem_bytes,
                      int64_t block_tokens, const int32_t *sel,
                      int64_t n_sel, uint8_t *out) {
  int64_t s, h, r, t;
  int64_t head_bytes = head_dim * elem_bytes;
  int64_t out_tokens = n_sel * block_tokens;
  for (s = 0; s < n_seq; ++s)
    for (h = 0; h < n_kv_heads; ++h)
      for (r = 0; r < n_sel; ++r) {
        int64_t blk = sel[(s * n_kv_heads + h) * n_sel + r];
        if (blk < 0 || (blk + 1) * block_tokens > seq_stride_tokens) return -1;
        for (t = 0; t < block_tokens; ++t) {
          int64_t src_tok = blk * block_tokens + t;
          int64_t dst_tok = r * block_tokens + t;
          memcpy(out + ((s * out_tokens + dst_tok) * n_kv_heads + h) * head_bytes,
                 plane + ((s * seq_stride_tokens + src_tok) * n_kv_heads + h) * head_bytes,
                 (size_t)head_bytes);
        }
      }
  return 0;
}

int64_t orc_copy_plan(const int64_t *local_offset, const int64_t *local_stride,
                      const int64_t *canonical_offset,
                      const int64_t *canonical_stride,
                      const int64_t *num_fragments,
                      const int64_t *fragment_size, int64_t n_runs,
                      int gpu_to_cpu, int64_t *frag_src, int64_t *frag_dst,
                      int64_t *frag_sizes, int64_t cap) {
  int64_t r, i, n = 0;
  for (r = 0; r < n_runs; ++r)
    for (i = 0; i < num_fragments[r]; ++i) {
      int64_t local = local_offset[r] + i * local_stride[r];
      int64_t canonical = canonical_offset[r] + i * canonical_stride[r];
      if (n >= cap) return -1;
      frag_src[n] = gpu_to_cpu ? local : canonical;
      frag_dst[n] = gpu_to_cpu ? canonical : local;
      frag_sizes[n] = fragment_size[r];
      ++n;
    }
  return n;
}

void orc_fragment_ptrs(const uint64_t *src_bases, const uint64_t *dst_bases,
                       int64_t n_blocks, const int64_t *frag_src,
                       const int64_t *frag_dst, const int64_t *frag_sizes,
                       int64_t n_frags, uint64_t *out_src, uint64_t *out_dst,
                       int64_t *out_sizes) {
  int64_t b, f;
  for (b = 0; b < n_blocks; ++b)
    for (f = 0; f < n_frags; ++f) {
      out_src[b * n_frags + f] = src_bases[b] + (uint64_t)frag_src[f];
      out_dst[b * n_frags + f] = dst_bases[b] + (uint64_t)frag_dst[f];
      out_sizes[b * n_frags + f] = frag_sizes[f];
    }
}

static const uint8_t *cell_row(const orc_cache *c, const uint8_t *head,
                               const uint8_t *tail, int64_t b, int64_t j) {
  int64_t rb = orc_row_bytes(c->dtype, c->n_kv_heads, c->head_dim);
  if (j < c->n_vram) return head + (b * c->head_seq_stride_rows + j) * rb;
  return tail + (b * c->tail_seq_stride_rows + (j - c->n_vram)) * rb;
}

/* Scratch bound: head_dim never exceeds this in the oracle. */
#define ORC_MAX_D 1024

void orc_attn_partial(const orc_cache *c, int64_t b, int64_t kv_head,
                      const double *q, double scale, int64_t c0, int64_t c1,
                      double *m, double *l, double *acc) {
  int64_t D = c->head_dim, j, d;
  double kd[ORC_MAX_D], vd[ORC_MAX_D];
  double mx = -INFINITY, sum = 0.0;
  for (d = 0; d < D; ++d) acc[d] = 0.0;
  /* pass 1: the maximum logit */
  for (j = c0; j < c1; ++j) {
    double s = 0.0;
    orc_load_head(cell_row(c, c->k_head, c->k_tail, b, j), c->dtype, D, kv_head, kd);
    for (d = 0; d < D; ++d) s += q[d] * kd[d];
    s *= scale;
    if (s > mx) mx = s;
  }
  /* pass 2: exp-weights and the weighted sum of V */
  if (c1 > c0) {
    for (j = c0; j < c1; ++j) {
      double s = 0.0, p;
      orc_load_head(cell_row(c, c->k_head, c->k_tail, b, j), c->dtype, D, kv_head, kd);
      orc_load_head(cell_row(c, c->v_head, c->v_tail, b, j), c->dtype, D, kv_head, vd);
      for (d = 0; d < D; ++d) s += q[d] * kd[d];
      s *= scale;
      p = exp(s - mx);
      sum += p;
      for (d = 0; d < D; ++d) acc[d] += p * vd[d];
    }
  }
  *m = mx;
  *l = sum;
}

void orc_fold(double *m, double *l, double *acc, double m_b, double l_b,
              const double *acc_b, int64_t head_dim) {
  double m_new = *m > m_b ? *m : m_b;
  double alpha = *m > -INFINITY ? exp(*m - m_new) : 0.0;
  double beta = m_b > -INFINITY ? exp(m_b - m_new) : 0.0;
  int64_t d;
  for (d = 0; d < head_dim; ++d) acc[d] = alpha * acc[d] + beta * acc_b[d];
  *l = alpha * *l + beta * l_b;
  *m = m_new;
}

static void load_q(const uint16_t *q, int q_dtype, int64_t D, double *out) {
  int64_t d;
  for (d = 0; d < D; ++d)
    out[d] = q_dtype == ORC_F16 ? orc_half_to_double(q[d])
                                : orc_bf16_to_double(q[d]);
}

void orc_attn_decode(const orc_cache *c, const uint16_t *q, int q_dtype,
                     int64_t batch, int64_t n_q_heads,
                     const int32_t *ctx_len, double scale, double *out) {
  int64_t D = c->head_dim;
  int64_t group = n_q_heads / c->n_kv_heads;
  int64_t task;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (task = 0; task < batch * n_q_heads; ++task) {
    int64_t b = task / n_q_heads, h = task % n_q_heads, d;
    double qd[ORC_MAX_D], m, l;
    double *o = out + task * D;
    load_q(q + task * D, q_dtype, D, qd);
    orc_attn_partial(c, b, h / group, qd, scale, 0, ctx_len[b], &m, &l, o);
    /* final normalisation o = acc / max(l, 1e-30): an empty context gives 0 */
    if (l < 1e-30) l = 1e-30;
    for (d = 0; d < D; ++d) o[d] /= l;
  }
}

void orc_attn_prefill(const orc_cache *c, const uint16_t *q, int q_dtype,
                      int64_t rows, int64_t q_pos0, int64_t n_q_heads,
                      int64_t ctx_len, double scale, double *out) {
  int64_t D = c->head_dim;
  int64_t group = n_q_heads / c->n_kv_heads;
  int64_t task;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (task = 0; task < rows * n_q_heads; ++task) {
    int64_t i = task / n_q_heads, h = task % n_q_heads, d;
    int64_t end = q_pos0 + i + 1; /* causal: cells 0 .. q_pos0 + i */
    double qd[ORC_MAX_D], m, l;
    double *o = out + task * D;
    if (end > ctx_len) end = ctx_len;
    load_q(q + task * D, q_dtype, D, qd);
    orc_attn_partial(c, 0, h / group, qd, scale, 0, end, &m, &l, o);
    if (l < 1e-30) l = 1e-30;
    for (d = 0; d < D; ++d) o[d] /= l;
  }
}

int orc_staging_worthwhile(int64_t rows, int64_t k_pad, int64_t num_pages_used,
                           int64_t page_size, int enabled) {
  return enabled && rows * k_pad > 2 * num_pages_used * page_size;
}

/* Row of position p in the paged planes, or NULL when p is padding. */
static const uint8_t *paged_row(const uint8_t *pages, int64_t p, int64_t page_size,
                                const int32_t *block_table, int64_t num_pages_used,
                                int64_t row_bytes) {
  if (p < 0 || p >= num_pages_used * page_size) return NULL;
  return pages + ((int64_t)block_table[p / page_size] * page_size + p % page_size) * row_bytes;
}

void orc_attn_sparse_rows(const uint8_t *k_pages, const uint8_t *v_pages,
                          int dtype, int64_t page_size, int64_t n_kv_heads,
                          int64_t head_dim, const int32_t *block_table,
                          int64_t num_pages_used, const int32_t *indices,
                          int64_t rows, int64_t k_pad, const uint16_t *q,
                          int q_dtype, int64_t n_q_heads, double scale,
                          double *out) {
  int64_t D = head_dim, group = n_q_heads / n_kv_heads;
  int64_t rb = orc_row_bytes(dtype, n_kv_heads, head_dim);
  int64_t task;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (task = 0; task < rows * n_q_heads; ++task) {
    int64_t r = task / n_q_heads, h = task % n_q_heads, g = h / group, k, d;
    const int32_t *sel = indices + r * k_pad;
    double qd[ORC_MAX_D], kd[ORC_MAX_D], vd[ORC_MAX_D];
    double mx = -INFINITY, sum = 0.0;
    double *o = out + task * D;
    load_q(q + task * D, q_dtype, D, qd);
    for (d = 0; d < D; ++d) o[d] = 0.0;
    /* pass 1: the maximum logit over the selected positions */
    for (k = 0; k < k_pad; ++k) {
      const uint8_t *kr = paged_row(k_pages, sel[k], page_size, block_table, num_pages_used, rb);
      double s = 0.0;
      if (!kr) continue;
      orc_load_head(kr, dtype, D, g, kd);
      for (d = 0; d < D; ++d) s += qd[d] * kd[d];
      s *= scale;
      if (s > mx) mx = s;
    }
    /* pass 2: exp-weights and the weighted sum of V */
    for (k = 0; k < k_pad; ++k) {
      const uint8_t *kr = paged_row(k_pages, sel[k], page_size, block_table, num_pages_used, rb);
      const uint8_t *vr = paged_row(v_pages, sel[k], page_size, block_table, num_pages_used, rb);
      double s = 0.0, p;
      if (!kr) continue;
      orc_load_head(kr, dtype, D, g, kd);
      orc_load_head(vr, dtype, D, g, vd);
      for (d = 0; d < D; ++d) s += qd[d] * kd[d];
      s *= scale;
      p = exp(s - mx);
      sum += p;
      for (d = 0; d < D; ++d) o[d] += p * vd[d];
    }
    if (sum < 1e-30) sum = 1e-30;
    for (d = 0; d < D; ++d) o[d] /= sum;
  }
}

uint16_t orc_float_to_half_bits(float x) {
  /* decompose |x| = m * 2^e exactly in binary64, then round m to the
   * binary16 grid at that exponent */
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  double a = fabs((double)x);
  int e;
  double m, q, r;
  long long n;
  if (isnan(x)) return (uint16_t)(sign | 0x7e00u);
  if (isinf(x)) return (uint16_t)(sign | 0x7c00u);
  if (a == 0.0) return sign;
  frexp(a, &e);                      /* a = f * 2^e, f in [0.5, 1) */
  /* binary16 spacing: 2^(e-11) for normals (e >= -13), 2^-24 below */
  {
    int ulp_exp = e - 11;
    if (ulp_exp < -24) ulp_exp = -24;
    m = ldexp(a, -ulp_exp);          /* a in units of the spacing */
    q = floor(m);
    r = m - q;
    n = (long long)q;
    if (r > 0.5 || (r == 0.5 && (n & 1))) n += 1;
    a = ldexp((double)n, ulp_exp);   /* rounded magnitude */
  }
  if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u);  /* overflow */
  if (a < ldexp(1.0, -14)) {         /* subnormal (or rounded up to min normal) */
    n = (long long)ldexp(a, 24);
    return (uint16_t)(sign | (uint16_t)n);
  }
  frexp(a, &e);
  {
    int be = e - 1 + 15;             /* biased exponent */
    long long frac = (long long)ldexp(a, 11 - e) - 1024;  /* 10 fraction bits */
    return (uint16_t)(sign | (uint16_t)(be << 10) | (uint16_t)frac);
  }
}

void orc_quantize_q8_0_block(const float *x, uint8_t *blk) {
  float amax = 0.0f, d, id;
  uint16_t dh;
  int i;
  for (i = 0; i < 32; ++i) {
    float ax = fabsf(x[i]);
    if (ax > amax) amax = ax;
  }
  d = amax / 127.0f;
  id = d != 0.0f ? 1.0f / d : 0.0f;
  dh = orc_float_to_half_bits(d);
  blk[0] = (uint8_t)(dh & 0xff);
  blk[1] = (uint8_t)(dh >> 8);
  for (i = 0; i < 32; ++i) {
    float v = x[i] * id;
    blk[2 + i] = (uint8_t)(int8_t)roundf(v);
  }
}

int orc_append_kv(const uint8_t *k_new, const uint8_t *v_new, int src_dtype,
                  int64_t n_new, int64_t pos0, int64_t n_kv_heads,
                  int64_t head_dim, uint8_t *k_head, uint8_t *v_head,
                  uint8_t *k_tail, uint8_t *v_tail, int dtype,
                  int64_t n_vram) {
  int64_t t, h, b, d;
  int64_t src_row = n_kv_heads * head_dim * 2;
  int64_t rb = orc_row_bytes(dtype, n_kv_heads, head_dim);
  if (src_dtype != ORC_F16 && src_dtype != ORC_BF16) return -1;
  if (dtype != ORC_Q8_0 && dtype != src_dtype) return -1;
  if (rb == 0) return -1;
  for (t = 0; t < n_new; ++t) {
    int64_t j = pos0 + t;
    int which;
    for (which = 0; which < 2; ++which) {
      const uint8_t *src = (which ? v_new : k_new) + t * src_row;
      uint8_t *dst = j < n_vram ? (which ? v_head : k_head) + j * rb
                                : (which ? v_tail : k_tail) + (j - n_vram) * rb;
      if (dtype != ORC_Q8_0) {
        memcpy(dst, src, (size_t)rb);
        continue;
      }
      for (h = 0; h < n_kv_heads; ++h) {
        for (b = 0; b < head_dim / 32; ++b) {
          float x[32];
          for (d = 0; d < 32; ++d) {
            const uint8_t *e = src + (h * head_dim + b * 32 + d) * 2;
            uint16_t bits = (uint16_t)(e[0] | (e[1] << 8));
            /* exact: every fp16 / bf16 value is a binary32 value */
            x[d] = (float)(src_dtype == ORC_F16 ? orc_half_to_double(bits)
                                                : orc_bf16_to_double(bits));
          }
          orc_quantize_q8_0_block(x, dst + (h * (head_dim / 32) + b) * 34);
        }
      }
    }
  }
  return 0;
}

int orc_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
  return omp_get_max_threads();
#else
  (void)n;
  return 1;
#endif
}
