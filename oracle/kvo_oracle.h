/*
 * kvo_oracle.h -- plain CPU oracle for the tiered KV-cache hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  This library is the slow, obviously-correct
 * statement of what the GPU library computes.  It is linked by the tests, by
 * the package's smoke check and by the benchmark's CPU-baseline leg, and by
 * nothing else.  It shares no source, header, table or helper with the CUDA
 * library: every conversion (fp16/bf16 bit decoding, q8_0 blocks) is written
 * out again here from its definition.
 *
 * Floating point is evaluated in IEEE binary64 ("double"); compile with
 * -ffp-contract=off so no fused multiply-add changes the rounding between
 * the x86 development machine and the Arm GPU host.
 *
 * Storage formats read by the oracle (raw bytes, exactly what the GPU side
 * reads):
 *   dtype 0 = fp16   IEEE binary16, little endian
 *   dtype 1 = bf16   upper 16 bits of an IEEE binary32, little endian
 *   dtype 2 = q8_0   34-byte block { uint16 d (fp16 bits); int8 qs[32] },
 *                    value[i] = d * qs[i]; a cell row holds n_kv_heads heads,
 *                    each head_dim/32 consecutive blocks.
 *
 * Parity pins (checked by the CPU test-suite, against things other than this
 * file): fp16/bf16 decoding against numpy/torch over all 65,536 patterns;
 * sub-block pointers against a brute-force enumeration of the (block, j)
 * grid; swap against numpy slicing and the D2H-then-H2D round trip;
 * gather against numpy fancy indexing; attention against scipy's softmax with
 * numpy matmuls, and against closed forms (one cell gives v, q = 0 gives the
 * mean of v, a constant-per-head V gives the kv-head index, the causal
 * boundary gives pos/2 for V = position); the fold against the one-shot
 * softmax over the union of buckets; the sparse-row attention against a
 * numpy/scipy gather-and-softmax (padding, order, duplicates, one selection
 * gives v, every earlier position gives the causal prefill row); the staging
 * rule against the page's own worked example.
 */
#ifndef KVO_ORACLE_H
#define KVO_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_Q8_0 = 2 };

/* Exact decodings of the two 16-bit float formats. */
double orc_half_to_double(uint16_t bits);
double orc_bf16_to_double(uint16_t bits);

/* Bytes of one cell row (n_kv_heads heads of head_dim values) in a dtype;
 * 0 for an unknown dtype or a q8_0 head_dim that is not a multiple of 32. */
int64_t orc_row_bytes(int dtype, int64_t n_kv_heads, int64_t head_dim);

/* Decode head `head` of one cell row into head_dim doubles. */
void orc_load_head(const uint8_t *row, int dtype, int64_t head_dim,
                   int64_t head, double *out);

/* vLLM gpu_worker.py, compute_sub_block_ptrs: pointer of sub-block j of
 * block b is base + b*row_stride + j*(row_bytes/bpc); the (n_ids x bpc) grid
 * is flattened row-major and out = flat[skip : skip + n_out].
 * Returns 0, or -1 on an argument the page's asserts reject
 * (skip >= bpc, row_bytes % bpc != 0) or on n_out beyond the grid. */
int orc_sub_block_ptrs(const int64_t *block_ids, int64_t n_ids,
                       int64_t blocks_per_chunk, int64_t skip_count,
                       uint64_t base, int64_t row_stride_bytes,
                       int64_t row_bytes, uint64_t *out, int64_t n_out);

/* vLLM gpu_worker.py, transfer_async -> swap_blocks_batch: for i in
 * index order, copy sizes[i] bytes from address src[i] to address dst[i]
 * (all host addresses here). */
void orc_swap_blocks(const uint64_t *src, const uint64_t *dst,
                     const int64_t *sizes, int64_t n);

/* ExLlamaV3 qsa-kv-offload patch, staged gather (index_select of whole
 * pages): for each sequence s, kv head h and rank r, block sel[s][h][r]
 * (block_tokens tokens) of plane [s][token][h][:] is copied to
 * out[s][r*block_tokens + t][h][:] for t < block_tokens.
 * Planes are [n_seq][seq_stride_tokens][n_kv_heads][head_dim] elements of
 * elem_bytes; out is [n_seq][n_sel*block_tokens][n_kv_heads][head_dim].
 * Returns 0, or -1 when a selected block lies outside the plane. */
int orc_gather_blocks(const uint8_t *plane, int64_t n_seq,
                      int64_t seq_stride_tokens, int64_t n_kv_heads,
                      int64_t head_dim, int64_t elem_bytes,
                      int64_t block_tokens, const int32_t *sel,
                      int64_t n_sel, uint8_t *out);

/* vLLM gpu_worker.py, _build_copy_plan: run r of a ref's mapping has
 * num_fragments[r] fragments of fragment_size[r] bytes; fragment i sits at
 * local_offset[r] + i*local_stride[r] in the worker's block and at
 * canonical_offset[r] + i*canonical_stride[r] in the canonical block.
 * Fragments are listed run by run; source/destination offsets are (local,
 * canonical) for a GPU->CPU transfer and (canonical, local) otherwise.
 * Returns the fragment count, or -1 if it exceeds cap. */
int64_t orc_copy_plan(const int64_t *local_offset, const int64_t *local_stride,
                      const int64_t *canonical_offset,
                      const int64_t *canonical_stride,
                      const int64_t *num_fragments,
                      const int64_t *fragment_size, int64_t n_runs,
                      int gpu_to_cpu, int64_t *frag_src, int64_t *frag_dst,
                      int64_t *frag_sizes, int64_t cap);

/* vLLM gpu_worker.py, _fill_canonical_ops (step 3): one descriptor per
 * (block, fragment), block-major: out[b*n_frags + f] = base[b] + offset[f],
 * sizes[b*n_frags + f] = frag_sizes[f]. */
void orc_fragment_ptrs(const uint64_t *src_bases, const uint64_t *dst_bases,
                       int64_t n_blocks, const int64_t *frag_src,
                       const int64_t *frag_dst, const int64_t *frag_sizes,
                       int64_t n_frags, uint64_t *out_src, uint64_t *out_dst,
                       int64_t *out_sizes);

/* Tiered cache addressing (llama.cpp PR "tiered KV cache (--kv-vram-cells)"):
 * cell j of sequence b lives at
 *   head + (b*head_seq_stride_rows + j) * row_bytes          if j <  n_vram
 *   tail + (b*tail_seq_stride_rows + j - n_vram) * row_bytes if j >= n_vram
 */
typedef struct {
  const uint8_t *k_head, *v_head, *k_tail, *v_tail;
  int64_t head_seq_stride_rows, tail_seq_stride_rows;
  int64_t n_vram;
  int dtype;
  int64_t n_kv_heads, head_dim;
} orc_cache;

/* Softmax attention over cells [c0, c1) of sequence b for one q head
 * (already decoded to doubles), kv head = q_head / (n_q_heads/n_kv_heads).
 * Unnormalised partial: m = max_j s_j, l = sum_j exp(s_j - m),
 * acc[d] = sum_j exp(s_j - m) v_j[d], with s_j = scale * q . k_j.
 * An empty range gives m = -inf, l = 0, acc = 0. */
void orc_attn_partial(const orc_cache *c, int64_t b, int64_t kv_head,
                      const double *q, double scale, int64_t c0, int64_t c1,
                      double *m, double *l, double *acc);

/* One-step online-softmax fold (ExLlamaV3 qsa-kv-offload patch, the fold of
 * a bucket's partial (o, m, l) into the running (acc, m, l)):
 *   m' = max(m, m_b); alpha = exp(m - m') (0 if m = -inf);
 *   beta = exp(m_b - m') (0 if m_b = -inf);
 *   acc = alpha*acc + beta*acc_b; l = alpha*l + beta*l_b; m = m'. */
void orc_fold(double *m, double *l, double *acc, double m_b, double l_b,
              const double *acc_b, int64_t head_dim);

/* GQA decode: out[b][h][:] = softmax_j(scale * q[b][h] . k_j) v_j over
 * cells j < ctx_len[b] of sequence b.  q is [batch][n_q_heads][head_dim] of
 * q_dtype (fp16 or bf16).  out is [batch][n_q_heads][head_dim] doubles. */
void orc_attn_decode(const orc_cache *c, const uint16_t *q, int q_dtype,
                     int64_t batch, int64_t n_q_heads,
                     const int32_t *ctx_len, double scale, double *out);

/* Causal chunked prefill for one sequence: row i of q ([rows][n_q_heads]
 * [head_dim], bf16 or fp16) sits at position q_pos0 + i and attends cells
 * j <= q_pos0 + i (and j < ctx_len).  out is [rows][n_q_heads][head_dim]. */
void orc_attn_prefill(const orc_cache *c, const uint16_t *q, int q_dtype,
                      int64_t rows, int64_t q_pos0, int64_t n_q_heads,
                      int64_t ctx_len, double scale, double *out);

/* ExLlamaV3 qsa-kv-offload patch, qsa_staging_worthwhile: staging the page
 * range through the VRAM arena pays when the direct gather would read more
 * cache positions (rows * k_pad, every row its own selection) than twice the
 * positions staging reads once (num_pages_used * page_size).  Returns 1 or 0
 * (0 as well when staging is disabled). */
int orc_staging_worthwhile(int64_t rows, int64_t k_pad, int64_t num_pages_used,
                           int64_t page_size, int enabled);

/* ExLlamaV3 qsa-kv-offload patch, qsa_sparse_attend_rows(_staged): query
 * row r (n_q_heads heads of head_dim, fp16 or bf16) attends to the cache
 * positions indices[r][0 .. k_pad) that are >= 0 and below
 * num_pages_used * page_size; the others are padding.  Position p is slot
 * p % page_size of page block_table[p / page_size] of the paged planes
 * k_pages / v_pages ([pages][page_size][n_kv_heads][head_dim], fp16 or bf16),
 * and q head h reads kv head h / (n_q_heads / n_kv_heads):
 *     out[r][h] = sum_p softmax_p(scale * q[r][h] . k_p) v_p
 * over the selected positions (a position listed twice counts twice).  A row
 * with no selection gives 0 (acc / max(l, 1e-30)). */
void orc_attn_sparse_rows(const uint8_t *k_pages, const uint8_t *v_pages,
                          int dtype, int64_t page_size, int64_t n_kv_heads,
                          int64_t head_dim, const int32_t *block_table,
                          int64_t num_pages_used, const int32_t *indices,
                          int64_t rows, int64_t k_pad, const uint16_t *q,
                          int q_dtype, int64_t n_q_heads, double scale,
                          double *out);

/* IEEE binary32 -> binary16 bits, round to nearest, ties to even (with
 * subnormals, overflow to infinity, NaN kept quiet). */
uint16_t orc_float_to_half_bits(float x);

/* q8_0 quantisation of one 32-value block (the usual q8_0 rule; the pages
 * name the format but not the rounding, so this is a stated reading),
 * evaluated in binary32): amax = max|x|, d = amax / 127, id = d ? 1/d : 0,
 * qs[i] = round-half-away-from-zero(x[i] * id); the block stores d as fp16.
 * Writes 34 bytes {fp16 d; int8 qs[32]}. */
void orc_quantize_q8_0_block(const float *x, uint8_t *blk);

/* Append (write path of the tiered cache): tokens t < n_new of k_new / v_new
 * ([n_new][n_kv_heads][head_dim], src dtype fp16 or bf16) become cells
 * pos0 + t of one sequence: cell j < n_vram goes to head row j, cell
 * j >= n_vram to tail row j - n_vram, stored in the cache dtype (a copy for
 * fp16/bf16 equal to the source dtype; q8_0 quantised per 32-value block of
 * each head).  The cache pointers are those of an orc_cache (k_head ...
 * v_tail), written through.  Returns 0, or -1 on a dtype pair the cache
 * cannot hold. */
int orc_append_kv(const uint8_t *k_new, const uint8_t *v_new, int src_dtype,
                  int64_t n_new, int64_t pos0, int64_t n_kv_heads,
                  int64_t head_dim, uint8_t *k_head, uint8_t *v_head,
                  uint8_t *k_tail, uint8_t *v_tail, int dtype,
                  int64_t n_vram);

/* Worker threads used by orc_attn_decode / orc_attn_prefill (independent
 * (row, head) outputs are distributed; each is computed exactly as in the
 * serial loop).  Returns the count in effect; 1 without OpenMP. */
int orc_set_threads(int n);

#ifdef __cplusplus
}
#endif
#endif
