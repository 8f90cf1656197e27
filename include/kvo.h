/*
 * kvo.h -- C ABI of libkvo, a GB300 (sm_103a) library for an LLM KV cache
 * that lives partly in VRAM and partly in pinned, device-mapped host memory.
 *
 * Conventions shared by every entry point:
 *   - The caller owns every buffer.  The library allocates no memory of its
 *     own accord: only the VMM tiers kvo_vmm_tier_create makes on request
 *     (freed by kvo_vmm_tier_destroy), and the fixed device scratch array of
 *     kvo_attn_decode_tiered_noalloc.
 *   - "device-accessible" means device memory (cudaMalloc / a framework's
 *     allocator), pinned host memory that is mapped into the device's
 *     address space (cudaHostAlloc(..., Mapped) / cudaHostRegister(...,
 *     Mapped)), or a range of a VMM tier; all are passed by the same unified
 *     virtual address.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  All calls except kvo_sub_block_ptrs are stream-ordered and
 *     asynchronous: they return once the work is enqueued, do no host
 *     synchronisation, and every buffer must stay valid until the stream has
 *     passed the enqueued work.
 *   - Every call returns a kvo_status.  Nothing aborts or throws.  An
 *     argument the host can check is rejected before anything is enqueued;
 *     kvo_last_error() then holds a one-line reason (thread-local).
 *     Asynchronous CUDA faults surface as KVO_ERR_CUDA on a later call or at
 *     the caller's synchronisation.  Values the host cannot see (selected
 *     block ids in device memory) are range-checked by the kernels, which
 *     skip an out-of-range item and set a bit read by kvo_device_errors().
 *   - There is no CPU fallback: a combination a kernel does not implement
 *     returns KVO_ERR_UNSUPPORTED.
 */
#ifndef KVO_H
#define KVO_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KVO_OK = 0,
  KVO_ERR_ARG = -1,          /* a size, count or pointer is invalid            */
  KVO_ERR_ALIGN = -2,        /* a pointer or row size breaks a 16-byte rule    */
  KVO_ERR_NOT_MAPPED = -3,   /* a buffer is not device-accessible              */
  KVO_ERR_UNSUPPORTED = -4,  /* dtype / head_dim / group size not implemented  */
  KVO_ERR_CUDA = -5,         /* a CUDA runtime call failed                     */
  KVO_ERR_WORKSPACE = -6     /* workspace missing or smaller than required     */
} kvo_status;

typedef enum {
  KVO_F16 = 0,   /* IEEE binary16                                           */
  KVO_BF16 = 1,  /* bfloat16                                                */
  KVO_Q8_0 = 2   /* 34-byte block {fp16 d; int8 qs[32]}, value = d * qs[i];   */
                 /* a cell row holds n_kv_heads heads of head_dim/32 blocks  */
} kvo_dtype;

/* Static text for a status code. */
const char *kvo_status_string(int status);

/* Detail of the last failing call on this host thread ("" if none). */
const char *kvo_last_error(void);

/* Bits set by kernels that met a condition the host could not check:
 *   bit 0 (1): a gather selection outside its plane (the block was skipped);
 *   bit 1 (2): a sparse-rows page-table entry outside the planes (its picks
 *              counted as padding);
 *   bit 2 (4): a bounded barrier wait gave up (about 2 s without progress;
 *              the kernel wound down after its own copies and MMAs landed,
 *              and its output is not valid);
 *   bit 3 (8): a CTA could not align its shared memory and exited;
 *   bit 4 (16): the tensor-core prefill over a bf16 cache met a V value of
 *              magnitude 65520 or more (or infinite), which its fp16 PV
 *              product cannot hold; that call's output is not valid.
 * Synchronises the device; clears the bits when `clear` is non-zero.  For
 * tests and debugging, not for hot loops. */
int kvo_device_errors(uint32_t *bits, int clear);

/* kvo_selftest_wait_timeout -- runs the library's bounded barrier wait (the
 * one every tensor-core prefill wait uses) on a barrier that nothing
 * completes, with limit_ns in place of the kernels' ~2 s: the wait gives up,
 * sets bit 2 of kvo_device_errors() and the kernel returns.  For testing the
 * failure path without a fault; the context stays usable.  The pages have no
 * counterpart.  Errors: KVO_ERR_ARG (limit_ns 0 or above 10 s),
 * KVO_ERR_CUDA. */
int kvo_selftest_wait_timeout(uint64_t limit_ns, void *stream);

/* ------------------------------------------------------------------------
 * kvo_sub_block_ptrs -- host function, synchronous, no CUDA.
 *
 * vLLM gpu_worker.py (v1 CPU KV offload), compute_sub_block_ptrs: block b
 * of a paged tensor is split into blocks_per_chunk sub-blocks of
 * page = row_bytes / blocks_per_chunk bytes; sub-block j of block b is at
 *     base + b * row_stride_bytes + j * page.
 * The (n_ids x blocks_per_chunk) grid is flattened row-major and
 *     out[i] = flat[skip_count + i],  0 <= i < n_out
 * i.e. (k, j) = divmod(i + skip_count, blocks_per_chunk), block b = ids[k].
 * row_stride_bytes may exceed row_bytes (a non-contiguous host tensor).
 *
 * block_ids: host int64[n_ids]; out: host int64[n_out] (addresses as int64,
 * the descriptor type kvo_swap_blocks_batch takes).
 * Errors: KVO_ERR_ARG if skip_count >= blocks_per_chunk (the page's assert),
 * row_bytes % blocks_per_chunk != 0 with blocks_per_chunk > 1 (the page's
 * assert), n_out + skip_count > n_ids * blocks_per_chunk, a negative size,
 * or a NULL array with a non-zero count.
 * ---------------------------------------------------------------------- */
int kvo_sub_block_ptrs(const int64_t *block_ids, int64_t n_ids,
                       int64_t blocks_per_chunk, int64_t skip_count,
                       uint64_t base, int64_t row_stride_bytes,
                       int64_t row_bytes, int64_t *out, int64_t n_out);

/* ------------------------------------------------------------------------
 * kvo_shard_range -- host function, synchronous, no CUDA: the contiguous
 * share of n_units work units (swap descriptors, sequences of a gather or a
 * decode batch) that rank `rank` of `world` processes takes.
 *
 * vLLM gpu_worker.py (transfer_async: each block's descriptors are
 * independent) and the ExLlamaV3 qsa-kv-offload patch (each sequence's
 * selection is independent): the path splits with no exchange step, so one
 * process per GPU takes
 *     [*lo, *hi) = [floor(n_units * rank / world), floor(n_units * (rank + 1) / world))
 * -- the ranks' ranges are disjoint, cover [0, n_units) exactly once, in
 * rank order, and differ in size by at most one unit.  A rank's call then
 * passes the descriptor arrays offset by *lo (count *hi - *lo), or the
 * sequence-indexed buffers offset by *lo sequences.
 * Errors: KVO_ERR_ARG (n_units < 0, world < 1, rank outside [0, world),
 *   NULL lo or hi).
 * ---------------------------------------------------------------------- */
int kvo_shard_range(int64_t n_units, int64_t world, int64_t rank, int64_t *lo,
                    int64_t *hi);

/* ------------------------------------------------------------------------
 * kvo_copy_plan / kvo_fragment_ptrs -- host functions, synchronous, no CUDA:
 * descriptors for a canonical host layout, fed to kvo_swap_blocks_batch.
 *
 * vLLM gpu_worker.py, _build_copy_plan: in a canonical layout one cache
 * block is scattered as fragments that come from mapping runs.  Run r has
 * num_fragments[r] fragments of fragment_size[r] bytes; fragment i sits at
 * local_offset[r] + i * local_stride[r] in the worker's block and at
 * canonical_offset[r] + i * canonical_stride[r] in the canonical block.
 * kvo_copy_plan lists the fragments run by run into frag_src / frag_dst /
 * frag_sizes (int64[capacity], host): source and destination offsets are
 * (local, canonical) when gpu_to_cpu is non-zero, (canonical, local)
 * otherwise; *n_frags receives the count.
 *
 * vLLM gpu_worker.py, _fill_canonical_ops (its step 3): kvo_fragment_ptrs
 * expands per-block base addresses (e.g. from kvo_sub_block_ptrs) and the
 * plan into one descriptor per (block, fragment), block-major:
 *     out_src[b * n_frags + f] = src_bases[b] + frag_src[f]
 *     out_dst[b * n_frags + f] = dst_bases[b] + frag_dst[f]
 *     out_sizes[b * n_frags + f] = frag_sizes[f]
 * All arrays are host int64.  (The pages' multi-rank writer rotation is not
 * part of this.)
 * Errors: KVO_ERR_ARG for negative counts or sizes, NULL arrays with a
 * non-zero count, or more fragments than capacity.
 * ---------------------------------------------------------------------- */
int kvo_copy_plan(const int64_t *local_offset, const int64_t *local_stride,
                  const int64_t *canonical_offset,
                  const int64_t *canonical_stride,
                  const int64_t *num_fragments, const int64_t *fragment_size,
                  int64_t n_runs, int gpu_to_cpu, int64_t *frag_src,
                  int64_t *frag_dst, int64_t *frag_sizes, int64_t capacity,
                  int64_t *n_frags);

int kvo_fragment_ptrs(const int64_t *src_bases, const int64_t *dst_bases,
                      int64_t n_blocks, const int64_t *frag_src,
                      const int64_t *frag_dst, const int64_t *frag_sizes,
                      int64_t n_frags, int64_t *out_src, int64_t *out_dst,
                      int64_t *out_sizes);

/* ------------------------------------------------------------------------
 * kvo_swap_blocks_batch -- batched block copy between a paged device cache
 * and pinned host blocks.
 *
 * vLLM gpu_worker.py, transfer_async -> swap_blocks_batch(src, dst, sizes,
 * is_src_access_order_any): for every i < n, copy sizes[i] bytes from
 * address src[i] to address dst[i].  Ranges must not overlap; the order in
 * which descriptors are executed is unspecified.
 *
 * src, dst, sizes: int64[n] descriptor arrays in pinned host memory (the
 *   page's pooled pinned buffers).  In SM mode the kernel reads them through
 *   the device mapping while it runs; in copy-engine mode the host reads them
 *   during this call.
 * Each src[i] / dst[i] must be device-accessible; the library does not
 *   check descriptor targets (it would have to look up every one of them).
 *   Any alignment and size
 *   is accepted; descriptors whose two addresses and size are 16-byte
 *   multiples take the 16-byte vector path, others an 8-, 4- or 1-byte path.
 * flags: KVO_SWAP_H2D or KVO_SWAP_D2H (the direction; informational: both
 *   modes serve both); KVO_SWAP_SRC_ORDER_ANY (the page's
 *   is_src_access_order_any: the source is not written while the copy runs)
 *   is accepted and has no effect -- both modes read every source byte
 *   exactly once, in whatever order, so there is nothing a read-only or
 *   reordered path would save; KVO_SWAP_FORCE_CE selects the copy engine (one
 *   cudaMemcpyAsync per run of descriptors whose source and destination both
 *   continue the previous one; the host reads the descriptors during the
 *   call).  Default (and KVO_SWAP_FORCE_SM): the SM kernel, which reads the
 *   descriptors through the device mapping while it runs.  The default is a
 *   crossover measured on GB300 (2 KiB - 1 MiB pages, 64 and 2,048
 *   descriptors, both directions): the SM kernel is the faster mode in every
 *   cell -- a copy-engine call costs ~1.7 us to issue, and the copy engine
 *   moves 1 MiB copies at 126-147 GB/s against the SM kernel's 205-211 GB/s.
 *   A batch of at most KVO_SWAP_SHORT_BATCH descriptors in pinned host memory
 *   has its sizes read on the host (to cut large copies into pieces that
 *   spread over every SM).
 * n == 0 is a no-op.
 * Errors: KVO_ERR_ARG (n < 0, NULL arrays, both FORCE flags),
 *   KVO_ERR_NOT_MAPPED (descriptor arrays not device-accessible in SM mode,
 *   or not host-readable in copy-engine mode), KVO_ERR_CUDA.
 * ---------------------------------------------------------------------- */
#define KVO_SWAP_H2D 0x1u
#define KVO_SWAP_D2H 0x2u
#define KVO_SWAP_SRC_ORDER_ANY 0x4u
#define KVO_SWAP_FORCE_SM 0x8u
#define KVO_SWAP_FORCE_CE 0x10u
#define KVO_SWAP_SHORT_BATCH 64

int kvo_swap_blocks_batch(const int64_t *src, const int64_t *dst,
                          const int64_t *sizes, int64_t n, uint32_t flags,
                          void *stream);

/* ------------------------------------------------------------------------
 * kvo_gather_blocks -- top-k block gather from host-resident K/V planes.
 *
 * ExLlamaV3 qsa-kv-offload patch: K/V planes stay in pinned, mapped host
 * memory and only the selected blocks are read (the staged prefill copies
 * them into a VRAM arena with index_select of whole pages).  For sequence s,
 * kv head h and rank r < n_sel, block sel[s][h][r] (block_tokens tokens) is
 * copied:
 *     k_out[s][r*block_tokens + t][h][:] = k_plane[s][sel*block_tokens + t][h][:]
 * for t < block_tokens, and the same for V.
 *
 * k_plane, v_plane: [n_seq][seq_stride_tokens][n_kv_heads][head_dim] of
 *   dtype (pinned mapped host, or device memory).
 * sel: device-accessible int32 [n_seq][n_kv_heads][n_sel].
 * k_out, v_out: device [n_seq][n_sel*block_tokens][n_kv_heads][head_dim].
 * dtype: KVO_F16 or KVO_BF16; head_dim * 2 must be a multiple of 16 and all
 *   four buffers 16-byte aligned.
 * A selection outside [0, seq_stride_tokens / block_tokens) is skipped (its
 *   destination rows are left as they were) and sets bit 0 of
 *   kvo_device_errors().
 * Errors: KVO_ERR_ARG, KVO_ERR_ALIGN, KVO_ERR_NOT_MAPPED,
 *   KVO_ERR_UNSUPPORTED (q8_0), KVO_ERR_CUDA.
 * ---------------------------------------------------------------------- */
int kvo_gather_blocks(const void *k_plane, const void *v_plane, int64_t n_seq,
                      int64_t seq_stride_tokens, int64_t n_kv_heads,
                      int64_t head_dim, int dtype, int64_t block_tokens,
                      const int32_t *sel, int64_t n_sel, void *k_out,
                      void *v_out, void *stream);

/* ------------------------------------------------------------------------
 * kvo_attn_decode_tiered -- GQA decode attention over a tiered cache.
 *
 * llama.cpp PR "tiered KV cache (--kv-vram-cells)": cells [0, N) of each
 * sequence's K/V sit in VRAM and cells [N, L) in pinned host memory, and the
 * attention arithmetic does not depend on where a cell lives (output is
 * bit-identical to an all-VRAM cache).  For sequence b and q head h
 * (kv head g = h / (n_q_heads / n_kv_heads)):
 *     out[b][h] = sum_j softmax_j(scale * q[b][h] . k[b][j][g]) v[b][j][g]
 * over cells j < ctx_len[b], computed as split-K flash-decoding: fixed
 * cell ranges (a function of max_ctx, batch and the device's SM count only)
 * give partial (m, l, acc) in fp32, combined in a fixed order.  F16/BF16
 * caches: products q * k are exact (16-bit x 16-bit) and summed in fp32.
 * Q8_0 caches: each query head's slice of dims is rounded once to 16-bit
 * integers n with step s = max|q| / 32767 (|q - s n| <= s / 2), the block
 * dot products with the int8 values are exact integer sums, scaled by d * s
 * in fp32.  P * V runs in fp32.  An empty context gives 0.
 *
 * Cell row j of sequence b (n_kv_heads * head_dim values, or n_kv_heads *
 * head_dim/32 q8_0 blocks):
 *     j <  N: k_vram + (b * vram_seq_stride_rows + j)     * row_bytes
 *     j >= N: k_host + (b * host_seq_stride_rows + j - N) * row_bytes
 * (the same for V).  k_vram/v_vram may be NULL when N == 0.
 * k_host == v_host == NULL with N > 0: one range per plane, as a VMM tier
 *   (kvo_vmm_tier_create) holds it -- the tail continues right after the
 *   VRAM cells: k_host = k_vram + N * row_bytes, host_seq_stride_rows =
 *   vram_seq_stride_rows.
 * Memory kinds are taken per range: a range that is device memory
 *   throughout is read with cp.async; anything else (pinned host memory, the
 *   host tail of a VMM tier, a range crossing from a tier's VRAM head into its
 *   tail) with plain 16-byte loads.
 * q: device [batch][n_q_heads][head_dim] of q_dtype: the cache's 16-bit
 *   type for an F16 or BF16 cache, F16 for a Q8_0 cache (other pairs return
 *   KVO_ERR_UNSUPPORTED).
 * kv_dtype: F16, BF16 or Q8_0.  head_dim: 64 or 128.  Group size
 *   n_q_heads / n_kv_heads: 1..8.  n_kv_heads <= 8.  row_bytes and every
 *   base pointer 16-byte aligned.
 * ctx_len: device int32 [batch], each in [0, max_ctx].
 * staging_k / staging_v: NULL = the kernel reads host cells directly
 *   (SM loads through the device mapping).  Otherwise VRAM buffers of
 *   batch * (max_ctx - N) rows each: the host rows [N, max_ctx) are copied
 *   there by the copy engine, and the kernel reads that all-VRAM view.  The
 *   copy runs on a library stream (ordered after the work already on
 *   `stream`, and `stream` waits for it before the call's last kernel), in
 *   up to four parts cut at split boundaries when the decode spans more than
 *   one wave of CTAs; each part's splits are decoded while the next part is
 *   in flight.  The results are bit-identical to the direct read and to an
 *   all-VRAM cache.  Staged calls from several host threads are serialised
 *   inside the library while they enqueue.
 * out: device fp32 [batch][n_q_heads][head_dim].
 * workspace: device, at least kvo_attn_decode_workspace_bytes(...) bytes,
 *   16-byte aligned (split partials).
 * Errors: KVO_ERR_ARG, KVO_ERR_ALIGN, KVO_ERR_NOT_MAPPED,
 *   KVO_ERR_UNSUPPORTED, KVO_ERR_WORKSPACE, KVO_ERR_CUDA.
 * ---------------------------------------------------------------------- */
size_t kvo_attn_decode_workspace_bytes(int64_t batch, int64_t n_q_heads,
                                       int64_t head_dim, int64_t max_ctx);

/* kvo_attn_decode_launches -- how many kernels one kvo_attn_decode_tiered
 * call with these sizes launches on its stream (0 for batch 0, a negative
 * kvo_status for a negative size).  Direct: 2 (split, combine).  Staged with
 * host rows: the split kernel runs once per copy part (plus once for the
 * chunks wholly in VRAM when it overlaps the copy), then the combine: 2 to
 * 6.  Depends on the current device's SM count.  Host function. */
int kvo_attn_decode_launches(int64_t batch, int64_t max_ctx, int64_t head_dim,
                             int64_t n_vram_cells, int staged);

int kvo_attn_decode_tiered(const void *q, int q_dtype, int64_t batch,
                           int64_t n_q_heads, int64_t n_kv_heads,
                           int64_t head_dim, const void *k_vram,
                           const void *v_vram, int64_t vram_seq_stride_rows,
                           const void *k_host, const void *v_host,
                           int64_t host_seq_stride_rows, int kv_dtype,
                           const int32_t *ctx_len, int64_t max_ctx,
                           int64_t n_vram_cells, float scale, void *staging_k,
                           void *staging_v, float *out, void *workspace,
                           size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * kvo_attn_decode_tiered_noalloc -- the same decode with no workspace
 * argument.  The source pages have no counterpart: this entry point exists
 * for callers that cannot give the library a device buffer, for example a
 * serving loop whose device memory was reserved up front by a framework's
 * caching allocator (a separate cudaMalloc there can fail, fragment the
 * pool or synchronise the device), or a plain C host without a device
 * allocator of its own.
 *
 * Arguments, layouts and errors are those of kvo_attn_decode_tiered, minus
 * workspace / workspace_bytes.  The split partials live in one file-scope
 * device array of KVO_NOALLOC_SCRATCH_BYTES (8 MiB) that every GPU loading
 * the library holds until the process exits; the call itself allocates
 * nothing (no cudaMalloc, no cudaFree).  The split length is the regular
 * one when its partials fit; otherwise the context is cut into the fewest
 * splits the array holds (KVO_NOALLOC_SCRATCH_BYTES / (batch * n_q_heads *
 * (head_dim + 2) * 4) of them), each a whole number of 32-cell tiles, so
 * results agree with kvo_attn_decode_tiered within the decode tolerance
 * (not bit for bit when the lengths differ).  Staged and direct calls with
 * the same sizes use the same splits and give the same bits.
 *   - batch * n_q_heads * (head_dim + 2) * 4 > KVO_NOALLOC_SCRATCH_BYTES
 *     returns KVO_ERR_WORKSPACE.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current, under a lock); make
 *     that first call before any stream capture.  The address is kept for
 *     the life of the process: after a cudaDeviceReset of a device the
 *     entry point must not be called on it again.
 *   - The first staged call on a device whose work spans more than one wave
 *     of CTAs creates the library's copy stream and events (no device
 *     memory); make it, too, before any stream capture.
 *   - Every call shares the array and leaves its partials there.  Calls
 *     whose GPU work overlaps (two streams, or two host threads) race on it;
 *     order them on one stream or serialise them.  No part of the array needs
 *     clearing: each call writes every partial before reading it.
 * ---------------------------------------------------------------------- */
#define KVO_NOALLOC_SCRATCH_BYTES (8 << 20)

int kvo_attn_decode_tiered_noalloc(const void *q, int q_dtype, int64_t batch,
                                   int64_t n_q_heads, int64_t n_kv_heads,
                                   int64_t head_dim, const void *k_vram,
                                   const void *v_vram,
                                   int64_t vram_seq_stride_rows,
                                   const void *k_host, const void *v_host,
                                   int64_t host_seq_stride_rows, int kv_dtype,
                                   const int32_t *ctx_len, int64_t max_ctx,
                                   int64_t n_vram_cells, float scale,
                                   void *staging_k, void *staging_v,
                                   float *out, void *stream);

/* ------------------------------------------------------------------------
 * kvo_vmm_tier_create -- one device virtual range holding a VRAM head of
 * head_bytes, then a host-memory tail of tail_bytes, and optionally a second
 * range (the all-VRAM alias) that maps the same head pages followed by a
 * VRAM staging buffer of stage_bytes.
 *
 * llama.cpp PR #319 "tiered KV cache (--kv-vram-cells): VRAM head,
 * pinned-host tail in one VMM range", the tier buffer and its review: the
 * tail is cuMemCreate memory on the host NUMA node the device reports
 * (CU_DEVICE_ATTRIBUTE_HOST_NUMA_ID; node 0 where the host has no NUMA),
 * mapped after the head with device read/write access.  A KV plane of L
 * cells of row_bytes keeps cells [0, N) in VRAM and [N, L) in host memory
 * when head_bytes = N * row_bytes; the decode and prefill entry points then
 * take k_vram = base and k_host = NULL (one base pointer).  Staging through
 * the alias: staging_k = alias + N * row_bytes holds cells [N, ...) so that
 * the alias reads as an all-VRAM plane; this needs N * row_bytes ==
 * head_mapped.
 *
 * Each size is rounded up to kvo_vmm_granularity(device) and returned in
 * *head_mapped, *tail_mapped, *stage_mapped (any may be NULL).  *base and
 * *alias (NULL when stage_bytes == 0) are device addresses, *tier the handle
 * for kvo_vmm_tier_destroy.  The host tail is reachable from the device
 * only: fill it with copies (cudaMemcpy, kvo_swap_blocks_batch, the append
 * path).  The library knows every live tier's ranges and reads the host part
 * with plain loads only (never cp.async or TMA).  The caller's current
 * device is left as it was.
 * Errors: KVO_ERR_ARG (NULL base/tier, an empty head or tail, stage_bytes
 *   without alias, no such device), KVO_ERR_UNSUPPORTED (the driver lacks
 *   the virtual-memory calls, or refuses them), KVO_ERR_CUDA (allocation or
 *   mapping failed; nothing is left allocated).  Callers that want the
 *   page's fallback allocate plain device memory on an error.
 * ---------------------------------------------------------------------- */
int kvo_vmm_granularity(int device, size_t *bytes);

int kvo_vmm_tier_create(int device, size_t head_bytes, size_t tail_bytes,
                        size_t stage_bytes, void **base, void **alias,
                        size_t *head_mapped, size_t *tail_mapped,
                        size_t *stage_mapped, void **tier);

/* kvo_vmm_tier_destroy -- waits for the tier's device to go idle, then
 * unmaps and frees every range of the tier.  NULL is a no-op. */
int kvo_vmm_tier_destroy(void *tier);

/* ------------------------------------------------------------------------
 * kvo_staging_worthwhile -- the staged/direct rule of the sparse rows.
 *
 * ExLlamaV3 patch "QSA KV cache host-RAM offload", qsa_staging_worthwhile:
 * the direct gather reads rows * k_pad cache positions (every row its own
 * selection, re-reading shared pages), staging reads num_pages_used *
 * page_size positions once.  Returns 1 when rows * k_pad > 2 *
 * num_pages_used * page_size, else 0 (also for a negative size).  Pure host
 * function.
 * ---------------------------------------------------------------------- */
int kvo_staging_worthwhile(int64_t rows, int64_t k_pad, int64_t num_pages_used,
                           int64_t page_size);

/* ------------------------------------------------------------------------
 * kvo_dense_staging_worthwhile -- the staged/direct rule of the dense calls
 * (kvo_attn_decode_tiered with staging_k/v, kvo_attn_prefill_tiered with an
 * arena), the measured counterpart of kvo_staging_worthwhile.
 *
 * llama.cpp PR #319 "tiered KV cache (--kv-vram-cells)" stages the used host
 * rows through VRAM by DMA because SM reads of host memory were slow on its
 * PCIe GPUs; on GB300 the SM kernels read the host tail at the full link
 * rate, so the choice is measured (staged vs direct, GB300, over host tails
 * of 1,024 - 176,128 cells and VRAM heads of 8,192 - 94,208 cells for the
 * q8_0 decode of 48 q / 8 kv heads x 128, and over 1 - 2,048 query rows for
 * the bf16 prefill of 32 q / 8 kv heads x 128 with a 32 MiB arena):
 *   prefill != 0: staging wins at every measured row count (8.7 against
 *     12.9 ms at 1 row, 5.5 against 25.9 ms at 256 rows, 9.5 against 126 ms
 *     at 2,048 rows): the direct kernels read the tail once per query tile of
 *     each kv head, on few CTAs at small row counts.
 *     Returns 1 whenever n_tail_cells > 0.
 *   prefill == 0 (decode, one query row per sequence): direct wins unless the
 *     VRAM head is long enough to hide the copy of the tail: staging pays off
 *     (by up to 21 %) when n_vram_cells >= 65,536 and 5 * n_tail_cells <=
 *     n_vram_cells -- the copy then runs while the VRAM cells are decoded.
 *     Elsewhere direct is faster by up to 20 %, or within a few per cent.
 *     Against the measured table the rule's choice is never more than 7 %
 *     slower than the faster mode.
 * Returns 0 for n_tail_cells <= 0 and for negative sizes.  Pure host
 * function.
 * ---------------------------------------------------------------------- */
int kvo_dense_staging_worthwhile(int prefill, int64_t n_vram_cells, int64_t n_tail_cells);

/* ------------------------------------------------------------------------
 * kvo_attn_sparse_rows -- QSA sparse attention of query rows over a paged,
 * host-resident K/V cache, direct or staged through a VRAM arena.
 *
 * ExLlamaV3 patch "QSA KV cache host-RAM offload": qsa_sparse_attend_rows
 * (direct) and qsa_sparse_attend_rows_staged.  Row r (q [rows][n_q_heads]
 * [head_dim] of q_dtype == dtype) attends to the cache positions
 * indices[r][0 .. k_pad) that are >= 0 and < num_pages_used * page_size
 * (anything else is padding).  Position p is slot p % page_size of page
 * block_table[p / page_size] of the planes k_pages / v_pages
 * ([n_pages][page_size][n_kv_heads][head_dim], F16 or BF16); q head h reads
 * kv head h / (n_q_heads / n_kv_heads):
 *     out[r][h] = sum_p softmax_p(scale * q[r][h] . k_p) v_p
 * (a position listed twice counts twice; a row with no selection gives 0).
 *   arena == NULL (or num_pages_used == 0): direct -- every row reads its
 *     picks through the host mapping, rows_per_launch rows per launch.
 *   arena != NULL: staged -- the pages in use are walked in buckets; each
 *     bucket is gathered into an arena slot (its K pages, then its V pages),
 *     every row block is scored against it, and its partial (m, l, acc) is
 *     folded into a running state; after the last bucket
 *     out = acc / max(l, 1e-30).  With page_bytes = page_size * n_kv_heads *
 *     head_dim * 2, the arena holds two slots of arena_bytes / (4 *
 *     page_bytes) pages when that is >= 1 (the next bucket is gathered on a
 *     library stream while the current one is scored), else one slot of
 *     arena_bytes / (2 * page_bytes) pages; a bucket never exceeds
 *     num_pages_used pages.  At least 2 pages must fit (KVO_ERR_ARG
 *     otherwise).
 *   Staged and direct agree within the attention tolerance, not bit for bit.
 * q, out (fp32 [rows][n_q_heads][head_dim]), workspace, arena: device
 *   memory, 16-byte aligned.  indices (int32 [rows][k_pad]) and block_table
 *   (int32 [num_pages_used]): device-accessible.  k_pages / v_pages: pinned
 *   mapped host (or device) memory, 16-byte aligned.
 * head_dim 64 or 128; group 1..8; n_kv_heads <= 8.
 * A block_table entry outside [0, n_pages) is skipped (its picks count as
 *   padding) and sets bit 1 of kvo_device_errors().
 * Staged mode first groups every row's picks by bucket (order kept within a
 *   bucket, padding dropped) so that each bucket scores only its own picks;
 *   at most 51,199 buckets.
 * workspace: at least kvo_attn_sparse_rows_workspace_bytes(rows, n_q_heads,
 *   n_kv_heads, head_dim, k_pad, rows_per_launch, page_size, num_pages_used,
 *   arena_bytes) bytes (the same arguments as the call).
 * Errors: KVO_ERR_ARG, KVO_ERR_ALIGN, KVO_ERR_NOT_MAPPED,
 *   KVO_ERR_UNSUPPORTED, KVO_ERR_WORKSPACE, KVO_ERR_CUDA.
 * ---------------------------------------------------------------------- */
size_t kvo_attn_sparse_rows_workspace_bytes(int64_t rows, int64_t n_q_heads,
                                            int64_t n_kv_heads, int64_t head_dim,
                                            int64_t k_pad,
                                            int64_t rows_per_launch,
                                            int64_t page_size,
                                            int64_t num_pages_used,
                                            size_t arena_bytes);

int kvo_attn_sparse_rows(const void *q, int q_dtype, int64_t rows,
                         int64_t n_q_heads, int64_t n_kv_heads,
                         int64_t head_dim, const void *k_pages,
                         const void *v_pages, int dtype, int64_t page_size,
                         int64_t n_pages, const int32_t *block_table,
                         int64_t num_pages_used, const int32_t *indices,
                         int64_t k_pad, float scale, void *arena,
                         size_t arena_bytes, int64_t rows_per_launch,
                         float *out, void *workspace, size_t workspace_bytes,
                         void *stream);

/* ------------------------------------------------------------------------
 * kvo_copy_pages_host -- copy one page's first tokens between host planes.
 *
 * ExLlamaV3 patch "QSA KV cache host-RAM offload", copy_page: host-resident
 * pages are copied by the CPU, not by a device kernel reading and writing
 * across the host link.  The call first drains `stream` (queued GPU work may
 * still read or write the pages), then copies num_tokens * token_bytes bytes
 * from page from_page to page to_page (pages of page_tokens * token_bytes
 * bytes) for K (src_k -> dst_k) and V (src_v -> dst_v); overlapping ranges
 * are allowed.  Synchronous; the planes must be host memory (pinned or not).
 * Errors: KVO_ERR_ARG (num_tokens > page_tokens, negative sizes, NULL),
 *   KVO_ERR_NOT_MAPPED (a device pointer, or a plane inside a VMM tier,
 *   which the CPU cannot address), KVO_ERR_CUDA (the drain).
 * ---------------------------------------------------------------------- */
int kvo_copy_pages_host(const void *src_k, const void *src_v, void *dst_k,
                        void *dst_v, int64_t page_tokens, int64_t token_bytes,
                        int64_t from_page, int64_t to_page, int64_t num_tokens,
                        void *stream);

/* ------------------------------------------------------------------------
 * kvo_append_kv_tiered -- write path: new tokens into a tiered cache.
 *
 * ExLlamaV3 qsa-kv-offload patch (the paged cache update that writes new
 * tokens' K/V into the host-resident planes) and llama.cpp PR "tiered KV
 * cache": token t < n_new of k_new / v_new becomes cell pos0 + t of one
 * sequence, stored in the tier that holds it -- VRAM head row j for j < N,
 * pinned host tail row j - N for j >= N -- in the cache dtype.
 *   kv_dtype == src_dtype (F16 or BF16): the rows are copied.
 *   kv_dtype == Q8_0: each 32-value block of each head is quantised in
 *     fp32: amax = max|x|, d = amax / 127, q = round-half-away-from-zero(
 *     x * (1/d)) (0 when d == 0), stored as {fp16 d (round to nearest
 *     even); int8 q[32]}.  The pages name the q8_0 format, not its rounding:
 *     this rule is the library's stated reading.  q8_0 rows hold at most
 *     2048 values (n_kv_heads * head_dim).
 *
 * k_new, v_new: device-accessible [n_new][n_kv_heads][head_dim] of src_dtype
 *   (F16 or BF16), 16-byte aligned.
 * k_vram, v_vram: the head, min(N, capacity_cells) rows; k_host, v_host:
 *   the tail, capacity_cells - N rows (either may be NULL if never touched).
 *   Rows of n_kv_heads * head_dim values or n_kv_heads * head_dim/32 q8_0
 *   blocks; f16/bf16 tiers 16-byte aligned, q8_0 tiers 2-byte aligned.
 * Errors: KVO_ERR_ARG (cells past capacity_cells, bad sizes),
 *   KVO_ERR_UNSUPPORTED (dtype pair), KVO_ERR_ALIGN, KVO_ERR_NOT_MAPPED,
 *   KVO_ERR_CUDA.
 * ---------------------------------------------------------------------- */
int kvo_append_kv_tiered(const void *k_new, const void *v_new, int src_dtype,
                         int64_t n_new, int64_t pos0, int64_t n_kv_heads,
                         int64_t head_dim, void *k_vram, void *v_vram,
                         void *k_host, void *v_host, int kv_dtype,
                         int64_t n_vram_cells, int64_t capacity_cells,
                         void *stream);

/* ------------------------------------------------------------------------
 * kvo_attn_prefill_tiered -- causal chunked-prefill GQA attention over a
 * tiered cache (one sequence).
 *
 * Query row i (0 <= i < rows) sits at position q_pos0 + i and attends the
 * cells j <= q_pos0 + i, j < ctx_len:
 *     out[i][h] = sum_j softmax_j(scale * q[i][h] . k[j][g]) v[j][g],
 *     g = h / (n_q_heads / n_kv_heads).
 * Cells [0, N) are read from k_vram/v_vram, cells [N, ctx_len) from
 * k_host/v_host (row j - N), rows of n_kv_heads * head_dim values.
 * k_host == v_host == NULL: one range per plane (a VMM tier), the tail at
 * k_vram + N * row_bytes.
 *
 * Staged mode (arena != NULL; ExLlamaV3 qsa-kv-offload patch,
 * qsa_sparse_attend_rows_staged): the host tail is walked in buckets.  The
 * arena is used as two slots of arena_bytes / (4 * row_bytes) cells of K and
 * of V (one slot of arena_bytes / (2 * row_bytes) cells if a slot would hold
 * no row); each bucket is copied host -> slot once by the copy engine on a
 * library-owned side stream (created on first use, joined back into
 * `stream` before the call's work ends), so the next bucket's copy overlaps
 * the current bucket's scoring.  Every query row is scored against a bucket
 * in launches of rows_per_launch rows, and each launch folds its partial
 * (m, l, acc) into the running softmax
 *     m' = max(m, m_b), acc = e^(m-m') acc + e^(m_b-m') acc_b,
 *     l = e^(m-m') l + e^(m_b-m') l_b
 * (a bucket a row cannot see contributes nothing); the end result is
 * acc / max(l, 1e-30).  Each host byte crosses the link once per call.
 * Direct mode (arena == NULL): the kernel reads the tail from host memory
 * for every query tile.
 *
 * Precision: scores and sums in fp32; the softmax weights enter the PV
 *   product as fp16 (11 significant bits), and so do the V values of a bf16
 *   cache (converted on chip: exact for magnitudes in [2^-14, 65504], to
 *   within 2^-25 below that; larger values set bit 4 of kvo_device_errors()).
 * q: device [rows][n_q_heads][head_dim], dtype = kv_dtype (F16 or BF16:
 *   the tensor-core tiles take one operand type).  head_dim: 128.  Group
 *   size: 1, 2, 4 or 8.  Rows and base pointers 16-byte aligned.
 * arena: device, >= 2 cell rows of K and of V, 16-byte aligned.
 * out: device fp32 [rows][n_q_heads][head_dim]; also used as the running
 *   accumulator between launches.
 * workspace: device, kvo_attn_prefill_workspace_bytes(rows, n_q_heads)
 *   bytes (running m and l).
 * Errors: KVO_ERR_ARG, KVO_ERR_ALIGN, KVO_ERR_NOT_MAPPED,
 *   KVO_ERR_UNSUPPORTED, KVO_ERR_WORKSPACE, KVO_ERR_CUDA.
 * ---------------------------------------------------------------------- */
size_t kvo_attn_prefill_workspace_bytes(int64_t rows, int64_t n_q_heads);

int kvo_attn_prefill_tiered(const void *q, int64_t rows, int64_t q_pos0,
                            int64_t n_q_heads, int64_t n_kv_heads,
                            int64_t head_dim, const void *k_vram,
                            const void *v_vram, const void *k_host,
                            const void *v_host, int kv_dtype, int64_t ctx_len,
                            int64_t n_vram_cells, float scale, void *arena,
                            size_t arena_bytes, int64_t rows_per_launch,
                            float *out, void *workspace,
                            size_t workspace_bytes, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* KVO_H */
