// Internal helpers shared by the libkvo translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <stddef.h>

#include "../../include/kvo.h"

namespace kvo {

// Record a one-line reason for the failing call (thread-local) and return st.
int fail(int st, const char *fmt, ...);
// Clear the thread-local reason at the start of an entry point.
void clear_error();
// Map a CUDA error to KVO_ERR_CUDA with its text; KVO_OK for cudaSuccess.
int cuda_status(cudaError_t e, const char *what);

enum Access { kDeviceMem = 1, kMappedHost = 2 };
// Classify [p, p + bytes): returns kDeviceMem, kMappedHost or 0 (not
// device-accessible: unregistered pageable memory, NULL, or a range with a
// byte in no allocation).  The range is walked allocation by allocation, so a
// gap between two allocations is found; a range over allocations of both
// kinds counts as kMappedHost (device-accessible, not all device memory).
int classify(const void *p, size_t bytes);
// 1: p lies in the host-backed tail of a live VMM tier; 0: in a tier's VRAM
// range; -1: in no tier.  *range_end (if given) receives the end of the
// tier range holding p.
int vmm_host_backed(const void *p, uintptr_t *range_end = nullptr);
// [*lo, *hi): the allocation (or reserved range) holding p, from the driver's
// pointer attributes; false when the driver cannot say.
bool alloc_range(const void *p, uintptr_t *lo, uintptr_t *hi);

int num_sms();                       // SMs of the current device (cached)

// Library streams for staged work: a side stream that fills one arena slot
// while the caller's stream scores the other, and a second launch stream so
// that two row blocks run concurrently.  One set per user (0: prefill,
// 1: sparse rows, 2: staged decode) and device, created on first use; every use forks from and
// joins back into the caller's stream, under the user's own mutex.
struct Ring {
  cudaStream_t side = nullptr, comp2 = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr, join2 = nullptr;
  cudaEvent_t ready[2] = {nullptr, nullptr}, freed[2] = {nullptr, nullptr}, done2[2] = {nullptr, nullptr};
  cudaEvent_t part[4] = {nullptr, nullptr, nullptr, nullptr};
};
Ring *ring(int which);               // nullptr when the streams cannot be created (which: 0..2)
inline bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Device-side error bits set by kernels that skipped an out-of-range item.
enum DeviceErrorBits : uint32_t {
  kErrGatherSel = 1u,     // a gather selection outside its plane (skipped)
  kErrPageTable = 2u,     // a page-table entry outside the planes (skipped)
  kErrWaitTimeout = 4u,   // a bounded barrier wait gave up (the kernel wound down)
  kErrSmemAlign = 8u,     // a CTA could not align its shared memory and exited
  kErrF16Range = 16u      // a bf16 V value outside fp16's range met the fp16 PV product
};
uint32_t *device_error_word();       // address of the per-device word (nullptr on failure)

// Launchers implemented in the kernel translation units.  They assume the
// entry point already validated every argument.
// max_size: the largest descriptor size when the host knows it (a short
// batch whose sizes it read), else -1.
cudaError_t launch_swap_sm(const int64_t *src, const int64_t *dst, const int64_t *sizes, int64_t n,
                           int64_t max_size, cudaStream_t st);

cudaError_t launch_gather(const void *k_plane, const void *v_plane, int64_t n_seq,
                          int64_t seq_stride_tokens, int64_t n_kv_heads, int64_t head_bytes,
                          int64_t block_tokens, const int32_t *sel, int64_t n_sel,
                          void *k_out, void *v_out, uint32_t *err, cudaStream_t st);

struct DecodeArgs {
  const void *q; int q_dtype;
  int batch, n_q_heads, n_kv_heads, head_dim, group;
  const uint8_t *k_lo, *v_lo;  int64_t lo_seq_stride_rows;   // cells [0, N)
  const uint8_t *k_hi, *v_hi;  int64_t hi_seq_stride_rows;   // cells [N, L), row j - N
  int hi_device;               // k_hi / v_hi are device memory (staging, or a device tail)
  int kv_dtype; int64_t row_bytes;
  const int32_t *ctx_len; int64_t max_ctx, n_vram;
  float scale_log2;            // scale * log2(e)
  float *out;
  float *part_acc, *part_ml;   // workspace: [B][splits][Hq][D], [B][splits][Hq][2]
  int split_cells, n_splits;
  // Items this launch computes: [item_lo, item_hi) (item_hi < 0: all).
  // phase 0: split kernel then combine; 1: split kernel only; 2: combine only.
  int64_t item_lo = 0, item_hi = -1;
  int phase = 0;
  // Deal the chunks in the order 0, n-1, 1, n-2, ... instead of 0, 1, 2, ...
  // (a direct call with host rows): the first wave then mixes VRAM chunks and
  // host chunks, so the host link is busy while the VRAM chunks are decoded.
  // Which CTA computes a chunk changes none of its bits.
  int interleave = 0;
  // Running softmax state folded by the combine kernel (null: plain decode,
  // out = the normalised result).  init: this launch starts the state;
  // finalize: this launch writes out = acc / max(l, 1e-30).
  float *run_acc = nullptr, *run_ml = nullptr;   // [B][Hq][D], [B][Hq][2]
  int init = 1, finalize = 1;
  // Sparse rows (QSA): cell k of work row b is cache position
  // indices[b * max_ctx + k]; positions outside [win_lo, win_hi) are padding.
  // staged: position j is row j - win_lo of k_lo / v_lo (the arena); else row
  // block_table[j / page_size] * page_size + j % page_size of k_hi / v_hi.
  const int32_t *indices = nullptr;              // null for the decode
  // Staged mode: row b's picks of this bucket are indices[b * max_ctx +
  // offs[b * offs_stride + bucket] ...] up to offs[... + bucket + 1].
  const int32_t *offs = nullptr;
  int64_t offs_stride = 0, bucket = 0;
  int64_t win_lo = 0, win_hi = 0;
  const int32_t *block_table = nullptr;
  int64_t page_size = 1, n_pages_total = 0;
  int sparse_staged = 0;
  // Every row the launch reads is device-resident: the split kernel runs one
  // continuous copy ring over all of a CTA's items.
  int all_ring = 0;
  // At most this many CTAs for the split kernel (0: one per SM), leaving SMs
  // free for a kernel that runs beside it on another stream.
  int grid_cap = 0;
  // Selection mode with one chunk per row and a running state: the split
  // kernel folds each row's chunk into run_acc / run_ml itself (no combine).
  int fold_in_split = 0;
  int pre_rows = 0;             // set by the launcher: rows' query / running state prefetched
  uint32_t *err = nullptr;     // device error word (sparse: bad page-table entries)
};
// Split geometry for a decode: fixed cell ranges that depend on max_ctx and
// batch only (never on N or on staging), so tiered and all-VRAM runs match.
void decode_geometry(int64_t batch, int64_t max_ctx, int64_t head_dim, int *split_cells,
                     int *n_splits);
size_t decode_workspace_bytes(int64_t batch, int64_t n_q_heads, int64_t head_dim,
                              int64_t max_ctx);
int launch_decode(const DecodeArgs &a, cudaStream_t st);   // kvo_status
// Staged decode schedule: chunks [0, c_v) are decoded while the copy runs,
// then copy part p covers chunks [ch_lo[p], ch_hi[p]) (cut at chunk
// boundaries, the host rows among them).
struct StagedPlan {
  int64_t c_v = 0;
  int parts = 1;
  int64_t ch_lo[4] = {0, 0, 0, 0}, ch_hi[4] = {0, 0, 0, 0};
};
StagedPlan staged_plan(int64_t batch, int split_cells, int n_splits, int64_t n_vram);
// Staged decode: the host rows [a.n_vram, a.max_ctx) of every sequence
// (k_host / v_host, host_stride rows apart) are copied to staging_k /
// staging_v ([batch][max_ctx - n_vram] rows) on a library stream in parts cut
// at chunk boundaries; each part's chunks are decoded once it has landed, the
// combine runs last.  Takes a's all-VRAM view fields from the arguments.
int launch_decode_staged(DecodeArgs a, const void *k_host, const void *v_host, int64_t host_stride,
                         void *staging_k, void *staging_v, cudaStream_t st);   // kvo_status
// Sparse rows: the split kernel in selection mode (fp16 / bf16 caches), then
// the combine (with the running-state fold when a.run_acc is set).
int launch_sparse_rows(const DecodeArgs &a, cudaStream_t st);   // kvo_status
// Copy pages block_table[p0 .. p0 + n) of the K and V planes (page_bytes each)
// to arena slots 0 .. n-1; entries outside [0, n_pages_total) are skipped and
// set kErrPageTable.  beside: the copy runs beside a split kernel that
// leaves it a few SMs (one wide CTA per SM); else up to four CTAs per SM.
cudaError_t launch_page_gather(const void *k_pages, const void *v_pages, int64_t page_bytes,
                               const int32_t *block_table, int64_t p0, int64_t n,
                               int64_t n_pages_total, void *k_arena, void *v_arena, uint32_t *err,
                               bool beside, cudaStream_t st);

struct PrefillArgs {
  const uint16_t *q;           // [rows][Hq][D] (rows of this launch start at q)
  int rows;                    // rows in this launch
  int64_t pos0;                // position of the first row of this launch
  int n_q_heads, n_kv_heads, head_dim, group, dtype;
  int64_t row_bytes;
  const uint8_t *k_lo, *v_lo;  // cells < N: k_lo + j * row_bytes
  const uint8_t *k_hi, *v_hi;  // cells >= N: k_hi + (j - hi_origin) * row_bytes
  int64_t hi_origin, n_vram;
  int64_t c0, c1;              // cell range of this launch
  float scale_log2;
  float *acc;                  // [rows][Hq][D] running accumulator / output
  float *ml;                   // [rows][Hq][2] running (m, l) in log2 units
  int init, finalize;
};
int launch_prefill(const PrefillArgs &a, cudaStream_t st);  // kvo_status (mma.sync, any memory)
// tcgen05 + TMA path for a device-resident segment: cells [a.c0, a.c1) are
// rows (c - a.hi_origin) of k_seg / v_seg (seg_rows rows).
int launch_prefill_tc(const PrefillArgs &a, const void *k_seg, const void *v_seg, int64_t seg_rows,
                      cudaStream_t st);
// tcgen05 path for a host-memory segment (rows (c - a.hi_origin) of a.k_hi /
// a.v_hi), filled with plain loads.
int launch_prefill_tc_host(const PrefillArgs &a, cudaStream_t st);

struct AppendArgs {
  const uint8_t *k_new, *v_new;  // [n_new][n_kv_heads][head_dim] of src_dtype
  int src_dtype, kv_dtype;
  int64_t n_new, pos0, n_kv_heads, head_dim, row_bytes;   // row_bytes: cache row
  uint8_t *k_lo, *v_lo;          // cells < n_vram: row j
  uint8_t *k_hi, *v_hi;          // cells >= n_vram: row j - n_vram
  int64_t n_vram;
};
int launch_append(const AppendArgs &a, cudaStream_t st);   // kvo_status

}  // namespace kvo
