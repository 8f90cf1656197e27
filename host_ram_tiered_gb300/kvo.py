"""Thin ctypes binding of libkvo (include/kvo.h), same names as the C ABI.

Argument marshalling only: every step of the path runs in the library's
CUDA kernels.  Buffers may be passed as torch tensors (their data pointer is
used) or as integer addresses; streams as ``torch.cuda.Stream`` or a raw
handle.  A non-zero status raises :class:`KvoError`.  If the library has
not been built, loading it raises: there is no Python or CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

F16, BF16, Q8_0 = 0, 1, 2
KVO_SWAP_H2D = 0x1
KVO_SWAP_D2H = 0x2
KVO_SWAP_SRC_ORDER_ANY = 0x4
KVO_SWAP_FORCE_SM = 0x8
KVO_SWAP_FORCE_CE = 0x10
KVO_SWAP_SHORT_BATCH = 64
KVO_NOALLOC_SCRATCH_BYTES = 8 << 20

STATUS = {0: "KVO_OK", -1: "KVO_ERR_ARG", -2: "KVO_ERR_ALIGN", -3: "KVO_ERR_NOT_MAPPED",
          -4: "KVO_ERR_UNSUPPORTED", -5: "KVO_ERR_CUDA", -6: "KVO_ERR_WORKSPACE"}

# Every symbol include/kvo.h declares, with (restype, argtypes).
_i64, _u64, _vp, _u32, _int, _f32, _sz = (ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p,
                                          ctypes.c_uint32, ctypes.c_int, ctypes.c_float,
                                          ctypes.c_size_t)
SIGNATURES = {
    "kvo_status_string": (ctypes.c_char_p, [_int]),
    "kvo_last_error": (ctypes.c_char_p, []),
    "kvo_device_errors": (_int, [_vp, _int]),
    "kvo_selftest_wait_timeout": (_int, [_u64, _vp]),
    "kvo_sub_block_ptrs": (_int, [_vp, _i64, _i64, _i64, _u64, _i64, _i64, _vp, _i64]),
    "kvo_shard_range": (_int, [_i64, _i64, _i64, _vp, _vp]),
    "kvo_copy_plan": (_int, [_vp] * 6 + [_i64, _int, _vp, _vp, _vp, _i64, _vp]),
    "kvo_fragment_ptrs": (_int, [_vp, _vp, _i64, _vp, _vp, _vp, _i64, _vp, _vp, _vp]),
    "kvo_swap_blocks_batch": (_int, [_vp, _vp, _vp, _i64, _u32, _vp]),
    "kvo_gather_blocks": (_int, [_vp, _vp, _i64, _i64, _i64, _i64, _int, _i64, _vp, _i64, _vp,
                                 _vp, _vp]),
    "kvo_attn_decode_workspace_bytes": (_sz, [_i64, _i64, _i64, _i64]),
    "kvo_attn_decode_launches": (_int, [_i64, _i64, _i64, _i64, _int]),
    "kvo_vmm_granularity": (_int, [_int, _vp]),
    "kvo_vmm_tier_create": (_int, [_int, _sz, _sz, _sz, _vp, _vp, _vp, _vp, _vp, _vp]),
    "kvo_vmm_tier_destroy": (_int, [_vp]),
    "kvo_attn_decode_tiered": (_int, [_vp, _int, _i64, _i64, _i64, _i64, _vp, _vp, _i64, _vp, _vp,
                                      _i64, _int, _vp, _i64, _i64, _f32, _vp, _vp, _vp, _vp, _sz,
                                      _vp]),
    "kvo_attn_decode_tiered_noalloc": (_int, [_vp, _int, _i64, _i64, _i64, _i64, _vp, _vp, _i64, _vp,
                                              _vp, _i64, _int, _vp, _i64, _i64, _f32, _vp, _vp, _vp,
                                              _vp]),
    "kvo_append_kv_tiered": (_int, [_vp, _vp, _int, _i64, _i64, _i64, _i64, _vp, _vp, _vp, _vp,
                                    _int, _i64, _i64, _vp]),
    "kvo_staging_worthwhile": (_int, [_i64, _i64, _i64, _i64]),
    "kvo_dense_staging_worthwhile": (_int, [_int, _i64, _i64]),
    "kvo_attn_sparse_rows_workspace_bytes": (_sz, [_i64] * 8 + [_sz]),
    "kvo_attn_sparse_rows": (_int, [_vp, _int, _i64, _i64, _i64, _i64, _vp, _vp, _int, _i64, _i64,
                                    _vp, _i64, _vp, _i64, _f32, _vp, _sz, _i64, _vp, _vp, _sz, _vp]),
    "kvo_copy_pages_host": (_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _vp]),
    "kvo_attn_prefill_workspace_bytes": (_sz, [_i64, _i64]),
    "kvo_attn_prefill_tiered": (_int, [_vp, _i64, _i64, _i64, _i64, _i64, _vp, _vp, _vp, _vp,
                                       _int, _i64, _i64, _f32, _vp, _sz, _i64, _vp, _vp, _sz,
                                       _vp]),
}


class KvoError(RuntimeError):
    def __init__(self, status: int, func: str, detail: str):
        self.status = status
        super().__init__(f"{func}: {STATUS.get(status, status)}: {detail}")


_lib = None


def lib_path() -> str:
    return _build.LIB_PATH


def load():
    """Load the in-tree libkvo.so (build it first with build.build())."""
    global _lib
    if _lib is None:
        path = lib_path()
        if not os.path.exists(path):
            raise ImportError(f"libkvo.so is not built ({path}); run host_ram_tiered_gb300.build.build()")
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _p(x) -> int | None:
    """Address of a tensor / numpy array / int / None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    return x.data_ptr()


def _s(stream) -> int | None:
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st: int, name: str) -> None:
    if st != 0:
        raise KvoError(st, name, load().kvo_last_error().decode(errors="replace"))


def kvo_status_string(status: int) -> str:
    return load().kvo_status_string(status).decode()


def kvo_last_error() -> str:
    return load().kvo_last_error().decode(errors="replace")


def kvo_device_errors(clear: bool = True) -> int:
    bits = ctypes.c_uint32(0)
    _check(load().kvo_device_errors(ctypes.addressof(bits), int(clear)), "kvo_device_errors")
    return bits.value


def kvo_selftest_wait_timeout(limit_ns, stream=None) -> None:
    _check(load().kvo_selftest_wait_timeout(limit_ns, _s(stream)), "kvo_selftest_wait_timeout")


def kvo_sub_block_ptrs(block_ids, n_ids, blocks_per_chunk, skip_count, base, row_stride_bytes,
                       row_bytes, out, n_out) -> None:
    _check(load().kvo_sub_block_ptrs(_p(block_ids), n_ids, blocks_per_chunk, skip_count, base,
                                     row_stride_bytes, row_bytes, _p(out), n_out),
           "kvo_sub_block_ptrs")


def kvo_shard_range(n_units, world, rank) -> tuple[int, int]:
    """[lo, hi): rank's contiguous share of n_units work units."""
    lo, hi = ctypes.c_int64(0), ctypes.c_int64(0)
    _check(load().kvo_shard_range(n_units, world, rank, ctypes.addressof(lo), ctypes.addressof(hi)),
           "kvo_shard_range")
    return lo.value, hi.value


def kvo_copy_plan(local_offset, local_stride, canonical_offset, canonical_stride, num_fragments,
                  fragment_size, n_runs, gpu_to_cpu, frag_src, frag_dst, frag_sizes, capacity) -> int:
    """Returns the fragment count written to frag_src / frag_dst / frag_sizes."""
    n = ctypes.c_int64(0)
    _check(load().kvo_copy_plan(_p(local_offset), _p(local_stride), _p(canonical_offset),
                                _p(canonical_stride), _p(num_fragments), _p(fragment_size), n_runs,
                                int(gpu_to_cpu), _p(frag_src), _p(frag_dst), _p(frag_sizes), capacity,
                                ctypes.addressof(n)), "kvo_copy_plan")
    return n.value


def kvo_fragment_ptrs(src_bases, dst_bases, n_blocks, frag_src, frag_dst, frag_sizes, n_frags,
                      out_src, out_dst, out_sizes) -> None:
    _check(load().kvo_fragment_ptrs(_p(src_bases), _p(dst_bases), n_blocks, _p(frag_src),
                                    _p(frag_dst), _p(frag_sizes), n_frags, _p(out_src), _p(out_dst),
                                    _p(out_sizes)), "kvo_fragment_ptrs")


def kvo_swap_blocks_batch(src, dst, sizes, n, flags, stream=None) -> None:
    _check(load().kvo_swap_blocks_batch(_p(src), _p(dst), _p(sizes), n, flags, _s(stream)),
           "kvo_swap_blocks_batch")


def kvo_gather_blocks(k_plane, v_plane, n_seq, seq_stride_tokens, n_kv_heads, head_dim, dtype,
                      block_tokens, sel, n_sel, k_out, v_out, stream=None) -> None:
    _check(load().kvo_gather_blocks(_p(k_plane), _p(v_plane), n_seq, seq_stride_tokens, n_kv_heads,
                                    head_dim, dtype, block_tokens, _p(sel), n_sel, _p(k_out),
                                    _p(v_out), _s(stream)), "kvo_gather_blocks")


def kvo_attn_decode_workspace_bytes(batch, n_q_heads, head_dim, max_ctx) -> int:
    return load().kvo_attn_decode_workspace_bytes(batch, n_q_heads, head_dim, max_ctx)


def kvo_attn_decode_launches(batch, max_ctx, head_dim, n_vram_cells, staged) -> int:
    return load().kvo_attn_decode_launches(batch, max_ctx, head_dim, n_vram_cells, int(bool(staged)))


def kvo_vmm_granularity(device) -> int:
    """Granularity of a VMM tier's ranges; raises KvoError when VMM is unavailable."""
    out = ctypes.c_size_t(0)
    _check(load().kvo_vmm_granularity(device, ctypes.byref(out)), "kvo_vmm_granularity")
    return out.value


def kvo_vmm_tier_create(device, head_bytes, tail_bytes, stage_bytes=0):
    """One VA range (VRAM head + host tail) and, with stage_bytes > 0, the
    all-VRAM alias. Returns a dict: base, alias, head, tail, stage (mapped
    sizes) and tier (the handle for kvo_vmm_tier_destroy)."""
    base, alias, tier = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_void_p()
    hm, tm, sm = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(load().kvo_vmm_tier_create(device, head_bytes, tail_bytes, stage_bytes, ctypes.byref(base),
                                      ctypes.byref(alias), ctypes.byref(hm), ctypes.byref(tm), ctypes.byref(sm),
                                      ctypes.byref(tier)), "kvo_vmm_tier_create")
    return {"base": base.value, "alias": alias.value, "head": hm.value, "tail": tm.value, "stage": sm.value,
            "tier": tier.value}


def kvo_vmm_tier_destroy(tier) -> None:
    _check(load().kvo_vmm_tier_destroy(tier), "kvo_vmm_tier_destroy")


def kvo_attn_decode_tiered(q, q_dtype, batch, n_q_heads, n_kv_heads, head_dim, k_vram, v_vram,
                           vram_seq_stride_rows, k_host, v_host, host_seq_stride_rows, kv_dtype,
                           ctx_len, max_ctx, n_vram_cells, scale, staging_k, staging_v, out,
                           workspace, workspace_bytes, stream=None) -> None:
    _check(load().kvo_attn_decode_tiered(
        _p(q), q_dtype, batch, n_q_heads, n_kv_heads, head_dim, _p(k_vram), _p(v_vram),
        vram_seq_stride_rows, _p(k_host), _p(v_host), host_seq_stride_rows, kv_dtype, _p(ctx_len),
        max_ctx, n_vram_cells, scale, _p(staging_k), _p(staging_v), _p(out), _p(workspace),
        workspace_bytes, _s(stream)), "kvo_attn_decode_tiered")


def kvo_attn_decode_tiered_noalloc(q, q_dtype, batch, n_q_heads, n_kv_heads, head_dim, k_vram,
                                   v_vram, vram_seq_stride_rows, k_host, v_host,
                                   host_seq_stride_rows, kv_dtype, ctx_len, max_ctx, n_vram_cells,
                                   scale, staging_k, staging_v, out, stream=None) -> None:
    """kvo_attn_decode_tiered for callers that cannot provide a workspace: the
    partials go to the library's fixed 8 MiB device scratch array."""
    _check(load().kvo_attn_decode_tiered_noalloc(
        _p(q), q_dtype, batch, n_q_heads, n_kv_heads, head_dim, _p(k_vram), _p(v_vram),
        vram_seq_stride_rows, _p(k_host), _p(v_host), host_seq_stride_rows, kv_dtype, _p(ctx_len),
        max_ctx, n_vram_cells, scale, _p(staging_k), _p(staging_v), _p(out), _s(stream)),
        "kvo_attn_decode_tiered_noalloc")


def kvo_append_kv_tiered(k_new, v_new, src_dtype, n_new, pos0, n_kv_heads, head_dim, k_vram,
                         v_vram, k_host, v_host, kv_dtype, n_vram_cells, capacity_cells,
                         stream=None) -> None:
    _check(load().kvo_append_kv_tiered(
        _p(k_new), _p(v_new), src_dtype, n_new, pos0, n_kv_heads, head_dim, _p(k_vram), _p(v_vram),
        _p(k_host), _p(v_host), kv_dtype, n_vram_cells, capacity_cells, _s(stream)),
        "kvo_append_kv_tiered")


def kvo_attn_prefill_workspace_bytes(rows, n_q_heads) -> int:
    return load().kvo_attn_prefill_workspace_bytes(rows, n_q_heads)


def kvo_attn_prefill_tiered(q, rows, q_pos0, n_q_heads, n_kv_heads, head_dim, k_vram, v_vram,
                            k_host, v_host, kv_dtype, ctx_len, n_vram_cells, scale, arena,
                            arena_bytes, rows_per_launch, out, workspace, workspace_bytes,
                            stream=None) -> None:
    _check(load().kvo_attn_prefill_tiered(
        _p(q), rows, q_pos0, n_q_heads, n_kv_heads, head_dim, _p(k_vram), _p(v_vram), _p(k_host),
        _p(v_host), kv_dtype, ctx_len, n_vram_cells, scale, _p(arena), arena_bytes,
        rows_per_launch, _p(out), _p(workspace), workspace_bytes, _s(stream)),
        "kvo_attn_prefill_tiered")


def kvo_dense_staging_worthwhile(prefill, n_vram_cells, n_tail_cells) -> bool:
    return bool(load().kvo_dense_staging_worthwhile(int(prefill), n_vram_cells, n_tail_cells))


def kvo_staging_worthwhile(rows, k_pad, num_pages_used, page_size) -> bool:
    return bool(load().kvo_staging_worthwhile(rows, k_pad, num_pages_used, page_size))


def kvo_attn_sparse_rows_workspace_bytes(rows, n_q_heads, n_kv_heads, head_dim, k_pad, rows_per_launch,
                                         page_size, num_pages_used, arena_bytes) -> int:
    return load().kvo_attn_sparse_rows_workspace_bytes(rows, n_q_heads, n_kv_heads, head_dim, k_pad,
                                                       rows_per_launch, page_size, num_pages_used,
                                                       arena_bytes)


def kvo_attn_sparse_rows(q, q_dtype, rows, n_q_heads, n_kv_heads, head_dim, k_pages, v_pages, dtype,
                         page_size, n_pages, block_table, num_pages_used, indices, k_pad, scale, arena,
                         arena_bytes, rows_per_launch, out, workspace, workspace_bytes, stream=None) -> None:
    _check(load().kvo_attn_sparse_rows(
        _p(q), q_dtype, rows, n_q_heads, n_kv_heads, head_dim, _p(k_pages), _p(v_pages), dtype,
        page_size, n_pages, _p(block_table), num_pages_used, _p(indices), k_pad, scale, _p(arena),
        arena_bytes, rows_per_launch, _p(out), _p(workspace), workspace_bytes, _s(stream)),
        "kvo_attn_sparse_rows")


def kvo_copy_pages_host(src_k, src_v, dst_k, dst_v, page_tokens, token_bytes, from_page, to_page,
                        num_tokens, stream=None) -> None:
    _check(load().kvo_copy_pages_host(_p(src_k), _p(src_v), _p(dst_k), _p(dst_v), page_tokens,
                                      token_bytes, from_page, to_page, num_tokens, _s(stream)),
           "kvo_copy_pages_host")
