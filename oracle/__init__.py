"""ctypes binding of the plain-C CPU oracle (``kvo_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the smoke check in
``__graft_entry__`` and by ``bench.py``'s CPU-baseline leg, never by the
library.  It shares no code with the CUDA library; inputs come from
``host_ram_tiered_gb300.synth`` (seeded generators holding none of the
method's arithmetic), outputs are fp64 numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvo_oracle.so")
SOURCES = [os.path.join(_HERE, "kvo_oracle.c")]

F16, BF16, Q8_0 = 0, 1, 2

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp64, no FMA contraction, OpenMP)."""
    newest = max(os.path.getmtime(s) for s in SOURCES + [os.path.join(_HERE, "kvo_oracle.h")])
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= newest:
        return LIB_PATH
    tmp = LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-o", tmp] + SOURCES + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


class Cache(ctypes.Structure):
    _fields_ = [
        ("k_head", ctypes.c_void_p), ("v_head", ctypes.c_void_p),
        ("k_tail", ctypes.c_void_p), ("v_tail", ctypes.c_void_p),
        ("head_seq_stride_rows", ctypes.c_int64), ("tail_seq_stride_rows", ctypes.c_int64),
        ("n_vram", ctypes.c_int64), ("dtype", ctypes.c_int),
        ("n_kv_heads", ctypes.c_int64), ("head_dim", ctypes.c_int64),
    ]


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(LIB_PATH)
        i64, vp, dbl = ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
        L.orc_half_to_double.argtypes = [ctypes.c_uint16]
        L.orc_half_to_double.restype = dbl
        L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.orc_bf16_to_double.restype = dbl
        L.orc_row_bytes.argtypes = [ctypes.c_int, i64, i64]
        L.orc_row_bytes.restype = i64
        L.orc_load_head.argtypes = [vp, ctypes.c_int, i64, i64, vp]
        L.orc_sub_block_ptrs.argtypes = [vp, i64, i64, i64, ctypes.c_uint64, i64, i64, vp, i64]
        L.orc_sub_block_ptrs.restype = ctypes.c_int
        L.orc_swap_blocks.argtypes = [vp, vp, vp, i64]
        L.orc_gather_blocks.argtypes = [vp, i64, i64, i64, i64, i64, i64, vp, i64, vp]
        L.orc_gather_blocks.restype = ctypes.c_int
        L.orc_attn_partial.argtypes = [ctypes.POINTER(Cache), i64, i64, vp, dbl, i64, i64, vp, vp, vp]
        L.orc_fold.argtypes = [vp, vp, vp, dbl, dbl, vp, i64]
        L.orc_attn_decode.argtypes = [ctypes.POINTER(Cache), vp, ctypes.c_int, i64, i64, vp, dbl, vp]
        L.orc_attn_prefill.argtypes = [ctypes.POINTER(Cache), vp, ctypes.c_int, i64, i64, i64, i64, dbl, vp]
        L.orc_float_to_half_bits.argtypes = [ctypes.c_float]
        L.orc_float_to_half_bits.restype = ctypes.c_uint16
        L.orc_quantize_q8_0_block.argtypes = [vp, vp]
        L.orc_append_kv.argtypes = [vp, vp, ctypes.c_int, i64, i64, i64, i64, vp, vp, vp, vp,
                                    ctypes.c_int, i64]
        L.orc_append_kv.restype = ctypes.c_int
        L.orc_copy_plan.argtypes = [vp] * 6 + [i64, ctypes.c_int, vp, vp, vp, i64]
        L.orc_copy_plan.restype = i64
        L.orc_fragment_ptrs.argtypes = [vp, vp, i64, vp, vp, vp, i64, vp, vp, vp]
        L.orc_staging_worthwhile.argtypes = [i64, i64, i64, i64, ctypes.c_int]
        L.orc_staging_worthwhile.restype = ctypes.c_int
        L.orc_attn_sparse_rows.argtypes = [vp, vp, ctypes.c_int, i64, i64, i64, vp, i64, vp, i64, i64,
                                           vp, ctypes.c_int, i64, dbl, vp]
        L.orc_set_threads.argtypes = [ctypes.c_int]
        L.orc_set_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(a) -> int:
    """Address of a numpy array (C-contiguous) or an int address."""
    if isinstance(a, int):
        return a
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def set_threads(n: int) -> int:
    return lib().orc_set_threads(int(n))


def half_to_double(bits: int) -> float:
    return lib().orc_half_to_double(bits)


def bf16_to_double(bits: int) -> float:
    return lib().orc_bf16_to_double(bits)


def row_bytes(dtype: int, n_kv_heads: int, head_dim: int) -> int:
    return lib().orc_row_bytes(dtype, n_kv_heads, head_dim)


def load_head(row: np.ndarray, dtype: int, head_dim: int, head: int) -> np.ndarray:
    out = np.empty(head_dim, np.float64)
    lib().orc_load_head(_ptr(row), dtype, head_dim, head, _ptr(out))
    return out


def sub_block_ptrs(block_ids, blocks_per_chunk, skip_count, base, row_stride_bytes,
                   row_bytes_, n_out):
    ids = np.ascontiguousarray(block_ids, dtype=np.int64)
    out = np.zeros(max(n_out, 0), np.uint64)
    rc = lib().orc_sub_block_ptrs(_ptr(ids), len(ids), blocks_per_chunk, skip_count,
                                  base, row_stride_bytes, row_bytes_,
                                  _ptr(out) if n_out > 0 else None, n_out)
    if rc != 0:
        raise ValueError("orc_sub_block_ptrs rejected its arguments")
    return out


def swap_blocks(src: np.ndarray, dst: np.ndarray, sizes: np.ndarray) -> None:
    src = np.ascontiguousarray(src, np.uint64)
    dst = np.ascontiguousarray(dst, np.uint64)
    sizes = np.ascontiguousarray(sizes, np.int64)
    lib().orc_swap_blocks(_ptr(src), _ptr(dst), _ptr(sizes), len(sizes))


def gather_blocks(plane: np.ndarray, n_seq, seq_stride_tokens, n_kv_heads, head_dim,
                  elem_bytes, block_tokens, sel: np.ndarray) -> np.ndarray:
    sel = np.ascontiguousarray(sel, np.int32)
    n_sel = sel.shape[-1]
    out = np.empty(n_seq * n_sel * block_tokens * n_kv_heads * head_dim * elem_bytes, np.uint8)
    rc = lib().orc_gather_blocks(_ptr(plane), n_seq, seq_stride_tokens, n_kv_heads, head_dim,
                                 elem_bytes, block_tokens, _ptr(sel), n_sel, _ptr(out))
    if rc != 0:
        raise ValueError("orc_gather_blocks: a selected block lies outside the plane")
    return out


def make_cache(k_head, v_head, k_tail, v_tail, head_seq_stride_rows, tail_seq_stride_rows,
               n_vram, dtype, n_kv_heads, head_dim) -> Cache:
    """Keep the numpy arrays alive in the caller; the struct holds raw addresses."""
    def p(a):
        return None if a is None else _ptr(a)
    return Cache(p(k_head), p(v_head), p(k_tail), p(v_tail), head_seq_stride_rows,
                 tail_seq_stride_rows, n_vram, dtype, n_kv_heads, head_dim)


def copy_plan(runs, gpu_to_cpu: bool):
    """runs: list of (local_offset, local_stride, canonical_offset,
    canonical_stride, num_fragments, fragment_size)."""
    cols = [np.ascontiguousarray([r[k] for r in runs], np.int64) for k in range(6)]
    cap = int(sum(r[4] for r in runs)) + 1
    fs, fd, fz = (np.zeros(cap, np.int64) for _ in range(3))
    n = lib().orc_copy_plan(*[_ptr(c) for c in cols], len(runs), int(gpu_to_cpu), _ptr(fs), _ptr(fd),
                            _ptr(fz), cap)
    if n < 0:
        raise ValueError("orc_copy_plan: capacity")
    return fs[:n].copy(), fd[:n].copy(), fz[:n].copy()


def fragment_ptrs(src_bases, dst_bases, frag_src, frag_dst, frag_sizes):
    sb = np.ascontiguousarray(src_bases, np.uint64)
    db = np.ascontiguousarray(dst_bases, np.uint64)
    fs = np.ascontiguousarray(frag_src, np.int64)
    fd = np.ascontiguousarray(frag_dst, np.int64)
    fz = np.ascontiguousarray(frag_sizes, np.int64)
    nb, nf = sb.size, fs.size
    os_, od, oz = np.zeros(nb * nf, np.uint64), np.zeros(nb * nf, np.uint64), np.zeros(nb * nf, np.int64)
    if nb * nf:
        lib().orc_fragment_ptrs(_ptr(sb), _ptr(db), nb, _ptr(fs), _ptr(fd), _ptr(fz), nf, _ptr(os_),
                                _ptr(od), _ptr(oz))
    return os_, od, oz


def float_to_half_bits(x: float) -> int:
    return lib().orc_float_to_half_bits(x)


def quantize_q8_0_block(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float32)
    assert x.size == 32
    out = np.empty(34, np.uint8)
    lib().orc_quantize_q8_0_block(_ptr(x), _ptr(out))
    return out


def append_kv(k_new, v_new, src_dtype, n_new, pos0, n_kv_heads, head_dim, k_head, v_head,
              k_tail, v_tail, dtype, n_vram) -> None:
    """Writes through the given numpy buffers (None where a tier is absent)."""
    def p(a):
        return None if a is None else _ptr(a)
    rc = lib().orc_append_kv(_ptr(k_new), _ptr(v_new), src_dtype, n_new, pos0, n_kv_heads,
                             head_dim, p(k_head), p(v_head), p(k_tail), p(v_tail), dtype, n_vram)
    if rc != 0:
        raise ValueError("orc_append_kv: unsupported dtype pair")


def attn_partial(cache: Cache, b, kv_head, q: np.ndarray, scale, c0, c1):
    q = np.ascontiguousarray(q, np.float64)
    m = np.zeros(1, np.float64)
    l = np.zeros(1, np.float64)
    acc = np.zeros(cache.head_dim, np.float64)
    lib().orc_attn_partial(ctypes.byref(cache), b, kv_head, _ptr(q), scale, c0, c1,
                           _ptr(m), _ptr(l), _ptr(acc))
    return float(m[0]), float(l[0]), acc


def fold(m, l, acc, m_b, l_b, acc_b):
    """Returns the folded (m, l, acc); inputs are not modified."""
    mm = np.array([m], np.float64)
    ll = np.array([l], np.float64)
    aa = np.array(acc, np.float64, copy=True)
    bb = np.ascontiguousarray(acc_b, np.float64)
    lib().orc_fold(_ptr(mm), _ptr(ll), _ptr(aa), m_b, l_b, _ptr(bb), len(aa))
    return float(mm[0]), float(ll[0]), aa


def attn_decode(cache: Cache, q: np.ndarray, q_dtype, batch, n_q_heads, ctx_len, scale):
    q = np.ascontiguousarray(q, np.uint16)
    ctx = np.ascontiguousarray(ctx_len, np.int32)
    out = np.empty((batch, n_q_heads, cache.head_dim), np.float64)
    lib().orc_attn_decode(ctypes.byref(cache), _ptr(q), q_dtype, batch, n_q_heads, _ptr(ctx),
                          scale, _ptr(out))
    return out


def staging_worthwhile(rows, k_pad, num_pages_used, page_size, enabled=True) -> bool:
    return bool(lib().orc_staging_worthwhile(rows, k_pad, num_pages_used, page_size, int(enabled)))


def attn_sparse_rows(k_pages: np.ndarray, v_pages: np.ndarray, dtype, page_size, n_kv_heads, head_dim,
                     block_table, num_pages_used, indices, q: np.ndarray, q_dtype, n_q_heads, scale):
    """k_pages / v_pages: raw bytes [pages][page_size][n_kv_heads][head_dim];
    indices: int32 [rows][k_pad] (negative = padding); q: uint16 [rows][n_q_heads][head_dim].
    Returns float64 [rows][n_q_heads][head_dim]."""
    kp = np.ascontiguousarray(k_pages).view(np.uint8)
    vp_ = np.ascontiguousarray(v_pages).view(np.uint8)
    bt = np.ascontiguousarray(block_table, np.int32)
    idx = np.ascontiguousarray(indices, np.int32)
    rows, k_pad = idx.shape
    q = np.ascontiguousarray(q, np.uint16)
    out = np.empty((rows, n_q_heads, head_dim), np.float64)
    lib().orc_attn_sparse_rows(_ptr(kp), _ptr(vp_), dtype, page_size, n_kv_heads, head_dim, _ptr(bt),
                               num_pages_used, _ptr(idx), rows, k_pad, _ptr(q), q_dtype, n_q_heads,
                               scale, _ptr(out))
    return out


def attn_prefill(cache: Cache, q: np.ndarray, q_dtype, rows, q_pos0, n_q_heads, ctx_len, scale):
    q = np.ascontiguousarray(q, np.uint16)
    out = np.empty((rows, n_q_heads, cache.head_dim), np.float64)
    lib().orc_attn_prefill(ctypes.byref(cache), _ptr(q), q_dtype, rows, q_pos0, n_q_heads,
                           ctx_len, scale, _ptr(out))
    return out
