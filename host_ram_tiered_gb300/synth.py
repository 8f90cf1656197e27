"""Seeded synthetic inputs for the tiered KV-cache path.

This module only draws random numbers and packs them into the storage
formats the library reads; it holds none of the method's arithmetic.  The
GPU tests, the CPU oracle's tests and the benchmark all take their inputs
from here, so both sides of every parity check read the same bytes.

Recipe (seed = 1234 + workload index; independent substreams per tensor):
  * fp16 / bf16 values ~ N(0, 1): numpy PCG64 normals in float32, rounded to
    the 16-bit format with round-to-nearest-even.
  * q8_0 blocks: qs ~ U{-127..127} (int8), d ~ U(0.001, 0.02) rounded to fp16.
  * block ids: seeded permutations (numpy ``Generator.permutation``).
  * Very large planes (gigabytes) are filled from a seeded N(0, 1) pool of
    ``POOL_ELEMS`` values: chunk c of ``CHUNK_ELEMS`` elements copies the pool
    starting at a seeded random offset.  The marginal distribution is the
    same; a wrongly addressed block still reads different values.
"""
from __future__ import annotations

import numpy as np

POOL_ELEMS = (1 << 24) + 4099      # not a power of two: chunk offsets never line up
CHUNK_ELEMS = 1 << 20


def rng(seed: int, stream: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream])))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    bias = 0x7FFF + ((u >> 16) & 1)
    return ((u + bias) >> 16).astype(np.uint16)


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """Round to IEEE binary16 (numpy rounds to nearest even); uint16 bits."""
    return np.asarray(x, np.float32).astype(np.float16).view(np.uint16)


def normal_bits(shape, dtype: str, gen: np.random.Generator) -> np.ndarray:
    """N(0,1) values as uint16 bits of 'f16' or 'bf16'."""
    x = gen.standard_normal(size=shape, dtype=np.float32)
    return f32_to_f16_bits(x) if dtype == "f16" else f32_to_bf16_bits(x)


def q8_0_rows(n_rows: int, n_kv_heads: int, head_dim: int, gen: np.random.Generator) -> np.ndarray:
    """Cell rows of q8_0 blocks: [n_rows][n_kv_heads * head_dim/32 * 34] uint8.

    Each 34-byte block is {fp16 scale d (little endian); int8 qs[32]}."""
    nb = n_rows * n_kv_heads * (head_dim // 32)
    d = gen.uniform(0.001, 0.02, size=nb).astype(np.float32)
    qs = gen.integers(-127, 128, size=(nb, 32), dtype=np.int16).astype(np.int8)
    blocks = np.empty((nb, 34), np.uint8)
    blocks[:, 0:2] = f32_to_f16_bits(d).reshape(nb, 1).view(np.uint8).reshape(nb, 2)
    blocks[:, 2:] = qs.view(np.uint8)
    return blocks.reshape(n_rows, -1)


def fill_normal_bits_large(out_u16: np.ndarray, dtype: str, seed: int, stream: int) -> None:
    """Fill a large uint16 array (any shape, C-contiguous) from a seeded pool."""
    flat = out_u16.reshape(-1)
    gen = rng(seed, stream)
    pool = normal_bits(POOL_ELEMS, dtype, gen)
    pool2 = np.concatenate([pool, pool[:CHUNK_ELEMS]])
    n = flat.size
    n_chunks = (n + CHUNK_ELEMS - 1) // CHUNK_ELEMS
    offs = gen.integers(0, POOL_ELEMS, size=n_chunks)
    for c in range(n_chunks):
        a = c * CHUNK_ELEMS
        b = min(n, a + CHUNK_ELEMS)
        o = int(offs[c])
        flat[a:b] = pool2[o:o + (b - a)]


def fill_bytes_large(out_u8: np.ndarray, seed: int, stream: int) -> None:
    """Fill a large byte array with seeded random bytes (pool-tiled as above)."""
    flat = out_u8.reshape(-1)
    gen = rng(seed, stream)
    pool = gen.integers(0, 256, size=POOL_ELEMS, dtype=np.uint8)
    pool2 = np.concatenate([pool, pool[:CHUNK_ELEMS]])
    n = flat.size
    n_chunks = (n + CHUNK_ELEMS - 1) // CHUNK_ELEMS
    offs = gen.integers(0, POOL_ELEMS, size=n_chunks)
    for c in range(n_chunks):
        a = c * CHUNK_ELEMS
        b = min(n, a + CHUNK_ELEMS)
        o = int(offs[c])
        flat[a:b] = pool2[o:o + (b - a)]


def topk_selection(n_seq: int, n_kv_heads: int, n_blocks: int, k: int,
                   gen: np.random.Generator) -> np.ndarray:
    """Per (sequence, kv head): k-1 block ids drawn without replacement from
    [0, n_blocks-1) plus the last block n_blocks-1, sorted ascending. int32."""
    sel = np.empty((n_seq, n_kv_heads, k), np.int32)
    for s in range(n_seq):
        for h in range(n_kv_heads):
            pick = gen.choice(n_blocks - 1, size=k - 1, replace=False)
            sel[s, h, :k - 1] = np.sort(pick)
            sel[s, h, k - 1] = n_blocks - 1
    return sel


def row_selections(rows: int, k_pad: int, first_pos: int, n_pick: int,
                   gen: np.random.Generator, pad_frac: float = 0.0) -> np.ndarray:
    """Per query row i (at position first_pos + i): n_pick distinct cache
    positions drawn uniformly from [0, first_pos + i], in random order, then
    -1 padding up to k_pad; with pad_frac > 0 about that fraction of the picks
    is replaced by -1 as well.  int32 [rows][k_pad]."""
    out = np.full((rows, k_pad), -1, np.int32)
    for i in range(rows):
        hi = first_pos + i + 1
        n = min(n_pick, hi)
        pick = np.unique(gen.integers(0, hi, size=n + n // 4 + 8))
        while pick.size < n:
            pick = np.unique(np.concatenate([pick, gen.integers(0, hi, size=n)]))
        pick = gen.permutation(gen.permutation(pick)[:n])
        out[i, :n] = pick
    if pad_frac > 0:
        out[gen.random(out.shape) < pad_frac] = -1
    return out
