"""Shared helpers of the GPU parity tests: buffers, tiered layouts, metrics."""
from __future__ import annotations

import math

import numpy as np

import oracle
from host_ram_tiered_gb300 import kvo, synth


def torch():
    import torch as t
    return t


def pinned(nbytes: int):
    """Pinned, device-mapped host bytes (cudaHostAlloc through torch)."""
    t = torch()
    return t.empty(max(nbytes, 1), dtype=t.uint8, pin_memory=True)


def host_np(buf, shape=None, dtype=np.uint8) -> np.ndarray:
    """numpy view of a CPU (pinned) torch uint8 buffer."""
    a = buf.numpy().view(dtype)
    return a.reshape(shape) if shape is not None else a


def to_dev(a: np.ndarray):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(a).reshape(-1).view(np.uint8).copy()).cuda()


def to_pinned(a: np.ndarray):
    t = torch()
    flat = np.ascontiguousarray(a).reshape(-1).view(np.uint8)
    buf = pinned(flat.size)
    buf.numpy()[:flat.size] = flat
    return buf


def dev_bytes(x) -> np.ndarray:
    return x.cpu().numpy().view(np.uint8)


def normwise_rel_err(out: np.ndarray, ref: np.ndarray) -> float:
    """max over (row, head) of max_d |o - r| / max_d |r|."""
    o = out.reshape(-1, out.shape[-1]).astype(np.float64)
    r = ref.reshape(-1, ref.shape[-1])
    num = np.abs(o - r).max(axis=1)
    den = np.maximum(np.abs(r).max(axis=1), 1e-300)
    return float((num / den).max())


def cells(L: int, hkv: int, d: int, dtype: int, gen) -> tuple[np.ndarray, np.ndarray]:
    """K and V cell rows [L][row_bytes] (uint8) of a dtype, seeded."""
    if dtype == oracle.Q8_0:
        return synth.q8_0_rows(L, hkv, d, gen), synth.q8_0_rows(L, hkv, d, gen)
    name = "f16" if dtype == oracle.F16 else "bf16"
    k = synth.normal_bits((L, hkv * d), name, gen).view(np.uint8).reshape(L, -1)
    v = synth.normal_bits((L, hkv * d), name, gen).view(np.uint8).reshape(L, -1)
    return np.ascontiguousarray(k), np.ascontiguousarray(v)


class Tiered:
    """A batch of sequences' K/V cells, split at N into a device head
    [B][N] and a pinned host tail [B][L - N], plus the oracle's view."""

    def __init__(self, k: np.ndarray, v: np.ndarray, n_vram: int, batch: int = 1):
        # k, v: [B * L][row_bytes] uint8, sequence-major
        self.batch = batch
        self.L = k.shape[0] // batch
        self.rb = k.shape[1]
        self.n = min(n_vram, self.L)
        kb = k.reshape(batch, self.L, self.rb)
        vb = v.reshape(batch, self.L, self.rb)
        self.k_head_np = np.ascontiguousarray(kb[:, :self.n])
        self.v_head_np = np.ascontiguousarray(vb[:, :self.n])
        self.k_tail_np = np.ascontiguousarray(kb[:, self.n:])
        self.v_tail_np = np.ascontiguousarray(vb[:, self.n:])
        self.k_head = to_dev(self.k_head_np) if self.n > 0 else None
        self.v_head = to_dev(self.v_head_np) if self.n > 0 else None
        self.k_tail = to_pinned(self.k_tail_np) if self.n < self.L else None
        self.v_tail = to_pinned(self.v_tail_np) if self.n < self.L else None

    def oracle_cache(self, dtype, hkv, d):
        def p(a):
            return a if a.size else None
        return oracle.make_cache(p(self.k_head_np), p(self.v_head_np), p(self.k_tail_np),
                                 p(self.v_tail_np), self.n, self.L - self.n, self.n, dtype, hkv, d)


def run_decode(tc: Tiered, q_dev, q_dtype, hq, hkv, d, kv_dtype, ctx_dev, scale, staging=False,
               stream=None):
    t = torch()
    B, L = tc.batch, tc.L
    out = t.empty(B * hq * d, dtype=t.float32, device="cuda")
    ws_bytes = kvo.kvo_attn_decode_workspace_bytes(B, hq, d, L)
    ws = t.empty(max(ws_bytes, 16), dtype=t.uint8, device="cuda")
    sk = sv = None
    if staging and tc.n < L:
        sk = t.empty(B * (L - tc.n) * tc.rb, dtype=t.uint8, device="cuda")
        sv = t.empty_like(sk)
    kvo.kvo_attn_decode_tiered(q_dev, q_dtype, B, hq, hkv, d, tc.k_head, tc.v_head, tc.n,
                               tc.k_tail, tc.v_tail, L - tc.n, kv_dtype, ctx_dev, L, tc.n, scale,
                               sk, sv, out, ws, ws_bytes, stream)
    t.cuda.synchronize()
    return out.cpu().numpy().reshape(B, hq, d)


def scale_for(d: int) -> float:
    return 1.0 / math.sqrt(d)
