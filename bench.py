#!/usr/bin/env python3
"""Benchmark of the tiered KV-cache hot path on GB300 (one JSON line).

Headline: tiered q8_0 decode (48 q heads / 8 kv heads x 128, batch 1, one
layer) at a 184,320-cell context with cells [0, 8192) in VRAM and the rest
in pinned host memory -- microseconds per step, host-link GB/s and the
fraction of the measured pinned-copy peak.  The same line carries every
other row of the path measured on its own workload: the batched block swap
(32 layers x K,V, 2048 blocks per direction, 32 KiB and 2 KiB pages), the
top-k gather from 8 GiB host planes plus the sparse decode over the gathered
4096 tokens, the other decode contexts and VRAM splits with staging on and
off, and the tiered chunked prefill (2048 rows over 262,144 cells, staged
through a 32 MiB arena and direct).

All inputs are seeded synthetic data (host_ram_tiered_gb300.synth).  The
timed region starts with every input resident where the workload puts it
(VRAM head, pinned host tail); each timed step is bracketed by CUDA events
on the launching stream, and L2 is flushed (a 256 MiB device write) between
timed steps.  ``--impl reference`` times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from host_ram_tiered_gb300 import synth  # noqa: E402

METRIC = "tiered-KV decode µs/step & host-link GB/s (% of measured pinned-copy peak)"
HEADLINE = "q8_0_decode_L184320_N8192_direct"
SEED0 = 1234


def torch():
    import torch as t
    return t


def kvo():
    from host_ram_tiered_gb300 import kvo as k
    return k


# ----------------------------------------------------------------- buffers

def pinned(nbytes):
    t = torch()
    return t.empty(max(int(nbytes), 1), dtype=t.uint8, pin_memory=True)


def dev(nbytes):
    t = torch()
    return t.empty(max(int(nbytes), 1), dtype=t.uint8, device="cuda")


def pinned_i64(a):
    buf = pinned(a.size * 8)
    buf.numpy().view(np.int64)[:a.size] = a
    return buf


# ----------------------------------------------------------------- timing

class Timer:
    """K timed steps on one stream, each bracketed by CUDA events, L2 flushed
    in between (outside the events)."""

    def __init__(self):
        t = torch()
        self.stream = t.cuda.current_stream()
        self.flush_buf = t.empty(256 << 20, dtype=t.uint8, device="cuda")

    def flush(self):
        self.flush_buf.fill_(1)

    def run(self, step, steps, warmup, flush=True):
        t = torch()
        for _ in range(warmup):
            step()
        t.cuda.synchronize()
        evs = [(t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in evs:
            if flush:
                self.flush()
            a.record(self.stream)
            step()
            b.record(self.stream)
        t.cuda.synchronize()
        ms = [a.elapsed_time(b) for a, b in evs]
        return sum(ms), ms


def measure_link_peak(timer):
    """Pinned-copy peak per direction: cudaMemcpyAsync of 1 GiB, best of 5."""
    t = torch()
    n = 1 << 30
    h = pinned(n)
    d = dev(n)
    out = {}
    for name, fn in (("h2d", lambda: d.copy_(h, non_blocking=True)),
                     ("d2h", lambda: h.copy_(d, non_blocking=True))):
        _, ms = timer.run(fn, 5, 2, flush=False)
        out[name] = n / (min(ms) * 1e-3) / 1e9
    del h, d
    return out


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.rows, self.proc = [], None
        dev_idx = os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0] or "0"
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", dev_idx, f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            try:
                sm.append(float(r[0]))
                mx.append(float(r[1]))
            except (ValueError, IndexError):
                continue
            for i, nm in enumerate(names):
                if len(r) > 4 + i and r[4 + i].lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- tiny paged cache (swap + decode)

def tiny_setup(seed=SEED0):
    """Tiny case: 2 layers x K,V paged fp16 (16 tokens x 8 heads x 128 = 32 KiB
    pages), 64 seeded blocks swapped between 128-block pools; decode for one
    sequence, 32 q / 8 kv heads, 1024 cells with 512 in VRAM."""
    t = torch()
    k = kvo()
    g = synth.rng(seed, 1)
    page, nt, pool, nb = 32768, 4, 128, 64
    d = dev(nt * pool * page)
    h = pinned(nt * pool * page)
    synth.fill_bytes_large(h.numpy(), seed, 2)
    gids = g.permutation(pool)[:nb].astype(np.int64)
    hids = g.permutation(pool)[:nb].astype(np.int64)
    gp = np.empty(nt * nb, np.int64)
    hp = np.empty(nt * nb, np.int64)
    for i in range(nt):
        k.kvo_sub_block_ptrs(gids.ctypes.data, nb, 1, 0, d.data_ptr() + i * pool * page, page, page,
                             gp[i * nb:].ctypes.data, nb)
        k.kvo_sub_block_ptrs(hids.ctypes.data, nb, 1, 0, h.data_ptr() + i * pool * page, page, page,
                             hp[i * nb:].ctypes.data, nb)
    st = {"dev": d, "host": h, "n_desc": nt * nb, "bytes": nt * nb * page,
          "sizes": pinned_i64(np.full(nt * nb, page, np.int64)),
          "h2d_src": pinned_i64(hp), "h2d_dst": pinned_i64(gp),
          "d2h_src": pinned_i64(gp), "d2h_dst": pinned_i64(hp)}
    L, N, hq, hkv, D = 1024, 512, 32, 8, 128
    rb = hkv * D * 2
    kc = synth.normal_bits((L, hkv * D), "f16", g).view(np.uint8).reshape(L, rb)
    vc = synth.normal_bits((L, hkv * D), "f16", g).view(np.uint8).reshape(L, rb)
    q = synth.normal_bits((1, hq, D), "f16", g)
    st.update({"k_head": t.from_numpy(kc[:N].copy().reshape(-1)).cuda(),
               "v_head": t.from_numpy(vc[:N].copy().reshape(-1)).cuda(),
               "k_tail": t.from_numpy(kc[N:].copy().reshape(-1)).pin_memory(),
               "v_tail": t.from_numpy(vc[N:].copy().reshape(-1)).pin_memory(),
               "q": t.from_numpy(q.view(np.int16).reshape(-1).copy()).cuda(),
               "ctx": t.tensor([L], dtype=t.int32, device="cuda"),
               "out": t.empty(hq * D, dtype=t.float32, device="cuda"),
               "stage_k": dev((L - N) * rb), "stage_v": dev((L - N) * rb),
               "L": L, "N": N, "hq": hq, "hkv": hkv, "rb": rb})
    st["ws_bytes"] = k.kvo_attn_decode_workspace_bytes(1, hq, D, L)
    st["ws"] = dev(st["ws_bytes"])
    return st


def tiny_decode(st, staging):
    k = kvo()
    L, N = st["L"], st["N"]
    k.kvo_attn_decode_tiered(st["q"], k.F16, 1, st["hq"], st["hkv"], 128, st["k_head"], st["v_head"], N,
                             st["k_tail"], st["v_tail"], L - N, k.F16, st["ctx"], L, N,
                             1.0 / math.sqrt(128), st["stage_k"] if staging else None,
                             st["stage_v"] if staging else None, st["out"], st["ws"], st["ws_bytes"])


# ----------------------------------------------------------------- 32-layer offload swap

SWAP_TENSORS, SWAP_GPU_BLOCKS, SWAP_HOST_CHUNKS, SWAP_BLOCKS, SWAP_BPC, SWAP_SKIP = 64, 4096, 640, 2048, 4, 1


def swap_setup(page, seed=SEED0 + 1):
    """vLLM-style CPU offload swap: 64 paged tensors (32 layers x K,V), 2048
    seeded GPU block ids per direction, host chunks of 4 pages with a row
    stride of 1.5 x the chunk, skip 1 on the first chunk."""
    k = kvo()
    row = SWAP_BPC * page
    stride = row * 3 // 2
    gpu_bytes = SWAP_GPU_BLOCKS * page
    host_bytes = SWAP_HOST_CHUNKS * stride
    d = dev(SWAP_TENSORS * gpu_bytes)
    h = pinned(SWAP_TENSORS * host_bytes)
    init = np.empty(SWAP_TENSORS * gpu_bytes, np.uint8)
    synth.fill_bytes_large(init, seed, 2)
    d.copy_(torch().from_numpy(init))
    synth.fill_bytes_large(h.numpy(), seed, 3)
    g = synth.rng(seed, 4)
    gpu_ids = g.permutation(SWAP_GPU_BLOCKS)[:SWAP_BLOCKS].astype(np.int64)
    need = -(-(SWAP_BLOCKS + SWAP_SKIP) // SWAP_BPC)
    host_ids = g.permutation(SWAP_HOST_CHUNKS)[:need].astype(np.int64)
    n_desc = SWAP_TENSORS * SWAP_BLOCKS
    hp = np.empty(n_desc, np.int64)
    gp = np.empty(n_desc, np.int64)
    for i in range(SWAP_TENSORS):
        k.kvo_sub_block_ptrs(host_ids.ctypes.data, need, SWAP_BPC, SWAP_SKIP, h.data_ptr() + i * host_bytes,
                             stride, row, hp[i * SWAP_BLOCKS:].ctypes.data, SWAP_BLOCKS)
        k.kvo_sub_block_ptrs(gpu_ids.ctypes.data, SWAP_BLOCKS, 1, 0, d.data_ptr() + i * gpu_bytes,
                             page, page, gp[i * SWAP_BLOCKS:].ctypes.data, SWAP_BLOCKS)
    sizes = pinned_i64(np.full(n_desc, page, np.int64))
    st = {"page": page, "dev": d, "host": h, "n_desc": n_desc, "sizes": sizes,
          "h2d_src": pinned_i64(hp), "h2d_dst": pinned_i64(gp),
          "d2h_src": pinned_i64(gp), "d2h_dst": pinned_i64(hp),
          "bytes": n_desc * page, "init_dev": init, "host_ids": host_ids, "gpu_ids": gpu_ids}
    st["init_dev_sample"] = lambda off, n: init[off:off + n]
    st["d2h_src_np"], st["d2h_dst_np"] = gp, hp
    return st


def swap_run(st, h2d, flags=0, shard=None):
    """One swap direction; shard = (lo, hi) takes descriptors [lo, hi) only."""
    k = kvo()
    lo, hi = shard if shard is not None else (0, st["n_desc"])
    if hi <= lo:
        return
    src, dst = (st["h2d_src"], st["h2d_dst"]) if h2d else (st["d2h_src"], st["d2h_dst"])
    k.kvo_swap_blocks_batch(src.data_ptr() + 8 * lo, dst.data_ptr() + 8 * lo, st["sizes"].data_ptr() + 8 * lo,
                            hi - lo, (k.KVO_SWAP_H2D | k.KVO_SWAP_SRC_ORDER_ANY if h2d else k.KVO_SWAP_D2H) | flags)


# SM copies against the copy engine: page sizes (KiB) and descriptor counts of
# the crossover sweep, each a set of seeded random block ids in 2,560-page pools.
SWEEP_PAGES_KIB = (2, 8, 32, 128, 1024)
SWEEP_COUNTS = (64, 2048)
SWEEP_POOL = 2560


def swap_sweep_setup(page, seed=SEED0 + 5):
    """Device and pinned pools of SWEEP_POOL pages, descriptors for the largest
    count (smaller counts take a prefix)."""
    k = kvo()
    d = dev(SWEEP_POOL * page)
    h = pinned(SWEEP_POOL * page)
    synth.fill_bytes_large(h.numpy(), seed, page)
    g = synth.rng(seed, page)
    n = max(SWEEP_COUNTS)
    gids = g.permutation(SWEEP_POOL)[:n].astype(np.int64)
    hids = g.permutation(SWEEP_POOL)[:n].astype(np.int64)
    gp = np.empty(n, np.int64)
    hp = np.empty(n, np.int64)
    k.kvo_sub_block_ptrs(gids.ctypes.data, n, 1, 0, d.data_ptr(), page, page, gp.ctypes.data, n)
    k.kvo_sub_block_ptrs(hids.ctypes.data, n, 1, 0, h.data_ptr(), page, page, hp.ctypes.data, n)
    return {"page": page, "dev": d, "host": h, "gp": pinned_i64(gp), "hp": pinned_i64(hp),
            "sizes": pinned_i64(np.full(n, page, np.int64))}


def swap_sweep_run(st, h2d, n, ce):
    k = kvo()
    src, dst = (st["hp"], st["gp"]) if h2d else (st["gp"], st["hp"])
    k.kvo_swap_blocks_batch(src, dst, st["sizes"], n,
                            (k.KVO_SWAP_H2D if h2d else k.KVO_SWAP_D2H) |
                            (k.KVO_SWAP_FORCE_CE if ce else k.KVO_SWAP_FORCE_SM))


# ----------------------------------------------------------------- q8_0 tiered decode

DEC_HQ, DEC_HKV, DEC_D = 48, 8, 128
# VRAM heads and host-tail sizes (cells) of the staged/direct decode sweep
DEC_SWEEP_NS = (8192, 32768, 65536, 94208)
DEC_SWEEP_TAILS = (1024, 2048, 4096, 8192, 16384, 32768)
DEC_LS = (29696, 96256, 184320)
DEC_NS = (8192, 94208)


def dec_setup(seed=SEED0 + 2, l_max=max(DEC_LS), n_max=max(DEC_NS)):
    """llama.cpp-style tiered decode, q8_0 K/V (blocks of 32 int8 uniform in
    [-127, 127] and an fp16 scale ~U(0.001, 0.02)), one layer, batch 1."""
    t = torch()
    g = synth.rng(seed, 1)
    rb = DEC_HKV * (DEC_D // 32) * 34
    k_all = pinned(l_max * rb)
    v_all = pinned(l_max * rb)
    chunk = 16384
    for c0 in range(0, l_max, chunk):
        n = min(chunk, l_max - c0)
        k_all.numpy()[c0 * rb:(c0 + n) * rb] = synth.q8_0_rows(n, DEC_HKV, DEC_D, g).reshape(-1)
        v_all.numpy()[c0 * rb:(c0 + n) * rb] = synth.q8_0_rows(n, DEC_HKV, DEC_D, g).reshape(-1)
    q = synth.normal_bits((1, DEC_HQ, DEC_D), "f16", g)
    st = {"rb": rb, "k_host": k_all, "v_host": v_all,
          "k_dev": k_all[:n_max * rb].cuda(), "v_dev": v_all[:n_max * rb].cuda(),
          "k_dev_all": k_all.cuda(), "v_dev_all": v_all.cuda(),
          "q_np": q, "q": t.from_numpy(q.view(np.int16).reshape(-1).copy()).cuda(),
          "out": t.empty(DEC_HQ * DEC_D, dtype=t.float32, device="cuda"),
          "stage_k": dev(l_max * rb), "stage_v": dev(l_max * rb)}
    st["ws_bytes"] = kvo().kvo_attn_decode_workspace_bytes(1, DEC_HQ, DEC_D, l_max)
    st["ws"] = dev(st["ws_bytes"])
    st["ctx"] = {}
    return st


def dec_ctx(st, L):
    t = torch()
    if L not in st["ctx"]:
        st["ctx"][L] = t.tensor([L], dtype=t.int32, device="cuda")
    return st["ctx"][L]


def dec_run(st, L, N, staging=False, all_vram=False, q=None, out=None):
    k = kvo()
    rb = st["rb"]
    ws_bytes = k.kvo_attn_decode_workspace_bytes(1, DEC_HQ, DEC_D, L)
    if all_vram:
        kh, vh, kt, vt, n = st["k_dev_all"], st["v_dev_all"], None, None, L
    else:
        n = min(N, L)
        kh, vh = st["k_dev"], st["v_dev"]
        kt = st["k_host"].data_ptr() + n * rb
        vt = st["v_host"].data_ptr() + n * rb
    k.kvo_attn_decode_tiered(q if q is not None else st["q"], k.F16, 1, DEC_HQ, DEC_HKV, DEC_D,
                             kh, vh, n, kt, vt, L - n, k.Q8_0, dec_ctx(st, L), L, n,
                             1.0 / math.sqrt(DEC_D),
                             st["stage_k"] if staging else None, st["stage_v"] if staging else None,
                             out if out is not None else st["out"], st["ws"], ws_bytes)


VMM_RAN = [False]


def vmm_setup(st, L=184320, N=8192):
    """The headline decode's K/V planes copied into two VMM tiers (a VRAM head of
    N cells, then a host-NUMA tail in the same device range)."""
    k = kvo()
    t = torch()
    rb = st["rb"]
    try:
        tk = k.kvo_vmm_tier_create(0, N * rb, (L - N) * rb)
        tv = k.kvo_vmm_tier_create(0, N * rb, (L - N) * rb)
    except k.KvoError as e:
        return {"unavailable": str(e)}
    chunk = 1 << 16
    offs = np.arange(0, L * rb, chunk, dtype=np.int64)
    sizes = t.from_numpy(np.minimum(chunk, L * rb - offs).astype(np.int64)).cuda()
    for src, tier in ((st["k_dev_all"], tk), (st["v_dev_all"], tv)):
        k.kvo_swap_blocks_batch(t.from_numpy(src.data_ptr() + offs).cuda(), t.from_numpy(tier["base"] + offs).cuda(),
                                sizes, len(offs), k.KVO_SWAP_H2D | k.KVO_SWAP_FORCE_SM)
    t.cuda.synchronize()
    return {"tk": tk, "tv": tv, "L": L, "N": N}


def vmm_run(st, vm, staging=False):
    """Decode over the tiers through one base pointer per plane (staging: the
    host tail copied to a VRAM buffer by the copy engine first)."""
    k = kvo()
    L, N = vm["L"], vm["N"]
    k.kvo_attn_decode_tiered(st["q"], k.F16, 1, DEC_HQ, DEC_HKV, DEC_D, vm["tk"]["base"], vm["tv"]["base"], L,
                             None, None, L, k.Q8_0, dec_ctx(st, L), L, N, 1.0 / math.sqrt(DEC_D),
                             st["stage_k"] if staging else None, st["stage_v"] if staging else None,
                             st["out"], st["ws"], k.kvo_attn_decode_workspace_bytes(1, DEC_HQ, DEC_D, L))


def k_launches_staged_headline():
    return kvo().kvo_attn_decode_launches(1, 184320, DEC_D, 8192, 1)


def vmm_free(vm):
    k = kvo()
    for key in ("tk", "tv"):
        if key in vm:
            k.kvo_vmm_tier_destroy(vm[key]["tier"])


def dec_bytes(L, N):
    rb2 = 2 * DEC_HKV * (DEC_D // 32) * 34
    return max(L - N, 0) * rb2, min(L, N) * rb2


# ----------------------------------------------------------------- top-k block gather + sparse decode

TOPK_S, TOPK_T, TOPK_HQ, TOPK_HKV, TOPK_D, TOPK_BLK, TOPK_K = 8, 1 << 20, 16, 4, 128, 64, 64


def topk_setup(seed=SEED0 + 3, shard=None):
    """QSA-style sparse decode: bf16 K/V planes [8][2^20][4][128] in pinned
    host memory, 64 of 16,384 blocks per (sequence, kv head) selected
    without replacement (the last block always), gathered into VRAM, then
    decode over the 4096 gathered tokens.  shard = (lo, hi): this process
    holds and computes sequences [lo, hi) only (the other sequences' planes
    are not allocated)."""
    t = torch()
    lo, hi = shard if shard is not None else (0, TOPK_S)
    plane = (hi - lo) * TOPK_T * TOPK_HKV * TOPK_D
    k_plane = pinned(plane * 2)
    v_plane = pinned(plane * 2)
    synth.fill_normal_bits_large(k_plane.numpy().view(np.uint16), "bf16", seed, 1)
    synth.fill_normal_bits_large(v_plane.numpy().view(np.uint16), "bf16", seed, 2)
    g = synth.rng(seed, 3)
    sel = synth.topk_selection(TOPK_S, TOPK_HKV, TOPK_T // TOPK_BLK, TOPK_K, g)[lo:hi]
    q = synth.normal_bits((TOPK_S, TOPK_HQ, TOPK_D), "bf16", g)[lo:hi]
    tok = TOPK_K * TOPK_BLK
    n = hi - lo
    out_bytes = n * tok * TOPK_HKV * TOPK_D * 2
    st = {"k_plane": k_plane, "v_plane": v_plane, "sel_np": sel, "n_seq": n,
          "sel": t.from_numpy(sel.reshape(-1).copy()).cuda(),
          "kg": dev(out_bytes), "vg": dev(out_bytes), "q_np": q,
          "q": t.from_numpy(q.view(np.int16).reshape(-1).copy()).cuda(),
          "ctx": t.full((n,), tok, dtype=t.int32, device="cuda"),
          "out": t.empty(n * TOPK_HQ * TOPK_D, dtype=t.float32, device="cuda"),
          "gather_bytes": 2 * out_bytes}
    st["ws_bytes"] = kvo().kvo_attn_decode_workspace_bytes(n, TOPK_HQ, TOPK_D, tok)
    st["ws"] = dev(st["ws_bytes"])
    return st


def topk_gather(st):
    k = kvo()
    k.kvo_gather_blocks(st["k_plane"], st["v_plane"], st["n_seq"], TOPK_T, TOPK_HKV, TOPK_D, k.BF16, TOPK_BLK,
                        st["sel"], TOPK_K, st["kg"], st["vg"])


def topk_decode(st):
    k = kvo()
    tok = TOPK_K * TOPK_BLK
    k.kvo_attn_decode_tiered(st["q"], k.BF16, st["n_seq"], TOPK_HQ, TOPK_HKV, TOPK_D, st["kg"], st["vg"], tok,
                             None, None, 0, k.BF16, st["ctx"], tok, tok, 1.0 / math.sqrt(TOPK_D),
                             None, None, st["out"], st["ws"], st["ws_bytes"])


# ----------------------------------------------------------------- tiered chunked prefill

PF_R, PF_POS0, PF_L, PF_HQ, PF_HKV, PF_D, PF_N = 2048, 260096, 262144, 32, 8, 128, 65536
PF_ARENA, PF_RPL = 32 << 20, 1024
# FP32 multiply-adds per second on CUDA cores: 152 SMs x 128 lanes x 2.07 GHz
FP32_FMA_PEAK = 152 * 128 * 2.07e9


def pf_setup(seed=SEED0 + 4):
    """Tiered chunked prefill: 2048 query rows at positions 260,096-262,143,
    bf16 K/V cells [262,144][8][128], cells [0, 65,536) in VRAM, the tail in
    pinned host memory; staged through a 32 MiB arena, 1024 rows a launch."""
    t = torch()
    rb = PF_HKV * PF_D * 2
    g_seed = seed
    k_host = pinned((PF_L - PF_N) * rb)
    v_host = pinned((PF_L - PF_N) * rb)
    k_head = np.empty(PF_N * rb // 2, np.uint16)
    v_head = np.empty(PF_N * rb // 2, np.uint16)
    synth.fill_normal_bits_large(k_head, "bf16", g_seed, 1)
    synth.fill_normal_bits_large(v_head, "bf16", g_seed, 2)
    synth.fill_normal_bits_large(k_host.numpy().view(np.uint16), "bf16", g_seed, 3)
    synth.fill_normal_bits_large(v_host.numpy().view(np.uint16), "bf16", g_seed, 4)
    q = synth.normal_bits((PF_R, PF_HQ, PF_D), "bf16", synth.rng(g_seed, 5))
    st = {"rb": rb, "k_host": k_host, "v_host": v_host, "k_head_np": k_head, "v_head_np": v_head,
          "k_head": t.from_numpy(k_head.view(np.int16)).cuda(),
          "v_head": t.from_numpy(v_head.view(np.int16)).cuda(), "q_np": q,
          "q": t.from_numpy(q.view(np.int16).reshape(-1).copy()).cuda(),
          "arena": dev(PF_ARENA),
          "out": t.empty(PF_R * PF_HQ * PF_D, dtype=t.float32, device="cuda")}
    st["ws_bytes"] = kvo().kvo_attn_prefill_workspace_bytes(PF_R, PF_HQ)
    st["ws"] = dev(st["ws_bytes"])
    return st


def pf_run(st, staged=True, q=None, out=None):
    k = kvo()
    k.kvo_attn_prefill_tiered(q if q is not None else st["q"], PF_R, PF_POS0, PF_HQ, PF_HKV, PF_D,
                              st["k_head"], st["v_head"], st["k_host"], st["v_host"], k.BF16, PF_L,
                              PF_N, 1.0 / math.sqrt(PF_D),
                              st["arena"] if staged else None, PF_ARENA if staged else 0, PF_RPL,
                              out if out is not None else st["out"], st["ws"], st["ws_bytes"])


# Query-row counts of the staged/direct crossover sweep: the last `rows`
# positions of the 262,144-cell context, the same cells and tiers as above.
PF_SWEEP_ROWS = (1, 4, 16, 64, 256)


def pf_run_rows(st, rows, staged):
    k = kvo()
    k.kvo_attn_prefill_tiered(st["q"], rows, PF_L - rows, PF_HQ, PF_HKV, PF_D, st["k_head"], st["v_head"],
                              st["k_host"], st["v_host"], k.BF16, PF_L, PF_N, 1.0 / math.sqrt(PF_D),
                              st["arena"] if staged else None, PF_ARENA if staged else 0,
                              min(PF_RPL, rows), st["out"], st["ws"], st["ws_bytes"])


def pf_flops(rows=PF_R, pos0=PF_POS0):
    # causal: row i sees pos0 + i + 1 cells; QK^T and PV are 2 flops per MAC each
    cells = sum(pos0 + i + 1 for i in range(rows))
    return 4.0 * PF_HQ * PF_D * cells


# ----------------------------------------------------------------- QSA sparse rows (next row)

# ExLlamaV3 QSA offload prefill: 2048 query rows, each picking 2080 cache
# positions, over a paged fp16 host cache of 262,144 positions (1,024 pages
# of 256 tokens, 32 q / 8 kv heads x 128), staged through a 32 MiB arena.
SR_R, SR_POS0, SR_L, SR_PS, SR_KPAD = 2048, 260096, 262144, 256, 2080
SR_HQ, SR_HKV, SR_D, SR_ARENA, SR_RPL = 32, 8, 128, 32 << 20, 1024


def sr_setup(seed=SEED0 + 6):
    t = torch()
    n_pages = SR_L // SR_PS
    page_bytes = SR_PS * SR_HKV * SR_D * 2
    k_pages = pinned(n_pages * page_bytes)
    v_pages = pinned(n_pages * page_bytes)
    synth.fill_normal_bits_large(k_pages.numpy().view(np.uint16), "f16", seed, 1)
    synth.fill_normal_bits_large(v_pages.numpy().view(np.uint16), "f16", seed, 2)
    g = synth.rng(seed, 3)
    bt = g.permutation(n_pages).astype(np.int32)
    idx = synth.row_selections(SR_R, SR_KPAD, SR_POS0, SR_KPAD, synth.rng(seed, 4))
    q = synth.normal_bits((SR_R, SR_HQ, SR_D), "f16", synth.rng(seed, 5))
    st = {"n_pages": n_pages, "page_bytes": page_bytes, "k_pages": k_pages, "v_pages": v_pages,
          "bt_np": bt, "idx_np": idx, "q_np": q, "bt": t.from_numpy(bt).cuda(),
          "idx": t.from_numpy(idx.reshape(-1).copy()).cuda(),
          "q": t.from_numpy(q.view(np.int16).reshape(-1).copy()).cuda(), "arena": dev(SR_ARENA),
          "out": t.empty(SR_R * SR_HQ * SR_D, dtype=t.float32, device="cuda")}
    k = kvo()
    st["ws_bytes"] = max(k.kvo_attn_sparse_rows_workspace_bytes(SR_R, SR_HQ, SR_HKV, SR_D, SR_KPAD, SR_RPL,
                                                                SR_PS, n_pages, a)
                         for a in (0, SR_ARENA))
    st["ws"] = dev(st["ws_bytes"])
    return st


def sr_run(st, staged=True):
    k = kvo()
    k.kvo_attn_sparse_rows(st["q"], k.F16, SR_R, SR_HQ, SR_HKV, SR_D, st["k_pages"], st["v_pages"], k.F16,
                           SR_PS, st["n_pages"], st["bt"], st["n_pages"], st["idx"], SR_KPAD,
                           1.0 / math.sqrt(SR_D), st["arena"] if staged else None, SR_ARENA if staged else 0,
                           SR_RPL, st["out"], st["ws"], st["ws_bytes"])


# ----------------------------------------------------------------- write path (append)

def append_setup(seed=SEED0 + 5):
    """Appends into the host tails of the q8_0 decode cache and the bf16 prefill cache: one
    decode token (q8_0) and one 2048-token prefill chunk (q8_0 and bf16)."""
    t = torch()
    g = synth.rng(seed, 1)
    n = 2048
    st = {"n": n}
    for name, hkv in (("q8", DEC_HKV), ("bf", PF_HKV)):
        x = synth.normal_bits((n, hkv * 128), "bf16" if name == "bf" else "f16", g)
        st[name + "_k"] = t.from_numpy(x.view(np.int16).reshape(-1).copy()).cuda()
        st[name + "_v"] = t.from_numpy(x[::-1].copy().view(np.int16).reshape(-1)).cuda()
    st["q8_rb"] = DEC_HKV * 4 * 34
    st["bf_rb"] = PF_HKV * 128 * 2
    cap = 8192 + 4096
    st["cap"] = cap
    st["q8_tail_k"] = pinned((cap - 8192) * st["q8_rb"])
    st["q8_tail_v"] = pinned((cap - 8192) * st["q8_rb"])
    st["bf_tail_k"] = pinned((cap - 8192) * st["bf_rb"])
    st["bf_tail_v"] = pinned((cap - 8192) * st["bf_rb"])
    st["q8_head"] = dev(8192 * st["q8_rb"])
    st["bf_head"] = dev(8192 * st["bf_rb"])
    return st


def append_run(st, which, n_tokens):
    k = kvo()
    q8 = which == "q8"
    k.kvo_append_kv_tiered(st[which + "_k"], st[which + "_v"], k.F16 if q8 else k.BF16, n_tokens,
                           8192 + 1000, DEC_HKV if q8 else PF_HKV, 128, st[which + "_head"],
                           st[which + "_head"], st[which + "_tail_k"], st[which + "_tail_v"],
                           k.Q8_0 if q8 else k.BF16, 8192, st["cap"])


# ----------------------------------------------------------------- CPU oracle arm

def oracle_c3_step(L, heads=DEC_HQ):
    """fp64 oracle decode of the headline workload (q8_0, L cells, N split),
    on host copies of the same seeded inputs."""
    import oracle
    g = synth.rng(SEED0 + 2, 1)
    rb = DEC_HKV * (DEC_D // 32) * 34
    k = np.empty((L, rb), np.uint8)
    v = np.empty((L, rb), np.uint8)
    chunk = 16384
    for c0 in range(0, max(DEC_LS), chunk):
        n = min(chunk, max(DEC_LS) - c0)
        kk = synth.q8_0_rows(n, DEC_HKV, DEC_D, g)
        vv = synth.q8_0_rows(n, DEC_HKV, DEC_D, g)
        if c0 < L:
            m = min(n, L - c0)
            k[c0:c0 + m] = kk[:m]
            v[c0:c0 + m] = vv[:m]
    q = synth.normal_bits((1, DEC_HQ, DEC_D), "f16", g)
    N = 8192
    kh, vh = np.ascontiguousarray(k[:N]), np.ascontiguousarray(v[:N])
    kt, vt = np.ascontiguousarray(k[N:]), np.ascontiguousarray(v[N:])
    cache = oracle.make_cache(kh, vh, kt, vt, N, L - N, N, oracle.Q8_0, DEC_HKV, DEC_D)
    keep = (kh, vh, kt, vt)
    qs = np.ascontiguousarray(q[:, :heads])

    def step():
        return oracle.attn_decode(cache, qs, oracle.F16, 1, heads, [L], 1.0 / math.sqrt(DEC_D))
    return step, keep


def headline_config():
    return {"workload": HEADLINE, "L": 184320, "n_vram_cells": 8192, "q_heads": DEC_HQ,
            "kv_heads": DEC_HKV, "head_dim": DEC_D, "kv_dtype": "q8_0", "batch": 1,
            "staging": False, "l2": "flushed between timed steps (256 MiB write)"}


def run_reference(args):
    import oracle
    oracle.build()
    threads = oracle.set_threads(os.cpu_count() or 1)
    L = max(DEC_LS)
    # Every step is the whole headline decode (all 48 query heads over the
    # 184,320 cells, parallel over heads on the host's cores): about 2 s on
    # 16 Grace cores, so the default 20 + 5 steps end within a minute.
    step, keep = oracle_c3_step(L, DEC_HQ)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    us = dt / args.steps * 1e6
    host_b, dev_b = dec_bytes(L, 8192)
    line = {"impl": "reference", "metric": METRIC, "value": us, "unit": "us/step",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": us / 1e3, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": headline_config(),
            "cpu_baseline": {"value": us, "unit": "us/step", "cores": threads, "kind": "oracle",
                             "sample": f"the whole headline step ({DEC_HQ} query heads x {L} cells), "
                                       f"{args.steps} timed steps, no scaling"},
            "e2e": {"value": us, "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "host_gbs_equiv": host_b / (us * 1e-6) / 1e9}
    return line


# ----------------------------------------------------------------- main

def rank_info():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    t = torch()
    import torch.distributed as dist
    v = t.tensor([x], dtype=t.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(v, op=dist.ReduceOp.MAX)
    return float(v.item())


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="kvo", choices=["kvo", "reference"])
    ap.add_argument("--rows", default="all",
                    help="comma list of head (headline decode only), tiny, swap, swapsweep (SM copies vs the copy "
                         "engine over page sizes), decode, vmm (the headline decode "
                         "over VMM tiers), topk, prefill, append, sparse (QSA sparse rows), decode_vram (the 184,320-"
                         "cell all-VRAM decode alone; not in 'all') (default: all rows at one GPU, the headline alone "
                         "under torchrun)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--split", default="replicas", choices=["replicas", "shards"],
                    help="under torchrun: every rank runs the whole workload (replicas, weak scaling), or the "
                         "swap descriptors and the top-k sequences are divided among the ranks by "
                         "kvo_shard_range (shards, strong scaling; the headline decode of one sequence stays "
                         "a replica)")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)
    rank, world, local = rank_info()

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return 0

    t = torch()
    t.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    from host_ram_tiered_gb300 import build
    build.build()
    k = kvo()
    k.load()
    # Every row at one GPU.  Under torchrun each rank replicates the workload,
    # so the default there is the headline alone (the full set would pin about
    # 30 GB of host memory per rank).
    if args.rows == "all" and world > 1:
        rows = {"head", "swap", "topk"} if args.split == "shards" else {"head"}
    elif args.rows == "all":
        rows = {"head", "tiny", "swap", "swapsweep", "decode", "decsweep", "vmm", "topk", "prefill", "pfsweep",
                "append", "sparse"}
    else:
        rows = set(args.rows.split(","))
    timer = Timer()
    peaks = measure_link_peak(timer)
    hbm = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))).get("hbm_gbs", 6789.0) \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else 6800.0
    K, W = args.steps, args.warmup
    results = {}

    def shard(n_units):
        """This rank's contiguous share [lo, hi) of n_units (everything without --split shards)."""
        if world == 1 or args.split != "shards":
            return 0, n_units
        return k.kvo_shard_range(n_units, world, rank)

    def bar():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        t.cuda.synchronize()

    clocks = Clocks()
    # ---- headline: q8_0 tiered decode at L = 184,320, N = 8,192, direct
    head = None
    if "decode" in rows or "head" in rows or "vmm" in rows or "decsweep" in rows:
        st3 = dec_setup()
        bar()
        tot, ms = timer.run(lambda: dec_run(st3, 184320, 8192), K, W)
        tot = max_over_ranks(tot, world)
        us = tot / K * 1e3
        hb, db = dec_bytes(184320, 8192)
        head = {"us": us, "host_bytes": hb, "dev_bytes": db, "ms": ms}
        results[HEADLINE] = {"us_per_step": us, "host_gbs": hb / (us * 1e-6) / 1e9,
                             "frac_link_peak": hb / (us * 1e-6) / 1e9 / peaks["h2d"]}
        # e2e through the C-ABI with host buffers: q from pinned host, out back to pinned host
        q_h = t.from_numpy(st3["q_np"].view(np.int16).reshape(-1).copy()).pin_memory()
        o_h = t.empty(DEC_HQ * DEC_D, dtype=t.float32).pin_memory()
        q_d = t.empty_like(st3["q"])
        o_d = t.empty_like(st3["out"])

        def e2e_step():
            q_d.copy_(q_h, non_blocking=True)
            dec_run(st3, 184320, 8192, q=q_d, out=o_d)
            o_h.copy_(o_d, non_blocking=True)
        tot_e, _ = timer.run(e2e_step, K, W)
        tot_e = max_over_ranks(tot_e, world)
        head["e2e_us"] = tot_e / K * 1e3
        head["e2e_h2d"] = q_h.numel() * 2
        head["e2e_d2h"] = o_h.numel() * 4
        if "decode" in rows:
            for L in DEC_LS:
                for N in DEC_NS:
                    for staging in (False, True):
                        if L <= N and staging:
                            continue
                        tot, _ = timer.run(lambda: dec_run(st3, L, N, staging=staging), K, W)
                        us_r = max_over_ranks(tot, world) / K * 1e3
                        hb_r, db_r = dec_bytes(L, N)
                        if staging:
                            db_r += 2 * hb_r
                        key = f"q8_0_decode_L{L}_N{N}_{'staged' if staging else 'direct'}"
                        t_star = max(hb_r / (peaks['h2d'] * 1e9), db_r / (hbm * 1e9))
                        results[key] = {"us_per_step": us_r, "host_gbs": hb_r / (us_r * 1e-6) / 1e9,
                                        "roofline_frac": t_star / (us_r * 1e-6)}
                tot, _ = timer.run(lambda: dec_run(st3, L, 0, all_vram=True), K, W)
                us_r = max_over_ranks(tot, world) / K * 1e3
                db_r = L * 2 * DEC_HKV * (DEC_D // 32) * 34
                results[f"q8_0_decode_L{L}_all_vram"] = {
                    "us_per_step": us_r, "hbm_gbs": db_r / (us_r * 1e-6) / 1e9,
                    "roofline_frac": db_r / (hbm * 1e9) / (us_r * 1e-6)}
        if "decsweep" in rows:
            # staged vs direct over the size of the host tail, at both VRAM splits
            for N in DEC_SWEEP_NS:
                for tail in DEC_SWEEP_TAILS:
                    L = N + tail
                    for staging in (False, True):
                        tot, _ = timer.run(lambda: dec_run(st3, L, N, staging=staging), K, W)
                        us_r = max_over_ranks(tot, world) / K * 1e3
                        hb_r, _ = dec_bytes(L, N)
                        results[f"decsweep_N{N}_tail{tail}_{'staged' if staging else 'direct'}"] = {
                            "us_per_step": us_r, "host_gbs": hb_r / (us_r * 1e-6) / 1e9}
        if "vmm" in rows:
            # the headline decode over one VMM range per plane (host-NUMA tail)
            vm = vmm_setup(st3)
            if "unavailable" in vm:
                results["q8_0_decode_L184320_N8192_vmm_tier"] = {"unavailable": vm["unavailable"]}
            else:
                try:
                    for staging in (False, True):
                        tot, _ = timer.run(lambda: vmm_run(st3, vm, staging), K, W)
                        VMM_RAN[0] = True
                        us_r = max_over_ranks(tot, world) / K * 1e3
                        hb_r, db_r = dec_bytes(184320, 8192)
                        if staging:
                            db_r += 2 * hb_r
                        t_star = max(hb_r / (peaks['h2d'] * 1e9), db_r / (hbm * 1e9))
                        results[f"q8_0_decode_L184320_N8192_vmm_tier_{'staged' if staging else 'direct'}"] = {
                            "us_per_step": us_r, "host_gbs": hb_r / (us_r * 1e-6) / 1e9,
                            "roofline_frac": t_star / (us_r * 1e-6)}
                finally:
                    vmm_free(vm)
        del st3
    if "decode_vram" in rows and "decode" not in rows:
        st3 = dec_setup()
        L = max(DEC_LS)
        tot, _ = timer.run(lambda: dec_run(st3, L, 0, all_vram=True), K, W)
        us_r = max_over_ranks(tot, world) / K * 1e3
        db_r = L * 2 * DEC_HKV * (DEC_D // 32) * 34
        results[f"q8_0_decode_L{L}_all_vram"] = {
            "us_per_step": us_r, "hbm_gbs": db_r / (us_r * 1e-6) / 1e9,
            "roofline_frac": db_r / (hbm * 1e9) / (us_r * 1e-6)}
        del st3
    # ---- tiny paged cache (latency-bound: microseconds, fractions not meaningful)
    if "tiny" in rows:
        st1 = tiny_setup()
        for h2d in (True, False):
            tot, _ = timer.run(lambda: swap_run(st1, h2d), K, W)
            us_r = max_over_ranks(tot, world) / K * 1e3
            results[f"tiny_swap_64blocks_{'h2d' if h2d else 'd2h'}"] = {
                "us_per_step": us_r, "host_gbs": st1["bytes"] / (us_r * 1e-6) / 1e9}
        for staging in (False, True):
            tot, _ = timer.run(lambda: tiny_decode(st1, staging), K, W)
            us_r = max_over_ranks(tot, world) / K * 1e3
            results[f"tiny_f16_decode_L1024_N512_{'staged' if staging else 'direct'}"] = {"us_per_step": us_r}
        del st1
    # ---- 32-layer offload swap
    if "swap" in rows:
        for page in (32768, 2048):
            st2 = swap_setup(page)
            sh = shard(st2["n_desc"])
            for h2d in (True, False):
                tot, _ = timer.run(lambda: swap_run(st2, h2d, shard=sh), K, W)
                us_r = max_over_ranks(tot, world) / K * 1e3
                # whole-job bytes: every rank's share (the whole list once when sharded)
                job_bytes = st2["bytes"] * (1 if args.split == "shards" else world)
                gbs = job_bytes / (us_r * 1e-6) / 1e9
                pk = peaks["h2d" if h2d else "d2h"] * world
                results[f"swap_{page // 1024}KiB_{'h2d' if h2d else 'd2h'}"] = {
                    "us_per_step": us_r, "host_gbs": gbs, "roofline_frac": gbs / pk,
                    "descriptors": st2["n_desc"], "mode": "sm",
                    "scaling": "strong" if args.split == "shards" and world > 1 else "weak"}
            del st2
            t.cuda.empty_cache()
    # ---- SM copies vs the copy engine over page sizes and descriptor counts
    if "swapsweep" in rows:
        for pk_kib in SWEEP_PAGES_KIB:
            st8 = swap_sweep_setup(pk_kib << 10)
            for n in SWEEP_COUNTS:
                for h2d in (True, False):
                    for ce in (False, True):
                        tot, _ = timer.run(lambda: swap_sweep_run(st8, h2d, n, ce), K, W)
                        us_r = max_over_ranks(tot, world) / K * 1e3
                        gbs = n * (pk_kib << 10) / (us_r * 1e-6) / 1e9
                        pk = peaks["h2d" if h2d else "d2h"]
                        results[f"swapsweep_{pk_kib}KiB_x{n}_{'h2d' if h2d else 'd2h'}_{'ce' if ce else 'sm'}"] = {
                            "us_per_step": us_r, "host_gbs": gbs, "roofline_frac": gbs / pk}
            del st8
            t.cuda.empty_cache()
    # ---- top-k gather + sparse decode
    if "topk" in rows:
        sh = shard(TOPK_S)
        st4 = topk_setup(shard=sh)
        # whole-job bytes: 8 sequences once when sharded, once per rank as replicas
        full_bytes = 2 * TOPK_S * TOPK_K * TOPK_BLK * TOPK_HKV * TOPK_D * 2
        job_bytes = full_bytes if args.split == "shards" else full_bytes * world
        scal = "strong" if args.split == "shards" and world > 1 else "weak"
        tot, _ = timer.run(lambda: topk_gather(st4), K, W)
        us_r = max_over_ranks(tot, world) / K * 1e3
        gbs = job_bytes / (us_r * 1e-6) / 1e9
        results["topk_gather_8seq_64blocks"] = {"us_per_step": us_r, "host_gbs": gbs,
                                                "roofline_frac": gbs / (peaks["h2d"] * world), "scaling": scal}
        topk_gather(st4)
        tot, _ = timer.run(lambda: topk_decode(st4), K, W)
        us_r = max_over_ranks(tot, world) / K * 1e3
        gbs = job_bytes / (us_r * 1e-6) / 1e9
        results["topk_sparse_decode_8x4096"] = {"us_per_step": us_r, "hbm_gbs": gbs,
                                                "roofline_frac": gbs / (hbm * world), "scaling": scal}
        del st4
    # ---- write path: appends into the host tail
    if "append" in rows:
        st6 = append_setup()
        for which, n_tok in (("q8", 1), ("q8", 2048), ("bf", 2048)):
            tot, _ = timer.run(lambda: append_run(st6, which, n_tok), K, W)
            us_r = max_over_ranks(tot, world) / K * 1e3
            host_b = 2 * n_tok * st6[which + "_rb"]
            gbs = host_b / (us_r * 1e-6) / 1e9
            results[f"append_{'q8_0' if which == 'q8' else 'bf16'}_{n_tok}tok_host"] = {
                "us_per_step": us_r, "host_gbs": gbs, "roofline_frac": gbs / peaks["d2h"],
                "host_bytes": host_b}
        del st6
    # ---- QSA sparse rows (staged through the arena vs direct)
    if "sparse" in rows:
        st7 = sr_setup()
        host_staged = 2 * st7["n_pages"] * st7["page_bytes"]
        host_direct = 2 * SR_R * SR_KPAD * SR_HKV * SR_D * 2
        fma = 2.0 * SR_R * SR_KPAD * SR_HQ * SR_D
        for staged in (True, False):
            steps = K if staged else max(1, min(K, 2))
            tot, _ = timer.run(lambda: sr_run(st7, staged), steps, min(W, 3))
            us_r = max_over_ranks(tot, world) / steps * 1e3
            hb = host_staged if staged else host_direct
            gbs = hb / (us_r * 1e-6) / 1e9
            t_star = max(hb / (peaks["h2d"] * 1e9), fma / FP32_FMA_PEAK)
            results[f"qsa_sparse_rows_R2048_K2080_{'staged' if staged else 'direct'}"] = {
                "us_per_step": us_r, "host_gbs": gbs, "roofline_frac": t_star / (us_r * 1e-6),
                "rows_per_s": SR_R / (us_r * 1e-6)}
        del st7
    # ---- tiered chunked prefill
    if "prefill" in rows or "pfsweep" in rows:
        st5 = pf_setup()
        fl = pf_flops()
        tail_b = (PF_L - PF_N) * st5["rb"] * 2
        bf16 = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))).get("bf16_tflops", 1932.2) \
            if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else 1900.0
        for staged in ((True, False) if "prefill" in rows else ()):
            steps = K if staged else max(1, min(K, 3))
            tot, _ = timer.run(lambda: pf_run(st5, staged), steps, min(W, 3))
            us_r = max_over_ranks(tot, world) / steps * 1e3
            tfs = fl / (us_r * 1e-6) / 1e12
            t_star = max(fl / (bf16 * 1e12), tail_b / (peaks["h2d"] * 1e9))
            results[f"prefill_R2048_L262144_N65536_{'staged' if staged else 'direct'}"] = {
                "us_per_step": us_r, "tflops": tfs, "tensor_frac": tfs / bf16,
                "roofline_frac": t_star / (us_r * 1e-6), "tokens_per_s": PF_R / (us_r * 1e-6)}
        if "pfsweep" in rows:
            # staged vs direct over the number of query rows: the direct kernel reads the host
            # tail once per query tile of each kv head, the staged call once per call
            for r in PF_SWEEP_ROWS:
                for staged in (True, False):
                    steps = K if staged else max(1, min(K, 3))
                    tot, _ = timer.run(lambda: pf_run_rows(st5, r, staged), steps, min(W, 3))
                    us_r = max_over_ranks(tot, world) / steps * 1e3
                    results[f"pfsweep_R{r}_{'staged' if staged else 'direct'}"] = {
                        "us_per_step": us_r, "host_gbs": tail_b / (us_r * 1e-6) / 1e9,
                        "tflops": pf_flops(r, PF_L - r) / (us_r * 1e-6) / 1e12}
        del st5
    clk = clocks.stop()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline()
    if rank == 0 and head is None:
        # a subset of rows without the headline (profiling runs)
        print(json.dumps({"metric": METRIC, "value": None, "unit": "us/step", "n_gpus": world,
                          "steps": K, "warmup": W, "rows": results, "clocks": clk}), flush=True)
    elif rank == 0:
        us = head["us"]
        achieved = head["host_bytes"] / (us * 1e-6) / 1e9
        line = {
            "metric": METRIC, "value": us, "unit": "us/step", "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": us / 1e3, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "q8_0 K/V x f16 q, f32 accumulate",
            "data": "synthetic (seeded)",
            "config": headline_config(),
            "host_gbs": achieved, "link_peak_gbs": peaks,
            "roofline": {"bound": "host_link", "achieved": achieved, "peak": peaks["h2d"], "unit": "GB/s",
                         "frac": achieved / peaks["h2d"], "traffic": profiled_traffic(),
                         "traffic_note": "dram__bytes_read+write of decode_split_kernel per launch (one ncu "
                                         "capture of this workload); host-link bytes are not DRAM traffic",
                         "peak_source": "pinned cudaMemcpyAsync H2D 1 GiB, best of 5, measured in this run",
                         "kernel": "decode_split_kernel + decode_combine_kernel (one C-ABI call)"},
            "e2e": {"value": head["e2e_us"], "unit": "us/step", "h2d_bytes_per_step": head["e2e_h2d"],
                    "d2h_bytes_per_step": head["e2e_d2h"]},
            "gpu_launches": gpu_launch_count(K, rows),
            "clocks": clk, "cpu_baseline": cpu, "rows": results,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def decode_source_sha256():
    """sha256 of the decode kernel source (the kernels the headline times)."""
    import hashlib
    h = hashlib.sha256()
    for name in ("decode_impl.cuh", "decode_dispatch.cuh", "decode.cu"):
        with open(os.path.join(ROOT, "host_ram_tiered_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


# DRAM bytes per launch of the headline decode kernel (dram__bytes_read.sum +
# dram__bytes_write.sum of decode_split_kernel, one ncu capture of the headline
# workload), with the sha256 of the decode kernel source it was taken on.
HEADLINE_TRAFFIC = {"bytes_per_launch": 18083072,
                    "decode_source_sha256": "949d0ded6b22820a885c80af5437208ec5d52bad15f8156a5fcdfabcb24dc1b1"}


def profiled_traffic():
    """The captured DRAM traffic of the headline decode kernel; None once the
    decode kernel source differs from the one the capture was taken on."""
    if HEADLINE_TRAFFIC["decode_source_sha256"] != decode_source_sha256():
        return None
    return HEADLINE_TRAFFIC["bytes_per_launch"]


def gpu_launch_count(K, rows):
    """Kernels of libkvo launched in the timed regions (own kernels only)."""
    n = 0
    if "decode" in rows or "head" in rows or "vmm" in rows or "decsweep" in rows:
        n += 2 * K * 2                             # headline decode + its e2e: split + combine
    if "vmm" in rows and VMM_RAN[0]:
        # the headline decode over VMM tiers, direct and staged
        n += 2 * K + K * k_launches_staged_headline()
    k = kvo()
    if "decode" in rows:
        # 11 tiered variants (a staged call runs the split kernel once per copy part) + 3
        # all-VRAM (split + combine)
        for L in DEC_LS:
            for N in DEC_NS:
                for staging in (False, True):
                    if not (L <= N and staging):
                        n += K * k.kvo_attn_decode_launches(1, L, DEC_D, N, staging)
            n += 2 * K
    elif "decode_vram" in rows:
        n += 2 * K                                 # the 184,320-cell all-VRAM decode
    if "decsweep" in rows:
        for N in DEC_SWEEP_NS:
            for tail in DEC_SWEEP_TAILS:
                n += K * sum(k.kvo_attn_decode_launches(1, N + tail, DEC_D, N, s) for s in (False, True))
    if "tiny" in rows:
        # swap both ways; decode direct + staged
        n += K * 2 + K * sum(k.kvo_attn_decode_launches(1, 1024, 128, 512, s) for s in (False, True))
    if "swap" in rows:
        n += K * 4                                 # 2 pages x 2 directions, one swap kernel each
    if "swapsweep" in rows:
        # SM mode: one swap kernel per row (page sizes x counts x directions); the copy-engine
        # rows launch no kernel
        n += K * len(SWEEP_PAGES_KIB) * len(SWEEP_COUNTS) * 2
    if "topk" in rows:
        n += K + 2 * K                             # gather; decode split + combine
    if "append" in rows:
        n += 3 * K                                 # three appends, one kernel each
    if "prefill" in rows:
        # staged: VRAM head (2 row blocks) + 48 arena buckets of 4096 cells x 2 row blocks;
        # direct: head + host tail, 2 row blocks each
        n += K * (2 + 48 * 2) + min(K, 3) * 4
    if "pfsweep" in rows:
        # one row block per call: staged = VRAM head + 48 buckets, direct = head + tail
        n += len(PF_SWEEP_ROWS) * (K * 49 + max(1, min(K, 3)) * 2)
    if "sparse" in rows:
        # staged: partition + buckets x (page gather + 2 row blocks x a split kernel that folds
        # its one chunk per row itself), the arena holding two slots of arena / (4 page_bytes)
        # pages; direct: 2 row blocks x (split + combine)
        page_bytes = SR_PS * SR_HKV * SR_D * 2
        slot = SR_ARENA // (4 * page_bytes)
        buckets = -(-(SR_L // SR_PS) // slot)
        n += K * (1 + buckets * (1 + 2)) + max(1, min(K, 2)) * 4
    return n


def cpu_baseline():
    """The fp64 oracle timed on this host's cores on the headline workload:
    whole steps (all 48 query heads over the 184,320 cells, parallel over
    heads), as many as fit in about 10 s."""
    import oracle
    oracle.build()
    threads = oracle.set_threads(os.cpu_count() or 1)
    step, keep = oracle_c3_step(max(DEC_LS), DEC_HQ)
    step()
    t0 = time.perf_counter()
    n = 0
    while time.perf_counter() - t0 < 10.0 and n < 20:
        step()
        n += 1
    dt = (time.perf_counter() - t0) / n
    out = {"value": dt * 1e6, "unit": "us/step", "cores": threads, "kind": "oracle",
           "sample": f"whole headline steps ({DEC_HQ} query heads x {max(DEC_LS)} cells), {n} steps after one "
                     f"untimed, no scaling"}
    out["rows"] = cpu_rows(threads)
    return out


def _timed(fn, budget_s=3.0, max_n=20, warm=True):
    if warm:
        fn()
    t0 = time.perf_counter()
    n = 0
    while n < 1 or (time.perf_counter() - t0 < budget_s and n < max_n):
        fn()
        n += 1
    return (time.perf_counter() - t0) / n


def _pool_run(pool, parts):
    """Run the callables in `parts` on the thread pool and wait (the oracle's
    ctypes calls release the GIL, so the parts run on separate cores)."""
    for f in [pool.submit(p) for p in parts]:
        f.result()


def _split(n, k):
    return [(n * i // k, n * (i + 1) // k) for i in range(k) if n * i // k < n * (i + 1) // k]


def cpu_rows(threads):
    """The oracle on bounded samples of the other rows, scaled to one step of
    each workload.  The swap and gather oracles are plain memcpy loops: each is
    timed on one thread and on `threads` threads that each take a contiguous
    range of descriptors (swap) or of sequences (gather).  The attention
    oracles run on `threads` cores."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    res = {}
    pool = ThreadPoolExecutor(threads)

    def swap_rows(name, page, nd, total):
        src = np.zeros(nd * page, np.uint8)
        dst = np.zeros(nd * page, np.uint8)
        perm = synth.rng(SEED0 + 1, 9).permutation(nd)
        s_ptr = (src.ctypes.data + perm.astype(np.uint64) * page).astype(np.uint64)
        d_ptr = (dst.ctypes.data + np.arange(nd, dtype=np.uint64) * page).astype(np.uint64)
        sizes = np.full(nd, page, np.int64)
        scale = total / nd
        sample = (f"{nd} of {total:,} descriptors, scaled x{scale:g}" if nd < total
                  else f"the full {total:,} descriptors")
        dt1 = _timed(lambda: oracle.swap_blocks(s_ptr, d_ptr, sizes))
        parts = [lambda a=a, b=b: oracle.swap_blocks(s_ptr[a:b], d_ptr[a:b], sizes[a:b])
                 for a, b in _split(nd, threads)]
        dtn = _timed(lambda: _pool_run(pool, parts))
        res[name] = {"value": dt1 * 1e6 * scale, "unit": "us/step", "sample": sample, "cores": 1,
                     "all_cores": {"value": dtn * 1e6 * scale, "cores": threads}}

    # C1: 4 tensors x 64 blocks of 32 KiB per direction (the whole step)
    swap_rows("tiny_swap_64blocks", 32768, 256, 256)
    # C2: 32 KiB pages, 4,096 of the 131,072 descriptors; 2 KiB pages, all of them
    swap_rows("swap_32KiB", 32768, 4096, 131072)
    swap_rows("swap_2KiB", 2048, 131072, 131072)
    # C1 decode: one sequence, 32 q / 8 kv heads x 128 fp16, 1,024 cells (512 in the head)
    g = synth.rng(SEED0, 10)
    kt = synth.normal_bits((1024, 8 * 128), "f16", g).view(np.uint8)
    vt = synth.normal_bits((1024, 8 * 128), "f16", g).view(np.uint8)
    qt = synth.normal_bits((1, 32, 128), "f16", g)
    kh, vh, ktl, vtl = (np.ascontiguousarray(x) for x in (kt[:512], vt[:512], kt[512:], vt[512:]))
    cache = oracle.make_cache(kh, vh, ktl, vtl, 512, 512, 512, oracle.F16, 8, 128)
    dt = _timed(lambda: oracle.attn_decode(cache, qt, oracle.F16, 1, 32, [1024], 1.0 / math.sqrt(128)))
    res["tiny_f16_decode_L1024_N512"] = {"value": dt * 1e6, "unit": "us/step", "sample": "full step",
                                         "cores": threads}
    # gather: 64 blocks of 64 tokens per (sequence, kv head), 8 x 4 x 128 bf16 planes of 65,536 tokens
    # (the same 64 MiB copied as the full 2^20-token planes)
    T = 65536
    plane = np.zeros((TOPK_S, T, TOPK_HKV, TOPK_D), np.uint16)
    sel = synth.topk_selection(TOPK_S, TOPK_HKV, T // 64, 64, synth.rng(SEED0 + 3, 9))
    dt1 = _timed(lambda: oracle.gather_blocks(plane, TOPK_S, T, TOPK_HKV, TOPK_D, 2, 64, sel))
    parts = [lambda a=a, b=b: oracle.gather_blocks(plane[a:b], b - a, T, TOPK_HKV, TOPK_D, 2, 64, sel[a:b])
             for a, b in _split(TOPK_S, min(threads, TOPK_S))]
    dtn = _timed(lambda: _pool_run(pool, parts))
    res["topk_gather_8seq_64blocks"] = {
        "value": dt1 * 1e6 * 2, "unit": "us/step", "cores": 1,
        "sample": "K plane only (x2 for K and V), 65,536-token planes, full selection",
        "all_cores": {"value": dtn * 1e6 * 2, "cores": min(threads, TOPK_S)}}
    del plane
    pool.shutdown()
    # sparse decode over the 4,096 gathered cells: full size
    g = synth.rng(SEED0 + 3, 10)
    cells = TOPK_S * 4096
    kb = synth.normal_bits((cells, TOPK_HKV * TOPK_D), "bf16", g).view(np.uint8)
    vb = synth.normal_bits((cells, TOPK_HKV * TOPK_D), "bf16", g).view(np.uint8)
    qb = synth.normal_bits((TOPK_S, TOPK_HQ, TOPK_D), "bf16", g)
    cache = oracle.make_cache(kb, vb, None, None, 4096, 0, 4096, oracle.BF16, TOPK_HKV, TOPK_D)
    dt = _timed(lambda: oracle.attn_decode(cache, qb, oracle.BF16, TOPK_S, TOPK_HQ, [4096] * TOPK_S,
                                           1.0 / math.sqrt(TOPK_D)))
    res["topk_sparse_decode_8x4096"] = {"value": dt * 1e6, "unit": "us/step", "sample": "full step", "cores": threads}
    del kb, vb
    # prefill: 2 of the 2,048 rows (all 32 heads) over the full 262,144 cells
    rb = PF_HKV * PF_D * 2
    kc = np.empty(PF_L * rb // 2, np.uint16)
    vc = np.empty(PF_L * rb // 2, np.uint16)
    synth.fill_normal_bits_large(kc, "bf16", SEED0 + 4, 11)
    synth.fill_normal_bits_large(vc, "bf16", SEED0 + 4, 12)
    q5 = synth.normal_bits((2, PF_HQ, PF_D), "bf16", synth.rng(SEED0 + 4, 13))
    cache = oracle.make_cache(kc.view(np.uint8), vc.view(np.uint8), None, None, PF_L, 0, PF_L, oracle.BF16,
                              PF_HKV, PF_D)
    dt = _timed(lambda: oracle.attn_prefill(cache, q5, oracle.BF16, 2, PF_POS0 + PF_R - 2, PF_HQ, PF_L,
                                            1.0 / math.sqrt(PF_D)), budget_s=0.0, max_n=1, warm=False)
    res["pf_prefill"] = {"value": dt * 1e6 * (PF_R / 2), "unit": "us/step",
                         "sample": "2 of 2,048 rows (the last positions, 64 tasks), one run, scaled x1024",
                         "cores": threads}
    del kc, vc
    return res


if __name__ == "__main__":
    sys.exit(main())
