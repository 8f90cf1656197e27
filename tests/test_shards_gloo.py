"""Multi-GPU split of the path, checked on CPU with two gloo ranks: each rank
takes its kvo_shard_range share of the work units (swap descriptors, gather
sequences, decode sequences), computes it (the oracle stands in for the
kernels here), and the ranks' results put together equal the one-rank result.
The path has no exchange step: the only collective is the test's own
all-gather of the results."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

WORLD = 2


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _problems():
    """The same seeded inputs on every rank."""
    from host_ram_tiered_gb300 import synth
    g = synth.rng(777)
    # gather: 5 sequences x 2 kv heads, planes of 512 tokens x 64 dims (bf16 bits), 6 of 8 blocks
    S, T, H, D, blk, k = 5, 512, 2, 64, 64, 6
    plane = synth.normal_bits((S, T, H, D), "bf16", g)
    sel = synth.topk_selection(S, H, T // blk, k, g)
    # swap: 37 descriptors of ragged sizes from a source pool into disjoint destination slots
    n = 37
    sizes = g.integers(1, 300, size=n).astype(np.int64)
    src_pool = g.integers(0, 256, size=64 * 512, dtype=np.uint8)
    slot = g.permutation(64)[:n]
    src_off = (g.permutation(64)[:n] * 512).astype(np.int64)
    dst_off = (slot * 512).astype(np.int64)
    dst_init = g.integers(0, 256, size=64 * 512, dtype=np.uint8)
    # decode: 5 sequences, 4 q / 2 kv heads x 64, fp16 cells, ragged lengths
    B, L, hq, hkv = 5, 300, 4, 2
    kc = synth.normal_bits((B * L, hkv * D), "f16", g).view(np.uint8)
    vc = synth.normal_bits((B * L, hkv * D), "f16", g).view(np.uint8)
    q = synth.normal_bits((B, hq, D), "f16", g)
    lens = [300, 1, 157, 299, 64]
    return dict(S=S, T=T, H=H, D=D, blk=blk, k=k, plane=plane, sel=sel, n=n, sizes=sizes,
                src_pool=src_pool, src_off=src_off, dst_off=dst_off, dst_init=dst_init,
                B=B, L=L, hq=hq, hkv=hkv, kc=kc, vc=vc, q=q, lens=lens)


def _gather(p, lo, hi):
    import oracle
    return oracle.gather_blocks(np.ascontiguousarray(p["plane"][lo:hi]), hi - lo, p["T"], p["H"], p["D"], 2,
                                p["blk"], p["sel"][lo:hi])


def _swap(p, lo, hi):
    import oracle
    dst = p["dst_init"].copy()
    src = (p["src_off"][lo:hi].astype(np.uint64) + np.uint64(p["src_pool"].ctypes.data))
    dd = (p["dst_off"][lo:hi].astype(np.uint64) + np.uint64(dst.ctypes.data))
    oracle.swap_blocks(src, dd, p["sizes"][lo:hi])
    return dst


def _decode(p, lo, hi):
    import oracle
    if hi == lo:
        return np.zeros((0, p["hq"], p["D"]))
    L, rb = p["L"], p["kc"].shape[1]
    kc = np.ascontiguousarray(p["kc"].reshape(p["B"], L, rb)[lo:hi]).reshape(-1, rb)
    vc = np.ascontiguousarray(p["vc"].reshape(p["B"], L, rb)[lo:hi]).reshape(-1, rb)
    c = oracle.make_cache(kc, vc, None, None, L, 0, L, oracle.F16, p["hkv"], p["D"])
    return oracle.attn_decode(c, p["q"][lo:hi], oracle.F16, hi - lo, p["hq"], p["lens"][lo:hi],
                              1 / np.sqrt(p["D"]))


def _worker(rank, port, out):
    import torch.distributed as dist

    from host_ram_tiered_gb300 import kvo
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    p = _problems()
    res = {}
    for name, n_units, fn in (("gather", p["S"], _gather), ("swap", p["n"], _swap),
                              ("decode", p["B"], _decode)):
        lo, hi = kvo.kvo_shard_range(n_units, WORLD, rank)
        parts = [None] * WORLD
        dist.all_gather_object(parts, (lo, hi, fn(p, lo, hi)))
        res[name] = parts
    if rank == 0:
        out["res"] = res
    dist.destroy_process_group()


def test_two_rank_shards_reassemble_the_one_rank_result(kvo_lib):
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, out)) for r in range(WORLD)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    res = out["res"]
    p = _problems()
    for name, n_units in (("gather", p["S"]), ("swap", p["n"]), ("decode", p["B"])):
        ranges = [(lo, hi) for lo, hi, _ in res[name]]
        # disjoint, complete, in rank order: every unit exactly once
        assert ranges[0][0] == 0 and ranges[-1][1] == n_units
        assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
        assert all(hi > lo for lo, hi in ranges)
    # gather and decode: the per-rank outputs concatenate to the one-rank output
    g_parts = [r for _, _, r in res["gather"]]
    assert np.array_equal(np.concatenate(g_parts), _gather(p, 0, p["S"]))
    d_parts = [r for _, _, r in res["decode"]]
    assert np.array_equal(np.concatenate(d_parts), _decode(p, 0, p["B"]))
    # swap: each destination slot comes from the rank that owns its descriptor; bytes that
    # no descriptor targets are unchanged on every rank
    whole = _swap(p, 0, p["n"])
    merged = p["dst_init"].copy()
    for lo, hi, dst in res["swap"]:
        for i in range(lo, hi):
            a = int(p["dst_off"][i])
            merged[a:a + int(p["sizes"][i])] = dst[a:a + int(p["sizes"][i])]
        touched = np.zeros(dst.size, bool)
        for i in range(lo, hi):
            touched[int(p["dst_off"][i]):int(p["dst_off"][i]) + int(p["sizes"][i])] = True
        assert np.array_equal(dst[~touched], p["dst_init"][~touched])
    assert np.array_equal(merged, whole)
