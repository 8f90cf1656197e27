"""GPU tests of the VMM tier: a VRAM head and a host-NUMA tail in one device
virtual range (llama.cpp PR #319 "tiered KV cache (--kv-vram-cells): VRAM
head, pinned-host tail in one VMM range"), with the all-VRAM staging alias.
Decode and prefill read a tier through one base pointer; the results are the
bits of the two-buffer call and of an all-VRAM cache, and the oracle's within
the attention tolerance."""
import math

import numpy as np
import pytest

import oracle
from helpers import Tiered, cells, normwise_rel_err, run_decode, scale_for, torch
from host_ram_tiered_gb300 import kvo, synth

pytestmark = pytest.mark.gpu

REL_TOL = 2e-3
CHUNK = 1 << 16


def _tier(head, tail, stage=0):
    try:
        return kvo.kvo_vmm_tier_create(0, head, tail, stage)
    except kvo.KvoError as e:
        if e.status == -4:                                 # KVO_ERR_UNSUPPORTED
            pytest.skip(f"VMM tier not supported by this driver: {e}")
        raise


def _copy(dst_addr, src_addr, n, d2h=False):
    """n bytes src -> dst through the SM swap kernel (any device-accessible memory)."""
    t = torch()
    offs = np.arange(0, n, CHUNK, dtype=np.int64)
    sizes = np.minimum(CHUNK, n - offs).astype(np.int64)
    dev = lambda a: t.from_numpy(np.ascontiguousarray(a)).cuda()
    flags = (kvo.KVO_SWAP_D2H if d2h else kvo.KVO_SWAP_H2D) | kvo.KVO_SWAP_FORCE_SM
    kvo.kvo_swap_blocks_batch(dev(src_addr + offs), dev(dst_addr + offs), dev(sizes), len(offs), flags)
    t.cuda.synchronize()


def _decode(q, hq, hkv, d, kv_dt, k_vram, v_vram, k_host, v_host, L, N, scale, sk=None, sv=None):
    t = torch()
    out = t.empty(hq * d, dtype=t.float32, device="cuda")
    wsb = kvo.kvo_attn_decode_workspace_bytes(1, hq, d, L)
    ws = t.empty(max(wsb, 16), dtype=t.uint8, device="cuda")
    ctx = t.tensor([L], dtype=t.int32, device="cuda")
    qdt = kvo.BF16 if kv_dt == kvo.BF16 else kvo.F16
    kvo.kvo_attn_decode_tiered(q, qdt, 1, hq, hkv, d, k_vram, v_vram, L, k_host, v_host, L - N, kv_dt, ctx, L,
                               N, scale, sk, sv, out, ws, wsb)
    t.cuda.synchronize()
    return out.cpu().numpy().reshape(1, hq, d)


def test_bf16_tier_one_pointer_two_pointer_and_staged_alias_are_bit_identical():
    t = torch()
    gran = kvo.kvo_vmm_granularity(0)
    hq, hkv, d = 32, 8, 128
    rb = hkv * d * 2
    N = gran // rb                                         # head exactly one granule of rows
    L = N + 1500
    g = synth.rng(41, 1)
    k, v = cells(L, hkv, d, oracle.BF16, g)
    q_np = synth.normal_bits((1, hq, d), "bf16", g)
    q = t.from_numpy(q_np.view(np.int16).reshape(-1).copy()).cuda()
    s = scale_for(d)
    tk = _tier(N * rb, (L - N) * rb, (L - N) * rb)
    tv = _tier(N * rb, (L - N) * rb, (L - N) * rb)
    try:
        assert tk["head"] == N * rb and tk["alias"]
        kd, vd = t.from_numpy(k.reshape(-1).copy()).cuda(), t.from_numpy(v.reshape(-1).copy()).cuda()
        _copy(tk["base"], kd.data_ptr(), L * rb)
        _copy(tv["base"], vd.data_ptr(), L * rb)
        one = _decode(q, hq, hkv, d, kvo.BF16, tk["base"], tv["base"], None, None, L, N, s)
        two = _decode(q, hq, hkv, d, kvo.BF16, tk["base"], tv["base"], tk["base"] + N * rb, tv["base"] + N * rb,
                      L, N, s)
        stg = _decode(q, hq, hkv, d, kvo.BF16, tk["base"], tv["base"], None, None, L, N, s,
                      tk["alias"] + N * rb, tv["alias"] + N * rb)
        ref = run_decode(Tiered(k, v, L), q, kvo.BF16, hq, hkv, d, kvo.BF16, t.tensor([L], dtype=t.int32,
                                                                                      device="cuda"), s)
        for o in (one, two, stg):
            assert np.array_equal(o.view(np.uint32), ref.view(np.uint32))
        tc = Tiered(k, v, N)
        exp = oracle.attn_decode(tc.oracle_cache(oracle.BF16, hkv, d), q_np, oracle.BF16, 1, hq, [L], s)
        assert normwise_rel_err(one, exp) <= REL_TOL
    finally:
        kvo.kvo_vmm_tier_destroy(tk["tier"])
        kvo.kvo_vmm_tier_destroy(tv["tier"])


def test_q8_0_tier_boundary_inside_a_granule():
    # The head is rounded up to the granularity, so the cells from N to the
    # end of the VRAM granule lie in VRAM but are read as tail cells: the
    # tail range crosses from the head into the host memory.
    t = torch()
    hq, hkv, d = 48, 8, 128
    rb = hkv * (d // 32) * 34
    N, L = 3000, 5200
    g = synth.rng(41, 2)
    k, v = cells(L, hkv, d, oracle.Q8_0, g)
    q_np = synth.normal_bits((1, hq, d), "f16", g)
    q = t.from_numpy(q_np.view(np.int16).reshape(-1).copy()).cuda()
    s = scale_for(d)
    tk = _tier(N * rb, (L - N) * rb)
    tv = _tier(N * rb, (L - N) * rb)
    try:
        kd, vd = t.from_numpy(k.reshape(-1).copy()).cuda(), t.from_numpy(v.reshape(-1).copy()).cuda()
        _copy(tk["base"], kd.data_ptr(), L * rb)
        _copy(tv["base"], vd.data_ptr(), L * rb)
        one = _decode(q, hq, hkv, d, kvo.Q8_0, tk["base"], tv["base"], None, None, L, N, s)
        ref = run_decode(Tiered(k, v, L), q, kvo.F16, hq, hkv, d, kvo.Q8_0,
                         t.tensor([L], dtype=t.int32, device="cuda"), s)
        assert np.array_equal(one.view(np.uint32), ref.view(np.uint32))
        # a VRAM head claimed past the device granules reaches host memory: refused
        n_bad = tk["head"] // rb + 1
        with pytest.raises(kvo.KvoError) as e:
            _decode(q, hq, hkv, d, kvo.Q8_0, tk["base"], tv["base"], None, None, L, n_bad, s)
        assert e.value.status == -3                        # KVO_ERR_NOT_MAPPED
        # the CPU page copy cannot address a tier: refused before any access
        with pytest.raises(kvo.KvoError) as e:
            kvo.kvo_copy_pages_host(tk["base"] + tk["head"], tv["base"] + tv["head"], tk["base"] + tk["head"],
                                    tv["base"] + tv["head"], 16, rb, 0, 1, 16)
        assert e.value.status == -3
        # staging buffers in the host tail: refused (they must be device memory)
        with pytest.raises(kvo.KvoError) as e:
            _decode(q, hq, hkv, d, kvo.Q8_0, tk["base"], tv["base"], None, None, L, N, s,
                    tk["base"] + tk["head"], tv["base"] + tv["head"])
        assert e.value.status == -3
    finally:
        kvo.kvo_vmm_tier_destroy(tk["tier"])
        kvo.kvo_vmm_tier_destroy(tv["tier"])


def test_prefill_and_append_over_a_tier():
    # The append path writes the cache into the tier (head rows to VRAM, the
    # rest to the host tail); the bytes read back are the source's, and the
    # prefill over the tier (one pointer, direct and through an arena) gives
    # the two-pointer bits and the oracle's values.
    t = torch()
    hq, hkv, d = 16, 4, 128
    rb = hkv * d * 2
    N, L, R = 700, 1900, 96
    g = synth.rng(41, 3)
    k, v = cells(L, hkv, d, oracle.BF16, g)
    q_np = synth.normal_bits((R, hq, d), "bf16", g)
    q = t.from_numpy(q_np.view(np.int16).reshape(-1).copy()).cuda()
    s = 1 / math.sqrt(d)
    tk = _tier(N * rb, (L - N) * rb)
    tv = _tier(N * rb, (L - N) * rb)
    try:
        kd, vd = t.from_numpy(k.reshape(-1).copy()).cuda(), t.from_numpy(v.reshape(-1).copy()).cuda()
        kvo.kvo_append_kv_tiered(kd, vd, kvo.BF16, L, 0, hkv, d, tk["base"], tv["base"], tk["base"] + N * rb,
                                 tv["base"] + N * rb, kvo.BF16, N, L)
        t.cuda.synchronize()
        back = t.empty(L * rb, dtype=t.uint8, device="cuda")
        _copy(back.data_ptr(), tk["base"], L * rb, d2h=True)
        assert np.array_equal(back.cpu().numpy(), k.reshape(-1))

        def prefill(k_host, v_host, arena_cells):
            out = t.full((R * hq * d,), float("nan"), dtype=t.float32, device="cuda")
            wsb = kvo.kvo_attn_prefill_workspace_bytes(R, hq)
            ws = t.empty(wsb, dtype=t.uint8, device="cuda")
            ab = 2 * arena_cells * rb
            arena = t.empty(ab, dtype=t.uint8, device="cuda") if arena_cells else None
            kvo.kvo_attn_prefill_tiered(q, R, L - R, hq, hkv, d, tk["base"], tv["base"], k_host, v_host, kvo.BF16,
                                        L, N, s, arena, ab, 48, out, ws, wsb)
            t.cuda.synchronize()
            return out.cpu().numpy().reshape(R, hq, d)

        one = prefill(None, None, 0)
        two = prefill(tk["base"] + N * rb, tv["base"] + N * rb, 0)
        staged = prefill(None, None, 256)
        assert np.array_equal(one.view(np.uint32), two.view(np.uint32))
        tc = Tiered(k, v, N)
        exp = oracle.attn_prefill(tc.oracle_cache(oracle.BF16, hkv, d), q_np, oracle.BF16, R, L - R, hq, L, s)
        assert normwise_rel_err(one, exp) <= REL_TOL
        assert normwise_rel_err(staged, exp) <= REL_TOL
    finally:
        kvo.kvo_vmm_tier_destroy(tk["tier"])
        kvo.kvo_vmm_tier_destroy(tv["tier"])
