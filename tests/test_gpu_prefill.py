"""GPU parity of kvo_attn_prefill_tiered (causal chunked prefill over a
tiered cache, staged through an arena or read directly) against the fp64
oracle: normwise relative error <= 2e-3 per (row, head)."""
import math

import numpy as np
import pytest

import oracle
from helpers import Tiered, cells, normwise_rel_err, torch
from host_ram_tiered_gb300 import kvo, synth

pytestmark = pytest.mark.gpu

REL_TOL = 2e-3


def _prefill(tc, q_np, rows, pos0, hq, hkv, d, dt, ctx_len, scale, arena_cells, rpl):
    t = torch()
    q = t.from_numpy(q_np.view(np.int16).reshape(-1).copy()).cuda()
    out = t.full((rows * hq * d,), float("nan"), dtype=t.float32, device="cuda")
    wsb = kvo.kvo_attn_prefill_workspace_bytes(rows, hq)
    ws = t.empty(wsb, dtype=t.uint8, device="cuda")
    arena = None
    ab = 0
    if arena_cells:
        ab = 2 * arena_cells * tc.rb + 48                 # not a multiple of a row pair: rounds down
        arena = t.empty(ab, dtype=t.uint8, device="cuda")
    kvo.kvo_attn_prefill_tiered(q, rows, pos0, hq, hkv, d, tc.k_head, tc.v_head, tc.k_tail,
                                tc.v_tail, dt, ctx_len, tc.n, scale, arena, ab, rpl, out, ws, wsb)
    t.cuda.synchronize()
    return out.cpu().numpy().reshape(rows, hq, d)


def _ref(tc, q_np, rows, pos0, hq, hkv, d, odt, ctx_len, scale):
    return oracle.attn_prefill(tc.oracle_cache(odt, hkv, d), q_np, odt, rows, pos0, hq, ctx_len, scale)


@pytest.mark.parametrize("arena_cells,rpl", [(128, 48), (0, 100), (1000, 0), (64, 7)])
def test_prefill_staged_and_direct_match_oracle(arena_cells, rpl):
    g = synth.rng(1238, arena_cells + rpl)
    R, pos0, L, N, hq, hkv, d = 100, 900, 1000, 300, 8, 2, 128
    k, v = cells(L, hkv, d, oracle.BF16, g)
    q = synth.normal_bits((R, hq, d), "bf16", g)
    tc = Tiered(k, v, N)
    s = 1 / math.sqrt(d)
    out = _prefill(tc, q, R, pos0, hq, hkv, d, kvo.BF16, L, s, arena_cells, rpl)
    ref = _ref(tc, q, R, pos0, hq, hkv, d, oracle.BF16, L, s)
    assert normwise_rel_err(out, ref) <= REL_TOL


@pytest.mark.parametrize("hq,hkv,dt", [(4, 4, oracle.F16), (16, 8, oracle.BF16), (16, 2, oracle.F16)])
def test_group_sizes(hq, hkv, dt):
    g = synth.rng(11, hq * 10 + hkv)
    R, pos0, L, N, d = 77, 400, 477, 123, 128
    k, v = cells(L, hkv, d, dt, g)
    q = synth.normal_bits((R, hq, d), "f16" if dt == oracle.F16 else "bf16", g)
    tc = Tiered(k, v, N)
    out = _prefill(tc, q, R, pos0, hq, hkv, d, dt, L, 0.09, 96, 40)
    ref = _ref(tc, q, R, pos0, hq, hkv, d, dt, L, 0.09)
    assert normwise_rel_err(out, ref) <= REL_TOL


@pytest.mark.parametrize("N", [0, 999, 5000])
def test_all_host_all_vram_and_rows_past_the_context(N):
    g = synth.rng(12, N)
    R, pos0, L, hq, hkv, d = 64, 980, 1000, 8, 2, 128     # rows 20.. see only cells < 1000
    k, v = cells(L, hkv, d, oracle.BF16, g)
    q = synth.normal_bits((R, hq, d), "bf16", g)
    tc = Tiered(k, v, N)
    out_s = _prefill(tc, q, R, pos0, hq, hkv, d, kvo.BF16, L, 0.1, 200, 32)
    out_d = _prefill(tc, q, R, pos0, hq, hkv, d, kvo.BF16, L, 0.1, 0, 32)
    ref = _ref(tc, q, R, pos0, hq, hkv, d, oracle.BF16, L, 0.1)
    assert normwise_rel_err(out_s, ref) <= REL_TOL
    assert normwise_rel_err(out_d, ref) <= REL_TOL


def test_first_row_sees_one_cell():
    g = synth.rng(13)
    R, L, hq, hkv, d = 40, 40, 4, 2, 128                  # a prefill from position 0
    k, v = cells(L, hkv, d, oracle.BF16, g)
    q = synth.normal_bits((R, hq, d), "bf16", g)
    tc = Tiered(k, v, 16)
    out = _prefill(tc, q, R, 0, hq, hkv, d, kvo.BF16, L, 0.1, 8, 16)
    ref = _ref(tc, q, R, 0, hq, hkv, d, oracle.BF16, L, 0.1)
    assert normwise_rel_err(out, ref) <= REL_TOL


@pytest.mark.parametrize("hq,hkv,dt,R", [(8, 2, oracle.BF16, 160), (16, 2, oracle.F16, 80),
                                          (4, 4, oracle.BF16, 520)])
def test_direct_tensor_core_path_over_host_rows(hq, hkv, dt, R):
    # rows x group >= 512: the host tail is read in place by the tensor-core kernel's producer
    # warp (plain loads into the swizzled tiles); a ragged last tile and rows whose causal range
    # ends inside the tail
    G = hq // hkv
    assert R * G >= 512
    g = synth.rng(1240, hq * 1000 + R)
    L, N, d = 1100, 300, 128
    pos0 = L - R - 7                                    # the last 7 cells lie past every row
    tc = Tiered(*cells(L, hkv, d, dt, g), N)
    q = synth.normal_bits((R, hq, d), "f16" if dt == oracle.F16 else "bf16", g)
    out = _prefill(tc, q, R, pos0, hq, hkv, d, dt, L, 0.09, 0, R)
    ref = _ref(tc, q, R, pos0, hq, hkv, d, dt, L, 0.09)
    assert normwise_rel_err(out, ref) <= REL_TOL


@pytest.mark.parametrize("arena_cells", [256, 0])
def test_bf16_value_beyond_fp16_range_sets_bit_4(arena_cells):
    # The PV product takes the weights and the V values of a bf16 cache as fp16: a cached V value
    # of 65536 cannot be held and must be reported (staged: V tiles by TMA from the arena;
    # direct, rows x group >= 512: V tiles loaded from host memory by the producer warp)
    g = synth.rng(1241, arena_cells)
    R, pos0, L, N, hq, hkv, d = 128, 900, 1000, 600, 8, 2, 128
    k, v = cells(L, hkv, d, oracle.BF16, g)
    q = synth.normal_bits((R, hq, d), "bf16", g)
    kvo.kvo_device_errors(clear=True)
    _prefill(Tiered(k, v, N), q, R, pos0, hq, hkv, d, kvo.BF16, L, 0.1, arena_cells, R)
    assert kvo.kvo_device_errors(clear=True) & 16 == 0
    v_big = v.copy()
    v_big[700, 2 * d + 6: 2 * d + 8] = (0x80, 0x47)    # cell 700 (host tail), kv head 1, dim 3: 65536
    _prefill(Tiered(k, v_big, N), q, R, pos0, hq, hkv, d, kvo.BF16, L, 0.1, arena_cells, R)
    assert kvo.kvo_device_errors(clear=True) & 16


def test_prefill_argument_errors():
    t = torch()
    x = t.zeros(1 << 16, dtype=t.uint8, device="cuda")
    o = t.zeros(1 << 16, dtype=t.float32, device="cuda")
    for dt, d, st in ((kvo.Q8_0, 128, -4), (kvo.BF16, 64, -4)):
        with pytest.raises(kvo.KvoError) as e:
            kvo.kvo_attn_prefill_tiered(x, 4, 0, 4, 2, d, x, x, None, None, dt, 4, 4, 0.1, None, 0, 0,
                                        o, x, 1 << 16)
        assert e.value.status == st
    with pytest.raises(kvo.KvoError) as e:
        kvo.kvo_attn_prefill_tiered(x, 4, 0, 4, 2, 128, x, x, None, None, kvo.BF16, 4, 4, 0.1, None,
                                    0, 0, o, x, 8)
    assert e.value.status == -6


@pytest.mark.parametrize("staged", [True, False])
def test_c5_full_size_sampled_rows(staged):
    # 2048 rows at positions 260,096..262,143 over 262,144 bf16 cells, 32/8 heads,
    # N = 65,536, 32 MiB arena, 1024 rows per launch -- the benchmark's launch.
    from bench import (PF_D, PF_HKV, PF_HQ, PF_L, PF_N, PF_POS0, PF_R, pf_run, pf_setup)
    st = pf_setup()
    pf_run(st, staged=staged)
    torch().cuda.synchronize()
    out = st["out"].cpu().numpy().reshape(PF_R, PF_HQ, PF_D)
    rb = st["rb"]
    kh = st["k_head_np"].view(np.uint8).reshape(PF_N, rb)
    vh = st["v_head_np"].view(np.uint8).reshape(PF_N, rb)
    kt = st["k_host"].numpy().reshape(PF_L - PF_N, rb)
    vt = st["v_host"].numpy().reshape(PF_L - PF_N, rb)
    cache = oracle.make_cache(kh, vh, kt, vt, PF_N, PF_L - PF_N, PF_N, oracle.BF16, PF_HKV, PF_D)
    g = synth.rng(77, int(staged))
    rows = sorted(set([0, 1, 1023, 1024, 2046, 2047] + g.choice(PF_R, 10, replace=False).tolist()))
    for i in rows:
        ref = oracle.attn_prefill(cache, st["q_np"][i:i + 1], oracle.BF16, 1, PF_POS0 + i, PF_HQ,
                                  PF_L, 1.0 / math.sqrt(PF_D))
        assert normwise_rel_err(out[i:i + 1], ref) <= REL_TOL, i
