"""GPU parity of kvo_gather_blocks against the oracle's memcpy gather:
bit-exact, at a small ragged shape and at the full 8 x 2^20-token planes."""
import numpy as np
import pytest

import oracle
from helpers import pinned, to_pinned, torch
from host_ram_tiered_gb300 import kvo, synth

pytestmark = pytest.mark.gpu


def _gather(kp, vp, S, T, H, D, dt, blk, sel_np, k):
    t = torch()
    sel = t.from_numpy(np.ascontiguousarray(sel_np, np.int32).reshape(-1).copy()).cuda()
    n_out = S * k * blk * H * D * 2
    ko = t.full((n_out,), 7, dtype=t.uint8, device="cuda")
    vo = t.full((n_out,), 7, dtype=t.uint8, device="cuda")
    kvo.kvo_gather_blocks(kp, vp, S, T, H, D, dt, blk, sel, k, ko, vo)
    t.cuda.synchronize()
    return ko.cpu().numpy(), vo.cpu().numpy()


@pytest.mark.parametrize("S,T,H,D,blk,k,dt", [(3, 64 * 37, 4, 128, 64, 9, kvo.BF16),
                                               (2, 16 * 50, 2, 64, 16, 5, kvo.F16),
                                               (1, 64 * 3, 1, 128, 64, 3, kvo.BF16)])
def test_gather_matches_oracle(S, T, H, D, blk, k, dt):
    g = synth.rng(1237, S * 100 + k)
    name = "bf16" if dt == kvo.BF16 else "f16"
    kpl = synth.normal_bits((S, T, H, D), name, g)
    vpl = synth.normal_bits((S, T, H, D), name, g)
    sel = synth.topk_selection(S, H, T // blk, k, g)
    ko, vo = _gather(to_pinned(kpl), to_pinned(vpl), S, T, H, D, dt, blk, sel, k)
    assert np.array_equal(ko, oracle.gather_blocks(kpl, S, T, H, D, 2, blk, sel))
    assert np.array_equal(vo, oracle.gather_blocks(vpl, S, T, H, D, 2, blk, sel))
    assert kvo.kvo_device_errors() == 0


def test_gather_from_device_planes_too():
    t = torch()
    g = synth.rng(5)
    S, T, H, D, blk, k = 2, 64 * 10, 4, 128, 64, 4
    kpl = synth.normal_bits((S, T, H, D), "bf16", g)
    sel = synth.topk_selection(S, H, T // blk, k, g)
    kd = t.from_numpy(kpl.view(np.int16).reshape(-1).copy()).cuda()
    ko, vo = _gather(kd, kd, S, T, H, D, kvo.BF16, blk, sel, k)
    assert np.array_equal(ko, oracle.gather_blocks(kpl, S, T, H, D, 2, blk, sel))


def test_out_of_range_selection_is_skipped_and_flagged():
    g = synth.rng(6)
    S, T, H, D, blk, k = 1, 64 * 8, 2, 128, 64, 3
    kpl = synth.normal_bits((S, T, H, D), "bf16", g)
    sel = np.array([[[0, 3, 7], [1, 8, 2]]], np.int32)         # 8 is past the plane's last block
    kvo.kvo_device_errors(clear=True)
    ko, _ = _gather(to_pinned(kpl), to_pinned(kpl), S, T, H, D, kvo.BF16, blk, sel, k)
    assert kvo.kvo_device_errors(clear=True) & 1
    out = ko.view(np.uint16).reshape(S, k * blk, H, D)
    assert (ko.reshape(S, k * blk, H, D * 2)[0, blk:2 * blk, 1] == 7).all()   # skipped item untouched
    good = sel.copy()
    good[0, 1, 1] = 4
    exp = oracle.gather_blocks(kpl, S, T, H, D, 2, blk, good).view(np.uint16).reshape(S, k * blk, H, D)
    assert np.array_equal(out[:, :, 0], exp[:, :, 0])
    assert np.array_equal(out[0, :blk, 1], exp[0, :blk, 1])
    assert np.array_equal(out[0, 2 * blk:, 1], exp[0, 2 * blk:, 1])


def test_gather_rejects_pageable_and_q8_0():
    t = torch()
    plane = np.zeros(64 * 128, np.uint16)
    o = t.zeros(64 * 128 * 2, dtype=t.uint8, device="cuda")
    sel = t.zeros(1, dtype=t.int32, device="cuda")
    with pytest.raises(kvo.KvoError) as e:
        kvo.kvo_gather_blocks(plane.ctypes.data, plane.ctypes.data, 1, 64, 1, 128, kvo.BF16, 64, sel, 1, o, o)
    assert e.value.status == -3
    with pytest.raises(kvo.KvoError) as e:
        kvo.kvo_gather_blocks(o, o, 1, 64, 1, 128, kvo.Q8_0, 64, sel, 1, o, o)
    assert e.value.status == -4


def test_c4_full_size_gather_bit_exact():
    # 8 sequences x 2^20 tokens x 4 kv heads x 128 bf16 planes (8 GiB each) in
    # pinned host memory; 64 blocks of 64 tokens per (sequence, kv head).
    from bench import TOPK_BLK, TOPK_D, TOPK_HKV, TOPK_K, TOPK_S, TOPK_T, topk_gather, topk_setup
    st = topk_setup()
    topk_gather(st)
    torch().cuda.synchronize()
    kp = st["k_plane"].numpy()
    vp = st["v_plane"].numpy()
    exp_k = oracle.gather_blocks(kp, TOPK_S, TOPK_T, TOPK_HKV, TOPK_D, 2, TOPK_BLK, st["sel_np"])
    exp_v = oracle.gather_blocks(vp, TOPK_S, TOPK_T, TOPK_HKV, TOPK_D, 2, TOPK_BLK, st["sel_np"])
    assert np.array_equal(st["kg"].cpu().numpy(), exp_k)
    assert np.array_equal(st["vg"].cpu().numpy(), exp_v)
    assert kvo.kvo_device_errors() == 0
