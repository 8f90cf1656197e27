"""GPU parity of kvo_attn_sparse_rows (QSA sparse rows over a paged host
cache, ExLlamaV3 patch "QSA KV cache host-RAM offload") against the fp64
oracle: direct, staged in one bucket and in many, with padding, empty rows
and a bad page-table entry; plus the host-side page copy."""
import math

import numpy as np
import pytest

import oracle
from helpers import normwise_rel_err, pinned, to_pinned, torch
from host_ram_tiered_gb300 import kvo, synth

pytestmark = pytest.mark.gpu

REL_TOL = 2e-3


def _planes(n_pages, ps, hkv, d, name, g):
    k = synth.normal_bits((n_pages, ps, hkv, d), name, g)
    v = synth.normal_bits((n_pages, ps, hkv, d), name, g)
    return k, v


def _run(q_dev, dt, rows, hq, hkv, d, kp, vp, ps, n_pages, bt_dev, npu, idx_dev, k_pad, scale,
         arena_pages=0, rows_per_launch=1 << 20):
    t = torch()
    page_bytes = ps * hkv * d * 2
    arena_bytes = 2 * arena_pages * page_bytes
    arena = t.empty(max(arena_bytes, 16), dtype=t.uint8, device="cuda") if arena_pages else None
    wsb = kvo.kvo_attn_sparse_rows_workspace_bytes(rows, hq, hkv, d, k_pad, rows_per_launch, ps, npu,
                                                   arena_bytes)
    ws = t.empty(max(wsb, 16), dtype=t.uint8, device="cuda")
    out = t.full((rows * hq * d,), float("nan"), dtype=t.float32, device="cuda")
    kvo.kvo_attn_sparse_rows(q_dev, dt, rows, hq, hkv, d, kp, vp, dt, ps, n_pages, bt_dev, npu, idx_dev,
                             k_pad, scale, arena, arena_bytes, rows_per_launch, out, ws, wsb)
    t.cuda.synchronize()
    return out.cpu().numpy().reshape(rows, hq, d)


@pytest.mark.parametrize("dt,hq,hkv,d,rows", [(kvo.F16, 8, 2, 128, 200), (kvo.BF16, 16, 4, 64, 37),
                                               (kvo.F16, 6, 1, 128, 170)])
def test_sparse_rows_direct_and_staged_match_oracle(dt, hq, hkv, d, rows):
    t = torch()
    g = synth.rng(1301, hq * 1000 + rows)
    name = "bf16" if dt == kvo.BF16 else "f16"
    n_pages, ps, npu, k_pad = 48, 16, 40, 96
    k, v = _planes(n_pages, ps, hkv, d, name, g)
    kp, vp = to_pinned(k), to_pinned(v)
    bt = g.permutation(n_pages).astype(np.int32)[:npu].copy()
    idx = synth.row_selections(rows, k_pad, npu * ps - rows - 8, 80, g, pad_frac=0.15)
    idx[3, 10:20] = npu * ps + 5                            # past the pages in use: padding
    idx[0, :] = -1                                          # a row with nothing selected
    q = synth.normal_bits((rows, hq, d), name, g)
    scale = 1 / math.sqrt(d)
    ref = oracle.attn_sparse_rows(k, v, dt, ps, hkv, d, bt, npu, idx, q, dt, hq, scale)
    q_dev = t.from_numpy(q.view(np.int16).reshape(-1).copy()).cuda()
    bt_dev = t.from_numpy(bt).cuda()
    idx_dev = t.from_numpy(idx.reshape(-1).copy()).cuda()
    runs = {"direct": _run(q_dev, dt, rows, hq, hkv, d, kp, vp, ps, n_pages, bt_dev, npu, idx_dev, k_pad,
                           scale),
            # arena of 2 * arena_pages pages: two slots of arena_pages / 2 pages each when that is >= 1
            "one_bucket": _run(q_dev, dt, rows, hq, hkv, d, kp, vp, ps, n_pages, bt_dev, npu, idx_dev, k_pad,
                               scale, arena_pages=2 * npu),
            "two_slots_20_buckets": _run(q_dev, dt, rows, hq, hkv, d, kp, vp, ps, n_pages, bt_dev, npu, idx_dev,
                                         k_pad, scale, arena_pages=5, rows_per_launch=64),
            "one_slot_40_buckets": _run(q_dev, dt, rows, hq, hkv, d, kp, vp, ps, n_pages, bt_dev, npu, idx_dev,
                                        k_pad, scale, arena_pages=1)}
    for name_, out in runs.items():
        assert np.all(out[0] == 0.0), name_
        assert normwise_rel_err(out[1:], ref[1:]) <= REL_TOL, name_


def test_sparse_rows_single_pick_gives_v_and_bad_page_is_flagged():
    t = torch()
    g = synth.rng(1302)
    hq, hkv, d, n_pages, ps, npu, k_pad, rows = 4, 1, 128, 6, 32, 6, 64, 3
    k, v = _planes(n_pages, ps, hkv, d, "f16", g)
    kp, vp = to_pinned(k), to_pinned(v)
    bt = np.arange(n_pages, dtype=np.int32)[::-1].copy()
    idx = np.full((rows, k_pad), -1, np.int32)
    idx[0, 7] = 77                                          # one pick: out = v of position 77
    idx[1, :40] = np.arange(40)
    idx[2, :40] = np.arange(40) + 150
    q = synth.normal_bits((rows, hq, d), "f16", g)
    q_dev = t.from_numpy(q.view(np.int16).reshape(-1).copy()).cuda()
    idx_dev = t.from_numpy(idx.reshape(-1).copy()).cuda()
    kvo.kvo_device_errors(clear=True)
    out = _run(q_dev, kvo.F16, rows, hq, hkv, d, kp, vp, ps, n_pages, t.from_numpy(bt).cuda(), npu, idx_dev,
               k_pad, 0.1)
    v77 = v[bt[77 // ps], 77 % ps, 0].view(np.float16).astype(np.float32)
    for h in range(hq):
        assert np.array_equal(out[0, h], v77)
    assert kvo.kvo_device_errors(clear=True) == 0
    bad = bt.copy()
    bad[4] = n_pages + 3                                    # page 4 holds positions 128..159
    out2 = _run(q_dev, kvo.F16, rows, hq, hkv, d, kp, vp, ps, n_pages, t.from_numpy(bad).cuda(), npu, idx_dev,
                k_pad, 0.1)
    assert kvo.kvo_device_errors(clear=True) & 2
    assert np.all(np.isfinite(out2))
    ref = oracle.attn_sparse_rows(k, v, kvo.F16, ps, hkv, d, bt, npu, idx, q, kvo.F16, hq, 0.1)
    assert normwise_rel_err(out2[:2], ref[:2]) <= REL_TOL    # rows that never touch page 4


def test_sparse_rows_argument_errors():
    t = torch()
    hq, hkv, d, n_pages, ps, npu, k_pad, rows = 4, 1, 128, 4, 16, 4, 32, 2
    kp = pinned(n_pages * ps * hkv * d * 2)
    vp = pinned(n_pages * ps * hkv * d * 2)
    q = t.zeros(rows * hq * d, dtype=t.int16, device="cuda")
    idx = t.zeros(rows * k_pad, dtype=t.int32, device="cuda")
    bt = t.arange(n_pages, dtype=t.int32, device="cuda")
    out = t.empty(rows * hq * d, dtype=t.float32, device="cuda")
    wsb = kvo.kvo_attn_sparse_rows_workspace_bytes(rows, hq, hkv, d, k_pad, 64, ps, npu, 0)
    ws = t.empty(wsb, dtype=t.uint8, device="cuda")
    pageable = np.zeros(n_pages * ps * hkv * d * 2, np.uint8)
    small_arena = t.empty(ps * hkv * d * 2, dtype=t.uint8, device="cuda")
    base = dict(q=q, q_dtype=kvo.F16, rows=rows, n_q_heads=hq, n_kv_heads=hkv, head_dim=d, k_pages=kp,
                v_pages=vp, dtype=kvo.F16, page_size=ps, n_pages=n_pages, block_table=bt,
                num_pages_used=npu, indices=idx, k_pad=k_pad, scale=0.1, arena=None, arena_bytes=0,
                rows_per_launch=64, out=out, workspace=ws, workspace_bytes=wsb)
    cases = [(dict(k_pages=pageable.ctypes.data), -3), (dict(q_dtype=kvo.BF16), -4),
             (dict(dtype=kvo.Q8_0, q_dtype=kvo.Q8_0), -4), (dict(workspace_bytes=wsb - 16), -6),
             (dict(arena=small_arena, arena_bytes=small_arena.numel()), -1),
             (dict(num_pages_used=n_pages + 1), -1), (dict(head_dim=96), -4)]
    for change, status in cases:
        with pytest.raises(kvo.KvoError) as e:
            kvo.kvo_attn_sparse_rows(**dict(base, **change))
        assert e.value.status == status, change


def test_copy_pages_host_sees_queued_gpu_writes():
    # A D2H swap queued on a stream writes page 3 of the host K/V planes;
    # the host copy of page 3 -> page 5 must see the swapped bytes.
    t = torch()
    g = synth.rng(1303)
    ps, tok, n_pages = 64, 512, 8
    page = ps * tok
    hk, hv = pinned(n_pages * page), pinned(n_pages * page)
    hk.numpy()[:] = 0
    hv.numpy()[:] = 0
    src_k = t.from_numpy(g.integers(0, 256, page, dtype=np.uint8)).cuda()
    src_v = t.from_numpy(g.integers(0, 256, page, dtype=np.uint8)).cuda()
    d = np.array([src_k.data_ptr(), src_v.data_ptr()], np.int64)
    h = np.array([hk.data_ptr() + 3 * page, hv.data_ptr() + 3 * page], np.int64)
    z = np.array([page, page], np.int64)
    dd, hh, zz = to_pinned(d), to_pinned(h), to_pinned(z)
    s = t.cuda.Stream()
    kvo.kvo_swap_blocks_batch(dd, hh, zz, 2, kvo.KVO_SWAP_D2H, s)
    kvo.kvo_copy_pages_host(hk, hv, hk, hv, ps, tok, 3, 5, 40, s)
    got_k = hk.numpy()[5 * page: 5 * page + 40 * tok]
    got_v = hv.numpy()[5 * page: 5 * page + 40 * tok]
    assert np.array_equal(got_k, src_k.cpu().numpy()[:40 * tok])
    assert np.array_equal(got_v, src_v.cpu().numpy()[:40 * tok])
    assert np.all(hk.numpy()[5 * page + 40 * tok: 6 * page] == 0)      # past num_tokens: untouched
    with pytest.raises(kvo.KvoError) as e:
        kvo.kvo_copy_pages_host(hk, hv, hk, hv, ps, tok, 3, 5, ps + 1, s)
    assert e.value.status == -1
    dev = t.empty(page, dtype=t.uint8, device="cuda")
    with pytest.raises(kvo.KvoError) as e:
        kvo.kvo_copy_pages_host(dev, hv, hk, hv, ps, tok, 0, 1, 4, s)
    assert e.value.status == -3


def test_full_size_qsa_prefill_sampled_rows():
    # 2048 rows x 2080 picks over 262,144 fp16 positions in 1,024 host pages of 256,
    # 32 q / 8 kv heads x 128, staged through a 32 MiB arena (32 buckets) and direct;
    # 24 sampled rows against the oracle.
    from bench import SR_D, SR_HKV, SR_HQ, SR_KPAD, SR_PS, sr_run, sr_setup
    t = torch()
    st = sr_setup()
    kp = st["k_pages"].numpy()
    vp = st["v_pages"].numpy()
    rows = np.linspace(0, 2047, 24).astype(int)
    ref = oracle.attn_sparse_rows(kp, vp, oracle.F16, SR_PS, SR_HKV, SR_D, st["bt_np"], st["n_pages"],
                                  st["idx_np"][rows], st["q_np"][rows], oracle.F16, SR_HQ,
                                  1.0 / math.sqrt(SR_D))
    for staged in (True, False):
        st["out"].fill_(float("nan"))
        sr_run(st, staged)
        t.cuda.synchronize()
        out = st["out"].cpu().numpy().reshape(-1, SR_HQ, SR_D)
        assert np.all(np.isfinite(out)), staged
        assert normwise_rel_err(out[rows], ref) <= REL_TOL, staged
