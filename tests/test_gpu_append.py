"""GPU parity of kvo_append_kv_tiered (the write path of the tiered cache)
against the oracle's append: byte-exact cache contents, for copies and for
q8_0 quantisation, with the appended range crossing the VRAM/host boundary;
then a decode over the appended cache matches the oracle's decode."""
import math

import numpy as np
import pytest

import oracle
from helpers import normwise_rel_err, pinned, torch
from host_ram_tiered_gb300 import kvo, synth

pytestmark = pytest.mark.gpu


def _run(dt, src_dt, H, D, N, cap, pos0, n_new, seed):
    t = torch()
    g = synth.rng(seed, dt)
    name = "bf16" if src_dt == oracle.BF16 else "f16"
    kn = synth.normal_bits((n_new, H * D), name, g).view(np.uint8).reshape(n_new, -1).copy()
    vn = synth.normal_bits((n_new, H * D), name, g).view(np.uint8).reshape(n_new, -1).copy()
    rb = oracle.row_bytes(dt, H, D)
    n_lo = min(N, cap)
    # pre-fill both tiers with seeded cells of the cache dtype: untouched cells
    # must survive, and the whole cache stays a valid one to attend over
    if dt == oracle.Q8_0:
        kh0, vh0 = synth.q8_0_rows(n_lo, H, D, g), synth.q8_0_rows(n_lo, H, D, g)
        kt0, vt0 = synth.q8_0_rows(cap - n_lo, H, D, g), synth.q8_0_rows(cap - n_lo, H, D, g)
    else:
        nm = "bf16" if dt == oracle.BF16 else "f16"
        kh0, vh0, kt0, vt0 = [synth.normal_bits((n, H * D), nm, g).view(np.uint8).reshape(n, rb).copy()
                              for n in (n_lo, n_lo, cap - n_lo, cap - n_lo)]
    kh = t.from_numpy(kh0.reshape(-1).copy()).cuda()
    vh = t.from_numpy(vh0.reshape(-1).copy()).cuda()
    kt = pinned(kt0.size); kt.numpy()[:kt0.size] = kt0.reshape(-1)
    vt = pinned(vt0.size); vt.numpy()[:vt0.size] = vt0.reshape(-1)
    kn_d = t.from_numpy(kn.reshape(-1)).cuda()
    vn_d = t.from_numpy(vn.reshape(-1)).cuda()
    kvo.kvo_append_kv_tiered(kn_d, vn_d, src_dt, n_new, pos0, H, D, kh, vh, kt, vt, dt, N, cap)
    t.cuda.synchronize()
    ek, ev, etk, etv = kh0.copy(), vh0.copy(), kt0.copy(), vt0.copy()
    oracle.append_kv(kn, vn, src_dt, n_new, pos0, H, D, ek, ev, etk, etv, dt, n_lo)
    assert np.array_equal(kh.cpu().numpy(), ek.reshape(-1))
    assert np.array_equal(vh.cpu().numpy(), ev.reshape(-1))
    assert np.array_equal(kt.numpy()[:kt0.size], etk.reshape(-1))
    assert np.array_equal(vt.numpy()[:vt0.size], etv.reshape(-1))
    return ek, ev, etk, etv, (kh, vh, kt, vt)


@pytest.mark.parametrize("dt,src", [(oracle.Q8_0, oracle.BF16), (oracle.Q8_0, oracle.F16),
                                    (oracle.BF16, oracle.BF16), (oracle.F16, oracle.F16)])
def test_append_crossing_the_tier_boundary(dt, src):
    _run(dt, src, 8, 128, 300, 1000, 250, 131, seed=1240)


def test_append_single_decode_token_into_the_host_tail_and_decode():
    # one decode step: one token appended at the tail, then attention over all cells
    t = torch()
    H, D, N, cap, hq = 8, 128, 100, 400, 48
    ek, ev, etk, etv, dev = _run(oracle.Q8_0, oracle.F16, H, D, N, cap, 399, 1, seed=1241)
    kh, vh, kt, vt = dev
    # decode a query over the whole cache; the oracle reads its own appended copy
    q = synth.normal_bits((1, hq, D), "f16", synth.rng(1242))
    qd = t.from_numpy(q.view(np.int16).reshape(-1).copy()).cuda()
    ctx = t.tensor([cap], dtype=t.int32, device="cuda")
    out = t.empty(hq * D, dtype=t.float32, device="cuda")
    wsb = kvo.kvo_attn_decode_workspace_bytes(1, hq, D, cap)
    ws = t.empty(wsb, dtype=t.uint8, device="cuda")
    kvo.kvo_attn_decode_tiered(qd, kvo.F16, 1, hq, H, D, kh, vh, N, kt, vt, cap - N, kvo.Q8_0, ctx,
                               cap, N, 1 / math.sqrt(D), None, None, out, ws, wsb)
    t.cuda.synchronize()
    cache = oracle.make_cache(ek, ev, etk, etv, N, cap - N, N, oracle.Q8_0, H, D)
    ref = oracle.attn_decode(cache, q, oracle.F16, 1, hq, [cap], 1 / math.sqrt(D))
    assert normwise_rel_err(out.cpu().numpy().reshape(1, hq, D), ref) <= 2e-3


def test_append_argument_errors():
    t = torch()
    x = t.zeros(1 << 16, dtype=t.uint8, device="cuda")
    with pytest.raises(kvo.KvoError) as e:                      # past the capacity
        kvo.kvo_append_kv_tiered(x, x, kvo.F16, 4, 8, 2, 64, x, x, None, None, kvo.F16, 16, 10)
    assert e.value.status == -1
    with pytest.raises(kvo.KvoError) as e:                      # f16 source into a bf16 cache
        kvo.kvo_append_kv_tiered(x, x, kvo.F16, 4, 0, 2, 64, x, x, None, None, kvo.BF16, 16, 16)
    assert e.value.status == -4
    pageable = np.zeros(1 << 16, np.uint8)
    with pytest.raises(kvo.KvoError) as e:                      # tail not mapped
        kvo.kvo_append_kv_tiered(x, x, kvo.F16, 4, 0, 2, 64, x, x, pageable.ctypes.data,
                                 pageable.ctypes.data, kvo.F16, 2, 16)
    assert e.value.status == -3
