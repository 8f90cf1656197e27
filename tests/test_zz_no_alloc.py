"""kvo_attn_decode_tiered_noalloc: the decode entry point for callers that
cannot hand the library a workspace (memory reserved up front by a
framework's allocator, or a C host with no device allocator).  Its partials
live in the library's fixed device scratch array; its output must match the
workspace entry point's within the decode tolerance, on two calls in a row
(the second call finds the first call's partials still in the array)."""
import math

import numpy as np
import pytest

import oracle
from helpers import Tiered, cells, normwise_rel_err, run_decode, torch
from host_ram_tiered_gb300 import kvo, synth

pytestmark = pytest.mark.gpu

REL_TOL = 2e-3


def _noalloc(tc, q_dev, hq, hkv, d, kv_dtype, ctx, scale):
    t = torch()
    out = t.empty(tc.batch * hq * d, dtype=t.float32, device="cuda")
    kvo.kvo_attn_decode_tiered_noalloc(q_dev, kvo.F16, tc.batch, hq, hkv, d, tc.k_head, tc.v_head,
                                       tc.n, tc.k_tail, tc.v_tail, tc.L - tc.n, kv_dtype, ctx, tc.L,
                                       tc.n, scale, None, None, out)
    t.cuda.synchronize()
    return out.cpu().numpy().reshape(tc.batch, hq, d)


@pytest.mark.parametrize("L,N,kvdt,hq,hkv", [(184320, 8192, oracle.Q8_0, 48, 8),
                                             (3001, 700, oracle.F16, 32, 8)])
def test_noalloc_matches_workspace_entry_point_twice(L, N, kvdt, hq, hkv):
    t = torch()
    d = 128
    g = synth.rng(4321, L)
    k, v = cells(L, hkv, d, kvdt, g)
    tc = Tiered(k, v, N)
    scale = 1 / math.sqrt(d)
    ctx = t.tensor([L], dtype=t.int32, device="cuda")
    for call in range(2):
        q = synth.normal_bits((1, hq, d), "f16", synth.rng(4321, 100 + call))
        qd = t.from_numpy(q.view(np.int16).reshape(-1).copy()).cuda()
        ref = run_decode(tc, qd, kvo.F16, hq, hkv, d, kvdt, ctx, scale)
        got = _noalloc(tc, qd, hq, hkv, d, kvdt, ctx, scale)
        assert normwise_rel_err(got, ref.astype(np.float64)) <= REL_TOL, call
        if kvdt == oracle.Q8_0:
            assert np.abs(got - ref).max() <= 1e-2


def test_noalloc_rejects_what_does_not_fit():
    t = torch()
    x = t.zeros(1 << 12, dtype=t.uint8, device="cuda")
    ctx = t.ones(1, dtype=t.int32, device="cuda")
    o = t.zeros(1 << 12, dtype=t.float32, device="cuda")
    # 8192 sequences x 8 heads x 130 floats > 8 MiB: rejected before any launch
    with pytest.raises(kvo.KvoError) as e:
        kvo.kvo_attn_decode_tiered_noalloc(x, kvo.F16, 8192, 8, 8, 128, x, x, 1, None, None, 0,
                                           kvo.F16, ctx, 1, 1, 0.1, None, None, o)
    assert e.value.status == -6


def test_noalloc_lengthens_the_split_when_the_partials_do_not_fit():
    # 64 sequences x 48 heads: the regular chunks' partials exceed the 8 MiB
    # scratch, so the no-workspace call runs with longer chunks; the result must
    # still meet the decode tolerance against the oracle and the workspace call.
    t = torch()
    B, hq, hkv, d, L = 64, 48, 8, 128, 3000
    g = synth.rng(4322)
    k, v = cells(B * L, hkv, d, oracle.F16, g)
    tc = Tiered(k.reshape(B * L, -1), v.reshape(B * L, -1), 1000, batch=B)
    lens = [L - 37 * i for i in range(B)]
    ctx = t.tensor(lens, dtype=t.int32, device="cuda")
    q = synth.normal_bits((B, hq, d), "f16", g)
    qd = t.from_numpy(q.view(np.int16).reshape(-1).copy()).cuda()
    scale = 1 / math.sqrt(d)
    assert kvo.kvo_attn_decode_workspace_bytes(B, hq, d, L) > 8 << 20
    got = _noalloc(tc, qd, hq, hkv, d, oracle.F16, ctx, scale)
    ref = run_decode(tc, qd, kvo.F16, hq, hkv, d, oracle.F16, ctx, scale)
    assert normwise_rel_err(got, ref.astype(np.float64)) <= REL_TOL
    want = oracle.attn_decode(tc.oracle_cache(oracle.F16, hkv, d), q, oracle.F16, B, hq, lens, scale)
    assert normwise_rel_err(got, want) <= REL_TOL
