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


def _noalloc_call(tc, q_dev, hq, hkv, d, kv_dtype, ctx, scale, staged):
    t = torch()
    out = t.full((tc.batch * hq * d,), float("nan"), dtype=t.float32, device="cuda")
    sk = sv = None
    if staged:
        sk = t.empty(tc.batch * (tc.L - tc.n) * tc.rb, dtype=t.uint8, device="cuda")
        sv = t.empty_like(sk)
    kvo.kvo_attn_decode_tiered_noalloc(q_dev, kvo.F16 if kv_dtype != oracle.BF16 else kvo.BF16,
                                       tc.batch, hq, hkv, d, tc.k_head, tc.v_head, tc.n, tc.k_tail,
                                       tc.v_tail, tc.L - tc.n, kv_dtype, ctx, tc.L, tc.n, scale, sk, sv,
                                       out)
    t.cuda.synchronize()
    return out.cpu().numpy().reshape(tc.batch, hq, d)


def _oracle_rows(tc, kvdt, hkv, d, q, hq, lens, scale, seqs):
    """The fp64 oracle for the sequences `seqs` of a Tiered batch, one at a time."""
    want = {}
    for b in seqs:
        def p(a):
            return a if a.size else None
        c = oracle.make_cache(p(tc.k_head_np[b]), p(tc.v_head_np[b]), p(tc.k_tail_np[b]),
                              p(tc.v_tail_np[b]), tc.n, tc.L - tc.n, tc.n, kvdt, hkv, d)
        want[b] = oracle.attn_decode(c, q[b:b + 1], oracle.F16 if kvdt != oracle.BF16 else oracle.BF16,
                                     1, hq, [lens[b]], scale)[0]
    return want


def test_noalloc_splits_far_longer_than_the_regular_chunks_q8_0():
    # 64 sequences x 48 query heads: the 8 MiB scratch holds 5 splits per sequence, so
    # 9,600 cells run as 5 splits of 1,920 cells (three times the regular 640-cell
    # maximum), over a tiered cache with ragged lengths.  Checked against the fp64 oracle
    # on sampled sequences (every head) and against the workspace call on all of them;
    # the staged no-workspace call must give the direct one's bits.
    t = torch()
    B, hq, hkv, d, L, N = 64, 48, 8, 128, 9600, 4000
    assert (8 << 20) // (B * hq * (d + 2) * 4) == 5
    g = synth.rng(4323)
    k, v = cells(B * L, hkv, d, oracle.Q8_0, g)
    tc = Tiered(k, v, N, batch=B)
    del k, v
    lens = [L - 131 * i for i in range(B)]
    lens[5] = 1                                  # a one-cell sequence
    lens[9] = N                                  # exactly the VRAM head
    ctx = t.tensor(lens, dtype=t.int32, device="cuda")
    q = synth.normal_bits((B, hq, d), "f16", g)
    qd = t.from_numpy(q.view(np.int16).reshape(-1).copy()).cuda()
    scale = 1 / math.sqrt(d)
    got = _noalloc_call(tc, qd, hq, hkv, d, oracle.Q8_0, ctx, scale, staged=False)
    assert np.isfinite(got).all()
    ref = run_decode(tc, qd, kvo.F16, hq, hkv, d, oracle.Q8_0, ctx, scale)
    assert normwise_rel_err(got, ref.astype(np.float64)) <= REL_TOL
    assert np.abs(got - ref).max() <= 1e-2
    want = _oracle_rows(tc, oracle.Q8_0, hkv, d, q, hq, lens, scale, [0, 5, 9, 33, 63])
    for b, w in want.items():
        assert normwise_rel_err(got[b], w) <= REL_TOL, b
        assert np.abs(got[b] - w).max() <= 1e-2, b
    staged = _noalloc_call(tc, qd, hq, hkv, d, oracle.Q8_0, ctx, scale, staged=True)
    assert np.array_equal(staged.view(np.uint32), got.view(np.uint32))


def test_noalloc_one_split_per_sequence_f16():
    # 128 sequences x 64 query heads: one split per sequence fits (4.3 MB of partials), so
    # each sequence's 2,999 cells are one chunk of 3,008 cells.
    t = torch()
    B, hq, hkv, d, L, N = 128, 64, 8, 128, 2999, 1200
    assert (8 << 20) // (B * hq * (d + 2) * 4) == 1
    g = synth.rng(4324)
    k, v = cells(B * L, hkv, d, oracle.F16, g)
    tc = Tiered(k, v, N, batch=B)
    del k, v
    lens = [L - 23 * i for i in range(B)]
    ctx = t.tensor(lens, dtype=t.int32, device="cuda")
    q = synth.normal_bits((B, hq, d), "f16", g)
    qd = t.from_numpy(q.view(np.int16).reshape(-1).copy()).cuda()
    scale = 1 / math.sqrt(d)
    got = _noalloc_call(tc, qd, hq, hkv, d, oracle.F16, ctx, scale, staged=False)
    ref = run_decode(tc, qd, kvo.F16, hq, hkv, d, oracle.F16, ctx, scale)
    assert normwise_rel_err(got, ref.astype(np.float64)) <= REL_TOL
    want = _oracle_rows(tc, oracle.F16, hkv, d, q, hq, lens, scale, [0, 64, 127])
    for b, w in want.items():
        assert normwise_rel_err(got[b], w) <= REL_TOL, b


def test_noalloc_staged_matches_direct_and_the_workspace_call_bit_for_bit():
    # Four sequences of 30,000 cells, 5,000 in VRAM: the partials of the regular splits fit,
    # so the no-workspace call uses the workspace call's splits; staged, it copies the tail
    # in two parts on the library stream.  Two calls in a row, each bit-identical to the
    # direct no-workspace call and to the staged workspace call.
    t = torch()
    B, L, hq, hkv, d, N = 4, 30000, 8, 2, 128, 5000
    g = synth.rng(4325)
    k, v = cells(B * L, hkv, d, oracle.BF16, g)
    tc = Tiered(k, v, N, batch=B)
    lens = [L, 2500, 11111, L - 1]
    ctx = t.tensor(lens, dtype=t.int32, device="cuda")
    scale = 1 / math.sqrt(d)
    assert kvo.kvo_attn_decode_launches(B, L, d, N, 1) == 4
    for call in range(2):
        q = synth.normal_bits((B, hq, d), "bf16", synth.rng(4325, 10 + call))
        qd = t.from_numpy(q.view(np.int16).reshape(-1).copy()).cuda()
        direct = _noalloc_call(tc, qd, hq, hkv, d, oracle.BF16, ctx, scale, staged=False)
        staged = _noalloc_call(tc, qd, hq, hkv, d, oracle.BF16, ctx, scale, staged=True)
        ws_staged = run_decode(tc, qd, kvo.BF16, hq, hkv, d, oracle.BF16, ctx, scale, staging=True)
        assert np.array_equal(staged.view(np.uint32), direct.view(np.uint32)), call
        assert np.array_equal(staged.view(np.uint32), ws_staged.view(np.uint32)), call
        want = _oracle_rows(tc, oracle.BF16, hkv, d, q, hq, lens, scale, [0, 2])
        for b, w in want.items():
            assert normwise_rel_err(staged[b], w) <= REL_TOL, (call, b)
