"""GPU parity of kvo_attn_decode_tiered against the fp64 oracle (normwise
relative error <= 2e-3; q8_0 also <= 1e-2 absolute), and the pages'
invariant: a tiered cache gives output bit-identical to the same kernel on
an all-VRAM cache, with staging on and off."""
import math

import numpy as np
import pytest

import oracle
from helpers import Tiered, cells, normwise_rel_err, run_decode, scale_for, torch
from host_ram_tiered_gb300 import kvo, synth

pytestmark = pytest.mark.gpu

REL_TOL = 2e-3
Q8_ABS_TOL = 1e-2


def _q(batch, hq, d, name, gen):
    t = torch()
    q = synth.normal_bits((batch, hq, d), name, gen)
    return q, t.from_numpy(q.view(np.int16).reshape(-1).copy()).cuda()


def _ctx(lens):
    t = torch()
    return t.tensor(list(lens), dtype=t.int32, device="cuda")


def _oracle(tc, q, q_dt, hq, hkv, d, kv_dt, lens, scale):
    c = tc.oracle_cache(kv_dt, hkv, d)
    return oracle.attn_decode(c, q, q_dt, tc.batch, hq, lens, scale)


@pytest.mark.parametrize("staging", [False, True])
def test_c1_tiny_decode_tiered_equals_all_vram(staging):
    # 1 sequence, 32 q heads / 8 kv heads x 128, fp16, context 1024, N = 512.
    g = synth.rng(1234, 20)
    L, hq, hkv, d = 1024, 32, 8, 128
    k, v = cells(L, hkv, d, oracle.F16, g)
    q, qd = _q(1, hq, d, "f16", g)
    ctx = _ctx([L])
    s = scale_for(d)
    tiered = Tiered(k, v, 512)
    out = run_decode(tiered, qd, kvo.F16, hq, hkv, d, kvo.F16, ctx, s, staging=staging)
    ref = _oracle(tiered, q, oracle.F16, hq, hkv, d, oracle.F16, [L], s)
    assert normwise_rel_err(out, ref) <= REL_TOL
    allv = run_decode(Tiered(k, v, L), qd, kvo.F16, hq, hkv, d, kvo.F16, ctx, s)
    assert np.array_equal(out.view(np.uint32), allv.view(np.uint32))
    host_only = run_decode(Tiered(k, v, 0), qd, kvo.F16, hq, hkv, d, kvo.F16, ctx, s, staging=staging)
    assert np.array_equal(host_only.view(np.uint32), allv.view(np.uint32))


def test_q8_0_ragged_context_and_splits():
    g = synth.rng(1236, 21)
    L, hq, hkv, d = 3001, 48, 8, 128
    k, v = cells(L, hkv, d, oracle.Q8_0, g)
    q, qd = _q(1, hq, d, "f16", g)
    ctx = _ctx([L])
    s = scale_for(d)
    outs = []
    for n in (0, 700, 2999, L):
        for staging in (False, True):
            tc = Tiered(k, v, n)
            outs.append(run_decode(tc, qd, kvo.F16, hq, hkv, d, kvo.Q8_0, ctx, s, staging=staging))
    ref = _oracle(Tiered(k, v, 700), q, oracle.F16, hq, hkv, d, oracle.Q8_0, [L], s)
    assert normwise_rel_err(outs[0], ref) <= REL_TOL
    assert np.abs(outs[0] - ref).max() <= Q8_ABS_TOL
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32))


def test_batch_with_ragged_and_empty_contexts():
    g = synth.rng(7, 22)
    B, L, hq, hkv, d = 4, 777, 16, 4, 128
    k, v = cells(B * L, hkv, d, oracle.BF16, g)
    q, qd = _q(B, hq, d, "bf16", g)
    lens = [0, 1, 333, L]
    s = 0.0883
    tc = Tiered(k, v, 100, batch=B)
    out = run_decode(tc, qd, kvo.BF16, hq, hkv, d, kvo.BF16, _ctx(lens), s)
    ref = _oracle(tc, q, oracle.BF16, hq, hkv, d, oracle.BF16, lens, s)
    assert (out[0] == 0).all()
    assert normwise_rel_err(out[1:], ref[1:]) <= REL_TOL
    allv = run_decode(Tiered(k, v, L, batch=B), qd, kvo.BF16, hq, hkv, d, kvo.BF16, _ctx(lens), s)
    assert np.array_equal(out.view(np.uint32), allv.view(np.uint32))


def test_staged_copy_in_parts_is_bit_identical():
    # Four sequences of up to 30,000 cells: 73 chunks of 416 cells each, 292
    # work items or two waves of CTAs, so the staged call decodes the chunks wholly in VRAM
    # while the host tail is copied in two parts, and each part's chunks as
    # it lands (four launches: the VRAM chunks, two parts, the combine).  Ragged lengths:
    # full, inside the VRAM head, ending inside a part, one short of full.
    g = synth.rng(31, 23)
    B, L, hq, hkv, d, N = 4, 30000, 8, 2, 128, 5000
    k, v = cells(B * L, hkv, d, oracle.BF16, g)
    q, qd = _q(B, hq, d, "bf16", g)
    lens = [L, 2500, 11111, L - 1]
    s = scale_for(d)
    assert kvo.kvo_attn_decode_launches(B, L, d, N, 1) == 4
    tc = Tiered(k, v, N, batch=B)
    staged = run_decode(tc, qd, kvo.BF16, hq, hkv, d, kvo.BF16, _ctx(lens), s, staging=True)
    direct = run_decode(tc, qd, kvo.BF16, hq, hkv, d, kvo.BF16, _ctx(lens), s)
    allv = run_decode(Tiered(k, v, L, batch=B), qd, kvo.BF16, hq, hkv, d, kvo.BF16, _ctx(lens), s)
    assert np.array_equal(staged.view(np.uint32), direct.view(np.uint32))
    assert np.array_equal(staged.view(np.uint32), allv.view(np.uint32))
    ref = _oracle(tc, q, oracle.BF16, hq, hkv, d, oracle.BF16, lens, s)
    assert normwise_rel_err(staged, ref) <= REL_TOL


@pytest.mark.parametrize("hq,hkv,d,kvdt", [(8, 8, 128, oracle.F16), (64, 8, 128, oracle.BF16),
                                           (12, 4, 64, oracle.Q8_0), (7, 1, 64, oracle.F16),
                                           (40, 8, 64, oracle.BF16)])
def test_group_sizes_and_head_dims(hq, hkv, d, kvdt):
    g = synth.rng(8, hq * 1000 + d)
    L = 517
    k, v = cells(L, hkv, d, kvdt, g)
    # q is the cache's 16-bit type (fp16 for a q8_0 cache)
    bf = kvdt == oracle.BF16
    q, qd = _q(1, hq, d, "bf16" if bf else "f16", g)
    s = scale_for(d)
    tc = Tiered(k, v, 200)
    out = run_decode(tc, qd, kvo.BF16 if bf else kvo.F16, hq, hkv, d, kvdt, _ctx([L]), s, staging=True)
    ref = _oracle(tc, q, oracle.BF16 if bf else oracle.F16, hq, hkv, d, kvdt, [L], s)
    assert normwise_rel_err(out, ref) <= REL_TOL


def test_argument_errors():
    t = torch()
    g = synth.rng(9)
    L, hq, hkv, d = 64, 8, 2, 128
    k, v = cells(L, hkv, d, oracle.F16, g)
    q, qd = _q(1, hq, d, "f16", g)
    tc = Tiered(k, v, 32)
    out = t.empty(hq * d, dtype=t.float32, device="cuda")
    need = kvo.kvo_attn_decode_workspace_bytes(1, hq, d, L)
    ws = t.empty(need, dtype=t.uint8, device="cuda")
    ctx = _ctx([L])
    pageable = np.zeros(L * tc.rb, np.uint8)
    cases = [
        (dict(k_host=pageable.ctypes.data), -3),
        (dict(workspace_bytes=need - 16), -6),
        (dict(n_q_heads=18), -4),                     # group 9
        (dict(head_dim=96), -4),
        (dict(q_dtype=kvo.Q8_0), -4),
        (dict(q_dtype=kvo.BF16), -4),                 # q must be the cache's 16-bit type
        (dict(kv_dtype=kvo.BF16), -4),
    ]
    base = dict(q=qd, q_dtype=kvo.F16, batch=1, n_q_heads=hq, n_kv_heads=hkv, head_dim=d,
                k_vram=tc.k_head, v_vram=tc.v_head, vram_seq_stride_rows=32, k_host=tc.k_tail,
                v_host=tc.v_tail, host_seq_stride_rows=L - 32, kv_dtype=kvo.F16, ctx_len=ctx,
                max_ctx=L, n_vram_cells=32, scale=0.1, staging_k=None, staging_v=None, out=out,
                workspace=ws, workspace_bytes=need)
    for change, status in cases:
        args = dict(base, **change)
        with pytest.raises(kvo.KvoError) as e:
            kvo.kvo_attn_decode_tiered(**args)
        assert e.value.status == status, change


@pytest.mark.parametrize("L", [29696, 96256, 184320])
def test_c3_full_size_tiered_staged_all_vram_bit_identical(L):
    # llama.cpp-style q8_0 decode, 48/8 heads x 128; N in {8192, 94208}; staging on/off.
    from bench import DEC_D, DEC_HKV, DEC_HQ, dec_run, dec_setup
    t = torch()
    st = dec_setup()
    outs = {}
    for N in (8192, 94208):
        for staging in (False, True):
            o = t.empty(DEC_HQ * DEC_D, dtype=t.float32, device="cuda")
            dec_run(st, L, N, staging=staging, out=o)
            outs[(N, staging)] = o
    o = t.empty(DEC_HQ * DEC_D, dtype=t.float32, device="cuda")
    dec_run(st, L, 0, all_vram=True, out=o)
    t.cuda.synchronize()
    allv = o.cpu().numpy()
    for key, x in outs.items():
        assert np.array_equal(x.cpu().numpy().view(np.uint32), allv.view(np.uint32)), key
    rb = st["rb"]
    kh = st["k_host"].numpy()[:L * rb].reshape(L, rb)
    vh = st["v_host"].numpy()[:L * rb].reshape(L, rb)
    cache = oracle.make_cache(None, None, kh, vh, 0, L, 0, oracle.Q8_0, DEC_HKV, DEC_D)
    ref = oracle.attn_decode(cache, st["q_np"], oracle.F16, 1, DEC_HQ, [L], 1.0 / math.sqrt(DEC_D))
    got = allv.reshape(1, DEC_HQ, DEC_D)
    assert normwise_rel_err(got, ref) <= REL_TOL
    assert np.abs(got - ref).max() <= Q8_ABS_TOL


def test_c4_sparse_decode_over_gathered_tokens():
    from bench import TOPK_D, TOPK_HKV, TOPK_HQ, TOPK_K, TOPK_BLK, TOPK_S, topk_decode, topk_gather, topk_setup
    st = topk_setup()
    topk_gather(st)
    topk_decode(st)
    torch().cuda.synchronize()
    from bench import TOPK_T
    tok = TOPK_K * TOPK_BLK
    # the oracle's own gather of the same host planes (never the GPU's output)
    kg = oracle.gather_blocks(st["k_plane"].numpy(), TOPK_S, TOPK_T, TOPK_HKV, TOPK_D, 2, TOPK_BLK,
                              st["sel_np"]).reshape(TOPK_S * tok, -1)
    vg = oracle.gather_blocks(st["v_plane"].numpy(), TOPK_S, TOPK_T, TOPK_HKV, TOPK_D, 2, TOPK_BLK,
                              st["sel_np"]).reshape(TOPK_S * tok, -1)
    cache = oracle.make_cache(kg, vg, None, None, tok, 0, tok, oracle.BF16, TOPK_HKV, TOPK_D)
    ref = oracle.attn_decode(cache, st["q_np"], oracle.BF16, TOPK_S, TOPK_HQ, [tok] * TOPK_S,
                             1.0 / math.sqrt(TOPK_D))
    out = st["out"].cpu().numpy().reshape(TOPK_S, TOPK_HQ, TOPK_D)
    assert normwise_rel_err(out, ref) <= REL_TOL
