"""The tiered decode inside a CUDA graph (the question the llama.cpp PR #319
review asks of the staging path): the direct call and the staged call -- whose
copy parts run on a library stream forked from and joined back into the
captured stream, and whose combine is a programmatic dependent launch --
replay from a captured graph with the bits of the eager calls, also after the
query is updated in place."""
import numpy as np
import pytest

import oracle
from helpers import Tiered, cells, scale_for, torch
from host_ram_tiered_gb300 import kvo, synth

pytestmark = pytest.mark.gpu


def test_decode_direct_and_staged_replay_from_cuda_graphs():
    t = torch()
    # four sequences of 30,000 cells, 5,000 in VRAM: two waves of work items,
    # so the staged call copies the tail in two parts
    B, L, hq, hkv, d, N = 4, 30000, 8, 2, 128, 5000
    g = synth.rng(51, 1)
    k, v = cells(B * L, hkv, d, oracle.BF16, g)
    tc = Tiered(k, v, N, batch=B)
    q_a = t.from_numpy(synth.normal_bits((B, hq, d), "bf16", g).view(np.int16).reshape(-1).copy()).cuda()
    q_b = t.from_numpy(synth.normal_bits((B, hq, d), "bf16", g).view(np.int16).reshape(-1).copy()).cuda()
    ctx = t.tensor([L, 2500, 11111, L - 1], dtype=t.int32, device="cuda")
    s = scale_for(d)
    wsb = kvo.kvo_attn_decode_workspace_bytes(B, hq, d, L)
    ws = t.empty(wsb, dtype=t.uint8, device="cuda")
    sk = t.empty(B * (L - N) * tc.rb, dtype=t.uint8, device="cuda")
    sv = t.empty_like(sk)
    q = t.empty_like(q_a)
    assert kvo.kvo_attn_decode_launches(B, L, d, N, 1) == 4

    def call(out, staged, stream=None):
        kvo.kvo_attn_decode_tiered(q, kvo.BF16, B, hq, hkv, d, tc.k_head, tc.v_head, N, tc.k_tail, tc.v_tail,
                                   L - N, kvo.BF16, ctx, L, N, s, sk if staged else None, sv if staged else None,
                                   out, ws, wsb, stream)

    for staged in (False, True):
        eager = {}
        for name, src in (("a", q_a), ("b", q_b)):
            q.copy_(src)
            o = t.empty(B * hq * d, dtype=t.float32, device="cuda")
            call(o, staged)
            t.cuda.synchronize()
            eager[name] = o.cpu().numpy()
        q.copy_(q_a)
        out = t.full((B * hq * d,), float("nan"), dtype=t.float32, device="cuda")
        side = t.cuda.Stream()
        side.wait_stream(t.cuda.current_stream())
        with t.cuda.stream(side):
            call(out, staged, t.cuda.current_stream())          # warm-up outside the capture
        t.cuda.current_stream().wait_stream(side)
        t.cuda.synchronize()
        graph = t.cuda.CUDAGraph()
        with t.cuda.graph(graph, capture_error_mode="relaxed"):
            call(out, staged, t.cuda.current_stream())
        out.fill_(float("nan"))
        graph.replay()
        t.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy().view(np.uint32), eager["a"].view(np.uint32)), staged
        q.copy_(q_b)                                              # new query, same graph
        graph.replay()
        t.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy().view(np.uint32), eager["b"].view(np.uint32)), staged
        del graph


def _graph_matches_eager(call, out, bufs):
    """Eager call, then capture + replay; the replay's bits must equal the
    eager ones for every (name, source) the captured input buffer takes."""
    t = torch()
    dst, sources = bufs
    eager = {}
    for name, src in sources:
        dst.copy_(src)
        out.fill_(float("nan"))
        call(None)
        t.cuda.synchronize()
        eager[name] = out.cpu().numpy().copy()
    dst.copy_(sources[0][1])
    side = t.cuda.Stream()
    side.wait_stream(t.cuda.current_stream())
    with t.cuda.stream(side):
        call(t.cuda.current_stream())                      # warm-up outside the capture
    t.cuda.current_stream().wait_stream(side)
    t.cuda.synchronize()
    graph = t.cuda.CUDAGraph()
    with t.cuda.graph(graph, capture_error_mode="relaxed"):
        call(t.cuda.current_stream())
    for name, src in sources:
        dst.copy_(src)
        out.fill_(float("nan"))
        graph.replay()
        t.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy().view(np.uint32), eager[name].view(np.uint32)), name


def test_staged_prefill_replays_from_a_cuda_graph():
    # two arena slots (the copy engine on a library stream, one bucket ahead)
    # and row blocks alternating between the captured and a library stream
    t = torch()
    R, pos0, L, N, hq, hkv, d = 100, 900, 1000, 300, 8, 2, 128
    g = synth.rng(51, 2)
    k, v = cells(L, hkv, d, oracle.BF16, g)
    tc = Tiered(k, v, N)
    qa = t.from_numpy(synth.normal_bits((R, hq, d), "bf16", g).view(np.int16).reshape(-1).copy()).cuda()
    qb = t.from_numpy(synth.normal_bits((R, hq, d), "bf16", g).view(np.int16).reshape(-1).copy()).cuda()
    q = t.empty_like(qa)
    out = t.empty(R * hq * d, dtype=t.float32, device="cuda")
    wsb = kvo.kvo_attn_prefill_workspace_bytes(R, hq)
    ws = t.empty(wsb, dtype=t.uint8, device="cuda")
    ab = 2 * 128 * tc.rb
    arena = t.empty(ab, dtype=t.uint8, device="cuda")

    def call(stream):
        kvo.kvo_attn_prefill_tiered(q, R, pos0, hq, hkv, d, tc.k_head, tc.v_head, tc.k_tail, tc.v_tail, kvo.BF16,
                                    L, N, 0.0883, arena, ab, 48, out, ws, wsb, stream)

    _graph_matches_eager(call, out, (q, [("a", qa), ("b", qb)]))


def test_staged_sparse_rows_replay_from_a_cuda_graph():
    # partition once per call, then per bucket a page gather into one of two
    # arena slots on a library stream and the split launches that fold
    t = torch()
    rows, hq, hkv, d = 200, 8, 2, 128
    n_pages, ps, npu, k_pad = 48, 16, 40, 96
    g = synth.rng(51, 3)
    kp = synth.normal_bits((n_pages, ps, hkv, d), "f16", g)
    vp = synth.normal_bits((n_pages, ps, hkv, d), "f16", g)
    kpin = t.from_numpy(kp.view(np.uint8).reshape(-1).copy()).pin_memory()
    vpin = t.from_numpy(vp.view(np.uint8).reshape(-1).copy()).pin_memory()
    bt = t.from_numpy(g.permutation(n_pages).astype(np.int32)[:npu].copy()).cuda()
    idx = t.from_numpy(synth.row_selections(rows, k_pad, npu * ps - rows - 8, 80, g, pad_frac=0.1)
                       .reshape(-1).copy()).cuda()
    qa = t.from_numpy(synth.normal_bits((rows, hq, d), "f16", g).view(np.int16).reshape(-1).copy()).cuda()
    qb = t.from_numpy(synth.normal_bits((rows, hq, d), "f16", g).view(np.int16).reshape(-1).copy()).cuda()
    q = t.empty_like(qa)
    page_bytes = ps * hkv * d * 2
    ab = 2 * 5 * page_bytes
    arena = t.empty(ab, dtype=t.uint8, device="cuda")
    wsb = kvo.kvo_attn_sparse_rows_workspace_bytes(rows, hq, hkv, d, k_pad, 64, ps, npu, ab)
    ws = t.empty(wsb, dtype=t.uint8, device="cuda")
    out = t.empty(rows * hq * d, dtype=t.float32, device="cuda")

    def call(stream):
        kvo.kvo_attn_sparse_rows(q, kvo.F16, rows, hq, hkv, d, kpin, vpin, kvo.F16, ps, n_pages, bt, npu, idx, k_pad,
                                 1 / np.sqrt(d), arena, ab, 64, out, ws, wsb, stream)

    _graph_matches_eager(call, out, (q, [("a", qa), ("b", qb)]))
