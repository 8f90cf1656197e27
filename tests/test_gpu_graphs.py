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
    # four sequences of 30,000 cells, 5,000 in VRAM: five waves of work items,
    # so the staged call copies the tail in four parts
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
    assert kvo.kvo_attn_decode_launches(B, L, d, N, 1) == 6

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
