"""Failure detection without a GPU fault: every barrier wait of the library's
tensor-core kernels is bounded; when one runs out, the waiter sets bit 2 of
kvo_device_errors() and the kernel winds down and returns.  The self-test
entry point runs that same wait on a barrier that nothing completes, with a
short limit, and the context must stay usable afterwards."""
import math

import numpy as np
import pytest

import oracle
from helpers import Tiered, cells, normwise_rel_err, run_decode, torch
from host_ram_tiered_gb300 import kvo, synth

pytestmark = pytest.mark.gpu

WAIT_TIMEOUT_BIT = 4


def test_bounded_wait_runs_out_sets_the_error_bit_and_the_context_stays_usable():
    t = torch()
    kvo.kvo_device_errors(clear=True)
    start, stop = t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True)
    start.record()
    kvo.kvo_selftest_wait_timeout(50_000_000, t.cuda.current_stream())   # 50 ms, nothing arrives
    stop.record()
    t.cuda.synchronize()
    ms = start.elapsed_time(stop)
    assert 45.0 <= ms < 2000.0, ms                   # it waited about the limit, then gave up
    bits = kvo.kvo_device_errors(clear=True)
    assert bits & WAIT_TIMEOUT_BIT, bits
    assert kvo.kvo_device_errors(clear=True) == 0    # cleared
    # the context still runs the library's kernels, with correct results
    d, hq, hkv, L, N = 128, 32, 8, 1024, 512
    g = synth.rng(4400)
    k, v = cells(L, hkv, d, oracle.F16, g)
    tc = Tiered(k, v, N)
    q = synth.normal_bits((1, hq, d), "f16", g)
    qd = t.from_numpy(q.view(np.int16).reshape(-1).copy()).cuda()
    ctx = t.tensor([L], dtype=t.int32, device="cuda")
    scale = 1 / math.sqrt(d)
    got = run_decode(tc, qd, kvo.F16, hq, hkv, d, oracle.F16, ctx, scale)
    want = oracle.attn_decode(tc.oracle_cache(oracle.F16, hkv, d), q, oracle.F16, 1, hq, [L], scale)
    assert normwise_rel_err(got, want) <= 2e-3
    assert kvo.kvo_device_errors(clear=True) == 0
