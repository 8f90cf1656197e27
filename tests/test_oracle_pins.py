"""Pins of the CPU oracle against things other than itself (no GPU).

Each test checks the oracle against a library routine, a closed form, an
invariant the source pages state, or a brute-force enumeration, chosen so
that a dropped term, a wrong sign or index or a transposed operand in the
oracle fails at least one of them.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from host_ram_tiered_gb300 import synth


# ---------------------------------------------------------------- formats

def test_half_decoding_matches_numpy_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_decoding_matches_torch_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_generator_bf16_rounding_is_torch_rne():
    x = synth.rng(7).standard_normal(200000, dtype=np.float32) * 37.0
    ours = synth.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_row_bytes():
    assert oracle.row_bytes(oracle.Q8_0, 8, 128) == 1088      # 8 heads x 4 blocks x 34 B
    assert oracle.row_bytes(oracle.F16, 8, 128) == 2048
    assert oracle.row_bytes(oracle.BF16, 4, 128) == 1024
    assert oracle.row_bytes(oracle.Q8_0, 8, 100) == 0


def test_q8_0_hand_values():
    # head_dim 64 -> 2 blocks per head, 2 heads -> 4 blocks in the row
    row = np.zeros(4 * 34, np.uint8)
    scales = [0x3800, 0xB400, 0x1234, 0x3C00]           # 0.5, -0.25, small, 1.0
    for blk, sc in enumerate(scales):
        row[blk * 34: blk * 34 + 2] = np.array([sc], np.uint16).view(np.uint8)
        row[blk * 34 + 2: blk * 34 + 34] = (np.arange(-16, 16) * (blk + 1)).astype(np.int8).view(np.uint8)
    h0 = oracle.load_head(row, oracle.Q8_0, 64, 0)
    h1 = oracle.load_head(row, oracle.Q8_0, 64, 1)
    assert h0[0] == 0.5 * -16 and h0[31] == 0.5 * 15
    assert h0[32] == -0.25 * -32 and h0[63] == -0.25 * 30
    small = float(np.array([0x1234], np.uint16).view(np.float16)[0])
    assert h1[5] == small * (-11 * 3)
    assert h1[32 + 31] == 1.0 * (15 * 4)


# ---------------------------------------------------------------- pointers

def _brute_sub_block_ptrs(ids, bpc, skip, base, stride, row_bytes, n):
    page = row_bytes // bpc
    grid = []
    for b in ids:
        for j in range(bpc):
            grid.append(base + int(b) * stride + j * page)
    return grid[skip: skip + n]


@pytest.mark.parametrize("bpc,skip,n", [(1, 0, 7), (4, 0, 16), (4, 1, 13), (4, 3, 10), (3, 2, 1)])
def test_sub_block_ptrs_brute_force(bpc, skip, n):
    g = synth.rng(3, bpc * 10 + skip)
    ids = g.permutation(50)[:8].astype(np.int64)
    base, row_bytes = 0x7F0000001000, bpc * 2048
    stride = row_bytes * 3 // 2
    n = min(n, len(ids) * bpc - skip)
    got = oracle.sub_block_ptrs(ids, bpc, skip, base, stride, row_bytes, n)
    assert got.tolist() == _brute_sub_block_ptrs(ids, bpc, skip, base, stride, row_bytes, n)


def test_sub_block_ptrs_rejects_page_asserts():
    ids = np.arange(4)
    with pytest.raises(ValueError):
        oracle.sub_block_ptrs(ids, 4, 4, 0, 1024, 1024, 4)       # skip >= bpc
    with pytest.raises(ValueError):
        oracle.sub_block_ptrs(ids, 3, 0, 0, 1024, 1024, 4)       # row % bpc != 0
    with pytest.raises(ValueError):
        oracle.sub_block_ptrs(ids, 4, 1, 0, 1024, 1024, 16)      # beyond the grid


def test_group_walk_consumes_cdiv_chunks():
    # transfer_async: a group of 2048 GPU blocks starting at logical block 1 consumes
    # cdiv(2048 + 1, 4) = 513 host chunks; 512 would not cover it.
    n, bpc, skip = 2048, 4, 1
    need = -(-(n + skip) // bpc)
    assert need == 513
    ids = np.arange(need)
    oracle.sub_block_ptrs(ids, bpc, skip, 0, 16, 16, n)
    with pytest.raises(ValueError):
        oracle.sub_block_ptrs(ids[:512], bpc, skip, 0, 16, 16, n)


# ---------------------------------------------------------------- swap

def test_swap_matches_numpy_slices_and_round_trips():
    g = synth.rng(11)
    page = 256
    dev = g.integers(0, 256, size=(32, page), dtype=np.uint8)          # "device" pool
    host = np.zeros((20, page + 64), np.uint8)                         # padded host rows
    host[:, page:] = 0xA5                                              # canaries
    dev_ids = g.permutation(32)[:12]
    host_ids = g.permutation(20)[:12]
    src = np.array([dev[i].ctypes.data for i in dev_ids], np.uint64)
    dst = np.array([host[i].ctypes.data for i in host_ids], np.uint64)
    sizes = np.full(12, page, np.int64)
    expect = host.copy()
    expect[host_ids, :page] = dev[dev_ids]
    oracle.swap_blocks(src, dst, sizes)
    assert np.array_equal(host, expect)
    assert (host[:, page:] == 0xA5).all()
    # H2D back into a clean device pool: round trip is byte-identical
    dev2 = np.zeros_like(dev)
    src2 = dst
    dst2 = np.array([dev2[i].ctypes.data for i in dev_ids], np.uint64)
    oracle.swap_blocks(src2, dst2, sizes)
    assert np.array_equal(dev2[dev_ids], dev[dev_ids])
    untouched = np.setdiff1d(np.arange(32), dev_ids)
    assert (dev2[untouched] == 0).all()


def test_swap_zero_descriptors_is_noop():
    oracle.swap_blocks(np.zeros(0, np.uint64), np.zeros(0, np.uint64), np.zeros(0, np.int64))


# ---------------------------------------------------------------- gather

def test_gather_matches_numpy_fancy_indexing():
    g = synth.rng(5)
    S, T, H, D, blk, k = 3, 12 * 8, 2, 16, 8, 4
    plane = synth.normal_bits((S, T, H, D), "bf16", g)
    sel = synth.topk_selection(S, H, T // blk, k, g)
    got = oracle.gather_blocks(plane, S, T, H, D, 2, blk, sel).view(np.uint16).reshape(S, k * blk, H, D)
    for s in range(S):
        for h in range(H):
            toks = (sel[s, h][:, None] * blk + np.arange(blk)[None, :]).reshape(-1)
            assert np.array_equal(got[s, :, h, :], plane[s, toks, h, :])


def test_gather_rejects_block_outside_plane():
    plane = np.zeros((1, 16, 1, 4), np.uint16)
    with pytest.raises(ValueError):
        oracle.gather_blocks(plane, 1, 16, 1, 4, 2, 8, np.array([[[2]]], np.int32))


def test_topk_selection_shape_and_last_block():
    sel = synth.topk_selection(2, 3, 100, 10, synth.rng(1))
    assert (sel[..., -1] == 99).all()
    for s in range(2):
        for h in range(3):
            assert len(set(sel[s, h].tolist())) == 10
            assert (np.diff(sel[s, h]) > 0).all()


# ---------------------------------------------------------------- attention

def _decode_values(raw, dtype, H, D):
    """Decode raw storage to float64 with numpy/torch (independent of the oracle)."""
    if dtype == oracle.F16:
        return raw.view(np.float16).astype(np.float64).reshape(raw.shape[0], H, D)
    if dtype == oracle.BF16:
        t = torch.from_numpy(raw.view(np.int16)).view(torch.bfloat16).to(torch.float64)
        return t.numpy().reshape(raw.shape[0], H, D)
    nb = D // 32
    blocks = raw.reshape(raw.shape[0], H, nb, 34)
    d = blocks[..., 0:2].copy().view(np.float16).astype(np.float64)      # [n, H, nb, 1]
    qs = blocks[..., 2:].copy().view(np.int8).astype(np.float64)          # [n, H, nb, 32]
    return (d * qs).reshape(raw.shape[0], H, D)


def _cells(L, H, D, dtype, g):
    if dtype == oracle.Q8_0:
        k = synth.q8_0_rows(L, H, D, g)
        v = synth.q8_0_rows(L, H, D, g)
    else:
        name = "f16" if dtype == oracle.F16 else "bf16"
        k = synth.normal_bits((L, H * D), name, g).view(np.uint8).reshape(L, -1)
        v = synth.normal_bits((L, H * D), name, g).view(np.uint8).reshape(L, -1)
    return np.ascontiguousarray(k), np.ascontiguousarray(v)


def _tiered(k, v, n_vram, dtype, H, D):
    n_vram = min(n_vram, k.shape[0])
    kh, vh = np.ascontiguousarray(k[:n_vram]), np.ascontiguousarray(v[:n_vram])
    kt, vt = np.ascontiguousarray(k[n_vram:]), np.ascontiguousarray(v[n_vram:])
    keep = (kh, vh, kt, vt)
    c = oracle.make_cache(kh if kh.size else None, vh if vh.size else None,
                          kt if kt.size else None, vt if vt.size else None,
                          n_vram, k.shape[0] - n_vram, n_vram, dtype, H, D)
    return c, keep


@pytest.mark.parametrize("dtype,Hq,Hkv,D,L", [(oracle.F16, 8, 2, 32, 37),
                                              (oracle.BF16, 6, 2, 64, 50),
                                              (oracle.Q8_0, 6, 2, 64, 45)])
def test_decode_matches_scipy_softmax(dtype, Hq, Hkv, D, L):
    g = synth.rng(21, dtype)
    k, v = _cells(L, Hkv, D, dtype, g)
    qname = "bf16" if dtype == oracle.BF16 else "f16"
    q = synth.normal_bits((1, Hq, D), qname, g)
    c, keep = _tiered(k, v, 17, dtype, Hkv, D)
    scale = 1 / math.sqrt(D)
    got = oracle.attn_decode(c, q, oracle.BF16 if qname == "bf16" else oracle.F16, 1, Hq,
                             [L], scale)
    K = _decode_values(k, dtype, Hkv, D)
    V = _decode_values(v, dtype, Hkv, D)
    Q = _decode_values(q.reshape(1, -1).view(np.uint8), oracle.BF16 if qname == "bf16" else oracle.F16, Hq, D)[0]
    G = Hq // Hkv
    for h in range(Hq):
        s = scale * (K[:, h // G, :] @ Q[h])
        p = scipy.special.softmax(s)
        ref = p @ V[:, h // G, :]
        np.testing.assert_allclose(got[0, h], ref, rtol=1e-12, atol=1e-13)


def test_single_cell_gives_v_and_empty_context_gives_zero():
    g = synth.rng(2)
    k, v = _cells(3, 2, 32, oracle.F16, g)
    c, keep = _tiered(k, v, 1, oracle.F16, 2, 32)
    q = synth.normal_bits((2, 4, 32), "f16", g)
    out = oracle.attn_decode(c, q, oracle.F16, 1, 4, [1], 0.3)
    V = _decode_values(v, oracle.F16, 2, 32)
    for h in range(4):
        assert np.array_equal(out[0, h], V[0, h // 2])
    out0 = oracle.attn_decode(c, q, oracle.F16, 1, 4, [0], 0.3)
    assert (out0 == 0).all()


def test_zero_query_gives_mean_of_v():
    g = synth.rng(4)
    L = 29
    k, v = _cells(L, 2, 32, oracle.BF16, g)
    c, keep = _tiered(k, v, 10, oracle.BF16, 2, 32)
    q = np.zeros((1, 4, 32), np.uint16)
    out = oracle.attn_decode(c, q, oracle.BF16, 1, 4, [L], 0.125)
    V = _decode_values(v, oracle.BF16, 2, 32)
    for h in range(4):
        np.testing.assert_allclose(out[0, h], V[:, h // 2, :].mean(axis=0), rtol=0, atol=1e-15)


def test_gqa_head_map_is_contiguous_groups():
    # The staged kernel's q head is kv_head * group + r: a V that is constant g on
    # kv head g makes every q head h return exactly h // group.
    Hq, Hkv, D, L = 12, 3, 32, 9
    vals = np.zeros((L, Hkv, D), np.float16)
    for gh in range(Hkv):
        vals[:, gh, :] = gh
    v = vals.view(np.uint16).view(np.uint8).reshape(L, -1).copy()
    k = synth.normal_bits((L, Hkv * D), "f16", synth.rng(8)).view(np.uint8).reshape(L, -1).copy()
    c, keep = _tiered(k, v, 4, oracle.F16, Hkv, D)
    q = synth.normal_bits((1, Hq, D), "f16", synth.rng(9))
    out = oracle.attn_decode(c, q, oracle.F16, 1, Hq, [L], 0.2)
    for h in range(Hq):
        assert np.allclose(out[0, h], h // (Hq // Hkv), rtol=0, atol=1e-14)


def test_dominant_logit_selects_its_value():
    D, L = 32, 6
    kf = np.zeros((L, 1, D), np.float16)
    kf[3, 0, :] = 8.0
    k = kf.view(np.uint16).view(np.uint8).reshape(L, -1).copy()
    v = synth.normal_bits((L, D), "f16", synth.rng(10)).view(np.uint8).reshape(L, -1).copy()
    c, keep = _tiered(k, v, 2, oracle.F16, 1, D)
    q = np.full((1, 1, D), 0x4000, np.uint16)                      # 2.0
    out = oracle.attn_decode(c, q, oracle.F16, 1, 1, [L], 1.0)     # logit 512 vs 0
    V = _decode_values(v, oracle.F16, 1, D)
    np.testing.assert_allclose(out[0, 0], V[3, 0], rtol=0, atol=1e-200)


def test_prefill_causal_boundary_closed_form():
    # V = position on dim 0, q = 0: row at position p returns mean(0..p) = p/2.
    Hkv, D, L, R, pos0 = 1, 32, 40, 8, 30
    vals = np.zeros((L, Hkv, D), np.float16)
    vals[:, 0, 0] = np.arange(L)
    v = vals.view(np.uint16).view(np.uint8).reshape(L, -1).copy()
    k = synth.normal_bits((L, D), "f16", synth.rng(12)).view(np.uint8).reshape(L, -1).copy()
    c, keep = _tiered(k, v, 13, oracle.F16, Hkv, D)
    q = np.zeros((R, 2, D), np.uint16)
    out = oracle.attn_prefill(c, q, oracle.F16, R, pos0, 2, L, 0.1)
    for i in range(R):
        assert abs(out[i, 0, 0] - (pos0 + i) / 2) < 1e-12
        assert abs(out[i, 1, 0] - (pos0 + i) / 2) < 1e-12


def test_prefill_row_equals_decode_at_its_position():
    g = synth.rng(13)
    Hq, Hkv, D, L, R, pos0 = 4, 2, 32, 30, 5, 24
    k, v = _cells(L, Hkv, D, oracle.BF16, g)
    c, keep = _tiered(k, v, 11, oracle.BF16, Hkv, D)
    q = synth.normal_bits((R, Hq, D), "bf16", g)
    pre = oracle.attn_prefill(c, q, oracle.BF16, R, pos0, Hq, L, 0.17)
    for i in range(R):
        dec = oracle.attn_decode(c, q[i:i + 1], oracle.BF16, 1, Hq, [pos0 + i + 1], 0.17)
        assert np.array_equal(pre[i], dec[0])


@pytest.mark.parametrize("dtype", [oracle.F16, oracle.Q8_0])
def test_tier_split_does_not_change_the_result(dtype):
    g = synth.rng(14, dtype)
    L, Hkv, D = 33, 2, 64
    k, v = _cells(L, Hkv, D, dtype, g)
    q = synth.normal_bits((1, 4, D), "f16", g)
    c_all, keep_all = _tiered(k, v, L, dtype, Hkv, D)
    ref = oracle.attn_decode(c_all, q, oracle.F16, 1, 4, [L], 0.1)
    for n in (0, 1, 16, 32):
        c, keep = _tiered(k, v, n, dtype, Hkv, D)
        assert np.array_equal(oracle.attn_decode(c, q, oracle.F16, 1, 4, [L], 0.1), ref)


def test_fold_over_buckets_equals_one_shot():
    g = synth.rng(15)
    L, D = 70, 32
    k, v = _cells(L, 1, D, oracle.F16, g)
    c, keep = _tiered(k, v, 20, oracle.F16, 1, D)
    qd = g.standard_normal(D)
    m1, l1, a1 = oracle.attn_partial(c, 0, 0, qd, 0.3, 0, L)
    cuts = [0, 5, 5, 31, 32, 69, L]                         # includes an empty bucket
    m, l, acc = -math.inf, 0.0, np.zeros(D)
    for a, b in zip(cuts[:-1], cuts[1:]):
        mb, lb, ab = oracle.attn_partial(c, 0, 0, qd, 0.3, a, b)
        if a == b:
            assert mb == -math.inf and lb == 0 and (ab == 0).all()
        m, l, acc = oracle.fold(m, l, acc, mb, lb, ab)
    assert m == m1
    np.testing.assert_allclose(l, l1, rtol=1e-13)
    np.testing.assert_allclose(acc / l, a1 / l1, rtol=1e-12, atol=1e-14)
    # and against scipy's softmax over the union of the buckets
    K = _decode_values(k, oracle.F16, 1, D)[:, 0]
    V = _decode_values(v, oracle.F16, 1, D)[:, 0]
    np.testing.assert_allclose(acc / l, scipy.special.softmax(0.3 * K @ qd) @ V, rtol=1e-12, atol=1e-14)


def test_prefill_matches_scipy_with_mask():
    g = synth.rng(16)
    Hq, Hkv, D, L, R, pos0 = 6, 3, 32, 26, 7, 19
    k, v = _cells(L, Hkv, D, oracle.BF16, g)
    c, keep = _tiered(k, v, 9, oracle.BF16, Hkv, D)
    q = synth.normal_bits((R, Hq, D), "bf16", g)
    out = oracle.attn_prefill(c, q, oracle.BF16, R, pos0, Hq, L, 0.2)
    K = _decode_values(k, oracle.BF16, Hkv, D)
    V = _decode_values(v, oracle.BF16, Hkv, D)
    Q = _decode_values(q.reshape(R, -1).view(np.uint8), oracle.BF16, Hq, D)
    for i in range(R):
        mask = np.arange(L) <= pos0 + i
        for h in range(Hq):
            s = 0.2 * (K[:, h // 2, :] @ Q[i, h])
            s[~mask] = -np.inf
            np.testing.assert_allclose(out[i, h], scipy.special.softmax(s) @ V[:, h // 2, :],
                                       rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- q8_0 write path

def test_half_rounding_matches_numpy_on_many_values():
    g = synth.rng(31)
    x = np.concatenate([g.standard_normal(20000).astype(np.float32) * s
                        for s in (1e-6, 1e-3, 1.0, 100.0, 30000.0)])
    x = np.concatenate([x, np.float32([65504.0, 65519.0, 65520.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26])])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = np.array([oracle.float_to_half_bits(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, ref)


def test_q8_0_quantise_hand_block():
    # amax 127 gives d = 1 exactly: the codes are the values themselves
    x = np.arange(-16, 16, dtype=np.float32) * 4.0
    x[0] = -127.0
    blk = oracle.quantize_q8_0_block(x)
    assert blk[0:2].view(np.uint16)[0] == 0x3C00                        # fp16 1.0
    assert np.array_equal(blk[2:].view(np.int8), x.astype(np.int8))
    zero = oracle.quantize_q8_0_block(np.zeros(32, np.float32))
    assert (zero == 0).all()
    # ties round away from zero: x = 0.5 * d
    x = np.zeros(32, np.float32)
    x[0], x[1], x[2] = 127.0, 0.5, -0.5
    q = oracle.quantize_q8_0_block(x)[2:].view(np.int8)
    assert q[1] == 1 and q[2] == -1


def test_q8_0_quantise_error_bound_and_scale():
    g = synth.rng(32)
    for _ in range(200):
        x = (g.standard_normal(32) * g.uniform(1e-3, 50)).astype(np.float32)
        blk = oracle.quantize_q8_0_block(x)
        d16 = float(blk[0:2].view(np.float16)[0])
        q = blk[2:].view(np.int8).astype(np.float64)
        amax = float(np.abs(x).max())
        assert np.abs(q).max() == 127                                    # the max hits the end code
        assert abs(d16 - amax / 127) <= 2 ** -11 * amax / 127            # fp16 rounding of d
        d32 = np.float32(amax) / np.float32(127)
        assert np.all(np.abs(x - d32 * q) <= 0.5 * d32 * (1 + 1e-6))     # half a step


def test_append_places_cells_in_their_tiers():
    g = synth.rng(33)
    H, D, N, cap, n_new, pos0 = 2, 64, 10, 30, 8, 6
    for dt in (oracle.F16, oracle.BF16, oracle.Q8_0):
        src_dt = oracle.BF16 if dt == oracle.Q8_0 else dt
        name = "bf16" if src_dt == oracle.BF16 else "f16"
        kn = synth.normal_bits((n_new, H * D), name, g).view(np.uint8).reshape(n_new, -1).copy()
        vn = synth.normal_bits((n_new, H * D), name, g).view(np.uint8).reshape(n_new, -1).copy()
        rb = oracle.row_bytes(dt, H, D)
        kh = np.zeros((N, rb), np.uint8); vh = np.zeros((N, rb), np.uint8)
        kt = np.zeros((cap - N, rb), np.uint8); vt = np.zeros((cap - N, rb), np.uint8)
        oracle.append_kv(kn, vn, src_dt, n_new, pos0, H, D, kh, vh, kt, vt, dt, N)
        # untouched rows stay zero; written rows decode back to the inputs
        assert (kh[:pos0] == 0).all() and (kt[pos0 + n_new - N:] == 0).all()
        for t in range(n_new):
            j = pos0 + t
            row = kh[j] if j < N else kt[j - N]
            for h in range(H):
                got = oracle.load_head(row, dt, D, h)
                src = (kn[t].view(np.uint16)[h * D:(h + 1) * D])
                x = (src.view(np.float16).astype(np.float64) if src_dt == oracle.F16 else
                     torch.from_numpy(src.view(np.int16).copy()).view(torch.bfloat16).double().numpy())
                if dt == oracle.Q8_0:
                    # half a quantisation step, plus the fp16 rounding of d times |q| <= 127
                    step = np.abs(x).reshape(-1, 32).max(axis=1) / 127
                    bound = (0.5 + 127 * 2.0 ** -11) * step[:, None] + 1e-12
                    assert np.all(np.abs(got - x).reshape(-1, 32) <= bound)
                else:
                    assert np.array_equal(got, x)


# ---------------------------------------------------------------- canonical fragments

# vLLM gpu_worker.py, _build_copy_plan and _fill_canonical_ops: the expected lists
# below are written out by hand from the run definitions, not computed.

_TWO_RUNS = [(64, 1024, 0, 300, 3, 100),      # 3 fragments of 100 B: local 64 + 1024 i, canonical 300 i
             (5000, 200, 2000, 40, 2, 32)]    # 2 fragments of 32 B: local 5000 + 200 i, canonical 2000 + 40 i


def test_copy_plan_gpu_to_cpu_hand_written():
    fs, fd, fz = oracle.copy_plan(_TWO_RUNS, True)
    # source = worker-local offsets, destination = canonical offsets, run by run
    assert fs.tolist() == [64, 1088, 2112, 5000, 5200]
    assert fd.tolist() == [0, 300, 600, 2000, 2040]
    assert fz.tolist() == [100, 100, 100, 32, 32]


def test_copy_plan_cpu_to_gpu_hand_written():
    fs, fd, fz = oracle.copy_plan(_TWO_RUNS, False)
    # source = canonical offsets, destination = worker-local offsets
    assert fs.tolist() == [0, 300, 600, 2000, 2040]
    assert fd.tolist() == [64, 1088, 2112, 5000, 5200]
    assert fz.tolist() == [100, 100, 100, 32, 32]


def test_copy_plan_empty_run_contributes_nothing():
    fs, fd, fz = oracle.copy_plan([(0, 8, 0, 8, 0, 8), (16, 0, 32, 0, 1, 4)], True)
    assert (fs.tolist(), fd.tolist(), fz.tolist()) == ([16], [32], [4])


def test_fragment_ptrs_hand_written_block_major():
    os_, od, oz = oracle.fragment_ptrs([1000, 50000], [7000, 90000], [0, 300], [10, 20], [300, 600])
    # block 0's two fragments, then block 1's
    assert os_.tolist() == [1000, 1300, 50000, 50300]
    assert od.tolist() == [7010, 7020, 90010, 90020]
    assert oz.tolist() == [300, 600, 300, 600]


def _head_major_runs(tokens, heads, slice_bytes):
    """One run per head: its `tokens` slices leave the token-major block with the
    row stride and pack contiguously in the head-major block."""
    return [(h * slice_bytes, heads * slice_bytes, h * tokens * slice_bytes, slice_bytes, tokens,
             slice_bytes) for h in range(heads)]


def test_canonical_copy_is_the_head_major_transpose():
    # 6 blocks of 16 tokens x 8 heads x 256 B (128 fp16 dims): the canonical host block is
    # the token-major device block with its token and head axes exchanged.
    g = synth.rng(37)
    T, H, S, nb = 16, 8, 256, 6
    page = T * H * S
    local = g.integers(0, 256, size=(nb, T, H, S), dtype=np.uint8)
    canon = np.zeros((nb, H, T, S), np.uint8)
    runs = _head_major_runs(T, H, S)
    fs, fd, fz = oracle.copy_plan(runs, True)
    lb = np.uint64(local.ctypes.data) + np.arange(nb, dtype=np.uint64) * np.uint64(page)
    cb = np.uint64(canon.ctypes.data) + np.arange(nb, dtype=np.uint64) * np.uint64(page)
    oracle.swap_blocks(*oracle.fragment_ptrs(lb, cb, fs, fd, fz))
    for b in range(nb):
        assert np.array_equal(canon[b], local[b].reshape(T, H, S).transpose(1, 0, 2))
    # and back: canonical -> a fresh local buffer restores the token-major blocks
    back = np.zeros_like(local)
    bb = np.uint64(back.ctypes.data) + np.arange(nb, dtype=np.uint64) * np.uint64(page)
    fs, fd, fz = oracle.copy_plan(runs, False)
    oracle.swap_blocks(*oracle.fragment_ptrs(cb, bb, fs, fd, fz))
    assert np.array_equal(back, local)


def test_canonical_copy_with_a_padded_local_row():
    # local rows padded to 3 heads' worth of slices for 2 heads: the padding slice of
    # every token is never read, and the canonical block is still the transpose.
    g = synth.rng(38)
    T, H, S = 4, 2, 16
    local = g.integers(0, 256, size=(T, 3, S), dtype=np.uint8)
    canon = np.zeros((H, T, S), np.uint8)
    runs = [(h * S, 3 * S, h * T * S, S, T, S) for h in range(H)]
    fs, fd, fz = oracle.copy_plan(runs, True)
    oracle.swap_blocks(*oracle.fragment_ptrs([local.ctypes.data], [canon.ctypes.data], fs, fd, fz))
    assert np.array_equal(canon, local[:, :H, :].transpose(1, 0, 2))


# ---------------------------------------------------------------- sparse rows (QSA staged prefill)

def test_staging_policy_golden_cases():
    path = __file__.replace("test_oracle_pins.py", "golden/staging_policy.txt")
    cases = [list(map(int, ln.split())) for ln in open(path) if ln.strip() and not ln.startswith("#")]
    assert cases
    for rows, k_pad, npu, ps, want in cases:
        assert oracle.staging_worthwhile(rows, k_pad, npu, ps) == bool(want)
        assert not oracle.staging_worthwhile(rows, k_pad, npu, ps, enabled=False)
    # the boundary is strict: rows * k_pad == 2 * pages * page_size stays direct
    assert not oracle.staging_worthwhile(2, 64, 1, 64)
    assert oracle.staging_worthwhile(2, 65, 1, 64)


def _paged(pages, ps, H, D, dtype, g):
    raw_k, raw_v = _cells(pages * ps, H, D, dtype, g)
    return raw_k.reshape(pages, ps, -1), raw_v.reshape(pages, ps, -1)


def _sparse_ref(kp, vp, dtype, ps, H, D, bt, npu, idx, Q, Hq, scale):
    """numpy/scipy brute force: gather each row's selected positions by page
    table, softmax over them, weight V."""
    K = _decode_values(kp.reshape(-1, kp.shape[-1]), dtype, H, D).reshape(kp.shape[0], ps, H, D)
    V = _decode_values(vp.reshape(-1, vp.shape[-1]), dtype, H, D).reshape(kp.shape[0], ps, H, D)
    G = Hq // H
    out = np.zeros((idx.shape[0], Hq, D))
    for r in range(idx.shape[0]):
        pos = [int(p) for p in idx[r] if 0 <= p < npu * ps]
        if not pos:
            continue
        pg = np.array([bt[p // ps] for p in pos])
        sl = np.array([p % ps for p in pos])
        for h in range(Hq):
            kk = K[pg, sl, h // G, :]
            vv = V[pg, sl, h // G, :]
            p = scipy.special.softmax(scale * (kk @ Q[r, h]))
            out[r, h] = p @ vv
    return out


@pytest.mark.parametrize("dtype", [oracle.F16, oracle.BF16])
def test_sparse_rows_match_scipy_bruteforce(dtype):
    g = synth.rng(61, dtype)
    pages, ps, H, D, Hq, rows, k_pad, npu = 7, 4, 2, 32, 6, 5, 12, 6
    kp, vp = _paged(pages, ps, H, D, dtype, g)
    bt = g.permutation(pages).astype(np.int32)
    idx = g.integers(-1, npu * ps + 3, size=(rows, k_pad)).astype(np.int32)   # -1 pads, some past the pages
    idx[0, :] = -1                                                          # a row with no selection
    idx[1, 1:] = -1                                                         # a row with one
    qname = "bf16" if dtype == oracle.BF16 else "f16"
    q = synth.normal_bits((rows, Hq, D), qname, g)
    scale = 1 / math.sqrt(D)
    got = oracle.attn_sparse_rows(kp, vp, dtype, ps, H, D, bt, npu, idx, q, dtype, Hq, scale)
    Q = _decode_values(q.reshape(rows, -1).view(np.uint8), dtype, Hq, D)
    ref = _sparse_ref(kp, vp, dtype, ps, H, D, bt, npu, idx, Q, Hq, scale)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)
    assert np.all(got[0] == 0.0)
    j = int(idx[1, 0])
    if 0 <= j < npu * ps:                                                   # one selection: o = v exactly
        V = _decode_values(vp.reshape(-1, vp.shape[-1]), dtype, H, D).reshape(pages, ps, H, D)
        for h in range(Hq):
            assert np.array_equal(got[1, h], V[bt[j // ps], j % ps, h // (Hq // H)])


def test_sparse_rows_padding_order_and_duplicates():
    g = synth.rng(62)
    pages, ps, H, D, Hq, k_pad, npu = 6, 8, 2, 64, 4, 20, 6
    kp, vp = _paged(pages, ps, H, D, oracle.F16, g)
    bt = g.permutation(pages).astype(np.int32)
    base = g.choice(npu * ps, size=k_pad, replace=False).astype(np.int32)
    q = synth.normal_bits((1, Hq, D), "f16", g)
    scale = 0.125
    a = oracle.attn_sparse_rows(kp, vp, oracle.F16, ps, H, D, bt, npu, base[None], q, oracle.F16, Hq, scale)
    padded = np.concatenate([g.permutation(base), np.full(12, -1, np.int32)])[None]
    b = oracle.attn_sparse_rows(kp, vp, oracle.F16, ps, H, D, bt, npu, padded, q, oracle.F16, Hq, scale)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-14)
    # a position listed twice weighs twice: equal to duplicating it in the brute force
    dup = np.concatenate([base, base[:1]])[None]
    c = oracle.attn_sparse_rows(kp, vp, oracle.F16, ps, H, D, bt, npu, dup, q, oracle.F16, Hq, scale)
    Q = _decode_values(q.reshape(1, -1).view(np.uint8), oracle.F16, Hq, D)
    ref = _sparse_ref(kp, vp, oracle.F16, ps, H, D, bt, npu, dup, Q, Hq, scale)
    np.testing.assert_allclose(c, ref, rtol=1e-12, atol=1e-13)
    assert np.abs(c - a).max() > 1e-6


def test_sparse_rows_over_all_earlier_positions_is_causal_prefill():
    # identity page table, row i selects every position <= its own: the causal prefill row
    g = synth.rng(63)
    pages, ps, H, D, Hq, rows = 5, 8, 2, 32, 4, 6
    L = pages * ps
    kp, vp = _paged(pages, ps, H, D, oracle.F16, g)
    pos0 = L - rows
    idx = np.full((rows, L), -1, np.int32)
    for i in range(rows):
        idx[i, : pos0 + i + 1] = np.arange(pos0 + i + 1)
    q = synth.normal_bits((rows, Hq, D), "f16", g)
    got = oracle.attn_sparse_rows(kp, vp, oracle.F16, ps, H, D, np.arange(pages, dtype=np.int32), pages,
                                  idx, q, oracle.F16, Hq, 0.2)
    k = np.ascontiguousarray(kp.reshape(L, -1))
    v = np.ascontiguousarray(vp.reshape(L, -1))
    c, keep = _tiered(k, v, L, oracle.F16, H, D)
    ref = oracle.attn_prefill(c, q, oracle.F16, rows, pos0, Hq, L, 0.2)
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-14)
