"""GPU parity of kvo_swap_blocks_batch (and the descriptors kvo_sub_block_ptrs
builds) against the oracle's memcpy swap: bit-exact, plus the D2H-then-H2D
round trip and untouched canary bytes."""
import numpy as np
import pytest

import oracle
from helpers import pinned, torch
from host_ram_tiered_gb300 import kvo, synth

pytestmark = pytest.mark.gpu


def _ptrs(ids, bpc, skip, base, stride, row_bytes, n):
    ids = np.ascontiguousarray(ids, np.int64)
    out = np.zeros(n, np.int64)
    kvo.kvo_sub_block_ptrs(ids.ctypes.data, len(ids), bpc, skip, base, stride, row_bytes,
                           out.ctypes.data, n)
    exp = oracle.sub_block_ptrs(ids, bpc, skip, base, stride, row_bytes, n)
    assert np.array_equal(out.view(np.uint64), exp)
    return out


class Pools:
    """n_tensors paged device tensors [gpu_blocks][page] and host tensors
    [host_chunks][row_stride] (row = bpc pages), each its own allocation
    region inside one device / one pinned slab."""

    def __init__(self, n_tensors, gpu_blocks, host_chunks, page, bpc, row_stride, seed):
        t = torch()
        self.n_tensors, self.page, self.bpc, self.row_stride = n_tensors, page, bpc, row_stride
        self.gpu_bytes = gpu_blocks * page
        self.host_bytes = host_chunks * row_stride
        self.dev = t.empty(n_tensors * self.gpu_bytes, dtype=t.uint8, device="cuda")
        self.host = pinned(n_tensors * self.host_bytes)
        g = synth.rng(seed, 1)
        init_dev = np.empty(n_tensors * self.gpu_bytes, np.uint8)
        synth.fill_bytes_large(init_dev, seed, 2)
        self.dev.copy_(t.from_numpy(init_dev))
        synth.fill_bytes_large(self.host.numpy(), seed, 3)
        self.init_dev = init_dev

    def dev_base(self, i):
        return self.dev.data_ptr() + i * self.gpu_bytes

    def host_base(self, i):
        return self.host.data_ptr() + i * self.host_bytes


def _descs(pools, gpu_ids, host_ids, skip, h2d, n):
    """Descriptors of one direction for every tensor (transfer_async order)."""
    src, dst = [], []
    for i in range(pools.n_tensors):
        hp = _ptrs(host_ids, pools.bpc, skip, pools.host_base(i), pools.row_stride,
                   pools.bpc * pools.page, n)
        gp = _ptrs(gpu_ids, 1, 0, pools.dev_base(i), pools.page, pools.page, n)
        src.append(hp if h2d else gp)
        dst.append(gp if h2d else hp)
    return np.concatenate(src), np.concatenate(dst)


def _pinned_i64(a):
    buf = pinned(a.size * 8)
    buf.numpy().view(np.int64)[:a.size] = a
    return buf


def _swap(src, dst, page, flags):
    n = src.size
    s, d = _pinned_i64(src), _pinned_i64(dst)
    z = _pinned_i64(np.full(n, page, np.int64))
    kvo.kvo_swap_blocks_batch(s, d, z, n, flags)
    torch().cuda.synchronize()


def _host_addr_map(pools):
    """numpy arrays of the host slab and a device mirror for the oracle."""
    return pools.host.numpy()


def _oracle_swap(src, dst, page, base_map):
    """Run the oracle memcpy swap on host mirrors: addresses are translated
    from (device | pinned) ranges to numpy mirror ranges."""
    (dev_base, dev_mirror), (host_base, host_mirror) = base_map

    def tr(a):
        out = np.empty_like(a, dtype=np.uint64)
        in_dev = (a >= dev_base) & (a < dev_base + dev_mirror.size)
        out[in_dev] = (a[in_dev] - dev_base).astype(np.uint64) + np.uint64(dev_mirror.ctypes.data)
        out[~in_dev] = (a[~in_dev] - host_base).astype(np.uint64) + np.uint64(host_mirror.ctypes.data)
        return out

    oracle.swap_blocks(tr(src), tr(dst), np.full(src.size, page, np.int64))


@pytest.mark.parametrize("mode", [0, kvo.KVO_SWAP_FORCE_SM, kvo.KVO_SWAP_FORCE_CE])
def test_c1_swap_64_blocks_round_trip(mode):
    # 2 layers x K,V; 32 KiB pages (16 tokens x 8 heads x 128 x fp16); pools of 128.
    page, nt = 32768, 4
    pools = Pools(nt, 128, 128, page, 1, page, seed=1234)
    g = synth.rng(1234, 10)
    gpu_ids = g.permutation(128)[:64]
    host_ids = g.permutation(128)[:64]
    dev_mirror = pools.init_dev.copy()
    host_mirror = pools.host.numpy().copy()
    bm = ((pools.dev.data_ptr(), dev_mirror), (pools.host.data_ptr(), host_mirror))
    # D2H
    src, dst = _descs(pools, gpu_ids, host_ids, 0, False, 64)
    _swap(src, dst, page, kvo.KVO_SWAP_D2H | mode)
    _oracle_swap(src, dst, page, bm)
    assert np.array_equal(pools.host.numpy(), host_mirror)
    # H2D into a cleared device pool: the blocks come back byte-identical
    pools.dev.zero_()
    dev_mirror[:] = 0
    src, dst = _descs(pools, gpu_ids, host_ids, 0, True, 64)
    _swap(src, dst, page, kvo.KVO_SWAP_H2D | kvo.KVO_SWAP_SRC_ORDER_ANY | mode)
    _oracle_swap(src, dst, page, bm)
    got = pools.dev.cpu().numpy()
    assert np.array_equal(got, dev_mirror)
    # round trip: the swapped blocks equal the original device blocks
    for i in range(nt):
        o = pools.init_dev[i * pools.gpu_bytes:(i + 1) * pools.gpu_bytes].reshape(128, page)
        r = got[i * pools.gpu_bytes:(i + 1) * pools.gpu_bytes].reshape(128, page)
        assert np.array_equal(r[gpu_ids], o[gpu_ids])
        others = np.setdiff1d(np.arange(128), gpu_ids)
        assert (r[others] == 0).all()


@pytest.mark.parametrize("page,n_tensors,n_blocks", [(2048, 8, 301), (32768, 4, 77)])
def test_c2_shape_swap_bpc4_skip1(page, n_tensors, n_blocks):
    # blocks_per_chunk 4, skip 1 on the first chunk, host row stride 1.5 x row;
    # a ragged block count (not a multiple of 4).
    bpc = 4
    need = -(-(n_blocks + 1) // bpc)
    pools = Pools(n_tensors, 512, need + 20, page, bpc, bpc * page * 3 // 2, seed=1235)
    g = synth.rng(1235, 11)
    gpu_ids = g.permutation(512)[:n_blocks]
    host_ids = g.permutation(need + 20)[:need]
    dev_mirror = pools.init_dev.copy()
    host_mirror = pools.host.numpy().copy()
    bm = ((pools.dev.data_ptr(), dev_mirror), (pools.host.data_ptr(), host_mirror))
    src, dst = _descs(pools, gpu_ids, host_ids, 1, False, n_blocks)
    _swap(src, dst, page, kvo.KVO_SWAP_D2H)
    _oracle_swap(src, dst, page, bm)
    assert np.array_equal(pools.host.numpy(), host_mirror)      # incl. the untouched 1/3 of rows
    pools.dev.zero_()
    dev_mirror[:] = 0
    src, dst = _descs(pools, gpu_ids, host_ids, 1, True, n_blocks)
    _swap(src, dst, page, kvo.KVO_SWAP_H2D | kvo.KVO_SWAP_SRC_ORDER_ANY)
    _oracle_swap(src, dst, page, bm)
    assert np.array_equal(pools.dev.cpu().numpy(), dev_mirror)


def test_unaligned_and_odd_sizes_with_canaries():
    t = torch()
    g = synth.rng(9)
    dev = t.zeros(1 << 20, dtype=t.uint8, device="cuda")
    host = pinned(1 << 20)
    hn = host.numpy()
    hn[:] = g.integers(0, 256, size=hn.size, dtype=np.uint8)
    sizes = np.array([1, 3, 8, 24, 1000, 4096, 4100, 16, 77, 65536], np.int64)
    soffs = np.array([5, 64, 131, 256, 1001, 8192, 20000, 30001, 40003, 100000], np.int64)
    doffs = np.array([0, 17, 40, 200, 4000, 12288, 20480, 30000, 40000, 200000], np.int64)
    src = soffs + host.data_ptr()
    dst = doffs + dev.data_ptr()
    s, d, z = _pinned_i64(src), _pinned_i64(dst), _pinned_i64(sizes)
    kvo.kvo_swap_blocks_batch(s, d, z, sizes.size, kvo.KVO_SWAP_H2D | kvo.KVO_SWAP_FORCE_SM)
    t.cuda.synchronize()
    got = dev.cpu().numpy()
    exp = np.zeros(1 << 20, np.uint8)
    oracle.swap_blocks(soffs.astype(np.uint64) + np.uint64(hn.ctypes.data),
                       doffs.astype(np.uint64) + np.uint64(exp.ctypes.data), sizes)
    assert np.array_equal(got, exp)


def test_copy_engine_merges_contiguous_runs():
    t = torch()
    dev = t.zeros(1 << 22, dtype=t.uint8, device="cuda")
    host = pinned(1 << 22)
    host.numpy()[:] = synth.rng(3).integers(0, 256, size=1 << 22, dtype=np.uint8)
    n = 64
    sizes = np.full(n, 1 << 16, np.int64)
    src = host.data_ptr() + np.arange(n, dtype=np.int64) * (1 << 16)
    dst = dev.data_ptr() + np.arange(n, dtype=np.int64) * (1 << 16)
    kvo.kvo_swap_blocks_batch(_pinned_i64(src), _pinned_i64(dst), _pinned_i64(sizes), n,
                              kvo.KVO_SWAP_H2D | kvo.KVO_SWAP_FORCE_CE)
    t.cuda.synchronize()
    assert np.array_equal(dev.cpu().numpy(), host.numpy())


def test_descriptor_arrays_must_be_mapped():
    t = torch()
    dev = t.zeros(4096, dtype=t.uint8, device="cuda")
    pageable = np.array([dev.data_ptr()], np.int64)
    with pytest.raises(kvo.KvoError) as e:
        kvo.kvo_swap_blocks_batch(pageable.ctypes.data, pageable.ctypes.data, pageable.ctypes.data,
                                  1, kvo.KVO_SWAP_FORCE_SM)
    assert e.value.status == -3


def _equal_chunked(a: np.ndarray, b: np.ndarray, chunk: int = 1 << 28) -> bool:
    """Byte equality of two large flat arrays without a full-size temporary."""
    if a.size != b.size:
        return False
    return all(np.array_equal(a[i:i + chunk], b[i:i + chunk]) for i in range(0, a.size, chunk))


@pytest.mark.parametrize("page", [32768, 2048])
def test_c2_full_size_swap_whole_pools(page):
    # The full 32-layer offload swap, in the launch configuration the benchmark times:
    # 64 tensors (32 layers x K,V), 2048 blocks per direction, bpc 4, skip 1, host stride
    # 1.5 x row.  Every byte of both pools is compared with the oracle's memcpy run on host
    # mirrors: D2H, then H2D from a host pool refilled with fresh bytes, so that the H2D
    # direction writes values the device never held.
    from bench import swap_setup, swap_run
    t = torch()
    st = swap_setup(page, seed=1235)
    host, dev = st["host"], st["dev"]
    host_np_ = host.numpy()
    dev_mirror = st["init_dev"]                 # the device pool's initial bytes
    host_mirror = host_np_.copy()
    gp, hp = st["d2h_src_np"], st["d2h_dst_np"]
    dev_base, host_base = dev.data_ptr(), host.data_ptr()

    def on(mirror, addrs, base):
        return (addrs - base).astype(np.uint64) + np.uint64(mirror.ctypes.data)

    sizes = np.full(st["n_desc"], page, np.int64)
    swap_run(st, h2d=False)
    t.cuda.synchronize()
    oracle.swap_blocks(on(dev_mirror, gp, dev_base), on(host_mirror, hp, host_base), sizes)
    assert _equal_chunked(host_np_, host_mirror)
    assert _equal_chunked(dev.cpu().numpy(), dev_mirror)
    synth.fill_bytes_large(host_np_, 1235, 7)
    np.copyto(host_mirror, host_np_)
    swap_run(st, h2d=True)
    t.cuda.synchronize()
    oracle.swap_blocks(on(host_mirror, hp, host_base), on(dev_mirror, gp, dev_base), sizes)
    assert _equal_chunked(dev.cpu().numpy(), dev_mirror)
    assert _equal_chunked(host_np_, host_mirror)


@pytest.mark.parametrize("gpu_to_cpu", [True, False])
def test_canonical_fragment_swap(gpu_to_cpu):
    # A 32 KiB device block (16 tokens x 8 heads x 128 fp16) stored canonically on the
    # host head-major: fragment (token t, head h) of 256 B moves from t*2048 + h*256
    # locally to h*4096 + t*256 canonically -- 8 runs of 16 fragments each.
    t = torch()
    g = synth.rng(36, int(gpu_to_cpu))
    page, nb, pool = 32768, 24, 64
    runs = [(h * 256, 2048, h * 4096, 256, 16, 256) for h in range(8)]
    cols = [np.array([r[k] for r in runs], np.int64) for k in range(6)]
    fs, fd, fz = (np.zeros(128, np.int64) for _ in range(3))
    nf = kvo.kvo_copy_plan(*cols, len(runs), gpu_to_cpu, fs, fd, fz, 128)
    dev = t.from_numpy(g.integers(0, 256, size=pool * page, dtype=np.uint8)).cuda()
    host = pinned(pool * page)
    host.numpy()[:] = g.integers(0, 256, size=pool * page, dtype=np.uint8)
    dev_ids = g.permutation(pool)[:nb]
    host_ids = g.permutation(pool)[:nb]
    dev_b = (dev.data_ptr() + dev_ids * page).astype(np.int64)
    host_b = (host.data_ptr() + host_ids * page).astype(np.int64)
    sb, db = (dev_b, host_b) if gpu_to_cpu else (host_b, dev_b)
    n = nb * nf
    os_, od, oz = (np.zeros(n, np.int64) for _ in range(3))
    kvo.kvo_fragment_ptrs(sb, db, nb, fs[:nf], fd[:nf], fz[:nf], nf, os_, od, oz)
    dev_mirror = dev.cpu().numpy().copy()
    host_mirror = host.numpy().copy()
    kvo.kvo_swap_blocks_batch(_pinned_i64(os_), _pinned_i64(od), _pinned_i64(oz), n,
                              kvo.KVO_SWAP_D2H if gpu_to_cpu else kvo.KVO_SWAP_H2D)
    t.cuda.synchronize()
    # oracle: the same plan and descriptors, built by the oracle, on host mirrors
    es, ed, ez = oracle.copy_plan(runs, gpu_to_cpu)
    mb_dev = (np.uint64(dev_mirror.ctypes.data) + (dev_ids * page).astype(np.uint64))
    mb_host = (np.uint64(host_mirror.ctypes.data) + (host_ids * page).astype(np.uint64))
    msb, mdb = (mb_dev, mb_host) if gpu_to_cpu else (mb_host, mb_dev)
    rs, rd, rz = oracle.fragment_ptrs(msb, mdb, es, ed, ez)
    oracle.swap_blocks(rs, rd, rz)
    got_host, got_dev = host.numpy(), dev.cpu().numpy()
    assert np.array_equal(got_host, host_mirror)
    assert np.array_equal(got_dev, dev_mirror)
    # the meaning, independent of the plan: a canonical host block is its device block with
    # the token and head axes exchanged ([16][8][256 B] token-major <-> [8][16][256 B] head-major)
    for di, hi in zip(dev_ids, host_ids):
        d_blk = got_dev[di * page:(di + 1) * page].reshape(16, 8, 256)
        h_blk = got_host[hi * page:(hi + 1) * page].reshape(8, 16, 256)
        assert np.array_equal(h_blk, d_blk.transpose(1, 0, 2))
