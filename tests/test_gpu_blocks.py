"""Whole-block copies (pa_copy_blocks) through the C ABI, against the oracle's block copy.

Copy-on-write inside one device pool, swap out to page-locked host memory and swap in to other
device blocks: every destination pool must equal the oracle's bit for bit, and every block no
pair names must be left untouched.
"""

from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DeviceLayer, host_bits
from paged_kv_cache_244_gb300 import _build
from paged_kv_cache_244_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    _build.build()
    from paged_kv_cache_244_gb300 import binding
    return binding


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


def check_status_clean(pa):
    rc, flags = pa.get_device_status()
    assert rc == 0 and flags == 0, (rc, hex(flags))


def random_pools(rng, n, num_blocks, hkv):
    """n pools of random bf16 bit patterns (NaNs and signed zeros included)."""
    return [rng.integers(0, 1 << 16, (num_blocks, hkv, W.BLOCK_SIZE, W.HEAD_DIM), dtype=np.uint16)
            for _ in range(n)]


def to_dev(a):
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()


def bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("hkv", [1, 2, 4, 8])
def test_copy_on_write_in_one_pool(pa, orc, hkv):
    """K and V of 28 layers (56 caches), 40 pairs from used blocks to fresh ones."""
    rng = np.random.default_rng(100 + hkv)
    pools = random_pools(rng, 56, 96, hkv)
    frm = rng.permutation(48)[:40]
    to = 48 + rng.permutation(48)[:40]
    pairs = np.stack([frm, to], axis=1).astype(np.int64)
    want = [p.copy() for p in pools]
    assert orc.copy_blocks(want, want, pairs) == 0
    dev = [to_dev(p) for p in pools]
    pa.copy_blocks(dev, dev, torch.from_numpy(pairs).cuda())
    torch.cuda.synchronize()
    for c in range(56):
        assert np.array_equal(bits(dev[c]), want[c]), c
    check_status_clean(pa)


def test_swap_out_and_in_preserves_decode(pa, orc):
    """Swap every block of the mix64 batch out to page-locked host memory, then in to other
    blocks of a fresh device pool; with the block tables remapped, decode gives the same
    output bits as before the swap."""
    w = W.make("mix64")
    d = DeviceLayer(w)
    before = pa.decode(d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens,
                       w.max_context_len, w.scale)
    used = np.unique(np.concatenate(
        [w.block_tables[s, :(int(w.context_lens[s]) + 15) // 16] for s in range(w.num_seqs)]))
    n = used.shape[0]
    host = [torch.empty((n,) + tuple(d.k_cache.shape[1:]), dtype=torch.bfloat16).pin_memory()
            for _ in range(2)]
    out_pairs = torch.from_numpy(np.stack([used, np.arange(n)], axis=1).astype(np.int64)).cuda()
    pa.copy_blocks([d.k_cache, d.v_cache], host, out_pairs)                       # swap out
    rng = np.random.default_rng(5)
    fresh = rng.permutation(w.num_blocks)[:n]
    k2 = torch.full_like(d.k_cache, float("nan"))
    v2 = torch.full_like(d.v_cache, float("nan"))
    in_pairs = torch.from_numpy(np.stack([np.arange(n), fresh], axis=1).astype(np.int64)).pin_memory()
    pa.copy_blocks(host, [k2, v2], in_pairs)                                      # swap in
    torch.cuda.synchronize()
    # host copies and device copies against the oracle
    want_host = [np.zeros((n,) + w.k_cache.shape[2:], np.uint16) for _ in range(2)]
    orc.copy_blocks([w.k_cache[0], w.v_cache[0]], want_host, np.stack([used, np.arange(n)], 1))
    assert np.array_equal(bits(host[0]), want_host[0])
    assert np.array_equal(bits(host[1]), want_host[1])
    remap = np.full(w.num_blocks, -1, np.int64)
    remap[used] = fresh
    bt = w.block_tables.copy()
    for s in range(w.num_seqs):
        nb = (int(w.context_lens[s]) + 15) // 16
        bt[s, :nb] = remap[bt[s, :nb]]
    after = pa.decode(d.q, k2, v2, torch.from_numpy(bt).cuda(), d.context_lens,
                      w.max_context_len, w.scale)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(after), host_bits(before))
    # blocks no pair named keep their fill
    untouched = np.setdiff1d(np.arange(w.num_blocks), fresh)
    assert torch.isnan(k2[torch.from_numpy(untouched).cuda()]).all()
    check_status_clean(pa)


def test_out_of_range_pairs_are_flagged_and_skipped(pa, orc):
    rng = np.random.default_rng(11)
    src = random_pools(rng, 4, 10, 2)
    dst = [np.zeros((8, 2, W.BLOCK_SIZE, W.HEAD_DIM), np.uint16) for _ in range(4)]
    pairs = np.array([[0, 0], [10, 1], [-1, 2], [3, 8], [4, -5], [9, 7]], np.int64)
    want = [x.copy() for x in dst]
    assert orc.copy_blocks(src, want, pairs) == 4
    s_dev, d_dev = [to_dev(x) for x in src], [to_dev(x) for x in dst]
    pa.copy_blocks(s_dev, d_dev, torch.from_numpy(pairs).cuda())
    rc, flags = pa.get_device_status()
    assert rc == pa.PA_ERR_DEVICE_OOB and flags == pa.PA_FLAG_BLOCK_ID_OOB
    for c in range(4):
        assert np.array_equal(bits(d_dev[c]), want[c])
    check_status_clean(pa)


def test_pageable_host_memory_is_refused(pa):
    """A pool in ordinary (pageable) host memory is refused before anything is launched."""
    dev = torch.zeros((4, 2, W.BLOCK_SIZE, W.HEAD_DIM), dtype=torch.bfloat16, device="cuda")
    pageable = torch.zeros((4, 2, W.BLOCK_SIZE, W.HEAD_DIM), dtype=torch.bfloat16)
    assert not pageable.is_pinned()
    pairs = torch.tensor([[0, 1]], dtype=torch.int64, device="cuda")
    arr = ctypes.c_void_p * 1
    dims = pa.make_dims(2, 2)
    rc = pa.lib().pa_copy_blocks(ctypes.byref(dims), 1, ctypes.cast(arr(dev.data_ptr()), ctypes.c_void_p), 4,
                                 ctypes.cast(arr(pageable.data_ptr()), ctypes.c_void_p), 4,
                                 ctypes.c_void_p(pairs.data_ptr()), 1, None)
    assert rc == pa.PA_ERR_MEMORY
    with pytest.raises(ValueError):
        pa.copy_blocks([dev], [pageable], pairs)
    torch.cuda.synchronize()
    check_status_clean(pa)


def test_copy_blocks_in_a_cuda_graph(pa, orc):
    """Captured once, replayed with new pair lists written into the same buffer."""
    rng = np.random.default_rng(12)
    pools = random_pools(rng, 6, 64, 2)
    dev = [to_dev(p) for p in pools]
    ref = [p.copy() for p in pools]
    pairs = torch.zeros((16, 2), dtype=torch.int64, device="cuda")
    pairs[:, 0] = torch.arange(16)
    pairs[:, 1] = torch.arange(16) + 16
    pa.copy_blocks(dev, dev, pairs)
    orc.copy_blocks(ref, ref, pairs.cpu().numpy())
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        pa.copy_blocks(dev, dev, pairs)
    for r in range(2):
        frm = rng.permutation(32)[:16]
        to = 32 + rng.permutation(32)[:16]
        new = np.stack([frm, to], 1).astype(np.int64)
        pairs.copy_(torch.from_numpy(new))
        graph.replay()
        orc.copy_blocks(ref, ref, new)
        torch.cuda.synchronize()
        for c in range(6):
            assert np.array_equal(bits(dev[c]), ref[c]), (r, c)
    check_status_clean(pa)
