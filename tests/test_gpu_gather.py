"""pa_gather_checksum(_fp8): the decode kernels' gather of K/V tiles without the attention.

The expected value is the checksum's plain definition, computed here with numpy from the
host caches: for every (sequence, KV head), the XOR of all 32-bit words of its K and V rows
t < context length, reached through the block table (a bf16 row is 64 words, an E4M3 row
32).  XOR does not depend on the order of the work, so the result is compared bit for bit.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_helpers import dev, dev_bf16
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


def expected_xor(k_cache, v_cache, block_tables, context_lens, max_context_len):
    """[S, Hkv] uint32: XOR of the words of each (sequence, KV head)'s K and V rows."""
    S = len(context_lens)
    Hkv = k_cache.shape[1]
    out = np.zeros((S, Hkv), dtype=np.uint32)
    for s in range(S):
        n = int(min(max(int(context_lens[s]), 0), max_context_len))
        if n == 0:
            continue
        blocks = block_tables[s, :(n + 15) // 16]
        for g in range(Hkv):
            for cache in (k_cache, v_cache):
                rows = np.ascontiguousarray(cache[blocks, g]).reshape(-1, 128)[:n]
                out[s, g] ^= np.bitwise_xor.reduce(rows.view(np.uint32), axis=None)
    return out


def run(pa, w, kc, vc, bt, ctx, maxctx):
    put = dev if kc.dtype == np.uint8 else dev_bf16
    got = pa.gather_checksum(put(kc), put(vc), dev(bt), dev(ctx), maxctx, w.num_q_heads)
    torch.cuda.synchronize()
    return got.cpu().numpy().view(np.uint32)


def e4m3_caches(w, seed):
    """Seeded random code bytes in the E4M3 cache layout (the checksum reads them as stored)."""
    rng = np.random.default_rng(seed)
    shape = (w.num_blocks, w.num_kv_heads, 16, 128)
    return rng.integers(0, 256, size=shape, dtype=np.uint8), rng.integers(0, 256, size=shape, dtype=np.uint8)


@pytest.mark.parametrize("name", W.WORKLOADS)
def test_gather_checksum_matches_definition(pa, name):
    w = W.make(name)
    want = expected_xor(w.k_cache[0], w.v_cache[0], w.block_tables, w.context_lens, w.max_context_len)
    got = run(pa, w, w.k_cache[0], w.v_cache[0], w.block_tables, w.context_lens, w.max_context_len)
    assert np.array_equal(got, want)
    rc, flags = pa.get_device_status()
    assert rc == 0 and flags == 0, (rc, hex(flags))


@pytest.mark.parametrize("name", W.WORKLOADS)
def test_gather_checksum_fp8_matches_definition(pa, name):
    w = W.make(name)
    k8, v8 = e4m3_caches(w, 3100 + W.WORKLOADS.index(name))
    want = expected_xor(k8, v8, w.block_tables, w.context_lens, w.max_context_len)
    got = run(pa, w, k8, v8, w.block_tables, w.context_lens, w.max_context_len)
    assert np.array_equal(got, want)
    rc, flags = pa.get_device_status()
    assert rc == 0 and flags == 0, (rc, hex(flags))


def test_gather_checksum_ignores_entries_past_the_context(pa):
    """Table entries past each context are out of range here; they are never read or flagged,
    and the checksum is unchanged.  Stale cache rows past the context (NaN canaries) do not
    enter it."""
    w = W.make("mix64")
    bt = w.block_tables.copy()
    for s in range(w.num_seqs):
        bt[s, (int(w.context_lens[s]) + 15) // 16:] = w.num_blocks + 7
    want = expected_xor(w.k_cache[0], w.v_cache[0], w.block_tables, w.context_lens, w.max_context_len)
    got = run(pa, w, w.k_cache[0], w.v_cache[0], bt, w.context_lens, w.max_context_len)
    assert np.array_equal(got, want)
    rc, flags = pa.get_device_status()
    assert rc == 0 and flags == 0, (rc, hex(flags))


def test_gather_checksum_flags_bad_block_ids_and_xors_into_out(pa):
    """An out-of-range id inside a context skips that block and raises the block-id flag; the
    output is XORed into, so a second call on the same buffer returns it to zero."""
    w = W.make("tiny")
    bt = w.block_tables.copy()
    bt[1, 1] = -3
    out = torch.zeros((w.num_seqs, w.num_kv_heads), dtype=torch.int32, device="cuda")
    for _ in range(2):
        pa.gather_checksum(dev_bf16(w.k_cache[0]), dev_bf16(w.v_cache[0]), dev(bt),
                           dev(w.context_lens), w.max_context_len, w.num_q_heads, out_xor=out)
    torch.cuda.synchronize()
    assert not out.any()
    rc, flags = pa.get_device_status()
    assert flags & pa.PA_FLAG_BLOCK_ID_OOB
