"""The fused decode step (pa_decode_step) through the C ABI, against the fp64 oracle.

The step must equal pa_rope_kv_store (position context_len - 1, the slot at that position of
the block table) followed by pa_decode, except that q is left unrotated in memory.  Bars as
everywhere: V stores and untouched cache bytes bit-exact, rotated K within 1 bf16 ulp, output
within |gpu - oracle| <= 1e-2 + 1e-2 |oracle|.  The expected values come from the oracle's
own store followed by its own decode.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (DeviceLayer, assert_out_close, bf16_ulp_distance, dev, dev_bf16,
                         host_bits)
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


def run_step(pa, d, w, partition_tokens=None, cos_sin=None):
    P = w.partition_tokens if partition_tokens is None else partition_tokens
    out = pa.decode_step(d.q, d.k, d.v, d.cos_sin if cos_sin is None else cos_sin, d.k_cache,
                         d.v_cache, d.block_tables, d.context_lens, w.max_context_len, w.scale,
                         partition_tokens=P)
    torch.cuda.synchronize()
    return host_bits(out)


def expected(orc, w, layer=0, context_lens=None, max_pos=None, qkv=None):
    """The oracle's store then decode: (out_f64, k_cache, v_cache).  Sequences with no
    context or whose position has no cos/sin row store nothing and keep q unrotated.
    qkv replaces the layer's new-token (q, k, v)."""
    ctx = w.context_lens if context_lens is None else context_lens
    cos_sin = w.cos_sin if max_pos is None else w.cos_sin[:max_pos]
    q0, k0, v0 = (w.q[layer], w.k[layer], w.v[layer]) if qkv is None else qkv
    kc, vc = w.k_cache[layer].copy(), w.v_cache[layer].copy()
    q = q0.copy()
    pos = ctx.astype(np.int64) - 1
    live = (ctx > 0) & (pos < cos_sin.shape[0])
    if live.any():
        blk = w.block_tables[np.arange(w.num_seqs), np.maximum(pos, 0) // W.BLOCK_SIZE].astype(np.int64)
        slots = blk * W.BLOCK_SIZE + np.maximum(pos, 0) % W.BLOCK_SIZE
        q[live] = orc.rope_kv_store(q0[live], k0[live], v0[live], pos[live].astype(np.int32),
                                    cos_sin, slots[live], kc, vc)
    ref, _ = orc.decode(q, kc, vc, w.block_tables, ctx, w.scale)
    return ref, kc, vc


def check_caches(d, kc_ref, vc_ref):
    assert np.array_equal(host_bits(d.v_cache), vc_ref)
    kc = host_bits(d.k_cache)
    assert bf16_ulp_distance(kc, kc_ref).max() <= 1


@pytest.mark.parametrize("name", W.WORKLOADS)
def test_decode_step_matches_oracle(pa, orc, name):
    w = W.make(name)
    for layer in sorted({0, w.num_layers - 1}):
        d = DeviceLayer(w, layer)
        got = run_step(pa, d, w)
        ref, kc_ref, vc_ref = expected(orc, w, layer)
        assert np.array_equal(host_bits(d.q), w.q[layer])          # q is not modified
        check_caches(d, kc_ref, vc_ref)
        # outside the new slots the K cache is untouched, bit for bit
        kc = host_bits(d.k_cache)
        blk, off = np.divmod(w.slot_mapping, W.BLOCK_SIZE)
        mask = np.ones(kc.shape, bool)
        mask[blk, :, off] = False
        assert np.array_equal(kc[mask], w.k_cache[layer][mask])
        assert_out_close(got, ref, f"{name} layer {layer}")
    check_status_clean(pa)


@pytest.mark.parametrize("name", ["tiny", "mix64", "long4"])
def test_decode_step_equals_store_then_decode(pa, orc, name):
    """Same kernels' arithmetic either way: the caches and the output agree bit for bit with
    pa_rope_kv_store followed by pa_decode on the same grid."""
    w = W.make(name)
    a = DeviceLayer(w)
    got = run_step(pa, a, w)
    b = DeviceLayer(w)
    pa.rope_kv_store(b.q, b.k, b.v, b.positions, b.cos_sin, b.slot_mapping, b.k_cache, b.v_cache)
    two = pa.decode(b.q, b.k_cache, b.v_cache, b.block_tables, b.context_lens, w.max_context_len,
                    w.scale, partition_tokens=w.partition_tokens)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(a.k_cache), host_bits(b.k_cache))
    assert np.array_equal(host_bits(a.v_cache), host_bits(b.v_cache))
    assert np.array_equal(got, host_bits(two))
    check_status_clean(pa)


def test_decode_step_edge_context_lengths(pa, orc):
    """The new token first, last and alone in its block; one-token contexts; every split."""
    ctxs = [1, 2, 15, 16, 17, 31, 32, 33, 255, 256, 257, 511, 512, 513, 1000, 3]
    w = W.build("step_edges", ctxs, 400, 91, max_blocks=70)
    ref, kc_ref, vc_ref = expected(orc, w)
    for P in (0, 16, 256):
        d = DeviceLayer(w)
        got = run_step(pa, d, w, partition_tokens=P)
        check_caches(d, kc_ref, vc_ref)
        assert_out_close(got, ref, f"P={P}")
    check_status_clean(pa)


@pytest.mark.parametrize("hq,hkv", [(12, 2), (8, 8), (16, 2), (6, 2), (4, 1), (14, 2), (32, 4)])
def test_decode_step_group_sizes(pa, orc, hq, hkv):
    w = W.build("step_groups", [5, 40, 300, 700], 120, 92, num_q_heads=hq, num_kv_heads=hkv)
    ref, kc_ref, vc_ref = expected(orc, w)
    for P in (0, 64):
        d = DeviceLayer(w)
        got = run_step(pa, d, w, partition_tokens=P)
        check_caches(d, kc_ref, vc_ref)
        assert_out_close(got, ref, f"{hq}/{hkv} P={P}")
    check_status_clean(pa)


def test_decode_step_zero_context_stores_nothing(pa, orc):
    w = W.build("step_zero", [30, 50, 20], 16, 93)
    ctx = w.context_lens.copy()
    ctx[1] = 0
    ref, kc_ref, vc_ref = expected(orc, w, context_lens=ctx)
    for P in (0, 16):
        d = DeviceLayer(w)
        d.context_lens = dev(ctx)
        got = run_step(pa, d, w, partition_tokens=P)
        assert (got[1] == 0).all()
        check_caches(d, kc_ref, vc_ref)
        assert_out_close(got, ref)
    check_status_clean(pa)


def test_decode_step_position_without_rope_row_is_flagged(pa, orc):
    """n - 1 >= max_pos: that token is left as the store kernel leaves it (q unrotated,
    nothing stored), the rest of the batch is unaffected, and the flag is raised."""
    # canary 0: the slot left unwritten holds zeros (not NaN), so sequence 1's output, which
    # attends over it, is finite and comparable too
    w = W.build("step_pos", [30, 50, 20], 16, 94, canary=0)
    max_pos = 40                          # sequence 1 (position 49) has no row
    ref, kc_ref, vc_ref = expected(orc, w, max_pos=max_pos)
    d = DeviceLayer(w)
    got = run_step(pa, d, w, partition_tokens=0, cos_sin=d.cos_sin[:max_pos].contiguous())
    rc, flags = pa.get_device_status()
    assert rc == pa.PA_ERR_DEVICE_OOB and flags == pa.PA_FLAG_POSITION_OOB
    check_caches(d, kc_ref, vc_ref)
    assert_out_close(got, ref)
    check_status_clean(pa)


def test_decode_step_out_of_range_new_block_is_flagged(pa, orc):
    """The block of a sequence's new token is out of range: flagged, skipped (never written),
    the other sequences still stored and attended."""
    w = W.build("step_blk", [30, 50, 20], 16, 95)
    bt = w.block_tables.copy()
    bt[2, (20 - 1) // 16] = w.num_blocks + 7
    d = DeviceLayer(w)
    d.block_tables = dev(bt)
    before_k, before_v = host_bits(d.k_cache), host_bits(d.v_cache)
    got = run_step(pa, d, w, partition_tokens=0)
    rc, flags = pa.get_device_status()
    assert flags == pa.PA_FLAG_BLOCK_ID_OOB
    # sequences 0 and 1 as the oracle has them; sequence 2's store never happened
    ref, kc_ref, vc_ref = expected(orc, w)
    blk, off = divmod(int(w.slot_mapping[2]), W.BLOCK_SIZE)
    kc_ref[blk, :, off], vc_ref[blk, :, off] = before_k[blk, :, off], before_v[blk, :, off]
    check_caches(d, kc_ref, vc_ref)
    assert_out_close(got[:2], ref[:2])
    check_status_clean(pa)


@pytest.mark.parametrize("P", [0, 16])
def test_decode_step_replayed_from_a_cuda_graph(pa, orc, P):
    """A captured step reads whatever its frozen buffers hold at replay: new q, k and v
    overwrite the same slots and give the oracle's result for them."""
    w = W.build("step_graph", [40, 300, 700, 17], 200, 96)
    d = DeviceLayer(w)
    ws = pa.decode_workspace(d.q, d.k_cache, w.max_context_len, P)
    out = torch.empty_like(d.q)

    def call():
        pa.decode_step(d.q, d.k, d.v, d.cos_sin, d.k_cache, d.v_cache, d.block_tables,
                       d.context_lens, w.max_context_len, w.scale, partition_tokens=P,
                       workspace=ws, out=out)

    call()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    rng = W.SplitMix64(97 + P)
    for _ in range(3):
        qkv = tuple(rng.normal_bf16(a.size, 1.0).reshape(a.shape) for a in (w.q[0], w.k[0], w.v[0]))
        for t, a in zip((d.q, d.k, d.v), qkv):
            t.copy_(dev_bf16(a))
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        ref, kc_ref, vc_ref = expected(orc, w, qkv=qkv)
        check_caches(d, kc_ref, vc_ref)
        assert_out_close(host_bits(out), ref, f"P={P}")
    check_status_clean(pa)
