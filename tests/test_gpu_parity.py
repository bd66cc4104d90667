"""CUDA path (through the C ABI) against the fp64 oracle, element by element.

Bars: slot placement and V stores bit-exact; rotated q and K within 1 bf16 ulp; attention
output within |gpu - oracle| <= 1e-2 + 1e-2 |oracle|.  Every decode comparison feeds both
sides identical inputs that the oracle (never the GPU) produced.
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


_cache = {}


def workload(name):
    if name not in _cache:
        _cache[name] = W.make(name)
    return _cache[name]


def oracle_store(orc, w, layer=0):
    """Oracle's RoPE + store for one layer: (rotated q, k_cache, v_cache) host arrays."""
    kc, vc = w.k_cache[layer].copy(), w.v_cache[layer].copy()
    q = orc.rope_kv_store(w.q[layer], w.k[layer], w.v[layer], w.positions, w.cos_sin,
                          w.slot_mapping, kc, vc)
    return q, kc, vc


def check_status_clean(pa):
    rc, flags = pa.get_device_status()
    assert rc == 0 and flags == 0, (rc, hex(flags))


# ------------------------------------------------------------------ rope + KV store ----

@pytest.mark.parametrize("name", W.WORKLOADS)
def test_rope_kv_store_matches_oracle(pa, orc, name):
    w = workload(name)
    for layer in sorted({0, w.num_layers - 1}):
        d = DeviceLayer(w, layer)
        pa.rope_kv_store(d.q, d.k, d.v, d.positions, d.cos_sin, d.slot_mapping, d.k_cache, d.v_cache)
        torch.cuda.synchronize()
        q_ref, kc_ref, vc_ref = oracle_store(orc, w, layer)
        assert bf16_ulp_distance(host_bits(d.q), q_ref).max() <= 1
        # V and everything outside the written slots: bit-exact.  K at the slots: <= 1 ulp.
        assert np.array_equal(host_bits(d.v_cache), vc_ref)
        kc = host_bits(d.k_cache)
        assert bf16_ulp_distance(kc, kc_ref).max() <= 1
        blk, off = np.divmod(w.slot_mapping, W.BLOCK_SIZE)
        mask = np.ones(kc.shape, bool)
        mask[blk, :, off] = False
        assert np.array_equal(kc[mask], w.k_cache[layer][mask])
    check_status_clean(pa)


# -------------------------------------------------------------------------- decode ----

def run_decode(pa, d, w, partition_tokens=None, max_context_len=None):
    P = w.partition_tokens if partition_tokens is None else partition_tokens
    out = pa.decode(d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens,
                    max_context_len or w.max_context_len, w.scale, partition_tokens=P)
    torch.cuda.synchronize()
    return host_bits(out)


@pytest.mark.parametrize("name", W.WORKLOADS)
def test_decode_matches_oracle(pa, orc, name):
    w = workload(name)
    for layer in sorted({0, w.num_layers - 1}):
        q, kc, vc = oracle_store(orc, w, layer)
        ref, _ = orc.decode(q, kc, vc, w.block_tables, w.context_lens, w.scale)
        d = DeviceLayer(w, layer, q=q, k_cache=kc, v_cache=vc)
        assert_out_close(run_decode(pa, d, w), ref, f"{name} layer {layer}")
    check_status_clean(pa)


@pytest.mark.parametrize("name", ["tiny", "mix64"])
def test_chained_step_matches_oracle(pa, orc, name):
    """GPU rope+store then GPU decode, against the oracle's own chain."""
    w = workload(name)
    d = DeviceLayer(w)
    pa.rope_kv_store(d.q, d.k, d.v, d.positions, d.cos_sin, d.slot_mapping, d.k_cache, d.v_cache)
    got = run_decode(pa, d, w)
    q, kc, vc = oracle_store(orc, w)
    ref, _ = orc.decode(q, kc, vc, w.block_tables, w.context_lens, w.scale)
    assert_out_close(got, ref, name)
    check_status_clean(pa)


@pytest.mark.parametrize("P", [16, 32, 64, 128, 512, 4096])
def test_decode_partition_sizes(pa, orc, P):
    w = W.build("parts", [1, 16, 17, 100, 511, 512, 513, 1500, 4096], 800, 77)
    q, kc, vc = oracle_store(orc, w)
    ref, _ = orc.decode(q, kc, vc, w.block_tables, w.context_lens, w.scale)
    d = DeviceLayer(w, q=q, k_cache=kc, v_cache=vc)
    assert_out_close(run_decode(pa, d, w, partition_tokens=P), ref, f"P={P}")
    check_status_clean(pa)


def test_decode_edge_context_lengths(pa, orc):
    ctxs = [1, 2, 15, 16, 17, 31, 32, 33, 255, 256, 257, 511, 512, 513, 1000, 3]
    w = W.build("edges", ctxs, 400, 78, max_blocks=70)
    q, kc, vc = oracle_store(orc, w)
    bt = w.block_tables.copy()
    bt[bt < 0] = 123456789        # garbage past each context: must never be read
    ref, _ = orc.decode(q, kc, vc, bt, w.context_lens, w.scale)
    d = DeviceLayer(w, q=q, k_cache=kc, v_cache=vc)
    d.block_tables = dev(bt)
    for P in (0, 16, 256):
        assert_out_close(run_decode(pa, d, w, partition_tokens=P), ref, f"P={P}")
    check_status_clean(pa)


@pytest.mark.parametrize("hq,hkv", [(12, 2), (8, 8), (16, 2), (6, 2), (4, 1), (14, 2), (10, 2),
                                    (32, 4)])
def test_decode_group_sizes(pa, orc, hq, hkv):
    w = W.build("groups", [5, 40, 300, 700], 120, 79, num_q_heads=hq, num_kv_heads=hkv)
    q, kc, vc = oracle_store(orc, w)
    ref, _ = orc.decode(q, kc, vc, w.block_tables, w.context_lens, w.scale)
    d = DeviceLayer(w, q=q, k_cache=kc, v_cache=vc)
    for P in (0, 64):
        assert_out_close(run_decode(pa, d, w, partition_tokens=P), ref, f"{hq}/{hkv} P={P}")
    check_status_clean(pa)


def test_decode_zero_context_gives_zero_rows(pa, orc):
    w = W.build("zero", [30, 50, 20], 16, 80)
    q, kc, vc = oracle_store(orc, w)
    ctx = w.context_lens.copy()
    ctx[1] = 0
    ref, _ = orc.decode(q, kc, vc, w.block_tables, ctx, w.scale)
    d = DeviceLayer(w, q=q, k_cache=kc, v_cache=vc)
    d.context_lens = dev(ctx)
    for P in (0, 16):
        got = run_decode(pa, d, w, partition_tokens=P)
        assert (got[1] == 0).all()
        assert_out_close(got, ref)
    check_status_clean(pa)


def test_decode_reuses_one_workspace_across_shapes(pa, orc):
    """One zero-filled workspace serves calls of different shapes and split modes in a row;
    repeated calls give identical results."""
    big = workload("mix64")
    need = max(pa.decode_workspace_size(12, 2, big.num_seqs, big.max_context_len, P) for P in (0, 64))
    ws = torch.zeros((need + 3) // 4, dtype=torch.float32, device="cuda")
    cases = [("mix64", 0), ("tiny", 0), ("mix64", 64), ("long4", 512), ("mix64", 0)]
    seen = {}
    for name, P in cases:
        w = workload(name)
        q, kc, vc = oracle_store(orc, w)
        ref, _ = orc.decode(q, kc, vc, w.block_tables, w.context_lens, w.scale)
        d = DeviceLayer(w, q=q, k_cache=kc, v_cache=vc)
        assert pa.decode_workspace_size(12, 2, w.num_seqs, w.max_context_len, P) <= ws.numel() * 4
        out = pa.decode(d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens,
                        w.max_context_len, w.scale, partition_tokens=P, workspace=ws)
        torch.cuda.synchronize()
        got = host_bits(out)
        assert_out_close(got, ref, f"{name} P={P}")
        if (name, P) in seen:
            assert np.array_equal(got, seen[(name, P)])
        seen[(name, P)] = got
    check_status_clean(pa)


# --------------------------------------------------------- device-side range checks ----

def test_out_of_range_block_id_is_flagged_and_skipped(pa, orc):
    w = W.build("oob", [40, 40], 16, 81)
    q, kc, vc = oracle_store(orc, w)
    ref, _ = orc.decode(q, kc, vc, w.block_tables, w.context_lens, w.scale)
    bt = w.block_tables.copy()
    bt[1, 1] = w.num_blocks + 5          # sequence 1 now names a block that does not exist
    d = DeviceLayer(w, q=q, k_cache=kc, v_cache=vc)
    d.block_tables = dev(bt)
    check_status_clean(pa)
    got = run_decode(pa, d, w, partition_tokens=0)
    rc, flags = pa.get_device_status()
    assert rc == pa.PA_ERR_DEVICE_OOB and flags & pa.PA_FLAG_BLOCK_ID_OOB
    assert_out_close(got[:1], ref[:1], "untouched sequence")
    check_status_clean(pa)               # read-and-clear


def test_context_len_beyond_bound_is_flagged(pa, orc):
    w = W.build("ctxoob", [40, 20], 16, 82)
    q, kc, vc = oracle_store(orc, w)
    d = DeviceLayer(w, q=q, k_cache=kc, v_cache=vc)
    ctx = w.context_lens.copy()
    ctx[1] = 41                          # above max_context_len = 40
    d.context_lens = dev(ctx)
    run_decode(pa, d, w)
    rc, flags = pa.get_device_status()
    assert flags & pa.PA_FLAG_CONTEXT_LEN_OOB


def test_bad_slot_and_position_are_flagged(pa, orc):
    w = W.build("slotoob", [20, 30, 10], 8, 83)
    d = DeviceLayer(w)
    slots = w.slot_mapping.copy()
    slots[0] = w.num_blocks * W.BLOCK_SIZE + 3
    slots[2] = -1                        # padding token: silently skipped
    pos = w.positions.copy()
    pos[1] = w.cos_sin.shape[0] + 10
    d.slot_mapping = dev(slots)
    d.positions = dev(pos)
    before_v = host_bits(d.v_cache)
    pa.rope_kv_store(d.q, d.k, d.v, d.positions, d.cos_sin, d.slot_mapping, d.k_cache, d.v_cache)
    rc, flags = pa.get_device_status()
    assert flags & pa.PA_FLAG_SLOT_OOB and flags & pa.PA_FLAG_POSITION_OOB
    assert np.array_equal(host_bits(d.v_cache), before_v)   # nothing was stored
    check_status_clean(pa)


def test_bounded_wait_times_out_and_reports(pa):
    """A wait on a barrier that nothing completes gives up, raises the timeout flag, and the
    GPU keeps working afterwards (a decode right after still matches the oracle)."""
    check_status_clean(pa)
    pa.selftest_wait_timeout(2000)          # 2 ms
    rc, flags = pa.get_device_status()
    assert rc == pa.PA_ERR_TIMEOUT and flags == pa.PA_FLAG_TIMEOUT
    check_status_clean(pa)
    orc = oracle.default()
    w = W.build("after_timeout", [40, 17], 16, 84)
    q, kc, vc = oracle_store(orc, w)
    ref, _ = orc.decode(q, kc, vc, w.block_tables, w.context_lens, w.scale)
    d = DeviceLayer(w, q=q, k_cache=kc, v_cache=vc)
    assert_out_close(run_decode(pa, d, w), ref)


@pytest.mark.parametrize("P", [0, 16])
def test_decode_replayed_from_a_cuda_graph(pa, orc, P):
    """A graph freezes the call's arguments: every replay reads the q its buffer holds then
    and gives that q's result (the workspace carries nothing from one call to the next)."""
    w = W.build("graph", [40, 300, 700, 17], 200, 85)
    q, kc, vc = oracle_store(orc, w)
    d = DeviceLayer(w, q=q, k_cache=kc, v_cache=vc)
    ws = pa.decode_workspace(d.q, d.k_cache, w.max_context_len, P)
    out = torch.empty_like(d.q)

    def call():
        pa.decode(d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens, w.max_context_len,
                  w.scale, partition_tokens=P, workspace=ws, out=out)

    call()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    rng = W.SplitMix64(86 + P)
    for _ in range(3):
        q2 = rng.normal_bf16(q.size, 1.0).reshape(q.shape)
        d.q.copy_(dev_bf16(q2))
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        ref, _ = orc.decode(q2, kc, vc, w.block_tables, w.context_lens, w.scale)
        assert_out_close(host_bits(out), ref, f"P={P}")
    check_status_clean(pa)
