"""Seeded random sweeps of the CUDA path against the fp64 oracle.

Each case draws a batch size, context lengths (short, block-aligned, ragged and long mixed),
a GQA shape, a split size and a pool layout from a seeded generator. It then checks, with the
same bars as the targeted tests:
- decode;
- the fused step (every other case with early metadata);
- the E4M3 decode;
- prefill.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DeviceLayer, assert_out_close, bf16_ulp_distance, dev, dev_bf16, host_bits
from paged_kv_cache_244_gb300 import _build
from paged_kv_cache_244_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SHAPES = [(12, 2), (8, 8), (16, 2), (4, 1), (32, 4), (6, 2), (7, 1)]


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


def draw_case(seed):
    rng = np.random.default_rng(seed)
    S = int(rng.integers(1, 24))
    kinds = rng.integers(0, 4, S)
    ctx = np.where(kinds == 0, rng.integers(1, 17, S),                      # within one block
          np.where(kinds == 1, 16 * rng.integers(1, 40, S),                 # block-aligned
          np.where(kinds == 2, rng.integers(17, 700, S),                    # ragged
                   rng.integers(700, 3000, S)))).astype(np.int32)           # long
    hq, hkv = SHAPES[int(rng.integers(0, len(SHAPES)))]
    P = int(rng.choice([0, 0, 16, 32, 64, 256, 512]))
    need = int(((ctx + 15) // 16).sum())
    pool = need + int(rng.integers(0, 64))
    return ctx, hq, hkv, P, pool


@pytest.mark.parametrize("seed", range(8))
def test_random_decode_and_step(pa, orc, seed):
    ctx, hq, hkv, P, pool = draw_case(1000 + seed)
    w = W.build("rand", ctx, pool, 2000 + seed, num_q_heads=hq, num_kv_heads=hkv)
    # decode on oracle-stored inputs
    kc, vc = w.k_cache[0].copy(), w.v_cache[0].copy()
    q = orc.rope_kv_store(w.q[0], w.k[0], w.v[0], w.positions, w.cos_sin, w.slot_mapping, kc, vc)
    ref, _ = orc.decode(q, kc, vc, w.block_tables, w.context_lens, w.scale)
    d = DeviceLayer(w, q=q, k_cache=kc, v_cache=vc)
    out = pa.decode(d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens, w.max_context_len,
                    w.scale, partition_tokens=P)
    torch.cuda.synchronize()
    assert_out_close(host_bits(out), ref, f"decode seed {seed} P={P} {hq}/{hkv}")
    # the fused step from the unrotated inputs; odd seeds with early metadata (the tables were
    # uploaded by copies, and the decode above does not write them)
    e = DeviceLayer(w)
    got = pa.decode_step(e.q, e.k, e.v, e.cos_sin, e.k_cache, e.v_cache, e.block_tables,
                         e.context_lens, w.max_context_len, w.scale, partition_tokens=P,
                         early_metadata=bool(seed % 2))
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(e.v_cache), vc)
    assert bf16_ulp_distance(host_bits(e.k_cache), kc).max() <= 1
    assert_out_close(host_bits(got), ref, f"step seed {seed}")
    check_status_clean(pa)


@pytest.mark.parametrize("seed", range(6))
def test_random_decode_fp8(pa, orc, seed):
    ctx, hq, hkv, P, pool = draw_case(3000 + seed)
    w = W.build("rand8", ctx, pool, 4000 + seed, num_q_heads=hq, num_kv_heads=hkv)
    kc, vc = w.k_cache[0].copy(), w.v_cache[0].copy()
    q = orc.rope_kv_store(w.q[0], w.k[0], w.v[0], w.positions, w.cos_sin, w.slot_mapping, kc, vc)
    rng = np.random.default_rng(seed)
    ks = rng.uniform(2.0, 8.0, hkv).astype(np.float32) / 448
    vs = rng.uniform(2.0, 8.0, hkv).astype(np.float32) / 448
    k8, v8 = orc.quantize_cache(kc, ks), orc.quantize_cache(vc, vs)
    ref, _ = orc.decode_fp8(q, k8, v8, ks, vs, w.block_tables, w.context_lens, w.scale)
    out = pa.decode_fp8(dev_bf16(q), dev(k8), dev(v8), dev(ks), dev(vs), dev(w.block_tables),
                        dev(w.context_lens), w.max_context_len, w.scale, partition_tokens=P)
    torch.cuda.synchronize()
    assert_out_close(host_bits(out), ref, f"fp8 seed {seed} P={P} {hq}/{hkv}")
    check_status_clean(pa)


@pytest.mark.parametrize("seed", range(6))
def test_random_prefill(pa, orc, seed):
    rng = np.random.default_rng(5000 + seed)
    S = int(rng.integers(1, 8))
    ctx = rng.integers(1, 600, S).astype(np.int32)
    ql = np.array([int(rng.integers(1, c + 1)) for c in ctx], np.int32)
    hq, hkv = SHAPES[int(rng.integers(0, len(SHAPES)))]
    pool = int(((ctx + 15) // 16).sum()) + 8
    w = W.build_prefill("randpf", ctx, ql, pool, 6000 + seed, num_q_heads=hq, num_kv_heads=hkv)
    ref, _ = orc.prefill(w.q, w.q_start, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale)
    got = pa.prefill(dev_bf16(w.q), dev(w.q_start), dev_bf16(w.k_cache), dev_bf16(w.v_cache),
                     dev(w.block_tables), dev(w.context_lens), w.max_query_len, w.max_context_len,
                     w.scale)
    torch.cuda.synchronize()
    assert_out_close(host_bits(got), ref, f"prefill seed {seed} {hq}/{hkv}")
    check_status_clean(pa)
