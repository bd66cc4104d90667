"""Scores over a wide and drifting range, against the fp64 oracle.

The standard workloads draw q and K from N(0, 1), so their logits (scale * q.k * log2 e) span a
few units and a running softmax maximum settles within the first block.  The kernels move a
row's softmax shift only when its maximum passes the shift by more than 8 (log2 domain), so
those workloads never exercise a moving shift after the first block.  Here the maximum climbs
through the context by several times that slack, or falls, or the logits spread over hundreds
of units:

- "rise": each past K row scaled by a factor growing linearly from 0.25 to 8 with its position;
- "fall": the same factor reversed (the first tokens dominate, later ones underflow);
- "wide": q and K drawn with sigma 6, V brought back to sigma 1 (P is rounded to bf16, so the
  output error scales with the V rows it weights; the bar is set for rows of that size).

Decode (even split and fixed partitions), the fused step, the E4M3 decode and prefill.  Bars as
everywhere: output within 1e-2 + 1e-2 |oracle|, V stores bit-exact, K within 1 ulp.
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

CTX = [2048, 1500, 900, 37, 16, 1]
PROFILES = ("rise", "fall", "wide")


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


def ramp(profile, n):
    t = np.arange(n, dtype=np.float64)
    f = 0.25 + 7.75 * t / max(n - 1, 1)
    return f if profile == "rise" else f[::-1]


def scale_rows(cache, block_tables, lens, profile):
    """Multiply K row t of sequence s (t < lens[s]) by ramp(profile, lens[s])[t], rounded to bf16."""
    for s, n in enumerate(lens):
        n = int(n)
        if n <= 0:
            continue
        t = np.arange(n)
        blk = block_tables[s, t // W.BLOCK_SIZE].astype(np.int64)
        off = t % W.BLOCK_SIZE
        rows = W.bf16_bits_to_f32(cache[blk, :, off, :]).astype(np.float64)
        rows *= ramp(profile, n)[:, None, None]
        cache[blk, :, off, :] = W.f32_to_bf16_bits(rows.astype(np.float32))


def scaled(bits, factor):
    """bf16 bit patterns times `factor`, rounded to bf16."""
    return W.f32_to_bf16_bits((W.bf16_bits_to_f32(bits).astype(np.float64) * factor).astype(np.float32))


def decode_workload(profile, seed):
    sigma = 6.0 if profile == "wide" else 1.0
    ctx = np.asarray(CTX, np.int32)
    w = W.build(f"range_{profile}", ctx, int(((ctx + 15) // 16).sum()) + 8, seed, sigma=sigma)
    if profile == "wide":
        w.v_cache[0] = scaled(w.v_cache[0], 1.0 / sigma)
        w.v[0] = scaled(w.v[0], 1.0 / sigma)
    else:  # past tokens only: the new token's slot still holds the canary
        scale_rows(w.k_cache[0], w.block_tables, ctx - 1, profile)
    return w


@pytest.mark.parametrize("profile", PROFILES)
def test_decode_and_step_over_wide_score_ranges(pa, orc, profile):
    w = decode_workload(profile, 0x5A0 + PROFILES.index(profile))
    kc, vc = w.k_cache[0].copy(), w.v_cache[0].copy()
    q = orc.rope_kv_store(w.q[0], w.k[0], w.v[0], w.positions, w.cos_sin, w.slot_mapping, kc, vc)
    ref, _ = orc.decode(q, kc, vc, w.block_tables, w.context_lens, w.scale)
    d = DeviceLayer(w, q=q, k_cache=kc, v_cache=vc)
    for P in (0, 64, 512):
        out = pa.decode(d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens, w.max_context_len,
                        w.scale, partition_tokens=P)
        torch.cuda.synchronize()
        assert_out_close(host_bits(out), ref, f"decode {profile} P={P}")
    e = DeviceLayer(w)
    got = pa.decode_step(e.q, e.k, e.v, e.cos_sin, e.k_cache, e.v_cache, e.block_tables, e.context_lens,
                         w.max_context_len, w.scale)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(e.v_cache), vc)
    assert bf16_ulp_distance(host_bits(e.k_cache), kc).max() <= 1
    assert_out_close(host_bits(got), ref, f"step {profile}")
    check_status_clean(pa)


@pytest.mark.parametrize("profile", PROFILES)
def test_decode_fp8_over_wide_score_ranges(pa, orc, profile):
    w = decode_workload(profile, 0x5B0 + PROFILES.index(profile))
    kc, vc = w.k_cache[0].copy(), w.v_cache[0].copy()
    q = orc.rope_kv_store(w.q[0], w.k[0], w.v[0], w.positions, w.cos_sin, w.slot_mapping, kc, vc)

    def head_scales(cache):
        used = np.zeros(cache.shape[0], bool)
        used[w.block_tables[w.block_tables >= 0]] = True
        x = np.abs(W.bf16_bits_to_f32(cache[used]).astype(np.float64))
        x[~np.isfinite(x)] = 0.0
        return (np.maximum(x.max(axis=(0, 2, 3)), 1e-3) / 448.0).astype(np.float32)

    ks, vs = head_scales(kc), head_scales(vc)
    k8, v8 = orc.quantize_cache(kc, ks), orc.quantize_cache(vc, vs)
    ref8, _ = orc.decode_fp8(q, k8, v8, ks, vs, w.block_tables, w.context_lens, w.scale)
    for P in (0, 512):
        out8 = pa.decode_fp8(dev_bf16(q), dev(k8), dev(v8), dev(ks), dev(vs), dev(w.block_tables),
                             dev(w.context_lens), w.max_context_len, w.scale, partition_tokens=P)
        torch.cuda.synchronize()
        assert_out_close(host_bits(out8), ref8, f"fp8 {profile} P={P}")
    check_status_clean(pa)


@pytest.mark.parametrize("profile", PROFILES)
def test_prefill_over_wide_score_ranges(pa, orc, profile):
    sigma = 6.0 if profile == "wide" else 1.0
    ctx = np.asarray([700, 320, 97, 16], np.int32)
    ql = np.asarray([700, 64, 97, 5], np.int32)
    w = W.build_prefill(f"range_pf_{profile}", ctx, ql, int(((ctx + 15) // 16).sum()) + 4,
                        0x5C0 + PROFILES.index(profile), sigma=sigma)
    if profile == "wide":
        w.v_cache[...] = scaled(w.v_cache, 1.0 / sigma)
    else:
        scale_rows(w.k_cache, w.block_tables, ctx, profile)
    ref, _ = orc.prefill(w.q, w.q_start, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale)
    got = pa.prefill(dev_bf16(w.q), dev(w.q_start), dev_bf16(w.k_cache), dev_bf16(w.v_cache),
                     dev(w.block_tables), dev(w.context_lens), w.max_query_len, w.max_context_len,
                     w.scale)
    torch.cuda.synchronize()
    assert_out_close(host_bits(got), ref, f"prefill {profile}")
    check_status_clean(pa)
