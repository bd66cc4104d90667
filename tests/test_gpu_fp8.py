"""FP8 (E4M3) KV cache through the C ABI, against the fp64 oracle.

Bars:
- V codes: bit-exact.
- K codes: within one E4M3 step. The rotated k the codes come from may differ by one bf16
  ulp between fp32 and fp64 rotation.
- Rotated q: within 1 bf16 ulp.
- Attention output over the same codes: within 1e-2 + 1e-2 |oracle|, as for bf16 caches.

Every decode input (q, codes, scales) is produced by the oracle or by the seeded generator,
never by the GPU.
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


def head_scales(cache_bits, margin=1.0):
    """One scale per KV head: the largest finite magnitude of that head's cache over 448."""
    x = W.bf16_bits_to_f32(cache_bits).astype(np.float64)
    x[~np.isfinite(x)] = 0.0
    amax = np.abs(x).max(axis=(0, 2, 3))
    return (np.maximum(amax, 1e-3) * margin / 448.0).astype(np.float32)


def e4m3_step_distance(a, b):
    def ordered(x):
        x = x.astype(np.int32)
        mag = x & 0x7F
        return np.where(x & 0x80, -mag, mag)
    return np.abs(ordered(a) - ordered(b))


class Fp8Layer:
    """A layer with E4M3 caches quantised by the oracle from the workload's bf16 caches."""

    def __init__(self, orc, w, layer=0, margin=1.0):
        self.ks = head_scales(w.k_cache[layer], margin)
        self.vs = head_scales(w.v_cache[layer], margin)
        self.k8 = orc.quantize_cache(w.k_cache[layer], self.ks)
        self.v8 = orc.quantize_cache(w.v_cache[layer], self.vs)
        self.d = DeviceLayer(w, layer)
        self.k8_dev = dev(self.k8)
        self.v8_dev = dev(self.v8)
        self.ks_dev = dev(self.ks)
        self.vs_dev = dev(self.vs)


def oracle_store_fp8(orc, w, f, layer=0):
    k8, v8 = f.k8.copy(), f.v8.copy()
    q = orc.rope_kv_store_fp8(w.q[layer], w.k[layer], w.v[layer], w.positions, w.cos_sin,
                              w.slot_mapping, k8, v8, f.ks, f.vs)
    return q, k8, v8


@pytest.mark.parametrize("name", W.WORKLOADS)
def test_rope_kv_store_fp8_matches_oracle(pa, orc, name):
    w = W.make(name)
    f = Fp8Layer(orc, w)
    d = f.d
    pa.rope_kv_store_fp8(d.q, d.k, d.v, d.positions, d.cos_sin, d.slot_mapping, f.k8_dev, f.v8_dev,
                         f.ks_dev, f.vs_dev)
    torch.cuda.synchronize()
    q_ref, k_ref, v_ref = oracle_store_fp8(orc, w, f)
    assert bf16_ulp_distance(host_bits(d.q), q_ref).max() <= 1
    assert np.array_equal(f.v8_dev.cpu().numpy(), v_ref)
    k_got = f.k8_dev.cpu().numpy()
    assert e4m3_step_distance(k_got, k_ref).max() <= 1
    # outside the new slots nothing moved
    blk, off = np.divmod(w.slot_mapping, W.BLOCK_SIZE)
    mask = np.ones(k_got.shape, bool)
    mask[blk, :, off] = False
    assert np.array_equal(k_got[mask], f.k8[mask])
    check_status_clean(pa)


@pytest.mark.parametrize("name", W.WORKLOADS)
def test_decode_fp8_matches_oracle(pa, orc, name):
    w = W.make(name)
    for layer in sorted({0, w.num_layers - 1}):
        f = Fp8Layer(orc, w, layer)
        q, k8, v8 = oracle_store_fp8(orc, w, f, layer)
        ref, _ = orc.decode_fp8(q, k8, v8, f.ks, f.vs, w.block_tables, w.context_lens, w.scale)
        d = f.d
        out = pa.decode_fp8(dev_bf16(q), dev(k8), dev(v8), f.ks_dev, f.vs_dev, d.block_tables,
                            d.context_lens, w.max_context_len, w.scale,
                            partition_tokens=w.partition_tokens)
        torch.cuda.synchronize()
        assert_out_close(host_bits(out), ref, f"{name} layer {layer}")
    check_status_clean(pa)


def test_decode_fp8_edges_splits_and_groups(pa, orc):
    ctxs = [1, 2, 15, 16, 17, 31, 32, 33, 255, 256, 257, 511, 512, 513, 1000, 3]
    for hq, hkv in ((12, 2), (8, 8), (16, 2), (4, 1), (32, 4)):
        w = W.build("fp8_edges", ctxs, 400, 97, max_blocks=70, num_q_heads=hq, num_kv_heads=hkv)
        f = Fp8Layer(orc, w)
        q, k8, v8 = oracle_store_fp8(orc, w, f)
        ref, _ = orc.decode_fp8(q, k8, v8, f.ks, f.vs, w.block_tables, w.context_lens, w.scale)
        for P in (0, 16, 256):
            out = pa.decode_fp8(dev_bf16(q), dev(k8), dev(v8), f.ks_dev, f.vs_dev, f.d.block_tables,
                                f.d.context_lens, w.max_context_len, w.scale, partition_tokens=P)
            torch.cuda.synchronize()
            assert_out_close(host_bits(out), ref, f"{hq}/{hkv} P={P}")
    check_status_clean(pa)


def test_decode_fp8_subnormal_codes(pa, orc):
    """Scales 2^13 x (largest magnitude / 448) put the largest code near 0.055, so most codes
    fall in the E4M3 subnormal range (below 2^-6): the exact widening must keep them."""
    w = W.build("fp8_sub", [40, 300, 17], 64, 98)
    f = Fp8Layer(orc, w, margin=8192.0)
    q, k8, v8 = oracle_store_fp8(orc, w, f)
    used = np.concatenate([k8[w.block_tables[s, :(int(c) + 15) // 16]].ravel()
                           for s, c in enumerate(w.context_lens)])
    assert ((used & 0x78) == 0).mean() > 0.5          # exponent field 0: subnormal or zero
    ref, _ = orc.decode_fp8(q, k8, v8, f.ks, f.vs, w.block_tables, w.context_lens, w.scale)
    out = pa.decode_fp8(dev_bf16(q), dev(k8), dev(v8), f.ks_dev, f.vs_dev, f.d.block_tables,
                        f.d.context_lens, w.max_context_len, w.scale)
    torch.cuda.synchronize()
    assert_out_close(host_bits(out), ref)
    check_status_clean(pa)


@pytest.mark.parametrize("name", ["tiny", "mix64", "long4"])
def test_decode_step_fp8_matches_oracle_and_two_calls(pa, orc, name):
    w = W.make(name)
    f = Fp8Layer(orc, w)
    a_k8, a_v8 = dev(f.k8), dev(f.v8)
    d = f.d
    got = pa.decode_step_fp8(d.q, d.k, d.v, d.cos_sin, a_k8, a_v8, f.ks_dev, f.vs_dev,
                             d.block_tables, d.context_lens, w.max_context_len, w.scale,
                             partition_tokens=w.partition_tokens)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(d.q), w.q[0])               # q is not modified
    q_ref, k_ref, v_ref = oracle_store_fp8(orc, w, f)
    ref, _ = orc.decode_fp8(q_ref, k_ref, v_ref, f.ks, f.vs, w.block_tables, w.context_lens, w.scale)
    assert np.array_equal(a_v8.cpu().numpy(), v_ref)
    assert e4m3_step_distance(a_k8.cpu().numpy(), k_ref).max() <= 1
    assert_out_close(host_bits(got), ref, name)
    # the same as the FP8 store followed by the FP8 decode, bit for bit
    b = DeviceLayer(w)
    b_k8, b_v8 = dev(f.k8), dev(f.v8)
    pa.rope_kv_store_fp8(b.q, b.k, b.v, b.positions, b.cos_sin, b.slot_mapping, b_k8, b_v8,
                         f.ks_dev, f.vs_dev)
    two = pa.decode_fp8(b.q, b_k8, b_v8, f.ks_dev, f.vs_dev, b.block_tables, b.context_lens,
                        w.max_context_len, w.scale, partition_tokens=w.partition_tokens)
    torch.cuda.synchronize()
    assert np.array_equal(a_k8.cpu().numpy(), b_k8.cpu().numpy())
    assert np.array_equal(a_v8.cpu().numpy(), b_v8.cpu().numpy())
    assert np.array_equal(host_bits(got), host_bits(two))
    check_status_clean(pa)


def test_fp8_cache_error_against_bf16_cache(pa, orc):
    """Not a parity bar: how far the E4M3 cache moves the mix64 output from the bf16 cache
    (amax scales), reported and bounded loosely to catch a gross scale error."""
    w = W.make("mix64")
    f = Fp8Layer(orc, w)
    q, k8, v8 = oracle_store_fp8(orc, w, f)
    d = f.d
    out8 = pa.decode_fp8(dev_bf16(q), dev(k8), dev(v8), f.ks_dev, f.vs_dev, d.block_tables,
                         d.context_lens, w.max_context_len, w.scale)
    kc, vc = w.k_cache[0].copy(), w.v_cache[0].copy()
    q16 = orc.rope_kv_store(w.q[0], w.k[0], w.v[0], w.positions, w.cos_sin, w.slot_mapping, kc, vc)
    ref16, _ = orc.decode(q16, kc, vc, w.block_tables, w.context_lens, w.scale)
    torch.cuda.synchronize()
    got = W.bf16_bits_to_f32(host_bits(out8)).astype(np.float64)
    err = np.abs(got - ref16)
    print(f"E4M3 cache vs bf16 cache on mix64: max |diff| {err.max():.4f}, mean {err.mean():.5f}")
    assert err.max() < 0.25 and err.mean() < 0.02
    check_status_clean(pa)
