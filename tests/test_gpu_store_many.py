"""pa_rope_kv_store and pa_rope_kv_store_fp8 at prompt sizes, against the fp64 oracle.

The store kernel has two shapes, chosen by the token count (up to 2048 tokens: every vector of
a token loaded at once; more: fewer registers, more warps per SM).  These cases run both, with
head counts that take one and several groups of passes, padding tokens (slot -1) among them,
and random positions and slots.  Bars as for the decode-size store: q and rotated K within 1
bf16 ulp (E4M3 K within one code step), V bit-exact, every other cache byte untouched.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import bf16_ulp_distance, dev, dev_bf16, host_bits
from paged_kv_cache_244_gb300 import _build
from paged_kv_cache_244_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_POS = 4096


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


def tokens(T, hq, hkv, seed):
    """Seeded new-token rows, positions, slots (every 97th token a padding slot) and a
    randomly filled bf16 cache pool."""
    rng = W.SplitMix64(seed)
    q = rng.normal_bf16(T * hq * 128, 1.0).reshape(T, hq, 128)
    k = rng.normal_bf16(T * hkv * 128, 1.0).reshape(T, hkv, 128)
    v = rng.normal_bf16(T * hkv * 128, 1.0).reshape(T, hkv, 128)
    nb = (T + 15) // 16 + 8
    kc = rng.normal_bf16(nb * hkv * 16 * 128, 1.0).reshape(nb, hkv, 16, 128)
    vc = rng.normal_bf16(nb * hkv * 16 * 128, 1.0).reshape(nb, hkv, 16, 128)
    gen = np.random.default_rng(seed)
    pos = gen.integers(0, MAX_POS, T).astype(np.int32)
    slots = gen.permutation(nb * 16)[:T].astype(np.int64)
    slots[::97] = -1
    return q, k, v, pos, slots, kc, vc


def untouched_mask(shape, slots):
    live = slots[slots >= 0]
    blk, off = np.divmod(live, W.BLOCK_SIZE)
    mask = np.ones(shape, bool)
    mask[blk, :, off] = False
    return mask


@pytest.mark.parametrize("T,hq,hkv", [(2048, 12, 2), (2049, 12, 2), (6000, 12, 2), (3000, 32, 4),
                                      (2500, 8, 8), (700, 32, 4)])
def test_store_at_prompt_sizes_matches_oracle(pa, orc, T, hq, hkv):
    q, k, v, pos, slots, kc, vc = tokens(T, hq, hkv, 300 + T + hq)
    cos_sin = W.rope_cos_sin_table(MAX_POS)
    kc_ref, vc_ref = kc.copy(), vc.copy()
    q_ref = orc.rope_kv_store(q, k, v, pos, cos_sin, slots, kc_ref, vc_ref)
    dq, dkc, dvc = dev_bf16(q), dev_bf16(kc), dev_bf16(vc)
    pa.rope_kv_store(dq, dev_bf16(k), dev_bf16(v), dev(pos), dev(cos_sin), dev(slots), dkc, dvc)
    torch.cuda.synchronize()
    assert bf16_ulp_distance(host_bits(dq), q_ref).max() <= 1
    assert np.array_equal(host_bits(dvc), vc_ref)
    got_k = host_bits(dkc)
    assert bf16_ulp_distance(got_k, kc_ref).max() <= 1
    mask = untouched_mask(kc.shape, slots)
    assert np.array_equal(got_k[mask], kc[mask])
    check_status_clean(pa)


def e4m3_step_distance(a, b):
    def ordered(x):
        x = x.astype(np.int32)
        mag = x & 0x7F
        return np.where(x & 0x80, -mag, mag)
    return np.abs(ordered(a) - ordered(b))


@pytest.mark.parametrize("T,hq,hkv", [(2048, 12, 2), (5000, 12, 2), (3000, 32, 4)])
def test_store_fp8_at_prompt_sizes_matches_oracle(pa, orc, T, hq, hkv):
    q, k, v, pos, slots, kc, vc = tokens(T, hq, hkv, 400 + T + hq)
    cos_sin = W.rope_cos_sin_table(MAX_POS)
    gen = np.random.default_rng(T)
    ks = gen.uniform(2.0, 6.0, hkv).astype(np.float32) / 448
    vs = gen.uniform(2.0, 6.0, hkv).astype(np.float32) / 448
    k8, v8 = orc.quantize_cache(kc, ks), orc.quantize_cache(vc, vs)
    k_ref, v_ref = k8.copy(), v8.copy()
    q_ref = orc.rope_kv_store_fp8(q, k, v, pos, cos_sin, slots, k_ref, v_ref, ks, vs)
    dq, dk8, dv8 = dev_bf16(q), dev(k8), dev(v8)
    pa.rope_kv_store_fp8(dq, dev_bf16(k), dev_bf16(v), dev(pos), dev(cos_sin), dev(slots), dk8, dv8,
                         dev(ks), dev(vs))
    torch.cuda.synchronize()
    assert bf16_ulp_distance(host_bits(dq), q_ref).max() <= 1
    assert np.array_equal(dv8.cpu().numpy(), v_ref)
    got_k = dk8.cpu().numpy()
    assert e4m3_step_distance(got_k, k_ref).max() <= 1
    mask = untouched_mask(k8.shape, slots)
    assert np.array_equal(got_k[mask], k8[mask])
    check_status_clean(pa)
