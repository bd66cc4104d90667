"""The entry points at the limits pa.h states, against the fp64 oracle.

- 8,192 sequences in one call: the block-count prefix fills its shared-memory area, in the
  bf16 and E4M3 layouts and in the fused step.
- Many KV heads, up to the 4,096 allowed: the KV head index travels packed in a job word.
- pa_copy_blocks over the most caches one call takes (256: K and V of 128 layers).
Bars as everywhere: output within 1e-2 + 1e-2 |oracle|, V stores bit-exact, K within 1 ulp.
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


def stored(orc, w):
    kc, vc = w.k_cache[0].copy(), w.v_cache[0].copy()
    q = orc.rope_kv_store(w.q[0], w.k[0], w.v[0], w.positions, w.cos_sin, w.slot_mapping, kc, vc)
    ref, _ = orc.decode(q, kc, vc, w.block_tables, w.context_lens, w.scale)
    return q, kc, vc, ref


def test_most_sequences_per_call(pa, orc):
    """8,192 sequences of 1 to 40 tokens: decode, fused step and E4M3 decode."""
    rng = np.random.default_rng(8192)
    ctx = rng.integers(1, 41, 8192).astype(np.int32)
    w = W.build("max_seqs", ctx, int(((ctx + 15) // 16).sum()) + 16, 8193)
    q, kc, vc, ref = stored(orc, w)
    d = DeviceLayer(w, q=q, k_cache=kc, v_cache=vc)
    out = pa.decode(d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens, w.max_context_len, w.scale)
    torch.cuda.synchronize()
    assert_out_close(host_bits(out), ref, "decode")
    e = DeviceLayer(w)
    got = pa.decode_step(e.q, e.k, e.v, e.cos_sin, e.k_cache, e.v_cache, e.block_tables, e.context_lens,
                         w.max_context_len, w.scale)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(e.v_cache), vc)
    assert bf16_ulp_distance(host_bits(e.k_cache), kc).max() <= 1
    assert_out_close(host_bits(got), ref, "step")
    ks = np.full(2, 5.0 / 448, np.float32)
    vs = np.full(2, 5.0 / 448, np.float32)
    k8, v8 = orc.quantize_cache(kc, ks), orc.quantize_cache(vc, vs)
    ref8, _ = orc.decode_fp8(q, k8, v8, ks, vs, w.block_tables, w.context_lens, w.scale)
    out8 = pa.decode_fp8(dev_bf16(q), dev(k8), dev(v8), dev(ks), dev(vs), dev(w.block_tables),
                         dev(w.context_lens), w.max_context_len, w.scale)
    torch.cuda.synchronize()
    assert_out_close(host_bits(out8), ref8, "fp8")
    check_status_clean(pa)


@pytest.mark.parametrize("hq,hkv", [(64, 64), (512, 64), (4096, 4096)])
def test_many_kv_heads(pa, orc, hq, hkv):
    ctx = [1, 20, 33] if hkv < 4096 else [1, 18]
    w = W.build(f"heads{hkv}", ctx, int(sum((c + 15) // 16 for c in ctx)) + 2, hkv + hq,
                num_q_heads=hq, num_kv_heads=hkv)
    q, kc, vc, ref = stored(orc, w)
    d = DeviceLayer(w, q=q, k_cache=kc, v_cache=vc)
    out = pa.decode(d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens, w.max_context_len, w.scale)
    torch.cuda.synchronize()
    assert_out_close(host_bits(out), ref, f"decode {hq}/{hkv}")
    e = DeviceLayer(w)
    got = pa.decode_step(e.q, e.k, e.v, e.cos_sin, e.k_cache, e.v_cache, e.block_tables, e.context_lens,
                         w.max_context_len, w.scale, early_metadata=True)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(e.v_cache), vc)
    assert bf16_ulp_distance(host_bits(e.k_cache), kc).max() <= 1
    assert_out_close(host_bits(got), ref, f"step {hq}/{hkv}")
    check_status_clean(pa)


def test_copy_blocks_most_caches(pa, orc):
    """256 caches of 24 blocks, 10 copy-on-write pairs: every pool as the oracle's copy."""
    rng = np.random.default_rng(256)
    pools = [rng.integers(0, 1 << 16, (24, 2, W.BLOCK_SIZE, W.HEAD_DIM), dtype=np.uint16)
             for _ in range(pa.PA_MAX_BLOCK_CACHES)]
    frm = rng.permutation(12)[:10]
    to = 12 + rng.permutation(12)[:10]
    pairs = np.stack([frm, to], axis=1).astype(np.int64)
    want = [p.copy() for p in pools]
    assert orc.copy_blocks(want, want, pairs) == 0
    devp = [torch.from_numpy(p.view(np.int16)).view(torch.bfloat16).cuda() for p in pools]
    pa.copy_blocks(devp, devp, torch.from_numpy(pairs).cuda())
    torch.cuda.synchronize()
    for c in range(len(pools)):
        assert np.array_equal(devp[c].view(torch.int16).cpu().numpy().view(np.uint16), want[c]), c
    check_status_clean(pa)
