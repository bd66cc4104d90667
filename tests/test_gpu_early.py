"""The fused decode step with PA_STEP_EARLY_METADATA, through the C ABI.

With the flag the decode kernel reads lengths and block tables before the preceding kernel
on the stream has finished, and waits for it before its first copy and its first write.  The
arithmetic is the same, so:
- one call gives the same bits as the call without the flag;
- layers launched back to back on one stream, step after step (the intended use), give the
  oracle's result for every layer and step, eagerly and replayed from a CUDA graph.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_out_close, bf16_ulp_distance, dev, dev_bf16, host_bits
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


class Layers:
    """Every layer of a workload on the GPU, sharing one block table and one length array."""

    def __init__(self, w: W.Workload):
        self.k_cache = [dev_bf16(w.k_cache[i]) for i in range(w.num_layers)]
        self.v_cache = [dev_bf16(w.v_cache[i]) for i in range(w.num_layers)]
        self.cos_sin = dev(w.cos_sin)
        self.block_tables = dev(w.block_tables)


def step_inputs(w, seed):
    """New-token q, k, v of every layer for one step (host bf16 bits)."""
    rng = W.SplitMix64(seed)
    return [tuple(rng.normal_bf16(a.size, 1.0).reshape(a.shape) for a in (w.q[0], w.k[0], w.v[0]))
            for _ in range(w.num_layers)]


def oracle_step(orc, w, kc, vc, ctx, qkv):
    """The oracle's store of the new token at position ctx - 1, then its decode; kc, vc are
    updated in place.  Returns the fp64 output."""
    q0, k0, v0 = qkv
    pos = ctx.astype(np.int64) - 1
    blk = w.block_tables[np.arange(w.num_seqs), pos // W.BLOCK_SIZE].astype(np.int64)
    slots = blk * W.BLOCK_SIZE + pos % W.BLOCK_SIZE
    q = orc.rope_kv_store(q0, k0, v0, pos.astype(np.int32), w.cos_sin, slots, kc, vc)
    ref, _ = orc.decode(q, kc, vc, w.block_tables, ctx, w.scale)
    return ref


@pytest.mark.parametrize("name,P", [("tiny", 0), ("mix64", 0), ("long4", 512), ("prefix32", 0),
                                    ("mix64", 64)])
def test_early_metadata_gives_the_same_bits(pa, name, P):
    w = W.make(name)
    outs, caches = [], []
    for early in (False, True):
        kc, vc = dev_bf16(w.k_cache[0]), dev_bf16(w.v_cache[0])
        out = pa.decode_step(dev_bf16(w.q[0]), dev_bf16(w.k[0]), dev_bf16(w.v[0]), dev(w.cos_sin), kc,
                             vc, dev(w.block_tables), dev(w.context_lens), w.max_context_len,
                             w.scale, partition_tokens=P, early_metadata=early)
        torch.cuda.synchronize()
        outs.append(host_bits(out))
        caches.append((host_bits(kc), host_bits(vc)))
    assert np.array_equal(outs[0], outs[1])
    assert np.array_equal(caches[0][0], caches[1][0]) and np.array_equal(caches[0][1], caches[1][1])
    check_status_clean(pa)


@pytest.mark.parametrize("P", [0, 64])
def test_early_metadata_layers_back_to_back(pa, orc, P):
    """Two steps of a 4-layer model, every layer's step launched right after the previous
    one with the flag, nothing synchronised in between.  Step 2 appends one more token to
    every sequence (the same blocks: no length is a multiple of 16)."""
    ctx1 = np.array([17, 40, 300, 701, 1001, 3, 250, 2047], np.int32)
    w = W.build("early_chain", ctx1, 400, 131, num_layers=4, max_blocks=130)
    ctx2 = ctx1 + 1
    w.cos_sin = W.rope_cos_sin_table(int(ctx2.max()))      # rows for step 2's positions too
    d = Layers(w)
    lens = [dev(ctx1), dev(ctx2)]
    steps = [step_inputs(w, 132), step_inputs(w, 133)]
    dev_in = [[tuple(dev_bf16(a) for a in qkv) for qkv in s] for s in steps]
    maxctx = int(ctx2.max())
    ws = pa.decode_workspace(dev_in[0][0][0], d.k_cache[0], maxctx, P)
    outs = [[torch.empty_like(dev_in[0][0][0]) for _ in range(w.num_layers)] for _ in range(2)]
    for s in range(2):
        for i in range(w.num_layers):
            q, k, v = dev_in[s][i]
            pa.decode_step(q, k, v, d.cos_sin, d.k_cache[i], d.v_cache[i], d.block_tables, lens[s],
                           maxctx, w.scale, partition_tokens=P, workspace=ws, out=outs[s][i],
                           early_metadata=True)
    torch.cuda.synchronize()
    for i in range(w.num_layers):
        kc, vc = w.k_cache[i].copy(), w.v_cache[i].copy()
        for s, ctx in enumerate((ctx1, ctx2)):
            ref = oracle_step(orc, w, kc, vc, ctx, steps[s][i])
            assert_out_close(host_bits(outs[s][i]), ref, f"step {s} layer {i}")
        assert np.array_equal(host_bits(d.v_cache[i]), vc)
        assert bf16_ulp_distance(host_bits(d.k_cache[i]), kc).max() <= 1
    check_status_clean(pa)


@pytest.mark.parametrize("name", ["mix64", "long4"])
def test_early_metadata_full_size_chain(pa, orc, name):
    """Three layers of a full-size workload back to back with the flag and one shared
    workspace: each layer's kernel resolves its work while the kernels of the layer before are
    still running (the merge lets it launch as soon as the merge starts), and every layer must
    still give the oracle's result."""
    base = W.make(name)
    L = 3
    d_kc = [dev_bf16(base.k_cache[0]) for _ in range(L)]
    d_vc = [dev_bf16(base.v_cache[0]) for _ in range(L)]
    rng_inputs = [tuple(W.SplitMix64(170 + i).normal_bf16(a.size, 1.0).reshape(a.shape)
                        for a in (base.q[0], base.k[0], base.v[0])) for i in range(L)]
    dev_in = [tuple(dev_bf16(a) for a in t) for t in rng_inputs]
    cos_sin, bt, ctx = dev(base.cos_sin), dev(base.block_tables), dev(base.context_lens)
    P = base.partition_tokens
    ws = pa.decode_workspace(dev_in[0][0], d_kc[0], base.max_context_len, P)
    outs = [torch.empty_like(dev_in[0][0]) for _ in range(L)]
    for i in range(L):
        q, k, v = dev_in[i]
        pa.decode_step(q, k, v, cos_sin, d_kc[i], d_vc[i], bt, ctx, base.max_context_len,
                       base.scale, partition_tokens=P, workspace=ws, out=outs[i],
                       early_metadata=i > 0)
    torch.cuda.synchronize()
    for i in range(L):
        kc, vc = base.k_cache[0].copy(), base.v_cache[0].copy()
        ref = oracle_step(orc, base, kc, vc, base.context_lens, rng_inputs[i])
        assert_out_close(host_bits(outs[i]), ref, f"{name} layer {i}")
        assert np.array_equal(host_bits(d_vc[i]), vc)
    check_status_clean(pa)


def test_early_metadata_layers_in_a_cuda_graph(pa, orc):
    """The same chain captured once and replayed: each replay appends the next token."""
    ctx0 = np.array([33, 90, 517, 1500], np.int32)
    w = W.build("early_graph", ctx0, 300, 141, num_layers=3, max_blocks=100)
    w.cos_sin = W.rope_cos_sin_table(int(ctx0.max()) + 8)  # rows for the replays' positions
    d = Layers(w)
    lens = dev(ctx0)
    qkv_dev = [tuple(dev_bf16(a) for a in qkv) for qkv in step_inputs(w, 142)]
    maxctx = int(ctx0.max()) + 8
    ws = pa.decode_workspace(qkv_dev[0][0], d.k_cache[0], maxctx, 0)
    outs = [torch.empty_like(qkv_dev[0][0]) for _ in range(w.num_layers)]

    def chain():
        for i in range(w.num_layers):
            q, k, v = qkv_dev[i]
            pa.decode_step(q, k, v, d.cos_sin, d.k_cache[i], d.v_cache[i], d.block_tables, lens,
                           maxctx, w.scale, workspace=ws, out=outs[i], early_metadata=True)

    kc = [w.k_cache[i].copy() for i in range(w.num_layers)]
    vc = [w.v_cache[i].copy() for i in range(w.num_layers)]
    ctx = ctx0.copy()
    host_qkv = step_inputs(w, 142)
    chain()                                    # step at ctx0 (also warms the library up)
    torch.cuda.synchronize()
    for i in range(w.num_layers):
        oracle_step(orc, w, kc[i], vc[i], ctx, host_qkv[i])
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        chain()
    for rep in range(3):                       # each replay: one more token per sequence
        ctx = ctx + 1
        lens.copy_(dev(ctx))
        host_qkv = step_inputs(w, 150 + rep)
        for t, qkv in zip(qkv_dev, host_qkv):
            for dst, src in zip(t, qkv):
                dst.copy_(dev_bf16(src))
        torch.cuda.synchronize()      # the copy kernel above writes the lengths the replay reads early
        graph.replay()
        torch.cuda.synchronize()
        for i in range(w.num_layers):
            ref = oracle_step(orc, w, kc[i], vc[i], ctx, host_qkv[i])
            assert_out_close(host_bits(outs[i]), ref, f"replay {rep} layer {i}")
            assert np.array_equal(host_bits(d.v_cache[i]), vc[i])
    check_status_clean(pa)


def test_early_metadata_fp8_step_gives_the_same_bits(pa):
    w = W.make("mix64")
    kc16 = dev_bf16(w.k_cache[0]).float()
    vc16 = dev_bf16(w.v_cache[0]).float()

    def codes(c):
        scale = (c.abs().nan_to_num(0.0).amax(dim=(0, 2, 3)).clamp_min(1e-3) / 448.0).contiguous()
        q8 = (c / scale[None, :, None, None]).clamp(-448, 448).to(torch.float8_e4m3fn)
        return q8.view(torch.uint8).contiguous(), scale

    k8, ks = codes(kc16)
    v8, vs = codes(vc16)
    outs, caches = [], []
    for early in (False, True):
        kc, vc = k8.clone(), v8.clone()
        out = pa.decode_step_fp8(dev_bf16(w.q[0]), dev_bf16(w.k[0]), dev_bf16(w.v[0]), dev(w.cos_sin),
                                 kc, vc, ks, vs, dev(w.block_tables), dev(w.context_lens),
                                 w.max_context_len, w.scale, early_metadata=early)
        torch.cuda.synchronize()
        outs.append(host_bits(out))
        caches.append((kc.cpu().numpy(), vc.cpu().numpy()))
    assert np.array_equal(outs[0], outs[1])
    assert np.array_equal(caches[0][0], caches[1][0]) and np.array_equal(caches[0][1], caches[1][1])
    check_status_clean(pa)
