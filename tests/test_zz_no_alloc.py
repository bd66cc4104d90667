"""pa_decode_static_workspace: decode for callers that cannot allocate device memory.

Some callers may not allocate while a decode step runs: an engine that has handed all free
HBM to its KV-cache pool, a plugin whose enqueue path forbids allocation, a real-time loop
that must not take allocator locks.  This entry point runs the same decode with the
library's built-in scratch array instead of a caller-provided workspace.  The test calls it
through the C ABI and checks it bit for bit against pa_decode with a caller workspace and
against the fp64 oracle, on two calls in a row with different inputs after a call that left
NaN partials in the scratch (the scratch keeps the previous call's contents), and checks that
a call needing more scratch than the array holds is refused without launching anything.
This file is collected last so that a failure here stops a -x run after every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import OUT_ATOL, OUT_RTOL, DeviceLayer, host_bits
from paged_kv_cache_244_gb300 import _build
from paged_kv_cache_244_gb300 import workloads as W

pytestmark = pytest.mark.gpu

STATIC_BYTES = 8 << 20   # PA_STATIC_WORKSPACE_BYTES in include/pa.h


@pytest.fixture(scope="module")
def pa():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    _build.build()
    from paged_kv_cache_244_gb300 import binding
    L = binding.lib()
    f = L.pa_decode_static_workspace
    p, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [ctypes.POINTER(binding.pa_dims), i, p, p, p, i, p, i, p, i, ctypes.c_float, i, p, p]
    f.restype = i
    return binding


def call_static(pa, d, w, P, out):
    dims = pa.make_dims(w.num_q_heads, w.num_kv_heads)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    return pa.lib().pa_decode_static_workspace(
        ctypes.byref(dims), w.num_seqs, ptr(d.q), ptr(d.k_cache), ptr(d.v_cache), w.num_blocks,
        ptr(d.block_tables), w.max_blocks, ptr(d.context_lens), w.max_context_len, w.scale, P,
        ptr(out), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def prepared(name, orc):
    w = W.make(name)
    kc, vc = w.k_cache[0].copy(), w.v_cache[0].copy()
    q = orc.rope_kv_store(w.q[0], w.k[0], w.v[0], w.positions, w.cos_sin, w.slot_mapping, kc, vc)
    return w, DeviceLayer(w, q=q, k_cache=kc, v_cache=vc)


def test_static_workspace_matches_decode_on_two_calls(pa):
    """The static entry point runs the same kernels with the same split as pa_decode, so its
    output is the same bits; both agree with the oracle.  Before the two calls, a call of a
    different shape with a NaN query fills the scratch with NaN partial results, so a call that
    read a partial it did not write itself would show NaN or differ."""
    orc = oracle.default()
    w0, d0 = prepared("prefix32", orc)
    d0.q.fill_(float("nan"))
    poison = torch.empty_like(d0.q)
    assert call_static(pa, d0, w0, 512, poison) == pa.PA_OK
    torch.cuda.synchronize()
    assert torch.isnan(poison.float()).all()
    for name in ("mix64", "long4"):               # two calls in a row, different shapes
        w, d = prepared(name, orc)
        P = w.partition_tokens            # mix64: even split; long4: 512-token partitions
        need = pa.decode_workspace_size(w.num_q_heads, w.num_kv_heads, w.num_seqs,
                                        w.max_context_len, P)
        assert 0 < need <= STATIC_BYTES
        ref = pa.decode(d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens,
                        w.max_context_len, w.scale, partition_tokens=P)
        out = torch.full_like(d.q, float("nan"))
        assert call_static(pa, d, w, P, out) == pa.PA_OK
        torch.cuda.synchronize()
        got = host_bits(out)
        assert np.array_equal(got, host_bits(ref)), name
        q = W.bf16_bits_to_f32(host_bits(d.q)).astype(np.float64)
        kc = host_bits(d.k_cache)
        vc = host_bits(d.v_cache)
        want, _ = orc.decode(host_bits(d.q), kc, vc, w.block_tables, w.context_lens, w.scale)
        g = W.bf16_bits_to_f32(got).astype(np.float64)
        assert np.isfinite(g).all() and np.isfinite(q).all()
        assert (np.abs(g - want) <= OUT_ATOL + OUT_RTOL * np.abs(want)).all(), name
        rc, flags = pa.get_device_status()
        assert rc == 0 and flags == 0


def test_static_workspace_refuses_oversized_requests(pa):
    orc = oracle.default()
    w, d = prepared("mix64", orc)
    need = pa.decode_workspace_size(w.num_q_heads, w.num_kv_heads, w.num_seqs,
                                    w.max_context_len, 16)     # one range per block: too many
    assert need > STATIC_BYTES
    out = torch.zeros_like(d.q)
    assert call_static(pa, d, w, 16, out) == pa.PA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert (host_bits(out) == 0).all()           # nothing was launched
