"""pa_stage_copy through the C ABI: host -> device, device -> host and device -> device copies
are byte-exact at sizes from one 16-byte word to several MiB (ragged against the kernel's
grid), pageable host memory is refused, and a copy issued right after a kernel on the same
stream sees that kernel's writes."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_helpers import dev, dev_bf16, host_bits
from paged_kv_cache_244_gb300 import _build
from paged_kv_cache_244_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SIZES = [16, 4096 + 16, 327424, (1 << 20) + 48, 9 * (1 << 20) + 16 * 257]


@pytest.fixture(scope="module")
def pa():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    _build.build()
    from paged_kv_cache_244_gb300 import binding
    return binding


def seeded_bytes(n, seed):
    words = W.SplitMix64(seed).uint64((n + 7) // 8)
    return np.frombuffer(words.tobytes(), dtype=np.uint8)[:n].copy()


@pytest.mark.parametrize("n", SIZES)
def test_host_to_device_to_host(pa, n):
    src = torch.from_numpy(seeded_bytes(n, 700 + n)).pin_memory()
    d = torch.full((n,), 0xA5, dtype=torch.uint8, device="cuda")
    pa.stage_copy(d, src)
    back = torch.zeros(n, dtype=torch.uint8).pin_memory()
    pa.stage_copy(back, d)
    torch.cuda.synchronize()
    assert torch.equal(d.cpu(), src)
    assert torch.equal(back, src)


@pytest.mark.parametrize("n", SIZES[:3])
def test_device_to_device(pa, n):
    a = torch.from_numpy(seeded_bytes(n, 900 + n)).cuda()
    b = torch.zeros(n, dtype=torch.uint8, device="cuda")
    pa.stage_copy(b, a)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_pageable_host_memory_is_refused(pa):
    src = torch.from_numpy(seeded_bytes(4096, 5))          # not pinned
    d = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        pa.stage_copy(d, src)                               # the binding refuses it
    import ctypes
    rc = pa.lib().pa_stage_copy(ctypes.c_void_p(d.data_ptr()), ctypes.c_void_p(src.data_ptr()), 4096, None)
    assert rc == pa.PA_ERR_MEMORY                           # and so does the library


def test_copy_after_a_kernel_sees_its_output(pa):
    """The decode step's output read back by the next call on the stream, no synchronisation
    in between: the staging kernel waits for the decode kernels before it reads."""
    w = W.make("mix64")
    kc, vc = dev_bf16(w.k_cache[0]), dev_bf16(w.v_cache[0])
    out = pa.decode_step(dev_bf16(w.q[0]), dev_bf16(w.k[0]), dev_bf16(w.v[0]), dev(w.cos_sin), kc, vc,
                         dev(w.block_tables), dev(w.context_lens), w.max_context_len, w.scale)
    h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    pa.stage_copy(h, out)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(out), h.view(torch.int16).numpy().view(np.uint16))
