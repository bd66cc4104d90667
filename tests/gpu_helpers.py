"""Helpers for the GPU tests: upload host workloads, compare bf16 results with the oracle."""

from __future__ import annotations

import numpy as np
import torch

from paged_kv_cache_244_gb300 import workloads as W

OUT_ATOL = 1e-2   # |gpu - oracle| <= 1e-2 + 1e-2 |oracle| for the bf16 attention output
OUT_RTOL = 1e-2


def dev_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in units in the last place between bf16 bit patterns (+0 and -0 equal)."""
    def ordered(x):
        x = x.astype(np.int32)
        mag = x & 0x7FFF
        return np.where(x & 0x8000, -mag, mag)
    return np.abs(ordered(a) - ordered(b))


def assert_out_close(gpu_bits: np.ndarray, ref_f64: np.ndarray, what: str = "out"):
    g = W.bf16_bits_to_f32(gpu_bits).astype(np.float64)
    err = np.abs(g - ref_f64)
    bound = OUT_ATOL + OUT_RTOL * np.abs(ref_f64)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first "
                             f"{[(tuple(i), g[tuple(i)], ref_f64[tuple(i)]) for i in idx]}")


class DeviceLayer:
    """One layer of a workload on the GPU (caches, new-token tensors, tables)."""

    def __init__(self, w: W.Workload, layer: int = 0, q=None, k_cache=None, v_cache=None):
        self.q = dev_bf16(w.q[layer] if q is None else q)
        self.k = dev_bf16(w.k[layer])
        self.v = dev_bf16(w.v[layer])
        self.k_cache = dev_bf16(w.k_cache[layer] if k_cache is None else k_cache)
        self.v_cache = dev_bf16(w.v_cache[layer] if v_cache is None else v_cache)
        self.positions = dev(w.positions)
        self.slot_mapping = dev(w.slot_mapping)
        self.cos_sin = dev(w.cos_sin)
        self.block_tables = dev(w.block_tables)
        self.context_lens = dev(w.context_lens)
