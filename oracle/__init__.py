"""fp64 CPU oracle for paged GQA decode attention and the fused RoPE + KV-cache store.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code with the CUDA
library in ``paged_kv_cache_244_gb300`` and the library never imports it.

The arithmetic lives in ``oracle.cpp`` (plain C++17, double precision, one thread per
(sequence, KV head) unit).  This module only compiles it with the host C++ compiler and
marshals numpy arrays into it.  The citations for each definition are in ``oracle.cpp``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
SOURCE = _HERE / "oracle.cpp"
LIBRARY = _HERE / "liboracle.so"


def build(force: bool = False, src: Path = SOURCE, out: Path = LIBRARY) -> Path:
    """Compile an oracle source file into a shared library (g++, -O2, strict fp)."""
    src, out = Path(src), Path(out)
    if force or not out.exists() or out.stat().st_mtime < src.stat().st_mtime:
        tmp = out.with_name(out.name + f".tmp{os.getpid()}")
        cmd = ["g++", "-std=c++17", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC",
               "-shared", "-pthread", str(src), "-o", str(tmp)]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class Oracle:
    """numpy front end to one compiled copy of oracle.cpp."""

    def __init__(self, lib_path: Path):
        lib = ctypes.CDLL(str(lib_path))
        p, i, d = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_to_f64.restype = d
        lib.orc_f64_to_bf16.argtypes = [d]
        lib.orc_f64_to_bf16.restype = ctypes.c_uint16
        lib.orc_rope_rotate_f64.argtypes = [p, i, p, p]
        lib.orc_rope_rotate_f64.restype = i
        lib.orc_rope_kv_store.argtypes = [i, i, i, i, i, p, p, p, p, p, i, p, p, p, i]
        lib.orc_rope_kv_store.restype = i
        lib.orc_decode.argtypes = [i, i, i, i, i, p, p, p, i, p, i, p, d, i, p, p]
        lib.orc_decode.restype = i
        lib.orc_decode_partitioned.argtypes = [i, i, i, i, i, p, p, p, i, p, i, p, d, i, i, p]
        lib.orc_decode_partitioned.restype = i
        lib.orc_prefill.argtypes = [i, i, i, i, i, p, p, p, p, p, i, p, i, d, i, p, p]
        lib.orc_prefill.restype = i
        lib.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_to_f64.restype = d
        lib.orc_f64_to_e4m3.argtypes = [d]
        lib.orc_f64_to_e4m3.restype = ctypes.c_uint8
        lib.orc_quantize_cache.argtypes = [ctypes.c_int64, i, i, i, p, p, p]
        lib.orc_quantize_cache.restype = i
        lib.orc_rope_kv_store_fp8.argtypes = [i, i, i, i, i, p, p, p, p, p, i, p, p, p, i, p, p]
        lib.orc_rope_kv_store_fp8.restype = i
        lib.orc_decode_fp8.argtypes = [i, i, i, i, i, p, p, p, p, p, i, p, i, p, d, i, p, p]
        lib.orc_decode_fp8.restype = i
        lib.orc_copy_blocks.argtypes = [i, ctypes.c_int64, p, ctypes.c_int64, p, ctypes.c_int64, p, i]
        lib.orc_copy_blocks.restype = ctypes.c_int64
        lib.orc_hardware_threads.argtypes = []
        lib.orc_hardware_threads.restype = i
        self.lib = lib

    def prefill(self, q, q_start, k_cache, v_cache, block_tables, context_lens, scale, nthreads=0):
        """Paged (chunked) prefill: query i of sequence s, at position
        context_lens[s] - n_s + i, attends causally to its cached tokens 0..position.
        q [T, Hq, D] bf16 bits, q_start [S + 1]; returns (out fp64 [T, Hq, D], out bf16 bits)."""
        q = _c(q, np.uint16)
        qs = _c(q_start, np.int32)
        kc, vc = _c(k_cache, np.uint16), _c(v_cache, np.uint16)
        bt = _c(block_tables, np.int32)
        ctx = _c(context_lens, np.int32)
        T, Hq, D = q.shape
        nb, Hkv, B, _ = kc.shape
        S = ctx.shape[0]
        assert qs.shape == (S + 1,) and qs[-1] == T
        out = np.empty((T, Hq, D), np.float64)
        outb = np.empty((T, Hq, D), np.uint16)
        rc = self.lib.orc_prefill(S, Hq, Hkv, D, B, _ptr(q), _ptr(qs), _ptr(ctx), _ptr(kc), _ptr(vc),
                                  nb, _ptr(bt), bt.shape[1] if bt.ndim == 2 else 0, float(scale),
                                  int(nthreads), _ptr(out), _ptr(outb))
        if rc != 0:
            raise ValueError("orc_prefill rejected its arguments")
        return out, outb

    # ---- FP8 (E4M3) KV cache -----------------------------------------------------------
    def e4m3_to_f64(self, code: int) -> float:
        return float(self.lib.orc_e4m3_to_f64(int(code) & 0xFF))

    def f64_to_e4m3(self, x: float) -> int:
        """E4M3 code nearest to x, ties to even, saturating to +-448 (NaN stays NaN)."""
        return int(self.lib.orc_f64_to_e4m3(float(x)))

    def quantize_cache(self, cache_bits, scale) -> np.ndarray:
        """E4M3 codes of a bf16 cache [num_blocks, Hkv, B, D] (bits) with one fp32 scale per
        KV head: code of fp32(x) * fp32(1 / scale)."""
        src = _c(cache_bits, np.uint16)
        nb, Hkv, B, D = src.shape
        scale = _c(scale, np.float32)
        assert scale.shape == (Hkv,)
        dst = np.empty(src.shape, np.uint8)
        if self.lib.orc_quantize_cache(src.size, Hkv, B, D, _ptr(src), _ptr(scale), _ptr(dst)) != 0:
            raise ValueError("orc_quantize_cache rejected its arguments")
        return dst

    def rope_kv_store_fp8(self, q, k, v, positions, cos_sin, slot_mapping, k_cache, v_cache,
                          k_scale, v_scale):
        """As rope_kv_store, into uint8 E4M3 caches with per-KV-head scales (in place)."""
        q = np.array(q, dtype=np.uint16, copy=True, order="C")
        k, v = _c(k, np.uint16), _c(v, np.uint16)
        positions = _c(positions, np.int32)
        cos_sin = _c(cos_sin, np.float32)
        slot_mapping = _c(slot_mapping, np.int64)
        k_scale, v_scale = _c(k_scale, np.float32), _c(v_scale, np.float32)
        for c in (k_cache, v_cache):
            assert c.dtype == np.uint8 and c.flags.c_contiguous
        T, Hq, D = q.shape
        nb, Hkv, B, D2 = k_cache.shape
        assert D2 == D and k.shape == (T, Hkv, D) and v.shape == (T, Hkv, D)
        assert k_scale.shape == (Hkv,) and v_scale.shape == (Hkv,)
        rc = self.lib.orc_rope_kv_store_fp8(T, Hq, Hkv, D, B, _ptr(q), _ptr(k), _ptr(v),
                                            _ptr(positions), _ptr(cos_sin), cos_sin.shape[0],
                                            _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), nb,
                                            _ptr(k_scale), _ptr(v_scale))
        if rc != 0:
            raise ValueError("orc_rope_kv_store_fp8 rejected its arguments")
        return q

    def decode_fp8(self, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                   scale, nthreads=0):
        """Decode over uint8 E4M3 caches; returns (out fp64 [S, Hq, D], out bf16 bits)."""
        q = _c(q, np.uint16)
        kc, vc = _c(k_cache, np.uint8), _c(v_cache, np.uint8)
        ks, vs = _c(k_scale, np.float32), _c(v_scale, np.float32)
        bt = _c(block_tables, np.int32)
        ctx = _c(context_lens, np.int32)
        S, Hq, D = q.shape
        nb, Hkv, B, _ = kc.shape
        out = np.empty((S, Hq, D), np.float64)
        outb = np.empty((S, Hq, D), np.uint16)
        rc = self.lib.orc_decode_fp8(S, Hq, Hkv, D, B, _ptr(q), _ptr(kc), _ptr(vc), _ptr(ks),
                                     _ptr(vs), nb, _ptr(bt), bt.shape[1] if bt.ndim == 2 else 0,
                                     _ptr(ctx), float(scale), int(nthreads), _ptr(out), _ptr(outb))
        if rc != 0:
            raise ValueError("orc_decode_fp8 rejected its arguments")
        return out, outb

    def copy_blocks(self, src, dst, pairs) -> int:
        """Block copy (copy-on-write, swap out / in): for each (from, to) row of `pairs` and
        each pool index c, dst[c][to] = src[c][from].  src, dst: lists of equally shaped
        [num_blocks, ...] uint16 arrays (dst written in place).  Returns the pairs skipped
        because a block id is outside its pool."""
        assert len(src) == len(dst)
        for a in list(src) + list(dst):
            assert a.dtype == np.uint16 and a.flags.c_contiguous
        block_elems = int(np.prod(src[0].shape[1:])) if src else 1
        for a in list(src) + list(dst):
            assert int(np.prod(a.shape[1:])) == block_elems
        pairs = _c(pairs, np.int64).reshape(-1, 2)
        arr = ctypes.c_void_p * max(1, len(src))
        sp = arr(*[a.ctypes.data for a in src])
        dp = arr(*[a.ctypes.data for a in dst])
        src_blocks = src[0].shape[0] if src else 0
        dst_blocks = dst[0].shape[0] if dst else 0
        rc = self.lib.orc_copy_blocks(len(src), block_elems, ctypes.cast(sp, ctypes.c_void_p),
                                      src_blocks, ctypes.cast(dp, ctypes.c_void_p), dst_blocks,
                                      _ptr(pairs), pairs.shape[0])
        if rc < 0:
            raise ValueError("orc_copy_blocks rejected its arguments")
        return int(rc)

    def hardware_threads(self) -> int:
        return int(self.lib.orc_hardware_threads())

    def bf16_to_f64(self, bits: int) -> float:
        return float(self.lib.orc_bf16_to_f64(int(bits) & 0xFFFF))

    def f64_to_bf16(self, x: float) -> int:
        """bf16 bit pattern nearest to x, ties to even (one rounding from double)."""
        return int(self.lib.orc_f64_to_bf16(float(x)))

    def rope_rotate_f64(self, x_bits, cos_sin_row) -> np.ndarray:
        """rotate_half RoPE of one head vector (bf16 bits) by one [cos | sin] row, in double."""
        x = _c(x_bits, np.uint16)
        row = _c(cos_sin_row, np.float32)
        y = np.empty(x.shape[0], np.float64)
        if self.lib.orc_rope_rotate_f64(_ptr(x), x.shape[0], _ptr(row), _ptr(y)) != 0:
            raise ValueError("orc_rope_rotate_f64 rejected its arguments")
        return y

    def rope_kv_store(self, q, k, v, positions, cos_sin, slot_mapping, k_cache, v_cache):
        """Fused RoPE + KV-cache store on host arrays of bf16 bits (uint16).

        Returns the rotated copy of q [T, Hq, D]; k_cache / v_cache [num_blocks, Hkv, B, D]
        (C-contiguous uint16) receive rotated k and raw v at slot_mapping, in place.
        """
        q = np.array(q, dtype=np.uint16, copy=True, order="C")
        k, v = _c(k, np.uint16), _c(v, np.uint16)
        positions = _c(positions, np.int32)
        cos_sin = _c(cos_sin, np.float32)
        slot_mapping = _c(slot_mapping, np.int64)
        for c in (k_cache, v_cache):
            assert c.dtype == np.uint16 and c.flags.c_contiguous
        T, Hq, D = q.shape
        nb, Hkv, B, D2 = k_cache.shape
        assert D2 == D and k.shape == (T, Hkv, D) and v.shape == (T, Hkv, D)
        rc = self.lib.orc_rope_kv_store(T, Hq, Hkv, D, B, _ptr(q), _ptr(k), _ptr(v),
                                        _ptr(positions), _ptr(cos_sin), cos_sin.shape[0],
                                        _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), nb)
        if rc != 0:
            raise ValueError("orc_rope_kv_store rejected its arguments")
        return q

    def decode(self, q, k_cache, v_cache, block_tables, context_lens, scale, nthreads=0):
        """Unsplit paged decode.  Returns (out_f64 [S,Hq,D], out_bf16 bits [S,Hq,D])."""
        q = _c(q, np.uint16)
        k_cache, v_cache = _c(k_cache, np.uint16), _c(v_cache, np.uint16)
        bt = _c(block_tables, np.int32)
        ctx = _c(context_lens, np.int32)
        S, Hq, D = q.shape
        nb, Hkv, B, _ = k_cache.shape
        out = np.zeros((S, Hq, D), np.float64)
        outb = np.zeros((S, Hq, D), np.uint16)
        rc = self.lib.orc_decode(S, Hq, Hkv, D, B, _ptr(q), _ptr(k_cache), _ptr(v_cache), nb,
                                 _ptr(bt), bt.shape[1], _ptr(ctx), float(scale), int(nthreads),
                                 _ptr(out), _ptr(outb))
        if rc != 0:
            raise ValueError("orc_decode rejected its arguments")
        return out, outb

    def decode_partitioned(self, q, k_cache, v_cache, block_tables, context_lens, scale,
                           partition_tokens, nthreads=0):
        """Flash-Decode form: per-partition (m, l, o) merged by log-sum-exp.  Returns out_f64."""
        q = _c(q, np.uint16)
        k_cache, v_cache = _c(k_cache, np.uint16), _c(v_cache, np.uint16)
        bt = _c(block_tables, np.int32)
        ctx = _c(context_lens, np.int32)
        S, Hq, D = q.shape
        nb, Hkv, B, _ = k_cache.shape
        out = np.zeros((S, Hq, D), np.float64)
        rc = self.lib.orc_decode_partitioned(S, Hq, Hkv, D, B, _ptr(q), _ptr(k_cache),
                                             _ptr(v_cache), nb, _ptr(bt), bt.shape[1], _ptr(ctx),
                                             float(scale), int(partition_tokens), int(nthreads),
                                             _ptr(out))
        if rc != 0:
            raise ValueError("orc_decode_partitioned rejected its arguments")
        return out


_default: Oracle | None = None


def default() -> Oracle:
    """The oracle compiled from oracle.cpp (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default
