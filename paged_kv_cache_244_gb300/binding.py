"""Thin Python binding of the C ABI in include/pa.h (argument marshalling only).

Every function here checks tensor devices, dtypes, shapes and contiguity, passes raw
device pointers and the current CUDA stream to libpa_gb300.so, and turns a negative return
code into PaError.  All computation happens in the library's CUDA kernels: there is no
fallback, and using any function without the compiled library raises at once.
"""

from __future__ import annotations

import ctypes
from pathlib import Path

import torch

LIBRARY = Path(__file__).resolve().parent / "libpa_gb300.so"

PA_OK = 0
PA_ERR_NULL = -1
PA_ERR_SHAPE = -2
PA_ERR_RANGE = -3
PA_ERR_WORKSPACE = -4
PA_ERR_CUDA = -5
PA_ERR_DEVICE_OOB = -6
PA_ERR_TIMEOUT = -7
PA_ERR_ALIGN = -8
PA_ERR_MEMORY = -9
PA_MAX_BLOCK_CACHES = 256
PA_STEP_EARLY_METADATA = 0x1

PA_FLAG_BLOCK_ID_OOB = 0x1
PA_FLAG_CONTEXT_LEN_OOB = 0x2
PA_FLAG_SLOT_OOB = 0x4
PA_FLAG_POSITION_OOB = 0x8
PA_FLAG_TIMEOUT = 0x10


class PaError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} ({code})")
        self.code = code


class pa_dims(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32)]


_lib = None


def lib():
    """The loaded C library with argument types declared (raises if it was never built)."""
    global _lib
    if _lib is None:
        if not LIBRARY.exists():
            raise RuntimeError(f"{LIBRARY.name} is not built: run __graft_entry__.build() "
                               "(the CUDA kernels are the only implementation)")
        L = ctypes.CDLL(str(LIBRARY))
        p, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        pd = ctypes.POINTER(pa_dims)
        L.pa_rope_kv_store.argtypes = [pd, i, p, p, p, p, p, i, p, p, p, i, p]
        L.pa_rope_kv_store.restype = i
        L.pa_decode_partition_tokens.argtypes = [pd, i, i, i]
        L.pa_decode_partition_tokens.restype = i
        L.pa_decode_workspace_size.argtypes = [pd, i, i, i]
        L.pa_decode_workspace_size.restype = ctypes.c_size_t
        L.pa_decode.argtypes = [pd, i, p, p, p, i, p, i, p, i, f, i, p, ctypes.c_size_t, p, p]
        L.pa_decode.restype = i
        L.pa_decode_step.argtypes = [pd, i, p, p, p, p, i, p, p, i, p, i, p, i, f, i, p,
                                     ctypes.c_size_t, p, ctypes.c_uint, p]
        L.pa_decode_step.restype = i
        L.pa_rope_kv_store_fp8.argtypes = [pd, i, p, p, p, p, p, i, p, p, p, i, p, p, p]
        L.pa_rope_kv_store_fp8.restype = i
        L.pa_decode_fp8.argtypes = [pd, i, p, p, p, p, p, i, p, i, p, i, f, i, p, ctypes.c_size_t,
                                    p, p]
        L.pa_decode_fp8.restype = i
        L.pa_decode_step_fp8.argtypes = [pd, i, p, p, p, p, i, p, p, p, p, i, p, i, p, i, f, i, p,
                                         ctypes.c_size_t, p, ctypes.c_uint, p]
        L.pa_decode_step_fp8.restype = i
        L.pa_gather_checksum.argtypes = [pd, i, p, p, i, p, i, p, i, p, p]
        L.pa_gather_checksum.restype = i
        L.pa_gather_checksum_fp8.argtypes = [pd, i, p, p, i, p, i, p, i, p, p]
        L.pa_gather_checksum_fp8.restype = i
        L.pa_prefill.argtypes = [pd, i, i, p, p, i, p, p, i, p, i, p, i, f, p, p]
        L.pa_prefill.restype = i
        L.pa_copy_blocks.argtypes = [pd, i, p, ctypes.c_int64, p, ctypes.c_int64, p, i, p]
        L.pa_copy_blocks.restype = i
        L.pa_stage_copy.argtypes = [p, p, ctypes.c_size_t, p]
        L.pa_stage_copy.restype = i
        L.pa_set_timing_jitter.argtypes = [ctypes.c_uint32, ctypes.c_uint32]
        L.pa_set_timing_jitter.restype = i
        L.pa_get_device_status.argtypes = [p, ctypes.POINTER(ctypes.c_uint32)]
        L.pa_get_device_status.restype = i
        L.pa_selftest_wait_timeout.argtypes = [ctypes.c_uint32, p]
        L.pa_selftest_wait_timeout.restype = i
        L.pa_status_string.argtypes = [i]
        L.pa_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().pa_status_string(int(code)).decode()


def _check(code: int, what: str):
    if code != PA_OK:
        raise PaError(code, what)


def _dev_ptr(t: torch.Tensor | None, name: str, dtype=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_dims(num_q_heads: int, num_kv_heads: int, head_dim: int = 128, block_size: int = 16):
    return pa_dims(num_q_heads, num_kv_heads, head_dim, block_size)


def rope_kv_store(q, k, v, positions, cos_sin, slot_mapping, k_cache, v_cache, stream=None):
    """Fused RoPE + KV-cache store (pa_rope_kv_store): rotates q in place, writes the caches.

    q [T, Hq, D] bf16; k, v [T, Hkv, D] bf16; positions [T] int32; cos_sin [max_pos, D] fp32;
    slot_mapping [T] int64; k_cache, v_cache [num_blocks, Hkv, B, D] bf16.
    """
    T, Hq, D = q.shape
    nb, Hkv, B, D2 = k_cache.shape
    if D2 != D or tuple(k.shape) != (T, Hkv, D) or tuple(v.shape) != (T, Hkv, D):
        raise ValueError("shape mismatch between q, k, v and the caches")
    if tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache and v_cache differ in shape")
    if positions.shape != (T,) or slot_mapping.shape != (T,) or cos_sin.shape[1] != D:
        raise ValueError("positions / slot_mapping / cos_sin shape mismatch")
    dims = make_dims(Hq, Hkv, D, B)
    bf = torch.bfloat16
    rc = lib().pa_rope_kv_store(
        ctypes.byref(dims), T, _dev_ptr(q, "q", bf), _dev_ptr(k, "k", bf), _dev_ptr(v, "v", bf),
        _dev_ptr(positions, "positions", torch.int32), _dev_ptr(cos_sin, "cos_sin", torch.float32),
        cos_sin.shape[0], _dev_ptr(slot_mapping, "slot_mapping", torch.int64),
        _dev_ptr(k_cache, "k_cache", bf), _dev_ptr(v_cache, "v_cache", bf), nb, _stream(stream))
    _check(rc, "pa_rope_kv_store")


def decode_partition_tokens(num_q_heads, num_kv_heads, num_seqs, max_context_len,
                            partition_tokens=0, head_dim=128, block_size=16) -> int:
    dims = make_dims(num_q_heads, num_kv_heads, head_dim, block_size)
    rc = lib().pa_decode_partition_tokens(ctypes.byref(dims), num_seqs, max_context_len,
                                          partition_tokens)
    if rc < 0:
        raise PaError(rc, "pa_decode_partition_tokens")
    return rc


def decode_workspace_size(num_q_heads, num_kv_heads, num_seqs, max_context_len,
                          partition_tokens=0, head_dim=128, block_size=16) -> int:
    dims = make_dims(num_q_heads, num_kv_heads, head_dim, block_size)
    return int(lib().pa_decode_workspace_size(ctypes.byref(dims), num_seqs, max_context_len,
                                              partition_tokens))


def decode_workspace(q, k_cache, max_context_len, partition_tokens=0) -> torch.Tensor:
    """Allocate the workspace pa_decode needs for these shapes (no initialisation needed)."""
    S, Hq, D = q.shape
    _, Hkv, B, _ = k_cache.shape
    n = decode_workspace_size(Hq, Hkv, S, max_context_len, partition_tokens, D, B)
    if n == 0:
        raise PaError(PA_ERR_RANGE, "pa_decode_workspace_size")
    return torch.empty((n + 3) // 4, dtype=torch.float32, device=q.device)


def decode(q, k_cache, v_cache, block_tables, context_lens, max_context_len, scale,
           partition_tokens=0, workspace=None, out=None, stream=None):
    """Paged GQA decode attention (pa_decode).  Returns out [S, Hq, D] bf16.

    q [S, Hq, D] bf16; k_cache, v_cache [num_blocks, Hkv, B, D] bf16; block_tables
    [S, max_blocks] int32; context_lens [S] int32; max_context_len a host int bounding them.
    `workspace` (from decode_workspace) is allocated here when None.
    """
    S, Hq, D = q.shape
    nb, Hkv, B, D2 = k_cache.shape
    if D2 != D or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("cache shape mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("block_tables / context_lens shape mismatch")
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = decode_workspace(q, k_cache, max_context_len, partition_tokens)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    dims = make_dims(Hq, Hkv, D, B)
    bf = torch.bfloat16
    rc = lib().pa_decode(
        ctypes.byref(dims), S, _dev_ptr(q, "q", bf), _dev_ptr(k_cache, "k_cache", bf),
        _dev_ptr(v_cache, "v_cache", bf), nb, _dev_ptr(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev_ptr(context_lens, "context_lens", torch.int32),
        int(max_context_len), float(scale), int(partition_tokens), _dev_ptr(workspace, "workspace"),
        ws_bytes, _dev_ptr(out, "out", bf), _stream(stream))
    _check(rc, "pa_decode")
    return out


def decode_step(q, k, v, cos_sin, k_cache, v_cache, block_tables, context_lens, max_context_len,
                scale, partition_tokens=0, workspace=None, out=None, stream=None,
                early_metadata=False):
    """One fused decode step (pa_decode_step): RoPE + KV store of each sequence's new token at
    position context_lens[s] - 1, then decode attention, in one launch.  Returns out.

    q [S, Hq, D] bf16, NOT rotated (left unchanged); k, v [S, Hkv, D] bf16 (the new token);
    cos_sin [max_pos, D] fp32; the rest as for decode().  The caches get the new K and V.
    early_metadata sets PA_STEP_EARLY_METADATA: the caller promises that no kernel still
    running on the stream writes context_lens or block_tables, and the kernel resolves its
    work from them before the preceding kernel has finished.
    """
    S, Hq, D = q.shape
    nb, Hkv, B, D2 = k_cache.shape
    if D2 != D or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("cache shape mismatch")
    if tuple(k.shape) != (S, Hkv, D) or tuple(v.shape) != (S, Hkv, D):
        raise ValueError("k / v shape mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("block_tables / context_lens shape mismatch")
    if cos_sin.dim() != 2 or cos_sin.shape[1] != D:
        raise ValueError("cos_sin shape mismatch")
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = decode_workspace(q, k_cache, max_context_len, partition_tokens)
    ws_bytes = workspace.numel() * workspace.element_size()
    dims = make_dims(Hq, Hkv, D, B)
    bf = torch.bfloat16
    rc = lib().pa_decode_step(
        ctypes.byref(dims), S, _dev_ptr(q, "q", bf), _dev_ptr(k, "k", bf), _dev_ptr(v, "v", bf),
        _dev_ptr(cos_sin, "cos_sin", torch.float32), cos_sin.shape[0],
        _dev_ptr(k_cache, "k_cache", bf), _dev_ptr(v_cache, "v_cache", bf), nb,
        _dev_ptr(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _dev_ptr(context_lens, "context_lens", torch.int32), int(max_context_len), float(scale),
        int(partition_tokens), _dev_ptr(workspace, "workspace"), ws_bytes, _dev_ptr(out, "out", bf),
        PA_STEP_EARLY_METADATA if early_metadata else 0, _stream(stream))
    _check(rc, "pa_decode_step")
    return out


def prefill(q, q_start, k_cache, v_cache, block_tables, context_lens, max_query_len,
            max_context_len, scale, out=None, stream=None):
    """Paged (chunked) prefill attention (pa_prefill).  Returns out [T, Hq, D] bf16.

    q [T, Hq, D] bf16 (rotated); q_start [S + 1] int32 (rows of each sequence); context_lens
    [S] int32 (cached tokens including the new ones); max_query_len / max_context_len host
    bounds; caches and block_tables as for decode().
    """
    T, Hq, D = q.shape
    nb, Hkv, B, D2 = k_cache.shape
    S = context_lens.shape[0]
    if D2 != D or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("cache shape mismatch")
    if q_start.shape != (S + 1,) or block_tables.dim() != 2 or block_tables.shape[0] != S:
        raise ValueError("q_start / block_tables shape mismatch")
    if out is None:
        out = torch.empty_like(q)
    dims = make_dims(Hq, Hkv, D, B)
    bf = torch.bfloat16
    rc = lib().pa_prefill(
        ctypes.byref(dims), S, T, _dev_ptr(q, "q", bf), _dev_ptr(q_start, "q_start", torch.int32),
        int(max_query_len), _dev_ptr(k_cache, "k_cache", bf), _dev_ptr(v_cache, "v_cache", bf), nb,
        _dev_ptr(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _dev_ptr(context_lens, "context_lens", torch.int32), int(max_context_len), float(scale),
        _dev_ptr(out, "out", bf), _stream(stream))
    _check(rc, "pa_prefill")
    return out


# ---- FP8 (E4M3) caches: uint8 tensors of codes, fp32 scales [Hkv] per KV head ----------

def _fp8_args(k_cache, v_cache, k_scale, v_scale):
    nb, Hkv, B, D = k_cache.shape
    if tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache and v_cache differ in shape")
    if tuple(k_scale.shape) != (Hkv,) or tuple(v_scale.shape) != (Hkv,):
        raise ValueError("k_scale and v_scale must be [num_kv_heads] float32")
    u8, f32 = torch.uint8, torch.float32
    return (nb, Hkv, B, D, _dev_ptr(k_cache, "k_cache", u8), _dev_ptr(v_cache, "v_cache", u8),
            _dev_ptr(k_scale, "k_scale", f32), _dev_ptr(v_scale, "v_scale", f32))


def rope_kv_store_fp8(q, k, v, positions, cos_sin, slot_mapping, k_cache, v_cache, k_scale,
                      v_scale, stream=None):
    """pa_rope_kv_store_fp8: q rotated in place (bf16); rotated k and v stored as E4M3 codes
    (k_cache, v_cache uint8 [num_blocks, Hkv, B, D]) with per-KV-head scales."""
    T, Hq, D = q.shape
    nb, Hkv, B, D2, kc, vc, ks, vs = _fp8_args(k_cache, v_cache, k_scale, v_scale)
    if D2 != D or tuple(k.shape) != (T, Hkv, D) or tuple(v.shape) != (T, Hkv, D):
        raise ValueError("shape mismatch between q, k, v and the caches")
    if positions.shape != (T,) or slot_mapping.shape != (T,) or cos_sin.shape[1] != D:
        raise ValueError("positions / slot_mapping / cos_sin shape mismatch")
    dims = make_dims(Hq, Hkv, D, B)
    bf = torch.bfloat16
    rc = lib().pa_rope_kv_store_fp8(
        ctypes.byref(dims), T, _dev_ptr(q, "q", bf), _dev_ptr(k, "k", bf), _dev_ptr(v, "v", bf),
        _dev_ptr(positions, "positions", torch.int32), _dev_ptr(cos_sin, "cos_sin", torch.float32),
        cos_sin.shape[0], _dev_ptr(slot_mapping, "slot_mapping", torch.int64), kc, vc, nb, ks, vs,
        _stream(stream))
    _check(rc, "pa_rope_kv_store_fp8")


def gather_checksum(k_cache, v_cache, block_tables, context_lens, max_context_len, num_q_heads,
                    out_xor=None, stream=None):
    """pa_gather_checksum (bf16 caches) or pa_gather_checksum_fp8 (uint8 E4M3 caches): XOR of the
    tile words of every (sequence, KV head)'s context, read through the block tables the way
    the decode reads them.  out_xor [S, Hkv] int32 (zero-filled here when None) is XORed into
    and returned."""
    nb, Hkv, B, D = k_cache.shape
    S = context_lens.shape[0]
    if tuple(v_cache.shape) != tuple(k_cache.shape) or block_tables.shape[0] != S:
        raise ValueError("shape mismatch between the caches, block_tables and context_lens")
    fp8 = k_cache.dtype == torch.uint8
    dt = torch.uint8 if fp8 else torch.bfloat16
    if out_xor is None:
        out_xor = torch.zeros((S, Hkv), dtype=torch.int32, device=k_cache.device)
    dims = make_dims(num_q_heads, Hkv, D, B)
    fn = lib().pa_gather_checksum_fp8 if fp8 else lib().pa_gather_checksum
    rc = fn(ctypes.byref(dims), S, _dev_ptr(k_cache, "k_cache", dt), _dev_ptr(v_cache, "v_cache", dt), nb,
            _dev_ptr(block_tables, "block_tables", torch.int32), block_tables.shape[1],
            _dev_ptr(context_lens, "context_lens", torch.int32), int(max_context_len),
            _dev_ptr(out_xor, "out_xor", torch.int32), _stream(stream))
    _check(rc, "pa_gather_checksum_fp8" if fp8 else "pa_gather_checksum")
    return out_xor


def decode_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
               max_context_len, scale, partition_tokens=0, workspace=None, out=None, stream=None):
    """pa_decode_fp8: decode attention over E4M3 caches.  Returns out [S, Hq, D] bf16."""
    S, Hq, D = q.shape
    nb, Hkv, B, D2, kc, vc, ks, vs = _fp8_args(k_cache, v_cache, k_scale, v_scale)
    if D2 != D or block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = decode_workspace(q, k_cache, max_context_len, partition_tokens)
    dims = make_dims(Hq, Hkv, D, B)
    rc = lib().pa_decode_fp8(
        ctypes.byref(dims), S, _dev_ptr(q, "q", torch.bfloat16), kc, vc, ks, vs, nb,
        _dev_ptr(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _dev_ptr(context_lens, "context_lens", torch.int32), int(max_context_len), float(scale),
        int(partition_tokens), _dev_ptr(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _dev_ptr(out, "out", torch.bfloat16),
        _stream(stream))
    _check(rc, "pa_decode_fp8")
    return out


def decode_step_fp8(q, k, v, cos_sin, k_cache, v_cache, k_scale, v_scale, block_tables,
                    context_lens, max_context_len, scale, partition_tokens=0, workspace=None,
                    out=None, stream=None, early_metadata=False):
    """pa_decode_step_fp8: the fused step over E4M3 caches (q left unchanged); early_metadata
    as for decode_step."""
    S, Hq, D = q.shape
    nb, Hkv, B, D2, kc, vc, ks, vs = _fp8_args(k_cache, v_cache, k_scale, v_scale)
    if D2 != D or tuple(k.shape) != (S, Hkv, D) or tuple(v.shape) != (S, Hkv, D):
        raise ValueError("k / v shape mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("block_tables / context_lens shape mismatch")
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = decode_workspace(q, k_cache, max_context_len, partition_tokens)
    dims = make_dims(Hq, Hkv, D, B)
    bf = torch.bfloat16
    rc = lib().pa_decode_step_fp8(
        ctypes.byref(dims), S, _dev_ptr(q, "q", bf), _dev_ptr(k, "k", bf), _dev_ptr(v, "v", bf),
        _dev_ptr(cos_sin, "cos_sin", torch.float32), cos_sin.shape[0], kc, vc, ks, vs, nb,
        _dev_ptr(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _dev_ptr(context_lens, "context_lens", torch.int32), int(max_context_len), float(scale),
        int(partition_tokens), _dev_ptr(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _dev_ptr(out, "out", bf),
        PA_STEP_EARLY_METADATA if early_metadata else 0, _stream(stream))
    _check(rc, "pa_decode_step_fp8")
    return out


def _pool_ptr(t: torch.Tensor, name: str):
    """A block pool: a contiguous bf16 tensor on the GPU or in page-locked host memory."""
    if t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be bfloat16, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if not t.is_cuda and not t.is_pinned():
        raise ValueError(f"{name} must be a CUDA tensor or page-locked (pin_memory) host tensor")
    return t.data_ptr()


def copy_blocks(src_caches, dst_caches, block_pairs, stream=None):
    """Whole-block copies (pa_copy_blocks): for each row (from, to) of block_pairs and each
    cache c, dst_caches[c][to] = src_caches[c][from].  Copy-on-write inside one pool (pass the
    same list twice) or swap out / in between GPU pools and page-locked host pools.

    src_caches, dst_caches: equally long lists of [num_blocks, Hkv, B, D] bf16 tensors (CUDA
    or pinned host; all sources one pool size, all destinations one pool size); block_pairs:
    [n, 2] int64 (CUDA or pinned host).
    """
    if len(src_caches) != len(dst_caches) or not src_caches:
        raise ValueError("src_caches and dst_caches must be non-empty lists of equal length")
    n_src, Hkv, B, D = src_caches[0].shape
    n_dst = dst_caches[0].shape[0]
    for t in src_caches:
        if tuple(t.shape) != (n_src, Hkv, B, D):
            raise ValueError("source pools differ in shape")
    for t in dst_caches:
        if tuple(t.shape) != (n_dst, Hkv, B, D):
            raise ValueError("destination pools differ in shape")
    if block_pairs.dtype != torch.int64 or block_pairs.dim() != 2 or block_pairs.shape[1] != 2:
        raise ValueError("block_pairs must be an [n, 2] int64 tensor")
    if not block_pairs.is_contiguous() or not (block_pairs.is_cuda or block_pairs.is_pinned()):
        raise ValueError("block_pairs must be contiguous, on the GPU or in pinned host memory")
    n = len(src_caches)
    arr = ctypes.c_void_p * n
    src = arr(*[_pool_ptr(t, "src_caches") for t in src_caches])
    dst = arr(*[_pool_ptr(t, "dst_caches") for t in dst_caches])
    dims = make_dims(Hkv, Hkv, D, B)
    rc = lib().pa_copy_blocks(ctypes.byref(dims), n, ctypes.cast(src, ctypes.c_void_p), n_src,
                              ctypes.cast(dst, ctypes.c_void_p), n_dst,
                              ctypes.c_void_p(block_pairs.data_ptr()), block_pairs.shape[0],
                              _stream(stream))
    _check(rc, "pa_copy_blocks")


def stage_copy(dst, src, stream=None):
    """One-kernel copy of a tensor's bytes (pa_stage_copy): dst and src contiguous, on the GPU
    or in pinned host memory, the same number of bytes (a multiple of 16), 16-byte aligned.
    For staging a step's packed inputs and reading its outputs around the step's calls."""
    for t, nm in ((dst, "dst"), (src, "src")):
        if not t.is_contiguous() or not (t.is_cuda or t.is_pinned()):
            raise ValueError(f"{nm} must be contiguous, on the GPU or in pinned host memory")
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise ValueError("dst and src differ in size")
    _check(lib().pa_stage_copy(ctypes.c_void_p(dst.data_ptr()), ctypes.c_void_p(src.data_ptr()),
                               nbytes, _stream(stream)), "pa_stage_copy")


def set_timing_jitter(max_ns: int, seed: int = 0):
    """Test hook (pa_set_timing_jitter): pipeline roles of the prefill kernel sleep up to max_ns
    at each step from the next launch on; 0 turns it off."""
    _check(lib().pa_set_timing_jitter(int(max_ns), int(seed) & 0xFFFFFFFF), "pa_set_timing_jitter")


def selftest_wait_timeout(limit_us: int = 1000, stream=None):
    """Launch the bounded-wait self-test (a wait that must run out); read the result with
    get_device_status(), which then reports PA_ERR_TIMEOUT with PA_FLAG_TIMEOUT set."""
    _check(lib().pa_selftest_wait_timeout(int(limit_us), _stream(stream)), "pa_selftest_wait_timeout")


def get_device_status(stream=None) -> tuple[int, int]:
    """Synchronise the stream and read+clear the device status word: (code, flags)."""
    flags = ctypes.c_uint32(0)
    rc = lib().pa_get_device_status(_stream(stream), ctypes.byref(flags))
    return rc, int(flags.value)
