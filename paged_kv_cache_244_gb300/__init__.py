"""Paged GQA decode attention and fused RoPE + KV-cache store for GB300 (sm_103a).

The computation is in hand-written CUDA kernels behind the C ABI of include/pa.h
(libpa_gb300.so, built by ``_build.build()``).  ``binding`` is the thin ctypes front end
over PyTorch tensors; ``workloads`` makes seeded synthetic inputs.
"""

__all__ = ["binding", "workloads"]
