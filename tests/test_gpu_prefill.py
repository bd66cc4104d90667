"""Paged (chunked) prefill attention (pa_prefill) through the C ABI, against the fp64 oracle.

Output bar as for decode: |gpu - oracle| <= 1e-2 + 1e-2 |oracle|, element by element.

- Small cases (full prefill, chunked prefill, one-token chunks, every GQA group size) are
  compared in full.
- The two full-size workloads are compared on sampled query tokens. Query i of sequence s
  alone is the oracle prefill of one token at position p with context p + 1 through the same
  block table (the causal definition makes that its whole input).
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_out_close, dev, dev_bf16, host_bits
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


def run_prefill(pa, w, out=None, context_lens=None, q_start=None):
    ctx = w.context_lens if context_lens is None else context_lens
    qs = w.q_start if q_start is None else q_start
    got = pa.prefill(dev_bf16(w.q), dev(qs), dev_bf16(w.k_cache), dev_bf16(w.v_cache),
                     dev(w.block_tables), dev(ctx), w.max_query_len, w.max_context_len, w.scale,
                     out=out)
    torch.cuda.synchronize()
    return host_bits(got)


@pytest.mark.parametrize("hq,hkv", [(12, 2), (8, 8), (16, 2), (6, 2), (4, 1), (14, 2), (10, 2), (32, 4)])
def test_prefill_small_matches_oracle(pa, orc, hq, hkv):
    """Full prefills, chunks continuing earlier tokens, one-token chunks, a chunk ending on a
    block boundary, a 16-token tile boundary and a ragged tail."""
    ctx = [1, 15, 16, 17, 100, 300, 64, 513]
    ql = [1, 15, 10, 17, 37, 64, 1, 130]
    w = W.build_prefill("pf_small", ctx, ql, 120, 101, num_q_heads=hq, num_kv_heads=hkv)
    ref, _ = orc.prefill(w.q, w.q_start, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale)
    assert np.isfinite(ref).all()
    assert_out_close(run_prefill(pa, w), ref, f"{hq}/{hkv}")
    check_status_clean(pa)


def test_prefill_one_token_per_sequence_matches_decode_oracle(pa, orc):
    w = W.build_prefill("pf_one", [1, 17, 40, 333, 2048], [1] * 5, 200, 102)
    ref_pf, _ = orc.prefill(w.q, w.q_start, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale)
    ref_dec, _ = orc.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale)
    assert np.array_equal(ref_pf, ref_dec)
    assert_out_close(run_prefill(pa, w), ref_dec)
    check_status_clean(pa)


def sampled_reference(orc, w, samples):
    """Oracle rows for the sampled (sequence, query) pairs, one one-token prefill each."""
    S = len(samples)
    q = np.stack([w.q[w.q_start[s] + i] for s, i in samples])
    pos = np.array([w.context_lens[s] - (w.q_start[s + 1] - w.q_start[s]) + i for s, i in samples], np.int32)
    bt = np.stack([w.block_tables[s] for s, _ in samples])
    ref, _ = orc.prefill(q, np.arange(S + 1, dtype=np.int32), w.k_cache, w.v_cache, bt, pos + 1, w.scale)
    return ref


@pytest.mark.parametrize("name", W.PREFILL_WORKLOADS)
def test_prefill_full_size_sampled(pa, orc, name):
    w = W.make_prefill(name)
    got = run_prefill(pa, w)
    rng = np.random.default_rng(103)
    samples = []
    for s in range(w.num_seqs):
        n = int(w.q_start[s + 1] - w.q_start[s])
        picks = set(rng.integers(0, n, 6).tolist()) | {0, n - 1, min(15, n - 1), min(16, n - 1)}
        samples += [(s, int(i)) for i in sorted(picks)]
    ref = sampled_reference(orc, w, samples)
    rows = np.array([w.q_start[s] + i for s, i in samples])
    assert_out_close(got[rows], ref, name)
    assert np.isfinite(W.bf16_bits_to_f32(got)).all()
    check_status_clean(pa)


@pytest.mark.parametrize("name", W.PREFILL_WORKLOADS)
def test_prefill_full_size_every_row(pa, orc, name):
    """Both full-size prefill workloads, every query row of every head against the oracle's
    whole prefill: the last-wave tiles (the cheapest, scheduled last) included."""
    w = W.make_prefill(name)
    got = run_prefill(pa, w)
    ref, _ = orc.prefill(w.q, w.q_start, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale)
    assert_out_close(got, ref, name)
    check_status_clean(pa)


def test_prefill_bad_sequences_are_flagged_and_skipped(pa, orc):
    w = W.build_prefill("pf_bad", [40, 50, 30], [40, 20, 30], 32, 104)
    ctx = w.context_lens.copy()
    ctx[1] = 10                                   # fewer cached tokens than new ones
    out = torch.full((w.num_tokens, w.q.shape[1], w.q.shape[2]), 7.0, dtype=torch.bfloat16, device="cuda")
    got = run_prefill(pa, w, out=out, context_lens=ctx)
    rc, flags = pa.get_device_status()
    assert rc == pa.PA_ERR_DEVICE_OOB and flags == pa.PA_FLAG_CONTEXT_LEN_OOB
    ref, _ = orc.prefill(w.q, w.q_start, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale)
    s1 = slice(int(w.q_start[1]), int(w.q_start[2]))
    assert (W.bf16_bits_to_f32(got[s1]) == 7.0).all()          # untouched
    for s in (0, 2):
        rows = slice(int(w.q_start[s]), int(w.q_start[s + 1]))
        assert_out_close(got[rows], ref[rows])
    check_status_clean(pa)


def test_prefill_out_of_range_block_is_flagged(pa, orc):
    w = W.build_prefill("pf_blk", [40, 50], [40, 50], 16, 105)
    bt = w.block_tables.copy()
    bt[1, 2] = w.num_blocks + 3
    got = pa.prefill(dev_bf16(w.q), dev(w.q_start), dev_bf16(w.k_cache), dev_bf16(w.v_cache),
                     dev(bt), dev(w.context_lens), w.max_query_len, w.max_context_len, w.scale)
    rc, flags = pa.get_device_status()
    assert flags == pa.PA_FLAG_BLOCK_ID_OOB
    ref, _ = orc.prefill(w.q, w.q_start, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale)
    rows = slice(0, int(w.q_start[1]))                          # sequence 0 is untouched by it
    assert_out_close(host_bits(got)[rows], ref[rows])
    check_status_clean(pa)


def test_prefill_first_block_out_of_range(pa, orc):
    """Sequence 1's first block id is out of range: that block is skipped.  Its queries 0-15 see
    keys of block 0 only, so every key of theirs is skipped and they store zeros (the tile's
    first P V never runs for them).  Query i >= 16 attends over keys 16..i alone, which is the
    oracle's decode of that query over the block table shifted by one block (attention depends
    on the set of keys, and RoPE is already in K)."""
    w = W.build_prefill("pf_blk0", [40, 50], [40, 50], 16, 106)
    bt = w.block_tables.copy()
    bt[1, 0] = -1
    got = host_bits(pa.prefill(dev_bf16(w.q), dev(w.q_start), dev_bf16(w.k_cache), dev_bf16(w.v_cache),
                               dev(bt), dev(w.context_lens), w.max_query_len, w.max_context_len, w.scale))
    rc, flags = pa.get_device_status()
    assert flags == pa.PA_FLAG_BLOCK_ID_OOB
    q1 = int(w.q_start[1])
    assert (W.bf16_bits_to_f32(got[q1:q1 + 16]) == 0.0).all()
    rows = np.arange(16, int(w.context_lens[1]))
    shifted = np.tile(w.block_tables[1, 1:], (len(rows), 1))
    ref, _ = orc.decode(w.q[q1 + rows], w.k_cache, w.v_cache, shifted, (rows - 15).astype(np.int32), w.scale)
    assert_out_close(got[q1 + rows], ref, "shifted")
    ref_all, _ = orc.prefill(w.q, w.q_start, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale)
    assert_out_close(got[:q1], ref_all[:q1], "untouched sequence")
    check_status_clean(pa)


@pytest.mark.parametrize("hq,hkv,ctx,ql", [(2, 2, [4100, 1200], [300, 130]), (12, 2, [9000, 777], [150, 40])])
def test_prefill_long_contexts_every_row(pa, orc, hq, hkv, ctx, ql):
    """Chunks late in long contexts (many 64-key stages, block ids read window after window) and
    G = 1 (128 queries per tile, every row its own query): every row against the oracle."""
    nb = sum((c + 15) // 16 for c in ctx) + 9
    w = W.build_prefill("pf_long", ctx, ql, nb, 107, num_q_heads=hq, num_kv_heads=hkv)
    ref, _ = orc.prefill(w.q, w.q_start, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale)
    assert_out_close(run_prefill(pa, w), ref, f"{hq}/{hkv}")
    check_status_clean(pa)


@pytest.mark.parametrize("name,seed,max_ns", [("chunked16", 11, 3000), ("prefill4x2048", 12, 3000),
                                              ("pf_long", 13, 8000), ("pf_long", 14, 500)])
def test_prefill_under_timing_jitter_gives_the_same_bits(pa, name, seed, max_ns):
    """Race check: with pseudo-random sleeps at every pipeline step of every role (TMA warps,
    MMA warp, softmax warps), the barriers see orders of arrival that undisturbed runs rarely
    take; the output must be bit-identical (the arithmetic does not depend on timing) and no
    wait may time out.  A wait that a late look can find two phases on fails here."""
    if name == "pf_long":
        ctx, ql = [9000, 777, 4100], [150, 40, 300]
        w = W.build_prefill("pf_long", ctx, ql, sum((c + 15) // 16 for c in ctx) + 9, 109)
    else:
        w = W.make_prefill(name)
    want = run_prefill(pa, w)
    check_status_clean(pa)
    pa.set_timing_jitter(max_ns, seed)
    try:
        got = run_prefill(pa, w)
    finally:
        pa.set_timing_jitter(0)
    check_status_clean(pa)
    assert np.array_equal(got, want)
