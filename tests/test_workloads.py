"""Host logic of the seeded input generator (CPU only)."""

import numpy as np
import pytest

from paged_kv_cache_244_gb300 import workloads as W


def test_splitmix64_reference_values():
    # First outputs of splitmix64 seeded with 0 (Vigna's reference generator).
    z = W.SplitMix64(0).uint64(3)
    assert [int(x) for x in z] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_normal_draws_have_the_stated_moments():
    x = W.bf16_bits_to_f32(W.SplitMix64(7).normal_bf16(200000, 0.5)).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 0.5) < 0.01


def test_f32_to_bf16_rounds_to_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.0 + 2 ** -8 + 2 ** -20], np.float32)
    assert list(W.f32_to_bf16_bits(x)) == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x3F81]


@pytest.mark.parametrize("name", ["tiny", "prefix32"])
def test_workload_is_deterministic(name):
    a, b = W.make(name), W.make(name)
    for f in ("q", "k", "v", "k_cache", "v_cache", "block_tables", "slot_mapping"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f


@pytest.mark.parametrize("name", W.WORKLOADS)
def test_block_tables_and_slots_are_consistent(name):
    w = W.make(name)
    B = W.BLOCK_SIZE
    shared = w.meta["shared_prefix_blocks"]
    owned = []
    for s in range(w.num_seqs):
        ctx = int(w.context_lens[s])
        n = (ctx + B - 1) // B
        row = w.block_tables[s]
        assert (row[:n] >= 0).all() and (row[:n] < w.num_blocks).all()
        assert (row[n:] == -1).all()
        owned += list(row[shared:n])
        # the new token is the last one of the context and its slot is in the table
        assert w.positions[s] == ctx - 1
        blk, off = divmod(int(w.slot_mapping[s]), B)
        assert blk == row[(ctx - 1) // B] and off == (ctx - 1) % B
        # its slot still holds the canary (written by the store step)
        assert (w.k_cache[:, blk, :, off] == W.BF16_NAN).all()
    assert len(set(owned)) == len(owned), "a non-shared block is handed out twice"
    if shared:
        assert (w.block_tables[:, :shared] == w.block_tables[0, :shared]).all()
        assert not set(owned) & set(w.block_tables[0, :shared].tolist())


def test_named_shapes():
    assert list(W.make("tiny").context_lens) == [17, 40]
    m = W.make("mix64")
    assert m.num_seqs == 64 and m.context_lens.min() >= 64 and m.context_lens.max() <= 4096
    assert list(W.make("long4").context_lens) == [8192, 8192, 32768, 32768]
    assert W.make("long4").partition_tokens == 512
    q = W.make("qwen_b1")
    assert q.num_layers == 28 and q.k_cache.shape == (28, 128, 2, 16, 128)
    p = W.make("prefix32")
    assert p.unique_kv_bytes_per_layer() < p.kv_bytes_per_layer() // 10


def test_shards_cover_every_sequence_once():
    w = W.make("tiny")
    parts = [W.shard(w, r, 2) for r in range(2)]
    assert sum(p.num_seqs for p in parts) == w.num_seqs
    assert np.array_equal(np.concatenate([p.context_lens for p in parts]), w.context_lens)
