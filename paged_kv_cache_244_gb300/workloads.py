"""Seeded synthetic inputs for paged decode attention: caches, block tables, new tokens.

This module makes inputs only.  It holds none of the attention or RoPE arithmetic: it draws
random bf16 values, lays out block tables the way a block allocator would hand out blocks,
and builds the fp32 cos/sin table a model would precompute.  Both the CUDA path and the
oracle consume what it returns.

Random numbers: splitmix64 (Steele, Lea, Flood 2014; constants from Vigna's public
reference) drives everything.  Normal draws use Box-Muller in float64, then round to bf16
(round-to-nearest-even on the fp32 bit pattern).  Everything is a pure function of the seed.

Shapes follow Qwen2.5-1.5B attention: 12 query heads, 2 KV heads (GQA group of 6),
head_dim 128, 16-token cache blocks, RoPE theta 1e6.

Workloads (seed = 0x244 + index):
  tiny      2 seqs, context_lens {17, 40}, pool of 16 blocks, N(0, 0.5^2)
  qwen_b1   1 seq, context 2048, 28 layers each with its own 128-block cache
  mix64     64 seqs, context_lens uniform in [64, 4096], pool of 20000 scattered blocks
  prefix32  32 seqs sharing a 2000-token prefix (125 shared block ids) + 64-token suffixes
  long4     4 seqs, context_lens {8192, 8192, 32768, 32768}, 512-token partitions

Every context length counts the new token.  The new token of each sequence sits at
position context_len - 1; its slot in the cache is left holding the canary value and is
written by the RoPE + KV-store step.  Cache slots no sequence owns, and slots past the end
of a sequence, hold a bf16 NaN canary so that a kernel that reads them shows it.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

NUM_Q_HEADS = 12
NUM_KV_HEADS = 2
HEAD_DIM = 128
BLOCK_SIZE = 16
ROPE_THETA = 1.0e6
BF16_NAN = 0x7FC0

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


class SplitMix64:
    """Counter-based splitmix64 stream: output i is mix(seed + (i + 1) * golden)."""

    def __init__(self, seed: int):
        self.seed = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
        self.count = 0

    def uint64(self, n: int) -> np.ndarray:
        with np.errstate(over="ignore"):
            i = np.arange(self.count + 1, self.count + n + 1, dtype=np.uint64)
            z = self.seed + i * _GOLDEN
            z = (z ^ (z >> np.uint64(30))) * _M1
            z = (z ^ (z >> np.uint64(27))) * _M2
            z = z ^ (z >> np.uint64(31))
        self.count += n
        return z

    def uniform01(self, n: int) -> np.ndarray:
        """n doubles in [0, 1) from the top 53 bits."""
        return (self.uint64(n) >> np.uint64(11)).astype(np.float64) * (1.0 / (1 << 53))

    def integers(self, n: int, lo: int, hi: int) -> np.ndarray:
        """n integers uniform in [lo, hi] (inclusive; modulo bias below 2^-40)."""
        span = np.uint64(hi - lo + 1)
        return (self.uint64(n) % span).astype(np.int64) + lo

    def permutation(self, n: int) -> np.ndarray:
        """A permutation of 0..n-1 (argsort of n random 64-bit keys)."""
        return np.argsort(self.uint64(n), kind="stable").astype(np.int64)

    def normal_bf16(self, n: int, sigma: float) -> np.ndarray:
        """n draws of N(0, sigma^2) rounded to bf16, as uint16 bit patterns."""
        out = np.empty(n, np.uint16)
        pos = 0
        while pos < n:
            m = min(_CHUNK, n - pos)
            pairs = (m + 1) // 2
            u1 = 1.0 - self.uniform01(pairs)          # (0, 1]
            u2 = self.uniform01(pairs)
            r = np.sqrt(-2.0 * np.log(u1)) * sigma
            a = 2.0 * np.pi * u2
            z = np.empty(2 * pairs, np.float64)
            z[0::2] = r * np.cos(a)
            z[1::2] = r * np.sin(a)
            out[pos:pos + m] = f32_to_bf16_bits(z[:m].astype(np.float32))
            pos += m
        return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (inputs here are finite)."""
    b = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def rope_cos_sin_table(max_pos: int, head_dim: int = HEAD_DIM, theta: float = ROPE_THETA):
    """The model's precomputed RoPE table: fp32 [max_pos, head_dim] = [cos | sin] halves.

    Row p, column i < head_dim/2 holds cos(p * theta^(-2i/head_dim)); column head_dim/2 + i
    holds the sine.  Angles and trig are evaluated in float64 and rounded once to fp32, so
    large positions keep full fp32 accuracy.  The kernels take this table as input.
    """
    half = head_dim // 2
    inv_freq = theta ** (-(2.0 * np.arange(half, dtype=np.float64)) / head_dim)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    tab = np.empty((max_pos, head_dim), np.float32)
    tab[:, :half] = np.cos(ang).astype(np.float32)
    tab[:, half:] = np.sin(ang).astype(np.float32)
    return tab


@dataclass
class Workload:
    """One decode step's inputs for `num_layers` layers (host arrays, bf16 as uint16 bits)."""

    name: str
    num_layers: int
    context_lens: np.ndarray            # int32 [S], includes the new token
    block_tables: np.ndarray            # int32 [S, max_blocks]; unused entries -1
    num_blocks: int                     # physical blocks per layer cache
    q: np.ndarray                       # uint16 [L, S, Hq, D]  new token, before RoPE
    k: np.ndarray                       # uint16 [L, S, Hkv, D]
    v: np.ndarray                       # uint16 [L, S, Hkv, D]
    positions: np.ndarray               # int32 [S] = context_lens - 1
    slot_mapping: np.ndarray            # int64 [S] new token's slot
    cos_sin: np.ndarray                 # fp32 [max_pos, D]
    k_cache: np.ndarray                 # uint16 [L, num_blocks, Hkv, B, D]
    v_cache: np.ndarray                 # uint16 [L, num_blocks, Hkv, B, D]
    partition_tokens: int = 0           # 0: let the library choose
    sigma: float = 1.0
    seed: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def num_q_heads(self) -> int:
        return int(self.q.shape[2])

    @property
    def num_kv_heads(self) -> int:
        return int(self.k_cache.shape[2])

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(HEAD_DIM))

    def kv_bytes_per_layer(self) -> int:
        """K and V bytes one decode pass reads per layer: sum(ctx) * Hkv * D * 2 B * 2."""
        return int(self.context_lens.astype(np.int64).sum()) * self.num_kv_heads * HEAD_DIM * 2 * 2

    def unique_kv_bytes_per_layer(self) -> int:
        """Bytes of distinct (physical block, token) slots read, for shared-prefix tables."""
        seen = set()
        total = 0
        for s in range(self.num_seqs):
            ctx = int(self.context_lens[s])
            for j in range((ctx + BLOCK_SIZE - 1) // BLOCK_SIZE):
                blk = int(self.block_tables[s, j])
                n = min(BLOCK_SIZE, ctx - j * BLOCK_SIZE)
                if blk in seen:
                    continue
                seen.add(blk)
                total += n
        return total * self.num_kv_heads * HEAD_DIM * 2 * 2


def _slots_for(block_tables, positions):
    blk = block_tables[np.arange(positions.shape[0]), positions // BLOCK_SIZE].astype(np.int64)
    return blk * BLOCK_SIZE + (positions % BLOCK_SIZE)


def build(name: str, context_lens, num_blocks: int, seed: int, *, sigma: float = 1.0,
          num_layers: int = 1, shared_prefix_blocks: int = 0, partition_tokens: int = 0,
          max_blocks: int | None = None, canary: int = BF16_NAN,
          num_q_heads: int = NUM_Q_HEADS, num_kv_heads: int = NUM_KV_HEADS) -> Workload:
    """General builder.

    Block allocation: one seeded shuffle of the pool's ids; the first `shared_prefix_blocks`
    ids become a prefix every sequence maps at logical blocks 0.. (shared physical blocks,
    as prefix caching hands them out), then each sequence takes its remaining blocks from
    the shuffled list in order.  One block table serves all layers; each layer has its
    own cache tensor.
    """
    ctx = np.asarray(context_lens, np.int32)
    S = ctx.shape[0]
    rng = SplitMix64(seed)
    nblk = (ctx.astype(np.int64) + BLOCK_SIZE - 1) // BLOCK_SIZE
    mb = int(nblk.max()) if S else 1
    if max_blocks is None:
        max_blocks = max(mb, 1)
    assert max_blocks >= mb
    if shared_prefix_blocks:
        assert (nblk > shared_prefix_blocks).all(), "suffix must own the new token's block"
    need = shared_prefix_blocks + int((nblk - shared_prefix_blocks).sum())
    assert need <= num_blocks, f"pool too small: need {need} blocks, have {num_blocks}"
    pool = rng.permutation(num_blocks)
    bt = np.full((S, max_blocks), -1, np.int32)
    cursor = shared_prefix_blocks
    for s in range(S):
        bt[s, :shared_prefix_blocks] = pool[:shared_prefix_blocks]
        own = int(nblk[s]) - shared_prefix_blocks
        bt[s, shared_prefix_blocks:shared_prefix_blocks + own] = pool[cursor:cursor + own]
        cursor += own

    positions = (ctx - 1).astype(np.int32)
    slots = _slots_for(bt, positions.astype(np.int64)) if S else np.zeros(0, np.int64)
    max_pos = max(int(ctx.max()) if S else 1, 1)
    cos_sin = rope_cos_sin_table(max_pos)

    L = num_layers
    Hq, Hkv = num_q_heads, num_kv_heads
    shape_cache = (L, num_blocks, Hkv, BLOCK_SIZE, HEAD_DIM)
    k_cache = np.full(shape_cache, canary, np.uint16)
    v_cache = np.full(shape_cache, canary, np.uint16)
    tile = Hkv * BLOCK_SIZE * HEAD_DIM
    for layer in range(L):
        for cache in (k_cache, v_cache):
            if shared_prefix_blocks:
                ids = pool[:shared_prefix_blocks]
                cache[layer, ids] = rng.normal_bf16(ids.shape[0] * tile, sigma).reshape(
                    ids.shape[0], Hkv, BLOCK_SIZE, HEAD_DIM)
            for s in range(S):
                ids = bt[s, shared_prefix_blocks:nblk[s]].astype(np.int64)
                if ids.shape[0] == 0:
                    continue
                cache[layer, ids] = rng.normal_bf16(ids.shape[0] * tile, sigma).reshape(
                    ids.shape[0], Hkv, BLOCK_SIZE, HEAD_DIM)
                # The new token's slot and everything after it in the last block are not
                # past tokens: they keep the canary.
                last = int(bt[s, nblk[s] - 1])
                first_free = int(positions[s]) % BLOCK_SIZE
                cache[layer, last, :, first_free:, :] = canary
    q = rng.normal_bf16(L * S * Hq * HEAD_DIM, sigma).reshape(L, S, Hq, HEAD_DIM)
    k = rng.normal_bf16(L * S * Hkv * HEAD_DIM, sigma).reshape(L, S, Hkv, HEAD_DIM)
    v = rng.normal_bf16(L * S * Hkv * HEAD_DIM, sigma).reshape(L, S, Hkv, HEAD_DIM)
    return Workload(name=name, num_layers=L, context_lens=ctx, block_tables=bt,
                    num_blocks=num_blocks, q=q, k=k, v=v, positions=positions,
                    slot_mapping=slots.astype(np.int64), cos_sin=cos_sin, k_cache=k_cache,
                    v_cache=v_cache, partition_tokens=partition_tokens, sigma=sigma, seed=seed,
                    meta={"shared_prefix_blocks": shared_prefix_blocks})


WORKLOADS = ("tiny", "qwen_b1", "mix64", "prefix32", "long4")


def make(name: str, seed: int | None = None) -> Workload:
    """One of the five named workloads (module docstring), seeded 0x244 + its index."""
    idx = WORKLOADS.index(name)
    if seed is None:
        seed = 0x244 + idx
    if name == "tiny":
        return build(name, [17, 40], 16, seed, sigma=0.5)
    if name == "qwen_b1":
        return build(name, [2048], 128, seed, num_layers=28)
    if name == "mix64":
        ctx = SplitMix64(seed ^ 0xC0FFEE).integers(64, 64, 4096).astype(np.int32)
        return build(name, ctx, 20000, seed)
    if name == "prefix32":
        return build(name, [2064] * 32, 512, seed, shared_prefix_blocks=125)
    if name == "long4":
        return build(name, [8192, 8192, 32768, 32768], 5120, seed, partition_tokens=512)
    raise KeyError(name)


@dataclass
class PrefillWorkload:
    """One layer's inputs of a paged (chunked) prefill: sequence s brings q_lens[s] new tokens
    at the end of its context_lens[s] cached tokens, all of which are in the cache."""

    name: str
    context_lens: np.ndarray            # int32 [S], cached tokens including the new ones
    q_start: np.ndarray                 # int32 [S + 1], rows of q per sequence
    block_tables: np.ndarray            # int32 [S, max_blocks]; unused entries -1
    num_blocks: int
    q: np.ndarray                       # uint16 [T, Hq, D], already rotated
    k_cache: np.ndarray                 # uint16 [num_blocks, Hkv, B, D]
    v_cache: np.ndarray
    seed: int = 0

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.q_start[-1])

    @property
    def q_lens(self) -> np.ndarray:
        return np.diff(self.q_start).astype(np.int32)

    @property
    def max_query_len(self) -> int:
        return int(self.q_lens.max()) if self.num_seqs else 0

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(HEAD_DIM))

    def attention_flops(self) -> int:
        """Multiply-adds x 2 of q.K and p.V over the causal pairs: query i of s sees
        context_lens[s] - n_s + i + 1 keys; 4 * Hq * D flops per (query, key) pair."""
        total = 0
        Hq = int(self.q.shape[1])
        for ctx, n in zip(self.context_lens.astype(np.int64), self.q_lens.astype(np.int64)):
            first = ctx - n + 1                          # keys seen by the first new query
            total += n * first + n * (n - 1) // 2
        return int(total) * 4 * Hq * HEAD_DIM


def build_prefill(name: str, context_lens, q_lens, num_blocks: int, seed: int, *,
                  sigma: float = 1.0, num_q_heads: int = NUM_Q_HEADS,
                  num_kv_heads: int = NUM_KV_HEADS, canary: int = BF16_NAN) -> PrefillWorkload:
    """Seeded prefill inputs: blocks from one shuffle of the pool, every cached token N(0, sigma)
    in bf16, every other slot the canary, q N(0, sigma) for the new tokens."""
    rng = SplitMix64(seed)
    ctx = np.asarray(context_lens, np.int32)
    ql = np.asarray(q_lens, np.int32)
    assert ctx.shape == ql.shape and (ql <= ctx).all() and (ql >= 0).all()
    S = ctx.shape[0]
    nblk = (ctx.astype(np.int64) + BLOCK_SIZE - 1) // BLOCK_SIZE
    maxb = max(int(nblk.max()) if S else 1, 1)
    assert int(nblk.sum()) <= num_blocks, "pool too small"
    pool = rng.permutation(num_blocks)
    bt = np.full((S, maxb), -1, np.int32)
    cur = 0
    for s_ in range(S):
        bt[s_, :nblk[s_]] = pool[cur:cur + nblk[s_]]
        cur += int(nblk[s_])
    shape = (num_blocks, num_kv_heads, BLOCK_SIZE, HEAD_DIM)
    kc = np.full(shape, canary, np.uint16)
    vc = np.full(shape, canary, np.uint16)
    tile = num_kv_heads * BLOCK_SIZE * HEAD_DIM
    for cache in (kc, vc):
        for s_ in range(S):
            ids = bt[s_, :nblk[s_]].astype(np.int64)
            if ids.shape[0] == 0:
                continue
            cache[ids] = rng.normal_bf16(ids.shape[0] * tile, sigma).reshape(ids.shape[0], num_kv_heads,
                                                                             BLOCK_SIZE, HEAD_DIM)
            tail = int(ctx[s_]) - (int(nblk[s_]) - 1) * BLOCK_SIZE   # valid slots in the last block
            cache[int(bt[s_, nblk[s_] - 1]), :, tail:, :] = canary
    qs = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    T = int(qs[-1])
    q = rng.normal_bf16(T * num_q_heads * HEAD_DIM, sigma).reshape(T, num_q_heads, HEAD_DIM)
    return PrefillWorkload(name=name, context_lens=ctx, q_start=qs, block_tables=bt,
                           num_blocks=num_blocks, q=q, k_cache=kc, v_cache=vc, seed=seed)


PREFILL_WORKLOADS = ("prefill4x2048", "chunked16")


def make_prefill(name: str, seed: int | None = None) -> PrefillWorkload:
    """Named prefill workloads: prefill4x2048 = 4 prompts of 2048 tokens prefilled whole;
    chunked16 = 16 sequences each adding a 256-token chunk to 1792 prefilled tokens."""
    idx = PREFILL_WORKLOADS.index(name)
    if seed is None:
        seed = 0x2440 + idx
    if name == "prefill4x2048":
        return build_prefill(name, [2048] * 4, [2048] * 4, 4 * 128 + 64, seed)
    if name == "chunked16":
        return build_prefill(name, [2048] * 16, [256] * 16, 16 * 128 + 64, seed)
    raise KeyError(name)


def shard(w: Workload, rank: int, world: int) -> Workload:
    """Rank `rank`'s share of a workload's sequences (contiguous split; caches shared)."""
    S = w.num_seqs
    lo = (S * rank) // world
    hi = (S * (rank + 1)) // world
    sl = slice(lo, hi)
    return Workload(name=w.name, num_layers=w.num_layers, context_lens=w.context_lens[sl].copy(),
                    block_tables=w.block_tables[sl].copy(), num_blocks=w.num_blocks,
                    q=w.q[:, sl].copy(), k=w.k[:, sl].copy(), v=w.v[:, sl].copy(),
                    positions=w.positions[sl].copy(), slot_mapping=w.slot_mapping[sl].copy(),
                    cos_sin=w.cos_sin, k_cache=w.k_cache, v_cache=w.v_cache,
                    partition_tokens=w.partition_tokens, sigma=w.sigma, seed=w.seed,
                    meta=dict(w.meta, shard=(rank, world)))
