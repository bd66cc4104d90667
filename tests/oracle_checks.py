"""Pins for the fp64 oracle: checks against what the pages and the mathematics fix.

Each check takes an ``oracle.Oracle`` and raises AssertionError when the oracle disagrees
with something other than itself: closed forms, invariants, brute force over every bf16
value, dense attention through a library softmax, textbook trig values.  The same checks run
against deliberately broken copies of the oracle (tests/test_oracle_mutants.py) to show that
a plausible mistake anywhere in it fails at least one of them.

Passages pinned (page title, section):
  * "从零实现 LLM 推理引擎：深挖 vLLM 的六大核心优化", §3.1 Paged KV Cache: 16-token blocks,
    block_table maps logical to physical blocks.  -> dense equivalence, permutation
    invariance, canary slots ignored.
  * "Pico-vLLM：从零手写的工业级LLM推理引擎实现", §1 模型实现层: RoPE (rotate_half), GQA.
    -> unit-vector rotations, norm, relative position; KV-head mapping.
  * same page, §2 Kernel层: decode kernel computes softmax attention of one new token;
    fused RoPE + KV cache store.  -> closed forms, slot placement.
  * same page, §H200上的详细对比: Flash Decode.  -> partitioned merge equals unsplit.
"""

from __future__ import annotations

import math

import numpy as np
from scipy.special import softmax

from paged_kv_cache_244_gb300 import workloads as W

D = W.HEAD_DIM
HALF = D // 2
B = W.BLOCK_SIZE
THETA = W.ROPE_THETA


# ----------------------------------------------------------------------------- bf16 ----

def _bf16_of(x: float) -> int:
    """Brute-force bf16 RNE: nearest of all non-negative bf16 values (inf as 2^128)."""
    bits = np.arange(0, 0x7F81, dtype=np.uint32)
    vals = (bits << np.uint32(16)).view(np.float32).astype(np.float64)
    vals[-1] = 2.0 ** 128
    a = abs(x)
    i = int(np.searchsorted(vals, a))
    if i == vals.shape[0]:
        b = 0x7F80
    elif vals[i] == a:
        b = i
    else:
        lo, hi = i - 1, i
        dlo, dhi = a - vals[lo], vals[hi] - a
        b = lo if dlo < dhi else hi if dhi < dlo else (lo if lo % 2 == 0 else hi)
    return b | (0x8000 if math.copysign(1.0, x) < 0 else 0)


def check_bf16_widen(orc):
    bits = np.arange(0x10000, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        ref = (bits << np.uint32(16)).view(np.float32).astype(np.float64)
    for b in list(range(0, 0x10000, 97)) + [0x0000, 0x8000, 0x0001, 0x7F7F, 0xFF7F, 0x3F80]:
        got = orc.bf16_to_f64(b)
        assert got == ref[b] or (math.isnan(got) and math.isnan(ref[b])), (hex(b), got, ref[b])


def check_bf16_narrow_bruteforce(orc):
    rng = W.SplitMix64(11)
    xs = []
    # random magnitudes across the whole exponent range, both signs
    e = rng.integers(400, -140, 130)
    m = rng.uniform01(400) + 0.5
    sgn = np.where(rng.integers(400, 0, 1) == 1, -1.0, 1.0)
    xs += list(sgn * np.ldexp(m, e))
    # exact midpoints between consecutive bf16 values (ties) and their neighbours
    for b in [0x3F80, 0x3F81, 0x4000, 0x0001, 0x0002, 0x007F, 0x0080, 0x7F7E, 0x7F7F, 0x4480]:
        lo = orc_free_value(b)
        hi = orc_free_value(b + 1)
        mid = (lo + hi) / 2.0
        xs += [mid, -mid, math.nextafter(mid, 0.0), math.nextafter(mid, math.inf)]
    xs += [0.0, -0.0, 1.0, -1.0, 2.0 ** -134, 2.0 ** -135, 3.0 * 2.0 ** -135, 3.4e38, 3.5e38]
    for x in xs:
        got = orc.f64_to_bf16(float(x))
        want = _bf16_of(float(x))
        assert got == want, (x, hex(got), hex(want))
    assert orc.f64_to_bf16(math.inf) == 0x7F80
    assert orc.f64_to_bf16(-math.inf) == 0xFF80
    assert (orc.f64_to_bf16(math.nan) & 0x7FFF) > 0x7F80


def orc_free_value(b: int) -> float:
    """Value of a bf16 bit pattern, computed by numpy (no oracle involved)."""
    return float(np.array([b << 16], np.uint32).view(np.float32)[0])


# ----------------------------------------------------------------------------- RoPE ----

def _unit(i):
    x = np.zeros(D, np.float64)
    x[i] = 1.0
    return W.f32_to_bf16_bits(x.astype(np.float32))


def check_rope_identity_at_pos0(orc):
    tab = W.rope_cos_sin_table(4)
    x = W.SplitMix64(3).normal_bf16(D, 1.0)
    y = orc.rope_rotate_f64(x, tab[0])
    assert np.array_equal(y, W.bf16_bits_to_f32(x).astype(np.float64))


def check_rope_unit_vectors(orc):
    """e_i at position p rotates to (cos, sin)(p * w_i) at (i, i + D/2): rotate_half pairing.

    Closed forms of the frequency theta^(-2i/D) at theta = 1e6, D = 128:
    w_0 = 1, w_16 = 10^-1.5, w_32 = 10^-3, w_48 = 10^-4.5.
    """
    tab = W.rope_cos_sin_table(40000)
    w = {0: 1.0, 16: 10.0 ** -1.5, 32: 1.0e-3, 48: 10.0 ** -4.5}
    for p in (1, 2, 7, 2047, 32767):
        for i, wi in w.items():
            c, s = math.cos(p * wi), math.sin(p * wi)
            y = orc.rope_rotate_f64(_unit(i), tab[p])
            want = np.zeros(D)
            want[i], want[HALF + i] = c, s
            assert np.allclose(y, want, rtol=0, atol=2e-7), (p, i)
            y = orc.rope_rotate_f64(_unit(HALF + i), tab[p])
            want = np.zeros(D)
            want[i], want[HALF + i] = -s, c
            assert np.allclose(y, want, rtol=0, atol=2e-7), (p, i, "upper")


def check_rope_pair_norm(orc):
    tab = W.rope_cos_sin_table(5000)
    rng = W.SplitMix64(5)
    for p in (3, 100, 4999):
        x = rng.normal_bf16(D, 1.0)
        xf = W.bf16_bits_to_f32(x).astype(np.float64)
        y = orc.rope_rotate_f64(x, tab[p])
        n_in = xf[:HALF] ** 2 + xf[HALF:] ** 2
        n_out = y[:HALF] ** 2 + y[HALF:] ** 2
        assert np.allclose(n_out, n_in, rtol=1e-6, atol=1e-12)


def check_rope_relative_position(orc):
    """<R_m q, R_n k> depends only on m - n."""
    tab = W.rope_cos_sin_table(9000)
    rng = W.SplitMix64(6)
    q = rng.normal_bf16(D, 1.0)
    k = rng.normal_bf16(D, 1.0)
    for m, n in ((10, 3), (500, 17), (8000, 4000)):
        base = orc.rope_rotate_f64(q, tab[m]) @ orc.rope_rotate_f64(k, tab[n])
        for shift in (1, 37, 900):
            other = orc.rope_rotate_f64(q, tab[m + shift]) @ orc.rope_rotate_f64(k, tab[n + shift])
            assert abs(other - base) < 1e-4, (m, n, shift, base, other)
    # and it does depend on m - n
    a = orc.rope_rotate_f64(q, tab[10]) @ orc.rope_rotate_f64(k, tab[3])
    b = orc.rope_rotate_f64(q, tab[11]) @ orc.rope_rotate_f64(k, tab[3])
    assert abs(a - b) > 1e-3


def check_rope_kv_store_placement(orc):
    """V lands bit-exact at its slot, K lands rotated, nothing else in the caches changes."""
    rng = W.SplitMix64(8)
    T, Hq, Hkv, nb = 5, 12, 2, 6
    q = rng.normal_bf16(T * Hq * D, 1.0).reshape(T, Hq, D)
    k = rng.normal_bf16(T * Hkv * D, 1.0).reshape(T, Hkv, D)
    v = rng.normal_bf16(T * Hkv * D, 1.0).reshape(T, Hkv, D)
    positions = np.array([0, 5, 16, 95, 40], np.int32)
    slots = np.array([3, 17, 5 * 16 + 15, -1, 2 * 16], np.int64)
    tab = W.rope_cos_sin_table(96)
    kc = np.full((nb, Hkv, B, D), 0x1234, np.uint16)
    vc = np.full((nb, Hkv, B, D), 0x4321, np.uint16)
    q2 = orc.rope_kv_store(q, k, v, positions, tab, slots, kc, vc)
    touched = np.zeros((nb, B), bool)
    for t in range(T):
        for h in range(Hq):
            want = [orc.f64_to_bf16(x) for x in orc.rope_rotate_f64(q[t, h], tab[positions[t]])]
            assert np.array_equal(q2[t, h], np.array(want, np.uint16)), (t, h)
        if slots[t] < 0:
            continue
        blk, off = divmod(int(slots[t]), B)
        touched[blk, off] = True
        for h in range(Hkv):
            assert np.array_equal(vc[blk, h, off], v[t, h])
            want = [orc.f64_to_bf16(x) for x in orc.rope_rotate_f64(k[t, h], tab[positions[t]])]
            assert np.array_equal(kc[blk, h, off], np.array(want, np.uint16))
    for blk in range(nb):
        for off in range(B):
            if not touched[blk, off]:
                assert (kc[blk, :, off] == 0x1234).all() and (vc[blk, :, off] == 0x4321).all()
    # pos 0 leaves k unchanged bit for bit
    assert np.array_equal(kc[0, :, 3], k[0])


# --------------------------------------------------------------------------- decode ----

def _paged_from_dense(Kd, Vd, nb, rng, fill=W.BF16_NAN):
    """Scatter dense per-sequence K/V [S][Hkv][ctx_s][D] into a paged cache via a random
    block permutation.  Returns (k_cache, v_cache, block_tables)."""
    S = len(Kd)
    Hkv = Kd[0].shape[0]
    ctxs = [k.shape[1] for k in Kd]
    nblk = [(c + B - 1) // B for c in ctxs]
    perm = rng.permutation(nb)
    maxb = max(max(nblk), 1)
    bt = np.full((S, maxb), -1, np.int32)
    kc = np.full((nb, Hkv, B, D), fill, np.uint16)
    vc = np.full((nb, Hkv, B, D), fill, np.uint16)
    cur = 0
    for s in range(S):
        for j in range(nblk[s]):
            blk = int(perm[cur])
            cur += 1
            bt[s, j] = blk
            lo, hi = j * B, min(ctxs[s], (j + 1) * B)
            kc[blk, :, : hi - lo] = Kd[s][:, lo:hi]
            vc[blk, :, : hi - lo] = Vd[s][:, lo:hi]
    return kc, vc, bt


def _dense_attention(q, Kd, Vd, scale):
    """softmax(scale q K^T) V per query head with scipy's softmax, on contiguous K/V."""
    S, Hq, _ = q.shape
    Hkv = Kd[0].shape[0]
    G = Hq // Hkv
    out = np.zeros((S, Hq, D))
    for s in range(S):
        for h in range(Hq):
            K = W.bf16_bits_to_f32(Kd[s][h // G]).astype(np.float64)
            V = W.bf16_bits_to_f32(Vd[s][h // G]).astype(np.float64)
            if K.shape[0] == 0:
                continue
            qh = W.bf16_bits_to_f32(q[s, h]).astype(np.float64)
            p = softmax(scale * (K @ qh))
            out[s, h] = p @ V
    return out


def check_decode_dense_equivalence(orc):
    rng = W.SplitMix64(21)
    ctxs = [1, 15, 16, 17, 40, 100]
    Hq, Hkv = 12, 2
    Kd = [rng.normal_bf16(Hkv * c * D, 1.0).reshape(Hkv, c, D) for c in ctxs]
    Vd = [rng.normal_bf16(Hkv * c * D, 1.0).reshape(Hkv, c, D) for c in ctxs]
    q = rng.normal_bf16(len(ctxs) * Hq * D, 1.0).reshape(len(ctxs), Hq, D)
    kc, vc, bt = _paged_from_dense(Kd, Vd, 32, rng)
    scale = 1.0 / math.sqrt(D)
    got, gotb = orc.decode(q, kc, vc, bt, np.array(ctxs, np.int32), scale)
    want = _dense_attention(q, Kd, Vd, scale)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-13)
    assert np.isfinite(got).all()
    # the bf16 output is the nearest bf16 of the fp64 output
    flat = got.reshape(-1)
    for idx in range(0, flat.shape[0], 331):
        assert gotb.reshape(-1)[idx] == _bf16_of(float(flat[idx]))


def _tiny_after_store(orc):
    """The tiny workload after its fused RoPE + store step: (workload, rotated q, caches)."""
    w = W.make("tiny")
    kc, vc = w.k_cache[0].copy(), w.v_cache[0].copy()
    q = orc.rope_kv_store(w.q[0], w.k[0], w.v[0], w.positions, w.cos_sin, w.slot_mapping, kc, vc)
    return w, q, kc, vc


def check_decode_block_permutation_invariance(orc):
    w, q, kc, vc = _tiny_after_store(orc)
    out1, b1 = orc.decode(q, kc, vc, w.block_tables, w.context_lens, w.scale)
    assert np.isfinite(out1).all()
    pi = W.SplitMix64(99).permutation(w.num_blocks)
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[pi] = kc
    vc2[pi] = vc
    bt2 = np.where(w.block_tables >= 0, pi[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    out2, b2 = orc.decode(q, kc2, vc2, bt2, w.context_lens, w.scale)
    assert np.array_equal(out1, out2) and np.array_equal(b1, b2)


def _small_case(ctx, Kfill, Vfill, qfill, Hq=12, Hkv=2):
    """One sequence with explicit dense K/V, paged through a shuffled pool."""
    rng = W.SplitMix64(1234)
    Kd = [Kfill]
    Vd = [Vfill]
    q = qfill[None]
    kc, vc, bt = _paged_from_dense(Kd, Vd, max(4, (ctx + B - 1) // B + 2), rng)
    return q, kc, vc, bt, np.array([ctx], np.int32)


def check_decode_ctx1_returns_v(orc):
    rng = W.SplitMix64(31)
    K = rng.normal_bf16(2 * 1 * D, 3.0).reshape(2, 1, D)
    V = rng.normal_bf16(2 * 1 * D, 3.0).reshape(2, 1, D)
    q = rng.normal_bf16(12 * D, 3.0).reshape(12, D)
    args = _small_case(1, K, V, q)
    out, outb = orc.decode(*args, 1.0 / math.sqrt(D))
    for h in range(12):
        assert np.array_equal(outb[0, h], V[h // 6, 0])
        assert np.array_equal(out[0, h], W.bf16_bits_to_f32(V[h // 6, 0]).astype(np.float64))


def check_decode_identical_keys_mean(orc):
    rng = W.SplitMix64(32)
    ctx = 37
    k1 = rng.normal_bf16(2 * D, 1.0).reshape(2, 1, D)
    K = np.repeat(k1, ctx, axis=1)
    V = rng.normal_bf16(2 * ctx * D, 1.0).reshape(2, ctx, D)
    q = rng.normal_bf16(12 * D, 1.0).reshape(12, D)
    out, _ = orc.decode(*_small_case(ctx, K, V, q), 1.0 / math.sqrt(D))
    for h in range(12):
        mean = W.bf16_bits_to_f32(V[h // 6]).astype(np.float64).mean(axis=0)
        assert np.allclose(out[0, h], mean, rtol=1e-13, atol=1e-14)


def check_decode_gqa_head_mapping(orc):
    """V constant (g + 1) on KV head g: every query head h reads KV head h // (Hq / Hkv)."""
    rng = W.SplitMix64(33)
    for Hq, Hkv in ((12, 2), (8, 4), (6, 1)):
        ctx = 21
        K = rng.normal_bf16(Hkv * ctx * D, 1.0).reshape(Hkv, ctx, D)
        V = np.stack([np.full((ctx, D), W.f32_to_bf16_bits(np.float32([g + 1]))[0], np.uint16)
                      for g in range(Hkv)])
        q = rng.normal_bf16(Hq * D, 1.0).reshape(Hq, D)
        out, _ = orc.decode(*_small_case(ctx, K, V, q, Hq, Hkv), 0.1)
        G = Hq // Hkv
        for h in range(Hq):
            assert np.allclose(out[0, h], h // G + 1, rtol=1e-14), (Hq, Hkv, h)


def check_decode_two_token_logistic(orc):
    """Two keys with q.k1 - q.k2 = a: weight on v1 is the logistic sigma(scale * a)."""
    for a, scale in ((8.0, 1.0 / math.sqrt(D)), (3.0, 0.5), (-5.0, 1.0 / math.sqrt(D))):
        q = np.zeros((12, D), np.uint16)
        q[:, 0] = W.f32_to_bf16_bits(np.float32([a]))[0]
        K = np.zeros((2, 2, D), np.uint16)
        K[:, 0, 0] = W.f32_to_bf16_bits(np.float32([1.0]))[0]
        rng = W.SplitMix64(34)
        V = rng.normal_bf16(2 * 2 * D, 1.0).reshape(2, 2, D)
        out, _ = orc.decode(*_small_case(2, K, V, q), scale)
        w1 = 1.0 / (1.0 + math.exp(-scale * a))
        for h in range(12):
            Vf = W.bf16_bits_to_f32(V[h // 6]).astype(np.float64)
            assert np.allclose(out[0, h], w1 * Vf[0] + (1 - w1) * Vf[1], rtol=1e-12, atol=1e-14)


def check_decode_large_scores_stable(orc):
    """Scores near 1000 (exp would overflow without the max shift): one key dominates."""
    q = np.zeros((12, D), np.uint16)
    q[:, 0] = W.f32_to_bf16_bits(np.float32([128.0]))[0]
    ctx = 5
    K = np.zeros((2, ctx, D), np.uint16)
    for t in range(ctx):
        K[:, t, 0] = W.f32_to_bf16_bits(np.float32([100.0 - 10.0 * (t != 3)]))[0]
    V = W.SplitMix64(35).normal_bf16(2 * ctx * D, 1.0).reshape(2, ctx, D)
    out, _ = orc.decode(*_small_case(ctx, K, V, q), 1.0 / math.sqrt(D))
    assert np.isfinite(out).all()
    for h in range(12):
        assert np.allclose(out[0, h], W.bf16_bits_to_f32(V[h // 6, 3]), rtol=0, atol=1e-12)


def check_decode_ignores_canaries_and_unused_entries(orc):
    """Slots past context_len, unused blocks and table entries past the context are never read."""
    w, q, kc, vc = _tiny_after_store(orc)
    bt = w.block_tables.copy()
    bt[bt < 0] = 10 ** 6               # garbage, not just -1
    out, _ = orc.decode(q, kc, vc, bt, w.context_lens, w.scale)
    assert np.isfinite(out).all()
    # the canaries are really there: slots past the end of sequence 0's last block
    last = w.block_tables[0, (w.context_lens[0] - 1) // B]
    assert (kc[last, :, w.context_lens[0] % B:] == W.BF16_NAN).all()


def check_decode_empty_context(orc):
    w, q, kc, vc = _tiny_after_store(orc)
    ctx = w.context_lens.copy()
    ctx[0] = 0
    out, outb = orc.decode(q, kc, vc, w.block_tables, ctx, w.scale)
    assert (out[0] == 0).all() and (outb[0] == 0).all()
    assert np.isfinite(out[1]).all() and (out[1] != 0).any()


def check_store_then_decode_matches_dense(orc):
    """After the fused store, decode over context_len includes the new token at ctx - 1."""
    w, q, kc, vc = _tiny_after_store(orc)
    got, _ = orc.decode(q, kc, vc, w.block_tables, w.context_lens, w.scale)
    Kd, Vd = [], []
    for s in range(w.num_seqs):
        c = int(w.context_lens[s])
        Ks = np.empty((2, c, D), np.uint16)
        Vs = np.empty((2, c, D), np.uint16)
        for t in range(c - 1):
            blk = w.block_tables[s, t // B]
            Ks[:, t] = w.k_cache[0][blk, :, t % B]
            Vs[:, t] = w.v_cache[0][blk, :, t % B]
        for h in range(2):
            Ks[h, c - 1] = [orc.f64_to_bf16(x) for x in
                            orc.rope_rotate_f64(w.k[0, s, h], w.cos_sin[c - 1])]
            Vs[h, c - 1] = w.v[0, s, h]
        Kd.append(Ks)
        Vd.append(Vs)
    want = _dense_attention(q, Kd, Vd, w.scale)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-13)


def check_flash_decode_merge_equals_unsplit(orc):
    rng = W.SplitMix64(41)
    ctxs = [1, 16, 17, 100, 515]
    Hq, Hkv = 12, 2
    Kd = [rng.normal_bf16(Hkv * c * D, 2.0).reshape(Hkv, c, D) for c in ctxs]
    Vd = [rng.normal_bf16(Hkv * c * D, 1.0).reshape(Hkv, c, D) for c in ctxs]
    q = rng.normal_bf16(len(ctxs) * Hq * D, 1.0).reshape(len(ctxs), Hq, D)
    kc, vc, bt = _paged_from_dense(Kd, Vd, 64, rng)
    ctx = np.array(ctxs, np.int32)
    scale = 1.0 / math.sqrt(D)
    ref, _ = orc.decode(q, kc, vc, bt, ctx, scale)
    for P in (1, 5, 16, 48, 512, 4096):
        got = orc.decode_partitioned(q, kc, vc, bt, ctx, scale, P)
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-14), P


def check_copy_blocks_matches_fancy_indexing(orc):
    """Block copy between pools = numpy's own indexed assignment, bit for bit (NaN and
    signed-zero patterns included); blocks not named as destinations are untouched."""
    rng = np.random.default_rng(7)
    src = [rng.integers(0, 1 << 16, (40, 2, 16, D), dtype=np.uint16) for _ in range(5)]
    dst = [rng.integers(0, 1 << 16, (30, 2, 16, D), dtype=np.uint16) for _ in range(5)]
    want = [d.copy() for d in dst]
    frm = rng.permutation(40)[:17]
    to = rng.permutation(30)[:17]
    for c in range(5):
        want[c][to] = src[c][frm]
    assert orc.copy_blocks(src, dst, np.stack([frm, to], axis=1)) == 0
    for c in range(5):
        assert np.array_equal(dst[c], want[c])


def check_copy_blocks_skips_out_of_range_pairs(orc):
    rng = np.random.default_rng(8)
    src = [rng.integers(0, 1 << 16, (8, 1, 16, D), dtype=np.uint16) for _ in range(2)]
    dst = [np.zeros((6, 1, 16, D), np.uint16) for _ in range(2)]
    pairs = [[0, 0], [8, 1], [-1, 2], [3, 6], [4, -5], [7, 5]]
    assert orc.copy_blocks(src, dst, pairs) == 4
    for c in range(2):
        assert np.array_equal(dst[c][0], src[c][0]) and np.array_equal(dst[c][5], src[c][7])
        assert not dst[c][1:5].any()


def check_swap_out_in_preserves_decode(orc):
    """Swap every block of a batch out to a CPU pool and back in to other GPU blocks, with
    the block tables remapped: the decode output is the same to the last bit of fp64."""
    w, q, kc, vc = _tiny_after_store(orc)
    S = w.num_seqs
    used = sorted({int(b) for s in range(S)
                   for b in w.block_tables[s, :(int(w.context_lens[s]) + 15) // 16]})
    ref, _ = orc.decode(q, kc, vc, w.block_tables, w.context_lens, w.scale)
    assert np.isfinite(ref).all()
    cpu = [np.zeros((len(used),) + kc.shape[1:], np.uint16) for _ in range(2)]
    orc.copy_blocks([kc, vc], cpu, [[b, i] for i, b in enumerate(used)])           # swap out
    rng = np.random.default_rng(9)
    fresh = rng.permutation(kc.shape[0])[:len(used)]                                 # new ids
    kc2 = np.full_like(kc, W.BF16_NAN)
    vc2 = np.full_like(vc, W.BF16_NAN)
    orc.copy_blocks(cpu, [kc2, vc2], [[i, int(f)] for i, f in enumerate(fresh)])    # swap in
    remap = {b: int(f) for b, f in zip(used, fresh)}
    bt = w.block_tables.copy()
    for s in range(S):
        for j in range((int(w.context_lens[s]) + 15) // 16):
            bt[s, j] = remap[int(bt[s, j])]
    got, _ = orc.decode(q, kc2, vc2, bt, w.context_lens, w.scale)
    assert np.array_equal(got, ref)


# ---- paged (chunked) prefill -------------------------------------------------------------

def _prefill_case(seed, ctxs, Hq=12, Hkv=2, nb=64):
    rng = W.SplitMix64(seed)
    Kd = [rng.normal_bf16(Hkv * c * D, 1.5).reshape(Hkv, c, D) for c in ctxs]
    Vd = [rng.normal_bf16(Hkv * c * D, 1.0).reshape(Hkv, c, D) for c in ctxs]
    kc, vc, bt = _paged_from_dense(Kd, Vd, nb, rng)
    return rng, Kd, Vd, kc, vc, bt


def check_prefill_full_equals_dense_causal(orc):
    """Full prefill (the whole context is new) = causal dense attention (scipy softmax over
    tokens 0..i for query i) on contiguous K/V."""
    ctxs = [1, 17, 70]
    Hq, Hkv = 12, 2
    rng, Kd, Vd, kc, vc, bt = _prefill_case(51, ctxs)
    T = sum(ctxs)
    q = rng.normal_bf16(T * Hq * D, 1.0).reshape(T, Hq, D)
    qs = np.concatenate([[0], np.cumsum(ctxs)]).astype(np.int32)
    scale = 1.0 / math.sqrt(D)
    got, _ = orc.prefill(q, qs, kc, vc, bt, np.array(ctxs, np.int32), scale)
    for s, c in enumerate(ctxs):
        for i in range(c):
            for h in range(Hq):
                K = W.bf16_bits_to_f32(Kd[s][h // 6][:i + 1]).astype(np.float64)
                V = W.bf16_bits_to_f32(Vd[s][h // 6][:i + 1]).astype(np.float64)
                qh = W.bf16_bits_to_f32(q[qs[s] + i, h]).astype(np.float64)
                ref = softmax(scale * (K @ qh)) @ V
                assert np.allclose(got[qs[s] + i, h], ref, rtol=1e-12, atol=1e-14), (s, i, h)


def check_prefill_one_token_is_decode(orc):
    w, q, kc, vc = _tiny_after_store(orc)
    S = w.num_seqs
    got, _ = orc.prefill(q, np.arange(S + 1, dtype=np.int32), kc, vc, w.block_tables,
                         w.context_lens, w.scale)
    ref, _ = orc.decode(q, kc, vc, w.block_tables, w.context_lens, w.scale)
    assert np.array_equal(got, ref)


def check_prefill_chunks_compose(orc):
    """A prompt prefilled in two chunks gives, token for token, the one-chunk result."""
    ctxs = [40, 93]
    Hq = 12
    rng, Kd, Vd, kc, vc, bt = _prefill_case(52, ctxs)
    T = sum(ctxs)
    q = rng.normal_bf16(T * Hq * D, 1.0).reshape(T, Hq, D)
    qs = np.concatenate([[0], np.cumsum(ctxs)]).astype(np.int32)
    ctx = np.array(ctxs, np.int32)
    whole, _ = orc.prefill(q, qs, kc, vc, bt, ctx, 0.09)
    cut = [13, 64]                                       # first chunks
    q1 = np.concatenate([q[qs[s]:qs[s] + cut[s]] for s in range(2)])
    a, _ = orc.prefill(q1, np.array([0, cut[0], sum(cut)], np.int32), kc, vc, bt,
                       np.array(cut, np.int32), 0.09)
    q2 = np.concatenate([q[qs[s] + cut[s]:qs[s + 1]] for s in range(2)])
    n2 = [ctxs[s] - cut[s] for s in range(2)]
    b, _ = orc.prefill(q2, np.array([0, n2[0], sum(n2)], np.int32), kc, vc, bt, ctx, 0.09)
    for s in range(2):
        assert np.array_equal(whole[qs[s]:qs[s] + cut[s]], a[sum(cut[:s]):sum(cut[:s + 1])])
        assert np.array_equal(whole[qs[s] + cut[s]:qs[s + 1]], b[sum(n2[:s]):sum(n2[:s + 1])])


def check_prefill_is_causal(orc):
    """Changing the K/V of token j changes exactly the outputs of queries at positions >= j."""
    ctxs = [50]
    Hq = 12
    rng, Kd, Vd, kc, vc, bt = _prefill_case(53, ctxs)
    q = rng.normal_bf16(50 * Hq * D, 1.0).reshape(50, Hq, D)
    qs = np.array([0, 50], np.int32)
    ctx = np.array([50], np.int32)
    before, _ = orc.prefill(q, qs, kc, vc, bt, ctx, 0.09)
    j = 29
    blk, off = int(bt[0, j // 16]), j % 16
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[blk, :, off] = rng.normal_bf16(2 * D, 3.0).reshape(2, D)
    vc2[blk, :, off] = rng.normal_bf16(2 * D, 3.0).reshape(2, D)
    after, _ = orc.prefill(q, qs, kc2, vc2, bt, ctx, 0.09)
    assert np.array_equal(after[:j], before[:j])
    assert (np.abs(after[j:] - before[j:]).max(axis=(1, 2)) > 0).all()


# ---- FP8 (E4M3) KV cache ------------------------------------------------------------------
# The independent reference for the E4M3 format is PyTorch's own float8_e4m3fn conversion.

def _torch_e4m3_decode(codes):
    import torch
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _torch_e4m3_encode(x_f32):
    import torch
    t = torch.from_numpy(np.asarray(x_f32, np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def check_e4m3_decode_all_codes(orc):
    want = _torch_e4m3_decode(np.arange(256))
    for c in range(256):
        got = orc.e4m3_to_f64(c)
        if np.isnan(want[c]):
            assert np.isnan(got), c
        else:
            assert got == want[c] and np.signbit(got) == np.signbit(want[c]), (c, got, want[c])
    # the format's landmarks: max 448, smallest normal 2^-6, smallest subnormal 2^-9
    assert orc.e4m3_to_f64(0x7E) == 448.0 and orc.e4m3_to_f64(0x08) == 2.0 ** -6
    assert orc.e4m3_to_f64(0x01) == 2.0 ** -9


def check_e4m3_encode_rne_and_saturation(orc):
    codes = np.arange(0x7E + 1)
    vals = _torch_e4m3_decode(codes)
    mids = (vals[:-1] + vals[1:]) / 2               # exact ties (fp32-representable)
    rng = np.random.default_rng(21)
    rand = np.ldexp(rng.uniform(1, 2, 4000), rng.integers(-12, 9, 4000))
    xs = np.concatenate([vals, mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9), rand])
    xs = np.concatenate([xs, -xs]).astype(np.float32)
    xs = xs[np.abs(xs) <= 448]
    want = _torch_e4m3_encode(xs)
    got = np.array([orc.f64_to_e4m3(float(x)) for x in xs], np.uint8)
    assert np.array_equal(got, want)
    for big in (448.5, 464.0, 480.0, 1e6, float("inf")):
        assert orc.f64_to_e4m3(big) == 0x7E and orc.f64_to_e4m3(-big) == 0xFE
    assert orc.f64_to_e4m3(float("nan")) & 0x7F == 0x7F


def check_quantize_cache_definition(orc):
    """code = E4M3(fp32(x) * fp32(1 / scale_g)) with g the element's KV head."""
    rng = W.SplitMix64(22)
    cache = rng.normal_bf16(6 * 2 * 16 * D, 2.0).reshape(6, 2, 16, D)
    scale = np.array([4.5 / 448, 7.0 / 448], np.float32)
    got = orc.quantize_cache(cache, scale)
    x = W.bf16_bits_to_f32(cache)
    inv = (np.float32(1.0) / scale).astype(np.float32)
    y = (x * inv[None, :, None, None]).astype(np.float32)
    inside = np.abs(y) <= 448
    assert inside.mean() > 0.9 and (~inside).any()       # both regimes are exercised
    assert np.array_equal(got[inside], _torch_e4m3_encode(y[inside]))
    assert np.array_equal(got[~inside], np.where(y[~inside] > 0, 0x7E, 0xFE).astype(np.uint8))


def check_quantize_decides_in_fp32(orc):
    """The code is taken from fp32(x) * fp32(1 / scale), the kernels' precision, not from the
    exact quotient: over every bf16 value in range, with scale 7 (where the two differ for 25
    values), the oracle agrees with the fp32 product everywhere."""
    bits = np.arange(0x3C00, 0x43E0, dtype=np.uint16)          # ~0.0078 .. ~450
    pad = -bits.size % (16 * D)
    bits = np.concatenate([bits, np.zeros(pad, np.uint16)])     # whole 16 x D rows
    x = W.bf16_bits_to_f32(bits).astype(np.float32)
    for sc in (7.0, 3.0, 0.7):
        s32 = np.float32(sc)
        y32 = (x * (np.float32(1.0) / s32)).astype(np.float32)
        got = orc.quantize_cache(bits.reshape(-1, 1, 16, D), np.array([s32], np.float32)).reshape(-1)
        m = np.abs(y32) <= 448
        assert np.array_equal(got[m], _torch_e4m3_encode(y32[m])), sc


def _fp8_case(orc, seed=23):
    rng = W.SplitMix64(seed)
    ctxs = [1, 16, 17, 100, 333]
    Hq, Hkv = 12, 2
    Kd = [rng.normal_bf16(Hkv * c * D, 1.0).reshape(Hkv, c, D) for c in ctxs]
    Vd = [rng.normal_bf16(Hkv * c * D, 1.0).reshape(Hkv, c, D) for c in ctxs]
    q = rng.normal_bf16(len(ctxs) * Hq * D, 1.0).reshape(len(ctxs), Hq, D)
    kc, vc, bt = _paged_from_dense(Kd, Vd, 48, rng, fill=0)
    ks = np.array([5.0 / 448, 4.0 / 448], np.float32)
    vs = np.array([4.5 / 448, 6.0 / 448], np.float32)
    return q, orc.quantize_cache(kc, ks), orc.quantize_cache(vc, vs), ks, vs, bt, np.array(ctxs, np.int32)


def check_decode_fp8_dense_equivalence(orc):
    """FP8 decode = dense fp64 attention over the exactly dequantised K, V (torch decode)."""
    q, k8, v8, ks, vs, bt, ctx = _fp8_case(orc)
    scale = 1.0 / math.sqrt(D)
    got, _ = orc.decode_fp8(q, k8, v8, ks, vs, bt, ctx, scale)
    kd = _torch_e4m3_decode(k8) * ks.astype(np.float64)[None, :, None, None]
    vd = _torch_e4m3_decode(v8) * vs.astype(np.float64)[None, :, None, None]
    for s, c in enumerate(ctx):
        blocks = bt[s, :(int(c) + 15) // 16]
        Kd = kd[blocks].transpose(1, 0, 2, 3).reshape(2, -1, D)[:, :c]
        Vd = vd[blocks].transpose(1, 0, 2, 3).reshape(2, -1, D)[:, :c]
        qs = W.bf16_bits_to_f32(q[s]).astype(np.float64)
        for h in range(12):
            g = h // 6
            ref = softmax(scale * (Kd[g] @ qs[h])) @ Vd[g]
            assert np.allclose(got[s, h], ref, rtol=1e-12, atol=1e-14), (s, h)


def check_rope_kv_store_fp8_is_bf16_store_then_quantise(orc):
    """The FP8 store equals the bf16 store followed by quantisation of the stored rows."""
    w = W.make("tiny")
    ks = np.array([3.0 / 448, 5.0 / 448], np.float32)
    vs = np.array([2.0 / 448, 4.0 / 448], np.float32)
    kc16, vc16 = w.k_cache[0].copy(), w.v_cache[0].copy()
    q16 = orc.rope_kv_store(w.q[0], w.k[0], w.v[0], w.positions, w.cos_sin, w.slot_mapping, kc16, vc16)
    kc8 = np.zeros(kc16.shape, np.uint8)
    vc8 = np.zeros(vc16.shape, np.uint8)
    q8 = orc.rope_kv_store_fp8(w.q[0], w.k[0], w.v[0], w.positions, w.cos_sin, w.slot_mapping,
                               kc8, vc8, ks, vs)
    assert np.array_equal(q8, q16)
    blk, off = np.divmod(w.slot_mapping, W.BLOCK_SIZE)
    for i in range(len(blk)):
        krow = kc16[blk[i], :, off[i]]
        vrow = vc16[blk[i], :, off[i]]
        for g in range(2):
            inv_k = np.float32(1.0) / ks[g]
            inv_v = np.float32(1.0) / vs[g]
            want_k = _torch_e4m3_encode((W.bf16_bits_to_f32(krow[g]) * inv_k).astype(np.float32))
            want_v = _torch_e4m3_encode((W.bf16_bits_to_f32(vrow[g]) * inv_v).astype(np.float32))
            assert np.array_equal(kc8[blk[i], g, off[i]], want_k)
            assert np.array_equal(vc8[blk[i], g, off[i]], want_v)
    mask = np.ones(kc8.shape, bool)
    mask[blk, :, off] = False
    assert not kc8[mask].any() and not vc8[mask].any()


ALL_CHECKS = [
    check_bf16_widen,
    check_bf16_narrow_bruteforce,
    check_rope_identity_at_pos0,
    check_rope_unit_vectors,
    check_rope_pair_norm,
    check_rope_relative_position,
    check_rope_kv_store_placement,
    check_decode_dense_equivalence,
    check_decode_block_permutation_invariance,
    check_decode_ctx1_returns_v,
    check_decode_identical_keys_mean,
    check_decode_gqa_head_mapping,
    check_decode_two_token_logistic,
    check_decode_large_scores_stable,
    check_decode_ignores_canaries_and_unused_entries,
    check_decode_empty_context,
    check_store_then_decode_matches_dense,
    check_flash_decode_merge_equals_unsplit,
    check_copy_blocks_matches_fancy_indexing,
    check_copy_blocks_skips_out_of_range_pairs,
    check_swap_out_in_preserves_decode,
    check_e4m3_decode_all_codes,
    check_e4m3_encode_rne_and_saturation,
    check_quantize_cache_definition,
    check_quantize_decides_in_fp32,
    check_decode_fp8_dense_equivalence,
    check_rope_kv_store_fp8_is_bf16_store_then_quantise,
    check_prefill_full_equals_dense_causal,
    check_prefill_one_token_is_decode,
    check_prefill_chunks_compose,
    check_prefill_is_causal,
]
