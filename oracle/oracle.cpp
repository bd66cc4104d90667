// Paged GQA decode attention and fused RoPE + KV-cache store: plain fp64 CPU oracle.
//
// TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only tests/, __graft_entry__.smoke() and the
// CPU-baseline leg of bench.py may load, call or link this file.  It shares no code,
// header, table or helper with the CUDA library under paged_kv_cache_244_gb300/, and the
// library never calls it.
//
// Every function below is the plain definition of what the method computes, written out
// with no blocking, fusion or reordering beyond what that definition states:
//
//  * Paged KV cache.  The cache is an array of fixed 16-token physical blocks; each
//    sequence owns a block table that maps its logical block j to a physical block id,
//    so token t of the sequence lives in physical block block_table[t / 16] at offset
//    t % 16.  ("从零实现 LLM 推理引擎：深挖 vLLM 的六大核心优化", §3.1 Paged KV Cache:
//    16 tokens per block, block_table as a page table; "nano-vllm：vLLM 极简实现与大模型
//    推理流程解析", FAQ 2: logical-to-physical block mapping table.)
//  * The new token's slot is (physical block of its position) * 16 + position % 16, the
//    plain reading of append_slot (same page, §3.2 Continuous Batching).
//  * GQA: consecutive groups of G = Hq / Hkv query heads share one KV head; query head h
//    reads KV head h / G.  ("Pico-vLLM：从零手写的工业级LLM推理引擎实现", §核心技术架构解析
//    1. 模型实现层: GQA.)
//  * RoPE in the rotate_half form: for i < D/2, with (c, s) = (cos, sin) of the token's
//    angle for frequency i,
//        y[i]       = x[i] * c - x[i + D/2] * s
//        y[i + D/2] = x[i + D/2] * c + x[i] * s
//    (same page and section: RoPE, rotate_half computed in place; §2. Kernel层: fused
//    RoPE + KV cache store).  The cos/sin values are an input table, one fp32 row of
//    [cos(0..D/2-1) | sin(0..D/2-1)] per position.
//  * Single-token decode: each query head attends over all context_len cached tokens of
//    its sequence (the token just stored included): softmax(scale * q K^T) V
//    (same page, §2. Kernel层: PagedAttention Decode Kernel).
//  * Flash Decode: the context is cut into partitions; each gives (m_p, l_p, o_p) and an
//    exp-weighted merge gives the same result as the unsplit softmax (same page, §H200上的
//    详细对比 names Flash Decode; the merge is the standard log-sum-exp identity, the plain
//    reading since the page gives no formula).
//
// Arithmetic: bf16 inputs are widened exactly to double; every sum, exp and product is in
// double; results are rounded once to bf16 with round-to-nearest-even.
//
// Cache layout (the pages leave it open): k_cache and v_cache are each
// [num_blocks][Hkv][block_size][D] bf16, row-major.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

double widen_bf16(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

// Round a double to the nearest bf16 (8 significant bits, exponent range of fp32), ties to
// even, in one step.  The quantum of the binade of |x| is 2^(e-8) where |x| in
// [2^(e-1), 2^e); below 2^-126 the quantum is fixed at 2^-133 (bf16 subnormals).
uint16_t narrow_bf16(double x) {
  if (std::isnan(x)) return 0x7FC0;
  if (std::isinf(x)) return x > 0 ? 0x7F80 : 0xFF80;
  if (x == 0.0) return std::signbit(x) ? 0x8000 : 0x0000;
  int e = 0;
  std::frexp(x, &e);  // |x| = m * 2^e, m in [0.5, 1)
  int qexp = e - 8;
  if (qexp < -133) qexp = -133;
  double scaled = std::ldexp(x, -qexp);     // exact: power-of-two scaling
  double r = std::nearbyint(scaled);        // default rounding mode: nearest, ties to even
  double y = std::ldexp(r, qexp);           // exact, representable in bf16 or overflowing
  const double max_bf16 = std::ldexp(255.0, 120);  // (2 - 2^-7) * 2^127
  if (std::fabs(y) > max_bf16) return y > 0 ? 0x7F80 : 0xFF80;
  float f = static_cast<float>(y);          // exact: y has at most 8 significant bits
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  return static_cast<uint16_t>(u >> 16);
}

// FP8 E4M3 (the OCP "E4M3FN" format): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
// bits; exponent 0 holds the subnormals m/8 * 2^-6; S.1111.111 is NaN; no infinities, so the
// largest finite magnitude is 1.75 * 2^8 = 448.
double e4m3_value(uint8_t b) {
  const int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
  double v;
  if (e == 15 && m == 7) v = std::numeric_limits<double>::quiet_NaN();
  else if (e == 0) v = std::ldexp(m / 8.0, -6);
  else v = std::ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -v : v;
}

// Nearest E4M3 code to x, ties to even, magnitudes beyond 448 (infinities included) clamped to
// 448 ("saturate to finite"); NaN gives the NaN code.  The quantum is 2^-9 below 2^-6 and
// 2^(e-3) in the binade [2^e, 2^(e+1)).
uint8_t e4m3_encode(double x) {
  if (std::isnan(x)) return std::signbit(x) ? 0xFF : 0x7F;
  const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  const double a = std::fabs(x);
  if (a >= 448.0) return sign | 0x7E;
  int qexp = -9;                              // subnormal quantum
  if (a >= std::ldexp(1.0, -6)) {
    int e = 0;
    std::frexp(a, &e);                        // a in [2^(e-1), 2^e)
    qexp = (e - 1) - 3;
  }
  const double q = std::nearbyint(std::ldexp(a, -qexp));  // ties to even
  const double y = std::ldexp(q, qexp);       // the rounded magnitude, exact
  if (y >= 448.0) return sign | 0x7E;         // cannot happen below 448, kept for clarity
  if (y < std::ldexp(1.0, -6)) return sign | static_cast<uint8_t>(q);       // subnormal or 2^-6
  int e = 0;
  std::frexp(y, &e);
  const int ef = (e - 1) + 7;                  // biased exponent of y
  const int m = static_cast<int>(std::ldexp(y, -(e - 1)) * 8.0) - 8;
  return sign | static_cast<uint8_t>((ef << 3) | m);
}

// The value a stored code is taken from: the bf16 input times the reciprocal of the scale,
// both in fp32 with round-to-nearest (the precision the kernels quantise in).
double quant_input(uint16_t x_bf16, float scale) {
  const float inv = 1.0f / scale;
  const float y = static_cast<float>(widen_bf16(x_bf16)) * inv;
  return static_cast<double>(y);
}

size_t cache_index(int blk, int h, int off, int d, int Hkv, int B, int D) {
  return ((static_cast<size_t>(blk) * Hkv + h) * B + off) * static_cast<size_t>(D) + d;
}

// Rotate one head vector of length D by the angles of one cos/sin table row.
void rotate_half(const uint16_t* x, int D, const float* cs_row, double* y) {
  const int half = D / 2;
  for (int i = 0; i < half; ++i) {
    const double c = static_cast<double>(cs_row[i]);
    const double s = static_cast<double>(cs_row[half + i]);
    const double a = widen_bf16(x[i]);
    const double b = widen_bf16(x[half + i]);
    y[i] = a * c - b * s;
    y[half + i] = b * c + a * s;
  }
}

bool shape_ok(int Hq, int Hkv, int D, int B) {
  return Hq > 0 && Hkv > 0 && Hq % Hkv == 0 && D > 0 && D % 2 == 0 && B > 0;
}

int pick_threads(int nthreads, int units) {
  int n = nthreads;
  if (n <= 0) n = static_cast<int>(std::thread::hardware_concurrency());
  if (n <= 0) n = 1;
  return std::max(1, std::min(n, units));
}

// Run fn(unit) for unit in [0, units); unit u is always computed by exactly one thread
// (thread u % n), so results do not depend on the thread count.
template <class F>
void parallel_units(int units, int nthreads, F fn) {
  const int n = pick_threads(nthreads, units);
  if (n == 1) {
    for (int u = 0; u < units; ++u) fn(u);
    return;
  }
  std::vector<std::thread> pool;
  pool.reserve(n);
  for (int t = 0; t < n; ++t)
    pool.emplace_back([=] {
      for (int u = t; u < units; u += n) fn(u);
    });
  for (auto& th : pool) th.join();
}

// Scores of one query head over tokens [t0, t1) of one sequence, in double.
void head_scores(const uint16_t* qh, const uint16_t* k_cache, const int32_t* bt_row, int g,
                 int t0, int t1, int Hkv, int B, int D, double scale, double* scores) {
  for (int t = t0; t < t1; ++t) {
    const int blk = bt_row[t / B];
    const int off = t % B;
    double dot = 0.0;
    for (int d = 0; d < D; ++d)
      dot += widen_bf16(qh[d]) * widen_bf16(k_cache[cache_index(blk, g, off, d, Hkv, B, D)]);
    scores[t - t0] = scale * dot;
  }
}

bool table_ok(const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
              int num_seqs, int num_blocks, int B) {
  for (int s = 0; s < num_seqs; ++s) {
    const int ctx = context_lens[s];
    if (ctx < 0 || ctx > max_blocks * B) return false;
    const int nblk = (ctx + B - 1) / B;
    for (int j = 0; j < nblk; ++j) {
      const int blk = block_tables[static_cast<size_t>(s) * max_blocks + j];
      if (blk < 0 || blk >= num_blocks) return false;
    }
  }
  return true;
}

}  // namespace

extern "C" {

double orc_bf16_to_f64(uint16_t b) { return widen_bf16(b); }

uint16_t orc_f64_to_bf16(double x) { return narrow_bf16(x); }

// Rotated head vector in double, before rounding (for pinning the rotation itself).
int orc_rope_rotate_f64(const uint16_t* x, int D, const float* cs_row, double* y) {
  if (!x || !cs_row || !y || D <= 0 || D % 2) return -1;
  rotate_half(x, D, cs_row, y);
  return 0;
}

// Fused RoPE + KV-cache store for num_tokens new tokens.
//   q [T][Hq][D] bf16, rotated in place;  k, v [T][Hkv][D] bf16 (read only)
//   positions [T]; cos_sin [max_pos][D] fp32 = [cos | sin] halves
//   slot_mapping [T]: slot = physical block * B + offset; a negative slot skips the store
//   k_cache, v_cache [num_blocks][Hkv][B][D] bf16: rotated k and raw v written at the slot
// Returns 0, or -1 on a bad argument (nothing is written then).
int orc_rope_kv_store(int T, int Hq, int Hkv, int D, int B, uint16_t* q, const uint16_t* k,
                      const uint16_t* v, const int32_t* positions, const float* cos_sin,
                      int max_pos, const int64_t* slot_mapping, uint16_t* k_cache,
                      uint16_t* v_cache, int num_blocks) {
  if (T < 0 || !shape_ok(Hq, Hkv, D, B)) return -1;
  if (T == 0) return 0;
  if (!q || !k || !v || !positions || !cos_sin || !slot_mapping || !k_cache || !v_cache) return -1;
  for (int t = 0; t < T; ++t) {
    if (positions[t] < 0 || positions[t] >= max_pos) return -1;
    if (slot_mapping[t] >= static_cast<int64_t>(num_blocks) * B) return -1;
  }
  std::vector<double> y(D);
  for (int t = 0; t < T; ++t) {
    const float* row = cos_sin + static_cast<size_t>(positions[t]) * D;
    for (int h = 0; h < Hq; ++h) {
      uint16_t* qh = q + (static_cast<size_t>(t) * Hq + h) * D;
      rotate_half(qh, D, row, y.data());
      for (int d = 0; d < D; ++d) qh[d] = narrow_bf16(y[d]);
    }
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    const int blk = static_cast<int>(slot / B);
    const int off = static_cast<int>(slot % B);
    for (int h = 0; h < Hkv; ++h) {
      const uint16_t* kh = k + (static_cast<size_t>(t) * Hkv + h) * D;
      const uint16_t* vh = v + (static_cast<size_t>(t) * Hkv + h) * D;
      rotate_half(kh, D, row, y.data());
      for (int d = 0; d < D; ++d) {
        k_cache[cache_index(blk, h, off, d, Hkv, B, D)] = narrow_bf16(y[d]);
        v_cache[cache_index(blk, h, off, d, Hkv, B, D)] = vh[d];
      }
    }
  }
  return 0;
}

// Single-token paged decode attention, unsplit.
//   q [S][Hq][D] bf16; block_tables [S][max_blocks]; context_lens [S]
//   out_f64 [S][Hq][D] (may be null), out_bf16 [S][Hq][D] (may be null)
// A sequence with context_len 0 gets an all-zero output.
int orc_decode(int S, int Hq, int Hkv, int D, int B, const uint16_t* q, const uint16_t* k_cache,
               const uint16_t* v_cache, int num_blocks, const int32_t* block_tables,
               int max_blocks, const int32_t* context_lens, double scale, int nthreads,
               double* out_f64, uint16_t* out_bf16) {
  if (S < 0 || !shape_ok(Hq, Hkv, D, B) || max_blocks < 0) return -1;
  if (S == 0) return 0;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens) return -1;
  if (!table_ok(block_tables, max_blocks, context_lens, S, num_blocks, B)) return -1;
  const int G = Hq / Hkv;
  parallel_units(S * Hkv, nthreads, [&](int unit) {
    const int s = unit / Hkv;
    const int g = unit % Hkv;
    const int ctx = context_lens[s];
    const int32_t* bt_row = block_tables + static_cast<size_t>(s) * max_blocks;
    std::vector<double> scores(std::max(ctx, 1));
    std::vector<double> o(D);
    for (int h = g * G; h < (g + 1) * G; ++h) {
      const size_t obase = (static_cast<size_t>(s) * Hq + h) * D;
      std::fill(o.begin(), o.end(), 0.0);
      if (ctx > 0) {
        head_scores(q + obase, k_cache, bt_row, g, 0, ctx, Hkv, B, D, scale, scores.data());
        const double m = *std::max_element(scores.begin(), scores.begin() + ctx);
        double l = 0.0;
        for (int t = 0; t < ctx; ++t) {
          const double p = std::exp(scores[t] - m);
          l += p;
          const int blk = bt_row[t / B];
          const int off = t % B;
          for (int d = 0; d < D; ++d)
            o[d] += p * widen_bf16(v_cache[cache_index(blk, g, off, d, Hkv, B, D)]);
        }
        for (int d = 0; d < D; ++d) o[d] /= l;
      }
      for (int d = 0; d < D; ++d) {
        if (out_f64) out_f64[obase + d] = o[d];
        if (out_bf16) out_bf16[obase + d] = narrow_bf16(o[d]);
      }
    }
  });
  return 0;
}

// Flash Decode: the same attention, computed partition by partition and merged.
// Partition p covers tokens [p*P, min((p+1)*P, ctx)).  Each gives
//   m_p = max score,  l_p = sum exp(s - m_p),  o_p = sum exp(s - m_p) v / l_p
// and the merge is
//   M = max_p m_p,  out = sum_p exp(m_p - M) l_p o_p / sum_p exp(m_p - M) l_p.
// The result equals orc_decode's up to rounding order.
int orc_decode_partitioned(int S, int Hq, int Hkv, int D, int B, const uint16_t* q,
                           const uint16_t* k_cache, const uint16_t* v_cache, int num_blocks,
                           const int32_t* block_tables, int max_blocks,
                           const int32_t* context_lens, double scale, int partition_tokens,
                           int nthreads, double* out_f64) {
  if (S < 0 || !shape_ok(Hq, Hkv, D, B) || partition_tokens <= 0 || max_blocks < 0) return -1;
  if (S == 0) return 0;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out_f64) return -1;
  if (!table_ok(block_tables, max_blocks, context_lens, S, num_blocks, B)) return -1;
  const int G = Hq / Hkv;
  const int P = partition_tokens;
  parallel_units(S * Hkv, nthreads, [&](int unit) {
    const int s = unit / Hkv;
    const int g = unit % Hkv;
    const int ctx = context_lens[s];
    const int32_t* bt_row = block_tables + static_cast<size_t>(s) * max_blocks;
    const int nparts = (ctx + P - 1) / P;
    std::vector<double> scores(P), mp(nparts), lp(nparts), op(static_cast<size_t>(nparts) * D);
    for (int h = g * G; h < (g + 1) * G; ++h) {
      const size_t obase = (static_cast<size_t>(s) * Hq + h) * D;
      for (int p = 0; p < nparts; ++p) {
        const int t0 = p * P;
        const int t1 = std::min(ctx, t0 + P);
        head_scores(q + obase, k_cache, bt_row, g, t0, t1, Hkv, B, D, scale, scores.data());
        const double m = *std::max_element(scores.begin(), scores.begin() + (t1 - t0));
        double l = 0.0;
        double* o = op.data() + static_cast<size_t>(p) * D;
        std::fill(o, o + D, 0.0);
        for (int t = t0; t < t1; ++t) {
          const double w = std::exp(scores[t - t0] - m);
          l += w;
          const int blk = bt_row[t / B];
          const int off = t % B;
          for (int d = 0; d < D; ++d)
            o[d] += w * widen_bf16(v_cache[cache_index(blk, g, off, d, Hkv, B, D)]);
        }
        for (int d = 0; d < D; ++d) o[d] /= l;
        mp[p] = m;
        lp[p] = l;
      }
      for (int d = 0; d < D; ++d) out_f64[obase + d] = 0.0;
      if (nparts == 0) continue;
      const double M = *std::max_element(mp.begin(), mp.end());
      double L = 0.0;
      for (int p = 0; p < nparts; ++p) L += std::exp(mp[p] - M) * lp[p];
      for (int p = 0; p < nparts; ++p) {
        const double w = std::exp(mp[p] - M) * lp[p] / L;
        for (int d = 0; d < D; ++d) out_f64[obase + d] += w * op[static_cast<size_t>(p) * D + d];
      }
    }
  });
  return 0;
}

// Block copy between two block pools: copy-on-write inside one pool, swap out / swap in
// between the GPU pool and a CPU pool.  ("从零实现 LLM 推理引擎：深挖 vLLM 的六大核心优化",
// §3.4 Prefix Caching / Copy-on-Write: a block shared by several sequences (ref_count > 1) is
// replaced, before it is written, by a freshly allocated block, which must hold the same
// contents; §3.5 CPU Swap: swap_out moves a sequence's KV blocks to CPU memory and records the
// mapping, swap_in allocates new GPU blocks and restores them from it.)
//   src[c], dst[c]  pools of `src_blocks` / `dst_blocks` blocks of `block_elems` bf16 each,
//                   for every cache c < num_caches (e.g. K and V of every layer)
//   pairs           [num_pairs][2] = (source block, destination block)
// For each pair in order and each cache: dst[c][pair.dst] = src[c][pair.src], every element.
// A pair naming a block outside its pool is skipped.  Returns the number of pairs skipped,
// or -1 on a bad argument.
int64_t orc_copy_blocks(int num_caches, int64_t block_elems, const uint16_t* const* src,
                        int64_t src_blocks, uint16_t* const* dst, int64_t dst_blocks,
                        const int64_t* pairs, int num_pairs) {
  if (num_caches < 0 || block_elems <= 0 || num_pairs < 0 || src_blocks < 0 || dst_blocks < 0)
    return -1;
  if (num_pairs > 0 && (!pairs || !src || !dst)) return -1;
  int64_t skipped = 0;
  for (int i = 0; i < num_pairs; ++i) {
    const int64_t from = pairs[2 * i], to = pairs[2 * i + 1];
    if (from < 0 || from >= src_blocks || to < 0 || to >= dst_blocks) {
      ++skipped;
      continue;
    }
    for (int c = 0; c < num_caches; ++c)
      for (int64_t e = 0; e < block_elems; ++e)
        dst[c][to * block_elems + e] = src[c][from * block_elems + e];
  }
  return skipped;
}

// Paged prefill / chunked prefill: sequence s brings n_s = q_start[s+1] - q_start[s] new
// query tokens whose K and V are already in the cache, and context_lens[s] counts every cached
// token including them, so query i of s sits at position p = context_lens[s] - n_s + i and
// attends, causally, to the cached tokens 0..p of its sequence ("Pico-vLLM：从零手写的工业级LLM
// 推理引擎实现", §2 Kernel层: PagedAttention Prefill Kernel, after the FlashAttention work;
// "从零实现 LLM 推理引擎：深挖 vLLM 的六大核心优化", §3.3 Chunked Prefill: a prompt is prefilled
// in chunks, each continuing from the tokens already prefilled).  A full prefill is the case
// context_lens[s] = n_s; one new token (n_s = 1) is the decode.
//   q [T][Hq][D] bf16 (T = q_start[S]), out [T][Hq][D].
int orc_prefill(int S, int Hq, int Hkv, int D, int B, const uint16_t* q, const int32_t* q_start,
                const int32_t* context_lens, const uint16_t* k_cache, const uint16_t* v_cache,
                int num_blocks, const int32_t* block_tables, int max_blocks, double scale,
                int nthreads, double* out_f64, uint16_t* out_bf16) {
  if (S < 0 || !shape_ok(Hq, Hkv, D, B) || max_blocks < 0) return -1;
  if (S == 0) return 0;
  if (!q || !q_start || !context_lens || !k_cache || !v_cache || !block_tables) return -1;
  if (q_start[0] != 0) return -1;
  for (int s = 0; s < S; ++s) {
    const int n = q_start[s + 1] - q_start[s];
    if (n < 0 || context_lens[s] < n) return -1;
  }
  if (!table_ok(block_tables, max_blocks, context_lens, S, num_blocks, B)) return -1;
  const int G = Hq / Hkv;
  parallel_units(S * Hkv, nthreads, [&](int unit) {
    const int s = unit / Hkv;
    const int g = unit % Hkv;
    const int ctx = context_lens[s];
    const int n = q_start[s + 1] - q_start[s];
    const int32_t* bt_row = block_tables + static_cast<size_t>(s) * max_blocks;
    std::vector<double> scores(std::max(ctx, 1));
    std::vector<double> o(D);
    for (int i = 0; i < n; ++i) {
      const int pos = ctx - n + i;          // attends to tokens 0..pos
      for (int h = g * G; h < (g + 1) * G; ++h) {
        const size_t obase = (static_cast<size_t>(q_start[s] + i) * Hq + h) * D;
        head_scores(q + obase, k_cache, bt_row, g, 0, pos + 1, Hkv, B, D, scale, scores.data());
        const double m = *std::max_element(scores.begin(), scores.begin() + pos + 1);
        double l = 0.0;
        std::fill(o.begin(), o.end(), 0.0);
        for (int t = 0; t <= pos; ++t) {
          const double p = std::exp(scores[t] - m);
          l += p;
          const int blk = bt_row[t / B];
          const int off = t % B;
          for (int d = 0; d < D; ++d)
            o[d] += p * widen_bf16(v_cache[cache_index(blk, g, off, d, Hkv, B, D)]);
        }
        for (int d = 0; d < D; ++d) {
          o[d] /= l;
          if (out_f64) out_f64[obase + d] = o[d];
          if (out_bf16) out_bf16[obase + d] = narrow_bf16(o[d]);
        }
      }
    }
  });
  return 0;
}

// ---- FP8 (E4M3) KV cache with one scale per KV head --------------------------------------
// The pages name low-precision quantisation as a way to cut memory and raise inference speed
// ("nano-vllm：vLLM 极简实现与大模型推理流程解析", §学习要点: FP8 or INT4 quantisation with
// almost no loss of accuracy; "从零实现15倍加速：一个纯PyTorch LLM推理引擎的技术剖析", §未来展望:
// INT8 / FP16 quantisation to save memory and bandwidth) but give no format.  The plain
// reading for the KV cache: each cached K (V) element is stored as the E4M3 code of
// x / scale_g, where scale_g is the K (V) scale of its KV head, and read back as
// code * scale_g.

double orc_e4m3_to_f64(uint8_t b) { return e4m3_value(b); }

uint8_t orc_f64_to_e4m3(double x) { return e4m3_encode(x); }

// Quantise n bf16 values of head-major cache rows: element i belongs to KV head
// (i / (B * D)) % Hkv, the layout [num_blocks][Hkv][B][D].
int orc_quantize_cache(int64_t n, int Hkv, int B, int D, const uint16_t* src, const float* scale,
                       uint8_t* dst) {
  if (n < 0 || Hkv <= 0 || B <= 0 || D <= 0 || (n > 0 && (!src || !scale || !dst))) return -1;
  const int64_t per_head = static_cast<int64_t>(B) * D;
  for (int64_t i = 0; i < n; ++i) {
    const int g = static_cast<int>((i / per_head) % Hkv);
    dst[i] = e4m3_encode(quant_input(src[i], scale[g]));
  }
  return 0;
}

// RoPE + KV-cache store into FP8 caches: q is rotated in place exactly as orc_rope_kv_store
// does (bf16); k is rotated and rounded to bf16 as there, then stored as the E4M3 code of
// k_rot / k_scale[h]; v is stored as the code of v / v_scale[h].
int orc_rope_kv_store_fp8(int T, int Hq, int Hkv, int D, int B, uint16_t* q, const uint16_t* k,
                          const uint16_t* v, const int32_t* positions, const float* cos_sin,
                          int max_pos, const int64_t* slot_mapping, uint8_t* k_cache,
                          uint8_t* v_cache, int num_blocks, const float* k_scale,
                          const float* v_scale) {
  if (T < 0 || !shape_ok(Hq, Hkv, D, B)) return -1;
  if (T == 0) return 0;
  if (!q || !k || !v || !positions || !cos_sin || !slot_mapping || !k_cache || !v_cache ||
      !k_scale || !v_scale)
    return -1;
  for (int t = 0; t < T; ++t) {
    if (positions[t] < 0 || positions[t] >= max_pos) return -1;
    if (slot_mapping[t] >= static_cast<int64_t>(num_blocks) * B) return -1;
  }
  std::vector<double> y(D);
  for (int t = 0; t < T; ++t) {
    const float* row = cos_sin + static_cast<size_t>(positions[t]) * D;
    for (int h = 0; h < Hq; ++h) {
      uint16_t* qh = q + (static_cast<size_t>(t) * Hq + h) * D;
      rotate_half(qh, D, row, y.data());
      for (int d = 0; d < D; ++d) qh[d] = narrow_bf16(y[d]);
    }
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    const int blk = static_cast<int>(slot / B);
    const int off = static_cast<int>(slot % B);
    for (int h = 0; h < Hkv; ++h) {
      const uint16_t* kh = k + (static_cast<size_t>(t) * Hkv + h) * D;
      const uint16_t* vh = v + (static_cast<size_t>(t) * Hkv + h) * D;
      rotate_half(kh, D, row, y.data());
      for (int d = 0; d < D; ++d) {
        k_cache[cache_index(blk, h, off, d, Hkv, B, D)] =
            e4m3_encode(quant_input(narrow_bf16(y[d]), k_scale[h]));
        v_cache[cache_index(blk, h, off, d, Hkv, B, D)] = e4m3_encode(quant_input(vh[d], v_scale[h]));
      }
    }
  }
  return 0;
}

// Decode over FP8 caches: the same single-token attention as orc_decode, each cached element
// read as code * scale of its KV head (exact in double).
int orc_decode_fp8(int S, int Hq, int Hkv, int D, int B, const uint16_t* q, const uint8_t* k_cache,
                   const uint8_t* v_cache, const float* k_scale, const float* v_scale,
                   int num_blocks, const int32_t* block_tables, int max_blocks,
                   const int32_t* context_lens, double scale, int nthreads, double* out_f64,
                   uint16_t* out_bf16) {
  if (S < 0 || !shape_ok(Hq, Hkv, D, B) || max_blocks < 0) return -1;
  if (S == 0) return 0;
  if (!q || !k_cache || !v_cache || !k_scale || !v_scale || !block_tables || !context_lens)
    return -1;
  if (!table_ok(block_tables, max_blocks, context_lens, S, num_blocks, B)) return -1;
  const int G = Hq / Hkv;
  parallel_units(S * Hkv, nthreads, [&](int unit) {
    const int s = unit / Hkv;
    const int g = unit % Hkv;
    const int ctx = context_lens[s];
    const int32_t* bt_row = block_tables + static_cast<size_t>(s) * max_blocks;
    const double ks = static_cast<double>(k_scale[g]);
    const double vs = static_cast<double>(v_scale[g]);
    std::vector<double> scores(std::max(ctx, 1));
    std::vector<double> o(D);
    for (int h = g * G; h < (g + 1) * G; ++h) {
      const size_t obase = (static_cast<size_t>(s) * Hq + h) * D;
      std::fill(o.begin(), o.end(), 0.0);
      if (ctx > 0) {
        for (int t = 0; t < ctx; ++t) {
          const int blk = bt_row[t / B];
          const int off = t % B;
          double dot = 0.0;
          for (int d = 0; d < D; ++d)
            dot += widen_bf16(q[obase + d]) *
                   (e4m3_value(k_cache[cache_index(blk, g, off, d, Hkv, B, D)]) * ks);
          scores[t] = scale * dot;
        }
        const double m = *std::max_element(scores.begin(), scores.begin() + ctx);
        double l = 0.0;
        for (int t = 0; t < ctx; ++t) {
          const double p = std::exp(scores[t] - m);
          l += p;
          const int blk = bt_row[t / B];
          const int off = t % B;
          for (int d = 0; d < D; ++d)
            o[d] += p * (e4m3_value(v_cache[cache_index(blk, g, off, d, Hkv, B, D)]) * vs);
        }
        for (int d = 0; d < D; ++d) o[d] /= l;
      }
      for (int d = 0; d < D; ++d) {
        if (out_f64) out_f64[obase + d] = o[d];
        if (out_bf16) out_bf16[obase + d] = narrow_bf16(o[d]);
      }
    }
  });
  return 0;
}

int orc_hardware_threads(void) {
  const unsigned n = std::thread::hardware_concurrency();
  return n ? static_cast<int>(n) : 1;
}

}  // extern "C"
