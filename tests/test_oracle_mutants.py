"""Planted mistakes in a copy of the oracle must each fail at least one pin (CPU only).

Each mutant is oracle.cpp with one plausible slip (a flipped sign, a dropped term, a wrong
index or head mapping, the wrong rounding), compiled into a temporary library.  The pins of
oracle_checks.py run against it in a child process (a slip in indexing can crash the
mutant, which also counts as detected); a mutant that passes every pin would mean the pins
cannot tell that slip from the method, so the test fails.
"""

import json
import subprocess
import sys
from pathlib import Path

import pytest

import oracle

ROOT = Path(__file__).resolve().parents[1]

_CHILD = """
import json, sys
sys.path[:0] = [sys.argv[2], sys.argv[2] + '/tests']
import oracle, oracle_checks
orc = oracle.Oracle(sys.argv[1])
caught = []
for check in oracle_checks.ALL_CHECKS:
    try:
        check(orc)
    except (AssertionError, ValueError):
        caught.append(check.__name__)
    print(json.dumps(caught), flush=True)
"""

MUTANTS = {
    "rope_sign": ("y[i] = a * c - b * s;", "y[i] = a * c + b * s;"),
    "rope_sin_is_cos": ("const double s = static_cast<double>(cs_row[half + i]);",
                        "const double s = static_cast<double>(cs_row[i]);"),
    "rope_pairing": ("const double b = widen_bf16(x[half + i]);",
                     "const double b = widen_bf16(x[(i + 1) % D]);"),
    "q_not_written_back": ("for (int d = 0; d < D; ++d) qh[d] = narrow_bf16(y[d]);", ""),
    "store_k_unrotated": ("k_cache[cache_index(blk, h, off, d, Hkv, B, D)] = narrow_bf16(y[d]);",
                          "k_cache[cache_index(blk, h, off, d, Hkv, B, D)] = kh[d];"),
    "store_v_wrong_offset": ("v_cache[cache_index(blk, h, off, d, Hkv, B, D)] = vh[d];",
                             "v_cache[cache_index(blk, h, (off + 1) % B, d, Hkv, B, D)] = vh[d];"),
    "gqa_interleaved": ("for (int h = g * G; h < (g + 1) * G; ++h) {\n"
                        "      const size_t obase = (static_cast<size_t>(s) * Hq + h) * D;\n"
                        "      std::fill(",
                        "for (int h = g; h < Hq; h += Hkv) {\n"
                        "      const size_t obase = (static_cast<size_t>(s) * Hq + h) * D;\n"
                        "      std::fill("),
    "no_scale": ("scores[t - t0] = scale * dot;", "scores[t - t0] = dot;"),
    "context_off_by_one": ("const int ctx = context_lens[s];\n"
                           "    const int32_t* bt_row = block_tables + static_cast<size_t>(s) * max_blocks;\n"
                           "    std::vector<double> scores(std::max(ctx, 1));",
                           "const int ctx = context_lens[s] > 1 ? context_lens[s] - 1 : context_lens[s];\n"
                           "    const int32_t* bt_row = block_tables + static_cast<size_t>(s) * max_blocks;\n"
                           "    std::vector<double> scores(std::max(ctx, 1));"),
    "block_offset": ("const int off = t % B;", "const int off = (t + 1) % B;"),
    "block_index": ("const int blk = bt_row[t / B];", "const int blk = bt_row[(t + B - 1) / B];"),
    "no_max_shift": ("const double p = std::exp(scores[t] - m);",
                     "const double p = std::exp(scores[t]);"),
    "no_normalisation": ("o[d] /= l;", "o[d] /= 1.0;"),
    "v_read_from_k": ("o[d] += p * widen_bf16(v_cache[", "o[d] += p * widen_bf16(k_cache["),
    "round_ties_away": ("std::nearbyint(scaled)", "std::round(scaled)"),
    "no_subnormals": ("if (qexp < -133) qexp = -133;", "if (qexp < -126) qexp = -126;"),
    "widen_shift": ("uint32_t u = static_cast<uint32_t>(b) << 16;",
                    "uint32_t u = static_cast<uint32_t>(b) << 15;"),
    "merge_drops_l": ("const double w = std::exp(mp[p] - M) * lp[p] / L;",
                      "const double w = std::exp(mp[p] - M) / L;"),
    "copy_ids_swapped": ("dst[c][to * block_elems + e] = src[c][from * block_elems + e];",
                         "dst[c][from * block_elems + e] = src[c][to * block_elems + e];"),
    "copy_first_cache_only": ("for (int c = 0; c < num_caches; ++c)\n      for (int64_t e = 0;",
                              "for (int c = 0; c < 1; ++c)\n      for (int64_t e = 0;"),
    "copy_skips_last_element": ("for (int64_t e = 0; e < block_elems; ++e)",
                                "for (int64_t e = 0; e + 1 < block_elems; ++e)"),
    "e4m3_bias_8": ("else v = std::ldexp(1.0 + m / 8.0, e - 7);",
                    "else v = std::ldexp(1.0 + m / 8.0, e - 8);"),
    "e4m3_ties_away": ("const double q = std::nearbyint(std::ldexp(a, -qexp));  // ties to even",
                       "const double q = std::round(std::ldexp(a, -qexp));"),
    "e4m3_no_saturation": ("if (a >= 448.0) return sign | 0x7E;", "if (a >= 448.0) return sign | 0x7F;"),
    "quantise_divides_in_double": ("const float y = static_cast<float>(widen_bf16(x_bf16)) * inv;",
                                   "const float y = static_cast<float>(widen_bf16(x_bf16) / scale);"),
    "fp8_store_k_with_v_scale": ("e4m3_encode(quant_input(narrow_bf16(y[d]), k_scale[h]));",
                                 "e4m3_encode(quant_input(narrow_bf16(y[d]), v_scale[h]));"),
    "fp8_decode_drops_k_scale": ("(e4m3_value(k_cache[cache_index(blk, g, off, d, Hkv, B, D)]) * ks);",
                                 "(e4m3_value(k_cache[cache_index(blk, g, off, d, Hkv, B, D)]) * 1.0);"),
    "prefill_position_from_start": ("const int pos = ctx - n + i;          // attends to tokens 0..pos",
                                    "const int pos = i;"),
    "prefill_sum_drops_last": ("for (int t = 0; t <= pos; ++t) {", "for (int t = 0; t < pos; ++t) {"),
    "prefill_q_row_stride": ("const size_t obase = (static_cast<size_t>(q_start[s] + i) * Hq + h) * D;",
                             "const size_t obase = (static_cast<size_t>(q_start[s] + i) * Hkv + h) * D;"),
    "fp8_decode_wrong_v_head": ("o[d] += p * (e4m3_value(v_cache[cache_index(blk, g, off, d, Hkv, B, D)]) * vs);",
                                "o[d] += p * (e4m3_value(v_cache[cache_index(blk, (g + 1) % Hkv, off, d, Hkv, B, D)]) * vs);"),
}


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    return tmp_path_factory.mktemp("oracle_mutants")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, mutant_dir):
    old, new = MUTANTS[name]
    src = oracle.SOURCE.read_text()
    assert old in src, f"mutation site for {name} no longer in oracle.cpp"
    mutated = src.replace(old, new)
    path = Path(mutant_dir) / f"{name}.cpp"
    path.write_text(mutated)
    lib = oracle.build(force=True, src=path, out=Path(mutant_dir) / f"lib{name}.so")
    r = subprocess.run([sys.executable, "-c", _CHILD, str(lib), str(ROOT)], capture_output=True,
                       text=True, timeout=300)
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("[")]
    caught = json.loads(lines[-1]) if lines else []
    crashed = r.returncode != 0
    assert caught or crashed, f"no pin catches mutant {name}"
