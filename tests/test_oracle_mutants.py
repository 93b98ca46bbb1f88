"""Mutation test for the oracle's pins (no GPU).

Each case plants one plausible mistake in a copy of the oracle's C source
(a dropped term, a wrong sign, a wrong index, a transposed operand), builds
it, and runs every pin against the broken build in a child process. The
pins pass on the real oracle (test_oracle_pins.py); here at least one of them
must fail for every mutant, otherwise the pins would not have noticed that
mistake in the oracle.
"""
import os
import subprocess
import sys
import textwrap

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "paged_attn_oracle.c")

MUTANTS = {
    "page_index_mod": ("p->max_blocks + t / p->bs]", "p->max_blocks + t % p->bs]"),
    "slot_index_div": ("int off = t % p->bs;", "int off = t / p->bs;"),
    "gqa_head_modulo": ("int h = hq / G;", "int h = hq % p->Hkv;"),
    "cache_head_slot_transposed": ("(((int64_t)blk * p->bs + off) * p->Hkv + h) * p->D",
                                   "(((int64_t)blk * p->Hkv + h) * p->bs + off) * p->D"),
    "q_index_transposed": ("p->q + ((int64_t)b * p->Hq + hq) * p->D",
                           "p->q + ((int64_t)hq * p->B + b) * p->D"),
    "dropped_scale": ("return p->scale * dot;", "return dot;"),
    "softmax_sign": ("double w = exp(s[t - t0] - m);", "double w = exp(m - s[t - t0]);"),
    "no_max_shift": ("double w = exp(s[t - t0] - m);", "double w = exp(s[t - t0]);"),
    "no_normalisation": ("for (int d = 0; d < p->D; ++d) o[d] /= l;", "(void)l;"),
    "v_reads_k": ("kv_value(p, p->v_cache, p->v_scale", "kv_value(p, p->k_cache, p->v_scale"),
    "off_by_one_context": ("attend_range(p, b, hq, 0, p->context_lens[b],",
                           "attend_range(p, b, hq, 0, p->context_lens[b] - (p->context_lens[b] > 1),"),
    "split_lse_drops_log": ("lse[idx] = (l > 0.0) ? m + log(l) : -INFINITY;",
                            "lse[idx] = (l > 0.0) ? m : -INFINITY;"),
    "merge_weight_sign": ("double w = exp(l - M);", "double w = exp(M - l);"),
    "merge_no_normalisation": ("for (int d = 0; d < D; ++d) orow[d] /= wsum;", "(void)wsum;"),
    "bf16_exponent_bias": ("exp - 127 - 7", "exp - 127 - 8"),
    "fp16_subnormal_scale": ("ldexp((double)frac, -14 - 10)", "ldexp((double)frac, -15 - 10)"),
    "rne_ties_away": ("r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;", "r = fl + 1.0;"),
    "e4m3_bias": ("else v = ldexp(8.0 + m, e - 7 - 3);", "else v = ldexp(8.0 + m, e - 8 - 3);"),
    "e4m3_subnormal": ("if (e == 0) v = ldexp((double)m, -9);", "if (e == 0) v = ldexp((double)m, -10);"),
    "kv_scale_wrong_head": ("return head_scale ? x * head_scale[h] : x;",
                            "return head_scale ? x * head_scale[(h + 1) % p->Hkv] : x;"),
    "k_uses_v_scale": ("kv_value(p, p->k_cache, p->k_scale", "kv_value(p, p->k_cache, p->v_scale"),
    "copy_direction": ("k_cache[dst * block_bytes + j] = k_cache[src * block_bytes + j];",
                       "k_cache[src * block_bytes + j] = k_cache[dst * block_bytes + j];"),
    "gather_page_index": ("int32_t blk = block_table[(int64_t)b * max_blocks + t / block_size];",
                          "int32_t blk = block_table[(int64_t)b * max_blocks + t % block_size];"),
    "gather_no_advance": ("      ++row;\n", "\n"),
    "scatter_writes_padding": ("    if (slot < 0) continue;\n    if (slot >= num_slots)",
                               "    if (slot < 0) slot = 0;\n    if (slot >= num_slots)"),
    "remap_by_position": ("*e = new_id[*e];", "*e = new_id[p];"),
    "rows_b_hq_swapped": ("      b = j->rows[2 * r];\n      hq = j->rows[2 * r + 1];",
                          "      b = j->rows[2 * r + 1];\n      hq = j->rows[2 * r];"),
    "rows_pair_stride": ("      b = j->rows[2 * r];\n", "      b = j->rows[r];\n"),
    "rows_ignored": ("    if (j->rows) {\n      b = j->rows", "    if (0) {\n      b = j->rows"),
    "rope_second_sign": ("double yb = xb * c + xa * s;", "double yb = xb * c - xa * s;"),
    "rope_first_sign": ("double ya = xa * c - xb * s;", "double ya = xa * c + xb * s;"),
    "rope_neox_pairing": ("int b = neox ? j + half : 2 * j + 1;",
                          "int b = neox ? rot_dim - 1 - j : 2 * j + 1;"),
    "rope_interleaved_pairing": ("int a = neox ? j : 2 * j;", "int a = neox ? j : j;"),
    "rope_sin_from_cos_half": ("s = (double)cs[half + j];", "s = (double)cs[j];"),
    "rope_table_row_stride": ("cos_sin + (int64_t)pos * rot_dim;",
                              "cos_sin + (int64_t)pos * (rot_dim / 2);"),
    "rope_cache_head_stride": ("int64_t dst = (slot * Hkv + h) * D;",
                               "int64_t dst = (slot + h * Hkv) * D;"),
    "rope_v_copies_k": ("v_cache[dst + d] = v[src + d];", "v_cache[dst + d] = k[src + d];"),
    "rope_writes_padding_slot": ("if (slot < 0 || slot >= num_slots) continue;",
                                 "if (slot >= num_slots) continue; if (slot < 0) slot = 0;"),
}

RUNNER = textwrap.dedent("""
    import sys
    sys.path[:0] = [{root!r}, {tests!r}]
    import oracle, oracle_pins
    lib = oracle.load({so!r})
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except Exception as e:  # any failure counts as the mistake being caught
            failed.append(pin.__name__)
    print("FAILED_PINS", ",".join(failed))
""")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutant_src = tmp_path / "mutant.c"
    mutant_src.write_text(src.replace(old, new))
    so = str(tmp_path / "libmutant.so")
    oracle.compile_oracle(str(mutant_src), so)
    code = RUNNER.format(root=ROOT, tests=os.path.join(ROOT, "tests"), so=so)
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                         timeout=600)
    if res.returncode != 0:
        return  # the broken oracle crashed under the pins: caught
    line = [ln for ln in res.stdout.splitlines() if ln.startswith("FAILED_PINS")]
    assert line, res.stdout + res.stderr
    failed = line[0].split(" ", 1)[1].strip() if " " in line[0] else ""
    assert failed, f"no pin caught the mutant {name}"
