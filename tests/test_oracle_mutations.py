"""The pins have teeth: each plausible mistake, planted in a copy of the
oracle's C source on the CPU, makes at least one pin fail.

Each mutant is compiled into a temporary directory and its pins are run in a
child process, so a mutant that misbehaves cannot take the test run down.
"""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "causal_off_by_one": ("int n_keys = pos + 1;", "int n_keys = pos > 0 ? pos : 1;"),
    "top_left_causal": ("int pos = seq_len - qo_len + j;", "int pos = j;"),
    "gqa_interleaved": ("int kvh = h / G;", "int kvh = h % a->Hkv;"),
    "scale_dropped": ("s[t] = a->sm_scale * dot;", "s[t] = dot;"),
    "softmax_sign": ("double w = exp(s[t] - m);", "double w = exp(m - s[t]);"),
    "values_from_keys": ("o[d] += w * kv_elem(a, 1,", "o[d] += w * kv_elem(a, 0,"),
    "page_index_mod": ("int64_t block = table[t / a->p];\n    if", "int64_t block = table[(t / a->p) % 2];\n    if"),
    "lse_log2": ("*lse = m + log(l);", "*lse = m + log2(l);"),
    "nhd_layout": ("return (((size_t)block * (size_t)Hkv + (size_t)kvh) * (size_t)p + (size_t)off) * (size_t)D",
                   "return (((size_t)block * (size_t)p + (size_t)off) * (size_t)Hkv + (size_t)kvh) * (size_t)D"),
    "append_offset": ("    int off = (int)(slot % block_size);\n    if (block >= num_blocks) return ORACLE_ERR_INDEX;\n"
                      "    for (int h = 0; h < num_kv_heads; ++h) {\n      for (int d = 0;",
                      "    int off = (int)((slot + 1) % block_size);\n    if (block >= num_blocks) return ORACLE_ERR_INDEX;\n"
                      "    for (int h = 0; h < num_kv_heads; ++h) {\n      for (int d = 0;"),
    "q8_append_offset": ("          memcpy(s + (size_t)off * head_dim + 32 * g, codes, 32);",
                         "          memcpy(s + (size_t)((off + 1) % block_size) * head_dim + 32 * g, codes, 32);"),
    "merge_weight_sign": ("double wa = exp(la - M), wb = exp(lb - M);", "double wa = exp(M - la), wb = exp(lb - M);"),
    "merge_lse_dropped": ("lse_out[i] = M + log(wa + wb);", "lse_out[i] = M;"),
    "normalise_dropped": ("for (int d = 0; d < a->D; ++d) o[d] /= l;", ""),
    "round_truncates": ("double r = ldexp(rint(ldexp(m, 8)), e - 8);", "double r = ldexp(trunc(ldexp(m, 8)), e - 8);"),
    "copy_keys_only": ("          v_cache[to] = v_cache[from];\n", ""),
    "copy_one_head": ("    for (int h = 0; h < num_kv_heads; ++h)\n      for (int off = 0; off < block_size; ++off)",
                      "    for (int h = 0; h < 1; ++h)\n      for (int off = 0; off < block_size; ++off)"),
    "copy_reversed": ("          k_cache[to] = k_cache[from];", "          k_cache[from] = k_cache[to];"),
    "q8_scale_128": ("float d = amax / 127.0f;", "float d = amax / 128.0f;"),
    "q8_code_trunc": ("float t = rintf((float)bf16_to_double(x[i]) / d16);",
                      "float t = truncf((float)bf16_to_double(x[i]) / d16);"),
    "q8_scale_index": ("2 * ((size_t)off * (D / 32) + d / 32)", "2 * ((size_t)off * (D / 32) + d / 64)"),
    "step_slot_next": ("int64_t pos = L - 1;", "int64_t pos = L;"),
    "step_slot_offset": ("slots[r] = block * block_size + pos % block_size;",
                         "slots[r] = block * block_size + pos / block_size;"),
    "step_padding_written": ("    if (L == 0) continue;\n    if (L < 0 ||", "    if (L < 0 ||"),
    "step_bound_ignored": ("if (L < 0 || L > max_seq_len ||", "if (L < 0 ||"),
    "f16_round_trunc": ("r = ldexp(rint(ldexp(m, 11)), e - 11);", "r = ldexp(trunc(ldexp(m, 11)), e - 11);"),
    "q_row_of_request": ("a->q + ((size_t)tok * (size_t)a->Hq + (size_t)h)", "a->q + ((size_t)r * (size_t)a->Hq + (size_t)h)"),
    "q_head_of_group": ("a->q + ((size_t)tok * (size_t)a->Hq + (size_t)h)",
                        "a->q + ((size_t)tok * (size_t)a->Hq + (size_t)(kvh * G))"),
    "table_row_stride": ("a->block_tables + (size_t)r * (size_t)a->max_blocks_per_req;",
                         "a->block_tables + (size_t)r * (size_t)(a->max_blocks_per_req - 1);"),
    "request_boundary": ("if (tok >= a->qo_indptr[r] && tok < a->qo_indptr[r + 1]) return r;",
                         "if (tok >= a->qo_indptr[r] && tok <= a->qo_indptr[r + 1]) return r;"),
    "append_src_head_stride": ("size_t src = ((size_t)i * (size_t)num_kv_heads + (size_t)h) * (size_t)head_dim",
                               "size_t src = ((size_t)h * (size_t)n_tokens + (size_t)i) * (size_t)head_dim"),
    "append_skip_kept": ("    if (slot < 0) continue;\n    int64_t block = slot / block_size;\n"
                         "    int off = (int)(slot % block_size);\n    if (block >= num_blocks) return ORACLE_ERR_INDEX;\n"
                         "    for (int h = 0; h < num_kv_heads; ++h) {\n      for (int d = 0;",
                         "    if (slot < 0) slot = 0;\n    int64_t block = slot / block_size;\n"
                         "    int off = (int)(slot % block_size);\n    if (block >= num_blocks) return ORACLE_ERR_INDEX;\n"
                         "    for (int h = 0; h < num_kv_heads; ++h) {\n      for (int d = 0;"),
    "q8_clamp_128": ("c = t > 127.0f ? 127 : (t < -127.0f ? -127 : (int)t);",
                     "c = t > 127.0f ? 127 : (t < -128.0f ? -128 : (int)t);"),
    "q8_amax_signed": ("float v = (float)fabs(bf16_to_double(x[i]));", "float v = (float)bf16_to_double(x[i]);"),
    "q8_scale_unrounded": ("float t = rintf((float)bf16_to_double(x[i]) / d16);",
                           "float t = rintf((float)bf16_to_double(x[i]) / d);"),
    "f16_subnormal_flushed": ("if (r < ldexp(1.0, -14)) return sign | (uint16_t)ldexp(r, 24);",
                              "if (r < ldexp(1.0, -14)) return sign;"),
    "f16_overflow_late": ("if (r >= 65520.0 || isinf(a)) return sign | 0x7c00;",
                          "if (r >= 131072.0 || isinf(a)) return sign | 0x7c00;"),
    "round_ties_away": ("double r = ldexp(rint(ldexp(m, 8)), e - 8);", "double r = ldexp(round(ldexp(m, 8)), e - 8);"),
    "f16_ties_away": ("r = ldexp(rint(ldexp(m, 11)), e - 11);", "r = ldexp(round(ldexp(m, 11)), e - 11);"),
    "sampled_head_swapped": ("int e = attend_one(&a, request_of(&a, sample_tok[i]), sample_tok[i], sample_head[i], s,",
                             "int e = attend_one(&a, request_of(&a, sample_tok[i]), sample_tok[i], sample_head[i] ^ 1, s,"),
    "merge_other_part_zero": ("double ta = wa > 0.0 ? wa * va : 0.0, tb = wb > 0.0 ? wb * vb : 0.0;",
                              "double ta = wa > 0.0 ? wa * va : 0.0, tb = 0.0;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutant_src = tmp_path / "mutant.c"
    mutant_src.write_text(src.replace(old, new))
    lib = oracle.compile_oracle(str(mutant_src), str(tmp_path / "libmutant.so"))
    res = subprocess.run([sys.executable, "-m", "tests.oracle_pins", lib], cwd=ROOT, capture_output=True, text=True,
                         timeout=300)
    assert res.returncode != 0, f"no pin caught mutant {name}:\n{res.stdout}\n{res.stderr}"


def test_unmutated_copy_passes(tmp_path):
    lib = oracle.compile_oracle(oracle.SOURCE, str(tmp_path / "libcopy.so"))
    res = subprocess.run([sys.executable, "-m", "tests.oracle_pins", lib], cwd=ROOT, capture_output=True, text=True,
                         timeout=300)
    assert res.returncode == 0, res.stdout + res.stderr
