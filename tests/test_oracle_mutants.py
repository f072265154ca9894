"""Plant single mistakes into a copy of the oracle and check the pins catch them.

Each mutant is one textual edit of oracle.c of the kind a careless restatement
of the pages could make (a dropped ReLU, a transposed operand, a strict
threshold, a reversed tie-break, a wrong E4M3 bias, ...).  The mutated copy is
compiled into a temporary directory and all pins run against it in a child
process (a crash counts as caught).  The test fails if any mutant survives.
"""
import json
import os
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle

TESTS = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(TESTS)

MUTANTS = {
    "relu_dropped": ("double relu = dot > 0.0 ? dot : 0.0;", "double relu = dot;"),
    "relu_after_weight": ("x += (double)w[h] * relu;",
                          "x += ((double)w[h] * dot > 0.0 ? (double)w[h] * dot : 0.0) + 0.0 * relu;"),
    "weight_dropped": ("x += (double)w[h] * relu;", "x += relu;"),
    "q_transposed": ("orc_bf16(q[(size_t)h * d + j])", "orc_bf16(q[(size_t)j * n_h + h])"),
    "k_shifted": ("* k[j];", "* k[(j + 1) % d];"),
    "threshold_strict": ("if (best >= thr)", "if (best > thr)"),
    "union_by_min": ("if (sig > best) best = sig;", "if (l == 0 || sig < best) best = sig;"),
    "sigmoid_sign": ("return 1.0 / (1.0 + exp(-x));", "return 1.0 / (1.0 + exp(x));"),
    "mask_bit_reversed": ("if (best >= thr) mask[b * words + (s >> 5)] |= 1u << (s & 31);",
                          "if (best >= thr) mask[b * words + (s >> 5)] |= 1u << (31 - (s & 31));"),
    "ensemble_mask_bit_reversed": ("if (e >= thr) mask[b * words + (s >> 5)] |= 1u << (s & 31);",
                                   "if (e >= thr) mask[b * words + (s >> 5)] |= 1u << (31 - (s & 31));"),
    "tie_higher_id_first": ("return a->id < b->id ? -1 : 1;", "return a->id > b->id ? -1 : 1;"),
    "rank_ascending": ("if (xa > xb) return -1;\n  if (xa < xb) return 1;",
                       "if (xa < xb) return -1;\n  if (xa > xb) return 1;"),
    "output_not_id_sorted": ("qsort(c, (size_t)m, sizeof(orc_cand), orc_id_cmp);", ""),
    "k_minus_one": ("int64_t m = n < k ? n : k;", "int64_t m = n < k ? n : k - 1;"),
    "pad_zero": ("idx_out[i] = i < m ? (int32_t)c[i].id : -1;", "idx_out[i] = i < m ? (int32_t)c[i].id : 0;"),
    "e4m3_bias_8": ("ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    "e4m3_subnormal_scale": ("ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)"),
    "e4m3_no_nan": ("if (e == 0xF && m == 0x7) return NAN;", ""),
    "fp8_scale_ignored": ("float kv = (float)orc_e4m3(code) * scale;", "float kv = (float)orc_e4m3(code);"),
    "fp8_dequant_in_fp64": ("float kv = (float)orc_e4m3(code) * scale;",
                            "double kv = orc_e4m3(code) * (double)scale;"),
    "paged_id_from_physical": ("int64_t chunk = lp * page_size + o;", "int64_t chunk = p * page_size + o;"),
    "paged_mask_ignored": ("        if (mrow) {\n          int64_t word", "        if (0) {\n          int64_t word"),
    "paged_mask_group_ignored": ("res_mask + (qi / mask_group) * mask_ld", "res_mask + qi * mask_ld"),
    "paged_masked_kept_at_neg_inf": ("if (!((bits >> (chunk & 31)) & 1u)) continue;",
                                     "if (!((bits >> (chunk & 31)) & 1u)) x = -INFINITY;"),
    "paged_remap_ignored": ("    if (id_mode) /* translate", "    if (0) /* translate"),
    "paged_remap_to_logical_offset": ("(int32_t)(page_phys[qi * R + j] * page_size + chunk % page_size)",
                                      "(int32_t)(page_phys[qi * R + j] * page_size)"),
    "paged_mask_past_row": ("uint32_t bits = word < mask_ld ? mrow[word] : 0u;",
                            "uint32_t bits = word < mask_ld ? mrow[word] : ~0u;"),
    "paged_bf16_pool_row_shifted": ("kbf + (size_t)row * d", "kbf + (size_t)(row ^ 1) * d"),
    "paged_nres_ignored": ("int64_t nr = n_res ? n_res[qi] : R;", "int64_t nr = R;"),
    "causal_inclusive": ("int64_t lim = pos / ratio;", "int64_t lim = pos / ratio + 1;"),
    "causal_token_not_chunk": ("int64_t lim = pos / ratio;", "int64_t lim = pos;"),
    "nan_ranks_high": ("double xa = isnan(a->x) ? -INFINITY : a->x;", "double xa = isnan(a->x) ? INFINITY : a->x;"),
    "memindex_fp8_scale_from_wrong_layer": ("const float sc = scale[b * sstride_b + l * sstride_l + s];",
                                            "const float sc = scale[b * sstride_b + s];"),
    "memindex_fp8_key_stride_swapped": ("const uint8_t* ks = k8 + b * stride_b + l * stride_l + s * d;",
                                        "const uint8_t* ks = k8 + l * stride_b + b * stride_l + s * d;"),
    "recall_keeps_empty_pages": ("if (density > 0) {", "if (density >= 0) {"),
    "recall_recent_short": ("if (s < sink || s >= S - recent) resident = 1;",
                            "if (s < sink || s > S - recent) resident = 1;"),
    "recall_sink_long": ("if (s < sink || s >= S - recent) resident = 1;",
                         "if (s <= sink || s >= S - recent) resident = 1;"),
    "recall_partial_page_overrun": ("s < (p + 1) * page_size && s < S; ++s)", "s < (p + 1) * page_size; ++s)"),
    "ensemble_sigmoid_of_mean_logit": (
        "for (int64_t l = 0; l < L; ++l) sum += orc_sigmoid(x[((size_t)b * L + l) * S + s]);\n        e = sum / (double)L;",
        "for (int64_t l = 0; l < L; ++l) sum += x[((size_t)b * L + l) * S + s];\n        e = orc_sigmoid(sum / (double)L);"),
    "ensemble_mode_ignored": ("      if (mode == 0) {\n        e = -1.0;", "      if (1) {\n        e = -1.0;"),
    "ensemble_sum_not_mean": ("e = sum / (double)L;", "e = sum;"),
    "ensemble_threshold_strict": ("if (e >= thr) mask", "if (e > thr) mask"),
    "unpack_scale_offset": ("memcpy(&scale_out[i], row + d, sizeof(float));",
                            "memcpy(&scale_out[i], row + d - 4, sizeof(float));"),
    "unpack_row_stride_d": ("const uint8_t* row = ck + (size_t)i * (size_t)(d + 4);",
                            "const uint8_t* row = ck + (size_t)i * (size_t)d;"),
    "rmsnorm_sum_not_mean": ("double inv = 1.0 / sqrt(ss / (double)n + eps);", "double inv = 1.0 / sqrt(ss + eps);"),
    "rmsnorm_eps_outside": ("double inv = 1.0 / sqrt(ss / (double)n + eps);", "double inv = 1.0 / (sqrt(ss / (double)n) + eps);"),
    "rmsnorm_gain_ignored": ("y[i] = x[i] * inv * orc_bf16(g[i]);", "y[i] = x[i] * inv;"),
    "yarn_blend_swapped": ("return (1.0 - gamma) * theta / factor + gamma * theta;",
                           "return gamma * theta / factor + (1.0 - gamma) * theta;"),
    "yarn_turns_without_2pi": ("double r = orig_len * theta / two_pi;", "double r = orig_len * theta;"),
    "yarn_exponent_per_dim": ("double theta = pow(base, -2.0 * (double)i / (double)rope_dim);",
                              "double theta = pow(base, -(double)i / (double)rope_dim);"),
    "rope_half_split_pairs": ("double x0 = xr[2 * i], x1 = xr[2 * i + 1];\n    xr[2 * i] = x0 * c - x1 * sn;\n    xr[2 * i + 1] = x0 * sn + x1 * c;",
                              "double x0 = xr[i], x1 = xr[i + rope_dim / 2];\n    xr[i] = x0 * c - x1 * sn;\n    xr[i + rope_dim / 2] = x0 * sn + x1 * c;"),
    "rope_on_first_dims": ("double* xr = x + head_dim - rope_dim;", "double* xr = x;"),
    "rope_reverse_turn": ("xr[2 * i] = x0 * c - x1 * sn;", "xr[2 * i] = x0 * c + x1 * sn;"),
    "hadamard_unnormalised": ("double norm = 1.0 / sqrt((double)n);", "double norm = 1.0;"),
    "hadamard_or_not_and": ("__builtin_popcount((unsigned)(i & j))", "__builtin_popcount((unsigned)(i | j))"),
    "chain_wq_b_transposed": ("acc += orc_bf16(wq_b[(size_t)j * r + i]) * c[i];",
                              "acc += orc_bf16(wq_b[(size_t)i * (n_h * head_dim) + j]) * c[i];"),
    "chain_weight_scale_missing": ("w_out[(size_t)t * n_h + hh] = acc * ws;", "w_out[(size_t)t * n_h + hh] = acc;"),
    "chain_hadamard_before_rope": (
        "      orc_rope_yarn(uh, head_dim, rope_dim, pos[t], base, factor, orig_len, beta_fast, beta_slow);\n      orc_hadamard(uh, head_dim, q_out + ((size_t)t * n_h + hh) * head_dim);",
        "      double* qo = q_out + ((size_t)t * n_h + hh) * head_dim;\n      orc_hadamard(uh, head_dim, qo);\n      orc_rope_yarn(qo, head_dim, rope_dim, pos[t], base, factor, orig_len, beta_fast, beta_slow);"),
    "recall_bit_reversed": ("int resident = (mask[b * words + (s >> 5)] >> (s & 31)) & 1u;",
                            "int resident = (mask[b * words + (s >> 5)] >> (31 - (s & 31))) & 1u;"),
}

RUNNER = r"""
import json, sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, pins
o = oracle.Oracle({so!r})
failed = []
for p in pins.ALL_PINS:
    try:
        p(o)
    except Exception as e:
        failed.append(p.__name__)
print(json.dumps(failed))
"""


def _run_mutant(name, old, new, tmp):
    src = open(oracle.SRC).read()
    assert src.count(old) == 1, f"mutant {name}: target occurs {src.count(old)} times"
    path = os.path.join(tmp, f"{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    so = os.path.join(tmp, f"lib{name}.so")
    oracle.compile_oracle(path, so, extra=("-w",))
    code = RUNNER.format(root=ROOT, tests=TESTS, so=so)
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600, env=env)
    if r.returncode != 0:
        return name, ["<crashed>"]
    return name, json.loads(r.stdout.strip().splitlines()[-1])


def test_every_mutant_is_caught():
    with tempfile.TemporaryDirectory() as tmp:
        with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
            results = dict(ex.map(lambda kv: _run_mutant(kv[0], *kv[1], tmp), MUTANTS.items()))
    survivors = [n for n, failed in results.items() if not failed]
    assert not survivors, f"mutants not caught by any pin: {survivors}"


def test_unmutated_copy_passes_all_pins():
    with tempfile.TemporaryDirectory() as tmp:
        name, failed = _run_mutant("identity", "ORC_API int orc_num_threads(void) {",
                                   "ORC_API int orc_num_threads(void) {", tmp)
    assert failed == [], failed
