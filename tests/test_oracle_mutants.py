"""Mutation check of the oracle's pins.

Each case plants one plausible mistake in a copy of the oracle's C source
(a dropped term, a wrong sign or index, a transposed operand, a wrong tie
rule ...), builds it on the CPU, and runs the pin tests against it: the pins
must fail for every mutant.  The real oracle is never modified.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "qsa_oracle.c")

MUTANTS = {
    "mean_drops_fourth_key": (
        "    s = s + (float)oracle_bf16_to_double(raw[3 * QSA_D + d]);\n", ""),
    "rope_wrong_sign": (
        "k[i + half] = u[i + half] * c + u[i] * s;", "k[i + half] = u[i + half] * c - u[i] * s;"),
    "rope_wrong_frequency": ("-2.0 * (double)i / (double)QSA_D", "-1.0 * (double)i / (double)QSA_D"),
    "rope_interleaved_pairs": (
        "    k[i] = u[i] * c - u[i + half] * s;\n    k[i + half] = u[i + half] * c + u[i] * s;",
        "    if (i % 2 == 0) { k[i] = u[i] * c - u[i + 1] * s; k[i + 1] = u[i + 1] * c + u[i] * s; }\n"
        "    k[i + half] = u[i + half];"),
    "no_normalisation": ("(double)m[d] / norm", "(double)m[d]"),
    "no_relu": ("acc += dot > 0.0 ? dot : 0.0;", "acc += dot;"),
    "three_heads": ("for (int h = 0; h < QSA_H; ++h) {\n    double dot",
                    "for (int h = 0; h < QSA_H - 1; ++h) {\n    double dot"),
    "q_transposed": ("oracle_bf16_to_double(q[h * QSA_D + d])", "oracle_bf16_to_double(q[d * QSA_H + h])"),
    "wrong_scale": ("return (float)(acc / sqrt((double)QSA_D));", "return (float)(acc / 8.0);"),
    "ties_to_higher_index": ("  if (a < b) return 0;\n  return ia < ib;", "  if (a < b) return 0;\n  return ia > ib;"),
    "nan_ranks_first": ("    return nb;  /* the non-NaN one ranks first */", "    return na;"),
    "output_not_ascending": (
        "  qsort(out_idx, (size_t)m, sizeof(int32_t), cmp_index);\n", ""),
    "slot_page_offset_swapped": (
        "return (int64_t)pt_row[pos / page_size] * page_size + pos % page_size;",
        "return (int64_t)pt_row[pos % page_size] * page_size + pos / page_size;"),
    "pool_row_not_divided": (
        "return oracle_slot_of(pt_row, QSA_C * b, page_size) / QSA_C;",
        "return oracle_slot_of(pt_row, b, page_size);"),
    "incomplete_block_scored": (
        "int64_t nb = row_len[t] / QSA_C;", "int64_t nb = (row_len[t] + QSA_C - 1) / QSA_C;"),
    "pending_off_by_one": (
        "for (int64_t p = (L / QSA_C) * QSA_C; p < L; ++p)",
        "for (int64_t p = (L / QSA_C) * QSA_C + 1; p <= L; ++p)"),
    "expand_block_not_times_4": (
        "out_pos[w++] = QSA_C * sel[j] + c;", "out_pos[w++] = sel[j] + c;"),
    "bf16_truncates": ("double r = nearbyint(x / q) * q;", "double r = trunc(x / q) * q;"),
    "indexshare_tail_from_cap_len": (
        "for (int64_t p = QSA_C * nb0; p < L; ++p) {", "for (int64_t p = cap_len; p < L; ++p) {"),
    "indexshare_no_causal_cut": ("      if (p >= L) continue;\n", ""),
    "indexshare_incomplete_block_kept": ("    if (b >= nb0) {\n      flags |= 2;\n      continue;\n    }\n", ""),
    "append_first_new_key_from_ring": ("const uint16_t* src = q >= p0 ? keys", "const uint16_t* src = q > p0 ? keys"),
    "append_ring_slot_by_call_index": ("memcpy(rr + ((p0 + i) % QSA_C) * QSA_D", "memcpy(rr + (i % QSA_C) * QSA_D"),
    "attn_kv_head_modulo": ("int64_t g = h / group;", "int64_t g = h % h_kv;"),
    "attn_no_max_subtraction": ("double w = exp(logit[j] - mx);", "double w = exp(logit[j]);"),
    "attn_mask_reads_slot_0": ("      if (s < 0) continue;\n      if (s >= n_slots) {",
                               "      if (s < 0) s = 0;\n      if (s >= n_slots) {"),
    "attn_nan_when_all_masked": ("out[h * d + e] = sum > 0.0 ? (float)(acc[e] / sum) : 0.0f;",
                                 "out[h * d + e] = (float)(acc[e] / sum);"),
    "attn_no_scale": ("      logit[j] = scale * dot;", "      logit[j] = dot;"),
    "rope_queries_wrong_sign": ("y[i + half] = oracle_bf16_round(v * c + u * s);",
                                "y[i + half] = oracle_bf16_round(v * c - u * s);"),
    "rope_queries_position_off_by_one": ("double theta = (double)pos[t] * inv_freq;",
                                         "double theta = (double)(pos[t] + 1) * inv_freq;"),
    "e4m3_truncates": ("double r = a == 0.0 ? 0.0 : nearbyint(a / ldexp(1.0, qexp)) * ldexp(1.0, qexp);",
                       "double r = a == 0.0 ? 0.0 : floor(a / ldexp(1.0, qexp)) * ldexp(1.0, qexp);"),
    "e4m3_no_saturation": ("  if (r > 448.0) r = 448.0;        /* saturate */\n", ""),
    "fp8_scale_wrong_range": ("const float scale = mx / 448.0f;", "const float scale = mx / 256.0f;"),
    "fp8_score_no_relu": ("total += hdot > 0.0 ? hdot : 0.0;", "total += hdot;"),
    "fp8_query_not_binary16": ("hdot += oracle_f16_round(oracle_bf16_to_double(qh[d]))",
                               "hdot += oracle_bf16_to_double(qh[d])"),
    "f16_no_subnormal_quantum": ("  if (qexp < -24) qexp = -24;\n", ""),
    "gate_before_relu": ("const double rect = hd > 0.0 ? hd : 0.0;\n    sum_w += (double)g[hg] * rect;",
                         "const double gd = (double)g[hg] * hd;\n    sum_w += gd > 0.0 ? gd : 0.0;"),
    "gate_of_the_next_head": ("sum_w += (double)g[hg] * rect;", "sum_w += (double)g[(hg + 1) % QSA_H] * rect;"),
    "gated_rows_share_row_0_gates": ("gates + t * QSA_H,", "gates,"),
    "indexshare_no_drafted_columns": (
        "int64_t width = QSA_C * k_blk + (QSA_C - 1) + n_extra;\n  int64_t nb0",
        "int64_t width = QSA_C * k_blk + (QSA_C - 1);\n  int64_t nb0"),
}


def _run_mutant(name, tmpdir):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique/found"
    mdir = os.path.join(tmpdir, name)
    os.makedirs(mdir, exist_ok=True)
    csrc = os.path.join(mdir, "m.c")
    lib = os.path.join(mdir, "libm.so")
    open(csrc, "w").write(src.replace(old, new))
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                           "-o", lib, csrc, "-lm"])
    env = dict(os.environ, QSA_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py"),
                        os.path.join(ROOT, "tests", "test_oracle_prologue.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode


def test_every_planted_mistake_fails_a_pin(tmp_path):
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
        codes = dict(zip(MUTANTS, ex.map(lambda n: _run_mutant(n, str(tmp_path)), MUTANTS)))
    survivors = [n for n, c in codes.items() if c == 0]
    assert not survivors, f"mutants not caught by the pins: {survivors}"
    # a mutant that writes outside its buffers may also crash the run (e.g.
    # pool_row_not_divided); any non-zero exit is a detection
