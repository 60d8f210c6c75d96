"""The oracle's pins catch plausible mistakes (CPU).  Each mutant below is oracle.c with one
plausible error planted in it (a dropped term, a wrong comparison, a wrong index or
constant).  The mutant is compiled into its own library, and the oracle pin suites run
against it through ORACLE_LIB.  The test requires every mutant to fail at least one pin.
The mistakes are planted in the oracle only, on the CPU; nothing here touches the CUDA path.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")
PINS = ["tests/test_oracle.py", "tests/test_oracle_samplers.py",
        "tests/test_oracle_value_sampling.py", "tests/test_oracle_held_set.py"]

# name -> [(exact text in oracle.c, replacement)]; each text must occur exactly once
MUTANTS = {
    # the method
    "scores without 1/sqrt(d)": [
        ("const double inv_sqrt_d = 1.0 / sqrt((double)d);", "const double inv_sqrt_d = 1.0;")],
    "CDF search with <= for <": [("    if (t < C[i]) return i;", "    if (t <= C[i]) return i;")],
    "inclusion probability pi = p": [
        ("      pi[count] = -expm1((double)M * log1p(-p[i]));", "      pi[count] = p[i];")],
    "GQA mixture of query head 0 only": [
        ("  for (int g = 0; g < G; ++g) {\n    const int hq = h * G + g;\n    for (int i = 0; i < n; ++i) {",
         "  for (int g = 0; g < 1; ++g) {\n    const int hq = h * G + g;\n    for (int i = 0; i < n; ++i) {"),
        ("  for (int i = 0; i < n; ++i) p[i] /= (double)G;", "")],
    "query heads strided across KV heads": [
        ("    const int hq = h * G + g;\n    for (int i = 0; i < n; ++i) {",
         "    const int hq = g * pr->num_kv_heads + h;\n    for (int i = 0; i < n; ++i) {")],
    "representative divides by T, not the valid count": [
        ("rep[k] = c > 0 ? sum / (double)c : 0.0;", "rep[k] = c > 0 ? sum / (double)T : 0.0;")],
    "draw counter words swapped": [
        ("uint64_t oracle_draw_point(uint64_t seed, int b, int h, int r, uint64_t Z) {\n"
         "  uint32_t ctr[4] = {(uint32_t)r, (uint32_t)h, (uint32_t)b, 0u};",
         "uint64_t oracle_draw_point(uint64_t seed, int b, int h, int r, uint64_t Z) {\n"
         "  uint32_t ctr[4] = {(uint32_t)h, (uint32_t)r, (uint32_t)b, 0u};")],
    "wrong Weyl constant": [("      k0 += 0x9E3779B9u;", "      k0 += 0x9E3779B7u;")],
    "unweighted denominator": [("        den[g] += w * e;", "        den[g] += e;")],
    "padded slots counted in a partial team": [
        ("  return rest < pr->team_size ? rest : pr->team_size;", "  return pr->team_size;")],
    "values read from KV head 0": [
        ("          num[g * d + k] += w * e * elem(pr->v_pool, pr->dtype, kv_index(pr, page, h, t, k));",
         "          num[g * d + k] += w * e * elem(pr->v_pool, pr->dtype, kv_index(pr, page, 0, t, k));")],
    "token scores against keys of KV head 0": [
        ("    dot += q_elem(pr, b, hq, k) * elem(pr->k_pool, pr->dtype, kv_index(pr, page, h, t, k));",
         "    dot += q_elem(pr, b, hq, k) * elem(pr->k_pool, pr->dtype, kv_index(pr, page, 0, t, k));")],
    "exclusive CDF": [
        ("    run += oracle_fixed_prob(p[i]);\n    C[i] = run;",
         "    C[i] = run;\n    run += oracle_fixed_prob(p[i]);")],
    "inclusion probability of M - 1 draws": [
        ("      pi[count] = -expm1((double)M * log1p(-p[i]));",
         "      pi[count] = -expm1((double)(M - 1) * log1p(-p[i]));")],
    "page table ignored": [
        ("  return pr->page_table[(int64_t)b * pr->max_teams + i];",
         "  return (int64_t)b * pr->max_teams + i;")],
    "weight pi instead of 1/pi": [
        ("      const double w = 1.0 / pi[c];\n      for (int t = 0; t < len; ++t) {",
         "      const double w = pi[c];\n      for (int t = 0; t < len; ++t) {")],
    "draw uniform without the 1/2": [
        ("  oracle_philox4x32_10(ctr, key, w);\n"
         "  unsigned __int128 prod = (unsigned __int128)(2ull * w[0] + 1ull) * Z;\n"
         "  return (uint64_t)(prod >> 33);\n}\n\n/* M i.i.d. draws",
         "  oracle_philox4x32_10(ctr, key, w);\n"
         "  unsigned __int128 prod = (unsigned __int128)(2ull * w[0]) * Z;\n"
         "  return (uint64_t)(prod >> 33);\n}\n\n/* M i.i.d. draws")],
    "sampled set in descending order": [
        ("  int count = 0;\n  for (int i = 0; i < n; ++i) {\n    int hit = 0;",
         "  int count = 0;\n  for (int i = n - 1; i >= 0; --i) {\n    int hit = 0;")],
    "team probabilities summed over the heads": [
        ("  for (int i = 0; i < n; ++i) p[i] /= (double)G;", "")],
    "bf16 read from the low half-word": [
        ("    uint32_t w = (uint32_t)((const uint16_t*)base)[idx] << 16;",
         "    uint32_t w = (uint32_t)((const uint16_t*)base)[idx];")],
    # the next rows
    "systematic uniform from draw 1": [
        ("  const uint64_t t_u = oracle_draw_point(seed, b, h, 0, Z);",
         "  const uint64_t t_u = oracle_draw_point(seed, b, h, 1, Z);")],
    "mixture left out of the whole step": [("  oracle_mix(q, n, alpha, q);\n", "")],
    "value rows averaged without 1/S": [
        ("token_score(pr, b, hq, h, page, j) - shift[g]) / r[j] / S;",
         "token_score(pr, b, hq, h, page, j) - shift[g]) / r[j];")],
    "systematic weight without min(1, .)": [
        ("      recip[count] = fmin(1.0, (double)M * q[i]);", "      recip[count] = (double)M * q[i];")],
    "Hansen-Hurwitz weight ignores the draw count": [
        ("      recip[count] = (double)M * q[i] / (double)c;", "      recip[count] = (double)M * q[i];")],
    "mixture adds alpha instead of alpha / n": [
        ("q[i] = (1.0 - alpha) * p[i] + alpha / (double)n;", "q[i] = (1.0 - alpha) * p[i] + alpha;")],
    "systematic points spaced 1/(M+1)": [
        ("  return (uint64_t)(num / (unsigned __int128)(uint64_t)M);",
         "  return (uint64_t)(num / (unsigned __int128)(uint64_t)(M + 1));")],
    "value-row weight without 1/r": [
        ("token_score(pr, b, hq, h, page, j) - shift[g]) / r[j] / S;",
         "token_score(pr, b, hq, h, page, j) - shift[g]) / S;")],
    "row distribution without the 1/G": [
        ("      r[t] += exp(token_score(pr, b, h * G + g, h, page, t) - m) / z / (double)G;",
         "      r[t] += exp(token_score(pr, b, h * G + g, h, page, t) - m) / z;")],
    "row-draw counter word 3 = team instead of 1 + team": [
        ("(uint32_t)b, (uint32_t)(1 + team)};", "(uint32_t)b, (uint32_t)team};")],
    "value-row denominator from the drawn rows only": [
        ("      for (int t = 0; t < len; ++t) den[g] += w * exp(token_score(pr, b, hq, h, page, t) - shift[g]);",
         "      for (int k = 0; k < S; ++k) den[g] += w * exp(token_score(pr, b, hq, h, page, idx[c * S + k]) - shift[g]) / r[idx[c * S + k]] / S;")],
}


def _mutate(src, edits):
    for old, new in edits:
        assert src.count(old) == 1, f"mutation anchor occurs {src.count(old)} times: {old[:60]!r}"
        src = src.replace(old, new)
    return src


def _run_pins(name, edits, tmp):
    tag = "".join(c if c.isalnum() else "_" for c in name)
    c_path = os.path.join(tmp, tag + ".c")
    so_path = os.path.join(tmp, tag + ".so")
    with open(SRC) as f:
        text = _mutate(f.read(), edits)
    with open(c_path, "w") as f:
        f.write(text)
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-shared",
                    "-fPIC", "-o", so_path, c_path, "-lm"], check=True, capture_output=True)
    env = dict(os.environ, ORACLE_LIB=so_path)
    r = subprocess.run([sys.executable, "-m", "pytest", *PINS, "-x", "-q", "-p", "no:cacheprovider",
                        "-m", "not gpu"], cwd=ROOT, env=env, capture_output=True, text=True)
    failed = [ln for ln in r.stdout.splitlines() if ln.startswith("FAILED")]
    return name, r.returncode, failed


def test_every_mutant_fails_a_pin(tmp_path):
    with ThreadPoolExecutor(max(1, min(8, os.cpu_count() or 1))) as ex:
        results = list(ex.map(lambda kv: _run_pins(kv[0], kv[1], str(tmp_path)), MUTANTS.items()))
    survivors = [name for name, rc, _ in results if rc != 1]
    assert not survivors, f"mutants no pin caught (or that broke collection): {survivors}"


def test_anchors_are_unique():
    with open(SRC) as f:
        src = f.read()
    for name, edits in MUTANTS.items():
        _mutate(src, edits)
