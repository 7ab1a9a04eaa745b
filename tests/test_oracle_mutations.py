"""Plant plausible mistakes in copies of the oracle source and check that the
pins catch every one.  The mistakes live only in temporary copies on the CPU;
the real oracle is untouched.  CPU only."""
import os
import shutil
import subprocess

import pytest

import oracle
import oracle_pins as P

MUTANTS = [
    ("accept ratio inverted", "ratio = p / q;", "ratio = q / p;"),
    ("residual sign flipped", "double r = w_out[v] - q[v];", "double r = q[v] - w_out[v];"),
    ("accept test not strict", "(double)u_accept[di] < ratio", "(double)u_accept[di] <= ratio"),
    ("target rows lose the per-request bonus offset",
     "return (int64_t)cu[i] + i + j;", "return (int64_t)cu[i] + j;"),
    ("argmax ties go to the highest index", "if (l > best) {", "if (l >= best) {"),
    ("temperature multiplies instead of divides", "s += exp((l - m) / T);",
     "s += exp((l - m) * T);"),
    ("inverse CDF boundary not strict", "if (C > target)", "if (C >= target)"),
    ("D-cut ties prefer the higher request", "return a->i < b->i ? -1 : 1;",
     "return a->i > b->i ? -1 : 1;"),
    ("D-cut ignores min_gain", "int64_t keep = eligible < budget ? eligible : budget;",
     "int64_t keep = budget < n ? budget : n;"),
    ("last rejection instead of first", "if (!accept && a == k)", "if (!accept)"),
    ("residual fallback removed", "if (any) {", "if (1) {"),
    ("D-cut prefix product off by one",
     "P = P * conf[(int64_t)i * Kmax + (d - 1)];\n            cand[c].P = P;",
     "cand[c].P = P;\n            P = P * conf[(int64_t)i * Kmax + (d - 1)];"),
    ("q read from the target row",
     "err = softmax_at(draft, dtype, di, V, T, x, &q);",
     "err = softmax_at(target, dtype, target_row(cu, i, j), V, T, x, &q);"),
    ("final draw from the previous target row",
     "err = oracle_final_weights(target, draft, dtype, V, T, target_row(cu, i, a), drow,",
     "err = oracle_final_weights(target, draft, dtype, V, T, target_row(cu, i, a > 0 ? a - 1 : a), drow,"),
    ("greedy compares every draft against row 0",
     "while (a < k && tokens[draft_index(cu, i, a, draft_stride)] == g[a])",
     "while (a < k && tokens[draft_index(cu, i, a, draft_stride)] == g[0])"),
    ("greedy final token from the row before the mismatch", "y = g[a];",
     "y = g[a > 0 ? a - 1 : 0];"),
    ("padded draft stride ignored",
     "return draft_stride > 0 ? (int64_t)i * draft_stride + j : (int64_t)cu[i] + j;",
     "return (int64_t)cu[i] + j;"),
    ("softmax numerator drops the max shift",
     "p_out[v] = exp((logit_at(logits, dtype, row, V, v) - m) / T) / s;",
     "p_out[v] = exp(logit_at(logits, dtype, row, V, v) / T) / s;"),
    ("inverse CDF forgets to scale u by S", "double target = u * S;", "double target = u;"),
    ("cost table interpolates from the wrong end",
     "table[d] = cost_value[seg] + rise * frac;", "table[d] = cost_value[seg + 1] - rise * frac;"),
    ("cost variant stops at the first request that does not fit",
     "if (total + c <= max_cost) {", "if (total + c > max_cost) break; {"),
    ("cost variant benefit forgets the depth factor",
     "double b = P * (double)d / oracle_dcut_cost(d);", "double b = P / oracle_dcut_cost(d);"),
    ("confidence reads the wrong row", "err = softmax_at(draft, dtype, r, V, T, x, &c);",
     "err = softmax_at(draft, dtype, r > 0 ? r - 1 : r, V, T, x, &c);"),
    ("greedy confidence ignores the argmax", "c = (err == ORC_OK && g == x) ? 1.0 : 0.0;",
     "c = 1.0;"),
    ("draft sample reads the next row", "err = oracle_softmax_row(draft, dtype, r, V, T, w);",
     "err = oracle_softmax_row(draft, dtype, r + 1 < (int64_t)B * Kmax ? r + 1 : r, V, T, w);"),
    ("draft sample conf of the wrong entry", "out_conf[r] = (float)w[x];",
     "out_conf[r] = (float)w[x > 0 ? x - 1 : x];"),
    ("acceptance counts an untested position", "            if (a >= j)\n                out_reached[j] += 1;",
     "            if (a >= j - 1)\n                out_reached[j] += 1;"),
    ("acceptance mean over every request", "    *out_mean = n > 0 ? (double)total / (double)n : 0.0;",
     "    *out_mean = B > 0 ? (double)total / (double)B : 0.0;"),
    ("cost variant keeps the last maximising depth", "if (b > best) { /* strict",
     "if (b >= best) { /* strict"),
    ("an underflowed q accepts even when p is 0", "ratio = p > 0 ? INFINITY : 0.0;",
     "ratio = INFINITY;"),
    ("expected length counts one depth too many",
     "            for (int32_t d = 1; d <= out_depth[i]; ++d) {\n                P = P * conf",
     "            for (int32_t d = 1; d <= out_depth[i] + (out_depth[i] < Kmax); ++d) {\n                P = P * conf"),
    ("cost table clamps long depths to the shortest cost", "        table[d] = cost_value[4];",
     "        table[d] = cost_value[0];"),
    ("acceptance counts the first rejection as accepted", "            if (a > j)\n                out_accepted[j] += 1;",
     "            if (a >= j)\n                out_accepted[j] += 1;"),
    ("D-cut keeps only products strictly above min_gain", "            if (P >= min_gain)",
     "            if (P > min_gain)"),
    ("cost variant sorts ascending",
     "if (a->benefit > b->benefit)\n        return -1;\n    if (a->benefit < b->benefit)\n        return 1;",
     "if (a->benefit < b->benefit)\n        return -1;\n    if (a->benefit > b->benefit)\n        return 1;"),
    ("final CDF exclusive instead of inclusive",
     "        C += cdf_out[v];\n        cdf_out[v] = C;",
     "        const double w_v = cdf_out[v];\n        cdf_out[v] = C;\n        C += w_v;"),
    ("final CDF at a = K reads the next draft row",
     "    int64_t drow = a < k ? draft_index(cu, i, a, draft_stride) : -1;\n    int st = oracle_final_weights",
     "    int64_t drow = a <= k ? draft_index(cu, i, a, draft_stride) : -1;\n    int st = oracle_final_weights"),
    ("final CDF from the previous target row",
     "    int st = oracle_final_weights(target, draft, dtype, V, T, target_row(cu, i, a), drow,\n                                  cdf_out, NULL);",
     "    int st = oracle_final_weights(target, draft, dtype, V, T, target_row(cu, i, a > 0 ? a - 1 : a), drow,\n                                  cdf_out, NULL);"),
    ("diagnostic S of p instead of the weights", "out_final[4 * (int64_t)i + 1] = S;",
     "out_final[4 * (int64_t)i + 1] = 1.0;"),
    ("diagnostic C(y-1) stops one weight short", "for (int64_t t = 0; t < v; ++t)",
     "for (int64_t t = 0; t + 1 < v; ++t)"),
    ("diagnostic u*S without S", "*uS_out = u * S;", "*uS_out = u;"),
]


def _pins_in_cost_order():
    cheap = [p for p in P.ALL_PINS if p is not P.pin_lossless_chi_square]

    def chi(lib):
        P.pin_lossless_chi_square(lib, n=200_000, batch=200_000)
    return cheap + [chi]


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    d = tmp_path_factory.mktemp("oracle_mutants")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(mutant_dir, name, old, new):
    src = open(oracle.SRC).read()
    assert src.count(old) >= 1, f"mutation site for '{name}' not found in oracle.c"
    mutated = src.replace(old, new)
    tag = "".join(c if c.isalnum() else "_" for c in name)
    c_path = os.path.join(mutant_dir, f"{tag}.c")
    so_path = os.path.join(mutant_dir, f"lib{tag}.so")
    with open(c_path, "w") as f:
        f.write(mutated)
    subprocess.run(["gcc", *oracle.CFLAGS, "-w", "-o", so_path, c_path, "-lm"], check=True)
    lib = oracle.load(so_path)
    for pin in _pins_in_cost_order():
        try:
            pin(lib)
        except AssertionError:
            return  # caught
    pytest.fail(f"no pin caught the planted mistake '{name}'")


def test_unmutated_copy_passes(mutant_dir):
    """The harness itself: an unmodified copy passes every pin."""
    c_path = os.path.join(mutant_dir, "clean.c")
    so_path = os.path.join(mutant_dir, "libclean.so")
    shutil.copy(oracle.SRC, c_path)
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", so_path, c_path, "-lm"], check=True)
    lib = oracle.load(so_path)
    for pin in _pins_in_cost_order():
        pin(lib)
