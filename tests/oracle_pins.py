"""Pins of the CPU oracle against what the mathematics and the pages fix.

Each ``pin_*`` function takes a loaded oracle library (ctypes CDLL) and raises
AssertionError on a mismatch.  test_oracle_pins.py runs them against the real
oracle; test_oracle_mutations.py runs them against deliberately broken copies
of the oracle source, to show that a plausible mistake fails at least one pin.

Nothing here calls the oracle to produce its own expected values: expected
values are closed forms, library routines (numpy / scipy), brute force written
here, hand-worked fixtures under tests/golden/, or statistical laws.
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
from scipy import special, stats

import oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16 bit patterns (for values exactly
    representable in bf16 this is just the upper half of the word)."""
    f = np.ascontiguousarray(np.asarray(x, np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def _ref_softmax(l, T):
    """Library softmax in fp64 (scipy)."""
    return special.softmax(np.asarray(l, np.float64) / T)


# ---------------------------------------------------------------------------
# softmax with temperature
# ---------------------------------------------------------------------------


def pin_softmax_closed_form_v2(lib):
    """V = 2: p(0) = 1 / (1 + exp((l1 - l0) / T)) (the logistic function)."""
    for l0, l1, T in [(0.0, 1.0, 1.0), (2.5, -1.25, 0.7), (-3.0, 4.0, 2.0),
                      (1.0, 1.0, 0.3), (10.0, -10.0, 1.0)]:
        row = np.array([[l0, l1]], np.float32)
        st, p = O.softmax_row(row, 0, T, lib=lib)
        assert st == O.OK
        e = 1.0 / (1.0 + math.exp((float(np.float32(l1)) - float(np.float32(l0))) / T))
        assert abs(p[0] - e) <= 1e-14 * max(e, 1e-300), (l0, l1, T, p, e)
        assert abs(p[1] - (1 - e)) <= 1e-13, (l0, l1, T, p, e)


def pin_softmax_matches_library(lib):
    """Random rows against scipy.special.softmax in fp64, f32 and bf16 inputs."""
    rng = np.random.default_rng(1)
    for V, T in [(7, 1.0), (1024, 0.7), (333, 1.7)]:
        l = (rng.standard_normal((3, V)) * 3).astype(np.float32)
        for r in range(3):
            st, p = O.softmax_row(l, r, T, lib=lib)
            assert st == O.OK
            np.testing.assert_allclose(p, _ref_softmax(l[r], T), rtol=1e-12, atol=0)
        bits = _to_bf16_bits(l)
        exact = (bits.astype(np.uint32) << 16).view(np.float32)
        for r in range(3):
            st, p = O.softmax_row(bits, r, T, lib=lib)
            assert st == O.OK
            np.testing.assert_allclose(p, _ref_softmax(exact[r], T), rtol=1e-12, atol=0)


def pin_softmax_invariances(lib):
    """Shift invariance, p_T(l) = p_1(l / T), sum to one, masked entries."""
    rng = np.random.default_rng(2)
    V = 257
    grid = rng.integers(-256, 256, size=V) / 64.0  # exact in fp32 and after +/-3 or /0.5
    base = grid.astype(np.float32)[None, :]
    shifted = (grid + 3.0).astype(np.float32)[None, :]
    _, p0 = O.softmax_row(base, 0, 1.0, lib=lib)
    _, p1 = O.softmax_row(shifted, 0, 1.0, lib=lib)
    np.testing.assert_allclose(p0, p1, rtol=1e-14, atol=0)
    assert abs(p0.sum() - 1.0) < 1e-12
    _, pT = O.softmax_row(base, 0, 0.5, lib=lib)
    scaled = (grid / 0.5).astype(np.float32)[None, :]
    _, pS = O.softmax_row(scaled, 0, 1.0, lib=lib)
    np.testing.assert_allclose(pT, pS, rtol=1e-14, atol=0)
    masked = base.copy()
    masked[0, ::3] = -np.inf
    st, pm = O.softmax_row(masked, 0, 1.0, lib=lib)
    assert st == O.OK and np.all(pm[::3] == 0.0)
    np.testing.assert_allclose(pm, _ref_softmax(masked[0], 1.0), rtol=1e-12)


def pin_softmax_errors(lib):
    """NaN, +inf and an all-masked row are errors; T <= 0 is an argument error."""
    for bad in (np.nan, np.inf):
        row = np.zeros((1, 5), np.float32)
        row[0, 2] = bad
        assert O.softmax_row(row, 0, 1.0, lib=lib)[0] == O.ERR_NONFINITE
    row = np.full((1, 5), -np.inf, np.float32)
    assert O.softmax_row(row, 0, 1.0, lib=lib)[0] == O.ERR_NONFINITE
    assert O.softmax_row(np.zeros((1, 5), np.float32), 0, 0.0, lib=lib)[0] == O.ERR_INVALID_ARG


# ---------------------------------------------------------------------------
# argmax and inverse CDF
# ---------------------------------------------------------------------------


def pin_argmax(lib):
    """numpy.argmax (first occurrence) on rows with planted ties, f32 and bf16."""
    rng = np.random.default_rng(3)
    l = rng.integers(-20, 20, size=(40, 129)).astype(np.float32)  # many ties
    for r in range(l.shape[0]):
        st, a = O.argmax_row(l, r, lib=lib)
        assert st == O.OK and a == int(np.argmax(l[r])), (r, a)
    bits = _to_bf16_bits(l)
    for r in range(l.shape[0]):
        st, a = O.argmax_row(bits, r, lib=lib)
        assert st == O.OK and a == int(np.argmax(l[r]))
    row = np.full((1, 6), -np.inf, np.float32)
    row[0, 4] = -1.0
    assert O.argmax_row(row, 0, lib=lib) == (O.OK, 4)
    row[0, 4] = np.nan
    assert O.argmax_row(row, 0, lib=lib)[0] == O.ERR_NONFINITE


def pin_inverse_cdf(lib):
    """Smallest v with C(v) > u*S equals searchsorted(cumsum, u*S, 'right')."""
    rng = np.random.default_rng(4)
    for _ in range(200):
        V = int(rng.integers(1, 50))
        w = rng.random(V)
        w[rng.random(V) < 0.3] = 0.0
        if w.sum() == 0:
            w[-1] = 0.5
        u = float(rng.random())
        v, uS, S = O.inverse_cdf(w, u, lib=lib)
        C = np.cumsum(w)
        assert v == int(np.searchsorted(C, u * C[-1], side="right")), (w, u, v)
        assert w[v] > 0
    w = np.array([0.0, 0.0, 0.3, 0.0, 0.7, 0.0])
    assert O.inverse_cdf(w, 0.0, lib=lib)[0] == 2           # u -> 0: first w > 0
    assert O.inverse_cdf(w, np.nextafter(1.0, 0.0), lib=lib)[0] == 4  # u -> 1: last w > 0
    assert O.inverse_cdf(w, 0.3, lib=lib)[0] == 4           # C(2) = 0.3 is not > 0.3
    assert O.inverse_cdf(np.zeros(4), 0.5, lib=lib)[0] == -1


# ---------------------------------------------------------------------------
# greedy verification
# ---------------------------------------------------------------------------


def _brute_greedy(target, tokens, k):
    """Greedy verification written out with Python loops (lowest-index argmax)."""
    out_tok, out_len = [], []
    row = 0
    d = 0
    for ki in k:
        rows = target[row: row + ki + 1]
        drafts = tokens[d: d + ki]
        g = []
        for r in rows:
            best, arg = -math.inf, -1
            for v, x in enumerate(r):
                if x > best:
                    best, arg = x, v
            g.append(arg)
        a = 0
        while a < ki and drafts[a] == g[a]:
            a += 1
        emitted = list(drafts[:a]) + [g[a]] + [-1] * (ki - a)
        out_tok += emitted
        out_len.append(a)
        row += ki + 1
        d += ki
    return np.array(out_tok, np.int32), np.array(out_len, np.int32)


def pin_greedy_golden(lib):
    g = _golden("greedy_layout.json")
    V = g["V"]
    target = np.zeros((len(g["target_peaks"]), V), np.float32)
    for r, peaks in enumerate(g["target_peaks"]):
        target[r, peaks] = 5.0
    k = np.array(g["k"], np.int32)
    cu = np.concatenate([[0], np.cumsum(k)]).astype(np.int32)
    res = O.verify_greedy(target, np.array(g["draft_tokens"], np.int32), cu, lib=lib)
    assert res.status == O.OK
    assert res.accept_len.tolist() == g["expected_accept_len"], res.accept_len
    assert res.tokens.tolist() == g["expected_tokens"], res.tokens
    # the sampling entry at T = 0 is the greedy verification
    r2 = O.verify_sample(target, None, np.array(g["draft_tokens"], np.int32), cu, 0.0,
                         np.zeros(6, np.float32), np.zeros(4, np.float32), lib=lib)
    assert r2.tokens.tolist() == g["expected_tokens"]


def pin_greedy_brute_force(lib):
    rng = np.random.default_rng(5)
    for trial in range(30):
        B = int(rng.integers(1, 6))
        V = int(rng.integers(2, 9))
        k = rng.integers(0, 5, size=B).astype(np.int32)
        cu = np.concatenate([[0], np.cumsum(k)]).astype(np.int32)
        target = rng.integers(-3, 3, size=(int(k.sum()) + B, V)).astype(np.float32)
        # drafts mostly equal to the target argmax so long prefixes occur
        g = np.argmax(target, axis=1)
        tokens = []
        row = 0
        for ki in k:
            for j in range(ki):
                tokens.append(int(g[row + j]) if rng.random() < 0.8 else int(rng.integers(0, V)))
            row += ki + 1
        tokens = np.array(tokens, np.int32)
        res = O.verify_greedy(target, tokens, cu, lib=lib)
        et, el = _brute_greedy(target.tolist(), tokens.tolist(), k.tolist())
        assert res.status == O.OK
        assert np.array_equal(res.tokens, et), (trial, res.tokens, et)
        assert np.array_equal(res.accept_len, el), (trial, res.accept_len, el)


def pin_greedy_padded_layout(lib):
    """Padded draft side: request i's drafts at i*stride + j give the same result."""
    rng = np.random.default_rng(6)
    B, V, stride = 4, 6, 5
    k = np.array([3, 0, 5, 2], np.int32)
    cu = np.concatenate([[0], np.cumsum(k)]).astype(np.int32)
    target = rng.integers(-3, 3, size=(int(k.sum()) + B, V)).astype(np.float32)
    packed = rng.integers(0, V, size=int(k.sum())).astype(np.int32)
    padded = np.full(B * stride, 99, np.int32)  # 99: out of range, must never be read
    for i in range(B):
        padded[i * stride: i * stride + k[i]] = packed[cu[i]: cu[i + 1]]
    a = O.verify_greedy(target, packed, cu, lib=lib)
    b = O.verify_greedy(target, padded, cu, draft_stride=stride, lib=lib)
    assert a.status == O.OK and b.status == O.OK
    assert np.array_equal(a.tokens, b.tokens) and np.array_equal(a.accept_len, b.accept_len)


def pin_greedy_errors(lib):
    target = np.zeros((3, 4), np.float32)
    target[:, 1] = 1.0
    cu = np.array([0, 1, 1], np.int32)
    res = O.verify_greedy(target, np.array([7], np.int32), cu, lib=lib)  # token >= V
    assert res.status == O.ERR_INVALID_ARG and res.accept_len.tolist() == [-1, 0]
    assert res.tokens.tolist() == [-1, -1, 1]
    bad = target.copy()
    bad[2, 0] = np.nan
    res = O.verify_greedy(bad, np.array([1], np.int32), cu, lib=lib)
    assert res.status == O.ERR_NONFINITE and res.accept_len.tolist() == [1, -1]
    res = O.verify_greedy(target, np.array([1], np.int32), np.array([1, 1, 1], np.int32),
                          lib=lib)
    assert res.status == O.ERR_INVALID_ARG
    # a NaN past the first mismatch is still an error (every row is read)
    t4 = target.copy()
    t4[1, 3] = np.nan
    res = O.verify_greedy(t4, np.array([0], np.int32), cu, lib=lib)  # mismatch at 0
    assert res.status == O.ERR_NONFINITE and res.accept_len.tolist() == [-1, 0]


# ---------------------------------------------------------------------------
# sampling verification
# ---------------------------------------------------------------------------


def _batch_rows(case, L):
    def val(x):
        if x == "L":
            return L
        if x == "-inf":
            return -np.inf
        return float(x)
    t = np.array([[val(x) for x in r] for r in case["target"]], np.float32)
    d = np.array([[val(x) for x in r] for r in case["draft"]], np.float32)
    return t, d


def pin_sample_golden(lib):
    g = _golden("sample_v2.json")
    for case in g["cases"]:
        t, d = _batch_rows(case, g["L"])
        k = case["k"]
        cu = np.array([0, k], np.int32)
        res = O.verify_sample(t, d, np.array(case["tokens"], np.int32), cu, g["temperature"],
                              np.array(case["u_accept"], np.float32),
                              np.array([case["u_final"]], np.float32), lib=lib)
        assert res.status == O.OK, case["name"]
        assert res.accept_len.tolist() == [case["expected_accept_len"]], (case["name"], res)
        assert res.tokens.tolist() == case["expected_tokens"], (case["name"], res.tokens)
        np.testing.assert_allclose(res.p, case["expected_p"], rtol=1e-6, atol=1e-12)
        np.testing.assert_allclose(res.q, case["expected_q"], rtol=1e-6, atol=1e-12)


def _replicated(p_logits, q_logits, n, rng, T):
    """n requests with identical target rows (K+1) and draft rows (K); drafted
    tokens drawn from q_j = softmax(draft row j / T) with numpy."""
    K = len(q_logits)
    V = len(p_logits[0])
    target = np.tile(np.asarray(p_logits, np.float32), (n, 1))
    draft = np.tile(np.asarray(q_logits, np.float32), (n, 1))
    toks = np.empty((n, K), np.int32)
    for j in range(K):
        q = _ref_softmax(np.asarray(q_logits[j], np.float32), T)
        toks[:, j] = rng.choice(V, size=n, p=q / q.sum())
    cu = (np.arange(n + 1) * K).astype(np.int32)
    ua = rng.random(n * K).astype(np.float32)
    uf = rng.random(n).astype(np.float32)
    return target, draft, toks.reshape(-1), cu, ua, uf


def _chi2_ok(counts, probs, alpha=1e-3):
    n = counts.sum()
    exp = probs * n
    keep = exp >= 5
    c = np.append(counts[keep], counts[~keep].sum())
    e = np.append(exp[keep], exp[~keep].sum())
    if e[-1] < 5:  # fold a small remainder into the largest bin
        j = int(np.argmax(e[:-1]))
        c[j] += c[-1]
        e[j] += e[-1]
        c, e = c[:-1], e[:-1]
    chi2 = float(((c - e) ** 2 / e).sum())
    dof = len(c) - 1
    return stats.chi2.sf(chi2, dof) > alpha, chi2, dof


PAIRS = {
    # name: (target logits rows 0..2, draft logits rows 0..1)
    "random": ([[0.3, -1.2, 2.0, 0.0, 1.1, -0.4, 0.7, -2.0],
                [1.5, 0.2, -0.3, 0.9, -1.0, 0.4, 0.0, 0.6],
                [-0.5, 0.8, 0.1, 1.7, -0.2, 0.3, -1.1, 0.9]],
               [[1.0, 0.4, 0.5, -0.6, 1.9, 0.1, -0.3, -0.8],
                [0.2, 1.4, -0.9, 0.0, 0.5, 1.2, -0.4, 0.3]]),
    "disjointish": ([[3.0, 2.5, 2.0, 0.0, -1.0, -1.0, -2.0, -2.0],
                     [-2.0, -1.0, 0.0, 1.0, 2.0, 3.0, 0.5, 0.0],
                     [0.0, 0.0, 1.0, 1.0, 2.0, 2.0, 0.5, 0.5]],
                    [[-2.0, -2.0, -1.0, 0.0, 1.0, 2.0, 2.5, 3.0],
                     [3.0, 2.0, 1.0, 0.0, -1.0, -2.0, 0.0, 0.5]]),
    "onehot_q": ([[0.5, 0.0, 1.0, -0.5, 0.2, 0.8, -1.0, 0.3],
                  [0.0, 1.0, 0.0, 1.0, 0.0, 1.0, 0.0, 1.0],
                  [1.2, -0.3, 0.4, 0.0, 0.9, -0.7, 0.1, 0.6]],
                 [[-np.inf, -np.inf, 0.0, -np.inf, -np.inf, -np.inf, -np.inf, -np.inf],
                  [-np.inf, 0.0, -np.inf, -np.inf, -np.inf, -np.inf, -np.inf, -np.inf]]),
}


def pin_lossless_chi_square(lib, n=1_000_000, temperatures=(0.7, 1.0), pairs=None,
                            seed=7, batch=250_000):
    """Emitted tokens follow the target law: position 0 ~ p_0; position 1 given
    position 0 accepted ~ p_1; the bonus token given both accepted ~ p_2.
    Pearson chi-square, alpha = 1e-3 per check."""
    rng = np.random.default_rng(seed)
    for name in (pairs or PAIRS):
        p_rows, q_rows = PAIRS[name]
        for T in temperatures:
            V = len(p_rows[0])
            c0 = np.zeros(V, np.int64)
            c1 = np.zeros(V, np.int64)
            c2 = np.zeros(V, np.int64)
            acc0 = 0
            done = 0
            while done < n:
                m = min(batch, n - done)
                t, d, tok, cu, ua, uf = _replicated(p_rows, q_rows, m, rng, T)
                res = O.verify_sample(t, d, tok, cu, T, ua, uf, lib=lib)
                assert res.status == O.OK
                toks = res.tokens.reshape(m, 3)
                a = res.accept_len
                c0 += np.bincount(toks[:, 0], minlength=V)
                c1 += np.bincount(toks[a >= 1, 1], minlength=V)
                c2 += np.bincount(toks[a == 2, 2], minlength=V)
                acc0 += int((a >= 1).sum())
                done += m
            for j, c in enumerate((c0, c1, c2)):
                if c.sum() < 1000:
                    continue
                p = _ref_softmax(np.asarray(p_rows[j], np.float32), T)
                ok, chi2, dof = _chi2_ok(c, p)
                assert ok, (name, T, j, chi2, dof, c.tolist())
            # acceptance probability at position 0 = sum_v min(p, q) = 1 - TV(p, q)
            p0 = _ref_softmax(np.asarray(p_rows[0], np.float32), T)
            q0 = _ref_softmax(np.asarray(q_rows[0], np.float32), T)
            alpha = float(np.minimum(p0, q0).sum())
            sd = math.sqrt(max(alpha * (1 - alpha), 1e-12) / n)
            assert abs(acc0 / n - alpha) < 5 * sd + 1e-12, (name, T, acc0 / n, alpha)


def pin_q_equals_p_accepts_all(lib):
    """q = p: the ratio is exactly 1, so every u < 1 accepts and a = K."""
    rng = np.random.default_rng(8)
    n, K, V = 2000, 3, 16
    rows = (rng.standard_normal((K + 1, V)) * 2).astype(np.float32)
    t = np.tile(rows, (n, 1))
    d = np.tile(rows[:K], (n, 1))
    tok = rng.integers(0, V, size=n * K).astype(np.int32)
    cu = (np.arange(n + 1) * K).astype(np.int32)
    ua = rng.random(n * K).astype(np.float32)
    ua[:50] = np.nextafter(np.float32(1), np.float32(0))
    res = O.verify_sample(t, d, tok, cu, 0.9, ua, rng.random(n).astype(np.float32), lib=lib)
    assert res.status == O.OK and np.all(res.accept_len == K)
    np.testing.assert_array_equal(res.p, res.q)


def pin_residual_closed_forms(lib):
    """q one-hot at x: the residual is p with x removed.  Identical rows: the
    residual is all zero and the draw falls back to p."""
    rng = np.random.default_rng(9)
    V = 10
    t = (rng.standard_normal((1, V)) * 1.5).astype(np.float32)
    d = np.full((1, V), -np.inf, np.float32)
    x = 4
    d[0, x] = 0.0
    st, w, fb = O.final_weights(t, d, 0, 0, 1.3, lib=lib)
    assert st == O.OK and fb == 0
    p = _ref_softmax(t[0], 1.3)
    e = p.copy()
    e[x] = 0.0
    np.testing.assert_allclose(w, e, rtol=1e-12, atol=1e-300)
    st, w, fb = O.final_weights(t, t, 0, 0, 1.3, lib=lib)
    assert st == O.OK and fb == 1
    np.testing.assert_allclose(w, p, rtol=1e-12)
    # general pair: w = max(0, p - q) from library softmaxes
    d2 = (rng.standard_normal((1, V))).astype(np.float32)
    st, w, fb = O.final_weights(t, d2, 0, 0, 0.8, lib=lib)
    e = np.maximum(0.0, _ref_softmax(t[0], 0.8) - _ref_softmax(d2[0], 0.8))
    np.testing.assert_allclose(w, e, rtol=1e-10, atol=1e-15)
    # bonus row (no draft row): w = p
    st, w, fb = O.final_weights(t, None, 0, -1, 0.8, lib=lib)
    np.testing.assert_allclose(w, _ref_softmax(t[0], 0.8), rtol=1e-12)


def pin_sample_outputs_layout(lib):
    """p_j, q_j of every drafted position (also after the first rejection),
    packed vs padded draft side, ragged depths including 0."""
    rng = np.random.default_rng(10)
    B, V, stride = 5, 12, 6
    k = np.array([2, 0, 6, 1, 3], np.int32)
    cu = np.concatenate([[0], np.cumsum(k)]).astype(np.int32)
    T = 0.8
    t = (rng.standard_normal((int(k.sum()) + B, V)) * 2).astype(np.float32)
    dp = (rng.standard_normal((int(k.sum()), V)) * 2).astype(np.float32)
    tok = rng.integers(0, V, size=int(k.sum())).astype(np.int32)
    ua = rng.random(int(k.sum())).astype(np.float32)
    uf = rng.random(B).astype(np.float32)
    res = O.verify_sample(t, dp, tok, cu, T, ua, uf, lib=lib)
    assert res.status == O.OK
    for i in range(B):
        for j in range(k[i]):
            di = cu[i] + j
            p = _ref_softmax(t[cu[i] + i + j], T)[tok[di]]
            q = _ref_softmax(dp[di], T)[tok[di]]
            assert abs(res.p[di] - p) <= 1e-6 * p and abs(res.q[di] - q) <= 1e-6 * q
            assert abs(res.ratio[di] - p / q) <= 1e-12 * (p / q)
        a = res.accept_len[i]
        assert 0 <= a <= k[i]
        acc = [ua[cu[i] + j] < res.ratio[cu[i] + j] for j in range(k[i])]
        assert a == (acc.index(False) if False in acc else k[i])
        row = res.tokens[cu[i] + i: cu[i] + i + k[i] + 1]
        assert row[:a].tolist() == tok[cu[i]: cu[i] + a].tolist()
        assert row[a] >= 0 and all(x == -1 for x in row[a + 1:])
    dpad = np.zeros((B * stride, V), np.float32)
    tpad = np.full(B * stride, 0, np.int32)
    upad = np.zeros(B * stride, np.float32)
    for i in range(B):
        dpad[i * stride: i * stride + k[i]] = dp[cu[i]: cu[i + 1]]
        tpad[i * stride: i * stride + k[i]] = tok[cu[i]: cu[i + 1]]
        upad[i * stride: i * stride + k[i]] = ua[cu[i]: cu[i + 1]]
    r2 = O.verify_sample(t, dpad, tpad, cu, T, upad, uf, draft_stride=stride, lib=lib)
    assert np.array_equal(r2.tokens, res.tokens) and np.array_equal(r2.accept_len,
                                                                     res.accept_len)


def _ref_final_weights(t_row, d_row, T):
    """Final-draw weights from library softmaxes: max(0, p - q) after a
    rejection (p when that is all zero), p alone for the bonus row."""
    p = _ref_softmax(t_row, T)
    if d_row is None:
        return p
    w = np.maximum(0.0, p - _ref_softmax(d_row, T))
    return w if w.sum() > 0 else p


def pin_final_cdf_and_diagnostics(lib):
    """The final draw's running sum C and the per-request diagnostic
    {u*S, S, C(y-1), C(y)} (which decide the GPU parity exemption) against a
    numpy cumsum of weights built from scipy softmaxes: every accepted length
    a = 0..K of every request (a < K residual rows, a = K the bonus row, no
    draft row), identical rows (all-zero residual, p fallback), packed and
    padded draft sides."""
    rng = np.random.default_rng(21)
    B, V, T, stride = 5, 37, 0.9, 4
    k = np.array([3, 0, 4, 1, 2], np.int32)
    cu = np.concatenate([[0], np.cumsum(k)]).astype(np.int32)
    nd = int(k.sum())
    t = (rng.standard_normal((nd + B, V)) * 1.7).astype(np.float32)
    d = (t[np.concatenate([np.arange(cu[i] + i, cu[i] + i + k[i]) for i in range(B)])]
         + rng.standard_normal((nd, V)).astype(np.float32) * 0.8).astype(np.float32)
    d[cu[4] + 1] = t[cu[4] + 4 + 1]  # request 4, position 1: q = p (all-zero residual)
    tok = rng.integers(0, V, size=nd).astype(np.int32)
    dpad = np.zeros((B * stride, V), np.float32)
    for i in range(B):
        dpad[i * stride: i * stride + k[i]] = d[cu[i]: cu[i + 1]]
    for draft, dstride in ((d, 0), (dpad, stride)):
        for i in range(B):
            for a in range(k[i] + 1):
                drow = None
                if a < k[i]:
                    drow = draft[i * dstride + a] if dstride else draft[cu[i] + a]
                st, C = O.final_cdf(t, draft, cu, i, a, T, draft_stride=dstride, lib=lib)
                assert st == O.OK, (i, a, st)
                e = np.cumsum(_ref_final_weights(t[cu[i] + i + a], drow, T))
                np.testing.assert_allclose(C, e, rtol=1e-11, atol=1e-15,
                                           err_msg=f"request {i}, a={a}, stride {dstride}")
            st, _ = O.final_cdf(t, draft, cu, i, k[i] + 1, T, draft_stride=dstride, lib=lib)
            assert st == O.ERR_INVALID_ARG
    # the diagnostic of a verification call: u*S, S, C(y-1), C(y) around the
    # drawn y, with C(y-1) <= u*S < C(y); request 2 accepts every draft (u = 0
    # with identical rows), so its draw is from the bonus row
    # requests 0, 3 and 4 reject at a chosen position: the drafter puts +6 on
    # its drafted token there, so q(x) >> p(x), and u = 0.5 rejects
    d2 = d.copy()
    d2[cu[2]: cu[3]] = t[cu[2] + 2: cu[2] + 2 + k[2]]
    ua = rng.random(nd).astype(np.float32)
    ua[cu[2]: cu[3]] = 0.0
    want = {0: 1, 3: 0, 4: 0}
    for i, j in want.items():
        ua[cu[i]: cu[i] + j] = 0.0
        d2[cu[i]: cu[i] + j] = t[cu[i] + i: cu[i] + i + j]  # q = p before j: accepted
        d2[cu[i] + j, tok[cu[i] + j]] += 6.0
        ua[cu[i] + j] = 0.5
    uf = rng.random(B).astype(np.float32)
    res = O.verify_sample(t, d2, tok, cu, T, ua, uf, lib=lib)
    assert res.status == O.OK and res.accept_len.tolist() == [1, 0, 4, 0, 0]
    for i in range(B):
        a = int(res.accept_len[i])
        drow = d2[cu[i] + a] if a < k[i] else None
        w = _ref_final_weights(t[cu[i] + i + a], drow, T)
        C = np.cumsum(w)
        y = int(res.tokens[cu[i] + i + a])
        assert y == int(np.searchsorted(C, float(uf[i]) * C[-1], side="right")), (i, y)
        uS, S, lo, hi = res.final[i]
        assert abs(S - C[-1]) <= 1e-12 * C[-1], (i, S, C[-1])
        assert abs(uS - float(uf[i]) * C[-1]) <= 1e-12 * C[-1], (i, uS)
        assert abs(lo - (C[y - 1] if y > 0 else 0.0)) <= 1e-12 * C[-1], (i, lo)
        assert abs(hi - C[y]) <= 1e-12 * C[-1], (i, hi)
        assert lo <= uS < hi, (i, lo, uS, hi)


def pin_sample_errors(lib):
    t = np.zeros((3, 4), np.float32)
    d = np.zeros((1, 4), np.float32)
    cu = np.array([0, 1, 1], np.int32)
    u1 = np.array([0.5], np.float32)
    u2 = np.array([0.5, 0.5], np.float32)
    res = O.verify_sample(t, d, np.array([4], np.int32), cu, 1.0, u1, u2, lib=lib)
    assert res.status == O.ERR_INVALID_ARG and res.accept_len.tolist() == [-1, 0]
    d2 = d.copy()
    d2[0, 3] = np.inf
    res = O.verify_sample(t, d2, np.array([1], np.int32), cu, 1.0, u1, u2, lib=lib)
    assert res.status == O.ERR_NONFINITE and res.accept_len[0] == -1
    res = O.verify_sample(t, d, np.array([1], np.int32), cu, -1.0, u1, u2, lib=lib)
    assert res.status == O.ERR_INVALID_ARG
    # every row of a request is read: a NaN in the bonus row is an error even
    # when position 0 rejects (p(x) = 0 forces the rejection here)
    t3 = np.zeros((3, 4), np.float32)
    t3[0, 1] = -np.inf
    t3[1, 2] = np.nan
    res = O.verify_sample(t3, d, np.array([1], np.int32), cu, 1.0, np.zeros(1, np.float32),
                          u2, lib=lib)
    assert res.status == O.ERR_NONFINITE and res.accept_len.tolist() == [-1, 0]


# ---------------------------------------------------------------------------
# D-cut
# ---------------------------------------------------------------------------


def _prefix_products_f32(conf_row, n):
    """fp32 running products, one rounding per factor (numpy float32 multiply)."""
    out = []
    P = np.float32(1.0)
    for j in range(n):
        P = np.float32(P * np.float32(conf_row[j]))
        out.append(P)
    return out


def _brute_dcut(conf, kmax, budget, min_gain):
    """Enumerate every depth vector with 0 <= depth_i <= kmax_i, sum <= budget,
    using only positions with P >= min_gain; maximise the expected accepted
    tokens sum_i sum_{d <= depth_i} P_{i,d}; among optima keep the one that
    verifies the most positions, then the lexicographically largest."""
    P = [_prefix_products_f32(conf[i], kmax[i]) for i in range(len(kmax))]
    caps = [sum(1 for x in P[i] if x >= min_gain) for i in range(len(kmax))]
    best = None
    for depths in itertools.product(*[range(c + 1) for c in caps]):
        if sum(depths) > budget:
            continue
        val = sum(sum(float(x) for x in P[i][:depths[i]]) for i in range(len(kmax)))
        key = (round(val, 12), sum(depths), depths)
        if best is None or key > best[0]:
            best = (key, depths, val)
    return list(best[1]), best[2]


def pin_dcut_golden(lib):
    for case in _golden("dcut_ties.json")["cases"]:
        conf = np.array(case["conf"], np.float32)
        res = O.dcut_allocate(conf, np.array(case["kmax"], np.int32), case["budget"],
                              case["min_gain"], lib=lib)
        assert res.status == O.OK
        assert res.depth.tolist() == case["expected_depth"], (case["name"], res.depth)
        assert res.cu.tolist() == [0] + np.cumsum(case["expected_depth"]).tolist()


def pin_dcut_brute_force(lib):
    rng = np.random.default_rng(11)
    for trial in range(60):
        B = int(rng.integers(1, 5))
        Kmax = int(rng.integers(1, 5))
        kmax = rng.integers(0, Kmax + 1, size=B).astype(np.int32)
        conf = rng.uniform(0.05, 1.0, size=(B, Kmax)).astype(np.float32)
        min_gain = float(rng.choice([0.0, 0.0, 0.3]))
        for budget in range(0, int(kmax.sum()) + 2):
            res = O.dcut_allocate(conf, kmax, budget, min_gain, lib=lib)
            assert res.status == O.OK
            depths, val = _brute_dcut(conf.tolist(), kmax.tolist(), budget, min_gain)
            assert res.depth.tolist() == depths, (trial, budget, res.depth, depths)
            assert abs(res.expected.sum() - val) <= 1e-9 * max(1.0, val)


def pin_dcut_expected_len(lib):
    rng = np.random.default_rng(12)
    B, Kmax = 6, 16
    conf = (rng.beta(8, 2, size=(B, Kmax)) * 0.95 ** np.arange(Kmax)).astype(np.float32)
    kmax = np.full(B, Kmax, np.int32)
    res = O.dcut_allocate(conf, kmax, 40, 0.0, lib=lib)
    assert res.status == O.OK and int(res.depth.sum()) == 40
    for i in range(B):
        P = np.cumprod(conf[i].astype(np.float32), dtype=np.float32)
        assert abs(res.expected[i] - float(P[:res.depth[i]].astype(np.float64).sum())) < 1e-12
    # depth is monotone in the budget
    prev = np.zeros(B, np.int32)
    for budget in range(0, B * Kmax + 1, 7):
        d = O.dcut_allocate(conf, kmax, budget, 0.0, lib=lib).depth
        assert np.all(d >= prev)
        prev = d


def pin_dcut_errors(lib):
    ok = np.array([[0.5, 0.5]], np.float32)
    km = np.array([2], np.int32)
    assert O.dcut_allocate(ok, km, 1, lib=lib).status == O.OK
    assert O.dcut_allocate(np.array([[0.5, 1.5]], np.float32), km, 1,
                           lib=lib).status == O.ERR_INVALID_ARG
    assert O.dcut_allocate(np.array([[np.nan, 0.5]], np.float32), km, 1,
                           lib=lib).status == O.ERR_INVALID_ARG
    assert O.dcut_allocate(ok, np.array([3], np.int32), 1, lib=lib).status == O.ERR_INVALID_ARG
    assert O.dcut_allocate(ok, km, -1, lib=lib).status == O.ERR_INVALID_ARG


ALL_PINS = [
    pin_softmax_closed_form_v2, pin_softmax_matches_library, pin_softmax_invariances,
    pin_softmax_errors, pin_argmax, pin_inverse_cdf, pin_greedy_golden,
    pin_greedy_brute_force, pin_greedy_padded_layout, pin_greedy_errors, pin_sample_golden,
    pin_lossless_chi_square, pin_q_equals_p_accepts_all, pin_residual_closed_forms,
    pin_sample_outputs_layout, pin_final_cdf_and_diagnostics, pin_sample_errors,
    pin_dcut_golden, pin_dcut_brute_force,
    pin_dcut_expected_len, pin_dcut_errors,
]


# ---------------------------------------------------------------------------
# D-cut, cost-unit variant
# ---------------------------------------------------------------------------


def _padded(conf_rows):
    K = max(len(r) for r in conf_rows)
    c = np.zeros((len(conf_rows), K), np.float32)
    for i, r in enumerate(conf_rows):
        c[i, :len(r)] = r
    return c


def pin_dcut_cost_table(lib):
    """Hand-interpolated latency table (tests/golden/dcut_cost.json)."""
    g = _golden("dcut_cost.json")
    for d, want in g["cost_table"]:
        got = O.dcut_cost(d, lib=lib)
        assert abs(got - want) <= 1e-15, (d, got, want)


def pin_dcut_cost_golden(lib):
    g = _golden("dcut_cost.json")
    for case in g["cases"]:
        r = O.dcut_schedule_cost(_padded(case["conf"]), np.array(case["kmax"], np.int32),
                                 case["max_cost"], lib=lib)
        assert r.status == O.OK, case["name"]
        assert r.depth.tolist() == case["expected_depth"], (case["name"], r.depth)
        assert r.cu.tolist() == [0] + np.cumsum(case["expected_depth"]).tolist(), case["name"]


def pin_dcut_cost_invariants(lib):
    """Random batches: the admitted total stays within the budget (costs read
    from the hand table), every depth lies in 1..kmax or is 0, and a budget
    above every request's cost admits every request that drafted something."""
    g = _golden("dcut_cost.json")
    table = dict((int(d), c) for d, c in g["cost_table"])
    full = {d: table.get(d) for d in range(0, 33)}
    rng = np.random.default_rng(11)
    for trial in range(40):
        B = int(rng.integers(1, 9))
        Kmax = int(rng.integers(1, 9))
        kmax = rng.integers(0, Kmax + 1, size=B).astype(np.int32)
        conf = rng.random((B, Kmax)).astype(np.float32)
        budget = float(rng.choice([0.5, 1.0, 2.5, 4.0, 100.0]))
        r = O.dcut_schedule_cost(conf, kmax, budget, lib=lib)
        assert r.status == O.OK
        d = r.depth
        assert np.all((d == 0) | ((d >= 1) & (d <= kmax))), (kmax, d)
        known = [full[int(x)] for x in d if x > 0 and full[int(x)] is not None]
        if len(known) == int((d > 0).sum()):
            assert sum(known) <= budget + 1e-12, (d, budget)
        if budget >= 3.0 * B:
            assert np.all((d > 0) == (kmax > 0)), (kmax, d)


def pin_dcut_cost_errors(lib):
    c = np.array([[0.5, 1.5]], np.float32)
    assert O.dcut_schedule_cost(c, np.array([2], np.int32), 4.0, lib=lib).status == \
        O.ERR_INVALID_ARG
    assert O.dcut_schedule_cost(np.zeros((1, 2), np.float32), np.array([3], np.int32), 4.0,
                                lib=lib).status == O.ERR_INVALID_ARG
    assert O.dcut_schedule_cost(np.zeros((1, 2), np.float32), np.array([2], np.int32),
                                float("nan"), lib=lib).status == O.ERR_INVALID_ARG


ALL_PINS += [pin_dcut_cost_table, pin_dcut_cost_golden, pin_dcut_cost_invariants,
             pin_dcut_cost_errors]


# ---------------------------------------------------------------------------
# prefix confidence of drafted tokens
# ---------------------------------------------------------------------------


def pin_draft_confidence(lib):
    """q(x) against scipy's softmax in fp64 (f32 and bf16 rows); T = 0 against
    numpy's first-occurrence argmax; zeros past kmax; errors."""
    rng = np.random.default_rng(21)
    B, Kmax, V = 5, 4, 37
    l = (rng.standard_normal((B * Kmax, V)) * 2).astype(np.float32)
    tok = rng.integers(0, V, size=B * Kmax).astype(np.int32)
    kmax = np.array([4, 0, 2, 3, 1], np.int32)
    for T in (0.6, 1.0, 1.7):
        for rows, exact in ((l, l), (_to_bf16_bits(l), None)):
            if exact is None:
                exact = (rows.astype(np.uint32) << 16).view(np.float32)
            st, c = O.draft_confidence(rows, tok, kmax, T, lib=lib)
            assert st == O.OK
            for i in range(B):
                for j in range(Kmax):
                    r = i * Kmax + j
                    want = _ref_softmax(exact[r], T)[tok[r]] if j < kmax[i] else 0.0
                    assert abs(c[i, j] - want) <= 1e-6 * max(want, 1e-30), (T, i, j, c[i, j], want)
    ties = rng.integers(-3, 3, size=(B * Kmax, V)).astype(np.float32)  # many ties
    g = np.argmax(ties, axis=1)
    tok2 = np.where(rng.random(B * Kmax) < 0.5, g, (g + 1) % V).astype(np.int32)
    st, c = O.draft_confidence(ties, tok2, kmax, 0.0, lib=lib)
    assert st == O.OK
    for i in range(B):
        for j in range(Kmax):
            r = i * Kmax + j
            want = (1.0 if tok2[r] == g[r] else 0.0) if j < kmax[i] else 0.0
            assert c[i, j] == want, (i, j)
    bad = l.copy()
    bad[2 * Kmax + 1, 5] = np.nan  # request 2, position 1 (inside kmax = 2)
    st, c = O.draft_confidence(bad, tok, kmax, 1.0, lib=lib)
    assert st == O.ERR_NONFINITE and np.isnan(c[2, 1]) and not np.isnan(c[2, 0])
    tok3 = tok.copy()
    tok3[0] = V
    st, c = O.draft_confidence(l, tok3, kmax, 1.0, lib=lib)
    assert st == O.ERR_INVALID_ARG and np.isnan(c[0, 0])
    assert O.draft_confidence(l, tok, np.array([4, 0, 2, 3, 5], np.int32), 1.0,
                              lib=lib)[0] == O.ERR_INVALID_ARG


ALL_PINS += [pin_draft_confidence]


# ---------------------------------------------------------------------------
# drafted tokens and acceptance statistics
# ---------------------------------------------------------------------------


def pin_draft_sample(lib):
    """x = searchsorted(cumsum(scipy softmax), u*S, 'right') on random rows
    (f32, bf16); conf = q(x); T = 0: numpy's first-occurrence argmax; rows
    past kmax give -1; errors."""
    rng = np.random.default_rng(31)
    B, Kmax, V = 6, 3, 41
    l = (rng.standard_normal((B * Kmax, V)) * 2).astype(np.float32)
    l[rng.random(l.shape) < 0.2] = -np.inf  # masked entries never drawn
    kmax = np.array([3, 1, 0, 2, 3, 3], np.int32)
    u = rng.random(B * Kmax).astype(np.float32)
    for T in (0.7, 1.0):
        for rows, exact in ((l, l), (_to_bf16_bits(l), None)):
            if exact is None:
                exact = (rows.astype(np.uint32) << 16).view(np.float32)
            st, tok, conf = O.draft_sample(rows, kmax, Kmax, T, u, lib=lib)
            assert st == O.OK
            for i in range(B):
                for j in range(Kmax):
                    r = i * Kmax + j
                    if j >= kmax[i]:
                        assert tok[r] == -1 and conf[r] == 0.0
                        continue
                    q = _ref_softmax(exact[r], T)
                    C = np.cumsum(q)
                    want = int(np.searchsorted(C, float(u[r]) * C[-1], side="right"))
                    assert tok[r] == want, (T, i, j, tok[r], want)
                    assert abs(conf[r] - q[want]) <= 1e-6 * q[want]
    g = np.argmax(l, axis=1)
    st, tok, conf = O.draft_sample(l, kmax, Kmax, 0.0, u, lib=lib)
    assert st == O.OK
    for i in range(B):
        for j in range(Kmax):
            r = i * Kmax + j
            assert tok[r] == (g[r] if j < kmax[i] else -1)
    bad = l.copy()
    bad[1, 3] = np.inf  # request 0, position 1
    st, tok, conf = O.draft_sample(bad, kmax, Kmax, 1.0, u, lib=lib)
    assert st == O.ERR_NONFINITE and tok[1] == -1 and np.isnan(conf[1]) and tok[0] >= 0


def pin_draft_sample_chi_square(lib):
    """The drawn tokens follow softmax(l / T): Pearson chi-square, alpha 1e-3."""
    rng = np.random.default_rng(32)
    row = np.array([0.3, -1.2, 2.0, 0.0, 1.1, -0.4, 0.7, -2.0], np.float32)
    n = 200_000
    rows = np.tile(row, (n, 1))
    u = rng.random(n).astype(np.float32)
    for T in (0.7, 1.0):
        st, tok, _ = O.draft_sample(rows, np.ones(n, np.int32), 1, T, u, lib=lib)
        assert st == O.OK
        ok, chi2, dof = _chi2_ok(np.bincount(tok, minlength=8), _ref_softmax(row, T))
        assert ok, (T, chi2, dof)


def pin_acceptance_stats(lib):
    g = _golden("acceptance_stats.json")
    k = np.array(g["k"], np.int32)
    cu = np.concatenate([[0], np.cumsum(k)]).astype(np.int32)
    st, reached, accepted, mean = O.acceptance_stats(np.array(g["accept_len"], np.int32), cu,
                                                     g["Kmax"], lib=lib)
    assert st == O.OK
    assert reached.tolist() == g["expected_reached"], reached
    assert accepted.tolist() == g["expected_accepted"], accepted
    assert abs(mean - g["expected_mean"]) < 1e-15
    # a length beyond its request's K is an error
    bad = np.array(g["accept_len"], np.int32)
    bad[1] = 3
    assert O.acceptance_stats(bad, cu, g["Kmax"], lib=lib)[0] == O.ERR_INVALID_ARG


ALL_PINS += [pin_draft_sample, pin_draft_sample_chi_square, pin_acceptance_stats]


def pin_masked_in_both_rows_rejects(lib):
    """The drafted token masked in both the target and the draft row: p = q = 0,
    so no u in [0, 1) accepts it (the limit of min(1, p/q) with p = 0 is 0;
    an underflowed q only accepts when p > 0).  The residual max(0, p - q) is
    then identically zero on the uniform rows below, so the token is drawn
    from p itself: u_final = 0.6 over p = (1/2, 1/2, 0) picks token 1."""
    ninf = float("-inf")
    target = np.array([[0.0, 0.0, ninf], [0.0, 0.0, ninf]], np.float32)  # rows 0 and bonus
    draft = np.array([[0.0, 0.0, ninf]], np.float32)
    for u in (0.0, 0.5, 0.999):
        r = O.verify_sample(target, draft, np.array([2], np.int32), np.array([0, 1], np.int32),
                            1.0, np.array([u], np.float32), np.array([0.6], np.float32), lib=lib)
        assert r.status == O.OK
        assert r.accept_len.tolist() == [0], (u, r.accept_len)
        assert r.tokens.tolist() == [1, -1], (u, r.tokens)


ALL_PINS += [pin_masked_in_both_rows_rejects]
