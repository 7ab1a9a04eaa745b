"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bar: see tests/parity.py (bit-exact tokens / lengths / depths, accept
decisions exempt only within 1e-6 of p/q, final tokens exempt only within
1e-6*S of a CDF boundary, p and q within 1e-5 relative)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle as O
import parity
from draft_verification_02_b300 import specverify as sv
from draft_verification_02_b300 import workloads as W
from draft_verification_02_b300.verifier import Verifier

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
MAX_EXEMPT = 2  # per test; the expected rate is ~1e-5 per decision


def run_gpu(batch, rows=None, cu=None):
    batch = batch.to("cuda")
    v = Verifier(batch.B, rows or batch.n_target_rows, batch.V)
    out = v.verify(batch, rows, cu_draft=cu)
    torch.cuda.synchronize()
    return batch, out, v


def check_batch(batch, reqs=None, rows=None):
    batch, out, v = run_gpu(batch, rows)
    assert v.device_status() == sv.SPEC_OK
    rep = parity.compare_batch(batch, out, reqs)
    assert rep["exempt_accept"] + rep["exempt_final"] <= MAX_EXEMPT, rep
    return rep


def ragged_batch(B, V, T, dtype, seed, kmax=16, kmin=0, draft_stride=0, sigma=2.0,
                 noise=1.0, mask_frac=0.0):
    """Hand-sized batch through the workload generator's recipe."""
    g = torch.Generator().manual_seed(seed)
    k = torch.randint(kmin, kmax + 1, (B,), generator=g, dtype=torch.int32)
    w = W.Workload("custom", B=B, V=V, dtype=dtype, seed=seed, k=None, k_range=(kmin, kmax),
                   target_sigma=sigma, draft_sigma=(noise,))
    b = W.make_verify_batch(w, T, "cpu", depths=k, draft_stride=draft_stride)
    if mask_frac:
        m = torch.rand(b.target_logits.shape, generator=g) < mask_frac
        b.target_logits[m] = float("-inf")
        md = torch.rand(b.draft_logits.shape, generator=g) < mask_frac
        b.draft_logits[md] = float("-inf")
        # keep the drafted tokens themselves drawable from q
        d_idx = torch.arange(b.draft_tokens.numel())
        b.draft_logits[d_idx, b.draft_tokens.long()] = 1.0
    return b


def pad_to_loose_bound(b, rows):
    """Grow the row buffers of a packed or padded batch to a host bound of
    `rows` target rows, the rows past the real ones NaN (a kernel that read
    one would poison its request)."""
    V, dt = b.V, b.target_logits.dtype
    nan = float("nan")
    b.target_logits = torch.cat(
        [b.target_logits, torch.full((rows - b.n_target_rows, V), nan, dtype=dt)])
    if b.draft_stride == 0:
        extra = rows - b.B - b.draft_logits.shape[0]
        b.draft_logits = torch.cat([b.draft_logits, torch.full((extra, V), nan, dtype=dt)])
        b.draft_tokens = torch.cat([b.draft_tokens, torch.zeros(extra, dtype=torch.int32)])
        b.u_accept = torch.cat([b.u_accept, torch.full((extra,), 0.5)])
    return b


# ---------------------------------------------------------------------------
# small configurations, every request compared
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_tiny_config(T):
    check_batch(W.make_verify_batch(W.TINY, T, "cpu"))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [1, 7, 1000, 4099, 12345, 40000])
@pytest.mark.parametrize("T", [0.0, 0.7, 1.0])
def test_shapes(V, dtype, T):
    """Several chunks and a ragged tail; V*e not a multiple of 16 takes the
    plain-load path; depths 0..32 including empty requests."""
    b = ragged_batch(6, V, T, dtype, seed=V * 7 + int(T * 10), kmax=32)
    check_batch(b)


@pytest.mark.parametrize("T", [0.0, 0.7])
def test_padded_draft_layout(T):
    b = ragged_batch(9, 5000, T, "bf16", seed=3, kmax=8, draft_stride=8)
    check_batch(b)


@pytest.mark.parametrize("V,dtype", [(5000, "bf16"), (4099, "f32")])
@pytest.mark.parametrize("T", [0.7, 1.0])
def test_four_cta_draws_at_full_depth(V, dtype, T):
    """A batch large enough that each draw takes a cluster of 4 CTAs (more
    than half a request per SM), with most requests at the largest depth
    (65 rows: one more than the cluster's share, merged by every CTA)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    b = ragged_batch(sms // 2 + 4, V, T, dtype, seed=V + int(T * 10), kmin=28, kmax=32)
    assert int(b.k.max()) == 32
    check_batch(b)


@pytest.mark.parametrize("T", [0.0, 0.7, 1.0, 1.3])
def test_masked_vocabulary(T):
    b = ragged_batch(8, 3000, T, "bf16", seed=4, kmax=6, mask_frac=0.3)
    check_batch(b)


def test_drafted_token_masked_in_target_rejects():
    b = ragged_batch(4, 2048, 1.0, "f32", seed=5, kmin=2, kmax=4)
    for i in range(4):
        t0 = int(b.cu_draft[i]) + i
        b.target_logits[t0, b.draft_tokens[int(b.cu_draft[i])].long()] = float("-inf")
    batch, out, v = run_gpu(b)
    assert torch.all(out["accept_len"].cpu() == 0)
    parity.compare_batch(batch, out)


def test_drafted_token_masked_in_both_rows_rejects():
    """p = q = 0 for the drafted token: rejected for every u (an underflowed q
    accepts only when p > 0), then the residual is drawn as usual."""
    b = ragged_batch(4, 2048, 1.0, "f32", seed=7, kmin=2, kmax=4)
    b.u_accept[:] = 0.0  # the most permissive uniform still rejects
    for i in range(4):
        t0, d0 = int(b.cu_draft[i]) + i, int(b.cu_draft[i])
        x = b.draft_tokens[d0].long()
        b.target_logits[t0, x] = float("-inf")
        b.draft_logits[d0, x] = float("-inf")
    batch, out, v = run_gpu(b)
    assert torch.all(out["accept_len"].cpu() == 0)
    assert v.device_status() == sv.SPEC_OK
    rep = parity.compare_batch(batch, out)
    assert rep["exempt_final"] <= MAX_EXEMPT, rep


def test_identical_rows_accept_everything():
    """q = p makes p/q = 1, so every u < 1 accepts.  The kernels sum the
    target and draft rows in different orders, so their p/q is 1 only to
    fp32 rounding; u sits just outside the 1e-6 band in which an accept
    decision may differ from the oracle's, and the band's edge itself is
    compared by parity (u = 1 - 2^-24 there)."""
    b = ragged_batch(8, 3000, 0.8, "bf16", seed=6, kmin=1, kmax=10)
    for i in range(8):
        K = int(b.k[i])
        t0, d0 = int(b.cu_draft[i]) + i, int(b.cu_draft[i])
        b.draft_logits[d0:d0 + K] = b.target_logits[t0:t0 + K]
    b.u_accept[:] = 1.0 - 2.0 ** -16
    batch, out, v = run_gpu(b)
    assert torch.equal(out["accept_len"].cpu(), b.k)
    parity.compare_batch(batch, out)
    b.u_accept[:] = float(np.nextafter(np.float32(1), np.float32(0)))
    batch, out, v = run_gpu(b)
    rep = parity.compare_batch(batch, out)
    assert rep["exempt_accept"] <= b.B, rep


@pytest.mark.parametrize("T", [0.7, 1.0])
def test_one_hot_draft(T):
    b = ragged_batch(6, 512, T, "f32", seed=7, kmin=1, kmax=5)
    b.draft_logits[:] = float("-inf")
    rows = torch.arange(b.draft_logits.shape[0])
    b.draft_logits[rows, b.draft_tokens.long()] = 0.0
    check_batch(b)


@pytest.mark.parametrize("name", ["greedy", "sample"])
def test_golden_fixtures_on_gpu(name):
    if name == "greedy":
        g = json.load(open(os.path.join(GOLDEN, "greedy_layout.json")))
        V = g["V"]
        t = np.zeros((len(g["target_peaks"]), V), np.float32)
        for r, pk in enumerate(g["target_peaks"]):
            t[r, pk] = 5.0
        b = W.batch_from_rows(t.tolist(), [], g["draft_tokens"], g["k"],
                              [0.0] * len(g["draft_tokens"]), [0.0] * len(g["k"]), 0.0)
        batch, out, v = run_gpu(b)
        assert out["accept_len"].cpu().tolist() == g["expected_accept_len"]
        assert out["tokens"].cpu().tolist() == g["expected_tokens"]
        return
    g = json.load(open(os.path.join(GOLDEN, "sample_v2.json")))
    for case in g["cases"]:
        def val(x):
            return {"L": g["L"], "-inf": float("-inf")}.get(x, x) if isinstance(x, str) else x
        t = [[val(x) for x in r] for r in case["target"]]
        d = [[val(x) for x in r] for r in case["draft"]]
        b = W.batch_from_rows(t, d, case["tokens"], [case["k"]], case["u_accept"],
                              [case["u_final"]], g["temperature"])
        batch, out, v = run_gpu(b)
        assert out["accept_len"].cpu().tolist() == [case["expected_accept_len"]], case["name"]
        assert out["tokens"].cpu().tolist() == case["expected_tokens"], case["name"]
        np.testing.assert_allclose(out["p"].cpu().numpy()[:case["k"]], case["expected_p"],
                                   rtol=1e-6, atol=1e-12)
        np.testing.assert_allclose(out["q"].cpu().numpy()[:case["k"]], case["expected_q"],
                                   rtol=1e-6, atol=1e-12)


# ---------------------------------------------------------------------------
# the workloads at full size
# ---------------------------------------------------------------------------


def test_mtp_config_full():
    check_batch(W.make_verify_batch(W.MTP, 1.0, "cuda"))


@pytest.mark.parametrize("T", [0.0, 0.7])
def test_block_config_full(T):
    check_batch(W.make_verify_batch(W.BLOCK, T, "cuda"))


def test_dcut_config_full():
    """Config 4: D-cut on the device, its offsets feed the ragged verify
    directly (no host round trip), drafts padded to Kmax per request."""
    w = W.DCUT
    prob = W.make_dcut_problem(w, "cuda")
    v = Verifier(w.B, W.max_target_rows(w), w.V)
    d = v.dcut(prob.conf, prob.kmax, prob.budget)
    torch.cuda.synchronize()
    o = O.dcut_allocate(prob.conf.cpu().numpy(), prob.kmax.cpu().numpy(), prob.budget)
    assert o.status == O.OK
    assert d["depth"].cpu().numpy().tolist() == o.depth.tolist()
    assert d["cu"].cpu().numpy().tolist() == o.cu.tolist()
    np.testing.assert_allclose(d["expected"].cpu().numpy(), o.expected, rtol=1e-6)
    assert int(o.depth.sum()) == w.budget
    batch = W.make_verify_batch(w, 1.0, "cuda", depths=torch.from_numpy(o.depth),
                                draft_stride=w.kmax)
    rows = W.max_target_rows(w)
    # pad the target side to the host bound the grid is sized for
    t = torch.zeros((rows, w.V), dtype=batch.target_logits.dtype, device="cuda")
    t[:batch.target_logits.shape[0]] = batch.target_logits
    batch.target_logits = t
    out = v.verify(batch, rows, cu_draft=d["cu"])
    torch.cuda.synchronize()
    assert v.device_status() == sv.SPEC_OK
    rep = parity.compare_batch(batch, out)
    assert rep["exempt_accept"] + rep["exempt_final"] <= MAX_EXEMPT, rep


@pytest.mark.parametrize("pair", range(18))
def test_ragged_sweep(pair):
    """Every request against the oracle at one temperature per (B, V) pair
    (T = 0.7, the sampling path); the other two temperatures on every request
    for B <= 16 and on a seeded sample (first, last and ten more) above."""
    w = W.ragged(pair)
    for T in W.RAGGED_T:
        batch = W.make_verify_batch(w, T, "cuda")
        if w.B <= 16 or T == 0.7:
            reqs = None
        else:
            rng = np.random.default_rng(pair)
            reqs = sorted({0, w.B - 1, *rng.choice(w.B, 10, replace=False).tolist()})
        check_batch(batch, reqs)


# ---------------------------------------------------------------------------
# properties
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("T", [0.0, 0.7])
def test_repeat_calls_are_bit_identical(T):
    batch = W.make_verify_batch(W.ragged(10), T, "cuda")
    v = Verifier(batch.B, batch.n_target_rows, batch.V)
    a = v.verify(batch)
    b = v.verify(batch)
    torch.cuda.synchronize()
    for k in ("tokens", "accept_len", "p", "q"):
        assert torch.equal(a[k].view(torch.int32), b[k].view(torch.int32)), k


def _replicated(p_rows, q_rows, n, rng, T):
    K = len(q_rows)
    V = len(p_rows[0])
    target = np.tile(np.asarray(p_rows, np.float32), (n, 1))
    draft = np.tile(np.asarray(q_rows, np.float32), (n, 1))
    toks = np.empty((n, K), np.int32)
    from scipy import special
    for j in range(K):
        q = special.softmax(np.asarray(q_rows[j], np.float64) / T)
        toks[:, j] = rng.choice(V, size=n, p=q / q.sum())
    cu = (np.arange(n + 1) * K).astype(np.int32)
    return target, draft, toks.reshape(-1), cu


@pytest.mark.parametrize("pair", ["random", "disjointish", "onehot_q"])
@pytest.mark.parametrize("T", [0.7, 1.0])
def test_lossless_chi_square_gpu(pair, T):
    """10^6 seeded trials on V = 8 through the GPU: emitted tokens follow the
    target law (position 0; position 1 given one acceptance; the bonus token
    given two), and P(accept at 0) = sum_v min(p, q)."""
    import oracle_pins as P
    from scipy import special
    p_rows, q_rows = P.PAIRS[pair]
    rng = np.random.default_rng(123)
    n_total, n = 1_000_000, 4096
    V = 8
    c = [np.zeros(V, np.int64) for _ in range(3)]
    acc0 = 0
    v = Verifier(n, 3 * n, V)
    done = 0
    while done < n_total:
        m = min(n, n_total - done)
        t, d, tok, cu = _replicated(p_rows, q_rows, m, rng, T)
        ua = rng.random(2 * m).astype(np.float32)
        uf = rng.random(m).astype(np.float32)
        b = W.VerifyBatch(B=m, V=V, dtype="f32", temperature=T,
                          k=torch.full((m,), 2, dtype=torch.int32),
                          cu_draft=torch.from_numpy(cu), target_logits=torch.from_numpy(t),
                          draft_logits=torch.from_numpy(d), draft_tokens=torch.from_numpy(tok),
                          u_accept=torch.from_numpy(ua), u_final=torch.from_numpy(uf)).to("cuda")
        out = v.verify(b)
        toks = out["tokens"].cpu().numpy().reshape(m, 3)
        a = out["accept_len"].cpu().numpy()
        c[0] += np.bincount(toks[:, 0], minlength=V)
        c[1] += np.bincount(toks[a >= 1, 1], minlength=V)
        c[2] += np.bincount(toks[a == 2, 2], minlength=V)
        acc0 += int((a >= 1).sum())
        done += m
    assert v.device_status() == sv.SPEC_OK
    for j in range(3):
        if c[j].sum() < 1000:
            continue
        pj = special.softmax(np.asarray(p_rows[j], np.float64) / T)
        ok, chi2, dof = P._chi2_ok(c[j], pj)
        assert ok, (pair, T, j, chi2, dof)
    p0 = special.softmax(np.asarray(p_rows[0], np.float64) / T)
    q0 = special.softmax(np.asarray(q_rows[0], np.float64) / T)
    alpha = float(np.minimum(p0, q0).sum())
    sd = np.sqrt(max(alpha * (1 - alpha), 1e-12) / n_total)
    assert abs(acc0 / n_total - alpha) < 5 * sd + 1e-12


# ---------------------------------------------------------------------------
# errors: host checks, device status and poisoned outputs
# ---------------------------------------------------------------------------


def test_nonfinite_logits_poison_only_their_request():
    b = ragged_batch(5, 2000, 1.0, "bf16", seed=8, kmin=1, kmax=4)
    b.target_logits[int(b.cu_draft[2]) + 2, 17] = float("nan")
    b.draft_logits[int(b.cu_draft[4]), 3] = float("inf")
    batch, out, v = run_gpu(b)
    assert v.device_status() == sv.SPEC_ERR_NONFINITE
    assert v.device_status() == sv.SPEC_OK  # read clears
    lens = out["accept_len"].cpu().tolist()
    assert lens[2] == -1 and lens[4] == -1
    h = parity.to_host(batch)
    o = O.verify_sample(h["target"], h["draft"], h["tokens"], h["cu"], 1.0, h["u_accept"],
                        h["u_final"])
    assert o.status == O.ERR_NONFINITE
    assert lens == o.accept_len.tolist()
    assert out["tokens"].cpu().tolist() == o.tokens.tolist()


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_fully_masked_row_and_bad_token(T):
    b = ragged_batch(4, 1024, T, "f32", seed=9, kmin=1, kmax=3)
    b.target_logits[int(b.cu_draft[1]) + 1 + int(b.k[1])] = float("-inf")  # bonus row masked
    b.draft_tokens[int(b.cu_draft[3])] = 1024  # out of range
    batch, out, v = run_gpu(b)
    st = v.device_status()
    assert st == sv.SPEC_ERR_INVALID_ARG  # precedence over NONFINITE
    lens = out["accept_len"].cpu().tolist()
    assert lens[1] == -1 and lens[3] == -1 and lens[0] >= 0 and lens[2] >= 0


def test_malformed_offsets_poison_everything():
    b = ragged_batch(4, 1024, 1.0, "bf16", seed=10, kmin=2, kmax=3)
    rows = b.n_target_rows
    bad_cu = b.cu_draft.clone()
    bad_cu[2] = bad_cu[1] - 1  # decreasing
    batch = b.to("cuda")
    v = Verifier(b.B, rows, b.V)
    out = v.verify(batch, rows, cu_draft=bad_cu.cuda())
    assert v.device_status() == sv.SPEC_ERR_INVALID_ARG
    assert torch.all(out["accept_len"].cpu() == -1)
    assert torch.all(out["tokens"].cpu() == -1)
    # the workspace stays usable: a good call afterwards is correct
    out2 = v.verify(batch, rows)
    torch.cuda.synchronize()
    assert v.device_status() == sv.SPEC_OK
    parity.compare_batch(batch, out2)


def test_host_argument_errors():
    b = ragged_batch(3, 256, 1.0, "f32", seed=11, kmin=1, kmax=2).to("cuda")
    rows = b.n_target_rows
    v = Verifier(b.B, rows, b.V)
    out = v.outputs(b)
    small = torch.zeros(16, dtype=torch.uint8, device="cuda")
    assert sv.spec_verify_sample(b.target_logits, b.draft_logits, b.draft_tokens, b.cu_draft,
                                 b.B, b.V, rows, 0, 1.0, b.u_accept, b.u_final, out["tokens"],
                                 out["accept_len"], None, None, small) == sv.SPEC_ERR_WORKSPACE
    assert sv.spec_verify_sample(b.target_logits, b.draft_logits, b.draft_tokens, b.cu_draft,
                                 b.B, b.V, rows, 0, -1.0, b.u_accept, b.u_final, out["tokens"],
                                 out["accept_len"], None, None,
                                 v.workspace) == sv.SPEC_ERR_INVALID_ARG
    assert sv.spec_verify_greedy(b.target_logits, b.draft_tokens, b.cu_draft, b.B, b.V,
                                 b.B - 1 if b.B > 1 else 0, 0, out["tokens"], out["accept_len"],
                                 v.workspace) == sv.SPEC_ERR_INVALID_ARG
    with pytest.raises(ValueError):  # host tensor never reaches the library
        sv.spec_verify_greedy(b.target_logits.cpu(), b.draft_tokens, b.cu_draft, b.B, b.V,
                              rows, 0, out["tokens"], out["accept_len"], v.workspace)


# ---------------------------------------------------------------------------
# D-cut
# ---------------------------------------------------------------------------


def test_dcut_random_against_oracle():
    rng = np.random.default_rng(21)
    v = Verifier(128, 128, 1)
    for trial in range(60):
        B = int(rng.integers(0, 129))
        Kmax = int(rng.integers(0, 33))
        if B * Kmax > sv.SPEC_DCUT_MAX_CANDIDATES:
            continue
        kmax = rng.integers(0, Kmax + 1, size=B).astype(np.int32)
        conf = (rng.beta(8, 2, size=(B, Kmax)) * 0.95 ** np.arange(Kmax)).astype(np.float32)
        if trial % 5 == 0:  # exact ties: powers of two and repeated rows
            conf = (0.5 ** rng.integers(0, 3, size=(B, Kmax))).astype(np.float32)
        budget = int(rng.integers(0, max(1, int(kmax.sum()) + 5)))
        min_gain = float(rng.choice([0.0, 0.0, 0.1, 0.5]))
        d = v.dcut(torch.from_numpy(conf).cuda(), torch.from_numpy(kmax).cuda(), budget,
                   min_gain)
        o = O.dcut_allocate(conf, kmax, budget, min_gain)
        assert o.status == O.OK
        assert d["depth"].cpu().numpy()[:B].tolist() == o.depth.tolist(), trial
        assert d["cu"].cpu().numpy().tolist() == o.cu.tolist(), trial
        if B:
            np.testing.assert_allclose(d["expected"].cpu().numpy()[:B], o.expected, rtol=1e-6,
                                       atol=1e-7)
    assert v.device_status() == sv.SPEC_OK


@pytest.mark.parametrize("B,Kmax", [(256, 32), (4096, 2), (1000, 8), (37, 5)])
def test_dcut_large_against_oracle(B, Kmax):
    """Many candidates per thread (up to SPEC_DCUT_MAX_CANDIDATES), exact ties
    across requests, budgets below, at and above the eligible count."""
    rng = np.random.default_rng(B * 100 + Kmax)
    v = Verifier(B, B, 1)
    kmax = rng.integers(0, Kmax + 1, size=B).astype(np.int32)
    for ties in (False, True):
        conf = (rng.beta(8, 2, size=(B, Kmax)) * 0.95 ** np.arange(Kmax)).astype(np.float32)
        if ties:
            conf = (0.5 ** rng.integers(0, 3, size=(B, Kmax))).astype(np.float32)
        total = int(kmax.sum())
        for budget in (0, 1, total // 3, total, total + 7):
            for min_gain in (0.0, 0.3):
                d = v.dcut(torch.from_numpy(conf).cuda(), torch.from_numpy(kmax).cuda(), budget,
                           min_gain)
                o = O.dcut_allocate(conf, kmax, budget, min_gain)
                assert o.status == O.OK
                assert d["depth"].cpu().numpy()[:B].tolist() == o.depth.tolist(), (budget, ties)
                assert d["cu"].cpu().numpy().tolist() == o.cu.tolist(), (budget, ties)
    assert v.device_status() == sv.SPEC_OK


def test_dcut_golden_on_gpu():
    v = Verifier(4, 4, 1)
    for case in json.load(open(os.path.join(GOLDEN, "dcut_ties.json")))["cases"]:
        d = v.dcut(torch.tensor(case["conf"], dtype=torch.float32, device="cuda"),
                   torch.tensor(case["kmax"], dtype=torch.int32, device="cuda"),
                   case["budget"], case["min_gain"])
        assert d["depth"].cpu().tolist() == case["expected_depth"], case["name"]


def test_dcut_invalid_confidence():
    v = Verifier(4, 4, 1)
    conf = torch.tensor([[0.5, 1.5], [0.2, 0.1]], device="cuda")
    d = v.dcut(conf, torch.tensor([2, 2], dtype=torch.int32, device="cuda"), 2)
    assert v.device_status() == sv.SPEC_ERR_INVALID_ARG
    assert d["depth"].cpu().tolist() == [-1, -1] and d["cu"].cpu().tolist() == [-1, -1, -1]


# ---------------------------------------------------------------------------
# launches and the trace hook
# ---------------------------------------------------------------------------


def test_launch_counts_and_trace():
    batch = W.make_verify_batch(W.MTP, 1.0, "cuda")
    v = Verifier(batch.B, batch.n_target_rows, batch.V)
    v.verify(batch)
    torch.cuda.synchronize()
    n0 = sv.spec_kernel_launch_count()
    v.verify(batch)
    assert sv.spec_kernel_launch_count() - n0 == 2
    g = W.make_verify_batch(W.TINY, 0.0, "cuda")
    vg = Verifier(g.B, g.n_target_rows, g.V)
    n0 = sv.spec_kernel_launch_count()
    vg.verify(g)
    assert sv.spec_kernel_launch_count() - n0 == 2
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    assert sv.spec_set_trace(ev) == sv.SPEC_OK
    v.verify(batch)
    assert sv.spec_set_trace(None) == sv.SPEC_OK
    torch.cuda.synchronize()
    assert ev[0].elapsed_time(ev[1]) > 0 and ev[1].elapsed_time(ev[2]) > 0


@pytest.mark.parametrize("T,stride", [(0.0, 0), (0.7, 0), (1.0, 8), (0.0, 8)])
def test_loose_row_bound_reads_only_real_rows(T, stride):
    """max_target_rows far above the real count, as when the offsets come
    from the device with only a host bound: the streaming pass splits the
    real rows afresh once it has read the offsets (dropping its speculative
    first copies), the finish kernel finds the partials under the same split,
    and the rows past the real count (NaN here) are never read."""
    B, V = 12, 20000
    b = ragged_batch(B, V, T, "bf16", seed=41, kmin=0, kmax=8, draft_stride=stride)
    loose = B * 33
    b = pad_to_loose_bound(b, loose)
    batch, out, v = run_gpu(b, rows=loose)
    assert v.device_status() == sv.SPEC_OK
    rep = parity.compare_batch(batch, out)
    assert rep["exempt_accept"] + rep["exempt_final"] <= MAX_EXEMPT, rep


@pytest.mark.parametrize("T,stride", [(0.0, 0), (0.7, 0), (1.0, 8)])
def test_loose_bound_over_a_long_host_split(T, stride):
    """The largest host bound the call accepts, long enough that the host's
    split balances bytes with units below the largest, over a few real rows:
    the re-split keeps the host's units over the real rows, and every kernel
    that reads the partials derives the same split from the offsets."""
    B, V = 16, 151936
    b = ragged_batch(B, V, T, "bf16", seed=43, kmin=0, kmax=8, draft_stride=stride)
    loose = B * 33  # the largest bound the call accepts
    b = pad_to_loose_bound(b, loose)
    batch, out, v = run_gpu(b, rows=loose)
    assert v.device_status() == sv.SPEC_OK
    rep = parity.compare_batch(batch, out)
    assert rep["exempt_accept"] + rep["exempt_final"] <= MAX_EXEMPT, rep
