"""GPU parity of the drafter's step and of the acceptance statistics.

spec_draft_sample: drafted tokens x ~ q by the inverse CDF at u (T > 0), or
the lowest-index maximum (T = 0), and q(x); against oracle.draft_sample.
Bar: tokens bit-exact, except a draw whose u*S lies within 1e-6*S of the
oracle's running sum at the boundary between the two tokens (at most 2 per
test); q(x) within 1e-5 relative; T = 0 exact.

spec_acceptance_stats: integer counts and the mean, bit-exact against
oracle.acceptance_stats."""
import numpy as np
import pytest
import torch

import oracle as O
import parity
from draft_verification_02_b300 import specverify as sv
from draft_verification_02_b300 import workloads as W
from draft_verification_02_b300.verifier import Verifier

pytestmark = pytest.mark.gpu

FINAL_BAND = parity.FINAL_BAND


def _inputs(B, Kmax, V, dtype, seed, full=False):
    g = torch.Generator().manual_seed(seed)
    d = torch.randn((B * Kmax, V), generator=g) * 2.0
    d = d.to(torch.bfloat16 if dtype == "bf16" else torch.float32).contiguous()
    kmax = (torch.full((B,), Kmax, dtype=torch.int32) if full else
            torch.randint(0, Kmax + 1, (B,), generator=g, dtype=torch.int32))
    u = torch.rand(B * Kmax, generator=g, dtype=torch.float32)
    if u.numel() >= 2:
        u[0] = 0.0
        u[-1] = float(np.nextafter(np.float32(1), np.float32(0)))
    return d, kmax, u.contiguous()


def _run(d, kmax, u, B, Kmax, V, T):
    v = Verifier(B, B * (Kmax + 1), V)
    out = v.draft(d.cuda(), kmax.cuda(), Kmax, T, None if T == 0 else u.cuda())
    torch.cuda.synchronize()
    st = v.device_status()
    n = B * Kmax
    return out["tokens"][:n].cpu().numpy(), out["conf"][:n].cpu().numpy(), st


def _compare(d, u, T, got_t, got_c, want_t, want_c, rows=None):
    """Tokens equal except inside the CDF-boundary band; q(x) within 1e-5.
    Compares the given rows (all by default)."""
    rows = np.arange(got_t.size) if rows is None else np.asarray(rows)
    got_t, got_c, want_t, want_c = got_t[rows], got_c[rows], want_t[rows], want_c[rows].copy()
    exempt = 0
    for k in np.nonzero(got_t != want_t)[0]:
        r = int(rows[k])
        y_g, y_o = int(got_t[k]), int(want_t[k])
        assert T > 0 and y_g >= 0 and y_o >= 0, (r, y_g, y_o)
        st, w = O.softmax_row(d, r, T)
        assert st == O.OK
        _, uS, S = O.inverse_cdf(w, float(u[r]))
        C = np.cumsum(w)
        lo, hi = min(y_g, y_o), max(y_g, y_o)
        near = abs(C[hi - 1] - uS) <= FINAL_BAND * S and abs(C[lo] - uS) <= FINAL_BAND * S
        assert near, (r, y_g, y_o, uS, C[lo], C[hi - 1], S)
        exempt += 1
        want_c[k] = w[y_g]  # q at the GPU's token
    assert exempt <= 2, exempt
    if T == 0:
        assert np.array_equal(got_c, want_c)
    else:
        tiny = want_c < 1e-30
        np.testing.assert_allclose(got_c[~tiny], want_c[~tiny], rtol=1e-5, atol=0)
        assert np.all(np.abs(got_c[tiny] - want_c[tiny]) <= 1e-35)
    return exempt


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("T", [0.0, 0.7, 1.0])
@pytest.mark.parametrize("B,Kmax,V", [
    (2, 4, 50000),    # 8 rows of several slices each, a short last slice
    (5, 3, 1001),     # rows not 16-byte multiples (plain loads), one partial slice
    (16, 16, 32000),
    (64, 8, 128000),  # 512 rows, more rows than resident CTAs
])
def test_draft_sample_against_oracle(B, Kmax, V, T, dtype):
    d, kmax, u = _inputs(B, Kmax, V, dtype, seed=B * 131 + Kmax * 7 + V)
    got_t, got_c, st = _run(d, kmax, u, B, Kmax, V, T)
    assert st == sv.SPEC_OK
    ost, want_t, want_c = O.draft_sample(d, kmax, Kmax, T, u)
    assert ost == O.OK
    live = (np.arange(Kmax)[None, :] < kmax.numpy()[:, None]).reshape(-1)
    assert np.all(got_t[~live] == -1) and np.all(got_c[~live] == 0)
    _compare(d, u, T, got_t, got_c, want_t, want_c)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_draft_greedy_ties_take_the_lowest_index(dtype):
    """T = 0: rows with their maximum repeated take its lowest index, as the
    oracle (and numpy's argmax) do; rows with a NaN are errors."""
    B, Kmax, V = 6, 4, 40000
    g = torch.Generator().manual_seed(51)
    d = torch.randint(-3, 3, (B * Kmax, V), generator=g).float()  # many ties everywhere
    d[5, 31000] = 7.0
    d[5, 12] = 7.0  # lowest of two maxima far apart
    d = d.to(torch.bfloat16 if dtype == "bf16" else torch.float32)
    kmax = torch.full((B,), Kmax, dtype=torch.int32)
    got_t, got_c, st = _run(d, kmax, torch.zeros(B * Kmax), B, Kmax, V, 0.0)
    assert st == sv.SPEC_OK
    want = np.argmax(d.float().numpy(), axis=1)
    assert got_t.tolist() == want.tolist() and got_t[5] == 12
    assert np.all(got_c == 1.0)


def test_draft_sample_follows_u():
    """Over one row drawn at many u, the tokens are non-decreasing in u and
    each token's share of a fine u grid matches q within the grid step."""
    V, T, n = 64, 1.0, 4096
    g = torch.Generator().manual_seed(3)
    row = torch.randn(V, generator=g) * 1.5
    d = row.repeat(n, 1).contiguous()
    kmax = torch.full((n,), 1, dtype=torch.int32)
    u = ((torch.arange(n, dtype=torch.float64) + 0.5) / n).float()
    got_t, got_c, st = _run(d, kmax, u, n, 1, V, T)
    assert st == sv.SPEC_OK
    assert np.all(np.diff(got_t) >= 0)
    _, q = O.softmax_row(d, 0, T)
    share = np.bincount(got_t, minlength=V) / n
    assert np.all(np.abs(share - q) <= 2.0 / n)  # one grid step at each end of a bucket


def test_draft_sample_errors():
    B, Kmax, V = 4, 3, 512
    d, kmax, u = _inputs(B, Kmax, V, "f32", seed=9, full=True)
    d[4, 11] = float("nan")  # request 1, position 1
    got_t, got_c, st = _run(d, kmax, u, B, Kmax, V, 1.0)
    assert st == sv.SPEC_ERR_NONFINITE
    assert got_t[4] == -1 and np.isnan(got_c[4])
    ost, want_t, want_c = O.draft_sample(d, kmax, Kmax, 1.0, u)
    assert ost == O.ERR_NONFINITE
    _compare(d, u, 1.0, got_t, got_c, want_t, want_c, rows=np.delete(np.arange(B * Kmax), 4))
    # kmax outside [0, Kmax]: rows of that request poisoned, status INVALID
    d, kmax, u = _inputs(B, Kmax, V, "f32", seed=10, full=True)
    kmax[2] = Kmax + 1
    got_t, got_c, st = _run(d, kmax, u, B, Kmax, V, 1.0)
    assert st == sv.SPEC_ERR_INVALID_ARG
    assert np.all(got_t[6:9] == -1) and np.all(np.isnan(got_c[6:9]))
    assert np.all(got_t[:6] >= 0) and np.all(got_t[9:] >= 0)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_draft_sample_degenerate_rows(dtype):
    """V = 1 (the only token, q = 1); rows with most entries masked; an
    all-masked row is an error for that row only."""
    d, kmax, u = _inputs(3, 2, 1, dtype, seed=41, full=True)
    got_t, got_c, st = _run(d, kmax, u, 3, 2, 1, 1.0)
    assert st == sv.SPEC_OK
    assert np.all(got_t == 0) and np.allclose(got_c, 1.0, rtol=1e-6)
    B, Kmax, V = 2, 2, 5000
    d, kmax, u = _inputs(B, Kmax, V, dtype, seed=42, full=True)
    g = torch.Generator().manual_seed(43)
    d[torch.rand(d.shape, generator=g) < 0.999] = float("-inf")  # about 5 live entries per row
    d[1, :] = float("-inf")                                     # request 0, position 1: nothing live
    got_t, got_c, st = _run(d, kmax, u, B, Kmax, V, 0.8)
    assert st == sv.SPEC_ERR_NONFINITE
    assert got_t[1] == -1 and np.isnan(got_c[1])
    ost, want_t, want_c = O.draft_sample(d, kmax, Kmax, 0.8, u)
    assert ost == O.ERR_NONFINITE
    _compare(d, u, 0.8, got_t, got_c, want_t, want_c, rows=[0, 2, 3])


def test_draft_sample_empty_and_host_checks():
    v = Verifier(1, 2, 100)
    t = torch.zeros(1, dtype=torch.int32, device="cuda")
    c = torch.zeros(1, device="cuda")
    d = torch.zeros((1, 100), device="cuda")
    assert sv.spec_draft_sample(d, t, 0, 1, 100, 1.0, c, t, c, v.workspace) == sv.SPEC_OK
    k = torch.ones(1, dtype=torch.int32, device="cuda")
    assert sv.spec_draft_sample(d, k, 1, 1, 100, -1.0, c, t, c, v.workspace) == \
        sv.SPEC_ERR_INVALID_ARG
    assert sv.LIB.spec_draft_sample(d.data_ptr(), 0, k.data_ptr(), 1, 1, 100, 1.0, None,
                                    t.data_ptr(), c.data_ptr(), v.workspace.data_ptr(),
                                    v.workspace.numel(), None) == sv.SPEC_ERR_INVALID_ARG


def _stats(accept_len, cu, Kmax):
    v = Verifier(1, 2, 16)
    out = v.acceptance_stats(accept_len.cuda(), cu.cuda(), Kmax, check=False)
    torch.cuda.synchronize()
    st = v.device_status()
    return (out["reached"][:Kmax].cpu().numpy(), out["accepted"][:Kmax].cpu().numpy(),
            float(out["mean"].item()), st)


@pytest.mark.parametrize("B,Kmax,seed", [(1, 1, 0), (7, 5, 1), (256, 16, 2), (4096, 32, 3)])
def test_acceptance_stats_against_oracle(B, Kmax, seed):
    g = torch.Generator().manual_seed(seed)
    k = torch.randint(0, Kmax + 1, (B,), generator=g, dtype=torch.int32)
    a = (torch.rand(B, generator=g) * (k.float() + 1)).floor().to(torch.int32)
    a[torch.rand(B, generator=g) < 0.05] = -1  # poisoned requests are left out
    cu = torch.zeros(B + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(k, 0)
    r, acc, mean, st = _stats(a, cu, Kmax)
    assert st == sv.SPEC_OK
    ost, wr, wa, wm = O.acceptance_stats(a, cu, Kmax)
    assert ost == O.OK
    assert np.array_equal(r, wr) and np.array_equal(acc, wa)
    assert mean == float(np.float32(wm))


def test_acceptance_stats_invalid_and_empty():
    a = torch.tensor([1, 3], dtype=torch.int32)
    cu = torch.tensor([0, 2, 4], dtype=torch.int32)  # request 1 accepts 3 of 2
    r, acc, mean, st = _stats(a, cu, 4)
    assert st == sv.SPEC_ERR_INVALID_ARG
    assert np.all(r == -1) and np.all(acc == -1) and np.isnan(mean)
    assert O.acceptance_stats(a, cu, 4)[0] == O.ERR_INVALID_ARG
    v = Verifier(1, 2, 16)
    m = torch.full((1,), -3.0, device="cuda")
    assert sv.spec_acceptance_stats(None, None, 0, 0, None, None, m, v.workspace) == sv.SPEC_OK
    torch.cuda.synchronize()
    assert m.item() == 0.0 and v.device_status() == sv.SPEC_OK


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_drafting_chain(T):
    """Drafter logits -> drafted tokens and q(x) -> D-cut depths -> verification
    of the drafted tokens -> acceptance statistics, all on the device with no
    host round trip; every stage against the oracle."""
    B, Kmax, V, budget = 24, 8, 32000, 96
    w = W.Workload("draft_chain", B=B, V=V, dtype="bf16", seed=91, kmax=Kmax, budget=budget)
    full = W.make_verify_batch(w, T, "cuda", depths=torch.full((B,), Kmax, dtype=torch.int32),
                               draft_stride=Kmax)
    v = Verifier(B, B * (Kmax + 1), V)
    kmax = torch.full((B,), Kmax, dtype=torch.int32, device="cuda")
    g = torch.Generator().manual_seed(17)
    u = torch.rand(B * Kmax, generator=g).cuda()
    dr = v.draft(full.draft_logits, kmax, Kmax, T, u)
    d = v.dcut(dr["conf"][:B * Kmax].view(B, Kmax), kmax, budget)
    torch.cuda.synchronize()
    ost, want_t, want_c = O.draft_sample(full.draft_logits, kmax, Kmax, T, u)
    assert ost == O.OK
    got_t = dr["tokens"][:B * Kmax].cpu().numpy()
    got_c = dr["conf"][:B * Kmax].cpu().numpy()
    _compare(full.draft_logits, u.cpu(), T, got_t, got_c, want_t, want_c)
    o = O.dcut_allocate(got_c.reshape(B, Kmax), kmax.cpu().numpy(), budget)
    assert d["depth"].cpu().numpy().tolist() == o.depth.tolist()
    batch = W.make_verify_batch(w, T, "cuda", depths=torch.from_numpy(o.depth),
                                draft_stride=Kmax)
    batch.draft_logits = full.draft_logits
    batch.draft_tokens = dr["tokens"][:B * Kmax]
    rows = budget + B
    t = torch.zeros((rows, V), dtype=batch.target_logits.dtype, device="cuda")
    t[:batch.target_logits.shape[0]] = batch.target_logits
    batch.target_logits = t
    out = v.verify(batch, rows, cu_draft=d["cu"])
    stats = v.acceptance_stats(out["accept_len"], d["cu"], Kmax)
    torch.cuda.synchronize()
    assert v.device_status() == sv.SPEC_OK
    rep = parity.compare_batch(batch, out)
    assert rep["exempt_accept"] + rep["exempt_final"] <= 2, rep
    ost, wr, wa, wm = O.acceptance_stats(out["accept_len"].cpu(), d["cu"].cpu(), Kmax)
    assert ost == O.OK
    assert np.array_equal(stats["reached"][:Kmax].cpu().numpy(), wr)
    assert np.array_equal(stats["accepted"][:Kmax].cpu().numpy(), wa)
    assert stats["mean"].item() == float(np.float32(wm))
