"""GPU parity of spec_draft_confidence (q_{i,j}(x_{i,j}) from the drafter's
logits, the per-request prefix confidence D-cut ranks) against the oracle,
and the chained path: drafter logits -> confidence -> D-cut -> verification.

Bar: confidences within 1e-5 relative (as p and q of the verification
path); at T = 0 exactly 0 or 1."""
import numpy as np
import pytest
import torch

import oracle as O
import parity
from draft_verification_02_b300 import specverify as sv
from draft_verification_02_b300 import workloads as W
from draft_verification_02_b300.verifier import Verifier

pytestmark = pytest.mark.gpu


def _inputs(B, Kmax, V, dtype, seed, T):
    g = torch.Generator().manual_seed(seed)
    d = torch.randn((B * Kmax, V), generator=g) * 2.0
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    d = d.to(tdt)
    df = d.float()
    if T > 0:
        gum = -torch.log(-torch.log1p(-torch.rand(df.shape, generator=g, dtype=torch.float64)))
        tok = torch.argmax(df.double() / T + gum, dim=1)
    else:
        tok = torch.argmax(df, dim=1)
        flip = torch.rand(B * Kmax, generator=g) < 0.3  # some drafts off the argmax
        tok = torch.where(flip, (tok + 1) % V, tok)
    kmax = torch.randint(0, Kmax + 1, (B,), generator=g, dtype=torch.int32)
    return d.contiguous(), tok.to(torch.int32).contiguous(), kmax


def _run(d, tok, kmax, B, Kmax, V, T):
    v = Verifier(B, B * (Kmax + 1), V)
    out = torch.full((max(B * Kmax, 1),), -7.0, device="cuda")
    st = sv.spec_draft_confidence(d.cuda(), tok.cuda(), kmax.cuda(), B, Kmax, V, T, out,
                                  v.workspace)
    assert st == sv.SPEC_OK
    torch.cuda.synchronize()
    return out[:B * Kmax].cpu().numpy().reshape(B, Kmax), v


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("T", [0.0, 0.7, 1.0])
@pytest.mark.parametrize("B,Kmax,V", [(3, 4, 1000), (16, 16, 32000), (64, 16, 128000)])
def test_confidence_against_oracle(B, Kmax, V, T, dtype):
    d, tok, kmax = _inputs(B, Kmax, V, dtype, seed=B * 31 + Kmax + V, T=T)
    got, v = _run(d, tok, kmax, B, Kmax, V, T)
    assert v.device_status() == sv.SPEC_OK
    st, want = O.draft_confidence(d, tok, kmax, T)
    assert st == O.OK
    if T == 0:
        assert np.array_equal(got, want)
    else:
        tiny = want < 1e-30
        np.testing.assert_allclose(got[~tiny], want[~tiny], rtol=1e-5, atol=0)
        assert np.all(np.abs(got[tiny] - want[tiny]) <= 1e-35)


def test_confidence_errors_poison_rows():
    B, Kmax, V = 4, 3, 512
    d, tok, kmax = _inputs(B, Kmax, V, "f32", seed=5, T=1.0)
    kmax[:] = Kmax
    d[4, 7] = float("nan")  # request 1, position 1
    tok[9] = V              # request 3, position 0
    got, v = _run(d, tok, kmax, B, Kmax, V, 1.0)
    st = v.device_status()
    assert st == sv.SPEC_ERR_INVALID_ARG  # precedence over NONFINITE
    assert np.isnan(got[1, 1]) and np.isnan(got[3, 0])
    assert np.isfinite(got[0]).all() and np.isfinite(got[2]).all()


def test_confidence_feeds_dcut_and_verification():
    """The drafter's logits give the confidences, D-cut allocates depth from
    them on the device, and the verification reads the offsets D-cut wrote:
    no host round trip, every stage against the oracle."""
    B, Kmax, V, T, budget = 32, 16, 32000, 1.0, 128
    w = W.Workload("chain", B=B, V=V, dtype="bf16", seed=77, kmax=Kmax, budget=budget)
    full = W.make_verify_batch(w, T, "cuda", depths=torch.full((B,), Kmax, dtype=torch.int32),
                               draft_stride=Kmax)
    rows = budget + B
    v = Verifier(B, B * (Kmax + 1), V)
    kmax = torch.full((B,), Kmax, dtype=torch.int32, device="cuda")
    conf = torch.empty(B * Kmax, device="cuda")
    assert sv.spec_draft_confidence(full.draft_logits, full.draft_tokens, kmax, B, Kmax, V, T,
                                    conf, v.workspace) == sv.SPEC_OK
    d = v.dcut(conf.view(B, Kmax), kmax, budget)
    torch.cuda.synchronize()
    st, want_conf = O.draft_confidence(full.draft_logits, full.draft_tokens, kmax, T)
    assert st == O.OK
    np.testing.assert_allclose(conf.cpu().numpy().reshape(B, Kmax), want_conf, rtol=1e-5,
                               atol=1e-35)
    o = O.dcut_allocate(conf.view(B, Kmax).cpu().numpy(), kmax.cpu().numpy(), budget)
    assert d["depth"].cpu().numpy().tolist() == o.depth.tolist()
    depth = torch.from_numpy(o.depth)
    # the verification batch: target rows for the chosen depths, drafts padded to Kmax
    batch = W.make_verify_batch(w, T, "cuda", depths=depth, draft_stride=Kmax)
    batch.draft_logits = full.draft_logits
    batch.draft_tokens = full.draft_tokens
    t = torch.zeros((rows, V), dtype=batch.target_logits.dtype, device="cuda")
    t[:batch.target_logits.shape[0]] = batch.target_logits
    batch.target_logits = t
    out = v.verify(batch, rows, cu_draft=d["cu"])
    torch.cuda.synchronize()
    assert v.device_status() == sv.SPEC_OK
    rep = parity.compare_batch(batch, out)
    assert rep["exempt_accept"] + rep["exempt_final"] <= 2, rep
