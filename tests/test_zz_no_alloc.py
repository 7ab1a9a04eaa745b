"""spec_verify_sample_static: verification for callers that cannot allocate
device memory (an engine whose pool owns all of HBM, a plugin whose host
runtime forbids outside allocations).  It uses the library's fixed scratch
array instead of a workspace; its results must equal spec_verify_sample's on
the same inputs, call after call, since every call reuses that one array.

This file is collected last on purpose, so that a run which stops at the
first failure has already run every other test."""
import pytest
import torch

from draft_verification_02_b300 import specverify as sv
from draft_verification_02_b300 import workloads as W
from draft_verification_02_b300.verifier import Verifier

pytestmark = pytest.mark.gpu

P_RTOL = 1e-5  # the parity tests' bar for p and q


def _batch(seed, T, B, V, dtype="bf16"):
    g = torch.Generator().manual_seed(seed)
    k = torch.randint(0, 17, (B,), generator=g, dtype=torch.int32)
    w = W.Workload("no_alloc", B=B, V=V, dtype=dtype, seed=seed, k_range=(0, 16))
    return W.make_verify_batch(w, T, "cuda", depths=k)


def _outputs(b):
    nd = max(b.draft_tokens.numel(), 1)
    return {"tokens": torch.full((b.n_target_rows,), -7, dtype=torch.int32, device="cuda"),
            "accept_len": torch.full((b.B,), -7, dtype=torch.int32, device="cuda"),
            "p": torch.full((nd,), float("nan"), device="cuda"),
            "q": torch.full((nd,), float("nan"), device="cuda")}


def _static_call(b, o):
    return sv.spec_verify_sample_static(
        b.target_logits, b.draft_logits, b.draft_tokens, b.cu_draft, b.B, b.V,
        b.n_target_rows, b.draft_stride, b.temperature, b.u_accept, b.u_final, o["tokens"],
        o["accept_len"], o["p"], o["q"])


def test_static_scratch_matches_workspace_entry_point_on_consecutive_calls():
    # two different batches in a row (sampling, then greedy, then sampling at
    # another vocabulary), so each call starts from the previous call's scratch
    cases = [(31, 1.0, 24, 32000), (32, 0.0, 16, 128000), (33, 0.7, 40, 151936)]
    for seed, T, B, V in cases:
        b = _batch(seed, T, B, V)
        ref = Verifier(b.B, b.n_target_rows, b.V).verify(b)
        o = _outputs(b)
        assert _static_call(b, o) == sv.SPEC_OK
        torch.cuda.synchronize()
        assert torch.equal(o["accept_len"], ref["accept_len"]), (seed, T)
        assert torch.equal(o["tokens"], ref["tokens"]), (seed, T)
        assert bool((o["accept_len"] >= 0).all())
        if T > 0:
            n = b.draft_tokens.numel()
            torch.testing.assert_close(o["p"][:n], ref["p"][:n], rtol=P_RTOL, atol=0)
            torch.testing.assert_close(o["q"][:n], ref["q"][:n], rtol=P_RTOL, atol=0)


def test_static_scratch_rejects_sizes_beyond_its_array():
    B, V = 4096, 151936
    rows = B * 17
    need = sv.spec_workspace_size(B, rows, V)
    assert need > sv.SPEC_STATIC_SCRATCH_BYTES
    t = torch.zeros((1, 16), dtype=torch.bfloat16, device="cuda")
    i32 = torch.zeros(16, dtype=torch.int32, device="cuda")
    f32 = torch.zeros(16, dtype=torch.float32, device="cuda")
    # the library checks sizes before touching any buffer, so small stand-in
    # tensors are enough: nothing is enqueued
    st = sv.LIB.spec_verify_sample_static(
        t.data_ptr(), t.data_ptr(), sv.SPEC_BF16, i32.data_ptr(), i32.data_ptr(), B, V, rows, 0,
        1.0, f32.data_ptr(), f32.data_ptr(), i32.data_ptr(), i32.data_ptr(), None, None, None)
    assert st == sv.SPEC_ERR_WORKSPACE
    torch.cuda.synchronize()


def test_static_scratch_data_error_then_clean_call_against_the_oracle():
    """A request with a NaN logit is poisoned (accepted length -1, tokens -1)
    and the others match the oracle; the next call on clean inputs starts
    from the scratch the failed call left and matches the oracle everywhere."""
    import parity
    b = _batch(41, 1.0, 12, 32000)
    bad = 5
    row = int(b.cu_draft[bad]) + bad  # request 5's first target row
    b.target_logits[row, 123] = float("nan")
    o = _outputs(b)
    assert _static_call(b, o) == sv.SPEC_OK
    torch.cuda.synchronize()
    assert int(o["accept_len"][bad]) == -1
    K = int(b.k[bad])
    assert bool((o["tokens"][row:row + K + 1] == -1).all())
    good = [i for i in range(b.B) if i != bad]
    rep = parity.compare_batch(b, o, good)
    assert rep["exempt_accept"] + rep["exempt_final"] <= 2, rep
    clean = _batch(42, 1.0, 12, 32000)
    o2 = _outputs(clean)
    assert _static_call(clean, o2) == sv.SPEC_OK
    torch.cuda.synchronize()
    assert bool((o2["accept_len"] >= 0).all())
    rep = parity.compare_batch(clean, o2)
    assert rep["exempt_accept"] + rep["exempt_final"] <= 2, rep
