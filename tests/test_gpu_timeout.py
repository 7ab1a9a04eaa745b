"""The timeout path of the verification kernels, without a GPU fault.

spec_test_expire_wait(unit) makes the streaming pass treat the bounded wait
for one unit's copy as expired once that copy has landed: the expiry branch
runs (status flag, one more bounded wait for every copy still in flight,
the warp stops) and nothing is left in flight.  The finish kernel then
poisons every output.  The test checks the status the host reads, the
poisoned outputs, and that a call after re-zeroing the workspace is correct
again."""
import pytest
import torch

from draft_verification_02_b300 import specverify as sv
from draft_verification_02_b300 import workloads as W
from draft_verification_02_b300.verifier import Verifier
import parity


@pytest.mark.gpu
@pytest.mark.parametrize("T", [0.0, 1.0])
@pytest.mark.parametrize("unit", [0, 37])
def test_expired_wait_flags_timeout_poisons_and_recovers(T, unit):
    batch = W.make_verify_batch(W.MTP, T, "cuda")  # bf16 rows of 256000 bytes: bulk copies
    v = Verifier(batch.B, batch.n_target_rows, batch.V)
    assert sv.spec_test_expire_wait(unit) == sv.SPEC_OK
    try:
        out = v.verify(batch, check=False)
    finally:
        assert sv.spec_test_expire_wait(-1) == sv.SPEC_OK
    torch.cuda.synchronize()
    assert out["status"] == sv.SPEC_OK  # the launch itself succeeded
    assert v.device_status() == sv.SPEC_ERR_TIMEOUT
    assert (out["accept_len"] == -1).all()
    assert (out["tokens"] == -1).all()
    # after a timeout the workspace is zeroed again, as the header says
    sv.check(sv.spec_workspace_init(v.workspace), "workspace init")
    out2 = v.verify(batch)
    torch.cuda.synchronize()
    assert v.device_status() == sv.SPEC_OK
    rep = parity.compare_batch(batch, out2)
    assert rep["exempt_accept"] + rep["exempt_final"] <= 2


@pytest.mark.gpu
def test_expiry_hook_is_off_by_default():
    batch = W.make_verify_batch(W.TINY, 1.0, "cuda")
    v = Verifier(batch.B, batch.n_target_rows, batch.V)
    out = v.verify(batch)
    torch.cuda.synchronize()
    assert v.device_status() == sv.SPEC_OK
    assert (out["accept_len"] >= 0).all()
