"""GPU parity of vocabulary-sharded verification: a batch's logits split into
N column ranges (what the ranks of a tensor-parallel target hold), verified
shard by shard on one device through the C ABI (the exchanges stood in for
by stacking and an element-wise max), against the oracle on the whole
vocabulary.  Same bar as tests/parity.py; every shard must end with the same
outputs bit for bit."""
import numpy as np
import pytest
import torch

import parity
from draft_verification_02_b300 import specverify as sv
from draft_verification_02_b300 import workloads as W
from draft_verification_02_b300.sharded import (Shard, shard_bounds, shard_columns,
                                                verify_sharded_local)
from test_gpu_verify import MAX_EXEMPT, pad_to_loose_bound, ragged_batch

pytestmark = pytest.mark.gpu


def run_sharded(batch, bounds, rows=None):
    batch = batch.to("cuda")
    rows = rows or batch.n_target_rows
    T = batch.temperature
    shards = [Shard(batch.B, rows, bounds, r, batch.draft_stride)
              for r in range(len(bounds) - 1)]
    targets = shard_columns(batch.target_logits, bounds)
    drafts = shard_columns(batch.draft_logits if T > 0 else None, bounds)
    outs = verify_sharded_local(shards, targets, drafts, batch.draft_tokens, batch.cu_draft, T,
                                batch.u_accept, batch.u_final)
    torch.cuda.synchronize()
    status = [sv.spec_get_device_status(s.workspace) for s in shards]
    return batch, outs, status


def assert_shards_agree(outs):
    for o in outs[1:]:
        for k in ("tokens", "accept_len", "p", "q"):
            torch.testing.assert_close(o[k], outs[0][k], rtol=0, atol=0, equal_nan=True)


def check_sharded(batch, bounds, reqs=None, max_exempt=MAX_EXEMPT):
    batch, outs, status = run_sharded(batch, bounds)
    assert status == [sv.SPEC_OK] * (len(bounds) - 1)
    assert_shards_agree(outs)
    rep = parity.compare_batch(batch, outs[0], reqs)
    assert rep["exempt_accept"] + rep["exempt_final"] <= max_exempt, rep
    return batch, outs


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [0.0, 0.7, 1.0])
@pytest.mark.parametrize("V,N", [(1000, 1), (4099, 2), (12345, 3), (40000, 8), (32000, 4)])
def test_sharded_matches_oracle(V, N, T, dtype):
    """Ragged depths 0..32 with empty requests; uneven shard widths (4099 /
    2, 12345 / 3) whose rows are not 16-byte multiples take the plain-load
    path of the streaming pass and the draw."""
    b = ragged_batch(8, V, T, dtype, seed=V + 31 * N + int(T * 10), kmax=32)
    check_sharded(b, shard_bounds(V, N))


@pytest.mark.parametrize("T", [0.0, 0.7])
def test_sharded_padded_draft_layout(T):
    b = ragged_batch(9, 5000, T, "bf16", seed=13, kmax=8, draft_stride=8)
    check_sharded(b, shard_bounds(5000, 4))


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_drafted_tokens_at_shard_boundaries(T):
    """Drafted tokens on the first and last column of every shard: the
    shard holding each one supplies its logit; at T = 0 the target's maxima
    are put there too, so the drafts are accepted across shards."""
    V, N = 6000, 3
    bounds = shard_bounds(V, N)
    edges = sorted({v for r in range(N) for v in (bounds[r], bounds[r + 1] - 1)})
    b = ragged_batch(6, V, T, "f32", seed=17, kmin=3, kmax=6)
    for n in range(b.draft_tokens.numel()):
        b.draft_tokens[n] = edges[n % len(edges)]
    if T == 0:
        for i in range(b.B):
            K, t0, d0 = int(b.k[i]), int(b.cu_draft[i]) + i, int(b.cu_draft[i])
            for j in range(K - 1):  # accept all but the last draft
                b.target_logits[t0 + j, b.draft_tokens[d0 + j].long()] = 50.0
    _, outs = check_sharded(b, bounds)
    if T == 0:
        assert torch.all(outs[0]["accept_len"].cpu() >= torch.clamp(b.k - 1, min=0))


def test_greedy_ties_across_shards_take_the_lowest_index():
    """Equal maxima in two shards (and twice inside one shard): the lowest
    global index wins, as in the unsharded verification."""
    V, N = 4096, 4
    bounds = shard_bounds(V, N)
    b = ragged_batch(4, V, 0.0, "f32", seed=19, kmin=2, kmax=4)
    rows = b.target_logits.shape[0]
    for r in range(rows):
        lo, hi = bounds[1] + 5 + r, bounds[3] + 7
        b.target_logits[r, hi] = 30.0
        b.target_logits[r, lo] = 30.0
        b.target_logits[r, lo + 1] = 30.0
    _, outs = check_sharded(b, bounds)
    tok = outs[0]["tokens"].cpu()
    for i in range(b.B):
        a = int(outs[0]["accept_len"][i])
        t0 = int(b.cu_draft[i]) + i
        assert int(tok[t0 + a]) == bounds[1] + 5 + t0 + a


def test_identical_rows_accept_everything_sharded():
    b = ragged_batch(8, 3000, 0.8, "bf16", seed=6, kmin=1, kmax=10)
    for i in range(8):
        K = int(b.k[i])
        t0, d0 = int(b.cu_draft[i]) + i, int(b.cu_draft[i])
        b.draft_logits[d0:d0 + K] = b.target_logits[t0:t0 + K]
    b.u_accept[:] = 1.0 - 2.0 ** -16
    batch, outs = check_sharded(b, shard_bounds(3000, 3))
    assert torch.equal(outs[0]["accept_len"].cpu(), b.k)


def test_final_draws_come_from_several_shards():
    """Flat target rows and concentrated drafts: rejections are common and
    the residual mass spreads over the whole vocabulary, so the drawing
    shard varies from request to request."""
    V, N = 8000, 4
    bounds = shard_bounds(V, N)
    b = ragged_batch(24, V, 1.0, "f32", seed=23, kmin=1, kmax=3, sigma=0.1, noise=4.0)
    _, outs = check_sharded(b, bounds)
    tok = outs[0]["tokens"].cpu()
    owners = set()
    for i in range(b.B):
        a = int(outs[0]["accept_len"][i])
        y = int(tok[int(b.cu_draft[i]) + i + a])
        owners.add(int(np.searchsorted(bounds, y, side="right")) - 1)
    assert len(owners) >= 3, owners


def test_nonfinite_in_one_shard_poisons_only_its_request():
    V, N = 5000, 4
    bounds = shard_bounds(V, N)
    b = ragged_batch(6, V, 1.0, "bf16", seed=29, kmin=2, kmax=5)
    bad = 3
    t0 = int(b.cu_draft[bad]) + bad
    b.target_logits[t0 + 1, bounds[2] + 9] = float("nan")
    batch, outs, status = run_sharded(b, bounds)
    assert_shards_agree(outs)
    # every shard sees the NaN in the gathered records and poisons alike
    assert status == [sv.SPEC_ERR_NONFINITE] * N
    assert int(outs[0]["accept_len"][bad]) == -1
    K = int(b.k[bad])
    assert bool((outs[0]["tokens"][t0:t0 + K + 1] == -1).all())
    good = [i for i in range(b.B) if i != bad]
    parity.compare_batch(batch, outs[0], good)


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_malformed_offsets_poison_everything_sharded(T):
    """Decreasing offsets: every shard's row pass flags them and every
    shard poisons every output; the same shards then verify a clean batch."""
    V, N = 3000, 2
    bounds = shard_bounds(V, N)
    b = ragged_batch(5, V, T, "f32", seed=31, kmin=1, kmax=3).to("cuda")
    rows = b.n_target_rows
    shards = [Shard(b.B, rows, bounds, r) for r in range(N)]
    targets = shard_columns(b.target_logits, bounds)
    drafts = shard_columns(b.draft_logits if T > 0 else None, bounds)
    bad_cu = b.cu_draft.clone()
    bad_cu[2] = bad_cu[1] - 1
    outs = verify_sharded_local(shards, targets, drafts, b.draft_tokens, bad_cu, T,
                                b.u_accept, b.u_final)
    torch.cuda.synchronize()
    assert [sv.spec_get_device_status(s.workspace) for s in shards] == [sv.SPEC_ERR_INVALID_ARG] * N
    for o in outs:
        assert bool((o["accept_len"] == -1).all())
        assert bool((o["tokens"] == -1).all())
    outs = verify_sharded_local(shards, targets, drafts, b.draft_tokens, b.cu_draft, T,
                                b.u_accept, b.u_final)
    torch.cuda.synchronize()
    assert [sv.spec_get_device_status(s.workspace) for s in shards] == [sv.SPEC_OK] * N
    assert_shards_agree(outs)
    parity.compare_batch(b, outs[0])


def test_tp8_large_vocabulary_sampled():
    """The largest configuration's shape (B = 128, V = 151936, K_i ~ U{1..16},
    T = 0.7) split as a TP = 8 target would be (8 x 18992 columns); requests
    sampled for the oracle."""
    w = W.get("ragged17")
    b = W.make_verify_batch(w, 0.7, "cuda", depths=W.make_depths(w, "cpu", 0))
    reqs = list(range(0, w.B, 11))
    check_sharded(b, shard_bounds(w.V, 8), reqs=reqs)


def test_repeat_calls_are_bit_identical_sharded():
    b = ragged_batch(10, 20000, 0.9, "bf16", seed=37, kmax=12).to("cuda")
    bounds = shard_bounds(20000, 4)
    _, first, _ = run_sharded(b, bounds)
    _, again, _ = run_sharded(b, bounds)
    for k in ("tokens", "accept_len", "p", "q"):
        torch.testing.assert_close(again[0][k], first[0][k], rtol=0, atol=0, equal_nan=True)


@pytest.mark.parametrize("T", [0.0, 0.9])
def test_sharded_loose_row_bound(T):
    """A host bound far above the real rows (NaN past them): each shard's
    streaming pass re-splits the real rows and its row merge follows."""
    B, V = 10, 9000
    b = pad_to_loose_bound(ragged_batch(B, V, T, "f32", seed=43, kmax=6), B * 20)
    batch, outs, status = run_sharded(b, shard_bounds(V, 3), rows=B * 20)
    assert status == [sv.SPEC_OK] * 3
    assert_shards_agree(outs)
    parity.compare_batch(batch, outs[0])


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_expired_wait_on_one_shard_flags_it_and_poisons_its_outputs(T):
    """The forced-expiry hook on shard 0's streaming pass: shard 0's status
    says TIMEOUT and its accept step poisons every output it holds (the other
    shards cannot see it, so the verification's outputs are unspecified, as
    the header states); after its workspace is zeroed the same shards verify
    correctly."""
    V, N = 12000, 2
    bounds = shard_bounds(V, N)
    b = ragged_batch(6, V, T, "bf16", seed=47, kmin=2, kmax=6).to("cuda")
    rows = b.n_target_rows
    shards = [Shard(b.B, rows, bounds, r) for r in range(N)]
    targets = shard_columns(b.target_logits, bounds)
    drafts = shard_columns(b.draft_logits if T > 0 else None, bounds)
    outs = [s.outputs() for s in shards]
    assert sv.spec_test_expire_wait(3) == sv.SPEC_OK
    try:
        recs0 = shards[0].row_stats(targets[0], drafts[0], b.draft_tokens, b.cu_draft, T).clone()
    finally:
        assert sv.spec_test_expire_wait(-1) == sv.SPEC_OK
    recs1 = shards[1].row_stats(targets[1], drafts[1], b.draft_tokens, b.cu_draft, T).clone()
    rows_all = torch.stack([recs0, recs1])
    shards[0].accept(rows_all, b.draft_tokens, b.cu_draft, T, b.u_accept, outs[0])
    torch.cuda.synchronize()
    assert sv.spec_get_device_status(shards[0].workspace) == sv.SPEC_ERR_TIMEOUT
    assert bool((outs[0]["accept_len"] == -1).all())
    assert bool((outs[0]["tokens"] == -1).all())
    sv.check(sv.spec_workspace_init(shards[0].workspace), "workspace init")
    sv.check(sv.spec_workspace_init(shards[1].workspace), "workspace init")
    outs = verify_sharded_local(shards, targets, drafts, b.draft_tokens, b.cu_draft, T,
                                b.u_accept, b.u_final)
    torch.cuda.synchronize()
    assert [sv.spec_get_device_status(s.workspace) for s in shards] == [sv.SPEC_OK] * N
    parity.compare_batch(b, outs[0])


@pytest.mark.parametrize("T", [0.0, 0.8])
def test_distributed_driver_over_nccl_with_one_rank(T):
    """verify_sharded with its real exchanges (torch.distributed over NCCL
    on this GPU) in a group of one rank holding the whole vocabulary: the
    all-gathers and the max all-reduce run on device tensors, and the
    result is the oracle's."""
    import torch.distributed as dist
    from draft_verification_02_b300.sharded import DistExchange, verify_sharded
    V = 9000
    b = ragged_batch(8, V, T, "bf16", seed=53, kmax=8).to("cuda")
    dist.init_process_group("nccl", store=dist.HashStore(), rank=0, world_size=1,
                            device_id=torch.device("cuda", 0))
    try:
        shard = Shard(b.B, b.n_target_rows, [0, V], 0)
        out = verify_sharded(shard, DistExchange(), b.target_logits,
                             b.draft_logits if T > 0 else None, b.draft_tokens, b.cu_draft, T,
                             b.u_accept, b.u_final)
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    assert sv.spec_get_device_status(shard.workspace) == sv.SPEC_OK
    rep = parity.compare_batch(b, out)
    assert rep["exempt_accept"] + rep["exempt_final"] <= MAX_EXEMPT, rep
