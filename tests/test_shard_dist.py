"""The sharded verification driver on CPU: its exchanges across world-size-2
gloo ranks (draft_verification_02_b300.sharded.verify_sharded over
torch.distributed), and the one-device driver.  A shard's four kernel calls
are stood in for by an fp64 numpy model with the same tensors and the same
semantics (records of 4 numbers per row, masses of 4 per request), written
from the definitions: per-shard softmax statistics merged by the log-sum-exp
rule, p(x) from the shard that holds x, the accept test u < p/q, and the
inverse CDF of max(0, p - q) walked shard by shard.  So what is tested here is
the driver: the order of the steps, the shard order of every gathered tensor
and the final element-wise max; the result must equal the oracle's
verification over the whole vocabulary."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle as O
from draft_verification_02_b300 import workloads as W
from draft_verification_02_b300.sharded import shard_bounds, verify_sharded, verify_sharded_local

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


class ModelShard:
    """fp64 model of draft_verification_02_b300.sharded.Shard (packed draft
    layout).  Records: [m, gx or global argmax, s, 0] with s = sum
    exp((l - m) / T) over the shard's columns; masses: [sum w, 0, sum p, 0]."""

    def __init__(self, B, max_rows, bounds, r):
        self.B, self.max_rows, self.bounds, self.r = B, max_rows, list(bounds), r
        self.vb, self.ve = bounds[r], bounds[r + 1]
        self.state = {}

    def outputs(self):
        nd = max(self.max_rows - self.B, 1)
        return {"tokens": torch.full((self.max_rows,), -7, dtype=torch.int32),
                "accept_len": torch.full((self.B,), -7, dtype=torch.int32),
                "p": torch.full((nd,), float("nan"), dtype=torch.float64),
                "q": torch.full((nd,), float("nan"), dtype=torch.float64)}

    def _requests(self, cu):
        for i in range(self.B):
            yield i, int(cu[i]), int(cu[i + 1]) - int(cu[i])

    def row_stats(self, target, draft, tokens, cu, T):
        t = target.double().numpy()
        d = draft.double().numpy() if draft is not None else None
        tok, cu = tokens.numpy(), cu.numpy()
        rec = np.zeros((self.max_rows + self.max_rows - self.B, 4))

        def stats(row, x):
            m = row.max()
            if T == 0:
                return [m, self.vb + int(np.argmax(row)), 0.0, 0.0]
            s = np.exp((row - m) / T).sum()
            owned = x is not None and self.vb <= x < self.ve
            return [m, row[x - self.vb] if owned else 0.0, s, 0.0]
        for i, c, K in self._requests(cu):
            t0 = c + i
            for j in range(K + 1):
                rec[t0 + j] = stats(t[t0 + j], int(tok[c + j]) if j < K else None)
            if T > 0:
                for j in range(K):
                    rec[self.max_rows + c + j] = stats(d[c + j], int(tok[c + j]))
        return torch.from_numpy(rec)

    def accept(self, rows_all, tokens, cu, T, u_accept, out):
        R = rows_all.numpy()
        tok, cu = tokens.numpy(), cu.numpy()
        ua = u_accept.numpy() if u_accept is not None else None
        N = len(self.bounds) - 1
        for i, c, K in self._requests(cu):
            t0 = c + i
            if T == 0:
                g = []
                for j in range(K + 1):
                    vals = R[:, t0 + j, 0]
                    best = vals.max()
                    g.append(int(min(R[r, t0 + j, 1] for r in range(N) if vals[r] == best)))
                a = next((j for j in range(K) if int(tok[c + j]) != g[j]), K)
                row = [int(tok[c + j]) if j < a else (g[a] if j == a else -1)
                       for j in range(K + 1)]
            else:
                def merged(rec):
                    m = R[:, rec, 0].max()
                    return m, float((R[:, rec, 2] * np.exp((R[:, rec, 0] - m) / T)).sum())

                def prob(rec, x):
                    m, s = merged(rec)
                    owner = int(np.searchsorted(self.bounds, x, side="right")) - 1
                    return np.exp((R[owner, rec, 1] - m) / T) / s
                a = K
                for j in range(K):
                    x = int(tok[c + j])
                    p, q = prob(t0 + j, x), prob(self.max_rows + c + j, x)
                    out["p"][c + j], out["q"][c + j] = p, q
                    if a == K and not ua[c + j] < (p / q if q > 0 else (np.inf if p > 0 else 0)):
                        a = j
                row = [int(tok[c + j]) if j < a else -1 for j in range(K + 1)]
                self.state[i] = (a, K, t0, merged(t0 + a),
                                 merged(self.max_rows + c + a) if a < K else None, c)
            out["tokens"][t0:t0 + K + 1] = torch.tensor(row, dtype=torch.int32)
            out["accept_len"][i] = a

    def _weights(self, target, draft, i, T):
        a, K, t0, (mt, st), dstat, c = self.state[i]
        p = np.exp((target[t0 + a].double().numpy() - mt) / T) / st
        if dstat is None:
            return p, p
        md, sd = dstat
        q = np.exp((draft[c + a].double().numpy() - md) / T) / sd
        return np.maximum(p - q, 0.0), p

    def final_mass(self, target, draft):
        T = self.T
        m = np.zeros((self.B, 4))
        for i in range(self.B):
            w, p = self._weights(target, draft, i, T)
            m[i] = [w.sum(), 0.0, p.sum(), 0.0]
        return torch.from_numpy(m)

    def final_draw(self, target, draft, mass_all, u_final, out_tokens):
        T = self.T
        M = mass_all.numpy()
        for i in range(self.B):
            a, K, t0 = self.state[i][:3]
            col = 0
            if a < K and M[:, i, 0].sum() == 0:
                col = 2  # an all-zero residual: draw from p
            cum = np.cumsum(M[:, i, col])
            tgt = float(u_final[i]) * cum[-1]
            hit = np.nonzero(cum > tgt)[0]
            owner = int(hit[0]) if len(hit) else int(np.nonzero(M[:, i, col] > 0)[0][-1])
            if owner != self.r:
                out_tokens[t0 + a] = -1
                continue
            w, p = self._weights(target, draft, i, T)
            w = p if col == 2 else w
            base = cum[owner - 1] if owner > 0 else 0.0
            c = base + np.cumsum(w)
            k = np.nonzero(c > tgt)[0]
            v = int(k[0]) if len(k) else int(np.nonzero(w > 0)[0][-1])
            out_tokens[t0 + a] = self.vb + v


def _batch(T, V, B=6, seed=3):
    g = torch.Generator().manual_seed(seed)
    k = torch.randint(0, 9, (B,), generator=g, dtype=torch.int32)
    w = W.Workload("shard_cpu", B=B, V=V, dtype="f32", seed=seed, k_range=(0, 8))
    return W.make_verify_batch(w, T, "cpu", depths=k)


def _oracle(b):
    h = {"target": b.target_logits.numpy(), "draft": b.draft_logits.numpy(),
         "tokens": b.draft_tokens.numpy(), "cu": b.cu_draft.numpy()}
    if b.temperature == 0:
        return O.verify_greedy(h["target"], h["tokens"], h["cu"])
    return O.verify_sample(h["target"], h["draft"], h["tokens"], h["cu"], b.temperature,
                           b.u_accept.numpy(), b.u_final.numpy())


def _check(b, out):
    o = _oracle(b)
    assert out["accept_len"].tolist() == o.accept_len.tolist()
    assert out["tokens"].tolist() == o.tokens.tolist()
    if b.temperature > 0:
        nd = b.draft_tokens.numel()
        np.testing.assert_allclose(out["p"][:nd].numpy(), o.p, rtol=1e-6, atol=0)  # oracle p, q: fp32
        np.testing.assert_allclose(out["q"][:nd].numpy(), o.q, rtol=1e-6, atol=0)


def _shards(b, bounds):
    shards = []
    for r in range(len(bounds) - 1):
        s = ModelShard(b.B, b.n_target_rows, bounds, r)
        s.T = b.temperature
        shards.append(s)
    cols = [slice(bounds[r], bounds[r + 1]) for r in range(len(bounds) - 1)]
    targets = [b.target_logits[:, c] for c in cols]
    drafts = [b.draft_logits[:, c] if b.temperature > 0 else None for c in cols]
    return shards, targets, drafts


@pytest.mark.parametrize("T", [0.0, 0.7, 1.0])
@pytest.mark.parametrize("N", [1, 3])
def test_local_driver_with_model_shards_equals_the_oracle(T, N):
    b = _batch(T, 997, seed=5 + N)
    shards, targets, drafts = _shards(b, shard_bounds(997, N))
    outs = verify_sharded_local(shards, targets, drafts, b.draft_tokens, b.cu_draft, T,
                                b.u_accept, b.u_final)
    for o in outs:
        _check(b, o)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q, T, V):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import torch.distributed as dist
    from draft_verification_02_b300.sharded import DistExchange
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _batch(T, V, seed=11)  # the same seeded batch on every rank
        bounds = shard_bounds(V, world)
        shard = ModelShard(b.B, b.n_target_rows, bounds, rank)
        shard.T = T
        c = slice(bounds[rank], bounds[rank + 1])
        out = verify_sharded(shard, DistExchange(), b.target_logits[:, c].contiguous(),
                             b.draft_logits[:, c].contiguous() if T > 0 else None,
                             b.draft_tokens, b.cu_draft, T, b.u_accept, b.u_final)
        q.put((rank, {k: v.clone() for k, v in out.items()}))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_two_gloo_ranks_exchange_records_and_agree_with_the_oracle(T):
    world, V = 2, 1001  # uneven shards: 501 + 500 columns
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q, T, V)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=180) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    b = _batch(T, V, seed=11)
    for r in range(world):
        _check(b, res[r])
    assert res[0]["tokens"].tolist() == res[1]["tokens"].tolist()


def test_shard_bounds_and_columns():
    """The vocabulary split: contiguous ranges in shard order covering [0, V)
    with widths differing by at most one (the first V % N one wider), every
    count from 1 to the limit, refused beyond it or beyond V; each shard's
    columns put side by side give the logits back."""
    from draft_verification_02_b300 import specverify as sv
    from draft_verification_02_b300.sharded import shard_columns
    for V in (1, 2, 7, 1000, 18992, 151936):
        for n in range(1, min(V, sv.SPEC_MAX_SHARDS) + 1):
            b = shard_bounds(V, n)
            w = np.diff(b)
            assert b[0] == 0 and b[-1] == V and len(b) == n + 1
            assert w.min() >= 1 and w.max() - w.min() <= 1
            assert (w[:V % n] == w.max()).all() and (w[V % n:] == V // n).all()
        for bad in (0, min(V, sv.SPEC_MAX_SHARDS) + 1):
            with pytest.raises(ValueError):
                shard_bounds(V, bad)
    x = torch.randn(5, 1003)
    for n in (1, 3, 8):
        b = shard_bounds(1003, n)
        cols = shard_columns(x, b)
        assert all(c.is_contiguous() and c.shape == (5, b[r + 1] - b[r])
                   for r, c in enumerate(cols))
        assert torch.equal(torch.cat(cols, dim=1), x)
    assert shard_columns(None, shard_bounds(10, 2)) == [None, None]
