"""Vocabulary-sharded verification: one shard's four calls of the C ABI, and
the drivers that run them with the exchanges in between.

A target served tensor-parallel splits its output projection by vocabulary
(TP = 8 in "Tencent Hunyuan Turns Speculative Decoding Into a Full Open-Source
Stack", "Key numbers (Hy3-295B-A21B, TP=8)"), so each rank holds its own
columns of every logit row.  Each rank reduces those columns (spec_shard_*);
between the calls only small records cross ranks:

  1. row_stats    -> 16 bytes per row          all-gather (shard order)
  2. accept       (the same on every rank; T = 0 ends here)
  3. final_mass   -> 16 bytes per request      all-gather (shard order)
  4. final_draw   -> the drawing rank's token   element-wise max of out_tokens

verify_sharded runs one rank's part over a torch.distributed group (NCCL on
GPUs; the collectives are plain all_gather / all_reduce of small tensors).
verify_sharded_local runs several shards held on one device, with stacking
and an element-wise max standing in for the collectives.  Nothing here
computes: every step of the verification runs in the library's kernels.
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import torch

from . import specverify as sv


def shard_bounds(V: int, n_shards: int) -> List[int]:
    """Contiguous, near-equal vocabulary ranges (the first V % n get one more)."""
    if not 1 <= n_shards <= min(V, sv.SPEC_MAX_SHARDS):
        raise ValueError(f"cannot split V={V} into {n_shards} shards")
    base, extra = divmod(V, n_shards)
    out = [0]
    for r in range(n_shards):
        out.append(out[-1] + base + (1 if r < extra else 0))
    return out


def shard_columns(logits: Optional[torch.Tensor], shard_begin: Sequence[int]) -> list:
    """Each shard's columns of a [rows, V] logit tensor as contiguous tensors
    (what each rank of a tensor-parallel group holds)."""
    n = len(shard_begin) - 1
    if logits is None:
        return [None] * n
    return [logits[:, shard_begin[r]:shard_begin[r + 1]].contiguous() for r in range(n)]


class Shard:
    """One shard's workspace and exchange buffers, for up to B requests and
    max_target_rows rows; its columns are [shard_begin[shard], shard_begin[shard + 1])."""

    def __init__(self, B: int, max_target_rows: int, shard_begin: Sequence[int], shard: int,
                 draft_stride: int = 0, device="cuda"):
        self.B, self.max_target_rows, self.draft_stride = B, max_target_rows, draft_stride
        self.shard_begin = [int(v) for v in shard_begin]
        self.n_shards = len(self.shard_begin) - 1
        self.shard = shard
        self.v_begin, self.v_end = self.shard_begin[shard], self.shard_begin[shard + 1]
        self.device = torch.device(device)
        nbytes = sv.spec_shard_workspace_size(B, max_target_rows, self.v_end - self.v_begin)
        n_rec = sv.spec_shard_row_count(B, max_target_rows, draft_stride)
        if nbytes == 0 or n_rec < 0:
            raise ValueError("invalid shard sizes")
        # zero-filled: the workspace's first-use rule
        self.workspace = torch.zeros(nbytes, dtype=torch.uint8, device=self.device)
        self.rows = torch.zeros((n_rec, sv.SHARD_RECORD_FLOATS), dtype=torch.float32,
                                device=self.device)
        self.mass = torch.zeros((max(B, 1), sv.SHARD_RECORD_FLOATS), dtype=torch.float32,
                                device=self.device)

    def outputs(self) -> dict:
        nd = max(self.B * self.draft_stride if self.draft_stride else
                 self.max_target_rows - self.B, 1)
        dev = self.device
        return {
            "tokens": torch.full((self.max_target_rows,), -7, dtype=torch.int32, device=dev),
            "accept_len": torch.full((self.B,), -7, dtype=torch.int32, device=dev),
            "p": torch.full((nd,), float("nan"), dtype=torch.float32, device=dev),
            "q": torch.full((nd,), float("nan"), dtype=torch.float32, device=dev),
        }

    # -- the four steps ------------------------------------------------------

    def row_stats(self, target, draft, tokens, cu, temperature, stream=None) -> torch.Tensor:
        sv.check(sv.spec_shard_row_stats(target, draft, tokens, cu, self.B, self.v_begin,
                                         self.v_end, self.max_target_rows, self.draft_stride,
                                         temperature, self.rows, self.workspace, stream),
                 "shard row stats")
        return self.rows

    def accept(self, rows_all, tokens, cu, temperature, u_accept, out, stream=None) -> None:
        sv.check(sv.spec_shard_accept(rows_all, self.n_shards, self.shard_begin, tokens, cu,
                                      self.B, self.max_target_rows, self.draft_stride,
                                      temperature, u_accept, out["tokens"], out["accept_len"],
                                      out.get("p"), out.get("q"), self.workspace, stream),
                 "shard accept")

    def final_mass(self, target, draft, stream=None) -> torch.Tensor:
        sv.check(sv.spec_shard_final_mass(target, draft, self.B, self.v_begin, self.v_end,
                                          self.max_target_rows, self.draft_stride, self.mass,
                                          self.workspace, stream), "shard final mass")
        return self.mass

    def final_draw(self, target, draft, mass_all, u_final, out_tokens, stream=None) -> None:
        sv.check(sv.spec_shard_final_draw(target, draft, mass_all, self.n_shards, self.shard,
                                          self.B, self.v_begin, self.v_end,
                                          self.max_target_rows, self.draft_stride, u_final,
                                          out_tokens, self.workspace, stream),
                 "shard final draw")


class DistExchange:
    """The three exchanges over a torch.distributed group (rank r = shard r)."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group

    def all_gather(self, t: torch.Tensor) -> torch.Tensor:
        n = self.dist.get_world_size(self.group)
        parts = [torch.empty_like(t) for _ in range(n)]
        self.dist.all_gather(parts, t.contiguous(), group=self.group)
        return torch.stack(parts)

    def max_(self, t: torch.Tensor) -> None:
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX, group=self.group)


def verify_sharded(shard, exchange, target, draft, tokens, cu, temperature, u_accept, u_final,
                   out: Optional[dict] = None) -> dict:
    """One rank's part of a sharded verification; every rank of the group
    calls it together with its own columns (target, draft) and the same
    tokens, offsets and uniforms.  Returns the whole verification's outputs
    (the same on every rank)."""
    out = out if out is not None else shard.outputs()
    rows_all = exchange.all_gather(shard.row_stats(target, draft, tokens, cu, temperature))
    shard.accept(rows_all, tokens, cu, temperature, u_accept, out)
    if temperature > 0:
        mass_all = exchange.all_gather(shard.final_mass(target, draft))
        shard.final_draw(target, draft, mass_all, u_final, out["tokens"])
        exchange.max_(out["tokens"])
    return out


def verify_sharded_local(shards: Sequence[Shard], targets, drafts, tokens, cu, temperature,
                         u_accept, u_final, outs: Optional[list] = None) -> list:
    """Several shards held on one device: the same steps in the same order,
    each exchange replaced by stacking (all-gather) or an element-wise max.
    Returns one output dict per shard; they are equal."""
    outs = outs if outs is not None else [s.outputs() for s in shards]
    # (each shard's records live in its own buffer; stacking copies them)
    rows_all = torch.stack([s.row_stats(t, d, tokens, cu, temperature)
                            for s, t, d in zip(shards, targets, drafts)])
    for s, o in zip(shards, outs):
        s.accept(rows_all, tokens, cu, temperature, u_accept, o)
    if temperature > 0:
        mass_all = torch.stack([s.final_mass(t, d) for s, t, d in zip(shards, targets, drafts)])
        for s, t, d, o in zip(shards, targets, drafts, outs):
            s.final_draw(t, d, mass_all, u_final, o["tokens"])
        top = torch.stack([o["tokens"] for o in outs]).amax(0)
        for o in outs:
            o["tokens"].copy_(top)
    return outs
