"""Convenience layer over the C-ABI binding: owns a workspace, allocates the
output tensors and turns status codes into exceptions.  Every call goes
through specverify (the C ABI); nothing here computes."""
from __future__ import annotations

from typing import Optional

import torch

from . import specverify as sv
from .workloads import VerifyBatch


class Verifier:
    """Workspace sized for up to B requests, max_target_rows rows and vocabulary V."""

    def __init__(self, B: int, max_target_rows: int, V: int, device="cuda"):
        self.B, self.max_target_rows, self.V = B, max_target_rows, V
        nbytes = sv.spec_workspace_size(B, max_target_rows, V)
        if nbytes == 0:
            raise ValueError("invalid workspace sizes")
        # torch.zeros already satisfies the zero-fill-before-first-use rule
        self.workspace = torch.zeros(nbytes, dtype=torch.uint8, device=device)
        self.device = torch.device(device)

    def outputs(self, batch: VerifyBatch, max_target_rows: Optional[int] = None) -> dict:
        rows = max_target_rows or batch.n_target_rows
        nd = batch.draft_tokens.numel()
        dev = self.device
        return {
            "tokens": torch.full((rows,), -7, dtype=torch.int32, device=dev),
            "accept_len": torch.full((batch.B,), -7, dtype=torch.int32, device=dev),
            "p": torch.full((max(nd, 1),), float("nan"), dtype=torch.float32, device=dev),
            "q": torch.full((max(nd, 1),), float("nan"), dtype=torch.float32, device=dev),
        }

    def verify(self, batch: VerifyBatch, max_target_rows: Optional[int] = None,
               out: Optional[dict] = None, stream=None, cu_draft: Optional[torch.Tensor] = None,
               check: bool = True) -> dict:
        """Run spec_verify_sample (T > 0) or spec_verify_greedy (T = 0) on a batch
        whose tensors live on this device.  cu_draft overrides batch.cu_draft
        (e.g. offsets produced on the device by dcut_allocate)."""
        rows = max_target_rows or batch.n_target_rows
        out = out if out is not None else self.outputs(batch, rows)
        cu = cu_draft if cu_draft is not None else batch.cu_draft
        if batch.temperature == 0:
            st = sv.spec_verify_greedy(batch.target_logits, batch.draft_tokens, cu, batch.B,
                                       batch.V, rows, batch.draft_stride, out["tokens"],
                                       out["accept_len"], self.workspace, stream)
        else:
            st = sv.spec_verify_sample(batch.target_logits, batch.draft_logits,
                                       batch.draft_tokens, cu, batch.B, batch.V, rows,
                                       batch.draft_stride, batch.temperature, batch.u_accept,
                                       batch.u_final, out["tokens"], out["accept_len"],
                                       out["p"], out["q"], self.workspace, stream)
        if check:
            sv.check(st, "verify")
        out["status"] = st
        return out

    def dcut(self, conf: torch.Tensor, kmax: torch.Tensor, budget: int, min_gain: float = 0.0,
             stream=None, check: bool = True) -> dict:
        B, Kmax = (conf.shape[0], conf.shape[1]) if conf.dim() == 2 else (kmax.numel(), 0)
        dev = self.device
        out = {"depth": torch.full((max(B, 1),), -7, dtype=torch.int32, device=dev),
               "cu": torch.full((B + 1,), -7, dtype=torch.int32, device=dev),
               "expected": torch.full((max(B, 1),), float("nan"), dtype=torch.float32,
                                      device=dev)}
        st = sv.dcut_allocate(conf, kmax, B, Kmax, budget, min_gain, out["depth"], out["cu"],
                              out["expected"], self.workspace, stream)
        if check:
            sv.check(st, "dcut_allocate")
        out["status"] = st
        return out

    def draft(self, draft_logits: torch.Tensor, kmax: torch.Tensor, Kmax: int,
              temperature: float, u_draft: Optional[torch.Tensor] = None, stream=None,
              check: bool = True) -> dict:
        """Drafted tokens and their q(x) from [B*Kmax][V] drafter logits (the
        workspace must hold B*(Kmax+1) target rows)."""
        B = kmax.numel()
        n = B * Kmax
        V = draft_logits.shape[-1]
        dev = self.device
        out = {"tokens": torch.full((max(n, 1),), -7, dtype=torch.int32, device=dev),
               "conf": torch.full((max(n, 1),), float("nan"), dtype=torch.float32, device=dev)}
        st = sv.spec_draft_sample(draft_logits, kmax, B, Kmax, V, temperature, u_draft,
                                  out["tokens"], out["conf"], self.workspace, stream)
        if check:
            sv.check(st, "draft_sample")
        out["status"] = st
        return out

    def acceptance_stats(self, accept_len: torch.Tensor, cu_draft: torch.Tensor, Kmax: int,
                         stream=None, check: bool = True) -> dict:
        """Per-position reached/accepted counts and the mean accepted length."""
        B = accept_len.numel()
        dev = self.device
        out = {"reached": torch.full((max(Kmax, 1),), -7, dtype=torch.int32, device=dev),
               "accepted": torch.full((max(Kmax, 1),), -7, dtype=torch.int32, device=dev),
               "mean": torch.full((1,), float("nan"), dtype=torch.float32, device=dev)}
        st = sv.spec_acceptance_stats(accept_len, cu_draft, B, Kmax, out["reached"],
                                      out["accepted"], out["mean"], self.workspace, stream)
        if check:
            sv.check(st, "acceptance_stats")
        out["status"] = st
        return out

    def device_status(self, stream=None) -> int:
        return sv.spec_get_device_status(self.workspace, stream)
