"""Seeded synthetic inputs for batched draft verification and D-cut.

This module only draws random inputs: logits, drafted tokens, uniforms and
per-position draft confidences.  It holds none of the verification arithmetic
(no softmax statistics, no accept test, no residual, no ranking), so both the
CUDA path and the CPU oracle may consume what it produces.

The shapes and distributions stand in for the workloads the AngelSpec pages
describe (MTP drafts of depth 3, block-diffusion blocks, concurrency 4-64,
vocabularies of 32k-152k; "Tencent Hunyuan Turns Speculative Decoding Into a
Full Open-Source Stack", "Key numbers"); the logits there come from trained
Hy3 / Qwen3 models, which are not available, so every value here is synthetic.

Layout (shared with the C-ABI): request i verifies k[i] drafted tokens.
``cu_draft[i]`` is the exclusive prefix sum of k.  Target row j of request i
is row ``cu_draft[i] + i + j`` of ``target_logits`` (j = k[i] is the bonus
row).  Draft-side arrays (draft rows, drafted tokens, accept uniforms) use the
draft index ``cu_draft[i] + j`` (packed, ``draft_stride == 0``) or
``i * draft_stride + j`` (padded, ``draft_stride > 0``).

Drafted tokens are drawn from the drafter's law q = softmax(d / T) by the
Gumbel-max construction (argmax of d/T plus Gumbel noise), which samples that
law exactly without forming it; at T = 0 the drafter is greedy (argmax of d).
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import torch

# ---------------------------------------------------------------------------
# workload specifications
# ---------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, value recipe and seed."""

    name: str
    B: int
    V: int
    dtype: str                 # "f32" or "bf16"
    seed: int
    k: Optional[int] = None    # fixed verified depth per request, or None
    k_range: Optional[tuple] = None  # (lo, hi) inclusive uniform depth per request
    kmax: int = 0              # drafted tokens per request (D-cut workloads)
    budget: int = 0            # D-cut verify-token budget
    target_sigma: float = 2.0
    peak: float = 0.0          # planted +peak at one uniformly drawn index per target row
    draft_sigma: tuple = (1.0,)  # per-position draft noise sigma (last value repeats)
    temperatures: tuple = (1.0,)


def _linear_sigmas(lo: float, hi: float, n: int) -> tuple:
    return tuple(lo + (hi - lo) * j / (n - 1) for j in range(n))


TINY = Workload("tiny", B=4, V=1024, dtype="f32", seed=0, k=4, target_sigma=2.0,
                draft_sigma=(1.0,), temperatures=(0.0, 1.0))
MTP = Workload("mtp", B=16, V=128000, dtype="bf16", seed=1, k=3, target_sigma=3.0,
               peak=8.0, draft_sigma=(1.5,), temperatures=(1.0,))
BLOCK = Workload("block", B=32, V=151936, dtype="bf16", seed=2, k=16, target_sigma=3.0,
                 draft_sigma=_linear_sigmas(0.5, 3.0, 16), temperatures=(0.0, 0.7))
DCUT = Workload("dcut", B=64, V=128000, dtype="bf16", seed=3, kmax=16, budget=256,
                target_sigma=2.0, draft_sigma=(1.0,), temperatures=(1.0,))

RAGGED_B = (4, 8, 16, 32, 64, 128)
RAGGED_V = (32000, 128000, 151936)
RAGGED_T = (0.0, 0.7, 1.0)


def ragged(pair_index: int) -> Workload:
    """The ragged sweep: 18 (B, V) pairs in B-major order, seeds 10..27."""
    if not 0 <= pair_index < len(RAGGED_B) * len(RAGGED_V):
        raise ValueError(f"ragged pair index {pair_index} out of range")
    B = RAGGED_B[pair_index // len(RAGGED_V)]
    V = RAGGED_V[pair_index % len(RAGGED_V)]
    return Workload(f"ragged_B{B}_V{V}", B=B, V=V, dtype="bf16", seed=10 + pair_index,
                    k_range=(1, 16), target_sigma=2.0, draft_sigma=(1.0,),
                    temperatures=RAGGED_T)


WORKLOADS = {w.name: w for w in (TINY, MTP, BLOCK, DCUT)}


def get(name: str) -> Workload:
    if name in WORKLOADS:
        return WORKLOADS[name]
    if name.startswith("ragged"):
        # accept "ragged<k>" or "ragged_B<B>_V<V>"
        rest = name[len("ragged"):]
        if rest.isdigit():
            return ragged(int(rest))
        for k in range(len(RAGGED_B) * len(RAGGED_V)):
            if ragged(k).name == name:
                return ragged(k)
    raise KeyError(name)


# ---------------------------------------------------------------------------
# containers
# ---------------------------------------------------------------------------


@dataclasses.dataclass
class VerifyBatch:
    """Inputs of one verification call (all tensors on one device)."""

    B: int
    V: int
    dtype: str
    temperature: float
    k: torch.Tensor              # int32 [B]
    cu_draft: torch.Tensor       # int32 [B+1]
    target_logits: torch.Tensor  # [sum(k)+B, V] float32 or bfloat16
    draft_logits: torch.Tensor   # [rows, V] (packed sum(k) or padded B*draft_stride)
    draft_tokens: torch.Tensor   # int32, draft index
    u_accept: torch.Tensor       # float32 in [0,1), draft index
    u_final: torch.Tensor        # float32 in [0,1), [B]
    draft_stride: int = 0

    @property
    def n_draft(self) -> int:
        return int(self.k.sum().item())

    @property
    def n_target_rows(self) -> int:
        return self.n_draft + self.B

    def to(self, device) -> "VerifyBatch":
        fields = {}
        for f in dataclasses.fields(self):
            v = getattr(self, f.name)
            fields[f.name] = v.to(device) if isinstance(v, torch.Tensor) else v
        return VerifyBatch(**fields)

    def algorithmic_bytes(self) -> int:
        """Logit bytes the method must read once: target rows, plus draft rows at T > 0."""
        e = 4 if self.dtype == "f32" else 2
        rows = self.n_target_rows + (self.n_draft if self.temperature > 0 else 0)
        return rows * self.V * e


@dataclasses.dataclass
class DcutProblem:
    conf: torch.Tensor   # float32 [B, Kmax], c in [0,1]
    kmax: torch.Tensor   # int32 [B]
    budget: int


# ---------------------------------------------------------------------------
# generators
# ---------------------------------------------------------------------------

_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _rep_seed(seed: int, rep: int) -> int:
    return seed + 1_000_003 * rep


def _uniform(g, n, device) -> torch.Tensor:
    return torch.rand(n, generator=g, device=device, dtype=torch.float32)


def _gumbel_argmax(rows_f32: torch.Tensor, temperature: float, g, device,
                   chunk_rows: int = 64) -> torch.Tensor:
    """Draft token per row: argmax(d/T + Gumbel) (exact draw from softmax(d/T))."""
    out = torch.empty(rows_f32.shape[0], dtype=torch.int64, device=device)
    for r0 in range(0, rows_f32.shape[0], chunk_rows):
        r1 = min(rows_f32.shape[0], r0 + chunk_rows)
        u = torch.rand((r1 - r0, rows_f32.shape[1]), generator=g, device=device,
                       dtype=torch.float64)
        gumbel = -torch.log(-torch.log1p(-u))  # u in [0,1) -> 1-u in (0,1]
        score = rows_f32[r0:r1].double() / temperature + gumbel
        out[r0:r1] = torch.argmax(score, dim=1)
    return out


def make_depths(w: Workload, device="cpu", rep: int = 0) -> torch.Tensor:
    """Verified depth per request for fixed-depth and ragged workloads."""
    if w.k is not None:
        return torch.full((w.B,), w.k, dtype=torch.int32, device=device)
    if w.k_range is not None:
        g = _gen(device, _rep_seed(w.seed, rep) ^ 0x5EED)
        lo, hi = w.k_range
        return torch.randint(lo, hi + 1, (w.B,), generator=g, device=device,
                             dtype=torch.int32)
    raise ValueError(f"workload {w.name} has no fixed depths (D-cut decides them)")


def make_dcut_problem(w: Workload, device="cpu", rep: int = 0) -> DcutProblem:
    """Per-position draft confidence c[i,j] = b[i,j] * 0.95**j with b ~ Beta(8,2).

    Beta(8,2) is drawn as X/(X+Y) with X ~ Gamma(8), Y ~ Gamma(2), each Gamma
    of integer shape a sum of unit exponentials (-log of a uniform).
    """
    if w.kmax <= 0:
        raise ValueError(f"workload {w.name} is not a D-cut workload")
    g = _gen(device, _rep_seed(w.seed, rep) ^ 0xDC)
    u = torch.rand((w.B, w.kmax, 10), generator=g, device=device, dtype=torch.float64)
    e = -torch.log1p(-u)                      # unit exponentials
    x = e[..., :8].sum(-1)
    y = e[..., 8:].sum(-1)
    b = x / (x + y)
    decay = 0.95 ** torch.arange(w.kmax, device=device, dtype=torch.float64)
    conf = (b * decay).to(torch.float32).clamp_(0.0, 1.0)
    kmax = torch.full((w.B,), w.kmax, dtype=torch.int32, device=device)
    return DcutProblem(conf=conf.contiguous(), kmax=kmax, budget=w.budget)


def make_verify_batch(w: Workload, temperature: float, device="cpu", rep: int = 0,
                      depths: Optional[torch.Tensor] = None,
                      draft_stride: int = 0) -> VerifyBatch:
    """Draw one verification batch.

    Draw order from one generator seeded with the workload seed (``rep`` > 0
    gives independent copies used to rotate inputs past the L2 cache):
    target logits N(0, target_sigma^2) -> planted peaks -> draft noise ->
    drafted tokens (Gumbel noise, or argmax at T = 0) -> u_accept -> u_final.
    ``depths`` overrides the workload's verified depth per request (D-cut).
    With ``draft_stride`` > 0 the draft side is padded to draft_stride rows
    per request; rows at j >= depth are drawn too (a drafter produces them)
    but are never verified.
    """
    device = torch.device(device)
    k = (depths.to(device=device, dtype=torch.int32) if depths is not None
         else make_depths(w, device, rep))
    B, V = w.B, w.V
    if k.numel() != B:
        raise ValueError("depths must have one entry per request")
    if draft_stride and int(k.max().item() if B else 0) > draft_stride:
        raise ValueError("draft_stride smaller than a depth")
    g = _gen(device, _rep_seed(w.seed, rep))
    cu = torch.zeros(B + 1, dtype=torch.int32, device=device)
    cu[1:] = torch.cumsum(k, 0)
    n_draft = int(cu[-1].item())

    # one logical target row per (request, position 0..depth); padded drafts
    # also need logical rows up to draft_stride for the unverified positions
    depth_rows = (k + 1) if not draft_stride else torch.full_like(k, draft_stride + 1)
    n_logical = int(depth_rows.sum().item())
    tgt = torch.randn((n_logical, V), generator=g, device=device,
                      dtype=torch.float32) * w.target_sigma
    if w.peak:
        idx = torch.randint(0, V, (n_logical,), generator=g, device=device)
        tgt[torch.arange(n_logical, device=device), idx] += w.peak
    # position of every logical row inside its request
    starts = torch.zeros(B + 1, dtype=torch.int64, device=device)
    starts[1:] = torch.cumsum(depth_rows.long(), 0)
    pos = (torch.arange(n_logical, device=device)
           - torch.repeat_interleave(starts[:-1], depth_rows.long()))
    sig = torch.tensor(w.draft_sigma, dtype=torch.float32, device=device)
    sig_row = sig[pos.clamp(max=len(w.draft_sigma) - 1)]
    noise = torch.randn((n_logical, V), generator=g, device=device, dtype=torch.float32)
    drf = tgt + noise * sig_row[:, None]

    tdt = _TORCH_DTYPE[w.dtype]
    req_of_row = torch.repeat_interleave(torch.arange(B, device=device), depth_rows.long())
    # target rows actually verified: j <= k[i]
    keep_t = pos <= k.long()[req_of_row]
    target_logits = tgt[keep_t].to(tdt).contiguous()
    # draft rows: j < k[i] (packed) or j < draft_stride (padded)
    if draft_stride:
        keep_d = pos < draft_stride
    else:
        keep_d = pos < k.long()[req_of_row]
    draft_logits = drf[keep_d].to(tdt).contiguous()
    del tgt, drf, noise

    # drafted tokens come from the (rounded) draft logits
    d_exact = draft_logits.float()
    if temperature > 0:
        tokens = _gumbel_argmax(d_exact, temperature, g, device)
    else:
        tokens = torch.argmax(d_exact, dim=1)
    del d_exact
    n_drows = draft_logits.shape[0]
    u_accept = _uniform(g, n_drows, device)
    u_final = _uniform(g, B, device)
    return VerifyBatch(B=B, V=V, dtype=w.dtype, temperature=float(temperature), k=k,
                       cu_draft=cu, target_logits=target_logits,
                       draft_logits=draft_logits,
                       draft_tokens=tokens.to(torch.int32).contiguous(),
                       u_accept=u_accept, u_final=u_final,
                       draft_stride=int(draft_stride))


def batch_from_rows(target_rows: Sequence, draft_rows: Sequence, tokens: Sequence,
                    k: Sequence[int], u_accept: Sequence[float], u_final: Sequence[float],
                    temperature: float, dtype: str = "f32") -> VerifyBatch:
    """Assemble a packed batch from explicit rows (hand-built cases and fixtures)."""
    tdt = _TORCH_DTYPE[dtype]
    k_t = torch.tensor(list(k), dtype=torch.int32)
    B = k_t.numel()
    cu = torch.zeros(B + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(k_t, 0)
    t = torch.tensor(target_rows, dtype=torch.float32).to(tdt)
    V = t.shape[1]
    d = (torch.tensor(draft_rows, dtype=torch.float32).to(tdt) if len(draft_rows)
         else torch.zeros((0, V), dtype=tdt))
    return VerifyBatch(B=B, V=V, dtype=dtype, temperature=float(temperature), k=k_t,
                       cu_draft=cu, target_logits=t.contiguous(),
                       draft_logits=d.contiguous(),
                       draft_tokens=torch.tensor(list(tokens), dtype=torch.int32),
                       u_accept=torch.tensor(list(u_accept), dtype=torch.float32),
                       u_final=torch.tensor(list(u_final), dtype=torch.float32))


def max_target_rows(w: Workload) -> int:
    """Host-known upper bound on target rows for a workload (grid sizing)."""
    if w.kmax:
        return w.budget + w.B
    if w.k is not None:
        return w.B * (w.k + 1)
    return w.B * (w.k_range[1] + 1)


def describe(w: Workload) -> str:
    parts = [f"B={w.B}", f"V={w.V}", w.dtype]
    if w.k is not None:
        parts.append(f"K={w.k}")
    if w.k_range is not None:
        parts.append(f"K~U{{{w.k_range[0]}..{w.k_range[1]}}}")
    if w.kmax:
        parts.append(f"Kmax={w.kmax} budget={w.budget}")
    return f"{w.name}: " + ", ".join(parts)


__all__ = [
    "Workload", "VerifyBatch", "DcutProblem", "TINY", "MTP", "BLOCK", "DCUT",
    "RAGGED_B", "RAGGED_V", "RAGGED_T", "ragged", "get", "make_depths",
    "make_dcut_problem", "make_verify_batch", "batch_from_rows", "max_target_rows",
    "describe",
]
