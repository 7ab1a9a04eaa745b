"""ctypes binding of libspecverify.so (include/specverify.h), same names.

Argument marshalling only: tensors become device pointers, the stream
defaults to torch's current stream, and buffer sizes and devices are checked
against what each call will touch, so that no host pointer and no undersized
buffer ever reaches a kernel.  Every step of the computation runs in the
library's CUDA kernels; there is no CPU fallback.  Importing this module
raises if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# SPECVERIFY_LIB selects another in-tree build of the same library (the
# tests use it for the bounds-checked build, libspecverify_debug.so)
LIB_PATH = os.path.join(_HERE, os.environ.get("SPECVERIFY_LIB", "libspecverify.so"))

SPEC_OK = 0
SPEC_ERR_INVALID_ARG = -1
SPEC_ERR_WORKSPACE = -2
SPEC_ERR_CUDA = -3
SPEC_ERR_NONFINITE = -4
SPEC_ERR_TIMEOUT = -5
SPEC_F32, SPEC_BF16 = 0, 1
SPEC_MAX_DRAFT = 32
SPEC_MAX_BATCH = 4096
SPEC_DCUT_MAX_CANDIDATES = 8192

EXPORTS = ("spec_workspace_size", "spec_workspace_init", "spec_verify_greedy",
           "spec_verify_sample", "dcut_allocate", "spec_get_device_status",
           "spec_status_string", "spec_set_trace", "spec_kernel_launch_count",
           "spec_verify_sample_static", "dcut_allocate_cost", "spec_draft_confidence",
           "spec_draft_sample", "spec_acceptance_stats", "spec_test_expire_wait",
           "spec_shard_workspace_size", "spec_shard_row_count", "spec_shard_row_stats",
           "spec_shard_accept", "spec_shard_final_mass", "spec_shard_final_draw")
SPEC_MAX_SHARDS = 32
SHARD_RECORD_FLOATS = 4  # spec_shard_row and spec_shard_mass: 16 bytes each
SPEC_STATIC_SCRATCH_BYTES = 1 << 20


class SpecError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__(f"{where}: {spec_status_string(status)} (status {status})")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing; build it with `python -m draft_verification_02_b300.build`."
            " The verification path runs only in its CUDA kernels and has no fallback.")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, F32, SZ = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                            ctypes.c_size_t)
    INT = ctypes.c_int
    lib.spec_workspace_size.argtypes = [I32, I64, I32]
    lib.spec_workspace_size.restype = SZ
    lib.spec_workspace_init.argtypes = [P, SZ, P]
    lib.spec_workspace_init.restype = INT
    lib.spec_verify_greedy.argtypes = [P, INT, P, P, I32, I32, I64, I32, P, P, P, SZ, P]
    lib.spec_verify_greedy.restype = INT
    lib.spec_verify_sample.argtypes = [P, P, INT, P, P, I32, I32, I64, I32, F32, P, P, P, P,
                                       P, P, P, SZ, P]
    lib.spec_verify_sample.restype = INT
    lib.spec_verify_sample_static.argtypes = [P, P, INT, P, P, I32, I32, I64, I32, F32, P, P,
                                              P, P, P, P, P]
    lib.spec_verify_sample_static.restype = INT
    lib.dcut_allocate.argtypes = [P, P, I32, I32, I32, F32, P, P, P, P, SZ, P]
    lib.dcut_allocate_cost.argtypes = [P, P, I32, I32, ctypes.c_double, P, P, P, P, SZ, P]
    lib.dcut_allocate_cost.restype = INT
    lib.spec_draft_confidence.argtypes = [P, INT, P, P, I32, I32, I32, F32, P, P, SZ, P]
    lib.spec_draft_confidence.restype = INT
    lib.spec_draft_sample.argtypes = [P, INT, P, I32, I32, I32, F32, P, P, P, P, SZ, P]
    lib.spec_draft_sample.restype = INT
    lib.spec_acceptance_stats.argtypes = [P, P, I32, I32, P, P, P, P, SZ, P]
    lib.spec_acceptance_stats.restype = INT
    lib.dcut_allocate.restype = INT
    lib.spec_get_device_status.argtypes = [P, P]
    lib.spec_get_device_status.restype = INT
    lib.spec_status_string.argtypes = [INT]
    lib.spec_status_string.restype = ctypes.c_char_p
    lib.spec_set_trace.argtypes = [ctypes.POINTER(ctypes.c_void_p), INT]
    lib.spec_set_trace.restype = INT
    lib.spec_kernel_launch_count.argtypes = []
    lib.spec_kernel_launch_count.restype = I64
    lib.spec_test_expire_wait.argtypes = [I64]
    lib.spec_test_expire_wait.restype = INT
    lib.spec_shard_workspace_size.argtypes = [I32, I64, I32]
    lib.spec_shard_workspace_size.restype = SZ
    lib.spec_shard_row_count.argtypes = [I32, I64, I32]
    lib.spec_shard_row_count.restype = I64
    lib.spec_shard_row_stats.argtypes = [P, P, INT, P, P, I32, I32, I32, I64, I32, F32, P, P, SZ,
                                         P]
    lib.spec_shard_row_stats.restype = INT
    lib.spec_shard_accept.argtypes = [P, I32, ctypes.POINTER(I32), P, P, I32, I64, I32, F32, P,
                                      P, P, P, P, P, SZ, P]
    lib.spec_shard_accept.restype = INT
    lib.spec_shard_final_mass.argtypes = [P, P, INT, I32, I32, I32, I64, I32, P, P, SZ, P]
    lib.spec_shard_final_mass.restype = INT
    lib.spec_shard_final_draw.argtypes = [P, P, INT, P, I32, I32, I32, I32, I32, I64, I32, P, P,
                                          P, SZ, P]
    lib.spec_shard_final_draw.restype = INT
    return lib


LIB = _load()

# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------


def _dev(t, name, dtype=None, min_numel=0, allow_none=False):
    """Device pointer of a contiguous CUDA tensor with at least min_numel elements."""
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (device memory)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.numel() < min_numel:
        raise ValueError(f"{name} holds {t.numel()} elements, needs at least {min_numel}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SPEC_F32
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _draft_extent(B, max_target_rows, draft_stride):
    return B * draft_stride if draft_stride > 0 else max_target_rows - B


# ---------------------------------------------------------------------------
# the C ABI, one function per entry point
# ---------------------------------------------------------------------------


def spec_workspace_size(B: int, max_target_rows: int, V: int) -> int:
    return int(LIB.spec_workspace_size(B, max_target_rows, V))


def spec_workspace_init(workspace: torch.Tensor, stream=None) -> int:
    ptr = _dev(workspace, "workspace")
    return LIB.spec_workspace_init(ptr, workspace.numel() * workspace.element_size(),
                                   _stream(stream))


def spec_verify_greedy(target_logits, draft_tokens, cu_draft, B: int, V: int,
                       max_target_rows: int, draft_stride: int, out_tokens, out_accept_len,
                       workspace, stream=None) -> int:
    if B == 0:
        return SPEC_OK
    nd = _draft_extent(B, max_target_rows, draft_stride)
    return LIB.spec_verify_greedy(
        _dev(target_logits, "target_logits", min_numel=max_target_rows * V),
        dtype_code(target_logits),
        _dev(draft_tokens, "draft_tokens", torch.int32, nd, allow_none=nd == 0),
        _dev(cu_draft, "cu_draft", torch.int32, B + 1), B, V, max_target_rows, draft_stride,
        _dev(out_tokens, "out_tokens", torch.int32, max_target_rows),
        _dev(out_accept_len, "out_accept_len", torch.int32, B),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream))


def spec_verify_sample(target_logits, draft_logits, draft_tokens, cu_draft, B: int, V: int,
                       max_target_rows: int, draft_stride: int, temperature: float, u_accept,
                       u_final, out_tokens, out_accept_len, out_p, out_q, workspace,
                       stream=None) -> int:
    if B == 0:
        return SPEC_OK
    nd = _draft_extent(B, max_target_rows, draft_stride)
    code = dtype_code(target_logits)
    greedy = temperature == 0
    if not greedy and draft_logits is not None and draft_logits.dtype != target_logits.dtype:
        raise TypeError("target and draft logits must share a dtype")
    need_draft = (not greedy) and nd > 0
    return LIB.spec_verify_sample(
        _dev(target_logits, "target_logits", min_numel=max_target_rows * V),
        _dev(draft_logits, "draft_logits", min_numel=nd * V, allow_none=not need_draft),
        code,
        _dev(draft_tokens, "draft_tokens", torch.int32, nd, allow_none=nd == 0),
        _dev(cu_draft, "cu_draft", torch.int32, B + 1), B, V, max_target_rows, draft_stride,
        float(temperature),
        _dev(u_accept, "u_accept", torch.float32, nd, allow_none=not need_draft),
        _dev(u_final, "u_final", torch.float32, B, allow_none=greedy),
        _dev(out_tokens, "out_tokens", torch.int32, max_target_rows),
        _dev(out_accept_len, "out_accept_len", torch.int32, B),
        _dev(out_p, "out_p", torch.float32, nd, allow_none=True),
        _dev(out_q, "out_q", torch.float32, nd, allow_none=True),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream))


def spec_verify_sample_static(target_logits, draft_logits, draft_tokens, cu_draft, B: int,
                              V: int, max_target_rows: int, draft_stride: int,
                              temperature: float, u_accept, u_final, out_tokens,
                              out_accept_len, out_p, out_q, stream=None) -> int:
    """spec_verify_sample with the library's fixed scratch array instead of a
    workspace: for callers that cannot allocate device memory."""
    if B == 0:
        return SPEC_OK
    nd = _draft_extent(B, max_target_rows, draft_stride)
    code = dtype_code(target_logits)
    greedy = temperature == 0
    if not greedy and draft_logits is not None and draft_logits.dtype != target_logits.dtype:
        raise TypeError("target and draft logits must share a dtype")
    need_draft = (not greedy) and nd > 0
    return LIB.spec_verify_sample_static(
        _dev(target_logits, "target_logits", min_numel=max_target_rows * V),
        _dev(draft_logits, "draft_logits", min_numel=nd * V, allow_none=not need_draft),
        code,
        _dev(draft_tokens, "draft_tokens", torch.int32, nd, allow_none=nd == 0),
        _dev(cu_draft, "cu_draft", torch.int32, B + 1), B, V, max_target_rows, draft_stride,
        float(temperature),
        _dev(u_accept, "u_accept", torch.float32, nd, allow_none=not need_draft),
        _dev(u_final, "u_final", torch.float32, B, allow_none=greedy),
        _dev(out_tokens, "out_tokens", torch.int32, max_target_rows),
        _dev(out_accept_len, "out_accept_len", torch.int32, B),
        _dev(out_p, "out_p", torch.float32, nd, allow_none=True),
        _dev(out_q, "out_q", torch.float32, nd, allow_none=True),
        _stream(stream))


def dcut_allocate(conf, kmax, B: int, Kmax: int, budget: int, min_gain: float, out_depth,
                  out_cu, out_expected_len, workspace, stream=None) -> int:
    return LIB.dcut_allocate(
        _dev(conf, "conf", torch.float32, B * Kmax, allow_none=B * Kmax == 0),
        _dev(kmax, "kmax", torch.int32, B, allow_none=B == 0), B, Kmax, budget,
        float(min_gain),
        _dev(out_depth, "out_depth", torch.int32, B, allow_none=B == 0),
        _dev(out_cu, "out_cu", torch.int32, B + 1),
        _dev(out_expected_len, "out_expected_len", torch.float32, B, allow_none=True),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream))


def dcut_allocate_cost(conf, kmax, B: int, Kmax: int, max_cost: float, out_depth, out_cu,
                       out_benefit, workspace, stream=None) -> int:
    return LIB.dcut_allocate_cost(
        _dev(conf, "conf", torch.float32, B * Kmax, allow_none=B * Kmax == 0),
        _dev(kmax, "kmax", torch.int32, B, allow_none=B == 0), B, Kmax, float(max_cost),
        _dev(out_depth, "out_depth", torch.int32, B, allow_none=B == 0),
        _dev(out_cu, "out_cu", torch.int32, B + 1),
        _dev(out_benefit, "out_benefit", torch.float64, B, allow_none=True),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream))


def spec_draft_confidence(draft_logits, draft_tokens, kmax, B: int, Kmax: int, V: int,
                          temperature: float, out_conf, workspace, stream=None) -> int:
    n = B * Kmax
    if n == 0:
        return SPEC_OK
    return LIB.spec_draft_confidence(
        _dev(draft_logits, "draft_logits", min_numel=n * V), dtype_code(draft_logits),
        _dev(draft_tokens, "draft_tokens", torch.int32, n),
        _dev(kmax, "kmax", torch.int32, B), B, Kmax, V, float(temperature),
        _dev(out_conf, "out_conf", torch.float32, n),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream))


def spec_draft_sample(draft_logits, kmax, B: int, Kmax: int, V: int, temperature: float, u_draft,
                      out_tokens, out_conf, workspace, stream=None) -> int:
    n = B * Kmax
    if n == 0:
        return SPEC_OK
    return LIB.spec_draft_sample(
        _dev(draft_logits, "draft_logits", min_numel=n * V), dtype_code(draft_logits),
        _dev(kmax, "kmax", torch.int32, B), B, Kmax, V, float(temperature),
        _dev(u_draft, "u_draft", torch.float32, n, allow_none=temperature == 0),
        _dev(out_tokens, "out_tokens", torch.int32, n),
        _dev(out_conf, "out_conf", torch.float32, n),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream))


def spec_acceptance_stats(accept_len, cu_draft, B: int, Kmax: int, out_reached, out_accepted,
                          out_mean, workspace, stream=None) -> int:
    return LIB.spec_acceptance_stats(
        _dev(accept_len, "accept_len", torch.int32, B, allow_none=B == 0),
        _dev(cu_draft, "cu_draft", torch.int32, B + 1, allow_none=B == 0), B, Kmax,
        _dev(out_reached, "out_reached", torch.int32, Kmax, allow_none=Kmax == 0),
        _dev(out_accepted, "out_accepted", torch.int32, Kmax, allow_none=Kmax == 0),
        _dev(out_mean, "out_mean", torch.float32, 1),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream))


# ---- vocabulary-sharded verification (records: float32 tensors of 4 per row / request)


def spec_shard_workspace_size(B: int, max_target_rows: int, V_shard: int) -> int:
    return int(LIB.spec_shard_workspace_size(B, max_target_rows, V_shard))


def spec_shard_row_count(B: int, max_target_rows: int, draft_stride: int) -> int:
    return int(LIB.spec_shard_row_count(B, max_target_rows, draft_stride))


def _records(t, name, n):
    return _dev(t, name, torch.float32, n * SHARD_RECORD_FLOATS)


def spec_shard_row_stats(target_shard, draft_shard, draft_tokens, cu_draft, B: int, v_begin: int,
                         v_end: int, max_target_rows: int, draft_stride: int, temperature: float,
                         out_rows, workspace, stream=None) -> int:
    if B == 0:
        return SPEC_OK
    Vs = v_end - v_begin
    nd = _draft_extent(B, max_target_rows, draft_stride)
    greedy = temperature == 0
    need_draft = (not greedy) and nd > 0
    if need_draft and draft_shard is not None and draft_shard.dtype != target_shard.dtype:
        raise TypeError("target and draft logits must share a dtype")
    return LIB.spec_shard_row_stats(
        _dev(target_shard, "target_shard", min_numel=max_target_rows * Vs),
        _dev(draft_shard, "draft_shard", min_numel=nd * Vs, allow_none=not need_draft),
        dtype_code(target_shard),
        _dev(draft_tokens, "draft_tokens", torch.int32, nd, allow_none=nd == 0),
        _dev(cu_draft, "cu_draft", torch.int32, B + 1), B, v_begin, v_end, max_target_rows,
        draft_stride, float(temperature),
        _records(out_rows, "out_rows", spec_shard_row_count(B, max_target_rows, draft_stride)),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream))


def spec_shard_accept(rows_all, n_shards: int, shard_begin, draft_tokens, cu_draft, B: int,
                      max_target_rows: int, draft_stride: int, temperature: float, u_accept,
                      out_tokens, out_accept_len, out_p, out_q, workspace, stream=None) -> int:
    """shard_begin: a host sequence of n_shards + 1 ints."""
    if B == 0:
        return SPEC_OK
    begin = [int(v) for v in shard_begin]
    if len(begin) != n_shards + 1:
        raise ValueError("shard_begin must hold n_shards + 1 entries")
    nd = _draft_extent(B, max_target_rows, draft_stride)
    greedy = temperature == 0
    n_rec = spec_shard_row_count(B, max_target_rows, draft_stride)
    return LIB.spec_shard_accept(
        _records(rows_all, "rows_all", n_shards * n_rec), n_shards,
        (ctypes.c_int32 * len(begin))(*begin),
        _dev(draft_tokens, "draft_tokens", torch.int32, nd, allow_none=nd == 0),
        _dev(cu_draft, "cu_draft", torch.int32, B + 1), B, max_target_rows, draft_stride,
        float(temperature),
        _dev(u_accept, "u_accept", torch.float32, nd, allow_none=greedy or nd == 0),
        _dev(out_tokens, "out_tokens", torch.int32, max_target_rows),
        _dev(out_accept_len, "out_accept_len", torch.int32, B),
        _dev(out_p, "out_p", torch.float32, nd, allow_none=True),
        _dev(out_q, "out_q", torch.float32, nd, allow_none=True),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream))


def spec_shard_final_mass(target_shard, draft_shard, B: int, v_begin: int, v_end: int,
                          max_target_rows: int, draft_stride: int, out_mass, workspace,
                          stream=None) -> int:
    if B == 0:
        return SPEC_OK
    Vs = v_end - v_begin
    nd = _draft_extent(B, max_target_rows, draft_stride)
    return LIB.spec_shard_final_mass(
        _dev(target_shard, "target_shard", min_numel=max_target_rows * Vs),
        _dev(draft_shard, "draft_shard", min_numel=nd * Vs, allow_none=nd == 0),
        dtype_code(target_shard), B, v_begin, v_end, max_target_rows, draft_stride,
        _records(out_mass, "out_mass", B),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream))


def spec_shard_final_draw(target_shard, draft_shard, mass_all, n_shards: int, shard: int, B: int,
                          v_begin: int, v_end: int, max_target_rows: int, draft_stride: int,
                          u_final, out_tokens, workspace, stream=None) -> int:
    if B == 0:
        return SPEC_OK
    Vs = v_end - v_begin
    nd = _draft_extent(B, max_target_rows, draft_stride)
    return LIB.spec_shard_final_draw(
        _dev(target_shard, "target_shard", min_numel=max_target_rows * Vs),
        _dev(draft_shard, "draft_shard", min_numel=nd * Vs, allow_none=nd == 0),
        dtype_code(target_shard), _records(mass_all, "mass_all", n_shards * B), n_shards, shard,
        B, v_begin, v_end, max_target_rows, draft_stride,
        _dev(u_final, "u_final", torch.float32, B),
        _dev(out_tokens, "out_tokens", torch.int32, max_target_rows),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream))


def spec_get_device_status(workspace, stream=None) -> int:
    return LIB.spec_get_device_status(_dev(workspace, "workspace"), _stream(stream))


def spec_status_string(status: int) -> str:
    return LIB.spec_status_string(int(status)).decode()


def spec_set_trace(events) -> int:
    """events: list of torch.cuda.Event (recorded by the next calls), or None."""
    if not events:
        return LIB.spec_set_trace(None, 0)
    handles = []
    for e in events:
        if e.cuda_event == 0:  # torch creates the event lazily
            e.record()
        handles.append(e.cuda_event)
    arr = (ctypes.c_void_p * len(handles))(*handles)
    return LIB.spec_set_trace(arr, len(handles))


def spec_kernel_launch_count() -> int:
    return int(LIB.spec_kernel_launch_count())


def spec_test_expire_wait(item: int) -> int:
    """Test hook (see the header): -1 turns it off."""
    return int(LIB.spec_test_expire_wait(int(item)))


def check(status: int, where: str = "") -> None:
    if status != SPEC_OK:
        raise SpecError(status, where)


__all__ = list(EXPORTS) + ["SpecError", "check", "dtype_code", "LIB", "LIB_PATH"]
