"""The C-ABI library on the CPU: it loads, exports every symbol the header
declares, and its host-side checks reject bad arguments before touching a
GPU.  No compute call is made here."""
import ctypes
import os
import re

import pytest
import torch

from draft_verification_02_b300 import specverify as sv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specverify.h")
FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: every call below fails its checks first


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(
        r"^(?:size_t|int|int64_t|const char \*)\s*\**\s*(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_api():
    names = declared_functions()
    for n in ("spec_verify_greedy", "spec_verify_sample", "dcut_allocate",
              "spec_workspace_size", "spec_get_device_status", "spec_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(sv.LIB_PATH)
    for n in declared_functions():
        assert hasattr(lib, n), n
        assert n in sv.EXPORTS, n
        assert callable(getattr(sv, n)), n


def test_workspace_size():
    assert sv.spec_workspace_size(-1, 10, 10) == 0
    assert sv.spec_workspace_size(0, 0, 0) > 0  # status word only
    a = sv.spec_workspace_size(16, 64, 128000)
    b = sv.spec_workspace_size(32, 544, 151936)
    assert 0 < a < b
    assert sv.spec_workspace_size(4, 20, 1 << 30) == 0  # vocabulary beyond the chunk limit


def test_status_strings():
    for code in (0, -1, -2, -3, -4, -5):
        assert sv.spec_status_string(code) and sv.spec_status_string(code) != "unknown status"
    assert sv.spec_status_string(42) == "unknown status"


def test_host_checks_reject_before_any_launch():
    L = sv.LIB
    null = None
    # greedy: negative batch, bad dtype, max rows below B, stride negative
    assert L.spec_verify_greedy(FAKE, 0, FAKE, FAKE, -1, 10, 10, 0, FAKE, FAKE, FAKE, 1 << 20,
                                null) == sv.SPEC_ERR_INVALID_ARG
    assert L.spec_verify_greedy(FAKE, 7, FAKE, FAKE, 2, 10, 4, 0, FAKE, FAKE, FAKE, 1 << 20,
                                null) == sv.SPEC_ERR_INVALID_ARG
    assert L.spec_verify_greedy(FAKE, 0, FAKE, FAKE, 4, 10, 3, 0, FAKE, FAKE, FAKE, 1 << 20,
                                null) == sv.SPEC_ERR_INVALID_ARG
    assert L.spec_verify_greedy(FAKE, 0, FAKE, FAKE, 4, 10, 8, -1, FAKE, FAKE, FAKE, 1 << 20,
                                null) == sv.SPEC_ERR_INVALID_ARG
    assert L.spec_verify_greedy(FAKE, 0, FAKE, FAKE, 4, 10, 8, 0, FAKE, FAKE, null, 0,
                                null) == sv.SPEC_ERR_WORKSPACE
    assert L.spec_verify_greedy(FAKE, 0, FAKE, FAKE, 4, 10, 8, 0, FAKE, FAKE, FAKE, 16,
                                null) == sv.SPEC_ERR_WORKSPACE
    assert L.spec_verify_greedy(null, 0, FAKE, FAKE, 4, 10, 8, 0, FAKE, FAKE, FAKE, 1 << 20,
                                null) == sv.SPEC_ERR_INVALID_ARG
    # B = 0 is a no-op
    assert L.spec_verify_greedy(null, 0, null, null, 0, 10, 0, 0, null, null, null, 0,
                                null) == sv.SPEC_OK
    # sampling: negative, NaN and infinite temperatures; missing draft logits
    for T in (-1.0, float("nan"), float("inf")):
        assert L.spec_verify_sample(FAKE, FAKE, 0, FAKE, FAKE, 2, 10, 6, 0, T, FAKE, FAKE, FAKE,
                                    FAKE, null, null, FAKE, 1 << 20,
                                    null) == sv.SPEC_ERR_INVALID_ARG
    assert L.spec_verify_sample(FAKE, null, 0, FAKE, FAKE, 2, 10, 6, 0, 1.0, FAKE, FAKE, FAKE,
                                FAKE, null, null, FAKE, 1 << 20, null) == sv.SPEC_ERR_INVALID_ARG
    assert L.spec_verify_sample(FAKE, FAKE, 0, FAKE, FAKE, 2, 10, 6, 0, 1.0, FAKE, FAKE, FAKE,
                                FAKE, null, null, FAKE, 8, null) == sv.SPEC_ERR_WORKSPACE
    # D-cut
    assert L.dcut_allocate(FAKE, FAKE, -1, 4, 4, 0.0, FAKE, FAKE, null, FAKE, 1 << 20,
                           null) == sv.SPEC_ERR_INVALID_ARG
    assert L.dcut_allocate(FAKE, FAKE, 4, 33, 4, 0.0, FAKE, FAKE, null, FAKE, 1 << 20,
                           null) == sv.SPEC_ERR_INVALID_ARG
    assert L.dcut_allocate(FAKE, FAKE, 4, 4, -1, 0.0, FAKE, FAKE, null, FAKE, 1 << 20,
                           null) == sv.SPEC_ERR_INVALID_ARG
    assert L.dcut_allocate(FAKE, FAKE, 4, 4, 4, float("nan"), FAKE, FAKE, null, FAKE, 1 << 20,
                           null) == sv.SPEC_ERR_INVALID_ARG
    assert L.dcut_allocate(FAKE, FAKE, 1024, 16, 4, 0.0, FAKE, FAKE, null, FAKE, 1 << 20,
                           null) == sv.SPEC_ERR_INVALID_ARG  # 16384 candidates
    assert L.dcut_allocate(FAKE, FAKE, 4, 4, 4, 0.0, FAKE, FAKE, null, null, 0,
                           null) == sv.SPEC_ERR_WORKSPACE
    # D-cut, cost-unit variant
    assert L.dcut_allocate_cost(FAKE, FAKE, -1, 4, 4.0, FAKE, FAKE, null, FAKE, 1 << 20,
                                null) == sv.SPEC_ERR_INVALID_ARG
    assert L.dcut_allocate_cost(FAKE, FAKE, 4, 33, 4.0, FAKE, FAKE, null, FAKE, 1 << 20,
                                null) == sv.SPEC_ERR_INVALID_ARG
    assert L.dcut_allocate_cost(FAKE, FAKE, 4, 4, float("nan"), FAKE, FAKE, null, FAKE, 1 << 20,
                                null) == sv.SPEC_ERR_INVALID_ARG
    assert L.dcut_allocate_cost(FAKE, FAKE, 4097, 4, 4.0, FAKE, FAKE, null, FAKE, 1 << 20,
                                null) == sv.SPEC_ERR_INVALID_ARG
    assert L.dcut_allocate_cost(FAKE, FAKE, 4, 4, 4.0, FAKE, FAKE, null, null, 0,
                                null) == sv.SPEC_ERR_WORKSPACE


def test_trace_hook_arguments():
    assert sv.LIB.spec_set_trace(None, 0) == sv.SPEC_OK
    assert sv.LIB.spec_set_trace(None, 2) == sv.SPEC_ERR_INVALID_ARG
    arr = (ctypes.c_void_p * 17)()
    assert sv.LIB.spec_set_trace(arr, 17) == sv.SPEC_ERR_INVALID_ARG
    assert sv.spec_kernel_launch_count() >= 0


def test_binding_refuses_host_tensors():
    t = torch.zeros((4, 8))
    i32 = torch.zeros(8, dtype=torch.int32)
    ws = torch.zeros(1 << 16, dtype=torch.uint8)
    with pytest.raises(ValueError):
        sv.spec_verify_greedy(t, i32, torch.zeros(3, dtype=torch.int32), 2, 8, 4, 0, i32,
                              i32[:2], ws)
    with pytest.raises(ValueError):
        sv.dcut_allocate(torch.zeros((2, 2)), torch.zeros(2, dtype=torch.int32), 2, 2, 2, 0.0,
                         i32[:2], i32[:3], None, ws)


def test_expiry_hook_arguments():
    """The test-only expiry hook takes a unit index or -1 (off)."""
    assert sv.spec_test_expire_wait(-2) == sv.SPEC_ERR_INVALID_ARG
    assert sv.spec_test_expire_wait(5) == sv.SPEC_OK
    assert sv.spec_test_expire_wait(-1) == sv.SPEC_OK


def test_shard_host_checks_reject_before_any_launch():
    L = sv.LIB
    I = ctypes.c_int32
    assert sv.spec_shard_row_count(4, 20, 0) == 20 + 16
    assert sv.spec_shard_row_count(4, 20, 6) == 20 + 24
    assert sv.spec_shard_row_count(4, 3, 0) == -1
    assert sv.spec_shard_workspace_size(4, 20, 1000) > sv.spec_workspace_size(4, 20, 1000)
    assert sv.spec_shard_workspace_size(4, 20, 0) == 0
    # an empty shard, no shard, a first bound that is not 0
    for begin, n in (((0, 10, 10), 2), ((0, 10, 20), 0), ((1, 10, 20), 2)):
        arr = (I * 3)(*begin)
        assert L.spec_shard_accept(FAKE, n, arr, FAKE, FAKE, 1, 2, 0, 1.0, FAKE, FAKE, FAKE,
                                   None, None, FAKE, 1 << 20, None) == sv.SPEC_ERR_INVALID_ARG
    arr = (I * 3)(0, 10, 20)
    assert L.spec_shard_accept(FAKE, 2, None, FAKE, FAKE, 1, 2, 0, 1.0, FAKE, FAKE, FAKE, None,
                               None, FAKE, 1 << 20, None) == sv.SPEC_ERR_INVALID_ARG
    assert L.spec_shard_accept(FAKE, 2, arr, FAKE, FAKE, 1, 2, 0, 1.0, FAKE, FAKE, FAKE, None,
                               None, FAKE, 16, None) == sv.SPEC_ERR_WORKSPACE
    assert L.spec_shard_accept(FAKE, 2, arr, FAKE, FAKE, 1, 2, 0, 1.0, None, FAKE, FAKE, None,
                               None, FAKE, 1 << 20, None) == sv.SPEC_ERR_INVALID_ARG  # no u_accept
    # the drawing shard's index out of range; an empty column range
    assert L.spec_shard_final_draw(FAKE, FAKE, 0, FAKE, 2, 2, 1, 0, 10, 2, 0, FAKE, FAKE, FAKE,
                                   1 << 20, None) == sv.SPEC_ERR_INVALID_ARG
    assert L.spec_shard_row_stats(FAKE, FAKE, 0, FAKE, FAKE, 1, 10, 10, 2, 0, 1.0, FAKE, FAKE,
                                  1 << 20, None) == sv.SPEC_ERR_INVALID_ARG
    assert L.spec_shard_row_stats(FAKE, FAKE, 0, FAKE, FAKE, 1, 0, 10, 2, 0, -1.0, FAKE, FAKE,
                                  1 << 20, None) == sv.SPEC_ERR_INVALID_ARG
    # the draw's slice table: 64 slices of 12288 f32 columns at most
    assert L.spec_shard_final_mass(FAKE, FAKE, 0, 1, 0, 64 * 12288 + 1, 2, 0, FAKE, FAKE,
                                   1 << 30, None) == sv.SPEC_ERR_INVALID_ARG
    # B = 0 is a no-op for every step
    assert L.spec_shard_row_stats(None, None, 0, None, None, 0, 0, 10, 0, 0, 1.0, None, None, 0,
                                  None) == sv.SPEC_OK
    assert L.spec_shard_final_mass(None, None, 0, 0, 0, 10, 0, 0, None, None, 0,
                                   None) == sv.SPEC_OK
