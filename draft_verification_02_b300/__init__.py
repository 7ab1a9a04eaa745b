"""B300 (sm_103a) batched draft verification and D-cut.

The C-ABI binding (``specverify``) loads ``libspecverify.so`` and raises if it
is missing: the verification path runs only in the library's CUDA kernels.
``workloads`` (seeded synthetic inputs) imports without the library.
"""
import importlib

_BINDING_NAMES = {
    "spec_workspace_size", "spec_workspace_init", "spec_verify_greedy", "spec_verify_sample",
    "dcut_allocate", "spec_get_device_status", "spec_status_string", "spec_set_trace",
    "spec_kernel_launch_count", "spec_verify_sample_static", "dcut_allocate_cost",
    "spec_draft_confidence", "spec_draft_sample", "spec_acceptance_stats",
    "spec_shard_workspace_size", "spec_shard_row_count", "spec_shard_row_stats",
    "spec_shard_accept", "spec_shard_final_mass", "spec_shard_final_draw",
    "SpecError", "check",
}


def __getattr__(name):
    if name in _BINDING_NAMES:
        return getattr(importlib.import_module(".specverify", __name__), name)
    if name == "Verifier":
        return importlib.import_module(".verifier", __name__).Verifier
    if name in ("Shard", "verify_sharded", "verify_sharded_local"):
        return getattr(importlib.import_module(".sharded", __name__), name)
    raise AttributeError(name)
