"""GB300-native (sm_103a) Gated DeltaNet recurrence: decode, per-token state
capture for speculative-decode rollback, and long prefill.

The compute lives in ``libgdn_gb300.so`` (CUDA kernels behind the C ABI of
``include/gdn.h``); this package is its thin Python binding plus the
parameter packer and the seeded synthetic-input generator.
"""
from .params import (FLAG_DECAY_AFTER, FLAG_KHEAD_DIV, N_PARAMS, PATH_AUTO, PATH_CHUNKED,
                     PATH_CHUNKED_TF32, PATH_SCAN, pack_params, q_scale_bits)

__all__ = ["FLAG_DECAY_AFTER", "FLAG_KHEAD_DIV", "N_PARAMS", "PATH_AUTO", "PATH_CHUNKED",
           "PATH_CHUNKED_TF32", "PATH_SCAN", "pack_params", "q_scale_bits", "gdn_forward", "gdn_forward_capture",
           "gdn_last_error", "gdn_path_name", "gdn_commit_capture", "gdn_forward_layers",
           "gdn_forward_host", "gdn_forward_ws", "gdn_workspace_size", "HostPipeline", "GdnError"]

_NATIVE = ("gdn_forward", "gdn_forward_capture", "gdn_last_error", "gdn_path_name",
           "gdn_commit_capture", "gdn_forward_layers", "gdn_forward_host", "gdn_forward_ws",
           "gdn_workspace_size", "HostPipeline", "GdnError")


def __getattr__(name):
    # The native binding loads on first use, so importing the package (for
    # the parameter packer or the input generator) needs no GPU library.
    if name in _NATIVE:
        from . import _native
        return getattr(_native, name)
    raise AttributeError(name)
