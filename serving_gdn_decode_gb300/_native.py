"""ctypes binding of libgdn_gb300.so.

Argument marshalling only: every step of the recurrence runs in the CUDA
library.  There is no fallback: if the library is missing or cannot load,
every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import numpy as np

from .params import N_PARAMS

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgdn_gb300.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "gdn.h")

GDN_OK = 0
GDN_ERR_INVALID_ARGUMENT = 1
GDN_ERR_UNSUPPORTED = 2
GDN_ERR_CUDA = 3
STATUS_NAMES = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARGUMENT", 2: "GDN_ERR_UNSUPPORTED",
                3: "GDN_ERR_CUDA"}

_lock = threading.Lock()
_lib = None


class GdnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status
        self.message = message


def lib() -> ctypes.CDLL:
    """Load libgdn_gb300.so (built by ``serving_gdn_decode_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with `python -m serving_gdn_decode_gb300.build`"
                    " (there is no CPU fallback)")
            L = ctypes.CDLL(LIB_PATH)
            vp, sz, u32p = ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(ctypes.c_uint32)
            L.gdn_forward.argtypes = [vp] * 8 + [u32p, sz, vp]
            L.gdn_forward.restype = ctypes.c_int
            L.gdn_forward_capture.argtypes = [vp] * 8 + [u32p, sz, vp, sz, vp]
            L.gdn_forward_capture.restype = ctypes.c_int
            L.gdn_last_error.argtypes = []
            L.gdn_last_error.restype = ctypes.c_char_p
            L.gdn_path_name.argtypes = [u32p, sz, ctypes.c_int, ctypes.POINTER(ctypes.c_char_p)]
            L.gdn_path_name.restype = ctypes.c_int
            _lib = L
    return _lib


def header_functions() -> list[str]:
    """Names of the functions include/gdn.h declares."""
    with open(HEADER_PATH) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_0-9]+)\s*\(", text)))


def _params_arg(params):
    p = np.ascontiguousarray(np.asarray(params, dtype=np.uint32)).reshape(-1)
    return p, p.ctypes.data_as(ctypes.POINTER(ctypes.c_uint32)), p.size


def gdn_last_error() -> str:
    return lib().gdn_last_error().decode()


def gdn_path_name(params, capture: bool = False) -> str:
    p, pp, n = _params_arg(params)
    name = ctypes.c_char_p()
    st = lib().gdn_path_name(pp, n, 1 if capture else 0, ctypes.byref(name))
    if st != GDN_OK:
        raise GdnError(st, gdn_last_error())
    return name.value.decode()


# ---------------------------------------------------------------- raw calls

def forward_raw(q, k, v, g, beta, state_in, output, state_out, params, stream=0) -> int:
    """Call gdn_forward with integer device addresses; returns the status."""
    p, pp, n = _params_arg(params)
    return lib().gdn_forward(q, k, v, g, beta, state_in, output, state_out, pp, n, stream)


def forward_capture_raw(q, k, v, g, beta, state_in, output, state_out, params, state_capture,
                        state_capture_elems, stream=0) -> int:
    """Call gdn_forward_capture with integer device addresses; returns the status."""
    p, pp, n = _params_arg(params)
    return lib().gdn_forward_capture(q, k, v, g, beta, state_in, output, state_out, pp, n,
                                     state_capture, state_capture_elems, stream)


# ---------------------------------------------------------------- torch tensors

def _check(name, t, expect_numel, allow_larger=False):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.float32:
        raise GdnError(GDN_ERR_INVALID_ARGUMENT, f"{name} must be f32 (got {t.dtype})")
    if not t.is_cuda:
        raise GdnError(GDN_ERR_INVALID_ARGUMENT, f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise GdnError(GDN_ERR_INVALID_ARGUMENT, f"{name} must be contiguous")
    n = t.numel()
    if (n != expect_numel) and not (allow_larger and n > expect_numel):
        raise GdnError(GDN_ERR_INVALID_ARGUMENT,
                       f"{name} element count {n} != expected {expect_numel}")
    return t.data_ptr()


def _sizes(params):
    p = np.asarray(params, dtype=np.uint32).reshape(-1)
    if p.size < N_PARAMS:
        raise GdnError(GDN_ERR_INVALID_ARGUMENT, f"params has {p.size} u32, expected >= 9")
    dk, dv, nk, nv, nt, ns = (int(x) for x in p[:6])
    return dict(qk=dk * nk * nt * ns, v=dv * nv * nt * ns, sc=nv * nt * ns,
                state=dk * dv * nv * ns, ns=ns, nt=nt)


def _stream(stream, device):
    import torch
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def gdn_forward(q, k, v, g, beta, state_in, output, state_out, params, stream=None) -> None:
    """Run gdn_forward on torch CUDA tensors (flat f32, the layouts of
    include/gdn.h).  Checks dtype, device, contiguity and element counts
    (the per-buffer checks of `validate` in gated_delta_net_decode.rs), then
    hands the device pointers to the C ABI.  Raises GdnError on failure."""
    s = _sizes(params)
    ptrs = [_check("q", q, s["qk"]), _check("k", k, s["qk"]), _check("v", v, s["v"]),
            _check("g", g, s["sc"]), _check("beta", beta, s["sc"]),
            _check("state_in", state_in, s["state"]), _check("output", output, s["v"]),
            _check("state_out", state_out, s["state"])]
    st = forward_raw(*ptrs, params, _stream(stream, q.device))
    if st != GDN_OK:
        raise GdnError(st, gdn_last_error())


def gdn_forward_capture(q, k, v, g, beta, state_in, output, state_out, params, state_capture,
                        stream=None) -> None:
    """gdn_forward plus the per-token state written to ``state_capture``
    ([D_k, D_v, n_v, n_tokens, n_seqs]; may be larger than needed when
    n_seqs == 1, as dispatch_gated_delta_net_decode_with_capture allows)."""
    s = _sizes(params)
    ptrs = [_check("q", q, s["qk"]), _check("k", k, s["qk"]), _check("v", v, s["v"]),
            _check("g", g, s["sc"]), _check("beta", beta, s["sc"]),
            _check("state_in", state_in, s["state"]), _check("output", output, s["v"]),
            _check("state_out", state_out, s["state"])]
    cap = _check("state_capture", state_capture, s["state"] * s["nt"], allow_larger=s["ns"] == 1)
    st = forward_capture_raw(*ptrs, params, cap, state_capture.numel(),
                             _stream(stream, q.device))
    if st != GDN_OK:
        raise GdnError(st, gdn_last_error())
