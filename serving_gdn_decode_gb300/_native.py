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


class LayerBuffers(ctypes.Structure):
    """Mirror of gdn_layer_buffers and gdn_layer_buffers_bf16 (include/gdn.h):
    nine pointers in the same order in both."""
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "k", "v", "g", "beta", "state_in", "output",
                                                "state_out", "state_capture")]


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
            L.gdn_commit_capture.argtypes = [vp, sz, vp, vp, u32p, sz, vp]
            L.gdn_commit_capture.restype = ctypes.c_int
            L.gdn_forward_layers.argtypes = [ctypes.POINTER(LayerBuffers), sz, u32p, sz, ctypes.c_int,
                                             sz, vp]
            L.gdn_forward_layers.restype = ctypes.c_int
            L.gdn_forward_bf16.argtypes = L.gdn_forward.argtypes
            L.gdn_forward_bf16.restype = ctypes.c_int
            L.gdn_forward_capture_bf16.argtypes = L.gdn_forward_capture.argtypes
            L.gdn_forward_capture_bf16.restype = ctypes.c_int
            L.gdn_forward_layers_bf16.argtypes = L.gdn_forward_layers.argtypes
            L.gdn_forward_layers_bf16.restype = ctypes.c_int
            L.gdn_forward_ws.argtypes = [vp] * 8 + [u32p, sz, vp, sz, vp]
            L.gdn_forward_ws.restype = ctypes.c_int
            L.gdn_forward_ws_bf16.argtypes = L.gdn_forward_ws.argtypes
            L.gdn_forward_ws_bf16.restype = ctypes.c_int
            L.gdn_workspace_size.argtypes = [u32p, sz, ctypes.POINTER(ctypes.c_size_t)]
            L.gdn_workspace_size.restype = ctypes.c_int
            L.gdn_forward_chunked_noalloc.argtypes = [vp] * 8 + [u32p, sz, vp]
            L.gdn_forward_chunked_noalloc.restype = ctypes.c_int
            L.gdn_device_status.argtypes = [u32p, ctypes.c_int, vp]
            L.gdn_device_status.restype = ctypes.c_int
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


GDN_DEVICE_WAIT_TIMEOUT = 0x1


def gdn_device_status(reset: bool = False, stream=0) -> int:
    """The library's device status word on the current device (0 = no
    failure; GDN_DEVICE_WAIT_TIMEOUT when a chunked kernel's bounded wait ran
    out), after all work enqueued on ``stream`` so far (the call synchronises
    that stream); cleared afterwards when ``reset``."""
    out = ctypes.c_uint32()
    st = lib().gdn_device_status(ctypes.byref(out), 1 if reset else 0, _stream_ptr(stream))
    if st != GDN_OK:
        raise GdnError(st, gdn_last_error())
    return int(out.value)


def _stream_ptr(stream) -> int:
    if stream is None or isinstance(stream, int):
        return int(stream or 0)
    return int(getattr(stream, "cuda_stream", stream))


def gdn_workspace_size(params) -> int:
    """Bytes of device workspace gdn_forward_ws needs for ``params`` (0 off
    the chunked path)."""
    p, pp, n = _params_arg(params)
    out = ctypes.c_size_t()
    st = lib().gdn_workspace_size(pp, n, ctypes.byref(out))
    if st != GDN_OK:
        raise GdnError(st, gdn_last_error())
    return out.value


# ---------------------------------------------------------------- raw calls

def forward_raw(q, k, v, g, beta, state_in, output, state_out, params, stream=0,
                bf16=False) -> int:
    """Call gdn_forward (gdn_forward_bf16 when ``bf16``) with integer device
    addresses; returns the status."""
    p, pp, n = _params_arg(params)
    fn = lib().gdn_forward_bf16 if bf16 else lib().gdn_forward
    return fn(q, k, v, g, beta, state_in, output, state_out, pp, n, stream)


def forward_ws_raw(q, k, v, g, beta, state_in, output, state_out, params, workspace,
                   workspace_bytes, stream=0, bf16=False) -> int:
    """Call gdn_forward_ws (gdn_forward_ws_bf16 when ``bf16``) with integer
    device addresses; returns the status."""
    p, pp, n = _params_arg(params)
    fn = lib().gdn_forward_ws_bf16 if bf16 else lib().gdn_forward_ws
    return fn(q, k, v, g, beta, state_in, output, state_out, pp, n, workspace, workspace_bytes, stream)


def forward_chunked_noalloc_raw(q, k, v, g, beta, state_in, output, state_out, params,
                                stream=0) -> int:
    """Call gdn_forward_chunked_noalloc (two-pass chunked prefill on the
    library's fixed scratch) with integer device addresses; returns the
    status."""
    p, pp, n = _params_arg(params)
    return lib().gdn_forward_chunked_noalloc(q, k, v, g, beta, state_in, output, state_out, pp, n,
                                             stream)


def forward_capture_raw(q, k, v, g, beta, state_in, output, state_out, params, state_capture,
                        state_capture_elems, stream=0, bf16=False) -> int:
    """Call gdn_forward_capture (gdn_forward_capture_bf16 when ``bf16``) with
    integer device addresses; returns the status."""
    p, pp, n = _params_arg(params)
    fn = lib().gdn_forward_capture_bf16 if bf16 else lib().gdn_forward_capture
    return fn(q, k, v, g, beta, state_in, output, state_out, pp, n, state_capture,
              state_capture_elems, stream)


def forward_layers_raw(layers, params, with_capture=False, state_capture_elems=0, stream=0,
                       bf16=False) -> int:
    """Call gdn_forward_layers (gdn_forward_layers_bf16 when ``bf16``) with
    per-layer tuples of 9 integer device addresses (q, k, v, g, beta,
    state_in, output, state_out, state_capture); returns the status."""
    p, pp, n = _params_arg(params)
    arr = (LayerBuffers * max(1, len(layers)))(*[LayerBuffers(*lay) for lay in layers])
    fn = lib().gdn_forward_layers_bf16 if bf16 else lib().gdn_forward_layers
    return fn(arr if layers else None, len(layers), pp, n, 1 if with_capture else 0,
              state_capture_elems, stream)


def commit_capture_raw(state_capture, state_capture_elems, accepted_idx, state, params,
                       stream=0) -> int:
    """Call gdn_commit_capture with integer device addresses; returns the status."""
    p, pp, n = _params_arg(params)
    return lib().gdn_commit_capture(state_capture, state_capture_elems, accepted_idx, state, pp, n,
                                    stream)


# ---------------------------------------------------------------- torch tensors

def _dtype_name(dtype) -> str:
    import torch
    return "bf16" if dtype == torch.bfloat16 else "f32"


def _check(name, t, expect_numel, allow_larger=False, dtype=None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    dtype = torch.float32 if dtype is None else dtype
    if t.dtype != dtype:
        raise GdnError(GDN_ERR_INVALID_ARGUMENT,
                       f"{name} must be {_dtype_name(dtype)} (got {t.dtype})")
    if not t.is_cuda:
        raise GdnError(GDN_ERR_INVALID_ARGUMENT, f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise GdnError(GDN_ERR_INVALID_ARGUMENT, f"{name} must be contiguous")
    n = t.numel()
    if (n != expect_numel) and not (allow_larger and n > expect_numel):
        raise GdnError(GDN_ERR_INVALID_ARGUMENT,
                       f"{name} element count {n} != expected {expect_numel}")
    return t.data_ptr()


def _act_dtype(q):
    """Activation dtype of a call, taken from q: f32 (gdn_forward) or bf16
    (gdn_forward_bf16); k, v and output must match it."""
    import torch
    if isinstance(q, torch.Tensor) and q.dtype in (torch.float32, torch.bfloat16):
        return q.dtype
    raise GdnError(GDN_ERR_INVALID_ARGUMENT,
                   f"q must be an f32 or bf16 torch.Tensor (got {getattr(q, 'dtype', type(q))})")


def _check_dtypes(prefix, act, k, v, g, beta, state_in, output, state_out):
    """Every buffer's dtype, before any other check, so that a mixed-dtype
    call is reported as such."""
    import torch
    f32 = torch.float32
    for name, t, want in (("k", k, act), ("v", v, act), ("g", g, f32), ("beta", beta, f32),
                          ("state_in", state_in, f32), ("output", output, act),
                          ("state_out", state_out, f32)):
        if isinstance(t, torch.Tensor) and t.dtype != want:
            raise GdnError(GDN_ERR_INVALID_ARGUMENT,
                           f"{prefix}{name} must be {_dtype_name(want)} (got {t.dtype})")


def _act_ptrs(prefix, q, k, v, g, beta, state_in, output, state_out, s):
    """Checked device addresses of the eight buffers of one call, and whether
    the activations (q, k, v, output) are bf16."""
    import torch
    act = _act_dtype(q)
    _check_dtypes(prefix, act, k, v, g, beta, state_in, output, state_out)
    ptrs = [_check(prefix + "q", q, s["qk"], dtype=act), _check(prefix + "k", k, s["qk"], dtype=act),
            _check(prefix + "v", v, s["v"], dtype=act), _check(prefix + "g", g, s["sc"]),
            _check(prefix + "beta", beta, s["sc"]),
            _check(prefix + "state_in", state_in, s["state"]),
            _check(prefix + "output", output, s["v"], dtype=act),
            _check(prefix + "state_out", state_out, s["state"])]
    return ptrs, act == torch.bfloat16


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
    """Run gdn_forward on torch CUDA tensors (flat, the layouts of
    include/gdn.h).  q, k, v and output are all f32, or all bf16 (then
    gdn_forward_bf16 runs); g, beta and the states are f32.  Checks dtype,
    device, contiguity and element counts (the per-buffer checks of
    `validate` in gated_delta_net_decode.rs), then hands the device pointers
    to the C ABI.  Raises GdnError on failure."""
    s = _sizes(params)
    ptrs, bf16 = _act_ptrs("", q, k, v, g, beta, state_in, output, state_out, s)
    st = forward_raw(*ptrs, params, _stream(stream, q.device), bf16=bf16)
    if st != GDN_OK:
        raise GdnError(st, gdn_last_error())


def gdn_forward_capture(q, k, v, g, beta, state_in, output, state_out, params, state_capture,
                        stream=None) -> None:
    """gdn_forward plus the per-token state written to ``state_capture``
    ([D_k, D_v, n_v, n_tokens, n_seqs]; may be larger than needed when
    n_seqs == 1, as dispatch_gated_delta_net_decode_with_capture allows)."""
    s = _sizes(params)
    ptrs, bf16 = _act_ptrs("", q, k, v, g, beta, state_in, output, state_out, s)
    cap = _check("state_capture", state_capture, s["state"] * s["nt"], allow_larger=s["ns"] == 1)
    st = forward_capture_raw(*ptrs, params, cap, state_capture.numel(),
                             _stream(stream, q.device), bf16=bf16)
    if st != GDN_OK:
        raise GdnError(st, gdn_last_error())


def gdn_forward_ws(q, k, v, g, beta, state_in, output, state_out, params, workspace,
                   stream=None) -> None:
    """gdn_forward with a device workspace (a contiguous CUDA tensor of any
    dtype holding at least gdn_workspace_size(params) bytes, or None when that
    is 0).  On the chunked path the two-pass form runs; elsewhere as
    gdn_forward.  q, k, v and output all f32, or all bf16 (then
    gdn_forward_ws_bf16 runs)."""
    import torch
    s = _sizes(params)
    ptrs, bf16 = _act_ptrs("", q, k, v, g, beta, state_in, output, state_out, s)
    if workspace is None:
        wp, wb = None, 0
    else:
        if (not isinstance(workspace, torch.Tensor) or not workspace.is_cuda
                or not workspace.is_contiguous()):
            raise GdnError(GDN_ERR_INVALID_ARGUMENT, "workspace must be a contiguous CUDA tensor")
        wp, wb = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    st = forward_ws_raw(*ptrs, params, wp, wb, _stream(stream, q.device), bf16=bf16)
    if st != GDN_OK:
        raise GdnError(st, gdn_last_error())


def gdn_commit_capture(state_capture, accepted_idx, state, params, stream=None) -> None:
    """Speculative-decode rollback on torch CUDA tensors: for every sequence s
    with 0 <= accepted_idx[s] < n_tokens, state[.., s] = state_capture[.., accepted_idx[s], s];
    other sequences keep their state.  ``accepted_idx`` is an int32 CUDA tensor
    of n_seqs entries (read on the device)."""
    import torch
    s = _sizes(params)
    cap = _check("state_capture", state_capture, s["state"] * s["nt"], allow_larger=s["ns"] == 1)
    stp = _check("state", state, s["state"])
    if (not isinstance(accepted_idx, torch.Tensor) or accepted_idx.dtype != torch.int32
            or not accepted_idx.is_cuda or not accepted_idx.is_contiguous()
            or accepted_idx.numel() != s["ns"]):
        raise GdnError(GDN_ERR_INVALID_ARGUMENT,
                       "accepted_idx must be a contiguous int32 CUDA tensor of n_seqs entries")
    st = commit_capture_raw(cap, state_capture.numel(), accepted_idx.data_ptr(), stp, params,
                            _stream(stream, state.device))
    if st != GDN_OK:
        raise GdnError(st, gdn_last_error())


def gdn_forward_layers(layers, params, with_capture: bool = False, stream=None) -> None:
    """gdn_forward (or gdn_forward_capture) on several problems of one shape,
    such as the linear-attention layers of a forward pass: ``layers`` is a list
    of dicts with torch CUDA tensors under the keys q, k, v, g, beta, state_in,
    output, state_out (and state_capture when ``with_capture``).  On the decode
    path all layers run in one launch (per 64 layers).  Activations are f32
    or bf16, the same for every layer."""
    s = _sizes(params)
    rows, cap_elems = [], 0
    dev = None
    bf16 = None
    for i, L in enumerate(layers):
        ptrs, b = _act_ptrs(f"layers[{i}].", L["q"], L["k"], L["v"], L["g"], L["beta"],
                            L["state_in"], L["output"], L["state_out"], s)
        if bf16 is not None and b != bf16:
            raise GdnError(GDN_ERR_INVALID_ARGUMENT, "activation dtypes differ between layers")
        bf16 = b
        if with_capture:
            c = L["state_capture"]
            ptrs.append(_check(f"layers[{i}].state_capture", c, s["state"] * s["nt"],
                               allow_larger=s["ns"] == 1))
            if i == 0:
                cap_elems = c.numel()
            elif c.numel() != cap_elems:
                raise GdnError(GDN_ERR_INVALID_ARGUMENT, "state_capture sizes differ between layers")
        else:
            ptrs.append(None)
        rows.append(ptrs)
        dev = L["q"].device
    if not rows:
        raise GdnError(GDN_ERR_INVALID_ARGUMENT, "no layers")
    st = forward_layers_raw(rows, params, with_capture, cap_elems, _stream(stream, dev), bf16=bf16)
    if st != GDN_OK:
        raise GdnError(st, gdn_last_error())


# ---------------------------------------------------------------- host buffers

def _check_host(name, t, expect_numel, dtype):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.is_cuda or not t.is_pinned() or not t.is_contiguous() or t.dtype != dtype:
        raise GdnError(GDN_ERR_INVALID_ARGUMENT,
                       f"{name} must be a contiguous {_dtype_name(dtype)} pinned host tensor")
    if t.numel() != expect_numel:
        raise GdnError(GDN_ERR_INVALID_ARGUMENT,
                       f"{name} element count {t.numel()} != expected {expect_numel}")
    return t.data_ptr()


def gdn_forward_host(q, k, v, g, beta, state_in, output, state_out, params, state_capture=None,
                     stream=None, device=None) -> None:
    """gdn_forward (gdn_forward_capture when ``state_capture`` is given) on
    PINNED HOST tensors, zero-copy: the kernel reads the inputs from host
    memory and writes output, state and capture back to host memory itself,
    over the CPU-GPU link, with no staging copy.  Pinned host memory is
    device-accessible, and under CUDA's unified addressing (every 64-bit
    platform) its device address is its host address, so the host pointers
    go to the C ABI unchanged.  Same dtype rules as gdn_forward (q, k, v and
    output f32 or all bf16).  Runs on ``stream`` (default: the current stream
    of ``device``, default the current device) and does not block the host:
    synchronise before reading the results."""
    import torch
    s = _sizes(params)
    act = _act_dtype(q)
    f32 = torch.float32
    _check_dtypes("", act, k, v, g, beta, state_in, output, state_out)
    ptrs = [_check_host("q", q, s["qk"], act), _check_host("k", k, s["qk"], act),
            _check_host("v", v, s["v"], act), _check_host("g", g, s["sc"], f32),
            _check_host("beta", beta, s["sc"], f32),
            _check_host("state_in", state_in, s["state"], f32),
            _check_host("output", output, s["v"], act),
            _check_host("state_out", state_out, s["state"], f32)]
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    strm = _stream(stream, dev)
    bf16 = act == torch.bfloat16
    if state_capture is None:
        st = forward_raw(*ptrs, params, strm, bf16=bf16)
    else:
        need = s["state"] * s["nt"]
        n_cap = state_capture.numel() if isinstance(state_capture, torch.Tensor) else -1
        cap = _check_host("state_capture", state_capture,
                          max(n_cap, need) if s["ns"] == 1 else need, f32)
        st = forward_capture_raw(*ptrs, params, cap, state_capture.numel(), strm, bf16=bf16)
    if st != GDN_OK:
        raise GdnError(st, gdn_last_error())


class HostPipeline:
    """Run gdn_forward on PINNED HOST tensors, end to end.

    Sequences are independent and n_seqs is the outermost dimension of every
    buffer.  q, k, v, g, beta (small) are copied in with one copy each; the
    state, which dominates the bytes, is cut into `groups` groups of sequences
    so that group i's state is copied in on one stream while group i-1 runs
    and group i-2's new state is copied out on a third stream (the two copy
    directions overlap).  Device buffers of the full problem size are
    allocated once (by torch) at construction and reused by every call.
    """

    SMALL_INPUTS = ("q", "k", "v", "g", "beta")

    def __init__(self, params, groups: int = 4, device=None):
        import torch
        p = np.asarray(params, dtype=np.uint32).reshape(-1)
        self.params = p.copy()
        dk, dv, nk, nv, nt, ns = (int(x) for x in p[:6])
        self.ns = ns
        self.group = max(1, -(-ns // max(1, groups)))
        self.per_seq = dict(q=dk * nk * nt, k=dk * nk * nt, v=dv * nv * nt, g=nv * nt,
                            beta=nv * nt, state_in=dk * dv * nv, output=dv * nv * nt,
                            state_out=dk * dv * nv)
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        self.device = dev
        self.buf = {k: torch.empty(n * ns, dtype=torch.float32, device=dev)
                    for k, n in self.per_seq.items()}
        self.s_in = torch.cuda.Stream(dev)
        self.s_run = torch.cuda.Stream(dev)
        self.s_out = torch.cuda.Stream(dev)

    def h2d_bytes(self) -> int:
        return 4 * self.ns * sum(self.per_seq[k] for k in self.SMALL_INPUTS + ("state_in",))

    def d2h_bytes(self) -> int:
        return 4 * self.ns * (self.per_seq["output"] + self.per_seq["state_out"])

    def __call__(self, q, k, v, g, beta, state_in, output, state_out, stream=None):
        """Inputs and outputs: flat f32 pinned host tensors in the layouts of
        include/gdn.h.  Work is ordered after `stream` (default: the current
        stream), and `stream` waits for all of it; the host does not block."""
        import torch
        host = dict(q=q, k=k, v=v, g=g, beta=beta, state_in=state_in, output=output,
                    state_out=state_out)
        for name, t in host.items():
            if t.is_cuda or not t.is_pinned() or t.dtype != torch.float32 or not t.is_contiguous():
                raise GdnError(GDN_ERR_INVALID_ARGUMENT,
                               f"{name} must be a contiguous f32 pinned host tensor")
            if t.numel() != self.per_seq[name] * self.ns:
                raise GdnError(GDN_ERR_INVALID_ARGUMENT,
                               f"{name} element count {t.numel()} != {self.per_seq[name] * self.ns}")
        base = torch.cuda.current_stream(self.device) if stream is None else stream
        for s in (self.s_in, self.s_run, self.s_out):
            s.wait_stream(base)
        buf = self.buf
        with torch.cuda.stream(self.s_in):
            for name in self.SMALL_INPUTS:
                buf[name].copy_(host[name], non_blocking=True)
        m_st = self.per_seq["state_in"]
        for s0 in range(0, self.ns, self.group):
            n = min(self.group, self.ns - s0)
            sl = slice(s0 * m_st, (s0 + n) * m_st)
            with torch.cuda.stream(self.s_in):
                buf["state_in"][sl].copy_(host["state_in"][sl], non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(self.s_in)
            with torch.cuda.stream(self.s_run):
                self.s_run.wait_event(ev_in)
                p = self.params.copy()
                p[5] = n
                args = [buf[x][s0 * self.per_seq[x]:(s0 + n) * self.per_seq[x]] for x in
                        ("q", "k", "v", "g", "beta", "state_in", "output", "state_out")]
                gdn_forward(*args, p, stream=self.s_run)
                ev_run = torch.cuda.Event()
                ev_run.record(self.s_run)
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(ev_run)
                host["state_out"][sl].copy_(buf["state_out"][sl], non_blocking=True)
        with torch.cuda.stream(self.s_out):
            self.s_out.wait_stream(self.s_run)
            host["output"].copy_(buf["output"], non_blocking=True)
        for s in (self.s_in, self.s_run, self.s_out):
            base.wait_stream(s)
