"""Double-precision CPU oracle of the Gated DeltaNet recurrence.

TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the
benchmark's CPU-baseline leg are the only callers.  The CUDA library and its
Python binding never import this package, and this package imports nothing
from them.

The arithmetic lives in ``gdn_oracle.c`` (plain C, double precision,
threaded over (seq, value-head) pairs); this module builds it with gcc and
marshals numpy arrays to it.  ``build()`` compiles the C source; ``forward``
and ``forward_heads`` run it.

Layouts, parameters and the two flag readings are documented in the C file.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB = os.path.join(_HERE, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
BAD_ARGUMENT = 1
NO_MEMORY = 2


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c into libgdn_oracle.so next to it (gcc, no FMA
    contraction so results are the same on x86-64 and aarch64)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-pthread", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
            lib.gdn_oracle_forward.argtypes = [vp, sz, vp, vp, vp, vp, vp, vp, i, vp, vp, vp, i]
            lib.gdn_oracle_forward.restype = i
            lib.gdn_oracle_forward_heads.argtypes = [vp, sz, vp, vp, vp, vp, vp, vp, i, vp, sz,
                                                     vp, vp, vp, i]
            lib.gdn_oracle_forward_heads.restype = i
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(a):
    return np.ascontiguousarray(np.asarray(a), dtype=np.float32).reshape(-1)


def _state(a):
    a = np.asarray(a)
    if a.dtype == np.float64:
        return np.ascontiguousarray(a).reshape(-1), 1
    return _f32(a), 0


def _params(params):
    return np.ascontiguousarray(np.asarray(params, dtype=np.uint32)).reshape(-1)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


class OracleError(RuntimeError):
    pass


def forward(params, q, k, v, g, beta, state_in, capture: bool = False, n_threads: int | None = None):
    """Run the whole problem.

    Returns ``(output, state_out, state_capture)`` as flat float64 arrays in
    the pages' innermost-first layouts (``state_capture`` is None unless
    ``capture``).  ``state_in`` may be float32 or float64.
    """
    lib = _load()
    p = _params(params)
    dk, dv, nk, nv, nt, ns = (int(x) for x in p[:6])
    out = np.empty(dv * nv * nt * ns, dtype=np.float64)
    st = np.empty(dk * dv * nv * ns, dtype=np.float64)
    cap = np.empty(dk * dv * nv * nt * ns, dtype=np.float64) if capture else None
    qa, ka, va, ga, ba = (_f32(x) for x in (q, k, v, g, beta))
    sa, s64 = _state(state_in)
    rc = lib.gdn_oracle_forward(_ptr(p), p.size, _ptr(qa), _ptr(ka), _ptr(va), _ptr(ga), _ptr(ba),
                                _ptr(sa), s64, _ptr(out), _ptr(st), _ptr(cap),
                                n_threads or default_threads())
    if rc != OK:
        raise OracleError(f"gdn_oracle_forward returned {rc}")
    return out, st, cap


def forward_heads(params, q, k, v, g, beta, state_in, heads, capture: bool = False,
                  n_threads: int | None = None):
    """Run only the listed heads (``head = s * n_v_heads + vh``) of a
    full-layout problem.

    Returns compact float64 arrays ``output [n][T][D_v]``,
    ``state_out [n][D_v][D_k]`` and ``state_capture [n][T][D_v][D_k]``
    (None unless ``capture``).
    """
    lib = _load()
    p = _params(params)
    dk, dv, nk, nv, nt, ns = (int(x) for x in p[:6])
    h = np.ascontiguousarray(np.asarray(heads, dtype=np.uint32)).reshape(-1)
    n = h.size
    out = np.empty((n, nt, dv), dtype=np.float64)
    st = np.empty((n, dv, dk), dtype=np.float64)
    cap = np.empty((n, nt, dv, dk), dtype=np.float64) if capture else None
    qa, ka, va, ga, ba = (_f32(x) for x in (q, k, v, g, beta))
    sa, s64 = _state(state_in)
    rc = lib.gdn_oracle_forward_heads(_ptr(p), p.size, _ptr(qa), _ptr(ka), _ptr(va), _ptr(ga),
                                      _ptr(ba), _ptr(sa), s64, _ptr(h), n, _ptr(out), _ptr(st),
                                      _ptr(cap), n_threads or default_threads())
    if rc != OK:
        raise OracleError(f"gdn_oracle_forward_heads returned {rc}")
    return out, st, cap
