"""The lazy-decay form that the FP32 scan kernel evaluates, written out in
float64 numpy, against the oracle's token-by-token recurrence.

The scan keeps the state as S = c * St, c the product of the decays since the
last fold.  Over a chunk of 16 tokens, with G_t the prefix sums of g from the
chunk's first token and c_t = e^-G_t (c = 1 entering the chunk):

    x     = St @ k_t
    delta = (v_t - c' x) beta_t        c' = c_t (decay-first), c_{t-1} (decay-after)
    St   += (delta / c_t) k_t^T
    y_t   = q_scale c_t (St @ q_t),    state_capture[t] = c_t St

and c is folded into St at the chunk's end.  A chunk in which some |G_t|
exceeds 40 runs the plain recurrence instead (explicit decay each token).
The GPU tests hold the kernel to the oracle within its float32 bar; this
test shows on the CPU that the form itself is exact up to float64 rounding.
"""
import numpy as np
import pytest

from serving_gdn_decode_gb300.params import PATH_SCAN
from serving_gdn_decode_gb300.workloads import Workload, make_inputs

TC = 16
MAX_LOG = 40.0


def _q_scale(params):
    bits = int(params[8])
    return 1.0 if bits == 0 else float(np.array([bits], dtype=np.uint32).view(np.float32)[0])


def scan_forward(params, q, k, v, g, beta, state_in, stats=None, mutate=None):
    """The lazy-decay form above for a whole problem; returns flat (output,
    state_out, state_capture) in the library's innermost-first layouts."""
    dk, dv, nk, nv, nt, ns = (int(x) for x in params[:6])
    decay_after = bool(int(params[6]) & 1)
    khead_div = bool(int(params[6]) & 2)
    qs = _q_scale(params)
    q = q.astype(np.float64).reshape(ns, nt, nk, dk)
    k = k.astype(np.float64).reshape(ns, nt, nk, dk)
    v = v.astype(np.float64).reshape(ns, nt, nv, dv)
    g = g.astype(np.float64).reshape(ns, nt, nv)
    beta = beta.astype(np.float64).reshape(ns, nt, nv)
    state = state_in.astype(np.float64).reshape(ns, nv, dv, dk)
    out = np.zeros((ns, nt, nv, dv))
    cap = np.zeros((ns, nt, nv, dv, dk))
    st_out = np.zeros_like(state)
    if stats is not None:
        stats.update(lazy=0, explicit=0)
    for s in range(ns):
        for vh in range(nv):
            kh = vh // (nv // nk) if khead_div else vh % nk
            St = state[s, vh].copy()
            for t0 in range(0, nt, TC):
                ts = range(t0, min(nt, t0 + TC))
                G = np.cumsum(g[s, t0:t0 + len(ts), vh])
                explicit = bool(np.any(np.abs(G) > MAX_LOG))
                if stats is not None:
                    stats["explicit" if explicit else "lazy"] += 1
                c_prev = 1.0
                for n, t in enumerate(ts):
                    kt, qt, vt, b = k[s, t, kh], q[s, t, kh], v[s, t, vh], beta[s, t, vh]
                    if explicit:
                        alpha = np.exp(-g[s, t, vh])
                        if decay_after:
                            St = alpha * St + b * np.outer(vt - St @ kt, kt)
                        else:
                            St = alpha * St
                            St = St + b * np.outer(vt - St @ kt, kt)
                        out[s, t, vh] = qs * (St @ qt)
                        cap[s, t, vh] = St
                        continue
                    c_t = np.exp(-G[n])
                    x = St @ kt
                    c_sk = c_prev if decay_after else c_t
                    if mutate == "c_sk_swapped":
                        c_sk = c_t if decay_after else c_prev
                    delta = (vt - c_sk * x) * b
                    St = St + np.outer(delta / (c_t if mutate != "no_divide" else 1.0), kt)
                    y_scale = c_t if mutate != "y_without_c" else 1.0
                    out[s, t, vh] = qs * y_scale * (St @ qt)
                    cap[s, t, vh] = c_t * St
                    c_prev = c_t
                if not explicit and mutate != "no_fold":
                    St = c_prev * St
            st_out[s, vh] = St
    return out.reshape(-1), st_out.reshape(-1), cap.reshape(-1)


def _max_rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def _gates(w, kind, rng):
    if kind == "plain":
        return rng.uniform(0.0, 0.5, w.scalar_elems).astype(np.float32)
    if kind == "negative":  # growing states: c > 1
        return rng.uniform(-0.12, 0.0, w.scalar_elems).astype(np.float32)
    g = rng.uniform(0.0, 0.5, w.scalar_elems).astype(np.float32)
    g[3::29] = 60.0  # |G| > 40 inside some chunks
    return g


@pytest.mark.parametrize("decay_after", [False, True], ids=["decay-first", "decay-after"])
@pytest.mark.parametrize("khead_div", [False, True], ids=["mod", "div"])
@pytest.mark.parametrize("gates", ["plain", "negative", "extreme"])
def test_lazy_scan_is_the_recurrence(oracle_mod, decay_after, khead_div, gates):
    # 37 tokens: two full chunks and a ragged one; D_v != D_k
    w = Workload("scan-algebra", 16, 8, 2, 4, 37, 2)
    x = make_inputs(w, 91)
    x["g"] = _gates(w, gates, np.random.default_rng(92))
    p = w.params(path=PATH_SCAN, decay_after=decay_after, khead_div=khead_div)
    ro, rs, rc = oracle_mod.forward(p, **x, capture=True)
    stats = {}
    so, ss, sc = scan_forward(p, **x, stats=stats)
    assert _max_rel(so, ro) < 1e-10
    assert _max_rel(ss, rs) < 1e-10
    assert _max_rel(sc, rc) < 1e-10
    assert (stats["explicit"] > 0) == (gates == "extreme")
    assert stats["lazy"] > 0


@pytest.mark.parametrize("mutate", ["c_sk_swapped", "no_divide", "y_without_c", "no_fold"])
@pytest.mark.parametrize("decay_after", [False, True], ids=["decay-first", "decay-after"])
def test_a_planted_mistake_is_caught(oracle_mod, mutate, decay_after):
    # each slip in the lazy form (the other token's scale in delta, the update
    # not divided by c_t, y without c_t, no fold at the chunk's end) moves the
    # result far outside the bar
    w = Workload("scan-algebra", 16, 8, 2, 4, 37, 2)
    x = make_inputs(w, 93)
    p = w.params(path=PATH_SCAN, decay_after=decay_after)
    ro, rs, rc = oracle_mod.forward(p, **x, capture=True)
    so, ss, sc = scan_forward(p, **x, mutate=mutate)
    assert max(_max_rel(so, ro), _max_rel(ss, rs), _max_rel(sc, rc)) > 1e-4
