"""The chunk equations that the two-pass chunked prefill evaluates, written
out in float64 numpy, against the oracle's token-by-token recurrence.

The GPU parity tests show that the kernels reach the oracle's results within
the TF32 bar; this test shows, exactly up to float64 rounding and without a
GPU, that the equations the kernels implement are the recurrence.  Per
(seq, value head) and 64-token chunk, with G the prefix sums of g over the
chunk, gamma = e^-G, the state kept as S = c * St:

  chunk pass:  A[r, i] = beta_r e^-(G_r' - G_i) k_r.k_i   (i < r; G_r' = G_r,
                                                           or G_{r-1} with
                                                           decay-after)
               T = (I + A)^-1,  T'' = T diag(beta)
               P'[r, i] = q_scale e^-(G_r - G_i) q_r.k_i  (i <= r)
  state pass:  X = St K^T,  Z = St Q^T
               W = V^T - X diag(c gamma)                  (gamma' = e^-G' with
                                                           decay-after)
               U = W T''^T
               Y = Z diag(c q_scale gamma) + U P'^T      (the chunk's outputs)
               St += U diag(e^(G_i - G_C) / c') K,  c' = c e^-G_C

with c folded into St when it leaves [2^-30, 2^30], and, for a chunk whose
|G| exceeds 40 somewhere, St decayed by c e^-G_C before the update and c' = 1.

The one-pass kernel groups the same products differently (form "one_pass"):

  U^T  = V^T T''^T + X (-T')^T,   T' = c T diag(beta gamma)   (gamma' with
                                                               decay-after)
  Y^T  = St Q'^T + U^T P'^T,      Q' = c q_scale diag(gamma) Q
  St  += U^T K'^T,                K' = diag(e^(G_i - G_C) / c') K
"""
import numpy as np
import pytest

from serving_gdn_decode_gb300.params import PATH_CHUNKED
from serving_gdn_decode_gb300.workloads import Workload, make_inputs

C = 64
MAX_LOG = 40.0
LO, HI = 2.0 ** -30, 2.0 ** 30


def _q_scale(params):
    bits = int(params[8])
    return 1.0 if bits == 0 else float(np.array([bits], dtype=np.uint32).view(np.float32)[0])


def chunk_forward(params, q, k, v, g, beta, state_in, stats=None, mutate=None, form="two_pass"):
    """The chunk equations above for a whole problem; flat arrays in and out
    in the library's innermost-first layouts.  `stats` (a dict) counts the
    renorm and extreme-chunk branches taken; `mutate` plants one mistake, to
    show that the comparison catches it."""
    if stats is not None:
        stats.update(renorm=0, extreme=0)
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
    st_out = np.zeros_like(state)
    for s in range(ns):
        for vh in range(nv):
            kh = vh // (nv // nk) if khead_div else vh % nk
            St, c = state[s, vh].copy(), 1.0
            for t0 in range(0, nt, C):
                sl = slice(t0, min(nt, t0 + C))
                K, Q, V = k[s, sl, kh], q[s, sl, kh], v[s, sl, vh]
                gc, b = g[s, sl, vh], beta[s, sl, vh]
                n = len(gc)
                G = np.cumsum(gc)
                Gp = G - gc
                GC = G[-1]
                gam, gamp = np.exp(-G), np.exp(-Gp)
                extreme = bool(np.any(np.abs(G) > MAX_LOG))
                # the lazy scale entering the chunk (folded into St if out of range)
                if c < LO or c > HI:
                    St *= c
                    c = 1.0
                    if stats is not None:
                        stats["renorm"] += 1
                if extreme:
                    fold, c_next = c * np.exp(-GC), 1.0
                    if stats is not None:
                        stats["extreme"] += 1
                else:
                    fold, c_next = 1.0, c * np.exp(-GC)
                # chunk pass
                Ga = Gp if decay_after else G
                r_idx, i_idx = np.arange(n)[:, None], np.arange(n)[None, :]
                lower = i_idx < r_idx if mutate != "diag_in_A" else i_idx <= r_idx
                A = np.where(lower, b[:, None] * np.exp(G[None, :] - Ga[:, None]) * (K @ K.T), 0.0)
                T = np.linalg.inv(np.eye(n) + A)
                Tpp = T * (b[None, :] if mutate != "beta_rows" else b[:, None])
                P = np.where(i_idx <= r_idx, qs * np.exp(G[None, :] - G[:, None]) * (Q @ K.T), 0.0)
                kts = np.exp(G - GC) if mutate != "kts_sign" else np.exp(GC - G)
                if form == "two_pass":
                    X, Z = St @ K.T, St @ Q.T
                    W = V.T - X * (c * (gamp if decay_after else gam))[None, :]
                    U = W @ Tpp.T
                    Y = U @ P.T
                    if mutate != "no_Z":
                        Y = Y + Z * (c * qs * gam)[None, :]
                    St = St * fold + (U * (kts / c_next)[None, :]) @ K
                else:
                    X = St @ K.T
                    Tp = c * T * (b * (gamp if decay_after else gam))[None, :]
                    U = V.T @ Tpp.T + X @ (-Tp).T
                    Qp = (c * qs * gam)[:, None] * Q
                    Y = U @ P.T
                    if mutate != "no_Z":
                        Y = Y + St @ Qp.T
                    Kp = (kts / c_next)[:, None] * K
                    St = St * fold + U @ Kp
                out[s, sl, vh] = Y.T
                c = c_next
            st_out[s, vh] = c * St
    return out.reshape(-1), st_out.reshape(-1)


def _max_rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


@pytest.mark.parametrize("decay_after", [False, True], ids=["decay-first", "decay-after"])
@pytest.mark.parametrize("khead_div", [False, True], ids=["mod", "div"])
@pytest.mark.parametrize("gates", ["plain", "long", "extreme"])
@pytest.mark.parametrize("form", ["two_pass", "one_pass"])
def test_chunk_equations_are_the_recurrence(oracle_mod, decay_after, khead_div, gates, form):
    # 150 tokens: two full chunks and a ragged one; D = 16 keeps the oracle quick
    # (the equations do not depend on D)
    w = Workload("algebra", 16, 16, 2, 4, 150, 2)
    x = make_inputs(w, 81)
    rng = np.random.default_rng(82)
    if gates == "plain":
        # gentle decay: neither branch taken
        x["g"] = rng.uniform(0.0, 0.05, w.scalar_elems).astype(np.float32)
    elif gates == "long":
        # decay sums past 2^-30 within the window: the lazy scale is folded back
        x["g"] = rng.uniform(0.2, 0.6, w.scalar_elems).astype(np.float32)
    elif gates == "extreme":
        g = rng.uniform(0.0, 0.5, w.scalar_elems).astype(np.float32)
        g[5::37] = 60.0  # |G| > 40 inside a chunk
        x["g"] = g
    p = w.params(path=PATH_CHUNKED, decay_after=decay_after, khead_div=khead_div)
    ro, rs, _ = oracle_mod.forward(p, **x)
    stats = {}
    co, cs = chunk_forward(p, **x, stats=stats, form=form)
    assert _max_rel(co, ro) < 1e-10
    assert _max_rel(cs, rs) < 1e-10
    assert (stats["renorm"] > 0) == (gates == "long")
    assert (stats["extreme"] > 0) == (gates == "extreme")


@pytest.mark.parametrize("mutate", ["diag_in_A", "beta_rows", "no_Z", "kts_sign", "flags"])
@pytest.mark.parametrize("form", ["two_pass", "one_pass"])
def test_a_planted_mistake_is_caught(oracle_mod, mutate, form):
    # each plausible slip in the equations (the diagonal inside A, beta scaling
    # rows instead of columns, the inter-chunk output term dropped, the key
    # decay of the state update inverted, decay-first read as decay-after)
    # moves the result far outside the bar
    w = Workload("algebra", 16, 16, 2, 4, 150, 2)
    x = make_inputs(w, 83)
    p = w.params(path=PATH_CHUNKED)
    ro, rs, _ = oracle_mod.forward(p, **x)
    if mutate == "flags":
        co, cs = chunk_forward(w.params(path=PATH_CHUNKED, decay_after=True), **x, form=form)
    else:
        co, cs = chunk_forward(p, **x, mutate=mutate, form=form)
    assert max(_max_rel(co, ro), _max_rel(cs, rs)) > 1e-4
