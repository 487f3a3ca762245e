"""Pins of the double-precision oracle to things other than itself.

Every test here runs on the CPU.  Each pin is chosen so that a plausible slip
in the oracle (a dropped term, a wrong sign or index, a transposed operand, a
swapped flag, a wrong stride) fails at least one of them:

* hand-derived worked cases (``tests/golden/hand_cases.json``);
* closed forms: beta = 0 reduces the recurrence to repeated scaling, checked
  with numpy GEMV; g = 0, beta = 1 and an exactly unit-norm key give S'k = v;
* an independent formulation: the matrix form of the gated delta rule,
  ``S' = alpha*S*(I - beta*k*k^T) + beta*v*k^T`` (decay-first) and
  ``S' = S*(alpha*I - beta*k*k^T) + beta*v*k^T`` (decay-after), written with
  numpy matrices over arrays reshaped from the pages' layout table;
* invariants: capture's last slice equals state_out, capture prefixes, chained
  calls equal one call, the map is linear in (state_in, v), the two k_head
  mappings and the two decay orders are not no-ops.
"""
import json
import math
import os

import numpy as np
import pytest

from serving_gdn_decode_gb300.params import pack_params
from serving_gdn_decode_gb300.workloads import WORKLOADS, Workload, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")
LN2_F32 = float(np.float32(math.log(2.0)))


def _load_cases():
    with open(GOLDEN) as f:
        data = json.load(f)
    return data["tolerance_abs"], data["cases"]


TOL, CASES = _load_cases()


def _arr(x):
    return np.array([LN2_F32 if e == "ln2" else e for e in x], dtype=np.float32)


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_hand_cases(oracle_mod, case):
    dk, dv, nk, nv, nt, ns = case["dims"]
    for flags in case["flags"]:
        params = np.array([dk, dv, nk, nv, nt, ns, flags, 0, case["q_scale_bits"]], dtype=np.uint32)
        want_cap = "state_capture" in case
        out, st, cap = oracle_mod.forward(params, _arr(case["q"]), _arr(case["k"]), _arr(case["v"]),
                                          _arr(case["g"]), _arr(case["beta"]),
                                          _arr(case["state_in"]), capture=want_cap, n_threads=1)
        np.testing.assert_allclose(out, np.array(case["output"], float), rtol=0, atol=TOL,
                                   err_msg=f"{case['name']} flags={flags} output")
        np.testing.assert_allclose(st, np.array(case["state_out"], float), rtol=0, atol=TOL,
                                   err_msg=f"{case['name']} flags={flags} state_out")
        if want_cap:
            np.testing.assert_allclose(cap, np.array(case["state_capture"], float), rtol=0,
                                       atol=TOL, err_msg=f"{case['name']} flags={flags} capture")


# ---------------------------------------------------------------- helpers

def _small(dk=8, dv=12, nk=2, nv=4, nt=5, ns=3, seed=1, zero_state=False):
    w = Workload("small", dk, dv, nk, nv, nt, ns, zero_state=zero_state)
    return w, make_inputs(w, seed)


def _views(w, x):
    """Reshape flat arrays per the 'Memory layouts' table (innermost first)."""
    q = x["q"].astype(np.float64).reshape(w.n_seqs, w.n_tokens, w.n_k_heads, w.d_k)
    k = x["k"].astype(np.float64).reshape(w.n_seqs, w.n_tokens, w.n_k_heads, w.d_k)
    v = x["v"].astype(np.float64).reshape(w.n_seqs, w.n_tokens, w.n_v_heads, w.d_v)
    g = x["g"].astype(np.float64).reshape(w.n_seqs, w.n_tokens, w.n_v_heads)
    b = x["beta"].astype(np.float64).reshape(w.n_seqs, w.n_tokens, w.n_v_heads)
    s0 = np.asarray(x["state_in"], dtype=np.float64).reshape(w.n_seqs, w.n_v_heads, w.d_v, w.d_k)
    return q, k, v, g, b, s0


def _khead(w, vh, div):
    return vh // (w.n_v_heads // w.n_k_heads) if div else vh % w.n_k_heads


def _matrix_form(w, x, decay_after, div, q_scale):
    q, k, v, g, b, s0 = _views(w, x)
    out = np.zeros((w.n_seqs, w.n_tokens, w.n_v_heads, w.d_v))
    st = np.zeros_like(s0)
    cap = np.zeros((w.n_seqs, w.n_tokens, w.n_v_heads, w.d_v, w.d_k))
    eye = np.eye(w.d_k)
    for s in range(w.n_seqs):
        for vh in range(w.n_v_heads):
            kh = _khead(w, vh, div)
            S = s0[s, vh].copy()
            for t in range(w.n_tokens):
                a = math.exp(-g[s, t, vh])
                beta = b[s, t, vh]
                kk = k[s, t, kh][:, None]
                if decay_after:
                    S = S @ (a * eye - beta * (kk @ kk.T)) + beta * (v[s, t, vh][:, None] @ kk.T)
                else:
                    S = a * S @ (eye - beta * (kk @ kk.T)) + beta * (v[s, t, vh][:, None] @ kk.T)
                out[s, t, vh] = q_scale * (S @ q[s, t, kh])
                cap[s, t, vh] = S
            st[s, vh] = S
    return out.reshape(-1), st.reshape(-1), cap.reshape(-1)


# ---------------------------------------------------------------- pins

@pytest.mark.parametrize("decay_after", [False, True])
@pytest.mark.parametrize("div", [False, True])
@pytest.mark.parametrize("dims", [(8, 12, 2, 4, 5, 3), (4, 4, 1, 2, 3, 1), (16, 8, 3, 6, 4, 2)])
def test_matrix_form_agrees(oracle_mod, decay_after, div, dims):
    w, x = _small(*dims)
    qs = 0.375
    p = pack_params(*dims, q_scale=qs, decay_after=decay_after, khead_div=div)
    out, st, cap = oracle_mod.forward(p, **x, capture=True, n_threads=3)
    mo, ms, mc = _matrix_form(w, x, decay_after, div, qs)
    for a, b, name in ((out, mo, "output"), (st, ms, "state"), (cap, mc, "capture")):
        err = np.max(np.abs(a - b)) / np.max(np.abs(b))
        assert err < 1e-12, (name, err)


@pytest.mark.parametrize("decay_after", [False, True])
def test_beta_zero_is_pure_decay(oracle_mod, decay_after):
    """beta = 0: S_T = (prod_t alpha_t) S0 and y_t = q_scale * (prod_{tau<=t} alpha_tau) S0 q_t."""
    w, x = _small(dk=8, dv=6, nk=2, nv=4, nt=6, ns=2, seed=3)
    x["beta"] = np.zeros_like(x["beta"])
    qs = 0.25
    p = pack_params(8, 6, 2, 4, 6, 2, q_scale=qs, decay_after=decay_after)
    out, st, _ = oracle_mod.forward(p, **x)
    q, _, _, g, _, s0 = _views(w, x)
    out = out.reshape(w.n_seqs, w.n_tokens, w.n_v_heads, w.d_v)
    st = st.reshape(s0.shape)
    for s in range(w.n_seqs):
        for vh in range(w.n_v_heads):
            kh = vh % w.n_k_heads
            c = 1.0
            for t in range(w.n_tokens):
                c *= math.exp(-g[s, t, vh])
                np.testing.assert_allclose(out[s, t, vh], qs * c * np.dot(s0[s, vh], q[s, t, kh]),
                                           rtol=1e-13, atol=1e-15)
            np.testing.assert_allclose(st[s, vh], c * s0[s, vh], rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("decay_after", [False, True])
def test_unit_key_gives_exact_recall(oracle_mod, decay_after):
    """g = 0, beta = 1 and ||k|| = 1 exactly: the updated state maps k to v."""
    rng = np.random.default_rng(7)
    dk, dv, nt = 16, 8, 5
    w = Workload("unit", dk, dv, 1, 1, nt, 1)
    x = make_inputs(w, 11)
    # 16 entries of +-1/4: squared norm is exactly 1 in binary floating point.
    x["k"] = (rng.choice([-0.25, 0.25], size=w.qk_elems)).astype(np.float32)
    x["g"] = np.zeros_like(x["g"])
    x["beta"] = np.ones_like(x["beta"])
    p = pack_params(dk, dv, 1, 1, nt, 1, decay_after=decay_after)
    _, _, cap = oracle_mod.forward(p, **x, capture=True)
    cap = cap.reshape(nt, dv, dk)
    k = x["k"].astype(np.float64).reshape(nt, dk)
    v = x["v"].astype(np.float64).reshape(nt, dv)
    for t in range(nt):
        np.testing.assert_allclose(cap[t] @ k[t], v[t], rtol=0, atol=1e-12)


def test_decay_orders_differ_by_closed_form(oracle_mod):
    """One token: decay-first minus decay-after = beta*(1-alpha)*(S0 k) k^T."""
    w, x = _small(dk=8, dv=5, nk=1, nv=1, nt=1, ns=1, seed=5)
    p0 = pack_params(8, 5, 1, 1, 1, 1)
    p1 = pack_params(8, 5, 1, 1, 1, 1, decay_after=True)
    _, s_first, _ = oracle_mod.forward(p0, **x)
    _, s_after, _ = oracle_mod.forward(p1, **x)
    _, k, _, g, b, s0 = _views(w, x)
    a = math.exp(-g[0, 0, 0])
    kk = k[0, 0, 0]
    want = b[0, 0, 0] * (1 - a) * np.outer(s0[0, 0] @ kk, kk)
    got = (s_first - s_after).reshape(5, 8)
    assert np.max(np.abs(want)) > 1e-3  # the pin must not be vacuous
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-14)


def test_khead_mapping_flag_is_not_a_noop(oracle_mod):
    _, x = _small(dk=8, dv=4, nk=2, nv=4, nt=2, ns=1, seed=9)
    o0, _, _ = oracle_mod.forward(pack_params(8, 4, 2, 4, 2, 1), **x)
    o1, _, _ = oracle_mod.forward(pack_params(8, 4, 2, 4, 2, 1, khead_div=True), **x)
    o0 = o0.reshape(2, 4, 4)
    o1 = o1.reshape(2, 4, 4)
    # v-heads 0 and 3 map to the same k-head under both readings, 1 and 2 swap.
    np.testing.assert_array_equal(o0[:, [0, 3]], o1[:, [0, 3]])
    assert np.max(np.abs(o0[:, [1, 2]] - o1[:, [1, 2]])) > 1e-3


def test_capture_last_slice_and_prefixes(oracle_mod):
    """state_capture[..., T-1, ...] == state_out, and slice t equals the
    state_out of the same problem cut to t+1 tokens (the determinism contract
    of dispatch_gated_delta_net_decode_with_capture)."""
    w, x = _small(dk=8, dv=6, nk=2, nv=4, nt=5, ns=2, seed=13)
    p = pack_params(8, 6, 2, 4, 5, 2, q_scale=0.5)
    out, st, cap = oracle_mod.forward(p, **x, capture=True)
    cap = cap.reshape(2, 5, -1)
    np.testing.assert_array_equal(cap[:, -1].reshape(-1), st)
    for t in range(5):
        xt = _cut_tokens(w, x, 0, t + 1)
        _, st_t, _ = oracle_mod.forward(pack_params(8, 6, 2, 4, t + 1, 2, q_scale=0.5), **xt)
        np.testing.assert_array_equal(cap[:, t].reshape(-1), st_t)


def _cut_tokens(w, x, t0, t1):
    """Tokens [t0, t1) of every per-token input, state_in unchanged."""
    def cut(a, inner):
        return np.ascontiguousarray(a.reshape(w.n_seqs, w.n_tokens, inner)[:, t0:t1]).reshape(-1)
    return {"q": cut(x["q"], w.n_k_heads * w.d_k), "k": cut(x["k"], w.n_k_heads * w.d_k),
            "v": cut(x["v"], w.n_v_heads * w.d_v), "g": cut(x["g"], w.n_v_heads),
            "beta": cut(x["beta"], w.n_v_heads), "state_in": x["state_in"]}


@pytest.mark.parametrize("flags", [(False, False), (True, True)])
def test_chained_calls_equal_one_call(oracle_mod, flags):
    w, x = _small(dk=8, dv=6, nk=2, nv=4, nt=7, ns=2, seed=17)
    da, dv_ = flags
    out, st, _ = oracle_mod.forward(pack_params(8, 6, 2, 4, 7, 2, 0.3, da, dv_), **x)
    a = _cut_tokens(w, x, 0, 3)
    o1, s1, _ = oracle_mod.forward(pack_params(8, 6, 2, 4, 3, 2, 0.3, da, dv_), **a)
    b = _cut_tokens(w, x, 3, 7)
    b["state_in"] = s1  # f64 state carried exactly
    o2, s2, _ = oracle_mod.forward(pack_params(8, 6, 2, 4, 4, 2, 0.3, da, dv_), **b)
    out = out.reshape(2, 7, -1)
    np.testing.assert_array_equal(out[:, :3].reshape(-1), o1)
    np.testing.assert_array_equal(out[:, 3:].reshape(-1), o2)
    np.testing.assert_array_equal(st, s2)


def test_linear_in_state_and_values(oracle_mod):
    """For fixed q, k, g, beta the map (S0, V) -> (Y, S_T, capture) is linear,
    and doubling is exact in binary floating point."""
    _, x = _small(dk=8, dv=6, nk=2, nv=4, nt=4, ns=2, seed=19)
    p = pack_params(8, 6, 2, 4, 4, 2, q_scale=0.7)
    o, s, c = oracle_mod.forward(p, **x, capture=True)
    x2 = dict(x, v=x["v"] * np.float32(2), state_in=x["state_in"] * np.float32(2))
    o2, s2, c2 = oracle_mod.forward(p, **x2, capture=True)
    np.testing.assert_array_equal(o2, 2 * o)
    np.testing.assert_array_equal(s2, 2 * s)
    np.testing.assert_array_equal(c2, 2 * c)


def test_q_scale_bits(oracle_mod):
    """q_scale_bits == 0 means 1.0 (capture kernel page, 'Buffer bindings');
    non-zero bits are the f32 scale applied at writeback."""
    _, x = _small(dk=8, dv=6, nk=1, nv=2, nt=3, ns=1, seed=23)
    base = pack_params(8, 6, 1, 2, 3, 1)
    assert base[8] == 0
    o0, s0, _ = oracle_mod.forward(base, **x)
    o1, s1, _ = oracle_mod.forward(pack_params(8, 6, 1, 2, 3, 1, q_scale=1.0), **x)
    oh, sh, _ = oracle_mod.forward(pack_params(8, 6, 1, 2, 3, 1, q_scale=0.5), **x)
    np.testing.assert_array_equal(o0, o1)
    np.testing.assert_array_equal(oh, 0.5 * o0)
    np.testing.assert_array_equal(s0, sh)  # the scale never touches the state


def test_heads_subset_matches_full(oracle_mod):
    w, x = _small(dk=8, dv=6, nk=2, nv=4, nt=3, ns=3, seed=29)
    p = pack_params(8, 6, 2, 4, 3, 3, q_scale=0.5, khead_div=True)
    out, st, cap = oracle_mod.forward(p, **x, capture=True)
    heads = [11, 0, 5]
    ho, hs, hc = oracle_mod.forward_heads(p, **x, heads=heads, capture=True)
    out = out.reshape(3, 3, 4, 6)
    st = st.reshape(3, 4, 6, 8)
    cap = cap.reshape(3, 3, 4, 6, 8)
    for n, h in enumerate(heads):
        s, vh = divmod(h, 4)
        np.testing.assert_array_equal(ho[n], out[s, :, vh])
        np.testing.assert_array_equal(hs[n], st[s, vh])
        np.testing.assert_array_equal(hc[n], cap[s, :, vh])


@pytest.mark.parametrize("bad", [
    dict(n_params=8), dict(slot=0, value=0), dict(slot=1, value=0), dict(slot=2, value=0),
    dict(slot=3, value=0), dict(slot=4, value=0), dict(slot=5, value=0),
    dict(slot=3, value=3),          # n_v % n_k != 0 (n_k = 2)
    dict(slot=7, value=1),          # reserved slot
    dict(slot=6, value=0x10),       # unknown flag bit
    dict(slot=6, value=0x80000000),  # unknown flag bit
])
def test_oracle_rejects_what_the_pages_reject(oracle_mod, bad):
    _, x = _small(dk=8, dv=6, nk=2, nv=4, nt=2, ns=1)
    p = pack_params(8, 6, 2, 4, 2, 1)
    if "n_params" in bad:
        p = p[: bad["n_params"]]
    else:
        p[bad["slot"]] = bad["value"]
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.forward(p, **x)


@pytest.mark.parametrize("path", [0, 1, 2, 3])
def test_oracle_ignores_the_path_bits(oracle_mod, path):
    # params[6] bits 2-3 choose a GPU kernel; the recurrence is the same
    _, x = _small(dk=8, dv=6, nk=2, nv=4, nt=3, ns=2)
    ref = oracle_mod.forward(pack_params(8, 6, 2, 4, 3, 2), **x)
    got = oracle_mod.forward(pack_params(8, 6, 2, 4, 3, 2, path=path), **x)
    for a, b in zip(got[:2], ref[:2]):
        np.testing.assert_array_equal(a, b)


def test_tiny_workload_runs_and_is_finite(oracle_mod):
    w = WORKLOADS["tiny"]
    x = make_inputs(w, 0)
    out, st, cap = oracle_mod.forward(w.params(), **x, capture=True)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(st))
    np.testing.assert_array_equal(cap.reshape(w.n_tokens, -1)[-1], st)
