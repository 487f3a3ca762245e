"""GPU invariants, edge cases and ragged shapes, through the C ABI.

* bitwise properties that need no oracle: capture's last slice equals
  state_out; chained calls equal one call on the decode path (the scan path
  folds its lazy decay at chunk boundaries counted from the call's first
  token, so there chaining holds within tolerance); doubling (state_in, v)
  doubles every result; in-place equals out-of-place;
* no write outside the caller's buffers (guard bands), and the unused tail of
  an oversized capture buffer (allowed when n_seqs == 1) stays untouched;
* ragged shapes (several CTAs with a partial last one, token chunks with a
  partial last chunk), every supported D_k, D_v != D_k, against the oracle.
"""
import numpy as np
import pytest

from gpu_helpers import assert_close, run_gpu, to_dev
from serving_gdn_decode_gb300.params import PATH_CHUNKED, PATH_SCAN, pack_params
from serving_gdn_decode_gb300.workloads import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as t
    assert t.cuda.is_available(), "GPU tests need a CUDA device"
    from serving_gdn_decode_gb300 import build
    build.build()
    return t


def _cut(w, x, t0, t1):
    def cut(a, inner):
        return np.ascontiguousarray(a.reshape(w.n_seqs, w.n_tokens, inner)[:, t0:t1]).reshape(-1)
    return {"q": cut(x["q"], w.n_k_heads * w.d_k), "k": cut(x["k"], w.n_k_heads * w.d_k),
            "v": cut(x["v"], w.n_v_heads * w.d_v), "g": cut(x["g"], w.n_v_heads),
            "beta": cut(x["beta"], w.n_v_heads), "state_in": x["state_in"]}


@pytest.mark.parametrize("path,nt,split", [(0, 12, 5), (0, 16, 1), (PATH_SCAN, 40, 17),
                                           (PATH_SCAN, 9, 1)])
def test_chained_equals_one_call(torch, path, nt, split):
    w = Workload("chain", 128, 64, 2, 4, nt, 3)
    x = make_inputs(w, 5)
    out, st, _ = run_gpu(w, x, w.params(path=path))
    wa, wb = w.with_(n_tokens=split), w.with_(n_tokens=nt - split)
    xa = _cut(w, x, 0, split)
    oa, sa, _ = run_gpu(wa, xa, wa.params(path=path))
    xb = _cut(w, x, split, nt)
    xb["state_in"] = sa
    ob, sb, _ = run_gpu(wb, xb, wb.params(path=path))
    o = out.reshape(w.n_seqs, nt, -1)
    if path == PATH_SCAN:
        assert_close("output", oa, o[:, :split].reshape(-1).astype(np.float64), split)
        assert_close("output", ob, o[:, split:].reshape(-1).astype(np.float64), nt - split)
        assert_close("state_out", sb, st.astype(np.float64), nt)
        return
    np.testing.assert_array_equal(o[:, :split].reshape(-1), oa)
    np.testing.assert_array_equal(o[:, split:].reshape(-1), ob)
    np.testing.assert_array_equal(st, sb)


@pytest.mark.parametrize("name", ["tiny", "spec_capture"])
def test_capture_last_slice_is_state_out(torch, name):
    w = WORKLOADS[name]
    x = make_inputs(w, 7)
    _, st, cap = run_gpu(w, x, w.params(), capture=True)
    np.testing.assert_array_equal(cap.reshape(w.n_seqs, w.n_tokens, -1)[:, -1].reshape(-1), st)


def test_doubling_is_exact(torch):
    w = Workload("lin", 128, 128, 4, 8, 6, 2)
    x = make_inputs(w, 9)
    p = w.params()
    o, s, c = run_gpu(w, x, p, capture=True)
    x2 = dict(x, v=x["v"] * np.float32(2), state_in=x["state_in"] * np.float32(2))
    o2, s2, c2 = run_gpu(w, x2, p, capture=True)
    np.testing.assert_array_equal(o2, 2 * o)
    np.testing.assert_array_equal(s2, 2 * s)
    np.testing.assert_array_equal(c2, 2 * c)


@pytest.mark.parametrize("capture", [False, True])
def test_in_place_equals_out_of_place(torch, capture):
    w = Workload("inplace", 128, 96, 2, 6, 3, 4)
    x = make_inputs(w, 11)
    a = run_gpu(w, x, w.params(), capture=capture)
    b = run_gpu(w, x, w.params(), capture=capture, in_place=True)
    for u, v in zip(a, b):
        if u is not None:
            np.testing.assert_array_equal(u, v)


@pytest.mark.parametrize("path,capture,workspace", [
    (PATH_SCAN, False, False), (PATH_SCAN, True, False),
    (PATH_CHUNKED, False, False), (PATH_CHUNKED, False, True)],
    ids=["scan", "scan-capture", "chunked-one-pass", "chunked-two-pass"])
def test_in_place_equals_out_of_place_long(torch, path, capture, workspace):
    """state_in == state_out on the prefill kernels: 100 tokens (one full
    64-token chunk and a partial one; six full 16-token scan chunks and a
    partial one), bit for bit equal to the out-of-place call.  Each of these
    kernels reads and writes the state through its own code."""
    w = Workload("inplace_long", 128, 128, 2, 4, 100, 2)
    x = make_inputs(w, 12)
    p = w.params(path=path)
    a = run_gpu(w, x, p, capture=capture, workspace=workspace)
    b = run_gpu(w, x, p, capture=capture, workspace=workspace, in_place=True)
    for u, v in zip(a, b):
        if u is not None:
            np.testing.assert_array_equal(u, v)


def test_device_status_clean_after_normal_runs(torch):
    """The device status word stays 0 through normal calls on every chunked
    form (no bounded wait runs out), and reading it with reset leaves 0."""
    from serving_gdn_decode_gb300 import _native as nat
    w = Workload("status", 128, 128, 2, 4, 130, 2)
    x = make_inputs(w, 14)
    nat.gdn_device_status(reset=True)
    for ws in (False, True):
        run_gpu(w, x, w.params(path=PATH_CHUNKED), workspace=ws)
    assert nat.gdn_device_status() == 0
    assert nat.gdn_device_status(reset=True) == 0
    assert nat.gdn_device_status(stream=torch.cuda.current_stream()) == 0


def test_guard_bands_untouched(torch):
    """Every output lives inside a larger buffer filled with a sentinel; only
    the exact output ranges may change."""
    from serving_gdn_decode_gb300 import _native as nat
    w = Workload("guard", 64, 50, 2, 4, 3, 2)
    x = make_inputs(w, 13)
    d = to_dev(x)
    pad = 64  # floats (256 bytes) on each side keeps 16-byte alignment
    sentinel = 12345.0

    def padded(n):
        return torch.full((n + 2 * pad,), sentinel, dtype=torch.float32, device="cuda")

    bo, bs, bc = padded(w.v_elems), padded(w.state_elems), padded(w.capture_elems)
    out, st, cap = (b[pad:pad + n] for b, n in ((bo, w.v_elems), (bs, w.state_elems),
                                                  (bc, w.capture_elems)))
    nat.gdn_forward_capture(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state_in"], out, st,
                            w.params(), cap)
    torch.cuda.synchronize()
    for b, n in ((bo, w.v_elems), (bs, w.state_elems), (bc, w.capture_elems)):
        h = b.cpu().numpy()
        assert np.all(h[:pad] == sentinel) and np.all(h[pad + n:] == sentinel)
        assert not np.any(h[pad:pad + n] == sentinel)


def test_oversized_capture_tail_untouched_single_seq(torch, oracle_mod):
    """n_seqs == 1 may pass a larger capture buffer (sized for the deepest
    speculation); elements past n_tokens * state elements stay untouched."""
    from serving_gdn_decode_gb300 import _native as nat
    w = Workload("spec1", 128, 128, 4, 8, 3, 1)
    x = make_inputs(w, 17)
    d = to_dev(x)
    extra = 5 * w.state_elems
    cap = torch.full((w.capture_elems + extra,), -7.0, dtype=torch.float32, device="cuda")
    out = torch.empty(w.v_elems, dtype=torch.float32, device="cuda")
    st = torch.empty(w.state_elems, dtype=torch.float32, device="cuda")
    nat.gdn_forward_capture(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state_in"], out, st,
                            w.params(), cap)
    torch.cuda.synchronize()
    h = cap.cpu().numpy()
    assert np.all(h[w.capture_elems:] == -7.0)
    _, _, rc = oracle_mod.forward(w.params(), **x, capture=True)
    assert_close("state_capture", h[:w.capture_elems], rc, w.n_tokens)


RAGGED = [
    # (d_k, d_v, n_k, n_v, n_tokens, n_seqs, path)
    (128, 100, 2, 6, 3, 2, 0),      # 4 row blocks, last one partial
    (128, 4, 1, 1, 1, 1, 0),        # smallest D_v for D_k = 128
    (128, 36, 3, 3, 8, 2, 0),       # n_v == n_k
    (64, 130, 1, 3, 5, 2, 0),       # D_k = 64, D_v > D_k
    (64, 2, 2, 2, 2, 1, 0),
    (32, 33, 3, 3, 2, 3, 0),        # D_k = 32, odd D_v
    (32, 1, 1, 1, 9, 1, 0),         # one row
    (32, 32, 1, 3, 4, 1, 0),        # D_k = 32, three value heads, four tokens
    (32, 32, 1, 2, 8, 1, PATH_SCAN),
    (128, 128, 16, 32, 37, 2, PATH_SCAN),   # 3 token chunks, partial last one
    (64, 70, 2, 4, 100, 1, PATH_SCAN),
    (128, 64, 1, 2, 17, 2, 0),      # auto path just past the decode window
    (128, 128, 2, 4, 100, 2, 0),    # auto: chunked, or the token loop with capture
    (64, 64, 2, 4, 60, 1, 0),       # auto: the scan, or the token loop with capture
]


@pytest.mark.parametrize("shape", RAGGED, ids=[str(s) for s in RAGGED])
@pytest.mark.parametrize("flags", [dict(), dict(decay_after=True, khead_div=True)],
                         ids=["default", "after-div"])
@pytest.mark.parametrize("capture", [False, True], ids=["plain", "capture"])
def test_ragged_shapes_vs_oracle(torch, oracle_mod, shape, flags, capture):
    dk, dv, nk, nv, nt, ns, path = shape
    w = Workload("ragged", dk, dv, nk, nv, nt, ns)
    x = make_inputs(w, 19)
    p = w.params(path=path, **flags)
    out, st, cap = run_gpu(w, x, p, capture=capture)
    ro, rs, rc = oracle_mod.forward(p, **x, capture=capture)
    assert_close("output", out, ro, nt)
    assert_close("state_out", st, rs, nt)
    if capture:
        assert_close("state_capture", cap, rc, nt)


@pytest.mark.parametrize("gate", ["large", "negative", "mixed"])
@pytest.mark.parametrize("decay_after", [False, True])
@pytest.mark.parametrize("capture", [False, True], ids=["plain", "capture"])
def test_scan_extreme_gates_vs_oracle(torch, oracle_mod, gate, decay_after, capture):
    """Gates far outside U[0, 0.5): the scan kernel's lazy decay must fall back
    to explicit decay in chunks where the running log-scale leaves [-40, 40]."""
    w = Workload("gates", 128, 64, 2, 4, 70, 2)
    x = make_inputs(w, 41)
    rng = np.random.default_rng(43)
    if gate == "large":
        x["g"] = rng.uniform(0.0, 8.0, w.scalar_elems).astype(np.float32)
    elif gate == "negative":
        x["g"] = rng.uniform(-0.12, 0.0, w.scalar_elems).astype(np.float32)
    else:  # some chunks lazy, some explicit, some tokens with alpha underflowing to 0
        g = rng.uniform(0.0, 0.5, w.scalar_elems).astype(np.float32)
        g[::7] = 60.0
        g[5::23] = 200.0
        x["g"] = g
    p = w.params(path=PATH_SCAN, decay_after=decay_after)
    out, st, cap = run_gpu(w, x, p, capture=capture)
    ro, rs, rc = oracle_mod.forward(p, **x, capture=capture)
    assert_close("output", out, ro, w.n_tokens)
    assert_close("state_out", st, rs, w.n_tokens)
    if capture:
        assert_close("state_capture", cap, rc, w.n_tokens)


def test_decode_and_scan_shapes_agree(torch):
    w = Workload("paths", 128, 128, 4, 8, 6, 3)
    x = make_inputs(w, 23)
    a = run_gpu(w, x, w.params(path=0), capture=True)
    b = run_gpu(w, x, w.params(path=PATH_SCAN), capture=True)
    for u, v in zip(a, b):
        assert_close("paths", u, v.astype(np.float64), w.n_tokens)


def test_unit_key_recall_on_gpu(torch):
    """g = 0, beta = 1 and ||k|| = 1 exactly (D_k = 64 entries of +-1/8):
    the updated state maps k to v, up to f32 rounding."""
    rng = np.random.default_rng(29)
    w = Workload("recall", 64, 48, 2, 4, 4, 2)
    x = make_inputs(w, 29)
    x["k"] = rng.choice([-0.125, 0.125], size=w.qk_elems).astype(np.float32)
    x["g"] = np.zeros_like(x["g"])
    x["beta"] = np.ones_like(x["beta"])
    _, _, cap = run_gpu(w, x, w.params(), capture=True)
    cap = cap.reshape(w.n_seqs, w.n_tokens, w.n_v_heads, w.d_v, w.d_k).astype(np.float64)
    k = x["k"].reshape(w.n_seqs, w.n_tokens, w.n_k_heads, w.d_k).astype(np.float64)
    v = x["v"].reshape(w.n_seqs, w.n_tokens, w.n_v_heads, w.d_v).astype(np.float64)
    for s in range(w.n_seqs):
        for t in range(w.n_tokens):
            for vh in range(w.n_v_heads):
                got = cap[s, t, vh] @ k[s, t, vh % w.n_k_heads]
                np.testing.assert_allclose(got, v[s, t, vh], rtol=0, atol=2e-5)


def test_beta_zero_pure_decay_on_gpu(torch):
    w = Workload("decay", 128, 64, 2, 4, 5, 2)
    x = make_inputs(w, 31)
    x["beta"] = np.zeros_like(x["beta"])
    _, st, _ = run_gpu(w, x, w.params())
    g = x["g"].reshape(w.n_seqs, w.n_tokens, w.n_v_heads).astype(np.float64)
    c = np.exp(-g.sum(axis=1))  # [S, n_v]
    s0 = x["state_in"].reshape(w.n_seqs, w.n_v_heads, -1).astype(np.float64)
    want = (c[:, :, None] * s0).reshape(-1)
    np.testing.assert_allclose(st, want, rtol=1e-5, atol=1e-7)


def test_non_default_stream(torch):
    w = Workload("stream", 128, 128, 2, 4, 2, 2)
    x = make_inputs(w, 37)
    a = run_gpu(w, x, w.params())
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        d = to_dev(x)
        b = run_gpu(w, x, w.params(), stream=s, dev=d)
    for u, v in zip(a, b):
        if u is not None:
            np.testing.assert_array_equal(u, v)
