"""GPU tests of the bf16-activation entry points (gdn_forward_bf16,
gdn_forward_capture_bf16, gdn_forward_layers_bf16): q, k, v and output in
bfloat16, g, beta, state and capture in f32 ("Dtype / precision" of
gated_delta_net.rs, mlx-native 0.4.0: f32 accumulation, bf16 I/O as the
later variant).

q, k and v are drawn on the bf16 grid (``make_inputs(act="bf16")``), so the
bf16 path, the f32 path and the oracle all read the same values.  Two bars:

* against the oracle: state_out and state_capture within the f32 bar of
  gpu_helpers; output within half a bf16 ulp of the oracle on top of that
  bar.  Half an ulp of a bf16 value y is at most 2^-8 |y|, so for
  n_tokens <= 8 every element obeys
  |y - y_ref| <= 2^-8 (|y_ref| + E) + E with E = 1e-4 max|y_ref|, and for
  longer windows rel-L2(y, y_ref) <= 1e-3 + 2^-8;
* against the f32 path on the same values: state_out and state_capture bit
  for bit, and output equal, bit for bit, to the f32 path's output rounded to
  nearest-even bf16 -- the header's contract that only the final store of y
  differs.  This holds on the chunked path too: there the bf16 kernel leaves
  out the products whose lo half is zero (bf16 inputs are their own hi
  halves), which add nothing in the f32 kernel.
"""
import numpy as np
import pytest

from gpu_helpers import (MAXABS_TOL, RELL2_TOL, SPLIT_RELL2_TOL, assert_close, assert_rel_l2, gather_heads,
                         run_gpu, sample_heads)
from serving_gdn_decode_gb300.params import PATH_CHUNKED, PATH_CHUNKED_TF32, PATH_SCAN
from serving_gdn_decode_gb300.workloads import Workload, make_inputs, round_to_bf16

pytestmark = pytest.mark.gpu

HALF_ULP = 2.0 ** -8


@pytest.fixture(scope="module")
def torch():
    import torch as t
    assert t.cuda.is_available(), "GPU tests need a CUDA device"
    from serving_gdn_decode_gb300 import build
    build.build()
    return t


def _dev_bf16(torch, x):
    """Device tensors: q, k, v as bf16 (exact: the values are on the bf16
    grid), the rest f32."""
    d = {}
    for n, a in x.items():
        t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
        if n in ("q", "k", "v"):
            b = t.to(torch.bfloat16)
            assert torch.equal(b.float(), t), f"{n} is not on the bf16 grid"
            t = b
        d[n] = t
    return d


def run_bf16(torch, w, x, params, capture=False, in_place=False, workspace=False):
    """Run the bf16 path (gdn_forward_ws_bf16 with a workspace of
    gdn_workspace_size's bytes when ``workspace``).  Returns numpy (output as
    f32 values, state_out, capture|None)."""
    from serving_gdn_decode_gb300 import _native as nat
    d = _dev_bf16(torch, x)
    out = torch.empty(w.v_elems, dtype=torch.bfloat16, device="cuda")
    st_in = d["state_in"]
    st = st_in.clone() if in_place else torch.empty(w.state_elems, dtype=torch.float32, device="cuda")
    if in_place:
        st_in = st
    if capture:
        cap = torch.empty(w.capture_elems, dtype=torch.float32, device="cuda")
        nat.gdn_forward_capture(d["q"], d["k"], d["v"], d["g"], d["beta"], st_in, out, st, params,
                                cap)
    elif workspace:
        cap = None
        ws = torch.empty(max(16, nat.gdn_workspace_size(params)), dtype=torch.uint8, device="cuda")
        nat.gdn_forward_ws(d["q"], d["k"], d["v"], d["g"], d["beta"], st_in, out, st, params, ws)
    else:
        cap = None
        nat.gdn_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], st_in, out, st, params)
    torch.cuda.synchronize()
    return (out.float().cpu().numpy(), st.cpu().numpy(),
            None if cap is None else cap.cpu().numpy())


def assert_output_bf16(y, y_ref, n_tokens):
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    assert np.all(np.isfinite(y)), "output: non-finite values"
    assert np.array_equal(round_to_bf16(y.astype(np.float32)), y.astype(np.float32)), \
        "output: values off the bf16 grid"
    if n_tokens > 8:
        d = y - y_ref
        e = float(np.sqrt(np.sum(d * d)) / max(np.sqrt(np.sum(y_ref * y_ref)), 1e-300))
        assert e <= RELL2_TOL + HALF_ULP, f"output: rel-L2 {e:.3e} > {RELL2_TOL + HALF_ULP:.3e}"
        return
    E = MAXABS_TOL * float(np.max(np.abs(y_ref)))
    bound = HALF_ULP * (np.abs(y_ref) + E) + E
    worst = float(np.max(np.abs(y - y_ref) - bound))
    assert worst <= 0.0, f"output: {int(np.sum(np.abs(y - y_ref) > bound))} elements past " \
                         f"half a bf16 ulp + {MAXABS_TOL:g} (worst excess {worst:.3e})"


CASES = [  # (d_k, d_v, n_k, n_v, n_tokens, n_seqs, capture, path)
    (32, 32, 1, 2, 8, 1, True, 0),          # the tiny workload's shape
    (128, 128, 4, 8, 1, 3, False, 0),       # decode
    (128, 128, 2, 4, 4, 2, True, 0),        # speculative verify window with capture
    (64, 96, 2, 6, 3, 2, False, 0),         # D_v != D_k, two cells per lane
    (32, 34, 1, 3, 2, 1, True, 0),          # even D_v far below the CTA's 128 rows
    (128, 136, 2, 2, 3, 2, False, 0),       # ragged last row block (136 = 4*32 + 8)
    (128, 128, 2, 4, 40, 2, True, 0),       # auto scan: 2 full 16-token chunks + 8
    (64, 64, 1, 2, 5, 1, True, PATH_SCAN),  # forced scan, one partial chunk
    (128, 128, 2, 4, 130, 2, False, 0),     # auto chunked: 2 full 64-token chunks + 2
    (128, 128, 2, 6, 9, 2, False, PATH_CHUNKED),   # forced chunked, one partial chunk
    (128, 128, 1, 2, 64, 1, False, PATH_CHUNKED),  # exactly one chunk
]
FLAGS = [dict(), dict(decay_after=True), dict(khead_div=True),
         dict(decay_after=True, khead_div=True)]


@pytest.mark.parametrize("flags", FLAGS, ids=["df-mod", "da-mod", "df-div", "da-div"])
@pytest.mark.parametrize("case", CASES, ids=[str(c) for c in CASES])
def test_bf16_parity_and_f32_identity(torch, oracle_mod, case, flags):
    dk, dv, nk, nv, nt, ns, capture, path = case
    w = Workload("bf16", dk, dv, nk, nv, nt, ns)
    p = w.params(path=path, q_scale=0.5 if flags.get("khead_div") else "default", **flags)
    x = make_inputs(w, 7, act="bf16")
    out, st, cap = run_bf16(torch, w, x, p, capture=capture)

    ro, rs, rc = oracle_mod.forward(p, **x, capture=capture)
    assert_output_bf16(out, ro, nt)
    assert_close("state_out", st, rs, nt)
    if capture:
        assert_close("state_capture", cap, rc, nt)

    fo, fs, fc = run_gpu(w, x, p, capture=capture)
    assert np.array_equal(st.view(np.uint32), fs.view(np.uint32)), "state_out differs from f32 path"
    if capture:
        assert np.array_equal(cap.view(np.uint32), fc.view(np.uint32)), \
            "state_capture differs from f32 path"
    assert np.array_equal(out.view(np.uint32), round_to_bf16(fo).view(np.uint32)), \
        "output is not the f32 path's output rounded to bf16"


TWO_PASS = [  # (n_k, n_v, n_tokens, n_seqs, path)
    (2, 4, 130, 2, 0),             # automatic: the chunked form, 2 full chunks + 2
    (2, 6, 9, 2, PATH_CHUNKED),    # one partial chunk
    (1, 8, 64, 1, PATH_CHUNKED),   # exactly one chunk, eight value heads on one key head
    (4, 4, 70, 1, PATH_CHUNKED),   # one value head per key head
]


@pytest.mark.parametrize("flags", [dict(), dict(decay_after=True, khead_div=True)], ids=["df-mod", "da-div"])
@pytest.mark.parametrize("case", TWO_PASS, ids=[str(c) for c in TWO_PASS])
def test_bf16_two_pass_parity_and_f32_identity(torch, oracle_mod, case, flags):
    """gdn_forward_ws_bf16: the two-pass chunked form with bf16 activations,
    against the oracle and, bit for bit, against gdn_forward_ws on the same
    widened values (output: that output rounded to bf16)."""
    nk, nv, nt, ns, path = case
    w = Workload("bf16", 128, 128, nk, nv, nt, ns)
    p = w.params(path=path, **flags)
    x = make_inputs(w, 13, act="bf16")
    out, st, _ = run_bf16(torch, w, x, p, workspace=True)
    ro, rs, _ = oracle_mod.forward(p, **x)
    assert_output_bf16(out, ro, nt)
    assert_close("state_out", st, rs, nt)
    fo, fs, _ = run_gpu(w, x, p, workspace=True)
    assert np.array_equal(st.view(np.uint32), fs.view(np.uint32)), "state_out differs from the f32 two-pass form"
    assert np.array_equal(out.view(np.uint32), round_to_bf16(fo).view(np.uint32)), \
        "output is not the f32 two-pass form's output rounded to bf16"


@pytest.mark.parametrize("workspace", [False, True], ids=["one-pass", "two-pass"])
def test_bf16_chunked_segments_and_in_place(torch, workspace):
    """More (seq, value head) chains than SMs (160 chains of 16 chunks): both
    chunked forms cut the chains into segments over launches.  With bf16
    activations the state equals the f32 form's on the same values bit for
    bit and the output equals its output rounded to bf16, out of place and in
    place (state_in == state_out)."""
    w = Workload("bf16seg", 128, 128, 2, 40, 1000, 4)
    p = w.params(path=PATH_CHUNKED, decay_after=True)
    x = make_inputs(w, 17, act="bf16")
    fo, fs, _ = run_gpu(w, x, p, workspace=workspace)
    for in_place in (False, True):
        out, st, _ = run_bf16(torch, w, x, p, in_place=in_place, workspace=workspace)
        assert np.array_equal(st.view(np.uint32), fs.view(np.uint32)), f"state_out (in place: {in_place})"
        assert np.array_equal(out.view(np.uint32), round_to_bf16(fo).view(np.uint32)), f"output (in place: {in_place})"


def test_bf16_in_place_decode(torch, oracle_mod):
    w = Workload("bf16", 128, 128, 4, 8, 1, 4)
    p = w.params()
    x = make_inputs(w, 11, act="bf16")
    out, st, _ = run_bf16(torch, w, x, p, in_place=True)
    ro, rs, _ = oracle_mod.forward(p, **x)
    assert_output_bf16(out, ro, 1)
    assert_close("state_out", st, rs, 1)


@pytest.mark.parametrize("path", [0, PATH_SCAN], ids=["auto-chunked", "scan"])
def test_bf16_long_window_sampled(torch, oracle_mod, path):
    """A 600-token prefill (9 full 64-token chunks + 24; 37 full 16-token
    scan chunks + 8) on the automatic path (the chunked form) and on the
    forced scan, sampled heads; the chunked state also within the split-bf16
    bar."""
    w = Workload("bf16", 128, 128, 2, 6, 600, 2, zero_state=True)
    p = w.params(path=path)
    x = make_inputs(w, 3, act="bf16")
    out, st, _ = run_bf16(torch, w, x, p)
    heads = sample_heads(w, 4, seed=2)
    ro, rs, _ = oracle_mod.forward_heads(p, **x, heads=heads)
    go, gs, _ = gather_heads(w, out, st, None, heads)
    assert_output_bf16(go, ro, w.n_tokens)
    assert_close("state_out", gs, rs, w.n_tokens)
    if path == 0:
        assert_rel_l2("state_out", gs, rs, SPLIT_RELL2_TOL)


@pytest.mark.parametrize("capture", [False, True])
def test_bf16_layers_equal_per_layer_calls(torch, capture):
    from serving_gdn_decode_gb300 import _native as nat
    w = Workload("bf16", 128, 128, 2, 4, 3 if capture else 1, 2)
    p = w.params(decay_after=capture)
    xs = [make_inputs(w, 40 + i, act="bf16") for i in range(5)]
    layers = []
    for x in xs:
        d = _dev_bf16(torch, x)
        d["output"] = torch.empty(w.v_elems, dtype=torch.bfloat16, device="cuda")
        d["state_out"] = torch.empty(w.state_elems, dtype=torch.float32, device="cuda")
        if capture:
            d["state_capture"] = torch.empty(w.capture_elems, dtype=torch.float32, device="cuda")
        layers.append(d)
    nat.gdn_forward_layers(layers, p, with_capture=capture)
    torch.cuda.synchronize()
    for x, d in zip(xs, layers):
        ro, rs, rc = run_bf16(torch, w, x, p, capture=capture)
        assert np.array_equal(d["output"].float().cpu().numpy().view(np.uint32), ro.view(np.uint32))
        assert np.array_equal(d["state_out"].cpu().numpy().view(np.uint32), rs.view(np.uint32))
        if capture:
            assert np.array_equal(d["state_capture"].cpu().numpy().view(np.uint32),
                                  rc.view(np.uint32))


def test_bf16_path_rejects_tf32_chunked(torch):
    """bf16 activations take the chunked path with split operands only."""
    from serving_gdn_decode_gb300 import _native as nat
    w = Workload("bf16", 128, 128, 1, 1, 64, 1)
    x = make_inputs(w, 0, act="bf16")
    with pytest.raises(nat.GdnError, match="f32 activations"):
        run_bf16(torch, w, x, w.params(path=PATH_CHUNKED_TF32))
