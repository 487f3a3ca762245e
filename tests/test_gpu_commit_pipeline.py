"""GPU tests of the speculative-decode rollback commit and of the pinned-host
pipeline, through the C ABI.

* gdn_commit_capture is a gather: the committed state must equal the chosen
  capture slice bit for bit (and that slice matches the oracle's state after
  accepted_idx + 1 tokens within the parity bar); out-of-range indices keep
  the sequence's state.
* HostPipeline splits the batch over groups of sequences, and gdn_forward_host
  runs the kernel on pinned host buffers (zero-copy); every sequence is
  computed by the same kernel code, so results equal one device call bit for
  bit.
"""
import numpy as np
import pytest

from gpu_helpers import assert_close, run_gpu, to_dev
from serving_gdn_decode_gb300.workloads import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as t
    assert t.cuda.is_available(), "GPU tests need a CUDA device"
    from serving_gdn_decode_gb300 import build
    build.build()
    return t


@pytest.mark.parametrize("name,ns", [("spec_capture", None), ("tiny", None), ("spec_capture", 1)])
def test_commit_gathers_accepted_slice(torch, oracle_mod, name, ns):
    from serving_gdn_decode_gb300 import _native as nat
    w = WORKLOADS[name] if ns is None else WORKLOADS[name].with_(n_seqs=ns)
    x = make_inputs(w, 3)
    d = to_dev(x)
    p = w.params()
    out = torch.empty(w.v_elems, dtype=torch.float32, device="cuda")
    st = torch.empty(w.state_elems, dtype=torch.float32, device="cuda")
    cap = torch.empty(w.capture_elems, dtype=torch.float32, device="cuda")
    nat.gdn_forward_capture(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state_in"], out, st, p, cap)
    rng = np.random.default_rng(5)
    idx = rng.integers(-1, w.n_tokens + 1, size=w.n_seqs).astype(np.int32)  # includes -1 and T
    idx[0] = w.n_tokens - 1
    active = d["state_in"].clone()
    nat.gdn_commit_capture(cap, torch.from_numpy(idx).cuda(), active, p)
    torch.cuda.synchronize()
    got = active.cpu().numpy().reshape(w.n_seqs, -1)
    capn = cap.cpu().numpy().reshape(w.n_seqs, w.n_tokens, -1)
    s0 = x["state_in"].reshape(w.n_seqs, -1)
    for s in range(w.n_seqs):
        want = capn[s, idx[s]] if 0 <= idx[s] < w.n_tokens else s0[s]
        np.testing.assert_array_equal(got[s], want)
    np.testing.assert_array_equal(got[0], st.cpu().numpy().reshape(w.n_seqs, -1)[0])
    # the committed state is the recurrence's state after idx+1 tokens
    _, _, rc = oracle_mod.forward(p, **x, capture=True)
    rc = rc.reshape(w.n_seqs, w.n_tokens, -1)
    sel = [s for s in range(w.n_seqs) if 0 <= idx[s] < w.n_tokens]
    assert_close("committed", np.stack([got[s] for s in sel]),
                 np.stack([rc[s, idx[s]] for s in sel]), w.n_tokens)


@pytest.mark.parametrize("groups", [1, 3, 4, 19, 64])
def test_host_pipeline_equals_device_call(torch, groups):
    from serving_gdn_decode_gb300 import _native as nat
    w = Workload("pipe", 128, 128, 4, 8, 2, 19)
    x = make_inputs(w, 7)
    p = w.params()
    ref_out, ref_st, _ = run_gpu(w, x, p)
    host = {k: torch.from_numpy(v).pin_memory() for k, v in x.items()}
    out = torch.zeros(w.v_elems, dtype=torch.float32).pin_memory()
    st = torch.zeros(w.state_elems, dtype=torch.float32).pin_memory()
    pipe = nat.HostPipeline(p, groups=groups)
    for _ in range(2):  # buffers are reused across calls
        pipe(host["q"], host["k"], host["v"], host["g"], host["beta"], host["state_in"], out, st)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out.numpy(), ref_out)
        np.testing.assert_array_equal(st.numpy(), ref_st)
    assert pipe.h2d_bytes() == 4 * sum(v.size for v in x.values())
    assert pipe.d2h_bytes() == 4 * (w.v_elems + w.state_elems)


def test_host_pipeline_rejects_device_tensors(torch):
    from serving_gdn_decode_gb300 import _native as nat
    w = Workload("pipe", 128, 128, 4, 8, 2, 4)
    pipe = nat.HostPipeline(w.params())
    t = torch.zeros(4, device="cuda")
    with pytest.raises(nat.GdnError):
        pipe(t, t, t, t, t, t, t, t)


ZC_CASES = [  # (workload, capture, act, path)
    (Workload("zc", 128, 128, 4, 8, 1, 6), False, "f32", 0),        # decode
    (Workload("zc", 128, 128, 2, 4, 4, 3), True, "f32", 0),         # capture window
    (Workload("zc", 64, 96, 2, 6, 40, 2), True, "f32", 0),          # scan path
    (Workload("zc", 128, 128, 4, 8, 3, 5), True, "bf16", 0),        # bf16 activations
]


@pytest.mark.parametrize("case", ZC_CASES, ids=["decode", "capture", "scan", "bf16"])
def test_zero_copy_host_call_equals_device_call(torch, case):
    """gdn_forward_host runs the same kernel on pinned host buffers: results
    equal the device-buffer call bit for bit."""
    from serving_gdn_decode_gb300 import _native as nat
    w, capture, act, path = case
    x = make_inputs(w, 21, act=act)
    p = w.params(path=path)
    adt = torch.bfloat16 if act == "bf16" else torch.float32

    def on(dev):
        t = {k: torch.from_numpy(v) for k, v in x.items()}
        for k in ("q", "k", "v"):
            t[k] = t[k].to(adt)
        t = {k: (v.cuda() if dev else v.pin_memory()) for k, v in t.items()}
        mk = (lambda n, d: torch.zeros(n, dtype=d, device="cuda")) if dev else \
            (lambda n, d: torch.zeros(n, dtype=d).pin_memory())
        out, st = mk(w.v_elems, adt), mk(w.state_elems, torch.float32)
        cap = mk(w.capture_elems, torch.float32) if capture else None
        args = (t["q"], t["k"], t["v"], t["g"], t["beta"], t["state_in"], out, st, p)
        if dev:
            if capture:
                nat.gdn_forward_capture(*args, cap)
            else:
                nat.gdn_forward(*args)
        else:
            nat.gdn_forward_host(*args, state_capture=cap)
        torch.cuda.synchronize()
        return [None if a is None else a.cpu().view(torch.int16 if a.dtype == torch.bfloat16
                                                   else torch.int32).numpy() for a in (out, st, cap)]

    for a, b in zip(on(False), on(True)):
        if b is not None:
            np.testing.assert_array_equal(a, b)


def test_zero_copy_rejects_device_and_pageable(torch):
    from serving_gdn_decode_gb300 import _native as nat
    w = Workload("zc", 32, 32, 1, 2, 1, 1)
    x = {k: torch.from_numpy(v).pin_memory() for k, v in make_inputs(w, 0).items()}
    out = torch.zeros(w.v_elems).pin_memory()
    st = torch.zeros(w.state_elems).pin_memory()
    with pytest.raises(nat.GdnError, match="pinned host"):
        nat.gdn_forward_host(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state_in"],
                             torch.zeros(w.v_elems), st, w.params())     # pageable output
    with pytest.raises(nat.GdnError, match="pinned host"):
        nat.gdn_forward_host(x["q"].cuda(), x["k"], x["v"], x["g"], x["beta"], x["state_in"],
                             out, st, w.params())
