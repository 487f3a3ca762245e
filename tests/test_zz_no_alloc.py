"""GPU test of gdn_forward_chunked_noalloc, the entry point for callers that
cannot allocate device memory -- code that only receives device buffers
from a framework owning all device memory, or loops that must not call
cudaMalloc.  It runs the two-pass chunked prefill with its chunk scratch in
a fixed 32 MiB array inside the library instead of a caller workspace.

Through the C ABI, two calls in a row (different inputs, so anything left
in the shared scratch by the first call would show in the second) must give
what gdn_forward_ws gives with its own workspace, and what the oracle gives,
within the long-window bar of the other GPU tests; an in-place call
(state_in == state_out) must equal the out-of-place one bit for bit; a
problem needing more than the fixed scratch is refused with a clear error.
The file is named to be collected last.
"""
import numpy as np
import pytest

from gpu_helpers import assert_close, run_gpu, to_dev
from serving_gdn_decode_gb300.params import PATH_CHUNKED
from serving_gdn_decode_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as t
    assert t.cuda.is_available(), "GPU tests need a CUDA device"
    from serving_gdn_decode_gb300 import build
    build.build()
    return t


def _noalloc(torch, w, x, params, in_place=False):
    from serving_gdn_decode_gb300 import _native as nat
    d = to_dev(x)
    out = torch.empty(w.v_elems, dtype=torch.float32, device="cuda")
    st = d["state_in"].clone() if in_place else torch.empty(w.state_elems, dtype=torch.float32,
                                                            device="cuda")
    st_in = st if in_place else d["state_in"]
    stream = torch.cuda.current_stream().cuda_stream
    rc = nat.forward_chunked_noalloc_raw(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(),
                                         d["g"].data_ptr(), d["beta"].data_ptr(),
                                         st_in.data_ptr(), out.data_ptr(), st.data_ptr(),
                                         params, stream)
    assert rc == nat.GDN_OK, nat.gdn_last_error()
    torch.cuda.synchronize()
    return out.cpu().numpy(), st.cpu().numpy()


def test_noalloc_matches_workspace_entry_point_twice(torch, oracle_mod):
    # 4 value heads x 2 seqs x 5 chunks (300 tokens: 4 full chunks + 44)
    w = Workload("noalloc", 128, 128, 2, 4, 300, 2)
    for call, seed in enumerate((71, 72)):
        x = make_inputs(w, seed)
        p = w.params(path=PATH_CHUNKED, decay_after=call == 1)
        out, st = _noalloc(torch, w, x, p)
        ref_out, ref_st, _ = run_gpu(w, x, p, workspace=True)
        assert_close("output", out, ref_out.astype(np.float64), w.n_tokens)
        assert_close("state_out", st, ref_st.astype(np.float64), w.n_tokens)
        # and against the oracle directly, for both this call and the
        # workspace call it was compared with
        ro, rs, _ = oracle_mod.forward(p, **x)
        for o, s_ in ((out, st), (ref_out, ref_st)):
            assert_close("output", o, ro, w.n_tokens)
            assert_close("state_out", s_, rs, w.n_tokens)


def test_noalloc_in_place(torch):
    w = Workload("noalloc_inplace", 128, 128, 2, 4, 100, 2)
    x = make_inputs(w, 75)
    p = w.params(path=PATH_CHUNKED)
    out, st = _noalloc(torch, w, x, p)
    out2, st2 = _noalloc(torch, w, x, p, in_place=True)
    np.testing.assert_array_equal(out2, out)
    np.testing.assert_array_equal(st2, st)


def test_noalloc_refuses_more_than_its_scratch(torch):
    from serving_gdn_decode_gb300 import _native as nat
    # 16 seqs x 17 chunks x (4 x 32 KB + 2 x 96 KB) = 85 MiB > 32 MiB; real
    # buffers of that shape, so the refusal is the only thing tested
    w = Workload("noalloc_big", 128, 128, 2, 4, 1025, 16)
    x = to_dev(make_inputs(w, 73))
    out = torch.empty(w.v_elems, dtype=torch.float32, device="cuda")
    st = torch.empty(w.state_elems, dtype=torch.float32, device="cuda")
    rc = nat.forward_chunked_noalloc_raw(x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(),
                                         x["g"].data_ptr(), x["beta"].data_ptr(),
                                         x["state_in"].data_ptr(), out.data_ptr(), st.data_ptr(),
                                         w.params(path=PATH_CHUNKED))
    assert rc == nat.GDN_ERR_INVALID_ARGUMENT
    assert "gdn_forward_ws" in nat.gdn_last_error()


def test_noalloc_beyond_the_two_pass_group_limit(torch):
    # 40 value heads on one key head: the entry point runs the one-pass form,
    # which needs no scratch, and matches gdn_forward exactly
    w = Workload("noalloc_g40", 128, 128, 1, 40, 70, 1)
    x = make_inputs(w, 74)
    p = w.params(path=PATH_CHUNKED)
    out, st = _noalloc(torch, w, x, p)
    ref_out, ref_st, _ = run_gpu(w, x, p)
    np.testing.assert_array_equal(out, ref_out)
    np.testing.assert_array_equal(st, ref_st)
