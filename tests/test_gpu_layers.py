"""GPU tests of gdn_forward_layers: several problems of one shape in one call
must give exactly what one gdn_forward (or gdn_forward_capture) per problem
gives -- the same kernel code runs on every (layer, seq, head)."""
import numpy as np
import pytest

from gpu_helpers import assert_close, run_gpu, to_dev
from serving_gdn_decode_gb300.params import PATH_SCAN
from serving_gdn_decode_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as t
    assert t.cuda.is_available(), "GPU tests need a CUDA device"
    from serving_gdn_decode_gb300 import build
    build.build()
    return t


def _run_layers(torch, w, xs, params, capture):
    from serving_gdn_decode_gb300 import _native as nat
    layers = []
    for x in xs:
        d = to_dev(x)
        d["output"] = torch.empty(w.v_elems, dtype=torch.float32, device="cuda")
        d["state_out"] = torch.empty(w.state_elems, dtype=torch.float32, device="cuda")
        if capture:
            d["state_capture"] = torch.empty(w.capture_elems, dtype=torch.float32, device="cuda")
        layers.append(d)
    nat.gdn_forward_layers(layers, params, with_capture=capture)
    torch.cuda.synchronize()
    return [(d["output"].cpu().numpy(), d["state_out"].cpu().numpy(),
             d["state_capture"].cpu().numpy() if capture else None) for d in layers]


CASES = [  # (d_k, d_v, n_k, n_v, n_tokens, n_seqs, n_layers, capture, path)
    (128, 128, 4, 8, 1, 3, 1, False, 0),
    (128, 128, 4, 8, 1, 3, 5, False, 0),
    (128, 128, 2, 4, 4, 2, 70, True, 0),     # two launches (64 + 6 layers), capture
    (64, 96, 2, 6, 3, 2, 9, False, 0),
    (32, 33, 1, 3, 2, 1, 4, True, 0),
    (32, 32, 1, 3, 1, 1, 3, False, 0),        # D_k = 32 decode, three layers
    (128, 64, 2, 4, 20, 2, 3, False, 0),      # past the decode window: one launch per layer
    (128, 128, 2, 4, 5, 1, 3, True, PATH_SCAN),
]


@pytest.mark.parametrize("case", CASES, ids=[str(c) for c in CASES])
def test_layers_equal_per_layer_calls(torch, oracle_mod, case):
    dk, dv, nk, nv, nt, ns, nl, capture, path = case
    w = Workload("layers", dk, dv, nk, nv, nt, ns)
    p = w.params(path=path, decay_after=nl % 2 == 0, khead_div=nl % 3 == 0)
    xs = [make_inputs(w, 100 + i) for i in range(nl)]
    got = _run_layers(torch, w, xs, p, capture)
    for i, x in enumerate(xs):
        ref = run_gpu(w, x, p, capture=capture)
        for a, b in zip(got[i], ref):
            if b is not None:
                np.testing.assert_array_equal(a, b)
    ro, rs, rc = oracle_mod.forward(p, **xs[-1], capture=capture)
    assert_close("output", got[-1][0], ro, nt)
    assert_close("state_out", got[-1][1], rs, nt)
