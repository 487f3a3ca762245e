"""Host-side tests of the C ABI (no GPU needed).

* the library loads and exports every function include/gdn.h declares;
* argument checks return the documented status before anything is enqueued.

Buffer-check cases pass made-up device addresses, so each of them has
exactly one invalid argument and must be rejected on the host.  They are
skipped where a CUDA device is visible: there a wrongly accepted call would
launch a kernel on those addresses.
"""
import ctypes

import numpy as np
import pytest

from serving_gdn_decode_gb300 import _native as nat
from serving_gdn_decode_gb300.params import PATH_CHUNKED, PATH_CHUNKED_TF32, PATH_SCAN, pack_params
from serving_gdn_decode_gb300.workloads import WORKLOADS, Workload


@pytest.fixture(scope="module")
def L():
    from serving_gdn_decode_gb300 import build
    build.build()
    return nat.lib()


def _has_cuda_device():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


no_device = pytest.mark.skipif(_has_cuda_device(), reason="fake-address cases run only without a GPU")


def test_exports_every_declared_function(L):
    names = nat.header_functions()
    assert {"gdn_forward", "gdn_forward_capture", "gdn_last_error", "gdn_path_name"} <= set(names)
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/gdn.h but not exported"


def test_header_constants_match_binding():
    text = open(nat.HEADER_PATH).read()
    for name, val in (("GDN_OK", 0), ("GDN_ERR_INVALID_ARGUMENT", 1), ("GDN_ERR_UNSUPPORTED", 2),
                      ("GDN_ERR_CUDA", 3)):
        assert f"{name} = {val}" in text
    assert "#define GDN_N_PARAMS 9" in text
    assert "#define GDN_FLAG_DECAY_AFTER 0x1u" in text and "#define GDN_FLAG_KHEAD_DIV 0x2u" in text


def test_device_status_constants_and_null(L):
    text = open(nat.HEADER_PATH).read()
    assert "#define GDN_DEVICE_WAIT_TIMEOUT 0x1u" in text
    assert nat.GDN_DEVICE_WAIT_TIMEOUT == 0x1
    # a NULL result pointer is refused before any CUDA call
    assert L.gdn_device_status(None, 0, None) == nat.GDN_ERR_INVALID_ARGUMENT
    assert "status is NULL" in nat.gdn_last_error()


# ---------------------------------------------------------------- params-only checks

def _path(p, capture=False):
    return nat.gdn_path_name(p, capture)


def test_path_choice(L):
    assert _path(WORKLOADS["decode"].params()) == "token_loop_decode"
    assert _path(WORKLOADS["decode_wide_gqa"].params(khead_div=True)) == "token_loop_decode"
    assert _path(WORKLOADS["spec_capture"].params(), True) == "token_loop_decode_capture"
    assert _path(WORKLOADS["long_prefill"].params()) == "chunked"
    assert _path(WORKLOADS["long_prefill"].params(path=PATH_SCAN)) == "scan"
    assert _path(WORKLOADS["long_prefill"].params(path=PATH_CHUNKED_TF32)) == "chunked_tf32"
    assert _path(WORKLOADS["tiny"].params(path=PATH_SCAN), True) == "scan_capture"
    assert _path(WORKLOADS["decode"].with_(n_tokens=16).params()) == "token_loop_decode"
    assert _path(WORKLOADS["decode"].with_(n_tokens=17).params()) == "scan"
    # the automatic choice takes the chunked form from 48 tokens on, where it covers the shape
    assert _path(WORKLOADS["decode"].with_(n_tokens=47).params()) == "scan"
    assert _path(WORKLOADS["decode"].with_(n_tokens=48).params()) == "chunked"
    # every capture window takes the token loop under the automatic choice
    assert _path(WORKLOADS["long_prefill"].params(), True) == "token_loop_decode_capture"
    assert _path(pack_params(64, 64, 2, 4, 4096, 1)) == "scan"
    assert _path(pack_params(128, 64, 2, 4, 4096, 1)) == "scan"


@pytest.mark.parametrize("mutate,status", [
    (lambda p: p[:8], nat.GDN_ERR_INVALID_ARGUMENT),                 # fewer than 9 u32
    (lambda p: _set(p, 0, 0), nat.GDN_ERR_INVALID_ARGUMENT),         # D_k = 0
    (lambda p: _set(p, 1, 0), nat.GDN_ERR_INVALID_ARGUMENT),         # D_v = 0
    (lambda p: _set(p, 2, 0), nat.GDN_ERR_INVALID_ARGUMENT),         # n_k = 0
    (lambda p: _set(p, 3, 0), nat.GDN_ERR_INVALID_ARGUMENT),         # n_v = 0
    (lambda p: _set(p, 4, 0), nat.GDN_ERR_INVALID_ARGUMENT),         # n_tokens = 0
    (lambda p: _set(p, 5, 0), nat.GDN_ERR_INVALID_ARGUMENT),         # n_seqs = 0
    (lambda p: _set(p, 3, 24), nat.GDN_ERR_INVALID_ARGUMENT),        # n_v % n_k != 0
    (lambda p: _set(p, 0, 48), nat.GDN_ERR_INVALID_ARGUMENT),        # D_k % 32 != 0
    (lambda p: _set(p, 0, 160), nat.GDN_ERR_INVALID_ARGUMENT),       # D_k/32 > 4
    (lambda p: _set(p, 0, 96), nat.GDN_ERR_UNSUPPORTED),             # D_k/32 = 3
    (lambda p: _set(p, 1, 126), nat.GDN_ERR_INVALID_ARGUMENT),       # D_v % (D_k/32) != 0
    (lambda p: _set(p, 7, 1), nat.GDN_ERR_INVALID_ARGUMENT),         # reserved slot
    (lambda p: _set(p, 6, 0x10), nat.GDN_ERR_INVALID_ARGUMENT),      # unknown flag bit
])
def test_params_rejected(L, mutate, status):
    p = mutate(WORKLOADS["decode"].params())
    with pytest.raises(nat.GdnError) as e:
        _path(p)
    assert e.value.status == status
    assert nat.gdn_last_error() != ""


def _set(p, i, val):
    p = p.copy()
    p[i] = val
    return p


def test_chunked_forced_with_capture_is_unsupported(L):
    with pytest.raises(nat.GdnError) as e:
        _path(WORKLOADS["spec_capture"].params(path=PATH_CHUNKED), capture=True)
    assert e.value.status == nat.GDN_ERR_UNSUPPORTED


def test_chunked_path_shapes(L):
    assert _path(WORKLOADS["long_prefill"].params(path=PATH_CHUNKED)) == "chunked"
    for dk, dv in ((64, 64), (128, 64), (32, 32)):
        with pytest.raises(nat.GdnError) as e:
            _path(pack_params(dk, dv, 1, 2, 100, 1, path=PATH_CHUNKED))
        assert e.value.status == nat.GDN_ERR_UNSUPPORTED


def test_supported_head_dims(L):
    for dk in (32, 64, 128):
        nsg = dk // 32
        for dv in (nsg, 3 * nsg, 128, 200 - 200 % nsg):
            assert _path(pack_params(dk, dv, 2, 6, 3, 2)) == "token_loop_decode"


# ---------------------------------------------------------------- buffer checks (fake addresses)

GAP = 1 << 32


class Fake:
    """Disjoint, 256-byte aligned made-up device addresses for each buffer."""

    def __init__(self, w, capture=False):
        self.w = w
        names = ["q", "k", "v", "g", "beta", "state_in", "output", "state_out", "state_capture"]
        self.addr = {n: (i + 1) * GAP for i, n in enumerate(names)}
        self.cap_elems = w.capture_elems

    def call(self, params=None, capture=False, bf16=False, **over):
        a = dict(self.addr, **over)
        p = self.w.params() if params is None else params
        args = [a[n] for n in ("q", "k", "v", "g", "beta", "state_in", "output", "state_out")]
        if capture:
            return nat.forward_capture_raw(*args, p, a["state_capture"],
                                           over.get("cap_elems", self.cap_elems), bf16=bf16)
        return nat.forward_raw(*args, p, bf16=bf16)


SMALL = WORKLOADS["decode"].with_(n_seqs=2, n_tokens=3)
SMALL1 = WORKLOADS["decode"].with_(n_seqs=1, n_tokens=3)


@no_device
@pytest.mark.parametrize("name", ["q", "k", "v", "g", "beta", "state_in", "output", "state_out"])
def test_null_buffer(L, name):
    f = Fake(SMALL)
    assert f.call(**{name: 0}) == nat.GDN_ERR_INVALID_ARGUMENT
    assert name in nat.gdn_last_error()


@no_device
@pytest.mark.parametrize("name,off", [("q", 4), ("k", 8), ("state_in", 4), ("state_out", 12),
                                      ("v", 2), ("g", 1), ("beta", 3), ("output", 2)])
def test_misaligned_buffer(L, name, off):
    f = Fake(SMALL)
    assert f.call(**{name: f.addr[name] + off}) == nat.GDN_ERR_INVALID_ARGUMENT
    assert "aligned" in nat.gdn_last_error()


@no_device
def test_partial_state_alias_rejected(L):
    f = Fake(SMALL)
    assert f.call(state_out=f.addr["state_in"] + 16) == nat.GDN_ERR_INVALID_ARGUMENT
    assert "overlap" in nat.gdn_last_error()


@no_device
@pytest.mark.parametrize("victim", ["q", "v", "state_in", "state_out"])
def test_output_overlap_rejected(L, victim):
    f = Fake(SMALL)
    assert f.call(output=f.addr[victim] + 16) == nat.GDN_ERR_INVALID_ARGUMENT


@no_device
def test_state_out_overlapping_input_rejected(L):
    f = Fake(SMALL)
    assert f.call(state_out=f.addr["k"]) == nat.GDN_ERR_INVALID_ARGUMENT


@no_device
def test_capture_size_rules(L):
    f = Fake(SMALL, capture=True)
    need = SMALL.capture_elems
    # n_seqs > 1: exact size only
    assert f.call(capture=True, cap_elems=need + 4) == nat.GDN_ERR_INVALID_ARGUMENT
    assert f.call(capture=True, cap_elems=need - 4) == nat.GDN_ERR_INVALID_ARGUMENT
    # n_seqs == 1: smaller is rejected (larger is accepted; not called here)
    f1 = Fake(SMALL1, capture=True)
    assert f1.call(capture=True, cap_elems=SMALL1.capture_elems - 1) == nat.GDN_ERR_INVALID_ARGUMENT
    assert f.call(capture=True, state_capture=0) == nat.GDN_ERR_INVALID_ARGUMENT
    assert f.call(capture=True, state_capture=f.addr["state_capture"] + 4) == \
        nat.GDN_ERR_INVALID_ARGUMENT
    assert f.call(capture=True, state_capture=f.addr["state_out"]) == nat.GDN_ERR_INVALID_ARGUMENT
    assert f.call(capture=True, state_capture=f.addr["v"] + 64) == nat.GDN_ERR_INVALID_ARGUMENT


@no_device
def test_invalid_params_through_forward(L):
    f = Fake(SMALL)
    p = SMALL.params()
    p[3] = 17
    assert f.call(params=p) == nat.GDN_ERR_INVALID_ARGUMENT
    assert f.call(params=SMALL.params()[:8]) == nat.GDN_ERR_INVALID_ARGUMENT
    assert nat.lib().gdn_forward(*([GAP] * 8), None, 9, None) == nat.GDN_ERR_INVALID_ARGUMENT


def test_capture_memory_cost_matches_pages():
    """'Memory cost' section of gated_delta_net_decode_capture.metal: D_k = D_v =
    128, n_v = 8, n_seqs = 1, K+1 = 4 tokens -> 128*128*8*4*4 bytes = 2 MB per
    linear-attention layer."""
    w = WORKLOADS["spec_capture"].with_(n_v_heads=8, n_seqs=1, n_tokens=4)
    assert w.capture_elems * 4 == 2 * 1024 * 1024
    assert WORKLOADS["spec_capture"].capture_elems * 4 == 256 * 1024 * 1024


def test_binding_rejects_before_calling():
    torch = pytest.importorskip("torch")
    x = torch.zeros(4)
    with pytest.raises(nat.GdnError):
        nat.gdn_forward(x, x, x, x, x, x, x, x, pack_params(32, 32, 1, 1, 1, 1))


# ---------------------------------------------------------------- rollback commit checks

@no_device
def test_commit_checks(L):
    w = SMALL
    cap, idx, st = 1 * GAP, 2 * GAP, 3 * GAP
    p = w.params()
    ok_elems = w.capture_elems
    assert nat.commit_capture_raw(0, ok_elems, idx, st, p) == nat.GDN_ERR_INVALID_ARGUMENT
    assert nat.commit_capture_raw(cap, ok_elems, 0, st, p) == nat.GDN_ERR_INVALID_ARGUMENT
    assert nat.commit_capture_raw(cap, ok_elems, idx, 0, p) == nat.GDN_ERR_INVALID_ARGUMENT
    assert nat.commit_capture_raw(cap + 8, ok_elems, idx, st, p) == nat.GDN_ERR_INVALID_ARGUMENT
    assert nat.commit_capture_raw(cap, ok_elems, idx + 2, st, p) == nat.GDN_ERR_INVALID_ARGUMENT
    assert nat.commit_capture_raw(cap, ok_elems + 4, idx, st, p) == nat.GDN_ERR_INVALID_ARGUMENT
    assert nat.commit_capture_raw(cap, ok_elems, idx, cap + 64, p) == nat.GDN_ERR_INVALID_ARGUMENT
    assert nat.commit_capture_raw(cap, ok_elems, idx, idx, p) == nat.GDN_ERR_INVALID_ARGUMENT
    assert nat.commit_capture_raw(cap, ok_elems, idx, st, p[:8]) == nat.GDN_ERR_INVALID_ARGUMENT
    w1 = SMALL1
    assert nat.commit_capture_raw(cap, w1.capture_elems - 1, idx, st, w1.params()) == \
        nat.GDN_ERR_INVALID_ARGUMENT


# ---------------------------------------------------------------- multi-layer checks

def _layer_rows(n, base=1 << 36):
    names = ["q", "k", "v", "g", "beta", "state_in", "output", "state_out", "state_capture"]
    return [[base + (9 * i + j) * GAP for j in range(len(names))] for i in range(n)]


@no_device
def test_layers_checks(L):
    p = SMALL.params()
    assert nat.forward_layers_raw([], p) == nat.GDN_ERR_INVALID_ARGUMENT
    rows = _layer_rows(3)
    rows[1][0] = 0                                     # layer 1: q is NULL
    assert nat.forward_layers_raw(rows, p) == nat.GDN_ERR_INVALID_ARGUMENT
    assert "layer 1" in nat.gdn_last_error()
    rows = _layer_rows(3)
    rows[2][6] = rows[0][1] + 64                       # layer 2's output inside layer 0's k
    assert nat.forward_layers_raw(rows, p) == nat.GDN_ERR_INVALID_ARGUMENT
    assert "layer 2" in nat.gdn_last_error() and "layer 0" in nat.gdn_last_error()
    rows = _layer_rows(2)
    rows[1][7] = rows[0][7]                            # two layers write the same state
    assert nat.forward_layers_raw(rows, p) == nat.GDN_ERR_INVALID_ARGUMENT
    assert nat.forward_layers_raw(_layer_rows(2), p[:8]) == nat.GDN_ERR_INVALID_ARGUMENT
    rows = _layer_rows(2)
    assert nat.forward_layers_raw(rows, p, with_capture=True,
                                  state_capture_elems=SMALL.capture_elems - 4) == \
        nat.GDN_ERR_INVALID_ARGUMENT


@no_device
def test_layers_count_limit(L):
    rows = _layer_rows(1025, base=1 << 40)
    assert nat.forward_layers_raw(rows, SMALL.params()) == nat.GDN_ERR_INVALID_ARGUMENT


# ---------------------------------------------------------------- bf16 activations

@no_device
@pytest.mark.parametrize("name,off", [("q", 8), ("k", 2), ("v", 2), ("output", 1), ("g", 2),
                                      ("state_in", 8)])
def test_bf16_misaligned_buffer(L, name, off):
    f = Fake(SMALL)
    assert f.call(bf16=True, **{name: f.addr[name] + off}) == nat.GDN_ERR_INVALID_ARGUMENT
    assert "aligned" in nat.gdn_last_error()


@no_device
def test_bf16_spans_are_two_bytes(L):
    """With bf16 activations, v and output take 2 bytes per element: an output
    placed right after v's bf16 extent passes every host check (the launch
    then fails here for want of a device), while the same placement overlaps
    v's f32 extent."""
    f = Fake(SMALL)
    after_v = f.addr["v"] + SMALL.v_elems * 2
    assert f.call(bf16=True, output=after_v) == nat.GDN_ERR_CUDA
    assert f.call(output=after_v) == nat.GDN_ERR_INVALID_ARGUMENT
    # 2-byte aligned output is enough for bf16, not for f32
    assert f.call(bf16=True, output=f.addr["output"] + 2) == nat.GDN_ERR_CUDA
    assert f.call(output=f.addr["output"] + 2) == nat.GDN_ERR_INVALID_ARGUMENT


@no_device
def test_bf16_unsupported_shapes(L):
    odd = WORKLOADS["tiny"].with_(d_v=33)
    assert Fake(odd).call(bf16=True) == nat.GDN_ERR_UNSUPPORTED
    assert "even D_v" in nat.gdn_last_error()
    assert Fake(odd).call() != nat.GDN_ERR_UNSUPPORTED       # f32 takes odd D_v
    w = WORKLOADS["long_prefill"].with_(n_tokens=64, n_seqs=1)
    # bf16 activations take the chunked path with split operands, not with TF32 ones
    assert Fake(w).call(params=w.params(path=PATH_CHUNKED_TF32), bf16=True) == nat.GDN_ERR_UNSUPPORTED
    assert "f32 activations" in nat.gdn_last_error()
    assert Fake(w).call(params=w.params(path=PATH_CHUNKED), bf16=True) == nat.GDN_ERR_CUDA  # host checks pass
    assert Fake(w).call(params=w.params(), bf16=True) == nat.GDN_ERR_CUDA


@no_device
def test_bf16_layers_checks(L):
    p = SMALL.params()
    rows = _layer_rows(2)
    rows[1][2] += 2                                    # layer 1: v only 2-byte aligned
    assert nat.forward_layers_raw(rows, p, bf16=True) == nat.GDN_ERR_INVALID_ARGUMENT
    assert "layer 1" in nat.gdn_last_error()
    rows = _layer_rows(2)
    rows[1][6] = rows[0][2] + SMALL.v_elems * 2 - 2    # layer 1's output on layer 0's last v
    assert nat.forward_layers_raw(rows, p, bf16=True) == nat.GDN_ERR_INVALID_ARGUMENT


def test_binding_bf16_dtype_rules():
    torch = pytest.importorskip("torch")
    w = WORKLOADS["tiny"]
    p = w.params()
    bf, f32 = torch.bfloat16, torch.float32
    t = {n: torch.zeros(getattr(w, f"{e}_elems"), dtype=d) for n, e, d in (
        ("q", "qk", bf), ("k", "qk", bf), ("v", "v", bf), ("g", "scalar", f32),
        ("beta", "scalar", f32), ("state_in", "state", f32), ("output", "v", bf),
        ("state_out", "state", f32))}
    with pytest.raises(nat.GdnError, match="k must be bf16"):
        nat.gdn_forward(**dict(t, k=t["k"].float()), params=p)
    with pytest.raises(nat.GdnError, match="g must be f32"):
        nat.gdn_forward(**dict(t, g=t["g"].to(bf)), params=p)
    with pytest.raises(nat.GdnError, match="q must be an f32 or bf16"):
        nat.gdn_forward(**dict(t, q=t["q"].half()), params=p)
    with pytest.raises(nat.GdnError, match="CUDA tensor"):   # all dtypes right: device check
        nat.gdn_forward(**t, params=p)
    with pytest.raises(nat.GdnError, match="pinned host"):   # zero-copy call: pageable memory
        nat.gdn_forward_host(**t, params=p)


def test_round_to_bf16_matches_torch():
    """The input generator's bf16 rounding (round to nearest, ties to even)
    against torch's float32 -> bfloat16 conversion, bit for bit, on random
    values, halfway cases, zeros, subnormals and values near the f32 limit."""
    torch = pytest.importorskip("torch")
    from serving_gdn_decode_gb300.workloads import round_to_bf16
    x = np.random.default_rng(1).standard_normal(1 << 16).astype(np.float32) * np.float32(3)
    x = np.concatenate([x, np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, -1.00390625,
                                     3.0e38, -1e-40, 1e-38], np.float32)])
    a = round_to_bf16(x)
    b = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


# ---------------------------------------------------------------- two-pass workspace

def test_workspace_size_values(L):
    w = WORKLOADS["long_prefill"].with_(n_tokens=200, n_seqs=3)
    # per (seq, chunk): 32 KB per value head (48) + 96 KB per key head (16); 3 seqs x 4 chunks
    assert nat.gdn_workspace_size(w.params(path=PATH_CHUNKED)) == 3 * 4 * (48 * 32768 + 16 * 98304)
    # auto: the chunked form from 48 tokens on, in two passes given a workspace from 512
    # tokens on (the one pass is the faster form below), else the scan
    assert nat.gdn_workspace_size(w.params()) == 0
    w600 = w.with_(n_tokens=600)
    assert nat.gdn_workspace_size(w600.params()) == nat.gdn_workspace_size(w600.params(path=PATH_CHUNKED))
    assert nat.gdn_workspace_size(w600.with_(n_tokens=511).params()) == 0
    assert nat.gdn_workspace_size(w600.with_(n_tokens=512).params()) == 3 * 8 * (48 * 32768 + 16 * 98304)
    assert nat.gdn_workspace_size(w.params(path=PATH_CHUNKED_TF32)) == \
        nat.gdn_workspace_size(w.params(path=PATH_CHUNKED))       # same layout sizes
    assert nat.gdn_workspace_size(w.with_(n_tokens=47).params()) == 0
    assert nat.gdn_workspace_size(w.params(path=PATH_SCAN)) == 0
    assert nat.gdn_workspace_size(SMALL.params()) == 0               # decode
    with pytest.raises(nat.GdnError):
        nat.gdn_workspace_size(SMALL.params()[:8])


@no_device
def test_workspace_checks(L):
    w = WORKLOADS["long_prefill"].with_(n_tokens=100, n_seqs=1)
    p = w.params(path=PATH_CHUNKED)
    need = nat.gdn_workspace_size(p)
    f = Fake(w)
    args = [f.addr[n] for n in ("q", "k", "v", "g", "beta", "state_in", "output", "state_out")]
    ws = 10 * GAP
    assert nat.forward_ws_raw(*args, p, 0, need) == nat.GDN_ERR_INVALID_ARGUMENT
    assert "NULL" in nat.gdn_last_error()
    assert nat.forward_ws_raw(*args, p, ws + 8, need) == nat.GDN_ERR_INVALID_ARGUMENT
    assert nat.forward_ws_raw(*args, p, ws, need - 16) == nat.GDN_ERR_INVALID_ARGUMENT
    assert nat.forward_ws_raw(*args, p, f.addr["v"] + 64, need) == nat.GDN_ERR_INVALID_ARGUMENT
    assert "overlaps" in nat.gdn_last_error()
    # a good workspace passes every host check (the launch then fails here for want of a device)
    assert nat.forward_ws_raw(*args, p, ws, need) == nat.GDN_ERR_CUDA
    # off the chunked path the workspace is not needed
    assert nat.forward_ws_raw(*args, w.params(path=PATH_SCAN), 0, 0) == nat.GDN_ERR_CUDA
    # the automatic choice at 100 tokens is the one-pass chunked form (the faster below 512
    # tokens), which needs none; from 512 tokens on it is the two-pass form, which needs it
    assert nat.forward_ws_raw(*args, w.params(), 0, 0) == nat.GDN_ERR_CUDA
    w6 = w.with_(n_tokens=600)
    f6 = Fake(w6)
    args6 = [f6.addr[n] for n in ("q", "k", "v", "g", "beta", "state_in", "output", "state_out")]
    need6 = nat.gdn_workspace_size(w6.params())
    assert need6 == nat.gdn_workspace_size(w6.params(path=PATH_CHUNKED)) > 0
    assert nat.forward_ws_raw(*args6, w6.params(), 0, need6) == nat.GDN_ERR_INVALID_ARGUMENT
    assert nat.forward_ws_raw(*args6, w6.params(), 10 * GAP, need6) == nat.GDN_ERR_CUDA


@no_device
def test_workspace_bf16_checks(L):
    """gdn_forward_ws_bf16: the workspace checks of gdn_forward_ws with the
    bf16 checks of gdn_forward_bf16; the TF32 chunked path is refused."""
    w = WORKLOADS["long_prefill"].with_(n_tokens=100, n_seqs=1)
    p = w.params(path=PATH_CHUNKED)
    need = nat.gdn_workspace_size(p)
    f = Fake(w)
    args = [f.addr[n] for n in ("q", "k", "v", "g", "beta", "state_in", "output", "state_out")]
    ws = 10 * GAP
    assert nat.forward_ws_raw(*args, p, 0, need, bf16=True) == nat.GDN_ERR_INVALID_ARGUMENT
    assert nat.forward_ws_raw(*args, p, ws, need - 16, bf16=True) == nat.GDN_ERR_INVALID_ARGUMENT
    assert nat.forward_ws_raw(*args, p, ws, need, bf16=True) == nat.GDN_ERR_CUDA   # host checks pass
    assert nat.forward_ws_raw(*args, w.params(), ws, need, bf16=True) == nat.GDN_ERR_CUDA
    assert nat.forward_ws_raw(*args, w.params(path=PATH_CHUNKED_TF32), ws, need, bf16=True) == \
        nat.GDN_ERR_UNSUPPORTED
    assert "f32 activations" in nat.gdn_last_error()
    v2 = list(args)
    v2[2] += 2                                               # bf16 v 2-byte aligned only
    assert nat.forward_ws_raw(*v2, p, ws, need, bf16=True) == nat.GDN_ERR_INVALID_ARGUMENT


@no_device
def test_noalloc_host_checks(L):
    """gdn_forward_chunked_noalloc: the fixed 32 MiB scratch holds 16 chunks
    of 16 value and 16 key heads (2 MiB each); one more chunk is refused
    before anything is enqueued, and a
    problem that fits passes every host check (the launch then fails here for
    want of a device).  Non-chunked path bits and shapes are refused."""
    def call(w, params=None, **over):
        f = Fake(w)
        a = dict(f.addr, **over)
        args = [a[n] for n in ("q", "k", "v", "g", "beta", "state_in", "output", "state_out")]
        return nat.forward_chunked_noalloc_raw(*args, w.params(path=PATH_CHUNKED) if params is None
                                               else params)
    fits = WORKLOADS["long_prefill"].with_(n_v_heads=16, n_k_heads=16, n_seqs=1, n_tokens=1024)
    assert call(fits) == nat.GDN_ERR_CUDA                       # 16 chunks x 2 MiB = 32 MiB
    over = fits.with_(n_tokens=1025)                            # 17 chunks
    assert call(over) == nat.GDN_ERR_INVALID_ARGUMENT
    assert "gdn_forward_ws" in nat.gdn_last_error()
    assert call(fits, params=fits.params()) == nat.GDN_ERR_CUDA  # auto path bits: chunked
    assert call(fits, params=fits.params(path=PATH_SCAN)) == nat.GDN_ERR_INVALID_ARGUMENT
    small = WORKLOADS["tiny"].with_(n_tokens=64)
    assert call(small) == nat.GDN_ERR_UNSUPPORTED               # D_k = 32
    assert call(fits, output=Fake(fits).addr["q"]) == nat.GDN_ERR_INVALID_ARGUMENT


@no_device
def test_two_pass_needs_aligned_v(L):
    w = WORKLOADS["long_prefill"].with_(n_tokens=100, n_seqs=1)
    p = w.params(path=PATH_CHUNKED)
    f = Fake(w)
    args = [f.addr[n] for n in ("q", "k", "v", "g", "beta", "state_in", "output", "state_out")]
    args[2] += 4                                             # v 4-byte aligned only
    assert nat.forward_ws_raw(*args, p, 10 * GAP, nat.gdn_workspace_size(p)) == \
        nat.GDN_ERR_INVALID_ARGUMENT
    assert "16-byte" in nat.gdn_last_error()
    assert nat.forward_chunked_noalloc_raw(*args, w.with_(n_tokens=64).params(path=PATH_CHUNKED)) == \
        nat.GDN_ERR_INVALID_ARGUMENT


@no_device
def test_chunked_path_needs_aligned_v(L):
    # the chunked path copies v rows 16 bytes at a time (one-pass form, two-pass
    # form and layer table alike); the other paths take a 4-byte-aligned v
    w = Workload("cv", 128, 128, 2, 4, 100, 1)
    f = Fake(w)
    v4 = f.addr["v"] + 4
    assert f.call(params=w.params(path=PATH_CHUNKED), v=v4) == nat.GDN_ERR_INVALID_ARGUMENT
    assert "16-byte" in nat.gdn_last_error()
    assert f.call(params=w.params(path=PATH_SCAN), v=v4) == nat.GDN_ERR_CUDA  # host checks pass
    # the automatic choice falls back to the scan for such a v (host checks pass)
    assert f.call(params=w.params(), v=v4) == nat.GDN_ERR_CUDA
    rows = _layer_rows(2)
    rows[1][2] += 4
    assert nat.forward_layers_raw(rows, w.params(path=PATH_CHUNKED)) == nat.GDN_ERR_INVALID_ARGUMENT
    assert "layer 1" in nat.gdn_last_error() and "16-byte" in nat.gdn_last_error()
    assert nat.forward_layers_raw(rows, w.params()) == nat.GDN_ERR_CUDA  # auto: the scan for every layer


@no_device
def test_two_pass_group_limit(L):
    # more than 32 value heads per key head: no workspace, the one-pass form runs
    w40 = Workload("g40", 128, 128, 1, 40, 100, 1)
    assert nat.gdn_workspace_size(w40.params(path=PATH_CHUNKED)) == 0
    w32 = Workload("g32", 128, 128, 1, 32, 100, 1)
    assert nat.gdn_workspace_size(w32.params(path=PATH_CHUNKED)) == 2 * (32 * 32768 + 98304)
    f = Fake(w40)
    args = [f.addr[n] for n in ("q", "k", "v", "g", "beta", "state_in", "output", "state_out")]
    # a NULL workspace is then fine (host checks pass; the launch fails here for want of a device)
    assert nat.forward_ws_raw(*args, w40.params(path=PATH_CHUNKED), 0, 0) == nat.GDN_ERR_CUDA
