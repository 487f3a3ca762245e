"""Parity of the CUDA path with the double-precision oracle on the five
workloads at their full sizes, every flag combination, through the C ABI.

Small workloads compare every element; at full size the oracle runs on every
head where that takes seconds (decode, capture) and on a seeded sample of
heads elsewhere (wide-GQA decode, long prefill), comparing those heads
element by element.
"""
import numpy as np
import pytest

from gpu_helpers import (SPLIT_RELL2_TOL, assert_close, assert_rel_l2, gather_heads, run_gpu, sample_heads,
                         to_dev)
from serving_gdn_decode_gb300.params import PATH_AUTO, PATH_SCAN
from serving_gdn_decode_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

FLAGS = [dict(), dict(decay_after=True), dict(khead_div=True),
         dict(decay_after=True, khead_div=True)]
FLAG_IDS = ["decay_first-mod", "decay_after-mod", "decay_first-div", "decay_after-div"]


@pytest.fixture(scope="module")
def cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from serving_gdn_decode_gb300 import build
    build.build()
    return torch


_cache = {}


def _inputs(name):
    if name not in _cache:
        _cache.clear()
        w = WORKLOADS[name]
        x = make_inputs(w, 0)
        _cache[name] = (w, x, to_dev(x))
    return _cache[name]


@pytest.mark.parametrize("flags", FLAGS, ids=FLAG_IDS)
@pytest.mark.parametrize("capture", [False, True], ids=["plain", "capture"])
def test_tiny(cuda, oracle_mod, flags, capture):
    w, x, d = _inputs("tiny")
    p = w.params(**flags)
    out, st, cap = run_gpu(w, x, p, capture=capture, dev=d)
    ro, rs, rc = oracle_mod.forward(p, **x, capture=capture)
    assert_close("output", out, ro, w.n_tokens)
    assert_close("state_out", st, rs, w.n_tokens)
    if capture:
        assert_close("state_capture", cap, rc, w.n_tokens)


@pytest.mark.parametrize("flags", FLAGS, ids=FLAG_IDS)
def test_decode_full(cuda, oracle_mod, flags):
    w, x, d = _inputs("decode")
    p = w.params(**flags)
    out, st, _ = run_gpu(w, x, p, dev=d)
    ro, rs, _ = oracle_mod.forward(p, **x)
    assert_close("output", out, ro, w.n_tokens)
    assert_close("state_out", st, rs, w.n_tokens)


def test_decode_in_place_as_benchmarked(cuda, oracle_mod):
    """The benchmark's launch: state_in == state_out (in-place update)."""
    w, x, d = _inputs("decode")
    p = w.params()
    out, st, _ = run_gpu(w, x, p, in_place=True, dev=d)
    heads = sample_heads(w, 64, seed=1)
    ro, rs, _ = oracle_mod.forward_heads(p, **x, heads=heads)
    go, gs, _ = gather_heads(w, out, st, None, heads)
    assert_close("output", go, ro, w.n_tokens)
    assert_close("state_out", gs, rs, w.n_tokens)


@pytest.mark.parametrize("flags", FLAGS, ids=FLAG_IDS)
def test_decode_wide_gqa_sampled(cuda, oracle_mod, flags):
    w, x, d = _inputs("decode_wide_gqa")
    p = w.params(**flags)
    out, st, _ = run_gpu(w, x, p, dev=d)
    heads = sample_heads(w, 96, seed=2)
    ro, rs, _ = oracle_mod.forward_heads(p, **x, heads=heads)
    go, gs, _ = gather_heads(w, out, st, None, heads)
    assert_close("output", go, ro, w.n_tokens)
    assert_close("state_out", gs, rs, w.n_tokens)


@pytest.mark.parametrize("flags", FLAGS, ids=FLAG_IDS)
def test_spec_capture_full(cuda, oracle_mod, flags):
    w, x, d = _inputs("spec_capture")
    p = w.params(**flags)
    out, st, cap = run_gpu(w, x, p, capture=True, dev=d)
    ro, rs, rc = oracle_mod.forward(p, **x, capture=True)
    assert_close("output", out, ro, w.n_tokens)
    assert_close("state_out", st, rs, w.n_tokens)
    assert_close("state_capture", cap, rc, w.n_tokens)
    # determinism contract: last capture slice is bit-identical to state_out
    np.testing.assert_array_equal(cap.reshape(w.n_seqs, w.n_tokens, -1)[:, -1].reshape(-1),
                                  st.reshape(w.n_seqs, -1).reshape(-1))


@pytest.mark.parametrize("flags", FLAGS, ids=FLAG_IDS)
@pytest.mark.parametrize("path", [PATH_AUTO, PATH_SCAN], ids=["auto", "scan"])
def test_long_prefill_sampled(cuda, oracle_mod, flags, path):
    """The automatic choice (the split-bf16 chunked form, one pass) and the
    FP32 scan forced, on sampled heads at full size."""
    w, x, d = _inputs("long_prefill")
    p = w.params(path=path, **flags)
    out, st, _ = run_gpu(w, x, p, dev=d)
    heads = sample_heads(w, 8, seed=3)
    ro, rs, _ = oracle_mod.forward_heads(p, **x, heads=heads)
    go, gs, _ = gather_heads(w, out, st, None, heads)
    assert_close("output", go, ro, w.n_tokens)
    assert_close("state_out", gs, rs, w.n_tokens)
    if path == PATH_AUTO:
        assert_rel_l2("output", go, ro, SPLIT_RELL2_TOL)
        assert_rel_l2("state_out", gs, rs, SPLIT_RELL2_TOL)
