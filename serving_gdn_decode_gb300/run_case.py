"""Run one workload through the C ABI a few times on cuda:0 (no timing).

For profiler captures and quick checks, e.g.::

    python -m serving_gdn_decode_gb300.run_case decode --calls 3
    python -m serving_gdn_decode_gb300.run_case long_prefill --tokens 512 --path scan
    python -m serving_gdn_decode_gb300.run_case long_prefill --tokens 512 --path chunked --two-pass
    python -m serving_gdn_decode_gb300.run_case long_prefill --tokens 512 --path chunked_tf32
"""
from __future__ import annotations

import argparse

from .params import PATH_AUTO, PATH_CHUNKED, PATH_CHUNKED_TF32, PATH_SCAN
from .workloads import WORKLOADS, make_inputs

PATHS = {"auto": PATH_AUTO, "scan": PATH_SCAN, "chunked": PATH_CHUNKED, "chunked_tf32": PATH_CHUNKED_TF32}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("workload", choices=sorted(WORKLOADS))
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--path", choices=sorted(PATHS), default="auto")
    ap.add_argument("--tokens", type=int, default=None, help="override n_tokens")
    ap.add_argument("--seqs", type=int, default=None, help="override n_seqs")
    ap.add_argument("--capture", action="store_true", help="use gdn_forward_capture")
    ap.add_argument("--decay-after", action="store_true")
    ap.add_argument("--khead-div", action="store_true")
    ap.add_argument("--two-pass", action="store_true",
                    help="use gdn_forward_ws with a workspace (two-pass form on the chunked path)")
    ap.add_argument("--commit", action="store_true",
                    help="after each capture call, commit a random accepted token per sequence")
    ap.add_argument("--bf16", action="store_true", help="bf16 activations (q, k, v, output)")
    a = ap.parse_args(argv)

    import torch

    from . import _native as nat
    w = WORKLOADS[a.workload]
    if a.tokens:
        w = w.with_(n_tokens=a.tokens)
    if a.seqs:
        w = w.with_(n_seqs=a.seqs)
    capture = a.capture or w.capture
    x = make_inputs(w, 0, act="bf16" if a.bf16 else "f32")
    dev = torch.device("cuda:0")
    d = {k: torch.from_numpy(v).to(dev) for k, v in x.items()}
    if a.bf16:
        for n in ("q", "k", "v"):
            d[n] = d[n].to(torch.bfloat16)
    out = torch.empty(w.v_elems, dtype=torch.bfloat16 if a.bf16 else torch.float32, device=dev)
    st = torch.empty(w.state_elems, dtype=torch.float32, device=dev)
    cap = torch.empty(w.capture_elems, dtype=torch.float32, device=dev) if capture else None
    p = w.params(decay_after=a.decay_after, khead_div=a.khead_div, path=PATHS[a.path])
    if a.commit:
        import numpy as np
        capture = True
        cap = torch.empty(w.capture_elems, dtype=torch.float32, device=dev)
        idx = torch.from_numpy(np.random.default_rng(0).integers(0, w.n_tokens, w.n_seqs)
                               .astype(np.int32)).to(dev)
    ws = None
    if a.two_pass:
        ws = torch.empty(max(16, nat.gdn_workspace_size(p)), dtype=torch.uint8, device=dev)
    for _ in range(a.calls):
        if ws is not None:
            nat.gdn_forward_ws(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state_in"], out, st, p, ws)
        elif capture:
            nat.gdn_forward_capture(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state_in"], out,
                                    st, p, cap)
            if a.commit:
                nat.gdn_commit_capture(cap, idx, st, p)
        else:
            nat.gdn_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state_in"], out, st, p)
    torch.cuda.synchronize()
    print(f"{w.name}: {nat.gdn_path_name(p, capture)} x{a.calls} ok "
          f"({w.algorithmic_bytes() / 1e6:.1f} MB algorithmic per call)")


if __name__ == "__main__":
    main()
