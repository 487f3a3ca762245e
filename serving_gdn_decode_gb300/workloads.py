"""Seeded synthetic inputs for the Gated DeltaNet recurrence.

This module only draws random numbers in the pages' layouts; it holds none of
the recurrence, and both the CUDA path's tests and the oracle's tests take
their inputs from it.

Recipe (the same for every workload):

* numpy ``default_rng(seed)`` (PCG64), drawn in the fixed order
  q, k, v, g, beta, state_in;
* q, k ~ N(0, 1), then each (token, seq, k_head) vector of length D_k is
  divided by its Euclidean norm, computed in float64, then rounded to f32;
* v ~ N(0, 1); g ~ U[0, 0.5); beta ~ U[0, 1);
* state_in ~ N(0, sigma=0.1), or zeros for the long-prefill workload;
* output scale q_scale = 1/sqrt(D_k).

Layouts (innermost first) are those of the "Memory layouts" table of
``gated_delta_net.rs`` (mlx-native 0.4.0): q, k ``[D_k, n_k, T, S]``,
v ``[D_v, n_v, T, S]``, g, beta ``[n_v, T, S]``, state ``[D_k, D_v, n_v, S]``.
Arrays are returned flat (C order of the reversed shape).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np

from .params import pack_params


@dataclass(frozen=True)
class Workload:
    name: str
    d_k: int
    d_v: int
    n_k_heads: int
    n_v_heads: int
    n_tokens: int
    n_seqs: int
    capture: bool = False
    zero_state: bool = False

    @property
    def q_scale(self) -> float:
        return 1.0 / math.sqrt(self.d_k)

    @property
    def heads(self) -> int:
        return self.n_v_heads * self.n_seqs

    @property
    def state_elems(self) -> int:
        return self.d_k * self.d_v * self.n_v_heads * self.n_seqs

    @property
    def qk_elems(self) -> int:
        return self.d_k * self.n_k_heads * self.n_tokens * self.n_seqs

    @property
    def v_elems(self) -> int:
        return self.d_v * self.n_v_heads * self.n_tokens * self.n_seqs

    @property
    def scalar_elems(self) -> int:
        return self.n_v_heads * self.n_tokens * self.n_seqs

    @property
    def capture_elems(self) -> int:
        return self.state_elems * self.n_tokens

    def params(self, decay_after: bool = False, khead_div: bool = False, path: int = 0,
               q_scale: float | None | str = "default") -> np.ndarray:
        qs = self.q_scale if q_scale == "default" else q_scale
        return pack_params(self.d_k, self.d_v, self.n_k_heads, self.n_v_heads, self.n_tokens,
                           self.n_seqs, q_scale=qs, decay_after=decay_after,
                           khead_div=khead_div, path=path)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    def algorithmic_bytes(self, act: str = "f32") -> int:
        """Bytes the method must move once per call: every input read once,
        every output written once (q and k counted once although several value
        heads read them).  ``act="bf16"``: q, k, v and output take 2 bytes."""
        f = 4
        a = 2 if act == "bf16" else 4
        b = 2 * self.state_elems * f            # state_in read + state_out write
        b += 2 * self.qk_elems * a              # q, k
        b += 2 * self.v_elems * a               # v, output
        b += 2 * self.scalar_elems * f          # g, beta
        if self.capture:
            b += self.capture_elems * f         # state_capture write
        return b

    def flops(self) -> int:
        """7 flops per state element per token: decay 1, S@k 2, update 2, S@q 2."""
        return 7 * self.d_k * self.d_v * self.n_v_heads * self.n_seqs * self.n_tokens


WORKLOADS = {
    "tiny": Workload("tiny", 32, 32, 1, 2, 8, 1),
    "decode": Workload("decode", 128, 128, 16, 32, 1, 64),
    "decode_wide_gqa": Workload("decode_wide_gqa", 128, 128, 16, 48, 1, 256),
    "spec_capture": Workload("spec_capture", 128, 128, 16, 32, 4, 32, capture=True),
    "long_prefill": Workload("long_prefill", 128, 128, 16, 48, 4096, 4, zero_state=True),
}


def _unit_rows(rng: np.random.Generator, n_vec: int, dim: int) -> np.ndarray:
    x = rng.standard_normal((n_vec, dim), dtype=np.float32).astype(np.float64)
    x /= np.sqrt(np.sum(x * x, axis=1, keepdims=True))
    return x.astype(np.float32).reshape(-1)


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even), returned
    as float32 arrays holding exactly those values.  Finite inputs only."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def make_inputs(w: Workload, seed: int = 0, act: str = "f32") -> dict[str, np.ndarray]:
    """Draw the seeded inputs of ``w`` as flat float32 arrays.  With
    ``act="bf16"`` q, k and v are rounded to bfloat16 values (still stored as
    float32 here, so they widen exactly on either side of a comparison)."""
    if act not in ("f32", "bf16"):
        raise ValueError(f"act must be 'f32' or 'bf16', not {act!r}")
    rng = np.random.default_rng(seed)
    n_vec = w.n_k_heads * w.n_tokens * w.n_seqs
    q = _unit_rows(rng, n_vec, w.d_k)
    k = _unit_rows(rng, n_vec, w.d_k)
    v = rng.standard_normal(w.v_elems, dtype=np.float32)
    if act == "bf16":
        q, k, v = round_to_bf16(q), round_to_bf16(k), round_to_bf16(v)
    g = (rng.random(w.scalar_elems, dtype=np.float32) * np.float32(0.5)).astype(np.float32)
    beta = rng.random(w.scalar_elems, dtype=np.float32)
    if w.zero_state:
        state = np.zeros(w.state_elems, dtype=np.float32)
    else:
        state = rng.standard_normal(w.state_elems, dtype=np.float32) * np.float32(0.1)
    return {"q": q, "k": k, "v": v, "g": g, "beta": beta, "state_in": state}
