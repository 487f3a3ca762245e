"""The 9-u32 parameter block and its flag bits.

Slots 0-5 and 8 follow the "Buffer bindings" section of
``gated_delta_net_decode_capture.metal`` (mlx-native 0.9.2):
``(D_k, D_v, n_k_heads, n_v_heads, n_tokens, n_seqs, 0, 0, q_scale_bits)``,
where ``q_scale_bits`` holds the f32 bits of the output scale and 0 means
"no scale" (1.0), as the "Buffer / params contract" section of
``gated_delta_net_decode.rs`` (mlx-native 0.21.1) states.

The pages always write 0 to slots 6 and 7.  This library reads slot 6 as flag
bits, with 0 selecting the pages' kernel behaviour, and keeps slot 7 reserved
(must be 0):

* bit 0 -- decay-after: the state is decayed after ``S@k`` (the recurrence in
  the module doc of ``gated_delta_net.rs``, mlx-native 0.4.0) instead of
  before it (the capture kernel's step order);
* bit 1 -- ``k_head = v_head / (n_v_heads / n_k_heads)`` (the "GQA broadcast"
  section of ``gated_delta_net.rs``) instead of ``v_head % n_k_heads`` (the
  capture kernel);
* bits 2-3 -- path choice: 0 automatic, 1 token-loop scan, 2 chunked prefill
  (split-bf16 tensor-core operands), 3 chunked prefill with TF32 operands.

This module only packs numbers; it holds none of the recurrence.
"""
from __future__ import annotations

import numpy as np

N_PARAMS = 9

FLAG_DECAY_AFTER = 0x1
FLAG_KHEAD_DIV = 0x2
PATH_AUTO = 0
PATH_SCAN = 1
PATH_CHUNKED = 2
PATH_CHUNKED_TF32 = 3
PATH_SHIFT = 2


def q_scale_bits(q_scale: float | None) -> int:
    """f32 bit pattern of ``q_scale``; None (or 1.0 requested as 'none') -> 0."""
    if q_scale is None:
        return 0
    bits = int(np.array([q_scale], dtype=np.float32).view(np.uint32)[0])
    if bits == 0:
        raise ValueError("q_scale = +0.0 cannot be encoded: bits 0 mean 'no scale' (1.0)")
    return bits


def pack_params(d_k: int, d_v: int, n_k_heads: int, n_v_heads: int, n_tokens: int,
                n_seqs: int, q_scale: float | None = None, decay_after: bool = False,
                khead_div: bool = False, path: int = PATH_AUTO) -> np.ndarray:
    """Pack the 9-u32 parameter block (the capture kernel page's params
    layout, with this library's flag bits in slot 6)."""
    flags = (FLAG_DECAY_AFTER if decay_after else 0) | (FLAG_KHEAD_DIV if khead_div else 0)
    flags |= (int(path) & 0x3) << PATH_SHIFT
    return np.array([d_k, d_v, n_k_heads, n_v_heads, n_tokens, n_seqs, flags, 0,
                     q_scale_bits(q_scale)], dtype=np.uint32)


def unpack_dims(params) -> tuple[int, int, int, int, int, int]:
    p = np.asarray(params, dtype=np.uint32).reshape(-1)
    return tuple(int(x) for x in p[:6])  # type: ignore[return-value]
