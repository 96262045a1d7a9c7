"""Oracle of the QKV projection with rotary position embedding that feeds a
decode step, in fp64.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use this module.  The CUDA library and its
binding never import it, and it shares no code with them.

What it computes.  "Understanding and Exploiting Diagonal Attention Sparsity
in Autoregressive Image Generation" (arXiv 2609.19702), section 2, "LLM-aligned
decoding behavior": every decoder layer turns the hidden state of the newest
token into a query, key and value (the QKV projection) before causal
self-attention; section 5.3, Fig. 16(b), times that projection as its own
part of each decode step.  For one layer and one decode step:

    [q | k | v] = x W^T                 x: [B, hidden], W: [3 H d, hidden]
    q, k <- RoPE(q, pos), RoPE(k, pos)   per head; v is not rotated

Readings taken where the page is silent (the models it names are
LLaMA-style decoders):

* W is stored as a linear layer's weight, [out_features, in_features], with
  the q rows of all heads first (head-major, d rows per head), then the k
  rows, then the v rows; there is no bias.
* The outputs are ordered as the decode streams are, s = b * H + h, each a
  d-vector.
* RoPE is the rotate-half form with base 10000: element j and element
  j + d/2 of a head (j < d/2) are rotated together by the angle
  pos * base^(-2 j / d).
* The position of decode token t is L_p + t (the prompt holds 0 .. L_p - 1).
"""
from __future__ import annotations

import numpy as np

MUTATIONS = ("transpose", "swap_qk", "rope_v", "rope_sign", "rope_interleaved", "rope_base", "pos_off")


def rope(u: np.ndarray, pos: float, base: float = 10000.0, mutation: str | None = None) -> np.ndarray:
    """Rotary embedding of the last axis of u (length d, even) at position
    pos: the pair (u[j], u[j + d/2]) is turned by pos * base^(-2j/d)."""
    u = np.asarray(u, dtype=np.float64)
    d = u.shape[-1]
    half = d // 2
    if mutation == "rope_base":
        base = 1000.0
    if mutation == "pos_off":
        pos = pos + 1
    theta = base ** (-2.0 * np.arange(half, dtype=np.float64) / d)
    c = np.cos(pos * theta)
    s = np.sin(pos * theta)
    if mutation == "rope_sign":
        s = -s
    if mutation == "rope_interleaved":
        a, b = u[..., 0::2], u[..., 1::2]
        out = np.empty_like(u)
        out[..., 0::2] = a * c - b * s
        out[..., 1::2] = b * c + a * s
        return out
    a, b = u[..., :half], u[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def qkv_rope(x: np.ndarray, W: np.ndarray, heads: int, head_dim: int, pos: int, base: float = 10000.0,
             mutation: str | None = None):
    """q, k, v of one decode step: each [B * heads, head_dim] fp64, stream
    s = b * heads + h."""
    x = np.asarray(x, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    B, hidden = x.shape
    HD = heads * head_dim
    assert W.shape == (3 * HD, hidden), (W.shape, (3 * HD, hidden))
    if mutation == "transpose":
        y = x @ W.reshape(hidden, 3 * HD)
    else:
        y = x @ W.T
    q = y[:, :HD].reshape(B * heads, head_dim)
    k = y[:, HD:2 * HD].reshape(B * heads, head_dim)
    v = y[:, 2 * HD:].reshape(B * heads, head_dim)
    if mutation == "swap_qk":
        q, k = k, q
    rmut = mutation if mutation in ("rope_sign", "rope_interleaved", "rope_base", "pos_off") else None
    q = rope(q, pos, base, rmut)
    k = rope(k, pos, base, rmut)
    if mutation == "rope_v":
        v = rope(v, pos, base)
    return q, k, v
