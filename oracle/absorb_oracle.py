"""fp64 reference for the weight-absorption BMMs on either side of MLA decode.

TEST INFRASTRUCTURE.  Only tests, the smoke check and the benchmark's
CPU-baseline leg may use it; it shares no code with the GPU path.  Every step
is the page's bmm written out in float64 with a library batched matmul
(numpy.matmul over the head axis), no blocking or reordering.

What it computes ("DeepSeek V3/R1 Inference Efficiency (2): Reverse-
Engineering the Production Deployment", §2.4.1, Compute):

  * QKV projection, Q''' = bmm(Q'', W_UK^T): bmm([128, bs, 128], [128, 128,
    512]).  With the key up-projection absorbed, each head's 128 "nope" query
    dims are mapped into the 512-dim latent space the cache rows live in:

        q_latent[t, h, c] = sum_d q_nope[t, h, d] * W_UK[h, c, d]

    W_UK[h] is [c = 512, d = 128] (the page's table lists it as
    [128, 512, 128]); a key head is k_nope = W_UK[h] @ latent, so
    q_nope . k_nope = q_latent . latent.
  * O projection, O' = bmm(PV, W_UV): [n_head, bs, c] @ [n_head, c, d].  The
    value up-projection is applied after the attention:

        out[t, h, d] = sum_c O[t, h, c] * W_UV[h, c, d]

Inputs are raw bf16 bit patterns (uint16), decoded exactly; outputs float64.
Tokens t index the flattened (request, query token) pairs of a decode step,
in the [T, heads, dims] layout the attention itself reads and writes.

Pins: tests/test_absorb_oracle.py (brute-force loops, the absorption
identities that motivate the BMMs, identity weights, planted transposes).
"""

from __future__ import annotations

import numpy as np

from .mla_oracle import bf16_bits_to_f64

D_NOPE = 128  # d: per-head query / value head dim
D_LATENT = 512  # c: latent dims of a cache row


def absorb_q(q_nope_bits: np.ndarray, w_uk_bits: np.ndarray) -> np.ndarray:
    """q_nope [T, H, d] (bf16 bits), W_UK [H, c, d] -> q_latent [T, H, c] (float64)."""
    q = bf16_bits_to_f64(np.asarray(q_nope_bits))
    w = bf16_bits_to_f64(np.asarray(w_uk_bits))
    if q.ndim != 3 or w.ndim != 3 or q.shape[1] != w.shape[0] or q.shape[2] != w.shape[2]:
        raise ValueError("expected q_nope [T, H, d] and W_UK [H, c, d]")
    # bmm([H, T, d], [H, d, c]) = Q'' @ W_UK^T per head, back to [T, H, c]
    return np.matmul(q.transpose(1, 0, 2), w.transpose(0, 2, 1)).transpose(1, 0, 2)


def absorb_o(o_bits: np.ndarray, w_uv_bits: np.ndarray) -> np.ndarray:
    """O [T, H, c] (bf16 bits), W_UV [H, c, d] -> O' [T, H, d] (float64)."""
    o = bf16_bits_to_f64(np.asarray(o_bits))
    w = bf16_bits_to_f64(np.asarray(w_uv_bits))
    if o.ndim != 3 or w.ndim != 3 or o.shape[1] != w.shape[0] or o.shape[2] != w.shape[1]:
        raise ValueError("expected O [T, H, c] and W_UV [H, c, d]")
    # bmm([H, T, c], [H, c, d]) per head, back to [T, H, d]
    return np.matmul(o.transpose(1, 0, 2), w).transpose(1, 0, 2)
