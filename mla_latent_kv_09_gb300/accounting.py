"""Algorithmic work of one MLA decode step (what the roofline is taken on).

FLOPs follow the absorbed-MLA count of "DeepSeek V3/R1 Inference Efficiency
(2)", §2.4.1 (Compute, "MLA/MQA attention"): Q^T@K = 2*bs*s'*n_head*(c+r)
and P@V = 2*bs*s'*n_head*c, i.e. 2*128*576 + 2*128*512 = 278,528 flops per
(query token, visible cache token).

Bytes are the minimum traffic: every visible latent row (576 bf16 = 1152 B,
or a 656-byte FP8 row) read once per request (both MTP tokens share it),
plus per (request, query
token) the 128x576 bf16 query block, the 128x512 output block and the 128
fp32 LSE values, plus 4 B per block-table entry, top-k index and length
read.  Partial results of split requests, L2 re-reads and duplicated work
are implementation overhead and are not counted.
"""

from __future__ import annotations

import numpy as np

H, D_QK, D_V, PAGE = 128, 576, 512, 64
FLOPS_PER_QT = 2 * H * D_QK + 2 * H * D_V  # 278,528
ROW_BYTES = D_QK * 2
FP8_ROW_BYTES = 656  # 512 E4M3 codes, 4 scale bytes, 12 unused, 64 bf16 RoPE dims


def visible_counts(cache_lens, s_q: int, causal: bool, topk_idx=None) -> np.ndarray:
    """[B, s_q] number of cache positions each query token attends to."""
    lens = np.maximum(np.asarray(cache_lens, dtype=np.int64), 0)
    if topk_idx is not None:
        idx = np.asarray(topk_idx)
        return ((idx >= 0) & (idx < lens[:, None, None])).sum(axis=-1)
    t = np.arange(s_q)[None, :]
    n = lens[:, None] - s_q + t + 1 if causal else np.broadcast_to(lens[:, None], (lens.size, s_q))
    return np.maximum(n, 0)


def step_flops(cache_lens, s_q: int, causal: bool, topk_idx=None) -> int:
    return int(visible_counts(cache_lens, s_q, causal, topk_idx).sum()) * FLOPS_PER_QT


def step_bytes(cache_lens, s_q: int, causal: bool, topk_idx=None, out_bytes_per_elem: int = 2,
               row_bytes: int = ROW_BYTES) -> int:
    lens = np.maximum(np.asarray(cache_lens, dtype=np.int64), 0)
    B = lens.size
    if topk_idx is not None:
        idx = np.asarray(topk_idx)
        rows = 0
        for b in range(B):
            v = idx[b].reshape(-1)
            rows += np.unique(v[(v >= 0) & (v < lens[b])]).size
        table = rows  # one block-table entry looked up per gathered row
        extra = idx.size * 4
    else:
        rows = int(lens.sum())
        table = int(((lens + PAGE - 1) // PAGE).sum())
        extra = 0
    per_qt = H * D_QK * 2 + H * D_V * out_bytes_per_elem + H * 4
    return int(rows * row_bytes + B * s_q * per_qt + 4 * table + extra + 4 * B)


# Weight-absorption BMMs on either side of the attention ("DeepSeek V3/R1
# Inference Efficiency (2)", §2.4.1, Compute): the query side maps each head's
# 128 "nope" dims into the 512-dim latent space through W_UK, the output side
# maps the 512-dim head output back to 128 dims through W_UV.  T tokens are
# (request, query token) pairs.
D_NOPE = 128


def absorb_q_flops(num_tokens: int) -> int:
    return 2 * H * num_tokens * D_NOPE * D_V


def absorb_o_flops(num_tokens: int) -> int:
    return 2 * H * num_tokens * D_V * D_NOPE


def absorb_q_bytes(num_tokens: int, with_pe: bool = True) -> int:
    """q_nope in, W_UK, the 512 latent dims out (plus the 64 RoPE dims copied)."""
    pe = 2 * num_tokens * H * (D_QK - D_V) * 2 if with_pe else 0
    return num_tokens * H * D_NOPE * 2 + H * D_V * D_NOPE * 2 + num_tokens * H * D_V * 2 + pe


def absorb_o_bytes(num_tokens: int) -> int:
    """O in, W_UV, O' out."""
    return num_tokens * H * D_V * 2 + H * D_V * D_NOPE * 2 + num_tokens * H * D_NOPE * 2


# Sparse-attention indexer ("The 31-Millisecond Smoking Gun", DSA indexer):
# per visible (query token, position) one 64-head x 128-dim product with the
# index key, ReLU, a weighted head sum.  Bytes: every visible index key (256 B)
# read once per query token, the 64 x 128 bf16 index query and 64 fp32 head
# weights per query token, and the int32 list written; the fp32 scores that
# pass between the two kernels are an intermediate and not counted.
IDX_HEADS, IDX_DIM = 64, 128


def indexer_flops(cache_lens, s_q: int, causal: bool) -> int:
    n = int(visible_counts(cache_lens, s_q, causal).sum())
    return n * (2 * IDX_HEADS * IDX_DIM + 3 * IDX_HEADS)


def indexer_bytes(cache_lens, s_q: int, causal: bool, topk: int) -> int:
    n = int(visible_counts(cache_lens, s_q, causal).sum())
    B = np.asarray(cache_lens).size
    return n * IDX_DIM * 2 + B * s_q * (IDX_HEADS * IDX_DIM * 2 + IDX_HEADS * 4 + topk * 4)
