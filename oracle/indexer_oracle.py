"""fp64 reference for the sparse-attention indexer: token scores and top-k.

TEST INFRASTRUCTURE.  Only tests, the smoke check and the benchmark's
CPU-baseline leg may use it; it shares no code with the GPU path.

What it computes.  "The 31-Millisecond Smoking Gun" (the DeepSeek-V4-Flash
architecture paragraph and "Potential mistake: Overlooking the indexer")
describes sparse token selection (DSA): every decode step an indexer scores
each cached token of a request (a [requests, positions, 64] tensor of
scores) and attention then runs over the selected tokens only (the top-2048
lists the sparse decode consumes).  The pages name neither the score formula
nor the tie rule; the reading taken here is the published DSA "lightning
indexer" form with the [.., 64] axis as 64 index heads:

    I[b, t, j] = sum_h w[b, t, h] * ReLU(q_I[b, t, h, :] . k_I[row(b, j), :])

for the visible positions j of query token t (all j < len_b, or j <= len_b -
s_q + t with the causal mask), with index keys k_I of 128 dims cached per
token in the same pages as the latent rows (row(b, j) through the block
table), bf16 q_I and k_I, fp32 head weights w.  Selection: the k visible
positions with the largest score, ties broken by the smaller position; the
list is written in increasing position order, padded with -1 when fewer than
k positions are visible.

Pins: tests/test_indexer_oracle.py.
"""

from __future__ import annotations

import numpy as np

from .mla_oracle import PAGE, bf16_bits_to_f64

H_IDX = 64  # index heads
D_IDX = 128  # index key dims


def index_rows(block_table_row: np.ndarray, n: int) -> np.ndarray:
    """Pool rows of logical positions 0 .. n-1 through one block-table row."""
    j = np.arange(n, dtype=np.int64)
    pages = np.asarray(block_table_row, dtype=np.int64)[j // PAGE]
    if n and (pages < 0).any():
        raise ValueError("block table entry < 0 inside the cache")
    return pages * PAGE + j % PAGE


def visible_count(cache_len: int, s_q: int, t: int, causal: bool) -> int:
    n = cache_len - s_q + t + 1 if causal else cache_len
    return max(0, min(n, cache_len))


def indexer_scores(q_bits: np.ndarray, w: np.ndarray, k_bits: np.ndarray, block_table: np.ndarray,
                   cache_lens: np.ndarray, causal: bool = False) -> list:
    """Scores of every visible position.

    q_bits:  uint16 bf16 bits [B, s_q, 64, 128]
    w:       float [B, s_q, 64]
    k_bits:  uint16 bf16 bits [num_pages, 64, 128] (index keys, paged)
    Returns a list over b of float64 arrays [s_q, n_t] -- as a list of lists:
    out[b][t] is the score vector of the visible positions 0 .. n_t - 1.
    """
    q = bf16_bits_to_f64(np.asarray(q_bits))
    kv = bf16_bits_to_f64(np.asarray(k_bits)).reshape(-1, D_IDX)
    w = np.asarray(w, dtype=np.float64)
    B, s_q, H, D = q.shape
    if H != H_IDX or D != D_IDX or w.shape != (B, s_q, H):
        raise ValueError("expected q [B, s_q, 64, 128] and w [B, s_q, 64]")
    out = []
    for b in range(B):
        L = int(cache_lens[b])
        rows = index_rows(block_table[b], max(L, 0))
        keys = kv[rows]  # [L, 128]
        per_t = []
        for t in range(s_q):
            n = visible_count(L, s_q, t, causal)
            dots = keys[:n] @ q[b, t].T  # [n, 64]
            per_t.append(np.maximum(dots, 0.0) @ w[b, t])
        out.append(per_t)
    return out


def topk_select(scores: np.ndarray, k: int) -> np.ndarray:
    """The k largest entries of a score vector (ties: smaller position
    first), as increasing positions, padded with -1 to length k."""
    s = np.asarray(scores)
    n = s.shape[0]
    order = sorted(range(n), key=lambda j: (-s[j], j))  # plain definition; n is small in the pins
    chosen = np.sort(np.asarray(order[:k], dtype=np.int64))
    out = np.full(k, -1, dtype=np.int64)
    out[:chosen.size] = chosen
    return out


def topk_select_fast(scores: np.ndarray, k: int) -> np.ndarray:
    """topk_select for long vectors: a stable sort on the negated scores is
    the same (score descending, position ascending) order."""
    s = np.asarray(scores)
    order = np.argsort(-s, kind="stable")[:k]
    chosen = np.sort(order.astype(np.int64))
    out = np.full(k, -1, dtype=np.int64)
    out[:chosen.size] = chosen
    return out


def indexer_topk(q_bits, w, k_bits, block_table, cache_lens, k: int, causal: bool = False) -> np.ndarray:
    """Index lists [B, s_q, k] (int64) of the indexer's top-k per query token."""
    sc = indexer_scores(q_bits, w, k_bits, block_table, cache_lens, causal)
    B, s_q = len(sc), len(sc[0]) if sc else 0
    out = np.full((B, s_q, k), -1, dtype=np.int64)
    for b in range(B):
        for t in range(s_q):
            out[b, t] = topk_select_fast(sc[b][t], k)
    return out
