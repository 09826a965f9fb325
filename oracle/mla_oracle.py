"""fp64 reference for weight-absorbed MLA decode over a paged latent KV cache.

TEST INFRASTRUCTURE.  This module is the oracle that the CUDA path is checked
against.  Only tests, the smoke check and the benchmark's CPU-baseline /
reference legs may use it.  It is deliberately slow and plain: every step is
the textbook definition, written with numpy in float64, with no blocking,
fusion, online softmax or reordering.

What it computes
----------------
"DeepSeek V3/R1 Inference Efficiency (2): Reverse-Engineering the Production
Deployment", §2.4.1 (Compute, "MLA/MQA attention"): at decode time the
up-projection of the key is absorbed into the query, so every one of the
n_head = 128 query heads carries c + r = 512 + 64 = 576 dimensions and all
heads attend, MQA-style, to ONE shared cached latent row per token.  The score
contraction runs over c + r = 576 dims (the Q^T@K term, 2*bs*s'*n_head*(c+r)
flops) and the value is the c = 512 latent dims of the same row (the P@V term,
2*bs*s'*n_head*c flops).  The cache rows live in fixed-size pages reached
through a block table ("How DeepSeek Inference Works", table of levers:
"KV-cache layout (MLA, paging)").

For one request b, query token t and head h, with V the visible positions:

    s_j = sigma * sum_{d<576} q[b,t,h,d] * kv[row(j), d]        (j in V)
    m   = max_j s_j,   w_j = exp(s_j - m),   Z = sum_j w_j
    O[d] = sum_j w_j * kv[row(j), d] / Z                         (d < 512)
    LSE  = m + ln Z

Readings taken where the pages are silent (each is listed in the design notes):
  * sigma is the float32 value of the caller's softmax scale, widened exactly.
  * LSE is the natural log and includes sigma.
  * Causal two-token decode (MTP, "The 31-Millisecond Smoking Gun", NextN):
    cache_len counts both new tokens; token t sees positions [0, L - s_q + t].
  * An empty visible set gives O = 0 and LSE = -inf.
  * Sparse top-k ("The 31-Millisecond Smoking Gun", DSA sparse decode): the
    index list holds logical positions of the request's own sequence, -1 means
    "no entry"; causality is then carried by the list itself.

Parity pins live in tests/test_oracle.py (brute force in extended precision,
closed forms and invariants).  Every function below is pinned there.
"""

from __future__ import annotations

import numpy as np

D_QK = 576  # c + r: latent (512) + decoupled RoPE key (64)
D_V = 512  # c: the value is the latent part of the same row
PAGE = 64  # tokens per cache page


# --------------------------------------------------------------------------
# bf16 <-> fp64, by bit manipulation only
# --------------------------------------------------------------------------

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Decode raw bf16 bit patterns (uint16) to float64 exactly.

    A bf16 value is the top half of an IEEE binary32 pattern, so shifting the
    16 bits into the high half of a uint32 gives the float32 with the same
    value; widening float32 to float64 is exact.
    """
    b = np.asarray(bits)
    if b.dtype != np.uint16:
        raise TypeError("expected raw bf16 bits as uint16")
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 to bf16 (round to nearest, ties to even), return bits.

    Rounds in one step from float64 (no float32 intermediate, so no double
    rounding): with a = |x| = f * 2**e (0.5 <= f < 1), the bf16 quantum is
    2**(e - 8) for normals (8 significant bits) and 2**-133 below the normal
    range; a / quantum is split into integer and fractional parts and the
    fraction is compared against one half.  Inputs must be finite and inside
    the bf16 range, which holds for attention outputs (convex combinations of
    bf16 values).
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, e = np.frexp(a)
    quantum = np.where(e - 1 < -126, 2.0 ** -133, np.ldexp(1.0, e - 8))
    n = a / quantum  # exact: quantum is a power of two
    fl = np.floor(n)
    rem = n - fl
    up = (rem > 0.5) | ((rem == 0.5) & (np.fmod(fl, 2.0) == 1.0))
    r = (fl + up) * quantum
    f32 = r.astype(np.float32)  # exact: r has at most 8 significant bits
    if not np.all(np.isfinite(f32)):
        raise OverflowError("value outside bf16 range")
    bits = (f32.view(np.uint32) >> 16).astype(np.uint16) & np.uint16(0x7FFF)
    return np.where(np.signbit(x), bits | np.uint16(0x8000), bits).astype(np.uint16)


# --------------------------------------------------------------------------
# which cache positions a query token sees, and where they live
# --------------------------------------------------------------------------

def visible_positions(cache_len: int, s_q: int, t: int, causal: bool,
                      topk_row: np.ndarray | None = None) -> np.ndarray:
    """Logical cache positions visible to query token t of a request.

    Dense: all of [0, cache_len), or with the causal two-token reading
    [0, cache_len - s_q + t].  Sparse: the non-negative entries of the
    request's top-k list, in list order (duplicates are not allowed; an entry
    at or beyond cache_len is an error).
    """
    L = int(cache_len)
    if L < 0:
        raise ValueError("negative cache length")
    if topk_row is not None:
        idx = np.asarray(topk_row, dtype=np.int64)
        idx = idx[idx >= 0]
        if idx.size and int(idx.max()) >= L:
            raise ValueError("top-k index beyond the cache length")
        if np.unique(idx).size != idx.size:
            raise ValueError("duplicate top-k index")
        return idx
    n = L - s_q + t + 1 if causal else L
    return np.arange(max(n, 0), dtype=np.int64)


def physical_rows(block_table_row: np.ndarray, positions: np.ndarray,
                  num_pages: int) -> np.ndarray:
    """Logical position j -> pool row block_table[j // 64] * 64 + j % 64."""
    pos = np.asarray(positions, dtype=np.int64)
    pages = np.asarray(block_table_row, dtype=np.int64)[pos // PAGE]
    if pages.size and (pages.min() < 0 or pages.max() >= num_pages):
        raise ValueError("block table entry outside the page pool")
    return pages * PAGE + pos % PAGE


# --------------------------------------------------------------------------
# the attention itself
# --------------------------------------------------------------------------

def softmax_weights(q_head: np.ndarray, kv_rows: np.ndarray,
                    scale: float) -> np.ndarray:
    """w_j / Z for one head: exp(s_j - m) / sum_k exp(s_k - m)."""
    sigma = float(np.float32(scale))
    s = sigma * (np.asarray(kv_rows, np.float64) @ np.asarray(q_head, np.float64))
    if s.size == 0:
        return s
    w = np.exp(s - s.max())
    return w / w.sum()


def attend(q_heads: np.ndarray, kv_rows: np.ndarray, scale: float):
    """Attention of H query heads over n cached latent rows.

    q_heads: float64 [H, 576]; kv_rows: float64 [n, 576].
    Returns O float64 [H, 512] and LSE float64 [H].
    """
    q_heads = np.asarray(q_heads, dtype=np.float64)
    kv_rows = np.asarray(kv_rows, dtype=np.float64)
    H = q_heads.shape[0]
    if kv_rows.shape[0] == 0:
        return np.zeros((H, D_V)), np.full(H, -np.inf)
    sigma = float(np.float32(scale))
    s = sigma * (q_heads @ kv_rows.T)  # [H, n], contraction over c + r = 576
    m = s.max(axis=1)
    w = np.exp(s - m[:, None])
    z = w.sum(axis=1)
    o = (w @ kv_rows[:, :D_V]) / z[:, None]  # value = first c = 512 dims
    lse = m + np.log(z)
    return o, lse


def mla_decode(q_bits: np.ndarray, kv_bits: np.ndarray, block_table: np.ndarray,
               cache_lens: np.ndarray, softmax_scale: float, causal: bool = False,
               topk_idx: np.ndarray | None = None, select=None):
    """Oracle for one decode call.

    q_bits:      uint16 (bf16 bits) [B, s_q, H, 576]
    kv_bits:     uint16 (bf16 bits) [num_pages, 64, 576]
    block_table: int32 [B, max_pages]
    cache_lens:  int32 [B]
    topk_idx:    optional int32 [B, s_q, k]
    select:      optional iterable of (b, t) pairs; only those are computed and
                 the rest of the outputs are left as NaN.
    Returns O float64 [B, s_q, H, 512] and LSE float64 [B, s_q, H].
    """
    q_bits = np.asarray(q_bits)
    kv_bits = np.asarray(kv_bits)
    B, s_q, H, dq = q_bits.shape
    if dq != D_QK or kv_bits.shape[1:] != (PAGE, D_QK):
        raise ValueError("unexpected q or cache shape")
    num_pages = kv_bits.shape[0]
    pool = kv_bits.reshape(num_pages * PAGE, D_QK)
    o = np.full((B, s_q, H, D_V), np.nan)
    lse = np.full((B, s_q, H), np.nan)
    pairs = [(b, t) for b in range(B) for t in range(s_q)] if select is None else list(select)
    for b, t in pairs:
        row_idx = None if topk_idx is None else topk_idx[b, t]
        pos = visible_positions(int(cache_lens[b]), s_q, t, causal, row_idx)
        rows = physical_rows(block_table[b], pos, num_pages)
        kv = bf16_bits_to_f64(pool[rows])
        qh = bf16_bits_to_f64(q_bits[b, t])
        o[b, t], lse[b, t] = attend(qh, kv, softmax_scale)
    return o, lse


def combine(parts):
    """Merge attention results over disjoint position sets.

    parts: list of (O_s [..., 512], LSE_s [...]) where each O_s is normalised
    over its own subset.  LSE = ln sum_s exp(LSE_s) and
    O = sum_s exp(LSE_s - LSE) * O_s; subsets that saw nothing (LSE_s = -inf)
    carry zero weight, and if every subset is empty the result is O = 0,
    LSE = -inf.
    """
    lses = np.stack([np.asarray(p[1], np.float64) for p in parts])  # [S, ...]
    outs = np.stack([np.asarray(p[0], np.float64) for p in parts])  # [S, ..., 512]
    mx = lses.max(axis=0)
    safe = np.where(np.isfinite(mx), mx, 0.0)
    e = np.exp(lses - safe)  # exp(-inf) = 0
    tot = e.sum(axis=0)
    lse = np.where(tot > 0, safe + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
    wgt = np.where(tot > 0, e / np.where(tot > 0, tot, 1.0), 0.0)
    o = (wgt[..., None] * outs).sum(axis=0)
    return o, lse
