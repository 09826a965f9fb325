"""Pins for the fp64 indexer oracle (token scores and top-k selection).

The score is I[b, t, j] = sum_h w[b, t, h] * ReLU(q_I[b, t, h] . k_I[j]) over
the visible positions (reading of "The 31-Millisecond Smoking Gun", the
DeepSeek-V4-Flash architecture paragraph and the indexer passage: 64 index
heads, scores per position, top-k lists for the sparse decode).  The pins
check it against brute-force loops, planted mistakes (ReLU after the head
sum, weights dropped, a transposed head axis, the causal offset), paging
invariance, and the selection against a sort and its tie rule.
"""

import numpy as np
import pytest

import oracle
from oracle import indexer_oracle as io


def _bits(rng, shape, scale=1.0):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def _case(rng, lens, s_q=1, pages_extra=2, shuffle=True):
    B = len(lens)
    npages = [(L + 63) // 64 for L in lens]
    total = sum(npages) + pages_extra
    perm = rng.permutation(total) if shuffle else np.arange(total)
    width = max(1, max(npages))
    table = np.full((B, width), -1, dtype=np.int32)
    c = 0
    for b, n in enumerate(npages):
        table[b, :n] = perm[c:c + n]
        c += n
    q = _bits(rng, (B, s_q, io.H_IDX, io.D_IDX))
    w = rng.standard_normal((B, s_q, io.H_IDX)).astype(np.float32)
    k = _bits(rng, (total, 64, io.D_IDX))
    return q, w, k, table, np.asarray(lens, dtype=np.int32)


def _brute(q, w, k, table, lens, causal):
    qf, kf = oracle.bf16_bits_to_f64(q), oracle.bf16_bits_to_f64(k)
    B, s_q = q.shape[:2]
    out = []
    for b in range(B):
        per_t = []
        for t in range(s_q):
            n = int(lens[b]) - s_q + t + 1 if causal else int(lens[b])
            n = max(0, min(n, int(lens[b])))
            sc = []
            for j in range(n):
                row = kf[table[b, j // 64], j % 64]
                tot = 0.0
                for h in range(io.H_IDX):
                    d = 0.0
                    for i in range(io.D_IDX):
                        d += qf[b, t, h, i] * row[i]
                    tot += float(w[b, t, h]) * max(d, 0.0)
                sc.append(tot)
            per_t.append(np.array(sc))
        out.append(per_t)
    return out


@pytest.mark.parametrize("causal", [False, True])
def test_scores_match_brute_force_across_pages(causal):
    rng = np.random.default_rng(1)
    q, w, k, table, lens = _case(rng, [3, 70], s_q=2)
    got = io.indexer_scores(q, w, k, table, lens, causal=causal)
    ref = _brute(q, w, k, table, lens, causal)
    for b in range(2):
        for t in range(2):
            assert got[b][t].shape == ref[b][t].shape
            assert np.allclose(got[b][t], ref[b][t], rtol=1e-12, atol=1e-9)


def test_planted_mistakes_are_caught():
    rng = np.random.default_rng(2)
    q, w, k, table, lens = _case(rng, [130])
    good = io.indexer_scores(q, w, k, table, lens)[0][0]
    qf = oracle.bf16_bits_to_f64(q)[0, 0]
    keys = oracle.bf16_bits_to_f64(k).reshape(-1, io.D_IDX)[io.index_rows(table[0], 130)]
    dots = keys @ qf.T
    relu_after_sum = np.maximum(dots @ w[0, 0].astype(np.float64), 0.0)
    no_weights = np.maximum(dots, 0.0).sum(axis=1)
    no_relu = dots @ w[0, 0].astype(np.float64)
    for wrong in (relu_after_sum, no_weights, no_relu):
        assert not np.allclose(good, wrong)
    assert np.allclose(good, np.maximum(dots, 0.0) @ w[0, 0].astype(np.float64))
    # causal offset: token t of s_q sees len - s_q + t + 1 positions
    assert io.visible_count(10, 2, 0, True) == 9 and io.visible_count(10, 2, 1, True) == 10
    assert io.visible_count(1, 4, 0, True) == 0 and io.visible_count(5, 4, 3, False) == 5


def test_scores_do_not_depend_on_page_placement():
    rng = np.random.default_rng(3)
    q, w, k, table, lens = _case(rng, [200], shuffle=False)
    a = io.indexer_scores(q, w, k, table, lens)[0][0]
    perm = rng.permutation(k.shape[0])
    inv = np.argsort(perm)
    b = io.indexer_scores(q, w, k[perm], np.where(table >= 0, inv[np.maximum(table, 0)], -1), lens)[0][0]
    assert np.array_equal(a, b)


def test_negative_dot_products_contribute_nothing():
    rng = np.random.default_rng(4)
    q, w, k, table, lens = _case(rng, [64])
    w[:] = 1.0
    neg_q = q ^ np.uint16(0x8000)  # flipping every sign negates every dot product
    a = io.indexer_scores(q, w, k, table, lens)[0][0]
    b = io.indexer_scores(neg_q, w, k, table, lens)[0][0]
    dots = oracle.bf16_bits_to_f64(k).reshape(-1, io.D_IDX)[io.index_rows(table[0], 64)] @ \
        oracle.bf16_bits_to_f64(q)[0, 0].T
    assert np.allclose(a + b, np.abs(dots).sum(axis=1))


def test_topk_selects_the_largest_and_lists_them_in_position_order():
    rng = np.random.default_rng(5)
    s = rng.standard_normal(1000)
    got = io.topk_select(s, 37)
    want = np.sort(np.argsort(-s)[:37])
    assert np.array_equal(got, want)
    assert np.array_equal(io.topk_select_fast(s, 37), got)


def test_topk_ties_take_the_smaller_positions_and_short_lists_pad():
    s = np.array([1.0, 3.0, 2.0, 3.0, 2.0, 2.0, 0.5])
    assert list(io.topk_select(s, 3)) == [1, 2, 3]      # 3, 3, then the first 2.0
    assert list(io.topk_select(s, 4)) == [1, 2, 3, 4]
    assert list(io.topk_select(s, 9)) == [0, 1, 2, 3, 4, 5, 6, -1, -1]
    assert list(io.topk_select(np.zeros(0), 2)) == [-1, -1]
    for k in (1, 3, 4, 6, 7, 9):
        assert np.array_equal(io.topk_select_fast(s, k), io.topk_select(s, k))
    # all equal: the first k positions
    assert list(io.topk_select(np.full(10, -2.5), 4)) == [0, 1, 2, 3]


def test_indexer_topk_feeds_the_sparse_decode_format():
    rng = np.random.default_rng(6)
    q, w, k, table, lens = _case(rng, [300, 20], s_q=2)
    lists = io.indexer_topk(q, w, k, table, lens, 32, causal=True)
    assert lists.shape == (2, 2, 32)
    for b in range(2):
        for t in range(2):
            n = io.visible_count(int(lens[b]), 2, t, True)
            row = lists[b, t]
            valid = row[row >= 0]
            assert valid.size == min(32, n) and np.all(np.diff(valid) > 0) and valid.max(initial=-1) < n
            assert np.all(row[valid.size:] == -1)
