"""Parity of the sparse-attention indexer (scores, top-k lists) against the
fp64 oracle (GPU required).

Scores: the kernel multiplies bf16 operands exactly, accumulates each head's
128-term dot product in fp32 on the tensor cores and sums the 64 weighted
ReLU terms in fp32, so |gpu - ref| <= 2^-14 * sum_h |w_h| |q_h|.|k| (the fp32
rounding of ~200 accumulations, with a wide margin).  Top-k: a floating-point
decision, so the oracle's selection runs on the GPU's own fp32 scores and
the lists must match bit for bit; the lists are also checked against the
oracle's scores (every selected position scores at least the best rejected
one, within the score bound).
"""

import numpy as np
import pytest
import torch

import mla_latent_kv_09_gb300 as m
import oracle
import workloads as wl
from oracle import indexer_oracle as io

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    from mla_latent_kv_09_gb300 import build
    build.build()
    m.load()
    assert torch.cuda.is_available()


def bits(t):
    return wl.bf16_bits(t.contiguous())


def oracle_scores(w, ix, causal, rows=None):
    q, wt, k = bits(ix.q_idx), ix.w_idx.cpu().numpy(), bits(ix.k_cache)
    table, lens = w.block_table.cpu().numpy(), w.cache_lens.cpu().numpy()
    if rows is not None:
        q, wt, table, lens = q[rows], wt[rows], table[rows], lens[rows]
    ref = io.indexer_scores(q, wt, k, table, lens, causal=causal)
    absref = io.indexer_scores(q & 0x7FFF, np.abs(wt), k & 0x7FFF, table, lens, causal=causal)
    return ref, absref


def check_scores(got, ref, absref, rows):
    for i, b in enumerate(rows):
        for t in range(len(ref[i])):
            n = ref[i][t].shape[0]
            g = got[b, t, :n].astype(np.float64)
            bound = 2.0 ** -14 * absref[i][t] + 1e-30
            assert np.all(np.abs(g - ref[i][t]) <= bound), (b, t, np.abs(g - ref[i][t]).max())


def run(w, ix, causal=False, topk=None):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sc = m.indexer_scores(ix.q_idx, ix.w_idx, ix.k_cache, w.block_table, w.cache_lens, causal=causal, status=status)
    lists = None
    if topk:
        lists = m.topk_indices(sc, w.cache_lens, topk, causal=causal, status=status)
    torch.cuda.synchronize()
    assert m.mla_workspace_status(status) == m.MLA_OK
    return sc.cpu().numpy(), (None if lists is None else lists.cpu().numpy())


@pytest.mark.parametrize("s_q,causal", [(1, False), (2, True), (3, True)])
def test_scores_match_the_oracle(s_q, causal):
    w = wl.make_workload("idx", [1, 63, 64, 130, 1000, 2047], s_q=s_q, causal=causal, seed=80 + s_q, device="cuda")
    ix = wl.make_indexer(w, seed=5)
    got, _ = run(w, ix, causal)
    rows = list(range(w.batch))
    ref, absref = oracle_scores(w, ix, causal)
    check_scores(got, ref, absref, rows)


def test_scores_leave_positions_past_the_visible_count_untouched():
    w = wl.make_workload("idx2", [5, 200], seed=90, device="cuda", max_pages=8)
    ix = wl.make_indexer(w, seed=6)
    sc = torch.full((2, 1, 512), 7.0, dtype=torch.float32, device="cuda")
    m.indexer_scores(ix.q_idx, ix.w_idx, ix.k_cache, w.block_table, w.cache_lens, scores=sc)
    torch.cuda.synchronize()
    got = sc.cpu().numpy()
    assert np.all(got[0, 0, 5:] == 7.0) and np.all(got[1, 0, 200:] == 7.0)
    assert not np.any(got[1, 0, :200] == 7.0)


@pytest.mark.parametrize("s_q,causal", [(1, False), (2, True)])
def test_topk_matches_the_oracle_on_the_kernels_scores(s_q, causal):
    w = wl.make_workload("idxk", [3000, 40, 2048, 2049, 9000], s_q=s_q, causal=causal, seed=91, device="cuda")
    ix = wl.make_indexer(w, seed=7)
    sc, lists = run(w, ix, causal, topk=2048)
    lens = w.cache_lens.cpu().numpy()
    for b in range(w.batch):
        for t in range(s_q):
            n = io.visible_count(int(lens[b]), s_q, t, causal)
            want = io.topk_select_fast(sc[b, t, :n], 2048)
            assert np.array_equal(lists[b, t], want), (b, t)


def test_topk_ties_take_the_smaller_positions():
    # scores with many exact ties (a few distinct values, zeros of both signs)
    B, L, k = 3, 6000, 700
    lens = torch.tensor([L, 5000, 800], dtype=torch.int32, device="cuda")
    rng = np.random.default_rng(8)
    vals = rng.integers(-3, 4, size=(B, 1, L)).astype(np.float32) * 0.5
    vals[0, 0, ::7] = -0.0
    sc = torch.from_numpy(vals).cuda()
    out = m.topk_indices(sc, lens, k)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    for b in range(B):
        n = int(lens[b])
        assert np.array_equal(got[b, 0], io.topk_select_fast(vals[b, 0, :n].astype(np.float64), k)), b


def test_topk_of_short_rows_lists_every_visible_position():
    lens = torch.tensor([0, 1, 100, 2048], dtype=torch.int32, device="cuda")
    sc = torch.randn((4, 1, 2048), device="cuda")
    got = m.topk_indices(sc, lens, 2048).cpu().numpy()
    for b, n in enumerate([0, 1, 100, 2048]):
        assert np.array_equal(got[b, 0, :n], np.arange(n)) and np.all(got[b, 0, n:] == -1)


def test_indexer_at_the_sparse_workload_size_sampled():
    # 80 requests of 65536 cached tokens, top-2048: scores of two requests
    # against the oracle, every list against the oracle's selection on the
    # kernel's scores
    w = wl.make_config("sparse_b80", device="cuda")
    ix = wl.make_indexer(w, seed=9)
    sc, lists = run(w, ix, topk=2048)
    rows = [0, 79]
    ref, absref = oracle_scores(w, ix, False, rows=rows)
    check_scores(sc, ref, absref, rows)
    for b in (0, 13, 79):
        assert np.array_equal(lists[b, 0], io.topk_select_fast(sc[b, 0, :65536], 2048))
        # the selection is consistent with the exact scores too (up to the score bound)
        r, a = (ref[rows.index(b)][0], absref[rows.index(b)][0]) if b in rows else (None, None)
        if r is not None:
            sel = np.zeros(65536, bool)
            sel[lists[b, 0]] = True
            tol = 2.0 ** -13 * a.max()
            assert r[sel].min() >= r[~sel].max() - tol


def test_indexer_lists_drive_the_sparse_decode():
    # indexer -> top-k -> sparse attention, against the oracle's attention
    # over the same lists
    w = wl.make_workload("chain", [3000, 700, 5000], s_q=2, causal=True, seed=92, device="cuda")
    ix = wl.make_indexer(w, seed=10)
    _, lists = run(w, ix, True, topk=512)
    idx = torch.from_numpy(lists).cuda()
    o, lse = m.decode_step(w.q, w.kv, w.block_table, w.cache_lens, w.softmax_scale, topk_idx=idx, out_fp32=True)
    torch.cuda.synchronize()
    h = wl.host_arrays(w)
    o_ref, lse_ref = oracle.mla_decode(h["q_bits"], h["kv_bits"], h["block_table"], h["cache_lens"],
                                       h["softmax_scale"], topk_idx=lists)
    err = np.abs(o.cpu().numpy() - o_ref)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= 1e-3


def test_indexer_calls_replay_bit_exact_from_a_cuda_graph():
    w = wl.make_workload("g", [4000, 900], seed=93, device="cuda")
    ix = wl.make_indexer(w, seed=11)
    eager, lists = run(w, ix, topk=256)
    sc = torch.zeros((2, 1, w.block_table.shape[1] * 64), dtype=torch.float32, device="cuda")
    out = torch.zeros((2, 1, 256), dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            m.indexer_scores(ix.q_idx, ix.w_idx, ix.k_cache, w.block_table, w.cache_lens, scores=sc, stream=s)
            m.topk_indices(sc, w.cache_lens, 256, out=out, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), lists)
    n = w.cache_lens.cpu().numpy()
    for b in range(2):
        assert np.array_equal(sc.cpu().numpy()[b, 0, :n[b]], eager[b, 0, :n[b]])
