"""The seeded input generator: determinism and the stated structure."""

import numpy as np
import torch

import workloads as wl


def test_same_seed_same_bytes_and_other_seed_differs():
    a = wl.make_config("mtp_b64", seed=3, batch=4, length=300)
    b = wl.make_config("mtp_b64", seed=3, batch=4, length=300)
    c = wl.make_config("mtp_b64", seed=4, batch=4, length=300)
    assert torch.equal(a.q.view(torch.int16), b.q.view(torch.int16))
    assert torch.equal(a.kv.view(torch.int16), b.kv.view(torch.int16))
    assert torch.equal(a.block_table, b.block_table)
    assert not torch.equal(a.q.view(torch.int16), c.q.view(torch.int16))


def test_block_table_is_a_bijection_onto_the_pool():
    w = wl.make_config("uniform_b32", batch=8, length=700)
    t = w.block_table.numpy()
    npg = (700 + 63) // 64
    used = t[:, :npg].reshape(-1)
    assert sorted(used.tolist()) == list(range(w.num_pages))
    assert (t[:, npg:] == -1).all()


def test_mtp_lengths_and_table_tail():
    w = wl.make_config("mtp_b64", seed=0)
    L = w.cache_lens.numpy()
    assert w.s_q == 2 and w.causal and w.batch == 64
    assert L.min() >= 1 and L.max() <= 8192
    t = w.block_table.numpy()
    for b in range(w.batch):
        n = (L[b] + 63) // 64
        assert (t[b, :n] >= 0).all() and (t[b, n:] == -1).all()


def test_sparse_lists_are_sorted_distinct_and_padded():
    w = wl.make_config("sparse_b80", batch=6, length=5000)
    idx = w.topk_idx.numpy()
    assert idx.shape == (6, 1, 2048)
    for row in idx.reshape(-1, 2048):
        valid = row[row >= 0]
        pad = (row < 0).sum()
        assert 0 <= pad <= 300
        assert (row[:valid.size] >= 0).all() and (row[valid.size:] == -1).all()
        assert (np.diff(valid) > 0).all() and valid.max() < 5000


def test_spiked_rows_are_about_five_percent_and_exact_powers_of_two():
    w = wl.make_config("long_b128", batch=2, length=4096)
    base = wl.make_workload("x", [4096] * 2, seed=0)
    a = w.kv.float().view(-1, 576)
    b = base.kv.float().view(-1, 576)
    ratio_rows = (a != b).any(dim=1)
    frac = ratio_rows.float().mean().item()
    assert 0.035 < frac < 0.065
    assert torch.equal(a[ratio_rows], b[ratio_rows] * 8)


def test_single_config_identity_table():
    w = wl.make_config("single")
    assert w.block_table.tolist() == [[0, 1, 2, 3]]
    assert w.cache_lens.tolist() == [256]
    assert abs(w.softmax_scale - 1 / 192 ** 0.5) < 1e-15
