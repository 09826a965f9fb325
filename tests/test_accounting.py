"""The algorithmic work the roofline is taken on: FLOPs pinned by the worked
decode example of "DeepSeek V3/R1 Inference Efficiency (2)" (§2.4.1, MLA/MQA
attention: 47.2 + 41.9 = 89.1 GFLOP for bs = 64, s' = 5000), visible-position
counts and minimum bytes checked by hand on small cases."""

import json
import os

import numpy as np

from mla_latent_kv_09_gb300 import accounting as acc

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "decode_flops_deepseek_v3r1.json")

# per (request, query token): 128 x 576 bf16 query, 128 x 512 bf16 output, 128 fp32 LSE
PER_QT_BYTES = 128 * 576 * 2 + 128 * 512 * 2 + 128 * 4


def test_flops_reproduce_the_pages_worked_decode_example():
    g = json.load(open(GOLDEN))
    bs, s_prime = g["bs"], g["s_prime"]
    total = acc.step_flops(np.full(bs, s_prime), 1, False)
    assert round(total / 1e9, 1) == g["attention_gflops"]
    # the two terms the pages print, from the per-(token, position) split
    qk = bs * s_prime * 2 * g["n_head"] * (g["c"] + g["r"])
    pv = bs * s_prime * 2 * g["n_head"] * g["c"]
    assert round(qk / 1e9, 1) == g["qk_gflops"] and round(pv / 1e9, 1) == g["pv_gflops"]
    assert total == qk + pv


def test_visible_counts_causal_dense_and_topk():
    lens = [1, 5, 0]
    assert acc.visible_counts(lens, 2, True).tolist() == [[0, 1], [4, 5], [0, 0]]
    assert acc.visible_counts(lens, 2, False).tolist() == [[1, 1], [5, 5], [0, 0]]
    assert acc.visible_counts(lens, 1, True).tolist() == [[1], [5], [0]]
    idx = np.array([[[0, 3, -1, 7]]])  # 7 is past the 5 cached positions
    assert acc.visible_counts([5], 1, False, idx).tolist() == [[2]]


def test_bytes_by_hand():
    # one request, one page, one query token: 64 rows, one table entry, one length
    assert acc.step_bytes([64], 1, False) == 64 * 1152 + PER_QT_BYTES + 4 + 4
    # two query tokens read each cached row once
    assert acc.step_bytes([64], 2, True) == 64 * 1152 + 2 * PER_QT_BYTES + 4 + 4
    # 65 rows span two pages
    assert acc.step_bytes([65], 1, False) == 65 * 1152 + PER_QT_BYTES + 2 * 4 + 4
    # top-k: rows are the union of the tokens' valid entries; every index is read
    idx = np.array([[[0, 5, -1], [5, 9, 200]]])  # 200 is past the 100 cached positions
    rows = 3  # {0, 5, 9}
    assert acc.step_bytes([100], 2, False, idx) == rows * 1152 + 2 * PER_QT_BYTES + 4 * rows + 4 * idx.size + 4


def test_bench_workload_totals():
    import workloads as wl
    w = wl.make_config("mtp_b64", seed=0)
    lens = w.cache_lens.numpy()
    assert acc.step_flops(lens, 2, True) == 152_655_069_184
    assert acc.step_bytes(lens, 2, True) == 351_464_412
