"""Parity of the CUDA decode path against the fp64 oracle (GPU required).

Tolerances (the stated acceptance bar for this operation): O max-abs <= 2e-2,
O mean-abs <= 2e-3, LSE abs <= 1e-3.  Reading of the "fp32-accumulated bf16"
output: the bar is checked on the fp32 O the kernels produce before the final
cast (MLA_FLAG_OUT_FP32 - same kernels, only the store differs) for every
workload; the production bf16 O is also checked, against the plain bar where
|O| is small, and where rows scaled x8 make |O| reach ~30 (long_b128), against
2e-2 + 2^-8 * |O_ref| (the bf16 half-ulp at that magnitude plus the bar).
"""

import numpy as np
import pytest
import torch

import mla_latent_kv_09_gb300 as m
import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _build():
    from mla_latent_kv_09_gb300 import build
    build.build()
    m.load()
    assert torch.cuda.is_available()


def run(w, out_fp32=True, num_units=0, validate=False, q=None, kv=None, table=None, topk_idx="same",
        bf16_pv=False):
    ws = m.Workspace(w.batch, w.s_q, num_units, w.q.device)
    ws.buf.fill_(0x7F)  # nothing the step leaves unwritten may pass as a result
    o, lse = m.decode_step(w.q if q is None else q, w.kv if kv is None else kv,
                           w.block_table if table is None else table, w.cache_lens, w.softmax_scale,
                           causal=w.causal, topk_idx=w.topk_idx if topk_idx == "same" else topk_idx,
                           out_fp32=out_fp32, num_units=num_units, validate=validate, bf16_pv=bf16_pv,
                           workspace=ws)
    torch.cuda.synchronize()
    assert m.mla_workspace_status(ws.buf) == m.MLA_OK  # no device wait ran out
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def reference(w, select=None):
    h = wl.host_arrays(w)
    return oracle.mla_decode(h["q_bits"], h["kv_bits"], h["block_table"], h["cache_lens"],
                             h["softmax_scale"], causal=h["causal"], topk_idx=h["topk_idx"],
                             select=select)


def assert_close(o, lse, o_ref, lse_ref, select=None, bf16_scaled=False):
    if select is not None:
        idx = tuple(np.array(select).T)
        o, lse, o_ref, lse_ref = o[idx], lse[idx], o_ref[idx], lse_ref[idx]
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse), fin), "empty rows must give LSE = -inf exactly"
    assert np.all(o[~fin] == 0), "empty rows must give O = 0"
    err = np.abs(o - o_ref)
    if bf16_scaled:
        assert np.all(err <= O_MAX + 2.0 ** -8 * np.abs(o_ref)), err.max()
    else:
        assert err.max() <= O_MAX, f"O max-abs {err.max():.3e}"
        assert err.mean() <= O_MEAN, f"O mean-abs {err.mean():.3e}"
    if fin.any():
        le = np.abs(lse[fin] - lse_ref[fin]).max()
        assert le <= LSE_MAX, f"LSE max-abs {le:.3e}"


# ---------------------------------------------------------------- workloads, small sizes (full compare)

SMALL = [
    ("single", {}),
    ("uniform_b32", dict(batch=4, length=1000)),
    ("mtp_b64", dict(batch=8, length=1000)),
    ("long_b128", dict(batch=3, length=3000)),
    ("sparse_b80", dict(batch=4, length=5000)),
]


@pytest.mark.parametrize("name,kw", SMALL, ids=[s[0] for s in SMALL])
def test_small_workloads_fp32_and_bf16(name, kw):
    w = wl.make_config(name, device="cuda", **kw)
    o_ref, lse_ref = reference(w)
    o, lse = run(w, out_fp32=True)
    assert_close(o, lse, o_ref, lse_ref)
    ob, lseb = run(w, out_fp32=False)
    assert_close(ob, lseb, o_ref, lse_ref, bf16_scaled=(name == "long_b128"))
    assert np.array_equal(lse, lseb)


# ---------------------------------------------------------------- full sizes, sampled rows

FULL = [("uniform_b32", 6), ("mtp_b64", 8), ("long_b128", 3), ("sparse_b80", 4)]


@pytest.mark.parametrize("name,nsample", FULL, ids=[f[0] for f in FULL])
def test_full_size_workloads_sampled(name, nsample):
    w = wl.make_config(name, device="cuda")
    rng = np.random.default_rng(5)
    bs = sorted(rng.choice(w.batch, nsample, replace=False).tolist())
    sel = [(b, t) for b in bs for t in range(w.s_q)]
    o, lse = run(w, out_fp32=True)
    o_ref, lse_ref = reference(w, select=sel)
    assert_close(o, lse, o_ref, lse_ref, select=sel)
    ob, lseb = run(w, out_fp32=False)
    assert_close(ob, lseb, o_ref, lse_ref, select=sel, bf16_scaled=(name == "long_b128"))


# ---------------------------------------------------------------- edge cases

@pytest.mark.parametrize("L", [1, 2, 63, 64, 65, 127, 129, 8192])
def test_lengths_around_tile_edges(L):
    w = wl.make_workload(f"len{L}", [L, 3 * L + 1], seed=L, device="cuda")
    o_ref, lse_ref = reference(w)
    o, lse = run(w)
    assert_close(o, lse, o_ref, lse_ref)


def test_one_request_split_across_many_units_matches_unsplit():
    w = wl.make_workload("long1", [8192], seed=3, device="cuda")
    o_ref, lse_ref = reference(w)
    o_many, lse_many = run(w)  # default: the request is cut across ~22 units
    o_one, lse_one = run(w, num_units=1)  # one unit: no split, no combine
    assert_close(o_many, lse_many, o_ref, lse_ref)
    assert_close(o_one, lse_one, o_ref, lse_ref)
    assert np.abs(o_many - o_one).max() <= O_MAX


def test_causal_two_tokens_with_empty_first_row():
    # L = 1: token 0 sees nothing (O = 0, LSE = -inf), token 1 sees one row
    w = wl.make_workload("c", [1, 2, 65, 130], s_q=2, causal=True, seed=9, device="cuda")
    o_ref, lse_ref = reference(w)
    o, lse = run(w)
    assert np.all(np.isneginf(lse[0, 0])) and np.all(o[0, 0] == 0)
    assert_close(o, lse, o_ref, lse_ref)


def test_zero_length_request_gives_empty_result():
    w = wl.make_workload("z", [0, 100, 0], seed=4, device="cuda")
    o, lse = run(w)
    o_ref, lse_ref = reference(w)
    assert np.all(np.isneginf(lse[0])) and np.all(o[0] == 0) and np.all(np.isneginf(lse[2]))
    assert_close(o, lse, o_ref, lse_ref)


def test_sparse_lists_with_one_entry_and_with_none():
    w = wl.make_workload("s", [3000, 3000], topk=128, seed=6, device="cuda")
    idx = w.topk_idx.clone()
    idx[0, 0, :] = -1
    idx[0, 0, 77] = 1234  # a single visible row, placed mid-list
    idx[1, 0, :] = -1  # nothing visible
    w.topk_idx = idx
    o_ref, lse_ref = reference(w)
    o, lse = run(w)
    assert np.all(np.isneginf(lse[1])) and np.all(o[1] == 0)
    assert_close(o, lse, o_ref, lse_ref)


def test_garbage_past_the_end_of_the_last_page_is_ignored():
    w = wl.make_workload("g", [70, 10], shuffle=False, seed=8, device="cuda")
    o_ref, lse_ref = reference(w)
    kv = w.kv.clone()
    flat = kv.view(-1, 576)
    nan = torch.tensor(float("nan"), dtype=torch.bfloat16, device="cuda")
    flat[70:128] = nan  # rows 70..127 of request 0's pages lie past its length
    flat[128 + 10:192] = nan
    o, lse = run(w, kv=kv)
    assert np.isfinite(o).all()
    assert_close(o, lse, o_ref, lse_ref)


# ---------------------------------------------------------------- two query tokens (paired-SM kernel)

@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
@pytest.mark.parametrize("L", [1, 2, 63, 64, 65, 127, 128, 129, 191, 255, 257])
def test_two_token_lengths_around_tile_edges(L, causal):
    # tiles are two pages: lengths that end in the first page of a tile, at a
    # page edge, one past it, and in the second page
    w = wl.make_workload(f"mtp{L}", [L, 2 * L + 3, 129], s_q=2, causal=causal, seed=L, device="cuda")
    o_ref, lse_ref = reference(w)
    o, lse = run(w)
    assert_close(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("bf16_pv", [False, True], ids=["f16pv", "bf16pv"])
def test_two_token_value_precision_modes(bf16_pv):
    w = wl.make_config("mtp_b64", device="cuda", batch=6, length=3000)
    o_ref, lse_ref = reference(w)
    o, lse = run(w, bf16_pv=bf16_pv)
    assert_close(o, lse, o_ref, lse_ref)
    ob, _ = run(w, out_fp32=False, bf16_pv=bf16_pv)
    assert_close(ob, lse, o_ref, lse_ref)


def test_two_token_full_size_bf16_pv_sampled():
    w = wl.make_config("mtp_b64", device="cuda")
    sel = [(b, t) for b in (3, 17, 40, 63) for t in range(2)]
    o, lse = run(w, bf16_pv=True)
    o_ref, lse_ref = reference(w, select=sel)
    assert_close(o, lse, o_ref, lse_ref, select=sel)


def test_two_token_peaked_softmax_default_mode_meets_the_bar():
    # 5% of the cache rows scaled x8: a few keys dominate each softmax row, so
    # the rounding of the largest weights reaches O almost unattenuated.  The
    # default (fp16 weights and values) must meet the bar on fp32 O, and the
    # bf16 O within its half-ulp at |O| ~ 30 as for the long-context workload.
    w = wl.make_workload("mtp_spiked", [6000, 3000, 129], s_q=2, causal=True, spike_frac=0.05, seed=31,
                         device="cuda")
    o_ref, lse_ref = reference(w)
    o, lse = run(w)
    assert_close(o, lse, o_ref, lse_ref)
    ob, lseb = run(w, out_fp32=False)
    assert_close(ob, lseb, o_ref, lse_ref, bf16_scaled=True)


def test_two_token_peaked_softmax_bf16_mode_stays_within_its_stated_error():
    # MLA_FLAG_BF16_PV keeps 8 significant bits on the weights: on the same
    # peaked input its O error is a few times the bar (an fp64 emulation of
    # the kernel's rounding gives max-abs 0.03-0.05, mean-abs ~1.3e-3), and
    # the partial rows of split requests are bf16 too (one more rounding of
    # those rows, <= 2^-9 relative); the LSE does not depend on the value
    # precision and still meets its bar
    w = wl.make_workload("mtp_spiked", [6000, 3000, 129], s_q=2, causal=True, spike_frac=0.05, seed=31,
                         device="cuda")
    o_ref, lse_ref = reference(w)
    o, lse = run(w, bf16_pv=True)
    err = np.abs(o - o_ref)
    assert err.max() <= 0.1 and err.mean() <= 4e-3, (err.max(), err.mean())
    fin = np.isfinite(lse_ref)
    assert np.abs(lse[fin] - lse_ref[fin]).max() <= LSE_MAX


def test_two_token_split_across_units_matches_single_unit():
    w = wl.make_workload("mtp_long", [8192, 300], s_q=2, causal=True, seed=21, device="cuda")
    o_ref, lse_ref = reference(w)
    o_many, lse_many = run(w)
    o_one, lse_one = run(w, num_units=1)
    assert_close(o_many, lse_many, o_ref, lse_ref)
    assert_close(o_one, lse_one, o_ref, lse_ref)


def test_two_token_garbage_past_the_end_is_ignored():
    # request 0 has 70 rows: its tile spans pages 0-1, rows 70..127 are past the end
    w = wl.make_workload("g2", [70, 10], s_q=2, causal=True, shuffle=False, seed=8, device="cuda")
    o_ref, lse_ref = reference(w)
    kv = w.kv.clone()
    flat = kv.view(-1, 576)
    nan = torch.tensor(float("nan"), dtype=torch.bfloat16, device="cuda")
    flat[70:128] = nan
    flat[128 + 10:192] = nan
    o, lse = run(w, kv=kv)
    assert np.isfinite(o).all()
    assert_close(o, lse, o_ref, lse_ref)


def test_two_token_sparse_uses_per_token_lists():
    w = wl.make_workload("s2", [3000, 1500], s_q=2, topk=256, seed=23, device="cuda")
    o_ref, lse_ref = reference(w)
    o, lse = run(w)
    assert_close(o, lse, o_ref, lse_ref)


def test_many_short_requests_beyond_the_plans_shared_table():
    # 5,000 requests (the plan keeps at most 4,096 in shared memory and walks
    # the rest through global memory), lengths 0..300 with empty ones;
    # sampled requests against the oracle, empty ones O = 0, LSE = -inf
    lens = np.random.default_rng(77).integers(0, 301, size=5000)
    lens[::97] = 0
    w = wl.make_workload("many", lens, seed=78, device="cuda")
    o, lse = run(w)
    sel = [(b, 0) for b in (0, 1, 97, 1234, 4095, 4096, 4097, 4999)]
    o_ref, lse_ref = reference(w, select=sel)
    assert_close(o, lse, o_ref, lse_ref, select=sel)


# ---------------------------------------------------------------- more than two query tokens (s_q = 3 .. 8)

@pytest.mark.parametrize("s_q", [3, 4, 8])
def test_multi_token_causal_lengths_around_tile_edges(s_q):
    # lengths below s_q leave the first tokens with nothing visible (O = 0,
    # LSE = -inf); the others end around page edges
    lens = [1, 2, s_q, s_q + 1, 63, 64, 65, 64 + s_q, 700]
    w = wl.make_workload(f"mtp{s_q}", lens, s_q=s_q, causal=True, seed=60 + s_q, device="cuda")
    o_ref, lse_ref = reference(w)
    o, lse = run(w)
    assert_close(o, lse, o_ref, lse_ref)
    ob, _ = run(w, out_fp32=False)
    assert_close(ob, lse, o_ref, lse_ref)


def test_multi_token_without_causal_mask():
    w = wl.make_workload("mtp3nc", [5, 129, 1000], s_q=3, causal=False, seed=70, device="cuda")
    o_ref, lse_ref = reference(w)
    o, lse = run(w)
    assert_close(o, lse, o_ref, lse_ref)


def test_multi_token_sparse_uses_per_token_lists():
    w = wl.make_workload("s4", [3000, 1500, 70], s_q=4, topk=256, pad_range=(0, 40), seed=71, device="cuda")
    o_ref, lse_ref = reference(w)
    o, lse = run(w)
    assert_close(o, lse, o_ref, lse_ref)


def test_multi_token_split_across_units_matches_single_unit():
    w = wl.make_workload("mtp4s", [4000, 37, 2500], s_q=4, causal=True, seed=72, device="cuda")
    o_ref, lse_ref = reference(w)
    o1, l1 = run(w, num_units=1)
    assert_close(o1, l1, o_ref, lse_ref)
    o2, l2 = run(w)
    assert_close(o2, l2, o_ref, lse_ref)


def test_multi_token_full_size_sampled():
    # 64 requests of U{1..8192} cached tokens, four query tokens each
    lens = np.random.default_rng(73).integers(1, 8193, size=64)
    w = wl.make_workload("mtp4_b64", lens, s_q=4, causal=True, seed=73, device="cuda", max_pages=128)
    sel = [(b, t) for b in (0, 21, 42, 63) for t in range(4)]
    o, lse = run(w)
    o_ref, lse_ref = reference(w, select=sel)
    assert_close(o, lse, o_ref, lse_ref, select=sel)


# ---------------------------------------------------------------- invariants

def test_page_permutation_gives_identical_output():
    w = wl.make_config("uniform_b32", device="cuda", batch=3, length=900)
    o1, l1 = run(w)
    perm = torch.randperm(w.num_pages, generator=torch.Generator().manual_seed(1)).cuda()
    inv = torch.argsort(perm)
    kv2 = w.kv[perm]
    t = w.block_table.long()
    table2 = torch.where(t >= 0, inv[t.clamp(min=0)], t).int()
    o2, l2 = run(w, kv=kv2, table=table2)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_repeated_calls_are_bit_identical():
    w = wl.make_config("mtp_b64", device="cuda", batch=16, length=3000)
    a = run(w)
    b = run(w)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("s_q,out_fp32", [(1, False), (1, True), (2, False)])
def test_output_aligned_to_16_bytes_only(s_q, out_fp32):
    # the caller's O need only be 16-byte aligned: the kernels then avoid
    # their 32-byte stores, with the same bits
    w = wl.make_workload("al", [700, 1500, 65], s_q=s_q, causal=s_q > 1, seed=41, device="cuda")
    o_a, l_a = run(w, out_fp32=out_fp32)
    dt = torch.float32 if out_fp32 else torch.bfloat16
    n = w.batch * s_q * 128 * 512
    shift = 16 // torch.empty((), dtype=dt).element_size()
    base = torch.empty(n + 64, dtype=dt, device="cuda")
    off = (-(base.data_ptr() // base.element_size()) % (32 // base.element_size())) + shift
    out = base[off:off + n].view(w.batch, s_q, 128, 512)
    assert out.data_ptr() % 32 == 16
    o, l = m.decode_step(w.q, w.kv, w.block_table, w.cache_lens, w.softmax_scale, causal=w.causal,
                         out_fp32=out_fp32, out=out)
    torch.cuda.synchronize()
    assert np.array_equal(o.float().cpu().numpy().astype(np.float64), o_a)
    assert np.array_equal(l.cpu().numpy().astype(np.float64), l_a)


# ---------------------------------------------------------------- split requests and their combine

@pytest.mark.parametrize("s_q,causal,length,units", [(1, False, 64 * 300, 40), (2, True, 128 * 300, 36)])
def test_a_request_split_over_more_than_32_units_is_combined(s_q, causal, length, units):
    # more than 32 splits: the combine takes the weights of splits 32.. on its
    # slow path (one lane holds one split's LSE); the short second request is whole
    w = wl.make_workload("many", [length, 500], s_q=s_q, causal=causal, seed=31, device="cuda")
    _, rm = m.mla_decode_plan_host(w.cache_lens.cpu().numpy(), s_q, 0, units)
    assert rm[0, 1] > 32
    o_ref, lse_ref = reference(w)
    for out_fp32 in (True, False):
        o, lse = run(w, num_units=units, out_fp32=out_fp32)
        assert_close(o, lse, o_ref, lse_ref, bf16_scaled=not out_fp32)


@pytest.mark.parametrize("s_q,causal,topk", [(1, False, 0), (2, True, 0), (2, False, 1024)])
def test_decode_repeated_on_one_plan_gives_the_same_result(s_q, causal, topk):
    # the plan is read-only to the attention and combine kernels: a second
    # decode + combine on the same plan (no new mla_decode_plan) gives the
    # same bits
    w = wl.make_workload("rep", [5000, 2500, 700, 9000], s_q=s_q, causal=causal, topk=topk, seed=33,
                         device="cuda")
    o1, l1 = run(w)
    ws = m.Workspace(w.batch, w.s_q, 0, w.q.device)
    U = ws.num_units
    flags = (m.MLA_FLAG_CAUSAL if causal else 0) | m.MLA_FLAG_OUT_FP32
    B = w.batch
    m.mla_decode_plan(w.cache_lens, B, s_q, topk, U, ws.buf, ws.nbytes)
    for _ in range(2):
        o = torch.full((B, s_q, 128, 512), float("nan"), device="cuda")
        lse = torch.full((B, s_q, 128), float("nan"), device="cuda")
        m.mla_decode(w.q, w.kv, w.kv.shape[0], w.block_table, w.block_table.stride(0), w.cache_lens, B, s_q,
                     128, w.softmax_scale, w.topk_idx, topk, flags, U, ws.buf, ws.nbytes, o, lse)
        m.mla_combine(ws.buf, ws.nbytes, B, s_q, 128, flags, U, o, lse)
        torch.cuda.synchronize()
        assert m.mla_workspace_status(ws.buf) == m.MLA_OK
        assert np.array_equal(o.cpu().numpy(), o1) and np.array_equal(lse.cpu().numpy(), l1)


def test_two_token_page_permutation_gives_identical_output():
    w = wl.make_config("mtp_b64", device="cuda", batch=3, length=900)
    o1, l1 = run(w)
    perm = torch.randperm(w.num_pages, generator=torch.Generator().manual_seed(2)).cuda()
    inv = torch.argsort(perm)
    t = w.block_table.long()
    table2 = torch.where(t >= 0, inv[t.clamp(min=0)], t).int()
    o2, l2 = run(w, kv=w.kv[perm], table=table2)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_sparse_full_index_list_matches_dense():
    # with one unit both paths visit the same rows in the same order, so the
    # row gather must reproduce the TMA page path exactly
    w = wl.make_workload("d", [700, 1000], seed=12, device="cuda")
    od, ld = run(w, num_units=1)
    idx = torch.full((2, 1, 1024), -1, dtype=torch.int32)
    idx[0, 0, :700] = torch.arange(700)
    idx[1, 0, :1000] = torch.arange(1000)
    os_, ls = run(w, topk_idx=idx.cuda(), num_units=1)
    assert np.array_equal(od, os_) and np.array_equal(ld, ls)


# ---------------------------------------------------------------- validate mode

def test_validate_reports_bad_table_and_bad_index():
    w = wl.make_workload("v", [200, 300], seed=2, device="cuda")
    run(w, validate=True)  # clean inputs pass
    bad = w.block_table.clone()
    bad[1, 2] = w.num_pages + 5
    with pytest.raises(m.MlaError) as e:
        run(w, table=bad, validate=True)
    assert e.value.status == m.MLA_ERR_BAD_TABLE
    ws = wl.make_workload("vs", [200, 300], topk=64, seed=2, device="cuda")
    idx = ws.topk_idx.clone()
    idx[0, 0, 3] = 250  # beyond request 0's 200 tokens
    with pytest.raises(m.MlaError) as e:
        run(ws, topk_idx=idx, validate=True)
    assert e.value.status == m.MLA_ERR_BAD_INDEX


def test_validated_step_is_asynchronous_and_capturable():
    # the check, the attention and the combine are recorded in a CUDA graph
    # (no host synchronisation inside the calls); a clean replay matches the
    # unvalidated step bit for bit; after a table entry is poisoned in place,
    # a replay reports MLA_ERR_BAD_TABLE and leaves O and LSE unwritten
    w = wl.make_workload("vg", [200, 300], seed=2, device="cuda")
    dev = torch.device("cuda")
    ws = m.Workspace(2, 1, 0, dev)
    U = ws.num_units
    out = torch.empty((2, 1, 128, 512), dtype=torch.float32, device=dev)
    lse = torch.empty((2, 1, 128), dtype=torch.float32, device=dev)
    table = w.block_table.clone()
    flags = m.MLA_FLAG_VALIDATE | m.MLA_FLAG_OUT_FP32

    def step():
        st = torch.cuda.current_stream()
        m.mla_decode_plan(w.cache_lens, 2, 1, 0, U, ws.buf, ws.nbytes, st)
        m.mla_decode(w.q, w.kv, w.num_pages, table, table.stride(0), w.cache_lens, 2, 1, 128, w.softmax_scale,
                     None, 0, flags, U, ws.buf, ws.nbytes, out, lse, st)
        m.mla_combine(ws.buf, ws.nbytes, 2, 1, 128, flags, U, out, lse, st)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    out.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert m.mla_workspace_status(ws.buf) == m.MLA_OK
    o_ref, l_ref = run(w, num_units=U)
    assert np.array_equal(out.cpu().numpy(), o_ref) and np.array_equal(lse.cpu().numpy(), l_ref)
    table[1, 2] = w.num_pages + 5
    out.fill_(float("nan"))
    lse.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert m.mla_workspace_status(ws.buf) == m.MLA_ERR_BAD_TABLE
    assert torch.isnan(out).all() and torch.isnan(lse).all()


def _poke_value(kv, table, b, pos, dim, value):
    flat = kv.view(-1, 576)
    row = int(table[b, pos // 64]) * 64 + pos % 64
    flat[row, dim] = value


def test_validate_reports_value_dims_that_do_not_fit_fp16():
    w = wl.make_workload("vr", [100, 200], seed=3, device="cuda")
    # outside what the step reads or outside the value dims: no error
    kv = w.kv.clone()
    _poke_value(kv, w.block_table, 1, 150, 530, 70000.0)  # a RoPE dim (scores only)
    _poke_value(kv, w.block_table, 0, 110, 7, float("inf"))  # past request 0's 100 tokens
    run(w, kv=kv, validate=True)
    # a visible value dim beyond fp16's range, and a NaN one
    for v in (70000.0, float("nan")):
        bad = kv.clone()
        _poke_value(bad, w.block_table, 1, 150, 7, v)
        with pytest.raises(m.MlaError) as e:
            run(w, kv=bad, validate=True)
        assert e.value.status == m.MLA_ERR_VALUE_RANGE
    # the two-token path: fp16 by default (checked), bf16 on request (no limit)
    w2 = wl.make_workload("vr2", [100, 200], s_q=2, causal=True, seed=3, device="cuda")
    bad = w2.kv.clone()
    _poke_value(bad, w2.block_table, 1, 150, 7, 70000.0)
    with pytest.raises(m.MlaError) as e:
        run(w2, kv=bad, validate=True)
    assert e.value.status == m.MLA_ERR_VALUE_RANGE
    o, lse = run(w2, kv=bad, validate=True, bf16_pv=True)
    h = wl.host_arrays(w2)
    h_kv = wl.bf16_bits(bad)
    o_ref, lse_ref = oracle.mla_decode(h["q_bits"], h_kv, h["block_table"], h["cache_lens"], h["softmax_scale"],
                                       causal=True)
    # dims 0..511 are key dims too: the poked row's scores reach ~1e4 x the
    # scale, where fp32 accumulation of the 576-term product keeps ~5 digits,
    # so the LSE is compared relatively; O carries up to 70000 x a weight in
    # that dim, where the bf16 value product's relative error bound applies
    fin = np.isfinite(lse_ref)
    assert np.all(np.abs(lse[fin] - lse_ref[fin]) <= LSE_MAX + 4e-5 * np.abs(lse_ref[fin]))
    assert np.all(np.abs(o - o_ref) <= O_MAX + 2.0 ** -7 * np.abs(o_ref))


# ---------------------------------------------------------------- failure path (bounded waits)

def test_a_wait_that_runs_out_reports_timeout_and_the_context_stays_usable():
    # one CTA waits on a barrier nothing completes: the bounded wait gives up
    # (about 2 s), records MLA_ERR_TIMEOUT and the kernel returns; no fault
    ws = m.Workspace(1, 1, 0, torch.device("cuda:0"))
    m.mla_selftest_wait_timeout(ws.buf, ws.nbytes)
    assert m.mla_workspace_status(ws.buf) == m.MLA_ERR_TIMEOUT
    assert torch.cuda.is_available() and torch.zeros(4, device="cuda").sum().item() == 0.0
    w = wl.make_workload("after-timeout", [300, 41], s_q=2, causal=True, seed=5, device="cuda")
    o, lse = run(w)
    assert_close(o, lse, *reference(w))
