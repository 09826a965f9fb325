"""Parity of the FP8-cache decode path (MLA_FLAG_KV_FP8) against the fp64
oracle over the same FP8 rows, with the bar of the bf16 path: O max-abs
<= 2e-2, mean-abs <= 2e-3, LSE <= 1e-3 (GPU required).  Because the rows'
power-of-two scales make every cached value exact in fp16 within its range,
the FP8 path must also agree to 1e-5 with the bf16 path on a bf16 cache
holding the same values."""

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


def run(w, kv=None, table=None, out_fp32=True, num_units=0, validate=False, bf16_pv=False):
    ws = m.Workspace(w.batch, w.s_q, num_units, w.q.device)
    ws.buf.fill_(0x7F)  # nothing the step leaves unwritten may pass as a result
    o, lse = m.decode_step(w.q, w.kv if kv is None else kv, w.block_table if table is None else table,
                           w.cache_lens, w.softmax_scale, causal=w.causal, topk_idx=w.topk_idx,
                           out_fp32=out_fp32, num_units=num_units, validate=validate, bf16_pv=bf16_pv,
                           workspace=ws)
    torch.cuda.synchronize()
    assert m.mla_workspace_status(ws.buf) == m.MLA_OK  # no device wait ran out
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def reference(w, select=None, kv=None):
    h = wl.host_arrays(w)
    pool = h["kv_fp8"] if kv is None else kv.cpu().numpy()
    return oracle.mla_decode_fp8(h["q_bits"], pool, h["block_table"], h["cache_lens"], h["softmax_scale"],
                                 causal=h["causal"], topk_idx=h["topk_idx"], select=select)


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


def bf16_copy(w):
    """The workload's FP8 pool as a bf16 pool of the same values (exact)."""
    vals = oracle.fp8_rows_to_f64(w.kv.cpu().numpy())
    bits = oracle.f64_to_bf16_bits(vals)
    assert np.array_equal(oracle.bf16_bits_to_f64(bits), vals)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(w.kv.device)


SMALL = [
    ("single_fp8", {}),
    ("uniform_b32_fp8", dict(batch=4, length=1000)),
    ("long_b128_fp8", dict(batch=3, length=3000)),
    ("sparse_b80_fp8", dict(batch=4, length=5000)),
    ("mtp4_b64_fp8", dict(batch=4, length=700)),
    ("mtp_b64_fp8", dict(batch=4, length=1500)),
]


@pytest.mark.parametrize("name,kw", SMALL, ids=[s[0] for s in SMALL])
def test_small_workloads(name, kw):
    w = wl.make_config(name, device="cuda", **kw)
    assert w.kv_fp8
    o_ref, lse_ref = reference(w)
    o, lse = run(w, out_fp32=True)
    assert_close(o, lse, o_ref, lse_ref)
    ob, lseb = run(w, out_fp32=False)
    assert_close(ob, lseb, o_ref, lse_ref, bf16_scaled=name.startswith("long"))
    assert np.array_equal(lse, lseb)


@pytest.mark.parametrize("name", ["single_fp8", "uniform_b32_fp8", "sparse_b80_fp8", "mtp4_b64_fp8"])
def test_matches_the_bf16_path_on_the_same_values(name):
    # the same cached values through the bf16 path: both value products are
    # fp16 on the same values; the FP8 path's scores take Q and K in fp16,
    # where a bf16 query dim below 2^-14 in magnitude rounds to an fp16
    # subnormal (an absolute change under 2^-25): agreement to 1e-5, where a
    # misplaced dim or scale would cost O(1)
    w = wl.make_config(name, device="cuda", batch=3, length=900)
    o8, l8 = run(w)
    o16, l16 = run(w, kv=bf16_copy(w))
    assert np.abs(o8 - o16).max() <= 1e-5 and np.abs(l8 - l16).max() <= 1e-5


FULL = [("uniform_b32_fp8", 6), ("long_b128_fp8", 3), ("sparse_b80_fp8", 4), ("mtp_b64_fp8", 4)]


@pytest.mark.parametrize("name,nsample", FULL, ids=[f[0] for f in FULL])
def test_full_size_workloads_sampled(name, nsample):
    w = wl.make_config(name, device="cuda")
    rng = np.random.default_rng(7)
    bs = sorted(rng.choice(w.batch, nsample, replace=False).tolist())
    sel = [(b, 0) for b in bs]
    o, lse = run(w)
    o_ref, lse_ref = reference(w, select=sel)
    assert_close(o, lse, o_ref, lse_ref, select=sel)


@pytest.mark.parametrize("L", [1, 2, 63, 64, 65, 129, 4000])
def test_lengths_around_tile_edges(L):
    w = wl.make_workload(f"f8len{L}", [L, 3 * L + 1], seed=L, device="cuda", kv_fp8=True)
    o_ref, lse_ref = reference(w)
    o, lse = run(w)
    assert_close(o, lse, o_ref, lse_ref)


def test_split_across_units_and_one_unit():
    w = wl.make_workload("f8long", [8192, 100, 0, 3000], seed=4, device="cuda", kv_fp8=True)
    o_ref, lse_ref = reference(w)
    for units in (0, 1, 7):
        o, lse = run(w, num_units=units)
        assert_close(o, lse, o_ref, lse_ref)


def test_page_order_does_not_matter():
    w = wl.make_workload("f8perm", [700, 300], seed=6, device="cuda", kv_fp8=True)
    o1, l1 = run(w)
    P = w.kv.shape[0]
    perm = torch.from_numpy(np.random.default_rng(1).permutation(P)).to("cuda")
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(P, device="cuda")
    kv2 = w.kv[perm].contiguous()              # page p of the new pool is old page perm[p]
    tbl = w.block_table.clone()
    ok = tbl >= 0
    tbl[ok] = inv[tbl[ok].long()].int()
    o2, l2 = run(w, kv=kv2, table=tbl)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_garbage_rows_past_the_cache_end_are_not_read():
    w = wl.make_workload("f8tail", [70, 130, 1], seed=8, device="cuda", kv_fp8=True, shuffle=False)
    kv = w.kv.clone()
    lens = w.cache_lens.cpu().numpy()
    tbl = w.block_table.cpu().numpy()
    for b, L in enumerate(lens):
        pg, r0 = tbl[b, (L - 1) // 64], L % 64
        if r0:
            kv[pg, r0:, :512] = 0x7F   # NaN codes
            kv[pg, r0:, 512:516] = 0xFF  # NaN scales
    o_ref, lse_ref = reference(w)
    o, lse = run(w, kv=kv)
    assert np.all(np.isfinite(o))
    assert_close(o, lse, o_ref, lse_ref)


def _status_of(w, kv):
    try:
        run(w, kv=kv, validate=True)
        return m.MLA_OK
    except m.MlaError as e:
        return e.status


def test_validate_flags_bad_rows():
    w = wl.make_workload("f8val", [100, 40], seed=9, device="cuda", kv_fp8=True, shuffle=False)
    assert _status_of(w, w.kv) == m.MLA_OK
    pg = int(w.block_table[0, 1])
    for patch, want in [((slice(512, 513), 0xFF), m.MLA_ERR_VALUE_RANGE),   # NaN scale
                        ((slice(7, 8), 0xFF), m.MLA_ERR_VALUE_RANGE),       # NaN code
                        ((slice(512, 516), 136), None)]:                   # large scale: depends on codes
        kv = w.kv.clone()
        kv[pg, 5, patch[0]] = patch[1]
        got = _status_of(w, kv)
        if want is None:
            v = oracle.fp8_rows_to_f64(kv[pg, 5].cpu().numpy())[:512]
            want = m.MLA_OK if np.abs(v).max() < 65536 else m.MLA_ERR_VALUE_RANGE
        assert got == want, (patch, got, want)
    kv = w.kv.clone()
    kv[pg, 5, 512:516] = 136
    kv[pg, 5, 0] = 0x7E  # 448 * 2^9 = 229376: out of the fp16 range
    assert _status_of(w, kv) == m.MLA_ERR_VALUE_RANGE


@pytest.mark.parametrize("units", [0, 1, 5])
def test_two_token_dense_runs_on_two_page_tiles(units):
    # s_q = 2 over a dense FP8 cache: the one-token kernel on the plan's
    # 128-row tiles, each split in two; lengths around the tile and page
    # edges (1, 64, 65, 128, 129, 191), causal, requests split across units
    lens = [1, 64, 65, 128, 129, 191, 3000, 6000]
    w = wl.make_workload("f8mtp", lens, s_q=2, causal=True, seed=17, device="cuda", kv_fp8=True)
    o_ref, lse_ref = reference(w)
    o, lse = run(w, num_units=units)
    assert_close(o, lse, o_ref, lse_ref)


def test_two_token_dense_with_bf16_partials():
    # MLA_FLAG_BF16_PV on this path only stores split requests' partial rows
    # in bf16 (8 significant bits, read back by the combine as bf16): the
    # bar holds with split requests
    w = wl.make_workload("f8mtpb", [5000, 3000, 700], s_q=2, causal=True, seed=19, device="cuda", kv_fp8=True)
    o_ref, lse_ref = reference(w)
    o, lse = run(w, bf16_pv=True)
    assert_close(o, lse, o_ref, lse_ref)
