"""Pins for the fp64 oracle, independent of the oracle's own formulas.

Each test checks the oracle against something other than itself: values
computed by a different route (multiprecision brute force with no max
subtraction), closed forms, invariants that the definition of attention fixes,
and special cases that reduce to plain means.  The last group plants mistakes
in copies of the oracle and checks that the pins catch them.

Definition being pinned: "DeepSeek V3/R1 Inference Efficiency (2)", §2.4.1
(Compute, "MLA/MQA attention"): scores over c + r = 576 dims of one shared
latent row per token, values = the c = 512 latent dims of that row.
"""

import math

import mpmath
import numpy as np
import pytest

import oracle
from oracle import mla_oracle as om

SCALE = 1.0 / math.sqrt(192.0)


def _bits(rng, shape, scale=1.0):
    """Random bf16 bit patterns of N(0, scale^2) values (test-local helper)."""
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)  # truncation is fine for inputs


def _tiny_case(rng, B, s_q, H, lens, shuffle=True, extra_pages=1):
    lens = np.asarray(lens)
    npg = (lens + om.PAGE - 1) // om.PAGE
    total = int(npg.sum()) + extra_pages
    order = rng.permutation(total) if shuffle else np.arange(total)
    table = np.full((B, max(1, int(npg.max()))), -1, np.int32)
    c = 0
    for b in range(B):
        table[b, :npg[b]] = order[c:c + npg[b]]
        c += npg[b]
    q = _bits(rng, (B, s_q, H, om.D_QK))
    kv = _bits(rng, (total, om.PAGE, om.D_QK))
    return q, kv, table, lens.astype(np.int32)


# --------------------------------------------------------------------------
# bf16 conversion pins
# --------------------------------------------------------------------------

def test_bf16_decode_known_patterns():
    bits = np.array([0x3F80, 0xC049, 0x0000, 0x8000, 0x7F7F, 0x0001, 0x4000, 0x3E80],
                    dtype=np.uint16)
    want = [1.0, -3.140625, 0.0, -0.0, 3.3895313892515355e38, 2.0 ** -133, 2.0, 0.25]
    got = oracle.bf16_bits_to_f64(bits)
    assert got.tolist() == want
    assert np.signbit(got[3])


def test_bf16_round_is_nearest_ties_even():
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-30, 30, 4000),
                        [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 1e-40]])
    bits = oracle.f64_to_bf16_bits(x)
    r = oracle.bf16_bits_to_f64(bits)
    up = oracle.bf16_bits_to_f64((bits.astype(np.int64) + 1).astype(np.uint16))
    dn = oracle.bf16_bits_to_f64(np.where(bits & 0x7FFF, bits.astype(np.int64) - 1,
                                          bits).astype(np.uint16))
    err = np.abs(x - r)
    assert np.all(err <= np.abs(x - up)) and np.all(err <= np.abs(x - dn))
    # exact ties go to the even significand
    assert oracle.f64_to_bf16_bits(np.array([1.0 + 2 ** -8]))[0] == 0x3F80
    assert oracle.f64_to_bf16_bits(np.array([1.0 + 3 * 2 ** -8]))[0] == 0x3F82


# --------------------------------------------------------------------------
# brute force by another route: multiprecision, no max subtraction
# --------------------------------------------------------------------------

def _mp_attention(q_row_bits, kv_rows_bits, scale):
    mpmath.mp.dps = 40
    sig = mpmath.mpf(float(np.float32(scale)))
    qv = [mpmath.mpf(float(v)) for v in oracle.bf16_bits_to_f64(q_row_bits)]
    rows = oracle.bf16_bits_to_f64(kv_rows_bits)
    if rows.shape[0] == 0:
        return np.zeros(om.D_V), -math.inf
    ex = []
    for r in rows:
        s = sig * mpmath.fsum(qv[d] * mpmath.mpf(float(r[d])) for d in range(om.D_QK))
        ex.append(mpmath.exp(s))
    z = mpmath.fsum(ex)
    o = [float(mpmath.fsum(ex[j] * mpmath.mpf(float(rows[j][d])) for j in range(len(ex))) / z)
         for d in range(om.D_V)]
    return np.array(o), float(mpmath.log(z))


@pytest.mark.parametrize("L,s_q,causal", [(1, 1, False), (3, 1, False), (65, 1, False),
                                          (66, 2, True), (2, 2, True)])
def test_oracle_matches_multiprecision_brute_force(L, s_q, causal):
    rng = np.random.default_rng(100 + L)
    q, kv, table, lens = _tiny_case(rng, 1, s_q, 2, [L])
    o, lse = oracle.mla_decode(q, kv, table, lens, SCALE, causal=causal)
    pool = kv.reshape(-1, om.D_QK)
    for t in range(s_q):
        n = L - s_q + t + 1 if causal else L
        # position j of the request lives on page table[0, j // 64], slot j % 64
        rows = np.array([pool[table[0, j // 64] * 64 + j % 64] for j in range(n)]).reshape(n, -1)
        for h in range(2):
            want_o, want_lse = _mp_attention(q[0, t, h], rows, SCALE)
            np.testing.assert_allclose(o[0, t, h], want_o, rtol=1e-12, atol=1e-13)
            assert abs(lse[0, t, h] - want_lse) <= 1e-12 * max(1.0, abs(want_lse))


def test_softmax_weights_match_brute_force_and_sum_to_one():
    rng = np.random.default_rng(3)
    q = oracle.bf16_bits_to_f64(_bits(rng, (om.D_QK,)))
    rows = oracle.bf16_bits_to_f64(_bits(rng, (9, om.D_QK), scale=3.0))
    w = oracle.softmax_weights(q, rows, SCALE)
    mpmath.mp.dps = 40
    sig = mpmath.mpf(float(np.float32(SCALE)))
    ex = [mpmath.exp(sig * mpmath.fsum(mpmath.mpf(float(a)) * mpmath.mpf(float(b))
                                       for a, b in zip(q, r))) for r in rows]
    z = mpmath.fsum(ex)
    np.testing.assert_allclose(w, [float(e / z) for e in ex], rtol=1e-12)
    assert abs(w.sum() - 1.0) < 1e-14


# --------------------------------------------------------------------------
# closed forms and special cases
# --------------------------------------------------------------------------

def test_single_token_returns_its_value_row():
    rng = np.random.default_rng(11)
    q, kv, table, lens = _tiny_case(rng, 1, 1, 8, [1])
    o, lse = oracle.mla_decode(q, kv, table, lens, SCALE)
    row = oracle.bf16_bits_to_f64(kv.reshape(-1, om.D_QK)[table[0, 0] * 64])
    for h in range(8):
        assert np.array_equal(o[0, 0, h], row[:om.D_V])
        s0 = float(np.float32(SCALE)) * float(oracle.bf16_bits_to_f64(q[0, 0, h]) @ row)
        assert abs(lse[0, 0, h] - s0) < 1e-12


def test_equal_scores_give_mean_of_values():
    """Rows share the RoPE part, q lives only in the RoPE dims: all scores are
    equal, so O is the plain mean of the value rows and LSE = s + ln L."""
    rng = np.random.default_rng(12)
    L = 100
    q, kv, table, lens = _tiny_case(rng, 1, 1, 4, [L])
    q[..., :om.D_V] = 0
    pool = kv.reshape(-1, om.D_QK)
    pool[:, om.D_V:] = pool[0, om.D_V:]
    o, lse = oracle.mla_decode(q, kv, table, lens, SCALE)
    rows = np.array([pool[table[0, j // 64] * 64 + j % 64] for j in range(L)])
    vals = oracle.bf16_bits_to_f64(rows)
    mean = vals[:, :om.D_V].mean(axis=0)
    for h in range(4):
        np.testing.assert_allclose(o[0, 0, h], mean, rtol=1e-13, atol=1e-14)
        s = float(np.float32(SCALE)) * float(oracle.bf16_bits_to_f64(q[0, 0, h]) @ vals[0])
        assert abs(lse[0, 0, h] - (s + math.log(L))) < 1e-12


def test_zero_query_gives_uniform_mean_and_log_length():
    rng = np.random.default_rng(13)
    L = 77
    q, kv, table, lens = _tiny_case(rng, 1, 1, 2, [L])
    q[:] = 0
    o, lse = oracle.mla_decode(q, kv, table, lens, SCALE)
    pool = kv.reshape(-1, om.D_QK)
    rows = oracle.bf16_bits_to_f64(np.array([pool[table[0, j // 64] * 64 + j % 64]
                                             for j in range(L)]))
    np.testing.assert_allclose(o[0, 0, 0], rows[:, :om.D_V].mean(0), rtol=1e-13, atol=1e-14)
    assert abs(lse[0, 0, 1] - math.log(L)) < 1e-14


def test_all_ones_values_give_ones():
    rng = np.random.default_rng(14)
    q, kv, table, lens = _tiny_case(rng, 1, 1, 3, [130])
    kv[..., :om.D_V] = 0x3F80  # value part = 1.0, RoPE part random
    o, _ = oracle.mla_decode(q, kv, table, lens, SCALE)
    np.testing.assert_allclose(o[0, 0], 1.0, rtol=0, atol=1e-14)


def test_empty_visible_set():
    rng = np.random.default_rng(15)
    q, kv, table, lens = _tiny_case(rng, 2, 2, 2, [1, 0])
    o, lse = oracle.mla_decode(q, kv, table, lens, SCALE, causal=True)
    # request 0: token 0 sees nothing (L - 2 + 0 + 1 = 0); request 1 has no cache
    assert np.all(o[0, 0] == 0) and np.all(lse[0, 0] == -np.inf)
    assert np.all(o[1] == 0) and np.all(lse[1] == -np.inf)
    assert np.all(np.isfinite(lse[0, 1]))


def test_scale_is_taken_as_float32():
    rng = np.random.default_rng(16)
    q, kv, table, lens = _tiny_case(rng, 1, 1, 2, [5])
    a = oracle.mla_decode(q, kv, table, lens, SCALE)
    b = oracle.mla_decode(q, kv, table, lens, float(np.float32(SCALE)))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------

def test_page_permutation_is_bit_identical():
    rng = np.random.default_rng(21)
    q, kv, table, lens = _tiny_case(rng, 3, 1, 4, [200, 64, 129], shuffle=False)
    o1, l1 = oracle.mla_decode(q, kv, table, lens, SCALE)
    perm = rng.permutation(kv.shape[0])  # new page p holds old page perm[p]
    inv = np.argsort(perm)
    kv2 = kv[perm]
    table2 = np.where(table >= 0, inv[np.maximum(table, 0)], -1).astype(np.int32)
    o2, l2 = oracle.mla_decode(q, kv2, table2, lens, SCALE)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("cuts", [[1], [64], [10, 70, 71], [5, 6, 7, 8, 100]])
def test_split_then_combine_equals_unsplit(cuts):
    rng = np.random.default_rng(22)
    L = 150
    q, kv, table, lens = _tiny_case(rng, 1, 1, 5, [L])
    o, lse = oracle.mla_decode(q, kv, table, lens, SCALE)
    qh = oracle.bf16_bits_to_f64(q[0, 0])
    pos = np.arange(L)
    rows = oracle.physical_rows(table[0], pos, kv.shape[0])
    pool = oracle.bf16_bits_to_f64(kv.reshape(-1, om.D_QK))
    edges = [0] + cuts + [L]
    parts = [oracle.attend(qh, pool[rows[a:b]], SCALE) for a, b in zip(edges[:-1], edges[1:])]
    oc, lc = oracle.combine(parts)
    np.testing.assert_allclose(oc, o[0, 0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lc, lse[0, 0], rtol=1e-13)


def test_combine_ignores_empty_parts_and_handles_all_empty():
    rng = np.random.default_rng(23)
    o = rng.standard_normal((3, 512))
    lse = rng.standard_normal(3)
    empty = (np.zeros((3, 512)), np.full(3, -np.inf))
    oc, lc = oracle.combine([empty, (o, lse), empty])
    assert np.array_equal(oc, o) and np.array_equal(lc, lse)
    oe, le = oracle.combine([empty, empty])
    assert np.all(oe == 0) and np.all(le == -np.inf)


def test_two_token_causal_matches_single_token_calls():
    rng = np.random.default_rng(24)
    L = 131
    q, kv, table, lens = _tiny_case(rng, 1, 2, 3, [L])
    o2, l2 = oracle.mla_decode(q, kv, table, lens, SCALE, causal=True)
    o_last, l_last = oracle.mla_decode(q[:, 1:], kv, table, lens, SCALE)
    o_first, l_first = oracle.mla_decode(q[:, :1], kv, table, lens - 1, SCALE)
    assert np.array_equal(o2[:, 1:], o_last) and np.array_equal(l2[:, 1:], l_last)
    assert np.array_equal(o2[:, :1], o_first) and np.array_equal(l2[:, :1], l_first)


@pytest.mark.parametrize("s_q", [3, 4])
def test_multi_token_causal_matches_single_token_calls(s_q):
    # token t of an s_q-token causal step attends exactly like a one-token
    # step over the first L - s_q + t + 1 cached tokens
    rng = np.random.default_rng(40 + s_q)
    L = 66
    q, kv, table, lens = _tiny_case(rng, 1, s_q, 3, [L])
    o, l = oracle.mla_decode(q, kv, table, lens, SCALE, causal=True)
    for t in range(s_q):
        o1, l1 = oracle.mla_decode(q[:, t:t + 1], kv, table, lens - (s_q - 1 - t), SCALE)
        assert np.array_equal(o[:, t:t + 1], o1) and np.array_equal(l[:, t:t + 1], l1)


def test_sparse_full_list_equals_dense_and_is_order_free():
    rng = np.random.default_rng(25)
    L = 90
    q, kv, table, lens = _tiny_case(rng, 1, 1, 3, [L])
    od, ld = oracle.mla_decode(q, kv, table, lens, SCALE)
    idx = np.arange(L, dtype=np.int32).reshape(1, 1, L)
    os_, ls = oracle.mla_decode(q, kv, table, lens, SCALE, topk_idx=idx)
    assert np.array_equal(od, os_) and np.array_equal(ld, ls)
    shuffled = rng.permutation(L).astype(np.int32).reshape(1, 1, L)
    op, lp = oracle.mla_decode(q, kv, table, lens, SCALE, topk_idx=shuffled)
    np.testing.assert_allclose(op, od, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lp, ld, rtol=1e-13)


def test_sparse_padding_equals_trimmed_list():
    rng = np.random.default_rng(26)
    L = 300
    q, kv, table, lens = _tiny_case(rng, 1, 1, 2, [L])
    sel = np.sort(rng.choice(L, 40, replace=False)).astype(np.int32)
    padded = np.concatenate([sel, -np.ones(24, np.int32)]).reshape(1, 1, -1)
    o1, l1 = oracle.mla_decode(q, kv, table, lens, SCALE, topk_idx=padded)
    o2, l2 = oracle.mla_decode(q, kv, table, lens, SCALE, topk_idx=sel.reshape(1, 1, -1))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # the same rows, taken densely from a request whose cache holds only them
    pool = kv.reshape(-1, om.D_QK)
    rows = pool[oracle.physical_rows(table[0], sel, kv.shape[0])]
    kv3 = np.zeros((1, 64, om.D_QK), np.uint16)
    kv3[0, :40] = rows
    o3, l3 = oracle.mla_decode(q, kv3, np.zeros((1, 1), np.int32), np.array([40], np.int32), SCALE)
    np.testing.assert_allclose(o1, o3, rtol=1e-12, atol=1e-14)


def test_bad_inputs_are_rejected():
    rng = np.random.default_rng(27)
    q, kv, table, lens = _tiny_case(rng, 1, 1, 2, [10])
    with pytest.raises(ValueError):
        oracle.mla_decode(q, kv, table, lens, SCALE, topk_idx=np.array([[[10]]], np.int32))
    with pytest.raises(ValueError):
        oracle.mla_decode(q, kv, table, lens, SCALE, topk_idx=np.array([[[3, 3]]], np.int32))
    bad = table.copy()
    bad[0, 0] = kv.shape[0]
    with pytest.raises(ValueError):
        oracle.mla_decode(q, kv, bad, lens, SCALE)


def test_select_computes_only_the_requested_pairs():
    rng = np.random.default_rng(28)
    q, kv, table, lens = _tiny_case(rng, 3, 2, 2, [5, 70, 9])
    full_o, full_l = oracle.mla_decode(q, kv, table, lens, SCALE, causal=True)
    o, lse = oracle.mla_decode(q, kv, table, lens, SCALE, causal=True, select=[(1, 0), (2, 1)])
    assert np.array_equal(o[1, 0], full_o[1, 0]) and np.array_equal(lse[2, 1], full_l[2, 1])
    assert np.isnan(o[0, 0]).all() and np.isnan(lse[1, 1]).all()


# --------------------------------------------------------------------------
# planted mistakes: copies of the oracle with one plausible bug each must fail
# the multiprecision pin
# --------------------------------------------------------------------------

_ATTEND = om.attend


def _attend_no_rope(q, rows, scale):  # dropped the RoPE term of the score
    o, _ = _ATTEND(q, rows, scale)
    _, lse = _ATTEND(q[:, :512], rows[:, :512], scale)
    s = float(np.float32(scale)) * (q[:, :512] @ rows[:, :512].T)
    w = np.exp(s - s.max(1, keepdims=True))
    return (w @ rows[:, :512]) / w.sum(1, keepdims=True), lse


def _attend_value_offset(q, rows, scale):  # value taken from the wrong 512 dims
    o, lse = _ATTEND(q, rows, scale)
    if rows.shape[0]:
        s = float(np.float32(scale)) * (q @ rows.T)
        w = np.exp(s - s.max(1, keepdims=True))
        o = (w @ rows[:, 64:]) / w.sum(1, keepdims=True)
    return o, lse


def _attend_log2(q, rows, scale):  # LSE in the wrong base
    o, lse = _ATTEND(q, rows, scale)
    return o, lse / math.log(2.0)


def _attend_no_scale(q, rows, scale):  # softmax scale forgotten
    return _ATTEND(q, rows, 1.0)


@pytest.mark.parametrize("mutant", [_attend_no_rope, _attend_value_offset, _attend_log2,
                                    _attend_no_scale])
def test_planted_mistakes_are_caught(monkeypatch, mutant):
    rng = np.random.default_rng(31)
    q, kv, table, lens = _tiny_case(rng, 1, 1, 1, [3])
    monkeypatch.setattr(om, "attend", mutant)
    o, lse = om.mla_decode(q, kv, table, lens, SCALE)
    pool = kv.reshape(-1, om.D_QK)
    rows = np.array([pool[table[0, j // 64] * 64 + j % 64] for j in range(3)])
    want_o, want_lse = _mp_attention(q[0, 0, 0], rows, SCALE)
    close = np.allclose(o[0, 0, 0], want_o, rtol=1e-9) and abs(lse[0, 0, 0] - want_lse) < 1e-9
    assert not close


def test_planted_causal_off_by_one_is_caught():
    rng = np.random.default_rng(32)
    q, kv, table, lens = _tiny_case(rng, 1, 2, 1, [4])
    good = om.mla_decode(q, kv, table, lens, SCALE, causal=True)
    orig = om.visible_positions

    def shifted(L, s_q, t, causal, topk_row=None):
        return orig(L, s_q, t + 1 if causal else t, causal, topk_row)[:L]

    try:
        om.visible_positions = shifted
        bad = om.mla_decode(q, kv, table, lens, SCALE, causal=True)
    finally:
        om.visible_positions = orig
    pool = kv.reshape(-1, om.D_QK)
    rows = np.array([pool[table[0, j // 64] * 64 + j % 64] for j in range(3)])
    want_o, _ = _mp_attention(q[0, 0, 0], rows, SCALE)
    np.testing.assert_allclose(good[0][0, 0, 0], want_o, rtol=1e-12, atol=1e-13)
    assert not np.allclose(bad[0][0, 0, 0], want_o, rtol=1e-9)
