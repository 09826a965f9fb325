"""Pins for the fp64 oracle of the weight-absorption BMMs.

Definitions pinned ("DeepSeek V3/R1 Inference Efficiency (2)", §2.4.1,
Compute): Q''' = bmm(Q'', W_UK^T) maps each head's 128 query "nope" dims into
the 512-dim latent space, O' = bmm(PV, W_UV) maps the attention output of each
head back to 128 dims.  The pins check the oracle against brute-force loops,
against the identities that make absorption valid (a query absorbed through
W_UK scores a latent row exactly as the unabsorbed query scores the key
W_UK up-projects from that row; the value up-projection commutes with the
attention's weighted sum), against identity weights, and plant a transposed
weight to show the identities catch it.
"""

import json
import os

import numpy as np

import oracle
from oracle import absorb_oracle as ao
from mla_latent_kv_09_gb300 import accounting as acc

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "absorb_flops_deepseek_v3r1.json")


def _bits(rng, shape, scale=1.0):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def _f(bits):
    return oracle.bf16_bits_to_f64(bits)


def test_brute_force_loops_on_small_shapes():
    rng = np.random.default_rng(0)
    T, H, d, c = 3, 2, 5, 7
    q, wk = _bits(rng, (T, H, d)), _bits(rng, (H, c, d))
    o, wv = _bits(rng, (T, H, c)), _bits(rng, (H, c, d))
    got_q, got_o = ao.absorb_q(q, wk), ao.absorb_o(o, wv)
    qf, wkf, of, wvf = _f(q), _f(wk), _f(o), _f(wv)
    for t in range(T):
        for h in range(H):
            for ci in range(c):
                s = 0.0
                for di in range(d):
                    s += qf[t, h, di] * wkf[h, ci, di]
                assert abs(got_q[t, h, ci] - s) <= 1e-12 * (1 + abs(s))
            for di in range(d):
                s = 0.0
                for ci in range(c):
                    s += of[t, h, ci] * wvf[h, ci, di]
                assert abs(got_o[t, h, di] - s) <= 1e-12 * (1 + abs(s))


def _query_identity_holds(absorb, q, wk, latent):
    # unabsorbed: key head = W_UK[h] @ latent row, scored by the nope query;
    # absorbed: the latent row scored by the absorbed query
    qf, wkf, lf = _f(q), _f(wk), _f(latent)
    keys = np.einsum("hcd,jc->jhd", wkf, lf)             # [rows, H, d]
    direct = np.einsum("thd,jhd->thj", qf, keys)          # [T, H, rows]
    absorbed = np.einsum("thc,jc->thj", absorb(q, wk), lf)
    return np.allclose(direct, absorbed, rtol=1e-10, atol=1e-9)


def test_absorbed_query_scores_latent_rows_like_the_up_projected_keys():
    rng = np.random.default_rng(1)
    q = _bits(rng, (4, 3, ao.D_NOPE))
    wk = _bits(rng, (3, ao.D_LATENT, ao.D_NOPE), 0.05)
    latent = _bits(rng, (6, ao.D_LATENT))
    assert _query_identity_holds(ao.absorb_q, q, wk, latent)


def test_value_projection_commutes_with_the_weighted_sum():
    # the attention output is O = sum_j p_j latent_j; projecting every latent
    # row's value head W_UV[h]^T latent_j first and then taking the same
    # weighted sum must agree with projecting O once (up to O's bf16 rounding,
    # at most 2^-9 relative per element, bounded through |O| @ |W_UV|)
    rng = np.random.default_rng(2)
    H, rows = 3, 9
    latent = _f(_bits(rng, (rows, ao.D_LATENT)))
    p = rng.random((2, H, rows))
    p /= p.sum(axis=-1, keepdims=True)
    o = np.einsum("thj,jc->thc", p, latent)
    o_bits = oracle.f64_to_bf16_bits(o)
    wv = _bits(rng, (H, ao.D_LATENT, ao.D_NOPE), 0.05)
    per_row = np.einsum("hcd,jc->jhd", _f(wv), latent)
    expect = np.einsum("thj,jhd->thd", p, per_row)
    bound = 2.0 ** -9 * np.einsum("thc,hcd->thd", np.abs(o), np.abs(_f(wv))) + 1e-12
    got = ao.absorb_o(o_bits, wv)
    assert (np.abs(got - expect) <= bound).all()
    # a value weight used as its transpose's slice (wrong head) breaks it
    assert not (np.abs(ao.absorb_o(o_bits, wv[::-1].copy()) - expect) <= bound).all()


def test_identity_weights_copy_the_inputs():
    rng = np.random.default_rng(3)
    T, H = 2, 4
    q = _bits(rng, (T, H, ao.D_NOPE))
    eye_k = np.zeros((H, ao.D_LATENT, ao.D_NOPE), np.uint16)
    eye_k[:, np.arange(ao.D_NOPE), np.arange(ao.D_NOPE)] = 0x3F80  # 1.0
    out = ao.absorb_q(q, eye_k)
    assert np.array_equal(out[:, :, :ao.D_NOPE], _f(q)) and not out[:, :, ao.D_NOPE:].any()
    o = _bits(rng, (T, H, ao.D_LATENT))
    eye_v = np.zeros((H, ao.D_LATENT, ao.D_NOPE), np.uint16)
    eye_v[:, np.arange(ao.D_NOPE), np.arange(ao.D_NOPE)] = 0x3F80
    assert np.array_equal(ao.absorb_o(o, eye_v), _f(o)[:, :, :ao.D_NOPE])


def test_a_transposed_weight_is_caught():
    # planted mistake: W_UK read as [H, d, c] instead of [H, c, d] (square dims
    # so that the wrong contraction still runs)
    rng = np.random.default_rng(4)
    n = 16
    q, wk, latent = _bits(rng, (2, 2, n)), _bits(rng, (2, n, n)), _bits(rng, (5, n))
    wrong = lambda a, w: np.einsum("thd,hdc->thc", _f(a), _f(w))  # noqa: E731
    assert _query_identity_holds(ao.absorb_q, q, wk, latent)
    assert not _query_identity_holds(wrong, q, wk, latent)


def test_flops_reproduce_the_pages_worked_example():
    g = json.load(open(GOLDEN))
    bs = g["bs"]
    assert round(acc.absorb_q_flops(bs) / 1e9, 2) == g["absorb_q_gflops"]
    assert round(acc.absorb_o_flops(bs) / 1e9, 1) == g["absorb_o_gflops"]
