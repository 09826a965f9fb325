"""Parity of the weight-absorption BMMs (query through W_UK, output through
W_UV) against the fp64 oracle (GPU required).

Bound: both kernels multiply bf16 operands exactly, accumulate in fp32 on the
tensor cores and round the sum to bf16 once, so element by element

    |gpu - ref| <= 2^-8 |ref| + K 2^-23 sum_k |a_k b_k|

(the first term covers the final bf16 rounding with a factor 2 to spare, the
second any fp32 accumulation order over the K = 128 or 512 terms).  The RoPE
dims the query-side call passes through must be bit-exact copies.
"""

import numpy as np
import pytest
import torch

import mla_latent_kv_09_gb300 as m
import oracle
import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    from mla_latent_kv_09_gb300 import build
    build.build()
    m.load()
    assert torch.cuda.is_available()


def bits(t):
    return wl.bf16_bits(t.contiguous())


def status_word():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def assert_status_ok(status):
    assert m.mla_workspace_status(status) == m.MLA_OK


def assert_within_bound(got, ref, absref, K):
    err = np.abs(got - ref)
    bound = 2.0 ** -8 * np.abs(ref) + K * 2.0 ** -23 * absref
    bad = err > bound
    assert not bad.any(), f"{bad.sum()} elements out of bound; worst excess {(err - bound).max():.3e}"


def check_q(inp, out, tokens=None):
    """out [T, H, >=512] against the oracle (on the listed tokens only, if given)."""
    q = bits(inp.q_nope)
    w = bits(inp.w_uk)
    got = out[..., :512].float().cpu().numpy()
    if tokens is not None:
        q, got = q[tokens], got[tokens]
    ref = oracle.absorb_q(q, w)
    absref = oracle.absorb_q(q & 0x7FFF, w & 0x7FFF)
    assert_within_bound(got, ref, absref, 128)


def check_o(inp, out, tokens=None):
    o = bits(inp.o)
    w = bits(inp.w_uv)
    got = out.float().cpu().numpy()
    if tokens is not None:
        o, got = o[tokens], got[tokens]
    ref = oracle.absorb_o(o, w)
    absref = oracle.absorb_o(o & 0x7FFF, w & 0x7FFF)
    assert_within_bound(got, ref, absref, 512)


# ---------------------------------------------------------------- query side

@pytest.mark.parametrize("T", [1, 2, 37, 128, 200, 300])
def test_query_absorption_matches_the_oracle(T):
    inp = wl.make_absorb(T, seed=T, device="cuda")
    status = status_word()
    out = m.absorb_q(inp.q_nope, inp.w_uk, inp.q_pe, status=status)
    torch.cuda.synchronize()
    assert out.shape == (T, 128, 576)
    check_q(inp, out)
    assert np.array_equal(bits(out[..., 512:]), bits(inp.q_pe)), "RoPE dims must pass through unchanged"
    assert_status_ok(status)


@pytest.mark.parametrize("H,T", [(1, 130), (16, 257), (64, 5)])
def test_query_absorption_for_fewer_heads_without_rope(H, T):
    inp = wl.make_absorb(T, num_heads=H, seed=100 + H, device="cuda")
    status = status_word()
    out = m.absorb_q(inp.q_nope, inp.w_uk, status=status)
    torch.cuda.synchronize()
    assert out.shape == (T, H, 512)
    check_q(inp, out)
    assert_status_ok(status)


def test_query_absorption_writes_only_its_rows_and_dims():
    # rows 640 wide and 3 extra tokens, all preset to a sentinel: only dims
    # 0..575 of the first T tokens may change
    T, H = 150, 128
    inp = wl.make_absorb(T, seed=7, device="cuda")
    big = torch.full((T + 3, H, 640), -7.0, dtype=torch.bfloat16, device="cuda")
    before = bits(big)
    status = status_word()
    m.absorb_q(inp.q_nope, inp.w_uk, inp.q_pe, out=big[:T, :, :576], status=status)
    torch.cuda.synchronize()
    after = bits(big)
    assert np.array_equal(after[:, :, 576:], before[:, :, 576:])
    assert np.array_equal(after[T:], before[T:])
    check_q(inp, big[:T])
    assert_status_ok(status)


def test_query_absorption_at_a_prefill_sized_step_sampled():
    # 4096 tokens (32 tiles): 48 sampled tokens against the oracle, and the
    # RoPE pass-through everywhere
    T = 4096
    inp = wl.make_absorb(T, seed=11, device="cuda")
    out = m.absorb_q(inp.q_nope, inp.w_uk, inp.q_pe)
    torch.cuda.synchronize()
    tokens = np.sort(np.random.default_rng(0).choice(T, 48, replace=False))
    tokens[-1] = T - 1
    check_q(inp, out, tokens)
    assert np.array_equal(bits(out[..., 512:]), bits(inp.q_pe))


# ---------------------------------------------------------------- output side

@pytest.mark.parametrize("T", [1, 64, 128, 200, 300])
def test_output_absorption_matches_the_oracle(T):
    inp = wl.make_absorb(T, seed=50 + T, device="cuda")
    status = status_word()
    out = m.absorb_o(inp.o, inp.w_uv, status=status)
    torch.cuda.synchronize()
    assert out.shape == (T, 128, 128)
    check_o(inp, out)
    assert_status_ok(status)


@pytest.mark.parametrize("H,T", [(1, 3), (16, 129)])
def test_output_absorption_for_fewer_heads(H, T):
    inp = wl.make_absorb(T, num_heads=H, seed=200 + H, device="cuda")
    out = m.absorb_o(inp.o, inp.w_uv)
    torch.cuda.synchronize()
    check_o(inp, out)


def test_output_absorption_writes_only_its_rows_and_reads_strided_input():
    T, H = 131, 128
    inp = wl.make_absorb(T, seed=9, device="cuda")
    wide = torch.zeros((T, H, 520), dtype=torch.bfloat16, device="cuda")  # input rows 520 apart
    wide[..., :512] = inp.o
    big = torch.full((T + 2, H, 136), 3.0, dtype=torch.bfloat16, device="cuda")
    before = bits(big)
    m.absorb_o(wide[..., :512], inp.w_uv, out=big[:T, :, :128])
    torch.cuda.synchronize()
    after = bits(big)
    assert np.array_equal(after[:, :, 128:], before[:, :, 128:])
    assert np.array_equal(after[T:], before[T:])
    check_o(inp, big[:T, :, :128])


def test_output_absorption_at_a_prefill_sized_step_sampled():
    T = 4096
    inp = wl.make_absorb(T, seed=12, device="cuda")
    out = m.absorb_o(inp.o, inp.w_uv)
    torch.cuda.synchronize()
    tokens = np.sort(np.random.default_rng(1).choice(T, 48, replace=False))
    tokens[0] = 0
    check_o(inp, out, tokens)


# ---------------------------------------------------------------- the layer around the attention

def test_absorb_decode_absorb_matches_the_oracle_chain():
    # query absorption writes the attention's query in place, the attention
    # runs on it, the output absorption reads the attention's output; the
    # oracle chain rounds its intermediates to bf16 at the same two points
    w = wl.make_config("mtp_b64", seed=3, device="cuda", batch=4, length=700)
    B, s_q, H = w.batch, w.s_q, 128
    T = B * s_q
    inp = wl.make_absorb(T, seed=4, device="cuda")
    q = torch.empty((B, s_q, H, 576), dtype=torch.bfloat16, device="cuda")
    m.absorb_q(inp.q_nope, inp.w_uk, inp.q_pe, out=q.view(T, H, 576))
    o, lse = m.decode_step(q, w.kv, w.block_table, w.cache_lens, w.softmax_scale, causal=True)
    out = m.absorb_o(o.view(T, H, 512), inp.w_uv)
    torch.cuda.synchronize()

    q_lat = oracle.f64_to_bf16_bits(oracle.absorb_q(bits(inp.q_nope), bits(inp.w_uk)))
    q_bits = np.concatenate([q_lat, bits(inp.q_pe)], axis=-1).reshape(B, s_q, H, 576)
    h = wl.host_arrays(w)
    o_ref, lse_ref = oracle.mla_decode(q_bits, h["kv_bits"], h["block_table"], h["cache_lens"],
                                       h["softmax_scale"], causal=True)
    o_ref_bits = oracle.f64_to_bf16_bits(o_ref).reshape(T, H, 512)
    out_ref = oracle.absorb_o(o_ref_bits, bits(inp.w_uv))
    err = np.abs(out.float().cpu().numpy() - out_ref)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, (err.max(), err.mean())
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= 1e-3


def test_absorption_calls_replay_bit_exact_from_a_cuda_graph():
    T = 96
    inp = wl.make_absorb(T, seed=5, device="cuda")
    qo = torch.empty((T, 128, 576), dtype=torch.bfloat16, device="cuda")
    oo = torch.empty((T, 128, 128), dtype=torch.bfloat16, device="cuda")
    status = status_word()
    eager_q = m.absorb_q(inp.q_nope, inp.w_uk, inp.q_pe, status=status).clone()
    eager_o = m.absorb_o(inp.o, inp.w_uv, status=status).clone()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            m.absorb_q(inp.q_nope, inp.w_uk, inp.q_pe, out=qo, status=status, stream=s)
            m.absorb_o(inp.o, inp.w_uv, out=oo, status=status, stream=s)
    qo.zero_()
    oo.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(qo, eager_q) and torch.equal(oo, eager_o)
    assert_status_ok(status)
