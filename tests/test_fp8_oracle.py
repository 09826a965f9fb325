"""Pins of the FP8-cache oracle (oracle/fp8_oracle.py): the E4M3 and UE8M0
decodings against the encodings' definitions and torch's own float8 types,
the 656-byte row layout, and attention over an FP8 cache against the
independently pinned bf16 oracle on the same values."""

import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8_oracle as f8

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_ue8m0_values.json")


def _golden(kind):
    d = json.load(open(GOLDEN))[kind]
    codes = np.array([int(k, 16) for k in d], dtype=np.uint8)
    vals = np.array([np.nan if v == "nan" else float(v) for v in d.values()])
    return codes, vals


def test_e4m3_values_of_the_definition():
    codes, want = _golden("e4m3")
    got = f8.e4m3_to_f64(codes)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(want[ok]))  # 0x80 is -0


def test_e4m3_matches_torch_float8_on_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = f8.e4m3_to_f64(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[~np.isnan(ref)], ref[~np.isnan(ref)])


def test_e4m3_structure():
    v = f8.e4m3_to_f64(np.arange(256, dtype=np.uint8))
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)          # codes 0x00 .. 0x7E increase
    assert pos[-1] == 448.0 and pos[1] == 2.0 ** -9
    assert np.array_equal(v[0x80:0xFF], -pos)  # sign bit negates
    assert np.flatnonzero(np.isnan(v)).tolist() == [0x7F, 0xFF]


def test_ue8m0_values():
    codes, want = _golden("ue8m0")
    got = f8.ue8m0_to_f64(codes)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    assert np.array_equal(got[~np.isnan(want)], want[~np.isnan(want)])
    all_codes = np.arange(255, dtype=np.uint8)
    assert np.array_equal(f8.ue8m0_to_f64(all_codes), np.ldexp(1.0, all_codes.astype(np.int64) - 127))
    if hasattr(torch, "float8_e8m0fnu"):
        ref = torch.from_numpy(np.arange(256, dtype=np.uint8)).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
        got = f8.ue8m0_to_f64(np.arange(256, dtype=np.uint8))
        assert np.array_equal(np.isnan(got), np.isnan(ref))
        assert np.array_equal(got[~np.isnan(ref)], ref[~np.isnan(ref)])


def _row(latent_codes, scale_bytes, rope_bits):
    r = np.zeros(656, dtype=np.uint8)
    r[:512] = latent_codes
    r[512:516] = scale_bytes
    r[528:656] = np.asarray(rope_bits, dtype=np.uint16).view(np.uint8)  # little-endian host order
    return r


def test_row_layout():
    # every latent code 1.0; group g scaled by 2**g; RoPE dims 0.5, -3.0, ...
    rope = np.array([0x3F00, 0xC040] * 32, dtype=np.uint16)  # bf16 0.5, -3.0
    r = _row(np.full(512, 0x38, np.uint8), [127, 128, 129, 130], rope)
    v = f8.fp8_rows_to_f64(r)
    want = np.concatenate([np.repeat([1.0, 2.0, 4.0, 8.0], 128), np.tile([0.5, -3.0], 32)])
    assert v.shape == (576,) and np.array_equal(v, want)
    # the planted mistakes this catches: 64-dim groups, big-endian RoPE
    assert not np.array_equal(np.repeat([1.0, 2.0, 4.0, 8.0, 1.0, 2.0, 4.0, 8.0], 64), want[:512])
    assert not np.array_equal(oracle.bf16_bits_to_f64(rope.byteswap()), want[512:])


def test_padding_bytes_are_ignored():
    rng = np.random.default_rng(3)
    r = _row(rng.integers(0, 0x7F, 512).astype(np.uint8), [126, 127, 128, 129],
             rng.integers(0, 0x4000, 64).astype(np.uint16))
    r2 = r.copy()
    r2[516:528] = 0xFF
    assert np.array_equal(f8.fp8_rows_to_f64(r), f8.fp8_rows_to_f64(r2))


def _fp8_case(seed, lens, s_q=1, causal=False, topk=0, num_extra=3):
    """Random FP8 pool (finite codes, scales 2^-3 .. 2^3) and the bf16 pool
    holding exactly the same values, with q, table and lists."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens)
    npg = (lens + 63) // 64
    P = int(npg.sum()) + num_extra
    lat = rng.integers(0, 0x7F, (P, 64, 512)).astype(np.uint8)
    lat |= (rng.integers(0, 2, lat.shape) << 7).astype(np.uint8)
    lat[lat == 0xFF] = 0x7E
    sc = rng.integers(124, 131, (P, 64, 4)).astype(np.uint8)
    rope = (rng.standard_normal((P, 64, 64)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    pool = np.zeros((P, 64, 656), np.uint8)
    pool[..., :512] = lat
    pool[..., 512:516] = sc
    pool[..., 528:] = rope.view(np.uint8).reshape(P, 64, 128)
    vals = f8.fp8_rows_to_f64(pool)
    bits = oracle.f64_to_bf16_bits(vals)
    assert np.array_equal(oracle.bf16_bits_to_f64(bits), vals)  # every value is exact in bf16
    perm = rng.permutation(P)
    table = np.full((len(lens), max(1, npg.max())), -1, np.int32)
    c = 0
    for b, n in enumerate(npg):
        table[b, :n] = perm[c:c + n]
        c += n
    q = (rng.standard_normal((len(lens), s_q, 128, 576)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    idx = None
    if topk:
        idx = np.full((len(lens), s_q, topk), -1, np.int32)
        for b, L in enumerate(lens):
            for t in range(s_q):
                n = min(topk - 3, L)
                idx[b, t, :n] = np.sort(rng.choice(L, size=n, replace=False))
    return q, pool, bits, table, lens.astype(np.int32), idx


@pytest.mark.parametrize("lens,s_q,causal,topk", [([70, 1, 130], 1, False, 0), ([65, 200], 3, True, 0),
                                                  ([300, 90], 1, False, 40), ([0, 5], 1, False, 0)])
def test_fp8_attention_equals_bf16_attention_on_the_same_values(lens, s_q, causal, topk):
    q, pool, bits, table, L, idx = _fp8_case(11, lens, s_q, causal, topk)
    scale = 1.0 / np.sqrt(192.0)
    o8, l8 = f8.mla_decode_fp8(q, pool, table, L, scale, causal=causal, topk_idx=idx)
    o16, l16 = oracle.mla_decode(q, bits, table, L, scale, causal=causal, topk_idx=idx)
    assert np.array_equal(o8, o16, equal_nan=True) and np.array_equal(l8, l16, equal_nan=True)


def test_scales_change_the_result():
    q, pool, bits, table, L, _ = _fp8_case(12, [100])
    scale = 1.0 / np.sqrt(192.0)
    o1, _ = f8.mla_decode_fp8(q, pool, table, L, scale)
    p2 = pool.copy()
    p2[..., 513] += 1  # group 1 of every row doubled
    o2, _ = f8.mla_decode_fp8(q, p2, table, L, scale)
    v1 = f8.fp8_rows_to_f64(pool)
    v2 = f8.fp8_rows_to_f64(p2)
    assert np.array_equal(v2[..., 128:256], 2 * v1[..., 128:256])
    assert np.array_equal(v2[..., :128], v1[..., :128]) and np.array_equal(v2[..., 256:], v1[..., 256:])
    assert not np.allclose(o1, o2)
