"""fp64 reference for MLA decode over an FP8 latent cache.

TEST INFRASTRUCTURE.  Like the rest of this package, only tests, the smoke
check and the benchmark's CPU-baseline / reference legs may use it.

What it computes
----------------
"The 31-Millisecond Smoking Gun" (the DeepSeek-V4-Flash architecture
paragraph) caches the MLA latent in FP8, and "How DeepSeek Inference Works"
(levers table, the "Precision" row) names FP8 as the lever that shrinks the
KV cache.  The pages give no byte format.  The reading used here (listed with
the other readings in the design notes):

  * one cached token is a 656-byte row:
      bytes [0, 512)    the 512 latent dims, OCP FP8 E4M3 (1 sign bit, 4
                        exponent bits with bias 7, 3 mantissa bits; exponent
                        0 is subnormal; S.1111.111 is NaN; no infinities)
      bytes [512, 516)  one UE8M0 scale per 128-dim group of the latent
                        (scale = 2 ** (byte - 127); byte 255 is NaN)
      bytes [516, 528)  unused (zero)
      bytes [528, 656)  the 64 RoPE dims in bf16, little-endian
  * latent dim d of a row is e4m3(byte d) * scale[d // 128]; the RoPE dims are
    the bf16 values as in the bf16 cache.

Power-of-two group scales keep the product of a code and its scale exactly
representable in bf16 (and in fp16 within its range), so the attention reads
exactly the values the cache encodes; the attention itself is the one of
mla_oracle.attend.
"""

from __future__ import annotations

import numpy as np

from .mla_oracle import D_QK, PAGE, attend, bf16_bits_to_f64, physical_rows, visible_positions

ROW_BYTES = 656   # bytes per cached token
LATENT = 512      # FP8 latent dims
GROUP = 128       # latent dims per scale
SCALE_OFF = 512   # offset of the four scale bytes
ROPE_OFF = 528    # offset of the 64 bf16 RoPE dims
ROPE = D_QK - LATENT


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """OCP FP8 E4M3 codes -> float64, from the format's definition."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = (1.0 + m / 8.0) * np.exp2(e - 7.0)
    sub = (m / 8.0) * np.exp2(-6.0)
    v = sign * np.where(e == 0, sub, normal)
    return np.where((e == 0xF) & (m == 0x7), np.nan, v)


def ue8m0_to_f64(codes: np.ndarray) -> np.ndarray:
    """UE8M0 scale bytes -> float64: 2 ** (byte - 127); 255 is NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    return np.where(c == 255, np.nan, np.exp2(c - 127.0))


def fp8_rows_to_f64(rows: np.ndarray) -> np.ndarray:
    """Cached rows uint8 [..., 656] -> their 576 dims as float64 [..., 576]."""
    rows = np.asarray(rows, dtype=np.uint8)
    if rows.shape[-1] != ROW_BYTES:
        raise ValueError("an FP8 cache row has 656 bytes")
    lat = e4m3_to_f64(rows[..., :LATENT])
    scale = ue8m0_to_f64(rows[..., SCALE_OFF:SCALE_OFF + LATENT // GROUP])
    lat = lat * np.repeat(scale, GROUP, axis=-1)
    rope_bits = rows[..., ROPE_OFF:ROPE_OFF + 2 * ROPE].astype(np.uint16)
    rope_bits = rope_bits[..., 0::2] | (rope_bits[..., 1::2] << 8)  # little-endian bf16
    return np.concatenate([lat, bf16_bits_to_f64(rope_bits)], axis=-1)


def mla_decode_fp8(q_bits: np.ndarray, kv_fp8: np.ndarray, block_table: np.ndarray,
                   cache_lens: np.ndarray, softmax_scale: float, causal: bool = False,
                   topk_idx: np.ndarray | None = None, select=None):
    """Oracle for one decode call over an FP8 cache.

    q_bits:  uint16 (bf16 bits) [B, s_q, H, 576]
    kv_fp8:  uint8 [num_pages, 64, 656]
    Other arguments and the outputs are those of mla_oracle.mla_decode.
    """
    q_bits = np.asarray(q_bits)
    kv_fp8 = np.asarray(kv_fp8, dtype=np.uint8)
    B, s_q, H, dq = q_bits.shape
    if dq != D_QK or kv_fp8.shape[1:] != (PAGE, ROW_BYTES):
        raise ValueError("unexpected q or cache shape")
    num_pages = kv_fp8.shape[0]
    pool = kv_fp8.reshape(num_pages * PAGE, ROW_BYTES)
    o = np.full((B, s_q, H, LATENT), np.nan)
    lse = np.full((B, s_q, H), np.nan)
    pairs = [(b, t) for b in range(B) for t in range(s_q)] if select is None else list(select)
    for b, t in pairs:
        row_idx = None if topk_idx is None else topk_idx[b, t]
        pos = visible_positions(int(cache_lens[b]), s_q, t, causal, row_idx)
        rows = physical_rows(block_table[b], pos, num_pages)
        kv = fp8_rows_to_f64(pool[rows])
        qh = bf16_bits_to_f64(q_bits[b, t])
        o[b, t], lse[b, t] = attend(qh, kv, softmax_scale)
    return o, lse
