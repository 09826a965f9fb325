"""Seeded synthetic inputs for MLA decode: the one module both sides share.

This module only draws random inputs; it holds none of the attention
arithmetic.  The CUDA path and the CPU oracle are both fed from it.

Shapes follow the decode workloads the pages describe: 128 weight-absorbed
query heads of 576 dims (512 latent + 64 RoPE), one 576-dim bf16 latent row
per cached token, 64-token pages in a shared pool reached through a block
table ("DeepSeek V3/R1 Inference Efficiency (2)", §2.4.1, decode shapes;
"How DeepSeek Inference Works", levers table, "KV-cache layout (MLA,
paging)").  Batch points 32/64/80/128 mirror the pages' decode batch sizes
(b = 64 per microbatch in §2.4; batch 32 and 80 in "The Premise That
Wasn't").

Structure (lengths, page permutations, top-k lists, pad counts, spiked rows)
comes from numpy's Philox generator keyed by (seed, stream id), so it is the
same on every machine.  The N(0,1) values come from torch's generator on the
target device, drawn in fixed-size chunks, so a run is reproducible on one
device; both sides of a parity test read the same bytes.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

H = 128
D_QK = 576
D_V = 512
PAGE = 64
SCALE = 1.0 / math.sqrt(192.0)  # 1/sqrt(d + r), d = 128, r = 64

_CHUNK_ELEMS = 1 << 26  # elements drawn per randn call


@dataclasses.dataclass
class Workload:
    name: str
    q: torch.Tensor  # bf16 [B, s_q, H, 576]
    kv: torch.Tensor  # bf16 [num_pages, 64, 576], or uint8 [num_pages, 64, 656] FP8 rows
    block_table: torch.Tensor  # int32 [B, max_pages]
    cache_lens: torch.Tensor  # int32 [B]
    topk_idx: torch.Tensor | None  # int32 [B, s_q, k] or None
    softmax_scale: float
    causal: bool

    @property
    def batch(self) -> int:
        return self.q.shape[0]

    @property
    def s_q(self) -> int:
        return self.q.shape[1]

    @property
    def num_pages(self) -> int:
        return self.kv.shape[0]

    @property
    def topk(self) -> int:
        return 0 if self.topk_idx is None else self.topk_idx.shape[-1]

    @property
    def kv_fp8(self) -> bool:
        return self.kv.dtype == torch.uint8


def _np_rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, stream])))


def _randn_bf16(shape, seed: int, stream: int, device, scale: float = 1.0) -> torch.Tensor:
    """N(0, scale^2) rounded to bf16, drawn in fixed chunks on `device`."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000003 + stream)
    n = flat.numel()
    for lo in range(0, n, _CHUNK_ELEMS):
        hi = min(n, lo + _CHUNK_ELEMS)
        x = torch.randn(hi - lo, generator=g, device=device, dtype=torch.float32)
        flat[lo:hi] = (x if scale == 1.0 else x * scale).to(torch.bfloat16)
    return out


FP8_ROW = 656  # bytes of an FP8 cache row: 512 E4M3 codes, 4 UE8M0 scales, 12 unused, 64 bf16 RoPE dims


def _fp8_pool(num_pages: int, seed: int, device, spike_rows=None) -> torch.Tensor:
    """An FP8 cache pool uint8 [num_pages, 64, 656] whose values are N(0,1)
    like the bf16 pool's, quantised the way a cache writer would: each
    128-dim group gets a UE8M0 scale byte 121 + d, d drawn from {0, 1, 2}
    (scales 2^-6 .. 2^-4), and its codes are N(0,1) draws times 2^(6 - d)
    cast to E4M3 by torch (clamped to +-448).  RoPE dims N(0,1) in bf16, the
    12 unused bytes zero.  spike_rows: pool rows whose four scale bytes get
    +3 (values x 8, exact)."""
    rows = num_pages * PAGE
    pool = torch.zeros((rows, FP8_ROW), dtype=torch.uint8, device=device)
    d = _np_rng(seed, 8).integers(0, 3, size=(rows, 4)).astype(np.uint8)
    mult = torch.from_numpy(np.exp2(6.0 - d).astype(np.float32)).to(device)
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000003 + 7)
    step = max(1, _CHUNK_ELEMS // 512)
    for lo in range(0, rows, step):
        hi = min(rows, lo + step)
        x = torch.randn((hi - lo, 4, 128), generator=g, device=device, dtype=torch.float32)
        x = (x * mult[lo:hi, :, None]).clamp_(-448.0, 448.0)
        pool[lo:hi, :512] = x.reshape(hi - lo, 512).to(torch.float8_e4m3fn).view(torch.uint8)
    sc = 121 + d
    if spike_rows is not None and len(spike_rows):
        sc[spike_rows] += 3
    pool[:, 512:516] = torch.from_numpy(sc).to(device)
    rope = _randn_bf16((rows, 64), seed, 9, device)
    pool[:, 528:] = rope.view(torch.uint8)
    return pool.view(num_pages, PAGE, FP8_ROW)


def make_workload(name: str, lens, s_q: int = 1, causal: bool = False, *,
                  topk: int = 0, pad_range=(0, 0), spike_frac: float = 0.0,
                  shuffle: bool = True, extra_pages: int = 0, seed: int = 0,
                  device="cpu", max_pages: int | None = None, kv_fp8: bool = False) -> Workload:
    """Build one decode call's inputs.

    lens:        per-request cache lengths (tokens).
    topk:        if > 0, each (request, token) gets a sorted list of
                 topk - pad distinct positions drawn uniformly from
                 [0, len), followed by pad entries of -1, pad ~ U{pad_range}.
    spike_frac:  fraction of pool rows multiplied by 8 (exact in bf16).
    shuffle:     pages of all requests are placed in the pool in a seeded
                 random order; otherwise request b's pages are contiguous.
    extra_pages: unused pool pages appended (filled with data too).
    max_pages:   width of the block table; unused entries hold -1.
    kv_fp8:      the pool is FP8 rows (see _fp8_pool) instead of bf16.
    """
    lens = np.asarray(lens, dtype=np.int64)
    B = lens.size
    npages_req = (lens + PAGE - 1) // PAGE
    total = int(npages_req.sum()) + int(extra_pages)
    width = int(max(1, npages_req.max() if B else 1)) if max_pages is None else int(max_pages)
    rng = _np_rng(seed, 1)
    order = rng.permutation(total) if shuffle else np.arange(total)
    table = np.full((B, width), -1, dtype=np.int32)
    cursor = 0
    for b in range(B):
        n = int(npages_req[b])
        table[b, :n] = order[cursor:cursor + n]
        cursor += n

    q = _randn_bf16((B, s_q, H, D_QK), seed, 2, device)
    if kv_fp8:
        spikes = None
        if spike_frac > 0:
            spikes = np.nonzero(_np_rng(seed, 4).random(max(total, 1) * PAGE) < spike_frac)[0]
        kv = _fp8_pool(max(total, 1), seed, device, spikes)
    else:
        kv = _randn_bf16((max(total, 1), PAGE, D_QK), seed, 3, device)
    if spike_frac > 0 and not kv_fp8:
        rows = np.nonzero(_np_rng(seed, 4).random(kv.shape[0] * PAGE) < spike_frac)[0]
        idx = torch.from_numpy(rows).to(device)
        flat = kv.view(-1, D_QK)
        flat[idx] = flat[idx] * 8

    topk_t = None
    if topk > 0:
        rng_k = _np_rng(seed, 5)
        lo, hi = pad_range
        idx = np.full((B, s_q, topk), -1, dtype=np.int32)
        for b in range(B):
            for t in range(s_q):
                pad = int(rng_k.integers(lo, hi + 1)) if hi > lo else int(lo)
                n = max(0, min(topk - pad, int(lens[b])))
                pos = np.sort(rng_k.choice(int(lens[b]), size=n, replace=False))
                idx[b, t, :n] = pos
        topk_t = torch.from_numpy(idx).to(device)

    return Workload(
        name=name, q=q, kv=kv,
        block_table=torch.from_numpy(table).to(device),
        cache_lens=torch.from_numpy(lens.astype(np.int32)).to(device),
        topk_idx=topk_t, softmax_scale=SCALE, causal=causal)


# The five decode workloads (full sizes).
CONFIGS = ("single", "uniform_b32", "mtp_b64", "long_b128", "sparse_b80")


def make_config(name: str, seed: int = 0, device="cpu", batch: int | None = None,
                length: int | None = None, kv_fp8: bool = False) -> Workload:
    """One of the five named workloads; `batch` / `length` shrink it for tests.

    single       B=1, L=256 (4 pages, identity block table), s_q=1
    uniform_b32  B=32, every L=4096, shuffled pool
    mtp_b64      B=64, s_q=2 causal, L ~ U{1..8192}, shuffled pool, table
                 entries past each request's pages = -1
    long_b128    B=128, every L=32768, 5% of pool rows scaled x8
    sparse_b80   B=80, every L=65536, top-2048 sorted distinct positions with
                 the last 0..300 entries padded with -1
    mtp4_b64     (beyond the five) mtp_b64's requests with four causal query
                 tokens each: speculative decoding with three draft tokens
    <name>_fp8   (or kv_fp8=True) the same over an FP8 cache of the same shape
                 (the FP8 latent cache; see _fp8_pool)
    """
    if name.endswith("_fp8"):
        w = make_config(name[:-4], seed, device, batch, length, kv_fp8=True)
        w.name = name
        return w
    kw = dict(seed=seed, device=device, kv_fp8=kv_fp8)
    if name == "single":
        return make_workload(name, [length or 256], shuffle=False, **kw)
    if name == "uniform_b32":
        B = batch or 32
        return make_workload(name, [length or 4096] * B, **kw)
    if name in ("mtp_b64", "mtp4_b64"):
        B = batch or 64
        top = length or 8192
        lens = _np_rng(seed, 6).integers(1, top + 1, size=B)
        return make_workload(name, lens, s_q=2 if name == "mtp_b64" else 4, causal=True,
                             max_pages=(top + PAGE - 1) // PAGE, **kw)
    if name == "long_b128":
        B = batch or 128
        return make_workload(name, [length or 32768] * B, spike_frac=0.05, **kw)
    if name == "sparse_b80":
        B = batch or 80
        L = length or 65536
        k = min(2048, L)
        return make_workload(name, [L] * B, topk=k, pad_range=(0, min(300, k)), **kw)
    raise KeyError(name)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Host copy of a bf16 tensor as raw uint16 bit patterns."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def host_arrays(w: Workload):
    """The workload as numpy arrays (bf16 as uint16 bits) for the oracle; an
    FP8 pool comes as its uint8 rows under kv_fp8 (kv_bits is then None)."""
    fp8 = w.kv_fp8
    return dict(
        q_bits=bf16_bits(w.q), kv_bits=None if fp8 else bf16_bits(w.kv),
        kv_fp8=w.kv.cpu().numpy() if fp8 else None,
        block_table=w.block_table.cpu().numpy(), cache_lens=w.cache_lens.cpu().numpy(),
        softmax_scale=w.softmax_scale, causal=w.causal,
        topk_idx=None if w.topk_idx is None else w.topk_idx.cpu().numpy())


# ---------------------------------------------------------------- absorption BMMs
D_NOPE, D_ROPE = 128, 64


@dataclasses.dataclass
class AbsorbInputs:
    q_proj: torch.Tensor  # bf16 [T, H, 192]: per head 128 "nope" dims, then 64 RoPE dims
    o: torch.Tensor       # bf16 [T, H, 512]: an attention output in the latent space
    w_uk: torch.Tensor    # bf16 [H, 512, 128]
    w_uv: torch.Tensor    # bf16 [H, 512, 128]

    @property
    def q_nope(self) -> torch.Tensor:
        return self.q_proj[..., :D_NOPE]

    @property
    def q_pe(self) -> torch.Tensor:
        return self.q_proj[..., D_NOPE:]


def make_absorb(num_tokens: int, num_heads: int = H, seed: int = 0, device="cpu") -> AbsorbInputs:
    """Inputs of the two weight-absorption BMMs for a step of `num_tokens`
    (request, query token) pairs ("DeepSeek V3/R1 Inference Efficiency (2)",
    §2.4.1: q_nope [n_head, bs, 128], W_UK and W_UV [n_head, 512, 128]).
    Activations are N(0,1); weights are random-init N(0, 1/fan_in) (fan_in =
    128 for W_UK, whose contraction runs over d, 512 for W_UV, over c), so
    that both outputs are O(1).  The query projection output is one
    [T, H, 192] tensor, as the query up-projection produces it."""
    q = _randn_bf16((num_tokens, num_heads, D_NOPE + D_ROPE), seed, 20, device)
    o = _randn_bf16((num_tokens, num_heads, D_V), seed, 21, device)
    w_uk = _randn_bf16((num_heads, D_V, D_NOPE), seed, 22, device, scale=1.0 / math.sqrt(D_NOPE))
    w_uv = _randn_bf16((num_heads, D_V, D_NOPE), seed, 23, device, scale=1.0 / math.sqrt(D_V))
    return AbsorbInputs(q_proj=q, o=o, w_uk=w_uk, w_uv=w_uv)


# ---------------------------------------------------------------- sparse-attention indexer
H_IDX, D_IDX = 64, 128


@dataclasses.dataclass
class IndexerInputs:
    q_idx: torch.Tensor    # bf16 [B, s_q, 64, 128]
    w_idx: torch.Tensor    # fp32 [B, s_q, 64]
    k_cache: torch.Tensor  # bf16 [num_pages, 64, 128]: index keys, same pages as the latent pool


def make_indexer(w: Workload, seed: int = 0) -> IndexerInputs:
    """Indexer inputs for a decode workload: one 128-dim index key per cached
    token in the workload's pages (same block table), index queries of 64
    heads per query token, head weights N(0, 1/64).  Keys and queries N(0,1)
    in bf16."""
    dev = w.q.device
    B, s_q = w.batch, w.s_q
    q = _randn_bf16((B, s_q, H_IDX, D_IDX), seed, 30, dev)
    k = _randn_bf16((w.num_pages, PAGE, D_IDX), seed, 31, dev)
    g = torch.Generator(device=dev)
    g.manual_seed(seed * 1000003 + 32)
    wt = torch.randn((B, s_q, H_IDX), generator=g, device=dev, dtype=torch.float32) / 8.0
    return IndexerInputs(q_idx=q, w_idx=wt, k_cache=k)
