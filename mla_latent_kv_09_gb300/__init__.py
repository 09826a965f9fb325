"""GB300 (sm_103a) weight-absorbed MLA decode over a paged latent KV cache.

The computation lives in libmla_decode.so (CUDA, hand-written tcgen05/TMA
kernels); this package is its Python face:

  * the C-ABI entry points under their C names (mla_decode_plan, mla_decode,
    mla_combine, ...) taking raw pointers or torch tensors;
  * `decode_step`, which allocates the outputs and runs plan -> decode ->
    combine on the current stream;
  * `decode_step_host`, the same call for host-resident inputs (copies in,
    runs, copies the outputs back);
  * `absorb_q` / `absorb_o`, the weight-absorption BMMs on either side of
    the attention (query through W_UK, output through W_UV);
  * `indexer_scores` / `topk_indices`, the sparse-attention indexer that
    produces the top-k lists the sparse decode consumes.

PyTorch is used only to allocate device memory and to name streams.
"""

from __future__ import annotations

from ._binding import (  # noqa: F401
    MLA_ERR_BAD_INDEX,
    MLA_ERR_BAD_TABLE,
    MLA_ERR_CUDA,
    MLA_ERR_DEVICE,
    MLA_ERR_INVALID_ARG,
    MLA_ERR_TIMEOUT,
    MLA_ERR_UNSUPPORTED,
    MLA_ERR_VALUE_RANGE,
    MLA_ERR_WORKSPACE,
    MLA_FLAG_CAUSAL,
    MLA_FLAG_BF16_PV,
    MLA_FLAG_KV_FP8,
    MLA_FLAG_OUT_FP32,
    MLA_FLAG_VALIDATE,
    MLA_OK,
    SIGNATURES,
    MlaError,
    load,
    mla_absorb_o,
    mla_absorb_q,
    mla_indexer_scores,
    mla_topk,
    mla_combine,
    mla_decode,
    mla_decode_noalloc,
    mla_noalloc_status,
    mla_noalloc_workspace,
    mla_decode_plan,
    mla_decode_plan_host,
    mla_decode_workspace_size,
    mla_default_num_units,
    mla_status_string,
    mla_workspace_status,
    mla_selftest_wait_timeout,
)

NUM_HEADS = 128
D_QK = 576
D_V = 512
PAGE = 64


class Workspace:
    """A device workspace sized for (batch, s_q, num_units)."""

    def __init__(self, batch: int, s_q: int, num_units: int = 0, device=None):
        import torch
        self.batch, self.s_q = batch, s_q
        self.num_units = num_units or mla_default_num_units(s_q)
        self.nbytes = mla_decode_workspace_size(batch, s_q, NUM_HEADS, self.num_units)
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device or "cuda")


def decode_step(q, kv_cache, block_table, cache_lens, softmax_scale: float, *, causal: bool = False,
                topk_idx=None, out_fp32: bool = False, validate: bool = False, bf16_pv: bool = False,
                num_units: int = 0, workspace: Workspace | None = None, out=None, lse=None, stream=None):
    """One MLA decode step on device tensors: plan, attention, combine.

    q [B, s_q, 128, 576] bf16; kv_cache [num_pages, 64, 576] bf16, or
    uint8 [num_pages, 64, 656] FP8 rows (MLA_FLAG_KV_FP8 is then set);
    block_table [B, W] int32; cache_lens [B] int32; topk_idx [B, s_q, k]
    int32 or None.  bf16_pv selects MLA_FLAG_BF16_PV (two-token dense path:
    faster, less precise value product).  With validate=True the inputs are
    checked on the device first and the step's status is read back (a host
    synchronisation) and raised as MlaError if it is not MLA_OK.
    Returns (O [B, s_q, 128, 512] bf16 or fp32, LSE fp32).
    """
    import torch
    B, s_q = q.shape[0], q.shape[1]
    if workspace is None:
        workspace = Workspace(B, s_q, num_units, q.device)
    U = workspace.num_units
    if out is None:
        out = torch.empty((B, s_q, NUM_HEADS, D_V), dtype=torch.float32 if out_fp32 else torch.bfloat16,
                          device=q.device)
    if lse is None:
        lse = torch.empty((B, s_q, NUM_HEADS), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    topk = 0 if topk_idx is None else topk_idx.shape[-1]
    flags = (MLA_FLAG_CAUSAL if causal else 0) | (MLA_FLAG_OUT_FP32 if out_fp32 else 0) | (
        MLA_FLAG_VALIDATE if validate else 0) | (MLA_FLAG_BF16_PV if bf16_pv else 0)
    if kv_cache.dtype == torch.uint8:
        flags |= MLA_FLAG_KV_FP8
    mla_decode_plan(cache_lens, B, s_q, topk, U, workspace.buf, workspace.nbytes, stream)
    mla_decode(q, kv_cache, kv_cache.shape[0], block_table, block_table.stride(0), cache_lens, B, s_q,
               NUM_HEADS, softmax_scale, topk_idx, topk, flags, U, workspace.buf, workspace.nbytes, out,
               lse, stream)
    mla_combine(workspace.buf, workspace.nbytes, B, s_q, NUM_HEADS, flags, U, out, lse, stream)
    if validate:
        # the check runs on the device; its outcome is read back here (the
        # C calls themselves never synchronise for it)
        status = mla_workspace_status(workspace.buf, stream)
        if status != MLA_OK:
            raise MlaError("mla_decode (validate)", status)
    return out, lse


def decode_step_host(q, kv_cache, block_table, cache_lens, softmax_scale: float, *, device="cuda",
                     causal: bool = False, topk_idx=None, out_fp32: bool = False, bf16_pv: bool = False,
                     num_units: int = 0,
                     workspace: Workspace | None = None, dev_buffers=None, out_host=None, lse_host=None):
    """decode_step for HOST tensors (pinned for speed): H2D copies, the step,
    D2H copies of O and LSE.  `dev_buffers` may hold preallocated device
    tensors with the same keys as the inputs to avoid allocation per call."""
    import torch
    d = dev_buffers or {}

    def up(name, t):
        if t is None:
            return None
        dst = d.get(name)
        if dst is None:
            dst = torch.empty(t.shape, dtype=t.dtype, device=device)
        dst.copy_(t, non_blocking=True)
        return dst

    o, l = decode_step(up("q", q), up("kv_cache", kv_cache), up("block_table", block_table),
                       up("cache_lens", cache_lens), softmax_scale, causal=causal,
                       topk_idx=up("topk_idx", topk_idx), out_fp32=out_fp32, bf16_pv=bf16_pv,
                       num_units=num_units,
                       workspace=workspace, out=d.get("out"), lse=d.get("lse"))
    if out_host is None:
        out_host = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    if lse_host is None:
        lse_host = torch.empty(l.shape, dtype=l.dtype, pin_memory=True)
    out_host.copy_(o, non_blocking=True)
    lse_host.copy_(l, non_blocking=True)
    torch.cuda.current_stream(device).synchronize()
    return out_host, lse_host


def _rows(t, dims: int, name: str) -> int:
    """Row stride of a token-major [T, H, dims] activation whose rows may be
    spaced wider than `dims` (e.g. a slice of a [T, H, 192] tensor)."""
    if t.dim() != 3 or t.shape[2] != dims or t.stride(2) != 1 or t.stride(0) != t.shape[1] * t.stride(1):
        raise ValueError(f"{name}: expected [T, H, {dims}] with unit stride in the last dim and rows "
                         "evenly spaced over (token, head)")
    return t.stride(1)


def absorb_q(q_nope, w_uk, q_pe=None, *, out=None, status=None, stream=None):
    """Query-side absorption: q_latent[t, h] = W_UK[h] @ q_nope[t, h].

    q_nope [T, H, 128] bf16 (rows may be strided, e.g. [..., :128] of a
    [T, H, 192] projection output), w_uk [H, 512, 128] bf16, q_pe [T, H, 64]
    bf16 with the same row stride, or None.  Returns `out`, by default a new
    [T, H, 576] tensor (the decode attention's query) with the RoPE dims in
    512..575, or [T, H, 512] without q_pe.  `status` (int32 device tensor,
    one element) receives MLA_ERR_TIMEOUT if a device wait runs out.
    """
    import torch
    T, H = q_nope.shape[0], q_nope.shape[1]
    q_stride = _rows(q_nope, 128, "q_nope")
    if q_pe is not None and _rows(q_pe, 64, "q_pe") != q_stride:
        raise ValueError("q_pe must have the row stride of q_nope")
    if out is None:
        out = torch.empty((T, H, D_QK if q_pe is not None else D_V), dtype=torch.bfloat16, device=q_nope.device)
    out_stride = _rows(out, out.shape[2], "out")
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=q_nope.device)
    if stream is None:
        stream = torch.cuda.current_stream(q_nope.device)
    mla_absorb_q(q_nope, q_pe, q_stride, w_uk, T, H, out, out_stride, status, stream)
    return out


def absorb_o(o, w_uv, *, out=None, status=None, stream=None):
    """Output-side absorption: out[t, h] = O[t, h] @ W_UV[h].

    o [T, H, 512] bf16 (the decode attention's output), w_uv [H, 512, 128]
    bf16.  Returns `out`, by default a new [T, H, 128] bf16 tensor.
    """
    import torch
    T, H = o.shape[0], o.shape[1]
    o_stride = _rows(o, 512, "o")
    if out is None:
        out = torch.empty((T, H, 128), dtype=torch.bfloat16, device=o.device)
    out_stride = _rows(out, 128, "out")
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=o.device)
    if stream is None:
        stream = torch.cuda.current_stream(o.device)
    mla_absorb_o(o, o_stride, w_uv, T, H, out, out_stride, status, stream)
    return out


def indexer_scores(q_idx, w_idx, k_idx_cache, block_table, cache_lens, *, causal: bool = False,
                   max_len: int | None = None, scores=None, status=None, stream=None):
    """Index scores of every visible position.

    q_idx [B, s_q, 64, 128] bf16, w_idx [B, s_q, 64] fp32, k_idx_cache
    [num_pages, 64, 128] bf16 (paged like the latent cache, same block
    table).  Returns `scores` (default a new fp32 [B, s_q, max_len] tensor;
    positions past a token's visible count are left unwritten).
    """
    import torch
    B, s_q = q_idx.shape[0], q_idx.shape[1]
    if max_len is None:
        max_len = block_table.shape[1] * PAGE
    if scores is None:
        stride = (max_len + 3) // 4 * 4
        scores = torch.empty((B, s_q, stride), dtype=torch.float32, device=q_idx.device)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=q_idx.device)
    if stream is None:
        stream = torch.cuda.current_stream(q_idx.device)
    mla_indexer_scores(q_idx, w_idx, k_idx_cache, k_idx_cache.shape[0], block_table, block_table.stride(0),
                       cache_lens, B, s_q, MLA_FLAG_CAUSAL if causal else 0, max_len, scores, scores.stride(1),
                       status, stream)
    return scores


def topk_indices(scores, cache_lens, topk: int, *, causal: bool = False, max_len: int | None = None, out=None,
                 status=None, stream=None):
    """Top-k lists [B, s_q, topk] int32 (increasing positions, -1 padded)
    from index scores [B, s_q, stride] (as `indexer_scores` returns them)."""
    import torch
    B, s_q = scores.shape[0], scores.shape[1]
    if max_len is None:
        max_len = scores.shape[2]
    if out is None:
        out = torch.empty((B, s_q, topk), dtype=torch.int32, device=scores.device)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=scores.device)
    if stream is None:
        stream = torch.cuda.current_stream(scores.device)
    mla_topk(scores, scores.stride(1), cache_lens, B, s_q, MLA_FLAG_CAUSAL if causal else 0, max_len, topk, out,
             status, stream)
    return out
