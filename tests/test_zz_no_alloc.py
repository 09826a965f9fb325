"""The decode step that allocates nothing (mla_decode_noalloc).

Some callers cannot allocate device memory while a decode step runs - a
serving runtime that records the step into a CUDA graph, or a program with a
fixed device-memory budget.  mla_decode_noalloc keeps its workspace in an
array inside the library.  These tests call it through the C ABI and check
it against the allocating entry point on two calls in a row (the second call
reuses whatever the first one left in the shared array).  The file is named
so that pytest collects it last.
"""

import ctypes

import numpy as np
import pytest
import torch

import mla_latent_kv_09_gb300 as m
import workloads as wl

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _build():
    from mla_latent_kv_09_gb300 import build
    build.build()
    m.load()
    assert torch.cuda.is_available()


def _noalloc(w, out_fp32):
    B, s_q = w.batch, w.s_q
    out = torch.empty((B, s_q, 128, 512), dtype=torch.float32 if out_fp32 else torch.bfloat16, device="cuda")
    lse = torch.empty((B, s_q, 128), dtype=torch.float32, device="cuda")
    flags = (m.MLA_FLAG_CAUSAL if w.causal else 0) | (m.MLA_FLAG_OUT_FP32 if out_fp32 else 0)
    rc = m.load().mla_decode_noalloc(
        w.q.data_ptr(), w.kv.data_ptr(), w.num_pages, w.block_table.data_ptr(), w.block_table.stride(0),
        w.cache_lens.data_ptr(), B, s_q, 128, ctypes.c_float(w.softmax_scale),
        None if w.topk_idx is None else w.topk_idx.data_ptr(), w.topk, flags, out.data_ptr(), lse.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert rc == m.MLA_OK, m.mla_status_string(rc)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _close(a, b):
    (oa, la), (ob, lb) = a, b
    err = np.abs(oa - ob)
    assert err.max() <= O_MAX and err.mean() <= O_MEAN
    fin = np.isfinite(lb)
    assert np.array_equal(np.isfinite(la), fin)
    assert np.abs(la[fin] - lb[fin]).max() <= LSE_MAX


@pytest.mark.parametrize("name,kw", [("mtp_b64", dict(batch=16, length=3000)),
                                     ("uniform_b32", dict(batch=8, length=2000)),
                                     ("sparse_b80", dict(batch=4, length=5000))])
def test_noalloc_matches_allocating_entry_point_twice(name, kw):
    w = wl.make_config(name, device="cuda", **kw)
    o_ref, l_ref = m.decode_step(w.q, w.kv, w.block_table, w.cache_lens, w.softmax_scale, causal=w.causal,
                                 topk_idx=w.topk_idx, out_fp32=True)
    torch.cuda.synchronize()
    ref = (o_ref.cpu().numpy(), l_ref.cpu().numpy())
    first = _noalloc(w, out_fp32=True)
    second = _noalloc(w, out_fp32=True)
    _close(first, ref)
    _close(second, ref)
    bf = _noalloc(w, out_fp32=False)
    _close(bf, ref)


def test_noalloc_rejects_a_batch_beyond_its_workspace():
    # the workspace needs 16 B of request metadata per request: 4M requests
    # cannot fit in 48 MiB whatever the unit count
    rc = m.load().mla_decode_noalloc(1 << 20, 1 << 20, 1, 1 << 20, 1, 1 << 20, 4 << 20, 1, 128,
                                     ctypes.c_float(0.07), None, 0, 0, 1 << 20, 1 << 20, None)
    assert rc == m.MLA_ERR_WORKSPACE
