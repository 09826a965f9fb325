"""The decode step that allocates nothing (mla_decode_noalloc).

Some callers cannot allocate device memory while a decode step runs - a
serving runtime that records the step into a CUDA graph, or a program with a
fixed device-memory budget.  mla_decode_noalloc keeps its workspace in an
array inside the library.  These tests call it through the C ABI and check
it against the allocating entry point on two calls in a row (the second call
reuses whatever the first one left in the shared array) and expect the same
bits, since both run the same plan and kernels.  The file is named so that
pytest collects it last.
"""

import ctypes

import numpy as np
import pytest
import torch

import mla_latent_kv_09_gb300 as m
import workloads as wl

pytestmark = pytest.mark.gpu


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


def _allocating(w, out_fp32):
    # the allocating entry points with the unit count the built-in workspace
    # gets for these sizes (the default: the workspace fits), so the plan and
    # every kernel's arithmetic are the same and the outputs must be too
    o, l = m.decode_step(w.q, w.kv, w.block_table, w.cache_lens, w.softmax_scale, causal=w.causal,
                         topk_idx=w.topk_idx, out_fp32=out_fp32, num_units=m.mla_default_num_units(w.s_q))
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), l.cpu().numpy()


def _same(a, b):
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("name,kw", [("mtp_b64", dict(batch=16, length=3000)),
                                     ("uniform_b32", dict(batch=8, length=2000)),
                                     ("sparse_b80", dict(batch=4, length=5000)),
                                     ("mtp4_b64", dict(batch=12, length=2500))])
def test_noalloc_matches_allocating_entry_point_twice(name, kw):
    w = wl.make_config(name, device="cuda", **kw)
    ref = _allocating(w, out_fp32=True)
    _same(_noalloc(w, out_fp32=True), ref)
    _same(_noalloc(w, out_fp32=True), ref)  # the array now holds the first call's state
    _same(_noalloc(w, out_fp32=False), _allocating(w, out_fp32=False))
    assert m.mla_noalloc_status() == m.MLA_OK


def test_noalloc_calls_of_changing_shape_leave_nothing_behind():
    # a larger call first (more requests, split slots in use), then smaller
    # ones of other kinds: each must equal its allocating twin exactly
    seq = [wl.make_config("mtp_b64", device="cuda", batch=16, length=6000),
           wl.make_config("sparse_b80", device="cuda", batch=4, length=5000),
           wl.make_config("uniform_b32", device="cuda", batch=8, length=2000),
           wl.make_config("mtp_b64", device="cuda", batch=3, length=500)]
    for w in seq:
        _same(_noalloc(w, out_fp32=True), _allocating(w, out_fp32=True))


def test_noalloc_reports_device_errors_through_its_status_query():
    # a wait that runs out inside the built-in array is reported by
    # mla_noalloc_status; the next call resets the status and is exact again
    ptr, nbytes = m.mla_noalloc_workspace()
    assert ptr and nbytes >= 256
    m.mla_selftest_wait_timeout(ptr, nbytes)
    assert m.mla_noalloc_status() == m.MLA_ERR_TIMEOUT
    w = wl.make_config("uniform_b32", device="cuda", batch=4, length=700)
    _same(_noalloc(w, out_fp32=True), _allocating(w, out_fp32=True))
    assert m.mla_noalloc_status() == m.MLA_OK
    # a failed validation is reported the same way, with O left unwritten
    kv = w.kv.clone()
    row = int(w.block_table[2, 3]) * 64 + 5  # position 197 of request 2 (700 tokens)
    kv.view(-1, 576)[row, 11] = float("inf")
    out = torch.full((4, 1, 128, 512), 7.0, dtype=torch.float32, device="cuda")
    lse = torch.empty((4, 1, 128), dtype=torch.float32, device="cuda")
    rc = m.load().mla_decode_noalloc(
        w.q.data_ptr(), kv.data_ptr(), w.num_pages, w.block_table.data_ptr(), w.block_table.stride(0),
        w.cache_lens.data_ptr(), 4, 1, 128, ctypes.c_float(w.softmax_scale), None, 0,
        m.MLA_FLAG_VALIDATE | m.MLA_FLAG_OUT_FP32, out.data_ptr(), lse.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert rc == m.MLA_OK
    assert m.mla_noalloc_status() == m.MLA_ERR_VALUE_RANGE
    assert bool((out == 7.0).all())


def test_noalloc_rejects_a_batch_beyond_its_workspace():
    # the workspace needs 16 B of request metadata per request: 4M requests
    # cannot fit in 48 MiB whatever the unit count
    rc = m.load().mla_decode_noalloc(1 << 20, 1 << 20, 1, 1 << 20, 1, 1 << 20, 4 << 20, 1, 128,
                                     ctypes.c_float(0.07), None, 0, 0, 1 << 20, 1 << 20, None)
    assert rc == m.MLA_ERR_WORKSPACE
