"""The C-ABI library builds for sm_103a, loads, and exports every declared
entry point; host-side argument checks answer without touching a GPU."""

import ctypes
import os
import re

import pytest

import mla_latent_kv_09_gb300 as m
from mla_latent_kv_09_gb300 import build as mbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


def declared_functions():
    text = "\n".join(open(h).read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(mla_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    mbuild.build()
    return m.load()


def test_header_declares_the_three_calls_and_helpers():
    names = declared_functions()
    for n in ["mla_decode_plan", "mla_decode", "mla_combine", "mla_decode_workspace_size",
              "mla_status_string", "mla_default_num_units", "mla_decode_plan_host",
              "mla_workspace_status", "mla_selftest_wait_timeout", "mla_absorb_q", "mla_absorb_o"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in m.SIGNATURES, name


def test_status_strings(lib):
    for code in range(0, 9):
        s = m.mla_status_string(code)
        assert s.startswith("MLA_")
    assert m.mla_status_string(99) == "unknown mla_status"


def test_workspace_size_is_pure_host_arithmetic(lib):
    n = m.mla_decode_workspace_size(64, 2, 128, 38)
    slots = 2 * 38
    # 16-bit partial rows and fp32 partial LSEs per slot and token, plus the plan
    assert n >= slots * 2 * 128 * (512 * 2 + 4) + 64 * 16
    assert n < slots * 2 * 128 * 512 * 4  # half the bytes fp32 partial rows would take
    with pytest.raises(m.MlaError):
        m.mla_decode_workspace_size(64, 2, 64, 38)  # 64 heads: unsupported
    with pytest.raises(m.MlaError):
        m.mla_decode_workspace_size(0, 1, 128, 10)


def test_null_pointers_and_bad_shapes_are_rejected_before_any_launch(lib):
    # every argument check below happens on the host, before the device is touched
    f = lib.mla_decode
    ok_ptr = 1 << 20
    args = [ok_ptr, ok_ptr, 10, ok_ptr, 4, ok_ptr, 2, 1, 128, 0.07, None, 0, 0, 8, ok_ptr, 1 << 30,
            ok_ptr, ok_ptr, None]
    a = list(args); a[0] = None
    assert f(*a) == m.MLA_ERR_INVALID_ARG
    a = list(args); a[8] = 64
    assert f(*a) == m.MLA_ERR_UNSUPPORTED
    a = list(args); a[7] = 9  # s_q beyond MLA_MAX_SQ
    assert f(*a) == m.MLA_ERR_UNSUPPORTED
    a = list(args); a[0] = ok_ptr + 8  # q not 16-byte aligned
    assert f(*a) == m.MLA_ERR_INVALID_ARG
    a = list(args); a[10] = ok_ptr  # index list without a length
    assert f(*a) == m.MLA_ERR_INVALID_ARG
    a = list(args); a[12] = 1 << 7  # unknown flag
    assert f(*a) == m.MLA_ERR_INVALID_ARG
    a = list(args); a[9] = float("nan")
    assert f(*a) == m.MLA_ERR_INVALID_ARG
    assert lib.mla_combine(None, 0, 1, 1, 128, 0, 1, ok_ptr, ok_ptr, None) == m.MLA_ERR_INVALID_ARG
    assert lib.mla_decode_plan(None, 1, 1, 0, 1, ok_ptr, 1 << 20, None) == m.MLA_ERR_INVALID_ARG
    assert lib.mla_selftest_wait_timeout(None, 1 << 20, None) == m.MLA_ERR_INVALID_ARG
    assert lib.mla_selftest_wait_timeout(ok_ptr, 64, None) == m.MLA_ERR_INVALID_ARG  # smaller than the header
    assert lib.mla_selftest_wait_timeout(ok_ptr + 16, 1 << 20, None) == m.MLA_ERR_INVALID_ARG  # misaligned


def test_absorption_calls_check_their_arguments_on_the_host(lib):
    ok = 1 << 20
    q = [ok, ok + 256, 192, ok, 128, 128, ok, 576, ok, None]  # q_nope, q_pe, q_stride, w_uk, T, H, out, out_stride, status
    o = [ok, 512, ok, 128, 128, ok, 128, ok, None]            # o, o_stride, w_uv, T, H, out, out_stride, status
    for f, good, bad in [
        (lib.mla_absorb_q, q, [(0, None), (3, None), (6, None), (8, None), (0, ok + 8), (1, ok + 8),
                               (8, ok + 2), (2, 120), (2, 196), (7, 512), (7, 580), (4, -1)]),
        (lib.mla_absorb_o, o, [(0, None), (2, None), (5, None), (7, None), (0, ok + 8), (5, ok + 4),
                               (1, 504), (1, 516), (6, 120), (3, -1)]),
    ]:
        for i, v in bad:
            a = list(good); a[i] = v
            assert f(*a) == m.MLA_ERR_INVALID_ARG, (f.__name__, i, v)
        for h in (0, 129):  # head counts outside 1..128
            a = list(good); a[5 if f is lib.mla_absorb_q else 4] = h
            assert f(*a) == m.MLA_ERR_UNSUPPORTED
    # without the RoPE rows the output may be 512 wide; zero tokens launch
    # nothing (MLA_ERR_DEVICE where no GPU is present)
    a = list(q); a[1] = None; a[7] = 512; a[4] = 0
    assert lib.mla_absorb_q(*a) in (m.MLA_OK, m.MLA_ERR_DEVICE)


def test_indexer_calls_check_their_arguments_on_the_host(lib):
    ok = 1 << 20
    sc = [ok, ok, ok, 10, ok, 4, ok, 2, 1, 0, 256, ok, 256, ok, None]
    for i, v in [(0, None), (1, None), (2, None), (4, None), (6, None), (11, None), (13, None), (0, ok + 8),
                 (3, 0), (5, 0), (7, 0), (9, 8), (10, 257), (12, 255), (12, 254), (13, ok + 2)]:
        a = list(sc); a[i] = v
        assert lib.mla_indexer_scores(*a) == m.MLA_ERR_INVALID_ARG, (i, v)
    a = list(sc); a[8] = 9
    assert lib.mla_indexer_scores(*a) == m.MLA_ERR_UNSUPPORTED
    tk = [ok, 256, ok, 2, 1, 0, 256, 64, ok, ok, None]
    for i, v in [(0, None), (2, None), (8, None), (9, None), (7, 0), (7, 65537), (1, 100), (8, ok + 2)]:
        a = list(tk); a[i] = v
        assert lib.mla_topk(*a) == m.MLA_ERR_INVALID_ARG, (i, v)


def test_python_binding_raises_when_library_missing(tmp_path):
    from mla_latent_kv_09_gb300 import _binding
    saved = _binding._lib
    try:
        _binding._lib = None
        with pytest.raises(RuntimeError):
            _binding.load(str(tmp_path / "nope.so"))
    finally:
        _binding._lib = saved
