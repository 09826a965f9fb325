"""Host mirror of the split-KV planner: every (request, tile) is covered
exactly once, in order, by equally loaded unit ranges, and the split and
slot bookkeeping the combine step relies on is consistent."""

import numpy as np
import pytest

import mla_latent_kv_09_gb300 as m
from mla_latent_kv_09_gb300 import build as mbuild

C0 = 2  # per-split fixed cost in tiles (matches the planner)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mbuild.build()
    m.load()


def expand(um, rm):
    """Per unit: list of (request, tile) pairs it processes, in order."""
    B = rm.shape[0]
    units = []
    for bb, bt, eb, et, fs in um:
        work = []
        b = bb
        while b < B and (b < eb or (b == eb and et > 0)):
            t0 = bt if b == bb else 0
            t1 = et if b == eb else rm[b, 0]
            work += [(b, t) for t in range(t0, t1)]
            b += 1
        units.append(work)
    return units


def check_plan(lens, U, topk=0, s_q=1):
    um, rm = m.mla_decode_plan_host(lens, s_q, topk, U)
    lens = np.asarray(lens)
    rows = 128 if (s_q == 2 and topk == 0) else 64  # the two-token dense kernel takes two pages per tile
    ntiles = np.array([(k + rows - 1) // rows for k in ([topk] * len(lens) if topk else np.maximum(lens, 0))])
    assert np.array_equal(rm[:, 0], ntiles)
    units = expand(um, rm)
    flat = [w for u in units for w in u]
    want = [(b, t) for b in range(len(lens)) for t in range(ntiles[b])]
    assert flat == want  # each (request, tile) exactly once, in order
    # split counts: number of units touching each request
    touch = np.zeros(len(lens), int)
    for u in units:
        for b in sorted({b for b, _ in u}):
            touch[b] += 1
    assert np.array_equal(rm[:, 1], touch)
    # slots: split requests get disjoint consecutive ranges; <= 2U in total
    used = []
    for b in range(len(lens)):
        if rm[b, 1] > 1:
            used += list(range(rm[b, 2], rm[b, 2] + rm[b, 1]))
    assert len(used) == len(set(used)) and len(used) <= 2 * U
    # first_split: the split index of a unit's first segment
    seen = np.zeros(len(lens), int)
    for ui, u in enumerate(units):
        if not u:
            continue
        b0 = u[0][0]
        assert um[ui, 4] == seen[b0]
        for b in sorted({b for b, _ in u}):
            seen[b] += 1
    # balance: unit cost (tiles + C0 per segment) within W + C0 of the mean
    costs = [len(u) + C0 * len({b for b, _ in u}) for u in units]
    total = int(sum(n + C0 for n in ntiles if n > 0))
    W = max(-(-total // U), C0 + 4)
    assert max(costs) <= W + C0
    return um, rm, units


@pytest.mark.parametrize("seed", range(12))
def test_random_lengths(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 200))
    lens = rng.integers(0, 9000, B)
    lens[rng.random(B) < 0.1] = 0
    U = int(rng.integers(1, 200))
    check_plan(lens, U)


@pytest.mark.parametrize("seed", range(6))
def test_random_lengths_two_tokens(seed):
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 200))
    lens = rng.integers(0, 9000, B)
    lens[rng.random(B) < 0.1] = 0
    U = int(rng.integers(1, 60))
    check_plan(lens, U, s_q=2)
    check_plan(lens, U, topk=int(rng.integers(1, 3000)), s_q=2)


def test_decode_workload_shapes():
    check_plan([4096] * 32, 74)
    check_plan(np.random.default_rng(0).integers(1, 8193, 64), 36, s_q=2)
    check_plan([32768] * 128, 74)
    check_plan([65536] * 80, 74, topk=2048)
    check_plan([256], 74)


def test_one_long_request_is_split_across_all_units():
    um, rm, units = check_plan([8192], 64)
    # 128 tiles + C0, at least C0 + 4 cost per unit -> 22 units
    assert rm[0, 1] == sum(1 for u in units if u) == -(-130 // (C0 + 4))


def test_single_unit_never_splits():
    um, rm, units = check_plan([100, 5000, 1, 64], 1)
    assert (rm[:, 1] == 1).all()


def test_two_token_tiles_are_two_pages():
    um, rm, units = check_plan([1, 64, 65, 128, 129, 8192], 4, s_q=2)
    assert list(rm[:, 0]) == [1, 1, 1, 1, 2, 64]


def test_empty_requests_have_no_work():
    um, rm, units = check_plan([0, 0, 70, 0], 8)
    assert rm[0, 1] == 0 and rm[1, 1] == 0 and rm[3, 1] == 0 and rm[2, 1] >= 1


def test_balance_on_uniform_batch_is_tight():
    um, rm, units = check_plan([4096] * 32, 74)
    sizes = [len(u) for u in units]
    # makespan: no unit holds more than W = ceil(total cost / U) tiles
    assert max(sizes) <= -(-(32 * (64 + C0)) // 74)
    assert sum(1 for x in sizes if x) >= 72


# ---------------------------------------------------------------- device plan vs host mirror

def _align256(x):
    return (x + 255) // 256 * 256


def ws_offsets(B, s_q, U):
    """Byte offsets of the workspace's unit table and request table, and its
    size: header (64 ints), unit table (U x 5 ints), request table (B x 4
    ints), fp32 partial LSE and 16-bit partial O (2U slots), each 256-byte
    aligned."""
    off_units = _align256(64 * 4)
    off_reqs = off_units + _align256(U * 5 * 4)
    slots = 2 * U
    total = (off_reqs + _align256(B * 4 * 4) + _align256(slots * s_q * 128 * 4)
             + _align256(slots * s_q * 128 * 512 * 2))
    return off_units, off_reqs, total


@pytest.mark.parametrize("B,s_q,U", [(1, 1, 1), (64, 2, 36), (200, 1, 74), (37, 2, 5)])
def test_workspace_offsets_match_the_library(B, s_q, U):
    assert ws_offsets(B, s_q, U)[2] == m.mla_decode_workspace_size(B, s_q, 128, U)


@pytest.mark.gpu
@pytest.mark.parametrize("seed", range(4))
def test_device_plan_matches_host_plan_bit_exactly(seed):
    import torch
    rng = np.random.default_rng(500 + seed)
    for s_q, topk in [(1, 0), (2, 0), (2, 512), (1, 2048)]:
        B = int(rng.integers(1, 200)) if seed < 3 else int(rng.integers(4097, 6000))  # beyond the smem table
        U = int(rng.integers(1, 80))
        lens = rng.integers(0, 9000, B).astype(np.int32)
        lens[rng.random(B) < 0.1] = 0
        um_h, rm_h = m.mla_decode_plan_host(lens, s_q, topk, U)
        ws = m.Workspace(B, s_q, U, torch.device("cuda:0"))
        ws.buf.fill_(0xAB)  # stale bytes must all be overwritten
        m.mla_decode_plan(torch.from_numpy(lens).cuda(), B, s_q, topk, U, ws.buf, ws.nbytes)
        torch.cuda.synchronize()
        assert m.mla_workspace_status(ws.buf) == 0
        raw = ws.buf.cpu().numpy()
        off_u, off_r, _ = ws_offsets(B, s_q, U)
        um_d = raw[off_u:off_u + U * 20].view(np.int32).reshape(U, 5)
        rm_d = raw[off_r:off_r + B * 16].view(np.int32).reshape(B, 4)
        assert np.array_equal(um_d, um_h), (s_q, topk, B, U)
        assert np.array_equal(rm_d, rm_h), (s_q, topk, B, U)
