"""Benchmark of one MLA decode step (plan + attention + combine) on GB300.

Default workload: the B=64 variable-length two-token (MTP, causal) decode
step - 64 requests, cache lengths ~U{1..8192}, 128 heads x 576 dims, 64-token
pages in a shuffled pool, bf16 inputs ~N(0,1) - the batch-64 decode shape
the pages quote (b = 64 per microbatch).  Inputs are synthetic and resident
in HBM; the pool exceeds L2 and L2 is also flushed (256 MB write) before
every timed step.

Before the headline workload the same step is timed on the four other
decode workloads (one request of 256 tokens; B=32 at 4096 tokens; B=128 at
32768 tokens with 5% of rows x8; B=80 top-2048 of 65536) and on the B=64
requests with four causal query tokens (mtp4_b64), each with its roofline
figures and a bounded oracle sample on the host cores, reported under
`other_workloads`.  The weight-absorption BMMs either side of the
attention (query through W_UK, output through W_UV) are timed alone at the
headline step's 128 tokens and at 64 tokens, under `absorb`; the
sparse-attention indexer (scores + top-2048 lists) on the sparse workload's
shape under `indexer`.

Prints ONE JSON line.  `value` is the whole-job attention throughput in
TFLOP/s (algorithmic FLOPs of every rank's steps / max-over-ranks time);
microseconds per call, HBM GB/s and the roofline fractions ride along.
`--impl reference` times the fp64 CPU oracle instead (rank 0 only).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA decode us/call, TFLOPS and HBM GB/s as % of GB300 roofline (B=64)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
COMMON_SOURCES = ["ptx.cuh", "common.cuh", "kernel_common.cuh", "plan.cuh"]


TWO_TOKEN_DENSE = {"mtp_b64"}  # workloads with s_q = 2 and no top-k lists


def kernel_sources(workload: str):
    """Sources of the attention kernel a workload runs: two-token dense
    requests take the paired-SM kernel, everything else the one-token one."""
    return (["mtp_kernel.cu"] if workload in TWO_TOKEN_DENSE else ["decode_kernel.cu"]) + COMMON_SOURCES


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_hash(workload: str) -> str:
    h = hashlib.sha256()
    for f in kernel_sources(workload):
        h.update(open(os.path.join(ROOT, "mla_latent_kv_09_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str):
    """DRAM bytes per decode launch from a committed ncu capture, if it was
    taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path))
    e = d.get(workload)
    if not e or e.get("kernel_hash") != kernel_hash(workload):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        # raw samples go to $MLA_BENCH_LOG_DIR (default: the temporary directory)
        log_dir = os.environ.get("MLA_BENCH_LOG_DIR") or tempfile.gettempdir()
        self.path = os.path.join(log_dir, f"clocks_bench_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        self.proc.wait()
        self.f.close()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def oracle_sample(w, host, reqs):
    """Run the fp64 oracle on requests `reqs` (all their query tokens)."""
    import oracle
    sel = [(b, t) for b in reqs for t in range(w.s_q)]
    if host["kv_fp8"] is not None:  # an FP8 cache
        oracle.mla_decode_fp8(host["q_bits"], host["kv_fp8"], host["block_table"], host["cache_lens"],
                              host["softmax_scale"], causal=host["causal"], topk_idx=host["topk_idx"], select=sel)
        return
    oracle.mla_decode(host["q_bits"], host["kv_bits"], host["block_table"], host["cache_lens"],
                      host["softmax_scale"], causal=host["causal"], topk_idx=host["topk_idx"], select=sel)


def sample_flops(w, host, reqs):
    from mla_latent_kv_09_gb300 import accounting as acc
    import numpy as np
    counts = acc.visible_counts(host["cache_lens"], w.s_q, w.causal, host["topk_idx"])
    return int(np.asarray(counts)[list(reqs)].sum()) * acc.FLOPS_PER_QT


def cpu_baseline(w, host, budget_s: float):
    """The oracle timed on this host's cores over a bounded sample of the
    workload: whole requests, in order, until about budget_s seconds."""
    reqs, t0 = [], time.perf_counter()
    for b in range(w.batch):
        oracle_sample(w, host, [b])
        reqs.append(b)
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    fl = sample_flops(w, host, reqs)
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{len(reqs)} of {w.batch} requests (all {w.s_q} query tokens each), "
                      f"{dt:.1f} s, numpy fp64 with BLAS on all host cores"}


def run_reference(args, world, rank):
    if rank != 0:
        return
    import workloads as wl
    w = wl.make_config(args.config, device="cpu")
    host = wl.host_arrays(w)
    order = list(range(w.batch))
    for i in range(args.warmup):
        oracle_sample(w, host, [order[i % w.batch]])
    times, flops = [], 0
    t_all = time.perf_counter()
    for i in range(args.steps):
        b = order[i % w.batch]
        t0 = time.perf_counter()
        oracle_sample(w, host, [b])
        times.append(time.perf_counter() - t0)
        flops += sample_flops(w, host, [b])
    dt = time.perf_counter() - t_all
    val = flops / dt / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": args.config, "batch": w.batch, "s_q": w.s_q, "heads": 128,
                       "d_qk": 576, "d_v": 512, "page": 64, "causal": w.causal,
                       "step": "one request (all query tokens) of the workload per step"},
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"{args.steps} steps of one request each, cycling through "
                                       f"the {w.batch} requests"},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def kernel_name(w) -> str:
    # two query tokens over a dense bf16 cache take the paired-SM kernel; an
    # FP8 cache (and everything else) the one-token kernel
    return "mla_decode_mtp_kernel" if (w.s_q == 2 and not w.topk and not w.kv_fp8) else "mla_decode_kernel"


def time_step(m, w, args, dev, world, sampler=None):
    """Times plan + decode + combine on one resident workload.

    Host-launched steps with an event between kernels give the per-kernel
    split; the timed figure is a CUDA graph of the three calls, replayed
    (checked bit-identical to the host-launched output).  256 MB of L2 are
    flushed before every step, outside the events."""
    import torch

    B, s_q = w.batch, w.s_q
    ws = m.Workspace(B, s_q, args.num_units, dev)
    out = torch.empty((B, s_q, 128, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, s_q, 128), dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    topk = w.topk
    flags = (m.MLA_FLAG_CAUSAL if w.causal else 0) | (m.MLA_FLAG_BF16_PV if args.bf16_pv else 0)
    if w.kv_fp8:
        flags |= m.MLA_FLAG_KV_FP8
    U = ws.num_units

    # every call goes to the stream current at call time (the capture stream
    # while a CUDA graph of the step is recorded)
    def plan():
        m.mla_decode_plan(w.cache_lens, B, s_q, topk, U, ws.buf, ws.nbytes, torch.cuda.current_stream(dev))

    def decode():
        m.mla_decode(w.q, w.kv, w.num_pages, w.block_table, w.block_table.stride(0), w.cache_lens, B, s_q,
                     128, w.softmax_scale, w.topk_idx, topk, flags, U, ws.buf, ws.nbytes, out, lse,
                     torch.cuda.current_stream(dev))

    def combine():
        m.mla_combine(ws.buf, ws.nbytes, B, s_q, 128, flags, U, out, lse, torch.cuda.current_stream(dev))

    for _ in range(args.warmup):
        flush.zero_()
        plan(); decode(); combine()
    torch.cuda.synchronize()
    status = m.mla_workspace_status(ws.buf, stream.cuda_stream)
    if status != 0:
        raise RuntimeError(f"{w.name}: device status after warm-up: {m.mla_status_string(status)}")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()
        e = ev[i]
        e[0].record(stream)
        plan()
        e[1].record(stream)
        decode()
        e[2].record(stream)
        combine()
        e[3].record(stream)
    torch.cuda.synchronize()
    r = {"launch_ms": sum(e[0].elapsed_time(e[3]) for e in ev) / args.steps,
         "dec_ms": sum(e[1].elapsed_time(e[2]) for e in ev) / args.steps,
         "plan_ms": sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps,
         "comb_ms": sum(e[2].elapsed_time(e[3]) for e in ev) / args.steps,
         "num_units": U, "flags": flags}
    r["step_ms"] = r["launch_ms"]
    t_wall = time.perf_counter()
    if not args.no_graph:
        # the step as a serving loop runs it: plan + decode + combine recorded
        # once in a CUDA graph (the decode and combine kernels are programmatic
        # dependents of the kernel before them) and replayed
        ref_out, ref_lse = out.clone(), lse.clone()
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            plan(); decode(); combine()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(graph):
            plan(); decode(); combine()
        for _ in range(args.warmup):
            flush.zero_()
            graph.replay()
        torch.cuda.synchronize()
        evg = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        if sampler is not None:
            sampler.start()
            time.sleep(0.3)
        barrier(world)
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            evg[i][0].record(stream)
            graph.replay()
            evg[i][1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        r["step_ms"] = sum(e[0].elapsed_time(e[1]) for e in evg) / args.steps
        status = m.mla_workspace_status(ws.buf, stream.cuda_stream)
        if status != 0:
            raise RuntimeError(f"{w.name}: device status after the graph replays: {m.mla_status_string(status)}")
        if not (torch.equal(out, ref_out) and torch.equal(lse, ref_lse)):
            raise RuntimeError(f"{w.name}: graph replays changed the output of the step")
    r["wall_s"] = time.perf_counter() - t_wall
    r["ws"], r["out"], r["lse"] = ws, out, lse
    return r


def roofline_of(w, r, pk, pk_kind, step_ms):
    """Algorithmic work of the workload and its roofline figures: `roofline`
    for the attention kernel alone (its event time), `frac_roofline` for the
    whole call (plan + attention + combine)."""
    from mla_latent_kv_09_gb300 import accounting as acc
    host_lens = w.cache_lens.cpu().numpy()
    host_topk = None if w.topk_idx is None else w.topk_idx.cpu().numpy()
    flops = acc.step_flops(host_lens, w.s_q, w.causal, host_topk)
    nbytes = acc.step_bytes(host_lens, w.s_q, w.causal, host_topk,
                            row_bytes=acc.FP8_ROW_BYTES if w.kv_fp8 else acc.ROW_BYTES)
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    bound = "tensor" if flops / nbytes > ridge else "hbm"
    dec_s = r["dec_ms"] * 1e-3
    if bound == "tensor":
        achieved, peak, unit = flops / dec_s / 1e12, pk["bf16_tflops"], "TFLOP/s"
    else:
        achieved, peak, unit = nbytes / dec_s / 1e9, pk["hbm_gbs"], "GB/s"
    step_s = step_ms * 1e-3
    return {
        "flops": flops, "nbytes": nbytes, "bound": bound,
        "tflops": flops / step_s / 1e12, "hbm_gbs": nbytes / step_s / 1e9,
        "frac_tensor_peak": flops / step_s / 1e12 / pk["bf16_tflops"],
        "frac_hbm_peak": nbytes / step_s / 1e9 / pk["hbm_gbs"],
        "frac_roofline": max(flops / (pk["bf16_tflops"] * 1e12), nbytes / (pk["hbm_gbs"] * 1e9)) / step_s,
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "traffic": measured_traffic(w.name), "kernel": kernel_name(w),
                     "scope": "attention kernel alone (its CUDA-event time); frac_roofline covers the whole call",
                     "peak_source": f"{pk_kind} (burst)"},
    }


ABSORB_SOURCES = ["absorb_kernel.cu", "kernel_common.cuh", "common.cuh", "ptx.cuh"]
INDEXER_SOURCES = ["indexer_kernel.cu", "kernel_common.cuh", "common.cuh", "ptx.cuh"]


def indexer_traffic():
    """DRAM bytes per launch of the indexer scores kernel at the sparse
    workload's size, from the committed (scaled) ncu record, if it was taken
    on the current source (else None)."""
    path = os.path.join(ROOT, "profiles", "indexer_traffic.json")
    if not os.path.exists(path):
        return None
    h = hashlib.sha256()
    for f in INDEXER_SOURCES:
        h.update(open(os.path.join(ROOT, "mla_latent_kv_09_gb300", "csrc", f), "rb").read())
    e = json.load(open(path)).get("mla_indexer_scores_kernel/sparse_b80")
    if not e or e.get("kernel_hash") != h.hexdigest()[:16]:
        return None
    return e.get("dram_bytes_per_launch")


def absorb_hash() -> str:
    h = hashlib.sha256()
    for f in ABSORB_SOURCES:
        h.update(open(os.path.join(ROOT, "mla_latent_kv_09_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def absorb_traffic(kernel: str, tokens: int):
    """DRAM bytes per launch of an absorption kernel from a committed ncu
    capture on the current source (else None)."""
    path = os.path.join(ROOT, "profiles", "absorb_traffic.json")
    if not os.path.exists(path):
        return None
    e = json.load(open(path)).get(f"{kernel}/T{tokens}")
    if not e or e.get("kernel_hash") != absorb_hash():
        return None
    return e.get("dram_bytes_per_launch")


def time_absorb(m, args, dev, tokens: int, pk, pk_kind, with_cpu: bool):
    """The weight-absorption BMMs around the attention for one step of
    `tokens` (request, query token) pairs, 128 heads: each call timed alone
    with CUDA events, 256 MB of L2 flushed before every launch (the inputs,
    ~40 MB, would otherwise stay in L2)."""
    import torch

    import workloads as wl
    from mla_latent_kv_09_gb300 import accounting as acc

    inp = wl.make_absorb(tokens, seed=args.seed, device=dev)
    q_out = torch.empty((tokens, 128, 576), dtype=torch.bfloat16, device=dev)
    o_out = torch.empty((tokens, 128, 128), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    calls = {
        "q": (lambda: m.absorb_q(inp.q_nope, inp.w_uk, inp.q_pe, out=q_out, status=status, stream=stream),
              acc.absorb_q_flops(tokens), acc.absorb_q_bytes(tokens), "mla_absorb_q_kernel"),
        "o": (lambda: m.absorb_o(inp.o, inp.w_uv, out=o_out, status=status, stream=stream),
              acc.absorb_o_flops(tokens), acc.absorb_o_bytes(tokens), "mla_absorb_o_kernel"),
    }
    res = {"tokens": tokens, "heads": 128}
    n = max(args.steps, 20)
    for key, (fn, flops, nbytes, kname) in calls.items():
        for _ in range(max(args.warmup, 3)):
            flush.zero_()
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        torch.cuda.synchronize()
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        us = sum(a.elapsed_time(b) for a, b in ev) / n * 1e3
        gbs = nbytes / (us * 1e-6) / 1e9
        res[key] = {"us": us, "gflop": flops / 1e9, "algorithmic_mb": nbytes / 1e6, "tflops": flops / (us * 1e-6) / 1e12,
                    "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                                 "frac": gbs / pk["hbm_gbs"], "traffic": absorb_traffic(kname, tokens),
                                 "kernel": kname, "peak_source": f"{pk_kind} (burst)"}}
    if m.mla_workspace_status(status, stream.cuda_stream) != 0:
        raise RuntimeError("absorption kernels reported a device status")
    if with_cpu:
        import oracle
        t0 = time.perf_counter()
        oracle.absorb_q(wl.bf16_bits(inp.q_nope.contiguous()), wl.bf16_bits(inp.w_uk))
        oracle.absorb_o(wl.bf16_bits(inp.o), wl.bf16_bits(inp.w_uv))
        dt = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": dt * 1e6, "unit": "us for both calls", "cores": torch.get_num_threads(),
                               "kind": "oracle", "sample": f"both calls once at {tokens} tokens (fp64, numpy matmul)"}
    del inp, q_out, o_out, flush
    torch.cuda.empty_cache()
    return res


def time_indexer(m, args, dev, pk, pk_kind, with_cpu: bool):
    """The sparse-attention indexer on the sparse workload's shape (80
    requests of 65,536 cached tokens, one query token, top-2048): index
    scores, then the top-k lists, each timed alone with CUDA events and 256 MB
    of L2 flushed before every launch; the pair as one graph."""
    import numpy as np
    import torch

    import workloads as wl
    from mla_latent_kv_09_gb300 import accounting as acc

    w = wl.make_config("sparse_b80", seed=args.seed, device=dev)
    ix = wl.make_indexer(w, seed=args.seed)
    k = 2048
    B, s_q = w.batch, w.s_q
    max_len = w.block_table.shape[1] * 64
    scores = torch.empty((B, s_q, max_len), dtype=torch.float32, device=dev)
    lists = torch.empty((B, s_q, k), dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def f_scores():
        m.indexer_scores(ix.q_idx, ix.w_idx, ix.k_cache, w.block_table, w.cache_lens, scores=scores,
                         status=status, stream=torch.cuda.current_stream(dev))

    def f_topk():
        m.topk_indices(scores, w.cache_lens, k, out=lists, status=status, stream=torch.cuda.current_stream(dev))

    def timed(fn, n):
        for _ in range(max(args.warmup, 3)):
            flush.zero_()
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        torch.cuda.synchronize()
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev) / n * 1e3

    n = max(min(args.steps, 200), 20)
    us_s = timed(f_scores, n)
    us_k = timed(f_topk, n)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        f_scores(); f_topk()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        f_scores(); f_topk()
    us_g = timed(graph.replay, n)
    if m.mla_workspace_status(status, stream.cuda_stream) != 0:
        raise RuntimeError("indexer: a kernel reported a device status")
    lens = w.cache_lens.cpu().numpy()
    nbytes = acc.indexer_bytes(lens, s_q, False, k)
    key_bytes = int(lens.sum()) * 256
    gbs = key_bytes / (us_s * 1e-6) / 1e9
    res = {"workload": "sparse_b80 shape: 80 x 65536 cached tokens, 64 index heads x 128 dims, top-2048",
           "us_scores": us_s, "us_topk": us_k, "us_per_call": us_g,
           "algorithmic_mb": nbytes / 1e6, "gflop": acc.indexer_flops(lens, s_q, False) / 1e9,
           "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                        "frac": gbs / pk["hbm_gbs"], "traffic": indexer_traffic(),
                        "kernel": "mla_indexer_scores_kernel",
                        "scope": "scores kernel alone: index-key bytes / its event time",
                        "peak_source": f"{pk_kind} (burst)"},
           "frac_roofline_call": nbytes / (pk["hbm_gbs"] * 1e9) / (us_g * 1e-6),
           "launch": "scores and top-k each timed alone; us_per_call = CUDA graph of both"}
    if with_cpu:
        from oracle import indexer_oracle as io
        # request 0's own pages only (the whole pool would not fit the host as fp64)
        pages0 = w.block_table[0].long()
        kc = wl.bf16_bits(ix.k_cache[pages0])
        table0 = np.arange(pages0.numel(), dtype=np.int32)[None, :]
        q, wt = wl.bf16_bits(ix.q_idx[:1]), ix.w_idx[:1].cpu().numpy()
        t0 = time.perf_counter()
        io.indexer_topk(q, wt, kc, table0, lens[:1], k)
        dt = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": dt * 1e6 * B, "unit": "us per call (one request timed, x 80)",
                               "cores": torch.get_num_threads(), "kind": "oracle",
                               "sample": "indexer scores + top-2048 of one request of 65536 tokens (fp64 numpy)"}
    del w, ix, scores, lists, flush
    torch.cuda.empty_cache()
    return res


def time_layer(m, w, args, dev, ws):
    """The attention block of one decode step as a serving loop runs it: plan,
    query absorption (writing the attention's query in place), attention,
    combine and output absorption, recorded once in a CUDA graph and replayed
    with 256 MB of L2 flushed before every replay.  Random-init W_UK / W_UV
    of the model's shapes; the query projection output is synthetic."""
    import torch

    import workloads as wl

    B, s_q = w.batch, w.s_q
    T = B * s_q
    inp = wl.make_absorb(T, seed=args.seed + 1, device=dev)
    q = torch.empty((B, s_q, 128, 576), dtype=torch.bfloat16, device=dev)
    out = torch.empty((B, s_q, 128, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, s_q, 128), dtype=torch.float32, device=dev)
    o_proj_in = torch.empty((T, 128, 128), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flags = (m.MLA_FLAG_CAUSAL if w.causal else 0) | (m.MLA_FLAG_BF16_PV if args.bf16_pv else 0)
    U = ws.num_units

    def block():
        # the plan reads only the lengths, so it goes first: the query
        # absorption's weight loads then overlap it (programmatic dependent
        # launch), and the attention waits for the absorption, which waited
        # for the plan
        st = torch.cuda.current_stream(dev)
        m.mla_decode_plan(w.cache_lens, B, s_q, w.topk, U, ws.buf, ws.nbytes, st)
        m.absorb_q(inp.q_nope, inp.w_uk, inp.q_pe, out=q.view(T, 128, 576), status=status, stream=st)
        m.mla_decode(q, w.kv, w.num_pages, w.block_table, w.block_table.stride(0), w.cache_lens, B, s_q, 128,
                     w.softmax_scale, w.topk_idx, w.topk, flags, U, ws.buf, ws.nbytes, out, lse, st)
        m.mla_combine(ws.buf, ws.nbytes, B, s_q, 128, flags, U, out, lse, st)
        m.absorb_o(out.view(T, 128, 512), inp.w_uv, out=o_proj_in, status=status, stream=st)

    stream = torch.cuda.current_stream(dev)
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        block()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    ref = o_proj_in.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        block()
    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        graph.replay()
    n = max(args.steps, 20)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    torch.cuda.synchronize()
    for a, b in ev:
        flush.zero_()
        a.record(stream)
        graph.replay()
        b.record(stream)
    torch.cuda.synchronize()
    if m.mla_workspace_status(status, stream.cuda_stream) != 0 or m.mla_workspace_status(ws.buf, stream.cuda_stream):
        raise RuntimeError("attention block: a kernel reported a device status")
    if not torch.equal(o_proj_in, ref):
        raise RuntimeError("attention block: graph replays changed the output")
    us = sum(a.elapsed_time(b) for a, b in ev) / n * 1e3
    del inp, q, out, lse, o_proj_in, flush
    torch.cuda.empty_cache()
    return {"us_per_call": us, "tokens": T,
            "launch": "CUDA graph of plan, absorb_q, decode, combine, absorb_o (programmatic dependent launches)",
            "l2": "256 MB L2 flush before every replay"}


def run_ours(args, world, rank, local):
    import torch

    import mla_latent_kv_09_gb300 as m
    import workloads as wl
    from mla_latent_kv_09_gb300 import build as mbuild

    mbuild.build()
    m.load()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pk, pk_kind = peaks()

    # the other workloads first (one at a time, freed after), the headline last
    others = {}
    extra = [c for c in (args.also or "").split(",") if c and c not in (args.config, "none")]
    for name in extra:
        w = wl.make_config(name, seed=args.seed + rank, device=dev)
        r = time_step(m, w, args, dev, world)
        step_ms = max_over_ranks(r["step_ms"], world)
        rf = roofline_of(w, r, pk, pk_kind, step_ms)
        entry = {"batch": w.batch, "s_q": w.s_q, "causal": w.causal, "topk": w.topk, "num_units": r["num_units"],
                 "kv_cache": "fp8 (656-byte rows: E4M3 latent, UE8M0 group scales, bf16 RoPE)" if w.kv_fp8 else "bf16",
                 "us_per_call": step_ms * 1e3, "us_per_call_host_launches": r["launch_ms"] * 1e3,
                 "us_decode_kernel": r["dec_ms"] * 1e3, "us_plan": r["plan_ms"] * 1e3,
                 "us_combine": r["comb_ms"] * 1e3, "algorithmic_gflop": rf["flops"] / 1e9,
                 "algorithmic_mb": rf["nbytes"] / 1e6, "tflops": rf["tflops"], "hbm_gbs": rf["hbm_gbs"],
                 "frac_roofline": rf["frac_roofline"], "roofline": rf["roofline"]}
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            entry["cpu_baseline"] = cpu_baseline(w, wl.host_arrays(w), args.cpu_budget_other)
        others[name] = entry
        del w, r
        torch.cuda.empty_cache()

    # the absorption BMMs either side of the attention, at the headline
    # step's 128 tokens (64 requests x 2) and at the pages' bs = 64
    absorb = None
    if not args.no_absorb:
        absorb = {f"T{t}": time_absorb(m, args, dev, t, pk, pk_kind, rank == 0 and world == 1
                                       and not args.no_cpu_baseline) for t in (128, 64)}
        absorb["page_context"] = ("H800 estimates at bs=64 (context only): 10 us for the query-side and 8 us "
                                  "for the output-side BMM")

    indexer = None
    if not args.no_indexer:
        indexer = time_indexer(m, args, dev, pk, pk_kind, rank == 0 and world == 1 and not args.no_cpu_baseline)

    w = wl.make_config(args.config, seed=args.seed + rank, device=dev, batch=args.batch, length=args.length)
    B, s_q = w.batch, w.s_q
    sampler = ClockSampler(local)
    r = time_step(m, w, args, dev, world, sampler=sampler)
    clocks = sampler.stop()
    if absorb is not None:
        absorb["layer"] = time_layer(m, w, args, dev, r["ws"])
    step_ms_max = max_over_ranks(r["step_ms"], world)
    rf = roofline_of(w, r, pk, pk_kind, step_ms_max)
    flops = rf["flops"]
    value = world * flops / (step_ms_max * 1e-3) / 1e12
    ws, out, lse = r["ws"], r["out"], r["lse"]

    # end to end through the host-buffer API: inputs copied in, O/LSE copied out, every step
    e2e = None
    if not args.no_e2e:
        pin = {k: t.cpu().pin_memory() for k, t in
               [("q", w.q), ("kv_cache", w.kv), ("block_table", w.block_table), ("cache_lens", w.cache_lens)]
               + ([("topk_idx", w.topk_idx)] if w.topk_idx is not None else [])}
        dbuf = {"q": w.q, "kv_cache": w.kv, "block_table": w.block_table, "cache_lens": w.cache_lens,
                "topk_idx": w.topk_idx, "out": out, "lse": lse}
        o_h = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        l_h = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
        h2d = sum(t.numel() * t.element_size() for t in pin.values())
        d2h = o_h.numel() * o_h.element_size() + l_h.numel() * l_h.element_size()
        n_e2e = max(3, min(args.steps, args.e2e_steps))

        def e2e_step():
            m.decode_step_host(pin["q"], pin["kv_cache"], pin["block_table"], pin["cache_lens"],
                               w.softmax_scale, device=dev, causal=w.causal, topk_idx=pin.get("topk_idx"),
                               bf16_pv=args.bf16_pv, workspace=ws, dev_buffers=dbuf, out_host=o_h,
                               lse_host=l_h)

        for _ in range(3):
            e2e_step()
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            e2e_step()
        torch.cuda.synchronize()
        dt = max_over_ranks((time.perf_counter() - t0) / n_e2e, world)
        e2e = {"value": world * flops / dt / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "steps": n_e2e, "ms_per_step": 1e3 * dt}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, wl.host_arrays(w), args.cpu_budget)

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.config + ("" if args.batch is None and args.length is None else " (reduced)"),
                   "batch": B, "s_q": s_q, "heads": 128, "d_qk": 576, "d_v": 512,
                   "page": 64, "causal": w.causal, "topk": w.topk, "num_units": r["num_units"],
                   "value_product": "bf16 P and V" if args.bf16_pv else "fp16 P and V",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "256 MB L2 flush before every timed step; cache pool exceeds L2",
                   "algorithmic_gflop": flops / 1e9, "algorithmic_mb": rf["nbytes"] / 1e6},
        "us_per_call": step_ms_max * 1e3,
        "launch": "CUDA graph of plan + decode + combine, replayed" if not args.no_graph
                  else "plan, decode, combine launched from the host",
        "us_per_call_host_launches": r["launch_ms"] * 1e3,
        "us_decode_kernel": r["dec_ms"] * 1e3, "us_plan": r["plan_ms"] * 1e3, "us_combine": r["comb_ms"] * 1e3,
        "tflops": rf["tflops"], "hbm_gbs": rf["hbm_gbs"],
        "frac_tensor_peak": rf["frac_tensor_peak"], "frac_hbm_peak": rf["frac_hbm_peak"],
        "frac_roofline": rf["frac_roofline"],
        "roofline": rf["roofline"],
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "wall_s_timed_region": r["wall_s"],
        "other_workloads": others,
        "absorb": absorb,
        "indexer": indexer,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="mtp_b64")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--batch", type=int, default=None,
                    help="shrink the headline workload to this many requests (profiling runs)")
    ap.add_argument("--length", type=int, default=None,
                    help="shrink the headline workload's cache length (profiling runs)")
    ap.add_argument("--num-units", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="time the step from host launches instead of a CUDA graph replay")
    ap.add_argument("--bf16-pv", action="store_true",
                    help="two-token dense path: value product with bf16 P and V (MLA_FLAG_BF16_PV)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-indexer", action="store_true",
                    help="skip timing the sparse-attention indexer (scores + top-k)")
    ap.add_argument("--no-absorb", action="store_true",
                    help="skip timing the weight-absorption BMMs around the attention")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle work for the headline workload's CPU baseline")
    ap.add_argument("--cpu-budget-other", type=float, default=4.0,
                    help="seconds of oracle work for each other workload's CPU baseline")
    ap.add_argument("--also", default="single,uniform_b32,long_b128,sparse_b80,mtp4_b64,"
                                      "uniform_b32_fp8,long_b128_fp8,sparse_b80_fp8,mtp_b64_fp8",
                    help="other workloads timed before the headline one (comma-separated; 'none' for none)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
