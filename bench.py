#!/usr/bin/env python
"""Benchmark of one DSA layer step on GB300 (query-tokens/s per layer and the
roofline fraction of the dominant kernel).

A step is one call of the fused dsa_decode (indexer -> exact top-2048 ->
sparse MLA) over one batch, on one layer's paged caches.  Consecutive steps
rotate through `--layers` independent layer copies (by default as many as make
the rotated caches at least eight times the 129 MB L2, between 2 and 24 -- the
model has 24 full-attention layers), so that every step reads its caches from
HBM.

Default workload: agentic multi-token decode, 64 requests of 131072 positions
with 5 causal query tokens each (the largest decode batch).  `--config`
selects another: c0_tiny, c1_batched, c2_agentic, c3a_long_fp8,
c3b_long_mxfp4, c4_prefill_append.

Timing: every timed step is replayed from a captured CUDA graph (whatever
--steps is), with the graph pieces built before the timed region.

Arms
  --impl ours       (default) the CUDA library through its C ABI.
  --impl reference  the CPU oracle (plain fp64 C) as it stands, on the host
                    cores, on a bounded sample of the same workload.

Multi-GPU (torchrun, one process per GPU): replicas only -- each rank runs the
same workload on its own GPU with no data-path collective (weak scaling); the
timing takes the maximum over ranks.
"""
import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "DSA decode query-tokens/s per layer; achieved HBM GB/s vs GB300 roofline"
UNIT = "query-tokens/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1200)
    ap.add_argument("--warmup", type=int, default=24)
    ap.add_argument("--config", default="c2_agentic")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=0,
                    help="layer copies rotated step by step; 0 = enough for 8x the L2")
    ap.add_argument("--requests", type=int, default=0,
                    help="keep only the first N requests of the workload (profiling at a "
                         "smaller scale with the same per-request shape); 0 = all")
    ap.add_argument("--query-tokens", type=int, default=0,
                    help="keep the first N query tokens of each request, its context ending "
                         "at the last kept token (profiling at a smaller scale with the same "
                         "causal rows); 0 = all")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="bounded CPU-oracle sample for the cpu_baseline field")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--soak-seconds", type=float, default=1.5,
                    help="extra untimed replay while GPU clocks are sampled")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the NVFP4 / DCP / fused-front measurements")
    ap.add_argument("--batch-invariant", action="store_true",
                    help="run the sparse MLA under the batch-invariant plan (every token "
                         "whole; dsa_set_batch_invariant)")
    return ap.parse_args()


def cuda_runtime():
    """The CUDA runtime library through ctypes (for the end-to-end leg's
    copies and event waits), or None when it cannot be loaded."""
    for name in ("libcudart.so.13", "libcudart.so",
                 os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "lib64", "libcudart.so")):
        try:
            rt = ctypes.CDLL(name)
        except OSError:
            continue
        for fn in ("cudaSetDevice", "cudaMemcpyAsync", "cudaEventRecord", "cudaStreamWaitEvent"):
            getattr(rt, fn).restype = ctypes.c_int
        return rt
    return None


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def config_shape(name):
    import dsa_inputs as di
    lens, nq, fmt, seed = di.config_shape(name)
    q_counts = [nq] * len(lens) if isinstance(nq, int) else list(nq)
    return lens, q_counts, fmt, seed


# ---- CPU oracle (baseline and reference arm) --------------------------------

def oracle_step(layer, rows):
    import oracle
    ob = oracle.Batch(layer.q_offsets, layer.seq_lens, layer.block_table, layer.num_pages)
    t0 = time.perf_counter()
    oracle.decode(ob, layer.q8, layer.qscale, layer.w, layer.index_pages, layer.key_format,
                  layer.q_lat, layer.latent_pages, layer.kv_scale, layer.sm_scale, rows=rows)
    return time.perf_counter() - t0


def oracle_sample_layer(cfg, threads):
    """A bounded sample of the workload for the CPU oracle: the first requests
    of the batch (same per-request shape: context lengths, query tokens,
    causal rule, value recipe), enough of them to give every host thread a
    query row, built on the host.  The rate metric is per query token, so the
    sample measures it directly."""
    import dsa_inputs as di
    lens, q_counts, fmt, seed = config_shape(cfg)
    n, rows = 0, 0
    while n < len(lens) and rows < threads:
        rows += q_counts[n]
        n += 1
    lens, q_counts = lens[:n], q_counts[:n]
    return di.make_layer(lens, q_counts, fmt, seed), lens, q_counts


def cpu_baseline(cfg, seconds):
    """The oracle on the host cores: steps over the sample's query rows (in
    parallel over rows) until about `seconds` of CPU work."""
    import oracle
    threads = max(1, oracle.num_threads())
    layer, lens, q_counts = oracle_sample_layer(cfg, threads)
    T = sum(q_counts)
    rows_per_step = min(T, threads)
    done_rows, spent, steps = 0, 0.0, 0
    while spent < seconds and steps < 64:
        rows = [(done_rows + i) % T for i in range(rows_per_step)]
        spent += oracle_step(layer, rows)
        done_rows += rows_per_step
        steps += 1
    return {"value": done_rows / spent, "unit": UNIT,
            "cores": min(rows_per_step, threads), "kind": "oracle",
            "sample": "%d oracle step(s) of %d query rows (full indexer over the row's "
                      "context, top-2048, MLA), from the first %d request(s) of %s "
                      "(ctx %d..%d), %.1f s" % (steps, rows_per_step, len(lens), cfg,
                                               min(lens), max(lens), spent)}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    import oracle
    threads = max(1, oracle.num_threads())
    layer, lens, q_counts = oracle_sample_layer(args.config, threads)
    full_lens, full_q, _, _ = config_shape(args.config)
    T = sum(q_counts)
    rows_per_step = min(T, threads)
    # size each step so that warm-up + timed steps end within ~150 s
    probe = oracle_step(layer, list(range(rows_per_step)))
    budget = 150.0 / max(1, args.steps + args.warmup)
    while rows_per_step > 1 and probe > budget:
        rows_per_step = max(1, rows_per_step // 2)
        probe = oracle_step(layer, list(range(rows_per_step)))
    cursor = 0
    for _ in range(args.warmup):
        oracle_step(layer, [(cursor + i) % T for i in range(rows_per_step)])
        cursor += rows_per_step
    spent = 0.0
    for _ in range(args.steps):
        spent += oracle_step(layer, [(cursor + i) % T for i in range(rows_per_step)])
        cursor += rows_per_step
    rows = args.steps * rows_per_step
    value = rows / spent
    cores = min(rows_per_step, threads)
    sample = ("%d query rows per step (full indexer over the row's context, top-2048, MLA) "
              "from the first %d request(s) of %s" % (rows_per_step, len(lens), args.config))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * spent / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.config, "requests": len(full_lens),
                       "seq_lens": [min(full_lens), max(full_lens)],
                       "query_tokens": sum(full_q)},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---- clocks -----------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.path = tempfile.mktemp(prefix="dsa_clocks_", suffix=".csv")
        self.proc = None
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    sm.append(float(parts[0]))
                    mx.append(float(parts[1]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[4:8]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---- GPU arm ----------------------------------------------------------------

def job_elapsed(elapsed, world, device):
    """The job's time: the longest of the ranks' timed regions, returned on
    every rank (one all-reduce over the process group's backend: NCCL on the
    GPUs, gloo in the CPU tests)."""
    if world == 1:
        return elapsed
    import torch
    import torch.distributed as dist
    t = torch.tensor([elapsed], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world, tokens_per_rank, steps, elapsed):
    """Whole-job query tokens/s: every rank's tokens over the job's time
    (replicas, so per-rank work is fixed as ranks are added: weak scaling)."""
    return world * tokens_per_rank * steps / elapsed


# Sources each kernel's DRAM traffic depends on (its own file and the shared
# device headers): a recorded traffic figure is used only while these hash to
# the value it was measured at.
KERNEL_SOURCES = {
    "indexer": ["indexer_tc.cu", "common.cuh", "sm100.cuh"],
    "topk": ["topk.cu", "topk_rows.cu", "common.cuh", "sm100.cuh"],
    "sparse_mla": ["sparse_mla.cu", "common.cuh", "sm100.cuh"],
}


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dsa_sparse_attention_step_gb300", "csrc")
    for n in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, n), "rb") as f:
            h.update(n.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, cfg):
    """DRAM bytes (read + write) per full-size launch from a committed ncu
    summary, when it was measured on the kernel's current sources; else None.
    A capture of a smaller case carries `scale` (full launch / captured launch,
    by units processed) and is scaled here."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        e = rec[kernel][cfg]
        if e.get("measured_at_hash") != kernel_source_hash(kernel):
            return None
        return float(e["dram_bytes_per_captured_launch"]) * float(e.get("scale", 1.0))
    except Exception:
        return None


def auto_layers(lens, fmt, l2_bytes=129e6):
    """Layer copies to rotate: enough that the rotated caches exceed 8x the L2,
    at least 2 and at most 24 (the model's full-attention layer count)."""
    kb = 8448 if fmt == 0 else 4352
    per_layer = sum((s + 63) // 64 for s in lens) * (kb + 36864)
    n = int(-(-8 * l2_bytes // per_layer))
    return max(2, min(24, n))


def graph_pieces(first, n, L):
    """Split n consecutive steps starting at layer `first` into runs that each
    stay within one pass over the L layers: (start layer, length) pairs."""
    out = []
    i = first % L
    while n > 0:
        k = min(n, L - i)
        out.append((i, k))
        n -= k
        i = (i + k) % L
    return out


def run_ours(args, rank, world, local):
    import torch
    import torch.distributed as dist

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.config, args.cpu_seconds)

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    import dsa_inputs as di
    import dsa_sparse_attention_step_gb300 as dsa
    from dsa_sparse_attention_step_gb300 import workload as wl
    dsa.load()
    if args.batch_invariant:
        dsa.dsa_set_batch_invariant(True)

    lens, q_counts, fmt, seed = config_shape(args.config)
    if args.requests > 0:
        lens, q_counts = lens[:args.requests], q_counts[:args.requests]
    if args.query_tokens > 0:
        lens = [n - max(0, q - args.query_tokens) for n, q in zip(lens, q_counts)]
        q_counts = [min(q, args.query_tokens) for q in q_counts]
    T = sum(q_counts)
    L = args.layers if args.layers > 0 else auto_layers(lens, fmt)
    dev = torch.device("cuda", local)
    layers, batches = [], []
    for l in range(L):
        lay = di.make_layer(lens, q_counts, fmt, seed + 7919 * (l + 1) + 104729 * rank,
                            device=dev)
        layers.append(lay)
        batches.append(dsa.Batch(lay.q_offsets, lay.seq_lens, lay.block_table, lay.num_pages,
                                 lens, q_counts))
    cache_bytes = sum(l.index_pages.numel() + l.latent_pages.numel() for l in layers)
    # the step's outputs share one device buffer, so that the end-to-end leg
    # reads them back with one copy
    out_bytes = T * 96 * 512 * 2
    obuf = torch.empty(out_bytes + T * dsa.TOPK * 4, dtype=torch.uint8, device=dev)
    out = obuf[:out_bytes].view(torch.bfloat16).view(T, 96, 512)
    idx = obuf[out_bytes:].view(torch.int32).view(T, dsa.TOPK)
    lse = torch.empty(T, 96, dtype=torch.float32, device=dev)
    ws = torch.empty(dsa.dsa_decode_workspace_size(batches[0]), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    # prefill-append: a step first writes the new tokens' keys and latents into
    # the paged caches, then runs the step over them
    append = args.config == "c4_prefill_append"
    payloads = [di.append_payload(lay, seed + 31 * l) for l, lay in enumerate(layers)] if append else None

    def step(i, s=None):
        lay, b = layers[i % L], batches[i % L]
        if append:
            keys, lat = payloads[i % L]
            dsa.dsa_append_cache(b, keys, lat, lay.kv_scale, lay.index_pages, lay.latent_pages, fmt,
                                 status, stream=s)
        dsa.dsa_decode(b, lay.q8, lay.qscale, lay.w, lay.index_pages, fmt, lay.q_lat,
                       lay.latent_pages, lay.kv_scale, lay.sm_scale, dsa.TOPK, out, lse, idx,
                       ws, status, stream=s)

    # eager warm-up of every layer (module loading, lazy set-up), then graphs:
    # one per (start layer, length) piece, all captured before timing
    with torch.cuda.stream(stream):
        for i in range(L):
            step(i, stream)
    stream.synchronize()
    graphs = {}

    def graph(start, n):
        if (start, n) not in graphs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(start, start + n):
                    step(i, stream)
            graphs[(start, n)] = g
        return graphs[(start, n)]

    warm_pieces = graph_pieces(0, args.warmup, L)
    timed_pieces = graph_pieces(args.warmup, args.steps, L)
    for s0, n in warm_pieces + timed_pieces:
        graph(s0, n)

    def replay(pieces):
        with torch.cuda.stream(stream):
            for s0, n in pieces:
                graphs[(s0, n)].replay()

    replay(warm_pieces)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ev0.record(stream)
    replay(timed_pieces)
    ev1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    # graph replays do not pass through the library's launch counter: count
    # the kernels of one step by a direct call, then scale to the timed steps
    c0 = dsa.dsa_launch_count()
    with torch.cuda.stream(stream):
        step(0, stream)
    per_step_launches = dsa.dsa_launch_count() - c0
    gpu_launches = per_step_launches * args.steps
    elapsed = job_elapsed(ev0.elapsed_time(ev1) / 1000.0, world, dev)
    # keep the GPU busy a little longer while the clock sampler runs
    soak = graph_pieces(0, L, L)
    t_end = time.time() + args.soak_seconds
    while time.time() < t_end:
        replay(soak)
        torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    st = int(status.item())
    if st != 0:
        raise RuntimeError("device status %d (%s)" % (st, dsa.dsa_status_string(st)))
    del graphs

    # ---- per-kernel durations (graphs of L launches of one entry point) ----
    ld = ((max(lens) + 127) // 128) * 128
    scores = ws[:T * ld * 4].view(torch.float32).view(T, ld)
    kern = {}

    def time_graph(fn, reps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            for i in range(L):
                fn(i)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for i in range(L):
                fn(i)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            a.record(stream)
            for _ in range(reps):
                g.replay()
            b.record(stream)
        stream.synchronize()
        return a.elapsed_time(b) / 1000.0 / (reps * L)

    reps = max(3, min(200, args.steps // L))
    kern["indexer"] = time_graph(
        lambda i: dsa.dsa_index_scores(batches[i], layers[i].q8, layers[i].qscale, layers[i].w,
                                       layers[i].index_pages, fmt, scores, ld, status,
                                       stream=stream), reps)
    topk_ws = torch.empty(max(16, dsa.dsa_topk_workspace_size(batches[0])), dtype=torch.uint8,
                          device=dev)
    kern["topk"] = time_graph(
        lambda i: dsa.dsa_topk(batches[i], scores, ld, dsa.TOPK, idx, topk_ws, stream=stream),
        reps)
    mla_ws = torch.empty(max(16, dsa.dsa_sparse_mla_workspace_size(batches[0])),
                         dtype=torch.uint8, device=dev)
    kern["sparse_mla"] = time_graph(
        lambda i: dsa.dsa_sparse_mla(batches[i], layers[i].q_lat, layers[i].latent_pages,
                                     layers[i].kv_scale, layers[i].sm_scale, idx, dsa.TOPK, out,
                                     lse, mla_ws, status, stream=stream), reps)
    kbytes = {"indexer": wl.indexer_bytes(lens, q_counts, fmt),
              "topk": wl.topk_bytes(lens, q_counts),
              "sparse_mla": wl.mla_bytes(lens, q_counts)}
    dominant = max(kern, key=kern.get)
    hbm, bf16, src = peaks()
    hashes = {k: kernel_source_hash(k) for k in KERNEL_SOURCES}
    if args.config == "c4_prefill_append":
        # the prefill-append indexer is a dense causal FP8 GEMM: its roofline is
        # the FP8 tensor peak (the measured bf16 GEMM rate x the nominal 2x of
        # FP8 over bf16), for the indexer kernel alone; the kernel runs inside
        # a multi-millisecond step, so the sustained rate is reported as well
        dominant = "indexer"
        flops = wl.indexer_flops(lens, q_counts)
        fp8_peak = 2.0 * bf16
        achieved = flops / kern["indexer"] / 1e12
        sustained = None
        try:
            with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
                sustained = 2.0 * float(json.load(f)["bf16_tflops_sustained"])
        except Exception:
            pass
        roofline = {"bound": "tensor", "kernel": "indexer", "achieved": achieved,
                    "peak": fp8_peak, "unit": "TFLOP/s", "frac": achieved / fp8_peak,
                    "traffic": recorded_traffic("indexer", args.config),
                    "peak_source": src + " (bf16 GEMM burst x 2 for FP8)",
                    "frac_of_sustained": (achieved / sustained) if sustained else None,
                    "algorithmic_flops_per_launch": flops,
                    "avg_launch_us": kern["indexer"] * 1e6,
                    "kernels_us": {k: v * 1e6 for k, v in kern.items()},
                    "source_hashes": hashes}
    else:
        achieved = kbytes[dominant] / kern[dominant] / 1e9
        traffic = recorded_traffic(dominant, args.config)
        roofline = {"bound": "hbm", "kernel": dominant, "achieved": achieved, "peak": hbm,
                    "unit": "GB/s", "frac": achieved / hbm, "traffic": traffic,
                    "peak_source": src + " (burst copy)",
                    "algorithmic_bytes_per_launch": kbytes[dominant],
                    "avg_launch_us": kern[dominant] * 1e6,
                    "kernels_us": {k: v * 1e6 for k, v in kern.items()},
                    "kernels_frac": {k: kbytes[k] / kern[k] / 1e9 / hbm for k in kern},
                    "source_hashes": hashes}

    # ---- the other rows of the path, on the same workload --------------------
    extras = None
    if rank == 0 and not args.no_extras and not append:
        extras = measure_extras(args, dsa, di, wl, lens, q_counts, fmt, seed, L, layers, batches,
                                scores, ld, idx, stream, time_graph, hbm, bf16)

    # ---- end to end through the public API with host buffers --------------
    # per step: one pinned-host -> device copy of the step's inputs (queries
    # and request metadata packed in one staging buffer), the step, and one
    # device -> pinned-host copy of its outputs (attention output and indices).
    # The copies run on their own streams, double-buffered, so that step i's
    # outputs go back and step i + 1's inputs come in while step i + 1 (resp.
    # step i) computes, as an engine pipelines them.
    e2e = None
    if rank == 0:
        def pack(tensors):
            offs, o = [], 0
            for t in tensors:
                offs.append(o)
                o += (t.numel() * t.element_size() + 255) // 256 * 256
            buf = torch.empty(o, dtype=torch.uint8).pin_memory()
            for t, off in zip(tensors, offs):
                n = t.numel() * t.element_size()
                buf[off:off + n].copy_(t.contiguous().view(-1).view(torch.uint8))
            return buf, offs

        def host_inputs(j):
            lay = layers[j]
            ts = [lay.q8, lay.qscale, lay.w, lay.q_lat, lay.q_offsets, lay.seq_lens,
                  lay.block_table]
            if append:
                ts += list(payloads[j])
            return [t.cpu() for t in ts]

        hin = [pack(host_inputs(j)) for j in range(L)]
        shapes = [(t.dtype, tuple(t.shape)) for t in host_inputs(0)]
        nbytes_in = hin[0][0].numel()
        offs = hin[0][1]
        # two device staging slots, alternated step by step
        din = [torch.empty(nbytes_in, dtype=torch.uint8, device=dev) for _ in range(2)]

        def views(buf):
            v = []
            for (dt, shp), off in zip(shapes, offs):
                n = 1
                for d in shp:
                    n *= d
                esz = torch.empty(0, dtype=dt).element_size()
                v.append(buf[off:off + n * esz].view(dt).view(shp))
            return v

        dviews = [views(b) for b in din]
        dbatch = [dsa.Batch(v[4], v[5], v[6], layers[0].num_pages, lens, q_counts)
                  for v in dviews]
        # two output slots (attention output and indices in one buffer each)
        obufs = [obuf, torch.empty_like(obuf)]
        oviews = [(ob[:out_bytes].view(torch.bfloat16).view(T, 96, 512),
                   ob[out_bytes:].view(torch.int32).view(T, dsa.TOPK)) for ob in obufs]
        houts = [torch.empty(obuf.numel(), dtype=torch.uint8).pin_memory() for _ in range(2)]
        h2d = nbytes_in
        d2h = obuf.numel()
        s_in = torch.cuda.Stream(device=dev)
        s_out = torch.cuda.Stream(device=dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]     # slot's inputs on the device
        ev_done = [torch.cuda.Event() for _ in range(2)]   # slot's step finished
        ev_out = [torch.cuda.Event() for _ in range(2)]    # slot's outputs back on the host
        for e in ev_in + ev_done + ev_out:
            e.record(stream)
        # the step as a user's serving loop issues it: the library's calls
        # prepared once per (layer, slot), the copies and event waits as plain
        # CUDA runtime calls on the same streams and events
        calls = [[dsa.prepare_decode(dbatch[slot], dviews[slot][0], dviews[slot][1],
                                     dviews[slot][2], layers[j].index_pages, fmt, dviews[slot][3],
                                     layers[j].latent_pages, layers[j].kv_scale,
                                     layers[j].sm_scale, dsa.TOPK, oviews[slot][0], lse,
                                     oviews[slot][1], ws, status, stream=stream)
                  for slot in range(2)] for j in range(L)]
        acalls = [[dsa.prepare_append_cache(dbatch[slot], dviews[slot][7], dviews[slot][8],
                                            layers[j].kv_scale, layers[j].index_pages,
                                            layers[j].latent_pages, fmt, status, stream=stream)
                   for slot in range(2)] for j in range(L)] if append else None
        rt = cuda_runtime()
        if rt is not None and rt.cudaSetDevice(ctypes.c_int(dev.index or 0)) != 0:
            rt = None

        def e2e_step_rt(i):
            j = i % L
            slot = i % 2
            h_in, h_done, h_out = rt_ev_in[slot], rt_ev_done[slot], rt_ev_out[slot]
            ok = (rt.cudaStreamWaitEvent(rt_s_in, h_done, 0) == 0 and
                  rt.cudaMemcpyAsync(rt_din[slot], rt_hin[j], rt_nin, 1, rt_s_in) == 0 and
                  rt.cudaEventRecord(h_in, rt_s_in) == 0 and
                  rt.cudaStreamWaitEvent(rt_s, h_in, 0) == 0 and
                  rt.cudaStreamWaitEvent(rt_s, h_out, 0) == 0)
            if append:
                acalls[j][slot]()
            calls[j][slot]()
            ok = ok and (rt.cudaEventRecord(h_done, rt_s) == 0 and
                         rt.cudaStreamWaitEvent(rt_s_out, h_done, 0) == 0 and
                         rt.cudaMemcpyAsync(rt_hout[slot], rt_obuf[slot], rt_nout, 2, rt_s_out) == 0 and
                         rt.cudaEventRecord(h_out, rt_s_out) == 0)
            if not ok:
                raise RuntimeError("CUDA runtime call failed in the end-to-end step")

        if rt is not None:
            vp, sz = ctypes.c_void_p, ctypes.c_size_t
            rt_s, rt_s_in, rt_s_out = (vp(x.cuda_stream) for x in (stream, s_in, s_out))
            rt_ev_in = [vp(e.cuda_event) for e in ev_in]
            rt_ev_done = [vp(e.cuda_event) for e in ev_done]
            rt_ev_out = [vp(e.cuda_event) for e in ev_out]
            rt_din = [vp(b.data_ptr()) for b in din]
            rt_hin = [vp(h[0].data_ptr()) for h in hin]
            rt_hout = [vp(b.data_ptr()) for b in houts]
            rt_obuf = [vp(b.data_ptr()) for b in obufs]
            rt_nin, rt_nout = sz(nbytes_in), sz(obuf.numel())

        def e2e_step_torch(i):
            j = i % L
            slot = i % 2
            lay = layers[j]
            # inputs: once the step that last used this slot has finished
            s_in.wait_event(ev_done[slot])
            with torch.cuda.stream(s_in):
                din[slot].copy_(hin[j][0], non_blocking=True)
            ev_in[slot].record(s_in)
            stream.wait_event(ev_in[slot])
            stream.wait_event(ev_out[slot])  # the slot's previous outputs have left
            v = dviews[slot]
            o_att, o_idx = oviews[slot]
            if append:
                dsa.dsa_append_cache(dbatch[slot], v[7], v[8], lay.kv_scale,
                                     lay.index_pages, lay.latent_pages, fmt, status, stream=stream)
            # the block table copied in belongs to layer j's pools
            dsa.dsa_decode(dbatch[slot], v[0], v[1], v[2], lay.index_pages, fmt, v[3],
                           lay.latent_pages, lay.kv_scale, lay.sm_scale, dsa.TOPK, o_att, lse,
                           o_idx, ws, status, stream=stream)
            ev_done[slot].record(stream)
            s_out.wait_event(ev_done[slot])
            with torch.cuda.stream(s_out):
                houts[slot].copy_(obufs[slot], non_blocking=True)
            ev_out[slot].record(s_out)

        e2e_step = e2e_step_rt if rt is not None else e2e_step_torch
        for i in range(max(3, min(args.warmup, 2 * L))):
            e2e_step(i)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for ev in ev_done + ev_out:  # the first steps may start at once
            ev.record(stream)
        n_e2e = max(1, min(args.steps, 480))
        for i in range(n_e2e):
            e2e_step(i)
        for ev in ev_out:  # the last outputs are on the host
            stream.wait_event(ev)
        b.record(stream)
        torch.cuda.synchronize()
        te = a.elapsed_time(b) / 1000.0
        e2e = {"value": T * n_e2e / te, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "note": "per step: one pinned H2D copy of the packed queries and metadata" +
                       (" and the new tokens' keys and latents, dsa_append_cache" if append else "") +
                       ", dsa_decode (eager launches through the C ABI, arguments prepared "
                       "once per layer and slot), one D2H copy of output and indices; copies "
                       "on their own streams, double-buffered (step i's results return and "
                       "step i+1's inputs arrive while a step computes); caches resident" +
                       ("" if rt is not None else "; copies and event waits through PyTorch")}

    if rank == 0:
        step_b = wl.step_bytes(lens, q_counts, fmt)
        value = job_value(world, T, args.steps, elapsed)
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1000.0 * elapsed / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "fp8/bf16->fp32",
                "data": "synthetic",
                "config": {"workload": args.config, "requests": len(lens),
                           "seq_lens": [min(lens), max(lens)], "query_tokens": T,
                           "layers_rotated": L, "cache_bytes_rotated": cache_bytes,
                           "l2": "inputs larger than L2: %d layer copies, %.2f GB of caches "
                                 "rotated" % (L, cache_bytes / 1e9),
                           "timing": "CUDA graphs of the timed steps, replayed back to back",
                           "step": "dsa_append_cache + dsa_decode" if args.config == "c4_prefill_append"
                                   else "dsa_decode",
                           "parallelism": "replicas" if world > 1 else "single",
                           "mla_plan": "batch-invariant (every token whole)"
                                       if args.batch_invariant else "default (split last wave)"},
                "step_hbm_gbs": step_b / (elapsed / args.steps) / 1e9,
                "step_frac": step_b / (elapsed / args.steps) / 1e9 / hbm,
                "step_bytes": step_b,
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "extras": extras,
                "gpu_launches": gpu_launches, "clocks": clocks}
        print(json.dumps(line))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def measure_extras(args, dsa, di, wl, lens, q_counts, fmt, seed, L, layers, batches, scores, ld,
                   idx, stream, time_graph, hbm, bf16):
    """Per-launch times of the other rows of the path on the bench workload,
    each timed like the step's kernels (graphs of L launches, CUDA events):
    sparse MLA over NVFP4 latents, the DCP merge for W = 8 ranks with the
    per-rank attention and LSE combine, and the fused indexer front."""
    import torch
    dev = scores.device
    T = sum(q_counts)
    reps = max(3, min(50, args.steps // L))
    out = {}
    # NVFP4 latents: same requests and page placement, 352-B latent pages
    nv = [di.make_layer(lens, q_counts, fmt, seed + 7919 * (l + 1), device=dev,
                        latent_format=di.LATENT_NVFP4) for l in range(L)]
    o = torch.empty(T, 96, 512, dtype=torch.bfloat16, device=dev)
    ls = torch.empty(T, 96, dtype=torch.float32, device=dev)
    mws = torch.empty(max(16, dsa.dsa_sparse_mla_workspace_size(batches[0])), dtype=torch.uint8,
                      device=dev)
    t_nv = time_graph(lambda i: dsa.dsa_sparse_mla_ex(
        batches[i], nv[i].q_lat, nv[i].latent_pages, dsa.LATENT_NVFP4, nv[i].kv_scale,
        nv[i].sm_scale, idx, dsa.TOPK, o, ls, mws, stream=stream), reps)
    b_nv = wl.mla_bytes(lens, q_counts, wl.NVFP4_LATENT_BYTES)
    out["sparse_mla_nvfp4"] = {"us": t_nv * 1e6, "algorithmic_bytes": b_nv,
                               "gbs": b_nv / t_nv / 1e9, "frac_of_hbm": b_nv / t_nv / 1e9 / hbm}
    del nv
    # DCP, W = 8: candidate merge on the step's scores, then per-rank attention
    W = 8
    if max(lens) <= 65536 * W:
        cand = -(-3 * dsa.TOPK // (2 * W))
        didx = torch.empty(T, dsa.TOPK, dtype=torch.int32, device=dev)
        ridx = torch.empty(W, T, dsa.TOPK, dtype=torch.int32, device=dev)
        res = torch.zeros(T, W, dtype=torch.int32, device=dev)
        dws = torch.empty(dsa.dsa_dcp_topk_workspace_size(batches[0], W), dtype=torch.uint8,
                          device=dev)
        # the scores buffer holds the last layer's rows
        j = L - 1
        t_merge = time_graph(lambda i: dsa.dsa_dcp_topk(batches[j], scores, ld, W, 0, dsa.TOPK,
                                                        didx, ridx, res, dws, stream=stream), reps)
        parts = torch.empty(W, T, 96, 512, dtype=torch.bfloat16, device=dev)
        plse = torch.empty(W, T, 96, dtype=torch.float32, device=dev)

        def attend(i):
            for r in range(W):
                dsa.dsa_sparse_mla(batches[j], layers[j].q_lat, layers[j].latent_pages,
                                   layers[j].kv_scale, layers[j].sm_scale, ridx[r], dsa.TOPK,
                                   parts[r], plse[r], mws, stream=stream)
            dsa.dsa_lse_combine(T, W, parts, plse, o, ls, stream=stream)
        t_att = time_graph(attend, max(3, reps // 4))
        ex_c, ex_g = wl.dcp_exchange_bytes(W, cand)
        out["dcp8"] = {"merge_us": t_merge * 1e6, "attention_and_combine_us": t_att * 1e6,
                       "resent_row_rank_fraction": float(res.float().mean().item()),
                       "exchange_bytes_per_row": ex_c, "generic_merge_bytes_per_row": ex_g,
                       "exchange_reduction": ex_g / ex_c,
                       "note": "W ranks emulated on one GPU: the exchange is a device buffer"}
    # fused indexer front for the workload's T tokens (synthetic projections)
    g = torch.Generator(device=dev).manual_seed(seed)
    mk = lambda *sh, k: (torch.randn(*sh, generator=g, device=dev) / k ** 0.5).to(torch.bfloat16)
    q_c = torch.randn(T, wl.FRONT_QLAT, generator=g, device=dev).to(torch.bfloat16)
    x = torch.randn(T, wl.FRONT_HIDDEN, generator=g, device=dev).to(torch.bfloat16)
    w_q, w_k, w_w = mk(4096, wl.FRONT_QLAT, k=wl.FRONT_QLAT), mk(128, wl.FRONT_HIDDEN, k=wl.FRONT_HIDDEN), \
        mk(32, wl.FRONT_HIDDEN, k=wl.FRONT_HIDDEN)
    q8 = torch.empty(T, 32, 128, dtype=torch.uint8, device=dev)
    qs = torch.empty(T, 32, dtype=torch.float32, device=dev)
    ww = torch.empty(T, 32, dtype=torch.float32, device=dev)
    pages = layers[0].index_pages.clone() if fmt == di.KEYS_FP8 else None
    t_front = time_graph(lambda i: dsa.dsa_indexer_front(batches[0], q_c, x, w_q, w_k, w_w, q8, qs,
                                                         ww, pages, fmt, stream=stream), reps)
    fb, ff = wl.front_bytes(T), wl.front_flops(T)
    out["indexer_front"] = {"us": t_front * 1e6, "algorithmic_bytes": fb, "flops": ff,
                            "frac_of_hbm": fb / t_front / 1e9 / hbm,
                            "frac_of_bf16_tensor": ff / t_front / 1e12 / bf16}
    return out


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    return run_ours(args, rank, world, local)


if __name__ == "__main__":
    sys.exit(main())
