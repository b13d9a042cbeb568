"""Benchmark of the H2O heavy-hitter KV-cache hot path on GB300.

One step = the whole hot path over one batch of synthetic input: prefill of the
prompt (causal attention, column-sum scores, top-h + recent selection,
compaction into the cache) followed by every decode step of the workload
(attention over the cache, score accumulation, eviction, slot overwrite), the
decode steps replayed from one CUDA graph. The metric is decode tokens per
second: batch x decode steps per step, divided by the step's time (prefill
included).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                  [--kv bf16|fp8] [--layout slots|ring] [--batch B] [--layers L] [--quick]

--batch / --layers shrink a workload (same shapes otherwise) and --quick skips
every measurement but the timed step; both are for small profiler captures,
and the line's config then names the change.

With --gpus N > 1 (launched by torchrun) every rank runs its own full-size
batch (independent sequences; no collective on the data path) and the time is
the maximum over ranks.

--impl reference times the CPU oracle (fp64, one process per host core) on a
bounded sample of rows of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import multiprocessing as mp
import os
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import (WORKLOADS, decode_bytes_per_row_step, head_direction,  # noqa: E402
                       prefill_bytes_per_row, prefill_flops_per_row, row_tokens)

METRIC = "H2O decode tokens/s/GPU at 20% KV budget; achieved HBM GB/s vs peak"
UNIT = "tokens/s"
PREFILL_LAUNCHES = 5  # reset, forward, column sums, select, gather
ORACLE_ROW_BLOCK = 1024  # query rows per block of the oracle's prefill


# --------------------------------------------------------------------------- CPU oracle leg
def _oracle_rows_timed(job):
    """Pool worker: runs the oracle on a list of rows; returns the compute seconds."""
    os.environ["OPENBLAS_NUM_THREADS"] = "1"
    import oracle
    from workloads import bf16_bits_to_f64

    w, rows_bits = job
    t0 = time.perf_counter()
    for q, k, v in rows_bits:
        # row_block bounds the oracle's memory (a T x T block per call otherwise)
        oracle.run_row(bf16_bits_to_f64(q), bf16_bits_to_f64(k), bf16_bits_to_f64(v), w.prompt,
                       w.steps, w.h, w.r, row_block=ORACLE_ROW_BLOCK, keep_sets=False)
    return time.perf_counter() - t0


def _oracle_row_flops(w):
    """Rough fp64 work of one oracle row: causal prefill plus the decode steps."""
    return 4 * w.head_dim * w.prompt * w.prompt + 4 * w.steps * w.k * w.head_dim


def _sample_rows(w, n):
    rng = np.random.default_rng(12345)
    idx = rng.choice(w.batch * w.heads, size=min(n, w.batch * w.heads), replace=False)
    return [(int(i) // w.heads, int(i) % w.heads) for i in sorted(idx)]


class OracleTimer:
    """Times the CPU oracle on sampled rows with one spawn process per core."""

    def __init__(self, w, rows_per_core=None):
        self.w = w
        if rows_per_core is None:  # about 10-30 s of oracle work per run
            rows_per_core = 2 if _oracle_row_flops(w) < 1e11 else 1
        self.cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
        self.pool = mp.get_context("spawn").Pool(self.cores)
        rows = _sample_rows(w, rows_per_core * self.cores)
        self.rows = rows
        bits = [row_tokens(w, 0, b, j, head_direction(w, 0, j)) for b, j in rows]
        self.jobs = [(w, bits[i::self.cores]) for i in range(self.cores) if bits[i::self.cores]]

    def run_once(self):
        t0 = time.perf_counter()
        self.pool.map(_oracle_rows_timed, self.jobs, chunksize=1)
        wall = time.perf_counter() - t0
        return self.tokens() / wall, wall

    def tokens(self):
        """Decode tokens the sampled rows stand for: a token passes through every
        head of every layer, so it is rows / (heads x layers) x steps."""
        w = self.w
        return len(self.rows) / (w.heads * w.layers) * w.steps

    def describe(self):
        w = self.w
        return (f"{len(self.rows)} of {w.batch * w.heads} (batch, head) rows of {w.name}, each a full "
                f"prefill of {w.prompt} tokens plus {w.steps} decode steps; tokens counted as "
                f"rows / (heads x layers) x steps")

    def close(self):
        self.pool.close()
        self.pool.join()


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of the SM clock and the throttle reasons, every 25 ms,
    over a window that spans the warm-up and the timed region; the samples
    taken inside the timed region (host wall-clock bounds) are reported apart."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device_index: int):
        self.proc = None
        self.dev = device_index
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "25"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def mark(self, t0: float, t1: float):
        """Host wall-clock bounds (time.time()) of the timed region."""
        self.t0, self.t1 = t0, t1

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return self.summarize(out)

    def summarize(self, out: str):
        """The clock record of nvidia-smi's CSV lines (FIELDS, no header, no
        units): median and minimum SM clock and the throttle reasons seen,
        over the samples inside the timed region when there are at least 3."""
        import datetime
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]),
                             {n for n, v in zip(self.NAMES, parts[5:9]) if v.lower().startswith("active")}))
            except ValueError:
                continue
        if not rows:
            return None
        inside = [r for r in rows if self.t0 is not None and self.t0 <= r[0] <= self.t1]
        use = inside if len(inside) >= 3 else rows
        reasons = set().union(*(r[3] for r in use))
        return {"sm_mhz": float(np.median([r[1] for r in use])),
                "sm_max_mhz": max(r[2] for r in rows), "reasons": sorted(reasons),
                "samples": len(use), "samples_in_timed_region": len(inside),
                "window": "timed region" if use is inside else "warm-up and timed region",
                "sm_mhz_min": float(min(r[1] for r in use)), "interval_ms": 25}


# --------------------------------------------------------------------------- helpers
def _peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


DECODE_SOURCES = ("decode.cu", "decode_kernel.cuh")  # the per-step decode kernel's source


def _profiled_traffic(kernel_files, workload: str, rows: int, root: str = ROOT):
    """DRAM bytes per launch of `rows` rows from a committed ncu summary, if it
    was taken on the current source of the kernel (the sha256 of its files,
    concatenated in order, is recorded in the summary). The summary states the
    rows its figure is for; a row reads only its own cache, so the traffic is
    scaled in proportion to the rows."""
    path = os.path.join(root, "profiles", f"decode_kernel_{workload}.md")
    try:
        txt = open(path).read()
    except OSError:
        return None
    m = re.search(r"source_sha256[^:\n]*:\s*([0-9a-f]{64})", txt)
    b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not (m and b):
        return None
    src = b"".join(open(os.path.join(root, "h2o_heavy_hitter_gb300", "csrc", f), "rb").read()
                   for f in kernel_files)
    if hashlib.sha256(src).hexdigest() != m.group(1):
        return None
    r = re.search(r"traffic_rows:\s*([0-9]+)", txt)
    return float(b.group(1)) * (rows / int(r.group(1)) if r else 1.0)


def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_layer_seed(rank: int) -> int:
    """Layer index used to seed a rank's inputs: every rank draws an independent batch."""
    return rank


def max_over_ranks(value: float, pg, device=None) -> float:
    """Maximum of a per-rank value over all ranks (identity without a process group)."""
    if pg is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- reference arm
def run_reference(args, w):
    ws, rank, _ = _dist_env()
    if rank != 0:
        return
    timer = OracleTimer(w, rows_per_core=1)
    try:
        for _ in range(args.warmup):
            timer.run_once()
        vals, walls = [], []
        for _ in range(args.steps):
            v, wall = timer.run_once()
            vals.append(v)
            walls.append(wall)
    finally:
        timer.close()
    value = float(timer.tokens() * args.steps / sum(walls))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(walls) / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": _config(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": timer.cores, "kind": "oracle",
                         "sample": timer.describe()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


MAX_DISTINCT_ROWS = 512    # distinct seeded rows per input layer; larger batches repeat them
MAX_DISTINCT_LAYERS = 2    # distinct seeded input layers; deeper stacks cycle through them
L2_FALLBACK_BYTES = 129 << 20
MAX_CYCLED_LAYERS = 64     # tiny caches stay latency-bound; they are not cycled


def _layer_cache_bytes(w, kv="bf16"):
    """Device bytes of one layer's cache: K, V (bf16, or E4M3 codes plus two fp32
    scales), score (fp32), position (int32)."""
    per_slot = 4 * w.head_dim + 8 if kv == "bf16" else 2 * w.head_dim + 16
    return w.rows_per_layer * w.k * per_slot


def _default_steps(w):
    """Timed steps so that the timed region stays within about 20 s (3 .. 200)."""
    est = (w.layers * w.steps * decode_bytes_per_row_step(w.k, w.head_dim) * w.rows_per_layer / 4e12
           + w.layers * prefill_flops_per_row(w.prompt, w.head_dim) * w.rows_per_layer / 3e14)
    return int(max(3, min(200, 20.0 / max(est, 1e-9))))


def _data_desc(w):
    rows, layers = w.rows_per_layer, w.layers
    s = "synthetic: seeded N(0,1) q/k/v plus a power-law shared key direction per head; no weights"
    if rows > MAX_DISTINCT_ROWS:
        s += f"; {MAX_DISTINCT_ROWS} distinct seeded rows per layer, repeated over the {rows} rows"
    if layers > MAX_DISTINCT_LAYERS:
        s += (f"; {MAX_DISTINCT_LAYERS} distinct seeded input layers cycled over the {layers} "
              "layers (each layer keeps its own cache)")
    return s


def _config(w, l2_bytes=L2_FALLBACK_BYTES, kv="bf16"):
    cache = _layer_cache_bytes(w, kv) * w.layers
    l2 = ("inputs larger than L2 (prompt Q/K/V read every step); "
          + ("the decode caches of all layers exceed L2" if cache > l2_bytes else
             "the decode cache fits in L2 and stays resident across the decode steps of a step "
             "(roofline.achieved is measured with the caches of several layers cycled through "
             "L2, as a deep model's are; roofline.achieved_in_step is the L2-resident figure)"))
    return {"workload": w.name, "layers": w.layers, "batch": w.batch, "heads": w.heads,
            "head_dim": w.head_dim, "prompt": w.prompt, "decode_steps": w.steps, "h": w.h, "r": w.r,
            "zipf_alpha": w.alpha,
            "step": (f"prefill of {w.prompt} tokens for each of {w.layers} layer(s), then "
                     f"{w.steps} decode steps through every layer (one CUDA graph)"),
            "tokens_per_step": w.batch * w.steps,
            "l2": l2, "parallelism": "one replica per GPU (independent batches)"}


def _gen_layer(w, seed_layer):
    """bf16 bits [3, B, H, N, d] of one input layer (rows beyond MAX_DISTINCT_ROWS repeat)."""
    B, H, N, d = w.batch, w.heads, w.tokens, w.head_dim
    bits = np.empty((3, B * H, N, d), dtype=np.uint16)
    dirs = [head_direction(w, seed_layer, j) for j in range(H)]
    nd = min(B * H, MAX_DISTINCT_ROWS)
    for i in range(nd):
        b, j = divmod(i, H)
        bits[:, i] = np.stack(row_tokens(w, seed_layer, b, j, dirs[j]))
    for i in range(nd, B * H):
        bits[:, i] = bits[:, i % nd]
    return bits.reshape(3, B, H, N, d)


# --------------------------------------------------------------------------- our arm
def _end_to_end(args, ctx, graph, L, S, dp, ds, hp, hs, dec_out, stream, prefill_all, capture,
                barrier, pg, dev):
    """The step through the public API with host buffers: every step copies its
    inputs (the prompts and the decode steps' q, k, v) from pinned host memory
    and reads its result -- the decode outputs of the last layer -- back into
    pinned host memory (the prefill's attention output would feed the next
    model layer on the device). Two device input sets and separate copy streams
    let step i's copies overlap the neighbouring steps' compute. Returns
    (milliseconds for the timed steps, timed steps)."""
    import torch
    h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    sets = [(dp, ds, dec_out, graph)]
    dp2 = [[torch.empty_like(x) for x in lay] for lay in dp]
    ds2 = [[torch.empty_like(x) for x in lay] for lay in ds]
    out2 = torch.empty_like(dec_out)
    with torch.cuda.stream(stream):
        prefill_all(ctx, L, dp2)
        sets.append((dp2, ds2, out2, capture(ctx, L, S, ds2, out2)))
    h_out = [torch.empty(dec_out.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    copied = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    read = [torch.cuda.Event() for _ in range(2)]
    torch.cuda.synchronize()

    def e2e_step(i):
        b = i % 2
        pdev, sdev, odev, g_b = sets[b]
        if i >= 2:
            h2d_s.wait_event(done[b])  # step i - 2 no longer reads this input set
        with torch.cuda.stream(h2d_s):
            for dl, hl in zip(pdev + sdev, hp + hs):
                for dst, src in zip(dl, hl):
                    dst.copy_(src, non_blocking=True)
            copied[b].record(h2d_s)
        stream.wait_event(copied[b])
        if i >= 2:
            stream.wait_event(read[b])  # step i - 2's result has been read out
        with torch.cuda.stream(stream):
            prefill_all(ctx, L, pdev)
            g_b.replay()
            done[b].record(stream)
        d2h_s.wait_event(done[b])
        with torch.cuda.stream(d2h_s):
            h_out[b].copy_(odev, non_blocking=True)
            read[b].record(d2h_s)

    e2e_steps = max(4, args.steps // 4)
    for i in range(2):  # warm both input sets
        e2e_step(i)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(h2d_s)
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(d2h_s)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), pg, dev)
    del sets
    return e2e_ms, e2e_steps


def run_ours(args, w):
    import torch

    ws, rank, local = _dist_env()
    timer = OracleTimer(w) if (rank == 0 and not args.no_cpu_baseline) else None
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    from __graft_entry__ import build
    build()
    import h2o_heavy_hitter_gb300 as h2o

    B, H, d, T, S, L = w.batch, w.heads, w.head_dim, w.prompt, w.steps, w.layers
    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)
                   or L2_FALLBACK_BYTES)
    # Inputs: each rank draws its own seeds (independent batches).
    t0 = time.perf_counter()
    nl = min(L, MAX_DISTINCT_LAYERS)

    def host(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)

    hp, hs = [], []  # per input layer: prompt [B,H,T,d] x3, decode inputs [S,B,H,d] x3 (pinned)
    for li in range(nl):
        bits = _gen_layer(w, rank_layer_seed(rank) * MAX_DISTINCT_LAYERS + li)
        hp.append([host(bits[i][:, :, :T]).pin_memory() for i in range(3)])
        hs.append([host(bits[i][:, :, T:].transpose(2, 0, 1, 3)).pin_memory() for i in range(3)])
        del bits
    gen_s = time.perf_counter() - t0
    dp = [[x.to(dev) for x in lay] for lay in hp]
    ds = [[x.to(dev) for x in lay] for lay in hs]
    # One output buffer per phase, written by every layer in turn (a following
    # model layer would consume it); the last layer's values are the step's result.
    pre_out = torch.empty((B, H, T, d), dtype=torch.float32, device=dev)
    dec_out = torch.empty((S, B, H, d), dtype=torch.float32, device=dev)

    ctx = h2o.h2o_create(L, B, H, d, w.h, w.r, kv=args.kv, layout=args.layout)
    stream = torch.cuda.Stream(device=dev)

    def prefill_all(c, layers, prompt=None):
        """A new prompt for every layer: empty the layers, then prefill each."""
        prompt = dp if prompt is None else prompt
        h2o.h2o_reset(c, -1)
        for layer in range(layers):
            h2o.h2o_prefill(c, layer, *prompt[layer % nl], out=pre_out)

    def capture(c, layers, steps, inputs=None, outs=None):
        inputs = ds if inputs is None else inputs
        outs = dec_out if outs is None else outs
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for s in range(steps):
                for layer in range(layers):
                    x = inputs[layer % nl]
                    h2o.h2o_decode_step(c, layer, x[0][s], x[1][s], x[2][s], outs[s])
        return g

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        prefill_all(ctx, L)
        graph = capture(ctx, L, S)
    torch.cuda.synchronize()

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        prefill_all(ctx, L)
        if ev is not None:
            ev[1].record(stream)
        graph.replay()
        if ev is not None:
            ev[2].record(stream)

    def barrier():
        if pg is not None:
            pg.barrier()

    with torch.cuda.stream(stream):
        step()  # first pass (module loading, first touches); the warm-up follows
    torch.cuda.synchronize()

    # ---- device-resident timed region (clock samples from the warm-up on)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                          else local)
    clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    with torch.cuda.stream(stream):
        start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        end.record(stream)
    torch.cuda.synchronize()
    clocks.mark(wall0, time.time())
    clk = clocks.stop()
    barrier()
    elapsed_ms = max_over_ranks(start.elapsed_time(end), pg, dev)
    prefill_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
    decode_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in evs]))

    quick = args.quick
    # ---- end to end through the public API with host buffers (_end_to_end)
    h2d = sum(x.numel() * 2 for lay in hp + hs for x in lay)
    d2h = dec_out.numel() * 4
    e2e_ms = e2e_steps = None
    if not quick:
        e2e_ms, e2e_steps = _end_to_end(args, ctx, graph, L, S, dp, ds, hp, hs, dec_out, stream,
                                        prefill_all, capture, barrier, pg, dev)
    del graph

    # ---- decode with the caches cycled through L2: when one layer's caches fit
    # in L2, a graph of decode steps over enough copies of the layer (more than
    # twice the L2 size in all) makes every launch read its cache from HBM, as
    # the layers of a deep model would, with launches still back to back.
    cycled_ms, n_cycle = None, 0
    need = -(-2 * l2_bytes // _layer_cache_bytes(w, args.kv))
    if (not quick and _layer_cache_bytes(w, args.kv) * L <= l2_bytes
            and need <= MAX_CYCLED_LAYERS):
        n_cycle = max(2, need)
        ctx_c = h2o.h2o_create(n_cycle, B, H, d, w.h, w.r, kv=args.kv, layout=args.layout)
        sc = min(S, 32)
        with torch.cuda.stream(stream):
            prefill_all(ctx_c, n_cycle)
            g_c = capture(ctx_c, n_cycle, sc)
            times = []
            for rep_i in range(4):  # the first replay warms up
                prefill_all(ctx_c, n_cycle)
                c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                c0.record(stream)
                g_c.replay()
                c1.record(stream)
                times.append((c0, c1))
        torch.cuda.synchronize()
        cycled_ms = float(np.mean([a.elapsed_time(b_) for a, b_ in times[1:]])) / (sc * n_cycle)
        del g_c
        h2o.h2o_sync_check(ctx_c)
        ctx_c.close()

    # ---- single decode launches with L2 flushed before each (HBM-cold and
    # launch-isolated: the pessimistic reference point). The flush writes a
    # buffer twice the size of L2 and reads it back, so L2 holds clean lines.
    flush = torch.empty(max(256 << 20, 2 * l2_bytes), dtype=torch.uint8, device=dev)
    cold = []
    n_cold = 0 if quick else min(S, 64)
    with torch.cuda.stream(stream):
        prefill_all(ctx, L)
        for s in range(n_cold):
            flush.fill_(s & 0xff)
            flush.sum(dtype=torch.int64)
            a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            x = ds[0]
            h2o.h2o_decode_step(ctx, 0, x[0][s], x[1][s], x[2][s], dec_out[s])
            b_.record(stream)
            cold.append((a, b_))
    torch.cuda.synchronize()
    cold_ms = float(np.mean([a.elapsed_time(b_) for a, b_ in cold[1:]])) if n_cold > 1 else None
    del flush

    # ---- the same decode steps with every step of a layer in one launch
    # (h2o_decode_steps: one CTA per row loops over the steps). Not the
    # headline: it needs all steps' inputs in advance (a teacher-forced pass),
    # while the timed step above launches once per step, as generation does.
    multi_ms = None
    if w.k <= 8192 and args.layout == "slots" and not quick:
        with torch.cuda.stream(stream):
            prefill_all(ctx, L)
            g_m = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_m, stream=stream):
                for layer in range(L):
                    x = ds[layer % nl]
                    h2o.h2o_decode_steps(ctx, layer, x[0], x[1], x[2], dec_out)
            mt = []
            for _ in range(max(3, min(args.steps, 20))):
                prefill_all(ctx, L)
                a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                g_m.replay()
                b_.record(stream)
                mt.append((a, b_))
        torch.cuda.synchronize()
        multi_ms = float(np.mean([a.elapsed_time(b_) for a, b_ in mt[1:]]))
        del g_m
    h2o.h2o_sync_check(ctx)
    ctx.close()

    if rank != 0:
        if pg is not None:
            pg.destroy_process_group()
        return

    peaks, peak_kind = _peaks()
    rows = B * H
    bytes_per_launch = decode_bytes_per_row_step(w.k, d, args.kv, args.layout, w.h) * rows
    dec_launch_ms = decode_ms / (S * L)  # graph replay: launch gaps included
    achieved = bytes_per_launch / (dec_launch_ms * 1e-3) / 1e9
    hbm = float(peaks["hbm_gbs"])
    pflops = prefill_flops_per_row(T, d) * rows * L
    pre_tflops = pflops / (prefill_ms * 1e-3) / 1e12
    # The prefill's ceiling is the lower of the tensor peak and what HBM can
    # feed at its arithmetic intensity (short prompts fall under the ridge).
    pbytes = prefill_bytes_per_row(T, d, w.k, args.kv) * rows * L
    tensor_peak = float(peaks["bf16_tflops"])
    hbm_ceiling = pflops / pbytes * float(peaks["hbm_gbs"]) / 1e3
    pre_ceiling = min(tensor_peak, hbm_ceiling)
    tokens = B * S * args.steps * ws
    value = tokens / (elapsed_ms * 1e-3)
    roof = {"kernel": "h2o decode_kernel", "bound": "hbm", "peak": hbm, "unit": "GB/s",
            "traffic": (_profiled_traffic(DECODE_SOURCES, w.name, rows)
                        if args.kv == "bf16" and args.layout == "slots" else None),
            "bytes_per_launch": bytes_per_launch, "peak_source": f"{peak_kind} hbm_gbs"}
    if cycled_ms is not None:
        # The layer's cache fits in L2, so inside the timed step it is read
        # from L2. The headline figure is the HBM-bound one: the same decode
        # launches with the caches of several layers cycled through L2.
        a_c = bytes_per_launch / (cycled_ms * 1e-3) / 1e9
        roof.update({"achieved": a_c, "frac": a_c / hbm, "launch_ms": cycled_ms,
                     "measured": (f"decode launches of {n_cycle} layers' caches cycled through L2 "
                                  "(each launch reads its cache from HBM), CUDA events around "
                                  "graph replays"),
                     "achieved_in_step": achieved, "frac_in_step": achieved / hbm,
                     "launch_ms_in_step": dec_launch_ms,
                     "in_step": "the timed step's decode launches, cache resident in L2"})
    else:
        resident = _layer_cache_bytes(w, args.kv) * L <= l2_bytes
        roof.update({"achieved": achieved, "frac": achieved / hbm, "launch_ms": dec_launch_ms,
                     "measured": ("the timed step's decode launches (CUDA events over the "
                                  "graph replays; " + (
                                      "the caches fit in L2, so this is an L2-assisted figure: "
                                      "the L2-cycled measurement was skipped" if resident else
                                      "the caches exceed L2") + ")")})
    if cold_ms is not None:
        achieved_cold = bytes_per_launch / (cold_ms * 1e-3) / 1e9
        roof.update({"achieved_l2_flushed": achieved_cold, "frac_l2_flushed": achieved_cold / hbm,
                     "launch_ms_l2_flushed": cold_ms})
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": _data_desc(w),
        "config": dict(_config(w, l2_bytes, args.kv), kv_cache=args.kv, cache_layout=args.layout),
        "roofline": roof,
        "phases": {"prefill_ms": prefill_ms, "decode_ms": decode_ms,
                   "prefill_tokens_per_s": B * T * L / (prefill_ms * 1e-3),
                   "prefill_tflops": pre_tflops,
                   "prefill_frac_bf16": pre_tflops / tensor_peak,
                   "prefill_bytes": pbytes,
                   "prefill_ceiling_tflops": pre_ceiling,
                   "prefill_ceiling_bound": "tensor" if tensor_peak <= hbm_ceiling else "hbm",
                   "prefill_frac_of_ceiling": pre_tflops / pre_ceiling,
                   "decode_only_tokens_per_s": B * S / (decode_ms * 1e-3),
                   "input_generation_s": gen_s},
        "e2e": ({"value": B * S * e2e_steps * ws / (e2e_ms * 1e-3), "unit": UNIT,
                 "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
                if e2e_ms is not None else None),
        "gpu_launches": (PREFILL_LAUNCHES + S) * L * args.steps,
        "clocks": clk,
    }
    if multi_ms is not None:
        a_m = bytes_per_launch * S * L / (multi_ms * 1e-3) / 1e9
        line["decode_multistep"] = {
            "call": "h2o_decode_steps, one launch per layer for all its decode steps",
            "decode_ms": multi_ms, "us_per_layer_step": 1e3 * multi_ms / (S * L),
            "decode_only_tokens_per_s": B * S / (multi_ms * 1e-3),
            "step_tokens_per_s": B * S / ((multi_ms + prefill_ms) * 1e-3),
            "achieved_l2_assisted": a_m, "frac_l2_assisted": a_m / hbm, "unit": "GB/s",
            "note": ("same algorithmic bytes per row-step as the per-step kernel; the rows that "
                     "run together keep their caches in L2 from one step to the next, so this "
                     "is not an HBM fraction")}
    if timer is not None:
        v, wall = timer.run_once()
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": timer.cores, "kind": "oracle",
                                "sample": timer.describe(), "wall_s": wall}
        timer.close()
    print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 200, fewer for heavy workloads)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="opt-6.7b-layer", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kv", default="bf16", choices=["bf16", "fp8"],
                    help="cache storage: bf16, or E4M3 codes with per-token scales")
    ap.add_argument("--batch", type=int, default=None, help="override the workload's batch")
    ap.add_argument("--layers", type=int, default=None, help="override the workload's layers")
    ap.add_argument("--quick", action="store_true",
                    help="time the step only (no end-to-end, cycled, flushed, multi-step or CPU legs)")
    ap.add_argument("--layout", default="slots", choices=["slots", "ring"],
                    help="cache layout: slot-indexed, or heavy slots plus a circular recent window")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    w = WORKLOADS[args.workload]
    if args.batch or args.layers:
        over = {k: v for k, v in (("batch", args.batch), ("layers", args.layers)) if v}
        w = w.with_(name=w.name + " (" + ", ".join(f"{k} {v}" for k, v in over.items()) + ")", **over)
    if args.quick:
        args.no_cpu_baseline = True
    if args.steps is None:
        args.steps = _default_steps(w)
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
