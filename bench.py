"""Benchmark of one paged-decode step: cache write + PagedAttention decode.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload llama3_8b|long_ctx|mixed_prefix|gqa8_70b|gqa8_70b_bs32|tiny_fp32]

A step is one pass of the whole hot path over one seeded synthetic batch:
pa_write_cache (each sequence's newest token into the pool) then pa_decode.
The default workload is the Llama-3-8B-shaped batch (64 sequences, 32/8 heads,
head 128, block 16, contexts uniform in [512, 4096], bf16).  Its valid K/V
(~0.6 GB) is larger than L2, so no flush is needed between steps.

Output: one JSON line (rank 0).  `value` is effective GB/s = algorithmic bytes
of the step (K+V over the valid contexts, q, out, the valid block-table
entries, context lengths, the write's rows and slots) / device time.
Under torchrun with N>1 every rank runs an independent replica (no collective
on the data path); the max time over ranks is used and `value` sums all ranks.
"""

from __future__ import annotations

import argparse
import ctypes
import math
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from paged_kv_cache_292_gb300 import workloads  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
# Sources the decode kernel's device code is compiled from; their hash tags
# the committed ncu traffic so that a changed kernel reports traffic null.
KERNEL_SRCS = [os.path.join(ROOT, "paged_kv_cache_292_gb300", "csrc", f)
               for f in ("pa_decode_kernel.cuh", "pa_device.cuh", "pa_schedule.h")]
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024

WORKLOADS = {
    "llama3_8b": ("llama3_8b", None),
    "long_ctx": ("long_ctx", None),
    "mixed_prefix": ("mixed_prefix", None),
    "gqa8_70b": ("gqa8_70b", 16),
    "gqa8_70b_bs32": ("gqa8_70b", 32),
    "tiny_fp32": ("tiny_fp32", None),
}


def step_bytes(w, queries: int = 1, kv_fp8: bool = False) -> dict:
    """Algorithmic bytes of one step (nothing that a perfect kernel could avoid):
    the decode reads K+V over the valid contexts (one byte per element for FP8
    pools), the queries, the valid block-table entries and the lengths, and
    writes the outputs; the cache write reads each new token's K/V rows and
    stores them (quantised for FP8 pools) with an int64 slot per token.
    `queries` new tokens per sequence sit at positions c - Q .. c - 1; those at
    negative positions are not written."""
    sp = w.spec
    e = 4 if sp.dtype == "f32" else 2
    pe = 1 if kv_fp8 else e
    Q = queries
    ctx = w.context_lens.numpy().astype(np.int64)
    nblk = -(-ctx // sp.block_size)
    kv = int(ctx.sum()) * 2 * sp.num_kv_heads * sp.head_size * pe
    qo = 2 * sp.num_seqs * Q * sp.num_heads * sp.head_size * e
    tables = 4 * int(nblk.sum()) + 4 * sp.num_seqs
    decode = kv + qo + tables
    wr_tokens = int(np.minimum(ctx, Q).sum()) if Q > 1 else int((w.slot_mapping.numpy() >= 0).sum())
    row = sp.num_kv_heads * sp.head_size
    write = wr_tokens * 2 * row * (e + pe) + 8 * sp.num_seqs * Q
    return {"decode": decode, "write": write, "step": decode + write, "kv_logical": kv}


def read_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _code_only(text: str) -> str:
    """Source text without comments and blank space, so that edits to comments
    leave the hash (and the measured traffic it keys) unchanged."""
    import re

    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_hash() -> str:
    h = hashlib.sha256()
    for path in KERNEL_SRCS:
        with open(path, encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def traffic_key(workload: str, kv: str = "native", queries: int = 1, block_size=None,
                separate: bool = False) -> str:
    """Key of one bench variant in profiles/traffic.json, e.g. "llama3_8b/fp8"."""
    key = workload
    if separate:
        key += "/separate"
    if kv == "fp8":
        key += "/fp8"
    if queries > 1:
        key += f"/q{queries}"
    if block_size is not None:
        key += f"/bs{block_size}"
    return key


def read_traffic(key: str):
    """Per-launch DRAM bytes of the decode kernel from the committed ncu summary,
    or None if missing or taken on a different kernel source."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
        rec = t.get(key)
        if rec and rec.get("kernel_sha") == kernel_hash():
            return float(rec["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [[c.strip() for c in line.split(",")] for line in out.strip().splitlines() if line.strip()]
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            for i, n in enumerate(names):
                if r[5 + i].lower().startswith("active"):
                    reasons.add(n)
        return {
            "sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(smax) if smax else None,
            "reasons": sorted(reasons),
            "samples": len(sm),
        }


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(ms: float, world: int, device=None) -> float:
    """The slowest rank's time: the whole job is done only when every replica is."""
    if world <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(step_bytes_per_rank: int, world: int, ms_per_step: float) -> float:
    """Weak scaling: every rank runs its own replica, so the job moves world x the bytes."""
    return world * step_bytes_per_rank / (ms_per_step * 1e-3) / 1e9


def make_replica(name: str, rank: int, block_size=None):
    spec_name, bs = WORKLOADS[name]
    bs = block_size or bs
    sp = workloads.spec(spec_name)
    if rank:
        sp = workloads.dataclasses.replace(sp, seed=sp.seed + 1000 * rank)
    return workloads.make_workload(sp, block_size=bs, prewritten=False)


# ---------------------------------------------------------------------------
# CPU oracle timing (reported baseline only)
# ---------------------------------------------------------------------------


def time_oracle(w, budget_s: float, max_seqs: int = None):
    """Run the fp64 oracle (as it stands) on a bounded sample of the batch:
    the cache write of the sampled sequences' new tokens, then their decode.
    Returns (seconds, bytes of that sample, description)."""
    import oracle

    sp = w.spec
    e = 4 if sp.dtype == "f32" else 2
    bs = sp.block_size
    order = list(range(sp.num_seqs)) * 1000  # repeat the batch until the budget is spent
    ctx_all = w.context_lens.numpy().astype(np.int64)
    done, secs, nbytes = 0, 0.0, 0
    for s in order:
        if max_seqs is not None and done >= max_seqs:
            break
        if secs >= budget_s and done > 0:
            break
        c = int(ctx_all[s])
        n = -(-c // bs)
        ids = w.block_tables[s, :n].long()
        # Compact this sequence's blocks (plumbing, not timed).
        view = torch.int32 if sp.dtype == "f32" else torch.int16
        kc = w.k_cache[ids].view(view).numpy()
        vc = w.v_cache[ids].view(view).numpy()
        slot = int(w.slot_mapping[s])
        local_slot = (n - 1) * bs + slot % bs
        bt = np.arange(n)[None, :]
        q = w.q[s : s + 1].double().numpy()
        kn = w.k_new[s : s + 1].view(view).numpy()
        vn = w.v_new[s : s + 1].view(view).numpy()
        t0 = time.perf_counter()
        k2, v2 = oracle.write_cache(kc, vc, kn, vn, np.array([local_slot]), bs)
        k64 = torch.from_numpy(k2).view(w.k_cache.dtype).double().numpy()
        v64 = torch.from_numpy(v2).view(w.v_cache.dtype).double().numpy()
        oracle.decode(q, k64, v64, bt, np.array([c]), w.scale, bs)
        secs += time.perf_counter() - t0
        nbytes += c * 2 * sp.num_kv_heads * sp.head_size * e + 2 * sp.num_heads * sp.head_size * e + 4 * n + 4
        nbytes += 2 * 2 * sp.num_kv_heads * sp.head_size * e + 8
        done += 1
    desc = (f"{done} sequence decodes ({done / sp.num_seqs:.2f} x the {sp.num_seqs}-sequence batch; "
            f"write + decode per sequence), fp64 NumPy oracle")
    return secs, nbytes, desc


def unique_kv_bytes(w, e: int) -> int:
    """K+V bytes of the distinct pool slots the batch reads (a shared prefix
    counted once), beside the logical bytes that count it per sequence."""
    bs = w.spec.block_size
    seen = np.zeros(w.num_blocks * bs, dtype=bool)
    bt, ctx = w.block_tables.numpy(), w.context_lens.numpy()
    for s_, c in enumerate(ctx.tolist()):
        n = -(-c // bs)
        slots = (bt[s_, :n].astype(np.int64)[:, None] * bs + np.arange(bs)).reshape(-1)[:c]
        seen[slots] = True
    return int(seen.sum()) * 2 * w.spec.num_kv_heads * w.spec.head_size * e


def oracle_single_thread(workload: str, budget_s: float):
    """The oracle sample again in a child process with one BLAS/OpenMP thread."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-sample", "--workload", workload,
                            "--cpu-budget", str(budget_s)], env=env, capture_output=True, text=True, timeout=300)
        d = json.loads(r.stdout.strip().splitlines()[-1])
        return {"value": d["bytes"] / d["seconds"] / 1e9, "unit": "GB/s", "cores": 1, "sample": d["sample"]}
    except Exception:
        return None


def run_oracle_sample(args):
    w = make_replica(args.workload, 0, args.block_size)
    secs, nbytes, desc = time_oracle(w, budget_s=args.cpu_budget)
    print(json.dumps({"seconds": secs, "bytes": nbytes, "sample": desc}), flush=True)
    return 0


def cpu_threads() -> int:
    try:
        import threadpoolctl  # noqa: F401

        from threadpoolctl import threadpool_info

        n = max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
        return int(n)
    except Exception:
        return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))


# ---------------------------------------------------------------------------
# Reference arm: the oracle on the host cores
# ---------------------------------------------------------------------------


def run_reference(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    w = make_replica(args.workload, 0)
    by = step_bytes(w)
    per_step_budget = 20.0 / max(1, args.steps + args.warmup)
    for _ in range(args.warmup):
        time_oracle(w, per_step_budget)
    secs, nbytes = 0.0, 0
    for _ in range(args.steps):
        s, b, desc = time_oracle(w, per_step_budget)
        secs += s
        nbytes += b
    gbs = nbytes / secs / 1e9
    ms = secs / args.steps * 1e3
    line = {
        "impl": "reference",
        "metric": "paged decode attention: effective KV GB/s (% of GB300 HBM peak), us/step",
        "value": gbs, "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1), PCG64)",
        "config": {"workload": args.workload, "sample": desc, "full_step_bytes": by["step"]},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cpu_threads(), "kind": "oracle", "sample": desc},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------


def measure(args, lib, dev, world, rank, local, cpu_baseline=True):
    """Time one workload (args.workload) on this rank: region 1 (K steps back
    to back), region 2 (events around each call), end to end from host
    buffers.  Every rank takes part (barriers, max over ranks); rank 0 gets the
    JSON line, the others None."""
    from paged_kv_cache_292_gb300 import binding

    w = make_replica(args.workload, rank, args.block_size)
    sp = w.spec
    Q = args.queries
    fp8 = args.kv == "fp8"
    if fp8 and sp.dtype != "bf16":
        raise SystemExit("--kv fp8 needs a bf16 workload (bf16 queries and new rows)")
    by = step_bytes(w, Q, fp8)
    S, H, D = w.q.shape
    Hk, bs, NB, MB = sp.num_kv_heads, sp.block_size, w.num_blocks, w.max_blocks_per_seq
    dt = binding.dtype_code(w.q.dtype)
    g = {k: getattr(w, k).to(dev) for k in ("q", "k_cache", "v_cache", "block_tables", "context_lens",
                                             "slot_mapping", "k_new", "v_new")}
    if Q > 1:
        # Several new tokens per sequence (positions c-Q .. c-1): their query
        # rows, their K/V rows and their slots; the pool already holds them.
        mq = workloads.multi_query_step(w, Q)
        for k, v in zip(("q", "k_new", "v_new", "slot_mapping"), mq):
            g[k] = v.to(dev)
    if fp8:
        # E4M3 pools (one scale per pool); the prompt's K/V quantised once here.
        k_scale = v_scale = 1.0
        g["k_cache"] = (g["k_cache"].float() / k_scale).to(torch.float8_e4m3fn).view(torch.uint8)
        g["v_cache"] = (g["v_cache"].float() / v_scale).to(torch.float8_e4m3fn).view(torch.uint8)
    n_new = S * Q
    out = torch.empty_like(g["q"])
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    ws_bytes = (lib.pa_decode_workspace_size(S, H, Hk, D, 0) if Q == 1
                else lib.pa_decode_mq_workspace_size(S, Q, H, Hk, D, 0))
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)  # merge tickets start at zero
    P = binding._ptr

    # The step: the newest tokens' cache write and the decode.  bf16 queries
    # run both in one launch (pa_decode_append, pa_decode_fp8_append or, with
    # several queries per sequence, pa_decode_mq_append) unless --step
    # separate asks for the cache write and the decode as two launches.
    fused = args.step == "fused" and sp.dtype == "bf16"
    # With more than 8 (query, head) columns per KV head the appending call
    # writes the rows with its own kernel ahead of the decode: two launches.
    launches = 1 if fused and (H // Hk) * Q <= 8 else 2

    def write(gg, sh=sh):
        if fused:
            return
        if fp8:
            rc = lib.pa_write_cache_fp8(P(gg["k_new"]), P(gg["v_new"]), P(gg["slot_mapping"]), P(g["k_cache"]),
                                        P(g["v_cache"]), n_new, Hk, D, bs, NB, k_scale, v_scale, sh, dt, None)
        else:
            rc = lib.pa_write_cache(P(gg["k_new"]), P(gg["v_new"]), P(gg["slot_mapping"]), P(g["k_cache"]),
                                    P(g["v_cache"]), n_new, Hk, D, bs, NB, sh, dt)
        if rc:
            raise RuntimeError(binding.pa_last_error())

    def decode(gg, o, sh=sh):
        if fused and fp8 and Q > 1:
            rc = lib.pa_decode_fp8_mq_append(P(o), P(gg["q"]), P(gg["k_new"]), P(gg["v_new"]), P(g["k_cache"]),
                                             P(g["v_cache"]), P(gg["block_tables"]), P(gg["context_lens"]), S, Q, H,
                                             Hk, D, bs, MB, w.scale, k_scale, v_scale, sh, 0, P(ws), ws_bytes, 0,
                                             None)
        elif fused and fp8:
            rc = lib.pa_decode_fp8_append(P(o), P(gg["q"]), P(gg["k_new"]), P(gg["v_new"]), P(g["k_cache"]),
                                          P(g["v_cache"]), P(gg["block_tables"]), P(gg["context_lens"]), S, H, Hk, D,
                                          bs, MB, w.scale, k_scale, v_scale, sh, 0, P(ws), ws_bytes, 0, None)
        elif fused and Q > 1:
            rc = lib.pa_decode_mq_append(P(o), P(gg["q"]), P(gg["k_new"]), P(gg["v_new"]), P(g["k_cache"]),
                                         P(g["v_cache"]), P(gg["block_tables"]), P(gg["context_lens"]), S, Q, H, Hk,
                                         D, bs, MB, w.scale, sh, dt, 0, P(ws), ws_bytes, 0, None)
        elif fused:
            rc = lib.pa_decode_append(P(o), P(gg["q"]), P(gg["k_new"]), P(gg["v_new"]), P(g["k_cache"]),
                                      P(g["v_cache"]), P(gg["block_tables"]), P(gg["context_lens"]), S, H, Hk, D,
                                      bs, MB, w.scale, sh, dt, 0, P(ws), ws_bytes, 0, None)
        elif fp8 and Q > 1:
            rc = lib.pa_decode_fp8_mq(P(o), P(gg["q"]), P(g["k_cache"]), P(g["v_cache"]), P(gg["block_tables"]),
                                      P(gg["context_lens"]), S, Q, H, Hk, D, bs, MB, w.scale, k_scale, v_scale, sh,
                                      0, P(ws), ws_bytes, 0, None)
        elif fp8:
            rc = lib.pa_decode_fp8(P(o), P(gg["q"]), P(g["k_cache"]), P(g["v_cache"]), P(gg["block_tables"]),
                                   P(gg["context_lens"]), S, H, Hk, D, bs, MB, w.scale, k_scale, v_scale, sh, 0,
                                   P(ws), ws_bytes, 0, None)
        elif Q == 1:
            rc = lib.pa_decode_ws(P(o), P(gg["q"]), P(g["k_cache"]), P(g["v_cache"]), P(gg["block_tables"]),
                                  P(gg["context_lens"]), S, H, Hk, D, bs, MB, w.scale, sh, dt, P(ws), ws_bytes)
        else:
            rc = lib.pa_decode_mq(P(o), P(gg["q"]), P(g["k_cache"]), P(g["v_cache"]), P(gg["block_tables"]),
                                  P(gg["context_lens"]), S, Q, H, Hk, D, bs, MB, w.scale, sh, dt, 0, P(ws),
                                  ws_bytes, 0, None)
        if rc:
            raise RuntimeError(binding.pa_last_error())

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # ---- device-resident timing ----
    for _ in range(args.warmup):
        write(g)
        decode(g, out)
    torch.cuda.synchronize(dev)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    torch.cuda.synchronize(dev)
    # Timed region 1: K whole steps back to back (the step's kernels are
    # chained with programmatic dependent launch, so no events in between).
    if args.graph:
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)  # capture needs a stream other than the legacy default
        with torch.cuda.graph(graph, stream=cap):
            write(g, cap.cuda_stream)
            decode(g, out, cap.cuda_stream)
        torch.cuda.synchronize(dev)
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize(dev)
    t_start.record(stream)
    for _ in range(args.steps):
        if args.graph:
            graph.replay()
        else:
            write(g)
            decode(g, out)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    # Timed region 2: the same K steps with events around each pa_decode call
    # on the launch stream, for the decode kernels' own duration (roofline).
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    wev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        wev[i][0].record(stream)
        write(g)
        wev[i][1].record(stream)
        ev[i][0].record(stream)
        decode(g, out)
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    dec_ms = statistics.fmean(a.elapsed_time(b) for a, b in ev)
    wr_ms = statistics.fmean(a.elapsed_time(b) for a, b in wev)
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_step = total_ms / args.steps
    value = job_throughput(by["step"], world, ms_step)

    # ---- end to end through the public API, host buffers ----
    # The step's inputs sit packed in one pinned host buffer (one upload per
    # step); device inputs and outputs are double-buffered so that the upload
    # of step i+1 and the read-back of step i overlap the kernels of step i.
    names = ("q", "block_tables", "context_lens", "slot_mapping", "k_new", "v_new")
    offs, total = {}, 0
    for k in names:
        offs[k] = total
        total += -(-g[k].numel() * g[k].element_size() // 256) * 256
    host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
    for k in names:
        nb = g[k].numel() * g[k].element_size()
        host_buf[offs[k]:offs[k] + nb].copy_(g[k].cpu().contiguous().view(-1).view(torch.uint8))
    h2d = sum(g[k].numel() * g[k].element_size() for k in names)
    dev_buf = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]

    def views(buf):
        return {k: buf[offs[k]:offs[k] + g[k].numel() * g[k].element_size()].view(g[k].dtype).view(g[k].shape)
                for k in names}

    dev_in = [views(b) for b in dev_buf]
    out_dev = [out, torch.empty_like(out)]
    out_host = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    d2h = out_host[0].numel() * out_host[0].element_size()
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_up = [torch.cuda.Event() for _ in range(2)]
    ev_run = [torch.cuda.Event() for _ in range(2)]
    ev_down = [torch.cuda.Event() for _ in range(2)]
    cur = torch.cuda.current_stream(dev)
    e2e_steps = max(10, min(args.steps, 1000))

    def e2e_step(i):
        b = i % 2
        if i >= 2:
            up.wait_event(ev_run[b])  # step i-2's kernels are done with dev_buf[b]
        with torch.cuda.stream(up):
            dev_buf[b].copy_(host_buf, non_blocking=True)
        ev_up[b].record(up)
        cur.wait_event(ev_up[b])
        if i >= 2:
            cur.wait_event(ev_down[b])  # step i-2's output has left out_dev[b]
        write(dev_in[b])
        decode(dev_in[b], out_dev[b])
        ev_run[b].record(cur)
        down.wait_event(ev_run[b])
        with torch.cuda.stream(down):
            out_host[b].copy_(out_dev[b], non_blocking=True)
        ev_down[b].record(down)

    def e2e_run(n):
        up.wait_stream(cur)
        down.wait_stream(cur)
        for i in range(n):
            e2e_step(i)
        cur.wait_stream(up)
        cur.wait_stream(down)

    e2e_run(max(3, args.warmup))
    torch.cuda.synchronize(dev)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(e2e_steps)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    e2e_value = job_throughput(by["step"], world, e2e_ms)

    if rank != 0:
        return None

    peak, peak_kind = read_peaks()
    # The roofline kernel's average launch duration.  A fused step is one
    # launch, so region 1 (launches back to back, events only around the whole
    # region) gives it directly, and that launch also moves the cache write's
    # bytes.  With a separate write, region 2's events around each decode call
    # isolate the decode kernel; they also keep each launch from overlapping
    # the one before, so that figure is a little high.
    kern_ms = ms_step if fused else dec_ms
    achieved = (by["step"] if fused else by["decode"]) / (kern_ms * 1e-3) / 1e9
    traffic = read_traffic(traffic_key(args.workload, args.kv, args.queries, args.block_size,
                                       separate=not fused and args.step == "separate"))
    line = {
        "metric": "paged decode attention: effective KV GB/s (% of GB300 HBM peak), us/step",
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "us_per_step": ms_step * 1e3,
        "pct_of_hbm_peak": 100.0 * value / world / peak,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8_e4m3" if fp8 else ("bf16" if sp.dtype == "bf16" else "f32"),
        "data": "synthetic (seeded N(0,1) K/V/q via PCG64, cast RNE to bf16; shuffled block pool)",
        "config": {
            "workload": args.workload,
            "num_seqs": S, "num_heads": H, "num_kv_heads": Hk, "head_size": D, "block_size": bs,
            "num_physical_blocks": NB, "context_tokens": int(w.context_lens.sum()),
            "step_bytes": by["step"], "decode_bytes": by["decode"], "write_bytes": by["write"],
            "unique_kv_bytes": unique_kv_bytes(w, 1 if fp8 else (2 if sp.dtype == "bf16" else 4)),
            "write_us": None if fused else wr_ms * 1e3,
            "step": ((("pa_decode_fp8_mq_append" if Q > 1 else "pa_decode_fp8_append") if fp8
                      else "pa_decode_mq_append" if Q > 1 else "pa_decode_append") +
                     (" (cache write fused into the decode, one launch)" if launches == 1
                      else " (row-writing kernel chained ahead of the decode, two launches)") if fused
                     else "cache write + decode (two launches)"),
            "l2": f"inputs larger than L2: {by['kv_logical'] / 1e9:.3f} GB of K/V read per step vs "
                  f"{L2_BYTES / 1e6:.0f} MB L2; no flush",
            "replicas": world,
            "queries_per_seq": Q,
            "kv_pool": "fp8_e4m3" if fp8 else sp.dtype,
            "launch": "CUDA graph replay" if args.graph else "eager (programmatic dependent launch)",
        },
        "roofline": {
            "kernel": ("pa_decode_kernel (one launch per step: cache write and decode; split sequences merged "
                       "in-kernel)" if launches == 1 else
                       "pa_append_rows_kernel + pa_decode_kernel (step bytes over the step time)" if fused else
                       "pa_decode_kernel (one launch per decode call; split sequences merged in-kernel)"),
            "bound": "hbm",
            "achieved": achieved,
            "peak": peak,
            "peak_source": f"{peak_kind} hbm_gbs",
            "unit": "GB/s",
            "frac": achieved / peak,
            "traffic": traffic,
            "decode_us": kern_ms * 1e3,
            "decode_us_per_call_events": dec_ms * 1e3,
            "timing": (f"region 1: back-to-back steps, {launches} launch(es) each" if fused
                       else "region 2: events around each decode call"),
        },
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms,
                "note": "per-step inputs (q, new K/V, slots, tables, lengths) uploaded from one pinned host "
                        "buffer and the output read back every step, double-buffered so transfers of adjacent "
                        "steps overlap the kernels; the paged pool is device-resident state"},
        "gpu_launches": launches * args.steps,  # launches per step in region 1
        "clocks": clk,
    }
    if cpu_baseline and args.cpu_baseline:
        secs, nbytes, desc = time_oracle(w, budget_s=args.cpu_budget)
        line["cpu_baseline"] = {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": cpu_threads(),
                                "kind": "oracle", "sample": desc, "seconds": secs}
        if args.workload in ("tiny_fp32", "llama3_8b") and Q == 1 and not fp8 and args.block_size is None:
            one = oracle_single_thread(args.workload, budget_s=min(5.0, args.cpu_budget))
            if one is not None:
                line["cpu_baseline"]["single_thread"] = one
    return line


# The second workload the default run also times: the long-context batch
# (8 sequences of 32768 tokens, every sequence split across ranges and merged).
SECONDARY = {"llama3_8b": "long_ctx"}


def run_ours(args):
    from paged_kv_cache_292_gb300 import binding
    from paged_kv_cache_292_gb300 import build as pa_build

    world, rank, local = dist_setup()
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 1
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    pa_build.build()
    lib = binding.load()

    line = measure(args, lib, dev, world, rank, local)
    second = SECONDARY.get(args.workload) if args.secondary else None
    if second and args.kv == "native" and args.queries == 1 and args.block_size is None and not args.graph:
        torch.cuda.empty_cache()
        sargs = argparse.Namespace(**vars(args))
        sargs.workload = second
        sargs.steps = max(1, min(args.steps, 2000))
        sl = measure(sargs, lib, dev, world, rank, local, cpu_baseline=False)
        if line is not None:
            keep = ("metric", "value", "unit", "ms_per_step", "us_per_step", "pct_of_hbm_peak", "steps", "warmup",
                    "dtype", "roofline", "e2e", "gpu_launches", "clocks")
            sec = {k: sl[k] for k in keep}
            sec["config"] = {k: sl["config"][k] for k in ("workload", "num_seqs", "num_heads", "num_kv_heads",
                                                            "head_size", "block_size", "context_tokens", "step_bytes",
                                                            "decode_bytes", "step", "l2")}
            line["secondary"] = {second: sec}
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_loop(args):
    """Steady-state decode driven by the host block manager, K steps.

    Each step: one batched pa_bm_append (one new token per sequence, blocks
    allocated on demand), export of block tables and lengths into a pinned
    host buffer, its host-to-device copy, the cache write and the decode.  The
    timed region covers the host work too (wall clock, synchronised at both
    ends)."""
    from paged_kv_cache_292_gb300 import binding
    from paged_kv_cache_292_gb300 import build as pa_build

    pa_build.build()
    lib = binding.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    spec_name, bs0 = WORKLOADS[args.workload]
    sp = workloads.spec(spec_name)
    bs = args.block_size or bs0 or sp.block_size
    S, H, Hk, D = sp.num_seqs, sp.num_heads, sp.num_kv_heads, sp.head_size
    ctx0 = workloads._draw_context_lens(dataclasses_replace(sp, block_size=bs))
    steps = args.steps
    mb = -(-(int(ctx0.max()) + steps + args.warmup + 1) // bs)
    nb = int(sum(-(-(int(c) + steps + args.warmup + 1) // bs) for c in ctx0)) + S
    tdt = torch.bfloat16 if sp.dtype == "bf16" else torch.float32
    gen = torch.Generator(device=dev).manual_seed(sp.seed)
    k_cache = torch.randn((nb, bs, Hk, D), generator=gen, device=dev).to(tdt)
    v_cache = torch.randn((nb, bs, Hk, D), generator=gen, device=dev).to(tdt)
    q = torch.randn((S, H, D), generator=gen, device=dev).to(tdt)
    k_new = torch.randn((S, Hk, D), generator=gen, device=dev).to(tdt)
    v_new = torch.randn((S, Hk, D), generator=gen, device=dev).to(tdt)
    bm = binding.BlockManager(nb, bs, S, mb)
    for s_, c in enumerate(ctx0.tolist()):
        bm.append(s_, c - 1)  # the prompt's K/V already sits in the (random) pool
    seqs = torch.arange(S, dtype=torch.int32)
    ones = torch.ones(S, dtype=torch.int32)
    # Per step the manager's slots, tables and lengths go up in one copy from
    # a packed pinned buffer.  Two buffer sets (host and device) alternate:
    # the host refills set b only after its previous upload completed, and the
    # upload into device set b waits until the kernels that last read it are
    # done, so uploads run on their own stream beside the previous decode.
    lay, total = {}, 0
    for k, n, dt in (("slots", S, torch.int64), ("tables", S * mb, torch.int32), ("lens", S, torch.int32)):
        lay[k] = (total, n, dt)
        total += -(-n * torch.empty(0, dtype=dt).element_size() // 256) * 256

    def carve(buf):
        v = {k: buf[o:o + n * torch.empty(0, dtype=dt).element_size()].view(dt) for k, (o, n, dt) in lay.items()}
        v["tables"] = v["tables"].view(S, mb)
        return v

    bufs = []
    for _ in range(2):
        hb = torch.empty(total, dtype=torch.uint8).pin_memory()
        db = torch.empty(total, dtype=torch.uint8, device=dev)
        bufs.append(dict(hbuf=hb, dbuf=db, h=carve(hb), d=carve(db), copied=torch.cuda.Event(),
                         used=torch.cuda.Event()))
    copies_h = torch.empty(2 * S, dtype=torch.int32)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    ws_bytes = lib.pa_decode_workspace_size(S, H, Hk, D, 0)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    up = torch.cuda.Stream(dev)
    sh = stream.cuda_stream
    P = binding._ptr
    nc, nd = ctypes.c_int(0), ctypes.c_int(0)
    host_s = 0.0
    it = 0

    def step():
        nonlocal host_s, it
        b = bufs[it % 2]
        it += 1
        b["copied"].synchronize()  # the upload that last read this host set is done
        t0 = time.perf_counter()
        h, d = b["h"], b["d"]
        rc = lib.pa_bm_append_batch(bm._h, S, P(seqs), P(ones), P(h["slots"]), P(copies_h), ctypes.addressof(nc),
                                    ctypes.addressof(nd))
        rc = rc or lib.pa_bm_export(bm._h, P(h["tables"]), P(h["lens"]))
        host_s += time.perf_counter() - t0
        if rc:
            raise RuntimeError(binding.pa_last_error())
        up.wait_event(b["used"])  # the kernels that last read this device set are done
        with torch.cuda.stream(up):
            b["dbuf"].copy_(b["hbuf"], non_blocking=True)
        b["copied"].record(up)
        stream.wait_event(b["copied"])
        if tdt == torch.bfloat16 and args.step == "fused":
            # The newest token sits at position len - 1, where the manager put its slot.
            rc = lib.pa_decode_append(P(out), P(q), P(k_new), P(v_new), P(k_cache), P(v_cache), P(d["tables"]),
                                      P(d["lens"]), S, H, Hk, D, bs, mb, 1 / math.sqrt(D), sh,
                                      binding.dtype_code(tdt), nb, P(ws), ws_bytes, 0, P(err))
        else:
            rc = lib.pa_write_cache(P(k_new), P(v_new), P(d["slots"]), P(k_cache), P(v_cache), S, Hk, D, bs, nb,
                                    sh, binding.dtype_code(tdt))
            rc = rc or lib.pa_decode_ex(P(out), P(q), P(k_cache), P(v_cache), P(d["tables"]), P(d["lens"]), S, H,
                                        Hk, D, bs, mb, 1 / math.sqrt(D), sh, binding.dtype_code(tdt), nb, P(ws),
                                        ws_bytes, 0, P(err))
        if rc:
            raise RuntimeError(binding.pa_last_error())
        b["used"].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    tokens0 = int(sum(bm.context_len(s_) for s_ in range(S)))
    host_s = 0.0
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t0
    if int(err.item()) != 0:
        raise RuntimeError(f"device reported error bits {int(err.item())}")
    tokens1 = int(sum(bm.context_len(s_) for s_ in range(S)))
    e = 2 if sp.dtype == "bf16" else 4
    mean_tokens = (tokens0 + tokens1) / 2
    kv = mean_tokens * 2 * Hk * D * e
    line = {
        "metric": "steady-state paged decode loop (block manager + cache write + decode), us/step",
        "value": wall / steps * 1e6, "unit": "us/step", "higher_is_better": False, "steps": steps,
        "warmup": args.warmup, "host_manager_us_per_step": host_s / steps * 1e6,
        "effective_kv_gbs": kv / (wall / steps) / 1e9, "n_gpus": 1, "dtype": sp.dtype, "data": "synthetic",
        "config": {"workload": args.workload, "num_seqs": S, "block_size": bs, "num_physical_blocks": nb,
                   "context_tokens_start": tokens0, "context_tokens_end": tokens1,
                   "step": ("pa_decode_append (cache write fused into the decode)"
                            if tdt == torch.bfloat16 and args.step == "fused" else "pa_write_cache + pa_decode_ex")},
    }
    print(json.dumps(line), flush=True)
    bm.close()
    return 0


def dataclasses_replace(sp, **kw):
    import dataclasses

    return dataclasses.replace(sp, **kw)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(WORKLOADS), default="llama3_8b")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--graph", action="store_true",
                    help="time replays of the step captured in a CUDA graph (region 1) instead of eager calls")
    ap.add_argument("--block-size", type=int, default=None, help="override the workload's block size")
    ap.add_argument("--queries", type=int, default=1,
                    help="query tokens per sequence (several: causal multi-query step via pa_decode_mq)")
    ap.add_argument("--kv", choices=["native", "fp8"], default="native",
                    help="KV pool element type: the workload's own, or E4M3 FP8 (quantising write + FP8 decode)")
    ap.add_argument("--no-secondary", dest="secondary", action="store_false",
                    help="the Llama-shaped default run also times the long-context batch (nested under "
                         "'secondary'); this turns that off")
    ap.add_argument("--oracle-sample", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--step", choices=["fused", "separate"], default="fused",
                    help="one-query bf16/FP8 steps: cache write fused into the decode launch (default) or a "
                         "separate cache-write launch")
    ap.add_argument("--loop", action="store_true",
                    help="steady-state decode loop driven by the host block manager (separate metric)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.oracle_sample:
        return run_oracle_sample(args)
    if args.impl == "reference":
        return run_reference(args)
    if args.loop:
        return run_loop(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
