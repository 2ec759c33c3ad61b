#!/usr/bin/env python
"""Benchmark of the GB300 variable-size all-to-all (a2av).

Workload (one "step" = one a2av over the whole batch): W=4 ranks, 4 GiB of
rows of 7168 bf16 (14336 B) per rank, uniform random bits, splits ~
Multinomial(rows, 1/4 each), seed 0 -- the top point of the 1 MiB .. 4 GiB
payload sweep of "[a2av] Improve tuning for 4 GPUs" (pytorch PR 154580,
"Before"/"After" tables).  The whole sweep is also timed and reported.

Metric: moved GB/s = bytes moved per step / step time (GB = 1e9), and the
fraction of the HBM roofline = 2 x moved bytes / time / HBM peak.  The page's
BusBw (per-rank bytes / time) is reported beside it for context.

Timing: CUDA events on the launching stream around every launch, after
warm-up, bracketed by barrier + synchronize; inputs (16 GiB) exceed the L2, and
the sweep flushes L2 between launches.  The CPU oracle is timed on a bounded
sample (whole peers' outputs) on one host core, and its result is compared
with the GPU's, outside every timed region.

Multi-GPU: the exchange emulates its ranks inside one GPU, so N GPUs run N
independent replicas ("replicas only"), each on its own copy of the workload;
value = all replicas' bytes / the slowest replica's time.

``--impl reference`` times the CPU oracle alone as the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "a2av moved GB/s and fraction of GB300 HBM roofline vs payload size"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
ROW_BYTES = 7168 * 2
W = 4


# ------------------------------------------------------------ arithmetic --
def moved_bytes(splits, row_bytes) -> int:
    """Bytes one exchange moves: every row once (read once, written once)."""
    return int(np.asarray(splits, dtype=np.int64).sum()) * int(row_bytes)


def algorithmic_bytes(splits, row_bytes) -> int:
    """DRAM bytes an ideal exchange touches: read + write of every row, the
    split matrix read (8 W^2) and out_splits_offsets written (16 W^2)."""
    Wn = np.asarray(splits).shape[0]
    return 2 * moved_bytes(splits, row_bytes) + 24 * Wn * Wn


def busbw_gbps(per_rank_bytes: float, seconds: float) -> float:
    """The page's BusBw: per-rank payload bytes / time, GB = 1e9."""
    return per_rank_bytes / seconds / 1e9


def workload_name(per_rank_bytes: int) -> str:
    return (f"a2av W={W}, {per_rank_bytes / 2**20:g} MiB/rank of 7168-bf16 rows "
            f"(14336 B), uniform random bits, in_splits ~ Multinomial(rows, 1/4), seed 0")


# -------------------------------------------------------------- process --
def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def dist_init(backend: str):
    import torch.distributed as dist
    rank, _, world = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return world


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def reduce_max(x: float, device=None) -> float:
    """Maximum of x over ranks (x itself without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Aggregate throughput: every rank's units over the slowest rank's time."""
    return units_per_rank * world / max_seconds


# --------------------------------------------------------------- clocks --
class ClockSampler:
    """nvidia-smi clock and throttle-reason samples during a timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.gpu, self.period = gpu_index, period_ms
        self.proc, self.path = None, None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.path is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 9:
                rows.append(f)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k] == "Active"})
        loaded = [s for s in sm if s > 0.5 * max(sm)] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows),
                "power_w_median": statistics.median([num(r[3]) for r in rows
                                                     if num(r[3]) is not None] or [0])}


# ------------------------------------------------------------ roofline --
def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        for key in ("hbm_gbs", "hbm_GBps", "hbm_copy_gbs"):
            if key in d and d[key]:
                return float(d[key]), "of measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "of fallback"


# The sources each family of kernels is compiled from: the fused dispatch's
# and fused combine's kernels (dispatch_*, combine_*) live in dispatch.cu,
# every other kernel in a2av.cu; both include the
# shared device header and the C header (a2av_handle.h is host-only).
_SHARED_SOURCES = ["variable_size_all_gb300/csrc/a2av_device.cuh", "include/a2av.h"]


def kernel_sources(kernel: str) -> list:
    own = "dispatch.cu" if kernel.startswith(("dispatch_", "combine_")) else "a2av.cu"
    return [f"variable_size_all_gb300/csrc/{own}"] + _SHARED_SOURCES


def code_only(text: str) -> str:
    """C/CUDA source without comments and with whitespace collapsed: what the
    compiler sees, so that editing a comment keeps a kernel's counters."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_sha(kernel: str = "a2av_bulk_kernel") -> str:
    """Hash of the code (comments aside) of the CUDA sources the named kernel
    is built from."""
    h = hashlib.sha256()
    for rel in kernel_sources(kernel):
        h.update(rel.encode())
        h.update(code_only(open(os.path.join(ROOT, rel), encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def workload_key(args) -> str:
    """The workload part of a traffic.json key: the config name plus what
    differs from its defaults (cfg3 hidden size, tokens, per-rank dedup; cfg5
    batch)."""
    k = args.workload
    if k == "cfg3":
        k += (f"_h{args.hidden}" if args.hidden != 7168 else "") + \
             (f"_t{args.tokens}" if args.tokens != 8192 else "") + ("_dedup" if args.dedup else "")
    elif k == "cfg5" and args.batch != 8192:
        k += f"_b{args.batch}"
    return k


def measured_traffic(kernel: str, algo_bytes: int):
    """DRAM bytes per launch from the committed ncu summary of this kernel on
    this workload ("kernel:workload"), scaled to this launch's algorithmic
    bytes; None when absent or taken on other source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(path))
    except (OSError, ValueError):
        return None
    e = d.get(kernel)
    if not e or e.get("source_sha") != kernel_source_sha(kernel.split(":")[0]):
        return None
    return int(round(e["dram_bytes"] / e["algorithmic_bytes"] * algo_bytes))


# -------------------------------------------------------------- oracle ----
def time_oracle(inputs, splits, row_bytes, budget_s: float, peers=None, check=None):
    """Run the CPU oracle peer by peer (one host thread) until the budget is
    spent; returns (seconds, bytes moved, peers done).  ``check(p, out, so)``,
    if given, sees each peer's output outside the timed part."""
    import oracle
    o = oracle.default()
    Wn = len(inputs)
    peers = list(range(Wn)) if peers is None else peers
    spent, moved, done = 0.0, 0, []
    for p in peers:
        buf = np.empty(int(splits[:, p].sum()) * row_bytes, dtype=np.uint8)
        so = np.empty((2, Wn), dtype=np.int64)
        t0 = time.perf_counter()
        rc = o.dest(inputs, splits, p, buf, so, row_bytes)
        spent += time.perf_counter() - t0
        assert rc == 0
        moved += buf.size
        done.append(p)
        if check is not None:
            check(p, buf, so)
        del buf
        if spent >= budget_s:
            break
    return spent, moved, done


# ----------------------------------------------------------------- ours ----
L2_BYTES = 129 * 10**6
WORKLOADS = ("cfg2", "cfg1", "cfg3", "cfg4", "cfg5")


def describe(name: str, per_rank_bytes: int, seed: int, tokens: int = 8192,
             batch: int = 8192, dedup: bool = False, hidden: int = 7168) -> str:
    if name == "cfg2":
        return workload_name(per_rank_bytes)
    if name == "cfg3" and dedup:
        return (describe(name, per_rank_bytes, seed, tokens, batch, hidden=hidden).replace(
            "top-2 of 64 experts", "top-2 of 64 experts, one row per distinct (token, "
            "destination rank) pair"))
    if name == "cfg3" and (tokens != 8192 or hidden != 7168):
        return (f"a2av W=8 MoE dispatch: {tokens} tokens/rank, hidden {hidden} bf16 "
                f"({2 * hidden} B rows), top-2 of 64 experts (8 per rank), Zipf(1.2) popularity "
                f"shuffled per seed, seed {seed}")
    if name == "cfg5" and batch != 8192:
        return (f"a2av W=2 embedding keys: 26 features x {batch} bags per rank, "
                f"min(Poisson(3), 20) int64 keys per bag, U[0, 1e7), feature mod 2 ownership, "
                f"seed {seed}")
    return {
        "cfg1": "a2av W=4, 4096 rows/rank of 128 bf16 (256 B), N(0,1) bf16, "
                "in_splits ~ Multinomial(4096, 1/4)",
        "cfg3": "a2av W=8 MoE dispatch: 8192 tokens/rank, hidden 7168 bf16 (14336 B rows), "
                "top-2 of 64 experts (8 per rank), Zipf(1.2) popularity shuffled per seed",
        "cfg4": "a2av W=8, 2^20 rows/rank of 13 int8 bytes (unaligned), "
                "in_splits ~ Multinomial(2^20, Dirichlet(0.1))",
        "cfg5": "a2av W=2 embedding keys: 26 features x 8192 bags per rank, "
                "min(Poisson(3), 20) int64 keys per bag, U[0, 1e7), feature mod 2 ownership",
    }[name] + f", seed {seed}"


def machine() -> dict:
    """The GPU's name, the host CPU model and the host's core count, recorded
    with every line (the oracle baseline runs on one of those cores)."""
    info = {"nproc": os.cpu_count()}
    try:
        import torch
        if torch.cuda.is_available():
            info["gpu"] = torch.cuda.get_device_name()
    except Exception:  # noqa: BLE001 -- a name is context, never a reason to fail
        pass
    try:
        for line in open("/proc/cpuinfo"):
            key = line.split(":")[0].strip().lower()
            if key in ("model name", "cpu part", "hardware") and ":" in line:
                info.setdefault("cpu_model", line.split(":", 1)[1].strip())
    except OSError:
        pass
    return info


def emit(line: dict) -> None:
    line["machine"] = machine()
    print(json.dumps(line), flush=True)


def host_memory_available() -> int:
    """MemAvailable from /proc/meminfo, bytes (0 if unreadable)."""
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def host_bytes_needed(args, world: int) -> int:
    """Pinned host memory all local ranks hold for the cfg2 line: each rank's
    inputs (the e2e sources) and the e2e outputs, W buffers of P bytes each."""
    return world * 2 * W * args.per_rank_bytes


def load_workload(args, torch):
    """The workload's inputs in pinned host memory (also the e2e sources).
    The payload is never reduced to fit: a host without room for every local
    rank's buffers is refused with the numbers."""
    import workloads as wl
    if args.workload == "cfg2":
        P = args.per_rank_bytes
        _, _, world = dist_env()
        avail = host_memory_available()
        need = host_bytes_needed(args, world)
        if avail and need > 0.85 * avail:
            raise SystemExit(f"bench.py: {world} rank(s) at {P / 2**30:g} GiB per emulated rank "
                             f"need {need / 2**30:.0f} GiB of pinned host memory (inputs and e2e "
                             f"outputs); {avail / 2**30:.0f} GiB available. Refusing rather than "
                             f"running a smaller configuration.")
        nbytes = (P // ROW_BYTES) * ROW_BYTES
        h_in = [torch.empty(nbytes, dtype=torch.uint8, pin_memory=True) for _ in range(W)]
        w = wl.cfg2(P, seed=args.seed, buffers=[t.numpy() for t in h_in])
    else:
        gen = {"cfg1": wl.cfg1,
               "cfg3": lambda s: wl.cfg3(s, tokens=args.tokens, dedup=args.dedup,
                                         hidden=args.hidden),
               "cfg4": wl.cfg4, "cfg5": lambda s: wl.cfg5(s, batch=args.batch)}
        w = gen[args.workload](args.seed)
        h_in = [torch.from_numpy(b).pin_memory() for b in w.inputs]
    return w, h_in


def run_ours(args, light=False):
    """One exchange workload (a2av_run, or a2av_combine with --op combine).
    Returns the JSON line.  ``light``: the timed steps, the roofline and a
    full bit-exact check against the oracle only (an entry of the cfg2 line's
    ``configs`` block)."""
    import torch
    import variable_size_all_gb300 as a2av
    import workloads as wl

    rank, local, world = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init("nccl")
    a2av.build()
    path_id = {"auto": a2av.PATH_AUTO, "vector": a2av.PATH_VECTOR, "bulk": a2av.PATH_BULK,
               "staged": a2av.PATH_STAGED}[args.path]

    t0 = time.time()
    w, h_in = load_workload(args, torch)
    gen_s = time.time() - t0
    Wn, rb, S = w.W, w.row_bytes, w.splits
    P = args.per_rank_bytes
    in_bytes = [t.numel() for t in h_in]
    recv = [int(S[:, p].sum()) * rb for p in range(Wn)]
    T = moved_bytes(S, rb)
    d_in = [t.to(dev) for t in h_in]
    d_out = [torch.empty(n, dtype=torch.uint8, device=dev) for n in recv]
    d_S = torch.from_numpy(S).to(dev)
    d_so = torch.empty((Wn, 2, Wn), dtype=torch.int64, device=dev)
    eng = a2av.A2av(Wn, path=path_id, ctas_per_sm=args.ctas_per_sm)
    stream = torch.cuda.current_stream()
    # Inputs larger than twice the L2 stream from HBM anyway; smaller ones get
    # the L2 flushed before every timed launch by reading 512 MiB (a read leaves
    # clean lines, so no earlier write-back lands inside the timed launch).
    cold = sum(in_bytes) < 2 * L2_BYTES
    flush = torch.ones(128 << 20, dtype=torch.int32, device=dev)

    def step(ins=d_in, outs=d_out, splits=d_S):
        eng.run(ins, splits, outs, d_so, rb, stream=stream)

    if args.op == "combine":
        # The reverse exchange: its inputs are the forward exchange's outputs,
        # made once on the device (untimed); a step sends every row home.
        step()
        torch.cuda.synchronize()
        if eng.status() != a2av.OK:
            raise SystemExit("device reported an error in the forward exchange")
        c_in, c_dso = d_out, d_so.clone()
        c_out = [torch.empty_like(t) for t in d_in]
        c_so = torch.empty_like(d_so)

        def step(ins=c_in, outs=c_out, splits=c_dso):  # noqa: F811
            eng.combine(ins, splits, outs, c_so, rb, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if eng.status() != a2av.OK:
        raise SystemExit("device reported an error during warm-up")
    launch = eng.last_launch()

    # ---- timed region: exactly K steps, one kernel launch each ----------
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    t_begin, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        barrier()
        torch.cuda.synchronize()
        t_begin.record(stream)
        for a, b in ev:
            if cold:
                flush.sum()
            a.record(stream)
            step()
            b.record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        barrier()
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    # with flushes in between, a step's time is its launch's own duration
    timed_s = (sum(launch_ms) if cold else t_begin.elapsed_time(t_end)) / 1e3
    if eng.status() != a2av.OK:
        raise SystemExit("device reported an error during the timed region")
    max_s = reduce_max(timed_s, dev)
    value = whole_job_value(T * K / 1e9, world, max_s)
    avg_launch_s = statistics.mean(launch_ms) / 1e3
    med_launch_s = statistics.median(launch_ms) / 1e3

    # ---- launch cost: eager calls vs one captured CUDA graph replayed -----
    # (back to back, no flush: what a caller issuing many small exchanges pays)
    graph_us = eager_us = None
    if cold and world == 1 and not light:
        g_stream = torch.cuda.Stream()
        g_stream.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=g_stream):
            if args.op == "combine":
                eng.combine(c_in, c_dso, c_out, c_so, rb, stream=g_stream)
            else:
                eng.run(d_in, d_S, d_out, d_so, rb, stream=g_stream)
        torch.cuda.synchronize()
        reps = 200
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            graph.replay()
        b.record(stream)
        torch.cuda.synchronize()
        graph_us = a.elapsed_time(b) * 1e3 / reps
        a.record(stream)
        for _ in range(reps):
            step()
        b.record(stream)
        torch.cuda.synchronize()
        eager_us = a.elapsed_time(b) * 1e3 / reps
        if eng.status() != a2av.OK:
            raise SystemExit("device reported an error during graph replay")
        del graph

    # ---- roofline of the (only) kernel -----------------------------------
    algo = algorithmic_bytes(S, rb)
    peak, peak_kind = hbm_peak()
    kname = {a2av.PATH_BULK: "a2av_bulk_kernel", a2av.PATH_STAGED: "a2av_staged_kernel",
             a2av.PATH_VECTOR: "a2av_vector_kernel"}[launch["path"]]
    achieved = algo / avg_launch_s / 1e9
    roofline = {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1),
                "peak": peak, "peak_source": peak_kind, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": measured_traffic(f"{kname}:{workload_key(args)}", algo),
                "algorithmic_bytes_per_launch": algo}

    # ---- the same bytes through a device-to-device copy, interleaved -------
    # (exchange and copy alternate, 20 of each, the L2 treated as in the timed
    # region; the ratio of the medians is the exchange's speed against the
    # practical copy ceiling measured side by side)
    d2d_gbps = vs_copy = None
    if not light:
        src = torch.cat([t for t in d_in])
        dst = torch.empty_like(src)
        for _ in range(3):
            dst.copy_(src)
        t_x, t_c = [], []
        for _ in range(20):
            for fn, acc in ((step, t_x), (lambda: dst.copy_(src), t_c)):
                if cold:
                    flush.sum()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                b.synchronize()
                acc.append(a.elapsed_time(b) / 1e3)
        d2d_gbps = src.numel() / statistics.median(t_c) / 1e9
        vs_copy = statistics.median(t_c) / statistics.median(t_x)
        roofline["vs_same_run_copy"] = round(vs_copy, 4)
        roofline["same_run_copy"] = {"GBps_moved": round(d2d_gbps, 1), "reps": 20,
                                     "what": "torch device-to-device copy of the same bytes, "
                                             "interleaved with the exchange"}
        del src, dst
        if eng.status() != a2av.OK:
            raise SystemExit("device reported an error during the interleaved comparison")

    # ---- payload sweep (cold L2 between launches) --------------------------
    sweep = []
    if args.workload == "cfg2" and args.op == "dispatch" and not args.no_sweep and not light:
        for Pk in wl.CFG2_SWEEP_BYTES:
            if Pk > P:
                break
            Sk = wl.cfg2_splits(Pk, args.seed)
            nk = (Pk // ROW_BYTES) * ROW_BYTES
            ins = [t[:nk] for t in d_in]  # prefix of the same draw = cfg2(Pk)'s inputs
            outs = [t[: int(Sk[:, p].sum()) * ROW_BYTES] for p, t in enumerate(d_out)]
            dSk = torch.from_numpy(Sk).to(dev)
            for _ in range(3):
                step(ins, outs, dSk)
            times = []
            for _ in range(args.sweep_reps):
                flush.sum()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                step(ins, outs, dSk)
                b.record(stream)
                b.synchronize()
                times.append(a.elapsed_time(b) / 1e3)
            t_med = statistics.median(times)
            Tk = moved_bytes(Sk, ROW_BYTES)
            point = {"per_rank_MiB": Pk / 2**20, "moved_bytes": Tk,
                     "us_median": round(t_med * 1e6, 2),
                     "us_mean": round(statistics.mean(times) * 1e6, 2),
                     "us_min": round(min(times) * 1e6, 2),
                     "moved_GBps": round(Tk / t_med / 1e9, 1),
                     "busbw_GBps": round(busbw_gbps(nk, t_med), 1),
                     "hbm_frac": round(algorithmic_bytes(Sk, ROW_BYTES) / t_med / 1e9 / peak, 4)}
            if 4 * Pk <= L2_BYTES // 2 and world == 1:
                # warm L2: one captured exchange replayed back to back
                gs = torch.cuda.Stream()
                gs.wait_stream(stream)
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=gs):
                    eng.run(ins, dSk, outs, d_so, ROW_BYTES, stream=gs)
                torch.cuda.synchronize()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for _ in range(100):
                    graph.replay()
                b.record(stream)
                torch.cuda.synchronize()
                warm = a.elapsed_time(b) / 1e3 / 100
                point["us_warm_graph"] = round(warm * 1e6, 2)
                point["moved_GBps_warm"] = round(Tk / warm / 1e9, 1)
                del graph
            sweep.append(point)
        if eng.status() != a2av.OK:
            raise SystemExit("device reported an error during the sweep")
    del flush

    # ---- end to end through the public API, host buffers ------------------
    e2e = None
    if not args.no_e2e and not light:
        if args.op == "combine":
            # host copies of the combine's own inputs (the forward outputs)
            e_src = [t.cpu().pin_memory() for t in c_in]
            e_dev, e_sp, e_spd = c_in, c_dso.cpu().pin_memory(), c_dso
            e_outs, e_so = c_out, c_so
        else:
            e_src, e_dev, e_sp, e_spd = h_in, d_in, torch.from_numpy(S).pin_memory(), d_S
            e_outs, e_so = d_out, d_so
        h_out = [torch.empty(t.numel(), dtype=torch.uint8, pin_memory=True) for t in e_outs]
        h_so = torch.empty((Wn, 2, Wn), dtype=torch.int64, pin_memory=True)

        def e2e_step():
            for h, d in zip(e_src, e_dev):
                d.copy_(h, non_blocking=True)
            e_spd.copy_(e_sp, non_blocking=True)
            step()
            for h, d in zip(h_out, e_outs):
                h.copy_(d, non_blocking=True)
            h_so.copy_(e_so, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        Ke = args.e2e_steps
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(Ke):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        barrier()
        e_s = reduce_max(a.elapsed_time(b) / 1e3, dev)
        copy_e2e = {"value": round(whole_job_value(T * Ke / 1e9, world, e_s), 2), "unit": UNIT,
                    "h2d_bytes_per_step": sum(t.numel() for t in e_src) + e_sp.numel() * 8,
                    "d2h_bytes_per_step": sum(t.numel() for t in h_out) + 2 * Wn * Wn * 8,
                    "steps": Ke, "mode": "copy: H2D of the inputs and splits, the exchange, "
                                         "D2H of the outputs and offsets (one stream)"}
        if eng.status() != a2av.OK:
            raise SystemExit("device reported an error during the e2e run")
        # Zero-copy: the same call with the pinned host buffers themselves; the
        # kernel reads the inputs and writes the outputs over the host link.
        zc = a2av.A2av(Wn, path=a2av.PATH_VECTOR, ctas_per_sm=args.ctas_per_sm)
        for t in h_out:
            t.fill_(0xEE)

        def zc_step():
            e_spd.copy_(e_sp, non_blocking=True)
            (zc.combine if args.op == "combine" else zc.run)(e_src, e_spd, h_out, e_so, rb,
                                                              stream=stream)
            h_so.copy_(e_so, non_blocking=True)

        zc_step()
        torch.cuda.synchronize()
        zc_ok = all(torch.equal(h_out[k], e_outs[k].cpu()) for k in range(Wn))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(Ke):
            zc_step()
        b.record(stream)
        torch.cuda.synchronize()
        barrier()
        z_s = reduce_max(a.elapsed_time(b) / 1e3, dev)
        if zc.status() != a2av.OK or not zc_ok:
            raise SystemExit("zero-copy exchange failed or differs from the device run")
        zc.close()
        zero_e2e = {"value": round(whole_job_value(T * Ke / 1e9, world, z_s), 2), "unit": UNIT,
                    "h2d_bytes_per_step": copy_e2e["h2d_bytes_per_step"],
                    "d2h_bytes_per_step": sum(t.numel() for t in h_out) + 2 * Wn * Wn * 8,
                    "steps": Ke, "mode": "zero-copy: the exchange reads the pinned host inputs "
                                         "and writes the pinned host outputs itself (vector "
                                         "engine over NVLink-C2C); splits H2D",
                    "bit_exact_vs_device_run": zc_ok}
        e2e = zero_e2e if zero_e2e["value"] >= copy_e2e["value"] else copy_e2e
        e2e["other"] = copy_e2e if e2e is zero_e2e else zero_e2e

    # ---- CPU oracle: baseline timing and a parity check of this run -------
    cpu = None
    parity = None
    if rank == 0 and world == 1 and (light or not args.no_cpu_baseline) and args.op == "combine":
        import oracle
        inputs = [t.numpy() for t in h_in]
        mid, dso = oracle.default().exchange(inputs, S, rb)
        back = [np.empty_like(b) for b in inputs]
        cso = np.empty((Wn, 2, Wn), dtype=np.int64)
        t0 = time.perf_counter()
        assert oracle.default().combine(mid, dso, back, cso, rb) == 0
        spent = time.perf_counter() - t0
        cpu = {"value": round(T / spent / 1e9, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": "the whole reverse exchange of the same workload", "seconds": round(spent, 3)}
        # parity: the round trip is the identity, on the device and on the oracle
        ok = all(torch.equal(c_out[r], d_in[r]) for r in range(Wn))
        ok = ok and np.array_equal(c_so.cpu().numpy(), cso)
        ok = ok and all(np.array_equal(back[r], inputs[r]) for r in range(Wn))
        parity = {"bit_exact": bool(ok), "check": "combine(dispatch(x)) == x on GPU and oracle; "
                                                  "offsets equal the oracle's"}
        if not ok:
            raise SystemExit("the GPU's reverse exchange does not return the inputs")
    elif rank == 0 and world == 1 and (light or not args.no_cpu_baseline):
        inputs = [t.numpy() for t in h_in]
        mismatched = []

        def compare(p, buf, so):
            if not (np.array_equal(d_out[p].cpu().numpy(), buf)
                    and np.array_equal(d_so[p].cpu().numpy(), so)):
                mismatched.append(p)

        spent, moved, peers = time_oracle(inputs, S, rb, float("inf") if light else args.cpu_budget,
                                          check=compare)
        cpu = {"value": round(moved / spent / 1e9, 3), "unit": UNIT, "cores": 1,
               "kind": "oracle",
               "sample": f"peers {peers} of the same exchange "
                         f"({moved / 2**30:.3f} GiB of the {T / 2**30:.3f} GiB moved per step)",
               "seconds": round(spent, 3)}
        parity = {"bit_exact": not mismatched, "peers_checked": peers}
        if mismatched:
            raise SystemExit(f"GPU output differs from the oracle on peers {mismatched}")

    eng.close()
    per_rank = statistics.mean(in_bytes)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(max_s * 1e3 / K, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic (seeded numpy draws; no dataset)",
        "config": exchange_config(args, Wn, rb, int(per_rank), T, cold, world),
        "launch": {"engine": kname, "grid": launch["grid"], "block": launch["block"],
                   "timing": ("L2 flushed (512 MiB read) before every timed launch; step time = "
                              "the launch's CUDA-event duration") if cold else
                             "step time = CUDA events bracketing the K steps"},
        "hbm_fraction": round(2 * T / (max_s / K) / 1e9 / peak, 4),
        "busbw_GBps": round(busbw_gbps(per_rank, max_s / K), 1),
        "launch_us_median": round(med_launch_s * 1e6, 2),
        "back_to_back_us": None if graph_us is None else {
            "eager_python_calls": round(eager_us, 2), "cuda_graph_replay": round(graph_us, 2),
            "note": "per exchange, 200 in a row, warm L2; the graph replays one captured "
                    "call (device-resident splits keep it valid when they change)"},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": K,
        "clocks": clocks.summary(),
        "d2d_memcpy_GBps": None if d2d_gbps is None else round(d2d_gbps, 1),
        "sweep": sweep,
        "parity": parity,
        "input_generation_s": round(gen_s, 2),
    }
    return line


def exchange_config(args, Wn, rb, per_rank, T, cold, world):
    """The `config` of an exchange line -- the same dict on both arms."""
    return {"workload": describe(args.workload, args.per_rank_bytes, args.seed, args.tokens,
                                 args.batch, args.dedup, hidden=args.hidden),
            "name": args.workload, "op": args.op, "ranks": Wn, "row_bytes": rb,
            "per_rank_bytes": per_rank, "moved_bytes_per_step": T,
            "l2": ("inputs smaller than the GPU's L2: flushed (a 512 MiB read) before every "
                   "timed launch") if cold else "inputs larger than the GPU's L2 (no flush)",
            "parallelism": f"{Wn} emulated ranks per replica, {world} replica(s)"}


# The other four exchange configurations and the MoE fused dispatch and
# combine, each an entry of the default (cfg2) line: timed steps, roofline
# and a bit-exact check against the oracle outside the timed region.
CONFIG_ENTRIES = [
    ("cfg1", dict(workload="cfg1")),
    ("cfg3", dict(workload="cfg3")),
    ("cfg4", dict(workload="cfg4", seed=0)),
    ("cfg5", dict(workload="cfg5")),
    ("cfg3_fused_dispatch", dict(workload="cfg3", op="fused_dispatch")),
    ("cfg3_fused_combine", dict(workload="cfg3", op="fused_combine")),
]


def config_block(args) -> dict:
    import copy
    import torch
    out = {}
    for name, over in CONFIG_ENTRIES:
        a = copy.copy(args)
        a.workload, a.op, a.seed = over["workload"], over.get("op", "dispatch"), over.get("seed", 0)
        a.steps, a.warmup = 20, 3
        a.tokens, a.hidden, a.batch, a.dedup = 8192, 7168, 8192, False
        a.path, a.ctas_per_sm = "auto", 0
        a.no_cpu_baseline = False  # (the entry's bit-exact check runs with it)
        torch.cuda.empty_cache()
        if a.op == "fused_dispatch":
            line = run_fused_dispatch(a, light=True)
        elif a.op == "fused_combine":
            line = run_fused_combine(a, light=True)
        else:
            line = run_ours(a, light=True)
        r = line["roofline"]
        out[name] = {"workload": line["config"]["workload"], "op": a.op,
                     "us_per_step": round(line["ms_per_step"] * 1e3, 2),
                     "moved_GBps": line["value"], "kernel": r["kernel"], "frac": r["frac"],
                     "traffic": r["traffic"], "algorithmic_bytes": r["algorithmic_bytes_per_launch"],
                     "launches_per_step": line["gpu_launches"] // line["steps"],
                     "bit_exact": None if line["parity"] is None else line["parity"]["bit_exact"],
                     "clocks": line["clocks"]}
    return out


# ------------------------------------------------------ fused dispatch ----
# A spin kernel this long (about 1 ms at 2.07 GHz) runs ahead of every timed
# call of a multi-launch op, so that the host has enqueued the whole op before
# its first event is reached: the events then bracket device time only.  (A
# shorter spin, 125 us, let occasional host pauses of the Python binding land
# between the events.)
SPIN_CYCLES = 1 << 21


def _timed(torch, stream, fn, reps, cold, flush):
    """Median and mean device time of fn over reps calls (seconds), and the
    mean host time of one call (seconds, the Python binding and the launches,
    measured while the GPU is still busy with the spin kernel)."""
    ts, host = [], []
    for _ in range(reps):
        with torch.cuda.stream(stream):
            if cold:
                flush.sum()
            torch.cuda._sleep(SPIN_CYCLES)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        t0 = time.perf_counter()
        fn()
        host.append(time.perf_counter() - t0)
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b) / 1e3)
    return statistics.median(ts), statistics.mean(ts), statistics.mean(host)


def run_fused_dispatch(args, light=False):
    """a2av_dispatch on unsorted MoE or embedding-key items, against the
    unfused path (torch stable sort + row gather, then a2av_run).  Returns
    the JSON line; ``light`` skips the unfused path and the bound call (an
    entry of the cfg2 line's ``configs`` block)."""
    import torch
    import variable_size_all_gb300 as a2av
    import workloads as wl
    import oracle

    rank, local, world = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init("nccl")
    a2av.build()
    if args.workload not in ("cfg3", "cfg5"):
        raise SystemExit("--op fused_dispatch needs --workload cfg3 or cfg5")
    w = (wl.cfg3(args.seed, tokens=args.tokens, dedup=args.dedup, hidden=args.hidden)
         if args.workload == "cfg3" else wl.cfg5(args.seed, batch=args.batch))
    K, rows, src, key = wl.dispatch_items(w)
    Wn, rb, S = w.W, w.row_bytes, w.splits
    m = [k.size for k in key]
    T = moved_bytes(S, rb)
    d_rows = [torch.from_numpy(r).to(dev) for r in rows]
    d_src = [torch.from_numpy(x).to(dev) for x in src]
    d_key = [torch.from_numpy(x).to(dev) for x in key]
    d_pos = [torch.empty(x, dtype=torch.int64, device=dev) for x in m]
    recv = [int(S[:, p].sum()) * rb for p in range(Wn)]
    d_out = [torch.empty(n, dtype=torch.uint8, device=dev) for n in recv]
    d_so = torch.empty((Wn, 2, Wn), dtype=torch.int64, device=dev)
    eng = a2av.A2av(Wn)
    stream = torch.cuda.current_stream()
    cold = sum(r.size for r in rows) < 2 * L2_BYTES
    flush = torch.ones(128 << 20, dtype=torch.int32, device=dev)

    def fused():
        eng.dispatch(d_rows, d_src, d_key, K, d_out, d_so, d_pos, rb, stream=stream)

    u_out = [torch.empty_like(t) for t in d_out]
    u_so = torch.empty_like(d_so)

    def unfused():
        gathered, counts = [], []
        for r in range(Wn):
            order = torch.sort(d_key[r], stable=True).indices
            gathered.append(d_rows[r].view(-1, rb).index_select(0, d_src[r][order]).view(-1))
            counts.append(torch.bincount(d_key[r] // K, minlength=Wn))
        splits = torch.stack(counts).to(torch.int64)
        eng.run(gathered, splits, u_out, u_so, rb, stream=stream)

    for _ in range(args.warmup):
        fused()
        if not light:
            unfused()
    torch.cuda.synchronize()
    if eng.status() != a2av.OK:
        raise SystemExit("device reported an error during warm-up")
    with ClockSampler(local) as clocks:
        barrier()
        torch.cuda.synchronize()
        f_med, f_mean, f_host = _timed(torch, stream, fused, args.steps, cold, flush)
        torch.cuda.synchronize()
        barrier()
    u_med = u_mean = u_host = b_med = b_mean = b_host = None
    if not light:
        u_med, u_mean, u_host = _timed(torch, stream, unfused, max(3, args.steps // 4), cold,
                                       flush)
        # the same dispatch marshalled once (A2av.bind_dispatch): the host's share per call
        bound = eng.bind_dispatch(d_rows, d_src, d_key, K, d_out, d_so, d_pos, rb, stream=stream)
        b_med, b_mean, b_host = _timed(torch, stream, bound, args.steps, cold, flush)
    if eng.status() != a2av.OK:
        raise SystemExit("device reported an error during the timed region")
    max_s = reduce_max(f_mean, dev)
    value = whole_job_value(T / 1e9, world, max_s)
    # ideal traffic: every distinct source row read once (a token routed to
    # two experts is read once), every moved row written once, each item's
    # key and source row read once and its position written once
    items = sum(m)
    distinct = sum(int(np.unique(x).size) for x in src) * rb
    algo = distinct + T + items * (4 + 4 + 8) + 24 * Wn * Wn
    peak, peak_kind = hbm_peak()
    # the kernels the library enqueued for this dispatch (a2av_last_dispatch)
    chain = eng.last_dispatch()
    copy_kernel = chain["copy_kernel"]
    roofline = {"bound": "hbm", "kernel": f"a2av_dispatch (chain ending in {copy_kernel})",
                "achieved": round(algo / f_mean / 1e9, 1), "peak": peak, "peak_source": peak_kind,
                "unit": "GB/s", "frac": round(algo / f_mean / 1e9 / peak, 4),
                "traffic": measured_traffic(f"{copy_kernel}:{workload_key(args)}", algo),
                "algorithmic_bytes_per_launch": algo}
    cpu = parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        t0 = time.perf_counter()
        ref, ref_so, ref_pos, _ = oracle.default().dispatch_exchange(K, rows, src, key, rb)
        spent = time.perf_counter() - t0
        ok = all(np.array_equal(d_out[p].cpu().numpy(), ref[p]) for p in range(Wn))
        ok = ok and np.array_equal(d_so.cpu().numpy(), ref_so)
        ok = ok and all(np.array_equal(d_pos[r].cpu().numpy(), ref_pos[r]) for r in range(Wn))
        if not light:
            ok = ok and all(torch.equal(u_out[p], d_out[p]) for p in range(Wn))
        parity = {"bit_exact": bool(ok), "check": "outputs, offsets and positions equal the "
                                                  "oracle's" + ("" if light else
                                                                "; the unfused path agrees")}
        cpu = {"value": round(T / spent / 1e9, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": "the whole fused dispatch of the same workload", "seconds": round(spent, 3)}
        if not ok:
            raise SystemExit("fused dispatch differs from the oracle")
    eng.close()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(max_s * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic (seeded numpy draws; no dataset)",
        "config": {"workload": describe(args.workload, args.per_rank_bytes, args.seed,
                                        args.tokens, args.batch, args.dedup, hidden=args.hidden) +
                   " -- items unsorted (token-major / feature-major), grouped on the device",
                   "name": args.workload, "op": "fused_dispatch", "ranks": Wn, "row_bytes": rb,
                   "items": items, "keys_per_peer": K, "moved_bytes_per_step": T,
                   "l2": ("L2 flushed (512 MiB read) before every timed launch" if cold else
                          "inputs larger than L2"),
                   "timing": f"CUDA events around the dispatch ({chain['memsets']} memset and "
                             f"{chain['kernels']} kernel{'s' if chain['kernels'] != 1 else ''}, ending in {copy_kernel}), "
                             "mean over steps; a spin kernel ahead of each call keeps the "
                             "host's call time outside the events (fused_host_call_us)"},
        "unfused_torch_sort_gather_a2av": None if light else {
            "ms_mean": round(u_mean * 1e3, 4), "ms_median": round(u_med * 1e3, 4),
            "value": round(T / u_mean / 1e9, 2), "unit": UNIT,
            "host_call_us": round(u_host * 1e6, 1)},
        "fused_ms_median": round(f_med * 1e3, 4),
        "fused_host_call_us": round(f_host * 1e6, 1),
        "bound_call": None if light else {
            "ms_mean": round(b_mean * 1e3, 4), "ms_median": round(b_med * 1e3, 4),
            "host_call_us": round(b_host * 1e6, 1),
            "note": "A2av.bind_dispatch: arguments marshalled once"},
        "speedup_vs_unfused": None if light else round(u_mean / f_mean, 3),
        "roofline": roofline, "cpu_baseline": cpu, "e2e": None,
        "gpu_launches": chain["kernels"] * args.steps,
        "clocks": clocks.summary(), "parity": parity,
    }
    return line


# ------------------------------------------------------------- overlap ----
def run_fused_combine(args, light=False):
    """a2av_combine_items after a fused dispatch (cfg3, cfg5): every item's row
    back from the peers into item order, against the plain reverse exchange
    followed by a torch gather by sorted position.  Returns the JSON line;
    ``light`` skips the unfused path."""
    import torch
    import variable_size_all_gb300 as a2av
    import workloads as wl
    import oracle

    rank, local, world = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init("nccl")
    a2av.build()
    if args.workload not in ("cfg3", "cfg5"):
        raise SystemExit("--op fused_combine needs --workload cfg3 or cfg5")
    w = (wl.cfg3(args.seed, tokens=args.tokens, dedup=args.dedup, hidden=args.hidden)
         if args.workload == "cfg3" else wl.cfg5(args.seed, batch=args.batch))
    K, rows, src, key = wl.dispatch_items(w)
    Wn, rb, S = w.W, w.row_bytes, w.splits
    m = [k.size for k in key]
    T = moved_bytes(S, rb)
    d_rows = [torch.from_numpy(r).to(dev) for r in rows]
    d_src = [torch.from_numpy(x).to(dev) for x in src]
    d_key = [torch.from_numpy(x).to(dev) for x in key]
    d_pos = [torch.empty(x, dtype=torch.int64, device=dev) for x in m]
    d_out = [torch.empty(int(S[:, p].sum()) * rb, dtype=torch.uint8, device=dev)
             for p in range(Wn)]
    d_so = torch.empty((Wn, 2, Wn), dtype=torch.int64, device=dev)
    d_isp = torch.empty((Wn, Wn), dtype=torch.int64, device=dev)
    eng = a2av.A2av(Wn)
    stream = torch.cuda.current_stream()
    eng.dispatch(d_rows, d_src, d_key, K, d_out, d_so, d_pos, rb, in_splits=d_isp)
    items = [torch.empty(x * rb, dtype=torch.uint8, device=dev) for x in m]
    back = [torch.empty(int(S[r].sum()) * rb, dtype=torch.uint8, device=dev) for r in range(Wn)]
    cso = torch.empty_like(d_so)
    u_items = [torch.empty_like(t) for t in items]
    cold = sum(t.numel() for t in d_out) < 2 * L2_BYTES
    flush = torch.ones(128 << 20, dtype=torch.int32, device=dev)
    call = eng.bind_combine_items(d_out, d_isp, d_key, d_pos, K, items, rb, stream=stream)

    def unfused():
        eng.combine(d_out, d_so, back, cso, rb, stream=stream)
        for r in range(Wn):
            torch.index_select(back[r].view(-1, rb), 0, d_pos[r], out=u_items[r].view(-1, rb))

    for _ in range(args.warmup):
        call()
        if not light:
            unfused()
    torch.cuda.synchronize()
    if eng.status() != a2av.OK:
        raise SystemExit("device reported an error during warm-up")
    with ClockSampler(local) as clocks:
        barrier()
        torch.cuda.synchronize()
        f_med, f_mean, f_host = _timed(torch, stream, call, args.steps, cold, flush)
        torch.cuda.synchronize()
        barrier()
    u_med = u_mean = u_host = None
    if not light:
        u_med, u_mean, u_host = _timed(torch, stream, unfused, max(3, args.steps // 4), cold,
                                       flush)
    if eng.status() != a2av.OK:
        raise SystemExit("device reported an error during the timed region")
    max_s = reduce_max(f_mean, dev)
    value = whole_job_value(T / 1e9, world, max_s)
    # ideal traffic: every peer row read once, every item row written once,
    # each item's key and position read once
    algo = T + sum(m) * rb + sum(m) * (4 + 8) + 24 * Wn * Wn
    peak, peak_kind = hbm_peak()
    chain = eng.last_dispatch()  # the kernels the library enqueued for the combine
    copy_kernel = chain["copy_kernel"]
    roofline = {"bound": "hbm", "kernel": f"a2av_combine_items ({chain['kernels']} kernel"
                                          f"{'s' if chain['kernels'] != 1 else ''}, "
                                          f"ending in {copy_kernel})",
                "achieved": round(algo / f_mean / 1e9, 1), "peak": peak, "peak_source": peak_kind,
                "unit": "GB/s", "frac": round(algo / f_mean / 1e9 / peak, 4),
                "traffic": measured_traffic(f"{copy_kernel}:{workload_key(args)}_combine", algo),
                "algorithmic_bytes_per_launch": algo}
    cpu = parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        o = oracle.default()
        peers = [t.cpu().numpy() for t in d_out]
        Sg = d_isp.cpu().numpy()
        pos = [t.cpu().numpy() for t in d_pos]
        t0 = time.perf_counter()
        ref = o.combine_items_exchange(K, peers, Sg, key, pos, rb)
        spent = time.perf_counter() - t0
        ok = all(np.array_equal(items[r].cpu().numpy(), ref[r]) for r in range(Wn))
        ok = ok and all(np.array_equal(ref[r], rows[r].reshape(-1, rb)[src[r]].reshape(-1))
                        for r in range(Wn))
        if not light:
            ok = ok and all(torch.equal(u_items[r], items[r]) for r in range(Wn))
        parity = {"bit_exact": bool(ok), "check": "item rows equal the oracle's and the items' "
                                                  "source rows" + ("" if light else
                                                                   "; the unfused path agrees")}
        cpu = {"value": round(T / spent / 1e9, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": "the whole fused combine of the same workload", "seconds": round(spent, 3)}
        if not ok:
            raise SystemExit("fused combine differs from the oracle")
    eng.close()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(max_s * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic (seeded numpy draws; no dataset)",
        "config": {"workload": describe(args.workload, 0, args.seed, args.tokens, args.batch,
                                        args.dedup, hidden=args.hidden) +
                   " -- after the fused dispatch, every item's row back in item order",
                   "name": args.workload, "op": "fused_combine", "ranks": Wn, "row_bytes": rb,
                   "items": sum(m), "moved_bytes_per_step": T,
                   "l2": ("L2 flushed (512 MiB read) before every timed launch" if cold else
                          "inputs larger than L2"),
                   "timing": f"CUDA events around the bound call ({chain['memsets']} memset and "
                             f"{chain['kernels']} kernels), mean over steps; a spin kernel ahead "
                             "of each call"},
        "unfused_combine_then_gather": None if light else {
            "ms_mean": round(u_mean * 1e3, 4), "ms_median": round(u_med * 1e3, 4),
            "host_call_us": round(u_host * 1e6, 1)},
        "fused_ms_median": round(f_med * 1e3, 4), "fused_host_call_us": round(f_host * 1e6, 1),
        "speedup_vs_unfused": None if light else round(u_mean / f_mean, 3),
        "roofline": roofline, "cpu_baseline": cpu, "e2e": None,
        "gpu_launches": chain["kernels"] * args.steps,
        "clocks": clocks.summary(), "parity": parity,
    }
    return line


def device_exchange(torch, dev, w):
    """Device inputs, splits, outputs and out_splits_offsets for workload w."""
    S, rb = w.splits, w.row_bytes
    d_in = [torch.from_numpy(b).to(dev) for b in w.inputs]
    d_out = [torch.empty(int(S[:, p].sum()) * rb, dtype=torch.uint8, device=dev)
             for p in range(w.W)]
    return (d_in, torch.from_numpy(S).to(dev), d_out,
            torch.empty((w.W, 2, w.W), dtype=torch.int64, device=dev))


def run_kjt(args):
    """The keyed-jagged exchange of an embedding batch (cfg5): the int32 bag
    lengths and the int64 keys, two a2av_run calls per step -- the key
    exchange torchrec PR 2570 moves to its own stream, with the lengths that
    cut the keys into bags.  Timed as one stream (PDL lets the keys' launch
    overlap the lengths' tail), without PDL, on two streams, and as one
    captured CUDA graph."""
    import torch
    import variable_size_all_gb300 as a2av
    import workloads as wl

    rank, local, world = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init("nccl")
    a2av.build()
    if args.workload != "cfg5":
        raise SystemExit("--op kjt runs the keyed-jagged exchange: --workload cfg5")
    w = wl.cfg5(args.seed, batch=args.batch)
    lw = wl.cfg5_lengths(w)
    parts = [lw, w]
    Wn = w.W
    T = sum(moved_bytes(x.splits, x.row_bytes) for x in parts)
    bufs = [device_exchange(torch, dev, x) for x in parts]
    eng = a2av.A2av(Wn)
    saved = os.environ.get("A2AV_PDL")
    os.environ["A2AV_PDL"] = "0"  # read once, when the handle is made
    try:
        eng_plain = a2av.A2av(Wn)
    finally:
        if saved is None:
            del os.environ["A2AV_PDL"]
        else:
            os.environ["A2AV_PDL"] = saved
    stream, side = torch.cuda.current_stream(), torch.cuda.Stream()
    flush = torch.ones(128 << 20, dtype=torch.int32, device=dev)

    def one_stream(e=eng, st=stream):
        for (d_in, d_S, d_out, d_so), x in zip(bufs, parts):
            e.run(d_in, d_S, d_out, d_so, x.row_bytes, stream=st)

    def two_streams():
        fork = torch.cuda.Event()
        fork.record(stream)
        side.wait_event(fork)
        (l_in, l_S, l_out, l_so), (k_in, k_S, k_out, k_so) = bufs
        eng.run(l_in, l_S, l_out, l_so, lw.row_bytes, stream=side)
        eng.run(k_in, k_S, k_out, k_so, w.row_bytes, stream=stream)
        join = torch.cuda.Event()
        join.record(side)
        stream.wait_event(join)

    for _ in range(args.warmup):
        one_stream()
        one_stream(eng_plain)
        two_streams()
    torch.cuda.synchronize()
    g_stream = torch.cuda.Stream()
    g_stream.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=g_stream):
        one_stream(eng, g_stream)
    torch.cuda.synchronize()
    def one_launch():
        eng.run_multi([(*b, x.row_bytes) for b, x in zip(bufs, parts)])

    for _ in range(args.warmup):
        one_launch()
    bound = eng.bind_run_multi([(*b, x.row_bytes) for b, x in zip(bufs, parts)], stream=stream)
    variants = {"one_launch": one_launch, "one_launch_bound": bound, "one_stream_pdl": one_stream,
                "one_stream_no_pdl": lambda: one_stream(eng_plain),
                "two_streams": two_streams, "cuda_graph": graph.replay}
    times = {}
    with ClockSampler(local) as clocks:
        barrier()
        torch.cuda.synchronize()
        for name, fn in variants.items():
            times[name] = _timed(torch, stream, fn, args.steps, True, flush)
        torch.cuda.synchronize()
        barrier()
    for e in (eng, eng_plain):
        if e.status() != a2av.OK:
            raise SystemExit("device reported an error during the timed region")
    t_mean = times["one_launch"][1]
    max_s = reduce_max(t_mean, dev)
    value = whole_job_value(T / 1e9, world, max_s)
    algo = sum(algorithmic_bytes(x.splits, x.row_bytes) for x in parts)
    peak, peak_kind = hbm_peak()
    roofline = {"bound": "hbm", "kernel": "a2av_staged_multi_kernel (lengths and keys, one launch)",
                "achieved": round(algo / t_mean / 1e9, 1), "peak": peak, "peak_source": peak_kind,
                "unit": "GB/s", "frac": round(algo / t_mean / 1e9 / peak, 4),
                "traffic": measured_traffic("a2av_staged_multi_kernel:cfg5_kjt", algo),
                "algorithmic_bytes_per_launch": algo}
    alone = {}  # each exchange by itself
    for (d_in, d_S, d_out, d_so), x in zip(bufs, parts):
        alone[x.name] = _timed(torch, stream, lambda: eng.run(d_in, d_S, d_out, d_so, x.row_bytes),
                               args.steps, True, flush)[1]
    cpu = parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        t0 = time.perf_counter()
        refs = [oracle.default().exchange(x.inputs, x.splits, x.row_bytes) for x in parts]
        spent = time.perf_counter() - t0
        ok = True
        for (_, _, d_out, d_so), (ref, ref_so) in zip(bufs, refs):
            ok = ok and np.array_equal(d_so.cpu().numpy(), ref_so)
            ok = ok and all(np.array_equal(d_out[p].cpu().numpy(), ref[p]) for p in range(Wn))
        # the received lengths count the received keys, per source rank
        l_out, l_so = bufs[0][2], bufs[0][3].cpu().numpy()
        k_so = bufs[1][3].cpu().numpy()
        for p in range(Wn):
            got = l_out[p].cpu().numpy().view(np.int32)
            for r in range(Wn):
                o0, n0 = int(l_so[p][1][r]), int(l_so[p][0][r])
                ok = ok and int(got[o0:o0 + n0].sum()) == int(k_so[p][0][r])
        parity = {"bit_exact": bool(ok), "check": "lengths and keys equal the oracle's; the "
                                                  "received lengths sum to the received key counts"}
        cpu = {"value": round(T / spent / 1e9, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": "both exchanges (lengths, keys) of the same batch",
               "seconds": round(spent, 3)}
        if not ok:
            raise SystemExit("keyed-jagged exchange differs from the oracle")
    eng.close()
    eng_plain.close()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(max_s * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic (seeded numpy draws; no dataset)",
        "config": {"workload": describe("cfg5", 0, args.seed, batch=args.batch) +
                   " -- with its bag lengths (int32, one per feature and bag): both "
                   "exchanges in one a2av_run_multi launch per step", "name": "cfg5",
                   "op": "kjt", "ranks": Wn,
                   "moved_bytes_per_step": T,
                   "l2": "L2 flushed (512 MiB read) before every timed step",
                   "timing": "CUDA events around the step, mean over steps; a spin kernel "
                             "ahead of each step keeps the host's call time outside"},
        "variants_us": {k: {"mean": round(v[1] * 1e6, 2), "median": round(v[0] * 1e6, 2),
                            "host_call": round(v[2] * 1e6, 1)} for k, v in times.items()},
        "alone_us": {k: round(v * 1e6, 2) for k, v in alone.items()},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": None, "gpu_launches": args.steps,
        "clocks": clocks.summary(), "parity": parity,
    }
    if rank == 0:
        emit(line)


def run_overlap(args):
    """The exchange on a side stream while a bf16 GEMM runs on the main one:
    each alone, then both at once (the separate-stream idea of torchrec PR
    2570, measured here as HBM interference inside one GPU)."""
    import torch
    import variable_size_all_gb300 as a2av
    import workloads as wl

    rank, local, world = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init("nccl")
    a2av.build()
    if args.workload == "cfg3":
        w = wl.cfg3(args.seed, tokens=args.tokens, dedup=args.dedup, hidden=args.hidden)
        parts = [w]  # the MoE token exchange
    elif args.workload == "cfg5":
        w = wl.cfg5(args.seed, batch=args.batch)
        parts = [wl.cfg5_lengths(w), w]  # a keyed-jagged batch: bag lengths, then keys
    else:
        raise SystemExit("--op overlap runs the MoE exchange (cfg3) or the keyed-jagged "
                         "exchange of bag lengths and keys (cfg5)")
    Wn = w.W
    T = sum(moved_bytes(x.splits, x.row_bytes) for x in parts)
    bufs = [device_exchange(torch, dev, x) for x in parts]
    n = args.gemm_n
    A = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
    B = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
    C = torch.empty(n, n, device=dev, dtype=torch.bfloat16)
    eng = a2av.A2av(Wn)
    main, side = torch.cuda.current_stream(), torch.cuda.Stream()
    reps = args.steps

    def gemms():
        for _ in range(reps):
            torch.matmul(A, B, out=C)

    def exchanges():
        for _ in range(reps):
            for (d_in, d_S, d_out, d_so), x in zip(bufs, parts):
                eng.run(d_in, d_S, d_out, d_so, x.row_bytes, stream=side)

    def span(fn_main, fn_side):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c, d = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(main)
        side.wait_event(a)
        if fn_main:
            fn_main()
        b.record(main)
        with torch.cuda.stream(side):
            c.record(side)
            if fn_side:
                fn_side()
            d.record(side)
        main.wait_stream(side)
        torch.cuda.synchronize()
        wall = max(a.elapsed_time(b), a.elapsed_time(d)) / 1e3
        return a.elapsed_time(b) / 1e3, c.elapsed_time(d) / 1e3, wall

    for _ in range(2):
        span(gemms, exchanges)
    g_alone = span(gemms, None)[0]
    x_alone = span(None, exchanges)[1]
    with ClockSampler(local) as clocks:
        g_both, x_both, wall = span(gemms, exchanges)
    # The same with the side stream at the highest priority: the block
    # scheduler then hands SMs freed by the GEMMs to the exchange first.
    lo, hi = torch.cuda.Stream.priority_range() if hasattr(torch.cuda.Stream, "priority_range") \
        else (0, -1)
    side = torch.cuda.Stream(priority=min(lo, hi))
    for _ in range(2):
        span(gemms, exchanges)
    g_hp, x_hp, wall_hp = span(gemms, exchanges)
    if eng.status() != a2av.OK:
        raise SystemExit("device reported an error")
    eng.close()
    parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        ok = True
        for (_, _, d_out, d_so), x in zip(bufs, parts):
            ref, ref_so = oracle.default().exchange(x.inputs, x.splits, x.row_bytes)
            ok = ok and np.array_equal(d_so.cpu().numpy(), ref_so)
            ok = ok and all(np.array_equal(d_out[p].cpu().numpy(), ref[p]) for p in range(Wn))
        parity = {"bit_exact": bool(ok), "check": "outputs and offsets equal the oracle's"}
        if not ok:
            raise SystemExit("overlapped exchange differs from the oracle")
    flops = 2.0 * n * n * n * reps
    line = {
        "metric": METRIC, "value": round(T * reps / x_both / 1e9, 2), "unit": UNIT,
        "n_gpus": world, "steps": reps, "warmup": 2, "ms_per_step": round(x_both / reps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic",
        "config": {"workload": describe(args.workload, 0, args.seed, args.tokens, args.batch,
                                        args.dedup, hidden=args.hidden) +
                   (" (bag lengths, int32, then keys: two a2av_run per step)"
                    if args.workload == "cfg5" else "") +
                   f" on a side stream, with {reps} bf16 GEMMs {n}x{n}x{n} on the main stream",
                   "name": args.workload, "op": "overlap"},
        "exchange_alone_GBps": round(T * reps / x_alone / 1e9, 2),
        "exchange_overlapped_GBps": round(T * reps / x_both / 1e9, 2),
        "gemm_alone_TFLOPs": round(flops / g_alone / 1e12, 1),
        "gemm_overlapped_TFLOPs": round(flops / g_both / 1e12, 1),
        "serial_ms": round((g_alone + x_alone) * 1e3, 3), "overlapped_wall_ms": round(wall * 1e3, 3),
        "overlap_saving": round(1 - wall / (g_alone + x_alone), 4),
        "high_priority_side_stream": {
            "exchange_overlapped_GBps": round(T * reps / x_hp / 1e9, 2),
            "exchange_ms_per_step": round(x_hp / reps * 1e3, 4),
            "gemm_overlapped_TFLOPs": round(flops / g_hp / 1e12, 1),
            "overlapped_wall_ms": round(wall_hp * 1e3, 3),
            "overlap_saving": round(1 - wall_hp / (g_alone + x_alone), 4)},
        "gpu_launches": reps * len(parts), "clocks": clocks.summary(), "roofline": None,
        "cpu_baseline": None, "e2e": None, "parity": parity,
    }
    if rank == 0:
        emit(line)


# ------------------------------------------------------------ reference ----
def run_reference(args):
    """The CPU oracle as the reference arm: each step runs it on one peer's
    whole output of the same workload (a bounded sample), one host core."""
    rank, _, world = dist_env()
    if rank != 0:
        return
    import workloads as wl
    P = args.per_rank_bytes
    if args.workload == "cfg2":
        w = wl.cfg2(P, seed=args.seed)
    else:
        w = {"cfg1": wl.cfg1,
             "cfg3": lambda s: wl.cfg3(s, tokens=args.tokens, dedup=args.dedup,
                                       hidden=args.hidden),
             "cfg4": wl.cfg4,
             "cfg5": lambda s: wl.cfg5(s, batch=args.batch)}[args.workload](args.seed)
    S, inputs, rb, Wn = w.splits, w.inputs, w.row_bytes, w.W
    K, Wm = args.steps, args.warmup
    for k in range(Wm):
        time_oracle(inputs, S, rb, 0.0, peers=[k % Wn])
    total_s, total_b = 0.0, 0
    for k in range(K):
        s, b, _ = time_oracle(inputs, S, rb, 0.0, peers=[k % Wn])
        total_s += s
        total_b += b
    value = total_b / total_s / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": world, "steps": K, "warmup": Wm, "ms_per_step": round(total_s * 1e3 / K, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic (seeded numpy draws; no dataset)",
        # the same config dict as this workload's GPU line
        "config": exchange_config(args, Wn, rb, int(statistics.mean(b.size for b in inputs)),
                                  moved_bytes(S, rb), sum(b.size for b in inputs) < 2 * L2_BYTES,
                                  world),
        "implementation": "the CPU oracle (C, one host core)",
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"one peer's whole output per step (peer = step mod {Wn})"},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    emit(line)


def free_port() -> int:
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def spawn_replicas(n: int, argv, script=None) -> int:
    """Start n local processes of this script with the rank variables a
    torchrun launch sets (rendezvous on 127.0.0.1); returns the worst exit
    code.  Only rank 0 prints the JSON line."""
    script = script or os.path.abspath(__file__)
    port = free_port()
    procs = []
    for r in range(n):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(n),
                   LOCAL_WORLD_SIZE=str(n), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, script, *argv], env=env))
    codes = [p.wait() for p in procs]
    return max(codes, key=abs)


def main(argv=None):
    argv = list(sys.argv[1:] if argv is None else argv)
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=WORKLOADS, default="cfg2")
    ap.add_argument("--op", choices=["dispatch", "combine", "fused_dispatch", "fused_combine",
                                     "overlap", "kjt"],
                    default="dispatch",
                    help="dispatch = a2av_run; combine = a2av_combine on its outputs; "
                         "fused_dispatch = a2av_dispatch on unsorted items (cfg3, cfg5); "
                         "overlap = the exchange (cfg3; cfg5: bag lengths and keys) on a side "
                         "stream beside bf16 GEMMs; kjt = cfg5 bag lengths + keys in one "
                         "a2av_run_multi launch (and as two a2av_run calls)")
    ap.add_argument("--gemm-n", type=int, default=8192)
    ap.add_argument("--tokens", type=int, default=8192, help="cfg3 tokens per rank")
    ap.add_argument("--batch", type=int, default=8192, help="cfg5 bags per feature and rank")
    ap.add_argument("--hidden", type=int, default=7168, help="cfg3 hidden size (bf16 elements)")
    ap.add_argument("--dedup", action="store_true",
                    help="cfg3: one row per distinct (token, destination rank) pair")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--per-rank-bytes", type=int, default=1 << 32, help="cfg2 payload per rank")
    ap.add_argument("--path", choices=["auto", "vector", "bulk", "staged"], default="auto")
    ap.add_argument("--ctas-per-sm", type=int, default=0)
    ap.add_argument("--sweep-reps", type=int, default=20)
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="cfg2 line: skip the other workloads' block (configs)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # timing rule: at least 3 warm-up steps
    world_env = os.environ.get("WORLD_SIZE")
    if world_env is None and args.gpus > 1:
        # N replicas without an external launcher: one process per GPU here
        raise SystemExit(spawn_replicas(args.gpus, argv))
    if world_env is not None and int(world_env) != args.gpus:
        raise SystemExit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world_env}: "
                         "launch one process per GPU (torchrun --nproc-per-node N, or "
                         "bench.py --gpus N alone)")
    if args.impl == "reference":
        run_reference(args)
    elif args.op == "fused_dispatch":
        line = run_fused_dispatch(args)
        if dist_env()[0] == 0:
            emit(line)
    elif args.op == "overlap":
        run_overlap(args)
    elif args.op == "kjt":
        run_kjt(args)
    elif args.op == "fused_combine":
        line = run_fused_combine(args)
        if dist_env()[0] == 0:
            emit(line)
    else:
        line = run_ours(args)
        if args.workload == "cfg2" and args.op == "dispatch" and not args.no_configs:
            line["configs"] = config_block(args)
        if dist_env()[0] == 0:
            emit(line)


if __name__ == "__main__":
    main()
