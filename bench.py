"""Benchmark of the speculative-decoding verify step on one GB300 (or N, one process each).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config 0..4] [--mode sampling|greedy] [--all]

A step is one sampling-mode verify call (row statistics, first-reject scan, residual or bonus
race: every step of the path) over one batch of the throughput-stress workload (B=256,
gamma=12, V=152064 bf16; 1.95 GB of logits, larger than L2, so no flush is needed between
steps).  Rank 0 prints one JSON line:

  value        verified logit rows per second, B*(gamma+1) rows per call, inputs resident
  e2e          the same through the C ABI with the step's inputs copied from pinned host
               memory and the outputs read back inside the timed region
  roofline     the row-statistics kernel (the dominant one): one read of every logit per
               launch / its CUDA-event duration, against the measured HBM copy bandwidth
  cpu_baseline the CPU oracle on a bounded sample of the same workload, on 1 host core

``--impl reference`` times the CPU oracle as the reference arm (there is no reference code to
install: the pages describe the method only).  With ``--gpus N`` (N > 1) the script starts N
ranks itself, one process per GPU, unless a launcher such as torchrun already set WORLD_SIZE;
every rank verifies its own batch (global sequence indices offset by rank) with no collective
on the data path, and the line reports the slowest rank's time.  The line also carries a
sustained leg (the step for over a second, clocks sampled inside it) and ``per_config``: the
other four workloads (and the greedy modes) with rotating input copies where one copy fits in
L2, each with its kernel split, roofline fraction and the oracle's one-core rate.
"""
from __future__ import annotations

import argparse
import contextlib
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "spec-verify logit rows/s (B*(gamma+1) rows of V) and achieved HBM GB/s vs peak"
UNIT = "rows/s"

# DRAM traffic of one row-statistics launch on the throughput workload, from the ncu capture
# summarised in profiles/ (dram__bytes_read.sum + dram__bytes_write.sum), with the hash of
# the code it was taken on (the element types and the row-statistics kernel with the piece
# choice and the helpers it calls); reported as null once that code has changed.
NCU_TRAFFIC = {"bytes": 1949927680, "sources_sha1": "26041dca03e6079a385837ca77d81ca2ff8828bc"}
ROW_STATS_SPAN = ("inline int pick_piece_len(", "// Per-position entropies and KL divergence")


@contextlib.contextmanager
def nvtx(name: str):
    """An NVTX range around a phase of the run (host markers only, outside the timed kernel
    work), so that a profiler can select it (`ncu --nvtx --nvtx-include name/`); nothing if
    torch has no NVTX."""
    import torch
    try:
        torch.cuda.nvtx.range_push(name)
        pushed = True
    except Exception:
        pushed = False
    try:
        yield
    finally:
        if pushed:
            torch.cuda.nvtx.range_pop()


def kernel_sources_sha1() -> str:
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "speculative_decoding_verification_31_gb300", "csrc")
    with open(os.path.join(csrc, "device_common.cuh"), "rb") as fh:
        h.update(fh.read())
    with open(os.path.join(csrc, "kernels.cuh"), "r") as fh:
        text = fh.read()
    a = text.index(ROW_STATS_SPAN[0])
    h.update(text[a:text.index(ROW_STATS_SPAN[1], a)].encode())
    return h.hexdigest()


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


# -------------------------------------------------------------------------------------------
# clocks during the timed region
# -------------------------------------------------------------------------------------------

CLOCK_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: int, interval_ms: int = 50):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(gpu_index), "-lms", str(interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]
        return self.lines

    @staticmethod
    def summarise(lines, t0: float, t1: float):
        rows = []
        for l in lines:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts, float(parts[2]), float(parts[3]), parts[5:]))
            except (ValueError, IndexError):
                continue
        if not rows:
            return None
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        window = "timed region"
        if len(inside) < 2:
            inside = [r for r in rows if r[0] <= t1 + 0.05][-5:] or rows[-5:]
            window = "nearest samples (timed region shorter than the sampling interval)"
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inside:
            for name, v in zip(names, r[3][1:5]):
                if v.strip().lower() in ("active", "1", "yes"):
                    reasons.add(name)
        return {"sm_mhz": float(np.median([r[1] for r in inside])),
                "sm_max_mhz": float(max(r[2] for r in inside)),
                "reasons": sorted(reasons), "samples": len(inside), "window": window}


# -------------------------------------------------------------------------------------------
# helpers
# -------------------------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def to_torch(a: np.ndarray, dtype: str):
    import torch
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))


def cpu_oracle_rate(w, seed: int, budget_s: float, max_seqs: int):
    """Time the CPU oracle on whole sequences of workload w (cycling through its first
    max_seqs sequences, in batches sized to the remaining budget) until about budget_s
    seconds.  Returns (rows/s, sequences verified, seconds)."""
    import oracle
    orc = oracle.get()
    done, rows, t_total = 0, 0, 0.0
    n, pool = 1, min(max_seqs, w.B)
    while t_total < budget_s:
        lo = done % pool
        k = min(n, pool - lo)
        sl = slice(lo, lo + k)
        t0 = time.perf_counter()
        orc.verify(w.target[sl], w.draft[sl], w.tokens[sl], w.T[sl], w.Td[sl], seed, b_base=lo)
        t_total += time.perf_counter() - t0
        done += k
        rows += k * (w.gamma + 1)
        per = t_total / done
        n = max(1, int((budget_s - t_total) / per)) if per > 0 else 1
    return rows / t_total, done, t_total


# -------------------------------------------------------------------------------------------
# our arm
# -------------------------------------------------------------------------------------------

def early_exit_rows_read(n: np.ndarray, gamma: int) -> tuple[int, int]:
    """Logit rows the early-exit path streams for accepted counts n (target and draft rows of
    every position up to the first rejection, plus the bonus row when all are accepted), and
    the rows the race then reads again."""
    streamed = raced = 0
    for j in n.tolist():
        if j < 0:
            continue
        streamed += 2 * (j + 1) if j < gamma else 2 * gamma + 1
        raced += 2 if j < gamma else 1
    return streamed, raced


def device_copies(w, dev, l2: int, greedy: bool):
    """The workload's logits on the device, as `copies` back-to-back copies whose total
    exceeds twice L2 when one copy alone would not (calls rotate over them, so every call
    reads HBM, not a warm L2); one copy otherwise.  Returns (targets, drafts, copies)."""
    import torch
    nbytes = w.bytes_greedy() if greedy else w.bytes_sampling()
    copies = 1 if nbytes > 2 * l2 else int(-(-2 * l2 // nbytes)) + 1
    t = to_torch(w.target, w.dtype).to(dev)
    d = to_torch(w.draft, w.dtype).to(dev)
    tb = t.unsqueeze(0).expand(copies, *t.shape).contiguous()
    db = d.unsqueeze(0).expand(copies, *d.shape).contiguous()
    return tb, db, copies


def time_calls(call, n: int, stream) -> float:
    """Mean ms per call over n calls (call(k) issues call k), CUDA events on `stream`, after
    warm-up calls."""
    import torch
    for k in range(5):
        call(k)
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for k in range(n):
        call(k)
    s1.record(stream)
    torch.cuda.synchronize()
    return s0.elapsed_time(s1) / n


def time_graph_calls(call, copies: int, stream):
    """Mean ms per call when the calls are replayed from a CUDA graph (no host work between
    them): the graph holds one call per input copy (at most 4096, at least 50 calls), and is
    replayed until about 0.2 s have passed.  Returns (ms per call, calls timed), or
    (None, error text) when the calls cannot be captured."""
    import torch
    n = min(copies, 4096) if copies > 1 else 50
    g = torch.cuda.CUDAGraph()
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for k in range(3):
                call(k)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            for k in range(n):
                call(k)
        torch.cuda.synchronize()
    except Exception as e:  # a launch that stream capture does not take
        torch.cuda.synchronize()
        return None, f"{type(e).__name__}: {str(e)[:120]}"
    g.replay()
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    g.replay()
    s1.record(stream)
    torch.cuda.synchronize()
    reps = max(1, int(200.0 / max(s0.elapsed_time(s1), 1e-3)))
    s0.record(stream)
    for _ in range(reps):
        g.replay()
    s1.record(stream)
    torch.cuda.synchronize()
    return s0.elapsed_time(s1) / (reps * n), reps * n


def kernel_split_ms(call_events, n: int, nkern: int, stream) -> list:
    """Mean CUDA-event time of each of a call's nkern kernels over n calls (events recorded
    between the kernels, which also turns their programmatic launch off)."""
    import torch
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nkern + 1)] for _ in range(n)]
    for e in evs:
        for ev in e:
            ev.record(stream)
    torch.cuda.synchronize()
    for k in range(n):
        call_events(k, evs[k])
    torch.cuda.synchronize()
    return [float(np.mean([e[i].elapsed_time(e[i + 1]) for e in evs])) for i in range(nkern)]


def measure_config(sv, cfg: int, dev, stream, seed: int, seq_base: int, l2: int, peak: float,
                   cpu_seconds: float):
    """One named workload on this GPU: the default sampling call, the early-exit call and
    (where the workload has one) the greedy call, each as us/call, rows/s, GB/s of one read
    of the logits and its fraction of the measured HBM bandwidth, with the split between the
    call's kernels; and the CPU oracle on one core over a bounded sample."""
    import torch
    import workloads
    out = {"workload": workloads.CONFIG_NAMES[cfg]}
    modes = ["sampling", "early_exit"] + (["greedy"] if cfg in (1, 3, 4) else [])
    if cfg == 4:
        modes = ["greedy"]  # the sampling paths of this workload are the line's headline
    w_s = None
    for mode in modes:
        greedy = mode == "greedy"
        w = workloads.config(cfg, greedy=greedy)
        if not greedy:
            w_s = w
        tb, db, copies = device_copies(w, dev, l2, greedy)
        tok = torch.from_numpy(w.tokens).to(dev)
        Tq, Tdq = torch.from_numpy(w.T).to(dev), torch.from_numpy(w.Td).to(dev)
        kw = dict(T_per_seq=Tq, Td_per_seq=Tdq) if cfg == 3 else {}
        out_t = torch.empty((w.B, w.gamma + 1), dtype=torch.int32, device=dev)
        out_n = torch.empty((w.B,), dtype=torch.int32, device=dev)
        flags = sv.SPEC_FLAG_EARLY_EXIT if mode == "early_exit" else 0

        def call(k, events=None):
            c = k % copies
            if greedy:
                sv.spec_verify_greedy_ex(tb[c], tok, out_t, out_n, prof_events=events)
            else:
                sv.spec_verify_ex(tb[c], db[c], tok, float(w.T[0]), float(w.Td[0]), seed, out_t,
                                  out_n, seq_index_base=seq_base, flags=flags,
                                  prof_events=events, **kw)

        with nvtx(f"workload {cfg} {mode}"):
            est = time_calls(call, 20, stream)
            n = int(max(200, min(20000, 250.0 / max(est, 1e-3))))
            ms_api = time_calls(call, n, stream)
            ms, ng = time_graph_calls(call, copies, stream)
        status = sv.spec_verify_check()
        nbytes = w.bytes_greedy() if greedy else w.bytes_sampling()
        timing = "CUDA graph replay of the calls (device time, no host work between calls)"
        if ms is None:  # not capturable: the Python loop's time
            timing, ms, ng = f"Python loop (graph capture failed: {ng})", ms_api, n
        entry = {"us_per_call": ms * 1e3, "rows_per_s": w.rows / (ms / 1e3), "calls": ng,
                 "timing": timing,
                 "us_per_call_python_api": ms_api * 1e3,
                 "GBps_one_read": nbytes / (ms / 1e3) / 1e9,
                 "frac_of_measured_hbm": nbytes / (ms / 1e3) / 1e9 / peak,
                 "inputs": (f"{copies} rotating copies ({copies * nbytes / 1e6:.0f} MB > 2x L2)"
                            if copies > 1 else "one copy, larger than 2x L2"),
                 "status": status}
        if mode == "early_exit":
            streamed, raced = early_exit_rows_read(out_n.cpu().numpy(), w.gamma)
            es_ = 2 if w.dtype == "bf16" else 4
            entry["logit_bytes_read_per_call"] = (streamed + raced) * w.V * es_
            entry["note"] = ("same outputs; reads rows only up to each sequence's first "
                             "rejection: GBps_one_read is the full read's bytes over this time")
        else:
            names = ["row_argmax", "scan_greedy"] if greedy else ["row_stats", "scan_race"]
            kms = kernel_split_ms(lambda k, ev: call(k, ev), min(n, 500), 2, stream)
            entry["kernel_us"] = {nm: v * 1e3 for nm, v in zip(names, kms)}
            entry["dominant"] = names[0]
            entry["dominant_frac_of_measured_hbm"] = nbytes / (kms[0] / 1e3) / 1e9 / peak
        out[mode] = entry
        del tb, db
    if w_s is not None and cpu_seconds > 0:
        rate, nseq, secs = cpu_oracle_rate(w_s, seed, cpu_seconds, max_seqs=w_s.B)
        out["cpu_oracle"] = {"rows_per_s": rate, "cores": 1,
                             "sample": f"{nseq} sequence verifications (cycling over the {w_s.B} of the "
                                       f"workload), {secs:.2f} s, single-threaded C"}
    return out


def run_ours(args):
    import torch
    import workloads
    import speculative_decoding_verification_31_gb300 as sv

    ws_, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws_ > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    sv.load_library()

    cfg = args.config
    w = workloads.config(cfg, greedy=(args.mode == "greedy"))
    t = to_torch(w.target, w.dtype).to(dev)
    d = to_torch(w.draft, w.dtype).to(dev)
    tok = torch.from_numpy(w.tokens).to(dev)
    Tq = torch.from_numpy(w.T).to(dev)
    Tdq = torch.from_numpy(w.Td).to(dev)
    per_seq = cfg == 3
    out_t = torch.empty((w.B, w.gamma + 1), dtype=torch.int32, device=dev)
    out_n = torch.empty((w.B,), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    seq_base = rank * w.B
    greedy = args.mode == "greedy"
    nkern = 2  # sampling: row_stats, scan_race; greedy: row_argmax, scan_greedy

    def step(events=None, tgt=t, drf=d, tk=tok):
        if greedy:
            sv.spec_verify_greedy_ex(tgt, tk, out_t, out_n, prof_events=events)
        else:
            kw = dict(T_per_seq=Tq, Td_per_seq=Tdq) if per_seq else {}
            sv.spec_verify_ex(tgt, drf, tk, float(w.T[0]), float(w.Td[0]), args.seed, out_t,
                              out_n, seq_index_base=seq_base, prof_events=events, **kw)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    status = sv.spec_verify_check()
    if status != sv.SPEC_OK:
        raise RuntimeError(f"device status after warm-up: {sv.spec_verify_strerror(status)}")

    K = args.steps
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.15 if sampler else 0)
    if ws_ > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with nvtx("timed steps"):
        h0 = time.time()
        start.record(stream)
        for k in range(K):
            step()
        end.record(stream)
        torch.cuda.synchronize()
        h1 = time.time()
    if ws_ > 1:
        torch.distributed.barrier()
    clocks = None
    if sampler:
        clocks = ClockSampler.summarise(sampler.stop(), h0, h1)
    ms = start.elapsed_time(end)
    # Sustained leg: the same step for at least a second (however few steps the timed region
    # above has), with the clocks sampled inside it.
    sustained = None
    if not args.no_sustained:
        Ks = int(np.ceil(args.sustained_seconds * 1e3 / max(ms / K, 1e-3)))
        sampler2 = ClockSampler(local) if rank == 0 else None
        time.sleep(0.15 if sampler2 else 0)
        if ws_ > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        g0 = time.time()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with nvtx("sustained steps"):
            s0.record(stream)
            for _ in range(Ks):
                step()
            s1.record(stream)
            torch.cuda.synchronize()
        g1 = time.time()
        sms = s0.elapsed_time(s1)
        if ws_ > 1:
            mt = torch.tensor([sms], device=dev, dtype=torch.float64)
            torch.distributed.all_reduce(mt, op=torch.distributed.ReduceOp.MAX)
            sms = float(mt.item())
        sustained = {"value": ws_ * w.rows * Ks / (sms / 1e3), "unit": UNIT, "steps": Ks,
                     "seconds": sms / 1e3, "ms_per_step": sms / Ks,
                     "clocks": ClockSampler.summarise(sampler2.stop(), g0, g1) if sampler2 else None}
    # Roofline pass: the same steps again with events around each kernel (an event between
    # the two kernels turns off the programmatic dependent launch, so these steps are not
    # the timed ones).
    Kr = min(K, 500)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nkern + 1)] for _ in range(Kr)]
    for e in evs:  # torch creates the CUDA event on first record: make the handles real
        for ev in e:
            ev.record(stream)
    torch.cuda.synchronize()
    with nvtx("roofline pass"):
        for k in range(Kr):
            step(evs[k])
        torch.cuda.synchronize()
    kern_ms = [float(np.mean([e[i].elapsed_time(e[i + 1]) for e in evs])) for i in range(nkern)]
    if ws_ > 1:
        mt = torch.tensor([ms], device=dev, dtype=torch.float64)
        torch.distributed.all_reduce(mt, op=torch.distributed.ReduceOp.MAX)
        ms = float(mt.item())
    status = sv.spec_verify_check()
    if status != sv.SPEC_OK:
        raise RuntimeError(f"device status after timing: {sv.spec_verify_strerror(status)}")

    ms_step = ms / K
    rows_total = ws_ * w.rows * K
    value = rows_total / (ms / 1e3)

    # roofline of the dominant kernel (row statistics / row argmax)
    alg_bytes = w.bytes_greedy() if greedy else w.bytes_sampling()
    peaks = measured_peaks()
    achieved = alg_bytes / (kern_ms[0] / 1e3) / 1e9
    traffic = None
    if NCU_TRAFFIC["bytes"] and NCU_TRAFFIC["sources_sha1"] == kernel_sources_sha1() and cfg == 4:
        traffic = NCU_TRAFFIC["bytes"]

    # the early-exit path (SPEC_FLAG_EARLY_EXIT) on the same inputs, with the bytes it reads
    early = None
    if not greedy:
        def estep():
            kw = dict(T_per_seq=Tq, Td_per_seq=Tdq) if per_seq else {}
            sv.spec_verify_ex(t, d, tok, float(w.T[0]), float(w.Td[0]), args.seed, out_t,
                              out_n, seq_index_base=seq_base, flags=sv.SPEC_FLAG_EARLY_EXIT, **kw)
        for _ in range(max(3, args.warmup)):
            estep()
        torch.cuda.synchronize()
        Kx = min(K, 1000)
        es0, es1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        es0.record(stream)
        for _ in range(Kx):
            estep()
        es1.record(stream)
        torch.cuda.synchronize()
        ems_x = es0.elapsed_time(es1) / Kx
        if ws_ > 1:
            mt = torch.tensor([ems_x], device=dev, dtype=torch.float64)
            torch.distributed.all_reduce(mt, op=torch.distributed.ReduceOp.MAX)
            ems_x = float(mt.item())
        streamed, raced = early_exit_rows_read(out_n.cpu().numpy(), w.gamma)
        es_ = 2 if w.dtype == "bf16" else 4
        early = {"value": ws_ * w.rows / (ems_x / 1e3), "unit": UNIT, "ms_per_step": ems_x,
                 "steps": Kx, "rows_streamed_per_call": streamed, "rows_raced_per_call": raced,
                 "logit_bytes_read_per_call": (streamed + raced) * w.V * es_,
                 "GBps_of_bytes_read": (streamed + raced) * w.V * es_ / (ems_x / 1e3) / 1e9,
                 "note": "same outputs as the full read; reads only rows up to each "
                         "sequence's first rejection (counted from this call's outputs)"}
        status = sv.spec_verify_check()
        if status != sv.SPEC_OK:
            raise RuntimeError(f"device status after early exit: {sv.spec_verify_strerror(status)}")

    # the same call also producing the per-position entropies and KL divergences
    stats = None
    if not greedy:
        stats_out = {"Hp": torch.empty((w.B, w.gamma + 1), dtype=torch.float32, device=dev),
                     "Hq": torch.empty((w.B, w.gamma), dtype=torch.float32, device=dev),
                     "KL": torch.empty((w.B, w.gamma), dtype=torch.float32, device=dev)}

        def sstep():
            kw = dict(T_per_seq=Tq, Td_per_seq=Tdq) if per_seq else {}
            sv.spec_verify_ex(t, d, tok, float(w.T[0]), float(w.Td[0]), args.seed, out_t,
                              out_n, seq_index_base=seq_base, position_stats=stats_out, **kw)
        for _ in range(3):
            sstep()
        torch.cuda.synchronize()
        Ks = min(K, 300)
        ss0, ss1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ss0.record(stream)
        for _ in range(Ks):
            sstep()
        ss1.record(stream)
        torch.cuda.synchronize()
        sms = ss0.elapsed_time(ss1) / Ks
        stats = {"value": ws_ * w.rows / (sms / 1e3), "unit": UNIT, "ms_per_step": sms,
                 "steps": Ks, "GBps_one_read": alg_bytes / (sms / 1e3) / 1e9,
                 "note": "same call with H(p_i), H(q_i), KL(p_i||q_i) for every position"}

    # End to end through the C ABI with HOST buffers (spec_verify_host): logits, draft tokens
    # and temperatures in pinned host memory, outputs written to pinned host memory; the
    # kernels read over the host link only the rows they need (early exit).  Beside it, for
    # context, the copy path: copy every input to the device, full-read verify, copy back.
    e2e = e2e_copy = None
    if not args.no_e2e:
        h_t = to_torch(w.target, w.dtype).pin_memory()
        h_d = to_torch(w.draft, w.dtype).pin_memory()
        h_tok = torch.from_numpy(w.tokens).pin_memory()
        h_T = torch.from_numpy(w.T).pin_memory()
        h_Td = torch.from_numpy(w.Td).pin_memory()
        h_out_t = torch.empty((w.B, w.gamma + 1), dtype=torch.int32).pin_memory()
        h_out_n = torch.empty((w.B,), dtype=torch.int32).pin_memory()
        Ke = max(3, min(K, args.e2e_steps))

        def timed(fn, k):
            for _ in range(2):
                fn()
            torch.cuda.synchronize()
            if ws_ > 1:
                torch.distributed.barrier()
            es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            es.record(stream)
            for _ in range(k):
                fn()
            ee.record(stream)
            torch.cuda.synchronize()
            ems = es.elapsed_time(ee)
            if ws_ > 1:
                mt = torch.tensor([ems], device=dev, dtype=torch.float64)
                torch.distributed.all_reduce(mt, op=torch.distributed.ReduceOp.MAX)
                ems = float(mt.item())
            return ems

        def copy_step():
            t.copy_(h_t, non_blocking=True)
            if not greedy:
                d.copy_(h_d, non_blocking=True)
            tok.copy_(h_tok, non_blocking=True)
            step()
            h_out_t.copy_(out_t, non_blocking=True)
            h_out_n.copy_(out_n, non_blocking=True)

        ems = timed(copy_step, Ke)
        h2d = h_t.numel() * h_t.element_size() + h_tok.numel() * 4
        if not greedy:
            h2d += h_d.numel() * h_d.element_size()
        e2e_copy = {"value": ws_ * w.rows * Ke / (ems / 1e3), "unit": UNIT,
                    "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(h_out_t.numel() * 4 + h_out_n.numel() * 4),
                    "steps": Ke, "path": "copy inputs to the device, full-read verify, copy back"}
        if greedy:
            e2e = e2e_copy
        else:
            def host_step():
                kw = dict(T_per_seq=h_T, Td_per_seq=h_Td) if per_seq else {}
                sv.spec_verify_host(h_t, h_d, h_tok, float(w.T[0]), float(w.Td[0]), args.seed,
                                    h_out_t, h_out_n, seq_index_base=seq_base, **kw)

            Kh = max(3, min(K, 4 * args.e2e_steps))
            ems = timed(host_step, Kh)
            streamed, raced = early_exit_rows_read(h_out_n.numpy(), w.gamma)
            es_ = 2 if w.dtype == "bf16" else 4
            # the raced rows are read from the device copy the kernel keeps of the rows it
            # streams, so only the streamed rows (and the small inputs) cross the link
            e2e = {"value": ws_ * w.rows * Kh / (ems / 1e3), "unit": UNIT,
                   "h2d_bytes_per_step": int(streamed * w.V * es_ + h_tok.numel() * 4),
                   "d2h_bytes_per_step": int(h_out_t.numel() * 4 + h_out_n.numel() * 4),
                   "steps": Kh,
                   "path": "spec_verify_host: pinned host buffers read and written in place over "
                           "the host link (no staging copy); early exit streams the rows up to each "
                           "sequence's first rejection, keeping a device copy of them for the race "
                           "(h2d bytes counted from the outputs)"}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rate, nseq, secs = cpu_oracle_rate(w, args.seed, args.cpu_seconds, max_seqs=w.B)
        cpu = {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{nseq} sequence verifications of the same workload's {w.B} "
                         f"({nseq * (w.gamma + 1)} rows, {secs:.1f} s, single-threaded C, fp64)"}

    per_config = None
    if not args.no_per_config:
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        per_config = {}
        for c in range(5):
            per_config[f"cfg{c}"] = measure_config(
                sv, c, dev, stream, args.seed, seq_base, l2, peaks["hbm_gbs"],
                args.cpu_seconds_per_config if rank == 0 and not args.no_cpu_baseline else 0.0)

    if ws_ > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws_, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded numpy generator; no dataset)",
        "config": {"workload": workloads.CONFIG_NAMES[cfg], "B": w.B, "gamma": w.gamma,
                   "V": w.V, "logits": w.dtype, "mode": args.mode,
                   "rows_per_call": w.rows, "bytes_per_call": alg_bytes,
                   "l2": "inputs larger than L2 (no flush)" if alg_bytes > 2 * 126e6
                   else "inputs smaller than L2 (warm-L2 number)",
                   "parallelism": f"replicas x{ws_} (batch per GPU fixed)"},
        "achieved_GBps_step": alg_bytes / (ms_step / 1e3) / 1e9,
        "kernel_ms": {n: v for n, v in zip(
            ["row_argmax", "scan_greedy"] if greedy else ["row_stats", "scan_race"], kern_ms)},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "kernel": "row_argmax" if greedy else "row_stats",
                     "peak_source": f"{peaks['source']} HBM copy bandwidth (MEASURED_PEAKS.json)"},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "e2e_copy": e2e_copy,
        "early_exit": early,
        "with_position_stats": stats,
        "sustained": sustained,
        "per_config": per_config,
        "gpu_launches": nkern * K,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


# -------------------------------------------------------------------------------------------
# reference arm: the CPU oracle
# -------------------------------------------------------------------------------------------

def run_reference(args):
    import workloads
    ws_, rank, local = dist_env()
    if rank != 0:
        return
    import oracle
    cfg = args.config
    w = workloads.config(cfg, greedy=(args.mode == "greedy"))
    orc = oracle.get()
    # one step = the oracle on a bounded sample of the workload's sequences
    n_seq = max(1, min(w.B, args.ref_seqs))

    def step(k):
        lo = (k * n_seq) % w.B
        sl = slice(lo, min(w.B, lo + n_seq))
        if args.mode == "greedy":
            orc.verify_greedy(w.target[sl], w.tokens[sl])
        else:
            orc.verify(w.target[sl], w.draft[sl], w.tokens[sl], w.T[sl], w.Td[sl], args.seed,
                       b_base=lo)
        return (sl.stop - sl.start) * (w.gamma + 1)

    for k in range(args.warmup):
        step(k)
    rows = 0
    t0 = time.perf_counter()
    for k in range(args.steps):
        rows += step(k)
    secs = time.perf_counter() - t0
    value = rows / secs
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws_, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "impl": "reference",
        "data": "synthetic (seeded numpy generator; no dataset)",
        "config": {"workload": workloads.CONFIG_NAMES[cfg], "B": w.B, "gamma": w.gamma,
                   "V": w.V, "logits": w.dtype, "mode": args.mode, "rows_per_call": w.rows,
                   "parallelism": "single host core"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{n_seq} sequences of {w.B} per step, single-threaded C"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_lmhead(sv, dev, B, gamma, V, d, steps=10):
    """Time the verify from hidden states (spec_verify_lmhead) and the unfused pipeline on
    seeded random bf16 hidden states and heads."""
    import torch
    g = torch.Generator(device=dev).manual_seed(0)
    ht = torch.randn((B, gamma + 1, d), generator=g, device=dev).to(torch.bfloat16)
    hd = (ht[:, :gamma].float() + 0.3 * torch.randn((B, gamma, d), generator=g, device=dev)).to(torch.bfloat16)
    wt = (torch.randn((V, d), generator=g, device=dev) * (6.0 / d ** 0.5)).to(torch.bfloat16)
    wd = (wt.float() + torch.randn((V, d), generator=g, device=dev) * (0.3 / d ** 0.5)).to(torch.bfloat16)
    tok = torch.randint(0, V, (B, gamma), generator=g, device=dev, dtype=torch.int32)
    out_t = torch.empty((B, gamma + 1), dtype=torch.int32, device=dev)
    out_n = torch.empty((B,), dtype=torch.int32, device=dev)

    def fused():
        sv.spec_verify_lmhead(ht, wt, hd, wd, tok, 1.0, 0.2, 0, out_t, out_n)

    def unfused():
        lt = torch.matmul(ht.reshape(-1, d), wt.t()).reshape(B, gamma + 1, V)
        ld = torch.matmul(hd.reshape(-1, d), wd.t()).reshape(B, gamma, V)
        sv.spec_verify_ex(lt, ld, tok, 1.0, 0.2, 0, out_t, out_n)

    def timeit(fn):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record()
        for _ in range(steps):
            fn()
        s1.record()
        torch.cuda.synchronize()
        return s0.elapsed_time(s1) / steps

    fms = timeit(fused)
    status = sv.spec_verify_check()
    ums = timeit(unfused)
    rows = B * (gamma + 1)
    flops = 2.0 * B * (2 * gamma + 1) * V * d
    return {"fused_ms": fms, "unfused_ms": ums, "rows_per_s": rows / (fms / 1e3),
            "unfused_rows_per_s": rows / (ums / 1e3), "tflops": flops / (fms / 1e3) / 1e12,
            "status": status}


def run_table(args):
    """Every named workload -- the default sampling call, the early-exit call, the call with
    per-position statistics, and the greedy mode -- then the token trees and the verify from
    hidden states, as a table on stderr (calls issued from Python, CUDA events).  Workloads
    smaller than twice L2 are timed twice: on one resident copy (warm L2) and rotating over
    enough copies to exceed twice L2 (cold)."""
    import torch
    import workloads
    import speculative_decoding_verification_31_gb300 as sv
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sv.load_library()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    rows_out = []
    for cfg in range(5):
        for greedy in ([False, True] if cfg in (1, 3, 4) else [False]):
            w = workloads.config(cfg, greedy=greedy)
            nbytes = w.bytes_greedy() if greedy else w.bytes_sampling()
            copies = 1 if nbytes > 2 * l2 else min(64, -(-2 * l2 // nbytes) + 1)
            bufs = [(to_torch(w.target, w.dtype).to(dev),
                     to_torch(w.draft, w.dtype).to(dev)) for _ in range(copies)]
            tok = torch.from_numpy(w.tokens).to(dev)
            Tq, Tdq = torch.from_numpy(w.T).to(dev), torch.from_numpy(w.Td).to(dev)
            out_t = torch.empty((w.B, w.gamma + 1), dtype=torch.int32, device=dev)
            out_n = torch.empty((w.B,), dtype=torch.int32, device=dev)
            kw = dict(T_per_seq=Tq, Td_per_seq=Tdq) if cfg == 3 else {}
            stats_out = {"Hp": torch.empty((w.B, w.gamma + 1), dtype=torch.float32, device=dev),
                         "Hq": torch.empty((w.B, w.gamma), dtype=torch.float32, device=dev),
                         "KL": torch.empty((w.B, w.gamma), dtype=torch.float32, device=dev)}
            modes = [("greedy", None)] if greedy else [("two-kernel", 0),
                                                        ("early-exit", sv.SPEC_FLAG_EARLY_EXIT),
                                                        ("with H, KL", "stats")]
            for label, dbg in modes:
                for warm in ([False, True] if copies > 1 else [False]):
                    def call(k):
                        t, d = bufs[0 if warm else k % copies]
                        if greedy:
                            sv.spec_verify_greedy_ex(t, tok, out_t, out_n)
                        elif dbg == "stats":
                            sv.spec_verify_ex(t, d, tok, float(w.T[0]), float(w.Td[0]), 0, out_t,
                                              out_n, position_stats=stats_out, **kw)
                        else:
                            sv.spec_verify_ex(t, d, tok, float(w.T[0]), float(w.Td[0]), 0, out_t,
                                              out_n, flags=dbg, **kw)
                    for k in range(5):
                        call(k)
                    torch.cuda.synchronize()
                    n = max(20, min(2000, int(2e9 / max(nbytes, 1))))
                    s0 = torch.cuda.Event(enable_timing=True)
                    s1 = torch.cuda.Event(enable_timing=True)
                    s0.record()
                    for k in range(n):
                        call(k)
                    s1.record()
                    torch.cuda.synchronize()
                    us = s0.elapsed_time(s1) / n * 1e3
                    st = sv.spec_verify_check()
                    rows_out.append((cfg, label, "warm" if warm else ("cold" if copies > 1 else "> L2"),
                                     us, w.rows / us * 1e6, nbytes / us / 1e3, st))
    # static token trees (SubSpec's shape: depth 48, six children per main-path node)
    for B in (1, 8):
        tw = workloads.tree(workloads.deep_narrow_tree(48, 6), B=B, V=152064, dtype="bf16",
                            seed=1005, scale=5.0, sigma=workloads.DEEP_CHAIN_SIGMA, T=0.6, Td=0.2,
                            name=f"tree depth 48 x 6, B={B}")
        nbytes = tw.bytes()
        copies = 1 if nbytes > 2 * l2 else min(64, -(-2 * l2 // nbytes) + 1)
        bufs = [(to_torch(tw.target, tw.dtype).to(dev), to_torch(tw.draft, tw.dtype).to(dev))
                for _ in range(copies)]
        ttok = torch.from_numpy(tw.tokens).to(dev)
        tree = sv.Tree(tw.parent)
        t_out = torch.empty((B, tree.D + 1), dtype=torch.int32, device=dev)
        t_nodes = torch.empty((B, tree.D), dtype=torch.int32, device=dev)
        t_n = torch.empty((B,), dtype=torch.int32, device=dev)
        for warm in ([False, True] if copies > 1 else [False]):
            def tcall(k):
                t, d = bufs[0 if warm else k % copies]
                return sv.spec_verify_tree(t, d, ttok, tree, 0.6, 0.2, 0, out_tokens=t_out,
                                           out_nodes=t_nodes, out_n_accepted=t_n)
            for k in range(5):
                tcall(k)
            torch.cuda.synchronize()
            n = 200
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record()
            for k in range(n):
                _, _, nacc = tcall(k)
            s1.record()
            torch.cuda.synchronize()
            us = s0.elapsed_time(s1) / n * 1e3
            emitted = float(nacc.float().mean().item()) + 1.0
            rows_out.append((tw.name, f"tree (emits {emitted:.1f} tokens/seq)",
                             "warm" if warm else ("cold" if copies > 1 else "> L2"), us,
                             tw.rows() / us * 1e6, nbytes / us / 1e3, sv.spec_verify_check()))
    # the verify from hidden states (fused LM head, tensor cores) at the throughput shape,
    # against the unfused pipeline: the library GEMM (torch.matmul: cuBLAS) writing bf16
    # logits, then the logits verify reading them
    lm = run_lmhead(sv, dev, B=256, gamma=12, V=152064, d=4096)
    print("| verify from hidden states, B=256 gamma=12 V=152064 d=4096 | fused LM head "
          f"(tensor cores) | - | {lm['fused_ms'] * 1e3:.0f} | {lm['rows_per_s']:.3e} | "
          f"GEMM {lm['tflops']:.0f} TFLOP/s | {lm['status']} |", file=sys.stderr)
    print("| same | cuBLAS bf16 logits + logits verify | - | "
          f"{lm['unfused_ms'] * 1e3:.0f} | {lm['unfused_rows_per_s']:.3e} | - | 0 |", file=sys.stderr)
    print("| workload | path | L2 | us/call | rows/s | GB/s (one read of the logits) | status |",
          file=sys.stderr)
    print("|---|---|---|---|---|---|---|", file=sys.stderr)
    for cfg, label, l2s, us, rps, gbs, st in rows_out:
        print(f"| {cfg} | {label} | {l2s} | {us:.1f} | {rps:.3e} | {gbs:.0f} | {st} |",
              file=sys.stderr)


def launch_ranks(n: int, argv) -> int:
    """Run this script as n ranks, one process per GPU (LOCAL_RANK = RANK = 0..n-1, WORLD_SIZE =
    n, rendezvous on 127.0.0.1), as torchrun would; rank 0 prints the JSON line.  If a rank
    fails the others are stopped.  Returns the first non-zero exit status, else 0."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    procs = []
    for r in range(n):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(n),
                   LOCAL_WORLD_SIZE=str(n), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, os.path.abspath(__file__), *argv], env=env))
    rc = 0
    while procs:
        for p in list(procs):
            code = p.poll()
            if code is None:
                continue
            procs.remove(p)
            if code != 0 and rc == 0:
                rc = code
                for q in procs:  # the ranks this launcher started, by their own handles
                    q.terminate()
        time.sleep(0.05)
    return rc


def run_dry(args):
    """CPU only: every rank joins a gloo group, 'times' K steps that sleep (rank + 1) * 10 ms
    each, and rank 0 prints the line with the maximum over ranks, as the GPU run does."""
    import torch
    import torch.distributed as dist
    import workloads
    ws_, rank, _ = dist_env()
    if ws_ > 1:
        dist.init_process_group("gloo")
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        time.sleep((rank + 1) * 0.01)
    ms = (time.perf_counter() - t0) * 1e3
    ranks = [rank]
    if ws_ > 1:
        mt = torch.tensor([ms], dtype=torch.float64)
        dist.all_reduce(mt, op=dist.ReduceOp.MAX)
        ms = float(mt.item())
        got = [torch.zeros(1, dtype=torch.int64) for _ in range(ws_)]
        dist.all_gather(got, torch.tensor([rank], dtype=torch.int64))
        ranks = sorted(int(g.item()) for g in got)
        dist.destroy_process_group()
    if rank != 0:
        return
    B, gamma, V, _ = workloads.CONFIG_SHAPES[args.config]
    rows = B * (gamma + 1)
    print(json.dumps({"metric": METRIC, "value": ws_ * rows * args.steps / (ms / 1e3), "unit": UNIT,
                      "n_gpus": ws_, "steps": args.steps, "warmup": args.warmup,
                      "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
                      "dry_run": True, "ranks": ranks}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=4, choices=range(5))
    ap.add_argument("--mode", choices=["sampling", "greedy"], default="sampling")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--lmhead", action="store_true",
                    help="time the verify from hidden states (fused LM head) only, to stderr")
    ap.add_argument("--lm-steps", type=int, default=10)
    ap.add_argument("--all", action="store_true",
                    help="print a per-workload table (every path, trees, LM head) to stderr")
    ap.add_argument("--no-sustained", action="store_true")
    ap.add_argument("--sustained-seconds", type=float, default=1.2)
    ap.add_argument("--no-per-config", action="store_true")
    ap.add_argument("--cpu-seconds-per-config", type=float, default=2.0)
    ap.add_argument("--dry-run", action="store_true",
                    help="CPU only: exercise the rank launcher and the max-over-ranks timing on\n"
                         "gloo without touching a GPU (prints a line marked dry_run)")
    ap.add_argument("--ref-seqs", type=int, default=1,
                    help="sequences per reference step (one throughput-workload sequence is\n"
                         "about 0.04 s of oracle work)")
    args = ap.parse_args()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(launch_ranks(args.gpus, sys.argv[1:]))
    if args.dry_run:
        run_dry(args)
        return
    if args.lmhead:
        import torch
        import speculative_decoding_verification_31_gb300 as sv
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        sv.load_library()
        print(json.dumps(run_lmhead(sv, dev, B=256, gamma=12, V=152064, d=4096,
                                    steps=args.lm_steps)), file=sys.stderr)
        return
    if args.all:
        run_table(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
