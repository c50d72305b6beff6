"""Benchmark: KDA chunked prefill, 8 sequences x 2048 tokens, H=16, D=128.

One step = one kda_chunk_prefill_fwd call over the whole batch (every step of
the method runs inside that call's kernels).  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--kernel auto|tc|split|streamed|ref|helpers|pipe] [--workload 1]
                  [--no-cpu-baseline] [--stamps] [--range-call]

value       tokens/s of the whole job (all ranks), inputs resident in HBM;
            device time from CUDA events over exactly K steps, max over ranks.
e2e         the same metric through the C ABI with host buffers: pinned
            host -> device copies of every input, the call, device -> host
            copies of out and final_state, all inside the timed region.
roofline    the prefill call against the HBM roofline: algorithmic bytes per
            call / mean call time (CUDA events on the launch stream).  On the
            default workload AUTO runs one launch of the warp-specialised
            kernel; on the split path (few sequences x heads) it is the
            k-side kernel followed by the chain kernel, or (streamed, AUTO's
            choice where the chains leave half of the SMs free) the chain
            kernel running beside the k-side kernel.
launch_us   mean, median, min and max of the K per-call event times.
graph       the same call captured in a CUDA graph (8 calls per graph over the
            rotating input sets), replayed 60 times: microseconds per call.
cpu_baseline  the fp64 CPU oracle (test infrastructure) on a bounded sample
            of the same workload, on this host's cores (rank 0, N=1 only);
            cpu_baseline_1thread the same oracle on one thread.
--impl reference  times that oracle as the reference arm.
--stamps    the per-chunk phase breakdown of the warp-specialised kernel: builds
            the -DKDA_PHASE_STAMPS variant of the library and prints medians of
            the clock64 stamps of CTA 0 (not a bench line); with --kernel split
            or streamed, the timeline of the split path's CTAs instead.
--range-call  one call between cudaProfilerStart/Stop, for an ncu range replay
            of a call whose kernels overlap (not a bench line).

L2: the inputs (352 MB per step) exceed the 129 MB L2, and four copies of
them are rotated so that no step finds the previous step's data in L2.
Multi-GPU: every rank runs its own full batch (replicas; the prefill has no
exchange step), "scaling": "weak".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import kda_workloads as W  # noqa: E402

METRIC = "KDA prefill us/layer & tokens/s (8x2048, H=16, D=128); % of roofline"
UNIT = "tokens/s"
D = W.HEAD_DIM


def algorithmic_bytes(w: W.Workload) -> int:
    """Bytes the prefill must move at least once: q, k, v, g, out (bf16),
    beta (bf16), A_log and dt_bias (fp32), cu_seqlens, the state in and out."""
    T = sum(w.lengths)
    H, N = w.heads, w.num_seqs
    s = 4 if w.state_dtype == "f32" else 2
    return T * H * (5 * 2 * D + 2) + 2 * N * H * D * D * s + H * (D + 1) * 4 + (N + 1) * 4


def algorithmic_flops(w: W.Workload, C: int = 64) -> int:
    """Chunked-form tensor FLOPs with full C x C tiles: 2 D (5 C + 3 D) per token-head."""
    return sum(w.lengths) * w.heads * 2 * D * (5 * C + 3 * D)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# host-only translation unit (argument checks, planning, the C entry points): no device code
HOST_ONLY_SOURCES = ("kda_api.cu",)
# the sources a kernel is built from, where that is a strict subset (headers included): its
# committed traffic figure stays valid while these are unchanged.  Other kernels hash every
# device source.
_SPLIT_SOURCES = ("kda_kside_kernel.cu", "kda_chain_kernel.cu", "kda_chain_vs_kernel.cu",
                  "kda_chain_tc_kernel.cu", "kda_stream.cuh", "kda_internal.cuh", "kda_sm100.cuh",
                  "kda_tc_common.cuh")
KERNEL_SOURCES = {
    "kda_pipe_kernel": ("kda_pipe_kernel.cu", "kda_internal.cuh", "kda_sm100.cuh",
                        "kda_tc_common.cuh"),
    "kda_split_path": _SPLIT_SOURCES,
    "kda_split_streamed_path": _SPLIT_SOURCES,
}


def kernel_source_hash(kernel_name: str | None = None) -> str:
    """Hash of a kernel's CUDA sources (KERNEL_SOURCES, else every file but the host-only
    ones) with comments, phase stamps and blank space removed: it changes when kernel or
    launch code does, not when a comment, a stamp or a host-side entry point does."""
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "kda_gated_delta_chunk_gb300", "csrc")
    names = KERNEL_SOURCES.get(kernel_name) if kernel_name else None
    for name in sorted(os.listdir(csrc)):
        if not name.endswith((".cu", ".cuh")) or name in HOST_ONLY_SOURCES:
            continue
        if names is not None and name not in names:
            continue
        text = open(os.path.join(csrc, name), encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        text = re.sub(r"[PT]STAMP\([^;]*\);", " ", text)   # stamps: empty outside the stamps build
        text = " ".join(text.split())
        h.update(name.encode() + b"\0" + text.encode())
    return h.hexdigest()[:16]


def load_traffic(kernel_name: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current sources of that kernel and this workload (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    ent = d.get(kernel_name)
    if (not ent or ent.get("source_hash") != kernel_source_hash(kernel_name)
            or ent.get("workload") != workload):
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str):
        self.uuid = uuid
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.rows and time.time() - t0 < 5.0:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9 and self.uuid in parts[0]:
                self.rows.append((time.time(), parts))

    def stop(self, t_begin: float, t_end: float):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        inside = [p for (t, p) in self.rows if t_begin <= t <= t_end] or [p for (_, p) in self.rows]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4)
                          if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(inside[0][2]), "reasons": reasons,
                "samples": len(inside), "power_w_max": max((num(p[3]) or 0.0) for p in inside)}


def dist_setup(gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest x over the ranks (the job's time is the slowest rank's)."""
    if world == 1:
        return x
    on_gpu = torch.distributed.get_backend() == "nccl"
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if on_gpu else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def oracle_sample_run(inp, heads, num_threads=0):
    """The fp64 oracle on all sequences of the workload for the given heads (num_threads 0:
    all the cores the oracle finds)."""
    import oracle
    N = inp["cu_seqlens"].numel() - 1
    sub = W.select(inp, range(N), heads)
    f = lambda t: t.float().double().numpy()
    args = (f(sub["q"]), f(sub["k"]), f(sub["v"]), f(sub["g"]), f(sub["beta"]),
            f(sub["A_log"]), f(sub["dt_bias"]), sub["lower_bound"], sub["scale"],
            f(sub["initial_state"]), sub["cu_seqlens"].numpy())
    t0 = time.perf_counter()
    oracle.kda_oracle_fwd(*args, num_threads=num_threads)
    return time.perf_counter() - t0


def cpu_baseline(inp, w: W.Workload, budget_s: float = 10.0):
    """Time the oracle as it stands on a bounded sample of the workload: whole passes over
    all sequences and heads, repeated until about budget_s of CPU work (at least one); a
    workload too large for that runs on its first h heads instead."""
    import oracle
    oracle.build()
    T = sum(w.lengths)
    t1 = oracle_sample_run(inp, [0])
    h = int(max(1, min(w.heads, budget_s // max(t1, 1e-3))))
    heads = list(range(h))
    t = oracle_sample_run(inp, heads) if h > 1 else t1
    reps = int(max(1, min(100, budget_s // max(t, 1e-3))))
    for _ in range(reps - 1):
        t += oracle_sample_run(inp, heads)
    tok_per_s = T * h * reps / t / w.heads   # token-heads/s expressed as tokens of the H-head layer
    return {"value": tok_per_s, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"{w.name}: {reps} pass(es) over all {w.num_seqs} sequences x {h} of "
                      f"{w.heads} heads ({T * h * reps} token-heads, fp64, {t:.2f} s); "
                      f"tokens/s = token-heads/s / {w.heads}",
            "seconds": t}


def cpu_baseline_one_thread(inp, w: W.Workload, budget_s: float = 4.0):
    """The oracle on one host thread: whole passes over all sequences for as many heads as
    fit in about budget_s (at least one head, one pass)."""
    import oracle
    oracle.build()
    T = sum(w.lengths)
    t = oracle_sample_run(inp, [0], num_threads=1)
    h = 1
    while h < w.heads and t * (h + 1) / h <= budget_s:
        t += oracle_sample_run(inp, [h], num_threads=1)
        h += 1
    return {"value": T * h / t / w.heads, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{w.name}: all {w.num_seqs} sequences x {h} of {w.heads} heads on one "
                      f"thread ({T * h} token-heads, fp64, {t:.2f} s); tokens/s = token-heads/s "
                      f"/ {w.heads}", "seconds": t}


def graph_timing(step, stream, calls: int = 8, replays: int = 60):
    """The same call captured in a CUDA graph (`calls` calls over the rotating input sets per
    graph) and replayed `replays` times after 3 warm-up replays: microseconds per call."""
    g = torch.cuda.CUDAGraph()
    stream.synchronize()
    with torch.cuda.graph(g, stream=stream):
        for i in range(calls):
            step(i)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(replays):
            g.replay()
    e1.record(stream)
    e1.synchronize()
    return {"us_per_layer": 1e3 * e0.elapsed_time(e1) / (replays * calls),
            "replays": replays, "calls_per_replay": calls}


def run_reference(args, w):
    """Reference arm: the oracle as it stands, a bounded sample per step."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    inp = W.make_inputs(w)
    T = sum(w.lengths)
    for _ in range(args.warmup):
        oracle_sample_run(inp, [0])
    ts = [oracle_sample_run(inp, [0]) for _ in range(args.steps)]
    total = sum(ts)
    val = T * args.steps / total / w.heads
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "tokens": T, "seqs": w.num_seqs, "heads": w.heads,
                       "head_dim": D, "state": w.state_dtype,
                       "step": "oracle on all sequences x 1 head"},
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": oracle.max_threads(),
                             "kind": "oracle",
                             "sample": f"{w.name}: all {w.num_seqs} sequences x 1 of {w.heads} "
                                       f"heads per step; tokens/s = token-heads/s / {w.heads}"},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# phase stamps of the pipelined kernel: 32 slots per chunk (see kda_pipe_kernel.cu)
# chain stamp slots (CTA 0, thread 0) and the k-side ones (thread 128); 32 slots per chunk
CHAIN_SLOTS = {0: "stage part A full", 2: "v ready", 3: "G1a issued", 12: "S decayed",
               4: "G1a done", 5: "X_b stored", 26: "T full, T operands stored",
               28: "G1b done (thread 0)", 27: "QK operand stored", 6: "chain group past G1b",
               7: "U_b stored", 8: "G2 done", 10: "O stored"}
CHAIN_ORDER = [0, 2, 3, 12, 4, 5, 26, 28, 27, 6, 7, 8, 10]
KSIDE_SLOTS = {19: "loop top", 25: "input wait (MMA thread)", 16: "inputs landed",
               17: "gate and norms", 18: "factors, [Kg; Qg] free", 20: "tile rows done",
               21: "tiles fenced", 22: "A|QK MMA done", 1: "Ke and T parts free",
               24: "N, Ke stored", 29: "inverse, stage handed over"}
KSIDE_ORDER = [19, 25, 16, 17, 18, 20, 21, 22, 1, 24, 29]


def run_split_timeline(args, kda, w, d, dev):
    """Timeline of one split-path call (--kernel split or streamed) in the stamps build:
    when each k-side CTA and each warp-level chain CTA (P = 4, 8) started and ended, when
    each chain CTA's first record was ready (streamed), which k-side CTAs left their SM to
    the chains; microseconds from the first k-side CTA's start, (min, median, max)."""
    kernel = kda.KERNEL_SPLIT_STREAMED if args.kernel == "streamed" else kda.KERNEL_SPLIT
    T, H, N = sum(w.lengths), w.heads, w.num_seqs
    need = 1024 + ((T + 63) // 64 + N) * H * (66560 + 4)
    ws_bytes = need + 65536
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    off = (ws_bytes - 32768) & ~255
    for _ in range(max(3, args.warmup) + 1):
        ws[off:].zero_()
        kda.chunk_prefill_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"],
                              d["dt_bias"], d["lower_bound"], d["scale"], d["initial_state"],
                              d["cu_seqlens"], workspace=ws, kernel=kernel, vsplit=args.vsplit)
    torch.cuda.synchronize()
    st = kda.last_device_status(ws)
    if st != kda.OK:
        raise kda.KDAError(st, "device status")
    _, P, _ = kda.plan(T, N, H, ws_bytes, args.vsplit, kernel)
    words = ws[off:off + 32768].cpu().view(torch.int64).tolist()
    nk = min(512, 2 * torch.cuda.get_device_properties(dev).multi_processor_count)
    ks = [words[1024 + 4 * b:1024 + 4 * b + 4] for b in range(nk)]
    ks = [k for k in ks if k[0] > 0]
    ch = [words[4 * b:4 * b + 4] for b in range(min(256, N * H * P))]
    t0 = min(k[0] for k in ks)

    def q3(vals):
        vals = sorted((v - t0) / 1e3 for v in vals)
        return [round(vals[0], 1), round(vals[len(vals) // 2], 1), round(vals[-1], 1)] if vals else None
    res = {"workload": w.name, "path": "streamed" if kernel == kda.KERNEL_SPLIT_STREAMED else "split",
           "vsplit": P, "unit": "us from the first k-side CTA's start: min, median, max",
           "kside_ctas": len(ks), "kside_ctas_that_left_their_sm": sum(k[3] >= 65536 for k in ks),
           "kside_start": q3([k[0] for k in ks]), "kside_end": q3([k[1] for k in ks]),
           "kside_end_working_ctas": q3([k[1] for k in ks if k[3] < 65536])}
    if P >= 4:
        res.update({"chain_ctas": len(ch), "chain_start": q3([c[0] for c in ch]),
                    "chain_end": q3([c[2] for c in ch]),
                    "chain_sms_distinct": len({c[3] for c in ch})})
        if kernel == kda.KERNEL_SPLIT_STREAMED:
            res["chain_first_record_ready"] = q3([c[1] for c in ch])
    print(json.dumps(res, indent=1), flush=True)


def run_range_call(args):
    """One call of the workload between cudaProfilerStart and cudaProfilerStop (after
    max(3, --warmup) untimed calls), for `ncu --replay-mode app-range`: the DRAM traffic of a
    call whose kernels overlap (the streamed split path), which kernel replay serialises."""
    from kda_gated_delta_chunk_gb300 import build as kbuild
    import kda_gated_delta_chunk_gb300 as kda
    kbuild.build()
    kernel = {"auto": kda.KERNEL_AUTO, "tc": kda.KERNEL_TC, "ref": kda.KERNEL_REF,
              "split": kda.KERNEL_SPLIT, "streamed": kda.KERNEL_SPLIT_STREAMED,
              "helpers": kda.KERNEL_TC_HELPERS, "pipe": kda.KERNEL_PIPE}[args.kernel]
    w = W.workload(args.workload, args.n) if args.workload == 3 else W.workload(args.workload)
    dev = torch.device("cuda", torch.cuda.current_device())
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in W.make_inputs(w).items()}
    T, H, N = sum(w.lengths), w.heads, w.num_seqs
    ws = torch.zeros(max(kda.workspace_size(T, H, N), 1024 + ((T + 63) // 64 + N) * H * (66560 + 4)),
                     dtype=torch.uint8, device=dev)
    out, fin = torch.empty_like(d["q"]), torch.empty_like(d["initial_state"])

    def call():
        kda.chunk_prefill_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"],
                              d["dt_bias"], d["lower_bound"], d["scale"], d["initial_state"],
                              d["cu_seqlens"], out=out, final_state=fin, workspace=ws,
                              kernel=kernel, vsplit=args.vsplit)
    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    torch.cuda.profiler.start()
    call()
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    st = kda.last_device_status(ws)
    if st != kda.OK:
        raise kda.KDAError(st, "device status")
    path, P, launches = kda.plan(T, N, H, ws.numel(), args.vsplit, kernel)
    print(json.dumps({"workload": w.name, "path": path, "vsplit": P, "launches": launches}),
          flush=True)


def run_stamps(args):
    """Phase breakdown of KDA_KERNEL_PIPE: build the phase-stamp variant of the library
    (-DKDA_PHASE_STAMPS), run the workload a few times, read the clock64 stamps CTA 0 (the
    longest sequence, head 0) wrote per chunk, print medians over its inner chunks.  The
    k-side's stamps come from a thread of warp 19, which the inverse does not use: stamps
    taken by a warp inside a phase lengthen that phase."""
    from kda_gated_delta_chunk_gb300 import build as kbuild
    import kda_gated_delta_chunk_gb300 as kda
    path = kbuild.build(stamps=True)
    kda.use_library(path)
    w = W.workload(args.workload, args.n) if args.workload == 3 else W.workload(args.workload)
    dev = torch.device("cuda", torch.cuda.current_device())
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in W.make_inputs(w).items()}
    if args.kernel in ("split", "streamed"):
        return run_split_timeline(args, kda, w, d, dev)
    ws_bytes = 1 << 16
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    off = (ws_bytes - 16384) & ~255
    for _ in range(max(3, args.warmup) + 1):
        ws[off:].zero_()
        kda.chunk_prefill_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"],
                              d["dt_bias"], d["lower_bound"], d["scale"], d["initial_state"],
                              d["cu_seqlens"], workspace=ws, kernel=kda.KERNEL_PIPE)
    torch.cuda.synchronize()
    st = kda.last_device_status(ws)
    if st != kda.OK:
        raise kda.KDAError(st, "device status")
    stamps = ws[off:off + 16384].cpu().view(torch.int64).view(64, 32).tolist()
    nch = min(64, (max(w.lengths) + 63) // 64)
    inner = range(1, max(2, nch - 1))

    def med(a, b, prev=False):
        vals = [stamps[c][b] - (stamps[c - 1][a] if prev else stamps[c][a]) for c in inner]
        return statistics.median(vals) if vals else 0

    ks, cs = KSIDE_ORDER, CHAIN_ORDER
    res = {"workload": w.name, "chunks_of_cta0": nch, "unit": "SM cycles (clock64), median",
           "chunk_period": med(29, 29, True),
           "kside": {f"{KSIDE_SLOTS[a]} -> {KSIDE_SLOTS[b]}": med(a, b) for a, b in zip(ks, ks[1:])},
           "kside_wait_for_inputs (handover c-1 -> inputs landed c)": med(29, 16, True),
           "kside_mma_issue (tiles fenced -> MMA issued)": med(21, 31),
           "kside_next_inputs_issued (tiles fenced -> issued)": med(21, 30),
           "chain": {f"{CHAIN_SLOTS[a]} -> {CHAIN_SLOTS[b]}": med(a, b) for a, b in zip(cs, cs[1:])},
           "chain_wait_for_stage (O stored c-1 -> stage full c)": med(10, 0, True),
           "handover -> chain start": med(29, 0),
           "chain G1a done (c-1) -> kside factors, [Kg; Qg] free (c)": med(4, 18, True),
           "chain QK rows of D free (c-1) -> kside tiles fenced (c)": med(27, 21, True),
           "chain G2 done (c-1) -> kside Ke and T parts free (c)": med(8, 1, True)}
    print(json.dumps(res, indent=1), flush=True)


def run_decode(args):
    """Decode / speculative-verify step through kda_recurrent_fwd: 64 sequences x K tokens,
    H = 32, fp32 state.  The time is bound by reading and writing the state."""
    import kda_gated_delta_chunk_gb300 as kda
    from kda_gated_delta_chunk_gb300 import build as kbuild
    kbuild.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    K, N, H = args.decode, 64, 32
    w = W.custom([K] * N, H, seed=61)
    host = W.make_inputs(w)
    NB = 4
    sets = []
    for _ in range(NB):
        d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
        d["out"] = torch.empty_like(d["q"])
        d["fin"] = torch.empty_like(d["initial_state"])
        d["ws"] = torch.zeros(256, dtype=torch.uint8, device=dev)
        sets.append(d)
    stream = torch.cuda.Stream(dev)

    def step(i):
        d = sets[i % NB]
        kda.recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"],
                          d["lower_bound"], d["scale"], d["initial_state"], d["cu_seqlens"],
                          out=d["out"], final_state=d["fin"], workspace=d["ws"], stream=stream)
    for i in range(max(3, args.warmup)):
        step(i)
    stream.synchronize()
    steps = args.steps if args.steps > 0 else 200
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        step(i)
    e1.record(stream)
    e1.synchronize()
    t = e0.elapsed_time(e1) / 1e3 / steps
    T = N * K
    abytes = T * H * (5 * 2 * D + 2) + 2 * N * H * D * D * 4 + H * (D + 1) * 4 + (N + 1) * 4
    hbm, _, peak_kind = load_peaks()
    line = {"metric": "KDA decode step (recurrent form)", "value": T / t, "unit": UNIT,
            "n_gpus": 1, "steps": steps, "warmup": args.warmup, "ms_per_step": 1e3 * t,
            "higher_is_better": True, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"decode_{N}x{K}_h{H}", "seqs": N, "tokens_per_seq": K,
                       "heads": H, "head_dim": D, "state": "f32",
                       "l2": f"{abytes / 1e6:.0f} MB per step, 4 input sets rotated"},
            "roofline": {"bound": "hbm", "kernel": "kda_recurrent_kernel",
                         "achieved": abytes / t / 1e9, "peak": hbm, "unit": "GB/s",
                         "frac": abytes / t / 1e9 / hbm, "algorithmic_bytes_per_launch": abytes,
                         "peak_source": peak_kind,
                         "traffic": load_traffic("kda_recurrent_kernel", f"decode_{N}x{K}_h{H}")},
            "gpu_launches": steps}
    print(json.dumps(line), flush=True)


def run_scatter(args):
    """The benchmark workload written through a row map (a mixed step's non-speculative
    tokens into the layer output): the prefill with out_index, against the dense call and
    against the dense call followed by index_copy_ into the layer output."""
    import kda_gated_delta_chunk_gb300 as kda
    from kda_gated_delta_chunk_gb300 import build as kbuild
    kbuild.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    w = W.workload(1)
    host = W.make_inputs(w)
    T, H, N = sum(w.lengths), w.heads, w.num_seqs
    NB = 4
    gen = torch.Generator().manual_seed(71)
    rows = torch.randperm(T + 1024, generator=gen)[:T].to(torch.int32).to(dev)
    sets = []
    for _ in range(NB):
        d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
        d["out"] = torch.empty_like(d["q"])
        d["layer"] = torch.empty((T + 1024, H, D), dtype=torch.bfloat16, device=dev)
        d["fin"] = torch.empty_like(d["initial_state"])
        d["ws"] = kda.alloc_workspace(T, H, N, device=dev)
        sets.append(d)
    stream = torch.cuda.Stream(dev)

    def call(i, mode):
        d = sets[i % NB]
        a = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"],
             d["lower_bound"], d["scale"], d["initial_state"], d["cu_seqlens"])
        if mode == "scatter":
            kda.chunk_prefill_fwd(*a, out=d["layer"], final_state=d["fin"], workspace=d["ws"],
                                  stream=stream, out_index=rows)
        else:
            kda.chunk_prefill_fwd(*a, out=d["out"], final_state=d["fin"], workspace=d["ws"],
                                  stream=stream)
            if mode == "index_copy":
                with torch.cuda.stream(stream):
                    d["layer"].index_copy_(0, rows.long(), d["out"])
    steps = args.steps if args.steps > 0 else 100
    res = {}
    for mode in ("dense", "scatter", "index_copy"):
        for i in range(max(3, args.warmup)):
            call(i, mode)
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            call(i, mode)
        e1.record(stream)
        e1.synchronize()
        res[mode] = e0.elapsed_time(e1) / 1e3 / steps
    _, _, launches = kda.plan(T, N, H, sets[0]["ws"].numel(), -1, kda.KERNEL_AUTO)
    line = {"metric": "KDA prefill with a scattered output (mixed step)", "value": T / res["scatter"],
            "unit": UNIT, "n_gpus": 1, "steps": steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * res["scatter"], "higher_is_better": True, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": w.name + "_scatter", "rows": "random one-to-one map into "
                       f"{T + 1024} rows", "l2": "4 input sets rotated"},
            "us_dense": 1e6 * res["dense"], "us_scatter": 1e6 * res["scatter"],
            "us_dense_then_index_copy": 1e6 * res["index_copy"],
            "gpu_launches": steps * launches}
    print(json.dumps(line), flush=True)


def run_proj(args):
    """The low-M projections (kda_skinny_proj) at the shapes of the skinny-GEMM test in the
    projection-overlap PR report: k = 7168 -> 144, first 128 columns -> 1536, for m token
    rows.  64 distinct weight sets (157 MB, more than L2) are rotated so the weights come
    from HBM, as they would for the layers of a model; the same calls through torch's
    cuBLAS linear are timed beside it."""
    import kda_gated_delta_chunk_gb300 as kda
    from kda_gated_delta_chunk_gb300 import build as kbuild
    kbuild.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    K, NAB, R, NB = 7168, 144, 128, 1536
    NS = 64
    g = torch.Generator(device="cpu").manual_seed(81)
    w_ab = [torch.randn(NAB, K, generator=g).to(torch.bfloat16).to(dev) for _ in range(NS)]
    w_b = [torch.randn(NB, R, generator=g).to(torch.bfloat16).to(dev) for _ in range(NS)]
    ws = torch.zeros(kda.skinny_proj_workspace_size(K, NAB), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)
    hbm, _, peak_kind = load_peaks()
    rows = []
    for m in (1, 2, 8, 14):
        x = torch.randn(m, K, generator=g).to(torch.bfloat16).to(dev)
        y = torch.empty(m, NAB, dtype=torch.bfloat16, device=dev)
        z = torch.empty(m, NB, dtype=torch.bfloat16, device=dev)
        res = {}
        for mode in ("ours", "cublas"):
            def call(i):
                if mode == "ours":
                    kda.skinny_proj(x, w_ab[i % NS], w_b[i % NS], R, y=y, z=z, workspace=ws,
                                    stream=stream)
                else:
                    with torch.cuda.stream(stream):
                        yy = torch.nn.functional.linear(x, w_ab[i % NS])
                        torch.nn.functional.linear(yy[:, :R], w_b[i % NS])
            for i in range(NS):
                call(i)
            stream.synchronize()
            # one call per weight set captured in a CUDA graph (the host's per-call cost is
            # not part of the layer's time), replayed
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for i in range(NS):
                    call(i)
            with torch.cuda.stream(stream):   # replay() launches on the current stream
                for _ in range(3):
                    graph.replay()
                stream.synchronize()
                reps = 20
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(reps):
                    graph.replay()
                e1.record(stream)
            e1.synchronize()
            res[mode] = e0.elapsed_time(e1) / 1e3 / (reps * NS)
        abytes = 2 * (NAB * K + NB * R + m * K + m * NAB + m * NB)
        rows.append({"m": m, "us": 1e6 * res["ours"], "us_cublas": 1e6 * res["cublas"],
                     "algorithmic_bytes": abytes,
                     "achieved_gbs": abytes / res["ours"] / 1e9,
                     "frac": abytes / res["ours"] / 1e9 / hbm})
    r14 = rows[-1]
    line = {"metric": "KDA low-M projections (x 7168 -> 144 -> 1536), us per layer",
            "value": r14["us"], "unit": "us", "higher_is_better": False, "n_gpus": 1,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "skinny_proj_m14_k7168_n144_r128_n1536",
                       "l2": "64 weight sets rotated (157 MB)",
                       "timing": "64 calls captured in a CUDA graph, replayed 20 times"},
            "roofline": {"bound": "hbm", "kernel": "kda_skinny_proj", "achieved": r14["achieved_gbs"],
                         "peak": hbm, "unit": "GB/s", "frac": r14["frac"], "peak_source": peak_kind,
                         "algorithmic_bytes_per_launch": r14["algorithmic_bytes"],
                         "traffic": load_traffic("kda_skinny_proj",
                                                 "skinny_proj_m14_k7168_n144_r128_n1536")},
            "per_m": rows, "gpu_launches": 2}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0, help="timed steps (0: ~1.5 s worth)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--kernel", default="auto",
                    choices=["auto", "tc", "helpers", "split", "streamed", "ref", "pipe"])
    ap.add_argument("--workload", type=int, default=1)
    ap.add_argument("--n", type=int, default=None, help="sequences of the V-split workload (3)")
    ap.add_argument("--vsplit", type=int, default=-1, help="-1 automatic, or 1/2/4/8")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--profile-range", action="store_true",
                    help="run one call inside cudaProfilerStart/Stop after the warm-up, then exit")
    ap.add_argument("--proj", action="store_true",
                    help="time the low-M projections (kda_skinny_proj)")
    ap.add_argument("--scatter", action="store_true",
                    help="time the prefill writing through an output row map")
    ap.add_argument("--decode", type=int, default=0,
                    help="time a decode step (kda_recurrent_fwd) with this many tokens per sequence")
    ap.add_argument("--stamps", action="store_true",
                    help="per-chunk phase breakdown of the pipelined kernel from the phase-stamp "
                         "build (clock64 stamps of CTA 0), then exit")
    ap.add_argument("--range-call", action="store_true",
                    help="one prefill call (after --warmup calls) between cudaProfilerStart and "
                         "cudaProfilerStop, for an ncu range replay of the whole call, then exit")
    args = ap.parse_args()
    if args.stamps:
        return run_stamps(args)
    if args.range_call:
        return run_range_call(args)
    if args.decode > 0:
        return run_decode(args)
    if args.scatter:
        return run_scatter(args)
    if args.proj:
        return run_proj(args)
    w = W.workload(args.workload, args.n) if args.workload == 3 else W.workload(args.workload)
    if args.impl == "reference":
        if args.steps <= 0:
            args.steps = 5
        return run_reference(args, w)

    import kda_gated_delta_chunk_gb300 as kda
    from kda_gated_delta_chunk_gb300 import build as kbuild
    world, rank, local = dist_setup(args.gpus)
    if rank == 0:
        kbuild.build()
    barrier(world)
    kbuild.build()
    kernel = {"auto": kda.KERNEL_AUTO, "tc": kda.KERNEL_TC, "ref": kda.KERNEL_REF,
              "split": kda.KERNEL_SPLIT, "streamed": kda.KERNEL_SPLIT_STREAMED,
              "helpers": kda.KERNEL_TC_HELPERS, "pipe": kda.KERNEL_PIPE}[args.kernel]
    dev = torch.device("cuda", torch.cuda.current_device())
    rc = kda.device_check(dev.index)
    if rc != kda.OK:
        raise kda.KDAError(rc, "device check")

    host = W.make_inputs(w)
    T, H, N = sum(w.lengths), w.heads, w.num_seqs
    stream = torch.cuda.Stream(dev)
    NB = 4
    sets = []
    with torch.cuda.stream(stream):
        for _ in range(NB):
            d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
            d["out"] = torch.empty_like(d["q"])
            d["fin"] = torch.empty_like(d["initial_state"])
            d["ws"] = kda.alloc_workspace(T, H, N, device=dev)
            if kernel in (kda.KERNEL_SPLIT, kda.KERNEL_SPLIT_STREAMED,
                          kda.KERNEL_TC_HELPERS):   # records (+ claim words)
                n_ws = 1024 + ((T + 63) // 64 + N) * H * (66560 + 4)
                d["ws"] = torch.zeros(max(n_ws, d["ws"].numel()), dtype=torch.uint8, device=dev)
            sets.append(d)
    stream.synchronize()
    path, vsplit_used, launches_per_step = kda.plan(T, N, H, sets[0]["ws"].numel(), args.vsplit,
                                                    kernel)

    def step(i, ev_pair=None):
        d = sets[i % NB]
        if ev_pair is not None:
            ev_pair[0].record(stream)
        kda.chunk_prefill_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"],
                              d["dt_bias"], d["lower_bound"], d["scale"], d["initial_state"],
                              d["cu_seqlens"], out=d["out"], final_state=d["fin"],
                              workspace=d["ws"], stream=stream, kernel=kernel, vsplit=args.vsplit)
        if ev_pair is not None:
            ev_pair[1].record(stream)

    for i in range(max(3, args.warmup)):
        step(i)
    stream.synchronize()
    for d in sets:
        st = kda.last_device_status(d["ws"], stream)
        if st != kda.OK:
            raise kda.KDAError(st, "device status after warm-up")
    if args.profile_range:
        # one call between cudaProfilerStart/Stop, for a profiler that replays the range as a
        # whole (the grids of one call together, as they run in the timed loop)
        torch.cuda.profiler.start()
        step(0)
        stream.synchronize()
        torch.cuda.profiler.stop()
        return

    if args.steps <= 0:   # about 1.5 s of timed work so the clock sampler sees it
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(8):
            step(i)
        e1.record(stream)
        e1.synchronize()
        per = e0.elapsed_time(e1) / 8 / 1e3
        args.steps = int(min(20000, max(20, 1.5 / max(per, 1e-6))))
        if world > 1:
            t = torch.tensor([args.steps], device=dev)
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
            args.steps = int(t.item())

    K = args.steps
    uuid = str(torch.cuda.get_device_properties(dev).uuid)
    sampler = ClockSampler(uuid.replace("GPU-", ""))
    sampler.start()
    launch_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(K)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.time()
    start.record(stream)
    for i in range(K):
        step(i, launch_ev[i])
    stop.record(stream)
    stop.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    wall1 = time.time()
    clocks = sampler.stop(wall0, wall1)
    elapsed = start.elapsed_time(stop) / 1e3
    launch_s = [a.elapsed_time(b) / 1e3 for a, b in launch_ev]
    elapsed = max_over_ranks(elapsed, world)
    mean_launch = max_over_ranks(sum(launch_s) / K, world)
    for d in sets:
        st = kda.last_device_status(d["ws"], stream)
        if st != kda.OK:
            raise kda.KDAError(st, "device status after the timed steps")
    launch_us = sorted(1e6 * x for x in launch_s)
    launch_stats = {"mean": 1e6 * sum(launch_s) / K, "median": statistics.median(launch_us),
                    "min": launch_us[0], "max": launch_us[-1], "samples": K}
    # the same call under CUDA-graph replay (after the timed region, outside it)
    graph = graph_timing(step, stream) if world == 1 else None
    for d in sets:
        st = kda.last_device_status(d["ws"], stream)
        if st != kda.OK:
            raise kda.KDAError(st, "device status after the graph replays")

    # ---- end to end through the C ABI with host buffers.  Every step copies its inputs
    #      from pinned host memory and reads its out and final_state back; steps are
    #      pipelined over two device buffer sets and three streams (copy in, compute,
    #      copy out), so step i+1's inputs travel while step i computes.
    pinned = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
    out_h = [torch.empty(tuple(host["q"].shape), dtype=torch.bfloat16).pin_memory()
             for _ in range(2)]
    fin_h = [torch.empty(tuple(host["initial_state"].shape),
                         dtype=host["initial_state"].dtype).pin_memory() for _ in range(2)]
    names = ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "initial_state", "cu_seqlens")
    h2d = sum(pinned[k].numel() * pinned[k].element_size() for k in names)
    d2h = out_h[0].numel() * out_h[0].element_size() + fin_h[0].numel() * fin_h[0].element_size()
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_done = [torch.cuda.Event() for _ in range(2)]     # inputs of slot b copied in
    comp_done = [torch.cuda.Event() for _ in range(2)]   # slot b computed
    out_done = [torch.cuda.Event() for _ in range(2)]    # slot b's results copied out
    used = [False, False]

    def e2e_step(i):
        b = i % 2
        d = sets[b]
        if used[b]:
            s_in.wait_event(comp_done[b])     # the slot's previous step no longer reads it
        with torch.cuda.stream(s_in):
            for k in names:
                d[k].copy_(pinned[k], non_blocking=True)
        in_done[b].record(s_in)
        stream.wait_event(in_done[b])
        if used[b]:
            stream.wait_event(out_done[b])    # its previous results have been copied out
        kda.chunk_prefill_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"],
                              d["dt_bias"], d["lower_bound"], d["scale"], d["initial_state"],
                              d["cu_seqlens"], out=d["out"], final_state=d["fin"],
                              workspace=d["ws"], stream=stream, kernel=kernel)
        comp_done[b].record(stream)
        s_out.wait_event(comp_done[b])
        with torch.cuda.stream(s_out):
            out_h[b].copy_(d["out"], non_blocking=True)
            fin_h[b].copy_(d["fin"], non_blocking=True)
        out_done[b].record(s_out)
        used[b] = True

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    KE = max(1, args.e2e_steps)
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(KE):
        e2e_step(i)
    e1.record(s_out)
    e1.synchronize()
    barrier(world)
    e2e_elapsed = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    kernel_name = {kda.KERNEL_TC: "kda_tc_chunk_kernel", kda.KERNEL_REF: "kda_ref_chunk_kernel",
                   kda.KERNEL_SPLIT: "kda_split_path", kda.KERNEL_TC_HELPERS: "kda_tc_helpers_path",
                   kda.KERNEL_SPLIT_STREAMED: "kda_split_streamed_path",
                   kda.KERNEL_PIPE: "kda_pipe_kernel"}[path]
    hbm, tflops, peak_kind = load_peaks()
    abytes = algorithmic_bytes(w)
    achieved = abytes / mean_launch / 1e9
    value = world * T * K / elapsed
    us = 1e6 * elapsed / K
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": 1e3 * elapsed / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "tokens": T, "seqs": N, "heads": H, "head_dim": D,
                   "state": w.state_dtype, "chunk": 64, "kernel": args.kernel,
                   "path": kernel_name, "vsplit": vsplit_used,
                   "l2": f"inputs {algorithmic_bytes(w) / 1e6:.0f} MB per step, 4 input sets rotated",
                   "parallelism": f"replicas x{world}"},
        "us_per_layer": us,
        "roofline": {"bound": "hbm", "kernel": kernel_name, "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": load_traffic(kernel_name, w.name),
                     "algorithmic_bytes_per_launch": abytes,
                     "mean_launch_us": 1e6 * mean_launch, "peak_source": peak_kind,
                     "roofline_us": 1e6 * abytes / (hbm * 1e9),
                     "tensor_flops_per_launch": algorithmic_flops(w),
                     "tensor_frac": algorithmic_flops(w) / mean_launch / (tflops * 1e12)},
        "e2e": {"value": world * T * KE / e2e_elapsed, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": KE},
        "gpu_launches": K * launches_per_step,
        "clocks": clocks,
        "launch_us": launch_stats,
    }
    if graph is not None:
        line["graph"] = graph
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(host, w)
        line["cpu_baseline_1thread"] = cpu_baseline_one_thread(host, w)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
