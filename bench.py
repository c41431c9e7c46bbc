"""Benchmark of the hot path: one step = one pass over every hot-path kernel on the
Q4_K 18944 x 3584 weight (a Qwen2.5-7B FFN up/gate projection, synthetic):

  1. decode matvec, B = 1           (the Q-matvec HBM GB/s metric)
  2. activation quantise, M = 512
  3. prefill MMQ, M = 512           (the prefill MMQ TOPS metric)

Prints one JSON line.  `value` is the decode matvec's HBM throughput (algorithmic
bytes / kernel time, whole job = all ranks), timed over back-to-back calls on
rotating weight copies (> 3x the 135 MB L2) replayed from a CUDA graph; the
MMQ's int-op rate and the per-kernel rooflines are in the same line.  The K
timed steps (matvec + quantise + MMQ each) are one captured CUDA graph, replayed
once at the end of a sustained busy period of untimed replays of the same graph
(clocks are sampled over all of it).  `configs` holds every configuration of the
five workloads (Q8_0 896 x 896; Q4_K 18944 x 3584; Q6_K 3584 x 18944 at B = 1, 2,
4, 8; the Q4_K prefill at M = 512; the Q6_K 151936 x 3584 LM head at M = 1 and
M = 2048), each with its roofline.  `cpu_baseline` times the oracle on one core
and on all cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mq|reference]
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "q4_k_18944x3584: decode matvec B=1 + quantise + MMQ M=512"
METRIC = "Q-matvec HBM GB/s (% of peak); prefill MMQ int8 TOPS (% of tensor peak)"
QTYPE, N, K, B, M = 12, 18944, 3584, 1, 512
W_SEED, XD_SEED, XA_SEED = 102, 202, 204
ROT = 4  # prefill buffer sets rotated between steps (4 x ~220 MB >> L2)
L2_BYTES = 135e6
SOAK_S = 1.5  # seconds of sustained replays ending with the timed region

# algorithmic bytes / ops per launch (what the method must move or compute)
MV_BYTES = N * (K // 256) * 144 + B * K * 4 + B * N * 4
Q_BYTES = M * K * 4 + M * K + 2 * M * (K // 32) * 4 + M * K * 2
MMQ_OPS = 2 * M * N * K
SMI_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def max_over_ranks(values, ws, device):
    """Each rank's timings replaced by their maximum over the ranks (the slowest rank sets
    the job's time); any process-group backend, tensors on `device`."""
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    if ws > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job(per_rank_rate, ws):
    """Replicas (weak scaling): every rank processes the same units in the common (maximum)
    time, so the whole job's rate is the per-rank rate times the number of ranks."""
    return per_rank_rate * ws


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={SMI_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for nm, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


def src_sha(paths):
    """sha256[:16] of a source file, or of several files' bytes in the order given."""
    if isinstance(paths, str):
        paths = [paths]
    h = hashlib.sha256()
    for path in paths:
        h.update(open(path, "rb").read())
    return h.hexdigest()[:16]


def matvec_kernel_name(qtype, n, sms):
    """The matvec kernel the library launches for a weight of this type and row count: the
    persistent kernel for Q4_K / Q5_K / Q6_K weights of at least sms / 2 row groups of 128,
    else the split-K kernel."""
    import synth
    persistent = qtype in (12, 13, 14) and (n + 127) // 128 * 2 >= sms
    return ("matvec_kq_kernel" if persistent else "matvec_kernel") + f"<{synth.TYPE_NAME[qtype]}>"


def traffic_for(kernel_key, src):
    """DRAM bytes per launch from a committed ncu summary (profiles/traffic.txt: lines of
    `key dram_bytes_per_launch source_sha`), if the kernel source is unchanged since the
    counters were taken; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    for line in open(p):
        f = line.split()
        if len(f) >= 3 and not line.startswith("#") and f[0] == kernel_key:
            return float(f[1]) if f[2] == src_sha(src) else None
    return None


def _host_cpus():
    """(usable cores, CPU model line) of this host: os.sched_getaffinity and lscpu."""
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    model = "unknown"
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    return cores, model


def _timed(fn, min_s):
    """(seconds per call, calls) of fn() repeated until at least min_s seconds have passed."""
    n, t0 = 0, time.perf_counter()
    while True:
        fn()
        n += 1
        t = time.perf_counter() - t0
        if t >= min_s:
            return t / n, n


def cpu_baseline(budget_s: float = 16.0):
    """The oracle, as it stands, on the bench workload's own inputs: the decode matvec
    (GB/s, the value metric) and the prefill MMQ (TOPS), each on one core and on all
    cores (the OpenMP build of the same oracle.c: rows in parallel, per-row arithmetic
    unchanged).  One-core figures come from a sample of the call, extrapolated linearly
    (the work per row is fixed); all-core figures time the full decode call and a
    16-row slice of the prefill."""
    import oracle
    import synth
    Wb = synth.weights(QTYPE, N, K, W_SEED)
    xd = synth.activations(B, K, XD_SEED)
    xa = synth.activations(M, K, XA_SEED)
    qs, sc, _ = oracle.quantize_act(xa)
    cores, model = _host_cpus()
    threads = oracle.threads(True)
    q = budget_s / 4
    # decode matvec, one core: the first `rows` weight rows
    rows = 64
    while True:
        t1, _ = _timed(lambda: oracle.matvec(QTYPE, Wb, N, K, xd, 0, rows), 0.0)
        if t1 > q / 4 or rows >= N:
            break
        rows = min(N, rows * 4)
    t1, _ = _timed(lambda: oracle.matvec(QTYPE, Wb, N, K, xd, 0, rows), q)
    mv1 = (rows * (K // 256) * 144 + B * K * 4 + B * rows * 4) / t1 / 1e9
    # decode matvec, all cores: the whole call
    tall, nall = _timed(lambda: oracle.matvec(QTYPE, Wb, N, K, xd, parallel=True), q)
    mvall = MV_BYTES / tall / 1e9
    # prefill MMQ, 16 activation rows: one core against `nrow` weight rows, all cores
    # against all N rows
    mrows = list(range(16))
    nrow = 16
    while True:
        tm1, _ = _timed(lambda: oracle.mmq(QTYPE, Wb, N, K, qs, sc, mrows=mrows, n1=nrow), 0.0)
        if tm1 > q / 4 or nrow >= N:
            break
        nrow = min(N, nrow * 4)
    tm1, _ = _timed(lambda: oracle.mmq(QTYPE, Wb, N, K, qs, sc, mrows=mrows, n1=nrow), q)
    tmall, _ = _timed(lambda: oracle.mmq(QTYPE, Wb, N, K, qs, sc, mrows=mrows, parallel=True), q)
    mm1 = 2 * 16 * nrow * K / tm1 / 1e12
    mmall = 2 * 16 * N * K / tmall / 1e12
    return {
        "value": mvall, "unit": "GB/s", "cores": threads, "kind": "oracle",
        "sample": (f"decode matvec {N}x{K} B={B}: the full call on {threads} threads "
                   f"({nall} calls); prefill MMQ: activation rows 0..15 x all {N} weight "
                   f"rows on {threads} threads; plain C, fp64 accumulation"),
        "mmq_tops": mmall,
        "one_core": {"value": mv1, "unit": "GB/s", "mmq_tops": mm1, "cores": 1,
                     "sample": (f"decode matvec over weight rows 0..{rows} of {N}; MMQ of "
                                f"activation rows 0..15 x weight rows 0..{nrow}; rates per "
                                "row extrapolated linearly to the full calls")},
        "host": {"affinity_cpus": cores, "lscpu_model": model, "openmp_threads": threads},
    }


def workload_config(ws: int):
    """The `config` object of both arms' JSON lines."""
    return {"workload": WORKLOAD, "N": N, "K": K, "decode_B": B, "prefill_M": M,
            "qtype": "Q4_K", "seeds": {"W": W_SEED, "x_decode": XD_SEED, "x_prefill": XA_SEED},
            "l2": ("inputs larger than L2: decode weight copies rotated (> 3x L2 together); "
                   "each step's prefill moves ~180 MB between decode calls"),
            "parallelism": f"replicas x{ws}"}


def run_reference(args):
    """The reference arm: the oracle (all host cores), as it stands, on the same workload;
    each step one full decode matvec call (the value metric) plus a 16-row slice of the
    prefill MMQ.  Rank 0 alone runs it."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    import synth
    Wb = synth.weights(QTYPE, N, K, W_SEED)
    xd = synth.activations(B, K, XD_SEED)
    qs, sc, _ = oracle.quantize_act(synth.activations(M, K, XA_SEED))
    threads = oracle.threads(True)
    cores, model = _host_cpus()

    def step():
        t0 = time.perf_counter()
        oracle.matvec(QTYPE, Wb, N, K, xd, parallel=True)
        t1 = time.perf_counter()
        oracle.mmq(QTYPE, Wb, N, K, qs, sc, mrows=list(range(16)), parallel=True)
        return t1 - t0, time.perf_counter() - t1

    for _ in range(args.warmup):
        step()
    tm = [step() for _ in range(args.steps)]
    t_mv = statistics.median(a for a, _ in tm)
    t_mm = statistics.median(b for _, b in tm)
    v = MV_BYTES / t_mv / 1e9
    sample = (f"each step: the full decode matvec {N}x{K} B={B} and activation rows 0..15 of "
              f"the prefill MMQ (all {N} weight rows), on {threads} threads")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000 * sum(a + b for a, b in tm) / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(ws),
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample,
                             "host": {"affinity_cpus": cores, "lscpu_model": model}},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "mmq_tops": 2 * 16 * N * K / t_mm / 1e12}
    print(json.dumps(line))
    return 0


def graph_time_ms(fn, calls, trials=5):
    """Median over `trials` of the device time of one replay of a CUDA graph holding
    `fn(j)` for j < calls, divided by calls (events on the replay stream)."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for j in range(calls):
            fn(j)
    g.replay()
    torch.cuda.synchronize()
    out = []
    for _ in range(trials):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        out.append(e0.elapsed_time(e1) / calls)
    del g
    return statistics.median(out)


def profile_calls(kernel: str, calls: int, batch=None, workload=None, from_decode_plane=False):
    """Run `calls` launches of one hot-path kernel on the bench workload (or on the weight
    of another named workload) and exit: the program that ncu captures are taken of (one
    kernel, few launches, ~0.3 GB on device).  from_decode_plane: register the (Q4_K) weight
    with MQ_REG_MMQ_FROM_DECODE_PLANE."""
    import torch

    import gguf_block_quantized_q4_gb300 as mq
    from gguf_block_quantized_q4_gb300 import build as mqbuild
    import synth
    mqbuild.build()
    mq.init(0)
    qt, n, k, ws, xs = QTYPE, N, K, W_SEED, XD_SEED
    if workload:
        c = synth.WORKLOADS[workload]
        qt, n, k, ws, xs = c["qtype"], c["N"], c["K"], c["w_seed"], c["x_seed"]
    Wb = synth.weights(qt, n, k, ws)
    flags = mq.REG_NO_MMQ_PLANE if kernel == "matvec" else mq.REG_DEFAULT
    if from_decode_plane:
        flags = mq.REG_MMQ_FROM_DECODE_PLANE
    W = mq.register_weight(qt, Wb, n, k, flags)
    if kernel == "matvec":
        nb = batch or B
        x = torch.from_numpy(synth.activations(nb, k, xs)).cuda()
        y = torch.empty((nb, n), device="cuda")
        for _ in range(calls):
            mq.matvec(W, x, y)
    else:
        m = batch or M  # activation rows (the K = 3584 quantiser of C5 at --batch 2048)
        x = torch.from_numpy(synth.activations(m, k, XA_SEED)).cuda()
        xq = mq.quantize_act(x)
        y = torch.empty((m, n), device="cuda")
        for _ in range(calls):
            if kernel == "quantize":
                mq.quantize_act(x, xq)
            else:
                mq.mmq(W, xq, m, y)
    torch.cuda.synchronize()
    mq.stream_status()
    W.free()
    return 0


def chain_timing(links: int, reps: int = 200):
    """Per-link time of a decode chain of `links` Q8_0 896x896 matvecs (B = 1), issued
    eagerly and as one captured CUDA graph (a side measurement, not the bench line)."""
    import torch

    import gguf_block_quantized_q4_gb300 as mq
    from gguf_block_quantized_q4_gb300 import build as mqbuild
    import synth
    mqbuild.build()
    mq.init(0)
    Ws = [mq.register_weight(synth.Q8_0, synth.weights(synth.Q8_0, 896, 896, 300 + l), 896, 896,
                             mq.REG_NO_MMQ_PLANE) for l in range(links)]
    x = torch.from_numpy(synth.activations(1, 896, 7)).cuda()
    ys = [torch.empty((1, 896), device="cuda") for _ in range(links)]

    def chain():
        h = x
        for W, y in zip(Ws, ys):
            mq.matvec(W, h, y)
            h = y

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            chain()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        chain()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    out = {}
    for name, fn in (("eager", chain), ("graph", g.replay)):
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        out[name + "_us_per_link"] = e0.elapsed_time(e1) * 1e3 / (reps * links)
    mq.stream_status()
    for W in Ws:
        W.free()
    print(json.dumps({"chain": f"{links} x Q8_0 896x896 matvec, B=1", **out}))
    return 0


def ffn_gu_timing(reps: int = 20):
    """Fused gate/up (one matvec or MMQ over both weights, SwiGLU in the store) against
    the two plain calls, on the Q4_K 18944 x 3584 pair: a side measurement, not the bench
    line.  Graph replays of back-to-back calls on rotating buffers, CUDA events."""
    import torch

    import gguf_block_quantized_q4_gb300 as mq
    from gguf_block_quantized_q4_gb300 import build as mqbuild
    import synth
    mqbuild.build()
    mq.init(0)
    g, u = synth.weights(QTYPE, N, K, W_SEED), synth.weights(QTYPE, N, K, W_SEED + 1)
    rot = 4  # weight copies rotated so the decode weights come from HBM
    fused = [mq.register_ffn_gu(QTYPE, g, u, N, K) for _ in range(rot)]
    gates = [mq.register_weight(QTYPE, g, N, K) for _ in range(rot)]
    ups = [mq.register_weight(QTYPE, u, N, K) for _ in range(rot)]
    x = torch.from_numpy(synth.activations(B, K, XD_SEED)).cuda()
    xa = torch.from_numpy(synth.activations(M, K, XA_SEED)).cuda()
    xq = mq.quantize_act(xa)
    hy = torch.empty((M, N), device="cuda")
    gy, uy = torch.empty((M, N), device="cuda"), torch.empty((M, N), device="cuda")
    out = {}
    cases = {
        "matvec_fused_us": lambda i: mq.ffn_gu_matvec(fused[i % rot], x, hy[:B]),
        "matvec_two_calls_us": lambda i: (mq.matvec(gates[i % rot], x, gy[:B]),
                                          mq.matvec(ups[i % rot], x, uy[:B])),
        "mmq_fused_us": lambda i: mq.ffn_gu_mmq(fused[i % rot], xq, M, hy),
        "mmq_two_calls_us": lambda i: (mq.mmq(gates[i % rot], xq, M, gy),
                                       mq.mmq(ups[i % rot], xq, M, uy)),
    }
    for name, fn in cases.items():
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for i in range(3):
                fn(i)
        torch.cuda.current_stream().wait_stream(s)
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            for i in range(reps):
                fn(i)
        gr.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        gr.replay()
        e1.record()
        torch.cuda.synchronize()
        out[name] = e0.elapsed_time(e1) * 1e3 / reps
    mq.stream_status()
    for w in fused + gates + ups:
        w.free()
    print(json.dumps({"ffn_gu": f"Q4_K gate+up {N}x{K} each, decode B={B}, prefill M={M}",
                      **out}))
    return 0


def rotation(nbytes: float) -> int:
    """Copies of an input that together exceed 3x L2, so back-to-back calls read HBM."""
    return max(1, int(np.ceil(3 * L2_BYTES / nbytes)))


def roof(kernel, bound, achieved, peak, unit, ms, algorithmic, traffic=None, note=None):
    r = {"kernel": kernel, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
         "frac": achieved / peak, "traffic": traffic, "ms": ms}
    r["algorithmic_bytes" if bound == "hbm" else "algorithmic_ops"] = algorithmic
    if note:
        r["note"] = note
    return r


MMQ_PEAK_NOTE = ("the integer contraction runs exactly on the f16 tensor pipe (integer-valued "
                 "f16 operands, f32 accumulation): sm_103a has no tcgen05 kind::i8, and the "
                 "legacy int8 mma.sync path measured 151 TOPS on this GPU; frac is against the "
                 "measured bf16 burst peak (f16 runs at the bf16 rate)")


def measure_configs(mq, dev, hbm, bf16):
    """Every configuration of the five hot-path workloads: device time per call from graph
    replays of back-to-back calls on rotating inputs (median of 5), with its roofline."""
    import torch

    import synth
    WL = synth.WORKLOADS
    out = {}
    csrc = os.path.join(ROOT, "gguf_block_quantized_q4_gb300", "csrc")

    def mv_bytes(qtype, n, k, b):
        be, bb = synth.BLOCK[qtype]
        return n * (k // be) * bb + b * k * 4 + b * n * 4

    sms = torch.cuda.get_device_properties(dev).multi_processor_count

    def matvec_case(name, batches, rotate=True):
        c = WL[name]
        qt, n, k = c["qtype"], c["N"], c["K"]
        wb = synth.weights(qt, n, k, c["w_seed"])
        rot = rotation(len(wb)) if rotate else 1
        Ws = [mq.register_weight(qt, wb, n, k, mq.REG_NO_MMQ_PLANE) for _ in range(rot)]
        res = {}
        for b in batches:
            x = torch.from_numpy(synth.activations(b, k, c["x_seed"], c["x_scale"])).to(dev)
            ys = [torch.empty((b, n), device=dev) for _ in range(rot)]
            t = graph_time_ms(lambda j: mq.matvec(Ws[j % rot], x, ys[j % rot]),
                              max(8, 2 * rot) if rot > 1 else 20)
            by = mv_bytes(qt, n, k, b)
            res[b] = roof(matvec_kernel_name(qt, n, sms), "hbm", by / (t * 1e-3) / 1e9,
                          hbm, "GB/s", t, by)
            res[b]["weight_copies_rotated"] = rot
        return Ws, res

    # C1: Q8_0 896 x 896, B = 1 (L2-resident; launch-bound): us per call, eager and graphed
    Ws, r = matvec_case("q8_0_matvec_896x896", [1])
    c1 = r[1]
    x = torch.from_numpy(synth.activations(1, 896, 0)).to(dev)
    ys = [torch.empty((1, 896), device=dev) for _ in range(len(Ws))]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for j in range(20):
        mq.matvec(Ws[j % len(Ws)], x, ys[j % len(Ws)])
    reps = 2000
    torch.cuda.synchronize()
    e0.record()
    for j in range(reps):
        mq.matvec(Ws[j % len(Ws)], x, ys[j % len(Ws)])
    e1.record()
    torch.cuda.synchronize()
    eager_us = e0.elapsed_time(e1) * 1e3 / reps
    g1000 = graph_time_ms(lambda j: mq.matvec(Ws[j % len(Ws)], x, ys[j % len(Ws)]), 1000, 3)
    c1.update({"us_per_call_graph": c1["ms"] * 1e3, "us_per_call_eager": eager_us,
               "us_per_call_graph_1000": g1000 * 1e3,
               "note": ("0.86 MB, L2-resident when repeated: launch-bound, reported in us per "
                        "call; eager = back-to-back host launches through the Python binding")})
    out["c1_q8_0_matvec_896x896_b1"] = c1
    for W in Ws:
        W.free()
    # C2: Q4_K 18944 x 3584, B = 1
    Ws, r = matvec_case("q4_k_matvec_18944x3584", [1])
    out["c2_q4_k_matvec_18944x3584_b1"] = r[1]
    for W in Ws:
        W.free()
    # C3: Q6_K 3584 x 18944, B = 1, 2, 4, 8
    Ws, r = matvec_case("q6_k_matvec_3584x18944", [1, 2, 4, 8])
    for b in (1, 2, 4, 8):
        out[f"c3_q6_k_matvec_3584x18944_b{b}"] = r[b]
    for W in Ws:
        W.free()

    def prefill_case(name, key, rot):
        c = WL[name]
        qt, n, k, m = c["qtype"], c["N"], c["K"], c["M"][0]
        wb = synth.weights(qt, n, k, c["w_seed"])
        Ws = [mq.register_weight(qt, wb, n, k) for _ in range(rot)]
        xs = [torch.from_numpy(synth.activations(m, k, c["x_seed"], c["x_scale"])).to(dev)
              for _ in range(rot)]
        xq = [mq.act_buffer(m, k, dev) for _ in range(rot)]
        ys = [torch.empty((m, n), device=dev) for _ in range(rot)]
        tq = graph_time_ms(lambda j: mq.quantize_act(xs[j % rot], xq[j % rot]), 4 * rot)
        tm = graph_time_ms(lambda j: mq.mmq(Ws[j % rot], xq[j % rot], m, ys[j % rot]), 2 * rot)
        tf = graph_time_ms(lambda j: mq.mmq_fused(Ws[j % rot], xs[j % rot], xq[j % rot],
                                                  ys[j % rot]), 2 * rot)
        qbytes = m * k * 4 + m * k + 2 * m * (k // 32) * 4 + m * k * 2
        ops = 2 * m * n * k
        out[f"{key}_quantize"] = roof("quantize_act_kernel", "hbm", qbytes / (tq * 1e-3) / 1e9,
                                      hbm, "GB/s", tq, qbytes)
        out[f"{key}_mmq"] = roof(f"mmq_tc_kernel<{synth.TYPE_NAME[qt]}>", "tensor",
                                 ops / (tm * 1e-3) / 1e12, bf16, "TFLOP/s", tm, ops,
                                 note=MMQ_PEAK_NOTE)
        out[f"{key}_prefill_incl_quantise"] = {
            "two_kernels_ms": tq + tm, "fused_ms": tf,
            "two_kernels_tops": ops / ((tq + tm) * 1e-3) / 1e12,
            "fused_tops": ops / (tf * 1e-3) / 1e12}
        for W in Ws:
            W.free()

    # C4: Q4_K prefill, M = 512
    prefill_case("q4_k_mmq_512x18944x3584", "c4_q4_k_m512", 4)
    # C5: Q6_K LM head 151936 x 3584: M = 1 decode matvec, M = 2048 prefill
    Ws, r = matvec_case("q6_k_lm_head_151936x3584", [1], rotate=False)
    out["c5_q6_k_lm_head_151936x3584_m1"] = r[1]
    for W in Ws:
        W.free()
    prefill_case("q6_k_lm_head_151936x3584", "c5_q6_k_lm_head_m2048", 1)
    torch.cuda.synchronize()
    mq.stream_status()
    return out


def run_mq(args):
    import torch

    import gguf_block_quantized_q4_gb300 as mq
    from gguf_block_quantized_q4_gb300 import build as mqbuild
    import synth

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    mqbuild.build()
    mq.init(local)
    dev = torch.device("cuda", local)
    hbm, bf16, peak_src = peaks()

    Wb = synth.weights(QTYPE, N, K, W_SEED)
    # decode: RMV weight copies, > 3x L2 together, so back-to-back calls read HBM
    rmv = rotation(len(Wb))
    Wd = [mq.register_weight(QTYPE, Wb, N, K, mq.REG_NO_MMQ_PLANE) for _ in range(rmv)]
    Wp = [mq.register_weight(QTYPE, Wb, N, K) for _ in range(ROT)]
    xd_h = synth.activations(B, K, XD_SEED)
    xa_h = synth.activations(M, K, XA_SEED)
    xd = [torch.from_numpy(xd_h).to(dev) for _ in range(ROT)]
    xa = [torch.from_numpy(xa_h).to(dev) for _ in range(ROT)]
    yd = [torch.empty((B, N), device=dev) for _ in range(rmv)]
    xq = [torch.empty(mq.act_bytes(M, K), dtype=torch.uint8, device=dev) for _ in range(ROT)]
    ym = [torch.empty((M, N), device=dev) for _ in range(ROT)]

    def step(i):
        # one pass of the hot path: a decode matvec, then a prefill (quantise + MMQ); the
        # prefill's ~180 MB of traffic evicts the next decode weight from L2
        r = i % ROT
        mq.matvec(Wd[i % rmv], xd[r], yd[i % rmv])
        mq.quantize_act(xa[r], xq[r])
        mq.mmq(Wp[r], xq[r], M, ym[r])

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    mq.stream_status()

    # the K timed steps, captured once as a CUDA graph (no host launch gaps)
    g_steps = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_steps):
        for i in range(args.steps):
            step(i)
    g_steps.replay()  # untimed warm replay
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # Clocks are sampled over a sustained busy period that ends with the timed region: the
    # same step graph replayed (untimed) for >= SOAK_S seconds, then the K timed steps.
    t0 = time.perf_counter()
    g_steps.replay()
    torch.cuda.synchronize()
    soak_reps = max(1, int(np.ceil(SOAK_S / max(1e-6, time.perf_counter() - t0))))
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_soak = time.perf_counter()
        for _ in range(soak_reps):
            g_steps.replay()
        e0.record()
        g_steps.replay()
        e1.record()
        torch.cuda.synchronize()
        t_soak = time.perf_counter() - t_soak
    if ws > 1:
        torch.distributed.barrier()
    mq.stream_status()
    total_ms = e0.elapsed_time(e1)
    del g_steps

    # per-kernel device times: back-to-back calls on rotating buffers, graph replays
    t_mv = graph_time_ms(lambda j: mq.matvec(Wd[j % rmv], xd[j % ROT], yd[j % rmv]), 5 * rmv)
    t_q = graph_time_ms(lambda j: mq.quantize_act(xa[j % ROT], xq[j % ROT]), 4 * ROT)
    t_mm = graph_time_ms(lambda j: mq.mmq(Wp[j % ROT], xq[j % ROT], M, ym[j % ROT]), 2 * ROT)
    # the prefill with the quantisation inside the MMQ kernel (one cooperative launch)
    xqf = [mq.act_buffer(M, K, dev) for _ in range(ROT)]
    t_fu = graph_time_ms(lambda j: mq.mmq_fused(Wp[j % ROT], xa[j % ROT], xqf[j % ROT],
                                                ym[j % ROT]), 2 * ROT)
    mq.stream_status()
    total_ms, t_mv, t_q, t_mm, t_fu = max_over_ranks([total_ms, t_mv, t_q, t_mm, t_fu], ws, dev)

    # end to end through the public API, eager: pinned host inputs in, results back out
    stream = torch.cuda.current_stream()
    xd_p = torch.from_numpy(xd_h).pin_memory()
    xa_p = torch.from_numpy(xa_h).pin_memory()
    yd_p = torch.empty((B, N), dtype=torch.float32).pin_memory()
    ym_p = torch.empty((M, N), dtype=torch.float32).pin_memory()

    def e2e_step(i, ev):
        r = i % ROT
        # one C-ABI call each: H2D of x from pinned host memory, the kernel(s), D2H of y
        ev[0].record(stream)
        mq.matvec_host(Wd[i % rmv], xd_p, yd_p, xd[r], yd[i % rmv], stream)
        ev[1].record(stream)
        mq.mmq_host(Wp[r], xa_p, ym_p, xa[r], xq[r], ym[r], stream)
        ev[2].record(stream)

    eev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for i in range(args.warmup):
        e2e_step(i, eev[0])
    torch.cuda.synchronize()
    for i in range(args.steps):
        e2e_step(i, eev[i])
    torch.cuda.synchronize()
    te_mv = statistics.median(e[0].elapsed_time(e[1]) for e in eev)
    te_mm = statistics.median(e[1].elapsed_time(e[2]) for e in eev)
    te_mv, te_mm = max_over_ranks([te_mv, te_mm], ws, dev)
    assert np.isfinite(yd_p.numpy()).all() and np.isfinite(ym_p.numpy()).all()
    for w in Wd + Wp:
        w.free()
    del xq, xqf, ym
    torch.cuda.empty_cache()

    # every configuration of the five workloads (the step above covers two of them)
    configs = measure_configs(mq, dev, hbm, bf16) if not args.no_configs else None

    mv_gbs = MV_BYTES / (t_mv * 1e-3) / 1e9
    q_gbs = Q_BYTES / (t_q * 1e-3) / 1e9
    mm_tops = MMQ_OPS / (t_mm * 1e-3) / 1e12
    csrc = os.path.join(ROOT, "gguf_block_quantized_q4_gb300", "csrc")
    kern = {
        "matvec": roof("matvec_kq_kernel<Q4_K>", "hbm", mv_gbs, hbm, "GB/s", t_mv, MV_BYTES,
                       traffic_for("matvec_q4_k_b1", [os.path.join(csrc, "matvec_kq.cu"),
                                                      os.path.join(csrc, "mv_device.cuh")])),
        "quantize": roof("quantize_act_kernel", "hbm", q_gbs, hbm, "GB/s", t_q, Q_BYTES,
                         traffic_for("quantize_m512", [os.path.join(csrc, "quantize.cu"),
                                                       os.path.join(csrc, "quant_row.cuh")])),
        "mmq": roof("mmq_tc_kernel<Q4_K>", "tensor", mm_tops, bf16, "TFLOP/s", t_mm, MMQ_OPS,
                    traffic_for("mmq_q4_k_m512", [os.path.join(csrc, "mmq.cu"),
                                                  os.path.join(csrc, "quant_row.cuh")]),
                    note=MMQ_PEAK_NOTE),
    }
    dom = max(kern, key=lambda k: kern[k]["ms"])
    roofl = {k: kern[dom][k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic")}
    roofl["kernel"] = kern[dom]["kernel"]
    roofl["peak_source"] = (f"{peak_src} ({'hbm_gbs' if roofl['bound'] == 'hbm' else 'bf16_tflops'}"
                            " burst)")
    if "note" in kern[dom]:
        roofl["peak_note"] = kern[dom]["note"]
    e2e_mv = MV_BYTES / (te_mv * 1e-3) / 1e9
    e2e_mm = MMQ_OPS / (te_mm * 1e-3) / 1e12
    config = workload_config(ws)
    config["timing"] = (f"steps: one CUDA graph of K steps, timed once (exactly K steps) at the "
                        f"end of a sustained busy period of {soak_reps} untimed replays of the "
                        f"same graph ({t_soak:.2f} s in all, clocks sampled throughout); "
                        "per-kernel and per-config: graph replays of back-to-back calls on "
                        "rotating buffers, median of 5")
    line = {
        "metric": METRIC, "value": whole_job(mv_gbs, ws), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16xf16->f32",
        "data": "synthetic (seeded, Qwen2.5-7B FFN-shaped Q4_K weights, N(0,1) activations)",
        "config": config,
        "matvec_gbs": whole_job(mv_gbs, ws), "matvec_frac_of_hbm": mv_gbs / hbm,
        "matvec_frac_of_8tbs": mv_gbs / 8000.0,
        "mmq_tops": whole_job(mm_tops, ws), "mmq_frac_of_f16_peak": mm_tops / bf16,
        "quantize_gbs": whole_job(q_gbs, ws),
        "roofline": roofl, "kernels": kern,
        "configs": configs,
        "prefill_incl_quantise": {
            "two_kernels_ms": t_q + t_mm, "fused_ms": t_fu,
            "two_kernels_tops": whole_job(MMQ_OPS / ((t_q + t_mm) * 1e-3) / 1e12, ws),
            "fused_tops": whole_job(MMQ_OPS / (t_fu * 1e-3) / 1e12, ws),
            "note": "quantise + MMQ as two launches, and as mq_mmq_fused (one cooperative "
                    "launch); graph replays of back-to-back calls"},
        "e2e": {"value": whole_job(e2e_mv, ws), "unit": "GB/s",
                "h2d_bytes_per_step": B * K * 4 + M * K * 4,
                "d2h_bytes_per_step": B * N * 4 + M * N * 4,
                "mmq_tops": whole_job(e2e_mm, ws),
                "note": "eager calls of the C ABI with pinned host buffers (mq_matvec_host: "
                        "x pulled over the host link by a copy kernel that the matvec overlaps, "
                        "y stored by the matvec into host memory; mq_mmq_host: the quantiser "
                        "reads x from host memory, then the MMQ in up to four chunks of 128-row "
                        "tiles, each chunk's rows of y copied to the host while the next chunk "
                        "runs), device time per step "
                        "between events, medians"},
        "gpu_launches": 3 * args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(line))
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mq", choices=["mq", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration measurements of the five workloads")
    ap.add_argument("--kernel", choices=["matvec", "quantize", "mmq"],
                    help="profiling mode: only run --calls launches of this kernel")
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--workload", default=None,
                    help="profiling mode: the weight of this named workload instead of the "
                         "bench's (e.g. q6_k_matvec_3584x18944)")
    ap.add_argument("--batch", type=int, default=None,
                    help="profiling mode: the matvec's batch rows (1..8), or the quantiser's and "
                         "MMQ's activation rows (default: the bench's decode batch / prefill M)")
    ap.add_argument("--mmq-from-decode-plane", action="store_true",
                    help="profiling mode: register the Q4_K weight without the f16 plane (the "
                         "MMQ expands the decode-plane tiles in shared memory)")
    ap.add_argument("--chain", type=int, default=0,
                    help="time a decode chain of this many small matvecs, eager and graphed")
    ap.add_argument("--ffn-gu", action="store_true",
                    help="time the fused gate/up matvec and MMQ against two plain calls")
    args = ap.parse_args()
    if args.kernel:
        if args.batch is not None and not (1 <= args.batch <= (8 if args.kernel == "matvec" else 4096)):
            ap.error("--batch: 1..8 for the matvec, 1..4096 for the quantiser and the MMQ")
        if args.workload is not None:
            import synth
            if args.workload not in synth.WORKLOADS:
                ap.error(f"--workload: one of {', '.join(synth.WORKLOADS)}")
        return profile_calls(args.kernel, args.calls, args.batch, args.workload,
                             args.mmq_from_decode_plane)
    if args.chain:
        return chain_timing(args.chain)
    if args.ffn_gu:
        return ffn_gu_timing()
    if args.impl == "reference":
        return run_reference(args)
    args.warmup = max(args.warmup, 3)
    return run_mq(args)


if __name__ == "__main__":
    sys.exit(main())
