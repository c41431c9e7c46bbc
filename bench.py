"""Benchmark of the hot path: one step = one pass over every hot-path kernel on the
Q4_K 18944 x 3584 weight (a Qwen2.5-7B FFN up/gate projection, synthetic):

  1. decode matvec, B = 1           (the Q-matvec HBM GB/s metric)
  2. activation quantise, M = 512
  3. prefill MMQ, M = 512           (the prefill MMQ TOPS metric)

Prints one JSON line.  `value` is the decode matvec's HBM throughput (algorithmic
bytes / kernel time, whole job = all ranks), timed over back-to-back calls on
rotating weight copies (> 3x the 135 MB L2) replayed from a CUDA graph; the
MMQ's int-op rate and the per-kernel rooflines are in the same line.  The K
timed steps (matvec + quantise + MMQ each) are one captured CUDA graph.

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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "q4_k_18944x3584: decode matvec B=1 + quantise + MMQ M=512"
METRIC = "Q-matvec HBM GB/s (% of peak); prefill MMQ int8 TOPS (% of tensor peak)"
QTYPE, N, K, B, M = 12, 18944, 3584, 1, 512
W_SEED, XD_SEED, XA_SEED = 102, 202, 204
ROT = 4  # prefill buffer sets rotated between steps (4 x ~220 MB >> L2)
L2_BYTES = 135e6

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


def cpu_baseline(budget_s: float = 12.0):
    """The oracle, as it stands, on a bounded sample of the same workload (1 thread)."""
    import numpy as np

    import oracle
    import synth
    Wb = synth.weights(QTYPE, N, K, W_SEED)
    xd = synth.activations(B, K, XD_SEED)
    xa = synth.activations(M, K, XA_SEED)
    # decode matvec sample: the first `rows` weight rows
    rows, t = 256, 0.0
    while True:
        t0 = time.perf_counter()
        oracle.matvec(QTYPE, Wb, N, K, xd, 0, rows)
        t = time.perf_counter() - t0
        if t > budget_s / 4 or rows >= N:
            break
        rows = min(N, rows * 2)
    mv_bytes = rows * (K // 256) * 144 + B * K * 4 + B * rows * 4
    mv_gbs = mv_bytes / t / 1e9
    # prefill sample: quantise 1 activation row, MMQ against `nrow` weight rows
    qs, sc, _ = oracle.quantize_act(xa[:1])
    nrow, tm = 256, 0.0
    while True:
        t0 = time.perf_counter()
        oracle.mmq(QTYPE, Wb, N, K, qs, sc, mrows=[0], n0=0, n1=nrow)
        tm = time.perf_counter() - t0
        if tm > budget_s / 4 or nrow >= N:
            break
        nrow = min(N, nrow * 2)
    mmq_tops = 2 * 1 * nrow * K / tm / 1e12
    return {"value": mv_gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": (f"decode matvec over weight rows 0..{rows} of {N} (B=1), "
                       f"{t:.2f} s; MMQ of 1 activation row x {nrow} weight rows, {tm:.2f} s; "
                       "single-threaded plain C, fp64 accumulation"),
            "mmq_tops": mmq_tops, "seconds": t + tm}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    cb = cpu_baseline(budget_s=max(2.0, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        pass  # the oracle has no warm state; each step below is timed
    vals = []
    t_all = 0.0
    for _ in range(args.steps):
        c = cpu_baseline(budget_s=max(2.0, 60.0 / max(1, args.steps + args.warmup)))
        vals.append(c["value"])
        t_all += c["seconds"]
    v = statistics.median(vals) if vals else cb["value"]
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000 * t_all / max(1, args.steps), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": cb["sample"]},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "mmq_tops": cb["mmq_tops"]}
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


def profile_calls(kernel: str, calls: int, batch=None):
    """Run `calls` launches of one hot-path kernel on the bench workload and exit: the
    program that ncu captures are taken of (one kernel, few launches, ~0.3 GB on device)."""
    import torch

    import gguf_block_quantized_q4_gb300 as mq
    from gguf_block_quantized_q4_gb300 import build as mqbuild
    import synth
    mqbuild.build()
    mq.init(0)
    Wb = synth.weights(QTYPE, N, K, W_SEED)
    flags = mq.REG_NO_MMQ_PLANE if kernel == "matvec" else mq.REG_DEFAULT
    W = mq.register_weight(QTYPE, Wb, N, K, flags)
    if kernel == "matvec":
        nb = batch or B
        x = torch.from_numpy(synth.activations(nb, K, XD_SEED)).cuda()
        y = torch.empty((nb, N), device="cuda")
        for _ in range(calls):
            mq.matvec(W, x, y)
    else:
        x = torch.from_numpy(synth.activations(M, K, XA_SEED)).cuda()
        xq = mq.quantize_act(x)
        y = torch.empty((M, N), device="cuda")
        for _ in range(calls):
            if kernel == "quantize":
                mq.quantize_act(x, xq)
            else:
                mq.mmq(W, xq, M, y)
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


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mq", choices=["mq", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel", choices=["matvec", "quantize", "mmq"],
                    help="profiling mode: only run --calls launches of this kernel")
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--batch", type=int, choices=range(1, 9), default=None,
                    help="profiling mode, matvec: batch rows (default: the bench's decode batch)")
    ap.add_argument("--chain", type=int, default=0,
                    help="time a decode chain of this many small matvecs, eager and graphed")
    ap.add_argument("--ffn-gu", action="store_true",
                    help="time the fused gate/up matvec and MMQ against two plain calls")
    args = ap.parse_args()
    if args.kernel:
        return profile_calls(args.kernel, args.calls, args.batch)
    if args.chain:
        return chain_timing(args.chain)
    if args.ffn_gu:
        return ffn_gu_timing()
    if args.impl == "reference":
        return run_reference(args)
    args.warmup = max(args.warmup, 3)

    import numpy as np
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

    Wb = synth.weights(QTYPE, N, K, W_SEED)
    # decode: RMV weight copies, > 3x L2 together, so back-to-back calls read HBM
    rmv = int(np.ceil(3 * L2_BYTES / len(Wb)))
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
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        e0.record()
        g_steps.replay()
        e1.record()
        torch.cuda.synchronize()
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

    hbm, bf16, peak_src = peaks()
    mv_gbs = MV_BYTES / (t_mv * 1e-3) / 1e9
    q_gbs = Q_BYTES / (t_q * 1e-3) / 1e9
    mm_tops = MMQ_OPS / (t_mm * 1e-3) / 1e12
    csrc = os.path.join(ROOT, "gguf_block_quantized_q4_gb300", "csrc")
    kern = {
        "matvec": {"kernel": "matvec_kernel<Q4_K,NT=1>", "bound": "hbm", "achieved": mv_gbs,
                   "peak": hbm, "unit": "GB/s", "frac": mv_gbs / hbm,
                   "traffic": traffic_for("matvec_q4_k_b1", os.path.join(csrc, "matvec.cu")),
                   "ms": t_mv, "algorithmic_bytes": MV_BYTES},
        "quantize": {"kernel": "quantize_act_kernel", "bound": "hbm", "achieved": q_gbs,
                     "peak": hbm, "unit": "GB/s", "frac": q_gbs / hbm,
                     "traffic": traffic_for("quantize_m512", [os.path.join(csrc, "quantize.cu"),
                                                              os.path.join(csrc, "quant_row.cuh")]),
                     "ms": t_q, "algorithmic_bytes": Q_BYTES},
        "mmq": {"kernel": "mmq_tc_kernel<Q4_K>", "bound": "tensor", "achieved": mm_tops,
                "peak": bf16, "unit": "TFLOP/s", "frac": mm_tops / bf16,
                "traffic": traffic_for("mmq_q4_k_m512", os.path.join(csrc, "mmq.cu")),
                "ms": t_mm, "algorithmic_ops": MMQ_OPS},
    }
    dom = max(kern, key=lambda k: kern[k]["ms"])
    roof = {k: kern[dom][k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic")}
    roof["kernel"] = kern[dom]["kernel"]
    roof["peak_source"] = (f"{peak_src} ({'hbm_gbs' if roof['bound'] == 'hbm' else 'bf16_tflops'}"
                           " burst; f16 runs at the bf16 rate)")
    e2e_mv = MV_BYTES / (te_mv * 1e-3) / 1e9
    e2e_mm = MMQ_OPS / (te_mm * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": whole_job(mv_gbs, ws), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16xf16->f32",
        "data": "synthetic (seeded, Qwen2.5-7B FFN-shaped Q4_K weights, N(0,1) activations)",
        "config": {"workload": WORKLOAD, "N": N, "K": K, "decode_B": B, "prefill_M": M,
                   "l2": (f"inputs larger than L2: {rmv} decode weight copies rotated; each timed "
                          f"step's prefill moves ~180 MB between decode calls"),
                   "timing": ("steps: one CUDA graph of K steps; per-kernel: graph replays of "
                              "back-to-back calls on rotating buffers, median of 5"),
                   "parallelism": f"replicas x{ws}"},
        "matvec_gbs": whole_job(mv_gbs, ws), "matvec_frac_of_hbm": mv_gbs / hbm,
        "matvec_frac_of_8tbs": mv_gbs / 8000.0,
        "mmq_tops": whole_job(mm_tops, ws), "mmq_frac_of_f16_peak": mm_tops / bf16,
        "quantize_gbs": whole_job(q_gbs, ws),
        "roofline": roof, "kernels": kern,
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
                        "reads x from host memory, MMQ, D2H copy of y), device time per step "
                        "between events, medians"},
        "gpu_launches": 3 * args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(line))
    for w in Wd + Wp:
        w.free()
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
