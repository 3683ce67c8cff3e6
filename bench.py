#!/usr/bin/env python3
"""Benchmark of the quantized GEMV/GEMM hot path on GB300; prints ONE JSON line.

Headline workload (the metric "quant GEMV weight GB/s"): the decode GEMV,
M = 14336, K = 4096, N = 1, fp32 x ~ N(0,1), in Q8_0 and Q4_0. One step = one
pass of the decode hot path over one activation vector: qgemv(Q8_0) then
qgemv(Q4_0), dequantization fused. value = weight bytes streamed per second,
summed over all ranks (each rank runs an independent replica: the path does not
shard across GPUs, so N > 1 is "replicas only").

Timing: W warm-up steps, then exactly K steps bracketed by a barrier and a
device synchronize, timed with CUDA events on the launching stream; each step
is one CUDA-graph replay (the kernels are a few microseconds, shorter than a
Python launch). L2 is defeated by rotating through weight copies totalling
more than 3x the L2 size. Clocks are sampled with nvidia-smi during the timed
region. The per-kernel roofline uses each kernel's average duration from a
graph of back-to-back launches timed in the same run.

--impl reference times the CPU oracle (tests' reference implementation) on
the host cores for the same workload and metric.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quant GEMV weight GB/s (% of HBM peak); quant GEMM TFLOP/s per kind"
UNIT = "GB/s"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50000)
    ap.add_argument("--warmup", type=int, default=500)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-secondary", action="store_true", help="skip the per-kind GEMM/MoE/dequant table")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", default=None,
                    help="run one workload --reps times, untimed, and exit (a target for ncu): "
                         "gemv:<kind> (decode GEMV), gemm:<kind> (prefill GEMM of the kind's workload), "
                         "moe:<gate_up|down>:<T>, dequant:<kind>")
    ap.add_argument("--reps", type=int, default=3)
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK if k in d}, "measured"
    return dict(FALLBACK), "fallback"


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------
# distributed plumbing (replicas)
# ---------------------------------------------------------------------------
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = False

    def init(self, backend="nccl"):
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend)
            self.pg = True

    def barrier(self):
        if self.pg:
            import torch.distributed as dist
            dist.barrier()

    def max(self, v: float) -> float:
        if not self.pg:
            return v
        import torch
        import torch.distributed as dist
        dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
        t = torch.tensor([v], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            import torch.distributed as dist
            dist.destroy_process_group()


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# CPU oracle timing
# ---------------------------------------------------------------------------
def oracle_decode_rate(kinds, M, K, budget_s: float, threads: int):
    """Weight GB/s of the oracle on the decode workload (full M rows per kind)."""
    import oracle
    from gemv_mul_mm_gb300 import synth
    orc = oracle.load()
    c = synth.DECODE
    data = [(k, synth.workload_weights(c, k), synth.workload_x(c, k)) for k in kinds]
    wbytes = sum(w.size for _, w, _ in data)
    steps, t0 = 0, time.perf_counter()
    while True:
        for k, w, x in data:
            orc.gemm(k, w, M, K, x, 1, nthreads=threads)
        steps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return wbytes * steps / el / 1e9, steps, el, wbytes


def run_reference(a):
    d = Dist()
    if d.world > 1:
        d.init("gloo")
        if d.rank != 0:
            d.close()
            return
    from gemv_mul_mm_gb300 import synth
    import oracle
    c = synth.DECODE
    kinds, M, K = c["kinds"], c["M"], c["K"]
    threads = host_cores()
    orc = oracle.load()
    data = [(k, synth.workload_weights(c, k), synth.workload_x(c, k)) for k in kinds]
    rb = {k: synth.row_bytes(k, K) for k in kinds}

    def step(r0, rows):
        # one bounded sample of the decode pass: `rows` weight rows of each kind
        for k, w, x in data:
            orc.gemm(k, w[r0 * rb[k]:(r0 + rows) * rb[k]], rows, K, x, 1, nthreads=threads)

    t0 = time.perf_counter()
    step(0, M)
    t_full = time.perf_counter() - t0
    # size the sample so K steps take about a minute
    rows = int(min(M, max(32, M * (60.0 / max(1, a.steps)) / max(t_full, 1e-6))))
    for i in range(max(0, a.warmup)):
        step((i * rows) % (M - rows + 1), rows)
    t0 = time.perf_counter()
    for i in range(a.steps):
        step((i * rows) % (M - rows + 1), rows)
    el = time.perf_counter() - t0
    n_done = a.steps
    wbytes = sum(rows * rb[k] for k in kinds)
    value = wbytes * n_done / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": a.gpus, "steps": n_done, "warmup": a.warmup, "ms_per_step": round(el / n_done * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded splitmix64; shapes/distributions of the decode GEMV workload)",
        "config": {"workload": "decode GEMV M=14336 K=4096 N=1, Q8_0 + Q4_0, fp32 x",
                   "kinds": list(kinds), "weight_bytes_per_step": wbytes, "parallelism": "replicas"},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{rows} of {M} weight rows of each kind per step ({wbytes} weight bytes), "
                                   f"{'OpenMP' if orc.has_openmp else 'single-thread'} over rows"},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    d.close()


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def strip_comments(src: str) -> str:
    """C/C++ source without its comments and blank-line noise: what the
    compiler sees (string and character literals are kept as they are)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(l.rstrip() for l in "".join(out).splitlines() if l.strip())


def src_hash(*names):
    """Hash of the kernel sources as compiled: a change to the comments alone
    leaves it (and the DRAM counters taken under it) valid."""
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "gemv_mul_mm_gb300", "csrc", n), encoding="utf-8") as f:
            h.update(strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def traffic_for(kernel_key: str, srcs, path: str = None):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel source changed since the counters were taken."""
    p = path or os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel_key)
    if not e or e.get("src_sha") != src_hash(*srcs):
        return None
    return e.get("dram_bytes_per_launch")


def graph_of(fn, reps: int, stream):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(reps):
            fn(i)
    return g


def time_graph(g, replays: int, stream):
    """ms for `replays` replays of g on `stream` (CUDAGraph.replay launches on
    the current stream, so the replays run under a stream context)."""
    import torch
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        s.record(stream)
        for _ in range(replays):
            g.replay()
        e.record(stream)
    e.synchronize()
    return s.elapsed_time(e)


TRIALS = 8   # timed trials per figure; trial 0 is discarded (warm-up), best and median of the rest


def bench_graph(fn, copies, stream, reps=20, replays=5):
    """Per-launch ms of `fn` (best, median) over TRIALS trials of `replays`
    replays of one CUDA graph of `reps` launches, trial 0 discarded. The first
    call runs outside capture (workspace growth)."""
    import torch
    with torch.cuda.stream(stream):
        fn(0)
    torch.cuda.synchronize()
    g = graph_of(lambda i: fn(i % copies), reps, stream)
    t = [time_graph(g, replays, stream) / (reps * replays) for _ in range(TRIALS)][1:]
    return min(t), statistics.median(t)


def _us(best_med):
    return {"us": round(best_med[0] * 1e3, 3), "us_median": round(best_med[1] * 1e3, 3)}


def secondary_table(qmm, synth, l2_bytes, stream, pk):
    """Per-kind decode GEMV GB/s, GEMM TFLOP/s, MoE and dequant GB/s (one GPU,
    outside the headline's timed region). Returns the table and the outputs
    the CPU-oracle leg checks (host copies, with the inputs that made them)."""
    import numpy as np
    import torch
    out, jobs = {}, []
    sh = stream.cuda_stream

    def rot(host, nbytes):
        copies = max(1, math.ceil(3 * l2_bytes / nbytes))
        return [torch.from_numpy(host).cuda() for _ in range(copies)], copies

    # tiny Q4_0 qgemm (latency bound)
    c = synth.TINY
    wh, xh = synth.workload_weights(c, "Q4_0"), synth.workload_x(c, "Q4_0")
    w, x = torch.from_numpy(wh).cuda(), torch.from_numpy(xh).cuda()
    y = torch.empty((c["N"], c["M"]), device="cuda")
    bm = bench_graph(lambda i: qmm.qgemm("Q4_0", w, x, c["M"], c["K"], c["N"], Y=y, stream=sh), 1, stream)
    out["tiny_q4_0_qgemm"] = dict(_us(bm), path=qmm.last_path(),
                                  tflops=round(2 * c["M"] * c["K"] * c["N"] / (bm[0] * 1e-3) / 1e12, 4))
    torch.cuda.synchronize()
    jobs.append(dict(what="gemm_full", tag="tiny_q4_0_qgemm", kind="Q4_0", w=wh, x=xh, M=c["M"], K=c["K"],
                     N=c["N"], got=y.cpu().numpy()))

    # decode GEMV of every kind on the decode shape (fp32 x)
    c = synth.DECODE
    M, K = c["M"], c["K"]
    gemv = {}
    for kind in synth.KINDS:
        try:
            wh = (synth.workload_weights(c, kind) if kind in c["kinds"]
                  else synth.quant_weights(kind, M, K, synth.config_seed(1, kind)))
            xh = synth.workload_x(c, kind)
            ws, copies = rot(wh, wh.size)
            x = torch.from_numpy(xh).cuda()
            y = torch.empty(M, device="cuda")
            bm = bench_graph(lambda i: qmm.qgemv(kind, ws[i], x, M, K, y=y, stream=sh, weights_const=True),
                             copies, stream, reps=max(copies, 20))
            alg = wh.size + 4 * K + 4 * M
            gemv[kind] = dict(M=M, K=K, **_us(bm), path=qmm.last_path(),
                              weight_gbs=round(wh.size / (bm[0] * 1e-3) / 1e9, 1),
                              frac_of_hbm=round(alg / (bm[0] * 1e-3) / 1e9 / pk["hbm_gbs"], 4))
            torch.cuda.synchronize()
            jobs.append(dict(what="gemm_full", tag=f"gemv_{kind}", kind=kind, w=wh, x=xh, M=M, K=K, N=1,
                             got=y.cpu().numpy().reshape(1, M)))
            del ws
        except Exception as e:   # a failure here must not cost the bench line
            gemv[kind] = {"error": f"{type(e).__name__}: {e}"[:200]}
    out["gemv"] = gemv

    # load-time repacked layout (Q8_0, Q4_0): the decode shape, and a shape
    # with few rows (M 2048, K 14336: 64 row groups on the SMs) where the
    # reduction over K is split; the native streaming GEMV beside it
    rep = {}
    for kind in ("Q8_0", "Q4_0"):
        for (M2, K2) in ((c["M"], c["K"]), (2048, 14336)):
            try:
                wh = synth.quant_weights(kind, M2, K2, synth.config_seed(1, kind) + M2)
                xh = synth.activations(1, K2, 17 + M2, "f32")
                ws, copies = rot(wh, wh.size)
                rs = [qmm.qrepack(kind, w_, M2, K2) for w_ in ws]
                x = torch.from_numpy(xh).cuda()
                y = torch.empty(M2, device="cuda")
                row = {"M": M2, "K": K2}
                for name, fn in (("native", lambda i: qmm.qgemv(kind, ws[i], x, M2, K2, y=y, stream=sh,
                                                                 weights_const=True)),
                                 ("repacked", lambda i: qmm.qgemm_repacked(kind, rs[i], x, M2, K2, 1, Y=y, stream=sh,
                                                                           weights_const=True))):
                    bm = bench_graph(fn, copies, stream, reps=max(copies, 20))
                    alg = wh.size + 4 * K2 + 4 * M2
                    row[name] = dict(**_us(bm), weight_gbs=round(wh.size / (bm[0] * 1e-3) / 1e9, 1),
                                     frac_of_hbm=round(alg / (bm[0] * 1e-3) / 1e9 / pk["hbm_gbs"], 4))
                torch.cuda.synchronize()
                jobs.append(dict(what="gemm_full", tag=f"repacked_{kind}_M{M2}", kind=kind, w=wh, x=xh, M=M2, K=K2,
                                 N=1, got=y.cpu().numpy().reshape(1, M2)))
                rep[f"{kind}_M{M2}_K{K2}"] = row
                del ws, rs
            except Exception as e:
                rep[f"{kind}_M{M2}_K{K2}"] = {"error": f"{type(e).__name__}: {e}"[:200]}
    out["repacked_gemv"] = rep

    deq = {}

    def dequant_row(kind, ws, copies, M, K, wh):
        # bit-exact dequant to fp32: the weight bytes read plus 4 * M * K written
        try:
            o = torch.empty((M, K), device="cuda")
            bm = bench_graph(lambda i: qmm.qdequant(kind, ws[i], M, K, out=o, stream=sh), copies, stream,
                             reps=max(copies, 5), replays=3)
            byt = ws[0].numel() + 4 * M * K
            deq[kind] = dict(M=M, K=K, **_us(bm), gbs=round(byt / (bm[0] * 1e-3) / 1e9, 1),
                             frac_of_hbm=round(byt / (bm[0] * 1e-3) / 1e9 / pk["hbm_gbs"], 4))
            torch.cuda.synchronize()
            rows = np.unique(np.concatenate([[0, M - 1], np.random.default_rng(5).integers(0, M, 30)]))
            jobs.append(dict(what="dequant_rows", tag=f"dequant_{kind}", kind=kind, w=wh, M=M, K=K, rows=rows,
                             got=o[torch.from_numpy(rows).cuda()].cpu().numpy()))
            del o
        except Exception as e:
            deq[kind] = {"error": f"{type(e).__name__}: {e}"[:200]}

    # prefill GEMMs (and the dequant of the same tensors)
    gem = {}
    for cfg in (synth.KQUANT, synth.CODEBOOK, synth.LEGACY1):
        M, K, N = cfg["M"], cfg["K"], cfg["N"]
        xh = synth.workload_x(cfg, cfg["kinds"][0])
        X = torch.from_numpy(xh).cuda()
        Y = torch.empty((N, M), device="cuda")
        for kind in cfg["kinds"]:
            try:
                wh = synth.workload_weights(cfg, kind)
                ws, copies = rot(wh, wh.size)
                bm = bench_graph(lambda i: qmm.qgemm(kind, ws[i], X, M, K, N, Y=Y, stream=sh), copies, stream,
                                 reps=max(copies, 6), replays=3)
                tf = 2 * M * K * N / (bm[0] * 1e-3) / 1e12
                gem[kind] = dict(M=M, K=K, N=N, **_us(bm), tflops=round(tf, 2),
                                 frac_of_bf16_peak=round(tf / pk["bf16_tflops"], 4), path=qmm.last_path())
                torch.cuda.synchronize()
                jobs.append(dict(what="gemm_sampled", tag=f"gemm_{kind}", kind=kind, w=wh, x=xh, M=M, K=K, N=N,
                                 got=Y.cpu().numpy()))
                dequant_row(kind, ws, copies, M, K, wh)
                del ws
            except Exception as e:
                gem[kind] = {"error": f"{type(e).__name__}: {e}"[:200]}
    out["gemm"] = gem

    # MoE grouped: both projections of the layer
    moe = {}
    for which, T in [(w, T) for w in ("gate_up", "down") for T in synth.MOE["tokens"]]:
        p = synth.moe_problem(T, which)
        W = torch.from_numpy(p["w"]).cuda()
        X = torch.from_numpy(p["x"]).cuda()
        xr = torch.from_numpy(p["x_row"]).cuda()
        eid = torch.from_numpy(p["expert_id"]).cuda()
        Y = torch.empty((p["x_row"].size, p["M"]), device="cuda")
        bm = bench_graph(lambda i: qmm.qgemm_grouped(p["kind"], W, p["stride"], p["n_experts"], X, xr, eid,
                                                     p["M"], p["K"], Y=Y, stream=sh), 1, stream)
        distinct = len(set(p["expert_id"].tolist()))
        gbs = distinct * p["stride"] / (bm[0] * 1e-3) / 1e9
        moe[f"{which}_T{T}"] = dict(**_us(bm), distinct_experts=distinct, weight_gbs=round(gbs, 1),
                                    frac_of_hbm=round(gbs / pk["hbm_gbs"], 4))
        torch.cuda.synchronize()
        jobs.append(dict(what="grouped_sampled", tag=f"moe_{which}_T{T}", p=p, got=Y.cpu().numpy()))
        del W
    out["moe_q4_0"] = moe

    # the whole MoE feed-forward layer (gate_up, SwiGLU, down, top-k combine)
    layer = {}
    for T in synth.MOE["tokens"]:
        try:
            p = synth.moe_layer_problem(T)
            Wg, Wd = torch.from_numpy(p["w_gu"]).cuda(), torch.from_numpy(p["w_down"]).cuda()
            X = torch.from_numpy(p["x"]).cuda()
            ids, wt = torch.from_numpy(p["ids"]).cuda(), torch.from_numpy(p["w"]).cuda()
            Y = torch.empty((T, p["d_model"]), device="cuda")
            ws = torch.empty(qmm.qmoe_ffn_workspace_bytes(T, ids.shape[1], p["d_model"], p["d_ff"]),
                             dtype=torch.uint8, device="cuda")
            bm = bench_graph(lambda i: qmm.qmoe_ffn(p["kind"], Wg, p["gu_stride"], Wd, p["down_stride"],
                                                    p["n_experts"], X, ids, wt, p["d_model"], p["d_ff"], Y=Y,
                                                    workspace=ws, stream=sh), 1, stream)
            distinct = len(set(p["ids"].reshape(-1).tolist()))
            wbytes = distinct * (p["gu_stride"] + p["down_stride"])
            gbs = wbytes / (bm[0] * 1e-3) / 1e9
            layer[f"T{T}"] = dict(**_us(bm), distinct_experts=distinct, weight_bytes=wbytes,
                                  weight_gbs=round(gbs, 1), frac_of_hbm=round(gbs / pk["hbm_gbs"], 4))
            torch.cuda.synchronize()
            jobs.append(dict(what="moe_layer", tag=f"moe_layer_T{T}", p=p, got=Y.cpu().numpy()))
            del Wg, Wd
        except Exception as e:
            layer[f"T{T}"] = {"error": f"{type(e).__name__}: {e}"[:200]}
    out["moe_layer_q4_0"] = layer

    # dequant of the decode-shape kinds (the K-quant and codebook kinds were
    # timed above, beside each GEMM, on their GEMM tensors)
    c = synth.DECODE
    for kind in ("Q8_0", "Q4_0", "Q5_0"):
        wh = (synth.workload_weights(c, kind) if kind in c["kinds"]
              else synth.quant_weights(kind, c["M"], c["K"], synth.config_seed(1, kind)))
        dequant_row(kind, [torch.from_numpy(wh).cuda()], 1, c["M"], c["K"], wh)
    out["dequant"] = {k: deq[k] for k in synth.KINDS if k in deq}
    out["timing"] = (f"per launch, from CUDA graphs of back-to-back launches with rotated weight copies "
                     f"(>= 3x L2); best of {TRIALS - 1} trials after a discarded first one (us), "
                     f"and their median (us_median)")
    return out, jobs


def parity_report(orc, jobs, threads):
    """CPU-oracle leg: the largest |y - y_ref| / tol of each checked output of
    the secondary table (tol = 1e-3 * sum|w x| + 1e-6), and, for dequant,
    whether the sampled rows are bit-identical to the oracle's."""
    import numpy as np
    rep = {}
    for j in jobs:
        try:
            if j["what"] == "gemm_full":
                y, tol = orc.gemm(j["kind"], j["w"], j["M"], j["K"], j["x"], j["N"], nthreads=threads)
                r = float(np.max(np.abs(j["got"] - y) / tol))
                rep[j["tag"]] = {"max_err_over_tol": round(r, 5), "outputs": int(y.size)}
            elif j["what"] == "gemm_sampled":
                N, M = j["got"].shape
                rng = np.random.default_rng(11)
                n = np.concatenate([[0, N - 1], rng.integers(0, N, 600)])
                m = np.concatenate([[0, M - 1], rng.integers(0, M, 600)])
                y, tol = orc.gemm_at(j["kind"], j["w"], j["M"], j["K"], j["x"], n, m)
                r = float(np.max(np.abs(j["got"][n, m] - y) / tol))
                rep[j["tag"]] = {"max_err_over_tol": round(r, 5), "outputs": int(n.size), "sampled": True}
            elif j["what"] == "grouped_sampled":
                p, got = j["p"], j["got"]
                nr, M = got.shape
                rng = np.random.default_rng(13)
                ri = np.concatenate([[0, nr - 1], rng.integers(0, nr, 400)])
                mi = np.concatenate([[0, M - 1], rng.integers(0, M, 400)])
                y, tol = orc.grouped(p["kind"], p["w"], p["stride"], p["n_experts"], p["x"], p["x_row"],
                                     p["expert_id"], p["M"], p["K"], r_idx=ri, m_idx=mi)
                r = float(np.max(np.abs(got[ri, mi] - y) / tol))
                rep[j["tag"]] = {"max_err_over_tol": round(r, 5), "outputs": int(ri.size), "sampled": True}
            elif j["what"] == "moe_layer":
                p = j["p"]
                y, tol = orc.moe_ffn(p["kind"], p["w_gu"], p["gu_stride"], p["w_down"], p["down_stride"],
                                     p["n_experts"], p["x"], p["ids"], p["w"], p["d_model"], p["d_ff"],
                                     nthreads=threads)
                r = float(np.max(np.abs(j["got"] - y) / tol))
                rep[j["tag"]] = {"max_err_over_tol": round(r, 5), "outputs": int(y.size)}
            elif j["what"] == "dequant_rows":
                rb = j["w"].size // j["M"]
                bad = 0
                for i, r0 in enumerate(j["rows"]):
                    want = orc.dequant(j["kind"], j["w"][r0 * rb:(r0 + 1) * rb], 1, j["K"])[0]
                    g = j["got"][i]
                    diff = (g.view(np.uint32) != want.view(np.uint32)) & ~(np.isnan(g) & np.isnan(want))
                    bad += int(diff.sum())
                rep[j["tag"]] = {"bit_exact": bad == 0, "rows": int(len(j["rows"]))}
        except Exception as e:
            rep[j["tag"]] = {"error": f"{type(e).__name__}: {e}"[:200]}
    return rep


def run_ours(a):
    import numpy as np
    import torch

    d = Dist()
    d.init("nccl")
    torch.cuda.set_device(d.local)
    import __graft_entry__
    __graft_entry__.build()
    from gemv_mul_mm_gb300 import qmm, synth

    pk, pk_src = peaks()
    c = synth.DECODE
    kinds, M, K = c["kinds"], c["M"], c["K"]
    props = torch.cuda.get_device_properties(d.local)
    l2 = int(getattr(props, "L2_cache_size", 126 * 1024 * 1024))
    stream = torch.cuda.Stream()
    sh = stream.cuda_stream

    host_w = {k: synth.workload_weights(c, k) for k in kinds}
    host_x = {k: synth.workload_x(c, k) for k in kinds}
    wbytes = {k: host_w[k].size for k in kinds}
    step_bytes = sum(wbytes.values())
    copies = max(2, math.ceil(3 * l2 / step_bytes))
    with torch.cuda.stream(stream):
        W = {k: [torch.from_numpy(host_w[k]).cuda() for _ in range(copies)] for k in kinds}
        X = {k: torch.from_numpy(host_x[k]).cuda() for k in kinds}
        Y = {k: torch.empty(M, device="cuda") for k in kinds}
    torch.cuda.synchronize()

    def one_step(i):
        j = i % copies
        for k in kinds:
            qmm.qgemv(k, W[k][j], X[k], M, K, y=Y[k], stream=sh, weights_const=True)

    # Steps are replayed from CUDA graphs of R consecutive steps (rotating the
    # weight copies), plus one graph for the remainder, so exactly K steps run.
    R = copies * max(1, 40 // copies)
    g_main = graph_of(one_step, R, stream)
    rem = a.steps % R
    g_rem = graph_of(one_step, rem, stream) if rem else None
    time_graph(g_main, max(1, -(-max(3, a.warmup) // R)), stream)   # >= W warm-up steps
    if g_rem is not None:
        # a graph's first launch uploads it: keep that out of the timed region
        # (a short run may time the remainder graph alone)
        time_graph(g_rem, 2, stream)

    clocks = Clocks(d.local)
    ev_s, ev_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    n0 = qmm.launch_count()
    with torch.cuda.stream(stream):
        ev_s.record(stream)
        for _ in range(a.steps // R):
            g_main.replay()
        if g_rem is not None:
            g_rem.replay()
        ev_e.record(stream)
    ev_e.synchronize()
    torch.cuda.synchronize()
    d.barrier()
    # graph replays launch their kernels without passing through the library's
    # launch counter: each step holds len(kinds) of our kernels.
    launches = (qmm.launch_count() - n0) + a.steps * len(kinds)
    clk = clocks.stop()
    ms_total = d.max(ev_s.elapsed_time(ev_e))
    ms_step = ms_total / a.steps
    value = d.world * step_bytes * a.steps / (ms_total * 1e-3) / 1e9

    # per-kernel durations: graphs of back-to-back launches of one kind, on
    # the stream the kernels run on, best of TRIALS - 1 trials (and median)
    per = {}
    R = 4 * copies
    for k in kinds:
        g = graph_of(lambda i, k=k: qmm.qgemv(k, W[k][i % copies], X[k], M, K, y=Y[k], stream=sh,
                                              weights_const=True), R, stream)
        time_graph(g, 2, stream)
        rp = max(5, 2000 // R)
        t = [time_graph(g, rp, stream) / (R * rp) for _ in range(TRIALS)][1:]
        ms, med = min(t), statistics.median(t)
        alg = wbytes[k] + 4 * K + 4 * M
        per[k] = {"us": round(ms * 1e3, 3), "us_median": round(med * 1e3, 3),
                  "weight_gbs": round(wbytes[k] / (ms * 1e-3) / 1e9, 1),
                  "achieved_gbs": round(alg / (ms * 1e-3) / 1e9, 1), "alg_bytes": alg,
                  "frac": round(alg / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4)}
    dom = max(kinds, key=lambda k: per[k]["us"])
    traffic = traffic_for(f"k_gemv<{dom}>", ["k_gemv.cu", "decode.cuh", "sm100_async.cuh"])
    roofline = {"bound": "hbm", "kernel": f"k_gemv<{dom},1>", "achieved": per[dom]["achieved_gbs"],
                "peak": pk["hbm_gbs"], "peak_source": pk_src, "unit": "GB/s", "frac": per[dom]["frac"],
                "traffic": traffic, "alg_bytes_per_launch": per[dom]["alg_bytes"]}

    # end to end through the public API: every step copies the step's
    # activations (both x vectors, one pinned host buffer) to the device, runs
    # both GEMVs and copies both outputs back to one pinned host buffer; the
    # steps are replayed from a CUDA graph (a decode loop's usual form), so the
    # host's per-call cost stays out of the GPU's way
    hx = torch.from_numpy(np.stack([host_x[k].reshape(-1) for k in kinds])).pin_memory()
    hy = torch.empty((len(kinds), M), dtype=torch.float32).pin_memory()
    Xe = torch.empty((len(kinds), K), dtype=torch.float32, device="cuda")
    Ye = torch.empty((len(kinds), M), dtype=torch.float32, device="cuda")

    def e2e_step(i):
        j = i % copies
        Xe.copy_(hx, non_blocking=True)
        for ki, k in enumerate(kinds):
            qmm.qgemv(k, W[k][j], Xe[ki], M, K, y=Ye[ki], stream=sh, weights_const=True)
        hy.copy_(Ye, non_blocking=True)

    RE = copies * max(1, 40 // copies)
    with torch.cuda.stream(stream):
        e2e_step(0)
    torch.cuda.synchronize()
    g_e2e = graph_of(e2e_step, RE, stream)
    time_graph(g_e2e, 2, stream)
    n_rep = max(1, min(a.steps, 4000) // RE)
    n_e2e = n_rep * RE
    e2e_ms = d.max(time_graph(g_e2e, n_rep, stream))
    e2e = {"value": round(d.world * step_bytes * n_e2e / (e2e_ms * 1e-3) / 1e9, 1), "unit": UNIT,
           "h2d_bytes_per_step": sum(4 * K for _ in kinds), "d2h_bytes_per_step": sum(4 * M for _ in kinds),
           "steps": n_e2e, "ms_per_step": round(e2e_ms / n_e2e, 4),
           "how": "CUDA-graph replay of steps; each step: one H2D of both x from pinned memory, qgemv x2, "
                  "one D2H of both y to pinned memory"}

    sec, jobs = None, []
    if d.rank == 0 and d.world == 1 and not a.no_secondary:
        sec, jobs = secondary_table(qmm, synth, l2, stream, pk)

    # CPU-oracle leg: the oracle timed on the host cores (cpu_baseline), and
    # the same oracle's check of every output the secondary table produced
    cpu, parity = None, None
    if d.rank == 0 and d.world == 1 and not a.no_cpu_baseline:
        import oracle
        cores = host_cores()
        rate, steps, el, wb = oracle_decode_rate(kinds, M, K, 10.0, cores)
        cpu = {"value": round(rate, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{steps} full decode steps ({wb} weight bytes each) in {el:.1f} s"}
        try:   # the same oracle on one core, for scale
            r1, s1, e1, _ = oracle_decode_rate(kinds, M, K, 4.0, 1)
            cpu["single_thread"] = {"value": round(r1, 3), "unit": UNIT, "cores": 1,
                                    "sample": f"{s1} full decode steps in {e1:.1f} s"}
        except Exception as e:
            cpu["single_thread"] = {"error": f"{type(e).__name__}: {e}"[:200]}
        if jobs:
            parity = parity_report(oracle.load(), jobs, cores)

    if d.rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": d.world,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded splitmix64; shapes and distributions of the pages' decode workload)",
            "config": {"workload": "decode GEMV M=14336 K=4096 N=1, Q8_0 + Q4_0, fp32 x (one step = both)",
                       "weight_bytes_per_step": step_bytes, "parallelism": "replicas",
                       "l2_defeat": f"rotating {copies} weight copies ({copies * step_bytes / 1e6:.0f} MB > 3x L2 "
                                    f"{l2 / 1e6:.0f} MB)", "timing": "CUDA-graph replay per step, CUDA events",
                       "weight_prefetch": "on (weights constant; programmatic dependent launch)"},
            "per_kind": per, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches, "clocks": clk, "secondary": sec, "parity": parity,
        }
        print(json.dumps(line), flush=True)
    d.close()


def run_case(a):
    """One workload, --reps back-to-back calls on one stream, no timing: the
    launch an ncu capture selects with -k / -c."""
    import torch
    torch.cuda.set_device(0)
    import __graft_entry__
    __graft_entry__.build()
    from gemv_mul_mm_gb300 import qmm, synth
    what, _, arg = a.case.partition(":")
    if what == "gemv":
        c = synth.DECODE
        W = torch.from_numpy(synth.workload_weights(c, arg)).cuda()
        x = torch.from_numpy(synth.workload_x(c, arg)).cuda()
        fn = lambda: qmm.qgemv(arg, W, x, c["M"], c["K"], weights_const=True)
    elif what == "gemm":
        c = next(cf for cf in (synth.KQUANT, synth.CODEBOOK, synth.LEGACY1) if arg in cf["kinds"])
        W = torch.from_numpy(synth.workload_weights(c, arg)).cuda()
        X = torch.from_numpy(synth.workload_x(c, arg)).cuda()
        fn = lambda: qmm.qgemm(arg, W, X, c["M"], c["K"], c["N"])
    elif what == "moe":
        which, _, T = arg.partition(":")
        p = synth.moe_problem(int(T), which)
        W, X = torch.from_numpy(p["w"]).cuda(), torch.from_numpy(p["x"]).cuda()
        xr, eid = torch.from_numpy(p["x_row"]).cuda(), torch.from_numpy(p["expert_id"]).cuda()
        fn = lambda: qmm.qgemm_grouped(p["kind"], W, p["stride"], p["n_experts"], X, xr, eid, p["M"], p["K"])
    elif what == "dequant":
        c = next(cf for cf in (synth.DECODE, synth.KQUANT, synth.CODEBOOK, synth.LEGACY1) if arg in cf["kinds"])
        W = torch.from_numpy(synth.workload_weights(c, arg)).cuda()
        fn = lambda: qmm.qdequant(arg, W, c["M"], c["K"])
    else:
        raise SystemExit(f"unknown case {a.case!r}")
    for _ in range(a.reps):
        fn()
    torch.cuda.synchronize()
    rc = qmm.check_device_error()
    print(json.dumps({"case": a.case, "reps": a.reps, "device_error": rc}))
    if rc:
        raise SystemExit(1)


def main():
    a = parse()
    if a.case:
        run_case(a)
        return
    if a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)


if __name__ == "__main__":
    main()
