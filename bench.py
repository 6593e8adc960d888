#!/usr/bin/env python
"""Throughput of the fused cascaded reductions on GB300.

Headline (one JSON line on rank 0): split-KV decode attention, B=32, H=32,
L=32768, D=128, bf16 K/V (16 GiB), S segments -- one step is
rf_attn_decode_split + rf_state_merge over the whole batch; value = K/V bytes
per second (GB/s).  The inputs (16 GiB) are far larger than the 129 MB L2, so
no flush is needed between steps.

The same line carries:
  roofline      the decode-split kernel's algorithmic bytes per launch over its
                CUDA-event duration, against the measured HBM copy bandwidth;
                traffic = ncu DRAM bytes per launch (profiles/traffic.json, only
                while the kernel source is unchanged since the capture);
  e2e           the same metric through the public API with pinned HOST
                buffers: host->device copy of q, K, V and device->host read of
                the output inside the timed region;
  cpu_baseline  the float64 CPU oracle on a bounded sample of rows of the same
                workload, on the host's cores (one single-threaded worker per
                core);
  clocks        nvidia-smi samples taken during the timed region;
  pages_claim   the speedup the pages claim for their own system, with the
                hardware they name (context, not a target);
  paths         the fused one-launch decode step on the same inputs, the
                other cascades (single-row fp32 decode, both routing
                shapes, quantisation, FP8 GEMM, causal prefill, MLA decode,
                the single-row cascades at every fusion level, LayerNorm and
                RMSNorm) and the incremental vs non-incremental decode
                ablations, each timed on its own with its roofline.

``--impl reference`` times the CPU oracle alone as the reference arm (same
metric, unit and config; each step is a bounded sample of rows).

Multi-GPU (torchrun): every rank runs the whole decode batch on its own GPU
(independent replicas, no collective: the rows are independent), the time is
the max over ranks and value = all ranks' bytes / that time.
"""

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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused cascade throughput: decode KV GB/s, prefill TFLOP/s, % of GB300 roofline"
DECODE = dict(B=32, H=32, L=32768, D=128)
L2_BYTES = 129 * 1024 * 1024


# ----------------------------------------------------------------- helpers --

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# What the pages claim for their own system, as context beside the measured
# numbers (not a target: the pages give speedups, no absolute throughput).
PAGES_CLAIM = {
    "speedup": "2x to 5x over state-of-the-art AI compilers (TVM, PyTorch Dynamo)",
    "hardware": "NVIDIA A10 and H800",
    "workloads": "multi-head attention, multi-latent attention, MoE routing, FP8 quantise + GEMM",
    "source": "bookshelf explainer 'RedFuser: An Automatic Operator Fusion Framework for Cascaded "
              "Reductions on AI Accelerators', section 'If you remember only three things', item 3",
}


def file_sha(path):
    return hashlib.sha256(open(path, "rb").read()).hexdigest()


def ncu_traffic(kernel):
    """DRAM bytes per launch recorded from an ncu capture, if the kernel's
    source has not changed since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(kernel)
    if not rec:
        return None
    src = os.path.join(ROOT, rec["source"])
    if not os.path.exists(src) or file_sha(src) != rec["source_sha256"]:
        return None
    return rec["dram_bytes_per_launch"]


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during a timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.15)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        self.proc.wait()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), smax=float(f[2]), power=float(f[3]),
                                 hw=f[5], hwt=f[6], swt=f[7], swp=f[8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        busy = [r for r in rows if r["power"] > 300] or rows
        return {"sm_mhz": statistics.median(r["sm"] for r in busy),
                "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(r["power"] for r in rows)}


# ------------------------------------------------------ CPU oracle baseline --

_W = {}


def _oracle_worker_init(q_bits, k_bits, v_bits, scale):
    _W.update(q=q_bits, k=k_bits, v=v_bits, scale=scale)


def _oracle_decode_row(_):
    from oracle import attention, bf16
    out, m, l = attention.softmax_v_rows(bf16.decode(_W["q"]), bf16.decode(_W["k"]),
                                         bf16.decode(_W["v"]), _W["scale"])
    return float(out[0, 0])


class OracleDecodePool:
    """One single-threaded float64 oracle worker per host core, each holding
    one row (q, K, V) of the decode workload, drawn with the workload's
    recipe (seed 2) on the CPU."""

    def __init__(self, cores=None):
        import multiprocessing as mp
        import torch
        import synthetic_inputs as si
        self.cores = cores or len(os.sched_getaffinity(0))
        L, D = DECODE["L"], DECODE["D"]
        q, K, V = si.decode_inputs(1, L, D, torch.bfloat16, seed=2)
        bits = [t.view(torch.int16).numpy().copy() for t in (q, K, V)]
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"
        ctx = mp.get_context("spawn")
        self.pool = ctx.Pool(self.cores, initializer=_oracle_worker_init,
                             initargs=(*bits, si.decode_scale(D)))
        self.row_bytes = 2 * L * D * 2
        self.pool.map(_oracle_decode_row, range(self.cores))      # warm the workers

    def run(self, rows):
        t = time.perf_counter()
        self.pool.map(_oracle_decode_row, range(rows), chunksize=1)
        return time.perf_counter() - t

    def close(self):
        self.pool.close()
        self.pool.join()


def _oracle_path_samples(budget_s):
    """Runs in a spawned single-threaded worker: the float64 oracle of each
    cascade on a bounded sample of its workload, timed.  Returns
    {path: (units_done, unit, seconds, sample description)}."""
    import torch
    import synthetic_inputs as si
    from oracle import attention, bf16, fp8, mla, routing

    def timed(fn):
        n, t0 = 0, time.perf_counter()
        while True:
            fn()
            n += 1
            dt = time.perf_counter() - t0
            if dt >= budget_s:
                return n, dt

    res = {}
    q, K, V = (t.double().numpy() for t in si.decode_inputs(1, 4096, 64, torch.float32, seed=1))
    n, dt = timed(lambda: attention.softmax_v_rows(q, K, V, 0.125))
    res["single_row_decode_f32"] = (n * 2 * 4096 * 64 * 4, "B", dt, "the whole q[64], K, V [4096, 64]")
    for name, tokens in (("route_256", 2048), ("route_64", 8192)):
        cfg = si.FULL[name]
        x = si.routing_logits(tokens, cfg["E"], seed=si.SEEDS[name]).numpy()
        n, dt = timed(lambda: routing.softmax_topk(x, cfg["k"], True))
        res["routing_%dx%d_top%d" % (cfg["T"], cfg["E"], cfg["k"])] = (
            n * tokens * (cfg["E"] * 4 + cfg["k"] * 8), "B", dt,
            f"{tokens} of the {cfg['T']} tokens")
    cfg = si.FULL["quant_gemm"]
    xb, wq, sw = si.quant_gemm_inputs(cfg["M"], cfg["K"], cfg["N"], seed=4)
    xs = bf16.decode(xb[:256].view(torch.int16).numpy())
    n, dt = timed(lambda: fp8.absmax_quant(xs))
    res["absmax_quant_e4m3"] = (n * 256 * cfg["K"] * 3, "B", dt, f"256 of the {cfg['M']} rows")
    xq, sx = fp8.absmax_quant(bf16.decode(xb[:32].view(torch.int16).numpy()))
    wqn, swn = wq.numpy(), sw.numpy()
    n, dt = timed(lambda: fp8.scaled_gemm(xq, sx, wqn, swn))
    res["fp8_gemm"] = (n * 2.0 * 32 * cfg["N"] * cfg["K"], "FLOP", dt,
                       f"32 of the {cfg['M']} rows against all of Wq")
    cfg = si.FULL["prefill"]
    Q, Kp, Vp = si.prefill_inputs(1, 1, cfg["N"], cfg["D"], seed=5)
    Q, Kp, Vp = (t[0, 0].double().numpy() for t in (Q, Kp, Vp))
    rows = list(range(cfg["N"] // 2, cfg["N"] // 2 + 16))
    n, dt = timed(lambda: [attention.causal_attention_row(Q[i], Kp, Vp, cfg["D"] ** -0.5, i)
                           for i in rows])
    res["causal_prefill"] = (n * sum(4.0 * cfg["D"] * (i + 1) for i in rows), "FLOP", dt,
                             "16 query rows in the middle of one head (exact causal FLOPs)")
    cfg = si.FULL["mla"]
    qm, Cm = si.mla_inputs(1, cfg["H"], cfg["L"], cfg["Dk"], seed=si.SEEDS["mla"])
    qm, Cm = qm.double().numpy(), Cm.double().numpy()
    n, dt = timed(lambda: mla.mla_decode(qm, Cm, cfg["Dv"], si.mla_scale()))
    res["mla_decode"] = (n * cfg["L"] * cfg["Dk"] * 2, "B", dt,
                         f"one of the {cfg['B']} sequences ({cfg['H']} heads, the whole latent cache)")
    return res


def oracle_path_baselines(budget_s=1.5):
    """The oracle beside each GPU path, in one single-threaded spawned worker."""
    import multiprocessing as mp
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    with mp.get_context("spawn").Pool(1) as pool:
        res = pool.apply(_oracle_path_samples, (budget_s,))
    out = {}
    for path, (units, unit, dt, sample) in res.items():
        if unit == "B":
            out[path] = {"value": round(units / dt / 1e9, 4), "unit": "GB/s"}
        else:
            out[path] = {"value": round(units / dt / 1e12, 6), "unit": "TFLOP/s"}
        out[path].update({"cores": 1, "kind": "oracle", "sample": sample + f", {dt:.1f} s"})
    return out


def cpu_baseline(budget_s=10.0):
    pool = OracleDecodePool()
    rows, elapsed = 0, 0.0
    batch = pool.cores * 4
    while elapsed < budget_s:
        elapsed += pool.run(batch)
        rows += batch
    pool.close()
    return {"value": rows * pool.row_bytes / elapsed / 1e9, "unit": "GB/s", "cores": pool.cores,
            "kind": "oracle",
            "sample": f"{rows} rows of the decode workload (each q [128], K and V [32768, 128] bf16), "
                      f"float64 oracle, {elapsed:.1f} s on {pool.cores} single-threaded workers"}


# -------------------------------------------------------- multi-rank logic --

def max_over_ranks(value, world, device):
    """The largest of every rank's value (all ranks get it); the value itself
    on a single rank."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.item()


def job_gbs(bytes_per_rank_step, world, ms_step):
    """Whole-job throughput in GB/s: every rank processed its own bytes in the
    slowest rank's time."""
    return world * bytes_per_rank_step / (ms_step * 1e-3) / 1e9


# --------------------------------------------------------------- GPU timing --

def _events(torch, n):
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def time_graph(torch, calls, reps, warmup=3):
    """Capture ``calls`` (a list of zero-argument launchers) in one CUDA
    graph; time ``reps`` replays back to back (events between them); return
    the median replay's ms per call."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for c in calls:                       # eager warm-up outside capture
            c()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for c in calls:
            c()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    # one event pair per replay; the median replay, per call
    reps = max(reps, 5)
    ev = _events(torch, reps + 1)
    ev[0].record()
    for i in range(reps):
        g.replay()
        ev[i + 1].record()
    torch.cuda.synchronize()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(reps)]
    return statistics.median(per) / len(calls)


def roofline(bound, achieved, peak, unit, traffic):
    return {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": traffic}


def decode_ablation(torch, rf, peaks, q, K, V, scale, segments=(1, 2, 4, 8, 16, 32, 64),
                    workload=None):
    """Incremental vs non-incremental split-KV decode, for every segment count
    S: time of the segment-state kernel alone."""
    R, L, D = K.shape
    kv_bytes = 2 * K.numel() * K.element_size()
    res = {}
    for S in segments:
        sm = torch.empty(R, S, device="cuda")
        sl = torch.empty(R, S, device="cuda")
        sa = torch.empty(R, S, D, device="cuda")
        row = {}
        for name, fn in (("incremental", rf.rf_attn_decode_split),
                         ("non_incremental", rf.rf_attn_decode_split_twopass)):
            try:
                for _ in range(2):
                    fn(q, K, V, S, scale, sm, sl, sa)
            except rf.RFError as e:
                row[name] = {"unsupported": str(e)}
                continue
            a, b = _events(torch, 2)
            a.record()
            for _ in range(5):
                fn(q, K, V, S, scale, sm, sl, sa)
            b.record()
            torch.cuda.synchronize()
            ms = a.elapsed_time(b) / 5
            gbs = kv_bytes / (ms * 1e-3) / 1e9
            row[name] = {"ms": round(ms, 4), "GB/s": round(gbs, 1),
                         "frac": round(gbs / peaks["hbm_gbs"], 4)}
        res[f"S{S}"] = row
    res["workload"] = workload or (
        "segment-state kernel only, B=32 H=32 L=32768 D=128 bf16; the non-incremental kernel "
        "keeps a segment's scores in shared memory (segments of at most 16384 keys)")
    return res


def decode_ablation_short(torch, rf, peaks):
    """The same comparison on short per-block sequences: 16384 rows of L=512
    keys, D=64 fp32 (BERT-base's head width and sequence length), S = 1..8
    (512 down to 64 keys per block)."""
    import synthetic_inputs as si
    q, K, V = si.decode_inputs(16384, 512, 64, torch.float32, seed=7, device="cuda")
    res = decode_ablation(torch, rf, peaks, q, K, V, si.decode_scale(64), segments=(1, 2, 4, 8),
                          workload="segment-state kernel only, 16384 rows x L=512 keys, D=64 fp32 "
                                   "(BERT-base head width and sequence length); K/V 4.3 GB > L2")
    del q, K, V
    return res


def path_single_row(torch, rf, peaks):
    import synthetic_inputs as si
    cfg = si.FULL["decode_f32"]
    q, K, V = (t.cuda() for t in si.decode_inputs(1, cfg["L"], cfg["D"], torch.float32, seed=1))
    S = 32
    sm = torch.empty(1, S, device="cuda")
    sl = torch.empty(1, S, device="cuda")
    sa = torch.empty(1, S, cfg["D"], device="cuda")
    out = torch.empty(1, cfg["D"], device="cuda")
    scale = si.decode_scale(cfg["D"])

    def call():
        rf.rf_attn_decode_split(q, K, V, S, scale, sm, sl, sa)
        rf.rf_state_merge(sm, sl, sa, out)
    ms = time_graph(torch, [call] * 50, 20)
    counters = torch.zeros(1, dtype=torch.int32, device="cuda")
    fused_sweep = {}
    for Sf in (4, 8, 16, 32, 64):
        smf = torch.empty(1, Sf, device="cuda")
        slf = torch.empty(1, Sf, device="cuda")
        saf = torch.empty(1, Sf, cfg["D"], device="cuda")
        fused = lambda: rf.rf_attn_decode_fused(q, K, V, Sf, scale, smf, slf, saf, counters, out)
        fused_sweep[f"S{Sf}"] = round(time_graph(torch, [fused] * 50, 20) * 1e3, 2)
    best_fused = min(fused_sweep, key=fused_sweep.get)
    ms_fused = fused_sweep[best_fused] * 1e-3
    nbytes = 2 * cfg["L"] * cfg["D"] * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": "single-row decode fp32 q[64] K,V[4096,64], S=32 (latency bound; "
                        "graph of 50 back-to-back calls, inputs L2-resident)",
            "value": round(gbs, 1), "unit": "GB/s", "us_per_call": round(ms * 1e3, 2),
            "fused_us_per_call": round(ms_fused * 1e3, 2),
            "fused_note": f"rf_attn_decode_fused (the merge done by the row's last CTA, one "
                          f"launch), best segment count {best_fused[1:]}",
            "fused_us_by_segments": fused_sweep,
            "roofline": roofline("hbm", gbs, peaks["hbm_gbs"], "GB/s", None)}


def path_routing(torch, rf, peaks, name):
    import synthetic_inputs as si
    cfg = si.FULL[name]
    T, E, k = cfg["T"], cfg["E"], cfg["k"]
    x0 = si.routing_logits(T, E, seed=si.SEEDS[name]).cuda()
    nbytes = T * E * 4 + T * k * 8
    copies = max(2, -(-3 * L2_BYTES // (T * E * 4)))
    xs = [x0.clone() for _ in range(copies)]
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, device="cuda")
    calls = [(lambda x=x: rf.rf_softmax_topk(x, k, True, idx, w)) for x in xs] * 4
    ms = time_graph(torch, calls, 10)
    gbs = nbytes / (ms * 1e-3) / 1e9
    # the floor: one streaming read of the same logits (rf_stream_read), same
    # copies, same graph, same timing
    xor = torch.zeros(1, dtype=torch.int32, device="cuda")
    reads = [(lambda x=x: rf.rf_stream_read(x, xor)) for x in xs] * 4
    ms_floor = time_graph(torch, reads, 10)
    return {"workload": f"routing logits [{T} x {E}] fp32, top-{k}, renormalised; {copies} input "
                        f"copies rotated (> L2) in a CUDA graph",
            "value": round(gbs, 1), "unit": "GB/s", "us_per_call": round(ms * 1e3, 2),
            "read_floor": {"us_per_call": round(ms_floor * 1e3, 2),
                           "GB/s": round(T * E * 4 / (ms_floor * 1e-3) / 1e9, 1),
                           "routing_time_over_floor": round(ms / ms_floor, 3),
                           "how": "rf_stream_read over the same input copies in the same CUDA "
                                  "graph: one 16-byte streaming read of every logit, nothing else"},
            "roofline": roofline("hbm", gbs, peaks["hbm_gbs"], "GB/s", ncu_traffic(f"softmax_topk_{E}"))}


def path_quant(torch, rf, peaks):
    import synthetic_inputs as si
    cfg = si.FULL["quant_gemm"]
    M, K = cfg["M"], cfg["K"]
    x0, _, _ = si.quant_gemm_inputs(M, K, 256, seed=4)
    x0 = x0.cuda()
    copies = 4
    xs = [x0.clone() for _ in range(copies)]
    xq = torch.empty(M, K, dtype=torch.uint8, device="cuda")
    sx = torch.empty(M, device="cuda")
    calls = [(lambda x=x: rf.rf_absmax_quant_e4m3(x, xq, sx)) for x in xs] * 4
    ms = time_graph(torch, calls, 10)
    nbytes = M * K * 2 + M * K + M * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": f"abs-max -> e4m3 quantisation of X [{M} x {K}] bf16; {copies} input copies "
                        f"rotated (> L2) in a CUDA graph",
            "value": round(gbs, 1), "unit": "GB/s", "us_per_call": round(ms * 1e3, 2),
            "roofline": roofline("hbm", gbs, peaks["hbm_gbs"], "GB/s", ncu_traffic("absmax_quant"))}


def path_gemm(torch, rf, peaks):
    import synthetic_inputs as si
    cfg = si.FULL["quant_gemm"]
    M, K, N = cfg["M"], cfg["K"], cfg["N"]
    x, wq, sw = si.quant_gemm_inputs(M, K, N, seed=4)
    x, wq, sw = x.cuda(), wq.cuda(), sw.cuda()
    xq = torch.empty(M, K, dtype=torch.uint8, device="cuda")
    sx = torch.empty(M, device="cuda")
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    try:
        rf.rf_absmax_quant_e4m3(x, xq, sx)
        rf.rf_fp8_gemm_scaled(xq, sx, wq, sw, y)
    except rf.RFError as e:
        return {"skipped": str(e)}
    ms = time_graph(torch, [lambda: rf.rf_fp8_gemm_scaled(xq, sx, wq, sw, y)] * 10, 10)
    ms_both = time_graph(torch, [lambda: rf.rf_absmax_quant_fp8_gemm(x, wq, sw, xq, sx, y)] * 10, 10)
    tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
    fp8_peak = 2.0 * peaks["bf16_tflops"]     # fp8 dense rate is twice bf16's
    # the incremental form of the cascade (one kernel, running abs-max)
    y_inc = torch.empty_like(y)
    sx_inc = torch.empty_like(sx)
    ms_inc = time_graph(torch, [lambda: rf.rf_incremental_quant_fp8_gemm(x, wq, sw, y_inc, sx_inc)] * 10, 10)
    rf.rf_absmax_quant_fp8_gemm(x, wq, sw, xq, sx, y)
    rf.rf_incremental_quant_fp8_gemm(x, wq, sw, y_inc, sx_inc)
    torch.cuda.synchronize()
    # error of both against the exact product of the bf16 X and the (dequantised) weights,
    # on 64 rows, float64
    rows = torch.arange(0, M, M // 64)
    w64 = wq.view(torch.float8_e4m3fn).double() * sw.double()[:, None]
    exact = x[rows].double() @ w64.t()
    nrm = exact.norm().item()
    err_two = (y[rows].double() - exact).norm().item() / nrm
    err_inc = (y_inc[rows].double() - exact).norm().item() / nrm
    tf_inc = 2.0 * M * N * K / (ms_inc * 1e-3) / 1e12
    incremental = {"us_per_call": round(ms_inc * 1e3, 2),
                   "TFLOP/s": round(tf_inc, 1),
                   "us_two_phase_quant_plus_gemm": round(ms_both * 1e3, 2),
                   "rel_error_vs_exact_product": round(err_inc, 6),
                   "rel_error_two_phase": round(err_two, 6),
                   "roofline": roofline("tensor", tf_inc, fp8_peak, "TFLOP/s",
                                        ncu_traffic("fp8_incremental_cluster")),
                   "workload": f"one kernel: bf16 X [{M} x {K}] read in 128-column tiles, running "
                               f"abs-max, e4m3 tiles in shared memory, accumulator rescaled when the "
                               f"scale grows; clusters of CTAs that share a 128-row block quantise "
                               f"one row band each and copy the codes to the others; "
                               f"error = Frobenius norm over 64 rows"}
    return {"incremental_quant_gemm": incremental,
            "workload": f"FP8 GEMM Y[{M} x {N}] = Xq[{M} x {K}] Wq^T, e4m3, fp32 accumulate, bf16 out",
            "value": round(tf, 1), "unit": "TFLOP/s", "us_per_call": round(ms * 1e3, 2),
            "us_quant_plus_gemm": round(ms_both * 1e3, 2),
            "incremental_us_per_call": round(ms_inc * 1e3, 2),
            "roofline": roofline("tensor", tf, fp8_peak, "TFLOP/s", ncu_traffic("fp8_gemm_2sm")),
            "peak_note": "fp8 peak = 2 x measured bf16 burst (nominal fp8/bf16 ratio)"}


def path_prefill(torch, rf, peaks):
    import synthetic_inputs as si
    cfg = si.FULL["prefill"]
    B, H, N, D = cfg["B"], cfg["H"], cfg["N"], cfg["D"]
    q, k, v = si.prefill_inputs(B, H, N, D, seed=5, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(B, H, N, device="cuda")
    try:
        rf.rf_attn_prefill(q, k, v, True, D ** -0.5, out, lse)
    except rf.RFError as e:
        return {"skipped": str(e)}
    ms = time_graph(torch, [lambda: rf.rf_attn_prefill(q, k, v, True, D ** -0.5, out, lse)] * 3, 5)
    flops = 4.0 * B * H * D * N * (N + 1) / 2
    tf = flops / (ms * 1e-3) / 1e12
    return {"workload": f"causal prefill B={B} H={H} N={N} D={D} bf16 (exact causal FLOPs)",
            "value": round(tf, 1), "unit": "TFLOP/s", "ms_per_call": round(ms, 3),
            "roofline": roofline("tensor", tf, peaks["bf16_tflops"], "TFLOP/s", ncu_traffic("prefill"))}


def path_mla(torch, rf, peaks, only_segments=0):
    """Multi-latent attention decode: B=64 sequences x 16 query heads reading
    one shared latent cache each (L=32768 rows of 576 bf16), split into S
    segments and merged.  The 2.4 GB cache is larger than L2."""
    import synthetic_inputs as si
    cfg = si.FULL["mla"]
    B, H, L, Dk, Dv = cfg["B"], cfg["H"], cfg["L"], cfg["Dk"], cfg["Dv"]
    q, C = si.mla_inputs(B, H, L, Dk, seed=si.SEEDS["mla"], device="cuda")
    scale = si.mla_scale()
    cache_bytes = B * L * Dk * 2
    flops = 2.0 * B * H * L * (Dk + Dv)
    res = {"workload": f"MLA decode B={B} H={H} L={L} latent {Dk} (value {Dv}) bf16, fp32 "
                       f"accumulate, bf16 out; latent cache {cache_bytes / 1e9:.2f} GB > L2",
           "unit": "GB/s"}
    sweep = {}
    for S in ((only_segments,) if only_segments else (8, 16, 32, 64)):
        sm = torch.empty(B, H, S, device="cuda")
        sl = torch.empty(B, H, S, device="cuda")
        sa = torch.empty(B, H, S, Dv, device="cuda")
        out = torch.empty(B * H, Dv, device="cuda", dtype=torch.bfloat16)
        lse = torch.empty(B * H, device="cuda")
        split = lambda: rf.rf_mla_decode_split(q, C, S, scale, sm, sl, sa)
        merge = lambda: rf.rf_state_merge(sm.view(B * H, S), sl.view(B * H, S),
                                          sa.view(B * H, S, Dv), out, lse)

        def both():
            split()
            merge()
        ms = time_graph(torch, [both] * 3, 5)
        ms_split = time_graph(torch, [split] * 3, 5)
        state_bytes = B * H * S * (Dv + 2) * 4
        alg = cache_bytes + q.numel() * 2 + state_bytes
        sweep[f"S{S}"] = {"ms": round(ms, 4), "GB/s": round(cache_bytes / (ms * 1e-3) / 1e9, 1),
                          "split_ms": round(ms_split, 4),
                          "split_frac_hbm": round(alg / (ms_split * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                          "TFLOP/s": round(flops / (ms * 1e-3) / 1e12, 1)}
        del sm, sl, sa, out, lse
    best = min(sweep, key=lambda k: sweep[k]["ms"])
    S = int(best[1:])
    b = sweep[best]
    alg = cache_bytes + q.numel() * 2 + B * H * S * (Dv + 2) * 4
    res.update({"segments": S, "value": b["GB/s"], "ms_per_call": b["ms"],
                "TFLOP/s": b["TFLOP/s"],
                "tensor_frac": round(b["TFLOP/s"] / peaks["bf16_tflops"], 4),
                "roofline": roofline("hbm", alg / (b["split_ms"] * 1e-3) / 1e9, peaks["hbm_gbs"],
                                     "GB/s", ncu_traffic("mla_decode")),
                "roofline_kernel": {"name": "mla_decode_kernel", "avg_ms": b["split_ms"],
                                    "alg_bytes_per_launch": alg},
                "segments_sweep": sweep})
    return res


def path_row_cascades(torch, rf, peaks):
    """Single-row cascades at every fusion level: softmax rows of 1K-8K
    (256 MB in, 256 MB out), variance of [16384 x 4096], moment of inertia of
    [4096 x 4096] points (256 MB); all larger than L2."""
    names = {0: "unfused", 1: "thread", 2: "warp", 3: "block"}
    g = torch.Generator(device="cuda").manual_seed(11)
    res = {"softmax": {}, "variance": {}, "inertia": {}, "layer_norm": {}}

    def entry(ms, nbytes):
        gbs = nbytes / (ms * 1e-3) / 1e9
        return {"us": round(ms * 1e3, 2), "GB/s": round(gbs, 1), "frac": round(gbs / peaks["hbm_gbs"], 4)}

    for n in (1024, 2048, 4096, 8192):
        R = (1 << 26) // n
        x = torch.randn(R, n, device="cuda", generator=g)
        y = torch.empty_like(x)
        work = torch.empty(2 * R, device="cuda")
        res["softmax"][f"n{n}"] = {}
        for lvl, nm in names.items():
            ms = time_graph(torch, [lambda: rf.rf_row_softmax(x, y, lvl, work)] * 5, 5)
            res["softmax"][f"n{n}"][nm] = entry(ms, 2 * R * n * 4)
        del x, y, work
    xv = torch.randn(16384, 4096, device="cuda", generator=g)
    mean = torch.empty(16384, device="cuda")
    var = torch.empty(16384, device="cuda")
    for lvl, nm in names.items():
        ms = time_graph(torch, [lambda: rf.rf_row_variance(xv, mean, var, lvl)] * 5, 5)
        res["variance"][nm] = entry(ms, xv.numel() * 4)
    del xv
    mass = torch.rand(4096, 4096, device="cuda", generator=g) + 0.05
    pos = torch.randn(4096, 3, 4096, device="cuda", generator=g)
    cen = torch.empty(4096, 3, device="cuda")
    ine = torch.empty(4096, device="cuda")
    for lvl, nm in names.items():
        ms = time_graph(torch, [lambda: rf.rf_moment_of_inertia(mass, pos, cen, ine, lvl)] * 5, 5)
        res["inertia"][nm] = entry(ms, (mass.numel() + pos.numel()) * 4)
    del mass, pos
    xl = torch.randn(16384, 4096, device="cuda", generator=g)
    yl = torch.empty_like(xl)
    gam = torch.randn(4096, device="cuda", generator=g)
    bet = torch.randn(4096, device="cuda", generator=g)
    wl = torch.empty(2 * 16384, device="cuda")
    res["layer_norm"] = {}
    for lvl, nm in ((0, "unfused"), (1, "fused")):
        ms = time_graph(torch, [lambda: rf.rf_layer_norm(xl, gam, bet, 1e-5, yl, lvl, wl)] * 5, 5)
        res["layer_norm"][nm] = entry(ms, 2 * xl.numel() * 4)
    res["rms_norm"] = {}
    wr = torch.empty(16384, device="cuda")
    for lvl, nm in ((0, "unfused"), (1, "fused")):
        ms = time_graph(torch, [lambda: rf.rf_rms_norm(xl, gam, 1e-6, yl, lvl, wr)] * 5, 5)
        res["rms_norm"][nm] = entry(ms, 2 * xl.numel() * 4)
    del xl, yl
    res["workload"] = ("row softmax R = 2^26/n rows of n fp32 (read + write counted); variance "
                       "x [16384, 4096]; moment of inertia mass [4096, 4096] + pos [4096, 3, 4096]; "
                       "layer norm and RMS norm x, y [16384, 4096] (read + write counted); "
                       "CUDA graphs of 5 calls, inputs larger than L2")
    return res


# --------------------------------------------------------------------- arms --

def run_rf(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if world > 1:
            dist.barrier()

    import cascaded_reductions_gb300 as rf
    import synthetic_inputs as si

    peaks = measured_peaks()
    if args.only:
        # one cascade alone (used for profiler captures of a single kernel)
        fns = {"single_row": lambda: path_single_row(torch, rf, peaks),
               "routing_256": lambda: path_routing(torch, rf, peaks, "route_256"),
               "routing_64": lambda: path_routing(torch, rf, peaks, "route_64"),
               "quant": lambda: path_quant(torch, rf, peaks),
               "gemm": lambda: path_gemm(torch, rf, peaks),
               "prefill": lambda: path_prefill(torch, rf, peaks),
               "mla": lambda: path_mla(torch, rf, peaks, args.mla_segments),
               "rows": lambda: path_row_cascades(torch, rf, peaks),
               "ablation_short": lambda: decode_ablation_short(torch, rf, peaks),
               "ablation": lambda: decode_ablation(
                   torch, rf, peaks, *si.decode_inputs(1024, 32768, 128, torch.bfloat16, seed=2,
                                                       device="cuda"), si.decode_scale(128))}
        print(json.dumps({args.only: fns[args.only]()}), flush=True)
        return
    B, H, L, D = DECODE["B"], DECODE["H"], DECODE["L"], DECODE["D"]
    if args.rows:                      # smaller batch of rows (profiling captures)
        B, H = 1, args.rows
    R, S = B * H, args.segments
    scale = si.decode_scale(D)
    q, K, V = si.decode_inputs(R, L, D, torch.bfloat16, seed=2 + 1000 * rank, device="cuda")
    seg_m = torch.empty(R, S, device="cuda")
    seg_l = torch.empty(R, S, device="cuda")
    seg_acc = torch.empty(R, S, D, device="cuda")
    out = torch.empty(R, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(R, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        rf.rf_attn_decode_split(q, K, V, S, scale, seg_m, seg_l, seg_acc, stream)
        rf.rf_state_merge(seg_m, seg_l, seg_acc, out, lse, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    ev0, ev1 = _events(torch, 2)
    ka, kb = _events(torch, args.steps), _events(torch, args.steps)
    ev0.record(stream)
    for i in range(args.steps):
        ka[i].record(stream)
        rf.rf_attn_decode_split(q, K, V, S, scale, seg_m, seg_l, seg_acc, stream)
        kb[i].record(stream)
        rf.rf_state_merge(seg_m, seg_l, seg_acc, out, lse, stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms_total = max_over_ranks(ev0.elapsed_time(ev1), world, "cuda")
    kern_ms = statistics.mean(ka[i].elapsed_time(kb[i]) for i in range(args.steps))
    ms_step = ms_total / args.steps
    kv_bytes = 2 * R * L * D * 2
    value = job_gbs(kv_bytes, world, ms_step)
    alg_bytes = kv_bytes + R * D * 2 + R * S * (D + 2) * 4
    achieved = alg_bytes / (kern_ms * 1e-3) / 1e9

    # the HBM read ceiling: one streaming read of K (8 GiB at full size) with
    # the decode kernel's own 16-byte loads and nothing else
    xor = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(3):
        rf.rf_stream_read(K, xor, stream)
    n_read = 5
    ra, rb = _events(torch, 2)
    ra.record(stream)
    for _ in range(n_read):
        rf.rf_stream_read(K, xor, stream)
    rb.record(stream)
    torch.cuda.synchronize()
    k_bytes = K.numel() * K.element_size()
    read_ceiling = k_bytes / (ra.elapsed_time(rb) / n_read * 1e-3) / 1e9

    # end to end through the public API with pinned host buffers
    e2e = None
    if not args.no_e2e:
        hq = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
        hK = torch.empty(K.shape, dtype=K.dtype, pin_memory=True)
        hV = torch.empty(V.shape, dtype=V.dtype, pin_memory=True)
        hq.copy_(q)
        hK.copy_(K)
        hV.copy_(V)
        hout = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        torch.cuda.synchronize()

        def e2e_step():
            q.copy_(hq, non_blocking=True)
            K.copy_(hK, non_blocking=True)
            V.copy_(hV, non_blocking=True)
            step()
            hout.copy_(out, non_blocking=True)
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        barrier()
        n_e2e = max(3, min(args.steps, 10))
        a, b = _events(torch, 2)
        a.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(a.elapsed_time(b) / n_e2e, world, "cuda")
        h2d = q.numel() * 2 + K.numel() * 2 + V.numel() * 2
        e2e = {"value": round(job_gbs(kv_bytes, world, e_ms), 1), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": out.numel() * 2,
               "ms_per_step": round(e_ms, 3), "steps": n_e2e}
        del hq, hK, hV

    paths = {}
    if world == 1 and not args.decode_only:
        # the same step as one launch: each row's last CTA merges its states
        counters = torch.zeros(R, dtype=torch.int32, device="cuda")
        fused = lambda: rf.rf_attn_decode_fused(q, K, V, S, scale, seg_m, seg_l, seg_acc, counters,
                                                out, lse, stream)
        for _ in range(3):
            fused()
        a, b = _events(torch, 2)
        a.record(stream)
        for _ in range(args.steps):
            fused()
        b.record(stream)
        torch.cuda.synchronize()
        ms_f = a.elapsed_time(b) / args.steps
        paths["decode_fused_one_launch"] = {
            "ms_per_step": round(ms_f, 4), "GB/s": round(job_gbs(kv_bytes, world, ms_f), 1),
            "workload": "the headline step through rf_attn_decode_fused (split and merge in one "
                        "launch, the merge done by each row's last CTA)"}
        paths["decode_incremental_vs_non_incremental"] = decode_ablation(torch, rf, peaks, q, K, V,
                                                                         scale)
        paths["decode_incremental_vs_non_incremental_short"] = decode_ablation_short(torch, rf, peaks)
        del q, K, V
        torch.cuda.empty_cache()
        for name, fn in (("single_row_decode_f32", lambda: path_single_row(torch, rf, peaks)),
                         ("routing_16384x256_top8", lambda: path_routing(torch, rf, peaks, "route_256")),
                         ("routing_65536x64_top2", lambda: path_routing(torch, rf, peaks, "route_64")),
                         ("absmax_quant_e4m3", lambda: path_quant(torch, rf, peaks)),
                         ("fp8_gemm", lambda: path_gemm(torch, rf, peaks)),
                         ("causal_prefill", lambda: path_prefill(torch, rf, peaks)),
                         ("mla_decode", lambda: path_mla(torch, rf, peaks)),
                         ("row_cascades", lambda: path_row_cascades(torch, rf, peaks))):
            try:
                paths[name] = fn()
            except Exception as e:         # report, never hide: the line says what failed
                paths[name] = {"error": f"{type(e).__name__}: {e}"}
            torch.cuda.empty_cache()

    cpu = cpu_baseline(args.cpu_budget) if (rank == 0 and world == 1 and not args.no_cpu) else None
    if paths and rank == 0 and not args.no_cpu:
        for name, base in oracle_path_baselines().items():
            if name in paths and isinstance(paths[name], dict) and "value" in paths[name]:
                paths[name]["cpu_oracle"] = base

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded N(0,1), drawn on the GPU)",
            "config": {"workload": f"split-KV decode attention B={B} H={H} L={L} D={D} bf16, "
                                   f"S={S} segments, fp32 accumulate, bf16 out",
                       "segments": S, "accumulate": "f32",
                       "l2": "inputs (16 GiB K/V) larger than L2, no flush",
                       "parallelism": f"replicas x{world} (rows are independent; no collective)"},
            "roofline": roofline("hbm", achieved, peaks["hbm_gbs"], "GB/s",
                                 ncu_traffic("decode_split")),
            "roofline_kernel": {"name": "decode_split_kernel", "avg_ms": round(kern_ms, 4),
                                "alg_bytes_per_launch": alg_bytes,
                                "peak_source": f"{peaks['source']} hbm_gbs (burst copy)",
                                "frac_of_read_ceiling": round(achieved / read_ceiling, 4)},
            "read_ceiling_gbs": round(read_ceiling, 1),
            "read_ceiling_how": (f"rf_stream_read over K ({k_bytes} bytes): "
                                 f"one 16-byte streaming read of every byte, the decode kernel's "
                                 f"load, nothing else; mean of {n_read} calls"),
            "e2e": e2e,
            "gpu_launches": 2 * args.steps,
            "clocks": clk,
            "cpu_baseline": cpu,
            "pages_claim": PAGES_CLAIM,
            "paths": paths,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference(args):
    """The CPU oracle as the reference arm: each step is one batch of rows of
    the decode workload (one row per host core)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    pool = OracleDecodePool()
    batch = pool.cores
    for _ in range(args.warmup):
        pool.run(batch)
    t = sum(pool.run(batch) for _ in range(args.steps))
    pool.close()
    ms_step = t / args.steps * 1e3
    value = batch * pool.row_bytes / (ms_step * 1e-3) / 1e9
    B, H, L, D = DECODE["B"], DECODE["H"], DECODE["L"], DECODE["D"]
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1), drawn on the CPU)",
        "config": {"workload": f"split-KV decode attention B={B} H={H} L={L} D={D} bf16, "
                               f"S={args.segments} segments, fp32 accumulate, bf16 out",
                   "segments": args.segments},
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": pool.cores,
                         "kind": "oracle",
                         "sample": f"each step: {batch} rows (q [128], K and V [32768, 128] bf16) of the "
                                   f"decode workload through the float64 oracle, one row per core"},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["rf", "reference"], default="rf")
    ap.add_argument("--segments", type=int, default=16)
    ap.add_argument("--rows", type=int, default=0,
                    help="decode rows instead of B*H=1024 (small cases for ncu captures)")
    ap.add_argument("--decode-only", action="store_true", help="skip the other cascades")
    ap.add_argument("--only", choices=["single_row", "routing_256", "routing_64", "quant", "gemm", "mla",
                                       "prefill", "rows", "ablation", "ablation_short"],
                    help="time one other cascade alone")
    ap.add_argument("--mla-segments", type=int, default=0,
                    help="with --only mla: time this segment count alone (profiler captures)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle work")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)      # at least three untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_rf(args)


if __name__ == "__main__":
    main()
