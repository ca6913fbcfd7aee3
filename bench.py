"""Benchmark of the GB300 block-quantized GEMV / MoE FFN hot path.

One step = the dense batch-1 GEMV sweep: one 4096 x 4096 matrix per format
(Q8_0, Q4_0, Q4_K, Q5_K, Q6_K, NaN scale in row 1), x ~ N(0,1), seed 0.
`value` = algorithmic bytes of a step (weights + x + y) / device time, in
GB/s, with inputs resident in HBM; weights rotate through copies totalling
more than 4x the L2 so every step streams from HBM.  The same run measures
the MoE FFN decode layer (128 experts, top-8, hidden 2048, expert_dim 768)
in us/token, the dense SwiGLU FFN, and the 512-token MoE layer.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 launch with torch.distributed.run: each rank runs an independent
replica (the path has no exchange step), timing is the max over ranks.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantized GEMV weight GB/s & % of HBM peak; MoE FFN layer µs/token"
FORMATS = [("Q8_0", 1), ("Q4_0", 2), ("Q4_K", 3), ("Q5_K", 4), ("Q6_K", 5)]
ROWS = COLS = 4096


def l2_bytes(torch, dev):
    """L2 size of the device, queried at run time."""
    return int(torch.cuda.get_device_properties(dev).L2_cache_size)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def dist_init(n_gpus):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if os.environ.get("QMOE_BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def job_throughput(bytes_per_rank_step, ms_per_step, world):
    """Whole-job GB/s: every rank moved bytes_per_rank_step per step, and a
    step took ms_per_step (the slowest rank's time)."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


def max_over_ranks(v, world, device=None):
    """Max of a float across ranks (all-reduce MAX); identity for one rank."""
    if world == 1:
        return float(v)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class Clocks:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.rows = []
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.strip().splitlines():
            f = [c.strip() for c in line.split(",")]
            if len(f) >= 9:
                self.rows.append(f)

    def summary(self):
        if not getattr(self, "rows", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in self.rows for k in range(4)
                          if r[5 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


# ------------------------------------------------------------------ ours
def run_ours(args, rank, world):
    import torch

    import moe_ffn_gb300 as qm
    from moe_ffn_gb300 import synth

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    qm.build()
    qm.lib()
    stream = torch.cuda.current_stream()

    # ---- GEMV sweep: weights rotate over copies > 4x L2
    mats, bytes_w = {}, {}
    for name, qt in FORMATS:
        g = synth.rng(qt)
        W = synth.quant_matrix(g, qt, ROWS, COLS, nan_row=1)
        x = synth.normal(g, COLS)
        mats[name] = (qt, torch.from_numpy(W).to(dev), torch.from_numpy(x).to(dev))
        bytes_w[name] = W.nbytes
    set_bytes = sum(bytes_w.values())
    L2 = l2_bytes(torch, dev)
    n_copies = int(np.ceil(4 * L2 / set_bytes)) + 1
    copies = {n: [mats[n][1].clone() for _ in range(n_copies)] for n, _ in FORMATS}
    ys = {n: torch.empty(ROWS, device=dev) for n, _ in FORMATS}
    torch.cuda.synchronize()
    alg_step = sum(bytes_w[n] + 4 * COLS + 4 * ROWS for n, _ in FORMATS)

    def step(i):
        c = i % n_copies
        for n, _ in FORMATS:
            qt, _, x = mats[n]
            qm.qmv(qt, copies[n][c], ROWS, COLS, x, ys[n])

    # One graph holds n_copies steps (every copy once); the timed region
    # replays it.  Launch cost is paid at capture, as a serving loop would.
    clk = Clocks(local).__enter__()  # sampled across all timed GPU work below
    g_sweep = capture(torch, step, n_copies)
    replays = max(1, args.steps // n_copies)
    steps_timed = replays * n_copies
    for _ in range(max(1, args.warmup // n_copies + 1)):
        g_sweep.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    # the K-step timed region, repeated; the median repetition is reported
    regions = []
    for _ in range(args.repeats):
        barrier(world)
        torch.cuda.synchronize()
        regions.append(time_replays(torch, g_sweep, replays))
    ms_local = statistics.median(regions)
    barrier(world)
    ms_total = max_over_ranks(ms_local, world, dev)
    ms_step = ms_total / steps_timed
    value = job_throughput(alg_step, ms_step, world)

    # ---- per-format kernel timing (dominant kernel roofline): L launches
    # back to back in a graph on the launching stream, rotating copies
    peak, peak_kind = load_peaks()
    per_fmt = {}
    L = 4 * n_copies
    for n, _ in FORMATS:
        qt, _, x = mats[n]

        def one(i, qt=qt, n=n, x=x):
            qm.qmv(qt, copies[n][i % n_copies], ROWS, COLS, x, ys[n])
        gf = capture(torch, one, L)
        gf.replay()
        torch.cuda.synchronize()
        us = time_graph(torch, gf) * 1e3 / L
        alg = bytes_w[n] + 4 * COLS + 4 * ROWS
        per_fmt[n] = {"us": round(us, 3), "gbs": round(alg / us / 1e3, 1),
                      "frac": round(alg / us / 1e3 / peak, 3), "bytes": alg}
        del gf
    dom = max(per_fmt, key=lambda n: per_fmt[n]["us"])
    traffic = load_traffic(f"qmv_{dom}")

    # ---- end to end through the public API with host buffers: every step
    # copies x from pinned host memory, runs the five GEMVs and copies y
    # back; plain calls from Python, no graph.
    xs_host = {n: torch.from_numpy(synth.normal(synth.rng(100 + qt), COLS)).pin_memory()
               for n, qt in FORMATS}
    ys_host = {n: torch.empty(ROWS).pin_memory() for n, _ in FORMATS}
    xs_dev = {n: torch.empty(COLS, device=dev) for n, _ in FORMATS}

    def e2e_step(i):
        c = i % n_copies
        for n, _ in FORMATS:
            qt = mats[n][0]
            xs_dev[n].copy_(xs_host[n], non_blocking=True)
            qm.qmv(qt, copies[n][c], ROWS, COLS, xs_dev[n], ys[n], stream)
            ys_host[n].copy_(ys[n], non_blocking=True)

    e2e_steps = min(args.steps, 500)
    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / e2e_steps
    e2e_value = job_throughput(alg_step, e2e_ms, world)

    del copies, g_sweep
    torch.cuda.empty_cache()
    extra = {}
    if not args.skip_layers:
        extra = bench_layers(qm, synth, dev, stream, args)
    clk.__exit__(None, None, None)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": steps_timed, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "dense batch-1 GEMV sweep, 4096x4096 per format "
                               "Q8_0/Q4_0/Q4_K/Q5_K/Q6_K, NaN scale in row 1, seed 0",
                   "rows": ROWS, "cols": COLS, "weight_copies": n_copies,
                   "l2": "weights rotate over copies totalling > 4x L2 (no flush needed)",
                   "launch": f"CUDA graph of {n_copies} steps, replayed",
                   "timed_region": f"{steps_timed} steps, repeated {args.repeats} times; "
                                   "the median repetition",
                   "arithmetic": "GGUF blocks decoded exactly; f32 activations, f32 sums",
                   "parallelism": f"replicas{world}"},
        "roofline": {"bound": "hbm", "kernel": f"qmv_tile_kernel<{dom}>",
                     "achieved": per_fmt[dom]["gbs"], "peak": peak, "unit": "GB/s",
                     "frac": per_fmt[dom]["frac"], "traffic": traffic,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, burst copy)"},
        "per_format": per_fmt,
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s",
                "h2d_bytes_per_step": 4 * COLS * len(FORMATS),
                "d2h_bytes_per_step": 4 * ROWS * len(FORMATS),
                "how": "plain Python calls per step (no graph), pinned-host x in, y out"},
        "gpu_launches": steps_timed * len(FORMATS),
        "clocks": clk.summary(),
    }
    line.update(extra)
    if rank == 0 and world == 1 and not args.skip_cpu:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds, all_cores=True)
        line["cpu_baseline_1core"] = cpu_baseline(args.cpu_seconds)
    return line


def capture(torch, fn, n):
    """A CUDA graph of fn(0) .. fn(n-1).  fn is called once beforehand (outside
    the capture) so one-time library set-up does not happen while capturing."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn(0)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(n):
            fn(i)
    torch.cuda.synchronize()
    return g


def time_replays(torch, g, replays):
    """ms for `replays` back-to-back replays, CUDA events on the launching stream."""
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(st)
    for _ in range(replays):
        g.replay()
    e1.record(st)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def time_graph(torch, g, min_s=0.5, chunk_ms=25.0):
    """Median ms per replay of graph g over a timed span of at least min_s:
    chunks of about chunk_ms of back-to-back replays, each timed with CUDA
    events; the median of the chunks' per-replay times."""
    one = max(time_replays(torch, g, 2) / 2, 1e-3)
    per_chunk = max(1, int(chunk_ms / one))
    n_chunks = max(5, int(min_s * 1e3 / (per_chunk * one)) + 1)
    return statistics.median(time_replays(torch, g, per_chunk) / per_chunk
                             for _ in range(n_chunks))


GEMV_SOURCES = ("formats.cuh", "ptx.cuh", "stream.cuh")


def gemv_source_hash():
    import hashlib
    h = hashlib.sha256()
    for f in GEMV_SOURCES:
        with open(os.path.join(ROOT, "moe_ffn_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_traffic(key):
    """dram bytes per launch from the committed ncu summary, or None if the
    kernel's sources changed since that capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(p):
        d = json.load(open(p))
        v = d.get(key)
        if isinstance(v, dict) and v.get("src_sha256_16") == gemv_source_hash():
            return v.get("bytes_per_launch")
    return None


def bench_layers(qm, synth, dev, stream, args):
    """MoE decode (us/token), dense FFN (us/call), MoE 512-token layer
    (us/token); each captured in a CUDA graph and replayed."""
    import torch
    out = {}
    peak, _ = load_peaks()
    # MoE decode: NCOPY copies of the full stacks (391.6 MB each, 1.57 GB in
    # all) rotate call by call, and x rotates over 64 token vectors, so the
    # routing (and the experts read) varies per call and an expert's rows
    # come back to the same copy only every NCOPY calls.
    shp = synth.MOE_DECODE
    inp = synth.moe_inputs(0, **shp)
    g = synth.rng(99)
    xpool = torch.from_numpy(synth.normal(g, (64, shp["hidden"]))).to(dev)
    s = qm.moe_shape(shp["hidden"], shp["expert_dim"], shp["num_experts"], shp["top_k"], 1,
                     shp["gate"], shp["up"], shp["down"])
    NCOPY = 4
    dc = [{k: torch.from_numpy(inp[k]).to(dev) for k in ("router", "gate", "up", "down")}
          for _ in range(NCOPY)]
    d = dc[0]
    res = torch.from_numpy(inp["residual"]).to(dev)
    ws = torch.zeros(qm.moe_ffn_workspace_size(s), dtype=torch.uint8, device=dev)
    idx = torch.empty((1, shp["top_k"]), dtype=torch.int32, device=dev)

    def call(i):
        c = dc[i % NCOPY]
        qm.moe_ffn(c["router"], c["gate"], c["up"], c["down"], s, xpool[i % 64], res, idx, None,
                   ws)
    n = 64
    gm = capture(torch, call, n)
    gm.replay()
    us = time_graph(torch, gm) * 1e3 / n
    rb_g = qm.row_bytes(shp["gate"], shp["hidden"])
    rb_d = qm.row_bytes(shp["down"], shp["expert_dim"])
    alg = (shp["num_experts"] * shp["hidden"] * 4
           + shp["top_k"] * (2 * shp["expert_dim"] * rb_g + shp["hidden"] * rb_d)
           + 3 * shp["hidden"] * 4)
    out["moe_decode"] = {"us_per_token": round(us, 3), "alg_bytes": alg,
                         "gbs": round(alg / us / 1e3, 1), "frac": round(alg / us / 1e3 / peak, 3),
                         "launches_per_token": 1,
                         "launch": f"CUDA graph of {n} tokens over {NCOPY} stack copies "
                                   f"(1.57 GB), replayed for >= 0.5 s, median",
                         "workload": "hidden 2048, 128 experts, top-8, expert_dim 768, Q4_K/Q4_K/Q6_K"}
    # the same layer with ffn_norm fused in front (input = the hidden state)
    nw = torch.from_numpy(synth.norm_weight(synth.rng(98), shp["hidden"])).to(dev)
    hpool = xpool.clone()
    wsn = torch.zeros(qm.moe_ffn_rmsnorm_workspace_size(s), dtype=torch.uint8, device=dev)

    def ncall(i):
        c = dc[i % NCOPY]
        qm.moe_ffn_rmsnorm(c["router"], c["gate"], c["up"], c["down"], s, nw, 1e-6,
                           hpool[i % 64], idx, None, wsn)
    gn = capture(torch, ncall, n)
    gn.replay()
    usn = time_graph(torch, gn) * 1e3 / n
    out["moe_decode"]["us_per_token_with_ffn_norm"] = round(usn, 3)
    # small batches: T tokens per call, each routed expert read once per call
    xpool2 = torch.cat([xpool, xpool])
    per_expert = 2 * shp["expert_dim"] * rb_g + shp["hidden"] * rb_d
    batched = {}
    for T in (2, 4, 8, 16):
        sT = qm.moe_shape(shp["hidden"], shp["expert_dim"], shp["num_experts"], shp["top_k"], T,
                          shp["gate"], shp["up"], shp["down"])
        wsT = torch.zeros(qm.moe_ffn_workspace_size(sT), dtype=torch.uint8, device=dev)
        resT = torch.from_numpy(synth.normal(synth.rng(97), (T, shp["hidden"]))).to(dev)
        idxT = torch.empty((T, shp["top_k"]), dtype=torch.int32, device=dev)

        def bcall(i, T=T, sT=sT, wsT=wsT, resT=resT, idxT=idxT):
            j = (i * T) % 64
            c = dc[i % NCOPY]
            qm.moe_ffn(c["router"], c["gate"], c["up"], c["down"], sT, xpool2[j:j + T], resT,
                       idxT, None, wsT)
        nT = max(8, 64 // T)
        experts = []
        for i in range(nT):  # distinct experts each call reads
            bcall(i)
            experts.append(len(np.unique(idxT.cpu().numpy())))
        gb = capture(torch, bcall, nT)
        gb.replay()
        usb = time_graph(torch, gb) * 1e3 / nT
        ne = float(np.mean(experts))
        algb = shp["num_experts"] * shp["hidden"] * 4 + ne * per_expert + 3 * T * shp["hidden"] * 4
        batched[str(T)] = {"us_per_call": round(usb, 3), "us_per_token": round(usb / T, 3),
                           "experts_read": round(ne, 2), "gbs": round(algb / usb / 1e3, 1),
                           "frac": round(algb / usb / 1e3 / peak, 3)}
        del gb
    out["moe_decode"]["batched"] = batched
    out["moe_decode"]["batched_launch"] = ("CUDA graph of max(8, 64/T) calls of T tokens over "
                                           f"{NCOPY} stack copies, >= 0.5 s, median; alg bytes = "
                                           "router + distinct experts read + x, residual in/out")
    del d, dc, inp, gm, gn
    torch.cuda.empty_cache()

    # dense SwiGLU FFN: 114 MB weights, 5 copies rotating (> 4x L2)
    w = synth.DENSE_FFN
    fin = synth.ffn_inputs(0, **w)
    ncp = 5
    G = [torch.from_numpy(fin["gate"]).to(dev) for _ in range(ncp)]
    U = [torch.from_numpy(fin["up"]).to(dev) for _ in range(ncp)]
    D = [torch.from_numpy(fin["down"]).to(dev) for _ in range(ncp)]
    x = torch.from_numpy(fin["x"]).to(dev)
    r = torch.from_numpy(fin["residual"]).to(dev)
    ws = torch.empty(qm.ffn_swiglu_workspace_size(w["hidden"], w["inter"]), dtype=torch.uint8,
                     device=dev)

    def fcall(i):
        c = i % ncp
        qm.ffn_swiglu(G[c], U[c], D[c], w["gate"], w["up"], w["down"], w["hidden"], w["inter"],
                      x, r, ws)
    n = 2 * ncp
    gf = capture(torch, fcall, n)
    gf.replay()
    us = time_graph(torch, gf) * 1e3 / n
    alg = fin["gate"].nbytes + fin["up"].nbytes + fin["down"].nbytes + 4 * w["hidden"] * 3
    out["dense_ffn"] = {"us": round(us, 3), "alg_bytes": alg, "gbs": round(alg / us / 1e3, 1),
                        "frac": round(alg / us / 1e3 / peak, 3), "launches": 1,
                        "launch": f"CUDA graph of {n} calls over {ncp} weight copies, "
                                  ">= 0.5 s, median",
                        "workload": "hidden 4096, intermediate 14336, Q4_K/Q4_K/Q6_K"}
    del G, U, D, gf
    torch.cuda.empty_cache()

    # lm_head-sized GEMVs: vocab 151,936 x hidden 2048, F32 (1.24 GB) and
    # Q6_K (255 MB, two copies rotating)
    lm = {}
    V, Hd = 151936, 2048
    for name, qt in (("F32", 0), ("Q6_K", 5), ("Q8_0", 1)):
        g = synth.rng(151936 + qt)
        if qt == 0:
            Wl = torch.randn((V, Hd), device=dev) * 0.02
            nbytes = Wl.numel() * 4
            cps = [Wl]
        else:
            Wh = synth.quant_matrix(g, qt, V, Hd)
            nbytes = Wh.nbytes
            cps = [torch.from_numpy(Wh).to(dev) for _ in range(2)]
        xl = torch.from_numpy(synth.normal(g, Hd)).to(dev)
        yl = torch.empty(V, device=dev)

        def lcall(i, qt=qt, cps=cps, xl=xl, yl=yl):
            qm.qmv(qt, cps[i % len(cps)], V, Hd, xl, yl)
        nl = 4
        gl = capture(torch, lcall, nl)
        gl.replay()
        us = time_graph(torch, gl) * 1e3 / nl
        alg = nbytes + 4 * Hd + 4 * V
        lm[name] = {"us": round(us, 2), "gbs": round(alg / us / 1e3, 1),
                    "frac": round(alg / us / 1e3 / peak, 3), "bytes": alg}
        del gl, cps
        torch.cuda.empty_cache()
    out["lm_head_gemv"] = {"workload": "vocab 151936 x hidden 2048, one qmv call",
                           "launch": "CUDA graph of 4 calls, >= 0.5 s, median", **lm}

    # MoE 512-token layer
    shp = synth.MOE_PREFILL
    inp = synth.moe_inputs(0, **shp)
    s = qm.moe_shape(shp["hidden"], shp["expert_dim"], shp["num_experts"], shp["top_k"],
                     shp["n_tokens"], shp["gate"], shp["up"], shp["down"])
    d = {k: torch.from_numpy(inp[k]).to(dev) for k in ("router", "gate", "up", "down", "x",
                                                          "residual")}
    ws = torch.zeros(qm.moe_ffn_workspace_size(s), dtype=torch.uint8, device=dev)

    def pcall(i):
        qm.moe_ffn(d["router"], d["gate"], d["up"], d["down"], s, d["x"], d["residual"], None,
                   None, ws)
    gp = capture(torch, pcall, 1)
    gp.replay()
    us = time_graph(torch, gp) * 1e3
    rb_g = qm.row_bytes(shp["gate"], shp["hidden"])
    rb_d = qm.row_bytes(shp["down"], shp["expert_dim"])
    alg_w = shp["num_experts"] * (2 * shp["expert_dim"] * rb_g + shp["hidden"] * rb_d)
    alg = alg_w + shp["num_experts"] * shp["hidden"] * 4 + 3 * shp["n_tokens"] * shp["hidden"] * 4
    flops = 2 * shp["n_tokens"] * shp["top_k"] * 3 * shp["hidden"] * shp["expert_dim"]
    out["moe_prefill"] = {"us_per_call": round(us, 1),
                          "us_per_token": round(us / shp["n_tokens"], 3),
                          "alg_bytes": alg, "gbs": round(alg / us / 1e3, 1),
                          "frac_hbm": round(alg / us / 1e3 / peak, 4),
                          "expert_tflops": round(flops / us / 1e6, 2),
                          "launch": "CUDA graph of one call, replayed for >= 0.5 s, median",
                          "workload": "512 tokens, hidden 2048, 64 experts, top-8, "
                                      "expert_dim 1024, Q4_K/Q4_K/Q6_K"}
    return out


# ------------------------------------------------------------- the oracle
def oracle_sweep_setup():
    import oracle
    from moe_ffn_gb300 import synth
    oracle.build()
    data = []
    for name, qt in FORMATS:
        g = synth.rng(qt)
        W = synth.quant_matrix(g, qt, ROWS, COLS, nan_row=1)
        x = synth.normal(g, COLS)
        data.append((qt, W, x))
    return oracle, data


def _oracle_sweeps(seconds):
    """Whole sweeps (all five 4096x4096 GEMVs) of the oracle until `seconds`
    have passed, in this process: (sweeps, elapsed seconds)."""
    orc, data = oracle_sweep_setup()
    t0 = time.perf_counter()
    n = 0
    while True:
        for qt, W, x in data:
            orc.matvec(qt, W, ROWS, COLS, x)
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    return n, time.perf_counter() - t0


# Arm "CPU part" numbers (implementer 0x41) of the cores these hosts carry
ARM_PARTS = {"0xd4f": "Arm Neoverse V2", "0xd40": "Arm Neoverse V1", "0xd0c": "Arm Neoverse N1",
             "0xd49": "Arm Neoverse N2", "0xd8f": "Arm Neoverse V3"}


def cpu_model(cpuinfo="/proc/cpuinfo"):
    """The host CPU's name: x86 'model name', or an Arm core's part number
    with its name when known (e.g. 0xd4f, Neoverse V2 as in Grace)."""
    part = None
    try:
        for line in open(cpuinfo):
            k, _, v = line.partition(":")
            k, v = k.strip(), v.strip()
            if k in ("model name", "Model name"):
                return v
            if k == "CPU part" and part is None:
                part = v
    except OSError:
        pass
    if part:
        name = ARM_PARTS.get(part.lower())
        return f"{name} (CPU part {part})" if name else f"Arm CPU part {part}"
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline(seconds=12.0, all_cores=False):
    """The oracle as it stands (plain C, one thread per process), timed on this
    host on whole sweeps for about `seconds`: in this process, or (all_cores)
    in one spawned process per host core at once, the bytes of every
    process's sweeps over the wall time."""
    alg = sum(W.nbytes + 4 * COLS + 4 * ROWS for _, W, _ in oracle_sweep_setup()[1])
    if not all_cores:
        n, dt = _oracle_sweeps(seconds)
        return {"value": round(n * alg / dt / 1e9, 4), "unit": "GB/s", "cores": 1,
                "kind": "oracle",
                "sample": f"{n} full sweeps (5 x 4096x4096 GEMVs, decode-then-dot, fp64 "
                          f"accumulation) in {dt:.1f} s on one core of {cpu_model()}"}
    import multiprocessing as mp
    cores = os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    t0 = time.perf_counter()
    with ctx.Pool(cores) as pool:
        res = pool.map(_oracle_sweeps, [seconds] * cores)
    wall = time.perf_counter() - t0
    n = sum(r[0] for r in res)
    return {"value": round(n * alg / wall / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{n} full sweeps over {cores} processes (one oracle per core, "
                      f"{seconds:.0f} s each) in {wall:.1f} s wall on {cpu_model()}"}


def run_reference(args, rank, world):
    """The oracle, timed as the reference arm.  Each step is a bounded sample
    of the sweep: one whole 4096x4096 GEMV, the five formats in turn (about
    0.02 s of CPU work), so K steps take about K/50 s."""
    orc, data = oracle_sweep_setup()
    per = [W.nbytes + 4 * COLS + 4 * ROWS for _, W, _ in data]

    def step(i):
        qt, W, x = data[i % len(data)]
        orc.matvec(qt, W, ROWS, COLS, x)
        return per[i % len(data)]
    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    done = 0
    for i in range(args.steps):
        done += step(i)
    dt = time.perf_counter() - t0
    ms_step = dt * 1e3 / args.steps
    v = done / dt / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "dense batch-1 GEMV sweep, 4096x4096 per format "
                               "Q8_0/Q4_0/Q4_K/Q5_K/Q6_K, NaN scale in row 1, seed 0",
                   "rows": ROWS, "cols": COLS, "parallelism": "replicas1"},
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} single-format 4096x4096 GEMVs (formats in turn) after {args.warmup} warm-up"},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_profile_case(case, launches):
    """Minimal program for ncu: one workload, `launches` calls, nothing else.
    gemv:<FMT>[:rows] — one [rows]x4096 GEMV (default 4096 rows); moe[:T] — the decode layer
    for T tokens (default 1); ffn — the dense FFN."""
    import torch

    import moe_ffn_gb300 as qm
    from moe_ffn_gb300 import synth
    qm.build()
    dev = torch.device("cuda", 0)
    if case.startswith("gemv:"):
        parts = case.split(":")
        name = parts[1]
        rows = int(parts[2]) if len(parts) > 2 else ROWS
        qt = dict(FORMATS)[name]
        g = synth.rng(qt)
        W = torch.from_numpy(synth.quant_matrix(g, qt, rows, COLS, nan_row=1)).to(dev)
        x = torch.from_numpy(synth.normal(g, COLS)).to(dev)
        y = torch.empty(rows, device=dev)
        for _ in range(launches):
            qm.qmv(qt, W, rows, COLS, x, y)
    elif case == "moe" or case.startswith("moe:"):
        T = int(case.split(":")[1]) if ":" in case else 1
        shp = dict(synth.MOE_DECODE, n_tokens=T)
        inp = synth.moe_inputs(0, **shp)
        s = qm.moe_shape(shp["hidden"], shp["expert_dim"], shp["num_experts"], shp["top_k"], T,
                         shp["gate"], shp["up"], shp["down"])
        d = {k: torch.from_numpy(inp[k]).to(dev) for k in inp}
        ws = torch.zeros(qm.moe_ffn_workspace_size(s), dtype=torch.uint8, device=dev)
        for _ in range(launches):
            qm.moe_ffn(d["router"], d["gate"], d["up"], d["down"], s, d["x"], d["residual"],
                       None, None, ws)
    elif case == "moe_prefill":
        shp = synth.MOE_PREFILL
        inp = synth.moe_inputs(0, **shp)
        s = qm.moe_shape(shp["hidden"], shp["expert_dim"], shp["num_experts"], shp["top_k"],
                         shp["n_tokens"], shp["gate"], shp["up"], shp["down"])
        d = {k: torch.from_numpy(inp[k]).to(dev) for k in inp}
        ws = torch.zeros(qm.moe_ffn_workspace_size(s), dtype=torch.uint8, device=dev)
        for _ in range(launches):
            qm.moe_ffn(d["router"], d["gate"], d["up"], d["down"], s, d["x"], d["residual"],
                       None, None, ws)
    elif case == "ffn":
        w = synth.DENSE_FFN
        fin = synth.ffn_inputs(0, **w)
        d = {k: torch.from_numpy(fin[k]).to(dev) for k in fin}
        ws = torch.empty(qm.ffn_swiglu_workspace_size(w["hidden"], w["inter"]),
                         dtype=torch.uint8, device=dev)
        for _ in range(launches):
            qm.ffn_swiglu(d["gate"], d["up"], d["down"], w["gate"], w["up"], w["down"],
                          w["hidden"], w["inter"], d["x"], d["residual"], ws)
    else:
        raise SystemExit(f"unknown profile case {case}")
    torch.cuda.synchronize()
    st = qm.device_status()
    print(json.dumps({"profile_case": case, "launches": launches, "device_status": st}))
    return 0 if st == 0 else 1


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--skip-layers", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--repeats", type=int, default=50,
                    help="repetitions of the K-step timed region (the median is reported)")
    ap.add_argument("--profile", default=None,
                    help="run one small case for ncu (gemv:<FMT>, moe, ffn) and exit")
    args = ap.parse_args(argv)
    if args.profile:
        return run_profile_case(args.profile, args.steps)
    if args.warmup < 3:
        args.warmup = 3
    rank, world = dist_init(args.gpus)
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, 1)))
        return 0
    line = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
