"""Benchmark of the MAPL boundary codec on GB300: compress (+ residual VQ) and
reconstruct one micro-batch per step, as boundary tokens/s.

Default workload: d=1024, r=128, 16 x 2048 tokens, bf16, VQ with G=4 groups,
R=2 rounds, K=256 codes (8 bytes of indices per token).  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the reference arm) on a bounded
sample per step.  Under torchrun every rank runs its own micro-batches (the
codec is per token, no collective on the data path) and rank 0 prints.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "boundary tokens/s (compress+RVQ+reconstruct) and % roofline, d=1024 r=128"
UNIT = "tokens/s"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=200)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="vq_d1024_r128")
    p.add_argument("--e2e-steps", type=int, default=40)
    p.add_argument("--no-clocks", action="store_true")
    p.add_argument("--tokens", type=int, default=0,
                   help="tokens per step (default: the workload's micro-batch); for profiling")
    p.add_argument("--skip-cpu", action="store_true", help="skip the CPU-baseline timing")
    return p.parse_args()


# ----------------------------------------------------------------- helpers
def dist_setup(args=None, backend: str = "nccl"):
    """One process per GPU (torchrun env).  The codec shards by micro-batch:
    every rank compresses and reconstructs its own tokens and no collective
    touches the data path; the process group only carries the barrier and
    the max-over-ranks of the timings."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if ws > 1:
        import torch
        import torch.distributed as dist
        if backend == "nccl":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group(backend)
    return ws, rank


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, ws: int, max_ms: float) -> float:
    """Units all ranks processed in the timed region / the slowest rank's time."""
    return units_per_rank * ws / (max_ms * 1e-3)


def rank_seed(rank: int) -> int:
    """Each rank draws its own micro-batches (weak scaling: the work per rank
    is fixed, no two ranks process the same tokens)."""
    return rank


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, enabled=True):
        self.proc = None
        self.path = None
        if enabled:
            try:
                import tempfile
                fd, self.path = tempfile.mkstemp(prefix="mapl_clocks_", suffix=".csv")
                self.f = os.fdopen(fd, "w")
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                     "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
            except Exception:
                self.proc = None

    def stop(self, dev_index: int):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sms, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9 or not f[0].isdigit() or int(f[0]) != dev_index:
                continue
            try:
                sms.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sms:
            return None
        return {"sm_mhz": float(np.median(sms)), "sm_max_mhz": mx, "samples": len(sms),
                "reasons": sorted(reasons)}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


KERNEL_SOURCES = {"mapl_compress": "kernels_compress.cu", "mapl_decompress": "kernels_tc.cu"}


def kernel_source_hash(kernel: str) -> str:
    """Hash of the sources a kernel is built from: a profiled traffic figure
    is reported only while it still describes the kernel that runs."""
    h = hashlib.sha256()
    for name in (KERNEL_SOURCES[kernel], "ptx.cuh", "mapl_internal.h", "mapl_api.cu"):
        with open(os.path.join(ROOT, "pipeline_activation_compression_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        j = json.load(f)
    e = j.get(f"{kernel}:{workload}")
    if not e or e.get("source_hash") != kernel_source_hash(kernel):
        return None
    return float(e["dram_bytes_per_launch"])


def algorithmic_bytes(w, tids: np.ndarray):
    """Bytes a launch must move at minimum through HBM (algorithmic count):
    compress:   X (2d) + tid (4) + payload out, per token; unique anchor rows
                (2r each) and the parameters (A^T, M splits, codebooks) once.
    decompress: payload in + tid (4) + X_hat (2d), per token; unique anchor
                rows of the receiver and the parameters ([A | P'^T], codebooks).
    """
    N = tids.size
    payload = w.R * w.G if w.vq else 2 * w.r
    U = np.unique(tids).size
    books = (w.R * w.G * w.K * w.gd * 2) if w.vq else 0
    comp = N * (2 * w.d + 4 + payload) + U * 2 * w.r + 2 * w.d * w.r + 3 * 2 * w.r * w.r + books
    decomp = N * (payload + 4 + 2 * w.d) + U * 2 * w.r + 2 * w.d * 2 * w.r + books
    return float(comp), float(decomp), U


# ------------------------------------------------------------- CPU oracle
def oracle_step(b, w, rows):
    import oracle
    W = np.asarray
    from pipeline_activation_compression_gb300 import synth
    X = synth.widen(b["X"][rows])
    t = b["tids"][rows]
    Z = oracle.compress(X, t, synth.widen(b["A"]), synth.widen(b["E"]), synth.widen(b["P"]))
    if w.vq:
        C = synth.widen(b["C"])
        idx = oracle.rvq_encode(Z, C)["idx"]
        Zh = oracle.rvq_decode(idx, C)
    else:
        Zh = Z
    return oracle.reconstruct(Zh, t, synth.widen(b["A"]), synth.widen(b["E_next"]),
                              synth.widen(b["P_next"]))


def cpu_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def time_oracle(b, w, tokens: int, budget_s: float):
    """Oracle tokens/s on chunks of `tokens` rows until `budget_s` elapses."""
    rng = np.random.default_rng(0)
    done, t0 = 0, time.perf_counter()
    while True:
        rows = np.sort(rng.choice(b["tids"].size, size=tokens, replace=False))
        oracle_step(b, w, rows)
        done += tokens
        el = time.perf_counter() - t0
        if el >= budget_s:
            return done / el, done, el


# --------------------------------------------------------------- our arm
def run_ours(args, ws, rank):
    import torch
    import pipeline_activation_compression_gb300 as mapl
    from pipeline_activation_compression_gb300 import synth

    dev = torch.cuda.current_device()
    mapl.build()
    mapl.load_library()
    w = synth.WORKLOADS[args.workload]
    N = args.tokens or w.N
    b = synth.make_boundary(w, seed=rank_seed(rank), n_tokens=N)

    def to_dev(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
        return torch.from_numpy(a).cuda()

    dt = mapl.MAPL_BF16 if w.dtype == "bf16" else mapl.MAPL_F32
    cfg = mapl.make_config(w.d, w.r, w.V, w.G, w.R, w.K, dt)
    plan = mapl.mapl_plan_create(cfg, to_dev(b["A"]), to_dev(b["P"]), to_dev(b["P_next"]),
                                 to_dev(b["C"]) if w.vq else None)
    E, En = to_dev(b["E"]), to_dev(b["E_next"])
    t = to_dev(b["tids"])
    x0 = to_dev(b["X"])
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    xbytes = x0.numel() * x0.element_size()
    nsets = max(3, int(np.ceil(2 * l2 / xbytes)) + 1)
    Xs = [x0] + [x0.clone() for _ in range(nsets - 1)]
    Xh = [torch.empty(N, w.d, dtype=x0.dtype, device="cuda") for _ in range(nsets)]
    pay = [torch.empty(plan.payload_shape(N), dtype=plan.payload_dtype(), device="cuda")
           for _ in range(nsets)]
    stream = torch.cuda.current_stream()

    def step(i):
        k = i % nsets
        mapl.mapl_compress(plan, Xs[k], t, E, pay[k], stream)
        mapl.mapl_decompress(plan, pay[k], t, En, Xh[k], stream)

    for i in range(args.warmup):
        step(i)
    mapl.mapl_check(plan)
    torch.cuda.synchronize()

    K = args.steps
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * K + 1)]
    clocks = ClockSampler(enabled=(rank == 0 and not args.no_clocks))
    barrier(ws)
    torch.cuda.synchronize()
    ev[0].record(stream)
    for i in range(K):
        k = i % nsets
        mapl.mapl_compress(plan, Xs[k], t, E, pay[k], stream)
        ev[2 * i + 1].record(stream)
        mapl.mapl_decompress(plan, pay[k], t, En, Xh[k], stream)
        ev[2 * i + 2].record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clk = clocks.stop(dev) if rank == 0 else None
    mapl.mapl_check(plan)
    total_ms = ev[0].elapsed_time(ev[2 * K])
    comp_ms = np.array([ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(K)])
    dec_ms = np.array([ev[2 * i + 1].elapsed_time(ev[2 * i + 2]) for i in range(K)])
    total_ms = max_over_ranks(total_ms, ws)

    # the same steps captured once in a CUDA graph (one step per buffer set)
    # and replayed: reported beside the plain-launch number
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cap = torch.cuda.current_stream()
        for k in range(nsets):
            mapl.mapl_compress(plan, Xs[k], t, E, pay[k], cap)
            mapl.mapl_decompress(plan, pay[k], t, En, Xh[k], cap)
    reps = max(1, K // nsets)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    g0.record(stream)
    for _ in range(reps):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    graph_ms = max_over_ranks(g0.elapsed_time(g1), ws) / (reps * nsets)
    mapl.mapl_check(plan)

    # the device's plain write rate on the same rotating X_hat buffers: a
    # fill of N x d bf16 (no reads), the floor under decompress, whose
    # traffic is almost all X_hat writes
    for k in range(2 * nsets):
        Xh[k % nsets].fill_(0)
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    nf = 10 * nsets
    f0.record(stream)
    for k in range(nf):
        Xh[k % nsets].fill_(0)
    f1.record(stream)
    torch.cuda.synchronize()
    fill_ms = f0.elapsed_time(f1) / nf

    # end to end through the public API's host-buffer calls: X and tids from
    # pinned host memory in, the payload out to the host and back, X_hat out
    # to pinned host memory.  Consecutive steps rotate over six streams (each
    # with its own device workspace and host outputs), so one step's download
    # overlaps the next steps' uploads, as successive micro-batches of a
    # pipeline would (2 / 4 / 6 / 8 streams measured 55 / 63 / 72 / 72 M
    # tokens/s).  The host link (about 210 GB/s up, 190 down, 330 both ways)
    # bounds this number.
    Ke = args.e2e_steps
    xh_host = torch.from_numpy(np.ascontiguousarray(b["X"]).view(np.int16)).view(torch.bfloat16).pin_memory()
    t_host = torch.from_numpy(b["tids"]).pin_memory()
    NS = 6
    streams = [stream] + [torch.cuda.Stream() for _ in range(NS - 1)]
    wsz = mapl.mapl_host_workspace_size(plan, N)
    wsp = [torch.empty(wsz, dtype=torch.uint8, device="cuda") for _ in range(NS)]
    pay_h = [torch.empty(plan.payload_shape(N), dtype=plan.payload_dtype()).pin_memory()
             for _ in range(NS)]
    out_h = [torch.empty(N, w.d, dtype=torch.bfloat16).pin_memory() for _ in range(NS)]

    def e2e_step(k):
        j = k % NS
        mapl.mapl_compress_host(plan, xh_host, t_host, E, pay_h[j], wsp[j], streams[j])
        mapl.mapl_decompress_host(plan, pay_h[j], t_host, En, out_h[j], wsp[j], streams[j])

    for k in range(2 * NS):
        e2e_step(k)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    e0.record(streams[0])
    for sx in streams[1:]:
        sx.wait_event(e0)
    for k in range(Ke):
        e2e_step(k)
    for sx in streams[1:]:
        joined = torch.cuda.Event()
        joined.record(sx)
        streams[0].wait_event(joined)
    e1.record(streams[0])
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), ws)
    mapl.mapl_check(plan)

    if rank != 0:
        return None
    comp_b, dec_b, U = algorithmic_bytes(w, b["tids"])
    comp_avg, dec_avg = float(comp_ms.mean()), float(dec_ms.mean())
    dom = "mapl_compress" if comp_avg >= dec_avg else "mapl_decompress"
    dom_bytes, dom_ms = (comp_b, comp_avg) if dom == "mapl_compress" else (dec_b, dec_avg)
    peak, peak_kind = peaks()
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    step_bytes = comp_b + dec_b
    value = whole_job_rate(N * K, ws, total_ms)

    # backward pass (gradient through the same projector, and dL/dA), timed
    # apart from the forward step: one call each per iteration, CUDA events
    gxh = to_dev(synth.make_boundary_grad(w, n_tokens=N))
    gZ = torch.empty(N, w.r, dtype=torch.bfloat16, device="cuda")
    gX = torch.empty(N, w.d, dtype=torch.bfloat16, device="cuda")
    Zb = torch.empty(N, w.r, dtype=torch.bfloat16, device="cuda")
    dA = torch.empty(w.d, w.r, dtype=torch.float32, device="cuda")
    bw_calls = [
        ("grad_compress_us", lambda: mapl.mapl_grad_compress(plan, gxh, gZ, stream)),
        ("grad_decompress_us", lambda: mapl.mapl_grad_decompress(plan, gZ, gX, stream)),
        ("grad_A_us", lambda: mapl.mapl_grad_A(plan, x0, t, E, gZ, gxh, Zb, dA, stream)),
    ]
    backward = {}
    for key, fn in bw_calls:
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        nb = 200
        b0.record(stream)
        for _ in range(nb):
            fn()
        b1.record(stream)
        torch.cuda.synchronize()
        backward[key] = b0.elapsed_time(b1) / nb * 1e3
    mapl.mapl_check(plan)

    # SPEL projector update (batch of 3 boundaries, St(1024, 256) and
    # St(2048, 256), fp32) and the plan refresh after an A update
    from pipeline_activation_compression_gb300 import polar
    spel = {}
    co = polar.default_coeffs(5, 5)
    for sname in ("spel_d1024_r256", "spel_d2048_r256"):
        sw = synth.SPEL_WORKLOADS[sname]
        sp = synth.make_spel(sw)
        As = torch.from_numpy(sp["A"]).cuda()
        ms = torch.zeros_like(As)
        Gs = torch.from_numpy(next(synth.spel_gradients(sw))).cuda()
        wsp_s = torch.empty(mapl.mapl_spel_workspace_size(sw.d, sw.r, sw.batch) // 4 + 64,
                            dtype=torch.float32, device="cuda")
        for _ in range(3):
            mapl.mapl_spel_step(As, Gs, ms, sw.lr, sw.beta, co, 5, 5, wsp_s, stream)
        torch.cuda.synchronize()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ns = 50
        s0.record(stream)
        for _ in range(ns):
            mapl.mapl_spel_step(As, Gs, ms, sw.lr, sw.beta, co, 5, 5, wsp_s, stream)
        s1.record(stream)
        torch.cuda.synchronize()
        spel[sname + "_us"] = s0.elapsed_time(s1) / ns * 1e3
        if sname == "spel_d1024_r256":
            # the projector broadcast: three bf16 plans of this (d, r)
            # refreshed by the step itself, against the step followed by one
            # mapl_plan_update_A per boundary
            wr = synth.WORKLOADS["proj_d1024_r256"]
            br = synth.make_boundary(wr, n_tokens=8)
            cfg_r = mapl.make_config(wr.d, wr.r, wr.V, dtype=mapl.MAPL_BF16)
            plans_r = [mapl.mapl_plan_create(cfg_r, to_dev(br["A"]), to_dev(br["P"]),
                                             to_dev(br["P_next"])) for _ in range(sw.batch)]
            Ab = torch.empty(sw.batch, sw.d, sw.r, dtype=torch.bfloat16, device="cuda")

            def separate():
                mapl.mapl_spel_step(As, Gs, ms, sw.lr, sw.beta, co, 5, 5, wsp_s, stream)
                Ab.copy_(As)
                for q in range(sw.batch):
                    mapl.mapl_plan_update_A(plans_r[q], Ab[q], stream)

            def fused():
                mapl.mapl_spel_step_refresh(As, Gs, ms, sw.lr, sw.beta, co, 5, 5, plans_r,
                                            wsp_s, stream)

            for key, fn in (("spel_then_update_A_x3_us", separate),
                            ("spel_step_refresh_x3_us", fused)):
                for _ in range(3):
                    fn()
                torch.cuda.synchronize()
                s0.record(stream)
                for _ in range(ns):
                    fn()
                s1.record(stream)
                torch.cuda.synchronize()
                spel[key] = s0.elapsed_time(s1) / ns * 1e3
            for pr in plans_r:
                pr.destroy()
    A_dev = to_dev(b["A"])
    for _ in range(3):
        mapl.mapl_plan_update_A(plan, A_dev, stream)
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for _ in range(20):
        mapl.mapl_plan_update_A(plan, A_dev, stream)
    s1.record(stream)
    torch.cuda.synchronize()
    spel["plan_update_A_us"] = s0.elapsed_time(s1) / 20 * 1e3
    spel["note"] = ("one SPEL step for a batch of 3 boundaries (5 LMO + 5 retraction "
                    "PolarExpress iterations, fp32); plan refresh after an A update; the "
                    "step with the projector broadcast to 3 bf16 plans, separate vs fused")
    mapl.mapl_check(plan)

    # first-boundary anchor (the full token embedding E_emb, V x d): the same
    # workload with X = E_emb[tids] + signal, compress and decompress timed
    # apart with CUDA events over rotating buffer sets
    first = {}
    if w.dtype == "bf16" and 3 * w.r <= 512:
        be = synth.make_first_boundary(w, seed=rank, n_tokens=N)
        Pz = torch.zeros(w.r, w.d, dtype=torch.bfloat16, device="cuda")
        plan_e = mapl.mapl_plan_create(cfg, to_dev(be["A"]), Pz, Pz,
                                       to_dev(be["C"]) if w.vq else None)
        Ee = to_dev(be["E_emb"])
        mapl.mapl_plan_set_embedding_anchor(plan_e, Ee, stream)
        te = to_dev(be["tids"])
        xe = to_dev(be["X"])
        for k in range(nsets):
            Xs[k].copy_(xe)
        ne = 50
        for i in range(3):
            mapl.mapl_compress(plan_e, Xs[i % nsets], te, None, pay[i % nsets], stream)
            mapl.mapl_decompress(plan_e, pay[i % nsets], te, None, Xh[i % nsets], stream)
        torch.cuda.synchronize()
        fe = [torch.cuda.Event(enable_timing=True) for _ in range(2 * ne + 1)]
        fe[0].record(stream)
        for i in range(ne):
            k = i % nsets
            mapl.mapl_compress(plan_e, Xs[k], te, None, pay[k], stream)
            fe[2 * i + 1].record(stream)
            mapl.mapl_decompress(plan_e, pay[k], te, None, Xh[k], stream)
            fe[2 * i + 2].record(stream)
        torch.cuda.synchronize()
        mapl.mapl_check(plan_e)
        first = {
            "mapl_compress_us": float(np.mean([fe[2 * i].elapsed_time(fe[2 * i + 1])
                                               for i in range(ne)])) * 1e3,
            "mapl_decompress_us": float(np.mean([fe[2 * i + 1].elapsed_time(fe[2 * i + 2])
                                                 for i in range(ne)])) * 1e3,
            "tokens_per_s": N * ne / (fe[0].elapsed_time(fe[2 * ne]) * 1e-3),
        }
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        A_e = to_dev(be["A"])
        for _ in range(2):
            mapl.mapl_plan_update_A(plan_e, A_e, stream)
        s0.record(stream)
        for _ in range(10):
            mapl.mapl_plan_update_A(plan_e, A_e, stream)
        s1.record(stream)
        torch.cuda.synchronize()
        first["plan_update_A_us"] = s0.elapsed_time(s1) / 10 * 1e3
        first["note"] = ("anchor = token embedding (Fig. 2), Z = (X - E_emb[t]) A, "
                         "X_hat = Z_hat A^T + E_emb[t]; update_A includes the E_emb A table")
        plan_e.destroy()

    # CPU baseline: the oracle as it stands, bounded sample
    cps, done, el = (0.0, 0, 0.0) if args.skip_cpu else time_oracle(b, w, min(1024, N), 10.0)
    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "d": w.d, "r": w.r, "V": w.V, "G": w.G, "R": w.R,
                   "K": w.K, "tokens_per_step": N,
                   "micro_batch": f"{w.B}x{w.T}" if N == w.N else f"{N} tokens",
                   "payload_bytes_per_token": w.R * w.G if w.vq else 2 * w.r,
                   "l2": f"{nsets} rotating input/output sets ({2 * nsets * xbytes >> 20} MiB) > L2",
                   "step": "mapl_compress + mapl_decompress on one stream"},
        "kernels": {"mapl_compress_us": comp_avg * 1e3, "mapl_decompress_us": dec_avg * 1e3,
                    "step_GBps": step_bytes / (total_ms / K * 1e-3) / 1e9,
                    "unique_token_rows": U,
                    "x_hat_fill_us": fill_ms * 1e3,
                    "x_hat_fill_GBps": N * w.d * 2 / (fill_ms * 1e-3) / 1e9,
                    "decompress_vs_fill": fill_ms / dec_avg,
                    "fill_note": "torch fill_ of the same rotating X_hat buffers (writes "
                                 "only), timed after the step loop: the device's plain write "
                                 "rate, the floor under decompress"},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "algorithmic_bytes_per_launch": dom_bytes,
                     "traffic": profiled_traffic(dom, w.name),
                     "step_frac": (step_bytes / (total_ms / K * 1e-3) / 1e9) / peak},
        "e2e": {"value": whole_job_rate(N * Ke, ws, e2e_ms), "unit": UNIT,
                "h2d_bytes_per_step": int(xh_host.numel() * 2 + 2 * t_host.numel() * 4
                                          + pay_h[0].numel() * pay_h[0].element_size()),
                "d2h_bytes_per_step": int(out_h[0].numel() * 2
                                          + pay_h[0].numel() * pay_h[0].element_size()),
                "api": "mapl_compress_host + mapl_decompress_host, steps rotating "
                       "over six streams"},
        "backward": dict(backward, note="gZ = dL/dX_hat A, dL/dX = gZ A^T, dL/dA; same "
                         "workload, 200 calls each, inputs L2-warm"),
        "spel": spel,
        "first_boundary": first,
        "cuda_graph": {"value": whole_job_rate(N, ws, graph_ms), "unit": UNIT,
                       "ms_per_step": graph_ms, "steps": reps * nsets,
                       "note": "compress + decompress captured once per buffer set, replayed"},
        "gpu_launches": 2 * K,
        "cpu_baseline": {"value": cps, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                         "sample": f"{done} tokens of {w.name} in chunks of 1024 random rows, "
                                   f"{el:.1f} s (numpy fp64; BLAS threads for the GEMMs, "
                                   f"VQ search single-threaded)"},
    }
    if clk is not None:
        res["clocks"] = clk
    return res


# ---------------------------------------------------------- reference arm
def run_reference(args, ws, rank):
    from pipeline_activation_compression_gb300 import synth
    if rank != 0:
        return None
    w = synth.WORKLOADS[args.workload]
    b = synth.make_boundary(w, n_tokens=min(w.N, 8192))
    # per-token cost, then a per-step sample that keeps the run within minutes
    rate, _, _ = time_oracle(b, w, 256, 2.0)
    budget = 120.0
    per_step = int(max(1, min(1024, rate * budget / max(1, args.steps + args.warmup))))
    rng = np.random.default_rng(1)
    for _ in range(args.warmup):
        oracle_step(b, w, np.sort(rng.choice(b["tids"].size, per_step, replace=False)))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(b, w, np.sort(rng.choice(b["tids"].size, per_step, replace=False)))
    el = time.perf_counter() - t0
    value = per_step * args.steps / el
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "d": w.d, "r": w.r, "G": w.G, "R": w.R, "K": w.K,
                   "tokens_per_step": per_step},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                         "sample": f"{per_step} random tokens of {w.name} per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    ws, rank = dist_setup(args) if args.impl == "ours" else (
        int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")))
    if args.gpus != ws and ws > 1:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE {ws}")
    res = run_ours(args, ws, rank) if args.impl == "ours" else run_reference(args, ws, rank)
    if res is not None and rank == 0:
        print(json.dumps(res), flush=True)
    if ws > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
