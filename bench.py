"""Throughput benchmark of the chunk-forward kkt_solve step on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config NAME]

One step = one kkt_solve over the whole workload ((2, 16384, 32, 128), bf16 keys,
bf16 output by default) with inputs already resident in HBM.  The default
step's inputs and output (409 MB) exceed twice the 129 MB L2, so it is timed
back to back; a smaller workload is timed cold (a 512 MiB buffer is written
before each step, and only the steps are timed).  Prints one JSON line (rank 0).  Under torchrun every rank runs the same
workload on its own GPU (independent replicas: weak scaling, no data-path
collective); timing is the max over ranks.

--impl reference times the plain fp64 CPU oracle on the host cores instead (it
is the only other implementation of this step that exists here), each step a
bounded sample of tiles of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "token-heads/s and achieved HBM GB/s (% of GB300 peak) for kkt_solve, 1 GPU"
UNIT = "token-heads/s"
# Ascend 910B fused time for (2,16384,32,128) from the MindSpeed-Ops PR page's
# performance table: 4.9368 ms -> 1,048,576 token-heads / 4.9368 ms.
PAGE_FUSED_MS = {"B2_T16384_H32_K128": 4.9368}
NOMINAL_HBM_GBS = 8000.0             # GB300 HBM3e nominal (~8 TB/s), for the second fraction
L2_BYTES = 129 * 10**6               # GB300 L2 (two dies together)
L2_FLUSH_BYTES = 512 << 20           # written before each step of a small workload
SM_MAX_HZ = 2.07e9                   # GB300 maximum SM clock: turns a hold time into spin cycles


ELEM_BYTES = {"bf16": 2, "f16": 2, "f32": 4}


def bytes_per_token_head(wl, out_dtype: str) -> int:
    """Algorithmic HBM bytes per token-head: read k (K values), g (fp32), beta;
    write one output row of `chunk` values."""
    b = wl.K * ELEM_BYTES[wl.k_dtype]
    b += 4 if wl.use_g else 0
    b += ELEM_BYTES[wl.beta_dtype] if wl.use_beta else 0
    b += wl.chunk * ELEM_BYTES[out_dtype]
    return b


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_sha() -> str:
    """Hash of the kernel source file (the kernels, their launch code and the C
    entry points): a recorded ncu figure holds for this hash only."""
    import hashlib
    with open(os.path.join(ROOT, "gated_deltanet_chunked_gdr_gb300/csrc/gdr_kkt_solve.cu"), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(wl, out_dtype: str):
    """DRAM bytes per launch (read + write) from the committed ncu summary, or
    None when it was taken on another kernel source or another workload."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f).get(f"{wl.name}:{out_dtype}")
    if not d or d.get("source_sha") != kernel_source_sha():
        return None
    return d.get("dram_bytes_per_launch")


HOLD_LAUNCHES = 256                  # launches queued behind a hold (well inside the launch queue)
HOLD_MAX_S = 0.5


def hold_time(host_s_per_call: float, launches: int) -> float:
    """A hold long enough for the host to queue min(launches, HOLD_LAUNCHES) calls
    (four times the measured host time per call, plus 2 ms), at most HOLD_MAX_S.
    Beyond those, the host keeps ahead of a GPU that runs them back to back."""
    return min(HOLD_MAX_S, 2e-3 + 4 * host_s_per_call * min(launches, HOLD_LAUNCHES))


def hold_stream(stream, seconds: float) -> None:
    """Hold `stream` with a delay kernel of about `seconds` (torch's spin kernel), so
    that the launches queued behind it run back to back: the host's per-call latency
    is then not part of a device-timed region, whose first event follows the hold."""
    import torch
    with torch.cuda.stream(stream):
        torch.cuda._sleep(max(1, int(seconds * SM_MAX_HZ)))


def reduce_max(x: float, ws: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity when ws == 1)."""
    if ws <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(token_heads_per_rank: int, ms_per_step_max: float, ws: int) -> float:
    """Whole-job throughput: every rank processes its own copy of the workload."""
    return ws * token_heads_per_rank / (ms_per_step_max * 1e-3)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi clocks/throttle sampling while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str, path: str | None):
        self.proc = None
        self.path = path
        self.gpu_id = gpu_id

    def start(self):
        try:
            f = open(self.path, "w") if self.path else subprocess.PIPE
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=f, stderr=subprocess.DEVNULL, text=True)
            self._file = f if self.path else None
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        if self._file:
            self._file.close()
            out = open(self.path).read()
        rows = [r.split(",") for r in (out or "").strip().splitlines() if r.strip()]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for nm, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def run_reference(args, wl):
    """Reference arm: the fp64 CPU oracle, as it stands, on the host cores.  Each
    step is the oracle's whole-tensor call (heads split over the host cores) on
    the workload, or on a token prefix of it when K whole-workload steps would
    take more than about a minute."""
    import oracle
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    inp = workloads.make_inputs(wl)
    threads = min(os.cpu_count() or 1, wl.H)
    lead = inp["k"].shape[:2]
    ntok = lead[0] * lead[1]
    flat = {x: None if inp[x] is None else inp[x].reshape(1, ntok, *inp[x].shape[2:])
            for x in ("k", "g", "beta")}
    cu = inp["cu_seqlens"]
    if cu is None:      # fixed-length sequences, flattened: one packed batch of B sequences
        cu = np.arange(wl.B + 1, dtype=np.int32) * wl.T

    def run(rows):
        # Whole sequences up to `rows` tokens (the last one cut at `rows`).
        c = np.minimum(np.asarray(cu, dtype=np.int64), rows).astype(np.int32)
        oracle.kkt_solve_ref(flat["k"][:, :rows], None if flat["g"] is None else flat["g"][:, :rows],
                             None if flat["beta"] is None else flat["beta"][:, :rows], c,
                             chunk_size=wl.chunk, threads=threads)
        return int(c[-1]) * wl.H

    t0 = time.perf_counter()
    run(ntok)
    t_whole = time.perf_counter() - t0
    rows = ntok
    if t_whole * args.steps > 60.0:
        rows = max(wl.chunk, int(ntok * 60.0 / (t_whole * args.steps)) // wl.chunk * wl.chunk)
    for _ in range(args.warmup):
        run(rows)
    th = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        th += run(rows)
    dt = time.perf_counter() - t0
    value = th / dt
    sample = (f"the whole {wl.name} workload per step" if rows == ntok else
              f"the first {rows} of {ntok} token rows of {wl.name}, all heads, per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "T": wl.T, "H": wl.H, "K": wl.K, "chunk": wl.chunk,
                   "impl": "plain C fp64 oracle, heads split over host threads",
                   "token_rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _oracle_prefix(wl, inp, budget_s: float, threads: int):
    """The oracle's whole-tensor call (heads split over `threads` host threads,
    each running the plain C loop) on growing token prefixes of the first
    sequence, all heads, until about `budget_s` seconds of work is done."""
    import oracle
    s, e = workloads._sequence_bounds(wl)[0]
    kf = inp["k"].reshape(-1, wl.H, wl.K)
    gf = None if inp["g"] is None else inp["g"].reshape(-1, wl.H)
    bf = None if inp["beta"] is None else inp["beta"].reshape(-1, wl.H)
    rows, th, dt = min(wl.chunk, e - s), 0, 0.0
    while True:
        sl = slice(s, s + rows)
        t0 = time.perf_counter()
        oracle.kkt_solve_ref(kf[sl].unsqueeze(0), None if gf is None else gf[sl].unsqueeze(0),
                             None if bf is None else bf[sl].unsqueeze(0), chunk_size=wl.chunk, threads=threads)
        t = time.perf_counter() - t0
        th, dt = rows * wl.H, t
        if t >= budget_s / 4 or rows >= e - s:
            return rows, th, dt
        rows = min(e - s, rows * max(2, int(budget_s / 4 / max(t, 1e-3))) // wl.chunk * wl.chunk or wl.chunk)


def _oracle_whole(wl, inp, budget_s: float, threads: int):
    """The oracle's whole-tensor call on the entire workload, repeated until
    about `budget_s` seconds have passed (at least once)."""
    import oracle
    n, t0 = 0, time.perf_counter()
    while True:
        oracle.kkt_solve_ref(inp["k"], inp["g"], inp["beta"], inp["cu_seqlens"], chunk_size=wl.chunk,
                             threads=threads)
        n += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s or dt / n * (n + 1) > 1.5 * budget_s:
            return n, n * wl.token_heads, dt


def cpu_baseline(wl, inp, budget_s: float):
    """The oracle, as it stands, timed on the host: its whole-tensor call (heads
    split over the host cores, each thread running the plain C loop) on the
    entire workload, and on one core on a token prefix of the first sequence."""
    threads = min(os.cpu_count() or 1, wl.H)
    n, th, dt = _oracle_whole(wl, inp, budget_s / 2, threads)
    rows1, th1, dt1 = _oracle_prefix(wl, inp, budget_s / 2, 1)
    return {"value": th / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"the whole {wl.name} workload x {n} ({th} token-heads) in {dt:.2f} s, "
                      f"heads split over {threads} threads",
            "single_thread": {"value": th1 / dt1, "unit": UNIT, "cores": 1,
                              "sample": f"first {rows1} tokens x {wl.H} heads ({th1} token-heads) in {dt1:.2f} s"}}


def small_workload_lines(dev, stream, gdr, launches: int):
    """Cold-L2 timings of the smaller workloads, each through the same C-ABI call:
    a 512 MiB buffer is written before every launch, an event pair times the
    launch alone; the median is reported, with the warm back-to-back mean."""
    import torch
    codes = {"bf16": gdr.GDR_BF16, "f16": gdr.GDR_F16, "f32": gdr.GDR_F32}
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    lines = {}
    for name, out_dtype in (("B1_T256_H8_K128", "f32"), ("B2_T2000_H5_K128", "f32"),
                            ("B1_T8192_H8_K128", "bf16"), ("B1_T8192_H8_K128", "f32"),
                            ("varlen8_H16_K128", "f32")):
        wl = workloads.CONFIGS[name]
        inp = workloads.make_inputs(wl)
        k, g, beta = (inp[x].to(dev) for x in ("k", "g", "beta"))
        cu = None if inp["cu_seqlens"] is None else inp["cu_seqlens"].to(dev)
        B = wl.B
        odt = {"bf16": torch.bfloat16, "f32": torch.float32}[out_dtype]
        out = torch.empty((*k.shape[:3], 64), dtype=odt, device=dev)

        def step():
            rc = gdr.kkt_solve_ex_raw(k.data_ptr(), codes[wl.k_dtype], g.data_ptr(), beta.data_ptr(),
                                      codes[wl.beta_dtype], 0 if cu is None else cu.data_ptr(), B, k.shape[1],
                                      wl.H, wl.K, 64, codes[out_dtype], out.data_ptr(), stream.cuda_stream)
            if rc != gdr.GDR_OK:
                raise gdr.GdrError(rc, "gdr_kkt_solve_ex")

        for _ in range(5):
            step()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(launches)]
        with torch.cuda.stream(stream):
            for a, b in evs:
                flush.fill_(1.0)
                a.record(stream)
                step()
                b.record(stream)
            w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            hold_stream(stream, 2e-3 + 1e-4 * launches)
            w0.record(stream)
            for _ in range(launches):
                step()
            w1.record(stream)
        torch.cuda.synchronize(dev)
        us = sorted(a.elapsed_time(b) * 1e3 for a, b in evs)
        med = statistics.median(us)
        th = wl.token_heads
        lines[f"{name}:{out_dtype}"] = {
            "token_heads": th, "cold_median_us": med, "cold_p10_us": us[int(0.1 * (len(us) - 1))],
            "cold_p90_us": us[int(0.9 * (len(us) - 1))], "warm_mean_us": w0.elapsed_time(w1) * 1e3 / launches,
            "value": th / (med * 1e-6), "unit": UNIT,
            "hbm_gbs_cold": th * bytes_per_token_head(wl, out_dtype) / (med * 1e-6) / 1e9,
            "launches": launches}
    if gdr.device_status() != gdr.GDR_OK:
        raise RuntimeError("device status not ok after the small workloads")
    return lines


def link_bound(dev, tensors_h2d, tensors_d2h, reps: int = 5):
    """Plain page-locked copies of the step's own bytes, one cudaMemcpyAsync per
    tensor (torch's non-blocking copy): host-to-device alone, device-to-host
    alone, and both at once on two streams.  The concurrent time is the bound an
    end-to-end step can reach with perfect overlap of copies and kernel."""
    import torch
    dsts = [torch.empty_like(t, device=dev) for t in tensors_h2d]
    srcs = [torch.empty_like(t, device=dev) for t in tensors_d2h]
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def h2d(s):
        with torch.cuda.stream(s):
            for d, h in zip(dsts, tensors_h2d):
                d.copy_(h, non_blocking=True)

    def d2h(s):
        with torch.cuda.stream(s):
            for h, d in zip(tensors_d2h, srcs):
                h.copy_(d, non_blocking=True)

    def timed(fn):
        best = float("inf")
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize(dev)
            best = min(best, time.perf_counter() - t0)
        return best * 1e3

    bi = sum(t.numel() * t.element_size() for t in tensors_h2d)
    bo = sum(t.numel() * t.element_size() for t in tensors_d2h)
    ms_in = timed(lambda: h2d(s1))
    ms_out = timed(lambda: d2h(s2))
    ms_both = timed(lambda: (h2d(s1), d2h(s2)))
    return {"h2d_gbs": bi / (ms_in * 1e-3) / 1e9, "d2h_gbs": bo / (ms_out * 1e-3) / 1e9,
            "h2d_ms": ms_in, "d2h_ms": ms_out, "both_ms": ms_both,
            "link_gbs": (bi + bo) / (ms_both * 1e-3) / 1e9,
            "how": "best of %d host-timed runs of one cudaMemcpyAsync per tensor, page-locked" % reps}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="B2_T16384_H32_K128", choices=sorted(workloads.CONFIGS))
    ap.add_argument("--out-dtype", default=None, choices=["f32", "bf16", "f16"])
    ap.add_argument("--K", type=int, default=None, choices=[64, 128, 192, 256],
                    help="head dimension (default: the workload's, 128)")
    ap.add_argument("--k-dtype", default="bf16", choices=["bf16", "f16", "f32"])
    ap.add_argument("--chunk", type=int, default=64, choices=[64, 128])
    ap.add_argument("--beta-dtype", default="bf16", choices=["bf16", "f16", "f32"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clocks-csv", default=None)
    ap.add_argument("--no-small-workloads", action="store_true",
                    help="skip the cold-L2 timings of the smaller workloads (per_config)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    wl = workloads.CONFIGS[args.config]
    if args.K is not None and args.K != wl.K:
        wl = wl.with_(K=args.K, name=wl.name.replace(f"_K{wl.K}", f"_K{args.K}"))
    if args.k_dtype != wl.k_dtype or args.beta_dtype != wl.beta_dtype:
        wl = wl.with_(k_dtype=args.k_dtype, beta_dtype=args.beta_dtype,
                      name=f"{wl.name}_k{args.k_dtype}_beta{args.beta_dtype}")
    if args.chunk != wl.chunk:
        wl = wl.with_(chunk=args.chunk, name=f"{wl.name}_C{args.chunk}")
    out_dtype = args.out_dtype or wl.out_dtype
    if args.impl == "reference":
        return run_reference(args, wl)

    import torch
    import gated_deltanet_chunked_gdr_gb300 as gdr

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)

    inp = workloads.make_inputs(wl)
    k = inp["k"].to(dev)
    g = None if inp["g"] is None else inp["g"].to(dev)
    beta = None if inp["beta"] is None else inp["beta"].to(dev)
    cu = None if inp["cu_seqlens"] is None else inp["cu_seqlens"].to(dev)
    odt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[out_dtype]
    codes = {"bf16": gdr.GDR_BF16, "f16": gdr.GDR_F16, "f32": gdr.GDR_F32}
    out = torch.empty((*k.shape[:3], wl.chunk), dtype=odt, device=dev)
    stream = torch.cuda.Stream(dev)
    sh = stream.cuda_stream
    B = cu.numel() - 1 if cu is not None else k.shape[0]

    def step(o=out):
        rc = gdr.kkt_solve_ex_raw(k.data_ptr(), codes[wl.k_dtype], 0 if g is None else g.data_ptr(),
                                  0 if beta is None else beta.data_ptr(), codes[wl.beta_dtype],
                                  0 if cu is None else cu.data_ptr(), B, k.shape[1], wl.H, wl.K, wl.chunk,
                                  codes[out_dtype], o.data_ptr(), sh)
        if rc != gdr.GDR_OK:
            raise gdr.GdrError(rc, "gdr_kkt_solve_ex")

    def barrier():
        if ws > 1:
            torch.distributed.barrier()

    t_enq = []
    for _ in range(args.warmup):
        t0 = time.perf_counter()
        step()
        t_enq.append(time.perf_counter() - t0)
    enqueue_s = statistics.median(t_enq)                       # host time per call
    torch.cuda.synchronize(dev)
    if gdr.device_status() != gdr.GDR_OK:
        raise RuntimeError("device status not ok after warm-up")

    props = torch.cuda.get_device_properties(dev)
    gpu_id = str(getattr(props, "uuid", "") or "")
    gpu_id = ("GPU-" + gpu_id) if gpu_id and not gpu_id.startswith("GPU-") else (gpu_id or str(local))
    sampler = ClockSampler(gpu_id, args.clocks_csv if rank == 0 else None)
    th_rank = wl.token_heads
    step_bytes = th_rank * bytes_per_token_head(wl, out_dtype)
    # A step whose inputs and output fit in L2 would be timed warm: then a
    # buffer larger than L2 is written before every step and only the step
    # itself is timed, with a pair of events around each launch.
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev) \
        if step_bytes < 2 * L2_BYTES else None
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    per_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps)] if flush is not None else []
    barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)                                  # let the sampler start
    # Back-to-back steps are queued behind a hold long enough for the host to
    # enqueue the first HOLD_LAUNCHES of them (checked: the region's first event
    # must still be pending by then, else the hold is lengthened and the region
    # timed again); past those the host stays ahead of the GPU.
    hold_s, queued = hold_time(enqueue_s, args.steps), flush is not None
    for _attempt in range(3):
        if flush is None:
            hold_stream(stream, hold_s)
        ev0.record(stream)
        if flush is None:
            for n in range(args.steps):
                step()
                if n + 1 == min(args.steps, HOLD_LAUNCHES):
                    queued = not ev0.query()
        else:
            with torch.cuda.stream(stream):
                for a, b in per_step:
                    flush.fill_(1.0)
                    a.record(stream)
                    step()
                    b.record(stream)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        if queued:
            break
        hold_s = min(HOLD_MAX_S, 4 * hold_s)
    barrier()
    clocks = sampler.stop()
    if flush is None:
        ms_total = ev0.elapsed_time(ev1)
    else:
        ms_total = sum(a.elapsed_time(b) for a, b in per_step)
    ms_total = reduce_max(ms_total, ws, dev)
    ms_step = ms_total / args.steps

    # Spread of single launches (median, p10, p90), each launch between its own
    # pair of events; a small workload reuses its cold per-step times and adds
    # the warm mean of back-to-back launches for comparison.
    if flush is None:
        spread_n = min(args.steps, 500)
        per_launch = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                      for _ in range(spread_n)]
        hold_stream(stream, hold_time(3 * enqueue_s, spread_n))
        for a, b in per_launch:
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize(dev)
    else:
        per_launch = per_step
    us = sorted(a.elapsed_time(b) * 1e3 for a, b in per_launch)
    launch_stats = {"launches": len(us), "l2": "cold" if flush is not None else "not flushed (> 2 x L2)",
                    "queued_behind_hold": bool(queued) if flush is None else None,
                    "host_us_per_call": enqueue_s * 1e6,
                    "median_us": statistics.median(us),
                    "p10_us": us[int(0.1 * (len(us) - 1))], "p90_us": us[int(0.9 * (len(us) - 1))]}
    if flush is not None:
        w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        hold_stream(stream, hold_time(enqueue_s, args.steps))
        w0.record(stream)
        for _ in range(args.steps):
            step()
        w1.record(stream)
        torch.cuda.synchronize(dev)
        launch_stats["warm_mean_us"] = w0.elapsed_time(w1) * 1e3 / args.steps
    flushed = flush is not None
    del flush
    value = aggregate_value(th_rank, ms_step, ws)
    if gdr.device_status() != gdr.GDR_OK:
        raise RuntimeError("device status not ok after the timed region")

    # The unfused chain on the same inputs (A through HBM, two launches), timed
    # the same way: what the fusion saves on this GPU.
    A = torch.empty((*k.shape[:3], 64), dtype=torch.float32, device=dev)

    def kkt_half():
        rc = gdr.chunk_scaled_dot_kkt_raw(k.data_ptr(), codes[wl.k_dtype], 0 if g is None else g.data_ptr(),
                                          0 if beta is None else beta.data_ptr(), codes[wl.beta_dtype],
                                          0 if cu is None else cu.data_ptr(), B, k.shape[1], wl.H, wl.K,
                                          64, A.data_ptr(), sh)
        if rc != gdr.GDR_OK:
            raise gdr.GdrError(rc, "gdr_chunk_scaled_dot_kkt")

    def solve_half():
        rc = gdr.solve_tril_raw(A.data_ptr(), 0 if cu is None else cu.data_ptr(), B, k.shape[1], wl.H,
                                64, codes[out_dtype], out.data_ptr(), sh)
        if rc != gdr.GDR_OK:
            raise gdr.GdrError(rc, "gdr_solve_tril")

    chain_steps = max(10, min(args.steps, 2000))
    chain_ms = {}
    chain_runs = (("chain", (kkt_half, solve_half)), ("kkt", (kkt_half,)), ("solve", (solve_half,)))
    for name, fns in (chain_runs if wl.chunk == 64 and wl.k_dtype != "f32" else ()):
        for _ in range(3):
            for f in fns:
                f()
        torch.cuda.synchronize(dev)
        barrier()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        hold_stream(stream, hold_time(enqueue_s * len(fns), chain_steps))
        c0.record(stream)
        for _ in range(chain_steps):
            for f in fns:
                f()
        c1.record(stream)
        torch.cuda.synchronize(dev)
        chain_ms[name] = reduce_max(c0.elapsed_time(c1) / chain_steps, ws, dev)
    if gdr.device_status() != gdr.GDR_OK:
        raise RuntimeError("device status not ok after the unfused chain")
    del A
    if wl.chunk != 64 or wl.k_dtype == "f32":       # the chain takes 16-bit keys and chunk 64
        chain_ms = None

    # End to end through the C ABI's host-buffer call (gdr_kkt_solve_host): the
    # step's inputs in page-locked host memory, the output back in host memory;
    # the call copies them slice by slice over two streams around the kernel.
    # The device workspace is allocated once, outside the timed region.
    hk = inp["k"].pin_memory()
    hg = None if inp["g"] is None else inp["g"].pin_memory()
    hb = None if inp["beta"] is None else inp["beta"].pin_memory()
    hcu = None if inp["cu_seqlens"] is None else inp["cu_seqlens"].pin_memory()
    hout = torch.empty(out.shape, dtype=odt).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hk, hg, hb, hcu) if t is not None)
    d2h = hout.numel() * hout.element_size()
    e2e_ws = torch.empty(gdr.kkt_solve_host_workspace_bytes(codes[wl.k_dtype], B, k.shape[1], wl.H, wl.K,
                                                            wl.chunk, codes[out_dtype]),
                         dtype=torch.uint8, device=dev)

    def e2e_step():
        gdr.kkt_solve_host(hk, hg, hb, hcu, chunk_size=wl.chunk, output_dtype=odt, out=hout, workspace=e2e_ws,
                           stream=sh, device=dev)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = reduce_max(e0.elapsed_time(e1) / args.e2e_steps, ws, dev)
    barrier()
    link = link_bound(dev, [t for t in (hk, hg, hb, hcu) if t is not None], [hout])
    del e2e_ws
    default_line = (args.config == "B2_T16384_H32_K128" and wl.K == 128 and wl.chunk == 64
                    and wl.k_dtype == "bf16" and out_dtype == "bf16")
    per_config = (small_workload_lines(dev, stream, gdr, 50)
                  if default_line and not args.no_small_workloads else None)

    if rank == 0:
        peak, peak_kind = measured_peaks()
        bpt = bytes_per_token_head(wl, out_dtype)
        achieved = th_rank * bpt / (ms_step * 1e-3) / 1e9
        traffic = recorded_traffic(wl, out_dtype)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": (value / (th_rank / (PAGE_FUSED_MS[args.config] * 1e-3))
                            if args.config in PAGE_FUSED_MS and wl.K == 128 else None),
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": wl.name, "B": wl.B, "T": wl.T, "H": wl.H, "K": wl.K,
                       "chunk": wl.chunk, "k": wl.k_dtype, "g": "f32", "beta": wl.beta_dtype,
                       "out": out_dtype,
                       "compute": f"Gram {wl.k_dtype}x{wl.k_dtype}->f32 (tcgen05), gate/solve f32",
                       "l2": (f"no flush: inputs+output {step_bytes / 1e6:.0f} MB/step > 2 x L2"
                              if step_bytes >= 2 * L2_BYTES else
                              f"L2 flushed before every step ({L2_FLUSH_BYTES >> 20} MiB write); "
                              "only the step is timed (events around each launch)"),
                       "timing": ("CUDA events around the K launches, queued back to back behind a "
                                  "delay kernel (host call latency not timed)" if not flushed else
                                  "CUDA events around each launch"),
                       "parallelism": f"replicas x{ws} (independent tiles, no collective)",
                       "vs_baseline_ref": "Ascend 910B fused Triton time from the PR page table"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_kind": f"{peak_kind} hbm_gbs (copy)",
                         "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                         "nominal_peak": NOMINAL_HBM_GBS,
                         "bytes_per_token_head": bpt},
            "e2e": {"value": aggregate_value(th_rank, e2e_ms, ws), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms,
                    "call": "gdr_kkt_solve_host: page-locked host buffers, copies pipelined over two streams",
                    "link": link, "link_gbs": link["link_gbs"],
                    "of_link_bound": link["both_ms"] / e2e_ms},
            "per_config": per_config,
            "gpu_launches": args.steps,
            "launch_stats": launch_stats,
            "clocks": clocks,
            "unfused_chain": None if chain_ms is None else {
                "what": "gdr_chunk_scaled_dot_kkt then gdr_solve_tril (A fp32 through HBM), same inputs",
                "value": aggregate_value(th_rank, chain_ms["chain"], ws), "unit": UNIT,
                "ms_per_step": chain_ms["chain"], "steps": chain_steps, "launches_per_step": 2,
                "kkt_ms": chain_ms["kkt"], "solve_ms": chain_ms["solve"],
                "bytes_per_token_head": bpt + 2 * 64 * 4,
                "fused_speedup": chain_ms["chain"] / ms_step,
            },
        }
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(wl, inp, args.cpu_budget)
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
