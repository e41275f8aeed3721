"""Benchmark of the HC gated residual on GB300 (one JSON line on rank 0).

Workload (one "step"): the decode sweep -- one forward call at each of
M = 2, 4, 8, 16, 32 tokens, HC=4, HS=2560 (K=10240), r=320, bf16, seeded
synthetic inputs (weights ~ N(0, 1/sqrt(fan-in)), Wnorm ~ N(0, 0.1), R and y
~ N(0, 1), inj ~ N(0, 2)).  value = tokens per second over K timed steps.

Timing: the device-side number replays one CUDA graph per step (the five
calls), rotating over NSETS distinct weight+activation sets whose total
footprint exceeds twice the L2, so weights stream from HBM on every call.
The e2e number calls the public API eagerly with pinned host inputs copied in
and every output copied back inside the timed region.  Also reported: the
per-M latency table, the roofline of the decode kernel against the measured
HBM peak, SM clocks sampled during the timed region, and the fp64 CPU oracle
timed on a bounded sample (cpu_baseline).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

SWEEP = (2, 4, 8, 16, 32)
LAT_MS = (1,) + SWEEP      # per-M latency table: the single-token call as well
HC, HS, R_LOW = 4, 2560, 320
K_DIM = HC * HS
METRIC = "HC gated-residual µs/call & tokens/s vs M (HC4,HS2560,r320 bf16); % roofline"
WEIGHT_BYTES = 2 * (R_LOW + HC) * K_DIM + 2 * K_DIM * R_LOW + 2 * K_DIM     # Wd, Wi, Wu, Wnorm
ACT_BYTES_PER_TOKEN = (2 * K_DIM + 2 * HS + 4 * HC + 2 * K_DIM + 4 * HC + 4 * HC
                       + 4 * R_LOW + 2 * HS)                                   # R y inj R2 rrms inj_next lora x
FLOPS_PER_TOKEN = 2 * K_DIM * (R_LOW + HC + R_LOW)

# DRAM bytes (read + write) of one decode_kernel launch per M, from one ncu
# capture of this benchmark's decode calls (dram__bytes_read.sum +
# dram__bytes_write.sum; the capture's summary sits under profiles/).  They
# hold only for the kernel sources they were taken on: if those changed
# since, roofline.traffic is null and roofline.traffic_source says why.
DECODE_SOURCES = ("decode.cu", "hc_gr_internal.cuh", "tmap.h")
DECODE_TRAFFIC = {
    "sources_sha256": "cbdcd3472c86401ed797328aa1a5267fa4ec1f9d62f8a7b2f181069494d3bd4f",
    "bytes": {2: 13579691, 4: 13862656, 8: 14428501, 16: 15519147, 32: 16545536},
}


def code_only(text: str) -> str:
    """C/C++/CUDA source without comments, trailing blanks and blank lines."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(ln.rstrip() for ln in text.splitlines() if ln.strip())


def decode_sources_sha256() -> str:
    """Hash of the decode kernel's code: its sources with comments and blank
    lines removed, so that an edit of the prose alone keeps the capture."""
    import hashlib
    h = hashlib.sha256()
    for name in DECODE_SOURCES:
        with open(os.path.join(ROOT, "hyper_connection_gated_gb300", "csrc", name)) as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()


def decode_traffic_per_launch():
    """Mean measured DRAM bytes per launch over the sweep (None if the stored
    capture is stale) and a note on where the figure comes from."""
    if decode_sources_sha256() != DECODE_TRAFFIC["sources_sha256"]:
        return None, ("null: the decode kernel's sources changed since the stored ncu capture "
                      "(sources hash mismatch)")
    return (sum(DECODE_TRAFFIC["bytes"][M] for M in SWEEP) / len(SWEEP),
            "stored ncu capture of these kernel sources (dram__bytes_read.sum + "
            "dram__bytes_write.sum per launch, mean over the sweep); not measured in this run")


def max_over_ranks(value: float, world: int, device="cuda") -> float:
    """The largest of one float over all ranks (the slowest rank's time); the
    value itself on one rank."""
    if world <= 1:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_step: float, steps: int, world: int, seconds: float) -> float:
    """Whole-job units per second: every rank processes units_per_step per
    step (replicas, weak scaling), timed by the slowest rank."""
    return units_per_step * steps * world / seconds


def roofline_us(nbytes: float, flops: float, hbm_gbs: float, tflops: float):
    """Roofline time of one call (µs) and its bound: the larger of the HBM
    time for the algorithmic bytes and the tensor time for the flops."""
    t_hbm = nbytes / hbm_gbs / 1e3
    t_tc = flops / tflops / 1e6
    return (t_hbm, "hbm") if t_hbm >= t_tc else (t_tc, "tensor")


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during a region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- CPU baseline
_ORACLE_CASE = None


def _oracle_worker_init():
    """Pool worker set-up: the weights and the sweep's 32 token rows, once."""
    global _ORACLE_CASE
    from hyper_connection_gated_gb300 import inputs

    w = {k: inputs.bf16_bits_to_f64(v) for k, v in inputs.weights().items()}
    a = inputs.activations(32)
    _ORACLE_CASE = (w, inputs.bf16_bits_to_f64(a["R"]), inputs.bf16_bits_to_f64(a["y"]),
                    a["inj"].astype("f8"))


def _oracle_sweep(_: int) -> int:
    """One task of the all-cores baseline: one whole sweep (the five calls)
    through the oracle, as the single-core baseline runs it; returns tokens."""
    import oracle

    w, R, y, inj = _ORACLE_CASE
    for M in SWEEP:
        oracle.forward(R=R[:M], y=y[:M], inj=inj[:M], Wnorm=w["Wnorm"], Wd=w["Wd"], Wi=w["Wi"],
                       Wu=w["Wu"], eps=1e-6)
    return sum(SWEEP)


def _oracle_pool_run(seconds: float, cores: int) -> dict:
    """Sweeps over a spawn-started pool of `cores` single-threaded workers
    (one sweep per worker per round) until `seconds` have passed."""
    import multiprocessing

    ctx = multiprocessing.get_context("spawn")
    with ctx.Pool(cores, initializer=_oracle_worker_init) as pool:
        pool.map(_oracle_sweep, range(cores), chunksize=1)          # warm-up round
        t0, n, tok = time.perf_counter(), 0, 0
        while True:
            tok += sum(pool.map(_oracle_sweep, range(cores), chunksize=1))
            n += cores
            el = time.perf_counter() - t0
            if el >= seconds:
                break
    return {"tokens": tok, "seconds": el, "sweeps": n}


def cpu_baseline_all_cores(seconds: float = 10.0) -> dict:
    """The same oracle over every host core: independent sweeps, one per
    pool worker (one BLAS thread each) at a time, in a child process with no
    CUDA.  (One token per task reads the whole weight set for a single row
    and measured slower than one core running the batched calls.)"""
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    code = (f"import sys, json; sys.path.insert(0, {ROOT!r}); import bench; "
            f"print(json.dumps(bench._oracle_pool_run({seconds!r}, {cores!r})))")
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                         timeout=600, cwd=ROOT)
    if res.returncode != 0:
        return {"value": None, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                "error": res.stderr[-500:]}
    d = json.loads(res.stdout.strip().splitlines()[-1])
    return {"value": d["tokens"] / d["seconds"], "unit": "tokens/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{d['sweeps']} sweeps of M={list(SWEEP)} ({d['tokens']} tokens), one sweep "
                      f"per task over {cores} spawn-started workers, fp64 numpy, 1 BLAS thread "
                      f"each, {d['seconds']:.1f} s"}


def cpu_baseline(seconds: float = 12.0, max_steps: int | None = None, warmup: int = 0) -> dict:
    """The fp64 oracle, single-threaded BLAS, on the sweep's token mix.

    Runs in a child process with one BLAS thread so the core count is exact
    and no CUDA state is touched.  Repeats whole sweeps until `seconds` of
    CPU work (or max_steps sweeps) and returns tokens/s.
    """
    code = f"""
import sys, time, json
sys.path.insert(0, {ROOT!r})
import oracle
from hyper_connection_gated_gb300 import inputs
w = {{k: inputs.bf16_bits_to_f64(v) for k, v in inputs.weights().items()}}
a = inputs.activations(32)
R = inputs.bf16_bits_to_f64(a['R']); y = inputs.bf16_bits_to_f64(a['y']); inj = a['inj'].astype('f8')
sweep = {list(SWEEP)!r}
for _ in range({warmup}):
    for M in sweep:
        oracle.forward(R=R[:M], y=y[:M], inj=inj[:M], Wnorm=w['Wnorm'], Wd=w['Wd'], Wi=w['Wi'],
                       Wu=w['Wu'], eps=1e-6)
t0 = time.perf_counter(); n = 0; tok = 0
while True:
    for M in sweep:
        oracle.forward(R=R[:M], y=y[:M], inj=inj[:M], Wnorm=w['Wnorm'], Wd=w['Wd'], Wi=w['Wi'],
                       Wu=w['Wu'], eps=1e-6)
        tok += M
    n += 1
    el = time.perf_counter() - t0
    if el >= {seconds} or ({max_steps!r} is not None and n >= ({max_steps!r} or 0)):
        break
print(json.dumps({{"tokens": tok, "seconds": el, "sweeps": n}}))
"""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                         timeout=600)
    if res.returncode != 0:
        return {"value": None, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                "error": res.stderr[-500:]}
    d = json.loads(res.stdout.strip().splitlines()[-1])
    return {"value": d["tokens"] / d["seconds"], "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{d['sweeps']} sweeps of M={list(SWEEP)} ({d['tokens']} tokens), fp64 numpy, "
                      f"1 BLAS thread, {d['seconds']:.1f} s"}


# ---------------------------------------------------------------- main arm
def run_ours(args, rank, world):
    import numpy as np
    import torch

    from hyper_connection_gated_gb300 import HcGatedResidual, _native, inputs

    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 1024 * 1024)
    per_set = WEIGHT_BYTES + sum(SWEEP) * ACT_BYTES_PER_TOKEN
    nsets = max(4, int(np.ceil(2.0 * l2 / per_set)) + 1)

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to("cuda").view(torch.bfloat16)

    w = inputs.weights()
    a = inputs.activations(max(SWEEP))
    base = {k: bf(v) for k, v in w.items()}
    base.update(R=bf(a["R"]), y=bf(a["y"]), inj=torch.from_numpy(a["inj"]).cuda())
    sets = [{k: v.clone() for k, v in base.items()} for _ in range(nsets)]
    op = HcGatedResidual(max_M=max(SWEEP))
    outs = {M: [op.forward(s["R"][:M], s["y"][:M], s["inj"][:M], s["Wnorm"], s["Wu"],
                           Wd=s["Wd"], Wi=s["Wi"]) for s in sets] for M in LAT_MS}
    op.check()

    def prepared(M, j, pdl):
        s, o = sets[j], outs[M][j]
        ar = _native.Args()
        ar.pdl = 1 if pdl else 0
        ar.M, ar.HC, ar.HS, ar.r, ar.eps = M, HC, HS, R_LOW, 1e-6
        ar.R, ar.y, ar.inj, ar.ld_inj = s["R"].data_ptr(), s["y"].data_ptr(), s["inj"].data_ptr(), HC
        ar.Wnorm, ar.Wd, ar.Wi, ar.Wu = (s["Wnorm"].data_ptr(), s["Wd"].data_ptr(),
                                         s["Wi"].data_ptr(), s["Wu"].data_ptr())
        ar.R2, ar.rrms, ar.inj_next = o["R2"].data_ptr(), o["rrms"].data_ptr(), o["inj_next"].data_ptr()
        ar.x, ar.lora = o["x"].data_ptr(), o["lora"].data_ptr()
        return ar

    # pdl: each call may start its weight copies while the previous call in
    # the stream finishes (the library's programmatic-dependent-launch mode)
    args_tab = {(M, j, pdl): prepared(M, j, pdl) for M in LAT_MS for j in range(nsets)
                for pdl in (True, False)}
    stream = torch.cuda.Stream()

    def capture(calls):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for ar in calls:
                st = op.forward_raw(ar, torch.cuda.current_stream().cuda_stream)
                assert st == 0, st
        return g

    step_graphs = [capture([args_tab[(M, j, True)] for M in SWEEP]) for j in range(nsets)]
    per_m_graphs = {(M, pdl): capture([args_tab[(M, j, pdl)] for j in range(nsets)])
                    for M in LAT_MS for pdl in (True, False)}
    torch.cuda.synchronize()

    # per-M latency (graph replay, nsets calls per replay), both launch modes
    per_m, per_m_plain = {}, {}
    with torch.cuda.stream(stream):
        for M in LAT_MS:
            for pdl, dst in ((True, per_m), (False, per_m_plain)):
                gr = per_m_graphs[(M, pdl)]
                for _ in range(3):
                    gr.replay()
                samples = []
                for _ in range(5):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    for _ in range(4):
                        gr.replay()
                    e1.record(stream)
                    e1.synchronize()
                    samples.append(e0.elapsed_time(e1) * 1e3 / (4 * nsets))
                dst[M] = statistics.median(samples)

    # timed steps
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step_graphs[i % nsets].replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev) as clk:
        time.sleep(0.3)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for i in range(args.steps):
                step_graphs[i % nsets].replay()
            e1.record(stream)
        e1.synchronize()
        time.sleep(0.2)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    if world > 1:
        torch.distributed.barrier()
    ms = max_over_ranks(ms, world)
    op.check(stream)
    tokens_per_step = sum(SWEEP)
    value = job_throughput(tokens_per_step, args.steps, world, ms / 1e3)

    # e2e through the public API: each step copies all of its inputs in with
    # one host->device copy from a pinned staging buffer and all of its
    # outputs back with one device->host copy (views carve the buffers)
    def carve(specs):
        offs, total = [], 0
        for shape, dtype in specs:
            nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
            offs.append((total, nbytes, shape, dtype))
            total += (nbytes + 255) // 256 * 256
        return offs, total

    def views(buf, offs):
        return [buf[o:o + n].view(dt).view(shape) for o, n, shape, dt in offs]

    in_keys = ("R", "y", "inj")
    out_keys = tuple(outs[SWEEP[0]][0].keys())
    in_offs, in_total = carve([(tuple(base[k][:M].shape), base[k].dtype) for M in SWEEP for k in in_keys])
    out_offs, out_total = carve([(tuple(outs[M][0][k].shape), outs[M][0][k].dtype)
                                 for M in SWEEP for k in out_keys])
    # two buffer sets: step i+1's inputs copy in (own stream) while step i
    # computes, and step i's outputs copy back (a third stream) meanwhile;
    # the host reads every step's outputs, one step behind
    host_in_buf = torch.empty(in_total, dtype=torch.uint8).pin_memory()
    dev_in_buf = [torch.empty(in_total, dtype=torch.uint8, device="cuda") for _ in range(2)]
    host_out_buf = [torch.empty(out_total, dtype=torch.uint8).pin_memory() for _ in range(2)]
    dev_out_buf = [torch.empty(out_total, dtype=torch.uint8, device="cuda") for _ in range(2)]
    hv = views(host_in_buf, in_offs)
    dev_in, dev_out = [{}, {}], [{}, {}]
    for bsel in range(2):
        dv, dov = views(dev_in_buf[bsel], in_offs), views(dev_out_buf[bsel], out_offs)
        for i, M in enumerate(SWEEP):
            dev_in[bsel][M] = {k: dv[i * len(in_keys) + j] for j, k in enumerate(in_keys)}
            dev_out[bsel][M] = {k: dov[i * len(out_keys) + j] for j, k in enumerate(out_keys)}
    for i, M in enumerate(SWEEP):
        for j, k in enumerate(in_keys):
            hv[i * len(in_keys) + j].copy_(base[k][:M].cpu())
    h2d, d2h = sum(n for _, n, _, _ in in_offs), sum(n for _, n, _, _ in out_offs)
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    # one prepared call per buffer set, weight set and M: the loop below makes
    # one C-ABI call per forward, with no per-call Python validation
    e2e_args = {(bsel, j, M): op.prepare(dev_in[bsel][M]["R"], dev_in[bsel][M]["y"],
                                         dev_in[bsel][M]["inj"], sets[j]["Wnorm"], sets[j]["Wu"],
                                         Wd=sets[j]["Wd"], Wi=sets[j]["Wi"], out=dev_out[bsel][M],
                                         pdl=True)[0]
                for bsel in range(2) for j in range(nsets) for M in SWEEP}
    sh = stream.cuda_stream

    def e2e_run(nsteps):
        for i in range(nsteps):
            bsel, j = i % 2, i % nsets
            with torch.cuda.stream(h2d_s):
                if i >= 2:
                    h2d_s.wait_event(ev_comp[bsel])      # step i-2 has read this buffer
                dev_in_buf[bsel].copy_(host_in_buf, non_blocking=True)
                ev_in[bsel].record(h2d_s)
            stream.wait_event(ev_in[bsel])
            if i >= 2:
                stream.wait_event(ev_out[bsel])          # step i-2's outputs are home
            for M in SWEEP:
                op.launch(e2e_args[(bsel, j, M)], sh)
            ev_comp[bsel].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(ev_comp[bsel])
                host_out_buf[bsel].copy_(dev_out_buf[bsel], non_blocking=True)
                ev_out[bsel].record(d2h_s)
            if i >= 1:
                ev_out[(i - 1) % 2].synchronize()        # the host has step i-1's results
        ev_out[(nsteps - 1) % 2].synchronize()
        torch.cuda.synchronize()

    e2e_run(args.warmup)
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    e2e_run(args.steps)
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    e2e_value = job_throughput(tokens_per_step, args.steps, world, e2e_s)

    hbm, bf16_peak, peak_src = peaks()
    alg_bytes = sum(WEIGHT_BYTES + M * ACT_BYTES_PER_TOKEN for M in SWEEP)
    traffic, traffic_src = decode_traffic_per_launch()
    kernel_us = sum(per_m[M] for M in SWEEP)
    achieved = alg_bytes / (kernel_us * 1e-6) / 1e9
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,1/sqrt(fan-in)) weights)",
        "config": {"workload": "decode sweep M={2,4,8,16,32}, HC=4 HS=2560 r=320 bf16, "
                               "unfolded Wd/Wi", "tokens_per_step": tokens_per_step,
                   "l2": f"rotating {nsets} weight+input sets ({nsets * per_set / 1e6:.0f} MB > 2x L2)",
                   "timing": "CUDA graph replay, CUDA events on the launching stream",
                   "launch": "programmatic dependent launch (hc_gr_args.pdl = 1): a call's "
                             "weight copies overlap the previous call's tail",
                   "e2e": "public prepare() once per buffer set, then launch() (one C-ABI call) per "
                          "forward; per step one pinned host->device copy of all inputs and "
                          "one device->host copy of all outputs, on their own streams and double-"
                          "buffered (step i+1's copy-in and step i's copy-back overlap step i's "
                          "compute); the host waits for every step's outputs, one step behind",
                   "parallelism": f"replicas x{world}"},
        "clocks": clocks,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": len(SWEEP) * args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": traffic, "traffic_source": traffic_src,
                     "algorithmic_bytes_per_launch": alg_bytes / len(SWEEP),
                     "kernel": "decode_kernel (per launch, mean over the sweep: weights + activations)",
                     "peak_source": peak_src},
        "per_M_us": {str(M): per_m[M] for M in LAT_MS},
        "per_M_us_plain_launch": {str(M): per_m_plain[M] for M in LAT_MS},
        "per_M_roofline_frac": {str(M): (WEIGHT_BYTES + M * ACT_BYTES_PER_TOKEN) / hbm / 1e3
                                / per_m[M] for M in LAT_MS},
    }
    return line


def run_case(args):
    """A few plain forward calls of one shape (for ncu captures)."""
    import numpy as np
    import torch

    from hyper_connection_gated_gb300 import HcGatedResidual, inputs

    shape = inputs.WIDE if args.wide else inputs.DEFAULT
    M = args.M

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to("cuda").view(torch.bfloat16)

    w = {k: bf(v) for k, v in inputs.weights(shape).items()}
    a = inputs.activations(M, shape, distinct_rows=4096)
    R, y, inj = bf(a["R"]), bf(a["y"]), torch.from_numpy(a["inj"]).cuda()
    op = HcGatedResidual(max_M=M, HC=shape.HC, HS=shape.HS, r=shape.r)
    for _ in range(args.calls):
        if args.case == "combine":
            op.combine(R, y, inj)
        elif args.case == "mix":
            op.mix(R, w["Wnorm"], w["Wu"], Wd=w["Wd"], Wi=w["Wi"])
        else:
            path = {"auto": 0, "decode": 1, "prefill": 2}[args.case]
            op.forward(R, y, inj, w["Wnorm"], w["Wu"], Wd=w["Wd"], Wi=w["Wi"], force_path=path)
    op.check()
    torch.cuda.synchronize()
    print(f"case ok: {args.case} M={M} calls={args.calls}")


PREFILL_MS = (512, 1024, 2048, 4096, 8192, 16384, 32768, 65536)


def prefill_sweep(Ms=PREFILL_MS, reps: int = 5):
    """Per-M latency of the prefill path (graph replay, L2 defeated).

    Token rows repeat the generator's first 4096 rows.  Small M rotate over
    enough weight+activation copies to exceed twice the L2; from M=4096 on a
    single call's inputs already exceed the L2.  Mid-batch M also run the
    merged 336-row weight, unfolded and with (1 + Wnorm) folded in (the fold
    is input preparation, done once here with torch on the device).
    """
    import numpy as np
    import torch

    from hyper_connection_gated_gb300 import HcGatedResidual, inputs

    dev = torch.cuda.current_device()
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 << 20)

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to("cuda").view(torch.bfloat16)

    w = {k: bf(v) for k, v in inputs.weights().items()}
    base_rows = 4096
    a = inputs.activations(base_rows)
    R0, y0, inj0 = bf(a["R"]), bf(a["y"]), torch.from_numpy(a["inj"]).cuda()
    Wdi = torch.zeros((336, K_DIM), dtype=torch.bfloat16, device="cuda")
    Wdi[:R_LOW] = w["Wd"]
    Wdi[R_LOW:R_LOW + HC] = w["Wi"]
    Wdi_f = (Wdi.float() * (1.0 + w["Wnorm"].float())[None, :]).to(torch.bfloat16)
    hbm, tflops, _ = peaks()
    res = {}
    stream = torch.cuda.Stream()
    for M in Ms:
        per_set = WEIGHT_BYTES + M * ACT_BYTES_PER_TOKEN
        nsets = 1 if M >= 4096 else int(min(8, max(1, np.ceil(2.0 * l2 / per_set))))
        reps_rows = (M + base_rows - 1) // base_rows
        R = R0.repeat(reps_rows, 1, 1)[:M].contiguous()
        y = y0.repeat(reps_rows, 1)[:M].contiguous()
        inj = inj0.repeat(reps_rows, 1)[:M].contiguous()
        # (name, merged weight, folded, chained by programmatic dependent launch)
        variants = [("unfolded", None, False, False), ("unfolded_pdl", None, False, True)]
        if M <= 2048:
            variants += [("merged336", Wdi, False, False), ("merged336_folded", Wdi_f, True, False)]
        op = HcGatedResidual(max_M=M)
        for name, Wm, fold, pdl in variants:
            sets = [(R, y, inj, w) if j == 0 else
                    (R.clone(), y.clone(), inj.clone(), {k: v.clone() for k, v in w.items()})
                    for j in range(nsets)]
            mats = [Wm if (Wm is None or j == 0) else Wm.clone() for j in range(nsets)]
            outs = [{"R2": torch.empty_like(R), "rrms": torch.empty((M, HC), device="cuda"),
                     "inj_next": torch.empty((M, HC), device="cuda"),
                     "x": torch.empty((M, HS), dtype=torch.bfloat16, device="cuda"),
                     "lora": torch.empty((M, R_LOW), device="cuda")} for _ in range(nsets)]

            def call(j):
                Rj, yj, ij, wj = sets[j]
                kw = dict(Wdi=mats[j], fold_w=fold) if mats[j] is not None else dict(Wd=wj["Wd"], Wi=wj["Wi"])
                op.forward(Rj, yj, ij, wj["Wnorm"], wj["Wu"], out=outs[j], pdl=pdl, **kw)

            for j in range(nsets):
                call(j)
            op.check()
            g = torch.cuda.CUDAGraph()
            calls = max(nsets, 2)
            with torch.cuda.graph(g, stream=stream):
                for j in range(calls):
                    call(j % nsets)
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                for _ in range(2):
                    g.replay()
                samples = []
                for _ in range(reps):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    g.replay()
                    e1.record(stream)
                    e1.synchronize()
                    samples.append(e0.elapsed_time(e1) * 1e3 / calls)
            us = statistics.median(samples)
            roof_us, bound = roofline_us(per_set, M * FLOPS_PER_TOKEN, hbm, tflops)
            res.setdefault(str(M), {})[name] = {
                "us": us, "tokens_per_s": M / (us * 1e-6), "roofline_us": roof_us, "bound": bound,
                "roofline_frac": roof_us / us, "spread": (max(samples) - min(samples)) / us,
                "l2": f"{nsets} rotating sets" if nsets > 1 else "inputs > L2"}
            del sets, outs
        op.close()
        del R, y, inj
        torch.cuda.empty_cache()
    return res


CROSS_MS = (24, 32, 40, 48, 56, 64, 96, 128, 256, 511)


def crossover_sweep(Ms=CROSS_MS, reps: int = 5):
    """Decode kernel against prefill kernels for the same call, M around and
    past the decode kernel's limit (64 tokens): graph replay, weight+input
    sets rotating over more than twice the L2.  The library's M dispatch
    follows this table."""
    import numpy as np
    import torch

    from hyper_connection_gated_gb300 import PATH_DECODE, PATH_PREFILL, HcGatedResidual, inputs

    dev = torch.cuda.current_device()
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 << 20)

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to("cuda").view(torch.bfloat16)

    w = {k: bf(v) for k, v in inputs.weights().items()}
    Mmax = max(Ms)
    a = inputs.activations(Mmax)
    base = dict(w, R=bf(a["R"]), y=bf(a["y"]), inj=torch.from_numpy(a["inj"]).cuda())
    nsets = max(3, int(np.ceil(2.0 * l2 / (WEIGHT_BYTES + Mmax * ACT_BYTES_PER_TOKEN))) + 1)
    sets = [{k: v.clone() for k, v in base.items()} for _ in range(nsets)]
    hbm, tflops, _ = peaks()
    stream = torch.cuda.Stream()
    res = {}
    with HcGatedResidual(max_M=Mmax) as op:
        for M in Ms:
            row = {}
            for name, path in (("decode", PATH_DECODE), ("prefill", PATH_PREFILL)):
                if path == PATH_DECODE and M > 64:
                    continue
                outs = [None] * nsets

                def call(j):
                    s_ = sets[j]
                    outs[j] = op.forward(s_["R"][:M], s_["y"][:M], s_["inj"][:M], s_["Wnorm"], s_["Wu"],
                                         Wd=s_["Wd"], Wi=s_["Wi"], force_path=path, pdl=True,
                                         out=outs[j])
                for j in range(nsets):
                    call(j)
                op.check()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for j in range(nsets):
                        call(j)
                torch.cuda.synchronize()
                samples = []
                with torch.cuda.stream(stream):
                    g.replay()
                    for _ in range(reps):
                        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                        e0.record(stream)
                        g.replay()
                        e1.record(stream)
                        e1.synchronize()
                        samples.append(e0.elapsed_time(e1) * 1e3 / nsets)
                op.check()
                row[name] = statistics.median(samples)
            roof_us, _ = roofline_us(WEIGHT_BYTES + M * ACT_BYTES_PER_TOKEN, M * FLOPS_PER_TOKEN, hbm, tflops)
            row["roofline_us"] = roof_us
            res[str(M)] = row
    return res


WIDE_MS = (1, 8, 64, 1024, 8192)


def wide_sweep(Ms=WIDE_MS, reps: int = 5):
    """Per-M latency of the wide shape (HC=8, HS=4096, r=512; heavy-tailed R,
    y x10): decode path for M <= 32, prefill above, chosen by the library's
    dispatcher.  Graph replay; weight+input sets rotate over more than twice
    the L2 where one set fits in it."""
    import numpy as np
    import torch

    from hyper_connection_gated_gb300 import HcGatedResidual, inputs

    sh = inputs.WIDE
    K = sh.HC * sh.HS
    w_bytes = 2 * (sh.r + sh.HC) * K + 2 * K * sh.r + 2 * K
    a_bytes = 2 * K + 2 * sh.HS + 4 * sh.HC + 2 * K + 4 * sh.HC + 4 * sh.HC + 4 * sh.r + 2 * sh.HS
    dev = torch.cuda.current_device()
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 << 20)

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to("cuda").view(torch.bfloat16)

    w = {k: bf(v) for k, v in inputs.weights(sh).items()}
    base_rows = 1024
    a = inputs.activations(base_rows, sh)
    R0, y0, inj0 = bf(a["R"]), bf(a["y"]), torch.from_numpy(a["inj"]).cuda()
    flops_tok = 2 * K * (sh.r + sh.HC + sh.r)
    hbm, tflops, _ = peaks()
    res = {}
    stream = torch.cuda.Stream()
    for M in Ms:
        per_set = w_bytes + M * a_bytes
        nsets = int(min(4, max(1, np.ceil(2.0 * l2 / per_set))))
        reps_rows = (M + base_rows - 1) // base_rows
        R = R0.repeat(reps_rows, 1, 1)[:M].contiguous()
        y = y0.repeat(reps_rows, 1)[:M].contiguous()
        inj = inj0.repeat(reps_rows, 1)[:M].contiguous()
        op = HcGatedResidual(max_M=M, HC=sh.HC, HS=sh.HS, r=sh.r)
        sets = [(R, y, inj, w) if j == 0 else
                (R.clone(), y.clone(), inj.clone(), {k: v.clone() for k, v in w.items()})
                for j in range(nsets)]
        outs = [{"R2": torch.empty_like(R), "rrms": torch.empty((M, sh.HC), device="cuda"),
                 "inj_next": torch.empty((M, sh.HC), device="cuda"),
                 "x": torch.empty((M, sh.HS), dtype=torch.bfloat16, device="cuda"),
                 "lora": torch.empty((M, sh.r), device="cuda")} for _ in range(nsets)]

        def call(j):
            Rj, yj, ij, wj = sets[j]
            op.forward(Rj, yj, ij, wj["Wnorm"], wj["Wu"], Wd=wj["Wd"], Wi=wj["Wi"], out=outs[j])

        for j in range(nsets):
            call(j)
        op.check()
        g = torch.cuda.CUDAGraph()
        calls = max(nsets, 2)
        with torch.cuda.graph(g, stream=stream):
            for j in range(calls):
                call(j % nsets)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for _ in range(2):
                g.replay()
            samples = []
            for _ in range(reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                g.replay()
                e1.record(stream)
                e1.synchronize()
                samples.append(e0.elapsed_time(e1) * 1e3 / calls)
        us = statistics.median(samples)
        roof_us, bound = roofline_us(per_set, M * flops_tok, hbm, tflops)
        res[str(M)] = {"us": us, "tokens_per_s": M / (us * 1e-6), "roofline_us": roof_us, "bound": bound,
                       "roofline_frac": roof_us / us, "path": "decode" if M <= 32 else "prefill",
                       "l2": f"{nsets} rotating sets" if nsets > 1 else "inputs > L2"}
        op.close()
        del sets, outs, R, y, inj
        torch.cuda.empty_cache()
    return res


ENTRY_MS = {"combine": (32, 512, 8192, 65536), "mix": (2, 32, 512, 8192)}


def entry_sweep(reps: int = 5):
    """Per-M latency of the combine-only and mix-only entry points at the
    default shape (graph replay; sets rotate over more than twice the L2
    where one set fits in it).  combine: R, y, inj in and R2 out, no weights;
    mix: the fused path without y, inj and the R2 store."""
    import numpy as np
    import torch

    from hyper_connection_gated_gb300 import HcGatedResidual, inputs

    dev = torch.cuda.current_device()
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 << 20)
    comb_tok = 2 * K_DIM + 2 * HS + 4 * HC + 2 * K_DIM
    mix_tok = 2 * K_DIM + 4 * HC + 4 * HC + 4 * R_LOW + 2 * HS

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to("cuda").view(torch.bfloat16)

    w = {k: bf(v) for k, v in inputs.weights().items()}
    base_rows = 1024
    a = inputs.activations(base_rows)
    R0, y0, inj0 = bf(a["R"]), bf(a["y"]), torch.from_numpy(a["inj"]).cuda()
    hbm, tflops, _ = peaks()
    res = {}
    stream = torch.cuda.Stream()
    for kind, Ms in ENTRY_MS.items():
        res[kind] = {}
        for M in Ms:
            per_set = M * comb_tok if kind == "combine" else WEIGHT_BYTES + M * mix_tok
            nsets = int(min(256, max(1, np.ceil(2.0 * l2 / per_set))))
            reps_rows = (M + base_rows - 1) // base_rows
            R = R0.repeat(reps_rows, 1, 1)[:M].contiguous()
            y = y0.repeat(reps_rows, 1)[:M].contiguous()
            inj = inj0.repeat(reps_rows, 1)[:M].contiguous()
            op = HcGatedResidual(max_M=M)
            sets = [(R, y, inj, w) if j == 0 else
                    (R.clone(), y.clone(), inj.clone(),
                     w if kind == "combine" else {k: v.clone() for k, v in w.items()})
                    for j in range(nsets)]
            if kind == "combine":
                outs = [torch.empty_like(R) for _ in range(nsets)]
            else:
                outs = [{"rrms": torch.empty((M, HC), device="cuda"),
                         "inj_next": torch.empty((M, HC), device="cuda"),
                         "x": torch.empty((M, HS), dtype=torch.bfloat16, device="cuda"),
                         "lora": torch.empty((M, R_LOW), device="cuda")} for _ in range(nsets)]

            def call(j):
                Rj, yj, ij, wj = sets[j]
                if kind == "combine":
                    op.combine(Rj, yj, ij, out=outs[j])
                else:
                    op.mix(Rj, wj["Wnorm"], wj["Wu"], Wd=wj["Wd"], Wi=wj["Wi"], out=outs[j])

            for j in range(nsets):
                call(j)
            op.check()
            g = torch.cuda.CUDAGraph()
            calls = max(nsets, 2)
            with torch.cuda.graph(g, stream=stream):
                for j in range(calls):
                    call(j % nsets)
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                for _ in range(2):
                    g.replay()
                samples = []
                for _ in range(reps):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    g.replay()
                    e1.record(stream)
                    e1.synchronize()
                    samples.append(e0.elapsed_time(e1) * 1e3 / calls)
            us = statistics.median(samples)
            flops = 0 if kind == "combine" else M * FLOPS_PER_TOKEN
            roof_us, bound = roofline_us(per_set, flops, hbm, tflops)
            res[kind][str(M)] = {"us": us, "tokens_per_s": M / (us * 1e-6), "roofline_us": roof_us,
                                 "bound": bound, "roofline_frac": roof_us / us,
                                 "l2": f"{nsets} rotating sets" if nsets > 1 else "inputs > L2"}
            op.close()
            del sets, outs, R, y, inj
            torch.cuda.empty_cache()
    return res


TRACE_PHASES = {0: "start", 1: "prologue done", 2: "previous kernel done", 3: "COMBINE done",
                4: "issuer 0: boxes landed, MMAs issued", 5: "down MMAs complete",
                6: "pieces written", 7: "first block gathered", 8: "blocks reduced, h published",
                9: "h gathered", 10: "gate MMAs complete", 11: "x stored", 12: "end",
                13: "prologue barrier passed", 14: "thread 0: first box issued",
                15: "issuer 0: gate MMAs issued", 16: "last piece store issued (any thread)",
                17: "last piece word seen (any thread)", 18: "last thread out of its piece loop",
                19: "last thread past the shuffle tree", 20: "last thread past its sum store",
                21: "last thread done with the gate readback", 22: "last thread done with x",
                23: "last thread's first product readback",
                24: "issuer 0: first box landed", 25: "issuer 0: first MMAs issued",
                26: "last thread out of the gather loop", 27: "issuer 0: first chunk landed",
                28: "issuer 0: first gate MMAs issued", 29: "mix inputs landed",
                30: "down MMA completion seen", 31: "gate MMA completion seen",
                32: "thread 0: before the barrier init", 33: "thread 0: barriers initialised",
                34: "last thread at the prologue barrier"}
DOWN_PHASES = (0, 32, 33, 34, 13, 14, 1, 2, 3, 24, 25, 4, 30, 5, 23, 16, 6, 12)
UP_PHASES = (0, 32, 33, 34, 13, 14, 1, 2, 17, 18, 19, 20, 7, 8, 29, 26, 9, 27, 28, 15, 31, 10, 21, 22,
             11, 12)


def decode_trace(args):
    """Phase timeline of the decode kernel, from the library's HCGR_TRACE twin
    (libhc_gr_trace.so, built here if missing).  Per M: `--calls` traced calls
    after 5 warm-up calls, each on one of several weight+input sets whose
    total exceeds twice the L2 (so the weights come from HBM); plain launches,
    or with --trace-pdl each traced call chained after a previous decode call
    by programmatic dependent launch; --trace-hot uses one weight set, which
    stays in L2.  Prints, per phase and role, the min / median / max over the
    CTAs that passed it of the time since the grid's first CTA started (µs),
    each the median over the traced calls."""
    import ctypes

    import numpy as np
    import torch

    from hyper_connection_gated_gb300 import _native, build

    if not os.path.exists(build.LIB_TRACE):
        build.build(trace=True)
    lib = _native.load(build.LIB_TRACE)
    lib.hc_gr_trace_read.argtypes = [ctypes.c_void_p, ctypes.c_int]
    lib.hc_gr_trace_read.restype = ctypes.c_int
    _native._LIB = lib
    from hyper_connection_gated_gb300 import PATH_DECODE, HcGatedResidual, inputs

    shape = inputs.WIDE if args.wide else inputs.DEFAULT
    dev = torch.cuda.current_device()
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 << 20)
    wbytes = 2 * (shape.r + shape.HC) * shape.K + 2 * shape.K * shape.r
    nsets = 1 if args.trace_hot else max(3, int(np.ceil(2.0 * l2 / wbytes)) + 1)

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to("cuda").view(torch.bfloat16)

    w = {k: bf(v) for k, v in inputs.weights(shape).items()}
    a = inputs.activations(32, shape)
    base = dict(w, R=bf(a["R"]), y=bf(a["y"]), inj=torch.from_numpy(a["inj"]).cuda())
    sets = [{k: v.clone() for k, v in base.items()} for _ in range(nsets)]
    slots = 36
    n = 256 * slots
    buf = np.zeros(n, dtype=np.uint64)
    report = {}
    with HcGatedResidual(max_M=32, HC=shape.HC, HS=shape.HS, r=shape.r) as op:
        for M in [int(v) for v in args.trace_M.split(",")]:
            runs = []
            for rep in range(5 + args.calls):
                if args.trace_pdl:
                    s0 = sets[(rep + 1) % nsets]
                    op.forward(s0["R"][:M], s0["y"][:M], s0["inj"][:M], s0["Wnorm"], s0["Wu"],
                               Wd=s0["Wd"], Wi=s0["Wi"], force_path=PATH_DECODE)
                s1 = sets[rep % nsets]
                op.forward(s1["R"][:M], s1["y"][:M], s1["inj"][:M], s1["Wnorm"], s1["Wu"],
                           Wd=s1["Wd"], Wi=s1["Wi"], force_path=PATH_DECODE, pdl=args.trace_pdl)
                op.check()
                assert lib.hc_gr_trace_read(buf.ctypes.data, n) == 0
                if rep >= 5:
                    runs.append(buf.reshape(256, slots).astype(np.int64).copy())
            table = {}
            for role, phases, sel in (("down", DOWN_PHASES, 6), ("up", UP_PHASES, 11)):
                per_run = []
                for st in runs:
                    live = st[st[:, 0] > 0]
                    t0 = live[:, 0].min()
                    rows = live[live[:, sel] > 0]
                    # a phase some CTAs do not pass (no reducer block) keeps 0 there
                    per_run.append({ph: ((rows[rows[:, ph] > 0][:, ph] - t0) / 1e3) for ph in phases})
                table[role] = {
                    TRACE_PHASES[ph]: [round(float(np.median([np.min(r[ph]) for r in per_run])), 2),
                                       round(float(np.median([np.median(r[ph]) for r in per_run])), 2),
                                       round(float(np.median([np.max(r[ph]) for r in per_run])), 2)]
                    for ph in phases}
                table[role + "_ctas"] = int(len(runs[-1][(runs[-1][:, 0] > 0) & (runs[-1][:, sel] > 0)]))
            report[str(M)] = table
            print(f"M={M} ({'chained by programmatic dependent launch' if args.trace_pdl else 'plain launch'}, "
                  f"weights {'L2-resident' if args.trace_hot else 'from HBM'}): µs since the first CTA "
                  f"started, min / median / max over CTAs, median of {args.calls} calls")
            for role in ("down", "up"):
                print(f"  {role} CTAs ({table[role + '_ctas']}):")
                for name, v in table[role].items():
                    print(f"    {name:40s} {v[0]:7.2f} {v[1]:7.2f} {v[2]:7.2f}")
    print(json.dumps({"decode_trace": report, "shape": [shape.HC, shape.HS, shape.r],
                      "pdl": bool(args.trace_pdl), "hot": bool(args.trace_hot)}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", choices=["auto", "decode", "prefill", "combine", "mix"], default=None,
                    help="only run --calls forward calls of one shape (for profiling)")
    ap.add_argument("--M", type=int, default=32)
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--wide", action="store_true")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill-sweep", action="store_true",
                    help="skip the per-M table of the prefill path")
    ap.add_argument("--trace", action="store_true",
                    help="phase timeline of the decode kernel (diagnostic build)")
    ap.add_argument("--trace-M", default="1,8,32")
    ap.add_argument("--trace-pdl", action="store_true")
    ap.add_argument("--trace-hot", action="store_true")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.case is not None:
        run_case(args)
        return
    if args.trace:
        decode_trace(args)
        return

    if args.impl == "reference":
        # The reference arm is the fp64 CPU oracle on the host cores; rank 0 only.
        if rank != 0:
            return
        steps = args.steps
        res = cpu_baseline(seconds=1e9, max_steps=steps, warmup=args.warmup)
        line = {"impl": "reference", "metric": METRIC, "value": res["value"], "unit": "tokens/s",
                "n_gpus": 1, "steps": steps, "warmup": args.warmup,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": {"workload": "decode sweep M={2,4,8,16,32}, HC=4 "
                                                            "HS=2560 r=320 (fp64 oracle)"},
                "cpu_baseline": {k: res.get(k) for k in ("value", "unit", "cores", "kind", "sample")},
                "e2e": {"value": res["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    line = run_ours(args, rank, world)
    if rank == 0 and not args.no_prefill_sweep:
        line["crossover_us"] = crossover_sweep()
        line["prefill_sweep_us"] = prefill_sweep()
        line["wide_sweep_us"] = wide_sweep()
        line["entry_points_us"] = entry_sweep()
    if rank == 0:
        line["cpu_baseline"] = None if args.no_cpu_baseline else cpu_baseline()
        line["cpu_baseline_all_cores"] = None if args.no_cpu_baseline else cpu_baseline_all_cores()
        print(json.dumps(line))
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
