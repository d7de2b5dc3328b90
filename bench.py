"""Benchmark of the batch-1 quantized Llama decode step on GB300.

Default workload: Llama-3.1-70B-shaped model, Q4_K_M-style weight mix (45.7 GB
of weights read per token) resident in HBM, f16 KV cache prefilled to context
4096, greedy decode.  One step = one decode step (every kernel of the hot
path).  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload llama70b_q4_k_m|llama8b_q8_0|llama70b_q6_k_streamed|tiny]
                  [--no-sweep] [--no-extras] [--no-cpu-baseline] [--profile-gemv FMT ROWS COLS LAUNCHES]

value: tokens/s over the K timed steps, device-timed (CUDA events on the
launching stream around a device-resident greedy loop; inputs already in HBM).
e2e: tokens/s through nt_decode_step with the token copied host->device and
the result device->host every step.  Weights are far larger than L2 (129 MB),
so no flush is needed between steps.
After the main model is freed, rank 0 also measures (unless turned off): the
isolated dequant-GEMV sweep at the 70B layer shapes in five formats, the 8B Q8_0
decode step, and the 70B Q6_K step with 54 of 80 layers streamed from
page-locked host memory.
--impl reference times the oracle (the C restatement of the method) on one
host core, each step one decode step of the same architecture truncated to one
layer; tokens/s are projected to the whole model by weight+KV bytes.
With N > 1 (torchrun) every rank runs an independent replica (the step does
not shard); value = all ranks' tokens / max over ranks of the time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "batch-1 decode tok/s"
PAGES_8B_Q8_0_TOK_S = 48.9   # RTX 3090, Llama 8B Q8_0 (hada "Roadmap", Phase 1); context, other hardware


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=128)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="llama70b_q4_k_m",
                   choices=["llama8b_q8_0", "llama70b_q4_k_m", "llama70b_q6_k_streamed", "tiny"])
    p.add_argument("--no-sweep", action="store_true")
    p.add_argument("--no-extras", action="store_true", help="skip the 8B and streamed-70B extra measurements")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--profile-gemv", nargs=4, metavar=("FMT", "ROWS", "COLS", "LAUNCHES"))
    p.add_argument("--layer-skip", type=int, default=0, metavar="MAX",
                   help="calibrate per-layer similarity, then skip up to MAX layers at or above --skip-threshold")
    p.add_argument("--skip-threshold", type=float, default=0.98)
    p.add_argument("--resident", type=int, default=None, metavar="N",
                   help="keep layers [0, N) in device memory and stream the rest (0: every layer from the host tier)")
    p.add_argument("--speculative", type=int, default=0, metavar="K",
                   help="time self-speculative cycles of K draft tokens instead of plain steps")
    p.add_argument("--draft-layers", type=int, default=None,
                   help="draft model depth (default: the resident layers, else a quarter of the layers)")
    p.add_argument("--layers", type=int, default=None,
                   help="profiling aid: the workload's shapes with this many layers (not a bench line)")
    return p.parse_args(argv)


# ---------------------------------------------------------------- workloads --

def workload(name: str):
    return dict(_workload(name), key=name)


def _workload(name: str):
    from quantized_decode_dequant_gb300 import workloads as W
    if name == "llama8b_q8_0":
        return dict(spec=W.LLAMA_8B_Q8_0, ctx=W.LLAMA_8B_CTX, resident=None,
                    label="Llama-3.1-8B-shaped, Q8_0, ctx 512, batch 1", vs=PAGES_8B_Q8_0_TOK_S)
    if name == "llama70b_q4_k_m":
        return dict(spec=W.LLAMA_70B_Q4_K_M, ctx=W.LLAMA_70B_Q4_K_M_CTX, resident=None,
                    label="Llama-3.1-70B-shaped, Q4_K_M mix, ctx 4096, batch 1", vs=None)
    if name == "llama70b_q6_k_streamed":
        return dict(spec=W.LLAMA_70B_Q6_K, ctx=W.LLAMA_70B_Q6_K_CTX, resident=W.LLAMA_70B_Q6_K_RESIDENT,
                    label="Llama-3.1-70B-shaped, Q6_K, 26 layers resident, 54 streamed, ctx 1024", vs=None)
    return dict(spec=W.TINY, ctx=0, resident=None, label="tiny Llama (2 layers, hidden 512), Q8_0", vs=None)


def max_ctx_for(wl, steps: int, warmup: int) -> int:
    # every phase restarts at the prefilled context, so the longest phase bounds the cache
    return wl["ctx"] + max(steps, warmup, 8) + 8


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), source="measured")
    return dict(hbm_gbs=6800.0, source="fallback")


# --------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi samples every 200 ms during the timed region (clocks, throttle reasons)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                p = [x.strip() for x in line.split(",")]
                if len(p) >= 9:
                    rows.append(p)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(pw) if pw else None}


# -------------------------------------------------------------- distributed --

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world <= 1:
        return 0, 1, 0, None
    import torch
    import torch.distributed as dist
    rank, local = int(os.environ["RANK"]), int(os.environ.get("LOCAL_RANK", "0"))
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if backend == "nccl":
        torch.cuda.set_device(local)
    dist.init_process_group(backend=backend)
    return rank, world, local, dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def reduce_max(dist, value: float) -> float:
    """Max over ranks (the timing rule: the slowest replica sets the job time)."""
    if dist is None:
        return value
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: int, world: int, max_seconds: float) -> float:
    return units_per_rank * world / max_seconds


# ------------------------------------------------------------ CPU baseline --

class OracleSample:
    """The oracle on one layer of the workload: the same architecture truncated
    to one decoder layer (plus the embedding and the output head), weights
    generated and quantized with every host thread when it is built (outside
    any timed region), KV cache prefilled to the workload's context, then timed
    on ONE host thread -- the single-core baseline.  A full token's time is
    projected from a sample step by weight+KV bytes (the oracle's time is
    proportional to the bytes it dequantizes)."""

    def __init__(self, wl, n_steps: int):
        import oracle
        from quantized_decode_dequant_gb300 import workloads as W
        spec = dict(wl["spec"])
        self.sample = dict(spec, n_layers=1, max_ctx=max(wl["ctx"], 1) + n_steps + 2)
        self.model = oracle.Model(oracle.ModelSpec(**self.sample, seed=W.SEED_WEIGHTS),
                                  nthreads=os.cpu_count() or 1)
        self.model.set_threads(1)
        if wl["ctx"] > 0:
            self.model.kv_prefill(wl["ctx"], W.SEED_KV)
        self.tok = oracle.token(W.SEED_PROMPT, oracle.UID_TOKENS, 0, spec["vocab"])
        full = W.weight_bytes(spec) + W.kv_bytes(spec, wl["ctx"])
        part = W.weight_bytes(self.sample) + W.kv_bytes(self.sample, wl["ctx"])
        self.scale = full / part

    def step(self) -> float:
        t0 = time.perf_counter()
        _, self.tok, _ = self.model.decode_step(self.tok)
        return time.perf_counter() - t0

    def close(self):
        self.model.close()


def cpu_baseline(wl, n_steps: int = 3) -> dict:
    """Single-core oracle on a bounded sample of the workload (OracleSample):
    n_steps one-layer decode steps, each about 1-5 s on one core."""
    smp = OracleSample(wl, n_steps)
    try:
        times = [smp.step() for _ in range(n_steps)]
    finally:
        smp.close()
    dt = statistics.median(times)
    return {"value": 1.0 / (dt * smp.scale), "unit": "tok/s", "cores": 1, "kind": "oracle",
            "sample": (f"{n_steps} oracle decode steps of the architecture truncated to 1 decoder layer "
                       f"(ctx {wl['ctx']}, embedding and output head included) on one host thread: "
                       f"median {dt:.3f} s per sample step, measured; value = 1 / (that x {smp.scale:.1f}), "
                       f"the full model's weight+KV bytes over the sample's"),
            "sample_s_per_step": round(dt, 4), "projection_factor": round(smp.scale, 2),
            "gemv": oracle_gemv_rates()}


def oracle_gemv_rates(rows_sample: int = 64) -> dict:
    """The oracle's dequant-GEMV on one host core at the sweep's shapes: the
    first `rows_sample` rows of each matrix (generated and quantized outside the
    timed call), GB/s of weight bytes read."""
    import numpy as np

    import oracle
    from quantized_decode_dequant_gb300 import workloads as W
    out = {}
    for fmt in W.GEMV_FORMATS:
        for rows, cols in W.GEMV_SHAPES:
            b = oracle.qtensor_rows(fmt, rows, cols, 0, 1, 0.02, row0=0, nrows=rows_sample, nthreads=4)
            x = np.random.default_rng(1).standard_normal(cols).astype(np.float32)
            t0 = time.perf_counter()
            oracle.gemv(fmt, b, rows_sample, cols, x, nthreads=1)
            dt = time.perf_counter() - t0
            gb = rows_sample * cols // W.BLOCK_ELEMS[fmt] * W.BLOCK_BYTES[fmt] / 1e9
            out[f"{fmt} {rows}x{cols}"] = round(gb / dt, 3)
    return {"unit": "GB/s, 1 core", "sample": f"first {rows_sample} rows of each sweep shape", "rates": out}


def run_reference(args, wl, rank, world, dist):
    """The oracle as the reference arm: W warm-up and K timed sample steps
    (OracleSample, one host thread); ms_per_step is the measured time of a
    sample step, value the projected whole-model tokens/s."""
    if rank != 0:
        return
    smp = OracleSample(wl, args.steps + args.warmup)
    try:
        for _ in range(args.warmup):
            smp.step()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            smp.step()
        dt = (time.perf_counter() - t0) / args.steps
    finally:
        smp.close()
    value = 1.0 / (dt * smp.scale)
    sample = (f"each step: one oracle decode step of the architecture truncated to 1 decoder layer "
              f"(ctx {wl['ctx']}, embedding and output head included) on one host thread, measured "
              f"({dt * 1e3:.1f} ms); value = 1 / (step time x {smp.scale:.1f}), the full model's "
              f"weight+KV bytes over the sample's")
    line = {"metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": wl["label"], "parallelism": "replicas only"},
            "projection": {"measured_s_per_sample_step": dt, "factor": smp.scale,
                           "projected_s_per_token": dt * smp.scale},
            "cpu_baseline": {"value": value, "unit": "tok/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def per_kernel_launches(spec) -> int:
    """Kernels of one step on the per-kernel launch path: embedding, per layer the
    QKV GEMV (two launches when v has its own format and no two-format kernel
    takes the pair: a Q4_K q/k with a Q6_K v at widths of whole 1024-column
    tiles is one launch), attention, O, gate/up and down GEMVs, then the output
    GEMV and the argmax."""
    tq, tv = spec.get("t_q", "q8_0"), spec.get("t_v", "q8_0")
    pair = tq == "q4_k" and tv == "q6_k" and spec["hidden"] % 1024 == 0
    return 1 + spec["n_layers"] * (5 + int(tq != tv and not pair)) + 2


# DRAM bytes (read + write) per algorithmic byte of the step's GEMV launches, per
# workload, from the ncu captures summarised in profiles/, and the SHA-256 of the
# kernel sources they were taken on: a changed kernel reports no traffic.
GEMV_DRAM_PER_BYTE: dict[str, float] = {"llama70b_q4_k_m": 1.001, "llama8b_q8_0": 1.001}
GEMV_SOURCES = ("nt_gemv_pipe.cuh", "nt_gemv.cuh")
GEMV_SOURCES_SHA256 = "cf4e534df5faabd7f407b664d138d6fd1af6537ca9ce57866df263cdd2f533fb"


def gemv_sources_sha256() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in GEMV_SOURCES:
        with open(os.path.join(ROOT, "quantized_decode_dequant_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def gemv_traffic(bytes_per_launch: float, wl):
    ratio = GEMV_DRAM_PER_BYTE.get(wl.get("key", ""))
    if ratio is None or gemv_sources_sha256() != GEMV_SOURCES_SHA256:
        return None
    return round(bytes_per_launch * ratio)


# ------------------------------------------------------------------ GEMV --

def gemv_sweep(nt, torch, peak_gbs: float, l2_bytes: int) -> list[dict]:
    """Isolated dequant-GEMV sweep at the 70B layer shapes: back-to-back launches
    over weight copies that together exceed 4x L2, captured once in a CUDA graph
    so the host launch rate does not bound short kernels; median of 5 replays."""
    from quantized_decode_dequant_gb300 import workloads as W
    out = []
    stream = torch.cuda.current_stream()
    for fmt in W.GEMV_FORMATS:
        for rows, cols in W.GEMV_SHAPES:
            wbytes = rows * cols // W.BLOCK_ELEMS[fmt] * W.BLOCK_BYTES[fmt]
            copies = max(1, min(64, math.ceil(4 * l2_bytes / wbytes)))
            ts = [nt.nt_qtensor_create(fmt, rows, cols, 0, 1000 + i, 0.02) for i in range(copies)]
            try:
                x = torch.randn(cols, device="cuda")
                y = torch.empty(rows, device="cuda")
                launches = max(copies, 2 * copies if wbytes < 64 << 20 else copies)
                for i in range(copies):
                    nt.nt_gemv_q(ts[i], x.data_ptr(), y.data_ptr(), stream)
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    cs = torch.cuda.current_stream()
                    for i in range(launches):
                        nt.nt_gemv_q(ts[i % copies], x.data_ptr(), y.data_ptr(), cs)
                g.replay()
                times = []
                for _ in range(5):
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    g.replay()
                    b.record(stream)
                    b.synchronize()
                    times.append(a.elapsed_time(b) / launches)
                del g
                ms = statistics.median(times)
                algo = wbytes + 4 * (rows + cols)
                gbs = algo / (ms * 1e-3) / 1e9
                out.append({"fmt": fmt, "rows": rows, "cols": cols, "us": round(ms * 1e3, 2),
                            "GB_s": round(gbs, 1), "frac": round(gbs / peak_gbs, 3)})
            finally:
                for t in ts:
                    nt.nt_qtensor_destroy(t)
    return out


def profile_gemv(nt, torch, fmt: str, rows: int, cols: int, launches: int):
    """A few launches of one GEMV shape (for an ncu capture of a small case)."""
    t = nt.nt_qtensor_create(fmt, rows, cols, 0, 1, 0.02)
    x = torch.randn(cols, device="cuda")
    y = torch.empty(rows, device="cuda")
    for _ in range(launches):
        nt.nt_gemv_q(t, x.data_ptr(), y.data_ptr(), torch.cuda.current_stream())
    torch.cuda.synchronize()
    nt.nt_qtensor_destroy(t)
    print(json.dumps({"profile_gemv": [fmt, rows, cols, launches]}))


# ------------------------------------------------------------------ ours --

DTYPE = ("weights as block codes; GEMV: codes x activations in 16-bit fixed point per 32-column block "
         "(19-bit into the Q/K/V GEMV), exact int32 DP4A dot products, fp32 block scales and accumulation; "
         "attention: f16 KV cache, f16 hi+lo tensor-core products with fp32 accumulation, fp32 softmax")


def measure(nt, torch, wl, steps: int, warmup: int, args, dist, world: int, local: int, peaks: dict,
            primary: bool) -> dict:
    """One model of workload wl: W warm-up steps, K timed steps (device-timed
    greedy loop on the device for resident models; per-step nt_decode_step
    calls, layer copies inside, for streamed ones), the same K steps end to end
    through nt_decode_step, per-class device times and the roofline of the
    step's GEMV launches.  The model is freed before it returns."""
    from quantized_decode_dequant_gb300 import workloads as W
    spec = dict(wl["spec"], max_ctx=max_ctx_for(wl, steps, warmup))
    m = nt.nt_model_create(nt.make_config(**spec, seed=W.SEED_WEIGHTS))
    stream = torch.cuda.current_stream()
    out = {}
    try:
        tok0 = _prompt_token(spec["vocab"])
        streamed = wl["resident"] is not None
        if streamed:
            nt.nt_stream_layers(m, wl["resident"], 2)

        def reset():
            if wl["ctx"] > 0:
                nt.nt_kv_prefill(m, wl["ctx"], W.SEED_KV)
            else:
                nt.nt_kv_reset(m)

        skip_info = None
        if primary and args.layer_skip > 0:
            skip_info = calibrate_skip(nt, m, reset, tok0, spec, args.layer_skip, args.skip_threshold)

        # ---- warm-up
        reset()
        if streamed:
            t = tok0
            for _ in range(warmup):
                t = nt.nt_decode_step(m, t)
        else:
            nt.nt_decode_run(m, tok0, warmup, stream)
        torch.cuda.synchronize()

        # ---- timed
        reset()
        clocks = ClockSampler(local)
        n_draft = args.draft_layers if args.draft_layers is not None else (
            wl["resident"] if streamed else spec["n_layers"] // 4)
        with clocks:
            barrier(dist)
            torch.cuda.synchronize()
            if primary and args.speculative:
                # cycles until `steps` tokens are emitted; each cycle copies the
                # host-tier layers once for up to K tokens
                t0 = time.perf_counter()
                t, emitted, cycles, accepted, h2d_b, vw_b = tok0, 0, 0, 0, 0.0, 0.0
                while emitted < steps:
                    e, j = nt.nt_speculative_step(m, t, n_draft, args.speculative)
                    t = e[-1]
                    emitted += len(e)
                    cycles += 1
                    accepted += j
                    st = nt.nt_get_stats(m)
                    h2d_b += st.h2d_bytes
                    vw_b += st.verify_weight_bytes
                torch.cuda.synchronize()
                sec = (time.perf_counter() - t0) * steps / emitted
                out["speculative"] = {"k": args.speculative, "draft_layers": n_draft, "cycles": cycles,
                                      "tokens": emitted, "tokens_per_cycle": round(emitted / cycles, 3),
                                      "accepted_per_cycle": round(accepted / cycles, 3),
                                      "h2d_GB_per_token": round(h2d_b / emitted / 1e9, 3),
                                      "verify_weight_GB_per_cycle": round(vw_b / cycles / 1e9, 3),
                                      "verified_layers_weight_GB": round(
                                          (W.weight_bytes(dict(spec, n_layers=spec["n_layers"] - n_draft))
                                           - W.weight_bytes(dict(spec, n_layers=0))) / 1e9, 3),
                                      "note": "acceptance is meaningless on random weights; the cycle cost is "
                                              "the measurement (verification reads each verified layer's weights "
                                              "once per multi-token launch, not once per token)"}
            elif streamed:
                t0 = time.perf_counter()
                t = tok0
                h2d_b = h2d_ms = comp_ms = ov = 0.0
                lay_min, lay_max, slow_layers = [], [], []
                for _ in range(steps):
                    t = nt.nt_decode_step(m, t)
                    st = nt.nt_get_stats(m)
                    h2d_b += st.h2d_bytes
                    h2d_ms += st.h2d_ms
                    comp_ms += st.compute_ms
                    ov += st.overlap
                    if st.h2d_layer_min_idx >= 0:
                        lay_min.append(st.h2d_layer_min_GBs)
                        lay_max.append(st.h2d_layer_max_GBs)
                        slow_layers.append(st.h2d_layer_min_idx)
                torch.cuda.synchronize()
                sec = time.perf_counter() - t0
                out["streaming"] = {
                    "resident_layers": wl["resident"], "streamed_layers": spec["n_layers"] - wl["resident"],
                    "h2d_GB_s": round(h2d_b / (h2d_ms * 1e-3) / 1e9, 1) if h2d_ms else None,
                    "h2d_GB_per_step": round(h2d_b / steps / 1e9, 3), "overlap": round(ov / steps, 4),
                    "compute_ms_per_step": round(comp_ms / steps, 3),
                    "pcie_gen5_x16_nominal_GB_s": 64.0, "link": host_link(local),
                    "h2d_timing": "copy-stream CUDA events around each layer's copy",
                    "cpu_numa_node": cpu_numa_node(),
                    "h2d_layer_GB_s_min_max": [round(min(lay_min), 1), round(max(lay_max), 1)] if lay_min else None,
                    "h2d_slowest_layers": sorted(set(slow_layers))[:8]}
                pr = h2d_probe(torch, 1 << 30)
                out["streaming"].update({
                    "h2d_probe_GB_s": pr["best"], "h2d_probe_median_GB_s": pr["median"],
                    "h2d_probe_4GiB_GB_s": pr["sustained"],
                    "h2d_probe": "plain copies from page-locked memory in the same process right after the timed "
                                 "steps: best and median of 8 copies of 1 GiB, and one copy of 4 GiB"})
            else:
                ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                ev0.record(stream)
                nt.nt_decode_run(m, tok0, steps, stream)
                ev1.record(stream)
                torch.cuda.synchronize()
                sec = ev0.elapsed_time(ev1) * 1e-3
            barrier(dist)
        sec_max = reduce_max(dist, sec)
        out["value"] = job_throughput(steps, world, sec_max)
        out["ms_per_step"] = sec_max / steps * 1e3
        out["clocks"] = clocks.summary()
        out["first_tokens"] = None if streamed else nt.nt_get_tokens(m, max(wl["ctx"], 0), min(steps, 8)).tolist()

        # ---- e2e through the public call, host token in / result out every step
        # (a streamed step already runs through nt_decode_step: its timed loop is the e2e one)
        if streamed:
            e2e_value = out["value"]
        else:
            reset()
            barrier(dist)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            t = tok0
            for _ in range(steps):
                t = nt.nt_decode_step(m, t)
            e2e_value = job_throughput(steps, world, reduce_max(dist, time.perf_counter() - t0))
        out["e2e"] = {"value": e2e_value, "unit": "tok/s", "h2d_bytes_per_step": 4, "d2h_bytes_per_step": 8}

        # ---- per-class device times (event pair around every launch) and the roofline
        stats = nt.nt_get_stats(m)
        step_bytes = stats.weight_bytes + stats.kv_bytes_per_pos * (wl["ctx"] + steps / 2)
        if skip_info:   # skipped layers' weights and cache are not read
            frac_kv = 1.0 - skip_info["n_skipped"] / spec["n_layers"]
            step_bytes = (stats.weight_bytes - skip_info["weight_bytes_saved_per_token"]
                          + stats.kv_bytes_per_pos * frac_kv * (wl["ctx"] + steps / 2))
            out["layer_skip"] = skip_info
        out["step_roofline"] = {"bytes_per_step": step_bytes,
                                "achieved_GB_s": round(step_bytes / (out["ms_per_step"] * 1e-3) / 1e9, 1),
                                "frac": round(step_bytes / (out["ms_per_step"] * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                                "peak_GB_s": peaks["hbm_gbs"]}
        if not streamed:
            reset()
            n_prof = max(4, min(steps, 32))
            kt = nt.nt_profile_steps(m, tok0, n_prof)
            out["gpu_launches"] = int(kt.kernel_launches // n_prof * steps)
            out["kernel_classes"] = {
                name: {"launches_per_step": kt.launches[c] // n_prof, "ms_per_step": round(kt.ms[c] / n_prof, 4),
                       "GB_s": round(kt.bytes[c] / (kt.ms[c] * 1e-3) / 1e9, 1) if kt.ms[c] else None}
                for name, c in (("gemv", nt.KC_GEMV), ("attention", nt.KC_ATTN), ("other", nt.KC_OTHER))}
            out["kernel_classes"]["profiled_step_ms"] = round(kt.step_ms, 4)
            out["kernel_classes"]["source"] = "CUDA event pair around every launch (no overlap between launches)"
            # the dominant kernel: the step's GEMV launches replayed on their own, back to back
            reset()
            g_ms, g_bytes, g_n = nt.nt_profile_gemvs(m, 8)
            achieved = g_bytes / (g_ms * 1e-3) / 1e9
            out["roofline"] = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                               "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                               "traffic": gemv_traffic(g_bytes, wl),
                               "kernel": "k_gemv_pipe (fused dequant-GEMV: every GEMV launch of a step, "
                                         "graph-replayed back to back with programmatic dependent launch)",
                               "peak_source": peaks["source"], "bytes_per_launch": round(g_bytes),
                               "launches_per_step": g_n, "us_per_launch": round(g_ms * 1e3, 3),
                               "timing": "CUDA events around 8 replays of the GEMV graph on the launching stream"}
        else:
            out["gpu_launches"] = per_kernel_launches(wl["spec"]) * steps
    finally:
        nt.nt_model_destroy(m)
    return out


def host_link(local: int) -> str:
    """How the GPU reaches host memory: NVLink-C2C on Grace systems, else PCIe."""
    try:
        r = subprocess.run(["nvidia-smi", "-q", "-i", str(local)], capture_output=True, text=True, timeout=20)
        txt = r.stdout
    except (OSError, subprocess.SubprocessError):
        return "unknown"
    if "C2C" in txt or "c2c" in txt:
        return "NVLink-C2C"
    for line in txt.splitlines():
        if "PCIe Generation" in line or "Link Width" in line:
            return "PCIe"
    return "unknown"


def h2d_probe(torch, nbytes: int, reps: int = 8) -> dict:
    """GB/s of plain host-to-device copies of nbytes from page-locked memory (the
    rate the link gives a single copy, the bound of a layer copy): the best and
    the median of reps copies, and one copy of four times the size (sustained).
    The host memory and link are shared with the machine's other work, so the
    median and the long copy show what a burst's best hides."""
    src = torch.empty(4 * nbytes, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(4 * nbytes, dtype=torch.uint8, device="cuda")
    dst[:nbytes].copy_(src[:nbytes], non_blocking=True)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def once(n):
        ev0.record()
        dst[:n].copy_(src[:n], non_blocking=True)
        ev1.record()
        torch.cuda.synchronize()
        return n / (ev0.elapsed_time(ev1) * 1e-3) / 1e9

    rates = sorted(once(nbytes) for _ in range(reps))
    long = once(4 * nbytes)
    del src, dst
    return {"best": round(rates[-1], 1), "median": round(rates[len(rates) // 2], 1), "sustained": round(long, 1)}


def cpu_numa_node() -> int | None:
    """NUMA node of the CPU this process runs on (Linux sysfs), None if unknown."""
    try:
        with open("/proc/self/stat") as f:
            cpu = int(f.read().rsplit(")", 1)[1].split()[36])
        for d in os.listdir(f"/sys/devices/system/cpu/cpu{cpu}"):
            if d.startswith("node") and d[4:].isdigit():
                return int(d[4:])
    except (OSError, ValueError, IndexError):
        pass
    return None


def run_ours(args, wl, rank, world, local, dist):
    import torch

    from quantized_decode_dequant_gb300 import nt, workloads as W
    torch.cuda.set_device(local)
    nt.lib()
    if args.profile_gemv:
        fmt, r, c, n = args.profile_gemv
        profile_gemv(nt, torch, fmt, int(r), int(c), int(n))
        return
    peaks = measured_peaks()
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 0) or 0) or (126 << 20)
    main_m = measure(nt, torch, wl, args.steps, args.warmup, args, dist, world, local, peaks, primary=True)
    sweep = cpu = None
    extras = {}
    if rank == 0:
        if not args.no_sweep:
            sweep = gemv_sweep(nt, torch, peaks["hbm_gbs"], l2)
        plain = (args.layers is None and args.resident is None and not args.layer_skip and not args.speculative
                 and args.workload == "llama70b_q4_k_m")
        if plain and not args.no_extras:
            for name, steps, warm in (("llama8b_q8_0", W.LLAMA_8B_STEPS, 5),
                                      ("llama70b_q6_k_streamed", W.LLAMA_70B_Q6_K_STEPS, 3)):
                x = measure(nt, torch, workload(name), steps, warm, args, None, 1, local, peaks, primary=False)
                keep = ("value", "ms_per_step", "e2e", "step_roofline", "roofline", "streaming", "clocks")
                extras[name] = dict({k: x[k] for k in keep if k in x}, unit="tok/s", steps=steps, warmup=warm,
                                    workload=workload(name)["label"])
        if not args.no_cpu_baseline:
            cpu = cpu_baseline(wl)
    if rank != 0:
        return
    value = main_m["value"]
    line = {"metric": METRIC, "value": round(value, 3), "unit": "tok/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(main_m["ms_per_step"], 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": round(value / wl["vs"], 3) if wl["vs"] else None,
            "dtype": DTYPE,
            "data": "synthetic (seeded N(0,0.02) weights quantized on device; N(0,1) f16 KV prefill)",
            "config": {"workload": wl["label"], "model": "llama", "global_batch": 1, "seq_len": wl["ctx"],
                       "parallelism": "replicas only" if world > 1 else "single GPU",
                       "l2": "inputs larger than L2 (weights > 4x L2), no flush"},
            "roofline": main_m.get("roofline"), "step_roofline": main_m["step_roofline"],
            "kernel_classes": main_m.get("kernel_classes"), "cpu_baseline": cpu, "e2e": main_m["e2e"],
            "gpu_launches": main_m["gpu_launches"], "clocks": main_m["clocks"],
            "first_tokens": main_m["first_tokens"]}
    for k in ("streaming", "layer_skip", "speculative"):
        if k in main_m:
            line[k] = main_m[k]
    if extras:
        line["extras"] = extras
    if sweep:
        line["gemv_sweep"] = sweep
        line["gemv_sweep_min_frac"] = min(s["frac"] for s in sweep)
    print(json.dumps(line), flush=True)


def calibrate_skip(nt, m, reset, tok0, spec, max_skip: int, threshold: float, steps: int = 4) -> dict:
    """Per-layer cosine between the residual entering and leaving each layer,
    averaged over a few greedy steps from the prompt token, then the skip plan
    (layers at or above the threshold, at most max_skip) applied to the model."""
    import numpy as np

    from quantized_decode_dequant_gb300 import workloads as W
    reset()
    cos = np.zeros(spec["n_layers"])
    t = tok0
    for _ in range(steps):
        t, c = nt.nt_layer_similarity(m, t)
        cos += c
    cos /= steps
    mask = nt.nt_plan_layer_skip(cos, threshold, max_skip)
    nt.nt_set_layer_skip(m, mask)
    layer_bytes = W.weight_bytes(dict(spec, n_layers=1)) - W.weight_bytes(dict(spec, n_layers=0))
    skipped = [int(i) for i in np.flatnonzero(mask)]
    return {"threshold": threshold, "max_skip": max_skip, "calibration_steps": steps, "n_skipped": len(skipped),
            "skipped_layers": skipped, "layers_at_or_above_threshold": int((cos >= threshold).sum()),
            "cos_min_max": [round(float(cos.min()), 5), round(float(cos.max()), 5)],
            "weight_bytes_saved_per_token": layer_bytes * len(skipped),
            "note": "mechanism and bytes only: output quality cannot be judged on random weights"}


def _prompt_token(vocab: int) -> int:
    """Prompt token id: SplitMix64 output of the prompt stream's first counter, mod vocab."""
    gamma, seed, uid = 0x9E3779B97F4A7C15, 3, 0x300000
    z = (seed + gamma * ((uid << 40) + 1)) & (2**64 - 1)
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & (2**64 - 1)
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & (2**64 - 1)
    return (z ^ (z >> 31)) % vocab


def main(argv=None):
    args = parse_args(argv)
    rank, world, local, dist = dist_setup()
    wl = workload(args.workload)
    if args.layers is not None:
        wl = dict(wl, spec=dict(wl["spec"], n_layers=args.layers),
                  label=wl["label"] + f" (profiling case: {args.layers} layers)", vs=None)
    if args.resident is not None:
        n = max(0, min(args.resident, wl["spec"]["n_layers"]))
        wl = dict(wl, resident=n, vs=None,
                  label=wl["label"] + f" ({n} layers resident, {wl['spec']['n_layers'] - n} streamed)")
    try:
        if args.impl == "reference":
            run_reference(args, wl, rank, world, dist)
        else:
            run_ours(args, wl, rank, world, local, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
