"""Benchmark: exact attention forward + backward (one training step of the attention op)
on the non-causal workload B=4, H=16, N=2048, d=64 (bf16, scale 1/sqrt(d)), through the C ABI.

Prints ONE JSON line (rank 0). ``value`` is whole-job TFLOPS: forward FLOPs 4*B*H*N^2*d
(halved for causal) plus backward FLOPs 2.5x that, divided by the device time of the timed
steps (max over ranks). Each timed step runs fa_forward then fa_backward on inputs resident
in HBM; L2 is flushed (a 512 MiB write) between timed steps, outside the timed events.

``e2e``: the same step through fa_forward_backward_host on pinned host buffers -- copies of
Q, K, V, dO in and of O, LSE, dQ, dK, dV out inside the timed region, pipelined by the library
over chunks of heads so that copies overlap kernels.

After the timed step: ``configs`` (the five attention configurations, forward and backward),
``extensions`` (grouped KV heads, chunked prefill, sliding window, split-KV decode) and
``naive_vs_fused``, each timed alone with L2 flushed.

``--impl reference`` times the fp64 CPU oracle (the reference arm of this repository) on a
bounded sample of the same workload instead.
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

WORKLOAD = dict(name="B4 H16 N2048 d64 non-causal fwd+bwd", B=4, H=16, N=2048, d=64,
                causal=False, seed=1002)
# The five attention configurations the forward/backward targets are stated on, timed one by
# one after the main step (CUDA-event median of --config-reps repetitions, L2 flushed between
# repetitions). Q, K ~ N(0, qk_sigma^2), V, dO ~ N(0, 1), scale 1/sqrt(d).
CONFIGS = [
    dict(name="1: B1 H1 N256 d64 non-causal", B=1, H=1, N=256, d=64, causal=False, qk_sigma=1.0, seed=1001),
    dict(name="2: B4 H16 N2048 d64 non-causal", B=4, H=16, N=2048, d=64, causal=False, qk_sigma=1.0, seed=1002),
    dict(name="3: B8 H32 N8192 d128 causal", B=8, H=32, N=8192, d=128, causal=True, qk_sigma=1.0, seed=1003),
    dict(name="4: B1 H64 N16384 d128 causal, QK sd 3", B=1, H=64, N=16384, d=128, causal=True, qk_sigma=3.0, seed=1004),
    dict(name="4r: B1 H64 N16000 d128 causal, QK sd 3", B=1, H=64, N=16000, d=128, causal=True, qk_sigma=3.0, seed=1004),
    dict(name="5: B4 H16 N4096 d128 causal", B=4, H=16, N=4096, d=128, causal=True, qk_sigma=1.0, seed=1005),
]
# Workloads of the extensions (grouped KV heads, a query offset, a sliding window, split-KV
# decode), timed after the configurations the same way. Q, K, V, dO ~ N(0, 1), scale 1/sqrt(d).
EXTENSIONS = [
    dict(name="GQA B1 Hq32 Hkv8 N8192 d128 causal", B=1, Hq=32, Hkv=8, Tq=8192, Tk=8192, d=128,
         causal=True, window=-1, bwd=True, seed=2001),
    dict(name="chunked prefill Tq1024 of Tk16384 B1 Hq32 Hkv8 d128 causal", B=1, Hq=32, Hkv=8,
         Tq=1024, Tk=16384, d=128, causal=True, window=-1, bwd=True, seed=2002),
    dict(name="sliding window 4095 B1 Hq32 Hkv8 N16384 d128", B=1, Hq=32, Hkv=8, Tq=16384,
         Tk=16384, d=128, causal=True, window=4095, bwd=True, seed=2003),
    dict(name="decode Tq1 Tk16384 B1 Hq32 Hkv8 d128", B=1, Hq=32, Hkv=8, Tq=1, Tk=16384, d=128,
         causal=True, window=-1, bwd=False, seed=2004),
    dict(name="decode Tq1 Tk16384 B8 Hq32 Hkv8 d128", B=8, Hq=32, Hkv=8, Tq=1, Tk=16384, d=128,
         causal=True, window=-1, bwd=False, seed=2005),
]
FWD_KERNEL_SRC = os.path.join(ROOT, "exact_io_aware_fa_gb300", "csrc", "fa_fwd.cu")
BWD_KERNEL_SRC = os.path.join(ROOT, "exact_io_aware_fa_gb300", "csrc", "fa_bwd.cu")
TRAFFIC_JSON = os.path.join(ROOT, "profiles", "traffic.json")
# What the "dominant kernel" timing covers: one ABI call, timed by CUDA events around it.
KERNEL_LABEL = {
    "fa_bwd": "fa_backward call (fa_bwd_pre_kernel + fa_bwd_kernel + fa_bwd_dq_kernel)",
    "fa_fwd": "fa_forward call (fa_fwd_kernel)",
}
L2_FLUSH_BYTES = 512 << 20
METRIC = ("attention fwd+bwd TFLOPS (bf16 in, fp32 accumulate), 1 step = fa_forward + fa_backward"
          " on B4 H16 N2048 d64")


def select_workload(key):
    """The main step's workload: B4 H16 N2048 d64 non-causal by default (the metric's workload);
    `--config K` runs another configuration's fwd + bwd step instead (for profiling)."""
    global WORKLOAD, METRIC
    if key == "2":
        return
    cfg = next(c for c in CONFIGS if c["name"].split(":")[0] == key)
    WORKLOAD = dict(name=cfg["name"].split(": ", 1)[1] + " fwd+bwd", B=cfg["B"], H=cfg["H"],
                    N=cfg["N"], d=cfg["d"], causal=cfg["causal"], seed=cfg["seed"],
                    qk_sigma=cfg["qk_sigma"])
    METRIC = ("attention fwd+bwd TFLOPS (bf16 in, fp32 accumulate), 1 step = fa_forward + "
              "fa_backward on " + WORKLOAD["name"])


def workload_config(world=1):
    w = WORKLOAD
    return {"workload": w["name"], "global_batch": w["B"] * world, "seq_len": w["N"],
            "heads": w["H"], "head_dim": w["d"], "causal": w["causal"],
            "parallelism": f"heads-replica x{world}" if world > 1 else "single"}


def fwd_flops(B, H, N, d, causal):
    f = 4.0 * B * H * N * N * d
    return f / 2 if causal else f


def bwd_flops(B, H, N, d, causal):
    return 2.5 * fwd_flops(B, H, N, d, causal)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration, extension and naive-comparison blocks")
    ap.add_argument("--config-reps", type=int, default=20)
    ap.add_argument("--config", default="2", choices=["1", "2", "3", "4", "4r", "5"],
                    help="configuration of the main timed step (default 2)")
    ap.add_argument("--extensions-only", metavar="SUBSTRING", default=None,
                    help="only the extension workloads whose name contains SUBSTRING (one JSON "
                         "line; profiling)")
    ap.add_argument("--naive-only", action="store_true",
                    help="only the naive-vs-fused forward comparison (one JSON line; profiling)")
    return ap.parse_args()


def file_sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return dict(hbm_gbs=j["hbm_gbs"], bf16_tflops=j["bf16_tflops"],
                    bf16_tflops_sustained=j.get("bf16_tflops_sustained"), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                source="fallback")


# ---- distributed plumbing (one process per GPU; no data-path collective) -----------------

def dist_init(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", init_method="env://")
    return rank, world, local


def barrier(world):
    from exact_io_aware_fa_gb300 import dist as fadist
    fadist.barrier()


def max_over_ranks(x, world):
    from exact_io_aware_fa_gb300 import dist as fadist
    return fadist.max_over_ranks(x, device="cuda" if world > 1 else None)


# ---- clocks sampling ------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
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
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ---- oracle CPU baseline (bounded sample of the workload) -------------------------------------

def oracle_sample_time(heads, want_seconds=None):
    """Time the fp64 oracle forward + backward on `heads` heads of the workload; returns
    (seconds, flops_of_sample, cores)."""
    import oracle
    from exact_io_aware_fa_gb300 import synthetic
    w = WORKLOAD
    bits = synthetic.attention_inputs(1, heads, w["N"], w["d"], seed=w["seed"], with_dout=True)
    cores = oracle.default_threads()
    orc = oracle.Oracle(0, threads=cores)
    scale = 1.0 / math.sqrt(w["d"])
    t0 = time.perf_counter()
    orc.forward_bf16(bits["q"], bits["k"], bits["v"], w["causal"], scale)
    orc.backward_bf16(bits["q"], bits["k"], bits["v"], bits["do"], w["causal"], scale)
    dt = time.perf_counter() - t0
    fl = fwd_flops(1, heads, w["N"], w["d"], w["causal"]) + bwd_flops(1, heads, w["N"], w["d"], w["causal"])
    return dt, fl, cores


def _sample_rows(N, seed, n=32):
    """The parity tests' row sample: n seeded rows plus the tile-boundary rows."""
    import numpy as np
    rng = np.random.default_rng(seed)
    fixed = [0, 127, 128, 255, N - 129, N - 1]
    rows = set(int(x) for x in rng.integers(0, N, size=n)) | {r for r in fixed if 0 <= r < N}
    return np.array(sorted(rows), dtype=np.int64)


def oracle_config_extrapolation(cfg, heads=4, fwd_rows=128, backward=False):
    """Time the fp64 oracle on a sample of one large configuration and extrapolate the full
    oracle's time from the sample's FLOP rate (labelled as such). Forward: `fwd_rows` seeded
    query rows on each of `heads` heads. Backward (optional): the parity tests' row sample as
    query and key rows, which rebuilds every row's LSE and D."""
    import numpy as np
    import oracle
    from exact_io_aware_fa_gb300 import synthetic
    N, d, causal = cfg["N"], cfg["d"], cfg["causal"]
    bits = synthetic.attention_inputs(1, heads, N, d, seed=cfg["seed"], qk_sigma=cfg["qk_sigma"],
                                      with_dout=backward)
    threads = min(heads, oracle.default_threads())
    orc = oracle.Oracle(0, threads=threads)
    scale = 1.0 / math.sqrt(d)

    def vis(i):  # keys row i sees
        return (i + 1) if causal else N

    rows = np.sort(np.random.default_rng(cfg["seed"]).choice(N, size=min(fwd_rows, N),
                                                              replace=False)).astype(np.int64)
    t0 = time.perf_counter()
    orc.forward_rows_bf16(bits["q"], bits["k"], bits["v"], causal, scale, rows)
    t_fwd = time.perf_counter() - t0
    f_fwd = heads * sum(4.0 * vis(int(i)) * d for i in rows)
    full_f = fwd_flops(cfg["B"], cfg["H"], N, d, causal)
    out = {"sample": f"{heads} heads x {len(rows)} seeded query rows (forward)",
           "cores": threads, "fwd_sample_s": t_fwd, "fwd_tflops": f_fwd / t_fwd / 1e12,
           "fwd_full_s_extrapolated": full_f / (f_fwd / t_fwd),
           "label": "extrapolated: full-configuration FLOPs / the sample's FLOP rate"}
    if backward:
        rb = _sample_rows(N, cfg["seed"])
        t0 = time.perf_counter()
        orc.backward_rows_bf16(bits["q"], bits["k"], bits["v"], bits["do"], causal, scale, rb, rb)
        t_bwd = time.perf_counter() - t0
        # every row's LSE and D (score and dP rows), then per sampled query row its P, dS and
        # dQ rows, per sampled key row its P and dS columns, dK and dV
        all_vis = (N * (N + 1) / 2.0) if causal else float(N) * N
        f_bwd = heads * (4.0 * all_vis * d + sum(6.0 * vis(int(i)) * d for i in rb) +
                         sum(8.0 * ((N - int(j)) if causal else N) * d for j in rb))
        out["sample"] += f"; {len(rb)} query and key rows per head (backward)"
        out.update(bwd_sample_s=t_bwd, bwd_tflops=f_bwd / t_bwd / 1e12,
                   bwd_full_s_extrapolated=bwd_flops(cfg["B"], cfg["H"], N, d, causal) /
                   (f_bwd / t_bwd))
    return out


def run_reference(args, rank, world):
    if rank != 0:
        return
    w = WORKLOAD
    heads = 16
    for _ in range(args.warmup):
        oracle_sample_time(heads)
    total_t, total_f = 0.0, 0.0
    cores = 1
    for _ in range(args.steps):
        dt, fl, cores = oracle_sample_time(heads)
        total_t += dt
        total_f += fl
    value = total_f / total_t / 1e12
    line = {
        "impl": "reference", "metric": METRIC,
        "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": dict(workload_config(1), l2="n/a (CPU)",
                       sample=f"{heads} of {w['B'] * w['H']} heads per step (fp64 oracle)"),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{heads} heads of B4 H16 N2048 d64, fwd+bwd, per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---- naive (materialised) attention as the comparison point -----------------------------

def naive_vs_fused(api, dev, reps=10):
    """Forward time and peak device memory of naive materialised attention (S and P written to
    HBM; exact_io_aware_fa_gb300.naive) against the fused forward, on B4 H16 N2048 d64 and on
    T = 4096 ("15. FlashAttention", "Stretch exercises" item 1). Context only."""
    import torch
    from exact_io_aware_fa_gb300 import naive
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    out = []
    for (B, H, N, d) in ((4, 16, 2048, 64), (1, 16, 4096, 64)):
        g = torch.Generator(device=dev)
        g.manual_seed(4242)
        q, k, v = (torch.randn((B, H, N, d), generator=g, device=dev).to(torch.bfloat16)
                   for _ in range(3))
        res = {"workload": f"B{B} H{H} N{N} d{d} non-causal forward"}
        for name, fn in (("naive", lambda: naive.forward(q, k, v)),
                         ("fused", lambda: api.forward(q, k, v))):
            fn()
            torch.cuda.synchronize()
            base = torch.cuda.memory_allocated(dev)
            torch.cuda.reset_peak_memory_stats(dev)
            fn()
            torch.cuda.synchronize()
            peak = torch.cuda.max_memory_allocated(dev) - base
            ts = []
            for _ in range(reps):
                flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                fn()
                b.record()
                torch.cuda.synchronize()
                ts.append(a.elapsed_time(b))
            ms = statistics.median(ts)
            res[name] = {"ms": ms, "tflops": fwd_flops(B, H, N, d, False) / ms / 1e9,
                         "peak_bytes_beyond_inputs": int(peak)}
        res["speedup"] = res["naive"]["ms"] / res["fused"]["ms"]
        out.append(res)
        del q, k, v
        torch.cuda.empty_cache()
    return out


# ---- GPU arm -------------------------------------------------------------------------------------

def _traffic_record(kernel, workload):
    """A traffic.json record of `kernel` on `workload` whose kernel source is unchanged since
    the counters were taken, else None."""
    if not os.path.exists(TRAFFIC_JSON):
        return None
    with open(TRAFFIC_JSON) as f:
        tj = json.load(f)
    src = BWD_KERNEL_SRC if kernel == "fa_bwd" else FWD_KERNEL_SRC
    for ent in tj.get("records", []):
        if (ent.get("kernel") == kernel and ent.get("workload") == workload and
                ent.get("source_sha") == file_sha(src)):
            return ent
    return None


def time_configs(api, dev, reps, peaks):
    """Median fwd / bwd times of every configuration (CUDA events on the launching stream, L2
    flushed before each repetition, outside the events). Inputs: seeded device normals of each
    configuration's distribution, rounded to bf16."""
    import torch
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    s = stream.cuda_stream
    peak = peaks["bf16_tflops"]
    out = []
    for cfg in CONFIGS:
        B, H, N, d, causal = cfg["B"], cfg["H"], cfg["N"], cfg["d"], cfg["causal"]
        g = torch.Generator(device=dev)
        g.manual_seed(cfg["seed"])

        def normal(sigma):
            return (torch.randn((B, H, N, d), generator=g, device=dev) * sigma).to(torch.bfloat16)

        q, k = normal(cfg["qk_sigma"]), normal(cfg["qk_sigma"])
        v, do = normal(1.0), normal(1.0)
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
        ws = torch.empty(api.backward_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
        scale = 1.0 / math.sqrt(d)
        ci = int(causal)

        def fwd():
            st = api.forward_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), B, H, N, d, ci, scale, s)
            assert st == 0, api.status_string(st)

        def bwd():
            st = api.backward_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                  dv.data_ptr(), B, H, N, d, ci, scale, ws.data_ptr(), s)
            assert st == 0, api.status_string(st)

        def run(reps_, flushed):
            for _ in range(3):
                fwd()
                bwd()
            ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps_)]
            for e in ev:
                if flushed:
                    flush.zero_()
                e[0].record(stream)
                fwd()
                e[1].record(stream)
                bwd()
                e[2].record(stream)
            torch.cuda.synchronize()
            return (statistics.median(e[0].elapsed_time(e[1]) for e in ev),
                    statistics.median(e[1].elapsed_time(e[2]) for e in ev))

        fms, bms = run(reps, True)
        assert api.device_error() == 0
        ff, bf = fwd_flops(B, H, N, d, causal), bwd_flops(B, H, N, d, causal)
        ent = {"config": cfg["name"],
               "fwd": {"ms": fms, "tflops": ff / fms / 1e9, "frac_of_peak": ff / fms / 1e9 / peak},
               "bwd": {"ms": bms, "tflops": bf / bms / 1e9, "frac_of_peak": bf / bms / 1e9 / peak},
               "timing": f"median of {reps}, L2 flushed"}
        for kern, key, ms, fl in (("fa_fwd", "fwd", fms, ff), ("fa_bwd", "bwd", bms, bf)):
            rec = _traffic_record(kern, cfg["name"])
            if rec is not None:
                ent[key]["traffic"] = rec["bytes_per_launch"]
                ent[key]["hbm_gbs"] = rec["bytes_per_launch"] / (ms * 1e-3) / 1e9
                ent[key]["hbm_frac"] = ent[key]["hbm_gbs"] / peaks["hbm_gbs"]
        if cfg["seed"] == WORKLOAD["seed"]:
            wf, wb = run(reps, False)
            ent["warm_l2"] = {"fwd_ms": wf, "bwd_ms": wb, "fwd_tflops": ff / wf / 1e9,
                              "bwd_tflops": bf / wb / 1e9,
                              "timing": f"median of {reps}, L2 not flushed"}
        out.append(ent)
        del q, k, v, do, o, lse, dq, dk, dv, ws
        torch.cuda.empty_cache()
    return out


def visible_pairs(Tq, Tk, causal, window):
    """Query-key pairs a launch computes: query row i at key position Tk - Tq + i sees the keys
    up to it (causal) and, with a window, no more than `window` positions before it."""
    total = 0
    for i in range(Tq):
        p = Tk - Tq + i
        hi = min(p, Tk - 1) if causal else Tk - 1
        lo = max(0, p - window) if window >= 0 else 0
        total += max(0, hi - lo + 1)
    return total


def time_extensions(api, dev, reps, peaks, name_filter=None):
    """Median fwd (and bwd) times of the extension workloads, through the Python API with
    preallocated outputs and workspaces (CUDA events on the launching stream, L2 flushed before
    each repetition). FLOPs 4 * B * Hq * (visible pairs) * d, x2.5 for the backward; decode
    also reports its K and V bytes over the forward's time against the measured copy rate."""
    import torch
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    peak = peaks["bf16_tflops"]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out = []
    for ext in EXTENSIONS:
        if name_filter is not None and name_filter not in ext["name"]:
            continue
        B, Hq, Hkv, Tq, Tk, d = ext["B"], ext["Hq"], ext["Hkv"], ext["Tq"], ext["Tk"], ext["d"]
        causal, window = ext["causal"], ext["window"]
        g = torch.Generator(device=dev)
        g.manual_seed(ext["seed"])

        def normal(h, n):
            return torch.randn((B, h, n, d), generator=g, device=dev).to(torch.bfloat16)

        q, k, v, do = normal(Hq, Tq), normal(Hkv, Tk), normal(Hkv, Tk), normal(Hq, Tq)
        o = torch.empty_like(q)
        lse = torch.empty((B, Hq, Tq), dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        nsplit = api.choose_splits(B, Hq, Hkv, Tq, Tk, sms)
        fws = None
        if nsplit > 1:
            fws = torch.empty(api.splitkv_workspace_bytes(B, Hq, Tq, d, nsplit),
                              dtype=torch.uint8, device=dev)
        bws = torch.empty(api.backward_workspace_bytes(B, Hq, Tq, d), dtype=torch.uint8,
                          device=dev) if ext["bwd"] else None

        def fwd():
            api.forward(q, k, v, causal=causal, window=window, out=o, lse=lse, nsplit=nsplit,
                        workspace=fws)

        def bwd():
            api.backward(q, k, v, o, lse, do, causal=causal, window=window, dq=dq, dk=dk, dv=dv,
                         workspace=bws)

        def timed(fn):
            for _ in range(3):
                fn()
            ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(reps)]
            for e in ev:
                flush.zero_()
                e[0].record(stream)
                fn()
                e[1].record(stream)
            torch.cuda.synchronize()
            return statistics.median(e[0].elapsed_time(e[1]) for e in ev)

        fl = 4.0 * B * Hq * visible_pairs(Tq, Tk, causal, window) * d
        fms = timed(fwd)
        ent = {"workload": ext["name"], "nsplit": nsplit,
               "fwd": {"ms": fms, "tflops": fl / fms / 1e9, "frac_of_peak": fl / fms / 1e9 / peak},
               "timing": f"median of {reps}, L2 flushed"}
        if not ext["bwd"]:
            kv_bytes = 2 * B * Hkv * Tk * d * 2
            ent["fwd"]["kv_gbs"] = kv_bytes / (fms * 1e-3) / 1e9
            ent["fwd"]["kv_frac_of_hbm"] = ent["fwd"]["kv_gbs"] / peaks["hbm_gbs"]
        else:
            bms = timed(bwd)
            ent["bwd"] = {"ms": bms, "tflops": 2.5 * fl / bms / 1e9,
                          "frac_of_peak": 2.5 * fl / bms / 1e9 / peak}
        assert api.device_error() == 0
        out.append(ent)
        del q, k, v, do, o, lse, dq, dk, dv, fws, bws
        torch.cuda.empty_cache()
    return out


def run_ours(args, rank, world, local):
    import numpy as np
    import torch

    import __graft_entry__
    if rank == 0 or world == 1:
        __graft_entry__.build()
    barrier(world)
    from exact_io_aware_fa_gb300 import api, synthetic

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = WORKLOAD
    B, H, N, d, causal = w["B"], w["H"], w["N"], w["d"], w["causal"]
    scale = 1.0 / math.sqrt(d)
    # Weak scaling: every rank runs the full workload on its own heads (its own seed).
    from exact_io_aware_fa_gb300 import dist as fadist
    bits = synthetic.attention_inputs(B, H, N, d, seed=fadist.rank_seed(w["seed"], rank),
                                      qk_sigma=w.get("qk_sigma", 1.0), with_dout=True)

    def dev_t(b):
        return torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(dev)

    q, k, v, do = (dev_t(bits[n]) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    ws = torch.empty(api.backward_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    s = stream.cuda_stream
    ci = int(bool(causal))

    def step_fwd():
        st = api.forward_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                             lse.data_ptr(), B, H, N, d, ci, scale, s)
        assert st == 0, api.status_string(st)

    def step_bwd():
        st = api.backward_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                              lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                              dv.data_ptr(), B, H, N, d, ci, scale, ws.data_ptr(), s)
        assert st == 0, api.status_string(st)

    for _ in range(args.warmup):
        step_fwd()
        step_bwd()
        flush.zero_()
    torch.cuda.synchronize()
    assert api.device_error() == 0

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    for i in range(args.steps):
        e0, e1, e2 = ev[i]
        e0.record(stream)
        step_fwd()
        e1.record(stream)
        step_bwd()
        e2.record(stream)
        flush.zero_()  # L2 flush between timed steps (outside the events)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    assert api.device_error() == 0
    fwd_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps)]
    bwd_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(args.steps)]
    total_ms = sum(fwd_ms) + sum(bwd_ms)
    total_ms = max_over_ranks(total_ms, world)
    ff = fwd_flops(B, H, N, d, causal)
    bf = bwd_flops(B, H, N, d, causal)
    value = fadist.weak_scaling_value(ff + bf, args.steps, world, total_ms * 1e-3)
    peaks = load_peaks()
    fwd_med = statistics.median(fwd_ms)
    bwd_med = statistics.median(bwd_ms)
    fwd_tf = ff / (fwd_med * 1e-3) / 1e12
    bwd_tf = bf / (bwd_med * 1e-3) / 1e12
    dominant = "fa_bwd" if bwd_med >= fwd_med else "fa_fwd"
    dom_tf = bwd_tf if dominant == "fa_bwd" else fwd_tf
    dom_ms = bwd_med if dominant == "fa_bwd" else fwd_med

    cfg_name = next((c["name"] for c in CONFIGS
                     if (c["B"], c["H"], c["N"], c["d"], c["causal"]) == (B, H, N, d, causal)), None)
    rec = _traffic_record(dominant, cfg_name) if cfg_name else None
    traffic = rec["bytes_per_launch"] if rec else None

    # ---- end to end through the public API with host buffers ----------------------------------
    e2e = None
    if not args.no_e2e:
        hq, hk, hv, hdo = (torch.from_numpy(bits[n].view(np.int16)).view(torch.bfloat16).pin_memory()
                           for n in ("q", "k", "v", "do"))
        ho = torch.empty_like(hq).pin_memory()
        hlse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
        hdq, hdk, hdv = (torch.empty_like(hq).pin_memory() for _ in range(3))
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo))
        d2h = sum(t.numel() * t.element_size() for t in (ho, hlse, hdq, hdk, hdv))

        dbuf = torch.empty(api.host_step_device_bytes(B, H, H, N, N, d, 0), dtype=torch.uint8,
                           device=dev)

        def e2e_step():
            # fa_forward_backward_host: copies in, fa_forward_ex + fa_backward_ex, copies out,
            # pipelined over chunks of heads
            api.forward_backward_host(hq, hk, hv, hdo, causal=causal, scale=scale,
                                      out=(ho, hlse, hdq, hdk, hdv), device_buffer=dbuf,
                                      stream=stream.cuda_stream)

        for _ in range(max(1, args.warmup)):
            e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ea.record(stream)
        for _ in range(args.steps):
            e2e_step()
        eb.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(ea.elapsed_time(eb), world)
        e2e = {"value": fadist.weak_scaling_value(ff + bf, args.steps, world, e2e_ms * 1e-3),
               "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms / args.steps}

    configs = None
    extensions = None
    naive_cmp = None
    if not args.no_configs:
        configs = time_configs(api, dev, args.config_reps, peaks)
        extensions = time_extensions(api, dev, args.config_reps, peaks)
        naive_cmp = naive_vs_fused(api, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        heads = 8
        dt, fl, cores = oracle_sample_time(heads)
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"{heads} of 64 heads of the workload, fwd+bwd, {dt:.1f} s"}
        if not args.no_configs:
            cpu["configs"] = {c["name"]: oracle_config_extrapolation(c, backward=c["name"][0] == "5")
                              for c in CONFIGS if c["name"][:2] in ("3:", "4:", "5:")}

    if rank != 0:
        return
    line = {
        "metric": METRIC,
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(workload_config(world),
                       l2="flushed between timed steps (512 MiB write outside the events)"),
        "fwd": {"ms": fwd_med, "tflops": fwd_tf, "frac_of_peak": fwd_tf / peaks["bf16_tflops"],
                "timing": f"median of {args.steps} timed steps"},
        "bwd": {"ms": bwd_med, "tflops": bwd_tf, "frac_of_peak": bwd_tf / peaks["bf16_tflops"],
                "timing": f"median of {args.steps} timed steps"},
        "roofline": {"kernel": KERNEL_LABEL[dominant], "bound": "tensor", "achieved": dom_tf,
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": dom_tf / peaks["bf16_tflops"], "traffic": traffic,
                     "hbm_gbs": (traffic / (dom_ms * 1e-3) / 1e9) if traffic else None,
                     "peak_source": f"{peaks['source']} bf16 burst"},
        "configs": configs,
        "extensions": extensions,
        "naive_vs_fused": naive_cmp,
        "e2e": e2e,
        "gpu_launches": args.steps * 4,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def run_extensions_only(args):
    import torch

    import __graft_entry__
    __graft_entry__.build()
    from exact_io_aware_fa_gb300 import api
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    ext = time_extensions(api, dev, args.config_reps, load_peaks(), args.extensions_only)
    print(json.dumps({"extensions": ext}), flush=True)


def run_naive_only(args):
    import torch

    import __graft_entry__
    __graft_entry__.build()
    from exact_io_aware_fa_gb300 import api
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    print(json.dumps({"naive_vs_fused": naive_vs_fused(api, dev, reps=max(1, args.steps))}),
          flush=True)


def main():
    args = parse_args()
    select_workload(args.config)
    if args.naive_only:
        run_naive_only(args)
        return
    if args.extensions_only is not None:
        run_extensions_only(args)
        return
    rank, world, local = dist_init(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
