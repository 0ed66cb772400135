"""Benchmark of the activation-sparse gated FFN (TwELL) on GB300: tokens/s per
layer for the inference forward and the training step, with the roofline
fractions of each kernel.

Inference step = one pass of the inference hot path over one batch: the gate
GEMM with the TwELL-packing epilogue (twell_gate_pack) followed by the up+down
projection, on the faster (CUDA-event time at that workload) of the
tensor-core union-gather forward (twell_ffn_fwd_tc) and the CUDA-core fused
kernel (twell_ffn_fwd); both are timed and reported.  Training step = gate
GEMM, TwELL -> hybrid, hybrid forward, hybrid backward with the L1 term.

Workloads (seeded synthetic inputs, see workloads.py): the headline is the
1.5B-class layer (T=16384 tokens, d_model=2048, d_ff=8192, mean 1% active
with a heavy-tailed per-token density, TwELL width 16), the largest inference
layer; the 0.5B-class layer, the small gated-MLP layer, the decode sweep
(T = 1, 4, 16, 64, 256 at d_model=2048, d_ff=8192, 0.5%) and the 2B-class
training step are measured in the same run, each with its own entry.

Rooflines follow the method's algorithmic work: the gate is a dense
contraction (2 T D F flops on the tensor cores, or the bytes of x, W_g and
the TwELL where those take longer); the up+down projection must move x in, y
out, the W_u / W_d rows of every neuron active in some row and the TwELL
entries, and do 4 D flops per active entry on the FP32 FMA pipe; its binding
roofline is the larger of the two times.  The FMA peak is measured here by a
register-resident FMA probe (twell_probe_fma), HBM and bf16 tensor peaks come
from MEASURED_PEAKS.json.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle on a
bounded sample of the headline workload instead.

Timing: W warm-up steps, then K timed steps.  Before every timed step a
512 MiB buffer is written to flush the 129 MB L2; each step is bracketed by
CUDA events on the launching stream (the flush is outside them), and the
per-kernel times come from events around each kernel.  Multi-GPU runs (one
process per GPU under torchrun) are replicas: each rank runs the full batch,
and the job value is all ranks' tokens over the slowest rank's time.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse gated-FFN tokens/s per layer (fwd; fwd+bwd) on 1 GB300, % of roofline"


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch from
# the committed ncu captures in profiles/, valid only while the kernel's source
# is the one captured (sha256 of the .cu file); otherwise reported as null.
TRAFFIC = {
    # 1.5B-class layer (profiles/ffn_fwd_tc_1.5B_T16384.md)
    ("twell_ffn_fwd_tc_sorted", "1.5B-class T=16384 D=2048 F=8192 mean 1% heavy-tail W=16"): (
        780.73e6, "csrc/ffn_tc.cu", "e9eb6d8e73758029", "profiles/ffn_fwd_tc_1.5B_T16384.md"),
    ("twell_ffn_fwd_tc", "1.5B-class T=16384 D=2048 F=8192 mean 1% heavy-tail W=16"): (
        828.30e6, "csrc/ffn_tc.cu", "e9eb6d8e73758029", "profiles/ffn_fwd_tc_1.5B_T16384.md"),
    ("twell_ffn_fwd", "1.5B-class T=16384 D=2048 F=8192 mean 1% heavy-tail W=16"): (
        775.65e6, "csrc/ffn_fwd.cu", "2e583b71ad421583", "profiles/ffn_fwd_tc_1.5B_T16384.md"),
    ("twell_gate_pack", "1.5B-class T=16384 D=2048 F=8192 mean 1% heavy-tail W=16"): (
        149.95e6, "csrc/gate_pack.cu", "541fa10f1d139aef", "profiles/ffn_fwd_tc_1.5B_T16384.md"),
    # 0.5B-class layer (the same profile, second table)
    ("twell_ffn_fwd_tc", "0.5B-class T=8192 D=1536 F=6144 1% W=8"): (
        219.47e6, "csrc/ffn_tc.cu", "e9eb6d8e73758029", "profiles/ffn_fwd_tc_1.5B_T16384.md"),
    ("twell_ffn_fwd_tc_sorted", "0.5B-class T=8192 D=1536 F=6144 1% W=8"): (
        246.89e6, "csrc/ffn_tc.cu", "e9eb6d8e73758029", "profiles/ffn_fwd_tc_1.5B_T16384.md"),
    ("twell_ffn_fwd", "0.5B-class T=8192 D=1536 F=6144 1% W=8"): (
        105.89e6, "csrc/ffn_fwd.cu", "2e583b71ad421583", "profiles/ffn_fwd_tc_1.5B_T16384.md"),
    ("twell_gate_pack", "0.5B-class T=8192 D=1536 F=6144 1% W=8"): (
        45.03e6, "csrc/gate_pack.cu", "541fa10f1d139aef", "profiles/ffn_fwd_tc_1.5B_T16384.md"),
}


def _traffic(kernel, workload):
    import hashlib
    rec = TRAFFIC.get((kernel, workload))
    if rec is None:
        return None, None
    nbytes, src, sha, prof = rec
    path = os.path.join(ROOT, "activation_sparse_gated_gate_gb300", src)
    try:
        cur = hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]
    except OSError:
        return None, None
    return (nbytes, prof) if cur == sha else (None, None)


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(
            p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, interval_ms=200):
        self.index = index
        self.interval_ms = interval_ms
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
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
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}

    def watts(self):
        """Mean board power (nvidia-smi power.draw) over the samples, or None."""
        w = []
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) >= 4:
                try:
                    w.append(float(f[3]))
                except ValueError:
                    pass
        return statistics.mean(w) if w else None


def energy_per_token(fn, tokens, stream, dev_index, seconds=1.5):
    """Board energy per token of back-to-back steps fn(): mean nvidia-smi
    power.draw (sampled every 100 ms) times the steps' CUDA-event time,
    divided by the tokens processed.  Idle board power is included."""
    import torch
    fn()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    fn()
    b.record(stream)
    torch.cuda.synchronize()
    n = max(1, int(seconds * 1e3 / max(a.elapsed_time(b), 1e-3)))
    with ClockSampler(dev_index, interval_ms=100) as clk:
        time.sleep(0.3)  # let the sampler start before the loop
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    w = clk.watts()
    if w is None:
        return None
    return {"joules_per_token": w * ms * 1e-3 / (n * tokens), "watts": w,
            "steps": n, "ms_per_step": ms / n}


def max_over_ranks(value, device=None):
    """Max of a per-rank float over the process group (the identity without
    one).  The timed region's length is the slowest rank's."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank, world_size, max_ms_per_step):
    """Whole-job throughput of replicas: every rank processes its own batch
    of `tokens_per_rank` tokens per step; the step takes the slowest rank's
    time."""
    return world_size * tokens_per_rank / (max_ms_per_step / 1e3)


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local



# ----------------------------------------------------------------- CPU oracle

def oracle_step(w, rows):
    """The oracle's inference path on token rows ``rows``: fp64 gate, TwELL
    pack, TwELL-driven up/down projection."""
    import oracle
    x = w.x[rows]
    z = oracle.gate_preact(x, w.Wg_t)
    tw = oracle.twell_pack(z, 128, w.width)
    return oracle.ffn_forward_twell(x, tw, w.Wu_t, w.Wd)


def oracle_dense_step(w, rows):
    """The oracle's dense definition on token rows ``rows`` (fp64 matmuls
    over every neuron)."""
    import oracle
    return oracle.ffn_forward_rows(w.x, w.Wg_t, w.Wu_t, w.Wd, rows)


def time_oracle(w, budget_s=10.0, chunk=64, seed=0, kind="sparse"):
    """Tokens/s of one oracle path on sampled rows, run for about
    `budget_s` seconds of host CPU (at least one chunk)."""
    fn = oracle_step if kind == "sparse" else oracle_dense_step
    rng = np.random.default_rng(seed)
    done = 0
    t0 = time.perf_counter()
    while True:
        rows = np.sort(rng.choice(w.T, size=min(chunk, w.T), replace=False))
        fn(w, rows)
        done += len(rows)
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return done / el, done, el


_POOL_W = None


def _pool_init(cfg, T):
    # each worker keeps one BLAS thread (set in its environment before numpy
    # loads) and draws the workload itself from its seed
    global _POOL_W
    import workloads
    _POOL_W = workloads.config(cfg, T=T)


def _pool_chunk(args):
    kind, rows = args
    (oracle_step if kind == "sparse" else oracle_dense_step)(_POOL_W, rows)
    return len(rows)


_ONE_THREAD = {k: "1" for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
                                "BLIS_NUM_THREADS", "NUMEXPR_NUM_THREADS")}


def time_oracle_pool(cfg, T, kind, budget_s, procs, chunk=16, seed=0):
    """Tokens/s of an oracle path on all host cores: `procs` spawned worker
    processes with one BLAS thread each, fed chunks of sampled rows for
    about `budget_s` seconds (worker start-up excluded)."""
    import multiprocessing as mp
    import workloads
    w = workloads.config(cfg, T=T)
    ctx = mp.get_context("spawn")
    saved = {k: os.environ.get(k) for k in _ONE_THREAD}
    os.environ.update(_ONE_THREAD)
    try:
        pool = ctx.Pool(procs, initializer=_pool_init, initargs=(cfg, T))
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    rng = np.random.default_rng(seed)
    try:
        # warm every worker (workload drawn, modules loaded) before timing
        pool.map(_pool_chunk, [(kind, np.arange(1)) for _ in range(procs)], chunksize=1)
        done = 0
        t0 = time.perf_counter()
        while True:
            jobs = [(kind, np.sort(rng.choice(w.T, size=min(chunk, w.T), replace=False)))
                    for _ in range(procs)]
            done += sum(pool.map(_pool_chunk, jobs, chunksize=1))
            el = time.perf_counter() - t0
            if el >= budget_s:
                break
    finally:
        pool.terminate()
        pool.join()
    return done / el, done, el


def _one_thread_run(cfg, T, kind, budget_s):
    """The oracle path in a fresh spawned process with one BLAS thread."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    saved = {k: os.environ.get(k) for k in _ONE_THREAD}
    os.environ.update(_ONE_THREAD)
    try:
        with ctx.Pool(1, initializer=_pool_init, initargs=(cfg, T)) as pool:
            return pool.apply(_timed_in_worker, (kind, budget_s))
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def _timed_in_worker(kind, budget_s):
    oracle_step(_POOL_W, np.arange(1))  # modules and weight conversions warm
    return time_oracle(_POOL_W, budget_s=budget_s, chunk=16, kind=kind)


def cpu_baselines(cfg, T, budget_s):
    """The oracle timed on the host cores: its dense definition and its
    sparse (TwELL) inference path, each single-threaded and on every core.
    Returns the dict for the JSON line."""
    import workloads
    name = workloads.config(cfg, T=T).name
    procs = os.cpu_count() or 1
    res = {}
    for kind in ("sparse", "dense"):
        v1, n1, s1 = _one_thread_run(cfg, T, kind, budget_s)
        vn, nn, sn = time_oracle_pool(cfg, T, kind, budget_s, procs)
        res[kind] = {"one_thread": {"value": v1, "rows": n1, "seconds": s1, "cores": 1},
                     "all_cores": {"value": vn, "rows": nn, "seconds": sn, "cores": procs}}
    head = res["sparse"]["all_cores"]
    return {
        "value": head["value"], "unit": "tokens/s", "cores": procs, "kind": "oracle",
        "sample": (f"{head['rows']} sampled token rows of {name} in {head['seconds']:.1f} s "
                   f"on {procs} processes x 1 BLAS thread (fp64 gate, TwELL pack, fused "
                   "up/down)"),
        "nproc": procs,
        "paths": {k: {m: {"tokens_per_s": r[m]["value"], "cores": r[m]["cores"],
                          "rows": r[m]["rows"], "seconds": r[m]["seconds"]}
                      for m in ("one_thread", "all_cores")} for k, r in res.items()},
        "what": ("sparse = the oracle's TwELL inference path (fp64 gate matmul, TwELL pack, "
                 "up/down over active entries); dense = its dense fp64 definition; "
                 "one_thread = one process, one BLAS thread; all_cores = one spawned process "
                 "per core, one BLAS thread each, on sampled rows"),
    }


def run_reference(args, w, cfg):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    for _ in range(args.warmup):
        oracle_step(w, np.arange(min(16, w.T)))
    tot_rows = 0
    tot_s = 0.0
    for _ in range(args.steps):
        v, n, s = time_oracle(w, budget_s=args.ref_budget)
        tot_rows += n
        tot_s += s
    value = tot_rows / tot_s
    cores = os.cpu_count()
    sample = (f"{tot_rows} sampled token rows of {w.name} over {args.steps} steps "
              f"(gate fp64 matmul + TwELL pack + fused up/down in fp64; numpy with its "
              f"default BLAS threads)")
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * w.T / value, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "d_model": w.D, "d_ff": w.F,
                   "twell_width": w.width, "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out))
    return 0


# ------------------------------------------------------------- roofline math

def gate_roofline(T, D, F, nnz, ms, hbm_gbs, bf16_tflops):
    """Gate GEMM + TwELL pack: 2 T D F flops (tensor cores); bytes = x and
    W_g in (bf16) + the TwELL written (5 bytes per stored entry: fp32 value
    and u8 column; 1 byte per (row, tile) count).  The bound is whichever
    roofline time is longer (tensor for token blocks, HBM for decode)."""
    flops = 2.0 * T * D * F
    nbytes = 2.0 * T * D + 2.0 * F * D + 5.0 * nnz + T * (F // 128)
    t_tensor = flops / (bf16_tflops * 1e12)
    t_hbm = nbytes / (hbm_gbs * 1e9)
    t = ms * 1e-3
    out = {"flops": flops, "bytes": nbytes, "ms": ms,
           "tensor": {"achieved_tflops": flops / t / 1e12, "peak": bf16_tflops,
                      "frac": t_tensor / t, "t_us": t_tensor * 1e6},
           "hbm": {"achieved_gbs": nbytes / t / 1e9, "peak": hbm_gbs, "frac": t_hbm / t,
                   "t_us": t_hbm * 1e6}}
    out["bound"] = "tensor" if t_tensor >= t_hbm else "hbm"
    out["frac"] = out[out["bound"]]["frac"]
    return out


def updown_bytes(T, D, F, nnz, n_active):
    """Algorithmic bytes of the up+down projection: x in (bf16), y out (fp32,
    the library's output type), the W_u and W_d rows (bf16) of every neuron
    active in some row, the TwELL entries read (fp32 value + u8 column) and
    the (row, tile) counts."""
    return 2.0 * T * D + 4.0 * T * D + 4.0 * n_active * D + 5.0 * nnz + T * (F // 128)


def updown_roofline(T, D, F, nnz, n_active, ms, hbm_gbs, fma_tflops, bf16_tflops=None,
                    union_sum=None):
    """The up+down projection against the method's work: bytes
    (``updown_bytes``) over HBM, 4 D flops per active entry over the FP32 FMA
    peak; binding = the longer of the two times.  With ``union_sum`` (the sum
    over 128-token blocks of the block's union of active neurons), also the
    tensor-pipe fraction of the union GEMMs (2 * 2 * 128 * D flops per union
    neuron of a block), a property of the tensor-core formulation."""
    nbytes = updown_bytes(T, D, F, nnz, n_active)
    flops = 4.0 * D * nnz
    t = ms * 1e-3
    t_hbm = nbytes / (hbm_gbs * 1e9)
    t_fma = flops / (fma_tflops * 1e12)
    out = {"bytes": nbytes, "flops": flops, "ms": ms,
           "hbm": {"achieved_gbs": nbytes / t / 1e9, "peak": hbm_gbs, "frac": t_hbm / t,
                   "t_us": t_hbm * 1e6},
           "alu": {"achieved_tflops": flops / t / 1e12, "peak": fma_tflops, "frac": t_fma / t,
                   "t_us": t_fma * 1e6}}
    out["bound"] = "alu" if t_fma >= t_hbm else "hbm"
    out["binding"] = {"bound": out["bound"], "t_us": max(t_hbm, t_fma) * 1e6,
                      "frac": max(t_hbm, t_fma) / t}
    if union_sum is not None and bf16_tflops:
        uf = 2 * 2.0 * 128 * D * union_sum
        out["union_tensor_frac"] = uf / t / (bf16_tflops * 1e12)
        out["union_flops"] = uf
    return out


def decode_roofline(T, D, F, nnz, n_active, ms, hbm_gbs, fma_tflops, bf16_tflops):
    """The one-kernel decode forward (twell_ffn_decode: gate, TwELL and the
    up + down projection) against the method's work: bytes = x in (bf16),
    W_g, the W_u and W_d rows of every neuron active in some row, y out
    (fp32) and the TwELL written; flops = 2 T D F for the gate (tensor
    cores) and 4 D per active entry (FP32 FMA pipe); binding = the longest
    of the three roofline times."""
    nbytes = (2.0 * T * D + 2.0 * F * D + 4.0 * n_active * D + 4.0 * T * D + 5.0 * nnz
              + T * (F // 128))
    flops = 4.0 * D * nnz
    tflops = 2.0 * T * D * F
    t = ms * 1e-3
    times = {"hbm": nbytes / (hbm_gbs * 1e9), "alu": flops / (fma_tflops * 1e12),
             "tensor": tflops / (bf16_tflops * 1e12)}
    out = {"bytes": nbytes, "flops": flops, "tensor_flops": tflops, "ms": ms,
           "hbm": {"achieved_gbs": nbytes / t / 1e9, "peak": hbm_gbs,
                   "frac": times["hbm"] / t, "t_us": times["hbm"] * 1e6},
           "alu": {"achieved_tflops": flops / t / 1e12, "peak": fma_tflops,
                   "frac": times["alu"] / t, "t_us": times["alu"] * 1e6},
           "tensor": {"achieved_tflops": tflops / t / 1e12, "peak": bf16_tflops,
                      "frac": times["tensor"] / t, "t_us": times["tensor"] * 1e6}}
    b = max(times, key=times.get)
    out["bound"] = b
    out["binding"] = {"bound": b, "t_us": times[b] * 1e6, "frac": times[b] / t}
    return out


def train_rooflines(D, F, T, nnz_ell, n_dense, nnz_total, kernels_ms, hbm_gbs, fma_tflops,
                    bf16_tflops):
    """Per-kernel rooflines of the training step (method's work).
    Sparse products of the ELL rows: 4 D flops per entry forward (u and y),
    12 D backward (da, dx from dz and du, dW_g, dW_u, dW_d), on the FP32 FMA
    pipe; dense overflow rows: 2 and 6 dense products of 2 n_dense D F flops
    on the tensor cores (bf16 rate; the hi/lo operand splits are not
    counted).  Bytes: every operand read and result written once.  The
    kernel's bound is the sum of its compute times against its HBM time,
    whichever is longer."""
    n_t = F // 128
    out = {}
    t = kernels_ms["twell_gate_pack"]
    out["twell_gate_pack"] = gate_roofline(T, D, F, nnz_total, t, hbm_gbs, bf16_tflops)
    b = T * n_t + 5.0 * nnz_total + 5.0 * nnz_ell + T * n_t + 4.0 * n_dense * F + 12.0 * T
    t = kernels_ms["twell_to_hybrid"] * 1e-3
    out["twell_to_hybrid"] = {"bound": "hbm", "bytes": b, "frac": b / (hbm_gbs * 1e9) / t,
                              "achieved_gbs": b / t / 1e9, "peak": hbm_gbs,
                              "ms": t * 1e3}
    for name, sp, dn, nbytes in (
            ("hybrid_ffn_fwd", 4.0 * D * nnz_ell, 2 * 2.0 * n_dense * D * F,
             2.0 * T * D + 4.0 * F * D + 9.0 * nnz_ell + 4.0 * T * D + 8.0 * n_dense * F),
            ("hybrid_ffn_bwd", 12.0 * D * nnz_ell, 6 * 2.0 * n_dense * D * F,
             2.0 * T * D + 6.0 * F * D + 4.0 * T * D + 9.0 * nnz_ell + 4.0 * T * D
             + 12.0 * F * D + 8.0 * n_dense * F)):
        t = kernels_ms[name] * 1e-3
        t_fma = sp / (fma_tflops * 1e12)
        t_tc = dn / (bf16_tflops * 1e12)
        t_hbm = nbytes / (hbm_gbs * 1e9)
        t_c = t_fma + t_tc
        out[name] = {"bound": "alu+tensor" if t_c >= t_hbm else "hbm",
                     "sparse_flops": sp, "dense_flops": dn, "bytes": nbytes,
                     "t_alu_us": t_fma * 1e6, "t_tensor_us": t_tc * 1e6,
                     "t_hbm_us": t_hbm * 1e6, "frac": max(t_c, t_hbm) / t, "ms": t * 1e3,
                     "hbm_frac": t_hbm / t}
    return out


def measure_fma_peak(dev, stream, iters=200000, reps=5):
    """FP32 FMA peak from the library's probe (scalar FFMA and packed f32x2
    chains): median of `reps` CUDA-event-timed launches each; the larger rate
    is the peak.  Returns a dict with both and the SM clock seen."""
    import torch
    import activation_sparse_gated_gate_gb300 as tw
    res = {}
    with ClockSampler(dev.index if dev.index is not None else 0, interval_ms=50) as clk:
        time.sleep(0.15)
        for packed in (False, True):
            buf, flops = tw.twell_probe_fma(packed, 1000, stream=stream, device=dev)
            torch.cuda.synchronize()
            ts = []
            for _ in range(reps):
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                _, flops = tw.twell_probe_fma(packed, iters, out=buf, stream=stream, device=dev)
                b.record(stream)
                torch.cuda.synchronize()
                ts.append(a.elapsed_time(b))
            ms = statistics.median(ts)
            res["ffma2" if packed else "ffma"] = {"tflops": flops / (ms * 1e-3) / 1e12,
                                                  "ms": ms}
            if not torch.isfinite(buf).all():
                raise RuntimeError("FMA probe produced non-finite sums")
    s = clk.summary()
    peak = max(r["tflops"] for r in res.values())
    return {"tflops": peak, "ffma": res["ffma"], "ffma2": res["ffma2"],
            "sm_mhz": s.get("sm_mhz"), "clock_reasons": s.get("reasons"),
            "how": ("twell_probe_fma: 2 CTAs x 512 threads per SM, 16 independent register "
                    f"FMA chains per thread x {iters} rounds, median of {reps} CUDA-event "
                    "timings; peak = the faster of scalar FFMA and packed fma.rn.f32x2")}


# ------------------------------------------------------------------ GPU path

def _block_unions(h, T, F):
    """Sum over the 128-token blocks of the number of neurons active in some
    row of the block (the gate kernel's block bitmaps)."""
    bits = h.block_bits.cpu().numpy().view(np.uint8)
    return int(np.unpackbits(bits).sum())


def plan_sizes(T, parts):
    """Token chunk sizes of the end-to-end pipeline: whole 128-token blocks
    (the last chunk may end in a partial block) in proportion to `parts`,
    summing to T, empty chunks dropped."""
    blocks = (T + 127) // 128
    cuts = [blocks * sum(parts[:i]) // sum(parts) for i in range(len(parts) + 1)]
    sizes = [min(T, 128 * cuts[i + 1]) - min(T, 128 * cuts[i]) for i in range(len(parts))]
    return [n for n in sizes if n > 0]


def _timed(fn, flush, stream, warmup, steps):
    """Mean CUDA-event time (ms) of fn() on `stream`, L2 flushed before each."""
    import torch
    for _ in range(warmup):
        flush.zero_()
        fn()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for e in ev:
        flush.zero_()
        e[0].record(stream)
        fn()
        e[1].record(stream)
    torch.cuda.synchronize()
    return statistics.mean(e[0].elapsed_time(e[1]) for e in ev)


def dense_context_forward(x, Wg, Wu, Wd, flush, stream, warmup, steps):
    """Context only: the dense gated FFN y = (ReLU(x W_g) * (x W_u)) W_d with
    torch bf16 matmuls (cuBLAS) at the same shape, every neuron computed."""
    def f():
        import torch
        return (torch.relu(x @ Wg.t()) * (x @ Wu.t())) @ Wd
    return _timed(f, flush, stream, warmup, steps)


def _up(b, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).to(dev)


class InferCase:
    """Device buffers of one inference workload and its two steps."""

    def __init__(self, w, dev, stream):
        import torch
        import activation_sparse_gated_gate_gb300 as tw
        self.w = w
        self.dev = dev
        self.stream = stream
        self.x, self.Wg, self.Wu, self.Wd = (_up(a, dev) for a in (w.x, w.Wg_t, w.Wu_t, w.Wd))
        self.h = tw.TwELL(w.T, w.F, w.width, device=dev)
        self.y = torch.empty((w.T, w.D), dtype=torch.float32, device=dev)
        self.y_cc = torch.empty((w.T, w.D), dtype=torch.float32, device=dev)
        self.ws_tc = torch.empty((tw.twell_workspace_size(tw.WS_FFN_FWD_TC, w.T, w.D, w.F, 0,
                                                          0),), dtype=torch.uint8, device=dev)
        self.y_tcs = torch.empty((w.T, w.D), dtype=torch.float32, device=dev)
        self.ws_tcs = torch.empty((tw.twell_workspace_size(tw.WS_FFN_FWD_TC_SORTED, w.T, w.D,
                                                           w.F, 0, 0),),
                                  dtype=torch.uint8, device=dev)
        # the tensor-core forward's down GEMM takes W_d in fp16: converted once
        # per model, like any weight preparation, outside the timed steps
        self.Wd16 = tw.twell_to_f16(self.Wd)
        # decode batches: the one-kernel forward (its own TwELL and y)
        self.dec = w.T <= 256 and w.D > 64
        if self.dec:
            self.h_dec = tw.TwELL(w.T, w.F, w.width, device=dev)
            self.y_dec = torch.empty((w.T, w.D), dtype=torch.float32, device=dev)

    def gate(self, stream=None):
        import activation_sparse_gated_gate_gb300 as tw
        tw.twell_gate_pack(self.x, self.Wg, self.h, stream=stream or self.stream)

    def fwd_tc(self, stream=None):
        import activation_sparse_gated_gate_gb300 as tw
        tw.twell_ffn_fwd_tc(self.x, self.h, self.Wu, self.Wd, y=self.y, ws=self.ws_tc,
                            Wd_f16=self.Wd16, stream=stream or self.stream)

    def fwd_tcs(self, stream=None):
        import activation_sparse_gated_gate_gb300 as tw
        tw.twell_ffn_fwd_tc_sorted(self.x, self.h, self.Wu, self.Wd, y=self.y_tcs,
                                   ws=self.ws_tcs, Wd_f16=self.Wd16,
                                   stream=stream or self.stream)

    def fwd_cc(self, stream=None):
        import activation_sparse_gated_gate_gb300 as tw
        tw.twell_ffn_fwd(self.x, self.h, self.Wu, self.Wd, y=self.y_cc,
                         stream=stream or self.stream)

    def fwd(self, kind, stream=None):
        {"tc": self.fwd_tc, "tcs": self.fwd_tcs, "cc": self.fwd_cc}[kind](stream)

    def step_dec(self, stream=None):
        import activation_sparse_gated_gate_gb300 as tw
        tw.twell_ffn_decode(self.x, self.Wg, self.Wu, self.Wd, self.h_dec, y=self.y_dec,
                            stream=stream or self.stream)

    def active_union(self):
        """Neurons active in some row (one untimed pack with z exported)."""
        import torch
        import activation_sparse_gated_gate_gb300 as tw
        z = torch.empty((self.w.T, self.w.F), dtype=torch.float32, device=self.dev)
        tw.twell_gate_pack(self.x, self.Wg, self.h, z_debug=z, stream=self.stream)
        n = int((z > 0).any(dim=0).sum().item())
        del z
        return n


FWD_NAMES = {"tc": "twell_ffn_fwd_tc", "tcs": "twell_ffn_fwd_tc_sorted", "cc": "twell_ffn_fwd",
             "dec": "twell_ffn_decode"}
# kernels of the library launched by one forward call: union scan + up +
# down GEMMs; the sorted variant adds two sort kernels and the union bitmaps
# (with the copy of x); the CUDA-core forward is one kernel (the gate is one
# more); the decode call is its gate kernel, then above 8 tokens the
# CUDA-core kernel
FWD_LAUNCHES = {"tc": 3, "tcs": 6, "cc": 1, "dec": 2}


def iter_launches(kinds, T=None):
    """Library kernels per timed iteration of infer_entry: the gate graph,
    each forward's graph and each step's graph (gate + forward; the decode
    call's step is its gate kernel, followed above 8 tokens by the CUDA-core
    kernel)."""
    n = 1
    for kd in kinds:
        if kd == "dec":
            n += 1 if T is not None and T <= 8 else FWD_LAUNCHES["dec"]
        else:
            n += 1 + 2 * FWD_LAUNCHES[kd]
    return n


def _capture(dev, fn):
    """A CUDA graph of fn() captured on a side stream (one warm-up call
    first, so per-call setup such as kernel attributes happens outside)."""
    import torch
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        fn(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        fn(side)
    torch.cuda.synchronize()
    return g


def infer_entry(args, case, flush, peaks, fma, steps, warmup, forward="auto", clk=None):
    """Time one inference workload.  Each call (the gate; each forward:
    tensor-core, tensor-core on activity-sorted blocks, CUDA-core fused) and
    each step (the gate followed by one forward) is captured once as a CUDA
    graph and replayed, after an L2 flush, between CUDA events on the
    launching stream: graph replay keeps the GPU's per-launch processing
    (several microseconds per kernel or memset issued one by one) out of the
    decode-sized calls, as a decode loop would.  K iterations run every graph
    once.  Returns the entry dict (times, tokens/s, rooflines) and the raw
    times."""
    import torch
    w = case.w
    stream = case.stream
    hbm, bf16, _, src = peaks
    kinds = ("tc", "tcs", "cc") + (("dec",) if case.dec else ())
    n_active = case.active_union()
    graphs = {"gate": _capture(case.dev, lambda st: case.gate(st))}
    for kd in kinds:
        if kd == "dec":
            graphs["step_dec"] = _capture(case.dev, lambda st: case.step_dec(st))
            continue
        graphs[kd] = _capture(case.dev, lambda st, kd=kd: case.fwd(kd, st))
        graphs["step_" + kd] = _capture(case.dev,
                                        lambda st, kd=kd: (case.gate(st), case.fwd(kd, st)))
    order = ["gate"] + [k for kd in kinds
                        for k in (("step_dec",) if kd == "dec" else (kd, "step_" + kd))]
    for _ in range(warmup):
        for name in order:
            flush.zero_()
            graphs[name].replay()
    torch.cuda.synchronize()
    for hh in (case.h, case.h_dec) if case.dec else (case.h,):
        if int(hh.status.item()) != 0:
            raise RuntimeError(f"device status flags {int(hh.status.item())} ({w.name})")
    K = steps
    ev = {name: [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
          for name in order}
    for i in range(K):
        for name in order:
            e = ev[name][i]
            flush.zero_()
            e[0].record(stream)
            graphs[name].replay()
            e[1].record(stream)
    torch.cuda.synchronize()
    for hh in (case.h, case.h_dec) if case.dec else (case.h,):
        if int(hh.status.item()) != 0:
            raise RuntimeError(f"device status flags {int(hh.status.item())} ({w.name})")
    t = {name: statistics.mean(ev[name][i][0].elapsed_time(ev[name][i][1]) for i in range(K))
         for name in order}
    step = {kd: max_over_ranks(t["step_" + kd], case.dev) for kd in kinds}
    if forward == "dec" and not case.dec:
        forward = "auto"  # the one-kernel forward exists for decode batches only
    if forward not in ("auto",) + kinds:
        raise RuntimeError(f"--forward {forward}: not available for {w.name}")
    best = min(step, key=step.get) if forward == "auto" else forward
    checks = [("tc", case.y), ("tcs", case.y_tcs)] + ([("dec", case.y_dec)] if case.dec else [])
    for kd, yk in checks:
        rel = float((yk - case.y_cc).norm() / max(float(case.y_cc.norm()), 1e-30))
        if not rel < 5e-3:
            raise RuntimeError(f"{FWD_NAMES[kd]} and the CUDA-core forward differ (relative "
                               f"{rel:.2e}, {w.name})")
    nnz = int(case.h.cnt.to(torch.int64).sum().item())
    union_sum = _block_unions(case.h, w.T, w.F)
    g_ms = t["gate"]
    ms_step = step[best]
    ws_n = int(os.environ.get("WORLD_SIZE", "1"))
    kernels = {"twell_gate_pack": gate_roofline(w.T, w.D, w.F, nnz, g_ms, hbm, bf16)}
    for kd in kinds:
        if kd == "dec":
            kernels[FWD_NAMES[kd]] = decode_roofline(w.T, w.D, w.F, nnz, n_active,
                                                     t["step_dec"], hbm, fma, bf16)
            continue
        kernels[FWD_NAMES[kd]] = updown_roofline(
            w.T, w.D, w.F, nnz, n_active, t[kd], hbm, fma, bf16,
            union_sum if kd == "tc" else None)
    entry = {
        "workload": w.name, "T": w.T, "d_model": w.D, "d_ff": w.F, "twell_width": w.width,
        "nnz": nnz, "density": nnz / (w.T * w.F), "active_neurons": n_active,
        "block_union_mean": union_sum / ((w.T + 127) // 128),
        "tokens_per_s": job_tokens_per_s(w.T, ws_n, ms_step), "ms_per_step": ms_step,
        "forward": FWD_NAMES[best],
        "steps_ms": {FWD_NAMES[kd]: step[kd] for kd in kinds},
        "kernels": kernels,
        "timing": ("each call and each step captured as a CUDA graph, replayed after an L2 "
                   "flush between CUDA events; mean of K"),
    }
    entry["launches_per_iteration"] = iter_launches(kinds, w.T)
    fwd_ms = t["step_dec"] if best == "dec" else t[best]
    return entry, {"use": best, "fwd_ms": fwd_ms, "gate_ms": 0.0 if best == "dec" else g_ms,
                   "fwd_name": FWD_NAMES[best], "nnz": nnz, "n_active": n_active,
                   "union_sum": union_sum}


def layer_stack(case, flush, steps, warmup, peaks, fma, nnz, n_active, layers=8):
    """The decode step as a decoding loop runs it: `layers` layers, each with
    weights of its own, in one CUDA graph.  Layer l's W_g, W_u and W_d are
    layer 0's with the neurons permuted (the same computation and the same
    active counts, in other memory); the layers' weights (about 100 MB each
    at d_model 2048, d_ff 8192) together exceed L2 several times, so every
    layer reads them from DRAM, with one L2 flush per replay.  Per-layer time
    = the graph's time / layers: the graph's own launch cost (several
    microseconds, paid once per replay) no longer lands on a single layer."""
    import torch
    import activation_sparse_gated_gate_gb300 as tw
    w, dev = case.w, case.dev
    hbm, bf16, _, _ = peaks
    gen = torch.Generator().manual_seed(2024)
    lay = []
    for l in range(layers):
        if l == 0:
            Wg, Wu, Wd = case.Wg, case.Wu, case.Wd
        else:
            perm = torch.randperm(w.F, generator=gen).to(dev)
            Wg, Wu, Wd = (case.Wg[perm].contiguous(), case.Wu[perm].contiguous(),
                          case.Wd[perm].contiguous())
        lay.append((Wg, Wu, Wd, tw.TwELL(w.T, w.F, w.width, device=dev),
                    torch.empty((w.T, w.D), dtype=torch.float32, device=dev)))

    def run(st):
        for Wg, Wu, Wd, h, y in lay:
            tw.twell_ffn_decode(case.x, Wg, Wu, Wd, h, y=y, stream=st)

    graph = _capture(dev, run)
    for _ in range(warmup):
        flush.zero_()
        graph.replay()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for e in ev:
        flush.zero_()
        e[0].record(case.stream)
        graph.replay()
        e[1].record(case.stream)
    torch.cuda.synchronize()
    if any(int(h.status.item()) for _, _, _, h, _ in lay):
        raise RuntimeError(f"device status flags in the layer stack ({w.name})")
    # the same y in every layer (a permutation of the neurons changes no sum's terms)
    rel = float((lay[-1][4] - lay[0][4]).norm() / max(float(lay[0][4].norm()), 1e-30))
    if not rel < 1e-4:
        raise RuntimeError(f"layer stack: permuted layers differ ({rel:.2e}, {w.name})")
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev) / layers
    r = decode_roofline(w.T, w.D, w.F, nnz, n_active, ms, hbm, fma, bf16)
    return {"layers": layers, "ms_per_layer": ms,
            "tokens_per_s_per_layer": job_tokens_per_s(w.T, int(os.environ.get("WORLD_SIZE", "1")), ms),
            "hbm_frac": r["hbm"]["frac"], "binding": r["binding"],
            "how": ("twell_ffn_decode for each of the layers in one CUDA graph, one L2 flush per "
                    "replay (the layers' weights exceed L2); layer l's weights are layer 0's with "
                    "the neurons permuted; time per layer = graph time / layers")}


def headline_roofline(entry, raw, peaks, fma_meta):
    """The `roofline` object of the JSON line: the step's dominant kernel
    against its binding roofline, with the HBM view and (for the tensor-core
    forward) the union-GEMM tensor fraction beside it."""
    hbm, bf16, _, src = peaks
    k = entry["kernels"]
    if raw["gate_ms"] >= raw["fwd_ms"]:
        g = k["twell_gate_pack"]
        name = "twell_gate_pack"
        tr, prof = _traffic(name, entry["workload"])
        if g["bound"] == "tensor":
            return {"kernel": name, "bound": "tensor", "achieved": g["tensor"]["achieved_tflops"],
                    "peak": bf16, "unit": "TFLOP/s", "frac": g["tensor"]["frac"],
                    "peak_source": f"{src} bf16 burst", "traffic": tr, "traffic_source": prof,
                    "work": "2 T D F flops"}
        return {"kernel": name, "bound": "hbm", "achieved": g["hbm"]["achieved_gbs"],
                "peak": hbm, "unit": "GB/s", "frac": g["hbm"]["frac"],
                "peak_source": f"{src} HBM copy", "traffic": tr, "traffic_source": prof,
                "work": "bytes of x, W_g and the TwELL"}
    name = raw["fwd_name"]
    r = k[name]
    tr, prof = _traffic(name, entry["workload"])
    if name == "twell_ffn_decode":
        b = r["binding"]["bound"]
        unit = "GB/s" if b == "hbm" else "TFLOP/s"
        ach = r["hbm"]["achieved_gbs"] if b == "hbm" else (
            r["alu"]["achieved_tflops"] if b == "alu" else r["tensor"]["achieved_tflops"])
        return {"kernel": name, "bound": b, "achieved": ach, "peak": r[b]["peak"], "unit": unit,
                "frac": r["binding"]["frac"],
                "peak_source": {"hbm": f"{src} HBM copy", "alu": "measured FFMA (twell_probe_fma)",
                                "tensor": f"{src} bf16 burst"}[b],
                "traffic": tr, "traffic_source": prof,
                "work": ("the whole decode step in one kernel: bytes = x in + W_g + W_u/W_d rows "
                         "of every active neuron + y out (fp32) + TwELL written; flops = 2 T D F "
                         "(gate, tensor cores) and 4 D per active entry (FP32 FMA); binding = "
                         "the longest of the three times"),
                "algorithmic_bytes": r["bytes"], "algorithmic_flops": r["flops"],
                "hbm": {"achieved": r["hbm"]["achieved_gbs"], "peak": hbm, "unit": "GB/s",
                        "frac": r["hbm"]["frac"], "peak_source": f"{src} HBM copy"},
                "binding": r["binding"]}
    out = {"kernel": name, "bound": r["bound"]}
    if r["bound"] == "alu":
        out.update({"achieved": r["alu"]["achieved_tflops"], "peak": r["alu"]["peak"],
                    "unit": "TFLOP/s", "frac": r["alu"]["frac"],
                    "peak_source": "measured FFMA (twell_probe_fma)"})
    else:
        out.update({"achieved": r["hbm"]["achieved_gbs"], "peak": hbm, "unit": "GB/s",
                    "frac": r["hbm"]["frac"], "peak_source": f"{src} HBM copy"})
    out.update({
        "traffic": tr, "traffic_source": prof,
        "work": ("method's work: 4 D flops per active entry (FP32 FMA pipe) and bytes = x in "
                 "(bf16) + y out (fp32) + W_u/W_d rows of every active neuron + TwELL entries; "
                 "binding roofline = the longer of the two times"),
        "algorithmic_bytes": r["bytes"], "algorithmic_flops": r["flops"],
        "hbm": {"achieved": r["hbm"]["achieved_gbs"], "peak": hbm, "unit": "GB/s",
                "frac": r["hbm"]["frac"], "peak_source": f"{src} HBM copy"},
        "alu": {"achieved": r["alu"]["achieved_tflops"], "peak": r["alu"]["peak"],
                "unit": "TFLOP/s", "frac": r["alu"]["frac"],
                "peak_source": "measured FFMA (twell_probe_fma)"},
        "binding": r["binding"],
    })
    if "union_tensor_frac" in r:
        out["union_tensor_frac"] = r["union_tensor_frac"]
        out["union_tensor_what"] = ("tensor-pipe fraction of the forward's two GEMMs over each "
                                    "128-token block's union of active neurons, of measured "
                                    "bf16 burst (fp16 operands run at the bf16 rate)")
    return out


def dense_context_train(x, Wg, Wu, Wd, dy, lam, flush, stream, warmup, steps):
    """Context only: the dense gated FFN's forward + backward (loss = <y, dy>
    + lam * sum(h)) with torch bf16 autograd (cuBLAS).  Returns (ms, peak
    bytes allocated by the step above its inputs and weights, with the step's
    gradients as torch returns them (bf16), peak bytes with dx and the weight
    gradients converted to fp32 as the sparse step returns them)."""
    import torch
    leaves = [t.detach().requires_grad_(True) for t in (x, Wg, Wu, Wd)]
    dyb = dy.to(torch.bfloat16)

    def f():
        xx, g, u, d = leaves
        hh = torch.relu(xx @ g.t())
        yy = (hh * (xx @ u.t())) @ d
        loss = (yy * dyb).sum(dtype=torch.float32) + lam * hh.sum(dtype=torch.float32)
        return torch.autograd.grad(loss, leaves)
    ms = _timed(f, flush, stream, warmup, steps)
    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    grads = f()
    torch.cuda.synchronize()
    peak_bf16 = torch.cuda.max_memory_allocated() - base
    del grads
    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    grads = [gr.float() for gr in f()]
    torch.cuda.synchronize()
    peak_f32 = torch.cuda.max_memory_allocated() - base
    del grads
    return ms, peak_bf16, peak_f32


def run_train(args, dev, flush, stream, peaks, fma):
    """Training step of the 2B-class layer (T=16384, D=2304, F=9216, mean 5%
    active, 3% of rows above the ELL capacity C=32): gate GEMM with TwELL
    epilogue (W=32), TwELL->hybrid, hybrid forward, hybrid backward with the
    L1 term.  Both variants of the hybrid matmuls are timed: the tensor-core
    one (hybrid_ffn_*_tc, the headline) and the CUDA-core one.  Returns a
    dict for the JSON line (per-kernel event times and rooflines, peak
    memory)."""
    import torch

    import activation_sparse_gated_gate_gb300 as tw
    import workloads

    w = workloads.config(3)
    hbm, bf16, bf16_sus, src = peaks
    x, Wg, Wu, Wd = (_up(a, dev) for a in (w.x, w.Wg_t, w.Wu_t, w.Wd))
    dy = torch.from_numpy(w.dy).to(dev)
    max_dense = 1024
    f32 = torch.float32
    K = args.train_steps
    ws_n = int(os.environ.get("WORLD_SIZE", "1"))
    n_t = w.F // 128
    variants = {
        "tensor-core": (tw.hybrid_ffn_fwd_tc, tw.hybrid_ffn_bwd_tc, tw.WS_HYBRID_FWD_TC,
                        tw.WS_HYBRID_BWD_TC),
        "cuda-core": (tw.hybrid_ffn_fwd, tw.hybrid_ffn_bwd, tw.WS_HYBRID_FWD,
                      tw.WS_HYBRID_BWD),
    }
    # per-call fp16 weight copies inside the tensor-core workspaces (W_d in
    # the forward; W_g, W_u, W_d in the backward): a caller training many
    # steps would keep them per model, so the memory comparison leaves them out
    wcopy = {"tensor-core": (1 + 3) * w.F * w.D * 2, "cuda-core": 0}
    names = ["twell_gate_pack", "twell_to_hybrid", "hybrid_ffn_fwd", "hybrid_ffn_bwd"]
    out = {}
    for vname, (fwd, bwd, op_f, op_b) in variants.items():
        torch.cuda.synchronize()
        mem_base = torch.cuda.memory_allocated()
        torch.cuda.reset_peak_memory_stats()
        # TwELL width = ELL capacity: only dense-backup rows spill, at most
        # max_dense * n_t slices
        h = tw.TwELL(w.T, w.F, w.cap, spill_cap=max_dense * n_t, device=dev)
        hyb = tw.Hybrid(w.T, w.F, w.cap, max_dense, device=dev)
        y = torch.empty((w.T, w.D), dtype=f32, device=dev)
        u_ell = torch.empty((w.T, n_t, w.cap), dtype=f32, device=dev)
        U_dense = torch.empty((max_dense, w.F), dtype=f32, device=dev)
        dx = torch.empty((w.T, w.D), dtype=f32, device=dev)
        dW = [torch.empty((w.F, w.D), dtype=f32, device=dev) for _ in range(3)]
        ws_f = tw._workspace(tw.twell_workspace_size(op_f, w.T, w.D, w.F, w.cap, max_dense), dev)
        ws_b = tw._workspace(tw.twell_workspace_size(op_b, w.T, w.D, w.F, w.cap, max_dense), dev)

        def launch(i):
            if i == 0:
                tw.twell_gate_pack(x, Wg, h, stream=stream)
            elif i == 1:
                tw.twell_to_hybrid(h, hyb, stream=stream)
            elif i == 2:
                fwd(x, hyb, Wu, Wd, y=y, u_ell=u_ell, U_dense=U_dense, ws=ws_f, stream=stream)
            else:
                bwd(x, hyb, u_ell, U_dense, Wg, Wu, Wd, dy, w.l1_coeff, dx=dx, dWg_t=dW[0],
                    dWu_t=dW[1], dWd=dW[2], ws=ws_b, stream=stream)

        flush.zero_()
        for i in range(4):
            launch(i)
        torch.cuda.synchronize()
        # every buffer of the step is the caller's (the library allocates none);
        # the flush buffer predates the baseline
        mem = torch.cuda.max_memory_allocated() - mem_base
        for _ in range(max(1, args.warmup)):
            flush.zero_()
            for i in range(4):
                launch(i)
        torch.cuda.synchronize()
        if int(h.status.item()) or int(hyb.status.item()):
            raise RuntimeError(f"device status flags set in the {vname} training step")
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K)]
        for k in range(K):
            flush.zero_()
            ev[k][0].record(stream)
            for i in range(4):
                launch(i)
                ev[k][i + 1].record(stream)
        torch.cuda.synchronize()
        per = {n: statistics.mean(ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(K))
               for i, n in enumerate(names)}
        ms = max_over_ranks(sum(per.values()), dev)
        nnz = int(h.cnt.to(torch.int64).sum().item())
        n_ell = hyb.n_ell
        n_dense = min(hyb.n_dense, max_dense)
        nnz_ell = int(hyb.ell_cnt[:n_ell].to(torch.int64).sum().item())
        roof = train_rooflines(w.D, w.F, w.T, nnz_ell, n_dense, nnz, per, hbm, fma, bf16)
        out[vname] = {"ms_per_step": ms, "tokens_per_s": job_tokens_per_s(w.T, ws_n, ms),
                      "kernels_ms": per, "roofline": roof, "peak_memory_bytes": mem,
                      "peak_memory_bytes_without_weight_copies": mem - wcopy[vname]}
        del h, hyb, y, u_ell, U_dense, dx, dW, ws_f, ws_b
        torch.cuda.empty_cache()
    d_ms, d_mem16, d_mem32 = dense_context_train(x, Wg, Wu, Wd, dy, w.l1_coeff, flush, stream,
                                                 2, K)
    head = out["tensor-core"]
    ours_mem = head["peak_memory_bytes_without_weight_copies"]
    return {
        "metric": "sparse gated-FFN training step (fwd+bwd) tokens/s per layer",
        "value": head["tokens_per_s"], "unit": "tokens/s", "ms_per_step": head["ms_per_step"],
        "steps": K, "scaling": "weak",
        "dtype": ("bf16 in; fp16 operands for the ELL products (h u, scaled dy/dz/du, "
                  "weights); fp32 accumulate and gradients"),
        "variant": "tensor-core hybrid matmuls (hybrid_ffn_fwd_tc / hybrid_ffn_bwd_tc)",
        "config": {"workload": w.name, "T": w.T, "d_model": w.D, "d_ff": w.F, "cap": w.cap,
                   "l1_coeff": w.l1_coeff, "nnz": nnz, "density": nnz / (w.T * w.F),
                   "nnz_ell": nnz_ell, "n_dense": n_dense, "max_dense": max_dense,
                   "l2": "flushed (512 MiB write) before every step"},
        "kernels_ms": head["kernels_ms"],
        "roofline": head["roofline"],
        "roofline_peaks": {"fma_tflops": fma, "fma_source": "measured FFMA (twell_probe_fma)",
                           "bf16_tflops": bf16, "hbm_gbs": hbm, "source": src},
        "cuda_core": out["cuda-core"],
        "peak_memory": {
            "ours_bytes": ours_mem,
            "dense_torch_bytes": d_mem32,
            "ratio": ours_mem / d_mem32,
            "pages_claim": "up to -28% peak training memory (paper section 4, memory)",
            "scope": ("device bytes the step allocates above its inputs (x, dy) and bf16 "
                      "weights, both producing fp32 dx and fp32 dW_g, dW_u, dW_d: ours = TwELL "
                      "+ hybrid + y + u + dense-row U + dx + dW + workspaces, without the fp16 "
                      "weight copies a caller would keep per model; dense = torch autograd "
                      "activations + its bf16 gradients converted to fp32"),
            "ours_with_weight_copies_bytes": head["peak_memory_bytes"],
            "cuda_core_bytes": out["cuda-core"]["peak_memory_bytes"],
            "dense_torch_bf16_grads_bytes": d_mem16},
        "dense_context": {
            "ms_per_step": d_ms, "tokens_per_s": job_tokens_per_s(w.T, ws_n, d_ms),
            "what": "torch bf16 autograd fwd+bwd of the dense gated FFN (cuBLAS), context only"},
    }


def run_stack(args, dev, flush, stream, layers=4):
    """A residual stack of `layers` 2B-class FFN layers (T=16384, D=2304,
    F=9216, 5 % mean density, 3 % dense rows, C=32), trained through the
    torch.autograd wrapper (tensor-core hybrid) against the same stack as
    dense torch bf16 autograd (cuBLAS).  One step = forward + backward of
    all layers with the L1 term.  Returns a dict for the JSON line."""
    import torch

    from activation_sparse_gated_gate_gb300.autograd import SparseFFNStack
    import workloads

    ws = []
    for l in range(layers):
        wl = workloads.config(3, seed=l)
        if l == 0:
            w0 = wl
        ws.append(tuple(torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
            torch.bfloat16).to(dev) for a in (wl.Wg_t, wl.Wu_t, wl.Wd)))
    x = torch.from_numpy(np.ascontiguousarray(w0.x).view(np.int16)).view(torch.bfloat16).to(dev)
    dy = torch.from_numpy(w0.dy).to(dev)
    lam = w0.l1_coeff
    stack = SparseFFNStack(ws, l1_coeff=lam, cap=w0.cap, max_dense=1024, tensor_cores=True)
    xs = x.clone().requires_grad_(True)

    def ours():
        xs.grad = None
        for prm in stack.parameters():
            prm.grad = None
        (stack(xs) * dy).sum().backward()

    dense_w = [[t.detach().clone().requires_grad_(True) for t in layer] for layer in ws]
    xd = x.clone().requires_grad_(True)

    def dense():
        xd.grad = None
        loss = 0.0
        h_sum = 0.0
        S = xd.float()
        for Wg, Wu, Wd in dense_w:
            for t in (Wg, Wu, Wd):
                t.grad = None
            X = S.to(torch.bfloat16)
            hh = torch.relu(X @ Wg.t())
            y = (hh * (X @ Wu.t())) @ Wd
            y = torch.cat([y[:, :-1], torch.zeros_like(y[:, -1:])], dim=1)
            h_sum = h_sum + hh.sum(dtype=torch.float32)
            S = S + y.float()
        loss = (S * dy).sum() + lam * h_sum
        loss.backward()

    K = max(2, args.train_steps)
    t_ours = _timed(ours, flush, stream, 2, K)
    flags = stack.status_flags()
    if flags:
        raise RuntimeError(f"device status flags {flags} in the stack")
    t_dense = _timed(dense, flush, stream, 2, K)
    n = int(os.environ.get("WORLD_SIZE", "1"))
    return {
        "metric": "FFN-stack training step (fwd+bwd through torch.autograd) tokens/s",
        "layers": layers, "workload": w0.name + f", {layers} residual layers",
        "ours": {"ms_per_step": t_ours, "tokens_per_s": job_tokens_per_s(w0.T, n, t_ours),
                 "path": "SparseFFNStack (tensor-core hybrid via the C-ABI; fp32 residual "
                         "stream and master weights, bf16 layer inputs)"},
        "dense_context": {"ms_per_step": t_dense,
                          "tokens_per_s": job_tokens_per_s(w0.T, n, t_dense),
                          "path": "torch bf16 autograd (cuBLAS), same stack (fp32 residual "
                                  "stream, bf16 weights and layer inputs)"},
        "ratio": t_dense / t_ours,
    }



def e2e_pipeline(args, case, flush, K):
    """End to end through the public API with host buffers: pinned x in,
    y out.  The batch is cut into token chunks on three streams (copy in,
    compute, copy out) so one chunk's copies overlap another chunk's kernels;
    every byte of both copies is inside the timed region, which runs from
    before the first copy-in to after the last copy-out.  The step is bound
    by the first copy-in, the sum of the chunks' compute and the copies that
    follow the last compute: short first and last chunks shorten the ends,
    few chunks keep the per-chunk fixed costs down.  Each candidate plan
    (fractions of the batch) runs each chunk on the forward measured faster
    at its size; the fastest plan is then timed."""
    import torch
    import activation_sparse_gated_gate_gb300 as tw
    w, dev, stream = case.w, case.dev, case.stream
    x, y, Wg, Wu, Wd, Wd16 = case.x, case.y, case.Wg, case.Wu, case.Wd, case.Wd16
    xh = x.cpu().pin_memory()
    yh = torch.empty_like(y, device="cpu").pin_memory()
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    # candidate plans: fractions of the batch per chunk (host copies run at
    # about 200 GB/s each way, about as long as the compute at the largest
    # layers; six and eight chunks measured slower at the 1.5B-class layer:
    # 1.39-1.48 ms against 1.30 ms for 4:7:4:1)
    plans = {"4 equal": (1, 1, 1, 1), "1:3:3:1": (1, 3, 3, 1), "1:8:5:2": (1, 8, 5, 2),
             "4:7:4:1": (4, 7, 4, 1)}
    chunk_state = {}

    def chunk_bufs(n):
        # a TwELL and a tensor-core workspace per chunk (sized for n tokens
        # and either tensor-core forward)
        h_c = tw.TwELL(n, w.F, w.width, device=dev)
        ws_c = torch.empty((tw.twell_workspace_size(tw.WS_FFN_FWD_TC_SORTED, n, w.D, w.F, 0,
                                                    0),), dtype=torch.uint8, device=dev)
        return h_c, ws_c

    def chunk_fwd(a, b, hc, kind, st):
        tw.twell_gate_pack(x[a:b], Wg, hc[0], stream=st)
        if kind == "cc":
            tw.twell_ffn_fwd(x[a:b], hc[0], Wu, Wd, y=y[a:b], stream=st)
        else:
            tw.twell_ffn_fwd_tc(x[a:b], hc[0], Wu, Wd, y=y[a:b], ws=hc[1], Wd_f16=Wd16,
                                stream=st, sorted_rows=kind == "tcs")

    def chunk_ms(n, kind):
        # one chunk of n tokens, device-resident, mean of 3 after a warm-up
        key = (n, kind)
        if key not in chunk_state:
            hc = chunk_bufs(n)
            c_ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            for it in range(4):
                if it == 1:
                    c_ev[0].record(stream)
                chunk_fwd(0, n, hc, kind, stream)
            c_ev[1].record(stream)
            torch.cuda.synchronize()
            chunk_state[key] = c_ev[0].elapsed_time(c_ev[1]) / 3
        return chunk_state[key]

    def kind_for(n):
        if args.forward not in ("auto", "dec"):
            return args.forward
        return min(("tc", "tcs", "cc"), key=lambda kd: chunk_ms(n, kd))

    def build_plan(parts):
        sizes = plan_sizes(w.T, parts)
        bounds = [sum(sizes[:i]) for i in range(len(sizes) + 1)]
        bufs = [chunk_bufs(n) for n in sizes]
        fwds = [kind_for(n) for n in sizes]

        def pipelined_step(origin):
            # fork from `origin`, one chunk per stage on each stream, join back
            for st in (s_in, s_cmp, s_out):
                st.wait_stream(origin)
            for c in range(len(sizes)):
                a, b = bounds[c], bounds[c + 1]
                with torch.cuda.stream(s_in):
                    x[a:b].copy_(xh[a:b], non_blocking=True)
                s_cmp.wait_stream(s_in)
                with torch.cuda.stream(s_cmp):
                    chunk_fwd(a, b, bufs[c], fwds[c], s_cmp)
                s_out.wait_stream(s_cmp)
                with torch.cuda.stream(s_out):
                    yh[a:b].copy_(y[a:b], non_blocking=True)
            origin.wait_stream(s_out)

        # one pipelined step recorded as a CUDA graph: replaying it costs one
        # host call, so the step is not bound by per-call host overhead
        pipelined_step(stream)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.graph(graph, stream=cap):
            pipelined_step(cap)
        torch.cuda.synchronize()
        return {"sizes": sizes, "fwds": fwds, "bufs": bufs, "graph": graph}

    def replay_ms(plan, n):
        e_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        for i in range(n):
            flush.zero_()
            e_ev[i][0].record(stream)
            plan["graph"].replay()
            e_ev[i][1].record(stream)
        torch.cuda.synchronize()
        return [e[0].elapsed_time(e[1]) for e in e_ev]

    built = {name: build_plan(parts) for name, parts in plans.items()}
    trial = {name: statistics.median(replay_ms(pl, 5)) for name, pl in built.items()}
    plan_name = min(trial, key=trial.get)
    plan = built[plan_name]
    e2e_ms = max_over_ranks(sum(replay_ms(plan, K)) / K, dev)
    hs = [b[0] for b in plan["bufs"]]
    if any(int(hh.status.item()) for hh in hs):
        raise RuntimeError("device status flags set in the end-to-end run")
    if not torch.equal(yh.to(dev), y):
        raise RuntimeError("end-to-end result differs from the device result")
    ws_n = int(os.environ.get("WORLD_SIZE", "1"))
    return {"value": job_tokens_per_s(w.T, ws_n, e2e_ms), "unit": "tokens/s",
            "h2d_bytes_per_step": x.numel() * 2, "d2h_bytes_per_step": y.numel() * 4,
            "ms_per_step": e2e_ms,
            "pipeline": (f"token chunks {plan['sizes']} (plan {plan_name}, the fastest of "
                         f"{len(plans)} tried untimed), copy-in / compute / copy-out streams, "
                         "replayed as one CUDA graph"),
            "forward": [FWD_NAMES[f] for f in plan["fwds"]],
            "forward_choice": ("per chunk, the faster measured at its size"
                               if args.forward == "auto"
                               else f"fixed by --forward {args.forward}"),
            "plans_tried_ms": trial}


def run_ours(args, head_cfg):
    import torch
    import torch.distributed as dist

    import workloads

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    flush = torch.empty((0 if args.no_flush else 512) * 1024 * 1024, dtype=torch.uint8,
                        device=dev)
    stream = torch.cuda.current_stream(dev)
    peaks = _peaks()
    hbm, bf16, bf16_sus, src = peaks
    fma_meta = measure_fma_peak(dev, stream)
    fma = fma_meta["tflops"]

    # ---- headline: one inference workload, timed with the clocks sampled
    w = workloads.config(head_cfg, T=args.T)
    case = InferCase(w, dev, stream)
    K = args.steps
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        entry, raw = infer_entry(args, case, flush, peaks, fma, K, args.warmup, args.forward)
    if ws > 1:
        dist.barrier()
    clk_sum = clk.summary()
    roof = headline_roofline(entry, raw, peaks, fma_meta)
    dense_ms = dense_context_forward(case.x, case.Wg, case.Wu, case.Wd, flush, stream, 3, K)
    entry["dense_context"] = {"ms_per_step": dense_ms,
                              "tokens_per_s": job_tokens_per_s(w.T, ws, dense_ms),
                              "what": "torch bf16 dense gated FFN (cuBLAS), all neurons"}
    e2e = None if args.no_e2e else e2e_pipeline(args, case, flush, K)
    energy = None
    if not args.no_energy:
        step = ((lambda: case.step_dec()) if raw["use"] == "dec"
                else (lambda: (case.gate(), case.fwd(raw["use"]))))
        e_ours = energy_per_token(step, w.T, stream, local)
        e_dense = energy_per_token(
            lambda: (torch.relu(case.x @ case.Wg.t()) * (case.x @ case.Wu.t())) @ case.Wd,
            w.T, stream, local)
        if e_ours and e_dense:
            energy = {"ours": e_ours, "dense_context": e_dense,
                      "ratio": e_ours["joules_per_token"] / e_dense["joules_per_token"],
                      "workload": w.name,
                      "how": ("board power (nvidia-smi power.draw, 100 ms samples, idle power "
                              "included) x CUDA-event time of ~1.5 s of back-to-back steps, "
                              "no L2 flush, per token")}
    del case
    torch.cuda.empty_cache()

    # ---- every other inference workload, each with its own entry
    configs = {}
    if not args.no_sweep:
        others = [(c, None) for c in (2, 1, 0) if c != head_cfg or args.T is not None]
        others += [(4, T) for T in workloads.DECODE_T]
        for c, T in others:
            wc = workloads.config(c, T=T)
            cc = InferCase(wc, dev, stream)
            e, r = infer_entry(args, cc, flush, peaks, fma, max(K, 10), args.warmup,
                               args.forward)
            e["roofline"] = headline_roofline(e, r, peaks, fma_meta)
            if c == 4:
                e["layer_stack"] = layer_stack(cc, flush, max(K, 10), args.warmup, peaks, fma,
                                               r["nnz"], r["n_active"])
            configs[wc.name] = e
            del cc
            torch.cuda.empty_cache()

    value = entry["tokens_per_s"]
    ms_step = entry["ms_per_step"]
    use_tc = raw["use"] in ("tc", "tcs")
    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": ("bf16 in, fp16 h*u and W_d in the down GEMM, fp32 accumulate, fp32 y"
                  if use_tc else "bf16 in, fp32 accumulate (FP32 FMA), fp32 y"),
        "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "d_model": w.D, "d_ff": w.F,
                   "twell_width": w.width, "nnz": entry["nnz"],
                   "active_neurons": entry["active_neurons"], "density": entry["density"],
                   "l2": ("NOT flushed (profiling run)" if args.no_flush
                          else "flushed (512 MiB write) before every step"),
                   "parallelism": f"replicas x{ws}",
                   "weights": ("bf16 W_g, W_u, W_d resident; the tensor-core forward's fp16 "
                               "copy of W_d is made once per model (twell_to_f16) outside the "
                               "timed region")},
        "e2e": e2e,
        # our kernels in the headline's timed region: every iteration replays
        # the gate, each forward and each step once
        "gpu_launches": K * entry["launches_per_iteration"],
        "roofline": roof,
        "headline": entry,
        "configs": configs,
        "fma_peak": fma_meta,
        "forward": raw["fwd_name"],
        "forward_choice": ("the fastest of the measured steps" if args.forward == "auto"
                           else f"fixed by --forward {args.forward}"),
        "energy": energy,
        "clocks": clk_sum,
    }
    if not args.no_train:
        out["train"] = run_train(args, dev, flush, stream, peaks, fma)
        out["train"]["n_gpus"] = ws
        if not args.no_stack:
            out["train"]["stack"] = run_stack(args, dev, flush, stream)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baselines(head_cfg, args.T, args.cpu_budget)
    if rank == 0:
        print(json.dumps(out))
    if ws > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=2,
                    help="headline workload (workloads.config index; default 2 = 1.5B-class)")
    ap.add_argument("--T", type=int, default=None, help="token count override")
    ap.add_argument("--ref-budget", type=float, default=10.0)
    ap.add_argument("--cpu-budget", type=float, default=5.0,
                    help="seconds per CPU-baseline measurement (four of them)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the non-headline inference workloads")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end pipeline")
    ap.add_argument("--no-train", action="store_true", help="skip the training-step section")
    ap.add_argument("--train-steps", type=int, default=5)
    ap.add_argument("--no-energy", action="store_true", help="skip the energy-per-token section")
    ap.add_argument("--no-stack", action="store_true", help="skip the multi-layer stack section")
    ap.add_argument("--forward", default="auto", choices=["auto", "tc", "tcs", "cc", "dec"],
                    help="inference forward of the steps and the end-to-end pipeline: the "
                         "faster measured one (auto) or a fixed one (profiling runs, where a "
                         "profiler's per-launch overhead distorts the comparison)")
    ap.add_argument("--no-flush", action="store_true",
                    help="skip the L2 flush (profiling runs only; not a valid bench number)")
    args = ap.parse_args()
    if args.impl == "reference":
        import workloads
        return run_reference(args, workloads.config(args.config, T=args.T), args.config)
    return run_ours(args, args.config)


if __name__ == "__main__":
    sys.exit(main())
