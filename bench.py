"""Benchmark of the activation-sparse gated FFN (TwELL) inference step on GB300.

One step = one pass of the inference hot path over one batch: the gate GEMM
with the TwELL-packing epilogue (twell_gate_pack) followed by the up+down
projection.  The headline step uses the tensor-core union-gather forward
(twell_ffn_fwd_tc); the CUDA-core fused kernel (twell_ffn_fwd) is timed in the
same run and reported beside it.  Default workload: the 0.5B-class layer,
T=8192 tokens, d_model=1536, d_ff=6144, ~1% active gate neurons, TwELL width
8 (seeded synthetic inputs, see workloads.py).

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.

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
    ("twell_ffn_fwd", "0.5B-class T=8192 D=1536 F=6144 1% W=8"): (
        108.88e6, "csrc/ffn_fwd.cu", "fdba64ead7a8eeb0", "profiles/ffn_fwd_0.5B_T8192.md"),
    ("twell_gate_pack", "0.5B-class T=8192 D=1536 F=6144 1% W=8"): (
        44.64e6, "csrc/gate_pack.cu", "7161047be7ce0d3d", "profiles/gate_pack_0.5B_T8192.md"),
    # the call's three kernels (union scan, up and down GEMMs)
    ("twell_ffn_fwd_tc", "0.5B-class T=8192 D=1536 F=6144 1% W=8"): (
        216.6e6, "csrc/ffn_tc.cu", "484e1de77c067100", "profiles/ffn_fwd_tc_0.5B_T8192.md"),
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
    import oracle
    x = w.x[rows]
    z = oracle.gate_preact(x, w.Wg_t)
    tw = oracle.twell_pack(z, 128, w.width)
    return oracle.ffn_forward_twell(x, tw, w.Wu_t, w.Wd)


def time_oracle(w, budget_s=10.0, chunk=64, seed=0):
    """Tokens/s of the oracle's inference path on sampled rows, run for about
    `budget_s` seconds of host CPU (at least one chunk)."""
    rng = np.random.default_rng(seed)
    done = 0
    t0 = time.perf_counter()
    while True:
        rows = np.sort(rng.choice(w.T, size=min(chunk, w.T), replace=False))
        oracle_step(w, rows)
        done += len(rows)
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return done / el, done, el


def run_reference(args, w):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    for _ in range(args.warmup):
        oracle_step(w, np.arange(min(16, w.T)))
    vals = []
    tot_rows = 0
    tot_s = 0.0
    for _ in range(args.steps):
        v, n, s = time_oracle(w, budget_s=args.ref_budget)
        vals.append(v)
        tot_rows += n
        tot_s += s
    value = tot_rows / tot_s
    cores = os.cpu_count()
    sample = (f"{tot_rows} sampled token rows of {w.name} over {args.steps} steps "
              f"(gate fp64 matmul + TwELL pack + fused up/down in fp64)")
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


def fma_peak_tflops(sm_count, sm_mhz):
    """FP32 FMA peak: 128 FP32 lanes per SM (4 sub-partitions x 32), 2 flops
    per FMA, at the given SM clock."""
    return sm_count * 128 * 2 * sm_mhz * 1e6 / 1e12


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
    import torch

    def f():
        return (torch.relu(x @ Wg.t()) * (x @ Wu.t())) @ Wd
    return _timed(f, flush, stream, warmup, steps)


def dense_context_train(x, Wg, Wu, Wd, dy, lam, flush, stream, warmup, steps):
    """Context only: the dense gated FFN's forward + backward (loss = <y, dy>
    + lam * sum(h)) with torch bf16 autograd (cuBLAS).  Returns (ms, peak
    bytes allocated by the step above its inputs and weights)."""
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
    peak = torch.cuda.max_memory_allocated() - base
    del grads
    return ms, peak


def run_train(args, dev, flush, stream):
    """Training step of the 2B-class layer (T=16384, D=2304, F=9216, mean 5%
    active, 3% of rows above the ELL capacity C=32): gate GEMM with TwELL
    epilogue (W=32), TwELL->hybrid, hybrid forward, hybrid backward with the
    L1 term.  Both variants of the hybrid matmuls are timed: the tensor-core
    one (hybrid_ffn_*_tc, the headline) and the CUDA-core one.  Returns a
    dict for the JSON line (per-kernel event times, peak memory)."""
    import torch

    import activation_sparse_gated_gate_gb300 as tw
    import workloads

    w = workloads.config(3)

    def up(b):
        return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(
            torch.bfloat16).to(dev)

    x, Wg, Wu, Wd = up(w.x), up(w.Wg_t), up(w.Wu_t), up(w.Wd)
    dy = torch.from_numpy(w.dy).to(dev)
    max_dense = 1024
    f32 = torch.float32
    K = args.train_steps
    ws_n = int(os.environ.get("WORLD_SIZE", "1"))
    variants = {
        "tensor-core": (tw.hybrid_ffn_fwd_tc, tw.hybrid_ffn_bwd_tc, tw.WS_HYBRID_FWD_TC,
                        tw.WS_HYBRID_BWD_TC),
        "cuda-core": (tw.hybrid_ffn_fwd, tw.hybrid_ffn_bwd, tw.WS_HYBRID_FWD,
                      tw.WS_HYBRID_BWD),
    }
    names = ["twell_gate_pack", "twell_to_hybrid", "hybrid_ffn_fwd", "hybrid_ffn_bwd"]
    out = {}
    for vname, (fwd, bwd, op_f, op_b) in variants.items():
        torch.cuda.synchronize()
        mem_base = torch.cuda.memory_allocated()
        torch.cuda.reset_peak_memory_stats()
        # TwELL width = ELL capacity: only dense-backup rows spill, at most
        # max_dense * n_t slices
        h = tw.TwELL(w.T, w.F, w.cap, spill_cap=max_dense * (w.F // 128), device=dev)
        hyb = tw.Hybrid(w.T, w.F, w.cap, max_dense, device=dev)
        y = torch.empty((w.T, w.D), dtype=f32, device=dev)
        u_ell = torch.empty((w.T, w.F // 128, w.cap), dtype=f32, device=dev)
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
        out[vname] = {"ms_per_step": ms, "tokens_per_s": job_tokens_per_s(w.T, ws_n, ms),
                      "kernels_ms": per, "peak_memory_bytes": mem}
        nnz = int(h.cnt.to(torch.int64).sum().item())
        n_dense = hyb.n_dense
        del h, hyb, y, u_ell, U_dense, dx, dW, ws_f, ws_b
        torch.cuda.empty_cache()
    d_ms, d_mem = dense_context_train(x, Wg, Wu, Wd, dy, w.l1_coeff, flush, stream, 2, K)
    head = out["tensor-core"]
    return {
        "metric": "sparse gated-FFN training step (fwd+bwd) tokens/s per layer",
        "value": head["tokens_per_s"], "unit": "tokens/s", "ms_per_step": head["ms_per_step"],
        "steps": K, "scaling": "weak",
        "dtype": "bf16 in, fp32 accumulate / gradients",
        "variant": "tensor-core hybrid matmuls (hybrid_ffn_fwd_tc / hybrid_ffn_bwd_tc)",
        "config": {"workload": w.name, "T": w.T, "d_model": w.D, "d_ff": w.F, "cap": w.cap,
                   "l1_coeff": w.l1_coeff, "nnz": nnz, "density": nnz / (w.T * w.F),
                   "n_dense": n_dense, "max_dense": max_dense,
                   "l2": "flushed (512 MiB write) before every step"},
        "kernels_ms": head["kernels_ms"],
        "cuda_core": out["cuda-core"],
        "peak_memory": {
            "tensor_core_bytes": head["peak_memory_bytes"],
            "cuda_core_bytes": out["cuda-core"]["peak_memory_bytes"],
            "dense_torch_bytes": d_mem,
            "scope": ("device bytes the step allocates above its inputs (x, dy) and bf16 "
                      "weights: ours = TwELL + hybrid + y + u + dense-row U + dx + fp32 dW + "
                      "workspaces; dense = torch autograd activations + bf16 grads")},
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


def run_ours(args, w):
    import torch
    import torch.distributed as dist

    import activation_sparse_gated_gate_gb300 as tw

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)

    def up(b):
        return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(
            torch.bfloat16).to(dev)

    x, Wg, Wu, Wd = up(w.x), up(w.Wg_t), up(w.Wu_t), up(w.Wd)
    h = tw.TwELL(w.T, w.F, w.width, device=dev)
    y = torch.empty((w.T, w.D), dtype=torch.float32, device=dev)
    y_cc = torch.empty((w.T, w.D), dtype=torch.float32, device=dev)
    ws_tc = torch.empty((tw.twell_workspace_size(tw.WS_FFN_FWD_TC, w.T, w.D, w.F, 0, 0),),
                        dtype=torch.uint8, device=dev)
    # the tensor-core forward's down GEMM takes W_d in fp16: converted once,
    # like any per-model weight preparation, outside the timed steps
    Wd16 = tw.twell_to_f16(Wd)
    flush = torch.empty((0 if args.no_flush else 512) * 1024 * 1024, dtype=torch.uint8,
                        device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        tw.twell_gate_pack(x, Wg, h, stream=stream)
        tw.twell_ffn_fwd_tc(x, h, Wu, Wd, y=y, ws=ws_tc, Wd_f16=Wd16, stream=stream)

    def step_cc():
        tw.twell_gate_pack(x, Wg, h, stream=stream)
        tw.twell_ffn_fwd(x, h, Wu, Wd, y=y_cc, stream=stream)

    # active-neuron union (for the fused kernel's algorithmic bytes), from
    # one untimed pack with the gate pre-activations exported
    zdbg = torch.empty((w.T, w.F), dtype=torch.float32, device=dev)
    tw.twell_gate_pack(x, Wg, h, z_debug=zdbg, stream=stream)
    n_active = int((zdbg > 0).any(dim=0).sum().item())
    del zdbg
    for _ in range(args.warmup):
        flush.zero_()
        step()
        flush.zero_()
        step_cc()
    torch.cuda.synchronize()
    if int(h.status.item()) != 0:
        raise RuntimeError(f"device status flags {int(h.status.item())}")

    # Each timed iteration runs both steps, each after its own L2 flush: the
    # headline (gate + tensor-core forward) and the CUDA-core one (gate +
    # fused kernel); events split every step into its two calls.
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    evc = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for i in range(K):
            flush.zero_()
            ev[i][0].record(stream)
            tw.twell_gate_pack(x, Wg, h, stream=stream)
            ev[i][1].record(stream)
            tw.twell_ffn_fwd_tc(x, h, Wu, Wd, y=y, ws=ws_tc, Wd_f16=Wd16, stream=stream)
            ev[i][2].record(stream)
            flush.zero_()
            evc[i][0].record(stream)
            tw.twell_gate_pack(x, Wg, h, stream=stream)
            evc[i][1].record(stream)
            tw.twell_ffn_fwd(x, h, Wu, Wd, y=y_cc, stream=stream)
            evc[i][2].record(stream)
        torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    t_k1 = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    t_tc = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]
    t_k1c = [evc[i][0].elapsed_time(evc[i][1]) for i in range(K)]
    t_k2 = [evc[i][1].elapsed_time(evc[i][2]) for i in range(K)]
    tc_step_ms = max_over_ranks(sum(a + b for a, b in zip(t_k1, t_tc)), dev) / K
    cc_ms = max_over_ranks(sum(a + b for a, b in zip(t_k1c, t_k2)), dev) / K
    # the headline is the faster of the two measured forwards at this
    # workload (the tensor-core one needs many 128-token blocks to fill the
    # GPU; decode-sized batches favour the CUDA-core kernel)
    use_tc = tc_step_ms <= cc_ms if args.forward == "auto" else args.forward == "tc"
    ms_step = tc_step_ms if use_tc else cc_ms
    value = job_tokens_per_s(w.T, ws, ms_step)
    if int(h.status.item()) != 0:
        raise RuntimeError(f"device status flags {int(h.status.item())}")
    # the two forwards compute the same y up to the bf16 rounding of h u
    rel = float((y - y_cc).norm() / y_cc.norm())
    if not rel < 5e-3:
        raise RuntimeError(f"tensor-core and CUDA-core forwards differ (relative {rel:.2e})")

    # end to end through the public API with host buffers: pinned x in, y out.
    # The batch is cut into token chunks on three streams (copy in, compute,
    # copy out) so one chunk's copies overlap another chunk's kernels; every
    # byte of both copies is inside the timed region, which runs from before
    # the first copy-in to after the last copy-out.  The step is bound by
    # the first copy-in, the sum of the chunks' compute and the copies that
    # follow the last compute: short first and last chunks shorten the ends,
    # few chunks keep the per-chunk fixed costs down.  Each candidate plan
    # (fractions of the batch) runs each chunk on the forward measured
    # faster at its size; the fastest plan is then timed.
    xh = x.cpu().pin_memory()
    yh = torch.empty_like(y, device="cpu").pin_memory()
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    plans = {"4 equal": (1, 1, 1, 1), "1:3:3:1": (1, 3, 3, 1), "1:8:5:2": (1, 8, 5, 2),
             "4:7:4:1": (4, 7, 4, 1)}

    chunk_state = {}

    def chunk_bufs(n):
        # a TwELL and a tensor-core workspace per chunk (sized for n tokens)
        h_c = tw.TwELL(n, w.F, w.width, device=dev)
        ws_c = torch.empty((tw.twell_workspace_size(tw.WS_FFN_FWD_TC, n, w.D, w.F, 0, 0),),
                           dtype=torch.uint8, device=dev)
        return h_c, ws_c

    def chunk_fwd(a, b, hc, fwd_tc, st):
        tw.twell_gate_pack(x[a:b], Wg, hc[0], stream=st)
        if fwd_tc:
            tw.twell_ffn_fwd_tc(x[a:b], hc[0], Wu, Wd, y=y[a:b], ws=hc[1], Wd_f16=Wd16,
                                stream=st)
        else:
            tw.twell_ffn_fwd(x[a:b], hc[0], Wu, Wd, y=y[a:b], stream=st)

    def chunk_ms(n, fwd_tc):
        # one chunk of n tokens, device-resident, mean of 3 after a warm-up
        key = (n, fwd_tc)
        if key not in chunk_state:
            hc = chunk_bufs(n)
            c_ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            for it in range(4):
                if it == 1:
                    c_ev[0].record(stream)
                chunk_fwd(0, n, hc, fwd_tc, stream)
            c_ev[1].record(stream)
            torch.cuda.synchronize()
            chunk_state[key] = c_ev[0].elapsed_time(c_ev[1]) / 3
        return chunk_state[key]

    def use_tc_for(n):
        if args.forward != "auto":
            return args.forward == "tc"
        return chunk_ms(n, True) <= chunk_ms(n, False)

    def build_plan(parts):
        sizes = plan_sizes(w.T, parts)
        bounds = [sum(sizes[:i]) for i in range(len(sizes) + 1)]
        bufs = [chunk_bufs(n) for n in sizes]
        fwds = [use_tc_for(n) for n in sizes]

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
    h2d = x.numel() * 2
    d2h = y.numel() * 4

    clk_sum = clk.summary()
    hbm, bf16, bf16_sus, src = _peaks()
    k1_ms = statistics.mean(t_k1)
    k2_ms = statistics.mean(t_k2)
    tc_ms = statistics.mean(t_tc)
    nnz = int(h.cnt.to(torch.int64).sum().item())
    k1_flops = 2.0 * w.T * w.D * w.F
    k1_tf = k1_flops / (k1_ms * 1e-3) / 1e12
    # tensor-core forward: its two GEMMs over each 128-token block's union of
    # active neurons, 2 * 128 * D * |U| flops each (the algorithmic work of
    # the formulation; padding rows and union positions are not counted)
    blk_union = _block_unions(h, w.T, w.F)
    tc_flops = 2 * 2.0 * 128 * w.D * blk_union
    tc_tf = tc_flops / (tc_ms * 1e-3) / 1e12
    # fused kernel: algorithmic bytes = x in (bf16) + y out (fp32) + W_u/W_d
    # rows of every neuron active in some row + the TwELL entries read (5 B
    # per nnz: fp32 value + u8 column, 1 B per count)
    k2_bytes = w.T * w.D * (2 + 4) + n_active * w.D * 2 * 2 + 5 * nnz + w.T * (w.F // 128)
    k2_gbs = k2_bytes / (k2_ms * 1e-3) / 1e9
    kernels = {
        "twell_gate_pack": {"ms": k1_ms, "tflops": k1_tf, "frac_bf16": k1_tf / bf16},
        "twell_ffn_fwd_tc": {"ms": tc_ms, "tflops": tc_tf, "frac_bf16": tc_tf / bf16,
                             "block_union_mean": blk_union / ((w.T + 127) // 128),
                             "what": "union scan + up GEMM + down GEMM (one C-ABI call)"},
        "twell_ffn_fwd": {"ms": k2_ms, "gbs": k2_gbs, "frac_hbm": k2_gbs / hbm,
                          "flops": 4.0 * w.D * nnz},
    }
    # The fused CUDA-core kernel's binding roofline is the FP32 FMA pipe (4 D
    # flops per active entry against 152 SMs x 128 lanes x 2 flops x clock),
    # not HBM: its algorithmic bytes take a fraction of the time its FMAs
    # need.  Both fractions are reported.
    tr2, prof2 = _traffic("twell_ffn_fwd", w.name)
    k2_tf = kernels["twell_ffn_fwd"]["flops"] / (k2_ms * 1e-3) / 1e12
    fma = fma_peak_tflops(torch.cuda.get_device_properties(dev).multi_processor_count,
                          clk_sum.get("sm_max_mhz") or 2070.0)
    kernels["twell_ffn_fwd"]["tflops"] = k2_tf
    kernels["twell_ffn_fwd"]["frac_fma"] = k2_tf / fma
    roof_cc = {"kernel": "twell_ffn_fwd", "bound": "alu", "achieved": k2_tf, "peak": fma,
               "unit": "TFLOP/s", "frac": k2_tf / fma,
               "peak_source": "FP32 FMA peak derived from SM count, 128 lanes/SM, max SM clock",
               "traffic": tr2, "traffic_source": prof2, "algorithmic_bytes": k2_bytes,
               "hbm": {"achieved": k2_gbs, "peak": hbm, "unit": "GB/s", "frac": k2_gbs / hbm,
                       "peak_source": f"{src} HBM copy"}}
    # headline step: the larger of its two calls bounds it
    if k1_ms >= (tc_ms if use_tc else k2_ms):
        tr, prof = _traffic("twell_gate_pack", w.name)
        roof = {"kernel": "twell_gate_pack", "bound": "tensor", "achieved": k1_tf,
                "peak": bf16, "unit": "TFLOP/s", "frac": k1_tf / bf16,
                "peak_source": f"{src} bf16 burst", "traffic": tr, "traffic_source": prof}
    elif not use_tc:
        roof = roof_cc
    else:
        tr, prof = _traffic("twell_ffn_fwd_tc", w.name)
        roof = {"kernel": "twell_ffn_fwd_tc", "bound": "tensor", "achieved": tc_tf,
                "peak": bf16, "unit": "TFLOP/s", "frac": tc_tf / bf16,
                "peak_source": f"{src} bf16 burst",
                "what": ("one call: union scan + up GEMM + down GEMM; flops = the two GEMMs "
                         "over each 128-token block's union of active neurons"),
                "traffic": tr, "traffic_source": prof}
    dense_ms = dense_context_forward(x, Wg, Wu, Wd, flush, stream, 3, K)
    energy = None
    if not args.no_energy:
        e_ours = energy_per_token(step if use_tc else step_cc, w.T, stream, local)
        e_dense = energy_per_token(
            lambda: (torch.relu(x @ Wg.t()) * (x @ Wu.t())) @ Wd, w.T, stream, local)
        if e_ours and e_dense:
            energy = {"ours": e_ours, "dense_context": e_dense,
                      "ratio": e_ours["joules_per_token"] / e_dense["joules_per_token"],
                      "how": ("board power (nvidia-smi power.draw, 100 ms samples, idle power "
                              "included) x CUDA-event time of ~1.5 s of back-to-back steps, "
                              "no L2 flush, per token")}

    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "d_model": w.D, "d_ff": w.F,
                   "twell_width": w.width, "nnz": nnz, "active_neurons": n_active,
                   "density": nnz / (w.T * w.F),
                   "l2": ("NOT flushed (profiling run)" if args.no_flush
                          else "flushed (512 MiB write) before every step"),
                   "parallelism": f"replicas x{ws}"},
        "e2e": {"value": job_tokens_per_s(w.T, ws, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "pipeline": (f"token chunks {plan['sizes']} (plan {plan_name}, the fastest of "
                             f"{len(plans)} tried untimed), copy-in / compute / copy-out "
                             "streams, replayed as one CUDA graph"),
                "forward": [("tensor-core" if f else "CUDA-core") for f in plan["fwds"]],
                "forward_choice": ("per chunk, the faster measured at its size"
                                   if args.forward == "auto"
                                   else f"fixed by --forward {args.forward}"),
                "plans_tried_ms": trial},
        # our kernels in the timed region per iteration: gate, union scan, up
        # and down GEMMs (headline) + gate and fused kernel (CUDA-core step)
        "gpu_launches": 6 * K,
        "roofline": roof,
        "kernels": kernels,
        "forward": ("tensor-core union gather (twell_ffn_fwd_tc)" if use_tc
                    else "CUDA-core fused kernel (twell_ffn_fwd)"),
        "forward_choice": ("the faster of the two measured steps" if args.forward == "auto"
                           else f"fixed by --forward {args.forward}"),
        "tensor_core": {"ms_per_step": tc_step_ms,
                        "tokens_per_s": job_tokens_per_s(w.T, ws, tc_step_ms),
                        "what": "gate + tensor-core union-gather forward (twell_ffn_fwd_tc)"},
        "cuda_core": {"ms_per_step": cc_ms, "tokens_per_s": job_tokens_per_s(w.T, ws, cc_ms),
                      "what": "gate + fused CUDA-core up/down kernel (twell_ffn_fwd)",
                      "roofline": roof_cc, "relative_difference_to_headline": rel},
        "dense_context": {
            "ms_per_step": dense_ms, "tokens_per_s": job_tokens_per_s(w.T, ws, dense_ms),
            "what": "torch bf16 dense gated FFN (cuBLAS), all neurons, context only"},
        "energy": energy,
        "clocks": clk_sum,
    }
    if not args.no_train:
        out["train"] = run_train(args, dev, flush, stream)
        out["train"]["n_gpus"] = ws
        if not args.no_stack:
            out["train"]["stack"] = run_stack(args, dev, flush, stream)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        v, n, s = time_oracle(w, budget_s=args.ref_budget)
        out["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": os.cpu_count(),
                               "kind": "oracle",
                               "sample": f"{n} sampled token rows in {s:.1f} s (fp64 oracle)"}
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
    ap.add_argument("--config", type=int, default=1)
    ap.add_argument("--T", type=int, default=None, help="token count override")
    ap.add_argument("--ref-budget", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-train", action="store_true", help="skip the training-step section")
    ap.add_argument("--train-steps", type=int, default=5)
    ap.add_argument("--no-energy", action="store_true", help="skip the energy-per-token section")
    ap.add_argument("--no-stack", action="store_true", help="skip the multi-layer stack section")
    ap.add_argument("--forward", default="auto", choices=["auto", "tc", "cc"],
                    help="inference forward of the headline and the end-to-end pipeline: the "
                         "faster measured one (auto) or a fixed one (profiling runs, where a "
                         "profiler's per-launch overhead distorts the comparison)")
    ap.add_argument("--no-flush", action="store_true",
                    help="skip the L2 flush (profiling runs only; not a valid bench number)")
    args = ap.parse_args()
    import workloads
    w = workloads.config(args.config, T=args.T)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
