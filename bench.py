"""Benchmark of the sparse-attention forward stack on GB300.

Default workload: the pages' 60M-model shape at training length, a 16-layer stack with
B=8, H=8, N=1024, D=64, bf16 Q/K/V ~ N(0,1), W=12, Fibonacci base, staggered-linear alpha,
mask (integer-distance) path.  One step = the forward of all 16 layers (16 launches,
replayed from a CUDA graph), inputs resident in HBM.  Each layer has its own Q/K/V, so a
step touches 537 MB > the 129 MB L2: no flush is needed between steps.

Prints one JSON line (rank 0).  `--impl reference` times the float64 CPU oracle instead
(on the host cores, on a bounded sample of the same workload).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-attn fwd tokens/s and achieved HBM GB/s vs roofline, 1 GB300 (N=1024/4096)"
UNIT = "tokens/s"
HBM_FALLBACK_GBS = 6800.0

WORKLOADS = {
    # name: (B, H, N, L, W, base, schedule, mode, dtype, config id for the seeds)
    "linear-stack-n1024": dict(B=8, H=8, N=1024, L=16, W=12, base="fib", sched="linear",
                               mode="mask", dtype="bf16", cfg=1),
    "coprime-fib-n4096": dict(B=2, H=8, N=4096, L=16, W=12, base="fib", sched="coprime",
                              mode="mask", dtype="bf16", cfg=2),
    "coprime-pow2-n4096": dict(B=2, H=8, N=4096, L=16, W=12, base="pow2", sched="coprime",
                               mode="mask", dtype="bf16", cfg=12),
    "learned-interp-n1024": dict(B=8, H=8, N=1024, L=16, W=10, base="fib", sched="learned",
                                 mode="interp", dtype="bf16", cfg=3),
    "long-mask-n131072": dict(B=1, H=8, N=131072, L=1, W=12, base="fib", sched="const1.5",
                              mode="mask", dtype="bf16", cfg=4),
    "long-interp-n131072": dict(B=1, H=8, N=131072, L=1, W=12, base="fib", sched="const1.5",
                                mode="interp", dtype="bf16", cfg=4),
}
DEFAULT = "linear-stack-n1024"
SECONDARY = ["coprime-fib-n4096", "coprime-pow2-n4096", "learned-interp-n1024", "long-mask-n131072",
             "long-interp-n131072"]
BACKWARD = "learned-interp-n1024"  # the training configuration: interpolated path, learned alpha


def alphas_for(w):
    """Per-layer alpha of a workload for the GPU arm: the library's own schedule planner."""
    if w["sched"] == "linear":
        from fibonacci_offset_sparse_gb300 import fib_attn as fa
        return fa.fib_attn_schedule(fa.FIB_SCHED_LINEAR, w["L"])
    if w["sched"] == "coprime":
        from fibonacci_offset_sparse_gb300 import fib_attn as fa
        return fa.fib_attn_schedule(fa.FIB_SCHED_COPRIME, w["L"], 7)
    if w["sched"] == "learned":
        from fibonacci_offset_sparse_gb300 import inputs
        return list(inputs.learned_alpha(w["L"], w["cfg"]))
    return [1.5] * w["L"]


def oracle_alphas_for(w):
    """The same alphas for the oracle legs, from the oracle's own schedule (nothing of the
    library is loaded there)."""
    import oracle
    if w["sched"] in ("linear", "coprime"):
        return oracle.schedule(w["sched"], w["L"])
    if w["sched"] == "learned":
        from fibonacci_offset_sparse_gb300 import inputs
        return list(inputs.learned_alpha(w["L"], w["cfg"]))
    return [1.5] * w["L"]


def compulsory_bytes(w):
    elt = 2 if w["dtype"] == "bf16" else 4
    return w["B"] * w["H"] * w["N"] * 64 * elt * 4  # Q, K, V read once + O written once


def compulsory_bytes_bwd(w):
    elt = 2 if w["dtype"] == "bf16" else 4
    # Q, K, V, O, dO read once + dQ, dK, dV written once (LSE and Delta apart)
    return w["B"] * w["H"] * w["N"] * 64 * elt * 8


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return HBM_FALLBACK_GBS, "fallback"


def source_hash(files):
    """Hash of the code of the named kernel sources: `//` comments, surrounding blanks and
    empty lines are left out, so that a profile summary stays valid across comment edits."""
    h = hashlib.sha256()
    for fn in files:
        with open(os.path.join(ROOT, "fibonacci_offset_sparse_gb300", "csrc", fn)) as f:
            for line in f:
                code = line.split("//", 1)[0].strip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def kernel_source_hash():
    """Hash of the forward kernels' sources (a profile summary names the one it was taken on)."""
    return source_hash(("common.cuh", "tc_common.cuh", "fwd.cu", "fwd_tc.cu"))


def backward_source_hash():
    """Hash of the tensor-core backward's sources."""
    return source_hash(("common.cuh", "tc_common.cuh", "bwd_tc.cu"))


def profile_fields(name):
    """The `- key: value` fields of a committed profile summary (empty when it is absent)."""
    p = os.path.join(ROOT, "profiles", name)
    vals = {}
    if os.path.exists(p):
        for line in open(p):
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                vals[k.strip()] = v.strip()
    return vals


def ncu_traffic(workload):
    """DRAM bytes of one layer's forward from the committed ncu summary of this workload:
    {"layer": steady-state bytes of both kernels of a layer inside the stack, "attend": the
    attention kernel's bytes in that capture}, or None when the summary is absent or was taken
    on a different kernel source."""
    vals = profile_fields(f"fwd_{workload}.md")
    if vals.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    try:
        return {"layer": float(vals["layer_dram_bytes_steady"]), "attend": float(vals["attend_dram_bytes_steady"])}
    except Exception:
        return None


def ncu_traffic_bwd(workload):
    """Steady-state DRAM bytes of one backward layer (its three kernels) from the committed ncu
    summary, or None when it is absent or was taken on a different kernel source."""
    vals = profile_fields(f"bwd_{workload}.md")
    if vals.get("kernel_source_sha256_16") != backward_source_hash():
        return None
    try:
        return float(vals["layer_dram_bytes_steady"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock/throttle sampling, every 20 ms, started before the warm-up (the tool
    takes a while to start); summary() keeps the samples stamped inside the timed region
    marked by mark_start()/mark_end()."""
    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.5)  # let the first samples arrive before the timed region
        except Exception:
            self.proc = None
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        import datetime
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(f[1]), float(f[2]),
                             {n for n, v in zip(names, f[5:9]) if v.lower().startswith("active")}))
            except ValueError:
                continue
        inside = [r for r in rows if self.t0 is not None and self.t0 - 0.02 <= r[0] <= self.t1 + 0.02]
        # a timed region shorter than the sampling period may hold no sample: then the two
        # samples around it stand for it
        use = inside
        if not use and self.t0 is not None:
            mid = (self.t0 + self.t1) / 2
            use = sorted(rows, key=lambda r: abs(r[0] - mid))[:2]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = set().union(*(r[3] for r in use))
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": use[-1][2],
                "reasons": sorted(reasons), "samples": len(use), "samples_inside_timed_region": len(inside)}


# ----------------------------------------------------------------------------- ranks
def barrier(world):
    """All ranks meet here (a no-op for one process)."""
    if world > 1:
        import torch
        torch.distributed.barrier()


def max_over_ranks(x, world):
    """The largest value of x over the ranks (x itself for one process): the job's time is
    its slowest replica's.  Works on NCCL (a CUDA tensor) and gloo (a CPU tensor)."""
    if world == 1:
        return x
    import torch
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.distributed.get_backend() == "nccl" \
        else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_rank, world, ms):
    """Whole-job throughput: every rank processes units_per_rank (weak scaling) in ms."""
    return units_per_rank * world / (ms / 1e3)


# ----------------------------------------------------------------------------- GPU arm
def setup(w, device):
    import torch
    from fibonacci_offset_sparse_gb300 import fib_attn as fa
    from fibonacci_offset_sparse_gb300 import inputs
    bk = fa.FIB_BASE_FIBONACCI if w["base"] == "fib" else fa.FIB_BASE_POW2
    mode = fa.FIB_MODE_MASK if w["mode"] == "mask" else fa.FIB_MODE_INTERP
    alphas = alphas_for(w)
    plan = fa.fib_attn_plan_create(bk, alphas, w["W"], w["N"], mode)
    host = [inputs.qkv(w["B"], w["H"], w["N"], 64, w["cfg"], l, w["dtype"]) for l in range(w["L"])]
    dev = [tuple(t.to(device) for t in layer) for layer in host]
    outs = [torch.empty_like(d[0]) for d in dev]
    lses = [torch.empty(w["B"], w["H"], w["N"], dtype=torch.float32, device=device) for _ in dev]
    adev = None
    if w["mode"] == "interp":
        adev = torch.tensor(alphas, dtype=torch.float32, device=device)
    # The layer stack reuses one forward workspace (the prepared K/V are scratch that each
    # layer's attention consumes at once, as in a model); timing one half alone uses one
    # workspace per layer (`wss`), so that every launch reads its own layer's data.
    need = fa.fib_attn_fwd_workspace_size(plan, w["B"], w["H"], w["N"], dev[0][0].dtype)
    wss = [torch.empty(need, dtype=torch.uint8, device=device) if need else None for _ in dev]
    return plan, host, dev, outs, lses, adev, wss


def shared_ws(wss):
    """The stack's one workspace, repeated per layer."""
    return [wss[0]] * len(wss)


def run_stack(fa, plan, dev, outs, lses, adev, wss):
    for l, (q, k, v) in enumerate(dev):
        fa.fib_attn_fwd(plan, l, q, k, v, o=outs[l], lse=lses[l], alpha_dev=adev, workspace=wss[l])


def kernels_per_layer(wss):
    return 2 if wss[0] is not None else 1


def time_graph(torch, stream, device, fn, steps, warmup):
    """Milliseconds per replay of a CUDA graph of fn(), CUDA events on `stream`."""
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        fn()
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize(device)
    return e0.elapsed_time(e1) / steps


def time_halves(fa, torch, stream, device, plan, dev, outs, lses, adev, wss, steps, warmup):
    """Per-launch device time of each kernel of the bf16 forward, each timed alone: a graph
    of the L layers' attention launches (every layer's own prepared K/V, Q and O) and one
    of the L preparation launches."""
    if wss[0] is None:
        return None
    L = len(dev)

    def attend():
        for l, (q, _, _) in enumerate(dev):
            fa.fib_attn_fwd_attend(plan, l, q, wss[l], o=outs[l], lse=lses[l], alpha_dev=adev)

    def prepare():
        for l, (_, k, v) in enumerate(dev):
            fa.fib_attn_fwd_prepare_kv(plan, k, v, workspace=wss[l])

    with torch.cuda.stream(stream):
        prepare()
    t_att = time_graph(torch, stream, device, attend, steps, warmup) / L
    t_prep = time_graph(torch, stream, device, prepare, steps, warmup) / L
    return {"attend_ms": t_att, "prepare_ms": t_prep}


def time_device(w, steps, warmup, device, rank, world):
    import torch
    from fibonacci_offset_sparse_gb300 import fib_attn as fa
    plan, host, dev, outs, lses, adev, wss = setup(w, device)
    ws1 = shared_ws(wss)
    stream = torch.cuda.Stream(device)
    with torch.cuda.stream(stream):
        run_stack(fa, plan, dev, outs, lses, adev, ws1)  # first call outside capture
    torch.cuda.synchronize(device)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        run_stack(fa, plan, dev, outs, lses, adev, ws1)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(device.index if device.index is not None else 0) as clk:
        for _ in range(warmup):
            graph.replay()
        torch.cuda.synchronize(device)
        barrier(world)
        clk.mark_start()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(steps):
                graph.replay()
            e1.record(stream)
        torch.cuda.synchronize(device)
        clk.mark_end()
    ms = max_over_ranks(e0.elapsed_time(e1), world)
    kpl = kernels_per_layer(wss)
    res = dict(ms_total=ms, ms_per_step=ms / steps, launches=kpl * w["L"] * steps, clocks=clk.summary())
    # end to end through the public API: pinned host inputs -> device -> 16 layers -> host O
    pinned = [tuple(t.pin_memory() for t in layer) for layer in host]
    o_host = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
    h2d = sum(t.numel() * t.element_size() for layer in pinned for t in layer)
    d2h = sum(o.numel() * o.element_size() for o in o_host)
    e2e_steps = max(1, min(steps, 5))

    # Per layer: host->device copy on one stream, the forward on `stream`, device->host copy
    # of O on a third stream, so that layer l+1's copies overlap layer l's attention (the
    # host buffers are pinned).  Events order each layer's buffers across steps.
    h2d_stream, d2h_stream = torch.cuda.Stream(device), torch.cuda.Stream(device)
    L = len(pinned)
    copied = [torch.cuda.Event() for _ in range(L)]
    computed = [torch.cuda.Event() for _ in range(L)]
    returned = [torch.cuda.Event() for _ in range(L)]
    started = torch.cuda.Event()

    def e2e_step(first):
        for l, (q, k, v) in enumerate(pinned):
            with torch.cuda.stream(h2d_stream):
                h2d_stream.wait_event(started)
                if not first:
                    h2d_stream.wait_event(computed[l])  # the previous step is done with dev[l]
                dev[l][0].copy_(q, non_blocking=True)
                dev[l][1].copy_(k, non_blocking=True)
                dev[l][2].copy_(v, non_blocking=True)
                copied[l].record(h2d_stream)
            stream.wait_event(copied[l])
            if not first:
                stream.wait_event(returned[l])  # the previous step's O of layer l is on the host
            with torch.cuda.stream(stream):
                fa.fib_attn_fwd(plan, l, *dev[l], o=outs[l], lse=lses[l], alpha_dev=adev, workspace=ws1[l])
                computed[l].record(stream)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(computed[l])
                o_host[l].copy_(outs[l], non_blocking=True)
                returned[l].record(d2h_stream)
        stream.wait_stream(d2h_stream)  # the step ends when every O is on the host

    with torch.cuda.stream(stream):
        started.record(stream)
        e2e_step(True)
        torch.cuda.synchronize(device)
        e0.record(stream)
        started.record(stream)
        for s in range(e2e_steps):
            e2e_step(False)
        e1.record(stream)
    torch.cuda.synchronize(device)
    ms_e2e = max_over_ranks(e0.elapsed_time(e1), world)
    res.update(ms_e2e_per_step=ms_e2e / e2e_steps, h2d=h2d, d2h=d2h, e2e_steps=e2e_steps,
               e2e_launches=kpl * w["L"] * e2e_steps)
    res["halves"] = time_halves(fa, torch, stream, device, plan, dev, outs, lses, adev, wss, steps, warmup)
    plan.close()
    return res


def time_backward(w, steps, warmup, device, prepared=True, with_forward=False):
    """Backward of the L-layer stack (dQ, dK, dV and dalpha of every layer), replayed from a
    CUDA graph: milliseconds per step and per launch of the backward.  prepared: each layer's
    backward takes the K'/V' rows its forward prepared (fib_attn_bwd_prepared, as a training
    step that keeps the forward's workspace does); else it prepares them from k and v
    (fib_attn_bwd).  with_forward: the graph holds the forward of the stack, then its
    backward (a training step's attention: the layers' forwards keep their workspaces)."""
    import torch
    from fibonacci_offset_sparse_gb300 import fib_attn as fa
    from fibonacci_offset_sparse_gb300 import inputs
    plan, host, dev, outs, lses, adev, wss = setup(w, device)
    stream = torch.cuda.Stream(device)
    with torch.cuda.stream(stream):
        run_stack(fa, plan, dev, outs, lses, adev, wss)
    dOs = [inputs.upstream_grad(w["B"], w["H"], w["N"], 64, w["cfg"], l, w["dtype"]).to(device)
           for l in range(w["L"])]
    grads = [tuple(torch.empty_like(d[0]) for _ in range(3)) for d in dev]
    dal = [torch.empty(1, dtype=torch.float32, device=device) for _ in dev]
    # one backward workspace for the stack: the prepared rows and (P, dS) pairs are scratch
    # that each layer's backward consumes before the next layer's starts, as in a model
    need = fa.fib_attn_bwd_workspace_size(plan, w["B"], w["H"], w["N"])
    bws = [torch.empty(need, dtype=torch.uint8, device=device)] * len(dev)

    def bwd_stack():
        if with_forward:
            run_stack(fa, plan, dev, outs, lses, adev, wss)
        for l, (q, k, v) in enumerate(dev):
            if prepared:  # wss[l]: layer l's forward workspace, filled by run_stack above
                fa.fib_attn_bwd_prepared(plan, l, q, wss[l], outs[l], lses[l], dOs[l], *grads[l], dalpha=dal[l],
                                         alpha_dev=adev, workspace=bws[l])
            else:
                fa.fib_attn_bwd(plan, l, q, k, v, outs[l], lses[l], dOs[l], *grads[l], dalpha=dal[l],
                                alpha_dev=adev, workspace=bws[l])

    with torch.cuda.stream(stream):
        bwd_stack()
    torch.cuda.synchronize(device)
    ms = time_graph(torch, stream, device, bwd_stack, steps, warmup)
    plan.close()
    return {"ms_per_step": ms, "us_per_layer": ms * 1e3 / w["L"]}


def time_decode(mode, B, H, N, L, steps, warmup, device):
    """One new token at position N-1 against an N-row cache, through the L layers of a
    plan (Fibonacci base, alpha = 1.5, W = 12; interp takes alpha from the device as a
    learned alpha would): microseconds per token, replayed from a CUDA graph."""
    import torch
    from fibonacci_offset_sparse_gb300 import fib_attn as fa
    from fibonacci_offset_sparse_gb300 import inputs
    m = fa.FIB_MODE_MASK if mode == "mask" else fa.FIB_MODE_INTERP
    plan = fa.fib_attn_plan_create(fa.FIB_BASE_FIBONACCI, [1.5] * L, 12, N, m)
    adev = torch.full((L,), 1.5, dtype=torch.float32, device=device) if mode == "interp" else None
    caches = [tuple(t.to(device) for t in inputs.qkv(B, H, N, 64, 50, l, "bf16")[1:]) for l in range(L)]
    qs = [inputs.normal((B, H, 64), 51, l, inputs.TENSOR_Q, "bf16").to(device) for l in range(L)]
    outs = [torch.empty_like(q) for q in qs]
    stream = torch.cuda.Stream(device)

    def step():
        for l in range(L):
            fa.fib_attn_decode(plan, l, N - 1, qs[l], *caches[l], o=outs[l], alpha_dev=adev, want_lse=False)

    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize(device)
    ms = time_graph(torch, stream, device, step, steps, warmup)
    plan.close()
    return ms * 1e3


def time_dense_ours(w, device, reps=20):
    """Dense causal attention with the same RoPE through the library's own dense kernel
    (fib_attn_dense_fwd: K'/V' preparation + the dense blocked kernel), one layer of the
    workload's shape: milliseconds per layer, CUDA events on the launching stream."""
    import torch
    from fibonacci_offset_sparse_gb300 import fib_attn as fa
    from fibonacci_offset_sparse_gb300 import inputs
    plan = fa.fib_attn_plan_create(fa.FIB_BASE_FIBONACCI, [1.0], 1, w["N"], fa.FIB_MODE_MASK)
    q, k, v = (t.to(device) for t in inputs.qkv(w["B"], w["H"], w["N"], 64, w["cfg"], 0, w["dtype"]))
    o = torch.empty_like(q)
    lse = torch.empty(w["B"], w["H"], w["N"], dtype=torch.float32, device=device)
    need = int(fa.lib().fib_attn_dense_fwd_workspace_size(plan.handle, w["B"], w["H"], w["N"], fa.FIB_DTYPE_BF16))
    ws = torch.empty(need, dtype=torch.uint8, device=device)
    stream = torch.cuda.Stream(device)

    def one():
        fa.fib_attn_dense_fwd(plan, q, k, v, o=o, lse=lse, workspace=ws)

    with torch.cuda.stream(stream):
        one()
    torch.cuda.synchronize(device)
    ms = time_graph(torch, stream, device, one, reps, 3)
    plan.close()
    return ms


def time_dense_sdpa(w, device, reps=20):
    """Dense causal attention on the same shape through PyTorch's fused attention (a library
    kernel, timed only as the dense comparison point): milliseconds per layer."""
    import torch
    from fibonacci_offset_sparse_gb300 import inputs
    q, k, v = (t.to(device) for t in inputs.qkv(w["B"], w["H"], w["N"], 64, w["cfg"], 0, w["dtype"]))
    f = torch.nn.functional.scaled_dot_product_attention
    for _ in range(3):
        f(q, k, v, is_causal=True)
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        f(q, k, v, is_causal=True)
    e1.record()
    torch.cuda.synchronize(device)
    return e0.elapsed_time(e1) / reps


# ----------------------------------------------------------------------------- CPU oracle
def time_oracle(w, n_layers_sample, heads=None):
    """Oracle seconds per layer of the workload on a sample of layers and heads (every batch
    row, the full sequence); returns (seconds per full layer, sample description, seconds
    actually measured)."""
    import numpy as np  # noqa: F401
    import oracle
    from fibonacci_offset_sparse_gb300 import inputs
    alphas = oracle_alphas_for(w)
    base = (lambda N: oracle.fibonacci_base()) if w["base"] == "fib" else oracle.pow2_base
    if heads is None:
        heads = w["H"] if w["N"] <= 4096 else 1
    layers = list(range(min(n_layers_sample, w["L"])))
    t_total = 0.0
    for l in layers:
        q, k, v = inputs.qkv(w["B"], w["H"], w["N"], 64, w["cfg"], l, w["dtype"])
        qf, kf, vf = (inputs.as_f64(x[:, :heads]) for x in (q, k, v))
        t0 = time.perf_counter()
        oracle.attend(qf, kf, vf, alphas[l], base(w["N"]), w["W"], w["mode"])
        t_total += time.perf_counter() - t0
    frac_heads = heads / w["H"]
    per_layer = t_total / len(layers) / frac_heads
    desc = (f"oracle forward on {len(layers)} of {w['L']} layers" +
            (f", {heads} of {w['H']} heads" if heads < w["H"] else "") + ", float64 numpy, 1 thread")
    return per_layer, desc, t_total


def oracle_tokens_per_s(w, per_layer_s):
    return w["B"] * w["N"] / (per_layer_s * w["L"])


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT, choices=sorted(WORKLOADS))
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    w = WORKLOADS[args.workload]
    cfg = {"workload": args.workload, "B": w["B"], "H": w["H"], "N": w["N"], "D": 64, "layers": w["L"],
           "W": w["W"], "base": {"fib": "fibonacci 1..987", "pow2": "powers of two < N"}[w["base"]],
           "schedule": w["sched"], "path": w["mode"] + " forward",
           "l2": "no flush: each step reads every layer's own Q/K/V (inputs > L2 per step)"}

    if args.impl == "reference":
        if rank != 0:
            return
        # One reference step = the oracle's forward of one layer on two of the heads (every
        # batch row, the whole sequence): a bounded sample of the workload.  ms_per_step is the
        # time such a step takes; value is the workload's tokens/s at that measured rate (the
        # work grows linearly in layers and heads).
        sample_heads = min(2, w["H"])
        for _ in range(args.warmup):
            time_oracle(w, 1, sample_heads)
        step_s = []
        t0 = time.perf_counter()
        for s in range(args.steps):
            pl, desc, measured = time_oracle(w, 1, sample_heads)
            step_s.append(measured)
        el = time.perf_counter() - t0
        ms_step = statistics.mean(step_s) * 1e3
        per_layer = statistics.mean(step_s) * w["H"] / sample_heads
        v = oracle_tokens_per_s(w, per_layer)
        rcfg = dict(cfg, reference_step=f"oracle forward of 1 of {w['L']} layers on {sample_heads} of {w['H']} "
                                        f"heads (B={w['B']}, N={w['N']}); value = the {w['L']}-layer stack's "
                                        "tokens/s at the measured rate")
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic N(0,1), seeded", "config": rcfg,
                "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": desc,
                                 "host_cores_available": len(os.sched_getaffinity(0))},
                "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                "wall_s": el}
        print(json.dumps(line))
        return

    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    from fibonacci_offset_sparse_gb300 import fib_attn as fa
    fa.lib()  # fails loudly when the library is not built

    r = time_device(w, args.steps, args.warmup, device, rank, world)
    tokens_step = w["B"] * w["N"]
    value = job_value(tokens_step, world, r["ms_per_step"])
    e2e_value = job_value(tokens_step, world, r["ms_e2e_per_step"])
    peak, peak_kind = read_peaks()
    layer_s = r["ms_per_step"] / 1e3 / w["L"]
    # The roofline is taken over a layer's whole forward (K'/V' preparation + attention, the
    # launches a user's fib_attn_fwd makes), timed inside the step: the layer's compulsory
    # bytes (Q, K, V read once, O written once) over its time.  The attention kernel timed
    # alone (it reads the prepared K'/V' instead of K and V) is reported beside it.
    launch_s = r["halves"]["attend_ms"] / 1e3 if r["halves"] else layer_s
    algo = compulsory_bytes(w)
    achieved = algo / layer_s / 1e9
    traffic = ncu_traffic(args.workload)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w["dtype"],
        "data": "synthetic: i.i.d. N(0,1) Q/K/V per layer (seeded), shaped like the pages' 60M model",
        "config": cfg,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic["layer"] if traffic else None,
                     "peak_kind": peak_kind + (" (hbm_gbs, burst copy)" if peak_kind == "measured" else ""),
                     "algorithmic_bytes_per_launch": algo,
                     "avg_launch_us": layer_s * 1e6,
                     "kernel": ("one layer's forward: prep_kv_kernel + fwd_tc_kernel" if r["halves"]
                                else "one layer's forward: fwd_kernel"),
                     "traffic_note": "steady-state DRAM bytes of one layer's kernels inside the stack (ncu, "
                                     "caches not flushed between kernels)",
                     "attention_kernel": {
                         "avg_launch_us": launch_s * 1e6, "achieved": algo / launch_s / 1e9,
                         "frac": algo / launch_s / 1e9 / peak,
                         "traffic": traffic["attend"] if traffic else None,
                         "note": "fwd_tc_kernel timed alone; its bytes counted as the layer's compulsory ones "
                                 "(it reads the prepared K'/V' where the layer reads K and V)"}},
        "layer": {"us_per_layer": layer_s * 1e6,
                  "prepare_us_per_launch": r["halves"]["prepare_ms"] * 1e3 if r["halves"] else None,
                  "attend_us_per_launch": r["halves"]["attend_ms"] * 1e3 if r["halves"] else None,
                  "achieved_gbs": algo / layer_s / 1e9, "frac": algo / layer_s / 1e9 / peak,
                  "note": "compulsory bytes of a layer over its whole forward (both kernels)"},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": r["h2d"],
                "d2h_bytes_per_step": r["d2h"], "steps": r["e2e_steps"], "gpu_launches": r["e2e_launches"]},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
    }
    if not args.no_secondary and args.workload == DEFAULT:
        sec = {}
        for name in SECONDARY:
            ws = WORKLOADS[name]
            rs = time_device(ws, args.steps, args.warmup, device, rank, world)
            ls = rs["ms_per_step"] / 1e3 / ws["L"]
            la = rs["halves"]["attend_ms"] / 1e3 if rs["halves"] else ls
            ach = compulsory_bytes(ws) / la / 1e9
            sec[name] = {"value": ws["B"] * ws["N"] * world / (rs["ms_per_step"] / 1e3), "unit": UNIT,
                         "path": ws["mode"] + " forward", "layers": ws["L"],
                         "ms_per_step": rs["ms_per_step"], "us_per_layer": ls * 1e6,
                         "attend_us_per_launch": la * 1e6,
                         "prepare_us_per_launch": rs["halves"]["prepare_ms"] * 1e3 if rs["halves"] else None,
                         "achieved_gbs": compulsory_bytes(ws) / ls / 1e9,
                         "frac": compulsory_bytes(ws) / ls / 1e9 / peak,
                         "attend_achieved_gbs": ach, "attend_frac": ach / peak,
                         "layer_frac": compulsory_bytes(ws) / ls / 1e9 / peak, "traffic": ncu_traffic(name)}
        line["secondary"] = sec
        # the interpolated path's cost over the mask path on the same shapes (the pages quote
        # ~5x for their own implementation, hardware unstated)
        line["interp_over_mask"] = {
            "n1024_layer": sec["learned-interp-n1024"]["us_per_layer"] / (r["ms_per_step"] * 1e3 / WORKLOADS[DEFAULT]["L"]),
            "n131072_layer": sec["long-interp-n131072"]["us_per_layer"] / sec["long-mask-n131072"]["us_per_layer"],
            "note": "N=1024: learned-interp-n1024 (W=10) over linear-stack-n1024 (W=12); N=131072: same shape and W",
            "pages_quote": "~5x (hardware unstated)"}
        wb = WORKLOADS[BACKWARD]
        rb = time_backward(wb, args.steps, args.warmup, device)
        rb_alone = time_backward(wb, args.steps, args.warmup, device, prepared=False)
        rt = time_backward(wb, args.steps, args.warmup, device, with_forward=True)
        bb = compulsory_bytes_bwd(wb)
        dec = {m: time_decode(m, 1, 8, 4096, 16, args.steps, args.warmup, device) for m in ("mask", "interp")}
        line["decode"] = {"shape": "B=1, H=8, 16 layers, cache N=4096, new token at 4095, W=12, alpha=1.5",
                          "mask_us_per_token": dec["mask"], "interp_us_per_token": dec["interp"],
                          "interp_over_mask": dec["interp"] / dec["mask"]}
        line["backward"] = {"workload": BACKWARD,
                            "path": "interp backward (dQ, dK, dV, dalpha) from the forward's prepared K'/V' rows "
                                    "(fib_attn_bwd_prepared)",
                            "standalone": {"path": "fib_attn_bwd: K'/V' prepared from k and v in the backward",
                                           "ms_per_step": rb_alone["ms_per_step"],
                                           "us_per_layer": rb_alone["us_per_layer"],
                                           "frac": compulsory_bytes_bwd(wb) / (rb_alone["us_per_layer"] * 1e-6) / 1e9 / peak},
                            "value": wb["B"] * wb["N"] * world / (rb["ms_per_step"] / 1e3), "unit": UNIT,
                            "ms_per_step": rb["ms_per_step"], "us_per_layer": rb["us_per_layer"],
                            "compulsory_bytes_per_layer": bb,
                            "achieved_gbs": bb / (rb["us_per_layer"] * 1e-6) / 1e9,
                            "frac": bb / (rb["us_per_layer"] * 1e-6) / 1e9 / peak,
                            "traffic": ncu_traffic_bwd(BACKWARD)}
        tb = compulsory_bytes(wb) + bb
        line["train_step"] = {"workload": BACKWARD,
                              "path": "forward of the stack, then its backward from the kept K'/V' (one graph)",
                              "value": wb["B"] * wb["N"] * world / (rt["ms_per_step"] / 1e3), "unit": UNIT,
                              "ms_per_step": rt["ms_per_step"], "us_per_layer": rt["us_per_layer"],
                              "compulsory_bytes_per_layer": tb,
                              "achieved_gbs": tb / (rt["us_per_layer"] * 1e-6) / 1e9,
                              "frac": tb / (rt["us_per_layer"] * 1e-6) / 1e9 / peak}
    dense = {}
    for name in [args.workload] + (SECONDARY if args.workload == DEFAULT and not args.no_secondary else []):
        ws = WORKLOADS[name]
        if ws["mode"] != "mask":
            continue
        sparse_ms = (r["ms_per_step"] if name == args.workload else line["secondary"][name]["ms_per_step"]) / ws["L"]
        ours = time_dense_ours(ws, device)
        dense[name] = {"ms_per_layer": ours, "sparse_ms_per_layer": sparse_ms, "dense_over_sparse": ours / sparse_ms}
        try:  # a library kernel on the same shape, context only (it applies no RoPE)
            dense[name]["torch_sdpa_ms_per_layer_no_rope"] = time_dense_sdpa(ws, device)
        except Exception as exc:
            dense[name]["torch_sdpa_ms_per_layer_no_rope"] = f"unavailable: {str(exc)[:120]}"
    line["dense_causal"] = {"kind": "fib_attn_dense_fwd: dense causal attention with the same RoPE, "
                                    "K'/V' preparation + the library's dense kernel, one layer",
                            "layers": dense}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        per_layer, desc, _ = time_oracle(w, 3)
        line["cpu_baseline"] = {"value": oracle_tokens_per_s(w, per_layer), "unit": UNIT, "cores": 1,
                                "kind": "oracle", "sample": desc + ", scaled to the full stack",
                                "host_cores_available": len(os.sched_getaffinity(0))}
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


if __name__ == "__main__":
    main()
