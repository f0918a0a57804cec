"""Benchmark of the tensor-parallel FFN hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one pass of the whole path over one batch of the Llama-3-8B-shaped
SwiGLU workload (8192 tokens, d = 4096, d_ff = 14336, T_p = 8, bf16): packing
of W1/W3 (shard_columns) and W2 (shard_rows), forward with the g-operator
shard-sum, backward with the f-operator dx shard-sum and all weight
gradients.  `value` is the algorithmic fwd+bwd FLOP rate (6+12 N d d_ff per
step) with inputs resident in HBM; `e2e` repeats the step through the same
API with x and dy copied in from pinned host memory and y and dx copied back
inside the timed region.  The decode-shaped workload (Llama-3-70B SwiGLU,
32 tokens) is reported in `decode` as HBM GB/s of its compulsory bytes.

--impl reference times the float64 CPU oracle on the host cores on a bounded
sample of the same workload (the oracle is the reference of this build).
Under torchrun (N > 1) every rank runs its own replica on its own GPU (the
shards are virtual ranks inside one GPU, so ranks share no data) and the
line reports the whole-job rate over the slowest rank.
"""
from __future__ import annotations

import argparse
import json
import os
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "TP-FFN fwd+bwd TFLOP/s & % BF16 tensor peak; decode-path HBM GB/s"
MAIN = "llama3_8b_swiglu_bf16"
DECODE = "llama3_70b_decode_swiglu_bf16"

# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) come
# from a committed ncu summary whose JSON block records them together with a
# hash of the kernel sources they were captured from; when the sources have
# changed since, the roofline's traffic is null (stale counters are not
# reported).
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic_per_launch.md")
CSRC = os.path.join(ROOT, "megatron_tensor_transformer_w1_gb300", "csrc")


def kernel_source_sha16():
    """sha256 (first 16 hex digits) over every kernel source file, in name order."""
    import hashlib
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)):
        path = os.path.join(CSRC, name)
        if os.path.isfile(path):
            h.update(name.encode())
            h.update(open(path, "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(workload):
    """{kernel name: DRAM bytes per launch} of `workload` from the committed
    capture, or ({}, reason) when there is none for the current sources."""
    if not os.path.exists(TRAFFIC_FILE):
        return {}, "no committed capture"
    text = open(TRAFFIC_FILE).read()
    try:
        block = text.split("```json", 1)[1].split("```", 1)[0]
        d = json.loads(block)
    except (IndexError, ValueError):
        return {}, "capture summary unreadable"
    if d.get("source_sha16") != kernel_source_sha16():
        return {}, "kernels changed since the capture"
    return d.get("per_launch_bytes", {}).get(workload, {}), "ncu capture " + d.get("source_sha16", "")


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d.get("hbm_gbs", 6800.0), bf16=d.get("bf16_tflops", 1900.0),
                    bf16_sus=d.get("bf16_tflops_sustained", 1700.0), source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        exe = shutil.which("nvidia-smi")
        if exe:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen([exe, f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "100"], stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return None
        sms, maxes, reasons = [], [], set()
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sms.append(float(f[1]))
                maxes.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        os.unlink(self.path)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes), "samples": len(sms),
                "reasons": sorted(reasons)}


def _smi_id(dev):
    """nvidia-smi's id of a CUDA device: its UUID when PyTorch exposes it (the
    CUDA ordinal differs from nvidia-smi's index under CUDA_VISIBLE_DEVICES)."""
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [v for v in vis.split(",") if v.strip()]
        return ids[dev.index] if dev.index < len(ids) else str(dev.index)


# ------------------------------------------------------------- distributed
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        rank = int(os.environ["RANK"])
        local = int(os.environ.get("LOCAL_RANK", rank))
        return dict(world=world, rank=rank, local=local, dist=dist)
    return dict(world=1, rank=0, local=0, dist=None)


def dist_max(ctx, value):
    """Max over ranks (identity on one rank)."""
    if ctx["dist"] is None:
        return value
    import torch
    dev = torch.device("cuda", ctx["local"]) if torch.cuda.is_available() else torch.device("cpu")
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    ctx["dist"].all_reduce(t, op=ctx["dist"].ReduceOp.MAX)
    return float(t.item())


def dist_barrier(ctx):
    if ctx["dist"] is not None:
        ctx["dist"].barrier()


# --------------------------------------------------------------- our arm
def _device_inputs(w, dev, seed):
    """Seeded synthetic tensors generated on the device (same shapes and
    distributions as synth.make_inputs; the parity tests use the host ones)."""
    import torch
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16

    def draw(shape, std):
        t = torch.randn(*shape, generator=gen, device=dev, dtype=torch.float32)
        return (t * std).to(dt)

    s1 = w.w_std if w.w_std is not None else w.d ** -0.5
    s2 = w.w_std if w.w_std is not None else w.d_ff ** -0.5
    out = {"x": draw((w.N, w.d_in), 1.0)}
    out["W1"] = draw((w.d_ff, w.d), s1) if w.act != "none" else None
    out["W3"] = draw((w.d_ff, w.d), s1) if w.act == "swiglu" else None
    out["W2"] = draw((w.d, w.d_ff), s2)
    out["b1"] = draw((w.d_ff,), w.b_std) if w.bias else None
    out["b2"] = draw((w.d,), w.b_std) if w.bias else None
    out["dy"] = None if w.fwd_only else draw((w.N, w.d), 1.0)
    return out


def _kernel_work(w, name):
    """Algorithmic work of one launch: ('flop', F) or ('byte', B)."""
    N, d, dff, T = w.N, w.d, w.d_ff, w.T_p
    wide = 2 * dff if w.act == "swiglu" else dff
    flops = {"up_swiglu": 2 * N * d * 2 * dff, "up_gelu": 2 * N * d * dff, "down_fused_sum": 2 * N * dff * d,
             "down_partials": 2 * N * dff * d, "dgrad_h_swiglu": 2 * N * d * dff, "dgrad_h_gelu": 2 * N * d * dff,
             "dgrad_x_fused_sum": 2 * N * wide * d, "dgrad_x_partials": 2 * N * wide * d,
             "wgrad_w2": 2 * N * d * dff, "wgrad_w13": 2 * N * wide * d, "wgrad_w1": 2 * N * wide * d}
    if name in flops:
        return "flop", flops[name]
    if name.startswith("shard_sum"):
        return "byte", T * N * d * 4 + N * d * 2
    return "byte", 0


def run_ours(args, ctx):
    import torch
    from synth import WORKLOADS
    from megatron_tensor_transformer_w1_gb300 import tpffn as abi
    from megatron_tensor_transformer_w1_gb300.ffn import TensorParallelFFN

    dev = torch.device("cuda", ctx["local"])
    torch.cuda.set_device(dev)
    peaks = _peaks()
    w = WORKLOADS[MAIN]
    if args.tokens:
        w = w.replace(N=args.tokens)  # smaller token batch for profiler captures only
    inp = _device_inputs(w, dev, 20260000 + w.seed_index + 1000 * ctx["rank"])
    ffn = TensorParallelFFN(w.d, w.d_ff, w.T_p, w.act, "bf16", device=dev)
    fused = args.sum == "fused"
    flags = abi.TP_SUM_FUSED if fused else 0
    st = torch.cuda.current_stream(dev)
    plan = ffn.plan
    n = w.N
    w13p = torch.empty(abi.tp_ffn_packed_bytes(plan, abi.TP_PACK_COLUMNS), dtype=torch.uint8, device=dev)
    w2p = torch.empty(abi.tp_ffn_packed_bytes(plan, abi.TP_PACK_ROWS), dtype=torch.uint8, device=dev)
    saved = torch.empty(abi.tp_ffn_saved_bytes(plan, n), dtype=torch.uint8, device=dev)
    ws = torch.empty(abi.tp_ffn_workspace_bytes(plan, n, flags), dtype=torch.uint8, device=dev)
    y = torch.empty(n, w.d, dtype=torch.bfloat16, device=dev)
    dx = torch.empty_like(y)
    dw13p, dw2p = torch.empty_like(w13p), torch.empty_like(w2p)
    x, dy = inp["x"], inp["dy"]
    launches = [0]

    def step(f=flags, x=x, dy=dy, y=y, dx=dx):
        abi.check(abi.tp_ffn_shard_columns(plan, inp["W1"], inp["W3"], w13p, st), "shard_columns")
        abi.check(abi.tp_ffn_shard_rows(plan, inp["W2"], w2p, st), "shard_rows")
        abi.check(abi.tp_ffn_fwd(plan, n, x, w13p, w2p, None, None, y, None, saved, ws, ws.numel(), f, st), "fwd")
        c = 2 + abi.tp_ffn_last_launch_count(plan)
        abi.check(abi.tp_ffn_bwd(plan, n, x, w13p, w2p, saved, dy, dx, None, dw13p, dw2p, None, None, ws,
                                 ws.numel(), f, st), "bwd")
        launches[0] += c + abi.tp_ffn_last_launch_count(plan)

    flop_step = w.fwd_flops() + w.bwd_flops()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    abi.tp_ffn_kernel_times(plan, 0)  # clear
    launches[0] = 0
    dist_barrier(ctx)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(_smi_id(dev)) as clk:
        e0.record(st)
        for _ in range(args.steps):
            step(flags | abi.TP_FLAG_TIMING)
        e1.record(st)
        torch.cuda.synchronize(dev)
    dist_barrier(ctx)
    ms = e0.elapsed_time(e1) / args.steps
    ms = dist_max(ctx, ms)
    gpu_launches = launches[0]
    recs = abi.tp_ffn_kernel_times(plan, 100000)

    # dominant kernel and its roofline, from the per-launch events above
    per = {}
    for name, t in recs:
        per.setdefault(name, []).append(t)
    dom = max(per, key=lambda k: sum(per[k]))
    kind, work = _kernel_work(w, dom)
    avg_ms = sum(per[dom]) / len(per[dom])
    traffic, traffic_src = ncu_traffic(MAIN if w.N == WORKLOADS[MAIN].N else f"{MAIN}@{w.N}")
    if kind == "flop":
        # a kernel of about a millisecond, timed inside a 5 ms step: the burst
        # peak is the denominator; the fraction of the sustained peak (a
        # seconds-long GEMM loop under the power cap) is given beside it
        ach = work / (avg_ms * 1e-3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": round(ach, 1), "peak": peaks["bf16"],
                "unit": "TFLOP/s", "frac": round(ach / peaks["bf16"], 4),
                "peak_kind": f"bf16 burst ({peaks['source']})",
                "frac_of_sustained": round(ach / peaks["bf16_sus"], 4), "traffic": traffic.get(dom),
                "traffic_source": traffic_src, "work_per_launch": work, "launch_ms": round(avg_ms, 4)}
    else:
        ach = work / (avg_ms * 1e-3) / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm"], "unit": "GB/s",
                "frac": round(ach / peaks["hbm"], 4), "peak_kind": f"HBM copy ({peaks['source']})",
                "traffic": traffic.get(dom), "traffic_source": traffic_src, "work_per_launch": work,
                "launch_ms": round(avg_ms, 4)}
    kernels = {k: {"launches": len(v), "avg_ms": round(sum(v) / len(v), 4), "share": None} for k, v in per.items()}
    tot = sum(sum(v) for v in per.values())
    for k, v in per.items():
        kernels[k]["share"] = round(sum(v) / tot, 4)
        kind_k, work_k = _kernel_work(w, k)
        if work_k:
            rate = work_k / (kernels[k]["avg_ms"] * 1e-3)
            kernels[k]["rate"] = round(rate / (1e12 if kind_k == "flop" else 1e9), 1)
            kernels[k]["rate_unit"] = "TFLOP/s" if kind_k == "flop" else "GB/s"

    # end to end: every step's x, dy come in from pinned host memory and its
    # y, dx go back.  The copies run on a second stream with two sets of
    # device buffers, so step i+1's inputs arrive and step i's results leave
    # while step i / i+1 compute -- as a training loop would overlap them;
    # every copy of every timed step lies inside the timed region.
    hx = x.cpu().pin_memory()
    hdy = dy.cpu().pin_memory()
    hy = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for _ in range(2)]
    hdx = [torch.empty(dx.shape, dtype=dx.dtype).pin_memory() for _ in range(2)]
    xin = [torch.empty_like(x) for _ in range(2)]
    dyin = [torch.empty_like(dy) for _ in range(2)]
    yb, dxb = [y, torch.empty_like(y)], [dx, torch.empty_like(dx)]
    cs = torch.cuda.Stream(dev)

    def e2e_run(k, start=None):
        ev = lambda: torch.cuda.Event()
        in_ready, done, out_free = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        if start is not None:
            cs.wait_event(start)
        with torch.cuda.stream(cs):
            xin[0].copy_(hx, non_blocking=True)
            dyin[0].copy_(hdy, non_blocking=True)
            in_ready[0].record(cs)
        for i in range(k):
            b = i & 1
            st.wait_event(in_ready[b])
            if i >= 2:
                st.wait_event(out_free[b])  # step i-2's results have left these buffers
            step(flags, xin[b], dyin[b], yb[b], dxb[b])
            done[b].record(st)
            with torch.cuda.stream(cs):
                if i + 1 < k:
                    if i >= 1:
                        cs.wait_event(done[1 - b])  # step i-1 has read its inputs
                    xin[1 - b].copy_(hx, non_blocking=True)
                    dyin[1 - b].copy_(hdy, non_blocking=True)
                    in_ready[1 - b].record(cs)
                cs.wait_event(done[b])
                hy[b].copy_(yb[b], non_blocking=True)
                hdx[b].copy_(dxb[b], non_blocking=True)
                out_free[b].record(cs)
        st.wait_stream(cs)

    k_e2e = max(20, args.steps // 2)  # at least ~0.1 s, so that one host hiccup does not dominate
    e2e_run(3)
    torch.cuda.synchronize(dev)
    dist_barrier(ctx)
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(st)
    e2e_run(k_e2e, start=e2)
    e3.record(st)
    torch.cuda.synchronize(dev)
    e2e_ms = dist_max(ctx, e2.elapsed_time(e3) / k_e2e)
    h2d = (x.numel() + dy.numel()) * 2
    d2h = (y.numel() + dx.numel()) * 2

    decode = run_decode(args, ctx, dev, peaks) if not args.no_decode else None
    standalone = run_standalone_sum(dev, 10, peaks) if not args.no_extras else None
    workloads = run_all_workloads(dev, 10) if not args.no_extras else None
    seq_parallel = run_seq_parallel(dev, 10, peaks) if not args.no_extras else None
    attention = run_attention(dev, 10, peaks, args.sum) if not args.no_extras else None

    value = ctx["world"] * flop_step / (ms * 1e-3) / 1e12
    # Key order: the long tables first, the headline blocks (roofline,
    # e2e, decode, cpu_baseline) last, so that a reader of the line's tail
    # sees them.
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": ctx["world"],
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded on-device normals)",
        "config": {"workload": MAIN, "tokens": w.N, "d": w.d, "d_ff": w.d_ff, "T_p": w.T_p, "act": w.act,
                   "shard_sum": args.sum, "step": "shard_columns+shard_rows+fwd+bwd (incl. weight grads)",
                   "flop_per_step": flop_step, "l2": "no flush: per-step working set ~4.3 GB > 129 MB L2",
                   "parallelism": f"{w.T_p} virtual TP ranks per GPU; replicas across GPUs"},
        "attention_sublayer": attention,
        "sequence_parallel": seq_parallel,
        "workloads": workloads,
        "standalone_shard_sum": standalone,
        "kernels": kernels,
        "gpu_launches": gpu_launches,
        "clocks": clk.summary(),
        "e2e": {"value": round(ctx["world"] * flop_step / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": "pinned host buffers; a second stream, two device buffer sets (overlapped with compute)"},
        "frac_of_bf16_peak": {"burst": round(value / ctx['world'] / peaks["bf16"], 4),
                              "sustained": round(value / ctx['world'] / peaks["bf16_sus"], 4),
                              "peaks": peaks["source"]},
        "roofline": roof,
        "decode": decode,
    }
    if ctx["rank"] == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget)
    return line


def time_workload(w, dev, steps, fused, seed=0, overlap=False, graphs=True):
    """fwd and bwd of one workload through the C ABI: ms per call (CUDA
    events on the calling stream, around a plain loop of calls), the average
    per-kernel times (a second loop with an event pair around every launch),
    and ms per replay of the call captured in a CUDA graph."""
    import torch
    from megatron_tensor_transformer_w1_gb300 import tpffn as abi
    from megatron_tensor_transformer_w1_gb300.ffn import TensorParallelFFN
    inp = _device_inputs(w, dev, 20260000 + w.seed_index + seed)
    if w.act == "none":
        ffn = TensorParallelFFN(w.d, w.d_ff, w.T_p, "none", w.dtype, device=dev, n_heads=w.n_heads,
                                n_kv_heads=w.n_kv_heads, head_dim=w.head_dim)
    else:
        ffn = TensorParallelFFN(w.d, w.d_ff, w.T_p, w.act, w.dtype, device=dev)
    st = torch.cuda.current_stream(dev)
    w13p, w2p = ffn.pack(inp["W1"], inp["W2"], inp["W3"])
    res = {}

    def timed(fn):
        """ms per call from a plain loop (no per-launch events), the
        per-kernel times from a second loop with them, and ms per replay of
        the call captured once in a CUDA graph (no host launch cost)."""
        for _ in range(3):
            fn(0)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(steps):
            fn(0)
        e1.record(st)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / steps
        abi.tp_ffn_kernel_times(ffn.plan, 0)
        for _ in range(steps):
            fn(abi.TP_FLAG_TIMING)
        torch.cuda.synchronize(dev)
        per = {}
        for name, t in abi.tp_ffn_kernel_times(ffn.plan, 100000):
            per.setdefault(name, []).append(t)
        graph_ms = None
        if graphs:
            try:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    fn(0)
                g.replay()
                torch.cuda.synchronize(dev)
                e0.record(st)
                for _ in range(steps):
                    g.replay()
                e1.record(st)
                torch.cuda.synchronize(dev)
                graph_ms = round(e0.elapsed_time(e1) / steps, 4)
                del g
            except Exception as exc:  # report, do not fail the bench line
                graph_ms = f"capture failed: {type(exc).__name__}: {exc}"[:160]
        return ms, {k: round(sum(v) / len(v), 4) for k, v in per.items()}, graph_ms

    out = {}
    f = (abi.TP_SUM_FUSED if fused else 0) | (abi.TP_SUM_OVERLAP if overlap else 0)
    saved = None if w.fwd_only or w.act == "none" else torch.empty(
        abi.tp_ffn_saved_bytes(ffn.plan, w.N), dtype=torch.uint8, device=dev)
    ws = ffn.workspace(w.N, f)
    y = torch.empty(w.N, w.d, dtype=ffn.torch_dtype, device=dev)

    def fwd(extra):
        abi.check(abi.tp_ffn_fwd(ffn.plan, w.N, inp["x"], w13p, w2p, inp["b1"], inp["b2"], y, None, saved, ws,
                                 ws.numel(), f | extra, torch.cuda.current_stream(dev)), "fwd")

    out["fwd_ms"], out["fwd_kernels"], out["fwd_graph_ms"] = timed(fwd)
    out["fwd_tflops"] = round(w.fwd_flops() / (out["fwd_ms"] * 1e-3) / 1e12, 3)
    if isinstance(out["fwd_graph_ms"], float):
        out["fwd_graph_tflops"] = round(w.fwd_flops() / (out["fwd_graph_ms"] * 1e-3) / 1e12, 3)
    if not w.fwd_only:
        dx = torch.empty(w.N, w.d_in, dtype=ffn.torch_dtype, device=dev)
        dw13p = None if w13p is None else torch.empty_like(w13p)
        dw2p = torch.empty_like(w2p)
        db1 = torch.empty(w.d_ff, dtype=ffn.torch_dtype, device=dev) if w.bias and w.act == "gelu_tanh" else None
        db2 = torch.empty(w.d, dtype=ffn.torch_dtype, device=dev) if w.bias else None

        def bwd(extra):
            abi.check(abi.tp_ffn_bwd(ffn.plan, w.N, inp["x"], w13p, w2p, saved, inp["dy"], dx, None, dw13p, dw2p,
                                     db1, db2, ws, ws.numel(), f | extra, torch.cuda.current_stream(dev)), "bwd")

        out["bwd_ms"], out["bwd_kernels"], out["bwd_graph_ms"] = timed(bwd)
        out["bwd_tflops"] = round(w.bwd_flops() / (out["bwd_ms"] * 1e-3) / 1e12, 3)
        if isinstance(out["bwd_graph_ms"], float):
            out["bwd_graph_tflops"] = round(w.bwd_flops() / (out["bwd_graph_ms"] * 1e-3) / 1e12, 3)
    out["fwd_ms"] = round(out["fwd_ms"], 4)
    if "bwd_ms" in out:
        out["bwd_ms"] = round(out["bwd_ms"], 4)
    return out


def run_all_workloads(dev, steps):
    """fwd and bwd throughput of every workload (fused shard-sum), plus the
    standalone shard-sum kernel of the Llama-3-8B workload in HBM GB/s."""
    from synth import WORKLOADS
    table = {}
    for name, w in WORKLOADS.items():
        table[name] = time_workload(w, dev, steps, fused=not w.fwd_only)
        if w.fwd_only:
            nbytes = w.weight_bytes() + 2 * w.N * w.d * 2
            table[name]["fwd_hbm_gbs"] = round(nbytes / (table[name]["fwd_ms"] * 1e-3) / 1e9, 1)
    return table


def run_standalone_sum(dev, steps, peaks):
    """The standalone shard-sum kernel in HBM GB/s, and how much of it the
    overlapped variant (TP_SUM_OVERLAP) hides behind the row-sharded GEMM."""
    from synth import WORKLOADS
    w = WORKLOADS[MAIN]
    r = time_workload(w, dev, steps, fused=False, graphs=False)
    o = time_workload(w, dev, steps, fused=False, overlap=True, graphs=False)
    nbytes = w.T_p * w.N * w.d * 4 + w.N * w.d * 2  # fp32 partials read + bf16 result written
    out = {"workload": MAIN, "fwd_ms": r["fwd_ms"], "bwd_ms": r["bwd_ms"],
           "step_tflops_fwd_bwd": round((w.fwd_flops() + w.bwd_flops()) / ((r["fwd_ms"] + r["bwd_ms"]) * 1e-3) / 1e12, 2),
           "overlap": {"fwd_ms": o["fwd_ms"], "bwd_ms": o["bwd_ms"],
                       "step_tflops_fwd_bwd": round((w.fwd_flops() + w.bwd_flops()) /
                                                    ((o["fwd_ms"] + o["bwd_ms"]) * 1e-3) / 1e12, 2)}}
    sums = sum(ms for k, ms in list(r["fwd_kernels"].items()) + list(r["bwd_kernels"].items())
               if k.startswith("shard_sum"))
    if sums > 0:
        out["overlap"]["hidden_fraction_of_shard_sum"] = round(
            ((r["fwd_ms"] + r["bwd_ms"]) - (o["fwd_ms"] + o["bwd_ms"])) / sums, 3)
    for k, ms in list(r["fwd_kernels"].items()) + list(r["bwd_kernels"].items()):
        if k.startswith("shard_sum"):
            gbs = nbytes / (ms * 1e-3) / 1e9
            out[k] = {"ms": ms, "bytes": nbytes, "achieved_gbs": round(gbs, 1), "peak_gbs": peaks["hbm"],
                      "frac": round(gbs / peaks["hbm"], 4)}
    return out


def run_seq_parallel(dev, steps, peaks):
    """Sequence-parallel forms of the Llama-3-8B workload: fwd and bwd ms with
    per-rank token slices (all-gather + reduce-scatter), and the GB/s of the
    gather and reduce-scatter kernels."""
    import torch
    from synth import WORKLOADS
    from megatron_tensor_transformer_w1_gb300 import tpffn as abi
    from megatron_tensor_transformer_w1_gb300.ffn import TensorParallelFFN
    w = WORKLOADS[MAIN]
    inp = _device_inputs(w, dev, 20260000 + w.seed_index + 7)
    ffn = TensorParallelFFN(w.d, w.d_ff, w.T_p, w.act, "bf16", device=dev)
    st = torch.cuda.current_stream(dev)
    w13p, w2p = ffn.pack(inp["W1"], inp["W2"], inp["W3"])
    T, ns = w.T_p, w.N // w.T_p
    xs = [inp["x"][t * ns:(t + 1) * ns].clone() for t in range(T)]
    dys = [inp["dy"][t * ns:(t + 1) * ns].clone() for t in range(T)]
    ys = [torch.empty(ns, w.d, dtype=torch.bfloat16, device=dev) for _ in range(T)]
    dxs = [torch.empty(ns, w.d, dtype=torch.bfloat16, device=dev) for _ in range(T)]
    saved = torch.empty(abi.tp_ffn_saved_bytes(ffn.plan, w.N), dtype=torch.uint8, device=dev)
    dw13p, dw2p = torch.empty_like(w13p), torch.empty_like(w2p)
    out = {"workload": MAIN}
    for mode, flags in (("reduce_scatter", 0), ("fused_then_scatter", abi.TP_SUM_FUSED)):
        ws = torch.empty(abi.tp_ffn_seq_parallel_workspace_bytes(ffn.plan, w.N, flags), dtype=torch.uint8,
                         device=dev)

        def fwd(extra):
            abi.check(abi.tp_ffn_fwd_seq_parallel(ffn.plan, w.N, xs, w13p, w2p, None, None, ys, saved, ws,
                                                  ws.numel(), flags | extra, st), "fwd_sp")

        def bwd(extra):
            abi.check(abi.tp_ffn_bwd_seq_parallel(ffn.plan, w.N, xs, w13p, w2p, saved, dys, dxs, dw13p, dw2p, None,
                                                  None, ws, ws.numel(), flags | extra, st), "bwd_sp")

        res = {}
        for name, fn in (("fwd", fwd), ("bwd", bwd)):
            for _ in range(3):
                fn(0)
            torch.cuda.synchronize(dev)
            abi.tp_ffn_kernel_times(ffn.plan, 0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            for _ in range(steps):
                fn(abi.TP_FLAG_TIMING)
            e1.record(st)
            torch.cuda.synchronize(dev)
            res[name + "_ms"] = round(e0.elapsed_time(e1) / steps, 4)
            per = {}
            for k, t in abi.tp_ffn_kernel_times(ffn.plan, 100000):
                per.setdefault(k, []).append(t)
            for k, v in per.items():
                ms = sum(v) / len(v)
                if k.startswith("all_gather"):
                    nbytes = 2 * w.N * w.d * 2  # read slices + write the gathered tensor
                elif k.startswith("reduce_scatter"):
                    nbytes = w.T_p * w.N * w.d * 4 + w.N * w.d * 2
                elif k.startswith("scatter"):
                    nbytes = 2 * w.N * w.d * 2
                else:
                    continue
                res[k] = {"ms": round(ms, 4), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
                          "frac_of_hbm": round(nbytes / (ms * 1e-3) / 1e9 / peaks["hbm"], 4)}
        res["step_tflops_fwd_bwd"] = round((w.fwd_flops() + w.bwd_flops()) /
                                           ((res["fwd_ms"] + res["bwd_ms"]) * 1e-3) / 1e12, 2)
        out[mode] = res
    return out


def _attn_kernel_work(w, name):
    """FLOPs one launch of the attention sublayer executes (visible score
    entries only for the attention kernels: the dq kernel recomputes S and dP
    and forms dQ -- 3 products; the dk/dv kernel recomputes S^T and dP^T and
    forms dV and dK -- 4 products; the forward forms S and PV -- 2)."""
    n, d, nq, nk = w.N, w.d, w.H * w.hd, w.Hkv * w.hd
    half = w.core_flops() // 2  # one product over the visible pairs
    table = {"qkv_proj": 2 * n * d * (nq + 2 * nk), "attn_fwd": 2 * half, "down_fused_sum": 2 * n * nq * d,
             "down_partials": 2 * n * nq * d, "dgrad_heads": 2 * n * d * nq, "wgrad_rows": 2 * n * d * nq,
             "attn_bwd_dq": 3 * half, "attn_bwd_dkdv": 4 * half,
             "attn_dgrad_x_fused_sum": 2 * n * (nq + 2 * nk) * d, "attn_dgrad_x_partials": 2 * n * (nq + 2 * nk) * d,
             "attn_wgrad_qkv": 2 * n * (nq + 2 * nk) * d}
    return table.get(name)


def run_attention(dev, steps, peaks, sum_mode="fused"):
    """The whole head-sharded attention sublayer (fwd + bwd incl. weight
    gradients) on its two workloads: ms, TFLOP/s (FlashAttention counting:
    backward core = 2.5x forward core) and per-kernel times and rates."""
    import torch
    from synth import ATTN_WORKLOADS
    from megatron_tensor_transformer_w1_gb300 import tpffn as abi
    from megatron_tensor_transformer_w1_gb300.attention import TensorParallelAttention
    out = {}
    for name, w in ATTN_WORKLOADS.items():
        gen = torch.Generator(device=dev)
        gen.manual_seed(20260000 + w.seed_index)

        def draw(shape, std):
            return (torch.randn(*shape, generator=gen, device=dev) * std).to(torch.bfloat16)

        nq, nk = w.H * w.hd, w.Hkv * w.hd
        x, dy = draw((w.N, w.d), 1.0), draw((w.N, w.d), 1.0)
        attn = TensorParallelAttention(w.d, w.H, w.Hkv, w.hd, w.T_p, causal=w.causal, device=dev)
        wqkv, wo = attn.pack(draw((nq, w.d), w.d ** -0.5), draw((nk, w.d), w.d ** -0.5),
                             draw((nk, w.d), w.d ** -0.5), draw((w.d, nq), nq ** -0.5))
        st = torch.cuda.current_stream(dev)
        flags = abi.TP_SUM_FUSED if sum_mode == "fused" else 0
        y = torch.empty(w.N, w.d, dtype=torch.bfloat16, device=dev)
        dx = torch.empty_like(y)
        saved = torch.empty(abi.tp_attn_saved_bytes(attn.plan, w.B, w.S), dtype=torch.uint8, device=dev)
        dwqkv, dwo = torch.empty_like(wqkv), torch.empty_like(wo)
        ws = attn.workspace(w.B, w.S, flags)

        def fwd(extra=0):
            abi.check(abi.tp_attn_fwd(attn.plan, w.B, w.S, x, wqkv, wo, y, saved, ws, ws.numel(), flags | extra, st),
                      "attn_fwd")

        def bwd(extra=0):
            abi.check(abi.tp_attn_bwd(attn.plan, w.B, w.S, x, wqkv, wo, saved, dy, dx, dwqkv, dwo, ws, ws.numel(),
                                      flags | extra, st), "attn_bwd")

        res = {"B": w.B, "S": w.S, "d": w.d, "heads": w.H, "kv_heads": w.Hkv, "head_dim": w.hd, "T_p": w.T_p,
               "causal": w.causal, "shard_sum": sum_mode}
        for ph, fn in (("fwd", fwd), ("bwd", bwd)):
            for _ in range(3):
                fwd()
                fn()
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            for _ in range(steps):
                fn()
            e1.record(st)
            torch.cuda.synchronize(dev)
            res[ph + "_ms"] = round(e0.elapsed_time(e1) / steps, 4)
        flop = w.fwd_flops() + w.bwd_flops()
        res["flop_per_step"] = flop
        res["step_tflops_fwd_bwd"] = round(flop / ((res["fwd_ms"] + res["bwd_ms"]) * 1e-3) / 1e12, 2)
        res["frac_of_bf16_peak"] = round(res["step_tflops_fwd_bwd"] / peaks["bf16"], 4)
        # per-kernel breakdown (events around every launch)
        abi.tp_attn_kernel_times(attn.plan, 0)
        for _ in range(steps):
            fwd(abi.TP_FLAG_TIMING)
            bwd(abi.TP_FLAG_TIMING)
        per = {}
        for k, t in abi.tp_attn_kernel_times(attn.plan, 100000):
            per.setdefault(k, []).append(t)
        kern = {}
        for k, v in per.items():
            ms = sum(v) / len(v)
            e = {"ms": round(ms, 4)}
            f = _attn_kernel_work(w, k)
            if f:
                e["tflops"] = round(f / (ms * 1e-3) / 1e12, 1)
                e["frac_of_bf16_peak"] = round(f / (ms * 1e-3) / 1e12 / peaks["bf16"], 4)
            kern[k] = e
        res["kernels"] = kern
        out[name] = res
        del attn
    return out


def profile_attention(args):
    """A plain loop of attention-sublayer steps for profiler captures: no
    timing, no extras; --attn-batch shrinks the sequence count."""
    import torch
    from synth import ATTN_WORKLOADS
    from megatron_tensor_transformer_w1_gb300.attention import TensorParallelAttention
    w = ATTN_WORKLOADS[args.profile_attention]
    if args.attn_batch:
        w = w.replace(B=args.attn_batch)
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(20260000 + w.seed_index)

    def draw(shape, std):
        return (torch.randn(*shape, generator=gen, device=dev) * std).to(torch.bfloat16)

    nq, nk = w.H * w.hd, w.Hkv * w.hd
    attn = TensorParallelAttention(w.d, w.H, w.Hkv, w.hd, w.T_p, causal=w.causal, device=dev)
    wqkv, wo = attn.pack(draw((nq, w.d), w.d ** -0.5), draw((nk, w.d), w.d ** -0.5), draw((nk, w.d), w.d ** -0.5),
                         draw((w.d, nq), nq ** -0.5))
    x, dy = draw((w.N, w.d), 1.0), draw((w.N, w.d), 1.0)
    for _ in range(args.warmup + args.steps):
        y, saved = attn.forward(x, w.B, w.S, wqkv, wo, fused=args.sum == "fused")
        attn.backward(x, w.B, w.S, wqkv, wo, saved, dy, fused=args.sum == "fused")
    torch.cuda.synchronize(dev)
    return {"profile_attention": w.name, "B": w.B, "S": w.S, "steps": args.steps, "warmup": args.warmup}


def profile_ffn(args):
    """A plain loop of FFN steps for profiler captures: the Llama-3-8B shapes
    (--profile-workload picks another workload's, with its biases; --tokens
    overrides the token count), pack + forward + backward with the --sum mode,
    or with --profile-decode the decode-shaped forward alone; no timing, no
    extras, nothing else launched."""
    import torch
    from synth import WORKLOADS
    from megatron_tensor_transformer_w1_gb300 import tpffn as abi
    from megatron_tensor_transformer_w1_gb300.ffn import TensorParallelFFN
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = WORKLOADS[DECODE if args.profile_decode else (args.profile_workload or MAIN)]
    if args.tokens and not args.profile_decode:
        w = w.replace(N=args.tokens)
    inp = _device_inputs(w, dev, 20260000 + w.seed_index)
    ffn = TensorParallelFFN(w.d, w.d_ff, w.T_p, w.act, "bf16", device=dev)
    st, plan, n = torch.cuda.current_stream(dev), ffn.plan, w.N
    flags = abi.TP_SUM_FUSED if (args.sum == "fused" and not args.profile_decode) else 0
    w13p, w2p = ffn.pack(inp["W1"], inp["W2"], inp["W3"])
    ws = ffn.workspace(n, flags)
    y = torch.empty(n, w.d, dtype=torch.bfloat16, device=dev)
    if args.profile_decode:
        for _ in range(args.warmup + args.steps):
            abi.check(abi.tp_ffn_fwd(plan, n, inp["x"], w13p, w2p, None, None, y, None, None, ws, ws.numel(), 0, st),
                      "decode fwd")
    else:
        saved = torch.empty(abi.tp_ffn_saved_bytes(plan, n), dtype=torch.uint8, device=dev)
        dx = torch.empty_like(y)
        dw13p, dw2p = torch.empty_like(w13p), torch.empty_like(w2p)
        b1, b2 = (inp["b1"], inp["b2"]) if w.bias else (None, None)
        db1 = torch.empty(w.d_ff, dtype=torch.bfloat16, device=dev) if w.bias and w.act == "gelu_tanh" else None
        db2 = torch.empty(w.d, dtype=torch.bfloat16, device=dev) if w.bias else None
        for _ in range(args.warmup + args.steps):
            abi.check(abi.tp_ffn_shard_columns(plan, inp["W1"], inp["W3"], w13p, st), "shard_columns")
            abi.check(abi.tp_ffn_shard_rows(plan, inp["W2"], w2p, st), "shard_rows")
            abi.check(abi.tp_ffn_fwd(plan, n, inp["x"], w13p, w2p, b1, b2, y, None, saved, ws, ws.numel(), flags,
                                     st), "fwd")
            abi.check(abi.tp_ffn_bwd(plan, n, inp["x"], w13p, w2p, saved, inp["dy"], dx, None, dw13p, dw2p, db1,
                                     db2, ws, ws.numel(), flags, st), "bwd")
    torch.cuda.synchronize(dev)
    return {"profile": w.name, "tokens": n, "sum": args.sum, "steps": args.steps, "warmup": args.warmup}


def run_decode(args, ctx, dev, peaks):
    import torch
    from synth import WORKLOADS
    from megatron_tensor_transformer_w1_gb300 import tpffn as abi
    from megatron_tensor_transformer_w1_gb300.ffn import TensorParallelFFN
    w = WORKLOADS[DECODE]
    inp = _device_inputs(w, dev, 20260000 + w.seed_index)
    ffn = TensorParallelFFN(w.d, w.d_ff, w.T_p, w.act, "bf16", device=dev)
    plan, st, n = ffn.plan, torch.cuda.current_stream(dev), w.N
    w13p, w2p = ffn.pack(inp["W1"], inp["W2"], inp["W3"])
    ws = torch.empty(abi.tp_ffn_workspace_bytes(plan, n, 0), dtype=torch.uint8, device=dev)
    y = torch.empty(n, w.d, dtype=torch.bfloat16, device=dev)

    def step(f=0):
        abi.check(abi.tp_ffn_fwd(plan, n, inp["x"], w13p, w2p, None, None, y, None, None, ws, ws.numel(), f, st),
                  "decode fwd")

    for _ in range(5):
        step()
    torch.cuda.synchronize(dev)
    # the whole-step rate from a loop without per-kernel events: at 0.24 ms a
    # step, the six event records of the timing mode add about 5 %
    k = max(20, args.steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(k):
        step()
    e1.record(st)
    torch.cuda.synchronize(dev)
    ms = dist_max(ctx, e0.elapsed_time(e1) / k)
    # per-kernel times (roofline of the dominant kernel) from a second loop
    abi.tp_ffn_kernel_times(plan, 0)
    for _ in range(k):
        step(abi.TP_FLAG_TIMING)
    torch.cuda.synchronize(dev)
    recs = abi.tp_ffn_kernel_times(plan, 100000)
    per = {}
    for name, t in recs:
        per.setdefault(name, []).append(t)
    nbytes = w.weight_bytes() + 2 * w.N * w.d * 2  # weights + x + y
    gbs = ctx["world"] * nbytes / (ms * 1e-3) / 1e9
    dom = max(per, key=lambda q: sum(per[q]))
    dom_ms = sum(per[dom]) / len(per[dom])
    dom_bytes = {"up_swiglu": 2 * w.d_ff * w.d * 2 + w.N * w.d * 2 + w.N * w.d_ff * 2,
                 "down_partials": w.d_ff * w.d * 2 + w.N * w.d_ff * 2 + w.T_p * w.N * w.d * 4}.get(dom, 0)
    dach = dom_bytes / (dom_ms * 1e-3) / 1e9
    dtraffic, dsrc = ncu_traffic(DECODE)
    return {"workload": DECODE, "value": round(gbs, 1), "unit": "GB/s", "ms_per_step": round(ms, 4),
            "timing": "step time from a loop without per-kernel events; kernel times from a second loop with them",
            "bytes_per_step": nbytes, "frac_of_hbm_peak": round(gbs / ctx["world"] / peaks["hbm"], 4),
            "roofline": {"kernel": dom, "bound": "hbm", "achieved": round(dach, 1), "peak": peaks["hbm"],
                         "unit": "GB/s", "frac": round(dach / peaks["hbm"], 4),
                         "traffic": dtraffic.get(dom), "traffic_source": dsrc,
                         "launch_ms": round(dom_ms, 4)},
            "kernels": {q: {"launches": len(v), "avg_ms": round(sum(v) / len(v), 4)} for q, v in per.items()}}


# ------------------------------------------------------------ CPU oracle
def cpu_baseline(w, budget_s=15.0, seed=5):
    """The float64 oracle as it stands, on a bounded sample of the workload:
    sharded forward of R token rows, backward (dx) of R/2 rows, and the weight
    gradients of J hidden units (all their dW1/dW3 rows and dW2 columns).
    Rate = algorithmic FLOPs of those outputs / wall time."""
    import numpy as np
    import oracle
    from synth import make_inputs, to_f64

    inp = make_inputs(w)
    f = {k: to_f64(v) for k, v in inp.items()}
    P = oracle.FFN(f["x"], f["W2"], w.T_p, w.act, W1=f["W1"], W3=f["W3"], b1=f["b1"], b2=f["b2"])
    rng = np.random.default_rng(seed)
    per_row_fwd = w.fwd_flops() / w.N
    per_row_dx = (2 * w.d * w.d_ff) + (2 * w.d * w.d_ff * (2 if w.act == "swiglu" else 1))
    per_j_wgrad = 2 * w.N * w.d * ((2 if w.act == "swiglu" else 1) + 1)
    # calibrate on 8 rows, then size the sample to the budget
    t0 = time.perf_counter()
    P.forward_sharded(rng.choice(w.N, 8, replace=False))
    t_row = (time.perf_counter() - t0) / 8
    R = int(max(8, min(w.N, 0.45 * budget_s / max(t_row, 1e-6))))
    Rb = max(4, R // 2)
    J = 16
    rows = rng.choice(w.N, R, replace=False)
    t0 = time.perf_counter()
    P.forward_sharded(rows)
    P.backward_rows(f["dy"], rows[:Rb])
    P.wgrad_entries(f["dy"], rng.choice(w.d_ff, J, replace=False), np.arange(w.d), np.arange(w.d))
    el = time.perf_counter() - t0
    flops = R * per_row_fwd + Rb * per_row_dx + J * per_j_wgrad
    return {"value": round(flops / el / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle", "seconds": round(el, 2),
            "sample": f"{w.name}: sharded forward of {R} token rows, dx of {Rb} rows, weight gradients of "
                      f"{J} hidden units (all d inputs/outputs); float64, OpenMP over independent outputs"}


def run_reference(args, ctx):
    """--impl reference: the oracle, timed per step on a bounded sample."""
    import numpy as np
    import oracle
    from synth import WORKLOADS, make_inputs, to_f64
    w = WORKLOADS[MAIN]
    inp = make_inputs(w)
    f = {k: to_f64(v) for k, v in inp.items()}
    P = oracle.FFN(f["x"], f["W2"], w.T_p, w.act, W1=f["W1"], W3=f["W3"])
    rng = np.random.default_rng(1)
    R, Rb, J = 16, 8, 2
    per_row_fwd = w.fwd_flops() / w.N
    per_row_dx = 2 * w.d * w.d_ff * 3
    per_j = 2 * w.N * w.d * 3
    flops = R * per_row_fwd + Rb * per_row_dx + J * per_j

    def step():
        rows = rng.choice(w.N, R, replace=False)
        P.forward_sharded(rows)
        P.backward_rows(f["dy"], rows[:Rb])
        P.wgrad_entries(f["dy"], rng.choice(w.d_ff, J, replace=False), np.arange(w.d), np.arange(w.d))

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = (time.perf_counter() - t0) / args.steps
    value = flops / el / 1e12
    sample = (f"{w.name}: per step, sharded forward of {R} token rows, dx of {Rb} rows and the weight "
              f"gradients of {J} hidden units, float64 oracle on host cores")
    return {"metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": ctx["world"],
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded host normals)",
            "config": {"workload": MAIN, "tokens": w.N, "d": w.d, "d_ff": w.d_ff, "T_p": w.T_p, "act": w.act,
                       "flop_per_step": flops},
            "impl": "reference",
            "cpu_baseline": {"kind": "oracle", "cores": oracle.num_threads(), "sample": sample,
                             "value": round(value, 6), "unit": "TFLOP/s"},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=150)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sum", choices=["fused", "standalone"], default="fused")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the per-workload table and standalone-sum line")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--tokens", type=int, default=0, help="override the token count (profiler captures)")
    ap.add_argument("--profile-attention", default="", metavar="WORKLOAD",
                    help="only run --steps fwd+bwd steps of this attention workload (profiler captures)")
    ap.add_argument("--attn-batch", type=int, default=0, help="override the attention workload's sequence count")
    ap.add_argument("--profile-ffn", action="store_true",
                    help="only run --warmup + --steps plain FFN steps (profiler captures)")
    ap.add_argument("--profile-workload", default="", metavar="WORKLOAD",
                    help="with --profile-ffn: this workload's shapes instead of the Llama-3-8B ones")
    ap.add_argument("--profile-decode", action="store_true",
                    help="with --profile-ffn: the decode-shaped forward instead of the training step")
    args = ap.parse_args()
    ctx = dist_setup(args.gpus)
    if args.impl == "reference":
        if ctx["rank"] != 0:
            return 0
        print(json.dumps(run_reference(args, ctx)), flush=True)
        return 0
    if ctx["world"] > 1:
        import torch
        torch.cuda.set_device(ctx["local"])
        ctx["dist"].init_process_group("nccl", device_id=torch.device("cuda", ctx["local"]))
    import importlib
    importlib.import_module("__graft_entry__").build()
    if args.profile_attention:
        print(json.dumps(profile_attention(args)), flush=True)
        return 0
    if args.profile_ffn:
        print(json.dumps(profile_ffn(args)), flush=True)
        return 0
    line = run_ours(args, ctx)
    if ctx["rank"] == 0:
        print(json.dumps(line), flush=True)
    if ctx["dist"] is not None:
        ctx["dist"].destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
