#!/usr/bin/env python
"""Throughput of the S6 selective scan (forward + backward) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

One step = one forward (ssm_scan_fwd) and one backward (ssm_scan_bwd) over one
batch of the workload, inputs resident in HBM. Metric: G(token*channel)/s =
B*L*D / (t_fwd + t_bwd) / 1e9, summed over ranks. Each pass is timed with
CUDA events on the launching stream; L2 (129 MB) is flushed before every
pass, outside the timed segments, and the inputs are larger than L2 anyway.
After the timed region (unless --no-extras) the line also carries the
forward without checkpoints, decode throughput through ssm_step, and
`other_ops`: the path's other calls (conv1d, dt projection, GDN2, mLSTM)
timed briefly the way their own --op runs time them.

Multi-GPU: one process per GPU (torchrun). Every rank runs the same workload
as an independent replica (the scan needs no exchange between replicas);
the job's time is the max over ranks.

--impl reference times the oracle (plain sequential C++, fp32, all host
cores) on bounded samples of the same workload, on rank 0 only.

--op conv1d times the causal depthwise conv1d + SiLU in front of the scan
(ssm_conv1d_fwd + ssm_conv1d_bwd, K = 4) on the workload's B, L, D instead,
with its own metric, HBM roofline and oracle baseline.

--op dtproj times the dt projection with its fused softplus on the tensor
cores (ssm_dtproj_fwd + ssm_dtproj_bwd, dt_rank = D/32, a read in place from
an x_proj-shaped buffer) on the workload's B*L tokens and D channels.

--op gdn2 times the Gated DeltaNet-2 chunkwise forward (gdn2_chunk_fwd) on
a GDN2 workload (default gdn2-1.3b-like: 8 x 16 heads x 2048 tokens,
K = V = 128, chunks of 64): one step = one forward call. --op mlstm times
the mLSTM stabilized chunkwise forward (mlstm_chunk_fwd) the same way
(default mlstm-8x16x2048: 8 x 16 heads x 2048 tokens, K = V = 128).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time
from dataclasses import replace

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import gen  # noqa: E402

METRIC = "selective-scan fwd+bwd G(token·channel)/s on 1 GB300; % of HBM roofline"
UNIT = "G(token·channel)/s"
DEFAULT_WORKLOAD = "mamba1.4b-bf16"
FALLBACK_HBM_GBS = 6800.0
# Special-function unit: ex2.approx / lg2.approx / rcp.approx run on the XU
# pipe, whose peak ncu reports on GB300 as sm__inst_executed_pipe_xu
# .avg.peak_sustained = 1 warp-instruction per cycle per SM, i.e. 32 results
# per clock per SM; the SFU roofline is that rate at the SM count and the
# maximum SM clock.
SFU_EX2_PER_CLK_PER_SM = 32
# A "pass" is one C-ABI call; its kernels (the main one plus, when the
# sequence is split into L-groups, the aggregate pass and the carry scan)
# are timed together between CUDA events.
PASS_KERNELS = {"fwd": "ssm_scan_fwd (ssm_fwd_kernel; + ssm_fwd_kernel<AGG> and ssm_carry_kernel when L-groups > 1)",
                "bwd": "ssm_scan_bwd (ssm_bwd_agg_kernel + ssm_carry_kernel when L-groups > 1, then ssm_bwd_kernel)"}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ------------------------------------------------------------------ bytes
def algorithmic_bytes(w, pass_):
    """Bytes a pass must move at least once (no checkpoints, no workspace, no
    re-reads): e = I/O element size; per token-channel, per token, fixed."""
    e = 2 if w.io == "bf16" else 4
    tc, bl = w.B * w.L * w.D, w.B * w.L
    if pass_ == "fwd":   # read x, z (e), dt (4); write y (e); read Bm, Cm; A, Dskip, dt_bias
        return tc * (3 * e + 4) + bl * 2 * w.N * e + w.D * w.N * 4 + 2 * w.D * 4
    # bwd: read x, z, dy (e), dt (4); write dx, dz (e), d_dt (4); read Bm, Cm (e), write dB, dC (4);
    # read A, Dskip, dt_bias; write dA, dD, d_dt_bias
    return tc * (5 * e + 8) + bl * 2 * w.N * (e + 4) + w.D * w.N * 8 + 4 * w.D * 4


CONV_K = 4
CONV_METRIC = "conv1d+SiLU fwd+bwd G(token·channel)/s on 1 GB300; % of HBM roofline"


def conv_algorithmic_bytes(w, pass_, K=CONV_K):
    """Conv bytes moved at least once: the forward reads xin and writes x; the
    backward reads xin and dx and writes dxin (e bytes each per
    token-channel); both read w and bias, the forward reads and writes the
    [B, D, K-1] state, the backward writes dw, dbias and the state's gradient."""
    e = 2 if w.io == "bf16" else 4
    tc, small = w.B * w.L * w.D, w.D * (K + 1) * 4
    st = w.B * w.D * (K - 1) * 4
    if pass_ == "fwd":
        return tc * 2 * e + small + 2 * st
    return tc * 3 * e + 2 * small + 2 * st


DTPROJ_METRIC = "dt_proj+softplus fwd+bwd G(token·channel)/s on 1 GB300; % of HBM roofline"


def dtproj_rank(w):
    """dt_rank = d_model / 16 = D / 32 (Mamba's expand = 2)."""
    return max(16, w.D // 32)


def dtproj_algorithmic_bytes(w, pass_):
    """Bytes moved at least once: a (bf16 [M,R]) and w (bf16 [D,R]) read, bias read; the forward writes
    delta (fp32 [M,D]); the backward reads ddelta and writes dpre (fp32 [M,D]) and dbias."""
    M, R = w.B * w.L, dtproj_rank(w)
    ins = M * R * 2 + w.D * R * 2 + w.D * 4
    return ins + M * w.D * 4 if pass_ == "fwd" else ins + 2 * M * w.D * 4 + w.D * 4


def mufu_ops(w, pass_):
    """Special-function-unit results a pass needs (bf16 path): one exp2 per
    (token, channel, state) for the decay, plus per (token, channel) the
    softplus (exp2, log2), the gate's sigmoid (exp2, reciprocal) and, in the
    backward, the reciprocal behind sigmoid(dt + dt_bias)."""
    tc = w.B * w.L * w.D
    return tc * w.N + tc * (4 if pass_ == "fwd" else 5)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured", d
    except Exception:
        return FALLBACK_HBM_GBS, "fallback", {}


# The device sources each C-ABI call's kernels are compiled from: a committed
# DRAM-traffic figure is used only while these files are unchanged.
CALL_SOURCES = {
    "ssm_scan_fwd": ("ssm_fwd.cu", "ssm_common.cuh", "ssm_internal.h"),
    "ssm_scan_bwd": ("ssm_bwd.cu", "ssm_fwd.cu", "ssm_common.cuh", "ssm_internal.h"),
    "ssm_conv1d_fwd": ("ssm_conv.cu", "ssm_common.cuh", "ssm_internal.h"),
    "ssm_conv1d_bwd": ("ssm_conv.cu", "ssm_common.cuh", "ssm_internal.h"),
    "ssm_dtproj_fwd": ("ssm_dtproj.cu", "ssm_common.cuh", "ssm_internal.h"),
    "ssm_dtproj_bwd": ("ssm_dtproj.cu", "ssm_common.cuh", "ssm_internal.h"),
    "gdn2_chunk_fwd": ("gdn2.cu", "tc_common.cuh", "ssm_common.cuh", "ssm_internal.h"),
    "mlstm_chunk_fwd": ("mlstm.cu", "tc_common.cuh", "ssm_common.cuh", "ssm_internal.h"),
}


def strip_c_comments(src: str) -> str:
    """C/C++ source with comments removed and whitespace runs collapsed to
    one space (string and character literals kept as written)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(call):
    """Hash of the code (comments and layout ignored) of the sources a call's
    kernels are built from: stored counters stay valid across documentation
    edits and lapse with any change to the code."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "selective_state_space_07_gb300", "csrc")
    for fn in CALL_SOURCES[call]:
        with open(os.path.join(d, fn), encoding="utf-8") as f:
            h.update((fn + "\n" + strip_c_comments(f.read())).encode())
    return h.hexdigest()[:16]


def sfu_peak_per_s(peaks):
    """ex2 results per second at the maximum SM clock (MEASURED_PEAKS.json
    sm_max_mhz, else 2070 MHz) on the current device's SMs."""
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    mhz = float(peaks.get("sm_max_mhz", 2070.0)) if peaks else 2070.0
    return SFU_EX2_PER_CLK_PER_SM * sms * mhz * 1e6


def profiled_traffic(kernel, workload):
    """DRAM bytes per call (summed over the pass's kernels) from the committed
    ncu summary, if it was taken on the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        ent = d.get(kernel, {}).get(workload)
        if ent and ent.get("source_hash") == kernel_source_hash(kernel):
            return float(ent["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self):
        self.proc = None
        self.tmp = None

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "10"],
                                         stdout=self.tmp, stderr=subprocess.DEVNULL)
        except Exception as ex:  # nvidia-smi missing: report no clocks
            log("clock sampling unavailable:", ex)
            self.proc = None

    def stop(self, gpus):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(5)
        except Exception:
            self.proc.kill()
        self.tmp.flush()
        rows = []
        with open(self.tmp.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    idx = int(parts[0])
                except ValueError:
                    continue
                if idx in gpus:
                    rows.append(parts)
        os.unlink(self.tmp.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        reasons = set()
        for r in rows:
            for name, val in zip(self.NAMES, r[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_median": statistics.median(pw) if pw else None,
                "reasons": sorted(reasons), "samples": len(rows)}


def with_cycles(clk, ms):
    """The clock record plus the step's time in SM cycles at the median clock
    sampled under load (ms x MHz), which stays comparable across clock drift."""
    if clk and clk.get("sm_mhz"):
        clk = dict(clk, sm_cycles_per_step=round(ms * clk["sm_mhz"] * 1e3))
    return clk


# ------------------------------------------------------------------ dist
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init_dist(world, backend):
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend=backend)
        return dist
    return None


def max_over_ranks(values, dist, device):
    """Each value's maximum over the ranks (the job's time is its slowest
    replica's); values unchanged on one process."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def job_value(world, token_channels, ms):
    """Whole-job throughput in G(token*channel)/s: every rank processes its own
    replica of the workload, so the job does world * B*L*D per step."""
    return world * token_channels / (ms * 1e-3) / 1e9


def visible_gpu_ids(world):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [int(v) for v in vis.split(",") if v.strip().isdigit()][:world]
    return ids or list(range(world))


# ------------------------------------------------------------------ cpu work
def decode_throughput(ssm, dv, w, dev, stream, n_tok=64):
    """ssm_step at the workload's B and D (one token of every channel per
    call), timed over n_tok consecutive tokens of the resident inputs: as
    n_tok eager calls, and replayed from one CUDA graph that holds the same
    n_tok calls (launch cost out of the way)."""
    import torch
    state = torch.zeros(w.B, w.D, w.N, dtype=torch.float32, device=dev)
    cols = [{k: dv[k][:, t].contiguous() for k in ("x", "dt", "z", "Bm", "Cm")} for t in range(n_tok)]
    ys = [torch.empty(w.B, w.D, dtype=dv["x"].dtype, device=dev) for _ in range(n_tok)]

    def run():
        for t in range(n_tok):
            c = cols[t]
            ssm.step(state, c["x"], c["dt"], dv["A"], c["Bm"], c["Cm"], c["z"], dv["Dskip"], dv["dt_bias"],
                     y_t=ys[t])

    def timed(fn, reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        cur = torch.cuda.current_stream(dev)
        a.record(cur)
        for _ in range(reps):
            fn()
        b.record(cur)
        b.synchronize()
        return a.elapsed_time(b) / reps / n_tok

    run()
    eager_ms = timed(run, 5)
    graph_ms = None
    try:
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            run()
        torch.cuda.current_stream(dev).wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run()
        g.replay()
        graph_ms = timed(g.replay, 20)
    except Exception as ex:  # a torch without graph capture: report the eager number only
        log("decode graph capture failed:", ex)
    e = 2 if w.io == "bf16" else 4
    per_call = w.B * w.D * (3 * e + 4) + w.B * 2 * w.N * e + w.B * w.D * w.N * 8 + w.D * (w.N + 2) * 4
    best = graph_ms if graph_ms is not None else eager_ms
    return {"what": f"ssm_step, one token for all {w.B}x{w.D} channels per call",
            "us_per_call_eager": round(eager_ms * 1e3, 3),
            "us_per_call_graph": None if graph_ms is None else round(graph_ms * 1e3, 3),
            "tokens_per_s": round(w.B / (best * 1e-3), 1),
            "algorithmic_bytes_per_call": per_call,
            "achieved_gbs": round(per_call / (best * 1e-3) / 1e9, 1)}


def _row(w):
    """Batch row 0 of the workload (the generator is indexed by position, so
    a one-row draw equals the first row of the full draw)."""
    return gen.make_inputs(1, w.L, w.D, w.N, io=w.io, seed=w.seed, dt_std=w.dt_std, delta_target=w.delta_target)


def _sample(row, ds):
    return replace(row, D=ds, x=row.x[:, :, :ds], dt=row.dt[:, :, :ds], z=row.z[:, :, :ds],
                   dy=row.dy[:, :, :ds], A=row.A[:ds], Dskip=row.Dskip[:ds], dt_bias=row.dt_bias[:ds])


def _oracle_step(s, cores):
    import oracle
    t0 = time.perf_counter()
    oracle.fwd(s, "f32", cores)
    oracle.bwd(s, "f32", cores)
    return time.perf_counter() - t0


def cpu_baseline(w, budget_s=12.0):
    """The oracle as it stands (fp32 instantiation: the plain sequential loop
    per channel, threads over channels) timed on a bounded sample of the
    workload: batch row 0, all tokens, the first D_s channels (D_s sized for
    about budget_s of forward + backward), repeated up to the budget."""
    import oracle
    cores = oracle.hardware_threads()
    row = _row(w)
    ds = min(w.D, max(8, cores * 2))
    t = _oracle_step(_sample(row, ds), cores)
    ds = int(min(w.D, max(ds, ds * budget_s / max(t, 1e-3))) // 8 * 8)
    s = _sample(row, ds)
    ts = []
    while sum(ts) < budget_s and len(ts) < 50:
        ts.append(_oracle_step(s, cores))
    tc = w.L * ds * len(ts)
    # the same loop on one thread, on as many channels as take about a
    # tenth of a quarter of the budget, repeated for that quarter
    t1p = _oracle_step(_sample(row, min(w.D, 8)), 1)
    s1 = _sample(row, int(min(w.D, max(8, 8 * budget_s / 40 / max(t1p, 1e-4))) // 8 * 8))
    t1 = []
    while sum(t1) < budget_s / 4 and len(t1) < 50:
        t1.append(_oracle_step(s1, 1))
    return {"value": tc / sum(ts) / 1e9, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"batch row 0, first {ds} of {w.D} channels, all {w.L} tokens, fp32 oracle fwd+bwd, "
                      f"{len(ts)} repetitions, {sum(ts):.1f} s",
            "one_core": {"value": w.L * s1.D * len(t1) / sum(t1) / 1e9, "unit": UNIT, "cores": 1,
                         "sample": f"batch row 0, first {s1.D} channels, all {w.L} tokens, {len(t1)} repetitions, "
                                   f"{sum(t1):.1f} s"}}


def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    cores = oracle.hardware_threads()
    row = _row(w)
    # size each step so that warmup + steps fit in about 150 s
    per_step = 150.0 / max(1, args.steps + args.warmup)
    t = _oracle_step(_sample(row, 8), cores)
    ds = int(min(w.D, max(8, 8 * per_step / max(t, 1e-4))) // 8 * 8)
    s = _sample(row, ds)
    for _ in range(args.warmup):
        _oracle_step(s, cores)
    ts = [_oracle_step(s, cores) for _ in range(args.steps)]
    tc = w.L * ds
    total = sum(ts)
    val = tc * len(ts) / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / len(ts), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "L": w.L, "D": w.D, "N": w.N, "io_dtype": w.io,
                   "sample_per_step": f"batch row 0, first {ds} channels, all {w.L} tokens"},
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"per step: {tc} token-channels (batch row 0, first {ds} of {w.D} "
                                   f"channels), fp32 oracle fwd+bwd on {cores} threads"},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ ours
def chunk_decode_throughput(op, ssm, t, dev, n_tok=64):
    """The op's one-token step (mlstm_step or gdn2_step) at the workload's B and H, one token of every head
    per call, over the first n_tok tokens of the resident inputs from the workload's initial state: eager,
    and replayed from one CUDA graph that holds the same n_tok calls."""
    import torch
    B, H, T, K = t["q"].shape
    V = t["v"].shape[-1]
    if op == "mlstm":
        names = ("q", "k", "v", "igate", "fgate")
        st = (t["C0"].clone(), t["n0"].clone(), t["m0"].clone())
        per_call = B * H * (K * 2 * 2 + V * 2 * 2 + 2 * 4 + 2 * (K * V + K + 1) * 4)

        def call(c, h):
            ssm.mlstm_step(c["q"], c["k"], c["v"], c["igate"], c["fgate"], st, K ** -0.5, h=h)
    else:
        names = ("q", "k", "v", "g", "b", "w")
        st = t["state"].clone()
        per_call = B * H * (K * (3 * 2 + 4) + V * (2 * 2 + 2) + 2 * K * V * 4)

        def call(c, h):
            ssm.gdn2_step(c["q"], c["k"], c["v"], c["g"], c["b"], c["w"], st, K ** -0.5, out=h)
    cols = [{n: t[n][:, :, i].contiguous() for n in names} for i in range(n_tok)]
    hs = [torch.empty(B, H, V, dtype=torch.bfloat16, device=dev) for _ in range(n_tok)]

    def run():
        for i in range(n_tok):
            call(cols[i], hs[i])

    def timed(fn, reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        cur = torch.cuda.current_stream(dev)
        a.record(cur)
        for _ in range(reps):
            fn()
        b.record(cur)
        b.synchronize()
        return a.elapsed_time(b) / reps / n_tok

    run()
    eager_ms = timed(run, 5)
    graph_ms = None
    try:
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            run()
        torch.cuda.current_stream(dev).wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run()
        g.replay()
        graph_ms = timed(g.replay, 20)
    except Exception as ex:  # a torch without graph capture: report the eager number only
        log(f"{op} decode graph capture failed:", ex)
    best = graph_ms if graph_ms is not None else eager_ms
    return {"what": f"{op}_step, one token for all {B}x{H} heads per call (state read and written in place)",
            "us_per_call_eager": round(eager_ms * 1e3, 3),
            "us_per_call_graph": None if graph_ms is None else round(graph_ms * 1e3, 3),
            "tokens_per_s": round(B / (best * 1e-3), 1),
            "algorithmic_bytes_per_call": per_call,
            "hbm_frac": round(per_call / (best * 1e-3) / 1e9 / measured_peaks()[0], 4)}


def emit(args, line, dist):
    """End a run: print its JSON line (the command-line path), or hand the
    line back when bench.py collects it as an extra of the scan's run."""
    if dist:
        dist.destroy_process_group()
    if getattr(args, "collect", False):
        return line
    print(json.dumps(line), flush=True)
    return 0


def other_ops(args, w):
    """The path's other calls, each timed briefly after the scan's timed
    region (50 calls, the same L2 flush and CUDA events as its own --op run,
    no CPU baseline or e2e): conv1d + SiLU fwd+bwd and the dt projection
    fwd+bwd on the scan workload's shapes, the GDN2 and mLSTM chunkwise
    forwards on their default workloads."""
    sub = argparse.Namespace(**vars(args))
    sub.steps, sub.warmup, sub.no_cpu_baseline, sub.no_e2e, sub.collect = 50, 3, True, True, True
    runs = (("conv1d", lambda: run_conv(sub, w)), ("dtproj", lambda: run_dtproj(sub, w)),
            ("gdn2", lambda: run_chunk(sub, ChunkOp("gdn2"))), ("mlstm", lambda: run_chunk(sub, ChunkOp("mlstm"))))
    out = {}
    for name, fn in runs:
        try:
            line = fn()
        except Exception as ex:  # an extra must not sink the scan's line
            log(f"extra {name} failed: {ex}")
            continue
        rf = line["roofline"]
        out[name] = {"workload": line["config"]["workload"], "metric": line["metric"], "value": line["value"],
                     "unit": line["unit"], "ms_per_call": line["ms_per_step"], "steps": line["steps"],
                     "roofline": {k: rf.get(k) for k in ("bound", "kernel", "achieved", "peak", "unit", "frac",
                                                          "traffic")},
                     "gpu_launches": line["gpu_launches"], "status": line["status"],
                     "sm_mhz": (line.get("clocks") or {}).get("sm_mhz"),
                     "reasons": (line.get("clocks") or {}).get("reasons")}
    return out


def run_ours(args, w):
    import torch
    import selective_state_space_07_gb300 as ssm

    rank, world, local = dist_env()
    dist = init_dist(world, "nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ssm.build()

    t0 = time.time()
    inp = gen.workload_inputs(w.name)
    log(f"[rank {rank}] inputs generated in {time.time() - t0:.1f}s")
    io = torch.bfloat16 if w.io == "bf16" else torch.float32

    def up(a, dtype):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev, dtype)

    dv = {"x": up(inp.x, io), "z": up(inp.z, io), "Bm": up(inp.Bm, io), "Cm": up(inp.Cm, io),
          "dy": up(inp.dy, io), "dt": up(inp.dt, torch.float32), "A": up(inp.A, torch.float32),
          "Dskip": up(inp.Dskip, torch.float32), "dt_bias": up(inp.dt_bias, torch.float32)}
    del inp
    ws = ssm.Workspace(w.B, w.L, w.D, dev)
    y = torch.empty_like(dv["x"])
    ckpt = torch.empty(ssm.ckpt_elems(w.B, w.L, w.D), dtype=torch.float32, device=dev)
    grads = None
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    kw = dict(nsplit=args.nsplit, groups=args.groups)

    def fwd():
        ssm.scan_fwd(dv["x"], dv["dt"], dv["A"], dv["Bm"], dv["Cm"], dv["z"], dv["Dskip"], dv["dt_bias"],
                     y=y, ckpt=ckpt, workspace=ws, **kw)
        return ssm.last_launch_count()

    def bwd():
        nonlocal grads
        grads = ssm.scan_bwd(dv["x"], dv["dt"], dv["A"], dv["Bm"], dv["Cm"], dv["dy"], ckpt, dv["z"],
                             dv["Dskip"], dv["dt_bias"], out=grads, workspace=ws, **kw)
        grads.pop("workspace", None)
        return ssm.last_launch_count()

    for _ in range(args.warmup):
        flush.zero_()
        fwd()
        flush.zero_()
        bwd()
    torch.cuda.synchronize()
    if ssm.poll_status(ws) != 0:
        raise RuntimeError("non-finite outputs during warm-up")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks = ClockSampler()
    if rank == 0:
        clocks.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    launches = 0
    wall0 = time.perf_counter()
    for k in range(args.steps):
        e = ev[k]
        flush.zero_()
        e[0].record(stream)
        launches += fwd()
        e[1].record(stream)
        flush.zero_()
        e[2].record(stream)
        launches += bwd()
        e[3].record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop(set(visible_gpu_ids(world))) if rank == 0 else None
    tf = [e[0].elapsed_time(e[1]) for e in ev]
    tb = [e[2].elapsed_time(e[3]) for e in ev]
    ms_f, ms_b = sum(tf) / len(tf), sum(tb) / len(tb)
    ms_step = ms_f + ms_b
    ms_f, ms_b, ms_step = max_over_ranks([ms_f, ms_b, ms_step], dist, dev)
    status = ssm.poll_status(ws)
    tc = w.B * w.L * w.D
    value = job_value(world, tc, ms_step)

    # ---- the forward without checkpoints (inference: y and the last state only)
    ms_inf = None
    if not args.no_extras:
        h_last = torch.empty(w.B, w.D, w.N, dtype=torch.float32, device=dev)
        ts = []
        for k in range(max(3, min(args.steps, 50)) + 3):
            flush.zero_()
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record(stream)
            ssm.scan_fwd(dv["x"], dv["dt"], dv["A"], dv["Bm"], dv["Cm"], dv["z"], dv["Dskip"], dv["dt_bias"],
                         y=y, h_last=h_last, save_ckpt=False, workspace=ws, **kw)
            b_.record(stream)
            b_.synchronize()
            if k >= 3:
                ts.append(a_.elapsed_time(b_))
        ms_inf = max_over_ranks([sum(ts) / len(ts)], dist, dev)[0]
    decode = decode_throughput(ssm, dv, w, dev, stream) if not args.no_extras else None
    others = other_ops(args, w) if not args.no_extras and world == 1 else None

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        host = {k: v.detach().cpu().pin_memory() for k, v in dv.items() if v is not None}
        e2e_steps = max(3, min(args.steps, 20))
        # back-to-back calls through the host API: copies in, compute and
        # copies out of consecutive steps overlap on three streams
        pipe = ssm.HostPipeline(host, dev)
        res = None
        for _ in range(3):
            res = pipe.step(host, res)
        pipe.synchronize()
        es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist:
            dist.barrier()
        es.record(pipe.s_in)
        for _ in range(e2e_steps):
            res = pipe.step(host, res)
        ee.record(pipe.s_out)  # after the last step's last copy back
        pipe.synchronize()
        e2e_ms = es.elapsed_time(ee) / e2e_steps
        e2e_ms = max_over_ranks([e2e_ms], dist, dev)[0]
        e2e = {"value": round(job_value(world, tc, e2e_ms), 3), "unit": UNIT,
               "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in host.values()),
               "d2h_bytes_per_step": sum(v.numel() * v.element_size() for v in res.values()),
               "ms_per_step": round(e2e_ms, 4),
               "api": "HostPipeline.step (pinned host buffers; 3 streams, 2 device buffer sets)"}

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    peak, peak_kind, peaks = measured_peaks()
    sfu_peak = sfu_peak_per_s(peaks)
    rf, sfu = {}, {}
    for name, ms in (("fwd", ms_f), ("bwd", ms_b)):
        ab = algorithmic_bytes(w, name)
        ach = ab / (ms * 1e-3) / 1e9
        call = "ssm_scan_" + name
        rf[name] = {"bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                    "frac": round(ach / peak, 4), "peak_kind": peak_kind, "kernel": PASS_KERNELS[name],
                    "algorithmic_bytes_per_launch": ab, "ms_per_launch": round(ms, 5),
                    "traffic": profiled_traffic(call, w.name)}
        ops = mufu_ops(w, name) / (ms * 1e-3)
        sfu[name] = {"bound": "sfu", "achieved": round(ops / 1e12, 3), "peak": round(sfu_peak / 1e12, 3),
                     "unit": "Tex2/s", "frac": round(ops / sfu_peak, 4),
                     "peak_kind": "derived: ncu XU peak (1 warp-instruction = 32 results /clk/SM) x SMs x max SM clock"}
    dom = "bwd" if ms_b >= ms_f else "fwd"
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        try:
            cpu = cpu_baseline(w)
        except Exception as ex:
            log("cpu baseline failed:", ex)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "L": w.L, "D": w.D, "N": w.N, "io_dtype": w.io,
                   "seed": w.seed, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (129 MB) and a 512 MiB write flushes L2 before every pass",
                   "ms_fwd": round(ms_f, 5), "ms_bwd": round(ms_b, 5),
                   "hbm_frac_fwd": rf["fwd"]["frac"], "hbm_frac_bwd": rf["bwd"]["frac"]},
        "roofline": rf[dom],
        "roofline_other": rf["fwd" if dom == "bwd" else "bwd"],
        "fwd_inference": None if ms_inf is None else {
            "ms": round(ms_inf, 5), "what": "ssm_scan_fwd with ckpt = NULL (y and h_last only)",
            "hbm_frac": round(algorithmic_bytes(w, "fwd") / (ms_inf * 1e-3) / 1e9 / peak, 4)},
        "decode": decode,
        "other_ops": others,
        "sfu_roofline": sfu,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": with_cycles(clk, ms_step),
        "status": status,
        "wall_s_timed_loop": round(wall, 3),
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def _conv_oracle_step(c):
    import oracle
    t0 = time.perf_counter()
    oracle.conv_fwd(c.xin, c.w, c.bias, c.state, dtype="f32")
    oracle.conv_bwd(c.xin, c.w, c.dx, c.bias, c.state, dtype="f32")
    return time.perf_counter() - t0


def conv_cpu_sample(w, budget_s):
    """The conv oracle (fp32, one thread: plain loops per channel) on batch
    row 0, all tokens, the first D_s channels sized for about budget_s."""
    c = gen.make_conv_inputs(1, w.L, 64, CONV_K, io=w.io, seed=w.seed, with_state=True)
    t = _conv_oracle_step(c)
    ds = int(min(w.D, max(64, 64 * budget_s / max(t, 1e-4))) // 8 * 8)
    return gen.make_conv_inputs(1, w.L, ds, CONV_K, io=w.io, seed=w.seed, with_state=True), ds


def run_conv_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    c, ds = conv_cpu_sample(w, 150.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        _conv_oracle_step(c)
    ts = [_conv_oracle_step(c) for _ in range(args.steps)]
    total = sum(ts)
    val = w.L * ds * len(ts) / total / 1e9
    sample = f"per step: batch row 0, first {ds} of {w.D} channels, all {w.L} tokens, fp32 conv oracle fwd+bwd"
    line = {
        "impl": "reference", "metric": CONV_METRIC, "value": val, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(ts), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name + "-conv1d", "B": w.B, "L": w.L, "D": w.D, "K": CONV_K, "io_dtype": w.io},
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_conv(args, w):
    """The conv1d + SiLU pair on the workload's activations: one step = one
    ssm_conv1d_fwd and one ssm_conv1d_bwd, each timed with CUDA events after
    an L2 flush, inputs resident in HBM."""
    import torch
    import selective_state_space_07_gb300 as ssm

    rank, world, local = dist_env()
    dist = init_dist(world, "nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ssm.build()
    c = gen.make_conv_inputs(w.B, w.L, w.D, CONV_K, io=w.io, seed=w.seed, with_state=True)
    io = torch.bfloat16 if w.io == "bf16" else torch.float32

    def up(a, dtype=torch.float32):
        return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev, dtype)

    xin, dx = up(c.xin, io), up(c.dx, io)
    wt, bias, st = up(c.w), up(c.bias), up(c.state)
    del c
    x, dxin = torch.empty_like(xin), torch.empty_like(xin)
    st_out = torch.empty_like(st)
    ws = ssm.Workspace(1, 1, 8, dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    grads = None

    def fwd():
        ssm.conv1d_fwd(xin, wt, bias, st, x=x, state_out=st_out, workspace=ws)
        return ssm.last_launch_count()

    def bwd():
        nonlocal grads
        grads = ssm.conv1d_bwd(xin, wt, dx, bias, st, dxin=dxin, want_dstate=True, workspace=ws)
        return ssm.last_launch_count()

    for _ in range(args.warmup):
        flush.zero_()
        fwd()
        flush.zero_()
        bwd()
    torch.cuda.synchronize()
    if ssm.poll_status(ws) != 0:
        raise RuntimeError("non-finite outputs during warm-up")
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks = ClockSampler()
    if rank == 0:
        clocks.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    launches = 0
    for e in ev:
        flush.zero_()
        e[0].record(stream)
        launches += fwd()
        e[1].record(stream)
        flush.zero_()
        e[2].record(stream)
        launches += bwd()
        e[3].record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop(set(visible_gpu_ids(world))) if rank == 0 else None
    ms_f = sum(e[0].elapsed_time(e[1]) for e in ev) / len(ev)
    ms_b = sum(e[2].elapsed_time(e[3]) for e in ev) / len(ev)
    ms_f, ms_b = max_over_ranks([ms_f, ms_b], dist, dev)
    status = ssm.poll_status(ws)
    tc = w.B * w.L * w.D
    value = job_value(world, tc, ms_f + ms_b)

    # end to end: pinned host inputs in, both passes, results back, one stream
    e2e = None
    if not args.no_e2e:
        h_in = {"xin": xin.cpu().pin_memory(), "dx": dx.cpu().pin_memory()}
        h_out = {"x": torch.empty_like(h_in["xin"]).pin_memory(), "dxin": torch.empty_like(h_in["xin"]).pin_memory(),
                 "dw": torch.empty(w.D, CONV_K).pin_memory(), "dbias": torch.empty(w.D).pin_memory()}

        def e2e_step():
            xin.copy_(h_in["xin"], non_blocking=True)
            dx.copy_(h_in["dx"], non_blocking=True)
            fwd()
            bwd()
            h_out["x"].copy_(x, non_blocking=True)
            h_out["dxin"].copy_(dxin, non_blocking=True)
            h_out["dw"].copy_(grads["dw"], non_blocking=True)
            h_out["dbias"].copy_(grads["dbias"], non_blocking=True)

        for _ in range(3):
            e2e_step()
        n = max(3, min(args.steps, 20))
        es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        es.record(stream)
        for _ in range(n):
            e2e_step()
        ee.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks([es.elapsed_time(ee) / n], dist, dev)[0]
        e2e = {"value": round(job_value(world, tc, e2e_ms), 3), "unit": UNIT,
               "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in h_in.values()),
               "d2h_bytes_per_step": sum(v.numel() * v.element_size() for v in h_out.values()),
               "ms_per_step": round(e2e_ms, 4), "api": "conv1d_fwd + conv1d_bwd on one stream, pinned host copies"}
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0
    peak, peak_kind, _ = measured_peaks()
    rf = {}
    for name, ms in (("fwd", ms_f), ("bwd", ms_b)):
        ab = conv_algorithmic_bytes(w, name)
        ach = ab / (ms * 1e-3) / 1e9
        rf[name] = {"bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                    "frac": round(ach / peak, 4), "peak_kind": peak_kind, "kernel": f"ssm_conv_{name}_kernel",
                    "algorithmic_bytes_per_launch": ab, "ms_per_launch": round(ms, 5),
                    "traffic": profiled_traffic("ssm_conv1d_" + name, w.name)}
    dom = "bwd" if ms_b >= ms_f else "fwd"
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cs, ds = conv_cpu_sample(w, 6.0)
        ts = []
        while sum(ts) < 12.0 and len(ts) < 50:
            ts.append(_conv_oracle_step(cs))
        cpu = {"value": w.L * ds * len(ts) / sum(ts) / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"batch row 0, first {ds} of {w.D} channels, all {w.L} tokens, fp32 conv oracle "
                         f"fwd+bwd, {len(ts)} repetitions, {sum(ts):.1f} s"}
    line = {
        "metric": CONV_METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_f + ms_b, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name + "-conv1d", "B": w.B, "L": w.L, "D": w.D, "K": CONV_K, "io_dtype": w.io,
                   "seed": w.seed, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (129 MB) and a 512 MiB write flushes L2 before every pass",
                   "ms_fwd": round(ms_f, 5), "ms_bwd": round(ms_b, 5),
                   "hbm_frac_fwd": rf["fwd"]["frac"], "hbm_frac_bwd": rf["bwd"]["frac"]},
        "roofline": rf[dom], "roofline_other": rf["fwd" if dom == "bwd" else "bwd"],
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": with_cycles(clk, ms_f + ms_b),
        "status": status,
    }
    return emit(args, line, dist)


def _dtproj_oracle_step(a, wt, bias, dd):
    import oracle
    t0 = time.perf_counter()
    oracle.dtproj_fwd(a, wt, bias, dtype="f32")
    oracle.dtproj_bwd(a, wt, dd, bias, dtype="f32")
    return time.perf_counter() - t0


def dtproj_cpu_sample(w, budget_s):
    """The dt-projection oracle (fp32, one thread: plain loops) on the first rows of the workload, all D
    channels, sized for about budget_s."""
    R = dtproj_rank(w)
    c = gen.make_dtproj_inputs(1, 64, w.D, R, seed=w.seed)
    t = _dtproj_oracle_step(c.a[0], c.w, c.bias, c.ddelta[0])
    rows = int(min(w.B * w.L, max(64, 64 * budget_s / max(t, 1e-4))))
    c = gen.make_dtproj_inputs(1, rows, w.D, R, seed=w.seed)
    return (c.a[0], c.w, c.bias, c.ddelta[0]), rows


def run_dtproj_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    smp, rows = dtproj_cpu_sample(w, 150.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        _dtproj_oracle_step(*smp)
    ts = [_dtproj_oracle_step(*smp) for _ in range(args.steps)]
    total = sum(ts)
    val = rows * w.D * len(ts) / total / 1e9
    sample = f"per step: the first {rows} of {w.B * w.L} token rows, all {w.D} channels, fp32 dt-projection oracle fwd+bwd"
    line = {
        "impl": "reference", "metric": DTPROJ_METRIC, "value": val, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(ts), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name + "-dtproj", "M": w.B * w.L, "D": w.D, "R": dtproj_rank(w)},
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_dtproj(args, w):
    """ssm_dtproj_fwd + ssm_dtproj_bwd on the workload's tokens and channels: one step = one forward and
    one backward call, each timed with CUDA events after an L2 flush, inputs resident in HBM."""
    import torch
    import selective_state_space_07_gb300 as ssm

    rank, world, local = dist_env()
    dist = init_dist(world, "nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ssm.build()
    R = dtproj_rank(w)
    c = gen.make_dtproj_inputs(w.B, w.L, w.D, R, seed=w.seed)
    xp = torch.zeros(w.B, w.L, R + 32, dtype=torch.bfloat16, device=dev)  # x_proj output: dt_rank | B | C
    xp[..., :R] = torch.from_numpy(c.a).to(dev, torch.bfloat16)
    a = xp[..., :R]
    wt = torch.from_numpy(c.w).to(dev, torch.bfloat16)
    bias = torch.from_numpy(c.bias).to(dev)
    dd = torch.from_numpy(c.ddelta).to(dev)
    del c
    delta = torch.empty(w.B, w.L, w.D, dtype=torch.float32, device=dev)
    dpre = torch.empty_like(delta)
    ws = ssm.Workspace(1, 1, 8, dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    out = {}

    def fwd():
        ssm.dtproj_fwd(a, wt, bias, delta=delta, workspace=ws)
        return ssm.last_launch_count()

    def bwd():
        out.update(ssm.dtproj_bwd(a, wt, dd, bias, dpre=dpre, workspace=ws))
        return ssm.last_launch_count()

    for _ in range(args.warmup):
        flush.zero_()
        fwd()
        flush.zero_()
        bwd()
    torch.cuda.synchronize()
    st = ssm.poll_status(ws)
    if st != 0:
        raise RuntimeError(f"status {st} during warm-up")
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks = ClockSampler()
    if rank == 0:
        clocks.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    launches = 0
    for e in ev:
        flush.zero_()
        e[0].record(stream)
        launches += fwd()
        e[1].record(stream)
        flush.zero_()
        e[2].record(stream)
        launches += bwd()
        e[3].record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop(set(visible_gpu_ids(world))) if rank == 0 else None
    ms_f = sum(e[0].elapsed_time(e[1]) for e in ev) / len(ev)
    ms_b = sum(e[2].elapsed_time(e[3]) for e in ev) / len(ev)
    ms_f, ms_b = max_over_ranks([ms_f, ms_b], dist, dev)
    status = ssm.poll_status(ws)
    tc = w.B * w.L * w.D
    value = job_value(world, tc, ms_f + ms_b)

    e2e = None
    if not args.no_e2e:  # the x_proj buffer and ddelta in from pinned host memory, delta, dpre and dbias back
        h_in = {"xp": xp.cpu().pin_memory(), "dd": dd.cpu().pin_memory()}
        h_out = {"delta": torch.empty_like(delta, device="cpu").pin_memory(),
                 "dpre": torch.empty_like(dpre, device="cpu").pin_memory(),
                 "dbias": torch.empty(w.D).pin_memory()}

        def e2e_step():
            xp.copy_(h_in["xp"], non_blocking=True)
            dd.copy_(h_in["dd"], non_blocking=True)
            fwd()
            bwd()
            h_out["delta"].copy_(delta, non_blocking=True)
            h_out["dpre"].copy_(dpre, non_blocking=True)
            h_out["dbias"].copy_(out["dbias"], non_blocking=True)

        for _ in range(3):
            e2e_step()
        n = max(3, min(args.steps, 20))
        es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        es.record(stream)
        for _ in range(n):
            e2e_step()
        ee.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks([es.elapsed_time(ee) / n], dist, dev)[0]
        e2e = {"value": round(job_value(world, tc, e2e_ms), 3), "unit": UNIT,
               "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in h_in.values()),
               "d2h_bytes_per_step": sum(v.numel() * v.element_size() for v in h_out.values()),
               "ms_per_step": round(e2e_ms, 4), "api": "dtproj_fwd + dtproj_bwd on one stream, pinned host copies"}
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0
    peak, peak_kind, peaks = measured_peaks()
    flops = 2.0 * w.B * w.L * w.D * R
    tpk = float(peaks.get("bf16_tflops", 1900.0)) if peaks else 1900.0
    rf, tens = {}, {}
    for name, ms in (("fwd", ms_f), ("bwd", ms_b)):
        ab = dtproj_algorithmic_bytes(w, name)
        ach = ab / (ms * 1e-3) / 1e9
        rf[name] = {"bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                    "frac": round(ach / peak, 4), "peak_kind": peak_kind, "kernel": f"ssm_dtproj_kernel<{name == 'bwd'}>",
                    "algorithmic_bytes_per_launch": ab, "ms_per_launch": round(ms, 5),
                    "traffic": profiled_traffic("ssm_dtproj_" + name, w.name)}
        tf = flops / (ms * 1e-3) / 1e12
        tens[name] = {"bound": "tensor", "achieved": round(tf, 2), "peak": tpk, "unit": "TFLOP/s",
                      "frac": round(tf / tpk, 4), "peak_kind": "measured bf16 (burst)" if peaks else "fallback"}
    dom = "bwd" if ms_b >= ms_f else "fwd"
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        smp, rows = dtproj_cpu_sample(w, 6.0)
        ts = []
        while sum(ts) < 12.0 and len(ts) < 50:
            ts.append(_dtproj_oracle_step(*smp))
        cpu = {"value": rows * w.D * len(ts) / sum(ts) / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"the first {rows} of {w.B * w.L} token rows, all {w.D} channels, fp32 dt-projection "
                         f"oracle fwd+bwd, {len(ts)} repetitions, {sum(ts):.1f} s"}
    line = {
        "metric": DTPROJ_METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_f + ms_b, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name + "-dtproj", "M": w.B * w.L, "D": w.D, "R": R, "seed": w.seed,
                   "parallelism": f"replicas x{world}",
                   "l2": "outputs larger than L2 (129 MB) and a 512 MiB write flushes L2 before every pass",
                   "ms_fwd": round(ms_f, 5), "ms_bwd": round(ms_b, 5),
                   "hbm_frac_fwd": rf["fwd"]["frac"], "hbm_frac_bwd": rf["bwd"]["frac"]},
        "roofline": rf[dom], "roofline_other": rf["fwd" if dom == "bwd" else "bwd"], "tensor_roofline": tens,
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": with_cycles(clk, ms_f + ms_b),
        "status": status,
    }
    return emit(args, line, dist)


# ------------------------------------------------------------------ gdn2, mlstm
GDN2_METRIC = "gdn2 chunkwise forward M(token·head)/s on 1 GB300; % of HBM roofline"
MLSTM_METRIC = "mlstm chunkwise forward M(token·head)/s on 1 GB300; % of HBM roofline"
CHUNK_UNIT = "M(token·head)/s"
CHUNK = 64  # tokens per chunk of both chunked forwards


def gdn2_algorithmic_bytes(B, H, T, K, V):
    """Bytes the forward moves at least once: q, k, b (bf16) and g (fp32) per
    key channel, v and w (bf16) per value channel, out (bf16) per value
    channel, for every (token, head); the fp32 state read and written once
    per (batch, head)."""
    return B * H * T * (K * (3 * 2 + 4) + V * (2 * 2 + 2)) + 2 * B * H * K * V * 4


def gdn2_flops(B, H, T, K, V, c=CHUNK):
    """The method's multiply-add work per full chunk, 2 flops each: q k^T and
    (b k) k^T (2 c^2 K), the key-mean decay as a product (c^2 K), the WY rows
    W and U from the inverse (c^2 K + c^2 V), W S (c K V), the output's two
    terms (c^2 V + c K V) and the state update (c K V)."""
    per_chunk = 2 * (2 * c * c * K + c * c * K + c * c * (K + V) + 3 * c * K * V + c * c * V)
    return B * H * (T / c) * per_chunk


def mlstm_algorithmic_bytes(B, H, T, K, V):
    """Bytes the forward moves at least once: q, k (bf16) per key channel, v
    and h (bf16) per value channel and the two fp32 gate pre-activations, for
    every (token, head); the fp32 state (C, n, m) read and written once per
    (batch, head)."""
    return B * H * T * (K * 2 * 2 + V * 2 * 2 + 2 * 4) + 2 * B * H * (K * V + K + 1) * 4


def mlstm_flops(B, H, T, K, V, c=CHUNK):
    """The method's multiply-add work per full chunk, 2 flops each: q k^T
    (c^2 K), P v (c^2 V), the state's share of the output q C (c K V) and the
    state update sum gamma k v^T (c K V)."""
    return B * H * (T / c) * 2 * (c * c * K + c * c * V + 2 * c * K * V)


class ChunkOp:
    """One of the chunked forwards as bench.py times it: its workloads, the
    device tensors of a problem, the call, the oracle step and the roofline
    figures."""

    def __init__(self, op):
        self.op = op
        if op == "gdn2":
            self.metric, self.workloads, self.default = GDN2_METRIC, gen.GDN2_WORKLOADS, "gdn2-1.3b-like"
            self.call_name, self.kernel = "gdn2_chunk_fwd", "gdn2_chunk_fwd_kernel"
            self.bytes, self.flops = gdn2_algorithmic_bytes, gdn2_flops
        else:
            self.metric, self.workloads, self.default = MLSTM_METRIC, gen.MLSTM_WORKLOADS, "mlstm-8x16x2048"
            self.call_name, self.kernel = "mlstm_chunk_fwd", "mlstm_chunk_fwd_kernel"
            self.bytes, self.flops = mlstm_algorithmic_bytes, mlstm_flops

    def name(self, args):
        return args.workload if args.workload in self.workloads else self.default

    def inputs(self, B, H, T, K, V, seed):
        if self.op == "gdn2":
            return gen.make_gdn2_inputs(B, H, T, K, V, seed=seed)
        return gen.make_mlstm_inputs(B, H, T, K, V, seed=seed)

    def oracle_step(self, x, tmax):
        """Seconds the float64 oracle takes on head (0, 0), the first tmax tokens."""
        sl = lambda a: a[:1, :1, :tmax]  # noqa: E731
        t0 = time.perf_counter()
        if self.op == "gdn2":
            from oracle import gdn2_oracle
            gdn2_oracle.chunk_wy_forward(sl(x.q), sl(x.k), sl(x.v), sl(x.g), sl(x.b), sl(x.w), x.state[:1, :1],
                                         x.scale, chunk=CHUNK)
        else:
            from oracle import mlstm_oracle
            mlstm_oracle.chunkwise(sl(x.q), sl(x.k), sl(x.v), sl(x.igate), sl(x.fgate), x.C0[:1, :1], x.n0[:1, :1],
                                   x.m0[:1, :1], scale=x.scale, chunk=CHUNK)
        return time.perf_counter() - t0

    def cpu_sample(self, name, budget_s):
        """Head (0, 0) of the workload, the first tokens (whole chunks), sized for
        about budget_s of oracle time."""
        B, H, T, K, V, seed = self.workloads[name]
        x = self.inputs(1, 1, T, K, V, seed)
        t = self.oracle_step(x, CHUNK)
        tmax = int(min(T, max(CHUNK, CHUNK * budget_s / max(t, 1e-4))) // CHUNK * CHUNK)
        return x, tmax

    def device_setup(self, x, dev):
        """Device inputs, outputs and the call (returning the launch count)."""
        import torch
        import selective_state_space_07_gb300 as ssm
        bf, f32 = torch.bfloat16, torch.float32
        B, H, T, K, V = x.B, x.H, x.T, x.K, x.V
        scale = K ** -0.5
        ws = ssm.Workspace(1, 1, 8, dev)
        if self.op == "gdn2":
            t = {n: torch.from_numpy(getattr(x, n)).to(dev, bf) for n in ("q", "k", "v", "b", "w")}
            t["g"] = torch.from_numpy(x.g).to(dev, f32)
            t["state"] = torch.from_numpy(x.state).to(dev, f32)
            o = {"out": torch.empty(B, H, T, V, dtype=bf, device=dev),
                 "state": torch.empty(B, H, K, V, dtype=f32, device=dev)}

            def call():
                ssm.gdn2_fwd(t["q"], t["k"], t["v"], t["g"], t["b"], t["w"], t["state"], scale, out=o["out"],
                             state_out=o["state"], workspace=ws)
                return ssm.last_launch_count()
        else:
            t = {n: torch.from_numpy(getattr(x, n)).to(dev, bf) for n in ("q", "k", "v")}
            for n in ("igate", "fgate", "C0", "n0", "m0"):
                t[n] = torch.from_numpy(np.ascontiguousarray(getattr(x, n))).to(dev, f32)
            o = {"h": torch.empty(B, H, T, V, dtype=bf, device=dev), "C": torch.empty(B, H, K, V, dtype=f32, device=dev),
                 "n": torch.empty(B, H, K, dtype=f32, device=dev), "m": torch.empty(B, H, dtype=f32, device=dev)}

            def call():
                ssm.mlstm_fwd(t["q"], t["k"], t["v"], t["igate"], t["fgate"], (t["C0"], t["n0"], t["m0"]), scale,
                              h=o["h"], state_out=(o["C"], o["n"], o["m"]), workspace=ws)
                return ssm.last_launch_count()
        return t, o, call, ws


def run_chunk_reference(args, op):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    name = op.name(args)
    B, H, T, K, V, seed = op.workloads[name]
    x, tmax = op.cpu_sample(name, 150.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        op.oracle_step(x, tmax)
    ts = [op.oracle_step(x, tmax) for _ in range(args.steps)]
    total = sum(ts)
    val = tmax * len(ts) / total / 1e6
    sample = (f"per step: head (0, 0), the first {tmax} of {T} tokens, float64 numpy oracle of the chunked forward "
              f"(numpy's BLAS may thread its products over the host's cores)")
    line = {
        "impl": "reference", "metric": op.metric, "value": val, "unit": CHUNK_UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(ts), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": name, "B": B, "H": H, "T": T, "K": K, "V": V, "chunk": CHUNK},
        "cpu_baseline": {"value": val, "unit": CHUNK_UNIT, "cores": os.cpu_count(), "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": CHUNK_UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_chunk(args, op):
    """A chunked forward on its workload: one step = one forward call timed with
    CUDA events after an L2 flush, inputs resident in HBM."""
    import torch
    import selective_state_space_07_gb300 as ssm

    rank, world, local = dist_env()
    dist = init_dist(world, "nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ssm.build()
    name = op.name(args)
    B, H, T, K, V, seed = op.workloads[name]
    x = op.inputs(B, H, T, K, V, seed)
    t, outs, fwd, ws = op.device_setup(x, dev)
    del x
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        flush.zero_()
        fwd()
    torch.cuda.synchronize()
    if ssm.poll_status(ws) != 0:
        raise RuntimeError("non-zero status during warm-up")
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    clocks = ClockSampler()
    if rank == 0:
        clocks.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    launches = 0
    for e in ev:
        flush.zero_()
        e[0].record(stream)
        launches += fwd()
        e[1].record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop(set(visible_gpu_ids(world))) if rank == 0 else None
    ms = max_over_ranks([sum(e[0].elapsed_time(e[1]) for e in ev) / len(ev)], dist, dev)[0]
    status = ssm.poll_status(ws)
    units = B * H * T
    value = world * units / (ms * 1e-3) / 1e6
    decode = chunk_decode_throughput(op.op, ssm, t, dev) if not getattr(args, "no_extras", False) else None

    e2e = None
    if not args.no_e2e:  # inputs in from pinned host memory, the output and the final state back
        h_in = {n: v.cpu().pin_memory() for n, v in t.items()}
        h_out = {n: torch.empty_like(v, device="cpu").pin_memory() for n, v in outs.items()}

        def e2e_step():
            for n, v in h_in.items():
                t[n].copy_(v, non_blocking=True)
            fwd()
            for n, v in h_out.items():
                v.copy_(outs[n], non_blocking=True)

        for _ in range(3):
            e2e_step()
        n = max(3, min(args.steps, 20))
        es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        es.record(stream)
        for _ in range(n):
            e2e_step()
        ee.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks([es.elapsed_time(ee) / n], dist, dev)[0]
        e2e = {"value": round(world * units / (e2e_ms * 1e-3) / 1e6, 3), "unit": CHUNK_UNIT,
               "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in h_in.values()),
               "d2h_bytes_per_step": sum(v.numel() * v.element_size() for v in h_out.values()),
               "ms_per_step": round(e2e_ms, 4), "api": f"{op.op}_fwd on one stream, pinned host copies"}
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0
    peak, peak_kind, peaks = measured_peaks()
    ab = op.bytes(B, H, T, K, V)
    ach = ab / (ms * 1e-3) / 1e9
    rf = {"bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s", "frac": round(ach / peak, 4),
          "peak_kind": peak_kind, "kernel": op.kernel, "algorithmic_bytes_per_launch": ab,
          "ms_per_launch": round(ms, 5), "traffic": profiled_traffic(op.call_name, name)}
    fl = op.flops(B, H, T, K, V)
    tpk = float(peaks.get("bf16_tflops", 1900.0)) if peaks else 1900.0
    tf = fl / (ms * 1e-3) / 1e12
    tens = {"bound": "tensor", "achieved": round(tf, 2), "peak": tpk, "unit": "TFLOP/s", "frac": round(tf / tpk, 4),
            "peak_kind": "measured bf16 (burst)" if peaks else "fallback", "flops_per_launch": fl}
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        x1, tmax = op.cpu_sample(name, 6.0)
        ts = []
        while sum(ts) < 12.0 and len(ts) < 50:
            ts.append(op.oracle_step(x1, tmax))
        cpu = {"value": tmax * len(ts) / sum(ts) / 1e6, "unit": CHUNK_UNIT, "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"head (0, 0), the first {tmax} of {T} tokens, float64 numpy oracle (its BLAS may thread "
                         f"over the host's cores), {len(ts)} repetitions, {sum(ts):.1f} s"}
    line = {
        "metric": op.metric, "value": round(value, 3), "unit": CHUNK_UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": name, "B": B, "H": H, "T": T, "K": K, "V": V, "chunk": CHUNK, "seed": seed,
                   "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (129 MB) and a 512 MiB write flushes L2 before every call"},
        "roofline": rf, "tensor_roofline": tens, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
        "clocks": with_cycles(clk, ms), "status": status,
    }
    if decode is not None:
        line["decode"] = decode
    return emit(args, line, dist)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=list(gen.WORKLOAD_ORDER) + list(gen.GDN2_WORKLOADS) + list(gen.MLSTM_WORKLOADS))
    ap.add_argument("--nsplit", type=int, default=0, help="lanes per channel (0 = library's choice)")
    ap.add_argument("--groups", type=int, default=0, help="L-groups (0 = library's choice)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the inference-forward, decode and other-op timings after the scan's")
    ap.add_argument("--op", choices=("scan", "conv1d", "dtproj", "gdn2", "mlstm"), default="scan",
                    help="scan: the S6 scan fwd+bwd (default); conv1d: the conv1d + SiLU in front of it; "
                         "dtproj: the dt projection with its softplus; gdn2: the Gated DeltaNet-2 chunkwise forward; "
                         "mlstm: the mLSTM stabilized chunkwise forward")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.op in ("gdn2", "mlstm"):
        op = ChunkOp(args.op)
        if args.workload != DEFAULT_WORKLOAD and args.workload not in op.workloads:
            ap.error(f"--op {args.op} takes one of {sorted(op.workloads)}")
        return run_chunk_reference(args, op) if args.impl == "reference" else run_chunk(args, op)
    if args.workload in gen.GDN2_WORKLOADS or args.workload in gen.MLSTM_WORKLOADS:
        ap.error("a GDN2 or mLSTM workload needs --op gdn2 or --op mlstm")
    w = gen.WORKLOADS[args.workload]
    if args.op == "dtproj":
        return run_dtproj_reference(args, w) if args.impl == "reference" else run_dtproj(args, w)
    if args.op == "conv1d":
        return run_conv_reference(args, w) if args.impl == "reference" else run_conv(args, w)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
