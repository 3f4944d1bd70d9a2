"""Benchmark of the chunkwise GLA forward pass on GB300.

Workload: the GLA layer shaped like the 1.3B model, B=8, H=4, T=2048,
dk=256, dv=512, bf16 q/k/v, fp32 per-key log gate logsigmoid(N(0,1))/16,
S0 ~ 0.02 N(0,1); synthetic seeded inputs (no dataset exists for this).

One step = one whole forward pass (every stage of the plan) over one batch.
`value` is tokens/s over all ranks with inputs resident in HBM and L2
flushed between steps (a write then a read of buffers larger than L2, so
each step starts cold and no dirty flush lines are written back inside
it); `e2e` is the same metric through the C call gla_fwd_host, which takes
pinned host buffers and copies the inputs in and O, S_T back inside the
timed region (in slices of the batch that overlap copies and compute). With N > 1 ranks each rank runs its own
replica batch (the path shards over (b, h) with no exchange): weak scaling.

`--impl reference` times the fp64 CPU oracle on this machine's host cores
on a bounded sample of the same workload (it is the only other
implementation of this method available here).
"""
from __future__ import annotations

import argparse
import platform
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "gla_1p3b"
METRIC = "GLA fwd tokens/s and TFLOP/s (fraction of GB300 bf16 peak) at B=8,T=2048,dk256,dv512"
FALLBACK_HBM = 6800.0
FALLBACK_BF16 = 1900.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=WORKLOAD,
                    help="workload to time (default: the 1.3B-shaped GLA layer the metric is quoted on)")
    ap.add_argument("--segments", type=int, default=0, help="force the sequence split (0: planner decides)")
    ap.add_argument("--shape", default="", help="B,H,T,dk,dv: the workload's gate and dtype at another shape")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--direction", default="fwd", choices=["fwd", "bwd"],
                    help="bwd: time the backward pass (gla_bwd) instead and print its own line")
    ap.add_argument("--cpu-sample-rows", type=int, default=8,
                    help="batch rows of the workload the oracle runs for cpu_baseline")
    ap.add_argument("--ref-sample-rows", type=int, default=1,
                    help="batch rows per step of the reference arm")
    ap.add_argument("--other-workloads", default="linear_attn,scalar_decay,gla_long",
                    help="bf16 configurations also timed (same discipline) and reported inside the line "
                         "under config.other_workloads; empty: none")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM, FALLBACK_BF16, 1700.0, "fallback"


def workload(args):
    from chunkwise_gated_linear_gla_gb300 import inputs as gi
    w = gi.WORKLOADS[args.workload]
    if args.shape:
        B, H, T, dk, dv = (int(x) for x in args.shape.split(","))
        w = w.with_(name=f"{w.name}@{args.shape}", B=B, H=H, T=T, dk=dk, dv=dv)
    return w


def algorithmic(w):
    """Algorithmic FLOPs and bytes of one forward pass of workload w (per rank).

    FLOPs per token per head: 4 dk dv (state update + inter-chunk term) +
    (C+1)(dk+dv) (causal intra-chunk scores and their product with V).
    Bytes: q, k, v read and O written once (e bytes each element), the fp32
    log gate read once (dk values per token per head for the per-key gate, one for
    the per-token scalar gate, dk + dv for the bilinear gate), S0 read and S_T
    written once (fp32).
    """
    import torch
    e = 2 if w.dtype == torch.bfloat16 else 4
    BH, T, dk, dv, C = w.B * w.H, w.T, w.dk, w.dv, w.chunk
    gate_bytes = 4 * dk if w.gate == 2 else 4 if w.gate == 3 else 4 * (dk + dv) if w.gate == 4 else 0
    flops = BH * T * (4 * dk * dv + (C + 1) * (dk + dv))
    byts = BH * T * (e * (2 * dk + dv) + e * dv + gate_bytes) + BH * dk * dv * 4 * (2 if w.s0_std > 0 else 1)
    return flops, byts


def stage_bytes(w, name, split=None):
    """Compulsory bytes one launch of a stage moves (each operand once, bf16 tiles).

    Qt/Kt (Q (.) Lambda, K (.) Gamma) exist only with a gate; without one the
    chunk pass reads q and k directly. S0/S_T are counted when present. `split` is
    planned_split's (nseg, cps, sub, st_nseg, st_cps) of a sequence split.
    """
    nseg, _, _, st_nseg, st_cps = split or (1, 0, 1, 0, 0)
    BH, T, dk, dv, C = w.B * w.H, w.T, w.dk, w.dv, w.chunk
    nch = (T + C - 1) // C
    Tp = nch * C
    gated = w.gate != 0
    gate_in = T * dk * 4 if w.gate in (2, 4) else T * 4 if w.gate == 3 else 0
    bil = w.gate == 4
    s0 = BH * dk * dv * 4 if w.s0_std > 0 else 0
    st = BH * dk * dv * 4
    qk_tiles = (Tp if gated else T) * dk * 2 * 2
    gam = nch * dk * 4 if gated else 0
    if name == "gla_chunk_fused":
        # the whole pass in one kernel: q, k, v, the log gate read once, O written once, S0 / S_T
        return algorithmic(w)[1]
    sc = scores_in_chunk_pass(w)
    if name == "gla_chunk_prep":
        # per-head decay with dk <= 128: chunks whose decay stays within e^-60 (every chunk of the
        # workloads' lambda_h) leave Q (.) Lambda and their scores to the chunk pass, so the prep
        # reads only k and writes only K (.) Gamma
        if sc:
            return BH * (T * dk * 2 + Tp * dk * 2 + gam)
        return BH * (T * dk * 2 * 2 + gate_in + (Tp * dk * 2 * 2 if gated else 0) + nch * C * C * 2 + gam)
    if dk == 512 and name in ("gla_chunk_fwd", "gla_chunk_fwd_keys_hi"):
        # two chunk passes over key halves: each reads its half of Q (.) Lambda, K (.) Gamma, gamma,
        # S0 and writes its half of S_T; the first reads the scores and writes O as an fp32
        # partial, the second reads that partial and writes O
        half = BH * ((Tp * 256 * 2 * 2) + nch * 256 * 4 + T * dv * 2) + (s0 + st) // 2
        if name == "gla_chunk_fwd":
            return half + BH * (nch * C * C * 2 + T * dv * 4)
        return half + BH * (T * dv * 4 + T * dv * 2)
    if name == "gla_chunk_fwd":
        # split: each segment reads its start state, the last one writes S_T
        last_state = (s0 + st) if nseg == 1 else BH * nseg * dk * dv * 4 + st
        # bilinear gate: V (.) D' in place of v, plus log beta and the chunks' column decays
        bil_in = T * dv * 4 + nch * dv * 4 if bil else 0
        scores = 0 if sc else nch * C * C * 2   # formed in the pass (dk <= 128, no gate or per-head decay)
        return BH * (qk_tiles + scores + gam + T * dv * 2 * 2 + bil_in) + last_state
    if name == "gla_value_prep":
        return BH * (T * dv * (2 + 4 + 2) + nch * dv * 4)
    # the split's state pass covers the chunks before the last segment, in st_nseg pieces
    covered = st_nseg * st_cps
    if name == "gla_chunk_state":
        return BH * covered * (C * dk * 2 + C * dv * 2 + (dk * 4 if gated else 0)) + BH * st_nseg * dk * dv * 4
    if name == "gla_state_scan":
        return BH * (2 * st_nseg + 1) * dk * dv * 4 + s0 + BH * covered * dk * 4 * (1 if gated else 0)
    return 0


def scores_in_chunk_pass(w):
    """Whether the chunk pass forms the intra-chunk scores itself (same rule as csrc/gla_api.cu):
    dk <= 128 with no gate or a per-head decay (whose chunks all keep the query factor out at
    the workloads' decays)."""
    return w.dk <= 128 and w.gate in (0, 1) and "bfloat16" in str(w.dtype)


def planned_split(w, force, sms, state_ctas_per_sm=1, min_state_chunks=4):
    """The sequence split the library's planner picks (same rule as csrc/gla_api.cu):
    (segments per (b,h), chunks per segment, state-pass pieces per segment, state-pass
    pieces per (b,h), chunks per piece)."""
    nch = (w.T + w.chunk - 1) // w.chunk
    units = w.B * w.H * (w.dv // 128)
    if force > 0:
        n = min(force, nch)
    elif units * 2 > sms or nch < 16:
        n = 1
    else:
        n = max(1, min(sms // units, nch // 8))
    cps = (nch + n - 1) // n
    n = (nch + cps - 1) // cps
    if n == 1:
        return 1, cps, 1, 0, 0
    sub = 1
    for f in range(cps // min_state_chunks, 1, -1):
        if cps % f == 0 and (n - 1) * f * units <= sms * state_ctas_per_sm:
            sub = f
            break
    return n, cps, sub, (n - 1) * sub, cps // sub


def planned_segments(w, force, sms):
    """Segments per (b,h) the library's planner picks."""
    return planned_split(w, force, sms)[0]


def kernel_source_sha(name):
    files = {"gla_chunk_fused": ["gla_fused.cu", "sm100.cuh"],
             "gla_chunk_fwd": ["gla_chunk_fwd.cu", "sm100.cuh"],
             "gla_chunk_fwd_keys_hi": ["gla_chunk_fwd.cu", "sm100.cuh"],
             "gla_chunk_prep": ["gla_prep.cu", "sm100.cuh"],
             "gla_chunk_state": ["gla_state.cu", "sm100.cuh"],
             "gla_state_scan": ["gla_scan.cu"],
             "gla_value_prep": ["gla_vprep.cu"],
             "gla_bwd_state_sweep": ["gla_chunk_fwd.cu", "sm100.cuh"],
             "gla_bwd_dstate_sweep": ["gla_chunk_fwd.cu", "sm100.cuh"],
             "gla_bwd_boundary": ["gla_bwd_chunk.cu"],
             "gla_bwd_grads": ["gla_bwd_chunk.cu", "sm100.cuh"],
             "gla_bwd_gate_tail": ["gla_bwd.cu", "gla_bwd_chunk.cu"]}.get(name, [])
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "chunkwise_gated_linear_gla_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload, name, direction="fwd"):
    """DRAM bytes per launch of kernel `name` on `workload` (the backward's under
    "<workload>/bwd") from the committed ncu summary, if one was captured for that pair and the
    kernel's source still matches it."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            d = json.load(f)[workload if direction == "fwd" else f"{workload}/bwd"][name]
        if d.get("source_sha") != kernel_source_sha(name):
            return None
        return float(d["dram_bytes_per_launch"])
    except Exception:
        return None


class Clocks:
    """nvidia-smi sampling (200 ms) during the timed region."""

    FIELDS = "index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active," \
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown," \
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap"

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        sm.sort()
        med = sm[len(sm) // 2] if sm else None
        return {"sm_mhz": med, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(x, dist=None, device=None):
    """Largest value of x over all ranks (the job's time is its slowest rank's)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank, world, step_ms):
    """Whole-job throughput: every rank processes its own batch (weak scaling)."""
    return tokens_per_rank * world / (step_ms * 1e-3)


def run_reference(args, w):
    """The oracle (fp64 recurrence, C, all host cores) on a bounded sample of the workload."""
    import oracle
    from chunkwise_gated_linear_gla_gb300 import inputs as gi
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    oracle.build()
    rows = args.ref_sample_rows
    ws = w.with_(B=rows)
    x = gi.make_inputs(ws, seed=0)
    cores = oracle.default_threads()
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"], nthreads=cores,
                           log_b=x.get("log_b"))
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    tok = rows * w.T
    mean = sum(times) / len(times)
    value = tok / mean
    sample = f"{rows} of {w.B} batch rows (all {w.H} heads, T={w.T}) per step, {cpu_model()}"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{w.name} B={w.B} H={w.H} T={w.T} dk={w.dk} dv={w.dv}", "sample": sample},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def cpu_model():
    """The host CPU's name as /proc/cpuinfo gives it (Arm kernels give implementer/part codes)."""
    try:
        info = open("/proc/cpuinfo").read()
    except OSError:
        return platform.machine()
    for key in ("model name", "Model", "Hardware"):
        for line in info.splitlines():
            if line.startswith(key) and ":" in line:
                return line.split(":", 1)[1].strip()
    # Arm kernels name no model: map the (implementer, part) codes of common server cores
    arm = {("0x41", "0xd0c"): "Arm Neoverse N1", ("0x41", "0xd40"): "Arm Neoverse V1",
           ("0x41", "0xd49"): "Arm Neoverse N2", ("0x41", "0xd4f"): "Arm Neoverse V2"}
    get = lambda key: sorted({line.split(":", 1)[1].strip() for line in info.splitlines()
                              if line.startswith(key) and ":" in line})
    impl, part = get("CPU implementer"), get("CPU part")
    if len(impl) == 1 and len(part) == 1 and (impl[0], part[0]) in arm:
        return f"{arm[(impl[0], part[0])]} ({platform.machine()})"
    codes = impl + part
    return f"{platform.machine()} ({', '.join(codes)})" if codes else platform.machine()


def cpu_one_core(w):
    """Oracle tokens/s on one thread, from one head of one batch row (T capped at 2048),
    scaled to whole tokens (all H heads) so it compares with the all-core figure."""
    import oracle
    from chunkwise_gated_linear_gla_gb300 import inputs as gi
    ws = w.with_(B=1, H=1, T=min(w.T, 2048))
    x = gi.make_inputs(ws, seed=0)
    if x["gate"] == gi.GATE_HEAD_SCALAR:
        x["log_g"] = x["log_g"][:1]
    t0 = time.perf_counter()
    oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"], nthreads=1, log_b=x.get("log_b"))
    dt = time.perf_counter() - t0
    return ws.T / dt / w.H, f"1 head x T={ws.T}, {dt:.2f} s"


def cpu_baseline(w, rows):
    import oracle
    from chunkwise_gated_linear_gla_gb300 import inputs as gi
    oracle.build()
    x = gi.make_inputs(w.with_(B=rows), seed=0)
    cores = oracle.default_threads()
    # repeat the sample until about 10 s of CPU work has been timed (at most 40 passes)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"], nthreads=cores,
                           log_b=x.get("log_b"))
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= 10.0 or reps >= 40:
            break
    one, one_sample = cpu_one_core(w)
    return {"value": reps * rows * w.T / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{rows} of {w.B} batch rows (all {w.H} heads, T={w.T}) x {reps} passes, {dt:.1f} s",
            "cpu_model": cpu_model(), "value_1core": one, "sample_1core": one_sample}


# fp32 FFMA peak from the nominal unit counts: 152 SMs x 128 fp32 lanes x 2 FLOP x 2.07 GHz
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
BWD_METRIC = "GLA bwd tokens/s at B=8,T=2048,dk256,dv512 (gradients of q, k, v, log_g, S0)"


def bwd_chunk_form(w):
    """Whether gla_bwd takes its 64-row chunk form (tcgen05) for workload w."""
    from chunkwise_gated_linear_gla_gb300 import inputs as gi
    return (w.dtype != torch_f32() and w.dk in (128, 256) and w.dv % 128 == 0 and w.T > 0
            and w.gate != gi.GATE_BILINEAR)


def torch_f32():
    import torch
    return torch.float32


def algorithmic_bwd(w):
    """FLOPs of the backward per token per head. The chunk form (C = 64): 10 dk dv (the two
    state sweeps' updates and the dv, dk and dq products with the chunk states) +
    2 C (2 dv + 3 dk) (the scores, dO V^T, and A^T dO, dA K, dA^T Q within the chunk). The
    16-row forms (C = 16): 10 dk dv + 2 (C + 1)(dk + dv)."""
    if bwd_chunk_form(w):
        C = 64
        return w.B * w.H * w.T * (10 * w.dk * w.dv + 2 * C * (2 * w.dv + 3 * w.dk))
    C = 16
    return w.B * w.H * w.T * (10 * w.dk * w.dv + 2 * (C + 1) * (w.dk + w.dv))


def bwd_segments(w, sms):
    """The chunk form's sequence split of its two sweeps (the library's rule)."""
    nch = -(-w.T // 64)
    units = w.B * w.H * (w.dv // 128)
    if units * 2 > sms or nch < 16:
        return 1
    n = max(1, min(sms // units, nch // 8))
    cps = -(-nch // n)
    return -(-nch // cps)


def bwd_stage_bytes(w, name, glog=True, dst=True, s0=True, nseg=1):
    """Compulsory DRAM bytes of one launch of a chunk-form stage: what it must read and write
    once (inputs, the workspace tensors it consumes and produces, its outputs)."""
    from chunkwise_gated_linear_gla_gb300 import inputs as gi
    BH, T, dk, dv = w.B * w.H, w.T, w.dk, w.dv
    nch = -(-T // 64)
    Tp = nch * 64
    gated = w.gate != gi.GATE_NONE
    lg = {gi.GATE_PER_KEY: T * dk * 4, gi.GATE_TOKEN_SCALAR: T * 4}.get(w.gate, 0)
    st = dk * dv * 4
    if name == "gla_chunk_prep":
        b = 2 * T * dk * 2 + lg + nch * 64 * 64 * 2 + nch * dk * 4 + (2 * Tp * dk * 2 if gated else 0)
    elif name == "gla_bwd_state_sweep":
        b = T * dk * 2 + T * dv * 2 + nch * dk * 4 + nch * dv * dk * 2 + (st if s0 else 0) + (st if glog and dst else 0)
    elif name == "gla_bwd_dstate_sweep":
        b = T * dk * 2 + T * dv * 2 + nch * dk * 4 + nch * dv * dk * 2 + (st if dst else 0) + st
    elif name in ("gla_chunk_state", "gla_chunk_dstate"):
        b = T * dk * 2 + T * dv * 2 + nch * dk * 4 + nseg * st
    elif name in ("gla_state_scan", "gla_dstate_scan"):
        b = 2 * nseg * st + nch * dk * 4 + (st if (s0 if name == "gla_state_scan" else dst) else 0)
    elif name == "gla_bwd_boundary":
        b = 2 * st + dk * 4
    elif name == "gla_bwd_grads":
        b = (2 * nch * dv * dk * 2 + 2 * T * dv * 2 + 2 * Tp * dk * 2 + nch * 64 * 64 * 2 + nch * dk * 4 + lg
             + 2 * T * dk * 4 + T * dv * 4 + ((T * dk * 4 + nch * dk * 4) if glog else 0))
    elif name == "gla_bwd_gate_tail":
        b = 2 * T * dk * 4 + 4 * nch * dk * 4
    else:
        return None
    return BH * b


def run_backward(args, w):
    """Times gla_bwd (inputs resident in HBM, L2 flushed between steps) and prints one line.
    A step is the whole backward (its stages back to back through gla_bwd_stage, events only
    before and after); the per-stage breakdown comes from as many further steps with an event
    between stages."""
    import torch
    from chunkwise_gated_linear_gla_gb300 import binding as bnd
    from chunkwise_gated_linear_gla_gb300 import build as gbuild
    from chunkwise_gated_linear_gla_gb300 import inputs as gi
    torch.cuda.set_device(0)
    gbuild.build()
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        oracle.build()
        ws_ = w.with_(B=1, H=1, T=min(w.T, 512))
        xs = gi.make_inputs(ws_, seed=0)
        if xs["gate"] == gi.GATE_HEAD_SCALAR:
            xs["log_g"] = xs["log_g"][:1]
        dOs = torch.randn((1, 1, ws_.T, w.dv)).to(w.dtype)
        cores = oracle.default_threads()
        t0 = time.perf_counter()
        oracle.gla_backward(xs["q"], xs["k"], xs["v"], xs["log_g"], xs["gate"], xs["S0"], dOs, None, nthreads=cores,
                            log_b=xs.get("log_b"))
        dt = time.perf_counter() - t0
        cpu = {"value": ws_.T / dt / w.H, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": f"1 head x T={ws_.T} (one (b,h) job runs on one thread), {dt:.2f} s, {cpu_model()}"}
    x = gi.make_inputs(w, seed=0)
    dev = torch.device("cuda", 0)
    c = lambda t: None if t is None else t.to(dev)
    q, k, v, g, S0 = c(x["q"]), c(x["k"]), c(x["v"]), c(x["log_g"]), c(x["S0"])
    gen = torch.Generator().manual_seed(1)
    dO = torch.randn((w.B, w.H, w.T, w.dv), generator=gen).to(w.dtype).to(dev)
    dST = (torch.randn((w.B, w.H, w.dk, w.dv), generator=gen) * 0.1).to(dev)
    f32 = lambda *shape: torch.empty(shape, dtype=torch.float32, device=dev)
    dq, dk, dv = f32(w.B, w.H, w.T, w.dk), f32(w.B, w.H, w.T, w.dk), f32(w.B, w.H, w.T, w.dv)
    dg = None if g is None else torch.empty(g.shape, dtype=torch.float32, device=dev)
    dS0 = f32(w.B, w.H, w.dk, w.dv)
    lb = c(x.get("log_b"))
    db = None if lb is None else f32(w.B, w.H, w.T, w.dv)
    p = bnd.make_bwd_params(q, k, v, g, S0, dO, dST, dq, dk, dv, dg, dS0, gate=x["gate"], log_b=lb, dlog_b=db)
    nbytes = bnd.gla_bwd_workspace_size(p)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    p.workspace, p.workspace_bytes = ws.data_ptr(), nbytes
    nst = bnd.gla_bwd_num_stages(p)
    names = [bnd.gla_bwd_stage_name(p, i) for i in range(nst)]
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    clean = torch.zeros(64 * 1024 * 1024, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(evs=None):
        for i in range(nst):
            if evs is not None:
                evs[i].record(stream)
            bnd.gla_bwd_stage(p, i, stream)
        if evs is not None:
            evs[nst].record(stream)

    for _ in range(args.warmup):
        flush.zero_(); clean.sum()
        step()
    torch.cuda.synchronize()
    if bnd.gla_device_status(stream) != 0:
        raise SystemExit("device status error after warm-up")
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = Clocks(0)
    clocks.start()
    torch.cuda.synchronize()
    for a, b in pairs:
        flush.zero_(); clean.sum()
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    staged = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(args.steps)]
    for evs in staged:
        flush.zero_(); clean.sum()
        step(evs)
    torch.cuda.synchronize()
    if bnd.gla_device_status(stream) != 0:
        raise SystemExit("device status error in timed region")
    times = sorted(a.elapsed_time(b) for a, b in pairs)
    ms = sum(times) / len(times)
    stage_ms = [sum(e[i].elapsed_time(e[i + 1]) for e in staged) / len(staged) for i in range(nst)]
    flops = algorithmic_bwd(w)
    tflops = flops / (ms * 1e-3) / 1e12
    hbm, bf16_burst, _, src = peaks()
    dom = max(range(nst), key=lambda i: stage_ms[i])
    if bwd_chunk_form(w):
        glog, dst_ = g is not None, True
        nseg = bwd_segments(w, torch.cuda.get_device_properties(dev).multi_processor_count)
        per_kernel = []
        for n_, t_ in zip(names, stage_ms):
            b_ = bwd_stage_bytes(w, n_, glog=glog, dst=dst_, s0=S0 is not None, nseg=nseg)
            per_kernel.append({"kernel": n_, "ms": t_, "compulsory_bytes": b_,
                               "compulsory_gbs": b_ / (t_ * 1e-3) / 1e9, "dram_bytes_ncu": ncu_traffic(w.name, n_, "bwd")})
        dk_ = per_kernel[dom]
        roof = {"kernel": dk_["kernel"], "bound": "hbm", "achieved": dk_["compulsory_gbs"], "peak": hbm, "unit": "GB/s",
                "frac": dk_["compulsory_gbs"] / hbm, "traffic": dk_["dram_bytes_ncu"],
                "peak_source": f"{src} HBM copy bandwidth", "bytes_per_launch": dk_["compulsory_bytes"],
                "bytes_basis": "compulsory bytes of the kernel: its inputs, the workspace tensors it reads and "
                               "writes, its outputs, each once", "kernels": per_kernel,
                "pass_gbs": sum(k_["compulsory_bytes"] for k_ in per_kernel) / (ms * 1e-3) / 1e9}
        kind = "chunk form: 64-row chunks on tcgen05, bf16 operands, fp32 accumulation"
        launches_per_step = nst + (1 if "gla_bwd_gate_tail" in names else 0) + (
            1 if w.gate in (gi.GATE_TOKEN_SCALAR, gi.GATE_HEAD_SCALAR) else 0)
    elif w.dtype == torch.bfloat16 and w.dk in (64, 128, 256) and w.gate != gi.GATE_BILINEAR:
        roof = {"kernel": "gla_bwd (split form: 16-row chunks, mma.sync on hi + lo bf16 operands)", "bound": "tensor",
                "achieved": tflops, "peak": bf16_burst, "unit": "TFLOP/s", "frac": tflops / bf16_burst,
                "traffic": None, "peak_source": f"{src} dense bf16 (burst: the pass is timed alone)"}
        kind = "split form"
        launches_per_step = 4 + (1 if w.gate in (gi.GATE_TOKEN_SCALAR, gi.GATE_HEAD_SCALAR) else 0) - (
            1 if w.gate == 0 else 0)
    else:
        roof = {"kernel": "gla_bwd (CUDA cores, all stages)", "bound": "alu", "achieved": tflops,
                "peak": FP32_ALU_TFLOPS, "unit": "TFLOP/s", "frac": tflops / FP32_ALU_TFLOPS, "traffic": None,
                "peak_source": "nominal fp32 FFMA rate: 152 SMs x 128 lanes x 2 FLOP x 2.07 GHz"}
        kind = "CUDA-core form"
        launches_per_step = 4 + (1 if w.gate in (gi.GATE_TOKEN_SCALAR, gi.GATE_HEAD_SCALAR) else 0) - (
            1 if w.gate == 0 else 0)
    line = {
        "metric": BWD_METRIC, "value": w.B * w.T / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32" if w.dtype == torch.float32 else "bf16 in, f32 arithmetic",
        "data": "synthetic (seeded inputs of the workload; dO ~ N(0,1), dST ~ 0.1 N(0,1))",
        "config": {"workload": f"{w.name} backward: B={w.B} H={w.H} T={w.T} dk={w.dk} dv={w.dv}, "
                               f"gate={['none', 'per-head scalar', 'per-key', 'per-token scalar', 'bilinear'][w.gate]}",
                   "form": kind, "stages": names, "stage_ms": stage_ms,
                   "sweep_segments": nseg if bwd_chunk_form(w) else None,
                   "l2": "flushed between steps (256 MB write then 256 MB read, outside the timed events)",
                   "workspace_bytes": nbytes},
        "tflops": tflops, "tflops_frac_bf16_peak": tflops / bf16_burst,
        "roofline": roof,
        "timing": {"mean_ms": ms, "median_ms": times[len(times) // 2], "min_ms": times[0],
                   "note": "mean is the value's basis: whole passes, events only before and after each; "
                           "stage_ms comes from as many further steps with an event between stages"},
        "cpu_baseline": cpu,
        "e2e": None,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def time_plan(bnd, p, steps, warmup, stream, flush_l2, record_clocks=None):
    """Times the plan of params p with CUDA events on `stream`: `warmup` untimed steps,
    then `steps` timed ones, L2 flushed before each (outside the events). A step is the
    whole pass as gla_fwd_ex runs it (its stages back to back, nothing recorded between
    them, so a stage may start while the one before finishes); the per-stage breakdown
    comes from as many further steps with an event between stages. Returns (stage names,
    mean ms per stage, mean ms per step, sorted per-step ms, clocks)."""
    import torch
    nst = bnd.gla_fwd_num_stages(p)
    names = [bnd.gla_fwd_stage_name(p, i) for i in range(nst)]

    def step(evs=None):
        for i in range(nst):
            if evs is not None:
                evs[i].record(stream)
            bnd.gla_fwd_stage(p, i, stream)
        if evs is not None:
            evs[nst].record(stream)

    def whole(e0, e1):
        e0.record(stream)
        for i in range(nst):
            bnd.gla_fwd_stage(p, i, stream)
        e1.record(stream)

    for _ in range(warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    if bnd.gla_device_status(stream) != 0:
        raise SystemExit("device status error after warm-up")
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    if record_clocks:
        record_clocks.start()
    torch.cuda.synchronize()
    for s in range(steps):
        flush_l2()
        whole(*pairs[s])
    torch.cuda.synchronize()
    clk = record_clocks.stop() if record_clocks else None
    if bnd.gla_device_status(stream) != 0:
        raise SystemExit("device status error in timed region")
    per = sorted(a.elapsed_time(b) for a, b in pairs)
    evsets = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(steps)]
    for s in range(steps):
        flush_l2()
        step(evsets[s])
    torch.cuda.synchronize()
    if bnd.gla_device_status(stream) != 0:
        raise SystemExit("device status error in the stage-by-stage steps")
    stage_ms = [sum(e[i].elapsed_time(e[i + 1]) for e in evsets) / steps for i in range(nst)]
    return names, stage_ms, sum(per) / steps, per, clk


def other_workloads(bnd, gi, names_csv, args, dev, stream, flush_l2, hbm):
    """The other bf16 configurations, timed like the headline one and summarised."""
    import torch
    out = {}
    for name in [n for n in names_csv.split(",") if n]:
        w = gi.WORKLOADS[name]
        x = gi.make_inputs(w, seed=0)
        c = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
        O = torch.empty((w.B, w.H, w.T, w.dv), dtype=w.dtype, device=dev)
        ST = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device=dev)
        p = bnd.make_params(c["q"], c["k"], c["v"], c["log_g"], c["S0"], O, ST, gate=x["gate"])
        nb = bnd.gla_fwd_workspace_size(p)
        ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=dev)
        p.workspace, p.workspace_bytes = ws.data_ptr(), nb
        names, stage_ms, ms, per, _ = time_plan(bnd, p, min(args.steps, 20), max(3, min(args.warmup, 5)),
                                               stream, flush_l2)
        flops, byts = algorithmic(w)
        out[name] = {"shape": f"B={w.B} H={w.H} T={w.T} dk={w.dk} dv={w.dv}",
                     "gate": ["none", "per-head scalar", "per-key", "per-token scalar", "bilinear"][w.gate],
                     "ms_per_step": ms, "median_ms": per[len(per) // 2],
                     "tokens_per_s": w.B * w.T / (ms * 1e-3),
                     "tflops": flops / (ms * 1e-3) / 1e12,
                     "algorithmic_bytes": byts, "path_frac_hbm": byts / (ms * 1e-3) / 1e9 / hbm,
                     "stages": names, "stage_ms": stage_ms, "workspace_bytes": nb}
        del c, O, ST, ws, p
        torch.cuda.empty_cache()
    return out


def main():
    args = parse()
    from chunkwise_gated_linear_gla_gb300 import inputs as gi
    w = workload(args)
    if args.impl == "reference":
        run_reference(args, w)
        return
    if args.direction == "bwd":
        run_backward(args, w)
        return

    import torch
    import torch.distributed as dist
    import chunkwise_gated_linear_gla_gb300 as gla
    from chunkwise_gated_linear_gla_gb300 import binding as bnd
    from chunkwise_gated_linear_gla_gb300 import build as gbuild

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0:
        gbuild.build()
    if world > 1:
        dist.barrier()
    bnd.load()

    # CPU baseline first (before any GPU work of this process is in flight)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_sample_rows)

    x = gi.make_inputs(w, seed=rank)
    dev = torch.device("cuda", local)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    g = None if x["log_g"] is None else x["log_g"].to(dev)
    lb = None if x.get("log_b") is None else x["log_b"].to(dev)
    S0 = None if x["S0"] is None else x["S0"].to(dev)
    O = torch.empty((w.B, w.H, w.T, w.dv), dtype=w.dtype, device=dev)
    ST = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device=dev)
    p = bnd.make_params(q, k, v, g, S0, O, ST, force_segments=args.segments, log_b=lb)
    nbytes = bnd.gla_fwd_workspace_size(p)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    p.workspace, p.workspace_bytes = ws.data_ptr(), nbytes
    nst = bnd.gla_fwd_num_stages(p)
    names = [bnd.gla_fwd_stage_name(p, i) for i in range(nst)]
    # L2 flush between steps: a 256 MB write (> 129 MB of L2), then a 256 MB read of
    # another buffer, so the flush's own dirty lines are written back before the timed
    # events start and every step begins from a clean, cold L2
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    clean = torch.zeros(64 * 1024 * 1024, dtype=torch.int32, device=dev)

    def flush_l2():
        flush.zero_()
        clean.sum()
    stream = torch.cuda.current_stream(dev)

    def step(evs=None):
        for i in range(nst):
            if evs is not None:
                evs[i].record(stream)
            bnd.gla_fwd_stage(p, i, stream)
        if evs is not None:
            evs[nst].record(stream)

    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    if bnd.gla_device_status(stream) != 0:
        raise SystemExit("device status error after warm-up")

    # The timed steps: each the whole pass as gla_fwd_ex runs it, its stages back to back
    # with nothing recorded between them (a stage may start while the one before finishes),
    # an event before and after.
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = Clocks(torch.cuda.current_device()) if rank == 0 else None
    if clocks:
        clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for s in range(args.steps):
        flush_l2()
        pairs[s][0].record(stream)
        step()
        pairs[s][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    if bnd.gla_device_status(stream) != 0:
        raise SystemExit("device status error in timed region")
    per_step = sorted(a.elapsed_time(b) for a, b in pairs)
    step_ms = sum(per_step) / args.steps
    step_ms = max_over_ranks(step_ms, dist, dev)
    # the per-stage breakdown: as many further steps, an event between stages
    evsets = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(args.steps)]
    for s in range(args.steps):
        flush_l2()
        step(evsets[s])
    torch.cuda.synchronize()
    if bnd.gla_device_status(stream) != 0:
        raise SystemExit("device status error in the stage-by-stage steps")
    stage_ms = [sum(evs[i].elapsed_time(evs[i + 1]) for evs in evsets) / args.steps for i in range(nst)]

    # the same steps back to back without the flush (inputs partly in L2 from the step before)
    uevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in uevs:
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    unflushed = sorted(a.elapsed_time(b) for a, b in uevs)

    # end to end through gla_fwd_host: pinned host tensors in, host tensors out; the
    # library slices the batch so that copies in, compute and copies out overlap
    hx = {n: (None if x.get(n) is None else x[n].pin_memory()) for n in ("q", "k", "v", "log_g", "log_b", "S0")}
    hO = torch.empty(O.shape, dtype=O.dtype).pin_memory()
    hST = torch.empty(ST.shape, dtype=ST.dtype).pin_memory()
    hp = bnd.make_params(hx["q"], hx["k"], hx["v"], hx["log_g"], hx["S0"], hO, hST,
                         force_segments=args.segments, log_b=hx["log_b"])
    h2d = sum(t.numel() * t.element_size() for t in hx.values() if t is not None)
    d2h = hO.numel() * hO.element_size() + hST.numel() * hST.element_size()

    def e2e_step():
        bnd.gla_fwd_host(hp, 0, stream)

    for _ in range(max(2, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    # the host result must be the device result (slices may plan their own sequence
    # split, which changes the rounding, not the function)
    for got, ref in ((hO, O), (hST, ST)):
        r = ref.float().cpu()
        if not torch.isfinite(got.float()).all() or \
                float((got.float() - r).norm()) > 5e-3 * max(float(r.norm()), 1e-30):
            raise SystemExit("gla_fwd_host result differs from the device-path result")

    hbm, bf16, bf16_sus, src = peaks()
    others = None
    if rank == 0 and world == 1 and args.other_workloads and w.name == WORKLOAD and not args.shape:
        others = other_workloads(bnd, gi, args.other_workloads, args, dev, stream, flush_l2, hbm)
    # the same workload through the fused path (one kernel, no workspace), where it applies
    fused = None
    if rank == 0 and world == 1 and args.segments == 0:
        pf = bnd.make_params(q, k, v, g, S0, O, ST, log_b=lb, path=bnd.GLA_PATH_FUSED)
        if bnd.gla_fwd_num_stages(pf) == 1:
            fnames, fstage, fms, fper, _ = time_plan(bnd, pf, min(args.steps, 20), max(3, min(args.warmup, 5)),
                                                     stream, flush_l2)
            fused = {"path": "GLA_PATH_FUSED", "stages": fnames, "ms_per_step": fms,
                     "median_ms": fper[len(fper) // 2], "tokens_per_s": w.B * w.T / (fms * 1e-3),
                     "path_frac_hbm": algorithmic(w)[1] / (fms * 1e-3) / 1e9 / hbm, "workspace_bytes": 0,
                     "note": "opt-in path: the gate prep inside the chunk pass, shared by a cluster of the "
                             "head's dv-tile CTAs through distributed shared memory; not the value's basis"}
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    flops, byts = algorithmic(w)
    tokens = w.B * w.T * world
    value = job_tokens_per_s(w.B * w.T, world, step_ms)
    tflops = flops * world / (step_ms * 1e-3) / 1e12
    dom = max(range(nst), key=lambda i: stage_ms[i])
    dname = names[dom]
    split = planned_split(w, args.segments, torch.cuda.get_device_properties(dev).multi_processor_count) \
        if "gla_chunk_state" in names else None
    nseg = split[0] if split else 1
    if dname == "gla_fwd_simt":
        # the CUDA-core pass: fp32 FFMA work against the nominal FFMA rate
        alu = flops / (stage_ms[dom] * 1e-3) / 1e12
        roof = {"kernel": dname, "bound": "alu", "achieved": alu, "peak": FP32_ALU_TFLOPS, "unit": "TFLOP/s",
                "frac": alu / FP32_ALU_TFLOPS, "traffic": None,
                "peak_source": "nominal fp32 FFMA rate: 152 SMs x 128 lanes x 2 FLOP x 2.07 GHz",
                "flops_per_launch": flops}
    else:
        # achieved = the method's algorithmic bytes (q, k, v, log gate in; O out; S0 in, S_T out)
        # over the time of the kernels that move them: the one launch of a one-kernel plan, the
        # whole step otherwise (each kernel's own compulsory bytes are listed separately)
        span_ms = stage_ms[0] if nst == 1 else step_ms
        ach = byts / (span_ms * 1e-3) / 1e9
        per_kernel = [{"kernel": n, "ms": t, "compulsory_bytes": stage_bytes(w, n, split),
                       "compulsory_gbs": stage_bytes(w, n, split) / (t * 1e-3) / 1e9,
                       "dram_bytes_ncu": ncu_traffic(w.name, n)} for n, t in zip(names, stage_ms)]
        tr = [k["dram_bytes_ncu"] for k in per_kernel]
        traffic = sum(tr) if tr and all(t is not None for t in tr) else None
        roof = {"kernel": names[0] if nst == 1 else "+".join(names), "bound": "hbm", "achieved": ach,
                "peak": hbm, "unit": "GB/s", "frac": ach / hbm, "traffic": traffic,
                "traffic_over_algorithmic": None if traffic is None else traffic / byts,
                "peak_source": src, "bytes_per_launch": byts,
                "bytes_basis": "algorithmic: q, k, v, log gate read once, O written once, S0 read, S_T written",
                "kernels": per_kernel}
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == torch.bfloat16 else "f32",
        "data": "synthetic (seeded, shapes and distributions of the workload)",
        "config": {"workload": f"{w.name}: {w.notes}, B={w.B} H={w.H} T={w.T} dk={w.dk} dv={w.dv} chunk=64, "
                               f"gate={['none', 'per-head scalar', 'per-key', 'per-token scalar', 'bilinear'][w.gate]}, "
                               f"S0={'given' if w.s0_std > 0 else 'zero'}",
                   "B": w.B, "H": w.H, "T": w.T, "dk": w.dk, "dv": w.dv, "segments": nseg,
                   "state_pieces": split[3] if split else 0,
                   "l2": "flushed between steps (256 MB write then 256 MB read, outside the timed events)",
                   "stages": names, "stage_ms": stage_ms, "other_workloads": others, "fused_path": fused},
        "tflops": tflops, "tflops_frac_bf16_peak": tflops / bf16,
        "path_gbs": byts * world / (step_ms * 1e-3) / 1e9, "path_frac_hbm": byts / (step_ms * 1e-3) / 1e9 / hbm,
        "roofline": roof,
        "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "timing": {"mean_ms": step_ms, "median_ms": per_step[len(per_step) // 2], "min_ms": per_step[0],
                   "unflushed_median_ms": unflushed[len(unflushed) // 2],
                   "note": "mean is the value's basis: whole passes, events only before and after each; "
                           "stage_ms comes from as many further steps with an event between stages; "
                           "unflushed = the same steps back to back, no L2 flush"},
        "gpu_launches": nst * args.steps,
        "clocks": clk,
    }
    if cpu:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
