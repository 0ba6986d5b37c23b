"""Benchmark of the attention forward on B300: one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl fa|reference]

A step is one fa_fwd call over the whole batch of the workload (default: bf16,
causal, B=2 H=32 N=8192 d=128, the long-sequence throughput case).  The metric
is attention-forward TFLOP/s counting 4*B*H*N^2*d multiply-add FLOPs, halved for
causal masking, with inputs resident in device memory; the inputs (3 x 134 MB)
exceed the 126 MB L2, so no L2 flush is needed between steps.  The line also
carries:
  * roofline  -- achieved TFLOP/s of the kernel against the measured dense-bf16
                 tensor peak (MEASURED_PEAKS.json), with DRAM traffic per launch
                 from an ncu capture of the same kernel sources (null otherwise);
  * e2e       -- the same metric through the public API with the inputs copied
                 from pinned host memory and O, lse copied back inside each step;
  * cpu_baseline -- the float64 CPU oracle timed on a bounded sample (rank 0, N=1);
  * clocks    -- SM clocks and throttle reasons sampled during the timed region;
  * fwd_bwd   -- forward and backward (recompute) TFLOP/s of the training
                 workload, bf16 causal B=4 H=16 N=4096 d=128 (backward FLOPs
                 10*B*H*N^2*d, halved for causal);
  * configs   -- the other forward workloads (float32 B=1 H=1 N=256 d=64; bf16
                 causal B=4 H=16 N=2048 d=64; the padded x8 stress workload
                 B=8 H=16 N=1024 d=128), each with its roofline fraction;
  * standard  -- standard attention (S and P written to device memory in full)
                 next to the tiled forward on two workloads' shapes;
  * merge     -- the split-key merge, device-memory bound.
With --impl reference the float64 oracle itself is timed (rank 0 only).
Multi-GPU (torchrun): every rank runs its own replica of the workload, no data
exchange; value = all ranks' FLOPs / the slowest rank's time ("weak" scaling).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from online_softmax_14_b300.inputs import WORKLOADS, Workload, make_workload  # noqa: E402

METRIC = "attention fwd TFLOP/s at bf16 (causal halved) and % of B300 dense-BF16 peak"
DEFAULT_WORKLOAD = "bf16_causal_B2_H32_N8192_d128"
BWD_WORKLOAD = "bf16_causal_fwdbwd_B4_H16_N4096_d128"
FALLBACK_BF16_TFLOPS = 1800.0  # used only when MEASURED_PEAKS.json is absent
L2_BYTES = 126 * 1024 * 1024

# DRAM bytes (read + write) per launch of the forward kernel, from an ncu capture
# of that launch, valid only for the forward sources whose digest is recorded
# with it (kernel_src_digest).
NCU_TRAFFIC = {"bf16_causal_B2_H32_N8192_d128": {"bytes": 460500224 + 117432320,
                                                 "src_digest": "b16f9a4f2aba695f",
                                                 "how": "ncu dram__bytes_read.sum + dram__bytes_write.sum, "
                                                        "one launch of this workload"}}
# What the forward kernel is built from: its headers, and the host functions of
# fa_lib.cu that shape its launch (grid and work list).
FWD_HEADERS = ("fwd_tc.cuh", "ptx.cuh", "worklist.cuh", "exp2_poly.cuh")
FWD_HOST_FUNCTIONS = ("fa_status launch_tc(", "const fa::WorkList* work_list(", "int tiles_needed(",
                      "const fa::WorkList* fwd_work_list(")


def _function_text(src: str, head: str) -> str:
    """The text of the C++ function whose definition starts with `head`, up to
    its matching closing brace ('' when absent)."""
    i = src.find(head)
    if i < 0:
        return ""
    j = src.index("{", i)
    depth = 0
    for k in range(j, len(src)):
        depth += {"{": 1, "}": -1}.get(src[k], 0)
        if depth == 0:
            return src[i:k + 1]
    return src[i:]


def flops_per_step(w) -> float:
    f = 4.0 * w.B * w.H * w.N * w.N * w.d
    return f / 2 if w.causal else f


def max_over_ranks(x: float, dist, device) -> float:
    """The largest value of x over all ranks (x itself without a process group):
    a multi-GPU run is timed by its slowest rank."""
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank: float, world: int, ms_max: float) -> float:
    """Throughput of the whole job: every rank's FLOPs over the slowest rank's time."""
    return flops_per_rank * world / (ms_max * 1e-3) / 1e12


def bwd_flops(w) -> float:
    """Five N x N x d products per head (S, dP, dV, dK, dQ), halved for causal."""
    f = 10.0 * w.B * w.H * w.N * w.N * w.d
    return f / 2 if w.causal else f


def kernel_src_digest() -> str:
    """Digest of the sources the forward kernel and its launch are built from."""
    csrc = os.path.join(ROOT, "online_softmax_14_b300", "csrc")
    h = hashlib.sha256()
    for name in FWD_HEADERS:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    with open(os.path.join(csrc, "fa_lib.cu"), encoding="utf-8") as f:
        lib = f.read()
    for head in FWD_HOST_FUNCTIONS:
        h.update(_function_text(lib, head).encode())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"bf16_tflops": FALLBACK_BF16_TFLOPS}, "fallback"


# ------------------------------------------------------------------ clocks --
REASON_BITS = {0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
               0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class ClockSampler:
    """Samples the SM clock and the clock-event (throttle) reasons of one GPU in a
    background thread, through NVML when importable, else an nvidia-smi
    subprocess; only samples taken between mark_start() and mark_end() count."""

    def __init__(self, device_index: int, period_ms: int = 5):
        self.period_ms = period_ms
        self.samples = []  # (monotonic time, sm_mhz, reasons bitmask)
        self.max_mhz = None
        self.t0 = self.t1 = None
        self.error = ""
        props = torch.cuda.get_device_properties(device_index)
        bus = getattr(props, "pci_bus_id", None)
        self.pci = (f"{getattr(props, 'pci_domain_id', 0):08X}:{bus:02X}:{getattr(props, 'pci_device_id', 0):02X}.0"
                    if bus is not None else None)
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        self.index = vis.split(",")[device_index] if vis else str(device_index)
        self.nv = None
        try:
            import pynvml

            pynvml.nvmlInit()
            self.h = (pynvml.nvmlDeviceGetHandleByPciBusId(self.pci) if self.pci
                      else pynvml.nvmlDeviceGetHandleByIndex(int(self.index)))
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.nv = pynvml
        except Exception as e:
            self.error = f"nvml: {e!r}"

    def _nvml_loop(self):
        nv = self.nv
        get_r = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            try:
                self.samples.append((time.monotonic(), nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM),
                                     int(get_r(self.h))))
            except Exception:
                pass
            time.sleep(self.period_ms / 1000)

    def _smi_loop(self):
        import subprocess

        cmd = ["nvidia-smi", "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
               "--format=csv,noheader,nounits", "-lms", str(self.period_ms), "-i", self.pci or self.index]
        try:
            self._proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception as e:
            self.error += f"; nvidia-smi: {e!r}"
            return
        for line in self._proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            try:
                self.max_mhz = float(parts[1])
                self.samples.append((time.monotonic(), float(parts[0]), int(parts[2], 16)))
            except (ValueError, IndexError):
                continue

    def __enter__(self):
        self._stop = threading.Event()
        self._proc = None
        self._t = threading.Thread(target=self._nvml_loop if self.nv else self._smi_loop, daemon=True)
        self._t.start()
        deadline = time.monotonic() + 3.0  # let the first sample arrive
        while not self.samples and time.monotonic() < deadline:
            time.sleep(0.01)
        return self

    def mark_start(self):
        self.t0 = time.monotonic()

    def mark_end(self):
        self.t1 = time.monotonic()

    def __exit__(self, *a):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
        self._t.join(timeout=5)

    def summary(self):
        inside = [s for s in self.samples if self.t0 is not None and self.t0 <= s[0] <= (self.t1 or 1e30)]
        reasons = set()
        for _, _, r in inside:
            for bit, name in REASON_BITS.items():
                if r & bit:
                    reasons.add(name)
        out = {"sm_mhz": statistics.median([s[1] for s in inside]) if inside else None,
               "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons), "samples": len(inside),
               "source": "nvml" if self.nv else "nvidia-smi"}
        if self.error:
            out["note"] = self.error
        return out


# ------------------------------------------------------------ CPU oracle --
def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


def oracle_heads(w, inputs, heads, causal):
    import oracle

    t0 = time.perf_counter()
    for (b, h) in heads:
        sl = slice(b, b + 1)
        kl = None if inputs["kv_len"] is None else [int(inputs["kv_len"][b])]
        oracle.attention_fwd(inputs["q"][sl, h:h + 1], inputs["k"][sl, h:h + 1], inputs["v"][sl, h:h + 1],
                             inputs["scale"], causal=causal, kv_len=kl)
    return time.perf_counter() - t0


def cpu_baseline(w, inputs, budget_s=15.0):
    """The oracle, as it stands, on whole heads of the workload until ~budget_s."""
    per_head = flops_per_step(w) / (w.B * w.H)
    heads, t = [], 0.0
    i = 0
    while t < budget_s and i < w.B * w.H:
        bh = (i * 7) % (w.B * w.H)
        t += oracle_heads(w, inputs, [(bh // w.H, bh % w.H)], w.causal)
        heads.append(bh)
        i += 1
    return {"value": per_head * len(heads) / t / 1e12, "unit": "TFLOP/s", "cores": blas_threads(),
            "kind": "oracle",
            "sample": f"{len(heads)} whole (b,h) heads of {w.name} ({t:.1f} s, float64 NumPy, full N x N scores)"}


# ------------------------------------------------------------------- main --
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--shape", default=None,
                    help="B,H,N,d: a custom bf16 workload instead of --workload (profiling runs)")
    ap.add_argument("--causal", type=int, default=1, help="with --shape: causal mask (1) or not (0)")
    ap.add_argument("--impl", default="fa", choices=["fa", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=10, help="0 skips the end-to-end measurement")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0, help="0 skips the CPU oracle baseline")
    ap.add_argument("--ref-budget-s", type=float, default=120.0,
                    help="--impl reference: approximate wall time of the whole run")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--bwd-steps", type=int, default=20,
                    help="timed steps of the forward + backward workload (0 skips it)")
    ap.add_argument("--merge-steps", type=int, default=20,
                    help="timed steps of the split-key merge (0 skips it)")
    ap.add_argument("--config-steps", type=int, default=20,
                    help="timed steps of each of the other forward workloads (0 skips them)")
    ap.add_argument("--std-steps", type=int, default=3,
                    help="timed steps of standard attention on two workloads' shapes (0 skips it)")
    ap.add_argument("--bwd-shape", default=None,
                    help="B,H,N: a custom causal d=128 forward + backward workload (profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.shape:
        B, H, N, d = (int(x) for x in args.shape.split(","))
        w = Workload(f"bf16_{'causal' if args.causal else 'full'}_B{B}_H{H}_N{N}_d{d}", "bf16", B, H, N, d,
                     bool(args.causal))
    else:
        w = WORKLOADS[args.workload]

    if args.impl == "reference":
        return run_reference(args, w, rank, world)

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import online_softmax_14_b300 as fa

    inputs = make_workload(w, seed=args.seed + rank)
    dev = torch.device("cuda", local)
    q, k, v = (inputs[n].to(dev) for n in ("q", "k", "v"))
    kv = None if inputs["kv_len"] is None else inputs["kv_len"].to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    dt = fa.FA_BF16 if w.dtype == "bf16" else fa.FA_FP32
    stream = torch.cuda.current_stream(dev)

    def step():
        fa.fa_fwd_ex(dt, q, k, v, o, lse, kv, w.B, w.H, w.N, w.d, inputs["scale"], w.causal, stream)

    for _ in range(args.warmup):
        step()
    fa.fa_check_device_error(stream)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        clk.mark_start()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        clk.mark_end()
    if dist:
        dist.barrier()
    fa.fa_check_device_error(stream)
    ms = e0.elapsed_time(e1) / args.steps
    ms_max = max_over_ranks(ms, dist, dev)
    f_step = flops_per_step(w)
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v))
    value = whole_job_tflops(f_step, world, ms_max)
    achieved = f_step / (ms * 1e-3) / 1e12

    # ---- end to end: pinned host inputs -> device -> kernel -> host outputs
    e2e = run_e2e(args, w, inputs, step, q, k, v, kv, o, lse, stream, dev, dist, world, fa) \
        if args.e2e_steps > 0 else None

    peaks, peak_src = measured_peaks()
    peak = float(peaks["bf16_tflops"])
    digest = kernel_src_digest()
    tr = NCU_TRAFFIC.get(w.name)
    traffic = tr["bytes"] if tr and tr["src_digest"] == digest else None
    traffic_how = tr["how"] if traffic is not None else None

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic (seeded N(0,1), see online_softmax_14_b300/inputs.py)",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
                   "seed": args.seed, "inputs_exceed_l2": in_bytes > L2_BYTES, "l2_flush": False,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic, "traffic_source": traffic_how,
                     "peak_source": f"{peak_src} bf16_tflops (burst)", "src_digest": digest},
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
        "gpu": torch.cuda.get_device_name(dev),
    }
    if args.bwd_steps > 0 and not args.shape:
        line["fwd_bwd"] = run_fwd_bwd(args, fa, dev, stream, dist)
    if args.merge_steps > 0 and not args.shape:
        line["merge"] = run_merge(args, fa, w, dev, stream, peaks)
    if args.config_steps > 0 and not args.shape:
        line["configs"] = run_configs(args, fa, dev, stream, peaks)
    if args.std_steps > 0 and not args.shape:
        line["standard"] = run_standard(args, fa, dev, stream, peaks)
    if rank == 0 and world == 1 and args.cpu_budget_s > 0:
        line["cpu_baseline"] = cpu_baseline(w, inputs, args.cpu_budget_s)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def run_fwd_bwd(args, fa, dev, stream, dist):
    """Forward and backward of the training workload (bf16, causal, B=4 H=16
    N=4096 d=128, dO drawn after Q, K, V), each timed over --bwd-steps launches
    with CUDA events on the launching stream.  The backward is one fa_bwd call
    (three kernels: the row preprocess, dK/dV per key tile, dQ per query tile)."""
    w = WORKLOADS[BWD_WORKLOAD]
    if args.bwd_shape:
        B, H, N = (int(x) for x in args.bwd_shape.split(","))
        w = Workload(f"bf16_causal_fwdbwd_B{B}_H{H}_N{N}_d128", "bf16", B, H, N, 128, True, backward=True)
    inp = make_workload(w, seed=args.seed)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    dq = torch.empty(q.shape, dtype=torch.float32, device=dev)
    dk, dv = torch.empty_like(dq), torch.empty_like(dq)
    ws_bytes = fa.fa_bwd_workspace_size(w.B, w.H, w.N, w.d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)

    def fwd():
        fa.fa_fwd(q, k, v, o, lse, w.B, w.H, w.N, w.d, inp["scale"], w.causal, stream)

    def bwd():
        fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, ws_bytes, w.B, w.H, w.N, w.d, inp["scale"], w.causal, stream)

    def timed(fn):
        for _ in range(max(3, args.warmup)):
            fn()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.bwd_steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / args.bwd_steps

    ms_f = timed(fwd)
    ms_b = timed(bwd)
    fa.fa_check_device_error(stream)
    ff, fb = flops_per_step(w), bwd_flops(w)
    return {"workload": w.name, "steps": args.bwd_steps, "fwd_ms": round(ms_f, 4), "bwd_ms": round(ms_b, 4),
            "fwd_tflops": round(ff / ms_f / 1e9, 2), "bwd_tflops": round(fb / ms_b / 1e9, 2),
            "fwd_bwd_tflops": round((ff + fb) / (ms_f + ms_b) / 1e9, 2),
            "flops": {"fwd": ff, "bwd": fb, "bwd_formula": "10*B*H*N^2*d, halved for causal"},
            "gpu_launches_per_bwd": 3}


FP32_FFMA_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12  # 148 SMs x 128 FP32 lanes x 2 FLOP (FMA) x 2.032 GHz


def _time(fn, steps, warmup, stream):
    for _ in range(max(3, warmup)):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def run_configs(args, fa, dev, stream, peaks):
    """The other forward workloads, each timed over --config-steps launches with
    CUDA events on the launching stream, with its roofline fraction: the bf16
    ones against the measured dense-bf16 peak; the float32 one (CUDA cores)
    against the FP32 FMA rate of 148 SMs x 128 lanes x 2 FLOP at 2.032 GHz.  The
    padded stress workload reports the formula FLOPs (4*B*H*N^2*d) and the
    effective ones (4*H*d*N*sum(kv_len), the keys actually visible)."""
    out = {}
    peak = float(peaks["bf16_tflops"])
    for name in ("fp32_B1_H1_N256_d64", "bf16_causal_B4_H16_N2048_d64", "bf16_padded_stress_B8_H16_N1024_d128"):
        w = WORKLOADS[name]
        inp = make_workload(w, seed=args.seed)
        q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
        kv = None if inp["kv_len"] is None else inp["kv_len"].to(dev)
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
        dt = fa.FA_BF16 if w.dtype == "bf16" else fa.FA_FP32

        def step():
            fa.fa_fwd_ex(dt, q, k, v, o, lse, kv, w.B, w.H, w.N, w.d, inp["scale"], w.causal, stream)

        ms = _time(step, args.config_steps, args.warmup, stream)
        fa.fa_check_device_error(stream)
        f = flops_per_step(w)
        tf = f / ms / 1e9
        r = {"ms": round(ms, 5), "tflops": round(tf, 2), "dtype": w.dtype}
        if w.dtype == "bf16":
            r["roofline"] = {"bound": "tensor", "achieved": round(tf, 2), "peak": peak, "unit": "TFLOP/s",
                             "frac": round(tf / peak, 4), "peak_source": "measured bf16_tflops (burst)"}
        else:
            r["roofline"] = {"bound": "alu", "achieved": round(tf, 3), "peak": round(FP32_FFMA_TFLOPS, 1),
                             "unit": "TFLOP/s", "frac": round(tf / FP32_FFMA_TFLOPS, 5),
                             "peak_source": "derived: 148 SMs x 128 FP32 lanes x 2 FLOP x 2.032 GHz"}
        if w.padded:
            eff = 4.0 * w.H * w.d * w.N * float(inp["kv_len"].sum())
            r["effective_tflops"] = round(eff / ms / 1e9, 2)
            r["effective_frac"] = round(eff / ms / 1e9 / peak, 4)
            r["flops"] = {"formula": f, "effective": eff, "note": "effective counts only keys < kv_len[b]"}
        out[name] = r
    return out


def run_standard(args, fa, dev, stream, peaks):
    """Standard attention (fa_std_fwd: S = scale Q K^T written in full as float32,
    P = softmax(S) written as bf16, then O = P V) next to the tiled forward on
    the same inputs, for two workloads' shapes: time of each, the algorithmic
    device-memory bytes of each, and the share of the standard path's bytes that
    are the N x N matrices (the HBM-traffic exercise of the Exercises page)."""
    out = {}
    hbm = float(peaks.get("hbm_gbs", 6400.0))
    for name in ("bf16_causal_B4_H16_N2048_d64", "bf16_causal_B2_H32_N8192_d128"):
        w = WORKLOADS[name]
        inp = make_workload(w, seed=args.seed)
        q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
        nbytes = fa.fa_std_workspace_size(w.B, w.H, w.N)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)

        def std():
            fa.fa_std_fwd(q, k, v, o, lse, None, ws, nbytes, w.B, w.H, w.N, w.d, inp["scale"], w.causal, stream)

        def tiled():
            fa.fa_fwd(q, k, v, o, lse, w.B, w.H, w.N, w.d, inp["scale"], w.causal, stream)

        ms_std = _time(std, args.std_steps, 3, stream)
        ms_tiled = _time(tiled, max(args.std_steps, 10), 3, stream)
        fa.fa_check_device_error(stream)
        bh, n, d = w.B * w.H, w.N, w.d
        io = 4 * bh * n * d * 2 + bh * n * 4           # Q, K, V read; O written; lse written
        quad = bh * n * n * (4 + 4 + 2 + 2)             # S written and read (f32), P written and read (bf16)
        out[name] = {"ms_standard": round(ms_std, 4), "ms_tiled": round(ms_tiled, 4),
                     "speedup_tiled_over_standard": round(ms_std / ms_tiled, 2),
                     "bytes_standard": io + quad, "bytes_tiled": io,
                     "nxn_share_of_standard_bytes": round(quad / (io + quad), 5),
                     "standard_gbs": round((io + quad) / (ms_std * 1e-3) / 1e9, 1),
                     "standard_hbm_frac": round((io + quad) / (ms_std * 1e-3) / 1e9 / hbm, 4),
                     "workspace_bytes": nbytes, "launches_standard": 3, "launches_tiled": 1}
        del ws
        torch.cuda.empty_cache()
    return out


def run_merge(args, fa, w, dev, stream, peaks, n_parts=4):
    """Split-key merge of n_parts bf16 partial results of the workload's shape
    (as a split-key forward over n_parts key ranges would produce them), timed
    with CUDA events on the launching stream.  Device-memory bound: the
    algorithmic bytes are every part's O and lse read once and the merged O and
    lse written once."""
    g = torch.Generator(device="cpu").manual_seed(args.seed)
    R = w.B * w.H * w.N
    o_p = torch.randn(n_parts, w.B, w.H, w.N, w.d, generator=g).to(torch.bfloat16).to(dev)
    l_p = (torch.randn(n_parts, w.B, w.H, w.N, generator=g) * 4).to(dev)
    o = torch.empty(o_p.shape[1:], dtype=torch.bfloat16, device=dev)
    lse = torch.empty(l_p.shape[1:], dtype=torch.float32, device=dev)

    def step():
        fa.fa_merge(fa.FA_BF16, o_p, l_p, n_parts, o, lse, w.B, w.H, w.N, w.d, stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.merge_steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    fa.fa_check_device_error(stream)
    ms = a.elapsed_time(b) / args.merge_steps
    nbytes = n_parts * R * (w.d * 2 + 4) + R * (w.d * 2 + 4)
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak = float(peaks.get("hbm_gbs", 6400.0))
    return {"workload": f"{n_parts} bf16 parts of {w.name}", "steps": args.merge_steps, "ms": round(ms, 4),
            "bytes_per_call": nbytes,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4)}}


def run_e2e(args, w, inputs, step, q, k, v, kv, o, lse, stream, dev, dist, world, fa):
    """Same metric through the public API with host buffers: every step copies
    Q, K, V (and kv_len) from pinned host memory, runs fa_fwd_ex, and copies O
    and lse back to pinned host memory, all inside the timed region.

    The steps are pipelined the way a serving loop would run them: two sets of
    device buffers, the host-to-device copies on one stream, the kernel on the
    launching stream and the device-to-host copies on a third, ordered by
    events, so that step i+1's inputs travel while step i computes and step i-1's
    outputs come back.  The timed region runs from before the first copy-in to
    after the last copy-out."""
    f_step = flops_per_step(w)
    hq, hk, hv = (inputs[n].pin_memory() for n in ("q", "k", "v"))
    ho = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
    hl = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho[0].numel() * ho[0].element_size() + hl[0].numel() * hl[0].element_size()
    hkv = None
    if kv is not None:
        hkv = inputs["kv_len"].pin_memory()
        h2d += hkv.numel() * hkv.element_size()
    # buffer set 0 is the bench's own tensors; set 1 is a second copy
    dq = [q, torch.empty_like(q)]
    dk = [k, torch.empty_like(k)]
    dv = [v, torch.empty_like(v)]
    dkv = [kv, None if kv is None else torch.empty_like(kv)]
    do = [o, torch.empty_like(o)]
    dl = [lse, torch.empty_like(lse)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    dt = fa.FA_BF16 if w.dtype == "bf16" else fa.FA_FP32

    def run(n_steps):
        copied = [None, None]    # event: inputs of the set are on the device
        computed = [None, None]  # event: the kernel using the set has finished
        returned = [None, None]  # event: the outputs of the set are back on the host
        for i in range(n_steps):
            b = i & 1
            with torch.cuda.stream(s_in):
                if computed[b] is not None:
                    s_in.wait_event(computed[b])        # the kernel of step i-2 no longer reads set b
                dq[b].copy_(hq, non_blocking=True)
                dk[b].copy_(hk, non_blocking=True)
                dv[b].copy_(hv, non_blocking=True)
                if hkv is not None:
                    dkv[b].copy_(hkv, non_blocking=True)
                copied[b] = torch.cuda.Event()
                copied[b].record(s_in)
            stream.wait_event(copied[b])
            if returned[b] is not None:
                stream.wait_event(returned[b])          # step i-2's outputs have left set b
            fa.fa_fwd_ex(dt, dq[b], dk[b], dv[b], do[b], dl[b], dkv[b], w.B, w.H, w.N, w.d, inputs["scale"],
                         w.causal, stream)
            computed[b] = torch.cuda.Event()
            computed[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(computed[b])
                ho[b].copy_(do[b], non_blocking=True)
                hl[b].copy_(dl[b], non_blocking=True)
                returned[b] = torch.cuda.Event()
                returned[b].record(s_out)
        return returned

    run(2)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(s_in)
    with torch.cuda.stream(s_in):
        returned = run(args.e2e_steps)
    for ev in returned:
        if ev is not None:
            s_out.wait_event(ev)
    e3.record(s_out)
    torch.cuda.synchronize()
    fa.fa_check_device_error(stream)
    ms_e2e = e2.elapsed_time(e3) / args.e2e_steps
    ms_e2e = max_over_ranks(ms_e2e, dist, dev)
    e2e_value = whole_job_tflops(f_step, world, ms_e2e)
    return {"value": round(e2e_value, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(ms_e2e, 3),
            "pipelining": "two device buffer sets; copy-in, kernel and copy-out on three streams"}


def run_reference(args, w, rank, world):
    """The float64 CPU oracle on the host cores (rank 0 only).

    Each step evaluates the oracle, as it stands, on a bounded sample of the
    workload: the first R query rows of one (b, h) head (heads cycled), through
    the oracle's ordinary whole-matrix path.  Under the causal mask those rows see
    only keys < R, so the leading R x R block is exactly the first R rows of the
    full problem; without it they see every key.  R is calibrated so that the
    whole --warmup + --steps run takes about --ref-budget-s seconds.  FLOPs are
    counted for the rows sampled, 4 * d * (visible keys) per row: the GPU
    metric's unit.
    """
    if rank != 0:
        return
    import oracle

    inputs = make_workload(w, seed=args.seed)
    kl = None if inputs["kv_len"] is None else [int(x) for x in inputs["kv_len"]]

    def visible(b, i):
        n = w.N if kl is None else min(w.N, kl[b])
        return min(n, i + 1) if w.causal else n

    def one_step(n_rows, k):
        bh = (k * 7) % (w.B * w.H)
        b, h = bh // w.H, bh % w.H
        nk = n_rows if w.causal else w.N
        sl = (slice(b, b + 1), slice(h, h + 1))
        t0 = time.perf_counter()
        oracle.attention_fwd(inputs["q"][sl][:, :, :n_rows], inputs["k"][sl][:, :, :nk], inputs["v"][sl][:, :, :nk],
                             inputs["scale"], causal=w.causal, kv_len=None if kl is None else [kl[b]])
        dt = time.perf_counter() - t0
        return dt, sum(4.0 * w.d * visible(b, i) for i in range(n_rows))

    r0 = min(512, w.N)
    t_cal, _ = one_step(r0, 0)
    per_step_s = args.ref_budget_s / (args.steps + args.warmup)
    grow = per_step_s / max(t_cal, 1e-6)
    n_rows = int(r0 * (grow ** 0.5 if w.causal else grow))  # the work grows as R^2 (causal) or R
    n_rows = max(64, min(w.N, n_rows))
    for k in range(args.warmup):
        one_step(n_rows, k + 1)
    t_tot, f_tot = 0.0, 0.0
    for k in range(args.steps):
        dt, fl = one_step(n_rows, args.warmup + 1 + k)
        t_tot += dt
        f_tot += fl
    value = f_tot / t_tot / 1e12
    cores = blas_threads()
    sample = (f"the first {n_rows} query rows of one (b,h) head of {w.name} per step (heads cycled), "
              f"float64 NumPy oracle with the full score block materialised")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_tot / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1))",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


if __name__ == "__main__":
    main()
