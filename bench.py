#!/usr/bin/env python3
"""Benchmark of the FP8 linear-layer hot path on one B300 (or N replicas).

One step = one pass of the whole path over one batch of synthetic input, for
every linear of the workload and every scaling mode it uses:
  block mode:      token-group quantize of A, block quantize of W, GEMM
  per-tensor mode: per-tensor quantize of A and of W, GEMM
  per_channel (opt-in with --modes): per-tensor quantize of A, per-channel
                   (one scale per output row) quantize of W, GEMM
  block_fp8w / fused_fp8w (weights held in FP8, quantized once before any
                   timing, as a model's weights are at load time): per
                   linear the token-group quantize of A and the GEMM, or
                   the fused linear alone
  per_tensor_static (delayed scaling, opt-in with --modes): A quantized with
                   the scale held from earlier steps while its amax goes
                   into a ring of HIST_LEN slots, per-tensor quantize of W,
                   GEMM, then the next scale from the ring (after the GEMM,
                   which still needs the scale A was quantized with)
The two quantizations of a linear are independent: A's runs on a forked
stream while W's runs on the main one, and the GEMM follows both (the
fork and join are events inside the captured graph).
`value` is the step's GEMM FLOPs divided by the step time (TFLOP/s), inputs
resident in HBM.  L2 is defeated by rotating over enough copies of the
inputs that consecutive uses of one copy are more than 2x the L2 size apart.

Timed regions (CUDA events on the launching stream, synchronize + barrier on
both sides, max over ranks):
  step region:   exactly K steps, replayed as CUDA graphs of many steps so
                 host launch cost never paces the GPU.
  kernel region: every kernel of the step alone, min(K, 2048) back-to-back
                 launches (rotating input sets) in one CUDA graph between two
                 events; these per-launch durations feed `roofline` and
                 `kernels`.
  e2e region:    K steps (capped to ~2 s) through the public API with host
                 buffers: per step, H2D of A and W from pinned memory, the
                 path, D2H of C; consecutive steps overlap their uploads,
                 compute and read-backs on three streams.

`--impl reference` times the CPU oracle (the plain C reference of the same
path) on the host cores, on a bounded sample of the same workload: every
quantizer in full and the first rows of each GEMM (ORACLE_SAMPLE_FLOP in
all), extrapolated to all rows; the median over the sampled steps.  The GPU
arm's `cpu_baseline` times the same sample (median of 3 after one warm-up).

The default workload is the largest one (16384x8192 outlier activations
times an 8192x8192 weight, block-scaled).
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "FP8 scaled-GEMM TFLOP/s & % of dense FP8 peak; quantize GB/s & % of HBM peak"
DEFAULT_WORKLOAD = "outlier_16384x8192x8192"   # the largest workload: the block-scaled GEMM at scale
L2_BYTES_DEFAULT = 126 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
FP8_OVER_BF16 = 2.0  # nominal dense FP8 / BF16 tensor throughput ratio (4.5 / 2.25 PFLOP/s)
HIST_LEN = 16        # amax-history ring of the delayed-scaling mode
HIST_MARGIN = 0      # the recipe's margin (DelayedScaling(margin=0, interval=4))
MODES = ("block", "per_tensor", "per_tensor_static", "per_channel", "block_ue8m0", "fused", "block_fp8w", "fused_fp8w")
# Modes whose weights are held in FP8: quantized once when the buffers are
# set up (a model's weights are quantized at load time and stored in FP8),
# so a step is the per-token work only: the activation's token-group
# quantization and the GEMM, or the fused linear alone.
FP8W_MODES = ("block_fp8w", "fused_fp8w")
# A plain run prints one line per entry, the headline (the largest workload,
# block-scaled with FP32 scales) last: a decode batch of one token through
# the unfused and the fused linear (weights held in FP8), and the headline
# shape with power-of-two (UE8M0) scales on the tensor core's block-scaled
# MMA.
DEFAULT_LINES = (("llama2_7b_m1", "block_fp8w,fused_fp8w"), (DEFAULT_WORKLOAD, "block_ue8m0"), (DEFAULT_WORKLOAD, ""))


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=None,
                   help="one workload (default: the decode and UE8M0 lines, then the headline workload)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=0, help="0: same as --steps, capped to ~2 s")
    p.add_argument("--modes", default="",
                   help="override the workload's scaling modes: block, per_tensor, per_channel, "
                        "per_tensor_static, block_ue8m0, fused (comma list)")
    p.add_argument("--profile", type=int, default=0,
                   help="run N eager steps on one input set and exit (a small command for ncu captures)")
    a = p.parse_args()
    a.warmup = max(a.warmup, 3)
    return a


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def max_over_ranks(x, world, device):
    """The largest x over all ranks, returned on every rank (the slowest
    rank's time is the job's time); x itself when there is one rank."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world, flops_per_step, step_ms):
    """Whole-job TFLOP/s of `world` replicas that each ran one step of
    flops_per_step in step_ms (already the maximum over ranks)."""
    return world * flops_per_step / (step_ms * 1e-3) / 1e12


def workload_of(args):
    """The named synthetic workload, with --modes overriding its scaling modes."""
    import dataclasses

    import synth
    wl = synth.WORKLOADS[args.workload]
    if args.modes:
        modes = tuple(args.modes.split(","))
        bad = [m for m in modes if m not in MODES]
        if bad:
            raise SystemExit(f"unknown scaling mode(s) {bad}")
        wl = dataclasses.replace(wl, modes=modes)
    return wl


def config_of(args, wl):
    """The `config` object of the JSON line, identical in both arms."""
    return {"workload": args.workload, "description": wl.description,
            "linears": [[lin.name, lin.M, lin.N, lin.K] for lin in wl.linears], "modes": list(wl.modes),
            "in_dtype": wl.in_dtype, "out_dtype": wl.out_dtype,
            "l2": "defeated: the GPU arm rotates over enough input sets that consecutive uses of one set are "
                  "more than 2x the L2 size apart",
            "parallelism": f"replicas x{args.gpus}" if args.gpus > 1 else "single GPU"}


# ------------------------------------------------------------ algorithmic work
def kernel_plan(wl):
    """[(linear, mode, [(kernel name, bound, bytes, flops)])] of one step."""
    plan = []
    for lin in wl.linears:
        M, N, K = lin.M, lin.N, lin.K
        for mode in wl.modes:
            nb, kbn = (N + 127) // 128, K // 128
            if mode == "block_ue8m0":
                ks = [("quant_token_group_ue8m0", "hbm", M * K * 3 + M * kbn, 0),
                      ("quant_weight_block_ue8m0", "hbm", N * K * 3 + nb * kbn, 0),
                      ("gemm_block_ue8m0", None, M * K + N * K + M * kbn + nb * kbn + 2 * M * N, 2 * M * N * K)]
            elif mode == "fused":
                # the activation is read once in 16 bits and quantized inside the GEMM
                ks = [("quant_weight_block", "hbm", N * K * 3 + 4 * nb * kbn, 0),
                      ("linear_fused", None, M * K * 2 + N * K + 4 * nb * kbn + 2 * M * N, 2 * M * N * K)]
            elif mode == "block_fp8w":
                ks = [("quant_token_group", "hbm", M * K * 3 + 4 * M * kbn, 0),
                      ("gemm_block", None, M * K + N * K + 4 * M * kbn + 4 * nb * kbn + 2 * M * N, 2 * M * N * K)]
            elif mode == "fused_fp8w":
                ks = [("linear_fused", None, M * K * 2 + N * K + 4 * nb * kbn + 2 * M * N, 2 * M * N * K)]
            elif mode == "block":
                ks = [("quant_token_group", "hbm", M * K * 3 + 4 * M * (K // 128), 0),
                      ("quant_weight_block", "hbm", N * K * 3 + 4 * ((N + 127) // 128) * (K // 128), 0),
                      ("gemm_block", None, M * K + N * K + 4 * M * (K // 128) + 4 * ((N + 127) // 128) * (K // 128)
                       + 2 * M * N, 2 * M * N * K)]
            elif mode == "per_channel":
                ks = [("quant_per_tensor_act", "hbm", M * K * 3 + 4, 0),
                      ("quant_per_channel_weight", "hbm", N * K * 3 + 4 * N, 0),
                      ("gemm_per_channel", None, M * K + N * K + 4 + 4 * N + 2 * M * N, 2 * M * N * K)]
            elif mode == "per_tensor_static":
                ks = [("quant_static_act", "hbm", M * K * 3 + 8, 0),
                      ("quant_per_tensor_weight", "hbm", N * K * 3 + 4, 0),
                      ("gemm_per_tensor", None, M * K + N * K + 8 + 2 * M * N, 2 * M * N * K),
                      ("scale_from_history", "hbm", 4 * HIST_LEN + 4, 0)]
            else:
                ks = [("quant_per_tensor_act", "hbm", M * K * 3 + 4, 0),
                      ("quant_per_tensor_weight", "hbm", N * K * 3 + 4, 0),
                      ("gemm_per_tensor", None, M * K + N * K + 8 + 2 * M * N, 2 * M * N * K)]
            plan.append((lin, mode, ks))
    return plan


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {k: float(pk[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash():
    csrc = os.path.join(ROOT, "fp8_scaled_gemm_02_b300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if taken on the
    current kernel sources for this workload; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    ent = rec.get(workload, {}).get(kernel)
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks
THROTTLE_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                 0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x2: "applications_clocks_setting",
                 0x10: "sync_boost"}


class ClockSampler(threading.Thread):
    """Samples SM clock, max clock and throttle reasons every ~10 ms through
    NVML, or every 100 ms through `nvidia-smi -lms` when NVML is unusable."""

    def __init__(self, device_index):
        super().__init__(daemon=True)
        self.samples = []   # (host time, sm MHz, max MHz, reasons bitmask)
        self.stop_flag = threading.Event()
        self.ok = False
        self.source = None
        self.err = None
        self.max_mhz = None
        self.bus = None
        try:
            import torch
            props = torch.cuda.get_device_properties(device_index)
            self.bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
        except Exception:
            pass
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = (pynvml.nvmlDeviceGetHandleByPciBusId(self.bus.encode()) if self.bus
                      else pynvml.nvmlDeviceGetHandleByIndex(device_index))
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.ok, self.source = True, "nvml"
        except Exception as e:
            self.err = f"nvml: {e!r}"
            self.ok, self.source = True, "nvidia-smi"

    def run(self):
        if self.source == "nvml":
            nv = self.nv
            while not self.stop_flag.is_set():
                try:
                    sm = nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM)
                    try:
                        rs = nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
                    except Exception:
                        rs = nv.nvmlDeviceGetCurrentClocksThrottleReasons(self.h)
                    self.samples.append((time.perf_counter(), sm, self.max_mhz, int(rs)))
                except Exception:
                    pass
                time.sleep(0.01)
            return
        cmd = ["nvidia-smi", "--query-gpu=pci.bus_id,clocks.sm,clocks.max.sm,clocks_event_reasons.active",
               "--format=csv,noheader,nounits", "-lms", "50"]
        try:
            proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception as e:
            self.ok = False
            self.err = (self.err or "") + f"; nvidia-smi: {e!r}"
            return
        try:
            for line in proc.stdout:
                if self.stop_flag.is_set():
                    break
                f = [x.strip() for x in line.split(",")]
                if len(f) < 4:
                    continue
                if self.bus and f[0].lower()[-len("00:00.0"):] != self.bus.lower()[-len("00:00.0"):]:
                    continue
                try:
                    self.max_mhz = float(f[2])
                    self.samples.append((time.perf_counter(), float(f[1]), float(f[2]), int(f[3], 16)))
                except ValueError:
                    pass
        finally:
            proc.terminate()

    def summary(self, t0, t1, t_wide0):
        base = {"source": self.source}
        if self.err:
            base["note"] = self.err
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], **base}
        win = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed"
        if len(win) < 3:
            win = [s for s in self.samples if t_wide0 <= s[0] <= t1]
            window = "spinup+warmup+timed"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0, **base}
        reasons = set()
        for s in win:
            for bit, name in THROTTLE_BITS.items():
                if s[3] & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(s[1] for s in win), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(win), "window": window, **base}


# --------------------------------------------------------------- our path
def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import synth
    import fp8_scaled_gemm_02_b300 as F

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=dev)

    wl = workload_of(args)
    plan = kernel_plan(wl)
    td = {"f16": torch.float16, "bf16": torch.bfloat16}
    in_t, out_t = td[wl.in_dtype], td[wl.out_dtype]

    # host inputs (seeded, synthetic) and one device buffer set per rotation
    host_a, host_w = {}, {}
    for lin in wl.linears:
        if lin.K not in host_a:
            host_a[lin.K] = synth.activation(wl, lin)
        host_w[lin.name] = synth.weight(wl, lin)

    def to_t(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(in_t)

    set_bytes = 0
    for lin, mode, _ in plan:
        M, N, K = lin.M, lin.N, lin.K
        set_bytes += (M * K + N * K) * 3 + M * N * 2 + 4 * (M * K // 128 + N * K // 128 + 8)
    l2 = L2_BYTES_DEFAULT
    try:
        l2 = torch.cuda.get_device_properties(local).L2_cache_size or l2
    except Exception:
        pass
    R = max(2, math.ceil(2 * l2 / set_bytes) + 1)
    R = min(R, max(2, int(40e9 // set_bytes)))
    if args.profile:
        R = 1

    sets = []
    for r in range(R):
        bufs = {"a": {k: to_t(v).to(dev) for k, v in host_a.items()},
                "w": {k: to_t(v).to(dev) for k, v in host_w.items()}, "lin": []}
        for lin, mode, _ in plan:
            M, N, K = lin.M, lin.N, lin.K
            b = {"qa": torch.empty((M, K), dtype=torch.uint8, device=dev),
                 "qw": torch.empty((N, K), dtype=torch.uint8, device=dev),
                 "c": torch.empty((M, N), dtype=out_t, device=dev)}
            if mode in ("block", "fused", "block_fp8w", "fused_fp8w"):
                b["sa"] = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
                b["sw"] = torch.empty(((N + 127) // 128, K // 128), dtype=torch.float32, device=dev)
            elif mode == "block_ue8m0":
                b["sa"] = torch.empty((K // 128, M), dtype=torch.uint8, device=dev)
                b["sw"] = torch.empty(((N + 127) // 128, K // 128), dtype=torch.uint8, device=dev)
            else:
                b["sa"] = torch.empty(4, dtype=torch.float32, device=dev)[:1]
                b["sw"] = torch.empty(4, dtype=torch.float32, device=dev)[:1]
            if mode == "per_channel":
                b["sw"] = torch.empty(N, dtype=torch.float32, device=dev)
            if mode in FP8W_MODES:
                # the weight, quantized once (load time), outside every timed region
                F.fp8_quantize_weight_block(bufs["w"][lin.name], q=b["qw"], sb=b["sw"])
            if mode == "per_tensor_static":
                # the held scale starts at the activation's own (calibrated) scale
                F.fp8_quantize_per_tensor(bufs["a"][lin.K], q=b["qa"], scale=b["sa"])
                b["hist"] = torch.zeros(HIST_LEN, dtype=torch.float32, device=dev)
            bufs["lin"].append(b)
        sets.append(bufs)

    def linear_calls(r):
        """Per linear of the step for rotation set r: (activation quantize,
        weight quantize, GEMM, [calls after the GEMM]) as zero-argument
        callables, in the order of `plan`."""
        groups = []
        s = sets[r]
        for (lin, mode, ks), b in zip(plan, s["lin"]):
            a = s["a"][lin.K]
            w = s["w"][lin.name]
            post = []
            if mode == "fused":
                ca = None
                cw = lambda w=w, b=b: F.fp8_quantize_weight_block(w, q=b["qw"], sb=b["sw"])
                cg = lambda a=a, b=b: F.fp8_linear_token_group(a, b["qw"], b["sw"], c=b["c"])
            elif mode == "fused_fp8w":
                ca, cw = None, None
                cg = lambda a=a, b=b: F.fp8_linear_token_group(a, b["qw"], b["sw"], c=b["c"])
            elif mode == "block_fp8w":
                ca = lambda a=a, b=b: F.fp8_quantize_token_group(a, q=b["qa"], sa=b["sa"])
                cw = None
                cg = lambda b=b: F.fp8_gemm_scaled(b["qa"], b["sa"], b["qw"], b["sw"], out_dtype=out_t,
                                                   mode="block", c=b["c"])
            elif mode == "block_ue8m0":
                ca = lambda a=a, b=b: F.fp8_quantize_token_group_ue8m0(a, q=b["qa"], sa=b["sa"])
                cw = lambda w=w, b=b: F.fp8_quantize_weight_block_ue8m0(w, q=b["qw"], sb=b["sw"])
                cg = lambda b=b: F.fp8_gemm_scaled(b["qa"], b["sa"], b["qw"], b["sw"], out_dtype=out_t,
                                                   mode="block_ue8m0", c=b["c"])
            elif mode == "block":
                ca = lambda a=a, b=b: F.fp8_quantize_token_group(a, q=b["qa"], sa=b["sa"])
                cw = lambda w=w, b=b: F.fp8_quantize_weight_block(w, q=b["qw"], sb=b["sw"])
                cg = lambda b=b: F.fp8_gemm_scaled(b["qa"], b["sa"], b["qw"], b["sw"], out_dtype=out_t,
                                                   mode="block", c=b["c"])
            elif mode == "per_channel":
                ca = lambda a=a, b=b: F.fp8_quantize_per_tensor(a, q=b["qa"], scale=b["sa"])
                cw = lambda w=w, b=b: F.fp8_quantize_per_channel(w, q=b["qw"], sb=b["sw"])
                cg = lambda b=b: F.fp8_gemm_scaled(b["qa"], b["sa"], b["qw"], b["sw"], out_dtype=out_t,
                                                   mode="per_channel", c=b["c"])
            else:
                if mode == "per_tensor_static":
                    slot = r % HIST_LEN
                    ca = lambda a=a, b=b, slot=slot: F.fp8_quantize_per_tensor_static(
                        a, b["sa"], q=b["qa"], amax=b["hist"][slot:slot + 1])
                    post = [lambda b=b: F.fp8_scale_from_amax_history(b["hist"], HIST_MARGIN, scale=b["sa"])]
                else:
                    ca = lambda a=a, b=b: F.fp8_quantize_per_tensor(a, q=b["qa"], scale=b["sa"])
                cw = lambda w=w, b=b: F.fp8_quantize_per_tensor(w, q=b["qw"], scale=b["sw"])
                cg = lambda b=b: F.fp8_gemm_scaled(b["qa"], b["sa"], b["qw"], b["sw"], out_dtype=out_t,
                                                   mode="per_tensor", c=b["c"])
            groups.append((ca, cw, cg, post))
        return groups

    def kernel_calls(r):
        """The step's kernels for rotation set r, as zero-argument callables
        (the order of the kernels in `plan`)."""
        return [c for ca, cw, cg, post in linear_calls(r) for c in (ca, cw, cg, *post) if c is not None]

    side = torch.cuda.Stream(device=dev)

    def run_step(r, main):
        """One step on stream `main`: per linear, the activation is quantized
        on a forked stream while the weight is quantized on `main` (the two
        are independent), then the GEMM runs on `main` after both, followed
        by the linear's post-GEMM calls (the delayed-scaling update)."""
        for ca, cw, cg, post in linear_calls(r):
            if ca is None or cw is None:   # fused, or weights held in FP8: one chain on `main`
                for c in (ca, cw, cg, *post):
                    if c is not None:
                        c()
                continue
            ev_fork = torch.cuda.Event()
            ev_fork.record(main)
            side.wait_event(ev_fork)
            with torch.cuda.stream(side):
                ca()
            cw()
            ev_join = torch.cuda.Event()
            ev_join.record(side)
            main.wait_event(ev_join)
            cg()
            for c in post:
                c()

    kinfo = [k for _, _, ks in plan for k in ks]
    # the static quantizer launches a one-thread kernel that zeroes its amax slot, then the cast kernel
    launches_per_kernel = [2 if k[0] == "quant_static_act" else 1 for k in kinfo]

    # eager warm-up (sets kernel attributes, fills the descriptor cache)
    for r in range(R):
        for c in kernel_calls(r):
            c()
    torch.cuda.synchronize()
    assert F.fp8s_device_error() == 0

    if args.profile:
        for _ in range(args.profile - 1):
            for c in kernel_calls(0):
                c()
        torch.cuda.synchronize()
        assert F.fp8s_device_error() == 0
        if rank == 0:
            print(json.dumps({"profile_steps": args.profile, "workload": args.workload, "modes": list(wl.modes),
                              "kernels_per_step": len(kinfo)}))
        return

    # CUDA graphs.  Host launch cost must never pace the GPU, so each timed
    # region is one or a few graph launches:
    #   step region:   a graph of C consecutive steps (C a multiple of R),
    #                  replayed K // C times, plus a graph of the K % C rest;
    #   kernel region: per kernel of the step, one graph of Kk = min(K, 2048)
    #                  back-to-back launches of that kernel alone.
    stream = torch.cuda.Stream(device=dev)
    nk = len(kinfo)

    def capture(steps, only=None):
        """Graph of `steps` consecutive steps (rotating input sets); with
        `only` = j, just kernel j of each step (back to back on one stream)."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(steps):
                if only is None:
                    run_step(i % R, stream)
                else:
                    kernel_calls(i % R)[only]()
        return g

    K, W = args.steps, args.warmup
    C = min(K, max(R, (256 // R) * R))
    Kk = min(K, 2048)
    with torch.cuda.stream(stream):
        g_one = capture(1)
        g_chunk = capture(C)
        g_rest = capture(K % C) if K % C else None
        g_kern = [capture(Kk, only=j) for j in range(nk)]
    torch.cuda.synchronize()

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()

    def rank_max(x):
        return max_over_ranks(x, world, dev)

    sampler = ClockSampler(local)
    if sampler.ok:
        sampler.start()
    t_wide0 = time.perf_counter()
    with torch.cuda.stream(stream):
        # spin-up: ~0.3 s of steps so clocks settle and the sampler sees load
        t_end = time.perf_counter() + 0.3
        while time.perf_counter() < t_end:
            g_chunk.replay()
            stream.synchronize()
        for i in range(W):
            g_one.replay()
        barrier()

        # ---- step region: exactly K steps
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        ev0.record(stream)
        for _ in range(K // C):
            g_chunk.replay()
        if g_rest is not None:
            g_rest.replay()
        ev1.record(stream)
        barrier()
        t1 = time.perf_counter()
        step_ms = rank_max(ev0.elapsed_time(ev1)) / K

        # ---- kernel region: each kernel alone, Kk back-to-back launches
        kern_ms = []
        for j in range(nk):
            g_kern[j].replay()   # untimed pass
            barrier()
            ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ea.record(stream)
            g_kern[j].replay()
            eb.record(stream)
            barrier()
            kern_ms.append(rank_max(ea.elapsed_time(eb)) / Kk)
        kregion_step_ms = sum(kern_ms)
    sampler.stop_flag.set()
    assert F.fp8s_device_error() == 0, "a kernel's bounded wait expired during the benchmark"

    # ---- e2e region: public API with host buffers
    e2e = None
    if not args.no_e2e:
        pin_a = {k: to_t(v).pin_memory() for k, v in host_a.items()}
        pin_w = {k: to_t(v).pin_memory() for k, v in host_w.items()}
        # one pinned output buffer per linear and input set, so that the
        # read-back of step i never shares host memory with that of step i+1
        pin_c = [[torch.empty((lin.M, lin.N), dtype=out_t).pin_memory() for lin, _, _ in plan] for _ in range(R)]
        if all(m in FP8W_MODES for m in wl.modes):
            pin_w = {}   # weights held in FP8 on the device: a step uploads activations only
        h2d = sum(t.numel() * 2 for t in pin_a.values()) + sum(t.numel() * 2 for t in pin_w.values())
        d2h = sum(t.numel() * 2 for t in pin_c[0])
        up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev_in = [torch.cuda.Event() for _ in range(R)]      # set r's inputs have landed
        ev_done = [torch.cuda.Event() for _ in range(R)]    # set r's step has finished
        ev_out = [torch.cuda.Event() for _ in range(R)]     # set r's outputs have been read back
        used = [False] * R

        def e2e_step(i):
            """Step i on input set r = i % R, pipelined over three streams: the
            upload of step i+1 and the read-back of step i-1 overlap the
            compute of step i.  A set is re-uploaded only after its previous
            step finished, and recomputed only after its previous outputs
            were read back."""
            r = i % R
            s = sets[r]
            if used[r]:
                up.wait_event(ev_done[r])
            with torch.cuda.stream(up):
                for k, t in pin_a.items():
                    s["a"][k].copy_(t, non_blocking=True)
                for k, t in pin_w.items():
                    s["w"][k].copy_(t, non_blocking=True)
                ev_in[r].record(up)
            stream.wait_event(ev_in[r])
            if used[r]:
                stream.wait_event(ev_out[r])
            run_step(r, stream)
            ev_done[r].record(stream)
            down.wait_event(ev_done[r])
            with torch.cuda.stream(down):
                for b, hc in zip(s["lin"], pin_c[r]):
                    hc.copy_(b["c"], non_blocking=True)
                ev_out[r].record(down)
            used[r] = True

        with torch.cuda.stream(stream):
            for i in range(W):
                e2e_step(i)
            barrier()
            ke = args.e2e_steps or K
            probe0 = time.perf_counter()
            e2e_step(0)
            torch.cuda.synchronize()
            per = max(time.perf_counter() - probe0, 1e-6)
            ke = max(3, min(ke, int(2.0 / per)))
            barrier()
            ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ea.record(up)   # every stream is idle here: the region starts with the first upload
            stream.wait_event(ea)
            down.wait_event(ea)
            for i in range(ke):
                e2e_step(i)
            last = torch.cuda.Event()
            last.record(down)
            stream.wait_event(last)
            eb.record(stream)   # after the last read-back
            barrier()
            e2e_ms = rank_max(ea.elapsed_time(eb)) / ke
        flops_step = sum(k[3] for k in kinfo)
        e2e = {"value": round(replica_throughput(world, flops_step, e2e_ms), 4), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": ke, "ms_per_step": round(e2e_ms, 5),
               "copies": "pinned host buffers; uploads, compute and read-backs of consecutive steps overlap on "
                         "three streams"}

    # ---- numbers
    peaks, peaks_src = load_peaks()
    timed_s = step_ms * K / 1e3
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    fp8_peak_sus = peaks["bf16_tflops_sustained"] * FP8_OVER_BF16
    fp8_use = fp8_peak_sus if timed_s >= 1.0 else fp8_peak
    hbm = peaks["hbm_gbs"]
    kernels = []
    for (name, bound, nbytes, flops), ms in zip(kinfo, kern_ms):
        if bound is None:
            bound = "tensor" if flops / (fp8_use * 1e12) > nbytes / (hbm * 1e9) else "hbm"
        ent = {"kernel": name, "ms": round(ms, 6), "bound": bound, "bytes": nbytes, "flops": flops,
               "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1)}
        if flops:
            ent["TFLOP/s"] = round(flops / (ms * 1e-3) / 1e12, 2)
        ent["frac"] = round((ent["TFLOP/s"] / fp8_use) if bound == "tensor" else ent["GB/s"] / hbm, 4)
        kernels.append(ent)
    # dominant kernel = largest share of the kernel region (aggregated by name)
    agg = {}
    for k in kernels:
        a = agg.setdefault(k["kernel"], {"ms": 0.0, "bytes": 0, "flops": 0, "bound": k["bound"]})
        a["ms"] += k["ms"]
        a["bytes"] += k["bytes"]
        a["flops"] += k["flops"]
    dom = max(agg, key=lambda n: agg[n]["ms"])
    d = agg[dom]
    nl = sum(1 for k in kernels if k["kernel"] == dom)
    if d["bound"] == "tensor":
        ach = d["flops"] / (d["ms"] * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(ach, 2), "peak": round(fp8_use, 1), "unit": "TFLOP/s",
                "frac": round(ach / fp8_use, 4)}
        roof["peak_source"] = (f"{peaks_src} bf16 {'sustained' if fp8_use == fp8_peak_sus else 'burst'} "
                               f"x {FP8_OVER_BF16:g} (nominal FP8/BF16 ratio)")
    else:
        ach = d["bytes"] / (d["ms"] * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s", "frac": round(ach / hbm, 4),
                "peak_source": f"{peaks_src} hbm_gbs"}
    tr = recorded_traffic(dom, args.workload)
    roof["traffic"] = None if tr is None else tr * 1
    roof["kernel"] = dom
    roof["per_launch"] = {"bytes": d["bytes"] // nl, "flops": d["flops"] // nl, "ms": round(d["ms"] / nl, 6)}

    flops_step = sum(k[3] for k in kinfo)
    value = replica_throughput(world, flops_step, step_ms)
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(step_ms, 6), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 x e4m3 -> f32 accumulate", "data": "synthetic (seeded Philox normal / Student-t inputs)",
        "config": config_of(args, wl),
        "l2_rotation": f"{R} input sets ({R * set_bytes / 1e6:.0f} MB; L2 {l2 / 1e6:.0f} MB)",
        "roofline": roof,
        "kernels": kernels,
        "kernel_region": {"steps": Kk, "ms_per_step": round(kregion_step_ms, 6),
                          "timing": "each kernel alone: one CUDA graph of back-to-back launches over the "
                                    "rotating input sets, CUDA events around it"},
        "gpu_launches": K * sum(launches_per_kernel),
        "e2e": e2e,
        "clocks": sampler.summary(t0, t1, t_wide0),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl)
    if rank == 0:
        print(json.dumps(line), flush=True)


# ----------------------------------------------------------- CPU oracle arm
_INPUTS = {}


def workload_inputs(wl):
    """Host inputs of every linear (generated once per process)."""
    import synth
    if wl.name not in _INPUTS:
        acts, ws = {}, {}
        for lin in wl.linears:
            if lin.K not in acts:
                acts[lin.K] = synth.activation(wl, lin)
            ws[lin.name] = synth.weight(wl, lin)
        _INPUTS[wl.name] = (acts, ws)
    return _INPUTS[wl.name]


# FLOPs of oracle GEMM work in one sampled step (split evenly over the step's
# GEMMs; each GEMM runs its first rows and is extrapolated to all M rows).
# Fixed, so that the GPU arm's cpu_baseline and the reference arm time the
# same sample and report the same rate.
ORACLE_SAMPLE_FLOP = 2e10


def oracle_sample_rows(wl):
    """Rows of each GEMM in the sampled oracle step, in `kernel_plan` order."""
    nlin = len(wl.linears) * len(wl.modes)
    share = ORACLE_SAMPLE_FLOP / nlin
    return [int(max(1, min(lin.M, round(share / (2 * lin.N * lin.K))))) for lin in wl.linears for _ in wl.modes]


def oracle_step_sample(wl):
    """Times the oracle on one pass of the workload: every quantizer in full
    and, per GEMM, the first rows of `oracle_sample_rows`, extrapolated
    linearly to all M rows.  Returns (seconds per full step, description)."""
    import numpy as np

    import oracle

    total = 0.0
    parts = []
    acts, ws = workload_inputs(wl)
    rows_of = iter(oracle_sample_rows(wl))
    for lin in wl.linears:
        a, w = acts[lin.K], ws[lin.name]
        for mode in wl.modes:
            rows = next(rows_of)
            if mode == "per_tensor_static":
                s_held = oracle.scale_from_history(np.float32([oracle.amax(a, wl.in_dtype)]), 0)
                hist = np.zeros(HIST_LEN, np.float32)
            if mode in FP8W_MODES:   # the weight is quantized once, outside the timed step
                qw, sw = oracle.quantize_weight_block(w, wl.in_dtype)
            t = time.perf_counter()
            if mode in FP8W_MODES:
                qa, sa = oracle.quantize_token_group(a, wl.in_dtype)
            elif mode in ("block", "fused"):
                qa, sa = oracle.quantize_token_group(a, wl.in_dtype)
                qw, sw = oracle.quantize_weight_block(w, wl.in_dtype)
            elif mode == "block_ue8m0":
                qa, ca = oracle.quantize_token_group_ue8m0(a, wl.in_dtype)
                qw, cw = oracle.quantize_weight_block_ue8m0(w, wl.in_dtype)
                sa, sw = oracle.ue8m0_decode(ca), oracle.ue8m0_decode(cw)
            elif mode == "per_channel":
                qa, sa = oracle.quantize_per_tensor(a, wl.in_dtype)
                qw, sw = oracle.quantize_per_channel(w, wl.in_dtype)
            elif mode == "per_tensor_static":
                qa, sa = oracle.quantize_with_scale(a, wl.in_dtype, s_held), s_held
                hist[0] = oracle.amax(a, wl.in_dtype)
                qw, sw = oracle.quantize_per_tensor(w, wl.in_dtype)
            else:
                qa, sa = oracle.quantize_per_tensor(a, wl.in_dtype)
                qw, sw = oracle.quantize_per_tensor(w, wl.in_dtype)
            tq = time.perf_counter() - t
            t = time.perf_counter()
            if mode in ("block", "fused", "block_ue8m0") or mode in FP8W_MODES:
                oracle.gemm_block(qa, sa, qw, sw, rows=np.arange(rows))
            elif mode == "per_channel":
                oracle.gemm_per_channel(qa, sa, qw, sw, rows=np.arange(rows))
            else:
                oracle.gemm_per_tensor(qa, sa, qw, sw, rows=np.arange(rows))
            tg = time.perf_counter() - t
            if mode == "per_tensor_static":
                t = time.perf_counter()
                oracle.scale_from_history(hist, HIST_MARGIN)
                tq += time.perf_counter() - t
            total += tq + tg * lin.M / rows
            parts.append(f"{lin.name}/{mode}: quantize full, GEMM {rows}/{lin.M} rows")
    return total, "; ".join(parts)


def oracle_timing(wl, warmup, samples):
    """`warmup` untimed sampled steps, then the median of `samples` timed
    ones: (seconds per full step, description, thread count)."""
    import oracle
    for _ in range(warmup):
        oracle_step_sample(wl)
    times, desc = [], ""
    for _ in range(samples):
        t, desc = oracle_step_sample(wl)
        times.append(t)
    return statistics.median(times), desc, oracle.get_threads()


def step_flops(wl):
    return sum(2 * lin.M * lin.N * lin.K for lin in wl.linears) * len(wl.modes)


def baseline_entry(wl, seconds, desc, cores, warmup, samples):
    return {"value": round(step_flops(wl) / seconds / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{desc} (GEMM time extrapolated to all rows); median of {samples} sampled steps after "
                      f"{warmup} untimed",
            "s_per_step": round(seconds, 4), "samples": samples}


def cpu_baseline(wl, warmup=1, samples=3):
    t, desc, cores = oracle_timing(wl, warmup, samples)
    return baseline_entry(wl, t, desc, cores, warmup, samples)


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    wl = workload_of(args)
    t, desc, cores = oracle_timing(wl, args.warmup, args.steps)
    base = baseline_entry(wl, t, desc, cores, args.warmup, args.steps)
    value = base["value"]
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
        "config": config_of(args, wl),
        "cpu_baseline": base,
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def lines_of(args):
    """(workload, modes) of every line to print: the one asked for, or the
    default set with the headline workload last."""
    import copy
    todo = [(args.workload, args.modes)] if args.workload else list(DEFAULT_LINES)
    out = []
    for wl, modes in todo:
        a = copy.copy(args)
        a.workload, a.modes = wl, modes
        out.append(a)
    return out


def main():
    args = parse_args()
    for a in lines_of(args):
        if args.impl == "reference":
            run_reference(a)
        else:
            run_ours(a)
            import gc

            import torch
            gc.collect()
            torch.cuda.empty_cache()
    if args.impl != "reference" and dist_env()[1] > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
