#!/usr/bin/env python
"""Throughput of the INT8 quantized linear layer on GB300.

One step = one full pass of the layer's hot path, ck_int8_linear: the preparation kernel
(activation quantize into bf16 codes, plus the int8 -> bf16 weight widening) and the
tensor-core GEMM with the fused dequant/bias/bf16 epilogue, over one batch of seeded
synthetic inputs that are already resident in device memory.  Metric: 2*M*N*K / step
time, in TOPS.  The default workload is the largest per-row shape of the sweep,
80666 x 28672 x 5376 (PR #142, "Numbers from the sweep").

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

Without --steps the timed region runs as many steps as fill about 8 seconds (at least 20).

Under torchrun (N > 1) every rank runs its own copy of the workload on its own GPU
(independent problems, weak scaling, no collective on the data path); the step time is
the maximum over ranks.  Rank 0 prints one JSON line.

--impl reference times the CPU oracle (plain C, all host cores) on a bounded row
sample of the same workload; the other ranks exit without work.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from int8_weight_quantized_gb300 import synthetic  # noqa: E402

METRIC = "INT8 linear TOPS (2MNK/s, fused dequant) and % of GB300 dense INT8 peak"
# --path w8a16 times the layer's 16-bit-activation path instead (not the headline metric)
METRICS = {"int8": METRIC, "w8a16": "W8A16 linear TOPS (2MNK/s, bf16 activations x int8 weight codes)"}
UNIT = "TOPS"
WORKLOADS = {spec[0]: spec for spec in synthetic.ALL_WORKLOADS}
DEFAULT_WORKLOAD = synthetic.SWEEP[-1][0]  # per_row_80666x28672x5376
TIMED_SECONDS = 8.0  # target length of the timed region when --steps is not given
FLUSH_BYTES = 512 << 20  # > 129 MB of L2: written between steps (outside the timed events)
L2_BYTES = 129 << 20
CLEAN_BYTES = 256 << 20  # then read, so the step does not start by writing back the flush's dirty lines
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
PROFILE_INT8_PEAK = os.path.join(ROOT, "profiles", "int8_peak.json")
GEMM_SOURCES = ["int8_weight_quantized_gb300/csrc/gemm.cu", "int8_weight_quantized_gb300/csrc/ck_device.cuh",
                "int8_weight_quantized_gb300/csrc/gemm_common.cuh"]


# ---------------------------------------------------------------- helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier():
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()


def reduce_max(value, device="cpu"):
    """Maximum of a float over all ranks (identity when not distributed)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    """(bf16 TFLOP/s burst, sustained, HBM GB/s, provenance)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), \
            float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, 1700.0, 6800.0, "fallback"


def sources_sha256(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def int8_dense_peak():
    """GB300's dense int8 matrix rate as measured by the committed mma.sync tool, or None."""
    try:
        with open(PROFILE_INT8_PEAK) as f:
            return json.load(f)["int8_dense_peak"]
    except (OSError, KeyError, ValueError):
        return None


def profiled_traffic(workload):
    """DRAM bytes per GEMM launch from the committed ncu summary, or None when the
    summary is missing, is for another workload, or predates the current kernel source."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            d = json.load(f)["gemm"]
    except (OSError, KeyError, ValueError):
        return None
    if d.get("workload") != workload or d.get("source_sha256") != sources_sha256(GEMM_SOURCES):
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock, power and throttle reasons while running."""
    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device_index):
        self.proc = None
        self.out = None
        self.target = self._smi_id(device_index)

    @staticmethod
    def _smi_id(device_index):
        try:
            p = torch.cuda.get_device_properties(device_index)
            return "%08X:%02X:%02X.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        except Exception:
            return None

    def start(self):
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits", "-lms", "100"]
        if self.target:
            cmd[1:1] = ["-i", self.target]
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        lines = self.out.read().splitlines()
        self.out.close()
        os.unlink(self.out.name)
        return self.parse(lines)

    @classmethod
    def parse(cls, lines):
        sm, mx, reasons = [], [], set()
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != len(cls.FIELDS):
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(cls.REASONS, parts[5:]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def workload_config(spec, l2_note):
    name, M, N, K, mode, bias, frac, seed = spec
    return {"workload": name, "M": M, "N": N, "K": K, "mode": synthetic.MODE_NAMES[mode], "bias": bool(bias),
            "seed": seed, "l2": l2_note}


# ---------------------------------------------------------------- the CPU oracle arms
def oracle_step_rows(case, rows, path="int8"):
    """One oracle evaluation of the layer on the first `rows` rows (its own scale for
    tensorwise mode: the sample is the tensor)."""
    import numpy as np
    import oracle

    x = case.x[:rows].contiguous().view(torch.int16).numpy().view(np.uint16)
    if case.mode == synthetic.CONVROT:
        w, ws = case.meta["w_rot"]
    else:
        w, ws = case.w.numpy(), case.w_scale.numpy()
    b = None if case.bias is None else case.bias.contiguous().view(torch.int16).numpy().view(np.uint16)
    t0 = time.perf_counter()
    if path == "w8a16":
        oracle.w8a16_linear(x, w, ws, b, mode=case.mode)
    else:
        oracle.int8_linear(x, w, ws, b, mode=case.mode)
    return time.perf_counter() - t0


def prepare_oracle_case(spec):
    case = synthetic.case_from_spec(spec)
    if case.mode == synthetic.CONVROT:
        import oracle
        case.meta["w_rot"] = oracle.prepare_convrot_weight(case.w_float.numpy())
    return case


def cpu_baseline(spec, path="int8", budget_s=12.0):
    """The oracle as it stands, on a bounded row sample of the workload."""
    import oracle

    case = prepare_oracle_case(spec)
    M, N, K = case.M, case.N, case.K
    probe = min(M, max(8, oracle.num_threads()))
    t = oracle_step_rows(case, probe, path)
    rows = int(min(M, max(probe, probe * budget_s / max(t, 1e-6))))
    t = oracle_step_rows(case, rows, path)
    return {"value": 2.0 * rows * N * K / t / 1e12, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "first %d of %d rows x all %d columns, K=%d (%.1f s)" % (rows, M, N, K, t)}


def run_reference(args, spec):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle

    case = prepare_oracle_case(spec)
    M, N, K = case.M, case.N, case.K
    budget = 150.0  # seconds for warmup + timed steps together
    probe = min(M, max(4, oracle.num_threads()))
    t_probe = oracle_step_rows(case, probe, args.path)
    per_row = t_probe / probe
    steps = args.steps if args.steps is not None else 20
    rows = int(max(1, min(M, budget / (steps + args.warmup) / per_row)))
    for _ in range(args.warmup):
        oracle_step_rows(case, rows, args.path)
    times = [oracle_step_rows(case, rows, args.path) for _ in range(steps)]
    step_s = sum(times) / len(times)
    value = 2.0 * rows * N * K / step_s / 1e12
    sample = "first %d of %d rows x all %d columns, K=%d, per step" % (rows, M, N, K)
    line = {"impl": "reference", "metric": METRICS[args.path], "value": value, "unit": UNIT, "n_gpus": world,
            "steps": steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int8" if args.path == "int8" else "bf16",
            "data": "synthetic",
            "config": workload_config(spec, "n/a (host)"),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- the GPU arm
def run_ours(args, spec):
    import int8_weight_quantized_gb300 as ck
    from int8_weight_quantized_gb300 import build as ck_build

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    ck_build.build()
    dev = torch.device("cuda", local)

    name, M, N, K, mode, has_bias, frac, seed = spec
    case = synthetic.case_from_spec(spec)
    x = case.x.to(dev)
    if mode == synthetic.CONVROT:
        # the layer's stored weight W @ H^T, prepared once per layer (not part of a step)
        w, ws_ = ck.ck_convrot_prepare_weight(case.w_float.to(dev))
    else:
        w = case.w.to(dev)
        ws_ = case.w_scale.to(dev)
    b = None if case.bias is None else case.bias.to(dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    w8a16 = args.path == "w8a16"
    codes = None
    if w8a16:
        work = ck.workspace(ck.load_library().ck_w8a16_linear_workspace_size(M, N, K, mode), dev)
    elif args.weight_codes:
        # the weight's bf16 codes, prepared once per layer (outside the steps)
        codes = ck.ck_int8_weight_codes(w)
        work = ck.workspace(ck.load_library().ck_int8_linear_codes_workspace_size(M, N, K, mode), dev)
    else:
        work = ck.workspace(ck.ck_int8_linear_workspace_size(M, N, K, mode), dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    clean = torch.zeros(CLEAN_BYTES // 8, dtype=torch.int64, device=dev)
    sink = torch.empty((), dtype=torch.int64, device=dev)

    def flush_l2(i):
        flush.fill_(i & 0xFF)
        torch.sum(clean, dim=0, out=sink)

    ops = 2.0 * M * N * K

    def step():
        if w8a16:
            ck.ck_w8a16_linear(x, w, ws_, b, mode=mode, y=y, ws=work)
        elif codes is not None:
            ck.ck_int8_linear_codes(x, codes, ws_, b, mode=mode, y=y, ws=work)
        else:
            ck.ck_int8_linear(x, w, ws_, b, mode=mode, y=y, ws=work)

    for i in range(args.warmup):
        flush_l2(i)
        step()
    torch.cuda.synchronize()
    if ck.ck_device_error(clear=True) != 0:
        raise SystemExit("a kernel reported a wait timeout during warm-up")
    steps = args.steps
    if steps is None:
        # size the timed region from one more (untimed) step: about TIMED_SECONDS of steps
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush_l2(0)
        e0.record()
        step()
        e1.record()
        torch.cuda.synchronize()
        one = reduce_max(e0.elapsed_time(e1), dev)
        steps = int(min(4000, max(20, TIMED_SECONDS * 1e3 / max(one, 1e-3))))

    # ---- timed region: `steps` steps, device-resident inputs, L2 flushed between steps.
    # The library only counts its launches here (no events between its kernels, so their
    # programmatic launch overlap is what gets timed).
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    ck.ck_profile_begin(with_events=False)
    wall0 = time.perf_counter()
    for i, (e0, e1) in enumerate(evs):
        flush_l2(i)
        e0.record()
        step()
        e1.record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier()
    counts = ck.ck_profile_end()
    clocks = sampler.stop()
    step_ms_local = sum(a.elapsed_time(b_) for a, b_ in evs) / steps
    step_ms = reduce_max(step_ms_local, dev)
    value = world * ops / (step_ms * 1e-3) / 1e12
    if ck.ck_device_error(clear=True) != 0:
        raise SystemExit("a kernel reported a wait timeout in the timed region")

    # ---- per-kernel durations: the same loop with CUDA events around each library launch
    kt_steps = min(steps, 300)
    barrier()
    torch.cuda.synchronize()
    ck.ck_profile_begin(with_events=True)
    for i in range(kt_steps):
        flush_l2(i)
        step()
    torch.cuda.synchronize()
    prof = ck.ck_profile_end()

    # ---- roofline of the dominant kernel (the GEMM) and of the bandwidth-bound preparation
    bf16_peak, bf16_sust, hbm_peak, provenance = load_peaks()
    g_ms, g_n = prof["gemm"]
    p_ms = prof["quantize"][0] + prof["widen"][0]
    p_n = prof["quantize"][1] + prof["widen"][1]
    gemm_avg_ms = reduce_max(g_ms / max(g_n, 1), dev)
    achieved = ops / (gemm_avg_ms * 1e-3) / 1e12
    traffic = None if w8a16 else profiled_traffic(name)
    # The preparation launch.  Algorithmic bytes (the activation quantize alone): read x
    # (bf16) and write int8 codes, 3 B per element, plus 4 B per row scale; tensorwise
    # reads x twice (5 B per element).  Moved bytes (what the launch really does, the
    # bf16-operand engine's overhead included): x read, its codes written as bf16, the int8
    # weight read and written as bf16 codes.  The 16-bit path: the weight widening, plus
    # read x / write bf16(x @ H) for ConvRot.
    if w8a16:
        prep_alg = 4 * M * K if mode == synthetic.CONVROT else 0
        prep_moved = N * K + 2 * N * K + prep_alg
    else:
        prep_alg = (5 * M * K + 4) if mode == synthetic.TENSORWISE else (3 * M * K + 4 * M)
        prep_moved = 2 * M * K + 2 * M * K + (0 if codes is not None else N * K + 2 * N * K) + \
            (4 if mode == synthetic.TENSORWISE else 4 * M)
    p_step = max(p_ms, 1e-9) / kt_steps
    roofline = {"bound": "tensor", "achieved": achieved, "peak": bf16_peak, "unit": "TFLOP/s",
                "frac": achieved / bf16_peak, "traffic": traffic,
                "kernel": ("gemm_kernel<mixed> (tcgen05 kind::f16, bf16 activations x int8 codes, fp32 sum)" if w8a16
                           else "gemm_kernel (tcgen05 kind::f16 on int8 codes, exact int32, fused dequant)"),
                "peak_source": "%s bf16 dense, burst (cuBLAS); the engine this kernel runs on" % provenance,
                "peak_sustained": bf16_sust, "frac_sustained": achieved / bf16_sust,
                "avg_launch_ms": gemm_avg_ms, "timed_launches": g_n,
                "algorithmic_flops_per_launch": ops}
    i8 = int8_dense_peak()
    if i8 is not None and not w8a16:
        # the GPU's dense int8 matrix rate (its only int8 instruction, mma.sync): the layer,
        # exact on the bf16 engine, runs at a multiple of it
        roofline["int8_dense_peak"] = dict(i8, layer_over_peak=value / i8["value"],
                                           gemm_over_peak=achieved / i8["value"])
    kernels = {
        "gemm": {"ms_per_step": g_ms / kt_steps, "launches": g_n},
        "prep": {"ms_per_step": p_step, "launches": p_n,
                 "bytes_algorithmic": prep_alg, "bytes_moved": prep_moved,
                 "GB/s_algorithmic": prep_alg / (p_step * 1e-3) / 1e9,
                 "GB/s_moved": prep_moved / (p_step * 1e-3) / 1e9,
                 "frac_hbm_algorithmic": prep_alg / (p_step * 1e-3) / 1e9 / hbm_peak,
                 "frac_hbm_moved": prep_moved / (p_step * 1e-3) / 1e9 / hbm_peak},
    }
    if not w8a16:
        kernels["quantize_int8"] = time_quantize_int8(ck, x, mode, flush_l2, min(kt_steps, 200), hbm_peak, dev)

    # ---- end to end from and to pinned host memory.  The INT8 layer: its host-memory
    # entry point, which pipelines the copies with the kernels over row slabs.  The
    # 16-bit path: the copy in, the call, the copy out, in sequence.
    e2e_steps = max(20, min(steps, 100))
    x_host = torch.empty((M, K), dtype=torch.bfloat16, pin_memory=True)
    x_host.copy_(case.x)
    y_host = torch.empty((M, N), dtype=torch.bfloat16, pin_memory=True)
    host_ws = None if w8a16 else ck.workspace(
        ck.load_library().ck_int8_linear_host_workspace_size(M, N, K, mode, ck.OUT_BF16, 0), dev)
    if not w8a16:
        for _ in range(2):  # warm-up (the first call in a context makes the copy streams)
            ck.ck_int8_linear_host(x_host, w, ws_, b, mode=mode, y=y_host, ws=host_ws)
    e2e_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(e2e_steps)]
    barrier()
    torch.cuda.synchronize()
    for i, (e0, e1) in enumerate(e2e_evs):
        flush_l2(i)
        e0.record()
        if w8a16:
            x.copy_(x_host, non_blocking=True)
            step()
            y_host.copy_(y, non_blocking=True)
        else:
            ck.ck_int8_linear_host(x_host, w, ws_, b, mode=mode, y=y_host, ws=host_ws)
        e1.record()
    torch.cuda.synchronize()
    e2e_each = sorted(a.elapsed_time(b_) for a, b_ in e2e_evs)
    e2e_ms = reduce_max(sum(e2e_each) / e2e_steps, dev)
    e2e = {"value": world * ops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT, "h2d_bytes_per_step": x_host.numel() * 2,
           "d2h_bytes_per_step": y_host.numel() * 2, "ms_per_step": e2e_ms,
           # the host link stalls now and then for tens of ms; the median step shows the rest
           "median_ms_per_step": e2e_each[len(e2e_each) // 2], "max_ms_per_step": e2e_each[-1],
           "entry": "ck_w8a16_linear with torch copies" if w8a16 else "ck_int8_linear_host (slab-pipelined copies)"}

    line = {"metric": METRICS[args.path], "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int8" if not w8a16 else "bf16", "data": "synthetic",
            "config": dict(workload_config(spec, "flushed between steps (%d MiB write, then %d MiB read); inputs %s L2" % (
                FLUSH_BYTES >> 20, CLEAN_BYTES >> 20, "larger than" if M * K * 2 > L2_BYTES else "smaller than")),
                           **({"weight": "bf16 codes prepared once per layer (ck_int8_linear_codes)"} if codes is not None
                              else {})),
            "roofline": roofline, "kernels": kernels, "e2e": e2e, "clocks": clocks,
            "gpu_launches": int(sum(n for _, n in counts.values())), "timed_wall_s": wall}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(spec, args.path)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()
    return 0


def time_quantize_int8(ck, x, mode, flush_l2, n, hbm_peak, dev):
    """The stand-alone activation quantize (ck_quantize_int8_rowwise, rotated for ConvRot,
    or ck_quantize_int8_tensorwise): bf16 x in, int8 codes and fp32 scales out, each launch
    bracketed by CUDA events on the launching stream.  L2 is flushed before each launch
    unless x alone is larger than L2 (then launches follow each other, as in a stream of
    calls, and no launch finds its input in L2)."""
    M, K = x.shape
    tw = mode == synthetic.TENSORWISE
    q = torch.empty((M, K), dtype=torch.int8, device=dev)
    xs = torch.empty((1 if tw else M,), dtype=torch.float32, device=dev)

    def run():
        if tw:
            ck.ck_quantize_int8_tensorwise(x, q=q, x_scale=xs)
        else:
            ck.ck_quantize_int8_rowwise(x, rotate=(mode == synthetic.CONVROT), q=q, x_scale=xs)

    for i in range(3):
        flush_l2(i)
        run()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    flush = 2 * M * K <= L2_BYTES
    torch.cuda.synchronize()
    for i, (e0, e1) in enumerate(evs):
        if flush:
            flush_l2(i)
        e0.record()
        run()
        e1.record()
    torch.cuda.synchronize()
    ms = reduce_max(sum(a.elapsed_time(b) for a, b in evs) / n, dev)
    nbytes = (5 * M * K + 4) if tw else (3 * M * K + 4 * M)
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"entry": "ck_quantize_int8_tensorwise" if tw else "ck_quantize_int8_rowwise",
            "rotate": mode == synthetic.CONVROT, "ms": ms, "launches": n, "l2_flushed": flush,
            "bytes_algorithmic": nbytes,
            "GB/s": gbs, "frac_hbm": gbs / hbm_peak, "peak_hbm_gbs": hbm_peak}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: as many as fill about %g s, at least 20)" % TIMED_SECONDS)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--weight-codes", action="store_true",
                    help="run the INT8 layer on the weight's bf16 codes prepared once (ck_int8_linear_codes) "
                         "instead of widening the int8 weight in every step")
    ap.add_argument("--path", choices=sorted(METRICS), default="int8",
                    help="int8: the INT8 layer (the headline); w8a16: its 16-bit-activation path")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    spec = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, spec)
    return run_ours(args, spec)


if __name__ == "__main__":
    sys.exit(main())
