"""Benchmark of the block-scaled quantized GEMM hot path on GB300.

One step = one pass of every row of the hot path over its workload, inputs resident in HBM:
  1. MXFP8 GEMM        M = N = K = 8192   (E4M3 + UE8M0 per 32 along K, per-row variance)
  2. fp16 GEMM         M = N = K = 4096
  3. W4A16 GEMM        M = 4096, N = 14336, K = 4096 (int4 weights, UE8M0 per 32)
  4. W8 decode GEMV    M = 1, 8, 16; N = 28672, K = 8192, each M as a run of four consecutive
                       launches (a decode step's GEMVs; weights rotate over three copies)
Each kernel is timed with CUDA events on the stream it is launched on.  The headline ``value``
is the MXFP8 8192^3 GEMM in TFLOP/s; the GEMV in GB/s and the other rows are reported beside it.

``--impl reference`` times the CPU oracle (test infrastructure, plain fp64 C) on a bounded sample
of the same workload instead.  Under torchrun (N > 1) every rank runs the whole step on its own
GPU (independent problems, no collective: weak scaling); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import datetime
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
SPEC_FP8_TFLOPS = 4500.0
SPEC_F16_TFLOPS = 2250.0
SPEC_FP4_TFLOPS = 13500.0
SPEC_HBM_GBS = 8000.0
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
METRIC = "MXFP8 GEMM TFLOP/s at 8192^3 (% of GB300 FP8 peak); W8 GEMV GB/s (% of HBM)"
WORKLOAD = "mxfp8_8192 + w4a16_prefill + f16_4096 + w8_decode(M=1,8,16)"


def _traffic(record: str):
    """DRAM bytes per call from a committed ncu traffic record under profiles/ (its line
    "traffic_bytes_per_call: N sha1(<source>): <hash> ..."), or None when the record is missing
    or any of the kernel sources it names has changed since the counters were taken."""
    import hashlib
    import re
    root = os.path.dirname(os.path.abspath(__file__))
    try:
        text = open(os.path.join(root, "profiles", record)).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_call: (\d+)((?: sha1\([\w.]+\): [0-9a-f]+)+)", text)
    if not m:
        return None
    csrc = os.path.join(root, "block_scaled_quantized_tcgen05_gb300", "csrc")
    for name, want in re.findall(r"sha1\(([\w.]+)\): ([0-9a-f]+)", m.group(2)):
        try:
            with open(os.path.join(csrc, name), "rb") as f:
                if hashlib.sha1(f.read()).hexdigest() != want:
                    return None
        except OSError:
            return None
    return int(m.group(1))


def max_over_ranks(values, ws: int, device):
    """Element-wise maximum of a list of floats over all ranks of the default process group
    (the identity at world size 1): every rank's timings become the slowest rank's."""
    if ws <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def whole_job_rate(ws: int, work_per_rank: float, ms: float) -> float:
    """Throughput of the whole job: the work all ranks did over the (max-over-ranks) time."""
    return ws * work_per_rank / (ms * 1e-3)


def _peaks():
    try:
        with open(PEAKS_PATH) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK), "fallback"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 50 ms during the timed region."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.bus_id = bus_id
        self.proc = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "50"]
        if self.bus_id:
            cmd += ["-i", self.bus_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None

    def stop(self, t_begin: float | None = None, t_end: float | None = None):
        """Summarise the samples taken between t_begin and t_end (host wall-clock seconds, the
        timed region); all samples when no window is given or none falls inside it."""
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]), float(parts[3]), parts[4:8]))
            except ValueError:
                continue
        inside = [r for r in rows if t_begin is not None and t_begin <= r[0] <= t_end]
        use = inside if inside else rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in use:
            for n, v in zip(names, r[4]):
                if v.lower() == "active":
                    reasons.add(n)
        sm = [r[1] for r in use]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_min_mhz": min(sm) if sm else None,
                "sm_max_mhz": max(r[2] for r in use) if use else None,
                "power_w_median": statistics.median(r[3] for r in use) if use else None,
                "samples": len(use), "samples_in_timed_region": len(inside),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------------------ our arm
def run_ours(args, ws, rank, local):
    import torch

    import block_scaled_quantized_tcgen05_gb300 as q
    from block_scaled_quantized_tcgen05_gb300 import synth

    q.build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    # ------------------------------------------------------------- inputs (resident in HBM)
    only = args.only
    want = (lambda k: only is None or only == k)
    mx = None
    if want("mxfp8") or only == "epilogue":
        mx = synth.workload("mxfp8_8192")
        a, sa, b, sb = (mx[k].to(dev) for k in ("a", "sa", "b", "sb"))
        A8 = q.qgemm_create_tensor(q.E4M3, a, sa)
        B8 = q.qgemm_create_tensor(q.E4M3, b, sb)
        C8 = torch.empty(8192, 8192, dtype=torch.float16, device=dev)
        # fused-epilogue variants: C = relu(A B^T), and C = relu(A B^T + C) on its own buffer
        C8r = torch.empty(8192, 8192, dtype=torch.float16, device=dev)
        C8a = torch.zeros(8192, 8192, dtype=torch.float16, device=dev)
    if only == "mxfp4":      # the FP4 row, timed on its own: 8192^3 E2M1 with UE8M0 scales
        m4 = synth.workload("mxfp4_8192")
        A4 = q.qgemm_create_tensor(q.E2M1, m4["a"].to(dev), m4["sa"].to(dev))
        B4 = q.qgemm_create_tensor(q.E2M1, m4["b"].to(dev), m4["sb"].to(dev))
        C4 = torch.empty(8192, 8192, dtype=torch.float16, device=dev)
        del m4
    if only == "w4a16_f16s":   # int4 weights with fp16 block scales, the prefill shape
        wf = synth.workload("w4a16_f16s_prefill")
        wfa, wfw, wfs = wf["a"].to(dev), wf["w"].to(dev), wf["sw"].to(dev)
        wfc = torch.empty(4096, 14336, dtype=torch.float16, device=dev)
        del wf
    if only == "attention":   # fused attention, 32 heads x 4096 x 4096 x 128
        at = synth.workload("attn_prefill")
        atq, atk, atv = at["q"].to(dev), at["k"].to(dev), at["v"].to(dev)
        ato = torch.empty_like(atq)
        at_scale = at["scale"]
        del at
    if want("f16"):
        f = synth.workload("f16_4096")
        fa, fb = f["a"].to(dev), f["b"].to(dev)
        fc = torch.empty(4096, 4096, dtype=torch.float16, device=dev)
        del f
    if want("w4a16"):
        w4 = synth.workload("w4a16_prefill")
        w4a = w4["a"].to(dev)
        W4 = q.qgemm_create_tensor(q.INT4, w4["w"].to(dev), w4["sw"].to(dev))
        w4c = torch.empty(4096, 14336, dtype=torch.float16, device=dev)
        del w4
    if want("gemv"):
        gv = synth.workload("w8_decode", M=16)
        W8s = []
        # three weight copies (727 MB): with two, ncu saw 27 MB of a 242 MB stream still hit in L2
        for copy in range(3):
            w8 = gv["w"].to(dev) if copy == 0 else gv["w"].to(dev).clone()
            s8 = gv["sw"].to(dev) if copy == 0 else gv["sw"].to(dev).clone()
            W8s.append(q.qgemm_create_tensor(q.INT8, w8, s8))
        X16 = gv["x"].to(dev)
        Ys = {m: torch.empty(m, 28672, dtype=torch.float16, device=dev) for m in (1, 8, 16)}
        del gv

    # the decode GEMVs run after the fp16 GEMM (33 MB of output) rather than after W4A16, whose
    # 117 MB of output is still being written back from L2 when the next kernel starts
    all_kernels = ["mxfp8", "w4a16", "f16", "gemv_m1", "gemv_m8", "gemv_m16"]
    kernels = [k for k in all_kernels if want(k.split("_")[0])]
    if only == "epilogue":   # the fused output epilogues on the MXFP8 workload
        kernels = ["mxfp8", "mxfp8_relu", "mxfp8_accrelu"]
    if only == "mxfp4":
        kernels = ["mxfp4"]
    if only == "w4a16_f16s":
        kernels = ["w4a16_f16s"]
    if only == "attention":
        kernels = ["attention"]
    stream = torch.cuda.current_stream()
    gemv_count = [0]
    # SM clock during the MXFP8 GEMM: a probe issued right after each timed GEMM on the same
    # stream starts once the GEMM's CTAs all run (a programmatic dependent), reads cycles and
    # global time over 200 us of the GEMM's ~330 us and completes with the GEMM
    probe_buf = torch.zeros(max(1, args.steps), 2, dtype=torch.int64, device=dev)
    probe_gemv = torch.zeros(max(1, args.steps), 2, dtype=torch.int64, device=dev)
    PROBE_NS = 200_000
    PROBE_GEMV_NS = 20_000        # inside the last M = 1 decode GEMV of a run (about 39 us)
    probe_on = [False, 0]
    # GEMVs are timed as runs of consecutive launches, as a decode step issues them; a CUDA event
    # between two kernels costs each one the whole kernel boundary (about 4 us here)
    GEMV_RUN = 4

    def launch(k, i):
        if k == "mxfp8":
            q.qgemm_mxfp8(A8, B8, C8)
        elif k == "mxfp8_relu":
            q.qgemm_mxfp8_ex(A8, B8, C8r, relu=True)
        elif k == "mxfp8_accrelu":
            q.qgemm_mxfp8_ex(A8, B8, C8a, accumulate=True, relu=True)
        elif k == "mxfp4":
            q.qgemm_mxfp4(A4, B4, C4)
        elif k == "w4a16_f16s":
            q.qgemm_w4a16_f16s(wfa, wfw, wfs, wfc)
        elif k == "attention":
            q.qgemm_attention(atq, atk, atv, ato, scale=at_scale)
        elif k == "f16":
            q.gemm_f16(fa, fb, fc)
        elif k == "w4a16":
            q.qgemm_w4a16(w4a, W4, w4c)
        else:
            # a decode run: GEMV_RUN launches back to back (each a programmatic dependent of the
            # one before), consecutive launches reading different weight copies (727 MB in all)
            m = int(k[6:])
            for _ in range(GEMV_RUN):
                q.qgemm_w8_gemv(X16[:m], W8s[gemv_count[0] % 3], Ys[m])
                if m == 1 and _ == GEMV_RUN - 1 and probe_on[0]:
                    q.qgemm_sm_clock_probe(PROBE_GEMV_NS, probe_gemv[probe_on[1]])
                gemv_count[0] += 1

    def step(i, ev=None):
        if ev is not None:
            ev[0].record(stream)
        probe_on[0], probe_on[1] = ev is not None, i
        for j, k in enumerate(kernels):
            launch(k, i)
            if ev is not None and k == "mxfp8":
                q.qgemm_sm_clock_probe(PROBE_NS, probe_buf[i])
            if ev is not None:
                ev[j + 1].record(stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if q.qgemm_poll_device_error() != 0:
        raise RuntimeError("a kernel wait timed out during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(kernels) + 1)]
           for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    bus = None
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id
    except Exception:
        pass
    sampler = ClockSampler(bus if rank == 0 else None)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    wall0 = time.time()
    t0.record(stream)
    for i in range(args.steps):
        step(i, evs[i])
    t1.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    clocks = sampler.stop(wall0, wall1) if rank == 0 else None
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    if q.qgemm_poll_device_error() != 0:
        raise RuntimeError("a kernel wait timed out during the timed region")

    total_ms = t0.elapsed_time(t1)
    if clocks is not None:
        clocks["smi_sm_mhz"] = clocks["sm_mhz"]
        if "mxfp8" in kernels:
            pr = probe_buf.cpu().tolist()
            mhz = [1e3 * c / n for c, n in pr[:args.steps] if n > 0]
            if mhz:
                clocks["sm_mhz"] = round(statistics.median(mhz), 1)
                clocks["sm_mhz_source"] = ("median over the timed steps of a clock64 / globaltimer "
                                           "probe run beside the MXFP8 GEMM (200 us of each launch)")
                clocks["probe_mhz_min_max"] = [round(min(mhz), 1), round(max(mhz), 1)]
        if "gemv_m1" in kernels:
            pr = probe_gemv.cpu().tolist()
            mhz = [1e3 * c / n for c, n in pr[:args.steps] if n > 0]
            if mhz:
                clocks["sm_mhz_during_gemv_m1"] = round(statistics.median(mhz), 1)
    per = {k: [evs[i][j].elapsed_time(evs[i][j + 1]) / (GEMV_RUN if k.startswith("gemv") else 1)
               for i in range(args.steps)]
           for j, k in enumerate(kernels)}
    mean = {k: sum(v) / len(v) for k, v in per.items()}
    median = {k: statistics.median(v) for k, v in per.items()}
    agg = max_over_ranks([total_ms] + [mean[k] for k in kernels] + [median[k] for k in kernels],
                         ws, dev)
    total_ms = agg[0]
    mean = {k: agg[1 + j] for j, k in enumerate(kernels)}
    median = {k: agg[1 + len(kernels) + j] for j, k in enumerate(kernels)}

    # ----------------------------------------------------------- e2e through host buffers
    e2e = None
    if rank == 0 and mx is not None and not args.no_e2e:
        e2e = e2e_mxfp8(q, torch, dev, a, sa, b, sb, reps=max(3, min(10, args.steps)))

    # ---------------------------------------------------------- derived numbers
    flops = {"mxfp8": 2.0 * 8192 ** 3, "f16": 2.0 * 4096 ** 3, "w4a16": 2.0 * 4096 * 14336 * 4096,
             "w4a16_f16s": 2.0 * 4096 * 14336 * 4096, "attention": 4.0 * 32 * 4096 * 4096 * 128}
    gemv_bytes = {m: 28672 * 8192 + 28672 * 256 + m * 8192 * 2 + m * 28672 * 2 for m in (1, 8, 16)}
    peaks, peak_kind = _peaks()
    fp8_peak_sust = 2.0 * peaks.get("bf16_tflops_sustained", FALLBACK["bf16_tflops_sustained"])
    fp8_peak_burst = 2.0 * peaks.get("bf16_tflops", FALLBACK["bf16_tflops"])
    hbm = peaks.get("hbm_gbs", FALLBACK["hbm_gbs"])
    secondary = {}
    for k in kernels:
        if k in ("f16", "w4a16", "w4a16_f16s", "attention"):
            tf = flops[k] / (mean[k] * 1e-3) / 1e12
            secondary[k] = {"us": round(mean[k] * 1e3, 2), "us_median": round(median[k] * 1e3, 2),
                            "tflops": round(tf, 1),
                            "frac_of_f16_spec_2250": round(tf / SPEC_F16_TFLOPS, 4),
                            "frac_of_measured_bf16_sustained": round(
                                tf / peaks.get("bf16_tflops_sustained", 1700.0), 4)}
        elif k.startswith("gemv"):
            m = int(k[6:])
            gbs = gemv_bytes[m] / (mean[k] * 1e-3) / 1e9
            secondary[k] = {"us": round(mean[k] * 1e3, 2), "us_median": round(median[k] * 1e3, 2),
                            "gbs": round(gbs, 1),
                            "frac_of_measured_hbm": round(gbs / hbm, 4),
                            "frac_of_spec_hbm_8000": round(gbs / SPEC_HBM_GBS, 4),
                            "timing": f"per launch, over runs of {GEMV_RUN} consecutive launches"}
    for k in ("mxfp8_relu", "mxfp8_accrelu"):
        if k in mean:
            tf = flops["mxfp8"] / (mean[k] * 1e-3) / 1e12
            secondary[k] = {"us": round(mean[k] * 1e3, 2), "us_median": round(median[k] * 1e3, 2),
                            "tflops": round(tf, 1), "frac_of_fp8_spec_4500": round(tf / SPEC_FP8_TFLOPS, 4),
                            "epilogue": "C = relu(A B^T)" if k == "mxfp8_relu"
                            else "C = relu(A B^T + C): reads the old C (+134 MB)"}
    if "mxfp4" in mean:
        tf = 2.0 * 8192 ** 3 / (mean["mxfp4"] * 1e-3) / 1e12
        fp4_peak_sust = 6.0 * peaks.get("bf16_tflops_sustained", FALLBACK["bf16_tflops_sustained"])
        secondary["mxfp4"] = {"us": round(mean["mxfp4"] * 1e3, 2),
                              "us_median": round(median["mxfp4"] * 1e3, 2),
                              "tflops": round(tf, 1),
                              "frac_of_fp4_spec_13500": round(tf / SPEC_FP4_TFLOPS, 4),
                              "frac_of_measured_bf16_sustained_x6": round(tf / fp4_peak_sust, 4),
                              "kernel": "qgemm_mxfp4 = sf_pack_kernel<2> + mx_pair_kernel<E2M1>",
                              "algorithmic_bytes": 2 * 8192 * 4096 + 2 * 8192 * 256
                              + 2 * 8192 * 8192}
    mx_tflops = None
    if "mxfp8" in mean:
        mx_tflops = flops["mxfp8"] / (mean["mxfp8"] * 1e-3) / 1e12
        secondary["mxfp8"] = {"us": round(mean["mxfp8"] * 1e3, 2),
                              "us_median": round(median["mxfp8"] * 1e3, 2),
                              "tflops": round(mx_tflops, 1),
                              "frac_of_fp8_spec_4500": round(mx_tflops / SPEC_FP8_TFLOPS, 4)}
    value = (whole_job_rate(ws, flops["mxfp8"], mean["mxfp8"]) / 1e12
             if mx_tflops is not None else None)
    # one qgemm_mxfp8 call at 8192^3 is two launches (scale repack + CTA-pair GEMM), one
    # qgemm_w4a16 call two (the GEMM + the outlier-row pass), one attention call one (the
    # persistent kernel merges the units its key-tile ranges split; the flags it zeroes first
    # are a driver memset, not a kernel of this library)
    launches = sum(2 if k.startswith("mxfp") or k == "w4a16"
                   else GEMV_RUN if k.startswith("gemv") else 1 for k in kernels) * args.steps
    launches += args.steps * (("mxfp8" in kernels) + ("gemv_m1" in kernels))   # clock probes
    line = {
        "metric": METRIC, "value": round(value, 2) if value is not None else None,
        "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3+ue8m0",
        "data": "synthetic (seeded, shapes and distributions of the workloads)",
        "config": {"workload": WORKLOAD if only is None else only,
                   "headline": "mxfp8_8192 M=N=K=8192",
                   "parallelism": f"replicas x{ws}",
                   "l2": "inputs larger than L2: each kernel's inputs are evicted by the rest of "
                         "the step (>129 MB between reuses); GEMV weights rotate over 3 copies"},
        "roofline": None if mx_tflops is None else {
            "kernel": "qgemm_mxfp8 = sf_pack_kernel<1> + mx_pair_kernel<FmtE4M3>", "bound": "tensor",
            "achieved": round(mx_tflops, 1), "peak": round(fp8_peak_burst, 1),
            "unit": "TFLOP/s", "frac": round(mx_tflops / fp8_peak_burst, 4),
            "peak_source": f"{peak_kind} bf16 burst x 2 (nominal fp8/bf16 ratio), the larger "
                           "of the two measured peaks and so the stricter denominator; the "
                           "sustained one (a seconds-long loop at the power-capped clock) is "
                           f"frac_of_measured_sustained; timed region {round(total_ms, 1)} ms",
            "frac_of_measured_sustained": round(mx_tflops / fp8_peak_sust, 4),
            "frac_of_spec_4500": round(mx_tflops / SPEC_FP8_TFLOPS, 4),
            "traffic": _traffic("mxfp8_pair_8192_traffic.txt"),
            "traffic_unit": "bytes per call (ncu, dram read + write)",
            "algorithmic_bytes": 2 * 8192 * 8192 + 2 * 8192 * 256 + 2 * 8192 * 8192},
        "roofline_gemv": None if "gemv_m1" not in mean else {
            "kernel": "qgemm_w8_gemv = w8_gemv_kernel, M = 1 (the decode row of the metric), "
                      f"average launch of runs of {GEMV_RUN} back-to-back launches",
            "bound": "hbm", "achieved": secondary["gemv_m1"]["gbs"], "peak": hbm, "unit": "GB/s",
            "frac": round(secondary["gemv_m1"]["gbs"] / hbm, 4),
            "peak_source": f"{peak_kind} HBM copy bandwidth",
            "frac_of_spec_8000": round(secondary["gemv_m1"]["gbs"] / SPEC_HBM_GBS, 4),
            "traffic": _traffic("w8_gemv_decode_traffic.txt"),
            "traffic_unit": "bytes per launch (ncu, dram read + write)",
            "algorithmic_bytes": gemv_bytes[1]},
        "kernels": secondary,
        "gpu_launches": launches,
        "clocks": clocks,
        "e2e": e2e,
    }
    if rank == 0 and mx is not None and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_rows, mx)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return line


def e2e_mxfp8(q, torch, dev, a, sa, b, sb, reps):
    """The same metric through the public host-memory C-ABI call, qgemm_mxfp8_host: every step
    uploads A, B and their scales from pinned host buffers, runs the GEMM and downloads C into a
    pinned host buffer.  Steps alternate between two streams, so one step's uploads overlap the
    previous step's download (the library keeps two device buffer sets for that)."""
    ha, hsa, hb, hsb = (t.cpu().pin_memory() for t in (a, sa, b, sb))
    hc = [torch.empty(8192, 8192, dtype=torch.float16).pin_memory() for _ in range(2)]
    A = q.qgemm_create_tensor(q.E4M3, ha, hsa)
    B = q.qgemm_create_tensor(q.E4M3, hb, hsb)
    streams = [torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)]
    cur = torch.cuda.current_stream()

    def run(n):
        for i in range(n):
            q.qgemm_mxfp8_host(A, B, hc[i % 2], stream=streams[i % 2])

    run(2)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    for st in streams:
        st.wait_stream(cur)
    run(reps)
    for st in streams:
        cur.wait_stream(st)
    e1.record(cur)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    bi = sum(t.numel() * t.element_size() for t in (ha, hsa, hb, hsb))
    bo = hc[0].numel() * hc[0].element_size()
    return {"value": round(2.0 * 8192 ** 3 / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "ms_per_call": round(ms, 3),
            "api": "qgemm_mxfp8_host (host operands and output; steps on two streams)"}


# --------------------------------------------------------------------- CPU oracle timing
def cpu_baseline(rows: int, d):
    """The oracle (plain fp64 C, OpenMP over all host cores) on a sample of the MXFP8 8192^3
    workload: `rows` output rows x all 8192 columns, decode of A rows and all of B included."""
    import numpy as np

    import oracle
    oracle.build()
    a, sa, b, sb = (d[k].numpy() for k in ("a", "sa", "b", "sb"))
    sel = np.arange(rows)
    t = time.perf_counter()
    oracle.mxfp8(a, sa, b, sb, rows=sel)
    dt = time.perf_counter() - t
    flops = 2.0 * rows * 8192 * 8192
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    omp = os.environ.get("OMP_NUM_THREADS")
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s",
            "cores": int(omp) if omp else cores, "kind": "oracle",
            "sample": f"MXFP8 8192^3: {rows} rows x 8192 cols x K=8192 (fp64 decode + dot), "
                      f"{dt:.2f} s"}


def run_reference(args, ws, rank):
    """Reference arm: the CPU oracle as it stands, each step a bounded sample of the workload."""
    if rank != 0:
        return None
    import numpy as np

    import oracle
    from block_scaled_quantized_tcgen05_gb300 import synth
    oracle.build()
    d = synth.workload("mxfp8_8192")
    a, sa, b, sb = (d[k].numpy() for k in ("a", "sa", "b", "sb"))
    rows = args.ref_rows
    for i in range(args.warmup):
        oracle.mxfp8(a, sa, b, sb, rows=np.arange(i % 8, i % 8 + 1))
    t = time.perf_counter()
    for i in range(args.steps):
        sel = (np.arange(rows) + i * rows) % 8192
        oracle.mxfp8(a, sa, b, sb, rows=sel)
    dt = time.perf_counter() - t
    flops = 2.0 * rows * 8192 * 8192 * args.steps
    value = flops / dt / 1e12
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, shapes and distributions of the workloads)",
        "config": {"workload": "mxfp8_8192 M=N=K=8192 (oracle on a row sample per step)"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"{rows} output rows x 8192 cols x K=8192 per step"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def _swizzle_scales_for_cublaslt(s):
    """UE8M0 scale plane [R, C] -> the 128 x 4 tiled order cuBLASLt reads for VEC32 block scales:
    rows padded to 128 and columns to 4 (zero bytes), tiles in row-major tile order, and inside a
    tile the byte of (row 32 a + b, column c) at 16 b + 4 a + c."""
    import torch
    R, C = s.shape
    Rp, Cp = (R + 127) // 128 * 128, (C + 3) // 4 * 4
    pad = torch.zeros(Rp, Cp, dtype=torch.uint8, device=s.device)
    pad[:R, :C] = s
    t = pad.view(Rp // 128, 4, 32, Cp // 4, 4).permute(0, 3, 2, 1, 4).contiguous()
    return t.view(-1)


def run_libref(args):
    """Library reference points on this GPU, in one process beside our kernels, on the benchmark's
    own data: cuBLASLt's block-scaled FP8 GEMM (E4M3 with UE8M0 scales per 32 along K, through
    torch._scaled_mm) against qgemm_mxfp8 at 8192^3, and cuBLAS fp16 (torch.matmul) against
    gemm_f16 at 4096^3.  CUDA events, `warmup` launches then the mean of `steps` back-to-back
    launches of each."""
    import numpy as np
    import torch

    import block_scaled_quantized_tcgen05_gb300 as q
    from block_scaled_quantized_tcgen05_gb300 import synth
    q.build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()

    def timed(fn):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps

    out = {"impl": "library-reference", "torch": torch.__version__, "steps": args.steps,
           "gpu": torch.cuda.get_device_name(dev)}
    mx = synth.workload("mxfp8_8192")
    a, sa, b, sb = (mx[k].to(dev) for k in ("a", "sa", "b", "sb"))
    A8 = q.qgemm_create_tensor(q.E4M3, a, sa)
    B8 = q.qgemm_create_tensor(q.E4M3, b, sb)
    C8 = torch.empty(8192, 8192, dtype=torch.float16, device=dev)
    ms = timed(lambda: q.qgemm_mxfp8(A8, B8, C8))
    out["qgemm_mxfp8_8192"] = {"us": round(ms * 1e3, 1),
                               "tflops": round(2 * 8192 ** 3 / (ms * 1e-3) / 1e12, 1)}
    try:
        fa8 = a.view(torch.float8_e4m3fn)
        fb8 = b.view(torch.float8_e4m3fn)
        ssa = _swizzle_scales_for_cublaslt(sa).view(torch.float8_e8m0fnu)
        ssb = _swizzle_scales_for_cublaslt(sb).view(torch.float8_e8m0fnu)
        ref_dtype = torch.float16
        try:
            Cl = torch._scaled_mm(fa8, fb8.t(), ssa, ssb, out_dtype=ref_dtype)
        except Exception:
            ref_dtype = torch.bfloat16
            Cl = torch._scaled_mm(fa8, fb8.t(), ssa, ssb, out_dtype=ref_dtype)
        torch.cuda.synchronize()
        ms = timed(lambda: torch._scaled_mm(fa8, fb8.t(), ssa, ssb, out_dtype=ref_dtype))
        # the two products must agree (same decoded operands): relative to sum |a b| on 64 rows
        rows = torch.arange(0, 8192, 128, device=dev)
        da = (a[rows].view(torch.float8_e4m3fn).float().view(64, 256, 32)
              * torch.exp2(sa[rows].float() - 127).unsqueeze(2)).view(64, 8192)
        db = (b.view(torch.float8_e4m3fn).float().view(8192, 256, 32)
              * torch.exp2(sb.float() - 127).unsqueeze(2)).view(8192, 8192)
        mag = (da.abs() @ db.abs().t())
        dif = (Cl[rows].float() - C8[rows].float()).abs() / mag.clamp_min(1e-30)
        out["cublaslt_mxfp8_8192"] = {
            "us": round(ms * 1e3, 1), "tflops": round(2 * 8192 ** 3 / (ms * 1e-3) / 1e12, 1),
            "call": f"torch._scaled_mm(E4M3 [M,K], E4M3 [N,K]^T, UE8M0 per 32 (128x4 tiled), "
                    f"out {str(ref_dtype).replace('torch.', '')})",
            "max_abs_diff_over_sum_abs_ab_vs_qgemm_mxfp8": float(dif.max())}
    except Exception as ex:          # the installed torch has no MX path for this GPU
        out["cublaslt_mxfp8_8192"] = {"unavailable": f"{type(ex).__name__}: {ex}"[:300]}
    del a, sa, b, sb, C8, mx
    f = synth.workload("f16_4096")
    fa, fb = f["a"].to(dev), f["b"].to(dev)
    fc = torch.empty(4096, 4096, dtype=torch.float16, device=dev)
    ms = timed(lambda: q.gemm_f16(fa, fb, fc))
    out["gemm_f16_4096"] = {"us": round(ms * 1e3, 1),
                            "tflops": round(2 * 4096 ** 3 / (ms * 1e-3) / 1e12, 1)}
    ms = timed(lambda: torch.matmul(fa, fb))
    tc = torch.matmul(fa, fb)
    torch.cuda.synchronize()
    out["cublas_f16_4096"] = {"us": round(ms * 1e3, 1),
                              "tflops": round(2 * 4096 ** 3 / (ms * 1e-3) / 1e12, 1),
                              "call": "torch.matmul(fp16 [4096,4096], fp16 [4096,4096])",
                              "max_abs_diff_vs_gemm_f16": float((tc.float() - fc.float()).abs().max())}
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-rows", type=int, default=4096)
    ap.add_argument("--ref-rows", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--only", default=None,
                    choices=["mxfp8", "f16", "w4a16", "gemv", "epilogue", "mxfp4", "w4a16_f16s",
                             "attention", "libref"],
                    help="run one row of the hot path only (profiling); 'epilogue': MXFP8 8192^3 "
                         "plain, with C = relu(A B^T) and with C = relu(A B^T + C); 'mxfp4': the "
                         "FP4 (E2M1) GEMM at 8192^3; 'w4a16_f16s': int4 with fp16 block scales, "
                         "4096 x 14336 x 4096; 'attention': fused attention, 32 heads x 4096 x "
                         "4096 x 128; 'libref': cuBLASLt block-scaled FP8 at 8192^3 and cuBLAS "
                         "fp16 at 4096^3 beside qgemm_mxfp8 and gemm_f16, same data")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = _dist()
    if args.impl == "reference":
        line = run_reference(args, ws, rank)
    elif args.only == "libref":
        line = run_libref(args) if rank == 0 else None
    else:
        line = run_ours(args, ws, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
