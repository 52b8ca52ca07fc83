"""Benchmark: FP16 -> FP32 GEMM throughput on GB300 through the library's C ABI.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {ours,reference}]
                  [--workload {gemm,softmax}] [--configs] [--sustained SECONDS]
                  [--sustained-leg SECONDS]
  python bench.py --splits [--steps S]
  python bench.py --case M N K [--launches L] [--warmup W] [--cta-group G] [--tile-n T]
                  [--stages S] [--group-m G] [--max-ctas C] [--stream-k 0|1|2] [--flush-l2]

A step is one C = A.B call on the 8192 x 8192 x 8192 workload (A, B drawn N(0,1) from
seed 4, rounded to FP16).  The inputs (256 MiB) are larger than L2, so no flush is needed
between steps.  Prints one JSON line (rank 0).  Under torchrun with N > 1 every rank runs
its own replica on its own GPU (the problem does not need a collective); the time is the
maximum over ranks and the value the aggregate throughput.

After the timed steps the line adds: the end-to-end figure through the host-buffer call,
4096^3 with L2 flushed before each launch (`secondary`), 8192^3 with L2 flushed (`cold_l2`),
and 4096^3 and 8192^3 back to back for --sustained-leg seconds with the SM clock sampled
inside each loop (`sustained`).  The roofline's `frac` divides by the measured cuBLAS bf16
peak; `frac_per_clock` divides the sustained 8192^3 rate by SMs x 8192 FLOP/clk x the median
SM clock of that loop, the device's dense FP16 rate at the clock it actually ran.

--impl reference times the CPU oracle (the plain FP64-accumulating definition) on the
host cores over a bounded sample of the same workload.

--workload softmax measures the second, bandwidth-bound workload instead: the fused row
softmax of a 65536 x 1024 FP32 matrix (N(0,1), seed 2; 256 MiB in, 256 MiB out, larger
than L2), one softmax_rows_f32 call per step, in GB/s of algorithmic traffic (read MN +
write MN), with the page's own 4096 x 1024 case (L2 flushed before each launch) beside it.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = (8192, 8192, 8192)
SEED = 4
SECONDARY = (4096, 4096, 4096)
METRIC = "FP16->FP32 GEMM TFLOP/s at 4096^3/8192^3; % of GB300 dense FP16 tensor peak"
UNIT = "TFLOP/s"
FALLBACK_PEAK_TFLOPS = 1900.0
L2_FLUSH_BYTES = 512 << 20
SUSTAINED_SECONDS = 0.25
# Dense FP16/BF16 tensor rate of one SM per clock (kind::f16 MMAs with FP32 accumulation):
# the per-clock denominator, peak = SMs x this x SM clock.
TENSOR_FLOP_PER_CLK_SM = 8192
MAX_SM_MHZ = 2070.0
# device code of the measured kernels (a committed ncu figure holds while these are unchanged
# and the plan it was taken with is the plan the bench runs)
KERNEL_SOURCES = ("gemm_sm103a.cu", "ptx_sm103a.cuh", "tile_sched.h", "gemm_internal.h")
SOFTMAX_SOURCES = ("softmax_sm103a.cu", "ptx_sm103a.cuh", "gemm_internal.h")
SOFTMAX_WORKLOAD = (65536, 1024)
SOFTMAX_SEED = 2
SOFTMAX_METRIC = "fused row softmax GB/s (read MN + write MN FP32); % of measured HBM copy bandwidth"
SOFTMAX_UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target length of the CPU-oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=["gemm", "softmax"], default="gemm")
    ap.add_argument("--configs", action="store_true",
                    help="instead of the benchmark line, time every workload shape (one JSON line each)")
    ap.add_argument("--sustained", type=float, default=0.0, metavar="SECONDS",
                    help="instead of the benchmark line, run 4096^3 and 8192^3 back to back for SECONDS each "
                         "and report TFLOP/s with the SM clocks and power seen (one JSON line each)")
    ap.add_argument("--sustained-leg", type=float, default=4.0, metavar="SECONDS",
                    help="length of the back-to-back 4096^3 and 8192^3 loops that follow the timed steps in the "
                         "benchmark line (clock-sampled; they give the per-clock fraction); 0 leaves them out")
    # one shape, for profiling and sweeps
    ap.add_argument("--case", type=int, nargs=3, metavar=("M", "N", "K"),
                    help="instead of the benchmark line, time C = A.B on one shape (inputs drawn on the device) "
                         "and print the per-launch device times")
    ap.add_argument("--launches", type=int, default=3, help="--case: timed launches")
    ap.add_argument("--tile-n", type=int, default=0)
    ap.add_argument("--stages", type=int, default=0)
    ap.add_argument("--group-m", type=int, default=0)
    ap.add_argument("--max-ctas", type=int, default=0)
    ap.add_argument("--cta-group", type=int, default=0)
    ap.add_argument("--stream-k", type=int, default=0, help="--case: 1 = whole tiles only, 2 = force split tiles")
    ap.add_argument("--flush-l2", action="store_true", help="--case: write 512 MiB before each launch")
    ap.add_argument("--splits", action="store_true",
                    help="instead of the benchmark line, time each work-split form (whole tiles, two-part split "
                         "tail, stream-K) against the planner's choice on shapes where they differ")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def dist_max(value, dist, device):
    """Maximum of a per-rank float over the process group (all ranks receive it)."""
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(world, flops_per_rank, ms_max):
    """Whole-job throughput: every rank runs its own replica of the step; the slowest rank's
    time bounds the job."""
    return world * flops_per_rank / (ms_max * 1e-3) / 1e12


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0.0)), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_PEAK_TFLOPS, None, "fallback"


def hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def code_text(text):
    """C/C++ source with its comments removed and its whitespace collapsed to single spaces
    (string and character literals kept as they are)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
            out.append(" ")
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_hash(sources=KERNEL_SOURCES):
    """Hash of the device sources' code: comments and layout are left out, so that an edit
    of a comment does not retire a profile taken on the same code."""
    h = hashlib.sha256()
    for name in sources:
        with open(os.path.join(ROOT, "tensor_core_tiled_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(code_text(f.read()).encode())
    return h.hexdigest()[:16]


def traffic_per_launch(name="gemm_8192_dram_traffic.json", sources=KERNEL_SOURCES, plan=None):
    """DRAM bytes (read + write) per launch of the measured kernel from the committed ncu
    summary, or None if absent, taken on a different kernel source, or (when the summary
    records one) under a different launch plan."""
    path = os.path.join(ROOT, "profiles", name)
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_hash") != kernel_hash(sources):
        return None
    if plan is not None and "plan" in d and any(plan.get(k) != v for k, v in d["plan"].items()):
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks/throttle sampling in the background (timestamps in host time)."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.samples = []
        self._stop = threading.Event()
        self._thr = None

    def _run(self):
        try:
            proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                     "--format=csv,noheader,nounits", "-lms", "50"],
                                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        try:
            for line in proc.stdout:
                self.samples.append((time.time(), [x.strip() for x in line.split(",")]))
                if self._stop.is_set():
                    break
        finally:
            proc.terminate()
            try:
                proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                proc.kill()

    def start(self):
        self._thr = threading.Thread(target=self._run, daemon=True)
        self._thr.start()
        time.sleep(0.3)

    def stop(self):
        self._stop.set()
        if self._thr:
            self._thr.join(timeout=10)

    def summary(self, t0, t1):
        inside = [s for (t, s) in self.samples if t0 <= t <= t1]
        window = "timed region"
        if not inside and self.samples:
            nearest = min(self.samples, key=lambda ts: min(abs(ts[0] - t0), abs(ts[0] - t1)))
            inside = [nearest[1]]
            window = "nearest sample (timed region shorter than the sampling period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(s[1]) for s in inside if len(s) > 1 and num(s[1]) is not None]
        mx = [num(s[2]) for s in inside if len(s) > 2 and num(s[2]) is not None]
        pw = [num(s[3]) for s in inside if len(s) > 3 and num(s[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for s in inside:
            for i, n in enumerate(names):
                if len(s) > 5 + i and s[5 + i].lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "reasons": sorted(reasons),
                "samples": len(inside), "window": window}


def make_inputs(M, N, K, seed):
    import numpy as np
    from tensor_core_tiled_gb300 import inputs
    rng = np.random.default_rng(seed)
    return inputs.normal_pair(rng, M, N, K)


def _oracle_rate(A, B, rows=4):
    """Rows per second of the oracle on this host (a short calibration run)."""
    import oracle
    oracle.build()
    t0 = time.perf_counter()
    oracle.gemm_rows_f32(A, B, 0, rows)
    return rows / max(time.perf_counter() - t0, 1e-9)


def _oracle_sample(A, B, rows):
    """Time the oracle on rows [0, rows) of the product; returns (seconds, flops)."""
    import oracle
    N, K = B.shape[1], A.shape[1]
    t0 = time.perf_counter()
    oracle.gemm_rows_f32(A, B, 0, rows)
    return time.perf_counter() - t0, 2.0 * rows * N * K


def _baseline_record(A, B, rows, secs, flops):
    import oracle
    M, K = A.shape
    N = B.shape[1]
    return {"value": flops / secs / 1e12, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"rows 0..{rows - 1} of the {M}x{N}x{K} seed-{SEED} product ({rows * N} outputs, "
                      f"{flops / 1e9:.1f} GFLOP in {secs:.2f} s), FP64 accumulation, all host threads"}


def cpu_baseline(A, B, target_seconds):
    """The oracle as it stands, timed on a bounded sample: leading rows of the same product."""
    rate = _oracle_rate(A, B)
    rows = int(max(1, min(A.shape[0], rate * target_seconds)))
    secs, flops = _oracle_sample(A, B, rows)
    return _baseline_record(A, B, rows, secs, flops)


def back_to_back(launch, seconds, sampler, warm_seconds=1.0):
    """Launches `launch` back to back for `seconds` (after `warm_seconds` of warm-up), in
    batches of about 0.1 s, timed by one CUDA event pair around the whole loop; the clocks
    are the sampler's summary over the loop.  Returns (ms per launch, launches, clocks)."""
    import torch
    t_end = time.time() + warm_seconds
    while time.time() < t_end:
        for _ in range(10):
            launch()
        torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(10):
        launch()
    e1.record()
    torch.cuda.synchronize()
    per = max(1, int(0.1 / max(e0.elapsed_time(e1) / 10 / 1e3, 1e-9)))
    launches = 0
    t0 = time.time()
    e0.record()
    while time.time() - t0 < seconds:
        for _ in range(per):
            launch()
        launches += per
        torch.cuda.synchronize()
    e1.record()
    torch.cuda.synchronize()
    t1 = time.time()
    return e0.elapsed_time(e1) / launches, launches, sampler.summary(t0, t1)


def per_clock_peak_tflops(sms, mhz):
    """Dense FP16 tensor peak of the device at an SM clock of `mhz`, in TFLOP/s."""
    return sms * TENSOR_FLOP_PER_CLK_SM * mhz * 1e6 / 1e12


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    M, N, K = WORKLOAD
    A, B = make_inputs(M, N, K, SEED)
    # each step: a bounded sample sized so that warm-up + steps take about cpu_seconds * 6
    per_step = max(0.02, 6.0 * args.cpu_seconds / max(1, args.steps + args.warmup))
    rate = _oracle_rate(A, B)
    rows = int(max(1, min(M, rate * per_step)))
    for _ in range(args.warmup):
        _oracle_sample(A, B, rows)
    secs = flops = 0.0
    for _ in range(args.steps):
        s, f = _oracle_sample(A, B, rows)
        secs += s
        flops += f
    value = flops / secs / 1e12
    rec = _baseline_record(A, B, rows, secs / args.steps, flops / args.steps)
    rec["value"] = value
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": f"gemm_f16_f32 {M}x{N}x{K}, A and B N(0,1) FP16 "
                                                        f"from seed {SEED}, FP32 output",
                                            "M": M, "N": N, "K": K},
            "cpu_baseline": rec,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import numpy as np
    import torch

    import tensor_core_tiled_gb300 as tct
    from tensor_core_tiled_gb300 import build as lib_build

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        dist = None
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    if rank == 0:
        lib_build.build()
    if dist:
        dist.barrier()
    tct.load()

    M, N, K = WORKLOAD
    A16, B16 = make_inputs(M, N, K, SEED)
    hA = torch.from_numpy(A16.view(np.int16)).view(torch.float16).pin_memory()
    hB = torch.from_numpy(B16.view(np.int16)).view(torch.float16).pin_memory()
    dA = hA.to(dev)
    dB = hB.to(dev)
    dC = torch.empty((M, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    flops = 2.0 * M * N * K

    def launch():
        st = tct.gemm_f16_f32(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), M, N, K, K, N, N, sp)
        if st:
            raise tct.GemmError(st, "gemm_f16_f32")

    for _ in range(max(3, args.warmup)):
        launch()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    # ---- timed region: K launches, one event pair per launch on the launching stream
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_host0 = time.time()
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for e0, e1 in evs:
        e0.record(stream)
        launch()
        e1.record(stream)
    g1.record(stream)
    torch.cuda.synchronize()
    t_host1 = time.time()
    if dist:
        dist.barrier()
    total_ms = g0.elapsed_time(g1)
    launch_ms = [a.elapsed_time(b) for a, b in evs]
    sampler.stop()
    clocks = sampler.summary(t_host0, t_host1)

    # max over ranks of the timed region
    if dist:
        total_ms = dist_max(total_ms, dist, dev)
    ms_per_step = total_ms / args.steps
    value = aggregate_tflops(world, flops, ms_per_step)
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK

    # ---- end to end through the public host-buffer call: gemm_f16_f32_host copies A and B
    # from pinned memory, multiplies and copies C back into pinned memory (row blocks
    # pipelined across two copy streams and the GEMM), all inside the timed region.
    hC = torch.empty((M, N), dtype=torch.float32).pin_memory()
    e2e_steps = max(1, min(args.steps, 20))

    def e2e_step():
        st = tct.gemm_f16_f32_host(hA.data_ptr(), hB.data_ptr(), hC.data_ptr(), M, N, K, K, N, N, sp)
        if st:
            raise tct.GemmError(st, "gemm_f16_f32_host")

    for _ in range(3):  # warm-up: pools, copy streams and the host link settled
        e2e_step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    x0 = torch.cuda.Event(enable_timing=True)
    x1 = torch.cuda.Event(enable_timing=True)
    x0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    x1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = x0.elapsed_time(x1) / e2e_steps
    if dist:
        e2e_ms = dist_max(e2e_ms, dist, dev)
    e2e_value = aggregate_tflops(world, flops, e2e_ms)

    # ---- secondary workload: 4096^3 (inputs fit in L2, so L2 is flushed before each launch)
    m2, n2, k2 = SECONDARY
    sA, sB = make_inputs(m2, n2, k2, 2)
    sA = torch.from_numpy(sA.view(np.int16)).view(torch.float16).to(dev)
    sB = torch.from_numpy(sB.view(np.int16)).view(torch.float16).to(dev)
    sC = torch.empty((m2, n2), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def launch2():
        st = tct.gemm_f16_f32(sA.data_ptr(), sB.data_ptr(), sC.data_ptr(), m2, n2, k2, k2, n2, n2, sp)
        if st:
            raise tct.GemmError(st, "gemm_f16_f32")

    for _ in range(5):
        launch2()
    sec = []
    n_sec = max(5, min(args.steps, 100))
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_sec)]
    for a, b in pairs:
        flush.fill_(1.0)
        a.record(stream)
        launch2()
        b.record(stream)
    torch.cuda.synchronize()
    sec = [a.elapsed_time(b) for a, b in pairs]
    sec_ms = statistics.mean(sec)
    sec_tflops = 2.0 * m2 * n2 * k2 / (sec_ms * 1e-3) / 1e12
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK

    # ---- 8192^3 with L2 flushed (512 MiB written) before each launch: the cold-cache form
    cold = []
    cold_pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(max(5, min(args.steps, 20)))]
    for a, b in cold_pairs:
        flush.fill_(1.0)
        a.record(stream)
        launch()
        b.record(stream)
    torch.cuda.synchronize()
    cold = [a.elapsed_time(b) for a, b in cold_pairs]
    cold_ms = statistics.mean(cold)
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK

    # ---- back-to-back loops of 4096^3 and 8192^3 under the power cap, clocks sampled inside
    # the loop: the sustained figures and, from time x median clock, the per-clock fraction
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sustained = {}
    if args.sustained_leg > 0:
        sampler2 = ClockSampler(local)
        sampler2.start()
        try:
            for name, fn, f in (("4096^3", launch2, 2.0 * m2 * n2 * k2), ("8192^3", launch, flops)):
                ms_l, n_l, clk = back_to_back(fn, args.sustained_leg, sampler2)
                tf = f / (ms_l * 1e-3) / 1e12
                mhz = clk.get("sm_mhz")
                sustained[name] = {
                    "seconds": args.sustained_leg, "launches": n_l, "ms_per_launch": ms_l, "tflops": tf,
                    "sm_mhz_median": mhz, "clocks": clk,
                    "cycles_per_launch": ms_l * 1e-3 * mhz * 1e6 if mhz else None,
                    "frac_per_clock": tf / per_clock_peak_tflops(sms, mhz) if mhz else None}
        finally:
            sampler2.stop()
        assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK

    # ---- the tensor core's own rate per SM per clock, measured on this device (one CTA per
    # SM issuing back-to-back 128x256x16 MMAs, timed by the SM clock counter)
    probe_med, probe_lo, probe_hi = tct.gemm_tensor_rate_probe(1 << 16, sp)

    peak_burst, peak_sustained, peak_src = peaks()
    mean_launch = statistics.mean(launch_ms)
    achieved = flops / (mean_launch * 1e-3) / 1e12
    clock_peak_max = per_clock_peak_tflops(sms, MAX_SM_MHZ)
    s8 = sustained.get("8192^3", {})
    # A timed region of back-to-back launches longer than SUSTAINED_SECONDS runs under the
    # power cap: compare it with the sustained library figure, a short one with the burst one.
    region_s = total_ms * 1e-3
    if peak_sustained and region_s >= SUSTAINED_SECONDS:
        peak, peak_kind = peak_sustained, "sustained"
    else:
        peak, peak_kind = peak_burst, "burst"
    plan = tct.gemm_f16_f32_plan(M, N, K)
    plan2 = tct.gemm_f16_f32_plan(m2, n2, k2)

    line = None
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": f"gemm_f16_f32 {M}x{N}x{K}, A and B N(0,1) FP16 from seed {SEED}, "
                                   f"FP32 accumulate and output",
                       "M": M, "N": N, "K": K, "accumulate": "f32", "parallelism": f"replicas x{world}",
                       "l2": "inputs (256 MiB) larger than L2; no flush",
                       "tile": [plan["tile_m"], plan["tile_n"], plan["tile_k"]], "stages": plan["stages"],
                       "group_m": plan["group_m"], "grid": plan["grid"]},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                         "frac": achieved / peak, "traffic": traffic_per_launch(plan=plan),
                         "peak_source": f"{peak_src} cuBLAS bf16 {peak_kind} (timed region {region_s:.2f} s of "
                                        f"back-to-back launches; FP16 dense rate equals BF16)",
                         "peak_burst": peak_burst, "frac_of_burst": achieved / peak_burst,
                         "peak_sustained": peak_sustained,
                         "frac_of_sustained": (achieved / peak_sustained) if peak_sustained else None,
                         "kernel_ms_mean": mean_launch, "kernel_ms_min": min(launch_ms),
                         # the per-clock denominator: SMs x 8192 FLOP/clk x SM clock
                         "per_clock_peak_at_max_clock": clock_peak_max,
                         "frac_of_per_clock_peak_at_max_clock": achieved / clock_peak_max,
                         "frac_per_clock": s8.get("frac_per_clock"),
                         "tensor_flop_per_clk_sm_measured": {"median": probe_med, "min": probe_lo, "max": probe_hi,
                                                             "how": "gemm_tensor_rate_probe: one CTA per SM, 65536 "
                                                                    "back-to-back 128x256x16 kind::f16 MMAs, clock64"},
                         "frac_per_clock_source": (f"8192^3 back to back for {args.sustained_leg:g} s: "
                                                   f"TFLOP/s / ({sms} SMs x {TENSOR_FLOP_PER_CLK_SM} FLOP/clk x "
                                                   f"median SM clock sampled inside the loop)") if s8 else None},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(dA.numel() * 2 + dB.numel() * 2),
                    "d2h_bytes_per_step": int(dC.numel() * 4), "steps": e2e_steps, "ms_per_step": e2e_ms,
                    "api": "gemm_f16_f32_host (pinned host buffers; 4x4 blocks pipelined over H2D, GEMM, D2H)"},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "secondary": {"workload": f"gemm_f16_f32 {m2}x{n2}x{k2}, seed 2, L2 flushed before each launch",
                          "value": sec_tflops, "unit": UNIT, "frac_of_burst": sec_tflops / peak_burst,
                          "ms_mean": sec_ms, "launches": n_sec,
                          "tile": [plan2["tile_m"], plan2["tile_n"], plan2["tile_k"]], "waves": plan2["waves"],
                          "frac_of_per_clock_peak_at_max_clock": sec_tflops / clock_peak_max},
            "cold_l2": {"workload": f"gemm_f16_f32 {M}x{N}x{K}, seed {SEED}, L2 flushed (512 MiB written) "
                                    f"before each launch", "value": flops / (cold_ms * 1e-3) / 1e12, "unit": UNIT,
                        "ms_mean": cold_ms, "launches": len(cold)},
            "sustained": sustained,
            "kernel_hash": kernel_hash(),
        }
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(A16, B16, args.cpu_seconds)
        print(json.dumps(line), flush=True)
    return 0


CONFIG_SHAPES = [
    ("square 256^3, seed 0", (256, 256, 256)),
    ("ragged (300,200,150), seed 1", (300, 200, 150)),
    ("ragged (129,65,33), seed 1", (129, 65, 33)),
    ("ragged (1,1000,64), seed 1", (1, 1000, 64)),
    ("ragged (17,4097,31), seed 1", (17, 4097, 31)),
    ("square 4096^3, seed 2", (4096, 4096, 4096)),
    ("wave sweep 1792^3, seed 3", (1792, 1792, 1792)),
    ("wave sweep 1793^3, seed 3", (1793, 1793, 1793)),
    ("wave sweep 2048^3, seed 3", (2048, 2048, 2048)),
    ("wave sweep 3072^3, seed 3", (3072, 3072, 3072)),
    ("wave sweep 6144^3, seed 3", (6144, 6144, 6144)),
    ("large 8192^3, seed 4", (8192, 8192, 8192)),
    ("large 16384x16384x4096, seed 4", (16384, 16384, 4096)),
    ("skinny 128x16384x16384, seed 4", (128, 16384, 16384)),
]


def run_configs(args):
    """Every workload shape: median device time over launches (L2 flushed before each launch
    when the operands fit in L2), TFLOP/s, operand+result GB/s, and the plan's tile waves."""
    import numpy as np
    import torch

    import tensor_core_tiled_gb300 as tct
    from tensor_core_tiled_gb300 import build as lib_build

    lib_build.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    peak_burst, _, peak_src = peaks()
    hbm = None
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            hbm = float(json.load(f)["hbm_gbs"])
    except (OSError, KeyError, ValueError):
        pass
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    for label, (M, N, K) in CONFIG_SHAPES:
        g = torch.Generator(device=dev).manual_seed(0)
        A = torch.randn(M, K, device=dev, generator=g).half()
        B = torch.randn(K, N, device=dev, generator=g).half()
        C = torch.empty(M, N, device=dev)
        for _ in range(3):
            tct.matmul(A, B, C)
        fits = (A.numel() + B.numel()) * 2 < 100e6
        reps = max(5, min(args.steps, 50))
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in pairs:
            if fits:
                flush.fill_(1.0)
            a.record()
            tct.matmul(A, B, C)
            b.record()
        torch.cuda.synchronize()
        ms = statistics.median([a.elapsed_time(b) for a, b in pairs])
        # the vendor library on the same operands and the same timing (FP16 in, FP32 out)
        cublas_ms = None
        try:
            for _ in range(3):
                torch.mm(A, B, out_dtype=torch.float32)
            for a, b in pairs:
                if fits:
                    flush.fill_(1.0)
                a.record()
                torch.mm(A, B, out_dtype=torch.float32)
                b.record()
            torch.cuda.synchronize()
            cublas_ms = statistics.median([a.elapsed_time(b) for a, b in pairs])
        except (TypeError, RuntimeError):
            pass
        pl = tct.gemm_f16_f32_plan(M, N, K, lda=K, ldb=N)
        tiles = pl["tiles"]
        slots = sms // pl["cta_group"]
        byts = 2 * (M * K + K * N) + 4 * M * N
        line = {"workload": label, "M": M, "N": N, "K": K, "us": ms * 1e3, "tflops": 2 * M * N * K / ms / 1e9,
                "frac_of_burst": 2 * M * N * K / ms / 1e9 / peak_burst, "gbs": byts / ms / 1e6,
                "frac_of_hbm": (byts / ms / 1e6 / hbm) if hbm else None,
                "cta_group": pl["cta_group"], "tile": [pl["tile_m"], pl["tile_n"]], "stages": pl["stages"],
                "tiles": tiles, "units": pl["units"], "sm_slots": slots,
                "waves": -(-tiles // slots), "page_wave_utilization": tiles / (-(-tiles // slots) * slots),
                "split_tiles": pl["stream_k_tiles"], "effective_waves": pl["effective_waves"],
                "l2_flushed": fits, "repack": bool(pl["pack_a"] or pl["pack_b"]), "split_form": pl["split_form"],
                "cublas_us": cublas_ms * 1e3 if cublas_ms else None}
        print(json.dumps(line), flush=True)
        del A, B, C
    # operand storage and type at 8192^3: the four layouts of gemm_f32acc, FP16 then BF16
    n = 8192
    for dt in (torch.float16, torch.bfloat16):
        g = torch.Generator(device=dev).manual_seed(0)
        A = torch.randn(n, n, device=dev, generator=g).to(dt)
        B = torch.randn(n, n, device=dev, generator=g).to(dt)
        At, Bt = A.t().contiguous(), B.t().contiguous()
        C = torch.empty(n, n, device=dev)
        for name, a, b in (("NN", A, B), ("TN", At.t(), B), ("NT", A, Bt.t()), ("TT", At.t(), Bt.t())):
            for _ in range(3):
                tct.matmul(a, b, C)
            reps = max(5, min(args.steps, 30))
            pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
            for e0, e1 in pairs:
                e0.record()
                tct.matmul(a, b, C)
                e1.record()
            torch.cuda.synchronize()
            ms = statistics.median([e0.elapsed_time(e1) for e0, e1 in pairs])
            print(json.dumps({"workload": f"layout {name} {str(dt).split('.')[-1]} {n}^3", "us": ms * 1e3,
                              "tflops": 2 * n ** 3 / ms / 1e9, "frac_of_burst": 2 * n ** 3 / ms / 1e9 / peak_burst}),
                  flush=True)
        del A, B, At, Bt, C
    # epilogue variants at 8192^3 (gemm_ex): output type, alpha, beta * C, bias
    g = torch.Generator(device=dev).manual_seed(0)
    A = torch.randn(n, n, device=dev, generator=g).half()
    B = torch.randn(n, n, device=dev, generator=g).half()
    bias = torch.randn(n, device=dev, generator=g)
    for name, dt, kw in (("FP32 out", torch.float32, {}), ("FP16 out", torch.float16, {}),
                         ("BF16 out", torch.bfloat16, {}), ("alpha 0.5, FP32 out", torch.float32, {"alpha": 0.5}),
                         ("beta 1 (reads C), FP32 out", torch.float32, {"beta": 1.0}),
                         ("bias, FP32 out", torch.float32, {"bias": bias}),
                         ("beta 1, FP16 out", torch.float16, {"beta": 1.0}),
                         ("bias, BF16 out", torch.bfloat16, {"bias": bias})):
        C = torch.randn(n, n, device=dev, generator=g).to(dt)
        for _ in range(3):
            tct.gemm(A, B, C, **kw)
        reps = max(5, min(args.steps, 30))
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for e0, e1 in pairs:
            e0.record()
            tct.gemm(A, B, C, **kw)
            e1.record()
        torch.cuda.synchronize()
        ms = statistics.median([e0.elapsed_time(e1) for e0, e1 in pairs])
        print(json.dumps({"workload": f"epilogue {name} {n}^3", "us": ms * 1e3, "tflops": 2 * n ** 3 / ms / 1e9,
                          "frac_of_burst": 2 * n ** 3 / ms / 1e9 / peak_burst}), flush=True)
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK
    return 0


# Row-length sweep of the softmax: (M, N, leading dimension), 2^26 elements (256 MiB each
# way, above L2) unless stated; the last rows are not 16-byte aligned (ld = N + 1).
SOFTMAX_CONFIGS = [(4096, 1024, 1024)] + [((1 << 26) // n, n, n) for n in (
    128, 512, 1024, 2048, 4096, 8192, 16384, 32768, 65536, 131072, 262144, 1 << 20)] + [
    ((1 << 26) // 1000, 1000, 1001), ((1 << 26) // 20000, 20000, 20001)]


def run_softmax_configs(args):
    """Every softmax shape: median device time over launches (L2 flushed before each), GB/s of
    algorithmic traffic (read + write MN floats) and its fraction of the HBM copy peak."""
    import torch

    import tensor_core_tiled_gb300 as tct
    from tensor_core_tiled_gb300 import build as lib_build

    lib_build.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    peak, _ = hbm_peak()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    sp = torch.cuda.current_stream(dev).cuda_stream
    for M, N, ld in SOFTMAX_CONFIGS:
        g = torch.Generator(device=dev).manual_seed(0)
        X = torch.randn(M * ld, device=dev, generator=g)
        Y = torch.empty_like(X)

        def launch():
            st = tct.softmax_rows_f32(X.data_ptr(), Y.data_ptr(), M, N, ld, ld, sp)
            if st:
                raise tct.GemmError(st, "softmax_rows_f32")

        for _ in range(3):
            launch()
        reps = max(5, min(args.steps, 30))
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for e0, e1 in pairs:
            flush.fill_(1.0)
            e0.record()
            launch()
            e1.record()
        torch.cuda.synchronize()
        ms = statistics.median([e0.elapsed_time(e1) for e0, e1 in pairs])
        gbs = 8.0 * M * N / ms / 1e6
        print(json.dumps({"workload": f"softmax {M}x{N}" + (f" (ld {ld}, rows not 16-byte aligned)" if ld != N else ""),
                          "M": M, "N": N, "ld": ld, "us": ms * 1e3, "gbs": gbs, "frac_of_hbm": gbs / peak}), flush=True)
        del X, Y
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK
    return 0


# ---------------------------------------------------------------- softmax workload

def softmax_input(M, N, seed):
    import numpy as np
    from tensor_core_tiled_gb300 import inputs
    return inputs.normal_f32(np.random.default_rng(seed), M, N)


def _softmax_oracle_sample(X, rows):
    """Time the oracle's softmax on rows [0, rows); returns (seconds, algorithmic bytes)."""
    import oracle
    t0 = time.perf_counter()
    oracle.softmax_rows_f32(X[:rows])
    return time.perf_counter() - t0, 2.0 * 4 * rows * X.shape[1]


def _softmax_rows_for(X, seconds):
    import oracle
    oracle.build()
    probe = min(X.shape[0], 256)
    s, _ = _softmax_oracle_sample(X, probe)
    return int(max(1, min(X.shape[0], probe * seconds / max(s, 1e-9))))


def _softmax_baseline_record(X, rows, secs, byts):
    import oracle
    M, N = X.shape
    return {"value": byts / secs / 1e9, "unit": SOFTMAX_UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"rows 0..{rows - 1} of the {M}x{N} seed-{SOFTMAX_SEED} matrix ({rows * N} outputs in "
                      f"{secs:.2f} s), FP64 arithmetic, all host threads"}


def softmax_config(M, N):
    return {"workload": f"softmax_rows_f32 {M}x{N}, X N(0,1) FP32 from seed {SOFTMAX_SEED}, row softmax",
            "M": M, "N": N, "l2": "input and output (256 MiB each) larger than L2; no flush"}


def run_softmax_reference(args):
    rank, _, _ = dist_env()
    if rank != 0:
        return 0
    M, N = SOFTMAX_WORKLOAD
    X = softmax_input(M, N, SOFTMAX_SEED)
    per_step = max(0.02, 6.0 * args.cpu_seconds / max(1, args.steps + args.warmup))
    rows = _softmax_rows_for(X, per_step)
    for _ in range(args.warmup):
        _softmax_oracle_sample(X, rows)
    secs = byts = 0.0
    for _ in range(args.steps):
        s, b = _softmax_oracle_sample(X, rows)
        secs += s
        byts += b
    value = byts / secs / 1e9
    rec = _softmax_baseline_record(X, rows, secs / args.steps, byts / args.steps)
    rec["value"] = value
    line = {"impl": "reference", "metric": SOFTMAX_METRIC, "value": value, "unit": SOFTMAX_UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": softmax_config(M, N), "cpu_baseline": rec,
            "e2e": {"value": value, "unit": SOFTMAX_UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_softmax(args):
    import torch

    import tensor_core_tiled_gb300 as tct
    from tensor_core_tiled_gb300 import build as lib_build

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        dist = None
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    if rank == 0:
        lib_build.build()
    if dist:
        dist.barrier()
    tct.load()

    M, N = SOFTMAX_WORKLOAD
    X = softmax_input(M, N, SOFTMAX_SEED)
    hX = torch.from_numpy(X).pin_memory()
    dX = hX.to(dev)
    dY = torch.empty_like(dX)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    byts = 2.0 * 4 * M * N

    def launch(src=dX, dst=dY, m=M, n=N):
        st = tct.softmax_rows_f32(src.data_ptr(), dst.data_ptr(), m, n, n, n, sp)
        if st:
            raise tct.GemmError(st, "softmax_rows_f32")

    for _ in range(max(3, args.warmup)):
        launch()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_host0 = time.time()
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for e0, e1 in evs:
        e0.record(stream)
        launch()
        e1.record(stream)
    g1.record(stream)
    torch.cuda.synchronize()
    t_host1 = time.time()
    if dist:
        dist.barrier()
    total_ms = g0.elapsed_time(g1)
    launch_ms = [a.elapsed_time(b) for a, b in evs]
    sampler.stop()
    clocks = sampler.summary(t_host0, t_host1)
    if dist:
        total_ms = dist_max(total_ms, dist, dev)
    ms_per_step = total_ms / args.steps
    value = world * byts / (ms_per_step * 1e-3) / 1e9
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK

    # end to end through the host-buffer call: softmax_rows_f32_host copies X from pinned
    # memory, softmaxes it and copies Y back (row blocks pipelined), inside the timed region
    hY = torch.empty_like(hX).pin_memory()
    e2e_steps = max(1, min(args.steps, 20))

    def e2e_step():
        st = tct.softmax_rows_f32_host(hX.data_ptr(), hY.data_ptr(), M, N, N, N, sp)
        if st:
            raise tct.GemmError(st, "softmax_rows_f32_host")

    for _ in range(3):  # warm-up: pools, copy streams and the host link settled
        e2e_step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    x0 = torch.cuda.Event(enable_timing=True)
    x1 = torch.cuda.Event(enable_timing=True)
    x0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    x1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = x0.elapsed_time(x1) / e2e_steps
    if dist:
        e2e_ms = dist_max(e2e_ms, dist, dev)
    e2e_value = world * byts / (e2e_ms * 1e-3) / 1e9

    # the page's own case, 4096 x 1024 (16 MiB each way, inside L2): L2 flushed per launch
    m2, n2 = 4096, 1024
    sX = torch.from_numpy(softmax_input(m2, n2, SOFTMAX_SEED)).to(dev)
    sY = torch.empty_like(sX)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    for _ in range(5):
        launch(sX, sY, m2, n2)
    n_sec = max(5, min(args.steps, 100))
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_sec)]
    for a, b in pairs:
        flush.fill_(1.0)
        a.record(stream)
        launch(sX, sY, m2, n2)
        b.record(stream)
    torch.cuda.synchronize()
    sec_ms = statistics.mean([a.elapsed_time(b) for a, b in pairs])
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK

    peak, peak_src = hbm_peak()
    mean_launch = statistics.mean(launch_ms)
    achieved = byts / (mean_launch * 1e-3) / 1e9
    line = None
    if rank == 0:
        line = {
            "metric": SOFTMAX_METRIC, "value": value, "unit": SOFTMAX_UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": dict(softmax_config(M, N), parallelism=f"replicas x{world}"),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak,
                         "traffic": traffic_per_launch("softmax_65536x1024_dram_traffic.json", SOFTMAX_SOURCES),
                         "peak_source": f"{peak_src} HBM copy bandwidth (read + write bytes)",
                         "algorithmic_bytes_per_launch": byts,
                         "kernel_ms_mean": mean_launch, "kernel_ms_min": min(launch_ms)},
            "e2e": {"value": e2e_value, "unit": SOFTMAX_UNIT, "h2d_bytes_per_step": int(dX.numel() * 4),
                    "d2h_bytes_per_step": int(dY.numel() * 4), "steps": e2e_steps, "ms_per_step": e2e_ms,
                    "api": "softmax_rows_f32_host (pinned host buffers; row blocks pipelined over H2D, softmax, D2H)"},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "secondary": {"workload": f"softmax_rows_f32 {m2}x{n2} (the page's case), seed {SOFTMAX_SEED}, "
                                      f"L2 flushed before each launch",
                          "value": 2.0 * 4 * m2 * n2 / (sec_ms * 1e-3) / 1e9, "unit": SOFTMAX_UNIT,
                          "us_mean": sec_ms * 1e3, "launches": n_sec},
            "kernel_hash": kernel_hash(SOFTMAX_SOURCES),
        }
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            rows = _softmax_rows_for(X, args.cpu_seconds)
            secs, b = _softmax_oracle_sample(X, rows)
            line["cpu_baseline"] = _softmax_baseline_record(X, rows, secs, b)
        print(json.dumps(line), flush=True)
    return 0


SPLIT_SHAPES = [(256, 256, 65536), (128, 512, 32768), (512, 512, 16384), (1024, 1024, 32768), (1024, 1024, 8192),
                (128, 4096, 8192), (256, 256, 4096), (1792, 1792, 1792), (2048, 2048, 2048), (4096, 4096, 4096),
                (8192, 8192, 8192), (128, 16384, 16384)]
SPLIT_FORMS = (("whole tiles", {"stream_k": 1}), ("two-part split tail", {"stream_k": 2}),
               ("stream-K", {"stream_k": 3}), ("planner's choice", {}))


def run_splits(args):
    """Each work-split form on shapes where they differ: median device time over launches (L2
    flushed before each launch when the operands fit in L2), with the plan's form, the units
    sharing the stream-K k-blocks and the most pieces one tile is cut into."""
    import torch

    import tensor_core_tiled_gb300 as tct
    from tensor_core_tiled_gb300 import build as lib_build

    lib_build.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    for M, N, K in SPLIT_SHAPES:
        g = torch.Generator(device=dev).manual_seed(0)
        A = torch.randn(M, K, device=dev, generator=g).half()
        B = torch.randn(K, N, device=dev, generator=g).half()
        C = torch.empty(M, N, device=dev)
        fits = (A.numel() + B.numel()) * 2 < 100e6
        for name, opts in SPLIT_FORMS:
            try:
                pl = tct.gemm_f16_f32_plan(M, N, K, **opts)
            except tct.GemmError as e:
                print(json.dumps({"M": M, "N": N, "K": K, "form": name, "unavailable": str(e)}), flush=True)
                continue
            for _ in range(3):
                tct.matmul(A, B, C, **opts)
            reps = max(5, min(args.steps, 30))
            pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
            for a, b in pairs:
                if fits:
                    flush.fill_(1.0)
                a.record()
                tct.matmul(A, B, C, **opts)
                b.record()
            torch.cuda.synchronize()
            ms = statistics.median([a.elapsed_time(b) for a, b in pairs])
            print(json.dumps({"M": M, "N": N, "K": K, "form": name, "us": ms * 1e3,
                              "tflops": 2 * M * N * K / ms / 1e9, "cta_group": pl["cta_group"],
                              "tile": [pl["tile_m"], pl["tile_n"]], "split_form": pl["split_form"],
                              "split_tiles": pl["stream_k_tiles"], "sk_units": pl["sk_units"],
                              "pieces_or_parts": pl["split_parts_per_unit"], "l2_flushed": fits}), flush=True)
        del A, B, C
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK
    return 0


def run_sustained(args):
    """4096^3 and 8192^3 launched back to back for args.sustained seconds each (after a
    second of warm-up): whole-loop TFLOP/s by CUDA events, with the median SM clock, the
    largest power draw and the throttle reasons nvidia-smi reported during the loop."""
    import torch

    import tensor_core_tiled_gb300 as tct
    from tensor_core_tiled_gb300 import build as lib_build

    lib_build.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    peak_burst, peak_sus, _ = peaks()
    sampler = ClockSampler(0)
    sampler.start()
    try:
        for n, seed in ((4096, 2), (8192, SEED)):
            g = torch.Generator(device=dev).manual_seed(seed)
            A = torch.randn(n, n, device=dev, generator=g).half()
            B = torch.randn(n, n, device=dev, generator=g).half()
            C = torch.empty(n, n, device=dev)
            ms, launches, clk = back_to_back(lambda: tct.matmul(A, B, C), args.sustained, sampler)
            tflops = 2 * n ** 3 / ms / 1e9
            mhz = clk.get("sm_mhz")
            print(json.dumps({"workload": f"gemm_f16_f32 {n}^3 back to back", "seconds": args.sustained,
                              "launches": launches, "ms_per_launch": ms, "tflops": tflops,
                              "frac_of_sustained": tflops / peak_sus if peak_sus else None,
                              "frac_of_burst": tflops / peak_burst,
                              "frac_per_clock": tflops / per_clock_peak_tflops(sms, mhz) if mhz else None,
                              "clocks": clk, "device_status": tct.gemm_f16_f32_get_error()}), flush=True)
            del A, B, C
    finally:
        sampler.stop()


def run_case(args):
    """One shape, a few launches: per-launch device times (CUDA events), the launch plan and
    the device status, as one JSON line.  Inputs are N(0,1) FP16 drawn on the device, so the
    command starts quickly; meant for profiling one kernel on a chosen shape and for sweeps."""
    import torch

    import tensor_core_tiled_gb300 as tct
    from tensor_core_tiled_gb300 import build as lib_build

    lib_build.build()
    torch.cuda.set_device(0)
    M, N, K = args.case
    g = torch.Generator(device="cuda").manual_seed(0)
    A = torch.randn(M, K, device="cuda", generator=g).half()
    B = torch.randn(K, N, device="cuda", generator=g).half()
    C = torch.empty(M, N, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES // 4, device="cuda") if args.flush_l2 else None
    opts = dict(tile_n=args.tile_n, stages=args.stages, group_m=args.group_m, max_ctas=args.max_ctas,
                cta_group=args.cta_group, stream_k=args.stream_k)
    opts = {k: v for k, v in opts.items() if v}
    for _ in range(args.warmup):
        tct.matmul(A, B, C, **opts)
    torch.cuda.synchronize()
    times = []
    for _ in range(args.launches):
        if flush is not None:
            flush.fill_(1.0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        tct.matmul(A, B, C, **opts)
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    st = tct.gemm_f16_f32_get_error()
    flops = 2.0 * M * N * K
    best = min(times)
    plan = tct.gemm_f16_f32_plan(M, N, K, **opts)
    print(json.dumps({"shape": [M, N, K], "opts": opts, "ms": times, "best_ms": best,
                      "median_ms": statistics.median(times), "tflops_best": flops / best / 1e9,
                      "tflops_median": flops / statistics.median(times) / 1e9, "plan": plan,
                      "device_status": st}), flush=True)
    if st != tct.GEMM_OK:
        raise SystemExit(f"device status {st}")
    return 0


def main():
    args = parse()
    if args.workload == "softmax":
        if args.impl == "reference":
            return run_softmax_reference(args)
        return run_softmax_configs(args) if args.configs else run_softmax(args)
    if args.impl == "reference":
        return run_reference(args)
    if args.case:
        return run_case(args)
    if args.splits:
        return run_splits(args)
    if args.configs:
        return run_configs(args)
    if args.sustained > 0:
        return run_sustained(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
