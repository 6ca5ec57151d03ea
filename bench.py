#!/usr/bin/env python3
"""Throughput of the KroQuant MXFP4 activation quantizer on one GB300 (or N,
one process per GPU, weak scaling).

A step quantizes the FLUX.1-schnell-shaped layer pair of "KroQuant:
Kronecker-Structured Block Transforms for Efficient Post-Training
Quantization of Diffusion Transformers" (Sec. 4.1 models, Table 4 widths):
m = 4608 tokens (4096 image + 512 text) at d = 3072 and at d = 12288 (the
FFN-down input), bf16 activations with outlier channels (synthetic: per-token
lognormal(0, 0.7) x N(0, 1), 1 % of channels x U[30, 300]) and random
unit-determinant LU Kronecker factors per layer, quantized to MXFP4 with the
scale factors in the 128x4 tiled layout of block-scaled MMA.

Metric: GB/s moved = m * d * (2 + 1/2 + 1/32) bytes / time (bf16 read, packed
FP4 and E8M0 written), and the fraction of the measured HBM copy bandwidth.
Four input/output sets rotate so that no step reads data a recent step left
in L2 (~710 MB footprint against a 126 MB L2).

--impl reference times the CPU oracle (fp64, all host cores) on a bounded
row sample of the same workload and prints the same line.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KroQuant MXFP4 quantizer GB/s and % HBM peak; speedup vs diag-scale quantizer"
LAYERS = (("flux_3072", 4608, 3072), ("flux_ffn_down", 4608, 12288))
DOMINANT = 1                        # the d = 12288 launch dominates the step
SETS = 4
ROUND = 8 * SETS                    # steps per replay of a layer's CUDA graph
FALLBACK_HBM_GBS = 6800.0


def algo_bytes(m: int, d: int) -> float:
    """bf16 read + packed E2M1 written + one E8M0 byte per 32 elements."""
    return m * d * 2 + m * d / 2 + m * d / 32


STEP_BYTES = sum(algo_bytes(m, d) for _, m, d in LAYERS)


def round_lengths(steps: int) -> list:
    """The timed region's structure: rounds of min(steps left, ROUND) steps;
    each round replays every layer's CUDA graph of that many launches, so the
    launches run back to back in the same way whatever the step count."""
    out, left = [], steps
    while left > 0:
        out.append(min(left, ROUND))
        left -= out[-1]
    return out


def algo_bytes_dual(m: int, d: int) -> float:
    """kq_quantize_mxfp4_dual: the MXFP4 outputs plus the bf16 side output A T."""
    return algo_bytes(m, d) + m * d * 2


STEP_BYTES_DUAL = sum(algo_bytes_dual(m, d) for _, m, d in LAYERS)


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--variant", choices=("butterfly", "umma", "k2"), default="umma",
                    help="KroQuant kernel: tcgen05 on expanded records (umma, default), "
                         "tcgen05 building the records from the raw factors (k2), or the "
                         "CUDA-core butterfly")
    ap.add_argument("--isolated", type=int, default=20,
                    help="single-launch measurements of the dominant layer (isolated_launch)")
    ap.add_argument("--no-baselines", action="store_true",
                    help="skip the diagonal / Hadamard / bare-quantizer side measurements")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU time budget of the oracle baseline sample")
    ap.add_argument("--gemm", action="store_true",
                    help="table of the W4A4 consumer product (kind::mxf4) on the layer shapes")
    ap.add_argument("--profile", choices=("kroquant", "dual", "diag", "hadamard", "identity",
                                          "fwht", "gemm"),
                    help="profiling case for ncu: run one quantizer a few times and exit")
    ap.add_argument("--m", type=int, default=9216, help="rows of the profiling case")
    ap.add_argument("--d", type=int, default=12288, help="channels of the profiling case")
    ap.add_argument("--n", type=int, default=3072, help="output channels of the gemm profiling case")
    ap.add_argument("--launches", type=int, default=3, help="launches of the profiling case")
    ap.add_argument("--table", action="store_true",
                    help="per-launch medians of every kernel on every config shape (markdown)")
    ap.add_argument("--table3-only", action="store_true",
                    help="with --table: only the pages' Table 3 comparison (bf16 and fp16 input)")
    ap.add_argument("--table-reps", type=int, default=50, help="graph replays per kernel")
    ap.add_argument("--table-warmup", type=int, default=100, help="warm-up launches per kernel")
    ap.add_argument("--cpu-rate", nargs=3, type=int, metavar=("M", "D", "SECONDS"),
                    help="print the oracle's GB/s on an M x D KroQuant layer (row sample of "
                         "about SECONDS of CPU work; OMP_NUM_THREADS sets the cores)")
    return ap.parse_args()


# --------------------------------------------------------------- distributed --

class Dist:
    def __init__(self, use_cuda: bool):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if use_cuda else "gloo"
            if use_cuda:
                import torch
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            if self.pg.get_backend() == "nccl":
                import torch
                self.pg.barrier(device_ids=[torch.cuda.current_device()])
            else:
                self.pg.barrier()

    def max(self, x: float) -> float:
        return self._reduce(x, "max")

    def sum(self, x: float) -> float:
        return self._reduce(x, "sum")

    def _reduce(self, x: float, op: str) -> float:
        if self.pg is None:
            return x
        import torch
        dev = "cuda" if self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX if op == "max" else self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# ------------------------------------------------------------------ helpers --

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def fp4_peak():
    """Dense FP4 tensor peak: the measured bf16 GEMM rate times the nominal
    FP4 / bf16 ratio of the part (13.5 / 2.25 PFLOP/s)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]) * 6.0, "measured bf16 x 6"
    except (OSError, KeyError, ValueError):
        return 1900.0 * 6.0, "fallback bf16 x 6"


def gemm_case(m: int, n: int, k: int, seed: int, dev):
    """Operands of an m x n x k W4A4 product: random packed codes and E8M0
    bytes in [118, 136] (tiled layout), plus bf16 A and W of the same shapes
    for the reference product."""
    import numpy as np
    import torch
    from w4a4_mxfp4_activation_gb300 import kq, synth
    qa = torch.from_numpy(synth.packed_codes(m, k, seed)).to(dev)
    qw = torch.from_numpy(synth.packed_codes(n, k, seed + 1)).to(dev)
    sfa = torch.from_numpy(synth.scale_bytes(kq.kq_sf_bytes(m, k, 1), 1, seed + 2, 118, 136)
                           .reshape(-1)).to(dev)
    sfw = torch.from_numpy(synth.scale_bytes(kq.kq_sf_bytes(n, k, 1), 1, seed + 3, 118, 136)
                           .reshape(-1)).to(dev)
    a = torch.from_numpy(synth.activations(m, k, seed + 4, "flux").view(np.int16)).to(dev) \
        .view(torch.bfloat16)
    w = torch.from_numpy(synth.weights(n, k, seed + 5).view(np.int16)).to(dev).view(torch.bfloat16)
    return qa, sfa, qw, sfw, a, w


def time_launches(fn, stream, reps: int = 20, rounds: int = 5) -> float:
    """Median over `rounds` CUDA-event brackets of `reps` back-to-back calls
    (a CUDA graph of them) on `stream`: microseconds per call."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(3):
            fn()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(reps):
                fn()
        g.replay()
        stream.synchronize()
        out = []
        for _ in range(rounds):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            stream.synchronize()
            out.append(a.elapsed_time(b) * 1e3 / reps)
    return statistics.median(out)


def kernel_source_hash() -> str:
    """Hash of the sources that define the dominant kernel (the tcgen05
    quantizer): its device code, its launch configuration, the entry points
    that build its tensor maps and choose the path, and the build script
    that holds the compile command."""
    h = hashlib.sha256()
    pkg = os.path.join(ROOT, "w4a4_mxfp4_activation_gb300")
    csrc = os.path.join(pkg, "csrc")
    files = [os.path.join(csrc, f) for f in ("kq_umma.cu", "kq_device.cuh", "kq_internal.h",
                                             "kq_records.h", "kq_api.cu")]
    files.append(os.path.join(pkg, "build.py"))
    for path in files:
        h.update(os.path.basename(path).encode())
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        with open(path) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 4 and parts[0] == workload and parts[1] == kernel_source_hash():
                    return float(parts[3])
    except OSError:
        pass
    return None


_NVML_POLLER = r"""
import ctypes, sys, time
uuid, path = sys.argv[1], sys.argv[2]
L = ctypes.CDLL("libnvidia-ml.so.1")
assert L.nvmlInit_v2() == 0
h = ctypes.c_void_p()
assert L.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) == 0
reasons = getattr(L, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
    L.nvmlDeviceGetCurrentClocksThrottleReasons
mhz, mx, bits = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
assert L.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0
with open(path, "w", buffering=1) as f:
    f.write("ready\n")
    while True:
        t = time.monotonic()
        if (L.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0 and
                reasons(h, ctypes.byref(bits)) == 0):
            f.write(f"{t} {mhz.value} {mx.value} {bits.value}\n")
        time.sleep(0.0002)
"""


class ClockSampler:
    """SM clock and clock-event reasons of the benchmarked GPU, sampled while
    alive by a child process that polls NVML (read-only queries of the
    driver's libnvidia-ml) as fast as it answers; falls back to nvidia-smi
    writing to a file.  Samples carry time.monotonic() stamps, so those inside
    a window (the timed region) can be told from the rest; a separate process
    keeps sampling while this one waits on the GPU."""

    # nvmlClocksEventReasons bits
    REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                   "hw_thermal_slowdown": 0x40}
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None, out_dir: str | None = None):
        import tempfile
        self.uuid = uuid
        self.samples = []            # (monotonic time or None, sm MHz, max MHz, reason bits)
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".txt", dir=out_dir)
        os.close(fd)
        self.source = None
        self.proc = None
        if uuid:
            try:
                self.proc = subprocess.Popen([sys.executable, "-c", _NVML_POLLER, uuid, self.path],
                                             stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
                self.source = "nvml"
                for _ in range(100):                     # until its first line (<= 5 s)
                    if self.proc.poll() is not None or os.path.getsize(self.path) > 0:
                        break
                    time.sleep(0.05)
                if self.proc.poll() is not None:
                    self.proc = None
            except OSError:
                self.proc = None
        if self.proc is None:
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                     "-lms", "20", "-f", self.path], stdout=subprocess.DEVNULL,
                    stderr=subprocess.DEVNULL)
                self.source = "nvidia-smi"
            except OSError:
                self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
        try:
            with open(self.path) as f:
                lines = f.read().splitlines()
            os.unlink(self.path)
        except OSError:
            lines = []
        for line in lines:
            if self.source == "nvml":
                fl = line.split()
                if len(fl) == 4:
                    self.samples.append((float(fl[0]), float(fl[1]), float(fl[2]), int(fl[3])))
                continue
            fl = [x.strip() for x in line.split(",")]
            if len(fl) < 7 or (self.uuid and self.uuid not in fl[0] and fl[0] not in self.uuid):
                continue
            try:
                bits = sum(b for (name, b), v in zip(self.REASON_BITS.items(),
                                                     (fl[6], fl[3], fl[5], fl[4]))
                           if v.lower().startswith("active"))
                self.samples.append((None, float(fl[1]), float(fl[2]), bits))
            except ValueError:
                continue

    def summary(self, window=None):
        """Median SM clock, max clock and the throttle reasons seen, over the
        samples inside window = (t0, t1) (time.monotonic() seconds), or all."""
        pts = [x for x in self.samples
               if window is None or x[0] is None or window[0] <= x[0] <= window[1]]
        if not pts:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "source": self.source}
        reasons = sorted(name for name, b in self.REASON_BITS.items()
                         if any(p[3] & b for p in pts))
        return {"sm_mhz": statistics.median(p[1] for p in pts),
                "sm_max_mhz": max(p[2] for p in pts), "reasons": reasons, "samples": len(pts),
                "source": self.source}


def device_uuid(dev) -> str | None:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# ------------------------------------------------------------ CPU oracle --

def cpu_oracle_rate(rows_per_layer: int, seed: int = 0):
    """Times the oracle (transform + quantize, fp64, OpenMP over host cores)
    on the first rows of both layers; returns (GB/s, seconds, bytes)."""
    import numpy as np
    from oracle import kq_oracle as O
    from w4a4_mxfp4_activation_gb300 import synth
    inputs = []
    for i, (_, m, d) in enumerate(LAYERS):
        r = min(rows_per_layer, m)
        A = synth.activations(r, d, synth.SEED_A + 3 + seed, "flux")
        lu = synth.lu_params(d // 32, synth.SEED_FACTORS + 3 + i)
        F = O.lu_to_factors(lu.astype(np.float64), +1).astype(np.float32).astype(np.float64)
        inputs.append((A, d, F, r))
    t0 = time.perf_counter()
    nbytes = 0.0
    for A, d, F, r in inputs:
        y, bound = O.transform(A, d, "kron", F)
        O.quantize(y, bound, O.SF_BLOCKED_128x4)
        nbytes += algo_bytes(r, d)
    dt = time.perf_counter() - t0
    return nbytes / dt / 1e9, dt, nbytes


def cpu_cores() -> int:
    n = os.environ.get("OMP_NUM_THREADS")
    return int(n) if n and n.isdigit() else (os.cpu_count() or 1)


def cpu_baseline(budget_s: float):
    """The oracle on the host cores: a row sample of the step sized to about
    budget_s seconds; when the whole step takes less, whole steps repeated."""
    _, t16, _ = cpu_oracle_rate(16)
    rows = max(16, min(LAYERS[0][1], int(16 * budget_s / max(t16, 1e-3))))
    rate, dt, nbytes = cpu_oracle_rate(rows)
    passes = 1
    if rows == LAYERS[0][1] and dt < 0.5 * budget_s:
        extra = max(1, int((budget_s - dt) / max(dt, 1e-3)))
        for p in range(extra):
            _, d2, n2 = cpu_oracle_rate(rows, seed=1 + p)
            dt += d2
            nbytes += n2
        passes += extra
        rate = nbytes / dt / 1e9
    what = (f"all {rows} rows" if rows == LAYERS[0][1] else f"first {rows} rows")
    return {"value": round(rate, 4), "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{what} of each FLUX layer (m=4608, d=3072 and 12288), {passes} pass(es), "
                      f"{dt:.1f} s of CPU work"}


def run_reference(args, dist: Dist):
    if dist.rank != 0:
        return
    W, K = args.warmup, args.steps
    _, t16, _ = cpu_oracle_rate(16)
    per_step = 90.0 / max(K + W, 1)
    rows = max(1, min(LAYERS[0][1], int(16 * per_step / max(t16, 1e-6))))
    for w in range(W):
        cpu_oracle_rate(rows, seed=w)
    total_t, total_b = 0.0, 0.0
    for k in range(K):
        _, dt, nb = cpu_oracle_rate(rows, seed=k)
        total_t += dt
        total_b += nb
    value = total_b / total_t / 1e9
    line = {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": K, "warmup": W, "ms_per_step": round(1e3 * total_t / K, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": "flux_layer_pair_row_sample", "m": 4608, "d": [3072, 12288],
                       "rows_per_layer_per_step": rows, "transform": "kroquant",
                       "sf_layout": "blocked_128x4"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cpu_cores(),
                             "kind": "oracle",
                             "sample": f"first {rows} rows of each FLUX layer per step"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU --

def run_ours(args, dist: Dist):
    import numpy as np
    import torch
    from w4a4_mxfp4_activation_gb300 import kq, synth

    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.Stream(device=dev)
    layout = kq.KQ_SF_BLOCKED_128x4

    # ---- inputs resident in HBM: SETS rotating sets per layer
    A, Q, SF, F, KX = [], [], [], [], []
    host_A = []
    for li, (_, m, d) in enumerate(LAYERS):
        bits = synth.activations(m, d, synth.SEED_A + 3 + 100 * dist.rank + li, "flux")
        host = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).pin_memory()
        host_A.append(host)
        base = host.to(dev)
        A.append([torch.roll(base, shifts=137 * s, dims=0).contiguous() for s in range(SETS)])
        Q.append([torch.empty((m, d // 2), dtype=torch.uint8, device=dev) for _ in range(SETS)])
        SF.append([torch.empty(kq.kq_sf_bytes(m, d, layout), dtype=torch.uint8, device=dev)
                   for _ in range(SETS)])
        fac = kq.kq_lu_to_factors(synth.lu_params(d // 32, synth.SEED_FACTORS + 3 + li), +1)
        F.append(torch.from_numpy(fac).to(dev))
        KX.append(kq.kq_expand_blocks(F[-1], kq.KQ_K_BF16X3))
    torch.cuda.synchronize()

    def launch(kind, li, s):
        _, m, d = LAYERS[li]
        if kind == "kroquant":
            kind = args.variant
        if kind == "butterfly":
            kq.kq_quantize_mxfp4(A[li][s], d, factors=F[li], layout=layout, q=Q[li][s],
                                 sf=SF[li][s], variant=kq.VARIANT_BUTTERFLY, stream=stream)
        elif kind == "umma":
            kq.kq_quantize_mxfp4(A[li][s], d, K_expanded=KX[li], layout=layout, q=Q[li][s],
                                 sf=SF[li][s], stream=stream)
        elif kind == "k2":
            kq.kq_quantize_mxfp4(A[li][s], d, factors=F[li], layout=layout, q=Q[li][s],
                                 sf=SF[li][s], variant=kq.VARIANT_K2, stream=stream)
        elif kind == "dual":
            kq.kq_quantize_mxfp4_dual(A[li][s], KX[li], d, layout=layout, q=Q[li][s],
                                      sf=SF[li][s], at=AT[li][s], stream=stream)
        elif kind == "diag":
            kq.kq_smooth_quantize_mxfp4(A[li][s], DIAG[li], d, layout=layout, q=Q[li][s],
                                        sf=SF[li][s], stream=stream)
        elif kind == "hadamard":
            kq.kq_hadamard_quantize_mxfp4(A[li][s], d, layout=layout, q=Q[li][s], sf=SF[li][s],
                                          stream=stream)
        else:
            kq.kq_quantize_mxfp4(A[li][s], d, layout=layout, q=Q[li][s], sf=SF[li][s],
                                 stream=stream)

    DIAG = [torch.from_numpy(synth.smooth_scales(d)).to(dev) for _, _, d in LAYERS]
    # bf16 side outputs of the dual quantizer (allocated when it is measured)
    AT = [[None] * SETS for _ in LAYERS]

    def graphs_for(kind, lengths):
        """Per layer and per length L in `lengths`, a CUDA graph of L
        launches of that layer back to back, cycling through its SETS input
        sets, with programmatic dependent launch between them; and per
        (set, layer) a one-launch graph for the isolated measurement.  Each
        graph is replayed once here, untimed: a graph's first replay also
        uploads it to the device, a cost that no later replay pays."""
        per_len = {}
        single = [[None] * len(LAYERS) for _ in range(SETS)]
        with torch.cuda.stream(stream):
            for s in range(SETS):
                for li in range(len(LAYERS)):
                    launch(kind, li, s)              # warm the launch path before capture
            stream.synchronize()
            for n in sorted(set(x for x in lengths if x > 0)):
                per_len[n] = []
                for li in range(len(LAYERS)):
                    gr = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(gr, stream=stream):
                        for k in range(n):
                            launch(kind, li, k % SETS)
                    gr.replay()
                    per_len[n].append(gr)
            for s in range(SETS):
                for li in range(len(LAYERS)):
                    gr = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(gr, stream=stream):
                        launch(kind, li, s)
                    gr.replay()
                    single[s][li] = gr
        stream.synchronize()
        return per_len, single

    order = [DOMINANT] + [li for li in range(len(LAYERS)) if li != DOMINANT]

    def run_steps(g, steps, events):
        """`steps` steps (each: every layer once); with events, brackets
        every replay of the dominant layer's graph and returns the number of
        dominant launches inside each bracket."""
        per_len, _ = g
        counts = []
        for n in round_lengths(steps):
            for li in order:
                if events is not None and li == DOMINANT:
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    per_len[n][li].replay()
                    b.record(stream)
                    events.append((a, b))
                    counts.append(n)
                else:
                    per_len[n][li].replay()
        return counts

    def timed(kind, steps, warmup, per_launch=False, clocks=None):
        g = graphs_for(kind, round_lengths(steps) + round_lengths(warmup))
        events = [] if per_launch else None
        with torch.cuda.stream(stream):
            hw = time.monotonic()
            run_steps(g, warmup, None)
            stream.synchronize()
            dist.barrier()
            torch.cuda.synchronize()
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            h0 = time.monotonic()
            t0.record(stream)
            counts = run_steps(g, steps, events)
            t1.record(stream)
            stream.synchronize()
            h1 = time.monotonic()
            dist.barrier()
            torch.cuda.synchronize()
        ms = t0.elapsed_time(t1)
        # average duration of one dominant launch over the timed region
        launch_ms = ([sum(a.elapsed_time(b) for a, b in events) / sum(counts)]
                     if per_launch and events else [])
        return ms, launch_ms, (hw, h0, h1), g

    def isolated(kind, g, n):
        """Median CUDA-event time (ms) of one dominant-layer launch replayed
        alone (a one-launch graph between two events: no programmatic overlap
        with a neighbour, start-up and drain exposed), over n launches
        rotating through the input sets."""
        _, single = g
        out = []
        with torch.cuda.stream(stream):
            for k in range(n + 2):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                single[k % SETS][DOMINANT].replay()
                b.record(stream)
                b.synchronize()
                if k >= 2:
                    out.append(a.elapsed_time(b))
        return statistics.median(out)

    def launch_floor(n):
        """The same single-launch measurement on a one-element kernel: the
        time two events and a graph launch take with (almost) no work."""
        tiny = torch.zeros(1, device=dev)
        out = []
        with torch.cuda.stream(stream):
            tiny.add_(1.0)
            stream.synchronize()
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                tiny.add_(1.0)
            for k in range(n + 2):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                gr.replay()
                b.record(stream)
                b.synchronize()
                if k >= 2:
                    out.append(a.elapsed_time(b))
        return statistics.median(out)

    W, K = args.warmup, args.steps
    clock = ClockSampler(device_uuid(dev), os.environ.get("TMPDIR"))
    ms, launch_ms, (hw, h0, h1), g_main = timed("kroquant", K, W, per_launch=True)
    iso_ms = isolated("kroquant", g_main, max(3, args.isolated))
    h2 = time.monotonic()
    floor_ms = launch_floor(max(3, args.isolated))
    del g_main
    ms_max = dist.max(ms)
    total_bytes = dist.sum(STEP_BYTES * K)
    value = total_bytes / (ms_max * 1e-3) / 1e9
    peak, peak_src = hbm_peak()
    dom_m, dom_d = LAYERS[DOMINANT][1], LAYERS[DOMINANT][2]
    dom_ms = statistics.mean(launch_ms) if launch_ms else float("nan")
    achieved = algo_bytes(dom_m, dom_d) / (dom_ms * 1e-3) / 1e9
    workload = f"kq_quantize_mxfp4 {args.variant} m={dom_m} d={dom_d}"
    traffic = recorded_traffic(f"flux_ffn_down_{args.variant}")

    # ---- the dual quantizer (MXFP4 + the bf16 side output A T of the
    #      low-rank branch) on the same step
    side = None
    if not args.no_baselines:
        for li, (_, m, d) in enumerate(LAYERS):
            AT[li] = [torch.empty((m, d), dtype=torch.bfloat16, device=dev) for _ in range(SETS)]
        nd = max(ROUND, min(K, 8000))
        dms, dlaunch, _, _ = timed("dual", nd, W, per_launch=True)
        dms = dist.max(dms)
        side = {"metric": "kq_quantize_mxfp4_dual GB/s (MXFP4 + bf16 A T side output)",
                "value": round(dist.sum(STEP_BYTES_DUAL * nd) / (dms * 1e-3) / 1e9, 2),
                "unit": "GB/s", "bytes_per_element": 4.53125, "steps": nd,
                "ms_per_step": round(dms / nd, 5),
                "dominant_launch_ms": round(dlaunch[0], 5) if dlaunch else None,
                "dominant_frac": round(algo_bytes_dual(dom_m, dom_d) / (dlaunch[0] * 1e-3) / 1e9
                                       / peak, 4) if dlaunch else None,
                "traffic": recorded_traffic("flux_ffn_down_dual") if args.variant == "umma"
                else None}
        AT = [[None] * SETS for _ in LAYERS]
        torch.cuda.empty_cache()

    # ---- side measurements: the baselines built alongside
    # (same launch structure, steps and warm-up as the headline step; the
    #  diagonal kernel also in the isolated form)
    baselines = {}
    iso_diag_ms = None
    if not args.no_baselines:
        nb_steps = max(3, min(K, 4000))
        others = [v for v in ("butterfly", "umma", "k2") if v != args.variant]
        for kind in (*others, "diag", "hadamard", "identity"):
            bms, _, _, g = timed(kind, nb_steps, W)
            if kind == "diag":
                iso_diag_ms = isolated("diag", g, max(3, args.isolated))
            del g
            name = f"kroquant_{kind}" if kind in ("butterfly", "umma", "k2") else kind
            baselines[name] = round(STEP_BYTES * nb_steps / (dist.max(bms) * 1e-3) / 1e9, 2)
    clock.stop()
    # NVML answers in tens of ms, so few samples fall inside a timed region of
    # a millisecond: the reported window also holds the warm-up steps before
    # it and the isolated launches after it (the same kernels, back to back)
    clocks = dict(clock.summary((h0, h1)), window="timed region")
    if clocks["samples"] < 3:
        clocks = dict(clock.summary((hw, h2)), window="warm-up + timed region + isolated launches")
    run_clocks = clock.summary()
    if clocks["samples"] < 3:
        clocks = dict(run_clocks, window="whole run (no closer window holds 3 samples)")

    # ---- the consumer of the quantizer's output: the W4A4 product of the
    #      FFN-down layer (A_q: this step's quantized activations, 4608 x
    #      12288; W_q: 3072 x 12288 random codes and scales) on the FP4 tensor
    #      cores, with the bf16-dequantization route and the bf16 reference
    #      product A W^T for context
    consumer = None
    if not args.no_baselines:
        gm, gn, gk = dom_m, 3072, dom_d
        _, _, qw, sfw, ga, gw = gemm_case(gm, gn, gk, 9000 + dist.rank, dev)
        cq = torch.empty((gm, gn), dtype=torch.float32, device=dev)
        qa, sfa = Q[DOMINANT][0], SF[DOMINANT][0]
        us_fp4 = time_launches(lambda: kq.kq_w4a4_gemm(qa, sfa, qw, sfw, gm, gn, gk, c=cq,
                                                       stream=stream), stream)
        us_deq = time_launches(lambda: kq.kq_w4a4_gemm(qa, sfa, qw, sfw, gm, gn, gk, c=cq,
                                                       variant=kq.GEMM_DEQUANT_BF16,
                                                       stream=stream), stream, reps=4, rounds=3)
        us_ref = time_launches(lambda: kq.kq_bf16_gemm(ga, gw, c=cq, stream=stream), stream)
        flops = 2.0 * gm * gn * gk
        fpeak, fsrc = fp4_peak()
        consumer = {"metric": "kq_w4a4_gemm TFLOP/s (kind::mxf4, C = A_q W_q^T, fp32 out)",
                    "shape": f"{gm}x{gn}x{gk}", "us": round(us_fp4, 2),
                    "tflops": round(flops / us_fp4 / 1e6, 1), "peak_tflops": round(fpeak, 1),
                    "frac": round(flops / us_fp4 / 1e6 / fpeak, 4), "peak_source": fsrc,
                    "dequant_bf16_us": round(us_deq, 2), "bf16_reference_us": round(us_ref, 2)}
        del cq, qw, sfw, ga, gw
        torch.cuda.empty_cache()

    # ---- end to end through the public call with host buffers
    e2e_steps = max(3, min(K, 100))
    host_q = [torch.empty(Q[li][0].shape, dtype=torch.uint8).pin_memory() for li in range(2)]
    host_sf = [torch.empty(SF[li][0].shape, dtype=torch.uint8).pin_memory() for li in range(2)]
    h2d = sum(h.numel() * 2 for h in host_A)
    d2h = sum(t.numel() for t in host_q) + sum(t.numel() for t in host_sf)
    # Three streams: host->device copies, the quantizer launches, device->host
    # copies; step k uses buffer set k % SETS, and events keep a set's input
    # from being overwritten before its launches ran and its outputs from
    # being overwritten before they were copied out.  A step's copies thus
    # overlap the launches and copies of its neighbours.
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(SETS)]
    ev_done = [torch.cuda.Event() for _ in range(SETS)]
    ev_out = [torch.cuda.Event() for _ in range(SETS)]
    used = [False] * SETS

    def e2e_step(s):
        if used[s]:
            s_in.wait_event(ev_done[s])             # launches of the set's last use ran
        with torch.cuda.stream(s_in):
            for li in range(len(LAYERS)):
                A[li][s].copy_(host_A[li], non_blocking=True)
            ev_in[s].record(s_in)
        stream.wait_event(ev_in[s])
        if used[s]:
            stream.wait_event(ev_out[s])            # outputs of the set's last use copied out
        with torch.cuda.stream(stream):
            for li in range(len(LAYERS)):
                launch("kroquant", li, s)
            ev_done[s].record(stream)
        s_out.wait_event(ev_done[s])
        with torch.cuda.stream(s_out):
            for li in range(len(LAYERS)):
                host_q[li].copy_(Q[li][s], non_blocking=True)
                host_sf[li].copy_(SF[li][s], non_blocking=True)
            ev_out[s].record(s_out)
        used[s] = True

    for w in range(3):
        e2e_step(w % SETS)
    torch.cuda.synchronize()
    dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    for k in range(e2e_steps):
        e2e_step(k % SETS)
    for ev in ev_out:
        stream.wait_event(ev)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = dist.max(e0.elapsed_time(e1))
    e2e_value = dist.sum(STEP_BYTES * e2e_steps) / (e2e_ms * 1e-3) / 1e9

    cpu = cpu_baseline(args.cpu_seconds) if dist.rank == 0 and dist.world == 1 else None

    if dist.rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": dist.world,
            "steps": K, "warmup": W, "ms_per_step": round(ms_max / K, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": "flux_layer_pair", "m": 4608, "d": [3072, 12288],
                       "transform": f"kroquant_{args.variant}", "input": "bf16",
                       "output": "mxfp4 (e2m1 codes + e8m0 scales, 128x4 tiled)",
                       "l2": f"{SETS} rotating input/output sets, "
                             f"{SETS * STEP_BYTES / 1e6:.0f} MB footprint > L2",
                       "launch": f"rounds of min(steps left, {ROUND}) steps: per round and "
                                 "layer one CUDA graph of that many launches of the layer over "
                                 f"its {SETS} input sets (programmatic dependent launch between "
                                 "them); events around each dominant-layer graph",
                       "parallelism":
                           f"replicas x{dist.world} (rows independent, no exchange)"},
            "hbm_frac": round(value / dist.world / peak, 4),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                         "traffic_unit": "bytes per launch (ncu, cold L2; outputs left in L2)",
                         "kernel": workload, "launch_ms": round(dom_ms, 5),
                         "mode": "launches back to back inside the timed region's layer graphs",
                         "launch_us_x_sm_mhz": round(dom_ms * 1e3 * clocks["sm_mhz"], 1)
                         if clocks.get("sm_mhz") else None,
                         "peak_source": peak_src},
            "isolated_launch": {
                "us": round(iso_ms * 1e3, 3),
                "gbs": round(algo_bytes(dom_m, dom_d) / (iso_ms * 1e-3) / 1e9, 2),
                "frac": round(algo_bytes(dom_m, dom_d) / (iso_ms * 1e-3) / 1e9 / peak, 4),
                "launch_floor_us": round(floor_ms * 1e3, 3),
                "diag_us": round(iso_diag_ms * 1e3, 3) if iso_diag_ms else None,
                "vs_diag_scale": round(iso_diag_ms / iso_ms, 4) if iso_diag_ms else None,
                "how": "median over launches of one dominant-layer launch replayed alone as a "
                       "one-launch CUDA graph between two events (no overlap with a neighbour); "
                       "launch_floor_us is the same measurement of a one-element kernel"},
            "vs_diag_scale": round(value / dist.world / baselines["diag"], 4)
            if baselines.get("diag") else None,
            "baselines_gbs": baselines,
            "side_output": side,
            "consumer_gemm": consumer,
            "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps},
            "gpu_launches": K * len(LAYERS),
            "clocks": clocks,
            "clocks_whole_run": run_clocks,
        }
        if cpu is not None:
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)


def run_profile_case(args):
    """A few launches of one quantizer on one synthetic layer (for ncu)."""
    import numpy as np
    import torch
    from w4a4_mxfp4_activation_gb300 import kq, synth
    m, d = args.m, args.d
    bits = synth.activations(m, d, synth.SEED_A + 3, "flux")
    A = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    F = torch.from_numpy(kq.kq_lu_to_factors(synth.lu_params(d // 32, 7), +1)).cuda()
    s = torch.from_numpy(synth.smooth_scales(d)).cuda()
    layout = kq.KQ_SF_BLOCKED_128x4
    q = torch.empty((m, d // 2), dtype=torch.uint8, device="cuda")
    sf = torch.empty(kq.kq_sf_bytes(m, d, layout), dtype=torch.uint8, device="cuda")
    KX = (kq.kq_expand_blocks(F, kq.KQ_K_BF16X3)
          if args.variant == "umma" or args.profile == "dual" else None)
    at = torch.empty((m, d), dtype=torch.bfloat16, device="cuda") if args.profile == "dual" else None
    variant = {"butterfly": kq.VARIANT_BUTTERFLY, "umma": kq.VARIANT_UMMA,
               "k2": kq.VARIANT_K2}[args.variant]
    if args.profile == "gemm":
        n = args.n
        qa, sfa, qw, sfw, _, _ = gemm_case(m, n, d, 9000, "cuda")
        c = torch.empty((m, n), dtype=torch.float32, device="cuda")
        for _ in range(args.launches):
            kq.kq_w4a4_gemm(qa, sfa, qw, sfw, m, n, d, c=c)
        torch.cuda.synchronize()
        print(f"profile case done: gemm m={m} n={n} k={d} launches={args.launches}")
        return
    for _ in range(args.launches):
        if args.profile == "kroquant":
            kq.kq_quantize_mxfp4(A, d, factors=F if KX is None else None, K_expanded=KX,
                                 layout=layout, q=q, sf=sf, variant=variant)
        elif args.profile == "dual":
            kq.kq_quantize_mxfp4_dual(A, KX, d, layout=layout, q=q, sf=sf, at=at)
        elif args.profile == "diag":
            kq.kq_smooth_quantize_mxfp4(A, s, d, layout=layout, q=q, sf=sf)
        elif args.profile == "hadamard":
            kq.kq_hadamard_quantize_mxfp4(A, d, layout=layout, q=q, sf=sf)
        elif args.profile == "fwht":
            kq.kq_fwht_quantize_mxfp4(A, d, layout=layout, q=q, sf=sf)
        else:
            kq.kq_quantize_mxfp4(A, d, layout=layout, q=q, sf=sf)
    torch.cuda.synchronize()
    print(f"profile case done: {args.profile} m={m} d={d} launches={args.launches}")


# ------------------------------------------------------------- config table --

TABLE_CONFIGS = (
    ("0", (("cfg0_tiny", 256, 1152, "gauss_outlier8"),)),
    ("1", (("pixart_qkv", 4096, 1152, "pixart"), ("pixart_ffn_down", 4096, 4608, "pixart"))),
    ("2", (("sana_2240", 4096, 2240, "sana"), ("sana_5600", 4096, 5600, "sana"))),
    ("3", (("flux_3072", 4608, 3072, "flux"), ("flux_ffn_down", 4608, 12288, "flux"))),
    ("4", tuple((f"sweep_{m}x{d}", m, d, "flux") for m in (256, 1024, 4096, 16384, 65536)
                for d in (1152, 3072, 12288))),
)
TABLE_KERNELS = ("umma", "k2", "butterfly", "diag", "hadamard", "identity", "dual")


def oracle_rate_shape(m: int, d: int, seconds: float):
    """GB/s of the oracle (KroQuant transform + MXFP4, tiled scales) on a row
    sample of an m x d layer sized to about `seconds` of CPU work."""
    import numpy as np
    from oracle import kq_oracle as O
    from w4a4_mxfp4_activation_gb300 import synth

    def once(rows):
        A = synth.activations(rows, d, synth.SEED_A + 5, "flux")
        lu = synth.lu_params(d // 32, synth.SEED_FACTORS + 5)
        F = O.lu_to_factors(lu.astype(np.float64), +1).astype(np.float32).astype(np.float64)
        t0 = time.perf_counter()
        y, bound = O.transform(A, d, "kron", F)
        O.quantize(y, bound, O.SF_BLOCKED_128x4)
        return time.perf_counter() - t0

    t = once(min(m, 32))
    rows = max(1, min(m, int(min(m, 32) * seconds / max(t, 1e-4))))
    dt = once(rows)
    return algo_bytes(rows, d) / dt / 1e9, rows


def synth_seed(cfg: str) -> int:
    from w4a4_mxfp4_activation_gb300 import synth
    return synth.SEED_A + int(cfg)


def measure_shape(args, m, d, model, seed, kinds, peak):
    """Per-launch median time (us) of each kernel kind on one layer shape, in
    the bench's steady state: launches back to back from CUDA graphs,
    rotating over enough input/output sets that their footprint exceeds 3x
    the L2 (every launch reads its input from DRAM and evicts earlier
    outputs); the time per launch is the median over graph replays of the
    replay's CUDA-event time / its launches.  Returns ({kind: us}, sets)."""
    import numpy as np
    import torch
    from w4a4_mxfp4_activation_gb300 import kq, synth

    dev = torch.device("cuda", 0)
    layout = kq.KQ_SF_BLOCKED_128x4
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    stream = torch.cuda.Stream(device=dev)
    sets = max(4, int(np.ceil(3 * l2 / algo_bytes(m, d))))
    # the seeded generator for up to 4096 rows, tiled on the device
    rows = min(m, 4096)
    base = torch.from_numpy(synth.activations(rows, d, seed, model)
                            .view(np.int16)).to(dev).view(torch.bfloat16)
    A0 = base.repeat((m + rows - 1) // rows, 1)[:m].contiguous()
    del base
    A = [torch.roll(A0, shifts=37 * s, dims=0) for s in range(sets)]
    del A0
    A16 = None
    if any(k.endswith("_f16") for k in kinds):
        # the same model drawn in fp16 (PixArt-Sigma's format)
        base16 = torch.from_numpy(synth.activations(rows, d, seed, model, fmt="f16")
                                  .view(np.int16)).to(dev).view(torch.float16)
        B16 = base16.repeat((m + rows - 1) // rows, 1)[:m].contiguous()
        del base16
        A16 = [torch.roll(B16, shifts=37 * s, dims=0) for s in range(sets)]
        del B16
    F = torch.from_numpy(kq.kq_lu_to_factors(
        synth.lu_params(d // 32, synth.SEED_FACTORS + seed), +1)).to(dev)
    KX = kq.kq_expand_blocks(F, kq.KQ_K_BF16X3)
    S = torch.from_numpy(synth.smooth_scales(d)).to(dev)
    Q = [torch.empty((m, d // 2), dtype=torch.uint8, device=dev) for _ in range(sets)]
    SF = [torch.empty(kq.kq_sf_bytes(m, d, layout), dtype=torch.uint8, device=dev)
          for _ in range(sets)]
    AT = ([torch.empty((m, d), dtype=torch.bfloat16, device=dev) for _ in range(sets)]
          if "dual" in kinds else None)
    n_launch = max(sets, 32)

    def launch(kind, i):
        s = i % sets
        if kind == "umma":
            kq.kq_quantize_mxfp4(A[s], d, K_expanded=KX, layout=layout, q=Q[s], sf=SF[s],
                                 variant=kq.VARIANT_UMMA, stream=stream)
        elif kind == "butterfly":
            kq.kq_quantize_mxfp4(A[s], d, factors=F, layout=layout, q=Q[s], sf=SF[s],
                                 variant=kq.VARIANT_BUTTERFLY, stream=stream)
        elif kind == "k2":
            kq.kq_quantize_mxfp4(A[s], d, factors=F, layout=layout, q=Q[s], sf=SF[s],
                                 variant=kq.VARIANT_K2, stream=stream)
        elif kind == "dual":
            kq.kq_quantize_mxfp4_dual(A[s], KX, d, layout=layout, q=Q[s], sf=SF[s], at=AT[s],
                                      stream=stream)
        elif kind == "diag":
            kq.kq_smooth_quantize_mxfp4(A[s], S, d, layout=layout, q=Q[s], sf=SF[s],
                                        stream=stream)
        elif kind == "hadamard":
            kq.kq_hadamard_quantize_mxfp4(A[s], d, layout=layout, q=Q[s], sf=SF[s], stream=stream)
        elif kind == "fwht":
            kq.kq_fwht_quantize_mxfp4(A[s], d, layout=layout, q=Q[s], sf=SF[s], stream=stream)
        elif kind.endswith("_f16"):
            t = {"identity_f16": "identity", "diag_f16": "diag", "butterfly_f16": "kron",
                 "fwht_f16": "fwht"}[kind]
            prm = F if t == "kron" else (S if t == "diag" else None)
            kq.kq_quantize_mxfp4_ex(A16[s], t, prm, d, in_format=kq.KQ_IN_F16, layout=layout,
                                    q=Q[s], sf=SF[s], stream=stream)
        else:
            kq.kq_quantize_mxfp4(A[s], d, layout=layout, q=Q[s], sf=SF[s], stream=stream)

    us = {}
    for kind in kinds:
        with torch.cuda.stream(stream):
            for i in range(sets):
                launch(kind, i)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(n_launch):
                    launch(kind, i)
            reps = max(5, min(args.table_reps, int(2e5 // n_launch)))
            for _ in range(max(2, args.table_warmup // n_launch)):
                g.replay()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(reps)]
            for a, b in ev:
                a.record(stream)
                g.replay()
                b.record(stream)
            stream.synchronize()
        us[kind] = statistics.median(a.elapsed_time(b) for a, b in ev) / n_launch * 1e3
        del g
    del A, A16, Q, SF, KX, AT
    torch.cuda.empty_cache()
    return us, sets


# the pages' Table 3 shapes: power-of-two d, where the full-row FWHT applies
TABLE3_SHAPES = ((4096, 1024), (4096, 4096), (4096, 16384), (512, 4096), (512, 16384))


def run_table(args):
    """Steady-state GB/s of every kernel on every config shape, the pages'
    Table 3 comparison on GB300, and the oracle on the host cores."""
    import torch  # noqa: F401  (initializes CUDA before the measurements)
    peak, _ = hbm_peak()
    if args.table3_only:
        run_table3(args, peak)
        return
    print("| config | layer | m x d | sets | " + " | ".join(
        f"{k} GB/s (% peak)" if k in ("umma", "dual") else f"{k} GB/s"
        for k in TABLE_KERNELS) + " | umma / diag |")
    print("|" + "---|" * (len(TABLE_KERNELS) + 5))
    for cfg, layers in TABLE_CONFIGS:
        for name, m, d, model in layers:
            us, sets = measure_shape(args, m, d, model, synth_seed(cfg), TABLE_KERNELS, peak)
            gbs = {k: (algo_bytes_dual(m, d) if k == "dual" else algo_bytes(m, d)) / us[k] / 1e3
                   for k in TABLE_KERNELS}
            cells = [f"{gbs[k]:.0f} ({100 * gbs[k] / peak:.0f} %)" if k in ("umma", "dual")
                     else f"{gbs[k]:.0f}" for k in TABLE_KERNELS]
            print(f"| {cfg} | {name} | {m}x{d} | {sets} | " + " | ".join(cells) +
                  f" | {gbs['umma'] / gbs['diag']:.2f} |", flush=True)
    run_table3(args, peak)
    # the oracle on the host cores: all of them, then one
    print()
    print("| config | layer | oracle GB/s, all cores | oracle GB/s, 1 core |")
    print("|---|---|---|---|")
    for cfg, layers in TABLE_CONFIGS[:4]:
        for name, m, d, _ in layers:
            out = []
            for env_threads in (None, "1"):
                env = dict(os.environ)
                if env_threads:
                    env["OMP_NUM_THREADS"] = env_threads
                r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-rate",
                                    str(m), str(d), "3"], env=env, capture_output=True,
                                   text=True, check=True)
                out.append(r.stdout.strip())
            print(f"| {cfg} | {name} | {out[0]} | {out[1]} |", flush=True)
    print(f"\nhost: {os.cpu_count()} cores; per shape max(4, 3 L2 / set) rotating sets, "
          f"CUDA graphs of max(sets, 32) launches, median over up to {args.table_reps} replays")


def run_table3(args, peak):
    """[KQ] Table 3 on GB300 (bf16 and fp16 activations)."""
    # [KQ] Table 3 on GB300: latency (us) of the bare quantizer (Q4), the
    # diagonal scale (Scale), the dense-block tensor-core kernel (tcgen05,
    # K1's form), the kernel built from the factors (butterfly, K2's input)
    # and the full-row Walsh-Hadamard transform (FWHT), all with MXFP4 output
    kinds = ("identity", "diag", "umma", "k2", "butterfly", "fwht")
    print()
    print("| m | d | Q4 us | Scale us | tcgen05 (K1 records) us | tcgen05 (K2) us | butterfly us | "
          "FWHT us | Scale/tcgen05 | K1/K2 | Scale/butterfly | FWHT/tcgen05 | FWHT/butterfly |")
    print("|" + "---|" * 13)
    for m, d in TABLE3_SHAPES:
        us, _ = measure_shape(args, m, d, "flux", synth_seed("3"), kinds, peak)
        print(f"| {m} | {d} | " + " | ".join(f"{us[k]:.2f}" for k in kinds) +
              f" | {us['diag'] / us['umma']:.2f} | {us['umma'] / us['k2']:.2f} | "
              f"{us['diag'] / us['butterfly']:.2f} | "
              f"{us['fwht'] / us['umma']:.2f} | {us['fwht'] / us['butterfly']:.2f} |", flush=True)
    # the same with fp16 activations, the precision the pages time in: the
    # CUDA-core kernels (the tensor-core path reads bf16)
    kinds16 = ("identity_f16", "diag_f16", "butterfly_f16", "fwht_f16")
    print()
    print("fp16 activations (the pages' timing precision):")
    print()
    print("| m | d | Q4 us | Scale us | butterfly us | FWHT us | Scale/butterfly | FWHT/butterfly |")
    print("|" + "---|" * 8)
    for m, d in TABLE3_SHAPES:
        us, _ = measure_shape(args, m, d, "flux", synth_seed("3"), kinds16, peak)
        print(f"| {m} | {d} | " + " | ".join(f"{us[k]:.2f}" for k in kinds16) +
              f" | {us['diag_f16'] / us['butterfly_f16']:.2f} | "
              f"{us['fwht_f16'] / us['butterfly_f16']:.2f} |", flush=True)


GEMM_TABLE = (
    ("cfg0 projection", 256, 1152, 1152),
    ("PixArt-Sigma FFN up", 4096, 4608, 1152),
    ("PixArt-Sigma FFN down", 4096, 1152, 4608),
    ("SANA FFN up", 4096, 5600, 2240),
    ("SANA FFN down", 4096, 2240, 5600),
    ("FLUX projection", 4608, 3072, 3072),
    ("FLUX FFN up", 4608, 12288, 3072),
    ("FLUX FFN down", 4608, 3072, 12288),
)


def run_gemm_table(args):
    """The W4A4 product C = A_q W_q^T on the layer shapes (m tokens, n output
    channels, k input channels): the FP4 tensor-core kernel, the bf16
    dequantization route, the bf16 reference product A W^T of this library and
    of cuBLAS (torch.matmul)."""
    import torch
    from w4a4_mxfp4_activation_gb300 import kq
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=dev)
    fpeak, fsrc = fp4_peak()
    print(f"| layer | m x n x k | kind::mxf4 us | TFLOP/s | % of FP4 peak ({fpeak:.0f}, {fsrc}) | "
          "dequant-bf16 us | bf16 reference us | cuBLAS bf16 us | mxf4 / cuBLAS bf16 |")
    print("|" + "---|" * 9)
    for name, m, n, k in GEMM_TABLE:
        qa, sfa, qw, sfw, a, w = gemm_case(m, n, k, 9100, dev)
        c = torch.empty((m, n + (-n) % 4), dtype=torch.float32, device=dev)[:, :n]
        t4 = time_launches(lambda: kq.kq_w4a4_gemm(qa, sfa, qw, sfw, m, n, k, c=c, stream=stream),
                           stream)
        td = time_launches(lambda: kq.kq_w4a4_gemm(qa, sfa, qw, sfw, m, n, k, c=c,
                                                   variant=kq.GEMM_DEQUANT_BF16, stream=stream),
                           stream, reps=4, rounds=3)
        tb = time_launches(lambda: kq.kq_bf16_gemm(a, w, c=c, stream=stream), stream)
        tc = time_launches(lambda: torch.matmul(a, w.t()), stream)
        tf = 2.0 * m * n * k / t4 / 1e6
        print(f"| {name} | {m}x{n}x{k} | {t4:.2f} | {tf:.0f} | {100 * tf / fpeak:.1f} | {td:.1f} | "
              f"{tb:.2f} | {tc:.2f} | {tc / t4:.2f} |", flush=True)
        del qa, sfa, qw, sfw, a, w, c
        torch.cuda.empty_cache()
    print("\nmedian of 5 replays of a CUDA graph of 20 launches (4 for dequant-bf16), same stream; "
          "operands resident, random codes and scales")


def main():
    args = parse_args()
    if args.gemm:
        from w4a4_mxfp4_activation_gb300 import build
        build.build()
        run_gemm_table(args)
        return
    if args.cpu_rate:
        m, d, sec = args.cpu_rate
        rate, rows = oracle_rate_shape(m, d, float(sec))
        print(f"{rate:.3f} ({rows} rows, {cpu_cores()} cores)")
        return
    if args.table:
        from w4a4_mxfp4_activation_gb300 import build
        build.build()
        run_table(args)
        return
    if args.profile:
        from w4a4_mxfp4_activation_gb300 import build
        build.build()
        run_profile_case(args)
        return
    if args.impl == "reference":
        dist = Dist(use_cuda=False) if int(os.environ.get("WORLD_SIZE", "1")) > 1 else Dist(False)
        try:
            run_reference(args, dist)
        finally:
            dist.close()
        return
    import torch
    if not torch.cuda.is_available():
        print(json.dumps({"metric": METRIC, "error": "no CUDA device"}), flush=True)
        sys.exit(1)
    dist = Dist(use_cuda=True)
    torch.cuda.set_device(dist.local)
    from w4a4_mxfp4_activation_gb300 import build
    build.build()
    try:
        run_ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
