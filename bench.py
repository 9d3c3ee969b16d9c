"""Benchmark of the MXFP4 block-quantization hot path on GB300.

Headline (one JSON line on stdout, rank 0): dense activation quantize of a
4096 x 7168 BF16 matrix — GB/s counted as BF16 bytes read + code bytes
written + tiled scale bytes written, per step = one quantize launch on one
batch.  Inputs/outputs rotate over enough buffer sets to exceed 2x L2, so no
step finds its operands in L2.

Also reported in the same line:
  roofline      achieved GB/s of the quantize kernel vs the measured HBM copy
                peak, plus DRAM traffic from the committed ncu summary;
  e2e           the same metric through the public API with pinned host
                buffers (host->device copy of x and device->host copy of
                codes + scales inside the timed region, pipelined in row
                chunks over three streams);
  cpu_baseline  the CPU oracle on the host cores (bounded sample);
  rows          every other hot-path row measured on its own workload:
                dequantize, grouped MoE quantize, expert-weight quantize,
                w13 swap, edge-case matrix;
  clocks        nvidia-smi samples taken while the GPU was busy.

`--impl reference` times the CPU oracle instead (the only reference this
method has), on a bounded sample per step.

Multi-GPU: one process per GPU under torchrun; every rank quantizes its own
batch (weak scaling, no data exchange); the timed region is bracketed by a
barrier and the max over ranks is reported.
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MXFP4 quantize GB/s (in+out) and % of GB300 HBM peak, bit-exact vs oracle"
M_DENSE, K_DENSE = 4096, 7168
FALLBACK_HBM_GBS = 6800.0
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "quantize_dense_4096x7168.md")
QUANT_SOURCES = [os.path.join(ROOT, "mxfp4_block_quantization_gb300", "csrc", f)
                 for f in ("quantize.cu", "mxfp4_device.cuh")]


def quant_bytes(M, K):
    """Algorithmic bytes of one quantize: BF16 read + codes + tiled scales."""
    sK = K // 32
    scale = ((M + 127) // 128 * 128) * ((sK + 3) // 4 * 4)
    return 2 * M * K + M * K // 2 + scale


def dequant_bytes(M, K):
    sK = K // 32
    scale = ((M + 127) // 128 * 128) * ((sK + 3) // 4 * 4)
    return M * K // 2 + scale + 2 * M * K


# ------------------------------------------------------------ distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(elapsed_ms, nbytes, group=None):
    """Max elapsed time and summed bytes over all ranks (timing only)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return elapsed_ms, nbytes
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device=dev)
    b = torch.tensor([float(nbytes)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(b, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(b.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ----------------------------------------------------------------- peaks
def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_digest():
    h = hashlib.sha256()
    for p in QUANT_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu summary, or None when the
    summary is missing or the kernel source changed since it was taken."""
    try:
        text = open(PROFILE_SUMMARY).read()
    except OSError:
        return None
    m_src = re.search(r"kernel_source_digest:\s*([0-9a-f]+)", text)
    m_b = re.search(r"dram_bytes_per_launch_4096x7168:\s*([0-9.]+)", text)
    if not (m_src and m_b) or m_src.group(1) != source_digest():
        return None
    return float(m_b.group(1))


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (SM clock, max clock, throttle reasons) every 100 ms."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def wait_first(self, timeout=15.0):
        """Until the first sample arrives (nvidia-smi can take a second or more
        to start on a fresh box), at most `timeout` seconds: the settle period
        that follows is then sampled from its start."""
        t_end = time.time() + timeout
        while self.proc is not None and not self.samples and time.time() < t_end:
            if self.proc.poll() is not None:
                return
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        if self.proc is None:
            return None
        inside = [p for t, p in self.samples if t0 <= t <= t1]
        window = "timed"
        if not inside:
            inside = [p for t, p in self.samples if t0 - 1.5 <= t <= t1 + 0.5]
            window = "timed region shorter than the 100 ms sampling period: samples from the " \
                     "sustained warm-up just before it and the timed region"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        mx = [num(p[2]) for p in inside if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4)
                          if p[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside), "window": window}


# ------------------------------------------------------------ CPU oracle
def host_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_quantize_threads(xb, codes, scales, threads):
    """Run the unchanged single-threaded oracle over 128-row partitions on
    `threads` host threads (the C routine releases the GIL)."""
    import oracle
    M = xb.shape[0]
    tiles = (M + 127) // 128
    per = (tiles + threads - 1) // threads
    parts = [(t * 128, min(M, (t + per) * 128)) for t in range(0, tiles, per)]
    ths = [threading.Thread(target=oracle.quantize_rows_into, args=(xb, a, b, codes, scales))
           for a, b in parts]
    for t in ths:
        t.start()
    for t in ths:
        t.join()
    return len(parts)


def cpu_baseline(xb, min_seconds=2.0, max_reps=20):
    import numpy as np
    import oracle
    oracle.lib()
    M, K = xb.shape
    threads = host_threads()
    codes = np.zeros((M, K // 2), np.uint8)
    scales = np.zeros(quant_bytes(M, K) - 2 * M * K - M * K // 2, np.uint8)
    used = oracle_quantize_threads(xb, codes, scales, threads)   # warm-up + page-in
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle_quantize_threads(xb, codes, scales, threads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or reps >= max_reps:
            break
    gbs = quant_bytes(M, K) * reps / el / 1e9
    # the same oracle on one core, on the first 512 rows
    rows = min(M, 512)
    x1 = np.ascontiguousarray(xb[:rows])
    oracle.quantize(x1)
    reps1, t1 = 0, time.perf_counter()
    while True:
        oracle.quantize(x1)
        reps1 += 1
        el1 = time.perf_counter() - t1
        if el1 >= min_seconds / 2 or reps1 >= 4 * max_reps:
            break
    gbs1 = quant_bytes(rows, K) * reps1 / el1 / 1e9
    return {"value": round(gbs, 3), "unit": "GB/s", "cores": used, "kind": "oracle",
            "sample": f"full {M}x{K} matrix x {reps} passes, 128-row bands on {used} threads",
            "single_core_GB_per_s": round(gbs1, 4)}


# ---------------------------------------------------------- reference arm
def run_reference(args):
    """The CPU oracle (single-threaded, unchanged) as the reference arm: each
    step quantizes the first rows of the dense activation matrix, as many as
    keep the whole run within about two minutes.  Imports the oracle and the
    input generators only: the CUDA library is never loaded here."""
    import numpy as np
    import oracle
    import workloads as W
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    oracle.lib()
    xb_full = W.bf16_bits(W.dense_activation(1, M_DENSE, K_DENSE))
    # per-step sample: enough rows that the whole run ends in ~1-2 minutes
    steps_total = args.steps + args.warmup
    t0 = time.perf_counter()
    oracle.quantize(xb_full[:8])
    per_row = (time.perf_counter() - t0) / 8
    step_s = min(0.25, 90.0 / max(steps_total, 1))  # seconds of oracle work per step
    rows = int(max(1, min(M_DENSE, step_s / max(per_row, 1e-9))))
    xb = np.ascontiguousarray(xb_full[:rows])
    for _ in range(args.warmup):
        oracle.quantize(xb)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.quantize(xb)
    el = time.perf_counter() - t0
    nbytes = quant_bytes(rows, K_DENSE)
    gbs = nbytes * args.steps / el / 1e9
    sample = (f"first {rows} rows of the {M_DENSE}x{K_DENSE} dense activation per step "
              f"({nbytes} algorithmic bytes), single-threaded CPU oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"dense activation quantize, first {rows} rows of "
                               f"{M_DENSE}x{K_DENSE} BF16 (N(0,1) x 2^U(-8,8) per row, seed 1)",
                   "bytes_per_step": nbytes, "parallelism": "single host thread"},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm
class L2Sweep:
    """A read (by torch) of a buffer of 3x the L2 before each timed batch.
    It evicts whatever the L2 held, so the batch's first step starts cold
    like every later one, and it leaves only clean lines behind, so no
    write-back of earlier work lands inside the batch.  While the device
    reads it, the host has already queued the batch's launches, so a batch's
    device time holds no host launch latency."""

    def __init__(self, l2_bytes, device=None):
        import torch
        dev = device or "cuda"
        self.buf = torch.zeros(3 * l2_bytes // 4, dtype=torch.float32, device=dev)
        self.res = torch.zeros((), dtype=torch.float32, device=dev)

    def __call__(self):
        import torch
        torch.sum(self.buf, dim=0, out=self.res)


def time_batches(fn, stream, sweep, per_batch, batches, warmup=3):
    """fn(i) launched in `batches` batches of `per_batch` calls, each batch
    timed by CUDA events on `stream` after an L2 sweep.  Returns (mean,
    median) milliseconds per call: the mean over all calls, the median over
    batches of each batch's mean."""
    import torch
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(batches)]
    i = 0
    for s_, e_ in evs:
        sweep()
        s_.record(stream)
        for _ in range(per_batch):
            fn(i)
            i += 1
        e_.record(stream)
    torch.cuda.synchronize()
    per = [s_.elapsed_time(e_) / per_batch for s_, e_ in evs]
    return sum(per) / len(per), statistics.median(per)


def time_graph_batches(fn, stream, sweep, per_batch, batches, warmup=3):
    """time_batches with each batch captured once as a CUDA graph of its
    `per_batch` calls fn(i) on `stream` (not the default stream) and replayed
    after an L2 sweep: the host's per-call cost (the binding's argument checks
    and ctypes, 8-19 us a call) is then not in the time, which is the device
    time of the calls alone.  Returns (mean, median) milliseconds per call."""
    import torch
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(per_batch):
            fn(i)
    g.replay()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(batches)]
    for s_, e_ in evs:
        sweep()
        s_.record(stream)
        g.replay()
        e_.record(stream)
    torch.cuda.synchronize()
    per = [s_.elapsed_time(e_) / per_batch for s_, e_ in evs]
    del g
    return sum(per) / len(per), statistics.median(per)


def tiled_scale_index(M, K, device="cpu"):
    """[M, K/32] byte offsets of the scale bytes in the 128x4-tiled layout:
    chunk (r/128, c/4) of 512 bytes, byte (r%32)*16 + ((r%128)/32)*4 + c%4."""
    import torch
    r = torch.arange(M, device=device).view(M, 1)
    c = torch.arange(K // 32, device=device).view(1, K // 32)
    nkt = (K // 32 + 3) // 4
    return ((r // 128) * nkt + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4


def reconstruction_report(mx, x, codes, scales):
    """Reconstruction error of the headline matrix, from the GPU's own outputs
    (outside every timed region): relative L2 of dequantize(quantize(x))
    against x in float64, and the fraction of elements the E2M1 range clips,
    i.e. with |x| > 6 * 2^(s-127) for their block's scale byte s (read back
    from the 128x4-tiled layout)."""
    import torch
    M, K = x.shape
    y = mx.dequantize(codes, scales, M, K)
    xd, yd = x.double(), y.double()
    rel = float(torch.linalg.vector_norm(yd - xd) / torch.linalg.vector_norm(xd))
    s = scales[tiled_scale_index(M, K, x.device)].to(torch.float64)
    blk = torch.exp2(s - 127.0).repeat_interleave(32, dim=1)
    live = (s > 0).repeat_interleave(32, dim=1)
    sat = int(((xd.abs() > 6.0 * blk) & live).sum())
    return {"rel_l2": round(rel, 6), "clipped_frac": round(sat / (M * K), 6)}


def time_graph(fn, iters, replays=5):
    """Per-call device time of `iters` calls fn(i, stream) captured once in a
    CUDA graph on a side stream and replayed `replays` times: for kernels
    shorter than a Python call, so that the host's launch rate does not set
    the time.  Returns (mean, median over replays) milliseconds per call."""
    import torch
    side = torch.cuda.Stream()
    for i in range(3):
        fn(i, side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for i in range(iters):
            fn(i, side)
    per = []
    with torch.cuda.stream(side):
        g.replay()
        torch.cuda.synchronize()
        for _ in range(replays):
            s = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            s.record(side)
            g.replay()
            e.record(side)
            e.synchronize()
            per.append(s.elapsed_time(e) / iters)
    return sum(per) / len(per), statistics.median(per)


ROW_FIELDS = ["GB/s", "frac of measured peak", "mean us", "median us"]


def measure_rows(mx, W, stream, peak, l2_bytes, sweep):
    """Each remaining hot-path row on its own workload (device time, inputs
    resident in HBM, operands rotated or larger than L2, an L2 sweep before
    each timed batch, each batch a CUDA graph of its calls).  Every row is
    [GB/s, fraction of the peak, mean us, median us] over the row's
    algorithmic bytes; `extra` holds the unfused baselines the fused dispatch
    calls are compared with.  Runs on a stream of its own (graphs are not
    captured on the default stream); `stream` is replaced by it."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    prev = torch.cuda.current_stream()
    torch.cuda.set_stream(side)
    try:
        return _measure_rows(mx, W, side, peak, l2_bytes, sweep)
    finally:
        torch.cuda.synchronize()
        torch.cuda.set_stream(prev)


def _measure_rows(mx, W, stream, peak, l2_bytes, sweep):
    import torch
    rows, extra = {}, {}

    def row(name, nbytes, t):
        mean, med = t
        gbs = nbytes / (mean * 1e-3) / 1e9
        rows[name] = [round(gbs, 1), round(gbs / peak, 4), round(mean * 1e3, 2),
                      round(med * 1e3, 2)]

    def tb(fn, per_batch, batches=5):
        return time_graph_batches(fn, stream, sweep, per_batch, batches)

    # dequantize 4096 x 7168 (rotate buffers beyond 2x L2)
    M, K = M_DENSE, K_DENSE
    x = W.dense_activation(1, M, K, device="cuda")
    codes, scales = mx.quantize(x)
    nb = dequant_bytes(M, K)
    R = max(2, -(-2 * l2_bytes // nb) + 1)
    cs = [codes.clone() for _ in range(R)]
    ss = [scales.clone() for _ in range(R)]
    ys = [torch.empty((M, K), dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    row("dequant_4096x7168", nb,
        tb(lambda i: mx.mxfp4_dequantize(cs[i % R], ss[i % R], M, K, ys[i % R], stream), 40))
    del cs, ss, ys, x, codes, scales

    # the same activation in FP16 (same method, binary16 input)
    x16s = [W.dense_activation(1, M, K, device="cuda").to(torch.float16) for _ in range(R)]
    cs16 = [torch.empty((M, K // 2), dtype=torch.uint8, device="cuda") for _ in range(R)]
    ss16 = [torch.empty(M * 224, dtype=torch.uint8, device="cuda") for _ in range(R)]
    row("f16_quant_4096x7168", quant_bytes(M, K),
        tb(lambda i: mx.mxfp4_quantize_f16(x16s[i % R], cs16[i % R], ss16[i % R], stream), 40))
    del x16s, cs16, ss16

    # NVFP4 (16-element blocks, E4M3 scales, global scale 448*6/amax): quantize
    # and dequantize of the same 4096 x 7168 activation, and the FP16 quantize
    xs_nv = [W.dense_activation(1, M, K, device="cuda") for _ in range(R)]
    g_nv = torch.tensor([448.0 * 6.0 / float(xs_nv[0].float().abs().max())], device="cuda")
    sb_nv = mx.mxfp4_nvfp4_scale_bytes(M, K)
    cs_nv = [torch.empty((M, K // 2), dtype=torch.uint8, device="cuda") for _ in range(R)]
    ss_nv = [torch.empty(sb_nv, dtype=torch.uint8, device="cuda") for _ in range(R)]
    nb_nv = 2 * M * K + M * K // 2 + sb_nv
    row("nvfp4_quant_4096x7168", nb_nv,
        tb(lambda i: mx.mxfp4_quantize_nvfp4(xs_nv[i % R], g_nv, cs_nv[i % R], ss_nv[i % R],
                                             stream), 40))
    row("nvfp4_dequant_4096x7168", nb_nv,
        tb(lambda i: mx.mxfp4_dequantize_nvfp4(cs_nv[i % R], ss_nv[i % R], g_nv, M, K,
                                               xs_nv[i % R], stream), 40))
    for j in range(R):
        xs_nv[j] = xs_nv[j].to(torch.float16)
    row("nvfp4_f16_quant_4096x7168", nb_nv,
        tb(lambda i: mx.mxfp4_quantize_nvfp4_f16(xs_nv[i % R], g_nv, cs_nv[i % R], ss_nv[i % R],
                                                 stream), 40))
    del xs_nv, cs_nv, ss_nv

    # grouped MoE activations: 16384 tokens x top-8 over 384 experts, K = 7168
    g = W.moe_grouped(seed=2, device="cuda")
    total, K = g.x.shape
    E = g.num_experts
    T = g.x_tokens.shape[0]
    codes = torch.empty((total, K // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty(mx.mxfp4_grouped_scale_bytes_bound(total, E, K), dtype=torch.uint8,
                         device="cuda")
    sro = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    st = torch.empty(1, dtype=torch.int32, device="cuda")
    t_grouped = tb(lambda i: mx.mxfp4_quantize_grouped(g.x, g.offsets, codes, scales, sro, st,
                                                       stream), 6)
    padded = int(sro[-1].item())
    row("grouped_moe_131072x7168_E384",
        2 * total * K + total * K // 2 + padded * (K // 32) + 4 * (E + 1), t_grouped)
    g_nv = torch.full((E,), 448.0 * 6.0 / 5.0, device="cuda")
    sc_nv = torch.empty(mx.mxfp4_nvfp4_grouped_scale_bytes_bound(total, E, K), dtype=torch.uint8,
                        device="cuda")
    nb_nvg = 2 * total * K + total * K // 2 + padded * (K // 16) + 4 * (E + 1) + 4 * E
    row("nvfp4_grouped_moe_131072x7168_E384", nb_nvg,
        tb(lambda i: mx.mxfp4_quantize_nvfp4_grouped(g.x, g.offsets, g_nv, codes, sc_nv, sro, st,
                                                     stream), 6))

    # the same MoE batch with the dispatch fused in: token rows [16384, 7168]
    # read once + int32 route maps, against the unfused pair (torch
    # index_select materialising the 1.9 GB permuted matrix, then the grouped
    # quantize)
    xg = torch.empty_like(g.x)
    nb = 2 * T * K + 4 * total + total * K // 2 + padded * (K // 32) + 4 * (E + 1)
    t_unf = tb(lambda i: (torch.index_select(g.x_tokens, 0, g.row_index, out=xg),
                          mx.mxfp4_quantize_grouped(xg, g.offsets, codes, scales, sro, st,
                                                    stream)), 6)
    extra["unfused_gather_then_grouped_us"] = round(t_unf[0] * 1e3, 2)
    row("gather_moe_16384tok_top8", nb,
        tb(lambda i: mx.mxfp4_quantize_grouped_gather(g.x_tokens, g.row_index, g.offsets, codes,
                                                      scales, sro, st, stream), 6))
    ws = torch.empty(mx.mxfp4_gather_workspace_bytes(T, total, E, K), dtype=torch.uint8,
                     device="cuda")
    row("gather_ws_moe_16384tok_top8", nb,
        tb(lambda i: mx.mxfp4_quantize_grouped_gather_ws(g.x_tokens, g.row_index, g.offsets, ws,
                                                         codes, scales, sro, st, stream), 6))
    del ws
    row("scatter_moe_16384tok_top8", nb,
        tb(lambda i: mx.mxfp4_quantize_grouped_scatter(g.x_tokens, g.dest_rows, g.offsets, total,
                                                       codes, scales, sro, st, stream), 6))
    ws = torch.empty(mx.mxfp4_scatter_workspace_bytes(T, total, E, K), dtype=torch.uint8,
                     device="cuda")
    row("scatter_ws_moe_16384tok_top8", nb,
        tb(lambda i: mx.mxfp4_quantize_grouped_scatter_ws(g.x_tokens, g.dest_rows, g.offsets,
                                                          total, ws, codes, scales, sro, st,
                                                          stream), 6))
    del ws
    # the dispatch permutation itself, from the router's expert ids (every
    # route's expert read back from its row's segment): ids in, offsets,
    # token -> rows and row -> token out; then routed straight into the
    # scatter quantize with a workspace
    off_h = g.offsets.cpu()
    ids = (torch.searchsorted(off_h, g.dest_rows.cpu(), right=True) - 1).to(torch.int32).cuda()
    r_off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    r_dest = torch.empty_like(g.dest_rows)
    r_rows = torch.empty(total, dtype=torch.int32, device="cuda")
    r_ws = torch.empty(mx.mxfp4_route_workspace_bytes(T, g.dest_rows.shape[1], E),
                       dtype=torch.uint8, device="cuda")
    route = lambda i: mx.mxfp4_moe_route(ids, E, r_ws, r_off, r_dest, r_rows, st, stream)  # noqa: E731
    row("route_moe_16384tok_top8_E384", 12 * total + 4 * (E + 1), tb(route, 40))
    assert torch.equal(r_off, g.offsets) and torch.equal(r_dest, g.dest_rows)
    ws = torch.empty(mx.mxfp4_scatter_workspace_bytes(T, total, E, K), dtype=torch.uint8,
                     device="cuda")
    row("route_then_scatter_ws_moe", nb,
        tb(lambda i: (route(i), mx.mxfp4_quantize_grouped_scatter_ws(
            g.x_tokens, r_dest, r_off, total, ws, codes, scales, sro, st, stream)), 6))
    del ws
    # the NVFP4 experts quant with the same dispatch fused in; one global
    # scale shared by every expert, then a scale of its own per expert
    nb_nvs = 2 * T * K + 4 * total + total * K // 2 + padded * (K // 16) + 4 * (E + 1) + 4 * E
    t_nvu = tb(lambda i: (torch.index_select(g.x_tokens, 0, g.row_index, out=xg),
                          mx.mxfp4_quantize_nvfp4_grouped(xg, g.offsets, g_nv, codes, sc_nv, sro,
                                                          st, stream)), 6)
    extra["unfused_gather_then_nvfp4_grouped_us"] = round(t_nvu[0] * 1e3, 2)
    row("nvfp4_scatter_shared_g_moe", nb_nvs,
        tb(lambda i: mx.mxfp4_quantize_nvfp4_grouped_scatter(g.x_tokens, g.dest_rows, g.offsets,
                                                             total, g_nv, codes, sc_nv, sro, st,
                                                             stream), 6))
    ws = torch.empty(mx.mxfp4_nvfp4_scatter_workspace_bytes(total, E, K), dtype=torch.uint8,
                     device="cuda")
    row("nvfp4_scatter_ws_shared_g_moe", nb_nvs,
        tb(lambda i: mx.mxfp4_quantize_nvfp4_grouped_scatter_ws(g.x_tokens, g.dest_rows,
                                                                g.offsets, total, g_nv, ws, codes,
                                                                sc_nv, sro, st, stream), 6))
    g_own = 448.0 * 6.0 / torch.exp(torch.rand(E, generator=torch.Generator().manual_seed(2)) * 3.0)
    g_own = g_own.to("cuda")
    row("nvfp4_scatter_ws_own_g_moe", nb_nvs,
        tb(lambda i: mx.mxfp4_quantize_nvfp4_grouped_scatter_ws(g.x_tokens, g.dest_rows,
                                                                g.offsets, total, g_own, ws,
                                                                codes, sc_nv, sro, st, stream), 6))
    del sc_nv, ws, g, codes, scales, xg

    # expert weights: w13 [128, 1536, 2048], w2 [128, 2048, 768], then the swap
    w = W.expert_weights(3, device="cuda")
    E, two_n, H = w.w13.shape
    x13 = w.w13.view(E * two_n, H)
    x2 = w.w2.view(-1, w.w2.shape[2])
    c13 = torch.empty((E * two_n, H // 2), dtype=torch.uint8, device="cuda")
    s13 = torch.empty(mx.mxfp4_scale_bytes(E * two_n, H), dtype=torch.uint8, device="cuda")
    c2 = torch.empty((x2.shape[0], x2.shape[1] // 2), dtype=torch.uint8, device="cuda")
    s2 = torch.empty(mx.mxfp4_scale_bytes(*x2.shape), dtype=torch.uint8, device="cuda")
    row("w13_quant_196608x2048", quant_bytes(*x13.shape),
        tb(lambda i: mx.mxfp4_quantize(x13, c13, s13, stream), 6))
    row("w2_quant_262144x768", quant_bytes(*x2.shape),
        tb(lambda i: mx.mxfp4_quantize(x2, c2, s2, stream), 6))
    c_o = torch.empty_like(c13)
    s_o = torch.empty_like(s13)
    b13 = torch.empty(w.w13_bias.shape, dtype=torch.bfloat16, device="cuda")
    b2 = torch.empty(w.w2_bias.shape, dtype=torch.bfloat16, device="cuda")
    nb = 2 * (c13.numel() + s13.numel()) + w.w13_bias.numel() * 6 + w.w2_bias.numel() * 6
    row("swap_w13_E128_2N1536_K2048", nb,
        tb(lambda i: mx.mxfp4_swap_w13(c13, s13, w.w13_bias, E, two_n, H, 1, c_o, s_o, b13,
                                       w.w2_bias, b2, stream), 6))
    del w, c13, s13, c2, s2, c_o, s_o

    # edge-case matrix 1000 x 2880 (latency-scale; rotate 2x L2 worth of sets;
    # 500 launches replayed from one CUDA graph, the kernel being shorter than
    # a Python call)
    xe = W.edge_cases(4).cuda()
    nb = quant_bytes(1000, 2880)
    R = max(2, -(-2 * l2_bytes // nb) + 1)
    xs = [xe.clone() for _ in range(R)]
    cs = [torch.empty((1000, 1440), dtype=torch.uint8, device="cuda") for _ in range(R)]
    ss = [torch.empty(mx.mxfp4_scale_bytes(1000, 2880), dtype=torch.uint8, device="cuda")
          for _ in range(R)]
    row("edge_quant_1000x2880", nb,
        time_graph(lambda i, st: mx.mxfp4_quantize(xs[i % R], cs[i % R], ss[i % R], st), 500))
    return rows, extra


DISPATCH_CALLS = ("gather", "gather_ws", "scatter", "scatter_ws", "nvfp4_scatter",
                  "nvfp4_scatter_ws", "nvfp4_scatter_ws_own_g")
SINGLE_CALLS = DISPATCH_CALLS + ("dense", "w13", "route", "dequant", "nvfp4_dequant", "grouped",
                                  "swap")


def run_one_call(args):
    """--call NAME: one call repeated --reps times after one warm-up, and one
    JSON line with its mean CUDA-event time.  For profiling a single call
    (ncu -k on this command sees only its kernels).  NAME is a dispatch call
    on the MoE batch (16384 tokens x top-8 over 384 experts, K = 7168;
    nvfp4_scatter_ws_own_g with a global scale of its own per expert), the
    dense quantize of the 4096 x 7168 activation, the dense quantize of the
    w13 expert weights [128 x 1536, 2048], or the MXFP4 / NVFP4 dequantize of
    the quantized 4096 x 7168 activation (5 rotating input/output sets, 372 MB,
    so that no call finds its operands in the L2), the grouped quantize of the
    expert-sorted MoE batch (131072 x 7168, 384 experts), or the w13 swap of
    the quantized expert weights (128 experts, 2N = 1536, K = 2048, tiled
    scales and both biases)."""
    import torch
    import mxfp4_block_quantization_gb300 as mx
    import workloads as W
    if args.call in ("dequant", "nvfp4_dequant"):
        M, K, R = M_DENSE, K_DENSE, 5
        x = W.dense_activation(1, M, K, device="cuda")
        if args.call == "dequant":
            codes, scales = mx.quantize(x)
            nbytes = dequant_bytes(M, K)
        else:
            g_nv = torch.tensor([448.0 * 6.0 / float(x.float().abs().max())], device="cuda")
            codes, scales = mx.quantize_nvfp4(x, g_nv)
            nbytes = M * K // 2 + scales.numel() + 2 * M * K
        del x
        cs = [codes.clone() for _ in range(R)]
        ss = [scales.clone() for _ in range(R)]
        ys = [torch.empty((M, K), dtype=torch.bfloat16, device="cuda") for _ in range(R)]
        if args.call == "dequant":
            fn = lambda i: mx.mxfp4_dequantize(cs[i % R], ss[i % R], M, K, ys[i % R])  # noqa: E731
        else:
            fn = lambda i: mx.mxfp4_dequantize_nvfp4(cs[i % R], ss[i % R], g_nv, M, K,  # noqa: E731
                                                     ys[i % R])
        fn(0)
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for i in range(args.reps):
            fn(i + 1)
        t1.record()
        torch.cuda.synchronize()
        us = t0.elapsed_time(t1) * 1e3 / args.reps
        print(json.dumps({"call": args.call, "reps": args.reps, "us_per_call": round(us, 2),
                          "bytes_per_call": nbytes}))
        return 0
    if args.call == "swap":
        w = W.expert_weights(3, device="cuda")
        E, two_n, H = w.w13.shape
        c13, s13 = mx.quantize(w.w13.view(E * two_n, H))
        c_o, s_o = torch.empty_like(c13), torch.empty_like(s13)
        b13 = torch.empty(w.w13_bias.shape, dtype=torch.bfloat16, device="cuda")
        b2 = torch.empty(w.w2_bias.shape, dtype=torch.bfloat16, device="cuda")
        nbytes = 2 * (c13.numel() + s13.numel()) + 6 * (w.w13_bias.numel() + w.w2_bias.numel())
        fn = lambda: mx.mxfp4_swap_w13(c13, s13, w.w13_bias, E, two_n, H, 1, c_o, s_o,  # noqa: E731
                                       b13, w.w2_bias, b2)
        fn()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(args.reps):
            fn()
        t1.record()
        torch.cuda.synchronize()
        us = t0.elapsed_time(t1) * 1e3 / args.reps
        print(json.dumps({"call": "swap", "reps": args.reps, "us_per_call": round(us, 2),
                          "bytes_per_call": nbytes}))
        return 0
    if args.call in ("dense", "w13"):
        if args.call == "dense":
            x = W.dense_activation(1, M_DENSE, K_DENSE, device="cuda")
        else:
            w13 = W.expert_weights(3, device="cuda").w13
            x = w13.view(-1, w13.shape[2])
        codes = torch.empty((x.shape[0], x.shape[1] // 2), dtype=torch.uint8, device="cuda")
        scales = torch.empty(mx.mxfp4_scale_bytes(*x.shape), dtype=torch.uint8, device="cuda")
        fn = lambda: mx.mxfp4_quantize(x, codes, scales)  # noqa: E731
        fn()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(args.reps):
            fn()
        t1.record()
        torch.cuda.synchronize()
        us = t0.elapsed_time(t1) * 1e3 / args.reps
        print(json.dumps({"call": args.call, "reps": args.reps, "us_per_call": round(us, 2),
                          "bytes_per_call": quant_bytes(*x.shape)}))
        return 0
    g = W.moe_grouped(seed=2, device="cuda")
    T, K = g.x_tokens.shape
    total = g.row_index.numel()
    E = g.num_experts
    if args.call == "route":
        # the dispatch permutation of the batch from its routes' expert ids
        off_h = g.offsets.cpu()
        ids = (torch.searchsorted(off_h, g.dest_rows.cpu(), right=True) - 1).to(torch.int32)
        ids = ids.cuda()
        fn = lambda: mx.moe_route(ids, E)  # noqa: E731
        fn()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(args.reps):
            fn()
        t1.record()
        torch.cuda.synchronize()
        print(json.dumps({"call": "route", "reps": args.reps,
                          "us_per_call": round(t0.elapsed_time(t1) * 1e3 / args.reps, 2)}))
        return 0
    codes = torch.empty((total, K // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty(mx.mxfp4_grouped_scale_bytes_bound(total, E, K), dtype=torch.uint8,
                         device="cuda")
    sro = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    st = torch.empty(1, dtype=torch.int32, device="cuda")
    ws_bytes = {"gather_ws": lambda: mx.mxfp4_gather_workspace_bytes(T, total, E, K),
                "scatter_ws": lambda: mx.mxfp4_scatter_workspace_bytes(T, total, E, K),
                "nvfp4_scatter_ws": lambda: mx.mxfp4_nvfp4_scatter_workspace_bytes(total, E, K),
                "nvfp4_scatter_ws_own_g":
                    lambda: mx.mxfp4_nvfp4_scatter_workspace_bytes(total, E, K)}
    gs = torch.full((E,), 448.0 * 6.0 / 5.0, device="cuda")
    if args.call == "nvfp4_scatter_ws_own_g":
        gs = (448.0 * 6.0 / torch.exp(torch.rand(E, generator=torch.Generator().manual_seed(2))
                                      * 3.0)).to("cuda")
    if args.call.startswith("nvfp4"):
        scales = torch.empty(mx.mxfp4_nvfp4_grouped_scale_bytes_bound(total, E, K),
                             dtype=torch.uint8, device="cuda")
    ws = (torch.empty(ws_bytes[args.call](), dtype=torch.uint8, device="cuda")
          if args.call in ws_bytes else None)
    fn = {
        "grouped": lambda: mx.mxfp4_quantize_grouped(g.x, g.offsets, codes, scales, sro, st),
        "gather": lambda: mx.mxfp4_quantize_grouped_gather(g.x_tokens, g.row_index, g.offsets,
                                                           codes, scales, sro, st),
        "gather_ws": lambda: mx.mxfp4_quantize_grouped_gather_ws(
            g.x_tokens, g.row_index, g.offsets, ws, codes, scales, sro, st),
        "scatter": lambda: mx.mxfp4_quantize_grouped_scatter(g.x_tokens, g.dest_rows, g.offsets,
                                                             total, codes, scales, sro, st),
        "scatter_ws": lambda: mx.mxfp4_quantize_grouped_scatter_ws(
            g.x_tokens, g.dest_rows, g.offsets, total, ws, codes, scales, sro, st),
        "nvfp4_scatter": lambda: mx.mxfp4_quantize_nvfp4_grouped_scatter(
            g.x_tokens, g.dest_rows, g.offsets, total, gs, codes, scales, sro, st),
        "nvfp4_scatter_ws": lambda: mx.mxfp4_quantize_nvfp4_grouped_scatter_ws(
            g.x_tokens, g.dest_rows, g.offsets, total, gs, ws, codes, scales, sro, st),
    }
    fn["nvfp4_scatter_ws_own_g"] = fn["nvfp4_scatter_ws"]
    fn = fn[args.call]
    fn()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.reps):
        fn()
    t1.record()
    torch.cuda.synchronize()
    print(json.dumps({"call": args.call, "reps": args.reps, "status": int(st.item()),
                      "us_per_call": round(t0.elapsed_time(t1) * 1e3 / args.reps, 2)}))


def run_sweep(args):
    """--sweep: the dense quantize (BF16, K = 7168 and K = 2048) over a range of
    row counts, one JSON line per size: device time per call from CUDA-graph
    batches of back-to-back calls after an L2 sweep, the inputs and outputs
    rotated over enough sets that together they exceed twice the L2, so no
    call finds its operands there.  Shows where the kernel leaves the launch
    and latency regime and reaches the copy bandwidth."""
    import torch
    import mxfp4_block_quantization_gb300 as mx
    import workloads as W
    torch.cuda.set_device(0)
    peak, _ = hbm_peak()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    sweep = L2Sweep(l2)
    side = torch.cuda.Stream()
    torch.cuda.set_stream(side)
    for K in (7168, 2048):
        for M in (128, 512, 1024, 2048, 4096, 8192, 16384, 65536):
            nb = quant_bytes(M, K)
            R = max(2, -(-2 * l2 // nb) + 1)
            x = W.dense_activation(1, M, K, device="cuda")
            xs = [x] + [x.clone() for _ in range(R - 1)]
            cs = [torch.empty((M, K // 2), dtype=torch.uint8, device="cuda") for _ in range(R)]
            ss = [torch.empty(mx.mxfp4_scale_bytes(M, K), dtype=torch.uint8, device="cuda")
                  for _ in range(R)]
            per = max(R, min(200, -(-(1 << 30) // nb)))
            mean, med = time_graph_batches(
                lambda i: mx.mxfp4_quantize(xs[i % R], cs[i % R], ss[i % R], side), side, sweep,
                per, 5)
            gbs = nb / (mean * 1e-3) / 1e9
            print(json.dumps({"sweep": "dense quantize", "M": M, "K": K, "ctas":
                              ((M + 127) // 128) * ((K // 32 + 3) // 4), "us": round(mean * 1e3, 2),
                              "median_us": round(med * 1e3, 2), "GB_per_s": round(gbs, 1),
                              "frac_of_peak": round(gbs / peak, 4), "rotating_sets": R}),
                  flush=True)
            del xs, cs, ss, x
            torch.cuda.empty_cache()
    return 0


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    import mxfp4_block_quantization_gb300 as mx
    import workloads as W

    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    props = torch.cuda.get_device_properties(dev)
    l2_bytes = int(getattr(props, "L2_cache_size", 128 << 20))
    peak, peak_src = hbm_peak()

    # ---- inputs: the 4096 x 7168 activation, R rotating copies > 2x L2
    x0 = W.dense_activation(1, M_DENSE, K_DENSE, device=dev)
    nbytes = quant_bytes(M_DENSE, K_DENSE)
    R = max(2, -(-2 * l2_bytes // nbytes) + 1)
    xs = [x0.clone() for _ in range(R)]
    codes = [torch.empty((M_DENSE, K_DENSE // 2), dtype=torch.uint8, device=dev) for _ in range(R)]
    sb = mx.mxfp4_scale_bytes(M_DENSE, K_DENSE)
    scales = [torch.empty(sb, dtype=torch.uint8, device=dev) for _ in range(R)]
    # the timed loop calls the C entry point directly with pre-marshalled
    # pointers, so the host issue rate is not what is measured
    import ctypes
    sp = ctypes.c_void_p(stream.cuda_stream)
    argsets = [(ctypes.c_void_p(xs[i].data_ptr()), ctypes.c_void_p(codes[i].data_ptr()),
                ctypes.c_void_p(scales[i].data_ptr())) for i in range(R)]
    qfn = mx._lib.mxfp4_quantize

    def step(i):
        a = argsets[i % R]
        rc = qfn(a[0], M_DENSE, K_DENSE, K_DENSE, a[1], a[2], sp)
        if rc:
            raise mx.MXFP4Error(rc, "mxfp4_quantize")

    xb_all = W.bf16_bits(x0) if (rank == 0 and world == 1 and not args.no_cpu) else None

    # ---- warm-up: W steps, then keep the GPU busy ~1 s so clocks settle
    sweep = L2Sweep(l2_bytes, dev)
    clocks = ClockSampler(local)
    clocks.start()
    clocks.wait_first()
    for i in range(args.warmup):
        sweep()                       # its first calls carry torch's one-time host work
        step(i)
    torch.cuda.synchronize()
    t_end = time.time() + args.settle
    i = 0
    while time.time() < t_end:
        for _ in range(200):
            step(i)
            i += 1
        torch.cuda.synchronize()

    # ---- timed region: an L2 sweep (torch reads 3x L2) is queued first, so
    # that the first step finds a cold L2 like every later one and the host
    # has the steps queued by the time the sweep ends; the events bracket the
    # K steps alone
    barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    torch.cuda.nvtx.range_push(f"timed: {args.steps} x mxfp4_quantize {M_DENSE}x{K_DENSE}")
    sweep()
    ev0.record(stream)
    for i in range(args.steps):
        step(i)
    ev1.record(stream)
    torch.cuda.nvtx.range_pop()
    ev1.synchronize()
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier()
    clocks.stop()
    local_ms = ev0.elapsed_time(ev1)
    max_ms, total_bytes = aggregate(local_ms, nbytes * args.steps)
    ms_per_step = max_ms / args.steps
    value = total_bytes / (max_ms * 1e-3) / 1e9
    kernel_gbs = nbytes / (local_ms / args.steps * 1e-3) / 1e9
    # the same kernel over 25 more batches of K steps, at most 200 (outside
    # the timed region): the median over batches of the per-step time
    _, med_ms = time_batches(step, stream, sweep, min(args.steps, 200), 25)

    # ---- e2e through the public API with pinned host buffers: per step the
    # matrix goes host -> device in 4 row chunks on a copy stream, each chunk
    # is quantized on a compute stream as soon as it lands, and its codes and
    # scales go device -> host on a third stream.  The three overlap, also
    # across steps: a chunk's device buffers are reused as soon as the
    # previous step has consumed them (per-chunk events), so the host link
    # never waits for a step to drain.
    x_host = x0.cpu().pin_memory()
    c_host = torch.empty((M_DENSE, K_DENSE // 2), dtype=torch.uint8).pin_memory()
    s_host = torch.empty(sb, dtype=torch.uint8).pin_memory()
    x_dev = torch.empty_like(x0)
    c_dev = torch.empty_like(codes[0])
    s_dev = torch.empty_like(scales[0])
    n_chunks = args.e2e_chunks
    chunk_rows = M_DENSE // n_chunks                # a multiple of 128: whole scale tiles
    tile_bytes = sb // (M_DENSE // 128)
    s_h2d, s_comp, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    chunks = []
    for j in range(n_chunks):
        r0, r1 = j * chunk_rows, (j + 1) * chunk_rows
        a0, a1 = r0 // 128 * tile_bytes, r1 // 128 * tile_bytes
        chunks.append((x_host[r0:r1], x_dev[r0:r1], c_dev[r0:r1], s_dev[a0:a1], c_host[r0:r1],
                       s_host[a0:a1], torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()))
    ev_start, ev_done = torch.cuda.Event(), torch.cuda.Event()

    def e2e_run(n_steps):
        ev_start.record(stream)
        for s_ in (s_h2d, s_comp, s_d2h):
            s_.wait_event(ev_start)
        for _ in range(n_steps):
            for xh, xd, cd, sd, ch, sh, ev_in, ev_q, ev_out in chunks:
                s_h2d.wait_event(ev_q)        # the previous step has quantized xd
                with torch.cuda.stream(s_h2d):
                    xd.copy_(xh, non_blocking=True)
                ev_in.record(s_h2d)
                s_comp.wait_event(ev_in)
                s_comp.wait_event(ev_out)     # the previous step's cd, sd are on the host
                mx.mxfp4_quantize(xd, cd, sd, stream=s_comp)
                ev_q.record(s_comp)
                s_d2h.wait_event(ev_q)
                with torch.cuda.stream(s_d2h):
                    ch.copy_(cd, non_blocking=True)
                    sh.copy_(sd, non_blocking=True)
                ev_out.record(s_d2h)
        ev_done.record(s_d2h)
        stream.wait_event(ev_done)

    e2e_steps = max(3, min(args.steps, 50))
    e2e_run(3)
    torch.cuda.synchronize()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push(f"e2e: {e2e_steps} pipelined host->device / quantize / device->host steps")
    e0.record(stream)
    e2e_run(e2e_steps)
    e1.record(stream)
    torch.cuda.nvtx.range_pop()
    e1.synchronize()
    e2e_ms, e2e_bytes = aggregate(e0.elapsed_time(e1), nbytes * e2e_steps)
    e2e_val = e2e_bytes / (e2e_ms * 1e-3) / 1e9

    # the host link on its own, for context: the same bytes per step (x to the
    # device, codes and scales back) as whole-buffer copies on the two copy
    # streams, no kernel; the copy engines set this ceiling, not the library
    def link_run(n_steps):
        ev_start.record(stream)
        for s_ in (s_h2d, s_d2h):
            s_.wait_event(ev_start)
        for _ in range(n_steps):
            with torch.cuda.stream(s_h2d):
                x_dev.copy_(x_host, non_blocking=True)
            with torch.cuda.stream(s_d2h):
                c_host.copy_(c_dev, non_blocking=True)
                s_host.copy_(s_dev, non_blocking=True)
        ev_done.record(s_h2d)
        stream.wait_event(ev_done)
        ev_done.record(s_d2h)
        stream.wait_event(ev_done)

    link_run(3)
    torch.cuda.synchronize()
    e0.record(stream)
    link_run(e2e_steps)
    e1.record(stream)
    e1.synchronize()
    link_gbs = (x_host.numel() * 2 + c_host.numel() + s_host.numel()) * e2e_steps / (
        e0.elapsed_time(e1) * 1e-3) / 1e9

    quality = reconstruction_report(mx, x0, codes[0], scales[0]) if rank == 0 else None

    rows, extra = None, None
    if not args.no_rows:
        rows, extra = measure_rows(mx, W, stream, peak, l2_bytes, sweep)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(xb_all)

    traffic = profiled_traffic()
    if rank == 0:
        clk = clocks.summary(t_wall0, t_wall1)
        if clk is not None:
            clk.pop("window", None)
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {
                "workload": f"dense activation quantize {M_DENSE}x{K_DENSE} BF16, "
                            "N(0,1) x 2^U(-8,8) per row, seed 1",
                "bytes_per_step": nbytes,
                "l2": f"{R} rotating input/output sets ({R * nbytes / 1e6:.0f} MB > 2x L2); "
                      "a 3x L2 read evicts the L2 before the timed steps",
                "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            },
            "roofline": {"bound": "hbm", "achieved": round(kernel_gbs, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(kernel_gbs / peak, 4),
                         "peak_src": "measured burst copy" if peak_src == "measured"
                         else "fallback 6.8 TB/s",
                         "traffic": traffic, "traffic_src": "ncu DRAM read+write of a mid-sequence launch",
                         "kernel": "quantize_tiles_kernel",
                         "median_us": round(med_ms * 1e3, 3)},
            "e2e": {"value": round(e2e_val, 2), "unit": "GB/s",
                    "h2d_bytes_per_step": x_host.numel() * 2,
                    "d2h_bytes_per_step": c_host.numel() + s_host.numel(),
                    "host_link_GB_per_s": round(link_gbs, 2),
                    "frac_of_host_link": round(e2e_val / link_gbs, 4)},
            "gpu_launches": args.steps,
            "clocks": clk,
            "cpu_baseline": cpu,
            "quality": quality,
            "extra": extra,
            "rows_fields": ROW_FIELDS,
            "rows": rows,
        }
        print(json.dumps(line, separators=(",", ":")), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-rows", action="store_true", help="skip the per-row measurements")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--call", choices=SINGLE_CALLS,
                    help="only time this one call (for profiling)")
    ap.add_argument("--reps", type=int, default=5, help="repetitions of --call")
    ap.add_argument("--sweep", action="store_true",
                    help="the dense quantize over a range of sizes, one JSON line each")
    ap.add_argument("--e2e-chunks", type=int, default=4, choices=(1, 2, 4, 8, 16, 32),
                    help="row chunks per step of the pipelined e2e measurement")
    ap.add_argument("--settle", type=float, default=1.0,
                    help="seconds of untimed launches after the warm-up steps (clock settling)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.call:
        return run_one_call(args)
    if args.sweep:
        return run_sweep(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
