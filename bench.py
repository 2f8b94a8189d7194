"""Benchmark of the 4-bit weight-quantized linear on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one Llama-3.2-1B-shaped decode token: 16 layers x {q, k, v, o, gate, up, down}
plus lm_head, M = 1, group size 32, fp16 scales, every layer its own weight buffers
(698.4 MB per token, far above the 129 MB L2, so each token streams the whole model from
HBM and no L2 flush is needed).  The 113 q4lin_run calls of a token are captured once in
a CUDA graph and replayed; steps are timed with CUDA events on the replay stream.

Printed: one JSON line with the aggregate GB/s, ms/token, the roofline of the GEMV kernel,
an end-to-end figure through the public C API with host copies, clocks sampled during the
timed region, the oracle timed on the host cores (rank 0, N = 1), and extra measurements
(8B decode token, per-shape GEMV bandwidth, 2- to 4-row GEMVs, prefill TFLOP/s, the
training-path kernels).

N > 1 (torchrun): replicas only -- each rank runs the same token on its own GPU with no
collective on the data path; a barrier brackets the timed region and the slowest rank's
time is reported; value = bytes of all ranks / that time ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode GEMV HBM GB/s & ms/token; prefill TFLOP/s; % roofline on 1 GB300"
GROUP = 32
L2_BYTES = 129 << 20

# DRAM bytes (read + write) of the 65 launches of one 1B decode token, summed from one ncu
# launch list (dram__bytes_read.sum + dram__bytes_write.sum per launch; the summary is
# profiles/gemv_tma_token_1b_launches.md).  Valid only for the kernel source it was taken
# with: the sha256 prefix of gemv_tma.cu + ptx.cuh; any other source reports null.
TOKEN_TRAFFIC = {"bytes": 698246656, "launches": 65, "source_sha256": "0702c7c64ddbcf43"}


def gemv_source_sha():
    import hashlib
    h = hashlib.sha256()
    for f in ("gemv_tma.cu", "ptx.cuh"):
        with open(os.path.join(ROOT, "bit_weight_quantized_int4_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def token_traffic_per_launch(launches):
    t = TOKEN_TRAFFIC
    if launches != t["launches"] or gemv_source_sha() != t["source_sha256"]:
        return None
    return round(t["bytes"] / t["launches"])

# (name, N, K) per decoder layer, in layer order; lm_head last.
LAYER_1B = [("q", 2048, 2048), ("k", 512, 2048), ("v", 512, 2048), ("o", 2048, 2048),
            ("gate", 8192, 2048), ("up", 8192, 2048), ("down", 2048, 8192)]
LAYER_8B = [("q", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096), ("o", 4096, 4096),
            ("gate", 14336, 4096), ("up", 14336, 4096), ("down", 4096, 14336)]
MODELS = {
    "1b": dict(layers=16, layer=LAYER_1B, head=("lm_head", 128256, 2048),
               desc="Llama-3.2-1B-shaped decode token"),
    "8b": dict(layers=32, layer=LAYER_8B, head=("lm_head", 128256, 4096),
               desc="Llama-3.1-8B-shaped decode token"),
}
PREFILL_NK = [(2048, 2048), (512, 2048), (8192, 2048), (2048, 8192)]


def gemv_bytes(N, K, gs=GROUP, scale_bytes=2, bias=False):
    """Algorithmic bytes of one M=1 GEMV: packed weight + scales + x + out (+ bias)."""
    return N * ((K + 1) // 2) + (-(-K // gs)) * N * scale_bytes + 4 * K + 4 * N + (4 * N if bias else 0)


def token_shapes(model):
    m = MODELS[model]
    shapes = []
    for layer in range(m["layers"]):
        for name, N, K in m["layer"]:
            shapes.append((f"{name}{layer}", N, K))
    shapes.append(m["head"])
    return shapes


# ------------------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons every 20 ms around the timed region.

    mark_start() / mark_end() bracket the timed region on the host clock; the summary keeps
    the samples whose nvidia-smi timestamp falls inside it (widened by one sampling period
    on each side), and says how many there were."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 20

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="q4clk_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(2 * self.PERIOD_MS / 1000)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    @staticmethod
    def _stamp(text):
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(text, fmt).timestamp()
            except ValueError:
                pass
        return None

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append(dict(t=self._stamp(parts[0]), sm=float(parts[2]),
                                 smax=float(parts[3]),
                                 power=float(parts[4]) if parts[4] not in ("[N/A]", "") else None,
                                 hw=parts[6], hwt=parts[7], swt=parts[8], swp=parts[9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        slack = self.PERIOD_MS / 1000
        inside = [r for r in rows if r["t"] is not None and self.t0 is not None and
                  self.t1 is not None and self.t0 - slack <= r["t"] <= self.t1 + slack]
        use = inside or rows
        reasons = set()
        for r in use:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in use),
                "sm_max_mhz": max(r["smax"] for r in use),
                "samples": len(use), "samples_in_timed_region": len(inside),
                "timed_region_s": round(self.t1 - self.t0, 4) if self.t0 and self.t1 else None,
                "reasons": sorted(reasons)}


# -------------------------------------------------------------------------- distributed
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value, world, device=None):
    """Largest value over all ranks (the slowest rank's time)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------- our workload
# Projections of a layer that read the same activation (fused into one launch).
SHARED_INPUT = ({"q", "k", "v"}, {"gate", "up"})


def token_groups(model):
    """Consecutive shapes of a token that read the same x: [[(name, N, K), ...], ...]."""
    groups = []
    for name, N, K in token_shapes(model):
        base = name.rstrip("0123456789")
        if groups:
            prev = groups[-1][-1][0].rstrip("0123456789")
            same_layer = name[len(base):] == groups[-1][-1][0][len(prev):]
            if same_layer and any(base in g and prev in g for g in SHARED_INPUT):
                groups[-1].append((name, N, K))
                continue
        groups.append([(name, N, K)])
    return groups


class DecodeToken:
    """Device buffers of one model's decode token and the q4lin calls over them.

    Each group of projections that read the same activation (q/k/v, gate/up) has one x
    buffer and runs as one q4lin_run_grouped call (or as separate q4lin_run calls with
    grouped=False).  Every projection has its own weight, scale and output buffers."""

    def __init__(self, handle, model, device, seed_base=1000, grouped=True):
        import torch
        self.torch = torch
        self.h = handle
        self.grouped = grouped
        self.groups = token_groups(model)
        gen = torch.Generator(device=device)
        self.bufs = []  # per group: list of (N, K, w, s, out_offset)
        x_sizes, oo, i = [], 0, 0
        for grp in self.groups:
            entries = []
            for name, N, K in grp:
                gen.manual_seed(seed_base + i)
                i += 1
                w = torch.randint(0, 256, (N, (K + 1) // 2), dtype=torch.uint8, device=device,
                                  generator=gen)
                s = (torch.rand((-(-K // GROUP), N), device=device, generator=gen) * 0.015
                     + 0.005).to(torch.float16)
                entries.append((N, K, w, s, oo))
                oo += N
            self.bufs.append(entries)
            x_sizes.append(grp[0][2])
        # All activations of a token in one buffer, all outputs in another, so an
        # end-to-end step is one host->device and one device->host copy.
        self.x_offsets = [sum(x_sizes[:g]) for g in range(len(x_sizes))]
        self.x_all = torch.randn(sum(x_sizes), device=device, generator=gen)
        self.out_all = torch.empty(oo, device=device)
        self.bytes = sum(
            sum(N * ((K + 1) // 2) + (-(-K // GROUP)) * N * 2 + 4 * N for N, K, _, _, _ in entries)
            + 4 * entries[0][1] for entries in self.bufs)
        self.gemvs = sum(len(e) for e in self.bufs)
        self.launches = len(self.bufs) if grouped else self.gemvs

    def run(self, stream_ptr):
        from bit_weight_quantized_int4_gb300 import q4lin as q
        xb, ob = self.x_all.data_ptr(), self.out_all.data_ptr()
        for entries, xo in zip(self.bufs, self.x_offsets):
            probs = [(xb + 4 * xo, w.data_ptr(), s.data_ptr(), None, ob + 4 * oo, 1, N, K, GROUP,
                      q.Q4LIN_SCALE_F16) for N, K, w, s, oo in entries]
            if self.grouped and len(probs) > 1:
                st = q.q4lin_run_grouped(self.h, probs, stream_ptr)
            else:
                for pr in probs:
                    st = q.q4lin_run(self.h, *pr, stream_ptr)
                    if st != q.Q4LIN_OK:
                        break
            if st != q.Q4LIN_OK:
                raise q.Q4LinError(st, "q4lin_run")

    def head_output(self):
        N, _, _, _, oo = self.bufs[-1][-1]
        return self.out_all[oo:oo + N]

    def capture(self):
        torch = self.torch
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self.run(side.cuda_stream)          # loads every kernel before capture
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run(torch.cuda.current_stream().cuda_stream)
        return g


def time_graph(torch, graph, steps, warmup, world, clk=None):
    """ms per replay, CUDA events on the replay stream, barrier + sync on both sides (the
    clock sampler, if given, is told when the timed region starts and ends)."""
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            graph.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if clk is not None:
        clk.mark_start()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps):
            graph.replay()
        end.record(stream)
    torch.cuda.synchronize()
    if clk is not None:
        clk.mark_end()
    barrier(world)
    return start.elapsed_time(end) / steps


def measure_e2e(torch, token, graph, steps, warmup):
    """Per step: pinned host x -> device, the token's graph, lm_head logits -> pinned host."""
    x_host = torch.empty(token.x_all.numel(), dtype=torch.float32, pin_memory=True)
    x_host.copy_(token.x_all.cpu())
    head = token.head_output()
    out_host = torch.empty(head.numel(), dtype=torch.float32, pin_memory=True)
    stream = torch.cuda.Stream()

    def step():
        token.x_all.copy_(x_host, non_blocking=True)
        graph.replay()
        out_host.copy_(head, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps):
            step()
        end.record(stream)
    end.synchronize()
    ms = start.elapsed_time(end) / steps
    return ms, x_host.numel() * 4, out_host.numel() * 4


def graph_time_us(torch, launch, count, reps=1):
    """Device time per launch: `count` launches (launch(i, stream_ptr)) captured in one CUDA
    graph, replayed once untimed and `reps` times timed with CUDA events on the replay
    stream (no host launch overhead inside the timed region)."""
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        launch(0, side.cuda_stream)              # loads the kernels before capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(count):
            launch(i, torch.cuda.current_stream().cuda_stream)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(reps):
            g.replay()
        end.record(stream)
    end.synchronize()
    del g
    return start.elapsed_time(end) * 1000 / (count * reps)


def weight_copies(torch, N, K, bytes_each, l2_bytes=L2_BYTES, cap=1024):
    """Enough distinct (weight, scale) copies that cycling through them streams at least
    three L2 capacities, so every launch reads its weights from HBM."""
    copies = int(min(cap, max(2, -(-3 * l2_bytes // bytes_each))))
    ws = [torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device="cuda") for _ in range(copies)]
    ss = [(torch.rand((K // GROUP, N), device="cuda") * 0.015 + 0.005).half() for _ in range(copies)]
    return ws, ss


def shape_bandwidth(torch, handle, N, K, M=1):
    """GB/s of one GEMV shape (M activation rows) in isolation, every launch on its own
    weight copy (HBM-cold weights; x stays L2-resident as it would in a model)."""
    from bit_weight_quantized_int4_gb300 import q4lin as q
    b = gemv_bytes(N, K) + 4 * (M - 1) * (K + N)
    ws, ss = weight_copies(torch, N, K, b)
    x = torch.randn(M, K, device="cuda")
    out = torch.empty(M, N, device="cuda")

    def launch(i, sp):
        st = q.q4lin_run(handle, x.data_ptr(), ws[i % len(ws)].data_ptr(),
                         ss[i % len(ws)].data_ptr(), None, out.data_ptr(), M, N, K, GROUP,
                         q.Q4LIN_SCALE_F16, sp)
        assert st == q.Q4LIN_OK

    us = graph_time_us(torch, launch, len(ws))
    del ws, ss
    row = {"N": N, "K": K, "us": round(us, 3), "GB_s": round(b / us / 1e3, 1)}
    if M > 1:
        row["M"] = M
    return row


def prefill_tflops(torch, handle, M, N, K, reps=10):
    """TFLOP/s (2*M*N*K per launch) of one prefill shape: `reps` launches captured in a CUDA
    graph, device time from CUDA events around a replay."""
    from bit_weight_quantized_int4_gb300 import q4lin as q
    w = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device="cuda")
    s = torch.rand((K // GROUP, N), device="cuda") * 0.015 + 0.005
    bias = torch.randn(N, device="cuda") * 0.1
    x = torch.randn(M, K, device="cuda")
    out = torch.empty(M, N, device="cuda")
    st, path = q.q4lin_plan(handle, x.data_ptr(), w.data_ptr(), s.data_ptr(), bias.data_ptr(),
                            out.data_ptr(), M, N, K, GROUP, q.Q4LIN_SCALE_F32)

    def launch(i, sp):
        r = q.q4lin_run(handle, x.data_ptr(), w.data_ptr(), s.data_ptr(), bias.data_ptr(),
                        out.data_ptr(), M, N, K, GROUP, q.Q4LIN_SCALE_F32, sp)
        assert r == q.Q4LIN_OK

    us = graph_time_us(torch, launch, reps)
    return {"M": M, "N": N, "K": K, "path": q.PATH_NAMES[path], "us": round(us, 2),
            "TFLOP_s": round(2.0 * M * N * K / (us * 1e-6) / 1e12, 2)}


def backward_bandwidth(torch, handle, M, N, K):
    """Input gradient d_x[M,K] = d_out[M,N] @ dequant(W): device time per launch (CUDA graph,
    every launch on its own HBM-cold weight copy) and GB/s of the algorithmic bytes (packed
    codes + fp16 scales read once per 8 rows of d_out, d_out, d_x)."""
    from bit_weight_quantized_int4_gb300 import q4lin as q
    wbytes = gemv_bytes(N, K) - 4 * K - 4 * N
    ws, ss = weight_copies(torch, N, K, wbytes)
    d_out = torch.randn(M, N, device="cuda")
    d_x = torch.empty(M, K, device="cuda")

    def launch(i, sp):
        st = q.q4lin_run_backward_dx(handle, d_out.data_ptr(), ws[i % len(ws)].data_ptr(),
                                     ss[i % len(ws)].data_ptr(), d_x.data_ptr(), M, N, K,
                                     GROUP, q.Q4LIN_SCALE_F16, sp)
        assert st == q.Q4LIN_OK

    us = graph_time_us(torch, launch, len(ws))
    byts = wbytes * (-(-M // 8)) + 4 * M * N + 4 * M * K
    del ws, ss
    return {"op": "backward_dx", "M": M, "N": N, "K": K, "us": round(us, 3),
            "GB_s": round(byts / us / 1e3, 1)}


def requant_bandwidth(torch, handle, N, K):
    """Re-quantisation of fp32 latents [N,K]: device time and GB/s of latent + scales read
    and packed codes written."""
    from bit_weight_quantized_int4_gb300 import q4lin as q
    latent = torch.randn(N, K, device="cuda") * 0.05
    scales = (torch.rand((K // GROUP, N), device="cuda") * 0.015 + 0.005).half()
    codes = torch.empty(N, K // 2, dtype=torch.uint8, device="cuda")

    def launch(i, sp):
        st = q.q4lin_run_requant(handle, latent.data_ptr(), scales.data_ptr(), codes.data_ptr(),
                                 N, K, GROUP, q.Q4LIN_SCALE_F16, sp)
        assert st == q.Q4LIN_OK

    us = graph_time_us(torch, launch, 10)
    byts = 4 * N * K + 2 * (K // GROUP) * N + N * K // 2
    return {"op": "requant", "N": N, "K": K, "us": round(us, 3), "GB_s": round(byts / us / 1e3, 1)}


# ------------------------------------------------------------------------- CPU baseline
def cpu_baseline(min_seconds=10.0, row_fraction=8):
    """The fp64 oracle, as it stands, on the host cores: every matrix of a 1B decode
    token restricted to its first N/row_fraction rows, repeated until min_seconds."""
    import numpy as np
    import oracle
    rng = np.random.Generator(np.random.PCG64(7))
    mats, nbytes = [], 0
    for name, N, K in token_shapes("1b"):
        n = max(1, N // row_fraction)
        w = rng.integers(0, 256, size=(n, K // 2), dtype=np.uint8)
        s = rng.uniform(0.005, 0.02, size=(K // GROUP, n)).astype(np.float16)
        x = rng.standard_normal((1, K), dtype=np.float32)
        mats.append((x, w, s, K))
        nbytes += gemv_bytes(n, K)
    oracle.build()
    t0 = time.perf_counter()
    passes = 0
    while True:
        for x, w, s, K in mats:
            oracle.linear(x, w, s, None, K, GROUP)
        passes += 1
        if time.perf_counter() - t0 >= min_seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": round(nbytes * passes / dt / 1e9, 4), "unit": "GB/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": (f"1B decode token, first 1/{row_fraction} of the rows of each of the "
                       f"113 matrices ({nbytes / 1e6:.1f} MB), {passes} passes, {dt:.1f} s"),
            "ms_per_token_equiv": round(dt / passes * row_fraction * 1000, 1)}


def run_reference(args, world, rank):
    """The reference arm: the fp64 oracle on the host cores (no GPU work)."""
    if rank != 0:
        return 0
    for _ in range(args.warmup):
        cpu_baseline(min_seconds=0.0)
    # Each step repeats the bounded sample for at least 1 s, or less when there are many
    # steps, so that the whole arm takes about a minute of host time.
    per_step = min(1.0, 60.0 / max(1, args.steps))
    vals = [cpu_baseline(min_seconds=per_step) for _ in range(args.steps)]
    gbs = statistics.median(v["value"] for v in vals)
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": statistics.median(v["ms_per_token_equiv"] for v in vals),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config("1b"),
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": vals[0]["cores"],
                             "kind": "oracle", "sample": vals[0]["sample"]},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def token_bytes(model):
    """Algorithmic bytes of one decode token: every packed weight, scale and output once,
    and each activation once per group of projections that share it."""
    total = 0
    for grp in token_groups(model):
        total += 4 * grp[0][2]
        for _, N, K in grp:
            total += N * ((K + 1) // 2) + (-(-K // GROUP)) * N * 2 + 4 * N
    return total


def workload_config(model):
    shapes = token_shapes(model)
    b = token_bytes(model)
    return {"workload": f"{MODELS[model]['desc']}: {len(shapes)} q4 GEMVs (M=1, group 32, "
                        f"fp16 scales, distinct buffers per layer), {b / 1e6:.1f} MB per token",
            "bytes_per_step": b, "gemvs_per_step": len(shapes),
            "l2": "inputs larger than L2 (129 MB): every token streams from HBM; no flush",
            "parallelism": "replicas"}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return p["hbm_gbs"], p.get("bf16_tflops"), "measured"
    return 6800.0, 1900.0, "fallback"


CROSSOVER_M = (1, 2, 3, 4, 5, 7, 8, 12, 16, 24, 32, 33, 48, 64, 96, 128, 256, 512)
CROSSOVER_NK = ((2048, 2048), (8192, 2048), (2048, 8192), (128256, 2048), (1000, 2048),
                (4096, 14336), (14336, 4096))


def crossover():
    """Device time per launch of each forced path (CUDA-core row streaming, the generic
    FFMA kernel, the tensor-core GEMM) over M for several (N, K): one JSON row per (N, K, M).
    Every launch in a graph reads its own weight copy, so weights come from HBM."""
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    h = q.q4lin_create(0)
    paths = (("gemv", q.Q4LIN_PATH_GEMV), ("ffma", q.Q4LIN_PATH_FFMA), ("tc", q.Q4LIN_PATH_TC))
    for N, K in CROSSOVER_NK:
        ws, ss = weight_copies(torch, N, K, gemv_bytes(N, K), cap=64)
        for M in CROSSOVER_M:
            x = torch.randn(M, K, device="cuda")
            out = torch.empty(M, N, device="cuda")
            row = {"N": N, "K": K, "M": M, "copies": len(ws)}
            for name, path in paths:
                q.q4lin_set_option(h, q.Q4LIN_OPT_FORCE_PATH, path)
                st, _ = q.q4lin_plan(h, x.data_ptr(), ws[0].data_ptr(), ss[0].data_ptr(), None,
                                     out.data_ptr(), M, N, K, GROUP, q.Q4LIN_SCALE_F16)
                if st != q.Q4LIN_OK or (name == "ffma" and M * N * K > (1 << 34)):
                    row[name + "_us"] = None
                    continue

                def launch(i, sp):
                    r = q.q4lin_run(h, x.data_ptr(), ws[i % len(ws)].data_ptr(),
                                    ss[i % len(ws)].data_ptr(), None, out.data_ptr(), M, N, K,
                                    GROUP, q.Q4LIN_SCALE_F16, sp)
                    assert r == q.Q4LIN_OK

                row[name + "_us"] = round(graph_time_us(torch, launch, len(ws)), 2)
            q.q4lin_set_option(h, q.Q4LIN_OPT_FORCE_PATH, q.Q4LIN_PATH_AUTO)
            st, auto = q.q4lin_plan(h, x.data_ptr(), ws[0].data_ptr(), ss[0].data_ptr(), None,
                                    out.data_ptr(), M, N, K, GROUP, q.Q4LIN_SCALE_F16)
            row["auto"] = q.PATH_NAMES[auto]
            print(json.dumps(row), flush=True)
        del ws, ss
        torch.cuda.empty_cache()
    q.q4lin_destroy(h)
    return 0


def profile(spec):
    """A handful of launches of one op, nothing printed: a target for ncu."""
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    h = q.q4lin_create(0)
    kind, *dims = spec.split(":")
    if kind == "token":
        token = DecodeToken(h, dims[0], "cuda")
        for _ in range(3):
            token.run(torch.cuda.current_stream().cuda_stream)
    elif kind == "gemv":
        N, K = int(dims[0]), int(dims[1])
        shape_bandwidth(torch, h, N, K, int(dims[2]) if len(dims) > 2 else 1)
    elif kind == "prefill":
        M, N, K = (int(d) for d in dims)
        prefill_tflops(torch, h, M, N, K, reps=3)
    elif kind == "backward":
        M, N, K = (int(d) for d in dims)
        backward_bandwidth(torch, h, M, N, K)
    elif kind == "requant":
        N, K = (int(d) for d in dims)
        requant_bandwidth(torch, h, N, K)
    else:
        raise SystemExit(f"unknown profile spec {spec}")
    torch.cuda.synchronize()
    q.q4lin_destroy(h)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-group", action="store_true",
                    help="run every projection as its own q4lin_run call (113 launches per "
                         "1B token) instead of fusing those that share an input")
    ap.add_argument("--pdl", type=int, default=1, choices=[0, 1],
                    help="launch with programmatic dependent launch (kernels start "
                         "streaming weights while the previous one drains)")
    ap.add_argument("--crossover", action="store_true",
                    help="time the CUDA-core and tensor-core paths over M and print the "
                         "measured table (JSON) instead of the benchmark line")
    ap.add_argument("--profile", default=None,
                    help="run a few launches of one op and exit (for ncu): gemv:N:K[:M], "
                         "prefill:M:N:K, backward:M:N:K, requant:N:K or token:1b|8b")
    args = ap.parse_args()
    if args.profile:
        return profile(args.profile)
    if args.crossover:
        return crossover()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        return run_reference(args, world, rank)

    import torch
    torch.cuda.set_device(local)
    from bit_weight_quantized_int4_gb300 import q4lin as q
    h = q.q4lin_create(local)
    q.q4lin_set_option(h, q.Q4LIN_OPT_PDL, args.pdl)

    token = DecodeToken(h, "1b", "cuda", grouped=not args.no_group)
    graph = token.capture()
    with ClockSampler(local) as clk:
        ms = time_graph(torch, graph, args.steps, args.warmup, world, clk)
    clocks = clk.summary()
    ms_max = max_over_ranks(ms, world, device="cuda")
    total_bytes = token.bytes * world
    gbs = total_bytes / (ms_max * 1e-3) / 1e9
    hbm_peak, bf16_peak, peak_src = load_peaks()
    per_gpu_gbs = token.bytes / (ms * 1e-3) / 1e9

    e2e_ms, h2d, d2h = measure_e2e(torch, token, graph, args.steps, args.warmup)
    e2e_ms = max_over_ranks(e2e_ms, world, device="cuda")

    extra = {}
    if not args.no_extra and rank == 0:
        tok8 = DecodeToken(h, "8b", "cuda", seed_base=2000, grouped=not args.no_group)
        g8 = tok8.capture()
        ms8 = time_graph(torch, g8, max(5, args.steps // 4), 3, 1)
        extra["decode_8b"] = {"ms_per_token": round(ms8, 4),
                              "GB_s": round(tok8.bytes / (ms8 * 1e-3) / 1e9, 1),
                              "bytes_per_token": tok8.bytes, "launches": tok8.launches,
                              "gemvs": tok8.gemvs}
        del g8, tok8
        torch.cuda.empty_cache()
        seen, shapes = set(), []
        for _, N, K in token_shapes("1b") + token_shapes("8b") + [("fused", 22016, 4096)]:
            if (N, K) not in seen:
                seen.add((N, K))
                shapes.append(shape_bandwidth(torch, h, N, K))
        extra["gemv_shapes"] = shapes
        # A few activation rows (speculative decoding, small batches): the multi-row GEMV.
        extra["small_m"] = [shape_bandwidth(torch, h, N, K, M) for M in (2, 3, 4)
                            for N, K in ((8192, 2048), (2048, 8192), (128256, 2048))]
        extra["prefill"] = [prefill_tflops(torch, h, M, N, K)
                            for M in (128, 512, 2048) for N, K in PREFILL_NK]
        extra["training"] = ([backward_bandwidth(torch, h, M, N, K)
                              for M in (1, 8) for N, K in ((2048, 2048), (8192, 2048), (2048, 8192))]
                             + [requant_bandwidth(torch, h, N, K)
                                for N, K in ((2048, 2048), (8192, 2048), (2048, 8192))])

    line = {
        "metric": METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 4),
        "ms_per_token": round(ms_max, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(workload_config("1b"), pdl=bool(args.pdl), grouped=not args.no_group,
                       launches_per_step=token.launches),
        "roofline": {"bound": "hbm", "achieved": round(per_gpu_gbs, 1), "peak": hbm_peak,
                     "unit": "GB/s", "frac": round(per_gpu_gbs / hbm_peak, 4),
                     "traffic": token_traffic_per_launch(token.launches),
                     "traffic_unit": "bytes per launch (mean over the token)",
                     "algorithmic_bytes_per_launch": round(token.bytes / token.launches),
                     "kernel": f"gemv_tma_kernel (all {token.launches} launches of a token; "
                               "launch gaps included)", "peak_source": peak_src},
        "e2e": {"value": round(token.bytes * world / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "clocks": clocks,
        "gpu_launches": token.launches * args.steps,
        "gemvs_per_step": token.gemvs,
    }
    if extra:
        line["extra"] = extra
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(line))
    q.q4lin_destroy(h)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
