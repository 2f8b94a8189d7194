"""Benchmark of the 4-bit weight-quantized linear on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one Llama-3.1-8B-shaped decode token, the largest workload that fits one GPU:
32 layers x {q, k, v, o, gate, up, down} plus lm_head, M = 1, group size 32, fp16 scales,
every layer its own weight buffers (4230.8 MB per token, far above the 129 MB L2, so each
token streams the whole model from HBM and no L2 flush is needed).  The projections that
read the same activation (q/k/v, gate/up) run as one q4lin_run_grouped call; the 129
calls of a token are captured once in a CUDA graph and replayed, with programmatic
dependent launch, so each launch reads its x only after the previous one completed (the
dependency chain of a decoder).  Steps are timed with CUDA events on the replay stream.

Printed: one JSON line with the token's aggregate GB/s and ms/token, the roofline of the
decode GEMV, the roofline of the prefill GEMM (per-shape TFLOP/s against the tensor-core
peaks), an end-to-end figure that calls the public C API every step with host copies,
clocks sampled during the timed region, the oracle timed on the host cores (rank 0,
N = 1), the Llama-3.2-1B-shaped token, and extra per-shape measurements.  Per-shape
figures are the median over >= 100 timed launches after >= 20 warm-up launches, each
launch on its own weight copy (enough copies to stream three L2 capacities), so weights
come from HBM.

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
HEADLINE = "8b"

# DRAM bytes (read + written) of one launch of each launch shape of a decode token, from
# one-launch ncu captures (dram__bytes_read.sum + dram__bytes_write.sum; bench.py
# --profile launch:<model>:<kind>, each launch on its own cold weights).  Valid only for
# the kernel code they were taken with (gemv_source_sha); any other code reports null.
LAUNCH_TRAFFIC = {"source_sha256": "f530a05ba646638e", "bytes": {
    "8b:qkv": 14203648, "8b:o": 9482240, "8b:gateup": 66401536, "8b:down": 33116672,
    "8b:lm_head": 298558208, "1b:qkv": 3575808, "1b:o": 2395904, "1b:gateup": 18919168,
    "1b:down": 9507072, "1b:lm_head": 150955776}}


def gemv_source_sha():
    """sha256 prefix of the decode GEMV's code (gemv_tma.cu + ptx.cuh with // comments and
    blank lines removed: a comment edit does not invalidate the traffic captures)."""
    import hashlib
    h = hashlib.sha256()
    for f in ("gemv_tma.cu", "ptx.cuh"):
        with open(os.path.join(ROOT, "bit_weight_quantized_int4_gb300", "csrc", f)) as fh:
            code = [ln.split("//", 1)[0].rstrip() for ln in fh.read().splitlines()]
        h.update(("\n".join(ln for ln in code if ln) + "\n").encode())
    return h.hexdigest()[:16]


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
# Prefill (N, K) classes of a Llama-3.2-1B layer: q/o, k/v, gate/up, down.
PREFILL_NK = [(2048, 2048), (512, 2048), (8192, 2048), (2048, 8192)]
PREFILL_LAYER_COUNTS = {(2048, 2048): 2, (512, 2048): 2, (8192, 2048): 2, (2048, 8192): 1}
PREFILL_M = (128, 512, 2048)


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


def launch_kind(group):
    """Launch shape of a token group: qkv, o, gateup, down or lm_head."""
    names = "".join(n.rstrip("0123456789") for n, _, _ in group)
    return {"qkv": "qkv", "gateup": "gateup"}.get(names, names)


def token_bytes(model):
    """Algorithmic bytes of one decode token: every packed weight, scale and output once,
    and each activation once per group of projections that share it."""
    total = 0
    for grp in token_groups(model):
        total += 4 * grp[0][2]
        for _, N, K in grp:
            total += N * ((K + 1) // 2) + (-(-K // GROUP)) * N * 2 + 4 * N
    return total


def token_traffic_per_launch(model, source_sha=None, table=None):
    """Mean DRAM bytes per launch of a grouped decode token, from the per-launch-shape
    captures; None unless every launch shape was captured with the current source."""
    t = LAUNCH_TRAFFIC if table is None else table
    sha = gemv_source_sha() if source_sha is None else source_sha
    if not t.get("source_sha256") or sha != t["source_sha256"]:
        return None
    groups = token_groups(model)
    total = 0
    for g in groups:
        b = t["bytes"].get(f"{model}:{launch_kind(g)}")
        if b is None:
            return None
        total += b
    return round(total / len(groups))


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
class DecodeToken:
    """Device buffers of one model's decode token and the q4lin calls over them.

    Each group of projections that read the same activation (q/k/v, gate/up) has one x
    buffer.  grouped=True runs the whole token as one q4lin_run_grouped call (which fuses
    each group into one launch); grouped=False as one q4lin_run call per projection.
    Every projection has its own weight, scale and output buffers."""

    def __init__(self, handle, model, device, seed_base=1000, grouped=True):
        import torch
        self.torch = torch
        self.h = handle
        self.model = model
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
        self.bytes = token_bytes(model)
        self.gemvs = sum(len(e) for e in self.bufs)
        self.launches = len(self.bufs) if grouped else self.gemvs

    def problem_tuples(self):
        from bit_weight_quantized_int4_gb300 import q4lin as q
        xb, ob = self.x_all.data_ptr(), self.out_all.data_ptr()
        per_group = []
        for entries, xo in zip(self.bufs, self.x_offsets):
            per_group.append([(xb + 4 * xo, w.data_ptr(), s.data_ptr(), None, ob + 4 * oo, 1, N,
                               K, GROUP, q.Q4LIN_SCALE_F16) for N, K, w, s, oo in entries])
        return per_group

    def run(self, stream_ptr):
        from bit_weight_quantized_int4_gb300 import q4lin as q
        if self.grouped:
            # One call over the whole token, as a serving loop makes it: the library fuses
            # the projections that share an input.
            st = q.q4lin_run_grouped(self.h, [p for grp in self.problem_tuples() for p in grp],
                                     stream_ptr)
            if st != q.Q4LIN_OK:
                raise q.Q4LinError(st, "q4lin_run_grouped")
            return
        for probs in self.problem_tuples():
            for pr in probs:
                st = q.q4lin_run(self.h, *pr, stream_ptr)
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


def measure_e2e_api(torch, token, steps, warmup):
    """End to end through the public C API, every step: pinned host activations -> device,
    ONE q4lin_run_grouped call over all the token's projections (the library validates
    them, fuses those that share an input and launches; nothing is captured or replayed),
    the lm_head logits -> pinned host.  CUDA events on the stream bracket the steps, so
    host-side launch time that the GPU waits for is included."""
    from bit_weight_quantized_int4_gb300 import q4lin as q
    probs = [p for grp in token.problem_tuples() for p in grp]
    arr = (q.q4lin_problem_t * len(probs))(*[q.q4lin_problem_t(*p) for p in probs])
    x_host = torch.empty(token.x_all.numel(), dtype=torch.float32, pin_memory=True)
    x_host.copy_(token.x_all.cpu())
    head = token.head_output()
    out_host = torch.empty(head.numel(), dtype=torch.float32, pin_memory=True)
    stream = torch.cuda.Stream()

    def step():
        token.x_all.copy_(x_host, non_blocking=True)
        st = q.q4lin_run_grouped_array(token.h, arr, len(probs), stream.cuda_stream)
        if st != q.Q4LIN_OK:
            raise q.Q4LinError(st, "q4lin_run_grouped")
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


def measure_e2e_graph(torch, token, graph, steps, warmup):
    """The same copies around a replay of the token's captured graph."""
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
    return start.elapsed_time(end) / steps


def median_launch_us(torch, launch, count, min_reps=100, min_warmup=20):
    """Device time per launch: `count` launches (launch(i, stream_ptr), each on its own
    weight copy) captured in one CUDA graph; replays until >= min_warmup launches have run
    untimed, then timed replays (CUDA events on the replay stream, one pair per replay)
    until >= min_reps launches; returns (median over replays of replay time / count, reps)."""
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        launch(0, side.cuda_stream)              # loads the kernels before capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(count):
            launch(i, torch.cuda.current_stream().cuda_stream)
    stream = torch.cuda.Stream()
    warm = max(1, -(-min_warmup // count))
    replays = max(5, -(-min_reps // count))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(replays)]
    with torch.cuda.stream(stream):
        for _ in range(warm):
            g.replay()
        for a, b in evs:
            a.record(stream)
            g.replay()
            b.record(stream)
    torch.cuda.synchronize()
    times = [a.elapsed_time(b) * 1000 / count for a, b in evs]
    del g
    return statistics.median(times), replays * count


def copies_for(bytes_each, l2_bytes=L2_BYTES, cap=1024):
    """Distinct weight copies so that cycling through them streams >= 3 L2 capacities."""
    return int(min(cap, max(2, -(-3 * l2_bytes // bytes_each))))


def weight_copies(torch, N, K, bytes_each, scale_dtype=None, cap=1024):
    import torch as _t
    dt = scale_dtype if scale_dtype is not None else _t.float16
    copies = copies_for(bytes_each, cap=cap)
    ws = [torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device="cuda") for _ in range(copies)]
    ss = [(torch.rand((K // GROUP, N), device="cuda") * 0.015 + 0.005).to(dt) for _ in range(copies)]
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

    us, reps = median_launch_us(torch, launch, len(ws))
    del ws, ss
    row = {"N": N, "K": K, "us": round(us, 3), "GB_s": round(b / us / 1e3, 1), "reps": reps}
    if M > 1:
        row["M"] = M
    return row


def prefill_time(torch, handle, M, N, K, bias=True, min_reps=100, f16=False):
    """One prefill shape (fp32 scales, group 32, fp32 bias): median device time per launch
    over >= min_reps launches, each on its own HBM-cold weight copy, and TFLOP/s of
    2*M*N*K.  f16: with the tensor-core path's fp16 operands (Q4LIN_OPT_TC_F16; the time
    includes the conversion of x)."""
    from bit_weight_quantized_int4_gb300 import q4lin as q
    q.q4lin_set_option(handle, q.Q4LIN_OPT_TC_F16, int(f16))
    wbytes = N * K // 2 + (K // GROUP) * N * 4
    ws, ss = weight_copies(torch, N, K, wbytes, scale_dtype=torch.float32, cap=256)
    bvec = torch.randn(N, device="cuda") * 0.1
    x = torch.randn(M, K, device="cuda")
    out = torch.empty(M, N, device="cuda")
    bp = bvec.data_ptr() if bias else None
    st, kernel = q.q4lin_plan_kernel(handle, x.data_ptr(), ws[0].data_ptr(), ss[0].data_ptr(),
                                     bp, out.data_ptr(), M, N, K, GROUP, q.Q4LIN_SCALE_F32)
    assert st == q.Q4LIN_OK

    def launch(i, sp):
        r = q.q4lin_run(handle, x.data_ptr(), ws[i % len(ws)].data_ptr(),
                        ss[i % len(ws)].data_ptr(), bp, out.data_ptr(), M, N, K, GROUP,
                        q.Q4LIN_SCALE_F32, sp)
        assert r == q.Q4LIN_OK

    us, reps = median_launch_us(torch, launch, len(ws), min_reps=min_reps)
    q.q4lin_set_option(handle, q.Q4LIN_OPT_TC_F16, 0)
    del ws, ss
    return {"M": M, "N": N, "K": K, "kernel": q.KERNEL_NAMES[kernel], "us": round(us, 2),
            "TFLOP_s": round(2.0 * M * N * K / (us * 1e-6) / 1e12, 2), "reps": reps}


def backward_bandwidth(torch, handle, M, N, K):
    """Input gradient d_x[M,K] = d_out[M,N] @ dequant(W): median device time per launch
    (every launch on its own HBM-cold weight copy) and GB/s of the algorithmic bytes
    (packed codes + fp16 scales read once per 8 rows of d_out, d_out, d_x)."""
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

    us, reps = median_launch_us(torch, launch, len(ws))
    byts = wbytes * (-(-M // 8)) + 4 * M * N + 4 * M * K
    del ws, ss
    return {"op": "backward_dx", "M": M, "N": N, "K": K, "us": round(us, 3),
            "GB_s": round(byts / us / 1e3, 1), "reps": reps}


def requant_bandwidth(torch, handle, N, K):
    """Re-quantisation of fp32 latents [N,K]: median device time and GB/s of latent +
    scales read and packed codes written (latent copies rotated: HBM-cold)."""
    from bit_weight_quantized_int4_gb300 import q4lin as q
    byts = 4 * N * K + 2 * (K // GROUP) * N + N * K // 2
    n = copies_for(byts, cap=64)
    latents = [torch.randn(N, K, device="cuda") * 0.05 for _ in range(n)]
    scales = (torch.rand((K // GROUP, N), device="cuda") * 0.015 + 0.005).half()
    codes = torch.empty(N, K // 2, dtype=torch.uint8, device="cuda")

    def launch(i, sp):
        st = q.q4lin_run_requant(handle, latents[i % n].data_ptr(), scales.data_ptr(),
                                 codes.data_ptr(), N, K, GROUP, q.Q4LIN_SCALE_F16, sp)
        assert st == q.Q4LIN_OK

    us, reps = median_launch_us(torch, launch, n)
    del latents
    return {"op": "requant", "N": N, "K": K, "us": round(us, 3), "GB_s": round(byts / us / 1e3, 1),
            "reps": reps}


def cublas_tf32_tflops(torch, n=8192, reps=10):
    """Dense tf32 GEMM rate of this GPU through cuBLAS (torch.matmul on fp32 with tf32
    allowed), best of `reps` (burst): the tf32 tensor-core ceiling the prefill GEMM is
    compared with, measured the same way as the bf16 peak of the peaks file."""
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        a = torch.randn(n, n, device="cuda")
        b = torch.randn(n, n, device="cuda")
        for _ in range(3):
            torch.matmul(a, b)
        best = 1e30
        for _ in range(reps):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            torch.matmul(a, b)
            e.record()
            e.synchronize()
            best = min(best, s.elapsed_time(e))
        del a, b
        return round(2.0 * n ** 3 / (best * 1e-3) / 1e12, 1)
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


# The highest tf32 tensor rate seen on this part: a bare loop of tcgen05.mma kind::tf32
# (128 x 256 x 8 MMAs, A in tensor memory, zero operands, no loads), measured once on a
# GB300 at 2.07 GHz during development.  Reported beside the live cuBLAS figure, as the
# tighter denominator.
TF32_MMA_LOOP_TFLOPS = 1216.0


def prefill_roofline(torch, handle, bf16_peak):
    """Per-shape prefill TFLOP/s (Llama-3.2-1B layer shapes at M = 128 / 512 / 2048,
    bias on all but k/v) against the tensor-core peaks, and the 16-layer prefill time."""
    tf32_derived = round(bf16_peak * 1.1 / 2.25, 1) if bf16_peak else None
    tf32_cublas = cublas_tf32_tflops(torch)
    shapes = []
    for M in PREFILL_M:
        for N, K in PREFILL_NK:
            r = prefill_time(torch, handle, M, N, K, bias=(N != 512))
            r["frac_of_tf32_derived"] = round(r["TFLOP_s"] / tf32_derived, 4) if tf32_derived else None
            r["frac_of_tf32_cublas"] = round(r["TFLOP_s"] / tf32_cublas, 4)
            r["frac_of_tf32_mma_loop"] = round(r["TFLOP_s"] / TF32_MMA_LOOP_TFLOPS, 4)
            r["frac_of_bf16"] = round(r["TFLOP_s"] / bf16_peak, 4) if bf16_peak else None
            shapes.append(r)
    layer16 = []
    for M in PREFILL_M:
        t = sum(PREFILL_LAYER_COUNTS[(s["N"], s["K"])] * s["us"] for s in shapes if s["M"] == M)
        fl = sum(PREFILL_LAYER_COUNTS[(s["N"], s["K"])] * 2.0 * M * s["N"] * s["K"]
                 for s in shapes if s["M"] == M)
        layer16.append({"M": M, "ms": round(16 * t / 1000, 4),
                        "TFLOP_s": round(fl / (t * 1e-6) / 1e12, 2)})
    top = layer16[-1]
    # The same shapes with fp16 operands (kind::f16, twice the tf32 MMA rate), against the
    # dense 16-bit peak of the peaks file.
    shapes16 = []
    for M in PREFILL_M:
        for N, K in PREFILL_NK:
            r = prefill_time(torch, handle, M, N, K, bias=(N != 512), f16=True)
            r["frac_of_bf16"] = round(r["TFLOP_s"] / bf16_peak, 4) if bf16_peak else None
            shapes16.append(r)
    layer16_f16 = []
    for M in PREFILL_M:
        t = sum(PREFILL_LAYER_COUNTS[(s["N"], s["K"])] * s["us"] for s in shapes16 if s["M"] == M)
        fl = sum(PREFILL_LAYER_COUNTS[(s["N"], s["K"])] * 2.0 * M * s["N"] * s["K"]
                 for s in shapes16 if s["M"] == M)
        layer16_f16.append({"M": M, "ms": round(16 * t / 1000, 4),
                            "TFLOP_s": round(fl / (t * 1e-6) / 1e12, 2)})
    top16 = layer16_f16[-1]
    f16_block = {"kernel": "tc_wa_kernel with fp16 operands (Q4LIN_OPT_TC_F16: x converted by "
                           "x_to_f16_kernel, tcgen05.mma kind::f16)",
                 "achieved": top16["TFLOP_s"], "peak": bf16_peak, "unit": "TFLOP/s",
                 "frac": round(top16["TFLOP_s"] / bf16_peak, 4) if bf16_peak else None,
                 "peak_source": "bf16_tflops of the peaks file (dense 16-bit; fp16 = bf16 rate)",
                 "shapes": shapes16, "layer16": layer16_f16}
    return {"bound": "tensor", "kernel": "tc_wa_kernel (tcgen05.mma kind::tf32, TMEM accumulators)",
            "workload": "16-layer Llama-3.2-1B-shaped prefill GEMMs at M=2048 (fp32 scales, group 32)",
            "achieved": top["TFLOP_s"], "peak": tf32_cublas, "unit": "TFLOP/s",
            "frac": round(top["TFLOP_s"] / tf32_cublas, 4),
            "peak_source": "cuBLAS tf32 GEMM 8192^3 measured in this run (burst)",
            "tf32_derived_peak": tf32_derived,
            "tf32_derived_source": "bf16_tflops of the peaks file x 1.1/2.25 (nominal tf32 : bf16)",
            "frac_of_tf32_derived": round(top["TFLOP_s"] / tf32_derived, 4) if tf32_derived else None,
            "tf32_mma_loop_peak": TF32_MMA_LOOP_TFLOPS,
            "tf32_mma_loop_source": "bare tcgen05.mma kind::tf32 loop (128x256x8, A in TMEM), "
                                    "measured once on this part at 2.07 GHz",
            "frac_of_tf32_mma_loop": round(top["TFLOP_s"] / TF32_MMA_LOOP_TFLOPS, 4),
            "bf16_peak": bf16_peak,
            "frac_of_bf16": round(top["TFLOP_s"] / bf16_peak, 4) if bf16_peak else None,
            "timing": "median of >= 100 launches after >= 20 warm-up, weight copies rotated (HBM-cold)",
            "shapes": shapes, "layer16": layer16, "f16": f16_block}


# ------------------------------------------------------------------------- CPU baseline
def _cpu_shapes():
    """(label, N, K, scale dtype, rows of x) of every distinct shape the baseline times:
    the decode GEMVs of both tokens (fp16 scales) and the prefill classes (fp32 scales)."""
    seen, out = set(), []
    for model in ("1b", "8b"):
        for _, N, K in token_shapes(model):
            if (N, K) not in seen:
                seen.add((N, K))
                out.append((f"gemv {N}x{K}", N, K, "f16", 1))
    for N, K in PREFILL_NK:
        out.append((f"prefill {N}x{K}", N, K, "f32", 4))
    return out


def cpu_baseline_worker(target_s=0.4):
    """Runs in a child process (thread count from OMP_NUM_THREADS): the oracle on a row
    subset of every shape, sized to about target_s of work, scaled to the full shape."""
    import numpy as np
    import oracle
    oracle.build()
    rng = np.random.Generator(np.random.PCG64(7))
    res = []
    for label, N, K, sdt, M in _cpu_shapes():
        x = rng.standard_normal((M, K), dtype=np.float32)
        n = 16
        while True:
            w = rng.integers(0, 256, size=(n, K // 2), dtype=np.uint8)
            s = rng.uniform(0.005, 0.02, size=(K // GROUP, n)).astype(
                np.float16 if sdt == "f16" else np.float32)
            t0 = time.perf_counter()
            oracle.linear(x, w, s, None, K, GROUP)
            dt = time.perf_counter() - t0
            if dt >= target_s or n >= N:
                break
            n = min(N, max(2 * n, int(n * target_s / max(dt, 1e-4) * 1.2)))
        # Small shapes (all rows in less than target_s): repeat until target_s, keep the
        # fastest pass.
        reps, t_start = 1, time.perf_counter()
        while time.perf_counter() - t_start < target_s:
            t0 = time.perf_counter()
            oracle.linear(x, w, s, None, K, GROUP)
            dt = min(dt, time.perf_counter() - t0)
            reps += 1
        res.append({"label": label, "N": N, "K": K, "M": M, "rows_timed": n, "passes": reps,
                    "ms_full": dt * 1000 * N / n})
    return {"threads": oracle.num_threads(), "shapes": res}


def _run_worker(threads):
    env = dict(os.environ)
    if threads:
        env["OMP_NUM_THREADS"] = str(threads)
    else:
        env.pop("OMP_NUM_THREADS", None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--cpu-worker"],
                       capture_output=True, text=True, env=env, timeout=600)
    if r.returncode != 0:
        raise RuntimeError(f"cpu baseline worker failed: {r.stderr[-1000:]}")
    return json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])


def _cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return None


def cpu_baseline_summary(one, allc):
    """Combine the single-thread and all-core worker results into per-shape, per-token
    and per-16-layer-prefill figures."""
    def by_shape(r):
        return {(s["N"], s["K"], s["M"]): s for s in r["shapes"]}
    s1, sa = by_shape(one), by_shape(allc)
    per_shape = []
    for key, s in sa.items():
        N, K, M = key
        per_shape.append({"shape": s["label"], "M": M, "ms_1_thread": round(s1[key]["ms_full"], 2),
                          f"ms_{allc['threads']}_threads": round(s["ms_full"], 2),
                          "rows_timed": [s1[key]["rows_timed"], s["rows_timed"]]})
    tokens = {}
    for model in ("1b", "8b"):
        t1 = sum(s1[(N, K, 1)]["ms_full"] for _, N, K in token_shapes(model))
        ta = sum(sa[(N, K, 1)]["ms_full"] for _, N, K in token_shapes(model))
        b = token_bytes(model)
        tokens[model] = {"ms_1_thread": round(t1, 1), "ms_all": round(ta, 1),
                         "GB_s_1_thread": round(b / (t1 * 1e-3) / 1e9, 4),
                         "GB_s_all": round(b / (ta * 1e-3) / 1e9, 4)}
    prefill = []
    for M in PREFILL_M:
        t1 = sum(c * s1[(N, K, 4)]["ms_full"] * M / 4 for (N, K), c in PREFILL_LAYER_COUNTS.items())
        ta = sum(c * sa[(N, K, 4)]["ms_full"] * M / 4 for (N, K), c in PREFILL_LAYER_COUNTS.items())
        fl = sum(c * 2.0 * M * N * K for (N, K), c in PREFILL_LAYER_COUNTS.items())
        prefill.append({"M": M, "ms_16_layers_1_thread": round(16 * t1, 1),
                        "ms_16_layers_all": round(16 * ta, 1),
                        "GFLOP_s_all": round(fl / (ta * 1e-3) / 1e9, 2)})
    return per_shape, tokens, prefill


def cpu_baseline():
    """The fp64 oracle, as it stands, on the host cores, single-thread and all cores: every
    distinct shape on a row subset (about 0.4 s of work each), scaled to the full shape;
    per token (both models) and per 16-layer prefill.  value = the 8B token's GB/s on all
    cores."""
    t0 = time.perf_counter()
    one = _run_worker(1)
    allc = _run_worker(None)
    per_shape, tokens, prefill = cpu_baseline_summary(one, allc)
    dt = time.perf_counter() - t0
    return {"value": tokens[HEADLINE]["GB_s_all"], "unit": "GB/s", "cores": allc["threads"],
            "kind": "oracle", "cpu_model": _cpu_model(),
            "sample": (f"every distinct GEMV shape of the 1B and 8B decode tokens (fp16 scales) "
                       f"and the 4 prefill (N, K) classes (4 rows of x, fp32 scales), each on a "
                       f"row subset timed for ~0.4 s and scaled to the full rows; single-thread "
                       f"and {allc['threads']} threads; {dt:.1f} s of host time in all"),
            "ms_per_token": {m: v["ms_all"] for m, v in tokens.items()},
            "tokens": tokens, "per_shape": per_shape, "prefill_16_layers": prefill}


def reference_step(min_seconds):
    """One step of the reference arm: the oracle on all host cores over a fixed sample of
    the 8B decode token (the first 1/64 of the rows of each distinct shape, >= 16 rows),
    repeated for at least min_seconds; GB/s of the token scaled by the rows sampled."""
    import numpy as np
    import oracle
    oracle.build()
    rng = np.random.Generator(np.random.PCG64(11))
    counts = {}
    for _, N, K in token_shapes(HEADLINE):
        counts[(N, K)] = counts.get((N, K), 0) + 1
    mats = []
    for (N, K), c in counts.items():
        n = max(16, N // 64)
        mats.append((rng.standard_normal((1, K), dtype=np.float32),
                     rng.integers(0, 256, size=(n, K // 2), dtype=np.uint8),
                     rng.uniform(0.005, 0.02, size=(K // GROUP, n)).astype(np.float16),
                     N, K, n, c))
    t_token, passes = 0.0, 0
    t_start = time.perf_counter()
    while True:
        for x, w, s, N, K, n, c in mats:
            t0 = time.perf_counter()
            oracle.linear(x, w, s, None, K, GROUP)
            t_token += (time.perf_counter() - t0) * N / n * c
        passes += 1
        if time.perf_counter() - t_start >= min_seconds:
            break
    ms = t_token / passes * 1000
    return {"ms_per_token": ms, "GB_s": token_bytes(HEADLINE) / (ms * 1e-3) / 1e9,
            "threads": oracle.num_threads(), "passes": passes}


def run_reference(args, world, rank):
    """The reference arm: the fp64 oracle on the host cores (no GPU work)."""
    if rank != 0:
        return 0
    for _ in range(args.warmup):
        reference_step(0.0)
    per_step = min(1.0, 60.0 / max(1, args.steps))
    vals = [reference_step(per_step) for _ in range(args.steps)]
    gbs = statistics.median(v["GB_s"] for v in vals)
    sample = (f"{MODELS[HEADLINE]['desc']}: the first 1/64 of the rows (>= 16) of each distinct "
              f"matrix, timed and scaled by rows and occurrences, >= {per_step:.2f} s per step")
    line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(statistics.median(v["ms_per_token"] for v in vals), 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(HEADLINE),
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": vals[0]["threads"],
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


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
    """Device time per launch of each forced path (CUDA-core GEMV family, the generic FFMA
    kernel, the tensor-core GEMM, the small-M tensor-core GEMM) over M for several (N, K):
    one JSON row per (N, K, M),
    with the kernel each path runs and the one AUTO picks.  Every launch reads its own
    weight copy (HBM-cold); median over >= 20 launches."""
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    h = q.q4lin_create(0)
    q.q4lin_set_option(h, q.Q4LIN_OPT_PDL, 1)
    paths = (("gemv", q.Q4LIN_PATH_GEMV), ("ffma", q.Q4LIN_PATH_FFMA), ("tc", q.Q4LIN_PATH_TC),
             ("tc_small", q.Q4LIN_PATH_TC_SMALL))
    for N, K in CROSSOVER_NK:
        ws, ss = weight_copies(torch, N, K, gemv_bytes(N, K), cap=64)
        for M in CROSSOVER_M:
            x = torch.randn(M, K, device="cuda")
            out = torch.empty(M, N, device="cuda")
            row = {"N": N, "K": K, "M": M, "copies": len(ws)}
            for name, path in paths:
                q.q4lin_set_option(h, q.Q4LIN_OPT_FORCE_PATH, path)
                st, kern = q.q4lin_plan_kernel(h, x.data_ptr(), ws[0].data_ptr(),
                                               ss[0].data_ptr(), None, out.data_ptr(), M, N, K,
                                               GROUP, q.Q4LIN_SCALE_F16)
                if st != q.Q4LIN_OK or (name == "ffma" and M * N * K > (1 << 34)):
                    row[name + "_us"] = None
                    continue

                def launch(i, sp):
                    r = q.q4lin_run(h, x.data_ptr(), ws[i % len(ws)].data_ptr(),
                                    ss[i % len(ws)].data_ptr(), None, out.data_ptr(), M, N, K,
                                    GROUP, q.Q4LIN_SCALE_F16, sp)
                    assert r == q.Q4LIN_OK

                row[name + "_us"] = round(median_launch_us(torch, launch, len(ws), min_reps=20,
                                                           min_warmup=5)[0], 2)
                row[name + "_kernel"] = q.KERNEL_NAMES[kern]
            q.q4lin_set_option(h, q.Q4LIN_OPT_FORCE_PATH, q.Q4LIN_PATH_AUTO)
            st, auto = q.q4lin_plan_kernel(h, x.data_ptr(), ws[0].data_ptr(), ss[0].data_ptr(),
                                           None, out.data_ptr(), M, N, K, GROUP,
                                           q.Q4LIN_SCALE_F16)
            row["auto_kernel"] = q.KERNEL_NAMES[auto]
            print(json.dumps(row), flush=True)
        del ws, ss
        torch.cuda.empty_cache()
    q.q4lin_destroy(h)
    return 0


def profile(spec):
    """A handful of launches of one op, nothing printed: a target for ncu.

    launch:<model>:<kind> runs one launch shape of a decode token (qkv, o, gateup, down,
    lm_head) three times, each on its own freshly drawn weights."""
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    h = q.q4lin_create(0)
    kind, *dims = spec.split(":")
    if kind == "token":
        token = DecodeToken(h, dims[0], "cuda")
        for _ in range(3):
            token.run(torch.cuda.current_stream().cuda_stream)
    elif kind == "launch":
        model, lk = dims
        group = next(g for g in token_groups(model) if launch_kind(g) == lk)
        K = group[0][2]
        x = torch.randn(K, device="cuda")
        sp = torch.cuda.current_stream().cuda_stream
        for rep in range(3):
            probs, keep = [], []
            for _, N, _ in group:
                w = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device="cuda")
                s = (torch.rand((K // GROUP, N), device="cuda") * 0.015 + 0.005).half()
                o = torch.empty(N, device="cuda")
                keep += [w, s, o]
                probs.append((x.data_ptr(), w.data_ptr(), s.data_ptr(), None, o.data_ptr(), 1, N,
                              K, GROUP, q.Q4LIN_SCALE_F16))
            st = q.q4lin_run_grouped(h, probs, sp)
            assert st == q.Q4LIN_OK
            torch.cuda.synchronize()
    elif kind == "gemv":
        N, K = int(dims[0]), int(dims[1])
        shape_bandwidth(torch, h, N, K, int(dims[2]) if len(dims) > 2 else 1)
    elif kind in ("prefill", "prefill16"):
        M, N, K = (int(d) for d in dims)
        prefill_time(torch, h, M, N, K, min_reps=3, f16=kind == "prefill16")
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
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-group", action="store_true",
                    help="run every projection as its own q4lin_run call instead of fusing "
                         "those that share an input")
    ap.add_argument("--pdl", type=int, default=1, choices=[0, 1],
                    help="launch with programmatic dependent launch (kernels start "
                         "streaming weights while the previous one drains)")
    ap.add_argument("--crossover", action="store_true",
                    help="time the CUDA-core and tensor-core paths over M and print the "
                         "measured table (JSON) instead of the benchmark line")
    ap.add_argument("--profile", default=None,
                    help="run a few launches of one op and exit (for ncu): gemv:N:K[:M], "
                         "prefill:M:N:K, prefill16:M:N:K, backward:M:N:K, requant:N:K, "
                         "token:1b|8b or "
                         "launch:1b|8b:qkv|o|gateup|down|lm_head")
    ap.add_argument("--cpu-worker", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.cpu_worker:
        print(json.dumps(cpu_baseline_worker()))
        return 0
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
    hbm_peak, bf16_peak, peak_src = load_peaks()

    token = DecodeToken(h, HEADLINE, "cuda", grouped=not args.no_group)
    graph = token.capture()
    with ClockSampler(local) as clk:
        ms = time_graph(torch, graph, args.steps, args.warmup, world, clk)
    clocks = clk.summary()
    ms_max = max_over_ranks(ms, world, device="cuda")
    gbs = token.bytes * world / (ms_max * 1e-3) / 1e9
    per_gpu_gbs = token.bytes / (ms * 1e-3) / 1e9

    e2e_ms, h2d, d2h = measure_e2e_api(torch, token, args.steps, args.warmup)
    e2e_ms = max_over_ranks(e2e_ms, world, device="cuda")
    e2e_graph_ms = measure_e2e_graph(torch, token, graph, args.steps, args.warmup)
    launches = token.launches
    del graph, token
    torch.cuda.empty_cache()

    extra, prefill = {}, None
    tok1 = DecodeToken(h, "1b", "cuda", seed_base=2000, grouped=not args.no_group)
    g1 = tok1.capture()
    ms1 = time_graph(torch, g1, max(20, args.steps), 3, world)
    e2e1, _, _ = measure_e2e_api(torch, tok1, max(20, args.steps), 3)
    decode_1b = {"ms_per_token": round(ms1, 4), "GB_s": round(tok1.bytes / (ms1 * 1e-3) / 1e9, 1),
                 "frac_of_hbm": round(tok1.bytes / (ms1 * 1e-3) / 1e9 / hbm_peak, 4),
                 "bytes_per_token": tok1.bytes, "launches": tok1.launches, "gemvs": tok1.gemvs,
                 "e2e_api_ms": round(e2e1, 4),
                 "traffic_per_launch": token_traffic_per_launch("1b")}
    del g1, tok1
    torch.cuda.empty_cache()
    if not args.no_extra and rank == 0:
        prefill = prefill_roofline(torch, h, bf16_peak)
        seen, shapes = set(), []
        for _, N, K in token_shapes("1b") + token_shapes("8b") + [("fused", 22016, 4096)]:
            if (N, K) not in seen:
                seen.add((N, K))
                shapes.append(shape_bandwidth(torch, h, N, K))
        for s in shapes:
            s["frac_of_hbm"] = round(s["GB_s"] / hbm_peak, 4)
        extra["gemv_shapes"] = shapes
        # A few activation rows (speculative decoding, small batches): the multi-row GEMV,
        # and from 3 rows on large matrices (on few row blocks with its K split) the small-M
        # tensor-core GEMM (AUTO's choice; each row names the kernel that ran).
        from bit_weight_quantized_int4_gb300 import q4lin as q
        small = []
        for M in (2, 3, 4, 8, 16, 32):
            for N, K in ((8192, 2048), (2048, 8192), (128256, 2048), (28672, 4096), (4096, 4096),
                         (4096, 14336)):
                row = shape_bandwidth(torch, h, N, K, M)
                x = torch.empty(M, K, device="cuda")
                w = torch.empty(N, K // 2, dtype=torch.uint8, device="cuda")
                sc = torch.empty(K // GROUP, N, dtype=torch.float16, device="cuda")
                o = torch.empty(M, N, device="cuda")
                st, kern = q.q4lin_plan_kernel(h, x.data_ptr(), w.data_ptr(), sc.data_ptr(), None,
                                               o.data_ptr(), M, N, K, GROUP, q.Q4LIN_SCALE_F16)
                row["kernel"] = q.KERNEL_NAMES[kern] if st == q.Q4LIN_OK else None
                row["frac_of_hbm"] = round(row["GB_s"] / hbm_peak, 4)
                small.append(row)
        extra["small_m"] = small
        extra["training"] = ([backward_bandwidth(torch, h, M, N, K)
                              for M in (1, 8) for N, K in ((2048, 2048), (8192, 2048), (2048, 8192))]
                             + [requant_bandwidth(torch, h, N, K)
                                for N, K in ((2048, 2048), (8192, 2048), (2048, 8192))])

    line = {
        "metric": METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 4),
        "ms_per_token": round(ms_max, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(workload_config(HEADLINE), pdl=bool(args.pdl), grouped=not args.no_group,
                       launches_per_step=launches),
        "roofline": {"bound": "hbm", "achieved": round(per_gpu_gbs, 1), "peak": hbm_peak,
                     "unit": "GB/s", "frac": round(per_gpu_gbs / hbm_peak, 4),
                     "traffic": token_traffic_per_launch(HEADLINE),
                     "traffic_unit": "DRAM bytes per launch (mean over the token's launches)",
                     "algorithmic_bytes_per_launch": round(token_bytes(HEADLINE) / launches),
                     "kernel": f"gemv_tma_kernel (all {launches} launches of a token; "
                               "launch gaps included)", "peak_source": peak_src},
        "e2e": {"value": round(token_bytes(HEADLINE) * world / (e2e_ms * 1e-3) / 1e9, 1),
                "unit": "GB/s", "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "how": "one q4lin_run_grouped C-API call per step over all 225 projections "
                       "(validation, fusion and launches each step), pinned H2D of every "
                       "activation before it and D2H of the logits after it",
                "graph_replay_ms_per_step": round(e2e_graph_ms, 4)},
        "clocks": clocks,
        "gpu_launches": launches * args.steps,
        "decode_1b": decode_1b,
    }
    if prefill is not None:
        line["prefill_roofline"] = prefill
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
