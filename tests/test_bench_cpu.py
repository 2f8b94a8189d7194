"""Host logic of bench.py that needs no GPU: the clock sampler keeps only the nvidia-smi
samples taken inside the timed region and reports the throttle reasons seen there."""
import datetime
import os
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _write_log(path, t0, rows):
    with open(path, "w") as f:
        for dt, mhz, power_cap in rows:
            ts = datetime.datetime.fromtimestamp(t0 + dt).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
            cap = "Active" if power_cap else "Not Active"
            f.write(f"{ts}, 0, {mhz}, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, {cap}\n")


def test_clock_summary_keeps_the_timed_region():
    import bench
    c = bench.ClockSampler(0)
    fd, c.path = tempfile.mkstemp()
    os.close(fd)
    t0 = time.time()
    # Outside the region (idle, 2070 MHz) and inside it (1900 MHz, one power-cap sample).
    _write_log(c.path, t0, [(-0.5, 2070, False), (0.01, 1900, False), (0.05, 1900, True),
                            (0.09, 1900, False), (0.6, 2070, False)])
    c.proc = object()
    c.t0, c.t1 = t0, t0 + 0.1
    s = c.summary()
    assert s["samples_in_timed_region"] == 3 and s["samples"] == 3
    assert s["sm_mhz"] == 1900.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    assert not os.path.exists(c.path)


def test_clock_summary_without_samples_in_region_uses_all():
    import bench
    c = bench.ClockSampler(0)
    fd, c.path = tempfile.mkstemp()
    os.close(fd)
    t0 = time.time()
    _write_log(c.path, t0, [(-0.5, 2070, False), (0.6, 2070, False)])
    c.proc = object()
    c.t0, c.t1 = t0, t0 + 0.01
    s = c.summary()
    assert s["samples_in_timed_region"] == 0 and s["samples"] == 2
    assert s["sm_mhz"] == 2070.0 and s["reasons"] == []


def test_clock_summary_without_nvidia_smi():
    import bench
    c = bench.ClockSampler(0)
    assert c.summary()["reasons"] == ["nvidia-smi unavailable"]


def test_token_bytes_are_the_algorithmic_bytes():
    """Bytes of one decode token, the numerator of the bench's GB/s and roofline: every
    packed weight (N * K/2), fp16 group scale (K/32 * N * 2) and output (4N) once, and each
    activation (4K) once per group of projections that read it (q/k/v, o, gate/up, down,
    lm_head)."""
    import bench

    def matrix(N, K):
        return N * (K // 2) + (K // 32) * N * 2 + 4 * N

    for model, want in (("1b", 698053632), ("8b", 4230812672)):
        m = bench.MODELS[model]
        per_layer = sum(matrix(N, K) for _, N, K in m["layer"])
        per_layer += sum(4 * K for name, _, K in m["layer"] if name in ("q", "o", "gate", "down"))
        _, hN, hK = m["head"]
        total = m["layers"] * per_layer + matrix(hN, hK) + 4 * hK
        assert bench.token_bytes(model) == total == want


def test_token_groups_share_x():
    import bench
    groups = bench.token_groups("1b")
    assert len(groups) == 16 * 4 + 1
    assert [n.rstrip("0123456789") for n, _, _ in groups[0]] == ["q", "k", "v"]
    assert [n.rstrip("0123456789") for n, _, _ in groups[2]] == ["gate", "up"]
    assert groups[-1] == [("lm_head", 128256, 2048)]


def test_launch_kinds_of_a_token():
    import bench
    kinds = [bench.launch_kind(g) for g in bench.token_groups("8b")]
    assert kinds[:4] == ["qkv", "o", "gateup", "down"] and kinds[-1] == "lm_head"
    assert len(kinds) == 32 * 4 + 1


def test_token_traffic_needs_every_launch_shape_and_the_source():
    """Traffic per launch = captured bytes of each launch shape summed over the token's
    launches / launches; null unless the capture's source hash is the current one and
    every launch shape was captured."""
    import bench
    table = {"source_sha256": "abc", "bytes": {"8b:qkv": 1000, "8b:o": 200, "8b:gateup": 3000,
                                               "8b:down": 400, "8b:lm_head": 50000}}
    want = round((32 * (1000 + 200 + 3000 + 400) + 50000) / 129)
    assert bench.token_traffic_per_launch("8b", "abc", table) == want
    assert bench.token_traffic_per_launch("8b", "def", table) is None
    assert bench.token_traffic_per_launch("1b", "abc", table) is None
    assert bench.token_traffic_per_launch("8b", "abc", {"source_sha256": None, "bytes": {}}) is None


def test_cpu_baseline_summary_scales_shapes_to_tokens_and_prefill():
    """Per-token oracle time = sum over the token's GEMVs of the per-shape time; 16-layer
    prefill = 16 x sum over the layer's classes (count x per-4-row time x M / 4)."""
    import bench

    def worker(threads, ms):
        return {"threads": threads,
                "shapes": [{"label": l, "N": N, "K": K, "M": M, "rows_timed": 16,
                            "ms_full": ms(N, K, M)} for l, N, K, _, M in bench._cpu_shapes()]}
    one = worker(1, lambda N, K, M: N * K * M * 1e-6)
    allc = worker(16, lambda N, K, M: N * K * M * 1e-7)
    per_shape, tokens, prefill = bench.cpu_baseline_summary(one, allc)
    assert len(per_shape) == len(bench._cpu_shapes())
    t8 = sum(N * K * 1e-7 for _, N, K in bench.token_shapes("8b"))
    assert abs(tokens["8b"]["ms_all"] - round(t8, 1)) < 1e-9
    assert abs(tokens["8b"]["GB_s_all"] - round(bench.token_bytes("8b") / (t8 * 1e-3) / 1e9, 4)) < 1e-9
    p = {r["M"]: r for r in prefill}
    t = 16 * sum(c * N * K * 4 * 1e-6 * 2048 / 4 for (N, K), c in bench.PREFILL_LAYER_COUNTS.items())
    assert abs(p[2048]["ms_16_layers_1_thread"] - round(t, 1)) < 1e-9
