"""Reader for the hand-derived worked example under tests/golden/."""
import os

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_worked_example():
    rows = {}
    with open(os.path.join(GOLDEN_DIR, "worked_example_2x4x8.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            rows.setdefault(key, []).append(vals)
    ex = {k: int(rows[k][0][0]) for k in ("M", "N", "K", "group_size")}
    f32 = lambda k: np.array([[float(v) for v in r] for r in rows[k]], dtype=np.float32)
    f64 = lambda k: np.array([[float(v) for v in r] for r in rows[k]], dtype=np.float64)
    ex["x"] = f32("x")
    ex["qweight"] = np.array([[int(v, 16) for v in r] for r in rows["qweight"]], np.uint8)
    ex["scales"] = f32("scales")
    ex["bias"] = f32("bias")[0]
    ex["scales_per_channel"] = f32("scales_per_channel")[0]
    for k in ("out_nobias", "out_bias", "mag", "out_swapped_nobias",
              "out_per_channel_nobias"):
        ex[k] = f64(k)
    ex["bw_d_out"] = f32("bw_d_out")
    ex["bw_d_x"] = f64("bw_d_x")
    return ex


def load_requant_example():
    rows = {}
    with open(os.path.join(GOLDEN_DIR, "requant_example_2x8.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            rows.setdefault(key, []).append(vals)
    return {
        "scales": np.array([[float(v) for v in r] for r in rows["scales"]], np.float32),
        "latent": np.array([[float(v) for v in r] for r in rows["latent"]], np.float32),
        "qweight": np.array([[int(v, 16) for v in r] for r in rows["qweight"]], np.uint8),
        "group_size": 4,
    }
