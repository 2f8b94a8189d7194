"""Pins of the oracle's training-path routines (CPU only): the input gradient
d_x = d_out @ dequant(W) ("linear_q4gsw_backward") and the re-quantisation of fp32
latents to 4-bit codes ("q4gsw_requant").  Each routine is checked against something
other than itself: hand-derived examples, the adjoint identity with the (separately
pinned) forward oracle, a numpy dense brute force, special cases, and planted mistakes.
"""
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from bit_weight_quantized_int4_gb300 import synth
from tests._golden import load_requant_example, load_worked_example
from tests.test_oracle import dense_dequant


# ----------------------------------------------------------------- input gradient d_x
@pytest.mark.parametrize("scale_dtype", [np.float32, np.float16])
def test_backward_worked_example(scale_dtype):
    ex = load_worked_example()
    d_x, _ = oracle.backward_dx(ex["bw_d_out"], ex["qweight"], ex["scales"].astype(scale_dtype),
                                ex["K"], ex["group_size"])
    np.testing.assert_array_equal(d_x, ex["bw_d_x"])


@pytest.mark.parametrize("M,N,K,gs,f16", [(1, 64, 256, 32, True), (3, 37, 77, 8, False),
                                          (5, 129, 100, 100, False), (2, 16, 33, 1, True)])
def test_backward_adjoint_of_forward(M, N, K, gs, f16):
    """<d_out, W x> == <W^T d_out, x>: the gradient against the pinned forward oracle."""
    c = synth.make_case(M, N, K, gs, scale_f16=f16, bias=False, seed=M + N + K)
    rng = np.random.default_rng(K)
    d_out = rng.standard_normal((M, N)).astype(np.float32)
    fwd, fwd_mag = oracle.linear(c.x, c.qweight, c.scales, None, K, gs)
    d_x, d_mag = oracle.backward_dx(d_out, c.qweight, c.scales, K, gs)
    lhs = np.sum(d_out.astype(np.float64) * fwd)
    rhs = np.sum(d_x * c.x.astype(np.float64))
    bound = 1e-12 * (np.sum(np.abs(d_out) * fwd_mag) + np.sum(np.abs(c.x) * d_mag))
    assert abs(lhs - rhs) <= bound + 1e-300


@pytest.mark.parametrize("M,N,K,gs,f16,eh", [(4, 50, 64, 32, False, False),
                                             (2, 33, 65, 8, True, False),
                                             (3, 20, 96, 96, False, True)])
def test_backward_brute_force_dense(M, N, K, gs, f16, eh):
    c = synth.make_case(1, N, K, gs, scale_f16=f16, bias=False, seed=N * K)
    d_out = np.random.default_rng(N).standard_normal((M, N)).astype(np.float32)
    w = dense_dequant(c.qweight, c.scales, K, gs, even_high=eh)
    ref = d_out.astype(np.float64) @ w
    mag_ref = np.abs(d_out.astype(np.float64)) @ np.abs(w)
    d_x, mag = oracle.backward_dx(d_out, c.qweight, c.scales, K, gs, even_high=eh)
    assert np.all(np.abs(d_x - ref) <= 1e-12 * mag_ref + 1e-300)
    np.testing.assert_allclose(mag, mag_ref, rtol=1e-12)


def test_backward_codes_eight_give_zero():
    c = synth.make_case(1, 40, 64, 32, scale_f16=True, bias=False, seed=1)
    q = synth.fill_codes(40, 64, 8)
    d_out = np.random.default_rng(1).standard_normal((3, 40)).astype(np.float32)
    d_x, _ = oracle.backward_dx(d_out, q, c.scales, 64, 32)
    assert np.all(d_x == 0.0)


# --------------------------------------------------------------------------- requant
@pytest.mark.parametrize("even_high", [False, True])
def test_requant_hand_example(even_high):
    r = load_requant_example()
    q = oracle.requant(r["latent"], r["scales"], r["group_size"], even_high=even_high)
    want = r["qweight"]
    if even_high:
        want = ((want & 0x0F) << 4) | (want >> 4)
    np.testing.assert_array_equal(q, want)


@pytest.mark.parametrize("N,K,gs,f16,eh", [(16, 64, 32, False, False), (9, 77, 8, True, False),
                                           (31, 130, 130, False, True), (5, 33, 1, True, False)])
def test_requant_inverts_dequant(N, K, gs, f16, eh):
    """Latents that are exact dequantized weights re-quantise to the same codes."""
    c = synth.make_case(1, N, K, gs, scale_f16=f16, bias=False, seed=N + K)
    latent = dense_dequant(c.qweight, c.scales, K, gs, even_high=eh).astype(np.float32)
    q = oracle.requant(latent, c.scales, gs, even_high=eh)
    if K % 2:  # the padding nibble is the bias-zero code 8
        pad = (0x80 if not eh else 0x08)
        expect = c.qweight.copy()
        expect[:, -1] = (expect[:, -1] & (0x0F if not eh else 0xF0)) | pad
    else:
        expect = c.qweight
    np.testing.assert_array_equal(q, expect)


def test_requant_error_within_half_step():
    """|dequant(requant(latent)) - latent| <= scale / 2 inside the representable range."""
    rng = np.random.default_rng(5)
    N, K, gs = 20, 96, 32
    scales = rng.uniform(0.01, 0.1, (K // gs, N)).astype(np.float32)
    s_per_k = np.repeat(scales, gs, axis=0).T.astype(np.float64)
    latent = (rng.uniform(-7.4, 6.4, (N, K)) * s_per_k).astype(np.float32)
    q = oracle.requant(latent, scales, gs)
    back = dense_dequant(q, scales, K, gs)
    assert np.all(np.abs(back - latent.astype(np.float64)) <= 0.5 * s_per_k * (1 + 1e-6))


def test_requant_zero_scale_and_clamp():
    N, K, gs = 3, 8, 8
    latent = np.array([[1e9, -1e9, 0.3, -0.3, 7.4, -8.4, np.inf, -np.inf]] * N, np.float32)
    scales = np.array([[1.0, 0.0, 1.0]], np.float32)
    q = oracle.requant(latent, scales, gs)
    codes = np.stack([q & 0x0F, q >> 4], axis=-1).reshape(N, K)
    np.testing.assert_array_equal(codes[0], [15, 0, 8, 8, 15, 0, 15, 0])
    np.testing.assert_array_equal(codes[1], [8] * 8)


# ----------------------------------------------------------------- planted mistakes
MUTANTS = {
    "backward: nibble of (k, n) instead of (n, k)": (
        "int q = nibble_at(qweight, row_bytes, n, k, even_high);\n            double w",
        "int q = nibble_at(qweight, row_bytes, k % N, n % K, even_high);\n            double w"),
    "backward: offset 7": ("double w = (double)(q - 8) * scale_at(scales, scale_is_f16, N, k / group_size, n);",
                           "double w = (double)(q - 7) * scale_at(scales, scale_is_f16, N, k / group_size, n);"),
    "backward: group index from n": (
        "scale_at(scales, scale_is_f16, N, k / group_size, n);\n            double p",
        "scale_at(scales, scale_is_f16, N, n / group_size % ((K + group_size - 1) / group_size), n);\n            double p"),
    "backward: last n dropped": ("for (int64_t n = 0; n < N; ++n) {\n            int q",
                                 "for (int64_t n = 0; n < N - 1; ++n) {\n            int q"),
    "requant: round half away from zero": ("double r = rint((double)quotient);",
                                           "double r = round((double)quotient);"),
    "requant: clamp to 8": ("if (r > 7.0) r = 7.0;", "if (r > 8.0) r = 8.0;"),
    "requant: zero scale gives code 0": ("if (s == 0.0) continue;",
                                         "if (s == 0.0) { codes[j] = 0; continue; }"),
    "requant: nibble order swapped": ("int low = even_high ? codes[1] : codes[0];",
                                      "int low = even_high ? codes[0] : codes[1];"),
    "requant: group index k % gs": ("double s = scale_at(scales, scale_is_f16, N, k / group_size, n);\n                if (s == 0.0)",
                                    "double s = scale_at(scales, scale_is_f16, N, k % group_size % ((K + group_size - 1) / group_size), n);\n                if (s == 0.0)"),
}


def _train_pins_pass(lib_path):
    import ctypes
    lib = ctypes.CDLL(lib_path)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.q4o_backward_dx.argtypes = [vp, vp, vp, i32, i64, i64, i64, i64, i32, vp, vp]
    lib.q4o_requant.argtypes = [vp, vp, i32, i64, i64, i64, i32, vp]
    p = lambda a: a.ctypes.data_as(vp)

    def bw(d_out, q, s, K, gs):
        M, N = d_out.shape
        d_x = np.empty((M, K)); mag = np.empty((M, K))
        lib.q4o_backward_dx(p(d_out), p(q), p(s), int(s.dtype == np.float16), M, N, K, gs, 0,
                            p(d_x), p(mag))
        return d_x

    def rq(latent, s, gs):
        N, K = latent.shape
        out = np.empty((N, (K + 1) // 2), np.uint8)
        lib.q4o_requant(p(latent), p(s), int(s.dtype == np.float16), N, K, gs, 0, p(out))
        return out

    ex = load_worked_example()
    if not np.array_equal(bw(ex["bw_d_out"], ex["qweight"], ex["scales"], 8, 4), ex["bw_d_x"]):
        return False
    c = synth.make_case(1, 37, 77, 8, scale_f16=False, bias=False, seed=4)
    d_out = np.random.default_rng(4).standard_normal((3, 37)).astype(np.float32)
    w = dense_dequant(c.qweight, c.scales, 77, 8)
    ref, mag = d_out.astype(np.float64) @ w, np.abs(d_out.astype(np.float64)) @ np.abs(w)
    if not np.all(np.abs(bw(d_out, c.qweight, c.scales, 77, 8) - ref) <= 1e-12 * mag + 1e-300):
        return False
    r = load_requant_example()
    if not np.array_equal(rq(r["latent"], r["scales"], 4), r["qweight"]):
        return False
    c = synth.make_case(1, 9, 64, 8, scale_f16=False, bias=False, seed=9)
    latent = dense_dequant(c.qweight, c.scales, 64, 8).astype(np.float32)
    return np.array_equal(rq(latent, c.scales, 8), c.qweight)


def test_train_pins_catch_planted_mistakes():
    src = open(os.path.join(os.path.dirname(oracle.__file__), "q4_oracle.c")).read()
    tmp = tempfile.mkdtemp(prefix="q4o_tmut_")
    try:
        def build(text, name):
            path = os.path.join(tmp, f"{name}.c")
            with open(path, "w") as f:
                f.write(text)
            lib = os.path.join(tmp, f"lib{name}.so")
            subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", path, "-o", lib, "-lm"],
                           check=True)
            return lib

        assert _train_pins_pass(build(src, "unmutated"))
        for i, (name, (old, new)) in enumerate(MUTANTS.items()):
            assert src.count(old) == 1, f"mutation site for '{name}' not unique"
            assert not _train_pins_pass(build(src.replace(old, new), f"m{i}")), \
                f"planted mistake not caught: {name}"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
