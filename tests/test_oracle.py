"""Pins for the fp64 CPU oracle, against facts that do not come from the oracle itself.

- the hand-derived worked example (tests/golden/worked_example_2x4x8.txt);
- numpy's IEEE binary16 conversion for all 65536 bit patterns (the oracle decodes fp16
  scales with its own bit-field code);
- the identity "per-channel qcs4w == grouped q4gsw with group_size = K" between two
  separately written routines;
- brute force on tiny inputs: an explicitly dequantized dense fp64 weight, unpacked here
  with numpy bit operations, times x through numpy's matmul;
- exact invariants (all codes 8, scale doubling, row permutation, linearity in x, the
  odd-K padding nibble never read);
- planted mistakes: mutated copies of the oracle's C source must each fail a pin.
"""
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from bit_weight_quantized_int4_gb300 import synth
from tests._golden import load_worked_example


# ----------------------------------------------------------------------------- helpers
def dense_dequant(qweight, scales, K, group_size, even_high=False):
    """[N, K] float64 weights (q - 8) * scale, unpacked with numpy bit operations."""
    lo = (qweight & 0x0F).astype(np.int64)
    hi = (qweight >> 4).astype(np.int64)
    codes = np.empty((qweight.shape[0], 2 * qweight.shape[1]), np.int64)
    codes[:, 0::2], codes[:, 1::2] = (hi, lo) if even_high else (lo, hi)
    codes = codes[:, :K]
    s = scales.astype(np.float64)                        # [G, N]
    s_per_k = np.repeat(s, group_size, axis=0)[:K].T     # [N, K]
    return (codes - 8).astype(np.float64) * s_per_k


def brute_force(case, even_high=False):
    w = dense_dequant(case.qweight, case.scales, case.K, case.group_size, even_high)
    out = case.x.astype(np.float64) @ w.T
    if case.bias is not None:
        out = out + case.bias.astype(np.float64)
    mag = np.abs(case.x.astype(np.float64)) @ np.abs(w).T
    return out, mag


# ------------------------------------------------------------------------ worked example
@pytest.mark.parametrize("scale_dtype", [np.float32, np.float16])
def test_worked_example(scale_dtype):
    ex = load_worked_example()
    scales = ex["scales"].astype(scale_dtype)
    out, mag = oracle.linear(ex["x"], ex["qweight"], scales, None, ex["K"], ex["group_size"])
    np.testing.assert_array_equal(out, ex["out_nobias"])
    np.testing.assert_array_equal(mag, ex["mag"])
    out_b, mag_b = oracle.linear(ex["x"], ex["qweight"], scales, ex["bias"], ex["K"],
                                 ex["group_size"])
    np.testing.assert_array_equal(out_b, ex["out_bias"])
    np.testing.assert_array_equal(mag_b, ex["mag"])  # bias is not in the denominator


def test_worked_example_nibble_order_matters():
    ex = load_worked_example()
    out, _ = oracle.linear(ex["x"], ex["qweight"], ex["scales"], None, ex["K"],
                           ex["group_size"], even_high=True)
    np.testing.assert_array_equal(out, ex["out_swapped_nobias"])
    assert not np.array_equal(ex["out_swapped_nobias"], ex["out_nobias"])


@pytest.mark.parametrize("scale_dtype", [np.float32, np.float16])
def test_worked_example_per_channel(scale_dtype):
    ex = load_worked_example()
    s = ex["scales_per_channel"].astype(scale_dtype)
    out_g, _ = oracle.linear(ex["x"], ex["qweight"], s[None, :], None, ex["K"], ex["K"])
    out_c, _ = oracle.linear_qcs4w(ex["x"], ex["qweight"], s, None, ex["K"])
    np.testing.assert_array_equal(out_g, ex["out_per_channel_nobias"])
    np.testing.assert_array_equal(out_c, ex["out_per_channel_nobias"])


# ---------------------------------------------------------------------------- fp16 decode
def test_f16_decode_all_bit_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(b)) for b in bits])
    nan = np.isnan(want)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


# ------------------------------------------------------------------------------ identity
@pytest.mark.parametrize("K", [64, 255, 1000])
@pytest.mark.parametrize("f16", [False, True])
def test_identity_qcs4w_equals_grouped_gs_K(K, f16):
    c = synth.make_case(M=3, N=37, K=K, group_size=K, scale_f16=f16, bias=True, seed=K)
    out_g, mag_g = oracle.linear(c.x, c.qweight, c.scales, c.bias, K, K)
    out_c, mag_c = oracle.linear_qcs4w(c.x, c.qweight, c.scales[0], c.bias, K)
    # Two different summation orders in double: agreement up to double rounding.
    assert np.all(np.abs(out_g - out_c) <= 1e-12 * mag_g + 1e-300)
    assert np.allclose(mag_g, mag_c, rtol=1e-12, atol=0)


# ---------------------------------------------------------------------------- brute force
BRUTE_CASES = [
    # (M, N, K, group_size, f16, bias)
    (1, 16, 64, 32, False, False),
    (4, 64, 256, 32, False, True),
    (3, 33, 96, 8, True, True),
    (2, 17, 128, 64, True, False),
    (5, 9, 80, 80, False, True),     # group_size = K
    (2, 11, 75, 75, True, True),     # odd K, per-channel
    (3, 13, 77, 8, False, False),    # odd K, partial last group
    (2, 7, 10, 4, False, True),      # K not a multiple of group_size
    (8, 64, 250, 1, True, False),    # group_size 1
    (1, 5, 1, 1, False, True),       # K = 1
]


@pytest.mark.parametrize("M,N,K,gs,f16,bias", BRUTE_CASES)
def test_brute_force_dense_fp64(M, N, K, gs, f16, bias):
    c = synth.make_case(M, N, K, gs, scale_f16=f16, bias=bias, seed=M * 1000 + K)
    out, mag = oracle.linear(c.x, c.qweight, c.scales, c.bias, K, gs)
    ref, ref_mag = brute_force(c)
    assert np.all(np.abs(out - ref) <= 1e-12 * ref_mag + 1e-300)
    assert np.allclose(mag, ref_mag, rtol=1e-12, atol=0)


def test_brute_force_swapped_order():
    c = synth.make_case(3, 20, 64, 16, bias=True, seed=5)
    out, _ = oracle.linear(c.x, c.qweight, c.scales, c.bias, 64, 16, even_high=True)
    ref, ref_mag = brute_force(c, even_high=True)
    assert np.all(np.abs(out - ref) <= 1e-12 * ref_mag)


# ----------------------------------------------------------------------------- invariants
def test_all_codes_eight_gives_bias_exactly():
    c = synth.make_case(3, 40, 130, 32, bias=True, seed=11)
    q8 = synth.fill_codes(40, 130, 8)
    out, mag = oracle.linear(c.x, q8, c.scales, c.bias, 130, 32)
    np.testing.assert_array_equal(out, np.broadcast_to(c.bias.astype(np.float64), out.shape))
    np.testing.assert_array_equal(mag, 0.0)


def test_scale_doubling_is_exact():
    c = synth.make_case(2, 24, 96, 32, bias=False, seed=12)
    out1, _ = oracle.linear(c.x, c.qweight, c.scales, None, 96, 32)
    out2, _ = oracle.linear(c.x, c.qweight, c.scales * np.float32(2), None, 96, 32)
    np.testing.assert_array_equal(out2, 2.0 * out1)  # power-of-two scaling is exact


def test_row_permutation_permutes_output():
    c = synth.make_case(2, 31, 64, 16, scale_f16=True, bias=True, seed=13)
    perm = np.random.Generator(np.random.PCG64(99)).permutation(31)
    out, _ = oracle.linear(c.x, c.qweight, c.scales, c.bias, 64, 16)
    outp, _ = oracle.linear(c.x, c.qweight[perm], c.scales[:, perm], c.bias[perm], 64, 16)
    np.testing.assert_array_equal(outp, out[:, perm])


def test_linear_in_x():
    a = synth.make_dyadic_case(2, 19, 48, 16, seed=14)
    b = synth.make_dyadic_case(2, 19, 48, 16, seed=15)
    o1, m1 = oracle.linear(a.x, a.qweight, a.scales, None, 48, 16)
    o2, m2 = oracle.linear(b.x, a.qweight, a.scales, None, 48, 16)
    o12, _ = oracle.linear(a.x + b.x, a.qweight, a.scales, None, 48, 16)
    o3, _ = oracle.linear(np.float32(2) * a.x, a.qweight, a.scales, None, 48, 16)
    np.testing.assert_array_equal(o12, o1 + o2)   # dyadic inputs: all exact
    np.testing.assert_array_equal(o3, 2.0 * o1)


def test_odd_k_padding_nibble_is_not_read():
    c = synth.make_case(2, 12, 33, 8, bias=False, seed=16)
    q = c.qweight.copy()
    q[:, -1] ^= 0xF0  # flip only the padding (high) nibble of the last byte
    o1, _ = oracle.linear(c.x, c.qweight, c.scales, None, 33, 8)
    o2, _ = oracle.linear(c.x, q, c.scales, None, 33, 8)
    np.testing.assert_array_equal(o1, o2)


def test_sampled_elements_match_full():
    c = synth.make_case(5, 70, 100, 20, scale_f16=True, bias=True, seed=17)
    out, mag = oracle.linear(c.x, c.qweight, c.scales, c.bias, 100, 20)
    ms = np.array([0, 4, 2, 3, 4])
    ns = np.array([0, 69, 33, 1, 0])
    o, m = oracle.linear_at(c.x, c.qweight, c.scales, c.bias, 100, 20, ms, ns)
    np.testing.assert_array_equal(o, out[ms, ns])
    np.testing.assert_array_equal(m, mag[ms, ns])


def test_rejects_bad_arguments():
    c = synth.make_case(1, 4, 8, 4, seed=18)
    with pytest.raises(ValueError):
        oracle.linear(c.x, c.qweight, c.scales, None, 8, 3)  # scales shape wrong for gs=3
    with pytest.raises(ValueError):
        oracle.linear_at(c.x, c.qweight, c.scales, None, 8, 4, [1], [0])  # m out of range


# ------------------------------------------------------------------------ planted mistakes
MUTANTS = {
    "nibble order swapped": ("int take_low = even_high ? !k_is_even : k_is_even;",
                             "int take_low = even_high ? k_is_even : !k_is_even;"),
    "offset 7 instead of 8": ("double w = (double)(q - 8) * s;",
                              "double w = (double)(q - 7) * s;"),
    "group index k % gs": ("double s = scale_at(scales, scale_is_f16, N, k / group_size, n);\n        double w",
                           "double s = scale_at(scales, scale_is_f16, N, k % group_size, n);\n        double w"),
    # the worked example has G = 2 fp32 groups, so [n * 2 + g] reads scales as [N, G]
    "scale matrix transposed": ("((const float*)scales)[g * N + n]",
                                "((const float*)scales)[n * 2 + g]"),
    "bias dropped": ("out[i] = acc + (bias ? (double)bias[n] : 0.0);", "out[i] = acc;"),
    "last term dropped": ("for (int64_t k = 0; k < K; ++k) {\n        int q",
                          "for (int64_t k = 0; k < K - 1; ++k) {\n        int q"),
    "row stride floor(K/2)": ("int64_t row_bytes = (K + 1) / 2;\n    double acc",
                              "int64_t row_bytes = K / 2;\n    double acc"),
    "f16 exponent bias off by one": ("exponent - 25", "exponent - 24"),
}


def _build_mutant(src_text, tmpdir, name):
    path = os.path.join(tmpdir, f"{name}.c")
    with open(path, "w") as f:
        f.write(src_text)
    lib = os.path.join(tmpdir, f"lib{name}.so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", path, "-o", lib, "-lm"],
                   check=True)
    return lib


def _pins_pass(lib_path):
    """Run the worked example, a brute-force case and the fp16 decode on a mutant."""
    import ctypes
    lib = ctypes.CDLL(lib_path)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.q4o_linear.argtypes = [vp, vp, vp, i32, vp, i64, i64, i64, i64, i32, vp, vp]
    lib.q4o_f16_to_f64.argtypes = [ctypes.c_uint16]
    lib.q4o_f16_to_f64.restype = ctypes.c_double

    def run(x, q, s, b, K, gs):
        M, N = x.shape[0], q.shape[0]
        out = np.empty((M, N)); mag = np.empty((M, N))
        p = lambda a: None if a is None else a.ctypes.data_as(vp)
        lib.q4o_linear(p(x), p(q), p(s), int(s.dtype == np.float16), p(b), M, N, K, gs, 0,
                       p(out), p(mag))
        return out, mag

    ex = load_worked_example()
    out, _ = run(ex["x"], ex["qweight"], ex["scales"], ex["bias"], ex["K"], ex["group_size"])
    if not np.array_equal(out, ex["out_bias"]):
        return False
    c = synth.make_case(3, 13, 77, 8, scale_f16=True, bias=True, seed=3)
    out, _ = run(c.x, c.qweight, c.scales, c.bias, 77, 8)
    ref, ref_mag = brute_force(c)
    if not np.all(np.abs(out - ref) <= 1e-12 * ref_mag + 1e-300):
        return False
    for b in (0x3C00, 0x0001, 0x7BFF, 0xC000):
        if lib.q4o_f16_to_f64(b) != float(np.array([b], np.uint16).view(np.float16)[0]):
            return False
    return True


def test_pins_catch_planted_mistakes():
    src = open(os.path.join(os.path.dirname(oracle.__file__), "q4_oracle.c")).read()
    tmp = tempfile.mkdtemp(prefix="q4o_mut_")
    try:
        assert _pins_pass(_build_mutant(src, tmp, "unmutated"))
        for i, (name, (old, new)) in enumerate(MUTANTS.items()):
            assert src.count(old) == 1, f"mutation site for '{name}' not unique"
            lib = _build_mutant(src.replace(old, new), tmp, f"m{i}")
            assert not _pins_pass(lib), f"planted mistake not caught: {name}"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
