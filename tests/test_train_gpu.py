"""Parity of the training-path kernels (through the C ABI) with the fp64 CPU oracle:
the input gradient d_x = d_out @ dequant(W) (per element within 1e-5 * sum_n |d_out * w| +
1e-7; bit-exact on dyadic inputs) and the re-quantisation of fp32 latents (integer output:
bit-exact, including ties, zero scales, NaN / Inf latents and the odd-K padding nibble)."""
import numpy as np
import pytest

import oracle
from bit_weight_quantized_int4_gb300 import synth
from tests._golden import load_requant_example, load_worked_example
from tests._gpu import GUARD, SENTINEL, TOL_FP32, assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def handle():
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    assert torch.cuda.is_available()
    h = q.q4lin_create(0)
    yield h
    q.q4lin_destroy(h)


def run_backward(handle, c, even_high=False):
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    d_out, w, s = t(c.d_out), t(c.qweight), t(c.scales)
    buf = torch.full((c.M * c.K + GUARD,), float("nan"), dtype=torch.float32, device="cuda")
    buf[c.M * c.K:] = float(SENTINEL)
    q.q4lin_set_option(handle, q.Q4LIN_OPT_NIBBLE_EVEN_HIGH, int(even_high))
    sd = q.Q4LIN_SCALE_F16 if c.scale_f16 else q.Q4LIN_SCALE_F32
    st = q.q4lin_run_backward_dx(handle, d_out.data_ptr(), w.data_ptr(), s.data_ptr(),
                                 buf.data_ptr(), c.M, c.N, c.K, c.group_size, sd,
                                 torch.cuda.current_stream().cuda_stream)
    q.q4lin_set_option(handle, q.Q4LIN_OPT_NIBBLE_EVEN_HIGH, 0)
    assert st == q.Q4LIN_OK, q.q4lin_status_string(st)
    torch.cuda.synchronize()
    host = buf.cpu().numpy()
    assert np.all(host[c.M * c.K:] == SENTINEL), "write past the end of d_x"
    return host[:c.M * c.K].reshape(c.M, c.K)


def run_requant(handle, c, even_high=False):
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    Kp = (c.K + 1) // 2
    lat = torch.from_numpy(np.ascontiguousarray(c.latent)).cuda()
    s = torch.from_numpy(np.ascontiguousarray(c.scales)).cuda()
    buf = torch.full((c.N * Kp + GUARD,), 0xA5, dtype=torch.uint8, device="cuda")
    q.q4lin_set_option(handle, q.Q4LIN_OPT_NIBBLE_EVEN_HIGH, int(even_high))
    sd = q.Q4LIN_SCALE_F16 if c.scale_f16 else q.Q4LIN_SCALE_F32
    st = q.q4lin_run_requant(handle, lat.data_ptr(), s.data_ptr(), buf.data_ptr(), c.N, c.K,
                             c.group_size, sd, torch.cuda.current_stream().cuda_stream)
    q.q4lin_set_option(handle, q.Q4LIN_OPT_NIBBLE_EVEN_HIGH, 0)
    assert st == q.Q4LIN_OK, q.q4lin_status_string(st)
    torch.cuda.synchronize()
    host = buf.cpu().numpy()
    assert np.all(host[c.N * Kp:] == 0xA5), "write past the end of qweight"
    return host[:c.N * Kp].reshape(c.N, Kp)


# ----------------------------------------------------------------- input gradient d_x
BACKWARD_SHAPES = [
    # M, N, K, gs, f16
    (1, 2048, 2048, 32, True),      # decode-size row, rows split over CTAs
    (3, 515, 1000, 8, False),       # ragged k tile, ragged row splits
    (8, 64, 256, 64, True),         # one full tile of 8 d_out rows
    (13, 100, 96, 96, False),       # two d_out tiles, one group (per channel)
    (2, 37, 77, 7, True),           # generic kernel: odd K, group 7
    (5, 129, 4104, 8, False),       # K % 256 != 0 across many k tiles
    (1, 128256, 2048, 32, True),    # vocab-sized N: deep row split
]


@pytest.mark.parametrize("M,N,K,gs,f16", BACKWARD_SHAPES)
def test_backward_parity(handle, M, N, K, gs, f16):
    c = synth.make_backward_case(M, N, K, gs, scale_f16=f16, seed=M * 7 + K)
    out = run_backward(handle, c)
    ref, mag = oracle.backward_dx(c.d_out, c.qweight, c.scales, K, gs)
    assert_parity(out, ref, mag, TOL_FP32)


# Shapes taking the TMA-fed kernel (K % 32 == 0, N % 8 == 0, 16-byte aligned tensors, a
# group size that tiles 256 k or spans whole tiles): ragged k tiles and 64-row stages,
# partial d_out tiles, groups of 32..512 and per channel, both scale dtypes.
BACKWARD_TMA_SHAPES = [
    # M, N, K, gs, f16
    (3, 520, 1056, 32, False),     # K % 256 != 0, N % 64 != 0, MT = 4 with 3 rows
    (5, 1000, 2048, 128, True),    # MT = 8 with 5 rows
    (2, 4096, 4096, 512, True),    # a group spans two k tiles
    (9, 264, 768, 768, False),     # per channel, two d_out tiles
    (1, 8, 256, 256, False),       # one stage of 8 rows
    (4, 2048, 8192, 256, True),    # one group per k tile, rows split over CTAs
    (1, 8192, 2048, 64, False),    # deep row split, fp32 scales
    (8, 2048, 8192, 32, True),     # the benchmark's M = 8 shape
    (1, 8192, 2048, 32, True),     # the benchmark's M = 1 shape
    (1, 2048, 8192, 32, True),     # 16 consumer warps (1-2 rows of d_out, K >= 8192), cluster
    (2, 600, 9216, 64, False),     # 16 consumer warps, MT = 2, ragged N
    (1, 4096, 14336, 32, True),    # 16 consumer warps, rows split through the workspace
    (2, 4104, 1056, 32, False),    # 128-k tiles (two rows per warp pass), ragged K and N
    (1, 6000, 512, 256, True),     # 128-k tiles, a group spans two tiles
]


@pytest.mark.parametrize("M,N,K,gs,f16", BACKWARD_TMA_SHAPES)
def test_backward_tma_parity(handle, M, N, K, gs, f16):
    c = synth.make_backward_case(M, N, K, gs, scale_f16=f16, seed=M * 13 + N + K)
    out = run_backward(handle, c)
    ref, mag = oracle.backward_dx(c.d_out, c.qweight, c.scales, K, gs)
    assert_parity(out, ref, mag, TOL_FP32)


def test_backward_tma_nibble_even_high_and_repeat(handle):
    c = synth.make_backward_case(3, 256, 1024, 64, scale_f16=True, seed=6)
    ref, mag = oracle.backward_dx(c.d_out, c.qweight, c.scales, 1024, 64, even_high=True)
    out = run_backward(handle, c, even_high=True)
    assert_parity(out, ref, mag, TOL_FP32)
    np.testing.assert_array_equal(out, run_backward(handle, c, even_high=True))


@pytest.mark.parametrize("M,N,K,gs", [(4, 300, 512, 32), (9, 1000, 2048, 128), (1, 77, 40, 8),
                                      (1, 4096, 2048, 32), (2, 8192, 1024, 64)])
def test_backward_dyadic_bit_exact(handle, M, N, K, gs):
    c = synth.make_backward_case(M, N, K, gs, seed=N, dyadic=True)
    ref, _ = oracle.backward_dx(c.d_out, c.qweight, c.scales, K, gs)
    np.testing.assert_array_equal(run_backward(handle, c).astype(np.float64), ref)


def test_backward_worked_example(handle):
    ex = load_worked_example()
    c = synth.BackwardCase(2, 4, 8, 4, ex["bw_d_out"], ex["qweight"], ex["scales"])
    np.testing.assert_array_equal(run_backward(handle, c).astype(np.float64), ex["bw_d_x"])


def test_backward_nibble_even_high(handle):
    c = synth.make_backward_case(3, 250, 1024, 64, scale_f16=True, seed=5)
    ref, mag = oracle.backward_dx(c.d_out, c.qweight, c.scales, 1024, 64, even_high=True)
    assert_parity(run_backward(handle, c, even_high=True), ref, mag, TOL_FP32)


def test_backward_repeat_identical(handle):
    c = synth.make_backward_case(2, 4096, 2048, 32, seed=11)
    np.testing.assert_array_equal(run_backward(handle, c), run_backward(handle, c))


def test_backward_empty_rows_give_zeros(handle):
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    d_x = torch.full((3, 64), float("nan"), device="cuda")
    st = q.q4lin_run_backward_dx(handle, None, None, None, d_x.data_ptr(), 3, 0, 64, 32,
                                 q.Q4LIN_SCALE_F32, torch.cuda.current_stream().cuda_stream)
    assert st == q.Q4LIN_OK
    torch.cuda.synchronize()
    assert torch.all(d_x == 0).item()
    assert q.q4lin_run_backward_dx(handle, None, None, None, None, 0, 5, 64, 32,
                                   q.Q4LIN_SCALE_F32, 0) == q.Q4LIN_OK


def test_backward_rejects_overlap(handle):
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    c = synth.make_backward_case(2, 64, 64, 32, seed=1)
    buf = torch.zeros(4096, device="cuda")
    w = torch.from_numpy(c.qweight).cuda()
    s = torch.from_numpy(c.scales).cuda()
    st = q.q4lin_run_backward_dx(handle, buf.data_ptr(), w.data_ptr(), s.data_ptr(),
                                 buf.data_ptr() + 16, 2, 64, 64, 32, q.Q4LIN_SCALE_F32, 0)
    assert st == q.Q4LIN_ERR_INVALID_ARG


# --------------------------------------------------------------------------- requant
REQUANT_SHAPES = [
    # N, K, gs, f16
    (8192, 2048, 32, True),    # the benchmark's shape (16-k kernel)
    (40, 1040, 16, False),     # 16-k kernel, K % 32 == 16, groups of 16
    (64, 2048, 32, False),     # fast kernel
    (33, 4096, 4096, True),    # per channel, fp16 scales
    (100, 512, 64, False),
    (17, 77, 8, True),         # generic kernel: odd K (padding nibble 8)
    (5, 96, 24, False),        # group not a multiple of 32
]


@pytest.mark.parametrize("N,K,gs,f16", REQUANT_SHAPES)
@pytest.mark.parametrize("specials", [False, True])
def test_requant_bit_exact(handle, N, K, gs, f16, specials):
    c = synth.make_requant_case(N, K, gs, scale_f16=f16, seed=N + K, specials=specials)
    np.testing.assert_array_equal(run_requant(handle, c), oracle.requant(c.latent, c.scales, gs))


@pytest.mark.parametrize("f16", [False, True])
def test_requant_near_half_integers(handle, f16):
    """Latents whose fp32 quotients fall on, or within a few ulps of, half-integers (and
    of the clamp edges -8.5 / 7.5) under non-power-of-two scales: the rounding decision
    near a tie must be the one of the exact fp32 quotient."""
    rng = np.random.default_rng(17)
    N, K, gs = 64, 1024, 32
    s = rng.uniform(0.003, 0.05, size=(K // gs, N)).astype(np.float32)
    scales = s.astype(np.float16) if f16 else s
    s_used = np.repeat(scales.astype(np.float64), gs, axis=0).T  # [N, K]
    h = rng.integers(-9, 9, size=(N, K)) + 0.5
    ulps = rng.integers(-4, 5, size=(N, K))
    target = (h * s_used).astype(np.float32)
    latent = np.nextafter(target, np.where(ulps >= 0, np.inf, -np.inf).astype(np.float32))
    for _ in range(3):  # a few ulps either side, some exact
        step = np.abs(ulps) > 1
        latent = np.where(step, np.nextafter(latent, np.where(ulps >= 0, np.inf, -np.inf)
                                             .astype(np.float32)), latent)
        ulps = np.where(step, ulps - np.sign(ulps), ulps)
    latent = np.where(rng.random((N, K)) < 0.2, target, latent).astype(np.float32)
    c = synth.RequantCase(N, K, gs, latent, scales)
    np.testing.assert_array_equal(run_requant(handle, c), oracle.requant(latent, scales, gs))


def test_requant_hand_example(handle):
    r = load_requant_example()
    c = synth.RequantCase(2, 8, r["group_size"], r["latent"], r["scales"])
    np.testing.assert_array_equal(run_requant(handle, c), r["qweight"])


@pytest.mark.parametrize("K", [1024, 65])
def test_requant_nibble_even_high(handle, K):
    c = synth.make_requant_case(40, K, 32, seed=K, specials=True)
    np.testing.assert_array_equal(run_requant(handle, c, even_high=True),
                                  oracle.requant(c.latent, c.scales, 32, even_high=True))


def test_requant_then_forward_round_trip(handle):
    """Codes -> fp32 latents (the oracle's dequantized weights) -> requant on the GPU -> the
    same codes, and the forward of the requantized weight matches the original's."""
    from tests.test_oracle import dense_dequant
    case = synth.make_case(1, 256, 1024, 32, scale_f16=False, bias=False, seed=3)
    latent = dense_dequant(case.qweight, case.scales, 1024, 32).astype(np.float32)
    c = synth.RequantCase(256, 1024, 32, latent, case.scales)
    np.testing.assert_array_equal(run_requant(handle, c), case.qweight)
