"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle.

Every case is seeded and synthetic (bit_weight_quantized_int4_gb300.synth).  The output
is NaN-poisoned with 64 guard slots after it; the tolerance per element is
1e-5 * sum_k|x*w| + 1e-7 on the CUDA-core paths and 4e-3 * sum_k|x*w| + 1e-6 on the
tensor-core path.  Dyadic inputs and all-8 codes must come out bit-exact on every path.
"""
import numpy as np
import pytest

import oracle
from bit_weight_quantized_int4_gb300 import synth
from tests._golden import load_worked_example
from tests._gpu import TOL_FP32, TOL_TC, assert_parity, run_q4lin

pytestmark = pytest.mark.gpu

GEMV, FFMA, TC, AUTO = 1, 2, 3, 0
TC_SMALL = 4


@pytest.fixture(scope="module")
def handle():
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    assert torch.cuda.is_available()
    h = q.q4lin_create(0)
    yield h
    q.q4lin_destroy(h)


def tol_for(path):
    return TOL_TC if path in (TC, TC_SMALL) else TOL_FP32


def check_case(handle, case, path=AUTO, even_high=False):
    """Every element of out[M,N] against the oracle (full rows and columns: the oracle
    finishes the largest configs, 2048 x 8192 x 2048, in seconds on the host cores)."""
    out, used = run_q4lin(handle, case, path, even_high)
    ref, mag = oracle.linear(case.x, case.qweight, case.scales, case.bias, case.K,
                             case.group_size, even_high=even_high)
    assert_parity(out, ref, mag, tol_for(used))
    return out, used


# ------------------------------------------------------------------------ worked example
@pytest.mark.parametrize("path", [AUTO, FFMA])
@pytest.mark.parametrize("f16", [False, True])
def test_worked_example_exact(handle, path, f16):
    ex = load_worked_example()
    scales = ex["scales"].astype(np.float16 if f16 else np.float32)
    c = synth.Case(2, 4, 8, 4, ex["x"], ex["qweight"], scales, ex["bias"])
    out, _ = run_q4lin(handle, c, path)
    np.testing.assert_array_equal(out.astype(np.float64), ex["out_bias"])


# ---------------------------------------------------------------------------- tiny config
@pytest.mark.parametrize("path", [AUTO, GEMV, FFMA])
def test_tiny_config(handle, path):
    c = synth.make_case(4, 128, 256, 32, scale_f16=False, bias=False, seed=0)
    check_case(handle, c, path)


# ----------------------------------------------------------------------- decode shapes
DECODE_1B = [(2048, 2048), (512, 2048), (8192, 2048), (2048, 8192), (128256, 2048)]
DECODE_8B = [(4096, 4096), (1024, 4096), (14336, 4096), (4096, 14336), (22016, 4096),
             (128256, 4096)]


@pytest.mark.parametrize("N,K", DECODE_1B + DECODE_8B)
def test_decode_gemv_shapes(handle, N, K):
    c = synth.make_case(1, N, K, 32, scale_f16=True, bias=False, seed=1 + N % 97 + K)
    _, used = check_case(handle, c, AUTO)
    assert used == GEMV


# ------------------------------------------------------------------------ qcs4w edges
@pytest.mark.parametrize("M", [1, 7, 64])
def test_qcs4w_vocab_ragged(handle, M):
    c = synth.make_case(M, 128257, 4096, 4096, scale_f16=False, bias=False, seed=4)
    check_case(handle, c, AUTO)


@pytest.mark.parametrize("M", [1, 33])
def test_qcs4w_k2056(handle, M):
    c = synth.make_case(M, 1000, 2056, 2056, scale_f16=False, bias=False, seed=4)
    check_case(handle, c, AUTO)


def test_qcs4w_fp16_scales(handle):
    c = synth.make_case(3, 4097, 1024, 1024, scale_f16=True, bias=True, seed=41)
    check_case(handle, c, AUTO)


# --------------------------------------------------------------------- small M / ragged
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 7, 8, 9, 16])
@pytest.mark.parametrize("path", [GEMV, FFMA])
def test_small_m(handle, M, path):
    c = synth.make_case(M, 300, 512, 32, scale_f16=True, bias=True, seed=M)
    check_case(handle, c, path)


@pytest.mark.parametrize("N", [1, 7, 15, 17, 33, 127, 129, 1000, 4097])
def test_ragged_n_gemv(handle, N):
    c = synth.make_case(1, N, 1024, 32, scale_f16=True, bias=True, seed=N)
    check_case(handle, c, GEMV)


@pytest.mark.parametrize("gs", [32, 64, 128, 96, 4096, 100000])
def test_group_sizes_gemv(handle, gs):
    K = 4096 if gs != 96 else 1056
    G = -(-K // gs)
    c = synth.make_case(2, 257, K, gs, scale_f16=False, bias=True, seed=gs)
    assert c.scales.shape == (G, 257)
    check_case(handle, c, GEMV)


@pytest.mark.parametrize("K,gs", [(77, 8), (33, 33), (250, 1), (1000, 24), (2056, 8),
                                  (96, 64), (1, 1)])
def test_generic_shapes(handle, K, gs):
    c = synth.make_case(3, 45, K, gs, scale_f16=K % 2 == 0, bias=True, seed=K)
    _, used = check_case(handle, c, AUTO)
    if K % 32:
        assert used == FFMA


# --------------------------------------------------------------------------- options
@pytest.mark.parametrize("path", [GEMV, FFMA])
def test_nibble_even_high(handle, path):
    c = synth.make_case(3, 130, 512, 64, scale_f16=True, bias=True, seed=21)
    check_case(handle, c, path, even_high=True)


# ------------------------------------------------------------------------ exactness
@pytest.mark.parametrize("path", [GEMV, FFMA, AUTO])
@pytest.mark.parametrize("M", [1, 3, 6])
def test_dyadic_bit_exact(handle, path, M):
    c = synth.make_dyadic_case(M, 200, 1024, 32, scale_f16=(M % 2 == 1), bias=True, seed=M)
    out, _ = run_q4lin(handle, c, path)
    ref, _ = oracle.linear(c.x, c.qweight, c.scales, c.bias, c.K, c.group_size)
    np.testing.assert_array_equal(out.astype(np.float64), ref)


@pytest.mark.parametrize("path", [GEMV, FFMA, AUTO])
def test_all_codes_eight_gives_bias(handle, path):
    c = synth.make_case(2, 333, 2048, 32, scale_f16=True, bias=True, seed=9)
    c.qweight = synth.fill_codes(333, 2048, 8)
    out, _ = run_q4lin(handle, c, path)
    np.testing.assert_array_equal(out, np.broadcast_to(c.bias, out.shape))


def test_repeat_calls_identical(handle):
    c = synth.make_case(1, 5000, 2048, 32, scale_f16=True, bias=True, seed=31)
    a, _ = run_q4lin(handle, c, AUTO)
    b, _ = run_q4lin(handle, c, AUTO)
    np.testing.assert_array_equal(a, b)


# ------------------------------------------------------------------- host-side checks
def test_empty_problems_launch_nothing(handle):
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    out = torch.full((16,), 7.0, device="cuda")
    x = torch.zeros(64, device="cuda")
    w = torch.zeros(64, dtype=torch.uint8, device="cuda")
    s = torch.zeros(64, device="cuda")
    for M, N in [(0, 4), (4, 0), (0, 0)]:
        st = q.q4lin_run(handle, x.data_ptr(), w.data_ptr(), s.data_ptr(), None,
                         out.data_ptr(), M, N, 32, 32, 0, None)
        assert st == q.Q4LIN_OK
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)


def test_invalid_arguments(handle):
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    x = torch.zeros(4 * 64, device="cuda")
    w = torch.zeros(8 * 32, dtype=torch.uint8, device="cuda")
    s = torch.zeros(2 * 8, device="cuda")
    out = torch.zeros(4 * 8, device="cuda")
    P = lambda t: t.data_ptr()
    run = lambda *a: q.q4lin_run(handle, *a)
    ok = (P(x), P(w), P(s), None, P(out), 4, 8, 64, 32, 0, None)
    assert run(*ok) == q.Q4LIN_OK
    bad = [
        (P(x), P(w), P(s), None, P(out), 4, 8, 0, 32, 0, None),        # K == 0
        (P(x), P(w), P(s), None, P(out), -1, 8, 64, 32, 0, None),      # M < 0
        (P(x), P(w), P(s), None, P(out), 4, 8, 64, 0, 0, None),        # group_size 0
        (P(x), P(w), P(s), None, P(out), 4, 8, 64, 32, 2, None),       # scale dtype
        (None, P(w), P(s), None, P(out), 4, 8, 64, 32, 0, None),       # NULL x
        (P(x), P(w), P(s), None, P(x), 4, 8, 64, 32, 0, None),         # out aliases x
        (P(x), P(w), P(s), None, P(out) + 2, 4, 8, 64, 32, 0, None),   # misaligned out
        (P(x), P(w), P(s) + 2, None, P(out), 4, 8, 64, 32, 0, None),   # misaligned f32 scales
    ]
    for args in bad:
        assert run(*args) == q.Q4LIN_ERR_INVALID_ARG, args
    assert q.q4lin_set_option(handle, q.Q4LIN_OPT_FORCE_PATH, 9) == q.Q4LIN_ERR_INVALID_ARG
    assert q.q4lin_set_option(handle, 77, 0) == q.Q4LIN_ERR_INVALID_ARG


def test_unaligned_x_falls_back(handle):
    """x that is 4- but not 16-byte aligned: GEMV is ineligible, AUTO still correct."""
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    c = synth.make_case(2, 100, 256, 32, scale_f16=True, bias=False, seed=5)
    big = torch.zeros(2 * 256 + 1, device="cuda")
    big[1:] = torch.from_numpy(c.x.ravel()).cuda()
    x_view = big[1:]
    out, used = run_q4lin(handle, c, AUTO, x_dev=x_view)
    assert used == FFMA
    ref, mag = oracle.linear(c.x, c.qweight, c.scales, None, 256, 32)
    assert_parity(out, ref, mag, TOL_FP32)
    q.q4lin_set_option(handle, q.Q4LIN_OPT_FORCE_PATH, GEMV)
    w = torch.from_numpy(c.qweight).cuda()
    s = torch.from_numpy(c.scales).cuda()
    o = torch.empty(200, device="cuda")
    st = q.q4lin_run(handle, x_view.data_ptr(), w.data_ptr(), s.data_ptr(), None,
                     o.data_ptr(), 2, 100, 256, 32, 1, None)
    q.q4lin_set_option(handle, q.Q4LIN_OPT_FORCE_PATH, AUTO)
    assert st == q.Q4LIN_ERR_UNSUPPORTED


def test_side_stream(handle):
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    c = synth.make_case(1, 2048, 2048, 32, scale_f16=True, bias=True, seed=6)
    x, w, s, b = (torch.from_numpy(a).cuda() for a in (c.x, c.qweight, c.scales, c.bias))
    out = torch.full((1, 2048), float("nan"), device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    st = q.q4lin_run(handle, x.data_ptr(), w.data_ptr(), s.data_ptr(), b.data_ptr(),
                     out.data_ptr(), 1, 2048, 2048, 32, 1, side.cuda_stream)
    assert st == q.Q4LIN_OK
    side.synchronize()
    ref, mag = oracle.linear(c.x, c.qweight, c.scales, c.bias, 2048, 32)
    assert_parity(out.cpu().numpy(), ref, mag, TOL_FP32)


# -------------------------------------------------------------------- prefill shapes
PREFILL_NK = [(2048, 2048), (512, 2048), (8192, 2048), (2048, 8192)]


@pytest.mark.parametrize("M", [128, 512, 2048])
@pytest.mark.parametrize("N,K", PREFILL_NK)
def test_prefill_shapes(handle, M, N, K):
    c = synth.make_case(M, N, K, 32, scale_f16=False, bias=(N != 512), seed=3)
    _, used = check_case(handle, c, AUTO)
    assert used == TC


@pytest.mark.parametrize("M,K,N,gs", [(96, 2048, 256, 32), (70, 1024, 136, 32),
                                      (96, 2048, 256, 64), (96, 2048, 256, 8),
                                      (128, 8192, 2048, 32)])
def test_extra_page_shapes(handle, M, K, N, gs):
    c = synth.make_case(M, N, K, gs, scale_f16=False, bias=True, seed=12)
    check_case(handle, c, AUTO)


# ------------------------------------------------------------------- tensor-core path
TC_SHAPES = [
    # (M, N, K, gs, f16, bias)
    (4, 128, 256, 32, False, False),      # the tiny config
    (1, 300, 512, 32, True, True),        # M = 1 through the tensor cores (bm = 16)
    (17, 129, 96, 32, False, True),       # 3 k-stages (< pipeline depth), ragged M and N
    (70, 136, 1024, 32, False, True),     # the pages' partial-M / partial-N edge shape
    (96, 256, 2048, 64, True, False),
    (256, 384, 512, 128, False, True),
    (257, 200, 1024, 32, False, True),    # two M tiles
    (600, 1000, 768, 32, True, True),     # three M tiles, ragged everything
    (33, 1000, 4096, 4096, False, False), # per-channel
    (64, 128257, 4096, 4096, False, False),
    (40, 200, 320, 32, True, True),       # 5 stages: two MMA issuers with unequal shares
    (100, 520, 1120, 32, False, True),    # 17.5 stages (odd, last one half), two issuers
    (300, 1000, 736, 32, True, False),    # 11.5 stages on 128-row tiles
]


@pytest.mark.parametrize("M,N,K,gs,f16,bias", TC_SHAPES)
def test_tc_parity(handle, M, N, K, gs, f16, bias):
    c = synth.make_case(M, N, K, gs, scale_f16=f16, bias=bias, seed=M + N)
    _, used = check_case(handle, c, TC)
    assert used == TC


@pytest.mark.parametrize("M,N,K,gs,f16,bias", [
    (128, 2048, 2048, 32, False, True),   # 16 tiles of 128 rows: K split over 8-CTA clusters
    (64, 256, 8192, 128, True, False),    # one 256-row tile: 8-way split of long K
    (200, 520, 1024, 1024, False, True),  # per-channel scales applied after the exchange
    (9, 96, 512, 32, True, True),         # 16 stages over 4 CTAs, ragged N inside the slices
    (64, 1024, 4096, 128, True, True),    # 64-row tiles, two issuers, K split over 4 CTAs
])
def test_tc_split_k_parity_and_determinism(handle, M, N, K, gs, f16, bias):
    """Few output tiles: the K range is split over the CTAs of a cluster, whose partial
    tiles are added in rank order in distributed shared memory.  Parity with the oracle,
    and bitwise-identical results on a second call."""
    c = synth.make_case(M, N, K, gs, scale_f16=f16, bias=bias, seed=N + K)
    out1, used = check_case(handle, c, TC)
    assert used == TC
    out2, _ = run_q4lin(handle, c, TC)
    np.testing.assert_array_equal(out1, out2)


@pytest.mark.parametrize("M", [1, 5, 48, 300])
def test_tc_dyadic_bit_exact(handle, M):
    c = synth.make_dyadic_case(M, 260, 1024, 32, scale_f16=(M % 2 == 1), bias=True, seed=M)
    out, used = run_q4lin(handle, c, TC)
    assert used == TC
    ref, _ = oracle.linear(c.x, c.qweight, c.scales, c.bias, c.K, c.group_size)
    np.testing.assert_array_equal(out.astype(np.float64), ref)


def test_tc_all_codes_eight_gives_bias(handle):
    c = synth.make_case(40, 333, 2048, 32, scale_f16=True, bias=True, seed=9)
    c.qweight = synth.fill_codes(333, 2048, 8)
    out, _ = run_q4lin(handle, c, TC)
    np.testing.assert_array_equal(out, np.broadcast_to(c.bias, out.shape))


def test_tc_nibble_even_high(handle):
    c = synth.make_case(20, 130, 512, 64, scale_f16=True, bias=True, seed=21)
    check_case(handle, c, TC, even_high=True)


def test_tc_bounded_wait_times_out_cleanly(handle):
    """The producer skips its first copy (test hook), so the barrier the consumers wait
    on is never completed: their 1 ms bounded waits run out, the kernel records code 1
    and returns; the context stays usable and the next call is correct."""
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    c = synth.make_case(8, 256, 512, 32, scale_f16=False, bias=False, seed=77)
    st, code = q.q4lin_check_device_status(handle, None)
    assert (st, code) == (q.Q4LIN_OK, 0)
    q.q4lin_set_option(handle, q.Q4LIN_OPT_WAIT_LIMIT, 1_000_000)
    q.q4lin_set_option(handle, q.Q4LIN_OPT_TC_SKIP_FIRST_COPY, 1)
    try:
        run_q4lin(handle, c, TC)
    except AssertionError:
        pass  # the output of a timed-out call is undefined (NaN-poisoned here)
    finally:
        q.q4lin_set_option(handle, q.Q4LIN_OPT_TC_SKIP_FIRST_COPY, 0)
        q.q4lin_set_option(handle, q.Q4LIN_OPT_WAIT_LIMIT, 0)
    st, code = q.q4lin_check_device_status(handle, None)
    assert st == q.Q4LIN_ERR_TIMEOUT and code == 1
    st, code = q.q4lin_check_device_status(handle, None)
    assert (st, code) == (q.Q4LIN_OK, 0)
    torch.cuda.synchronize()
    check_case(handle, c, TC)


# ----------------------------------------------------- programmatic dependent launch
@pytest.mark.parametrize("pdl", [0, 1])
def test_dependent_chain(handle, pdl):
    """GEMVs chained on one stream, each reading the previous output as its x, with every
    buffer NaN-poisoned first.  With programmatic dependent launch a kernel starts
    streaming weights early but must read x only after its predecessor completed; each
    link is checked against the oracle applied to the input it actually received."""
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    dims = [2048, 4096, 1024, 2048, 8192, 2048]
    links = []
    for i in range(len(dims) - 1):
        K, N = dims[i], dims[i + 1]
        c = synth.make_case(1, N, K, 32, scale_f16=True, bias=(i % 2 == 0), seed=900 + i)
        links.append(c)
    bufs = [torch.from_numpy(links[0].x.ravel()).cuda()]
    bufs += [torch.full((d,), float("nan"), device="cuda") for d in dims[1:]]
    dev = [tuple(None if a is None else torch.from_numpy(a).cuda()
                 for a in (c.qweight, c.scales, c.bias)) for c in links]
    torch.cuda.synchronize()
    q.q4lin_set_option(handle, q.Q4LIN_OPT_PDL, pdl)
    try:
        stream = torch.cuda.current_stream().cuda_stream
        for i, c in enumerate(links):
            w, s, b = dev[i]
            st = q.q4lin_run(handle, bufs[i].data_ptr(), w.data_ptr(), s.data_ptr(),
                             None if b is None else b.data_ptr(), bufs[i + 1].data_ptr(),
                             1, c.N, c.K, 32, q.Q4LIN_SCALE_F16, stream)
            assert st == q.Q4LIN_OK
        torch.cuda.synchronize()
    finally:
        q.q4lin_set_option(handle, q.Q4LIN_OPT_PDL, 0)
    host = [b.cpu().numpy() for b in bufs]
    for i, c in enumerate(links):
        assert not np.isnan(host[i + 1]).any(), f"link {i} output has NaN"
        ref, mag = oracle.linear(host[i][None, :], c.qweight, c.scales, c.bias, c.K, 32)
        assert_parity(host[i + 1][None, :], ref, mag, TOL_FP32)


@pytest.mark.parametrize("pdl", [0, 1])
@pytest.mark.parametrize("M", [96, 300])
def test_tc_dependent_chain(handle, pdl, M):
    """Tensor-core GEMMs chained on one stream, each reading the previous output as its x,
    every buffer NaN-poisoned first.  With programmatic dependent launch the kernel
    streams packed weights before the dependency wait but loads x, reads the bias and
    writes out only after it; each link is checked against the oracle applied to the
    input it actually received.  M = 300 takes several activation tiles, M = 96 few
    tiles with K split over clusters (workspace exchange)."""
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    dims = [512, 1024, 256, 768, 2048]
    links = []
    for i in range(len(dims) - 1):
        K, N = dims[i], dims[i + 1]
        links.append(synth.make_case(M, N, K, 32, scale_f16=(i % 2 == 1), bias=(i % 2 == 0),
                                     seed=700 + i + M))
    bufs = [torch.from_numpy(np.ascontiguousarray(links[0].x)).cuda()]
    bufs += [torch.full((M, d), float("nan"), device="cuda") for d in dims[1:]]
    dev = [tuple(None if a is None else torch.from_numpy(a).cuda()
                 for a in (c.qweight, c.scales, c.bias)) for c in links]
    torch.cuda.synchronize()
    q.q4lin_set_option(handle, q.Q4LIN_OPT_PDL, pdl)
    q.q4lin_set_option(handle, q.Q4LIN_OPT_FORCE_PATH, TC)
    try:
        stream = torch.cuda.current_stream().cuda_stream
        for i, c in enumerate(links):
            w, s, b = dev[i]
            sd = q.Q4LIN_SCALE_F16 if c.scales.dtype == np.float16 else q.Q4LIN_SCALE_F32
            st = q.q4lin_run(handle, bufs[i].data_ptr(), w.data_ptr(), s.data_ptr(),
                             None if b is None else b.data_ptr(), bufs[i + 1].data_ptr(),
                             M, c.N, c.K, 32, sd, stream)
            assert st == q.Q4LIN_OK
        torch.cuda.synchronize()
    finally:
        q.q4lin_set_option(handle, q.Q4LIN_OPT_PDL, 0)
        q.q4lin_set_option(handle, q.Q4LIN_OPT_FORCE_PATH, AUTO)
    host = [b.cpu().numpy() for b in bufs]
    for i, c in enumerate(links):
        assert not np.isnan(host[i + 1]).any(), f"link {i} output has NaN"
        ref, mag = oracle.linear(host[i], c.qweight, c.scales, c.bias, c.K, 32)
        assert_parity(host[i + 1], ref, mag, TOL_TC)


# ------------------------------------------------------------- split K (decode GEMV)
@pytest.mark.parametrize("N,K,gs", [(512, 8192, 32), (64, 4096, 64), (2048, 2048, 32),
                                    (1000, 8192, 8192), (2047, 14336, 128), (4096, 14336, 32),
                                    (28672, 4096, 32), (2048, 8192, 32)])
def test_split_k_parity_and_determinism(handle, N, K, gs):
    """The decode GEMV cuts its (row block, 1024-k stage) units evenly over the CTAs, so
    row blocks are split across CTAs at uneven K boundaries (partial sums in the handle's
    scratch, summed in K order by the last CTA of each block): parity, and bit-identical
    results over repeated calls (the counters reset themselves)."""
    c = synth.make_case(1, N, K, gs, scale_f16=(gs != K), bias=True, seed=N + K)
    outs = [run_q4lin(handle, c, AUTO)[0] for _ in range(3)]
    ref, mag = oracle.linear(c.x, c.qweight, c.scales, c.bias, K, gs)
    assert_parity(outs[0], ref, mag, TOL_FP32)
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], outs[2])


# ------------------------------------------------------- TMA-fed GEMV, 2 <= M <= 4 rows
# Shapes that take the multi-row TMA GEMV (4 weight rows per thread, or 2 when that avoids
# splitting K: 8192 x 2048 and 5120 x 2048 here): at least 10 M weights, K % 32 == 0, K >= 512,
# N >= 16, a scale row of whole 16-byte units (N % 8 for fp16 scales, N % 4 for fp32), a
# power-of-two group size (or one group per row).  Covered: ragged N (not a multiple of the
# 64-row block), a K tail shorter than a 512-k stage, groups of 32..512 k inside a stage
# and wider than a stage, per-channel scales (fp16 and fp32), the smallest N with a K long
# enough for the 8-part split, fp32 and fp16 scales.
MR_SHAPES = [
    # N, K, gs, f16, bias
    (8192, 2048, 32, True, True),
    (10056, 1056, 32, False, True),
    (2048, 8192, 128, True, True),
    (4104, 4096, 1024, False, False),
    (168, 65536, 65536, True, True),
    (24, 524288, 524288, True, False),
    (2600, 4096, 64, False, True),
    (5120, 2048, 256, True, False),
    (5120, 2048, 512, False, False),
    (10000, 1024, 1024, False, True),
]


@pytest.mark.parametrize("M", [2, 3, 4])
@pytest.mark.parametrize("N,K,gs,f16,bias", MR_SHAPES)
def test_multirow_gemv_parity(handle, M, N, K, gs, f16, bias):
    c = synth.make_case(M, N, K, gs, scale_f16=f16, bias=bias, seed=7 * N + K + M)
    _, used = check_case(handle, c, AUTO)
    assert used == GEMV


@pytest.mark.parametrize("M", [2, 4])
def test_multirow_gemv_lm_head(handle, M):
    c = synth.make_case(M, 128256, 2048, 32, scale_f16=True, bias=False, seed=50 + M)
    check_case(handle, c, GEMV)


@pytest.mark.parametrize("M", [2, 3, 4])
@pytest.mark.parametrize("N,K", [(2568, 4096), (6144, 2048)])
def test_multirow_gemv_even_high(handle, M, N, K):
    """Even k in the high nibble, with 4 weight rows per thread and K split (2568 x 4096)
    and with 2 rows per thread and no split (6144 x 2048)."""
    c = synth.make_case(M, N, K, 64, scale_f16=True, bias=True, seed=60 + M + N)
    check_case(handle, c, GEMV, even_high=True)


@pytest.mark.parametrize("M", [2, 3, 4])
@pytest.mark.parametrize("f16", [False, True])
def test_multirow_gemv_dyadic_bit_exact(handle, M, f16):
    c = synth.make_dyadic_case(M, 2560, 4096, 32, scale_f16=f16, bias=True, seed=70 + M)
    out, _ = run_q4lin(handle, c, GEMV)
    ref, _ = oracle.linear(c.x, c.qweight, c.scales, c.bias, c.K, c.group_size)
    np.testing.assert_array_equal(out.astype(np.float64), ref)


def test_multirow_gemv_all_codes_eight(handle):
    c = synth.make_case(4, 5120, 2048, 32, scale_f16=True, bias=True, seed=80)
    c.qweight = synth.fill_codes(5120, 2048, 8)
    out, _ = run_q4lin(handle, c, GEMV)
    np.testing.assert_array_equal(out, np.broadcast_to(c.bias, out.shape))


@pytest.mark.parametrize("M", [2, 4])
def test_multirow_gemv_split_k_deterministic(handle, M):
    """Few row blocks, long K: the K range is cut into parts whose partial sums are added
    in part order; repeated calls give identical bits."""
    c = synth.make_case(M, 640, 16384, 32, scale_f16=True, bias=True, seed=90 + M)
    outs = [run_q4lin(handle, c, AUTO)[0] for _ in range(3)]
    ref, mag = oracle.linear(c.x, c.qweight, c.scales, c.bias, c.K, 32)
    assert_parity(outs[0], ref, mag, TOL_FP32)
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], outs[2])


@pytest.mark.parametrize("pdl", [0, 1])
@pytest.mark.parametrize("M", [2, 4])
def test_multirow_dependent_chain(handle, pdl, M):
    """Multi-row GEMVs chained on one stream, each reading the previous output as its x
    (NaN-poisoned first): with programmatic dependent launch the weights of the first
    stages are requested early, x only after the predecessor completed."""
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    dims = [2048, 4096, 1024, 2048, 8192, 2048]
    links = [synth.make_case(M, dims[i + 1], dims[i], 32, scale_f16=True, bias=(i % 2 == 0),
                             seed=950 + i) for i in range(len(dims) - 1)]
    bufs = [torch.from_numpy(links[0].x).cuda()]
    bufs += [torch.full((M, d), float("nan"), device="cuda") for d in dims[1:]]
    dev = [tuple(None if a is None else torch.from_numpy(a).cuda()
                 for a in (c.qweight, c.scales, c.bias)) for c in links]
    torch.cuda.synchronize()
    q.q4lin_set_option(handle, q.Q4LIN_OPT_PDL, pdl)
    try:
        stream = torch.cuda.current_stream().cuda_stream
        for i, c in enumerate(links):
            w, s, b = dev[i]
            st = q.q4lin_run(handle, bufs[i].data_ptr(), w.data_ptr(), s.data_ptr(),
                             None if b is None else b.data_ptr(), bufs[i + 1].data_ptr(),
                             M, c.N, c.K, 32, q.Q4LIN_SCALE_F16, stream)
            assert st == q.Q4LIN_OK
        torch.cuda.synchronize()
    finally:
        q.q4lin_set_option(handle, q.Q4LIN_OPT_PDL, 0)
    host = [b.cpu().numpy() for b in bufs]
    for i, c in enumerate(links):
        assert not np.isnan(host[i + 1]).any(), f"link {i} output has NaN"
        ref, mag = oracle.linear(host[i], c.qweight, c.scales, c.bias, c.K, 32)
        assert_parity(host[i + 1], ref, mag, TOL_FP32)


def test_multirow_bounded_wait_times_out_cleanly(handle):
    """The multi-row GEMV's producer issues no copies (test hook): every consumer wait
    runs out after 1 ms, the kernel records code 1, walks its remaining work items
    (split-K counters included) without waiting and returns; the context stays usable and
    the next call is correct and deterministic."""
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    c = synth.make_case(4, 640, 16384, 32, scale_f16=True, bias=True, seed=78)
    st, code = q.q4lin_check_device_status(handle, None)
    assert (st, code) == (q.Q4LIN_OK, 0)
    q.q4lin_set_option(handle, q.Q4LIN_OPT_WAIT_LIMIT, 1_000_000)
    q.q4lin_set_option(handle, q.Q4LIN_OPT_TC_SKIP_FIRST_COPY, 1)
    try:
        run_q4lin(handle, c, GEMV)
    except AssertionError:
        pass  # the output of a timed-out call is undefined (NaN-poisoned here)
    finally:
        q.q4lin_set_option(handle, q.Q4LIN_OPT_TC_SKIP_FIRST_COPY, 0)
        q.q4lin_set_option(handle, q.Q4LIN_OPT_WAIT_LIMIT, 0)
    st, code = q.q4lin_check_device_status(handle, None)
    assert st == q.Q4LIN_ERR_TIMEOUT and code == 1
    st, code = q.q4lin_check_device_status(handle, None)
    assert (st, code) == (q.Q4LIN_OK, 0)
    torch.cuda.synchronize()
    a, _ = check_case(handle, c, GEMV)
    b, _ = run_q4lin(handle, c, GEMV)
    np.testing.assert_array_equal(a, b)


# ------------------------------------------- decode GEMV: fixed-point (dp4a) arithmetic
# Shapes whose CTAs take at least two row blocks each (here 49152 x 2048 and 65536 x 1024,
# 64-row blocks, and 28672 x 4096, 32-row blocks) run the decode GEMV's fixed-point
# arithmetic: x converted per 32-k chunk to 32-bit fixed point, exact integer dot products
# of the codes (dp4a), one rounding per chunk.  A stage with Inf / NaN, or with a nonzero
# element more than 2^13 below its chunk's largest, stays on the fp32 path.  Every test
# checks that the planner chose the fixed-point kernel.  65536 x 1024 is a single 1024-k
# stage of x (no second copy group to wait for).
X8_SHAPES = [(49152, 2048), (28672, 4096), (65536, 1024)]
X8_N, X8_K = X8_SHAPES[0]


def _assert_fixed_point(handle, c):
    assert _kernel_of(handle, c) == "gemv_tma_fixed", "the shape no longer takes the fixed-point path"


def test_gemv_small_launch_stays_fp32(handle):
    """One row block per CTA: the conversion of x would not pay, the fp32 loop runs."""
    c = synth.make_case(1, 8192, 2048, 32, scale_f16=True, bias=True, seed=17)
    assert _kernel_of(handle, c) == "gemv_tma"


@pytest.mark.parametrize("N,K", X8_SHAPES)
@pytest.mark.parametrize("gs,f16", [(32, True), (32, False), (128, True), (None, False)])
def test_gemv_fixed_point_dyadic_bit_exact(handle, N, K, gs, f16):
    gs = gs or K
    c = synth.make_dyadic_case(1, N, K, gs, scale_f16=f16, bias=True, seed=N + gs)
    _assert_fixed_point(handle, c)
    out, used = run_q4lin(handle, c, AUTO)
    assert used == GEMV
    ref, _ = oracle.linear(c.x, c.qweight, c.scales, c.bias, c.K, c.group_size)
    np.testing.assert_array_equal(out.astype(np.float64), ref)


def test_gemv_fixed_point_all_codes_eight_gives_bias(handle):
    c = synth.make_case(1, X8_N, X8_K, 32, scale_f16=True, bias=True, seed=19)
    c.qweight = synth.fill_codes(X8_N, X8_K, 8)
    _assert_fixed_point(handle, c)
    out, _ = run_q4lin(handle, c, AUTO)
    np.testing.assert_array_equal(out, np.broadcast_to(c.bias, out.shape))


@pytest.mark.parametrize("N,K", X8_SHAPES)
def test_gemv_fixed_point_even_high(handle, N, K):
    c = synth.make_case(1, N, K, 32, scale_f16=True, bias=True, seed=23)
    _assert_fixed_point(handle, c)
    check_case(handle, c, AUTO, even_high=True)


def _assert_ieee_match(out, ref, mag):
    """NaN and +/-Inf positions equal to the oracle's, finite elements within the bar."""
    o = out.astype(np.float64)
    assert np.array_equal(np.isnan(o), np.isnan(ref)), "NaN positions differ"
    inf = np.isinf(ref)
    assert np.array_equal(np.isinf(o), inf), "Inf positions differ"
    assert np.array_equal(o[inf], ref[inf]), "Inf signs differ"
    fin = np.isfinite(ref)
    if fin.any():
        assert_parity(out[fin][None, :], ref[fin][None, :], mag[fin][None, :], TOL_FP32)


@pytest.mark.parametrize("case", ["pos_inf", "neg_and_pos_inf", "nan"])
def test_gemv_fixed_point_non_finite_x(handle, case):
    """Inf and NaN in x propagate as in IEEE arithmetic (Inf * 0 = NaN, Inf - Inf = NaN),
    element by element as the fp64 oracle computes them; the other chunks of the same
    launch stay on the fixed-point path."""
    c = synth.make_case(1, X8_N, X8_K, 32, scale_f16=True, bias=True, seed=29)
    _assert_fixed_point(handle, c)
    x = c.x.copy()
    if case == "pos_inf":
        x[0, 5] = np.inf
    elif case == "neg_and_pos_inf":
        x[0, 5] = np.inf
        x[0, 1500] = -np.inf
    else:
        x[0, 700] = np.nan
    c.x = x
    out, _ = run_q4lin(handle, c, AUTO)
    with np.errstate(invalid="ignore"):
        ref, mag = oracle.linear(c.x, c.qweight, c.scales, c.bias, c.K, 32)
    _assert_ieee_match(out, ref, mag)
    if case == "pos_inf":
        assert np.isnan(out).any() and np.isinf(out).any()


@pytest.mark.parametrize("ratio", [1e3, 1e4, 1e5, 1e7])
def test_gemv_fixed_point_dynamic_range(handle, ratio):
    """Every 32-k chunk holds one element `ratio` times larger than the rest, and for half
    of the rows that element's code is 8 (weight 0), so the tolerance comes only from the
    small elements: chunks within 2^13 of their largest are converted to fixed point
    (relative error <= 2^-18 per element), wider ones stay fp32; both stay in the bar."""
    N, K = X8_N, X8_K
    c = synth.make_case(1, N, K, 32, scale_f16=True, bias=True, seed=int(ratio) % 1000)
    _assert_fixed_point(handle, c)
    x = c.x.copy()
    x[0, 7::32] *= ratio
    c.x = x
    w = c.qweight.copy()
    rows = np.arange(0, N, 2)
    byte = 7 // 2  # k = 7 + 32 j sits in byte 16 j + 3, high nibble
    for j in range(K // 32):
        b = w[rows, 16 * j + byte]
        w[rows, 16 * j + byte] = (b & 0x0F) | 0x80
    c.qweight = w
    check_case(handle, c, AUTO)


def test_gemv_fixed_point_zero_and_subnormal_chunks(handle):
    """All-zero chunks, subnormal x and a chunk of equal values convert without error."""
    N, K = X8_N, X8_K
    c = synth.make_case(1, N, K, 32, scale_f16=False, bias=True, seed=37)
    _assert_fixed_point(handle, c)
    x = c.x.copy()
    x[0, :64] = 0.0
    x[0, 64:96] = np.float32(1e-40)
    x[0, 96:128] = np.float32(-3.0)
    x[0, 128:160] = np.float32(2.0 ** -120)
    c.x = x
    check_case(handle, c, AUTO)


# ------------------------------------------------ tensor-core GEMM with fp16 operands
# Q4LIN_OPT_TC_F16: x and the dequantized weights rounded to fp16 (x by a conversion
# kernel into the handle's scratch), tcgen05.mma kind::f16 with fp32 accumulation.
@pytest.fixture()
def f16_handle(handle):
    from bit_weight_quantized_int4_gb300 import q4lin as q
    assert q.q4lin_set_option(handle, q.Q4LIN_OPT_TC_F16, 1) == q.Q4LIN_OK
    yield handle
    q.q4lin_set_option(handle, q.Q4LIN_OPT_TC_F16, 0)


def _kernel_of(handle, c, path=AUTO):
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    from tests._gpu import device_case
    x, w, s, b = device_case(c)
    out = torch.empty(c.M, c.N, device="cuda")
    sd = q.Q4LIN_SCALE_F16 if c.scale_f16 else q.Q4LIN_SCALE_F32
    q.q4lin_set_option(handle, q.Q4LIN_OPT_FORCE_PATH, path)
    try:
        st, k = q.q4lin_plan_kernel(handle, x.data_ptr(), w.data_ptr(), s.data_ptr(),
                                    None if b is None else b.data_ptr(), out.data_ptr(), c.M,
                                    c.N, c.K, c.group_size, sd)
    finally:
        q.q4lin_set_option(handle, q.Q4LIN_OPT_FORCE_PATH, AUTO)
    assert st == q.Q4LIN_OK
    return q.KERNEL_NAMES[k]


@pytest.mark.parametrize("M,N,K,gs,f16,bias", TC_SHAPES)
def test_tc_f16_parity(f16_handle, M, N, K, gs, f16, bias):
    c = synth.make_case(M, N, K, gs, scale_f16=f16, bias=bias, seed=M + N + 1)
    assert _kernel_of(f16_handle, c, TC) == "tc_f16"
    _, used = check_case(f16_handle, c, TC)
    assert used == TC


@pytest.mark.parametrize("M,N,K", [(2048, 2048, 2048), (512, 8192, 2048), (128, 2048, 8192),
                                   (2048, 512, 2048)])
def test_tc_f16_prefill_shapes(f16_handle, M, N, K):
    c = synth.make_case(M, N, K, 32, scale_f16=False, bias=True, seed=M + K)
    assert _kernel_of(f16_handle, c) == "tc_f16"
    check_case(f16_handle, c, AUTO)


@pytest.mark.parametrize("M", [5, 48, 300])
def test_tc_f16_dyadic_bit_exact(f16_handle, M):
    c = synth.make_dyadic_case(M, 260, 1056, 32, scale_f16=(M % 2 == 1), bias=True, seed=M)
    out, used = run_q4lin(f16_handle, c, TC)
    assert used == TC
    ref, _ = oracle.linear(c.x, c.qweight, c.scales, c.bias, c.K, c.group_size)
    np.testing.assert_array_equal(out.astype(np.float64), ref)


@pytest.mark.parametrize("what", ["x", "scale"])
def test_tc_f16_out_of_range_is_reported(f16_handle, what):
    """A value that fp16 cannot hold (x >= 65520, or a scale above 8188 so that a weight
    passes 65504) records code 2 in the status word; the next in-range call is correct."""
    from bit_weight_quantized_int4_gb300 import q4lin as q
    c = synth.make_case(64, 256, 512, 32, scale_f16=False, bias=False, seed=5)
    bad = synth.make_case(64, 256, 512, 32, scale_f16=False, bias=False, seed=5)
    if what == "x":
        bad.x = bad.x.copy()
        bad.x[3, 17] = 1.0e5
    else:
        bad.scales = bad.scales.copy()
        bad.scales[2, 9] = 1.0e4
    assert q.q4lin_check_device_status(f16_handle, None) == (q.Q4LIN_OK, 0)
    run_q4lin(f16_handle, bad, TC)
    st, code = q.q4lin_check_device_status(f16_handle, None)
    assert st == q.Q4LIN_ERR_TIMEOUT and code == 2
    check_case(f16_handle, c, TC)
    assert q.q4lin_check_device_status(f16_handle, None) == (q.Q4LIN_OK, 0)


@pytest.mark.parametrize("pdl", [0, 1])
def test_tc_f16_dependent_chain(f16_handle, pdl):
    """fp16 GEMMs chained on one stream (each reads the previous output as x): the
    conversion of x runs after the preceding GEMM completed, the GEMM after the
    conversion; each link checked against the oracle on the input it received."""
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    M, dims = 200, [512, 1024, 256, 768]
    links = [synth.make_case(M, dims[i + 1], dims[i], 32, scale_f16=(i % 2 == 1),
                             bias=(i % 2 == 0), seed=800 + i) for i in range(len(dims) - 1)]
    bufs = [torch.from_numpy(np.ascontiguousarray(links[0].x)).cuda()]
    bufs += [torch.full((M, d), float("nan"), device="cuda") for d in dims[1:]]
    dev = [tuple(None if a is None else torch.from_numpy(a).cuda()
                 for a in (c.qweight, c.scales, c.bias)) for c in links]
    torch.cuda.synchronize()
    q.q4lin_set_option(f16_handle, q.Q4LIN_OPT_PDL, pdl)
    q.q4lin_set_option(f16_handle, q.Q4LIN_OPT_FORCE_PATH, TC)
    try:
        stream = torch.cuda.current_stream().cuda_stream
        for i, c in enumerate(links):
            w, s, b = dev[i]
            sd = q.Q4LIN_SCALE_F16 if c.scales.dtype == np.float16 else q.Q4LIN_SCALE_F32
            st = q.q4lin_run(f16_handle, bufs[i].data_ptr(), w.data_ptr(), s.data_ptr(),
                             None if b is None else b.data_ptr(), bufs[i + 1].data_ptr(),
                             M, c.N, c.K, 32, sd, stream)
            assert st == q.Q4LIN_OK
        torch.cuda.synchronize()
    finally:
        q.q4lin_set_option(f16_handle, q.Q4LIN_OPT_PDL, 0)
        q.q4lin_set_option(f16_handle, q.Q4LIN_OPT_FORCE_PATH, AUTO)
    host = [b.cpu().numpy() for b in bufs]
    for i, c in enumerate(links):
        assert not np.isnan(host[i + 1]).any(), f"link {i} output has NaN"
        ref, mag = oracle.linear(host[i], c.qweight, c.scales, c.bias, c.K, 32)
        assert_parity(host[i + 1], ref, mag, TOL_TC)
