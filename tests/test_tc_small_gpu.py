"""Parity of the tensor-core GEMM for 2 <= M <= 32 activation rows (Q4LIN_PATH_TC_SMALL,
bit_weight_quantized_int4_gb300/csrc/tc_small.cu) with the fp64 oracle, through the C ABI.

Every element of out[M, N] is checked at the tensor-core tolerance (4e-3 * sum_k|x*w| +
1e-6); dyadic inputs and all-8 codes must come out bit-exact.  Covered: every M from 2 to
32 (MMA width 16 up to 16 rows, 32 above), ragged N (rows past N in the last 128-row block), ragged K (a last 256-k stage that is
mostly past K), the longest K whose x stays resident and longer ones whose x streams,
group sizes from 32 to wider than a stage,
per-channel scales (fp16 and fp32), fp32 and fp16 group scales, bias or none, the
even-high nibble order, persistent CTAs over many blocks (more blocks than SMs), repeated
calls bit-identical, and a bounded wait that runs out cleanly.  Up to 8 rows (x resident,
K > 256) the kernel can multiply bf16 operands (x as bf16(x) + bf16(x - bf16(x))): by
default from 100 row blocks, forced here with Q4LIN_OPT_TC_SMALL_OPERANDS = 2 on smaller
matrices; tf32 is forced with 1.
"""
import numpy as np
import pytest

import oracle
from bit_weight_quantized_int4_gb300 import synth
from tests._gpu import TOL_TC, assert_parity, run_q4lin

pytestmark = pytest.mark.gpu

TC_SMALL = 4


@pytest.fixture(scope="module")
def handle():
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    assert torch.cuda.is_available()
    h = q.q4lin_create(0)
    yield h
    q.q4lin_destroy(h)


def check(handle, case, even_high=False):
    out, used = run_q4lin(handle, case, TC_SMALL, even_high)
    assert used == TC_SMALL
    ref, mag = oracle.linear(case.x, case.qweight, case.scales, case.bias, case.K,
                             case.group_size, even_high=even_high)
    assert_parity(out, ref, mag, TOL_TC)
    return out


@pytest.fixture
def bf16(handle):
    """The handle with bf16 operands wherever they apply, for one test."""
    from bit_weight_quantized_int4_gb300 import q4lin as q
    q.q4lin_set_option(handle, q.Q4LIN_OPT_TC_SMALL_OPERANDS, 2)
    yield handle
    q.q4lin_set_option(handle, q.Q4LIN_OPT_TC_SMALL_OPERANDS, 0)


def kernel_of(handle, case):
    """The kernel name q4lin_plan_kernel reports for the case on the forced small-M path."""
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    M, N, K = case.M, case.N, case.K
    x = torch.zeros(M, K, device="cuda")
    w = torch.zeros(N, K // 2, dtype=torch.uint8, device="cuda")
    s = torch.from_numpy(case.scales).cuda()
    out = torch.empty(M, N, device="cuda")
    q.q4lin_set_option(handle, q.Q4LIN_OPT_FORCE_PATH, TC_SMALL)
    try:
        st, k = q.q4lin_plan_kernel(handle, x.data_ptr(), w.data_ptr(), s.data_ptr(), None,
                                    out.data_ptr(), M, N, K, case.group_size,
                                    q.Q4LIN_SCALE_F16 if case.scale_f16 else q.Q4LIN_SCALE_F32)
    finally:
        q.q4lin_set_option(handle, q.Q4LIN_OPT_FORCE_PATH, 0)
    assert st == q.Q4LIN_OK
    return q.KERNEL_NAMES[k]


@pytest.mark.parametrize("M", list(range(2, 33)))
def test_every_m(handle, M):
    c = synth.make_case(M, 1000, 2048, 32, scale_f16=True, bias=True, seed=M)
    assert kernel_of(handle, c) == "tc_small"  # 8 row blocks: tf32 by default
    check(handle, c)


@pytest.mark.parametrize("M", list(range(2, 9)))
def test_every_m_bf16_operands(bf16, M):
    c = synth.make_case(M, 1000, 2048, 32, scale_f16=True, bias=True, seed=M)
    assert kernel_of(bf16, c) == "tc_small_bf16"
    check(bf16, c)


@pytest.mark.parametrize("M,N,K,gs,f16,kern", [
    (4, 1000, 256, 32, True, "tc_small"),         # one 256-k stage: tf32
    (4, 1000, 512, 32, True, "tc_small_bf16"),    # two stages
    (8, 384, 5120, 32, True, "tc_small"),         # resident, but an even ring < 4 stages
    (8, 384, 4096, 32, False, "tc_small_bf16"),   # four stages of the ring, fp32 scales
    (5, 520, 2048, 2048, False, "tc_small_bf16"),  # per channel, fp32
    (3, 200, 1056, 32, False, "tc_small_bf16"),   # ragged N and K (last stage mostly past K)
    (7, 1032, 1536, 1536, True, "tc_small_bf16"),  # per channel, fp16, ragged N
    (2, 4104, 2048, 64, True, "tc_small_bf16"),   # 33 blocks, group 64
    (6, 1024, 2048, 1024, True, "tc_small_bf16"),  # group wider than a stage
    (4, 2600, 8192, 32, True, "tc_small"),        # x streamed
    (9, 1000, 2048, 32, True, "tc_small"),        # more than 8 rows
])
def test_where_bf16_operands_apply(bf16, M, N, K, gs, f16, kern):
    c = synth.make_case(M, N, K, gs, scale_f16=f16, bias=True, seed=M + N + K)
    assert kernel_of(bf16, c) == kern
    check(bf16, c)


@pytest.mark.parametrize("M,N,kern", [(4, 12800, "tc_small_bf16"), (4, 12672, "tc_small"),
                                      (8, 12800, "tc_small_bf16"), (9, 12800, "tc_small")])
def test_default_operands_from_100_blocks(handle, M, N, kern):
    c = synth.make_case(M, N, 512, 32, scale_f16=True, bias=True, seed=M + N)
    assert kernel_of(handle, c) == kern
    check(handle, c)


@pytest.mark.parametrize("N,K,gs,f16,bias", [
    (128, 512, 32, True, True),        # one block, two stages
    (200, 1056, 32, False, True),      # ragged N and K (the last stage mostly past K)
    (4104, 2048, 64, True, False),     # ragged N over 33 blocks
    (2600, 2560, 128, False, True),    # the longest K that 16 resident rows of x allow
    (1024, 2048, 1024, True, True),    # group wider than a stage
    (520, 2048, 2048, False, True),    # per channel, fp32
    (136, 1536, 1536, True, False),    # per channel, fp16
])
def test_shapes(handle, N, K, gs, f16, bias):
    for M in (2, 7, 16, 17, 32):
        check(handle, synth.make_case(M, N, K, gs, scale_f16=f16, bias=bias, seed=N + K + M))


@pytest.mark.parametrize("N,K,gs,f16", [(384, 5120, 32, True), (1000, 4096, 64, False)])
@pytest.mark.parametrize("M", [2, 8])
def test_long_k_up_to_8_rows(handle, M, N, K, gs, f16):
    """Up to 8 rows, x is kept as 8-row chunks: K up to 5120 stays resident."""
    check(handle, synth.make_case(M, N, K, gs, scale_f16=f16, bias=True, seed=N + K + M))


@pytest.mark.parametrize("M,N,K,gs,f16", [
    (4, 2600, 8192, 32, True),      # 8-row chunks of x, too long to stay resident
    (12, 1000, 4096, 64, False),    # 16-row chunks, K > 2560
    (16, 700, 14336, 14336, True),  # per channel, long K
    (9, 3000, 2592, 32, True),      # just past the resident limit of 16-row chunks, ragged K
    (24, 1504, 2048, 32, True),     # 32-row chunks (MMA width 32)
])
def test_streamed_x(handle, M, N, K, gs, f16):
    """x too long to stay resident in shared memory: it streams through a ring of three
    256-k groups per CTA, released by the MMAs' commits."""
    check(handle, synth.make_case(M, N, K, gs, scale_f16=f16, bias=True, seed=N + K + M))


def test_streamed_x_dyadic_bit_exact(handle):
    c = synth.make_dyadic_case(12, 264, 4096, 32, scale_f16=True, bias=True, seed=12)
    out, used = run_q4lin(handle, c, TC_SMALL)
    assert used == TC_SMALL
    ref, _ = oracle.linear(c.x, c.qweight, c.scales, c.bias, c.K, c.group_size)
    np.testing.assert_array_equal(out.astype(np.float64), ref)


@pytest.mark.parametrize("M,mode", [(3, 0), (3, 1), (16, 0), (32, 0)])
def test_persistent_over_many_blocks(handle, M, mode):
    """More 128-row blocks than SMs (the vocabulary-sized head): each CTA takes several
    blocks with the accumulators double-buffered between them (bf16 operands by default
    at 3 rows, tf32 forced as well)."""
    from bit_weight_quantized_int4_gb300 import q4lin as q
    c = synth.make_case(M, 128256, 2048, 32, scale_f16=True, bias=True, seed=M)
    q.q4lin_set_option(handle, q.Q4LIN_OPT_TC_SMALL_OPERANDS, mode)
    try:
        assert kernel_of(handle, c) == ("tc_small_bf16" if M <= 8 and mode == 0 else "tc_small")
        check(handle, c)
    finally:
        q.q4lin_set_option(handle, q.Q4LIN_OPT_TC_SMALL_OPERANDS, 0)


def test_even_high(handle):
    check(handle, synth.make_case(5, 704, 2048, 64, scale_f16=True, bias=True, seed=3),
          even_high=True)


def test_even_high_bf16_operands(bf16):
    check(bf16, synth.make_case(5, 704, 2048, 64, scale_f16=True, bias=True, seed=4),
          even_high=True)


@pytest.mark.parametrize("M,f16,mode", [(2, True, 2), (5, False, 2), (8, True, 2), (3, True, 0),
                                        (9, False, 0), (16, True, 0), (24, False, 0), (32, True, 0)])
def test_dyadic_bit_exact(handle, M, f16, mode):
    from bit_weight_quantized_int4_gb300 import q4lin as q
    c = synth.make_dyadic_case(M, 264, 1024, 32, scale_f16=f16, bias=True, seed=M)
    q.q4lin_set_option(handle, q.Q4LIN_OPT_TC_SMALL_OPERANDS, mode)
    try:
        assert kernel_of(handle, c) == ("tc_small_bf16" if mode == 2 else "tc_small")
        out, used = run_q4lin(handle, c, TC_SMALL)
    finally:
        q.q4lin_set_option(handle, q.Q4LIN_OPT_TC_SMALL_OPERANDS, 0)
    assert used == TC_SMALL
    ref, _ = oracle.linear(c.x, c.qweight, c.scales, c.bias, c.K, c.group_size)
    np.testing.assert_array_equal(out.astype(np.float64), ref)


def test_all_codes_eight_gives_bias(handle):
    c = synth.make_case(6, 336, 2048, 32, scale_f16=True, bias=True, seed=9)
    c.qweight = synth.fill_codes(336, 2048, 8)
    out, _ = run_q4lin(handle, c, TC_SMALL)
    np.testing.assert_array_equal(out, np.broadcast_to(c.bias, out.shape))


def test_repeated_calls_bit_identical(handle):
    c = synth.make_case(8, 30000, 2048, 32, scale_f16=True, bias=True, seed=5)
    a = check(handle, c)
    b, _ = run_q4lin(handle, c, TC_SMALL)
    np.testing.assert_array_equal(a, b)


def test_ineligible_shapes_are_refused(handle):
    """M outside 2..32, K not a multiple of 32, or a group size that is not a power-of-two
    multiple of 32: the forced path reports Q4LIN_ERR_UNSUPPORTED and nothing runs."""
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    q.q4lin_set_option(handle, q.Q4LIN_OPT_FORCE_PATH, TC_SMALL)
    try:
        for M, N, K, gs in [(1, 256, 512, 32), (33, 256, 512, 32), (4, 256, 528, 48),
                            (4, 256, 1024, 96)]:
            c = synth.make_case(M, N, K, gs, scale_f16=False, bias=False, seed=1)
            x = torch.from_numpy(c.x).cuda()
            w = torch.from_numpy(c.qweight).cuda()
            s = torch.from_numpy(c.scales).cuda()
            out = torch.empty(M * N, device="cuda")
            st, _ = q.q4lin_plan(handle, x.data_ptr(), w.data_ptr(), s.data_ptr(), None,
                                 out.data_ptr(), M, N, K, gs, q.Q4LIN_SCALE_F32)
            assert st == q.Q4LIN_ERR_UNSUPPORTED, (M, N, K, gs)
    finally:
        q.q4lin_set_option(handle, q.Q4LIN_OPT_FORCE_PATH, 0)


@pytest.mark.parametrize("mode", [1, 2])
def test_bounded_wait_times_out_cleanly(handle, mode):
    """The producer skips its first copy (test hook), so the barrier the first slots wait on
    is never completed: the 1 ms bounded waits run out, the kernel records code 1, drains
    its MMAs, frees its tensor memory and returns; the next call is correct.  With bf16
    operands (mode 2) a stage holds two A slots, so the teams and issuers of the second
    stage get through their first slot before everything stops: no role may then run on
    into ring laps whose previous lap never happened."""
    from bit_weight_quantized_int4_gb300 import q4lin as q
    c = synth.make_case(4, 1024, 2048, 32, scale_f16=True, bias=False, seed=77)
    st, code = q.q4lin_check_device_status(handle, None)
    assert (st, code) == (q.Q4LIN_OK, 0)
    q.q4lin_set_option(handle, q.Q4LIN_OPT_TC_SMALL_OPERANDS, mode)
    assert kernel_of(handle, c) == ("tc_small_bf16" if mode == 2 else "tc_small")
    q.q4lin_set_option(handle, q.Q4LIN_OPT_WAIT_LIMIT, 1_000_000)
    q.q4lin_set_option(handle, q.Q4LIN_OPT_TC_SKIP_FIRST_COPY, 1)
    try:
        run_q4lin(handle, c, TC_SMALL)
    except AssertionError:
        pass  # the output of a timed-out call is undefined (NaN-poisoned here)
    finally:
        q.q4lin_set_option(handle, q.Q4LIN_OPT_TC_SKIP_FIRST_COPY, 0)
        q.q4lin_set_option(handle, q.Q4LIN_OPT_WAIT_LIMIT, 0)
    st, code = q.q4lin_check_device_status(handle, None)
    assert st == q.Q4LIN_ERR_TIMEOUT and code == 1
    st, code = q.q4lin_check_device_status(handle, None)
    assert (st, code) == (q.Q4LIN_OK, 0)
    try:
        check(handle, c)
    finally:
        q.q4lin_set_option(handle, q.Q4LIN_OPT_TC_SMALL_OPERANDS, 0)


@pytest.mark.parametrize("M,N,K,gs,f16,mode", [
    (8, 4096, 4096, 32, True, 0),     # 32 blocks: 4 parts of 4 stages
    (6, 6144, 4096, 64, False, 0),    # 48 blocks: 2 parts, fp32 scales
    (16, 2048, 8192, 128, True, 0),   # 16 blocks: 8 parts (x streamed through the ring)
    (5, 1000, 2048, 32, True, 0),     # 8 blocks, ragged N: 4 parts of 2 stages
    (3, 520, 4096, 4096, True, 0),    # per channel, 5 blocks
    (24, 1504, 2048, 32, True, 0),    # MMA width 32, 12 blocks
    (4, 2048, 2048, 32, True, 2),     # bf16 operands, 4 parts of 2 stages
    (8, 3000, 1024, 32, False, 2),    # bf16 operands, ragged N, 2 parts
])
def test_k_split(handle, M, N, K, gs, f16, mode):
    """Fewer 128-row blocks than half the SMs: each block is split over K into parts whose
    partial tiles the last part of the block adds (in part order) through the workspace."""
    from bit_weight_quantized_int4_gb300 import q4lin as q
    c = synth.make_case(M, N, K, gs, scale_f16=f16, bias=True, seed=M + N + K)
    q.q4lin_set_option(handle, q.Q4LIN_OPT_TC_SMALL_OPERANDS, mode)
    try:
        a = check(handle, c)
        b, _ = run_q4lin(handle, c, TC_SMALL)
        np.testing.assert_array_equal(a, b)  # the part order fixes the sum
    finally:
        q.q4lin_set_option(handle, q.Q4LIN_OPT_TC_SMALL_OPERANDS, 0)


@pytest.mark.parametrize("M,N,K", [(8, 2048, 4096), (4, 1000, 2048)])
def test_k_split_dyadic_bit_exact(handle, M, N, K):
    c = synth.make_dyadic_case(M, N, K, 32, scale_f16=True, bias=True, seed=N + K)
    out, used = run_q4lin(handle, c, TC_SMALL)
    assert used == TC_SMALL
    ref, _ = oracle.linear(c.x, c.qweight, c.scales, c.bias, c.K, c.group_size)
    np.testing.assert_array_equal(out.astype(np.float64), ref)


@pytest.mark.parametrize("pdl", [0, 1])
@pytest.mark.parametrize("M", [4, 12, 20])
def test_chain_with_dependent_launch(handle, M, pdl):
    """Four launches where each output is the next input, with programmatic dependent
    launch on and off: the weights stream before the dependency wait, x is read after it
    and out is written after it; each link is checked against the oracle applied to the
    input it actually received."""
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    dims = [512, 1024, 256, 768, 2048]
    links = [synth.make_case(M, dims[i + 1], dims[i], 32, scale_f16=(i % 2 == 1),
                             bias=(i % 2 == 0), seed=900 + i + M) for i in range(4)]
    bufs = [torch.from_numpy(np.ascontiguousarray(links[0].x)).cuda()]
    bufs += [torch.full((M, d), float("nan"), device="cuda") for d in dims[1:]]
    dev = [tuple(None if a is None else torch.from_numpy(a).cuda()
                 for a in (c.qweight, c.scales, c.bias)) for c in links]
    torch.cuda.synchronize()
    q.q4lin_set_option(handle, q.Q4LIN_OPT_PDL, pdl)
    q.q4lin_set_option(handle, q.Q4LIN_OPT_FORCE_PATH, TC_SMALL)
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
        q.q4lin_set_option(handle, q.Q4LIN_OPT_FORCE_PATH, 0)
    host = [b.cpu().numpy() for b in bufs]
    for i, c in enumerate(links):
        assert not np.isnan(host[i + 1]).any(), f"link {i} output has NaN"
        ref, mag = oracle.linear(host[i], c.qweight, c.scales, c.bias, c.K, 32)
        assert_parity(host[i + 1], ref, mag, TOL_TC)


def _auto_kernel(handle, M, N, K, f16=True):
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    x = torch.zeros(M, K, device="cuda")
    w = torch.zeros(N, K // 2, dtype=torch.uint8, device="cuda")
    s = torch.zeros(K // 32, N, dtype=torch.float16 if f16 else torch.float32, device="cuda")
    out = torch.empty(M, N, device="cuda")
    st, k = q.q4lin_plan_kernel(handle, x.data_ptr(), w.data_ptr(), s.data_ptr(), None,
                                out.data_ptr(), M, N, K, 32,
                                q.Q4LIN_SCALE_F16 if f16 else q.Q4LIN_SCALE_F32)
    assert st == q.Q4LIN_OK
    return q.KERNEL_NAMES[k]


@pytest.mark.parametrize("M,N,K,kernel", [
    (2, 128256, 2048, "multirow"),   # two rows: the multi-row GEMV is faster
    (3, 128256, 2048, "tc_small_bf16"),  # bf16 operands from 100 row blocks
    (4, 28672, 4096, "tc_small_bf16"),
    (3, 22016, 4096, "multirow"),    # a last wave of 20 blocks on 152 SMs
    (3, 14336, 4096, "multirow"),    # 3 rows on less than one wave (112 blocks)
    (3, 28672, 4096, "tc_small_bf16"),  # 224 blocks
    (4, 8192, 2048, "multirow"),     # 64 blocks at 3-4 rows
    (8, 8192, 2048, "tc_small"),     # 64 blocks of 8 stages
    (8, 4096, 4096, "tc_small"),     # 32 blocks of 16 stages: K split in 4 parts
    (16, 128256, 2048, "tc_small"),
    (16, 14336, 4096, "tc_small"),   # 16 rows of x for K = 4096 stream through a ring
    (8, 2048, 2048, "tc_small"),     # 16 blocks, 4 M weights: K split in 4 parts
    (8, 1000, 2048, "rowstream"),    # 2 M weights: the CUDA-core path
    (12, 2048, 8192, "tc_small"),    # 16 blocks of 32 stages: K split in 8 parts
    (4, 4096, 14336, "tc_small"),    # 4 rows, K split, long rows of >= 4096 rows
    (4, 4096, 4096, "multirow"),     # 3-4 rows keep the multi-row GEMV below 100 blocks
    (4, 2048, 8192, "multirow"),     # 4 rows on 2048 rows: the multi-row GEMV
    (12, 1000, 2048, "tc_small"),    # 9-16 rows: the K split at any size
    (24, 2048, 8192, "tc"),          # 17-32 rows on few blocks: the tile GEMM
    (24, 128256, 2048, "tc_small"),  # MMA width 32
    (24, 8192, 2048, "tc"),          # 64 blocks above 16 rows: the tile GEMM
])
def test_auto_dispatch(handle, M, N, K, kernel):
    assert _auto_kernel(handle, M, N, K) == kernel
