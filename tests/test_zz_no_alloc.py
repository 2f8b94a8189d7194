"""q4lin_run_static_scratch: the decode GEMV for callers that cannot allocate device
memory (during a stream capture that forbids allocation, inside a custom allocator, on
real-time paths).  Its split-K scratch is a fixed array in the library's device image.

Checked through the C ABI against the fp64 oracle at the tolerance of the CUDA-core
paths, and against the existing entry point (q4lin_run with a handle), on two calls in a
row; the second call reuses the array the first one left behind.  The largest accepted N
(16384) with a long K runs the split-K scratch at its capacity.  This file is collected
last."""
import numpy as np
import pytest

import oracle
from bit_weight_quantized_int4_gb300 import synth
from tests._gpu import TOL_FP32, assert_parity

pytestmark = pytest.mark.gpu


def _dev(c):
    import torch
    t = lambda a: None if a is None else torch.from_numpy(a).cuda()
    return t(c.x), t(c.qweight), t(c.scales), t(c.bias)


@pytest.mark.parametrize("N,K,gs,f16", [(2048, 8192, 32, True),     # split along K
                                        (1000, 8192, 8192, False),  # per-channel, split
                                        (512, 2048, 64, True),
                                        (16384, 8192, 32, True)])   # N at the limit
def test_static_scratch_matches_oracle_and_run(N, K, gs, f16):
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    h = q.q4lin_create(0)
    try:
        sd = q.Q4LIN_SCALE_F16 if f16 else q.Q4LIN_SCALE_F32
        stream = torch.cuda.current_stream().cuda_stream
        for call in range(2):  # two calls in a row, different inputs
            c = synth.make_case(1, N, K, gs, scale_f16=f16, bias=True, seed=300 + call)
            x, w, s, b = _dev(c)
            want = torch.full((N,), float("nan"), device="cuda")
            got = torch.full((N,), float("nan"), device="cuda")
            assert q.q4lin_run(h, x.data_ptr(), w.data_ptr(), s.data_ptr(), b.data_ptr(),
                               want.data_ptr(), 1, N, K, gs, sd, stream) == q.Q4LIN_OK
            assert q.q4lin_run_static_scratch(x.data_ptr(), w.data_ptr(), s.data_ptr(),
                                              b.data_ptr(), got.data_ptr(), N, K, gs, sd,
                                              stream) == q.Q4LIN_OK
            torch.cuda.synchronize()
            ref, mag = oracle.linear(c.x, c.qweight, c.scales, c.bias, K, gs)
            g = got.cpu().numpy()[None, :]
            assert_parity(g, ref, mag, TOL_FP32)
            a = want.cpu().numpy()[None, :].astype(np.float64)
            rel, ab = TOL_FP32
            assert np.all(np.abs(g.astype(np.float64) - a) <= rel * mag + ab)
    finally:
        q.q4lin_destroy(h)


def test_static_scratch_rejects_too_large():
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    N, K = 16385, 512
    w = torch.zeros((N, K // 2), dtype=torch.uint8, device="cuda")
    s = torch.zeros((K // 32, N), dtype=torch.float16, device="cuda")
    x = torch.zeros(K, device="cuda")
    out = torch.full((N,), 7.0, device="cuda")
    st = q.q4lin_run_static_scratch(x.data_ptr(), w.data_ptr(), s.data_ptr(), None,
                                    out.data_ptr(), N, K, 32, q.Q4LIN_SCALE_F16, None)
    assert st == q.Q4LIN_ERR_TOO_LARGE
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)
