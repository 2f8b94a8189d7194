"""q4lin_run_grouped: the result equals q4lin_run on each problem in order; runs of
M = 1 problems sharing x are fused into one launch (checked against the fp64 oracle)."""
import numpy as np
import pytest

import oracle
from bit_weight_quantized_int4_gb300 import synth
from tests._gpu import TOL_FP32, assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    from bit_weight_quantized_int4_gb300 import q4lin
    return q4lin


@pytest.fixture(scope="module")
def handle(q):
    h = q.q4lin_create(0)
    yield h
    q.q4lin_destroy(h)


def _problems(cases, x_shared=True):
    """Device buffers for cases; with x_shared every case reads cases[0].x."""
    import torch
    x0 = torch.from_numpy(cases[0].x).cuda()
    dev = []
    for c in cases:
        x = x0 if x_shared else torch.from_numpy(c.x).cuda()
        w = torch.from_numpy(c.qweight).cuda()
        s = torch.from_numpy(c.scales).cuda()
        b = None if c.bias is None else torch.from_numpy(c.bias).cuda()
        o = torch.full((c.M, c.N), float("nan"), device="cuda")
        dev.append((x, w, s, b, o))
    return dev


def _tuple(c, d, q):
    x, w, s, b, o = d
    return (x.data_ptr(), w.data_ptr(), s.data_ptr(), None if b is None else b.data_ptr(),
            o.data_ptr(), c.M, c.N, c.K, c.group_size,
            q.Q4LIN_SCALE_F16 if c.scale_f16 else q.Q4LIN_SCALE_F32)


def _check(cases, dev, x_shared=True):
    for c, d in zip(cases, dev):
        x = cases[0].x if x_shared else c.x
        out = d[4].cpu().numpy()
        ref, mag = oracle.linear(x, c.qweight, c.scales, c.bias, c.K, c.group_size)
        assert_parity(out, ref, mag, TOL_FP32)


@pytest.mark.parametrize("shapes", [
    [(2048, 2048), (512, 2048), (512, 2048)],          # q, k, v of a 1B layer
    [(8192, 2048), (8192, 2048)],                        # gate, up
    [(4096, 4096), (1024, 4096), (1024, 4096)],          # q, k, v of an 8B layer
    [(300, 1024), (77, 1024), (129, 1024), (64, 1024), (1000, 1024)],  # 5 > 4 per launch
])
def test_grouped_matches_oracle(handle, q, shapes):
    import torch
    cases = [synth.make_case(1, N, K, 32, scale_f16=True, bias=(i % 2 == 0), seed=50 + i)
             for i, (N, K) in enumerate(shapes)]
    dev = _problems(cases)
    st = q.q4lin_run_grouped(handle, [_tuple(c, d, q) for c, d in zip(cases, dev)],
                             torch.cuda.current_stream().cuda_stream)
    assert st == q.Q4LIN_OK
    torch.cuda.synchronize()
    _check(cases, dev)


def test_grouped_mixed_problems(handle, q):
    """Different K, M > 1 and per-channel problems in one call: runs are split."""
    import torch
    cases = [synth.make_case(1, 256, 1024, 32, scale_f16=True, bias=True, seed=60),
             synth.make_case(1, 128, 2048, 32, scale_f16=True, bias=False, seed=61),
             synth.make_case(5, 200, 512, 64, scale_f16=False, bias=True, seed=62),
             synth.make_case(1, 333, 4096, 4096, scale_f16=False, bias=False, seed=63)]
    dev = _problems(cases, x_shared=False)
    st = q.q4lin_run_grouped(handle, [_tuple(c, d, q) for c, d in zip(cases, dev)],
                             torch.cuda.current_stream().cuda_stream)
    assert st == q.Q4LIN_OK
    torch.cuda.synchronize()
    for c, d in zip(cases, dev):
        ref, mag = oracle.linear(c.x, c.qweight, c.scales, c.bias, c.K, c.group_size)
        tol = (4e-3, 1e-6) if c.M >= 4 else TOL_FP32
        assert_parity(d[4].cpu().numpy(), ref, mag, tol)


def test_grouped_aliasing_outputs_keep_sequential_semantics(handle, q):
    """Two problems writing the same out buffer must not be fused: the second wins."""
    import torch
    a = synth.make_case(1, 512, 2048, 32, scale_f16=True, seed=70)
    b = synth.make_case(1, 512, 2048, 32, scale_f16=True, seed=71)
    dev = _problems([a, b])
    shared_out = dev[0][4]
    ta = _tuple(a, dev[0], q)
    tb = list(_tuple(b, dev[1], q))
    tb[4] = shared_out.data_ptr()
    st = q.q4lin_run_grouped(handle, [ta, tuple(tb)], torch.cuda.current_stream().cuda_stream)
    assert st == q.Q4LIN_OK
    torch.cuda.synchronize()
    ref, mag = oracle.linear(a.x, b.qweight, b.scales, None, 2048, 32)
    assert_parity(shared_out.cpu().numpy(), ref, mag, TOL_FP32)


def test_grouped_validates_before_launching(handle, q):
    import torch
    cases = [synth.make_case(1, 256, 1024, 32, scale_f16=True, seed=80 + i) for i in range(3)]
    dev = _problems(cases)
    probs = [_tuple(c, d, q) for c, d in zip(cases, dev)]
    bad = list(probs[2])
    bad[7] = 0  # K == 0
    st = q.q4lin_run_grouped(handle, [probs[0], probs[1], tuple(bad)],
                             torch.cuda.current_stream().cuda_stream)
    assert st == q.Q4LIN_ERR_INVALID_ARG
    torch.cuda.synchronize()
    for d in dev:
        assert torch.isnan(d[4]).all(), "a problem ran although the call was rejected"
    assert q.q4lin_run_grouped(handle, [], None) == q.Q4LIN_OK
