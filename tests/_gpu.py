"""GPU-side helpers for the parity tests: run q4lin_run through the C ABI on a seeded
case, with the output NaN-poisoned and guard slots after the last element, and compare
with the fp64 oracle element by element."""
import numpy as np

GUARD = 64
SENTINEL = np.float32(12345.678)

# Per-element bars, |gpu - oracle| <= rel * sum_k |x * w| + abs.
TOL_FP32 = (1e-5, 1e-7)   # CUDA-core paths (fp32 FMA)
TOL_TC = (4e-3, 1e-6)     # tensor-core path (bf16 / tf32 operands, fp32 accumulate)


def device_case(case, device="cuda"):
    import torch
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(device)
    return t(case.x), t(case.qweight), t(case.scales), t(case.bias)


def run_q4lin(handle, case, path=0, even_high=False, x_dev=None):
    """Run one case through q4lin_run; returns (out [M,N] numpy, path used)."""
    import torch
    from bit_weight_quantized_int4_gb300 import q4lin as q
    x, w, s, b = device_case(case)
    if x_dev is not None:
        x = x_dev
    M, N, K, gs = case.M, case.N, case.K, case.group_size
    buf = torch.full((M * N + GUARD,), float("nan"), dtype=torch.float32, device="cuda")
    buf[M * N:] = float(SENTINEL)
    q.q4lin_set_option(handle, q.Q4LIN_OPT_FORCE_PATH, path)
    q.q4lin_set_option(handle, q.Q4LIN_OPT_NIBBLE_EVEN_HIGH, int(even_high))
    sd = q.Q4LIN_SCALE_F16 if case.scale_f16 else q.Q4LIN_SCALE_F32
    ptr = lambda a: None if a is None else a.data_ptr()
    st, used = q.q4lin_plan(handle, ptr(x), ptr(w), ptr(s), ptr(b), buf.data_ptr(), M, N, K,
                            gs, sd)
    assert st == q.Q4LIN_OK, q.q4lin_status_string(st)
    stream = torch.cuda.current_stream().cuda_stream
    st = q.q4lin_run(handle, ptr(x), ptr(w), ptr(s), ptr(b), buf.data_ptr(), M, N, K, gs,
                     sd, stream)
    assert st == q.Q4LIN_OK, q.q4lin_status_string(st)
    torch.cuda.synchronize()
    q.q4lin_set_option(handle, q.Q4LIN_OPT_FORCE_PATH, 0)
    q.q4lin_set_option(handle, q.Q4LIN_OPT_NIBBLE_EVEN_HIGH, 0)
    host = buf.cpu().numpy()
    assert np.all(host[M * N:] == SENTINEL), "write past the end of out"
    return host[:M * N].reshape(M, N), used


def assert_parity(out, ref, mag, tol):
    rel, ab = tol
    out64 = out.astype(np.float64)
    nan_ref = np.isnan(ref)
    assert np.array_equal(np.isnan(out64), nan_ref), "NaN positions differ (unwritten output?)"
    err = np.abs(out64 - ref)
    bound = rel * mag + ab
    bad = ~(err <= bound) & ~nan_ref
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{int(bad.sum())} of {bad.size} elements out of tolerance; first at {tuple(i)}: "
            f"gpu {out64[tuple(i)]!r} oracle {ref[tuple(i)]!r} bound {bound[tuple(i)]!r}")
    return float(np.max(err / np.maximum(bound, 1e-300))) if err.size else 0.0
