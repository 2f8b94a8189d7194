// q4lin.cpp -- C-ABI host layer: argument validation, path planning, dispatch, options.
//
// The guards mirror the fail-loud checks on the pages ("Add linear_qcs4w op",
// Implementation: packed row length ceil(K/2), enough scales; the K == 0 guard of the
// q4gsw training ops) and the "throw before any allocation" rule of "Add optimized
// linear_fp32 op": every check runs before anything is enqueued.  The path choice
// mirrors the pages' M-dispatch (M = 1 -> GEMV; M > 1 -> a GEMM chosen by a fail-closed
// eligibility test, "Add 256-thread steel q4gsw prefill GEMM") with a crossover measured
// on GB300 instead of shape thresholds.
#include "../../include/q4lin.h"

#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include <new>

#include "q4lin_internal.h"

struct q4lin_handle {
    int device = 0;
    int sm_count = 0;
    int max_smem_optin = 0;
    int force_path = Q4LIN_PATH_AUTO;
    int even_high = 0;
    int pdl = 0;
    int64_t wait_limit = 0;  // ns; 0: default
    int tc_skip_first_copy = 0;
    int tc_f16 = 0;
    int tc_small_operands = 0;
    int* d_status = nullptr;
    float* d_ws = nullptr;     // split-K partial sums
    int* d_tickets = nullptr;  // split-K row-block counters (zero between launches)
};

namespace {

constexpr int64_t kDefaultWaitLimit = 2000000000LL;  // 2 s of GPU global time
// Scratch of a handle: partial sums of split-K launches and their row-block counters.
constexpr int64_t kWsFloats = 1 << 24;   // 64 MiB (split-K partials; the fp16 copy of x)
constexpr int64_t kTickets = 1 << 14;    // 64 KiB

// M-dispatch between the CUDA-core kernels (the row-streaming kernel, which re-reads the
// weights for every 4 activation rows, so its time grows with M, and the TMA-fed multi-row
// GEMV for 2..4 rows) and the tensor-core GEMM (flat in M up to 64 rows).  Crossover table
// from a device-time sweep on GB300 (M = 1..512; N x K = 1000 x 2048, 2048 x 2048,
// 8192 x 2048, 2048 x 8192, 128256 x 2048, 4096 x 14336, 14336 x 4096; every launch on
// HBM-cold weights): the largest M for which the CUDA-core path is still faster, by the
// weight count N * K.
int64_t rowstream_max_m(const q4lin::Problem& p) {
    const double nk = (double)p.N * (double)p.K;
    if (nk < 3.0e6) return 16;
    if (nk < 8.0e6) return 8;
    return 4;
}

// For 2..4 rows the multi-row GEMV beats row streaming from about 10 M weights on (1.2x at
// 8192 x 2048, 1.7x at 128256 x 2048 and 4 rows); below that its fixed pipeline latency
// (~5 us) loses to row streaming (2048 x 2048: 6.2 against 4.3 us at 2 rows; 4096 x 2048:
// 6.5 against 6.0).
bool multirow_preferred(const q4lin::Problem& p) {
    return (double)p.N * (double)p.K >= 1.0e7 && q4lin::gemv_mr_eligible(p);
}

// 3..32 activation rows: the small-M tensor-core GEMM (one CTA per SM over 128-row weight
// blocks, each weight read once for all rows) where its blocks fill the SMs.  Its time is
// close to waves x stages of 256 k x ~1.05 us up to 16 rows (MMA width 16) and ~1.35 us
// above (width 32), flat in M (device time per launch on GB300, HBM-cold weights: 128256 x
// 2048 57 / 74 us, 28672 x 4096 33 / 43 us, 14336 x 4096 19 / 23 us, 8192 x 2048 9.1 /
// 12.0 us), against, at 3..4 rows, the multi-row GEMV (128256 x 2048: 66 / 79 us at 3 / 4
// rows; it stays ahead where a last wave of a few blocks doubles the small-M GEMM's time:
// 22016 x 4096 at 3 rows 27 against 33 us, and at 3 rows on less than one wave, 14336 x
// 4096 19.1 against 20.0) and, from 5 rows, the tile GEMM (128256 x 2048
// 111-115 us; above 16 rows it stays ahead on few blocks, 8192 x 2048 11.4 against 12.0 us).
// On fewer blocks than half the SMs the small-M GEMM splits K (see tc_small_parts): AUTO
// takes it at 5..8 rows from 4 M weights (8 rows: 4096 x 4096 9.5 against the tile GEMM's
// 11.8 us, 2048 x 8192 10.9 against 16.1, 2048 x 2048 6.1 against row streaming's 7.3), at
// 9..16 rows at any size (1000 x 2048 at 12 rows: 6.0 against 7.2), at 4 rows on long
// rows of >= 4096 rows (4096 x 14336: 19.7 against the multi-row GEMV's 21.9; within 5 %
// either way on shorter rows, and behind on 2048 x 8192, 10.9 against 10.5); above 16
// rows the split is within a few per cent of the tile GEMM either way (2048 x 8192 at 24
// rows 17.1 against 16.2; 2048 x 2048 10.2 against 7.3) and AUTO keeps the tile GEMM.  Two
// rows stay with the multi-row GEMV (50.5 against 57 us on 128256 x 2048).
bool tc_small_preferred(const q4lin::Problem& p, const q4lin::LaunchCtx& c) {
    if (p.M < 3 || p.M > 32 || !q4lin::tc_small_eligible(p, c)) return false;
    const int64_t blocks = (p.N + 127) / 128, sms = c.sm_count;
    const int64_t stages = (p.K + 255) / 256, tail = blocks % sms;
    const bool split = q4lin::tc_small_parts(p, c) > 1;
    if (p.M <= 4)
        return (blocks >= (p.M == 3 ? sms : 100) && (tail == 0 || 4 * tail > sms)) ||
               (p.M == 4 && split && p.N >= 4096 && p.K >= 8192);
    if (p.M <= 16)
        return blocks >= 100 || (stages <= 8 && blocks >= 40) ||
               (split && (p.M > 8 || p.N * p.K >= (4LL << 20)));
    return blocks >= 100;
}

class DeviceGuard {
   public:
    explicit DeviceGuard(int device) {
        if (cudaGetDevice(&prev_) != cudaSuccess) prev_ = -1;
        if (prev_ != device) ok_ = cudaSetDevice(device) == cudaSuccess;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev_ >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev_) cudaSetDevice(prev_);
    }
    bool ok() const { return ok_; }

   private:
    int prev_ = -1;
    bool ok_ = true;
};

bool mul_ok(int64_t a, int64_t b, int64_t* r) { return !__builtin_mul_overflow(a, b, r); }

bool overlaps(const void* a, int64_t abytes, const void* b, int64_t bbytes) {
    if (!a || !b || abytes <= 0 || bbytes <= 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + (uintptr_t)bbytes && b0 < a0 + (uintptr_t)abytes;
}

// Validation shared by q4lin_run and q4lin_plan.  On success fills `p` (except the
// out pointer for plan) and returns Q4LIN_OK; M == 0 or N == 0 is reported via *empty.
q4lin_status_t validate(q4lin_handle_t h, const float* x, const uint8_t* qweight,
                        const void* scales, const float* bias, const void* out, int64_t M,
                        int64_t N, int64_t K, int64_t group_size, int scale_dtype,
                        q4lin::Problem* p, bool* empty) {
    if (!h) return Q4LIN_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 1 || group_size < 1) return Q4LIN_ERR_INVALID_ARG;
    if (scale_dtype != Q4LIN_SCALE_F32 && scale_dtype != Q4LIN_SCALE_F16)
        return Q4LIN_ERR_INVALID_ARG;
    *empty = (M == 0 || N == 0);
    if (*empty) return Q4LIN_OK;
    if (!x || !qweight || !scales || !out) return Q4LIN_ERR_INVALID_ARG;
    const int64_t esize = scale_dtype == Q4LIN_SCALE_F16 ? 2 : 4;
    const int64_t Kp = (K + 1) / 2;
    const int64_t G = (K + group_size - 1) / group_size;
    int64_t xb, wb, sb, ob, t;
    if (!mul_ok(M, K, &t) || !mul_ok(t, 4, &xb)) return Q4LIN_ERR_INVALID_ARG;
    if (!mul_ok(N, Kp, &wb)) return Q4LIN_ERR_INVALID_ARG;
    if (!mul_ok(G, N, &t) || !mul_ok(t, esize, &sb)) return Q4LIN_ERR_INVALID_ARG;
    if (!mul_ok(M, N, &t) || !mul_ok(t, 4, &ob)) return Q4LIN_ERR_INVALID_ARG;
    const int64_t bb = bias ? N * 4 : 0;
    // Element alignment.
    if (reinterpret_cast<uintptr_t>(x) % 4 || reinterpret_cast<uintptr_t>(out) % 4 ||
        (bias && reinterpret_cast<uintptr_t>(bias) % 4) ||
        reinterpret_cast<uintptr_t>(scales) % esize)
        return Q4LIN_ERR_INVALID_ARG;
    // The output must not alias any input.
    if (overlaps(out, ob, x, xb) || overlaps(out, ob, qweight, wb) ||
        overlaps(out, ob, scales, sb) || overlaps(out, ob, bias, bb))
        return Q4LIN_ERR_INVALID_ARG;
    p->x = x;
    p->qweight = qweight;
    p->scales = scales;
    p->bias = bias;
    p->out = static_cast<float*>(const_cast<void*>(out));
    p->M = M;
    p->N = N;
    p->K = K;
    p->group_size = group_size;
    p->scale_f16 = scale_dtype == Q4LIN_SCALE_F16;
    p->even_high = h->even_high;
    return Q4LIN_OK;
}

q4lin::LaunchCtx make_ctx(q4lin_handle_t h, cudaStream_t stream) {
    q4lin::LaunchCtx c;
    c.stream = stream;
    c.sm_count = h->sm_count;
    c.max_smem_optin = h->max_smem_optin;
    c.pdl = h->pdl;
    c.status_word = h->d_status;
    c.wait_limit_ns = h->wait_limit > 0 ? h->wait_limit : kDefaultWaitLimit;
    c.tc_skip_first_copy = h->tc_skip_first_copy;
    c.tc_f16 = h->tc_f16;
    c.tc_small_operands = h->tc_small_operands;
    c.ws = h->d_ws;
    c.ws_floats = kWsFloats;
    c.tickets = h->d_tickets;
    c.ticket_count = kTickets;
    return c;
}

// Which kernel family runs the problem.
q4lin_status_t plan(q4lin_handle_t h, const q4lin::Problem& p, const q4lin::LaunchCtx& c,
                    int* path) {
    const bool row_ok = q4lin::rowstream_eligible(p);
    switch (h->force_path) {
        case Q4LIN_PATH_GEMV:
            if (!row_ok) return Q4LIN_ERR_UNSUPPORTED;
            *path = Q4LIN_PATH_GEMV;
            return Q4LIN_OK;
        case Q4LIN_PATH_FFMA:
            *path = Q4LIN_PATH_FFMA;
            return Q4LIN_OK;
        case Q4LIN_PATH_TC:
            if (!q4lin::tc_eligible(p, c)) return Q4LIN_ERR_UNSUPPORTED;
            *path = Q4LIN_PATH_TC;
            return Q4LIN_OK;
        case Q4LIN_PATH_TC_SMALL:
            if (!q4lin::tc_small_eligible(p, c)) return Q4LIN_ERR_UNSUPPORTED;
            *path = Q4LIN_PATH_TC_SMALL;
            return Q4LIN_OK;
        default:
            break;
    }
    if (tc_small_preferred(p, c)) {
        *path = Q4LIN_PATH_TC_SMALL;
    } else if (p.M > 1 && q4lin::tc_eligible(p, c) && (!row_ok || p.M > rowstream_max_m(p))) {
        *path = Q4LIN_PATH_TC;
    } else if (row_ok) {
        *path = Q4LIN_PATH_GEMV;
    } else {
        *path = Q4LIN_PATH_FFMA;
    }
    return Q4LIN_OK;
}

// The kernel behind a path for an M >= 1, N >= 1 problem (the dispatch of q4lin_run).
int kernel_of(const q4lin::Problem& p, const q4lin::LaunchCtx& c, int path) {
    switch (path) {
        case Q4LIN_PATH_TC: return q4lin::tc_uses_f16(p, c) ? Q4LIN_KERNEL_TC_F16 : Q4LIN_KERNEL_TC;
        case Q4LIN_PATH_TC_SMALL:
            return q4lin::tc_small_uses_bf16(p, c) ? Q4LIN_KERNEL_TC_SMALL_BF16 : Q4LIN_KERNEL_TC_SMALL;
        case Q4LIN_PATH_GEMV:
            if (q4lin::gemv_tma_eligible(p))
                return q4lin::gemv_tma_fixed_point(p, c) ? Q4LIN_KERNEL_GEMV_TMA_FIXED
                                                         : Q4LIN_KERNEL_GEMV_TMA;
            return multirow_preferred(p) ? Q4LIN_KERNEL_MULTIROW : Q4LIN_KERNEL_ROWSTREAM;
        default: return Q4LIN_KERNEL_GENERIC;
    }
}

}  // namespace

extern "C" {

q4lin_status_t q4lin_create(q4lin_handle_t* handle, int device) {
    if (!handle) return Q4LIN_ERR_INVALID_ARG;
    *handle = nullptr;
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess || device < 0 || device >= count) {
        cudaGetLastError();
        return Q4LIN_ERR_NO_DEVICE;
    }
    int major = 0, minor = 0, sms = 0, smem = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) !=
            cudaSuccess)
        return Q4LIN_ERR_CUDA;
    if (major != 10 || minor != 3) return Q4LIN_ERR_UNSUPPORTED;
    q4lin_handle* h = new (std::nothrow) q4lin_handle();
    if (!h) return Q4LIN_ERR_CUDA;
    h->device = device;
    h->sm_count = sms;
    h->max_smem_optin = smem;
    {
        DeviceGuard g(device);
        if (!g.ok() || cudaMalloc(&h->d_status, sizeof(int)) != cudaSuccess ||
            cudaMemset(h->d_status, 0, sizeof(int)) != cudaSuccess ||
            cudaMalloc(&h->d_ws, kWsFloats * sizeof(float)) != cudaSuccess ||
            cudaMalloc(&h->d_tickets, kTickets * sizeof(int)) != cudaSuccess ||
            cudaMemset(h->d_tickets, 0, kTickets * sizeof(int)) != cudaSuccess ||
            cudaDeviceSynchronize() != cudaSuccess) {
            if (h->d_status) cudaFree(h->d_status);
            if (h->d_ws) cudaFree(h->d_ws);
            if (h->d_tickets) cudaFree(h->d_tickets);
            delete h;
            return Q4LIN_ERR_CUDA;
        }
    }
    *handle = h;
    return Q4LIN_OK;
}

q4lin_status_t q4lin_destroy(q4lin_handle_t h) {
    if (!h) return Q4LIN_OK;
    {
        DeviceGuard g(h->device);
        if (h->d_status) cudaFree(h->d_status);
        if (h->d_ws) cudaFree(h->d_ws);
        if (h->d_tickets) cudaFree(h->d_tickets);
    }
    delete h;
    return Q4LIN_OK;
}

q4lin_status_t q4lin_plan(q4lin_handle_t h, const float* x, const uint8_t* qweight,
                          const void* scales, const float* bias, const float* out,
                          int64_t M, int64_t N, int64_t K, int64_t group_size,
                          int scale_dtype, int* path_out) {
    if (!path_out) return Q4LIN_ERR_INVALID_ARG;
    q4lin::Problem p;
    bool empty = false;
    q4lin_status_t st = validate(h, x, qweight, scales, bias, out, M, N, K, group_size,
                                 scale_dtype, &p, &empty);
    if (st != Q4LIN_OK) return st;
    if (empty) {
        *path_out = Q4LIN_PATH_AUTO;
        return Q4LIN_OK;
    }
    return plan(h, p, make_ctx(h, nullptr), path_out);
}

q4lin_status_t q4lin_plan_kernel(q4lin_handle_t h, const float* x, const uint8_t* qweight,
                                 const void* scales, const float* bias, const float* out,
                                 int64_t M, int64_t N, int64_t K, int64_t group_size,
                                 int scale_dtype, int* kernel_out) {
    if (!kernel_out) return Q4LIN_ERR_INVALID_ARG;
    q4lin::Problem p;
    bool empty = false;
    q4lin_status_t st = validate(h, x, qweight, scales, bias, out, M, N, K, group_size,
                                 scale_dtype, &p, &empty);
    if (st != Q4LIN_OK) return st;
    if (empty) {
        *kernel_out = Q4LIN_KERNEL_NONE;
        return Q4LIN_OK;
    }
    int path = 0;
    const q4lin::LaunchCtx c = make_ctx(h, nullptr);
    st = plan(h, p, c, &path);
    if (st != Q4LIN_OK) return st;
    *kernel_out = kernel_of(p, c, path);
    return Q4LIN_OK;
}

q4lin_status_t q4lin_run(q4lin_handle_t h, const float* x, const uint8_t* qweight,
                         const void* scales, const float* bias, float* out, int64_t M,
                         int64_t N, int64_t K, int64_t group_size, int scale_dtype,
                         void* stream) {
    q4lin::Problem p;
    bool empty = false;
    q4lin_status_t st = validate(h, x, qweight, scales, bias, out, M, N, K, group_size,
                                 scale_dtype, &p, &empty);
    if (st != Q4LIN_OK || empty) return st;
    const q4lin::LaunchCtx c = make_ctx(h, static_cast<cudaStream_t>(stream));
    int path = 0;
    st = plan(h, p, c, &path);
    if (st != Q4LIN_OK) return st;
    DeviceGuard g(h->device);
    if (!g.ok()) return Q4LIN_ERR_CUDA;
    cudaError_t err;
    switch (kernel_of(p, c, path)) {
        case Q4LIN_KERNEL_TC:
        case Q4LIN_KERNEL_TC_F16: err = q4lin::tc_launch(p, c); break;
        case Q4LIN_KERNEL_TC_SMALL:
        case Q4LIN_KERNEL_TC_SMALL_BF16: err = q4lin::tc_small_launch(p, c); break;
        case Q4LIN_KERNEL_GEMV_TMA:
        case Q4LIN_KERNEL_GEMV_TMA_FIXED: err = q4lin::gemv_tma_launch(p, c); break;
        case Q4LIN_KERNEL_MULTIROW: err = q4lin::gemv_mr_launch(p, c); break;
        case Q4LIN_KERNEL_ROWSTREAM: err = q4lin::rowstream_launch(p, c); break;
        default: err = q4lin::generic_launch(p, c); break;
    }
    if (err == cudaSuccess) err = cudaGetLastError();
    return err == cudaSuccess ? Q4LIN_OK : Q4LIN_ERR_CUDA;
}

q4lin_status_t q4lin_run_grouped(q4lin_handle_t h, const q4lin_problem_t* problems, int count,
                                 void* stream) {
    if (!h || count < 0 || (count > 0 && !problems)) return Q4LIN_ERR_INVALID_ARG;
    if (count == 0) return Q4LIN_OK;
    constexpr int kMax = 4;
    q4lin::Problem ps[kMax];
    const q4lin::LaunchCtx c = make_ctx(h, static_cast<cudaStream_t>(stream));
    // Validate everything first: an error means nothing was enqueued.
    for (int i = 0; i < count; ++i) {
        const q4lin_problem_t& q = problems[i];
        q4lin::Problem p;
        bool empty = false;
        q4lin_status_t st = validate(h, q.x, q.qweight, q.scales, q.bias, q.out, q.M, q.N, q.K,
                                     q.group_size, q.scale_dtype, &p, &empty);
        if (st != Q4LIN_OK) return st;
        int path = 0;
        if (!empty && (st = plan(h, p, c, &path)) != Q4LIN_OK) return st;
    }
    DeviceGuard g(h->device);
    if (!g.ok()) return Q4LIN_ERR_CUDA;
    const bool gemv_forced_off = h->force_path == Q4LIN_PATH_FFMA ||
                                 h->force_path == Q4LIN_PATH_TC ||
                                 h->force_path == Q4LIN_PATH_TC_SMALL;
    int i = 0;
    while (i < count) {
        // Gather a run of fusable problems starting at i.
        int n = 0;
        bool empty = false;
        const q4lin_problem_t* q = &problems[i];
        validate(h, q->x, q->qweight, q->scales, q->bias, q->out, q->M, q->N, q->K,
                 q->group_size, q->scale_dtype, &ps[0], &empty);
        if (!empty && !gemv_forced_off && q4lin::gemv_tma_eligible(ps[0])) {
            n = 1;
            while (n < kMax && n < q4lin::gemv_tma_max_group() && i + n < count) {
                const q4lin_problem_t& r = problems[i + n];
                q4lin::Problem pr;
                bool e2 = false;
                validate(h, r.x, r.qweight, r.scales, r.bias, r.out, r.M, r.N, r.K, r.group_size,
                         r.scale_dtype, &pr, &e2);
                if (e2 || !q4lin::gemv_tma_eligible(pr) || !q4lin::gemv_tma_groupable(ps[0], pr))
                    break;
                // Fused problems run concurrently: no output may touch another's buffers.
                bool clash = false;
                for (int k = 0; k < n && !clash; ++k) {
                    const int64_t ob_new = pr.N * 4, ob_old = ps[k].N * 4;
                    const int64_t es = pr.scale_f16 ? 2 : 4;
                    const int64_t G = (pr.K + pr.group_size - 1) / pr.group_size;
                    clash = overlaps(pr.out, ob_new, ps[k].out, ob_old) ||
                            overlaps(pr.out, ob_new, ps[k].qweight, ps[k].N * (ps[k].K / 2)) ||
                            overlaps(pr.out, ob_new, ps[k].scales, G * ps[k].N * es) ||
                            overlaps(pr.out, ob_new, ps[k].bias, ps[k].bias ? ob_old : 0) ||
                            overlaps(ps[k].out, ob_old, pr.qweight, pr.N * (pr.K / 2)) ||
                            overlaps(ps[k].out, ob_old, pr.scales, G * pr.N * es) ||
                            overlaps(ps[k].out, ob_old, pr.bias, pr.bias ? ob_new : 0);
                }
                if (clash) break;
                ps[n++] = pr;
            }
        }
        cudaError_t err = cudaSuccess;
        if (n >= 2) {
            err = q4lin::gemv_tma_launch_group(ps, n, c);
            i += n;
        } else {
            err = cudaSuccess;
            q4lin_status_t st = q4lin_run(h, q->x, q->qweight, q->scales, q->bias, q->out, q->M,
                                          q->N, q->K, q->group_size, q->scale_dtype, stream);
            if (st != Q4LIN_OK) return st;
            ++i;
        }
        if (err == cudaSuccess) err = cudaGetLastError();
        if (err != cudaSuccess) return Q4LIN_ERR_CUDA;
    }
    return Q4LIN_OK;
}

q4lin_status_t q4lin_run_backward_dx(q4lin_handle_t h, const float* d_out,
                                     const uint8_t* qweight, const void* scales, float* d_x,
                                     int64_t M, int64_t N, int64_t K, int64_t group_size,
                                     int scale_dtype, void* stream) {
    if (!h) return Q4LIN_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 1 || group_size < 1) return Q4LIN_ERR_INVALID_ARG;
    if (scale_dtype != Q4LIN_SCALE_F32 && scale_dtype != Q4LIN_SCALE_F16)
        return Q4LIN_ERR_INVALID_ARG;
    if (M == 0) return Q4LIN_OK;
    if (!d_x || (N > 0 && (!d_out || !qweight || !scales))) return Q4LIN_ERR_INVALID_ARG;
    const int64_t esize = scale_dtype == Q4LIN_SCALE_F16 ? 2 : 4;
    const int64_t Kp = (K + 1) / 2;
    const int64_t G = (K + group_size - 1) / group_size;
    int64_t db, wb, sb, xb, t;
    if (!mul_ok(M, N, &t) || !mul_ok(t, 4, &db)) return Q4LIN_ERR_INVALID_ARG;
    if (!mul_ok(N, Kp, &wb)) return Q4LIN_ERR_INVALID_ARG;
    if (!mul_ok(G, N, &t) || !mul_ok(t, esize, &sb)) return Q4LIN_ERR_INVALID_ARG;
    if (!mul_ok(M, K, &t) || !mul_ok(t, 4, &xb)) return Q4LIN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(d_x) % 4 || (d_out && reinterpret_cast<uintptr_t>(d_out) % 4) ||
        (scales && reinterpret_cast<uintptr_t>(scales) % esize))
        return Q4LIN_ERR_INVALID_ARG;
    if (overlaps(d_x, xb, d_out, db) || overlaps(d_x, xb, qweight, wb) ||
        overlaps(d_x, xb, scales, sb))
        return Q4LIN_ERR_INVALID_ARG;
    const q4lin::LaunchCtx c = make_ctx(h, static_cast<cudaStream_t>(stream));
    DeviceGuard g(h->device);
    if (!g.ok()) return Q4LIN_ERR_CUDA;
    cudaError_t err;
    if (N == 0) {
        err = cudaMemsetAsync(d_x, 0, (size_t)xb, c.stream);
    } else {
        q4lin::TrainProblem p;
        p.d_out = d_out;
        p.qweight = qweight;
        p.scales = scales;
        p.d_x = d_x;
        p.M = M;
        p.N = N;
        p.K = K;
        p.group_size = group_size;
        p.scale_f16 = scale_dtype == Q4LIN_SCALE_F16;
        p.even_high = h->even_high;
        err = q4lin::backward_dx_launch(p, c);
    }
    if (err == cudaSuccess) err = cudaGetLastError();
    return err == cudaSuccess ? Q4LIN_OK : Q4LIN_ERR_CUDA;
}

q4lin_status_t q4lin_run_requant(q4lin_handle_t h, const float* latent, const void* scales,
                                 uint8_t* qweight, int64_t N, int64_t K, int64_t group_size,
                                 int scale_dtype, void* stream) {
    if (!h) return Q4LIN_ERR_INVALID_ARG;
    if (N < 0 || K < 1 || group_size < 1) return Q4LIN_ERR_INVALID_ARG;
    if (scale_dtype != Q4LIN_SCALE_F32 && scale_dtype != Q4LIN_SCALE_F16)
        return Q4LIN_ERR_INVALID_ARG;
    if (N == 0) return Q4LIN_OK;
    if (!latent || !scales || !qweight) return Q4LIN_ERR_INVALID_ARG;
    const int64_t esize = scale_dtype == Q4LIN_SCALE_F16 ? 2 : 4;
    const int64_t Kp = (K + 1) / 2;
    const int64_t G = (K + group_size - 1) / group_size;
    int64_t lb, wb, sb, t;
    if (!mul_ok(N, K, &t) || !mul_ok(t, 4, &lb)) return Q4LIN_ERR_INVALID_ARG;
    if (!mul_ok(N, Kp, &wb)) return Q4LIN_ERR_INVALID_ARG;
    if (!mul_ok(G, N, &t) || !mul_ok(t, esize, &sb)) return Q4LIN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(latent) % 4 || reinterpret_cast<uintptr_t>(scales) % esize)
        return Q4LIN_ERR_INVALID_ARG;
    if (overlaps(qweight, wb, latent, lb) || overlaps(qweight, wb, scales, sb))
        return Q4LIN_ERR_INVALID_ARG;
    const q4lin::LaunchCtx c = make_ctx(h, static_cast<cudaStream_t>(stream));
    DeviceGuard g(h->device);
    if (!g.ok()) return Q4LIN_ERR_CUDA;
    q4lin::RequantProblem p;
    p.latent = latent;
    p.scales = scales;
    p.qweight = qweight;
    p.N = N;
    p.K = K;
    p.group_size = group_size;
    p.scale_f16 = scale_dtype == Q4LIN_SCALE_F16;
    p.even_high = h->even_high;
    cudaError_t err = q4lin::requant_launch(p, c);
    if (err == cudaSuccess) err = cudaGetLastError();
    return err == cudaSuccess ? Q4LIN_OK : Q4LIN_ERR_CUDA;
}

q4lin_status_t q4lin_set_option(q4lin_handle_t h, int option, int64_t value) {
    if (!h) return Q4LIN_ERR_INVALID_ARG;
    switch (option) {
        case Q4LIN_OPT_FORCE_PATH:
            if (value < Q4LIN_PATH_AUTO || value > Q4LIN_PATH_TC_SMALL) return Q4LIN_ERR_INVALID_ARG;
            h->force_path = (int)value;
            return Q4LIN_OK;
        case Q4LIN_OPT_NIBBLE_EVEN_HIGH:
            if (value != 0 && value != 1) return Q4LIN_ERR_INVALID_ARG;
            h->even_high = (int)value;
            return Q4LIN_OK;
        case Q4LIN_OPT_WAIT_LIMIT:
            h->wait_limit = value > 0 ? value : 0;
            return Q4LIN_OK;
        case Q4LIN_OPT_PDL:
            if (value != 0 && value != 1) return Q4LIN_ERR_INVALID_ARG;
            h->pdl = (int)value;
            return Q4LIN_OK;
        case Q4LIN_OPT_TC_SKIP_FIRST_COPY:
            if (value != 0 && value != 1) return Q4LIN_ERR_INVALID_ARG;
            h->tc_skip_first_copy = (int)value;
            return Q4LIN_OK;
        case Q4LIN_OPT_TC_F16:
            if (value != 0 && value != 1) return Q4LIN_ERR_INVALID_ARG;
            h->tc_f16 = (int)value;
            return Q4LIN_OK;
        case Q4LIN_OPT_TC_SMALL_OPERANDS:
            if (value < 0 || value > 2) return Q4LIN_ERR_INVALID_ARG;
            h->tc_small_operands = (int)value;
            return Q4LIN_OK;
        default:
            return Q4LIN_ERR_INVALID_ARG;
    }
}

q4lin_status_t q4lin_get_option(q4lin_handle_t h, int option, int64_t* value) {
    if (!h || !value) return Q4LIN_ERR_INVALID_ARG;
    switch (option) {
        case Q4LIN_OPT_FORCE_PATH: *value = h->force_path; return Q4LIN_OK;
        case Q4LIN_OPT_NIBBLE_EVEN_HIGH: *value = h->even_high; return Q4LIN_OK;
        case Q4LIN_OPT_WAIT_LIMIT:
            *value = h->wait_limit > 0 ? h->wait_limit : kDefaultWaitLimit;
            return Q4LIN_OK;
        case Q4LIN_OPT_PDL: *value = h->pdl; return Q4LIN_OK;
        case Q4LIN_OPT_TC_SKIP_FIRST_COPY: *value = h->tc_skip_first_copy; return Q4LIN_OK;
        case Q4LIN_OPT_TC_F16: *value = h->tc_f16; return Q4LIN_OK;
        case Q4LIN_OPT_TC_SMALL_OPERANDS: *value = h->tc_small_operands; return Q4LIN_OK;
        default: return Q4LIN_ERR_INVALID_ARG;
    }
}

q4lin_status_t q4lin_check_device_status(q4lin_handle_t h, void* stream, int* code_out) {
    if (!h || !code_out) return Q4LIN_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    if (!g.ok()) return Q4LIN_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int code = 0;
    if (cudaMemcpyAsync(&code, h->d_status, sizeof(int), cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaMemsetAsync(h->d_status, 0, sizeof(int), s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return Q4LIN_ERR_CUDA;
    *code_out = code;
    return code ? Q4LIN_ERR_TIMEOUT : Q4LIN_OK;
}

const char* q4lin_status_string(q4lin_status_t s) {
    switch (s) {
        case Q4LIN_OK: return "ok";
        case Q4LIN_ERR_INVALID_ARG: return "invalid argument";
        case Q4LIN_ERR_UNSUPPORTED: return "unsupported device or forced path";
        case Q4LIN_ERR_CUDA: return "CUDA error";
        case Q4LIN_ERR_TIMEOUT: return "device-side bounded wait ran out";
        case Q4LIN_ERR_NO_DEVICE: return "no such CUDA device";
        case Q4LIN_ERR_TOO_LARGE: return "problem exceeds a fixed capacity";
        default: return "unknown status";
    }
}

}  // extern "C"
