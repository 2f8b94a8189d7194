/*
 * q4lin.h -- C ABI of the GB300 (sm_103a) 4-bit group-symmetric weight-quantized linear.
 *
 *   out[m,n] = bias[n] + sum_k x[m,k] * (nib(W)[n,k] - 8) * scale[k / group_size, n]
 *
 * Sources of the operation ("[ExecuTorch][WebGPU] ..." pull-request pages):
 *   - "Add linear_qcs4w op (et_vk.linear_qcs4w)", Solution and Constraints (2)-(4): the
 *     per-term formula in[m,k] * (unpack_int4(w) - 8) * scale, the grouped scale index
 *     (k / group_size) * N + n, the +8-shifted signed int4, the packed [N, K/2] uint8
 *     weight whose LOW nibble holds the even k (the q4gsw packer's "(odd << 4) | even"),
 *     the per-output-channel case (one scale per n, i.e. group_size = K), and the
 *     fail-loud argument guards (K_packed == ceil(K/2), enough scales).
 *   - "Add fp32 matmul ops ... (linear_q4gsw_backward)", #20943: dequant = (code - 8) *
 *     scale with [num_groups, N] scales; the K == 0 guard of the sibling ops.
 *   - "Add optimized linear_fp32 op", Implementation: the optional bias (a dummy binding
 *     when absent) added once in the epilogue, v = v + bias[n].
 *   - "Add 256-thread steel q4gsw prefill GEMM", Solution/Implementation: M = 1 routes to
 *     a GEMV, M > 1 to GEMM kernels chosen by a fail-closed eligibility check.
 *
 * Conventions for every entry point:
 *   - Every buffer is owned by the caller.  q4lin_run allocates nothing, never
 *     synchronizes the device and only enqueues kernels on the given stream.  A handle
 *     owns its options, a 4-byte device status word and 64 MiB of device scratch plus
 *     64 KiB of counters (partial sums of launches that split K or the rows across CTAs:
 *     decode GEMV, tensor-core GEMM, small-M tensor-core GEMM, input gradient; the fp16
 *     copy of x of the fp16 tensor-core path), all allocated by q4lin_create.
 *   - Status codes, never exceptions, aborts or prints.  Arguments are validated before
 *     any launch: a non-OK status from validation means nothing was enqueued.
 *   - All device pointers must be device-accessible memory of the handle's device.
 *   - The handle's scratch is shared by its calls: calls on one handle must be ordered on
 *     the GPU (one stream, or streams ordered by events).  Use one handle per stream for
 *     calls that run concurrently.  q4lin_set_option must not race with q4lin_run on the
 *     same handle.
 */
#ifndef Q4LIN_H
#define Q4LIN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define Q4LIN_API __attribute__((visibility("default")))
#else
#define Q4LIN_API
#endif

typedef struct q4lin_handle* q4lin_handle_t;

typedef enum {
    Q4LIN_OK = 0,
    Q4LIN_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment, overlap or option     */
    Q4LIN_ERR_UNSUPPORTED = 2, /* device is not sm_103, or a forced path cannot run   */
    Q4LIN_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed                 */
    Q4LIN_ERR_TIMEOUT = 4,     /* a bounded device-side wait gave up (see status word) */
    Q4LIN_ERR_NO_DEVICE = 5,   /* no CUDA device with that ordinal                     */
    Q4LIN_ERR_TOO_LARGE = 6    /* exceeds a fixed capacity (q4lin_run_static_scratch)  */
} q4lin_status_t;

/* Element type of the scales array. */
typedef enum { Q4LIN_SCALE_F32 = 0, Q4LIN_SCALE_F16 = 1 } q4lin_scale_dtype_t;

/* Kernel families.  AUTO picks by M and shape (measured crossover); the others force. */
typedef enum {
    Q4LIN_PATH_AUTO = 0,
    Q4LIN_PATH_GEMV = 1,    /* CUDA-core GEMV family: TMA-fed decode GEMV (M = 1),
                               TMA-fed multi-row GEMV (2 <= M <= 4, >= 10 M weights),
                               else the row-streaming kernel (small M)                */
    Q4LIN_PATH_FFMA = 2,    /* generic CUDA-core kernel: any K, group size, alignment  */
    Q4LIN_PATH_TC = 3,      /* tcgen05 tensor-core GEMM (TMEM accumulators)            */
    Q4LIN_PATH_TC_SMALL = 4 /* tcgen05 GEMM for 2 <= M <= 32 activation rows: persistent
                               CTAs over 128-row weight blocks, each weight read once,
                               x resident in shared memory or streamed for long K
                               (K % 32 == 0, 16-byte aligned x and qweight; grouped
                               scales: a power-of-two multiple of 32 as group size and a
                               scale row of whole 16-byte units); on fewer blocks
                               than half the SMs it splits K and adds the parts
                               through the handle's workspace (deterministic order);
                               tensor-core tolerance.  AUTO takes it for 3..32 rows
                               where it measured fastest (large matrices, and with
                               the K split most smaller ones from 5 rows) */
} q4lin_path_t;

/* Options for q4lin_set_option / q4lin_get_option. */
typedef enum {
    /* q4lin_path_t; default AUTO.  A forced path that cannot run the shape makes
     * q4lin_run return Q4LIN_ERR_UNSUPPORTED. */
    Q4LIN_OPT_FORCE_PATH = 1,
    /* 0 (default): the low nibble of byte j holds k = 2j (the q4gsw packer).
     * 1: the high nibble holds k = 2j (the qcs4w AOT packer's "(even << 4) | odd"
     * order, "Add linear_qcs4w op", Constraints (2)). */
    Q4LIN_OPT_NIBBLE_EVEN_HIGH = 2,
    /* Time limit, in nanoseconds of the GPU's global timer, of every bounded
     * device-side wait (mbarrier polls) of the TMA-fed kernels (decode and multi-row
     * GEMV, tensor-core GEMM, input gradient); <= 0 restores the default (2 s).  When a
     * wait runs out the kernel records code 1 in the handle's status word, stops issuing
     * work, lets its own copies (and MMAs) in flight finish, frees its tensor memory and
     * returns; its output is then undefined. */
    Q4LIN_OPT_WAIT_LIMIT = 3,
    /* 1: launch with programmatic dependent launch, so a kernel may start streaming
     * its weights while the previous kernel on the stream drains (default 0).  The
     * preceding kernel must not write this call's qweight or scales. */
    Q4LIN_OPT_PDL = 4,
    /* Test hook, default 0.  1: the tensor-core kernel's copy engine skips the first
     * pipeline stage, and the multi-row GEMV's copy engine issues nothing, so the barrier
     * their consumers wait on is never completed and their bounded waits run out
     * (exercises the timeout path without faulting the GPU). */
    Q4LIN_OPT_TC_SKIP_FIRST_COPY = 5,
    /* 1: the tensor-core GEMM multiplies fp16 operands (x and the dequantized weights
     * (code - 8) * scale rounded to IEEE binary16, fp32 accumulation: tcgen05.mma
     * kind::f16, twice the tf32 rate) instead of tf32 (default 0).  Each product carries a
     * relative error below 2^-10, inside the tensor-core path's 4e-3 * sum|x*w| bar.
     * Values outside the fp16 range (|x| >= 65520, or a scale with |scale| > 8188) make
     * the call record code 2 in the status word; its output is then undefined.  x is
     * first converted into the handle's scratch (M * K * 2 bytes); a problem whose copy
     * does not fit there runs in tf32. */
    Q4LIN_OPT_TC_F16 = 6,
    /* Operands of the small-M tensor-core GEMM (Q4LIN_PATH_TC_SMALL).  Up to 8 rows, with
     * x resident in shared memory, K > 256 and room for an even weight ring of >= 4 stages,
     * it can multiply bf16 operands: the dequantized weights rounded to bf16, and x as the
     * two bf16 terms bf16(x) and bf16(x - bf16(x)), taken by the same MMA as extra columns;
     * each product then carries a relative error below 2^-9 + 2^-16, inside the tensor-core
     * path's 4e-3 * sum|x*w| bar, and bf16 keeps fp32's exponent range.  0 (default): bf16
     * where it applies and the matrix has >= 100 blocks of 128 rows (measured faster there),
     * else tf32; 1: tf32 always; 2: bf16 wherever it applies. */
    Q4LIN_OPT_TC_SMALL_OPERANDS = 7
} q4lin_option_t;

/* Create a handle for CUDA device `device`.  Queries the SM count and shared-memory
 * limit and allocates the 4-byte device status word and the handle's scratch.  Q4LIN_ERR_NO_DEVICE if the
 * ordinal does not exist, Q4LIN_ERR_UNSUPPORTED if it is not compute capability 10.3.
 * The caller's current device is left unchanged. */
Q4LIN_API q4lin_status_t q4lin_create(q4lin_handle_t* handle, int device);

/* Release the handle, its status word and its scratch.  NULL is accepted (no-op). */
Q4LIN_API q4lin_status_t q4lin_destroy(q4lin_handle_t handle);

/* out = x @ dequant(W)^T (+ bias), enqueued on `stream` (a cudaStream_t; NULL = the
 * legacy default stream).
 *
 *   x        float32 [M, K], row-major, contiguous, 4-byte aligned.
 *   qweight  uint8 [N, ceil(K/2)], row-major: byte (n, j) holds codes for k = 2j and
 *            k = 2j+1 (low/high nibble by default, see Q4LIN_OPT_NIBBLE_EVEN_HIGH);
 *            signed weight = code - 8.  For odd K the last high nibble is never read.
 *   scales   [ceil(K / group_size), N] row-major, float32 (scale_dtype 0, 4-byte
 *            aligned) or IEEE binary16 (scale_dtype 1, 2-byte aligned).  Per-channel
 *            (qcs4w) weights use group_size = K with a [1, N] (= [N]) array.
 *   bias     float32 [N], 4-byte aligned, or NULL for no bias.
 *   out      float32 [M, N], row-major, 4-byte aligned; must not overlap any input.
 *   M >= 0, N >= 0, K >= 1, group_size >= 1.  M == 0 or N == 0 returns Q4LIN_OK and
 *   launches nothing; K == 0 is Q4LIN_ERR_INVALID_ARG.
 * Any K, group size and alignment beyond the element alignment above is accepted;
 * shapes a fast kernel cannot take run on a slower one (never an error under AUTO).
 * Accumulation is fp32.  Q4LIN_ERR_CUDA reports a failed launch
 * (cudaGetLastError after enqueueing). */
Q4LIN_API q4lin_status_t q4lin_run(q4lin_handle_t handle, const float* x,
                                   const uint8_t* qweight, const void* scales,
                                   const float* bias, float* out, int64_t M, int64_t N,
                                   int64_t K, int64_t group_size, int scale_dtype,
                                   void* stream);

/* One problem of q4lin_run_grouped: the arguments of one q4lin_run call. */
typedef struct q4lin_problem {
    const float* x;
    const uint8_t* qweight;
    const void* scales;
    const float* bias; /* may be NULL */
    float* out;
    int64_t M, N, K, group_size;
    int scale_dtype;
} q4lin_problem_t;

/* Run `count` problems on `stream`; the result is that of calling q4lin_run on each in
 * order.  Consecutive M = 1 problems that read the same x with the same K, group size and
 * scale dtype (for example the q, k and v projections of a decoder layer, or its gate
 * and up projections) run as one launch, up to 4 per launch, when none of their outputs
 * overlaps another problem's buffers; everything else runs one call at a time.  This is
 * the fused decode launch that the pages' MLC fusion passes produce before the GEMV
 * schedule ("dlight.gpu.GEMV" notice: "fusion passes -> LowBatchGemvSpecialize").
 * Every problem is validated before anything is enqueued (same rules and status codes
 * as q4lin_run); `problems` is read during the call only.  count == 0 is Q4LIN_OK. */
Q4LIN_API q4lin_status_t q4lin_run_grouped(q4lin_handle_t handle,
                                           const q4lin_problem_t* problems, int count,
                                           void* stream);

/* Decode GEMV (M = 1) for callers that cannot allocate device memory.
 *
 * No counterpart on the pages: this entry point exists for callers that may not call
 * cudaMalloc -- code that runs while a stream is being captured into a CUDA graph in a
 * mode that forbids allocation, code inside a custom allocator or memory pool (where
 * allocating would recurse), and real-time paths where an allocation's latency or
 * failure is not allowed.  Such callers cannot create a handle (q4lin_create allocates),
 * so this call needs none: it runs the same decode GEMV as q4lin_run with M = 1, whose
 * split-K partial sums and counters live in a fixed array of about 537 KB that the
 * library reserves in the device code image; every GPU that loads the library holds it
 * until the process exits.  Nothing is allocated: no cudaMalloc, cudaFree or allocating
 * library routine.
 *
 *   Arguments as q4lin_run with M = 1 (x is [K], out is [N]); default nibble order, no
 *   PDL.  N must be at most 16384: larger N returns Q4LIN_ERR_TOO_LARGE and runs nothing.
 *   Shapes the TMA-fed GEMV cannot take (K % 32 != 0, K < 512, N < 32, x or qweight not
 *   16-byte aligned, group_size neither a multiple of 32 nor >= K) return
 *   Q4LIN_ERR_UNSUPPORTED.
 *   The first call on a device looks up the array's device address (once per device, on
 *   the current device); make that first call before any stream capture.  A device reset
 *   (cudaDeviceReset) destroys the array with the context: the next call on that device
 *   sees the new context and looks the address up again, so after a reset, too, make the
 *   first call before any capture.
 *   Every call shares the array and it keeps the last call's contents: each call clears
 *   the counters it needs (an asynchronous memset on `stream`) before its kernel.  Calls
 *   that overlap on the GPU race on the array: order them (one stream, or events).
 *   A bounded device-side wait that runs out is not reported by this entry point (the
 *   output is then undefined); the kernel still returns. */
Q4LIN_API q4lin_status_t q4lin_run_static_scratch(const float* x, const uint8_t* qweight,
                                                  const void* scales, const float* bias,
                                                  float* out, int64_t N, int64_t K,
                                                  int64_t group_size, int scale_dtype,
                                                  void* stream);

/* Input gradient of the linear on the same packed weights (the frozen 4-bit base of
 * adapter training):
 *
 *   d_x[m,k] = sum_n d_out[m,n] * (nib(W)[n,k] - 8) * scale[k / group_size, n]
 *
 * "[ExecuTorch][WebGPU] Add fp32 matmul ops ... (linear_q4gsw_backward)", #20943:
 * d_x[M,K] = d_out[M,N] @ dequant(W)[N,K], contracting over N, with the forward's weight
 * and scale layout.
 *   d_out   device fp32 [M, N] row-major (4-byte aligned)
 *   qweight, scales, K, group_size, scale_dtype: exactly as q4lin_run (the handle's
 *           Q4LIN_OPT_NIBBLE_EVEN_HIGH applies)
 *   d_x     device fp32 [M, K] row-major (4-byte aligned); must not overlap any input
 * Summation order over n is not specified (fp32 accumulation; results within
 * 1e-5 * sum_n |d_out * w| + 1e-7 of the fp64 definition), but it is fixed for a given
 * shape: repeated calls give identical bits.  M == 0 is Q4LIN_OK (nothing runs); N == 0
 * writes zeros to d_x.  Uses the handle's workspace when the rows are split over CTAs
 * (calls on one handle must be ordered on the GPU).  Validated before anything is
 * enqueued; same status codes as q4lin_run. */
Q4LIN_API q4lin_status_t q4lin_run_backward_dx(q4lin_handle_t handle, const float* d_out,
                                               const uint8_t* qweight, const void* scales,
                                               float* d_x, int64_t M, int64_t N, int64_t K,
                                               int64_t group_size, int scale_dtype,
                                               void* stream);

/* Straight-through re-quantisation of fp32 latent weights to packed 4-bit codes with
 * frozen scales, in the layout q4lin_run reads:
 *
 *   code[n,k] = clamp(round(latent[n,k] / scale[k / group_size, n]), -8, 7) + 8
 *
 * "[ExecuTorch][WebGPU] Add fp32 matmul ops ... (q4gsw_requant)", #20945: a zero scale
 * gives code 8.  The quotient is the IEEE fp32 quotient, round() rounds half to even,
 * a NaN quotient gives code 8, and for odd K the padding nibble of each row's last byte
 * is 8.  Bit-exact (integer output).
 *   latent  device fp32 [N, K] row-major (4-byte aligned)
 *   scales  device fp32 or fp16 [ceil(K/group_size), N], as q4lin_run
 *   qweight device uint8 [N, ceil(K/2)] output (low nibble = even k, or swapped when the
 *           handle's Q4LIN_OPT_NIBBLE_EVEN_HIGH is set); must not overlap any input
 * N == 0 is Q4LIN_OK (nothing runs).  Validated before anything is enqueued. */
Q4LIN_API q4lin_status_t q4lin_run_requant(q4lin_handle_t handle, const float* latent,
                                           const void* scales, uint8_t* qweight, int64_t N,
                                           int64_t K, int64_t group_size, int scale_dtype,
                                           void* stream);

/* The path q4lin_run would take for these arguments (no launch, no device access);
 * *path_out receives a q4lin_path_t other than AUTO.  Same validation and status codes
 * as q4lin_run.  For M == 0 or N == 0, *path_out is Q4LIN_PATH_AUTO (nothing runs). */
Q4LIN_API q4lin_status_t q4lin_plan(q4lin_handle_t handle, const float* x,
                                    const uint8_t* qweight, const void* scales,
                                    const float* bias, const float* out, int64_t M,
                                    int64_t N, int64_t K, int64_t group_size,
                                    int scale_dtype, int* path_out);

/* Kernels behind the paths (what q4lin_plan_kernel reports). */
typedef enum {
    Q4LIN_KERNEL_NONE = 0,      /* M == 0 or N == 0: nothing runs                          */
    Q4LIN_KERNEL_GEMV_TMA = 1,  /* TMA-fed decode GEMV (M = 1)                             */
    Q4LIN_KERNEL_MULTIROW = 2,  /* TMA-fed multi-row GEMV (2 <= M <= 4)                    */
    Q4LIN_KERNEL_ROWSTREAM = 3, /* row-streaming CUDA-core kernel (small M)                */
    Q4LIN_KERNEL_GENERIC = 4,   /* generic CUDA-core kernel (any K, group size, alignment) */
    Q4LIN_KERNEL_TC = 5,        /* tcgen05 tensor-core GEMM, tf32 operands                 */
    Q4LIN_KERNEL_TC_F16 = 6,    /* the same with fp16 operands (Q4LIN_OPT_TC_F16)          */
    Q4LIN_KERNEL_GEMV_TMA_FIXED = 7, /* the decode GEMV with exact fixed-point arithmetic: x as
                                      * 32-bit fixed point per 32-k chunk, codes times x by
                                      * dp4a; chosen when its CTAs take >= 2 row blocks each */
    Q4LIN_KERNEL_TC_SMALL = 8,  /* tcgen05 GEMM for 2 <= M <= 32 (Q4LIN_PATH_TC_SMALL), tf32 */
    Q4LIN_KERNEL_TC_SMALL_BF16 = 9 /* the same with bf16 operands (up to 8 rows, see
                                    * Q4LIN_OPT_TC_SMALL_OPERANDS) */
} q4lin_kernel_t;

/* The kernel q4lin_run would launch for these arguments (no launch, no device access);
 * *kernel_out receives a q4lin_kernel_t.  Same arguments, validation and status codes as
 * q4lin_plan; for M == 0 or N == 0, *kernel_out is Q4LIN_KERNEL_NONE. */
Q4LIN_API q4lin_status_t q4lin_plan_kernel(q4lin_handle_t handle, const float* x,
                                           const uint8_t* qweight, const void* scales,
                                           const float* bias, const float* out, int64_t M,
                                           int64_t N, int64_t K, int64_t group_size,
                                           int scale_dtype, int* kernel_out);

/* Set / read one q4lin_option_t.  Q4LIN_ERR_INVALID_ARG for an unknown option or an
 * out-of-range value. */
Q4LIN_API q4lin_status_t q4lin_set_option(q4lin_handle_t handle, int option,
                                          int64_t value);
Q4LIN_API q4lin_status_t q4lin_get_option(q4lin_handle_t handle, int option,
                                          int64_t* value);

/* Read and clear the handle's device status word after synchronizing `stream`.
 * *code_out = 0 if no kernel recorded a problem since the last call; otherwise the
 * first recorded code (1 = a bounded device-side wait ran out; 2 = a value outside the
 * fp16 range on the fp16 tensor-core path).
 * The word is shared by every call on the handle.
 * Returns Q4LIN_ERR_TIMEOUT when the code is non-zero, Q4LIN_OK otherwise. */
Q4LIN_API q4lin_status_t q4lin_check_device_status(q4lin_handle_t handle, void* stream,
                                                   int* code_out);

/* Static, never-NULL description of a status code. */
Q4LIN_API const char* q4lin_status_string(q4lin_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* Q4LIN_H */
