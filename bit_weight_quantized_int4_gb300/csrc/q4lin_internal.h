// Internal interface between the C-ABI host layer (q4lin.cpp) and the kernel files.
// Not installed; the public interface is include/q4lin.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace q4lin {

// Function attributes belong to the function's instance in one device's context: a kernel
// that needs more than 48 KiB of dynamic shared memory (or a carveout) gets them set once
// per device, on the first launch there (the caller has made the handle's device current).
// Thread-safe; concurrent first launches may both set them, which is harmless.
template <auto Kernel>
cudaError_t kernel_smem_once(int bytes, int carveout = -1) {
    static std::atomic<uint64_t> done{0};  // one bit per device ordinal < 64
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev >= 0 && dev < 64 ? (1ULL << dev) : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && carveout >= 0)
        e = cudaFuncSetAttribute(Kernel, cudaFuncAttributePreferredSharedMemoryCarveout, carveout);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
}

// cuTensorMapEncodeTiled of the driver, resolved once through the runtime (null when the
// driver does not provide it); used by every TMA-fed kernel to build its tensor maps.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder();

// One linear problem, already validated by the host layer.
struct Problem {
    const float* x;          // [M, K] fp32
    const uint8_t* qweight;  // [N, ceil(K/2)] packed codes
    const void* scales;      // [ceil(K/gs), N] fp32 or fp16
    const float* bias;       // [N] or nullptr
    float* out;              // [M, N] fp32
    int64_t M, N, K, group_size;
    int scale_f16;           // 1: binary16 scales, 0: fp32
    int even_high;           // 1: even k in the high nibble
};

// Per-launch context from the handle.
struct LaunchCtx {
    cudaStream_t stream;
    int sm_count;
    int max_smem_optin;      // bytes of opt-in shared memory per block
    int pdl;                 // launch with programmatic stream serialization
    int* status_word;        // device int, first nonzero code a kernel records
    int64_t wait_limit_ns;   // time limit of bounded device-side waits
    int tc_skip_first_copy;  // test hook: the TC producer skips stage 0
    int tc_f16 = 0;          // tensor-core GEMM with fp16 operands
    int tc_small_operands = 0;  // small-M GEMM: 0 auto, 1 tf32, 2 bf16 where it applies
    float* ws;               // scratch for split-K partial sums (may be null)
    int64_t ws_floats;
    int* tickets;            // per-row-block counters, zero between launches (may be null)
    int64_t ticket_count;
};

// Row-streaming CUDA-core kernel (decode GEMV, and small M with weight reuse across a
// tile of up to 4 activation rows).  Needs K % 32 == 0, 16-byte aligned x and qweight,
// and group_size % 32 == 0 or group_size >= K.
bool rowstream_eligible(const Problem& p);
cudaError_t rowstream_launch(const Problem& p, const LaunchCtx& c);

// Tiling of the TMA-fed decode GEMV that bounds its split-K scratch: row blocks of 16, 32
// or 64 rows, K split into at most 8 parts.  A launch that splits K uses parts x (row
// blocks x rows per block) partial sums and one counter per row block; a launch whose
// scratch does not fit the context's capacity does not split.
constexpr int kGemvMinRowBlock = 16;
constexpr int kGemvMaxRowBlock = 64;
constexpr int kGemvMaxParts = 8;

// TMA-fed decode GEMV (M = 1): persistent CTAs, a producer warp streams weight tiles
// into a shared-memory ring.  Needs K % 32 == 0, K >= 512, N >= 16, 16-byte aligned x and
// qweight, and group_size % 32 == 0 or group_size >= K.
bool gemv_tma_eligible(const Problem& p);
cudaError_t gemv_tma_launch(const Problem& p, const LaunchCtx& c);
// Whether gemv_tma_launch would run the problem with the exact fixed-point arithmetic (x
// as 32-bit fixed point per 32-k chunk, dp4a): when its CTAs process at least two row
// blocks each.
bool gemv_tma_fixed_point(const Problem& p, const LaunchCtx& c);
// Several eligible M = 1 problems that share x, K, group size, scale dtype and nibble
// order in one launch (at most gemv_tma_max_group()).
int gemv_tma_max_group();
bool gemv_tma_groupable(const Problem& a, const Problem& b);
cudaError_t gemv_tma_launch_group(const Problem* ps, int count, const LaunchCtx& c);

// TMA-fed GEMV for 2 <= M <= 4 activation rows: a producer warp streams the weight
// tile, its group scales and the x tile of each 512-k stage into a shared-memory ring;
// each widened code is used for all M rows.  Needs K % 32 == 0, K >= 512, N >= 16, a
// scale row of whole 16-byte units, 16-byte aligned x, qweight and scales, and a
// power-of-two group size that is a multiple of 32, or group_size >= K.
bool gemv_mr_eligible(const Problem& p);
cudaError_t gemv_mr_launch(const Problem& p, const LaunchCtx& c);

// Generic CUDA-core kernel: any K (odd included), any group size, any alignment.
cudaError_t generic_launch(const Problem& p, const LaunchCtx& c);

// Training-path problems on the same packed weights, validated by the host layer.
struct TrainProblem {  // d_x[M,K] = d_out[M,N] @ dequant(W)[N,K]
    const float* d_out;      // [M, N] fp32
    const uint8_t* qweight;  // [N, ceil(K/2)]
    const void* scales;      // [ceil(K/gs), N]
    float* d_x;              // [M, K] fp32
    int64_t M, N, K, group_size;
    int scale_f16, even_high;
};
struct RequantProblem {  // qweight[N, ceil(K/2)] = pack(clamp(round(latent / scale), -8, 7) + 8)
    const float* latent;  // [N, K] fp32
    const void* scales;   // [ceil(K/gs), N]
    uint8_t* qweight;     // [N, ceil(K/2)]
    int64_t N, K, group_size;
    int scale_f16, even_high;
};
cudaError_t backward_dx_launch(const TrainProblem& p, const LaunchCtx& c);
cudaError_t requant_launch(const RequantProblem& p, const LaunchCtx& c);

// tcgen05 tensor-core GEMM.  Eligibility and launch live in tc_gemm.cu.
bool tc_eligible(const Problem& p, const LaunchCtx& c);
// Whether tc_launch multiplies fp16 operands for this problem (the option is set and the
// fp16 copy of x fits the scratch).
bool tc_uses_f16(const Problem& p, const LaunchCtx& c);
cudaError_t tc_launch(const Problem& p, const LaunchCtx& c);

// tcgen05 GEMM for 2 <= M <= 32 activation rows (tc_small.cu): persistent CTAs over
// 128-row weight blocks, x resident in shared memory (or streamed for long K).  Needs
// K % 32 == 0, 16-byte aligned x and qweight, and for grouped scales a power-of-two
// multiple of 32 as group size with 16-byte aligned scale rows.
bool tc_small_eligible(const Problem& p, const LaunchCtx& c);
// Whether that kernel multiplies bf16 operands (up to 8 rows, x resident, K > 256; x
// split into bf16(x) and bf16(x - bf16(x)), the dequantized weights rounded to bf16)
// rather than tf32: by default from 100 row blocks, or as Q4LIN_OPT_TC_SMALL_OPERANDS says.
bool tc_small_uses_bf16(const Problem& p, const LaunchCtx& c);
// Parts of that kernel's K split (1: none): on matrices with fewer 128-row blocks than half
// the SMs, the largest of 2, 4 or 8 parts dividing the 256-k stages into runs of >= 2 whose
// items fit one wave, within the handle's split-K workspace and tickets.
int tc_small_parts(const Problem& p, const LaunchCtx& c);
cudaError_t tc_small_launch(const Problem& p, const LaunchCtx& c);

}  // namespace q4lin
