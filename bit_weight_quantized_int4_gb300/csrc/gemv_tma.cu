// gemv_tma.cu -- TMA-fed decode GEMV (M = 1) of the 4-bit weight-quantized linear.
//
//   out[n] = bias[n] + sum_g s[g,n] * sum_{k in g} x[k] * (code[n,k] - 8)
//
// (formula: "[ExecuTorch][WebGPU] Add linear_qcs4w op", Solution; the decode GEMV is the
// regime of the TVM "dlight.gpu.GEMV" WebGPU notice, whose lesson -- several rows per
// workgroup, a short reduction per row, and a predicated final store for a ragged vocab
// such as 128257 -- is kept here.)
//
// HBM-bound: every packed byte is read exactly once.  The design decouples the memory
// stream from the arithmetic:
//   producer warp (one lane): 2D TMA copies of weight tiles [rb rows x 256 bytes]
//     (= 512 k per row) into a 4-stage shared-memory ring, one mbarrier per stage.  The
//     copies are long contiguous row segments, so DRAM sees streaming reads; the ring
//     keeps up to 4 tiles (up to 128 KiB) in flight per SM without spending registers.
//   16 consumer warps (512 threads, 4 per SM sub-partition, enough to keep the issue
//     slots busy): thread = (chunk lane j in 0..15, row group r0); per tile it widens the
//     32 codes of chunk j of each of its V = rb/32 rows and dots them with the x chunk
//     (read once per tile from shared memory, where x is staged in padded 32-float chunks,
//     and reused across the V rows), scaling each 32-value chunk by its group scale; the
//     scales are fetched two tiles ahead.  A warp reads 512 contiguous bytes of the tile
//     per load (conflict-free).  Partial sums stay in registers across the whole row; the
//     16 chunk lanes of a row group are reduced with shuffles once per row block.
// The CTAs are persistent and walk row blocks; the pipeline runs across block boundaries.
// With programmatic dependent launch the producer starts streaming weights before the
// preceding kernel on the stream has finished; x, bias and out are touched only after
// griddepcontrol.wait.  Waits are bounded in time; a timeout records code 1 in the
// status word and the CTA drains its copies and returns.
#include <algorithm>
#include <mutex>

#include "ptx.cuh"
#include "q4lin_internal.h"

namespace q4lin {
namespace {
using namespace ptx;

constexpr int kCWarps = 16;                // consumer warps: 4 per SM sub-partition
constexpr int kCThreads = 32 * kCWarps;
constexpr int kThreadsG = kCThreads + 32;  // + the producer warp
constexpr int kSliceBytes = 256;           // packed bytes per row per tile
constexpr int kSliceK = 512;
constexpr int kStagesG = 4;
constexpr int kPrefetch = 2;               // tiles of scales loaded ahead
constexpr int kXPad = 36;                  // floats per 32-float x chunk in shared memory
constexpr int64_t kDrainNs = 4000000000LL;
constexpr int kMaxSmemG = 227 * 1024;

struct GArgs {
    const float* x;
    const void* scales;
    const float* bias;
    float* out;
    int64_t N, K, gs;
    int scale_f16, per_channel, svec, kslices, x_chunks;
    int64_t row_blocks;
    int* status;
    int64_t wait_ns;
};

// Shared memory: the stage ring, the barriers, then x (padded chunks of 32 floats).
__host__ __device__ constexpr int ring_bytes(int rb) { return kStagesG * rb * kSliceBytes; }
__host__ __device__ constexpr int x_offset(int rb) { return ring_bytes(rb) + 16 * kStagesG + 16; }
inline int smem_bytes_g(int rb, int64_t K) {
    return 128 + x_offset(rb) + (int)((K + kSliceK - 1) / kSliceK * 16) * kXPad * 4;
}

__device__ __forceinline__ float load_scale(const void* scales, int f16, int64_t idx) {
    if (f16) return __half2float(__ldg(reinterpret_cast<const __half*>(scales) + idx));
    return __ldg(reinterpret_cast<const float*>(scales) + idx);
}

// s[v] = scale[g, n0 + v] (0 past N or when !valid).
template <int V>
__device__ __forceinline__ void load_scales(const GArgs& a, int64_t g, int64_t n0, bool valid,
                                            float (&s)[V]) {
    const int64_t base = g * a.N + n0;
    if (valid && a.svec && n0 + V <= a.N) {
        if (a.scale_f16) {
            const __half* p = reinterpret_cast<const __half*>(a.scales) + base;
            if constexpr (V == 4) {
                const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
                const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
                const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
                s[0] = f0.x; s[1] = f0.y; s[2] = f1.x; s[3] = f1.y;
            } else if constexpr (V == 2) {
                const float2 f = __half22float2(__ldg(reinterpret_cast<const __half2*>(p)));
                s[0] = f.x; s[1] = f.y;
            } else {
                s[0] = __half2float(__ldg(p));
            }
        } else {
            const float* p = reinterpret_cast<const float*>(a.scales) + base;
            if constexpr (V == 4) {
                const float4 f = __ldg(reinterpret_cast<const float4*>(p));
                s[0] = f.x; s[1] = f.y; s[2] = f.z; s[3] = f.w;
            } else if constexpr (V == 2) {
                const float2 f = __ldg(reinterpret_cast<const float2*>(p));
                s[0] = f.x; s[1] = f.y;
            } else {
                s[0] = __ldg(p);
            }
        }
    } else {
#pragma unroll
        for (int v = 0; v < V; ++v)
            s[v] = (valid && n0 + v < a.N) ? load_scale(a.scales, a.scale_f16, base + v) : 0.f;
    }
}

// sum over the 32 values of one 16-byte chunk of x[t] * (code_t - 8).
template <bool EH>
__device__ __forceinline__ float chunk_dot(const uint4& wv, const float4 (&xv)[8]) {
    float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
    const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        float2 c[4];
        codes_word<EH>(words[w], c);
        const float4 p = xv[2 * w], q = xv[2 * w + 1];
        float2& acc = (w & 1) ? a1 : a0;
        acc = ffma2(c[0], make_float2(p.x, p.y), acc);
        acc = ffma2(c[1], make_float2(p.z, p.w), acc);
        acc = ffma2(c[2], make_float2(q.x, q.y), acc);
        acc = ffma2(c[3], make_float2(q.z, q.w), acc);
    }
    return (a0.x + a0.y) + (a1.x + a1.y);
}

template <int V, bool EH>
__global__ void __launch_bounds__(kThreadsG, 1)
    gemv_tma_kernel(const __grid_constant__ CUtensorMap tmap_w, const GArgs a) {
    constexpr int rb = 32 * V;  // rows per block: 32 row groups of V rows
    constexpr uint32_t tile_bytes = rb * kSliceBytes;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 127u) & ~127u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t bar_base = base + ring_bytes(rb);
    volatile int* failed =
        reinterpret_cast<volatile int*>(gbase + (bar_base + 16 * kStagesG - base));
    float* xs = reinterpret_cast<float*>(gbase + x_offset(rb));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto full = [&](int s) { return bar_base + 8u * s; };
    auto empty = [&](int s) { return bar_base + 8u * (kStagesG + s); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStagesG; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), kCWarps);
        }
        *failed = 0;
        mbar_init_fence();
    }
    __syncthreads();
    griddep_launch_dependents();

    if (warp == kCWarps) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tensormap(&tmap_w);
            int64_t t = 0;
            bool stop = false;
            for (int64_t blk = blockIdx.x; blk < a.row_blocks && !stop; blk += gridDim.x) {
                for (int ks = 0; ks < a.kslices; ++ks) {
                    const int s = (int)(t % kStagesG);
                    if (t >= kStagesG &&
                        !wait_bounded(empty(s), (uint32_t)((t / kStagesG) - 1) & 1, a.wait_ns,
                                      failed)) {
                        record_failure(a.status, failed);
                        stop = true;
                        break;
                    }
                    if (*failed) {
                        stop = true;
                        break;
                    }
                    mbar_arrive_expect_tx(full(s), tile_bytes);
                    tma_load_2d(base + s * tile_bytes, &tmap_w, ks * kSliceBytes, (int)(blk * rb),
                                full(s));
                    ++t;
                }
            }
            // The last armed tiles may still be landing; the CTA must not exit first.
            for (int64_t j = t > kStagesG ? t - kStagesG : 0; j < t; ++j)
                wait_bounded(full((int)(j % kStagesG)), (uint32_t)(j / kStagesG) & 1, kDrainNs,
                             nullptr);
        }
        return;
    }

    // ------------------------------------------------------------------ consumers
    const int j = threadIdx.x & 15;          // chunk lane within a 256-byte slice
    const int r0 = (threadIdx.x >> 4) * V;   // first of this thread's V rows in a block

    // Scales of this thread's tiles, kPrefetch tiles ahead of use (they do not depend
    // on the preceding kernel, so the first ones are requested before griddep_wait).
    float sc[kPrefetch + 1][V];
    int64_t pf_blk = blockIdx.x;
    int pf_ks = 0;
    auto fetch = [&](float (&dst)[V]) {
        if (pf_blk < a.row_blocks && !a.per_channel) {
            const int64_t k0 = (int64_t)pf_ks * kSliceK + j * 32;
            load_scales<V>(a, k0 < a.K ? k0 / a.gs : 0, pf_blk * rb + r0, k0 < a.K, dst);
        }
        if (++pf_ks == a.kslices) {
            pf_ks = 0;
            pf_blk += gridDim.x;
        }
    };
#pragma unroll
    for (int p = 0; p < kPrefetch; ++p) fetch(sc[p]);

    // x into shared memory once: chunk c (32 floats) at xs + c * kXPad; zero past K.
    griddep_wait();
    for (int i = threadIdx.x; i < a.x_chunks * 8; i += kCThreads) {
        const int c = i >> 3, q = i & 7;
        const int64_t k = (int64_t)c * 32 + q * 4;
        const float4 v = k < a.K ? __ldg(reinterpret_cast<const float4*>(a.x + k))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4*>(xs + c * kXPad + q * 4) = v;
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kCThreads) : "memory");

    int64_t t = 0;
    for (int64_t blk = blockIdx.x; blk < a.row_blocks; blk += gridDim.x) {
        const int64_t n0 = blk * rb + r0;
        float acc[V];
#pragma unroll
        for (int v = 0; v < V; ++v) acc[v] = 0.f;
        for (int ks = 0; ks < a.kslices; ++ks, ++t) {
            const int s = (int)(t % kStagesG);
            fetch(sc[kPrefetch]);
            float4 xv[8];
            const float* xc = xs + (ks * 16 + j) * kXPad;
#pragma unroll
            for (int i = 0; i < 8; ++i) xv[i] = *reinterpret_cast<const float4*>(xc + 4 * i);
            const bool got = __all_sync(
                0xffffffffu, wait_bounded(full(s), (uint32_t)(t / kStagesG) & 1, a.wait_ns, failed));
            if (!got) {
                if (lane == 0) record_failure(a.status, failed);
                return;
            }
            const uint32_t tile = base + s * tile_bytes;
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const uint4 wv = ld_shared_v4(tile + (r0 + v) * kSliceBytes + j * 16);
                const float d = chunk_dot<EH>(wv, xv);
                acc[v] = a.per_channel ? acc[v] + d : fmaf(d, sc[0][v], acc[v]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(s));
#pragma unroll
            for (int p = 0; p < kPrefetch; ++p)
#pragma unroll
                for (int v = 0; v < V; ++v) sc[p][v] = sc[p + 1][v];
        }
#pragma unroll
        for (int v = 0; v < V; ++v) {
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) acc[v] += __shfl_xor_sync(0xffffffffu, acc[v], o);
        }
        float mine = acc[0];
#pragma unroll
        for (int v = 1; v < V; ++v)
            if (j == v) mine = acc[v];
        const int64_t n = n0 + j;
        if (j < V && n < a.N) {
            if (a.per_channel) mine *= load_scale(a.scales, a.scale_f16, n);
            if (a.bias) mine += __ldg(a.bias + n);
            a.out[n] = mine;
        }
    }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

template <int V, bool EH>
cudaError_t launch_v(const CUtensorMap& tw, const GArgs& a, unsigned grid, const LaunchCtx& c) {
    static cudaError_t attr = cudaFuncSetAttribute(
        gemv_tma_kernel<V, EH>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmemG);
    if (attr != cudaSuccess) return attr;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreadsG);
    cfg.dynamicSmemBytes = smem_bytes_g(32 * V, a.K);
    cfg.stream = c.stream;
    cudaLaunchAttribute attrs[1];
    if (c.pdl) {
        attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attrs;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, gemv_tma_kernel<V, EH>, tw, a);
}

}  // namespace

bool gemv_tma_eligible(const Problem& p) {
    if (p.M != 1 || p.K % 32 != 0 || p.K < 2 * kSliceBytes || p.N < 32) return false;
    if (smem_bytes_g(128, p.K) > kMaxSmemG) return false;
    if (reinterpret_cast<uintptr_t>(p.x) % 16 || reinterpret_cast<uintptr_t>(p.qweight) % 16)
        return false;
    if (!(p.group_size >= p.K || p.group_size % 32 == 0)) return false;
    if (p.N > 0x7FFFFFFFLL) return false;
    return encode_fn() != nullptr;
}

cudaError_t gemv_tma_launch(const Problem& p, const LaunchCtx& c) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    // Rows per block: as large as the GPU stays busy with (more rows per thread reuse
    // the x chunk more), smaller for short matrices so every SM gets a block.
    int V = 4;
    if ((p.N + 127) / 128 < c.sm_count) V = 2;
    if ((p.N + 63) / 64 < c.sm_count) V = 1;
    const int rb = 32 * V;
    GArgs a;
    a.x = p.x;
    a.scales = p.scales;
    a.bias = p.bias;
    a.out = p.out;
    a.N = p.N;
    a.K = p.K;
    a.gs = p.group_size;
    a.scale_f16 = p.scale_f16;
    a.per_channel = p.group_size >= p.K;
    const int esize = p.scale_f16 ? 2 : 4;
    a.svec = (reinterpret_cast<uintptr_t>(p.scales) % 16 == 0) && (p.N % 4 == 0) && esize > 0;
    a.kslices = (int)((p.K + kSliceK - 1) / kSliceK);
    a.x_chunks = a.kslices * 16;
    a.row_blocks = (p.N + rb - 1) / rb;
    a.status = c.status_word;
    a.wait_ns = c.wait_limit_ns;

    CUtensorMap tw;
    const int64_t Kp = p.K / 2;
    const cuuint64_t dims[2] = {(cuuint64_t)Kp, (cuuint64_t)p.N};
    const cuuint64_t strides[1] = {(cuuint64_t)Kp};
    const cuuint32_t box[2] = {(cuuint32_t)kSliceBytes, (cuuint32_t)rb};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(p.qweight), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const unsigned grid = (unsigned)std::min<int64_t>(a.row_blocks, c.sm_count);
    const bool eh = p.even_high != 0;
    if (V == 4) return eh ? launch_v<4, true>(tw, a, grid, c) : launch_v<4, false>(tw, a, grid, c);
    if (V == 2) return eh ? launch_v<2, true>(tw, a, grid, c) : launch_v<2, false>(tw, a, grid, c);
    return eh ? launch_v<1, true>(tw, a, grid, c) : launch_v<1, false>(tw, a, grid, c);
}

}  // namespace q4lin
