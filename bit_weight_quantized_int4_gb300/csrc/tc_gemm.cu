// tc_gemm.cu -- tcgen05 tensor-core GEMM of the 4-bit weight-quantized linear (sm_103a).
//
//   out[m, n] = bias[n] + sum_k x[m, k] * (code[n, k] - 8) * scale[k / gs, n]
//
// (the formula of "[ExecuTorch][WebGPU] Add linear_qcs4w op", Solution; prefill, M > 1,
// is the regime of "Add 256-thread steel q4gsw prefill GEMM").  The page's kernel stages
// f32 activations and dequantized weights of a BK = 16 slice in shared memory and
// accumulates a 64x64 tile on CUDA cores; on GB300 the contraction goes to the 5th-gen
// tensor cores instead, and what survives of the page's design is its "dequantize once
// per packed word, read the group scale once" staging (the pwdq variant).
//
// Computed as D[n, m] = sum_k A[n, k] * B[m, k] with
//   A = dequantized weight tile, 128 rows of W (the MMA's M), written by CUDA cores into
//       shared memory as fp32 (read by the MMA as tf32), K-major, 128-byte swizzle;
//   B = x tile, bm rows of x (the MMA's N, 16..256), fp32 straight from HBM by TMA
//       (read as tf32), K-major, 128-byte swizzle;
//   D = fp32 accumulator in tensor memory (128 lanes x bm columns).
// tf32 keeps 10 explicit mantissa bits of each operand, so a product carries a relative
// error below 2^-9 -- inside the 4e-3 * sum|x*w| bar of the tensor-core path.
//
// Roles (320 threads, one CTA per 128 x bm output tile):
//   warp 0, one lane: TMA producer; per stage (32 k) the x tile [bm x 128 B] and the
//                     packed weight tile [128 rows x 16 B] land in a 4-stage ring.
//   warp 1:           allocates tensor memory; one lane issues 4 tcgen05.mma (K = 8
//                     each) per stage and commits each stage's completion to "empty".
//   warps 2-9:        two groups of 4 warps, each taking alternate stages (so one
//                     group's proxy fence and arrive overlap the other's work); one
//                     thread per weight row: widen 32 codes, multiply by the group
//                     scale, store the row into the swizzled A stage, fence, arrive on
//                     "a_ready"; at the end each warp reads its 32-lane slice of D with
//                     tcgen05.ld (the groups split the columns), adds the bias and
//                     stores out (predicated m < M, n < N).
// Every mbarrier wait is bounded in time (%globaltimer).  A wait that runs out records
// code 1 in the status word; the CTA then stops issuing work, waits for its own copies
// and MMAs in flight, frees its tensor memory and returns.
#include <algorithm>
#include <mutex>

#include "ptx.cuh"
#include "q4lin_internal.h"

namespace q4lin {
namespace {
using namespace ptx;

constexpr int kDequantGroups = 2;     // warp groups of 4 that dequantize alternate stages
constexpr int kThreadsTc = 64 + 128 * kDequantGroups;
constexpr int kRows = 128;            // weight rows per tile (MMA M)
constexpr int kStageK = 32;           // k per stage: 32 fp32 = one 128-byte swizzle row
constexpr int kStages = 4;
constexpr int kATile = kRows * 128;   // 16 KiB
constexpr int kWTile = kRows * 16;    // 2 KiB: 32 codes per row
constexpr int kMaxBm = 256;
constexpr int64_t kDrainLimitNs = 4000000000LL;
constexpr int kScaleAhead = 6;        // stages of group scales requested ahead of use

constexpr int smem_bytes_for(int bm) {
    return 1024 + kStages * (kATile + bm * 128 + kWTile) + 256;
}

struct TcArgs {
    const void* scales;
    const float* bias;
    float* out;
    int64_t M, N, K, gs;
    int scale_f16, per_channel, even_high;
    int bm, k_iters, tmem_cols;
    int gs_stages;  // group size in stages of 32 k (grouped scales)
    int gs_shift;   // log2(gs_stages) when a power of two, else -1
    int* status;
    int64_t wait_ns;
    int skip_first_copy;
};

__device__ __forceinline__ float load_scale(const void* scales, int f16, int64_t idx) {
    if (f16) return __half2float(__ldg(reinterpret_cast<const __half*>(scales) + idx));
    return __ldg(reinterpret_cast<const float*>(scales) + idx);
}

// Signed codes (c - 8) of the 8 nibbles of one packed word, in k order (nibble i holds
// k = i).  0x6400 is binary16 1024; OR-ing a 4-bit code into its mantissa gives 1024 + c,
// and one mixed-precision add widens it and subtracts 1032, exactly.
__device__ __forceinline__ void codes8(uint32_t w, float (&v)[8]) {
    const uint32_t h[4] = {(w & 0x000F000Fu) | 0x64006400u, ((w >> 4) & 0x000F000Fu) | 0x64006400u,
                           ((w >> 8) & 0x000F000Fu) | 0x64006400u,
                           ((w >> 12) & 0x000F000Fu) | 0x64006400u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        asm("{\n\t.reg .b16 l, u;\n\tmov.b32 {l, u}, %2;\n\t"
            "add.rn.f32.f16 %0, l, %3;\n\tadd.rn.f32.f16 %1, u, %3;\n\t}"
            : "=f"(v[i]), "=f"(v[i + 4])
            : "r"(h[i]), "f"(-1032.0f));
    }
}

__global__ void __launch_bounds__(kThreadsTc, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmap_x,
                   const __grid_constant__ CUtensorMap tmap_w, const TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const int bm = a.bm;
    const uint32_t a_base = base;
    const uint32_t b_base = a_base + kStages * kATile;
    const uint32_t w_base = b_base + kStages * bm * 128;
    const uint32_t bar_base = w_base + kStages * kWTile;
    const uint32_t accfull = bar_base + 8 * 3 * kStages;
    const uint32_t tmem_slot = accfull + 8;
    uint32_t* tmem_slot_ptr = reinterpret_cast<uint32_t*>(gbase + (tmem_slot - base));
    volatile int* failed = reinterpret_cast<volatile int*>(gbase + (tmem_slot + 4 - base));
    auto full = [&](int s) { return bar_base + 8u * s; };
    auto aready = [&](int s) { return bar_base + 8u * (kStages + s); };
    auto empty = [&](int s) { return bar_base + 8u * (2 * kStages + s); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(aready(s), 128);  // the 128 threads of the group that owns the stage
            mbar_init(empty(s), 1);
        }
        mbar_init(accfull, 1);
        *failed = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(tmem_slot, (uint32_t)a.tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_d = *tmem_slot_ptr;
    griddep_wait();

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ TMA producer
            const int m0 = (int)blockIdx.y * bm, n0 = (int)blockIdx.x * kRows;
            int it = 0;
            for (; it < a.k_iters; ++it) {
                const int s = it % kStages;
                if (it >= kStages &&
                    !wait_bounded(empty(s), ((it / kStages) - 1) & 1, a.wait_ns, failed)) {
                    record_failure(a.status, failed);
                    break;
                }
                if (*failed) break;
                if (a.skip_first_copy && it == 0) continue;
                mbar_arrive_expect_tx(full(s), (uint32_t)(bm * 128 + kWTile));
                tma_load_2d(b_base + s * bm * 128, &tmap_x, it * kStageK, m0, full(s));
                tma_load_2d(w_base + s * kWTile, &tmap_w, it * (kStageK / 2), n0, full(s));
            }
            // Copies of the last stages may still be landing; the CTA must not exit first.
            for (int j = it > kStages ? it - kStages : 0; j < it; ++j) {
                if (a.skip_first_copy && j == 0) continue;
                wait_bounded(full(j % kStages), (j / kStages) & 1, kDrainLimitNs, nullptr);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------------- MMA issuer
            const uint32_t idesc = tf32_idesc(kRows, bm);
            for (int it = 0; it < a.k_iters; ++it) {
                const int s = it % kStages;
                const uint32_t par = (it / kStages) & 1;
                if (!wait_bounded(full(s), par, a.wait_ns, failed) ||
                    !wait_bounded(aready(s), par, a.wait_ns, failed)) {
                    record_failure(a.status, failed);
                    break;
                }
                // The A stage was written through the generic proxy, fenced to the async
                // proxy by its writers before they arrived; the B stage came by TMA.  The
                // mbarrier waits above order both before these MMAs.
                const uint32_t ab = a_base + s * kATile, bb = b_base + s * bm * 128;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_tf32(tmem_d, sw128_desc(ab + kk * 32), sw128_desc(bb + kk * 32), idesc,
                             (it | kk) != 0);
                mma_commit(empty(s));
            }
            mma_commit(accfull);  // arrives once every MMA issued above has completed
        }
        __syncwarp();
    } else {
        // ------------------------------------------------- dequantization, epilogue
        const int group = (warp - 2) >> 2;  // dequantizes stages it % kDequantGroups == group
        const int quarter = warp & 3;       // the 32-lane slice of tensor memory this warp owns
        const int row = quarter * 32 + lane;
        const int64_t n = (int64_t)blockIdx.x * kRows + row;
        const bool row_ok = n < a.N;
        const uint32_t swz = (uint32_t)(row & 7);
        bool ok = true;
        // Group scales of this row for this group's stages, kScaleAhead of them ahead of
        // use (a global load takes longer than a stage of MMAs).  The loop is unrolled by
        // the ring size so each slot is a fixed register (no move of a pending load).
        float sc_ring[kScaleAhead];
        auto scale_of = [&](int it) -> float {
            if (!row_ok) return 0.f;
            if (a.per_channel || it >= a.k_iters) return 1.f;
            const int g = a.gs_shift >= 0 ? (it >> a.gs_shift) : it / a.gs_stages;
            return load_scale(a.scales, a.scale_f16, (int64_t)g * a.N + n);
        };
#pragma unroll
        for (int i = 0; i < kScaleAhead; ++i) sc_ring[i] = scale_of(group + i * kDequantGroups);
        constexpr int kStride = kScaleAhead * kDequantGroups;
        for (int it0 = group; it0 < a.k_iters && ok; it0 += kStride) {
#pragma unroll
            for (int u = 0; u < kScaleAhead; ++u) {
                const int it = it0 + u * kDequantGroups;
                if (it >= a.k_iters) break;
                const int s = it % kStages;
                if (!wait_bounded(full(s), (it / kStages) & 1, a.wait_ns, failed)) {
                    record_failure(a.status, failed);
                    ok = false;
                    break;
                }
                uint4 wv = ld_shared_v4(w_base + s * kWTile + row * 16);
                if (a.even_high) {
                    wv.x = ((wv.x & 0x0F0F0F0Fu) << 4) | ((wv.x >> 4) & 0x0F0F0F0Fu);
                    wv.y = ((wv.y & 0x0F0F0F0Fu) << 4) | ((wv.y >> 4) & 0x0F0F0F0Fu);
                    wv.z = ((wv.z & 0x0F0F0F0Fu) << 4) | ((wv.z >> 4) & 0x0F0F0F0Fu);
                    wv.w = ((wv.w & 0x0F0F0F0Fu) << 4) | ((wv.w >> 4) & 0x0F0F0F0Fu);
                }
                const float sc = sc_ring[u];
                sc_ring[u] = scale_of(it + kStride);
                const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
                const uint32_t arow = a_base + s * kATile + row * 128;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float v[8];
                    codes8(words[j], v);
#pragma unroll
                    for (int t = 0; t < 8; ++t) v[t] *= sc;
                    st_shared_v4(arow + (((2u * j) ^ swz) << 4), v[0], v[1], v[2], v[3]);
                    st_shared_v4(arow + (((2u * j + 1) ^ swz) << 4), v[4], v[5], v[6], v[7]);
                }
                fence_proxy_async_smem();
                mbar_arrive(aready(s));
            }
        }
        const bool acc_ok = wait_bounded(accfull, 0, ok ? a.wait_ns : kDrainLimitNs, nullptr);
        if (!acc_ok) record_failure(a.status, failed);
        tc_fence_after();
        const bool go = __all_sync(0xffffffffu, acc_ok && !*failed);
        if (go) {
            const float pc = (a.per_channel && row_ok) ? load_scale(a.scales, a.scale_f16, n) : 1.f;
            const float bs = (a.bias && row_ok) ? __ldg(a.bias + n) : 0.f;
            const int64_t m0 = (int64_t)blockIdx.y * bm;
            const uint32_t lane_base = tmem_d + ((uint32_t)(quarter * 32) << 16);
            for (int c0 = 16 * group; c0 < bm; c0 += 16 * kDequantGroups) {
                uint32_t r[16];
                tmem_ld16(lane_base + (uint32_t)c0, r);
                if (row_ok) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int64_t m = m0 + c0 + j;
                        if (m < a.M) a.out[m * a.N + n] = fmaf(__uint_as_float(r[j]), pc, bs);
                    }
                }
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_d, (uint32_t)a.tmem_cols);
    }
}

// ------------------------------------------------------------------------- host side
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

cudaError_t ensure_smem_attr() {
    static cudaError_t err = cudaErrorNotReady;
    static std::once_flag once;
    std::call_once(once, [] {
        err = cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   smem_bytes_for(kMaxBm));
    });
    return err;
}

}  // namespace

bool tc_eligible(const Problem& p, const LaunchCtx& c) {
    if (p.K % kStageK != 0) return false;
    if (reinterpret_cast<uintptr_t>(p.x) % 16 || reinterpret_cast<uintptr_t>(p.qweight) % 16)
        return false;
    if (!(p.group_size >= p.K || p.group_size % kStageK == 0)) return false;
    if (p.M > 65535LL * kMaxBm) return false;
    if (c.max_smem_optin < smem_bytes_for(kMaxBm)) return false;
    return encode_fn() != nullptr;
}

cudaError_t tc_launch(const Problem& p, const LaunchCtx& c) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    cudaError_t e = ensure_smem_attr();
    if (e != cudaSuccess) return e;
    // x rows per tile (the MMA's N).  Larger tiles reuse each dequantized weight tile
    // more; smaller ones give more CTAs.  Estimate waves x cycles per stage, where a
    // stage costs ~2 * bm cycles of tf32 MMA but no less than the CUDA-core dequant
    // (~160 cycles for 128 rows x 32 codes on 4 warps), and take the cheapest.
    const int64_t ntiles = (p.N + kRows - 1) / kRows;
    int bm = 16;
    int64_t mtiles = 0, best = -1;
    for (int cand = kMaxBm; cand >= 16; cand /= 2) {
        const int64_t mt = (p.M + cand - 1) / cand;
        if (mt > 65535) continue;
        const int64_t per_tile = (p.M + mt - 1) / mt;
        const int b = (int)std::min<int64_t>(cand, (per_tile + 15) / 16 * 16);
        const int64_t waves = (ntiles * mt + c.sm_count - 1) / c.sm_count;
        const int64_t cost = waves * std::max<int64_t>(2 * b, 160);
        if (best < 0 || cost < best) {
            best = cost;
            bm = b;
            mtiles = mt;
        }
    }
    int cols = 32;
    while (cols < bm) cols <<= 1;

    TcArgs a;
    a.scales = p.scales;
    a.bias = p.bias;
    a.out = p.out;
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.gs = p.group_size;
    a.scale_f16 = p.scale_f16;
    a.per_channel = p.group_size >= p.K;
    a.even_high = p.even_high;
    a.bm = bm;
    a.k_iters = (int)(p.K / kStageK);
    a.tmem_cols = cols;
    a.status = c.status_word;
    a.wait_ns = c.wait_limit_ns;
    a.skip_first_copy = c.tc_skip_first_copy;
    a.gs_stages = a.per_channel ? 1 : (int)(p.group_size / kStageK);
    a.gs_shift = -1;
    for (int sft = 0; sft < 31; ++sft)
        if ((1 << sft) == a.gs_stages) a.gs_shift = sft;

    CUtensorMap tx, tw;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)p.K, (cuuint64_t)p.M};
        const cuuint64_t strides[1] = {(cuuint64_t)p.K * 4};
        const cuuint32_t box[2] = {(cuuint32_t)kStageK, (cuuint32_t)bm};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(p.x), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const int64_t Kp = p.K / 2;
        const cuuint64_t dims[2] = {(cuuint64_t)Kp, (cuuint64_t)p.N};
        const cuuint64_t strides[1] = {(cuuint64_t)Kp};
        const cuuint32_t box[2] = {(cuuint32_t)(kStageK / 2), (cuuint32_t)kRows};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(p.qweight), dims,
                strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((p.N + kRows - 1) / kRows), (unsigned)mtiles);
    cfg.blockDim = dim3(kThreadsTc);
    cfg.dynamicSmemBytes = smem_bytes_for(bm);
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[1];
    if (c.pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, tc_gemm_kernel, tx, tw, a);
}

}  // namespace q4lin
