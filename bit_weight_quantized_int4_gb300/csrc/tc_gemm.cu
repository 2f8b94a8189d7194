// tc_gemm2.cu -- tcgen05 tensor-core GEMM of the 4-bit weight-quantized linear, with the
// activations as the MMA's A operand (sm_103a).
//
//   out[m, n] = bias[n] + sum_k x[m, k] * (code[n, k] - 8) * scale[k / gs, n]
//
// (the formula of "[ExecuTorch][WebGPU] Add linear_qcs4w op", Solution; prefill, M > 1, is
// the regime of "Add 256-thread steel q4gsw prefill GEMM", whose 64x64 CUDA-core tile with
// a BK = 16 shared-memory slice is replaced here by the 5th-generation tensor cores; what
// is kept from that page is its dequantize-once staging of the "pwdq" variant: each packed
// word is widened once per tile and its group scale read once.)
//
// D[m, n] = sum_k A[m, k] * B[n, k] with
//   A = x tile, 128 rows of x (the MMA's M), fp32 from HBM by TMA with the 128-byte
//       swizzle, read by the MMA as tf32 (K-major);
//   B = dequantized weight tile, bn rows of W (the MMA's N, 64..256), written by CUDA
//       cores into shared memory as fp32 (tf32 to the MMA), K-major, 128-byte swizzle;
//   D = fp32 accumulator in tensor memory: 128 lanes (m) x bn columns (n).
// Putting the weights on the MMA's N side keeps the MMAs wide (N = 256) even for a short
// prompt, and each stage of x (16 KiB) feeds 256 weight rows.  tf32 keeps 10 explicit
// mantissa bits of each operand: a product carries a relative error below 2^-9, inside
// the 4e-3 * sum|x*w| bar of the tensor-core path.
//
// Roles (320 threads, one CTA per 128 x bn output tile, a ring of 32-k stages):
//   warp 0, one lane: TMA producer: per stage the x tile [128 x 128 B] and the packed
//                     weight tile [bn rows x 16 B].
//   warp 1:           allocates tensor memory; one lane issues 4 tcgen05.mma (K = 8) per
//                     stage and commits each stage's completion to "empty".
//   warps 2-9:        two groups of 4 warps taking alternate stages; each thread widens
//                     the codes of bn/128 weight rows, applies the group scale, writes the
//                     rows into the swizzled B stage, fences them to the async proxy and
//                     arrives on "b_ready".  At the end each warp reads its 32 lanes (m)
//                     of D with tcgen05.ld (the groups split the columns), applies the
//                     channel scale and bias, and stores out (predicated m < M, n < N).
// Every mbarrier wait is bounded in time; a timeout records code 1 in the status word,
// after which the CTA stops issuing work, drains its copies and MMAs, frees its tensor
// memory and returns.
#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "ptx.cuh"
#include "q4lin_internal.h"

namespace q4lin {
namespace {
using namespace ptx;

constexpr int kGroups = 2;                   // dequantizing warp groups (alternate stages)
constexpr int kThreads2 = 64 + 128 * kGroups;
constexpr int kXRows = 128;                  // x rows per tile (MMA M)
constexpr int kStageK = 32;                  // 32 fp32 = one 128-byte swizzle row
constexpr int kATile = kXRows * 128;         // 16 KiB
constexpr int kMaxStages = 8;
constexpr int kScaleAhead = 4;               // stages of scales in flight per thread
constexpr int kWPrefetch = 8;                // stages per L2 prefetch block of packed weights
constexpr int64_t kDrainNs = 4000000000LL;
constexpr int kSmemLimit = 227 * 1024;

__host__ __device__ constexpr int stage_bytes(int bn) { return kATile + bn * 128 + bn * 16; }
// Shared memory: alignment slack, the stage ring, barriers (256 bytes), then the tile's
// bias and channel scales (2 x 256 floats) for the epilogue.
inline int smem_bytes(int bn, int stages) { return 1024 + stages * stage_bytes(bn) + 256 + 2048; }

struct Tc2Args {
    const void* scales;
    const float* bias;
    float* out;
    int64_t M, N, K;
    int scale_f16, per_channel;
    int bn, stages, k_iters, tmem_cols;
    int gs_stages, gs_shift;  // group size in stages; log2 of it or -1
    int out_vec;              // 16-byte stores of out are aligned
    int tma_out;              // out is written by TMA tensor stores from shared memory
    int* status;
    int64_t wait_ns;
    int skip_first_copy;
    // Split K over a cluster of `splitk` CTAs (1: no split): CTA rank r of the cluster
    // covers stages [r * kpp, (r + 1) * kpp) of the tile; the partial tiles meet in
    // distributed shared memory, where rank q adds the columns [q * sw, (q + 1) * sw) of
    // all partials in rank order (row stride rs floats in the exchange buffer).
    int splitk, kpp, sw, rs;
    int w_prefetch;  // pull 128-byte weight row segments into L2 ahead (few M tiles: the
                     // weights stream from DRAM once; with many M tiles they sit in L2)
};

__device__ __forceinline__ float load_scale(const void* scales, int f16, int64_t idx) {
    if (f16) return __half2float(__ldg(reinterpret_cast<const __half*>(scales) + idx));
    return __ldg(reinterpret_cast<const float*>(scales) + idx);
}
__device__ __forceinline__ uint32_t load_scale_bits(const void* scales, int f16, int64_t idx) {
    if (f16) return __ldg(reinterpret_cast<const unsigned short*>(scales) + idx);
    return __ldg(reinterpret_cast<const unsigned int*>(scales) + idx);
}
__device__ __forceinline__ float scale_from_bits(uint32_t bits, int f16) {
    return f16 ? __half2float(__ushort_as_half((unsigned short)bits)) : __uint_as_float(bits);
}

template <int RPT, bool EH>
__global__ void __launch_bounds__(kThreads2, 1)
    tc_xa_kernel(const __grid_constant__ CUtensorMap tmap_x,
                 const __grid_constant__ CUtensorMap tmap_w,
                 const __grid_constant__ CUtensorMap tmap_o,
                 const __grid_constant__ CUtensorMap tmap_wp, const Tc2Args a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const int bn = a.bn, S = a.stages;
    const uint32_t a_base = base;
    const uint32_t b_base = a_base + S * kATile;
    const uint32_t w_base = b_base + S * bn * 128;
    const uint32_t bar_base = w_base + S * bn * 16;
    const uint32_t accfull = bar_base + 8 * 3 * kMaxStages;
    const uint32_t tmem_slot = accfull + 24;
    const int P = a.splitk;
    const int rank = P > 1 ? (int)cluster_ctarank() : 0;
    const int ntile = (int)blockIdx.x / P;
    const int it_begin = rank * a.kpp;
    const int n_iters = min(a.kpp, a.k_iters - it_begin);
    uint32_t* tmem_slot_ptr = reinterpret_cast<uint32_t*>(gbase + (tmem_slot - base));
    volatile int* failed = reinterpret_cast<volatile int*>(gbase + (tmem_slot + 4 - base));
    float* s_bias = reinterpret_cast<float*>(gbase + (bar_base + 256 - base));  // [256]
    float* s_cscale = s_bias + 256;                                              // [256]
    auto full = [&](int s) { return bar_base + 8u * s; };
    auto bready = [&](int s) { return bar_base + 8u * (kMaxStages + s); };
    auto empty = [&](int s) { return bar_base + 8u * (2 * kMaxStages + s); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), 1);
            mbar_init(bready(s), 128);  // the 128 threads of the group that owns the stage
            mbar_init(empty(s), 1);
        }
        mbar_init(accfull, 1);
        *failed = 0;
        mbar_init_fence();
    }
    if (warp == 1) tmem_alloc(tmem_slot, (uint32_t)a.tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_d = *tmem_slot_ptr;
    // Peers arrive on this CTA's barriers only after every CTA has initialised its own.
    if (P > 1) cluster_sync_all();
    griddep_wait();

    bool epi_go = false;  // dequantization warps: the accumulator is complete and valid
    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ TMA producer
            prefetch_tensormap(&tmap_x);
            prefetch_tensormap(&tmap_w);
            prefetch_tensormap(&tmap_wp);
            const int m0 = (int)blockIdx.y * kXRows, n0 = ntile * bn;
            const uint32_t tx = (uint32_t)(kATile + bn * 16);
            int li = 0;
            for (; li < n_iters; ++li) {
                const int s = li % S;
                if (li >= S && !wait_bounded(empty(s), ((li / S) - 1) & 1, a.wait_ns, failed)) {
                    record_failure(a.status, failed);
                    break;
                }
                if (*failed) break;
                // The packed-weight tile of a stage is only 16 bytes per row; with few M
                // tiles, whole 128-byte row segments (eight stages) are pulled into L2 a
                // block ahead, so that DRAM streams long segments and the per-stage copies
                // hit L2.
                if (a.w_prefetch && (li & (kWPrefetch - 1)) == 0) {
                    const int first = li == 0 ? 0 : li + kWPrefetch;
                    for (int pb = first; pb <= li + kWPrefetch && pb < n_iters; pb += kWPrefetch)
                        tma_prefetch_l2_2d(&tmap_wp, (it_begin + pb) * (kStageK / 2), n0);
                }
                if (a.skip_first_copy && li == 0) continue;
                const int it = it_begin + li;
                mbar_arrive_expect_tx(full(s), tx);
                tma_load_2d(a_base + s * kATile, &tmap_x, it * kStageK, m0, full(s));
                tma_load_2d(w_base + s * bn * 16, &tmap_w, it * (kStageK / 2), n0, full(s));
            }
            // Copies of the last stages may still be landing; the CTA must not exit first.
            for (int j = li > S ? li - S : 0; j < li; ++j) {
                if (a.skip_first_copy && j == 0) continue;
                wait_bounded(full(j % S), (j / S) & 1, kDrainNs, nullptr);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------------- MMA issuer
            const uint32_t idesc = tf32_idesc(kXRows, bn);
            for (int it = 0; it < n_iters; ++it) {  // it: stage of this CTA's range
                const int s = it % S;
                const uint32_t par = (it / S) & 1;
                if (!wait_bounded(full(s), par, a.wait_ns, failed) ||
                    !wait_bounded(bready(s), par, a.wait_ns, failed)) {
                    record_failure(a.status, failed);
                    break;
                }
                // B was written through the generic proxy and fenced to the async proxy by
                // its writers before they arrived; A came by TMA.  The waits order both.
                const uint32_t ab = a_base + s * kATile, bb = b_base + s * bn * 128;
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
        const int group = (warp - 2) >> 2;
        const int tg = ((warp - 2) & 3) * 32 + lane;  // thread within its group
        const int64_t n0 = (int64_t)ntile * bn;
        // The tile's bias and channel scales, staged for the epilogue (their loads overlap
        // the main loop).
        for (int c = threadIdx.x - 64; c < bn; c += 128 * kGroups) {
            const int64_t n = n0 + c;
            s_bias[c] = (a.bias && n < a.N) ? __ldg(a.bias + n) : 0.f;
            s_cscale[c] = (a.per_channel && n < a.N) ? load_scale(a.scales, a.scale_f16, n) : 1.f;
        }
        bool ok = true;
        // Rows of the weight tile this thread widens: tg + 128 * i.
        int64_t nrow[RPT];
        bool rvalid[RPT];
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            const int r = tg + 128 * i;
            nrow[i] = n0 + r;
            rvalid[i] = r < bn && n0 + r < a.N;
        }
        // Group scales (raw bits) of this thread's rows for its group's stages,
        // kScaleAhead stages ahead; the loop is unrolled by the ring size so every slot
        // is a fixed register (no move of a pending load).
        uint32_t ring[kScaleAhead][RPT];
        auto fetch = [&](int it, uint32_t (&dst)[RPT]) {
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                uint32_t bits = 0;
                if (rvalid[i] && !a.per_channel && it < n_iters) {
                    const int git = it_begin + it;  // stage of the whole K
                    const int g = a.gs_shift >= 0 ? (git >> a.gs_shift) : git / a.gs_stages;
                    bits = load_scale_bits(a.scales, a.scale_f16, (int64_t)g * a.N + nrow[i]);
                }
                dst[i] = bits;
            }
        };
#pragma unroll
        for (int u = 0; u < kScaleAhead; ++u) fetch(group + u * kGroups, ring[u]);
        constexpr int kStride = kScaleAhead * kGroups;
        for (int it0 = group; it0 < n_iters && ok; it0 += kStride) {
#pragma unroll
            for (int u = 0; u < kScaleAhead; ++u) {
                const int it = it0 + u * kGroups;
                if (it >= n_iters) break;
                const int s = it % S;
                if (!wait_bounded(full(s), (it / S) & 1, a.wait_ns, failed)) {
                    record_failure(a.status, failed);
                    ok = false;
                    break;
                }
#pragma unroll
                for (int i = 0; i < RPT; ++i) {
                    const int r = tg + 128 * i;
                    if (r >= bn) continue;
                    const uint4 wv = ld_shared_v4(w_base + s * bn * 16 + r * 16);
                    float sc = 0.f;
                    if (rvalid[i]) sc = a.per_channel ? 1.f : scale_from_bits(ring[u][i], a.scale_f16);
                    const float2 sc2 = make_float2(sc, sc);
                    const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
                    const uint32_t brow = b_base + s * bn * 128 + r * 128;
                    const uint32_t swz = (uint32_t)(r & 7);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        float2 c[4];
                        codes_word<EH>(words[j], c);
#pragma unroll
                        for (int t = 0; t < 4; ++t) c[t] = fmul2(c[t], sc2);
                        st_shared_v4(brow + (((2u * j) ^ swz) << 4), c[0].x, c[0].y, c[1].x, c[1].y);
                        st_shared_v4(brow + (((2u * j + 1) ^ swz) << 4), c[2].x, c[2].y, c[3].x,
                                     c[3].y);
                    }
                }
                fetch(it + kStride, ring[u]);
                fence_proxy_async_smem();
                mbar_arrive(bready(s));
            }
        }
        const bool acc_ok = wait_bounded(accfull, 0, ok ? a.wait_ns : kDrainNs, nullptr);
        if (!acc_ok) record_failure(a.status, failed);
        tc_fence_after();
        asm volatile("bar.sync 2, %0;" ::"r"(128 * kGroups) : "memory");  // staged bias/scales
        const bool go = __all_sync(0xffffffffu, acc_ok && !*failed);
        epi_go = go;
        if (go && P == 1 && a.tma_out) {
            // The tile goes to shared memory (the free stage ring) as bn / 32 blocks of
            // [128 rows x 32 floats] in the 128-byte swizzle (16-byte unit u of row m at
            // u ^ (m & 7): a quarter-warp writes 8 distinct bank groups), then out by TMA
            // tensor stores (whole lines; rows >= M and columns >= N are not written).
            const int quarter = warp & 3;  // the 32-lane slice of tensor memory this warp owns
            const int ml = quarter * 32 + lane;
            const uint32_t lane_base = tmem_d + ((uint32_t)(quarter * 32) << 16);
            for (int c0 = 16 * group; c0 < bn; c0 += 16 * kGroups) {
                uint32_t r[16];
                tmem_ld16(lane_base + (uint32_t)c0, r);
                float v[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float val = __uint_as_float(r[j]);
                    if (a.per_channel) val *= s_cscale[c0 + j];
                    v[j] = val + s_bias[c0 + j];
                }
                const uint32_t row =
                    a_base + (uint32_t)(c0 / 32) * (kXRows * 128) + (uint32_t)ml * 128;
                const uint32_t u0 = (uint32_t)(c0 % 32) / 4;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    st_shared_v4(row + (((u0 + q) ^ ((uint32_t)ml & 7u)) << 4), v[4 * q],
                                 v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            }
            fence_proxy_async_smem();
        } else if (go && P == 1) {
            const int quarter = warp & 3;  // the 32-lane slice of tensor memory this warp owns
            const int64_t m = (int64_t)blockIdx.y * kXRows + quarter * 32 + lane;
            const bool m_ok = m < a.M;
            const uint32_t lane_base = tmem_d + ((uint32_t)(quarter * 32) << 16);
            float* orow = a.out + (m_ok ? m : 0) * a.N;
            for (int c0 = 16 * group; c0 < bn; c0 += 16 * kGroups) {
                uint32_t r[16];
                tmem_ld16(lane_base + (uint32_t)c0, r);
                const int64_t nb = n0 + c0;
                float v[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int64_t n = nb + j;
                    float val = __uint_as_float(r[j]);
                    if (n < a.N) {
                        if (a.per_channel) val *= s_cscale[c0 + j];
                        val += s_bias[c0 + j];
                    }
                    v[j] = val;
                }
                if (!m_ok) continue;
                if (a.out_vec && nb + 16 <= a.N) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<float4*>(orow + nb + 4 * q) =
                            make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (nb + j < a.N) orow[nb + j] = v[j];
                }
            }
        }
        if (P == 1 && a.tma_out) {
            asm volatile("bar.sync 2, %0;" ::"r"(128 * kGroups) : "memory");
            if (threadIdx.x == 64 && !*failed) {
                for (int b = 0; b < bn / 32 && n0 + 32 * b < a.N; ++b)
                    tma_store_2d(&tmap_o, (int)(n0 + 32 * b), (int)blockIdx.y * kXRows,
                                 a_base + (uint32_t)b * (kXRows * 128));
                bulk_commit();
                bulk_wait_read();
            }
        }
    }
    if (P > 1) {
        // ------------------------------------------- split K: reduce over the cluster
        // Shared memory (the free stage ring): send blocks [P][128][rs] (block q: columns
        // [q * sw, (q + 1) * sw) of this CTA's partial tile, rows padded to rs floats so a
        // quarter-warp writes 8 distinct bank groups), then this CTA's reduced slice
        // [128][sw].  Every thread reaches both cluster barriers: all earlier waits in this
        // kernel are bounded in time.
        const uint32_t blk_bytes = (uint32_t)(kXRows * a.rs * 4);
        const uint32_t send_base = a_base;
        const uint32_t slice_base = send_base + (uint32_t)P * blk_bytes;
        if (warp >= 2 && epi_go) {
            const int group = (warp - 2) >> 2;
            const int quarter = warp & 3;
            const int m = quarter * 32 + lane;
            const uint32_t lane_base = tmem_d + ((uint32_t)(quarter * 32) << 16);
            for (int c0 = 16 * group; c0 < bn; c0 += 16 * kGroups) {
                uint32_t r[16];
                tmem_ld16(lane_base + (uint32_t)c0, r);
                const int q = c0 / a.sw, cl = c0 - q * a.sw;
                const uint32_t dst =
                    send_base + (uint32_t)q * blk_bytes + (uint32_t)((m * a.rs + cl) * 4);
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4)
                    st_shared_v4(dst + 16 * v4, __uint_as_float(r[4 * v4]),
                                 __uint_as_float(r[4 * v4 + 1]), __uint_as_float(r[4 * v4 + 2]),
                                 __uint_as_float(r[4 * v4 + 3]));
            }
        }
        // 1. Every CTA of the cluster has staged its send blocks.
        cluster_sync_all();
        // 2. This CTA's column slice: read block `rank` of every CTA's send blocks (remote
        //    shared-memory loads, four columns at a time), add them in rank order, then the
        //    channel scale and bias, into the slice tile; one TMA store writes it out.
        if (warp >= 2) {
            const bool ok2 = __all_sync(0xffffffffu, epi_go);
            if (ok2) {
                float* slice = reinterpret_cast<float*>(gbase + (slice_base - base));
                const int cbase = rank * a.sw;
                const int q_shift = 31 - __clz(a.sw / 4);  // sw / 4 is a power of two
                const uint32_t my_blk = send_base + (uint32_t)rank * blk_bytes;
                for (int idx = threadIdx.x - 64; idx < kXRows * (a.sw / 4); idx += 128 * kGroups) {
                    const int m = idx >> q_shift, c = (idx & (a.sw / 4 - 1)) * 4;
                    const uint32_t off = my_blk + (uint32_t)((m * a.rs + c) * 4);
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int r = 0; r < P; ++r) {
                        const float4 t = ld_cluster_v4(map_shared_rank(off, (uint32_t)r));
                        v.x += t.x, v.y += t.y, v.z += t.z, v.w += t.w;
                    }
                    if (a.per_channel) {
                        v.x *= s_cscale[cbase + c], v.y *= s_cscale[cbase + c + 1];
                        v.z *= s_cscale[cbase + c + 2], v.w *= s_cscale[cbase + c + 3];
                    }
                    v.x += s_bias[cbase + c], v.y += s_bias[cbase + c + 1];
                    v.z += s_bias[cbase + c + 2], v.w += s_bias[cbase + c + 3];
                    *reinterpret_cast<float4*>(slice + m * a.sw + c) = v;
                }
                fence_proxy_async_smem();
            }
            asm volatile("bar.sync 2, %0;" ::"r"(128 * kGroups) : "memory");
            const int64_t ncol = (int64_t)ntile * bn + (int64_t)rank * a.sw;
            if (threadIdx.x == 64 && ok2 && !*failed && ncol < a.N) {
                tma_store_2d(&tmap_o, (int)ncol, (int)blockIdx.y * kXRows, slice_base);
                bulk_commit();
                bulk_wait_read();
            }
        }
        // 3. No CTA leaves while another may still read its send blocks.
        cluster_sync_all();
    }
    if (warp >= 2) tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_d, (uint32_t)a.tmem_cols);
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

template <int RPT, bool EH>
cudaError_t kernel_attr() {
    static cudaError_t attr = cudaFuncSetAttribute(
        tc_xa_kernel<RPT, EH>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    return attr;
}

int stages_for_bn(int bn, const LaunchCtx& c) {
    int stages = std::min(kMaxStages, (kSmemLimit - 1024 - 256 - 2048) / stage_bytes(bn));
    while (stages > 2 && smem_bytes(bn, stages) > c.max_smem_optin) --stages;
    return stages;
}

// How many clusters of P CTAs (tiles of bn weight rows) the device keeps resident at once
// (0 when that cannot be determined).  Cached per (device, bn, P).
int max_active_clusters(int bn, int P, const LaunchCtx& c) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_tuple(dev, bn, P);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(P * 64));
    cfg.blockDim = dim3(kThreads2);
    cfg.dynamicSmemBytes = smem_bytes(bn, stages_for_bn(bn, c));
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeClusterDimension;
    at.val.clusterDim.x = (unsigned)P;
    at.val.clusterDim.y = 1;
    at.val.clusterDim.z = 1;
    cfg.attrs = &at;
    cfg.numAttrs = 1;
    int n = 0;
    const cudaError_t e = bn > 128
        ? (kernel_attr<2, false>() == cudaSuccess
               ? cudaOccupancyMaxActiveClusters(&n, tc_xa_kernel<2, false>, &cfg) : cudaErrorUnknown)
        : (kernel_attr<1, false>() == cudaSuccess
               ? cudaOccupancyMaxActiveClusters(&n, tc_xa_kernel<1, false>, &cfg) : cudaErrorUnknown);
    if (e != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    cache[key] = n;
    return n;
}

template <int RPT, bool EH>
cudaError_t launch2(const CUtensorMap& tx, const CUtensorMap& tw, const CUtensorMap& to,
                    const CUtensorMap& twp, const Tc2Args& a, dim3 grid, const LaunchCtx& c) {
    const cudaError_t attr = kernel_attr<RPT, EH>();
    if (attr != cudaSuccess) return attr;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads2);
    cfg.dynamicSmemBytes = smem_bytes(a.bn, a.stages);
    cfg.stream = c.stream;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (c.pdl) {
        attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (a.splitk > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = (unsigned)a.splitk;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = na ? attrs : nullptr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, tc_xa_kernel<RPT, EH>, tx, tw, to, twp, a);
}

}  // namespace

bool tc_eligible(const Problem& p, const LaunchCtx& c) {
    if (p.K % kStageK != 0) return false;
    if (reinterpret_cast<uintptr_t>(p.x) % 16 || reinterpret_cast<uintptr_t>(p.qweight) % 16)
        return false;
    if (!(p.group_size >= p.K || p.group_size % kStageK == 0)) return false;
    if (p.M > 65535LL * kXRows || p.N > (1LL << 31) - 1) return false;
    if (c.max_smem_optin < smem_bytes(256, 4)) return false;
    return encode_fn() != nullptr;
}

cudaError_t tc_launch(const Problem& p, const LaunchCtx& c) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    // Weight rows per tile (the MMA's N) and the split of K over a cluster.  Wider tiles
    // make wider MMAs and feed more weight rows from each 16 KiB stage of x; narrower
    // ones give more CTAs.  When the tiles alone leave SMs idle, K is split over a
    // cluster of P CTAs (a power of two up to 8, at least 4 stages each, 16-column
    // slices).  Estimate: waves x stages per CTA x cycles per stage (an MMA stage costs
    // ~2 * bn cycles, a stage of x must arrive from L2, ~340 cycles at the L2 bandwidth
    // share of an SM when every SM streams, and the widening of bn rows needs ~bn cycles
    // of issue), plus ~2000 cycles for the exchange of partial tiles.
    const int64_t mtiles = (p.M + kXRows - 1) / kXRows;
    const int k_iters = (int)(p.K / kStageK);
    int bn = 256, splitk = 1;
    int64_t best = -1;
    for (int cand = 256; cand >= 64; cand /= 2) {
        const int64_t ntiles = (p.N + cand - 1) / cand;
        const int64_t tiles = ntiles * mtiles;
        // Split only into clusters that all stay resident at once (one wave), and only
        // with tiles of at most 128 rows (the exchange buffer must fit in the ring).
        int P = 1;
        while (P < 8 && cand <= 128 && tiles * P * 2 <= c.sm_count && k_iters % (2 * P) == 0 &&
               k_iters / (2 * P) >= 4 && cand / (2 * P) >= 16 && !c.tc_skip_first_copy &&
               max_active_clusters(cand, 2 * P, c) >= tiles)
            P *= 2;
        const int64_t ctas = tiles * P;
        const int64_t waves = (ctas + c.sm_count - 1) / c.sm_count;
        const int64_t busy = std::min<int64_t>(ctas, c.sm_count);
        const int64_t l2 = 340 * busy / c.sm_count;
        const int64_t cost = waves * (k_iters / P) * std::max<int64_t>({2LL * cand, l2, (int64_t)cand}) +
                             (P > 1 ? 2000 : 0);
        if (best < 0 || cost < best) {
            best = cost;
            bn = cand;
            splitk = P;
        }
    }
    const int stages = stages_for_bn(bn, c);
    int cols = 32;
    while (cols < bn) cols <<= 1;

    Tc2Args a;
    a.scales = p.scales;
    a.bias = p.bias;
    a.out = p.out;
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.scale_f16 = p.scale_f16;
    a.per_channel = p.group_size >= p.K;
    a.bn = bn;
    a.stages = stages;
    a.k_iters = k_iters;
    // The split-K exchange (send blocks [P][128][sw + 4] floats, the slice [128][sw]) must
    // fit in the stage ring, and its result goes out by TMA stores.
    if (!((reinterpret_cast<uintptr_t>(p.out) % 16 == 0) && (p.N % 4 == 0))) splitk = 1;
    while (splitk > 1 &&
           ((int64_t)splitk * kXRows * (bn / splitk + 4) + (int64_t)kXRows * (bn / splitk)) * 4 >
               (int64_t)stages * stage_bytes(bn))
        splitk /= 2;
    a.splitk = splitk;
    a.kpp = k_iters / splitk;
    a.sw = bn / splitk;
    a.rs = a.sw + 4;
    a.tmem_cols = cols;
    a.gs_stages = a.per_channel ? 1 : (int)(p.group_size / kStageK);
    a.gs_shift = -1;
    for (int sft = 0; sft < 31; ++sft)
        if ((1 << sft) == a.gs_stages) a.gs_shift = sft;
    a.out_vec = (reinterpret_cast<uintptr_t>(p.out) % 16 == 0) && (p.N % 4 == 0);
    a.tma_out = a.out_vec;
    a.w_prefetch = mtiles <= 2;
    a.status = c.status_word;
    a.wait_ns = c.wait_limit_ns;
    a.skip_first_copy = c.tc_skip_first_copy;

    CUtensorMap tx, tw;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)p.K, (cuuint64_t)p.M};
        const cuuint64_t strides[1] = {(cuuint64_t)p.K * 4};
        const cuuint32_t box[2] = {(cuuint32_t)kStageK, (cuuint32_t)kXRows};
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
        const cuuint32_t box[2] = {(cuuint32_t)(kStageK / 2), (cuuint32_t)bn};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(p.qweight), dims,
                strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    CUtensorMap twp;  // the packed weights in blocks of kWPrefetch stages (L2 prefetch)
    {
        const int64_t Kp = p.K / 2;
        const cuuint64_t dims[2] = {(cuuint64_t)Kp, (cuuint64_t)p.N};
        const cuuint64_t strides[1] = {(cuuint64_t)Kp};
        const cuuint32_t box[2] = {(cuuint32_t)(kWPrefetch * kStageK / 2), (cuuint32_t)bn};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&twp, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(p.qweight), dims,
                strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    CUtensorMap to = tx;  // unused unless a.tma_out
    if (a.tma_out) {
        // Non-split tiles: 32-column blocks in the 128-byte swizzle; split-K slices: sw
        // columns, unswizzled.
        const cuuint64_t dims[2] = {(cuuint64_t)p.N, (cuuint64_t)p.M};
        const cuuint64_t strides[1] = {(cuuint64_t)p.N * 4};
        const cuuint32_t box[2] = {(cuuint32_t)(splitk > 1 ? a.sw : 32), (cuuint32_t)kXRows};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&to, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p.out, dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE,
                splitk > 1 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const dim3 grid((unsigned)((p.N + bn - 1) / bn * splitk), (unsigned)mtiles);
    const bool eh = p.even_high != 0;
    if (bn > 128)
        return eh ? launch2<2, true>(tx, tw, to, twp, a, grid, c)
                  : launch2<2, false>(tx, tw, to, twp, a, grid, c);
    return eh ? launch2<1, true>(tx, tw, to, twp, a, grid, c)
              : launch2<1, false>(tx, tw, to, twp, a, grid, c);
}

}  // namespace q4lin
