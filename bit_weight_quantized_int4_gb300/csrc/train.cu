// train.cu -- training-path kernels on the same packed 4-bit weights (sm_103a).
//
// Input gradient of the linear (the frozen 4-bit base during adapter training):
//
//   d_x[m,k] = sum_n d_out[m,n] * (code[n,k] - 8) * scale[k / gs, n]
//
// ("[ExecuTorch][WebGPU] Add fp32 matmul ops ... (linear_q4gsw_backward)", #20943:
// d_x[M,K] = d_out[M,N] @ dequant(W)[N,K], contracting over N, with the forward's weight
// and scale layout.)  HBM-bound for a few activation rows: every packed byte is read once
// per tile of 8 rows of d_out.
//   backward_dx_kernel: a CTA owns 256 consecutive k (32 lanes x 8 k, one 32-bit word of
//     codes per lane and row: a warp reads 128 contiguous bytes of a weight row) and a
//     range of rows n; its 8 warps take every 8th row of the range.  Per row, the group
//     scale of the lane's 8 k (a group holds whole multiples of 8 k) is folded into the
//     d_out values (MT products, MT = 1, 2, 4 or 8 rows of d_out per pass), and each code
//     is widened with the byte-permute trick of
//     the forward (2^23 + byte, minus 2^23 + 8) and accumulated with MT FMAs.  The 8 warps'
//     partial sums are added in warp order through shared memory.  When the rows are split
//     over several CTAs (few k tiles), each writes its partial [MT, 256] tile to the
//     handle's workspace and the last CTA of the k tile (an atomic ticket) adds the parts
//     in split order: the result does not depend on which CTA finishes last.
//   backward_tma_kernel (the fast path when the tensors suit TMA): the same CTA tile of
//     256 k, fed by a producer warp that streams per stage the weight tile [64 rows x
//     128 B], the group scales of those rows [groups of the tile x 64] and d_out
//     [MT x 64] into a shared-memory ring with one TMA copy each; 8 consumer warps (16 for
//     1-2 rows of d_out on rows of >= 8192 k) take every 8th (16th) row of a stage (lane =
//     32-bit word of codes, 8 k).  For 1-2 rows of d_out on 2048-k rows of 4096-16384
//     rows the tile is 128 k (two rows per warp pass), which puts twice the CTAs on the
//     SMs.  The weight and scale
//     copies of the first ring of stages go out before the grid-dependency wait, their
//     d_out copies after it.  The rows are split over CTAs (multiples of 64 rows each);
//     when each CTA has at most 4 stages, the splits of a k tile are one thread-block
//     cluster that adds its partial tiles through distributed shared memory (in rank
//     order), else the partials are added through the workspace like above.
//   backward_dx_generic_kernel: one thread per (m, k), n ascending; any K, any group size,
//     any alignment.
//
// Re-quantisation of fp32 latent weights with frozen scales, packed like the forward
// reads them (low nibble = even k, or swapped when even_high):
//
//   code[n,k] = clamp(round(latent[n,k] / scale[k / gs, n]), -8, 7) + 8,  zero scale -> 8
//
// ("[ExecuTorch][WebGPU] Add fp32 matmul ops ... (q4gsw_requant)", #20945.)  The quotient
// is the IEEE fp32 quotient (__fdiv_rn), rounded half to even (rintf); a NaN quotient gives
// code 8, like a zero scale; for odd K the padding nibble is 8.
//   requant_wide_kernel: one thread per 16 k of a row (four float4 loads of latents in flight,
//     one 8-byte store); consecutive threads walk a row (coalesced loads and stores).
//   requant_kernel: the same with 4 k per thread (K % 4 == 0).
//   requant_generic_kernel: one thread per output byte (any K, any alignment).
#include <cuda_fp16.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "ptx.cuh"
#include "q4lin_internal.h"

namespace q4lin {
namespace {
using namespace ptx;

constexpr int kBwThreads = 256;
constexpr int kBwWarps = kBwThreads / 32;
constexpr int kBwK = 256;  // k per CTA tile: 32 lanes x 8
constexpr int kMT = 8;     // largest tile of d_out rows per pass

struct BwArgs {
    const float* d_out;
    const uint8_t* w;
    const void* scales;
    float* d_x;
    int64_t M, N, K, Kp, gs;
    int scale_f16, even_high;
    int k_tiles, splits;
    int64_t rows_per_split;
    float* ws;     // [splits][M][K] partials (splits > 1)
    int* tickets;  // [m_tiles * k_tiles], zero between launches
};

__device__ __forceinline__ float scale_value(const void* scales, int f16, int64_t idx) {
    if (f16) return __half2float(__ldg(reinterpret_cast<const __half*>(scales) + idx));
    return __ldg(reinterpret_cast<const float*>(scales) + idx);
}

// grid: x = k tile, y = split of the rows, z = tile of MT rows of d_out.  RB weight rows
// per warp are in flight at once (more when the d_out tile is short).
template <int MT>
__global__ void __launch_bounds__(kBwThreads, 2) backward_dx_kernel(const BwArgs a) {
    constexpr int kRB = MT >= 8 ? 4 : 32 / MT > 16 ? 16 : 32 / MT;
    constexpr int kHalf = MT >= 2 ? MT / 2 : 1;  // d_out rows per shared-memory pass
    __shared__ float red[kBwWarps][kHalf][kBwK];  // per-warp partial tiles
    __shared__ int s_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t k0 = (int64_t)blockIdx.x * kBwK + lane * 8;
    const int64_t m0 = (int64_t)blockIdx.z * MT;
    const int mt = a.M - m0 < MT ? (int)(a.M - m0) : MT;
    const int64_t n_begin = (int64_t)blockIdx.y * a.rows_per_split;
    const int64_t n_end = n_begin + a.rows_per_split < a.N ? n_begin + a.rows_per_split : a.N;
    const bool k_ok = k0 < a.K;  // K % 8 == 0: a lane's 8 k are all in or all out
    griddep_wait();

    float acc[MT][8];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[m][j] = 0.f;
    const int64_t g = k0 / a.gs;  // one group for the lane's 8 k (gs % 8 == 0)
    constexpr float kMagic = 8388616.0f;  // 2^23 + 8
    // Rows in batches of kRB per warp, every load of a batch issued before any use (the
    // rows are independent: kRB loads in flight per lane instead of one).
    for (int64_t nb = n_begin + warp; nb < n_end && k_ok; nb += kRB * kBwWarps) {
        uint32_t word[kRB];
        float s[kRB], dv[kRB][MT];
#pragma unroll
        for (int r = 0; r < kRB; ++r) {
            const int64_t n = nb + r * kBwWarps;
            const bool ok = n < n_end;
            word[r] = ok ? __ldg(reinterpret_cast<const uint32_t*>(a.w + n * a.Kp + k0 / 2))
                         : 0x88888888u;  // codes 8: contribute nothing
            s[r] = ok ? scale_value(a.scales, a.scale_f16, g * a.N + n) : 0.f;
#pragma unroll
            for (int m = 0; m < MT; ++m)
                dv[r][m] = (ok && m < mt) ? __ldg(a.d_out + (m0 + m) * a.N + n) : 0.f;
        }
#pragma unroll
        for (int r = 0; r < kRB; ++r) {
            float ds[MT];
#pragma unroll
            for (int m = 0; m < MT; ++m) ds[m] = dv[r][m] * s[r];
            const uint32_t lo = word[r] & 0x0F0F0F0Fu, hi = (word[r] >> 4) & 0x0F0F0F0Fu;
            const uint32_t ev = a.even_high ? hi : lo, od = a.even_high ? lo : hi;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const float ce = __uint_as_float(prmt(ev, 0x4B000000u, 0x7440u | b)) - kMagic;
                const float co = __uint_as_float(prmt(od, 0x4B000000u, 0x7440u | b)) - kMagic;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    acc[m][2 * b] = fmaf(ds[m], ce, acc[m][2 * b]);
                    acc[m][2 * b + 1] = fmaf(ds[m], co, acc[m][2 * b + 1]);
                }
            }
        }
    }
    // The CTA's partial tile, the 8 warps added in warp order through shared memory (two
    // halves of the d_out rows): thread t owns column t.
    const int c = threadIdx.x;
    const int64_t k = (int64_t)blockIdx.x * kBwK + c;
    float part[MT];
#pragma unroll
    for (int h0 = 0; h0 < MT; h0 += kHalf) {
#pragma unroll
        for (int m = 0; m < kHalf; ++m)
#pragma unroll
            for (int j = 0; j < 8; ++j) red[warp][m][lane * 8 + j] = acc[h0 + m][j];
        __syncthreads();
#pragma unroll
        for (int m = 0; m < kHalf; ++m) {
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < kBwWarps; ++w) v += red[w][m][c];
            part[h0 + m] = v;
        }
        __syncthreads();
    }
    if (a.splits == 1) {
        if (k < a.K)
            for (int m = 0; m < mt; ++m) a.d_x[(m0 + m) * a.K + k] = part[m];
        return;
    }
    // Split rows: partials to the workspace; the last CTA of this (m tile, k tile) adds
    // them in split order.
    if (k < a.K)
        for (int m = 0; m < mt; ++m)
            a.ws[((int64_t)blockIdx.y * a.M + m0 + m) * a.K + k] = part[m];
    // Partials before the ticket: the CTA barrier and one device-scope fence of the thread
    // that takes it; the last CTA's reads after it: that thread's second fence and barrier.
    __syncthreads();
    const int item = (int)(blockIdx.z * gridDim.x + blockIdx.x);
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = atomicAdd(a.tickets + item, 1) == a.splits - 1;
        __threadfence();
    }
    __syncthreads();
    if (!s_last) return;
    if (k < a.K)
        for (int m = 0; m < mt; ++m) {
            // Loads of 8 parts in flight at a time; still added in split order.
            const float* src = a.ws + (m0 + m) * a.K + k;
            const int64_t stride = a.M * a.K;
            float v = 0.f;
            int sp = 0;
            for (; sp + 8 <= a.splits; sp += 8) {
                float t[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) t[u] = __ldcg(src + (int64_t)(sp + u) * stride);
#pragma unroll
                for (int u = 0; u < 8; ++u) v += t[u];
            }
            for (; sp < a.splits; ++sp) v += __ldcg(src + (int64_t)sp * stride);
            a.d_x[(m0 + m) * a.K + k] = v;
        }
    if (threadIdx.x == 0) a.tickets[item] = 0;
}

__global__ void backward_dx_generic_kernel(const BwArgs a) {
    griddep_wait();
    const int64_t total = a.M * a.K;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = i / a.K, k = i % a.K;
        const int64_t g = k / a.gs;
        float acc = 0.f;
        for (int64_t n = 0; n < a.N; ++n) {
            const uint8_t byte = __ldg(a.w + n * a.Kp + k / 2);
            const bool low = ((k & 1) == 0) != (a.even_high != 0);
            const int code = low ? (byte & 0xF) : (byte >> 4);
            const float w = (float)(code - 8) * scale_value(a.scales, a.scale_f16, g * a.N + n);
            acc = fmaf(__ldg(a.d_out + m * a.N + n), w, acc);
        }
        a.d_x[i] = acc;
    }
}

// ------------------------------------------------------- TMA-fed input gradient
// Consumer warps CW: 8, or 16 for tiles of 1-2 rows of d_out on long rows (K >= 8192),
// where each CTA's loop is long enough for the extra warps to hide its latency (2048 x 8192
// at M = 1: 8.7 -> 7.1 us); on shorter rows the larger reduction and barriers cost more
// than they hide (8192 x 2048: 9.1 -> 9.5 us).  One producer warp besides.
constexpr int kBtKT = 256;                         // k per CTA tile: 128 bytes of a row
constexpr int kBtKTNarrow = 128;                   // or 64 bytes (more CTAs on short K)
constexpr int kBtRB = 64;                          // weight rows per stage
constexpr int kBtMaxStages = 8;
constexpr int64_t kDrainNs = 4000000000LL;
__host__ __device__ constexpr uint32_t bt_sc_off(int kt) { return kBtRB * kt / 2; }  // codes, then scales
// Scales are copied for 72 rows (fp16: 144-byte box rows) or 68 rows (fp32: 272 bytes): the
// lanes of a warp read up to 8 groups of one row, and the padded row stride puts them in
// different banks (a box row must be a multiple of 16 bytes).
constexpr int kBtScRows16 = kBtRB + 8, kBtScRows32 = kBtRB + 4;
__host__ __device__ constexpr uint32_t bt_do_off(int kt) { return bt_sc_off(kt) + 2304; }  // then d_out [MT x 64]

struct BtMaps {
    CUtensorMap w;   // uint8 [N, Kp], box {128, 64}
    CUtensorMap s;   // scales [G, N] (fp16 / fp32), box {64, GT}
    CUtensorMap d;   // d_out fp32 [M, N], box {64, MT}
};

struct BtArgs {
    float* d_x;
    float* ws;     // [m tiles x k tiles][splits][MT][256] partials (splits > 1)
    int* tickets;  // [m tiles x k tiles], zero between launches
    int* status;
    int64_t M, N, K;
    int gs_in_tile;       // group size when a k tile holds whole groups (gs <= 256), else 0
    int gs_shift256;      // then: group row of k tile kt = kt << gs_shift256
    int tiles_per_group;  // else: group row = kt / tiles_per_group
    int scale_f16, even_high;
    int sc_rows;  // staged scale rows per group (72 / 68)
    int splits, stages;
    int64_t rows_per_split;  // multiple of 64
    int cluster;             // > 1: the splits of a k tile form one cluster (splits == cluster)
    uint32_t stage_bytes, tx;
    int64_t wait_ns;
};

// grid: x = k tile, y = split of the rows, z = tile of MT rows of d_out.
template <int MT, int CW, int KT>
__global__ void __launch_bounds__(32 * CW + 32, 2)
    backward_tma_kernel(const __grid_constant__ BtMaps maps, const BtArgs a) {
    constexpr int kBtCWarps = CW;
    constexpr uint32_t kScOff = bt_sc_off(KT), kDoOff = bt_do_off(KT);
    // Lanes per weight row (one 32-bit word of codes, 8 k, each) and rows per warp pass.
    constexpr int LPR = KT / 8, RPI = 32 / LPR;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const int S = a.stages;
    // The partial-tile reduction reuses the ring: max(ring, [warps][MT][256] floats).
    const uint32_t ring = (uint32_t)S * a.stage_bytes;
    const uint32_t red_bytes = (uint32_t)kBtCWarps * MT * KT * 4;
    const uint32_t bar_base = base + (ring > red_bytes ? ring : red_bytes);
    volatile int* failed = reinterpret_cast<volatile int*>(gbase + (bar_base + 16 * kBtMaxStages - base));
    volatile int* s_last = failed + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto full = [&](int s) { return bar_base + 8u * s; };
    auto empty = [&](int s) { return bar_base + 8u * (kBtMaxStages + s); };

    const int kt = (int)blockIdx.x;
    const int64_t m0 = (int64_t)blockIdx.z * MT;
    const int64_t n_begin = (int64_t)blockIdx.y * a.rows_per_split;
    const int64_t n_end = n_begin + a.rows_per_split < a.N ? n_begin + a.rows_per_split : a.N;
    const int nst = n_end > n_begin ? (int)((n_end - n_begin + kBtRB - 1) / kBtRB) : 0;
    const int g_row = a.gs_in_tile ? kt << a.gs_shift256 : kt / a.tiles_per_group;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), kBtCWarps);
        }
        *failed = 0;
        mbar_init_fence();
    }
    __syncthreads();
    griddep_launch_dependents();

    if (warp == kBtCWarps) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tensormap(&maps.w);
            prefetch_tensormap(&maps.s);
            prefetch_tensormap(&maps.d);
            // The weights and scales do not depend on the preceding grid: the first ring of
            // stages streams them before griddepcontrol.wait, and only the d_out copies of
            // those stages wait for the release.  Their barriers count the weight bytes first
            // (expect_tx, no arrival; the phase cannot complete before the arrival) and the
            // d_out bytes with the one arrival after the wait.
            const int pre = nst < S ? nst : S;
            const uint32_t d_bytes = (uint32_t)(MT * kBtRB * 4);
            for (int li = 0; li < pre; ++li) {
                const int n = (int)(n_begin + (int64_t)li * kBtRB);
                const uint32_t sb = base + (uint32_t)li * a.stage_bytes;
                mbar_expect_tx(full(li), a.tx - d_bytes);
                tma_load_2d(sb, &maps.w, kt * (KT / 2), n, full(li));
                tma_load_2d(sb + kScOff, &maps.s, n, g_row, full(li));
            }
            griddep_wait();  // d_out comes from the preceding grid
            int li = 0, s = 0;
            uint32_t ph = 0;
            for (; li < nst; ++li) {
                if (li >= S && !wait_bounded(empty(s), ph ^ 1u, a.wait_ns, failed)) {
                    record_failure(a.status, failed);
                    break;
                }
                if (*failed) break;
                const int n = (int)(n_begin + (int64_t)li * kBtRB);
                const uint32_t sb = base + (uint32_t)s * a.stage_bytes;
                if (li < pre) {
                    mbar_arrive_expect_tx(full(s), d_bytes);
                } else {
                    mbar_arrive_expect_tx(full(s), a.tx);
                    tma_load_2d(sb, &maps.w, kt * (KT / 2), n, full(s));
                    tma_load_2d(sb + kScOff, &maps.s, n, g_row, full(s));
                }
                tma_load_2d(sb + kDoOff, &maps.d, n, (int)m0, full(s));
                if (++s == S) s = 0, ph ^= 1u;
            }
            // After a failure: the stages armed before the wait but not yet arrived on get
            // their arrival without a d_out copy, so that their phases complete when their
            // weight copies land; then the last armed copies are drained (the CTA must not
            // exit while copies into its shared memory are in flight).
            for (int q = li; q < pre; ++q) mbar_arrive(full(q));
            const int issued = li > pre ? li : pre;
            for (int q = issued > S ? issued - S : 0; q < issued; ++q)
                wait_bounded(full(q % S), (uint32_t)(q / S) & 1u, kDrainNs, nullptr);
        }
        if (a.cluster > 1) {
            // The producer warp takes part in the cluster's two barriers (below).
            __syncwarp();
            cluster_sync_all();
            cluster_sync_all();
        }
        return;
    }

    // ------------------------------------------------------------------ consumers
    // Lane = 32-bit word wl of codes (k = KT kt + 8 wl + j) of row hr of a pass: a warp
    // takes rows RPI (warp + CW i) + hr of every stage (one row per pass with 256-k tiles,
    // two with 128-k tiles); gl = the lane's group inside the tile.
    const int wl = lane % LPR, hr = lane / LPR;
    const int gl = a.gs_in_tile ? (wl * 8) / a.gs_in_tile : 0;
    // acc[m][b] = (k = 2b, k = 2b + 1) of the lane's 8 k: packed fp32x2 FMAs.
    float2 acc[MT][4];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[m][b] = make_float2(0.f, 0.f);
    int s = 0;
    uint32_t ph = 0;
    // After a timed-out wait (`dead`) the warp still walks every stage, without waiting or
    // computing, so that the consumer barriers and the split ticket are still reached.
    bool dead = false;
    for (int li = 0; li < nst; ++li) {
        const bool got =
            !dead && __all_sync(0xffffffffu, wait_bounded(full(s), ph, a.wait_ns, failed));
        if (!got && !dead) {
            if (lane == 0) record_failure(a.status, failed);
            dead = true;
        }
        if (got) {
            const uint8_t* stage = gbase + (uint32_t)s * a.stage_bytes;
            const uint32_t* wrow = reinterpret_cast<const uint32_t*>(stage) + wl;
            const __half* sc16 = reinterpret_cast<const __half*>(stage + kScOff) + gl * a.sc_rows;
            const float* sc32 = reinterpret_cast<const float*>(stage + kScOff) + gl * a.sc_rows;
            const float* dop = reinterpret_cast<const float*>(stage + kDoOff);
#pragma unroll 4
            for (int rr = 0; rr < kBtRB / (kBtCWarps * RPI); ++rr) {
                const int r = (warp + rr * kBtCWarps) * RPI + hr;
                const uint32_t word = wrow[r * (KT / 8)];
                const float sc = a.scale_f16 ? __half2float(sc16[r]) : sc32[r];
                float2 cv[4];  // (c - 8) of k = 2b, 2b + 1, exact
                if (a.even_high)
                    codes_word<true>(word, cv);
                else
                    codes_word<false>(word, cv);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const float d = dop[m * kBtRB + r] * sc;
                    const float2 d2 = make_float2(d, d);
#pragma unroll
                    for (int b = 0; b < 4; ++b) acc[m][b] = ffma2(d2, cv[b], acc[m][b]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(s));
        if (++s == S) s = 0, ph ^= 1u;
    }
    // The CTA's partial tile: the consumer warps added in warp order through shared memory
    // (the ring is free once every consumer warp has passed its last stage).
    if (RPI == 2) {
        // The warp's two rows of a pass are the same columns: half-warp hr = 1 adds onto 0.
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                acc[m][b].x += __shfl_down_sync(0xffffffffu, acc[m][b].x, LPR);
                acc[m][b].y += __shfl_down_sync(0xffffffffu, acc[m][b].y, LPR);
            }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kBtCWarps * 32) : "memory");
    float* red = reinterpret_cast<float*>(gbase);  // [warps][MT][KT]
    if (hr == 0)
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            float4* dst = reinterpret_cast<float4*>(red + (warp * MT + m) * KT + wl * 8);
            dst[0] = make_float4(acc[m][0].x, acc[m][0].y, acc[m][1].x, acc[m][1].y);
            dst[1] = make_float4(acc[m][2].x, acc[m][2].y, acc[m][3].x, acc[m][3].y);
        }
    asm volatile("bar.sync 1, %0;" ::"r"(kBtCWarps * 32) : "memory");
    const int mt = a.M - m0 < MT ? (int)(a.M - m0) : MT;
    // Consumer thread c < KT = column c of the tile (the others only take part in the
    // barriers).
    const int c = threadIdx.x;
    const bool col = kBtCWarps * 32 <= KT || c < KT;  // always, with 8 warps and 256-k tiles
    const int cc0 = col ? c : 0;
    const int64_t k = (int64_t)kt * KT + c;
    float part[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kBtCWarps; ++w) v += red[(w * MT + m) * KT + cc0];
        part[m] = v;
    }
    griddep_wait();  // (long complete: the d_out copies waited for it) before any store
    const bool store = !dead && !*failed;
    if (a.cluster > 1) {
        // The splits of this k tile are the CTAs of one cluster: each leaves its partial
        // tile [MT][256] in its own shared memory (warp 0's slots of `red`: column c was
        // read above by this thread only), and after the cluster barrier CTA rank r adds
        // columns [r * 256 / cluster, (r + 1) * 256 / cluster) of the MT rows over the
        // ranks in rank order (the result does not depend on timing) and stores them.
        // Thread c fetches column r * per + c % per of rank c / per for every row, all MT
        // remote loads in flight at once, into a local [MT][cluster][per] array (the other
        // warps' slots of `red`, free after the barrier); the rank-ordered sums then read
        // that.  No CTA leaves before the second barrier, so its partial stays readable.
        if (col)
#pragma unroll
            for (int m = 0; m < MT; ++m) red[m * KT + c] = part[m];
        cluster_sync_all();
        const uint32_t rank = cluster_ctarank();
        const int cs = a.cluster, per = KT / cs;
        float* stage = red + MT * KT;  // [MT][cs][per]
        if (col) {
            const int q = c / per, j = c % per, cl = (int)rank * per + j;
            const uint32_t src = mapa_shared(base + (uint32_t)cl * 4u, (uint32_t)q);
            float got[MT];
#pragma unroll
            for (int m = 0; m < MT; ++m) got[m] = ld_dsmem_f32(src + (uint32_t)(m * KT) * 4u);
#pragma unroll
            for (int m = 0; m < MT; ++m) stage[m * KT + c] = got[m];
        }
        asm volatile("bar.sync 1, %0;" ::"r"(kBtCWarps * 32) : "memory");
        for (int e = c; e < MT * per; e += kBtCWarps * 32) {
            const int m = e / per, jj = e % per, cc = (int)rank * per + jj;
            const float* sp = stage + m * KT + jj;
            float v = 0.f;
            for (int r = 0; r < cs; ++r) v += sp[r * per];
            const int64_t kk = (int64_t)kt * KT + cc;
            if (store && m < mt && kk < a.K) a.d_x[(m0 + m) * a.K + kk] = v;
        }
        cluster_sync_all();
        return;
    }
    if (a.splits == 1) {
        if (store && col && k < a.K)
            for (int m = 0; m < mt; ++m) a.d_x[(m0 + m) * a.K + k] = part[m];
        return;
    }
    // Split rows: partials to the workspace; the last CTA of this (m tile, k tile) adds
    // them in split order.
    const int64_t item = (int64_t)blockIdx.z * gridDim.x + blockIdx.x;
    float* wsi = a.ws + item * (int64_t)a.splits * MT * KT;
    if (col)
#pragma unroll
        for (int m = 0; m < MT; ++m) wsi[((int64_t)blockIdx.y * MT + m) * KT + c] = part[m];
    // Partials before the ticket: the barrier and one device-scope fence of the thread that
    // takes it; the last CTA's reads after it: that thread's second fence and barrier.
    asm volatile("bar.sync 1, %0;" ::"r"(kBtCWarps * 32) : "memory");
    if (threadIdx.x == 0) {
        __threadfence();
        *s_last = atomicAdd(a.tickets + item, 1) == a.splits - 1;
        __threadfence();
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kBtCWarps * 32) : "memory");
    if (!*s_last || !col) return;
    // The MT rows of the column together, the loads of PB parts of all of them in flight
    // at a time (MT * PB <= 32); every row still added in split order.
    constexpr int PB = MT >= 8 ? 4 : 32 / MT > 8 ? 8 : 32 / MT;
    const float* src = wsi + c;
    const int64_t stride = (int64_t)MT * KT;
    float v[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) v[m] = 0.f;
    for (int sp = 0; sp < a.splits; sp += PB) {
        float t[PB][MT];
#pragma unroll
        for (int u = 0; u < PB; ++u)
#pragma unroll
            for (int m = 0; m < MT; ++m)
                t[u][m] = sp + u < a.splits ? __ldcg(src + (int64_t)(sp + u) * stride + m * KT)
                                            : 0.f;
#pragma unroll
        for (int u = 0; u < PB; ++u)
#pragma unroll
            for (int m = 0; m < MT; ++m)
                if (sp + u < a.splits) v[m] += t[u][m];
    }
    if (store && !*failed && k < a.K)
#pragma unroll
        for (int m = 0; m < MT; ++m)
            if (m < mt) a.d_x[(m0 + m) * a.K + k] = v[m];
    if (threadIdx.x == 0) a.tickets[item] = 0;
}

struct RqArgs {
    const float* latent;
    const void* scales;
    uint8_t* w;
    int64_t N, K, Kp, gs;
    int scale_f16, even_high;
};

// The code of one latent: the fp32 quotient (correctly rounded division), converted to an
// integer rounding half to even (cvt.rni, which saturates and maps NaN to 0, i.e. code 8),
// clamped to [-8, 7] and offset by 8; a zero scale gives code 8.
__device__ __forceinline__ int requant_code(float l, float s) {
    const int c = s == 0.f ? 0 : __float2int_rn(__fdiv_rn(l, s));
    return min(max(c, -8), 7) + 8;
}

// One thread per 4 consecutive k (one float4 of latents, two output bytes); K % 4 == 0,
// 16-byte aligned latent rows.  A warp reads 512 contiguous bytes and writes 64.
__global__ void requant_kernel(const RqArgs a) {
    griddep_wait();
    const int64_t quads = a.K / 4;
    const int64_t total = a.N * quads;
    const int gs = (int)(a.gs < a.K ? a.gs : a.K);  // gs >= K: one group
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = i / quads;
        const int k0 = (int)(i - n * quads) * 4;
        const float4 u = __ldg(reinterpret_cast<const float4*>(a.latent + n * a.K + k0));
        const float l[4] = {u.x, u.y, u.z, u.w};
        int code[4];
        if (gs % 4 == 0) {  // the 4 k share one group
            const float sc = scale_value(a.scales, a.scale_f16, (int64_t)(k0 / gs) * a.N + n);
#pragma unroll
            for (int j = 0; j < 4; ++j) code[j] = requant_code(l[j], sc);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                code[j] = requant_code(l[j], scale_value(a.scales, a.scale_f16,
                                                         (int64_t)((k0 + j) / gs) * a.N + n));
        }
        const uint32_t b0 = a.even_high ? (code[1] | (code[0] << 4)) : (code[0] | (code[1] << 4));
        const uint32_t b1 = a.even_high ? (code[3] | (code[2] << 4)) : (code[2] | (code[3] << 4));
        *reinterpret_cast<uint16_t*>(a.w + n * a.Kp + k0 / 2) = (uint16_t)(b0 | (b1 << 8));
    }
}

// One thread per 4 * Q consecutive k of a row (Q = 4 or 8): Q float4 loads of latents in
// flight, one store of 2 * Q code bytes; K % (4 * Q) == 0, 16-byte aligned latents,
// (2 * Q)-byte aligned codes.  The nibble order is a template parameter.
template <int Q, bool EH>
__global__ void requant_wide_kernel(const RqArgs a) {
    constexpr int KC = 4 * Q;  // k per thread
    griddep_wait();
    const int64_t chunks = a.K / KC;
    const int64_t total = a.N * chunks;
    const int gs = (int)(a.gs < a.K ? a.gs : a.K);  // gs >= K: one group
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = i / chunks;
        const int k0 = (int)(i - n * chunks) * KC;
        const float4* src = reinterpret_cast<const float4*>(a.latent + n * a.K + k0);
        float l[KC];
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            const float4 u = __ldg(src + q);
            l[4 * q] = u.x, l[4 * q + 1] = u.y, l[4 * q + 2] = u.z, l[4 * q + 3] = u.w;
        }
        int code[KC];
        if (gs % 16 == 0) {  // every 16 k share one group
#pragma unroll
            for (int h = 0; h < KC / 16; ++h) {
                const float sc =
                    scale_value(a.scales, a.scale_f16, (int64_t)((k0 + 16 * h) / gs) * a.N + n);
#pragma unroll
                for (int j = 0; j < 16; ++j) code[16 * h + j] = requant_code(l[16 * h + j], sc);
            }
        } else {
#pragma unroll
            for (int j = 0; j < KC; ++j)
                code[j] = requant_code(l[j], scale_value(a.scales, a.scale_f16,
                                                         (int64_t)((k0 + j) / gs) * a.N + n));
        }
        uint32_t word[KC / 8];
#pragma unroll
        for (int h = 0; h < KC / 8; ++h) {
            uint32_t w = 0;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int e = code[8 * h + 2 * b], o = code[8 * h + 2 * b + 1];
                w |= (uint32_t)(EH ? (o | (e << 4)) : (e | (o << 4))) << (8 * b);
            }
            word[h] = w;
        }
        uint8_t* dst = a.w + n * a.Kp + k0 / 2;
        if (Q == 8)
            *reinterpret_cast<uint4*>(dst) = make_uint4(word[0], word[1 % (KC / 8)],
                                                        word[2 % (KC / 8)], word[3 % (KC / 8)]);
        else
            *reinterpret_cast<uint2*>(dst) = make_uint2(word[0], word[1 % (KC / 8)]);
    }
}

__global__ void requant_generic_kernel(const RqArgs a) {
    griddep_wait();
    const int64_t total = a.N * a.Kp;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = i / a.Kp, b = i % a.Kp;
        int codes[2] = {8, 8};
        for (int j = 0; j < 2; ++j) {
            const int64_t k = 2 * b + j;
            if (k >= a.K) break;
            codes[j] = requant_code(__ldg(a.latent + n * a.K + k),
                                    scale_value(a.scales, a.scale_f16, (k / a.gs) * a.N + n));
        }
        const int low = a.even_high ? codes[1] : codes[0];
        const int high = a.even_high ? codes[0] : codes[1];
        a.w[i] = (uint8_t)(low | (high << 4));
    }
}

template <typename Kern, typename Args>
cudaError_t launch(Kern k, const Args& a, dim3 grid, unsigned block, const LaunchCtx& c) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(block);
    cfg.stream = c.stream;
    cudaLaunchAttribute attrs[1];
    if (c.pdl) {
        attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attrs;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, k, a);
}

constexpr int kBtSmemLimit = 113 * 1024;  // two CTAs per SM

template <int MT, int CW, int KT>
cudaError_t launch_bt(const BtMaps& maps, const BtArgs& a, dim3 grid, int smem,
                      const LaunchCtx& c) {
    const cudaError_t attr = kernel_smem_once<backward_tma_kernel<MT, CW, KT>>(kBtSmemLimit);
    if (attr != cudaSuccess) return attr;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(32 * CW + 32);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = c.stream;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (c.pdl) {
        attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (a.cluster > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = 1;
        attrs[na].val.clusterDim.y = (unsigned)a.cluster;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = na ? attrs : nullptr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, backward_tma_kernel<MT, CW, KT>, maps, a);
}

// Whether clusters of `cs` CTAs (along y) of the MT instance with `smem` bytes can be
// resident on this device (cs > 8 needs the non-portable cluster size).  Cached per
// device, instance, cluster size and shared-memory size.
template <int MT, int CW, int KT>
bool bt_cluster_ok(int cs, int smem) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int>, bool> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const auto key = std::make_tuple(dev, cs, smem);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    bool ok = kernel_smem_once<backward_tma_kernel<MT, CW, KT>>(kBtSmemLimit) == cudaSuccess;
    if (ok && cs > 8)
        ok = cudaFuncSetAttribute(backward_tma_kernel<MT, CW, KT>,
                                  cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
    int n = 0;
    if (ok) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, (unsigned)cs, 1);
        cfg.blockDim = dim3(32 * CW + 32);
        cfg.dynamicSmemBytes = (size_t)smem;
        cudaLaunchAttribute at;
        at.id = cudaLaunchAttributeClusterDimension;
        at.val.clusterDim.x = 1;
        at.val.clusterDim.y = (unsigned)cs;
        at.val.clusterDim.z = 1;
        cfg.attrs = &at;
        cfg.numAttrs = 1;
        ok = cudaOccupancyMaxActiveClusters(&n, backward_tma_kernel<MT, CW, KT>, &cfg) == cudaSuccess && n > 0;
    }
    if (!ok) cudaGetLastError();
    cache[key] = ok;
    return ok;
}

// TMA needs 16-byte aligned bases and row strides (K % 32, N % 8) and a k tile of 256
// that holds whole groups or lies inside one (then so does a tile of 128).
bool bt_eligible(const TrainProblem& p) {
    auto al16 = [](const void* q) { return reinterpret_cast<uintptr_t>(q) % 16 == 0; };
    if (p.K % 32 != 0 || p.N % 8 != 0) return false;
    if (!al16(p.qweight) || !al16(p.scales) || !al16(p.d_out)) return false;
    const int64_t gs = p.group_size;
    if (gs < p.K && !(gs % 32 == 0 && ((gs <= kBtKT && kBtKT % gs == 0) || gs % kBtKT == 0)))
        return false;
    return tensor_map_encoder() != nullptr;
}

cudaError_t backward_tma_launch(const TrainProblem& p, const LaunchCtx& c) {
    EncodeTiledFn enc = tensor_map_encoder();
    const int MT = p.M <= 1 ? 1 : p.M <= 2 ? 2 : p.M <= 4 ? 4 : kMT;
    const bool wide = MT <= 2 && p.K >= 8192;  // 16 consumer warps (see backward_tma_kernel)
    const int CW = wide ? 16 : 8;
    // 128-k tiles (two rows per warp pass) where 256-k tiles in clusters of 16 would leave
    // SMs idle: 1-2 rows of d_out, fewer than sm_count / 16 tiles of 256 k, and 4-16 stages
    // of 64 rows per CTA of a 16-CTA cluster (8192 x 2048 at M = 1: 128 CTAs -> 256, 9.2 ->
    // 8.7 us).  With fewer rows the extra CTAs only add latency (2048 x 2048: 3.6 -> 4.5 us),
    // with more the clusters do not apply and the workspace hand-off grows (128256 x 2048:
    // 46.4 -> 51.2 us).
    const bool narrow = MT <= 2 && !wide && (p.K + kBtKT - 1) / kBtKT * 16 < c.sm_count &&
                        p.N >= 16 * 4 * kBtRB && p.N <= 16 * 16 * kBtRB;
    const int KTW = narrow ? kBtKTNarrow : kBtKT;
    const int64_t k_tiles = (p.K + KTW - 1) / KTW;
    const int64_t m_tiles = (p.M + MT - 1) / MT;
    const int64_t tiles = k_tiles * m_tiles;
    const bool one_group = p.group_size >= p.K;
    const int64_t G = one_group ? 1 : (p.K + p.group_size - 1) / p.group_size;
    const int gt = one_group || p.group_size >= KTW ? 1 : (int)(KTW / p.group_size);
    const uint32_t esz = p.scale_f16 ? 2 : 4;

    BtArgs a;
    a.d_x = p.d_x;
    a.ws = c.ws;
    a.tickets = c.tickets;
    a.status = c.status_word;
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    // Group row of k tile kt: kt * 256 / gs when a tile holds whole groups (gs in {32, 64,
    // 128, 256}: a shift by log2(256 / gs)), kt / (gs / 256) when a group spans tiles, 0
    // when one group covers K.
    a.gs_in_tile = 0;
    a.gs_shift256 = 0;
    a.tiles_per_group = 1;
    if (one_group) {
        a.tiles_per_group = (int)k_tiles;
    } else if (p.group_size <= KTW) {
        a.gs_in_tile = (int)p.group_size;
        while ((KTW >> a.gs_shift256) > p.group_size) ++a.gs_shift256;
    } else {
        a.tiles_per_group = (int)(p.group_size / KTW);
    }
    a.scale_f16 = p.scale_f16;
    a.even_high = p.even_high;
    a.wait_ns = c.wait_limit_ns;
    // Rows split so that one wave keeps about two CTAs on every SM, in multiples of 64 rows,
    // within the workspace and ticket capacity.
    int64_t splits = std::max<int64_t>(1, 2LL * c.sm_count / tiles);
    if (!c.ws || !c.tickets || tiles > c.ticket_count) splits = 1;
    while (splits > 1 && tiles * splits * MT * KTW > c.ws_floats) --splits;
    int64_t rows = (p.N + splits - 1) / splits;
    rows = (rows + kBtRB - 1) / kBtRB * kBtRB;
    splits = (p.N + rows - 1) / rows;
    if (splits > 65535 || m_tiles > 65535 || k_tiles > 0x7fffffff) return cudaErrorInvalidValue;
    a.stage_bytes = (uint32_t)((bt_do_off(KTW) + MT * kBtRB * 4 + 1023) / 1024 * 1024);
    // When the split above leaves each CTA at most 4 stages of rows, the hand-off through
    // the workspace (partials to L2, two device-scope fences and the ticket atomic, then
    // the last CTA's reads: ~3 us) dominates the launch; then one cluster of up to 16 CTAs
    // (one per row split) covers a k tile and the splits add their partials through
    // distributed shared memory.  Measured: 2048 x 2048 6.2 -> 3.6 us, 8192 x 2048
    // 10.8 -> 9.3 us at M = 1; with longer row ranges (14336 x 4096: 14.2 -> 20.9 us), or
    // 8 rows of d_out over 8 stages, the cluster's fewer CTAs lose more than the hand-off
    // costs, so those keep the workspace.
    a.cluster = 1;
    if (rows <= 4 * kBtRB || narrow) {
        int cs = 1;
        while (cs * 2 <= 16 && cs * 2 <= std::max<int64_t>(1, 2LL * c.sm_count / tiles)) cs *= 2;
        const int64_t rows_c = ((p.N + cs - 1) / cs + kBtRB - 1) / kBtRB * kBtRB;
        const int st_c = (int)std::min<int64_t>(kBtMaxStages, rows_c / kBtRB);
        const int ring_c = st_c * (int)a.stage_bytes, red_c = CW * MT * KTW * 4;
        const int smem_c = 1024 + (ring_c > red_c ? ring_c : red_c) + 256;
        bool ok = false;
        if (cs >= 2 && (MT <= 2 ? rows_c <= 16 * kBtRB : rows_c <= 4 * kBtRB) &&
            smem_c <= kBtSmemLimit) {
            switch (MT) {
                case 1: ok = wide     ? bt_cluster_ok<1, 16, kBtKT>(cs, smem_c)
                             : narrow ? bt_cluster_ok<1, 8, kBtKTNarrow>(cs, smem_c)
                                      : bt_cluster_ok<1, 8, kBtKT>(cs, smem_c);
                        break;
                case 2: ok = wide     ? bt_cluster_ok<2, 16, kBtKT>(cs, smem_c)
                             : narrow ? bt_cluster_ok<2, 8, kBtKTNarrow>(cs, smem_c)
                                      : bt_cluster_ok<2, 8, kBtKT>(cs, smem_c);
                        break;
                case 4: ok = bt_cluster_ok<4, 8, kBtKT>(cs, smem_c); break;
                default: ok = bt_cluster_ok<kMT, 8, kBtKT>(cs, smem_c); break;
            }
        }
        if (ok) {
            a.cluster = cs;
            splits = cs;
            rows = rows_c;
        }
    }
    a.splits = (int)splits;
    a.rows_per_split = rows;
    a.stages = (int)std::min<int64_t>(kBtMaxStages, rows / kBtRB);
    a.sc_rows = p.scale_f16 ? kBtScRows16 : kBtScRows32;
    a.tx = (uint32_t)(kBtRB * KTW / 2) + (uint32_t)gt * a.sc_rows * esz + (uint32_t)MT * kBtRB * 4;
    const int red = CW * MT * KTW * 4;
    const int ring = a.stages * (int)a.stage_bytes;
    const int smem = 1024 + (ring > red ? ring : red) + 256;
    if (smem > kBtSmemLimit) return cudaErrorInvalidValue;

    BtMaps maps;
    const cuuint32_t estr[2] = {1, 1};
    {
        const int64_t Kp = p.K / 2;
        const cuuint64_t dims[2] = {(cuuint64_t)Kp, (cuuint64_t)p.N};
        const cuuint64_t strides[1] = {(cuuint64_t)Kp};
        const cuuint32_t box[2] = {(cuuint32_t)(KTW / 2), (cuuint32_t)kBtRB};
        if (enc(&maps.w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(p.qweight), dims,
                strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)p.N, (cuuint64_t)G};
        const cuuint64_t strides[1] = {(cuuint64_t)p.N * esz};
        const cuuint32_t box[2] = {(cuuint32_t)a.sc_rows, (cuuint32_t)gt};
        if (enc(&maps.s, p.scale_f16 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT32, 2,
                const_cast<void*>(p.scales), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)p.N, (cuuint64_t)p.M};
        const cuuint64_t strides[1] = {(cuuint64_t)p.N * 4};
        const cuuint32_t box[2] = {(cuuint32_t)kBtRB, (cuuint32_t)MT};
        if (enc(&maps.d, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(p.d_out), dims,
                strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const dim3 grid((unsigned)k_tiles, (unsigned)splits, (unsigned)m_tiles);
    switch (MT) {
        case 1: return wide     ? launch_bt<1, 16, kBtKT>(maps, a, grid, smem, c)
                       : narrow ? launch_bt<1, 8, kBtKTNarrow>(maps, a, grid, smem, c)
                                : launch_bt<1, 8, kBtKT>(maps, a, grid, smem, c);
        case 2: return wide     ? launch_bt<2, 16, kBtKT>(maps, a, grid, smem, c)
                       : narrow ? launch_bt<2, 8, kBtKTNarrow>(maps, a, grid, smem, c)
                                : launch_bt<2, 8, kBtKT>(maps, a, grid, smem, c);
        case 4: return launch_bt<4, 8, kBtKT>(maps, a, grid, smem, c);
        default: return launch_bt<kMT, 8, kBtKT>(maps, a, grid, smem, c);
    }
}

}  // namespace

cudaError_t backward_dx_launch(const TrainProblem& p, const LaunchCtx& c) {
    BwArgs a;
    a.d_out = p.d_out;
    a.w = p.qweight;
    a.scales = p.scales;
    a.d_x = p.d_x;
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.Kp = (p.K + 1) / 2;
    a.gs = p.group_size;
    a.scale_f16 = p.scale_f16;
    a.even_high = p.even_high;
    a.ws = c.ws;
    a.tickets = c.tickets;
    if (bt_eligible(p)) return backward_tma_launch(p, c);
    const bool fast = p.K % 8 == 0 && p.group_size % 8 == 0 &&
                      reinterpret_cast<uintptr_t>(p.qweight) % 4 == 0;
    if (!fast) {
        a.k_tiles = 0;
        a.splits = 1;
        a.rows_per_split = p.N;
        const int64_t blocks = std::min<int64_t>((p.M * p.K + 255) / 256, 16LL * c.sm_count);
        return launch(backward_dx_generic_kernel, a, dim3((unsigned)blocks), 256, c);
    }
    a.k_tiles = (int)((p.K + kBwK - 1) / kBwK);
    const int MT = p.M <= 1 ? 1 : p.M <= 2 ? 2 : p.M <= 4 ? 4 : kMT;
    const int64_t m_tiles = (p.M + MT - 1) / MT;
    // Split the rows over CTAs so that one wave keeps ~2 CTAs on every SM, keeping >= 64
    // rows per split,
    // within the workspace ([splits][M][K] floats) and ticket capacity.
    const int64_t tiles = a.k_tiles * m_tiles;
    int64_t splits = std::max<int64_t>(1, 2LL * c.sm_count / tiles);  // one wave
    splits = std::min<int64_t>(splits, std::max<int64_t>(1, p.N / 64));
    if (!c.ws || !c.tickets || tiles > c.ticket_count) splits = 1;
    while (splits > 1 && splits * p.M * p.K > c.ws_floats) --splits;
    a.rows_per_split = (p.N + splits - 1) / splits;
    a.splits = (int)((p.N + a.rows_per_split - 1) / a.rows_per_split);
    if (a.splits < 1) a.splits = 1;
    if (m_tiles > 65535 || a.splits > 65535) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)a.k_tiles, (unsigned)a.splits, (unsigned)m_tiles);
    switch (MT) {
        case 1: return launch(backward_dx_kernel<1>, a, grid, kBwThreads, c);
        case 2: return launch(backward_dx_kernel<2>, a, grid, kBwThreads, c);
        case 4: return launch(backward_dx_kernel<4>, a, grid, kBwThreads, c);
        default: return launch(backward_dx_kernel<kMT>, a, grid, kBwThreads, c);
    }
}

cudaError_t requant_launch(const RequantProblem& p, const LaunchCtx& c) {
    RqArgs a;
    a.latent = p.latent;
    a.scales = p.scales;
    a.w = p.qweight;
    a.N = p.N;
    a.K = p.K;
    a.Kp = (p.K + 1) / 2;
    a.gs = p.group_size;
    a.scale_f16 = p.scale_f16;
    a.even_high = p.even_high;
    const uintptr_t wq = reinterpret_cast<uintptr_t>(p.qweight);
    const bool lat16 = reinterpret_cast<uintptr_t>(p.latent) % 16 == 0 && p.K < (1LL << 31);
    // (Eight float4 loads a thread, 32 k, measured slower than four on 8192 x 2048.)
    const bool w16 = lat16 && p.K % 16 == 0 && wq % 8 == 0;
    const bool fast = lat16 && p.K % 4 == 0 && wq % 2 == 0;
    const int64_t units = w16 ? p.N * (p.K / 16) : fast ? p.N * (p.K / 4) : p.N * a.Kp;
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((units + 255) / 256, 32LL * c.sm_count));
    const dim3 grid((unsigned)blocks);
    if (w16)
        return p.even_high ? launch(requant_wide_kernel<4, true>, a, grid, 256, c)
                           : launch(requant_wide_kernel<4, false>, a, grid, 256, c);
    return fast ? launch(requant_kernel, a, dim3((unsigned)blocks), 256, c)
                : launch(requant_generic_kernel, a, dim3((unsigned)blocks), 256, c);
}

}  // namespace q4lin
