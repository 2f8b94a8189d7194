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
//   requant_kernel: one thread per 4 k of a row (one float4 of latents, two output bytes);
//     consecutive threads walk a row (coalesced loads and stores).
//   requant_generic_kernel: one thread per output byte (any K, any alignment).
#include <cuda_fp16.h>

#include <algorithm>

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
    __threadfence();
    __syncthreads();
    const int item = (int)(blockIdx.z * gridDim.x + blockIdx.x);
    if (threadIdx.x == 0) s_last = atomicAdd(a.tickets + item, 1) == a.splits - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
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

struct RqArgs {
    const float* latent;
    const void* scales;
    uint8_t* w;
    int64_t N, K, Kp, gs;
    int scale_f16, even_high;
};

__device__ __forceinline__ int requant_code(float l, float s) {
    if (s == 0.f) return 8;
    const float q = __fdiv_rn(l, s);
    if (isnan(q)) return 8;
    const float r = fminf(fmaxf(rintf(q), -8.f), 7.f);
    return (int)r + 8;
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
    const bool fast = p.K % 4 == 0 && p.K < (1LL << 31) &&
                      reinterpret_cast<uintptr_t>(p.latent) % 16 == 0 &&
                      reinterpret_cast<uintptr_t>(p.qweight) % 2 == 0;
    const int64_t units = fast ? p.N * (p.K / 4) : p.N * a.Kp;
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((units + 255) / 256, 32LL * c.sm_count));
    return fast ? launch(requant_kernel, a, dim3((unsigned)blocks), 256, c)
                : launch(requant_generic_kernel, a, dim3((unsigned)blocks), 256, c);
}

}  // namespace q4lin
