// rowstream.cu -- CUDA-core kernels of the 4-bit weight-quantized linear (sm_103a).
//
//   out[m,n] = bias[n] + sum_g s[g,n] * sum_{k in g} x[m,k] * (code[n,k] - 8)
//
// The formula, the +8 offset, the [N, K/2] low-nibble-even packing and the grouped
// [ceil(K/gs), N] scales follow "[ExecuTorch][WebGPU] Add linear_qcs4w op", Solution and
// Constraints (2)-(3); the bias epilogue follows "Add optimized linear_fp32 op".
//
// rowstream_kernel (M = 1 decode GEMV, and M <= 4 per activation tile):
//   The decode GEMV is bound by HBM: every packed byte is read once.  Each thread owns
//   R consecutive weight rows and a strided set of 16-byte chunks (32 k-values, one
//   LDG.128 per row per chunk, coalesced along K).  The x chunk sits in registers and is
//   reused across the R rows; codes are widened in registers; lanes split K and reduce
//   with warp shuffles (then shared memory across warps that split K further).
//   Lane layout in a warp: lane = rg + 2 * cl, rg in {0,1} picks one of two row groups,
//   cl in [0,16) the chunk lane.  Two row groups per warp make one scale load
//   instruction read whole 32-byte sectors (R consecutive scales of one group per
//   thread, the neighbouring R in the other row group).
//   Prior art on the pages: the TVM decode-GEMV schedule "(TS, TR) = (8, 16)" (several
//   rows per workgroup, few reduction threads per row) -- kept as an idea (rows per
//   thread, a short lane reduction); the WGSL tiling itself is not used.  The ragged
//   tail (the page records a store 7 rows past the end at vocab 128257) is predicated:
//   rows >= N are never loaded or stored.
//
// generic_kernel: one warp per output element, lanes along K with byte loads; any K
//   (odd K: the padding nibble is never read), any group size, any alignment.
#include <cuda_fp16.h>

#include <algorithm>

#include "q4lin_internal.h"

namespace q4lin {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

struct RowArgs {
    const float* x;
    const uint8_t* w;
    const void* scales;
    const float* bias;
    float* out;
    int64_t M, N, K, Kp, gs;
    int chunks;        // K / 32 sixteen-byte chunks per weight row
    int wc;            // warps along K in a CTA (1, 2, 4, 8)
    int rows_per_cta;  // 2 * (kWarps / wc) * R
    int scale_f16;
    int svec;          // R consecutive scales of one group can be loaded as vectors
    int per_channel;   // one scale per row (group_size >= K)
};

// ------------------------------------------------------------------ small device helpers
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ld_stream_u2(const void* p) {
    uint2 v;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

// Programmatic dependent launch: wait until the preceding grid on the stream has
// completed (no-op when the kernel was not launched with the PDL attribute).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(d)
        : "l"(*reinterpret_cast<unsigned long long*>(&a)),
          "l"(*reinterpret_cast<unsigned long long*>(&b)),
          "l"(*reinterpret_cast<unsigned long long*>(&c)));
    return *reinterpret_cast<float2*>(&d);
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;"
        : "=l"(d)
        : "l"(*reinterpret_cast<unsigned long long*>(&a)),
          "l"(*reinterpret_cast<unsigned long long*>(&b)));
    return *reinterpret_cast<float2*>(&d);
}

// Widen the two binary16 halves of h and subtract 1032 in one mixed-precision add each.
__device__ __forceinline__ void halves_minus_1032(uint32_t h, float& lo, float& hi) {
    asm("{\n\t.reg .b16 l, u;\n\tmov.b32 {l, u}, %2;\n\t"
        "add.rn.f32.f16 %0, l, %3;\n\tadd.rn.f32.f16 %1, u, %3;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(h), "f"(-1032.0f));
}

// The eight signed codes (c - 8) of one packed 32-bit word, as exact floats in k order.
// Nibble i (bits 4i..4i+3) holds k = i by default, k = i ^ 1 with even k high.
// 0x6400 is binary16 1024.0; OR-ing a 4-bit code into its low mantissa bits gives
// 1024 + c exactly, and (1024 + c) - 1032 = c - 8 exactly in fp32.
template <bool EH>
__device__ __forceinline__ void codes8(uint32_t w, float (&v)[8]) {
    const uint32_t h0 = (w & 0x000F000Fu) | 0x64006400u;          // nibbles 0 | 4
    const uint32_t h1 = ((w >> 4) & 0x000F000Fu) | 0x64006400u;   // nibbles 1 | 5
    const uint32_t h2 = ((w >> 8) & 0x000F000Fu) | 0x64006400u;   // nibbles 2 | 6
    const uint32_t h3 = ((w >> 12) & 0x000F000Fu) | 0x64006400u;  // nibbles 3 | 7
    float n[8];
    halves_minus_1032(h0, n[0], n[4]);
    halves_minus_1032(h1, n[1], n[5]);
    halves_minus_1032(h2, n[2], n[6]);
    halves_minus_1032(h3, n[3], n[7]);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = n[EH ? (i ^ 1) : i];
}

__device__ __forceinline__ uint32_t word_of(const uint4& u, int j) {
    return j == 0 ? u.x : j == 1 ? u.y : j == 2 ? u.z : u.w;
}

// sum_{t<32} x[t] * (code_t - 8) for one 16-byte chunk; two fp32x2 chains.
template <bool EH>
__device__ __forceinline__ float chunk_dot(const uint4& wv, const float4 (&xv)[8]) {
    float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float v[8];
        codes8<EH>(word_of(wv, j), v);
        const float4 p = xv[2 * j], q = xv[2 * j + 1];
        float2& acc = (j & 1) ? a1 : a0;
        acc = ffma2(make_float2(v[0], v[1]), make_float2(p.x, p.y), acc);
        acc = ffma2(make_float2(v[2], v[3]), make_float2(p.z, p.w), acc);
        acc = ffma2(make_float2(v[4], v[5]), make_float2(q.x, q.y), acc);
        acc = ffma2(make_float2(v[6], v[7]), make_float2(q.z, q.w), acc);
    }
    return (a0.x + a0.y) + (a1.x + a1.y);
}

__device__ __forceinline__ float load_scale(const void* scales, int f16, int64_t idx) {
    if (f16) return __half2float(reinterpret_cast<const __half*>(scales)[idx]);
    return reinterpret_cast<const float*>(scales)[idx];
}

// Scales s[g, row0 .. row0+R) (zeros past N).
template <int R>
__device__ __forceinline__ void load_scales(const RowArgs& a, int64_t g, int64_t row0,
                                            float (&s)[R]) {
    const int64_t base = g * a.N + row0;
    if (a.svec && row0 + R <= a.N) {
        if (a.scale_f16) {
            const __half* p = reinterpret_cast<const __half*>(a.scales) + base;
            uint32_t u[R / 2];
            if constexpr (R == 8) {
                const uint4 t = ld_stream_u4(p);
                u[0] = t.x; u[1] = t.y; u[2] = t.z; u[3] = t.w;
            } else {
                const uint2 t = ld_stream_u2(p);
                u[0] = t.x; u[1] = t.y;
            }
#pragma unroll
            for (int i = 0; i < R / 2; ++i) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u[i]));
                s[2 * i] = f.x;
                s[2 * i + 1] = f.y;
            }
        } else {
            const float* p = reinterpret_cast<const float*>(a.scales) + base;
#pragma unroll
            for (int i = 0; i < R / 4; ++i) {
                const uint4 t = ld_stream_u4(p + 4 * i);
                s[4 * i] = __uint_as_float(t.x);
                s[4 * i + 1] = __uint_as_float(t.y);
                s[4 * i + 2] = __uint_as_float(t.z);
                s[4 * i + 3] = __uint_as_float(t.w);
            }
        }
    } else {
#pragma unroll
        for (int r = 0; r < R; ++r)
            s[r] = (row0 + r < a.N) ? load_scale(a.scales, a.scale_f16, base + r) : 0.f;
    }
}

// Sum V values per thread over the 16 chunk lanes of its row group (xor 2..16), then
// over the warps that split K (shared memory), and let lane cl of the row group finish
// value cl: returns true and sets `total` on the threads that own a value.
template <int V>
__device__ __forceinline__ bool reduce_rowgroup(const RowArgs& a, float (&val)[V],
                                                float* red, int warp, int rg, int cl,
                                                float& total) {
#pragma unroll
    for (int i = 0; i < V; ++i) {
#pragma unroll
        for (int o = 2; o < 32; o <<= 1) val[i] += __shfl_xor_sync(0xffffffffu, val[i], o);
    }
    float mine = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i)
        if (cl == i) mine = val[i];
    if (a.wc == 1) {
        total = mine;
        return cl < V;
    }
    // red layout: [warp][rg][V]
    if (cl < V) red[(warp * 2 + rg) * V + cl] = mine;
    __syncthreads();
    const int wc = warp % a.wc;
    bool owner = false;
    if (wc == 0 && cl < V) {
        float t = 0.f;
        for (int j = 0; j < a.wc; ++j) t += red[((warp + j) * 2 + rg) * V + cl];
        total = t;
        owner = true;
    }
    __syncthreads();  // red is reused by the next activation tile
    return owner;
}

__device__ __forceinline__ void store_out(const RowArgs& a, int64_t m, int64_t n, float v) {
    if (a.per_channel) v *= load_scale(a.scales, a.scale_f16, n);
    if (a.bias) v += a.bias[n];
    a.out[m * a.N + n] = v;
}

// ------------------------------------------------------------------------ M = 1 GEMV
template <int R, bool EH>
__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(const RowArgs a) {
    __shared__ float red[kWarps * 2 * R];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int wc = warp % a.wc, wr = warp / a.wc;
    const int rg = lane & 1, cl = lane >> 1;
    const int tc = wc * 16 + cl, TC = a.wc * 16;
    const int64_t row0 = (int64_t)blockIdx.x * a.rows_per_cta + (wr * 2 + rg) * R;

    griddep_wait();
    griddep_launch();
    for (int64_t m = blockIdx.y; m < a.M; m += gridDim.y) {
        float acc[R];
#pragma unroll
        for (int r = 0; r < R; ++r) acc[r] = 0.f;
        const float* xm = a.x + m * a.K;
        for (int c = tc; c < a.chunks; c += TC) {
            uint4 wv[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int64_t n = row0 + r;
                wv[r] = (n < a.N) ? ld_stream_u4(a.w + n * a.Kp + (int64_t)c * 16)
                                  : make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
            }
            float s[R] = {};
            if (!a.per_channel) load_scales<R>(a, ((int64_t)c * 32) / a.gs, row0, s);
            float4 xv[8];
            const float4* xp = reinterpret_cast<const float4*>(xm + (int64_t)c * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i) xv[i] = __ldg(xp + i);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float d = chunk_dot<EH>(wv[r], xv);
                acc[r] = a.per_channel ? acc[r] + d : fmaf(d, s[r], acc[r]);
            }
        }
        float total;
        if (reduce_rowgroup<R>(a, acc, red, warp, rg, cl, total)) {
            const int64_t n = row0 + cl;
            if (n < a.N) store_out(a, m, n, total);
        }
    }
}

// --------------------------------------------------------- small M (MR activation rows)
// Each dequantized weight is reused across MR rows of x; weights are pre-scaled
// w = (c - 8) * s in fp32 (per-channel: unscaled, the scale is applied at the end).
template <int MR, int R, bool EH>
__global__ void __launch_bounds__(kThreads, 2) smallm_kernel(const RowArgs a) {
    constexpr int V = R * MR;
    __shared__ float red[kWarps * 2 * V];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int wc = warp % a.wc, wr = warp / a.wc;
    const int rg = lane & 1, cl = lane >> 1;
    const int tc = wc * 16 + cl, TC = a.wc * 16;
    const int64_t row0 = (int64_t)blockIdx.x * a.rows_per_cta + (wr * 2 + rg) * R;

    griddep_wait();
    griddep_launch();
    for (int64_t mb = blockIdx.y; mb * MR < a.M; mb += gridDim.y) {
        const int64_t m0 = mb * MR;
        float2 acc[R][MR];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MR; ++m) acc[r][m] = make_float2(0.f, 0.f);
        for (int c = tc; c < a.chunks; c += TC) {
            uint4 wv[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int64_t n = row0 + r;
                wv[r] = (n < a.N) ? ld_stream_u4(a.w + n * a.Kp + (int64_t)c * 16)
                                  : make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
            }
            float s[R] = {};
            if (!a.per_channel) load_scales<R>(a, ((int64_t)c * 32) / a.gs, row0, s);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float4 xa[MR], xb[MR];
#pragma unroll
                for (int m = 0; m < MR; ++m) {
                    if (m0 + m < a.M) {
                        const float4* xp = reinterpret_cast<const float4*>(
                            a.x + (m0 + m) * a.K + (int64_t)c * 32 + 8 * j);
                        xa[m] = __ldg(xp);
                        xb[m] = __ldg(xp + 1);
                    } else {
                        xa[m] = make_float4(0.f, 0.f, 0.f, 0.f);
                        xb[m] = xa[m];
                    }
                }
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    float v[8];
                    codes8<EH>(word_of(wv[r], j), v);
                    float2 w0 = make_float2(v[0], v[1]), w1 = make_float2(v[2], v[3]);
                    float2 w2 = make_float2(v[4], v[5]), w3 = make_float2(v[6], v[7]);
                    if (!a.per_channel) {
                        const float2 ss = make_float2(s[r], s[r]);
                        w0 = fmul2(w0, ss); w1 = fmul2(w1, ss);
                        w2 = fmul2(w2, ss); w3 = fmul2(w3, ss);
                    }
#pragma unroll
                    for (int m = 0; m < MR; ++m) {
                        acc[r][m] = ffma2(w0, make_float2(xa[m].x, xa[m].y), acc[r][m]);
                        acc[r][m] = ffma2(w1, make_float2(xa[m].z, xa[m].w), acc[r][m]);
                        acc[r][m] = ffma2(w2, make_float2(xb[m].x, xb[m].y), acc[r][m]);
                        acc[r][m] = ffma2(w3, make_float2(xb[m].z, xb[m].w), acc[r][m]);
                    }
                }
            }
        }
        float val[V];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MR; ++m) val[m * R + r] = acc[r][m].x + acc[r][m].y;
        float total;
        // V may exceed the 16 chunk lanes: finish values cl and cl + 16 in two passes.
        if constexpr (V <= 16) {
            if (reduce_rowgroup<V>(a, val, red, warp, rg, cl, total)) {
                const int64_t n = row0 + cl % R, m = m0 + cl / R;
                if (n < a.N && m < a.M) store_out(a, m, n, total);
            }
        } else {
            float lo[16], hi[V - 16];
#pragma unroll
            for (int i = 0; i < 16; ++i) lo[i] = val[i];
#pragma unroll
            for (int i = 16; i < V; ++i) hi[i - 16] = val[i];
            if (reduce_rowgroup<16>(a, lo, red, warp, rg, cl, total)) {
                const int64_t n = row0 + cl % R, m = m0 + cl / R;
                if (n < a.N && m < a.M) store_out(a, m, n, total);
            }
            if (reduce_rowgroup<V - 16>(a, hi, red, warp, rg, cl, total)) {
                const int64_t n = row0 + (cl + 16) % R, m = m0 + (cl + 16) / R;
                if (n < a.N && m < a.M) store_out(a, m, n, total);
            }
        }
    }
}

// ------------------------------------------------------------------------ generic path
struct GenArgs {
    const float* x;
    const uint8_t* w;
    const void* scales;
    const float* bias;
    float* out;
    int64_t M, N, K, Kp, gs;
    int scale_f16;
};

template <bool EH>
__global__ void __launch_bounds__(kThreads) generic_kernel(const GenArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t warp_global = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int64_t warps_total = (int64_t)gridDim.x * kWarps;
    griddep_wait();
    griddep_launch();
    for (int64_t item = warp_global; item < a.M * a.N; item += warps_total) {
        const int64_t m = item / a.N, n = item % a.N;
        const float* xm = a.x + m * a.K;
        const uint8_t* wn = a.w + n * a.Kp;
        float acc = 0.f;
        for (int64_t k = lane; k < a.K; k += 32) {
            const uint8_t b = __ldg(wn + (k >> 1));
            const bool low = EH ? (k & 1) : !(k & 1);
            const int code = low ? (b & 0xF) : (b >> 4);
            const float s = load_scale(a.scales, a.scale_f16, (k / a.gs) * a.N + n);
            acc = fmaf(__ldg(xm + k), (float)(code - 8) * s, acc);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) a.out[m * a.N + n] = acc + (a.bias ? a.bias[n] : 0.f);
    }
}

template <typename Kern, typename Args>
cudaError_t launch(Kern kern, dim3 grid, const Args& args, const LaunchCtx& c) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[1];
    if (c.pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, args);
}

}  // namespace

bool rowstream_eligible(const Problem& p) {
    if (p.K % 32 != 0) return false;
    if (reinterpret_cast<uintptr_t>(p.x) % 16 || reinterpret_cast<uintptr_t>(p.qweight) % 16)
        return false;
    const bool per_channel = p.group_size >= p.K;
    return per_channel || p.group_size % 32 == 0;
}

cudaError_t rowstream_launch(const Problem& p, const LaunchCtx& c) {
    RowArgs a;
    a.x = p.x;
    a.w = p.qweight;
    a.scales = p.scales;
    a.bias = p.bias;
    a.out = p.out;
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.Kp = p.K / 2;
    a.gs = p.group_size;
    a.chunks = (int)(p.K / 32);
    a.scale_f16 = p.scale_f16;
    a.per_channel = p.group_size >= p.K;
    const int esize = p.scale_f16 ? 2 : 4;
    a.svec = (reinterpret_cast<uintptr_t>(p.scales) % 16 == 0) && ((p.N * esize) % 16 == 0);

    const int MR = p.M == 1 ? 1 : (p.M == 2 ? 2 : 4);
    const int64_t mblocks = (p.M + MR - 1) / MR;
    // Pick rows per thread R and warps along K so that the grid fills the GPU
    // (two resident CTAs per SM) while every thread keeps at least one chunk per row.
    const int64_t target = 2LL * c.sm_count;
    int best_R = MR == 4 ? 4 : 8, best_wc = 1;
    int64_t best_ctas = -1;
    const int r_options[2] = {8, 4};
    bool done = false;
    for (int ri = 0; ri < 2 && !done; ++ri) {
        const int R = r_options[ri];
        if (MR == 4 && R == 8) continue;
        for (int wc = 1; wc <= kWarps; wc *= 2) {
            if (wc > 1 && 16 * wc > a.chunks) break;
            const int rows = 2 * (kWarps / wc) * R;
            const int64_t ctas = ((p.N + rows - 1) / rows) * std::min<int64_t>(mblocks, 65535);
            if (ctas > best_ctas) {
                best_ctas = ctas;
                best_R = R;
                best_wc = wc;
            }
            if (ctas >= target) {
                done = true;
                break;
            }
        }
    }
    a.wc = best_wc;
    a.rows_per_cta = 2 * (kWarps / best_wc) * best_R;
    const dim3 grid((unsigned)((p.N + a.rows_per_cta - 1) / a.rows_per_cta),
                    (unsigned)std::min<int64_t>(mblocks, 65535));
    const bool eh = p.even_high != 0;
    if (MR == 1) {
        if (best_R == 8)
            return eh ? launch(gemv_kernel<8, true>, grid, a, c) : launch(gemv_kernel<8, false>, grid, a, c);
        return eh ? launch(gemv_kernel<4, true>, grid, a, c) : launch(gemv_kernel<4, false>, grid, a, c);
    }
    if (MR == 2) {
        if (best_R == 8)
            return eh ? launch(smallm_kernel<2, 8, true>, grid, a, c)
                      : launch(smallm_kernel<2, 8, false>, grid, a, c);
        return eh ? launch(smallm_kernel<2, 4, true>, grid, a, c)
                  : launch(smallm_kernel<2, 4, false>, grid, a, c);
    }
    return eh ? launch(smallm_kernel<4, 4, true>, grid, a, c) : launch(smallm_kernel<4, 4, false>, grid, a, c);
}

cudaError_t generic_launch(const Problem& p, const LaunchCtx& c) {
    GenArgs a;
    a.x = p.x;
    a.w = p.qweight;
    a.scales = p.scales;
    a.bias = p.bias;
    a.out = p.out;
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.Kp = (p.K + 1) / 2;
    a.gs = p.group_size;
    a.scale_f16 = p.scale_f16;
    const int64_t items = p.M * p.N;
    const int64_t want = (items + kWarps - 1) / kWarps;
    const unsigned blocks = (unsigned)std::min<int64_t>(want, 16LL * c.sm_count);
    return p.even_high ? launch(generic_kernel<true>, dim3(blocks), a, c)
                       : launch(generic_kernel<false>, dim3(blocks), a, c);
}

}  // namespace q4lin
