// gemv_tma.cu -- TMA-fed decode GEMV (M = 1) of the 4-bit weight-quantized linear.
//
//   out[n] = bias[n] + sum_g s[g,n] * sum_{k in g} x[k] * (code[n,k] - 8)
//
// (formula: "[ExecuTorch][WebGPU] Add linear_qcs4w op", Solution; the decode GEMV is the
// regime of the TVM "dlight.gpu.GEMV" WebGPU notice, whose lesson -- several rows per
// workgroup, a short reduction per row, and a predicated final store for a ragged vocab
// such as 128257 -- is kept here.)
//
// HBM-bound: every packed byte and every scale is read exactly once.  The memory stream
// is decoupled from the arithmetic:
//   producer warp (one lane): per stage, 2D TMA copies of the weight tile [rb rows x 512
//     bytes] (= 1024 k per row; the packed matrix viewed as 16-bit elements, so one box
//     spans the 512 bytes) and of the matching block of group
//     scales [1024 / group size groups x rb rows], all on one mbarrier, into a ring of
//     2..8 stages.  Weight rows are long contiguous segments, so DRAM sees streaming reads.
//   8 consumer warps (256 threads): thread = (chunk lane j in 0..15, row group of V rows);
//     per stage it widens chunks j and j + 16 (32 codes each) of each of its V rows and
//     dots them with the x chunks (read from shared memory, where x is staged in padded
//     32-float chunks, and reused across the V rows), scaling each chunk by its group
//     scale.  A quarter-warp reads 128 contiguous bytes of a weight row (conflict-free).
//     Partial sums stay in registers across the whole row; the 16 chunk lanes of a row
//     group are reduced with shuffles once per row block.
// A CTA is small enough (288 threads, at most 113 KiB of shared memory) that two fit on
// one SM: the CTAs of the next kernel on the stream can become resident while this one
// runs.  With programmatic dependent launch their producers then stream weights and
// scales (which do not depend on the preceding kernel) before griddepcontrol.wait; x,
// bias, out and the split-K workspace are touched only after it.
// Row blocks of long-K, short-N matrices are split along K across CTAs; the partial row
// sums go to a workspace and the last CTA of a row block adds them in part order (the
// result does not depend on which CTA finishes last).
// Waits are bounded in time; a timeout records code 1 in the status word and the CTA
// drains its copies and returns.
#include <algorithm>
#include <mutex>

#include "ptx.cuh"
#include "q4lin_internal.h"

namespace q4lin {
namespace {
using namespace ptx;

constexpr int kCWarps = 8;                 // consumer warps: 2 per SM sub-partition
constexpr int kCThreads = 32 * kCWarps;
constexpr int kThreadsG = kCThreads + 32;  // + the producer warp
constexpr int kRowGroups = kCThreads / 16; // 16 chunk lanes per row group
static_assert(kRowGroups == kGemvMinRowBlock && 4 * kRowGroups == kGemvMaxRowBlock,
              "row blocks of 16 row groups x V rows, V in {1, 2, 4}");
// Stage width: H chunk columns of 16 bytes per thread, i.e. 256 * H packed bytes (512 * H
// k) per row per stage.  H = 2 for every tile height (measured: halving the stage of the
// V = 4 tiles to fit a deeper ring made them slower, the per-stage overhead outweighs the
// extra depth).
__host__ __device__ constexpr int chunk_cols(int) { return 2; }
__host__ __device__ constexpr int stage_row_bytes(int V) { return 256 * chunk_cols(V); }
__host__ __device__ constexpr int stage_chunks(int V) { return 16 * chunk_cols(V); }
constexpr int kXPad = 36;                  // floats per 32-float x chunk in shared memory
constexpr int kMaxStages = 8;
constexpr int kCtaSmem = 113 * 1024;       // two CTAs per SM
constexpr int64_t kDrainNs = 4000000000LL;
constexpr int kMaxMats = 4;

// One weight matrix of a launch.  Several matrices that share x (the q/k/v projections
// of a layer, or gate/up) run in one launch over a virtual row space: matrix i owns the
// row blocks [blk_begin, blk_begin + ceil(N / rb)).
struct MatArgs {
    const void* scales;
    const float* bias;
    float* out;
    int64_t N;
    int64_t blk_begin;
};
struct TensorMaps {
    CUtensorMap w[kMaxMats];  // packed weights [N, K/4] 16-bit, box [rb rows x 512 bytes]
    CUtensorMap s[kMaxMats];  // group scales [G, N], box [groups per stage x rb rows]
};

struct GArgs {
    const float* x;
    MatArgs mat[kMaxMats];
    int nmat;
    int64_t K;
    int kstages;     // ceil(K / stage k)
    int x_chunks;    // kstages * chunks per stage
    int gs_shift;    // log2(group size / 32) (grouped scales)
    int stages;      // ring depth
    uint32_t stage_bytes, scale_off, stage_tx;
    int64_t row_blocks;
    // Split K: each row block's stages are cut into `parts` runs of `tpp` stages; a work
    // item is (row block, part).  With parts > 1 the items write partial row sums to
    // ws[part * ws_rows + row] and the last item of a row block (ticket count) adds them
    // in part order.
    int parts, tpp;
    int items;
    float* ws;       // [parts, ws_rows] partial sums (parts > 1)
    int* tickets;    // [row_blocks], zero between launches (the last item resets its own)
    int64_t ws_rows; // row_blocks * rows per block
    int* status;
    int64_t wait_ns;
};

// A CTA's walk over its work items: item = blockIdx.x + i * gridDim.x, item -> (row block
// blk = item / parts, part), covering stages [part * tpp, min((part + 1) * tpp, kstages)).
// One division per item, none per stage.
struct Cursor {
    int item, blk, part, ks, ks_end;
    __device__ __forceinline__ void set(const GArgs& a) {
        blk = item / a.parts;
        part = item - blk * a.parts;
        ks = part * a.tpp;
        ks_end = min(ks + a.tpp, a.kstages);
    }
    __device__ __forceinline__ void start(const GArgs& a) {
        item = (int)blockIdx.x;
        if (item < a.items) set(a);
    }
    __device__ __forceinline__ bool valid(const GArgs& a) const { return item < a.items; }
    // Move to the next stage; true when that finished the current item.
    __device__ __forceinline__ bool advance(const GArgs& a) {
        if (++ks < ks_end) return false;
        item += gridDim.x;
        if (item < a.items) set(a);
        return true;
    }
};

__host__ __device__ constexpr int x_bytes(int x_chunks) { return x_chunks * kXPad * 4; }
// Shared memory: the stage ring, then the barriers and flags (256 bytes), then x.
inline int smem_bytes_g(int stages, uint32_t stage_bytes, int x_chunks) {
    return 1024 + stages * (int)stage_bytes + 256 + x_bytes(x_chunks);
}

__device__ __forceinline__ float load_scale(const void* scales, int f16, int64_t idx) {
    if (f16) return __half2float(__ldg(reinterpret_cast<const __half*>(scales) + idx));
    return __ldg(reinterpret_cast<const float*>(scales) + idx);
}

// V consecutive group scales of one group row, from the staged scale block (shared
// memory; 2V or 4V bytes, aligned to their size).
template <int V, bool F16>
__device__ __forceinline__ void stage_scales(uint32_t addr, float (&s)[V]) {
    if (F16) {
        if (V == 4) {
            uint32_t a, b;
            asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(a), "=r"(b) : "r"(addr));
            const float2 p = __half22float2(*reinterpret_cast<__half2*>(&a));
            const float2 q = __half22float2(*reinterpret_cast<__half2*>(&b));
            s[0] = p.x, s[1 % V] = p.y, s[2 % V] = q.x, s[3 % V] = q.y;
        } else if (V == 2) {
            uint32_t a;
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(a) : "r"(addr));
            const float2 p = __half22float2(*reinterpret_cast<__half2*>(&a));
            s[0] = p.x, s[1 % V] = p.y;
        } else {
            unsigned short h;
            asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(addr));
            s[0] = __half2float(__ushort_as_half(h));
        }
    } else {
        if (V == 4) {
            float a, b, c, d;
            asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                         : "=f"(a), "=f"(b), "=f"(c), "=f"(d)
                         : "r"(addr));
            s[0] = a, s[1 % V] = b, s[2 % V] = c, s[3 % V] = d;
        } else if (V == 2) {
            float a, b;
            asm volatile("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(a), "=f"(b) : "r"(addr));
            s[0] = a, s[1 % V] = b;
        } else {
            float a;
            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(a) : "r"(addr));
            s[0] = a;
        }
    }
}

// Byte offset of `off` within group row g of the staged scale block, whose rows are
// IB = rows-per-block x scale-size bytes.  The block is staged with the TMA swizzle of its
// row width (32, 64 or 128 bytes; none for 256): 16-byte unit u of row g sits at unit
// u ^ f(g), so the 8 lanes of a quarter-warp, which read 8 different group rows at the
// same offset, hit 8 different bank groups.
template <int IB>
__device__ __forceinline__ uint32_t scale_slot(int g, int off) {
    if (IB > 128) return (uint32_t)(g * IB + off);
    const int f = IB == 128 ? (g & 7) : IB == 64 ? ((g >> 1) & 3) : ((g >> 2) & 1);
    return (uint32_t)(g * IB + ((((off >> 4) ^ f) << 4) | (off & 15)));
}

// Matrix that owns global row block blk (blk_begin ascending, matrix 0 begins at 0).
__device__ __forceinline__ int mat_of(const GArgs& a, int64_t blk) {
    int i = 0;
#pragma unroll
    for (int q = 1; q < kMaxMats; ++q)
        if (q < a.nmat && blk >= a.mat[q].blk_begin) i = q;
    return i;
}

// Products x[t] * (code_t - 8) of one 16-byte chunk (32 codes), summed as a float2 of
// (even-k sum, odd-k sum) where the lane fed from the HIGH nibbles carries a factor 16.
// Byte b of a word holds k = 2b in its low nibble and k = 2b + 1 in its high nibble
// (swapped when EH).  The low nibbles are isolated with one mask (w & 0x0F0F0F0F) and the
// high nibbles in place with another (w & 0xF0F0F0F0, i.e. 16 * code): no shift.  A byte
// permute builds the float 2^23 + byte (bit pattern 0x4B0000bb) and one packed add of
// -(2^23 + 8) (low lane) / -(2^23 + 128) (high lane) gives c - 8 and 16 * (c - 8), both
// exact.  The factor 16 is removed once per row (a power of two: exact).
template <bool EH>
__device__ __forceinline__ float2 chunk_dot(const uint4& wv, const float4 (&xv)[8]) {
    constexpr float kLo = -8388616.0f, kHi = -8388736.0f;
    const float2 bias = EH ? make_float2(kHi, kLo) : make_float2(kLo, kHi);
    float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
    const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const uint32_t lo = words[w] & 0x0F0F0F0Fu, hi = words[w] & 0xF0F0F0F0u;
        const uint32_t ev = EH ? hi : lo, od = EH ? lo : hi;
        const float4 p = xv[2 * w], q = xv[2 * w + 1];
        const float2 xs[4] = {make_float2(p.x, p.y), make_float2(p.z, p.w), make_float2(q.x, q.y),
                              make_float2(q.z, q.w)};
        float2& acc = (w & 1) ? a1 : a0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const float2 c = fadd2(make_float2(__uint_as_float(prmt(ev, 0x4B000000u, 0x7440u | b)),
                                               __uint_as_float(prmt(od, 0x4B000000u, 0x7440u | b))),
                                   bias);
            acc = ffma2(c, xs[b], acc);
        }
    }
    return fadd2(a0, a1);
}

template <int V, bool EH, bool PC, bool F16>
__global__ void __launch_bounds__(kThreadsG, 2)
    gemv_tma_kernel(const __grid_constant__ TensorMaps tmaps, const GArgs a) {
    constexpr int rb = kRowGroups * V;  // rows per block: 16 row groups of V rows
    constexpr int H = chunk_cols(V), kSRB = stage_row_bytes(V), kSC = stage_chunks(V);
    constexpr uint32_t esz = F16 ? 2 : 4;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // stages are 1024-byte aligned
    uint8_t* gbase = smem_raw + (base - raw);
    const int S = a.stages;
    const uint32_t bar_base = base + (uint32_t)S * a.stage_bytes;
    volatile int* failed = reinterpret_cast<volatile int*>(gbase + (bar_base + 16 * kMaxStages - base));
    volatile int* s_ticket = failed + 1;  // last-item decision, broadcast to the consumers
    float* xs = reinterpret_cast<float*>(gbase + (bar_base + 256 - base));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto full = [&](int s) { return bar_base + 8u * s; };
    auto empty = [&](int s) { return bar_base + 8u * (kMaxStages + s); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
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
            for (int q = 0; q < a.nmat; ++q) {
                prefetch_tensormap(&tmaps.w[q]);
                if (!PC) prefetch_tensormap(&tmaps.s[q]);
            }
            // Pull x toward L2 now, so that the read after griddepcontrol.wait is short.
            // L2 is where global memory is kept coherent: if the preceding kernel writes x
            // after this prefetch, the L2 line is updated and the later read sees it; no
            // copy of x enters this SM's L1 before the wait.
            const int64_t xb = a.K * 4;
            for (int64_t off = 0; off < xb; off += 32768)
                l2_prefetch_bulk(a.x + off / 4, (uint32_t)(xb - off < 32768 ? xb - off : 32768));
            int t = 0, s = 0;
            uint32_t ph = 0;
            Cursor cur;
            cur.start(a);
            while (cur.valid(a)) {
                if (t >= S && !wait_bounded(empty(s), ph ^ 1u, a.wait_ns, failed)) {
                    record_failure(a.status, failed);
                    break;
                }
                if (*failed) break;
                const int mi = mat_of(a, cur.blk);
                const int row0 = (int)((cur.blk - a.mat[mi].blk_begin) * rb);
                const uint32_t sb = base + (uint32_t)s * a.stage_bytes;
                mbar_arrive_expect_tx(full(s), a.stage_tx);
                tma_load_2d(sb, &tmaps.w[mi], cur.ks * (kSRB / 2), row0, full(s));
                if (!PC)
                    tma_load_2d(sb + a.scale_off, &tmaps.s[mi], row0,
                                (cur.ks * kSC) >> a.gs_shift, full(s));
                ++t;
                if (++s == S) s = 0, ph ^= 1u;
                cur.advance(a);
            }
            // The last armed stages may still be landing; the CTA must not exit first.
            for (int q = t > S ? t - S : 0; q < t; ++q)
                wait_bounded(full(q % S), (uint32_t)(q / S) & 1u, kDrainNs, nullptr);
        }
        return;
    }

    // ------------------------------------------------------------------ consumers
    const int j = threadIdx.x & 15;          // chunk lane within a 256-byte box row
    const int r0 = (threadIdx.x >> 4) * V;   // first of this thread's V rows in a block

    // x into shared memory once: chunk c (32 floats) at xs + c * kXPad; zero past K.
    // (Four loads in flight per thread before the shared-memory stores.)
    griddep_wait();
    for (int i0 = threadIdx.x; i0 < a.x_chunks * 8; i0 += 4 * kCThreads) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * kCThreads;
            const int64_t k = (int64_t)(i >> 3) * 32 + (i & 7) * 4;
            v[u] = (i < a.x_chunks * 8 && k < a.K) ? __ldg(reinterpret_cast<const float4*>(a.x + k))
                                                    : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * kCThreads;
            if (i < a.x_chunks * 8)
                *reinterpret_cast<float4*>(xs + (i >> 3) * kXPad + (i & 7) * 4) = v[u];
        }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kCThreads) : "memory");

    // Per row: (even-k, odd-k) partial sums, scaled per chunk by the group scale.
    float2 acc[V];
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] = make_float2(0.f, 0.f);
    Cursor cur;
    cur.start(a);
    // Where this thread's row of the current item goes, with its bias and (per channel)
    // scale, loaded when the item starts so that the loads overlap the item's stages.
    float* st_out = nullptr;
    float st_bias = 0.f, st_scale = 1.f;
    bool st_ok = false;
    auto prepare = [&](int blk) {
        const MatArgs& m = a.mat[mat_of(a, blk)];
        const int64_t n = (blk - m.blk_begin) * rb + r0 + j;
        st_ok = j < V && n < m.N;
        st_out = m.out + (st_ok ? n : 0);
        st_bias = (st_ok && m.bias) ? __ldg(m.bias + n) : 0.f;
        st_scale = (PC && st_ok) ? load_scale(m.scales, F16, n) : 1.f;
    };
    if (cur.valid(a)) prepare(cur.blk);
    int s = 0;
    uint32_t ph = 0;
    // Per-thread offsets: chunk lane j of the x chunks, the thread's rows of a weight
    // stage (row r at r * kSRB bytes, chunk column c at c * 16), its group-scale rows.
    const uint32_t xthr = smem_u32(xs) + (uint32_t)j * (kXPad * 4);
    const uint32_t w_off = (uint32_t)(r0 * kSRB + j * 16);
    uint32_t s_off[H];
#pragma unroll
    for (int h = 0; h < H; ++h)
        s_off[h] = a.scale_off + scale_slot<rb * esz>((h * 16 + j) >> a.gs_shift, r0 * esz);
    // After a timed-out wait (`dead`) the warp still walks every item, without waiting or
    // computing, so that all consumer warps reach the same named barriers and every split-K
    // ticket is still counted and reset; nothing is stored.
    bool dead = false;
    while (cur.valid(a)) {
        const bool got =
            !dead && __all_sync(0xffffffffu, wait_bounded(full(s), ph, a.wait_ns, failed));
        if (!got && !dead) {
            if (lane == 0) record_failure(a.status, failed);
            dead = true;
        }
        if (got) {
            const uint32_t sb = base + (uint32_t)s * a.stage_bytes;
            const uint32_t xc = xthr + (uint32_t)(cur.ks * kSC) * (kXPad * 4);
#pragma unroll
            for (int h = 0; h < H; ++h) {
                float4 xv[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint4 u = ld_shared_v4(xc + h * 16 * kXPad * 4 + 16 * i);
                    xv[i] = make_float4(__uint_as_float(u.x), __uint_as_float(u.y),
                                        __uint_as_float(u.z), __uint_as_float(u.w));
                }
                float sc[V];
                if (!PC) stage_scales<V, F16>(sb + s_off[h], sc);
                const uint32_t wrow = sb + w_off + h * 256;
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const uint4 wv = ld_shared_v4(wrow + v * kSRB);
                    const float2 d = chunk_dot<EH>(wv, xv);
                    acc[v] = PC ? fadd2(acc[v], d) : ffma2(d, make_float2(sc[v], sc[v]), acc[v]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(s));
        if (++s == S) s = 0, ph ^= 1u;
        const int blk = cur.blk;
        const int part = cur.part;
        if (cur.advance(a)) {
            // Item done: undo the factor 16 of the high-nibble lane, reduce the 16 chunk
            // lanes of each row; store (or hand the partial to the last item).
            float tot[V];
#pragma unroll
            for (int v = 0; v < V; ++v) {
                tot[v] = EH ? fmaf(acc[v].x, 0.0625f, acc[v].y) : fmaf(acc[v].y, 0.0625f, acc[v].x);
#pragma unroll
                for (int o = 1; o < 16; o <<= 1)
                    tot[v] += __shfl_xor_sync(0xffffffffu, tot[v], o);
                acc[v] = make_float2(0.f, 0.f);
            }
            float mine = tot[0];
#pragma unroll
            for (int v = 1; v < V; ++v)
                if (j == v) mine = tot[v];
            const int64_t vrow = (int64_t)blk * rb + r0 + j;  // row in the virtual row space
            bool finish = true;
            if (a.parts > 1) {
                if (j < V) a.ws[(int64_t)part * a.ws_rows + vrow] = mine;
                // The partial sums are ordered before the ticket by the CTA barrier and one
                // device-scope fence of the thread that takes it (cumulative); the last
                // item's reads after it by that thread's second fence and the next barrier.
                asm volatile("bar.sync 1, %0;" ::"r"(kCThreads) : "memory");
                if (threadIdx.x == 0) {
                    __threadfence();
                    const int t = atomicAdd(a.tickets + blk, 1);
                    __threadfence();
                    *s_ticket = t;
                }
                asm volatile("bar.sync 1, %0;" ::"r"(kCThreads) : "memory");
                finish = *s_ticket == a.parts - 1;
                if (finish) {
                    if (j < V) {
                        // All parts' loads in flight together (parts <= 8); added in order.
                        float t[8];
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            t[q] = q < a.parts ? __ldcg(a.ws + (int64_t)q * a.ws_rows + vrow) : 0.f;
                        mine = t[0];
#pragma unroll
                        for (int q = 1; q < 8; ++q)
                            if (q < a.parts) mine += t[q];
                    }
                    if (threadIdx.x == 0) a.tickets[blk] = 0;
                }
            }
            if (finish && st_ok && !*failed) {
                if (PC) mine *= st_scale;
                *st_out = mine + st_bias;
            }
            if (cur.valid(a)) prepare(cur.blk);
        }
    }
}

template <int V, bool EH, bool PC, bool F16>
cudaError_t launch_v(const TensorMaps& tm, const GArgs& a, unsigned grid, const LaunchCtx& c) {
    const cudaError_t attr = kernel_smem_once<gemv_tma_kernel<V, EH, PC, F16>>(kCtaSmem, 100);
    if (attr != cudaSuccess) return attr;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreadsG);
    cfg.dynamicSmemBytes = smem_bytes_g(a.stages, a.stage_bytes, a.x_chunks);
    cfg.stream = c.stream;
    cudaLaunchAttribute attrs[1];
    if (c.pdl) {
        attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attrs;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, gemv_tma_kernel<V, EH, PC, F16>, tm, a);
}

template <int V, bool EH, bool PC>
cudaError_t dispatch_f16(bool f16, const TensorMaps& tm, const GArgs& a, unsigned grid,
                         const LaunchCtx& c) {
    return f16 ? launch_v<V, EH, PC, true>(tm, a, grid, c) : launch_v<V, EH, PC, false>(tm, a, grid, c);
}
template <int V, bool EH>
cudaError_t dispatch_pc(bool pc, bool f16, const TensorMaps& tm, const GArgs& a, unsigned grid,
                        const LaunchCtx& c) {
    return pc ? dispatch_f16<V, EH, true>(f16, tm, a, grid, c)
              : dispatch_f16<V, EH, false>(f16, tm, a, grid, c);
}
template <int V>
cudaError_t dispatch_eh(bool eh, bool pc, bool f16, const TensorMaps& tm, const GArgs& a,
                        unsigned grid, const LaunchCtx& c) {
    return eh ? dispatch_pc<V, true>(pc, f16, tm, a, grid, c)
              : dispatch_pc<V, false>(pc, f16, tm, a, grid, c);
}
cudaError_t dispatch_v(int V, bool eh, bool pc, bool f16, const TensorMaps& tm, const GArgs& a,
                       unsigned grid, const LaunchCtx& c) {
    if (V == 4) return dispatch_eh<4>(eh, pc, f16, tm, a, grid, c);
    if (V == 2) return dispatch_eh<2>(eh, pc, f16, tm, a, grid, c);
    return dispatch_eh<1>(eh, pc, f16, tm, a, grid, c);
}

int log2_exact(int64_t v) {
    for (int s = 0; s < 62; ++s)
        if (((int64_t)1 << s) == v) return s;
    return -1;
}

// Bytes of one stage (weights, then the scale block rounded up to 128 bytes).
uint32_t stage_bytes_for(int V, bool pc, int esz, int gs_shift, uint32_t* scale_off,
                         uint32_t* tx) {
    const int rb = kRowGroups * V;
    const uint32_t wbytes = (uint32_t)(rb * stage_row_bytes(V));
    const int sc_log = chunk_cols(V) == 1 ? 4 : 5;  // log2(chunks per stage)
    const int gps = pc ? 0 : (gs_shift >= sc_log ? 1 : stage_chunks(V) >> gs_shift);
    const uint32_t sbytes = (uint32_t)(gps * rb * esz);
    *scale_off = wbytes;
    *tx = wbytes + sbytes;
    return wbytes + ((sbytes + 1023u) & ~1023u);  // keeps every stage 1024-byte aligned
}

}  // namespace

EncodeTiledFn tensor_map_encoder() {
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

bool gemv_tma_eligible(const Problem& p) {
    if (p.M != 1 || p.K % 32 != 0 || p.K < 512 || p.N < 16) return false;
    if (p.N > (1LL << 30) || p.K > (1LL << 24)) return false;
    if (reinterpret_cast<uintptr_t>(p.x) % 16 || reinterpret_cast<uintptr_t>(p.qweight) % 16)
        return false;
    const bool pc = p.group_size >= p.K;
    if (!pc) {
        // Group scales arrive by TMA: 16-byte aligned base and row stride, group size a
        // power-of-two multiple of 32.
        const int esz = p.scale_f16 ? 2 : 4;
        if (p.group_size % 32 != 0 || log2_exact(p.group_size / 32) < 0) return false;
        if (reinterpret_cast<uintptr_t>(p.scales) % 16 || (p.N * esz) % 16 != 0) return false;
    }
    // x staged whole, plus at least two stages of the smallest tile.
    const int x_chunks = (int)((p.K + 1023) / 1024) * stage_chunks(1);
    uint32_t so, tx;
    const uint32_t sb1 = stage_bytes_for(1, pc, p.scale_f16 ? 2 : 4,
                                         pc ? 0 : log2_exact(p.group_size / 32), &so, &tx);
    if (smem_bytes_g(2, sb1, x_chunks) > kCtaSmem) return false;
    return tensor_map_encoder() != nullptr;
}

int gemv_tma_max_group() { return kMaxMats; }

bool gemv_tma_groupable(const Problem& a, const Problem& b) {
    return a.x == b.x && a.K == b.K && a.group_size == b.group_size &&
           a.scale_f16 == b.scale_f16 && a.even_high == b.even_high &&
           (a.group_size >= a.K) == (b.group_size >= b.K);
}

cudaError_t gemv_tma_launch_group(const Problem* ps, int count, const LaunchCtx& c) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc || count < 1 || count > kMaxMats) return cudaErrorNotSupported;
    const Problem& p0 = ps[0];
    const bool pc = p0.group_size >= p0.K;
    const int esz = p0.scale_f16 ? 2 : 4;
    const int gs_shift = pc ? 0 : log2_exact(p0.group_size / 32);
    auto kstages_for = [&](int V) {
        const int sk = 512 * chunk_cols(V);
        return (int)((p0.K + sk - 1) / sk);
    };
    auto x_chunks_for = [&](int V) { return kstages_for(V) * stage_chunks(V); };
    const int slots = 2 * c.sm_count;
    auto blocks_for = [&](int V) {
        int64_t b = 0;
        for (int i = 0; i < count; ++i) b += (ps[i].N + kRowGroups * V - 1) / (kRowGroups * V);
        return b;
    };
    auto stages_for = [&](int V) {
        uint32_t so, tx;
        const uint32_t sb = stage_bytes_for(V, pc, esz, gs_shift, &so, &tx);
        const int room = kCtaSmem - smem_bytes_g(0, sb, x_chunks_for(V));
        return std::min<int>(kMaxStages, room / (int)sb);
    };
    // Tile shape (V rows per thread) and split-K parts from a cost model of the critical
    // CTA, fitted to measured launch times on GB300 (isolated GEMVs, 1B/8B decode shapes):
    //   cost = waves * (0.06 us per KiB of the CTA's weight bytes * eff(V)
    //                   + 2.1 us for the split-K handoff when parts > 1)
    // with waves = ceil(items / CTA slots).  eff(V) is the relative cost of a weight byte
    // (1.4, 1.1, 1.0 for V = 1, 2, 4: more rows per thread reuse each x chunk more).
    int V = 1, best_parts = 1;
    double best = 1e30;
    for (int v : {1, 2, 4}) {
        if (stages_for(v) < 2) continue;
        const int64_t blocks_v = blocks_for(v);
        const double eff = v == 1 ? 1.4 : (v == 2 ? 1.1 : 1.0);
        for (int parts = 1; parts <= kGemvMaxParts; parts *= 2) {
            const int kstages = kstages_for(v);
            if (parts > 1 && (kstages * 512 * chunk_cols(v) / parts < 2048 || !c.ws || !c.tickets ||
                              (int64_t)parts * blocks_v * kRowGroups * v > c.ws_floats ||
                              blocks_v > c.ticket_count))
                break;
            const int tpp = (kstages + parts - 1) / parts;
            const int64_t items = blocks_v * ((kstages + tpp - 1) / tpp);
            const double waves = (double)((items + slots - 1) / slots);
            const double kib = (double)kRowGroups * v * tpp * stage_row_bytes(v) / 1024.0;
            const double cost = waves * (0.06 * kib * eff + (parts > 1 ? 2.1 : 0.0));
            if (cost < best * 0.999) best = cost, V = v, best_parts = parts;
        }
    }
    const int rb = kRowGroups * V;
    GArgs a = {};
    a.x = p0.x;
    a.nmat = count;
    a.K = p0.K;
    const int kstages = kstages_for(V);
    a.kstages = kstages;
    a.x_chunks = x_chunks_for(V);
    a.gs_shift = gs_shift;
    a.stage_bytes = stage_bytes_for(V, pc, esz, gs_shift, &a.scale_off, &a.stage_tx);
    a.stages = stages_for(V);
    if (a.stages < 2) return cudaErrorNotSupported;
    a.status = c.status_word;
    a.wait_ns = c.wait_limit_ns;
    TensorMaps tm;
    int64_t blocks = 0;
    for (int i = 0; i < count; ++i) {
        const Problem& p = ps[i];
        a.mat[i].scales = p.scales;
        a.mat[i].bias = p.bias;
        a.mat[i].out = p.out;
        a.mat[i].N = p.N;
        a.mat[i].blk_begin = blocks;
        blocks += (p.N + rb - 1) / rb;
        {
            const cuuint64_t dims[2] = {(cuuint64_t)(p.K / 4), (cuuint64_t)p.N};
            const cuuint64_t strides[1] = {(cuuint64_t)(p.K / 2)};
            const cuuint32_t box[2] = {(cuuint32_t)(stage_row_bytes(V) / 2), (cuuint32_t)rb};
            const cuuint32_t estr[2] = {1, 1};
            if (enc(&tm.w[i], CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint8_t*>(p.qweight),
                    dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return cudaErrorInvalidValue;
        }
        if (!pc) {
            const int64_t G = (p.K + p.group_size - 1) / p.group_size;
            const int sc_log = chunk_cols(V) == 1 ? 4 : 5;
            const int gps = gs_shift >= sc_log ? 1 : stage_chunks(V) >> gs_shift;
            const cuuint64_t dims[2] = {(cuuint64_t)p.N, (cuuint64_t)G};
            const cuuint64_t strides[1] = {(cuuint64_t)(p.N * esz)};
            const cuuint32_t box[2] = {(cuuint32_t)rb, (cuuint32_t)gps};
            const cuuint32_t estr[2] = {1, 1};
            const int ib = rb * esz;
            const CUtensorMapSwizzle swz = ib == 32    ? CU_TENSOR_MAP_SWIZZLE_32B
                                           : ib == 64  ? CU_TENSOR_MAP_SWIZZLE_64B
                                           : ib == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                                       : CU_TENSOR_MAP_SWIZZLE_NONE;
            if (enc(&tm.s[i], p.scale_f16 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT32,
                    2, const_cast<void*>(p.scales), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return cudaErrorInvalidValue;
        } else {
            tm.s[i] = tm.w[i];  // unused
        }
    }
    for (int i = count; i < kMaxMats; ++i) {
        a.mat[i] = a.mat[count - 1];
        a.mat[i].blk_begin = blocks;  // never selected: begins past the last block
        tm.w[i] = tm.w[count - 1];
        tm.s[i] = tm.s[count - 1];
    }
    a.row_blocks = blocks;
    a.parts = best_parts;
    a.tpp = (kstages + a.parts - 1) / a.parts;
    a.parts = (kstages + a.tpp - 1) / a.tpp;  // no empty part
    a.items = (int)(blocks * a.parts);
    a.ws = c.ws;
    a.tickets = c.tickets;
    a.ws_rows = blocks * rb;
    const unsigned grid = (unsigned)std::min<int64_t>(a.items, slots);
    return dispatch_v(V, p0.even_high != 0, pc, p0.scale_f16 != 0, tm, a, grid, c);
}

cudaError_t gemv_tma_launch(const Problem& p, const LaunchCtx& c) {
    return gemv_tma_launch_group(&p, 1, c);
}

}  // namespace q4lin
