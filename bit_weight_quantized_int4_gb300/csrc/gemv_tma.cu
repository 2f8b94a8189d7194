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
//     scales are fetched three tiles ahead.  A warp reads 512 contiguous bytes of the tile
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
constexpr int kRingBytes = 128 * 1024;      // weight tiles in flight per SM
constexpr int kScaleRing = 4;              // tiles of scales in flight per thread
constexpr int kXPad = 36;                  // floats per 32-float x chunk in shared memory
constexpr int64_t kDrainNs = 4000000000LL;
constexpr int kMaxSmemG = 227 * 1024;
constexpr int kMaxMats = 4;

// One weight matrix of a launch.  Several matrices that share x (the q/k/v projections
// of a layer, or gate/up) run in one launch over a virtual row space: matrix i owns the
// row blocks [blk_begin, blk_begin + row_blocks).
struct MatArgs {
    const void* scales;
    const float* bias;
    float* out;
    int64_t N;
    int64_t blk_begin;
};
struct TensorMaps {
    CUtensorMap m[kMaxMats];
};

struct GArgs {
    const float* x;
    MatArgs mat[kMaxMats];
    int nmat;
    int64_t K, gs;
    int scale_f16, per_channel, kslices, x_chunks;
    int k_chunks;   // K / 32
    int gs_chunks;  // group size / 32 (grouped scales)
    int gs_shift;   // log2(gs_chunks) when a power of two, else -1
    int64_t row_blocks;
    // Split K: each row block's k-slices are cut into `parts` runs of `tpp` slices; a work
    // item is (row block, part).  With parts > 1 the items write partial row sums to
    // ws[part * ws_rows + row] and the last item of a row block (ticket count) adds them
    // in part order, so the result does not depend on which CTA finishes last.
    int parts, tpp;
    int items;
    float* ws;       // [parts, ws_rows] partial sums (parts > 1)
    int* tickets;    // [row_blocks], zero between launches (the last item resets its own)
    int64_t ws_rows; // row_blocks * rows per block
    int* status;
    int64_t wait_ns;
};

// A CTA's walk over its work items: item = blockIdx.x + i * gridDim.x, item -> (row block
// blk = item / parts, part), covering k-slices [part * tpp, min((part + 1) * tpp, kslices)).
// One division per item, none per tile.
struct Cursor {
    int item, blk, part, ks, ks_end;
    __device__ __forceinline__ void set(const GArgs& a) {
        blk = item / a.parts;
        part = item - blk * a.parts;
        ks = part * a.tpp;
        ks_end = min(ks + a.tpp, a.kslices);
    }
    __device__ __forceinline__ void start(const GArgs& a) {
        item = (int)blockIdx.x;
        if (item < a.items) set(a);
    }
    __device__ __forceinline__ bool valid(const GArgs& a) const { return item < a.items; }
    // Move to the next tile; true when that finished the current item.
    __device__ __forceinline__ bool advance(const GArgs& a) {
        if (++ks < ks_end) return false;
        item += gridDim.x;
        if (item < a.items) set(a);
        return true;
    }
};

// Ring depth for row blocks of rb rows: always kRingBytes of tiles (4, 8 or 16 stages).
__host__ __device__ constexpr int stages_for(int rb) { return kRingBytes / (rb * kSliceBytes); }
// Shared memory: the stage ring, the barriers, then x (padded chunks of 32 floats).
__host__ __device__ constexpr int ring_bytes(int rb) { return stages_for(rb) * rb * kSliceBytes; }
__host__ __device__ constexpr int x_offset(int rb) {
    return ring_bytes(rb) + 16 * stages_for(rb) + 16;
}
inline int smem_bytes_g(int rb, int64_t K) {
    return 128 + x_offset(rb) + (int)((K + kSliceK - 1) / kSliceK * 16) * kXPad * 4;
}

__device__ __forceinline__ float load_scale(const void* scales, int f16, int64_t idx) {
    if (f16) return __half2float(__ldg(reinterpret_cast<const __half*>(scales) + idx));
    return __ldg(reinterpret_cast<const float*>(scales) + idx);
}

// Raw bits of one scale (binary16 in the low half, or fp32).  Kept raw in the prefetch
// ring and converted only when used: converting at load time would make the thread wait
// for the load right away.
template <bool F16>
__device__ __forceinline__ uint32_t scale_bits(const void* scales, int64_t idx) {
    if (F16) return __ldg(reinterpret_cast<const unsigned short*>(scales) + idx);
    return __ldg(reinterpret_cast<const unsigned int*>(scales) + idx);
}
template <bool F16>
__device__ __forceinline__ float scale_value(uint32_t bits) {
    if (F16) return __half2float(__ushort_as_half((unsigned short)bits));
    return __uint_as_float(bits);
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
__global__ void __launch_bounds__(kThreadsG, 1)
    gemv_tma_kernel(const __grid_constant__ TensorMaps tmaps, const GArgs a) {
    constexpr int rb = 32 * V;  // rows per block: 32 row groups of V rows
    constexpr uint32_t tile_bytes = rb * kSliceBytes;
    constexpr int kStagesG = stages_for(rb);
    static_assert((kStagesG & (kStagesG - 1)) == 0, "ring depth must be a power of two");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 127u) & ~127u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t bar_base = base + ring_bytes(rb);
    volatile int* failed =
        reinterpret_cast<volatile int*>(gbase + (bar_base + 16 * kStagesG - base));
    volatile int* s_ticket = failed + 1;  // last-item decision, broadcast to the consumers
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
            for (int q = 0; q < a.nmat; ++q) prefetch_tensormap(&tmaps.m[q]);
            int t = 0;
            Cursor cur;
            cur.start(a);
            while (cur.valid(a)) {
                const int s = t & (kStagesG - 1);
                if (t >= kStagesG &&
                    !wait_bounded(empty(s), (uint32_t)((t / kStagesG) - 1) & 1, a.wait_ns, failed)) {
                    record_failure(a.status, failed);
                    break;
                }
                if (*failed) break;
                const int mi = mat_of(a, cur.blk);
                mbar_arrive_expect_tx(full(s), tile_bytes);
                tma_load_2d(base + s * tile_bytes, &tmaps.m[mi], cur.ks * kSliceBytes,
                            (int)((cur.blk - a.mat[mi].blk_begin) * rb), full(s));
                ++t;
                cur.advance(a);
            }
            // The last armed tiles may still be landing; the CTA must not exit first.
            for (int q = t > kStagesG ? t - kStagesG : 0; q < t; ++q)
                wait_bounded(full(q & (kStagesG - 1)), (uint32_t)(q / kStagesG) & 1, kDrainNs,
                             nullptr);
        }
        return;
    }

    // ------------------------------------------------------------------ consumers
    const int j = threadIdx.x & 15;          // chunk lane within a 256-byte slice
    const int r0 = (threadIdx.x >> 4) * V;   // first of this thread's V rows in a block

    // Scales of this thread's tiles, kScaleRing - 1 tiles ahead of use.  Tile t uses
    // ring slot t % kScaleRing and refills it for tile t + kScaleRing right after; the
    // tile loop is unrolled by the ring size so every slot has a fixed register (moving
    // a register whose load is in flight would wait for the load).  The first loads go
    // out before griddep_wait: scales do not depend on the preceding kernel.  Tile
    // coordinates advance incrementally (no integer division in the loop).
    int tiles_mine = 0;
    for (int it = blockIdx.x; it < a.items; it += gridDim.x) {
        const int part = it % a.parts;
        tiles_mine += min(a.tpp, a.kslices - part * a.tpp);
    }
    Cursor pf;
    pf.start(a);
    auto fetch_next = [&](uint32_t (&dst)[V]) {
        if (!PC && pf.valid(a)) {
            const int chunk = pf.ks * 16 + j;
            const int mi = mat_of(a, pf.blk);
            const MatArgs& m = a.mat[mi];
            const int64_t n0 = (pf.blk - m.blk_begin) * rb + r0;
            if (chunk < a.k_chunks) {
                const int g = a.gs_shift >= 0 ? (chunk >> a.gs_shift) : chunk / a.gs_chunks;
                const int64_t bi = (int64_t)g * m.N + n0;
                if (n0 + V <= m.N) {
#pragma unroll
                    for (int v = 0; v < V; ++v) dst[v] = scale_bits<F16>(m.scales, bi + v);
                } else {
#pragma unroll
                    for (int v = 0; v < V; ++v)
                        dst[v] = n0 + v < m.N ? scale_bits<F16>(m.scales, bi + v) : 0u;
                }
            } else {
#pragma unroll
                for (int v = 0; v < V; ++v) dst[v] = 0u;
            }
        }
        if (pf.valid(a)) pf.advance(a);
    };
    uint32_t sc[kScaleRing][V];
#pragma unroll
    for (int u = 0; u < kScaleRing; ++u) fetch_next(sc[u]);

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

    // Per row: (even-k, odd-k) partial sums, scaled per chunk by the group scale.
    float2 acc[V];
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] = make_float2(0.f, 0.f);
    Cursor cur;
    cur.start(a);
    const float* xrow = xs + j * kXPad;
    bool dead = false;
    for (int t0 = 0; t0 < tiles_mine && !dead; t0 += kScaleRing) {
#pragma unroll
        for (int u = 0; u < kScaleRing; ++u) {
            const int t = t0 + u;
            if (t >= tiles_mine) break;
            const int s = t & (kStagesG - 1);
            float4 xv[8];
            const float* xc = xrow + cur.ks * (16 * kXPad);
#pragma unroll
            for (int i = 0; i < 8; ++i) xv[i] = *reinterpret_cast<const float4*>(xc + 4 * i);
            const bool got = __all_sync(
                0xffffffffu, wait_bounded(full(s), (uint32_t)(t / kStagesG) & 1, a.wait_ns, failed));
            if (!got) {
                if (lane == 0) record_failure(a.status, failed);
                dead = true;
                break;
            }
            const uint32_t wrow = base + s * tile_bytes + r0 * kSliceBytes + j * 16;
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const uint4 wv = ld_shared_v4(wrow + v * kSliceBytes);
                const float2 d = chunk_dot<EH>(wv, xv);
                if (PC) {
                    acc[v] = fadd2(acc[v], d);
                } else {
                    const float sv = scale_value<F16>(sc[u][v]);
                    acc[v] = ffma2(d, make_float2(sv, sv), acc[v]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(s));
            fetch_next(sc[u]);
            const int blk = cur.blk;
            const int part = cur.part;
            if (cur.advance(a)) {
                // Item done: undo the factor 16 of the high-nibble lane, reduce the 16
                // chunk lanes of each row; store (or hand the partial to the last item).
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
                const MatArgs& m = a.mat[mat_of(a, blk)];
                const int64_t n = (blk - m.blk_begin) * rb + r0 + j;
                const int64_t vrow = (int64_t)blk * rb + r0 + j;  // row in the virtual row space
                bool finish = true;
                if (a.parts > 1) {
                    if (j < V) a.ws[(int64_t)part * a.ws_rows + vrow] = mine;
                    __threadfence();
                    asm volatile("bar.sync 1, %0;" ::"r"(kCThreads) : "memory");
                    if (threadIdx.x == 0) *s_ticket = atomicAdd(a.tickets + blk, 1);
                    asm volatile("bar.sync 1, %0;" ::"r"(kCThreads) : "memory");
                    finish = *s_ticket == a.parts - 1;
                    if (finish) {
                        __threadfence();
                        if (j < V) {
                            mine = 0.f;
                            for (int q = 0; q < a.parts; ++q)
                                mine += __ldcg(a.ws + (int64_t)q * a.ws_rows + vrow);
                        }
                        if (threadIdx.x == 0) a.tickets[blk] = 0;
                    }
                }
                if (finish && j < V && n < m.N) {
                    if (PC) mine *= scale_value<F16>(scale_bits<F16>(m.scales, n));
                    if (m.bias) mine += __ldg(m.bias + n);
                    m.out[n] = mine;
                }
            }
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

template <int V, bool EH, bool PC, bool F16>
cudaError_t launch_v(const TensorMaps& tm, const GArgs& a, unsigned grid, const LaunchCtx& c) {
    static cudaError_t attr = cudaFuncSetAttribute(
        gemv_tma_kernel<V, EH, PC, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmemG);
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

}  // namespace

bool gemv_tma_eligible(const Problem& p) {
    if (p.M != 1 || p.K % 32 != 0 || p.K < 2 * kSliceBytes || p.N < 32) return false;
    if (smem_bytes_g(128, p.K) > kMaxSmemG) return false;
    if (reinterpret_cast<uintptr_t>(p.x) % 16 || reinterpret_cast<uintptr_t>(p.qweight) % 16)
        return false;
    if (!(p.group_size >= p.K || p.group_size % 32 == 0)) return false;
    if (p.N > (1LL << 30)) return false;
    return encode_fn() != nullptr;
}

int gemv_tma_max_group() { return kMaxMats; }

bool gemv_tma_groupable(const Problem& a, const Problem& b) {
    return a.x == b.x && a.K == b.K && a.group_size == b.group_size &&
           a.scale_f16 == b.scale_f16 && a.even_high == b.even_high &&
           (a.group_size >= a.K) == (b.group_size >= b.K);
}

cudaError_t gemv_tma_launch_group(const Problem* ps, int count, const LaunchCtx& c) {
    EncodeTiledFn enc = encode_fn();
    if (!enc || count < 1 || count > kMaxMats) return cudaErrorNotSupported;
    const Problem& p0 = ps[0];
    int64_t rows = 0;
    for (int i = 0; i < count; ++i) rows += ps[i].N;
    // Rows per block: as large as the GPU stays busy with (more rows per thread reuse
    // the x chunk more), smaller for short matrices so every SM gets a block.
    int V = 4;
    if ((rows + 127) / 128 < c.sm_count) V = 2;
    if ((rows + 63) / 64 < c.sm_count) V = 1;
    const int rb = 32 * V;
    GArgs a = {};
    a.x = p0.x;
    a.nmat = count;
    a.K = p0.K;
    a.gs = p0.group_size;
    a.scale_f16 = p0.scale_f16;
    a.per_channel = p0.group_size >= p0.K;
    a.kslices = (int)((p0.K + kSliceK - 1) / kSliceK);
    a.x_chunks = a.kslices * 16;
    a.k_chunks = (int)(p0.K / 32);
    a.gs_chunks = a.per_channel ? 1 : (int)(p0.group_size / 32);
    a.gs_shift = -1;
    for (int sft = 0; sft < 31; ++sft)
        if ((1 << sft) == a.gs_chunks) a.gs_shift = sft;
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
        const int64_t Kp = p.K / 2;
        const cuuint64_t dims[2] = {(cuuint64_t)Kp, (cuuint64_t)p.N};
        const cuuint64_t strides[1] = {(cuuint64_t)Kp};
        const cuuint32_t box[2] = {(cuuint32_t)kSliceBytes, (cuuint32_t)rb};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&tm.m[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(p.qweight), dims,
                strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    for (int i = count; i < kMaxMats; ++i) {
        a.mat[i] = a.mat[count - 1];
        a.mat[i].blk_begin = blocks;  // never selected: begins past the last block
        tm.m[i] = tm.m[count - 1];
    }
    a.row_blocks = blocks;
    // Split K when the row blocks alone would leave SMs idle (the widening is ALU work,
    // so every SM should get a share), if the handle's workspace can hold the partials.
    // The partial-sum handoff costs a dependent round trip through L2, so a part keeps at
    // least 8 k-slices (4096 k): only long rows are split.
    a.parts = 1;
    if (blocks < c.sm_count && c.ws && c.tickets) {
        int parts = (int)std::min<int64_t>(c.sm_count / blocks, a.kslices / 8);
        while (parts > 1 && ((int64_t)parts * blocks * rb > c.ws_floats || blocks > c.ticket_count))
            --parts;
        a.parts = std::max(parts, 1);
    }
    a.tpp = (a.kslices + a.parts - 1) / a.parts;
    a.parts = (a.kslices + a.tpp - 1) / a.tpp;  // no empty part
    a.items = (int)(blocks * a.parts);
    a.ws = c.ws;
    a.tickets = c.tickets;
    a.ws_rows = blocks * rb;
    const unsigned grid = (unsigned)std::min<int64_t>(a.items, c.sm_count);
    return dispatch_v(V, p0.even_high != 0, a.per_channel != 0, a.scale_f16 != 0, tm, a, grid, c);
}

cudaError_t gemv_tma_launch(const Problem& p, const LaunchCtx& c) {
    return gemv_tma_launch_group(&p, 1, c);
}

}  // namespace q4lin
