// gemv_mr.cu -- TMA-fed GEMV for a few activation rows (2 <= M <= 4) of the 4-bit
// weight-quantized linear (sm_103a).
//
//   out[m, n] = bias[n] + sum_k x[m, k] * (code[n, k] - 8) * scale[k / gs, n]
//
// (the formula of "[ExecuTorch][WebGPU] Add linear_qcs4w op", Solution; the small-M
// regime below the tensor-core crossover, where each dequantized weight is reused across
// the M activation rows.)
//
// A producer warp streams per stage (512 k) the packed weights of a block of 16 V rows
// [16 V x 256 B] (V = 4, or 2 when 32-row blocks avoid a split of K that 64-row blocks
// need), their group scales [groups of the stage x (16 V + 8) fp16 / (16 V + 4) fp32 rows:
// the padded row stride spreads the 16 chunk lanes' group rows over the banks] and the x
// tile [MR rows x 512 k] (MR = M; a 3D box of 128-byte chunk rows with the 128-byte
// swizzle, so that the 16 chunk lanes reading the same offset of 16 chunks hit different
// banks) into a ring, all on one mbarrier; the weight and scale copies of the first
// stages go out before the grid-dependency wait, their x copies after it.
// Consumer thread = (chunk lane j of 16, row group of V rows): per stage it takes chunk j
// (32 k, one group) of its V rows, word by word (8 k, in a lane-rotated order that keeps
// the warp's code reads on 32 banks): it loads the x values of the MR rows once, widens
// each row's word once (byte permute + packed add, as in the M = 1 GEMV) and issues MR
// packed FMAs per pair of codes; the group scale multiplies the stage's unscaled sums
// once.  So x is read from shared memory once per V rows and each code is widened once
// for all MR rows.  The 16 chunk lanes of a row group are added with shuffles; lane j
// then holds all (m, row) sums and stores sum (j / V, j % V).  When the row blocks alone
// leave SMs idle, K is cut into parts; the parts write partial sums to the handle's
// workspace and the last item of a row block (an atomic ticket) adds them in part order
// (deterministic).  Every wait is bounded in time; after a timeout the warps walk their
// remaining items without waiting or computing, so the barriers and tickets are still
// reached.
#include <cuda_fp16.h>

#include <algorithm>

#include "ptx.cuh"
#include "q4lin_internal.h"

namespace q4lin {
namespace {
using namespace ptx;

constexpr int kMrCWarps = 8;                          // consumer warps
constexpr int kMrCThreads = 32 * kMrCWarps;
constexpr int kMrThreads = kMrCThreads + 32;          // + the producer warp
// V weight rows per consumer thread (4, or 2 when that saves a split of K): a block is
// 16 row groups of V rows.
__host__ __device__ constexpr int mr_rows(int V) { return 16 * V; }
constexpr int kMrStageK = 512;                        // k per stage: 16 chunks of 32
__host__ __device__ constexpr uint32_t mr_code_bytes(int V) { return mr_rows(V) * kMrStageK / 2; }
// Staged scale rows per group: the block's rows plus padding that spreads the 16 chunk
// lanes' group rows over the banks (a whole number of 16-byte units).
__host__ __device__ constexpr int mr_sc_rows(int V, bool f16) { return mr_rows(V) + (f16 ? 8 : 4); }
constexpr uint32_t kMrScBytes = 4608;                 // >= 16 groups x 68 fp32 rows (V = 4)
constexpr int kMrMaxStages = 8;
constexpr int kMrSmem = 113 * 1024;                   // two CTAs per SM
constexpr int64_t kMrDrainNs = 4000000000LL;

struct MrMaps {
    CUtensorMap w;  // uint8 [N, K/2], box {256, 16 V}
    CUtensorMap s;  // scales [G, N], box {16 V + 8 (fp16) / + 4 (fp32), groups per stage}
    CUtensorMap x;  // fp32 [M][K/32][32], box {32, 16, MR}, 128-byte swizzle
};

struct MrArgs {
    const float* bias;
    float* out;
    float* ws;       // [parts][MR][ws_rows] partial sums (parts > 1)
    int* tickets;    // [row_blocks], zero between launches
    int* status;
    int64_t M, N, ws_rows;
    int kstages, stages;
    uint32_t stage_bytes, tx;
    int gs_in_stage;       // group size when a stage holds whole groups (gs <= 512), else 0
    int gshift;            // then: group row of stage ks = ks << gshift
    int stages_per_group;  // else: group row = ks / stages_per_group
    int sc_rows;
    int parts, tpp, items;
    int64_t wait_ns;
    int skip_copies;  // test hook: the producer issues nothing, so the consumers' waits run out
};

// A CTA's walk over its work items (row block, part of K), as in the M = 1 GEMV.
struct MrCursor {
    int item, blk, part, ks, ks_end;
    __device__ __forceinline__ void set(const MrArgs& a) {
        blk = item / a.parts;
        part = item - blk * a.parts;
        ks = part * a.tpp;
        ks_end = min(ks + a.tpp, a.kstages);
    }
    __device__ __forceinline__ void start(const MrArgs& a) {
        item = (int)blockIdx.x;
        if (item < a.items) set(a);
    }
    __device__ __forceinline__ bool valid(const MrArgs& a) const { return item < a.items; }
    __device__ __forceinline__ bool advance(const MrArgs& a) {
        if (++ks < ks_end) return false;
        item += gridDim.x;
        if (item < a.items) set(a);
        return true;
    }
};

template <int MR, int V, bool EH, bool F16>
__global__ void __launch_bounds__(kMrThreads, 2)
    gemv_mr_kernel(const __grid_constant__ MrMaps maps, const MrArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const int S = a.stages;
    const uint32_t bar_base = base + (uint32_t)S * a.stage_bytes;
    volatile int* failed = reinterpret_cast<volatile int*>(gbase + (bar_base + 16 * kMrMaxStages - base));
    volatile int* s_ticket = failed + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto full = [&](int s) { return bar_base + 8u * s; };
    auto empty = [&](int s) { return bar_base + 8u * (kMrMaxStages + s); };
    constexpr uint32_t kXBytes = (uint32_t)MR * 2048;  // x tile, then codes, then scales
    constexpr int kRows = mr_rows(V);
    constexpr uint32_t kCodeBytes = mr_code_bytes(V);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), kMrCWarps);
        }
        *failed = 0;
        mbar_init_fence();
    }
    __syncthreads();
    griddep_launch_dependents();

    if (warp == kMrCWarps) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0 && !a.skip_copies) {
            prefetch_tensormap(&maps.w);
            prefetch_tensormap(&maps.s);
            prefetch_tensormap(&maps.x);
            int t = 0, s = 0;
            uint32_t ph = 0;
            MrCursor cur;
            cur.start(a);
            // The first stages are armed, and their weights and scales (which the preceding
            // grid does not write) requested, before griddepcontrol.wait; their x tiles
            // follow after it.
            int pre_ks[kMrMaxStages];
            while (cur.valid(a) && t < S) {
                const uint32_t sb = base + (uint32_t)t * a.stage_bytes;
                const int row0 = cur.blk * kRows;
                const int grow = a.gs_in_stage ? (cur.ks << a.gshift) : cur.ks / a.stages_per_group;
                mbar_arrive_expect_tx(full(t), a.tx);
                tma_load_2d(sb + kXBytes, &maps.w, cur.ks * (kMrStageK / 2), row0, full(t));
                tma_load_2d(sb + kXBytes + kCodeBytes, &maps.s, row0, grow, full(t));
                pre_ks[t] = cur.ks;
                ++t;
                cur.advance(a);
            }
            griddep_wait();  // x comes from the preceding grid
            for (int q = 0; q < t; ++q)
                tma_load_3d(base + (uint32_t)q * a.stage_bytes, &maps.x, 0,
                            pre_ks[q] * (kMrStageK / 32), 0, full(q));
            if (t == S) s = 0, ph = 1;
            else s = t;
            while (cur.valid(a)) {
                if (!wait_bounded(empty(s), ph ^ 1u, a.wait_ns, failed)) {
                    record_failure(a.status, failed);
                    break;
                }
                if (*failed) break;
                const uint32_t sb = base + (uint32_t)s * a.stage_bytes;
                const int row0 = cur.blk * kRows;
                const int grow = a.gs_in_stage ? (cur.ks << a.gshift) : cur.ks / a.stages_per_group;
                mbar_arrive_expect_tx(full(s), a.tx);
                tma_load_2d(sb + kXBytes, &maps.w, cur.ks * (kMrStageK / 2), row0, full(s));
                tma_load_2d(sb + kXBytes + kCodeBytes, &maps.s, row0, grow, full(s));
                tma_load_3d(sb, &maps.x, 0, cur.ks * (kMrStageK / 32), 0, full(s));
                ++t;
                if (++s == S) s = 0, ph ^= 1u;
                cur.advance(a);
            }
            for (int q = t > S ? t - S : 0; q < t; ++q)
                wait_bounded(full(q % S), (uint32_t)(q / S) & 1u, kMrDrainNs, nullptr);
        }
        return;
    }

    // ------------------------------------------------------------------ consumers
    const int j = threadIdx.x & 15;          // chunk lane: chunk j (32 k) of every stage
    const int rg = threadIdx.x >> 4;         // row group: rows V rg .. V rg + V - 1 of a block
    const int gl = a.gs_in_stage ? (j * 32) / a.gs_in_stage : 0;  // group row in the stage
    // A thread takes the 4 words of its chunk in a rotated order, so that the 32 lanes of a
    // warp (chunks j and j + 8 are 128 bytes apart, the two row groups V x 256 bytes apart)
    // read 32 different banks.
    const int rot = (j >> 3) + 2 * (rg & 1);
    constexpr uint32_t esz = F16 ? 2 : 4;
    // Per-thread offsets inside a stage: x chunk j of row m, 16-byte unit u at
    // m * 2048 + j * 128 + ((u ^ (j & 7)) << 4); the thread's code chunk of row v at
    // v * 256; its V consecutive scales of group row gl.
    const uint32_t x_off = (uint32_t)j * 128;
    const uint32_t w_off = kXBytes + (uint32_t)(rg * V) * 256 + (uint32_t)j * 16;
    const uint32_t s_off = kXBytes + kCodeBytes + ((uint32_t)gl * a.sc_rows + rg * V) * esz;
    // The products of a stage are summed unscaled over the thread's 32 k (one group: part,
    // even-k and odd-k sums) and the group scale is applied once per stage (acc.x).
    float2 acc[MR][V];
#pragma unroll
    for (int m = 0; m < MR; ++m)
#pragma unroll
        for (int v = 0; v < V; ++v) acc[m][v] = make_float2(0.f, 0.f);
    int s = 0;
    uint32_t ph = 0;
    bool dead = false;
    MrCursor cur;
    cur.start(a);
    while (cur.valid(a)) {
        const bool got =
            !dead && __all_sync(0xffffffffu, wait_bounded(full(s), ph, a.wait_ns, failed));
        if (!got && !dead) {
            if (lane == 0) record_failure(a.status, failed);
            dead = true;
        }
        if (got) {
            // Plain shared-memory loads (after the barrier wait, which orders them), so
            // that the compiler may schedule them early.
            const uint8_t* st = gbase + (size_t)s * a.stage_bytes;
            const uint8_t* xs = st + x_off;
            const uint8_t* cs = st + w_off;
            float sc[V];  // the V rows' scales of the thread's group row
            if constexpr (V == 4) {
                if (F16) {
                    const uint2 hv = *reinterpret_cast<const uint2*>(st + s_off);
                    const float2 p = __half22float2(*reinterpret_cast<const __half2*>(&hv.x));
                    const float2 q = __half22float2(*reinterpret_cast<const __half2*>(&hv.y));
                    sc[0] = p.x, sc[1] = p.y, sc[2] = q.x, sc[3] = q.y;
                } else {
                    const float4 f = *reinterpret_cast<const float4*>(st + s_off);
                    sc[0] = f.x, sc[1] = f.y, sc[2] = f.z, sc[3] = f.w;
                }
            } else {
                static_assert(V == 2, "4 or 2 rows per thread");
                const float2 f = F16 ? __half22float2(*reinterpret_cast<const __half2*>(st + s_off))
                                     : *reinterpret_cast<const float2*>(st + s_off);
                sc[0] = f.x, sc[1] = f.y;
            }
            float2 part[MR][V];
#pragma unroll
            for (int m = 0; m < MR; ++m)
#pragma unroll
                for (int v = 0; v < V; ++v) part[m][v] = make_float2(0.f, 0.f);
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                // Word we of each of the 4 rows: k = 32 j + 8 we + (0..7).
                const int we = (w + rot) & 3;
                uint32_t lo[V], hi[V];
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const uint32_t word = *reinterpret_cast<const uint32_t*>(cs + v * 256 + we * 4);
                    const uint32_t m4 = word & 0x0F0F0F0Fu, s4 = (word >> 4) & 0x0F0F0F0Fu;
                    lo[v] = EH ? s4 : m4;
                    hi[v] = EH ? m4 : s4;
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    // x of k = 32 j + 8 we + 4 h + (0..3) for the MR rows: unit 2 we + h.
                    const uint32_t xu = (uint32_t)((2 * we + h) ^ (j & 7)) << 4;
                    float2 xv[MR][2];
#pragma unroll
                    for (int m = 0; m < MR; ++m) {
                        const float4 p = *reinterpret_cast<const float4*>(xs + m * 2048 + xu);
                        xv[m][0] = make_float2(p.x, p.y);
                        xv[m][1] = make_float2(p.z, p.w);
                    }
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        // Pairs (k even, k odd) of bytes 2h and 2h + 1 as exact c - 8.
                        float2 c[2];
#pragma unroll
                        for (int b = 0; b < 2; ++b) {
                            const uint32_t sel = 0x7440u | (uint32_t)(2 * h + b);
                            c[b] = fadd2(make_float2(__uint_as_float(prmt(lo[v], 0x4B000000u, sel)),
                                                     __uint_as_float(prmt(hi[v], 0x4B000000u, sel))),
                                         make_float2(-8388616.0f, -8388616.0f));
                        }
#pragma unroll
                        for (int m = 0; m < MR; ++m)
#pragma unroll
                            for (int b = 0; b < 2; ++b) part[m][v] = ffma2(c[b], xv[m][b], part[m][v]);
                    }
                }
            }
#pragma unroll
            for (int m = 0; m < MR; ++m)
#pragma unroll
                for (int v = 0; v < V; ++v)
                    acc[m][v].x = fmaf(sc[v], part[m][v].x + part[m][v].y, acc[m][v].x);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(s));
        if (++s == S) s = 0, ph ^= 1u;
        const int blk = cur.blk, part = cur.part;
        if (cur.advance(a)) {
            // Item done: reduce the 16 chunk lanes of every (m, row); lane j keeps sum
            // (m, v) = (j / 4, j % 4).
            float mine = 0.f;
#pragma unroll
            for (int m = 0; m < MR; ++m)
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    float t = acc[m][v].x + acc[m][v].y;
#pragma unroll
                    for (int o = 1; o < 16; o <<= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                    if (j == m * V + v) mine = t;
                    acc[m][v] = make_float2(0.f, 0.f);
                }
            const int mj = j / V, vj = j % V;
            const int64_t nrow = (int64_t)blk * kRows + rg * V + vj;  // row of the matrix
            const bool mine_ok = mj < MR;
            griddep_wait();  // (long complete: the x copies waited for it) before any store
            bool finish = true;
            if (a.parts > 1) {
                if (mine_ok) a.ws[((int64_t)part * MR + mj) * a.ws_rows + nrow] = mine;
                // The consumers' partial sums are ordered before the ticket by the CTA
                // barrier and one device-scope fence of the thread that takes the ticket
                // (cumulative); the last item's reads are ordered after it by that thread's
                // second fence and the barrier that follows.
                asm volatile("bar.sync 1, %0;" ::"r"(kMrCThreads) : "memory");
                if (threadIdx.x == 0) {
                    __threadfence();
                    const int t = atomicAdd(a.tickets + blk, 1);
                    __threadfence();
                    *s_ticket = t;
                }
                asm volatile("bar.sync 1, %0;" ::"r"(kMrCThreads) : "memory");
                finish = *s_ticket == a.parts - 1;
                if (finish) {
                    if (mine_ok) {
                        // Parts added in part order: the sum does not depend on which
                        // item finished last.
                        const float* wp = a.ws + (int64_t)mj * a.ws_rows + nrow;
                        mine = __ldcg(wp);
                        for (int q = 1; q < a.parts; ++q) mine += __ldcg(wp + (int64_t)q * MR * a.ws_rows);
                    }
                    if (threadIdx.x == 0) a.tickets[blk] = 0;
                }
            }
            if (finish && mine_ok && mj < a.M && nrow < a.N && !dead && !*failed)
                a.out[mj * a.N + nrow] = mine + (a.bias ? __ldg(a.bias + nrow) : 0.f);
        }
    }
}

template <int MR, int V, bool EH, bool F16>
cudaError_t launch_mr(const MrMaps& maps, const MrArgs& a, unsigned grid, int smem,
                      const LaunchCtx& c) {
    const cudaError_t attr = kernel_smem_once<gemv_mr_kernel<MR, V, EH, F16>>(kMrSmem);
    if (attr != cudaSuccess) return attr;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kMrThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = c.stream;
    cudaLaunchAttribute attrs[1];
    if (c.pdl) {
        attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attrs;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, gemv_mr_kernel<MR, V, EH, F16>, maps, a);
}

template <int MR, int V>
cudaError_t launch_mr_v(bool eh, bool f16, const MrMaps& maps, const MrArgs& a, unsigned grid,
                        int smem, const LaunchCtx& c) {
    if (eh) return f16 ? launch_mr<MR, V, true, true>(maps, a, grid, smem, c)
                       : launch_mr<MR, V, true, false>(maps, a, grid, smem, c);
    return f16 ? launch_mr<MR, V, false, true>(maps, a, grid, smem, c)
               : launch_mr<MR, V, false, false>(maps, a, grid, smem, c);
}

// Parts of K per row block: split while the row blocks alone fill less than one wave of
// two CTAs per SM (at least two stages a part, within the workspace and ticket capacity).
int mr_parts(int64_t blocks, int kstages, int MR, int64_t ws_rows, const LaunchCtx& c) {
    const int64_t slots = 2LL * c.sm_count;
    int parts = 1;
    while (parts < 8 && blocks * parts * 2 <= slots && kstages / (parts * 2) >= 2 && c.ws &&
           c.tickets && blocks <= c.ticket_count &&
           (int64_t)(parts * 2) * MR * ws_rows <= c.ws_floats)
        parts *= 2;
    return parts;
}

int log2_exact_mr(int64_t v) {
    for (int s = 0; s < 31; ++s)
        if ((1LL << s) == v) return s;
    return -1;
}

}  // namespace

bool gemv_mr_eligible(const Problem& p) {
    auto al16 = [](const void* q) { return reinterpret_cast<uintptr_t>(q) % 16 == 0; };
    // The group scales arrive by TMA: a row stride of whole 16-byte units.
    if (p.M < 2 || p.M > 4 || p.K % 32 != 0 || p.K < kMrStageK || p.N < 16 ||
        (p.N * (p.scale_f16 ? 2 : 4)) % 16 != 0)
        return false;
    if (p.N > (1LL << 31) - mr_rows(4) || p.K > (1LL << 30)) return false;
    if (!al16(p.x) || !al16(p.qweight) || !al16(p.scales)) return false;
    const int64_t gs = p.group_size;
    if (gs < p.K && !(gs % 32 == 0 && log2_exact_mr(gs) >= 0)) return false;
    return tensor_map_encoder() != nullptr;
}

cudaError_t gemv_mr_launch(const Problem& p, const LaunchCtx& c) {
    EncodeTiledFn enc = tensor_map_encoder();
    const int MR = (int)p.M;  // 2, 3 or 4 rows of x per stage
    const bool one_group = p.group_size >= p.K;
    const uint32_t esz = p.scale_f16 ? 2 : 4;
    const int kstages = (int)((p.K + kMrStageK - 1) / kMrStageK);
    // 4 rows per thread, or 2 when that gives enough row blocks to need no split of K
    // while 4 would (measured: 8192 x 2048 at M = 2 / 4, 8.8 / 11.4 -> 7.2 / 9.8 us; where
    // both split, or neither, 4 is as fast or faster).
    int V = 4;
    {
        const int64_t b4 = (p.N + mr_rows(4) - 1) / mr_rows(4);
        const int64_t b2 = (p.N + mr_rows(2) - 1) / mr_rows(2);
        if (mr_parts(b4, kstages, MR, b4 * mr_rows(4), c) > 1 &&
            mr_parts(b2, kstages, MR, b2 * mr_rows(2), c) == 1)
            V = 2;
    }
    const int64_t blocks = (p.N + mr_rows(V) - 1) / mr_rows(V);

    MrArgs a = {};
    a.bias = p.bias;
    a.out = p.out;
    a.ws = c.ws;
    a.tickets = c.tickets;
    a.status = c.status_word;
    a.M = p.M;
    a.N = p.N;
    a.ws_rows = blocks * mr_rows(V);
    a.kstages = kstages;
    a.sc_rows = mr_sc_rows(V, p.scale_f16 != 0);
    a.wait_ns = c.wait_limit_ns;
    a.skip_copies = c.tc_skip_first_copy;
    // Group row of stage ks: ks * 512 / gs (gs <= 512: a shift), ks / (gs / 512), or 0.
    int gps = 1;
    a.gs_in_stage = 0;
    a.gshift = 0;
    a.stages_per_group = kstages;
    if (!one_group && p.group_size <= kMrStageK) {
        a.gs_in_stage = (int)p.group_size;
        gps = (int)(kMrStageK / p.group_size);
        a.gshift = log2_exact_mr(gps);
    } else if (!one_group) {
        a.stages_per_group = (int)(p.group_size / kMrStageK);
    }
    const int64_t G = one_group ? 1 : (p.K + p.group_size - 1) / p.group_size;
    a.stage_bytes = (uint32_t)((MR * 2048 + mr_code_bytes(V) + kMrScBytes + 1023) / 1024 * 1024);
    a.stages = std::min<int>(kMrMaxStages, (kMrSmem - 1024 - 256) / (int)a.stage_bytes);
    if (a.stages < 2) return cudaErrorNotSupported;
    a.tx = (uint32_t)MR * 2048 + mr_code_bytes(V) + (uint32_t)gps * a.sc_rows * esz;
    const int64_t slots = 2LL * c.sm_count;
    const int parts = mr_parts(blocks, kstages, MR, a.ws_rows, c);
    a.tpp = (kstages + parts - 1) / parts;
    a.parts = (kstages + a.tpp - 1) / a.tpp;
    if (blocks * a.parts > 0x7fffffff) return cudaErrorInvalidValue;
    a.items = (int)(blocks * a.parts);
    const int smem = 1024 + a.stages * (int)a.stage_bytes + 256;

    MrMaps maps;
    const cuuint32_t estr2[2] = {1, 1};
    {
        const int64_t Kp = p.K / 2;
        const cuuint64_t dims[2] = {(cuuint64_t)Kp, (cuuint64_t)p.N};
        const cuuint64_t strides[1] = {(cuuint64_t)Kp};
        const cuuint32_t box[2] = {(cuuint32_t)(kMrStageK / 2), (cuuint32_t)mr_rows(V)};
        if (enc(&maps.w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(p.qweight), dims,
                strides, box, estr2, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)p.N, (cuuint64_t)G};
        const cuuint64_t strides[1] = {(cuuint64_t)p.N * esz};
        const cuuint32_t box[2] = {(cuuint32_t)a.sc_rows, (cuuint32_t)gps};
        if (enc(&maps.s, p.scale_f16 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT32,
                2, const_cast<void*>(p.scales), dims, strides, box, estr2,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[3] = {32, (cuuint64_t)(p.K / 32), (cuuint64_t)p.M};
        const cuuint64_t strides[2] = {128, (cuuint64_t)p.K * 4};
        const cuuint32_t box[3] = {32, (cuuint32_t)(kMrStageK / 32), (cuuint32_t)MR};
        const cuuint32_t estr3[3] = {1, 1, 1};
        if (enc(&maps.x, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(p.x), dims, strides,
                box, estr3, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const unsigned grid = (unsigned)std::min<int64_t>(a.items, slots);
    const bool eh = p.even_high != 0, f16 = p.scale_f16 != 0;
    if (MR == 2) return V == 2 ? launch_mr_v<2, 2>(eh, f16, maps, a, grid, smem, c)
                               : launch_mr_v<2, 4>(eh, f16, maps, a, grid, smem, c);
    if (MR == 3) return V == 2 ? launch_mr_v<3, 2>(eh, f16, maps, a, grid, smem, c)
                               : launch_mr_v<3, 4>(eh, f16, maps, a, grid, smem, c);
    return V == 2 ? launch_mr_v<4, 2>(eh, f16, maps, a, grid, smem, c)
                  : launch_mr_v<4, 4>(eh, f16, maps, a, grid, smem, c);
}

}  // namespace q4lin
