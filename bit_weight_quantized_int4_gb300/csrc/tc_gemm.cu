// tc_gemm.cu -- tcgen05 tensor-core GEMM of the 4-bit weight-quantized linear, with the
// dequantized weights as the MMA's A operand in tensor memory (sm_103a).
//
//   out[m, n] = bias[n] + sum_k x[m, k] * (code[n, k] - 8) * scale[k / gs, n]
//
// (the formula of "[ExecuTorch][WebGPU] Add linear_qcs4w op", Solution; prefill, M > 1, is
// the regime of "Add 256-thread steel q4gsw prefill GEMM", whose 64x64 CUDA-core tile with
// a BK = 16 shared-memory slice is replaced here by the 5th-generation tensor cores; what
// is kept from that page is its dequantize-once staging of the "pwdq" variant: each packed
// word is widened once per tile and its group scale read once.)
//
// D[i, j] = sum_k A[i, k] * B[j, k] with
//   A = dequantized weight tile: 128 weight rows (the MMA's M; TMEM lane = weight row),
//       written by CUDA cores straight from registers into tensor memory (tcgen05.st), fp32
//       values read by the MMA as tf32, one 32-bit column per k;
//   B = x tile: bt activation rows (the MMA's N, 64..256), fp32 from HBM by TMA with the
//       128-byte swizzle, read as tf32 (K-major);
//   D = fp32 accumulator in tensor memory: 128 lanes (weight rows n) x bt columns (rows m).
// Keeping the dequantized weights out of shared memory leaves it the TMA writes and MMA
// reads of x plus the packed codes.  tf32 keeps 10 explicit mantissa bits of each
// operand: a product carries a relative error below 2^-9, inside the 4e-3 * sum|x*w| bar
// of the tensor-core path.
//
// A stage is 64 k (8 MMAs of K = 8).  What bounds a stage on this part is less the tensor
// core than the serial chains of single threads: a barrier wait, an expect-tx and a copy
// issue cost a producer thread ~600-700 cycles per iteration, an issuer thread's 8 MMAs and
// commit ~500.  So the stage is wide, its two x boxes come from two producer threads in
// different warps, and the packed weights arrive in blocks of four stages.
//
// Roles (640 threads, 672 with the second issuer; one CTA per [128 weight rows x bt
// activation rows] tile; tensor memory: D in columns [0, bt) (and D1 in [bt, 2 bt)), the A
// ring in [256, 256 + 64 * S)):
//   warps 0 and 2, one lane each: TMA producers of x: box j (j = 0, 1) of a stage is the
//                     tile [bt rows x 32 k] at k = 64 * stage + 32 * j (128-byte rows);
//                     with an even ring depth the producers take alternate stages (both
//                     boxes), else one box of every stage each.
//   warp 3, one lane: TMA producer of the packed weights: blocks [128 rows x 128 B]
//                     (256 k, four stages) with the 128-byte swizzle, a ring of two.
//   warps 1 (and 4):  warp 1 allocates tensor memory; one lane of each issues 8
//                     tcgen05.mma (K = 8, A from tensor memory) per stage and commits each
//                     stage's completion to "empty" (freeing the x slot and the A slot):
//                     for tiles of up to 128 activation rows (and an even ring depth) the
//                     two take alternate stages into two accumulators summed at the end,
//                     else warp 1 takes every stage.
//   then 16 warps:    four groups of 4 warps (as many as there are stages in the ring, so
//                     that a group always takes the same slot and waits on its barrier
//                     phase by phase) taking stages in turn; thread = weight row
//                     (its warp's lane quarter of tensor memory): once the MMAs that read
//                     the stage's A slot last have completed (not waiting for the stage's
//                     x, whose copy overlaps), it reads the row's 64
//                     codes of the stage (two 16-byte chunks of the swizzled block row),
//                     applies the group scales, stores the 64 values into the stage's A
//                     columns, and arrives on "a_ready".  At the end each warp reads its 32
//                     lanes of D with tcgen05.ld (the groups split the columns) and stores
//                     out: for one activation row the 32 lanes write 32 consecutive n
//                     (whole lines), with the channel scale and bias of the lane's row,
//                     predicated m < M, n < N.
//   When K % 64 == 32 the last stage has one half: its second box is not loaded, its
//   second half of A not written and its last 4 MMAs not issued.
//   Split K (few tiles): the CTAs of a cluster take disjoint K ranges of one tile; each
//                     writes the other ranks' columns of its partial tile to the workspace,
//                     and after a cluster barrier rank q adds the P partials of its column
//                     slice in rank order (deterministic; its own from tensor memory) and
//                     stores the slice.
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

// Control warps: two x producers, the MMA issuer(s), the W producer; DUAL kernels (tiles of
// up to 128 activation rows) have a second MMA issuer.
__host__ __device__ constexpr int ctl_warps(bool dual) { return dual ? 5 : 4; }
constexpr int kGroups = 4;                   // dequantizing warp groups (stages in turn)
__host__ __device__ constexpr int kernel_threads(bool dual) {
    return 32 * ctl_warps(dual) + 128 * kGroups;
}
constexpr int kWRows = 128;                  // weight rows per tile (MMA M = TMEM lanes)
constexpr int kStageK = 64;                  // k per stage: two 128-byte swizzle rows of x
constexpr int kHalfK = 32;
constexpr int kMaxStages = 4;                // A ring: 4 x 64 tensor-memory columns
static_assert(kMaxStages <= kGroups, "one dequantizing group per ring slot");
constexpr int kWBlkStages = 4;               // stages per packed-weight block (128 B a row)
constexpr int kWBlkBytes = kWRows * 128;     // 16 KiB
constexpr int kWSlots = 2;
constexpr int kScaleAhead = 2;               // stages of scales in flight per thread
constexpr int kACol0 = 256;                  // first tensor-memory column of the A ring
constexpr uint32_t kTmemCols = 512;
constexpr int64_t kDrainNs = 4000000000LL;
constexpr int kSmemLimit = 227 * 1024;

// A stage of x: two boxes [bt rows x 128 B] of fp32 (1024-byte aligned for the swizzle),
// or one box [bt rows x 128 B] of fp16 for the fp16-operand kernel.
__host__ __device__ constexpr int stage_bytes(int bt, bool h16) { return h16 ? bt * 128 : bt * 256; }
// Shared memory: alignment slack, the x ring, the weight ring, barriers (256 bytes); never
// less than 116 KiB, so that one CTA of this kernel holds an SM (it allocates all 512
// tensor-memory columns: a second one on the SM would block in tcgen05.alloc, and with
// clusters two such CTAs could wait on each other's peers).
constexpr int kOneCtaSmem = 116 * 1024;
inline int smem_bytes(int bt, int stages, bool h16) {
    return std::max(1024 + stages * stage_bytes(bt, h16) + kWSlots * kWBlkBytes + 256, kOneCtaSmem);
}

struct Tc2Args {
    const void* scales;
    const float* bias;
    float* out;
    int64_t M, N, K;
    int scale_f16, per_channel;
    int bt, stages, k_iters;
    int gs_halves, gs_shift;  // group size in 32-k halves; log2 of it or -1
    int* status;
    int64_t wait_ns;
    int skip_first_copy;
    // Split K over a cluster of `splitk` CTAs (1: no split): CTA rank r of the cluster
    // covers stages [r * kpp, (r + 1) * kpp) of the tile; rank q finishes the activation
    // rows [q * sw, (q + 1) * sw) of the tile.
    int splitk, kpp, sw;
    // Rows of the x box of the last activation tile: the rows it still holds, rounded up
    // to 8 (its own tensor map).  Rows of a box past the end of x cost the copy engine
    // nearly as much as real ones; the slot rows past them are never stored.
    int xrows_last;
    float* ws;  // split K: [tiles][P][P - 1][sw][128] partial columns exchanged through L2
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

// The 32 values (code - 8) * sc of one 16-byte chunk of packed codes, in k order.
template <bool EH>
__device__ __forceinline__ void dequant_chunk(const uint4 wv, float sc, uint32_t (&vals)[32]) {
    const float2 sc2 = make_float2(sc, sc);
    const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float2 c[4];
        codes_word<EH>(words[j], c);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float2 v = fmul2(c[t], sc2);
            vals[8 * j + 2 * t] = __float_as_uint(v.x);
            vals[8 * j + 2 * t + 1] = __float_as_uint(v.y);
        }
    }
}

// fp16 pairs (even k in the low half) of the 32 values of dequant_chunk.
template <bool EH>
__device__ __forceinline__ void dequant_chunk_h16(const uint4 wv, float sc, uint32_t* pairs) {
    uint32_t vals[32];
    dequant_chunk<EH>(wv, sc, vals);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const __half2 h = __floats2half2_rn(__uint_as_float(vals[2 * i]), __uint_as_float(vals[2 * i + 1]));
        pairs[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
}

// x fp32 -> fp16 (round to nearest even) for the fp16-operand GEMM, into the handle's
// scratch; code 2 in the status word when a finite value is outside the fp16 range
// (|x| >= 65520 rounds to infinity).  Under programmatic dependent launch the GEMM may
// start streaming its weights at once; it reads this kernel's output only after its own
// dependency wait (this grid's completion).
__global__ void __launch_bounds__(256) x_to_f16_kernel(const float4* __restrict__ x,
                                                       uint2* __restrict__ y, int64_t n4,
                                                       int* status) {
    griddep_launch_dependents();
    griddep_wait();
    bool bad = false;
    for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n4; i += (int64_t)gridDim.x * 256) {
        const float4 v = __ldg(x + i);
        bad |= (fabsf(v.x) >= 65520.f && isfinite(v.x)) || (fabsf(v.y) >= 65520.f && isfinite(v.y)) ||
               (fabsf(v.z) >= 65520.f && isfinite(v.z)) || (fabsf(v.w) >= 65520.f && isfinite(v.w));
        const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
        y[i] = make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
    }
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicCAS(status, 0, 2);
}

template <bool EH, bool DUAL, bool H16>
__global__ void __launch_bounds__(kernel_threads(DUAL), 1)
    tc_wa_kernel(const __grid_constant__ CUtensorMap tmap_x,
                 const __grid_constant__ CUtensorMap tmap_xl,
                 const __grid_constant__ CUtensorMap tmap_w, const Tc2Args a) {
    constexpr int kCtl = ctl_warps(DUAL);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const int bt = a.bt, S = a.stages;
    const uint32_t xbox = (uint32_t)bt * 128;
    const uint32_t sbytes = (uint32_t)stage_bytes(bt, H16);
    const uint32_t wring = base + (uint32_t)S * sbytes;
    const uint32_t bar_base = wring + (uint32_t)(kWSlots * kWBlkBytes);
    const uint32_t accfull = bar_base + 8 * (3 * kMaxStages + 2 * kWSlots);
    const uint32_t tmem_slot = accfull + 8;
    const int P = a.splitk;
    const int rank = P > 1 ? (int)cluster_ctarank() : 0;
    const int wtile = (int)blockIdx.x / P;
    const int it_begin = rank * a.kpp;
    const int n_iters = min(a.kpp, a.k_iters - it_begin);
    const int n_blk = (n_iters + kWBlkStages - 1) / kWBlkStages;
    // With an even ring depth the two x producers take alternate stages (both boxes each)
    // and, for tiles up to 128 activation rows, two MMA issuers take alternate stages into
    // two accumulators (D0 in columns [0, bt), D1 in [bt, 2 bt)), summed in the epilogue:
    // each slot then belongs to one producer and one issuer, which see its barrier phases
    // one by one.  A single thread's issue of 8 MMAs and its barrier work bound a stage at
    // narrow tiles.
    const bool alt = S % 2 == 0;
    const bool dual = DUAL && alt && bt <= 128 && n_iters >= 2;
    uint32_t* tmem_slot_ptr = reinterpret_cast<uint32_t*>(gbase + (tmem_slot - base));
    volatile int* failed = reinterpret_cast<volatile int*>(gbase + (tmem_slot + 4 - base));
    auto xslot = [&](int s) { return base + (uint32_t)s * sbytes; };
    auto wslot = [&](int b) { return wring + (uint32_t)(b * kWBlkBytes); };
    auto full = [&](int s) { return bar_base + 8u * s; };
    auto aready = [&](int s) { return bar_base + 8u * (kMaxStages + s); };
    auto empty = [&](int s) { return bar_base + 8u * (2 * kMaxStages + s); };
    auto wfull = [&](int b) { return bar_base + 8u * (3 * kMaxStages + b); };
    auto wempty = [&](int b) { return bar_base + 8u * (3 * kMaxStages + kWSlots + b); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), (alt || H16) ? 1 : 2);  // one producer a stage, or one a box
            mbar_init(aready(s), 128);  // the 128 threads of the group that owns the stage
            mbar_init(empty(s), 1);
        }
        for (int b = 0; b < kWSlots; ++b) {
            mbar_init(wfull(b), 1);
            mbar_init(wempty(b), 128 * kWBlkStages);  // every thread of every stage's group
        }
        mbar_init(accfull, DUAL ? 2 : 1);  // every MMA issuer commits it
        *failed = 0;
        mbar_init_fence();
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_d = *tmem_slot_ptr;
    // Programmatic dependent launch: the next grid may start launching now (its CTAs
    // become resident as this grid's leave).  Packed weights and scales do not depend on
    // the preceding grid and stream at once; x is loaded, and bias, out and the workspace
    // are touched, only after griddepcontrol.wait (x producers, epilogue threads).
    griddep_launch_dependents();

    const int64_t n0 = (int64_t)wtile * kWRows;
    const int64_t m0 = (int64_t)blockIdx.y * bt;
    bool epi_go = false;  // dequantization warps: the accumulator is complete and valid
    float row_cs = 1.f, row_b = 0.f;  // dequantization warps: channel scale, bias of row r
    if (warp == 0 || warp == 2) {
        if (lane == 0) {
            // ------------------------------------------------------ TMA producers of x
            const int pr = warp >> 1;  // producer 0 or 1
            const bool last_tile = blockIdx.y == gridDim.y - 1;
            const CUtensorMap* xmap = last_tile ? &tmap_xl : &tmap_x;
            const uint32_t xtx = (uint32_t)(last_tile ? a.xrows_last : bt) * 128;
            prefetch_tensormap(xmap);
            griddep_wait();
            // Stages of this producer: every stage (box pr) or, with alt, stages pr,
            // pr + 2, ... (both boxes).  Slot and phase kept incrementally.
            // (fp16 operands: a stage is one box; without alt producer 0 takes them all.)
            const int first = alt ? pr : 0, stride = alt ? 2 : 1;
            int s = 0;
            uint32_t ph = 0;  // parity of the slot's current use
            auto step = [&]() {
                if (++s == S) s = 0, ph ^= 1u;
            };
            for (int q = 0; q < first; ++q) step();
            int li = first;
            const int li_end = (H16 && !alt && pr == 1) ? 0 : n_iters;
            for (; li < li_end; li += stride) {
                if (li >= S && !wait_bounded(empty(s), ph ^ 1u, a.wait_ns, failed)) {
                    record_failure(a.status, failed);
                    break;
                }
                if (*failed) break;
                if (!(a.skip_first_copy && li == 0)) {
                    const int64_t k = (int64_t)(it_begin + li) * kStageK;
                    const bool two = k + kHalfK < a.K;  // else the last stage has one half
                    if (H16) {
                        // [rows x 64 k] of fp16; k past K reads as zeros.
                        mbar_arrive_expect_tx(full(s), xtx);
                        tma_load_2d(xslot(s), xmap, (int)k, (int)m0, full(s));
                    } else if (alt) {
                        mbar_arrive_expect_tx(full(s), two ? 2 * xtx : xtx);
                        tma_load_2d(xslot(s), xmap, (int)k, (int)m0, full(s));
                        if (two)
                            tma_load_2d(xslot(s) + xbox, xmap, (int)(k + kHalfK), (int)m0,
                                        full(s));
                    } else if (pr == 0 || two) {
                        mbar_arrive_expect_tx(full(s), xtx);
                        tma_load_2d(xslot(s) + (uint32_t)pr * xbox, xmap,
                                    (int)(k + kHalfK * pr), (int)m0, full(s));
                    } else {
                        mbar_arrive(full(s));  // the missing half of a last stage
                    }
                }
                for (int q = 0; q < stride; ++q) step();
            }
            // Copies of this producer's last stages may still be landing; the CTA must not
            // exit first.  (Its stages among the last S are the latest uses of their slots.)
            for (int q = li - stride; li_end > 0 && q >= first && q >= li - S; q -= stride) {
                if (a.skip_first_copy && q == 0) continue;
                wait_bounded(full(q % S), (q / S) & 1, kDrainNs, nullptr);
            }
        }
    } else if (warp == 3) {
        if (lane == 0) {
            // --------------------------------------------- TMA producer of packed weights
            prefetch_tensormap(&tmap_w);
            int bi = 0;
            for (; bi < n_blk; ++bi) {
                const int b = bi % kWSlots;
                if (bi >= kWSlots &&
                    !wait_bounded(wempty(b), ((bi / kWSlots) - 1) & 1, a.wait_ns, failed)) {
                    record_failure(a.status, failed);
                    break;
                }
                if (*failed) break;
                mbar_arrive_expect_tx(wfull(b), (uint32_t)kWBlkBytes);
                tma_load_2d(wslot(b), &tmap_w, (it_begin + bi * kWBlkStages) * (kStageK / 2),
                            (int)n0, wfull(b));
            }
            for (int q = bi > kWSlots ? bi - kWSlots : 0; q < bi; ++q)
                wait_bounded(wfull(q % kWSlots), (q / kWSlots) & 1, kDrainNs, nullptr);
        }
    } else if (warp == 1 || (DUAL && warp == 4)) {
        if (lane == 0) {
            // ------------------------------------------------------------ MMA issuers
            const int is = warp == 1 ? 0 : 1;
            const uint32_t idesc = H16 ? f16_idesc(kWRows, bt) : tf32_idesc(kWRows, bt);
            const int64_t k_two = a.K - kHalfK - (int64_t)it_begin * kStageK;
            const uint32_t dacc = tmem_d + (dual ? (uint32_t)(is * bt) : 0u);
            // Stages of this issuer: all (issuer 0, single), or is, is + 2, ... (dual).
            const int first = dual ? is : (is == 0 ? 0 : n_iters), stride = dual ? 2 : 1;
            int s = 0;
            uint32_t par = 0;
            auto step = [&]() {
                if (++s == S) s = 0, par ^= 1u;
            };
            for (int q = 0; q < first && q < S * 2; ++q) step();
            for (int it = first; it < n_iters; it += stride) {  // it: stage of this CTA's range
                if (!wait_bounded(aready(s), par, a.wait_ns, failed) ||
                    !wait_bounded(full(s), par, a.wait_ns, failed)) {
                    record_failure(a.status, failed);
                    break;
                }
                // A was written with tcgen05.st and fenced by its writers before they
                // arrived; B (x) came by TMA.  The waits order both.
                tc_fence_after();
                // Descriptors: +2 in the address field per 32 bytes (K = 8 tf32) along the
                // swizzle row, +xbox / 16 for the second box.
                const uint32_t acol = tmem_d + (uint32_t)(kACol0 + kStageK * s);
                const uint64_t d0 = sw128_desc(xslot(s));
                if (H16) {
                    // 4 MMAs of K = 16 (8 tensor-memory columns of fp16 pairs, 32 bytes along
                    // the swizzle row each).  A missing second half is zeros in both operands.
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_f16_ts(dacc, acol + 8 * kk, d0 + (uint64_t)(2 * kk), idesc,
                                   (it != first) || kk != 0);
                } else {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_tf32_ts(dacc, acol + 8 * kk, d0 + (uint64_t)(2 * kk), idesc,
                                    (it != first) || kk != 0);
                }
                if (!H16 && (int64_t)it * kStageK < k_two) {
                    const uint64_t d1 = d0 + (uint64_t)(xbox >> 4);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_tf32_ts(dacc, acol + kHalfK + 8 * kk, d1 + (uint64_t)(2 * kk), idesc,
                                    1u);
                }
                mma_commit(empty(s));
                for (int q = 0; q < stride; ++q) step();
            }
            mma_commit(accfull);  // arrives once every MMA issued above has completed
        }
        __syncwarp();
    } else {
        // ------------------------------------------------- dequantization, epilogue
        const int group = (warp - kCtl) >> 2;
        const int G = S;  // dequantizing groups (S <= kGroups): group g always takes slot g
        const int quarter = warp & 3;  // the 32-lane slice of tensor memory this warp owns
        const int r = quarter * 32 + lane;  // this thread's weight row in the tile
        const int64_t n = n0 + r;
        const bool rvalid = n < a.N;
        const uint32_t lane_base = tmem_d + ((uint32_t)(quarter * 32) << 16);
        // The row's channel scale, loaded now (its latency overlaps the loop); the bias
        // after the dependency wait below.
        const float cscale =
            (rvalid && a.per_channel) ? load_scale(a.scales, a.scale_f16, n) : 1.f;
        row_cs = cscale;
        bool ok = true;
        // Group scales (raw bits) of this row for its group's stages (both halves),
        // kScaleAhead stages ahead; the loop is unrolled by the ring size so every slot is
        // a fixed register.
        uint32_t ring[kScaleAhead][2];
        auto fetch = [&](int it, int h) {
            uint32_t bits = 0;
            if (rvalid && !a.per_channel && it < n_iters) {
                const int64_t half = (int64_t)(it_begin + it) * 2 + h;  // 32-k half of K
                if (half * kHalfK < a.K) {
                    const int64_t g = a.gs_shift >= 0 ? (half >> a.gs_shift) : half / a.gs_halves;
                    bits = load_scale_bits(a.scales, a.scale_f16, g * a.N + n);
                }
            }
            return bits;
        };
#pragma unroll
        for (int u = 0; u < kScaleAhead; ++u) {
            ring[u][0] = fetch(group + u * G, 0);
            ring[u][1] = fetch(group + u * G, 1);
        }
        const int stride = kScaleAhead * G;
        const int s = group;
        uint32_t ph = 0;  // parity of the slot's current use (this group's stage count)
        for (int it0 = group; group < G && it0 < n_iters && ok; it0 += stride) {
#pragma unroll
            for (int u = 0; u < kScaleAhead; ++u, ph ^= 1u) {
                const int it = it0 + u * G;
                if (it >= n_iters) break;
                const int bi = it / kWBlkStages, b = bi % kWSlots;
                // empty(s): the MMAs that read this A slot last have completed (the x copy
                // of the stage may still be landing: dequantization overlaps it);
                // wfull(b): the packed weights have landed.
                if ((it >= S && !wait_bounded(empty(s), ph ^ 1u, a.wait_ns, failed)) ||
                    !wait_bounded(wfull(b), (bi / kWSlots) & 1, a.wait_ns, failed)) {
                    record_failure(a.status, failed);
                    ok = false;
                    break;
                }
                tc_fence_after();
                // Chunk c of the block row sits at chunk c ^ (r % 8) (128-byte swizzle).
                const int c0 = 2 * (it % kWBlkStages);
                const uint32_t rowp = wslot(b) + (uint32_t)r * 128;
                const uint4 w0 = ld_shared_v4(rowp + ((uint32_t)(c0 ^ (r & 7)) << 4));
                const uint4 w1 = ld_shared_v4(rowp + ((uint32_t)((c0 + 1) ^ (r & 7)) << 4));
                mbar_arrive(wempty(b));
                const bool second = (int64_t)(it_begin + it) * kStageK + kHalfK < a.K;
                float sc0 = 0.f, sc1 = 0.f;
                if (rvalid) {
                    sc0 = a.per_channel ? 1.f : scale_from_bits(ring[u][0], a.scale_f16);
                    sc1 = a.per_channel ? 1.f : scale_from_bits(ring[u][1], a.scale_f16);
                }
                const uint32_t acol = lane_base + (uint32_t)(kACol0 + kStageK * s);
                uint32_t vals[32];
                if (H16) {
                    // 64 values as 32 fp16 pairs (zeros for a missing second half); a scale
                    // that would take (code - 8) * scale past the fp16 range is reported.
                    if (fabsf(sc0) > 8188.f || fabsf(sc1) > 8188.f) atomicCAS(a.status, 0, 2);
                    dequant_chunk_h16<EH>(w0, sc0, vals);
                    if (second) {
                        dequant_chunk_h16<EH>(w1, sc1, vals + 16);
                    } else {
#pragma unroll
                        for (int i = 16; i < 32; ++i) vals[i] = 0u;
                    }
                    tmem_st32_async(acol, vals);
                } else {
                    dequant_chunk<EH>(w0, sc0, vals);
                    tmem_st32_async(acol, vals);
                    if (second) {
                        dequant_chunk<EH>(w1, sc1, vals);
                        tmem_st32_async(acol + kHalfK, vals);
                    }
                }
                ring[u][0] = fetch(it + stride, 0);
                ring[u][1] = fetch(it + stride, 1);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(aready(s));
            }
        }
        const bool acc_ok = wait_bounded(accfull, 0, ok ? a.wait_ns : kDrainNs, nullptr);
        if (!acc_ok) record_failure(a.status, failed);
        griddep_wait();  // (long complete by now: the x copies waited for it)
        const float rbias = (rvalid && a.bias) ? __ldg(a.bias + n) : 0.f;
        row_b = rbias;
        tc_fence_after();
        const bool go = __all_sync(0xffffffffu, acc_ok && !*failed);
        epi_go = go;
        if (go && P == 1) {
            // Columns in chunks of 32 (one load and one wait each), the groups in turn; for
            // one activation row the 32 lanes store 32 consecutive n (whole lines).
            for (int c0 = 32 * group; c0 < bt; c0 += 32 * kGroups) {
                uint32_t v[32];
                tmem_ld32(lane_base + (uint32_t)c0, v);
                if (dual) {  // D0 + D1
                    uint32_t v1[32];
                    tmem_ld32(lane_base + (uint32_t)(bt + c0), v1);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        v[j] = __float_as_uint(__uint_as_float(v[j]) + __uint_as_float(v1[j]));
                }
                if (!rvalid) continue;
                float* dst = a.out + (m0 + c0) * a.N + n;
                const int64_t rows = a.M - (m0 + c0);
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j < rows) dst[(int64_t)j * a.N] = __uint_as_float(v[j]) * cscale + rbias;
            }
        }
    }
    if (P > 1) {
        // ------------------------------------------- split K: reduce over the cluster
        // Rank q owns the activation columns [q * sw, (q + 1) * sw) of the tile.  Every
        // CTA writes the other ranks' columns of its partial tile from tensor memory to
        // the workspace (slot j of a destination holds the partial of its j-th other rank,
        // in rank order; column-major, so the 32 lanes of a warp write 128 contiguous
        // bytes), the cluster barrier orders those writes before the reads, and each rank
        // adds the P partials of its columns in rank order (its own from tensor memory),
        // reading the peers' through L2, and stores.  (Distributed shared memory moved
        // these bytes several times slower than L2 on this part.)
        const int64_t tile_id = (int64_t)blockIdx.y * (gridDim.x / P) + wtile;
        float* wst = a.ws + tile_id * (int64_t)(P - 1) * kWRows * bt;
        if (warp >= kCtl && epi_go) {
            const int group = (warp - kCtl) >> 2;
            const int quarter = warp & 3;
            const int r = quarter * 32 + lane;
            const uint32_t lane_base = tmem_d + ((uint32_t)(quarter * 32) << 16);
            for (int c0 = 16 * group; c0 < bt; c0 += 16 * kGroups) {
                const int q = c0 / a.sw;
                if (q == rank) continue;
                uint32_t v[16];
                tmem_ld16(lane_base + (uint32_t)c0, v);
                if (dual) {  // D0 + D1
                    uint32_t v1[16];
                    tmem_ld16(lane_base + (uint32_t)(bt + c0), v1);
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        v[t] = __float_as_uint(__uint_as_float(v[t]) + __uint_as_float(v1[t]));
                }
                const int j = rank < q ? rank : rank - 1;  // this CTA's slot at rank q
                float* dst = wst + ((int64_t)(q * (P - 1) + j) * a.sw + (c0 - q * a.sw)) * kWRows + r;
#pragma unroll
                for (int t = 0; t < 16; ++t) dst[t * kWRows] = __uint_as_float(v[t]);
            }
        }
        // Every thread reaches this barrier (all earlier waits are bounded in time); its
        // release / acquire at cluster scope orders the workspace writes before the reads.
        cluster_sync_all();
        if (warp >= kCtl && __all_sync(0xffffffffu, epi_go && !*failed)) {
            const int group = (warp - kCtl) >> 2;
            const int quarter = warp & 3;
            const int r = quarter * 32 + lane;
            const int64_t n = n0 + r;
            const uint32_t lane_base = tmem_d + ((uint32_t)(quarter * 32) << 16);
            for (int c0 = 16 * group; c0 < a.sw; c0 += 16 * kGroups) {
                uint32_t own[16];
                tmem_ld16(lane_base + (uint32_t)(rank * a.sw + c0), own);
                if (dual) {  // D0 + D1
                    uint32_t own1[16];
                    tmem_ld16(lane_base + (uint32_t)(bt + rank * a.sw + c0), own1);
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        own[t] = __float_as_uint(__uint_as_float(own[t]) + __uint_as_float(own1[t]));
                }
                float acc[16];
#pragma unroll
                for (int t = 0; t < 16; ++t) acc[t] = 0.f;
                for (int q = 0; q < P; ++q) {
                    if (q == rank) {
#pragma unroll
                        for (int t = 0; t < 16; ++t) acc[t] += __uint_as_float(own[t]);
                    } else {
                        const int j = q < rank ? q : q - 1;
                        const float* src =
                            wst + ((int64_t)(rank * (P - 1) + j) * a.sw + c0) * kWRows + r;
                        float in[16];
#pragma unroll
                        for (int t = 0; t < 16; ++t) in[t] = __ldcg(src + t * kWRows);
#pragma unroll
                        for (int t = 0; t < 16; ++t) acc[t] += in[t];
                    }
                }
                // For one activation row the 32 lanes store 32 consecutive n; the row's
                // channel scale and bias (row_cs, row_b) were loaded before the main loop.
                if (n < a.N) {
                    const int64_t mb = m0 + rank * a.sw + c0;
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        if (mb + t < a.M) a.out[(mb + t) * a.N + n] = acc[t] * row_cs + row_b;
                }
            }
        }
    }
    if (warp >= kCtl) tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_d, kTmemCols);
    }
}

template <bool EH, bool DUAL, bool H16>
cudaError_t kernel_attr() {
    return kernel_smem_once<tc_wa_kernel<EH, DUAL, H16>>(kSmemLimit);
}

int stages_for_bt(int bt, bool h16, const LaunchCtx& c) {
    int stages = std::min(kMaxStages,
                          (kSmemLimit - 1024 - 256 - kWSlots * kWBlkBytes) / stage_bytes(bt, h16));
    while (stages > 2 && smem_bytes(bt, stages, h16) > c.max_smem_optin) --stages;
    return stages;
}

// How many clusters of P CTAs (tiles of bt activation rows) the device keeps resident at
// once (0 when that cannot be determined).  Cached per (device, bt, P).
int max_active_clusters(int bt, int P, const LaunchCtx& c) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_tuple(dev, bt, P);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(P * 64));
    const bool dual = bt <= 128;
    cfg.blockDim = dim3(kernel_threads(dual));
    cfg.dynamicSmemBytes = smem_bytes(bt, stages_for_bt(bt, false, c), false);
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeClusterDimension;
    at.val.clusterDim.x = (unsigned)P;
    at.val.clusterDim.y = 1;
    at.val.clusterDim.z = 1;
    cfg.attrs = &at;
    cfg.numAttrs = 1;
    int n = 0;
    cudaError_t e = cudaErrorUnknown;
    if (dual && kernel_attr<false, true, false>() == cudaSuccess)
        e = cudaOccupancyMaxActiveClusters(&n, tc_wa_kernel<false, true, false>, &cfg);
    else if (!dual && kernel_attr<false, false, false>() == cudaSuccess)
        e = cudaOccupancyMaxActiveClusters(&n, tc_wa_kernel<false, false, false>, &cfg);
    if (e != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    cache[key] = n;
    return n;
}

template <bool EH, bool DUAL, bool H16>
cudaError_t launch2(const CUtensorMap& tx, const CUtensorMap& txl, const CUtensorMap& tw,
                    const Tc2Args& a, dim3 grid, const LaunchCtx& c) {
    const cudaError_t attr = kernel_attr<EH, DUAL, H16>();
    if (attr != cudaSuccess) return attr;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kernel_threads(DUAL));
    cfg.dynamicSmemBytes = smem_bytes(a.bt, a.stages, H16);
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
    return cudaLaunchKernelEx(&cfg, tc_wa_kernel<EH, DUAL, H16>, tx, txl, tw, a);
}

// The fp16 copy of x [M, K] in the handle's scratch, before the GEMM on the same stream.
cudaError_t launch_x_to_f16(const Problem& p, uint2* y, const LaunchCtx& c) {
    const int64_t n4 = p.M * p.K / 4;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::min<int64_t>((n4 + 255) / 256, 8LL * c.sm_count));
    cfg.blockDim = dim3(256);
    cfg.stream = c.stream;
    cudaLaunchAttribute at[1];
    if (c.pdl) {
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, x_to_f16_kernel, reinterpret_cast<const float4*>(p.x), y, n4,
                              c.status_word);
}

// Floats of the scratch the fp16 copy of x takes (rounded up to 256 bytes).
int64_t x16_floats(const Problem& p) { return ((p.M * p.K * 2 + 255) / 256) * 64; }

}  // namespace

bool tc_eligible(const Problem& p, const LaunchCtx& c) {
    if (p.K % kHalfK != 0) return false;
    if (reinterpret_cast<uintptr_t>(p.x) % 16 || reinterpret_cast<uintptr_t>(p.qweight) % 16)
        return false;
    if (!(p.group_size >= p.K || p.group_size % kHalfK == 0)) return false;
    if (p.M > 65535LL * 64 || p.N > (1LL << 31) - 1) return false;
    if (c.max_smem_optin < smem_bytes(256, 2, false)) return false;
    return tensor_map_encoder() != nullptr;
}

bool tc_uses_f16(const Problem& p, const LaunchCtx& c) {
    // The fp16 copy of x may take at most half of the scratch (the rest is left to the
    // split-K exchange).
    return c.tc_f16 && c.ws && x16_floats(p) <= c.ws_floats / 2;
}

cudaError_t tc_launch(const Problem& p, const LaunchCtx& c) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const bool h16 = tc_uses_f16(p, c);
    float* const ws_split = h16 ? c.ws + x16_floats(p) : c.ws;
    const int64_t ws_split_floats = h16 ? c.ws_floats - x16_floats(p) : c.ws_floats;
    // Activation rows per tile (the MMA's N) and the split of K over a cluster.  Wider
    // tiles make wider MMAs; narrower ones give more CTAs.  When the tiles alone leave SMs
    // idle, K is split over a cluster of P CTAs (a power of two up to 8, at least 4 stages
    // each, 16-column slices, only if all the clusters stay resident at once).  Estimate:
    // waves x stages per CTA x cycles per stage, plus the split-K exchange (~30 cycles per
    // exchanged column of the 128-row partial tile: bt * (P - 1) / P of them); a 64-k
    // stage costs the larger of the tf32 MMAs (~4.2 * bt cycles) and the serial chains of
    // the producer and issuer threads (~700 cycles); ties go to the narrower tile.  (Fitted
    // to a sweep of forced tile heights over M = 64..2048.)
    const int64_t wtiles = (p.N + kWRows - 1) / kWRows;
    const int k_iters = (int)((p.K + kStageK - 1) / kStageK);
    int bt = 256, splitk = 1;
    int64_t best = -1;
    for (int cand = 256; cand >= 64; cand /= 2) {
        const int64_t mt = (p.M + cand - 1) / cand;
        if (mt > 65535) continue;
        const int64_t tiles = wtiles * mt;
        int P = 1;
        while (P < 8 && tiles * P * 2 <= c.sm_count && k_iters % (2 * P) == 0 &&
               k_iters / (2 * P) >= 4 && cand / (2 * P) >= 16 && !c.tc_skip_first_copy &&
               max_active_clusters(cand, 2 * P, c) >= tiles)
            P *= 2;
        const int64_t ctas = tiles * P;
        const int64_t waves = (ctas + c.sm_count - 1) / c.sm_count;
        const int64_t per_stage = std::max<int64_t>(700, (int64_t)(4.2 * cand));
        const int64_t cost =
            waves * (k_iters / P) * per_stage + (P > 1 ? 30LL * cand * (P - 1) / P : 0);
        if (best < 0 || cost <= best) {
            best = cost;
            bt = cand;
            splitk = P;
        }
    }
    const int stages = stages_for_bt(bt, h16, c);
    const int64_t mtiles = (p.M + bt - 1) / bt;
    // The split-K exchange ([tiles][P - 1][128][bt] floats) must fit in the workspace.
    while (splitk > 1 &&
           (!c.ws || wtiles * mtiles * (splitk - 1) * kWRows * bt > ws_split_floats))
        splitk /= 2;

    Tc2Args a;
    a.scales = p.scales;
    a.bias = p.bias;
    a.out = p.out;
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.scale_f16 = p.scale_f16;
    a.per_channel = p.group_size >= p.K;
    a.bt = bt;
    a.stages = stages;
    a.k_iters = k_iters;
    a.splitk = splitk;
    a.kpp = k_iters / splitk;
    a.sw = bt / splitk;
    a.ws = ws_split;
    a.gs_halves = a.per_channel ? 1 : (int)(p.group_size / kHalfK);
    a.gs_shift = -1;
    for (int sft = 0; sft < 31; ++sft)
        if ((1 << sft) == a.gs_halves) a.gs_shift = sft;
    a.status = c.status_word;
    a.wait_ns = c.wait_limit_ns;
    a.skip_first_copy = c.tc_skip_first_copy;

    a.xrows_last = (int)std::min<int64_t>(bt, (p.M - (mtiles - 1) * bt + 7) / 8 * 8);

    CUtensorMap tx, txl, tw;
    for (int last = 0; last < 2; ++last) {
        // x [M, K]: fp32 boxes [rows x 32 k], or fp16 boxes [rows x 64 k] of the copy in the
        // scratch; 128-byte rows either way.
        const cuuint64_t dims[2] = {(cuuint64_t)p.K, (cuuint64_t)p.M};
        const cuuint64_t strides[1] = {(cuuint64_t)p.K * (h16 ? 2 : 4)};
        const cuuint32_t box[2] = {(cuuint32_t)(h16 ? kStageK : kHalfK),
                                   (cuuint32_t)(last ? a.xrows_last : bt)};
        const cuuint32_t estr[2] = {1, 1};
        void* src = h16 ? static_cast<void*>(c.ws) : const_cast<float*>(p.x);
        if (enc(last ? &txl : &tx,
                h16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, src,
                dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        // Blocks of packed weights [128 rows x 128 B] (four stages), 128-byte swizzle.
        const int64_t Kp = p.K / 2;
        const cuuint64_t dims[2] = {(cuuint64_t)Kp, (cuuint64_t)p.N};
        const cuuint64_t strides[1] = {(cuuint64_t)Kp};
        const cuuint32_t box[2] = {(cuuint32_t)(kWBlkStages * kStageK / 2), (cuuint32_t)kWRows};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(p.qweight), dims,
                strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const dim3 grid((unsigned)(wtiles * splitk), (unsigned)mtiles);
    if (h16) {
        const cudaError_t e = launch_x_to_f16(p, reinterpret_cast<uint2*>(c.ws), c);
        if (e != cudaSuccess) return e;
        if (bt <= 128)
            return p.even_high ? launch2<true, true, true>(tx, txl, tw, a, grid, c)
                               : launch2<false, true, true>(tx, txl, tw, a, grid, c);
        return p.even_high ? launch2<true, false, true>(tx, txl, tw, a, grid, c)
                           : launch2<false, false, true>(tx, txl, tw, a, grid, c);
    }
    if (bt <= 128)
        return p.even_high ? launch2<true, true, false>(tx, txl, tw, a, grid, c)
                           : launch2<false, true, false>(tx, txl, tw, a, grid, c);
    return p.even_high ? launch2<true, false, false>(tx, txl, tw, a, grid, c)
                       : launch2<false, false, false>(tx, txl, tw, a, grid, c);
}

}  // namespace q4lin
