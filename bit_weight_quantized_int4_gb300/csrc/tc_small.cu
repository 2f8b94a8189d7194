// tc_small.cu -- tcgen05 tensor-core GEMM of the 4-bit weight-quantized linear for a few
// activation rows (2 <= M <= 32: batched or speculative decode), streaming the weights once.
//
//   out[m, n] = bias[n] + sum_k x[m, k] * (code[n, k] - 8) * scale[k / gs, n]
//
// (the formula of "[ExecuTorch][WebGPU] Add linear_qcs4w op", Solution.)
//
// D[n, m] = sum_k A[n, k] * B[m, k] per block of 128 weight rows, with
//   A = the block's dequantized weights (c - 8) * scale as fp32, written by CUDA cores into
//       tensor memory (lane = weight row, one column per k) and read by the MMA as tf32;
//   B = x, fp32 chunks of 32 k with the 128-byte swizzle, 8 rows a chunk when M <= 8, 16
//       up to 16 rows and 32 above (rows past M are zeros from the copy's out-of-bounds
//       fill; with 8-row chunks the MMA's rows 8-15 read the next chunk, which only D
//       columns m >= M see), read as tf32;
//   D = fp32 accumulators in tensor memory (128 lanes x BT columns: the MMA width BT is 16
//       up to 16 rows and 32 above).
// tf32 keeps 10 explicit mantissa bits of each operand: a product carries a relative error
// below 2^-9, inside the 4e-3 * sum|x*w| bar of the tensor-core path.
//
// bf16 operands (up to 8 rows, x resident, K > 256; by default from 100 row blocks, where
// they measured 2-5 % faster): A = (c - 8) * s rounded to bf16, two values per tensor-
// memory column, so that an A slot of 64 columns holds 128 k and an MMA (kind::f16, bf16 A
// and B) takes 16 k; B = x as 64-k chunks of 16 rows, rows 0-7 bf16(x) and rows 8-15 the
// remainder bf16(x - bf16(x)), converted by the dequantizing warps into shared memory at
// the start; the epilogue adds D columns m and m + 8.  A product then carries a relative
// error below 2^-9 + 2^-16 (the weight's rounding; x keeps 16 bits), and bf16 has fp32's
// exponent range, so no input range is excluded.
//
// At 16 columns an MMA is cheap for the tensor core but not for the thread that issues it:
// on GB300 one thread issues a tcgen05.mma of 128 x 16 x 8 about every 50-70 cycles
// whatever its width, and issuers in different warps add up.  So four issuer threads take
// the 64-k slots of A in turn (8 MMAs each), each into its own accumulator (summed in a
// fixed order at the end of the block), and four teams of four warps dequantize into a ring
// of six slots of tensor memory ahead of the MMAs.  (Measured on 128256 x 2048: 32-k slots
// in a ring of twelve 74 us, three teams 64.8 us, this layout 57 us; the loops advance their
// ring indices without divisions, and the roles off the issuers' path sleep between polls
// of their barriers, which together took 93.7 to 85 us.)
//
// Roles (800 threads, 832 with streamed x; one CTA per SM, persistent over the row blocks
// blockIdx.x + k grid):
//   warp 0, one lane:  TMA producer of the weights.  Per 256-k stage of a block: the codes
//                      [128 rows x 128 B] (128-byte swizzle) and the block's group scales
//                      [groups of the stage x 128 rows], into a ring of up to seven stages
//                      (what shared memory leaves next to x).  A stage is released once the
//                      dequantizing warps have read it.  The weights do not depend on the
//                      preceding kernel: no dependency wait.
//   warp 24, one lane: the fourth MMA issuer; when x fits next to three weight stages (K
//                      <= 5120 as 8-row chunks when M <= 8, K <= 2560 as 16-row chunks,
//                      K <= 1280 as 32-row chunks) it
//                      first copies the whole x after griddepcontrol.wait, resident for all
//                      the CTA's blocks, one 3D box of 8 chunks [rows x 32 k] per 256-k group
//                      on its own barrier (with bf16 operands the dequantizing warps convert
//                      x instead, and this thread only issues MMAs).
//   warp 25, one lane: (longer K only) streams x instead, one 256-k group per stage of the
//                      CTA's sequence through a ring of three, released by the MMAs'
//                      commits: ~5 % slower than resident x (28672 x 4096 at 12 rows 34.1 us
//                      against 33.0 resident at 8).
//   warps 1-3, lane 0: MMA issuers; slot i of the CTA's sequence goes to issuer i % 4:
//                      eight tcgen05.mma.kind::tf32 of K = 8, or kind::f16 of K = 16 with
//                      bf16 operands (A from tensor memory), then a
//                      commit that frees the A slot; after its last slot of a block, a commit
//                      to the block's "D full".  Warp 1 also allocates and frees the 512
//                      tensor-memory columns.
//   warps 4-7:         epilogue; warp w owns tensor-memory lanes 32 (w % 4) ...: adds the
//                      four accumulators of its rows, applies the channel scale and bias and
//                      stores out[m, n] for m < M, n < N (32 consecutive n per row m).
//   warps 8-23:        four dequantizing teams of four warps (one per lane quarter); team
//                      i % 4 writes slot i: each thread (one weight row) reads the row's two
//                      16-byte chunks of 32 codes and their group scales, and stores 64 fp32
//                      values with two tcgen05.st.  Per code: a byte permute puts it into the
//                      mantissa of a float v (v = 0.5 + c/256 for a low nibble, 1 + c/2048
//                      for a high one), and one packed FMA per pair gives the exactly
//                      rounded (c - 8) * s (256 s v - 136 s, 2048 s v - 2056 s; exact
//                      constants for fp16 and dyadic scales, within 2^-12 s otherwise, far
//                      below the tf32 rounding).  Per-channel scales are applied in the
//                      epilogue instead (A = c - 8 exactly).
//   Each CTA walks K from its own starting stage (blockIdx.x % stages, wrapping).
// K split (matrices with fewer 128-row blocks than half the SMs): each block is 2, 4 or 8
// work items over consecutive runs of its 256-k stages, one item per CTA; the epilogue
// writes an item's partial tile [columns x 128 rows] to the split-K workspace, takes the
// block's ticket, and the last item of the block adds the parts in part order (the sum
// does not depend on which CTA finishes last), applies the channel scale and bias, stores
// and resets the ticket.  After a timed-out wait the epilogue still walks every item so
// that every ticket is counted and reset.
// Tensor memory: accumulators [0, 8 BT) (two blocks in flight x four issuers x BT columns),
// the A ring [8 BT, 512) (six slots of 64 columns at BT = 16, four at BT = 32).  Slot i of
// the sequence takes ring position i % slots on lap i / slots, team i % 4 and issuer i % 4;
// with six positions a position's laps alternate between two teams (and two issuers), so
// each position has separate barriers for its even and its odd laps: every barrier is then
// waited on by one role, phase after phase (a parity wait that ran two phases ahead of its
// barrier would take the phase before the current one for the awaited one).  Every wait is bounded in time; a
// timeout records code 1 in the status word, each role stops, the issuers drain their
// MMAs, and the CTA frees its tensor memory and returns without storing.
#include <algorithm>

#include "ptx.cuh"
#include "q4lin_internal.h"

namespace q4lin {
namespace {
using namespace ptx;

constexpr int kRows = 128;                        // weight rows per block (MMA M)
constexpr int kBt = 32;                           // most activation rows (MMA N = 16 or 32)
constexpr int kStageK = 256;                      // k per stage (weights and x alike)
constexpr int kChunk = 32;                        // k per 16-byte chunk of a code row
constexpr int kChunksPerStage = kStageK / kChunk; // 8
constexpr int kSlotK = 64;                        // k per A slot: two chunks, 8 MMAs
constexpr int kSlotsPerStage = kStageK / kSlotK;  // 4
constexpr int kIssuers = 4;                       // warps 1-3 and the x producer's warp
constexpr int kTeams = 4;
// Tensor memory for MMA width BT: two blocks' accumulators (2 x issuers x BT columns), then
// the A ring of 64-k slots: six slots at BT = 16, four at BT = 32.
__host__ __device__ constexpr int acol0(int bt) { return 2 * kIssuers * bt; }
__host__ __device__ constexpr int aslots(int bt) { return (512 - acol0(bt)) / kSlotK; }
constexpr int kMaxASlots = aslots(16);
static_assert(aslots(32) >= kIssuers && aslots(32) >= kTeams && kSlotsPerStage >= kIssuers,
              "ring positions advance by less than a lap; every issuer has a slot per stage");
constexpr int kWBox = kRows * 128;                // codes of a stage: [128 rows x 128 B]
constexpr int kSMax = 8 * kRows * 4;              // scales: up to 8 groups x 128 rows
constexpr int kWStageBytes = kWBox + kSMax;       // 20 KiB
constexpr int kMaxWStages = 7;                    // weight ring: up to 140 KiB in flight
constexpr int kMinWStages = 3;
constexpr int kMaxXGroups = 20;                   // x resident: K <= 5120 (20 x 256 k)
constexpr int kXStages = 3;                       // x streamed: a ring of 256-k groups
constexpr int kWarps = 8 + 4 * kTeams + 2;
constexpr int kThreads = 32 * kWarps;
constexpr int kDeqWarp0 = 8;
constexpr int kIss3Warp = 8 + 4 * kTeams;          // the fourth MMA issuer (resident x: its loader)
constexpr int kXWarp = kIss3Warp + 1;              // the x producer of streamed x (launched only then)
constexpr int kBarBytes = 1024;
constexpr int kSmemCap = 227 * 1024;              // opt-in shared memory of a CTA
constexpr int64_t kDrainNs = 4000000000LL;
// bf16 operands (up to 8 rows): an A slot holds 128 k as 64 columns of bf16 pairs, two
// slots a stage; x is kept as 64-k chunks [16 rows x 128 B]: rows 0-7 the bf16 values
// x_hi = bf16(x), rows 8-15 the remainders x_lo = bf16(x - x_hi).
constexpr int kSlotKH = 128;
constexpr int kSlotsPerStageH = kStageK / kSlotKH;  // 2
constexpr int kChunkXH = 64;                        // k per x chunk (128 B of bf16)
constexpr int kXChunkBytesH = 16 * 128;
static_assert(kSlotKH / 2 == kSlotK, "a bf16 slot takes the columns of a tf32 slot");
static_assert(kStageK / kChunkXH * kXChunkBytesH == kChunksPerStage * 8 * 128,
              "a stage of bf16 x takes the bytes of a stage of 8-row fp32 x");

struct TsArgs {
    const float* x;       // bf16 operands: converted by the dequantizing warps
    int K;
    const void* scales;   // per channel: [N], read by the epilogue
    const float* bias;
    float* out;
    int M, N;
    int nst;              // stages per block: ceil(K / 256)
    int blocks;           // row blocks: ceil(N / 128)
    int gs_shift;         // log2(group_size / 32) (grouped scales)
    uint32_t w_tx;        // bytes of one stage's codes and scales
    int wst;              // stages of the weight ring
    int xrows;            // rows of x per chunk in shared memory: 8, 16 or 32 (by M)
    uint32_t x_bytes;     // x region: 8 chunks x xrows x 128 B per 256-k group, + 1 KiB
    int x_ring;           // 0: all of x resident; 1: streamed through a ring of kXStages
    int skip_first_copy;  // test hook: stage 0's codes are not requested
    // K split: each 128-row block is `parts` work items of nst / parts stages; CTA c takes
    // part c % parts of blocks c / parts, c / parts + grid / parts, ... (the grid is a
    // multiple of parts).  With parts > 1 the items leave their partial tiles in ws and
    // the last item of a block (ticket count) adds them in part order.
    int parts;
    float* ws;            // [blocks][parts][columns][128] partial tiles (parts > 1)
    int* tickets;         // [blocks], zero between launches (the last item resets its own)
    int* status;
    int64_t wait_ns;
};

// A bounded wait for the roles that are not on the MMA issuers' path (dequantizing warps,
// which run ahead, the epilogue, the producers): between polls the warp sleeps, so that
// the schedulers' issue slots go to the issuer threads instead of to polling.
static __device__ __noinline__ bool wait_backoff(uint32_t bar, uint32_t parity, int64_t limit_ns,
                                          const volatile int* failed, unsigned sleep_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer();
    while (true) {
        __nanosleep(sleep_ns);
        if (mbar_try_wait(bar, parity)) return true;
        if (failed && *failed) return false;
        if ((int64_t)(global_timer() - t0) > limit_ns) return false;
    }
}

__device__ __forceinline__ float ld_scale(const void* scales, bool f16, int64_t i) {
    if (f16) return __half2float(__ldg(reinterpret_cast<const __half*>(scales) + i));
    return __ldg(reinterpret_cast<const float*>(scales) + i);
}

// 32 fp32 values (c - 8) * s of one row's 16-byte chunk (k order) as raw bits.  Byte b of
// word q holds k = 8q + 2b in its low nibble and 8q + 2b + 1 in its high nibble (swapped
// when EH).  The permutes build v = 0.5 + c/256 (low nibble into byte 2 under 0x3F..) and
// v = 1 + c/2048 (high nibble, already << 4, into byte 1 under 0x3F80..); the FMA with the
// exact products 256 s, 2048 s and the offsets -136 s, -2056 s rounds (c - 8) s once.
template <bool EH>
__device__ __forceinline__ void dequant_chunk(const uint4 w4, float s, uint32_t (&v)[32]) {
    const float2 mul = EH ? make_float2(2048.f * s, 256.f * s) : make_float2(256.f * s, 2048.f * s);
    const float2 add = EH ? make_float2(-2056.f * s, -136.f * s) : make_float2(-136.f * s, -2056.f * s);
    const uint32_t words[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t lo = words[q] & 0x0F0F0F0Fu, hi = words[q] & 0xF0F0F0F0u;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const float vl = __uint_as_float(prmt(lo, 0x3F800000u, 0x7054u | (b << 8)));
            const float vh = __uint_as_float(prmt(hi, 0x3F800000u, 0x7604u | (b << 4)));
            const float2 r = ffma2(EH ? make_float2(vh, vl) : make_float2(vl, vh), mul, add);
            v[8 * q + 2 * b] = __float_as_uint(r.x);
            v[8 * q + 2 * b + 1] = __float_as_uint(r.y);
        }
    }
}

// Two fp32 values as a bf16 pair (round to nearest even), a in the low half.
__device__ __forceinline__ uint32_t bf16x2(float a, float b) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(b), "f"(a));
    return d;
}
// Instruction descriptor of kind::f16 with bf16 A and B (format 1), D fp32, both K-major.
__device__ __forceinline__ uint32_t bf16_idesc(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}
// Orders this thread's shared-memory stores before later reads by the tensor core.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// bf16 operands: x [M x K] into 64-k chunks [16 rows x 128 B] with the 128-byte swizzle
// (16-byte unit u of row r at unit u ^ (r % 8)): row m < 8 holds bf16(x), row m + 8 the
// remainder bf16(x - bf16(x)); rows past M and k past K are zeros.  Thread t of nthr
// takes units t, t + nthr, ... (8 k of one row each).
__device__ __forceinline__ void convert_x_bf16(const TsArgs& a, uint32_t xbase, int t, int nthr) {
    const int units = a.nst * (kStageK / kChunkXH) * 64;
    for (int e = t; e < units; e += nthr) {
        const int c = e >> 6, m = (e >> 3) & 7, u = e & 7;
        const int k0 = c * kChunkXH + u * 8;
        float v[8];
        if (m < a.M && k0 < a.K) {
            const float4* src = reinterpret_cast<const float4*>(a.x + (int64_t)m * a.K + k0);
            const float4 p = src[0], q = src[1];
            v[0] = p.x, v[1] = p.y, v[2] = p.z, v[3] = p.w, v[4] = q.x, v[5] = q.y, v[6] = q.z, v[7] = q.w;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = 0.f;
        }
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            hi[i] = bf16x2(v[2 * i], v[2 * i + 1]);
            // bf16 -> fp32 is exact (the top 16 bits); the remainders are exact in fp32.
            const float h0 = __uint_as_float(hi[i] << 16), h1 = __uint_as_float(hi[i] & 0xFFFF0000u);
            lo[i] = bf16x2(v[2 * i] - h0, v[2 * i + 1] - h1);
        }
        const uint32_t row = xbase + (uint32_t)(c * kXChunkBytesH) + ((uint32_t)(u ^ m) << 4);
        st_shared_v4(row + (uint32_t)(m * 128), hi[0], hi[1], hi[2], hi[3]);
        st_shared_v4(row + (uint32_t)((m + 8) * 128), lo[0], lo[1], lo[2], lo[3]);
    }
}

template <bool EH, bool PC, bool F16, bool XR, int BT, bool BF, bool KS>
__global__ void __launch_bounds__(XR ? kThreads : kThreads - 32, 1)
    tc_small_kernel(const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tms,
                    const __grid_constant__ CUtensorMap tmx, const TsArgs a) {
    constexpr int kAC0 = acol0(BT), kAS = aslots(BT);
    static_assert(!BF || (!XR && BT == 16), "bf16 operands: resident x, up to 8 rows");
    constexpr int SPS = BF ? kSlotsPerStageH : kSlotsPerStage;  // A slots per stage
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    // [x, resident: 256-k groups of 8 chunks [xrows x 128 B], + 1 KiB][weight ring][barriers]
    const uint32_t xbase = base;
    const uint32_t wbase = base + a.x_bytes;
    const uint32_t bar0 = wbase + (uint32_t)(a.wst * kWStageBytes);
    auto wstage = [&](int b) { return wbase + (uint32_t)(b * kWStageBytes); };
    constexpr int kB0 = 0, kB1 = kB0 + 2 * kMaxWStages, kBx = kB1 + kMaxXGroups,
                  kB2 = kBx + kXStages, kB3 = kB2 + 4 * kMaxASlots, kB4 = kB3 + 4;
    auto wfull = [&](int b) { return bar0 + 8u * (kB0 + b); };
    auto wempty = [&](int b) { return bar0 + 8u * (kB0 + kMaxWStages + b); };
    auto xfull = [&](int grp) { return bar0 + 8u * (kB1 + grp); };   // group, or ring slot
    auto xempty = [&](int b) { return bar0 + 8u * (kBx + b); };       // ring slot (streamed x)
    // A ring position p has one barrier pair for its even laps and one for its odd laps.
    // The slots go round the positions and the roles (issuers, teams) in turn, six
    // positions over four roles, so a position's laps alternate between two roles: each
    // barrier then has one role waiting on it, which takes its phases in order (a parity
    // wait must never run two phases ahead of its barrier: it would read the phase before
    // the current one as complete).
    auto afull = [&](int p, int lap) { return bar0 + 8u * (kB2 + 2 * p + (lap & 1)); };
    auto aempty = [&](int p, int lap) { return bar0 + 8u * (kB2 + 2 * kMaxASlots + 2 * p + (lap & 1)); };
    auto dfull = [&](int q) { return bar0 + 8u * (kB3 + q); };
    auto dempty = [&](int q) { return bar0 + 8u * (kB3 + 2 + q); };
    auto drain = [&](int u) { return bar0 + 8u * (kB4 + u); };
    static_assert(8 * (kB4 + kIssuers) <= 960, "barriers fit below the flags");
    volatile int* failed = reinterpret_cast<volatile int*>(gbase + (bar0 - base) + 960);
    const uint32_t tslot = bar0 + 968;
    volatile int* s_ticket = reinterpret_cast<volatile int*>(gbase + (bar0 - base) + 976);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int b = 0; b < a.wst; ++b) {
            mbar_init(wfull(b), 1);
            mbar_init(wempty(b), SPS * 4);  // the 4 dequantizing warps of each slot
        }
        // bf16 operands: xfull(0) completes once the 16 dequantizing warps converted x.
        for (int grp = 0; grp < (XR ? kXStages : a.nst); ++grp) mbar_init(xfull(grp), BF ? 16 : 1);
        for (int b = 0; b < kXStages; ++b) mbar_init(xempty(b), kSlotsPerStage);  // MMA commits
        for (int p = 0; p < kAS; ++p)
            for (int e = 0; e < 2; ++e) {
                mbar_init(afull(p, e), 4);
                mbar_init(aempty(p, e), 1);
            }
        for (int q = 0; q < 2; ++q) {
            mbar_init(dfull(q), kIssuers);
            mbar_init(dempty(q), 4);
        }
        for (int u = 0; u < kIssuers; ++u) mbar_init(drain(u), 1);
        *failed = 0;
        mbar_init_fence();
    }
    if (warp == 1) tmem_alloc(tslot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    uint32_t tmem;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(tmem) : "r"(tslot) : "memory");
    griddep_launch_dependents();

    // This CTA's work items: blockIdx.x, + gridDim.x, ... (item = block * parts + part, the
    // part the same for all of them); their stages and A slots in order.
    // (KS: K split instances; the others compile with one part.)
    const int parts = KS ? a.parts : 1, tpp = KS ? a.nst / parts : a.nst;
    const int my_part = KS ? (int)blockIdx.x % parts : 0;
    const int items = a.blocks * parts;
    const int my_blocks = (items - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
    auto blk_of = [&](int j) { return ((int)blockIdx.x + j * (int)gridDim.x) / parts; };
    const int n_stages = my_blocks * tpp;
    const int n_slots = n_stages * SPS;
    const int slots_per_block = tpp * SPS;
    // Each CTA walks K from its own starting stage (blockIdx.x % stages, wrapping), so
    // that the CTAs' concurrent weight requests spread over the column offsets of the
    // rows instead of all asking for the same 128 bytes of every row at once.
    const int rot = (int)((blockIdx.x / (unsigned)parts) % (unsigned)tpp);
    auto kstage = [&](int t) { return my_part * tpp + (t + rot < tpp ? t + rot : t + rot - tpp); };

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------- TMA producer of codes and scales
            // (independent of the preceding kernel: no dependency wait)
            prefetch_tensormap(&tmw);
            if (!PC) prefetch_tensormap(&tms);
            int g = 0;
            for (; g < n_stages; ++g) {
                const int b = g % a.wst, t = kstage(g % tpp);
                const int row0 = blk_of(g / tpp) * kRows;
                if (g >= a.wst &&
                    !wait_backoff(wempty(b), ((g / a.wst) - 1) & 1, a.wait_ns, failed, 64)) {
                    record_failure(a.status, failed);
                    break;
                }
                if (*failed) break;
                mbar_arrive_expect_tx(wfull(b), a.w_tx);
                if (a.skip_first_copy && g == 0) continue;
                tma_load_2d(wstage(b), &tmw, t * (kStageK / 2), row0, wfull(b));
                if (!PC)
                    tma_load_2d(wstage(b) + kWBox, &tms, row0, (t * kStageK) >> (a.gs_shift + 5),
                                wfull(b));
            }
            // The last requested stages may still be landing; the CTA must not exit first.
            for (int q = g > a.wst ? g - a.wst : 0; q < g; ++q) {
                if (a.skip_first_copy && q == 0) continue;
                wait_bounded(wfull(q % a.wst), (q / a.wst) & 1, kDrainNs, nullptr);
            }
        }
    } else if (warp == kXWarp) {
        if (lane == 0) {
            // ------------------------------------------------- TMA producer of streamed x
            // One 256-k group per stage of the CTA's sequence through a ring of kXStages,
            // released by the MMAs' commits (this warp is launched only in that mode).
            prefetch_tensormap(&tmx);
            griddep_wait();  // x belongs to the dependency chain
            const uint32_t gbytes = (uint32_t)(kChunksPerStage * a.xrows * 128);
            int g = 0;
            for (; g < n_stages; ++g) {
                const int b = g % kXStages;
                if (g >= kXStages && !wait_backoff(xempty(b), ((g / kXStages) - 1) & 1,
                                                   a.wait_ns, failed, 64)) {
                    record_failure(a.status, failed);
                    break;
                }
                if (*failed) break;
                mbar_arrive_expect_tx(xfull(b), gbytes);
                tma_load_3d(xbase + (uint32_t)b * gbytes, &tmx, 0, 0,
                            kstage(g % tpp) * kChunksPerStage, xfull(b));
            }
            for (int q = g > kXStages ? g - kXStages : 0; q < g; ++q)
                wait_bounded(xfull(q % kXStages), (q / kXStages) & 1, kDrainNs, nullptr);
        }
    } else if (warp <= 3 || warp == kIss3Warp) {
        if (lane == 0) {
            const int u = warp == kIss3Warp ? 3 : warp - 1;
            if (warp == kIss3Warp && !XR && !BF) {
                // --------------------------------------------------- TMA loads of resident x
                // All of x, read from L2 once per CTA (every CTA reads the same lines;
                // re-reading them per block made those L2 lines the bottleneck), in 256-k
                // groups on their own barriers, in the order of first use; then this thread
                // is the fourth MMA issuer.
                prefetch_tensormap(&tmx);
                griddep_wait();  // x belongs to the dependency chain
                const uint32_t gbytes = (uint32_t)(kChunksPerStage * a.xrows * 128);
                for (int q = 0; q < tpp; ++q) {  // the groups of this CTA's part
                    const int grp = kstage(q);
                    mbar_arrive_expect_tx(xfull(grp), gbytes);
                    tma_load_3d(xbase + (uint32_t)grp * gbytes, &tmx, 0, 0,
                                grp * kChunksPerStage, xfull(grp));
                }
            }
            // ------------------------------------------------------------- MMA issuers
            const uint32_t idesc = BF ? bf16_idesc(kRows, BT) : tf32_idesc(kRows, BT);
            // Slots u, u + kIssuers, ...: the block j, the slot's place in the block, its A ring
            // slot p and its lap there advance without divisions.
            int j = 0, in_blk = u, p = u, lap = 0;
            // Streamed x: the ring slot xb and phase xph of the current stage (an issuer
            // takes one slot of every stage, so they advance by one stage a slot).
            static_assert(kSlotsPerStage == kIssuers, "one slot of every stage per issuer");
            int xb = 0;
            uint32_t xph = 0;
            for (int i = u; i < n_slots; i += kIssuers) {
                while (in_blk >= slots_per_block) in_blk -= slots_per_block, ++j;
                const int par = j & 1;
                const int t = in_blk / SPS, sl = in_blk % SPS;
                const bool first = in_blk < kIssuers;
                const bool last = in_blk + kIssuers >= slots_per_block;
                if ((first && j >= 2 &&
                     !wait_bounded(dempty(par), ((j >> 1) - 1) & 1, a.wait_ns, failed)) ||
                    !wait_bounded(afull(p, lap), (lap >> 1) & 1, a.wait_ns, failed) ||
                    (!XR && !BF && j == 0 && !wait_bounded(xfull(kstage(t)), 0, a.wait_ns, failed)) ||
                    (BF && j == 0 && in_blk < kIssuers && !wait_bounded(xfull(0), 0, a.wait_ns, failed)) ||
                    (XR && !wait_bounded(xfull(xb), xph, a.wait_ns, failed))) {
                    record_failure(a.status, failed);
                    break;
                }
                // A was written by tcgen05.st and fenced by its writers before they arrived;
                // x came by TMA.  The waits order both.
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)((par * kIssuers + u) * BT);
                const uint32_t acol = tmem + (uint32_t)(kAC0 + p * kSlotK);
                // The slot's two x chunks in the resident copy (with 8 rows a chunk, rows 8-15
                // of the MMA's B read the next chunk: only D columns m >= 8 >= M see them); +2
                // in the descriptor's address field per 32 bytes (K = 8 tf32) along a row.
                if (BF) {
                    // bf16: the slot's two 64-k chunks of x [16 rows x 128 B]; an MMA takes
                    // 16 k (8 columns of A, 32 bytes of a row of x).
                    const int chunk = kstage(t) * (kStageK / kChunkXH) + sl * (kSlotKH / kChunkXH);
#pragma unroll
                    for (int h = 0; h < kSlotKH / kChunkXH; ++h) {
                        const uint64_t bd = sw128_desc(xbase + (uint32_t)((chunk + h) * kXChunkBytesH));
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_f16_ts(d, acol + 32 * h + 8 * kk, bd + (uint64_t)(2 * kk), idesc,
                                       (first && h == 0 && kk == 0) ? 0u : 1u);
                    }
                } else {
                    const int chunk = (XR ? xb : kstage(t)) * kChunksPerStage + sl * (kSlotK / kChunk);
#pragma unroll
                    for (int h = 0; h < kSlotK / kChunk; ++h) {
                        const uint64_t bd =
                            sw128_desc(xbase + (uint32_t)((chunk + h) * a.xrows * 128));
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_tf32_ts(d, acol + kChunk * h + 8 * kk, bd + (uint64_t)(2 * kk), idesc,
                                        (first && h == 0 && kk == 0) ? 0u : 1u);
                    }
                }
                mma_commit(aempty(p, lap));
                if (XR) mma_commit(xempty(xb));
                if (last) mma_commit(dfull(par));
                in_blk += kIssuers;
                if ((p += kIssuers) >= kAS) p -= kAS, ++lap;
                if (++xb == kXStages) xb = 0, xph ^= 1u;
            }
            // Every MMA this thread issued completes before the CTA frees tensor memory (and
            // the copies of resident x have landed).
            mma_commit(drain(u));
            wait_bounded(drain(u), 0, kDrainNs, nullptr);
            if (warp == kIss3Warp && !XR && !BF)
                for (int q = 0; q < tpp; ++q) wait_bounded(xfull(kstage(q)), 0, kDrainNs, nullptr);
        }
    } else if (warp < kDeqWarp0) {
        // ----------------------------------------------------------------- epilogue
        const int q = warp & 3;
        const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
        griddep_wait();  // bias, out belong to the dependency chain
        if constexpr (!KS) {
            for (int j = 0; j < my_blocks; ++j) {
                const int par = j & 1;
                if (!__all_sync(0xffffffffu,
                                wait_backoff(dfull(par), (j >> 1) & 1, a.wait_ns, failed, 256))) {
                    if (lane == 0) record_failure(a.status, failed);
                    break;
                }
                tc_fence_after();
                float acc[BT];
#pragma unroll
                for (int u = 0; u < kIssuers; ++u) {
#pragma unroll
                    for (int c = 0; c < BT; c += 16) {
                        uint32_t r[16];
                        tmem_ld16(lane_base + (uint32_t)((par * kIssuers + u) * BT + c), r);
#pragma unroll
                        for (int m = 0; m < 16; ++m)
                            acc[c + m] = u == 0 ? __uint_as_float(r[m]) : acc[c + m] + __uint_as_float(r[m]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(dempty(par));
                const int64_t n = ((int64_t)blockIdx.x + (int64_t)j * gridDim.x) * kRows + q * 32 + lane;
                if (n < a.N && !*failed) {
                    const float cs = PC ? ld_scale(a.scales, F16, n) : 1.f;
                    const float bv = a.bias ? __ldg(a.bias + n) : 0.f;
                    if (BF) {
                        // Columns m and m + 8: the products with x_hi and with x_lo.
#pragma unroll
                        for (int m = 0; m < 8; ++m)
                            if (m < a.M) a.out[(int64_t)m * a.N + n] = fmaf(acc[m] + acc[m + 8], cs, bv);
                    } else {
#pragma unroll
                        for (int m = 0; m < BT; ++m)
                            if (m < a.M) a.out[(int64_t)m * a.N + n] = fmaf(acc[m], cs, bv);
                    }
                }
            }
        } else {
            constexpr int MC = BF ? 8 : BT;  // output columns of a row (bf16: x_hi and x_lo added)
            const int r = q * 32 + lane;
            // After a timed-out wait the warps still walk every item (K split: every ticket is
            // counted and reset), without reading tensor memory or storing.
            bool dead = false;
            for (int j = 0; j < my_blocks; ++j) {
                const int par = j & 1;
                if (!dead && !__all_sync(0xffffffffu,
                                         wait_backoff(dfull(par), (j >> 1) & 1, a.wait_ns, failed, 256))) {
                    if (lane == 0) record_failure(a.status, failed);
                    dead = true;
                }
                if (dead && !KS) break;
                float acc[BT];
#pragma unroll
                for (int m = 0; m < BT; ++m) acc[m] = 0.f;
                if (!dead) {
                    tc_fence_after();
#pragma unroll
                    for (int u = 0; u < kIssuers; ++u) {
#pragma unroll
                        for (int c = 0; c < BT; c += 16) {
                            uint32_t rr[16];
                            tmem_ld16(lane_base + (uint32_t)((par * kIssuers + u) * BT + c), rr);
#pragma unroll
                            for (int m = 0; m < 16; ++m)
                                acc[c + m] = u == 0 ? __uint_as_float(rr[m]) : acc[c + m] + __uint_as_float(rr[m]);
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(dempty(par));
                    if (BF)
#pragma unroll
                        for (int m = 0; m < 8; ++m) acc[m] += acc[m + 8];  // x_hi and x_lo products
                }
                const int blk = blk_of(j);
                const int64_t n = (int64_t)blk * kRows + r;
                if (KS) {
                    // This item's partial tile to the workspace; the last item of the block (ticket)
                    // adds the parts in part order.  The partials are ordered before the ticket by
                    // the epilogue warps' barrier and one device-scope fence of the thread that
                    // takes it; the last item's reads after it by that thread's second fence.
                    float* wp = a.ws + ((int64_t)(blk * parts + my_part) * MC) * kRows + r;
                    if (!dead)
#pragma unroll
                        for (int m = 0; m < MC; ++m) wp[(int64_t)m * kRows] = acc[m];
                    asm volatile("bar.sync 1, 128;" ::: "memory");
                    if (q == 0 && lane == 0) {
                        __threadfence();
                        *s_ticket = atomicAdd(a.tickets + blk, 1);
                        __threadfence();
                    }
                    asm volatile("bar.sync 1, 128;" ::: "memory");
                    if (*s_ticket != parts - 1) continue;
                    const float* rp = a.ws + ((int64_t)blk * parts * MC) * kRows + r;
#pragma unroll
                    for (int m = 0; m < MC; ++m) acc[m] = 0.f;
                    for (int pp = 0; pp < parts; ++pp)
#pragma unroll
                        for (int m = 0; m < MC; ++m) acc[m] += __ldcg(rp + ((int64_t)pp * MC + m) * kRows);
                    if (q == 0 && lane == 0) a.tickets[blk] = 0;
                }
                if (!dead && n < a.N && !*failed) {
                    const float cs = PC ? ld_scale(a.scales, F16, n) : 1.f;
                    const float bv = a.bias ? __ldg(a.bias + n) : 0.f;
#pragma unroll
                    for (int m = 0; m < MC; ++m)
                        if (m < a.M) a.out[(int64_t)m * a.N + n] = fmaf(acc[m], cs, bv);
                }
            }
        }
    } else {
        // ---------------------------------------------------------- dequantization
        const int team = (warp - kDeqWarp0) >> 2;
        const int q = warp & 3;
        const int r = q * 32 + lane;  // this thread's weight row in the block
        const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
        // Slots team, team + kTeams, ...: stage (ring slot b, parity wph), slot sl in it, A
        // ring slot p (and its lap there), advanced without divisions.
        if (BF) {
            // x into its bf16 layout once per CTA (it comes from the preceding kernel), then
            // the tensor core may read it.
            griddep_wait();
            convert_x_bf16(a, xbase, (warp - kDeqWarp0) * 32 + lane, 4 * kTeams * 32);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(xfull(0));
        }
        int sl = team, b = 0, p = team, lap = 0;
        uint32_t wph = 0;
        for (int i = team; i < n_slots; i += kTeams) {
            while (sl >= SPS) {
                sl -= SPS;
                if (++b == a.wst) b = 0, wph ^= 1u;
            }
            // Waits are decided for the whole warp (its tcgen05 instructions are collective).
            // Lap L of the slot is written once the MMAs of lap L - 1 have completed.
            if (!__all_sync(0xffffffffu,
                            (lap == 0 || wait_backoff(aempty(p, lap - 1), ((lap - 1) >> 1) & 1,
                                                      a.wait_ns, failed, 32)) &&
                                wait_backoff(wfull(b), wph, a.wait_ns, failed, 32))) {
                if (lane == 0) record_failure(a.status, failed);
                break;
            }
            // The MMAs that read this slot last have completed (their commit): order the
            // overwrite after them.
            tc_fence_after();
            // The slot's chunks c of the block row; chunk c sits at chunk c ^ (r % 8)
            // (128-byte swizzle).  Their group scales are in the stage's scale block.
            constexpr int kCps = (BF ? kSlotKH : kSlotK) / kChunk;
            uint4 w[kCps];
            float sc[kCps];
#pragma unroll
            for (int h = 0; h < kCps; ++h) {
                const int c = kCps * sl + h;
                w[h] = ld_shared_v4(wstage(b) + (uint32_t)(r * 128) + ((uint32_t)(c ^ (r & 7)) << 4));
                sc[h] = 1.f;
                if (!PC) {
                    const int gl = (c * kChunk) >> (a.gs_shift + 5);
                    const uint8_t* sp = gbase + (wstage(b) - base) + kWBox;
                    sc[h] = F16 ? __half2float(reinterpret_cast<const __half*>(sp)[gl * kRows + r])
                                : reinterpret_cast<const float*>(sp)[gl * kRows + r];
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(wempty(b));  // the warp's reads of the stage are done
            if (BF) {
                // Two chunks (64 k) per store of 32 columns of bf16 pairs.
#pragma unroll
                for (int h2 = 0; h2 < kCps / 2; ++h2) {
                    uint32_t pk[32];
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t v[32];
                        dequant_chunk<EH>(w[2 * h2 + hh], sc[2 * h2 + hh], v);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            pk[16 * hh + i] = bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                    }
                    tmem_st32_async(lane_base + (uint32_t)(kAC0 + p * kSlotK + 32 * h2), pk);
                }
            } else {
#pragma unroll
                for (int h = 0; h < kCps; ++h) {
                    uint32_t v[32];
                    dequant_chunk<EH>(w[h], sc[h], v);
                    tmem_st32_async(lane_base + (uint32_t)(kAC0 + p * kSlotK + kChunk * h), v);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(afull(p, lap));
            sl += kTeams;
            if ((p += kTeams) >= kAS) p -= kAS, ++lap;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

template <bool EH, bool PC, bool F16, bool XR, int BT, bool BF, bool KS>
cudaError_t launch_ts_k(const CUtensorMap& tw, const CUtensorMap& ts, const CUtensorMap& tx,
                        const TsArgs& a, unsigned grid, int smem, const LaunchCtx& c) {
    constexpr auto kernel = tc_small_kernel<EH, PC, F16, XR, BT, BF, KS>;
    const cudaError_t attr = kernel_smem_once<kernel>(kSmemCap);
    if (attr != cudaSuccess) return attr;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(XR ? kThreads : kThreads - 32);  // the x producer warp: streamed x only
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = c.stream;
    cudaLaunchAttribute at[1];
    if (c.pdl) {
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kernel, tw, ts, tx, a);
}

template <bool EH, bool PC, bool F16, bool XR, int BT, bool BF>
cudaError_t launch_ts(const CUtensorMap& tw, const CUtensorMap& ts, const CUtensorMap& tx,
                      const TsArgs& a, unsigned grid, int smem, const LaunchCtx& c) {
    if (a.parts > 1) return launch_ts_k<EH, PC, F16, XR, BT, BF, true>(tw, ts, tx, a, grid, smem, c);
    return launch_ts_k<EH, PC, F16, XR, BT, BF, false>(tw, ts, tx, a, grid, smem, c);
}

template <bool XR, int BT, bool BF = false>
cudaError_t launch_eh(const Problem& p, const CUtensorMap& tw, const CUtensorMap& ts,
                      const CUtensorMap& tx, const TsArgs& a, unsigned grid, int smem,
                      const LaunchCtx& c) {
    const bool pc = p.group_size >= p.K, eh = p.even_high != 0, f16 = p.scale_f16 != 0;
    if (pc) {
        if (eh) return f16 ? launch_ts<true, true, true, XR, BT, BF>(tw, ts, tx, a, grid, smem, c)
                           : launch_ts<true, true, false, XR, BT, BF>(tw, ts, tx, a, grid, smem, c);
        return f16 ? launch_ts<false, true, true, XR, BT, BF>(tw, ts, tx, a, grid, smem, c)
                   : launch_ts<false, true, false, XR, BT, BF>(tw, ts, tx, a, grid, smem, c);
    }
    if (eh) return f16 ? launch_ts<true, false, true, XR, BT, BF>(tw, ts, tx, a, grid, smem, c)
                       : launch_ts<true, false, false, XR, BT, BF>(tw, ts, tx, a, grid, smem, c);
    return f16 ? launch_ts<false, false, true, XR, BT, BF>(tw, ts, tx, a, grid, smem, c)
               : launch_ts<false, false, false, XR, BT, BF>(tw, ts, tx, a, grid, smem, c);
}

int log2_pow2(int64_t v) {
    for (int s = 0; s < 62; ++s)
        if ((int64_t(1) << s) == v) return s;
    return -1;
}

// Shared memory: x (8 chunks x rows x 128 B per 256-k group: all groups when they fit
// next to at least kMinWStages weight stages, else a ring of kXStages; + 1 KiB that the
// 8-row layout's MMAs read past the last chunk), then as many weight stages as fit (at
// most kMaxWStages).  Returns the weight stages (0 if fewer than kMinWStages fit).
int ts_layout(const Problem& p, int smem_cap, uint32_t* x_bytes, int* xrows, int* x_ring,
              int* smem) {
    const int64_t nst = (p.K + kStageK - 1) / kStageK;
    *xrows = p.M <= 8 ? 8 : (p.M <= 16 ? 16 : 32);
    const int64_t gbytes = kChunksPerStage * *xrows * 128;
    const int64_t cap = (int64_t)std::min(smem_cap, kSmemCap) - 1024 - kBarBytes;
    *x_ring = !(nst <= kMaxXGroups && cap - (nst * gbytes + 1024) >= kMinWStages * kWStageBytes);
    *x_bytes = (uint32_t)((*x_ring ? kXStages : nst) * gbytes + 1024);
    const int wst = (int)std::min<int64_t>(kMaxWStages, (cap - *x_bytes) / kWStageBytes);
    if (wst < kMinWStages) return 0;
    *smem = 1024 + (int)*x_bytes + wst * kWStageBytes + kBarBytes;
    return wst;
}

}  // namespace

bool tc_small_eligible(const Problem& p, const LaunchCtx& c) {
    if (p.M < 2 || p.M > kBt || p.N < 1 || p.N > (1LL << 31) - kRows) return false;
    if (p.K % kChunk != 0 || p.K > (1LL << 30)) return false;
    if (reinterpret_cast<uintptr_t>(p.x) % 16 || reinterpret_cast<uintptr_t>(p.qweight) % 16)
        return false;
    if (p.group_size < p.K) {
        // Group scales arrive by TMA: 16-byte aligned base and row, and a group size that
        // is a power-of-two multiple of 32.
        const int esz = p.scale_f16 ? 2 : 4;
        if (p.group_size % kChunk != 0 || log2_pow2(p.group_size / kChunk) < 0) return false;
        if (reinterpret_cast<uintptr_t>(p.scales) % 16 || (p.N * esz) % 16 != 0) return false;
    }
    uint32_t xb;
    int xr, ring, smem;
    if (ts_layout(p, c.max_smem_optin, &xb, &xr, &ring, &smem) == 0) return false;
    return tensor_map_encoder() != nullptr;
}

// K split of the small-M GEMM for matrices with fewer 128-row blocks than SMs: the largest
// count of parts (2, 4 or 8, dividing the 256-k stages, at least two stages a part; bf16
// operands need two for every issuer to have a slot in every item) whose items still fit
// one wave, within the handle's workspace and tickets.  1: no split.  Measured at 8 rows
// (device time, HBM-cold): 4096 x 4096 17.1 -> 9.5 us (4 parts), 6144 x 4096 -> 12.6 (2),
// 4096 x 14336 -> 19.7 (4), 2048 x 2048 -> 5.9 (4); not on 8 stages of more than 48
// blocks (8192 x 2048: 9.1 unsplit, 9.5 in 2 parts).
int tc_small_parts(const Problem& p, const LaunchCtx& c) {
    const int64_t blocks = (p.N + kRows - 1) / kRows, nst = (p.K + kStageK - 1) / kStageK;
    if (!c.ws || !c.tickets || blocks > c.ticket_count || 2 * blocks > c.sm_count) return 1;
    if (nst <= 8 && blocks > 48) return 1;
    const int64_t cols = p.M > 16 ? 32 : 16;
    for (int parts = 8; parts >= 2; parts /= 2)
        if (nst % parts == 0 && nst / parts >= 2 && blocks * parts <= c.sm_count &&
            blocks * parts * cols * kRows <= c.ws_floats)
            return parts;
    return 1;
}

// bf16 operands (x split into two bf16 terms) where they apply: up to 8 rows, x resident,
// at least two 256-k stages (every issuer then has a slot in every block) and an even
// weight ring of at least four stages.  With two A slots a stage, even stages go to teams
// 0-1 and odd ones to teams 2-3; an even ring keeps each ring stage with one pair of teams,
// so that a team waits for every lap of the stages it reads (a parity wait must not run a
// lap ahead of the barrier).  By default from 100 row blocks of 128, where they were
// measured 2-5 % faster than tf32 (128256 x 2048 at 4 rows: 55.3 against 58.0 us; 14336 x
// 4096: 18.7 against 19.4), not on fewer (8192 x 2048: 10.1 against 9.2).
bool tc_small_uses_bf16(const Problem& p, const LaunchCtx& c) {
    if (c.tc_small_operands == 1 || p.M > 8 || p.K <= kStageK || !tc_small_eligible(p, c))
        return false;
    uint32_t xb;
    int xr, ring, smem;
    const int wst = ts_layout(p, c.max_smem_optin, &xb, &xr, &ring, &smem);
    if (ring || (wst & ~1) < 4) return false;
    return c.tc_small_operands == 2 || (p.N + kRows - 1) / kRows >= 100;
}

cudaError_t tc_small_launch(const Problem& p, const LaunchCtx& c) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc || !tc_small_eligible(p, c)) return cudaErrorNotSupported;
    const bool pc = p.group_size >= p.K;
    const int esz = p.scale_f16 ? 2 : 4;
    TsArgs a = {};
    a.x = p.x;
    a.K = (int)p.K;
    a.scales = p.scales;
    a.bias = p.bias;
    a.out = p.out;
    a.M = (int)p.M;
    a.N = (int)p.N;
    a.nst = (int)((p.K + kStageK - 1) / kStageK);
    a.blocks = (int)((p.N + kRows - 1) / kRows);
    a.gs_shift = pc ? 0 : log2_pow2(p.group_size / kChunk);
    const int gps = pc ? 0 : std::max(1, kStageK >> (a.gs_shift + 5));
    a.w_tx = (uint32_t)(kWBox + gps * kRows * esz);
    int smem = 0;
    a.wst = ts_layout(p, c.max_smem_optin, &a.x_bytes, &a.xrows, &a.x_ring, &smem);
    a.skip_first_copy = c.tc_skip_first_copy;
    a.status = c.status_word;
    a.wait_ns = c.wait_limit_ns;
    a.parts = tc_small_parts(p, c);
    a.ws = c.ws;
    a.tickets = c.tickets;

    CUtensorMap tw, ts, tx;
    const cuuint32_t e2[2] = {1, 1}, e3[3] = {1, 1, 1};
    {
        // Packed codes [N rows x K/2 bytes]: boxes [128 rows x 128 B], 128-byte swizzle.
        const cuuint64_t dims[2] = {(cuuint64_t)(p.K / 2), (cuuint64_t)p.N};
        const cuuint64_t strides[1] = {(cuuint64_t)(p.K / 2)};
        const cuuint32_t box[2] = {128, (cuuint32_t)kRows};
        if (enc(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(p.qweight), dims,
                strides, box, e2, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    if (!pc) {
        // Group scales [G groups x N]: boxes [gps groups x 128 rows] (gps = 256 / gs, or 1).
        const int64_t G = (p.K + p.group_size - 1) / p.group_size;
        const cuuint64_t dims[2] = {(cuuint64_t)p.N, (cuuint64_t)G};
        const cuuint64_t strides[1] = {(cuuint64_t)(p.N * esz)};
        const cuuint32_t box[2] = {(cuuint32_t)kRows, (cuuint32_t)gps};
        if (enc(&ts, p.scale_f16 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT32,
                2, const_cast<void*>(p.scales), dims, strides, box, e2, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    } else {
        ts = tw;  // unused
    }
    {
        // x [M rows x K] as (32 k, row, 32-k chunk): one box = 8 chunks of [16 rows x 128 B],
        // 128-byte swizzle; rows past M and chunks past K read as zeros.
        const cuuint64_t dims[3] = {32, (cuuint64_t)p.M, (cuuint64_t)(p.K / 32)};
        const cuuint64_t strides[2] = {(cuuint64_t)(p.K * 4), 128};
        const cuuint32_t box[3] = {32, (cuuint32_t)a.xrows, (cuuint32_t)kChunksPerStage};
        if (enc(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(p.x), dims, strides,
                box, e3, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const int64_t items = (int64_t)a.blocks * a.parts;
    const unsigned grid = (unsigned)(std::min<int64_t>(items, c.sm_count) / a.parts * a.parts);
    if (tc_small_uses_bf16(p, c)) {
        a.wst &= ~1;
        return launch_eh<false, 16, true>(p, tw, ts, tx, a, grid, smem, c);
    }
    if (p.M > 16)
        return a.x_ring ? launch_eh<true, 32>(p, tw, ts, tx, a, grid, smem, c)
                        : launch_eh<false, 32>(p, tw, ts, tx, a, grid, smem, c);
    return a.x_ring ? launch_eh<true, 16>(p, tw, ts, tx, a, grid, smem, c)
                    : launch_eh<false, 16>(p, tw, ts, tx, a, grid, smem, c);
}

}  // namespace q4lin
