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
//     spans the 512 bytes) and of the matching block of group scales [1024 / group size
//     groups x rb rows], all on one mbarrier, into a ring of 2..8 stages (the first
//     stage alone, then the rest of the ring once it has landed, so that every CTA's
//     first stage is ahead of the grid's later ones in the memory queues).  Weight rows
//     are long contiguous segments, so DRAM sees streaming reads.
//   8 consumer warps (256 threads): thread = (chunk lane j of CL, row group of V rows),
//     with (V, CL) = (2, 32) or (4, 32) for blocks of 16 or 32 rows and (4, 16) for 64;
//     per stage it takes chunks j, j + CL, ... (32 codes each) of each of its V rows, and
//     each x chunk it loads serves all V rows.
//     x is staged whole in shared memory once per CTA after the dependency wait (every
//     consumer thread copies 16-byte units, all in flight at once; the CTA's first stage
//     is a copy group of its own, so computing starts once it has landed), unit u of
//     32-k chunk c at unit u ^ (c % 8) of the chunk's 128-byte row.  A quarter-warp then reads
//     128 contiguous bytes of a weight row and 8 different 16-byte units of x, both
//     conflict-free.  Partial sums stay in registers for the whole row; the CL chunk lanes
//     of a row group are reduced with shuffles once per row block.
// Arithmetic (X8 instances): a tenth warp converts the staged x, stage by stage, in place
// into 32-bit fixed point per 32-k chunk (one chunk per lane, all in registers): with F
// the largest exponent field of the chunk, q = round(x * 2^(157 - F)) (|q| < 2^31; exact
// for every element within a factor 128 of the chunk's largest), stored as 4 byte slices;
// the consumers wait for a stage's conversion (its own mbarrier) at its first use.  A
// chunk's dot product sum_k (c_k - 8) * q_k is then exact integer arithmetic: 8 dp4a per 8
// codes (codes as unsigned bytes, one nibble mask each), with the -8 offset folded into
// the accumulators' starting values (-8 * sum_k q_k, split into two 16-bit halves); it is
// rounded once to fp32, scaled by 2^(F - 157) (exact) and accumulated with the group scale
// in fp32.  A stage holding Inf or NaN (IEEE propagation is unchanged) or a chunk with a
// nonzero element more than 2^13 below the chunk's largest keeps its fp32 values and takes
// the fp32 path, so every converted element has a relative error <= 2^-18.  fp32 instances
// (and such stages): the codes widened to exact floats by a byte permute
// (0x4B0000cc = 2^23 + c) and one packed add, fp32 FMA.
// A CTA is small enough (288 threads, 320 with the conversion warp, at most 113 KiB of
// shared memory) that two fit on one SM: the CTAs of the next kernel on the stream can become resident while this one
// runs.  With programmatic dependent launch their producers then stream weights and
// scales (which do not depend on the preceding kernel) before griddepcontrol.wait; x,
// bias, out and the split-K workspace are touched only after it.
// Row blocks of long-K, short-N matrices are split along K across CTAs; the partial row
// sums go to a workspace and the last CTA of a row block adds them in part order (the
// result does not depend on which CTA finishes last).  (A stream-K cut of the (row block,
// stage) units into equal runs per CTA was measured too: its split hand-offs cost more
// than its balance gained on the decode shapes.)
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
constexpr int kThreadsX8 = kThreadsG + 32; // + the x conversion warp (fixed-point instances)
// A consumer thread is (row group, chunk lane): CL chunk lanes (16 or 32) per row group,
// kCThreads / CL row groups of V rows each, so a row block has kCThreads / CL * V rows.
__host__ __device__ constexpr int rows_per_block(int V, int CL) { return kCThreads / CL * V; }
static_assert(rows_per_block(2, 32) == kGemvMinRowBlock && rows_per_block(4, 16) == kGemvMaxRowBlock,
              "row blocks of 16 to 64 rows");
constexpr int kSRB = 512;                  // packed bytes of a row per stage (1024 k)
constexpr int kSC = 32;                    // 32-k chunks per stage
constexpr int kXStageBytes = 4096;         // x of one stage: 32 chunk rows x 128 bytes
constexpr int kMetaBytes = 16;             // per chunk: factor, two offsets (one word unused)
constexpr int kMaxStages = 8;
constexpr int kMaxXStages = 32;            // K <= 32768 (x staged whole in shared memory)
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
    int kstages;     // ceil(K / 1024)
    int gs_shift;    // log2(group size / 32) (grouped scales)
    int stages;      // ring depth
    int burst;       // stages armed before the first one has landed (0: the whole ring)
    uint32_t stage_bytes, scale_off, stage_tx;
    uint32_t x_off, meta_off, bar_off;  // shared-memory layout, from the 1024-aligned base
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

// Shared memory: the stage ring, x (kstages x 4 KiB), the chunk metadata, then barriers
// and flags (512 bytes).
struct SmemLayout {
    uint32_t x_off, meta_off, bar_off, total;
};
inline SmemLayout smem_layout(int stages, uint32_t stage_bytes, int kstages) {
    SmemLayout l;
    l.x_off = (uint32_t)stages * stage_bytes;  // stage bytes are multiples of 1024
    l.meta_off = l.x_off + (uint32_t)kstages * kXStageBytes;
    l.bar_off = l.meta_off + (uint32_t)kstages * kSC * kMetaBytes;
    l.total = 1024 + l.bar_off + 512;
    return l;
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

// Address of 16-byte unit u (4 consecutive k) of 32-k chunk c in the staged x: chunk row
// c at c * 128 bytes, unit u at u ^ (c % 8), so that the 8 chunk lanes of a quarter-warp
// (8 consecutive chunks, same unit) hit 8 different bank groups.
__device__ __forceinline__ uint32_t x_unit(uint32_t xa, int c, int u) {
    return xa + (uint32_t)c * 128u + ((uint32_t)(u ^ (c & 7)) << 4);
}

// Matrix that owns global row block blk (blk_begin ascending, matrix 0 begins at 0).
__device__ __forceinline__ int mat_of(const GArgs& a, int64_t blk) {
    int i = 0;
#pragma unroll
    for (int q = 1; q < kMaxMats; ++q)
        if (q < a.nmat && blk >= a.mat[q].blk_begin) i = q;
    return i;
}

// fp32 chunk dot: products x[t] * (code_t - 8) of one 16-byte chunk (32 codes), summed as
// a float2 of (even-k sum, odd-k sum) where the lane fed from the HIGH nibbles carries a
// factor 16.  Byte b of a word holds k = 2b in its low nibble and k = 2b + 1 in its high
// nibble (swapped when EH).  The low nibbles are isolated with one mask (w & 0x0F0F0F0F)
// and the high nibbles in place with another (w & 0xF0F0F0F0, i.e. 16 * code): no shift.
// A byte permute builds the float 2^23 + byte (bit pattern 0x4B0000bb) and one packed add
// of -(2^23 + 8) (low lane) / -(2^23 + 128) (high lane) gives c - 8 and 16 * (c - 8), both
// exact.
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
template <bool EH>
__device__ __forceinline__ float chunk_dot_f32(const uint4& wv, const uint4 (&xu)[8]) {
    float4 xv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        xv[i] = make_float4(__uint_as_float(xu[i].x), __uint_as_float(xu[i].y),
                            __uint_as_float(xu[i].z), __uint_as_float(xu[i].w));
    const float2 d = chunk_dot<EH>(wv, xv);
    return EH ? fmaf(d.x, 0.0625f, d.y) : fmaf(d.y, 0.0625f, d.x);
}

// Fixed-point chunk dot: sum_k (c_k - 8) * q_k of one chunk, exact, rounded once to fp32.
// xu[2w] = (s0e, s1e, s0o, s1o) and xu[2w+1] = (s2e, s3e, s2o, s3o) for word w: slice s
// (byte 3 - s of q, slice 0 signed) of the even / odd k of the word, one byte per k.
// init = (-8 * sum_k (q_k >> 16), -8 * sum_k (q_k & 0xFFFF)).
template <bool EH>
__device__ __forceinline__ float chunk_dot_x8(const uint4& wv, const uint4 (&xu)[8], int init_hi,
                                              int init_lo) {
    int a0 = 0, a1 = init_hi, a2 = 0, a3 = init_lo;
    const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const uint32_t lo = words[w] & 0x0F0F0F0Fu, hi = (words[w] >> 4) & 0x0F0F0F0Fu;
        const uint32_t ev = EH ? hi : lo, od = EH ? lo : hi;  // codes of even / odd k
        const uint4 A = xu[2 * w], B = xu[2 * w + 1];
        a0 = dp4a_us(ev, A.x, a0);
        a0 = dp4a_us(od, A.z, a0);
        a1 = dp4a_uu(ev, A.y, a1);
        a1 = dp4a_uu(od, A.w, a1);
        a2 = dp4a_uu(ev, B.x, a2);
        a2 = dp4a_uu(od, B.z, a2);
        a3 = dp4a_uu(ev, B.y, a3);
        a3 = dp4a_uu(od, B.w, a3);
    }
    // |hi| < 2^23 and |lo| < 2^24: both convert exactly; one rounding in the fma.
    const int hi_v = a0 * 256 + a1, lo_v = a2 * 256 + a3;
    return fmaf((float)hi_v, 65536.f, (float)lo_v);
}

// 4 x 4 byte transpose: out[s] holds byte 3 - s of a, b, c, d (in that byte order), so
// out[0] is the top (signed) byte slice of the four values and out[3] the lowest.
__device__ __forceinline__ void byte_slices(uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                            uint32_t (&out)[4]) {
    const uint32_t t0 = prmt(a, b, 0x5140u), t1 = prmt(a, b, 0x7362u);
    const uint32_t t2 = prmt(c, d, 0x5140u), t3 = prmt(c, d, 0x7362u);
    out[3] = prmt(t0, t2, 0x5410u);
    out[2] = prmt(t0, t2, 0x7632u);
    out[1] = prmt(t1, t3, 0x5410u);
    out[0] = prmt(t1, t3, 0x7632u);
}

// The conversion warp's share of stage ks: lane j converts 32-k chunk c = 32 ks + j of
// the staged x in place, on its own (the whole chunk in registers: no shuffles, no CTA
// barrier), into the fixed-point layout that chunk_dot_x8 reads: with F the chunk's largest exponent field,
// q = round(x * 2^(157 - max(F, 31))), unit 2w = (s0e, s1e, s0o, s1o) and unit 2w + 1 =
// (s2e, s3e, s2o, s3o) for word w, where sXe / sXo is slice X (byte 3 - X of q) of the even
// / odd k of the word, one byte per k in k order; metadata (factor, -8 sum(q >> 16),
// -8 sum(q & 0xFFFF), 1).  If any chunk of the stage holds an Inf or NaN or a nonzero
// element more than 2^13 below its chunk's largest, the whole stage stays fp32 and every
// chunk's metadata word 3 is 0.  Returns whether the stage was converted.
__device__ __forceinline__ bool convert_x_chunk_lane(uint32_t xa, uint32_t meta, int ks, int lane) {
    const int c = ks * kSC + lane;
    uint32_t b[32];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const uint4 r = ld_shared_v4(x_unit(xa, c, u));
        b[4 * u] = r.x, b[4 * u + 1] = r.y, b[4 * u + 2] = r.z, b[4 * u + 3] = r.w;
    }
    // Largest exponent field F, and that of the smallest nonzero |x| (E; 255 when all are
    // zero): unsigned order of |x|'s bit pattern is exponent order.  (|x| - 1 wraps a zero
    // to the top, so the minimum skips zeros.)
    uint32_t amax = 0, amin1 = 0xFFFFFFFFu;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const uint32_t ab = b[i] & 0x7FFFFFFFu;
        amax = max(amax, ab);
        amin1 = min(amin1, ab - 1u);
    }
    const uint32_t F = amax >> 23;
    const uint32_t E = amin1 == 0xFFFFFFFFu ? 255u : max((amin1 + 1u) >> 23, 1u);
    const bool keep = __any_sync(0xffffffffu, F == 255u || E + 13u < F);
    if (keep) {
        st_shared_v4(meta + (uint32_t)c * kMetaBytes, 0u, 0u, 0u, 0u);
        return false;
    }
    const uint32_t Fm = max(F, 31u);
    const float mul = __uint_as_float((284u - min(Fm, 254u)) << 23);
    // Sums of the byte slices over the chunk (slice 0 signed): q >> 16 = 256 s0 + s1 and
    // q & 0xFFFF = 256 s2 + s3, so the offsets come from 8 dp4a per word.
    constexpr uint32_t kOnes = 0x01010101u;
    int s0 = 0, s1 = 0, s2 = 0, s3 = 0;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        uint32_t q[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = (uint32_t)__float2int_rn(__uint_as_float(b[8 * w + i]) * mul);
        uint32_t e[4], o[4];
        byte_slices(q[0], q[2], q[4], q[6], e);
        byte_slices(q[1], q[3], q[5], q[7], o);
        st_shared_v4(x_unit(xa, c, 2 * w), e[0], e[1], o[0], o[1]);
        st_shared_v4(x_unit(xa, c, 2 * w + 1), e[2], e[3], o[2], o[3]);
        s0 = dp4a_us(kOnes, e[0], dp4a_us(kOnes, o[0], s0));
        s1 = dp4a_uu(kOnes, e[1], dp4a_uu(kOnes, o[1], s1));
        s2 = dp4a_uu(kOnes, e[2], dp4a_uu(kOnes, o[2], s2));
        s3 = dp4a_uu(kOnes, e[3], dp4a_uu(kOnes, o[3], s3));
    }
    const int qh = s0 * 256 + s1, ql = s2 * 256 + s3;
    st_shared_v4(meta + (uint32_t)c * kMetaBytes, (Fm - 30u) << 23, (uint32_t)(-8 * qh),
                 (uint32_t)(-8 * ql), 1u);
    return true;
}

// One chunk of a stage for a thread's V rows: x chunk c from the staged x, the V rows'
// 16-byte code units at wrow + v * 512, their group scales at saddr; fixed-point (FX, with
// the chunk's metadata md: factor, two offsets) or fp32 arithmetic, accumulated into acc.
template <int V, bool EH, bool PC, bool F16, bool FX>
__device__ __forceinline__ void stage_chunk(uint32_t xa, int c, const uint4& md, uint32_t saddr,
                                            uint32_t wrow, float (&acc)[V]) {
    uint4 xu[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) xu[i] = ld_shared_v4(x_unit(xa, c, i));
    float sc[V];
    if (!PC) stage_scales<V, F16>(saddr, sc);
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const uint4 wv = ld_shared_v4(wrow + v * kSRB);
        const float t = FX ? chunk_dot_x8<EH>(wv, xu, (int)md.y, (int)md.z) * __uint_as_float(md.x)
                           : chunk_dot_f32<EH>(wv, xu);
        acc[v] = PC ? acc[v] + t : fmaf(t, sc[v], acc[v]);
    }
}

template <int V, int CL, bool EH, bool PC, bool F16, bool X8>
__global__ void __launch_bounds__(X8 ? kThreadsX8 : kThreadsG, 2)
    gemv_tma_kernel(const __grid_constant__ TensorMaps tmaps, const GArgs a) {
    constexpr int rb = rows_per_block(V, CL);  // row groups of V rows
    constexpr int H = kSC / CL;                // chunks of a stage per chunk lane
    constexpr uint32_t esz = F16 ? 2 : 4;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // stages are 1024-byte aligned
    uint8_t* gbase = smem_raw + (base - raw);
    const int S = a.stages;
    const uint32_t bar_base = base + a.bar_off;
    const uint32_t xa = base + a.x_off, meta = base + a.meta_off;
    volatile int* failed = reinterpret_cast<volatile int*>(gbase + a.bar_off + 16 * kMaxStages);
    volatile int* s_ticket = failed + 1;  // last-item decision, broadcast to the consumers
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto full = [&](int s) { return bar_base + 8u * s; };
    auto empty = [&](int s) { return bar_base + 8u * (kMaxStages + s); };
    // X8: stage ks of x converted by the conversion warp (its 32 lanes arrive).
    auto xconv = [&](int ks) { return bar_base + 256u + 8u * ks; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), kCWarps);
        }
        if (X8)
            for (int ks = 0; ks < a.kstages; ++ks) mbar_init(xconv(ks), 32);
        *failed = 0;
        mbar_init_fence();
    }
    __syncthreads();
    griddep_launch_dependents();
    // The stage of x this CTA uses first (its first item's first stage): it is copied
    // (and converted) ahead of the rest of x.
    const int ks_first = (int)blockIdx.x < a.items ? ((int)blockIdx.x % a.parts) * a.tpp : 0;

    if (warp == kCWarps) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            for (int q = 0; q < a.nmat; ++q) {
                prefetch_tensormap(&tmaps.w[q]);
                if (!PC) prefetch_tensormap(&tmaps.s[q]);
            }
            // Pull x toward L2 now, so that the consumers' reads after griddepcontrol.wait
            // are short.  L2 is where global memory is kept coherent: if the preceding
            // kernel writes x after this prefetch, the L2 line is updated and the later read
            // sees it; no copy of x enters this SM before the wait.
            const int64_t xb = a.K * 4;
            for (int64_t off = 0; off < xb; off += 32768)
                l2_prefetch_bulk(a.x + off / 4, (uint32_t)(xb - off < 32768 ? xb - off : 32768));
            int t = 0, s = 0;
            uint32_t ph = 0;
            Cursor cur;
            cur.start(a);
            while (cur.valid(a)) {
                // Arm `burst` stages, then wait for the first to land before arming the rest
                // of the ring: every CTA's first stage is then ahead of the grid's later
                // stages in the memory queues, and the consumers start sooner.
                if (t == a.burst && a.burst > 0 && a.burst < S &&
                    !wait_bounded(full(0), 0u, a.wait_ns, failed)) {
                    record_failure(a.status, failed);
                    break;
                }
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
                    tma_load_2d(sb + a.scale_off, &tmaps.s[mi], row0, (cur.ks * kSC) >> a.gs_shift,
                                full(s));
                ++t;
                if (++s == S) s = 0, ph ^= 1u;
                cur.advance(a);
            }
            // The last armed copies may still be landing; the CTA must not exit first.
            for (int q = t > S ? t - S : 0; q < t; ++q)
                wait_bounded(full(q % S), (uint32_t)(q / S) & 1u, kDrainNs, nullptr);
        }
        return;
    }
    if (X8 && warp == kCWarps + 1) {
        // ------------------------------------------------ x conversion (X8 instances)
        // The first stage of x once the consumers have staged it (named barrier 2), then
        // the rest once that has landed too (barrier 3), in the order the consumers first
        // use the stages, off their critical path; stage ks is released to them by its
        // mbarrier (every lane arrives after its stores).
        asm volatile("bar.sync 2, %0;" ::"r"(kCThreads + 32) : "memory");
        convert_x_chunk_lane(xa, meta, ks_first, lane);
        mbar_arrive(xconv(ks_first));
        asm volatile("bar.sync 3, %0;" ::"r"(kCThreads + 32) : "memory");
        for (int q = 1, ks = ks_first; q < a.kstages; ++q) {
            if (++ks == a.kstages) ks = 0;
            convert_x_chunk_lane(xa, meta, ks, lane);
            mbar_arrive(xconv(ks));
        }
        return;
    }

    // ------------------------------------------------------------------ consumers
    const int j = threadIdx.x & (CL - 1);    // chunk lane: chunks j, j + CL, ... of a stage
    const int r0 = (threadIdx.x / CL) * V;   // first of this thread's V rows in a block
    griddep_wait();  // x, bias, out and the workspace belong to the dependency chain
    // x into shared memory once: 16-byte unit i (k = 4 i .. 4 i + 3) of chunk i / 8 at its
    // swizzled place, zero past K.  Asynchronous copies, all in flight at once, one unit
    // per thread and stage: the CTA's first stage as one group, the rest as a second, so
    // that the consumers start on the first stage once it has landed.
    auto copy_x_stage = [&](int ks) {
        const int i = ks * kCThreads + threadIdx.x;
        const bool in = 4 * (int64_t)i < a.K;
        cp_async_16(x_unit(xa, i >> 3, i & 7),
                    in ? static_cast<const void*>(reinterpret_cast<const float4*>(a.x) + i) : a.x,
                    in ? 16u : 0u);
    };
    static_assert(kSC * 8 == kCThreads, "one 16-byte unit of x per consumer thread and stage");
    copy_x_stage(ks_first);
    cp_async_commit();
    for (int ks = 0; ks < a.kstages; ++ks)
        if (ks != ks_first) copy_x_stage(ks);
    cp_async_commit();
    cp_async_wait_group<1>();
    // X8: the conversion warp takes part (it converts the first stage next).
    if (X8)
        asm volatile("bar.sync 2, %0;" ::"r"(kCThreads + 32) : "memory");
    else
        asm volatile("bar.sync 1, %0;" ::"r"(kCThreads) : "memory");
    // The rest of x (possibly no copy): waited for at the first use of another stage, or
    // before leaving; either way once, with the conversion warp's second barrier.
    bool x_rest = false;
    auto wait_x_rest = [&]() {
        cp_async_wait_all();
        if (X8)
            asm volatile("bar.sync 3, %0;" ::"r"(kCThreads + 32) : "memory");
        else
            asm volatile("bar.sync 1, %0;" ::"r"(kCThreads) : "memory");
        x_rest = true;
    };

    // Per row: fp32 partial sum, scaled per chunk by the group scale.
    float acc[V];
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] = 0.f;
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
    // Per-thread offsets: the thread's rows of a weight stage (row r at r * kSRB bytes,
    // chunk column c at c * 16), its group-scale rows.
    const uint32_t w_off = (uint32_t)(r0 * kSRB + j * 16);
    uint32_t s_off[H];
#pragma unroll
    for (int h = 0; h < H; ++h)
        s_off[h] = a.scale_off + scale_slot<rb * esz>((h * CL + j) >> a.gs_shift, r0 * esz);
    uint32_t x_ready = X8 ? 0u : ~0u;  // stages of x this CTA has looked at
    uint32_t x_fixed = 0u;             // ... and converted to fixed point
    // After a timed-out wait (`dead`) the warp still walks every item, without waiting or
    // computing, so that all consumer warps reach the same named barriers and every split-K
    // ticket is still counted and reset; nothing is stored.
    bool dead = false;
    while (cur.valid(a)) {
        const int ks = cur.ks;
        // Every consumer warp walks the same items, so all of them reach this together.
        if (!x_rest && ks != ks_first) wait_x_rest();
        if (X8 && !((x_ready >> ks) & 1u)) {
            // First use of this stage of x by the CTA: wait for the conversion warp; the
            // metadata of the stage's first chunk says whether it was converted.
            if (!dead &&
                !__all_sync(0xffffffffu, wait_bounded(xconv(ks), 0u, a.wait_ns, failed))) {
                if (lane == 0) record_failure(a.status, failed);
                dead = true;
            }
            if (!dead && ld_shared_v4(meta + (uint32_t)(ks * kSC) * kMetaBytes).w != 0u)
                x_fixed |= 1u << ks;
            x_ready |= 1u << ks;
        }
        const bool got =
            !dead && __all_sync(0xffffffffu, wait_bounded(full(s), ph, a.wait_ns, failed));
        if (!got && !dead) {
            if (lane == 0) record_failure(a.status, failed);
            dead = true;
        }
        if (got) {
            const uint32_t sb = base + (uint32_t)s * a.stage_bytes;
            if (X8 && ((x_fixed >> ks) & 1u)) {
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    const int c = ks * kSC + h * CL + j;
                    stage_chunk<V, EH, PC, F16, true>(xa, c, ld_shared_v4(meta + (uint32_t)c * kMetaBytes),
                                                      sb + s_off[h], sb + w_off + h * CL * 16, acc);
                }
            } else {
#pragma unroll
                for (int h = 0; h < H; ++h)
                    stage_chunk<V, EH, PC, F16, false>(xa, ks * kSC + h * CL + j, make_uint4(0u, 0u, 0u, 0u),
                                                       sb + s_off[h], sb + w_off + h * CL * 16, acc);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(s));
        if (++s == S) s = 0, ph ^= 1u;
        const int blk = cur.blk;
        const int part = cur.part;
        if (cur.advance(a)) {
            // Item done: reduce the CL chunk lanes of each row; store (or hand the partial
            // to the last item).
            float tot[V];
#pragma unroll
            for (int v = 0; v < V; ++v) {
                tot[v] = acc[v];
#pragma unroll
                for (int o = 1; o < CL; o <<= 1)
                    tot[v] += __shfl_xor_sync(0xffffffffu, tot[v], o);
                acc[v] = 0.f;
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
                        float t[kGemvMaxParts];
#pragma unroll
                        for (int q = 0; q < kGemvMaxParts; ++q)
                            t[q] = q < a.parts ? __ldcg(a.ws + (int64_t)q * a.ws_rows + vrow) : 0.f;
                        mine = t[0];
#pragma unroll
                        for (int q = 1; q < kGemvMaxParts; ++q)
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
    // A CTA that used only its first stage still meets the conversion warp's barrier and
    // must not exit while copies of x are landing.
    if (!x_rest) wait_x_rest();
}

template <int V, int CL, bool EH, bool PC, bool F16, bool X8>
cudaError_t launch_v(const TensorMaps& tm, const GArgs& a, unsigned grid, uint32_t smem,
                     const LaunchCtx& c) {
    constexpr auto kernel = gemv_tma_kernel<V, CL, EH, PC, F16, X8>;
    const cudaError_t attr = kernel_smem_once<kernel>(kCtaSmem, 100);
    if (attr != cudaSuccess) return attr;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(X8 ? kThreadsX8 : kThreadsG);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = c.stream;
    cudaLaunchAttribute attrs[1];
    if (c.pdl) {
        attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attrs;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kernel, tm, a);
}

template <int V, int CL, bool EH, bool PC, bool F16>
cudaError_t dispatch_x8(bool x8, const TensorMaps& tm, const GArgs& a, unsigned grid,
                        uint32_t smem, const LaunchCtx& c) {
    return x8 ? launch_v<V, CL, EH, PC, F16, true>(tm, a, grid, smem, c)
              : launch_v<V, CL, EH, PC, F16, false>(tm, a, grid, smem, c);
}
template <int V, int CL, bool EH, bool PC>
cudaError_t dispatch_f16(bool f16, bool x8, const TensorMaps& tm, const GArgs& a, unsigned grid,
                         uint32_t smem, const LaunchCtx& c) {
    return f16 ? dispatch_x8<V, CL, EH, PC, true>(x8, tm, a, grid, smem, c)
               : dispatch_x8<V, CL, EH, PC, false>(x8, tm, a, grid, smem, c);
}
template <int V, int CL, bool EH>
cudaError_t dispatch_pc(bool pc, bool f16, bool x8, const TensorMaps& tm, const GArgs& a,
                        unsigned grid, uint32_t smem, const LaunchCtx& c) {
    return pc ? dispatch_f16<V, CL, EH, true>(f16, x8, tm, a, grid, smem, c)
              : dispatch_f16<V, CL, EH, false>(f16, x8, tm, a, grid, smem, c);
}
template <int V, int CL>
cudaError_t dispatch_eh(bool eh, bool pc, bool f16, bool x8, const TensorMaps& tm,
                        const GArgs& a, unsigned grid, uint32_t smem, const LaunchCtx& c) {
    return eh ? dispatch_pc<V, CL, true>(pc, f16, x8, tm, a, grid, smem, c)
              : dispatch_pc<V, CL, false>(pc, f16, x8, tm, a, grid, smem, c);
}

// Tiles of the decode GEMV: V rows per thread and CL chunk lanes per row group, so
// kCThreads / CL * V rows per block.  Rows 16 and 32 use 32 chunk lanes: each thread takes
// one chunk of a stage for its 2 or 4 rows, and a staged x chunk is read once per 2 or 4
// rows (with 16 chunk lanes the same heights would be 1 or 2 rows per thread, and x, read
// once per row or two, would bound the launch by shared-memory bandwidth).  Rows 64 keep
// 16 chunk lanes (4 rows per thread: 32 would need 8).  Listed so that at equal cost the
// taller block wins: it does twice the work per stage and per row-block reduction
// (measured: 128256 x 4096 55.3 us with 64-row blocks, 62.4 with 32).
struct Tile {
    int V, CL;
    int rows() const { return kCThreads / CL * V; }
};
constexpr Tile kTiles[] = {{4, 16}, {4, 32}, {2, 32}};

cudaError_t dispatch_tile(Tile t, bool eh, bool pc, bool f16, bool x8, const TensorMaps& tm,
                          const GArgs& a, unsigned grid, uint32_t smem, const LaunchCtx& c) {
    if (t.CL == 16) return dispatch_eh<4, 16>(eh, pc, f16, x8, tm, a, grid, smem, c);
    if (t.V == 4) return dispatch_eh<4, 32>(eh, pc, f16, x8, tm, a, grid, smem, c);
    return dispatch_eh<2, 32>(eh, pc, f16, x8, tm, a, grid, smem, c);
}

int log2_exact(int64_t v) {
    for (int s = 0; s < 62; ++s)
        if (((int64_t)1 << s) == v) return s;
    return -1;
}

// Bytes of one stage of rb rows (weights, then the scale block, rounded up to 1 KiB).
uint32_t stage_bytes_for(int rb, bool pc, int esz, int gs_shift, uint32_t* scale_off,
                         uint32_t* tx) {
    const uint32_t wbytes = (uint32_t)(rb * kSRB);
    const int gps = pc ? 0 : (gs_shift >= 5 ? 1 : kSC >> gs_shift);
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
    if (p.N > (1LL << 30) || p.K > (int64_t)kMaxXStages * 1024) return false;
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
    const int kstages = (int)((p.K + 1023) / 1024);
    uint32_t so, tx;
    const uint32_t sb1 = stage_bytes_for(kGemvMinRowBlock, pc, p.scale_f16 ? 2 : 4,
                                         pc ? 0 : log2_exact(p.group_size / 32), &so, &tx);
    if (smem_layout(2, sb1, kstages).total > (uint32_t)kCtaSmem) return false;
    return tensor_map_encoder() != nullptr;
}

int gemv_tma_max_group() { return kMaxMats; }

bool gemv_tma_groupable(const Problem& a, const Problem& b) {
    return a.x == b.x && a.K == b.K && a.group_size == b.group_size &&
           a.scale_f16 == b.scale_f16 && a.even_high == b.even_high &&
           (a.group_size >= a.K) == (b.group_size >= b.K);
}

namespace {

// Plans the launch of ps[0..count) (tile, split of K, grid, arithmetic) and, when `launch`,
// enqueues it; *x8_out (if given) receives whether the fixed-point instances are chosen.
cudaError_t gemv_group(const Problem* ps, int count, const LaunchCtx& c, bool launch,
                       bool* x8_out) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc || count < 1 || count > kMaxMats) return cudaErrorNotSupported;
    const Problem& p0 = ps[0];
    const bool pc = p0.group_size >= p0.K;
    const int esz = p0.scale_f16 ? 2 : 4;
    const int gs_shift = pc ? 0 : log2_exact(p0.group_size / 32);
    const int kstages = (int)((p0.K + 1023) / 1024);
    const int slots = 2 * c.sm_count;
    auto blocks_for = [&](int rb) {
        int64_t b = 0;
        for (int i = 0; i < count; ++i) b += (ps[i].N + rb - 1) / rb;
        return b;
    };
    auto stages_for = [&](int rb) {
        uint32_t so, tx;
        const uint32_t sb = stage_bytes_for(rb, pc, esz, gs_shift, &so, &tx);
        const int room = kCtaSmem - (int)smem_layout(0, sb, kstages).total;
        return std::min<int>(kMaxStages, room / (int)sb);
    };
    // Tile and split-K parts from a cost model of the critical CTA, fitted to measured
    // launch times on GB300 (isolated GEMVs, 1B/8B decode shapes):
    //   cost = waves * (0.06 us per KiB of the CTA's weight bytes * eff(tile)
    //                   + 0.8 us per item + 2.1 us for the split-K handoff when parts > 1)
    // with waves = ceil(items / CTA slots).  eff is the relative cost of a weight byte,
    // set by how many rows share each staged x chunk (V): 1.4, 1.1, 1.0 for V = 1, 2, 4.
    // The per-item term is each row block's reduction, store and pipeline turn: without it
    // the model chose 16-row blocks for a lone 14336 x 4096 (12.4 us; 64-row blocks 10.7)
    // and 22016 x 4096 (17.1 us; 32-row blocks 14.8).
    // Parts of at least 2048 k are weighed first.  Only when that picks a split are the finer
    // counts, down to one 1024-k stage per part, weighed too, and they win a tie: once K is
    // split, finer parts measured faster (2048 x 8192: 64-row blocks in 8 parts 5.86 us,
    // 32-row blocks in 4 parts 6.07; 512 x 8192 4.43 against 4.87), while turning an unsplit
    // plan into a split did not (1000 x 7168 in 4 parts 5.05 us, unsplit 4.76).
    Tile tile = kTiles[0];
    int best_parts = 1;
    double best = 1e30;
    bool fine_taken = false;
    for (int pass = 0; pass < 2 && (pass == 0 || best_parts > 1); ++pass) {
        for (const Tile t : kTiles) {
            const int rbt = t.rows();
            if (stages_for(rbt) < 2) continue;
            const int64_t blocks_t = blocks_for(rbt);
            const double eff = t.V == 1 ? 1.4 : (t.V == 2 ? 1.1 : 1.0);
            for (int parts = 1; parts <= kGemvMaxParts; parts *= 2) {
                if (parts > 1 && (parts > kstages || !c.ws || !c.tickets ||
                                  (int64_t)parts * blocks_t * rbt > c.ws_floats ||
                                  blocks_t > c.ticket_count))
                    break;
                const bool fine = parts > 1 && kstages * 1024 / parts < 2048;
                if (fine != (pass == 1)) {
                    if (fine) break;
                    continue;
                }
                const int tpp = (kstages + parts - 1) / parts;
                const int64_t items = blocks_t * ((kstages + tpp - 1) / tpp);
                const double waves = (double)((items + slots - 1) / slots);
                const double kib = (double)rbt * tpp * kSRB / 1024.0;
                const double cost = waves * (0.06 * kib * eff + 0.8 + (parts > 1 ? 2.1 : 0.0));
                if (pass == 1 && !fine_taken ? cost <= best : cost < best * 0.999) {
                    best = cost, tile = t, best_parts = parts;
                    fine_taken = pass == 1;
                }
            }
        }
    }
    const int rb = tile.rows();
    GArgs a = {};
    a.x = p0.x;
    a.nmat = count;
    a.K = p0.K;
    a.kstages = kstages;
    a.gs_shift = gs_shift;
    a.stage_bytes = stage_bytes_for(rb, pc, esz, gs_shift, &a.scale_off, &a.stage_tx);
    a.stages = stages_for(rb);
    a.burst = 1;
    if (a.stages < 2) return cudaErrorNotSupported;
    const SmemLayout lay = smem_layout(a.stages, a.stage_bytes, kstages);
    a.x_off = lay.x_off;
    a.meta_off = lay.meta_off;
    a.bar_off = lay.bar_off;
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
            const cuuint32_t box[2] = {(cuuint32_t)(kSRB / 2), (cuuint32_t)rb};
            const cuuint32_t estr[2] = {1, 1};
            if (enc(&tm.w[i], CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint8_t*>(p.qweight),
                    dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return cudaErrorInvalidValue;
        }
        if (!pc) {
            const int64_t G = (p.K + p.group_size - 1) / p.group_size;
            const int gps = gs_shift >= 5 ? 1 : kSC >> gs_shift;
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
    // Fixed-point dp4a arithmetic where its per-CTA conversion of x pays off: each CTA
    // converts the x stages it uses once, which the cheaper inner loop repays from about
    // two row blocks per CTA on (measured on the decode tokens: vocabulary-sized heads
    // 15 %, 8B gate/up 5 % faster; one block per CTA, as in q/k/v, o and down, 5-50 %
    // slower).
    const bool x8 = a.items >= 2 * (int64_t)grid;
    if (x8_out) *x8_out = x8;
    if (!launch) return cudaSuccess;
    return dispatch_tile(tile, p0.even_high != 0, pc, p0.scale_f16 != 0, x8, tm, a, grid, lay.total,
                         c);
}

}  // namespace

cudaError_t gemv_tma_launch_group(const Problem* ps, int count, const LaunchCtx& c) {
    return gemv_group(ps, count, c, true, nullptr);
}

cudaError_t gemv_tma_launch(const Problem& p, const LaunchCtx& c) {
    return gemv_group(&p, 1, c, true, nullptr);
}

bool gemv_tma_fixed_point(const Problem& p, const LaunchCtx& c) {
    bool x8 = false;
    return gemv_group(&p, 1, c, false, &x8) == cudaSuccess && x8;
}

}  // namespace q4lin
