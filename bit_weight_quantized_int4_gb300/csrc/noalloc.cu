// noalloc.cu -- the decode GEMV for callers that cannot allocate device memory.
//
// q4lin_create allocates (a status word and the split-K scratch), so a caller that may not
// call cudaMalloc cannot make a handle.  This entry point needs none: it runs the same
// TMA-fed decode GEMV (M = 1), and its split-K scratch -- partial sums, per-row-block
// counters and a status word -- lives in the file-scope array below, which every GPU
// that loads the library holds until the process exits.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/q4lin.h"
#include "q4lin_internal.h"

namespace {

// Largest N accepted: 16384 output rows.  The GEMV's smallest row block is 16 rows, so at
// most 1024 row blocks (one counter each); K is split into at most 8 parts, each holding
// one partial sum per row of the row blocks (the last block may extend up to 63 rows past
// N, for 64-row blocks).
constexpr int64_t kMaxRows = 16384;
constexpr int64_t kRowPad = 128;
constexpr int64_t kPartialFloats = q4lin::kGemvMaxParts * (kMaxRows + kRowPad);
constexpr int64_t kTicketWords = 1024;
constexpr int64_t kStatusWords = 64;
constexpr int64_t kScratchWords = kPartialFloats + kTicketWords + kStatusWords;  // ~537 KB
static_assert(kTicketWords * q4lin::kGemvMinRowBlock >= kMaxRows,
              "one counter per row block of the smallest height");
static_assert(kRowPad >= q4lin::kGemvMaxRowBlock - 1,
              "partial sums cover the rows of the last, partly filled row block");

// The scratch.  In host code this name is a host-side stand-in, not a device address:
// the address comes from cudaGetSymbolAddress (scratch_address below).
static __device__ __align__(256) float g_scratch[kScratchWords];

constexpr int kMaxDevices = 64;
// Per device: the device address of g_scratch and the unique id of the CUDA context it
// was looked up in.  A device reset destroys the context (and the module holding the
// array); the next call sees a new context id and looks the address up again.
struct ScratchSlot {
    void* addr = nullptr;
    unsigned long long ctx_id = 0;
    bool have_id = false;
};
ScratchSlot g_slots[kMaxDevices];
std::mutex g_setup_mutex;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (false if there is none or the driver
// does not provide the query).
bool current_context_id(unsigned long long* id) {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
        cudaGetLastError();
    });
    CUcontext ctx = nullptr;
    return get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx &&
           get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_scratch on the current device `device`: looked up on the first call
// there, and again whenever the device's context has changed since.
q4lin_status_t scratch_address(int device, void** addr) {
    if (device < 0 || device >= kMaxDevices) return Q4LIN_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    ScratchSlot& s = g_slots[device];
    unsigned long long id = 0;
    const bool have_id = current_context_id(&id);
    if (!s.addr || !have_id || !s.have_id || s.ctx_id != id) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            s.addr = nullptr;
            return Q4LIN_ERR_CUDA;
        }
        s.addr = p;
        s.have_id = current_context_id(&s.ctx_id);  // the lookup made the context current
    }
    *addr = s.addr;
    return Q4LIN_OK;
}

bool overlaps(const void* a, int64_t abytes, const void* b, int64_t bbytes) {
    if (!a || !b || abytes <= 0 || bbytes <= 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + (uintptr_t)bbytes && b0 < a0 + (uintptr_t)abytes;
}

}  // namespace

extern "C" q4lin_status_t q4lin_run_static_scratch(const float* x, const uint8_t* qweight,
                                                   const void* scales, const float* bias,
                                                   float* out, int64_t N, int64_t K,
                                                   int64_t group_size, int scale_dtype,
                                                   void* stream) {
    // Argument checks (the same rules as q4lin_run with M = 1), before anything runs.
    if (N < 0 || K < 1 || group_size < 1) return Q4LIN_ERR_INVALID_ARG;
    if (scale_dtype != Q4LIN_SCALE_F32 && scale_dtype != Q4LIN_SCALE_F16)
        return Q4LIN_ERR_INVALID_ARG;
    if (N == 0) return Q4LIN_OK;
    if (!x || !qweight || !scales || !out) return Q4LIN_ERR_INVALID_ARG;
    if (N > kMaxRows) return Q4LIN_ERR_TOO_LARGE;
    const int64_t esize = scale_dtype == Q4LIN_SCALE_F16 ? 2 : 4;
    const int64_t G = (K + group_size - 1) / group_size;
    if (K > (int64_t)1 << 40 || G * N > ((int64_t)1 << 50)) return Q4LIN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(x) % 4 || reinterpret_cast<uintptr_t>(out) % 4 ||
        (bias && reinterpret_cast<uintptr_t>(bias) % 4) ||
        reinterpret_cast<uintptr_t>(scales) % esize)
        return Q4LIN_ERR_INVALID_ARG;
    const int64_t ob = N * 4;
    if (overlaps(out, ob, x, K * 4) || overlaps(out, ob, qweight, N * ((K + 1) / 2)) ||
        overlaps(out, ob, scales, G * N * esize) || overlaps(out, ob, bias, bias ? N * 4 : 0))
        return Q4LIN_ERR_INVALID_ARG;

    q4lin::Problem p;
    p.x = x;
    p.qweight = qweight;
    p.scales = scales;
    p.bias = bias;
    p.out = out;
    p.M = 1;
    p.N = N;
    p.K = K;
    p.group_size = group_size;
    p.scale_f16 = scale_dtype == Q4LIN_SCALE_F16;
    p.even_high = 0;
    if (!q4lin::gemv_tma_eligible(p)) return Q4LIN_ERR_UNSUPPORTED;

    int device = 0, sms = 0, smem = 0;
    if (cudaGetDevice(&device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) !=
            cudaSuccess) {
        cudaGetLastError();
        return Q4LIN_ERR_CUDA;
    }
    void* scratch = nullptr;
    q4lin_status_t st = scratch_address(device, &scratch);
    if (st != Q4LIN_OK) return st;
    float* partials = static_cast<float*>(scratch);
    int* tickets = reinterpret_cast<int*>(partials + kPartialFloats);
    int* status = tickets + kTicketWords;

    q4lin::LaunchCtx c;
    c.stream = static_cast<cudaStream_t>(stream);
    c.sm_count = sms;
    c.max_smem_optin = smem;
    c.pdl = 0;
    c.status_word = status;
    c.wait_limit_ns = 2000000000LL;
    c.tc_skip_first_copy = 0;
    c.ws = partials;
    c.ws_floats = kPartialFloats;
    c.tickets = tickets;
    c.ticket_count = kTicketWords;
    // The counters must start at zero; the array keeps whatever the last call left.
    if (cudaMemsetAsync(tickets, 0, (kTicketWords + kStatusWords) * sizeof(int), c.stream) !=
        cudaSuccess) {
        cudaGetLastError();
        return Q4LIN_ERR_CUDA;
    }
    cudaError_t err = q4lin::gemv_tma_launch(p, c);
    if (err == cudaSuccess) err = cudaGetLastError();
    return err == cudaSuccess ? Q4LIN_OK : Q4LIN_ERR_CUDA;
}
