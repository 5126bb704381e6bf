// moe_plan_noalloc: the route-metadata stage without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they need the plan: a
// runtime that forbids cudaMalloc on its execution path (allocation would synchronise the
// device or break its memory accounting), or a plugin host that hands an operator its
// inputs and outputs but no scratch buffer. For them this entry point keeps its scratch in
// one file-scope device array instead of the workspace.
//
// The array is a fixed kNoallocScratchBytes (1,590,272 bytes) that every GPU which loads the
// library holds until the process exits. Every call shares it and it keeps the last call's
// contents; the launches clear what must start at zero (the header and the per-expert claim
// counters) themselves. Calls that overlap on the GPU -- on different streams, or from
// different host threads without ordering -- race on the array and give wrong plans.
//
// The kernels are the ones moe_plan launches; only the storage differs.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "internal.h"

namespace moe {

namespace {

constexpr int kNoallocMaxIds = 1 << 16;     // T*K routes per call
constexpr int kNoallocMaxExperts = 1024;
constexpr int kNoallocMaxPoolRows = kNoallocMaxIds + kNoallocMaxExperts * (kTileRows - 1);

// Regions (int32 units), in this order; the header and the claim counters must be adjacent
// because the route launch clears them with one memset.
constexpr int kOffHdr = 0;
constexpr int kOffClaim = kOffHdr + 64;
constexpr int kOffCounts = kOffClaim + kNoallocMaxExperts;
constexpr int kOffOffsets = kOffCounts + kNoallocMaxExperts;
constexpr int kOffPad = kOffOffsets + kNoallocMaxExperts + 64;
constexpr int kOffTiles = kOffPad + kNoallocMaxExperts + 64;
constexpr int kOffPos = kOffTiles + kNoallocMaxExperts + 64;
constexpr int kOffRowSrc = kOffPos + kNoallocMaxIds;
constexpr int kOffSlotRow = kOffRowSrc + kNoallocMaxIds;
constexpr int kOffPoolSrc = kOffSlotRow + kNoallocMaxIds;
constexpr int kNoallocScratchInts = kOffPoolSrc + kNoallocMaxPoolRows;
constexpr size_t kNoallocScratchBytes = sizeof(int32_t) * (size_t)kNoallocScratchInts;
static_assert(kNoallocScratchBytes == 1590272, "the size stated in include/moe_ffn.h");

// The scratch itself. In host code this name is a host-side stand-in, not a device address:
// the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) int32_t g_plan_scratch[kNoallocScratchInts];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
struct ScratchAddr {
    unsigned long long ctx_id;  // the context the address belongs to (IDs are never reused)
    int32_t* ptr;
};
ScratchAddr g_scratch[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// The unique ID of the calling thread's current context, through the driver entry points (no
// link-time dependency on libcuda).
cudaError_t current_context_id(unsigned long long* id) {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    if (!get_current || !get_id) return cudaErrorNotSupported;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorDeviceUninitialized;
    return get_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorDeviceUninitialized;
}

// Device address of g_plan_scratch in the current context of the current device. It is looked up
// once per device and looked up again when that device's context changes (after cudaDeviceReset
// the old address is no longer mapped). With no context current yet, the lookup itself makes the
// device's primary context current, and its ID is read afterwards.
cudaError_t scratch_address(int32_t** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    unsigned long long ctx = 0;
    const bool have_ctx = current_context_id(&ctx) == cudaSuccess;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!have_ctx || !g_scratch[dev].ptr || g_scratch[dev].ctx_id != ctx) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_plan_scratch);
        if (e != cudaSuccess) return e;
        if ((e = current_context_id(&ctx)) != cudaSuccess) return e;
        g_scratch[dev] = {ctx, static_cast<int32_t*>(ptr)};
    }
    *out = g_scratch[dev].ptr;
    return cudaSuccess;
}

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" MOE_API moe_status moe_plan_noalloc(const int32_t* topk_ids, const moe_dims* d, int32_t* counts,
                                               int32_t* offsets, int32_t* row_src, moe_stream_t stream) {
    // the same dims checks as moe_plan (which takes them in A16W16 mode), then this call's array limits
    if (!dims_ok(d, MOE_A16W16) || d->num_experts + d->num_shared_experts > kNoallocMaxExperts)
        return MOE_ERR_INVALID_ARG;
    const int E = d->num_experts + d->num_shared_experts, K = d->topk + d->num_shared_experts;
    const int64_t ids = (int64_t)d->num_tokens * K;  // the shared experts' slots included
    if (ids > kNoallocMaxIds) return MOE_ERR_INVALID_ARG;
    if (!counts || !offsets || (ids > 0 && (!topk_ids || !row_src))) return MOE_ERR_INVALID_ARG;
    int32_t* s = nullptr;
    if (scratch_address(&s) != cudaSuccess) return MOE_ERR_CUDA;
    Plan p{};
    p.T = d->num_tokens;
    p.H = d->hidden;
    p.I = d->intermediate;
    p.E = E;
    p.K = K;
    p.Er = d->num_experts;
    p.Kr = d->topk;
    p.mode = MOE_A16W16;
    p.pool_rows = ids + std::min<int64_t>(E, ids) * (kTileRows - 1);
    p.hdr = s + kOffHdr;
    p.claim = s + kOffClaim;
    p.counts = s + kOffCounts;
    p.offsets = s + kOffOffsets;
    p.pad_off = s + kOffPad;
    p.tile_off = s + kOffTiles;
    p.pos = s + kOffPos;
    p.row_src = s + kOffRowSrc;
    p.slot_row = s + kOffSlotRow;
    p.pool_src = s + kOffPoolSrc;
    cudaError_t e = launch_route(p, topk_ids, counts, offsets, row_src, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
