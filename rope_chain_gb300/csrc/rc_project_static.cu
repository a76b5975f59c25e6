// rc_kv_project_no_alloc: the K/V projection for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc or hand over a workspace: code that
// runs inside a host allocator's callback or a memory-pool hook, plug-ins
// whose host framework owns every device allocation, or service paths that
// must not touch the allocator at all once serving has started.  This entry
// point gives them the split-K projection anyway: its scratch is a
// file-scope device array that the library owns, so the caller passes only
// inputs and outputs.
//
// The array costs kScratchBytes (24 MiB) of device memory on every GPU that
// loads the library, until the process exits.  The first call on a device
// looks up the array's device address (cudaGetSymbolAddress, with that
// device current) and caches it; that first call should come before any
// stream capture.  All calls share it and it keeps the last
// call's contents, so two calls whose work overlaps on the GPU (different
// streams, or different host threads without ordering) race on it; order
// them on one stream.
#include "rope_chain.h"
#include "rc_internal.cuh"

#include <cstdio>
#include <mutex>

namespace {

// 24 MiB: on a 152-SM GB300 a split-K plan never needs more than
// (SMs) x 128 x 256 FP32 partials = 19.9 MB, and a persistent plan's tail
// split stays below that too (a host-only test sweeps the planner).
constexpr size_t kScratchBytes = RC_NO_ALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_project_scratch[kScratchBytes];

struct DeviceSlot {
    void *scratch = nullptr;     // device address of g_project_scratch
    int num_sms = 0;
};

std::mutex g_setup_mutex;
DeviceSlot g_slots[kMaxDevices];

// Once per device, with that device current: the array's device address
// (in host code the symbol is only a host-side stand-in) and the SM count.
cudaError_t device_setup(DeviceSlot **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    DeviceSlot &s = g_slots[dev];
    if (s.scratch == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_project_scratch);
        if (e != cudaSuccess)
            return e;
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return e;
        s.num_sms = n;
        s.scratch = p;
    }
    *out = &s;
    return cudaSuccess;
}

rc_status reject(rc_status s, const char *msg) {
    rc::set_last_error(msg);
    return s;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

}  // namespace

extern "C" {

rc_status rc_kv_project_no_alloc(const uint16_t *normed, const uint16_t *W, int32_t w_layout,
                                 uint16_t *out, int32_t L, int64_t T, int32_t D, int32_t N,
                                 cudaStream_t stream)
{
    // the checks rc_kv_project makes: sizes, layout, NULL, alignment, and
    // out overlapping normed or W
    const rc_status st = rc::check_project_call("rc_kv_project_no_alloc", normed, W, w_layout, out,
                                                L, T, D, N);
    if (st != RC_OK)
        return st;
    char msg[256];
    if (T == 0) {
        rc::set_last_error("");
        return RC_OK;
    }
    DeviceSlot *slot = nullptr;
    cudaError_t e = device_setup(&slot);
    if (e != cudaSuccess) {
        snprintf(msg, sizeof msg, "rc_kv_project_no_alloc: set-up failed: %s",
                 cudaGetErrorString(e));
        return reject(RC_ERR_CUDA, msg);
    }
    // No operand may lie inside the library's own scratch.
    if (overlaps(out, (size_t)L * T * N * 2, slot->scratch, kScratchBytes) ||
        overlaps(normed, (size_t)L * T * D * 2, slot->scratch, kScratchBytes) ||
        overlaps(W, (size_t)L * D * N * 2, slot->scratch, kScratchBytes))
        return reject(RC_ERR_INVALID_ARG,
                      "rc_kv_project_no_alloc: an operand overlaps the library's static scratch");
    // The same plan rc_kv_project makes with an unlimited workspace; a plan
    // whose partials do not fit the static array is refused, not shrunk.
    const rc::ProjectPlan plan = rc::plan_kv_project(L, T, D, N, slot->num_sms, SIZE_MAX);
    if (plan.workspace > kScratchBytes) {
        snprintf(msg, sizeof msg,
                 "rc_kv_project_no_alloc: these sizes need %zu bytes of split-K scratch; "
                 "the static scratch holds %zu",
                 plan.workspace, kScratchBytes);
        return reject(RC_ERR_UNSUPPORTED, msg);
    }
    // Nothing in the scratch has to start at zero when the call begins:
    // every FP32 partial the reduction reads is written earlier in the same
    // call, and the persistent kernel's tile counter (plans of eight rounds
    // of tiles or more) is zeroed by the call before its launch.
    const char *why = "launch";
    e = rc::launch_kv_project(normed, W, w_layout == RC_W_NK, out, L, T, D, N, plan,
                              static_cast<float *>(slot->scratch), stream, &why);
    if (e != cudaSuccess) {
        snprintf(msg, sizeof msg, "rc_kv_project_no_alloc: %s: %s", why, cudaGetErrorString(e));
        return reject(RC_ERR_CUDA, msg);
    }
    rc::set_last_error("");
    return RC_OK;
}

}  // extern "C"
