// noalloc.cu -- ctr_forward_noalloc: the forward pass for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc at all: code running inside a host framework whose
// allocator owns every device byte, code that must not allocate while a CUDA graph is being
// captured, or real-time audio callbacks where an allocation may block.  For them this
// entry point takes its scratch -- the packed weight, the staged input, the split-K
// partials and a status word -- from one file-scope device array of fixed size instead of
// a caller-bound workspace, and packs the weight itself on every call.  The caller passes
// only the plan, the inputs and the output.
//
// The array is a static __device__ object: the CUDA driver reserves it on every device that
// loads this library's module and keeps it until the process exits.  Its host-side name is
// only a stand-in; the device address comes from cudaGetSymbolAddress, once per device, with
// that device current, on the first call on that device.
#include <mutex>

#include "ctr_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr size_t kStatusBytes = 256;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices];

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device address of the scratch array on the current device (looked up once per device).
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

namespace ctr {
uint32_t *noalloc_status_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    return static_cast<uint32_t *>(g_scratch_addr[dev]);
}
}  // namespace ctr

extern "C" ctr_status ctr_forward_noalloc(ctr_plan_t pl, const void *x, const void *w,
                                          const void *bias, void *y, void *stream) {
    if (!pl || pl->chain_next) return CTR_ERR_INVALID_ARG;   // chaining needs bound workspaces
    if (pl->streaming) return CTR_ERR_UNSUPPORTED;   // carried frames need a bound workspace
    if (!w || !y || (!x && pl->B * pl->C_in * pl->in[0] * pl->in[1] > 0))
        return CTR_ERR_INVALID_ARG;
    if ((x && !aligned16(x)) || !aligned16(w) || !aligned16(y) || (bias && !aligned16(bias)))
        return CTR_ERR_MISALIGNED;
    const bool tc = pl->path == CTR_PATH_POLYPHASE || pl->path == CTR_PATH_COL2IM;
    const size_t packed_off = kStatusBytes;
    const size_t ws_off = packed_off + align256(tc ? pl->packed_bytes : 0);
    const size_t need = ws_off + (tc ? pl->ws_bytes_needed : 0);
    if (need > kNoAllocScratchBytes) return CTR_ERR_NO_WORKSPACE;
    if (pl->B == 0) return CTR_OK;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    void *base = nullptr;
    if (scratch_address(&base) != cudaSuccess) return CTR_ERR_CUDA;
    char *scratch = static_cast<char *>(base);
    uint32_t *status = reinterpret_cast<uint32_t *>(scratch);
    // The array keeps the previous call's contents: the status word must start at zero;
    // every other region is written in full before it is read.
    if (cudaMemsetAsync(status, 0, sizeof(uint32_t), st) != cudaSuccess) return CTR_ERR_CUDA;

    if (pl->path == CTR_PATH_GATHER) {
        // The gather kernel reads the weight in its torch layout; no scratch is needed.
        return ctr::launch_gather(pl, x, w, bias, y, st) == cudaSuccess ? CTR_OK : CTR_ERR_CUDA;
    }
    if (pl->path == CTR_PATH_DEPTHWISE)   // so does the depthwise kernel
        return ctr::launch_depthwise(pl, x, w, bias, y, st) == cudaSuccess ? CTR_OK : CTR_ERR_CUDA;
    void *w_packed = scratch + packed_off;
    if (ctr::launch_prepack(pl, w, w_packed, st) != cudaSuccess) return CTR_ERR_CUDA;
    if (pl->N_total == 0)
        return ctr::launch_fill_bias(pl, bias, y, st) == cudaSuccess ? CTR_OK : CTR_ERR_CUDA;

    const cudaError_t e = ctr::run_tc_path(pl, x, w_packed, bias, y, scratch + ws_off, status,
                                           nullptr, nullptr, st);
    return e == cudaSuccess ? CTR_OK : CTR_ERR_CUDA;
}
