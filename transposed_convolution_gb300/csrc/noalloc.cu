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

extern "C" ctr_status ctr_forward_noalloc(ctr_plan_t pl, const void *x, const void *w,
                                          const void *bias, void *y, void *stream) {
    if (!pl) return CTR_ERR_INVALID_ARG;
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
    void *w_packed = scratch + packed_off;
    if (ctr::launch_prepack(pl, w, w_packed, st) != cudaSuccess) return CTR_ERR_CUDA;
    if (pl->N_total == 0)
        return ctr::launch_fill_bias(pl, bias, y, st) == cudaSuccess ? CTR_OK : CTR_ERR_CUDA;

    char *ws = scratch + ws_off;
    void *xs = ws + pl->ws_off_stage;
    float *raw = pl->ws_raw_bytes ? reinterpret_cast<float *>(ws + pl->ws_off_raw) : nullptr;
    if (ctr::launch_stage_x(pl, x, xs, st) != cudaSuccess) return CTR_ERR_CUDA;

    const bool bf16 = pl->dtype == CTR_BF16;
    const int es = bf16 ? 2 : 4;
    const size_t a_plane = (size_t)pl->M_pad * pl->K_total * es;
    const size_t b_plane = (size_t)pl->N_total * pl->C_in_pad * es;
    CUtensorMap maps[4];
    bool ok = ctr::encode_2d(&maps[0], w_packed, bf16, pl->K_total, pl->M_pad, ctr::kBM) &&
              ctr::encode_2d(&maps[1], xs, bf16, pl->C_in_pad, pl->N_total, pl->block_n);
    if (!bf16) {
        ok = ok &&
             ctr::encode_2d(&maps[2], static_cast<char *>(w_packed) + a_plane, false, pl->K_total,
                            pl->M_pad, ctr::kBM) &&
             ctr::encode_2d(&maps[3], static_cast<char *>(xs) + b_plane, false, pl->C_in_pad,
                            pl->N_total, pl->block_n);
    } else {
        maps[2] = maps[0];
        maps[3] = maps[1];
    }
    if (!ok) return CTR_ERR_CUDA;

    ctr::GemmParams gp{};
    gp.num_m_tiles = pl->num_m_tiles;
    gp.num_n_tiles = pl->num_n_tiles;
    gp.splits = pl->splits;
    gp.num_tiles = pl->num_tiles;
    gp.kb_total = (int)(pl->K_total * es / ctr::kBKBytes);
    gp.kb_per_tap = (int)(pl->C_in_pad * es / ctr::kBKBytes);
    gp.kb_group = pl->kb_group;
    gp.mx = (int)pl->m[1];
    gp.Px = pl->P[1];
    const bool fused = pl->path == CTR_PATH_POLYPHASE && pl->splits == 1;
    gp.epi_mode = fused ? ctr::EPI_POLYPHASE : ctr::EPI_RAW;
    gp.epi = ctr::make_epi(pl, bias, y);
    gp.raw = raw;
    gp.raw_ld = (int64_t)pl->num_n_tiles * pl->block_n;
    gp.raw_split_stride = pl->M_pad * gp.raw_ld;
    gp.status = status;
    gp.wait_limit_ns = pl->wait_limit_ns;
    if (ctr::launch_gemm_tc(pl, maps, gp, st) != cudaSuccess) return CTR_ERR_CUDA;
    if (pl->path == CTR_PATH_POLYPHASE && !fused) {
        if (ctr::launch_splitk_reduce(pl, raw, gp.epi, gp.raw_ld, gp.raw_split_stride, st) !=
            cudaSuccess)
            return CTR_ERR_CUDA;
    } else if (pl->path == CTR_PATH_COL2IM) {
        if (ctr::launch_col2im(pl, raw, gp.raw_ld, bias, y, st) != cudaSuccess) return CTR_ERR_CUDA;
    }
    return CTR_OK;
}
