// ctr_internal.h -- plan state and kernel parameter blocks shared by the library's
// translation units (host and device).  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/ctr.h"
#include "per_device.h"

namespace ctr {

// Tile shape of the tensor-core GEMM: 128 rows (TMEM lanes) x BN columns.  The packed
// operands' K extents are multiples of 128 bytes (64 bf16 or 32 fp32); the kernel moves K
// in slices of 128 bytes (see gemm_slice_bytes).
constexpr int kBM = 128;
constexpr int kBKBytes = 128;

enum class Prec : int { BF16 = 0, F32 = 1, F16 = 2 };
constexpr bool is_16bit(Prec p) { return p != Prec::F32; }

// I/O element type of a plan: the ctr_dtype code (CTR_F32, CTR_BF16, CTR_F16).
enum IoType : int { IO_F32 = 0, IO_BF16 = 1, IO_F16 = 2 };
enum EpiMode : int { EPI_POLYPHASE = 0, EPI_RAW = 1 };

// Output-stage variants (chosen per plan on the host; see epilogue.cuh).
enum EpiKind : int {
    EPI_KIND_GENERIC = 0,
    EPI_KIND_1D_S1, EPI_KIND_1D_S2, EPI_KIND_1D_S4, EPI_KIND_1D_S8, EPI_KIND_1D_S16,
    EPI_KIND_1D_S32, EPI_KIND_2D_S2x2, EPI_KIND_2D_S4x4, EPI_KIND_1D_LARGE
};

// Output mapping of a GEMM result D[n, r] (shared by the fused epilogue and the split-K
// reduce).  Everything is in the 2-D form; 1-D plans have sy = 1, py = 0, Py = Qvy = 1,
// Hout = 1.
//   position n -> b = n / (Py*Px), qy = (n / Px) % Py, qx = n % Px (valid when b < B,
//                 qy < Qvy, qx < Qvx)
//   row r      -> oc = r / S_pad, j = r % S_pad (phase, valid when j < S), jy = j / sx,
//                 jx = j % sx
//   output     -> y[b, oc, sy*qy + jy - py, sx*qx + jx - px] when inside [0, Hout) x [0, Wout)
struct EpiParams {
    int S, S_pad, sx, sy, px, py;
    int64_t Px, Py, Qvx, Qvy;
    int64_t B, C_out, Hout, Wout;
    const void *bias;   // [C_out] in the I/O dtype, or nullptr
    void *y;
    int io;             // IoType of bias and y
    int act;            // ctr_act
    float slope;
    int kind;           // EpiKind
    int store_bytes;    // width of the aligned vector stores of interior runs (16, 8, 4, 2)
    int shift2;         // sx = 2 runs at odd columns stored as pairs across lanes (epilogue.cuh)
    // Chained output (out_staged = 1): y is the next plan's staged input, channels-last rows
    // of ys_cpad channels, output (oy, ox) of batch b at row (b*ys_Py + oy + ys_hy)*ys_Px +
    // ox + ys_hx; fp32 as the tf32 and cross planes (ptx::split_x), ys_lo elements apart.
    // The same output path writes a channels-last (NHWC) y: then ys_* describe y itself (no
    // halos, C_out channels per row) and ys_tf32 = 0 stores plain values.
    int out_staged;
    int64_t ys_Px, ys_Py, ys_hx, ys_hy, ys_cpad, ys_lo;
    int ys_tf32;        // fp32 values as the tf32 and cross planes (a staged operand)
    // Phase-major rows (pm_tc > 0, chained producers only): inside each tile of
    // pm_tc * S_pad rows, row j * pm_tc + c is phase j of the tile's channel c, so a 32-row
    // chunk holds whole channel runs of one (or a few) phases.
    int pm_tc;
};

// The tensor-core GEMM D[n, r] = sum_k Xs[n + shift(k), k] * A[r, k]: n runs over staged
// phase positions (TMEM lanes, 128 per tile), r over packed weight rows (TMEM columns, BN per
// tile).
struct GemmParams {
    int num_p_tiles, num_r_tiles, splits;
    int64_t num_tiles;
    // K counts below are in the kernel's slices (gemm_slice_bytes of the plan's dtype and BN).
    int kb_total;       // K slices over all taps
    int kb_per_tap;     // K slices per tap (C_in_pad * esize / slice bytes)
    int kb_group;       // K slices per tensor-core accumulation group (see gemm_tc.cu)
    int mx;             // taps along x: tap g -> (uy, ux) = (g / mx, g % mx)
    int64_t Px;         // position shift of one tap step along y
    int64_t shift0;     // staged row of tap 0 relative to the position (rb_y*Px + rb_x)
    int epi_mode;
    EpiParams epi;
    float *raw;         // EPI_RAW: D goes to raw[z][n][r] with leading dimension raw_ld
    int64_t raw_ld;
    int64_t raw_split_stride;
    uint32_t *status;   // device status word (bit flags of bounded waits that gave up)
    uint64_t wait_limit_ns;
    // Pipeline layout in shared memory (set by the host for the launch, see gemm_tc.cuh):
    // nstages stages of stage_bytes from a 1024-byte-aligned base, the barriers at bar_off.
    int nstages, stage_bytes, bar_off, smem_bytes;
    // Shared-X mode (1-D, 16-bit operands): a stage holds one X box of x_rows staged rows
    // (128 positions plus the taps' shifts) for one channel slice, and every tap's MMA reads
    // it through a descriptor that starts tap rows further down; the stage also holds the
    // taps' weight slices, unless the whole weight tile stays resident (wres) at wres_off.
    int xshare, x_rows, wres, wres_off;
    // X-ring mode (fp32 256-row tiles with four or more taps along x): the X boxes (x_rows rows,
    // both operand planes) of one channel slice and tap row sit in a ring of two slots at
    // xring_off, read by that row's mx taps through row-shifted descriptors; the weight
    // boxes (one plane of one tap) stream through the nstages-stage ring.  K is walked as
    // slices s = kc * (my * mx) + tap, so a split-K unit covers whole channel slices.
    int xring, xring_off, my;
};

// Shared-memory layout of one GEMM instantiation (gemm_tc.cu): default stage count and
// bytes, the dynamic shared-memory budget of one CTA, and the bytes of one K slice of a
// 128-position X box and of a block_n-row weight box (one plane).
struct GemmLayout {
    int stages, stage_bytes, smem_budget, slice_bytes, x_box_bytes, w_box_bytes, planes;
};
GemmLayout gemm_layout(Prec prec, int block_n);
constexpr int kGemmMaxStages = 12;
constexpr int kGemmBarBytes = 512;

// Status-word bits set by device code.
constexpr uint32_t kStatusTimeoutProducer = 1u << 0;
constexpr uint32_t kStatusTimeoutMma = 1u << 1;
constexpr uint32_t kStatusTimeoutEpilogue = 1u << 2;
constexpr uint32_t kStatusTimeoutDrain = 1u << 3;

}  // namespace ctr

struct ctr_plan_s {
    // Geometry in the 2-D form (index 0 = y/height, 1 = x/width).
    int ndim;
    int64_t B, C_in, C_out;
    int64_t in[2], k[2], s[2], p[2], op[2], out[2];
    int64_t dil[2];     // dilation (ctr_plan_set_dilation; 1 = none)
    int64_t pe[2];      // back pad (ctr_plan_set_pads; p is the front pad; default pe = p)
    int nhwc;           // ctr_plan_set_layout: x and y channels last
    int streaming;      // ctr_plan_set_streaming: carries the last m - 1 input frames
    int stream_saved_path;  // the forced path before streaming was turned on (restored after)
    int stream_ready;   // the carried frames were zeroed (ctr_plan_stream_reset)
    int dtype;
    int act;
    float slope;
    int path;           // chosen ctr_path (never AUTO)
    int forced_path;
    int forced_split;
    int forced_bn;      // 0 = automatic phase-row tile
    int64_t groups;     // ctr_plan_set_groups (1 = dense)
    int prepared;       // ctr_prepack_weight ran (status word allocated)
    int num_sms;

    // Tensor-core GEMM geometry (polyphase and col2im paths).  Per dimension the GEMM's
    // phase position Q and tap v read staged input row Q + rb + v, i.e. input index
    // Q + rb - hf + v; D[Q, (oc, j)] lands at output s*Q + j - ep.
    //   unpadded phases (the pages' form): Q indexes the unpadded output's phases, the
    //     packed tap of (v, j) is s*(mk-1-v) + j, hf = mk - 1, rb = 0, ep = p (the padding
    //     slice is applied at the store);
    //   output phases: Q indexes the output's own phases; with p = s*pq + pm the packed tap
    //     of (v, j) is s*(mk-1-v) + j + pm (zero outside the kernel), one more tap when
    //     pm > 0, hf = max(0, mk-1-pq), rb = max(0, pq-(mk-1)), ep = 0: every output run
    //     starts at s*Q, so the stores are aligned whatever the padding.
    int64_t m[2];       // GEMM taps per dim (polyphase), 1 for col2im
    int64_t mk[2];      // phase taps of the kernel, ceil(dilated extent / s)
    int64_t pm[2];      // padding remainder folded into the packed taps (output phases)
    int64_t hf[2];      // zero rows in front of the input in the staged layout
    int64_t rb[2];      // staged row of tap 0 relative to the phase position
    int64_t ep[2];      // output offset of the phase map (padding sliced at the store)
    int out_phases;     // 1: output phases, 0: unpadded phases
    int forced_origin;  // ctr_plan_set_phase_origin (CTR_PHASE_AUTO = choose)
    int64_t Qv[2];      // valid phase columns per dim
    int64_t P[2];       // staged pitch per dim (with halos)
    int S, S_pad;       // phases (polyphase) or taps (col2im) per output channel, padded
    int64_t C_in_pad;
    int64_t M_rows, M_pad;
    int64_t K_total;    // GEMM K = taps * C_in_pad
    int64_t N_total;    // GEMM columns = B * P[0] * P[1]
    int block_n;        // phase rows per tile (MMA N): 64, 128 or 256
    int splits;
    int kb_group;       // 128-byte K slices per accumulation group; >= all slices = no flush
    int num_p_tiles;    // tiles of 128 staged positions
    int num_r_tiles;    // tiles of block_n packed weight rows
    int64_t num_tiles;

    size_t packed_bytes;
    size_t ws_bytes_needed;
    size_t ws_off_stage;   // staged x (channels-last with halos)
    size_t ws_stage_bytes;
    size_t ws_off_raw;     // split-K partials or the col2im column buffer
    size_t ws_raw_bytes;
    size_t ws_off_state;   // streaming: the last m - 1 staged input frames of each batch item
    size_t ws_state_bytes;
    void *ws;
    size_t ws_bytes;

    // Chaining (ctr_plan_chain): this plan's output feeds chain_next's staged input.
    ctr_plan_s *chain_next;
    ctr_plan_s *chain_prev;
    void *chain_zeroed_ws;  // workspace whose staged buffer was zeroed for chained input
    int row_pm;             // packed rows phase-major within each tile (set for chained output)
    uint32_t *d_status;
    int status_device;
    uint64_t wait_limit_ns;
    cudaEvent_t ev_before, ev_after;   // optional timing events around the main kernel
};

namespace ctr {

// Launch with programmatic stream serialization: the kernel may be scheduled while the
// previous kernel of the stream is still running, so it must call ptx::griddep_wait() before
// its first global memory access; its launch and prologue then overlap the previous
// kernel's tail instead of following its completion.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// The current device's ordinal, or -1 when it cannot be read (set-up then runs every time).
inline int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return dev;
}

// Prefer the largest shared-memory carveout for a kernel (once per kernel and device: the
// attribute belongs to the current device's context), so that consecutive kernels of a
// forward pass do not reconfigure the SMs between them.
template <auto Kernel>
cudaError_t prefer_max_smem() {
    static PerDeviceOnce once;
    return once.run(current_device(), cudaSuccess, [] {
        return cudaFuncSetAttribute(Kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                    (int)cudaSharedmemCarveoutMaxShared);
    });
}

// Launch wrappers (each returns the cudaGetLastError() of its launches).
cudaError_t launch_gather(const ctr_plan_s *pl, const void *x, const void *w, const void *bias,
                          void *y, cudaStream_t st);
cudaError_t launch_copy_weight(const ctr_plan_s *pl, const void *w, void *w_packed,
                               cudaStream_t st);
cudaError_t launch_prepack(const ctr_plan_s *pl, const void *w, void *w_packed, cudaStream_t st);
cudaError_t launch_stage_x(const ctr_plan_s *pl, const void *x, void *xs, cudaStream_t st);
// The same staged operand from a channels-last (NHWC) x.
cudaError_t launch_stage_nhwc(const ctr_plan_s *pl, const void *x, void *xs, cudaStream_t st);
// Streaming plans: move the carried input frames into the staged input's leading halo and
// this call's last m - 1 frames into the carried state.
cudaError_t launch_stream_state(const ctr_plan_s *pl, void *xs, void *state, cudaStream_t st);
// Most frames a streaming plan carries (m - 1).
constexpr int kMaxStreamCarry = 16;
cudaError_t launch_splitk_reduce(const ctr_plan_s *pl, const float *raw, const EpiParams &ep,
                                 int64_t raw_ld, int64_t split_stride, cudaStream_t st);
// Leading dimension (floats) and split stride of the raw [z][n][r] buffer of a plan.
int64_t raw_ld_of(const ctr_plan_s *pl);
int64_t raw_split_stride_of(const ctr_plan_s *pl);
cudaError_t launch_col2im(const ctr_plan_s *pl, const float *col, int64_t col_ld,
                          const void *bias, void *y, cudaStream_t st);
cudaError_t launch_fill_bias(const ctr_plan_s *pl, const void *bias, void *y, cudaStream_t st);
// One input channel per group (groups = C_in, C_out a multiple of it): the depthwise kernel,
// for the x-direction kernel sizes and strides it is compiled for.
bool depthwise_supported(const ctr_plan_s *pl);
cudaError_t launch_depthwise(const ctr_plan_s *pl, const void *x, const void *w, const void *bias,
                             void *y, cudaStream_t st);
cudaError_t launch_gemm_tc(const ctr_plan_s *pl, const CUtensorMap *maps, const GemmParams &gp,
                           cudaStream_t st);

// 2-D tiled tensor map over a row-major [rows][inner] operand matrix of IoType io, box
// [box_rows][box_bytes], swizzled at box_bytes (128 or 64), zero fill (api.cu).
bool encode_2d(CUtensorMap *map, const void *base, int io, uint64_t inner, uint64_t rows,
               uint32_t box_rows, int box_bytes);

// Output mapping of a tensor-core plan (api.cu).
EpiParams make_epi(const ctr_plan_s *pl, const void *bias, void *y);

// The GEMM's shared-memory pipeline for a plan (api.cu): stage count and size, barrier
// offset, the shared-X and resident-weight modes.
void set_pipeline_layout(const ctr_plan_s *pl, GemmParams *gp);

// Staging (skipped when staged_in: a chained producer already wrote the staged input), GEMM
// and reduce/col2im of a tensor-core plan with explicit scratch (api.cu).  With chained_to
// set, the output goes to that plan's staged input instead of y.
cudaError_t run_tc_path(const ctr_plan_s *pl, const void *x, const void *w_packed,
                        const void *bias, void *y, char *ws, uint32_t *status,
                        cudaEvent_t ev_before, cudaEvent_t ev_after, cudaStream_t st,
                        const ctr_plan_s *chained_to = nullptr, bool staged_in = false);

// Two chained 1-D layers in one kernel (fused_pair.cu): whether a plan and the plan it is
// chained to qualify, and the launch (xs: the first plan's staged input).
bool fused_pair_supported(const ctr_plan_s *a);
cudaError_t launch_fused_pair(const ctr_plan_s *a, const void *xs, const void *wa_packed,
                              const void *bias_a, const void *wb_packed, const void *bias_b,
                              void *y, cudaStream_t st);

// Counter of launched kernels (monotonic, process-wide).
void count_launches(uint64_t n);
// Device address of ctr_forward_noalloc's status word on the current device, or nullptr when
// no allocation-free call has looked up its scratch on this device yet (noalloc.cu).
uint32_t *noalloc_status_word();
// Records a caller's timing event (an external event node under stream capture).
cudaError_t record_timing(cudaEvent_t ev, cudaStream_t st);

// Bytes of dynamic shared memory a GEMM instantiation uses.
size_t gemm_smem_bytes(Prec prec, int block_n);

// Width in bytes of the K slices a GEMM instantiation loads: 128, one 128-byte swizzle row.
// A TMA box row costs about the same whatever its width, so 128-byte rows move more bytes per
// SM than 64-byte ones (measured on GB300: 51 against 33 B per clock with four 48 KB stages
// in flight).  fp32 256-row tiles put one operand plane in each stage (gemm_tc.cuh), which
// keeps four stages for operands that come from HBM.
constexpr int gemm_slice_bytes(Prec, int) { return 128; }

// Largest phase-row tile whose accumulation groups fit the epilogue's registers.
constexpr int kMaxGroupedBN = 256;

}  // namespace ctr
