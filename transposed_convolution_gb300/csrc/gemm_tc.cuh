// gemm_tc.cuh -- the hot kernel: a persistent, warp-specialised implicit GEMM on the 5th-
// generation tensor cores (tcgen05 + TMEM), fed by TMA.  Instantiated in gemm_tc.cu (output
// in the torch layout) and gemm_tc_chain.cu (output into the next plan's staged input), two
// translation units that compile in parallel.
//
//   D[n, r] = sum over taps g and input channels ic of Xs[n + shift(g), ic] * A[r, g*C_in_pad + ic]
//
// For the polyphase path ("[XNNPACK] Lower dense transposed convs as one polyphase conv +
// depth to space", Summary) A is the phase-major prepacked weight, Xs the input staged
// channels-last with m - 1 zero positions on each side, and shift(g) = uy*Px + ux the tap
// offset, so that the m (or mH*mW) taps of the stride-1 phase convolution are m shifted TMA
// boxes of the same staged input: the zero halo is the convolution's padding m - 1.  For
// the col2im path ("[WebGPU] optimizations for audio models", ConvTranspose commit) there
// is one tap and D is the column buffer X[M, C_in] x W[C_in, k*C_out], transposed.
//
// The MMA's M dimension is the phase position n (128 per tile: TMEM lanes) and its N
// dimension the packed weight row r (BN = 64, 128 or 256 per tile: TMEM columns), so each
// epilogue thread owns one output position and writes its phases as contiguous runs.
//
// Warp roles (320 threads, one CTA per SM -- two for bf16 tiles of 64 rows -- persistent over
// output tiles):
//   warp 0      one lane issues TMA loads of Xs and A K-slices into a ring of stages;
//   warp 1      allocates TMEM; one lane issues tcgen05.mma into one of several TMEM
//               accumulators (128 lanes x BN fp32 columns) and commits to mbarriers;
//   warps 2..9  the epilogue: tcgen05.ld of the accumulator, then either the fused polyphase
//               output stage (bias, activation, interleave, slice; epilogue.cuh) or a raw
//               fp32 store of D (split-K partials, col2im columns).  A warp may read only
//               the TMEM lane quarter (warp id mod 4); two warps share each quarter, one
//               taking the first BN/2 columns and the other the rest.
// Several accumulators let the epilogue of tile i overlap the MMAs of tile i + 1.
//
// fp32 I/O: each operand value v is split as hi = tf32(v) and lo = v - hi, the idea of Ootomo
// and Yokota, "Recovering single precision accuracy from Tensor Cores while surpassing the
// FP32 theoretical peak performance" (IJHPCA 2022), who issue hi*hi, hi*lo and lo*hi as three
// tf32 MMAs.  Here the two cross products are one kind::f16 MMA on bf16 pairs instead: every
// 32-byte K step issues a bf16 MMA (16 bf16 = 8 K elements x (hi, lo), from the second
// operand plane; ptx::split_x / split_w) and a tf32 MMA of hi*hi (8 K elements, first plane)
// into the same fp32 accumulator.  The bf16 MMA of K 16 takes the tensor pipe as long as the
// tf32 MMA of K 8, so a K step costs two tf32 MMA times instead of three, and the
// shared-memory operand reads drop by the same third.  The bf16 roundings of the cross terms
// (each below 2^-11 of the product) cost at most about 2^-17 of a product's value, well
// inside fp32 I/O's accuracy bound.
//
// Stage layouts.  By default a stage holds one K slice (128 bytes of K) of every operand
// plane: the X box of the tap and the BN-row weight box.  fp32 256-row tiles hold one plane
// per stage instead (the tf32 plane's stage, then the cross plane's: four 48 KB stages fit),
// and with four or more taps along x they run in X-ring mode: the taps of one tap row read
// one shared X box (128 + mx - 1 rows, both planes) from a two-slot ring of its own, through
// descriptors that start one row further down per tap, while one-plane weight boxes stream
// through the stage ring.  16-bit 1-D plans may run in shared-X mode (set_pipeline_layout):
// one X box per channel slice in each stage, read by every tap the same way.
//
// Every mbarrier wait is bounded (wait_limit_ns of global time).  A wait that gives up sets
// a bit in the plan's status word and a CTA-wide abort flag; every role then stops, the
// producer waits for the TMA loads it issued, the MMA warp waits for its MMAs, and TMEM is
// freed before the CTA exits.
#pragma once

#include <algorithm>

#include "ctr_internal.h"
#include "epilogue.cuh"
#include "ptx.cuh"

namespace ctr {
namespace {

constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr int kSmemMax = 227 * 1024;

// CTAs per SM.  A bf16 tile of 64 phase rows has only a few K slices, and its output stage
// (one 32-column chunk per epilogue warp) takes far longer than its MMAs and loads: the
// eight epilogue warps are issue-bound on their dependent arithmetic and store chains.  Two
// CTAs per SM double the epilogue warps and independent tile pipelines an SM interleaves,
// each CTA with half the shared memory (fewer stages) and 256 TMEM columns.
constexpr int ctas_per_sm(Prec P, int BN) { return (is_16bit(P) && BN == 64) ? 2 : 1; }
constexpr uint64_t kDrainLimitNs = 2000000000ull;

template <Prec P, int BN>
struct Cfg {
    static constexpr int kPlanes = P == Prec::F32 ? 2 : 1;
    static constexpr int kSlice = gemm_slice_bytes(P, BN);  // K bytes per row per stage
    static constexpr int kElems = kSlice / (P == Prec::F32 ? 4 : 2);
    static constexpr int kKSteps = kSlice / 32;              // MMA K steps of 32 bytes
    static constexpr int kXBytes = kBM * kSlice;             // one 128-position Xs slice
    static constexpr int kWBytes = BN * kSlice;              // one BN-row weight slice
    // fp32 256-row tiles: each stage holds one operand plane of a K slice (the tf32 plane or
    // the cross plane), so four 48 KB stages of 128-byte rows fit; a K slice takes two
    // stages.  Otherwise a stage holds every plane of its K slice.
    static constexpr bool kPlaneStages = P == Prec::F32 && BN >= 256;
    static constexpr int kStagePlanes = kPlaneStages ? 1 : kPlanes;
    static constexpr int kStagesPerSlice = kPlaneStages ? kPlanes : 1;
    static constexpr int kStageBytes = kStagePlanes * (kXBytes + kWBytes);
    static constexpr int kBarBytes = kGemmBarBytes;
    static constexpr int kCtas = ctas_per_sm(P, BN);
    // Two CTAs share an SM's 228 KB (each also reserves 1 KB for the system).
    static constexpr int kSmemBudget = kCtas == 1 ? kSmemMax : 112 * 1024;
    static constexpr int kStagesRaw = (kSmemBudget - 1024 - kBarBytes) / kStageBytes;
    static constexpr int kStages = kStagesRaw > 8 ? 8 : kStagesRaw;
    static constexpr int kSmem = 1024 + kStages * kStageBytes + kBarBytes;
    // Grouped fp32 accumulation keeps its running sums in a TMEM region of BN columns
    // beside the accumulators for BN >= 128 (in registers they would not fit the 168 a
    // thread has with 10 warps per SM), in registers for BN = 64.
    static constexpr bool kTmemSum = P == Prec::F32 && BN >= 128;
    // TMEM accumulators: as many BN-column buffers as fit 512 columns (less the sum region),
    // at most 4, so the MMA can run several tiles ahead of the epilogue.
    static constexpr int kTmemBudget = 512 / kCtas;   // TMEM columns of one CTA
    static constexpr int kAccBufs = kTmemSum ? (kTmemBudget - BN) / BN
                                             : (kTmemBudget / BN > 4 ? 4 : kTmemBudget / BN);
    static constexpr uint32_t kSumCol = kAccBufs * BN;       // first column of the sum region
    // With a single accumulator the first group of a tile accumulates straight into the
    // sum region (nothing to fold); the later groups go through the accumulator.
    static constexpr bool kSumFirst = kTmemSum && kAccBufs == 1;
    static constexpr uint32_t kTmemCols = kAccBufs * BN + (kTmemSum ? BN : 0);
    static constexpr uint32_t kIdesc = ptx::idesc_f32acc(
        P == Prec::F32 ? ptx::kFmtTF32 : (P == Prec::F16 ? ptx::kFmtF16 : ptx::kFmtBF16), kBM, BN);
    // fp32 I/O: the cross products' MMA (bf16 pairs of the second operand plane).
    static constexpr uint32_t kIdescCross = ptx::idesc_f32acc(ptx::kFmtBF16, kBM, BN);
    static_assert(kStages >= 2, "at least two pipeline stages");
    static_assert(kTmemCols == 128 || kTmemCols == 256 || kTmemCols == 512,
                  "TMEM allocation is a power of two");
    static_assert(kAccBufs >= 1, "at least one accumulator");
};

struct TileCoord {
    int p0, r0;
    int z, kb0, kb1;
};

// Tile t -> (row tile fastest, then position tile, then split).  32-bit arithmetic: the host
// keeps tiles, positions and rows below 2^31 (64-bit divisions are long software sequences
// and every role decodes every tile).
__device__ __forceinline__ TileCoord decode_tile(uint32_t t, const GemmParams &gp, int bn) {
    TileCoord c;
    const uint32_t nr = (uint32_t)gp.num_r_tiles, np = (uint32_t)gp.num_p_tiles;
    const uint32_t rest = t / nr;
    const uint32_t r_tile = t - rest * nr;
    const uint32_t z = rest / np;
    const uint32_t p_tile = rest - z * np;
    c.z = (int)z;
    c.r0 = (int)(r_tile * (uint32_t)bn);
    c.p0 = (int)(p_tile * (uint32_t)kBM);
    const uint32_t sp = (uint32_t)gp.splits;
    if (gp.xring) {   // whole channel slices per split: slices kc * taps + tap
        const uint32_t kpt = (uint32_t)gp.kb_per_tap, taps = (uint32_t)(gp.mx * gp.my);
        c.kb0 = (int)((z * kpt / sp) * taps);
        c.kb1 = (int)(((z + 1) * kpt / sp) * taps);
        return c;
    }
    const uint32_t kbt = (uint32_t)gp.kb_total;
    c.kb0 = (int)(z * kbt / sp);
    c.kb1 = (int)((z + 1) * kbt / sp);
    return c;
}

__device__ __forceinline__ void give_up(volatile int *abort, uint32_t *status, uint32_t bit) {
    *abort = 1;
    atomicOr(status, bit);
}

// Output of one 32-column chunk (columns tc.r0 + 32c ..) of this thread's position: the fused
// polyphase output stage, or the raw fp32 values (split-K partials, col2im columns).  A
// function of its own, force-inlined, so that v stays in registers.
template <Prec P, bool CHAIN>
__device__ __forceinline__ void store_chunk_out(const GemmParams &gp, const TileCoord &tc,
                                                const PosInfo &ps, bool fused, int quad, int lane,
                                                int c, float (&v)[32]) {
    const int64_t r0 = tc.r0 + 32 * c;
    if (fused) {
        emit_cols<CHAIN ? kOutChain : kOutPlain,
                  P == Prec::BF16 ? kIoBF16 : (P == Prec::F16 ? kIoF16 : kIoF32)>(
            v, ps, r0, gp.epi, lane);
        return;
    }
    const int64_t pos = (int64_t)tc.p0 + 32 * quad + lane;
    float4 *dst = reinterpret_cast<float4 *>(gp.raw + (int64_t)tc.z * gp.raw_split_stride +
                                             pos * gp.raw_ld + r0);
#pragma unroll
    for (int i = 0; i < 8; ++i)
        dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

template <Prec P, int BN, bool CHAIN>
__global__ void __launch_bounds__(kThreads, ctas_per_sm(P, BN))
    gemm_tc_kernel(const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapW,
                   const __grid_constant__ CUtensorMap mapX2,
                   const __grid_constant__ CUtensorMap mapW2, const GemmParams gp) {
    using C = Cfg<P, BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *stage_base = smem;
    // The stage ring (nst stages of stage_bytes), then the barriers; the host sizes both.
    const int nst = gp.nstages;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + gp.bar_off);
    uint64_t *full = bars;
    uint64_t *empty = bars + kGemmMaxStages;
    uint64_t *tmem_full = bars + 2 * kGemmMaxStages;
    uint64_t *tmem_empty = tmem_full + C::kAccBufs;
    uint64_t *drain = tmem_empty + C::kAccBufs;
    uint64_t *sum_full = drain + 1;   // kSumFirst: a tile's first group is in the sum region
    uint64_t *sum_free = drain + 2;   // kSumFirst: the epilogue has read a tile's sums
    uint64_t *w_full = drain + 3;     // shared-X mode: the resident weight has landed
    uint64_t *xfull = drain + 4;      // X-ring mode: slot 0/1 holds its box
    uint64_t *xempty = drain + 6;     // X-ring mode: slot 0/1 may be refilled
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 8);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    auto x_slice = [&](int s, int plane) -> uint8_t * {
        return stage_base + s * gp.stage_bytes + plane * C::kXBytes;
    };
    auto w_slice = [&](int s, int plane) -> uint8_t * {
        return stage_base + s * gp.stage_bytes + C::kStagePlanes * C::kXBytes + plane * C::kWBytes;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < nst; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < C::kAccBufs; ++a) {
            ptx::mbar_init(&tmem_full[a], 1);
            ptx::mbar_init(&tmem_empty[a], kEpiWarps);
        }
        ptx::mbar_init(drain, 1);
        ptx::mbar_init(sum_full, 1);
        ptx::mbar_init(sum_free, kEpiWarps);
        ptx::mbar_init(w_full, 1);
        for (int q = 0; q < 2; ++q) {
            ptx::mbar_init(&xfull[q], 1);
            ptx::mbar_init(&xempty[q], 1);
        }
        *abort = 0;
        ptx::fence_mbar_init();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        ptx::tma_prefetch_desc(&mapX);
        ptx::tma_prefetch_desc(&mapW);
        if (P == Prec::F32) {
            ptx::tma_prefetch_desc(&mapX2);
            ptx::tma_prefetch_desc(&mapW2);
        }
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, C::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    // Everything above touched only shared memory, TMEM and the kernel parameters, so it may
    // overlap the previous kernel of the stream; global memory waits for it.
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    const uint32_t tmem_base = *tmem_slot;
    const uint64_t limit = gp.wait_limit_ns;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            bool w_issued = false;
            if constexpr (P != Prec::F32) {
                if (gp.xshare) {
                    // Shared-X mode: per tile and channel slice kc, one X box of x_rows rows at
                    // the tile's first tap row; the taps' weight slices with it, or the whole
                    // weight tile once, up front, when it stays resident.
                    const int x_bytes = gp.x_rows * C::kSlice;
                    const int taps = gp.mx;
                    if (gp.wres) {
                        uint8_t *wr = stage_base + gp.wres_off;
                        ptx::mbar_arrive_expect_tx(w_full, (uint32_t)(gp.kb_total * C::kWBytes));
                        for (int kb = 0; kb < gp.kb_total; ++kb)
                            ptx::tma_load_2d(wr + kb * C::kWBytes, &mapW, w_full, kb * C::kElems, 0);
                        w_issued = true;
                    }
                    const uint32_t stage_tx =
                        (uint32_t)(x_bytes + (gp.wres ? 0 : taps * C::kWBytes));
                    for (int64_t t = blockIdx.x; t < gp.num_tiles && !*abort; t += gridDim.x) {
                        const TileCoord tc = decode_tile((uint32_t)t, gp, BN);
                        for (int kc = 0; kc < gp.kb_per_tap; ++kc) {
                            if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, limit, abort)) {
                                if (!*abort) give_up(abort, gp.status, kStatusTimeoutProducer);
                                break;
                            }
                            ptx::mbar_arrive_expect_tx(&full[stage], stage_tx);
                            uint8_t *st = stage_base + stage * gp.stage_bytes;
                            ptx::tma_load_2d(st, &mapX, &full[stage], kc * C::kElems,
                                             (int32_t)(tc.p0 + gp.shift0));
                            if (!gp.wres)
                                for (int g = 0; g < taps; ++g)
                                    ptx::tma_load_2d(st + x_bytes + g * C::kWBytes, &mapW,
                                                     &full[stage],
                                                     (g * gp.kb_per_tap + kc) * C::kElems,
                                                     (int32_t)tc.r0);
                            ++issued;
                            if (++stage == nst) {
                                stage = 0;
                                phase ^= 1u;
                            }
                        }
                    }
                }
            }
            int64_t x_issued = 0;
            if constexpr (C::kPlaneStages) {
                if (gp.xring) {
                    // X-ring mode: per channel slice kc and tap row uy, one X box of both
                    // planes into the next ring slot; then per tap of the row and per plane,
                    // one weight box into the stage ring.
                    uint8_t *xr = stage_base + gp.xring_off;
                    const int x_bytes = gp.x_rows * C::kSlice;   // one plane of a box
                    const int taps = gp.mx * gp.my;
                    int slot = 0;
                    uint32_t xphase = 0;
                    bool stop = false;
                    for (int64_t t = blockIdx.x; t < gp.num_tiles && !*abort && !stop; t += gridDim.x) {
                        const TileCoord tc = decode_tile((uint32_t)t, gp, BN);
                        for (int kb = tc.kb0; kb < tc.kb1 && !stop; ++kb) {
                            const int kc = kb / taps;
                            const int g = kb - kc * taps;
                            const int uy = g / gp.mx;
                            if (g == uy * gp.mx) {
                                if (!ptx::mbar_wait(&xempty[slot], xphase ^ 1u, limit, abort)) {
                                    if (!*abort) give_up(abort, gp.status, kStatusTimeoutProducer);
                                    stop = true;
                                    break;
                                }
                                ptx::mbar_arrive_expect_tx(&xfull[slot], (uint32_t)(2 * x_bytes));
                                uint8_t *xb = xr + slot * 2 * x_bytes;
                                const int32_t x_k = kc * C::kElems;
                                const int32_t x_row = (int32_t)(tc.p0 + gp.shift0 + (int64_t)uy * gp.Px);
                                ptx::tma_load_2d(xb, &mapX, &xfull[slot], x_k, x_row);
                                ptx::tma_load_2d(xb + x_bytes, &mapX2, &xfull[slot], x_k, x_row);
                                ++x_issued;
                                if (++slot == 2) {
                                    slot = 0;
                                    xphase ^= 1u;
                                }
                            }
                            const int32_t w_k = (g * gp.kb_per_tap + kc) * C::kElems;
                            for (int pl = 0; pl < 2; ++pl) {
                                if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, limit, abort)) {
                                    if (!*abort) give_up(abort, gp.status, kStatusTimeoutProducer);
                                    stop = true;
                                    break;
                                }
                                ptx::mbar_arrive_expect_tx(&full[stage], (uint32_t)C::kWBytes);
                                ptx::tma_load_2d(stage_base + stage * gp.stage_bytes, pl ? &mapW2 : &mapW,
                                                 &full[stage], w_k, (int32_t)tc.r0);
                                ++issued;
                                if (++stage == nst) {
                                    stage = 0;
                                    phase ^= 1u;
                                }
                            }
                        }
                    }
                }
            }
            for (int64_t t = blockIdx.x; !gp.xshare && !gp.xring && t < gp.num_tiles && !*abort; t += gridDim.x) {
                const TileCoord tc = decode_tile((uint32_t)t, gp, BN);
                // Tap (uy, ux) and channel slice kc of K slice kb, stepped along with kb.
                const int g0 = tc.kb0 / gp.kb_per_tap;
                int kc = tc.kb0 - g0 * gp.kb_per_tap;
                int uy = g0 / gp.mx;
                int ux = g0 - uy * gp.mx;
                bool stop = false;
                for (int kb = tc.kb0; kb < tc.kb1 && !stop; ++kb) {
                    const int32_t x_k = kc * C::kElems;
                    const int32_t w_k = kb * C::kElems;
                    const int32_t x_row = (int32_t)(tc.p0 + gp.shift0 + (int64_t)uy * gp.Px + ux);
                    const int32_t w_row = (int32_t)tc.r0;
                    for (int sp = 0; sp < C::kStagesPerSlice; ++sp) {
                        if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, limit, abort)) {
                            if (!*abort) give_up(abort, gp.status, kStatusTimeoutProducer);
                            stop = true;
                            break;
                        }
                        ptx::mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
                        if constexpr (C::kPlaneStages) {
                            ptx::tma_load_2d(x_slice(stage, 0), sp ? &mapX2 : &mapX, &full[stage], x_k, x_row);
                            ptx::tma_load_2d(w_slice(stage, 0), sp ? &mapW2 : &mapW, &full[stage], w_k, w_row);
                        } else {
                            ptx::tma_load_2d(x_slice(stage, 0), &mapX, &full[stage], x_k, x_row);
                            ptx::tma_load_2d(w_slice(stage, 0), &mapW, &full[stage], w_k, w_row);
                            if (P == Prec::F32) {
                                ptx::tma_load_2d(x_slice(stage, 1), &mapX2, &full[stage], x_k, x_row);
                                ptx::tma_load_2d(w_slice(stage, 1), &mapW2, &full[stage], w_k, w_row);
                            }
                        }
                        ++issued;
                        if (++stage == nst) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (++kc == gp.kb_per_tap) {
                        kc = 0;
                        if (++ux == gp.mx) {
                            ux = 0;
                            ++uy;
                        }
                    }
                }
            }
            // Wait for the latest load into every stage, so no copy lands after exit.
            const int64_t pending = issued < nst ? issued : nst;
            for (int64_t s = 0; s < pending; ++s) {
                const int64_t idx = issued - 1 - s;
                if (!ptx::mbar_wait(&full[idx % nst], (uint32_t)((idx / nst) & 1),
                                    kDrainLimitNs, nullptr))
                    atomicOr(gp.status, kStatusTimeoutDrain);
            }
            if (w_issued && !ptx::mbar_wait(w_full, 0, kDrainLimitNs, nullptr))
                atomicOr(gp.status, kStatusTimeoutDrain);
            const int64_t x_pending = x_issued < 2 ? x_issued : 2;
            for (int64_t q = 0; q < x_pending; ++q) {
                const int64_t idx = x_issued - 1 - q;
                if (!ptx::mbar_wait(&xfull[idx % 2], (uint32_t)((idx / 2) & 1), kDrainLimitNs, nullptr))
                    atomicOr(gp.status, kStatusTimeoutDrain);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop; one elected lane issues each tcgen05 instruction.
        {
            int stage = 0;
            uint32_t phase = 0;
            int grp = 0;    // accumulator groups issued by this CTA (selects the TMEM buffer)
            int items = 0;  // tiles issued by this CTA (kSumFirst barrier phases)
            bool ok = true;
            if constexpr (P != Prec::F32) {
                if (gp.xshare) {
                    // Shared-X mode: one accumulation group per tile; for every channel slice
                    // the taps read the same X box, tap g starting g rows further down (a
                    // K-major 128-byte-swizzled operand may start at any row of its
                    // 1024-byte-aligned box: the swizzle follows the address bits).
                    const int x_bytes = gp.x_rows * C::kSlice;
                    const int taps = gp.mx;
                    uint8_t *wr = stage_base + gp.wres_off;
                    if (gp.wres && !ptx::mbar_wait_warp(w_full, 0, limit, abort)) {
                        if (lane == 0 && !*abort) give_up(abort, gp.status, kStatusTimeoutMma);
                        ok = false;
                    }
                    for (int64_t t = blockIdx.x; ok && t < gp.num_tiles && !ptx::abort_warp(abort); t += gridDim.x) {
                        const int acc = grp % C::kAccBufs;
                        const uint32_t acc_phase = (uint32_t)(grp / C::kAccBufs) & 1u;
                        if (!ptx::mbar_wait_warp(&tmem_empty[acc], acc_phase ^ 1u, limit, abort)) {
                            if (lane == 0 && !*abort) give_up(abort, gp.status, kStatusTimeoutMma);
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                        uint32_t accumulate = 0;
                        for (int kc = 0; kc < gp.kb_per_tap; ++kc) {
                            if (!ptx::mbar_wait_warp(&full[stage], phase, limit, abort)) {
                                if (lane == 0 && !*abort) give_up(abort, gp.status, kStatusTimeoutMma);
                                ok = false;
                                break;
                            }
                            ptx::tc_fence_after();
                            uint8_t *st = stage_base + stage * gp.stage_bytes;
                            for (int g = 0; g < taps; ++g) {
                                const uint64_t xd = ptx::sdesc_k<C::kSlice>(ptx::smem_u32(st + g * C::kSlice));
                                const uint8_t *wsl = gp.wres ? wr + (g * gp.kb_per_tap + kc) * C::kWBytes
                                                             : st + x_bytes + g * C::kWBytes;
                                const uint64_t wd = ptx::sdesc_k<C::kSlice>(ptx::smem_u32(wsl));
#pragma unroll
                                for (int k = 0; k < C::kKSteps; ++k) {
                                    const uint64_t dk = (uint64_t)(2 * k);
                                    if (ptx::elect_one())
                                        ptx::mma_f16(d_tmem, xd + dk, wd + dk, C::kIdesc, accumulate);
                                    accumulate = 1u;
                                }
                            }
                            if (ptx::elect_one()) ptx::mma_commit(&empty[stage]);
                            if (++stage == nst) {
                                stage = 0;
                                phase ^= 1u;
                            }
                        }
                        if (ok && ptx::elect_one()) ptx::mma_commit(&tmem_full[acc]);
                        ++grp;
                    }
                }
            }
            if constexpr (C::kPlaneStages) {
                if (gp.xring) {
                    // X-ring mode: tap ux of a row reads the row's X box through a descriptor
                    // that starts ux rows further down; the box's slot is released after the
                    // row's last tap.
                    const uint8_t *xr = stage_base + gp.xring_off;
                    const int x_bytes = gp.x_rows * C::kSlice;
                    const int taps = gp.mx * gp.my;
                    int slot = 0;
                    uint32_t xphase = 0;
                    for (int64_t t = blockIdx.x; ok && t < gp.num_tiles && !ptx::abort_warp(abort); t += gridDim.x, ++items) {
                        const TileCoord tc = decode_tile((uint32_t)t, gp, BN);
                        for (int kb = tc.kb0, gi = 0; ok && kb < tc.kb1; ++gi) {
                            const int kb_end = min(kb + gp.kb_group, tc.kb1);
                            const bool to_sum = C::kSumFirst && gi == 0;
                            const int acc = grp % C::kAccBufs;
                            if (to_sum) {
                                if (!ptx::mbar_wait_warp(sum_free, ((uint32_t)items & 1u) ^ 1u, limit, abort)) {
                                    if (lane == 0 && !*abort) give_up(abort, gp.status, kStatusTimeoutMma);
                                    ok = false;
                                    break;
                                }
                            } else {
                                const uint32_t acc_phase = (uint32_t)(grp / C::kAccBufs) & 1u;
                                if (!ptx::mbar_wait_warp(&tmem_empty[acc], acc_phase ^ 1u, limit, abort)) {
                                    if (lane == 0 && !*abort) give_up(abort, gp.status, kStatusTimeoutMma);
                                    ok = false;
                                    break;
                                }
                            }
                            ptx::tc_fence_after();
                            const uint32_t d_tmem =
                                tmem_base + (to_sum ? C::kSumCol : (uint32_t)(acc * BN));
                            uint32_t accumulate = 0;
                            for (; ok && kb < kb_end; ++kb) {
                                const int kc = kb / taps;
                                const int g = kb - kc * taps;
                                const int ux = g % gp.mx;
                                if (ux == 0) {
                                    if (!ptx::mbar_wait_warp(&xfull[slot], xphase, limit, abort)) {
                                        if (lane == 0 && !*abort) give_up(abort, gp.status, kStatusTimeoutMma);
                                        ok = false;
                                        break;
                                    }
                                    ptx::tc_fence_after();
                                }
                                const uint8_t *xb = xr + slot * 2 * x_bytes + ux * C::kSlice;
                                for (int pl = 0; pl < 2; ++pl) {
                                    if (!ptx::mbar_wait_warp(&full[stage], phase, limit, abort)) {
                                        if (lane == 0 && !*abort) give_up(abort, gp.status, kStatusTimeoutMma);
                                        ok = false;
                                        break;
                                    }
                                    ptx::tc_fence_after();
                                    const uint64_t xd = ptx::sdesc_k<C::kSlice>(ptx::smem_u32(xb + pl * x_bytes));
                                    const uint64_t wd = ptx::sdesc_k<C::kSlice>(
                                        ptx::smem_u32(stage_base + stage * gp.stage_bytes));
#pragma unroll
                                    for (int k = 0; k < C::kKSteps; ++k) {
                                        const uint64_t dk = (uint64_t)(2 * k);
                                        if (ptx::elect_one()) {
                                            if (pl == 0)
                                                ptx::mma_tf32(d_tmem, xd + dk, wd + dk, C::kIdesc, accumulate);
                                            else
                                                ptx::mma_f16(d_tmem, xd + dk, wd + dk, C::kIdescCross, 1u);
                                        }
                                        accumulate = 1u;
                                    }
                                    if (ptx::elect_one()) ptx::mma_commit(&empty[stage]);
                                    if (++stage == nst) {
                                        stage = 0;
                                        phase ^= 1u;
                                    }
                                }
                                if (!ok) break;
                                if (ux == gp.mx - 1) {   // the row's taps are issued: free its box
                                    if (ptx::elect_one()) ptx::mma_commit(&xempty[slot]);
                                    if (++slot == 2) {
                                        slot = 0;
                                        xphase ^= 1u;
                                    }
                                }
                            }
                            if (ok && ptx::elect_one()) ptx::mma_commit(to_sum ? sum_full : &tmem_full[acc]);
                            if (!to_sum) ++grp;
                        }
                    }
                }
            }
            for (int64_t t = blockIdx.x; !gp.xshare && !gp.xring && ok && t < gp.num_tiles && !ptx::abort_warp(abort); t += gridDim.x, ++items) {
                const TileCoord tc = decode_tile((uint32_t)t, gp, BN);
                for (int kb = tc.kb0, g = 0; ok && kb < tc.kb1; ++g) {
                    const int kb_end = min(kb + gp.kb_group, tc.kb1);
                    const bool to_sum = C::kSumFirst && g == 0;
                    const int acc = grp % C::kAccBufs;
                    if (to_sum) {
                        // The previous tile's sums must have been read.
                        if (!ptx::mbar_wait_warp(sum_free, ((uint32_t)items & 1u) ^ 1u, limit, abort)) {
                            if (lane == 0 && !*abort) give_up(abort, gp.status, kStatusTimeoutMma);
                            ok = false;
                            break;
                        }
                    } else {
                        const uint32_t acc_phase = (uint32_t)(grp / C::kAccBufs) & 1u;
                        if (!ptx::mbar_wait_warp(&tmem_empty[acc], acc_phase ^ 1u, limit, abort)) {
                            if (lane == 0 && !*abort) give_up(abort, gp.status, kStatusTimeoutMma);
                            ok = false;
                            break;
                        }
                    }
                    ptx::tc_fence_after();
                    const uint32_t d_tmem =
                        tmem_base + (to_sum ? C::kSumCol : (uint32_t)(acc * BN));
                    uint32_t accumulate = 0;
                    for (; ok && kb < kb_end; ++kb) {
                        for (int sp = 0; sp < C::kStagesPerSlice; ++sp) {
                            if (!ptx::mbar_wait_warp(&full[stage], phase, limit, abort)) {
                                if (lane == 0 && !*abort) give_up(abort, gp.status, kStatusTimeoutMma);
                                ok = false;
                                break;
                            }
                            ptx::tc_fence_after();
                            const uint64_t xd = ptx::sdesc_k<C::kSlice>(ptx::smem_u32(x_slice(stage, 0)));
                            const uint64_t wd = ptx::sdesc_k<C::kSlice>(ptx::smem_u32(w_slice(stage, 0)));
                            uint64_t xdl = 0, wdl = 0;
                            if (P == Prec::F32 && !C::kPlaneStages) {
                                xdl = ptx::sdesc_k<C::kSlice>(ptx::smem_u32(x_slice(stage, 1)));
                                wdl = ptx::sdesc_k<C::kSlice>(ptx::smem_u32(w_slice(stage, 1)));
                            }
#pragma unroll
                            for (int k = 0; k < C::kKSteps; ++k) {  // 32-byte K steps of the slice
                                // +2 in the descriptor's start-address field = +32 bytes
                                const uint64_t dk = (uint64_t)(2 * k);
                                if constexpr (C::kPlaneStages) {
                                    // the tf32 plane's stage first (hi*hi), then the cross
                                    // plane's (hi*lo + lo*hi)
                                    if (ptx::elect_one()) {
                                        if (sp == 0)
                                            ptx::mma_tf32(d_tmem, xd + dk, wd + dk, C::kIdesc, accumulate);
                                        else
                                            ptx::mma_f16(d_tmem, xd + dk, wd + dk, C::kIdescCross, 1u);
                                    }
                                } else if (P == Prec::F32) {
                                    if (ptx::elect_one()) {
                                        ptx::mma_f16(d_tmem, xdl + dk, wdl + dk, C::kIdescCross, accumulate);
                                        ptx::mma_tf32(d_tmem, xd + dk, wd + dk, C::kIdesc, 1u);
                                    }
                                } else {
                                    if (ptx::elect_one())
                                        ptx::mma_f16(d_tmem, xd + dk, wd + dk, C::kIdesc, accumulate);
                                }
                                accumulate = 1u;
                            }
                            if (ptx::elect_one())
                                ptx::mma_commit(&empty[stage]);  // frees the stage once these MMAs finish
                            if (++stage == nst) {
                                stage = 0;
                                phase ^= 1u;
                            }
                        }
                    }
                    if (ok && ptx::elect_one()) ptx::mma_commit(to_sum ? sum_full : &tmem_full[acc]);
                    if (!to_sum) ++grp;
                }
            }
            // Every MMA issued above completes before TMEM is freed.
            if (ptx::elect_one()) ptx::mma_commit(drain);
            __syncwarp();
            if (!ptx::mbar_wait_warp(drain, 0, kDrainLimitNs, nullptr) && lane == 0)
                atomicOr(gp.status, kStatusTimeoutDrain);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int quad = warp & 3;               // TMEM lanes 32*quad .. 32*quad + 31
        constexpr int kChunks = BN / 64;         // 32-column chunks per warp
        const int c_base = ((warp - 2) >> 2) * kChunks;  // this warp's first chunk
        const bool fused = gp.epi_mode == EPI_POLYPHASE;
        const uint32_t lane_addr = (uint32_t)(32 * quad) << 16;
        int grp = 0;
        int items = 0;   // kSumFirst: tiles whose sums this warp has read
        // Bounded wait of lane 0 on (bar, parity), uniform across the warp.
        auto warp_wait = [&](uint64_t *bar, uint32_t parity) -> bool {
            int ok = 1;
            if (lane == 0) {
                ok = ptx::mbar_wait(bar, parity, limit, abort) ? 1 : 0;
                if (!ok && !*abort) give_up(abort, gp.status, kStatusTimeoutEpilogue);
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            __syncwarp();
            return ok != 0;
        };
        auto wait_group = [&](int g) -> bool {
            const bool ok = warp_wait(&tmem_full[g % C::kAccBufs], (uint32_t)(g / C::kAccBufs) & 1u);
            if (ok) ptx::tc_fence_after();
            return ok;
        };
        auto release_group = [&](int g) {
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&tmem_empty[g % C::kAccBufs]);
        };
        auto tmem_chunk = [&](int g, int c, uint32_t (&u)[32]) {
            ptx::tmem_ld_32x32b_x32(
                tmem_base + lane_addr + (uint32_t)((g % C::kAccBufs) * BN + 32 * c), u);
        };
        auto sum_chunk_ld = [&](int c, uint32_t (&u)[32]) {
            ptx::tmem_ld_32x32b_x32(tmem_base + lane_addr + C::kSumCol + 32u * c, u);
        };
        bool ok = true;
        for (int64_t t = blockIdx.x; ok && t < gp.num_tiles; t += gridDim.x) {
            const TileCoord tc = decode_tile((uint32_t)t, gp, BN);
            const int ngroups = (tc.kb1 - tc.kb0 + gp.kb_group - 1) / gp.kb_group;
            PosInfo ps{};
            if (fused) ps = decode_pos(tc.p0 + 32 * quad + lane, gp.epi);
            if (C::kTmemSum && (C::kSumFirst || ngroups > 1)) {
                // Each group's partial is added, with fp32 round-to-nearest, into the TMEM sum
                // region (the first group is copied, or with a single accumulator was
                // accumulated there directly), and the accumulator is released at once; the
                // output stage then reads the finished sums.  Same arithmetic, in the same
                // order, as the register sums below.
                const int item = items++;
                for (int g = 0; g < ngroups; ++g) {
                    if (C::kSumFirst && g == 0) {
                        if (!(ok = warp_wait(sum_full, (uint32_t)item & 1u))) break;
                        ptx::tc_fence_after();
                        continue;
                    }
                    if (!(ok = wait_group(grp))) break;
#pragma unroll 1
                    for (int c = 0; c < kChunks; ++c) {
                        uint32_t u[32], w[32];
                        tmem_chunk(grp, c_base + c, u);
                        if (g > 0) {
                            sum_chunk_ld(c_base + c, w);
                            ptx::tmem_wait_ld();
#pragma unroll
                            for (int cc = 0; cc < 32; ++cc)
                                w[cc] = __float_as_uint(__uint_as_float(w[cc]) + __uint_as_float(u[cc]));
                        } else {
                            ptx::tmem_wait_ld();
#pragma unroll
                            for (int cc = 0; cc < 32; ++cc) w[cc] = u[cc];
                        }
                        ptx::tmem_st_32x32b_x32(tmem_base + lane_addr + C::kSumCol + 32u * (c_base + c), w);
                    }
                    ptx::tmem_wait_st();
                    release_group(grp);
                    ++grp;
                }
                if (!ok) break;
#pragma unroll 1
                for (int c = 0; c < kChunks; ++c) {
                    uint32_t u[32];
                    sum_chunk_ld(c_base + c, u);
                    ptx::tmem_wait_ld();
                    float v[32];
#pragma unroll
                    for (int cc = 0; cc < 32; ++cc) v[cc] = __uint_as_float(u[cc]);
                    store_chunk_out<P, CHAIN>(gp, tc, ps, fused, quad, lane, c_base + c, v);
                }
                if constexpr (C::kSumFirst) {   // the sum region may take the next tile
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(sum_free);
                }
            } else if (P != Prec::F32 || ngroups == 1) {
                // One accumulation group: straight from TMEM to the output stage.
                if (!(ok = wait_group(grp))) break;
#pragma unroll 1
                for (int c = 0; c < kChunks; ++c) {
                    uint32_t u[32];
                    tmem_chunk(grp, c_base + c, u);
                    ptx::tmem_wait_ld_regs(u);
                    if (c == kChunks - 1) release_group(grp);  // TMEM no longer needed
                    float v[32];
#pragma unroll
                    for (int cc = 0; cc < 32; ++cc) v[cc] = __uint_as_float(u[cc]);
                    store_chunk_out<P, CHAIN>(gp, tc, ps, fused, quad, lane, c_base + c, v);
                }
                ++grp;
            } else if constexpr (P == Prec::F32 && !C::kTmemSum) {
                // BN = 64 only.
                // Several groups: each group's partial leaves TMEM and is added, with fp32
                // round-to-nearest, into running sums held in registers (this thread's
                // position, this warp's BN/2 columns of the tile).  Keeps every tensor-core
                // accumulation chain short; see the group length chosen by the host.
                float sum[kChunks][32];
                for (int g = 0; g < ngroups; ++g, ++grp) {
                    if (!(ok = wait_group(grp))) break;
#pragma unroll
                    for (int c = 0; c < kChunks; ++c) {
                        uint32_t u[32];
                        tmem_chunk(grp, c_base + c, u);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int cc = 0; cc < 32; ++cc)
                            sum[c][cc] = g == 0 ? __uint_as_float(u[cc]) : sum[c][cc] + __uint_as_float(u[cc]);
                    }
                    release_group(grp);
                }
                if (!ok) break;
                // Unrolled (kChunks <= 2 here), so each chunk's sums die once stored.
#pragma unroll
                for (int c = 0; c < kChunks; ++c) store_chunk_out<P, CHAIN>(gp, tc, ps, fused, quad, lane, c_base + c, sum[c]);
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

template <Prec P, int BN, bool CHAIN>
cudaError_t launch_inst(const ctr_plan_s *pl, const CUtensorMap *maps, const GemmParams &gp,
                        cudaStream_t st) {
    using C = Cfg<P, BN>;
    // The dynamic shared-memory limit belongs to the current device's context: set it once
    // per device.
    static PerDeviceOnce once;
    cudaError_t ea = once.run(current_device(), cudaSuccess, [] {
        return cudaFuncSetAttribute(gemm_tc_kernel<P, BN, CHAIN>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBudget);
    });
    if (ea != cudaSuccess) return ea;
    if (gp.nstages < 2 || gp.nstages > kGemmMaxStages || gp.smem_bytes > C::kSmemBudget)
        return cudaErrorInvalidValue;
    const int64_t grid = std::min<int64_t>(gp.num_tiles, (int64_t)pl->num_sms * C::kCtas);
    const cudaError_t e = launch_pdl(gemm_tc_kernel<P, BN, CHAIN>, dim3((unsigned)grid),
                                     dim3(kThreads), (size_t)gp.smem_bytes, st, maps[0], maps[1],
                                     maps[2], maps[3], gp);
    if (e != cudaSuccess) return e;
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace
}  // namespace ctr
