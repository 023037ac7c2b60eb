// fused_pair.cu -- two chained 1-D upsampling layers in one kernel, the first layer's output
// kept in shared memory as the second layer's operand (ctr_forward_fused).
//
// A decoder's stack of upsamplers with an activation between them ("[XNNPACK] Lower dense
// transposed convs as one polyphase conv + depth to space", Test plan: two deconvolutions
// with an activation between; Summary: each layer one polyphase convolution) writes every
// intermediate to memory and reads it back.  For two small-channel layers that traffic is
// most of their bytes.  Here one CTA computes, per tile of the second layer's (B's) output
// phase positions, the slab of first-layer (A) outputs those positions read, and never
// stores it.  A tile is A's 128 positions; B's tile is 128 positions (one MMA group) or, when
// B's accumulators are 64 columns wide, up to 253 (two groups of 128), which uses all of the
// 2 x 128 outputs of A's tile:
//   warp 0      loads both packed weights once (they stay resident) and, per tile and
//               input channel slice, one box of A's staged input (128 positions plus A's
//               tap shifts);
//   warp 1      issues A's MMAs, tile after tile, and warp 18 B's, each as soon as its
//               operands and accumulator are free, so the tensor cores run one layer's
//               MMAs while the mid warps convert the other's tile;
//   warps 2..9  ("mid") read A's accumulator, add A's bias, apply its activation, round to
//               the I/O type and write the values as B's K-major, 128-byte-swizzled operand
//               box in shared memory: row r holds A's output a0 + r (zeros outside A's
//               output), every channel of it (one 128-byte row); two warps per TMEM lane
//               quarter, one phase each;
//   warps 10..17 run B's output stage (epilogue.cuh) on B's accumulator, two warps per lane
//               quarter splitting its columns;
//   warp 18     issues B's MMAs.
// Both MMAs read their operand boxes through descriptors that start tap rows further down
// (a K-major 128-byte-swizzled operand may start at any row of its 1024-byte-aligned box).
// The result is bit-identical to the two chained launches: the same products in the same
// order, the same single rounding of A's outputs.
//
// Every mbarrier wait is bounded, as in the GEMM kernel: a wait that gives up sets a status
// bit and the CTA's abort flag, and every role stops, drains its copies and MMAs and frees
// TMEM before the CTA exits.
#include <algorithm>
#include <cstring>

#include "ctr_internal.h"
#include "epilogue.cuh"
#include "ptx.cuh"

namespace ctr {
namespace {

constexpr int kFThreads = 608;
constexpr int kMidWarps = 8;     // warps 2..9
constexpr int kOutWarps = 8;     // warps 10..17
constexpr int kBWarp = 18;       // issues B's MMAs (warp 1 issues A's)
constexpr int kFMaxStages = 8;
constexpr int kRowBytes = 128;   // one K slice of 64 16-bit channels
constexpr uint64_t kFDrainNs = 2000000000ull;

struct FusedParams {
    int tiles_per_batch, num_tiles;
    int tile_q;   // B phase positions per tile (128, or up to 256 with two MMA groups)
    // layer A
    int kbA_per_tap, tapsA, x_rows_A, rbA, sA, epA;
    int64_t PA, LA_out;
    const void *biasA;
    int actA;
    float slopeA;
    // layer B
    int tapsB, x_rows_B, c0B;
    int64_t PB, QvB;
    EpiParams epiB;
    // shared memory: A's X stages, the resident weights, B's operand boxes, barriers
    int nstages, stage_bytes, wa_off, wb_off, bx_off, bar_off, smem_bytes;
    int kbA_total;
    uint32_t *status;
    uint64_t wait_limit_ns;
};

__device__ __forceinline__ void f_give_up(volatile int *abort, uint32_t *status, uint32_t bit) {
    *abort = 1;
    atomicOr(status, bit);
}

__device__ __forceinline__ int64_t floor_div(int64_t a, int64_t b) {
    const int64_t q = a / b;
    return (a % b != 0 && ((a < 0) != (b < 0))) ? q - 1 : q;
}

// The mid stage for one 32-column chunk of A's accumulator: phase j, channels ch0..ch0+31 of
// A's output position QA (one per lane), written to row r = sA*QA + j - epA - a0 of B's
// operand box when that row exists, as 4 swizzled 16-byte chunks.
template <typename T, bool ACT>
__device__ __forceinline__ void mid_chunk(float (&v)[32], uint8_t *box, int x_rows, int64_t oA,
                                          int64_t a0, int64_t LA_out, int ch0,
                                          const void *bias, float slope) {
    const int64_t r = oA - a0;
    if (r < 0 || r >= x_rows) return;
    uint32_t u[16];
    if (oA >= 0 && oA < LA_out) {
        const T *bsrc = bias ? static_cast<const T *>(bias) + ch0 : nullptr;
#pragma unroll
        for (int q = 0; q < 4; ++q) {   // 8 channels per bias vector
            float b[8];
            if (bsrc) {
                const uint4 w4 = __ldg(reinterpret_cast<const uint4 *>(bsrc + 8 * q));
                const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    b[2 * k] = io_lo<T>(ww[k]);
                    b[2 * k + 1] = io_hi<T>(ww[k]);
                }
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) b[k] = 0.0f;
            }
#pragma unroll
            for (int k = 0; k < 8; k += 2) {
                float a0v = v[8 * q + k] + b[k], a1v = v[8 * q + k + 1] + b[k + 1];
                if (ACT) {
                    a0v = a0v < 0.0f ? a0v * slope : a0v;
                    a1v = a1v < 0.0f ? a1v * slope : a1v;
                }
                u[(8 * q + k) / 2] = io_pack2<T>(a0v, a1v);
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < 16; ++k) u[k] = 0u;   // outside A's output: B reads zeros there
    }
    uint8_t *row = box + r * kRowBytes;
    const int sw = (int)(r & 7);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int cc = (ch0 >> 3) + q;   // 16-byte chunk of the 128-byte row
        *reinterpret_cast<uint4 *>(row + ((cc ^ sw) << 4)) =
            make_uint4(u[4 * q], u[4 * q + 1], u[4 * q + 2], u[4 * q + 3]);
    }
}

// KIND: layer B's output-stage variant compiled alone (EPI_KIND_1D_S2, the stride-2 layers),
// or -1 for the run-time dispatch over every variant.  One variant keeps the output warps'
// code small.
// NG: B's MMA groups of 128 positions per tile.  With NG = 2 a tile covers fp.tile_q <= 256
// of B's positions, fed by all sA * 128 outputs of A's 128-position tile (with NG = 1 only
// 128 + taps - 1 of them are used, and the neighbouring tile computes the rest again).
template <Prec P, int BNA, int BNB, int KIND, int NG>
__global__ void __launch_bounds__(kFThreads, 1)
    fused_pair_kernel(const __grid_constant__ CUtensorMap mapXA,
                      const __grid_constant__ CUtensorMap mapWA,
                      const __grid_constant__ CUtensorMap mapWB, const FusedParams fp) {
    using T = typename std::conditional<P == Prec::F16, __half, __nv_bfloat16>::type;
    constexpr uint32_t kFmt = P == Prec::F16 ? ptx::kFmtF16 : ptx::kFmtBF16;
    constexpr uint32_t kIdescA = ptx::idesc_f32acc(kFmt, kBM, BNA);
    constexpr uint32_t kIdescB = ptx::idesc_f32acc(kFmt, kBM, BNB);
    constexpr uint32_t kTmemCols = 2 * (BNA + NG * BNB) <= 256 ? 256 : 512;
    constexpr int kKSteps = kRowBytes / 32;
    static_assert(2 * (BNA + NG * BNB) <= 512, "two accumulators of each layer fit TMEM");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *wa = smem + fp.wa_off;
    uint8_t *wb = smem + fp.wb_off;
    uint8_t *bx = smem + fp.bx_off;
    const int box_bytes = fp.x_rows_B * kRowBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + fp.bar_off);
    uint64_t *full = bars;
    uint64_t *empty = bars + kFMaxStages;
    uint64_t *tA_full = bars + 2 * kFMaxStages;   // [2]
    uint64_t *tA_empty = tA_full + 2;              // [2], one arrival per mid warp
    uint64_t *bx_full = tA_empty + 2;              // [2], one arrival per mid warp
    uint64_t *bx_free = bx_full + 2;               // [2], B's MMAs done with the box
    uint64_t *tB_full = bx_free + 2;               // [2]
    uint64_t *tB_empty = tB_full + 2;              // [2], one arrival per final warp
    uint64_t *w_full = tB_empty + 2;
    uint64_t *drain = w_full + 1;      // warp 1's MMAs done
    uint64_t *drainB = drain + 1;      // warp 18's MMAs done
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drainB + 1);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nst = fp.nstages;

    if (threadIdx.x == 0) {
        for (int s = 0; s < nst; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(&tA_full[a], 1);
            ptx::mbar_init(&tA_empty[a], kMidWarps);
            ptx::mbar_init(&bx_full[a], kMidWarps);
            ptx::mbar_init(&bx_free[a], 1);
            ptx::mbar_init(&tB_full[a], 1);
            ptx::mbar_init(&tB_empty[a], kOutWarps);
        }
        ptx::mbar_init(w_full, 1);
        ptx::mbar_init(drain, 1);
        ptx::mbar_init(drainB, 1);
        *abort = 0;
        ptx::fence_mbar_init();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        ptx::tma_prefetch_desc(&mapXA);
        ptx::tma_prefetch_desc(&mapWA);
        ptx::tma_prefetch_desc(&mapWB);
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    const uint32_t tmem_base = *tmem_slot;
    const uint64_t limit = fp.wait_limit_ns;

    // Tile t -> batch item, the first B position q0 of the tile, the first A output a0 of
    // B's operand box and the first A position qa0 whose outputs cover it.
    auto tile_geo = [&](int t, int64_t &b, int64_t &q0, int64_t &a0, int64_t &qa0) {
        b = t / fp.tiles_per_batch;
        q0 = (int64_t)(t - b * fp.tiles_per_batch) * fp.tile_q;
        a0 = q0 + fp.c0B;
        qa0 = floor_div(a0 + fp.epA, fp.sA);
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint32_t w_bytes = (uint32_t)(fp.kbA_total * BNA * kRowBytes +
                                                fp.tapsB * BNB * kRowBytes);
            ptx::mbar_arrive_expect_tx(w_full, w_bytes);
            for (int kb = 0; kb < fp.kbA_total; ++kb)
                ptx::tma_load_2d(wa + kb * BNA * kRowBytes, &mapWA, w_full, kb * 64, 0);
            for (int g = 0; g < fp.tapsB; ++g)
                ptx::tma_load_2d(wb + g * BNB * kRowBytes, &mapWB, w_full, g * 64, 0);
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            for (int t = blockIdx.x; t < fp.num_tiles && !*abort; t += gridDim.x) {
                int64_t b, q0, a0, qa0;
                tile_geo(t, b, q0, a0, qa0);
                const int32_t row0 = (int32_t)(b * fp.PA + qa0 + fp.rbA);
                for (int kc = 0; kc < fp.kbA_per_tap; ++kc) {
                    if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, limit, abort)) {
                        if (!*abort) f_give_up(abort, fp.status, kStatusTimeoutProducer);
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(&full[stage], (uint32_t)fp.stage_bytes);
                    ptx::tma_load_2d(smem + stage * fp.stage_bytes, &mapXA, &full[stage],
                                     kc * 64, row0);
                    ++issued;
                    if (++stage == nst) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            const int64_t pending = issued < nst ? issued : nst;
            for (int64_t s = 0; s < pending; ++s) {
                const int64_t idx = issued - 1 - s;
                if (!ptx::mbar_wait(&full[idx % nst], (uint32_t)((idx / nst) & 1), kFDrainNs,
                                    nullptr))
                    atomicOr(fp.status, kStatusTimeoutDrain);
            }
            if (!ptx::mbar_wait(w_full, 0, kFDrainNs, nullptr)) atomicOr(fp.status, kStatusTimeoutDrain);
        }
    } else if (warp == 1 || warp == kBWarp) {
        // ------------------------------------------------------------ MMA issuers
        // Warp 1 issues A's MMAs, warp 18 B's.  Each whole warp runs its loop; one elected
        // lane issues each tcgen05 instruction, and each warp commits and drains its own.
        const bool is_a = warp == 1;
        bool ok = ptx::mbar_wait_warp(w_full, 0, limit, abort);
        if (!ok && lane == 0 && !*abort) f_give_up(abort, fp.status, kStatusTimeoutMma);
        if (is_a) {
            int stage = 0;
            uint32_t phase = 0;
            int na = 0;   // A tiles issued by this CTA
            for (int t = blockIdx.x; ok && t < fp.num_tiles && !ptx::abort_warp(abort);
                 t += gridDim.x, ++na) {
                const int acc = na & 1;
                if (!(ok = ptx::mbar_wait_warp(&tA_empty[acc], (((uint32_t)na >> 1) & 1u) ^ 1u,
                                               limit, abort)))
                    break;
                ptx::tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(acc * BNA);
                uint32_t accumulate = 0;
                for (int kc = 0; kc < fp.kbA_per_tap; ++kc) {
                    if (!(ok = ptx::mbar_wait_warp(&full[stage], phase, limit, abort))) break;
                    ptx::tc_fence_after();
                    uint8_t *st = smem + stage * fp.stage_bytes;
                    for (int g = 0; g < fp.tapsA; ++g) {
                        const uint64_t xd = ptx::sdesc_k<kRowBytes>(ptx::smem_u32(st + g * kRowBytes));
                        const uint64_t wd = ptx::sdesc_k<kRowBytes>(
                            ptx::smem_u32(wa + (g * fp.kbA_per_tap + kc) * BNA * kRowBytes));
#pragma unroll
                        for (int k = 0; k < kKSteps; ++k) {
                            if (ptx::elect_one()) ptx::mma_f16(d, xd + 2 * k, wd + 2 * k, kIdescA, accumulate);
                            accumulate = 1u;
                        }
                    }
                    if (ptx::elect_one()) ptx::mma_commit(&empty[stage]);
                    if (++stage == nst) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (ptx::elect_one()) ptx::mma_commit(&tA_full[acc]);
            }
        } else {
            int nb = 0;   // B tiles issued by this CTA
            for (int t = blockIdx.x; ok && t < fp.num_tiles && !ptx::abort_warp(abort);
                 t += gridDim.x, ++nb) {
                const int bb = nb & 1;
                const uint32_t par = ((uint32_t)nb >> 1) & 1u;
                if (!(ok = ptx::mbar_wait_warp(&bx_full[bb], par, limit, abort))) break;
                if (!(ok = ptx::mbar_wait_warp(&tB_empty[bb], par ^ 1u, limit, abort))) break;
                ptx::tc_fence_after();
                uint8_t *box = bx + bb * box_bytes;
#pragma unroll
                for (int h = 0; h < NG; ++h) {   // group h: positions 128h .. 128h + 127
                    const uint32_t d = tmem_base + (uint32_t)(2 * BNA + (bb * NG + h) * BNB);
                    uint32_t accumulate = 0;
                    for (int g = 0; g < fp.tapsB; ++g) {
                        const uint64_t xd = ptx::sdesc_k<kRowBytes>(
                            ptx::smem_u32(box + (kBM * h + g) * kRowBytes));
                        const uint64_t wd = ptx::sdesc_k<kRowBytes>(ptx::smem_u32(wb + g * BNB * kRowBytes));
#pragma unroll
                        for (int k = 0; k < kKSteps; ++k) {
                            if (ptx::elect_one()) ptx::mma_f16(d, xd + 2 * k, wd + 2 * k, kIdescB, accumulate);
                            accumulate = 1u;
                        }
                    }
                }
                if (ptx::elect_one()) {
                    ptx::mma_commit(&bx_free[bb]);
                    ptx::mma_commit(&tB_full[bb]);
                }
            }
        }
        if (!ok && lane == 0 && !*abort) f_give_up(abort, fp.status, kStatusTimeoutMma);
        uint64_t *my_drain = is_a ? drain : drainB;
        if (ptx::elect_one()) ptx::mma_commit(my_drain);
        __syncwarp();
        if (!ptx::mbar_wait_warp(my_drain, 0, kFDrainNs, nullptr) && lane == 0)
            atomicOr(fp.status, kStatusTimeoutDrain);
    } else if (warp < 2 + kMidWarps) {
        // ------------------------------------------------------------ mid: A -> B's operand
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;   // which half of A's columns (one phase)
        const uint32_t lane_addr = (uint32_t)(32 * quad) << 16;
        const bool act = fp.actA == CTR_ACT_LEAKY_RELU;
        int n = 0;
        auto warp_wait = [&](uint64_t *bar, uint32_t parity) -> bool {
            int okw = 1;
            if (lane == 0) {
                okw = ptx::mbar_wait(bar, parity, limit, abort) ? 1 : 0;
                if (!okw && !*abort) f_give_up(abort, fp.status, kStatusTimeoutEpilogue);
            }
            okw = __shfl_sync(0xffffffffu, okw, 0);
            __syncwarp();
            return okw != 0;
        };
        for (int t = blockIdx.x; t < fp.num_tiles; t += gridDim.x, ++n) {
            int64_t b, q0, a0, qa0;
            tile_geo(t, b, q0, a0, qa0);
            const int acc = n & 1;
            const uint32_t par = ((uint32_t)n >> 1) & 1u;
            if (!warp_wait(&tA_full[acc], par)) break;
            if (!warp_wait(&bx_free[acc], par ^ 1u)) break;
            ptx::tc_fence_after();
            uint8_t *box = bx + acc * box_bytes;
            const int64_t QA = qa0 + 32 * quad + lane;
#pragma unroll 1
            for (int c = half * (BNA / 64); c < (half + 1) * (BNA / 64); ++c) {
                uint32_t u[32];
                ptx::tmem_ld_32x32b_x32(tmem_base + lane_addr + (uint32_t)(acc * BNA + 32 * c), u);
                ptx::tmem_wait_ld_regs(u);
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(u[i]);
                // Phase-major rows: row 32c + i is phase (32c)/64, channel (32c) % 64 + i.
                const int j = (32 * c) / 64, ch0 = (32 * c) % 64;
                const int64_t oA = (int64_t)fp.sA * QA + j - fp.epA;
                if (act)
                    mid_chunk<T, true>(v, box, fp.x_rows_B, oA, a0, fp.LA_out, ch0, fp.biasA, fp.slopeA);
                else
                    mid_chunk<T, false>(v, box, fp.x_rows_B, oA, a0, fp.LA_out, ch0, fp.biasA, fp.slopeA);
            }
            ptx::tc_fence_before();
            // The box was written through the generic proxy; B's MMAs read it through the
            // async proxy.
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(&tA_empty[acc]);
                ptx::mbar_arrive(&bx_full[acc]);
            }
        }
    } else {
        // ------------------------------------------------------------ final: B's output
        const int quad = warp & 3;
        const int half = (warp - 2 - kMidWarps) >> 2;   // which half of B's columns
        const uint32_t lane_addr = (uint32_t)(32 * quad) << 16;
        constexpr int kIo = P == Prec::F16 ? kIoF16 : kIoBF16;
        int n = 0;
        auto warp_wait = [&](uint64_t *bar, uint32_t parity) -> bool {
            int okw = 1;
            if (lane == 0) {
                okw = ptx::mbar_wait(bar, parity, limit, abort) ? 1 : 0;
                if (!okw && !*abort) f_give_up(abort, fp.status, kStatusTimeoutEpilogue);
            }
            okw = __shfl_sync(0xffffffffu, okw, 0);
            __syncwarp();
            return okw != 0;
        };
        for (int t = blockIdx.x; t < fp.num_tiles; t += gridDim.x, ++n) {
            int64_t b, q0, a0, qa0;
            tile_geo(t, b, q0, a0, qa0);
            const int bb = n & 1;
            if (!warp_wait(&tB_full[bb], ((uint32_t)n >> 1) & 1u)) break;
            ptx::tc_fence_after();
            constexpr int kCh = BNB / 64;   // chunks per warp and group
#pragma unroll 1
            for (int h = 0; h < NG; ++h) {
            // A tile lies inside one batch item: its positions past the item's valid phase
            // positions (or past the tile's tile_q positions) would otherwise decode as the
            // next item's or the next tile's.
            const int64_t qi = kBM * h + 32 * quad + lane;
            const int64_t qb = q0 + qi;
            PosInfo ps = decode_pos(b * fp.PB + qb, fp.epiB);
            if (qb >= fp.QvB || qi >= fp.tile_q) ps.valid = false;
#pragma unroll 1
            for (int c = half * kCh; c < (half + 1) * kCh; ++c) {
                uint32_t u[32];
                ptx::tmem_ld_32x32b_x32(
                    tmem_base + lane_addr + (uint32_t)(2 * BNA + (bb * NG + h) * BNB + 32 * c), u);
                ptx::tmem_wait_ld_regs(u);
                if (h == NG - 1 && c == (half + 1) * kCh - 1) {
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(&tB_empty[bb]);
                }
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(u[i]);
                if constexpr (KIND == EPI_KIND_1D_S2)
                    emit_small<T, 2, 1>(v, ps, 32 * c, fp.epiB, lane);
                else
                    emit_cols<kOutPlain, kIo>(v, ps, 32 * c, fp.epiB, lane);
            }
            }
        }
    }

    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, kTmemCols);
    }
}

template <Prec P, int BNA, int BNB, int KIND, int NG>
cudaError_t launch_fused_inst(const ctr_plan_s *a, const CUtensorMap *maps, const FusedParams &fp,
                              cudaStream_t st) {
    static PerDeviceOnce once;
    cudaError_t e = once.run(current_device(), cudaSuccess, [] {
        return cudaFuncSetAttribute(fused_pair_kernel<P, BNA, BNB, KIND, NG>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    });
    if (e != cudaSuccess) return e;
    const int grid = std::min(fp.num_tiles, a->num_sms);
    e = launch_pdl(fused_pair_kernel<P, BNA, BNB, KIND, NG>, dim3((unsigned)grid), dim3(kFThreads),
                   (size_t)fp.smem_bytes, st, maps[0], maps[1], maps[2], fp);
    if (e != cudaSuccess) return e;
    count_launches(1);
    return cudaGetLastError();
}

// Shared-memory layout of a fused pair with ng MMA groups of B per tile; false when it does
// not fit.
bool fused_layout(const ctr_plan_s *a, const ctr_plan_s *b, int ng, FusedParams *fp) {
    const int64_t x_rows_A = (kBM + a->m[1] - 1 + 7) / 8 * 8;
    const int64_t x_rows_B = (ng * kBM + b->m[1] - 1 + 7) / 8 * 8;
    if (x_rows_A > 256 || x_rows_B > ng * kBM + 128) return false;
    const int64_t kbA_per_tap = a->C_in_pad / 64;
    const int64_t kbA_total = kbA_per_tap * a->m[1];
    const int64_t wa = kbA_total * a->block_n * kRowBytes;
    const int64_t wb = b->m[1] * b->block_n * kRowBytes;
    const int64_t bxb = 2 * x_rows_B * kRowBytes;
    const int64_t stage = x_rows_A * kRowBytes;
    const int64_t bars = 512;
    const int64_t avail = 227 * 1024 - 1024 - bars - wa - wb - bxb;
    const int64_t stages = std::min<int64_t>(avail / stage, kFMaxStages);
    if (stages < 2) return false;
    fp->x_rows_A = (int)x_rows_A;
    fp->x_rows_B = (int)x_rows_B;
    fp->kbA_per_tap = (int)kbA_per_tap;
    fp->kbA_total = (int)kbA_total;
    fp->nstages = (int)stages;
    fp->stage_bytes = (int)stage;
    fp->wa_off = (int)(stages * stage);
    fp->wb_off = (int)(fp->wa_off + wa);
    fp->bx_off = (int)(fp->wb_off + wb);
    fp->bar_off = (int)(fp->bx_off + bxb);
    fp->smem_bytes = 1024 + fp->bar_off + (int)bars;
    return true;
}

}  // namespace

bool fused_pair_supported(const ctr_plan_s *a) {
    const ctr_plan_s *b = a ? a->chain_next : nullptr;
    if (!b || a->dtype != b->dtype || a->dtype == CTR_F32) return false;
    if (a->path != CTR_PATH_POLYPHASE || b->path != CTR_PATH_POLYPHASE) return false;
    if (a->splits != 1 || b->splits != 1 || b->chain_next || b->nhwc || a->streaming) return false;
    if (a->ndim != 1 || b->ndim != 1) return false;
    // A: one row tile of 128 phase-major rows holding all 64 channels of its phases (the mid
    // stage writes whole 128-byte rows of B's operand), stride >= 2 (128 A positions then
    // cover B's 128 + taps - 1 operand rows).
    if (!a->row_pm || a->num_r_tiles != 1 || a->block_n != 128 || a->C_out != 64 ||
        a->block_n / a->S_pad != 64 || a->s[1] < 2)
        return false;
    // B: one 128-byte channel slice, one row tile of 64 or 128 rows.
    if (b->C_in_pad != 64 || b->num_r_tiles != 1 || (b->block_n != 64 && b->block_n != 128))
        return false;
    FusedParams fp;
    std::memset(&fp, 0, sizeof(fp));
    return fused_layout(a, b, 1, &fp);
}

namespace {

// B positions per tile with two MMA groups: A's 128-position tile gives sA * 128 operand rows
// starting up to sA - 1 rows before the tile's first row, and B's last position reads
// taps_B - 1 rows past its own; 0 when two groups do not apply (B's accumulators of 128
// columns would not fit TMEM twice, or the tile would not be longer than one group).
int64_t wide_tile_q(const ctr_plan_s *a, const ctr_plan_s *b) {
    if (b->block_n != 64) return 0;
    const int64_t q = std::min<int64_t>(2 * kBM, kBM * a->s[1] - (a->s[1] - 1) - (b->m[1] - 1));
    return q > kBM ? q : 0;
}

}  // namespace

cudaError_t launch_fused_pair(const ctr_plan_s *a, const void *xs, const void *wa_packed,
                              const void *bias_a, const void *wb_packed, const void *bias_b,
                              void *y, cudaStream_t st) {
    const ctr_plan_s *b = a->chain_next;
    FusedParams fp;
    std::memset(&fp, 0, sizeof(fp));
    int64_t tile_q = wide_tile_q(a, b);
    int ng = 2;
    if (tile_q == 0 || !fused_layout(a, b, 2, &fp)) {
        std::memset(&fp, 0, sizeof(fp));
        ng = 1;
        tile_q = kBM;
        if (!fused_layout(a, b, 1, &fp)) return cudaErrorInvalidValue;
    }
    CUtensorMap maps[3];
    if (!encode_2d(&maps[0], xs, a->dtype, a->C_in_pad, a->N_total, (uint32_t)fp.x_rows_A, kRowBytes) ||
        !encode_2d(&maps[1], wa_packed, a->dtype, a->K_total, a->M_pad, (uint32_t)a->block_n, kRowBytes) ||
        !encode_2d(&maps[2], wb_packed, b->dtype, b->K_total, b->M_pad, (uint32_t)b->block_n, kRowBytes))
        return cudaErrorInvalidValue;
    fp.tile_q = (int)tile_q;
    fp.tiles_per_batch = (int)((b->Qv[1] + tile_q - 1) / tile_q);
    fp.num_tiles = (int)(b->B * fp.tiles_per_batch);
    fp.tapsA = (int)a->m[1];
    fp.rbA = (int)a->rb[1];
    fp.sA = (int)a->s[1];
    fp.epA = (int)a->ep[1];
    fp.PA = a->P[1];
    fp.LA_out = a->out[1];
    fp.biasA = bias_a;
    fp.actA = a->act;
    fp.slopeA = a->slope;
    fp.tapsB = (int)b->m[1];
    fp.c0B = (int)(b->rb[1] - b->hf[1]);
    fp.PB = b->P[1];
    fp.QvB = b->Qv[1];
    fp.epiB = make_epi(b, bias_b, y);
    fp.status = a->d_status;
    fp.wait_limit_ns = a->wait_limit_ns;
    if (fp.num_tiles <= 0) return cudaSuccess;
    const bool f16 = a->dtype == CTR_F16;
    const bool s2 = fp.epiB.kind == EPI_KIND_1D_S2;
    if (ng == 2) {   // B tiles of 64 rows (wide_tile_q)
        if (s2)
            return f16 ? launch_fused_inst<Prec::F16, 128, 64, EPI_KIND_1D_S2, 2>(a, maps, fp, st)
                       : launch_fused_inst<Prec::BF16, 128, 64, EPI_KIND_1D_S2, 2>(a, maps, fp, st);
        return f16 ? launch_fused_inst<Prec::F16, 128, 64, -1, 2>(a, maps, fp, st)
                   : launch_fused_inst<Prec::BF16, 128, 64, -1, 2>(a, maps, fp, st);
    }
    if (b->block_n == 64)
        return f16 ? launch_fused_inst<Prec::F16, 128, 64, -1, 1>(a, maps, fp, st)
                   : launch_fused_inst<Prec::BF16, 128, 64, -1, 1>(a, maps, fp, st);
    if (s2)
        return f16 ? launch_fused_inst<Prec::F16, 128, 128, EPI_KIND_1D_S2, 1>(a, maps, fp, st)
                   : launch_fused_inst<Prec::BF16, 128, 128, EPI_KIND_1D_S2, 1>(a, maps, fp, st);
    return f16 ? launch_fused_inst<Prec::F16, 128, 128, -1, 1>(a, maps, fp, st)
               : launch_fused_inst<Prec::BF16, 128, 128, -1, 1>(a, maps, fp, st);
}

}  // namespace ctr
