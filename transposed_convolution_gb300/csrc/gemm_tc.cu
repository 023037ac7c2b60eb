// gemm_tc.cu -- the hot kernel: a persistent, warp-specialised implicit GEMM on the 5th-
// generation tensor cores (tcgen05 + TMEM), fed by TMA.
//
//   D[r, n] = sum over taps g and input channels ic of A[r, g*C_in_pad + ic] * Xs[n + shift(g), ic]
//
// For the polyphase path ("[XNNPACK] Lower dense transposed convs as one polyphase conv +
// depth to space", Summary) A is the phase-major prepacked weight, Xs the input staged
// channels-last with m - 1 zero positions on each side, and shift(g) = uy*Px + ux the tap
// offset, so that the m (or mH*mW) taps of the stride-1 phase convolution are m shifted TMA
// boxes of the same staged input: the zero halo is the convolution's padding m - 1.  For
// the col2im path ("[WebGPU] optimizations for audio models", ConvTranspose commit) there
// is one tap and D is the column buffer X[M, C_in] x W[C_in, k*C_out], transposed.
//
// Warp roles (192 threads, one CTA per SM, persistent over output tiles):
//   warp 0      one lane issues TMA loads of A and Xs K-slices into a ring of stages;
//   warp 1      allocates TMEM; one lane issues tcgen05.mma into one of two TMEM
//               accumulators (128 lanes x BN fp32 columns) and commits to mbarriers;
//   warps 2..5  the epilogue: tcgen05.ld of the accumulator, then either the fused polyphase
//               output stage (bias, activation, interleave, slice; epilogue.cuh) or a raw
//               fp32 store of D (split-K partials, col2im columns).
// Two accumulators let the epilogue of tile i overlap the MMAs of tile i + 1.
//
// 3xTF32 (fp32 I/O): both operands come as tf32 hi and lo planes (x = hi + lo, each
// rounded to tf32) and every K step issues lo*hi + hi*lo + hi*hi into the same fp32
// accumulator -- the split of Ootomo and Yokota, "Recovering single precision accuracy from
// Tensor Cores while surpassing the FP32 theoretical peak performance" (IJHPCA 2022).
//
// Every mbarrier wait is bounded (wait_limit_ns of global time).  A wait that gives up sets
// a bit in the plan's status word and a CTA-wide abort flag; every role then stops, the
// producer waits for the TMA loads it issued, the MMA warp waits for its MMAs, and TMEM is
// freed before the CTA exits.
#include <algorithm>

#include "ctr_internal.h"
#include "epilogue.cuh"
#include "ptx.cuh"

namespace ctr {
namespace {

constexpr int kThreads = 192;
constexpr int kEpiWarps = 4;
constexpr int kEpiTabBytes = (int)sizeof(GroupTables);  // per epilogue warp
constexpr int kEpiBytes = kEpiWarps * (32 * kEpiLdMax * 4 + kEpiTabBytes);
constexpr int kSmemBudget = 227 * 1024;
constexpr uint64_t kDrainLimitNs = 2000000000ull;

template <Prec P, int BN>
struct Cfg {
    static constexpr int kPlanes = P == Prec::TF32x3 ? 2 : 1;
    static constexpr int kABytes = kBM * kBKBytes;          // one 128-row A slice
    static constexpr int kBBytes = BN * kBKBytes;           // one BN-row Xs slice
    static constexpr int kStageBytes = kPlanes * (kABytes + kBBytes);
    static constexpr int kStagesRaw = (kSmemBudget - kEpiBytes - 2048) / kStageBytes;
    static constexpr int kStages = kStagesRaw > 8 ? 8 : kStagesRaw;
    static constexpr int kBarBytes = 256;
    static constexpr int kSmem = 1024 + kStages * kStageBytes + kEpiBytes + kBarBytes;
    static constexpr uint32_t kTmemCols = 2 * BN;
    static constexpr uint32_t kIdesc =
        ptx::idesc_f32acc(P == Prec::TF32x3 ? ptx::kFmtTF32 : ptx::kFmtBF16, kBM, BN);
    static_assert(kStages >= 2, "at least two pipeline stages");
    static_assert(kTmemCols == 256 || kTmemCols == 512, "TMEM allocation is a power of two");
};

struct TileCoord {
    int64_t m0, n0;
    int z, kb0, kb1;
};

__device__ __forceinline__ TileCoord decode_tile(int64_t t, const GemmParams &gp, int bn) {
    TileCoord c;
    const int64_t m_tile = t % gp.num_m_tiles;
    const int64_t rest = t / gp.num_m_tiles;
    const int64_t n_tile = rest % gp.num_n_tiles;
    c.z = (int)(rest / gp.num_n_tiles);
    c.m0 = m_tile * kBM;
    c.n0 = n_tile * bn;
    c.kb0 = (int)((int64_t)c.z * gp.kb_total / gp.splits);
    c.kb1 = (int)((int64_t)(c.z + 1) * gp.kb_total / gp.splits);
    return c;
}

__device__ __forceinline__ void give_up(volatile int *abort, uint32_t *status, uint32_t bit) {
    *abort = 1;
    atomicOr(status, bit);
}

template <Prec P, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                   const __grid_constant__ CUtensorMap mapA2,
                   const __grid_constant__ CUtensorMap mapB2, const GemmParams gp) {
    using C = Cfg<P, BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *stage_base = smem;
    float *epi_smem = reinterpret_cast<float *>(smem + C::kStages * C::kStageBytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kStages * C::kStageBytes + kEpiBytes);
    uint64_t *full = bars;
    uint64_t *empty = bars + C::kStages;
    uint64_t *tmem_full = bars + 2 * C::kStages;
    uint64_t *tmem_empty = tmem_full + 2;
    uint64_t *drain = tmem_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    auto a_slice = [&](int s, int plane) -> uint8_t * {
        return stage_base + s * C::kStageBytes + plane * C::kABytes;
    };
    auto b_slice = [&](int s, int plane) -> uint8_t * {
        return stage_base + s * C::kStageBytes + C::kPlanes * C::kABytes + plane * C::kBBytes;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(&tmem_full[a], 1);
            ptx::mbar_init(&tmem_empty[a], kEpiWarps);
        }
        ptx::mbar_init(drain, 1);
        *abort = 0;
        ptx::fence_mbar_init();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        ptx::tma_prefetch_desc(&mapA);
        ptx::tma_prefetch_desc(&mapB);
        if (P == Prec::TF32x3) {
            ptx::tma_prefetch_desc(&mapA2);
            ptx::tma_prefetch_desc(&mapB2);
        }
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, C::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint64_t limit = gp.wait_limit_ns;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            for (int64_t t = blockIdx.x; t < gp.num_tiles && !*abort; t += gridDim.x) {
                const TileCoord tc = decode_tile(t, gp, BN);
                for (int kb = tc.kb0; kb < tc.kb1; ++kb) {
                    if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, limit, abort)) {
                        if (!*abort) give_up(abort, gp.status, kStatusTimeoutProducer);
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
                    const int g = kb / gp.kb_per_tap;
                    const int kc = kb - g * gp.kb_per_tap;
                    const int uy = g / gp.mx;
                    const int ux = g - uy * gp.mx;
                    constexpr int kElems = P == Prec::TF32x3 ? 32 : 64;
                    const int32_t a_k = kb * kElems;
                    const int32_t b_k = kc * kElems;
                    const int32_t a_row = (int32_t)tc.m0;
                    const int32_t b_row = (int32_t)(tc.n0 + (int64_t)uy * gp.Px + ux);
                    ptx::tma_load_2d(a_slice(stage, 0), &mapA, &full[stage], a_k, a_row);
                    ptx::tma_load_2d(b_slice(stage, 0), &mapB, &full[stage], b_k, b_row);
                    if (P == Prec::TF32x3) {
                        ptx::tma_load_2d(a_slice(stage, 1), &mapA2, &full[stage], a_k, a_row);
                        ptx::tma_load_2d(b_slice(stage, 1), &mapB2, &full[stage], b_k, b_row);
                    }
                    ++issued;
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Wait for the latest load into every stage, so no copy lands after exit.
            const int64_t pending = issued < C::kStages ? issued : C::kStages;
            for (int64_t s = 0; s < pending; ++s) {
                const int64_t idx = issued - 1 - s;
                if (!ptx::mbar_wait(&full[idx % C::kStages], (uint32_t)((idx / C::kStages) & 1),
                                    kDrainLimitNs, nullptr))
                    atomicOr(gp.status, kStatusTimeoutDrain);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int grp = 0;  // accumulation groups issued by this CTA (selects the TMEM buffer)
            bool ok = true;
            for (int64_t t = blockIdx.x; ok && t < gp.num_tiles && !*abort; t += gridDim.x) {
                const TileCoord tc = decode_tile(t, gp, BN);
                for (int kb = tc.kb0; ok && kb < tc.kb1; ++grp) {
                    const int kb_end = min(kb + gp.kb_group, tc.kb1);
                    const int acc = grp & 1;
                    const uint32_t acc_phase = (uint32_t)(grp >> 1) & 1u;
                    if (!ptx::mbar_wait(&tmem_empty[acc], acc_phase ^ 1u, limit, abort)) {
                        if (!*abort) give_up(abort, gp.status, kStatusTimeoutMma);
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                    uint32_t accumulate = 0;
                    for (; kb < kb_end; ++kb) {
                        if (!ptx::mbar_wait(&full[stage], phase, limit, abort)) {
                            if (!*abort) give_up(abort, gp.status, kStatusTimeoutMma);
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        const uint32_t a_hi = ptx::smem_u32(a_slice(stage, 0));
                        const uint32_t b_hi = ptx::smem_u32(b_slice(stage, 0));
#pragma unroll
                        for (int k = 0; k < 4; ++k) {  // four 32-byte K steps per 128-byte slice
                            const uint64_t ad = ptx::sdesc_k_sw128(a_hi + 32 * k);
                            const uint64_t bd = ptx::sdesc_k_sw128(b_hi + 32 * k);
                            if (P == Prec::TF32x3) {
                                const uint32_t a_lo = ptx::smem_u32(a_slice(stage, 1));
                                const uint32_t b_lo = ptx::smem_u32(b_slice(stage, 1));
                                const uint64_t adl = ptx::sdesc_k_sw128(a_lo + 32 * k);
                                const uint64_t bdl = ptx::sdesc_k_sw128(b_lo + 32 * k);
                                ptx::mma_tf32(d_tmem, adl, bd, C::kIdesc, accumulate);
                                ptx::mma_tf32(d_tmem, ad, bdl, C::kIdesc, 1u);
                                ptx::mma_tf32(d_tmem, ad, bd, C::kIdesc, 1u);
                            } else {
                                ptx::mma_f16(d_tmem, ad, bd, C::kIdesc, accumulate);
                            }
                            accumulate = 1u;
                        }
                        ptx::mma_commit(&empty[stage]);  // frees the stage once these MMAs finish
                        if (++stage == C::kStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (ok) ptx::mma_commit(&tmem_full[acc]);
                }
            }
            // Every MMA issued above completes before TMEM is freed.
            ptx::mma_commit(drain);
            if (!ptx::mbar_wait(drain, 0, kDrainLimitNs, nullptr))
                atomicOr(gp.status, kStatusTimeoutDrain);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad + 31
        float *sm = epi_smem + (warp - 2) * 32 * kEpiLdMax;
        GroupTables *tab = reinterpret_cast<GroupTables *>(
            reinterpret_cast<uint8_t *>(epi_smem + kEpiWarps * 32 * kEpiLdMax) +
            (warp - 2) * kEpiTabBytes);
        const bool fused = gp.epi_mode == EPI_POLYPHASE;
        const int ld = fused ? gp.epi.epi_ld : 33;
        int grp = 0;
        // Wait for accumulation group g to land in TMEM; uniform across the warp.
        auto wait_group = [&](int g) -> bool {
            int ok = 1;
            if (lane == 0) {
                ok = ptx::mbar_wait(&tmem_full[g & 1], (uint32_t)(g >> 1) & 1u, limit, abort) ? 1 : 0;
                if (!ok && !*abort) give_up(abort, gp.status, kStatusTimeoutEpilogue);
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            __syncwarp();
            if (ok) ptx::tc_fence_after();
            return ok != 0;
        };
        auto release_group = [&](int g) {
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&tmem_empty[g & 1]);
        };
        // This lane's row of a 32-column chunk -> column-major staging block.
        auto stage_row = [&](const float (&v)[32]) {
#pragma unroll
            for (int cc = 0; cc < 32; ++cc) sm[cc * ld + lane] = v[cc];
            __syncwarp();
        };
        // Output stage of one staged 32-column chunk.
        auto store_chunk = [&](const TileCoord &tc, int c, const WarpRows &rows, ColCursor &cur) {
            const int64_t r0 = tc.m0 + 32 * quad;
            const int64_t n0 = tc.n0 + 32 * c;
            if (fused) {
                emit_block(sm, rows, cur, gp.epi, lane);
                col_advance(cur, 32, gp.epi);
            } else {
                float *dst = gp.raw + (int64_t)tc.z * gp.raw_split_stride + r0 * gp.raw_ld + n0 + lane;
#pragma unroll 4
                for (int i = 0; i < 32; ++i) dst[(int64_t)i * gp.raw_ld] = sm[lane * ld + i];
            }
            __syncwarp();
        };
        bool ok = true;
        for (int64_t t = blockIdx.x; ok && t < gp.num_tiles; t += gridDim.x) {
            const TileCoord tc = decode_tile(t, gp, BN);
            const int ngroups = (tc.kb1 - tc.kb0 + gp.kb_group - 1) / gp.kb_group;
            WarpRows rows{};
            ColCursor cur{};
            if (fused) {
                rows = warp_rows(tc.m0 + 32 * quad, gp.epi, lane, tab);
                cur = col_cursor(tc.n0, gp.epi);
            }
            if (P != Prec::TF32x3 || BN != 128 || ngroups == 1) {
                // One accumulation group: straight from TMEM to the output stage.
                if (!(ok = wait_group(grp))) break;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t u[32];
                    ptx::tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(32 * quad) << 16) +
                                                (uint32_t)((grp & 1) * BN + 32 * c), u);
                    ptx::tmem_wait_ld();
                    float v[32];
#pragma unroll
                    for (int cc = 0; cc < 32; ++cc) v[cc] = __uint_as_float(u[cc]);
                    if (c == BN / 32 - 1) release_group(grp);  // TMEM no longer needed
                    stage_row(v);
                    store_chunk(tc, c, rows, cur);
                }
                ++grp;
            } else if constexpr (P == Prec::TF32x3 && BN == 128) {
                // Several groups: each group's partial leaves TMEM and is added, with fp32
                // round-to-nearest, into running sums held in registers (this thread's row,
                // all 128 columns of the tile).  Keeps every tensor-core accumulation chain
                // short; see the group length chosen by the host.
                float sum[4][32];
                for (int g = 0; g < ngroups; ++g, ++grp) {
                    if (!(ok = wait_group(grp))) break;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t u[32];
                        ptx::tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(32 * quad) << 16) +
                                                    (uint32_t)((grp & 1) * BN + 32 * c), u);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int cc = 0; cc < 32; ++cc)
                            sum[c][cc] = g == 0 ? __uint_as_float(u[cc]) : sum[c][cc] + __uint_as_float(u[cc]);
                    }
                    release_group(grp);
                }
                if (!ok) break;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    stage_row(sum[c]);
                    store_chunk(tc, c, rows, cur);
                }
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

template <Prec P, int BN>
cudaError_t launch_inst(const ctr_plan_s *pl, const CUtensorMap *maps, const GemmParams &gp,
                        cudaStream_t st) {
    using C = Cfg<P, BN>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<P, BN>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int64_t grid = std::min<int64_t>(gp.num_tiles, pl->num_sms);
    gemm_tc_kernel<P, BN><<<(unsigned)grid, kThreads, C::kSmem, st>>>(maps[0], maps[1], maps[2],
                                                                      maps[3], gp);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

size_t gemm_smem_bytes(Prec prec, int block_n) {
    if (prec == Prec::BF16) return block_n == 256 ? Cfg<Prec::BF16, 256>::kSmem : Cfg<Prec::BF16, 128>::kSmem;
    return block_n == 256 ? Cfg<Prec::TF32x3, 256>::kSmem : Cfg<Prec::TF32x3, 128>::kSmem;
}

cudaError_t launch_gemm_tc(const ctr_plan_s *pl, const CUtensorMap *maps, const GemmParams &gp,
                           cudaStream_t st) {
    if (gp.num_tiles <= 0) return cudaSuccess;
    const bool bf16 = pl->dtype == CTR_BF16;
    if (bf16) {
        return pl->block_n == 256 ? launch_inst<Prec::BF16, 256>(pl, maps, gp, st)
                                  : launch_inst<Prec::BF16, 128>(pl, maps, gp, st);
    }
    return pl->block_n == 256 ? launch_inst<Prec::TF32x3, 256>(pl, maps, gp, st)
                              : launch_inst<Prec::TF32x3, 128>(pl, maps, gp, st);
}

}  // namespace ctr
