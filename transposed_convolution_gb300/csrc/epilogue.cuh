// epilogue.cuh -- output stage of the polyphase GEMM: bias, activation, the phase interleave
// and the padding slice, written straight from the accumulator registers.
//
// "[XNNPACK] Lower dense transposed convs as one polyphase conv + depth to space" (Summary)
// computes every output phase with one stride-1 convolution, then interleaves the phases
// (a view/permute/view in 1-D, a block-major depth_to_space in 2-D) and slices off the
// padding.  Here the GEMM is D[position, phase row]: TMEM lane = phase position n of the
// staged input, (b, qy, qx); TMEM column = phase row r = oc*S_pad + jy*sx + jx.  D[n, r]
// lands at y[b, oc, sy*qy + jy - py, sx*qx + jx - px] when that is inside the output, so the
// sx phases of one (oc, jy) held by one thread are sx consecutive outputs, and consecutive
// lanes (consecutive qx) continue the run.  The interleave and the slice are therefore just
// the store addresses: each thread writes its runs with aligned vector stores, and the warp's
// stores cover contiguous output rows.  The bias is added once, in fp32, before the
// activation and the single rounding to the I/O type ("[WebGPU] optimizations for audio
// models", review commit: f32 sums, bias bound once).
#pragma once

#include <cuda_bf16.h>

#include "ctr_internal.h"
#include "ptx.cuh"

namespace ctr {

__device__ __forceinline__ float load_io(const void *p, int64_t i, int bf16) {
    return bf16 ? __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i])
                : static_cast<const float *>(p)[i];
}

__device__ __forceinline__ void store_io(void *p, int64_t i, float v, int bf16) {
    if (bf16)
        static_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(v);
    else
        static_cast<float *>(p)[i] = v;
}

__device__ __forceinline__ float apply_act(float v, int act, float slope) {
    return (act == CTR_ACT_LEAKY_RELU && v < 0.0f) ? v * slope : v;
}

// Phase position of a GEMM row (one per thread).
struct PosInfo {
    int64_t b, qy, qx;
    bool valid;
};

// 32-bit arithmetic: the host keeps positions below 2^31 (see decode_tile).
__device__ __forceinline__ PosInfo decode_pos(int64_t n, const EpiParams &e) {
    PosInfo p;
    const uint32_t nn = (uint32_t)n, px = (uint32_t)e.Px, plane = (uint32_t)(e.Py * e.Px);
    const uint32_t b = nn / plane;
    const uint32_t rem = nn - b * plane;
    const uint32_t qy = rem / px;
    p.b = b;
    p.qy = qy;
    p.qx = rem - qy * px;
    p.valid = p.b < e.B && p.qy < e.Qvy && p.qx < e.Qvx;
    return p;
}

// Stores N consecutive outputs vals[0..N-1] at dst, as wbytes-wide stores (16, 8, 4 or the
// element size); dst is wbytes-aligned whenever wbytes > sizeof(T).
template <typename T, int N>
__device__ __forceinline__ void store_run(T *dst, const float *vals, int wbytes) {
    if constexpr (sizeof(T) == 4) {
        if (wbytes == 16 && N % 4 == 0) {
#pragma unroll
            for (int i = 0; i < N; i += 4)
                *reinterpret_cast<float4 *>(dst + i) =
                    make_float4(vals[i], vals[i + 1], vals[i + 2], vals[i + 3]);
            return;
        }
        if (wbytes == 8 && N % 2 == 0) {
#pragma unroll
            for (int i = 0; i < N; i += 2)
                *reinterpret_cast<float2 *>(dst + i) = make_float2(vals[i], vals[i + 1]);
            return;
        }
#pragma unroll
        for (int i = 0; i < N; ++i) dst[i] = vals[i];
    } else {
        if constexpr (N % 2 == 0) {
            if (wbytes >= 4) {
                uint32_t u[N / 2];
#pragma unroll
                for (int i = 0; i < N; i += 2) {
                    __nv_bfloat162 h = __floats2bfloat162_rn(vals[i], vals[i + 1]);
                    u[i / 2] = *reinterpret_cast<uint32_t *>(&h);
                }
                if constexpr (N % 8 == 0) {
                    if (wbytes == 16) {
#pragma unroll
                        for (int i = 0; i < N / 2; i += 4)
                            *reinterpret_cast<uint4 *>(dst + 2 * i) =
                                make_uint4(u[i], u[i + 1], u[i + 2], u[i + 3]);
                        return;
                    }
                }
                if constexpr (N % 4 == 0) {
                    if (wbytes >= 8) {
#pragma unroll
                        for (int i = 0; i < N / 2; i += 2)
                            *reinterpret_cast<uint2 *>(dst + 2 * i) = make_uint2(u[i], u[i + 1]);
                        return;
                    }
                }
#pragma unroll
                for (int i = 0; i < N / 2; ++i) *reinterpret_cast<uint32_t *>(dst + 2 * i) = u[i];
                return;
            }
        }
#pragma unroll
        for (int i = 0; i < N; ++i) dst[i] = __float2bfloat16_rn(vals[i]);
    }
}

// One run of NX consecutive outputs at dst (x = x0 .. x0+NX-1 of one output row) from
// v[0..NX-1]: bias, activation (slope_eff = 1 when there is none), then aligned vector
// stores inside the row, or element stores with bounds checks at its edges.
// LeakyReLU as one multiply and one max (slope <= 1) or min (slope > 1): equal to
// (a < 0 ? a * slope : a) for every a, NaN included; slope 1 is the identity.
__device__ __forceinline__ float leaky(float a, float slope_eff, bool use_min) {
    const float m = a * slope_eff;
    return use_min ? fminf(a, m) : fmaxf(a, m);
}

template <typename T, int NX>
__device__ __forceinline__ void emit_run(T *__restrict__ dst, int64_t x0, const float *v,
                                         float bias, float slope_eff, const EpiParams &e,
                                         bool interior) {
    const bool use_min = slope_eff > 1.0f;
    float t[NX];
#pragma unroll
    for (int i = 0; i < NX; ++i) t[i] = leaky(v[i] + bias, slope_eff, use_min);
    if (interior) {
        store_run<T, NX>(dst, t, e.store_bytes);
    } else {
#pragma unroll
        for (int i = 0; i < NX; ++i)
            if (x0 + i >= 0 && x0 + i < e.Wout) dst[i] = static_cast<T>(t[i]);
    }
}

// Bias of channel oc0 + lane for the first `count` lanes (0 elsewhere), so that a warp can
// share a chunk's biases by shuffles: one load per lane, issued before any output store.
__device__ __forceinline__ float lane_bias(const EpiParams &e, int64_t oc0, int count, int lane) {
    return (e.bias && lane < count && oc0 + lane < e.C_out) ? load_io(e.bias, oc0 + lane, e.out_bf16)
                                                            : 0.0f;
}

__device__ __forceinline__ float slope_of(const EpiParams &e) {
    return e.act == CTR_ACT_LEAKY_RELU ? e.slope : 1.0f;
}

// Output stage for whole phase sets: S = S_pad = SX * SY <= 32 (SX, SY compile-time), so the
// 32 columns r0 .. r0+31 of a chunk are G = 32/S whole channels.  Warp-collective: every
// lane passes the same r0 (its own position in ps).
template <typename T, int SX, int SY>
__device__ __forceinline__ void emit_small(const float (&v)[32], const PosInfo &ps, int64_t r0,
                                           const EpiParams &e, int lane) {
    constexpr int S = SX * SY;
    constexpr int G = 32 / S;
    const int64_t oc0 = r0 / S;
    const float bl = lane_bias(e, oc0, G, lane);
    const float slope_eff = slope_of(e);
    const int64_t x0 = (int64_t)SX * ps.qx - e.px;
    const int64_t oy0 = (int64_t)SY * ps.qy - e.py;
    const bool interior = x0 >= 0 && x0 + SX <= e.Wout;
    const int64_t cstride = e.Hout * e.Wout;
    // Channels of this chunk inside C_out (the same on every lane) and rows inside the
    // output for this lane's position, decided once for the chunk.
    const int64_t g_left = e.C_out - oc0;
    const int gmax = g_left < G ? (int)g_left : G;
    bool row_ok[SY];
#pragma unroll
    for (int jy = 0; jy < SY; ++jy) row_ok[jy] = ps.valid && oy0 + jy >= 0 && oy0 + jy < e.Hout;
    // Output of (oc0, oy0, x0); rows and channels below are offsets from it.
    T *__restrict__ dst = static_cast<T *>(e.y) + ((ps.b * e.C_out + oc0) * e.Hout + oy0) * e.Wout + x0;
    // Every lane runs the channel loop (the shuffles need the whole warp); lanes whose
    // position lies outside the output store nothing.
#pragma unroll
    for (int g = 0; g < G; ++g, dst += cstride) {
        if (g >= gmax) break;
        const float bias = __shfl_sync(0xffffffffu, bl, g);
#pragma unroll
        for (int jy = 0; jy < SY; ++jy)
            if (row_ok[jy])
                emit_run<T, SX>(dst + jy * e.Wout, x0, &v[g * S + jy * SX], bias, slope_eff, e,
                                interior);
    }
}

// Output stage for 1-D plans with S = S_pad a multiple of 32: the 32 columns of a chunk are 32
// consecutive phases j0 .. j0+31 of one channel, i.e. 32 consecutive outputs.
template <typename T>
__device__ __forceinline__ void emit_large(const float (&v)[32], const PosInfo &ps, int64_t r0,
                                           const EpiParams &e, int lane) {
    const int64_t oc = (uint32_t)r0 / (uint32_t)e.S_pad;
    const float bias = __shfl_sync(0xffffffffu, lane_bias(e, oc, 1, lane), 0);
    if (!ps.valid || oc >= e.C_out) return;
    const int64_t j0 = r0 - oc * e.S_pad;
    const int64_t x0 = (int64_t)e.sx * ps.qx + j0 - e.px;
    const bool interior = x0 >= 0 && x0 + 32 <= e.Wout;
    emit_run<T, 32>(static_cast<T *>(e.y) + (ps.b * e.C_out + oc) * e.Wout + x0, x0, v, bias,
                    slope_of(e), e, interior);
}

// Any plan: every output element on its own, with the full index map and bounds checks.
__device__ __forceinline__ void emit_generic(const float (&v)[32], const PosInfo &ps, int64_t r0,
                                             const EpiParams &e) {
    if (!ps.valid) return;
    const float slope_eff = slope_of(e);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const uint32_t r = (uint32_t)r0 + i;
        const uint32_t oc = r / (uint32_t)e.S_pad;
        const int j = (int)(r - oc * (uint32_t)e.S_pad);
        if (oc >= e.C_out || j >= e.S) continue;
        const int jy = j / e.sx, jx = j - (j / e.sx) * e.sx;
        const int64_t oy = (int64_t)e.sy * ps.qy + jy - e.py;
        const int64_t ox = (int64_t)e.sx * ps.qx + jx - e.px;
        if (oy < 0 || oy >= e.Hout || ox < 0 || ox >= e.Wout) continue;
        const float bias = e.bias ? load_io(e.bias, oc, e.out_bf16) : 0.0f;
        const float a = v[i] + bias;
        store_io(e.y, ((ps.b * e.C_out + oc) * e.Hout + oy) * e.Wout + ox,
                 a < 0.0f ? a * slope_eff : a, e.out_bf16);
    }
}

// ------------------------------------------------------------ chained output
// The same outputs written into the next plan's staged input (EpiParams::out_staged):
// channels-last, so the G channels of one output position are G consecutive elements.
// fp32 values are split into tf32 hi and lo planes exactly as the staging kernel does.

// Row of the staged buffer holding output (b, oy, ox).
__device__ __forceinline__ int64_t staged_row(const EpiParams &e, int64_t b, int64_t oy,
                                              int64_t ox) {
    return (b * e.ys_Py + oy + e.ys_hy) * e.ys_Px + ox + e.ys_hx;
}

// N consecutive channel values at dst (N * sizeof(T)-aligned): one plane for bf16, the hi
// and lo planes for fp32.
template <typename T, int N>
__device__ __forceinline__ void store_channels(T *dst, const float *vals, const EpiParams &e) {
    constexpr int kBytes = N * (int)sizeof(T) < 16 ? N * (int)sizeof(T) : 16;
    if constexpr (sizeof(T) == 2) {
        store_run<T, N>(dst, vals, kBytes);
    } else {
        float hi[N], lo[N];
#pragma unroll
        for (int i = 0; i < N; ++i) {
            hi[i] = ptx::to_tf32(vals[i]);
            lo[i] = ptx::to_tf32(vals[i] - hi[i]);
        }
        store_run<T, N>(dst, hi, kBytes);
        store_run<T, N>(dst + e.ys_lo, lo, kBytes);
    }
}

template <typename T, int SX, int SY>
__device__ __forceinline__ void emit_small_chain(const float (&v)[32], const PosInfo &ps,
                                                 int64_t r0, const EpiParams &e, int lane) {
    constexpr int S = SX * SY;
    constexpr int G = 32 / S;
    const int64_t oc0 = r0 / S;
    const float bl = lane_bias(e, oc0, G, lane);
    const float slope_eff = slope_of(e);
    const bool use_min = slope_eff > 1.0f;
    const int64_t g_left = e.C_out - oc0;
    const int gmax = g_left < G ? (int)g_left : G;
    // Bias and activation in place (every lane takes part in the shuffles).
    float t[32];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float bias = __shfl_sync(0xffffffffu, bl, g);
#pragma unroll
        for (int j = 0; j < S; ++j) t[g * S + j] = leaky(v[g * S + j] + bias, slope_eff, use_min);
    }
    if (!ps.valid) return;
    T *__restrict__ ys = static_cast<T *>(e.y);
#pragma unroll
    for (int jy = 0; jy < SY; ++jy) {
        const int64_t oy = (int64_t)SY * ps.qy + jy - e.py;
        if (oy < 0 || oy >= e.Hout) continue;
#pragma unroll
        for (int jx = 0; jx < SX; ++jx) {
            const int64_t ox = (int64_t)SX * ps.qx + jx - e.px;
            if (ox < 0 || ox >= e.Wout) continue;
            T *dst = ys + staged_row(e, ps.b, oy, ox) * e.ys_cpad + oc0;
            float c[G];
#pragma unroll
            for (int g = 0; g < G; ++g) c[g] = t[g * S + jy * SX + jx];
            if (gmax == G) {
                store_channels<T, G>(dst, c, e);
            } else {
#pragma unroll
                for (int g = 0; g < G; ++g)
                    if (g < gmax) store_channels<T, 1>(dst + g, &c[g], e);
            }
        }
    }
}

// Phase-major rows (EpiParams::pm_tc): the chunk's 32 columns are NJ = 32 / TCR phases of
// TCR = min(pm_tc, 32) consecutive channels each, so every phase is one run of TCR channel
// values at one output position.
template <typename T, int TCR>
__device__ __forceinline__ void emit_pm_chain(const float (&v)[32], const PosInfo &ps,
                                              int64_t r0, const EpiParams &e, int lane) {
    constexpr int NJ = 32 / TCR;
    const int tc = e.pm_tc;
    const int bn = tc * e.S_pad;
    const int64_t tile = r0 / bn;
    const int rl0 = (int)(r0 - tile * bn);
    const int j0 = rl0 / tc;
    const int64_t oc0 = tile * tc + (rl0 - j0 * tc);
    const float bl = lane_bias(e, oc0, TCR, lane);
    const float slope_eff = slope_of(e);
    const bool use_min = slope_eff > 1.0f;
    const int64_t c_left = e.C_out - oc0;
    const int cmax = c_left < TCR ? (int)c_left : TCR;
    float t[32];
#pragma unroll
    for (int i = 0; i < TCR; ++i) {
        const float bias = __shfl_sync(0xffffffffu, bl, i);
#pragma unroll
        for (int jj = 0; jj < NJ; ++jj)
            t[jj * TCR + i] = leaky(v[jj * TCR + i] + bias, slope_eff, use_min);
    }
    if (!ps.valid || cmax <= 0) return;
    T *__restrict__ ys = static_cast<T *>(e.y);
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) {
        const int j = j0 + jj;
        const int jy = j / e.sx, jx = j - (j / e.sx) * e.sx;
        const int64_t oy = (int64_t)e.sy * ps.qy + jy - e.py;
        const int64_t ox = (int64_t)e.sx * ps.qx + jx - e.px;
        if (oy < 0 || oy >= e.Hout || ox < 0 || ox >= e.Wout) continue;
        T *dst = ys + staged_row(e, ps.b, oy, ox) * e.ys_cpad + oc0;
        if (cmax == TCR) {
            store_channels<T, TCR>(dst, &t[jj * TCR], e);
        } else {
#pragma unroll
            for (int i = 0; i < TCR; ++i)
                if (i < cmax) store_channels<T, 1>(dst + i, &t[jj * TCR + i], e);
        }
    }
}

// Any plan, element by element.
__device__ __forceinline__ void emit_generic_chain(const float (&v)[32], const PosInfo &ps,
                                                   int64_t r0, const EpiParams &e) {
    if (!ps.valid) return;
    const float slope_eff = slope_of(e);
    const bool use_min = slope_eff > 1.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const uint32_t r = (uint32_t)r0 + i;
        const uint32_t oc = r / (uint32_t)e.S_pad;
        const int j = (int)(r - oc * (uint32_t)e.S_pad);
        if (oc >= e.C_out || j >= e.S) continue;
        const int jy = j / e.sx, jx = j - (j / e.sx) * e.sx;
        const int64_t oy = (int64_t)e.sy * ps.qy + jy - e.py;
        const int64_t ox = (int64_t)e.sx * ps.qx + jx - e.px;
        if (oy < 0 || oy >= e.Hout || ox < 0 || ox >= e.Wout) continue;
        const float bias = e.bias ? load_io(e.bias, oc, e.out_bf16) : 0.0f;
        const float val = leaky(v[i] + bias, slope_eff, use_min);
        const int64_t o = staged_row(e, ps.b, oy, ox) * e.ys_cpad + oc;
        if (e.out_bf16) {
            store_channels<__nv_bfloat16, 1>(static_cast<__nv_bfloat16 *>(e.y) + o, &val, e);
        } else {
            store_channels<float, 1>(static_cast<float *>(e.y) + o, &val, e);
        }
    }
}

// Output stage for the accumulator columns r0 .. r0+31 (r0 a multiple of 32) of one phase
// position per lane: v[i] = D[n, r0 + i].  Warp-collective: all 32 lanes of the warp call
// it together with the same r0, each with its own position.  kChain compiles in the chained
// output (EpiParams::out_staged); kernels without it keep their register budget.
template <bool kChain>
__device__ __forceinline__ void emit_cols(const float (&v)[32], const PosInfo &ps, int64_t r0,
                                          const EpiParams &e, int lane) {
    if (kChain && e.out_staged && e.pm_tc) {
#define CTR_PM(TCR)                                                        \
    if (e.out_bf16)                                                        \
        emit_pm_chain<__nv_bfloat16, TCR>(v, ps, r0, e, lane);             \
    else                                                                   \
        emit_pm_chain<float, TCR>(v, ps, r0, e, lane);                     \
    return
        switch (e.pm_tc >= 32 ? 32 : e.pm_tc) {
            case 2: CTR_PM(2);
            case 4: CTR_PM(4);
            case 8: CTR_PM(8);
            case 16: CTR_PM(16);
            default: CTR_PM(32);
        }
#undef CTR_PM
    }
    if (kChain && e.out_staged) {
#define CTR_CHAIN(SX, SY)                                                  \
    if (e.out_bf16)                                                        \
        emit_small_chain<__nv_bfloat16, SX, SY>(v, ps, r0, e, lane);       \
    else                                                                   \
        emit_small_chain<float, SX, SY>(v, ps, r0, e, lane);               \
    return
        switch (e.kind) {
            case EPI_KIND_1D_S1: CTR_CHAIN(1, 1);
            case EPI_KIND_1D_S2: CTR_CHAIN(2, 1);
            case EPI_KIND_1D_S4: CTR_CHAIN(4, 1);
            case EPI_KIND_1D_S8: CTR_CHAIN(8, 1);
            case EPI_KIND_2D_S2x2: CTR_CHAIN(2, 2);
            default:
                emit_generic_chain(v, ps, r0, e);
                return;
        }
#undef CTR_CHAIN
    }
#define CTR_SMALL(SX, SY)                                                  \
    if (e.out_bf16)                                                        \
        emit_small<__nv_bfloat16, SX, SY>(v, ps, r0, e, lane);             \
    else                                                                   \
        emit_small<float, SX, SY>(v, ps, r0, e, lane);                     \
    return
    switch (e.kind) {
        case EPI_KIND_1D_S1: CTR_SMALL(1, 1);
        case EPI_KIND_1D_S2: CTR_SMALL(2, 1);
        case EPI_KIND_1D_S4: CTR_SMALL(4, 1);
        case EPI_KIND_1D_S8: CTR_SMALL(8, 1);
        case EPI_KIND_1D_S16: CTR_SMALL(16, 1);
        case EPI_KIND_1D_S32: CTR_SMALL(32, 1);
        case EPI_KIND_2D_S2x2: CTR_SMALL(2, 2);
        case EPI_KIND_2D_S4x4: CTR_SMALL(4, 4);
        case EPI_KIND_1D_LARGE:
            if (e.out_bf16)
                emit_large<__nv_bfloat16>(v, ps, r0, e, lane);
            else
                emit_large<float>(v, ps, r0, e, lane);
            return;
        default:
            emit_generic(v, ps, r0, e);
            return;
    }
#undef CTR_SMALL
}

}  // namespace ctr
