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

__device__ __forceinline__ PosInfo decode_pos(int64_t n, const EpiParams &e) {
    PosInfo p;
    const int64_t plane = e.Py * e.Px;
    p.b = n / plane;
    const int64_t rem = n - p.b * plane;
    p.qy = rem / e.Px;
    p.qx = rem - p.qy * e.Px;
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

// One run of NX phases (jx = 0 .. NX-1 of one (oc, jy)) starting at v[0]: bias, activation,
// then either vector stores (interior) or per-element stores with bounds checks (row edges).
template <typename T, int NX>
__device__ __forceinline__ void emit_run(T *__restrict__ y, int64_t row, int64_t x0,
                                         const float *v, float bias, const EpiParams &e,
                                         bool interior) {
    float t[NX];
#pragma unroll
    for (int i = 0; i < NX; ++i) t[i] = apply_act(v[i] + bias, e.act, e.slope);
    if (interior) {
        store_run<T, NX>(y + row + x0, t, e.store_bytes);
    } else {
#pragma unroll
        for (int i = 0; i < NX; ++i)
            if (x0 + i >= 0 && x0 + i < e.Wout) y[row + x0 + i] = static_cast<T>(t[i]);
    }
}

// Output stage for whole phase sets: S = S_pad = SX * SY <= 32 (SX, SY compile-time), so the
// 32 columns r0 .. r0+31 of a chunk are 32/S whole channels.
template <typename T, int SX, int SY>
__device__ __forceinline__ void emit_small(const float (&v)[32], const PosInfo &ps, int64_t r0,
                                           const EpiParams &e) {
    constexpr int S = SX * SY;
    constexpr int G = 32 / S;
    T *__restrict__ y = static_cast<T *>(e.y);
    const int64_t oc0 = r0 / S;
    const int64_t x0 = (int64_t)SX * ps.qx - e.px;
    const bool interior = x0 >= 0 && x0 + SX <= e.Wout;
    const int64_t oy0 = (int64_t)SY * ps.qy - e.py;
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const int64_t oc = oc0 + g;
        if (oc >= e.C_out) break;
        const float bias = e.bias ? load_io(e.bias, oc, e.out_bf16) : 0.0f;
        const int64_t chan = (ps.b * e.C_out + oc) * e.Hout;
#pragma unroll
        for (int jy = 0; jy < SY; ++jy) {
            const int64_t oy = oy0 + jy;
            if (oy < 0 || oy >= e.Hout) continue;
            emit_run<T, SX>(y, (chan + oy) * e.Wout, x0, &v[g * S + jy * SX], bias, e, interior);
        }
    }
}

// Output stage for 1-D plans with S = S_pad a multiple of 32: the 32 columns of a chunk are 32
// consecutive phases j0 .. j0+31 of one channel, i.e. 32 consecutive outputs.
template <typename T>
__device__ __forceinline__ void emit_large(const float (&v)[32], const PosInfo &ps, int64_t r0,
                                           const EpiParams &e) {
    T *__restrict__ y = static_cast<T *>(e.y);
    const int64_t oc = r0 / e.S_pad;
    if (oc >= e.C_out) return;
    const int64_t j0 = r0 - oc * e.S_pad;
    const int64_t x0 = (int64_t)e.sx * ps.qx + j0 - e.px;
    const bool interior = x0 >= 0 && x0 + 32 <= e.Wout;
    const float bias = e.bias ? load_io(e.bias, oc, e.out_bf16) : 0.0f;
    emit_run<T, 32>(y, (ps.b * e.C_out + oc) * e.Wout, x0, v, bias, e, interior);
}

// Any plan: every output element on its own, with the full index map and bounds checks.
__device__ __forceinline__ void emit_generic(const float (&v)[32], const PosInfo &ps, int64_t r0,
                                             const EpiParams &e) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int64_t r = r0 + i;
        const int64_t oc = r / e.S_pad;
        const int j = (int)(r - oc * e.S_pad);
        if (oc >= e.C_out || j >= e.S) continue;
        const int jy = j / e.sx, jx = j - (j / e.sx) * e.sx;
        const int64_t oy = (int64_t)e.sy * ps.qy + jy - e.py;
        const int64_t ox = (int64_t)e.sx * ps.qx + jx - e.px;
        if (oy < 0 || oy >= e.Hout || ox < 0 || ox >= e.Wout) continue;
        const float bias = e.bias ? load_io(e.bias, oc, e.out_bf16) : 0.0f;
        store_io(e.y, ((ps.b * e.C_out + oc) * e.Hout + oy) * e.Wout + ox,
                 apply_act(v[i] + bias, e.act, e.slope), e.out_bf16);
    }
}

// Output stage for the accumulator columns r0 .. r0+31 (r0 a multiple of 32) of one phase
// position: v[i] = D[n, r0 + i].  Each thread works on its own position.
__device__ __forceinline__ void emit_cols(const float (&v)[32], const PosInfo &ps, int64_t r0,
                                          const EpiParams &e) {
    if (!ps.valid) return;
#define CTR_SMALL(SX, SY)                                                  \
    if (e.out_bf16)                                                        \
        emit_small<__nv_bfloat16, SX, SY>(v, ps, r0, e);                   \
    else                                                                   \
        emit_small<float, SX, SY>(v, ps, r0, e);                           \
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
                emit_large<__nv_bfloat16>(v, ps, r0, e);
            else
                emit_large<float>(v, ps, r0, e);
            return;
        default:
            emit_generic(v, ps, r0, e);
            return;
    }
#undef CTR_SMALL
}

}  // namespace ctr
