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
#include <cuda_fp16.h>

#include "ctr_internal.h"
#include "ptx.cuh"

namespace ctr {

// ------------------------------------------------------------ I/O element types
// fp32, bf16 and fp16 values: conversions from fp32 round to nearest, ties to even.
template <typename T> __device__ __forceinline__ T io_from_float(float v);
template <> __device__ __forceinline__ float io_from_float<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 io_from_float<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}
template <> __device__ __forceinline__ __half io_from_float<__half>(float v) {
    return __float2half_rn(v);
}
// Two 16-bit values in one 32-bit word, a in the low half.
template <typename T> __device__ __forceinline__ uint32_t io_pack2(float a, float b);
template <> __device__ __forceinline__ uint32_t io_pack2<__nv_bfloat16>(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
template <> __device__ __forceinline__ uint32_t io_pack2<__half>(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
// The low and high 16-bit values of a word, as fp32 (exact).
template <typename T> __device__ __forceinline__ float io_lo(uint32_t w);
template <typename T> __device__ __forceinline__ float io_hi(uint32_t w);
template <> __device__ __forceinline__ float io_lo<__nv_bfloat16>(uint32_t w) {
    return __uint_as_float(w << 16);
}
template <> __device__ __forceinline__ float io_hi<__nv_bfloat16>(uint32_t w) {
    return __uint_as_float(w & 0xFFFF0000u);
}
template <> __device__ __forceinline__ float io_lo<__half>(uint32_t w) {
    return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu)));
}
template <> __device__ __forceinline__ float io_hi<__half>(uint32_t w) {
    return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
}

__device__ __forceinline__ float load_io(const void *p, int64_t i, int io) {
    if (io == IO_BF16) return __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i]);
    if (io == IO_F16) return __half2float(static_cast<const __half *>(p)[i]);
    return static_cast<const float *>(p)[i];
}

__device__ __forceinline__ void store_io(void *p, int64_t i, float v, int io) {
    if (io == IO_BF16)
        static_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(v);
    else if (io == IO_F16)
        static_cast<__half *>(p)[i] = __float2half_rn(v);
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
                for (int i = 0; i < N; i += 2) u[i / 2] = io_pack2<T>(vals[i], vals[i + 1]);
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
        for (int i = 0; i < N; ++i) dst[i] = io_from_float<T>(vals[i]);
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
            if (x0 + i >= 0 && x0 + i < e.Wout) dst[i] = io_from_float<T>(t[i]);
    }
}

// Bias of channel oc0 + lane for the first `count` lanes (0 elsewhere), so that a warp can
// share a chunk's biases by shuffles: one load per lane, issued before any output store.
__device__ __forceinline__ float lane_bias(const EpiParams &e, int64_t oc0, int count, int lane) {
    return (e.bias && lane < count && oc0 + lane < e.C_out) ? load_io(e.bias, oc0 + lane, e.io)
                                                            : 0.0f;
}

__device__ __forceinline__ float slope_of(const EpiParams &e) {
    return e.act == CTR_ACT_LEAKY_RELU ? e.slope : 1.0f;
}

// ------------------------------------------------------------ fast chunk output
// Most chunks lie wholly inside the output: their channels exist and every lane's outputs
// are inside the output rows and columns.  The warp then takes a straight-line path, in
// place on the accumulator values: per block of channels whose biases fill one vector load
// (the same address on every lane: a broadcast), the bias is added, the activation applied
// and every run stored at a compile-time width.  No per-channel or per-run branches, so the
// compiler can interleave the channels' independent arithmetic and stores.  Other chunks
// take the element-wise paths.

// Biases of channels oc0 .. oc0+N-1 (all inside C_out) in one load of N * sizeof(T) <= 16
// bytes, or zeros.  oc0 is a multiple of N (a power of two) and the bias pointer 16-byte
// aligned, so the load is aligned.
template <typename T, int N>
__device__ __forceinline__ void load_bias_vec(const EpiParams &e, int64_t oc0, float (&b)[N]) {
    static_assert(N * sizeof(T) <= 16, "one vector load");
    if (!e.bias) {
#pragma unroll
        for (int i = 0; i < N; ++i) b[i] = 0.0f;
        return;
    }
    const T *src = static_cast<const T *>(e.bias) + oc0;
    if constexpr (sizeof(T) == 2 && N == 8) {
        const uint4 q = __ldg(reinterpret_cast<const uint4 *>(src));
        const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            b[2 * k] = io_lo<T>(w4[k]);
            b[2 * k + 1] = io_hi<T>(w4[k]);
        }
    } else if constexpr (sizeof(T) == 2 && N == 4) {
        const uint2 q = __ldg(reinterpret_cast<const uint2 *>(src));
        b[0] = io_lo<T>(q.x);
        b[1] = io_hi<T>(q.x);
        b[2] = io_lo<T>(q.y);
        b[3] = io_hi<T>(q.y);
    } else if constexpr (sizeof(T) == 4 && N == 4) {
        const float4 q = __ldg(reinterpret_cast<const float4 *>(src));
        b[0] = q.x;
        b[1] = q.y;
        b[2] = q.z;
        b[3] = q.w;
    } else if constexpr (sizeof(T) == 4 && N == 2) {
        const float2 q = __ldg(reinterpret_cast<const float2 *>(src));
        b[0] = q.x;
        b[1] = q.y;
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) b[i] = static_cast<float>(src[i]);
    }
}

// Channels per bias load: as many as fill 16 bytes, at most G.
template <typename T, int G>
__host__ __device__ constexpr int bias_block() {
    return G < (int)(16 / sizeof(T)) ? G : (int)(16 / sizeof(T));
}

// v[i] = act(v[i] + bias) for the n values at v (ACT: LeakyReLU with slope sl).
template <bool ACT, int N>
__device__ __forceinline__ void add_bias_act(float *v, float bias, float sl) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const float a = v[i] + bias;
        v[i] = ACT ? (a < 0.0f ? a * sl : a) : a;
    }
}

// N consecutive outputs at dst as VW-byte stores (dst VW-aligned).
template <typename T, int N, int VW>
__device__ __forceinline__ void store_vec(T *dst, const float *vals) {
    constexpr int kPer = VW / (int)sizeof(T);   // elements per store
    static_assert(N % kPer == 0, "run length is a multiple of the store width");
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int i = 0; i < N; i += kPer) {
            if constexpr (kPer == 4)
                *reinterpret_cast<float4 *>(dst + i) =
                    make_float4(vals[i], vals[i + 1], vals[i + 2], vals[i + 3]);
            else if constexpr (kPer == 2)
                *reinterpret_cast<float2 *>(dst + i) = make_float2(vals[i], vals[i + 1]);
            else
                dst[i] = vals[i];
        }
    } else {
        if constexpr (kPer == 1) {
#pragma unroll
            for (int i = 0; i < N; ++i) dst[i] = io_from_float<T>(vals[i]);
        } else {
            uint32_t u[N / 2];
#pragma unroll
            for (int i = 0; i < N; i += 2) u[i / 2] = io_pack2<T>(vals[i], vals[i + 1]);
#pragma unroll
            for (int i = 0; i < N / 2; i += kPer / 2) {
                if constexpr (kPer == 8)
                    *reinterpret_cast<uint4 *>(dst + 2 * i) =
                        make_uint4(u[i], u[i + 1], u[i + 2], u[i + 3]);
                else if constexpr (kPer == 4)
                    *reinterpret_cast<uint2 *>(dst + 2 * i) = make_uint2(u[i], u[i + 1]);
                else
                    *reinterpret_cast<uint32_t *>(dst + 2 * i) = u[i];
            }
        }
    }
}

// The whole-chunk output of emit_small: G = 32/S channels of SY runs of SX outputs each, the
// runs of channel g at dst + g*cstride + jy*wout, stored VW bytes at a time.
template <typename T, int SX, int SY, int VW, bool ACT>
__device__ __forceinline__ void small_chunk_fast(float (&v)[32], T *__restrict__ dst, int64_t oc0,
                                                 int64_t cstride, int64_t wout,
                                                 const EpiParams &e) {
    constexpr int S = SX * SY, G = 32 / S, GB = bias_block<T, G>();
#pragma unroll
    for (int g0 = 0; g0 < G; g0 += GB) {
        float b[GB];
        load_bias_vec<T, GB>(e, oc0 + g0, b);
#pragma unroll
        for (int g = 0; g < GB; ++g) {
            add_bias_act<ACT, S>(&v[(g0 + g) * S], b[g], e.slope);
#pragma unroll
            for (int jy = 0; jy < SY; ++jy)
                store_vec<T, SX, VW>(dst + (g0 + g) * cstride + jy * wout, &v[(g0 + g) * S + jy * SX]);
        }
    }
}

template <typename T, int SX, int SY, int VW>
__device__ __forceinline__ void small_chunk_fast_act(float (&v)[32], T *__restrict__ dst,
                                                     int64_t oc0, int64_t cstride, int64_t wout,
                                                     const EpiParams &e) {
    if (e.act == CTR_ACT_LEAKY_RELU)
        small_chunk_fast<T, SX, SY, VW, true>(v, dst, oc0, cstride, wout, e);
    else
        small_chunk_fast<T, SX, SY, VW, false>(v, dst, oc0, cstride, wout, e);
}

// Stride-2 columns with an odd px: a thread's two outputs of a row start at the odd column
// x0 = 2 qx - px, so neither they nor any pair of them is aligned for a 2-element store.
// Consecutive lanes hold consecutive qx of one output row, so the aligned pair (x0 + 1,
// x0 + 2) is this lane's second output and the next lane's first: each lane takes its right
// neighbour's first value by a shuffle and stores the pair at the even column x0 + 1.  A
// first output no left neighbour covers (lane 0, qx = 0, or a neighbour whose pair fell
// outside the row), and a second output with no pair, are stored alone.  Needs an even Wout
// and y aligned to two elements (every pair column is then aligned); every lane runs the
// channel and row loops for the shuffles, stores are predicated per lane.
template <typename T, int SY>
__device__ __forceinline__ void emit_small_shift2(float (&v)[32], const PosInfo &ps, int64_t r0,
                                                  const EpiParams &e, int lane) {
    constexpr int S = 2 * SY, G = 32 / S;
    const int64_t oc0 = r0 / S;
    const int64_t x0 = 2 * ps.qx - e.px;
    const int64_t oy0 = (int64_t)SY * ps.qy - e.py;
    // The next lane holds qx + 1 of the same row when both positions are valid and qx + 1
    // is a valid column position (Qvx <= the row pitch Px, so the row does not change).  The
    // neighbour's own flag is asked for: a caller may mark positions invalid beyond what
    // decode_pos knows (the end of a tile that does not end a row).
    const bool next_valid = __shfl_down_sync(0xffffffffu, ps.valid, 1);
    const bool next_adj = ps.valid && next_valid && lane < 31 && ps.qx + 1 < e.Qvx;
    const bool pair = next_adj && x0 + 1 >= 0 && x0 + 2 < e.Wout;
    const bool prev_pair = __shfl_up_sync(0xffffffffu, pair, 1) && lane > 0;
    const bool first = ps.valid && !prev_pair && x0 >= 0 && x0 < e.Wout;
    const bool second = ps.valid && !pair && x0 + 1 >= 0 && x0 + 1 < e.Wout;
    const bool any_single = __any_sync(0xffffffffu, first || second);
    const float bl = lane_bias(e, oc0, G, lane);
    const float slope_eff = slope_of(e);
    const bool use_min = slope_eff > 1.0f;
    const int64_t g_left = e.C_out - oc0;
    const int gmax = g_left < G ? (int)g_left : G;
    bool row_ok[SY];
#pragma unroll
    for (int jy = 0; jy < SY; ++jy) row_ok[jy] = ps.valid && oy0 + jy >= 0 && oy0 + jy < e.Hout;
    const int64_t cstride = e.Hout * e.Wout;
    T *__restrict__ dst = static_cast<T *>(e.y) + ((ps.b * e.C_out + oc0) * e.Hout + oy0) * e.Wout + x0;
#pragma unroll
    for (int g = 0; g < G; ++g, dst += cstride) {
        if (g >= gmax) break;
        const float bias = __shfl_sync(0xffffffffu, bl, g);
#pragma unroll
        for (int jy = 0; jy < SY; ++jy) {
            const float a = leaky(v[g * S + 2 * jy] + bias, slope_eff, use_min);
            const float b = leaky(v[g * S + 2 * jy + 1] + bias, slope_eff, use_min);
            const float n = __shfl_down_sync(0xffffffffu, a, 1);
            T *row = dst + jy * e.Wout;
            if (row_ok[jy]) {
                if (pair) {
                    const float pv[2] = {b, n};
                    store_vec<T, 2, 2 * (int)sizeof(T)>(row + 1, pv);
                }
                if (any_single) {
                    if (first) row[0] = io_from_float<T>(a);
                    if (second) row[1] = io_from_float<T>(b);
                }
            }
        }
    }
}

// Output stage for whole phase sets: S = S_pad = SX * SY <= 32 (SX, SY compile-time), so the
// 32 columns r0 .. r0+31 of a chunk are G = 32/S whole channels.  Warp-collective: every
// lane passes the same r0 (its own position in ps).
template <typename T, int SX, int SY>
__device__ __forceinline__ void emit_small(float (&v)[32], const PosInfo &ps, int64_t r0,
                                           const EpiParams &e, int lane) {
    constexpr int S = SX * SY;
    constexpr int G = 32 / S;
    constexpr int kRunBytes = SX * (int)sizeof(T);
    const int64_t oc0 = r0 / S;
    if constexpr (SX == 2) {
        if (e.shift2) {
            emit_small_shift2<T, SY>(v, ps, r0, e, lane);
            return;
        }
    }
    {
        const int64_t fx0 = (int64_t)SX * ps.qx - e.px, fy0 = (int64_t)SY * ps.qy - e.py;
        const bool inside = ps.valid && fx0 >= 0 && fx0 + SX <= e.Wout && fy0 >= 0 &&
                            fy0 + SY <= e.Hout;
        if (__all_sync(0xffffffffu, inside) && oc0 + G <= e.C_out) {
            T *dst = static_cast<T *>(e.y) + ((ps.b * e.C_out + oc0) * e.Hout + fy0) * e.Wout + fx0;
            const int64_t cs = e.Hout * e.Wout;
            if constexpr (kRunBytes % 16 == 0) {
                if (e.store_bytes == 16) {
                    small_chunk_fast_act<T, SX, SY, 16>(v, dst, oc0, cs, e.Wout, e);
                    return;
                }
            }
            if constexpr (kRunBytes % 8 == 0) {
                if (e.store_bytes == 8) {
                    small_chunk_fast_act<T, SX, SY, 8>(v, dst, oc0, cs, e.Wout, e);
                    return;
                }
            }
            if constexpr (kRunBytes % 4 == 0 && sizeof(T) == 2) {
                if (e.store_bytes == 4) {
                    small_chunk_fast_act<T, SX, SY, 4>(v, dst, oc0, cs, e.Wout, e);
                    return;
                }
            }
            small_chunk_fast_act<T, SX, SY, (int)sizeof(T)>(v, dst, oc0, cs, e.Wout, e);
            return;
        }
    }
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
        const float bias = e.bias ? load_io(e.bias, oc, e.io) : 0.0f;
        const float a = v[i] + bias;
        store_io(e.y, ((ps.b * e.C_out + oc) * e.Hout + oy) * e.Wout + ox,
                 a < 0.0f ? a * slope_eff : a, e.io);
    }
}

// ------------------------------------------------------------ chained output
// The same outputs written into the next plan's staged input (EpiParams::out_staged):
// channels-last, so the G channels of one output position are G consecutive elements.
// fp32 values are split into the tf32 and cross planes exactly as the staging kernel does.

// Row of the staged buffer holding output (b, oy, ox).
__device__ __forceinline__ int64_t staged_row(const EpiParams &e, int64_t b, int64_t oy,
                                              int64_t ox) {
    return (b * e.ys_Py + oy + e.ys_hy) * e.ys_Px + ox + e.ys_hx;
}

// N consecutive channel values at dst (N * sizeof(T)-aligned): one plane for 16-bit types;
// for fp32 the tf32 and cross planes of a staged operand, or the values of a channels-last y.
template <typename T, int N>
__device__ __forceinline__ void store_channels(T *dst, const float *vals, const EpiParams &e) {
    constexpr int kBytes = N * (int)sizeof(T) < 16 ? N * (int)sizeof(T) : 16;
    if constexpr (sizeof(T) == 2) {
        store_run<T, N>(dst, vals, kBytes);
    } else {
        if (!e.ys_tf32) {   // a channels-last y: the values themselves
            store_run<T, N>(dst, vals, kBytes);
            return;
        }
        float hi[N], cr[N];
#pragma unroll
        for (int i = 0; i < N; ++i) {
            uint32_t c;
            hi[i] = ptx::split_x(vals[i], c);
            cr[i] = __uint_as_float(c);
        }
        store_run<T, N>(dst, hi, kBytes);
        store_run<T, N>(dst + e.ys_lo, cr, kBytes);
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

// The whole-chunk output of emit_pm_chain: NJ = 32/TCR phases starting at phase (jy0, jx0),
// each a run of TCR channel values at one position of the staged input.
template <typename T, int TCR, bool ACT>
__device__ __forceinline__ void pm_chain_fast(float (&v)[32], const PosInfo &ps, int jy0, int jx0,
                                              int64_t oc0, const EpiParams &e) {
    constexpr int NJ = 32 / TCR, GB = bias_block<T, TCR>();
    T *__restrict__ ys = static_cast<T *>(e.y);
    // Staged row of phase (jy, jx): ((ybase + jy) * ys_Px + xbase + jx).
    const int64_t ybase = ps.b * e.ys_Py + (int64_t)e.sy * ps.qy - e.py + e.ys_hy;
    const int64_t xbase = (int64_t)e.sx * ps.qx - e.px + e.ys_hx;
#pragma unroll
    for (int c0 = 0; c0 < TCR; c0 += GB) {
        float b[GB];
        load_bias_vec<T, GB>(e, oc0 + c0, b);
        int jy = jy0, jx = jx0;
#pragma unroll
        for (int jj = 0; jj < NJ; ++jj) {
#pragma unroll
            for (int i = 0; i < GB; ++i) add_bias_act<ACT, 1>(&v[jj * TCR + c0 + i], b[i], e.slope);
            const int64_t row = (ybase + jy) * e.ys_Px + xbase + jx;
            store_channels<T, GB>(ys + row * e.ys_cpad + oc0 + c0, &v[jj * TCR + c0], e);
            if (++jx == e.sx) {
                jx = 0;
                ++jy;
            }
        }
    }
}

// Phase-major rows (EpiParams::pm_tc): the chunk's 32 columns are NJ = 32 / TCR phases of
// TCR = min(pm_tc, 32) consecutive channels each, so every phase is one run of TCR channel
// values at one output position.
template <typename T, int TCR>
__device__ __forceinline__ void emit_pm_chain(float (&v)[32], const PosInfo &ps,
                                              int64_t r0, const EpiParams &e, int lane) {
    constexpr int NJ = 32 / TCR;
    const int tc = e.pm_tc;
    const int bn = tc * e.S_pad;
    const int64_t tile = r0 / bn;
    const int rl0 = (int)(r0 - tile * bn);
    const int j0 = rl0 / tc;
    const int64_t oc0 = tile * tc + (rl0 - j0 * tc);
    {
        // Fast path: all TCR channels exist and every phase of the chunk lands inside the
        // output for every lane.  The NJ phases are NJ runs of TCR channel values, stored per
        // block of channels whose biases fill one vector load.
        const int jy0 = j0 / e.sx, jx0 = j0 - jy0 * e.sx;
        bool inside = ps.valid;
        {
            int jy = jy0, jx = jx0;
#pragma unroll
            for (int jj = 0; jj < NJ; ++jj) {
                const int64_t oy = (int64_t)e.sy * ps.qy + jy - e.py;
                const int64_t ox = (int64_t)e.sx * ps.qx + jx - e.px;
                inside = inside && oy >= 0 && oy < e.Hout && ox >= 0 && ox < e.Wout;
                if (++jx == e.sx) {
                    jx = 0;
                    ++jy;
                }
            }
        }
        if (__all_sync(0xffffffffu, inside) && oc0 + TCR <= e.C_out) {
            if (e.act == CTR_ACT_LEAKY_RELU)
                pm_chain_fast<T, TCR, true>(v, ps, jy0, jx0, oc0, e);
            else
                pm_chain_fast<T, TCR, false>(v, ps, jy0, jx0, oc0, e);
            return;
        }
    }
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
        const float bias = e.bias ? load_io(e.bias, oc, e.io) : 0.0f;
        const float val = leaky(v[i] + bias, slope_eff, use_min);
        const int64_t o = staged_row(e, ps.b, oy, ox) * e.ys_cpad + oc;
        if (e.io == IO_BF16) {
            store_channels<__nv_bfloat16, 1>(static_cast<__nv_bfloat16 *>(e.y) + o, &val, e);
        } else if (e.io == IO_F16) {
            store_channels<__half, 1>(static_cast<__half *>(e.y) + o, &val, e);
        } else {
            store_channels<float, 1>(static_cast<float *>(e.y) + o, &val, e);
        }
    }
}

// Which output stages a kernel compiles: the torch-layout output, the chained output into the
// next plan's staged input (EpiParams::out_staged), or both; and for which I/O type.  A GEMM
// instantiation takes one of each (its precision fixes the type), so it keeps its register
// budget; the split-K reduce takes everything.
enum : int { kOutPlain = 1, kOutChain = 2, kOutBoth = 3 };
enum : int { kIoAny = 0, kIoF32 = 1, kIoBF16 = 2, kIoF16 = 3 };

// Output stage for the accumulator columns r0 .. r0+31 (r0 a multiple of 32) of one phase
// position per lane: v[i] = D[n, r0 + i] (overwritten).  Warp-collective: all 32 lanes of the
// warp call it together with the same r0, each with its own position.
template <int kOut, int kIo>
__device__ __forceinline__ void emit_cols(float (&v)[32], const PosInfo &ps, int64_t r0,
                                          const EpiParams &e, int lane) {
// CTR_IO(FN, (bf16, args...), (fp16, args...), (fp32, args...)): call FN<T, args...> for
// the kernel's I/O type(s).
#define CTR_IO_CALL(FN, TARGS) FN<CTR_IO_EXPAND TARGS>(v, ps, r0, e, lane)
#define CTR_IO_EXPAND(...) __VA_ARGS__
#define CTR_IO(FN, BF_ARGS, H_ARGS, F_ARGS)                                \
    do {                                                                   \
        if constexpr (kIo == kIoBF16) {                                    \
            CTR_IO_CALL(FN, BF_ARGS);                                      \
        } else if constexpr (kIo == kIoF16) {                              \
            CTR_IO_CALL(FN, H_ARGS);                                       \
        } else if constexpr (kIo == kIoF32) {                              \
            CTR_IO_CALL(FN, F_ARGS);                                       \
        } else if (e.io == IO_BF16) {                                      \
            CTR_IO_CALL(FN, BF_ARGS);                                      \
        } else if (e.io == IO_F16) {                                       \
            CTR_IO_CALL(FN, H_ARGS);                                       \
        } else {                                                           \
            CTR_IO_CALL(FN, F_ARGS);                                       \
        }                                                                  \
        return;                                                            \
    } while (0)
    if constexpr ((kOut & kOutChain) != 0) {
        if (kOut == kOutChain || e.out_staged) {
            if (e.pm_tc) {
                switch (e.pm_tc >= 32 ? 32 : e.pm_tc) {
                    case 2: CTR_IO(emit_pm_chain, (__nv_bfloat16, 2), (__half, 2), (float, 2));
                    case 4: CTR_IO(emit_pm_chain, (__nv_bfloat16, 4), (__half, 4), (float, 4));
                    case 8: CTR_IO(emit_pm_chain, (__nv_bfloat16, 8), (__half, 8), (float, 8));
                    case 16: CTR_IO(emit_pm_chain, (__nv_bfloat16, 16), (__half, 16), (float, 16));
                    default: CTR_IO(emit_pm_chain, (__nv_bfloat16, 32), (__half, 32), (float, 32));
                }
            }
            switch (e.kind) {
                case EPI_KIND_1D_S1: CTR_IO(emit_small_chain, (__nv_bfloat16, 1, 1), (__half, 1, 1), (float, 1, 1));
                case EPI_KIND_1D_S2: CTR_IO(emit_small_chain, (__nv_bfloat16, 2, 1), (__half, 2, 1), (float, 2, 1));
                case EPI_KIND_1D_S4: CTR_IO(emit_small_chain, (__nv_bfloat16, 4, 1), (__half, 4, 1), (float, 4, 1));
                case EPI_KIND_1D_S8: CTR_IO(emit_small_chain, (__nv_bfloat16, 8, 1), (__half, 8, 1), (float, 8, 1));
                case EPI_KIND_2D_S2x2: CTR_IO(emit_small_chain, (__nv_bfloat16, 2, 2), (__half, 2, 2), (float, 2, 2));
                default:
                    emit_generic_chain(v, ps, r0, e);
                    return;
            }
        }
    }
    if constexpr ((kOut & kOutPlain) != 0) {
        switch (e.kind) {
            case EPI_KIND_1D_S1: CTR_IO(emit_small, (__nv_bfloat16, 1, 1), (__half, 1, 1), (float, 1, 1));
            case EPI_KIND_1D_S2: CTR_IO(emit_small, (__nv_bfloat16, 2, 1), (__half, 2, 1), (float, 2, 1));
            case EPI_KIND_1D_S4: CTR_IO(emit_small, (__nv_bfloat16, 4, 1), (__half, 4, 1), (float, 4, 1));
            case EPI_KIND_1D_S8: CTR_IO(emit_small, (__nv_bfloat16, 8, 1), (__half, 8, 1), (float, 8, 1));
            case EPI_KIND_1D_S16: CTR_IO(emit_small, (__nv_bfloat16, 16, 1), (__half, 16, 1), (float, 16, 1));
            case EPI_KIND_1D_S32: CTR_IO(emit_small, (__nv_bfloat16, 32, 1), (__half, 32, 1), (float, 32, 1));
            case EPI_KIND_2D_S2x2: CTR_IO(emit_small, (__nv_bfloat16, 2, 2), (__half, 2, 2), (float, 2, 2));
            case EPI_KIND_2D_S4x4: CTR_IO(emit_small, (__nv_bfloat16, 4, 4), (__half, 4, 4), (float, 4, 4));
            case EPI_KIND_1D_LARGE: CTR_IO(emit_large, (__nv_bfloat16), (__half), (float));
            default:
                emit_generic(v, ps, r0, e);
                return;
        }
    }
#undef CTR_IO
#undef CTR_IO_CALL
#undef CTR_IO_EXPAND
}

}  // namespace ctr
