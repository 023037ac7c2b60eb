// epilogue.cuh -- output stage of the polyphase GEMM: bias, activation, the phase interleave
// and the padding slice, written from a 32-row x 32-column block of D staged in shared memory.
//
// "[XNNPACK] Lower dense transposed convs as one polyphase conv + depth to space" (Summary)
// computes every output phase with one stride-1 convolution, then interleaves the phases
// (a view/permute/view in 1-D, a block-major depth_to_space in 2-D) and slices off the
// padding.  Here the three steps are one pass: GEMM row r holds phase (jy, jx) of channel oc
// and GEMM column n holds phase position (b, qy, qx), so D[r, n] lands at
// y[b, oc, sy*qy + jy - py, sx*qx + jx - px] when that is inside the output.  The bias is
// added once, in fp32, before the activation and the single rounding to the I/O type
// ("[WebGPU] optimizations for audio models", review commit: f32 sums, bias bound once).
//
// Work split per warp: the warp owns 32 consecutive GEMM rows.  Rows with the same
// (oc, jy) and consecutive jx form a "row group" whose outputs are contiguous along x for a
// run of consecutive qx, so lanes walk (qx, jx) with jx fastest and write consecutive
// addresses.  Row groups are found once per tile (warp ballots); the column position is
// advanced incrementally, so the per-element work is a shift, a mask, a shared load and a
// store.
#pragma once

#include <cuda_bf16.h>

#include "ctr_internal.h"

namespace ctr {

// Column-major staging block: element (row i, column c) at sm[c * ld + i].  The pitch is a
// per-plan value, ld = 32 + (row-group length mod 32) when that is at most kEpiLdMax (it
// makes the output-order reads conflict-free), else 33; the raw (split-K / col2im) stores
// use ld = 33.
constexpr int kEpiLdMax = 48;

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

// The warp's 32 rows, decoded once per tile.  Lane i describes row r0 + i.  For the fast
// output path the warp also keeps, per row group g of nj rows, the group's bias and the
// offset of its first output element relative to the chunk's base (shared-memory tables
// `gbias` and `goff` of 32 entries per warp).
struct WarpRows {
    uint32_t start_mask;  // lanes whose row starts a row group
    uint32_t stop_mask;   // start_mask | invalid rows: a group ends before the next set bit
    int oc, jy, jx;
    float bias;
    float *gbias;   // per group: bias
    int *gjy;       // per group: phase row jy
    int *gjx;       // per group: first phase column jx
    int64_t *goff;  // per group: oc * Hout * Wout (output channel offset)
};

// Group tables of one warp in shared memory (32 entries each).
struct GroupTables {
    int64_t goff[32];
    float gbias[32];
    int gjy[32];
    int gjx[32];
};

__device__ __forceinline__ WarpRows warp_rows(int64_t r0, const EpiParams &e, int lane,
                                              GroupTables *tab) {
    WarpRows w;
    const int64_t r = r0 + lane;
    const int64_t oc = r / e.S_pad;
    const int j = (int)(r - oc * e.S_pad);
    const bool valid = oc < e.C_out && j < e.S;
    w.jy = j / e.sx;
    w.jx = j - w.jy * e.sx;
    w.oc = (int)oc;
    w.bias = (valid && e.bias) ? load_io(e.bias, oc, e.out_bf16) : 0.0f;
    const bool start = valid && (lane == 0 || w.jx == 0);
    w.start_mask = __ballot_sync(0xffffffffu, start);
    w.stop_mask = w.start_mask | __ballot_sync(0xffffffffu, !valid);
    w.gbias = tab->gbias;
    w.gjy = tab->gjy;
    w.gjx = tab->gjx;
    w.goff = tab->goff;
    if (e.fast) {
        // Row group g starts at lane g * nj.
        const int src = (lane << e.lg_nj) & 31;
        const int goc = __shfl_sync(0xffffffffu, w.oc, src);
        const int gjy_l = __shfl_sync(0xffffffffu, w.jy, src);
        const int gjx = __shfl_sync(0xffffffffu, w.jx, src);
        const float gb = __shfl_sync(0xffffffffu, w.bias, src);
        if (lane < (32 >> e.lg_nj)) {
            tab->gbias[lane] = gb;
            tab->gjy[lane] = gjy_l;
            tab->gjx[lane] = gjx;
            tab->goff[lane] = (int64_t)goc * e.Hout * e.Wout;
        }
        __syncwarp();
    }
    return w;
}

// Position of a GEMM column in the staged input: batch item, phase row, phase column.
struct ColCursor {
    int64_t b, qy, qx;
};

__device__ __forceinline__ ColCursor col_cursor(int64_t n0, const EpiParams &e) {
    ColCursor c;
    const int64_t plane = e.Py * e.Px;
    c.b = n0 / plane;
    const int64_t rem = n0 - c.b * plane;
    c.qy = rem / e.Px;
    c.qx = rem - c.qy * e.Px;
    return c;
}

__device__ __forceinline__ void col_advance(ColCursor &c, int64_t by, const EpiParams &e) {
    c.qx += by;
    while (c.qx >= e.Px) {
        c.qx -= e.Px;
        if (++c.qy == e.Py) {
            c.qy = 0;
            ++c.b;
        }
    }
}

// Outputs of one row group (rows i0 .. i0+njx-1: phases jx_lo.. of (oc, jy)) over block
// columns c0 .. c0+nq-1 (phase positions qx .. qx+nq-1 of (b, qy)).
__device__ __forceinline__ void emit_run(const float *sm, int ld, int i0, int njx, int c0, int nq,
                                         int64_t b, int oc, int jy, int jx_lo, int64_t qy,
                                         int64_t qx, float bias, const EpiParams &e, int lane) {
    const int64_t oy = (int64_t)e.sy * qy + jy - e.py;
    if (oy < 0 || oy >= e.Hout) return;
    const int64_t row_base = ((b * e.C_out + oc) * e.Hout + oy) * e.Wout;
    const int64_t ox0 = (int64_t)e.sx * qx + jx_lo - e.px;
    const int count = nq * njx;
    const float *src = sm + c0 * ld + i0;
    if ((njx & (njx - 1)) == 0) {
        const int sh = __ffs(njx) - 1;
        for (int t = lane; t < count; t += 32) {
            const int dq = t >> sh;
            const int dj = t & (njx - 1);
            const int64_t ox = ox0 + (int64_t)e.sx * dq + dj;
            if (ox >= 0 && ox < e.Wout)
                store_io(e.y, row_base + ox, apply_act(src[dq * ld + dj] + bias, e.act, e.slope),
                         e.out_bf16);
        }
    } else {
        // t / njx for t < 1024, njx <= 32: (t * ceil(2^16 / njx)) >> 16 is exact there.
        const uint32_t magic = (65536u + (uint32_t)njx - 1u) / (uint32_t)njx;
        for (int t = lane; t < count; t += 32) {
            const int dq = (int)(((uint32_t)t * magic) >> 16);
            const int dj = t - dq * njx;
            const int64_t ox = ox0 + (int64_t)e.sx * dq + dj;
            if (ox >= 0 && ox < e.Wout)
                store_io(e.y, row_base + ox, apply_act(src[dq * ld + dj] + bias, e.act, e.slope),
                         e.out_bf16);
        }
    }
}

// Fast output stage for a warp whose 32 rows are 32/NJ full row groups of NJ = min(sx, 32)
// rows (plans with e.fast set).  It writes the block columns [c_lo, c_hi), all phase
// positions of one staged row (b, qy) starting at column qx of block column 0.  Lane l owns
// phase dj = l & (NJ - 1) of every group and block columns dq = (l >> LG) + ii * (32 / NJ);
// its 32 outputs are independent and fully unrolled: a shared load, the bias/activation and
// one store each.  MASKED adds per-element checks of the column range and of the output x
// range (row edges, chunks that cross a staged row); unmasked calls need [c_lo, c_hi) =
// [0, 32) with every output x inside the row.  Groups whose output row y is outside the
// output are skipped.
template <int LG, bool MASKED, typename T>
__device__ __forceinline__ void emit_fast_t(const float *__restrict__ sm, int ld,
                                            const float *__restrict__ gbias,
                                            const int *__restrict__ gjy,
                                            const int *__restrict__ gjx,
                                            const int64_t *__restrict__ goff,
                                            int64_t lane_base, int64_t ox_lane, int64_t ox_step,
                                            int64_t oy0, const EpiParams &e, int c_lo, int c_hi,
                                            int lane) {
    constexpr int NJ = 1 << LG;
    constexpr int G = 32 >> LG;
    constexpr int QSTEP = 32 >> LG;
    const int dq0 = lane >> LG;
    const float *src = sm + dq0 * ld + (lane & (NJ - 1));
    const int src_step = QSTEP * ld;
    T *__restrict__ y = static_cast<T *>(e.y);
    // All staged values first, so no shared load waits behind a global store.
    float v[32];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int ii = 0; ii < NJ; ++ii) v[g * NJ + ii] = src[g * NJ + ii * src_step];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const int64_t oy = oy0 + gjy[g];
        if (oy < 0 || oy >= e.Hout) continue;
        const float bg = gbias[g];
        const int jx = gjx[g];
        T *dst = y + (lane_base + goff[g] + oy * e.Wout + jx);
#pragma unroll
        for (int ii = 0; ii < NJ; ++ii) {
            if (MASKED) {
                const int dq = dq0 + ii * QSTEP;
                const int64_t ox = ox_lane + jx + ii * ox_step;
                if (dq < c_lo || dq >= c_hi || ox < 0 || ox >= e.Wout) continue;
            }
            float t = v[g * NJ + ii] + bg;
            if (e.act == CTR_ACT_LEAKY_RELU && t < 0.0f) t *= e.slope;
            if constexpr (sizeof(T) == 2)
                dst[ii * ox_step] = __float2bfloat16_rn(t);
            else
                dst[ii * ox_step] = t;
        }
    }
}

template <bool MASKED, typename T>
__device__ __forceinline__ void emit_fast(const float *sm, const WarpRows &rows, int64_t b,
                                          int64_t qy, int64_t qx, const EpiParams &e,
                                          int c_lo, int c_hi, int lane) {
    const int lg = e.lg_nj;
    const int dj = lane & ((1 << lg) - 1);
    const int dq0 = lane >> lg;
    // x of this lane's first element before the group's jx; the channel/jy part of the
    // address comes from the group tables, the row part from oy.
    const int64_t ox_lane = (int64_t)e.sx * (qx + dq0) + dj - e.px;
    const int64_t lane_base = b * e.C_out * e.Hout * e.Wout + ox_lane;
    const int64_t ox_step = (int64_t)e.sx * (32 >> lg);
    const int64_t oy0 = (int64_t)e.sy * qy - e.py;
    const int ld = e.epi_ld;
#define CTR_EMIT_FAST(L)                                                                          \
    emit_fast_t<L, MASKED, T>(sm, ld, rows.gbias, rows.gjy, rows.gjx, rows.goff, lane_base,     \
                              ox_lane, ox_step, oy0, e, c_lo, c_hi, lane)
    switch (lg) {
        case 0: CTR_EMIT_FAST(0); break;
        case 1: CTR_EMIT_FAST(1); break;
        case 2: CTR_EMIT_FAST(2); break;
        case 3: CTR_EMIT_FAST(3); break;
        case 4: CTR_EMIT_FAST(4); break;
        default: CTR_EMIT_FAST(5); break;
    }
#undef CTR_EMIT_FAST
}

// 16 bytes of output from 16/sizeof(T) consecutive fp32 values, rounded to T.
template <typename T>
__device__ __forceinline__ uint4 pack16(const float *v) {
    uint4 u;
    if constexpr (sizeof(T) == 2) {
        __nv_bfloat162 p0 = __floats2bfloat162_rn(v[0], v[1]);
        __nv_bfloat162 p1 = __floats2bfloat162_rn(v[2], v[3]);
        __nv_bfloat162 p2 = __floats2bfloat162_rn(v[4], v[5]);
        __nv_bfloat162 p3 = __floats2bfloat162_rn(v[6], v[7]);
        u.x = *reinterpret_cast<uint32_t *>(&p0);
        u.y = *reinterpret_cast<uint32_t *>(&p1);
        u.z = *reinterpret_cast<uint32_t *>(&p2);
        u.w = *reinterpret_cast<uint32_t *>(&p3);
    } else {
        u.x = __float_as_uint(v[0]);
        u.y = __float_as_uint(v[1]);
        u.z = __float_as_uint(v[2]);
        u.w = __float_as_uint(v[3]);
    }
    return u;
}

// Vector output stage of an interior chunk whose row groups are whole phase sets
// (nj = sx <= 32): the outputs of group g over the chunk are the contiguous range
// [out_lo, out_lo + 32*nj) of one output row, element e <-> (dq, dj) = (e >> lg, e & (nj-1))
// <-> staged value sm[dq * ld + g*nj + dj].  The range is written as 16-byte aligned vector
// stores (VE = 16/sizeof(T) elements per lane) plus a scalar head and tail up to the next
// 16-byte boundary; requires Wout % VE == 0 so every group has the same head.
template <typename T>
__device__ __forceinline__ void emit_vec(const float *__restrict__ sm, const WarpRows &rows,
                                         const ColCursor &cur, const EpiParams &e, int lane) {
    constexpr int VE = 16 / (int)sizeof(T);
    const int lg = e.lg_nj, nj = e.nj, ld = e.epi_ld;
    const int G = 32 >> lg;
    const int L = 32 * nj;                                        // elements per group
    const int64_t out_lo = (int64_t)e.sx * cur.qx - e.px;         // x of element 0
    const int64_t row0 = cur.b * e.C_out * e.Hout * e.Wout + ((int64_t)e.sy * cur.qy - e.py) * e.Wout;
    const int head = (int)((VE - ((row0 + out_lo) & (VE - 1))) & (VE - 1));
    const int nvec = (L - head) / VE;
    const int tail0 = head + nvec * VE;                            // first tail element
    const int nsc = head + (L - tail0);                            // scalars per group
    T *__restrict__ y = static_cast<T *>(e.y);
    auto value = [&](int g, int el) -> float {
        const float t = sm[(el >> lg) * ld + g * nj + (el & (nj - 1))] + rows.gbias[g];
        return (e.act == CTR_ACT_LEAKY_RELU && t < 0.0f) ? t * e.slope : t;
    };
    auto gbase = [&](int g) -> int64_t {
        return row0 + rows.goff[g] + (int64_t)rows.gjy[g] * e.Wout + rows.gjx[g] + out_lo;
    };
    // idx / d for idx < 2^10 and d <= 2^10: (idx * ceil(2^20 / d)) >> 20 is exact there.
    const uint32_t mv = nvec ? ((1u << 20) + (uint32_t)nvec - 1u) / (uint32_t)nvec : 0u;
    const int total = G * nvec;
    for (int idx = lane; idx < total; idx += 32) {
        const int g = (int)(((uint32_t)idx * mv) >> 20);
        const int k = idx - g * nvec;
        const int e0 = head + k * VE;
        float v[VE];
#pragma unroll
        for (int i = 0; i < VE; ++i) v[i] = value(g, e0 + i);
        *reinterpret_cast<uint4 *>(y + gbase(g) + e0) = pack16<T>(v);
    }
    if (nsc) {
        const uint32_t ms = ((1u << 20) + (uint32_t)nsc - 1u) / (uint32_t)nsc;
        for (int idx = lane; idx < G * nsc; idx += 32) {
            const int g = (int)(((uint32_t)idx * ms) >> 20);
            const int s = idx - g * nsc;
            const int el = s < head ? s : tail0 + (s - head);
            const float t = value(g, el);
            if constexpr (sizeof(T) == 2)
                y[gbase(g) + el] = __float2bfloat16_rn(t);
            else
                y[gbase(g) + el] = t;
        }
    }
}

// Write every output of the 32 x 32 block D[r0 .. r0+31, n0 .. n0+31] staged column-major
// in sm (pitch e.epi_ld).  `rows` describes r0 .. r0+31, `cur` the position of column n0.
// Called by all 32 lanes of a warp.
__device__ __forceinline__ void emit_block(const float *sm, const WarpRows &rows, ColCursor cur,
                                           const EpiParams &e, int lane) {
    const int ld = e.epi_ld;
    if (e.fast && rows.stop_mask == rows.start_mask) {
        // Uniform rows: every run of the chunk (one per staged row it touches) goes through
        // the fast path, unmasked when the whole chunk is interior.
        const bool interior = cur.b < e.B && cur.qy < e.Qvy && cur.qx + 32 <= e.Qvx &&
                              cur.qx + 32 <= e.Px && (int64_t)e.sx * cur.qx - e.px >= 0 &&
                              (int64_t)e.sx * (cur.qx + 32) - e.px <= e.Wout;
        if (interior) {
            const int ve = e.out_bf16 ? 8 : 4;
            const int64_t oy_lo = (int64_t)e.sy * cur.qy - e.py;
            if (e.sx <= 32 && e.Wout % ve == 0 && oy_lo >= 0 && oy_lo + e.sy <= e.Hout) {
                if (e.out_bf16)
                    emit_vec<__nv_bfloat16>(sm, rows, cur, e, lane);
                else
                    emit_vec<float>(sm, rows, cur, e, lane);
                return;
            }
            if (e.out_bf16)
                emit_fast<false, __nv_bfloat16>(sm, rows, cur.b, cur.qy, cur.qx, e, 0, 32, lane);
            else
                emit_fast<false, float>(sm, rows, cur.b, cur.qy, cur.qx, e, 0, 32, lane);
            return;
        }
        int c = 0;
        while (c < 32) {
            const int run = (int)min((int64_t)(32 - c), e.Px - cur.qx);
            if (cur.b < e.B && cur.qy < e.Qvy && cur.qx < e.Qvx) {
                const int nq = (int)min((int64_t)run, e.Qvx - cur.qx);
                // Block column c holds qx = cur.qx; block column 0 would hold cur.qx - c.
                if (e.out_bf16)
                    emit_fast<true, __nv_bfloat16>(sm, rows, cur.b, cur.qy, cur.qx - c, e, c,
                                                   c + nq, lane);
                else
                    emit_fast<true, float>(sm, rows, cur.b, cur.qy, cur.qx - c, e, c, c + nq,
                                           lane);
            }
            c += run;
            col_advance(cur, run, e);
        }
        return;
    }
    int c = 0;
    while (c < 32) {
        const int run = (int)min((int64_t)(32 - c), e.Px - cur.qx);
        if (cur.b < e.B && cur.qy < e.Qvy && cur.qx < e.Qvx) {
            const int nq = (int)min((int64_t)run, e.Qvx - cur.qx);
            uint32_t starts = rows.start_mask;
            while (starts) {
                const int i0 = __ffs(starts) - 1;
                starts &= starts - 1;
                const uint32_t after = i0 == 31 ? 0u : (0xffffffffu << (i0 + 1));
                const uint32_t stops = rows.stop_mask & after;
                const int njx = (stops ? __ffs(stops) - 1 : 32) - i0;
                const int oc = __shfl_sync(0xffffffffu, rows.oc, i0);
                const int jy = __shfl_sync(0xffffffffu, rows.jy, i0);
                const int jx = __shfl_sync(0xffffffffu, rows.jx, i0);
                const float bias = __shfl_sync(0xffffffffu, rows.bias, i0);
                emit_run(sm, ld, i0, njx, c, nq, cur.b, oc, jy, jx, cur.qy, cur.qx, bias, e, lane);
            }
        }
        c += run;
        col_advance(cur, run, e);
    }
}

}  // namespace ctr
