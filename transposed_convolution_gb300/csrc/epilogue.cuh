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
    float *gbias;
    int64_t *goff;
};

__device__ __forceinline__ WarpRows warp_rows(int64_t r0, const EpiParams &e, int lane,
                                              float *gbias, int64_t *goff) {
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
    w.gbias = gbias;
    w.goff = goff;
    if (e.fast) {
        // Row group g starts at lane g * nj.
        const int src = (lane << e.lg_nj) & 31;
        const int goc = __shfl_sync(0xffffffffu, w.oc, src);
        const int gjy = __shfl_sync(0xffffffffu, w.jy, src);
        const int gjx = __shfl_sync(0xffffffffu, w.jx, src);
        const float gb = __shfl_sync(0xffffffffu, w.bias, src);
        if (lane < (32 >> e.lg_nj)) {
            gbias[lane] = gb;
            goff[lane] = ((int64_t)goc * e.Hout + gjy) * e.Wout + gjx;
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

// Fast output stage of a full chunk: all 32 columns are valid phase positions of one staged
// row, every output of the chunk lies inside the output, and the 32 rows are 32/NJ full
// row groups of NJ = min(sx, 32) rows (plans with e.fast set; checked per chunk by the
// caller).  Lane l owns phase dj = l & (NJ - 1) of every group and columns
// dq = (l >> LG) + ii * (32 / NJ); the 32 outputs of a lane are independent and fully
// unrolled, each a shared load, the bias/activation and one store.
template <int LG, typename T>
__device__ __forceinline__ void emit_fast_t(const float *__restrict__ sm, int ld,
                                            const float *__restrict__ gbias,
                                            const int64_t *__restrict__ goff, int64_t lane_base,
                                            int64_t ox_step, T *__restrict__ y, int act,
                                            float slope, int lane) {
    constexpr int NJ = 1 << LG;
    constexpr int G = 32 >> LG;
    constexpr int QSTEP = 32 >> LG;
    const float *src = sm + (lane >> LG) * ld + (lane & (NJ - 1));
    const int src_step = QSTEP * ld;
    // All staged values first, so no shared load waits behind a global store.
    float v[32];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int ii = 0; ii < NJ; ++ii) v[g * NJ + ii] = src[g * NJ + ii * src_step];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float bg = gbias[g];
        T *dst = y + (lane_base + goff[g]);
#pragma unroll
        for (int ii = 0; ii < NJ; ++ii) {
            float t = v[g * NJ + ii] + bg;
            if (act == CTR_ACT_LEAKY_RELU && t < 0.0f) t *= slope;
            if constexpr (sizeof(T) == 2)
                dst[ii * ox_step] = __float2bfloat16_rn(t);
            else
                dst[ii * ox_step] = t;
        }
    }
}

template <typename T>
__device__ __forceinline__ void emit_fast(const float *sm, const WarpRows &rows,
                                          const ColCursor &cur, const EpiParams &e, int lane) {
    const int lg = e.lg_nj;
    const int dj = lane & ((1 << lg) - 1);
    const int dq0 = lane >> lg;
    // Output element of (group 0 start, column qx, row jy = 0) plus this lane's offset.
    const int64_t chunk_base = (cur.b * e.C_out * e.Hout + (int64_t)e.sy * cur.qy - e.py) * e.Wout +
                               (int64_t)e.sx * cur.qx - e.px;
    const int64_t lane_base = chunk_base + (int64_t)e.sx * dq0 + dj;
    const int64_t ox_step = (int64_t)e.sx * (32 >> lg);
    T *y = static_cast<T *>(e.y);
    const int ld = e.epi_ld;
    switch (lg) {
        case 0: emit_fast_t<0, T>(sm, ld, rows.gbias, rows.goff, lane_base, ox_step, y, e.act, e.slope, lane); break;
        case 1: emit_fast_t<1, T>(sm, ld, rows.gbias, rows.goff, lane_base, ox_step, y, e.act, e.slope, lane); break;
        case 2: emit_fast_t<2, T>(sm, ld, rows.gbias, rows.goff, lane_base, ox_step, y, e.act, e.slope, lane); break;
        case 3: emit_fast_t<3, T>(sm, ld, rows.gbias, rows.goff, lane_base, ox_step, y, e.act, e.slope, lane); break;
        case 4: emit_fast_t<4, T>(sm, ld, rows.gbias, rows.goff, lane_base, ox_step, y, e.act, e.slope, lane); break;
        default: emit_fast_t<5, T>(sm, ld, rows.gbias, rows.goff, lane_base, ox_step, y, e.act, e.slope, lane); break;
    }
}

// Write every output of the 32 x 32 block D[r0 .. r0+31, n0 .. n0+31] staged column-major
// in sm (pitch e.epi_ld).  `rows` describes r0 .. r0+31, `cur` the position of column n0.
// Called by all 32 lanes of a warp.
__device__ __forceinline__ void emit_block(const float *sm, const WarpRows &rows, ColCursor cur,
                                           const EpiParams &e, int lane) {
    const int ld = e.epi_ld;
    if (e.fast && rows.stop_mask == rows.start_mask && cur.b < e.B && cur.qy < e.Qvy &&
        cur.qx + 32 <= e.Qvx && cur.qx + 32 <= e.Px) {
        // All rows valid and the chunk inside one staged row; the outputs must also lie
        // inside the output (the first/last chunks of a row, and phase rows near the top
        // and bottom edge, fall back to the general path).
        const int64_t ox_lo = (int64_t)e.sx * cur.qx - e.px;
        const int64_t ox_hi = (int64_t)e.sx * (cur.qx + 32) - e.px;
        const int64_t oy_lo = (int64_t)e.sy * cur.qy - e.py;
        const int64_t oy_hi = oy_lo + e.sy;
        if (ox_lo >= 0 && ox_hi <= e.Wout && oy_lo >= 0 && oy_hi <= e.Hout) {
            if (e.out_bf16)
                emit_fast<__nv_bfloat16>(sm, rows, cur, e, lane);
            else
                emit_fast<float>(sm, rows, cur, e, lane);
            return;
        }
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
