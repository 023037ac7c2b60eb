// epilogue.cuh -- output stage of the polyphase GEMM: bias, activation, the phase interleave
// and the padding slice, written from a 32 x 32 block of D staged in shared memory.
//
// "[XNNPACK] Lower dense transposed convs as one polyphase conv + depth to space" (Summary)
// computes every output phase with one stride-1 convolution, then interleaves the phases
// (a view/permute/view in 1-D, a block-major depth_to_space in 2-D) and slices off the
// padding.  Here the three steps are one pass over registers: GEMM row r holds phase
// (jy, jx) of channel oc and GEMM column n holds phase position (b, qy, qx), so D[r, n]
// lands at y[b, oc, sy*qy + jy - py, sx*qx + jx - px] when that is inside the output.  The
// bias is added once, in fp32, before the activation and the single rounding to the I/O
// type ("[WebGPU] optimizations for audio models", review commit: f32 sums, bias bound once).
#pragma once

#include <cuda_bf16.h>

#include "ctr_internal.h"

namespace ctr {

constexpr int kEpiLd = 33;  // row pitch (floats) of a 32 x 32 staging block

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

// One run of outputs: rows i0 .. i0+njx-1 of the block (phases jx_lo .. jx_lo+njx-1 of
// (oc, jy)) times block columns c0 .. c0+nq-1 (phase positions qx .. qx+nq-1 of (b, qy)).
// Lanes walk (dq, dj) with dj fastest, so consecutive lanes write consecutive x.
__device__ __forceinline__ void emit_run(const float *sm, int i0, int njx, int c0, int nq,
                                         int64_t b, int64_t oc, int jy, int jx_lo, int64_t qy,
                                         int64_t qx, const EpiParams &e, float bval, int lane) {
    const int64_t oy = (int64_t)e.sy * qy + jy - e.py;
    if (oy < 0 || oy >= e.Hout) return;
    const int64_t row_base = ((b * e.C_out + oc) * e.Hout + oy) * e.Wout;
    const int64_t ox0 = (int64_t)e.sx * qx + jx_lo - e.px;
    const int count = nq * njx;
    // e / njx for e < 1024, njx <= 32: (e * ceil(2^16 / njx)) >> 16 is exact there.
    const uint32_t magic = (65536u + (uint32_t)njx - 1u) / (uint32_t)njx;
    for (int t = lane; t < count; t += 32) {
        const int dq = (int)(((uint32_t)t * magic) >> 16);
        const int dj = t - dq * njx;
        const int64_t ox = ox0 + (int64_t)e.sx * dq + dj;
        if (ox >= 0 && ox < e.Wout) {
            float v = sm[(i0 + dj) * kEpiLd + c0 + dq] + bval;
            store_io(e.y, row_base + ox, apply_act(v, e.act, e.slope), e.out_bf16);
        }
    }
}

// Write every output of the 32 x 32 block D[r0 .. r0+31, n0 .. n0+31] held in sm
// (sm[i * kEpiLd + c] = D[r0 + i, n0 + c]).  Called by all 32 lanes of a warp.
__device__ __forceinline__ void emit_block(const float *sm, int64_t r0, int64_t n0,
                                           const EpiParams &e, int lane) {
    // Column runs: maximal ranges of the block inside one staged row (b, qy).
    const int64_t plane = e.Py * e.Px;
    int64_t b = n0 / plane;
    int64_t rem = n0 - b * plane;
    int64_t qy = rem / e.Px;
    int64_t qx = rem - qy * e.Px;
    int c = 0;
    while (c < 32) {
        const int run = (int)min((int64_t)(32 - c), e.Px - qx);
        if (b < e.B && qy < e.Qvy && qx < e.Qvx) {
            const int nq = (int)min((int64_t)run, e.Qvx - qx);
            // Row groups: consecutive rows with the same (oc, jy).
            int i = 0;
            while (i < 32) {
                const int64_t r = r0 + i;
                const int64_t oc = r / e.S_pad;
                if (oc >= e.C_out) break;
                const int j = (int)(r - oc * e.S_pad);
                if (j >= e.S) {
                    i += e.S_pad - j;
                    continue;
                }
                const int jy = j / e.sx;
                const int jx_lo = j - jy * e.sx;
                const int njx = min(e.sx - jx_lo, 32 - i);
                const float bval = e.bias ? load_io(e.bias, oc, e.out_bf16) : 0.0f;
                emit_run(sm, i, njx, c, nq, b, oc, jy, jx_lo, qy, qx, e, bval, lane);
                i += njx;
            }
        }
        c += run;
        qx += run;
        if (qx == e.Px) {
            qx = 0;
            if (++qy == e.Py) {
                qy = 0;
                ++b;
            }
        }
    }
}

}  // namespace ctr
