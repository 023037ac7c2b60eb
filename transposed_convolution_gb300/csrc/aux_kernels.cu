// aux_kernels.cu -- the non-tensor-core kernels of the library:
//   prepack      torch weight -> phase-major GEMM rows (polyphase) or (oc, tap) rows (col2im)
//   stage_x      NC(H)W input -> channels-last rows with zero halos (tf32 hi/lo or bf16)
//   splitk_reduce  fixed-order sum of split-K partials, then the fused output stage
//   col2im       gather of the valid taps from the fp32 column buffer
//   gather       direct ConvTranspose for tiny channel counts
//   fill_bias    y = bias (or zeros) for an empty input on the col2im path
//   copy_weight  the gather path's "packed" weight (a plain copy)
#include <algorithm>
#include <cuda_bf16.h>

#include "ctr_internal.h"
#include "epilogue.cuh"
#include "ptx.cuh"

namespace ctr {
namespace {

constexpr int kBlock = 256;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

unsigned grid_for(int64_t n, int block) {
    const int64_t g = ceil_div(n, block);
    return (unsigned)std::min<int64_t>(std::max<int64_t>(g, 1), (int64_t)1 << 30);
}

// Geometry of a plan as plain values for the kernels below (2-D form).
struct Geo {
    int64_t B, C_in, C_out;
    int64_t H, W, ky, kx, sy, sx, py, px, Ho, Wo;
    int act;
    float slope;
    int bf16;
};

Geo geo_of(const ctr_plan_s *pl) {
    Geo g;
    g.B = pl->B;
    g.C_in = pl->C_in;
    g.C_out = pl->C_out;
    g.H = pl->in[0];
    g.W = pl->in[1];
    g.ky = pl->k[0];
    g.kx = pl->k[1];
    g.sy = pl->s[0];
    g.sx = pl->s[1];
    g.py = pl->p[0];
    g.px = pl->p[1];
    g.Ho = pl->out[0];
    g.Wo = pl->out[1];
    g.act = pl->act;
    g.slope = pl->slope;
    g.bf16 = pl->dtype == CTR_BF16 ? 1 : 0;
    return g;
}

// -------------------------------------------------------------------------- gather
// y[b, oc, oy, ox] = bias[oc] + sum over ic and the taps that reach (oy, ox): a tap ty
// contributes when (oy + py - ty) is a multiple of sy and the quotient is a valid input row
// ("[ExecuTorch][WebGPU] Add optimized conv2d op", Implementation: the gather form with the
// un-flipped weight).  fp32 accumulation on CUDA cores; one thread per output element.
__global__ void gather_kernel(const void *__restrict__ x, const void *__restrict__ w,
                              const void *__restrict__ bias, void *__restrict__ y, Geo g,
                              int64_t total) {
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t ox = idx % g.Wo;
        int64_t t = idx / g.Wo;
        const int64_t oy = t % g.Ho;
        t /= g.Ho;
        const int64_t oc = t % g.C_out;
        const int64_t b = t / g.C_out;
        float acc = 0.0f;
        const int64_t ry = oy + g.py, rx = ox + g.px;
        for (int64_t ty = ry % g.sy; ty < g.ky; ty += g.sy) {
            const int64_t iy = (ry - ty) / g.sy;
            if (iy < 0) break;
            if (iy >= g.H) continue;
            for (int64_t tx = rx % g.sx; tx < g.kx; tx += g.sx) {
                const int64_t ix = (rx - tx) / g.sx;
                if (ix < 0) break;
                if (ix >= g.W) continue;
                const int64_t xoff = ((b * g.C_in) * g.H + iy) * g.W + ix;
                const int64_t woff = ((oc * g.ky) + ty) * g.kx + tx;
                const int64_t xstride = g.H * g.W;
                const int64_t wstride = g.C_out * g.ky * g.kx;
                for (int64_t ic = 0; ic < g.C_in; ++ic)
                    acc = fmaf(load_io(x, xoff + ic * xstride, g.bf16),
                               load_io(w, woff + ic * wstride, g.bf16), acc);
            }
        }
        if (bias) acc += load_io(bias, oc, g.bf16);
        store_io(y, idx, apply_act(acc, g.act, g.slope), g.bf16);
    }
}

__global__ void fill_bias_kernel(const void *__restrict__ bias, void *__restrict__ y, Geo g,
                                 int64_t total) {
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t oc = (idx / (g.Ho * g.Wo)) % g.C_out;
        const float v = bias ? load_io(bias, oc, g.bf16) : 0.0f;
        store_io(y, idx, apply_act(v, g.act, g.slope), g.bf16);
    }
}

__global__ void copy_bytes_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                  int64_t n16, const uint8_t *__restrict__ src_tail,
                                  uint8_t *__restrict__ dst_tail, int tail) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n16;
         i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
    if (blockIdx.x == 0 && (int)threadIdx.x < tail) dst_tail[threadIdx.x] = src_tail[threadIdx.x];
}

// -------------------------------------------------------------------------- prepack
struct PackGeo {
    int64_t M_pad, K_total, C_in_pad, C_in, C_out;
    int64_t ky, kx, sy, sx, my, mx;
    int S, S_pad;
    int polyphase;
    int bf16;
};

// Polyphase rows ("[XNNPACK] Lower dense transposed convs as one polyphase conv + depth to
// space", Summary: phase-major ordering, taps flipped within a phase):
//   A[r = oc*S_pad + jy*sx + jx, k = (uy*mx + ux)*C_in_pad + ic]
//       = w[ic, oc, sy*(my-1-uy) + jy, sx*(mx-1-ux) + jx]    (0 past the kernel: the kernel
//                                                               is zero-padded to m*s taps)
// col2im rows ("[WebGPU] optimizations for audio models", ConvTranspose commit: W[C_in,
// kH*kW*C_out] prepacked to the GEMM layout):  A[r = oc*S_pad + t, k = ic] = w[ic, oc, t].
// Padding rows and channels are zero.  fp32 weights are split into tf32 hi and lo planes.
__global__ void prepack_kernel(const void *__restrict__ w, void *__restrict__ wp, PackGeo pg) {
    const int64_t total = pg.M_pad * pg.K_total;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = idx / pg.K_total;
        const int64_t kk = idx - r * pg.K_total;
        const int64_t g = kk / pg.C_in_pad;
        const int64_t ic = kk - g * pg.C_in_pad;
        const int64_t oc = r / pg.S_pad;
        const int64_t j = r - oc * pg.S_pad;
        float v = 0.0f;
        if (oc < pg.C_out && j < pg.S && ic < pg.C_in) {
            int64_t ty, tx;
            if (pg.polyphase) {
                const int64_t jy = j / pg.sx, jx = j - (j / pg.sx) * pg.sx;
                const int64_t uy = g / pg.mx, ux = g - (g / pg.mx) * pg.mx;
                ty = pg.sy * (pg.my - 1 - uy) + jy;
                tx = pg.sx * (pg.mx - 1 - ux) + jx;
            } else {
                ty = j / pg.kx;
                tx = j - ty * pg.kx;
            }
            if (ty < pg.ky && tx < pg.kx)
                v = load_io(w, ((ic * pg.C_out + oc) * pg.ky + ty) * pg.kx + tx, pg.bf16);
        }
        if (pg.bf16) {
            static_cast<__nv_bfloat16 *>(wp)[idx] = __float2bfloat16_rn(v);  // exact: v is bf16
        } else {
            const float hi = ptx::to_tf32(v);
            const float lo = ptx::to_tf32(v - hi);
            static_cast<float *>(wp)[idx] = hi;
            static_cast<float *>(wp)[total + idx] = lo;
        }
    }
}

// -------------------------------------------------------------------------- stage_x
struct StageGeo {
    int64_t B, C_in, C_in_pad, H, W, Py, Px, hy, hx, N_total;
    int bf16;
};

// xs[n][c] with n = (b*Py + py')*Px + px': x[b, c, py' - hy, px' - hx] inside the input and
// c < C_in, zero elsewhere (the halos are the polyphase conv's padding m - 1).  A block
// moves 256 consecutive staged positions x 32 channels through shared memory: each warp
// reads 4 channels along positions (32 loads in flight per lane, coalesced along x) and
// then writes 32 positions along channels (coalesced along c).  Positions are decoded once
// per lane and advanced incrementally.  fp32 input is written as tf32 hi and lo planes.
constexpr int kStagePos = 256;

__global__ void __launch_bounds__(256) stage_x_kernel(const void *__restrict__ x,
                                                      void *__restrict__ xs, StageGeo sg) {
    __shared__ float tile[kStagePos][33];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t n0 = (int64_t)blockIdx.x * kStagePos;
    const int64_t c0 = (int64_t)blockIdx.y * 32;
    const int64_t plane = sg.Py * sg.Px;
    const int64_t hw = sg.H * sg.W;
    // This lane's first position and its staged coordinates.
    int64_t n = n0 + lane;
    int64_t b = n / plane;
    int64_t rem = n - b * plane;
    int64_t py = rem / sg.Px;
    int64_t px = rem - py * sg.Px;
    int64_t xoff[kStagePos / 32];  // x offset of channel 0 at each of the lane's positions, -1 = zero
#pragma unroll
    for (int j = 0; j < kStagePos / 32; ++j) {
        const int64_t yy = py - sg.hy, xx = px - sg.hx;
        const bool in = n + 32 * j < sg.N_total && yy >= 0 && yy < sg.H && xx >= 0 && xx < sg.W;
        xoff[j] = in ? (b * sg.C_in * sg.H + yy) * sg.W + xx : -1;
        px += 32;
        while (px >= sg.Px) {
            px -= sg.Px;
            if (++py == sg.Py) {
                py = 0;
                ++b;
            }
        }
    }
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
        const int ci = warp * 4 + cc;
        const int64_t c = c0 + ci;
        const bool cvalid = c < sg.C_in;
#pragma unroll
        for (int j = 0; j < kStagePos / 32; ++j) {
            float v = 0.0f;
            if (cvalid && xoff[j] >= 0) v = load_io(x, xoff[j] + c * hw, sg.bf16);
            tile[lane + 32 * j][ci] = v;
        }
    }
    __syncthreads();
    const int64_t lo_off = sg.N_total * sg.C_in_pad;
#pragma unroll 4
    for (int p = warp; p < kStagePos; p += 8) {
        const int64_t np = n0 + p;
        if (np >= sg.N_total) break;
        const int64_t o = np * sg.C_in_pad + c0 + lane;
        const float v = tile[p][lane];
        if (sg.bf16) {
            static_cast<__nv_bfloat16 *>(xs)[o] = __float2bfloat16_rn(v);
        } else {
            const float hi = ptx::to_tf32(v);
            static_cast<float *>(xs)[o] = hi;
            static_cast<float *>(xs)[lo_off + o] = ptx::to_tf32(v - hi);
        }
    }
}

// -------------------------------------------------------------------------- split-K reduce
// One thread per (phase position n, 32-row chunk r0): sums the split-K partials
// raw[z][n][r0 .. r0+31] in a fixed order (z = 0, 1, ...) with 16-byte loads, then runs the
// same output stage as the fused epilogue.
__global__ void splitk_reduce_kernel(const float *__restrict__ raw, EpiParams ep, int64_t ld,
                                     int64_t split_stride, int splits, int64_t n_rows,
                                     int64_t r_chunks) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n_rows * r_chunks) return;
    const int64_t n = idx / r_chunks;
    const int64_t r0 = (idx - n * r_chunks) * 32;
    const float4 *p = reinterpret_cast<const float4 *>(raw + n * ld + r0);
    float v[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 a = p[i];
        v[4 * i] = a.x;
        v[4 * i + 1] = a.y;
        v[4 * i + 2] = a.z;
        v[4 * i + 3] = a.w;
    }
    for (int z = 1; z < splits; ++z) {
        const float4 *q = reinterpret_cast<const float4 *>(raw + z * split_stride + n * ld + r0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 a = q[i];
            v[4 * i] += a.x;
            v[4 * i + 1] += a.y;
            v[4 * i + 2] += a.z;
            v[4 * i + 3] += a.w;
        }
    }
    emit_cols(v, decode_pos(n, ep), r0, ep);
}

// -------------------------------------------------------------------------- col2im
// y[b, oc, oy, ox] = bias + sum of col[(b, iy, ix), (oc, ty, tx)] over the taps that reach
// (oy, ox) (the same divisibility rule as the gather kernel), summed over split-K partials
// in a fixed order.  Only reachable taps are visited ("[WebGPU] optimizations for audio
// models", review commit: each chunk gathers only into the box its rows reach).
__global__ void col2im_kernel(const float *__restrict__ col, int64_t ld, int64_t split_stride,
                              int splits, int S_pad, const void *__restrict__ bias,
                              void *__restrict__ y, Geo g, int64_t total) {
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t ox = idx % g.Wo;
        int64_t t = idx / g.Wo;
        const int64_t oy = t % g.Ho;
        t /= g.Ho;
        const int64_t oc = t % g.C_out;
        const int64_t b = t / g.C_out;
        float acc = bias ? load_io(bias, oc, g.bf16) : 0.0f;
        const int64_t ry = oy + g.py, rx = ox + g.px;
        for (int64_t ty = ry % g.sy; ty < g.ky; ty += g.sy) {
            const int64_t iy = (ry - ty) / g.sy;
            if (iy < 0) break;
            if (iy >= g.H) continue;
            for (int64_t tx = rx % g.sx; tx < g.kx; tx += g.sx) {
                const int64_t ix = (rx - tx) / g.sx;
                if (ix < 0) break;
                if (ix >= g.W) continue;
                const int64_t r = oc * S_pad + ty * g.kx + tx;
                const int64_t n = (b * g.H + iy) * g.W + ix;
                const float *p = col + n * ld + r;
                for (int z = 0; z < splits; ++z) acc += p[(int64_t)z * split_stride];
            }
        }
        store_io(y, idx, apply_act(acc, g.act, g.slope), g.bf16);
    }
}

}  // namespace

// ============================================================================ launchers

cudaError_t launch_gather(const ctr_plan_s *pl, const void *x, const void *w, const void *bias,
                          void *y, cudaStream_t st) {
    const Geo g = geo_of(pl);
    const int64_t total = g.B * g.C_out * g.Ho * g.Wo;
    if (total == 0) return cudaSuccess;
    gather_kernel<<<grid_for(total, kBlock), kBlock, 0, st>>>(x, w, bias, y, g, total);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_fill_bias(const ctr_plan_s *pl, const void *bias, void *y, cudaStream_t st) {
    const Geo g = geo_of(pl);
    const int64_t total = g.B * g.C_out * g.Ho * g.Wo;
    if (total == 0) return cudaSuccess;
    fill_bias_kernel<<<grid_for(total, kBlock), kBlock, 0, st>>>(bias, y, g, total);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_copy_weight(const ctr_plan_s *pl, const void *w, void *w_packed,
                               cudaStream_t st) {
    const int64_t bytes = (int64_t)pl->packed_bytes;
    const int64_t n16 = bytes / 16;
    const int tail = (int)(bytes - n16 * 16);
    copy_bytes_kernel<<<grid_for(std::max<int64_t>(n16, 1), kBlock), kBlock, 0, st>>>(
        static_cast<const uint4 *>(w), static_cast<uint4 *>(w_packed), n16,
        static_cast<const uint8_t *>(w) + n16 * 16, static_cast<uint8_t *>(w_packed) + n16 * 16,
        tail);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_prepack(const ctr_plan_s *pl, const void *w, void *w_packed, cudaStream_t st) {
    PackGeo pg;
    pg.M_pad = pl->M_pad;
    pg.K_total = pl->K_total;
    pg.C_in_pad = pl->C_in_pad;
    pg.C_in = pl->C_in;
    pg.C_out = pl->C_out;
    pg.ky = pl->k[0];
    pg.kx = pl->k[1];
    pg.sy = pl->s[0];
    pg.sx = pl->s[1];
    pg.my = pl->m[0];
    pg.mx = pl->m[1];
    pg.S = pl->S;
    pg.S_pad = pl->S_pad;
    pg.polyphase = pl->path == CTR_PATH_POLYPHASE ? 1 : 0;
    pg.bf16 = pl->dtype == CTR_BF16 ? 1 : 0;
    const int64_t total = pg.M_pad * pg.K_total;
    prepack_kernel<<<grid_for(total, kBlock), kBlock, 0, st>>>(w, w_packed, pg);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_stage_x(const ctr_plan_s *pl, const void *x, void *xs, cudaStream_t st) {
    StageGeo sg;
    sg.B = pl->B;
    sg.C_in = pl->C_in;
    sg.C_in_pad = pl->C_in_pad;
    sg.H = pl->in[0];
    sg.W = pl->in[1];
    sg.Py = pl->P[0];
    sg.Px = pl->P[1];
    sg.hy = pl->m[0] - 1;
    sg.hx = pl->m[1] - 1;
    sg.N_total = pl->N_total;
    sg.bf16 = pl->dtype == CTR_BF16 ? 1 : 0;
    if (sg.N_total == 0) return cudaSuccess;
    dim3 grid((unsigned)ceil_div(sg.N_total, kStagePos), (unsigned)(sg.C_in_pad / 32));
    stage_x_kernel<<<grid, 256, 0, st>>>(x, xs, sg);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_splitk_reduce(const ctr_plan_s *pl, const float *raw, const EpiParams &ep,
                                 int64_t raw_ld, int64_t split_stride, cudaStream_t st) {
    const int64_t n_rows = pl->N_total;
    const int64_t r_chunks = ceil_div(std::min<int64_t>(pl->M_rows, raw_ld), 32);
    const int64_t total = n_rows * r_chunks;
    if (total == 0) return cudaSuccess;
    splitk_reduce_kernel<<<grid_for(total, 128), 128, 0, st>>>(raw, ep, raw_ld, split_stride,
                                                             pl->splits, n_rows, r_chunks);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_col2im(const ctr_plan_s *pl, const float *col, int64_t col_ld,
                          const void *bias, void *y, cudaStream_t st) {
    const Geo g = geo_of(pl);
    const int64_t total = g.B * g.C_out * g.Ho * g.Wo;
    if (total == 0) return cudaSuccess;
    const int64_t split_stride = raw_split_stride_of(pl);
    col2im_kernel<<<grid_for(total, kBlock), kBlock, 0, st>>>(col, col_ld, split_stride,
                                                              pl->splits, pl->S_pad, bias, y, g,
                                                              total);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace ctr
