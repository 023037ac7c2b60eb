// depthwise.cu -- ConvTranspose with one input channel per group (groups = C_in, C_out = M *
// C_in; M = 1 is the depthwise upsampler).
//
// Output channel oc reads only input channel oc / M and its own k taps (the grouped weight
// [C_in][M][k...] of "[ExecuTorch][WebGPU] Add optimized conv2d op", Implementation, is the
// same memory as [C_out][k...]).  "[XNNPACK] Lower dense transposed convs as one polyphase
// conv + depth to space" (DecomposeDepthwiseConvTransposePass commit) rewrites such a layer
// as s*s stride-1 depthwise convolutions over the low-resolution input whose outputs are
// interleaved by a depth-to-space; here the interleave is the store order: each thread
// writes kDwV consecutive outputs of every output row of one phase row, and output ox takes
// the phase (ox + px) mod sx of the x taps.  With k = s every output has exactly one tap, the plain
// multiply of the same page's k = s upsampler.
//
// The work is a few multiply-adds per output byte, so the kernel is bound by HBM: inputs and
// taps are read through the L1 (a warp's 32 threads read one contiguous input segment), the
// outputs leave as 16-byte stores.  The x-direction kernel size, stride and padding phase are
// template parameters, and so are the row kernel size and stride: the taps that reach each
// of a thread's outputs and the input columns they read are then known at compile time, and
// those inputs and the taps sit in registers.  Geometries without a compiled kernel run on
// the gather kernel.
#include <algorithm>
#include <utility>
#include <cuda_bf16.h>

#include "ctr_internal.h"

namespace ctr {
namespace {

constexpr int kDwV = 8;       // outputs per thread and row (one 16-byte bf16 store, two for fp32)
constexpr int kDwBlock = 256;

struct DwGeo {
    int H, W, py, px, Ho, Wo;
    int Qy;                   // phase rows ceil((Ho + py) / sy)
    int R, bands;             // phase rows per thread; bands of blockDim.y * R phase rows
    int nch;                  // 16-byte copies per staged row
    int C_out, mult;          // mult = C_out / C_in
    int planes;               // B * C_out output planes
    int act;
    float slope;
    int vec;                  // Wo % kDwV == 0: whole chunks, 16-byte aligned stores
};

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

__device__ __forceinline__ void store_chunk(float *y, const float (&v)[kDwV]) {
    reinterpret_cast<float4 *>(y)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(y)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

__device__ __forceinline__ void store_chunk(__nv_bfloat16 *y, const float (&v)[kDwV]) {
    uint4 u;
    uint32_t *w = reinterpret_cast<uint32_t *>(&u);
#pragma unroll
    for (int i = 0; i < kDwV / 2; ++i) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t *>(&h);
    }
    *reinterpret_cast<uint4 *>(y) = u;
}

__device__ __forceinline__ void store_one(float *y, float v) { *y = v; }
__device__ __forceinline__ void store_one(__nv_bfloat16 *y, float v) { *y = __float2bfloat16_rn(v); }

// One input row's NX columns from bx on, as fp32.
template <typename T, int NX>
__device__ __forceinline__ void load_row(float (&v)[NX], const T *__restrict__ xr, int bx, int W,
                                         bool interior) {
    if (interior) {   // every column in [0, W): plain loads at fixed offsets
#pragma unroll
        for (int i = 0; i < NX; ++i) v[i] = to_f(xr[bx + i]);
    } else {          // a row end: clamped address, zero outside the row
#pragma unroll
        for (int i = 0; i < NX; ++i) {
            const int ix = bx + i;
            const float t = to_f(xr[min(max(ix, 0), W - 1)]);
            v[i] = (ix >= 0 && ix < W) ? t : 0.0f;
        }
    }
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
}

__host__ __device__ constexpr int floor_div(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

// A thread owns kDwV consecutive output columns of a run of R consecutive phase rows.  Phase
// row qy holds the output rows oy = SY*qy + jy - py (jy < SY), which all read input rows
// qy - uy (uy < MY) through the row taps ty = jy + SY*uy; consecutive phase rows share MY - 1
// input rows, so a run fetches each input row once.  The channel's KY x KX taps sit in
// registers for the whole plane.
//
// OFFX = px mod SX.  The first output column ox0 is a multiple of kDwV (and so of SX), so
// r0 = ox0 + px - OFFX is a multiple of SX and column ox0 + j lies at x phase (OFFX + j) mod
// SX and reads input column r0 / SX + (OFFX + j) / SX - ux through its tap ux.
//
// STAGED: a block covers a band of blockDim.y * R phase rows and blockDim.x chunks of one
// plane.  It first copies every input row and column the band reads (16-byte cp.async
// copies, zero where the window leaves the input) into shared memory, so all of the band's
// reads are in flight at once, then computes from there.  Needs W a multiple of 16 bytes.
// Otherwise each thread reads its columns straight from global memory.
template <typename T, int KX, int SX, int OFFX, int KY, int SY, bool STAGED>
__global__ void __launch_bounds__(kDwBlock, 4)
depthwise_kernel(const T *__restrict__ x, const T *__restrict__ w, const T *__restrict__ bias,
                 T *__restrict__ y, DwGeo g) {
    constexpr int MX = (KX + SX - 1) / SX;                 // x taps per phase
    constexpr int MY = (KY + SY - 1) / SY;                 // row taps per phase
    constexpr int NX = (OFFX + kDwV - 1) / SX + MX;        // input columns a thread reads
    constexpr int E = 16 / sizeof(T);                      // elements per 16-byte copy
    static_assert(kDwV % SX == 0, "a chunk must start at x phase 0");
    extern __shared__ __align__(16) unsigned char dw_smem[];
    T *xs = reinterpret_cast<T *>(dw_smem);

    const int ox_b = blockIdx.x * blockDim.x * kDwV;       // the block's first column
    const int ox0 = ox_b + threadIdx.x * kDwV;
    const bool col_ok = ox0 < g.Wo;
    const int bx = (ox0 + g.px - OFFX) / SX - (MX - 1);   // first input column read
    const bool interior = bx >= 0 && bx + NX <= g.W;
    const bool has_input = g.H > 0 && g.W > 0;
    // Staged window: columns from cs0 (a multiple of E at or before the block's first read
    // column), g.nch copies wide; rows from the band's first phase row - (MY - 1).
    const int cs0 = floor_div((ox_b + g.px - OFFX) / SX - (MX - 1), E) * E;
    const int pitch = g.nch * E;
    const int lx = bx - cs0;
    const int band_rows = blockDim.y * g.R;
    if (!STAGED && !col_ok) return;

    for (int plane = blockIdx.z; plane < g.planes; plane += gridDim.z) {
        const int oc = plane % g.C_out;
        const int xplane = g.mult == 1 ? plane : plane / g.mult;   // b * C_in + oc / M
        const float b = bias ? to_f(bias[oc]) : 0.0f;
        const T *xp = x + (int64_t)xplane * g.H * g.W;         // planes hold < 2^30 elements
        T *yp = y + (int64_t)plane * g.Ho * g.Wo + ox0;
        float wr[KY][KX];
        {
            const T *wp = w + (int64_t)oc * (KY * KX);
#pragma unroll
            for (int ty = 0; ty < KY; ++ty)
#pragma unroll
                for (int tx = 0; tx < KX; ++tx) wr[ty][tx] = to_f(wp[ty * KX + tx]);
        }
        for (int band = blockIdx.y; band < g.bands; band += gridDim.y) {
            const int ir0 = band * band_rows - (MY - 1);       // first staged input row
            if constexpr (STAGED) {
                // The band's phase rows that exist, and the MY - 1 rows above them.
                const int nrows = min(band_rows, g.Qy - band * band_rows) + MY - 1;
                const int tid = threadIdx.y * blockDim.x + threadIdx.x;
                for (int idx = tid; idx < nrows * g.nch; idx += blockDim.x * blockDim.y) {
                    const int r = idx / g.nch, c = idx - r * g.nch;
                    const int iy = ir0 + r, ix = cs0 + c * E;
                    T *dst = xs + r * pitch + c * E;
                    if (iy >= 0 && iy < g.H && ix >= 0 && ix < g.W)   // W % E == 0: whole copy in
                        cp_async16(dst, xp + iy * g.W + ix);
                    else
                        *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
                }
                cp_async_wait_all();
                __syncthreads();
            }
            // One input row's NX columns as fp32 (zero outside the input).
            auto fetch = [&](float (&v)[NX], int iy) {
                if constexpr (STAGED) {
                    const T *r = xs + (iy - ir0) * pitch + lx;
#pragma unroll
                    for (int i = 0; i < NX; ++i) v[i] = to_f(r[i]);
                } else {
                    if (has_input && iy >= 0 && iy < g.H) {
                        load_row(v, xp + iy * g.W, bx, g.W, interior);
                    } else {
#pragma unroll
                        for (int i = 0; i < NX; ++i) v[i] = 0.0f;
                    }
                }
            };
            const int qy0 = band * band_rows + threadIdx.y * g.R;
            const int qy1 = min(qy0 + g.R, g.Qy);
            if (col_ok && qy0 < qy1) {
                // In step qy, xv[uy] holds input row qy - uy: before the first step xv[uy]
                // holds row qy0 - 1 - uy, which the step's shift moves to xv[uy + 1].
                float xv[MY][NX];
#pragma unroll
                for (int uy = 0; uy + 1 < MY; ++uy) fetch(xv[uy], qy0 - 1 - uy);
                for (int qy = qy0; qy < qy1; ++qy) {
#pragma unroll
                    for (int uy = MY - 1; uy > 0; --uy)
#pragma unroll
                        for (int i = 0; i < NX; ++i) xv[uy][i] = xv[uy - 1][i];
                    fetch(xv[0], qy);
#pragma unroll
                    for (int jy = 0; jy < SY; ++jy) {
                        const int oy = SY * qy + jy - g.py;
                        if (oy < 0 || oy >= g.Ho) continue;
                        // y = bias + the taps in ascending (ty, tx) order, as the gather
                        // kernel sums them (the two agree bit for bit).
                        float acc[kDwV];
#pragma unroll
                        for (int j = 0; j < kDwV; ++j) acc[j] = b;
#pragma unroll
                        for (int uy = 0; uy < MY; ++uy) {
                            const int ty = jy + SY * uy;
                            if (ty >= KY) break;
#pragma unroll
                            for (int j = 0; j < kDwV; ++j) {
                                const int q = (OFFX + j) / SX, jx = (OFFX + j) % SX;
#pragma unroll
                                for (int ux = 0; ux < MX; ++ux) {
                                    if (jx + SX * ux < KX)
                                        acc[j] = fmaf(xv[uy][q - ux + MX - 1],
                                                      wr[ty][jx + SX * ux], acc[j]);
                                }
                            }
                        }
                        if (g.act == CTR_ACT_LEAKY_RELU) {
#pragma unroll
                            for (int j = 0; j < kDwV; ++j)
                                acc[j] = acc[j] < 0.0f ? acc[j] * g.slope : acc[j];
                        }
                        T *yr = yp + oy * g.Wo;
                        if (g.vec) {
                            store_chunk(yr, acc);
                        } else {
#pragma unroll
                            for (int j = 0; j < kDwV; ++j)
                                if (ox0 + j < g.Wo) store_one(yr + j, acc[j]);
                        }
                    }
                }
            }
            if constexpr (STAGED) __syncthreads();   // the window is refilled next
        }
    }
}

template <typename T>
using DwKernel = void (*)(const T *, const T *, const T *, T *, DwGeo);

template <typename T, int KX, int SX, int KY, int SY, int... O>
DwKernel<T> pick_phase(int off, bool staged, std::integer_sequence<int, O...>) {
    DwKernel<T> k = nullptr;
    ((off == O ? (k = staged ? depthwise_kernel<T, KX, SX, O, KY, SY, true>
                             : depthwise_kernel<T, KX, SX, O, KY, SY, false>,
                  0)
               : 0),
     ...);
    return k;
}

template <typename T, int KX, int SX, int KY, int SY>
DwKernel<T> pick(int off, bool staged) {
    return pick_phase<T, KX, SX, KY, SY>(off, staged, std::make_integer_sequence<int, SX>{});
}

// The compiled geometries: x (kernel, stride) pairs of the pages' upsamplers (k = 2s, k = s)
// and the odd k = 3, s = 2, with one row tap (1-D plans, or a 2-D kernel one row high), and
// the square 2-D kernels up to 4 x 4 (the image decoder's 4 x 4 / stride-2 filter).
template <typename T>
DwKernel<T> kernel_for(int kx, int sx, int off, int ky, int sy, bool staged = false) {
    const bool st = staged;
    if (ky == 1 && sy == 1) {
        if (sx == 2) return kx == 2 ? pick<T, 2, 2, 1, 1>(off, st) : kx == 3 ? pick<T, 3, 2, 1, 1>(off, st)
                          : kx == 4 ? pick<T, 4, 2, 1, 1>(off, st) : nullptr;
        if (sx == 4) return kx == 4 ? pick<T, 4, 4, 1, 1>(off, st)
                          : kx == 8 ? pick<T, 8, 4, 1, 1>(off, st) : nullptr;
        if (sx == 8) return kx == 8 ? pick<T, 8, 8, 1, 1>(off, st)
                          : kx == 16 ? pick<T, 16, 8, 1, 1>(off, st) : nullptr;
        return nullptr;
    }
    if (ky != kx || sy != sx) return nullptr;
    if (sx == 2) return kx == 2 ? pick<T, 2, 2, 2, 2>(off, st) : kx == 3 ? pick<T, 3, 2, 3, 2>(off, st)
                      : kx == 4 ? pick<T, 4, 2, 4, 2>(off, st) : nullptr;
    if (sx == 4 && kx == 4) return pick<T, 4, 4, 4, 4>(off, st);
    return nullptr;
}

DwGeo dw_geo_of(const ctr_plan_s *pl) {
    DwGeo g;
    g.H = (int)pl->in[0];
    g.W = (int)pl->in[1];
    g.py = (int)pl->p[0];
    g.px = (int)pl->p[1];
    g.Ho = (int)pl->out[0];
    g.Wo = (int)pl->out[1];
    g.Qy = (int)((pl->out[0] + pl->p[0] + pl->s[0] - 1) / pl->s[0]);
    g.C_out = (int)pl->C_out;
    g.mult = (int)(pl->C_out / pl->C_in);
    g.planes = (int)(pl->B * pl->C_out);
    g.act = pl->act;
    g.slope = pl->slope;
    g.vec = pl->out[1] % kDwV == 0;
    g.R = 1;
    g.bands = g.Qy;
    g.nch = 0;
    return g;
}

constexpr int kDwStageLimit = 48 * 1024;   // shared memory of a staged block

template <typename T>
cudaError_t launch_typed(const ctr_plan_s *pl, const void *x, const void *w, const void *bias,
                         void *y, cudaStream_t st) {
    const int kx = (int)pl->k[1], sx = (int)pl->s[1], ky = (int)pl->k[0], sy = (int)pl->s[0];
    const int off = (int)(pl->p[1] % pl->s[1]);
    DwGeo g = dw_geo_of(pl);
    // Block: tx threads along a row (enough chunks to cover it, up to the whole block) times
    // ty = kDwBlock / tx runs of R phase rows of the same plane: a band of ty * R phase rows.
    // R is the longest run (up to 8) that still leaves about two waves of blocks.
    const int64_t chunks = (g.Wo + kDwV - 1) / kDwV;
    int tx = 1;
    while (tx < kDwBlock && tx < chunks) tx *= 2;
    const int ty = kDwBlock / tx;
    const int64_t xblocks = (chunks + tx - 1) / tx;
    const int64_t want = 2 * 4 * (int64_t)std::max(pl->num_sms, 1);
    g.R = 8;
    while (g.R > 1 && ((int64_t)ty * (g.R / 2) >= g.Qy ||
                       xblocks * g.planes * ((g.Qy + ty * g.R - 1) / (ty * g.R)) < want))
        g.R /= 2;
    g.bands = (g.Qy + ty * g.R - 1) / (ty * g.R);
    // Staged when the input rows are whole 16-byte copies and the window fits.
    constexpr int E = 16 / sizeof(T);
    const int nx = (off + kDwV - 1) / sx + (kx + sx - 1) / sx;
    g.nch = ((tx - 1) * (kDwV / sx) + nx + 2 * E - 2) / E;
    const int64_t rows = std::min<int64_t>((int64_t)ty * g.R, g.Qy) + (ky + sy - 1) / sy - 1;
    const int64_t smem = rows * g.nch * 16;
    const bool staged = g.W % E == 0 && smem <= kDwStageLimit;
    const DwKernel<T> k = kernel_for<T>(kx, sx, off, ky, sy, staged);
    if (!k) return cudaErrorInvalidValue;
    const dim3 block(tx, ty);
    const dim3 grid((unsigned)xblocks, (unsigned)std::min<int64_t>(g.bands, 65535),
                    (unsigned)std::min<int64_t>(g.planes, 65535));
    k<<<grid, block, staged ? (size_t)smem : 0, st>>>(
        static_cast<const T *>(x), static_cast<const T *>(w), static_cast<const T *>(bias),
        static_cast<T *>(y), g);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

bool depthwise_supported(const ctr_plan_s *pl) {
    if (pl->groups != pl->C_in || pl->C_out % pl->C_in != 0) return false;
    if (pl->dtype == CTR_F16) return false;   // compiled for fp32 and bf16; fp16 uses gather
    if (pl->nhwc) return false;               // planes of NCHW tensors; NHWC uses gather
    if (pl->dil[0] != 1 || pl->dil[1] != 1) return false;   // taps compiled undilated
    // Planes, and offsets inside an input or output plane, in 32 bits.
    const int64_t lim = (int64_t)1 << 30;
    if (pl->B * pl->C_out >= lim || pl->out[0] * pl->out[1] >= lim ||
        pl->in[0] * pl->in[1] >= lim || pl->out[0] + pl->p[0] >= lim || pl->out[1] >= lim)
        return false;
    const int off = (int)(pl->p[1] % pl->s[1]);
    const int kx = (int)pl->k[1], sx = (int)pl->s[1], ky = (int)pl->k[0], sy = (int)pl->s[0];
    return pl->dtype == CTR_BF16 ? kernel_for<__nv_bfloat16>(kx, sx, off, ky, sy) != nullptr
                                 : kernel_for<float>(kx, sx, off, ky, sy) != nullptr;
}

cudaError_t launch_depthwise(const ctr_plan_s *pl, const void *x, const void *w, const void *bias,
                             void *y, cudaStream_t st) {
    if (pl->B * pl->C_out * pl->out[0] * pl->out[1] == 0) return cudaSuccess;
    return pl->dtype == CTR_BF16 ? launch_typed<__nv_bfloat16>(pl, x, w, bias, y, st)
                                 : launch_typed<float>(pl, x, w, bias, y, st);
}

}  // namespace ctr
