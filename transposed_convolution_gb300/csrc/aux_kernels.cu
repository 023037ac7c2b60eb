// aux_kernels.cu -- the non-tensor-core kernels of the library:
//   prepack      torch weight -> phase-major GEMM rows (polyphase) or (oc, tap) rows (col2im)
//   stage_x      NC(H)W input -> channels-last rows with zero halos (tf32 + cross, or 16-bit)
//   splitk_reduce  fixed-order sum of split-K partials, then the fused output stage
//   col2im       gather of the valid taps from the fp32 column buffer
//   gather       direct ConvTranspose for tiny channel counts and grouped convolutions
//   fill_bias    y = bias (or zeros) for an empty input on the col2im path
//   copy_weight  the gather path's "packed" weight (a plain copy)
#include <algorithm>
#include <type_traits>
#include <cuda_bf16.h>

#include "ctr_internal.h"
#include "epilogue.cuh"
#include "ptx.cuh"

namespace ctr {
namespace {

constexpr int kBlock = 256;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

unsigned grid_for(int64_t n, int block) {
    const int64_t g = ceil_div(n, block);
    return (unsigned)std::min<int64_t>(std::max<int64_t>(g, 1), (int64_t)1 << 30);
}

// Geometry of a plan as plain values for the kernels below (2-D form).
struct Geo {
    int64_t B, C_in, C_out;
    int64_t cin_g, cout_g;    // channels per group
    int64_t H, W, ky, kx, sy, sx, py, px, Ho, Wo;
    int64_t dy, dx;           // dilation
    int act;
    float slope;
    int io;           // IoType of x, w, bias and y
    int nhwc;         // x and y channels last
};

Geo geo_of(const ctr_plan_s *pl) {
    Geo g;
    g.B = pl->B;
    g.C_in = pl->C_in;
    g.C_out = pl->C_out;
    g.cin_g = pl->C_in / pl->groups;
    g.cout_g = pl->C_out / pl->groups;
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
    g.dy = pl->dil[0];
    g.dx = pl->dil[1];
    g.act = pl->act;
    g.slope = pl->slope;
    g.io = pl->dtype;   // IoType
    g.nhwc = pl->nhwc;
    return g;
}

// -------------------------------------------------------------------------- gather
// y[b, oc, oy, ox] = bias[oc] + sum over the input channels of oc's group and the taps that
// reach (oy, ox): a tap ty contributes when (oy + py - ty*dy) is a multiple of sy and the
// quotient is a valid input row ("[ExecuTorch][WebGPU] Add optimized conv2d op",
// Implementation: the gather form with the un-flipped weight, laid out [IC][OC/groups][k],
// and the dilation dH).  fp32 accumulation on CUDA cores, starting from the bias, taps in
// ascending (ty, tx) order; one thread per output element.
//
// Taps of one output along a dimension: r = o + p is the unpadded position, tap t reaches it
// from input (r - t*d)/s when that is a whole number in range.  Without dilation the first
// such tap is r mod s and the next ones follow every s taps; with dilation every tap is
// tested.  r - t*d only falls as t grows, so the loop ends at the first negative one.
struct TapRange {
    int64_t t0, step;
};

__device__ __forceinline__ TapRange tap_range(int64_t r, int64_t s, int64_t d) {
    return d == 1 ? TapRange{r % s, s} : TapRange{0, 1};
}
// Output element idx of a plan's y, NCHW or NHWC order.
struct OutIdx {
    int64_t b, oc, oy, ox;
};
__device__ __forceinline__ OutIdx out_index(int64_t idx, const Geo &g) {
    OutIdx o;
    if (g.nhwc) {
        o.oc = idx % g.C_out;
        int64_t t = idx / g.C_out;
        o.ox = t % g.Wo;
        t /= g.Wo;
        o.oy = t % g.Ho;
        o.b = t / g.Ho;
    } else {
        o.ox = idx % g.Wo;
        int64_t t = idx / g.Wo;
        o.oy = t % g.Ho;
        t /= g.Ho;
        o.oc = t % g.C_out;
        o.b = t / g.C_out;
    }
    return o;
}

__global__ void gather_kernel(const void *__restrict__ x, const void *__restrict__ w,
                              const void *__restrict__ bias, void *__restrict__ y, Geo g,
                              int64_t total) {
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const OutIdx o = out_index(idx, g);
        const int64_t ox = o.ox, oy = o.oy, oc = o.oc, b = o.b;
        const int64_t grp = oc / g.cout_g, ic0 = grp * g.cin_g;
        float acc = bias ? load_io(bias, oc, g.io) : 0.0f;
        const int64_t ry = oy + g.py, rx = ox + g.px;
        const TapRange try_ = tap_range(ry, g.sy, g.dy), trx = tap_range(rx, g.sx, g.dx);
        for (int64_t ty = try_.t0; ty < g.ky; ty += try_.step) {
            const int64_t ny = ry - ty * g.dy;
            if (ny < 0) break;
            if (ny % g.sy) continue;
            const int64_t iy = ny / g.sy;
            if (iy >= g.H) continue;
            for (int64_t tx = trx.t0; tx < g.kx; tx += trx.step) {
                const int64_t nx = rx - tx * g.dx;
                if (nx < 0) break;
                if (nx % g.sx) continue;
                const int64_t ix = nx / g.sx;
                if (ix >= g.W) continue;
                // input channel ic0 at (b, iy, ix) and the step between input channels
                const int64_t xoff = g.nhwc ? ((b * g.H + iy) * g.W + ix) * g.C_in + ic0
                                            : ((b * g.C_in + ic0) * g.H + iy) * g.W + ix;
                const int64_t xstride = g.nhwc ? 1 : g.H * g.W;
                const int64_t woff =
                    (((ic0 * g.cout_g + oc - grp * g.cout_g) * g.ky) + ty) * g.kx + tx;
                const int64_t wstride = g.cout_g * g.ky * g.kx;
                for (int64_t ic = 0; ic < g.cin_g; ++ic)
                    acc = fmaf(load_io(x, xoff + ic * xstride, g.io),
                               load_io(w, woff + ic * wstride, g.io), acc);
            }
        }
        store_io(y, idx, apply_act(acc, g.act, g.slope), g.io);
    }
}

__global__ void fill_bias_kernel(const void *__restrict__ bias, void *__restrict__ y, Geo g,
                                 int64_t total) {
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t oc = out_index(idx, g).oc;
        const float v = bias ? load_io(bias, oc, g.io) : 0.0f;
        store_io(y, idx, apply_act(v, g.act, g.slope), g.io);
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
    int64_t mky, mkx;     // phase taps of the kernel (my, mx count one more with a folded pm)
    int64_t pmy, pmx;     // padding remainder folded into the taps (output phases)
    int64_t dy, dx;       // dilation (polyphase rows of the zero-inserted kernel)
    int S, S_pad;
    int polyphase;
    int io;               // IoType of the weight and the packed operand
    int pm_tc, block_n;   // phase-major rows within tiles of block_n rows (pm_tc channels)
};

// Polyphase rows ("[XNNPACK] Lower dense transposed convs as one polyphase conv + depth to
// space", Summary: phase-major ordering, taps flipped within a phase):
//   A[r = oc*S_pad + jy*sx + jx, k = (uy*mx + ux)*C_in_pad + ic]
//       = w[ic, oc, sy*(mky-1-uy) + jy + pmy, sx*(mkx-1-ux) + jx + pmx]
// with 0 outside the kernel (the kernel is zero-padded to m*s taps).  pm = 0 gives the
// pages' phases of the unpadded output; pm = p mod s the phases of the output itself, whose
// phase j is the unpadded output's phase j + pm (the next position's phase j + pm - s when
// that reaches s, hence the extra tap).
// With dilation the polyphase rows come from the zero-inserted kernel: a dilated tap index
// e (per dimension) holds w[.., e / dil] when e is a multiple of dil and e / dil < k, and
// zero otherwise.
// col2im rows ("[WebGPU] optimizations for audio models", ConvTranspose commit: W[C_in,
// kH*kW*C_out] prepacked to the GEMM layout):  A[r = oc*S_pad + t, k = ic] = w[ic, oc, t].
// Padding rows and channels are zero.  fp32 weights are split into a tf32 plane and a plane
// of bf16 cross words (ptx::split_w).
// A chained producer (pm_tc > 0) orders the rows of each block_n-row tile phase-major
// instead: tile t, row j * pm_tc + c is phase j of channel t * pm_tc + c.
__global__ void prepack_kernel(const void *__restrict__ w, void *__restrict__ wp, PackGeo pg) {
    const int64_t total = pg.M_pad * pg.K_total;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = idx / pg.K_total;
        const int64_t kk = idx - r * pg.K_total;
        const int64_t g = kk / pg.C_in_pad;
        const int64_t ic = kk - g * pg.C_in_pad;
        int64_t oc, j;
        if (pg.pm_tc) {
            const int64_t t = r / pg.block_n, rl = r - t * pg.block_n;
            j = rl / pg.pm_tc;
            oc = t * pg.pm_tc + (rl - j * pg.pm_tc);
        } else {
            oc = r / pg.S_pad;
            j = r - oc * pg.S_pad;
        }
        float v = 0.0f;
        if (oc < pg.C_out && j < pg.S && ic < pg.C_in) {
            int64_t ty, tx;
            if (pg.polyphase) {
                const int64_t jy = j / pg.sx, jx = j - (j / pg.sx) * pg.sx;
                const int64_t uy = g / pg.mx, ux = g - (g / pg.mx) * pg.mx;
                ty = pg.sy * (pg.mky - 1 - uy) + jy + pg.pmy;
                tx = pg.sx * (pg.mkx - 1 - ux) + jx + pg.pmx;
                // Dilated tap index -> real tap (past the kernel when before the first tap or
                // between taps).
                ty = (ty < 0 || ty % pg.dy) ? pg.ky : ty / pg.dy;
                tx = (tx < 0 || tx % pg.dx) ? pg.kx : tx / pg.dx;
            } else {
                ty = j / pg.kx;
                tx = j - ty * pg.kx;
            }
            if (ty < pg.ky && tx < pg.kx)
                v = load_io(w, ((ic * pg.C_out + oc) * pg.ky + ty) * pg.kx + tx, pg.io);
        }
        if (pg.io == IO_BF16) {
            static_cast<__nv_bfloat16 *>(wp)[idx] = __float2bfloat16_rn(v);  // exact: v is bf16
        } else if (pg.io == IO_F16) {
            static_cast<__half *>(wp)[idx] = __float2half_rn(v);             // exact: v is fp16
        } else {
            uint32_t cross;
            static_cast<float *>(wp)[idx] = ptx::split_w(v, cross);
            static_cast<uint32_t *>(wp)[total + idx] = cross;
        }
    }
}

// -------------------------------------------------------------------------- stage_x
struct StageGeo {
    int64_t B, C_in, C_in_pad, H, W, Py, Px, hy, hx, N_total;
    int b16;   // 16-bit elements (bf16 or fp16), else fp32
};

// xs[n][c] with n = (b*Py + py')*Px + px': x[b, c, py' - hy, px' - hx] inside the input and
// c < C_in, zero elsewhere (the front halos hy, hx are the polyphase conv's padding m - 1,
// less the phase positions the output phases skip).  fp32 input is written as a tf32 plane
// and a plane of bf16 cross words (ptx::split_x).
//
// A block transposes one tile of 128 input positions (along x, within one staged row) by
// kStageC channels (64 bf16 or 32 fp32, i.e. 128 bytes of a staged row) through shared
// memory:
//   load   each warp reads whole 16-byte vectors along x (one or two channel rows per
//          instruction; element loads when the rows are not 16-byte aligned) and writes
//          them as float4s into tile[c][x];
//   store  each thread gathers the kOutVec channels of one 16-byte output vector at one
//          position and writes it; eight consecutive threads cover a 128-byte staged row.
// The tile is XOR-swizzled by 4-float groups, column group g of channel c stored at
// g ^ ((c / kOutVec) & 7), so both the float4 writes and the scalar reads of a warp hit 32
// different banks.  Tiles start at input x = 128 t (aligned for the 16-byte loads) and cover
// the input row; the first tile of a staged row also writes the zeros of the left halo
// (staged positions 0 .. hx-1) and the last one those past the tiles (up to Px).
constexpr int kStageThreads = 256;
constexpr int kStageTP = 128;

struct StageUnits {
    int64_t cchunks;   // C_in_pad / kStageC
    int64_t xtiles;    // tiles of 128 positions per staged row
    int64_t x_first;   // input x of the first tile of a row (0)
    int64_t tiles;     // rows * xtiles * cchunks
};

template <bool B16, bool VEC>
__global__ void __launch_bounds__(kStageThreads) stage_x_kernel(const void *__restrict__ x,
                                                               void *__restrict__ xs,
                                                               StageGeo sg, StageUnits su) {
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    // 16-bit inputs (bf16 or fp16) are moved as raw 16-bit payloads: placed in the high half
    // of an fp32 word in shared memory and taken back out unchanged, whatever the format.
    constexpr bool BF16 = B16;
    using T = typename std::conditional<B16, uint16_t, float>::type;
    constexpr int kStageC = BF16 ? 64 : 32;      // channels per tile (128 bytes of a row)
    constexpr int kInVec = 16 / sizeof(T);       // positions per 16-byte load
    constexpr int kOutVec = 16 / sizeof(T);      // channels per 16-byte store
    constexpr int kLoadItems = kStageC * (kStageTP / kInVec) / kStageThreads;
    constexpr int kStoreItems = kStageTP * (kStageC / kOutVec) / kStageThreads;
    __shared__ __align__(16) float tile[kStageC][kStageTP];
    const T *__restrict__ xin = static_cast<const T *>(x);
    const int64_t lo_off = sg.N_total * sg.C_in_pad;

    for (int64_t t = blockIdx.x; t < su.tiles; t += gridDim.x) {
        const int64_t cq = t % su.cchunks;
        const int64_t rest = t / su.cchunks;
        const int64_t xt = rest % su.xtiles;
        const int64_t row = rest / su.xtiles;      // b * Py + py'
        const int64_t b = row / sg.Py;
        const int64_t yy = row - b * sg.Py - sg.hy;
        const int64_t xx0 = su.x_first + kStageTP * xt;
        const int64_t c_base = cq * kStageC;
        const bool row_in = yy >= 0 && yy < sg.H;

#pragma unroll
        for (int it = 0; it < kLoadItems; ++it) {
            const int i = it * kStageThreads + threadIdx.x;
            const int c = i / (kStageTP / kInVec);
            const int v = i % (kStageTP / kInVec);
            const int64_t xx = xx0 + (int64_t)v * kInVec;
            const int64_t ch = c_base + c;
            float val[kInVec];
#pragma unroll
            for (int j = 0; j < kInVec; ++j) val[j] = 0.0f;
            if (row_in && ch < sg.C_in) {
                const T *src = xin + ((b * sg.C_in + ch) * sg.H + yy) * sg.W;
                if (VEC && xx >= 0 && xx + kInVec <= sg.W) {
                    const uint4 r = *reinterpret_cast<const uint4 *>(src + xx);
                    const uint32_t w4[4] = {r.x, r.y, r.z, r.w};
                    if constexpr (BF16) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            val[2 * j] = __uint_as_float(w4[j] << 16);
                            val[2 * j + 1] = __uint_as_float(w4[j] & 0xFFFF0000u);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j) val[j] = __uint_as_float(w4[j]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < kInVec; ++j)
                        if (xx + j >= 0 && xx + j < sg.W) {
                            if constexpr (BF16)
                                val[j] = __uint_as_float((uint32_t)src[xx + j] << 16);
                            else
                                val[j] = src[xx + j];
                        }
                }
            }
            const int sw = (c / kOutVec) & 7;
#pragma unroll
            for (int q = 0; q < kInVec / 4; ++q) {
                const int grp = (v * (kInVec / 4) + q) ^ sw;
                *reinterpret_cast<float4 *>(&tile[c][4 * grp]) =
                    make_float4(val[4 * q], val[4 * q + 1], val[4 * q + 2], val[4 * q + 3]);
            }
        }
        __syncthreads();

#pragma unroll
        for (int it = 0; it < kStoreItems; ++it) {
            const int i = it * kStageThreads + threadIdx.x;
            const int p = i / (kStageC / kOutVec);
            const int cg = i % (kStageC / kOutVec);
            const int64_t px = xx0 + p + sg.hx;
            if (px < 0 || px >= sg.Px) continue;
            const int col = (((p >> 2) ^ (cg & 7)) << 2) | (p & 3);
            float val[kOutVec];
#pragma unroll
            for (int k = 0; k < kOutVec; ++k) val[k] = tile[cg * kOutVec + k][col];
            const int64_t o = (row * sg.Px + px) * sg.C_in_pad + c_base + cg * kOutVec;
            if constexpr (BF16) {
                uint32_t w4[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)   // exact: the values came from bf16
                    w4[k] = (__float_as_uint(val[2 * k]) >> 16) |
                            (__float_as_uint(val[2 * k + 1]) & 0xFFFF0000u);
                *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(xs) + o) =
                    make_uint4(w4[0], w4[1], w4[2], w4[3]);
            } else {
                float hi[4];
                uint32_t cr[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) hi[k] = ptx::split_x(val[k], cr[k]);
                *reinterpret_cast<float4 *>(static_cast<float *>(xs) + o) =
                    make_float4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4 *>(static_cast<float *>(xs) + lo_off + o) =
                    make_uint4(cr[0], cr[1], cr[2], cr[3]);
            }
        }
        // Zeros of the staged positions no tile covers: the left halo (first tile of the
        // row) and the positions past the last tile (last tile of the row).
        auto zero_cols = [&](int64_t px_begin, int64_t px_end) {
            constexpr int kVecs = kStageC / kOutVec;
            const int64_t n_items = (px_end - px_begin) * kVecs;
            for (int64_t i = threadIdx.x; i < n_items; i += kStageThreads) {
                const int64_t px = px_begin + i / kVecs;
                const int64_t o = (row * sg.Px + px) * sg.C_in_pad + c_base + (i % kVecs) * kOutVec;
                *reinterpret_cast<uint4 *>(static_cast<T *>(xs) + o) = make_uint4(0u, 0u, 0u, 0u);
                if constexpr (!BF16)
                    *reinterpret_cast<uint4 *>(static_cast<float *>(xs) + lo_off + o) =
                        make_uint4(0u, 0u, 0u, 0u);
            }
        };
        if (xt == 0) zero_cols(0, sg.hx < sg.Px ? sg.hx : sg.Px);
        if (xt == su.xtiles - 1 && sg.hx + kStageTP * su.xtiles < sg.Px)
            zero_cols(sg.hx + kStageTP * su.xtiles, sg.Px);
        __syncthreads();   // the tile is reused by the next iteration
    }
}

// -------------------------------------------------------------------------- stage_nhwc
// The staged operand from a channels-last x: staged row n = (b*Py + py')*Px + px' holds
// x[b, py' - hy, px' - hx, 0 .. C_in) followed by zeros up to C_in_pad, or zeros outside the
// input.  One thread per 16-byte vector of a staged row: consecutive threads read and write
// consecutive bytes of one position.  fp32 input becomes the tf32 and cross planes; 16-bit input
// is moved as raw payloads.  VEC: x rows are whole 16-byte vectors (C_in * esize % 16 == 0).
template <bool B16, bool VEC>
__global__ void __launch_bounds__(256) stage_nhwc_kernel(const void *__restrict__ x,
                                                         void *__restrict__ xs, StageGeo sg,
                                                         int64_t total) {
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    using E = typename std::conditional<B16, uint16_t, uint32_t>::type;
    constexpr int kVec = 16 / (int)sizeof(E);           // elements per vector
    const int64_t vpr = sg.C_in_pad / kVec;             // vectors per staged row
    const int64_t lo_off = sg.N_total * sg.C_in_pad;    // elements to the cross plane
    const E *__restrict__ xe = static_cast<const E *>(x);
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = i / vpr;
        const int64_t c0 = (i - n * vpr) * kVec;
        const int64_t row = n / sg.Px;                  // b*Py + py'
        const int64_t px = n - row * sg.Px;
        const int64_t b = row / sg.Py;
        const int64_t yy = row - b * sg.Py - sg.hy, xx = px - sg.hx;
        E v[kVec];
#pragma unroll
        for (int k = 0; k < kVec; ++k) v[k] = 0;
        if (yy >= 0 && yy < sg.H && xx >= 0 && xx < sg.W && c0 < sg.C_in) {
            const E *src = xe + ((b * sg.H + yy) * sg.W + xx) * sg.C_in + c0;
            if (VEC && c0 + kVec <= sg.C_in) {
                const uint4 q = *reinterpret_cast<const uint4 *>(src);
                *reinterpret_cast<uint4 *>(v) = q;
            } else {
#pragma unroll
                for (int k = 0; k < kVec; ++k)
                    if (c0 + k < sg.C_in) v[k] = src[k];
            }
        }
        const int64_t o = n * sg.C_in_pad + c0;
        if constexpr (B16) {
            *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(xs) + o) = *reinterpret_cast<uint4 *>(v);
        } else {
            float hi[4];
            uint32_t cr[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) hi[k] = ptx::split_x(__uint_as_float(v[k]), cr[k]);
            *reinterpret_cast<float4 *>(static_cast<float *>(xs) + o) = make_float4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4 *>(static_cast<float *>(xs) + lo_off + o) =
                make_uint4(cr[0], cr[1], cr[2], cr[3]);
        }
    }
}

// -------------------------------------------------------------------------- split-K reduce
// One warp per (32 consecutive phase positions, 32-row chunk r0): sums the split-K partials
// raw[z][n][r0 .. r0+31] in a fixed order (z = 0, 1, ...), then runs the same output stage as
// the fused epilogue, which wants lane i to hold position n0 + i (positions padded to a
// multiple of 32; lanes past the end store nothing).  The partials are read coalesced: each
// 16-byte load instruction covers four positions' whole 128-byte runs (lane l: position
// n0 + 4i + l/8, rows r0 + 4(l%8) ..), and the sums reach their lanes through a 32 x 33
// shared tile (conflict-free both ways).  Each sum is the same sequence of fp32 additions as
// one thread per position would make.
constexpr int kReduceThreads = 64;

__global__ void __launch_bounds__(kReduceThreads)
    splitk_reduce_kernel(const float *__restrict__ raw, EpiParams ep, int64_t ld,
                         int64_t split_stride, int splits, int64_t n_rows, int64_t n_pad,
                         int64_t r_chunks) {
    __shared__ float tile[kReduceThreads / 32][32][33];
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n_pad * r_chunks) return;   // whole warps: n_pad * r_chunks is a multiple of 32
    const int lane = (int)(threadIdx.x & 31);
    float(*t)[33] = tile[threadIdx.x >> 5];
    const int64_t rc = idx / n_pad;
    const int64_t n = idx - rc * n_pad;     // this lane's position in the output stage
    const int64_t n0 = n - lane;
    const int64_t r0 = rc * 32;
    const int c4 = 4 * (lane & 7);
    const float *base = raw + r0 + c4;
    int64_t off[8];
    bool live[8];
    float4 sum[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t np = n0 + 4 * i + (lane >> 3);
        live[i] = np < n_rows;
        off[i] = np * ld;
        sum[i] = live[i] ? *reinterpret_cast<const float4 *>(base + off[i])
                         : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    // Two partials' loads in flight at once; the additions still run in split order.
    for (int z = 1; z < splits; z += 2) {
        float4 a[2][8];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            if (z + u >= splits) break;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                a[u][i] = live[i] ? *reinterpret_cast<const float4 *>(base + (z + u) * split_stride + off[i])
                                  : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            if (z + u >= splits) break;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                sum[i].x += a[u][i].x;
                sum[i].y += a[u][i].y;
                sum[i].z += a[u][i].z;
                sum[i].w += a[u][i].w;
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float *row = t[4 * i + (lane >> 3)] + c4;
        row[0] = sum[i].x;
        row[1] = sum[i].y;
        row[2] = sum[i].z;
        row[3] = sum[i].w;
    }
    __syncwarp();
    float v[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) v[r] = t[lane][r];
    // decode_pos marks positions at or past n_rows (= B * Py * Px) invalid.
    emit_cols<kOutBoth, kIoAny>(v, decode_pos(n, ep), r0, ep, lane);
}

// -------------------------------------------------------------------------- streaming
// A streaming 1-D plan computes its call's s*L output samples from the staged input with the
// previous call's last m - 1 frames in the leading halo (the polyphase conv reads frames
// q - (m - 1) .. q for phase position q).  One thread per (batch item, staged element column
// c, plane): it reads the carried frames and the new last frames first, then writes the halo
// and the new carried frames, so no element is read after another thread wrote it.  With
// fewer than m - 1 new frames the older carried frames shift down.
//   staged rows of batch item b: b*P + r, r = (m - 1) + frame;  state rows: b*(m - 1) + i
template <typename E>
__global__ void stream_state_kernel(E *__restrict__ xs, E *__restrict__ state, int64_t B,
                                    int64_t P, int64_t L, int carry, int64_t row_elems,
                                    int64_t xs_plane, int64_t st_plane, int planes) {
    const int64_t total = B * row_elems * planes;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t c = idx % row_elems;
        const int64_t rest = idx / row_elems;
        const int plane = (int)(rest % planes);
        const int64_t b = rest / planes;
        E *xp = xs + plane * xs_plane + b * P * row_elems + c;
        E *sp = state + plane * st_plane + b * carry * row_elems + c;
        E old[kMaxStreamCarry], nxt[kMaxStreamCarry];
#pragma unroll
        for (int i = 0; i < kMaxStreamCarry; ++i) {
            if (i >= carry) break;
            old[i] = sp[(int64_t)i * row_elems];
        }
#pragma unroll
        for (int i = 0; i < kMaxStreamCarry; ++i) {
            if (i >= carry) break;
            // frame L - carry + i of this call: staged row L + i, or an older carried frame
            nxt[i] = L + i < carry ? old[L + i] : xp[(L + i) * row_elems];
        }
#pragma unroll
        for (int i = 0; i < kMaxStreamCarry; ++i) {
            if (i >= carry) break;
            xp[(int64_t)i * row_elems] = old[i];
            sp[(int64_t)i * row_elems] = nxt[i];
        }
    }
}

// -------------------------------------------------------------------------- col2im
// y[b, oc, oy, ox] = bias + sum of col[(b, iy, ix), (oc, ty, tx)] over the taps that reach
// (oy, ox) (the same divisibility rule as the gather kernel), summed over split-K partials
// in a fixed order.  Only reachable taps are visited ("[WebGPU] optimizations for audio
// models", review commit: each chunk gathers only into the box its rows reach).
__global__ void col2im_kernel(const float *__restrict__ col, int64_t ld, int64_t split_stride,
                              int splits, int S_pad, const void *__restrict__ bias,
                              void *__restrict__ y, Geo g, int64_t total) {
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const OutIdx o = out_index(idx, g);
        const int64_t ox = o.ox, oy = o.oy, oc = o.oc, b = o.b;
        float acc = bias ? load_io(bias, oc, g.io) : 0.0f;
        const int64_t ry = oy + g.py, rx = ox + g.px;
        const TapRange try_ = tap_range(ry, g.sy, g.dy), trx = tap_range(rx, g.sx, g.dx);
        for (int64_t ty = try_.t0; ty < g.ky; ty += try_.step) {
            const int64_t ny = ry - ty * g.dy;
            if (ny < 0) break;
            if (ny % g.sy) continue;
            const int64_t iy = ny / g.sy;
            if (iy >= g.H) continue;
            for (int64_t tx = trx.t0; tx < g.kx; tx += trx.step) {
                const int64_t nx = rx - tx * g.dx;
                if (nx < 0) break;
                if (nx % g.sx) continue;
                const int64_t ix = nx / g.sx;
                if (ix >= g.W) continue;
                const int64_t r = oc * S_pad + ty * g.kx + tx;
                const int64_t n = (b * g.H + iy) * g.W + ix;
                const float *p = col + n * ld + r;
                for (int z = 0; z < splits; ++z) acc += p[(int64_t)z * split_stride];
            }
        }
        store_io(y, idx, apply_act(acc, g.act, g.slope), g.io);
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
    pg.mky = pl->mk[0];
    pg.mkx = pl->mk[1];
    pg.pmy = pl->pm[0];
    pg.pmx = pl->pm[1];
    pg.dy = pl->dil[0];
    pg.dx = pl->dil[1];
    pg.S = pl->S;
    pg.S_pad = pl->S_pad;
    pg.polyphase = pl->path == CTR_PATH_POLYPHASE ? 1 : 0;
    pg.io = pl->dtype;
    pg.pm_tc = pl->row_pm ? pl->block_n / pl->S_pad : 0;
    pg.block_n = pl->block_n;
    const int64_t total = pg.M_pad * pg.K_total;
    prepack_kernel<<<grid_for(total, kBlock), kBlock, 0, st>>>(w, w_packed, pg);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_stream_state(const ctr_plan_s *pl, void *xs, void *state, cudaStream_t st) {
    const int carry = (int)(pl->m[1] - 1);
    if (carry <= 0) return cudaSuccess;
    const bool bf16 = pl->dtype != CTR_F32;   // 16-bit elements (bf16 or fp16), one plane
    const int planes = bf16 ? 1 : 2;
    const int64_t xs_plane = pl->N_total * pl->C_in_pad;         // elements per staged plane
    const int64_t st_plane = pl->B * carry * pl->C_in_pad;
    const int64_t total = pl->B * pl->C_in_pad * planes;
    if (bf16) {
        stream_state_kernel<uint16_t><<<grid_for(total, kBlock), kBlock, 0, st>>>(
            static_cast<uint16_t *>(xs), static_cast<uint16_t *>(state), pl->B, pl->P[1],
            pl->in[1], carry, pl->C_in_pad, xs_plane, st_plane, planes);
    } else {
        stream_state_kernel<uint32_t><<<grid_for(total, kBlock), kBlock, 0, st>>>(
            static_cast<uint32_t *>(xs), static_cast<uint32_t *>(state), pl->B, pl->P[1],
            pl->in[1], carry, pl->C_in_pad, xs_plane, st_plane, planes);
    }
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
    sg.hy = pl->hf[0];
    sg.hx = pl->hf[1];
    sg.N_total = pl->N_total;
    sg.b16 = pl->dtype != CTR_F32;
    if (sg.N_total == 0) return cudaSuccess;
    StageUnits su;
    su.cchunks = sg.C_in_pad / (sg.b16 ? 64 : 32);
    su.x_first = 0;
    su.xtiles = std::max<int64_t>(1, ceil_div(sg.W, kStageTP));
    su.tiles = sg.B * sg.Py * su.xtiles * su.cchunks;
    const int64_t blocks = std::min<int64_t>(su.tiles, (int64_t)pl->num_sms * 8);
    const bool vec = (sg.W * (sg.b16 ? 2 : 4)) % 16 == 0;
    const dim3 grid((unsigned)blocks);
    cudaError_t e;
#define CTR_STAGE(B, V)                                                                   \
    if ((e = prefer_max_smem<stage_x_kernel<B, V>>()) != cudaSuccess) return e;          \
    e = launch_pdl(stage_x_kernel<B, V>, grid, dim3(kStageThreads), 0, st, x, xs, sg, su)
    if (sg.b16) {
        if (vec) { CTR_STAGE(true, true); } else { CTR_STAGE(true, false); }
    } else {
        if (vec) { CTR_STAGE(false, true); } else { CTR_STAGE(false, false); }
    }
#undef CTR_STAGE
    if (e != cudaSuccess) return e;
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_stage_nhwc(const ctr_plan_s *pl, const void *x, void *xs, cudaStream_t st) {
    StageGeo sg;
    sg.B = pl->B;
    sg.C_in = pl->C_in;
    sg.C_in_pad = pl->C_in_pad;
    sg.H = pl->in[0];
    sg.W = pl->in[1];
    sg.Py = pl->P[0];
    sg.Px = pl->P[1];
    sg.hy = pl->hf[0];
    sg.hx = pl->hf[1];
    sg.N_total = pl->N_total;
    sg.b16 = pl->dtype != CTR_F32;
    if (sg.N_total == 0) return cudaSuccess;
    const int es = sg.b16 ? 2 : 4;
    const int64_t total = sg.N_total * sg.C_in_pad * es / 16;
    const bool vec = (sg.C_in * es) % 16 == 0;
    const dim3 grid(grid_for(total, kBlock));
    cudaError_t e;
#define CTR_STAGE(B, V)                                                                   \
    if ((e = prefer_max_smem<stage_nhwc_kernel<B, V>>()) != cudaSuccess) return e;       \
    e = launch_pdl(stage_nhwc_kernel<B, V>, grid, dim3(kBlock), 0, st, x, xs, sg, total)
    if (sg.b16) {
        if (vec) { CTR_STAGE(true, true); } else { CTR_STAGE(true, false); }
    } else {
        if (vec) { CTR_STAGE(false, true); } else { CTR_STAGE(false, false); }
    }
#undef CTR_STAGE
    if (e != cudaSuccess) return e;
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_splitk_reduce(const ctr_plan_s *pl, const float *raw, const EpiParams &ep,
                                 int64_t raw_ld, int64_t split_stride, cudaStream_t st) {
    const int64_t n_rows = pl->N_total;
    const int64_t n_pad = round_up(n_rows, 32);
    // Channel-major rows: the first M_rows rows hold every output.  Phase-major rows (a
    // chained or channels-last output) spread the last tile's channels over its whole width,
    // so every packed row is visited; the output stage skips the padding channels.
    const int64_t r_rows = pl->row_pm ? raw_ld : std::min<int64_t>(pl->M_rows, raw_ld);
    const int64_t r_chunks = ceil_div(r_rows, 32);
    const int64_t total = n_pad * r_chunks;
    if (n_rows == 0 || r_chunks == 0) return cudaSuccess;
    cudaError_t e = prefer_max_smem<splitk_reduce_kernel>();
    if (e != cudaSuccess) return e;
    e = launch_pdl(splitk_reduce_kernel, dim3(grid_for(total, kReduceThreads)),
                   dim3(kReduceThreads), 0, st, raw, ep,
                   raw_ld, split_stride, pl->splits, n_rows, n_pad, r_chunks);
    if (e != cudaSuccess) return e;
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_col2im(const ctr_plan_s *pl, const float *col, int64_t col_ld,
                          const void *bias, void *y, cudaStream_t st) {
    const Geo g = geo_of(pl);
    const int64_t total = g.B * g.C_out * g.Ho * g.Wo;
    if (total == 0) return cudaSuccess;
    const int64_t split_stride = raw_split_stride_of(pl);
    cudaError_t e = prefer_max_smem<col2im_kernel>();
    if (e != cudaSuccess) return e;
    e = launch_pdl(col2im_kernel, dim3(grid_for(total, kBlock)), dim3(kBlock), 0, st, col,
                   col_ld, split_stride, pl->splits, pl->S_pad, bias, y, g, total);
    if (e != cudaSuccess) return e;
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace ctr
