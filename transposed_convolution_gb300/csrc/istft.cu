// istft.cu -- the inverse STFT as an inverse real FFT per frame, a synthesis window and an
// overlap-add.
//
// "[WebGPU] optimizations for audio models" (its description of the source-separation
// model) computes the inverse STFT as a ConvTranspose1d whose weight is the windowed inverse
// real-DFT basis: channel f of the input is the real part of bin f, channel n_fft/2 + 1 + f
// its imaginary part, the kernel is one frame (n_fft samples) and the stride is the hop, so
// the transposed convolution overlap-adds the frames.  Per frame that contraction is the
// windowed inverse real DFT
//
//     frame[t] = win[t] / N * ( Re X_0 + Re X_{N/2} (-1)^t
//                               + 2 sum_{0<f<N/2} (Re X_f cos(2 pi f t/N) - Im X_f sin(2 pi f t/N)) )
//
// (the imaginary parts of bins 0 and N/2 have zero weights), which an FFT computes in
// O(N log N) instead of O(N^2) operations.  The result is the same ConvTranspose: frames at
// stride hop, the padding slice, an optional bias.
//
// Inverse real DFT through a half-size complex FFT (M = N/2).  With x the inverse real DFT
// of X and the Hermitian extension X_{N-f} = conj(X_f):
//   x[2n]   = 1/N sum_{k<M} (X_k + conj(X_{M-k}))                 e^{2 pi i k n / M}
//   x[2n+1] = 1/N sum_{k<M} (X_k - conj(X_{M-k})) e^{2 pi i k/N}   e^{2 pi i k n / M}
// (split the sum over f into k and k + M).  Both bracketed sequences E_k, O_k are spectra of
// real sequences, so z = IDFT_M(E + i O), unnormalised, holds N x[2n] in its real part and
// N x[2n+1] in its imaginary part.  The length-M inverse transform is a mixed-radix Stockham
// autosort FFT between two shared-memory buffers (Govindaraju et al., "High performance
// discrete Fourier transforms on graphics processors", SC 2008): radix-16 passes, with one
// radix-2, -4 or -8 pass first when log2 M is not a multiple of 4, each butterfly's R points
// held in registers, so M = 2048 takes three passes over shared memory.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <new>

#include "ctr_internal.h"

struct ctr_istft_s {
    int64_t B, n_fft, hop, frames, pad, opad, L_out;
    int dtype;
    int fpb;                 // frames per block of the FFT kernel
    size_t smem;             // its dynamic shared memory
    size_t off_tw, off_win, off_frames, off_rows, ws_needed;
    void *ws;
    size_t ws_bytes;
    int window_set;
    cudaEvent_t ev_before, ev_after;   // optional timing events around the two kernels
};

namespace ctr {
namespace {

constexpr int kFftBlock = 256;

__device__ __forceinline__ float2 cadd(float2 a, float2 b) { return make_float2(a.x + b.x, a.y + b.y); }
__device__ __forceinline__ float2 csub(float2 a, float2 b) { return make_float2(a.x - b.x, a.y - b.y); }
__device__ __forceinline__ float2 cmul(float2 a, float2 b) {
    return make_float2(a.x * b.x - a.y * b.y, a.x * b.y + a.y * b.x);
}
__device__ __forceinline__ float2 conjf2(float2 a) { return make_float2(a.x, -a.y); }
__device__ __forceinline__ float2 times_i(float2 a) { return make_float2(-a.y, a.x); }

// tw[m] = e^{2 pi i m / N} (double-precision sincospi, rounded once), win[t] = window[t] / N
// (exact: N is a power of two).
__global__ void istft_init_kernel(float2 *__restrict__ tw, float *__restrict__ win,
                                  const float *__restrict__ window, int N) {
    for (int m = blockIdx.x * blockDim.x + threadIdx.x; m < N; m += gridDim.x * blockDim.x) {
        double s, c;
        sincospi(2.0 * (double)m / (double)N, &s, &c);
        tw[m] = make_float2((float)c, (float)s);
        win[m] = window[m] / (float)N;
    }
}

struct FftGeo {
    int T, C;                // frames, input channels (N + 2)
    int N, M, logM;          // frame length, half length, log2(M)
    int Mp;                  // pitch of the spectrum rows: M + 2 pairs (16-byte rows)
    int Ms;                  // pitch of a frame's FFT buffer in shared memory (padded indices)
    int fpb;                 // frames per block
};

// Onesided spectra, channel-major [b][c][t] (c < M + 1: real part of bin c, else imaginary
// part of bin c - M - 1), to frame-major complex rows Z[b][t][f] = (Re X_f, Im X_f), f <= M,
// rows of Mp float2.  One 32-bin x 32-frame tile per block through shared memory: a warp
// reads 32 consecutive frames of one channel and writes 32 consecutive bins of one frame, so
// both sides are coalesced (the FFT kernel then copies whole rows).  Every load of a thread
// is issued before the first shared-memory store.
constexpr int kTile = 32;

__global__ void __launch_bounds__(256)
spectrum_rows_kernel(const float *__restrict__ spec, float2 *__restrict__ Z, FftGeo g) {
    __shared__ float re[kTile][kTile + 1], im[kTile][kTile + 1];
    const int b = blockIdx.z;
    const int f0 = blockIdx.y * kTile, t0 = blockIdx.x * kTile;
    const int lx = threadIdx.x & 31, ly = threadIdx.x >> 5;
    const int M = g.M;
    const float *sb = spec + (int64_t)b * g.C * g.T;
    float a[kTile / 8], c[kTile / 8];
#pragma unroll
    for (int i = 0; i < kTile / 8; ++i) {
        const int f = f0 + ly + 8 * i, t = t0 + lx;
        const bool in = f <= M && t < g.T;
        a[i] = in ? __ldg(sb + (int64_t)f * g.T + t) : 0.0f;
        c[i] = in ? __ldg(sb + (int64_t)(M + 1 + f) * g.T + t) : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < kTile / 8; ++i) {
        re[ly + 8 * i][lx] = a[i];
        im[ly + 8 * i][lx] = c[i];
    }
    __syncthreads();
    float2 *zb = Z + (int64_t)b * g.T * g.Mp;
#pragma unroll
    for (int i = 0; i < kTile / 8; ++i) {
        const int r = ly + 8 * i;
        const int t = t0 + r, f = f0 + lx;
        if (t < g.T && f <= M) zb[(int64_t)t * g.Mp + f] = make_float2(re[lx][r], im[lx][r]);
    }
}

__device__ __forceinline__ void cp_async8(void *smem_dst, const void *gmem_src) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(d), "l"(gmem_src) : "memory");
}

// Shared-memory position of FFT element i: one pad entry after every 16, so that the strided
// accesses of the passes (stride 16 pairs in the first radix-16 pass) spread over all banks.
__device__ __forceinline__ int sidx(int i) { return i + (i >> 4); }

// In-place inverse DFT of R points, v[q] <- sum_r v[r] e^{+2 pi i r q / R}, natural order.
__device__ __forceinline__ void idft4(float2 &u0, float2 &u1, float2 &u2, float2 &u3) {
    const float2 a0 = cadd(u0, u2), a1 = csub(u0, u2);
    const float2 a2 = cadd(u1, u3), a3 = times_i(csub(u1, u3));   // e^{+2 pi i / 4} = i
    u0 = cadd(a0, a2);
    u1 = cadd(a1, a3);
    u2 = csub(a0, a2);
    u3 = csub(a1, a3);
}

// e^{+2 pi i m / 16} for m = 1 .. 9 (cos and sin of multiples of pi/8).
__device__ __forceinline__ float2 w16(int m) {
    constexpr float c1 = 0.92387953251128674f, s1 = 0.38268343236508979f,
                    h = 0.70710678118654752f;
    switch (m) {
        case 1: return make_float2(c1, s1);
        case 2: return make_float2(h, h);
        case 3: return make_float2(s1, c1);
        case 4: return make_float2(0.0f, 1.0f);
        case 6: return make_float2(-h, h);
        case 9: return make_float2(-c1, -s1);
        default: return make_float2(1.0f, 0.0f);
    }
}

template <int R>
__device__ __forceinline__ void idft(float2 (&v)[R]) {
    if constexpr (R == 2) {
        const float2 a = v[0];
        v[0] = cadd(a, v[1]);
        v[1] = csub(a, v[1]);
    } else if constexpr (R == 4) {
        idft4(v[0], v[1], v[2], v[3]);
    } else if constexpr (R == 8) {
        // Even and odd points: two 4-point transforms, then V_q = E_q + w^q O_q and
        // V_{q+4} = E_q - w^q O_q with w = e^{+2 pi i / 8}.
        idft4(v[0], v[2], v[4], v[6]);
        idft4(v[1], v[3], v[5], v[7]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 o = q == 0 ? v[1] : cmul(v[2 * q + 1], w16(2 * q));
            const float2 e = v[2 * q];
            v[2 * q] = cadd(e, o);
            v[2 * q + 1] = csub(e, o);
        }
        // v[2q] holds V_q, v[2q+1] holds V_{q+4}: back to natural order.
        float2 t[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            t[q] = v[2 * q];
            t[q + 4] = v[2 * q + 1];
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = t[q];
    } else {
        static_assert(R == 16, "radix 2, 4, 8 or 16");
        // r = 4 r1 + r2, q = q1 + 4 q2: 4-point transforms over r1 for each r2, the twiddle
        // e^{+2 pi i r2 q1 / 16}, then 4-point transforms over r2 for each q1.
#pragma unroll
        for (int r2 = 0; r2 < 4; ++r2) idft4(v[r2], v[4 + r2], v[8 + r2], v[12 + r2]);
        // v[4 q1 + r2] now holds A[r2][q1].
#pragma unroll
        for (int r2 = 1; r2 < 4; ++r2)
#pragma unroll
            for (int q1 = 1; q1 < 4; ++q1) v[4 * q1 + r2] = cmul(v[4 * q1 + r2], w16(r2 * q1));
#pragma unroll
        for (int q1 = 0; q1 < 4; ++q1) idft4(v[4 * q1], v[4 * q1 + 1], v[4 * q1 + 2], v[4 * q1 + 3]);
        // v[4 q1 + q2] now holds V[q1 + 4 q2]: transpose the 4x4 index.
        float2 t[16];
#pragma unroll
        for (int q1 = 0; q1 < 4; ++q1)
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2) t[q1 + 4 * q2] = v[4 * q1 + q2];
#pragma unroll
        for (int q = 0; q < 16; ++q) v[q] = t[q];
    }
}

// One Stockham pass of radix R over fpb frames, Ns points already combined: butterfly j reads
// in[j + r M/R], twiddles point r by w^r, w = e^{2 pi i (j mod Ns)/(Ns R)} = tw[(j mod Ns) N/(Ns R)],
// takes the R-point inverse DFT and writes out[(j - j mod Ns) R + j mod Ns + q Ns].
template <int R>
__device__ __forceinline__ void fft_pass(const float2 *in, float2 *out, const float2 *tw,
                                         const FftGeo &g, int Ns) {
    constexpr int kLogR = R == 2 ? 1 : R == 4 ? 2 : R == 8 ? 3 : 4;
    const int lognb = g.logM - kLogR;
    const int nb = 1 << lognb;
    const int tstep = g.N / (Ns * R);
    const int total = nb * g.fpb;
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
        const int f = i >> lognb, j = i & (nb - 1);
        const float2 *I = in + (size_t)f * g.Ms;
        float2 *O = out + (size_t)f * g.Ms;
        const int k = j & (Ns - 1);
        float2 v[R];
#pragma unroll
        for (int r = 0; r < R; ++r) v[r] = I[sidx(j + r * nb)];
        if (Ns > 1) {
            // w^r for w = e^{2 pi i k/(Ns R)}: w^{4a} from the table, w^{4a+b} = w^{4a} w^b
            // with w^2 = w w and w^3 = w^2 w (at most three roundings each), so a butterfly
            // loads R/4 twiddles (one for R = 2) instead of R - 1.
            float2 wr[R];
            wr[1] = __ldg(&tw[k * tstep]);
            if constexpr (R >= 4) {
                wr[2] = cmul(wr[1], wr[1]);
                wr[3] = cmul(wr[2], wr[1]);
            }
#pragma unroll
            for (int a = 1; a < R / 4; ++a) {
                const float2 wa = __ldg(&tw[4 * a * k * tstep]);
                wr[4 * a] = wa;
                wr[4 * a + 1] = cmul(wa, wr[1]);
                wr[4 * a + 2] = cmul(wa, wr[2]);
                wr[4 * a + 3] = cmul(wa, wr[3]);
            }
#pragma unroll
            for (int r = 1; r < R; ++r) v[r] = cmul(v[r], wr[r]);
        }
        idft<R>(v);
        const int o = (j - k) * R + k;
#pragma unroll
        for (int q = 0; q < R; ++q) O[sidx(o + q * Ns)] = v[q];
    }
}

// One block transforms fpb consecutive frames of one batch item: copies their spectrum rows,
// folds each into Z = E + iO (above), runs the inverse Stockham FFT and writes the windowed
// frames, fp32, to frames[b][t][N].
__global__ void __launch_bounds__(kFftBlock)
irfft_frames_kernel(const float2 *__restrict__ Zrows, const float2 *__restrict__ tw,
                    const float *__restrict__ win, float *__restrict__ frames, FftGeo g) {
    extern __shared__ __align__(16) unsigned char fft_smem[];
    const int M = g.M, N = g.N, fpb = g.fpb, Ms = g.Ms;
    float2 *bufA = reinterpret_cast<float2 *>(fft_smem);       // [fpb][Ms]
    float2 *bufB = bufA + (size_t)fpb * Ms;                     // [fpb][Ms]
    const int b = blockIdx.y;
    const int t0 = blockIdx.x * fpb;
    const int tid = threadIdx.x;

    // 1. Spectrum rows (bins 0..M), all copies in flight at once; frames past the end are
    //    zeros.  Pairs 2m, 2m + 1 stay adjacent under sidx, so each copy moves 8 bytes.
    for (int f = 0; f < fpb; ++f) {
        const int t = t0 + f;
        float2 *dst = bufA + (size_t)f * Ms;
        if (t < g.T) {
            const float2 *src = Zrows + ((int64_t)b * g.T + t) * g.Mp;
            for (int i = tid; i <= M; i += kFftBlock) cp_async8(dst + sidx(i), src + i);
        } else {
            for (int i = tid; i <= M; i += kFftBlock) dst[sidx(i)] = make_float2(0.f, 0.f);
        }
    }
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
    __syncthreads();

    // 2. Z_k = E_k + i O_k in place; a thread owns the pair (k, M - k), which read each other.
    //    Im X_0 and Im X_M do not enter (their basis rows are zero).
    const int npair = M / 2 + 1;
    for (int f = 0; f < fpb; ++f) {
        float2 *X = bufA + (size_t)f * Ms;
        for (int k = tid; k < npair; k += kFftBlock) {
            const int j = M - k;
            if (k == 0) {
                const float x0 = X[0].x, xm = X[sidx(M)].x;
                X[0] = make_float2(x0 + xm, x0 - xm);
            } else {
                const float2 xk = X[sidx(k)], xj = X[sidx(j)];
                const float2 ek = cadd(xk, conjf2(xj)), ok = cmul(csub(xk, conjf2(xj)), __ldg(&tw[k]));
                X[sidx(k)] = cadd(ek, times_i(ok));
                if (j != k) {
                    const float2 ej = cadd(xj, conjf2(xk)), oj = cmul(csub(xj, conjf2(xk)), __ldg(&tw[j]));
                    X[sidx(j)] = cadd(ej, times_i(oj));
                }
            }
        }
    }
    __syncthreads();

    // 3. Inverse FFT of length M (sign +): one radix-2/4/8 pass for log2 M mod 4, then
    //    radix-16 passes.
    float2 *in = bufA, *out = bufB;
    int Ns = 1;
    const int first = g.logM & 3;
    if (first) {
        if (first == 1) fft_pass<2>(in, out, tw, g, 1);
        else if (first == 2) fft_pass<4>(in, out, tw, g, 1);
        else fft_pass<8>(in, out, tw, g, 1);
        __syncthreads();
        float2 *t = in; in = out; out = t;
        Ns = 1 << first;
    }
    for (; Ns < M; Ns *= 16) {
        fft_pass<16>(in, out, tw, g, Ns);
        __syncthreads();
        float2 *t = in; in = out; out = t;
    }

    // 4. frame[2n] = win[2n] Re z_n / N, frame[2n + 1] = win[2n + 1] Im z_n / N.
    for (int f = 0; f < fpb; ++f) {
        const int t = t0 + f;
        if (t >= g.T) break;
        const float2 *zr = in + (size_t)f * Ms;
        float2 *fr = reinterpret_cast<float2 *>(frames + ((int64_t)b * g.T + t) * N);
        for (int n = tid; n < M; n += kFftBlock) {
            const float2 z = zr[sidx(n)];
            const float2 w2 = __ldg(reinterpret_cast<const float2 *>(win) + n);
            fr[n] = make_float2(z.x * w2.x, z.y * w2.y);
        }
    }
}

struct OlaGeo {
    int T, N, hop, pad, L_out;
    int vec;                 // 4 consecutive outputs per thread with 16-byte accesses
};

// y[b, 0, n'] = bias + sum over the frames k that cover n = n' + pad of frame_k[n - k hop],
// in ascending k (the overlap-add of the transposed convolution, as a gather: no atomics).
// blockIdx.y is the batch item; positions and frame offsets are 32-bit (checked at plan
// creation), the batch item's base 64-bit.  With hop, pad, N and L_out multiples of 4 a
// thread sums four consecutive outputs, which share their frames, with float4 loads and one
// float4 store (the same sums in the same order).
__global__ void istft_ola_kernel(const float *__restrict__ frames, const float *__restrict__ bias,
                                 float *__restrict__ y, OlaGeo g) {
    const float b0 = bias ? bias[0] : 0.0f;
    const float *fb = frames + (int64_t)blockIdx.y * g.T * g.N;
    float *yb = y + (int64_t)blockIdx.y * g.L_out;
    if (g.vec) {
        const int nq = g.L_out / 4;
        for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nq; i += gridDim.x * blockDim.x) {
            const int n = 4 * i + g.pad;
            const int k_hi = min(g.T - 1, n / g.hop);
            const int k_lo = n >= g.N ? (n - g.N) / g.hop + 1 : 0;
            float4 acc = make_float4(b0, b0, b0, b0);
            // Up to four frames' loads in flight before the first add (hop = N/4 has four);
            // any further frames follow one by one.  The sums keep ascending k.
            float4 v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                v[q] = k_lo + q <= k_hi
                           ? __ldg(reinterpret_cast<const float4 *>(fb + (int64_t)(k_lo + q) * (g.N - g.hop) + n))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (k_lo + q > k_hi) break;
                acc.x += v[q].x;
                acc.y += v[q].y;
                acc.z += v[q].z;
                acc.w += v[q].w;
            }
            for (int k = k_lo + 4; k <= k_hi; ++k) {
                const float4 u = __ldg(reinterpret_cast<const float4 *>(fb + (int64_t)k * (g.N - g.hop) + n));
                acc.x += u.x;
                acc.y += u.y;
                acc.z += u.z;
                acc.w += u.w;
            }
            reinterpret_cast<float4 *>(yb)[i] = acc;
        }
        return;
    }
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < g.L_out; i += gridDim.x * blockDim.x) {
        const int n = i + g.pad;
        const int k_hi = min(g.T - 1, n / g.hop);
        const int k_lo = n >= g.N ? (n - g.N) / g.hop + 1 : 0;
        float acc = b0;
        for (int k = k_lo; k <= k_hi; ++k) acc += fb[(int64_t)k * (g.N - g.hop) + n];
        yb[i] = acc;
    }
}

bool is_pow2(int64_t v) { return v > 0 && (v & (v - 1)) == 0; }
// Shared-memory pitch of one frame's FFT buffer: padded positions of bins 0..M (sidx(M) + 1),
// rounded up to an even count so every frame's buffer starts 16-byte aligned.
int64_t fft_pitch(int64_t M) { return ((M + (M >> 4) + 1) + 1) & ~(int64_t)1; }
size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }
bool aligned16p(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace ctr

using namespace ctr;

extern "C" {

ctr_status ctr_istft_create(ctr_istft_t *out, int64_t N, int64_t n_fft, int64_t hop,
                            int64_t frames, int64_t padding, int64_t output_padding, int dtype) {
    if (!out) return CTR_ERR_INVALID_ARG;
    *out = nullptr;
    if (dtype != CTR_F32 && dtype != CTR_BF16 && dtype != CTR_F16) return CTR_ERR_INVALID_ARG;
    if (N < 0 || frames < 0 || hop < 1 || padding < 0 || output_padding < 0 ||
        output_padding >= hop || !is_pow2(n_fft) || n_fft < 4 || n_fft > 8192)
        return CTR_ERR_INVALID_ARG;
    // Batch items are grid rows (<= 65535); positions, frames and offsets inside a batch
    // item's frames are 32-bit.
    const int64_t lim = (int64_t)1 << 30;
    if (N > 65535 || frames >= lim || hop >= lim || padding >= lim) return CTR_ERR_INVALID_ARG;
    const int64_t L_out = (frames - 1) * hop - 2 * padding + n_fft + output_padding;
    if (L_out < 1 || L_out + padding >= lim || frames * n_fft >= lim ||
        N * frames * n_fft >= ((int64_t)1 << 46))
        return CTR_ERR_INVALID_ARG;
    if (dtype != CTR_F32) return CTR_ERR_UNSUPPORTED;
    ctr_istft_s *p = new (std::nothrow) ctr_istft_s();
    if (!p) return CTR_ERR_INVALID_ARG;
    p->B = N;
    p->n_fft = n_fft;
    p->hop = hop;
    p->frames = frames;
    p->pad = padding;
    p->opad = output_padding;
    p->L_out = L_out;
    p->dtype = dtype;
    const int64_t M = n_fft / 2;
    p->fpb = (int)std::min<int64_t>(16, std::max<int64_t>(1, 4096 / M));   // ~64 KB a block
    p->smem = (size_t)p->fpb * 2 * fft_pitch(M) * sizeof(float2);
    p->off_tw = 0;
    p->off_win = align256((size_t)n_fft * sizeof(float2));
    p->off_frames = p->off_win + align256((size_t)n_fft * sizeof(float));
    p->off_rows = p->off_frames + align256((size_t)(N * frames * n_fft) * sizeof(float));
    p->ws_needed = p->off_rows + (size_t)(N * frames * (M + 2)) * sizeof(float2);
    *out = p;
    return CTR_OK;
}

ctr_status ctr_istft_output_length(ctr_istft_t p, int64_t *L_out) {
    if (!p || !L_out) return CTR_ERR_INVALID_ARG;
    *L_out = p->L_out;
    return CTR_OK;
}

size_t ctr_istft_workspace_bytes(ctr_istft_t p) { return p ? p->ws_needed : 0; }

ctr_status ctr_istft_bind_workspace(ctr_istft_t p, void *ws, size_t bytes) {
    if (!p || !ws) return CTR_ERR_INVALID_ARG;
    if (!aligned16p(ws)) return CTR_ERR_MISALIGNED;
    if (bytes < p->ws_needed) return CTR_ERR_NO_WORKSPACE;
    p->ws = ws;
    p->ws_bytes = bytes;
    p->window_set = 0;
    return CTR_OK;
}

ctr_status ctr_istft_set_window(ctr_istft_t p, const void *window, void *stream) {
    if (!p || !window) return CTR_ERR_INVALID_ARG;
    if (!aligned16p(window)) return CTR_ERR_MISALIGNED;
    if (!p->ws) return CTR_ERR_NO_WORKSPACE;
    char *ws = static_cast<char *>(p->ws);
    const int N = (int)p->n_fft;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaFuncSetAttribute(irfft_frames_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)p->smem) != cudaSuccess)
        return CTR_ERR_CUDA;
    istft_init_kernel<<<(N + 255) / 256, 256, 0, st>>>(
        reinterpret_cast<float2 *>(ws + p->off_tw), reinterpret_cast<float *>(ws + p->off_win),
        static_cast<const float *>(window), N);
    count_launches(1);
    if (cudaGetLastError() != cudaSuccess) return CTR_ERR_CUDA;
    p->window_set = 1;
    return CTR_OK;
}

ctr_status ctr_istft_forward(ctr_istft_t p, const void *spec, const void *bias, void *y,
                             void *stream) {
    if (!p || !y) return CTR_ERR_INVALID_ARG;
    if (!p->ws) return CTR_ERR_NO_WORKSPACE;
    if (!p->window_set) return CTR_ERR_NOT_PREPARED;
    if (!spec && p->B * p->frames > 0) return CTR_ERR_INVALID_ARG;
    if ((spec && !aligned16p(spec)) || !aligned16p(y) || (bias && !aligned16p(bias)))
        return CTR_ERR_MISALIGNED;
    if (p->B == 0) return CTR_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(p->ws);
    float *frames = reinterpret_cast<float *>(ws + p->off_frames);
    const bool timed = p->ev_before != nullptr;
    if (timed && record_timing(p->ev_before, st) != cudaSuccess) return CTR_ERR_CUDA;
    if (p->frames > 0) {
        FftGeo g;
        g.T = (int)p->frames;
        g.C = (int)(p->n_fft + 2);
        g.N = (int)p->n_fft;
        g.M = g.N / 2;
        g.Mp = g.M + 2;
        g.Ms = (int)fft_pitch(g.M);
        g.logM = 0;
        while ((1 << g.logM) < g.M) ++g.logM;
        g.fpb = p->fpb;
        float2 *rows = reinterpret_cast<float2 *>(ws + p->off_rows);
        const dim3 tgrid((unsigned)((p->frames + kTile - 1) / kTile),
                         (unsigned)((g.M + 1 + kTile - 1) / kTile), (unsigned)p->B);
        spectrum_rows_kernel<<<tgrid, 256, 0, st>>>(static_cast<const float *>(spec), rows, g);
        const dim3 grid((unsigned)((p->frames + p->fpb - 1) / p->fpb), (unsigned)p->B);
        irfft_frames_kernel<<<grid, kFftBlock, p->smem, st>>>(
            rows, reinterpret_cast<const float2 *>(ws + p->off_tw),
            reinterpret_cast<const float *>(ws + p->off_win), frames, g);
        count_launches(2);
        if (cudaGetLastError() != cudaSuccess) return CTR_ERR_CUDA;
    }
    OlaGeo o;
    o.T = (int)p->frames;
    o.N = (int)p->n_fft;
    o.hop = (int)p->hop;
    o.pad = (int)p->pad;
    o.L_out = (int)p->L_out;
    o.vec = (p->hop % 4 == 0 && p->pad % 4 == 0 && p->n_fft % 4 == 0 && p->L_out % 4 == 0) ? 1 : 0;
    const int64_t per_thread = o.vec ? 4 : 1;
    const int64_t oblocks = (p->L_out / per_thread + 255) / 256;
    const dim3 ogrid((unsigned)std::min<int64_t>(oblocks, (int64_t)1 << 20), (unsigned)p->B);
    istft_ola_kernel<<<ogrid, 256, 0, st>>>(frames, static_cast<const float *>(bias),
                                            static_cast<float *>(y), o);
    count_launches(1);
    if (cudaGetLastError() != cudaSuccess) return CTR_ERR_CUDA;
    if (timed && record_timing(p->ev_after, st) != cudaSuccess) return CTR_ERR_CUDA;
    return CTR_OK;
}

ctr_status ctr_istft_set_timing_events(ctr_istft_t p, void *before, void *after) {
    if (!p || (before == nullptr) != (after == nullptr)) return CTR_ERR_INVALID_ARG;
    p->ev_before = static_cast<cudaEvent_t>(before);
    p->ev_after = static_cast<cudaEvent_t>(after);
    return CTR_OK;
}

ctr_status ctr_istft_describe(ctr_istft_t p, char *buf, size_t len) {
    if (!p || !buf || len == 0) return CTR_ERR_INVALID_ARG;
    snprintf(buf, len, "istft n_fft=%lld hop=%lld frames=%lld pad=%lld L_out=%lld fpb=%d smem=%zu ws=%zu",
             (long long)p->n_fft, (long long)p->hop, (long long)p->frames, (long long)p->pad,
             (long long)p->L_out, p->fpb, p->smem, p->ws_needed);
    return CTR_OK;
}

void ctr_istft_destroy(ctr_istft_t p) { delete p; }

}  // extern "C"
