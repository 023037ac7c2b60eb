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
// N x[2n+1] in its imaginary part.  The length-M inverse transform is a Stockham autosort FFT
// in shared memory (radix-4 stages and one radix-2 stage when log2 M is odd; Govindaraju et
// al., "High performance discrete Fourier transforms on graphics processors", SC 2008).
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
    size_t off_tw, off_win, off_frames, ws_needed;
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
    int fpb;                 // frames per block
};

// One block transforms fpb consecutive frames of one batch item: loads their onesided
// spectra, folds each into Z = E + iO (above), runs the inverse Stockham FFT and writes the
// windowed frames, fp32, to frames[b][t][N].
__global__ void __launch_bounds__(kFftBlock)
irfft_frames_kernel(const float *__restrict__ spec, const float2 *__restrict__ tw,
                    const float *__restrict__ win, float *__restrict__ frames, FftGeo g) {
    extern __shared__ __align__(16) unsigned char fft_smem[];
    const int M = g.M, N = g.N, fpb = g.fpb;
    float2 *bufA = reinterpret_cast<float2 *>(fft_smem);       // [fpb][M + 1]
    float2 *bufB = bufA + (size_t)fpb * (M + 1);                // [fpb][M + 1]
    const int b = blockIdx.y;
    const int t0 = blockIdx.x * fpb;
    const int tid = threadIdx.x;
    const float *sp = spec + (int64_t)b * g.C * g.T;

    // 1. Spectra: bin f's real part in channel f, its imaginary part in channel M + 1 + f.
    //    Frame fastest, so a warp reads runs of consecutive frames of a channel.  4-byte
    //    cp.async copies: every load of the block is in flight at once.
    const int nload = 2 * (M + 1) * fpb;
    for (int i = tid; i < nload; i += kFftBlock) {
        const int c = i / fpb, f = i - c * fpb;
        const int t = t0 + f;
        float2 *X = bufA + (size_t)f * (M + 1);
        float *dst = c <= M ? &X[c].x : &X[c - (M + 1)].y;
        if (t < g.T) {
            const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(d),
                         "l"(sp + (int64_t)c * g.T + t)
                         : "memory");
        } else {
            *dst = 0.0f;
        }
    }
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
    __syncthreads();

    // 2. Z_k = E_k + i O_k in place; a thread owns the pair (k, M - k), which read each other.
    //    Im X_0 and Im X_M do not enter (their basis rows are zero).
    const int npair = M / 2 + 1;
    for (int i = tid; i < npair * fpb; i += kFftBlock) {
        const int f = i / npair, k = i - f * npair;
        float2 *X = bufA + (size_t)f * (M + 1);
        const int j = M - k;
        if (k == 0) {
            const float x0 = X[0].x, xm = X[M].x;
            X[0] = make_float2(x0 + xm, x0 - xm);
        } else {
            const float2 xk = X[k], xj = X[j];
            const float2 ek = cadd(xk, conjf2(xj)), ok = cmul(csub(xk, conjf2(xj)), tw[k]);
            X[k] = cadd(ek, times_i(ok));
            if (j != k) {
                const float2 ej = cadd(xj, conjf2(xk)), oj = cmul(csub(xj, conjf2(xk)), tw[j]);
                X[j] = cadd(ej, times_i(oj));
            }
        }
    }
    __syncthreads();

    // 3. Inverse FFT of length M (sign +).  Stage with radix R after Ns points are combined:
    //    butterfly j reads in[j + r M/R], twiddles point r by e^{2 pi i r (j mod Ns)/(Ns R)},
    //    takes the R-point DFT and writes out[(j - j mod Ns) R + j mod Ns + r Ns].
    float2 *in = bufA, *out = bufB;
    int Ns = 1;
    if (g.logM & 1) {   // one radix-2 stage first (Ns = 1: no twiddles)
        const int half = M / 2;
        for (int i = tid; i < half * fpb; i += kFftBlock) {
            const int f = i / half, j = i - f * half;
            const float2 *I = in + (size_t)f * (M + 1);
            float2 *O = out + (size_t)f * (M + 1);
            const float2 a = I[j], c = I[j + half];
            O[2 * j] = cadd(a, c);
            O[2 * j + 1] = csub(a, c);
        }
        __syncthreads();
        float2 *t = in; in = out; out = t;
        Ns = 2;
    }
    for (; Ns < M; Ns *= 4) {
        const int quarter = M / 4;
        const int tstep = N / (Ns * 4);    // e^{2 pi i r k / (4 Ns)} = tw[r k tstep]
        for (int i = tid; i < quarter * fpb; i += kFftBlock) {
            const int f = i / quarter, j = i - f * quarter;
            const float2 *I = in + (size_t)f * (M + 1);
            float2 *O = out + (size_t)f * (M + 1);
            const int k = j & (Ns - 1);
            float2 v0 = I[j], v1 = I[j + quarter], v2 = I[j + 2 * quarter], v3 = I[j + 3 * quarter];
            if (Ns > 1) {
                v1 = cmul(v1, tw[k * tstep]);
                v2 = cmul(v2, tw[2 * k * tstep]);
                v3 = cmul(v3, tw[3 * k * tstep]);
            }
            // 4-point inverse DFT: W = e^{+2 pi i / 4} = i.
            const float2 a0 = cadd(v0, v2), a1 = csub(v0, v2);
            const float2 a2 = cadd(v1, v3), a3 = times_i(csub(v1, v3));
            const int o = (j - k) * 4 + k;
            O[o] = cadd(a0, a2);
            O[o + Ns] = cadd(a1, a3);
            O[o + 2 * Ns] = csub(a0, a2);
            O[o + 3 * Ns] = csub(a1, a3);
        }
        __syncthreads();
        float2 *t = in; in = out; out = t;
    }

    // 4. frame[2n] = win[2n] Re z_n / N, frame[2n + 1] = win[2n + 1] Im z_n / N.
    for (int i = tid; i < M * fpb; i += kFftBlock) {
        const int f = i / M, n = i - f * M;
        const int t = t0 + f;
        if (t >= g.T) continue;
        const float2 z = in[(size_t)f * (M + 1) + n];
        const float2 w2 = reinterpret_cast<const float2 *>(win)[n];
        reinterpret_cast<float2 *>(frames + ((int64_t)b * g.T + t) * N)[n] =
            make_float2(z.x * w2.x, z.y * w2.y);
    }
}

struct OlaGeo {
    int T, N, hop, pad, L_out;
};

// y[b, 0, n'] = bias + sum over the frames k that cover n = n' + pad of frame_k[n - k hop],
// in ascending k (the overlap-add of the transposed convolution, as a gather: no atomics).
// blockIdx.y is the batch item; positions and frame offsets are 32-bit (checked at plan
// creation), the batch item's base 64-bit.
__global__ void istft_ola_kernel(const float *__restrict__ frames, const float *__restrict__ bias,
                                 float *__restrict__ y, OlaGeo g) {
    const float b0 = bias ? bias[0] : 0.0f;
    const float *fb = frames + (int64_t)blockIdx.y * g.T * g.N;
    float *yb = y + (int64_t)blockIdx.y * g.L_out;
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
    if (dtype != CTR_F32 && dtype != CTR_BF16) return CTR_ERR_INVALID_ARG;
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
    p->smem = (size_t)p->fpb * 2 * (M + 1) * sizeof(float2);
    p->off_tw = 0;
    p->off_win = align256((size_t)n_fft * sizeof(float2));
    p->off_frames = p->off_win + align256((size_t)n_fft * sizeof(float));
    p->ws_needed = p->off_frames + (size_t)(N * frames * n_fft) * sizeof(float);
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
        g.logM = 0;
        while ((1 << g.logM) < g.M) ++g.logM;
        g.fpb = p->fpb;
        const dim3 grid((unsigned)((p->frames + p->fpb - 1) / p->fpb), (unsigned)p->B);
        irfft_frames_kernel<<<grid, kFftBlock, p->smem, st>>>(
            static_cast<const float *>(spec), reinterpret_cast<const float2 *>(ws + p->off_tw),
            reinterpret_cast<const float *>(ws + p->off_win), frames, g);
        count_launches(1);
        if (cudaGetLastError() != cudaSuccess) return CTR_ERR_CUDA;
    }
    OlaGeo o;
    o.T = (int)p->frames;
    o.N = (int)p->n_fft;
    o.hop = (int)p->hop;
    o.pad = (int)p->pad;
    o.L_out = (int)p->L_out;
    const dim3 ogrid((unsigned)std::min<int64_t>((p->L_out + 255) / 256, (int64_t)1 << 20),
                     (unsigned)p->B);
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
