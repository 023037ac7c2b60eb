/*
 * ctr_oracle.c -- plain CPU oracle for transposed convolution: dense (groups = 1) and
 * grouped, including depthwise (groups = C_in = C_out), with dilation and separate front
 * and back pads.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark load this file's library.  The product library never links, loads or
 * calls it, and it shares no code, header or table with the CUDA path.
 *
 * What it computes: the scatter form of ConvTranspose, in double precision.
 *
 *   for every batch b, input channel ic, input position i, output channel oc of ic's
 *   group, tap t
 *       o = i*s - pb + t*d                               (per spatial dimension)
 *       if 0 <= o < L_out:  acc[b, oc, o] += x[b, ic, i] * w[ic, oc - g*C_out/G, t]
 *   y[b, oc, o] = bias[oc] + acc[b, oc, o]               (bias = 0 when absent)
 *
 * with L_out = (L_in - 1)*s + (k - 1)*d + 1 + op - pb - pe per dimension (front pad pb,
 * back pad pe, dilation d; the symmetric undilated case is (L_in - 1)*s - 2p + k + op),
 * G groups (input channel ic and output channel oc belong to group g when
 * ic / (C_in/G) = oc / (C_out/G) = g) and the weight in the un-flipped torch layout
 * w[C_in][C_out/G][k...].  Sources:
 *   - "[ExecuTorch][WebGPU] Add optimized conv2d op" (PR #20849), Implementation: the
 *     transposed kernel reads the weight un-flipped as [IC, OC/groups, KH, KW] (the grouped
 *     layout) and a tap kh reaches an output row oh when (oh + pH - kh*dH) is divisible by
 *     the stride and the quotient is in range -- the gather reading of the same scatter sum,
 *     dilation included;
 *   - "[XNNPACK] Lower dense transposed convs as one polyphase conv + depth to space"
 *     (PR #25037), Summary: the clean-upscale output size (H-1)s - 2p + k + op, and the
 *     padding slice: the output is the full (unpadded) result with pb positions cut at the
 *     front and pe at the back, output_padding positions added at the back;
 *   - "[WebGPU] optimizations for audio models" (PR #33978), ConvTranspose commits: the
 *     output starts from the bias (or zeros) and every tap contribution is summed onto it;
 *     an empty spatial input leaves the bias (or zeros) in a non-empty output; the
 *     ConvTranspose tests with pads, dilations or output_padding (the ONNX attributes, whose
 *     pads list a front and a back pad per dimension).
 *
 * 1-D is the 2-D code with a unit height (k = s = d = 1, no pads along y).
 *
 * Accumulation is in double; the caller rounds the result to the I/O precision.  OpenMP
 * splits the work into items (b, oc, chunk of input positions); every item owns a private
 * accumulator and the chunks are summed in a fixed order at the end, so the result does
 * not depend on the number of threads.  The chunk count depends on the problem only.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Output length of one spatial dimension with dilation d, front pad pb and back pad pe
 * (may be <= 0 for invalid geometry): the last tap of the last input lands at
 * (L_in - 1)*s + (k - 1)*d in the unpadded output, output_padding extends it at the back. */
int64_t ctr_oracle_output_size_ex(int64_t L_in, int64_t k, int64_t s, int64_t d, int64_t pb,
                                  int64_t pe, int64_t op)
{
    return (L_in - 1) * s + (k - 1) * d + 1 + op - pb - pe;
}

/* Output length without dilation, with the same pad p at both ends. */
int64_t ctr_oracle_output_size(int64_t L_in, int64_t k, int64_t s, int64_t p, int64_t op)
{
    return ctr_oracle_output_size_ex(L_in, k, s, 1, p, p, op);
}

/* Threads the oracle's parallel loops use (for reporting). */
int ctr_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Run the parallel loops on n threads (n >= 1), or on the OpenMP default when n <= 0.
 * Only the speed changes: every item sums into its own accumulator and the items are
 * combined in a fixed order, so the result is the same on any number of threads. */
void ctr_oracle_set_threads(int n)
{
#ifdef _OPENMP
    static int default_threads = 0;
    if (default_threads == 0) default_threads = omp_get_max_threads();
    omp_set_num_threads(n >= 1 ? n : default_threads);
#else
    (void)n;
#endif
}

/* Number of (input position, tap) pairs, over all spatial dimensions, that land inside
 * the output: the count of scalar contributions per (input channel, output channel)
 * pair.  Returns -1 on invalid geometry. */
int64_t ctr_oracle_landed_pairs(int ndim, const int64_t *in_sp, const int64_t *ker,
                                const int64_t *str, const int64_t *pad, const int64_t *opad)
{
    if (ndim < 1 || ndim > 2) return -1;
    int64_t total = 1;
    for (int d = 0; d < ndim; ++d) {
        int64_t L_out = ctr_oracle_output_size(in_sp[d], ker[d], str[d], pad[d], opad[d]);
        int64_t n = 0;
        for (int64_t i = 0; i < in_sp[d]; ++i)
            for (int64_t t = 0; t < ker[d]; ++t) {
                int64_t o = i * str[d] - pad[d] + t;
                if (o >= 0 && o < L_out) ++n;
            }
        total *= n;
    }
    return total;
}

/*
 * y = ConvTranspose(x, w) + bias with G groups, dilation and front/back pads, in double.
 *   x    [B][C_in][in_sp[0]]([in_sp[1]])            contiguous
 *   w    [C_in][C_out/G][ker[0]]([ker[1]])          contiguous, un-flipped torch layout
 *   bias [C_out] or NULL
 *   y    [B][C_out][L_out[0]]([L_out[1]])           contiguous, written in full
 *   dil, pad_b, pad_e, opad: per spatial dimension (dilation >= 1, pads >= 0, op >= 0)
 * Returns 0 on success, -1 on invalid arguments (G must divide C_in and C_out, every
 * output length must be positive), -2 when out of host memory.
 */
int ctr_oracle_conv_transpose_ex(int ndim, int64_t B, int64_t C_in, int64_t C_out, int64_t G,
                                 const int64_t *in_sp, const int64_t *ker, const int64_t *str,
                                 const int64_t *dil, const int64_t *pad_b, const int64_t *pad_e,
                                 const int64_t *opad, const double *x, const double *w,
                                 const double *bias, double *y)
{
    if (ndim < 1 || ndim > 2 || B < 0 || C_in < 1 || C_out < 1) return -1;
    if (G < 1 || C_in % G != 0 || C_out % G != 0) return -1;
    const int64_t cin_g = C_in / G, cout_g = C_out / G;

    /* Unit height for 1-D. */
    int64_t H = 1, kh = 1, sh = 1, dh = 1, ph = 0, peh = 0, oph = 0;
    int64_t W = in_sp[0], kw = ker[0], sw = str[0], dw = dil[0], pw = pad_b[0], pew = pad_e[0],
            opw = opad[0];
    if (ndim == 2) {
        H = in_sp[0]; kh = ker[0]; sh = str[0]; dh = dil[0]; ph = pad_b[0]; peh = pad_e[0];
        oph = opad[0];
        W = in_sp[1]; kw = ker[1]; sw = str[1]; dw = dil[1]; pw = pad_b[1]; pew = pad_e[1];
        opw = opad[1];
    }
    if (H < 0 || W < 0 || kh < 1 || kw < 1 || sh < 1 || sw < 1 || dh < 1 || dw < 1 ||
        ph < 0 || pw < 0 || peh < 0 || pew < 0 || oph < 0 || opw < 0)
        return -1;
    const int64_t Ho = ctr_oracle_output_size_ex(H, kh, sh, dh, ph, peh, oph);
    const int64_t Wo = ctr_oracle_output_size_ex(W, kw, sw, dw, pw, pew, opw);
    if (Ho <= 0 || Wo <= 0) return -1;

    const int64_t npos = H * W;          /* input positions per (b, ic) */
    const int64_t nout = Ho * Wo;        /* output positions per (b, oc) */
    const int64_t ntap = kh * kw;

    /* Chunks of input positions per (b, oc): enough items for the cores when B*C_out is
     * small.  A function of the problem only. */
    int64_t nchunk = 1;
    if (B * C_out < 32) nchunk = (32 + B * C_out - 1) / (B * C_out);
    if (nchunk > npos) nchunk = npos > 0 ? npos : 1;
    const int64_t nitem = B * C_out * nchunk;

    double *part = NULL;
    if (nitem > 0) {
        part = (double *)calloc((size_t)(nitem * nout), sizeof(double));
        if (!part) return -2;
    }

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t item = 0; item < nitem; ++item) {
        const int64_t chunk = item % nchunk;
        const int64_t oc = (item / nchunk) % C_out;
        const int64_t b = item / (nchunk * C_out);
        const int64_t pos_lo = npos * chunk / nchunk;
        const int64_t pos_hi = npos * (chunk + 1) / nchunk;
        const int64_t g = oc / cout_g, ocl = oc - g * cout_g;   /* group, channel in it */
        double *acc = part + item * nout;
        for (int64_t ic = g * cin_g; ic < (g + 1) * cin_g; ++ic) {
            const double *xp = x + (b * C_in + ic) * npos;
            const double *wp = w + (ic * cout_g + ocl) * ntap;
            for (int64_t pos = pos_lo; pos < pos_hi; ++pos) {
                const int64_t iy = pos / W, ix = pos % W;
                const double xv = xp[pos];
                for (int64_t ty = 0; ty < kh; ++ty) {
                    const int64_t oy = iy * sh - ph + ty * dh;
                    if (oy < 0 || oy >= Ho) continue;
                    /* Taps tx with 0 <= ix*sw - pw + tx*dw < Wo: the range check of the
                     * definition, written as loop bounds (ceilings of the two limits). */
                    const int64_t ox0 = ix * sw - pw;
                    const int64_t tx_lo = ox0 < 0 ? (-ox0 + dw - 1) / dw : 0;
                    int64_t tx_hi = ox0 < Wo ? (Wo - ox0 + dw - 1) / dw : 0;
                    if (tx_hi > kw) tx_hi = kw;
                    double *arow = acc + oy * Wo;
                    const double *wrow = wp + ty * kw;
                    for (int64_t tx = tx_lo; tx < tx_hi; ++tx)
                        arow[ox0 + tx * dw] += xv * wrow[tx];
                }
            }
        }
    }

    /* y = bias + sum of the chunk accumulators, chunks in increasing order. */
#pragma omp parallel for schedule(static)
    for (int64_t bo = 0; bo < B * C_out; ++bo) {
        const int64_t oc = bo % C_out;
        const double bv = bias ? bias[oc] : 0.0;
        double *yp = y + bo * nout;
        for (int64_t o = 0; o < nout; ++o) yp[o] = bv;
        for (int64_t c = 0; c < nchunk; ++c) {
            const double *acc = part + (bo * nchunk + c) * nout;
            for (int64_t o = 0; o < nout; ++o) yp[o] += acc[o];
        }
    }
    free(part);
    return 0;
}

/* Grouped transposed convolution without dilation, the same pad at both ends. */
int ctr_oracle_conv_transpose_groups(int ndim, int64_t B, int64_t C_in, int64_t C_out,
                                     int64_t G, const int64_t *in_sp, const int64_t *ker,
                                     const int64_t *str, const int64_t *pad,
                                     const int64_t *opad, const double *x, const double *w,
                                     const double *bias, double *y)
{
    const int64_t one[2] = {1, 1};
    return ctr_oracle_conv_transpose_ex(ndim, B, C_in, C_out, G, in_sp, ker, str, one, pad, pad,
                                        opad, x, w, bias, y);
}

/* Dense transposed convolution: the grouped one with one group. */
int ctr_oracle_conv_transpose(int ndim, int64_t B, int64_t C_in, int64_t C_out,
                              const int64_t *in_sp, const int64_t *ker, const int64_t *str,
                              const int64_t *pad, const int64_t *opad,
                              const double *x, const double *w, const double *bias, double *y)
{
    return ctr_oracle_conv_transpose_groups(ndim, B, C_in, C_out, 1, in_sp, ker, str, pad, opad,
                                            x, w, bias, y);
}
