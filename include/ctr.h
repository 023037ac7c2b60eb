/*
 * ctr.h -- C ABI of the GB300 (sm_103a) transposed-convolution library.
 *
 * The operation is dense (groups = 1) 1-D or 2-D ConvTranspose, in the scatter form
 *
 *     y[b, oc, i*s - p + t] += x[b, ic, i] * w[ic, oc, t]      (per spatial dimension)
 *     y[b, oc, o]           += bias[oc]
 *
 * with L_out = (L_in - 1)*s - 2p + k + op per spatial dimension and the weight in the
 * un-flipped torch layout [C_in][C_out][k...].  Sources:
 *   - "[ExecuTorch][WebGPU] Add optimized conv2d op" (PR #20849), Implementation and
 *     Constraints: the gather condition, the un-flipped [IC, OC, KH, KW] weight, the optional
 *     bias, output_padding < stride;
 *   - "[XNNPACK] Lower dense transposed convs as one polyphase conv + depth to space"
 *     (PR #25037), Summary: the polyphase lowering for k = m*s (one stride-1 conv with m
 *     taps, phase-major, then the phase interleave and the padding slice), which is the
 *     library's main path;
 *   - "[WebGPU] optimizations for audio models" (PR #33978), ConvTranspose commits: the
 *     X[M, C_in] x W[C_in, k*C_out] GEMM plus col2im path, the prepacked constant weight,
 *     f32 intermediates, the bias added once, the empty-input case.
 *
 * Call sequence:
 *     ctr_plan_create -> (ctr_plan_set_*) -> ctr_packed_weight_bytes / ctr_workspace_bytes
 *     -> ctr_prepack_weight (once per weight) -> ctr_plan_bind_workspace
 *     -> ctr_forward (any number of times) -> ctr_plan_check -> ctr_plan_destroy
 *
 * Conventions for every call:
 *   - Every call returns a ctr_status (or a size / string); nothing throws or aborts.
 *   - Device pointers are plain CUDA device addresses in the current device's context.
 *     Streams are cudaStream_t values passed as void* (NULL = the legacy default stream).
 *   - The caller owns every device buffer: x, w, w_packed, bias, y and the workspace.  The
 *     library never frees, keeps or aliases them beyond the call (and, for the workspace,
 *     the binding).  The plan owns its host metadata and a 4-byte device status word.
 *   - ctr_forward and ctr_prepack_weight are asynchronous on the given stream and never
 *     allocate, free or synchronise.
 *   - Tensors are contiguous, row-major, in the plan's I/O dtype:
 *         x    [N][C_in][L_in]            or [N][C_in][H][W]
 *         w    [C_in][C_out/G][k]         or [C_in][C_out/G][kH][kW]   (G groups, default 1)
 *         bias [C_out]                    (may be NULL)
 *         y    [N][C_out][L_out]          or [N][C_out][H_out][W_out]
 *     (x and y channels last with ctr_plan_set_layout(plan, CTR_LAYOUT_NHWC))
 *     and each must start on a 16-byte boundary (CTR_ERR_MISALIGNED otherwise).
 *   - A plan is not thread-safe: calls on one plan must not overlap on the host.  Two
 *     ctr_forward calls on one plan that run concurrently on the GPU (different streams)
 *     share its workspace and race; serialise them or use one plan per stream.
 */
#ifndef CTR_H
#define CTR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ctr_plan_s *ctr_plan_t;

typedef enum {
    CTR_OK = 0,
    CTR_ERR_INVALID_ARG = 1,     /* a size, geometry or handle is invalid */
    CTR_ERR_UNSUPPORTED = 2,     /* valid ConvTranspose this library does not implement */
    CTR_ERR_MISALIGNED = 3,      /* a pointer is not 16-byte aligned */
    CTR_ERR_NO_WORKSPACE = 4,    /* workspace needed but unbound or too small */
    CTR_ERR_CUDA = 5,            /* a CUDA runtime or launch error */
    CTR_ERR_DEVICE_TIMEOUT = 6,  /* a bounded device-side wait gave up (see ctr_plan_check) */
    CTR_ERR_NOT_PREPARED = 7     /* ctr_forward before ctr_prepack_weight on this plan */
} ctr_status;

typedef enum {
    CTR_F32 = 0,   /* fp32 I/O; each operand split as hi = tf32(v), lo = v - hi: hi*hi as a tf32
                      tensor-core product, hi*lo + lo*hi as bf16 products, fp32 accumulate
                      (rel_l2 within 1e-5 of fp32 arithmetic) */
    CTR_BF16 = 1,  /* bf16 I/O; bf16 tensor-core products, fp32 accumulate, one final rounding */
    CTR_F16 = 2    /* fp16 I/O; fp16 tensor-core products, fp32 accumulate and intermediates,
                      one final rounding ("[WebGPU] optimizations for audio models", review
                      commits: for float16 the packed weight and the K-padded input stay in the
                      I/O type while sums and column buffers are f32).  Not on the depthwise
                      kernel (grouped fp16 plans run the gather kernel) nor the iSTFT plan. */
} ctr_dtype;

typedef enum {
    CTR_ACT_NONE = 0,
    CTR_ACT_LEAKY_RELU = 1       /* y = y >= 0 ? y : slope * y, after the bias, before rounding */
} ctr_act;

typedef enum {
    CTR_PATH_AUTO = 0,
    CTR_PATH_POLYPHASE = 1,      /* polyphase implicit GEMM on tcgen05 (taps zero-padded to m*s) */
    CTR_PATH_COL2IM = 2,         /* tcgen05 GEMM into an fp32 column buffer, then col2im */
    CTR_PATH_GATHER = 3,         /* direct gather on CUDA cores (any groups) */
    CTR_PATH_DEPTHWISE = 4       /* one input channel per group (groups = C_in), CUDA cores */
} ctr_path;

/*
 * Create a plan.  Host only: validates the geometry, picks the path and the tiling.  The
 * only CUDA call reads the current device's SM count; without a GPU it assumes 152 SMs, so
 * plans can be created and inspected on a machine without one.
 *   out            receives the plan (set to NULL on failure)
 *   ndim           1 or 2 spatial dimensions
 *   N, C_in, C_out batch and channels: N >= 0, C_in >= 1, C_out >= 1
 *   in_spatial     ndim input sizes, each >= 0 (0 = empty input: y = bias or zeros)
 *   kernel         ndim kernel sizes >= 1
 *   stride         ndim strides >= 1
 *   padding        ndim paddings >= 0 (front and back; ctr_plan_set_pads separates them)
 *   output_padding ndim values with 0 <= op < stride (may be NULL = zeros)
 *   dtype          ctr_dtype (CTR_F32, CTR_BF16 or CTR_F16)
 * Every output size must be >= 1.  Groups, dilation and separate front/back pads are set
 * afterwards (ctr_plan_set_groups, ctr_plan_set_dilation, ctr_plan_set_pads; defaults: one
 * group, dilation 1, the back pad equal to `padding`).  Returns CTR_ERR_INVALID_ARG on any
 * violation.  A layer whose pads are only valid once separated or dilated (a front pad that,
 * taken on both sides, would leave no output) is created with zero padding and given its
 * pads by ctr_plan_set_pads, after ctr_plan_set_dilation.
 */
ctr_status ctr_plan_create(ctr_plan_t *out, int ndim, int64_t N, int64_t C_in, int64_t C_out,
                           const int64_t *in_spatial, const int64_t *kernel,
                           const int64_t *stride, const int64_t *padding,
                           const int64_t *output_padding, int dtype);

/*
 * Grouped transposed convolution (default 1 group): groups must divide C_in and C_out; the
 * weight is then [C_in][C_out/groups][k...] and output channel oc sums only the input
 * channels of its group ("[ExecuTorch][WebGPU] Add optimized conv2d op", Implementation:
 * the [IC, OC/groups, KH, KW] weight).  groups = C_in (C_out = M * C_in; M = 1 is the
 * depthwise upsampler of "[XNNPACK] Lower dense transposed convs as one polyphase conv +
 * depth to space", DecomposeDepthwiseConvTransposePass commit) runs on the depthwise path
 * (CTR_PATH_DEPTHWISE) for 1-D kernels with k/s in {2/2, 3/2, 4/2, 4/4, 8/4, 8/8, 16/8} and
 * square 2-D kernels 2x2/2, 3x3/2, 4x4/2, 4x4/4; other grouped plans run on the gather path.
 * The tensor-core paths need one group: forcing one on a grouped plan, or grouping a plan
 * forced onto one, returns CTR_ERR_UNSUPPORTED and leaves the plan unchanged.  Host only,
 * same ordering rule as ctr_plan_set_path; CTR_ERR_INVALID_ARG when groups does not divide
 * both channel counts, after ctr_prepack_weight, or on a chained plan.
 */
ctr_status ctr_plan_set_groups(ctr_plan_t plan, int64_t groups);

/*
 * Dilation (default 1 per dimension): taps are dil samples apart, so tap t of input i lands
 * at o = i*s - p_front + t*dil and L_out = (L_in - 1)*s + (k - 1)*dil + 1 + op - p_front -
 * p_back ("[ExecuTorch][WebGPU] Add optimized conv2d op", Implementation: the gather
 * condition (oh + pH - kh*dH) divisible by the stride; "[WebGPU] optimizations for audio
 * models": the ConvTranspose tests with pads, dilations or output_padding).
 *   dilation  ndim values >= 1
 * A dilated plan runs the col2im GEMM over its k real taps (C_in >= 16 and k*C_out >= 64)
 * or the gather kernel; a forced polyphase path packs the zero-inserted kernel of
 * (k - 1)*dil + 1 taps.  The depthwise path is undilated: forcing it on a dilated plan, or
 * dilating a plan forced onto it, returns CTR_ERR_UNSUPPORTED and leaves the plan unchanged.
 * Host only, with the same ordering rule as ctr_plan_set_path; CTR_ERR_INVALID_ARG for a
 * value < 1, an output size < 1, after ctr_prepack_weight, or on a chained plan (the plan is
 * then unchanged).
 */
ctr_status ctr_plan_set_dilation(ctr_plan_t plan, const int64_t *dilation);

/*
 * Separate front and back pads per dimension (the ONNX ConvTranspose `pads` attribute:
 * begin values, then end values), replacing the symmetric `padding` of ctr_plan_create.
 * The output is the unpadded result with p_front positions cut at the front and p_back at
 * the back (output_padding positions are added at the back first): L_out = (L_in - 1)*s +
 * (k - 1)*dil + 1 + op - p_front - p_back.  ("[XNNPACK] Lower dense transposed convs as one
 * polyphase conv + depth to space", Summary: the padding slice; "[WebGPU] optimizations for
 * audio models": the ConvTranspose tests with pads.)
 *   pads_begin, pads_end  ndim values >= 0 each
 * Every path takes any pads.  Host only, with the same ordering rule as ctr_plan_set_path;
 * CTR_ERR_INVALID_ARG for a negative pad, an output size < 1, after ctr_prepack_weight, or on
 * a chained plan (the plan is then unchanged).
 */
ctr_status ctr_plan_set_pads(ctr_plan_t plan, const int64_t *pads_begin, const int64_t *pads_end);

typedef enum {
    CTR_LAYOUT_NCHW = 0,   /* x [N][C_in][spatial...], y [N][C_out][out spatial...] (default) */
    CTR_LAYOUT_NHWC = 1    /* channels last: x [N][spatial...][C_in], y [N][out spatial...][C_out] */
} ctr_layout;

/*
 * Memory layout of x and y (default CTR_LAYOUT_NCHW); the weight keeps its torch layout.
 * Channels-last tensors are what image and audio pipelines often hold ("[XNNPACK] Lower dense
 * transposed convs as one polyphase conv + depth to space": the inpainting network's profile
 * spends a quarter of its time in NCHW <-> NHWC transposes around the deconvolutions).  The
 * tensor-core paths stage an NHWC input with a row copy (their staged operand is channels-last
 * already) and write an NHWC output from the same output stage that feeds a chained plan; the
 * gather kernel indexes NHWC directly.  The depthwise kernel is NCHW only (a grouped NHWC plan
 * runs the gather kernel) and so are streaming plans.  Host only, with the same ordering rule
 * as ctr_plan_set_path; CTR_ERR_INVALID_ARG for another value or after ctr_prepack_weight;
 * CTR_ERR_UNSUPPORTED on a streaming plan or one forced onto the depthwise path (the plan is
 * then unchanged).
 */
ctr_status ctr_plan_set_layout(ctr_plan_t plan, int layout);

typedef enum {
    CTR_AUTO_PAD_NOTSET = 0,      /* explicit pads (ctr_plan_create / ctr_plan_set_pads) */
    CTR_AUTO_PAD_SAME_UPPER = 1,  /* output = input * stride, odd total padding: extra at the end */
    CTR_AUTO_PAD_SAME_LOWER = 2,  /* output = input * stride, odd total padding: extra in front */
    CTR_AUTO_PAD_VALID = 3        /* no padding */
} ctr_auto_pad;

/*
 * The ONNX ConvTranspose `auto_pad` and `output_shape` attributes ("[WebGPU] optimizations
 * for audio models": the ConvTranspose tests run the ONNX operator's attributes), resolved
 * into the front and back pads of ctr_plan_set_pads.  Per dimension, with the plan's stride
 * s, kernel k, dilation d and output_padding op, the unpadded output has
 * full = (L_in - 1)*s + (k - 1)*d + 1 + op samples, and
 *   - output_shape given (any auto_pad): total = full - output_shape;
 *   - else SAME_UPPER / SAME_LOWER: total = full - L_in*s;
 *   - else VALID: no padding (total = 0);  NOTSET: the plan keeps its pads.
 * SAME_UPPER puts total/2 (rounded down) in front and the rest at the end; every other
 * setting puts the rest in front and total/2 at the end.  So the output is the unpadded
 * result's samples front .. full - back - 1, of length output_shape (or L_in*s).
 *   auto_pad      a ctr_auto_pad value
 *   output_shape  ndim output sizes, or NULL
 * A negative total (an output longer than the unpadded result) would need negative pads:
 * CTR_ERR_UNSUPPORTED.  Set dilation first (ctr_plan_set_dilation): the pads depend on it.
 * Host only, with the same ordering rule as ctr_plan_set_path; CTR_ERR_INVALID_ARG for an
 * unknown auto_pad, an output size < 1, after ctr_prepack_weight, or on a chained or
 * streaming plan (the plan is then unchanged).
 */
ctr_status ctr_plan_set_auto_pad(ctr_plan_t plan, int auto_pad, const int64_t *output_shape);

/*
 * Streaming 1-D ConvTranspose (default off): the input arrives as consecutive chunks of
 * L_in frames (a streaming audio decoder's upsampler), and each ctr_forward emits the
 * s*L_in output samples that its frames complete.  Concatenated, the outputs of a stream are
 * the unpadded ConvTranspose of the concatenated input, (L - 1)*s + k samples, without its
 * last k - s ("[XNNPACK] Lower dense transposed convs as one polyphase conv + depth to
 * space", Test plan and the Phonon fix: the overlap-add of a streaming decoder).  Those last
 * samples come out with the following chunk; zero frames flush them at the end of a stream.
 *
 * The polyphase form makes the state an input state. Output phase position q reads frames
 * q - (m - 1) .. q (m = ceil(k/s)). So the plan carries each batch item's last m - 1
 * input frames in its workspace and puts them in front of the next chunk. The
 * not-yet-complete output samples are not held back. Any chunk length works, including
 * chunks shorter than m - 1 frames.
 *
 * Requires: 1-D, padding = output_padding = 0, k >= s, one group, no dilation,
 * m - 1 <= 16, and the polyphase path.  The path is forced; a plan that cannot take it returns
 * CTR_ERR_UNSUPPORTED and stays unchanged.  Afterwards ctr_plan_output_shape reports
 * s*L_in. ctr_workspace_bytes includes the carried frames, B*(m - 1) staged rows.
 * ctr_plan_stream_reset must zero them before the first ctr_forward, after every
 * ctr_plan_bind_workspace, and to start a new stream (CTR_ERR_NOT_PREPARED otherwise).
 * Calls of one stream must run in stream order, one at a time: each reads the frames the
 * previous one carried.  ctr_forward_noalloc refuses streaming plans
 * (CTR_ERR_UNSUPPORTED).
 *
 * Host only, with the same ordering rule as ctr_plan_set_path.  CTR_ERR_INVALID_ARG for
 * enable not 0 or 1, after ctr_prepack_weight, or on a chained plan.  Once streaming, a
 * plan refuses ctr_plan_set_groups, _set_dilation, _set_pads and ctr_plan_chain
 * (CTR_ERR_INVALID_ARG), and ctr_plan_set_path with any path but the polyphase one
 * (CTR_ERR_UNSUPPORTED).  enable = 0 restores the plain plan, with the path it had before
 * streaming was turned on (the automatic path, or the one ctr_plan_set_path forced).
 */
ctr_status ctr_plan_set_streaming(ctr_plan_t plan, int enable);

/* Zero a streaming plan's carried input frames (asynchronous on `stream`): the next
 * ctr_forward starts a new stream.  CTR_ERR_INVALID_ARG when the plan is not streaming,
 * CTR_ERR_NO_WORKSPACE when its workspace is unbound or too small. */
ctr_status ctr_plan_stream_reset(ctr_plan_t plan, void *stream);

/* Fuse an activation into the output stage (default CTR_ACT_NONE).  Host only. */
ctr_status ctr_plan_set_activation(ctr_plan_t plan, int act, float negative_slope);

/*
 * Force a path (default CTR_PATH_AUTO) and optionally the split-K factor of the tensor-core
 * paths (0 = automatic, else 1..16).  Host only.  Must come before ctr_packed_weight_bytes,
 * ctr_workspace_bytes and ctr_prepack_weight, because the packed layout and the workspace
 * depend on the path; calling it after ctr_prepack_weight returns CTR_ERR_INVALID_ARG.
 * The tensor-core paths index tiles, staged input positions and packed weight rows in 32
 * bits: a plan that exceeds 2^31 of any of them runs the gather path when chosen
 * automatically, and forcing a tensor-core path on it returns CTR_ERR_UNSUPPORTED.
 * CTR_PATH_DEPTHWISE needs groups = C_in and a compiled geometry (ctr_plan_set_groups),
 * and the tensor-core paths one group; a path the plan cannot take returns
 * CTR_ERR_UNSUPPORTED and leaves the plan unchanged.
 */
ctr_status ctr_plan_set_path(ctr_plan_t plan, int path, int split_k);

typedef enum {
    CTR_PHASE_AUTO = 0,      /* the library chooses (below) */
    CTR_PHASE_UNPADDED = 1,  /* phases of the unpadded output, the padding sliced at the store */
    CTR_PHASE_OUTPUT = 2     /* phases of the output itself, the padding folded into the taps */
} ctr_phase_origin;

/*
 * Where the polyphase path's phase positions start.  "[XNNPACK] Lower dense transposed convs
 * as one polyphase conv + depth to space" (Summary) computes the phases of the unpadded
 * output and slices the padding off afterwards (CTR_PHASE_UNPADDED): output o = s*q + j - p,
 * so with p mod s != 0 every run of s phases starts at an odd offset and the output stage
 * writes elements one by one.  CTR_PHASE_OUTPUT re-indexes the phases by the output itself,
 * o = s*Q + J: with p = s*pq + pm, phase J takes the taps s*(m-1-v) + J + pm of the kernel
 * (zero where that is outside it), which needs one more tap per phase when pm > 0, and reads
 * input Q + pq - (m-1) + v.  Both compute the same sums of the same products; only zero
 * products are added or removed.  CTR_PHASE_AUTO takes the output phases when p mod s = 0
 * (no extra tap) and otherwise when the layer is bound by its output stores rather than by
 * its products (estimated from the tile model), for a plan whose output is not chained.
 * Streaming plans keep the unpadded phases.  A tuning and test override: host only, with the
 * same ordering rule as ctr_plan_set_path; CTR_ERR_INVALID_ARG for another value or after
 * ctr_prepack_weight.  Ignored by the paths other than polyphase.
 */
ctr_status ctr_plan_set_phase_origin(ctr_plan_t plan, int origin);

/*
 * Force the phase-row tile of the tensor-core paths: the number of packed weight rows one
 * output tile covers, i.e. the MMA N extent (0 = automatic, else 64, 128 or 256).  A tuning
 * and test override with no counterpart on the pages; every value gives the same result
 * bit for bit.  Host only, with the same ordering rule as ctr_plan_set_path; returns
 * CTR_ERR_INVALID_ARG for another value or after ctr_prepack_weight.
 */
ctr_status ctr_plan_set_tile(ctr_plan_t plan, int block_n);

/*
 * Chain two plans so that `plan`'s output feeds `next`'s input without a staging pass, as
 * in a decoder's stack of upsampling layers (two ConvTransposes with an activation between:
 * "[XNNPACK] Lower dense transposed convs as one polyphase conv + depth to space", Test
 * plan).  Afterwards:
 *   - ctr_forward(plan, x, w, bias, y = NULL, stream) writes its output, with bias and
 *     activation applied and rounded to the I/O type, straight into the channels-last
 *     staged-input layout inside next's workspace (fp32: as its tf32 and bf16-pair planes, exactly
 *     what next's staging would have made of the torch-layout output), and no y;
 *   - ctr_forward(next, x = NULL, ...) reads it from there instead of staging an x.
 * Results are bit-identical to the unchained calls.  Requirements (CTR_ERR_INVALID_ARG
 * otherwise): both plans on a tensor-core path (polyphase or col2im), the same dtype and
 * batch, next's C_in equal to plan's C_out and next's input spatial size equal to plan's
 * output size.  At each forward, next's workspace must be bound (CTR_ERR_NO_WORKSPACE)
 * and must not overlap plan's (CTR_ERR_INVALID_ARG); the first forward after binding
 * zeroes next's staged buffer once (its halos stay zero).  Run plan, then next, on the
 * same stream.  A chained plan packs its weight rows for this output (phase-major within
 * each tile), so ctr_plan_chain(plan, ...) must come before ctr_prepack_weight(plan)
 * (CTR_ERR_INVALID_ARG after it), and a plan packed for a chain whose other end was
 * destroyed refuses to run.  ctr_plan_chain(plan, NULL) unchains; destroying either plan
 * unchains both.  Host only; no counterpart of the call itself on the pages.
 */
ctr_status ctr_plan_chain(ctr_plan_t plan, ctr_plan_t next);

/*
 * Run a chained pair of layers -- plan and the plan it is chained to (ctr_plan_chain) -- as
 * one kernel that keeps the first layer's output in shared memory as the second layer's
 * operand, instead of writing it to the second plan's staged input and reading it back
 * (the two-layer stack of "[XNNPACK] Lower dense transposed convs as one polyphase conv +
 * depth to space", Test plan).  The result is bit-identical to ctr_forward(plan, x, ...)
 * followed by ctr_forward(next, NULL, ...).
 *   x            plan's input as for ctr_forward (NULL when a chained previous plan staged it)
 *   w_packed, bias        plan's packed weight and bias
 *   next_w_packed, next_bias   the next plan's
 *   y            the next plan's output
 * Needs (CTR_ERR_UNSUPPORTED otherwise, see ctr_plan_fusable): 1-D, bf16 or fp16, both on
 * the polyphase path without split-K; plan with stride >= 2 and exactly 64 output channels
 * in one tile of 128 phase rows; next with 64 input channels, one row tile of 64 or 128
 * rows, an NCHW output and no further chain.  Both plans prepacked (CTR_ERR_NOT_PREPARED)
 * and plan's workspace bound (CTR_ERR_NO_WORKSPACE); the next plan's workspace is not used.
 * Asynchronous on stream; device-side timeouts are reported by ctr_plan_check(plan, ...).
 * No counterpart of the call itself on the pages.
 */
ctr_status ctr_forward_fused(ctr_plan_t plan, const void *x, const void *w_packed,
                             const void *bias, const void *next_w_packed,
                             const void *next_bias, void *y, void *stream);

/* 1 when ctr_forward_fused can run plan and the plan it is chained to, else 0. */
int ctr_plan_fusable(ctr_plan_t plan);

/* The path the plan will run (a ctr_path other than AUTO), or -1 for a NULL plan. */
int ctr_plan_get_path(ctr_plan_t plan);

/* Write the ndim output sizes into out_spatial. */
ctr_status ctr_plan_output_shape(ctr_plan_t plan, int64_t *out_spatial);

/* Bytes of the packed weight buffer ctr_prepack_weight writes (0 for a NULL plan). */
size_t ctr_packed_weight_bytes(ctr_plan_t plan);

/* Bytes of device workspace ctr_forward needs (may be 0; 0 for a NULL plan). */
size_t ctr_workspace_bytes(ctr_plan_t plan);

/*
 * Bind a caller-owned device workspace of at least ctr_workspace_bytes(plan) bytes,
 * 256-byte aligned.  The binding lasts until the next bind or ctr_plan_destroy; the
 * workspace must stay allocated meanwhile.  Binding NULL with 0 bytes is allowed when the
 * plan needs no workspace.
 */
ctr_status ctr_plan_bind_workspace(ctr_plan_t plan, void *dev_ptr, size_t bytes);

/*
 * Pack a weight for this plan (once per weight; asynchronous on stream).
 *   w         device, [C_in][C_out/groups][k...] in the plan's dtype
 *   w_packed  device, ctr_packed_weight_bytes(plan) bytes, written in full
 * The packed weight is valid only for plans with the same geometry, dtype and path.  The
 * first call on a plan also allocates the plan's 4-byte device status word on the current
 * device (the only allocation the library makes).
 */
ctr_status ctr_prepack_weight(ctr_plan_t plan, const void *w, void *w_packed, void *stream);

/*
 * y = ConvTranspose(x, w) + bias, then the plan's activation, rounded once to the I/O dtype.
 *   x         device input, [N][C_in][spatial...]
 *   w_packed  device, written by ctr_prepack_weight for this plan's geometry
 *   bias      device [C_out] or NULL
 *   y         device output, [N][C_out][out spatial...], written in full
 *   stream    cudaStream_t as void*
 * Asynchronous; launch failures return CTR_ERR_CUDA.  Device-side errors (a bounded wait
 * that gave up) are reported by ctr_plan_check.  x and y must not overlap.  For a chained
 * plan (ctr_plan_chain) y must be NULL; for the plan it feeds, x may be NULL.
 */
ctr_status ctr_forward(ctr_plan_t plan, const void *x, const void *w_packed, const void *bias,
                       void *y, void *stream);

/*
 * ctr_forward for callers that cannot allocate device memory (a host framework whose
 * allocator owns all device memory, code running while a CUDA graph is captured, real-time
 * audio callbacks).  The source pages have no counterpart of this call.
 *   plan      a plan from ctr_plan_create; no ctr_prepack_weight, workspace binding or other
 *             device allocation is needed for it
 *   x, bias   device inputs as for ctr_forward (bias may be NULL)
 *   w         device weight in its torch layout [C_in][C_out][k...] (not packed: every call
 *             packs it into the library's scratch)
 *   y         device output as for ctr_forward
 *   stream    cudaStream_t as void*
 * Scratch (packed weight, staged input, split-K partials, a status word) lives in one
 * static 32 MiB device array that the CUDA driver reserves on each device that loads the
 * library and keeps until the process exits.  Plans needing more than that (the packed
 * weight plus ctr_workspace_bytes plus 256 bytes) get CTR_ERR_NO_WORKSPACE before anything
 * runs.  This call performs no cudaMalloc, cudaFree or other allocation.  Its first call on
 * a device looks up the array's device address (cudaGetSymbolAddress) with that device
 * current; make that first call before any stream capture.  Every call shares the one
 * array: calls whose GPU work overlaps (different streams, or several host threads) race on
 * it and must be serialised by the caller.  Bounded-wait timeouts are recorded in the
 * array's status word, which every call clears at its start (this call does not
 * synchronise); ctr_plan_check of any plan, on the same device, reads and clears it, so a
 * check right after a call reports that call's timeout.  Returns as ctr_forward otherwise.
 */
ctr_status ctr_forward_noalloc(ctr_plan_t plan, const void *x, const void *w, const void *bias,
                               void *y, void *stream);

/*
 * Synchronise stream, then read and clear the plan's device status word, and the status word
 * of ctr_forward_noalloc's scratch on the current device once an allocation-free call has
 * run there.  Returns CTR_OK, CTR_ERR_DEVICE_TIMEOUT when a kernel's bounded wait gave up
 * since the last check (its output is then incomplete), or CTR_ERR_CUDA.
 */
ctr_status ctr_plan_check(ctr_plan_t plan, void *stream);

/*
 * Limit, in nanoseconds, of every bounded device-side wait of the tensor-core kernels
 * (default 4e9).  A test hook: a tiny limit makes the waits give up on a healthy run, so
 * the timeout path can be exercised without a fault.  Host only.
 */
ctr_status ctr_plan_set_wait_limit_ns(ctr_plan_t plan, uint64_t limit_ns);

/*
 * Measurement hook: when both are non-NULL, every later ctr_forward records the
 * caller-owned CUDA events `before` and `after` (cudaEvent_t as void*) on its stream
 * immediately before and after the plan's main kernel (the tensor-core GEMM on the polyphase
 * and col2im paths, the gather kernel otherwise), so cudaEventElapsedTime gives that
 * kernel's own duration.  Pass NULL, NULL to stop.  Host only; the events must outlive
 * the calls that record them.  A ctr_forward captured into a CUDA graph records them as
 * external event nodes, so they time every replay.
 */
ctr_status ctr_plan_set_timing_events(ctr_plan_t plan, void *before, void *after);

/* Human-readable summary of the plan's path and tiling into buf (NUL-terminated). */
ctr_status ctr_plan_describe(ctr_plan_t plan, char *buf, size_t len);

/* Free the plan's host metadata and status word.  NULL is ignored.  Does not synchronise:
 * call it only after the plan's work on the GPU has finished. */
void ctr_plan_destroy(ctr_plan_t plan);

/* Static description of a status code. */
const char *ctr_status_string(ctr_status status);

/* Number of GPU kernels this library has launched in this process (a monotonic counter
 * for benchmarks and tests). */
uint64_t ctr_launch_count(void);

/* ------------------------------------------------------------------------------------
 * Inverse STFT through an inverse real FFT.
 *
 * The same result as ctr_forward on a 1-D plan with C_in = n_fft + 2, C_out = 1, kernel
 * n_fft, stride hop and the windowed inverse real-DFT basis as weight: channel f of the
 * input holds the real part of bin f (0 <= f <= n_fft/2), channel n_fft/2 + 1 + f its
 * imaginary part, and the weight rows are c_f win[t] cos(2 pi f t/N) / N and
 * -c_f win[t] sin(2 pi f t/N) / N (c_0 = c_{N/2} = 1, else 2).  "[WebGPU] optimizations for
 * audio models" computes the source-separation model's inverse STFT as that ConvTranspose1d;
 * here each frame is an inverse real FFT (O(n_fft log n_fft) instead of O(n_fft^2)), times
 * the window, and the frames are overlap-added at stride hop, sliced by the padding, plus
 * an optional scalar bias.
 *
 *   spec  device, [N][n_fft + 2][frames], fp32 (16-byte aligned)
 *   y     device, [N][1][L_out], fp32, L_out = (frames - 1)*hop - 2*padding + n_fft
 *         + output_padding (16-byte aligned)
 *   window  device, [n_fft] fp32 synthesis window (16-byte aligned)
 *   bias  device, [1] fp32 or NULL
 *
 * n_fft is a power of two in [4, 8192]; hop >= 1; 0 <= output_padding < hop; padding >= 0.
 * fp32 only: CTR_BF16 returns CTR_ERR_UNSUPPORTED.  The plan owns no device memory: the
 * caller binds a workspace of ctr_istft_workspace_bytes (twiddles, the scaled window, the
 * windowed frames, fp32 [N][frames][n_fft], and the spectra as frame-major complex rows,
 * [N][frames][n_fft/2 + 2] pairs) and sets the window once (a kernel on `stream`);
 * ctr_istft_forward then launches three kernels (the spectra to frame-major rows, the
 * per-frame FFT, then the overlap-add as a gather, summing frames in ascending order:
 * deterministic) and never allocates or synchronises.  Errors as for the ConvTranspose plan; CTR_ERR_NOT_PREPARED before
 * ctr_istft_set_window (rebinding the workspace clears it).
 * ------------------------------------------------------------------------------------ */
typedef struct ctr_istft_s *ctr_istft_t;

ctr_status ctr_istft_create(ctr_istft_t *out, int64_t N, int64_t n_fft, int64_t hop,
                            int64_t frames, int64_t padding, int64_t output_padding, int dtype);
ctr_status ctr_istft_output_length(ctr_istft_t plan, int64_t *L_out);
size_t ctr_istft_workspace_bytes(ctr_istft_t plan);
ctr_status ctr_istft_bind_workspace(ctr_istft_t plan, void *workspace, size_t bytes);
ctr_status ctr_istft_set_window(ctr_istft_t plan, const void *window, void *stream);
ctr_status ctr_istft_forward(ctr_istft_t plan, const void *spec, const void *bias, void *y,
                             void *stream);
ctr_status ctr_istft_describe(ctr_istft_t plan, char *buf, size_t len);
/* As ctr_plan_set_timing_events, around the kernels of ctr_istft_forward. */
ctr_status ctr_istft_set_timing_events(ctr_istft_t plan, void *before, void *after);
void ctr_istft_destroy(ctr_istft_t plan);

#ifdef __cplusplus
}
#endif

#endif /* CTR_H */
