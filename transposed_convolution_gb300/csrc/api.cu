// api.cu -- the library's C ABI: plan validation, path and tile choice, workspace layout,
// tensor-map encoding and the launch sequence of ctr_forward.
//
// Path choice follows the three lowerings on the source pages:
//   - polyphase ("[XNNPACK] Lower dense transposed convs as one polyphase conv + depth to
//     space", Summary): when every kernel size is a multiple of its stride and the phase
//     GEMM fills at least a 64-row MMA with K >= 16;
//   - GEMM + col2im ("[WebGPU] optimizations for audio models", ConvTranspose commit): for
//     group-1 convolutions with at least 16 input channels whose kernel is not a multiple
//     of the stride;
//   - the direct gather kernel ("[ExecuTorch][WebGPU] Add optimized conv2d op",
//     Implementation) for everything else, i.e. tiny channel counts.
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <cudaTypedefs.h>

#include "ctr_internal.h"
#include "epilogue.cuh"

using ctr::EpiParams;
using ctr::GemmParams;
using ctr::Prec;

namespace {

std::atomic<uint64_t> g_launches{0};

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }
size_t align256(size_t v) { return (v + 255) & ~size_t(255); }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t next_pow2(int64_t v) {
    int64_t r = 1;
    while (r < v) r <<= 1;
    return r;
}

int query_num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 152;
    }
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 152;
    }
    return n > 0 ? n : 152;
}

Prec prec_of(const ctr_plan_s *pl) {
    return pl->dtype == CTR_BF16 ? Prec::BF16 : pl->dtype == CTR_F16 ? Prec::F16 : Prec::F32;
}
bool io16(const ctr_plan_s *pl) { return pl->dtype != CTR_F32; }
int esize_io(const ctr_plan_s *pl) { return io16(pl) ? 2 : 4; }
// Elements of one 128-byte K slice in the GEMM operands.
int bk_elems(const ctr_plan_s *pl) { return io16(pl) ? 64 : 32; }
// Bytes per element of one GEMM operand plane, and number of planes (fp32: the tf32 plane
// and the plane of bf16 cross words).
int op_esize(const ctr_plan_s *pl) { return io16(pl) ? 2 : 4; }
int op_planes(const ctr_plan_s *pl) { return io16(pl) ? 1 : 2; }

bool is_tc_path(int path) { return path == CTR_PATH_POLYPHASE || path == CTR_PATH_COL2IM; }

// Estimated clocks of one K slice of a 128-position x BN-row tile on one SM (tensor pipe).
// fp32: a tf32 MMA and a bf16 MMA of twice the K per 32-byte K step, each at half the rate
// of a 16-bit MMA over the slice.
double slice_clocks(Prec prec, int bn) { return prec == Prec::F32 ? 4.0 * bn : 2.0 * bn; }

// 128-byte K slices per tensor-core accumulation group for fp32 I/O (512 fp32 K
// elements).  The tensor core's fp32 accumulation over a long K chain drifts well beyond
// fp32 summation with round-to-nearest (measured on GB300: rel_l2 2.3e-5 over 3300-element
// chains, a mean relative bias of -4.6e-5 over 4096 all-positive products), so the kernel
// moves the partial sum out of TMEM every group and adds it with round-to-nearest; the
// drift then scales with the group length only.  At 512 elements the all-positive worst
// case stays below the 1e-5 rel_l2 bound (a GPU test pins it) and random inputs give
// about 3e-6; 256 elements halve that but fold twice as often, which pauses the MMAs of
// 256-row tiles (codec upsampler step 46.2 vs 44.3 us).
constexpr int kTf32Group = 16;
constexpr int kNoGroup = 1 << 30;

int tf32_group() {
    // Diagnostic override of the group length (slices); 0 or negative disables grouping.
    const char *e = std::getenv("CTR_TF32_GROUP");
    if (!e || !*e) return kTf32Group;
    const int v = std::atoi(e);
    return v > 0 ? v : kNoGroup;
}

// Whether the GEMM runs in X-ring mode (gemm_tc.cuh): fp32 polyphase plans on 256-row
// tiles with at least four taps along x.  The taps of one tap row then share one staged-
// input box of 128 + mx - 1 rows (at most 256, a TMA box's height), and the split-K units
// take whole channel slices.  The operand bytes per K slice drop (by 24% at four taps), but
// the weight ring then holds 128 KB instead of 192, and an SM's TMA feed follows the bytes
// in flight: measured on GB300 with operands in HBM, the iSTFT (four taps) ran 163.9 ->
// 161.8 us and two-tap layers 2-3% slower, hence the four-tap threshold.
bool xring_eligible(const ctr_plan_s *pl, int bn, int splits) {
    if (prec_of(pl) != Prec::F32 || pl->path != CTR_PATH_POLYPHASE || bn != 256) return false;
    if (pl->m[1] < 4 || ctr::kBM + pl->m[1] - 1 > 256) return false;
    return splits <= pl->C_in_pad * 4 / ctr::kBKBytes;
}

// Choose the phase-row tile BN in {64, 128, 256} and the split-K factor: fewest estimated
// clocks, counting whole waves of tiles over the SMs, a tile's time from its MMA time, its
// operand-load time and its output time, and the extra pass over split-K partials.
// The tile a plan needs to run as one half of a fused chained pair (ctr_forward_fused):
// 128 rows for the first layer, its 64 channels x 2 phases in one tile; the second layer's
// rows in one tile of 64 or 128; both without split-K.  0 when the plan is not half of a
// pair of that shape (then the tile model chooses freely).
int fused_pair_bn(const ctr_plan_s *pl);

double choose_tiling(ctr_plan_s *pl, double epi_factor = 1.0) {
    const Prec prec = prec_of(pl);
    const int pair_bn = fused_pair_bn(pl);
    const int group = prec == Prec::F32 ? tf32_group() : kNoGroup;
    const int kb_total = (int)(pl->K_total * op_esize(pl) / ctr::kBKBytes);
    const int64_t num_p = std::max<int64_t>(1, ceil_div(pl->N_total, ctr::kBM));
    double best = 1e300;
    int best_bn = 128, best_sp = 1;
    // A forced split-K factor is clamped to the number of K slices.
    const int forced = pl->forced_split > 0 ? std::min(pl->forced_split, kb_total) : 0;
    for (int bn : {64, 128, 256}) {
        if (pl->forced_bn > 0 && bn != pl->forced_bn) continue;
        if (pl->forced_bn == 0 && pair_bn > 0 && bn != pair_bn) continue;
        const int64_t num_r = std::max<int64_t>(1, ceil_div(pl->M_rows, bn));
        for (int sp = 1; sp <= 16; ++sp) {
            if (forced > 0 && sp != forced) continue;
            if (forced == 0 && pair_bn > 0 && sp != 1) continue;
            if (sp > kb_total) break;
            if (sp > 1 && forced == 0 && kb_total / sp < 4) break;
            const double kbs = (double)ceil_div(kb_total, sp);
            if (bn > ctr::kMaxGroupedBN && kbs > group) continue;
            const int64_t tiles = num_p * num_r * sp;
            const int64_t waves = ceil_div(tiles, pl->num_sms);
            // Per tile: tensor-pipe time, operand loads from L2, and output writes at ~20 B
            // per clock per SM (the HBM share of one SM).
            const double mma = kbs * slice_clocks(prec, bn);
            const double epi = epi_factor * ctr::kBM * (double)bn * esize_io(pl) / 20.0 + 300.0;
            double t;
            if (prec == Prec::F32) {
                // Two operand planes, loaded at ~65 B per clock per SM (fitted to forced-tile
                // timings on GB300 with operands coming from HBM: inputs and weights rotated
                // past twice the L2).  A 256-row tile has one accumulator: its output stage
                // does not overlap the next work unit's MMAs, and folding each accumulation
                // group into the sums pauses them (~600 clocks).
                const double load = kbs * (ctr::kBM + bn) * (double)ctr::kBKBytes * 2 / 65.0;
                double unit = std::max(mma, load);
                if (bn == 256) {
                    unit += 600.0 * (std::ceil(kbs / std::min(kbs, (double)group)) - 1.0);
                    t = (double)waves * (unit + epi) + 2000.0;
                } else {
                    t = (double)waves * std::max(unit, epi) + epi + 2000.0;
                }
            } else {
                // One plane, operand loads at ~50 B per clock per SM.
                const double load = kbs * (ctr::kBM + bn) * (double)ctr::kBKBytes / 50.0;
                t = (double)waves * std::max(mma, std::max(load, epi)) + 2000.0;
            }
            if (sp > 1 || pl->path == CTR_PATH_COL2IM) {
                // partials written once and read once by the reduce (or col2im) pass, ~1.25
                // KB per clock for the whole GPU (measured: split-K 2 against 1)
                t += (double)(sp + 1) * num_p * ctr::kBM * num_r * bn * 4.0 / 1250.0;
            }
            if (t < best * 0.98) {
                best = t;
                best_bn = bn;
                best_sp = sp;
            }
        }
    }
    pl->block_n = best_bn;
    pl->splits = best_sp;
    pl->kb_group = best_bn <= ctr::kMaxGroupedBN ? group : kNoGroup;
    pl->num_p_tiles = (int)num_p;
    pl->num_r_tiles = (int)std::max<int64_t>(1, ceil_div(pl->M_rows, best_bn));
    pl->num_tiles = (int64_t)pl->num_p_tiles * pl->num_r_tiles * pl->splits;
    return best;
}

// Extent of the dilated kernel along dimension d: (k - 1)*dil + 1 samples, of which the k
// taps are every dil-th.
int64_t dilated_extent(const ctr_plan_s *pl, int d) { return (pl->k[d] - 1) * pl->dil[d] + 1; }

// Output length of dimension d: (L_in - 1)*s + (k - 1)*dil + 1 + op - p_front - p_back,
// i.e. (L_in - 1)*s - 2p + k + op without dilation and with equal pads.
int64_t output_length(const ctr_plan_s *pl, int d) {
    // A streaming plan emits the s*L_in samples its input frames complete (see
    // ctr_plan_set_streaming); its padding is 0.
    if (pl->streaming && d == 1) return pl->in[1] * pl->s[1];
    return (pl->in[d] - 1) * pl->s[d] + dilated_extent(pl, d) + pl->op[d] - pl->p[d] - pl->pe[d];
}

// Output lengths and the element counts derived from them; false when an output length is
// not positive or a count leaves the supported range (the plan is then left unchanged).
bool set_output_lengths(ctr_plan_s *pl) {
    const int64_t kLim = (int64_t)1 << 31;
    int64_t out[2];
    int64_t total_out = pl->B * pl->C_out;
    for (int d = 0; d < 2; ++d) {
        out[d] = output_length(pl, d);
        if (out[d] < 1 || out[d] >= kLim) return false;
        total_out *= out[d];
        if (total_out >= ((int64_t)1 << 46)) return false;
    }
    pl->out[0] = out[0];
    pl->out[1] = out[1];
    return true;
}

// Whether a chained pair has the shape the fused kernel takes (fused_pair.cu checks the
// rest, shared memory included): 16-bit 1-D polyphase layers, the first of stride 2 with 64
// output channels, the second with 64 input channels, at most 128 phase rows, an NCHW
// output and no further chain.
bool fusable_shape(const ctr_plan_s *a, const ctr_plan_s *b) {
    return a && b && a->dtype == b->dtype && a->dtype != CTR_F32 && a->ndim == 1 &&
           b->ndim == 1 && a->path == CTR_PATH_POLYPHASE && b->path == CTR_PATH_POLYPHASE &&
           a->s[1] == 2 && a->C_out == 64 && b->C_in == 64 && b->C_out * b->s[1] <= 128 &&
           !b->chain_next && !b->nhwc && !a->streaming && a->dil[1] == 1 && b->dil[1] == 1;
}

int fused_pair_bn(const ctr_plan_s *pl) {
    if (fusable_shape(pl, pl->chain_next)) return 128;
    if (fusable_shape(pl->chain_prev, pl)) return pl->C_out * pl->s[1] <= 64 ? 64 : 128;
    return 0;
}

// Phase geometry of the polyphase path per dimension (see ctr_plan_s): taps, halos, tap base,
// output offset, valid phase positions and the staged pitch, for unpadded phases
// (out_phases = 0) or output phases (1).
void phase_geometry(ctr_plan_s *pl, int out_phases) {
    for (int d = 0; d < 2; ++d) {
        const int64_t s = pl->s[d], mk = ceil_div(dilated_extent(pl, d), s);
        pl->mk[d] = mk;
        if (out_phases) {
            const int64_t pq = pl->p[d] / s, pm = pl->p[d] - pq * s;
            const int64_t c0 = pq - (mk - 1);    // input index of tap 0 at phase position 0
            pl->m[d] = mk + (pm > 0 ? 1 : 0);
            pl->pm[d] = pm;
            pl->hf[d] = std::max<int64_t>(0, -c0);
            pl->rb[d] = std::max<int64_t>(0, c0);
            pl->ep[d] = 0;
            pl->Qv[d] = ceil_div(pl->out[d], s);
            pl->P[d] = std::max(pl->hf[d] + pl->in[d], pl->rb[d] + pl->Qv[d] + pl->m[d] - 1);
        } else {
            pl->m[d] = mk;
            pl->pm[d] = 0;
            pl->hf[d] = mk - 1;
            pl->rb[d] = 0;
            pl->ep[d] = pl->p[d];
            pl->Qv[d] = ceil_div(pl->out[d] + pl->p[d], s);
            pl->P[d] = std::max(pl->in[d] + 2 * (mk - 1), pl->Qv[d] + mk - 1);
        }
    }
}

// Bytes of the widest aligned store of an interior output run (see make_epi): the run length
// (the x stride), the output offset of the phase map and the output row pitch must all be
// multiples of it.  Element size when nothing wider fits.
int run_store_bytes(const ctr_plan_s *pl, int64_t ex) {
    const int es = esize_io(pl);
    const int64_t run = pl->s[1] * es;
    for (int w : {16, 8, 4})
        if (run % w == 0 && (ex * es) % w == 0 && (pl->out[1] * es) % w == 0) return w;
    return es;
}

// Output phases when they cost no extra tap (p mod s = 0 in every dimension), and otherwise
// when the tile model, with element-wise stores priced at 2.5x (bf16) or 1.5x (fp32) the
// vector rate, expects them to be faster: a layer bound by its output stores rather than by
// its products.  A chained output goes to the next plan's channels-last staged input, where
// the runs of one position are channels, so it gains nothing from aligned runs.
int choose_phase_origin(ctr_plan_s *pl) {
    if (pl->streaming) return 0;   // the carried frames are the unpadded form's halo rows
    if (pl->forced_origin == CTR_PHASE_UNPADDED) return 0;
    if (pl->forced_origin == CTR_PHASE_OUTPUT) return 1;
    if (pl->p[0] % pl->s[0] == 0 && pl->p[1] % pl->s[1] == 0) return 1;
    if (pl->chain_next) return 0;
    const int es = esize_io(pl);
    const int w_pad = run_store_bytes(pl, pl->p[1]);
    const double f_pad = w_pad > es ? 1.0 : (es == 2 ? 2.5 : 1.5);
    const auto estimate = [&](int out_phases, double factor) {
        phase_geometry(pl, out_phases);
        pl->S_pad = (int)(pl->S <= ctr::kBM ? next_pow2(pl->S) : round_up(pl->S, ctr::kBM));
        pl->M_rows = pl->C_out * pl->S_pad;
        pl->M_pad = round_up(pl->M_rows, 64);
        pl->K_total = pl->m[0] * pl->m[1] * pl->C_in_pad;
        pl->N_total = pl->B * pl->P[0] * pl->P[1];
        return choose_tiling(pl, factor);
    };
    const double t_pad = estimate(0, f_pad);
    const double t_out = estimate(1, 1.0);
    return t_out < t_pad ? 1 : 0;
}

// A channels-last y whose rows of C_out channels are whole 16-byte vectors: the vectorised
// channels-last output stages apply; otherwise the element-wise one does.
bool nhwc_out_vector(const ctr_plan_s *pl) { return (pl->C_out * esize_io(pl)) % 16 == 0; }

// Derive the GEMM geometry, tiling, packed size and workspace layout from the path.
void layout_plan(ctr_plan_s *pl) {
    pl->packed_bytes = 0;
    pl->ws_bytes_needed = 0;
    pl->ws_off_stage = pl->ws_stage_bytes = pl->ws_off_raw = pl->ws_raw_bytes = 0;
    pl->chain_zeroed_ws = nullptr;   // the staged layout may change
    pl->row_pm = 0;
    pl->splits = 1;
    pl->block_n = 0;
    pl->num_tiles = 0;
    if (pl->path == CTR_PATH_GATHER || pl->path == CTR_PATH_DEPTHWISE) {
        // The torch weight [C_in][C_out/groups][k...], copied as is.
        pl->packed_bytes =
            (size_t)(pl->C_in * (pl->C_out / pl->groups) * pl->k[0] * pl->k[1]) * esize_io(pl);
        pl->S = pl->S_pad = 0;
        return;
    }
    const int bk = bk_elems(pl);
    pl->C_in_pad = round_up(pl->C_in, bk);
    if (pl->path == CTR_PATH_POLYPHASE) {
        pl->S = (int)(pl->s[0] * pl->s[1]);
        pl->out_phases = choose_phase_origin(pl);
        phase_geometry(pl, pl->out_phases);
    } else {  // col2im: plain GEMM over input positions, rows (oc, tap)
        pl->out_phases = 0;
        for (int d = 0; d < 2; ++d) {
            pl->m[d] = pl->mk[d] = 1;
            pl->pm[d] = pl->hf[d] = pl->rb[d] = 0;
            pl->ep[d] = pl->p[d];
            pl->Qv[d] = pl->in[d];
            pl->P[d] = pl->in[d];
        }
        pl->S = (int)(pl->k[0] * pl->k[1]);
    }
    pl->S_pad = (int)(pl->S <= ctr::kBM ? next_pow2(pl->S) : round_up(pl->S, ctr::kBM));
    pl->M_rows = pl->C_out * pl->S_pad;
    pl->M_pad = round_up(pl->M_rows, 64);
    pl->K_total = pl->m[0] * pl->m[1] * pl->C_in_pad;
    pl->N_total = pl->B * pl->P[0] * pl->P[1];
    choose_tiling(pl);
    // A chained producer packs its rows phase-major within each tile, so that the output
    // stage's 32-row chunks are runs of consecutive channels (contiguous in the next
    // plan's channels-last staged input).  Needs whole phase sets that divide the tile.
    // A channels-last y is written by the same output stage, when its rows of C_out channels
    // keep the 16-byte vector stores aligned.
    pl->row_pm = (pl->chain_next || (pl->nhwc && nhwc_out_vector(pl))) &&
                 pl->path == CTR_PATH_POLYPHASE && pl->S == pl->S_pad && pl->S_pad <= 32 &&
                 pl->block_n % pl->S_pad == 0 && pl->block_n / pl->S_pad >= 2;
    if (pl->row_pm) pl->M_pad = (int64_t)pl->num_r_tiles * pl->block_n;
    pl->packed_bytes = (size_t)pl->M_pad * pl->K_total * op_esize(pl) * op_planes(pl);
    pl->ws_off_stage = 0;
    pl->ws_stage_bytes = (size_t)pl->N_total * pl->C_in_pad * op_esize(pl) * op_planes(pl);
    size_t off = align256(pl->ws_stage_bytes);
    if (pl->path == CTR_PATH_COL2IM || pl->splits > 1) {
        pl->ws_off_raw = off;
        pl->ws_raw_bytes = (size_t)ctr::raw_split_stride_of(pl) * pl->splits * sizeof(float);
        off = align256(off + pl->ws_raw_bytes);
    }
    pl->ws_off_state = pl->ws_state_bytes = 0;
    if (pl->streaming && pl->m[1] > 1) {
        pl->ws_off_state = off;
        pl->ws_state_bytes =
            (size_t)pl->B * (pl->m[1] - 1) * pl->C_in_pad * op_esize(pl) * op_planes(pl);
        off = align256(off + pl->ws_state_bytes);
    }
    pl->ws_bytes_needed = (pl->ws_stage_bytes || pl->ws_raw_bytes) ? off : 0;
}

// Whether pl's output can feed nx's staged input directly (see ctr_plan_chain).
bool chain_compatible(const ctr_plan_s *pl, const ctr_plan_s *nx) {
    return pl->path == CTR_PATH_POLYPHASE &&
           (nx->path == CTR_PATH_POLYPHASE || nx->path == CTR_PATH_COL2IM) &&
           pl->dtype == nx->dtype && pl->B == nx->B && pl->ndim == nx->ndim &&
           nx->C_in == pl->C_out && nx->in[0] == pl->out[0] && nx->in[1] == pl->out[1];
}

// The tensor-core kernels index tiles, staged positions (with the largest tap shift) and
// packed rows in 32 bits.
bool tc_index_fits(const ctr_plan_s *pl) {
    const int64_t lim = (int64_t)1 << 31;
    const int64_t shift = pl->P[1] * (pl->rb[0] + pl->m[0] - 1) + pl->rb[1] + pl->m[1];
    return pl->num_p_tiles * (int64_t)ctr::kBM + shift < lim && pl->num_tiles < lim &&
           pl->M_pad + 256 < lim;
}

int choose_path(const ctr_plan_s *pl) {
    if (pl->forced_path != CTR_PATH_AUTO) return pl->forced_path;
    if (pl->groups > 1)   // the tensor-core paths contract over all input channels
        return ctr::depthwise_supported(pl) ? CTR_PATH_DEPTHWISE : CTR_PATH_GATHER;
    const int64_t T = pl->k[0] * pl->k[1];
    // Dilated taps: the polyphase rows of the zero-inserted kernel would be mostly zeros
    // (phases that no tap reaches), so a dilated plan runs the col2im GEMM over its real taps,
    // or the gather kernel.  Forcing polyphase stays possible (the prepack inserts the zeros).
    if (pl->dil[0] > 1 || pl->dil[1] > 1)
        return (pl->C_in >= 16 && T * pl->C_out >= 64) ? CTR_PATH_COL2IM : CTR_PATH_GATHER;
    const bool kdiv = (pl->k[0] % pl->s[0] == 0) && (pl->k[1] % pl->s[1] == 0);
    const int64_t S = pl->s[0] * pl->s[1];
    const int64_t mprod = ceil_div(pl->k[0], pl->s[0]) * ceil_div(pl->k[1], pl->s[1]);
    if (kdiv) return (S * pl->C_out >= 64 && pl->C_in * mprod >= 16) ? CTR_PATH_POLYPHASE
                                                                    : CTR_PATH_GATHER;
    return (pl->C_in >= 16 && T * pl->C_out >= 64) ? CTR_PATH_COL2IM : CTR_PATH_GATHER;
}

}  // namespace

namespace ctr {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    }
    return fn;
}

}  // namespace

// 2-D tiled tensor map over a row-major [rows][inner] matrix, box [box_rows][128 bytes],
// 128-byte swizzle (the K-major SWIZZLE_128B operand layout of tcgen05.mma), zero fill.
bool encode_2d(CUtensorMap *map, const void *base, int io, uint64_t inner, uint64_t rows,
               uint32_t box_rows, int box_bytes) {
    auto fn = get_encode_fn();
    if (!fn || (box_bytes != 128 && box_bytes != 64)) return false;
    const uint32_t es = io == IO_F32 ? 4 : 2;
    const CUtensorMapDataType dt = io == IO_BF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                   : io == IO_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner * es};
    cuuint32_t box[2] = {(cuuint32_t)(box_bytes / es), box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                    box_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

EpiParams make_epi(const ctr_plan_s *pl, const void *bias, void *y) {
    EpiParams e;
    e.S = pl->S;
    e.S_pad = pl->S_pad;
    e.sy = (int)pl->s[0];
    e.sx = (int)pl->s[1];
    e.py = (int)pl->ep[0];
    e.px = (int)pl->ep[1];
    e.Py = pl->P[0];
    e.Px = pl->P[1];
    e.Qvy = pl->Qv[0];
    e.Qvx = pl->Qv[1];
    e.B = pl->B;
    e.C_out = pl->C_out;
    e.Hout = pl->out[0];
    e.Wout = pl->out[1];
    e.bias = bias;
    e.y = y;
    e.io = pl->dtype;   // the ctr_dtype codes are the IoType codes
    e.act = pl->act;
    e.slope = pl->slope;
    // Output-stage variant: whole phase sets per 32-column chunk when S = S_pad is a power
    // of two <= 32 (1-D, or 2-D with sx = sy = 2 or 4), 32 consecutive phases of one
    // channel when a 1-D S is a multiple of 32, else the generic per-element stage.
    const int64_t sx = pl->s[1], sy = pl->s[0];
    const bool whole = pl->S == pl->S_pad;
    int nx = 0;  // run length of the fast variants
    e.kind = EPI_KIND_GENERIC;
    if (whole && sy == 1) {
        switch (sx) {
            case 1: e.kind = EPI_KIND_1D_S1; nx = 1; break;
            case 2: e.kind = EPI_KIND_1D_S2; nx = 2; break;
            case 4: e.kind = EPI_KIND_1D_S4; nx = 4; break;
            case 8: e.kind = EPI_KIND_1D_S8; nx = 8; break;
            case 16: e.kind = EPI_KIND_1D_S16; nx = 16; break;
            case 32: e.kind = EPI_KIND_1D_S32; nx = 32; break;
            default:
                if (sx % 32 == 0) {
                    e.kind = EPI_KIND_1D_LARGE;
                    nx = 32;
                }
        }
    } else if (whole && sx == sy && (sx == 2 || sx == 4)) {
        e.kind = sx == 2 ? EPI_KIND_2D_S2x2 : EPI_KIND_2D_S4x4;
        nx = (int)sx;
    }
    if (pl->nhwc && !nhwc_out_vector(pl)) e.kind = EPI_KIND_GENERIC;
    // Widest aligned store of an interior run: the run length, the run-to-run step of one
    // position (sx elements), the padding offset and the output row pitch must all be
    // multiples of it, so every thread and row share the same alignment.
    const int es = esize_io(pl);
    e.out_staged = 0;
    e.ys_Px = e.ys_Py = e.ys_hx = e.ys_hy = e.ys_cpad = e.ys_lo = 0;
    e.ys_tf32 = 0;
    e.pm_tc = pl->row_pm ? pl->block_n / pl->S_pad : 0;
    e.store_bytes = es;
    for (int w : {16, 8, 4}) {
        if (nx > 0 && (nx * es) % w == 0 && (sx * es) % w == 0 && (e.px * es) % w == 0 &&
            (pl->out[1] * es) % w == 0) {
            e.store_bytes = w;
            break;
        }
    }
    // Runs of sx = 2 outputs at odd columns (px odd): each lane stores its second output with
    // its right neighbour's first, an aligned pair, when rows keep that alignment (even Wout)
    // and y is aligned to two elements.
    e.shift2 = (e.kind == EPI_KIND_1D_S2 || e.kind == EPI_KIND_2D_S2x2) && (e.px & 1) &&
               pl->out[1] % 2 == 0 && reinterpret_cast<uintptr_t>(y) % (2 * es) == 0;
    return e;
}

int64_t raw_ld_of(const ctr_plan_s *pl) { return (int64_t)pl->num_r_tiles * pl->block_n; }

int64_t raw_split_stride_of(const ctr_plan_s *pl) {
    return (int64_t)pl->num_p_tiles * kBM * raw_ld_of(pl);
}

// The tensor-core paths after validation: stage x, encode the operand maps, run the GEMM
// (with timing events around it when given), then the split-K reduce or col2im.  ws holds
// the staged input and the raw partials at the plan's offsets; status is the device status
// word the GEMM reports bounded-wait timeouts into.
// Records a timing event.  Under stream capture it becomes an external event-record node,
// so every replay of the graph records it (a plain record would only order the graph);
// outside capture it is a plain record (the external flag is for capture only).
cudaError_t record_timing(cudaEvent_t ev, cudaStream_t st) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    const cudaError_t e = cudaStreamIsCapturing(st, &cs);
    if (e != cudaSuccess) return e;
    return cs == cudaStreamCaptureStatusActive
               ? cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal)
               : cudaEventRecord(ev, st);
}

// The GEMM's shared-memory pipeline for a plan: the instantiation's default stage ring, or
// the shared-X mode for 16-bit 1-D polyphase plans with several taps.  In that mode a stage
// holds one X box of 128 + (taps - 1) staged rows (rounded up to 8) per channel slice,
// which every tap reads through a shifted descriptor, instead of one 128-row box per tap;
// the whole weight tile stays resident when the plan has one row tile and it fits beside
// two X boxes.  It is taken when it keeps more tiles in flight than the default ring: the
// small-K layers whose loads, not their MMAs, set the pace.
void set_pipeline_layout(const ctr_plan_s *pl, GemmParams *gp) {
    const Prec prec = prec_of(pl);
    const GemmLayout lay = gemm_layout(prec, pl->block_n);
    gp->xshare = 0;
    gp->wres = 0;
    gp->x_rows = kBM;
    gp->nstages = lay.stages;
    gp->stage_bytes = lay.stage_bytes;
    gp->wres_off = 0;
    gp->bar_off = lay.stages * lay.stage_bytes;
    gp->smem_bytes = 1024 + gp->bar_off + kGemmBarBytes;
    gp->xring = 0;
    gp->xring_off = 0;
    gp->my = (int)pl->m[0];
    if (xring_eligible(pl, pl->block_n, pl->splits)) {
        // X-ring mode: the weight ring of one-plane, one-tap stages, then two X slots (a
        // box of both planes each), then the barriers.
        const int x_rows = (int)((kBM + pl->m[1] - 1 + 7) / 8 * 8);
        const int64_t slot_bytes = 2 * (int64_t)x_rows * lay.slice_bytes;
        const int64_t avail = lay.smem_budget - 1024 - kGemmBarBytes - 2 * slot_bytes;
        const int64_t stages = std::min<int64_t>(avail / lay.w_box_bytes, kGemmMaxStages);
        if (stages >= 3) {
            gp->xring = 1;
            gp->x_rows = x_rows;
            gp->nstages = (int)stages;
            gp->stage_bytes = lay.w_box_bytes;
            gp->xring_off = (int)(stages * lay.w_box_bytes);
            gp->bar_off = gp->xring_off + (int)(2 * slot_bytes);
            gp->smem_bytes = 1024 + gp->bar_off + kGemmBarBytes;
        }
        return;
    }
    if (!is_16bit(prec) || pl->path != CTR_PATH_POLYPHASE || pl->splits != 1 ||
        pl->m[0] != 1 || pl->m[1] < 2)
        return;
    const int x_rows = (int)((kBM + pl->m[1] - 1 + 7) / 8 * 8);
    if (x_rows > 256) return;
    const int64_t x_bytes = (int64_t)x_rows * lay.slice_bytes;
    const int64_t kb_total = pl->K_total * 2 / lay.slice_bytes;
    const int64_t kb_per_tap = pl->C_in_pad * 2 / lay.slice_bytes;
    const int64_t avail = lay.smem_budget - 1024 - kGemmBarBytes;
    const int64_t w_tile = kb_total * lay.w_box_bytes;
    int64_t stages, stage_bytes;
    int wres = 0;
    if (pl->num_r_tiles == 1 && w_tile + 2 * x_bytes <= avail) {
        wres = 1;
        stage_bytes = x_bytes;
        stages = (avail - w_tile) / x_bytes;
    } else {
        stage_bytes = x_bytes + pl->m[1] * lay.w_box_bytes;
        stages = avail / stage_bytes;
    }
    stages = std::min<int64_t>(stages, kGemmMaxStages);
    const double tiles_default = (double)lay.stages / (double)kb_total;
    const double tiles_shared = (double)stages / (double)kb_per_tap;
    if (stages < 2 || tiles_shared < 1.2 * tiles_default) return;
    gp->xshare = 1;
    gp->wres = wres;
    gp->x_rows = x_rows;
    gp->nstages = (int)stages;
    gp->stage_bytes = (int)stage_bytes;
    gp->wres_off = (int)(stages * stage_bytes);
    gp->bar_off = gp->wres_off + (wres ? (int)w_tile : 0);
    gp->smem_bytes = 1024 + gp->bar_off + kGemmBarBytes;
}

cudaError_t run_tc_path(const ctr_plan_s *pl, const void *x, const void *w_packed,
                        const void *bias, void *y, char *ws, uint32_t *status,
                        cudaEvent_t ev_before, cudaEvent_t ev_after, cudaStream_t st,
                        const ctr_plan_s *chained_to, bool staged_in) {
    cudaError_t e;
    void *xs = ws + pl->ws_off_stage;
    float *raw = pl->ws_raw_bytes ? reinterpret_cast<float *>(ws + pl->ws_off_raw) : nullptr;
    if (!staged_in && (e = pl->nhwc ? launch_stage_nhwc(pl, x, xs, st)
                                    : launch_stage_x(pl, x, xs, st)) != cudaSuccess)
        return e;
    if (pl->streaming &&
        (e = launch_stream_state(pl, xs, ws + pl->ws_off_state, st)) != cudaSuccess)
        return e;

    const bool h16 = io16(pl);   // bf16 or fp16 operands, one plane
    const int es = esize_io(pl);
    const size_t w_plane = (size_t)pl->M_pad * pl->K_total * es;
    const size_t x_plane = (size_t)pl->N_total * pl->C_in_pad * es;
    // maps: staged input (128-position boxes), packed weight (block_n-row boxes), lo planes;
    // every box is one K slice of the GEMM instantiation wide.
    const int sb = gemm_slice_bytes(prec_of(pl), pl->block_n);
    GemmParams gp;
    std::memset(&gp, 0, sizeof(gp));
    set_pipeline_layout(pl, &gp);
    CUtensorMap maps[4];
    bool ok = encode_2d(&maps[0], xs, pl->dtype, pl->C_in_pad, pl->N_total, (uint32_t)gp.x_rows, sb) &&
              encode_2d(&maps[1], w_packed, pl->dtype, pl->K_total, pl->M_pad, pl->block_n, sb);
    if (!h16) {
        ok = ok &&
             encode_2d(&maps[2], static_cast<char *>(xs) + x_plane, IO_F32, pl->C_in_pad,
                       pl->N_total, (uint32_t)gp.x_rows, sb) &&
             encode_2d(&maps[3], static_cast<const char *>(w_packed) + w_plane, IO_F32,
                       pl->K_total, pl->M_pad, pl->block_n, sb);
    } else {
        maps[2] = maps[0];
        maps[3] = maps[1];
    }
    if (!ok) return cudaErrorInvalidValue;

    gp.num_p_tiles = pl->num_p_tiles;
    gp.num_r_tiles = pl->num_r_tiles;
    gp.splits = pl->splits;
    gp.num_tiles = pl->num_tiles;
    gp.kb_total = (int)(pl->K_total * es / sb);
    gp.kb_per_tap = (int)(pl->C_in_pad * es / sb);
    gp.kb_group = pl->kb_group == kNoGroup ? kNoGroup : pl->kb_group * (kBKBytes / sb);
    gp.mx = (int)pl->m[1];
    gp.Px = pl->P[1];
    gp.shift0 = pl->rb[0] * pl->P[1] + pl->rb[1];
    const bool fused = pl->path == CTR_PATH_POLYPHASE && pl->splits == 1;
    gp.epi_mode = fused ? EPI_POLYPHASE : EPI_RAW;
    gp.epi = make_epi(pl, bias, y);
    if (chained_to) {
        // Output into the next plan's staged input (its staging geometry).
        const ctr_plan_s *nx = chained_to;
        gp.epi.out_staged = 1;
        gp.epi.y = static_cast<char *>(nx->ws) + nx->ws_off_stage;
        gp.epi.ys_Py = nx->P[0];
        gp.epi.ys_Px = nx->P[1];
        gp.epi.ys_hy = nx->hf[0];
        gp.epi.ys_hx = nx->hf[1];
        gp.epi.ys_cpad = nx->C_in_pad;
        gp.epi.ys_lo = nx->N_total * nx->C_in_pad;
        gp.epi.ys_tf32 = nx->dtype == CTR_F32;
    } else if (pl->nhwc) {
        // A channels-last y: the same channels-last output stage, on y itself.
        gp.epi.out_staged = 1;
        gp.epi.y = y;
        gp.epi.ys_Py = pl->out[0];
        gp.epi.ys_Px = pl->out[1];
        gp.epi.ys_hy = gp.epi.ys_hx = 0;
        gp.epi.ys_cpad = pl->C_out;
        gp.epi.ys_lo = 0;
        gp.epi.ys_tf32 = 0;
    }
    gp.raw = raw;
    gp.raw_ld = raw_ld_of(pl);
    gp.raw_split_stride = raw_split_stride_of(pl);
    gp.status = status;
    gp.wait_limit_ns = pl->wait_limit_ns;
    if (ev_before && (e = record_timing(ev_before, st)) != cudaSuccess) return e;
    if ((e = launch_gemm_tc(pl, maps, gp, st)) != cudaSuccess) return e;
    if (ev_after && (e = record_timing(ev_after, st)) != cudaSuccess) return e;
    if (pl->path == CTR_PATH_POLYPHASE && !fused)
        return launch_splitk_reduce(pl, raw, gp.epi, gp.raw_ld, gp.raw_split_stride, st);
    if (pl->path == CTR_PATH_COL2IM) return launch_col2im(pl, raw, gp.raw_ld, bias, y, st);
    return cudaSuccess;
}

}  // namespace ctr

using ctr::encode_2d;
using ctr::make_epi;

namespace ctr {
void count_launches(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
}  // namespace ctr

extern "C" {

const char *ctr_status_string(ctr_status s) {
    switch (s) {
        case CTR_OK: return "ok";
        case CTR_ERR_INVALID_ARG: return "invalid argument";
        case CTR_ERR_UNSUPPORTED: return "unsupported configuration";
        case CTR_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case CTR_ERR_NO_WORKSPACE: return "workspace unbound or too small";
        case CTR_ERR_CUDA: return "CUDA error";
        case CTR_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait gave up";
        case CTR_ERR_NOT_PREPARED: return "plan used before ctr_prepack_weight";
    }
    return "unknown status";
}

uint64_t ctr_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

ctr_status ctr_plan_create(ctr_plan_t *out, int ndim, int64_t N, int64_t C_in, int64_t C_out,
                           const int64_t *in_spatial, const int64_t *kernel,
                           const int64_t *stride, const int64_t *padding,
                           const int64_t *output_padding, int dtype) {
    if (!out) return CTR_ERR_INVALID_ARG;
    *out = nullptr;
    if (ndim != 1 && ndim != 2) return CTR_ERR_INVALID_ARG;
    if (!in_spatial || !kernel || !stride || !padding) return CTR_ERR_INVALID_ARG;
    if (N < 0 || C_in < 1 || C_out < 1) return CTR_ERR_INVALID_ARG;
    if (dtype != CTR_F32 && dtype != CTR_BF16 && dtype != CTR_F16) return CTR_ERR_INVALID_ARG;
    const int64_t kLim = (int64_t)1 << 31;
    if (N >= kLim || C_in >= kLim || C_out >= kLim) return CTR_ERR_INVALID_ARG;

    ctr_plan_s *pl = new (std::nothrow) ctr_plan_s();
    if (!pl) return CTR_ERR_INVALID_ARG;
    pl->ndim = ndim;
    pl->B = N;
    pl->C_in = C_in;
    pl->C_out = C_out;
    pl->dtype = dtype;
    pl->act = CTR_ACT_NONE;
    pl->slope = 0.0f;
    pl->forced_path = CTR_PATH_AUTO;
    pl->forced_origin = CTR_PHASE_AUTO;
    pl->stream_saved_path = CTR_PATH_AUTO;
    pl->forced_split = 0;
    pl->forced_bn = 0;
    pl->groups = 1;
    pl->chain_next = pl->chain_prev = nullptr;
    pl->chain_zeroed_ws = nullptr;
    pl->wait_limit_ns = 4000000000ull;
    // Unit leading dimension for 1-D.
    pl->in[0] = 1; pl->k[0] = 1; pl->s[0] = 1; pl->p[0] = 0; pl->op[0] = 0;
    pl->dil[0] = pl->dil[1] = 1;
    for (int d = 0; d < ndim; ++d) {
        const int dd = d + (2 - ndim);
        pl->in[dd] = in_spatial[d];
        pl->k[dd] = kernel[d];
        pl->s[dd] = stride[d];
        pl->p[dd] = padding[d];
        pl->op[dd] = output_padding ? output_padding[d] : 0;
    }
    int64_t total_out = N * C_out, total_in = N * C_in, total_w = C_in * C_out;
    for (int d = 0; d < 2; ++d) {
        const bool ok = pl->in[d] >= 0 && pl->in[d] < kLim && pl->k[d] >= 1 &&
                        pl->k[d] < kLim && pl->s[d] >= 1 && pl->s[d] < kLim && pl->p[d] >= 0 &&
                        pl->p[d] < kLim && pl->op[d] >= 0 && pl->op[d] < pl->s[d];
        if (!ok) { delete pl; return CTR_ERR_INVALID_ARG; }
        pl->pe[d] = pl->p[d];
        pl->out[d] = output_length(pl, d);
        if (pl->out[d] < 1 || pl->out[d] >= kLim) { delete pl; return CTR_ERR_INVALID_ARG; }
        total_out *= pl->out[d];
        total_in *= std::max<int64_t>(pl->in[d], 1);
        total_w *= pl->k[d];
        if (total_out >= ((int64_t)1 << 46) || total_in >= ((int64_t)1 << 46) ||
            total_w >= ((int64_t)1 << 46)) {
            delete pl;
            return CTR_ERR_INVALID_ARG;
        }
    }
    pl->num_sms = query_num_sms();
    pl->path = choose_path(pl);
    layout_plan(pl);
    if (is_tc_path(pl->path) && !tc_index_fits(pl)) {  // too large for 32-bit tile indexing
        pl->path = CTR_PATH_GATHER;
        layout_plan(pl);
    }
    *out = pl;
    return CTR_OK;
}

ctr_status ctr_plan_set_activation(ctr_plan_t pl, int act, float slope) {
    if (!pl || (act != CTR_ACT_NONE && act != CTR_ACT_LEAKY_RELU)) return CTR_ERR_INVALID_ARG;
    pl->act = act;
    pl->slope = slope;
    return CTR_OK;
}

// Whether the plan's geometry and groups can run on a forced path.
bool path_supported(const ctr_plan_s *pl, int path) {
    if (path == CTR_PATH_DEPTHWISE) return ctr::depthwise_supported(pl);
    if (is_tc_path(path)) return pl->groups == 1;
    return true;
}

// Re-derive the path and layout after a setting changed; a forced path the plan cannot take
// leaves the previous settings in place and reports CTR_ERR_UNSUPPORTED.
ctr_status reroute(ctr_plan_s *pl, int forced_path, int forced_split, int64_t groups) {
    const int old_path = pl->forced_path, old_split = pl->forced_split;
    const int64_t old_groups = pl->groups;
    pl->forced_path = forced_path;
    pl->forced_split = forced_split;
    pl->groups = groups;
    bool ok = forced_path == CTR_PATH_AUTO || path_supported(pl, forced_path);
    if (ok) {
        pl->path = choose_path(pl);
        layout_plan(pl);
        if (is_tc_path(pl->path) && !tc_index_fits(pl)) {
            ok = forced_path == CTR_PATH_AUTO;
            if (ok) {
                pl->path = CTR_PATH_GATHER;
                layout_plan(pl);
            }
        }
    }
    if (ok) return CTR_OK;
    pl->forced_path = old_path;
    pl->forced_split = old_split;
    pl->groups = old_groups;
    pl->path = choose_path(pl);
    layout_plan(pl);
    if (is_tc_path(pl->path) && !tc_index_fits(pl)) {
        pl->path = CTR_PATH_GATHER;
        layout_plan(pl);
    }
    return CTR_ERR_UNSUPPORTED;
}

ctr_status ctr_plan_set_path(ctr_plan_t pl, int path, int split_k) {
    if (!pl || path < CTR_PATH_AUTO || path > CTR_PATH_DEPTHWISE || split_k < 0 || split_k > 16)
        return CTR_ERR_INVALID_ARG;
    if (pl->prepared) return CTR_ERR_INVALID_ARG;
    if (pl->streaming && path != CTR_PATH_POLYPHASE && path != CTR_PATH_AUTO)
        return CTR_ERR_UNSUPPORTED;   // the carried frames are polyphase halo rows
    if (pl->streaming) path = CTR_PATH_POLYPHASE;
    return reroute(pl, path, split_k, pl->groups);
}

ctr_status ctr_plan_set_groups(ctr_plan_t pl, int64_t groups) {
    if (!pl || groups < 1 || pl->C_in % groups != 0 || pl->C_out % groups != 0)
        return CTR_ERR_INVALID_ARG;
    if (pl->prepared || pl->chain_next || pl->chain_prev || pl->streaming)
        return CTR_ERR_INVALID_ARG;
    return reroute(pl, pl->forced_path, pl->forced_split, groups);
}

// New dilation and pads (2-D form); the output lengths, path and layout follow.  Invalid
// geometry, or a forced path that cannot take it, leaves the plan as it was.
ctr_status set_geometry(ctr_plan_s *pl, const int64_t (&dil)[2], const int64_t (&pb)[2],
                        const int64_t (&pe)[2]) {
    const int64_t kLim = (int64_t)1 << 31;
    int64_t old_dil[2], old_p[2], old_pe[2], old_out[2];
    for (int d = 0; d < 2; ++d) {
        if (dil[d] < 1 || dil[d] >= kLim || pb[d] < 0 || pb[d] >= kLim || pe[d] < 0 ||
            pe[d] >= kLim || (pl->k[d] - 1) * dil[d] + 1 >= kLim)
            return CTR_ERR_INVALID_ARG;
        old_dil[d] = pl->dil[d];
        old_p[d] = pl->p[d];
        old_pe[d] = pl->pe[d];
        old_out[d] = pl->out[d];
    }
    auto restore = [&]() {
        for (int d = 0; d < 2; ++d) {
            pl->dil[d] = old_dil[d];
            pl->p[d] = old_p[d];
            pl->pe[d] = old_pe[d];
            pl->out[d] = old_out[d];
        }
    };
    for (int d = 0; d < 2; ++d) {
        pl->dil[d] = dil[d];
        pl->p[d] = pb[d];
        pl->pe[d] = pe[d];
    }
    if (!set_output_lengths(pl)) {
        restore();
        return CTR_ERR_INVALID_ARG;
    }
    const ctr_status st = reroute(pl, pl->forced_path, pl->forced_split, pl->groups);
    if (st != CTR_OK) {
        restore();
        reroute(pl, pl->forced_path, pl->forced_split, pl->groups);
    }
    return st;
}

ctr_status ctr_plan_set_dilation(ctr_plan_t pl, const int64_t *dilation) {
    if (!pl || !dilation) return CTR_ERR_INVALID_ARG;
    if (pl->prepared || pl->chain_next || pl->chain_prev || pl->streaming)
        return CTR_ERR_INVALID_ARG;
    int64_t dil[2] = {1, 1};
    for (int d = 0; d < pl->ndim; ++d) dil[d + (2 - pl->ndim)] = dilation[d];
    const int64_t pb[2] = {pl->p[0], pl->p[1]}, pe[2] = {pl->pe[0], pl->pe[1]};
    return set_geometry(pl, dil, pb, pe);
}

ctr_status ctr_plan_set_pads(ctr_plan_t pl, const int64_t *pads_begin, const int64_t *pads_end) {
    if (!pl || !pads_begin || !pads_end) return CTR_ERR_INVALID_ARG;
    if (pl->prepared || pl->chain_next || pl->chain_prev || pl->streaming)
        return CTR_ERR_INVALID_ARG;
    int64_t pb[2] = {0, 0}, pe[2] = {0, 0};
    for (int d = 0; d < pl->ndim; ++d) {
        pb[d + (2 - pl->ndim)] = pads_begin[d];
        pe[d + (2 - pl->ndim)] = pads_end[d];
    }
    const int64_t dil[2] = {pl->dil[0], pl->dil[1]};
    return set_geometry(pl, dil, pb, pe);
}

ctr_status ctr_plan_set_layout(ctr_plan_t pl, int layout) {
    if (!pl || (layout != CTR_LAYOUT_NCHW && layout != CTR_LAYOUT_NHWC)) return CTR_ERR_INVALID_ARG;
    if (pl->prepared) return CTR_ERR_INVALID_ARG;
    const int nhwc = layout == CTR_LAYOUT_NHWC;
    if (nhwc == pl->nhwc) return CTR_OK;
    if (nhwc && (pl->streaming || pl->forced_path == CTR_PATH_DEPTHWISE)) return CTR_ERR_UNSUPPORTED;
    pl->nhwc = nhwc;
    const ctr_status st = reroute(pl, pl->forced_path, pl->forced_split, pl->groups);
    if (st != CTR_OK) {
        pl->nhwc = !nhwc;
        reroute(pl, pl->forced_path, pl->forced_split, pl->groups);
    }
    return st;
}

ctr_status ctr_plan_set_auto_pad(ctr_plan_t pl, int auto_pad, const int64_t *output_shape) {
    if (!pl || auto_pad < CTR_AUTO_PAD_NOTSET || auto_pad > CTR_AUTO_PAD_VALID)
        return CTR_ERR_INVALID_ARG;
    if (pl->prepared || pl->chain_next || pl->chain_prev || pl->streaming)
        return CTR_ERR_INVALID_ARG;
    if (!output_shape && auto_pad == CTR_AUTO_PAD_NOTSET) return CTR_OK;   // explicit pads stay
    int64_t pb[2] = {0, 0}, pe[2] = {0, 0};
    for (int d = 2 - pl->ndim; d < 2; ++d) {
        const int64_t full = (pl->in[d] - 1) * pl->s[d] + dilated_extent(pl, d) + pl->op[d];
        int64_t total = 0;
        if (output_shape) {
            const int64_t want = output_shape[d - (2 - pl->ndim)];
            if (want < 1) return CTR_ERR_INVALID_ARG;
            total = full - want;
        } else if (auto_pad != CTR_AUTO_PAD_VALID) {
            total = full - pl->in[d] * pl->s[d];
        }
        if (total < 0) return CTR_ERR_UNSUPPORTED;
        if (auto_pad == CTR_AUTO_PAD_SAME_UPPER) {
            pb[d] = total / 2;
            pe[d] = total - pb[d];
        } else {
            pe[d] = total / 2;
            pb[d] = total - pe[d];
        }
    }
    const int64_t dil[2] = {pl->dil[0], pl->dil[1]};
    return set_geometry(pl, dil, pb, pe);
}

ctr_status ctr_plan_set_streaming(ctr_plan_t pl, int enable) {
    if (!pl || (enable != 0 && enable != 1)) return CTR_ERR_INVALID_ARG;
    if (pl->prepared || pl->chain_next || pl->chain_prev) return CTR_ERR_INVALID_ARG;
    if (enable == pl->streaming) return CTR_OK;
    if (!enable) {
        // Back to the plain plan, with the path the caller forced before streaming (if any).
        pl->streaming = 0;
        pl->stream_ready = 0;
        set_output_lengths(pl);
        return reroute(pl, pl->stream_saved_path, pl->forced_split, pl->groups);
    }
    // 1-D, no padding or output_padding, k >= s, one group, undilated, and a carry of at
    // most kMaxStreamCarry frames on the polyphase path.
    if (pl->ndim != 1 || pl->nhwc || pl->p[1] != 0 || pl->pe[1] != 0 || pl->op[1] != 0 ||
        pl->k[1] < pl->s[1] || pl->groups != 1 || pl->dil[1] != 1 ||
        ceil_div(pl->k[1], pl->s[1]) - 1 > ctr::kMaxStreamCarry)
        return CTR_ERR_UNSUPPORTED;
    if (pl->in[1] < 1) return CTR_ERR_INVALID_ARG;
    const int64_t old_out = pl->out[1];
    const int old_path = pl->forced_path;
    pl->streaming = 1;
    if (!set_output_lengths(pl)) {
        pl->streaming = 0;
        pl->out[1] = old_out;
        return CTR_ERR_INVALID_ARG;
    }
    const ctr_status st = reroute(pl, CTR_PATH_POLYPHASE, pl->forced_split, pl->groups);
    if (st != CTR_OK) {   // the plan as it was, its forced path included
        pl->streaming = 0;
        pl->out[1] = old_out;
        reroute(pl, old_path, pl->forced_split, pl->groups);
        return st;
    }
    pl->stream_saved_path = old_path;
    pl->stream_ready = 0;
    return CTR_OK;
}

ctr_status ctr_plan_stream_reset(ctr_plan_t pl, void *stream) {
    if (!pl || !pl->streaming) return CTR_ERR_INVALID_ARG;
    if (pl->ws_bytes_needed > 0 && (!pl->ws || pl->ws_bytes < pl->ws_bytes_needed))
        return CTR_ERR_NO_WORKSPACE;
    if (pl->ws_state_bytes &&
        cudaMemsetAsync(static_cast<char *>(pl->ws) + pl->ws_off_state, 0, pl->ws_state_bytes,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return CTR_ERR_CUDA;
    pl->stream_ready = 1;
    return CTR_OK;
}

ctr_status ctr_plan_set_phase_origin(ctr_plan_t pl, int origin) {
    if (!pl || origin < CTR_PHASE_AUTO || origin > CTR_PHASE_OUTPUT) return CTR_ERR_INVALID_ARG;
    if (pl->prepared) return CTR_ERR_INVALID_ARG;
    pl->forced_origin = origin;
    layout_plan(pl);
    if (is_tc_path(pl->path) && !tc_index_fits(pl)) {
        pl->forced_origin = CTR_PHASE_AUTO;
        layout_plan(pl);
        return CTR_ERR_UNSUPPORTED;
    }
    return CTR_OK;
}

ctr_status ctr_plan_set_tile(ctr_plan_t pl, int block_n) {
    if (!pl || (block_n != 0 && block_n != 64 && block_n != 128 && block_n != 256))
        return CTR_ERR_INVALID_ARG;
    if (pl->prepared) return CTR_ERR_INVALID_ARG;
    pl->forced_bn = block_n;
    layout_plan(pl);
    return CTR_OK;
}

int ctr_plan_get_path(ctr_plan_t pl) { return pl ? pl->path : -1; }

ctr_status ctr_plan_output_shape(ctr_plan_t pl, int64_t *out_spatial) {
    if (!pl || !out_spatial) return CTR_ERR_INVALID_ARG;
    for (int d = 0; d < pl->ndim; ++d) out_spatial[d] = pl->out[d + (2 - pl->ndim)];
    return CTR_OK;
}

size_t ctr_packed_weight_bytes(ctr_plan_t pl) { return pl ? pl->packed_bytes : 0; }
size_t ctr_workspace_bytes(ctr_plan_t pl) { return pl ? pl->ws_bytes_needed : 0; }

ctr_status ctr_plan_bind_workspace(ctr_plan_t pl, void *ptr, size_t bytes) {
    if (!pl) return CTR_ERR_INVALID_ARG;
    if (ptr == nullptr && bytes != 0) return CTR_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(ptr) & 255u) != 0) return CTR_ERR_MISALIGNED;
    if (bytes < pl->ws_bytes_needed) return CTR_ERR_NO_WORKSPACE;
    pl->ws = ptr;
    pl->ws_bytes = bytes;
    pl->stream_ready = 0;   // the carried frames live in the workspace
    return CTR_OK;
}

ctr_status ctr_plan_set_wait_limit_ns(ctr_plan_t pl, uint64_t limit_ns) {
    if (!pl) return CTR_ERR_INVALID_ARG;
    pl->wait_limit_ns = limit_ns;
    return CTR_OK;
}

ctr_status ctr_plan_set_timing_events(ctr_plan_t pl, void *before, void *after) {
    if (!pl || (before == nullptr) != (after == nullptr)) return CTR_ERR_INVALID_ARG;
    pl->ev_before = static_cast<cudaEvent_t>(before);
    pl->ev_after = static_cast<cudaEvent_t>(after);
    return CTR_OK;
}

ctr_status ctr_plan_describe(ctr_plan_t pl, char *buf, size_t len) {
    if (!pl || !buf || len == 0) return CTR_ERR_INVALID_ARG;
    const char *pname = pl->path == CTR_PATH_POLYPHASE    ? "polyphase"
                        : pl->path == CTR_PATH_COL2IM     ? "col2im"
                        : pl->path == CTR_PATH_DEPTHWISE  ? "depthwise"
                                                          : "gather";
    if (is_tc_path(pl->path)) {
        const EpiParams ep = make_epi(pl, nullptr, nullptr);
        snprintf(buf, len,
                 "path=%s prec=%s rows=%lld(pad %lld, BN %d, %d tiles) positions=%lld(%d tiles) "
                 "K=%lld splits=%d group=%d tiles=%lld sms=%d S=%d/%d taps=%lldx%lld%s "
                 "pitch=%lldx%lld epi=%d/%dB%s packed=%zu ws=%zu",
                 pname, pl->dtype == CTR_BF16 ? "bf16" : pl->dtype == CTR_F16 ? "f16" : "tf32+bf16x",
                 (long long)pl->M_rows,
                 (long long)pl->M_pad, pl->block_n, pl->num_r_tiles, (long long)pl->N_total,
                 pl->num_p_tiles, (long long)pl->K_total, pl->splits,
                 pl->kb_group == kNoGroup ? 0 : pl->kb_group, (long long)pl->num_tiles,
                 pl->num_sms, pl->S, pl->S_pad, (long long)pl->m[0], (long long)pl->m[1],
                 pl->out_phases ? " out-phases" : "",
                 (long long)pl->P[0], (long long)pl->P[1], ep.kind, ep.store_bytes,
                 ep.shift2 && pl->path == CTR_PATH_POLYPHASE && !pl->chain_next && !pl->nhwc
                     ? " pairs" : "",
                 pl->packed_bytes, pl->ws_bytes_needed);
    } else {
        snprintf(buf, len, "path=%s dtype=%s groups=%lld packed=%zu ws=0", pname,
                 pl->dtype == CTR_BF16 ? "bf16" : pl->dtype == CTR_F16 ? "f16" : "f32",
                 (long long)pl->groups, pl->packed_bytes);
    }
    if (is_tc_path(pl->path) && pl->block_n > 0) {
        GemmParams gp;
        std::memset(&gp, 0, sizeof(gp));
        ctr::set_pipeline_layout(pl, &gp);
        const size_t used = strlen(buf);
        if (used + 1 < len)
            snprintf(buf + used, len - used, " stages=%d%s", gp.nstages,
                     gp.xring ? " x-ring"
                              : gp.xshare ? (gp.wres ? " shared-x resident-w" : " shared-x") : "");
    }
    if (pl->nhwc) {
        const size_t used = strlen(buf);
        if (used + 1 < len) snprintf(buf + used, len - used, " nhwc");
    }
    if (pl->dil[0] > 1 || pl->dil[1] > 1 || pl->p[0] != pl->pe[0] || pl->p[1] != pl->pe[1]) {
        const size_t used = strlen(buf);
        if (used + 1 < len)
            snprintf(buf + used, len - used, " dil=%lldx%lld pads=%lldx%lld/%lldx%lld",
                     (long long)pl->dil[0], (long long)pl->dil[1], (long long)pl->p[0],
                     (long long)pl->p[1], (long long)pl->pe[0], (long long)pl->pe[1]);
    }
    return CTR_OK;
}

ctr_status ctr_prepack_weight(ctr_plan_t pl, const void *w, void *w_packed, void *stream) {
    if (!pl || !w || !w_packed) return CTR_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(w_packed)) return CTR_ERR_MISALIGNED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (!pl->d_status) {
        if (cudaGetDevice(&pl->status_device) != cudaSuccess) return CTR_ERR_CUDA;
        if (cudaMalloc(&pl->d_status, sizeof(uint32_t)) != cudaSuccess) {
            pl->d_status = nullptr;
            return CTR_ERR_CUDA;
        }
        if (cudaMemset(pl->d_status, 0, sizeof(uint32_t)) != cudaSuccess) return CTR_ERR_CUDA;
    }
    cudaError_t e = is_tc_path(pl->path) ? ctr::launch_prepack(pl, w, w_packed, st)
                                         : ctr::launch_copy_weight(pl, w, w_packed, st);
    if (e != cudaSuccess) return CTR_ERR_CUDA;
    pl->prepared = 1;
    return CTR_OK;
}

ctr_status ctr_forward(ctr_plan_t pl, const void *x, const void *w_packed, const void *bias,
                       void *y, void *stream) {
    if (!pl) return CTR_ERR_INVALID_ARG;
    if (!pl->prepared) return CTR_ERR_NOT_PREPARED;
    ctr_plan_s *nx = pl->chain_next;
    // A weight packed for a chained output (phase-major rows) needs that chain.
    if (pl->row_pm && !nx && !pl->nhwc) return CTR_ERR_INVALID_ARG;
    const bool staged_in = !x && pl->chain_prev != nullptr;  // input staged by the previous plan
    if (!w_packed || (nx ? y != nullptr : y == nullptr)) return CTR_ERR_INVALID_ARG;
    if (!x && !staged_in && pl->B * pl->C_in * pl->in[0] * pl->in[1] > 0)
        return CTR_ERR_INVALID_ARG;
    if ((x && !aligned16(x)) || !aligned16(w_packed) || (y && !aligned16(y)) ||
        (bias && !aligned16(bias)))
        return CTR_ERR_MISALIGNED;
    if (pl->ws_bytes_needed > 0 && (!pl->ws || pl->ws_bytes < pl->ws_bytes_needed))
        return CTR_ERR_NO_WORKSPACE;
    if (pl->streaming && !pl->stream_ready) return CTR_ERR_NOT_PREPARED;
    if (nx) {
        if (!chain_compatible(pl, nx)) return CTR_ERR_INVALID_ARG;
        if (!nx->ws || nx->ws_bytes < nx->ws_bytes_needed) return CTR_ERR_NO_WORKSPACE;
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(pl->ws), a1 = a0 + pl->ws_bytes;
        const uintptr_t b0 = reinterpret_cast<uintptr_t>(nx->ws), b1 = b0 + nx->ws_bytes;
        if (a0 < b1 && b0 < a1) return CTR_ERR_INVALID_ARG;
    }
    if (pl->B == 0) return CTR_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    const bool timed = pl->ev_before != nullptr;
    if (!is_tc_path(pl->path)) {
        if (timed && ctr::record_timing(pl->ev_before, st) != cudaSuccess) return CTR_ERR_CUDA;
        const cudaError_t e = pl->path == CTR_PATH_DEPTHWISE
                                  ? ctr::launch_depthwise(pl, x, w_packed, bias, y, st)
                                  : ctr::launch_gather(pl, x, w_packed, bias, y, st);
        if (e != cudaSuccess) return CTR_ERR_CUDA;
        if (timed && ctr::record_timing(pl->ev_after, st) != cudaSuccess) return CTR_ERR_CUDA;
        return CTR_OK;
    }
    if (pl->N_total == 0) {  // empty input on the col2im path: y = bias or zeros
        return ctr::launch_fill_bias(pl, bias, y, st) == cudaSuccess ? CTR_OK : CTR_ERR_CUDA;
    }
    if (nx && nx->chain_zeroed_ws != nx->ws) {
        // The producer writes only inside the input; the halos and padded channels of the
        // next plan's staged buffer must be zero (once per bound workspace).
        if (cudaMemsetAsync(static_cast<char *>(nx->ws) + nx->ws_off_stage, 0, nx->ws_stage_bytes,
                            st) != cudaSuccess)
            return CTR_ERR_CUDA;
        nx->chain_zeroed_ws = nx->ws;
    }
    const cudaError_t e = ctr::run_tc_path(pl, x, w_packed, bias, y, static_cast<char *>(pl->ws),
                                           pl->d_status, pl->ev_before, pl->ev_after, st, nx,
                                           staged_in);
    return e == cudaSuccess ? CTR_OK : CTR_ERR_CUDA;
}

int ctr_plan_fusable(ctr_plan_t pl) { return pl && ctr::fused_pair_supported(pl) ? 1 : 0; }

ctr_status ctr_forward_fused(ctr_plan_t pl, const void *x, const void *w_packed, const void *bias,
                             const void *next_w_packed, const void *next_bias, void *y,
                             void *stream) {
    if (!pl || !pl->chain_next) return CTR_ERR_INVALID_ARG;
    ctr_plan_s *nx = pl->chain_next;
    if (!pl->prepared || !nx->prepared) return CTR_ERR_NOT_PREPARED;
    if (!ctr::fused_pair_supported(pl)) return CTR_ERR_UNSUPPORTED;
    const bool staged_in = !x && pl->chain_prev != nullptr;
    if (!w_packed || !next_w_packed || !y) return CTR_ERR_INVALID_ARG;
    if (!x && !staged_in && pl->B * pl->C_in * pl->in[0] * pl->in[1] > 0)
        return CTR_ERR_INVALID_ARG;
    if ((x && !aligned16(x)) || !aligned16(w_packed) || !aligned16(next_w_packed) ||
        !aligned16(y) || (bias && !aligned16(bias)) || (next_bias && !aligned16(next_bias)))
        return CTR_ERR_MISALIGNED;
    if (!pl->ws || pl->ws_bytes < pl->ws_bytes_needed) return CTR_ERR_NO_WORKSPACE;
    if (pl->B == 0) return CTR_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(pl->ws);
    void *xs = ws + pl->ws_off_stage;
    cudaError_t e = cudaSuccess;
    if (!staged_in)
        e = pl->nhwc ? ctr::launch_stage_nhwc(pl, x, xs, st) : ctr::launch_stage_x(pl, x, xs, st);
    if (e != cudaSuccess) return CTR_ERR_CUDA;
    if (pl->ev_before && ctr::record_timing(pl->ev_before, st) != cudaSuccess) return CTR_ERR_CUDA;
    e = ctr::launch_fused_pair(pl, xs, w_packed, bias, next_w_packed, next_bias, y, st);
    if (e != cudaSuccess) return CTR_ERR_CUDA;
    if (pl->ev_after && ctr::record_timing(pl->ev_after, st) != cudaSuccess) return CTR_ERR_CUDA;
    return CTR_OK;
}

ctr_status ctr_plan_chain(ctr_plan_t pl, ctr_plan_t nx) {
    if (!pl || pl->prepared) return CTR_ERR_INVALID_ARG;   // the packed row order depends on it
    if (!nx) {
        ctr_plan_s *old = pl->chain_next;
        if (old) old->chain_prev = nullptr;
        pl->chain_next = nullptr;
        layout_plan(pl);
        if (old && !old->prepared) layout_plan(old);
        return CTR_OK;
    }
    if (nx == pl || !chain_compatible(pl, nx) || pl->streaming || nx->streaming)
        return CTR_ERR_INVALID_ARG;
    if (nx->chain_prev && nx->chain_prev != pl) return CTR_ERR_INVALID_ARG;
    if (pl->chain_next && pl->chain_next != nx) pl->chain_next->chain_prev = nullptr;
    pl->chain_next = nx;
    nx->chain_prev = pl;
    nx->chain_zeroed_ws = nullptr;
    layout_plan(pl);
    if (!nx->prepared) layout_plan(nx);   // a fusable pair picks the fused kernel's tiles
    return CTR_OK;
}

// Reads a device status word and clears it when set; true when it was set.
static ctr_status read_and_clear(uint32_t *word, bool *was_set) {
    uint32_t v = 0;
    if (cudaMemcpy(&v, word, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
        return CTR_ERR_CUDA;
    *was_set = v != 0;
    if (v != 0 && cudaMemset(word, 0, sizeof(uint32_t)) != cudaSuccess) return CTR_ERR_CUDA;
    return CTR_OK;
}

ctr_status ctr_plan_check(ctr_plan_t pl, void *stream) {
    if (!pl) return CTR_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return CTR_ERR_CUDA;
    bool timeout = false, set = false;
    ctr_status st;
    if (pl->d_status) {
        if ((st = read_and_clear(pl->d_status, &set)) != CTR_OK) return st;
        timeout = timeout || set;
    }
    // The allocation-free entry point reports into its scratch array's status word.
    if (uint32_t *w = ctr::noalloc_status_word()) {
        if ((st = read_and_clear(w, &set)) != CTR_OK) return st;
        timeout = timeout || set;
    }
    return timeout ? CTR_ERR_DEVICE_TIMEOUT : CTR_OK;
}

void ctr_plan_destroy(ctr_plan_t pl) {
    if (!pl) return;
    if (pl->chain_next) pl->chain_next->chain_prev = nullptr;
    if (pl->chain_prev) pl->chain_prev->chain_next = nullptr;
    if (pl->d_status) {
        int cur = 0;
        cudaGetDevice(&cur);
        if (cur != pl->status_device) cudaSetDevice(pl->status_device);
        cudaFree(pl->d_status);
        if (cur != pl->status_device) cudaSetDevice(cur);
    }
    delete pl;
}

}  // extern "C"
