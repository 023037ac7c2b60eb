// gemm_tc_f16.cu -- instantiations of the tensor-core GEMM (gemm_tc.cuh) for fp16 I/O: fp16
// operands (kind::f16 with the fp16 format), fp32 accumulation, both outputs (the torch
// layout and the next plan's staged input).  A translation unit of its own, so that it
// compiles in parallel with the fp32/bf16 ones.
#include "gemm_tc.cuh"

namespace ctr {

cudaError_t launch_gemm_tc_f16(const ctr_plan_s *pl, const CUtensorMap *maps,
                               const GemmParams &gp, cudaStream_t st) {
    if (gp.epi.out_staged) {
        switch (pl->block_n) {
            case 256: return launch_inst<Prec::F16, 256, true>(pl, maps, gp, st);
            case 128: return launch_inst<Prec::F16, 128, true>(pl, maps, gp, st);
            default: return launch_inst<Prec::F16, 64, true>(pl, maps, gp, st);
        }
    }
    switch (pl->block_n) {
        case 256: return launch_inst<Prec::F16, 256, false>(pl, maps, gp, st);
        case 128: return launch_inst<Prec::F16, 128, false>(pl, maps, gp, st);
        default: return launch_inst<Prec::F16, 64, false>(pl, maps, gp, st);
    }
}

}  // namespace ctr
