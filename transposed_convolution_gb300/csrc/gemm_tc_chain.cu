// gemm_tc_chain.cu -- instantiations of the tensor-core GEMM (gemm_tc.cuh) whose fused output
// stage writes into the next plan's staged input (ctr_plan_chain).
#include "gemm_tc.cuh"

namespace ctr {

cudaError_t launch_gemm_tc_chain(const ctr_plan_s *pl, const CUtensorMap *maps,
                                 const GemmParams &gp, cudaStream_t st) {
    if (pl->dtype == CTR_BF16) {
        switch (pl->block_n) {
            case 256: return launch_inst<Prec::BF16, 256, true>(pl, maps, gp, st);
            case 128: return launch_inst<Prec::BF16, 128, true>(pl, maps, gp, st);
            default: return launch_inst<Prec::BF16, 64, true>(pl, maps, gp, st);
        }
    }
    switch (pl->block_n) {
        case 256: return launch_inst<Prec::F32, 256, true>(pl, maps, gp, st);
        case 128: return launch_inst<Prec::F32, 128, true>(pl, maps, gp, st);
        default: return launch_inst<Prec::F32, 64, true>(pl, maps, gp, st);
    }
}

}  // namespace ctr
