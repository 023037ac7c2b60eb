// gemm_tc.cu -- instantiations of the tensor-core GEMM (gemm_tc.cuh) that write the torch
// layout, and the launch dispatch over precision, tile width and output.
#include "gemm_tc.cuh"

namespace ctr {

// gemm_tc_chain.cu: the instantiations whose output feeds the next plan's staged input.
cudaError_t launch_gemm_tc_chain(const ctr_plan_s *pl, const CUtensorMap *maps,
                                 const GemmParams &gp, cudaStream_t st);
// gemm_tc_f16.cu: the fp16 instantiations (both outputs).
cudaError_t launch_gemm_tc_f16(const ctr_plan_s *pl, const CUtensorMap *maps,
                               const GemmParams &gp, cudaStream_t st);

namespace {
template <Prec P, int BN>
cudaError_t launch_bn(const ctr_plan_s *pl, const CUtensorMap *maps, const GemmParams &gp,
                      cudaStream_t st) {
    return launch_inst<P, BN, false>(pl, maps, gp, st);
}
}  // namespace

namespace {
template <Prec P, int BN>
GemmLayout layout_of() {
    using C = Cfg<P, BN>;
    return GemmLayout{C::kStages, C::kStageBytes, C::kSmemBudget, C::kSlice, C::kXBytes,
                      C::kWBytes, C::kPlanes};
}
}  // namespace

GemmLayout gemm_layout(Prec prec, int block_n) {
    if (is_16bit(prec))   // fp16 and bf16 instantiations have the same layout
        return block_n == 256 ? layout_of<Prec::BF16, 256>()
               : block_n == 128 ? layout_of<Prec::BF16, 128>() : layout_of<Prec::BF16, 64>();
    return block_n == 256 ? layout_of<Prec::F32, 256>()
           : block_n == 128 ? layout_of<Prec::F32, 128>() : layout_of<Prec::F32, 64>();
}

size_t gemm_smem_bytes(Prec prec, int block_n) {
    if (is_16bit(prec))
        return block_n == 256 ? Cfg<Prec::BF16, 256>::kSmem
               : block_n == 128 ? Cfg<Prec::BF16, 128>::kSmem : Cfg<Prec::BF16, 64>::kSmem;
    return block_n == 256 ? Cfg<Prec::F32, 256>::kSmem
           : block_n == 128 ? Cfg<Prec::F32, 128>::kSmem : Cfg<Prec::F32, 64>::kSmem;
}

cudaError_t launch_gemm_tc(const ctr_plan_s *pl, const CUtensorMap *maps, const GemmParams &gp,
                           cudaStream_t st) {
    if (gp.num_tiles <= 0) return cudaSuccess;
    if (pl->dtype == CTR_F16) return launch_gemm_tc_f16(pl, maps, gp, st);
    if (gp.epi.out_staged) return launch_gemm_tc_chain(pl, maps, gp, st);
    if (pl->dtype == CTR_BF16) {
        switch (pl->block_n) {
            case 256: return launch_bn<Prec::BF16, 256>(pl, maps, gp, st);
            case 128: return launch_bn<Prec::BF16, 128>(pl, maps, gp, st);
            default: return launch_bn<Prec::BF16, 64>(pl, maps, gp, st);
        }
    }
    switch (pl->block_n) {
        case 256: return launch_bn<Prec::F32, 256>(pl, maps, gp, st);
        case 128: return launch_bn<Prec::F32, 128>(pl, maps, gp, st);
        default: return launch_bn<Prec::F32, 64>(pl, maps, gp, st);
    }
}

}  // namespace ctr
