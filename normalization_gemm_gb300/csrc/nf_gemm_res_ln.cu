// nf_gemm_res_ln.cu -- instantiations of the post-norm LayerNorm GEMM kernel
// with the residual add (H = X W + R before the statistics).
#include "nf_gemm_kernel.cuh"

namespace nf {

const GemmVariant* gemm_variants_res_ln(int* count) {
    static const GemmVariant v[] = {
        make_variant<EPI_POST_LN, 64, XCH_NONE, OPS_RESID>(), make_variant<EPI_POST_LN, 128, XCH_NONE, OPS_RESID>(),
        make_variant<EPI_POST_LN, 256, XCH_NONE, OPS_RESID>(), make_variant<EPI_POST_LN, 256, XCH_CLUSTER, OPS_RESID>(),
        make_variant<EPI_POST_LN, 256, XCH_GLOBAL, OPS_RESID>()};
    *count = 5;
    return v;
}

}  // namespace nf
