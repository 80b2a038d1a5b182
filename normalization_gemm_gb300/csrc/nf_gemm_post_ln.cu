// nf_gemm_post_ln.cu -- instantiations of the post-norm LayerNorm GEMM kernel
// (one translation unit per epilogue so the variants compile in parallel).
#include "nf_gemm_wide.cuh"

namespace nf {

const GemmVariant* gemm_variants_post_ln(int* count) {
    static const GemmVariant v[] = {
        make_variant<EPI_POST_LN, 64, XCH_NONE>(), make_variant<EPI_POST_LN, 128, XCH_NONE>(),
        make_variant<EPI_POST_LN, 256, XCH_NONE>(), make_variant<EPI_POST_LN, 256, XCH_CLUSTER>(),
        make_wide_variant<EPI_POST_LN, false>(), make_wide_variant<EPI_POST_LN, true>(),
        make_variant<EPI_POST_LN, 256, XCH_GLOBAL>(), make_variant<EPI_POST_LN, 256, XCH_GLOBAL, OPS_PAIR>()};
    *count = 8;
    return v;
}

}  // namespace nf
