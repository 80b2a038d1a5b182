// nf_gemm_post_ln.cu -- instantiations of the post-norm LayerNorm GEMM kernel
// (one translation unit per epilogue so the variants compile in parallel).
#include "nf_gemm_wide.cuh"

namespace nf {

const GemmVariant* gemm_variants_post_ln(int* count) {
    static const GemmVariant v[] = {
        make_variant<EPI_POST_LN, 64, false>(), make_variant<EPI_POST_LN, 128, false>(),
        make_variant<EPI_POST_LN, 256, false>(), make_variant<EPI_POST_LN, 256, true>(),
        make_wide_variant<EPI_POST_LN, false>(), make_wide_variant<EPI_POST_LN, true>()};
    *count = 6;
    return v;
}

}  // namespace nf
