// nf_gemm_post_rms.cu -- instantiations of the post-norm RMSNorm GEMM kernel
// (one translation unit per epilogue so the variants compile in parallel).
#include "nf_gemm_wide.cuh"

namespace nf {

const GemmVariant* gemm_variants_post_rms(int* count) {
    static const GemmVariant v[] = {
        make_variant<EPI_POST_RMS, 64, XCH_NONE>(), make_variant<EPI_POST_RMS, 128, XCH_NONE>(),
        make_variant<EPI_POST_RMS, 256, XCH_NONE>(), make_variant<EPI_POST_RMS, 256, XCH_CLUSTER>(),
        make_wide_variant<EPI_POST_RMS, false>(), make_wide_variant<EPI_POST_RMS, true>(),
        make_variant<EPI_POST_RMS, 256, XCH_GLOBAL>(), make_variant<EPI_POST_RMS, 256, XCH_GLOBAL, OPS_PAIR>()};
    *count = 8;
    return v;
}

}  // namespace nf
