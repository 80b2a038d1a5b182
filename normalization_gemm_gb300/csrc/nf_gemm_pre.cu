// nf_gemm_pre.cu -- instantiations of the Lazy Pre-Norm RMS GEMM kernel
// (one translation unit per epilogue so the variants compile in parallel).
#include "nf_gemm_kernel.cuh"

namespace nf {

const GemmVariant* gemm_variants_pre(int* count) {
    static const GemmVariant v[] = {
        make_variant<EPI_PRE_RMS, 64, XCH_NONE>(), make_variant<EPI_PRE_RMS, 128, XCH_NONE>(),
        make_variant<EPI_PRE_RMS, 256, XCH_NONE>(), make_variant<EPI_PRE_RMS, 256, XCH_NONE, OPS_PAIR>(),
        // the row sums of squares split over a row's tiles, gathered through L2
        make_variant<EPI_PRE_RMS, 256, XCH_GLOBAL>(), make_variant<EPI_PRE_RMS, 256, XCH_GLOBAL, OPS_PAIR>()};
    *count = 6;
    return v;
}

}  // namespace nf
