// nf_gemm_bwd_rms.cu -- instantiations of the GEMM whose epilogue is the
// RMSNorm backward (one translation unit per epilogue so the variants
// compile in parallel).
#include "nf_gemm_kernel.cuh"

namespace nf {

const GemmVariant* gemm_variants_bwd_rms(int* count) {
    static const GemmVariant v[] = {
        make_variant<EPI_BWD_RMS, 64, XCH_NONE>(), make_variant<EPI_BWD_RMS, 128, XCH_NONE>(),
        make_variant<EPI_BWD_RMS, 256, XCH_NONE>(), make_variant<EPI_BWD_RMS, 256, XCH_CLUSTER>(),
        make_variant<EPI_BWD_RMS, 256, XCH_GLOBAL>()};
    *count = 5;
    return v;
}

}  // namespace nf
