// nf_gemm_bwd_ln.cu -- instantiations of the GEMM whose epilogue is the
// LayerNorm backward (one translation unit per epilogue so the variants
// compile in parallel).
#include "nf_gemm_kernel.cuh"

namespace nf {

const GemmVariant* gemm_variants_bwd_ln(int* count) {
    static const GemmVariant v[] = {
        make_variant<EPI_BWD_LN, 64, XCH_NONE>(), make_variant<EPI_BWD_LN, 128, XCH_NONE>(),
        make_variant<EPI_BWD_LN, 256, XCH_NONE>(), make_variant<EPI_BWD_LN, 256, XCH_CLUSTER>(),
        make_variant<EPI_BWD_LN, 256, XCH_GLOBAL>()};
    *count = 5;
    return v;
}

}  // namespace nf
