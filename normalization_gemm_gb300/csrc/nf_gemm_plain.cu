// nf_gemm_plain.cu -- instantiations of the plain GEMM (unfused baseline) kernel
// (one translation unit per epilogue so the variants compile in parallel).
#include "nf_gemm_kernel.cuh"

namespace nf {

const GemmVariant* gemm_variants_plain(int* count) {
    static const GemmVariant v[] = {
        make_variant<EPI_PLAIN, 64, XCH_NONE>(), make_variant<EPI_PLAIN, 128, XCH_NONE>(),
        make_variant<EPI_PLAIN, 256, XCH_NONE>(), make_variant<EPI_PLAIN, 256, XCH_NONE, OPS_PAIR>()};
    *count = 4;
    return v;
}

}  // namespace nf
