// nf_gemm_trans_plain.cu -- plain GEMMs with a transposed operand: X stored
// K x M (Y = X^T W), optionally with each contraction row of X scaled by
// rstd (the rmsnorm of the stored matrix rebuilt on the fly: the Lazy
// Pre-Norm backward's dB = rmsnorm(A)^T dC), or W stored N x K (Y = X W^T).
#include "nf_gemm_kernel.cuh"

namespace nf {

const GemmVariant* gemm_variants_trans_plain(int* count) {
    static const GemmVariant v[] = {
        make_variant<EPI_PLAIN, 64, XCH_NONE, OPS_A_MN>(),
        make_variant<EPI_PLAIN, 128, XCH_NONE, OPS_A_MN>(),
        make_variant<EPI_PLAIN, 256, XCH_NONE, OPS_A_MN>(),
        make_variant<EPI_PLAIN, 64, XCH_NONE, OPS_A_MN | OPS_A_SCALE>(),
        make_variant<EPI_PLAIN, 128, XCH_NONE, OPS_A_MN | OPS_A_SCALE>(),
        make_variant<EPI_PLAIN, 256, XCH_NONE, OPS_A_MN | OPS_A_SCALE>(),
        make_variant<EPI_PLAIN, 64, XCH_NONE, OPS_B_K>(),
        make_variant<EPI_PLAIN, 128, XCH_NONE, OPS_B_K>(),
        make_variant<EPI_PLAIN, 256, XCH_NONE, OPS_B_K>()};
    *count = 9;
    return v;
}

}  // namespace nf
