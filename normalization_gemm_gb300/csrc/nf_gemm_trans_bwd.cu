// nf_gemm_trans_bwd.cu -- the RMSNorm-backward epilogue over X W^T (W stored
// N x K): the Lazy Pre-Norm backward's dA = rmsnorm_bwd(dC B^T; A, rstd),
// with B the forward's K x N weight read transposed.
#include "nf_gemm_kernel.cuh"

namespace nf {

const GemmVariant* gemm_variants_trans_bwd(int* count) {
    static const GemmVariant v[] = {
        make_variant<EPI_BWD_RMS, 64, XCH_NONE, OPS_B_K>(), make_variant<EPI_BWD_RMS, 128, XCH_NONE, OPS_B_K>(),
        make_variant<EPI_BWD_RMS, 256, XCH_NONE, OPS_B_K>(), make_variant<EPI_BWD_RMS, 256, XCH_CLUSTER, OPS_B_K>(),
        make_variant<EPI_BWD_RMS, 256, XCH_GLOBAL, OPS_B_K>()};
    *count = 5;
    return v;
}

}  // namespace nf
