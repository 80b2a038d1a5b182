// nf_splitk.cu -- second half of a split-K GEMM: adds the fp32 partial
// products of the contraction slices, in slice order, and writes Y in bf16.
//
// A GEMM with few output tiles and a long contraction (the weight gradient of
// the Lazy Pre-Norm backward, K x N over M, is the case in point) cuts the
// contraction into slices so that every SM holds one (tile, slice) unit; each
// unit stores its fp32 partial tile into plane s of the workspace.  The
// planes are at most one wave of 128 x 256 fp32 tiles, i.e. L2-resident when
// this kernel reads them back.  The order of the additions is fixed, so the
// result does not depend on the order in which the units finished.
#include "nf_internal.h"
#include "nf_ptx.cuh"

namespace nf {
namespace {

constexpr int SK_THREADS = 256;

// Thread i handles values [8i, 8i + 8): two float4 per plane, one uint4 out.
__global__ void __launch_bounds__(SK_THREADS) nf_splitk_reduce_kernel(const float4* __restrict__ ws, int slices,
                                                                      int64_t groups, uint4* __restrict__ y) {
    griddep_wait();  // the partials come from the GEMM launched just before
    griddep_launch_dependents();
    const int64_t plane = groups * 2;  // float4 per plane
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < groups; i += stride) {
        float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
        const float4* p = ws + 2 * i;
        for (int s = 0; s < slices; ++s, p += plane) {
            const float4 a = __ldcg(p), b = __ldcg(p + 1);
            acc[0] += a.x, acc[1] += a.y, acc[2] += a.z, acc[3] += a.w;
            acc[4] += b.x, acc[5] += b.y, acc[6] += b.z, acc[7] += b.w;
        }
        y[i] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                          pack_bf16x2(acc[6], acc[7]));
    }
}

}  // namespace

cudaError_t launch_splitk_reduce(const float* ws, int slices, int64_t elems, uint16_t* y, int sm_count, bool overlap,
                                 cudaStream_t stream) {
    const int64_t groups = elems / 8;
    if (groups == 0) return cudaSuccess;
    const int64_t blocks = (groups + SK_THREADS - 1) / SK_THREADS;
    const int64_t cap = static_cast<int64_t>(sm_count) * 4;
    const int grid = static_cast<int>(blocks < cap ? blocks : cap);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(SK_THREADS);
    cfg.stream = stream;
    if (overlap) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, nf_splitk_reduce_kernel, reinterpret_cast<const float4*>(ws), slices, groups,
                              reinterpret_cast<uint4*>(y));
}

}  // namespace nf
