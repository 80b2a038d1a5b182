// nf_splitk.cu -- second half of a split-K GEMM: adds the fp32 partial
// products of the contraction slices, in slice order, and writes the split
// tiles of Y in bf16.
//
// A plain GEMM splits tiles over the contraction in two cases: when it has
// few output tiles and a long contraction (the weight gradient of the Lazy
// Pre-Norm backward, K x N over M, is the case in point), every tile is split
// so that each SM holds one (tile, slice) unit; when a tensor-bound GEMM's
// last wave is at most half full, only that wave's tiles are split, so it
// takes a fraction of a tile's time.  Each split unit stores its fp32 partial
// tile into plane s of the workspace, tile-major; at most one wave of
// 128 x 256 fp32 tiles, i.e. L2-resident when this kernel reads them back.
// The order of the additions is fixed, so the result does not depend on the
// order in which the units finished.
#include "nf_internal.h"
#include "nf_ptx.cuh"

namespace nf {
namespace {

constexpr int SK_THREADS = 256;

// Thread i handles 8 consecutive columns of one row of one split tile: two
// float4 per plane, one uint4 out.
__global__ void __launch_bounds__(SK_THREADS) nf_splitk_reduce_kernel(const SplitkReduceArgs a) {
    griddep_wait();  // the partials come from the GEMM launched just before
    griddep_launch_dependents();
    const int gpr = a.tile_n / 8;                                   // 8-column groups per tile row
    const int64_t per_tile = static_cast<int64_t>(TILE_M) * gpr;    // groups per tile
    const int64_t groups = per_tile * a.sk_tiles;
    const int64_t plane = static_cast<int64_t>(a.sk_tiles) * TILE_M * a.tile_n / 4;  // float4 per plane
    const float4* ws = reinterpret_cast<const float4*>(a.ws);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < groups; i += stride) {
        const int tl = static_cast<int>(i / per_tile);
        const int rem = static_cast<int>(i - static_cast<int64_t>(tl) * per_tile);
        const int r = rem / gpr, c8 = rem - r * gpr;
        const int t = a.sk_base + tl;
        const int m = t / a.n_tiles, n = t - m * a.n_tiles;
        const int64_t grow = static_cast<int64_t>(m) * TILE_M + r;
        const int gcol = n * a.tile_n + c8 * 8;
        if (grow >= a.M || gcol >= a.N) continue;
        float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
        const float4* p = ws + ((static_cast<int64_t>(tl) * TILE_M + r) * a.tile_n + c8 * 8) / 4;
        for (int s = 0; s < a.slices; ++s, p += plane) {
            const float4 u = __ldcg(p), v = __ldcg(p + 1);
            acc[0] += u.x, acc[1] += u.y, acc[2] += u.z, acc[3] += u.w;
            acc[4] += v.x, acc[5] += v.y, acc[6] += v.z, acc[7] += v.w;
        }
        *reinterpret_cast<uint4*>(a.y + grow * a.N + gcol) =
            make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                       pack_bf16x2(acc[6], acc[7]));
    }
}

}  // namespace

cudaError_t launch_splitk_reduce(const SplitkReduceArgs& a, int sm_count, bool overlap, cudaStream_t stream) {
    const int64_t groups = static_cast<int64_t>(a.sk_tiles) * TILE_M * (a.tile_n / 8);
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
    return cudaLaunchKernelEx(&cfg, nf_splitk_reduce_kernel, a);
}

}  // namespace nf
