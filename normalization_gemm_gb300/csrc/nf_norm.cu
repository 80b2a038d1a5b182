// nf_norm.cu -- standalone LayerNorm / RMSNorm over rows: the separate,
// memory-bound normalization kernel of the unfused baseline (blog "Towards
// Free Normalization: Fusing Normalization into GEMM and Attention Kernels",
// §1: a GEMM followed by its own norm kernel, each row read and written once).
//
// Design: the kernel is HBM-bound, so it is built around 16-byte vector
// accesses and enough bytes in flight, not around tensor cores or TMA.
//   * A row of `cols` bf16 is 16-byte chunks; TPR threads (a power of two)
//     share a row, each holding CPT chunks (CPT * 8 values) in registers, so
//     the row is read from HBM exactly once and written once.
//   * Bytes in flight: the next row block's chunks are loaded (raw, 4
//     registers a chunk) before the current block is reduced, and gamma /
//     beta are read through the read-only cache where they are used rather
//     than held in registers, so four CTAs fit on an SM for rows of up to
//     4096 columns.
//   * Reductions: xor-shuffles inside a warp; for TPR > 32 a second step
//     through shared memory across the row's warps.
//   * LayerNorm takes two passes over the registers (mean, then squared
//     deviations), with biased variance and eps inside the root, as
//     torch.nn.LayerNorm; RMSNorm takes one.
//   * The grid is persistent (a multiple of the SM count); every CTA walks
//     blocks of rows so all its threads take the same trip count.
#include "nf_internal.h"
#include "nf_ptx.cuh"

namespace nf {

namespace {

constexpr int NORM_THREADS = 256;

__device__ __forceinline__ void unpack8(const uint4 q, float (&v)[8]) {
    v[0] = bf16lo(q.x); v[1] = bf16hi(q.x);
    v[2] = bf16lo(q.y); v[3] = bf16hi(q.y);
    v[4] = bf16lo(q.z); v[5] = bf16hi(q.z);
    v[6] = bf16lo(q.w); v[7] = bf16hi(q.w);
}

// Sum over the TPR threads of a row group (groups are aligned, TPR a power of 2).
template <int TPR>
__device__ __forceinline__ float group_sum(float x, float* red, int warp, int lane) {
    constexpr int W = TPR < 32 ? TPR : 32;
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if constexpr (TPR > 32) {
        constexpr int WPR = TPR / 32;  // warps per row
        if (lane == 0) red[warp] = x;
        __syncthreads();
        const int w0 = (warp / WPR) * WPR;
        float t = 0.0f;
#pragma unroll
        for (int i = 0; i < WPR; ++i) t += red[w0 + i];
        __syncthreads();
        x = t;
    }
    return x;
}

// This thread's CPT 16-byte chunks (t, t + TPR, ...) of `row`, raw; zeros
// past the row's end or for a row past the last.
template <int TPR, int CPT, bool STREAM>
__device__ __forceinline__ void load_row_chunks(const uint4* base, int64_t row, bool live, int t, int chunks,
                                                uint4 (&q)[CPT]) {
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int c = t + i * TPR;
        if (live && c < chunks)
            q[i] = STREAM ? __ldcs(base + row * chunks + c) : __ldcg(base + row * chunks + c);
        else
            q[i] = make_uint4(0u, 0u, 0u, 0u);
    }
}

// Occupancy target: 4 CTAs of 256 threads per SM (64 registers a thread)
// for the plain forward with rows of up to four chunks a thread, 2 for the
// residual forward and the backward (two tensors' chunks in flight), half
// that for rows of eight chunks a thread.  Bytes in flight come from the
// occupancy and from loading the next row block before reducing the current
// one.
template <int CPT, bool HEAVY>
struct NormOcc {
    static constexpr int MIN_BLOCKS = (HEAVY ? 2 : 4) / (CPT > 4 ? 2 : 1);
};

// Value e (0..7) of a chunk of 8 packed bf16.
__device__ __forceinline__ float chunk_val(const uint4& q, int e) {
    const uint32_t w = (e >> 1) == 0 ? q.x : (e >> 1) == 1 ? q.y : (e >> 1) == 2 ? q.z : q.w;
    return (e & 1) ? bf16hi(w) : bf16lo(w);
}

template <int TPR, int CPT, int KIND, bool RES>
__global__ void __launch_bounds__(NORM_THREADS, (NormOcc<CPT, RES>::MIN_BLOCKS)) nf_norm_rows_kernel(const NormArgs a) {
    constexpr int RPB = NORM_THREADS / TPR;  // rows per block-step
    __shared__ float red[NORM_THREADS / 32];
    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int lane = static_cast<int>(threadIdx.x & 31);
    const int t = static_cast<int>(threadIdx.x) % TPR;
    const int rg = static_cast<int>(threadIdx.x) / TPR;
    const int chunks = a.cols >> 3;
    const uint4* in = reinterpret_cast<const uint4*>(a.in);
    const uint4* res = reinterpret_cast<const uint4*>(a.res);
    uint4* out = reinterpret_cast<uint4*>(a.out);
    uint4* hout = reinterpret_cast<uint4*>(a.h_out);
    const uint4* gam = reinterpret_cast<const uint4*>(a.gamma);
    const uint4* bet = reinterpret_cast<const uint4*>(a.beta);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * RPB;
    // Warm L2 with this CTA's first two row blocks while a preceding grid may
    // still be running (a prefetch only fills L2, where that grid's writes
    // land, so the loads after the wait below never see stale data).
    if (threadIdx.x == 0) {
        for (int it = 0; it < 2; ++it) {
            const int64_t r = static_cast<int64_t>(blockIdx.x) * RPB + it * stride;
            if (r < a.rows) {
                const int64_t nr = a.rows - r < RPB ? a.rows - r : RPB;
                bulk_prefetch_l2(in + r * chunks, static_cast<uint32_t>(nr * chunks * 16));
            }
        }
    }
    griddep_wait();  // inputs may come from the kernel launched just before
    griddep_launch_dependents();

    int64_t r0 = static_cast<int64_t>(blockIdx.x) * RPB;
    // The plain forward keeps its chunks packed (the row block being reduced
    // in `cur`, the next one loading into `q`) and widens values where they
    // are used; the residual forward keeps the fp32 sum in v.
    uint4 q[CPT], qr[RES ? CPT : 1], cur[CPT];
    load_row_chunks<TPR, CPT, true>(in, r0 + rg, r0 + rg < a.rows, t, chunks, q);
    if constexpr (RES) load_row_chunks<TPR, CPT, false>(res, r0 + rg, r0 + rg < a.rows, t, chunks, qr);
    for (; r0 < a.rows; r0 += stride) {
        const int64_t row = r0 + rg;
        const bool live = row < a.rows;
        float v[RES ? CPT : 1][8];
#pragma unroll
        for (int i = 0; i < CPT; ++i) cur[i] = q[i];
        if constexpr (RES) {
            // Residual add before the norm; the sum (rounded to bf16) is the
            // updated residual stream.  The row's chunks of res were read
            // before this thread writes the same chunks of h_out, so h_out
            // may be res.
#pragma unroll
            for (int i = 0; i < CPT; ++i) {
                const int c = t + i * TPR;
                unpack8(cur[i], v[i]);
                float r[8];
                unpack8(qr[i], r);
#pragma unroll
                for (int e = 0; e < 8; ++e) v[i][e] += r[e];
                if (hout != nullptr && live && c < chunks)
                    __stcs(hout + row * chunks + c,
                           make_uint4(pack_bf16x2(v[i][0], v[i][1]), pack_bf16x2(v[i][2], v[i][3]),
                                      pack_bf16x2(v[i][4], v[i][5]), pack_bf16x2(v[i][6], v[i][7])));
            }
        }
        auto val = [&](int i, int e) -> float {
            if constexpr (RES) return v[i][e];
            else return chunk_val(cur[i], e);
        };
        // The next row block's loads go out before this block's reductions.
        {
            const int64_t nrow = row + stride;
            load_row_chunks<TPR, CPT, true>(in, nrow, nrow < a.rows, t, chunks, q);
            if constexpr (RES) load_row_chunks<TPR, CPT, false>(res, nrow, nrow < a.rows, t, chunks, qr);
        }
        float mean = 0.0f, rstd;
        if (KIND == 0) {
            float s = 0.0f;
#pragma unroll
            for (int i = 0; i < CPT; ++i)
#pragma unroll
                for (int e = 0; e < 8; ++e) s += val(i, e);
            mean = group_sum<TPR>(s, red, warp, lane) * a.inv_cols;
            float d2 = 0.0f;
#pragma unroll
            for (int i = 0; i < CPT; ++i) {
                const bool in_row = (t + i * TPR) < chunks;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float d = val(i, e) - mean;
                    d2 += in_row ? d * d : 0.0f;
                }
            }
            rstd = rsqrtf(fmaf(group_sum<TPR>(d2, red, warp, lane), a.inv_cols, a.eps));
        } else {
            float s = 0.0f;
#pragma unroll
            for (int i = 0; i < CPT; ++i)
#pragma unroll
                for (int e = 0; e < 8; ++e) s = fmaf(val(i, e), val(i, e), s);
            rstd = rsqrtf(fmaf(group_sum<TPR>(s, red, warp, lane), a.inv_cols, a.eps));
        }
        if (!live) continue;
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const int c = t + i * TPR;
            if (c < chunks) {
                // gamma / beta through the read-only cache (every row reuses them)
                float g[8], b[8];
                if (gam != nullptr) {
                    unpack8(__ldg(gam + c), g);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) g[e] = 1.0f;
                }
                if (KIND == 0 && bet != nullptr) {
                    unpack8(__ldg(bet + c), b);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) b[e] = 0.0f;
                }
                float y[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] = fmaf((val(i, e) - mean) * rstd, g[e], b[e]);
                uint4 o;
                o.x = pack_bf16x2(y[0], y[1]);
                o.y = pack_bf16x2(y[2], y[3]);
                o.z = pack_bf16x2(y[4], y[5]);
                o.w = pack_bf16x2(y[6], y[7]);
                __stcs(out + row * chunks + c, o);
            }
        }
        if (t == 0) {
            if (KIND == 0 && a.mean_out) a.mean_out[row] = mean;
            if (a.rstd_out) a.rstd_out[row] = rstd;
        }
    }
}

// Backward of the row normalization from the forward's saved statistics
// (blog "Towards Free Normalization: ...", §3 "What about backward?"; the
// unfused kernel the fused backward is compared with):
//   g = dY * gamma; xhat = (Z - mean) * rstd (LN) or Z * rstd (RMS);
//   dZ = rstd * (g - mean(g) - xhat * mean(g * xhat)), mean(g) for LN only.
// Same layout as the forward kernel: TPR threads per row, CPT 16-byte chunks
// of dY and of Z per thread in registers (the next row block's loaded ahead),
// each row read and written once.
template <int TPR, int CPT, int KIND>
__global__ void __launch_bounds__(NORM_THREADS, (NormOcc<CPT, true>::MIN_BLOCKS)) nf_norm_rows_bwd_kernel(const NormBwdArgs a) {
    constexpr int RPB = NORM_THREADS / TPR;
    __shared__ float red[NORM_THREADS / 32];
    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int lane = static_cast<int>(threadIdx.x & 31);
    const int t = static_cast<int>(threadIdx.x) % TPR;
    const int rg = static_cast<int>(threadIdx.x) / TPR;
    const int chunks = a.cols >> 3;
    const uint4* dyp = reinterpret_cast<const uint4*>(a.dy);
    const uint4* zp = reinterpret_cast<const uint4*>(a.z);
    const uint4* gam = reinterpret_cast<const uint4*>(a.gamma);
    uint4* out = reinterpret_cast<uint4*>(a.dz);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * RPB;
    // Warm L2 with the first row block of dY and Z (see the forward kernel).
    if (threadIdx.x == 0) {
        const int64_t r = static_cast<int64_t>(blockIdx.x) * RPB;
        if (r < a.rows) {
            const int64_t nr = a.rows - r < RPB ? a.rows - r : RPB;
            bulk_prefetch_l2(dyp + r * chunks, static_cast<uint32_t>(nr * chunks * 16));
            bulk_prefetch_l2(zp + r * chunks, static_cast<uint32_t>(nr * chunks * 16));
        }
    }
    griddep_wait();  // inputs may come from the kernel launched just before
    griddep_launch_dependents();

    int64_t r0 = static_cast<int64_t>(blockIdx.x) * RPB;
    uint4 qy[CPT], qz[CPT];
    load_row_chunks<TPR, CPT, true>(dyp, r0 + rg, r0 + rg < a.rows, t, chunks, qy);
    load_row_chunks<TPR, CPT, true>(zp, r0 + rg, r0 + rg < a.rows, t, chunks, qz);
    for (; r0 < a.rows; r0 += stride) {
        const int64_t row = r0 + rg;
        const bool live = row < a.rows;
        float gy[CPT][8], xh[CPT][8];
        const float mu = (KIND == 0 && live) ? a.mean[row] : 0.0f;
        const float rs = live ? a.rstd[row] : 0.0f;
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            unpack8(qy[i], gy[i]);
            unpack8(qz[i], xh[i]);
        }
        {  // the next row block's loads go out before this block's reductions
            const int64_t nrow = row + stride;
            load_row_chunks<TPR, CPT, true>(dyp, nrow, nrow < a.rows, t, chunks, qy);
            load_row_chunks<TPR, CPT, true>(zp, nrow, nrow < a.rows, t, chunks, qz);
        }
        float s1 = 0.0f, s2 = 0.0f;
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const int c = t + i * TPR;
            float g[8];
            if (gam != nullptr && c < chunks) {
                unpack8(__ldg(gam + c), g);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) g[e] = 1.0f;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                gy[i][e] *= g[e];                                      // g = dY * gamma
                xh[i][e] = (KIND == 0 ? xh[i][e] - mu : xh[i][e]) * rs;  // xhat
                s1 += gy[i][e];
                s2 = fmaf(gy[i][e], xh[i][e], s2);
            }
        }
        const float mg = KIND == 0 ? group_sum<TPR>(s1, red, warp, lane) * a.inv_cols : 0.0f;
        const float mgx = group_sum<TPR>(s2, red, warp, lane) * a.inv_cols;
        if (!live) continue;
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const int c = t + i * TPR;
            if (c < chunks) {
                float y[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] = rs * (gy[i][e] - mg - xh[i][e] * mgx);
                uint4 o;
                o.x = pack_bf16x2(y[0], y[1]);
                o.y = pack_bf16x2(y[2], y[3]);
                o.z = pack_bf16x2(y[4], y[5]);
                o.w = pack_bf16x2(y[6], y[7]);
                __stcs(out + row * chunks + c, o);
            }
        }
    }
}

template <int TPR, int CPT, int KIND>
cudaError_t launch_one(const NormArgs& a, int sm_count, bool overlap, cudaStream_t stream) {
    auto kern = a.res != nullptr ? nf_norm_rows_kernel<TPR, CPT, KIND, true> : nf_norm_rows_kernel<TPR, CPT, KIND, false>;
    constexpr int RPB = NORM_THREADS / TPR;
    static int per_sm[2] = {0, 0};  // occupancy of this variant (without, with residual), queried once
    int& occ = per_sm[a.res != nullptr ? 1 : 0];
    if (occ == 0) {
        int n = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, NORM_THREADS, 0);
        if (e != cudaSuccess) return e;
        occ = n < 1 ? 1 : n;
    }
    const int64_t steps = (a.rows + RPB - 1) / RPB;
    const int64_t cap = static_cast<int64_t>(sm_count) * occ;
    const int grid = static_cast<int>(steps < cap ? steps : cap);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(NORM_THREADS);
    cfg.stream = stream;
    if (overlap) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int KIND>
cudaError_t dispatch(const NormArgs& a, int sm_count, bool overlap, cudaStream_t stream) {
    const int chunks = a.cols >> 3;
    // TPR: the smallest power of two with TPR * 4 >= chunks (at most 256).
    if (chunks <= 4) return launch_one<1, 4, KIND>(a, sm_count, overlap, stream);
    if (chunks <= 8) return launch_one<2, 4, KIND>(a, sm_count, overlap, stream);
    if (chunks <= 16) return launch_one<4, 4, KIND>(a, sm_count, overlap, stream);
    if (chunks <= 32) return launch_one<8, 4, KIND>(a, sm_count, overlap, stream);
    if (chunks <= 64) return launch_one<16, 4, KIND>(a, sm_count, overlap, stream);
    if (chunks <= 128) return launch_one<32, 4, KIND>(a, sm_count, overlap, stream);
    if (chunks <= 256) return launch_one<64, 4, KIND>(a, sm_count, overlap, stream);
    if (chunks <= 512) return launch_one<128, 4, KIND>(a, sm_count, overlap, stream);
    if (chunks <= 1024) return launch_one<256, 4, KIND>(a, sm_count, overlap, stream);
    return launch_one<256, 8, KIND>(a, sm_count, overlap, stream);  // cols <= 16384
}

template <int TPR, int CPT, int KIND>
cudaError_t launch_one_bwd(const NormBwdArgs& a, int sm_count, bool overlap, cudaStream_t stream) {
    auto kern = nf_norm_rows_bwd_kernel<TPR, CPT, KIND>;
    constexpr int RPB = NORM_THREADS / TPR;
    static int per_sm = 0;  // occupancy of this variant, queried once
    if (per_sm == 0) {
        int n = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, NORM_THREADS, 0);
        if (e != cudaSuccess) return e;
        per_sm = n < 1 ? 1 : n;
    }
    const int64_t steps = (a.rows + RPB - 1) / RPB;
    const int64_t cap = static_cast<int64_t>(sm_count) * per_sm;
    const int grid = static_cast<int>(steps < cap ? steps : cap);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(NORM_THREADS);
    cfg.stream = stream;
    if (overlap) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int KIND>
cudaError_t dispatch_bwd(const NormBwdArgs& a, int sm_count, bool overlap, cudaStream_t stream) {
    const int chunks = a.cols >> 3;
    if (chunks <= 4) return launch_one_bwd<1, 4, KIND>(a, sm_count, overlap, stream);
    if (chunks <= 8) return launch_one_bwd<2, 4, KIND>(a, sm_count, overlap, stream);
    if (chunks <= 16) return launch_one_bwd<4, 4, KIND>(a, sm_count, overlap, stream);
    if (chunks <= 32) return launch_one_bwd<8, 4, KIND>(a, sm_count, overlap, stream);
    if (chunks <= 64) return launch_one_bwd<16, 4, KIND>(a, sm_count, overlap, stream);
    if (chunks <= 128) return launch_one_bwd<32, 4, KIND>(a, sm_count, overlap, stream);
    if (chunks <= 256) return launch_one_bwd<64, 4, KIND>(a, sm_count, overlap, stream);
    if (chunks <= 512) return launch_one_bwd<128, 4, KIND>(a, sm_count, overlap, stream);
    if (chunks <= 1024) return launch_one_bwd<256, 4, KIND>(a, sm_count, overlap, stream);
    return launch_one_bwd<256, 8, KIND>(a, sm_count, overlap, stream);  // cols <= 16384
}

}  // namespace

cudaError_t launch_norm_rows(const NormArgs& a, int kind, int sm_count, bool overlap, cudaStream_t stream) {
    return kind == 0 ? dispatch<0>(a, sm_count, overlap, stream) : dispatch<1>(a, sm_count, overlap, stream);
}

cudaError_t launch_norm_rows_bwd(const NormBwdArgs& a, int kind, int sm_count, bool overlap,
                                 cudaStream_t stream) {
    return kind == 0 ? dispatch_bwd<0>(a, sm_count, overlap, stream)
                     : dispatch_bwd<1>(a, sm_count, overlap, stream);
}

}  // namespace nf
