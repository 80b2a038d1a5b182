// nf_api.cu -- the C ABI declared in include/nf.h: argument validation, tensor
// maps, launch plans, launches, and the device status word.
//
// Blog: "Towards Free Normalization: Fusing Normalization into GEMM and
// Attention Kernels" -- §1 (unfused GEMM + norm baseline), §2 (Lazy Pre-Norm),
// §3 (Multi-CTA post-norm over a thread-block cluster).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "nf.h"
#include "nf_internal.h"
#include "nf_ptx.cuh"

namespace nf {
namespace {

// ---------------------------------------------------------------- errors
thread_local std::string g_last_error;

nf_status fail(nf_status s, const char* what) {
    g_last_error = what;
    return s;
}

nf_status fail_cuda(cudaError_t e, const char* what) {
    g_last_error = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
    return NF_ERR_CUDA;
}

// ---------------------------------------------------------------- device status
// Four words per the WaitGuard layout: code, wait site, block, tile.
__device__ uint32_t g_status_word[4];

__global__ void nf_selftest_wait_kernel(uint32_t* status, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // Nothing ever arrives on `bar`: the wait must give up after timeout_ns.
        const WaitGuard g{status, &abort_flag, timeout_ns};
        (void)mbar_wait(g, b, 0, SITE_SELFTEST, 0);
    }
    __syncthreads();
}

uint64_t g_timeout_ns = 2000000000ull;
// Programmatic dependent launch: a kernel's prologue may overlap the tail of
// the kernel before it on the stream (it waits in griddepcontrol.wait before
// touching global memory).
bool g_overlap = true;
// Post-norm column tile per CTA of a cluster: 0 = automatic, 256 or 512 forced.
int g_post_tile = 0;
// Column tile of plain and pre-norm GEMMs: 0 = automatic, 64, 128 or 256 forced.
int g_gemm_tile = 0;
// CTA pairs (cta_group::2) for plain and pre-norm GEMMs: 0 = automatic
// (tensor-bound shapes of 256-column tiles), 1 = never, 2 = whenever the
// tile allows.
int g_pair_mode = 0;
// Post-norm rows wider than 256 columns: 0 = automatic, else an Exchange mode.
int g_post_xch = 0;
// Lazy Pre-Norm row sums of squares split over a row's tiles: 0 = automatic
// (tensor-bound tiles), 1 = never, 2 = whenever the shape allows.
int g_pre_split = 0;
// A cooperative launch accepted the programmatic-serialization attribute.
bool g_coop_overlap_ok = true;
// A cooperative launch of clusters (CTA pairs with the L2 exchange) was accepted.
bool g_coop_cluster_ok = true;
// Split-K of plain GEMMs: 0 = automatic, 1 = never.
int g_splitk_mode = 0;
std::mutex g_mu;

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    int sm_count = 0;
    uint32_t* status = nullptr;
    // max co-resident clusters, per variant function and cluster size
    const void* occ_func[16] = {};
    int occ_cluster[16] = {};
    int occ_value[16] = {};
    int occ_n = 0;
    // kernels whose attributes were set on this device
    const void* attr_done[32] = {};
    int attr_n = 0;
    // resident CTAs per SM, per kernel (for cooperative grids)
    const void* blk_func[16] = {};
    int blk_value[16] = {};
    int blk_n = 0;
};
DeviceState g_dev[kMaxDevices];

// Global-exchange scratch, one buffer per (device, stream): launches on one
// stream run in order, so each buffer is used by one launch at a time.  The
// buffer holds the header and two counter banks of bank_ints each, then
// (256-byte aligned) stats_bytes of partial statistics.  A call that needs
// more replaces the stream's buffer with a larger one, allocated and cleared
// in stream order (cudaMallocAsync / cudaMemsetAsync: no host
// synchronization); the smaller one is kept for the life of the process,
// since a graph captured earlier may still use it.
struct XScratch {
    int dev = -1;
    cudaStream_t stream = nullptr;
    uint8_t* ptr = nullptr;
    size_t bytes = 0;
    int64_t bank_ints = 0;
    int64_t stats_bytes = 0;
    int64_t tag_bytes = 0;  // the pre-norm's tagged row sums (written by no other kernel)
    int* cnt() const { return reinterpret_cast<int*>(ptr); }
    unsigned long long* stats() const {
        return reinterpret_cast<unsigned long long*>(ptr + stats_offset(bank_ints));
    }
    unsigned long long* tags() const {
        return reinterpret_cast<unsigned long long*>(ptr + stats_offset(bank_ints) + stats_bytes);
    }
    static int64_t stats_offset(int64_t bank_ints) { return ((XCH_CNT0 + 2 * bank_ints) * 4 + 255) / 256 * 256; }
};
constexpr int kMaxScratch = 64;

// Fixed exchange scratch of nf_gemm_postnorm_ln_noalloc: a file-scope device
// array (header, two counter banks, partial statistics), so that entry point
// allocates nothing at any time.  Zero when set up on a device.
constexpr int64_t kNoAllocBankInts = 16384;      // 4 counters per row tile: m_tiles <= 4096
constexpr int64_t kNoAllocStatsBytes = 8 << 20;  // m_tiles * n_tiles <= 4096 (binds first: n_tiles >= 3)
constexpr int64_t kNoAllocStatsOffset = (XCH_CNT0 + 2 * kNoAllocBankInts) * 4;
constexpr int64_t kNoAllocBytes = kNoAllocStatsOffset + kNoAllocStatsBytes;
static_assert(kNoAllocStatsOffset % 256 == 0, "statistics region alignment");
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocBytes];
uint8_t* g_noalloc_ptr[64] = {};
XScratch g_xs[kMaxScratch];
int g_xs_n = 0;

nf_status device_state(DeviceState** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(NF_ERR_NO_DEVICE, "device index out of range");
    DeviceState& d = g_dev[dev];
    if (!d.ready) {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!d.ready) {
            int major = 0, minor = 0, sms = 0;
            if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
                return fail_cuda(e, "cudaDeviceGetAttribute");
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (major != 10 || minor != 3)
                return fail(NF_ERR_NO_DEVICE, "the kernels are built for sm_103a only");
            void* p = nullptr;
            if ((e = cudaGetSymbolAddress(&p, g_status_word)) != cudaSuccess)
                return fail_cuda(e, "cudaGetSymbolAddress(status)");
            d.status = static_cast<uint32_t*>(p);
            d.sm_count = sms;
            d.ready = true;
        }
    }
    *out = &d;
    return NF_OK;
}

// ---------------------------------------------------------------- tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Row-major bf16 matrix of `rows` x `cols` (row pitch cols * 2 bytes), read or
// written in boxes of box_rows x box_cols with 128-byte swizzle; out-of-bounds
// elements read as zero and are dropped on store.
nf_status make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_cols, int box_rows,
                   CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return fail(NF_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2u};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char msg[128];
        snprintf(msg, sizeof msg, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
        return fail(NF_ERR_CUDA, msg);
    }
    return NF_OK;
}

// ---------------------------------------------------------------- plans
enum Op { OP_PLAIN = 0, OP_PRE = 1, OP_POST_LN = 2, OP_POST_RMS = 3, OP_BWD_LN = 4, OP_BWD_RMS = 5 };

struct Plan {
    bool pair = false;  // CTA pair along M (cta_group::2), cluster of 2
    int splitk = 1;  // contraction slices of the split tiles (plain GEMM)
    int sk_base = 0, sk_tiles = 0;  // split-K: first split tile, split tiles
    int tile_n = 0;
    int xch = XCH_NONE;
    bool clustered = false;
    int cluster = 1;
    int m_tiles = 0, n_tiles = 0, k_tiles = 0;
    const GemmVariant* v = nullptr;
};

const GemmVariant* find_variant(int op, int tile_n, int xch, int ops = 0) {
    int n = 0;
    const GemmVariant* t = nullptr;
    if (ops != 0 && ops != OPS_PAIR) {
        if (op == OP_PLAIN) t = gemm_variants_trans_plain(&n);
        else if (op == OP_BWD_RMS) t = gemm_variants_trans_bwd(&n);
        else if (op == OP_POST_LN && ops == OPS_RESID) t = gemm_variants_res_ln(&n);
        else if (op == OP_POST_RMS && ops == OPS_RESID) t = gemm_variants_res_rms(&n);
        else return nullptr;
    } else switch (op) {
        case OP_PLAIN: t = gemm_variants_plain(&n); break;
        case OP_PRE: t = gemm_variants_pre(&n); break;
        case OP_POST_LN: t = gemm_variants_post_ln(&n); break;
        case OP_POST_RMS: t = gemm_variants_post_rms(&n); break;
        case OP_BWD_LN: t = gemm_variants_bwd_ln(&n); break;
        case OP_BWD_RMS: t = gemm_variants_bwd_rms(&n); break;
        default: return nullptr;
    }
    for (int i = 0; i < n; ++i)
        if (t[i].tile_n == tile_n && t[i].xch == xch && t[i].ops == ops) return &t[i];
    return nullptr;
}

// Whether a tile's share of HBM traffic takes longer than its MMA: its X rows
// (128 x K, read once per row tile and shared by the row's n_tiles CTAs) and
// its Y (128 x tile_n) against 2 * 128 * tile_n * K flops, at GB300's ratio of
// tensor throughput to HBM bandwidth (about 290 flop per byte).
bool tile_memory_bound(int64_t K, int tile_n, int n_tiles) {
    const double bytes = static_cast<double>(TILE_M) * K * 2 / n_tiles + static_cast<double>(TILE_M) * tile_n * 2;
    const double flops = 2.0 * TILE_M * tile_n * static_cast<double>(K);
    return flops < 290.0 * bytes;
}

// Tile choice.  Plain and pre-norm: the smallest of 64 / 128 / 256 columns
// that covers N, else 256.  Post-norm (blog §3): one CTA holds whole rows
// while N <= 256 (and, with 512 columns per CTA, while N <= 512).  Wider rows
// are split over CTAs that exchange partial row statistics:
//   through L2 between 256-column tiles of a cooperative grid that keeps
//   every SM busy -- the automatic choice when K >= 512, where a tile's
//   main loop outlasts the exchange and the cluster's co-residency limits
//   (GB300 holds 15 clusters of 8, i.e. 120 of 152 SMs) cost the most;
//   or, as on the blog, through DSMEM inside a thread-block cluster, with
//   256 columns per CTA (automatic for K < 512 up to N = 2048, a cluster of
//   <= 8) or 512 (two N = 256 MMAs per K step, a cluster of <= 8 for
//   N <= 4096).
// `sms`: SMs of the device.  The global exchange runs one CTA per SM and
// needs at least half as many CTAs as a row has tiles; with fewer the row
// goes to a cluster instead.
// A residual add (post-norm) takes the 256-column kernels only.
// The normalization backward (ops 4, 5) follows the same choice with
// 256-column CTAs only (no 512-column variant): L2 exchange for K >= 512 and
// N > 512, else a cluster of <= 16 (of 2 for N <= 512, which fits every SM).
nf_status plan_tiles(int op, int64_t M, int64_t N, int64_t K, int sms, Plan* p, int ops = 0) {
    const bool resid = (ops & OPS_RESID) != 0;
    const bool post = op == OP_POST_LN || op == OP_POST_RMS;
    const bool bwd = op == OP_BWD_LN || op == OP_BWD_RMS;
    p->tile_n = N <= 64 ? 64 : (N <= 128 ? 128 : 256);
    if ((op == OP_PLAIN || op == OP_PRE) && ops == 0 && g_gemm_tile != 0) p->tile_n = g_gemm_tile;
    p->xch = XCH_NONE;
    if (bwd && N > 256) {
        // Rows of two tiles: a cluster of 2, which co-resides on every SM.
        int mode = g_post_xch ? g_post_xch : ((K >= 512 && N > 512) ? XCH_GLOBAL : XCH_CLUSTER);
        if (mode == XCH_GLOBAL) {
            const int64_t nt = (N + 255) / 256, tiles = ((M + TILE_M - 1) / TILE_M) * nt;
            if (2 * (tiles < sms ? tiles : sms) < nt) mode = XCH_CLUSTER;
        }
        p->xch = mode;
        if (N > 16 * 256) return fail(NF_ERR_UNSUPPORTED_SHAPE, "N too large for the cluster");
    }
    if (post && N > 256) {
        int mode = g_post_xch, tile = g_post_tile;
        if (mode == 0) {
            if (N <= 512)
                mode = XCH_CLUSTER, tile = tile ? tile : 512;  // one 512-column CTA: no exchange
            else if (K >= 512)
                mode = XCH_GLOBAL;
            else
                mode = XCH_CLUSTER, tile = tile ? tile : (N <= 2048 ? 256 : 512);
        }
        if (mode == XCH_GLOBAL) {
            const int64_t nt = (N + 255) / 256, tiles = ((M + TILE_M - 1) / TILE_M) * nt;
            if (2 * (tiles < sms ? tiles : sms) < nt) mode = XCH_CLUSTER;
        }
        p->xch = mode;
        if (mode == XCH_CLUSTER) {
            p->tile_n = (tile == 256 || resid) ? 256 : 512;  // the 512-column kernel adds no residual
            if (N > static_cast<int64_t>(p->tile_n) * (p->tile_n == 512 ? 8 : 16))
                return fail(NF_ERR_UNSUPPORTED_SHAPE, "N too large for the cluster");
            if (N <= p->tile_n) p->xch = XCH_NONE;  // one wide CTA covers the row
        }
    }
    // Lazy Pre-Norm with 2..32 tiles of 256 columns a row: each tile sums the
    // squares of 1/n_tiles of the rows, and the row tile's tiles gather them
    // through L2 (the kernel's split sums of squares), instead of every tile
    // summing every row from its shared-memory stages -- on tensor-bound
    // tiles those reads take shared-memory bandwidth from the MMA (measured at
    // 8192 x 4096 x 4096 in CTA pairs: 159 us with every tile summing every
    // row, 143 us without the reads).  The gather needs the cooperative
    // persistent grid of the post-norm L2 exchange; <= 32 tiles a row keeps
    // 2 x resident CTAs (or pairs) >= n_tiles.  Automatic for tensor-bound
    // tiles with K >= 2048: memory-bound tiles keep the plain form (their last
    // wave is cut into 64-row units instead), and with a shorter contraction
    // the gather's latency and the cooperative launch cost about what the
    // shared reads saved (16384 x 1024 x 2048: 50.4 us split, 49.6 us not).
    if (op == OP_PRE && ops == 0 && p->tile_n == 256 && g_pre_split != 1) {
        const int64_t nt = (N + 255) / 256;
        if (nt >= 2 && nt <= 32 &&
            (g_pre_split == 2 || (K >= 2048 && !tile_memory_bound(K, 256, static_cast<int>(nt)))))
            p->xch = XCH_GLOBAL;
    }
    p->clustered = p->xch == XCH_CLUSTER;
    p->cluster = p->clustered ? static_cast<int>((N + p->tile_n - 1) / p->tile_n) : 1;
    p->m_tiles = static_cast<int>((M + TILE_M - 1) / TILE_M);
    p->n_tiles = ((post || bwd) && p->xch != XCH_GLOBAL) ? 1 : static_cast<int>((N + p->tile_n - 1) / p->tile_n);
    // CTA pair: two CTAs along M share each 256 x 256 tile's B (cta_group::2
    // MMAs), halving each CTA's B traffic and stage size, for tensor-bound
    // plain and pre-norm GEMMs of 256-column tiles -- unless a plain GEMM has
    // so few tiles that every one is split over the contraction (below).
    // Post-norm rows exchanged through L2 take pairs too (the exchange is
    // per 128-row tile, whichever CTA computes it).
    const int64_t tiles_all = static_cast<int64_t>(p->m_tiles) * p->n_tiles;
    const bool pair_op = ((op == OP_PLAIN || op == OP_PRE) && ops == 0) ||
                         (post && p->xch == XCH_GLOBAL && ops == 0);
    // (Automatic plans pair pre-norm GEMMs only with the split sums of
    // squares: with every tile summing every row, measured no faster in pairs.
    // Post-norm tiles of a shorter contraction are bound by their epilogue,
    // which a pair's two CTAs both wait for: K >= 2048.)
    p->pair = pair_op && p->tile_n == 256 && p->m_tiles >= 2 &&
              (g_pair_mode == 2 ||
               (g_pair_mode == 0 && (op != OP_PRE || p->xch == XCH_GLOBAL) &&
                !tile_memory_bound(K, p->tile_n, p->n_tiles) &&
                (!post || K >= 2048) &&
                !(op == OP_PLAIN && g_splitk_mode != 1 && 2 * tiles_all <= sms && (K + TILE_K - 1) / TILE_K >= 16)));
    if (p->pair) {
        ops = OPS_PAIR;
        p->cluster = 2;
    }
    p->v = find_variant(op, p->tile_n, p->xch, ops);
    if (!p->v) return fail(NF_ERR_UNSUPPORTED_SHAPE, "no kernel variant for this shape");
    p->k_tiles = static_cast<int>((K + p->v->tile_k - 1) / p->v->tile_k);
    // Split-K (plain GEMM), slices of >= 8 K-tiles, fp32 partials added by a
    // second kernel:
    //   * at most half as many output tiles as SMs: every tile is split, so
    //     that tiles x slices fills the SMs once;
    //   * tensor-bound tiles whose last, partial wave holds at most half the
    //     SMs: only that wave's tiles are split, so it takes a fraction of a
    //     tile's time instead of a whole one while most SMs idle.  (Memory-bound
    //     tiles cut that wave into 64-row halves instead, split_last_wave.)
    p->splitk = 1;
    p->sk_base = p->sk_tiles = 0;
    if (op == OP_PLAIN && g_splitk_mode != 1 && !p->pair) {
        const int tiles = p->m_tiles * p->n_tiles;
        const int kmax = p->k_tiles / 8;
        if (2 * tiles <= sms) {
            const int s = sms / tiles < kmax ? sms / tiles : kmax;
            if (s > 1) p->splitk = s, p->sk_tiles = tiles;
        } else if (!tile_memory_bound(K, p->tile_n, p->n_tiles)) {
            const int full = (tiles / sms) * sms, rest = tiles - full;
            const int s = rest > 0 ? (sms / rest < kmax ? sms / rest : kmax) : 0;
            if (rest > 0 && 2 * rest <= sms && s > 1) p->splitk = s, p->sk_base = full, p->sk_tiles = rest;
        }
    }
    return NF_OK;
}

// Memory-bound tiles whose last, partial wave holds at most half a wave of
// tiles: cut each of those tiles into two 64-row units so that the wave
// spreads over twice as many SMs.  (A half still runs the full MMA, so it
// gains only where the tile waits on memory; tensor-bound shapes keep whole
// tiles.)
void split_last_wave(int tiles, int grid, bool memory_bound, int32_t* units, int32_t* split_base) {
    *units = tiles;
    *split_base = tiles;
    if (!memory_bound || tiles <= grid) return;
    const int full = (tiles / grid) * grid;
    const int rest = tiles - full;
    if (rest > 0 && 2 * rest <= grid) {
        *split_base = full;
        *units = full + 2 * rest;
    }
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

nf_status check_gemm_args(int op, const void* X, const void* W, const void* Y, const void* gamma, const void* beta,
                          const float* mean_out, const float* rstd_out, int64_t M, int64_t N, int64_t K, float eps) {
    if (M < 0 || N < 1 || K < 1) return fail(NF_ERR_INVALID_ARG, "need M >= 0, N >= 1, K >= 1");
    // An empty X / Y (M == 0) may have a null base: nothing is ever accessed.
    if (M == 0) {
        X = X ? X : reinterpret_cast<const void*>(256);
        Y = Y ? Y : reinterpret_cast<const void*>(256);
    }
    if (!X || !W || !Y) return fail(NF_ERR_INVALID_ARG, "X, W and Y must be non-null");
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
        return fail(NF_ERR_UNSUPPORTED_SHAPE, "M, N and K must be below 2^31");
    if (op != OP_PLAIN && !(std::isfinite(eps) && eps >= 0.0f))
        return fail(NF_ERR_INVALID_ARG, "eps must be finite and >= 0");
    if (!aligned(X, 16) || !aligned(W, 16) || !aligned(Y, 16))
        return fail(NF_ERR_ALIGNMENT, "X, W and Y must be 16-byte aligned");
    if (K % 8 != 0 || N % 8 != 0)
        return fail(NF_ERR_ALIGNMENT, "K and N must be multiples of 8 (16-byte row pitch)");
    if ((gamma && !aligned(gamma, 2)) || (beta && !aligned(beta, 2)))
        return fail(NF_ERR_ALIGNMENT, "gamma and beta must be 2-byte aligned");
    if ((mean_out && !aligned(mean_out, 4)) || (rstd_out && !aligned(rstd_out, 4)))
        return fail(NF_ERR_ALIGNMENT, "mean_out and rstd_out must be 4-byte aligned");
    if (op >= OP_POST_LN && N > NF_POSTNORM_MAX_N)
        return fail(NF_ERR_UNSUPPORTED_SHAPE, "post-norm needs N <= 4096 (256 columns x 16-CTA cluster)");
    // Tile coordinates are int32: M rows plus one tile of slack.
    if (M > static_cast<int64_t>(INT32_MAX) - TILE_M) return fail(NF_ERR_UNSUPPORTED_SHAPE, "M too large");
    return NF_OK;
}

// Sets per-kernel attributes once per device.
nf_status prepare_kernel(DeviceState* d, const GemmVariant* v) {
    for (int i = 0; i < d->attr_n; ++i)
        if (d->attr_done[i] == v->func) return NF_OK;
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < d->attr_n; ++i)
        if (d->attr_done[i] == v->func) return NF_OK;
    cudaError_t e = cudaFuncSetAttribute(v->func, cudaFuncAttributeMaxDynamicSharedMemorySize, v->smem_bytes);
    if (e != cudaSuccess) return fail_cuda(e, "cudaFuncSetAttribute(max dynamic smem)");
    if (v->clustered) {
        e = cudaFuncSetAttribute(v->func, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return fail_cuda(e, "cudaFuncSetAttribute(non-portable cluster)");
    }
    if (d->attr_n < 32) d->attr_done[d->attr_n++] = v->func;
    return NF_OK;
}

nf_status max_clusters(DeviceState* d, const GemmVariant* v, int cluster, int* out) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        for (int i = 0; i < d->occ_n; ++i)
            if (d->occ_func[i] == v->func && d->occ_cluster[i] == cluster) {
                *out = d->occ_value[i];
                return NF_OK;
            }
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(cluster * 64));
    cfg.blockDim = dim3(static_cast<unsigned>(v->threads));
    cfg.dynamicSmemBytes = static_cast<size_t>(v->smem_bytes);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&n, v->func, &cfg);
    if (e != cudaSuccess) return fail_cuda(e, "cudaOccupancyMaxActiveClusters");
    if (n < 1) return fail(NF_ERR_UNSUPPORTED_SHAPE, "this cluster size cannot be co-resident on the device");
    std::lock_guard<std::mutex> lk(g_mu);
    if (d->occ_n < 16) {
        d->occ_func[d->occ_n] = v->func;
        d->occ_cluster[d->occ_n] = cluster;
        d->occ_value[d->occ_n] = n;
        ++d->occ_n;
    }
    *out = n;
    return NF_OK;
}

// Resident CTAs per SM of a variant (cached per device).
nf_status blocks_per_sm(DeviceState* d, const GemmVariant* v, int* out) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        for (int i = 0; i < d->blk_n; ++i)
            if (d->blk_func[i] == v->func) {
                *out = d->blk_value[i];
                return NF_OK;
            }
    }
    int n = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, v->func, v->threads,
                                                                  static_cast<size_t>(v->smem_bytes));
    if (e != cudaSuccess) return fail_cuda(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    if (n < 1) return fail(NF_ERR_UNSUPPORTED_SHAPE, "the kernel does not fit on an SM");
    std::lock_guard<std::mutex> lk(g_mu);
    if (d->blk_n < 16) {
        d->blk_func[d->blk_n] = v->func;
        d->blk_value[d->blk_n] = n;
        ++d->blk_n;
    }
    *out = n;
    return NF_OK;
}

// The stream's global-exchange scratch for m_tiles x n_tiles tiles.  Set up
// (or replaced by a larger one) in stream order, without synchronizing the
// host; refused while the stream is being captured into a graph.
nf_status xch_scratch(cudaStream_t stream, int m_tiles, int n_tiles, int** cnt, int32_t* bank,
                      unsigned long long** stats,
                      int64_t tag_rows = 0, unsigned long long** tags = nullptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
    const int64_t need_bank = xch_bank_ints(m_tiles), need_stats = xch_stats_bytes(m_tiles, n_tiles);
    const int64_t need_tags = tag_rows * 8;
    std::lock_guard<std::mutex> lk(g_mu);
    XScratch* x = nullptr;
    for (int i = 0; i < g_xs_n; ++i)
        if (g_xs[i].dev == dev && g_xs[i].stream == stream) x = &g_xs[i];
    if (x && x->bank_ints >= need_bank && x->stats_bytes >= need_stats && x->tag_bytes >= need_tags) {
        *cnt = x->cnt();
        *bank = static_cast<int32_t>(x->bank_ints);
        *stats = x->stats();
        if (tags) *tags = x->tags();
        return NF_OK;
    }
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if ((e = cudaStreamIsCapturing(stream, &cs)) != cudaSuccess) return fail_cuda(e, "cudaStreamIsCapturing");
    if (cs != cudaStreamCaptureStatusNone)
        return fail(NF_ERR_INVALID_ARG,
                    "exchange scratch is set up on the first call per stream (and enlarged for larger "
                    "shapes): make that call, or nf_reserve_scratch, before capturing the stream");
    if (!x && g_xs_n == kMaxScratch) return fail(NF_ERR_UNSUPPORTED_SHAPE, "too many streams with exchange scratch");
    int64_t bank_ints = need_bank, stats_bytes = need_stats, tag_bytes = need_tags;
    if (x) {
        bank_ints = bank_ints > x->bank_ints ? bank_ints : x->bank_ints;
        stats_bytes = stats_bytes > x->stats_bytes ? stats_bytes : x->stats_bytes;
        tag_bytes = tag_bytes > x->tag_bytes ? tag_bytes : x->tag_bytes;
    }
    // Round every region up so that modest growth reuses the buffer.
    bank_ints = (bank_ints + 4095) / 4096 * 4096;
    stats_bytes = (stats_bytes + (1 << 20) - 1) >> 20 << 20;
    tag_bytes = (tag_bytes + (1 << 20) - 1) >> 20 << 20;
    const size_t bytes = static_cast<size_t>(XScratch::stats_offset(bank_ints) + stats_bytes + tag_bytes);
    void* ptr = nullptr;
    if ((e = cudaMallocAsync(&ptr, bytes, stream)) != cudaSuccess) return fail_cuda(e, "cudaMallocAsync(exchange scratch)");
    if ((e = cudaMemsetAsync(ptr, 0, bytes, stream)) != cudaSuccess) {
        cudaFreeAsync(ptr, stream);
        return fail_cuda(e, "cudaMemsetAsync(exchange scratch)");
    }
    if (!x) {
        x = &g_xs[g_xs_n++];
        x->dev = dev;
        x->stream = stream;
    }
    // (the previous buffer, if any, stays allocated: see XScratch)
    x->ptr = static_cast<uint8_t*>(ptr);
    x->bytes = bytes;
    x->bank_ints = bank_ints;
    x->stats_bytes = stats_bytes;
    x->tag_bytes = tag_bytes;
    *cnt = x->cnt();
    *bank = static_cast<int32_t>(x->bank_ints);
    *stats = x->stats();
    if (tags) *tags = x->tags();
    return NF_OK;
}

// Split-K workspace, one per (device, stream), sized once for a full wave of
// 128 x 256 fp32 partial tiles (splitk x M x N <= SMs x 128 x 256).  Every
// value the reduction reads was written by the GEMM before it, so it needs no
// clearing.  The first call per stream allocates it in stream order (no host
// synchronization; refused during capture).
struct SKScratch {
    int dev = -1;
    cudaStream_t stream = nullptr;
    float* ptr = nullptr;
};
SKScratch g_sk[kMaxScratch];
int g_sk_n = 0;

nf_status splitk_scratch(cudaStream_t stream, int sm_count, float** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < g_sk_n; ++i)
        if (g_sk[i].dev == dev && g_sk[i].stream == stream) {
            *out = g_sk[i].ptr;
            return NF_OK;
        }
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if ((e = cudaStreamIsCapturing(stream, &cs)) != cudaSuccess) return fail_cuda(e, "cudaStreamIsCapturing");
    if (cs != cudaStreamCaptureStatusNone)
        return fail(NF_ERR_INVALID_ARG,
                    "the split-K workspace is set up on the first split GEMM per stream: make that call, or "
                    "nf_reserve_scratch, before capturing the stream");
    if (g_sk_n == kMaxScratch) return fail(NF_ERR_UNSUPPORTED_SHAPE, "too many streams with split-K workspaces");
    void* ptr = nullptr;
    const size_t bytes = static_cast<size_t>(sm_count) * TILE_M * 256 * sizeof(float);
    if ((e = cudaMallocAsync(&ptr, bytes, stream)) != cudaSuccess) return fail_cuda(e, "cudaMallocAsync(split-K workspace)");
    g_sk[g_sk_n].dev = dev;
    g_sk[g_sk_n].stream = stream;
    g_sk[g_sk_n].ptr = static_cast<float*>(ptr);
    ++g_sk_n;
    *out = static_cast<float*>(ptr);
    return NF_OK;
}

// The current device's fixed no-alloc scratch: address looked up and the
// array cleared (synchronously) on first use per device, which is refused
// while `stream` is being captured.
nf_status noalloc_scratch(cudaStream_t stream, uint8_t** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(NF_ERR_NO_DEVICE, "device index out of range");
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_noalloc_ptr[dev]) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if ((e = cudaStreamIsCapturing(stream, &cs)) != cudaSuccess) return fail_cuda(e, "cudaStreamIsCapturing");
        if (cs != cudaStreamCaptureStatusNone)
            return fail(NF_ERR_INVALID_ARG,
                        "the no-alloc scratch is cleared by the first call on each device: make that call before "
                        "capturing the stream");
        void* p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_noalloc_scratch)) != cudaSuccess)
            return fail_cuda(e, "cudaGetSymbolAddress(no-alloc scratch)");
        if ((e = cudaMemset(p, 0, static_cast<size_t>(kNoAllocBytes))) != cudaSuccess)
            return fail_cuda(e, "clear no-alloc scratch");
        if ((e = cudaDeviceSynchronize()) != cudaSuccess) return fail_cuda(e, "cudaDeviceSynchronize");
        g_noalloc_ptr[dev] = static_cast<uint8_t*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return NF_OK;
}

// fixed_scratch: the global exchange uses the no-alloc array instead of the
// stream's scratch buffer.
// ops (OperandFlags): OPS_A_MN -- X is stored K x M; OPS_A_SCALE -- and its
// row k is scaled by rstd_in[k] on the fly; OPS_B_K -- W is stored N x K.
nf_status run_gemm(int op, const void* X, const void* W, const void* gamma, const void* beta, void* Y, int64_t M,
                   int64_t N, int64_t K, float eps, float* mean_out, float* rstd_out, cudaStream_t stream,
                   bool fixed_scratch = false, const void* zin = nullptr, const float* mean_in = nullptr,
                   const float* rstd_in = nullptr, int ops = 0, void* xhat_out = nullptr,
                   const void* resid = nullptr, void* h_out = nullptr) {
    nf_status st = check_gemm_args(op, X, W, Y, gamma, beta, mean_out, rstd_out, M, N, K, eps);
    if (st != NF_OK) return st;
    if (h_out && !resid) return fail(NF_ERR_INVALID_ARG, "the residual output needs a residual");
    if (resid && op != OP_POST_LN && op != OP_POST_RMS)
        return fail(NF_ERR_INVALID_ARG, "a residual is added by the post-norm epilogues only");
    if (M == 0) return NF_OK;
    if ((resid && !aligned(resid, 16)) || (h_out && !aligned(h_out, 16)))
        return fail(NF_ERR_ALIGNMENT, "R and H must be 16-byte aligned");
    if ((ops & OPS_A_MN) && M % 8 != 0)
        return fail(NF_ERR_ALIGNMENT, "a transposed X (K x M) needs M a multiple of 8 (16-byte rows)");
    if ((ops & OPS_A_SCALE) && !rstd_in) return fail(NF_ERR_INVALID_ARG, "row scaling needs rstd");
    if ((ops & OPS_A_SCALE) && !aligned(rstd_in, 16))  // copied 64 values at a time with the ring stages
        return fail(NF_ERR_ALIGNMENT, "row scaling needs a 16-byte aligned rstd");
    if (op == OP_BWD_LN || op == OP_BWD_RMS) {
        if (!zin || !rstd_in || (op == OP_BWD_LN && !mean_in))
            return fail(NF_ERR_INVALID_ARG, "Z, rstd (and mean for LN) must be non-null");
        if (!aligned(zin, 16)) return fail(NF_ERR_ALIGNMENT, "Z must be 16-byte aligned");
        if ((mean_in && !aligned(mean_in, 4)) || !aligned(rstd_in, 4))
            return fail(NF_ERR_ALIGNMENT, "mean and rstd must be 4-byte aligned");
        if (xhat_out && !aligned(xhat_out, 16)) return fail(NF_ERR_ALIGNMENT, "xhat must be 16-byte aligned");
    }
    DeviceState* d = nullptr;
    if ((st = device_state(&d)) != NF_OK) return st;
    Plan p;
    if (resid) ops |= OPS_RESID;
    if ((st = plan_tiles(op, M, N, K, d->sm_count, &p, ops)) != NF_OK) return st;
    if ((st = prepare_kernel(d, p.v)) != NF_OK) return st;

    CUtensorMap tmX, tmW, tmY;
    const int tk = p.v->tile_k;  // 64: 128-byte rows of X; 32: 64-byte rows
    if (ops & OPS_A_MN) {  // X stored K x M: boxes of 64 K-rows x 64 output rows
        if ((st = make_map(&tmX, X, K, M, 64, 64)) != NF_OK) return st;
    } else if ((st = make_map(&tmX, X, M, K, tk, TILE_M,
                              tk == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B)) != NF_OK) {
        return st;
    }
    if (ops & OPS_B_K) {  // W stored N x K: boxes of tile_n output columns x 64 K
        if ((st = make_map(&tmW, W, N, K, tk, p.tile_n)) != NF_OK) return st;
    } else if ((st = make_map(&tmW, W, K, N, B_BOX_N, tk)) != NF_OK) {
        return st;
    }
    if ((st = make_map(&tmY, Y, M, N, STORE_COLS, STORE_ROWS)) != NF_OK) return st;

    GemmArgs a;
    a.M = static_cast<int32_t>(M);
    a.N = static_cast<int32_t>(N);
    a.K = static_cast<int32_t>(K);
    a.m_tiles = p.m_tiles;
    a.n_tiles = p.n_tiles;
    a.k_tiles = p.k_tiles;
    a.cluster = p.cluster;
    a.eps = eps;
    a.inv_len = op == OP_PRE ? 1.0f / static_cast<float>(K) : 1.0f / static_cast<float>(N);
    a.gamma = static_cast<const uint16_t*>(gamma);
    a.beta = static_cast<const uint16_t*>(beta);
    a.mean_out = mean_out;
    a.rstd_out = rstd_out;
    a.status = d->status;
    a.timeout_ns = g_timeout_ns;
    a.zin = static_cast<const uint16_t*>(zin);
    a.mean_in = mean_in;
    a.rstd_in = rstd_in;
    a.xcnt = nullptr;
    a.xbank = 0;
    a.xpart = nullptr;
    a.sstag = nullptr;
    a.splitk = p.splitk;
    a.sk_base = p.sk_base;
    a.sk_tiles = p.sk_tiles;
    a.ws = nullptr;
    a.xhat_out = (op == OP_BWD_LN || op == OP_BWD_RMS) ? static_cast<uint16_t*>(xhat_out) : nullptr;
    a.resid = static_cast<const uint16_t*>(resid);
    a.h_out = static_cast<uint16_t*>(h_out);

    int grid = 0;
    // Exchange scratch: post-norm partials of every (row tile, column tile);
    // the pre-norm's split sums of squares use only the counter header (for
    // the launch epoch) and their own region of tagged words, one per row.
    const int xnt = op == OP_PRE ? 0 : p.n_tiles;
    const int64_t xtag_rows = op == OP_PRE ? static_cast<int64_t>(p.m_tiles) * TILE_M : 0;
    a.units = p.m_tiles * p.n_tiles;
    a.split_base = a.units;
    if (p.pair) {
        // Pair tiles of 256 rows, one cluster of two CTAs each, persistent.
        // With the L2 exchange every cluster is resident at once (cooperative
        // launch); 2 x clusters >= n_tiles keeps the exchange deadlock free
        // (the argument of the kernel, per pair tile).
        int mc = 0;
        if ((st = max_clusters(d, p.v, 2, &mc)) != NF_OK) return st;
        a.units = ((p.m_tiles + 1) / 2) * p.n_tiles;
        a.split_base = a.units;
        const int clusters = a.units < mc ? a.units : mc;
        grid = clusters * 2;
        if (p.xch == XCH_GLOBAL) {
            if (2 * clusters < p.n_tiles) return fail(NF_ERR_UNSUPPORTED_SHAPE, "too few resident CTA pairs for the exchange");
            if (fixed_scratch) {
                if (xch_bank_ints(p.m_tiles) > kNoAllocBankInts ||
                    xch_stats_bytes(p.m_tiles, p.n_tiles) > kNoAllocStatsBytes)
                    return fail(NF_ERR_UNSUPPORTED_SHAPE,
                                "no-alloc post-norm: ceil(M/128) * ceil(N/256) must be <= 4096 (so M <= 2^19)");
                uint8_t* base = nullptr;
                if ((st = noalloc_scratch(stream, &base)) != NF_OK) return st;
                a.xcnt = reinterpret_cast<int*>(base);
                a.xbank = static_cast<int32_t>(kNoAllocBankInts);
                a.xpart = reinterpret_cast<unsigned long long*>(base + kNoAllocStatsOffset);
            } else if ((st = xch_scratch(stream, p.m_tiles, xnt, &a.xcnt, &a.xbank, &a.xpart, xtag_rows,
                                         &a.sstag)) != NF_OK) {
                return st;
            }
        }
    } else if (p.clustered) {
        int mc = 0;
        if ((st = max_clusters(d, p.v, p.cluster, &mc)) != NF_OK) return st;
        grid = (p.m_tiles < mc ? p.m_tiles : mc) * p.cluster;
    } else if (p.xch == XCH_GLOBAL) {
        // Every CTA resident at once (cooperative launch), tiles in order,
        // no split units.  grid >= n_tiles / 2 keeps the exchange deadlock
        // free (see the kernel); n_tiles <= 16 and tiles >= n_tiles.
        int per_sm = 0;
        if ((st = blocks_per_sm(d, p.v, &per_sm)) != NF_OK) return st;
        const int tiles = p.m_tiles * p.n_tiles;
        const int cap = per_sm * d->sm_count;
        grid = tiles < cap ? tiles : cap;
        if (2 * grid < p.n_tiles) return fail(NF_ERR_UNSUPPORTED_SHAPE, "too few resident CTAs for the exchange");
        if (fixed_scratch) {
            if (xch_bank_ints(p.m_tiles) > kNoAllocBankInts || xch_stats_bytes(p.m_tiles, p.n_tiles) > kNoAllocStatsBytes)
                return fail(NF_ERR_UNSUPPORTED_SHAPE,
                            "no-alloc post-norm: ceil(M/128) * ceil(N/256) must be <= 4096 (so M <= 2^19)");
            uint8_t* base = nullptr;
            if ((st = noalloc_scratch(stream, &base)) != NF_OK) return st;
            a.xcnt = reinterpret_cast<int*>(base);
            a.xbank = static_cast<int32_t>(kNoAllocBankInts);
            a.xpart = reinterpret_cast<unsigned long long*>(base + kNoAllocStatsOffset);
        } else if ((st = xch_scratch(stream, p.m_tiles, xnt, &a.xcnt, &a.xbank, &a.xpart, xtag_rows,
                                     &a.sstag)) != NF_OK) {
            return st;
        }
    } else if (p.splitk > 1) {
        // Whole tiles first (whole waves), then the split tiles' units, at most
        // one per CTA: sk_tiles x splitk <= SMs.
        if ((st = splitk_scratch(stream, d->sm_count, &a.ws)) != NF_OK) return st;
        a.units = p.sk_base + p.sk_tiles * p.splitk;
        a.split_base = a.units;
        grid = a.units < d->sm_count ? a.units : d->sm_count;
    } else {
        const int tiles = p.m_tiles * p.n_tiles;
        grid = tiles < d->sm_count ? tiles : d->sm_count;
        split_last_wave(tiles, grid, tile_memory_bound(K, p.tile_n, p.n_tiles), &a.units, &a.split_base);
    }

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[3];
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(p.v->threads));
    cfg.dynamicSmemBytes = static_cast<size_t>(p.v->smem_bytes);
    cfg.stream = stream;
    // Attributes: cluster (row cluster or CTA pair), cooperative (the L2
    // exchange needs every CTA resident), programmatic dependent launch.
    auto set_attrs = [&](bool coop, bool overlap) {
        int nattr = 0;
        if (p.clustered || p.pair) {
            attr[nattr].id = cudaLaunchAttributeClusterDimension;
            attr[nattr].val.clusterDim.x = static_cast<unsigned>(p.cluster);
            attr[nattr].val.clusterDim.y = 1;
            attr[nattr].val.clusterDim.z = 1;
            ++nattr;
        }
        if (coop) {
            attr[nattr].id = cudaLaunchAttributeCooperative;
            attr[nattr].val.cooperative = 1;
            ++nattr;
        }
        if (overlap) {
            attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[nattr].val.programmaticStreamSerializationAllowed = 1;
            ++nattr;
        }
        cfg.attrs = nattr ? attr : nullptr;
        cfg.numAttrs = static_cast<unsigned>(nattr);
    };
    bool coop = p.xch == XCH_GLOBAL && (!p.pair || g_coop_cluster_ok);
    bool overlap = g_overlap && (p.xch != XCH_GLOBAL || g_coop_overlap_ok);
    set_attrs(coop, overlap);
    void* kargs[4] = {&tmX, &tmW, &tmY, &a};
    cudaError_t e = cudaLaunchKernelExC(&cfg, p.v->func, kargs);
    if (e != cudaSuccess && coop && p.pair) {
        // The runtime refused a cooperative launch of clusters: CTA pairs then
        // rely on the grid fitting the device at once (it is sized from the
        // resident cluster count), without the guarantee.
        (void)cudaGetLastError();
        g_coop_cluster_ok = false;
        coop = false;
        set_attrs(coop, overlap);
        e = cudaLaunchKernelExC(&cfg, p.v->func, kargs);
    }
    if (e != cudaSuccess && overlap && p.xch == XCH_GLOBAL) {
        // The runtime refused programmatic serialization on a cooperative
        // launch: drop it for these launches from now on.
        (void)cudaGetLastError();
        g_coop_overlap_ok = false;
        overlap = false;
        set_attrs(coop, overlap);
        e = cudaLaunchKernelExC(&cfg, p.v->func, kargs);
    }
    if (e != cudaSuccess) return fail_cuda(e, "kernel launch");
    if (p.splitk > 1) {
        SplitkReduceArgs r;
        r.ws = a.ws;
        r.y = static_cast<uint16_t*>(Y);
        r.slices = p.splitk;
        r.sk_base = p.sk_base;
        r.sk_tiles = p.sk_tiles;
        r.n_tiles = p.n_tiles;
        r.tile_n = p.tile_n;
        r.M = a.M;
        r.N = a.N;
        if ((e = launch_splitk_reduce(r, d->sm_count, g_overlap, stream)) != cudaSuccess)
            return fail_cuda(e, "split-K reduction launch");
    }
    return NF_OK;
}

}  // namespace
}  // namespace nf

using namespace nf;

extern "C" {

nf_status nf_gemm_plain(const void* X, const void* W, void* Y, int64_t M, int64_t N, int64_t K, nf_stream stream) {
    return run_gemm(OP_PLAIN, X, W, nullptr, nullptr, Y, M, N, K, 0.0f, nullptr, nullptr,
                    reinterpret_cast<cudaStream_t>(stream));
}

nf_status nf_gemm_prenorm_rms(const void* X, const void* W, void* Y, int64_t M, int64_t N, int64_t K, float eps,
                              float* rstd_out, nf_stream stream) {
    return run_gemm(OP_PRE, X, W, nullptr, nullptr, Y, M, N, K, eps, nullptr, rstd_out,
                    reinterpret_cast<cudaStream_t>(stream));
}

nf_status nf_gemm_postnorm_ln(const void* X, const void* W, const void* gamma, const void* beta, void* Y, int64_t M,
                              int64_t N, int64_t K, float eps, float* mean_out, float* rstd_out, nf_stream stream) {
    return run_gemm(OP_POST_LN, X, W, gamma, beta, Y, M, N, K, eps, mean_out, rstd_out,
                    reinterpret_cast<cudaStream_t>(stream));
}

nf_status nf_gemm_postnorm_ln_noalloc(const void* X, const void* W, const void* gamma, const void* beta, void* Y,
                                      int64_t M, int64_t N, int64_t K, float eps, float* mean_out, float* rstd_out,
                                      nf_stream stream) {
    return run_gemm(OP_POST_LN, X, W, gamma, beta, Y, M, N, K, eps, mean_out, rstd_out,
                    reinterpret_cast<cudaStream_t>(stream), true);
}

nf_status nf_gemm_postnorm_ln_bwd(const void* A, const void* B, const void* Z, const void* gamma, const float* mean,
                                  const float* rstd, void* dZ, int64_t M, int64_t N, int64_t K, nf_stream stream) {
    return run_gemm(OP_BWD_LN, A, B, gamma, nullptr, dZ, M, N, K, 0.0f, nullptr, nullptr,
                    reinterpret_cast<cudaStream_t>(stream), false, Z, mean, rstd);
}

nf_status nf_gemm_postnorm_rms_bwd(const void* A, const void* B, const void* Z, const void* gamma, const float* rstd,
                                   void* dZ, int64_t M, int64_t N, int64_t K, nf_stream stream) {
    return run_gemm(OP_BWD_RMS, A, B, gamma, nullptr, dZ, M, N, K, 0.0f, nullptr, nullptr,
                    reinterpret_cast<cudaStream_t>(stream), false, Z, nullptr, rstd);
}

nf_status nf_gemm_plain_t(const void* X, const void* W, void* Y, int64_t M, int64_t N, int64_t K, int flags,
                          nf_stream stream) {
    if (flags & ~(NF_TRANS_X | NF_TRANS_W)) return fail(NF_ERR_INVALID_ARG, "flags: NF_TRANS_X | NF_TRANS_W");
    if ((flags & NF_TRANS_X) && (flags & NF_TRANS_W))
        return fail(NF_ERR_UNSUPPORTED_SHAPE, "only one operand may be transposed");
    const int ops = ((flags & NF_TRANS_X) ? OPS_A_MN : 0) | ((flags & NF_TRANS_W) ? OPS_B_K : 0);
    return run_gemm(OP_PLAIN, X, W, nullptr, nullptr, Y, M, N, K, 0.0f, nullptr, nullptr,
                    reinterpret_cast<cudaStream_t>(stream), false, nullptr, nullptr, nullptr, ops);
}

nf_status nf_gemm_prenorm_rms_bwd(const void* A, const void* B, const float* rstd, const void* dC, void* dA, void* dB,
                                  void* xhat, int64_t M, int64_t N, int64_t K, nf_stream stream) {
    if (M < 0 || N < 1 || K < 1) return fail(NF_ERR_INVALID_ARG, "need M >= 0, N >= 1, K >= 1");
    if (M == 0) return NF_OK;
    if (!A || !B || !rstd || !dC) return fail(NF_ERR_INVALID_ARG, "A, B, rstd and dC must be non-null");
    if (!dA && !dB) return NF_OK;
    if (M % 8 != 0 && dB) return fail(NF_ERR_ALIGNMENT, "dB needs M a multiple of 8 (A is read transposed)");
    if (K > NF_POSTNORM_MAX_N && dA)
        return fail(NF_ERR_UNSUPPORTED_SHAPE, "dA needs K <= 4096 (the RMS backward reduces over K)");
    nf_status st = NF_OK;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (xhat && !aligned(xhat, 16)) return fail(NF_ERR_ALIGNMENT, "xhat must be 16-byte aligned");
    const bool side = xhat && dA;  // the dA kernel writes xhat, dB reads it
    // dA = rmsnorm_bwd(dC B^T; A, rstd): a GEMM of M x K over N whose W (= B,
    // stored K x N) is read transposed, RMS-backward epilogue with Z = A
    // (and, with xhat, the side output xhat = bf16(A * rstd)).
    if (dA && (st = run_gemm(OP_BWD_RMS, dC, B, nullptr, nullptr, dA, M, K, N, 0.0f, nullptr, nullptr, s, false, A,
                             nullptr, rstd, OPS_B_K, side ? xhat : nullptr)) != NF_OK)
        return st;
    // dB = rmsnorm(A)^T dC: a GEMM of K x N over M whose X is read
    // transposed -- xhat as written above, or A with row m scaled by rstd[m]
    // in shared memory on the fly.
    if (dB && side &&
        (st = run_gemm(OP_PLAIN, xhat, dC, nullptr, nullptr, dB, K, N, M, 0.0f, nullptr, nullptr, s, false, nullptr,
                       nullptr, nullptr, OPS_A_MN)) != NF_OK)
        return st;
    if (dB && !side &&
        (st = run_gemm(OP_PLAIN, A, dC, nullptr, nullptr, dB, K, N, M, 0.0f, nullptr, nullptr, s, false, nullptr,
                       nullptr, rstd, OPS_A_MN | OPS_A_SCALE)) != NF_OK)
        return st;
    return NF_OK;
}

nf_status nf_gemm_postnorm_ln_res(const void* X, const void* W, const void* R, const void* gamma, const void* beta,
                                  void* Y, void* H, int64_t M, int64_t N, int64_t K, float eps, float* mean_out,
                                  float* rstd_out, nf_stream stream) {
    if (M > 0 && !R) return fail(NF_ERR_INVALID_ARG, "R must be non-null");
    return run_gemm(OP_POST_LN, X, W, gamma, beta, Y, M, N, K, eps, mean_out, rstd_out,
                    reinterpret_cast<cudaStream_t>(stream), false, nullptr, nullptr, nullptr, 0, nullptr, R, H);
}

nf_status nf_gemm_postnorm_rms_res(const void* X, const void* W, const void* R, const void* gamma, void* Y, void* H,
                                   int64_t M, int64_t N, int64_t K, float eps, float* rstd_out, nf_stream stream) {
    if (M > 0 && !R) return fail(NF_ERR_INVALID_ARG, "R must be non-null");
    return run_gemm(OP_POST_RMS, X, W, gamma, nullptr, Y, M, N, K, eps, nullptr, rstd_out,
                    reinterpret_cast<cudaStream_t>(stream), false, nullptr, nullptr, nullptr, 0, nullptr, R, H);
}

nf_status nf_flashnorm_attn_fwd(const void* Q, const void* K, const void* V, const int32_t* q_len, void* Out,
                                int64_t B, int64_t Lq, int64_t Lkv, int64_t H, int64_t D, int act, float eps1,
                                float eps2, nf_stream stream) {
    if (B < 0 || Lq < 0 || H < 1) return fail(NF_ERR_INVALID_ARG, "need B >= 0, Lq >= 0, H >= 1");
    if (act < NF_ACT_IDENTITY || act > NF_ACT_SILU) return fail(NF_ERR_INVALID_ARG, "act: identity, GELU or SiLU");
    if (!(std::isfinite(eps1) && eps1 >= 0.0f && std::isfinite(eps2) && eps2 >= 0.0f))
        return fail(NF_ERR_INVALID_ARG, "eps must be finite and >= 0");
    if (D != 128 || Lkv != 128) return fail(NF_ERR_UNSUPPORTED_SHAPE, "head dimension and K/V length must be 128");
    if (H > 8) return fail(NF_ERR_UNSUPPORTED_SHAPE, "at most 8 heads (one cluster of H CTAs)");
    if (Lq % 128 != 0) return fail(NF_ERR_UNSUPPORTED_SHAPE, "Lq must be a multiple of 128");
    if (B * Lq > INT32_MAX || B * Lkv > INT32_MAX) return fail(NF_ERR_UNSUPPORTED_SHAPE, "too many rows");
    if (B == 0 || Lq == 0) return NF_OK;
    if (!Q || !K || !V || !Out) return fail(NF_ERR_INVALID_ARG, "Q, K, V and Out must be non-null");
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(Out, 16) || (q_len && !aligned(q_len, 4)))
        return fail(NF_ERR_ALIGNMENT, "Q, K, V, Out must be 16-byte aligned, q_len 4-byte");
    DeviceState* d = nullptr;
    nf_status st = device_state(&d);
    if (st != NF_OK) return st;
    CUtensorMap maps[4];
    const int64_t hd = H * 128;
    if ((st = make_map(&maps[0], Q, B * Lq, hd, 64, 128)) != NF_OK) return st;
    if ((st = make_map(&maps[1], K, B * Lkv, hd, 64, 128)) != NF_OK) return st;
    if ((st = make_map(&maps[2], V, B * Lkv, hd, 64, 64)) != NF_OK) return st;
    if ((st = make_map(&maps[3], Out, B * Lq, hd, 64, 32)) != NF_OK) return st;
    FlashNormLaunch a;
    a.q_len = q_len;
    a.B = static_cast<int32_t>(B);
    a.Lq = static_cast<int32_t>(Lq);
    a.H = static_cast<int32_t>(H);
    a.act = act;
    a.eps1 = eps1;
    a.eps2 = eps2;
    a.status = d->status;
    a.timeout_ns = g_timeout_ns;
    cudaError_t e = launch_flashnorm_fwd(maps, a, g_overlap, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e, "FlashNormAttention launch");
    return NF_OK;
}

nf_status nf_gemm_postnorm_rms(const void* X, const void* W, const void* gamma, void* Y, int64_t M, int64_t N,
                               int64_t K, float eps, float* rstd_out, nf_stream stream) {
    return run_gemm(OP_POST_RMS, X, W, gamma, nullptr, Y, M, N, K, eps, nullptr, rstd_out,
                    reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace nf {
namespace {
nf_status norm_rows_impl(const void* in, const void* res, void* out, void* h_out, const void* gamma,
                         const void* beta, int64_t rows, int64_t cols, int kind, float eps, float* mean_out,
                         float* rstd_out, nf_stream stream) {
    if (kind != NF_NORM_LN && kind != NF_NORM_RMS) return fail(NF_ERR_INVALID_ARG, "kind must be LN or RMS");
    if (rows < 0 || cols < 1) return fail(NF_ERR_INVALID_ARG, "need rows >= 0 and cols >= 1");
    if (rows == 0) {  // empty tensors may have a null base: nothing is accessed
        in = in ? in : reinterpret_cast<const void*>(256);
        out = out ? out : reinterpret_cast<void*>(256);
    }
    if (!in || !out) return fail(NF_ERR_INVALID_ARG, "in and out must be non-null");
    if (!(std::isfinite(eps) && eps >= 0.0f)) return fail(NF_ERR_INVALID_ARG, "eps must be finite and >= 0");
    if (cols > NORM_MAX_COLS) return fail(NF_ERR_UNSUPPORTED_SHAPE, "cols must be <= 16384");
    if (cols % 8 != 0) return fail(NF_ERR_ALIGNMENT, "cols must be a multiple of 8 (16-byte rows)");
    if (!aligned(in, 16) || !aligned(out, 16)) return fail(NF_ERR_ALIGNMENT, "in and out must be 16-byte aligned");
    // gamma / beta are read as 16-byte vectors as well
    if ((gamma && !aligned(gamma, 16)) || (beta && !aligned(beta, 16)))
        return fail(NF_ERR_ALIGNMENT, "gamma and beta must be 16-byte aligned for nf_norm_rows");
    if ((mean_out && !aligned(mean_out, 4)) || (rstd_out && !aligned(rstd_out, 4)))
        return fail(NF_ERR_ALIGNMENT, "mean_out and rstd_out must be 4-byte aligned");
    if (h_out && !res) return fail(NF_ERR_INVALID_ARG, "the residual output needs a residual");
    if (rows > 0 && ((res && !aligned(res, 16)) || (h_out && !aligned(h_out, 16))))
        return fail(NF_ERR_ALIGNMENT, "the residual and its output must be 16-byte aligned");
    if (rows == 0) return NF_OK;
    DeviceState* d = nullptr;
    nf_status st = device_state(&d);
    if (st != NF_OK) return st;
    NormArgs a;
    a.res = res;
    a.h_out = h_out;
    a.in = in;
    a.out = out;
    a.gamma = static_cast<const uint16_t*>(gamma);
    a.beta = static_cast<const uint16_t*>(beta);
    a.rows = rows;
    a.cols = static_cast<int32_t>(cols);
    a.eps = eps;
    a.inv_cols = 1.0f / static_cast<float>(cols);
    a.mean_out = mean_out;
    a.rstd_out = rstd_out;
    cudaError_t e = launch_norm_rows(a, kind, d->sm_count, g_overlap, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e, "norm_rows launch");
    return NF_OK;
}
}  // namespace
}  // namespace nf

extern "C" {

nf_status nf_norm_rows(const void* in, void* out, const void* gamma, const void* beta, int64_t rows, int64_t cols,
                       int kind, float eps, float* mean_out, float* rstd_out, nf_stream stream) {
    return norm_rows_impl(in, nullptr, out, nullptr, gamma, beta, rows, cols, kind, eps, mean_out, rstd_out, stream);
}

nf_status nf_norm_rows_res(const void* in, const void* R, void* out, void* H, const void* gamma, const void* beta,
                           int64_t rows, int64_t cols, int kind, float eps, float* mean_out, float* rstd_out,
                           nf_stream stream) {
    if (rows > 0 && !R) return fail(NF_ERR_INVALID_ARG, "R must be non-null");
    return norm_rows_impl(in, R, out, H, gamma, beta, rows, cols, kind, eps, mean_out, rstd_out, stream);
}

nf_status nf_norm_rows_bwd(const void* dY, const void* Z, const void* gamma, const float* mean, const float* rstd,
                           void* dZ, int64_t rows, int64_t cols, int kind, nf_stream stream) {
    if (kind != NF_NORM_LN && kind != NF_NORM_RMS) return fail(NF_ERR_INVALID_ARG, "kind must be LN or RMS");
    if (rows < 0 || cols < 1) return fail(NF_ERR_INVALID_ARG, "need rows >= 0 and cols >= 1");
    if (rows == 0) return NF_OK;  // nothing is accessed
    if (!dY || !Z || !dZ || !rstd || (kind == NF_NORM_LN && !mean))
        return fail(NF_ERR_INVALID_ARG, "dY, Z, dZ, rstd (and mean for LN) must be non-null");
    if (cols > NORM_MAX_COLS) return fail(NF_ERR_UNSUPPORTED_SHAPE, "cols must be <= 16384");
    if (cols % 8 != 0) return fail(NF_ERR_ALIGNMENT, "cols must be a multiple of 8 (16-byte rows)");
    if (!aligned(dY, 16) || !aligned(Z, 16) || !aligned(dZ, 16))
        return fail(NF_ERR_ALIGNMENT, "dY, Z and dZ must be 16-byte aligned");
    if (gamma && !aligned(gamma, 16)) return fail(NF_ERR_ALIGNMENT, "gamma must be 16-byte aligned for nf_norm_rows_bwd");
    if ((mean && !aligned(mean, 4)) || !aligned(rstd, 4))
        return fail(NF_ERR_ALIGNMENT, "mean and rstd must be 4-byte aligned");
    DeviceState* d = nullptr;
    nf_status st = device_state(&d);
    if (st != NF_OK) return st;
    NormBwdArgs a;
    a.dy = dY;
    a.z = Z;
    a.gamma = static_cast<const uint16_t*>(gamma);
    a.mean = mean;
    a.rstd = rstd;
    a.dz = dZ;
    a.rows = rows;
    a.cols = static_cast<int32_t>(cols);
    a.inv_cols = 1.0f / static_cast<float>(cols);
    cudaError_t e = launch_norm_rows_bwd(a, kind, d->sm_count, g_overlap, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e, "norm_rows_bwd launch");
    return NF_OK;
}

nf_status nf_get_device_status(uint32_t* detail) {
    DeviceState* d = nullptr;
    nf_status st = device_state(&d);
    if (st != NF_OK) return st;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceSynchronize");
    uint32_t w[4] = {0, 0, 0, 0};
    e = cudaMemcpy(w, d->status, sizeof w, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail_cuda(e, "read status word");
    if (detail) memcpy(detail, w, sizeof w);
    return static_cast<nf_status>(w[0]);
}

nf_status nf_clear_device_status(void) {
    DeviceState* d = nullptr;
    nf_status st = device_state(&d);
    if (st != NF_OK) return st;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceSynchronize");
    const uint32_t z[4] = {0, 0, 0, 0};
    e = cudaMemcpy(d->status, z, sizeof z, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail_cuda(e, "clear status word");
    // A launch that gave up may have left exchange counters part-way.
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < g_xs_n; ++i)
        if (g_xs[i].dev == dev && g_xs[i].ptr) {
            e = cudaMemset(g_xs[i].ptr, 0, g_xs[i].bytes);
            if (e != cudaSuccess) return fail_cuda(e, "clear exchange scratch");
        }
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceSynchronize");
    return NF_OK;
}

nf_status nf_set_wait_timeout_ns(uint64_t ns) {
    if (ns < 1000ull || ns > 100000000000ull) return fail(NF_ERR_INVALID_ARG, "timeout must be in [1e3, 1e11] ns");
    g_timeout_ns = ns;
    return NF_OK;
}

nf_status nf_set_postnorm_tile_n(int tile_n) {
    if (tile_n != 0 && tile_n != 256 && tile_n != 512) return fail(NF_ERR_INVALID_ARG, "tile_n must be 0, 256 or 512");
    g_post_tile = tile_n;
    return NF_OK;
}

nf_status nf_set_gemm_tile_n(int tile_n) {
    if (tile_n != 0 && tile_n != 64 && tile_n != 128 && tile_n != 256)
        return fail(NF_ERR_INVALID_ARG, "tile_n must be 0, 64, 128 or 256");
    g_gemm_tile = tile_n;
    return NF_OK;
}

nf_status nf_set_gemm_pair(int mode) {
    if (mode != 0 && mode != 1 && mode != 2)
        return fail(NF_ERR_INVALID_ARG, "pair mode: 0 automatic, 1 never, 2 whenever the tile allows");
    g_pair_mode = mode;
    return NF_OK;
}

nf_status nf_set_prenorm_split(int mode) {
    if (mode < 0 || mode > 2)
        return fail(NF_ERR_INVALID_ARG, "pre-norm split: 0 automatic, 1 never, 2 whenever the shape allows");
    g_pre_split = mode;
    return NF_OK;
}

nf_status nf_set_postnorm_exchange(int mode) {
    if (mode != 0 && mode != NF_XCH_CLUSTER && mode != NF_XCH_GLOBAL)
        return fail(NF_ERR_INVALID_ARG, "mode must be 0 (automatic), 1 (cluster) or 2 (global)");
    g_post_xch = mode;
    return NF_OK;
}

nf_status nf_set_gemm_splitk(int mode) {
    if (mode != 0 && mode != 1) return fail(NF_ERR_INVALID_ARG, "split-K mode: 0 automatic, 1 never");
    g_splitk_mode = mode;
    return NF_OK;
}

nf_status nf_reserve_scratch(int64_t max_rows, int64_t max_cols, nf_stream stream) {
    if (max_rows < 0 || max_cols < 0) return fail(NF_ERR_INVALID_ARG, "sizes must be >= 0");
    if (max_rows > static_cast<int64_t>(INT32_MAX) - TILE_M || max_cols > NF_POSTNORM_MAX_N)
        return fail(NF_ERR_UNSUPPORTED_SHAPE, "max_rows < 2^31 - 128 and max_cols <= NF_POSTNORM_MAX_N");
    DeviceState* d = nullptr;
    nf_status st = device_state(&d);
    if (st != NF_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (max_rows > 0) {
        // Post-norm rows wider than one tile exchange per column tile; the
        // pre-norm's split sums of squares need a tagged word per row.
        int* cnt = nullptr;
        int32_t bank = 0;
        unsigned long long* stats = nullptr;
        const int m_tiles = static_cast<int>((max_rows + TILE_M - 1) / TILE_M);
        const int n_tiles = max_cols > 256 ? static_cast<int>((max_cols + 255) / 256) : 0;
        unsigned long long* tags = nullptr;
        if ((st = xch_scratch(s, m_tiles, n_tiles, &cnt, &bank, &stats, static_cast<int64_t>(m_tiles) * TILE_M,
                              &tags)) != NF_OK)
            return st;
    }
    float* ws = nullptr;
    return splitk_scratch(s, d->sm_count, &ws);
}

nf_status nf_set_launch_overlap(int enable) {
    g_overlap = enable != 0;
    return NF_OK;
}

nf_status nf_selftest_wait_timeout(uint64_t timeout_ns, nf_stream stream) {
    if (timeout_ns < 1000ull || timeout_ns > 10000000000ull)
        return fail(NF_ERR_INVALID_ARG, "timeout must be in [1e3, 1e10] ns");
    DeviceState* d = nullptr;
    nf_status st = device_state(&d);
    if (st != NF_OK) return st;
    nf_selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(d->status, timeout_ns);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail_cuda(e, "self-test launch");
    return NF_OK;
}

const char* nf_status_string(nf_status s) {
    switch (s) {
        case NF_OK: return "ok";
        case NF_ERR_INVALID_ARG: return "invalid argument";
        case NF_ERR_ALIGNMENT: return "misaligned pointer or row pitch";
        case NF_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case NF_ERR_CUDA: return "CUDA error";
        case NF_ERR_TIMEOUT: return "device wait timed out";
        case NF_ERR_NO_DEVICE: return "no usable sm_103 device";
    }
    return "unknown status";
}

const char* nf_last_error(void) { return g_last_error.c_str(); }

nf_status nf_plan_gemm(int op, int64_t M, int64_t N, int64_t K, int sm_count, nf_plan* out) {
    if (!out || op < 0 || op > 5 || sm_count < 1) return fail(NF_ERR_INVALID_ARG, "bad plan query");
    nf_status st = check_gemm_args(op, reinterpret_cast<const void*>(256), reinterpret_cast<const void*>(256),
                                   reinterpret_cast<const void*>(256), nullptr, nullptr, nullptr, nullptr, M, N, K,
                                   1e-5f);
    if (st != NF_OK) return st;
    Plan p;
    if ((st = plan_tiles(op, M > 0 ? M : 1, N, K, sm_count, &p)) != NF_OK) return st;
    out->tile_m = TILE_M;
    out->tile_n = p.tile_n;
    out->tile_k = p.v->tile_k;
    out->stages = p.v->stages;
    out->cluster = p.cluster;
    out->threads = p.v->threads;
    out->smem_bytes = p.v->smem_bytes;
    out->tmem_cols = p.v->tmem_cols;
    out->tiles = M > 0 ? p.m_tiles * p.n_tiles : 0;
    out->exchange = p.xch;
    out->splitk = p.splitk;
    out->split_tiles = p.splitk > 1 ? p.sk_tiles : 0;
    if (p.pair) {
        const int units = ((p.m_tiles + 1) / 2) * p.n_tiles, mc = sm_count / 2;
        out->grid = (units < mc ? units : mc) * 2;
    } else if (p.clustered) {
        const int mc = sm_count / p.cluster;
        out->grid = (p.m_tiles < mc ? p.m_tiles : mc) * p.cluster;
    } else if (p.splitk > 1) {
        const int units = p.sk_base + p.sk_tiles * p.splitk;
        out->grid = units < sm_count ? units : sm_count;
    } else {
        out->grid = out->tiles < sm_count ? out->tiles : sm_count;
    }
    return NF_OK;
}

int nf_abi_version(void) { return NF_ABI_VERSION; }

}  // extern "C"
