// nf_internal.h -- definitions shared by the kernel translation units and the
// host library: tile shapes, the shared-memory layout of each GEMM variant,
// the kernel argument block and the table of compiled variants.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace nf {

// ---------------------------------------------------------------- GEMM tiling
constexpr int TILE_M = 128;               // rows per CTA tile = TMEM lanes
constexpr int TILE_K = 64;                // bf16 K elements per stage = one 128-byte swizzle row
constexpr int UMMA_K = 16;                // K per tcgen05.mma of kind::f16
constexpr int B_BOX_N = 64;               // W is loaded as 64-column boxes (128 bytes per K row)
constexpr int A_STAGE_BYTES = TILE_M * TILE_K * 2;   // 16 KB
constexpr int B_BOX_BYTES = TILE_K * B_BOX_N * 2;    // 8 KB
constexpr int EPI_WARPS = 8;              // two warpgroups of 4: group g drains accumulator g
constexpr int STORE_COLS = 64;            // Y store box: 64 columns x 32 rows (one warp)
constexpr int STORE_ROWS = 32;
constexpr int STORE_BUF_BYTES = STORE_COLS * STORE_ROWS * 2;              // 4 KB
constexpr int STAGING_BYTES = EPI_WARPS * STORE_BUF_BYTES;                 // one box per warp
constexpr int MAX_CLUSTER = 16;           // post-norm: N <= 256 x 16
// Pre-norm with the row sums of squares split over a row's n_tiles >= 2 tiles:
// a tile sums R = ceil(128 / n_tiles) <= 64 rows, 8 R <= 512 16-byte chunks a
// stage, read by one warp in at most 16 loads a lane.
constexpr int SPLIT_SS_ITERS = 16;
constexpr int SMEM_OPTIN_LIMIT = 232448;  // 227 KB of dynamic shared memory per block
constexpr int MAX_STAGES = 8;

enum Epilogue : int {
    EPI_PLAIN = 0,
    EPI_PRE_RMS = 1,
    EPI_POST_LN = 2,
    EPI_POST_RMS = 3,
    EPI_BWD_LN = 4,   // dZ = LayerNorm backward of (X W) from saved statistics
    EPI_BWD_RMS = 5,  // dZ = RMSNorm backward of (X W) from saved statistics
};

// How the CTAs that share an output row exchange partial row statistics
// (post-norm with the row split over several CTAs).
enum Exchange : int {
    XCH_NONE = 0,     // one CTA owns whole rows
    XCH_CLUSTER = 1,  // the row's CTAs form a thread-block cluster; DSMEM
    XCH_GLOBAL = 2,   // the row's CTAs are any CTAs of a co-resident grid; L2
};

// Global-exchange scratch (device memory, zero when first set up), two
// regions whose sizes are fixed when the buffer is set up:
//   xcnt   int: [0] exit count, [2] launch epoch E (the last CTA to leave a
//          launch advances it), [3] row tiles of that launch; from XCH_CNT0
//          two banks of xbank ints, 4 per row tile, of which the first
//          counts the row tile's column tiles.  Launch E counts in bank
//          E & 1, which the launch before it cleared, and clears the other
//          bank, which that launch used: no counter is ever reset while it
//          may be read, and a launch that gave up part-way leaves nothing
//          behind.  A count only says when to look: no fence orders it with
//          the partials, which tell by their tags whether they are current.
//   xpart  (post-norm and its backward) two 64-bit words per (row tile,
//          column tile, tile row), 16-byte aligned: the launch's tag E + 1
//          in each word's high half and one float of the partial -- (mean,
//          M2), (sum of squares, 0) or the backward's two sums -- in its low
//          half.
//   tags   (pre-norm, split sums of squares) one such word per row, the
//          row's sum of squares in its low half.
// Each word is stored and read as one single-copy-atomic access, and E
// never repeats on one scratch buffer, so a word carrying the current tag is
// this launch's: it needs no fence and no clearing.
constexpr int XCH_CNT0 = 64;  // banks start 256 bytes in
__host__ __device__ inline int64_t xch_bank_ints(int m_tiles) { return static_cast<int64_t>(m_tiles) * 4; }
__host__ __device__ inline int64_t xch_stats_bytes(int m_tiles, int n_tiles) {
    return static_cast<int64_t>(m_tiles) * n_tiles * 128 * 16;
}

// Operand layouts (GemmCfg OPS bits).  Default: A K-major (X is M x K
// row-major), B MN-major (W is K x N row-major).
enum OperandFlags : int {
    OPS_A_MN = 1,     // A given as its transpose: X stored K x M row-major (Y = X^T W)
    OPS_A_SCALE = 2,  // with OPS_A_MN: each contraction row m of A scaled by rstd[m] in shared
                      // memory before the MMA (rmsnorm of the stored matrix rebuilt on the fly)
    OPS_B_K = 4,      // B given as its transpose: W stored N x K row-major (Y = X W^T)
    OPS_RESID = 8,    // post-norm: a residual R (M x N) added to X W before the statistics
    OPS_PAIR = 16,    // plain / pre-norm / post-norm with the L2 exchange: a cluster of two CTAs along M
                      // computes a 256-row tile with tcgen05 cta_group::2 MMAs (each CTA loads its 128
                      // rows of A and half of B)
};

template <int EPI, int TILE_N, int XCH, int OPS = 0>
struct GemmCfg {
    static constexpr bool kPre = EPI == EPI_PRE_RMS;
    static constexpr bool kPost = EPI == EPI_POST_LN || EPI == EPI_POST_RMS;
    static constexpr bool kLN = EPI == EPI_POST_LN;
    static constexpr bool kBwd = EPI == EPI_BWD_LN || EPI == EPI_BWD_RMS;
    static constexpr bool kBwdLN = EPI == EPI_BWD_LN;
    static constexpr bool kRow = kPost || kBwd;  // reduces over the output row (N)
    static constexpr bool CLUSTERED = XCH == XCH_CLUSTER;
    static constexpr bool kAMN = (OPS & OPS_A_MN) != 0;
    static constexpr bool kScaleA = (OPS & OPS_A_SCALE) != 0;
    static constexpr bool kBK = (OPS & OPS_B_K) != 0;
    static constexpr bool kRes = (OPS & OPS_RESID) != 0;
    static constexpr bool kPair = (OPS & OPS_PAIR) != 0;
    static_assert(!kPair || (OPS == OPS_PAIR && TILE_N == 256 &&
                             ((EPI == EPI_PLAIN && XCH == XCH_NONE) || EPI == EPI_PRE_RMS ||
                              ((EPI == EPI_POST_LN || EPI == EPI_POST_RMS) && XCH == XCH_GLOBAL))),
                  "the CTA pair is built for plain and pre-norm GEMMs of 256-column tiles and for "
                  "post-norm rows exchanged through L2");
    static_assert(!kRes || kPost, "the residual add belongs to the post-norm epilogues");
    static_assert(!kScaleA || (kAMN && EPI == EPI_PLAIN), "row scaling applies to a transposed A, plain epilogue");
    static_assert(TILE_N == 64 || TILE_N == 128 || TILE_N == 256, "tile_n");
    // Row exchanges: post-norm partial statistics (cluster or L2), or the
    // pre-norm's row sums of squares split over the row's tiles (L2).
    static_assert(XCH == XCH_NONE || (kRow && TILE_N == 256) ||
                      (kPre && XCH == XCH_GLOBAL && TILE_N == 256 && (OPS == 0 || OPS == OPS_PAIR)),
                  "row exchange only for post-norm, or the pre-norm's split sums of squares");

    static constexpr int B_STAGE_BYTES = TILE_K * (kPair ? TILE_N / 2 : TILE_N) * 2;  // this CTA's share of B
    static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
    // per-row partial statistics received from every CTA of the cluster,
    // double buffered by tile parity: [2][MAX_CLUSTER][TILE_M] x float2
    static constexpr int RECV_BYTES = CLUSTERED ? 2 * MAX_CLUSTER * TILE_M * 8 : 0;
    // gamma, beta (bf16) of the CTA's fixed column tile; the global exchange
    // moves across column tiles and keeps one slot per epilogue warpgroup,
    // refilled for each tile.
    static constexpr int AFFINE_BYTES = !kRow ? 0 : (XCH == XCH_GLOBAL ? 2 * (2 * TILE_N * 2) : 2 * TILE_N * 2);
    // TMEM accumulators: four when a tile has <= 128 columns and no row exchange
    // (4 x 128 columns fill TMEM), so the MMA can run up to three tiles ahead of
    // the epilogue, whose two warpgroups each alternate between two of them;
    // two otherwise.
    static constexpr int NACC = (TILE_N <= 128 && XCH == XCH_NONE && OPS == 0) ? 4 : 2;
    // full[8] empty[8] acc_full, acc_empty, ss_full, xch [NACC] mma_done aff_full[2] aff_empty[2]
    static constexpr int NSLOTS = 16 + 4 * NACC + 1 + 4;
    static constexpr int SS_BYTES = kPre ? NACC * TILE_M * 4 : 0;     // sum of squares [NACC][128]
    // A row scaling: each ring stage's 64 rstd values, copied with the stage.
    // (256-column tiles fit four stages at most, narrower ones up to eight.)
    static constexpr int RS_BYTES = kScaleA ? (TILE_N == 256 ? 4 : MAX_STAGES) * TILE_K * 4 : 0;
    // barriers (+ xformed[8], or a pre-norm pair's ardy[8]) + 4 words; the
    // global exchange adds xpub[2] and xrdy[2] after those
    static constexpr int BAR_BYTES = XCH == XCH_GLOBAL ? 352 : ((kScaleA || kPair || NACC == 4) ? 320 : 256);
    // The swizzled buffers need a 1 KB aligned base.  Dynamic shared memory
    // starts 1 KB aligned in practice; the global-exchange variant, whose
    // fourth pipeline stage needs the room, relies on that (and checks it at
    // run time), the others keep 1 KB of slack to realign.
    static constexpr int ALIGN_SLACK = XCH == XCH_GLOBAL ? 0 : 1024;
    static constexpr int FIXED_BYTES =
        ALIGN_SLACK + STAGING_BYTES + RECV_BYTES + AFFINE_BYTES + SS_BYTES + RS_BYTES + BAR_BYTES;
    static constexpr int STAGES_FIT = (SMEM_OPTIN_LIMIT - FIXED_BYTES) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > MAX_STAGES ? MAX_STAGES : STAGES_FIT;
    static_assert(STAGES >= 2, "pipeline needs two stages");
    static_assert(!kScaleA || RS_BYTES >= STAGES * TILE_K * 4, "one rstd slot per stage");
    static constexpr int SMEM_BYTES = FIXED_BYTES + STAGES * STAGE_BYTES;

    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_STAGE_BYTES;
    static constexpr int OFF_STG = OFF_B + STAGES * B_STAGE_BYTES;
    static constexpr int OFF_RECV = OFF_STG + STAGING_BYTES;
    static constexpr int OFF_AFF = OFF_RECV + RECV_BYTES;
    static constexpr int OFF_SS = OFF_AFF + AFFINE_BYTES;
    static constexpr int OFF_RS = OFF_SS + SS_BYTES;
    static constexpr int OFF_BAR = OFF_RS + RS_BYTES;
    static_assert(OFF_B % 1024 == 0 && OFF_STG % 1024 == 0, "swizzled buffers need 1 KB alignment");
    static_assert(NSLOTS * 8 + 16 <= (kScaleA ? 256 : BAR_BYTES), "barrier area + 4 words");
    static_assert(!kScaleA || 256 + 8 * 8 <= BAR_BYTES, "xformed[8] after the barrier area");

    static constexpr int PRODUCER_WARP = EPI_WARPS;       // 8
    static constexpr int MMA_WARP = EPI_WARPS + 1;        // 9
    static constexpr int SUMSQ_WARP0 = EPI_WARPS + 2;     // pre-norm: sum-of-squares warps 10-13;
                                                          // A row scaling: transform warps 10-13
    static constexpr int THREADS = (kPre || kScaleA ? EPI_WARPS + 6 : EPI_WARPS + 2) * 32;
    static constexpr int TMEM_COLS = NACC * TILE_N;        // the accumulator buffers
};

// Kernel argument block (passed by value).
struct GemmArgs {
    int32_t M, N, K;
    int32_t m_tiles, n_tiles, k_tiles;
    int32_t cluster;        // CTAs per cluster along N (1 = no cluster)
    int32_t units;          // unclustered: work units (tiles, with the last wave's tiles halved);
                            // CTA pair: 256-row pair tiles (ceil(m_tiles / 2) x n_tiles)
    int32_t split_base;     // unclustered: first half-tile unit (== units when nothing is split)
    float eps;
    float inv_len;          // 1/K (pre-norm) or 1/N (post-norm)
    const uint16_t* gamma;  // bf16, N entries, or null
    const uint16_t* beta;   // bf16, N entries, or null
    float* mean_out;        // M entries or null
    float* rstd_out;        // M entries or null
    uint32_t* status;       // device status word (4 x u32)
    uint64_t timeout_ns;
    const uint16_t* zin;    // backward: Z, M x N bf16 (the forward's norm input)
    const float* mean_in;   // backward LN: saved row means (M)
    const float* rstd_in;   // backward: saved row rstd (M); OPS_A_SCALE: rstd per contraction row (K)
    int* xcnt;              // global exchange only: XCH_CNT0 + 2 * xbank ints
    int32_t xbank;          // ints per counter bank, >= xch_bank_ints(m_tiles)
    unsigned long long* xpart;  // post-norm global exchange: >= xch_stats_bytes(m_tiles, n_tiles)
    int32_t splitk;         // plain GEMM: contraction slices of the split tiles (1 = none)
    int32_t sk_base;        // splitk > 1: first split unit (= first split tile); units before it are whole tiles
    int32_t sk_tiles;       // splitk > 1: split tiles (sk_base .. sk_base + sk_tiles - 1), each in splitk units
    float* ws;              // splitk > 1: fp32 partial tiles, [splitk][sk_tiles][TILE_M][TILE_N]
    unsigned long long* sstag;  // pre-norm, split sums of squares: one word per row, (launch tag << 32) | bits
                                // of the row's sum of squares, >= m_tiles * 128 words
    uint16_t* xhat_out;     // RMS backward (optional): bf16(Z * rstd), M x N, the rebuilt rmsnorm input
    const uint16_t* resid;  // post-norm (optional): R, M x N bf16, added to X W before the statistics
    uint16_t* h_out;        // with resid (optional): bf16(X W + R), M x N, the updated residual stream
};

// Wait sites recorded in the status word on a time-out.
enum WaitSite : uint32_t {
    SITE_PROD_EMPTY = 1,
    SITE_MMA_ACC_EMPTY = 2,
    SITE_MMA_FULL = 3,
    SITE_EPI_ACC_FULL = 4,
    SITE_EPI_SS_FULL = 5,
    SITE_EPI_XCH = 6,
    SITE_SS_FULL = 7,
    SITE_SS_ACC_EMPTY = 8,
    SITE_SELFTEST = 9,
    SITE_EPI_PAIR = 10,
    SITE_EPI_GXCH = 11,
    SITE_EPI_AFF = 12,
    SITE_SMEM_ALIGN = 13,  // code NF_ERR_ALIGNMENT: dynamic shared memory not 1 KB aligned
    SITE_CLUSTER_SHAPE = 14,  // code NF_ERR_INVALID_ARG: launched with a cluster size the variant does not use
    SITE_SPLIT_SS = 15,  // code NF_ERR_INVALID_ARG: pre-norm split sums of squares with fewer than two tiles a row
};

// One compiled GEMM variant.
struct GemmVariant {
    int epi, tile_n;
    bool clustered;  // xch == XCH_CLUSTER
    int xch;
    bool pair;       // OPS_PAIR: launched in clusters of two CTAs along M
    int ops;         // OperandFlags
    const void* func;
    int threads, smem_bytes, stages, tmem_cols;
    int tile_k;  // K per ring stage: 64 (X boxes 128-byte swizzled) or 32 (64-byte swizzled)
};

// Tables exported by the kernel translation units.
const GemmVariant* gemm_variants_plain(int* count);
const GemmVariant* gemm_variants_pre(int* count);
const GemmVariant* gemm_variants_post_ln(int* count);
const GemmVariant* gemm_variants_post_rms(int* count);
const GemmVariant* gemm_variants_bwd_ln(int* count);
const GemmVariant* gemm_variants_bwd_rms(int* count);
const GemmVariant* gemm_variants_trans_plain(int* count);  // plain GEMMs with OperandFlags
const GemmVariant* gemm_variants_trans_bwd(int* count);    // RMS-backward epilogue over X W^T
const GemmVariant* gemm_variants_res_ln(int* count);       // post-norm LayerNorm with a residual add
const GemmVariant* gemm_variants_res_rms(int* count);      // post-norm RMSNorm with a residual add

// ---------------------------------------------------------------- row norm
struct NormArgs {
    const void* in;
    void* out;
    const uint16_t* gamma;
    const uint16_t* beta;
    int64_t rows;
    int32_t cols;
    float eps;
    float inv_cols;
    float* mean_out;
    float* rstd_out;
    const void* res;        // optional residual (rows x cols bf16) added to `in` before the norm
    void* h_out;            // with res (optional): bf16(in + res), rows x cols
};

// Picks the variant for `cols` and launches it; returns the CUDA status.
cudaError_t launch_norm_rows(const NormArgs& a, int kind, int sm_count, bool overlap, cudaStream_t stream);

// Backward of the row normalization from saved statistics.
struct NormBwdArgs {
    const void* dy;        // rows x cols bf16
    const void* z;         // rows x cols bf16, the forward's norm input
    const uint16_t* gamma;  // bf16, cols entries, or null
    const float* mean;     // rows entries (LN), may be null for RMS
    const float* rstd;     // rows entries
    void* dz;              // rows x cols bf16
    int64_t rows;
    int32_t cols;
    float inv_cols;
};
cudaError_t launch_norm_rows_bwd(const NormBwdArgs& a, int kind, int sm_count, bool overlap, cudaStream_t stream);
// Largest supported cols.
constexpr int NORM_MAX_COLS = 16384;

// FlashNormAttention forward (nf_flashnorm.cu): head dimension and key /
// value length 128, up to 8 heads (one cluster of H CTAs per batch).
struct FlashNormLaunch {
    const int32_t* q_len;  // B entries or null
    int32_t B, Lq, H, act;
    float eps1, eps2;
    uint32_t* status;
    uint64_t timeout_ns;
};
// tmaps: four CUtensorMap, Q / K / V / Out viewed as [rows, H * 128] bf16 with
// the 128-byte swizzle and boxes {64, 128}, {64, 128}, {64, 64}, {64, 32}.
cudaError_t launch_flashnorm_fwd(const void* tmaps, const FlashNormLaunch& a, bool overlap, cudaStream_t stream);

// Split-K: for each split tile t = sk_base + i (i < sk_tiles), Y's tile
// (TILE_M x tile_n at row tile t / n_tiles, column tile t % n_tiles) in bf16 =
// the sum over `slices` of the fp32 partial tiles ws[s][i], added in slice
// order; only elements inside M x N are written.  N % 8 == 0.
struct SplitkReduceArgs {
    const float* ws;
    uint16_t* y;
    int32_t slices, sk_base, sk_tiles, n_tiles, tile_n;
    int32_t M, N;
};
cudaError_t launch_splitk_reduce(const SplitkReduceArgs& a, int sm_count, bool overlap, cudaStream_t stream);

}  // namespace nf
