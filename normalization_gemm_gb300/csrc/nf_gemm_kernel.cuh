// nf_gemm_kernel.cuh -- persistent, warp-specialized bf16 GEMM for sm_103a with
// the row normalization fused in.  One template covers the four epilogues:
//
//   EPI_PLAIN     Y = X W                         (blog §1 baseline GEMM)
//   EPI_PRE_RMS   Y = rstd(X) * (X W)              (blog §2 Lazy Pre-Norm)
//   EPI_POST_LN   Y = LayerNorm(X W) * g + b       (blog §3 Multi-CTA Norm)
//   EPI_POST_RMS  Y = RMSNorm(X W) * g             (blog §3 with RMSNorm)
//   EPI_BWD_LN    dZ = LayerNorm backward of dY = X W, from saved row
//   EPI_BWD_RMS   statistics (blog §3 "What about backward? Fusion
//                 regrouping": the norm's backward in the epilogue of the
//                 GEMM that produces its incoming gradient)
//
// Blog: "Towards Free Normalization: Fusing Normalization into GEMM and
// Attention Kernels".
//
// CTA roles (one CTA per SM, persistent over output tiles):
//   warps 0-7  epilogue, two warpgroups that alternate tiles: warp w of group
//              g = w / 4 reads TMEM lanes 32(w%4)..+31 of accumulator g, i.e.
//              one tile row per thread; normalizes; stores through a
//              128B-swizzled staging buffer with TMA, once per element.
//   warp 8     TMA producer (one elected lane): X and W K-tiles into a ring of
//              STAGES shared-memory stages.
//   warp 9     MMA issuer (one elected lane): tcgen05.mma 128 x TILE_N x 16
//              into one of NACC TMEM accumulators (two, or four for tiles of
//              <= 128 columns without a row exchange) so that the epilogue of
//              tile t overlaps the main loops of the tiles after it.
//   warps 10-13 (pre-norm only) sum of squares of each X row, read from the
//              same shared-memory stage the tensor cores consume, on CUDA
//              cores, in parallel with the MMA (blog §2 pseudocode:
//              square_sum += (tile_A * tile_A).sum(-1)); with the sums split
//              over a row's tiles, warp 10 alone sums the tile's share of rows.
//
// Shared-memory operands (128-byte swizzle, 1 KB aligned):
//   A stage  128 rows x 64 K, K-major: row r at r*128 bytes.
//   B stage  TILE_N/64 boxes of 64 K-rows x 64 N (MN-major, W is row-major
//            K x N), box i at i*8 KB, K-row k of a box at k*128 bytes.
//
// Waits on barriers that a remote event may complete (a CTA pair's full[s],
// whose bytes come from both CTAs; the first CTA's commits arriving in the
// second CTA) poll without the suspend-time hint; the first CTA waits for the
// peer's once-per-tile relay with test_wait (mbar_wait_remote).
//
// Pipeline barriers: full[s] (TMA bytes landed), empty[s] (MMA done with the
// stage; pre-norm: also all 128 sum-of-squares threads), acc_full[b] (MMA
// chain of a tile complete), acc_empty[b] (epilogue drained TMEM buffer b),
// ss_full[b] (row sums of squares of the tile ready), xch[b] (all partial row
// statistics of the cluster arrived).  Every wait is bounded in time; on
// expiry the kernel records NF_ERR_TIMEOUT, drains what it issued, frees TMEM
// and returns.
//
// CTA pair (OPS_PAIR: plain, pre-norm and globally exchanging post-norm GEMMs
// of 256-column tiles): a cluster of two CTAs along M computes a 256 x 256 tile with tcgen05
// cta_group::2 MMAs.  Each CTA's producer loads its own 128 rows of A and half
// of B's 256 columns into its own ring stage (32 KB instead of 48, so six
// stages fit), counted on the first CTA's full barrier; the first CTA's MMA
// thread issues the MMAs, which read both CTAs' stages and write each CTA's
// 128 rows into that CTA's TMEM, and its commits arrive on the barriers of
// both CTAs.  The second CTA's MMA warp relays its epilogue's "accumulator
// drained" to the first CTA.  Pre-norm: a sum-of-squares thread of the first
// CTA, once full[s] shows both CTAs' bytes landed, tells the second CTA's
// sum-of-squares warps (ardy[s]) with a relaxed remote arrive.  (Measured: with
// every tile summing all its rows the pre-norm pair runs no faster than one CTA
// per tile -- the plan pairs pre-norm GEMMs only with the split sums -- while a
// release arrive per stage, or a first CTA summing its peer's rows through
// distributed shared memory, was three times slower.)  Each CTA's epilogue is
// unchanged.
//
// Post-norm rows wider than one tile exchange partial row statistics between
// the CTAs that hold the row (XCH):
//   XCH_CLUSTER  the row's CTAs form a thread-block cluster along N and push
//                their partials into every peer's shared memory (DSMEM), as
//                in blog §3.
//   XCH_GLOBAL   the row's tiles are ordinary tiles of a persistent grid whose
//                CTAs are all resident at once (cooperative launch); partials
//                go through L2 as tagged words, with an arrival counter per
//                row tile that only says when to read them (no fence).
//                Tile t runs on CTA t mod G in order, G >= n_tiles / 2, so a
//                CTA's tiles t_i and t_{i-2} (which share a TMEM buffer) lie in
//                different row tiles and every wait points at an earlier row
//                tile: the exchange cannot deadlock.  This uses every SM,
//                whereas clusters of 8 or 16 co-reside on fewer of them.
#pragma once

#include <type_traits>

#include "nf_internal.h"
#include "nf_ptx.cuh"


// The producer loads W's tiles, which every wave of tiles reads again, with an
// evict-last L2 policy.
#ifndef NF_W_EVICT_LAST
#define NF_W_EVICT_LAST 1
#endif

namespace nf {

// Bounded wait used only while draining: ignores the abort flag and records
// nothing.
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > timeout_ns) return;
    }
}

__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t num_clusters_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// Keeps the compiler from using r[] before an earlier asm statement.
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31]));
}

// Loads NC 32-column chunks of this thread's TMEM lane starting at `taddr`,
// then waits once for all of them.
template <int NC>
__device__ __forceinline__ void tmem_load_seg(uint32_t taddr, uint32_t (&v)[NC][32]) {
#pragma unroll
    for (int c = 0; c < NC; ++c) tmem_ld32(taddr + static_cast<uint32_t>(c * 32), v[c]);
    tmem_ld_wait(v[0]);
#pragma unroll
    for (int c = 1; c < NC; ++c) reg_fence(v[c]);
}

// Bounded per-thread wait for a 64-bit word whose high half is `tag`; the
// word is returned in `w`.  False when the CTA is aborting or the time limit
// passed (recorded).
__device__ __forceinline__ bool tagged_wait(const WaitGuard& g, const unsigned long long* p, unsigned long long tag,
                                            unsigned long long& w, uint32_t site, uint32_t tile) {
    w = ld_relaxed_gpu_u64(p);
    if ((w & 0xffffffff00000000ull) == tag) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        __nanosleep(64);
        w = ld_relaxed_gpu_u64(p);
        if ((w & 0xffffffff00000000ull) == tag) return true;
        if (*g.abort_flag) return false;
        if (globaltimer_ns() - t0 > g.timeout_ns) {
            record_failure(g, 5u /* NF_ERR_TIMEOUT */, site, tile);
            return false;
        }
    }
}

// Where the epilogue finds gamma / beta.
enum AffSrc : int { AFF_NONE = 0, AFF_SMEM = 1 };

// 64 fp32 columns (two 32-column chunks) -> 32 packed bf16 pairs:
// y = x * scale + bias, then y * gamma + beta unless AFF == AFF_NONE (gamma /
// beta as bf16 in shared memory at saff_g / saff_b, 8 columns per 16-byte
// load).  Works on fp32 pairs: one f32x2 FMA per two columns.
template <int AFF>
__device__ __forceinline__ void convert64(const uint32_t (&va)[32], const uint32_t (&vb)[32], uint64_t scale2,
                                          uint64_t bias2, uint32_t saff_g, uint32_t saff_b, uint32_t (&pk)[32]) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const uint32_t* src = q < 4 ? va : vb;
        const int o = (q & 3) * 8;
        uint64_t y[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) y[e] = f2_fma(f2_pack(src[o + 2 * e], src[o + 2 * e + 1]), scale2, bias2);
        if (AFF != AFF_NONE) {
            const uint4 g = ld_shared_v4(saff_g + static_cast<uint32_t>(q * 16));
            const uint4 t = ld_shared_v4(saff_b + static_cast<uint32_t>(q * 16));
            y[0] = f2_fma(y[0], bf16x2_to_f2(g.x), bf16x2_to_f2(t.x));
            y[1] = f2_fma(y[1], bf16x2_to_f2(g.y), bf16x2_to_f2(t.y));
            y[2] = f2_fma(y[2], bf16x2_to_f2(g.z), bf16x2_to_f2(t.z));
            y[3] = f2_fma(y[3], bf16x2_to_f2(g.w), bf16x2_to_f2(t.w));
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float lo, hi;
            f2_unpack(y[e], lo, hi);
            pk[4 * q + e] = pack_bf16x2(lo, hi);
        }
    }
}

// Backward of 64 columns (two 32-column chunks of dY = X W) -> 32 packed
// bf16 pairs: dz = g * rstd + z * c1 + c0 with g = dY * gamma (AFF; gamma as
// bf16 in shared memory at saff_g) and z the saved forward input (zq, 64 bf16).
template <bool AFF>
__device__ __forceinline__ void convert64_bwd(const uint32_t (&va)[32], const uint32_t (&vb)[32],
                                              const uint4 (&zq)[8], uint32_t saff_g, uint64_t rs2, uint64_t c12,
                                              uint64_t c02, uint32_t (&pk)[32]) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const uint32_t* src = q < 4 ? va : vb;
        const int o = (q & 3) * 8;
        const uint32_t zw[4] = {zq[q].x, zq[q].y, zq[q].z, zq[q].w};
        uint32_t gw[4] = {0u, 0u, 0u, 0u};
        if (AFF) {
            const uint4 g = ld_shared_v4(saff_g + static_cast<uint32_t>(q * 16));
            gw[0] = g.x, gw[1] = g.y, gw[2] = g.z, gw[3] = g.w;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            uint64_t x2 = f2_pack(src[o + 2 * e], src[o + 2 * e + 1]);
            if (AFF) x2 = f2_fma(x2, bf16x2_to_f2(gw[e]), 0ull);
            const uint64_t y = f2_fma(x2, rs2, f2_fma(bf16x2_to_f2(zw[e]), c12, c02));
            float lo, hi;
            f2_unpack(y, lo, hi);
            pk[4 * q + e] = pack_bf16x2(lo, hi);
        }
    }
}

// 64 bf16 of a row of Z starting at p (16-byte aligned); 8-column groups at or
// past `valid` read as zero (N is a multiple of 8).  One thread per row: the
// loads of a segment can be issued ahead of the TMEM reads they pair with.
__device__ __forceinline__ void load_z64(const uint16_t* p, bool own, int valid, uint4 (&zq)[8]) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
        zq[q] = (own && q * 8 < valid) ? __ldg(reinterpret_cast<const uint4*>(p + q * 8)) : make_uint4(0, 0, 0, 0);
}

// A warp's 32 x 64 bf16 block through its 4 KB staging buffer (128-byte
// rows, 16-byte chunk e of row r at r * 128 + ((e ^ (r & 7)) << 4), the
// layout of the output staging).  Global memory is touched coalesced: lane l
// moves chunk l & 7 of rows (l >> 3) + 4 i, i.e. 4 full 128-byte lines per
// instruction, instead of one thread per row (32 lines per instruction).
// Rows at or past `nrows` and 8-column groups at or past `valid` read as
// zero and are not written.  Loads go through L2 (not the read-only path):
// the residual output may overwrite the residual in place, each block after
// it was read here.
__device__ __forceinline__ void stage_in64(uint32_t buf, const uint16_t* p, int64_t ld, int nrows, int valid,
                                           int lane) {
    const int c = lane & 7;
    uint4 q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = (lane >> 3) + 4 * i;
        q[i] = (r < nrows && c * 8 < valid) ? __ldcg(reinterpret_cast<const uint4*>(p + r * ld + c * 8))
                                            : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = (lane >> 3) + 4 * i;
        st_shared_v4(buf + static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4)), q[i].x, q[i].y, q[i].z, q[i].w);
    }
}

__device__ __forceinline__ void stage_out64(uint32_t buf, uint16_t* p, int64_t ld, int nrows, int valid, int lane) {
    const int c = lane & 7;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = (lane >> 3) + 4 * i;
        const uint4 q = ld_shared_v4(buf + static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4)));
        if (r < nrows && c * 8 < valid) *reinterpret_cast<uint4*>(p + r * ld + c * 8) = q;
    }
}

// v (64 fp32 columns of this lane's row, two 32-column chunks) += the row's 64
// bf16 in the staging buffer.
__device__ __forceinline__ void add_staged_row(uint32_t buf, int lane, uint32_t (&v)[2][32]) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const uint4 rq = ld_shared_v4(buf + static_cast<uint32_t>(lane * 128 + ((e ^ (lane & 7)) << 4)));
        const uint32_t rw[4] = {rq.x, rq.y, rq.z, rq.w};
        uint32_t* d = &v[e >> 2][(e & 3) * 8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            d[2 * k] = __float_as_uint(__uint_as_float(d[2 * k]) + bf16lo(rw[k]));
            d[2 * k + 1] = __float_as_uint(__uint_as_float(d[2 * k + 1]) + bf16hi(rw[k]));
        }
    }
}

// The row's 64 fp32 columns -> bf16 into the staging buffer (same layout).
__device__ __forceinline__ void put_staged_row(uint32_t buf, int lane, const uint32_t (&v)[2][32]) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const uint32_t* s = &v[e >> 2][(e & 3) * 8];
        st_shared_v4(buf + static_cast<uint32_t>(lane * 128 + ((e ^ (lane & 7)) << 4)),
                     pack_bf16x2(__uint_as_float(s[0]), __uint_as_float(s[1])),
                     pack_bf16x2(__uint_as_float(s[2]), __uint_as_float(s[3])),
                     pack_bf16x2(__uint_as_float(s[4]), __uint_as_float(s[5])),
                     pack_bf16x2(__uint_as_float(s[6]), __uint_as_float(s[7])));
    }
}

// Tile schedule: CTA-local work unit lt -> (m_tile, n_tile, first row, rows).
// Unclustered launches walk linear units; units from split_base on are the
// tiles of the last, partial wave cut into two 64-row halves, so that wave
// spreads over twice as many SMs.  A half still runs the 128-row MMA (the X
// box simply starts 64 rows further for the second half); only its own 64
// rows are stored.  A split-K launch (splitk > 1, plain GEMM) runs units
// [0, sk_base) as whole tiles and splits the sk_tiles tiles from sk_base on
// over the contraction, slice-major: unit sk_base + j is tile
// sk_base + j mod sk_tiles over slice s = j / sk_tiles, K-tiles
// [s k_tiles / splitk, (s+1) k_tiles / splitk).  (sk_base = 0 splits every
// tile; sk_base > 0 only the last, partial wave.)
struct TileSched {
    int first, step, count;  // m (clustered) or linear unit (unclustered) sequence
    int n_fixed;             // clustered: this CTA's n tile (its cluster rank)
    int n_tiles;
    int split_base;          // first half-tile unit (unclustered)
    int sk_base, sk_tiles;   // split-K: first split unit / tile, split tiles
    int splitk;              // contraction slices of the split tiles
    int k_tiles;
    bool clustered;
    bool pair;               // CTA pair: unit u is pair tile (u / n_tiles, u % n_tiles), this CTA's rows
    int pair_rank;           // 0 or 1: the pair tile's first or second 128 rows
    bool kflip;              // odd local units walk the contraction backwards
    // K-tiles of unit lt and its slice (-1 for a whole tile).
    __device__ __forceinline__ void krange(int lt, int& kt0, int& kt1, int& slice) const {
        const int u = first + lt * step;
        if (splitk <= 1 || u < sk_base) {
            kt0 = 0;
            kt1 = k_tiles;
            slice = -1;
            return;
        }
        slice = (u - sk_base) / sk_tiles;
        kt0 = static_cast<int>(static_cast<int64_t>(slice) * k_tiles / splitk);
        kt1 = static_cast<int>(static_cast<int64_t>(slice + 1) * k_tiles / splitk);
    }
    // Contraction step i of unit lt.  With kflip, every odd local unit walks
    // its K-tiles from the last down: a CTA's consecutive units are one wave
    // apart, so the next wave starts on the operand panels the previous one
    // read last, which L2 still holds.  (All CTAs of a wave walk the same way,
    // so CTAs sharing a panel still request it in step.)
    __device__ __forceinline__ int kstep(int lt, int kt0, int kt1, int i) const {
        return (kflip && (lt & 1)) ? kt1 - 1 - i : kt0 + i;
    }
    __device__ __forceinline__ void tile(int lt, int& m, int& n, int& row0, int& rows) const {
        int u = first + lt * step;
        if (splitk > 1 && u >= sk_base) u = sk_base + (u - sk_base) % sk_tiles;
        if (pair) {
            const int mp = u / n_tiles;
            n = u - mp * n_tiles;
            m = 2 * mp + pair_rank;
            row0 = m * TILE_M;
            rows = TILE_M;
            return;
        }
        if (clustered) {
            m = u;
            n = n_fixed;
            row0 = m * TILE_M;
            rows = TILE_M;
            return;
        }
        int t = u, half = -1;
        if (u >= split_base) {
            t = split_base + ((u - split_base) >> 1);
            half = (u - split_base) & 1;
        }
        m = t / n_tiles;
        n = t - m * n_tiles;
        row0 = m * TILE_M + (half == 1 ? TILE_M / 2 : 0);
        rows = half < 0 ? TILE_M : TILE_M / 2;
    }
};

template <int EPI, int TILE_N, int XCH, int OPS = 0>
__global__ void __launch_bounds__(GemmCfg<EPI, TILE_N, XCH, OPS>::THREADS, 1)
    nf_gemm_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                   const __grid_constant__ CUtensorMap tmY, const GemmArgs args) {
    using Cfg = GemmCfg<EPI, TILE_N, XCH, OPS>;
    constexpr bool CLUSTERED = XCH == XCH_CLUSTER;
    constexpr bool GLOBALX = XCH == XCH_GLOBAL;
    constexpr bool PAIR = Cfg::kPair;
    constexpr int STAGES = Cfg::STAGES;
    constexpr int NBOX = TILE_N / B_BOX_N;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    if (Cfg::ALIGN_SLACK == 0 && (raw & 1023u) != 0) {
        // No room to realign: report and leave before touching anything.
        if (threadIdx.x == 0 && atomicCAS(&args.status[0], 0u, 2u /* NF_ERR_ALIGNMENT */) == 0u) {
            atomicExch(&args.status[1], SITE_SMEM_ALIGN);
            atomicExch(&args.status[2], blockIdx.x);
        }
        return;
    }
    if (PAIR || CLUSTERED) {
        // The pair and row-cluster forms address their peers' shared memory and
        // (pairs) issue cta_group::2 instructions: a launch whose cluster is not
        // the one they were planned for leaves, reporting it, before any of that.
        const uint32_t want = PAIR ? 2u : static_cast<uint32_t>(args.cluster);
        if (cluster_nctarank() != want) {
            if (threadIdx.x == 0 && atomicCAS(&args.status[0], 0u, 1u /* NF_ERR_INVALID_ARG */) == 0u) {
                atomicExch(&args.status[1], SITE_CLUSTER_SHAPE);
                atomicExch(&args.status[2], blockIdx.x);
            }
            return;
        }
    }
    if (Cfg::kPre && GLOBALX && args.n_tiles < 2) {
        // Split sums of squares: two or more tiles a row keep each tile's share
        // within SPLIT_SS_ITERS loads a lane and stage.
        if (threadIdx.x == 0 && atomicCAS(&args.status[0], 0u, 1u /* NF_ERR_INVALID_ARG */) == 0u) {
            atomicExch(&args.status[1], SITE_SPLIT_SS);
            atomicExch(&args.status[2], blockIdx.x);
        }
        return;
    }
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const base_ptr = smem_raw + (base - raw);

    const uint32_t sA = base + Cfg::OFF_A;
    const uint32_t sB = base + Cfg::OFF_B;
    const uint32_t sStg = base + Cfg::OFF_STG;
    const uint32_t sRecv = base + Cfg::OFF_RECV;
    const uint32_t sBar = base + Cfg::OFF_BAR;
    const uint32_t sRS = base + Cfg::OFF_RS;  // A row scaling: rstd of each stage's 64 K-rows
    const uint32_t bar_full0 = sBar;             // [8]
    const uint32_t bar_empty0 = sBar + 8u * 8;   // [8]
    constexpr int NACC = Cfg::NACC;
    const uint32_t bar_accf0 = sBar + 8u * 16;               // [NACC]
    const uint32_t bar_acce0 = bar_accf0 + 8u * NACC;        // [NACC]
    const uint32_t bar_ssf0 = bar_acce0 + 8u * NACC;         // [NACC]
    const uint32_t bar_xch0 = bar_ssf0 + 8u * NACC;          // [NACC]
    const uint32_t bar_mma_done = bar_xch0 + 8u * NACC;
    const uint32_t bar_xf0 = sBar + 256u;        // [8] A row scaling: stage s transformed
    const uint32_t bar_pacc0 = bar_xch0;         // [NACC] CTA pair (first CTA): the peer's epilogue drained buffer b
    const uint32_t bar_ardy0 = sBar + 256u;      // [8] pre-norm CTA pair (second CTA): its A stage s has landed

    const uint32_t bar_afff0 = bar_mma_done + 8u;  // [2] global exchange: a group's affine slot filled
    const uint32_t bar_affe0 = bar_afff0 + 16u;    // [2] global exchange: a group's affine slot free
    const uint32_t bar_xpub0 = sBar + 320u;        // [2] global exchange: a group's 4 warps stored their partials
    const uint32_t bar_xrdy0 = sBar + 336u;        // [2] global exchange: the row tile's partials may be read
    uint32_t* const tmem_holder = reinterpret_cast<uint32_t*>(base_ptr + Cfg::OFF_BAR + 8 * Cfg::NSLOTS);
    volatile int* const abort_flag =
        reinterpret_cast<volatile int*>(base_ptr + Cfg::OFF_BAR + 8 * Cfg::NSLOTS + 4);
    float* const ss_buf = reinterpret_cast<float*>(base_ptr + Cfg::OFF_SS);
    uint16_t* const aff = reinterpret_cast<uint16_t*>(base_ptr + Cfg::OFF_AFF);
    volatile int* const epoch_sm =  // global exchange: launch epoch and the last launch's counter count
        reinterpret_cast<volatile int*>(base_ptr + Cfg::OFF_BAR + 8 * Cfg::NSLOTS + 8);

    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int lane = static_cast<int>(threadIdx.x & 31);
    const WaitGuard guard{args.status, abort_flag, args.timeout_ns};

    // ---- tile schedule
    TileSched sched;
    sched.clustered = CLUSTERED;
    sched.n_tiles = args.n_tiles;
    int my_rank = 0;
    sched.pair = PAIR;
    sched.pair_rank = 0;
    sched.kflip = Cfg::kAMN;
    if (PAIR) {
        my_rank = static_cast<int>(cluster_ctarank());
        const int cid = static_cast<int>(cluster_id_x());
        const int ncl = static_cast<int>(num_clusters_x());
        const int total = args.units;  // pair tiles
        sched.first = cid;
        sched.step = ncl;
        sched.count = cid < total ? (total - cid + ncl - 1) / ncl : 0;
        sched.n_fixed = 0;
        sched.split_base = total;
        sched.pair_rank = my_rank & 1;
    } else if (CLUSTERED) {
        my_rank = static_cast<int>(cluster_ctarank());
        const int cid = static_cast<int>(cluster_id_x());
        const int ncl = static_cast<int>(num_clusters_x());
        sched.first = cid;
        sched.step = ncl;
        sched.count = cid < args.m_tiles ? (args.m_tiles - cid + ncl - 1) / ncl : 0;
        sched.n_fixed = my_rank;
    } else {
        const int total = args.units;
        const int b = static_cast<int>(blockIdx.x);
        const int g = static_cast<int>(gridDim.x);
        sched.first = b;
        sched.step = g;
        sched.count = b < total ? (total - b + g - 1) / g : 0;
        sched.n_fixed = 0;
        sched.split_base = args.split_base;
    }
    sched.sk_base = args.sk_base;
    sched.sk_tiles = args.sk_tiles;
    sched.splitk = args.splitk;
    sched.k_tiles = args.k_tiles;
    const int count = sched.count;
    const int k_tiles = args.k_tiles;
    const bool lead = !PAIR || (my_rank & 1) == 0;  // CTA pair: the first CTA issues the MMAs
    const uint32_t xch_bytes = static_cast<uint32_t>(args.cluster) * TILE_M * 8u;

    // ---- set-up: barriers, TMEM, affine parameters
    if (threadIdx.x == 0) {
        // The tensor maps are kernel parameters, independent of any earlier
        // grid: fetch them while a preceding kernel may still be running.
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmW);
        prefetch_tmap(&tmY);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full0 + 8u * s, 1);
            // (pre-norm: and the sum-of-squares threads, or, with the sums
            // split over the row's tiles, its one sum-of-squares warp)
            mbar_init(bar_empty0 + 8u * s, 1 + (Cfg::kPre ? (GLOBALX ? 1 : 128) : 0));
        }
        for (int b = 0; b < NACC; ++b) {
            mbar_init(bar_accf0 + 8u * b, 1);
            mbar_init(bar_acce0 + 8u * b, 128);
            mbar_init(bar_ssf0 + 8u * b, 128);
            mbar_init(bar_xch0 + 8u * b, 1);  // (CTA pair: bar_pacc, one relayed arrival)
        }

        mbar_init(bar_mma_done, 1);
        if (PAIR && Cfg::kPre)
            for (int st = 0; st < STAGES; ++st) mbar_init(bar_ardy0 + 8u * st, 1);
        if (Cfg::kScaleA)
            for (int st = 0; st < STAGES; ++st) mbar_init(bar_xf0 + 8u * st, 128);  // the transform threads
        for (int g = 0; g < 2; ++g) {
            mbar_init(bar_afff0 + 8u * g, 4);  // one arrival per warp of the group
            mbar_init(bar_affe0 + 8u * g, 4);
            if (GLOBALX) {
                mbar_init(bar_xpub0 + 8u * g, 4);
                mbar_init(bar_xrdy0 + 8u * g, 1);
            }
        }
        *abort_flag = 0;
        fence_mbar_init();
        if (CLUSTERED) {
            // Arm the exchange barriers for local tiles 0 and 1 before any peer
            // can send (peers send only after the cluster barrier below).
            for (int b = 0; b < 2 && b < count; ++b) mbar_arrive_expect_tx(bar_xch0 + 8u * b, xch_bytes);
        }
    }
    if (warp == Cfg::PRODUCER_WARP) {
        if (PAIR) {  // the same columns in both CTAs of the pair
            tmem_alloc_pair(smem_u32(tmem_holder), Cfg::TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_holder), Cfg::TMEM_COLS);
            tmem_relinquish();
        }
    }
    // Warm L2 with this CTA's first ring-full of X K-tiles while a preceding
    // grid may still be running.  A prefetch only fills L2 lines, and L2 is
    // where that grid's writes land, so the loads below never see stale data.
    // The first use of a tensor map waits for its descriptor (about a
    // microsecond); the MMA warp, idle until the first stage lands, takes that
    // wait so the producer reaches its first load sooner (measured: -1.5 % at
    // 65536x128x128).  The pre-norm kernel keeps it on the producer (+1.3 % at
    // 8192x4096x4096 otherwise).
    constexpr int PF_WARP = Cfg::kPre ? Cfg::PRODUCER_WARP : Cfg::MMA_WARP;
    if (warp == PF_WARP && lane == 0 && count > 0) {
        int lt = 0, kt0, kt1, slice;
        sched.krange(0, kt0, kt1, slice);
        int ki = 0;
        for (int i = 0; i < STAGES && lt < count; ++i) {
            int m, n, row0, rows;
            sched.tile(lt, m, n, row0, rows);
            const int kt = sched.kstep(lt, kt0, kt1, ki);
            if (Cfg::kAMN) {
                tma_prefetch_l2_2d(&tmX, row0, kt * TILE_K);
                tma_prefetch_l2_2d(&tmX, row0 + 64, kt * TILE_K);
            } else {
                tma_prefetch_l2_2d(&tmX, kt * TILE_K, row0);
            }
            if (++ki == kt1 - kt0) {
                if (++lt < count) sched.krange(lt, kt0, kt1, slice);
                ki = 0;
            }
        }
    }
    // Everything above may overlap the tail of a preceding grid launched with
    // programmatic serialization; global memory is read or written only after
    // this (the prefetches above only warm L2).
    griddep_wait();
    griddep_launch_dependents();
    // Global exchange: launch E counts in bank E & 1.  Only the warps that
    // count or wait read E (gx_bank, below), after the pipeline has started:
    // an L2 round trip before the barrier would hold the producer back.  (E is
    // fixed for the launch: the last CTA to leave advances it, after every
    // thread's last use.)
    // One thread of the first epilogue warp reads E (and the last launch's
    // counter count) into shared memory; the epilogue warps and the
    // pre-norm's summing warp meet at a named barrier and take it from
    // there.  The CTA counts itself in after that barrier, so no warp of a
    // counted CTA reads E from L2 after the last CTA may have advanced it.
    constexpr int XWARPS = EPI_WARPS + (Cfg::kPre ? 1 : 0);  // warps meeting at named barrier 1
    auto gx_epoch = [&]() {
        if (threadIdx.x == 0) {
            epoch_sm[0] = ld_acquire_gpu(args.xcnt + 2);
            epoch_sm[1] = ld_acquire_gpu(args.xcnt + 3) * 4;
        }
        named_bar_sync(1, XWARPS * 32);
        return epoch_sm[0];
    };
    if (Cfg::kRow && !GLOBALX && threadIdx.x < 128) {
        // This CTA's columns never change: clustered CTAs keep their rank's
        // tile, unclustered post-norm has a single column tile.
        const int n0 = sched.n_fixed * TILE_N;
        for (int i = static_cast<int>(threadIdx.x); i < TILE_N; i += 128) {
            const int col = n0 + i;
            const bool in = col < args.N;
            aff[i] = (args.gamma && in) ? args.gamma[col] : static_cast<uint16_t>(0x3F80);  // 1.0
            aff[TILE_N + i] = (args.beta && in) ? args.beta[col] : static_cast<uint16_t>(0);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (CLUSTERED || PAIR) {  // barriers of every CTA initialised before any remote use
        cluster_arrive_release();
        cluster_wait_acquire();
    }
    const uint32_t tmem_base = *tmem_holder;

    if (warp == Cfg::PRODUCER_WARP) {
        // ================================================================ TMA producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued = 0;
            bool ok = true;
            const uint64_t wpol = NF_W_EVICT_LAST ? l2_policy_evict_last() : 0;
            for (int lt = 0; lt < count && ok; ++lt) {
                int m, n, row0, rows, kt0, kt1, slice;
                sched.tile(lt, m, n, row0, rows);
                sched.krange(lt, kt0, kt1, slice);
                for (int ki = 0; ki < kt1 - kt0; ++ki) {
                    const int kt = sched.kstep(lt, kt0, kt1, ki);
                    // (a slot's first fill never waits: the ring starts empty)
                    if (issued >= static_cast<uint32_t>(STAGES) &&
                        !mbar_wait<PAIR>(guard, bar_empty0 + 8u * s, ph ^ 1u, SITE_PROD_EMPTY, lt)) {
                        ok = false;
                        break;
                    }
                    if (PAIR) {
                        // Both CTAs' bytes are counted on the first CTA's full[s].
                        const uint32_t fl = bar_full0 + 8u * s;
                        const uint32_t fb = mapa_shared(fl, static_cast<uint32_t>(my_rank & ~1));
                        if (lead) mbar_arrive_expect_tx(fl, 2u * Cfg::STAGE_BYTES);
                        tma_load_2d_pair(sA + s * A_STAGE_BYTES, &tmX, fb, kt * TILE_K, row0);
#pragma unroll
                        for (int i = 0; i < NBOX / 2; ++i) {
                            const int col = n * TILE_N + sched.pair_rank * (TILE_N / 2) + i * B_BOX_N;
                            if (NF_W_EVICT_LAST)
                                tma_load_2d_pair_hint(sB + s * Cfg::B_STAGE_BYTES + i * B_BOX_BYTES, &tmW, fb, col,
                                                      kt * TILE_K, wpol);
                            else
                                tma_load_2d_pair(sB + s * Cfg::B_STAGE_BYTES + i * B_BOX_BYTES, &tmW, fb, col,
                                                 kt * TILE_K);
                        }
                        ++issued;
                        if (++s == STAGES) {
                            s = 0;
                            ph ^= 1u;
                        }
                        continue;
                    }
                    const uint32_t fb = bar_full0 + 8u * s;
                    if (Cfg::kScaleA) {
                        // The stage's 64 rstd values (fewer at the end of K) come
                        // with it: K % 8 == 0 keeps the byte count a multiple of 32.
                        const int nr = min(TILE_K, args.K - kt * TILE_K);
                        mbar_arrive_expect_tx(fb, Cfg::STAGE_BYTES + static_cast<uint32_t>(nr * 4));
                        bulk_load_g2s(sRS + static_cast<uint32_t>(s * TILE_K * 4), args.rstd_in + kt * TILE_K,
                                      static_cast<uint32_t>(nr * 4), fb);
                    } else {
                        mbar_arrive_expect_tx(fb, Cfg::STAGE_BYTES);
                    }
                    if (Cfg::kAMN) {
                        // X stored K x M: two boxes of 64 output rows x 64 K-rows
                        // (MN-major A: 128-byte rows along the output rows).
                        tma_load_2d(sA + s * A_STAGE_BYTES, &tmX, fb, row0, kt * TILE_K);
                        tma_load_2d(sA + s * A_STAGE_BYTES + B_BOX_BYTES, &tmX, fb, row0 + 64, kt * TILE_K);
                    } else {
                        tma_load_2d(sA + s * A_STAGE_BYTES, &tmX, fb, kt * TILE_K, row0);
                    }
                    if (Cfg::kBK) {
                        // W stored N x K: one box of TILE_N output columns x 64 K
                        // (K-major B: 128-byte rows along K, like A).
                        if (NF_W_EVICT_LAST)
                            tma_load_2d_hint(sB + s * Cfg::B_STAGE_BYTES, &tmW, fb, kt * TILE_K, n * TILE_N, wpol);
                        else
                            tma_load_2d(sB + s * Cfg::B_STAGE_BYTES, &tmW, fb, kt * TILE_K, n * TILE_N);
                    } else {
#pragma unroll
                        for (int i = 0; i < NBOX; ++i) {
                            if (NF_W_EVICT_LAST)
                                tma_load_2d_hint(sB + s * Cfg::B_STAGE_BYTES + i * B_BOX_BYTES, &tmW, fb,
                                                 n * TILE_N + i * B_BOX_N, kt * TILE_K, wpol);
                            else
                                tma_load_2d(sB + s * Cfg::B_STAGE_BYTES + i * B_BOX_BYTES, &tmW, fb,
                                            n * TILE_N + i * B_BOX_N, kt * TILE_K);
                        }
                    }
                    ++issued;
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // Drain: every load issued has landed before the CTA may exit.  (A
            // pair's loads are all counted on the first CTA's barriers, which
            // its producer drains; the pair meets at a cluster barrier before
            // either CTA exits.)
            for (int j = 0; j < STAGES && lead; ++j) {
                const uint32_t uj = static_cast<uint32_t>(j);
                if (issued > uj) {
                    const uint32_t fills = (issued - 1u - uj) / STAGES + 1u;
                    mbar_drain(bar_full0 + 8u * j, (fills - 1u) & 1u, args.timeout_ns);
                }
            }
        }
        __syncwarp();
    } else if (warp == Cfg::MMA_WARP) {
        // ================================================================ MMA issuer
        if (lane == 0 && PAIR && !lead) {
            // CTA pair, second CTA: relay "this CTA's epilogue drained
            // accumulator b" to the first CTA, whose MMA writes this CTA's TMEM.
            for (int lt = NACC; lt < count; ++lt) {
                const int b = lt % NACC;
                const uint32_t aph = static_cast<uint32_t>(lt / NACC) & 1u;
                if (!mbar_wait(guard, bar_acce0 + 8u * b, aph ^ 1u, SITE_MMA_ACC_EMPTY, lt)) break;
                mbar_arrive_remote(mapa_shared(bar_pacc0 + 8u * b, static_cast<uint32_t>(my_rank & ~1)));
            }
        } else if (lane == 0) {
            constexpr uint32_t IDESC = idesc_bf16_f32(PAIR ? 2 * TILE_M : TILE_M, TILE_N, !Cfg::kBK, Cfg::kAMN);
            // A transformed in shared memory is consumed after the transform
            // warps released the stage, not when its bytes landed.
            const uint32_t bar_ready0 = Cfg::kScaleA ? bar_xf0 : bar_full0;
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int lt = 0; lt < count && ok; ++lt) {
                const int b = lt % NACC;
                const uint32_t aph = static_cast<uint32_t>(lt / NACC) & 1u;
                if (!mbar_wait(guard, bar_acce0 + 8u * b, aph ^ 1u, SITE_MMA_ACC_EMPTY, lt)) break;
                if (PAIR && !mbar_wait_remote(guard, bar_pacc0 + 8u * b, aph ^ 1u, SITE_MMA_ACC_EMPTY, lt)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(b * TILE_N);
                int kt0, kt1, slice;
                sched.krange(lt, kt0, kt1, slice);
                for (int ki = 0; ki < kt1 - kt0; ++ki) {
                    // (a pair's full[s] also completes by the peer's bytes or
                    // arrival: polled without the suspend hint)
                    if (!mbar_wait<PAIR>(guard, bar_ready0 + 8u * s, ph, SITE_MMA_FULL, lt)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = sA + s * A_STAGE_BYTES;
                    const uint32_t b0 = sB + s * Cfg::B_STAGE_BYTES;
#pragma unroll
                    for (int j = 0; j < TILE_K / UMMA_K; ++j) {
                        // A: K-major, advance 16 elements = 32 bytes inside the
                        //    swizzled 128-byte row; 8-row groups 1 KB apart.
                        // B: MN-major, advance 16 K-rows = 2 KB; 8-row groups
                        //    1 KB apart, 64-column boxes 8 KB apart.
                        // (Transposed operands: MN-major A advances 2 KB per 16
                        //  K-rows with its two 64-row boxes 8 KB apart; K-major B
                        //  advances 32 bytes like A.  CTA pair: the same
                        //  descriptors address both CTAs' stages.)
                        const uint64_t adesc = Cfg::kAMN ? smem_desc_sw128(a0 + j * 2048, B_BOX_BYTES, 1024)
                                                         : smem_desc_sw128(a0 + j * 32, 16, 1024);
                        const uint64_t bdesc = Cfg::kBK ? smem_desc_sw128(b0 + j * 32, 16, 1024)
                                                        : smem_desc_sw128(b0 + j * 2048, B_BOX_BYTES, 1024);
                        if (PAIR)
                            mma_bf16_pair(d, adesc, bdesc, IDESC, (ki != 0 || j != 0) ? 1u : 0u);
                        else
                            mma_bf16(d, adesc, bdesc, IDESC, (ki != 0 || j != 0) ? 1u : 0u);
                    }
                    // stage free (in both CTAs of a pair) once these MMAs finish
                    if (PAIR)
                        mma_commit_pair(bar_empty0 + 8u * s);
                    else
                        mma_commit(bar_empty0 + 8u * s);
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                if (PAIR)  // accumulator b complete in both CTAs
                    mma_commit_pair(bar_accf0 + 8u * b);
                else
                    mma_commit(bar_accf0 + 8u * b);
            }
            // Everything issued has completed before TMEM can be released.
            if (PAIR)
                mma_commit_pair_local(bar_mma_done);
            else
                mma_commit(bar_mma_done);
            mbar_drain(bar_mma_done, 0, args.timeout_ns);
        }
        __syncwarp();
    } else if (warp < EPI_WARPS) {
        // ================================================================ epilogue
        // Global exchange: this launch's bank, and the other bank cleared --
        // the previous launch on this scratch counted there (it has completed;
        // the next launch counts there).  The epilogue warps do it while the
        // first tile's main loop runs.
        int* xbank = nullptr;
        unsigned long long xtag = 0;  // pre-norm, split sums: this launch's tag in a word's high half
        if (GLOBALX) {
            const int e = gx_epoch();
            xtag = static_cast<unsigned long long>(static_cast<uint32_t>(e) + 1u) << 32;
            const int prev_ints = epoch_sm[1];
            xbank = args.xcnt + XCH_CNT0 + (e & 1) * args.xbank;
            int* const other = args.xcnt + XCH_CNT0 + ((e + 1) & 1) * args.xbank;
            const int stride = static_cast<int>(gridDim.x) * EPI_WARPS * 32;
            for (int i = static_cast<int>(blockIdx.x) * EPI_WARPS * 32 + static_cast<int>(threadIdx.x); i < prev_ints;
                 i += stride)
                other[i] = 0;
            if (threadIdx.x == 0) {
                // Every CTA counts itself in once its warps hold E (the named
                // barrier above).  The last one resets the count, records how
                // many counters this launch uses (the next launch clears them)
                // and advances the epoch, which the next launch reads after
                // this one has completed.  Done here, in the first main loop's
                // shadow, not at exit, where its L2 round trips would delay the
                // kernel's end.
                int* const hdr = args.xcnt;
                if (atom_acq_rel_gpu_add(hdr, 1) == static_cast<int>(gridDim.x) - 1) {
                    hdr[0] = 0;
                    hdr[3] = args.m_tiles;
                    st_release_gpu(hdr + 2, e + 1);
                }
            }
        }
        // The global exchange of one tile's row partials (pa, pb), for the
        // group's four warps together, without a memory fence.  Each thread
        // stores its row's partials for column tile n as a pair of tagged
        // words (each carries this launch's tag beside its float, so a reader
        // can tell by the word itself whether it is current).  Once all four
        // warps have (xpub), the group's first warp adds one to row tile m's
        // count and waits, with relaxed loads, until all n_tiles column tiles
        // have counted; then (xrdy) every thread reads its row's n_tiles
        // pairs, again while any still carries an older tag.  The count and
        // the barriers only say when to look.  (A GPU-scope release on the
        // count and an acquire after it, one pair per warp, measured 3.7 us
        // slower at 16384 x 1024 x 2048, and one pair per warpgroup still
        // 3 us: such fences hold back the SM's operand loads.  Every thread
        // polling the tagged words alone, without the count, measured slower
        // still: the L2 traffic of the polling threads does the same.)  A
        // CTA pair's second CTA past M (m >= m_tiles) has no rows: it keeps
        // the group's barrier phases but stores, counts and reads nothing.
        // False (for the whole warp) when a wait gave up.
        auto xch_global = [&](int m, int n, int qtr, int row, int grp, uint32_t jph, float pa, float pb,
                              float2 (&pp)[MAX_CLUSTER], int lt) -> bool {
            const int nt = args.n_tiles;
            const bool real = m < args.m_tiles;  // (the same for the whole CTA)
            unsigned long long* const w = args.xpart + (static_cast<size_t>(real ? m : 0) * nt * TILE_M + row) * 2;
            if (real)
                st_relaxed_gpu_v2_u64(w + static_cast<size_t>(n) * TILE_M * 2, xtag | __float_as_uint(pa),
                                      xtag | __float_as_uint(pb));
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_xpub0 + 8u * grp);
            if (qtr == 0) {
                bool ok = __all_sync(0xffffffffu, mbar_wait(guard, bar_xpub0 + 8u * grp, jph, SITE_EPI_GXCH, lt));
                if (ok && real) {
                    int* const cnt = xbank + m * 4;
                    if (lane == 0) red_relaxed_gpu_add(cnt, 1);
                    ok = gwait_geq(guard, cnt, nt, SITE_EPI_GXCH, lt);
                }
                if (!ok) return false;  // (the other warps' xrdy wait then sees the abort flag)
                if (lane == 0) mbar_arrive(bar_xrdy0 + 8u * grp);
            }
            if (!__all_sync(0xffffffffu, mbar_wait(guard, bar_xrdy0 + 8u * grp, jph, SITE_EPI_GXCH, lt)))
                return false;
#pragma unroll
            for (int p = 0; p < MAX_CLUSTER; ++p) pp[p] = make_float2(0.0f, 0.0f);
            if (!real) return true;
            constexpr unsigned long long HI = 0xffffffff00000000ull;
            uint64_t t0 = 0;
            for (int round = 0;; ++round) {
                // All nt pairs each round, loaded before any is looked at.
                uint32_t stale = 0;
#pragma unroll
                for (int p = 0; p < MAX_CLUSTER; ++p)
                    if (p < nt) {
                        const ulonglong2 v = ld_relaxed_gpu_v2_u64(w + static_cast<size_t>(p) * TILE_M * 2);
                        stale |= static_cast<uint32_t>(((v.x & HI) != xtag) | ((v.y & HI) != xtag));
                        pp[p] = make_float2(__uint_as_float(static_cast<uint32_t>(v.x)),
                                            __uint_as_float(static_cast<uint32_t>(v.y)));
                    }
                if (__all_sync(0xffffffffu, stale == 0)) return true;
                if (round == 0) t0 = globaltimer_ns();
                __nanosleep(64);
                if (*guard.abort_flag) return false;
                if (globaltimer_ns() - t0 > guard.timeout_ns) {
                    record_failure(guard, 5u /* NF_ERR_TIMEOUT */, SITE_EPI_GXCH, lt);
                    return false;
                }
            }
        };
        // Two warpgroups alternate tiles: group g drains TMEM accumulator g, so
        // each group has two tiles' time for its chain of TMEM reads,
        // statistics, conversion and stores.  Warp (g, qtr) owns TMEM lane
        // quarter qtr (tile rows 32 qtr .. +31, one row per thread).  The row is
        // read in segments of 64 columns (two tcgen05.ld, one wait); post-norm
        // keeps the last segment in registers across the statistics exchange.
        constexpr int SEG = TILE_N < 64 ? TILE_N : 64;
        // Post-norm keeps the row's last segment in registers across the
        // statistics exchange, except the global exchange, whose partials of up
        // to 16 column tiles need those registers, and the residual add, whose
        // staging of R does: those read the segment (X W + R) again from TMEM.
        constexpr bool KEEP_SEG = Cfg::kPost && !GLOBALX && !Cfg::kRes;  // (the backward needs them for Z)
        // The global exchange's lane 0 counts and polls; another lane issues
        // the warp's bulk stores.
        constexpr int STORE_LANE = GLOBALX ? 31 : 0;
        constexpr int NC = SEG / 32;
        const int grp = warp >> 2;
        const int qtr = warp & 3;
        const int row = qtr * 32 + lane;  // tile row == TMEM lane
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(qtr * 32) << 16);
        const bool affine = Cfg::kRow && (args.gamma != nullptr || args.beta != nullptr);
        // gamma at saff, beta at saff + 2 TILE_N; the global exchange keeps one
        // such slot per group, refilled for each tile's columns.
        const uint32_t saff = smem_u32(aff) + (GLOBALX ? static_cast<uint32_t>(grp * 4 * TILE_N) : 0u);
        int aff_n = -1;  // global exchange: the column tile whose gamma / beta are in the slot
        for (int lt = grp; lt < count; lt += 2) {
            int m, n, row0, rows, kt0, kt1, slice;
            sched.tile(lt, m, n, row0, rows);
            sched.krange(lt, kt0, kt1, slice);
            const int b = lt % NACC;
            const uint32_t aph = static_cast<uint32_t>(lt / NACC) & 1u;
            const uint32_t jph = static_cast<uint32_t>(lt >> 1) & 1u;  // this group's tile count parity
            bool ok = true;
            const int nv = min(TILE_N, args.N - n * TILE_N);        // valid columns of this tile
            const int grow = row0 + row;                             // global row
            const bool own_row = row < rows && grow < args.M;
            const uint16_t* const zrow =
                Cfg::kBwd ? args.zin + static_cast<size_t>(own_row ? grow : 0) * args.N + n * TILE_N : nullptr;
            // This warp's 32-row block of the tile (wrows valid rows from wr0):
            // the residual R is read, and the residual output written, block by
            // block through the warp's staging buffer (coalesced 128-byte lines).
            const int wr0 = row0 + qtr * 32;
            const int wrows = max(0, min(32, min(rows - qtr * 32, args.M - wr0)));
            const size_t woff = static_cast<size_t>(wrows > 0 ? wr0 : 0) * args.N + n * TILE_N;
            const uint32_t wbuf = sStg + static_cast<uint32_t>(warp * STORE_BUF_BYTES);
            // Post-norm residual add: R's row in this tile is asked of L2 before
            // the accumulator wait; it is read once, in the statistics loop,
            // which writes X W + R back into TMEM.
            constexpr bool res = Cfg::kRes;
            if (res && own_row)  // nv * 2 bytes: N % 8 == 0 keeps it a multiple of 16
                bulk_prefetch_l2(args.resid + woff + static_cast<size_t>(row - qtr * 32) * args.N,
                                 static_cast<uint32_t>(nv * 2));
            if (GLOBALX && affine) {
                // -- this warp's quarter of the group's affine slot (64 columns),
                //    refilled only when the column tile changes, once the group's
                //    four warps are done with the previous tile; done before the
                //    accumulator is ready so the loads overlap the main loop.
                if (n != aff_n) {
                    ok = mbar_wait(guard, bar_affe0 + 8u * grp, jph ^ 1u, SITE_EPI_AFF, lt);
                    if (!__all_sync(0xffffffffu, ok)) break;
                    const int c = qtr * 64 + 2 * lane, col = n * TILE_N + c;  // N % 8 == 0: both or neither in
                    const bool in = col < args.N;
                    uint32_t g2 = 0x3F803F80u, b2 = 0u;
                    if (in && args.gamma)
                        g2 = static_cast<uint32_t>(args.gamma[col]) | (static_cast<uint32_t>(args.gamma[col + 1]) << 16);
                    if (in && args.beta)
                        b2 = static_cast<uint32_t>(args.beta[col]) | (static_cast<uint32_t>(args.beta[col + 1]) << 16);
                    st_shared_u32(saff + static_cast<uint32_t>(c * 2), g2);
                    st_shared_u32(saff + static_cast<uint32_t>((TILE_N + c) * 2), b2);
                    aff_n = n;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_afff0 + 8u * grp);
            }
            const int nseg = (nv + SEG - 1) / SEG;                   // segments holding them
            // Store only this unit's rows, and nothing past M.
            const int nstore = (qtr * 32 < rows && row0 + qtr * 32 < args.M) ? nv : 0;
            // Backward: the row's saved statistics, requested before the
            // accumulator wait (they do not depend on it).
            const float bmu = (Cfg::kBwdLN && own_row) ? args.mean_in[grow] : 0.0f;
            const float brs = (Cfg::kBwd && own_row) ? args.rstd_in[grow] : 0.0f;
            ok = mbar_wait<PAIR>(guard, bar_accf0 + 8u * b, aph, SITE_EPI_ACC_FULL, lt);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const uint32_t tacc = t_lane + static_cast<uint32_t>(b * TILE_N);
            float scale = 1.0f, bias = 0.0f;                         // y = acc * scale + bias
            bool released = false;
            uint32_t v[NC][32];


            if (Cfg::kPre) {
                float ss = 0.0f;
                if (GLOBALX) {
                    // The row's sum of squares, summed by one of the row tile's
                    // n_tiles tiles: poll the row's word until it carries this
                    // launch's tag.  (A CTA pair's second CTA past M has no
                    // rows: nothing to wait for.)
                    if (m < args.m_tiles) {
                        unsigned long long wv = 0;
                        ok = tagged_wait(guard, args.sstag + static_cast<size_t>(m) * TILE_M + row, xtag, wv,
                                         SITE_EPI_GXCH, lt);
                        if (!__all_sync(0xffffffffu, ok)) break;
                        ss = __uint_as_float(static_cast<uint32_t>(wv));
                    }
                } else {
                    ok = mbar_wait(guard, bar_ssf0 + 8u * b, aph, SITE_EPI_SS_FULL, lt);
                    if (!__all_sync(0xffffffffu, ok)) break;
                    ss = ss_buf[b * TILE_M + row];
                }
                // blog §2: rstd = rsqrt(square_sum / K + eps); acc *= rstd[:, None]
                scale = rsqrtf(fmaf(ss, args.inv_len, args.eps));
                if (n == 0 && args.rstd_out && own_row) args.rstd_out[grow] = scale;
            }

            float bc1 = 0.0f, bc0 = 0.0f;  // backward: dz = g * brs + z * bc1 + bc0

            if (Cfg::kBwd) {
                // -- backward partials of this CTA's nv columns: sum of g and of
                //    g * (z - mean), g = dY * gamma (xhat = (z - mean) * rstd).
                if (GLOBALX && affine) {  // gamma of this tile is in the group's slot
                    ok = mbar_wait(guard, bar_afff0 + 8u * grp, jph, SITE_EPI_AFF, lt);
                    if (!__all_sync(0xffffffffu, ok)) break;
                }
                const uint64_t mu2 = f2_splat(bmu);
                uint64_t a1[4] = {0, 0, 0, 0}, a2[4] = {0, 0, 0, 0};
                for (int sg = 0; sg < nseg; ++sg) {
                    uint4 zq[8];
                    load_z64(zrow + sg * SEG, own_row, nv - sg * SEG, zq);
                    tmem_load_seg<NC>(tacc + sg * SEG, v);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const uint32_t* src = v[q >> 2];
                        const int o = (q & 3) * 8;
                        const uint32_t zw[4] = {zq[q].x, zq[q].y, zq[q].z, zq[q].w};
                        uint32_t gw[4] = {0u, 0u, 0u, 0u};
                        if (affine && args.gamma) {
                            const uint4 gq = ld_shared_v4(saff + static_cast<uint32_t>((sg * SEG + q * 8) * 2));
                            gw[0] = gq.x, gw[1] = gq.y, gw[2] = gq.z, gw[3] = gq.w;
                        }
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            uint64_t g2 = f2_pack(src[o + 2 * e], src[o + 2 * e + 1]);
                            if (affine && args.gamma) g2 = f2_fma(g2, bf16x2_to_f2(gw[e]), 0ull);
                            const uint64_t d2 = f2_sub(bf16x2_to_f2(zw[e]), mu2);
                            a1[e] = f2_add(a1[e], g2);
                            a2[e] = f2_fma(g2, d2, a2[e]);
                        }
                    }
                }
                const float pa = f2_hsum(f2_add(f2_add(a1[0], a1[1]), f2_add(a1[2], a1[3])));
                const float pb = f2_hsum(f2_add(f2_add(a2[0], a2[1]), f2_add(a2[2], a2[3])));
                float s1 = pa, s2 = pb;  // sums over the whole row
                if (CLUSTERED) {
                    const uint32_t slot =
                        sRecv + static_cast<uint32_t>(((b * MAX_CLUSTER + my_rank) * TILE_M + row) * 8);
                    const uint32_t xbar = bar_xch0 + 8u * b;
                    for (int p = 0; p < args.cluster; ++p)
                        st_async_f32x2(mapa_shared(slot, p), pa, pb, mapa_shared(xbar, p));
                    ok = mbar_wait<true>(guard, xbar, aph, SITE_EPI_XCH, lt);
                    if (!__all_sync(0xffffffffu, ok)) break;
                    if (qtr == 0 && lane == 0 && lt + 2 < count) mbar_arrive_expect_tx(xbar, xch_bytes);
                    const float* recv = reinterpret_cast<const float*>(
                        base_ptr + Cfg::OFF_RECV + (b * MAX_CLUSTER * TILE_M + row) * 8);
                    s1 = s2 = 0.0f;
                    for (int p = 0; p < args.cluster; ++p) {
                        s1 += recv[p * TILE_M * 2];
                        s2 += recv[p * TILE_M * 2 + 1];
                    }
                } else if (GLOBALX) {
                    float2 pp[MAX_CLUSTER];
                    if (!xch_global(m, n, qtr, row, grp, jph, pa, pb, pp, lt)) break;
                    s1 = s2 = 0.0f;
#pragma unroll
                    for (int p = 0; p < MAX_CLUSTER; ++p) {
                        s1 += pp[p].x;
                        s2 += pp[p].y;
                    }
                }
                // dz = rstd (g - mean(g) - xhat mean(g xhat)), mean(g) for LN only:
                //    = g * rstd + z * bc1 + bc0.
                const float mg = Cfg::kBwdLN ? s1 * args.inv_len : 0.0f;
                const float mgx = brs * s2 * args.inv_len;
                bc1 = -brs * brs * mgx;
                bc0 = -brs * mg - bc1 * bmu;
            }

            if (Cfg::kPost) {
                // -- partial statistics of this CTA's nv columns (blog §3: each CTA
                //    reduces the partial row statistics of its tile).  LayerNorm
                //    uses sums shifted by the row's first value, sh, which keeps the
                //    one-pass variance accurate; four accumulators break the chains.
                // Column pairs go through f32x2 instructions; four pair accumulators.
                float sh = 0.0f;
                uint64_t a1[4] = {0, 0, 0, 0}, a2[4] = {0, 0, 0, 0};
                for (int sg = 0; sg < nseg; ++sg) {
                    tmem_load_seg<NC>(tacc + sg * SEG, v);
                    if (res) {
                        // R's block through the staging buffer (free once the last
                        // output store read it), added to the row; X W + R back
                        // into TMEM; H out the same way.
                        if (lane == STORE_LANE) bulk_wait_read<0>();
                        __syncwarp();
                        stage_in64(wbuf, args.resid + woff + sg * SEG, args.N, wrows, nv - sg * SEG, lane);
                        __syncwarp();
                        add_staged_row(wbuf, lane, v);
#pragma unroll
                        for (int c = 0; c < NC; ++c) tmem_st32(tacc + sg * SEG + c * 32, v[c]);
                        if (args.h_out != nullptr) {
                            __syncwarp();  // every lane has read its row of R
                            put_staged_row(wbuf, lane, v);
                            __syncwarp();
                            stage_out64(wbuf, args.h_out + woff + sg * SEG, args.N, wrows, nv - sg * SEG, lane);
                        }
                        __syncwarp();  // the buffer is read out before it is reused
                    }
                    if (Cfg::kLN && sg == 0) sh = __uint_as_float(v[0][0]);
                    const uint64_t sh2 = f2_splat(sh);
#pragma unroll
                    for (int c = 0; c < NC; ++c)
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const uint64_t x2 = f2_pack(v[c][2 * i], v[c][2 * i + 1]);
                            if (Cfg::kLN) {
                                const uint64_t d2 = f2_sub(x2, sh2);
                                a1[i & 3] = f2_add(a1[i & 3], d2);
                                a2[i & 3] = f2_fma(d2, d2, a2[i & 3]);
                            } else {
                                a2[i & 3] = f2_fma(x2, x2, a2[i & 3]);
                            }
                        }
                }
                if (res) tmem_st_wait();  // the finish loop reads X W + R back
                if (KEEP_SEG && nseg == 1) {  // the row is in registers: TMEM buffer b is free
                    tc_fence_before();
                    mbar_arrive(bar_acce0 + 8u * b);
                    released = true;
                }
                float pa, pb;  // partial: LN (mean_c, M2_c); RMS (sum of squares, 0)
                if (Cfg::kLN) {
                    // Columns past N inside the loaded segments hold exact zeros (W
                    // is zero-filled there); each added -sh to a1 and sh^2 to a2.
                    const float npad = static_cast<float>(nseg * SEG - nv);
                    const float inv_nv = 1.0f / static_cast<float>(nv);
                    const float s1 = f2_hsum(f2_add(f2_add(a1[0], a1[1]), f2_add(a1[2], a1[3]))) + npad * sh;
                    const float s2 = f2_hsum(f2_add(f2_add(a2[0], a2[1]), f2_add(a2[2], a2[3]))) - npad * sh * sh;
                    const float d1 = s1 * inv_nv;
                    pa = sh + d1;
                    pb = fmaxf(fmaf(-s1, d1, s2), 0.0f);
                } else {
                    pa = f2_hsum(f2_add(f2_add(a2[0], a2[1]), f2_add(a2[2], a2[3])));
                    pb = 0.0f;
                }

                float mean = 0.0f, sq;  // sq: M2 (LN) or sum of squares (RMS) over all N
                if (CLUSTERED) {
                    // -- exchange through distributed shared memory: push this
                    //    CTA's partial into slot [my_rank] of every CTA of the
                    //    cluster (itself included), then wait for all slots.
                    const uint32_t slot =
                        sRecv + static_cast<uint32_t>(((b * MAX_CLUSTER + my_rank) * TILE_M + row) * 8);
                    const uint32_t xbar = bar_xch0 + 8u * b;
                    for (int p = 0; p < args.cluster; ++p)
                        st_async_f32x2(mapa_shared(slot, p), pa, pb, mapa_shared(xbar, p));
                    ok = mbar_wait<true>(guard, xbar, aph, SITE_EPI_XCH, lt);
                    if (!__all_sync(0xffffffffu, ok)) break;
                    // Re-arm for local tile lt + 2.  Its data can arrive only after
                    // every CTA of the cluster got this CTA's tile lt+1 partials,
                    // which are sent after this point.
                    if (qtr == 0 && lane == 0 && lt + 2 < count) mbar_arrive_expect_tx(xbar, xch_bytes);
                    const float* recv = reinterpret_cast<const float*>(
                        base_ptr + Cfg::OFF_RECV + (b * MAX_CLUSTER * TILE_M + row) * 8);
                    if (Cfg::kLN) {
                        // Chan et al. pairwise merge of (count, mean, M2).
                        float msum = 0.0f;
                        for (int p = 0; p < args.cluster; ++p) {
                            const int np = min(TILE_N, args.N - p * TILE_N);
                            msum += static_cast<float>(np) * recv[p * TILE_M * 2];
                        }
                        mean = msum * args.inv_len;
                        sq = 0.0f;
                        for (int p = 0; p < args.cluster; ++p) {
                            const int np = min(TILE_N, args.N - p * TILE_N);
                            const float dm = recv[p * TILE_M * 2] - mean;
                            sq += recv[p * TILE_M * 2 + 1] + static_cast<float>(np) * dm * dm;
                        }
                    } else {
                        sq = 0.0f;
                        for (int p = 0; p < args.cluster; ++p) sq += recv[p * TILE_M * 2];
                    }
                } else if (GLOBALX) {
                    // -- exchange through L2: this row's partials for column
                    //    tile n out, those of all n_tiles column tiles of row
                    //    tile m in (xch_global above).
                    const int nt = args.n_tiles;
                    float2 pp[MAX_CLUSTER];
                    if (!xch_global(m, n, qtr, row, grp, jph, pa, pb, pp, lt)) break;
                    if (Cfg::kLN) {
                        // Chan et al. pairwise merge of (count, mean, M2).
                        float msum = 0.0f;
#pragma unroll
                        for (int p = 0; p < MAX_CLUSTER; ++p)
                            if (p < nt) msum += static_cast<float>(min(TILE_N, args.N - p * TILE_N)) * pp[p].x;
                        mean = msum * args.inv_len;
                        sq = 0.0f;
#pragma unroll
                        for (int p = 0; p < MAX_CLUSTER; ++p)
                            if (p < nt) {
                                const float dm = pp[p].x - mean;
                                sq += pp[p].y + static_cast<float>(min(TILE_N, args.N - p * TILE_N)) * dm * dm;
                            }
                    } else {
                        sq = 0.0f;
#pragma unroll
                        for (int p = 0; p < MAX_CLUSTER; ++p)
                            if (p < nt) sq += pp[p].x;
                    }
                } else {
                    mean = pa;
                    sq = Cfg::kLN ? pb : pa;
                }
                if (GLOBALX && affine) {  // the whole slot is written before the first conversion
                    ok = mbar_wait(guard, bar_afff0 + 8u * grp, jph, SITE_EPI_AFF, lt);
                    if (!__all_sync(0xffffffffu, ok)) break;
                }
                // LayerNorm: (acc - mean) * rsqrt(M2/N + eps); RMSNorm: acc * rsqrt(ss/N + eps)
                const float rstd = rsqrtf(fmaf(sq, args.inv_len, args.eps));
                scale = rstd;
                bias = Cfg::kLN ? -mean * rstd : 0.0f;
                if (n == 0 && own_row) {
                    if (Cfg::kLN && args.mean_out) args.mean_out[grow] = mean;
                    if (args.rstd_out) args.rstd_out[grow] = rstd;
                }
            }

            // -- normalize, convert, stage (128B swizzle) and store 64 columns at
            //    a time.  Post-norm starts with the segment it kept in registers.
            for (int k = 0; k < nseg; ++k) {
                const int sg = Cfg::kPost ? nseg - 1 - k : k;
                if (!(KEEP_SEG && k == 0)) {
                    tmem_load_seg<NC>(tacc + sg * SEG, v);
                    if (k == nseg - 1) {  // last TMEM read of this tile
                        tc_fence_before();
                        mbar_arrive(bar_acce0 + 8u * b);
                        released = true;
                    }
                }
                if (EPI == EPI_PLAIN && args.splitk > 1 && slice >= 0) {
                    // Split-K: the row's fp32 partial over this unit's slice of
                    // the contraction goes to the tile's slot in the slice's
                    // plane of the workspace; a second kernel adds the planes in
                    // order.
                    const int cw = sg * SEG;
                    if (own_row && cw < nv) {
                        const int tl = m * args.n_tiles + n - args.sk_base;  // split tile index
                        float* const dst =
                            args.ws + ((static_cast<size_t>(slice) * args.sk_tiles + tl) * TILE_M + row) * TILE_N + cw;
#pragma unroll
                        for (int q = 0; q < SEG / 4; ++q)
                            if (q * 4 < nv - cw) {
                                const uint32_t* src = &v[q >> 3][(q & 7) * 4];
                                __stcg(reinterpret_cast<float4*>(dst + q * 4),
                                       make_float4(__uint_as_float(src[0]), __uint_as_float(src[1]),
                                                   __uint_as_float(src[2]), __uint_as_float(src[3])));
                            }
                    }
                    continue;
                }
                // The segment's 64-column box goes through this warp's staging
                // buffer (128B swizzle) and one TMA store.
                constexpr int NQ = SEG / STORE_COLS;
                const int cs = sg * SEG;
                if (cs < nstore) {
                    const uint64_t scale2 = f2_splat(scale), bias2 = f2_splat(bias);
                    if (lane == STORE_LANE) bulk_wait_read<0>();  // the previous store has read the buffer
                    __syncwarp();
#pragma unroll
                    for (int q = 0; q < NQ; ++q) {
                        const int c0 = cs + q * STORE_COLS;
                        if (c0 < nstore) {
                            uint32_t pk[32];
                            if (Cfg::kBwd) {
                                uint4 zq[8];
                                load_z64(zrow + c0, own_row, nv - c0, zq);
                                if (args.xhat_out != nullptr && own_row) {
                                    // Side output: the normalized forward input
                                    // xhat = (z - mean) * rstd, rounded to bf16.
                                    uint16_t* const xp = args.xhat_out + static_cast<size_t>(grow) * args.N + n * TILE_N + c0;
#pragma unroll
                                    for (int e = 0; e < 8; ++e)
                                        if (e * 8 < nv - c0) {
                                            const uint32_t zw[4] = {zq[e].x, zq[e].y, zq[e].z, zq[e].w};
                                            uint32_t o[4];
#pragma unroll
                                            for (int k = 0; k < 4; ++k)
                                                o[k] = pack_bf16x2((bf16lo(zw[k]) - bmu) * brs, (bf16hi(zw[k]) - bmu) * brs);
                                            *reinterpret_cast<uint4*>(xp + e * 8) = make_uint4(o[0], o[1], o[2], o[3]);
                                        }
                                }
                                if (affine && args.gamma)
                                    convert64_bwd<true>(v[2 * q], v[2 * q + 1], zq, saff + c0 * 2, f2_splat(brs),
                                                        f2_splat(bc1), f2_splat(bc0), pk);
                                else
                                    convert64_bwd<false>(v[2 * q], v[2 * q + 1], zq, 0, f2_splat(brs),
                                                         f2_splat(bc1), f2_splat(bc0), pk);
                            } else if (affine) {
                                convert64<AFF_SMEM>(v[2 * q], v[2 * q + 1], scale2, bias2, saff + c0 * 2,
                                                    saff + (TILE_N + c0) * 2, pk);
                            } else {
                                convert64<AFF_NONE>(v[2 * q], v[2 * q + 1], scale2, bias2, 0, 0, pk);
                            }
                            const uint32_t rowp = sStg + static_cast<uint32_t>((warp + q) * STORE_BUF_BYTES) +
                                                  static_cast<uint32_t>(lane * 128);
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                st_shared_v4(rowp + (static_cast<uint32_t>(e ^ (lane & 7)) << 4), pk[4 * e],
                                             pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == STORE_LANE) {
#pragma unroll
                        for (int q = 0; q < NQ; ++q)
                            if (cs + q * STORE_COLS < nstore)
                                tma_store_2d(&tmY, sStg + static_cast<uint32_t>((warp + q) * STORE_BUF_BYTES),
                                             n * TILE_N + cs + q * STORE_COLS, row0 + qtr * 32);
                        bulk_commit();
                    }
                }
            }
            if (!released) {
                tc_fence_before();
                mbar_arrive(bar_acce0 + 8u * b);  // TMEM buffer b may be overwritten
            }
            if (GLOBALX && affine) {  // this warp is done with the group's affine slot
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_affe0 + 8u * grp);
            }
        }
        // Shared memory must outlive the stores' reads of it; their writes
        // complete with the grid.
        if (lane == STORE_LANE) bulk_wait_read<0>();
        __syncwarp();
    } else if (Cfg::kScaleA && warp >= Cfg::SUMSQ_WARP0) {
        // ================================================================ A row scaling
        // The stored matrix's rmsnorm rebuilt on the fly: contraction row m of
        // the transposed A (a 128-byte row of 64 output rows in one of the
        // stage's two boxes; the swizzle only permutes its 16-byte chunks) is
        // multiplied by rstd[m] and rounded back to bf16 before the MMA reads it.
        const int t = static_cast<int>(threadIdx.x) - Cfg::SUMSQ_WARP0 * 32;  // 0..127
        const int box = t >> 6, r = t & 63;
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int lt = 0; lt < count && ok; ++lt) {
            int kt0, kt1, slice;
            sched.krange(lt, kt0, kt1, slice);
            for (int ki = 0; ki < kt1 - kt0; ++ki) {
                const int kt = sched.kstep(lt, kt0, kt1, ki);
                if (!mbar_wait(guard, bar_full0 + 8u * s, ph, SITE_SS_FULL, lt)) {
                    ok = false;
                    break;
                }
                const int mrow = kt * TILE_K + r;
                const float sc = mrow < args.K ? ld_shared_f32(sRS + static_cast<uint32_t>((s * TILE_K + r) * 4)) : 0.0f;
                const uint32_t rbase = sA + s * A_STAGE_BYTES + static_cast<uint32_t>(box * B_BOX_BYTES + r * 128);
                // Rows are 128 bytes apart: each thread starts at a different
                // 16-byte chunk so a quarter-warp covers 8 bank groups.
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const uint32_t a = rbase + (static_cast<uint32_t>((q + r) & 7) << 4);
                    const uint4 w = ld_shared_v4(a);
                    const uint32_t in[4] = {w.x, w.y, w.z, w.w};
                    uint32_t o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[e] = pack_bf16x2(bf16lo(in[e]) * sc, bf16hi(in[e]) * sc);
                    st_shared_v4(a, o[0], o[1], o[2], o[3]);
                }
                fence_proxy_async_smem();  // the tensor cores read these writes
                mbar_arrive(bar_xf0 + 8u * s);
                if (++s == STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
    } else if (Cfg::kPre && GLOBALX && warp >= Cfg::SUMSQ_WARP0) {
        // ================================================================ row sums of squares, split
        // The n_tiles tiles of a row tile share the work on its rows (the
        // blog's CTAs each sum every row, a redundancy that costs shared-memory
        // bandwidth the tensor cores need): tile (m, n) sums rows
        // n R .. n R + R - 1, R = ceil(128 / n_tiles), over the whole
        // contraction, from the same stages the MMA reads -- one warp reading
        // 1/n_tiles of each A stage -- and stores each sum to L2 as one 64-bit
        // word carrying this launch's tag (plain stores: the warp, whose
        // arrivals free the ring's stages, never waits on L2).  The epilogue of
        // every tile of row tile m polls its row's word until it carries the
        // tag: one L2 round trip, with no counter, fence or second read (a
        // counter and a release fence took ~2.8 us from the accumulator's
        // completion to the sums in hand).  Deadlock freedom is that of the
        // post-norm exchange: a tile's publication needs only its own main
        // loop, which needs the epilogue of the CTA's tile two before it, which
        // lies in an earlier row tile (tiles in order, 2 G >= n_tiles).
        const int nt = args.n_tiles;  // >= 2 (checked at entry): R <= 64
        const int R = (TILE_M + nt - 1) / nt;
        if (warp == Cfg::SUMSQ_WARP0) {
            const unsigned long long tag = static_cast<unsigned long long>(static_cast<uint32_t>(gx_epoch()) + 1u) << 32;
            int s = 0;
            uint32_t ph = 0;
            for (int lt = 0; lt < count; ++lt) {
                int m, n, row0, rows;
                sched.tile(lt, m, n, row0, rows);
                const int r0 = n * R;
                const int nchunk = max(0, min(R, TILE_M - r0)) * 8;  // 16-byte chunks of those rows per stage
                const int nload = (nchunk + 31) >> 5;                   // loads a lane needs per stage (<= 16)
                // Lane l reads chunk l & 7 of rows (l >> 3) + 4 i, i < NL: a warp
                // load covers four whole 128-byte rows (no bank conflicts).  A
                // row past the tile's share reads chunk 0 of its first row
                // instead and is never published.
                float acc[SPLIT_SS_ITERS];
#pragma unroll
                for (int i = 0; i < SPLIT_SS_ITERS; ++i) acc[i] = 0.0f;
                // NL loads a lane and stage, fixed at compile time: all are
                // issued, unconditionally, before any is used, so a stage costs
                // one shared-memory latency, which the tensor cores' operand
                // reads stretch to a large part of a stage's MMA time.
                // (Measured: loads issued under per-load conditions were each
                // waited for in turn, and this warp fell a ring behind the MMA
                // and set its pace -- 8192 x 4096 x 4096 in CTA pairs 162 us
                // against 141 us.)
                auto tile_sums = [&](auto nl_tag) -> bool {
                    constexpr int NL = decltype(nl_tag)::value;
                    uint32_t off[NL > 0 ? NL : 1];
#pragma unroll
                    for (int i = 0; i < NL; ++i) {
                        const int c = lane + 32 * i;
                        const int cc = c < nchunk ? c : 0;
                        off[i] = static_cast<uint32_t>(r0 * 128 + (cc >> 3) * 128 + (cc & 7) * 16);
                    }
                    for (int kt = 0; kt < k_tiles; ++kt) {
                        const bool got = (!PAIR || lead)
                                             ? mbar_wait<2>(guard, bar_full0 + 8u * s, ph, SITE_SS_FULL, lt)
                                             : mbar_wait<2>(guard, bar_ardy0 + 8u * s, ph, SITE_SS_FULL, lt);
                        if (!__all_sync(0xffffffffu, got)) return false;
                        if (PAIR && lead && lane == 0)
                            mbar_arrive_remote_relaxed(
                                mapa_shared(bar_ardy0 + 8u * s, static_cast<uint32_t>(my_rank | 1)));
                        const uint32_t sbase = sA + s * A_STAGE_BYTES;
                        uint4 w[NL > 0 ? NL : 1];
#pragma unroll
                        for (int i = 0; i < NL; ++i) w[i] = ld_shared_v4(sbase + off[i]);
#pragma unroll
                        for (int i = 0; i < NL; ++i) {
                            float x, a = acc[i];
                            x = bf16lo(w[i].x); a = fmaf(x, x, a);
                            x = bf16hi(w[i].x); a = fmaf(x, x, a);
                            x = bf16lo(w[i].y); a = fmaf(x, x, a);
                            x = bf16hi(w[i].y); a = fmaf(x, x, a);
                            x = bf16lo(w[i].z); a = fmaf(x, x, a);
                            x = bf16hi(w[i].z); a = fmaf(x, x, a);
                            x = bf16lo(w[i].w); a = fmaf(x, x, a);
                            x = bf16hi(w[i].w); a = fmaf(x, x, a);
                            acc[i] = a;
                        }
                        __syncwarp();  // the warp's reads of the stage precede lane 0's arrival
                        if (lane == 0) mbar_arrive(bar_empty0 + 8u * s);
                        if (++s == STAGES) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                    return true;
                };
                // (the wait polls without the suspend hint: measured faster here)
                bool ok;
                if (nload == 0) ok = tile_sums(std::integral_constant<int, 0>{});
                else if (nload <= 1) ok = tile_sums(std::integral_constant<int, 1>{});
                else if (nload <= 2) ok = tile_sums(std::integral_constant<int, 2>{});
                else if (nload <= 4) ok = tile_sums(std::integral_constant<int, 4>{});
                else if (nload <= 8) ok = tile_sums(std::integral_constant<int, 8>{});
                else ok = tile_sums(std::integral_constant<int, 16>{});
                if (!ok) break;
                // Whole rows: add the eight chunks' sums (lanes 8j .. 8j + 7).
#pragma unroll
                for (int i = 0; i < SPLIT_SS_ITERS; ++i) {
                    acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], 1);
                    acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], 2);
                    acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], 4);
                }
                // One tagged word per row (a CTA pair's second CTA past M has
                // no rows: nothing to publish).
                if (m < args.m_tiles) {
                    unsigned long long* const dst = args.sstag + static_cast<size_t>(m) * TILE_M + r0;
#pragma unroll
                    for (int i = 0; i < SPLIT_SS_ITERS; ++i) {
                        const int r = (lane >> 3) + 4 * i;
                        if ((lane & 7) == 0 && 8 * r < nchunk)
                            st_relaxed_gpu_u64(dst + r, tag | __float_as_uint(acc[i]));
                    }
                }
            }
        }
    } else if (Cfg::kPre && warp >= Cfg::SUMSQ_WARP0) {
        // ================================================================ row sums of squares
        // (CTA pair: both CTAs' bytes are counted on the first CTA's full[s];
        // one of its sum-of-squares threads then tells the peer's, which wait
        // on their ardy[s], with a relaxed remote arrive -- it reports an event
        // the sender has observed.)
        const int row = static_cast<int>(threadIdx.x) - Cfg::SUMSQ_WARP0 * 32;  // 0..127
        int s = 0;
        uint32_t ph = 0;
        for (int lt = 0; lt < count; ++lt) {
            const int b = lt % NACC;
            const uint32_t aph = static_cast<uint32_t>(lt / NACC) & 1u;
            float acc0 = 0.0f, acc1 = 0.0f;
            bool ok = true;
            for (int kt = 0; kt < k_tiles; ++kt) {
                const bool got = (!PAIR || lead) ? mbar_wait(guard, bar_full0 + 8u * s, ph, SITE_SS_FULL, lt)
                                                 : mbar_wait<2>(guard, bar_ardy0 + 8u * s, ph, SITE_SS_FULL, lt);
                if (!got) {
                    ok = false;
                    break;
                }
                if (PAIR && lead && row == 0)
                    mbar_arrive_remote_relaxed(mapa_shared(bar_ardy0 + 8u * s, static_cast<uint32_t>(my_rank | 1)));
                // The row's 128 bytes are contiguous whatever the swizzle (it
                // only permutes 16-byte chunks within the row); start each
                // thread at a different chunk so the 8 threads of a quarter
                // warp hit 8 different bank groups.
                const uint32_t rbase = sA + s * A_STAGE_BYTES + static_cast<uint32_t>(row * 128);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const uint4 w = ld_shared_v4(rbase + (static_cast<uint32_t>((q + row) & 7) << 4));
                    float x;
                    x = bf16lo(w.x); acc0 = fmaf(x, x, acc0);
                    x = bf16hi(w.x); acc1 = fmaf(x, x, acc1);
                    x = bf16lo(w.y); acc0 = fmaf(x, x, acc0);
                    x = bf16hi(w.y); acc1 = fmaf(x, x, acc1);
                    x = bf16lo(w.z); acc0 = fmaf(x, x, acc0);
                    x = bf16hi(w.z); acc1 = fmaf(x, x, acc1);
                    x = bf16lo(w.w); acc0 = fmaf(x, x, acc0);
                    x = bf16hi(w.w); acc1 = fmaf(x, x, acc1);
                }
                mbar_arrive(bar_empty0 + 8u * s);
                if (++s == STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) break;
            // ss_buf[b] is free once the epilogue released accumulator b of tile lt-2.
            if (!mbar_wait(guard, bar_acce0 + 8u * b, aph ^ 1u, SITE_SS_ACC_EMPTY, lt)) break;
            ss_buf[b * TILE_M + row] = acc0 + acc1;
            mbar_arrive(bar_ssf0 + 8u * b);
        }
    }

    // ---- teardown
    tc_fence_before();
    __syncthreads();
    if (CLUSTERED || PAIR) {
        // No CTA leaves while a peer may still write into its shared memory
        // (or, in a pair, its TMEM).
        cluster_arrive_release();
        cluster_wait_acquire();
    }
    if (warp == Cfg::PRODUCER_WARP) {
        tc_fence_after();
        if (PAIR)
            tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
        else
            tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

template <int EPI, int TILE_N, int XCH, int OPS = 0>
GemmVariant make_variant() {
    using Cfg = GemmCfg<EPI, TILE_N, XCH, OPS>;
    return GemmVariant{EPI,
                       TILE_N,
                       XCH == XCH_CLUSTER,
                       XCH,
                       Cfg::kPair,
                       OPS,
                       reinterpret_cast<const void*>(&nf_gemm_kernel<EPI, TILE_N, XCH, OPS>),
                       Cfg::THREADS,
                       Cfg::SMEM_BYTES,
                       Cfg::STAGES,
                       Cfg::TMEM_COLS,
                       TILE_K};
}

}  // namespace nf
