// nf_gemm_wide.cuh -- post-norm GEMM with 512 output columns per CTA:
// Y = LayerNorm(X W) * g + b  or  RMSNorm(X W) * g, the row spread over a
// cluster of at most 8 CTAs (N <= 512 x 8 = 4096).  This is the tiling of the
// blog "Towards Free Normalization: Fusing Normalization into GEMM and
// Attention Kernels", §3: about 512 columns per CTA times the portable cluster
// size of 8.  On sm_103a a 512-column fp32 accumulator fills the whole tensor
// memory (two N = 256 MMAs per K step), so it is single-buffered; the shorter
// clusters fit more often on the GPU than 16-CTA clusters of 256 columns.
//
// CTA roles (one CTA per SM, persistent over the m tiles of its cluster):
//   warps 0-7  epilogue: warp w reads TMEM lane quarter w % 4 (tile rows
//              32(w%4)..+31, one per thread) and column half w / 4 (256
//              columns); the halves merge their row statistics through shared
//              memory, the CTAs of the cluster through distributed shared
//              memory (st.async); then each warp normalizes its columns and
//              stores them once through a 128B-swizzled staging box and TMA.
//   warp 8     TMA producer: X K-tiles of 128 x 32 (64-byte swizzle) and W
//              K-tiles of 32 x 512 (eight 32 x 64 boxes, 128-byte swizzle).
//   warp 9     MMA issuer: per 32-wide K-tile, 2 K steps x 2 column halves of
//              tcgen05.mma 128 x 256 x 16 into TMEM columns 0-255 / 256-511.
#pragma once

#include "nf_gemm_kernel.cuh"

namespace nf {

// Chan et al.'s merge of two (count, mean, M2) summaries into the first.
__device__ __forceinline__ void chan_merge(float na, float& mean_a, float& m2_a, float nb, float mean_b,
                                           float m2_b) {
    if (nb <= 0.0f) return;
    const float n = na + nb;
    const float d = mean_b - mean_a;
    mean_a = mean_a + d * (nb / n);
    m2_a = m2_a + m2_b + d * d * (na * nb / n);
}

template <int EPI, bool CLUSTERED>
struct WideCfg {
    static constexpr bool kLN = EPI == EPI_POST_LN;
    static_assert(EPI == EPI_POST_LN || EPI == EPI_POST_RMS, "post-norm only");
    static constexpr int TILE_N = 512;
    static constexpr int TK = 32;                              // K per stage
    static constexpr int HALF_N = 256;                         // N per MMA
    static constexpr int MAXC = 8;                             // cluster size limit
    static constexpr int A_STAGE = TILE_M * TK * 2;            // 8 KB
    static constexpr int B_BOX = TK * B_BOX_N * 2;             // 4 KB
    static constexpr int NBOX = TILE_N / B_BOX_N;              // 8
    static constexpr int B_STAGE = NBOX * B_BOX;               // 32 KB
    static constexpr int STAGE_BYTES = A_STAGE + B_STAGE;      // 40 KB
    static constexpr int RECV_BYTES = CLUSTERED ? 2 * MAXC * TILE_M * 8 : 0;
    static constexpr int AFFINE_BYTES = 2 * TILE_N * 2;
    static constexpr int PBUF_BYTES = 2 * 2 * TILE_M * 8;      // [parity][half][row] float2
    static constexpr int BAR_BYTES = 512;
    static constexpr int FIXED_BYTES =
        1024 + STAGING_BYTES + RECV_BYTES + AFFINE_BYTES + PBUF_BYTES + BAR_BYTES;
    static constexpr int STAGES_FIT = (SMEM_OPTIN_LIMIT - FIXED_BYTES) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > MAX_STAGES ? MAX_STAGES : STAGES_FIT;
    static_assert(STAGES >= 3, "ring");
    static constexpr int SMEM_BYTES = FIXED_BYTES + STAGES * STAGE_BYTES;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_STAGE;
    static constexpr int OFF_STG = OFF_B + STAGES * B_STAGE;
    static constexpr int OFF_RECV = OFF_STG + STAGING_BYTES;
    static constexpr int OFF_AFF = OFF_RECV + RECV_BYTES;
    static constexpr int OFF_PBUF = OFF_AFF + AFFINE_BYTES;
    static constexpr int OFF_BAR = OFF_PBUF + PBUF_BYTES;
    static_assert(OFF_B % 1024 == 0 && OFF_STG % 1024 == 0 && A_STAGE % 1024 == 0, "alignment");
    static constexpr int PRODUCER_WARP = 8;
    static constexpr int MMA_WARP = 9;
    static constexpr int THREADS = 320;
    static constexpr int TMEM_COLS = 512;
};

// Barrier slots of the wide kernel.
struct WideBars {
    static constexpr int FULL = 0;        // [MAX_STAGES]
    static constexpr int EMPTY = 8;       // [MAX_STAGES]
    static constexpr int ACC_FULL = 16;
    static constexpr int ACC_EMPTY = 17;  // 256 arrivals: every epilogue thread
    static constexpr int XCH = 18;        // [2] by tile parity
    static constexpr int PAIR = 20;       // [4 quarters][2 parities], 64 arrivals
    static constexpr int MMA_DONE = 28;
    static constexpr int COUNT = 29;
};

template <int EPI, bool CLUSTERED>
__global__ void __launch_bounds__(WideCfg<EPI, CLUSTERED>::THREADS, 1)
    nf_gemm_wide_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                        const __grid_constant__ CUtensorMap tmY, const GemmArgs args) {
    using Cfg = WideCfg<EPI, CLUSTERED>;
    constexpr int STAGES = Cfg::STAGES;
    constexpr int SEG = 64;
    constexpr int NC = SEG / 32;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const base_ptr = smem_raw + (base - raw);
    const uint32_t sA = base + Cfg::OFF_A;
    const uint32_t sB = base + Cfg::OFF_B;
    const uint32_t sStg = base + Cfg::OFF_STG;
    const uint32_t sRecv = base + Cfg::OFF_RECV;
    const uint32_t sBar = base + Cfg::OFF_BAR;
    auto bar = [&](int slot) { return sBar + 8u * static_cast<uint32_t>(slot); };
    uint32_t* const tmem_holder = reinterpret_cast<uint32_t*>(base_ptr + Cfg::OFF_BAR + 8 * WideBars::COUNT);
    volatile int* const abort_flag =
        reinterpret_cast<volatile int*>(base_ptr + Cfg::OFF_BAR + 8 * WideBars::COUNT + 4);
    float2* const pbuf = reinterpret_cast<float2*>(base_ptr + Cfg::OFF_PBUF);
    uint16_t* const aff = reinterpret_cast<uint16_t*>(base_ptr + Cfg::OFF_AFF);
    static_assert(8 * WideBars::COUNT + 8 <= Cfg::BAR_BYTES, "barrier area");

    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int lane = static_cast<int>(threadIdx.x & 31);
    const WaitGuard guard{args.status, abort_flag, args.timeout_ns};

    // ---- schedule: a cluster walks m tiles; this CTA owns column block n
    int my_rank = 0, first, step, count;
    if (CLUSTERED) {
        my_rank = static_cast<int>(cluster_ctarank());
        first = static_cast<int>(cluster_id_x());
        step = static_cast<int>(num_clusters_x());
    } else {
        first = static_cast<int>(blockIdx.x);
        step = static_cast<int>(gridDim.x);
    }
    count = first < args.m_tiles ? (args.m_tiles - first + step - 1) / step : 0;
    const int n = my_rank;
    const int k_tiles = args.k_tiles;
    const int nv = min(Cfg::TILE_N, args.N - n * Cfg::TILE_N);  // valid columns of this CTA
    const uint32_t xch_bytes = static_cast<uint32_t>(args.cluster) * TILE_M * 8u;

    // ---- set-up
    if (threadIdx.x == 0) {
        // The tensor maps are kernel parameters, independent of any earlier
        // grid: fetch them while a preceding kernel may still be running.
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmW);
        prefetch_tmap(&tmY);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar(WideBars::FULL + s), 1);
            mbar_init(bar(WideBars::EMPTY + s), 1);
        }
        mbar_init(bar(WideBars::ACC_FULL), 1);
        mbar_init(bar(WideBars::ACC_EMPTY), 256);
        mbar_init(bar(WideBars::XCH), 1);
        mbar_init(bar(WideBars::XCH + 1), 1);
        for (int i = 0; i < 8; ++i) mbar_init(bar(WideBars::PAIR + i), 64);
        mbar_init(bar(WideBars::MMA_DONE), 1);
        *abort_flag = 0;
        fence_mbar_init();
        if (CLUSTERED)
            for (int p = 0; p < 2 && p < count; ++p) mbar_arrive_expect_tx(bar(WideBars::XCH + p), xch_bytes);
    }
    if (warp == Cfg::PRODUCER_WARP) {
        tmem_alloc(smem_u32(tmem_holder), Cfg::TMEM_COLS);
        tmem_relinquish();
        // Warm L2 with this CTA's first ring-full of X K-tiles while a preceding
        // grid may still be running (a prefetch only fills L2, where that
        // grid's writes land, so the loads after the wait never see stale data).
        if (lane == 0) {
            int lt = 0, kt = 0;
            for (int i = 0; i < STAGES && lt < count; ++i) {
                tma_prefetch_l2_2d(&tmX, kt * Cfg::TK, (first + lt * step) * TILE_M);
                if (++kt == k_tiles) {
                    kt = 0;
                    ++lt;
                }
            }
        }
    }
    griddep_wait();
    griddep_launch_dependents();
    for (int i = static_cast<int>(threadIdx.x); i < Cfg::TILE_N; i += Cfg::THREADS) {
        const int col = n * Cfg::TILE_N + i;
        const bool in = col < args.N;
        aff[i] = (args.gamma && in) ? args.gamma[col] : static_cast<uint16_t>(0x3F80);  // 1.0
        aff[Cfg::TILE_N + i] = (args.beta && in) ? args.beta[col] : static_cast<uint16_t>(0);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (CLUSTERED) {
        cluster_arrive_release();
        cluster_wait_acquire();
    }
    const uint32_t tmem_base = *tmem_holder;

    if (warp == Cfg::PRODUCER_WARP) {
        // ================================================================ TMA producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0, issued = 0;
            bool ok = true;
            for (int lt = 0; lt < count && ok; ++lt) {
                const int m = first + lt * step;
                for (int kt = 0; kt < k_tiles; ++kt) {
                    if (!mbar_wait(guard, bar(WideBars::EMPTY + s), ph ^ 1u, SITE_PROD_EMPTY, lt)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = bar(WideBars::FULL + s);
                    mbar_arrive_expect_tx(fb, Cfg::STAGE_BYTES);
                    tma_load_2d(sA + s * Cfg::A_STAGE, &tmX, fb, kt * Cfg::TK, m * TILE_M);
#pragma unroll
                    for (int i = 0; i < Cfg::NBOX; ++i)
                        tma_load_2d(sB + s * Cfg::B_STAGE + i * Cfg::B_BOX, &tmW, fb,
                                    n * Cfg::TILE_N + i * B_BOX_N, kt * Cfg::TK);
                    ++issued;
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            for (int j = 0; j < STAGES; ++j) {
                const uint32_t uj = static_cast<uint32_t>(j);
                if (issued > uj) {
                    const uint32_t fills = (issued - 1u - uj) / STAGES + 1u;
                    mbar_drain(bar(WideBars::FULL + j), (fills - 1u) & 1u, args.timeout_ns);
                }
            }
        }
        __syncwarp();
    } else if (warp == Cfg::MMA_WARP) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC = idesc_bf16_f32(TILE_M, Cfg::HALF_N, true);
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int lt = 0; lt < count && ok; ++lt) {
                // single accumulator: wait until the epilogue drained the last tile
                if (!mbar_wait(guard, bar(WideBars::ACC_EMPTY), (static_cast<uint32_t>(lt) & 1u) ^ 1u,
                               SITE_MMA_ACC_EMPTY, lt))
                    break;
                tc_fence_after();
                for (int kt = 0; kt < k_tiles; ++kt) {
                    if (!mbar_wait(guard, bar(WideBars::FULL + s), ph, SITE_MMA_FULL, lt)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = sA + s * Cfg::A_STAGE;
                    const uint32_t b0 = sB + s * Cfg::B_STAGE;
#pragma unroll
                    for (int j = 0; j < Cfg::TK / UMMA_K; ++j) {
                        // A: K-major, 64-byte rows; advance 16 elements = 32 bytes;
                        //    8-row groups 512 bytes apart.
                        const uint64_t adesc = smem_desc_sw64(a0 + j * 32, 16, 512);
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            // B: MN-major, 64-column boxes of 32 K-rows (4 KB apart);
                            //    advance 16 K-rows = 2 KB; 8-row groups 1 KB apart.
                            const uint64_t bdesc =
                                smem_desc_sw128(b0 + hh * 4 * Cfg::B_BOX + j * 2048, Cfg::B_BOX, 1024);
                            mma_bf16(tmem_base + static_cast<uint32_t>(hh * Cfg::HALF_N), adesc, bdesc, IDESC,
                                     (kt | j) != 0 ? 1u : 0u);
                        }
                    }
                    mma_commit(bar(WideBars::EMPTY + s));
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(bar(WideBars::ACC_FULL));
            }
            mma_commit(bar(WideBars::MMA_DONE));
            mbar_drain(bar(WideBars::MMA_DONE), 0, args.timeout_ns);
        }
        __syncwarp();
    } else if (warp < 8) {
        // ================================================================ epilogue
        const int half = warp >> 2;   // column half: [256 half, 256 half + 256)
        const int qtr = warp & 3;     // TMEM lane quarter
        const int row = qtr * 32 + lane;
        const int col0 = half * Cfg::HALF_N;
        const uint32_t tacc = tmem_base + (static_cast<uint32_t>(qtr * 32) << 16) + static_cast<uint32_t>(col0);
        const bool affine = args.gamma != nullptr || args.beta != nullptr;
        const uint32_t saff = smem_u32(aff);
        const int nvw = max(0, min(Cfg::HALF_N, nv - col0));  // this warp's valid columns
        const int nseg = (nvw + SEG - 1) / SEG;
        uint32_t v[NC][32];
        for (int lt = 0; lt < count; ++lt) {
            const int m = first + lt * step;
            const uint32_t par = static_cast<uint32_t>(lt) & 1u;       // single buffer: phase = parity
            const int pb2 = lt & 1;                                    // exchange / pair buffer
            const uint32_t xph = static_cast<uint32_t>(lt >> 1) & 1u;  // their phase
            bool ok = mbar_wait(guard, bar(WideBars::ACC_FULL), par, SITE_EPI_ACC_FULL, lt);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const int grow = m * TILE_M + row;
            const int nstore = (m * TILE_M + qtr * 32 < args.M) ? nvw : 0;

            // -- statistics of this warp's columns (shifted sums on f32x2 pairs)
            float sh = 0.0f;
            uint64_t a1[4] = {0, 0, 0, 0}, a2[4] = {0, 0, 0, 0};
            for (int sg = 0; sg < nseg; ++sg) {
                tmem_load_seg<NC>(tacc + sg * SEG, v);
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
            float pa = 0.0f, pbv = 0.0f;  // LN (mean, M2) / RMS (sum of squares, 0) of the warp
            if (Cfg::kLN) {
                if (nvw > 0) {
                    // columns past N inside a loaded segment are exact zeros
                    const float npad = static_cast<float>(nseg * SEG - nvw);
                    const float inv = 1.0f / static_cast<float>(nvw);
                    const float s1 = f2_hsum(f2_add(f2_add(a1[0], a1[1]), f2_add(a1[2], a1[3]))) + npad * sh;
                    const float s2 = f2_hsum(f2_add(f2_add(a2[0], a2[1]), f2_add(a2[2], a2[3]))) - npad * sh * sh;
                    const float d1 = s1 * inv;
                    pa = sh + d1;
                    pbv = fmaxf(fmaf(-s1, d1, s2), 0.0f);
                }
            } else {
                pa = f2_hsum(f2_add(f2_add(a2[0], a2[1]), f2_add(a2[2], a2[3])));
            }
            // -- merge the two column halves of the row (bounded wait on an mbarrier)
            {
                float2* slot = pbuf + pb2 * 2 * TILE_M;
                slot[half * TILE_M + row] = make_float2(pa, pbv);
                const uint32_t pbar = bar(WideBars::PAIR + qtr * 2 + pb2);
                mbar_arrive(pbar);
                ok = mbar_wait(guard, pbar, xph, SITE_EPI_PAIR, lt);
                if (!__all_sync(0xffffffffu, ok)) break;
                const float2 s0 = slot[row];
                const float2 s1 = slot[TILE_M + row];
                if (Cfg::kLN) {
                    float mm = s0.x, m2 = s0.y;
                    chan_merge(static_cast<float>(min(Cfg::HALF_N, nv)), mm, m2,
                               static_cast<float>(max(0, nv - Cfg::HALF_N)), s1.x, s1.y);
                    pa = mm;
                    pbv = m2;
                } else {
                    pa = s0.x + s1.x;
                }
            }
            float mean = 0.0f, sq;
            if (CLUSTERED) {
                // -- exchange through distributed shared memory (blog §3)
                const uint32_t xbar = bar(WideBars::XCH + pb2);
                if (half == 0) {
                    const uint32_t slot =
                        sRecv + static_cast<uint32_t>(((pb2 * Cfg::MAXC + my_rank) * TILE_M + row) * 8);
                    for (int p = 0; p < args.cluster; ++p)
                        st_async_f32x2(mapa_shared(slot, p), pa, pbv, mapa_shared(xbar, p));
                }
                ok = mbar_wait<true>(guard, xbar, xph, SITE_EPI_XCH, lt);
                if (!__all_sync(0xffffffffu, ok)) break;
                // Re-arm for local tile lt + 2; its data can only arrive after every
                // CTA got this CTA's tile lt+1 partials, sent after this point.
                if (half == 0 && qtr == 0 && lane == 0 && lt + 2 < count) mbar_arrive_expect_tx(xbar, xch_bytes);
                const float* recv = reinterpret_cast<const float*>(
                    base_ptr + Cfg::OFF_RECV + (pb2 * Cfg::MAXC * TILE_M + row) * 8);
                if (Cfg::kLN) {
                    float nacc = static_cast<float>(min(Cfg::TILE_N, args.N));
                    mean = recv[0];
                    sq = recv[1];
                    for (int p = 1; p < args.cluster; ++p) {
                        const float np = static_cast<float>(min(Cfg::TILE_N, args.N - p * Cfg::TILE_N));
                        chan_merge(nacc, mean, sq, np, recv[p * TILE_M * 2], recv[p * TILE_M * 2 + 1]);
                        nacc += np;
                    }
                } else {
                    sq = 0.0f;
                    for (int p = 0; p < args.cluster; ++p) sq += recv[p * TILE_M * 2];
                }
            } else {
                mean = pa;
                sq = Cfg::kLN ? pbv : pa;
            }
            const float rstd = rsqrtf(fmaf(sq, args.inv_len, args.eps));
            const float bias = Cfg::kLN ? -mean * rstd : 0.0f;
            if (n == 0 && half == 0 && grow < args.M) {
                if (Cfg::kLN && args.mean_out) args.mean_out[grow] = mean;
                if (args.rstd_out) args.rstd_out[grow] = rstd;
            }

            // -- normalize and store, last segment first (still in registers)
            const uint64_t scale2 = f2_splat(rstd), bias2 = f2_splat(bias);
            for (int k = 0; k < nseg; ++k) {
                const int sg = nseg - 1 - k;
                if (k > 0) tmem_load_seg<NC>(tacc + sg * SEG, v);
                if (k == nseg - 1) {  // last TMEM read of this tile by this warp
                    tc_fence_before();
                    mbar_arrive(bar(WideBars::ACC_EMPTY));
                }
                const int c0 = sg * SEG;  // within this warp's half
                if (c0 < nstore) {
                    uint32_t pk[32];
                    if (affine)
                        convert64<AFF_SMEM>(v[0], v[1], scale2, bias2, saff + (col0 + c0) * 2,
                                            saff + (Cfg::TILE_N + col0 + c0) * 2, pk);
                    else
                        convert64<AFF_NONE>(v[0], v[1], scale2, bias2, 0, 0, pk);
                    const uint32_t sb = sStg + static_cast<uint32_t>(warp * STORE_BUF_BYTES);
                    if (lane == 0) bulk_wait_read<0>();  // the previous store has read the box
                    __syncwarp();
                    const uint32_t rowp = sb + static_cast<uint32_t>(lane * 128);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        st_shared_v4(rowp + (static_cast<uint32_t>(e ^ (lane & 7)) << 4), pk[4 * e],
                                     pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmY, sb, n * Cfg::TILE_N + col0 + c0, m * TILE_M + qtr * 32);
                        bulk_commit();
                    }
                }
            }
            if (nseg == 0) {  // no valid columns in this half: still release the buffer
                tc_fence_before();
                mbar_arrive(bar(WideBars::ACC_EMPTY));
            }
        }
        // Shared memory must outlive the stores' reads of it; their writes
        // complete with the grid.
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
    }

    // ---- teardown
    tc_fence_before();
    __syncthreads();
    if (CLUSTERED) {
        cluster_arrive_release();
        cluster_wait_acquire();
    }
    if (warp == Cfg::PRODUCER_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

template <int EPI, bool CLUSTERED>
GemmVariant make_wide_variant() {
    using Cfg = WideCfg<EPI, CLUSTERED>;
    return GemmVariant{EPI,
                       Cfg::TILE_N,
                       CLUSTERED,
                       CLUSTERED ? XCH_CLUSTER : XCH_NONE,
                       false,
                       0,
                       reinterpret_cast<const void*>(&nf_gemm_wide_kernel<EPI, CLUSTERED>),
                       Cfg::THREADS,
                       Cfg::SMEM_BYTES,
                       Cfg::STAGES,
                       Cfg::TMEM_COLS,
                       Cfg::TK};
}

}  // namespace nf
