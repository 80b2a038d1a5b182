// nf_flashnorm.cu -- FlashNormAttention forward for sm_103a: a LayerNorm
// prologue, a generalized dot-product attention over a short K/V sequence, a
// residual, an RMSNorm epilogue and a second residual, in one kernel (blog
// "Towards Free Normalization: Fusing Normalization into GEMM and Attention
// Kernels", §4, the fused short-K/V pseudocode).  Per batch b and query token:
//
//   ln_q = LayerNorm(q)                 over all H heads x D  (multi-CTA norm 1)
//   p    = act(ln_q[h] . K[b, :, h]^T)  per head, Lkv = 128 keys
//   o[h] = p . V[b, :, h] + ln_q[h]     (residual 1)
//   out  = RMSNorm(o) + q               over all H x D        (multi-CTA norm 2, residual 2)
//
// Layout: Q / Out [B, Lq, H, D], K / V [B, Lkv, H, D], bf16, D = Lkv = 128,
// seen by TMA as [B*L rows, H*D columns].  The grid is one cluster of H CTAs
// per batch (as in the blog: the cluster's CTAs share the batch index and take
// one head each); each CTA keeps its head's K and V in shared memory and walks
// the batch's 128-row query tiles (ceil(q_len[b] / 128) of them).
//
// CTA roles (192 threads):
//   warps 0-3  compute, one query row per thread (TMEM lane = row): the
//              LayerNorm (partial statistics over the CTA's 128 columns, pushed
//              to every CTA of the cluster with st.async, merged), writes
//              bf16(ln_q) as the first MMA's A operand and ln_q in fp32 into
//              the O accumulator (so residual 1 is the MMA's accumulate), the
//              activation of S into P (the second MMA's A operand), then the
//              RMSNorm of O (second exchange) and out = o * rstd + q, staged
//              over the q tile in shared memory and stored with TMA.
//   warp 4     TMA producer: K and V once, the q tiles into two buffers.
//   warp 5     MMA issuer: S = ln_q K^T and O += P V (tcgen05.mma, M = N = 128).
//
// Every wait is bounded; on expiry the kernel records NF_ERR_TIMEOUT with the
// site in the device status word, drains what it issued and returns.
#include "nf_internal.h"
#include "nf_ptx.cuh"

namespace nf {
namespace {

constexpr int FN_D = 128;                  // head dimension
constexpr int FN_LKV = 128;                // key / value length
constexpr int FN_ROWS = 128;               // query rows per tile
constexpr int FN_MAXH = 8;                 // heads per cluster (portable cluster size)
constexpr int FN_THREADS = 192;
constexpr int FN_PRODUCER_WARP = 4;
constexpr int FN_MMA_WARP = 5;
constexpr int FN_TILE_BYTES = FN_ROWS * FN_D * 2;  // 32 KB: a 128 x 128 bf16 tile
constexpr int FN_HALF_BYTES = FN_TILE_BYTES / 2;   // one 64-column box of 128 rows
constexpr int FN_RECV_BYTES = 2 * FN_MAXH * FN_ROWS * 8;  // [parity][cluster rank][row] float2

// Shared-memory layout (1 KB aligned base).
constexpr int FN_OFF_K = 0;                                  // K: 2 boxes of 128 keys x 64 d
constexpr int FN_OFF_V = FN_OFF_K + FN_TILE_BYTES;           // V: 2 K-tiles x 2 boxes of 64 keys x 64 d
constexpr int FN_OFF_Q = FN_OFF_V + FN_TILE_BYTES;           // q tiles [2], later the output staging
constexpr int FN_OFF_A = FN_OFF_Q + 2 * FN_TILE_BYTES;       // bf16(ln_q), then P
constexpr int FN_OFF_R1 = FN_OFF_A + FN_TILE_BYTES;          // LayerNorm partials received
constexpr int FN_OFF_R2 = FN_OFF_R1 + FN_RECV_BYTES;         // RMSNorm partials received
constexpr int FN_OFF_BAR = FN_OFF_R2 + FN_RECV_BYTES;
constexpr int FN_SMEM_BYTES = FN_OFF_BAR + 256 + 1024;       // barriers + words, 1 KB realignment slack
static_assert(FN_SMEM_BYTES <= SMEM_OPTIN_LIMIT, "shared memory");

enum FnSite : uint32_t {
    FN_SITE_KV = 20, FN_SITE_QFULL = 21, FN_SITE_QEMPTY = 22, FN_SITE_AREADY = 23, FN_SITE_SFULL = 24,
    FN_SITE_PREADY = 25, FN_SITE_OFULL = 26, FN_SITE_X1 = 27, FN_SITE_X2 = 28,
};

struct FnArgs {
    int32_t B, Lq, H;
    int32_t act;            // 0 identity, 1 GELU (tanh form), 2 SiLU
    float eps1, eps2;
    float inv_hd;           // 1 / (H * D)
    const int32_t* q_len;  // B entries or null (Lq each)
    uint32_t* status;
    uint64_t timeout_ns;
};

__device__ __forceinline__ float fn_act(float x, int act) {
    if (act == 1) return 0.5f * x * (1.0f + tanhf(0.7978845608028654f * fmaf(0.044715f * x, x * x, x)));
    if (act == 2) return x / (1.0f + expf(-x));
    return x;
}

// Address of 16-byte chunk c (0..15, 8 columns each) of row r in a 128-row,
// 128-column bf16 tile held as two 64-column boxes with the 128-byte swizzle.
__device__ __forceinline__ uint32_t fn_chunk(uint32_t base, int r, int c) {
    return base + static_cast<uint32_t>((c >> 3) * FN_HALF_BYTES + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t fn_cluster_id() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

// Bounded wait used only while draining: ignores the abort flag, records nothing.
__device__ __forceinline__ void fn_drain(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > timeout_ns) return;
}

__global__ void __launch_bounds__(FN_THREADS, 1)
    nf_flashnorm_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                            const FnArgs args) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const base_ptr = smem_raw + (base - raw);
    const uint32_t sK = base + FN_OFF_K, sV = base + FN_OFF_V, sQ = base + FN_OFF_Q, sA = base + FN_OFF_A;
    const uint32_t sR1 = base + FN_OFF_R1, sR2 = base + FN_OFF_R2, sBar = base + FN_OFF_BAR;
    const uint32_t bar_kv = sBar;               // K and V landed
    const uint32_t bar_qfull0 = sBar + 8;       // [2] q tile landed
    const uint32_t bar_qempty0 = sBar + 24;     // [2] q buffer free (its output store has read it)
    const uint32_t bar_aready = sBar + 40;      // bf16(ln_q) in sA and ln_q in O's TMEM columns
    const uint32_t bar_sfull = sBar + 48;       // S = ln_q K^T in TMEM
    const uint32_t bar_pready = sBar + 56;      // P in sA
    const uint32_t bar_ofull = sBar + 64;       // O = ln_q + P V in TMEM
    const uint32_t bar_x1 = sBar + 72;          // [2] LayerNorm partials of the cluster arrived
    const uint32_t bar_x2 = sBar + 88;          // [2] RMSNorm partials of the cluster arrived
    const uint32_t bar_mma_done = sBar + 104;
    uint32_t* const tmem_holder = reinterpret_cast<uint32_t*>(base_ptr + FN_OFF_BAR + 128);
    volatile int* const abort_flag = reinterpret_cast<volatile int*>(base_ptr + FN_OFF_BAR + 132);

    const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
    const int H = args.H;
    const int rank = static_cast<int>(cluster_ctarank());  // this CTA's head
    const int bidx = static_cast<int>(fn_cluster_id());     // this cluster's batch
    const uint32_t xbytes = static_cast<uint32_t>(H) * FN_ROWS * 8u;
    const WaitGuard guard{args.status, abort_flag, args.timeout_ns};

    if (threadIdx.x == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmO);
        mbar_init(bar_kv, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_qfull0 + 8u * i, 1);
            mbar_init(bar_qempty0 + 8u * i, 4);  // one arrival per compute warp
            mbar_init(bar_x1 + 8u * i, 1);
            mbar_init(bar_x2 + 8u * i, 1);
        }
        mbar_init(bar_aready, 128);
        mbar_init(bar_sfull, 1);
        mbar_init(bar_pready, 128);
        mbar_init(bar_ofull, 1);
        mbar_init(bar_mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == FN_PRODUCER_WARP) {
        tmem_alloc(smem_u32(tmem_holder), 256);  // S: columns 0-127, O: 128-255
        tmem_relinquish();
    }
    // Global memory (q_len included) is read only after the preceding grid.
    griddep_wait();
    griddep_launch_dependents();
    const int qlen = args.q_len ? min(max(args.q_len[bidx], 0), args.Lq) : args.Lq;
    const int tiles = (qlen + FN_ROWS - 1) / FN_ROWS;  // the same for every CTA of the cluster
    if (threadIdx.x == 0) {
        // Arm the exchange barriers of tiles 0 and 1 before any peer can send
        // (peers send only after the cluster barrier below).
        for (int i = 0; i < 2 && i < tiles; ++i) {
            mbar_arrive_expect_tx(bar_x1 + 8u * i, xbytes);
            mbar_arrive_expect_tx(bar_x2 + 8u * i, xbytes);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_arrive_release();
    cluster_wait_acquire();
    const uint32_t tmem_base = *tmem_holder;
    const int64_t qrow0 = static_cast<int64_t>(bidx) * args.Lq;  // the batch's first row in Q / Out
    const int col0 = rank * FN_D;                                 // this head's first column

    if (warp == FN_PRODUCER_WARP) {
        // ======================================================== TMA producer
        if (lane == 0 && tiles > 0) {
            mbar_arrive_expect_tx(bar_kv, 2 * FN_TILE_BYTES);
            const int krow = bidx * FN_LKV;
            for (int kt = 0; kt < 2; ++kt) {
                // K: 128 keys x 64 d (K-major B of S); V: 64 keys x 64 d boxes (MN-major B of O)
                tma_load_2d(sK + kt * FN_HALF_BYTES, &tmK, bar_kv, col0 + kt * 64, krow);
                for (int i = 0; i < 2; ++i)
                    tma_load_2d(sV + kt * FN_HALF_BYTES + i * (FN_HALF_BYTES / 2), &tmV, bar_kv, col0 + i * 64,
                                krow + kt * 64);
            }
            for (int it = 0; it < tiles; ++it) {
                const int qb = it & 1;
                const uint32_t ph = static_cast<uint32_t>(it >> 1) & 1u;
                if (!mbar_wait(guard, bar_qempty0 + 8u * qb, ph ^ 1u, FN_SITE_QEMPTY, it)) break;
                const uint32_t fb = bar_qfull0 + 8u * qb;
                mbar_arrive_expect_tx(fb, FN_TILE_BYTES);
                for (int half = 0; half < 2; ++half)
                    tma_load_2d(sQ + qb * FN_TILE_BYTES + half * FN_HALF_BYTES, &tmQ, fb, col0 + half * 64,
                                static_cast<int32_t>(qrow0 + it * FN_ROWS));
            }
            // Every load issued has landed before the CTA may exit.
            fn_drain(bar_kv, 0, args.timeout_ns);
            for (int j = 0; j < 2 && j < tiles; ++j) {
                const int last = j + ((tiles - 1 - j) / 2) * 2;  // the last tile that used buffer j
                fn_drain(bar_qfull0 + 8u * j, static_cast<uint32_t>(last >> 1) & 1u, args.timeout_ns);
            }
        }
        __syncwarp();
    } else if (warp == FN_MMA_WARP) {
        // ======================================================== MMA issuer
        if (lane == 0 && tiles > 0) {
            constexpr uint32_t IDESC_S = idesc_bf16_f32(FN_ROWS, FN_LKV, false);  // B = K (K-major)
            constexpr uint32_t IDESC_O = idesc_bf16_f32(FN_ROWS, FN_D, true);     // B = V (MN-major)
            const uint32_t tS = tmem_base, tO = tmem_base + 128u;
            bool ok = mbar_wait(guard, bar_kv, 0, FN_SITE_KV, 0);
            for (int it = 0; it < tiles && ok; ++it) {
                const uint32_t ph = static_cast<uint32_t>(it) & 1u;
                if (!(ok = mbar_wait(guard, bar_aready, ph, FN_SITE_AREADY, it))) break;
                tc_fence_after();
                for (int kt = 0; kt < 2; ++kt)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        mma_bf16(tS, smem_desc_sw128(sA + kt * FN_HALF_BYTES + j * 32, 16, 1024),
                                 smem_desc_sw128(sK + kt * FN_HALF_BYTES + j * 32, 16, 1024), IDESC_S,
                                 (kt | j) != 0 ? 1u : 0u);
                mma_commit(bar_sfull);
                if (!(ok = mbar_wait(guard, bar_pready, ph, FN_SITE_PREADY, it))) break;
                tc_fence_after();
                for (int kt = 0; kt < 2; ++kt)
#pragma unroll
                    for (int j = 0; j < 4; ++j)  // O already holds ln_q: accumulate from the first step
                        mma_bf16(tO, smem_desc_sw128(sA + kt * FN_HALF_BYTES + j * 32, 16, 1024),
                                 smem_desc_sw128(sV + kt * FN_HALF_BYTES + j * 2048, FN_HALF_BYTES / 2, 1024),
                                 IDESC_O, 1u);
                mma_commit(bar_ofull);
            }
            mma_commit(bar_mma_done);
            fn_drain(bar_mma_done, 0, args.timeout_ns);
        }
        __syncwarp();
    } else {
        // ======================================================== compute warps 0-3
        const int r = warp * 32 + lane;  // tile row == TMEM lane
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(warp * 32) << 16);
        const uint32_t tS = t_lane, tO = t_lane + 128u;
        for (int it = 0; it < tiles; ++it) {
            const int qb = it & 1;
            const uint32_t ph = static_cast<uint32_t>(it) & 1u, qph = static_cast<uint32_t>(it >> 1) & 1u;
            const int m0 = it * FN_ROWS;
            const bool valid = m0 + r < qlen;
            const uint32_t sq = sQ + static_cast<uint32_t>(qb * FN_TILE_BYTES);
            bool ok = mbar_wait(guard, bar_qfull0 + 8u * qb, qph, FN_SITE_QFULL, it);
            if (!__all_sync(0xffffffffu, ok)) break;

            // ---- LayerNorm: partial (mean, M2) over this CTA's 128 columns,
            //      sums shifted by the row's first value; rows past q_len are zero.
            float sh, a1 = 0.0f, a2 = 0.0f;
            {
                const uint4 w = ld_shared_v4(fn_chunk(sq, r, 0));
                sh = valid ? bf16lo(w.x) : 0.0f;
            }
#pragma unroll 4
            for (int c = 0; c < 16; ++c) {
                const uint4 w = ld_shared_v4(fn_chunk(sq, r, c));
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float d0 = (valid ? bf16lo(ww[e]) : 0.0f) - sh, d1 = (valid ? bf16hi(ww[e]) : 0.0f) - sh;
                    a1 += d0 + d1;
                    a2 = fmaf(d0, d0, fmaf(d1, d1, a2));
                }
            }
            const float mean_c = sh + a1 * (1.0f / FN_D);
            const float m2_c = fmaxf(fmaf(-a1, a1 * (1.0f / FN_D), a2), 0.0f);
            const int xp = it & 1;
            {
                // push to slot [rank] of every CTA of the cluster, wait for all H slots
                const uint32_t x1 = bar_x1 + 8u * xp;
                const uint32_t slot = sR1 + static_cast<uint32_t>(((xp * FN_MAXH + rank) * FN_ROWS + r) * 8);
                for (int p = 0; p < H; ++p) st_async_f32x2(mapa_shared(slot, p), mean_c, m2_c, mapa_shared(x1, p));
                ok = mbar_wait<true>(guard, x1, qph, FN_SITE_X1, it);
                if (!__all_sync(0xffffffffu, ok)) break;
                // Re-arm for tile it + 2: its partials can arrive only after every
                // CTA got this CTA's tile it + 1 partials, sent after this point.
                if (warp == 0 && lane == 0 && it + 2 < tiles) mbar_arrive_expect_tx(x1, xbytes);
            }
            const float* rv1 = reinterpret_cast<const float*>(base_ptr + FN_OFF_R1 + (xp * FN_MAXH * FN_ROWS + r) * 8);
            float msum = 0.0f;
            for (int p = 0; p < H; ++p) msum += rv1[p * FN_ROWS * 2];
            const float mean = msum / static_cast<float>(H);
            float m2 = 0.0f;
            for (int p = 0; p < H; ++p) {  // Chan et al. merge, D values per partial
                const float dm = rv1[p * FN_ROWS * 2] - mean;
                m2 += rv1[p * FN_ROWS * 2 + 1] + static_cast<float>(FN_D) * dm * dm;
            }
            const float rstd1 = rsqrtf(fmaf(m2, args.inv_hd, args.eps1));

            // ---- ln_q: bf16 into sA (the first MMA's A operand, K-major) and
            //      fp32 into O's TMEM columns (residual 1 through the MMA's accumulate).
#pragma unroll 1
            for (int seg = 0; seg < 4; ++seg) {
                uint32_t lv[32];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int c = seg * 4 + k;
                    const uint4 w = ld_shared_v4(fn_chunk(sq, r, c));
                    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
                    uint32_t pk[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float l0 = valid ? (bf16lo(ww[e]) - mean) * rstd1 : 0.0f;
                        const float l1 = valid ? (bf16hi(ww[e]) - mean) * rstd1 : 0.0f;
                        lv[k * 8 + 2 * e] = __float_as_uint(l0);
                        lv[k * 8 + 2 * e + 1] = __float_as_uint(l1);
                        pk[e] = pack_bf16x2(l0, l1);
                    }
                    st_shared_v4(fn_chunk(sA, r, c), pk[0], pk[1], pk[2], pk[3]);
                }
                tmem_st32(tO + static_cast<uint32_t>(seg * 32), lv);
            }
            tmem_st_wait();
            fence_proxy_async_smem();  // the tensor cores read sA
            tc_fence_before();
            mbar_arrive(bar_aready);

            // ---- activation: P = bf16(act(S)) into sA (the second MMA's A operand)
            ok = mbar_wait(guard, bar_sfull, ph, FN_SITE_SFULL, it);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
#pragma unroll 1
            for (int seg = 0; seg < 4; ++seg) {
                uint32_t v[32];
                tmem_ld32(tS + static_cast<uint32_t>(seg * 32), v);
                tmem_ld_wait(v);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    uint32_t pk[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        pk[e] = pack_bf16x2(fn_act(__uint_as_float(v[k * 8 + 2 * e]), args.act),
                                            fn_act(__uint_as_float(v[k * 8 + 2 * e + 1]), args.act));
                    st_shared_v4(fn_chunk(sA, r, seg * 4 + k), pk[0], pk[1], pk[2], pk[3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar_pready);

            // ---- RMSNorm of O over all heads (second exchange), out = o * rstd + q
            ok = mbar_wait(guard, bar_ofull, ph, FN_SITE_OFULL, it);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            float ss0 = 0.0f, ss1 = 0.0f;
#pragma unroll 1
            for (int seg = 0; seg < 4; ++seg) {
                uint32_t v[32];
                tmem_ld32(tO + static_cast<uint32_t>(seg * 32), v);
                tmem_ld_wait(v);
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const float o0 = __uint_as_float(v[i]), o1 = __uint_as_float(v[i + 1]);
                    ss0 = fmaf(o0, o0, ss0);
                    ss1 = fmaf(o1, o1, ss1);
                }
            }
            {
                const uint32_t x2 = bar_x2 + 8u * xp;
                const uint32_t slot = sR2 + static_cast<uint32_t>(((xp * FN_MAXH + rank) * FN_ROWS + r) * 8);
                for (int p = 0; p < H; ++p) st_async_f32x2(mapa_shared(slot, p), ss0 + ss1, 0.0f, mapa_shared(x2, p));
                ok = mbar_wait<true>(guard, x2, qph, FN_SITE_X2, it);
                if (!__all_sync(0xffffffffu, ok)) break;
                if (warp == 0 && lane == 0 && it + 2 < tiles) mbar_arrive_expect_tx(x2, xbytes);
            }
            const float* rv2 = reinterpret_cast<const float*>(base_ptr + FN_OFF_R2 + (xp * FN_MAXH * FN_ROWS + r) * 8);
            float tot = 0.0f;
            for (int p = 0; p < H; ++p) tot += rv2[p * FN_ROWS * 2];
            const float rstd2 = rsqrtf(fmaf(tot, args.inv_hd, args.eps2));
#pragma unroll 1
            for (int seg = 0; seg < 4; ++seg) {
                uint32_t v[32];
                tmem_ld32(tO + static_cast<uint32_t>(seg * 32), v);
                tmem_ld_wait(v);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t a = fn_chunk(sq, r, seg * 4 + k);  // q, overwritten in place by out
                    const uint4 w = ld_shared_v4(a);
                    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
                    uint32_t pk[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float y0 = valid ? fmaf(__uint_as_float(v[k * 8 + 2 * e]), rstd2, bf16lo(ww[e])) : 0.0f;
                        const float y1 = valid ? fmaf(__uint_as_float(v[k * 8 + 2 * e + 1]), rstd2, bf16hi(ww[e])) : 0.0f;
                        pk[e] = pack_bf16x2(y0, y1);
                    }
                    st_shared_v4(a, pk[0], pk[1], pk[2], pk[3]);
                }
            }
            fence_proxy_async_smem();  // the TMA store reads the staged rows
            __syncwarp();
            if (lane == 0) {
                // This warp's 32 rows, two 64-column boxes; none past the batch's
                // last 32-row group that holds a valid row.
                if (m0 + warp * 32 < qlen) {
                    for (int half = 0; half < 2; ++half)
                        tma_store_2d(&tmO, sq + static_cast<uint32_t>(half * FN_HALF_BYTES + warp * 32 * 128),
                                     col0 + half * 64, static_cast<int32_t>(qrow0 + m0 + warp * 32));
                    bulk_commit();
                    bulk_wait_read<0>();  // the buffer is read before the next q tile lands in it
                }
                mbar_arrive(bar_qempty0 + 8u * qb);
            }
            __syncwarp();
        }
    }

    // ---- teardown: no CTA leaves while a peer may still write into its shared memory
    tc_fence_before();
    __syncthreads();
    cluster_arrive_release();
    cluster_wait_acquire();
    if (warp == FN_PRODUCER_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 256);
    }
}

}  // namespace

cudaError_t launch_flashnorm_fwd(const void* tmaps, const FlashNormLaunch& a, bool overlap, cudaStream_t stream) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(nf_flashnorm_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             FN_SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const CUtensorMap* m = static_cast<const CUtensorMap*>(tmaps);
    FnArgs args;
    args.B = a.B;
    args.Lq = a.Lq;
    args.H = a.H;
    args.act = a.act;
    args.eps1 = a.eps1;
    args.eps2 = a.eps2;
    args.inv_hd = 1.0f / static_cast<float>(a.H * FN_D);
    args.q_len = a.q_len;
    args.status = a.status;
    args.timeout_ns = a.timeout_ns;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    int n = 0;
    cfg.gridDim = dim3(static_cast<unsigned>(a.B * a.H));
    cfg.blockDim = dim3(FN_THREADS);
    cfg.dynamicSmemBytes = FN_SMEM_BYTES;
    cfg.stream = stream;
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(a.H);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
    if (overlap) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = static_cast<unsigned>(n);
    return cudaLaunchKernelEx(&cfg, nf_flashnorm_fwd_kernel, m[0], m[1], m[2], m[3], args);
}

}  // namespace nf
