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
// seen by TMA as [B*L rows, H*D columns].  A cluster of H CTAs works on one
// batch at a time (as in the blog: the cluster's CTAs share the batch index and
// take one head each); each CTA keeps its head's K and V in shared memory and
// walks the batch's 128-row query tiles (ceil(q_len[b] / 128) of them).  The
// grid is persistent: as many clusters as are resident at once, each taking
// the next batch from a global counter when it starts the previous one (its
// rank 0 takes it and writes it into every CTA's batch ring), so set-up,
// teardown and the first loads are paid once per cluster rather than per batch,
// and jagged batches balance dynamically.  Query tiles are numbered across
// batches, so the q prefetch, the exchange slots and all phase parities run on
// through batch switches; a batch's K and V replace the previous ones once
// every group is done with them (the kvfree barrier).
//
// CTA roles, NG compute groups (NG = 2 for H <= 4; 1 above, where two groups'
// exchange slots for up to 16 partials per row would crowd out the q buffers):
//   warps 8g..8g+7  compute group g, tiles g, g + NG, ...; warp 8g + 4hf + q4
//              takes rows 32q4 .. 32q4 + 31 (its TMEM lane quarter) and the 64
//              columns of half hf, one half row per thread: the LayerNorm
//              (partial statistics over the 64 columns, pushed to every CTA of
//              the cluster with st.async, 2H partials per row merged);
//              bf16(ln_q) into TMEM as the first MMA's A operand; P =
//              bf16(act(S)) for keys 64hf .. 64hf + 63 into TMEM over S's
//              columns already read, the second MMA's A operand; o = P V + ln_q
//              (residual 1, ln_q recomputed from q in fp32), its RMSNorm
//              (second exchange) and out = o * rstd + q, staged over the q tile
//              and stored with TMA.  Two groups overlap one tile's exchanges
//              and MMAs with the other tile's CUDA-core work.
//   warp 8NG   TMA producer: the batch sequence, each batch's K and V, the q
//              tiles into NQ = 4 buffers (tile it into buffer it mod 4, with a
//              record of its batch, rows, K/V load and whether it is its
//              group's last tile of the batch), each refilled once its
//              tile's output stores have read it, so a group's next tile lands
//              while it computes the current one.
//   warp 8NG+1+g  MMA issuer of group g: S = ln_q K^T (two 64-key halves) and
//              O = P V (tcgen05.mma, A from TMEM, B from shared memory) in the
//              group's 256 TMEM columns (S / P 128, O / bf16(ln_q) 128); each
//              contraction runs in two halves, released as the compute group
//              writes the matching half of its A operand.
//
// Exchange slots: tile it uses slot it mod NG of each exchange, so slot s
// serves group s alone and a slot is reused by the same group's next tile,
// it + NG.  A peer sends its partials of tile it + NG to the LayerNorm slot
// only after its RMSNorm exchange of tile it completed, which needs every
// thread of this CTA's group to have sent its RMSNorm partial of tile it,
// which each does after reading its LayerNorm partials of tile it.  Likewise a
// peer sends to the RMSNorm slot for tile it + NG only after the LayerNorm
// exchange of tile it + NG, which each thread here joins after reading its
// RMSNorm partials of tile it.  So no slot is overwritten before it is read,
// and no slot's barrier completes a second phase before every thread here has
// waited on the first.
//
// Every wait is bounded; on expiry the kernel records NF_ERR_TIMEOUT with the
// site in the device status word, drains what it issued and returns.
#include <mutex>

#include "nf_internal.h"
#include "nf_ptx.cuh"

namespace nf {
namespace {

constexpr int FN_D = 128;                          // head dimension
constexpr int FN_LKV = 128;                        // key / value length
constexpr int FN_ROWS = 128;                       // query rows per tile
constexpr int FN_TILE_BYTES = FN_ROWS * FN_D * 2;  // 32 KB: a 128 x 128 bf16 tile
constexpr int FN_HALF_BYTES = FN_TILE_BYTES / 2;   // one 64-column box of 128 rows

template <int NG>
struct FnCfg {
    static constexpr int MAXH = NG == 2 ? 4 : 8;   // heads per cluster
    static constexpr int NSLOT = NG;               // exchange slots
    static constexpr int THREADS = (8 * NG + 1 + NG) * 32;
    static constexpr int PRODUCER_WARP = 8 * NG;
    static constexpr int MMA_WARP0 = 8 * NG + 1;
    static constexpr int NQ = 4;                                  // q tile buffers
    // received partials: [slot][cluster rank x column half][row] float2
    static constexpr int RECV_BYTES = NSLOT * 2 * MAXH * FN_ROWS * 8;
    // Shared-memory layout (1 KB aligned base).
    static constexpr int OFF_K = 0;                               // K: 2 boxes of 128 keys x 64 d
    static constexpr int OFF_V = OFF_K + FN_TILE_BYTES;           // V: 2 K-tiles x 2 boxes of 64 keys x 64 d
    static constexpr int OFF_Q = OFF_V + FN_TILE_BYTES;           // q tiles [NQ], later the output staging
    static constexpr int OFF_R1 = OFF_Q + NQ * FN_TILE_BYTES;     // LayerNorm partials received
    static constexpr int OFF_R2 = OFF_R1 + RECV_BYTES;            // RMSNorm partials received
    static constexpr int OFF_BAR = OFF_R2 + RECV_BYTES;
    static constexpr int SMEM_BYTES = OFF_BAR + 512 + 1024;       // barriers + words, 1 KB realignment slack
    static_assert(SMEM_BYTES <= SMEM_OPTIN_LIMIT, "shared memory");
    static constexpr int NB = 4;                                  // batch ring entries
    // barriers (8 bytes each): kv, qfull[NQ], qempty[NQ], GROUP_BARS per group
    // (below), x1[NSLOT], x2[NSLOT], bfull[NB], bempty[NB], kvfree
    static constexpr int B_KV = 0, B_QFULL = 1, B_QEMPTY = 1 + NQ, B_GROUP = 1 + 2 * NQ, GROUP_BARS = 8,
                         B_X1 = B_GROUP + GROUP_BARS * NG, B_X2 = B_X1 + NSLOT, B_BFULL = B_X2 + NSLOT,
                         B_BEMPTY = B_BFULL + NB, B_KVFREE = B_BEMPTY + NB, NBAR = B_KVFREE + 1;
    static_assert(NBAR * 8 <= 320, "barrier area");
    // words after the barriers: the batch ring (NB int32), the tile records
    // (NQ x FnTile), the TMEM base, the abort flag
    static constexpr int OFF_RING = 320, OFF_TILES = 384, OFF_TMEM_HOLDER = 504, OFF_ABORT = 508;
    static_assert(OFF_TILES + NQ * 20 <= OFF_TMEM_HOLDER, "tile records");
    static constexpr int TMEM_COLS = 256 * NG;     // per group: S 128 columns, O 128
};

// A group's barriers, by offset from its first: the two halves of the
// contraction of S (ln_q columns 0-63 / 64-127 written), the two 64-key halves
// of S (computed), the two 64-key halves of P (written), O (computed) and the
// MMA warp's final drain.
constexpr int G_AREADY = 0, G_SFULL = 2, G_PREADY = 4, G_OFULL = 6, G_MMA_DONE = 7;

enum FnSite : uint32_t {
    FN_SITE_KV = 20, FN_SITE_QFULL = 21, FN_SITE_QEMPTY = 22, FN_SITE_AREADY = 23, FN_SITE_SFULL = 24,
    FN_SITE_PREADY = 25, FN_SITE_OFULL = 26, FN_SITE_X1 = 27, FN_SITE_X2 = 28, FN_SITE_BATCH = 29,
    FN_SITE_BEMPTY = 30, FN_SITE_KVFREE = 31,
};

// What the producer tells the compute and MMA warps about the query tile in a
// q buffer: its batch (-1: no more tiles for this group), its first row within
// the batch, the batch's valid length, which K/V load (0, 1, ...) it uses and
// whether it is its group's last tile of the batch.
struct FnTile {
    int32_t b, m0, qlen, kv, last;
};
static_assert(sizeof(FnTile) == 20, "tile record");

struct FnArgs {
    int32_t B, Lq, H;
    int32_t act;            // 0 identity, 1 GELU (tanh form), 2 SiLU
    float eps1, eps2;
    float inv_hd;           // 1 / (H * D)
    const int32_t* q_len;  // B entries or null (Lq each)
    int32_t* sched;        // [0] next batch to hand out, [1] clusters done; zero between launches
    uint32_t* status;
    uint64_t timeout_ns;
};

// Hardware tanh (MUFU, about 2^-11 relative error: below the bf16 rounding
// that P gets before the second MMA).
__device__ __forceinline__ float fn_tanh(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// P = bf16(act(s)) for two S values held as 32-bit words, in packed fp32 pairs:
//   GELU (tanh form)  h + h tanh(u),  h = s / 2,  u = sqrt(2 / pi) (s + 0.044715 s^3)
//   SiLU              h + h tanh(h),  h = s / 2   (s sigmoid(s), written with tanh)
//   identity          s
template <int ACT>
__device__ __forceinline__ uint32_t fn_act_pack(uint32_t s0, uint32_t s1) {
    const uint64_t x = f2_pack(s0, s1);
    if (ACT == 0) return pack_bf16x2(__uint_as_float(s0), __uint_as_float(s1));
    const uint64_t h = f2_mul(x, f2_splat(0.5f));
    uint64_t u = h;
    if (ACT == 1) {
        constexpr float K0 = 0.7978845608028654f, K1 = 0.7978845608028654f * 0.044715f;
        u = f2_mul(x, f2_fma(f2_mul(x, x), f2_splat(K1), f2_splat(K0)));
    }
    float u0, u1;
    f2_unpack(u, u0, u1);
    const uint64_t th = f2_pack(__float_as_uint(fn_tanh(u0)), __float_as_uint(fn_tanh(u1)));
    return f2_to_bf16x2(f2_fma(h, th, h));
}

// Address of 16-byte chunk c (0..15, 8 columns each) of row r in a 128-row,
// 128-column bf16 tile held as two 64-column boxes with the 128-byte swizzle.
__device__ __forceinline__ uint32_t fn_chunk(uint32_t base, int r, int c) {
    return base + static_cast<uint32_t>((c >> 3) * FN_HALF_BYTES + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// The activation of one 64-key half of S (TMEM columns ts .. ts + 63 of this
// thread's row), as 32 bf16 pairs into the TMEM columns tp .. tp + 31, in two
// 32-key parts; tp <= ts, so each part's results land on columns already read.
template <int ACT>
__device__ __forceinline__ void fn_act_half(uint32_t ts, uint32_t tp) {
#pragma unroll 1
    for (int part = 0; part < 2; ++part) {
        uint32_t v[32], pk[16];
        tmem_ld32(ts + static_cast<uint32_t>(part * 32), v);
        tmem_ld_wait(v);
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = fn_act_pack<ACT>(v[2 * i], v[2 * i + 1]);
        tmem_st16(tp + static_cast<uint32_t>(part * 16), pk);
    }
}

// One 32-bit value into a (possibly remote) CTA's shared memory, completing 4
// bytes of the transaction count of the barrier at the same CTA.
__device__ __forceinline__ void fn_st_async_s32(uint32_t remote_addr, int32_t v, uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.s32 [%0], %1, [%2];" ::"r"(remote_addr),
                 "r"(v), "r"(remote_bar)
                 : "memory");
}

// Arrive on a barrier in a (possibly remote) CTA of the cluster, releasing this
// thread's earlier accesses at cluster scope.
__device__ __forceinline__ void fn_arrive_remote(uint32_t remote_bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar) : "memory");
}

// Bounded wait used only while draining: ignores the abort flag, records nothing.
__device__ __forceinline__ void fn_drain(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > timeout_ns) return;
}

template <int NG>
__global__ void __launch_bounds__(FnCfg<NG>::THREADS, 1)
    nf_flashnorm_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                            const FnArgs args) {
    using C = FnCfg<NG>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const base_ptr = smem_raw + (base - raw);
    const uint32_t sK = base + C::OFF_K, sV = base + C::OFF_V, sQ = base + C::OFF_Q;
    const uint32_t sR1 = base + C::OFF_R1, sR2 = base + C::OFF_R2, sBar = base + C::OFF_BAR;
    auto bar = [&](int slot) { return sBar + 8u * static_cast<uint32_t>(slot); };
    uint32_t* const tmem_holder = reinterpret_cast<uint32_t*>(base_ptr + C::OFF_BAR + C::OFF_TMEM_HOLDER);
    volatile int* const abort_flag = reinterpret_cast<volatile int*>(base_ptr + C::OFF_BAR + C::OFF_ABORT);

    const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
    const int H = args.H;
    const int rank = static_cast<int>(cluster_ctarank());  // this CTA's head
    const uint32_t xbytes = static_cast<uint32_t>(2 * H) * FN_ROWS * 8u;  // one partial per row and column half
    const WaitGuard guard{args.status, abort_flag, args.timeout_ns};
    const uint32_t sRing = sBar + C::OFF_RING;
    volatile int32_t* const ring = reinterpret_cast<volatile int32_t*>(base_ptr + C::OFF_BAR + C::OFF_RING);
    volatile FnTile* const tile_rec = reinterpret_cast<volatile FnTile*>(base_ptr + C::OFF_BAR + C::OFF_TILES);

    if (threadIdx.x == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmO);
        mbar_init(bar(C::B_KV), 1);
        for (int i = 0; i < C::NQ; ++i) {
            mbar_init(bar(C::B_QFULL + i), 1);
            mbar_init(bar(C::B_QEMPTY + i), 8);  // one arrival per warp of the group using the buffer
        }
        for (int g = 0; g < NG; ++g) {
            const int b0 = C::B_GROUP + g * C::GROUP_BARS;
            for (int h = 0; h < 2; ++h) {
                mbar_init(bar(b0 + G_AREADY + h), 128);  // every thread of the group
                mbar_init(bar(b0 + G_SFULL + h), 1);     // an MMA commit
                mbar_init(bar(b0 + G_PREADY + h), 128);
            }
            mbar_init(bar(b0 + G_OFULL), 1);
            mbar_init(bar(b0 + G_MMA_DONE), 1);
        }
        for (int s = 0; s < C::NSLOT; ++s) {
            mbar_init(bar(C::B_X1 + s), 1);
            mbar_init(bar(C::B_X2 + s), 1);
        }
        for (int s = 0; s < C::NB; ++s) {
            mbar_init(bar(C::B_BFULL + s), 1);  // the ring entry, written by the cluster's rank 0
            mbar_init(bar(C::B_BEMPTY + s), H);  // (rank 0's) every CTA has read the entry
        }
        // One phase per K/V load: every group is done with it (an MMA commit
        // after the group's last tile of the batch, or the producer's arrival for
        // a group without tiles in it).
        mbar_init(bar(C::B_KVFREE), NG);
        *abort_flag = 0;
        fence_mbar_init();
        // Arm the exchange and ring barriers before any peer can write (peers
        // write only after the cluster barrier below).
        for (int s = 0; s < C::NSLOT; ++s) {
            mbar_arrive_expect_tx(bar(C::B_X1 + s), xbytes);
            mbar_arrive_expect_tx(bar(C::B_X2 + s), xbytes);
        }
        for (int s = 0; s < C::NB; ++s) mbar_arrive_expect_tx(bar(C::B_BFULL + s), 4);
    }
    if (warp == C::PRODUCER_WARP) {
        tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish();
    }
    // Global memory (the scheduler words and q_len included) is touched only
    // after the preceding grid.
    griddep_wait();
    griddep_launch_dependents();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_arrive_release();
    cluster_wait_acquire();
    const uint32_t tmem_base = *tmem_holder;
    const int col0 = rank * FN_D;  // this head's first column

    if (warp == C::PRODUCER_WARP) {
        // ======================================================== TMA producer
        // The cluster walks batches handed out one at a time by a global
        // counter (the cluster's rank 0 takes them and publishes each in every
        // CTA's batch ring); the CTAs of a cluster see the same batches, hence
        // the same sequence of query tiles t = 0, 1, ...
        if (lane == 0) {
            int t = 0;          // query tiles issued
            int kv_loads = 0;   // K/V loads issued (one per batch with tiles)
            // rank 0: entry k of the ring = the next batch from the counter, or -1
            auto publish = [&](int k) -> bool {
                const int s = k % C::NB;
                if (k >= C::NB && !mbar_wait<true>(guard, bar(C::B_BEMPTY + s), static_cast<uint32_t>(k / C::NB - 1) & 1u,
                                                   FN_SITE_BEMPTY, k))
                    return false;
                const int i = atomicAdd(args.sched, 1);
                const int b = i < args.B ? i : -1;
                for (int p = 0; p < H; ++p)
                    fn_st_async_s32(mapa_shared(sRing + 4u * s, p), b, mapa_shared(bar(C::B_BFULL + s), p));
                return true;
            };
            bool ok = rank != 0 || publish(0);
            for (int nb = 0; ok; ++nb) {
                const int s = nb % C::NB;
                if (!(ok = mbar_wait<true>(guard, bar(C::B_BFULL + s), static_cast<uint32_t>(nb / C::NB) & 1u,
                                           FN_SITE_BATCH, nb)))
                    break;
                const int b = ring[s];
                mbar_arrive_expect_tx(bar(C::B_BFULL + s), 4);             // for entry nb + NB
                fn_arrive_remote(mapa_shared(bar(C::B_BEMPTY + s), 0));   // rank 0 may refill the entry
                if (b < 0) break;
                if (rank == 0 && !(ok = publish(nb + 1))) break;           // ahead of this batch's loads
                const int qlen = args.q_len ? min(max(args.q_len[b], 0), args.Lq) : args.Lq;
                const int tiles = (qlen + FN_ROWS - 1) / FN_ROWS;
                if (tiles == 0) continue;
                const int kv = kv_loads;  // this batch's K/V load
                const int64_t qrow0 = static_cast<int64_t>(b) * args.Lq;
                const int t_first = t;
                // q tile m of this batch into the next buffer, with its record
                auto issue_tile = [&](int m) -> bool {
                    const int qb = t % C::NQ;
                    if (!mbar_wait(guard, bar(C::B_QEMPTY + qb), (static_cast<uint32_t>(t / C::NQ) & 1u) ^ 1u,
                                   FN_SITE_QEMPTY, t))
                        return false;
                    tile_rec[qb].b = b;
                    tile_rec[qb].m0 = m * FN_ROWS;
                    tile_rec[qb].qlen = qlen;
                    tile_rec[qb].kv = kv;
                    tile_rec[qb].last = m + NG >= tiles ? 1 : 0;
                    const uint32_t fb = bar(C::B_QFULL + qb);
                    mbar_arrive_expect_tx(fb, FN_TILE_BYTES);  // releases the record with the phase
                    for (int half = 0; half < 2; ++half)
                        tma_load_2d(sQ + qb * FN_TILE_BYTES + half * FN_HALF_BYTES, &tmQ, fb, col0 + half * 64,
                                    static_cast<int32_t>(qrow0 + m * FN_ROWS));
                    ++t;
                    return true;
                };
                // Tiles whose buffer is already free go out before this batch's K and
                // V (at most NQ: their buffers were freed by earlier batches' tiles),
                // so their LayerNorm overlaps the wait below; the rest follow the
                // K/V load.  Only once the previous K/V load has landed, though: an
                // MMA warp whose group had no tile in the previous batch waits for
                // this batch's load by parity, which is exact only if the load
                // before it is complete.
                int m = 0;
                while (m < tiles && t < t_first + C::NQ &&
                       (kv == 0 || mbar_try_wait(bar(C::B_KV), static_cast<uint32_t>(kv - 1) & 1u)) &&
                       mbar_try_wait(bar(C::B_QEMPTY + t % C::NQ), (static_cast<uint32_t>(t / C::NQ) & 1u) ^ 1u))
                    if (!(ok = issue_tile(m++))) break;
                if (!ok) break;
                // K and V are overwritten once every group is done with the previous
                // load: phase kv - 1 of the kvfree barrier.  (Its phases run in step
                // with the loads, so the parity test cannot alias: a wait on a
                // barrier's per-tile phases, seen only at batch switches, could.)
                if (kv > 0 &&
                    !(ok = mbar_wait(guard, bar(C::B_KVFREE), static_cast<uint32_t>(kv - 1) & 1u, FN_SITE_KVFREE, t)))
                    break;
                mbar_arrive_expect_tx(bar(C::B_KV), 2 * FN_TILE_BYTES);
                const int krow = b * FN_LKV;
                for (int kt = 0; kt < 2; ++kt) {
                    // K: 128 keys x 64 d (K-major B of S); V: 64 keys x 64 d boxes (MN-major B of O)
                    tma_load_2d(sK + kt * FN_HALF_BYTES, &tmK, bar(C::B_KV), col0 + kt * 64, krow);
                    for (int i = 0; i < 2; ++i)
                        tma_load_2d(sV + kt * FN_HALF_BYTES + i * (FN_HALF_BYTES / 2), &tmV, bar(C::B_KV),
                                    col0 + i * 64, krow + kt * 64);
                }
                ++kv_loads;
                for (int n = tiles; n < NG; ++n) mbar_arrive(bar(C::B_KVFREE));  // each group without a tile here
                for (; m < tiles && ok; ++m) ok = issue_tile(m);
                if (!ok) break;
            }
            // Every load issued has landed before the CTA may exit (waited here,
            // before the end records below complete further phases of the q
            // buffers' barriers).
            const int loaded = t;  // tiles 0 .. loaded - 1 were loaded, in order
            if (kv_loads > 0) fn_drain(bar(C::B_KV), static_cast<uint32_t>(kv_loads - 1) & 1u, args.timeout_ns);
            for (int j = 0; j < C::NQ && j < loaded; ++j) {
                const int last = j + (loaded - 1 - j) / C::NQ * C::NQ;  // the last tile loaded into buffer j
                fn_drain(bar(C::B_QFULL + j), static_cast<uint32_t>(last / C::NQ) & 1u, args.timeout_ns);
            }
            // One end record per group (its next tile), so every group and MMA warp stops.
            for (int k = 0; k < NG && ok; ++k, ++t) {
                const int qb = t % C::NQ;
                if (!(ok = mbar_wait(guard, bar(C::B_QEMPTY + qb), (static_cast<uint32_t>(t / C::NQ) & 1u) ^ 1u,
                                     FN_SITE_QEMPTY, t)))
                    break;
                tile_rec[qb].b = -1;
                mbar_arrive(bar(C::B_QFULL + qb));
            }
            if (rank == 0) {
                // This cluster takes no more batches; the last cluster to finish
                // zeroes the counters for the next launch on this stream.
                __threadfence();
                const int clusters = static_cast<int>(gridDim.x) / H;
                if (atomicAdd(args.sched + 1, 1) == clusters - 1) {
                    atomicExch(args.sched, 0);
                    atomicExch(args.sched + 1, 0);
                }
            }
        }
        __syncwarp();
    } else if (warp >= C::MMA_WARP0) {
        // ======================================================== MMA issuer of group g
        const int g = warp - C::MMA_WARP0;
        const int b0 = C::B_GROUP + g * C::GROUP_BARS;
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_bf16_f32(FN_ROWS, FN_LKV / 2, false);  // B = K (K-major), 64 keys
            constexpr uint32_t IDESC_O = idesc_bf16_f32(FN_ROWS, FN_D, true);         // B = V (MN-major)
            const uint32_t tS = tmem_base + static_cast<uint32_t>(g * 256), tO = tS + 128u;
            // S half n (keys 64n..64n+63) += ln_q[:, 64kt..] K[64n.., 64kt..]^T, with
            // bf16(ln_q) in TMEM columns tO .. tO + 63 (8 columns per K step of 16)
            auto mma_s = [&](int n, int kt) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    mma_bf16_ts(tS + static_cast<uint32_t>(n * 64), tO + static_cast<uint32_t>(kt * 32 + j * 8),
                                smem_desc_sw128(sK + kt * FN_HALF_BYTES + n * (FN_HALF_BYTES / 2) + j * 32, 16, 1024),
                                IDESC_S, (kt | j) != 0 ? 1u : 0u);
            };
            bool ok = true;
            int kv_seen = -1;
            for (int it = g, k = 0; ok; it += NG, ++k) {
                const uint32_t ph = static_cast<uint32_t>(k) & 1u;
                // ln_q columns 0-63 written (or the group's end record seen)
                if (!(ok = mbar_wait(guard, bar(b0 + G_AREADY), ph, FN_SITE_AREADY, it))) break;
                const int kv = tile_rec[it % C::NQ].kv, last = tile_rec[it % C::NQ].last;
                if (tile_rec[it % C::NQ].b < 0) break;
                if (kv != kv_seen) {  // this tile's batch has its own K and V
                    if (!(ok = mbar_wait(guard, bar(C::B_KV), static_cast<uint32_t>(kv) & 1u, FN_SITE_KV, it))) break;
                    kv_seen = kv;
                }
                tc_fence_after();
                mma_s(0, 0);
                mma_s(1, 0);
                if (!(ok = mbar_wait(guard, bar(b0 + G_AREADY + 1), ph, FN_SITE_AREADY, it))) break;
                tc_fence_after();
                mma_s(0, 1);
                mma_commit(bar(b0 + G_SFULL));      // keys 0-63 done
                mma_s(1, 1);
                mma_commit(bar(b0 + G_SFULL + 1));  // keys 64-127 done
                // O = P V overwrites the columns that held bf16(ln_q): every S MMA is
                // complete first.  P's keys 64kt..64kt+63 are bf16 pairs in TMEM
                // columns tS + 64kt .. tS + 64kt + 31; keys 0-63 first.
                if (!(ok = mbar_wait(guard, bar(b0 + G_SFULL + 1), ph, FN_SITE_SFULL, it))) break;
                for (int kt = 0; kt < 2; ++kt) {
                    if (!(ok = mbar_wait(guard, bar(b0 + G_PREADY + kt), ph, FN_SITE_PREADY, it))) break;
                    tc_fence_after();
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        mma_bf16_ts(tO, tS + static_cast<uint32_t>(kt * 64 + j * 8),
                                    smem_desc_sw128(sV + kt * FN_HALF_BYTES + j * 2048, FN_HALF_BYTES / 2, 1024),
                                    IDESC_O, (kt | j) != 0 ? 1u : 0u);
                }
                if (!ok) break;
                mma_commit(bar(b0 + G_OFULL));
                if (last) mma_commit(bar(C::B_KVFREE));  // this group is done with this K and V
            }
            mma_commit(bar(b0 + G_MMA_DONE));
            fn_drain(bar(b0 + G_MMA_DONE), 0, args.timeout_ns);
        }
        __syncwarp();
    } else {
        // ======================================================== compute group g (warps 8g..8g+7)
        // Warp 8g + 4hf + q4 takes rows 32q4 .. 32q4 + 31 (its TMEM lane quarter)
        // and the 64 columns of half hf: one half row per thread.
        const int g = warp >> 3, gw = warp & 7, q4 = gw & 3, hf = gw >> 2;
        const int r = q4 * 32 + lane;  // tile row == TMEM lane
        const int b0 = C::B_GROUP + g * C::GROUP_BARS;
        const int pidx = rank * 2 + hf;  // this thread's partial in the exchanges
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q4 * 32) << 16) + static_cast<uint32_t>(g * 256);
        const uint32_t tS = t_lane, tO = t_lane + 128u;
        for (int it = g, k = 0;; it += NG, ++k) {
            const int qb = it % C::NQ;
            const uint32_t qph = static_cast<uint32_t>(it / C::NQ) & 1u;  // q buffer use count parity
            const uint32_t gph = static_cast<uint32_t>(k) & 1u;            // this group's tile count parity
            const int slot = it % C::NSLOT;
            const uint32_t xph = static_cast<uint32_t>(it / C::NSLOT) & 1u;
            const uint32_t sq = sQ + static_cast<uint32_t>(qb * FN_TILE_BYTES);
            bool ok = mbar_wait(guard, bar(C::B_QFULL + qb), qph, FN_SITE_QFULL, it);
            if (!__all_sync(0xffffffffu, ok)) break;
            const int tb = tile_rec[qb].b;
            if (tb < 0) {
                // No more tiles for this group; the MMA warp reads the same record.
                if (hf == 0) mbar_arrive(bar(b0 + G_AREADY));
                break;
            }
            const int m0 = tile_rec[qb].m0, qlen = tile_rec[qb].qlen;
            const int64_t qrow0 = static_cast<int64_t>(tb) * args.Lq;  // the batch's first row in Q / Out
            if (m0 + r >= qlen) {
                // A row past q_len: zero it once, so that every later step gives
                // exactly 0 for it, whatever the caller's buffer holds there.
#pragma unroll
                for (int c = 0; c < 8; ++c) st_shared_v4(fn_chunk(sq, r, hf * 8 + c), 0u, 0u, 0u, 0u);
            }

            // ---- LayerNorm: partial (mean, M2) over this thread's 64 columns, the
            //      sums shifted by the half row's first value, in packed fp32 pairs.
            float mean_c, m2_c;
            {
                const float sh = bf16lo(ld_shared_v4(fn_chunk(sq, r, hf * 8)).x);
                const uint64_t nsh = f2_splat(-sh);
                uint64_t s1a = 0, s1b = 0, s2a = 0, s2b = 0;  // (0.0f, 0.0f)
#pragma unroll
                for (int c = 0; c < 8; c += 2) {
                    const uint4 w0 = ld_shared_v4(fn_chunk(sq, r, hf * 8 + c));
                    const uint4 w1 = ld_shared_v4(fn_chunk(sq, r, hf * 8 + c + 1));
                    const uint32_t ww[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        const uint64_t d0 = f2_add(bf16x2_to_f2(ww[e]), nsh);
                        const uint64_t d1 = f2_add(bf16x2_to_f2(ww[e + 1]), nsh);
                        s1a = f2_add(s1a, d0);
                        s2a = f2_fma(d0, d0, s2a);
                        s1b = f2_add(s1b, d1);
                        s2b = f2_fma(d1, d1, s2b);
                    }
                }
                const float a1 = f2_hsum(f2_add(s1a, s1b)), a2 = f2_hsum(f2_add(s2a, s2b));
                mean_c = sh + a1 * (1.0f / 64.0f);
                m2_c = fmaxf(fmaf(-a1, a1 * (1.0f / 64.0f), a2), 0.0f);
            }
            {
                // push to partial [pidx] of every CTA of the cluster, wait for all 2H
                const uint32_t xb = bar(C::B_X1 + slot);
                const uint32_t dst =
                    sR1 + static_cast<uint32_t>(((slot * 2 * C::MAXH + pidx) * FN_ROWS + r) * 8);
                for (int p = 0; p < H; ++p) st_async_f32x2(mapa_shared(dst, p), mean_c, m2_c, mapa_shared(xb, p));
                ok = mbar_wait<true>(guard, xb, xph, FN_SITE_X1, it);
                if (!__all_sync(0xffffffffu, ok)) break;
                if (gw == 0 && lane == 0) mbar_arrive_expect_tx(xb, xbytes);  // for tile it + NSLOT
            }
            if (it >= NG && lane == 0) {
                // The output stores of this group's previous tile have read its q
                // buffer by now: the producer may refill it.
                bulk_wait_read<0>();
                mbar_arrive(bar(C::B_QEMPTY + (it - NG) % C::NQ));
            }
            // Chan et al. merge of the 2H partials (64 values each); all loads
            // issued before the first use.
            float2 pv[2 * C::MAXH];
            {
                const uint32_t rb = sR1 + static_cast<uint32_t>((slot * 2 * C::MAXH * FN_ROWS + r) * 8);
#pragma unroll
                for (int p = 0; p < 2 * C::MAXH; ++p)
                    pv[p] = p < 2 * H ? ld_shared_f32x2(rb + static_cast<uint32_t>(p * FN_ROWS * 8)) : make_float2(0.f, 0.f);
            }
            float msum = 0.0f;
#pragma unroll
            for (int p = 0; p < 2 * C::MAXH; ++p) msum += pv[p].x;
            const float mean = msum / static_cast<float>(2 * H);
            float m2 = 0.0f;
#pragma unroll
            for (int p = 0; p < 2 * C::MAXH; ++p) {
                const float dm = pv[p].x - mean;
                if (p < 2 * H) m2 += fmaf(64.0f * dm, dm, pv[p].y);
            }
            const float rstd1 = rsqrtf(fmaf(m2, args.inv_hd, args.eps1));
            // ln_q = (q - mean) rstd1 = q rstd1 - mean rstd1, in packed pairs
            const uint64_t rs = f2_splat(rstd1), nmr = f2_splat(-mean * rstd1);

            // ---- bf16(ln_q) of this half as bf16 pairs into TMEM columns
            //      tO + 32hf .. tO + 32hf + 31 (the first MMA's A operand): once the
            //      four warps of the half have written, that half of the
            //      contraction of S may run.
            {
                uint4 w[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) w[k] = ld_shared_v4(fn_chunk(sq, r, hf * 8 + k));
                uint32_t pk[32];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t ww[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) pk[k * 4 + e] = f2_to_bf16x2(f2_fma(bf16x2_to_f2(ww[e]), rs, nmr));
                }
                tmem_st32(tO + static_cast<uint32_t>(hf * 32), pk);
                tmem_st_wait();
                tc_fence_before();  // also orders this thread's reads of the last tile's S and O
                mbar_arrive(bar(b0 + G_AREADY + hf));
            }

            // ---- P = bf16(act(S)) for keys 64hf .. 64hf + 63 as bf16 pairs into the
            //      first 32 of S's TMEM columns for those keys (read just before, by
            //      this thread): the second MMA's A operand for that half.
            ok = mbar_wait(guard, bar(b0 + G_SFULL + hf), gph, FN_SITE_SFULL, it);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            {
                const uint32_t ts = tS + static_cast<uint32_t>(hf * 64);
                if (args.act == 1)
                    fn_act_half<1>(ts, ts);
                else if (args.act == 2)
                    fn_act_half<2>(ts, ts);
                else
                    fn_act_half<0>(ts, ts);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(b0 + G_PREADY + hf));
            }

            // ---- o = P V + ln_q (residual 1) for this half, written back over P V in
            //      TMEM, and its RMSNorm over all heads (second exchange);
            //      out = o rstd2 + q
            ok = mbar_wait(guard, bar(b0 + G_OFULL), gph, FN_SITE_OFULL, it);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            float ss;
            {
                uint64_t q0 = 0, q1 = 0;
#pragma unroll 1
                for (int seg = 0; seg < 2; ++seg) {
                    const uint32_t to = tO + static_cast<uint32_t>(hf * 64 + seg * 32);
                    uint32_t v[32];
                    tmem_ld32(to, v);
                    uint4 w[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) w[k] = ld_shared_v4(fn_chunk(sq, r, hf * 8 + seg * 4 + k));
                    tmem_ld_wait(v);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t ww[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int i = k * 8 + 2 * e;
                            const uint64_t o = f2_add(f2_pack(v[i], v[i + 1]), f2_fma(bf16x2_to_f2(ww[e]), rs, nmr));
                            if (e & 1)
                                q1 = f2_fma(o, o, q1);
                            else
                                q0 = f2_fma(o, o, q0);
                            float o0, o1;
                            f2_unpack(o, o0, o1);
                            v[i] = __float_as_uint(o0);
                            v[i + 1] = __float_as_uint(o1);
                        }
                    }
                    tmem_st32(to, v);
                }
                ss = f2_hsum(f2_add(q0, q1));
                tmem_st_wait();
            }
            {
                const uint32_t xb = bar(C::B_X2 + slot);
                const uint32_t dst =
                    sR2 + static_cast<uint32_t>(((slot * 2 * C::MAXH + pidx) * FN_ROWS + r) * 8);
                for (int p = 0; p < H; ++p) st_async_f32x2(mapa_shared(dst, p), ss, 0.0f, mapa_shared(xb, p));
                ok = mbar_wait<true>(guard, xb, xph, FN_SITE_X2, it);
                if (!__all_sync(0xffffffffu, ok)) break;
                if (gw == 0 && lane == 0) mbar_arrive_expect_tx(xb, xbytes);  // for tile it + NSLOT
            }
            float tot = 0.0f;
            {
                const uint32_t rb = sR2 + static_cast<uint32_t>((slot * 2 * C::MAXH * FN_ROWS + r) * 8);
                float pt[2 * C::MAXH];
#pragma unroll
                for (int p = 0; p < 2 * C::MAXH; ++p)
                    pt[p] = p < 2 * H ? ld_shared_f32(rb + static_cast<uint32_t>(p * FN_ROWS * 8)) : 0.0f;
#pragma unroll
                for (int p = 0; p < 2 * C::MAXH; ++p) tot += pt[p];
            }
            const float rstd2 = rsqrtf(fmaf(tot, args.inv_hd, args.eps2));
            {
                const uint64_t rr = f2_splat(rstd2);
#pragma unroll 1
                for (int seg = 0; seg < 2; ++seg) {
                    uint32_t v[32];
                    tmem_ld32(tO + static_cast<uint32_t>(hf * 64 + seg * 32), v);
                    uint4 w[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) w[k] = ld_shared_v4(fn_chunk(sq, r, hf * 8 + seg * 4 + k));
                    tmem_ld_wait(v);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t ww[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
                        uint32_t pk[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            pk[e] = f2_to_bf16x2(f2_fma(f2_pack(v[k * 8 + 2 * e], v[k * 8 + 2 * e + 1]), rr,
                                                        bf16x2_to_f2(ww[e])));
                        // q is overwritten in place by out
                        st_shared_v4(fn_chunk(sq, r, hf * 8 + seg * 4 + k), pk[0], pk[1], pk[2], pk[3]);
                    }
                }
            }
            fence_proxy_async_smem();  // the TMA store reads the staged rows
            __syncwarp();
            if (lane == 0) {
                // This warp's 32 rows of its 64-column box; none past the batch's
                // last 32-row group that holds a valid row.
                if (m0 + q4 * 32 < qlen)
                    tma_store_2d(&tmO, sq + static_cast<uint32_t>(hf * FN_HALF_BYTES + q4 * 32 * 128),
                                 col0 + hf * 64, static_cast<int32_t>(qrow0 + m0 + q4 * 32));
                bulk_commit();
            }
            __syncwarp();
        }
        if (lane == 0) bulk_wait_read<0>();  // shared memory outlives the stores' reads
        __syncwarp();
    }

    // ---- teardown: no CTA leaves while a peer may still write into its shared memory
    tc_fence_before();
    __syncthreads();
    cluster_arrive_release();
    cluster_wait_acquire();
    if (warp == C::PRODUCER_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// Scheduler words of the persistent grid, one pair per (device, stream): zero
// when the module loads, and zeroed again by the last cluster of every launch,
// so launches on one stream (which run one after the other) reuse them.
constexpr int kFnMaxSlots = 64;
__device__ int32_t g_fn_sched[kFnMaxSlots][2];

struct FnSlot {
    int device;
    cudaStream_t stream;
};
std::mutex g_fn_mu;
FnSlot g_fn_slots[kFnMaxSlots];
int g_fn_nslots = 0;

cudaError_t fn_sched_words(int device, cudaStream_t stream, int32_t** out) {
    std::lock_guard<std::mutex> lock(g_fn_mu);
    int idx = -1;
    for (int i = 0; i < g_fn_nslots && idx < 0; ++i)
        if (g_fn_slots[i].device == device && g_fn_slots[i].stream == stream) idx = i;
    if (idx < 0) {
        if (g_fn_nslots == kFnMaxSlots) return cudaErrorLaunchOutOfResources;  // too many streams
        idx = g_fn_nslots++;
        g_fn_slots[idx] = FnSlot{device, stream};
    }
    void* base = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&base, g_fn_sched);
    if (e != cudaSuccess) return e;
    *out = static_cast<int32_t*>(base) + 2 * idx;
    return cudaSuccess;
}

constexpr int kFnMaxDevices = 64;

template <int NG>
cudaError_t launch_fn(const CUtensorMap* m, FnArgs args, bool overlap, cudaStream_t stream) {
    using C = FnCfg<NG>;
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    if (device < 0 || device >= kFnMaxDevices) return cudaErrorInvalidDevice;
    static bool attr_set[kFnMaxDevices] = {};
    static int max_clusters[kFnMaxDevices][FnCfg<NG>::MAXH + 1] = {};
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(args.H);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int maxc = 0;
    {
        // Per-device set-up, once, under the launcher's lock.
        std::lock_guard<std::mutex> lock(g_fn_mu);
        if (!attr_set[device]) {
            e = cudaFuncSetAttribute(nf_flashnorm_fwd_kernel<NG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     C::SMEM_BYTES);
            if (e != cudaSuccess) return e;
            attr_set[device] = true;
        }
        int& cached = max_clusters[device][args.H];
        if (cached == 0) {
            // A persistent grid: as many clusters as can be resident at once.
            cfg.gridDim = dim3(static_cast<unsigned>(args.H));
            e = cudaOccupancyMaxActiveClusters(&cached, nf_flashnorm_fwd_kernel<NG>, &cfg);
            if (e != cudaSuccess) return e;
            if (cached <= 0) return cudaErrorInvalidConfiguration;
        }
        maxc = cached;
    }
    if ((e = fn_sched_words(device, stream, &args.sched)) != cudaSuccess) return e;
    const int clusters = args.B < maxc ? args.B : maxc;
    cfg.gridDim = dim3(static_cast<unsigned>(clusters * args.H));
    if (overlap) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, nf_flashnorm_fwd_kernel<NG>, m[0], m[1], m[2], m[3], args);
}

}  // namespace

cudaError_t launch_flashnorm_fwd(const void* tmaps, const FlashNormLaunch& a, bool overlap, cudaStream_t stream) {
    const CUtensorMap* m = static_cast<const CUtensorMap*>(tmaps);
    if (a.B <= 0) return cudaSuccess;
    FnArgs args;
    args.B = a.B;
    args.Lq = a.Lq;
    args.H = a.H;
    args.act = a.act;
    args.eps1 = a.eps1;
    args.eps2 = a.eps2;
    args.inv_hd = 1.0f / static_cast<float>(a.H * FN_D);
    args.q_len = a.q_len;
    args.sched = nullptr;
    args.status = a.status;
    args.timeout_ns = a.timeout_ns;
    // Two compute groups' exchange slots fit shared memory up to 4 heads per cluster.
    return a.H <= FnCfg<2>::MAXH ? launch_fn<2>(m, args, overlap, stream) : launch_fn<1>(m, args, overlap, stream);
}

}  // namespace nf
