/*
 * nf.h -- C ABI of the normalization-fused bf16 GEMM library (libnf.so).
 *
 * The library computes Y = X * W (X: M x K, W: K x N, bf16 in, fp32
 * accumulation, bf16 out) with a row-wise normalization fused into the GEMM,
 * as described in "Towards Free Normalization: Fusing Normalization into GEMM
 * and Attention Kernels" (PyTorch blog):
 *   - §2 "Lazy Pre-Norm":  Y = RMSNorm(X) * W, no affine;
 *   - §3 "Multi-CTA Norm": Y = LayerNorm(X * W) or RMSNorm(X * W), optional
 *     gamma / beta, the row spread over several CTAs that exchange partial
 *     row statistics (through DSMEM in a thread-block cluster, or through L2);
 * plus the unfused pair of the blog's §1 baseline (a plain GEMM and a
 * standalone row-norm kernel).
 *
 * Common rules for every compute entry point:
 *   Layout     All matrices are dense row-major bf16 (IEEE bfloat16 bit
 *              patterns), rows contiguous: X[i*K + k], W[k*N + j], Y[i*N + j].
 *              gamma / beta hold N bf16 values; mean / rstd outputs hold one
 *              fp32 per row.
 *   Memory     Every pointer is DEVICE memory of the current CUDA device,
 *              owned by the caller; the library keeps no reference after the
 *              call returns.  Y must not overlap any input.  Scratch memory
 *              owned by the library, one buffer of each kind per (device,
 *              stream): post-norm rows wider than 256 columns exchanged
 *              through L2 (the default, see nf_set_postnorm_exchange) use
 *              about 16 * M * ceil(N / 256) bytes, and Lazy Pre-Norm GEMMs
 *              with split row sums of squares (nf_set_prenorm_split) add
 *              8 * M bytes of their own to that buffer; GEMMs split over the
 *              contraction (nf_set_gemm_splitk) use SMs * 128 KB.  Rule: no
 *              compute call ever synchronizes the host with the device.  A
 *              call that finds its stream's buffer missing or too small
 *              allocates a large enough one in stream order (cudaMallocAsync
 *              and cudaMemsetAsync on `stream`); a buffer it replaces stays
 *              allocated for the life of the process, because graphs
 *              captured earlier may still use it.  nf_reserve_scratch sizes
 *              both buffers up front: after it, calls on that stream with
 *              shapes within its sizes allocate nothing.  While the stream
 *              is being captured, a call that would allocate fails with
 *              NF_ERR_INVALID_ARG; make it (or nf_reserve_scratch) before
 *              capture.  A captured graph keeps the buffers of the stream it
 *              was captured on, so its replays must not run concurrently
 *              with other work on that stream's buffers.
 *              nf_gemm_postnorm_ln_noalloc allocates nothing at any time.
 *   Alignment  X, W, Y (and in/out of nf_norm_rows) start on a 16-byte
 *              boundary; gamma / beta on 2 bytes; fp32 outputs on 4 bytes.
 *              K and N (cols for nf_norm_rows) are multiples of 8, so that
 *              every row starts on a 16-byte boundary.  Violations return
 *              NF_ERR_ALIGNMENT.
 *   Shapes     M == 0 is a no-op returning NF_OK (X and Y may then be NULL,
 *              as the base of an empty tensor can be).  N and K must be >= 1.
 *              M, N, K < 2^31.  Any M, N, K meeting these rules is handled,
 *              including ragged tails on every dimension.
 *   Streams    Work is enqueued on `stream` (NULL = the legacy default
 *              stream) and runs asynchronously; nothing synchronizes.  The
 *              first call on a device sets up per-device state (kernel
 *              attributes, the device status word); make it before any
 *              stream capture.  Later calls are capture-safe.
 *   Errors     A status code is returned; nothing is thrown across the ABI.
 *              Arguments are validated before anything is enqueued.  Launch
 *              failures return NF_ERR_CUDA (detail in nf_last_error()).
 *              Faults detected on the device (a pipeline wait that ran past
 *              its time limit) are recorded in the device status word, read
 *              with nf_get_device_status().
 *   Threads    Entry points are thread-safe.
 */
#ifndef NF_H
#define NF_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum nf_status {
    NF_OK = 0,
    NF_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad kind or eps */
    NF_ERR_ALIGNMENT = 2,         /* pointer or row pitch not aligned as required */
    NF_ERR_UNSUPPORTED_SHAPE = 3, /* a size beyond what the kernels support */
    NF_ERR_CUDA = 4,              /* a CUDA runtime / driver call failed */
    NF_ERR_TIMEOUT = 5,           /* a device-side wait exceeded its time limit */
    NF_ERR_NO_DEVICE = 6          /* no usable sm_103 device is current */
} nf_status;

/* Same type as cudaStream_t; declared here so that callers need no CUDA header. */
typedef struct CUstream_st* nf_stream;

#define NF_NORM_LN 0  /* LayerNorm: (x - mean) / sqrt(var + eps) * gamma + beta */
#define NF_NORM_RMS 1 /* RMSNorm:   x / sqrt(mean(x^2) + eps) * gamma          */

/* Post-norm N limit: one 256-column tile per CTA times a 16-CTA cluster. */
#define NF_POSTNORM_MAX_N 4096

/*
 * nf_gemm_plain -- Y = X * W.
 * The GEMM of the unfused baseline (blog §1: a GEMM kernel followed by a
 * separate normalization kernel).  fp32 accumulation, Y rounded to bf16
 * (round to nearest even).
 */
nf_status nf_gemm_plain(const void* X, const void* W, void* Y,
                        int64_t M, int64_t N, int64_t K, nf_stream stream);

/*
 * nf_gemm_plain_t -- Y = op(X) op(W) with one operand read transposed:
 * flags NF_TRANS_X: X is stored K x M row-major (Y = X^T W; needs M a
 * multiple of 8); NF_TRANS_W: W is stored N x K row-major (Y = X W^T).  Not
 * both.  Otherwise as nf_gemm_plain (Y is M x N row-major).  The unfused
 * baseline of the Lazy Pre-Norm backward uses both forms.
 */
#define NF_TRANS_X 1
#define NF_TRANS_W 4
nf_status nf_gemm_plain_t(const void* X, const void* W, void* Y, int64_t M,
                          int64_t N, int64_t K, int flags, nf_stream stream);

/*
 * nf_gemm_prenorm_rms -- Y = RMSNorm(X) * W, Lazy Pre-Norm (blog §2).
 * rstd_i = 1 / sqrt(sum_k X[i,k]^2 / K + eps) is accumulated from the same
 * shared-memory tiles of X the tensor cores consume, and applied to the fp32
 * accumulator in the epilogue: Y[i,:] = rstd_i * (X[i,:] * W), which equals
 * (rstd_i * X[i,:]) * W (the blog's §2 "Proof").  No gamma and no LayerNorm:
 * the blog's §2 limitations exclude both.  On tensor-bound shapes with
 * K >= 2048 and 2..32 column tiles of 256 a row, the tiles of a row share the
 * sums of squares
 * (nf_set_prenorm_split) through the stream's exchange scratch ("Memory").
 * rstd_out: optional (may be NULL), M fp32 values.
 * eps: finite and >= 0, else NF_ERR_INVALID_ARG.
 */
nf_status nf_gemm_prenorm_rms(const void* X, const void* W, void* Y,
                              int64_t M, int64_t N, int64_t K, float eps,
                              float* rstd_out, nf_stream stream);

/*
 * nf_gemm_postnorm_ln_res / nf_gemm_postnorm_rms_res -- residual add before
 * the post-norm, in the same epilogue:
 *   H = X W + R                       (fp32 accumulator plus R)
 *   Y = LayerNorm(H) * gamma + beta   (RMS: RMSNorm(H) * gamma)
 * The pattern of a transformer block's residual stream: the CUDA book chapter
 * "Element-wise 与算子融合", §8.4 (residual add followed by RMSNorm in one
 * kernel, the updated residual written back for the next layer) and §8.5.1
 * (the residual add taken into a GEMM's epilogue); the norm over the GEMM
 * output as blog §3.
 * R: M x N bf16 row-major device memory, 16-byte aligned, read once by the
 * kernel that owns each row segment.  H: optional (NULL) M x N bf16, 16-byte
 * aligned: bf16(H), the updated residual; H may be R itself (each element of
 * R is read before the same thread overwrites it).  Y must not overlap X, W,
 * R or H.  The statistics (mean_out, rstd_out) are those of H.  Same shapes,
 * alignment rules, exchanges and errors as nf_gemm_postnorm_ln, except that
 * the 512-column cluster kernel is not used (rows of 257..512 columns take a
 * cluster of two 256-column CTAs).
 */
nf_status nf_gemm_postnorm_ln_res(const void* X, const void* W, const void* R,
                                  const void* gamma, const void* beta, void* Y,
                                  void* H, int64_t M, int64_t N, int64_t K,
                                  float eps, float* mean_out, float* rstd_out,
                                  nf_stream stream);
nf_status nf_gemm_postnorm_rms_res(const void* X, const void* W, const void* R,
                                   const void* gamma, void* Y, void* H,
                                   int64_t M, int64_t N, int64_t K, float eps,
                                   float* rstd_out, nf_stream stream);

/*
 * nf_flashnorm_attn_fwd -- FlashNormAttention forward (blog §4, the fused
 * GDPA pseudocode over a short K/V sequence): for each batch b and query
 * token t < q_len[b], with q = Q[b, t, :, :] (H heads x D):
 *   ln_q = LayerNorm(q) over all H*D values (eps1, biased variance, no affine)
 *   per head h:  p = act(ln_q[h] . K[b, :, h, :]^T)            (Lkv keys)
 *                o[h] = p . V[b, :, h, :] + ln_q[h]            (residual 1)
 *   Out[b, t] = RMSNorm(o) over all H*D values (eps2, no affine) + q
 *                                                              (residual 2)
 * The two matmuls run on tensor cores with bf16 operands: ln_q and p enter
 * them rounded to bf16 (fp32 accumulation); the residuals and norms are fp32.
 * act: NF_ACT_IDENTITY, NF_ACT_GELU_TANH (x/2 (1 + tanh(sqrt(2/pi)(x + 0.044715
 * x^3)))) or NF_ACT_SILU (x / (1 + e^-x)); the pages name the activation
 * elementwise without fixing it.
 * Q, Out: [B, Lq, H, D]; K, V: [B, Lkv, H, D]; bf16 row-major device memory,
 * 16-byte aligned.  q_len: device int32[B] (4-byte aligned) or NULL (Lq for
 * every batch); rows t >= q_len[b] of Out are left as they were, except those
 * inside the last 32-row group holding a valid row, which are written as 0.
 * Supported: D = Lkv = 128, 1 <= H <= 8 (a thread-block cluster of H CTAs
 * works on one batch at a time and exchanges the row statistics of both norms
 * through distributed shared memory), Lq a multiple of 128; else
 * NF_ERR_UNSUPPORTED_SHAPE.
 * Scheduling: a persistent grid of as many clusters as fit on the device takes
 * batches one at a time from a counter the library keeps per (device, stream)
 * in device memory (no allocation; zero again when a launch ends).  Calls on
 * one stream run one after the other; calls on different streams may overlap.
 * The counters serve at most 64 (device, stream) pairs per process: a call
 * from a 65th pair fails with NF_ERR_CUDA.
 * Graphs: a CUDA graph captured from stream S keeps S's counter.  Its
 * replays must not overlap one another, nor calls made on S (replay it on S,
 * or order the replays with events); overlapping launches would share the
 * counter and skip each other's batches.
 */
#define NF_ACT_IDENTITY 0
#define NF_ACT_GELU_TANH 1
#define NF_ACT_SILU 2
nf_status nf_flashnorm_attn_fwd(const void* Q, const void* K, const void* V,
                                const int32_t* q_len, void* Out, int64_t B,
                                int64_t Lq, int64_t Lkv, int64_t H, int64_t D,
                                int act, float eps1, float eps2,
                                nf_stream stream);

/*
 * nf_gemm_prenorm_rms_bwd -- backward of C = RMSNorm(A) * B (Lazy Pre-Norm,
 * no affine), from the rstd the forward saved (blog §2, limitation 3: the
 * backward rebuilds rmsnorm(A) from A and rstd).  With xhat = A * rstd_i:
 *   dA = rstd_i * (dXhat - xhat * mean_k(dXhat * xhat)),  dXhat = dC B^T
 *        (the RMS-backward epilogue on a GEMM that reads B transposed);
 *   dB = xhat^T dC (a GEMM over M whose A operand is read transposed).
 * xhat: optional M x K bf16 buffer (16-byte aligned), owned by the caller.
 *   Given together with dA, the dA kernel's epilogue, which reads A and rstd
 *   anyway, also writes xhat = bf16(A * rstd_i) into it, and dB is a plain
 *   GEMM over that buffer.  NULL (or dA NULL): dB rebuilds xhat from A in
 *   shared memory, scaling each contraction row by rstd before the MMA -- no
 *   extra memory, but the rescaling competes with the tensor cores for
 *   shared-memory bandwidth.  Both forms round xhat to bf16 the same way.
 * A: M x K, B: K x N, dC: M x N, dA: M x K, dB: K x N, all bf16 row-major
 * device memory; rstd: M fp32 (16-byte aligned for dB).  dA or dB may be
 * NULL (not computed).  Same alignment rules as the forward; dB needs M a
 * multiple of 8 and dA K <= NF_POSTNORM_MAX_N.  Two to three kernels are
 * enqueued on `stream` (dB with few output tiles is split over the
 * contraction, see nf_set_gemm_splitk).
 */
nf_status nf_gemm_prenorm_rms_bwd(const void* A, const void* B,
                                  const float* rstd, const void* dC, void* dA,
                                  void* dB, void* xhat, int64_t M, int64_t N,
                                  int64_t K, nf_stream stream);

/*
 * nf_gemm_postnorm_ln -- Y = LayerNorm(X * W) over each row of N, Multi-CTA
 * post-norm (blog §3): each CTA holding a tile of the row reduces the partial
 * statistics of its tile, the partials are exchanged, and every CTA
 * normalizes before its single store.  N <= 256: one CTA holds whole rows.
 * Wider rows: the exchange runs through L2 between the 256-column tiles of a
 * cooperative grid (default), or, as on the blog, through distributed shared
 * memory inside a thread-block cluster spanning the row
 * (nf_set_postnorm_exchange).
 * LayerNorm as torch.nn.LayerNorm: biased variance, eps inside the root.
 * gamma, beta: optional (NULL = 1 and 0), N bf16 values each.
 * mean_out, rstd_out: optional, M fp32 values (row mean, 1/sqrt(var + eps)).
 * N <= NF_POSTNORM_MAX_N, else NF_ERR_UNSUPPORTED_SHAPE.
 */
nf_status nf_gemm_postnorm_ln(const void* X, const void* W, const void* gamma,
                              const void* beta, void* Y, int64_t M, int64_t N,
                              int64_t K, float eps, float* mean_out,
                              float* rstd_out, nf_stream stream);

/*
 * nf_gemm_postnorm_ln_noalloc -- nf_gemm_postnorm_ln that allocates no
 * memory at any time, on any call.  The blog has no counterpart: this is a
 * deployment variant.  Same arguments, plan, kernels and results as
 * nf_gemm_postnorm_ln.  Where that plan exchanges row statistics through L2,
 * the scratch is a fixed device array inside the library (about 8.1 MiB per
 * device, cleared on the first call on each device) instead of the
 * per-stream buffer.  Limit of that array: ceil(M / 128) * ceil(N / 256)
 * <= 4096 exchange tiles (which implies M <= 2^19), else
 * NF_ERR_UNSUPPORTED_SHAPE (only for shapes that use the L2 exchange).
 * The first such call on a device looks the array up and clears it with a
 * synchronous memset; make it before any stream capture (during a capture
 * it fails with NF_ERR_INVALID_ARG).
 * Races: the array is one per device, shared by every stream and every
 * thread.  Two calls that may run on the device at the same time (on
 * different streams, or from graphs replayed concurrently) corrupt each
 * other's exchange; the caller serializes them (one stream, or events).
 * Calls ordered on one stream are safe.
 */
nf_status nf_gemm_postnorm_ln_noalloc(const void* X, const void* W,
                                      const void* gamma, const void* beta,
                                      void* Y, int64_t M, int64_t N, int64_t K,
                                      float eps, float* mean_out,
                                      float* rstd_out, nf_stream stream);

/*
 * nf_gemm_postnorm_rms -- Y = RMSNorm(X * W) * gamma over each row of N
 * (blog §3 with RMSNorm).  gamma optional (NULL = 1); rstd_out optional.
 * N <= NF_POSTNORM_MAX_N, else NF_ERR_UNSUPPORTED_SHAPE.
 */
nf_status nf_gemm_postnorm_rms(const void* X, const void* W, const void* gamma,
                               void* Y, int64_t M, int64_t N, int64_t K,
                               float eps, float* rstd_out, nf_stream stream);

/*
 * nf_norm_rows -- standalone LayerNorm / RMSNorm of each row of `in`
 * (rows x cols) into `out`: the normalization kernel of the unfused baseline
 * (blog §1).  kind is NF_NORM_LN or NF_NORM_RMS; beta is ignored for RMSNorm;
 * mean_out is not written for RMSNorm.  cols <= 16384, else
 * NF_ERR_UNSUPPORTED_SHAPE.  `in` and `out` must not overlap.
 */
nf_status nf_norm_rows(const void* in, void* out, const void* gamma,
                       const void* beta, int64_t rows, int64_t cols, int kind,
                       float eps, float* mean_out, float* rstd_out,
                       nf_stream stream);

/* nf_norm_rows_res -- the unfused residual-add norm (CUDA book chapter
 * "Element-wise 与算子融合" §8.4): H = in + R, out = norm(H) as nf_norm_rows,
 * H (optional, may be R itself) = bf16(H).  R and H: rows x cols bf16,
 * 16-byte aligned; R non-null when rows > 0. */
nf_status nf_norm_rows_res(const void* in, const void* R, void* out, void* H,
                           const void* gamma, const void* beta, int64_t rows,
                           int64_t cols, int kind, float eps, float* mean_out,
                           float* rstd_out, nf_stream stream);

/*
 * nf_gemm_postnorm_ln_bwd -- dZ = LayerNorm backward of dY = A * B, the
 * norm's backward fused into the epilogue of the GEMM that produces its
 * incoming gradient (blog §3 "What about backward? Fusion regrouping": the
 * norm sits between two linears; the forward fuses it into the first one's
 * epilogue, the backward into the epilogue of the second one's input-gradient
 * GEMM dY = dOut * W2^T, so both directions are epilogue fusions with the
 * same multi-CTA structure).  With g = dY * gamma and xhat = (Z - mean_i) *
 * rstd_i:  dZ = rstd_i * (g - mean_j g - xhat * mean_j(g * xhat)); dY is
 * never rounded or stored.
 * A: M x K, B: K x N (row-major, e.g. W2^T), Z: M x N bf16 (the forward's
 * norm input, 16-byte aligned), gamma: optional N bf16, mean / rstd: the
 * forward's saved row statistics (M fp32 each, required), dZ: M x N bf16.
 * Same shape, alignment and N <= NF_POSTNORM_MAX_N rules as the forward;
 * rows wider than 256 columns exchange their two partial sums like the
 * forward (L2 for K >= 512, else a cluster).  dgamma / dbeta (column sums
 * over M) are not computed.
 */
nf_status nf_gemm_postnorm_ln_bwd(const void* A, const void* B, const void* Z,
                                  const void* gamma, const float* mean,
                                  const float* rstd, void* dZ, int64_t M,
                                  int64_t N, int64_t K, nf_stream stream);

/*
 * nf_gemm_postnorm_rms_bwd -- the same for RMSNorm: xhat = Z * rstd_i,
 * dZ = rstd_i * (g - xhat * mean_j(g * xhat)).
 */
nf_status nf_gemm_postnorm_rms_bwd(const void* A, const void* B, const void* Z,
                                   const void* gamma, const float* rstd,
                                   void* dZ, int64_t M, int64_t N, int64_t K,
                                   nf_stream stream);

/*
 * nf_norm_rows_bwd -- backward of LayerNorm / RMSNorm over each row, from
 * the statistics the forward pass saved (blog §3 "What about backward?"):
 *   g = dY * gamma;  xhat = (Z - mean_i) * rstd_i (LN) or Z * rstd_i (RMS);
 *   LN:  dZ = rstd_i * (g - mean_j g - xhat * mean_j(g * xhat))
 *   RMS: dZ = rstd_i * (g - xhat * mean_j(g * xhat)).
 * With Z's own statistics this is the gradient of sum(dY * norm(Z)) with
 * respect to Z (dgamma / dbeta are not computed).  The unfused kernel the
 * fused backward (nf_gemm_postnorm_ln_bwd / _rms_bwd) is compared with.
 * dY, Z, dZ: rows x cols bf16, 16-byte aligned, cols a multiple of 8 and
 * <= 16384; gamma: optional, cols bf16, 16-byte aligned; mean (LN only,
 * required) and rstd (required): rows fp32, device memory.  dZ must not
 * overlap dY or Z.  rows == 0 is a no-op.
 */
nf_status nf_norm_rows_bwd(const void* dY, const void* Z, const void* gamma,
                           const float* mean, const float* rstd, void* dZ,
                           int64_t rows, int64_t cols, int kind,
                           nf_stream stream);

/* ---------------------------------------------------------------------
 * Diagnostics and configuration (no counterpart in the blog).
 * ------------------------------------------------------------------- */

/* Synchronizes the current device, then returns the status recorded by the
 * kernels since the last clear: NF_OK, or NF_ERR_TIMEOUT when a pipeline wait
 * gave up (NF_ERR_ALIGNMENT: dynamic shared memory not 1 KB aligned;
 * NF_ERR_INVALID_ARG: a GEMM kernel found itself in a cluster of a size other
 * than the one its plan launches it with, as when a tool re-issues the launch
 * without its attributes, and returned before any work).  `detail` (may be
 * NULL) receives 4 words: code, wait site, block index, tile index of the
 * first failure. */
nf_status nf_get_device_status(uint32_t* detail);

/* Synchronizes the current device, resets its status word to NF_OK and
 * zeroes the library's post-norm exchange scratch on it. */
nf_status nf_clear_device_status(void);

/* Time limit for every device-side pipeline wait, in nanoseconds (default
 * 2e9).  After it a kernel records NF_ERR_TIMEOUT, stops its work, releases
 * its tensor memory and returns; the CUDA context stays usable. */
nf_status nf_set_wait_timeout_ns(uint64_t ns);

/* Programmatic dependent launch (default on): each kernel may be scheduled
 * while the kernel before it on the stream finishes; it performs its set-up
 * (barriers, tensor memory) and then waits for that kernel to complete before
 * touching global memory, so results are unchanged.  0 turns it off. */
nf_status nf_set_launch_overlap(int enable);

/* Column tile per CTA when post-norm rows go to a cluster: 0 (default)
 * automatic, 512 (a cluster of ceil(N/512) <= 8 CTAs; a row of N <= 512 then
 * needs no cluster) or 256 (clusters of up to 16 CTAs).  Applies to later
 * post-norm calls that use the cluster exchange. */
nf_status nf_set_postnorm_tile_n(int tile_n);

/* Column tile per CTA of plain and Lazy Pre-Norm GEMMs (nf_gemm_plain,
 * nf_gemm_prenorm_rms): 0 (default) automatic -- the
 * smallest of 64 / 128 / 256 that covers N, else 256 -- or 64, 128, 256
 * forced.  Applies to later calls. */
nf_status nf_set_gemm_tile_n(int tile_n);

/* CTA pairs for plain and Lazy Pre-Norm GEMMs: two CTAs of a cluster along M
 * compute one 256 x 256 output tile with tcgen05 cta_group::2 MMAs, each
 * loading its own 128 rows of X and half of W's 256 columns; post-norm rows
 * exchanged through L2 take them too.  mode 0 (default): plain GEMMs of
 * tensor-bound 256-column tiles (except those with so few tiles that each is
 * split over the contraction), pre-norm GEMMs whose row sums of squares are
 * split (nf_set_prenorm_split) and post-norm GEMMs with the L2 exchange and
 * K >= 2048; 1: never; 2: whenever the tile has 256 columns and M > 128.
 * Applies to later calls. */
nf_status nf_set_gemm_pair(int mode);

/* Lazy Pre-Norm row sums of squares, split.  Every CTA of the blog's §2
 * kernel sums the squares of all of its tile's rows from the shared-memory
 * stages of X, so the n_tiles = ceil(N / 256) tiles of a row each repeat the
 * same sums.  Split, tile n of a row tile sums only rows n R .. n R + R - 1
 * (R = ceil(128 / n_tiles)) over the whole of K, and the row tile's tiles
 * gather the 128 sums through L2 (scratch memory, see "Memory" above) before
 * their epilogues scale the accumulators; the tiles then run as a persistent
 * cooperative grid, like the post-norm L2 exchange.  The sums are the same up
 * to fp32 summation order.  mode 0 (default): when the 256-column tiles are
 * tensor-bound (their shared-memory reads would slow the MMA), K >= 2048 and
 * a row has 2..32 of them; 1: never; 2: whenever a row has 2..32 tiles of 256
 * columns.
 * Applies to later calls. */
nf_status nf_set_prenorm_split(int mode);

/* How post-norm rows wider than 256 columns exchange partial statistics:
 * 0 (default) automatic -- one 512-column CTA per row while N <= 512, else
 * NF_XCH_GLOBAL when K >= 512, else NF_XCH_CLUSTER; NF_XCH_CLUSTER: a
 * thread-block cluster spans the row and the partials go through
 * distributed shared memory (blog §3); NF_XCH_GLOBAL: 256-column tiles of a
 * persistent cooperative grid using every SM, partials through L2 (scratch
 * memory, see "Memory" above).  Applies to later calls. */
#define NF_XCH_CLUSTER 1
#define NF_XCH_GLOBAL 2
nf_status nf_set_postnorm_exchange(int mode);

/* Split-K of plain GEMMs (nf_gemm_plain, nf_gemm_plain_t and the weight
 * gradient of nf_gemm_prenorm_rms_bwd).  mode 0 (default): when the output
 * has at most half as many 128-row tiles as the device has SMs, the
 * contraction of every tile is cut into slices of >= 8 K-tiles, one
 * (tile, slice) per SM; when a tensor-bound GEMM's last, partial wave holds
 * at most half as many tiles as SMs, only that wave's tiles are split.  Each
 * split unit writes an fp32 partial tile into a per-stream workspace (SMs x
 * 128 KB, set up by nf_reserve_scratch or by the first such call on a
 * stream, which must not be inside a graph capture), and a second kernel
 * adds the slices in a fixed order and rounds to bf16, so results are
 * reproducible.  mode 1: never split.  Applies to later calls. */
nf_status nf_set_gemm_splitk(int mode);

/* Scratch set-up for `stream` (see "Memory" above): makes the stream's
 * exchange buffer large enough for post-norm calls (forward and backward) of
 * up to max_rows x max_cols and Lazy Pre-Norm calls of up to max_rows rows
 * (any N), and sets up its split-K workspace,
 * both in stream order without synchronizing the host.  Afterwards, calls on
 * the stream within those sizes allocate nothing and may be captured.
 * max_cols <= NF_POSTNORM_MAX_N.  Refused (NF_ERR_INVALID_ARG) while the
 * stream is being captured. */
nf_status nf_reserve_scratch(int64_t max_rows, int64_t max_cols, nf_stream stream);

/* Self-test of the time limit: launches one CTA that waits on a barrier no
 * thread ever arrives on, with limit `timeout_ns` (1e3..1e10).  After the
 * stream completes, nf_get_device_status() reports NF_ERR_TIMEOUT. */
nf_status nf_selftest_wait_timeout(uint64_t timeout_ns, nf_stream stream);

/* English text for a status code (static storage). */
const char* nf_status_string(nf_status status);

/* Detail of the last failing call on this thread ("" if none). */
const char* nf_last_error(void);

/* Launch plan the library would use; pure host function, no GPU needed.
 * op: 0 plain, 1 pre-norm RMS, 2 post-norm LN, 3 post-norm RMS,
 * 4 LN backward, 5 RMS backward.
 * sm_count: SMs of the device; the grid assumes every SM can hold one CTA
 * (for clusters, the library asks the driver for the real co-residency). */
typedef struct nf_plan {
    int32_t tile_m, tile_n, tile_k; /* CTA tile                            */
    int32_t stages;                 /* shared-memory ring depth            */
    int32_t cluster;                /* CTAs per cluster: along N for a row
                                       cluster, 2 along M for a CTA pair    */
    int32_t grid;                   /* persistent CTAs                      */
    int32_t threads;                /* threads per CTA                     */
    int32_t smem_bytes;             /* dynamic shared memory per CTA       */
    int32_t tmem_cols;              /* tensor-memory columns per CTA       */
    int32_t tiles;                  /* output tiles (M/tile_m x N/tile_n)  */
    int32_t exchange;               /* 0 none, NF_XCH_CLUSTER, NF_XCH_GLOBAL
                                       (pre-norm: the split row sums of
                                       squares gathered through L2)        */
    int32_t splitk;                 /* contraction slices (plain GEMM; 1 = none) */
    int32_t split_tiles;            /* tiles split over the contraction (the last ones) */
} nf_plan;
nf_status nf_plan_gemm(int op, int64_t M, int64_t N, int64_t K, int sm_count,
                       nf_plan* out);

/* ABI version of this header (bumped on any incompatible change). */
#define NF_ABI_VERSION 3
int nf_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* NF_H */
