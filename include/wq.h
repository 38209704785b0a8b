/*
 * wq.h -- C ABI of libwq, the W4A4 NVFP4 quantised projection for NVIDIA B300
 * (sm_103a).
 *
 * The operation (citations are page title + section):
 *   y = x W + b  computed as
 *   y = gA gW (Q4(xt_~O) . Q4(R'_~O)) + U Q + x_O W_O + b
 * where
 *   xt  = (x * inv_s) H             per-channel smoothing, then block-64 Walsh-Hadamard
 *                                   rotation (FoldQuantVLA, Key Contribution 2; QuantWAMs
 *                                   sec. 3.1 Eq. (1), Fig. 1(b));
 *   R'  = H diag(s) (W - P Q)       the inverse transform folded into the weight
 *                                   (FoldQuantVLA, Key Contribution 1, Proposition 1;
 *                                   QuantWAMs sec. 3.2: the Hadamard is fused into the weights);
 *   P Q                             the 16-bit low-rank protection branch (Q-WAM abstract,
 *                                   Action-Subspace Protection); P = bf16(L1 * inv_s),
 *                                   Q = bf16(L2), U = bf16(x P);
 *   O (Omega), x_O, W_O             the transformed channels kept in FP16 (QuantWAMs
 *                                   sec. 3.1, Eq. (3) Top-K mask; Fig. 1(d); sec. 4.2
 *                                   "Quantization configuration" exception path);
 *   Q4                              NVFP4: e2m1 codes, one unsigned e4m3 scale per 16
 *                                   consecutive K elements, one fp32 tensor scale
 *                                   (LatentQuant abstract; QuantWAMs sec. 4.2 "Backend":
 *                                   NVFP4 W4A4 kernels).  Activations use one fp32 scale per
 *                                   row, computed at run time (FoldQuantVLA, Key Contribution 2:
 *                                   dynamic per-token quantisation); weights one per tensor.
 *   NVFP4 rounding: g = amax / 2688; sc = e4m3_rn_satfinite((bmax / 6) / g);
 *   d = dec(sc) * g; code = e2m1_rn_satfinite(v / d) (0 when d == 0); each step one
 *   IEEE fp32 operation.
 *
 * Conventions for every entry point:
 *   - Device pointers must be 16-byte aligned.  "host" / "device" is stated per argument.
 *   - All calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream)
 *     unless stated otherwise.  Inputs are not modified.
 *   - Errors are returned as wq_status and never abort the process; wq_last_error()
 *     returns a thread-local message for the last failure.
 *   - NaN / Inf inputs are outside the contract.
 *   - Supported shapes: K % 64 == 0 and 64 <= K <= 16384; N % 16 == 0; 0 <= rank <= 64;
 *     0 <= n_outliers <= 64 (QuantWAMs sec. 4.2 keeps the top 2% of the input channels);
 *     M >= 0 (M == 0 is a no-op).  Anything else returns WQ_ERR_UNSUPPORTED.
 *   - Every launching entry point must be called with the handle's device current (the device
 *     that was current at wq_prepare_*); otherwise it returns WQ_ERR_INVALID.
 *   - A handle caches the tensor maps of the buffers it last saw; calls on one handle from
 *     several host threads are serialised by the handle and are safe.
 */
#ifndef WQ_H_
#define WQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define WQ_API __attribute__((visibility("default")))

typedef struct wq_weights *wq_weights_t;   /* opaque; owns library-allocated device memory */

typedef enum wq_status {
    WQ_OK = 0,
    WQ_ERR_INVALID = -1,       /* null pointer, negative size, unsorted Omega, bad enum  */
    WQ_ERR_UNSUPPORTED = -2,   /* shape or option outside the supported set               */
    WQ_ERR_CUDA = -3,          /* a CUDA runtime call failed (message in wq_last_error)   */
    WQ_ERR_OOM = -4,           /* device or host allocation failed                        */
    WQ_ERR_TIMEOUT = -5        /* a kernel gave up waiting on one of its barriers         */
} wq_status;

enum { WQ_MODE_W4A4 = 0, WQ_MODE_W8A8 = 1, WQ_MODE_W8A8_FP8 = 2, WQ_MODE_W4A8 = 3 };
enum { WQ_SCALE_LAYOUT_ROWMAJOR = 0, WQ_SCALE_LAYOUT_MMA = 1 };
/* Granularity of the activations' fp32 tensor scale g (4-bit layers):
 *   ROW     one g per row, from that row's amax at run time (FoldQuantVLA, Key Contribution 2:
 *           dynamic per-token quantisation; the default);
 *   TENSOR  one g for the whole [M, K] batch, from its amax at run time (two quantiser launches:
 *           the maximum, then the codes);
 *   STATIC  one calibrated g (wq_config.act_gscale) fixed at preparation; one pass, no amax.
 * g = amax / 2688 in the first two; the block scales and codes follow from g as in every mode. */
enum { WQ_ACT_SCALE_ROW = 0, WQ_ACT_SCALE_TENSOR = 1, WQ_ACT_SCALE_STATIC = 2 };
/* Order of the two activation transforms (4-bit layers with rotate = 1):
 *   SMOOTH_ROTATE  xt = (x diag(1/s)) H, weight R' = H diag(s) (W - P Q), P = bf16(diag(1/s) L1)
 *                  (FoldQuantVLA, Key Contribution 2: "channel scaling, block Hadamard"; default);
 *   ROTATE_SMOOTH  xt = (x H) diag(1/s), weight R' = diag(s) H (W - P Q), P = bf16(H diag(1/s) L1)
 *                  (QuantWAMs sec. 3.1 Eq. (1): A R S^-1).  L1, L2 are then the top-r factors of
 *                  diag(s) H W and s is taken in the rotated basis. */
enum { WQ_ORDER_SMOOTH_ROTATE = 0, WQ_ORDER_ROTATE_SMOOTH = 1 };

/* mode = WQ_MODE_W8A8 selects the selective 8-bit path (FoldQuantVLA, Key Contribution 3:
 * attention-output and FFN down projections kept at W8A8) in the same smoothed + rotated basis:
 * per-row activation scale a = amax / 127, per-output-column weight scale w = amax / 127,
 * q = round-half-even(v / scale) clamped to [-127, 127]; y = a[m] w[n] (sum_k qa qw) + b.
 * mode = WQ_MODE_W8A8_FP8 is the same 8-bit path in e4m3 (QuantWAMs sec. 4.2 "Backend": the
 * saliency-upgraded layers run FP8 W8A8 kernels): scales amax / 448, q = e4m3_rn_satfinite(v /
 * scale) with the quotient one IEEE fp32 division; one byte per value in HBM and tcgen05
 * kind::f8f6f4 MMAs.  rank and n_outliers must be 0 in both 8-bit modes.
 * mode = WQ_MODE_W4A8 is a 4-bit layer at an A8-protected step (QuantWAMs sec. 4.2 and sec. 5: one
 * of ten Fast-WAM action-denoising steps, 2/20 and 6/50 LingBot-VA steps keep 8-bit activations):
 * the same folded NVFP4 weights, low-rank branch and fp16 kept channels as WQ_MODE_W4A4 (same
 * options, rank and n_outliers allowed, act_scale WQ_ACT_SCALE_ROW), activations in e4m3 per token
 * (scale amax / 448 after the kept-channel split).  The tensor cores take both operands in bf16,
 * which holds every e4m3 value and every NVFP4 value dec(code) dec(scale) exactly (no tensor kind
 * multiplies e4m3 by e2m1 under NVFP4's e4m3-per-16 weight scales), so the handle stores the
 * weight values expanded to bf16 [N, K] next to the NVFP4 codes, and wq_linear_forward writes the
 * activation values as bf16 [M, K] (wq_workspace_bytes covers them).
 * project = 1 (Q-WAM abstract, Action-Subspace Protection: the 16-bit low-rank branch protects the
 * action subspace and the complementary weights AND activations are quantised): with the branch's
 * bf16 down-projection u = x P, the activation quantiser works on
 *     xt_c = xt - u Vt,   Vt[j][k] = bf16((H L1[:, j])[k] / ||L1[:, j]||^2)   (fp64, one rounding),
 * the complement of the span of L1 (the top-r left singular directions of diag(s) W) in the rotated
 * basis, one fp32 fma per rank term in the order j = 0 .. rank-1, before the kept-channel split.
 * The weights are unchanged: the complement R = W_s - L1 L2 has no component on the protected
 * directions (U_r^T R = 0 for L1 = U_r S_r), so xt_c R' = xt R' and y = xt_c R' + u Q + x_O W_O + b
 * equals the full activation's result up to the quantisation.  Needs rank > 0, WQ_MODE_W4A4, WQ_ACT_SCALE_ROW and WQ_ORDER_SMOOTH_ROTATE; the
 * quantiser then takes two launches (U, then both passes over the projected values). */
typedef struct wq_config {
    int K;            /* input features (reduction dimension)                              */
    int N;            /* output features                                                   */
    int rank;         /* low-rank branch rank r (0 disables the branch)                    */
    int n_outliers;   /* |Omega|, channels of the rotated basis kept in fp16 (0 disables)  */
    int rotate;       /* 1: block-64 Walsh-Hadamard rotation; 0: none                     */
    int mode;         /* WQ_MODE_W4A4 (wq_linear_forward) or WQ_MODE_W8A8 (..._w8a8)      */
    int act_scale;    /* WQ_ACT_SCALE_* (4-bit layers; W8A8 takes WQ_ACT_SCALE_ROW)        */
    float act_gscale; /* WQ_ACT_SCALE_STATIC: the calibrated g (> 0, finite); else ignored */
    int transform_order; /* WQ_ORDER_*: where the smoothing sits relative to the rotation  */
    int project;      /* 1: quantise the activation's complement of the protected subspace  */
                      /* (Q-WAM Action-Subspace Protection, below); 0: the full activation */
} wq_config;

/*
 * Fold and quantise one projection's weights (offline; FoldQuantVLA Key Contribution 1
 * "consistent folding"; Q-WAM ASP; QuantWAMs sec. 3.1 exception channels).
 *   cfg     host, shape and options.
 *   W       host fp32 [K, N] row-major (math convention y = x W).
 *   bias    host fp32 [N] or NULL.
 *   s       host fp32 [K] smoothing factors (> 0) or NULL for s = 1.
 *   L1, L2  host fp32 [K, r] and [r, N] (top-r factors of diag(s) W); NULL when r == 0.
 *   omega   host int32 [n_outliers], strictly ascending channel indices of the rotated
 *           basis, each < K; NULL when n_outliers == 0.
 *   stream  uploads are enqueued on it; the handle is usable by later work on any stream
 *           after the call returns (the call synchronises its uploads).
 *   out     receives the handle; free it with wq_free_weights().
 */
WQ_API wq_status wq_prepare_weights(const wq_config *cfg, const float *W, const float *bias,
                                    const float *s, const float *L1, const float *L2,
                                    const int32_t *omega, void *stream, wq_weights_t *out);

/* Copy the handle's configuration into *cfg (host). */
WQ_API wq_status wq_get_config(wq_weights_t h, wq_config *cfg);

/*
 * Row strides (in elements) of the 16-bit side operands that wq_quantize_activations writes
 * and wq_linear_forward_quantized reads: U is bf16 [M, *u_ld] and x_Omega fp16 [M, *xo_ld], where
 * each stride is the configured count (rank, n_outliers) rounded up to 16, 32 or 64 (0 when the
 * count is 0).  The columns beyond the count are written as zeros.  Host outputs; either may be NULL.
 */
WQ_API wq_status wq_side_strides(wq_weights_t h, int *u_ld, int *xo_ld);

/*
 * Bytes of device scratch that wq_linear_forward needs for M rows (the quantised
 * activations, their scales, per-row scales, U and x_Omega).  Returns 0 for a NULL handle.
 */
WQ_API size_t wq_workspace_bytes(wq_weights_t h, int M);

/*
 * The hot path: y = projection(x).
 *   x          device bf16 [M, K] row-major.
 *   y          device bf16 [M, N] row-major (written entirely; may not alias x).
 *   workspace  device scratch of at least wq_workspace_bytes(h, M) bytes, 256-byte aligned,
 *              owned by the caller; must not be used concurrently by another call.
 * Two kernels run on `stream`: the fused smooth + FWHT + NVFP4 activation quantiser and
 * the tcgen05 block-scaled FP4 GEMM with the fused epilogue (dequantisation, low-rank
 * branch, outlier slice, bias).  With the environment variable WQ_FUSED=1, a small batch
 * (see wq_forward_path) runs both in one thread-block-cluster kernel instead; the results
 * agree with the two-kernel path within the stated y tolerance (the row scales, codes and
 * scales are identical; fp32 partial sums may associate differently).
 */
WQ_API wq_status wq_linear_forward(wq_weights_t h, const void *x, int M, void *y,
                                   void *workspace, size_t workspace_bytes, void *stream);

#define WQ_PATH_TWO_KERNEL 0   /* quantiser kernel, then GEMM kernel */
#define WQ_PATH_FUSED 1        /* one cluster kernel (M <= 64, rank <= 32, K % 128 == 0) */
/*
 * Which path wq_linear_forward takes for M rows under the current environment (host query;
 * it may ask the CUDA runtime how many clusters fit on the device).  Returns a WQ_PATH_*
 * value, or WQ_ERR_INVALID for a NULL handle or M < 0.
 */
WQ_API int wq_forward_path(wq_weights_t h, int M);

#define WQ_QUANT_CLUSTER 0  /* a 16-row tile per cluster, K spread over its CTAs (few rows) */
#define WQ_QUANT_STREAM 1   /* persistent CTAs streaming row tiles (at least 2 x SMs of them) */
#define WQ_QUANT_RESIDENT 2 /* persistent CTAs keeping each row tile's transformed values in
                               registers: 4-bit layers, per-row scales, K <= 1536 (the default
                               for many rows there) */
/*
 * Which activation-quantiser schedule M rows take (host query).  Returns a WQ_QUANT_* value,
 * or WQ_ERR_INVALID for a NULL handle or M < 0.
 */
WQ_API int wq_quant_schedule(wq_weights_t h, int M);

#define WQ_GEMM_SINGLE 0   /* 128 x 128 tiles, one persistent CTA per SM */
#define WQ_GEMM_SPLITK 1   /* 128 x 128 tiles, K split over a thread-block cluster (few tiles) */
#define WQ_GEMM_WIDE 2     /* 256 x 256 tiles on CTA pairs, one accumulator (4-bit layers, many tiles) */
#define WQ_GEMM_WIDE_DB 3  /* 256 x 192 tiles on CTA pairs, two accumulators (4-bit layers, many tiles,
                              K <= 4096): the epilogue of one tile overlaps the next tile's MMAs */
/*
 * Which GEMM schedule the two-kernel path (and wq_linear_forward_quantized) uses for M rows
 * under the current environment (host query; it may ask the CUDA runtime how many clusters
 * fit).  Returns a WQ_GEMM_* value, or WQ_ERR_INVALID / WQ_ERR_CUDA.
 */
WQ_API int wq_gemm_schedule(wq_weights_t h, int M);

/*
 * Schedule knobs for tests and tuning (no counterpart on the pages; results never depend on them
 * beyond the stated tolerances).  Each knob starts from the environment variable of the same name,
 * read once at the library's first use, and afterwards changes only through this call.
 *   "WQ_FUSED" 0/1; "WQ_GEMM_SPLIT" 0 (auto) or 1..16; "WQ_GEMM_WIDE" -1 (auto), 0, 1;
 *   "WQ_GEMM_PUSH" -1 (auto) or 0 (pull form); "WQ_GEMM_STAGES" 0 (auto) or a ring depth;
 *   "WQ_QUANT_SCHEDULE" -1 (auto), 0 (cluster), 1 (stream), 2 (register-resident where it applies,
 *   else stream);
 *   "WQ_QUANT_SPLIT" 0 (auto) or 1..16;
 *   "WQ_QUANT_CTAS_PER_SM" 0 (auto) or a count;
 *   "WQ_GEMM_DB" -1 (auto), 0, 1: the two-accumulator form of the pair schedule off / on.
 * Process-wide; takes effect for launches issued after it returns.  Returns WQ_ERR_INVALID for an
 * unknown name.  wq_get_tuning returns the current value (or WQ_ERR_INVALID's value for an unknown name).
 */
WQ_API wq_status wq_set_tuning(const char *name, int value);
WQ_API int wq_get_tuning(const char *name);

/* Bytes of device scratch wq_linear_forward_host needs (workspace + x and y staging). */
WQ_API size_t wq_host_workspace_bytes(wq_weights_t h, int M);

/*
 * End-to-end variant over HOST buffers: copies x (host bf16 [M, K], pinned for the copies to
 * overlap) to the device, runs wq_linear_forward, copies y back to host bf16 [M, N].  From
 * M = 4096 rows the batch goes in up to eight row chunks whose uploads and downloads run on two
 * copy streams of the handle, overlapping each other and the kernels; the uploads start after the
 * work queued on `stream` before the call, and `stream` resumes only after the last download, so
 * y is valid once `stream` synchronises (as for a single chunk, which uses `stream` alone).
 * workspace: device, at least wq_host_workspace_bytes(h, M) bytes.  Calls that share a handle are
 * serialised on the host while they enqueue.
 */
WQ_API wq_status wq_linear_forward_host(wq_weights_t h, const void *x_host, int M, void *y_host,
                                        void *workspace, size_t workspace_bytes, void *stream);

/*
 * Run only the activation quantiser (for parity checks and for callers that keep the
 * quantised activations).  All outputs are device pointers:
 *   codes   uint8 [M, K/2]; element 2i of a row in the low nibble of byte i.  WQ_MODE_W4A8 handles:
 *           the e4m3 activation values as bf16 [M, K] instead (scales unused, may be NULL; gscale
 *           the per-row scale amax / 448).
 *   scales  e4m3 bytes: WQ_SCALE_LAYOUT_ROWMAJOR -> [M, K/16];
 *           WQ_SCALE_LAYOUT_MMA -> ceil(M/128) x (K/64) atoms of 512 bytes, atom (mb, kb)
 *           at offset (mb * K/64 + kb) * 512, row r of the 128-row block and 16-block j of
 *           the 64-block at byte (r % 32) * 16 + (r / 32) * 4 + j (the tcgen05
 *           block-scale layout the GEMM consumes).
 *   gscale  fp32 [M] tensor scales, one per row (equal in every row for WQ_ACT_SCALE_TENSOR and
 *           WQ_ACT_SCALE_STATIC).
 *   x_omega fp16 [M, xo_ld] (wq_side_strides); required when n_outliers > 0 (NULL otherwise).
 *   u       bf16 [M, u_ld] (wq_side_strides) or NULL (not computed when NULL).
 * For WQ_ACT_SCALE_TENSOR handles the batch maximum is gathered in a 4-byte device word owned by
 * the handle, so two such calls on one handle must not overlap on the GPU (wq_linear_forward keeps
 * that word in its workspace instead and has no such restriction).
 */
WQ_API wq_status wq_quantize_activations(wq_weights_t h, const void *x, int M, int scale_layout,
                                         uint8_t *codes, uint8_t *scales, float *gscale,
                                         void *x_omega, void *u, void *stream);

/*
 * GEMM + fused epilogue alone, on activations already quantised by
 * wq_quantize_activations(..., WQ_SCALE_LAYOUT_MMA, ...) (or, for a W8A8 handle, by
 * wq_quantize_activations_w8a8, with scales_mma NULL and gscale the per-row scale a).
 * All pointers are device:
 *   codes [M, K/2], scales_mma (MMA layout), gscale [M], u bf16 [M, rank] (required when
 *   rank > 0), x_omega fp16 [M, n_outliers] (required when n_outliers > 0), y bf16 [M, N].
 * One kernel runs on `stream`.
 */
WQ_API wq_status wq_linear_forward_quantized(wq_weights_t h, const uint8_t *codes, const uint8_t *scales_mma,
                                             const float *gscale, const void *u, const void *x_omega, int M,
                                             void *y, void *stream);

/*
 * Two chained 4-bit projections, with the second one's input quantised in the first one's GEMM
 * epilogue (the consistent folding of FoldQuantVLA, Key Contribution 1: the next consumer's
 * transform applied where its input is produced): no bf16 y is written and the second layer's
 * activation quantiser does not run.  The epilogue takes each output value as the bf16 that
 * wq_linear_forward would have stored, applies `next`'s smoothing and block-64 rotation along
 * this layer's N, moves `next`'s kept channels to x_omega and codes the rest in NVFP4 with
 * `next`'s fixed tensor scale -- bit-identical to wq_quantize_activations(next, that y).
 * Then wq_linear_forward_quantized(next, codes, scales_mma, gscale, NULL, x_omega, ...) finishes
 * the second layer.
 *   h        this layer (W4A4).
 *   next     the next layer: W4A4, next K == h's N, act_scale WQ_ACT_SCALE_STATIC (a per-row
 *            scale would need the whole row, which no output tile holds), rank 0 (its low-rank
 *            down-projection would need the whole row too); otherwise WQ_ERR_UNSUPPORTED.
 *   x        device bf16 [M, K] (this layer's input).
 *   codes    device uint8 [M, N/2]; scales_mma device, the MMA scale layout for K' = N;
 *   gscale   device fp32 [M] (every entry next's g); x_omega device fp16 [M, xo_ld of next]
 *            (required when next keeps channels, NULL otherwise).
 *   workspace  device, wq_workspace_bytes(h, M) bytes, 256-byte aligned.
 * Two kernels on `stream`: this layer's quantiser and its GEMM on the CTA-pair schedule.
 */
WQ_API wq_status wq_linear_forward_chain(wq_weights_t h, wq_weights_t next, const void *x, int M, uint8_t *codes,
                                         uint8_t *scales_mma, float *gscale, void *x_omega, void *workspace,
                                         size_t workspace_bytes, void *stream);

/*
 * The selective 8-bit projection (handle prepared with mode WQ_MODE_W8A8 or WQ_MODE_W8A8_FP8): the
 * 8-bit variant of the fused quantiser, then the tcgen05 GEMM -- on the int8 codes held as exact
 * bf16 integers (kind::f16), or on e4m3 bytes (kind::f8f6f4) -- with fp32 accumulation and the
 * epilogue y = a[m] w[n] acc + b.
 *   x, y, workspace  as for wq_linear_forward (workspace: wq_workspace_bytes(h, M)).
 */
WQ_API wq_status wq_linear_forward_w8a8(wq_weights_t h, const void *x, int M, void *y,
                                        void *workspace, size_t workspace_bytes, void *stream);

/*
 * The 8-bit quantiser alone (W8A8 handles), device outputs:
 *   codes  WQ_MODE_W8A8: bf16 [M, K] holding the integers q in [-127, 127] (scale a = amax / 127);
 *          WQ_MODE_W8A8_FP8: e4m3 bytes [M, K] (scale a = amax / 448).   scale fp32 [M].
 */
WQ_API wq_status wq_quantize_activations_w8a8(wq_weights_t h, const void *x, int M, void *codes,
                                              float *scale, void *stream);

/* 8-bit weights back to host (synchronous): q [N, K] bytes (K-major; int8 values, or e4m3 codes for
 * WQ_MODE_W8A8_FP8), w fp32 [N]. */
WQ_API wq_status wq_export_weights_w8a8(wq_weights_t h, int8_t *q, float *w);

/*
 * A video VAE's 3D convolution as an NVFP4 implicit GEMM (LatentQuant, Abstract: NVFP4 execution
 * of the Wan VAE).  The input is quantised once per voxel along channels (16-channel blocks,
 * e4m3 scales) with ONE fp32 scale for the whole [B, C_in, D, H, W] tensor (a GEMM row gathers
 * 27 voxels, so a per-voxel scale would not factor out); no smoothing or rotation.  The weight
 * is NVFP4 per output channel along K = (kd, kh, kw, c_in) with one fp32 scale per tensor.
 * y[b, n, v] = gx gw sum_{taps, c} A . W, bf16, stride 1, zero padding `pad`.
 *   w       host fp32 [C_out, C_in, kt, kh, kw];  C_in % 128 == 0, C_out % 16 == 0,
 *           kt kh kw C_in <= 16384.
 *   kt, kh, kw, pad  kernel extent and zero padding; the kernels implement the VAE's
 *           3 x 3 x 3 with padding 1 (the "same" convolution of the decoder's residual
 *           blocks) and return WQ_ERR_UNSUPPORTED for anything else.
 */
WQ_API wq_status wq_prepare_conv3d(const float *w, int C_in, int C_out, int kt, int kh, int kw, int pad,
                                   void *stream, wq_weights_t *out);

/* Device scratch for wq_conv3d_forward / wq_quantize_conv3d_input (B D H W voxels). */
WQ_API size_t wq_conv3d_workspace_bytes(wq_weights_t h, int B, int D, int H, int W);

/*
 *   x  device bf16 NCDHW [B, C_in, D, H, W];  y  device bf16 NCDHW [B, C_out, D, H, W];
 *   B >= 1, D H W % 8 == 0.  Three kernels on `stream`: |x| maxima, the per-voxel quantiser,
 *   the implicit GEMM (A rows gathered per tap by cp.async, zero-filled in the padding; taps
 *   never cross from one sample of the batch into another).
 */
WQ_API wq_status wq_conv3d_forward(wq_weights_t h, const void *x, int B, int D, int H, int W, void *y,
                                   void *workspace, size_t workspace_bytes, void *stream);

/* The conv input quantiser alone: codes [V, C_in/2], scales [V, C_in/16], g (one float),
 * all device; V = B D H W voxels numbered v = b D H W + (d H + h) W + w. */
WQ_API wq_status wq_quantize_conv3d_input(wq_weights_t h, const void *x, int B, int D, int H, int W,
                                          uint8_t *codes, uint8_t *scales, float *g,
                                          void *workspace, size_t workspace_bytes, void *stream);

/*
 * Copy the prepared weights back to host memory in canonical layouts (synchronous):
 *   codes uint8 [N, K/2]; scales e4m3 [N, K/16]; gW fp32 scalar; P bf16 [K, rank];
 *   Q bf16 [rank, N]; W_omega fp16 [n_outliers, N].  Any output may be NULL.
 */
WQ_API wq_status wq_export_weights(wq_weights_t h, uint8_t *codes, uint8_t *scales, float *gW,
                                   uint16_t *P, uint16_t *Q, uint16_t *W_omega);

/*
 * Synchronise `stream` and report whether a kernel of this handle set its device error
 * flag (a barrier wait that exceeded its time limit).  Clears the flag.
 * Returns WQ_OK or WQ_ERR_TIMEOUT (or WQ_ERR_CUDA).
 */
WQ_API wq_status wq_check_device_error(wq_weights_t h, void *stream);

/*
 * Self-test of the failure path that every kernel relies on (no counterpart on the pages).
 * One CTA waits on an mbarrier that nothing arrives on: the wait gives up after its limit
 * (WQ_WAIT_NS, 2 s of global time), records its site code in a device error flag and, through
 * the CTA's abort flag, releases a second waiter that started 0.5 s later before that waiter's
 * own limit.  No fault is raised and the context stays usable.  Synchronises the device.
 *   site       host int, out: the recorded site code (91 when the path works as designed)
 *   waited_ms  host double[2], out: how long the two waits lasted (the second one counted
 *              from its start, 0.5 s before its wait)
 *   released   host int, out: how many of the two waits returned without an arrival (2)
 * Returns WQ_ERR_TIMEOUT when a wait ran out (the status a forward reports through
 * wq_check_device_error in the same situation), WQ_OK if none did, WQ_ERR_CUDA on a launch
 * or copy failure, WQ_ERR_INVALID for a NULL output pointer.
 */
WQ_API wq_status wq_selftest_wait_timeout(int *site, double *waited_ms, int *released);

/*
 * Tensor-core issue-rate microbenchmark (no counterpart on the pages; a measurement utility).
 * On the current device, one thread per CTA (kind of MMA below) or per CTA pair issues `iters`
 * dense tcgen05.mma instructions back to back on fixed shared-memory operands into one TMEM
 * accumulator, with `copies` tcgen05.cp copies of scale atoms before each, on every SM at once,
 * timed on the device.  Synchronous; allocates and frees a few bytes of device memory.
 *   kind        0 = kind::mxf4nvf4 block-scaled e2m1 (K = 64 per instruction), 1 = kind::f16 bf16
 *               (K = 16), 2 = kind::f8f6f4 e4m3 (K = 32)
 *   n           N of the instruction, a multiple of 16 in [64, 256]; M = 128, or 256 with pair != 0
 *   copies      0..3 copies per MMA; copy_shape 0 = 32x128b.warpx4 (512 B), 1 = 128x256b (4 KiB)
 *   iters       1 .. 2^22 instructions per CTA
 *   feeder      who issues the copies: 0 the MMA thread (ordered before each MMA); 1 another warp,
 *               concurrently; 2 warps 1-3 write the same TMEM columns with tcgen05.st from registers
 *               instead (single CTA, copy_shape 0 only)
 *   zero_data   1: all-zero operands (0: a fixed pseudo-random pattern)
 *   accs        1, or 2 accumulators alternated instruction by instruction (N <= 128 for kind 0)
 *   tflops      host out: dense TFLOP/s summed over all SMs (2 M N K per instruction)
 *   ns_per_mma  host out: mean ns per instruction;  sm_mhz  host out: mean SM clock during the run
 * Returns WQ_ERR_INVALID for a bad argument, WQ_ERR_CUDA / WQ_ERR_TIMEOUT on a failed run.
 */
WQ_API wq_status wq_mma_peak(int kind, int n, int pair, int copies, int copy_shape, int iters, int feeder,
                             int zero_data, int accs, double *tflops, double *ns_per_mma, double *sm_mhz);

/*
 * On-device outlier calibration (QuantWAMs sec. 3.1, Eq. (1)-(3), one context): the pooled squared
 * energy of each channel of the transformed activation, z(c) = mean_t xt[t, c]^2, where xt is the
 * activation quantiser's transform of each row (the smoothing 1/s before or after the block-64
 * Walsh-Hadamard rotation, per transform_order; fp32 steps, fp64 squares and sums), and the Top-K
 * channels by z -- the Omega that wq_prepare_weights takes for the fp16 exception path.
 *   x        device bf16 [M, K] calibration activations (M >= 1; K % 64 == 0, K <= 16384).
 *   s        device fp32 [K] smoothing factors (> 0) or NULL for s = 1.
 *   rotate   1: block-64 FWHT; 0: none.   transform_order: WQ_ORDER_*.
 *   n_top    0 <= n_top <= K channels to select.
 *   z        device fp64 [K], out.   omega  device int32 [n_top], out: ascending channel indices,
 *            the n_top largest z (ties go to the lower index).
 *   workspace  device, wq_calibration_workspace_bytes(M, K) bytes, 256-byte aligned.
 * Four kernels on `stream`.  Returns WQ_ERR_INVALID / WQ_ERR_UNSUPPORTED on bad arguments.
 */
WQ_API size_t wq_calibration_workspace_bytes(int M, int K);
WQ_API wq_status wq_calibrate_outliers(const void *x, int M, int K, const float *s, int rotate, int transform_order,
                                       int n_top, double *z, int32_t *omega, void *workspace,
                                       size_t workspace_bytes, void *stream);

/* Release the handle and its device memory (synchronises the device first).  NULL is a no-op. */
WQ_API void wq_free_weights(wq_weights_t h);

/*
 * Forward without any device allocation by the caller or the library.
 * No counterpart on the pages: this entry point exists for deployment hosts that cannot
 * call cudaMalloc or hand out scratch buffers after start-up -- for instance a plugin
 * whose host engine owns every device allocation, or a real-time control loop that
 * forbids allocation once running so that its latency stays predictable.
 *   x, y    device bf16 [M, K] and [M, N], owned by the caller as in wq_linear_forward.
 * Scratch comes from one static device array of WQ_NOALLOC_SCRATCH_BYTES bytes, linked
 * into the library; every GPU that loads the library holds it until the process exits.
 * The first call on a device looks up that array's device address (a one-time set-up);
 * make that first call before any stream capture.  All calls share the one array and it
 * keeps the last call's contents (what must start at zero, the call clears), so calls whose
 * kernels overlap on the GPU -- on different streams, or through different handles --
 * race with each other: serialise them.  A call whose scratch need
 * wq_workspace_bytes(h, M) exceeds WQ_NOALLOC_SCRATCH_BYTES returns WQ_ERR_UNSUPPORTED.
 * It allocates nothing itself and otherwise behaves exactly like wq_linear_forward.
 */
#define WQ_NOALLOC_SCRATCH_BYTES (16u << 20)
WQ_API wq_status wq_linear_forward_noalloc(wq_weights_t h, const void *x, int M, void *y, void *stream);

/* Thread-local description of the last error ("" if none). */
WQ_API const char *wq_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* WQ_H_ */
