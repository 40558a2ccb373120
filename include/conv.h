/*
 * conv.h -- C ABI of the GB300 (sm_103a) forward 2D convolution library.
 *
 * Operation (one call = one layer):
 *
 *   y[n][ho][wo][co] = act( bias[co] + sum_{ci'<C_in/G} sum_{kh<Kh} sum_{kw<Kw}
 *                             x[n][ho*S + kh*D - P][wo*S + kw*D - P][g*C_in/G + ci']
 *                           * w[co][kh][kw][ci'] ),     g = co / (C_out/G)
 *
 * Input coordinates outside [0,H) x [0,W) read as zero.  act is ReLU when
 * CONV_FLAG_RELU is set, else identity.  Depthwise convolution is the case
 * G = C_in = C_out.
 *
 * Sources: the dot-product definition and index map of "GPU lesson 9: how a
 * GPU executes neural-network convolution" (lincklin.cn), section 2; zero
 * padding as an address test, section 26; the conv-as-GEMM mapping
 * M = C_out, N = N*H_out*W_out, K = C_in*Kh*Kw, section 19; bias and
 * activation fused after the sum, section 31.  Dilation, groups and the output
 * size H_out = floor((H + 2P - D(Kh-1) - 1)/S) + 1 follow "Convolution variants
 * and their matrix operations" (lpnh.cn/news/2674933), sections 2.2, 2.3, 4.2,
 * 4.3 and 6.2.  The same S, P, D apply to both spatial axes.
 *
 * Layouts (all dense, row-major, caller-owned device memory):
 *   x    [N][H][W][C_in]              (NHWC)
 *   w    [C_out][Kh][Kw][C_in/G]      (K order kh, kw, ci)
 *   bias [C_out], always FP32          (read only when CONV_FLAG_BIAS is set)
 *   y    [N][H_out][W_out][C_out]     (NHWC)
 * Element types: CONV_F32 -> x, w, y FP32 (y BF16 when CONV_FLAG_OUT_BF16);
 *                CONV_BF16 -> x, w, y BF16.  Accumulation is always FP32.
 *
 * Ownership: the plan is host memory owned by the caller between
 * conv_plan_create and conv_plan_destroy.  It owns no device memory and
 * allocates none.  A plan may be reused for any number of forwards with any
 * pointers of the right size, but not from two host threads at once (it caches
 * TMA descriptors keyed by pointer).
 *
 * Errors: every call returns a conv_status; no call prints, traps or aborts.
 * conv_forward is asynchronous on the given stream and never synchronises;
 * device-side wait timeouts (a safety net that fires only on a hang) are
 * latched in the plan's own device word, read by conv_plan_device_status (one
 * plan, in stream order) and by conv_device_status (every word, whole device).
 */
#ifndef CONV_GB300_CONV_H
#define CONV_GB300_CONV_H

#ifdef __cplusplus
extern "C" {
#endif

typedef struct conv_plan conv_plan;     /* opaque, host-owned */

typedef enum { CONV_F32 = 0, CONV_BF16 = 1 } conv_dtype;

enum {
    CONV_FLAG_BIAS = 1u,       /* add bias[co] after the sum                          */
    CONV_FLAG_RELU = 2u,       /* max(., 0) after the bias                            */
    CONV_FLAG_OUT_BF16 = 4u,   /* CONV_F32 only: write y as BF16 (round to nearest even) */
    CONV_FLAG_SM_PAIRS = 8u,   /* tensor-core GEMM paths: run each MMA on an SM pair
                                  (clusters of 2, 256 pixels per MMA, weight rows split
                                  between the two SMs) instead of one SM per 128 pixels.
                                  Without this flag or CONV_FLAG_ONE_SM the plan picks:
                                  pairs for ungrouped non-1x1 layers with 256 output
                                  channels per tile and at least 9 K-steps (taps x
                                  64-channel blocks), one SM otherwise */
    CONV_FLAG_TRANSPOSED = 16u, /* transposed convolution (see below)                 */
    CONV_FLAG_ONE_SM = 64u,    /* tensor-core GEMM paths: one SM per 128-pixel tile    */
    CONV_FLAG_PER_TAP = 128u,  /* stride-1 implicit GEMM: gather each tap's 128 input
                                  pixels as their own TMA box (every input pixel lands
                                  in shared memory once per tap) instead of the default
                                  halo tiles, where one box per 64-channel block holds
                                  the input under an 8 x 16 output tile plus the
                                  (K-1)*D border its taps reach and every tap reads it
                                  ("GPU lesson 9", sections 6 and 12-13: input reuse
                                  across a tile's taps).  Same results up to the order
                                  of the FP32 sum.  Ignored by other plans. */
    CONV_FLAG_WINOGRAD = 32u   /* FP32 3x3, stride 1, dilation 1, G = 1: Winograd F(2x2, 3x3)
                                  ("Convolution vs inner product", lnrq.cn, section 2.2;
                                  variants page, section 3.3): 4 multiplies per output
                                  instead of 9, rounding differs from the direct sum (the
                                  pages' precision caveat; it stays within FP32 tolerance
                                  on Kaiming-scale data).  Ignored for other plans. */
};

/*
 * Transposed convolution (CONV_FLAG_TRANSPOSED): the adjoint (matrix
 * transpose) of the convolution with the same S, P, D, G ("Convolution
 * variants and their matrix operations", sections 2.3 and 4.2: it upsamples;
 * S-1 zeros between neighbouring input pixels, then a stride-1 convolution;
 * in matrix form Y_col = W^T X).  Input pixel (i, j) of x [N][H][W][C_in]
 * adds x * w[co][kh][kw][ci'] to output (i*S + kh*D - P, j*S + kw*D - P) of
 * y [N][H_out][W_out][C_out]; positions outside the output are dropped:
 *
 *   y[n][ho][wo][co] = act( bias[co] + sum over ci' < C_in/G, kh, kw with
 *        i = (ho + P - kh*D)/S and j = (wo + P - kw*D)/S exact and inside the
 *        input of x[n][i][j][g*C_in/G + ci'] * w[co][kh][kw][ci'] ),
 *
 *   H_out = (H - 1)*S - 2P + D(Kh - 1) + 1, W_out likewise (no output padding;
 *   the pages give no formula, this is the adjoint's size).
 *
 * The weight keeps this library's layout [C_out][Kh][Kw][C_in/G] (a framework
 * weight [C_in][C_out/G][Kh][Kw] is permuted to it, not flipped).
 */

typedef enum {
    CONV_OK = 0,
    CONV_ERR_INVALID_ARG = 1,  /* bad size, NULL pointer or NULL plan                 */
    CONV_ERR_UNSUPPORTED = 2,  /* valid convolution this library does not run          */
    CONV_ERR_MISALIGNED = 3,   /* a device pointer is not 16-byte aligned              */
    CONV_ERR_CUDA = 4,         /* a CUDA runtime / driver call failed                  */
    CONV_ERR_NO_MEMORY = 5,    /* host allocation of the plan failed                   */
    CONV_ERR_TIMEOUT = 6       /* a device-side wait gave up (reported by conv_device_status) */
} conv_status;

/* Which kernel a plan runs (conv_plan_info).  A BF16 transposed plan runs the
 * implicit-GEMM kernel in its phase mode when C_in/G % 64 == 0, C_out/G % 16 == 0,
 * S <= 4, Kh, Kw <= 8, every output phase has at least one tap and S divides
 * H_out and W_out; other transposed plans run the direct kernel. */
typedef enum {
    CONV_PATH_DIRECT = 0,         /* CUDA-core direct loop, any shape                      */
    CONV_PATH_DEPTHWISE = 1,      /* FP32 depthwise, TMA halo tile in shared memory        */
    CONV_PATH_GEMM_1X1 = 2,       /* BF16 1x1 / stride 1 / pad 0: tcgen05 GEMM, tiled TMA  */
    CONV_PATH_IMPLICIT_GEMM = 3,  /* BF16 implicit GEMM: TMA im2col + tcgen05 + TMEM        */
    CONV_PATH_SMALL_K_GEMM = 4,   /* BF16, C_in*Kh*Kw <= 64 (e.g. a 3-channel stem): rows
                                     staged by bulk copy, K gathered in shared memory,
                                     tcgen05 + TMEM                                     */
    CONV_PATH_WINOGRAD = 5        /* FP32 Winograd F(2x2, 3x3) on CUDA cores (opt-in)     */
} conv_path;

/*
 * Create a plan for one convolution shape.  Validates the shape (all sizes
 * > 0, P >= 0, C_in % G == 0, C_out % G == 0, H_out >= 1, W_out >= 1,
 * CONV_FLAG_OUT_BF16 only with CONV_F32) and chooses the kernel.  Returns
 * CONV_ERR_INVALID_ARG for a bad shape or out == NULL, CONV_ERR_NO_MEMORY if
 * the host allocation fails, CONV_ERR_CUDA if the current device cannot be
 * queried.  On error *out is set to NULL.  The plan is tied to the CUDA device
 * current at creation: conv_forward / conv_forward_affine with another device
 * current return CONV_ERR_INVALID_ARG without launching.
 */
conv_status conv_plan_create(conv_plan **out, int N, int C_in, int H, int W, int C_out,
                             int Kh, int Kw, int S, int P, int D, int G,
                             conv_dtype dtype, unsigned flags);

/* Output extent, floor((H + 2P - D(K-1) - 1)/S) + 1 per axis. */
conv_status conv_plan_output_shape(const conv_plan *p, int *H_out, int *W_out);

/*
 * The chosen kernel (conv_path) and the logical GEMM extents of section 19 of
 * lesson 9: M = C_out, N = N*H_out*W_out, K = (C_in/G)*Kh*Kw (per group).  For
 * a transposed plan, the extents of its matrix form Y_col = W^T X (variants
 * page, section 4.2): M = C_out*Kh*Kw, N = N*H*W, K = C_in/G.
 * Any output pointer may be NULL.
 */
conv_status conv_plan_info(const conv_plan *p, int *path, long long *gemm_m,
                           long long *gemm_n, long long *gemm_k);

/*
 * Run the convolution on `stream` (a cudaStream_t; NULL = the legacy default
 * stream).  x, w, y must be non-NULL device pointers, 16-byte aligned; bias
 * must be a non-NULL 16-byte aligned device pointer when CONV_FLAG_BIAS is set
 * and is ignored otherwise.  y must not overlap x, w or bias.  Returns
 * CONV_ERR_INVALID_ARG / CONV_ERR_MISALIGNED without launching anything,
 * CONV_ERR_CUDA if a descriptor encode or the launch fails.  Asynchronous: the
 * return value does not cover faults that happen after the launch.
 */
conv_status conv_forward(conv_plan *p, const void *x, const void *w, const void *bias,
                         void *y, void *stream);

/*
 * conv_forward with a per-channel scale applied to the sum before the bias:
 *
 *   y[n][ho][wo][co] = act( scale[co] * sum + bias[co] )
 *
 * i.e. a batch normalisation folded into the epilogue (scale = gamma /
 * sqrt(var + eps), bias = beta - mean * scale): the per-channel "scale and
 * shift" step of lesson 9, section 31, fused with the bias and activation.
 * scale is a device pointer to C_out FP32 values, non-NULL and 16-byte
 * aligned; bias follows the plan's CONV_FLAG_BIAS as in conv_forward (without
 * it the shift is zero).  Same layouts, errors and asynchrony as conv_forward.
 */
conv_status conv_forward_affine(conv_plan *p, const void *x, const void *w, const void *scale,
                                const void *bias, void *y, void *stream);

/* Free the plan (host memory; its status word goes back to the pool).  Launches
 * still in flight keep running; a wait of theirs that gives up after this call may
 * latch its bit into the word's next owner.  NULL is accepted. */
conv_status conv_plan_destroy(conv_plan *p);

/* Static English text for a status code; never NULL. */
const char *conv_status_string(conv_status s);

/*
 * Synchronise the current device, then read and clear every status word the
 * library keeps on it: the library-wide word and every plan's own word (below).
 * *code receives 0 when no kernel hit a wait timeout since the last call, else
 * the OR of the bit sets naming the waits that gave up.  Returns
 * CONV_ERR_TIMEOUT when *code != 0, CONV_ERR_CUDA if the synchronisation or
 * read fails (a sticky fault from an earlier launch shows up here), else CONV_OK.
 */
conv_status conv_device_status(int *code);

/*
 * Each plan (conv_plan and conv_block_plan) takes its own device status word at
 * creation, from a fixed array of 1,024 per device (no allocation: creation clears
 * the word with a memset on the default stream); when all are taken it shares the
 * library-wide word.  This reads and clears the plan's word in the order of
 * `stream` (after the work queued on it, then waits for the stream only, not the
 * device): *code receives the bits of the plan's kernels whose waits gave up.
 * Returns CONV_ERR_TIMEOUT when *code != 0, CONV_ERR_INVALID_ARG for NULL
 * arguments or with another device current than the plan's, CONV_ERR_CUDA for a
 * host-only plan or a failed copy.  A plan used on several streams at once should
 * be read after all of them (the word is shared by its launches).
 */
conv_status conv_plan_device_status(const conv_plan *p, void *stream, int *code);

/* Number of SMs the plan's grid sizing uses (device property of the plan's device). */
int conv_plan_num_sms(const conv_plan *p);

/* Measured dense BF16 tensor rate (a measurement helper, not a convolution):
 * launches `grid` CTAs, one per SM (each holds more than half of an SM's shared
 * memory, so pass grid <= the SM count), and each issues `iters` (1..2^20)
 * back-to-back tcgen05.mma of M = 128, N = 256, K = 16 (BF16 in, FP32
 * accumulate in tensor memory) and writes the SM cycles from its first issue
 * to the last completion to cycles[cta] (a 8-byte aligned device array of
 * `grid` entries, caller-owned; 0 where the completion wait timed out, which
 * also sets conv_device_status).  FLOP per clock per SM =
 * 2 * 128 * 256 * 16 * iters / cycles[cta].  Asynchronous on `stream`.
 * Returns CONV_ERR_INVALID_ARG / CONV_ERR_MISALIGNED without launching, or
 * CONV_ERR_CUDA if the launch fails. */
conv_status conv_measure_mma_rate(int iters, unsigned long long *cycles, int grid, void *stream);

/*
 * Test aid, not a convolution: makes the kernels' bounded-wait failure path run.
 * Every mbarrier wait in this library's kernels gives up after a time limit
 * (2 s), sets a bit in the device status word, raises its CTA's abort flag so
 * the CTA's other roles leave their waits, frees tensor memory and returns (the
 * pipeline-hang detection of the failure-handling design; no trap, no fault).
 * This launches one CTA on `stream` in which one role waits on an mbarrier that
 * nothing completes, with a limit of `limit_ns` (1 .. 2e9 ns), and a second role
 * waits on another such barrier with the kernels' own 2 s limit.  The first gives
 * up after limit_ns and sets bit 2; the second leaves through the abort flag and
 * sets bit 4.  conv_device_status afterwards returns CONV_ERR_TIMEOUT with code
 * 6 and clears the word; the context stays usable.  If `elapsed_ns` is non-NULL
 * (device memory, 8-byte aligned) it receives how long the second role waited
 * (%globaltimer ns): at least limit_ns, far below 2 s.  Returns CONV_ERR_INVALID_ARG / CONV_ERR_MISALIGNED without launching,
 * CONV_ERR_CUDA if the launch fails.  Asynchronous.
 */
conv_status conv_check_wait_timeout(unsigned long long limit_ns, unsigned long long *elapsed_ns, void *stream);

/*
 * Launch configuration conv_forward uses for this plan: grid and block size
 * (CTAs, threads), dynamic shared memory per CTA in bytes, pipeline stages,
 * and CTAs per cluster (2 for SM pairs, else 1).  Any output pointer may be
 * NULL.  Returns CONV_ERR_INVALID_ARG for a NULL plan.
 */
conv_status conv_plan_launch_info(const conv_plan *p, int *grid, int *block, int *smem_bytes,
                                  int *stages, int *cluster);

/*
 * How a tensor-core GEMM plan (CONV_PATH_GEMM_1X1, CONV_PATH_IMPLICIT_GEMM) runs the
 * contraction (lesson 9, sections 21-24: the convolution as a GEMM over pixels x output
 * channels x C_in/G*Kh*Kw), for tests and tuning:
 *   mode              0 = 1x1 (A is the [pixels][C_in] matrix), 1 = TMA im2col (stride > 1),
 *                     2 = one input box per tap (stride 1 with CONV_FLAG_PER_TAP, or a halo
 *                     wider than a TMA box), 3 = phase (transposed), 4 = halo tiles;
 *   n_tile            output channels per tile (the accumulator's columns);
 *   pair              1: SM pairs (cta_group::2, 256 pixels per MMA);
 *   dual              1: two pixel tiles per CTA;
 *   resident_weights  1: every CTA keeps one n-tile, and that n-tile's weight rows for the
 *                     whole reduction sit in shared memory from its first tile on (loaded
 *                     once instead of once per tile);
 *   swapped           1: two tiles per CTA of 128 output channels with the operands swapped:
 *                     the weights are the MMA's M side and both tiles' 256 pixels its N
 *                     side (one M128 N256 MMA per K = 16 instead of two M128 N128).
 * Any output pointer may be NULL.  Returns CONV_ERR_INVALID_ARG for a NULL plan or one on
 * another path.
 */
conv_status conv_plan_gemm_config(const conv_plan *p, int *mode, int *n_tile, int *pair, int *dual,
                                  int *resident_weights, int *swapped);

/* ------------------------------------------------------------------------
 * Depthwise-separable block in one kernel: depthwise 3x3 (FP32) followed by
 * pointwise 1x1 (BF16 tensor cores), the two stages of "GPU lesson 9"
 * section 25, fused so the depthwise feature map never goes to memory (the
 * kernel fusion that section names to save its write and re-read):
 *
 *   t[n][ho][wo][c]  = bf16( act_dw( dw_scale[c] * sum_{kh,kw<3}
 *                        x[n][ho+kh-P][wo+kw-P][c] * w_dw[c][kh][kw] + dw_bias[c] ) )
 *   y[n][ho][wo][co] = act_pw( pw_scale[co] * sum_{c<C} t[n][ho][wo][c] * w_pw[co][c]
 *                        + pw_bias[co] )
 *
 * with H_out = H + 2P - 2, W_out = W + 2P - 2 (stride 1, dilation 1), input
 * pixels outside the image read as zero, bf16() round-to-nearest-even (the
 * pointwise GEMM's BF16 operand; the sum stays FP32), act_dw / act_pw ReLU when
 * CONV_BLOCK_DW_RELU / CONV_BLOCK_PW_RELU is set.
 *
 * Layouts (dense, caller-owned device memory, 16-byte aligned):
 *   x        [N][H][W][C]        FP32 (NHWC)
 *   w_dw     [C][3][3]           FP32
 *   dw_scale, dw_bias [C]        FP32, each may be NULL (scale 1, shift 0)
 *   w_pw     [C_out][C]          BF16
 *   pw_scale, pw_bias [C_out]    FP32, each may be NULL (scale 1, shift 0)
 *   y        [N][H_out][W_out][C_out]  BF16 (NHWC)
 * Supported: K = 3, 0 <= P <= 2, C % 64 == 0 and C <= 256, C_out % 32 == 0
 * (the output channels run as equal slices of at most 256, each a multiple
 * of 32, two slices in flight in tensor memory).  Other blocks get CONV_ERR_UNSUPPORTED from the create call
 * and run as two conv_forward calls (a depthwise plan with CONV_FLAG_OUT_BF16,
 * then a 1x1 plan).  The plan owns no device memory.
 * ------------------------------------------------------------------------ */
typedef struct conv_block_plan conv_block_plan; /* opaque, host-owned */

#define CONV_BLOCK_DW_RELU 1u
#define CONV_BLOCK_PW_RELU 2u

/*
 * Check the block's shape and choose its launch configuration.  *plan gets a
 * new plan, or NULL on error.  Like a convolution plan, it is tied to the
 * device current at creation (its forward returns CONV_ERR_INVALID_ARG with
 * another device current).  Returns CONV_ERR_INVALID_ARG for non-positive
 * sizes, an empty output or unknown flags, CONV_ERR_UNSUPPORTED for a valid
 * block outside the supported family above, CONV_ERR_CUDA if the device
 * cannot be queried.  Without a device a host-only plan is made (shape checks
 * only); its forward returns CONV_ERR_CUDA.
 */
conv_status conv_block_plan_create(conv_block_plan **plan, int N, int C, int H, int W, int C_out,
                                   int K, int P, unsigned flags);

/* Output extents of the block (H_out = H + 2P - 2, W_out = W + 2P - 2). */
conv_status conv_block_plan_output_shape(const conv_block_plan *p, int *H_out, int *W_out);

/*
 * Run the block on `stream` (a cudaStream_t; NULL = the legacy default
 * stream).  x, w_dw, w_pw, y must be non-NULL; every non-NULL pointer must be
 * 16-byte aligned (else CONV_ERR_MISALIGNED); y must not overlap any input.
 * Asynchronous like conv_forward; wait timeouts are latched for
 * conv_device_status.
 */
conv_status conv_block_forward(conv_block_plan *p, const void *x, const void *w_dw,
                               const void *dw_scale, const void *dw_bias, const void *w_pw,
                               const void *pw_scale, const void *pw_bias, void *y, void *stream);

/*
 * Launch configuration of conv_block_forward: grid and block size, dynamic
 * shared memory per CTA, halo-copy and weight-ring stages.  Any output
 * pointer may be NULL.
 */
conv_status conv_block_plan_launch_info(const conv_block_plan *p, int *grid, int *block,
                                        int *smem_bytes, int *halo_stages, int *weight_stages);

/* The block plan's own status word, read and cleared in the order of `stream`:
 * the same contract as conv_plan_device_status. */
conv_status conv_block_plan_device_status(const conv_block_plan *p, void *stream, int *code);

/* Free the block plan: the same contract as conv_plan_destroy.  NULL is accepted. */
conv_status conv_block_plan_destroy(conv_block_plan *p);

#ifdef __cplusplus
}
#endif

#endif /* CONV_GB300_CONV_H */
