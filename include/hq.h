/*
 * hq.h -- C ABI of the GB300 (sm_103a) quantized-weight matvec library (libhq.so).
 *
 * The library computes the bandwidth-bound decode product y = W_deq . x over
 * block-quantized weights, for 1..8 activation vectors in one pass, so that
 * every weight byte is streamed from HBM once per call.
 *
 * Sources (page title, section):
 *   - "One Native Stack for Private, Continuously-Learning AI", section "The
 *     Unified Quant Core": one quant-agnostic decode matvec over the ggml
 *     block formats Q8_0 (symmetric, 34 B per 32 weights) and Q4_0
 *     (symmetric, 18 B per 32 weights); the same core evaluates every routed
 *     MoE expert.  Section "The Central Efficiency Thesis", Lemma "QLoRA over
 *     the unified core is exact": y_i = sum_j What_ij x_j, What the CPU
 *     dequantization of the stored bytes, accumulated in f32.
 *   - "Economical Serving and the hanzo.ai Platform", subsection "The Roofline
 *     that Sets the Price": decode time per token is W/B (weight bytes over
 *     bandwidth); subsection "One Quant-Agnostic Core": per-format block
 *     decoder + traits record, reused by decode and MoE.
 *   - "Blue -- porting zen-nano (Qwen3-0.6B) to deterministic on-chain
 *     inference", section "Quantization recipe (validated)": per-output-channel
 *     symmetric int8 weights and gemmlowp requant
 *     (SaturatingRoundingDoublingHighMul, then RoundingDivideByPOT) to int8.
 *   - "DeepSeek-V4 on Hanzo Engine", section "A Fused Attention Kernel for
 *     512-Wide Latent Heads": speculative-verify widths q in [1, 8], hence
 *     n_vec in [1, 8].
 *
 * Conventions shared by every entry point
 *   - Pointers named W, x, y, ids, mult, shift, acc, out, scale are DEVICE
 *     pointers owned by the caller (cudaMalloc / PyTorch).  The library never
 *     allocates, frees or retains them, and keeps no state between calls other
 *     than a thread-local error string and a device fault word (below).
 *   - Every call is asynchronous and stream-ordered on `stream` (a
 *     cudaStream_t; NULL is the legacy default stream).  Arguments are
 *     validated on the host before any launch; a non-OK status means nothing
 *     was launched (except HQ_ERR_LAUNCH, which reports the launch failure).
 *     A fault inside a kernel surfaces at the caller's next synchronization.
 *   - Row-major layouts.  Quantized rows are packed blocks with no padding:
 *     row i of a Q8_0 matrix is bytes [i*cols/32*34, (i+1)*cols/32*34).
 *   - Block layouts (little-endian): Q8_0 = { uint16 fp16 d; int8 q[32] },
 *     w_j = d*q_j.  Q4_0 = { uint16 fp16 d; uint8 qs[16] }, element j (0..15)
 *     is the low nibble of qs[j] and element j+16 the high nibble,
 *     w = d*(n - 8).
 *   - Float paths accumulate in fp32 and are deterministic run to run (fixed
 *     reduction order, no float atomics).  They match the f64 definition
 *     within |y - y_ref| <= 1e-3 * sum_j |w_deq x_j| + 1e-5 per output.
 *     The int8 path is bit-exact.
 *   - Shapes: rows >= 1, cols >= 32, cols % 32 == 0 (int8: cols >= 4 and
 *     cols % 4 == 0), 1 <= n_vec <= 8.  W and x must be 16-byte aligned.
 *     When cols % 256 == 0 (every decode shape) the TMA-staged kernel runs;
 *     other legal shapes run a plain-load kernel that gives the same results
 *     to the same tolerance.  There is no CPU fallback.
 */
#ifndef HQ_H_
#define HQ_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *hq_stream_t;   /* identical to cudaStream_t */

typedef enum {
    HQ_OK = 0,
    HQ_ERR_NULL = -1,         /* a required pointer is NULL                        */
    HQ_ERR_SHAPE = -2,        /* rows/cols/n_experts/n_active out of range         */
    HQ_ERR_ALIGN = -3,        /* W or x not 16-byte aligned (y: 4-byte)            */
    HQ_ERR_NVEC = -4,         /* n_vec not in [1, 8]                               */
    HQ_ERR_LAUNCH = -5,       /* the CUDA launch failed (see hq_last_error)        */
    HQ_ERR_UNSUPPORTED = -6,  /* no sm_100-family GPU, or a value not representable */
    HQ_ERR_DEVICE = -7        /* a kernel reported a fault word (hq_device_fault)  */
} hq_status;

/* Format codes taken by hq_debug_plan. */
#define HQ_FMT_Q8_0 8
#define HQ_FMT_Q4_0 4
#define HQ_FMT_Q4_K 75      /* 'K' */
#define HQ_FMT_I8 1

/* Library version (major*10000 + minor*100 + patch). */
int hq_version(void);

/* Message for the last non-OK status returned on this host thread ("" if none). */
const char *hq_last_error(void);

/*
 * hq_matvec_q8_0 -- y[v][i] = sum_j w_deq[i][j] * x[v][j] for v < n_vec, i < rows.
 *   W  : Q8_0 blocks, rows x (cols/32) x 34 bytes, 16-byte aligned.
 *   x  : fp32 [n_vec][cols], 16-byte aligned.
 *   y  : fp32 [n_vec][rows], overwritten (not accumulated).
 * Accumulation is fp32; |y - y_exact| <= 1e-3 * sum_j |w_deq[i][j] * x[v][j]| + 1e-5
 * for finite x with |x| < 2^100 (beyond that a block's partial sum may
 * overflow).  Every quant is decoded to its signed value exactly before it
 * multiplies x, so the rounding is relative to the products |w x| themselves:
 * the bound holds at every n_vec for sparse or outlier-dominated blocks and
 * for x of any sign pattern or mean.
 * Source: "One Native Stack ...", section "The Unified Quant Core" (Q8_0,
 * 34 B/32) and the Lemma of section "The Central Efficiency Thesis".
 */
hq_status hq_matvec_q8_0(const void *W, const float *x, float *y,
                         int64_t rows, int64_t cols, int n_vec, hq_stream_t stream);

/*
 * hq_matvec_q4_0 -- as hq_matvec_q8_0 for Q4_0 blocks (rows x cols/32 x 18 B):
 * w = d * (n - 8), nibble order as in the conventions above; the same
 * accuracy and the same |x| < 2^100 precondition.
 * Source: "One Native Stack ...", section "The Unified Quant Core" (Q4_0, 18 B/32).
 */
hq_status hq_matvec_q4_0(const void *W, const float *x, float *y,
                         int64_t rows, int64_t cols, int n_vec, hq_stream_t stream);

/*
 * hq_matvec_q4_k -- as hq_matvec_q8_0 for Q4_K super-blocks: W is
 * rows x (cols/256) x 144 bytes, 16-byte aligned, cols % 256 == 0
 * (HQ_ERR_SHAPE otherwise).  A super-block is { fp16 d, fp16 dmin, uint8
 * scales[12], uint8 qs[128] }: sub-block j (32 weights, j = 0..7) has a
 * six-bit scale sc_j and min m_j -- for j < 4, sc_j = scales[j] & 63 and
 * m_j = scales[j+4] & 63; for j >= 4, sc_j = (scales[j+4] & 15) |
 * (scales[j-4] >> 6) << 4 and m_j = (scales[j+4] >> 4) | (scales[j] >> 6) << 4
 * -- and its quants are the low (even j) or high (odd j) nibbles of
 * qs[32*(j/2) .. +31]; w = d*sc_j*q - dmin*m_j.  Each weight is formed in fp32
 * (one rounding) before it multiplies x, so the accuracy statement and the
 * |x| < 2^100 precondition of hq_matvec_q8_0 hold unchanged.
 * Source: "One Native Stack ...", sections "The Unified Quant Core" (Q4_K is
 * one of the native formats) and "Ported Versus Novel" (formats taken
 * verbatim from ggml, whose Q4_K super-block this is); "Economical Serving
 * ...", subsection "One Quant-Agnostic Core, Not a Kernel-per-Quant Zoo"
 * (the Q4_K decode kernel).
 */
hq_status hq_matvec_q4_k(const void *W, const float *x, float *y,
                         int64_t rows, int64_t cols, int n_vec, hq_stream_t stream);


/*
 * hq_matvec_q8_0_lora, hq_matvec_q4_0_lora -- the float matvec of the same
 * format plus a QLoRA adapter over the frozen quantized base:
 *   y[v][i] = sum_j w_deq[i][j] x[v][j] + scale * sum_k B[i][k] (sum_j A[k][j] x[v][j]).
 *   lora_A    : bf16 [rank][cols] (raw bf16 bits), 16-byte aligned.
 *   lora_B    : bf16 [rows][rank], 2-byte aligned.
 *   scale     : alpha / r, finite.   rank : 1..64.
 *   workspace : caller-owned device memory of at least rank * n_vec floats,
 *               4-byte aligned; it receives u = A x (fp32 [n_vec][rank]) and
 *               must not be in use by other work until the call's kernels end.
 * W, x, y, rows, cols, n_vec and the accuracy are as for hq_matvec_q8_0; the
 * adapter term adds 1e-3 * |scale| * sum_k |B[i][k]| * sum_j |A[k][j] x[v][j]|
 * to the tolerance.  Two kernels run: the down projection u = A x, then the
 * matvec, which streams W once and adds scale * B u as it stores y.
 * Source: "One Native Stack ...", section "The Central Efficiency Thesis",
 * Lemma "QLoRA over the unified core is exact and base-weight-identical".
 */
hq_status hq_matvec_q8_0_lora(const void *W, const float *x, const uint16_t *lora_A,
                              const uint16_t *lora_B, float scale, int rank, float *workspace,
                              float *y, int64_t rows, int64_t cols, int n_vec, hq_stream_t stream);
hq_status hq_matvec_q4_0_lora(const void *W, const float *x, const uint16_t *lora_A,
                              const uint16_t *lora_B, float scale, int rank, float *workspace,
                              float *y, int64_t rows, int64_t cols, int n_vec, hq_stream_t stream);

/*
 * hq_matvec_q8_0_lora_noalloc -- hq_matvec_q8_0_lora without a workspace, for
 * callers that cannot allocate device memory.  Examples are code inside an
 * engine that hands all device memory to its own pre-sized pool, and a hot
 * path that must not call cudaMalloc / cudaFree, which may synchronize the
 * device.  Such a caller can pass no workspace for u = A x.
 *   Scratch: u lives in one file-scope array of 2 KB in the library's static
 *   device memory (64 x 8 fp32: the largest rank times the largest n_vec).
 *   Every GPU that loads the library holds it until the process exits.  A call
 *   with rank > 64 (or n_vec > 8) is rejected with HQ_ERR_SHAPE before any
 *   launch.  The call itself allocates nothing: no cudaMalloc, no cudaFree, no
 *   allocating library routine.
 *   Set-up: the library's first call on a device (this entry point or any
 *   other) looks up the scratch's device address with that device current.
 *   Make that first call before any stream capture.
 *   Sharing: every call on a device uses the same array, and nothing in it
 *   needs to start at zero (each call writes all of u before reading it).
 *   Calls of this entry point that overlap on the GPU (on different streams of
 *   one device) race on the array.  Calls on one stream are ordered and safe.
 * Arguments, validation, accuracy and kernels are those of hq_matvec_q8_0_lora.
 * Source: the paper has no counterpart (an allocation-free form of this
 * library's own QLoRA call).
 */
hq_status hq_matvec_q8_0_lora_noalloc(const void *W, const float *x, const uint16_t *lora_A,
                                      const uint16_t *lora_B, float scale, int rank, float *y,
                                      int64_t rows, int64_t cols, int n_vec, hq_stream_t stream);

/*
 * hq_matvec_i8_requant -- per-output-channel int8 GEMV with gemmlowp requant:
 *   acc = sum_j W[o][j] * x[v][j]  (int32; the caller keeps it in range:
 *         |W|, |x| <= 127 and cols < 133,000 always fit),
 *   y[v][o] = clamp(RDivByPOT(SRDHM(acc, mult[o]), shift[o]), -128, 127).
 *   W     : int8 [rows][cols], 16-byte aligned.   x : int8 [n_vec][cols], 16-byte aligned.
 *   mult  : int32 [rows] (any value).             shift : int32 [rows], each in [0, 31].
 *   y     : int8 [n_vec][rows].
 * SRDHM(a,b) is the high word of 2ab rounded to nearest (ties toward +inf),
 * saturating only at a = b = INT32_MIN; RDivByPOT(x,e) is x/2^e rounded to
 * nearest with ties away from zero.  Bit-exact.  A shift outside [0,31] is a
 * precondition violation (the kernel clamps it to that range).
 * Source: "Blue -- porting zen-nano ...", section "Quantization recipe
 * (validated)" and section "Gaps vs the current toy engine", item 3.
 */
hq_status hq_matvec_i8_requant(const int8_t *W, const int8_t *x,
                               const int32_t *mult, const int32_t *shift, int8_t *y,
                               int64_t rows, int64_t cols, int n_vec, hq_stream_t stream);

/*
 * hq_moe_matvec_q8_0 -- expert-indexed, grouped Q8_0 matvec for MoE decode.
 *   W_bank     : n_experts Q8_0 matrices of rows x cols, back to back
 *                (expert e starts at byte e*rows*cols/32*34), 16-byte aligned.
 *   expert_ids : int32 [n_vec][n_active], each in [0, n_experts).
 *   x          : fp32 [n_vec][cols] when x_per_slot == 0 (all slots of token t
 *                share x[t], as for gate/up), or [n_vec][n_active][cols] when
 *                x_per_slot == 1 (one input per slot, as for down).
 *   y          : fp32 [n_vec][n_active][rows]; y[t][k] = W_bank[ids[t][k]] . x(t,k).
 * Accuracy and the |x| < 2^100 precondition as for hq_matvec_q8_0.
 * Slots that pick the same expert are grouped so that each chosen expert's
 * bytes are streamed once per call.  No router weighting is applied (the
 * _combine variant below applies it).  An id
 * outside [0, n_experts) is a precondition violation: its outputs are set to
 * NaN and the device fault word gets HQ_FAULT_EXPERT_ID; nothing traps.
 * Source: "One Native Stack ...", section "The Unified Quant Core" (the MoE
 * path dispatches each routed expert through the same core); "Economical
 * Serving ...", subsection "The Roofline that Sets the Price" (MoE reads
 * only its active parameters).
 */
hq_status hq_moe_matvec_q8_0(const void *W_bank, const int32_t *expert_ids,
                             const float *x, int x_per_slot, float *y,
                             int64_t n_experts, int n_active, int64_t rows, int64_t cols,
                             int n_vec, hq_stream_t stream);

/*
 * hq_moe_matvec_q8_0_swiglu -- the grouped MoE matvec of an expert bank whose
 * gate and up matrices are stored as one matrix with their rows interleaved
 * (row 2i = gate row i, row 2i+1 = up row i; rows = 2 * intermediate, even),
 * with the SwiGLU gate applied as the outputs are stored:
 *   h[t][k][i] = silu(g) * u,  g = row 2i . x(t,k),  u = row 2i+1 . x(t,k),
 *   silu(z) = z / (1 + e^-z).
 *   h : fp32 [n_vec][n_active][rows / 2], 4-byte aligned; it is the x of the
 *       down projection (x_per_slot = 1).
 * Other arguments, grouping and the invalid-id behaviour (NaN outputs, fault
 * word) as for hq_moe_matvec_q8_0.  Accuracy: g and u are each within the
 * matvec tolerance e = 1e-3 * sum_j |w_deq * x| + 1e-5 of their exact values;
 * h is then within 1.1 * e_g * (|u| + e_u) + |silu(g)| * e_u, plus fp32
 * rounding, of silu(g) * u.
 * Source: "Blue -- porting zen-nano ...", section "Architecture" (each
 * layer's feed-forward is SwiGLU(gate, up, down)); the silu gate and the
 * row interleave are this library's readings.
 */
hq_status hq_moe_matvec_q8_0_swiglu(const void *W_bank, const int32_t *expert_ids, const float *x,
                                    int x_per_slot, float *h, int64_t n_experts, int n_active,
                                    int64_t rows, int64_t cols, int n_vec, hq_stream_t stream);

/*
 * hq_moe_matvec_q8_0_combine -- the grouped MoE matvec with the router-weighted
 * sum over each token's slots applied in the same launch:
 *   y[t][i] = sum_k router_w[t][k] * (W_bank[ids[t][k]] . x(t,k))[i].
 *   router_w : fp32 [n_vec][n_active], the router's weights for the chosen
 *              experts (the router itself is the caller's), 4-byte aligned.
 *   y        : fp32 [n_vec][rows], 4-byte aligned.
 * A cluster of up to 8 CTAs (as many as one wave of the grid allows) owns
 * each 32-row tile and splits the tile's expert groups among its CTAs; each
 * CTA keeps its weighted per-token sums in shared memory and the cluster's
 * leader adds them over distributed shared memory.  No atomics and no workspace; the summation order is fixed, so y
 * is the same bits on every run.  A token with an invalid expert id gets
 * NaN rows (and the fault word HQ_FAULT_EXPERT_ID).  Accuracy: |y - y_ref|
 * <= 1e-3 * sum_k |router_w[t][k]| * sum_j |w_deq * x| + 1e-5.  Other
 * arguments as for hq_moe_matvec_q8_0.
 * Source: "Economical Serving ...", paragraph "MoE is the cheapest-per-quality
 * tier" (a sparsely gated mixture: the output is the gate-weighted sum of the
 * chosen experts' outputs).
 */
hq_status hq_moe_matvec_q8_0_combine(const void *W_bank, const int32_t *expert_ids, const float *x,
                                     int x_per_slot, const float *router_w, float *y, int64_t n_experts,
                                     int n_active, int64_t rows, int64_t cols, int n_vec, hq_stream_t stream);

/*
 * hq_moe_matvec_q8_0_ex -- the three MoE calls above in one entry point, with
 * flags.
 *   epilogue : HQ_MOE_EPI_NONE (as hq_moe_matvec_q8_0; router_w unused),
 *              HQ_MOE_EPI_SWIGLU (as hq_moe_matvec_q8_0_swiglu) or
 *              HQ_MOE_EPI_COMBINE (as hq_moe_matvec_q8_0_combine).
 *   flags    : 0, or HQ_MOE_IDS_READY: the caller guarantees that expert_ids
 *              were written by work that completed before the kernel that
 *              precedes this call in the stream -- e.g. the down projection of
 *              an MoE feed-forward, whose ids the router wrote before the
 *              gate|up launch.  The kernel then reads the ids and starts its
 *              weight copies while that kernel is still running, waiting for
 *              it only before it reads x or writes y.  Ids written by the
 *              immediately preceding kernel break the guarantee (the kernel
 *              may read stale ids).
 * All other arguments, results and errors as for the calls above; unknown
 * epilogues or flags give HQ_ERR_UNSUPPORTED.
 * Source: as hq_moe_matvec_q8_0 ("One Native Stack ...", section "The
 * Unified Quant Core": every routed expert through the same core; "Economical
 * Serving ...", subsection "The Roofline that Sets the Price").
 */
#define HQ_MOE_EPI_NONE 0
#define HQ_MOE_EPI_SWIGLU 1
#define HQ_MOE_EPI_COMBINE 2
#define HQ_MOE_IDS_READY 1
hq_status hq_moe_matvec_q8_0_ex(const void *W_bank, const int32_t *expert_ids, const float *x, int x_per_slot,
                                const float *router_w, float *y, int64_t n_experts, int n_active, int64_t rows,
                                int64_t cols, int n_vec, int epilogue, int flags, hq_stream_t stream);

/*
 * Quantizers (the one-off data-preparation step, on the GPU).
 * hq_quantize_q8_0: W fp32 [rows][cols] (device) -> out Q8_0 blocks (device):
 *   d = max|w|/127 in fp32, stored fp16 (round to nearest even);
 *   q = round(w/d) (fp32 division, half away from zero), clamped to [-127,127];
 *   an all-zero block stores d = 0 and q = 0.
 * hq_quantize_q4_0: d = m/-8 with m the block's largest-|w| element (first
 *   on ties, sign kept), stored fp16; n = min(15, floor(w/d + 8.5)) (fp32);
 *   an all-zero block stores d = -0 and n = 8.
 * hq_quantize_i8_rows: scale[o] = max|W[o,:]|/127 (fp32),
 *   Wq = round(W/scale) clamped to [-127,127]; with rows = 1 this is the
 *   static per-tensor activation quantizer.
 * Requires rows >= 1 and cols % 32 == 0 (i8: cols >= 1).  Alignment: Q8_0 and
 * Q4_0 take W 16-byte aligned and out 2-byte aligned; the int8 quantizer takes
 * W and scale 4-byte aligned.  HQ_ERR_ALIGN otherwise.
 * Source: "One Native Stack ...", section "The Unified Quant Core" (formats
 * taken verbatim from ggml); "Blue -- porting zen-nano ...", section
 * "Quantization recipe (validated)".
 */
hq_status hq_quantize_q8_0(const float *W, void *out, int64_t rows, int64_t cols,
                           hq_stream_t stream);
hq_status hq_quantize_q4_0(const float *W, void *out, int64_t rows, int64_t cols,
                           hq_stream_t stream);
hq_status hq_quantize_i8_rows(const float *W, int8_t *Wq, float *scale,
                              int64_t rows, int64_t cols, hq_stream_t stream);
/*
 * hq_quantize_q4_k -- fp32 W [rows][cols] (4-byte aligned) to Q4_K
 * super-blocks in out (rows x cols/256 x 144 B, 16-byte aligned), cols % 256
 * == 0.  The pages give no encoder; this one is a plain min/max reading, per
 * sub-block of 32: mn = min(0, min w), scale = (max w - mn)/15, min = -mn;
 * d = (largest scale)/63 and dmin = (largest min)/63 stored fp16 (RNE);
 * sc = round(scale * 63/largest scale), m likewise (at most 63); then with
 * a = d*sc and b = dmin*m from the stored values, q = round((w + b)/a)
 * clamped to [0, 15] (0 when a == 0).  All in fp32, half away from zero.
 * Source: "One Native Stack ...", section "Ported Versus Novel" (ggml's Q4_K).
 */
hq_status hq_quantize_q4_k(const float *W, void *out, int64_t rows, int64_t cols, hq_stream_t stream);

/*
 * hq_requant_params -- HOST function: real multipliers M[i] in (0, 1) to
 * (mult, shift) with M ~= mult * 2^-31 * 2^-shift: M = f * 2^-shift with
 * f in [0.5, 1), mult = round(f * 2^31) (half away from zero; 2^31 becomes
 * 2^30 with shift - 1).  M, mult, shift are HOST arrays of n elements.
 * Returns HQ_ERR_UNSUPPORTED if some M is outside (0,1) or needs shift > 31.
 * Source: "Blue -- porting zen-nano ...", section "Quantization recipe
 * (validated)" (the requant multiplier s_a*s_w[o]/s_out as an integer pair).
 */
hq_status hq_requant_params(const double *M, int64_t n, int32_t *mult, int32_t *shift);

/*
 * hq_requant_i32_debug -- applies the device requant epilogue of
 * hq_matvec_i8_requant to arbitrary int32 accumulators, so that values the
 * GEMV cannot reach (INT32_MIN, INT32_MAX) are tested bit-exactly:
 * y[i] = requant(acc[i], mult[i % rows], shift[i % rows]).  Device pointers;
 * acc, y have n elements, mult, shift have rows elements.
 * Source: as hq_matvec_i8_requant.
 */
hq_status hq_requant_i32_debug(const int32_t *acc, const int32_t *mult, const int32_t *shift,
                               int8_t *y, int64_t n, int64_t rows, hq_stream_t stream);

/*
 * Device fault word.  Kernels never trap: a bounded wait that gives up (a
 * TMA transfer that never completes) or an out-of-range expert id sets a bit
 * in a per-device word and the kernel finishes without using the missing
 * data.  hq_device_fault() synchronizes the current device, returns the word
 * in *fault (0 = none) and clears it; it returns HQ_ERR_DEVICE if the word
 * was non-zero.  Bits 0..7 are the HQ_FAULT_* flags; when the first fault of
 * the word was a timeout, bits 9..31 hold the index of the CTA that gave up
 * and bit 8 is set if the waiter was a consumer warp (clear: the producer).
 */
#define HQ_FAULT_WAIT_TIMEOUT 1u   /* an mbarrier wait exceeded its time limit */
#define HQ_FAULT_EXPERT_ID    2u   /* an expert id outside [0, n_experts)      */
hq_status hq_device_fault(uint32_t *fault);

/*
 * hq_selftest_wait_timeout -- test-only exercise of the failure path: one CTA
 * of one warp waits on an mbarrier that nothing arrives on, with the matvec
 * kernels' bounded wait but a limit of `cycles` SM clock cycles
 * (1 <= cycles <= 4e9).  The wait gives up, sets HQ_FAULT_WAIT_TIMEOUT in the
 * fault word with CTA 0 and the consumer bit recorded, and the kernel returns:
 * nothing faults, traps or hangs, and the context stays usable.  Read the
 * result with hq_device_fault().
 * Source: none on the pages (a property of this implementation's waits).
 */
hq_status hq_selftest_wait_timeout(int64_t cycles, hq_stream_t stream);

/*
 * hq_launch_count -- the number of kernels the library has launched (or
 * recorded into a stream capture) in this process, on every device: a
 * monotone host-side counter for callers that account for launches.
 * Source: none on the pages (introspection of this implementation).
 */
uint64_t hq_launch_count(void);

/*
 * hq_debug_plan -- test-only: the launch geometry the library would choose for
 * a dense matvec of `rows` x `cols` at `n_vec` vectors, on a device with
 * `num_sms` SMs and `smem_optin` bytes of opt-in shared memory per CTA, for a
 * kernel of `regs` registers per thread.  Pure host arithmetic: no device is
 * touched, so it also runs on a machine without a GPU.
 *   fmt : 8 (Q8_0), 4 (Q4_0), 75 (Q4_K) or 1 (int8).  cols : a multiple of 256 (int8:
 *         128), the shapes the TMA-staged kernel serves.
 *   out : int64 [out_len >= HQ_PLAN_FIELDS], caller-owned host memory,
 *         filled with { policy (0 one owner per stage, 1 Q8_0 short rows,
 *         4 column-split stages; 2 and 3 are not used),
 *         consumer warps per CTA,
 *         rows per tile, grid (CTAs), K split (CTAs per cluster), ring stages,
 *         dynamic shared memory bytes, CTAs per SM of the launch bound,
 *         CTA slots (SMs x CTAs per SM the plan assumed), row tiles }.
 * Errors: HQ_ERR_NULL, HQ_ERR_SHAPE, HQ_ERR_NVEC, HQ_ERR_UNSUPPORTED (fmt).
 * Source: none on the pages (introspection of this implementation).
 */
#define HQ_PLAN_FIELDS 10
hq_status hq_debug_plan(int fmt, int n_vec, int64_t rows, int64_t cols, int num_sms, int smem_optin, int regs,
                        int64_t *out, int out_len);

#ifdef __cplusplus
}
#endif

#endif /* HQ_H_ */
