/*
 * attn.h - C ABI of the GB300 (sm_103a) fused attention library
 * (libattn_sm103.so): the forward pass, and its backward pass (attn_bwd).
 *
 * The operation (one call = one whole forward pass over every (b, h)):
 *
 *     S   = scale * Q K^T           (per head; K^T is the transpose of K)
 *     S   = -inf where key j > query i           (only when causal != 0)
 *     O   = softmax_rows(S) V
 *     LSE = log(sum_j exp(S_ij))    (natural log, per query row)
 *
 * computed block by block with the online softmax (running row max and row
 * sum, rescale of the partial output when the max grows, division by the
 * sum at the end) under a producer/consumer warp-specialised schedule.
 * Source: "Warp specialization" concept card (wikillm), sections
 * "Implementation sketch" (the consumer loop and its return value: output /
 * row_sum and row_max + log(row_sum)) and "Variants" (producer/consumer
 * roles, pingpong of two consumers); "Inside FlashAttention-3 &
 * Warp-Specialized CUDA Kernels" (tekromancy), sections 2 and 4 (TMA ring
 * with mbarriers, tcgen05.mma into Tensor Memory).  The pages leave the
 * scale, the mask convention and the layout open; this library takes:
 *   - scale multiplies Q K^T before the mask, the max and the exponential,
 *     so LSE is in units of the scaled scores;
 *   - causal: key j is visible to query i iff j <= i (square, top-left);
 *   - layout below.
 *
 * Layout.  Q, K, V and O are dense row-major [B, H, N, d] tensors (d
 * fastest), all with the same N (self-attention shape).  LSE is a dense
 * [B, H, N] fp32 tensor.  O has the input element type, except for e4m3
 * inputs, whose O is bf16.
 *
 * Memory.  Every pointer is a DEVICE pointer on the current CUDA device,
 * owned by the caller.  The library allocates and frees nothing and keeps
 * no state between calls apart from one device-side watchdog word per
 * device (see attn_fwd_status).  Inputs are only read; O and LSE are only
 * written, every element once.
 *
 * Asynchrony.  Calls enqueue one kernel on `stream` (NULL = the legacy
 * default stream) and return; results are valid once the stream has
 * synchronised.  Calls on different streams may run concurrently.
 *
 * Errors.  Every argument check runs before anything is enqueued; a call
 * that fails a check returns a nonzero attn_status_t and has no side
 * effects.  A failed kernel launch returns ATTN_ERR_CUDA.
 */
#ifndef WS_ATTN_H_
#define WS_ATTN_H_

#ifdef __cplusplus
extern "C" {
#endif

/* The CUDA runtime's stream type (cudaStream_t is a pointer to this). */
struct CUstream_st;

typedef enum {
    ATTN_FP32 = 0,      /* fp32 in, fp32 out, exact fp32 arithmetic (CUDA cores) */
    ATTN_FP16 = 1,      /* fp16 in, fp16 out, fp32 accumulation */
    ATTN_BF16 = 2,      /* bf16 in, bf16 out, fp32 accumulation */
    ATTN_FP8_E4M3 = 3   /* e4m3 in (descales 1.0 through attn_fwd), bf16 out */
} attn_dtype_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,   /* null pointer, size out of range, bad scale/causal/dtype */
    ATTN_ERR_UNSUPPORTED = 2,   /* head dim not built for this dtype, or kernel not runnable */
    ATTN_ERR_MISALIGNED = 3,    /* q/k/v/o not 16-byte aligned, or lse not 4-byte aligned */
    ATTN_ERR_DEVICE = 4,        /* no CUDA device, or the current device is not sm_103 */
    ATTN_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed */
    ATTN_ERR_TIMEOUT = 6        /* a device-side wait exceeded its limit (see attn_fwd_status) */
} attn_status_t;

/*
 * attn_fwd - one forward pass.
 *   q, k, v : [B, H, N, d] device tensors of `dtype`, 16-byte aligned.
 *   o       : [B, H, N, d] device output (dtype; bf16 for ATTN_FP8_E4M3),
 *             16-byte aligned.
 *   lse     : [B, H, N] fp32 device output, 4-byte aligned.
 *   B, H    : >= 1, B*H <= 2^24.
 *   N       : 1 <= N <= 2^24 and B*H*N <= 2^31 - 1; a final partial block
 *             of 128 keys is masked.
 *   d       : 64, 128 or 256 for fp16/bf16; 64 or 128 for fp32 and 128
 *             for e4m3.
 *   scale   : finite and > 0 (usually 1/sqrt(d)).
 *   causal  : 0 or 1.
 *   dtype   : an attn_dtype_t.
 * Returns ATTN_OK or an attn_status_t error code.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             int B, int H, int N, int d, float scale, int causal, int dtype,
             struct CUstream_st* stream);

/*
 * attn_fwd_workspace_size - bytes of device workspace attn_fwd_ws and
 * attn_fwd_fp8_ws need for head dim d and `dtype` on the current device
 * (it depends on the device's SM count, not on B, H or N); 0 where the
 * call never splits (ATTN_FP32, and d = 256, whose kernel runs whole items
 * only) or for an invalid d, dtype or device.
 */
unsigned long long attn_fwd_workspace_size(int d, int dtype);

/*
 * attn_fwd_split_advised - 1 when attn_fwd_ws's split of the leftover work
 * is expected to finish sooner than attn_fwd's whole rounds for this shape
 * on the current device, else 0; also 0 for invalid arguments.  The split
 * is advised only where the problem is a single partial round (fewer work
 * items than SMs) and its longest item is longer than a tail CTA's share
 * plus the split's own cost, both counted in key blocks.  Launches nothing.
 */
int attn_fwd_split_advised(int B, int H, int N, int d, int causal, int dtype);

/*
 * attn_fwd_ws - attn_fwd with a caller workspace, which lets the work that
 * is left over after whole rounds of one (b, h, query tile pair) item per
 * SM be split along the key axis: a second launch gives every CTA an
 * equal share of the leftover items' key blocks, and the partial results
 * of one query tile are merged with the exact rescaling of the online
 * softmax (each piece keeps its unnormalised O, row maximum m and row sum
 * l; the merge takes M = max m, weights exp2(m - M), and divides once).
 * That merge is the running-maximum rescaling of the "Warp specialization"
 * concept card, Implementation sketch (the consumer's update of the
 * running max, the rescale factor and the sum), applied across pieces
 * instead of across key blocks.  O and LSE are those of attn_fwd up to
 * floating-point reassociation of the row sums.
 *   workspace       : device memory, 256-byte aligned, at least
 *                     attn_fwd_workspace_size(d, dtype) bytes, owned by the
 *                     caller; its contents need no initialisation and are
 *                     scratch after the call.  One call at a time may use a
 *                     given workspace (calls on one stream are ordered).
 *   workspace_bytes : its size.
 * Other arguments and errors as attn_fwd; a null or short workspace is
 * ATTN_ERR_INVALID_ARG, a misaligned one ATTN_ERR_MISALIGNED.  Enqueues up
 * to two kernels (and a memset when no whole round exists).  ATTN_FP32
 * ignores the workspace.
 */
int attn_fwd_ws(const void* q, const void* k, const void* v, void* o, float* lse,
                int B, int H, int N, int d, float scale, int causal, int dtype,
                void* workspace, unsigned long long workspace_bytes,
                struct CUstream_st* stream);

/*
 * attn_fwd_fp8 - forward pass on e4m3 inputs quantised with per-tensor
 * scales: the real values are code * descale.  q_descale * k_descale is
 * folded into the softmax scale and v_descale is applied to O before the
 * bf16 rounding.  The probabilities are re-quantised to e4m3 (scale 1)
 * for the P.V product; the row sum uses them before that rounding.
 * Source: "Inside FlashAttention-3 & Warp-Specialized CUDA Kernels",
 * section 5 (FP8 E4M3 forward; per-tensor
 * scaling).  Arguments as attn_fwd with dtype ATTN_FP8_E4M3 (d = 128); the
 * descales must be finite and > 0.
 */
int attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int N, int d, float scale, int causal,
                 float q_descale, float k_descale, float v_descale,
                 struct CUstream_st* stream);

/*
 * attn_fwd_fp8_ws - attn_fwd_fp8 with the caller workspace of attn_fwd_ws
 * (same split of the leftover work, same workspace rules).
 */
int attn_fwd_fp8_ws(const void* q, const void* k, const void* v, void* o, float* lse,
                    int B, int H, int N, int d, float scale, int causal,
                    float q_descale, float k_descale, float v_descale,
                    void* workspace, unsigned long long workspace_bytes,
                    struct CUstream_st* stream);

/* Options of attn_fwd_opt and attn_fwd_fp8_opt (bitwise OR). */
#define ATTN_OPT_EXP2_FMA 1u

/*
 * attn_fwd_opt - attn_fwd with options.
 *   ATTN_OPT_EXP2_FMA : 4 of every 32 softmax exponentials are computed on
 *     the FMA pipe instead of the MUFU unit: x = n + f with n = round(x)
 *     (Cody and Waite's reduction), 2^f by a degree-3 polynomial fitted
 *     for the least largest relative error on [-1/2, 1/2] (7.5e-5 at most),
 *     n added to the exponent; x < -126 gives 0.  The exponential unit is
 *     the gap the "Inside FlashAttention-3 & Warp-Specialized CUDA Kernels"
 *     page names in its introduction (MUFU.EX2 throughput against the
 *     tensor cores); moving part of its work to the FMA pipe is this
 *     library's own measure, off by default because it measured slower on
 *     GB300 (the MUFU unit is not what bounds these kernels).  Built for
 *     ATTN_BF16 with d = 64 or 128 and ATTN_FP8_E4M3 with d = 128; other
 *     dtypes and head dims return ATTN_ERR_UNSUPPORTED.  No split of the
 *     leftover work (no workspace).
 *   opts = 0 is attn_fwd.  Unknown option bits are ATTN_ERR_INVALID_ARG.
 * Other arguments, results and errors as attn_fwd.
 */
int attn_fwd_opt(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int N, int d, float scale, int causal, int dtype,
                 unsigned int opts, struct CUstream_st* stream);

/*
 * attn_fwd_fp8_opt - attn_fwd_fp8 with the options of attn_fwd_opt
 * (ATTN_OPT_EXP2_FMA is built for d = 128).
 */
int attn_fwd_fp8_opt(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int H, int N, int d, float scale, int causal,
                     float q_descale, float k_descale, float v_descale,
                     unsigned int opts, struct CUstream_st* stream);

/*
 * attn_fwd_fp8_blockscaled - forward pass on e4m3 Q and K that carry one
 * fp32 scale per 128-row tile of each (b, h) (the real value of a row in
 * tile t is code * scale[bh][t]), as attn_quantize_fp8 produces them, and
 * e4m3 V with one per-tensor descale.  Per key block the softmax uses
 * scale * q_scale[tile] * k_scale[block]; everything else is attn_fwd_fp8.
 * Source: "Inside FlashAttention-3 & Warp-Specialized CUDA Kernels",
 * section 5 (block quantisation of FP8 attention
 * inputs).  q_scales and k_scales: device arrays [B * H, ceil(N / 128)],
 * 4-byte aligned, finite and > 0.  Other arguments as attn_fwd_fp8.
 */
int attn_fwd_fp8_blockscaled(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int H, int N, int d, float scale, int causal,
                             const float* q_scales, const float* k_scales, float v_descale,
                             struct CUstream_st* stream);

/*
 * attn_quantize_fp8 - e4m3 block quantisation of a [B, H, N, d] tensor (Q
 * or K), optionally after the 16 x 16 Walsh-Hadamard rotation of each group
 * of 16 consecutive channels.  The rotation H is orthonormal and symmetric,
 * so rotating both Q and K keeps Q K^T while spreading outlier channels
 * ("Inside FlashAttention-3 & Warp-Specialized CUDA Kernels", section 5).
 * Per 128-row tile of each (b, h): scale =
 * max|value| / 448 (1 for an all-zero tile), code = e4m3(value / scale):
 * the quotient correctly rounded to fp32, then rounded to e4m3 nearest
 * even, saturating at +-448.  The butterfly runs h = 1, 2, 4, 8 over pairs
 * (i, i + h) as (a + b, a - b) in fp32, then multiplies by 1/4.
 *   x      : input, dtype ATTN_FP32 / ATTN_FP16 / ATTN_BF16, 16-byte aligned.
 *   codes  : [B, H, N, d] e4m3 output, 16-byte aligned.
 *   scales : [B * H, ceil(N / 128)] fp32 output, 4-byte aligned.
 *   d      : 64 or 128.  hadamard: 0 or 1.
 * One kernel on `stream`; errors as attn_fwd.
 */
int attn_quantize_fp8(const void* x, void* codes, float* scales, int B, int H, int N, int d,
                      int dtype, int hadamard, struct CUstream_st* stream);

/*
 * attn_fwd_status - synchronises `stream`, then reports and clears the
 * device watchdog word of the current device.  Every wait inside the
 * kernels is bounded (about two seconds); a wait that runs out records
 * ATTN_ERR_TIMEOUT there and the kernel ends without writing the rest of
 * its outputs.  Returns ATTN_OK, ATTN_ERR_TIMEOUT, or ATTN_ERR_CUDA if
 * the synchronisation itself reports an error.
 */
int attn_fwd_status(struct CUstream_st* stream);

/*
 * attn_bwd_workspace_size - bytes of device workspace attn_bwd needs for
 * this shape: 8 bytes per query row, rows rounded up to whole 128-row tiles
 * per head (B * H * ceil(N / 128) * 128 * 8).  0 if a size is < 1.
 */
unsigned long long attn_bwd_workspace_size(int B, int H, int N);

/*
 * attn_bwd - backward pass: the gradients of the forward pass of attn_fwd
 * for an output gradient dO, using the forward's O and LSE:
 *     P_ij  = exp(scale q_i.k_j - LSE_i)   (0 where masked)
 *     D_i   = dO_i . O_i
 *     dS_ij = P_ij (dO_i . v_j - D_i)
 *     dV_j  = sum_i P_ij dO_i
 *     dQ_i  = scale sum_j dS_ij k_j
 *     dK_j  = scale sum_i dS_ij q_i
 * The LSE the forward returns (natural log, "Warp specialization" concept
 * card, section "Implementation sketch": row_max + log(row_sum)) is what
 * lets each block recompute its probabilities without a running max.
 *   q, k, v, o, dout : [B, H, N, d] device tensors of `dtype`, 16-byte aligned
 *                      (o and lse as returned by attn_fwd for these q, k, v,
 *                      scale and causal).
 *   lse              : [B, H, N] fp32, 4-byte aligned.
 *   dq, dk, dv       : [B, H, N, d] device outputs of `dtype`, 16-byte
 *                      aligned, every element written once.
 *   workspace        : device scratch of at least attn_bwd_workspace_size()
 *                      bytes, 16-byte aligned, owned by the caller; its
 *                      contents on entry do not matter and on return are
 *                      unspecified.  Calls that share a workspace must not
 *                      overlap on the device.
 *   dtype            : ATTN_FP16 or ATTN_BF16; d : 64 or 128; other
 *                      arguments as attn_fwd.
 * Three kernels are enqueued on `stream`.  Errors as attn_fwd, plus
 * ATTN_ERR_INVALID_ARG for a workspace that is missing or too small.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
             const float* lse, void* dq, void* dk, void* dv, void* workspace,
             unsigned long long workspace_bytes, int B, int H, int N, int d, float scale,
             int causal, int dtype, struct CUstream_st* stream);

/*
 * attn_bwd_noalloc - attn_bwd for callers that cannot allocate device
 * memory at call time (a program whose device memory all belongs to its own
 * pool, a plugin whose host framework owns every allocation, a step that
 * must not risk an allocation's latency or failure).  It takes no workspace:
 * the library keeps one 8 MiB array in device global memory for it, created
 * when the library is loaded on a device and held until the process exits.
 * The pages describe no counterpart; this is a deployment variant of
 * attn_bwd, with the same results.
 *   Limit: B * H * ceil(N / 128) * 128 <= 1,048,576 query rows; larger
 *   shapes return ATTN_ERR_INVALID_ARG without touching the device.
 *   The first call on a device looks up the array's device address (with
 *   that device current) and caches it; make that first call before any
 *   stream capture.  It allocates and frees nothing, here or later.
 *   All calls on a device share the one array, which keeps whatever the
 *   last call left in it (nothing in it needs to start zeroed).  Calls whose
 *   kernels overlap on the device race on it: issue them on one stream or
 *   order them.
 * Other arguments, errors and asynchrony as attn_bwd.
 */
int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                     float scale, int causal, int dtype, struct CUstream_st* stream);

/* attn_status_string - a static, human-readable name for a status code. */
const char* attn_status_string(int status);

/*
 * attn_watchdog_selftest - checks the watchdog path itself on the device:
 * launches one CTA that waits on an mbarrier nobody arrives on, with a
 * limit of `timeout_us` microseconds (1 .. 10^7).  The wait runs out, the
 * kernel records ATTN_ERR_TIMEOUT in the watchdog word and returns.  This
 * call then synchronises `stream` and returns what attn_fwd_status would
 * (ATTN_ERR_TIMEOUT when the watchdog works), clearing the word.  Not part
 * of the attention computation; it exists so the bounded-wait mechanism
 * can be tested without a real fault.
 */
int attn_watchdog_selftest(unsigned int timeout_us, struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif

#endif /* WS_ATTN_H_ */
