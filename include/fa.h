/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention library (libfa_gb300.so).
 *
 * The library computes exact scaled-dot-product attention
 *     S = scale * Q K^T  (S_ij = -inf for j > i when causal),
 *     P = softmax(S) row by row,  O = P V,
 * tiled so that S and P never reach device memory, and its gradient.  The
 * definitions follow "FLASH-ATTN" (taking-lying-flat), FlashAttention-2 >
 * Background (standard attention and its backward chain) and
 * FlashAttention-2 > FlashAttention-2 (online softmax with an unscaled output
 * accumulator, the LogSumExp statistic L = m + log(l), the causal mask and the
 * skip of fully masked blocks).  The pages write S = QK^T; the softmax scale
 * is this interface's explicit `scale` argument.
 *
 * Common conventions for every entry point
 *  - Tensors are dense, contiguous, row-major [B, H, N, d] (batch, head,
 *    sequence, head dimension); the statistics L and D are [B, H, N] fp32.
 *    Element types: bf16 for Q, K, V, O, dO, dQ, dK, dV; e4m3 bytes for the
 *    FP8 inputs.
 *  - All tensor pointers are DEVICE pointers owned by the caller; every
 *    pointer must be 16-byte aligned.  The library never allocates or frees
 *    memory, never synchronises the stream (fa_device_error excepted) and
 *    keeps no state between calls except a once-resolved driver entry point
 *    and a device error word per kernel family.
 *  - `stream` is a cudaStream_t passed as void*; NULL means the legacy
 *    default stream.  Launches are asynchronous on that stream.
 *  - CUDA graphs: the compute entry points only enqueue asynchronous work on
 *    `stream` (kernels, some launched with programmatic stream serialization,
 *    and memsets), so a call can be captured into a graph and replayed; the
 *    captured launches keep that call's pointers, sizes and scale.  Make the
 *    first call of each entry point outside a capture (it sets kernel
 *    attributes and loads modules).  fa_device_error, fa_measure_ex2_rate and
 *    the first fa_bwd_noalloc call on a device synchronise and cannot be
 *    captured.
 *  - Supported shapes: B, H, N >= 1, d in {64, 128}; B * H <= 2^31 / N.
 *    Rows past N in the last tile of a head are handled inside the kernels
 *    (loads past the end read zeros; masked keys get weight 0; nothing is
 *    stored past row N - 1).
 *  - scale must be finite and > 0 (usually 1/sqrt(d)).
 *  - Return value: FA_OK, or the first argument / launch error found; on an
 *    error nothing has been launched by that call, except FA_ERR_LAUNCH which
 *    reports a failed launch.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null pointer, B/H/N <= 0, bad scale, size overflow */
  FA_ERR_UNSUPPORTED = 2, /* d not in {64, 128}, or no sm_103 device current    */
  FA_ERR_ALIGNMENT = 3,   /* a tensor pointer not 16-byte aligned                */
  FA_ERR_LAUNCH = 4,      /* a kernel launch or tensor-map encoding failed       */
  FA_ERR_TIMEOUT = 5,     /* a kernel's bounded wait ran out (fa_device_error)   */
  FA_ERR_WORKSPACE = 6,   /* workspace missing or smaller than required          */
  FA_ERR_KERNEL_CONFIG = 7 /* the compiled kernel does not match the launch plan:
                              its register count differs from the one its
                              per-warpgroup register split assumes (a toolchain
                              change); nothing was launched                      */
} fa_status;

/*
 * Forward pass ("FLASH-ATTN", FlashAttention-2 > FlashAttention-2).
 *   q, k, v : [B,H,N,d] bf16, read only.
 *   o       : [B,H,N,d] bf16, written: O = softmax(scale*QK^T [+mask]) V.
 *   lse     : [B,H,N] fp32, written: L_i = ln sum_j exp(scale * q_i.k_j) over
 *             the unmasked keys (natural-log units of the scaled logits).
 *   causal  : 0 or 1 (mask S_ij = -inf for j > i, self-attention).
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 int causal, float scale, void* stream);

/*
 * Grouped-query forward ("FLASH-ATTN", FlashAttention-2 > FlashAttention-2,
 * multi-query and grouped-query attention: several query heads share one key
 * head and one value head, addressed by adjusting the head index instead of
 * copying K and V).  As fa_fwd, with
 *   q, o : [B,H,N,d] bf16;  k, v : [B,Hkv,N,d] bf16;  lse : [B,H,N] fp32,
 *   Hkv >= 1 dividing H; query head h uses key/value head h / (H / Hkv).
 * fa_fwd(...) is fa_fwd_gqa with Hkv = H.
 */
fa_status fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv, int N,
                     int d, int causal, float scale, void* stream);

/*
 * Bytes of device workspace fa_bwd needs: D ([B,H,N] fp32, 16-byte padded)
 * followed by the fp32 dQ accumulator ([B,H,N,d]).  0 on invalid sizes.
 */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Backward pass ("FLASH-ATTN", FlashAttention-2 > Background: dV = P^T dO,
 * dP = dO V^T, dS = dsoftmax(dP), dQ = dS K, dK = dS^T Q; P rebuilt from L as
 * in FlashAttention > Tiling and Recomputation).  With S = scale*QK^T the
 * gradients w.r.t. Q and K carry the factor `scale`.
 *   q, k, v, o, dO : [B,H,N,d] bf16 read only (o and lse from fa_fwd with the
 *                    same q, k, v, causal, scale).
 *   lse            : [B,H,N] fp32 read only.
 *   dq, dk, dv     : [B,H,N,d] bf16 written.
 *   workspace      : device buffer of at least fa_bwd_workspace_size() bytes;
 *                    contents on entry do not matter; overwritten.
 * Runs fa_bwd_preprocess, fa_bwd_main and fa_bwd_dq_convert on `stream`.
 * dQ is reduced with fp32 atomics, so its low bits may vary run to run.
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                 void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                 int causal, float scale, void* stream);

/*
 * Grouped-query backward (same section: the gradients of a shared key or
 * value head are the sums over the query heads that use it).  As fa_bwd, with
 *   q, o, dO, dq : [B,H,N,d] bf16;  k, v, dk, dv : [B,Hkv,N,d] bf16;
 *   lse : [B,H,N] fp32;  Hkv >= 1 dividing H;
 *   workspace : at least fa_bwd_workspace_size(B, H, N, d) bytes (per query
 *               head); with fa_bwd_gqa_workspace_size(B, H, Hkv, N, d) bytes
 *               the split described below may be used.
 * Each CTA owns one key/value head's block of keys and loops over all query
 * heads of its group, so dK and dV are summed on chip without atomics.  For
 * groups of four query heads or more, or key/value heads too few to fill the
 * GPU, and when the workspace holds fa_bwd_gqa_workspace_size bytes, each
 * CTA takes one query head instead and adds its part of dK and dV into fp32
 * accumulators in the workspace by reduce-adds (their low bits may then vary
 * run to run, as dQ's do), converted to bf16 at the end.
 * fa_bwd(...) is fa_bwd_gqa with Hkv = H.
 */
fa_status fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                     void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int H, int Hkv,
                     int N, int d, int causal, float scale, void* stream);

/*
 * Workspace bytes for fa_bwd_gqa: fa_bwd_workspace_size(B, H, N, d), plus two
 * fp32 [B,Hkv,N,d] accumulators when fa_bwd_gqa would split the query heads of
 * a group over CTAs (groups of four query heads or more, or fewer than two
 * waves of per-key/value-head CTAs).  0 for invalid shapes.  Host only; no GPU
 * needed.
 */
size_t fa_bwd_gqa_workspace_size(int B, int H, int Hkv, int N, int d);

/*
 * Backward step 1: D_i = sum_k dO_ik O_ik (fp32), which equals
 * sum_j P_ij dP_ij, the row term of the softmax Jacobian; also zeroes dq_acc.
 *   o, dO  : [B,H,N,d] bf16.  D: [B,H,N] fp32 out.  dq_acc: [B,H,N,d] fp32 out (zeros).
 */
fa_status fa_bwd_preprocess(const void* o, const void* dO, float* D, float* dq_acc, int B, int H, int N, int d,
                            void* stream);

/*
 * Backward step 2: one CTA per 128-key block of a head, Q blocks inner
 * ("FLASH-ATTN", FlashAttention-2 > Parallelism: the backward pass gives each
 * column block its own thread block and the blocks meet only in atomic adds
 * to dQ).  Writes dK = scale * dS^T Q and dV = P^T dO (bf16) and adds
 * dS K (unscaled, fp32) into dq_acc, which must hold zeros on entry (step 1).
 */
fa_status fa_bwd_main(const void* q, const void* k, const void* v, const float* lse, const void* dO,
                      const float* D, float* dq_acc, void* dk, void* dv, int B, int H, int N, int d, int causal,
                      float scale, void* stream);

/* Backward step 3: dq = bf16(scale * dq_acc), round to nearest even. */
fa_status fa_bwd_dq_convert(const float* dq_acc, void* dq, int B, int H, int N, int d, float scale, void* stream);

/*
 * FP8 forward ("FLASH-ATTN", FlashAttention-3 > Low-precision with FP8:
 * per-tensor scaling keeps one scalar per tensor).
 *   q8, k8, v8 : [B,H,N,d] e4m3 codes (1 byte each), d in {64, 128};
 *                X = delta_X * code.
 *   descale_q, descale_k, descale_v : DEVICE pointers to one fp32 each (delta).
 *   o   : [B,H,N,d] bf16 out, O = softmax(scale * (dq dk) q8 k8^T) (dv v8).
 *   lse : [B,H,N] fp32 out, natural-log LogSumExp of the scaled logits.
 * Inside, P is stored as e4m3 times 2^4 for the second product (the running
 * maximum is raised whenever P would pass 2^4, so P * 2^4 stays at or below
 * 256 < 448); the factor is removed in the final division
 * by the row sum.
 */
fa_status fa_fwd_fp8(const void* q8, const void* k8, const void* v8, const float* descale_q,
                     const float* descale_k, const float* descale_v, void* o, float* lse, int B, int H, int N,
                     int d, int causal, float scale, void* stream);

/*
 * FP8 storage for fa_fwd_fp8 ("FLASH-ATTN", FlashAttention-3 > Low-precision
 * with FP8: one scale per tensor, and incoherent processing -- Q and K are
 * multiplied by an orthogonal matrix before quantisation, which leaves QK^T
 * unchanged and spreads outliers; the matrix is a Hadamard transform as in
 * "FlashAttention 三代演进", 技术 4).
 *   x       : rows x d input, fp32 (x_dtype = 0) or bf16 (x_dtype = 1), device.
 *   hadamard: 1 to rotate each row by H/sqrt(d) (H the Sylvester Hadamard
 *             matrix; use it for Q and K, never for V), 0 to quantise as is.
 *   codes   : rows x d e4m3 codes out (1 byte each), device: e4m3_rne of
 *             y * 448 / max|y| (y as is if all zero), the product rounded
 *             once to fp32 and saturated at +-448.
 *   descale : one fp32 out, device: delta = max|y| / 448 (1 if all zero), so
 *             that y ~= delta * code.
 *   d in {64, 128}; rows >= 1.  Three launches on `stream`; the descale word
 *   holds the running maximum until the last one.
 */
fa_status fa_fp8_quantize(const void* x, int x_dtype, int hadamard, void* codes, float* descale, long long rows,
                          int d, void* stream);

/*
 * Causal attention with a sliding window ("FLASH-ATTN" lists sliding window
 * among the variants the kernels support; the pages do not define it, the
 * reading taken: query i sees keys j with i - window < j <= i, the `window`
 * most recent keys including its own).  Key blocks entirely outside every
 * row's window are skipped, so the work grows with N * window, not N^2.
 *   Arguments, layouts, results and errors as fa_fwd_gqa / fa_bwd_gqa, with
 *   `window` >= 1 in place of `causal` (window >= N is plain causal attention).
 */
fa_status fa_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv,
                        int N, int d, int window, float scale, void* stream);
fa_status fa_bwd_window(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                        void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int H, int Hkv,
                        int N, int d, int window, float scale, void* stream);

/*
 * Block sizes of the block-quantised FP8 path: one scale per 128 rows of Q
 * (the forward's query tile, B_r) and per 64 rows of K and of V (its key
 * block, B_c).
 */
#define FA_FP8_BLOCK_Q 128
#define FA_FP8_BLOCK_KV 64

/*
 * FP8 forward on block-quantised inputs ("FLASH-ATTN", FlashAttention-3 >
 * Low-precision with FP8, block quantisation: Q, K and V are cut into blocks
 * of B_r x d or B_c x d rows quantised each with its own scale; the kernel,
 * which works block by block, scales each block of S by the scales of its Q
 * and K blocks).
 *   q8, k8, v8 : [B,H,N,d] e4m3 codes, d in {64, 128}.
 *   descale_q  : DEVICE [B*H, ceil(N/128)] fp32, the scale of rows
 *                [128 b, 128 b + 128) of each head of Q.
 *   descale_k, descale_v : DEVICE [B*H, ceil(N/64)] fp32, per 64 rows of K
 *                and of V.  All scales positive and finite.
 *   o, lse, B, H, N, causal, scale, stream : as fa_fwd_fp8.
 * S for query block i and key block j is scale * dq_i dk_j q8 k8^T.  V's
 * block scale is applied to P's e4m3 operand relative to the largest V scale
 * of the head (P * 2^4 * dv_j / max dv, never above 448), and O is multiplied
 * by that largest scale at the end.  Where V's block scales differ, small P
 * values lose e4m3 precision; passing one V scale per head (the same value in
 * every block of descale_v) avoids that.
 */
fa_status fa_fwd_fp8_blocks(const void* q8, const void* k8, const void* v8, const float* descale_q,
                            const float* descale_k, const float* descale_v, void* o, float* lse, int B, int H,
                            int N, int d, int causal, float scale, void* stream);

/*
 * Block e4m3 storage for fa_fwd_fp8_blocks (block quantisation of the same
 * section; optional Hadamard rotation as in fa_fp8_quantize).
 *   x          : [seqs, N, d] input, fp32 (x_dtype = 0) or bf16 (x_dtype = 1),
 *                device.
 *   block_rows : rows per block, 1..1024 (FA_FP8_BLOCK_Q for Q,
 *                FA_FP8_BLOCK_KV for K and V); the last block of a sequence
 *                holds the remaining N mod block_rows rows, if any.
 *   codes      : [seqs, N, d] e4m3 codes out, device (rounded as in
 *                fa_fp8_quantize, with each block's own max|y|).
 *   descale    : [seqs, ceil(N / block_rows)] fp32 out, device: per block
 *                delta = max|y| / 448 (1 if the block is all zero).
 *   d in {64, 128}; seqs in 1..65535; N >= 1.  One launch on `stream`.
 */
fa_status fa_fp8_quantize_blocks(const void* x, int x_dtype, int hadamard, int block_rows, void* codes,
                                 float* descale, int seqs, int N, int d, void* stream);

/*
 * Decode: one query row per (batch, head) against a cache of N keys and
 * values -- the step that generates one token ("FlashAttention 三代演进": the
 * decode case is memory-bound, a single query against all keys, and is tiled
 * differently from the forward over whole sequences).  The row is standard
 * attention ("FLASH-ATTN", FlashAttention-2 > Background) with no mask: the
 * query sees every key of the cache.
 *   q   : [B, H, d] bf16 (the new token's query rows), device.
 *   k, v: [B, Hkv, N, d] bf16 (the cache), device; query head h reads key/value
 *         head h / (H / Hkv); H % Hkv == 0 and H / Hkv <= 16.
 *   o   : [B, H, d] bf16 out; lse : [B, H] fp32 out (natural-log LogSumExp of
 *         the scaled logits).
 *   workspace : device scratch of at least fa_decode_workspace_size(B, H,
 *         Hkv, N, d) bytes (per-chunk partial results), caller-owned; it holds
 *         nothing between calls.
 *   d in {64, 128}; N >= 1.  Two launches on `stream`: the chunks, then the
 *   merge of each row's chunks.
 */
size_t fa_decode_workspace_size(int B, int H, int Hkv, int N, int d);
fa_status fa_decode(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                    size_t workspace_bytes, int B, int H, int Hkv, int N, int d, float scale, void* stream);

/*
 * fa_bwd without a workspace argument, for callers that cannot allocate
 * device memory: a plugin inside another runtime that is handed only its
 * input and output tensors, or code on a path where cudaMalloc (which can
 * synchronise the device and can fail under memory pressure) is not allowed.
 * The pages have no counterpart to this entry point.
 *   Arguments, layouts and results are those of fa_bwd.
 *   Scratch: a 32 MiB array in the library's own device memory (present on
 *   every GPU that loads the library until the process exits).  Sizes whose
 *   fa_bwd_workspace_size() exceeds 32 MiB return FA_ERR_WORKSPACE before any
 *   launch.  All calls share the array; each call re-initialises what it
 *   reads, but calls that overlap on the GPU race, so order them on one
 *   stream.  The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current): make it before any
 *   stream capture.  Allocates nothing.
 */
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal,
                         float scale, void* stream);

/* Human-readable name of a status code (static string). */
const char* fa_status_string(fa_status s);

/*
 * Synchronises `stream`, then reads and clears the device error words of all
 * kernel families.  FA_ERR_TIMEOUT if any kernel recorded a wait that ran out
 * since the last call; FA_ERR_LAUNCH if the stream reports a CUDA error;
 * FA_OK otherwise.
 */
fa_status fa_device_error(void* stream);

/*
 * Measurement hook: the special-function unit's exp2 rate on this GPU, in
 * results per clock per SM (two CTAs of 512 threads per SM, each thread 8
 * independent ex2 -> FMA chains).  The softmax of every kernel here costs one
 * exp2 per score, so this rate bounds it ("FLASH-ATTN", FlashAttention-3:
 * the exponential unit is far slower than the tensor cores).
 *   scratch : caller-owned DEVICE buffer of at least
 *             fa_measure_ex2_rate_scratch_size() bytes (that size depends on
 *             the current device's SM count), 16-byte aligned; overwritten.
 * Synchronises `stream` (it reads the cycle counts back to the host).
 */
size_t fa_measure_ex2_rate_scratch_size(void);
fa_status fa_measure_ex2_rate(float* ex2_per_clock_per_sm, void* scratch, size_t scratch_bytes, void* stream);

/*
 * Test hook for the FMA-pipe exponential ("software exp2", named by the
 * FlashAttention-4 summary in "FlashAttention 源码级深度解析" as a Blackwell
 * lever): y[i] = 2^x[i] computed by the library's own polynomial (Cody-Waite
 * split x = n + f, |f| <= 1/2, a minimax polynomial of `degree` 2 or 3 for
 * 2^f, 2^n added into the exponent field; x below -126 is taken as -126), the
 * same device function the forward kernel can use for part of its
 * exponentials.  Maximum relative error 1.73e-3 at degree 2, 7.5e-5 at degree
 * 3, for x in [-125.5, 127]; below that the result stands in for zero (it is
 * at most 2^-125).
 *   x, y : DEVICE fp32 arrays of n elements (n >= 1), 16-byte aligned.
 */
fa_status fa_debug_exp2_poly(const float* x, float* y, long long n, int degree, void* stream);

/*
 * Test hook for the timeout path: launches one CTA whose thread waits on an
 * mbarrier that nothing ever completes, with a limit of about `limit_us`
 * microseconds (1..1000000); the kernel records a timeout and returns.  A
 * following fa_device_error() must report FA_ERR_TIMEOUT.
 */
fa_status fa_debug_wait_timeout(unsigned int limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
