/*
 * zyfa.h - C ABI of the GB300 (sm_103a) causal prefill attention library (libzyfa.so).
 *
 * The operation (ZYFA: Speed and Accuracy of FP8 FlashAttention on AMD CDNA4, abstract; spbcomputers.ru
 * ZYFA article, intro and FAQ "Это готовый сервер инференса?": a flash_attn_func-compatible kernel
 * library for causal forward attention in the prefill phase, FP8 e4m3 and BF16):
 *
 *     out[b, i, h, :] = sum_{j <= i} softmax_j(scale * q[b,i,h,:] . k[b,j,hk,:]) * v[b,j,hk,:]
 *     hk = h / (H / H_kv)   (grouped-query attention; H_kv == H is plain multi-head attention)
 *
 * FP8 numerics (same sources, abstract techniques (1) and (3); spbcomputers.ru article, section
 * "Три приёма"): probabilities are produced directly as e4m3 codes by one multiply-add and one
 * rounding ("Lean P": code(2^x) = rne(8x + 55.625)); every (row, 64-key block) of probabilities is
 * scaled up by a power of two before rounding and the scale is removed inside the PV product; the
 * output is normalised by the sum of the already-rounded probabilities.  BF16 numerics: probabilities
 * 2^(x - M) rounded to bf16, normalised by the sum of the rounded values.
 *
 * Memory layout (all tensors dense, row-major, flash_attn_func order, device memory):
 *     q   [B, S, H,    D_qk]   e4m3 (one byte per element) or bf16
 *     k   [B, S, H_kv, D_qk]   same type as q
 *     v   [B, S, H_kv, D_v ]   same type as q
 *     out [B, S, H,    D_v ]   bf16, written in full for every call with S > 0
 * Supported head shapes (D_qk, D_v): (64, 64), (128, 128), (192, 128) (the last one is the
 * DeepSeek-style multi-head latent attention shape, 128 "nope" + 64 rotary dims).
 * Inputs must be finite (no e4m3 NaN codes 0x7F / 0xFF, no bf16 Inf or NaN); the output for
 * non-finite inputs is unspecified.  A 64-key block whose scale lies more than 127 binades below its
 * row's reference contributes at most 2^-127 of its weight (its E8M0 scale is clamped).  FP8 scaled
 * scores (softmax_scale * descales * q.k) must stay below 2^16 binades in magnitude, where the
 * Lean-P offset 55.625 - 8e is still exact in fp32 (attention scores are many orders smaller).
 *
 * Per-device state: the library keeps, per device and for the life of the process, the device address
 * of its status word and of the allocation-free scratch, the shared-memory opt-in of each kernel and
 * two copy streams for the host-buffer entry point.  Do not use it across cudaDeviceReset() (or any
 * other teardown of a device's primary context) in the same process: those cached addresses,
 * attributes and streams would belong to the destroyed context.
 */
#ifndef ZYFA_H_
#define ZYFA_H_

#include <cuda_runtime.h>
#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ZYFA_DTYPE_E4M3 = 0, /* OCP FP8 e4m3 ("fn"): q, k, v hold bit patterns, one byte each */
  ZYFA_DTYPE_BF16 = 1
} zyfa_dtype_t;

typedef enum {
  ZYFA_OK = 0,
  ZYFA_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, H % H_kv != 0, bad scale, bad dtype */
  ZYFA_ERR_UNSUPPORTED = 2, /* head shape outside the supported list, or sizes beyond int range   */
  ZYFA_ERR_MISALIGNED = 3,  /* q, k, v or out not 16-byte aligned (TMA and vector stores need it) */
  ZYFA_ERR_CUDA = 4,        /* a CUDA runtime / driver call failed (launch, attribute, tensor map) */
  ZYFA_ERR_TIMEOUT = 5      /* a kernel gave up waiting on a pipeline barrier (see check_errors)  */
} zyfa_status_t;

/*
 * zyfa_attn_fwd_causal - causal forward attention, asynchronous on `stream`.
 *
 *   q, k, v, out   device pointers in the layout above; the caller owns them.  out must not alias
 *                  q, k or v.
 *   B, S, H, H_kv  batch, sequence length (queries and keys), query heads, key/value heads;
 *                  B, H, H_kv >= 1, S >= 0, H % H_kv == 0.  S == 0 returns ZYFA_OK with no launch.
 *   D_qk, D_v      head dims of q/k and of v/out, one of the supported pairs.
 *   softmax_scale  multiplier of q.k; 0 selects the flash_attn_func default (float)(1/sqrt(D_qk)).
 *                  Negative, NaN or infinite values are rejected.
 *   dtype          ZYFA_DTYPE_E4M3 or ZYFA_DTYPE_BF16 (type of q, k, v).
 *   q_descale, k_descale, v_descale
 *                  FP8 only: device pointers to one fp32 each, the per-tensor factor that turns a
 *                  stored e4m3 value into the real value (real = e4m3 * descale).  NULL means 1.0.
 *                  Ignored for BF16.  Read on the device, so no host synchronisation happens.
 *   stream         CUDA stream (0 = legacy default stream).
 *
 * Returns ZYFA_OK once the kernel is enqueued; argument errors are returned before anything is
 * enqueued.  The call allocates no memory, keeps no per-call state and may be issued concurrently
 * from several host threads.  Results are bitwise reproducible for identical inputs.  A kernel that
 * stops on a pipeline timeout records ZYFA_ERR_TIMEOUT in a per-device status word that
 * zyfa_check_errors() reports; the output of that launch is then unspecified.
 */
zyfa_status_t zyfa_attn_fwd_causal(const void* q, const void* k, const void* v, void* out, int B, int S,
                                   int H, int H_kv, int D_qk, int D_v, float softmax_scale,
                                   zyfa_dtype_t dtype, const float* q_descale, const float* k_descale,
                                   const float* v_descale, cudaStream_t stream);

/* How FP8 probabilities are produced (ZYFA abstract, technique (1); captivela ZYFA article, "Tiga Trik"). */
typedef enum {
  ZYFA_P_LEAN = 0,  /* Lean P: one multiply-add and one rounding per probability (the default)      */
  ZYFA_P_EXACT = 1, /* exact P: hardware exponential, then e4m3 rounding (the pages' comparison point) */
  ZYFA_P_EXACT_NO_BLOCK_SCALE = 2 /* exact P rounded against the row's running reference exponent,
                       with no per-64-key power-of-two scaling: the ablation of technique (2)
                       (spbcomputers.ru ZYFA article, "Три приёма").  The reference is the first
                       128-key tile's largest block exponent, raised to a later tile's when that
                       exceeds it by more than 8 binades; probabilities far below it round to 0. */
} zyfa_p_mode_t;

/* Optional behaviour of zyfa_attn_fwd_causal_ex.  A zero-initialised struct (or NULL) gives the
 * behaviour of zyfa_attn_fwd_causal. */
typedef struct {
  zyfa_p_mode_t p_mode;    /* FP8 only; BF16 always exponentiates exactly (ignored there)          */
  int descale_per_kv_head; /* FP8 only: 0 = each descale points to one float; 1 = to B*H_kv floats,
                              [b][hk], the descale of batch b and KV head hk (flash_attn_func's
                              (batch, nheads_k) descale tensors); query head h uses hk = h/(H/H_kv) */
  float* lse;              /* NULL, or a device pointer to B*H*S floats, [b][h][i], 4-byte aligned:
                              receives ln sum_{j<=i} exp(scale * q_i . k_j) in real (descaled) units,
                              from the same rounded weights that normalise the output */
} zyfa_fwd_options_t;

/*
 * zyfa_attn_fwd_causal_ex - zyfa_attn_fwd_causal with the options above (flash_attn_func's
 * softmax_lse output and per-(batch, KV head) descales; exact P for the Lean-P ablation).
 * `options` may be NULL.  Same layouts, ownership, asynchrony and errors as zyfa_attn_fwd_causal;
 * additionally ZYFA_ERR_INVALID_ARG for an unknown p_mode or a descale_per_kv_head other than 0/1,
 * ZYFA_ERR_MISALIGNED for an lse pointer that is not 4-byte aligned.
 */
zyfa_status_t zyfa_attn_fwd_causal_ex(const void* q, const void* k, const void* v, void* out, int B, int S,
                                      int H, int H_kv, int D_qk, int D_v, float softmax_scale,
                                      zyfa_dtype_t dtype, const float* q_descale, const float* k_descale,
                                      const float* v_descale, const zyfa_fwd_options_t* options,
                                      cudaStream_t stream);

/*
 * zyfa_attn_fwd_causal_host - zyfa_attn_fwd_causal for inputs and output in host memory, with the
 * transfers overlapped with the computation.
 *
 * The query rows are split into `chunks` equal groups of 256-row blocks (at most 64 and at most one per
 * block).  chunks = 0 selects the library's plan: with 32 blocks or more (S > 7,936), four equal
 * groups over the first 7/8 of the blocks and two short groups of 1/16 each at the end (the last
 * group's download cannot overlap any computation, so it is kept short); below that, four equal
 * groups.  Chunk c's rows of q, k and v are copied to the device buffers on an internal upload
 * stream; the kernel for chunk c's query rows then runs on `stream` (causality: those rows read keys
 * and values of chunks <= c only, all already uploaded); its output rows are copied back on an
 * internal download stream while later chunks compute.  `stream` waits for the last download, so
 * synchronising `stream` (or a later operation on it) sees the complete output in `out_host`.
 *
 *   q_host, k_host, v_host   host memory, layout as for zyfa_attn_fwd_causal; page-locked (pinned)
 *                            memory is needed for the copies to overlap (pageable memory works but
 *                            serialises them).  Read after earlier work on `stream`.
 *   out_host                 host memory [B,S,H,D_v] bf16, written by the call.
 *   q_dev, k_dev, v_dev, out_dev
 *                            device buffers of the full tensor sizes, 16-byte aligned, owned by the
 *                            caller (they hold the uploaded inputs and the output afterwards).
 *   q/k/v_descale            device pointers as for zyfa_attn_fwd_causal.
 *   chunks, stream           see above.
 * Other arguments and errors as zyfa_attn_fwd_causal (plus ZYFA_ERR_INVALID_ARG for null host
 * pointers or chunks < 0).  The two copy streams are created on the first call on a device and kept
 * for the life of the process; the call allocates no memory.
 */
zyfa_status_t zyfa_attn_fwd_causal_host(const void* q_host, const void* k_host, const void* v_host, void* out_host,
                                        void* q_dev, void* k_dev, void* v_dev, void* out_dev, int B, int S, int H,
                                        int H_kv, int D_qk, int D_v, float softmax_scale, zyfa_dtype_t dtype,
                                        const float* q_descale, const float* k_descale, const float* v_descale,
                                        int chunks, cudaStream_t stream);

/*
 * zyfa_hadamard_quantize_e4m3 - Hadamard rotation and per-tensor FP8 quantisation of Q or K, the
 * pre-pass that roughly halves the error input quantisation adds to attention (spbcomputers.ru ZYFA
 * article, FAQ "Что даёт поворот Адамара?"; captivela ZYFA article, "Angka Nyata").  Rotating Q and K
 * by the same orthogonal matrix leaves attention unchanged, so the codes go straight into
 * zyfa_attn_fwd_causal (V is not rotated).
 *
 *   x          device pointer, bf16 [rows][D] (e.g. q [B,S,H,D] with rows = B*S*H), 16-byte aligned.
 *   x8         device pointer, e4m3 codes [rows][D], 16-byte aligned; written in full.
 *   descale    device pointer to one float, 4-byte aligned: receives the per-tensor descale
 *              fl32(max|y| / 448) (1.0 if every rotated value is 0), ready to pass as q/k_descale.
 *   rows, D    rows >= 0 (0: nothing is done), D in {64, 128, 192}.
 *   workspace  device scratch of at least zyfa_hadamard_workspace_bytes(rows) bytes, 4-byte
 *              aligned, owned by the caller; its contents on entry do not matter.
 *
 * y = x R with R block-diagonal over the head dimension: normalised Walsh-Hadamard blocks of 128
 * (D = 128) or 64 (D = 64, 192), computed in fp32 by the radix-2 transform; codes =
 * rne_e4m3_satfinite(fl32(y * fl32(448 / max|y|))).  Two kernel launches on `stream`, asynchronous; allocates
 * nothing.  Errors: ZYFA_ERR_INVALID_ARG (null pointers, negative rows, short workspace),
 * ZYFA_ERR_UNSUPPORTED (D, or rows*D beyond 2^40), ZYFA_ERR_MISALIGNED, ZYFA_ERR_CUDA (launch).
 */
zyfa_status_t zyfa_hadamard_quantize_e4m3(const void* x, void* x8, float* descale, long long rows, int D,
                                          void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * zyfa_hadamard_quantize_qk_e4m3 - zyfa_hadamard_quantize_e4m3 for Q and K together (same passage):
 * the same rotation and quantisation, each tensor with its own per-tensor descale, in one launch per
 * pass instead of two.  Q's and K's 128-row blocks share one wave of CTAs, so the smaller tensor no
 * longer runs a partly empty wave of its own.
 *
 *   q, q8, q_descale, q_rows   Q's input, codes, descale and rows, as x, x8, descale, rows above.
 *   k, k8, k_descale, k_rows   the same for K.
 *   D                          the common head dimension, 64, 128 or 192.
 *   workspace                  at least zyfa_hadamard_workspace_bytes(q_rows) +
 *                              zyfa_hadamard_workspace_bytes(k_rows) bytes, 4-byte aligned.
 * Codes and descales equal those of two zyfa_hadamard_quantize_e4m3 calls, bit for bit.  Two kernel
 * launches on `stream`, asynchronous, allocates nothing; errors as zyfa_hadamard_quantize_e4m3 (either
 * tensor's).  If one of the two has no rows, only the other is processed.
 */
zyfa_status_t zyfa_hadamard_quantize_qk_e4m3(const void* q, void* q8, float* q_descale, long long q_rows,
                                             const void* k, void* k8, float* k_descale, long long k_rows, int D,
                                             void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * zyfa_hadamard_quantize_e4m3_noalloc - zyfa_hadamard_quantize_e4m3 without a workspace argument, for
 * callers that cannot allocate device memory on their call path: a serving runtime whose device
 * memory is planned up front and may not grow, or a plain C host program with no device allocator
 * from which to hand over scratch.  The pages describe no such call; it is a convenience of this
 * library.
 *
 * Same arguments, results and errors as zyfa_hadamard_quantize_e4m3, minus the workspace.  The
 * scratch (the partial maxima) is a fixed 128 KiB array inside the library that every GPU which loads
 * it holds until the process exits; it covers at most 4,194,304 rows per call, and larger calls return
 * ZYFA_ERR_UNSUPPORTED without doing anything.  The call allocates nothing.  Its first call on a
 * device looks up the array's device address (once per device, with that device current), so make
 * that first call before any stream capture.  All calls share the one array: calls that overlap on
 * the GPU (on different streams, or from several host threads, on the same device) race on it and
 * may produce wrong codes; serialise them.  Nothing in the array needs to start at zero: each call
 * writes every slot it later reads.
 */
zyfa_status_t zyfa_hadamard_quantize_e4m3_noalloc(const void* x, void* x8, float* descale, long long rows, int D,
                                                  cudaStream_t stream);

/* zyfa_hadamard_workspace_bytes - workspace zyfa_hadamard_quantize_e4m3 needs for `rows` rows:
 * one float per 128 rows (0 for rows <= 0).  Pure host arithmetic. */
size_t zyfa_hadamard_workspace_bytes(long long rows);

/*
 * zyfa_check_errors - synchronise `stream`, then read and clear the current device's status word.
 * Returns ZYFA_ERR_TIMEOUT if any kernel of this library timed out since the last check,
 * ZYFA_ERR_CUDA if the synchronisation itself failed, ZYFA_OK otherwise.
 */
zyfa_status_t zyfa_check_errors(cudaStream_t stream);

/*
 * zyfa_selftest_stalled_pipeline - exercise the timeout path without faulting or hanging the GPU.
 *
 * Enqueues the same kernel as zyfa_attn_fwd_causal (same arguments, default softmax scale, no
 * descales) with its load-issuing warp told to withhold every load.  Every other role then waits on
 * a barrier that never completes; each wait is bounded (about 2^31 SM clocks, roughly one second),
 * after which the kernel records ZYFA_ERR_TIMEOUT in the status word, waits for nothing it has in
 * flight, releases its tensor memory and returns, leaving the CUDA context usable.  `out` is not
 * written.  Returns the same argument errors as zyfa_attn_fwd_causal, else ZYFA_OK once enqueued;
 * the following zyfa_check_errors() then returns ZYFA_ERR_TIMEOUT.  For tests of error handling
 * only.  The pages describe no such call; it belongs to this library's failure detection.
 */
zyfa_status_t zyfa_selftest_stalled_pipeline(const void* q, const void* k, const void* v, void* out, int B, int S,
                                             int H, int H_kv, int D_qk, int D_v, zyfa_dtype_t dtype,
                                             cudaStream_t stream);

/* zyfa_status_string - static, human-readable name of a status code (never NULL). */
const char* zyfa_status_string(zyfa_status_t status);

/*
 * zyfa_kernel_launches - number of kernel launches one zyfa_attn_fwd_causal call with these sizes
 * enqueues (0 for S == 0, else 1).  Pure host arithmetic, for accounting in benchmarks.
 */
int zyfa_kernel_launches(int B, int S, int H);

/*
 * zyfa_probe_mma_rate - measure this GPU's dense tensor-core rate with the attention kernel's own
 * instruction forms (the denominator of "% of FP8 peak"; captivela ZYFA article, "Angka Nyata",
 * quotes FP8 prefill throughput as a share of the FP8 peak).
 *
 *   fp8        1: tcgen05.mma kind::f8f6f4 on e4m3 operands; 0: kind::f16 on bf16 operands.
 *   iters      MMA iterations per CTA (>= 1); one iteration is zyfa_probe_mma_flops_per_iter(fp8)
 *              floating-point operations (an M=128, N=256 product over 128 bytes of K).
 *   grid       CTAs to launch; one CTA occupies one SM (pass the SM count to load every SM).
 *   cycles     device array of `grid` long longs: each CTA's clock64 span from its first MMA issue
 *              to the completion of its last MMA.
 *   timed_out  device int; bit 0 is set if a CTA gave up waiting (a few seconds) for its MMAs.
 * Asynchronous on `stream`; the caller times the launch (CUDA events) and owns both buffers.  The
 * operands are synthetic values held in shared memory; nothing else is read or written.  Returns
 * ZYFA_ERR_INVALID_ARG for bad arguments, ZYFA_ERR_CUDA if the launch fails.
 */
zyfa_status_t zyfa_probe_mma_rate(int fp8, int iters, int grid, long long* cycles, int* timed_out,
                                  cudaStream_t stream);

/* zyfa_probe_mma_flops_per_iter - floating-point operations of one probe iteration per CTA. */
long long zyfa_probe_mma_flops_per_iter(int fp8);

/*
 * zyfa_probe_mma_form_rate - the tensor-core rate of one of the attention kernel's own MMA forms,
 * issued back to back with nothing else in the loop: what each kind of product in the kernel reaches
 * by itself, against which the kernel's schedule is judged.
 *
 *   form       0  FP8 score tile: M=128, N=128, D=128, both operands in shared memory;
 *              1  FP8 PV: block-scaled (e8m0 factors in tensor memory), M=128, N=144 (D_v = 128 plus the
 *                 16 row-sum columns), 128 keys, P in tensor memory, V in shared memory;
 *              2  form 0 followed by form 1;
 *              3  the FP8 score tile as two N=64 halves;
 *              4  BF16 score tile: M=128, N=128, D=128;
 *              5  BF16 score tile of the MLA shape: M=128, N=64, D=192.
 *   iters, grid, cycles, timed_out, stream: as for zyfa_probe_mma_rate; one iteration is
 *              zyfa_probe_mma_form_flops_per_iter(form) floating-point operations per CTA.
 * Returns ZYFA_ERR_INVALID_ARG for bad arguments, ZYFA_ERR_CUDA if the launch fails.  This call has
 * no counterpart in the pages: it is measurement support.
 */
zyfa_status_t zyfa_probe_mma_form_rate(int form, int iters, int grid, long long* cycles, int* timed_out,
                                       cudaStream_t stream);

/* zyfa_probe_mma_form_flops_per_iter - floating-point operations of one iteration of `form` (-1 if
 * the form is unknown). */
long long zyfa_probe_mma_form_flops_per_iter(int form);

#ifdef __cplusplus
}
#endif

#endif /* ZYFA_H_ */
