/*
 * lmce -- fused LM-head + token-level softmax cross-entropy, forward and backward,
 * with gradient-accumulation micro-steps, for GB300 (sm_103a).
 *
 * What one optimizer step computes (GPT-2 124M training pages):
 *   logits z = h . W^T with the tied, bias-free output projection W[V, C]
 *     ("How I trained my own GPT-2 124M on FineWeb-Edu", section 4, weight tying);
 *   per-row loss  l_n = logsumexp_v(z[n, :]) - z[n, y_n]  for y_n != ignore_id
 *     (same page, section 4: softmax, pick the target's probability, negative log);
 *   the gradient of  sum_k s_k * sum_n l_n  over the micro-steps k of one step,
 *     accumulated into an fp32 dW  (section 8.1, gradient accumulation);
 *   s_k = 1 / (valid targets over the whole step)  -- the global token mean -- or the
 *     pages' 1 / (valid targets of micro-step k * G)  ("Multi-GPU calculation of
 *     gradients for accelerated training", sections "Gradient accumulation averages
 *     across micro-steps" and "DDP averages gradients across processes").
 *   Pad targets are ignored by the loss (zerotofrontier "GPT", section "Document
 *   boundaries, packing and masking"); the ignore id is configurable, -100 by default.
 *
 * The N x V logits and dlogits never reach device memory.  On the default
 * tensor-core path (LMCE_PATH_TCGEN05) the first pass does store its bf16
 * exponentials 2^(z log2 e - m) -- one N x V array per micro-step, in the handle's
 * scratch -- so that dW is a single product; LMCE_PATH_TCGEN05_RECOMPUTE keeps every
 * N x V quantity on chip and recomputes the logit tiles for dW instead.
 *
 * Conventions for every function below:
 *   - Device pointers are CUDA device addresses on the current device; host pointers
 *     are ordinary host memory.  Rows are C-contiguous (row-major), no padding.
 *   - Every call returns an int status (LMCE_OK or an LMCE_ERR_* code) and never
 *     throws; no device code traps or asserts.
 *   - Calls on one handle must be issued from one host thread and enqueue on one
 *     stream (or on streams the caller orders).  Only lmce_finalize, lmce_dw_sumsq and
 *     the compacting micro-steps given n_valid = -1 block the host.
 *
 * Beyond the head, on the same pages' training step: lmce_microstep_compact skips rows
 * whose target is ignored, lmce_microstep_ln puts the final LayerNorm / RMSNorm (ln_f) in
 * front of the head, lmce_dw_sumsq gives dW's share of the global clip norm and lmce_adamw
 * applies the optimizer to W ("How I trained my own GPT-2 124M", sections 2.8 and 6;
 * "Reproduce GPT-2 124M", training configuration).
 */
#ifndef LMCE_H_
#define LMCE_H_

#include <stdint.h>

#if defined(__GNUC__)
#define LMCE_API __attribute__((visibility("default")))
#else
#define LMCE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------------------- */
#define LMCE_OK              0
#define LMCE_ERR_ARG         1  /* null pointer, bad size or dtype, unaligned pointer      */
#define LMCE_ERR_ARCH        2  /* the current device is not compute capability 10.3       */
#define LMCE_ERR_CUDA        3  /* a CUDA runtime call or kernel launch failed              */
#define LMCE_ERR_BAD_TARGET  4  /* a target was outside [0, V) and not ignore_id (finalize) */
#define LMCE_ERR_NO_VALID    5  /* the step has no valid target                             */
#define LMCE_ERR_NONFINITE   6  /* the summed loss is not finite (finalize)                 */
#define LMCE_ERR_STATE       7  /* call out of order (e.g. finalize before any micro-step)  */
#define LMCE_ERR_INTERNAL    8  /* a bounds check of the debug build failed (finalize)      */

/* ---- configuration ----------------------------------------------------------------- */
typedef enum { LMCE_BF16 = 0, LMCE_FP32 = 1 } lmce_dtype;

typedef enum {
  LMCE_NORM_GLOBAL = 0,     /* s = 1 / global_valid  (global token-weighted mean, default) */
  LMCE_NORM_MICRO_MEAN = 1  /* s = 1 / (valid targets of this micro-step * grad_accum_steps) */
} lmce_norm;

typedef enum {
  LMCE_PATH_AUTO = 0,       /* tensor-core path when the shape allows it, else SIMT; the
                               stored-exponential dW pass when its scratch fits in device
                               memory, else the recomputing one                          */
  LMCE_PATH_SIMT = 1,       /* fp32 FFMA kernels (any C <= 2048, any V, either dtype)    */
  LMCE_PATH_TCGEN05 = 2,    /* tcgen05/TMA kernels: bf16, C % 256 == 0, 256 <= C <= 1024:
                               one pass for logsumexp and dh (online softmax, exact repair of
                               rare out-of-range tiles) that also stores its bf16
                               exponentials, then dW as one product with them (no second
                               logits product); C > 768 runs each pass once per range of at
                               most 768 columns of the gradient.  Scratch: 2 bytes per
                               (max_N row, vocabulary entry rounded up to 256) and 16 C + 32
                               bytes per max_N row (rounded up to 256) beside the rest      */
  LMCE_PATH_TCGEN05_TWO_PASS = 3,  /* tensor cores, shapes as above, always a separate
                                     logsumexp pass before the dW and dh passes          */
  LMCE_PATH_TCGEN05_RECOMPUTE = 4  /* as LMCE_PATH_TCGEN05, but the dW pass recomputes the
                                      logits instead of storing the exponentials (no
                                      max_N x V scratch; a third more tensor work)        */
} lmce_path;

typedef struct lmce_config {
  int64_t C;                /* hidden size (columns of h and W)                              */
  int64_t V;                /* rows of W, padded vocabulary entries included                 */
  int64_t max_N;            /* most rows any micro-step will pass; sizes the library scratch */
  int32_t dtype;            /* lmce_dtype of hidden, W and dh                                */
  int32_t ignore_id;        /* target value that carries no loss (usually -100)              */
  int32_t norm;             /* lmce_norm                                                     */
  int32_t grad_accum_steps; /* G >= 1; used by LMCE_NORM_MICRO_MEAN                          */
  int32_t path;             /* lmce_path                                                     */
  int32_t flags;            /* 0 or an OR of the LMCE_ACCUMULATE_FROM_START, ... bits below  */
} lmce_config;

/* cfg.flags: the first micro-step after create or finalize ADDS its gradient to dW instead of
 * writing it, for a caller that has already written part of the step's gradient into the same
 * buffer (the embedding backward of the tied wte / lm_head matrix). */
#define LMCE_ACCUMULATE_FROM_START 1
/* cfg.flags: also allocate the scratch of lmce_microstep_compact (two [max_N, C] row buffers of
 * the input dtype and 16 bytes per row). */
#define LMCE_COMPACT_VALID_ROWS 2
/* cfg.flags: also allocate the scratch of lmce_microstep_ln (two [max_N, C] row buffers of the
 * input dtype, 8 bytes per row, and 8 * C bytes per 32 rows of parameter-gradient partials). */
#define LMCE_FINAL_NORM 4

/* lmce_microstep_ln: the kind of ln_f */
#define LMCE_LN_LAYERNORM 0
#define LMCE_LN_RMSNORM   1

typedef struct lmce_handle lmce_handle;

/*
 * lmce_create -- validate cfg, check the device, allocate the library scratch
 * (per-row logsumexp, per-block loss/count partials, the step accumulators and the
 * error word: about 12 * max_N + 64 KB of device memory, plus the tensor-core path's
 * buffers, the largest being the stored exponentials of LMCE_PATH_TCGEN05 -- see lmce_path)
 * and return a handle in *out.
 *   dW : device, fp32 [V, C], owned by the caller and kept by the handle until
 *        lmce_destroy.  The first lmce_microstep after create or finalize WRITES it
 *        (dW = this micro-step's gradient) unless cfg.flags has LMCE_ACCUMULATE_FROM_START;
 *        later ones ADD to it.
 * Errors: LMCE_ERR_ARG (null cfg/dW/out, C or V <= 0, max_N < 0, unknown dtype/norm/path,
 *         G < 1, unknown flags, a forced path the shape does not allow), LMCE_ERR_ARCH,
 *         LMCE_ERR_CUDA.
 */
LMCE_API int lmce_create(const lmce_config* cfg, float* dW, lmce_handle** out);

/*
 * lmce_microstep -- enqueue one micro-step on `stream` (a cudaStream_t; NULL = legacy
 * default stream) and return without waiting.  It computes, for this micro-batch, the
 * logits of the tied head, each row's softmax cross-entropy and its gradient ("How I
 * trained my own GPT-2 124M on FineWeb-Edu", section 4 "Implementing Loss Calculation"),
 * scaled by s_k and added into dW as backward adds into .grad between optimizer steps
 * (section 8.1 "Gradient Accumulation"; s_k as "Multi-GPU calculation of gradients for
 * accelerated training", section "Gradient accumulation averages across micro-steps").
 *   hidden      : device, dtype [N, C]  -- h, the final hidden states of N rows
 *   W           : device, dtype [V, C]  -- the tied wte / lm_head weight
 *   targets     : device, int32 [N]     -- next-token ids, or ignore_id
 *   N           : rows in this micro-step, 0 <= N <= max_N (N == 0 is a no-op micro-step)
 *   global_valid: LMCE_NORM_GLOBAL: valid targets over the whole optimizer step (all
 *                 micro-steps, all data-parallel ranks); ignored for MICRO_MEAN
 *   dh          : device, dtype [N, C], written (not accumulated): d(objective)/dh,
 *                 rounded to nearest-even from fp32 for bf16
 *   row_loss    : device, fp32 [N] or NULL; when given, receives every row's loss
 *                 (0 on ignored rows)
 * Out-of-range targets are treated as ignored and reported by lmce_finalize.
 * The tensor-core path needs hidden, W, dh and dW 16-byte aligned.
 * Errors: LMCE_ERR_ARG, LMCE_ERR_NO_VALID (GLOBAL norm with global_valid <= 0: dh is
 *         zeroed, dW untouched, nothing else is enqueued), LMCE_ERR_CUDA.
 */
LMCE_API int lmce_microstep(lmce_handle* h, const void* hidden, const void* W, const int32_t* targets,
                   int64_t N, int64_t global_valid, void* dh, float* row_loss, void* stream);

/*
 * lmce_microstep_compact -- lmce_microstep over the valid rows only.  A row whose target is
 * ignored (masked pad spans: zerotofrontier "GPT", section "Document boundaries, packing and
 * masking") adds nothing to the loss, dh or dW, so the library gathers the rows with a target in
 * [0, V), in their input order, runs both passes over those n_valid rows and scatters dh (and
 * row_loss) back, with zeros on the ignored rows.  The results equal lmce_microstep's up to the
 * summation order of dW (the valid rows sit in other tiles).
 *   n_valid : the valid targets of this micro-step (the caller counts them as it counts
 *             global_valid), 0 <= n_valid <= N; or -1: the library counts them and waits for the
 *             count on `stream` (this call then blocks).  A count that differs from the targets
 *             makes lmce_finalize return LMCE_ERR_ARG, with dh and dW of the step unusable.
 *   other arguments as lmce_microstep.  The handle must have been created with
 *   LMCE_COMPACT_VALID_ROWS.
 * Errors: LMCE_ERR_ARG (as lmce_microstep, n_valid < -1 or > N, no compaction scratch),
 *         LMCE_ERR_NO_VALID (as lmce_microstep), LMCE_ERR_CUDA.
 */
LMCE_API int lmce_microstep_compact(lmce_handle* h, const void* hidden, const void* W, const int32_t* targets,
                                    int64_t N, int64_t n_valid, int64_t global_valid, void* dh, float* row_loss,
                                    void* stream);

/*
 * lmce_microstep_ln -- lmce_microstep with the final normalisation ln_f in front ("How I trained
 * my own GPT-2 124M", section 2.8: LayerNorm; "Reproduce GPT-2 124M", model definition: RMSNorm):
 *   h  = ln_f(x) = (x - mean) * rstd * gamma + beta, per row, rstd = 1 / sqrt(var + eps) with the
 *        biased variance (RMSNorm: mean = 0, var = mean of x^2, no beta), computed in fp32 and
 *        rounded to the input dtype (nearest-even) for the head
 *   dx = the gradient through ln_f of the head's dh (bf16-rounded for bf16 handles):
 *        rstd * (g - mean_c(g) - xhat * mean_c(g * xhat)), g = dh * gamma, xhat = (x - mean) * rstd
 *        (RMSNorm: no mean_c(g) term)
 *   dgamma = sum over rows of dh * xhat, dbeta = sum over rows of dh, fp32, summed in a fixed order;
 *        written by the first micro-step of a step and added by later ones, exactly as dW.
 *   x       : device, dtype [N, C] -- the last block's output, row-major
 *   gamma   : device, fp32 [C];  beta : device, fp32 [C] or NULL (RMSNorm: must be NULL)
 *   ln_kind : LMCE_LN_LAYERNORM or LMCE_LN_RMSNORM;  eps >= 0 (torch's LayerNorm default: 1e-5)
 *   dx      : device, dtype [N, C], written
 *   dgamma  : device, fp32 [C];  dbeta : device, fp32 [C] or NULL (NULL when beta is NULL)
 *   W, targets, N, global_valid, row_loss, stream: as lmce_microstep.  The handle must have been
 *   created with LMCE_FINAL_NORM; h and dh live in its scratch.
 * Errors: LMCE_ERR_ARG (as lmce_microstep, a null gamma/dgamma, an unknown ln_kind, beta with
 *         RMSNorm, eps < 0, no ln_f scratch), LMCE_ERR_NO_VALID (GLOBAL norm with
 *         global_valid <= 0: dx is zeroed, dgamma, dbeta and dW untouched), LMCE_ERR_CUDA.
 */
LMCE_API int lmce_microstep_ln(lmce_handle* h, const void* x, const float* gamma, const float* beta, int32_t ln_kind,
                               float eps, const void* W, const int32_t* targets, int64_t N, int64_t global_valid,
                               void* dx, float* dgamma, float* dbeta, float* row_loss, void* stream);

/*
 * lmce_microstep_ln_compact -- lmce_microstep_ln over the valid rows only: the rows of x whose
 * target is in [0, V) are gathered in input order (as lmce_microstep_compact gathers h), ln_f, the
 * head and ln_f's backward run on those n_valid rows, and dx (and row_loss) are scattered back with
 * zeros on the ignored rows.  An ignored row's dh is zero, so its dx and its share of dgamma and
 * dbeta are zero too: the results equal lmce_microstep_ln's up to summation order.
 *   n_valid : as lmce_microstep_compact (-1: counted on the device, blocking).
 *   other arguments as lmce_microstep_ln.  The handle must have been created with both
 *   LMCE_FINAL_NORM and LMCE_COMPACT_VALID_ROWS.
 * Errors: as lmce_microstep_ln, and LMCE_ERR_ARG for n_valid < -1 or > N or a handle without
 *         the compaction scratch; a wrong n_valid is reported by lmce_finalize as LMCE_ERR_ARG.
 */
LMCE_API int lmce_microstep_ln_compact(lmce_handle* h, const void* x, const float* gamma, const float* beta,
                                       int32_t ln_kind, float eps, const void* W, const int32_t* targets, int64_t N,
                                       int64_t n_valid, int64_t global_valid, void* dx, float* dgamma, float* dbeta,
                                       float* row_loss, void* stream);

/*
 * lmce_finalize -- synchronise `stream`, read the step's results and reset the handle
 * for the next optimizer step (the next micro-step writes dW again).  It is the loss a
 * training loop reads once per step: the pages accumulate loss / G over the micro-steps
 * and read it after the last one ("How I trained my own GPT-2 124M", section 9, training
 * loop; "Multi-GPU calculation of gradients for accelerated training", section "Gradient
 * accumulation averages across micro-steps"), here as the objective sum_k s_k loss_k.
 *   loss_sum    : host, may be NULL -- sum of the valid rows' losses over the step
 *   valid_count : host, may be NULL -- valid targets seen over the step
 *   loss_mean   : host, may be NULL -- sum_k s_k * loss_sum_k, the objective whose gradient
 *                 dW holds: the token mean for GLOBAL norm on one rank, the pages'
 *                 sum_k mean_k / G for MICRO_MEAN; NaN when no target was valid
 * Errors: LMCE_ERR_STATE (no micro-step since create/finalize), LMCE_ERR_ARG (a compacted
 *         micro-step's n_valid was not its targets' count), LMCE_ERR_BAD_TARGET,
 *         LMCE_ERR_NONFINITE, LMCE_ERR_NO_VALID, LMCE_ERR_CUDA.  Results are written
 *         whenever the device values could be read, errors included.
 */
LMCE_API int lmce_finalize(lmce_handle* h, double* loss_sum, int64_t* valid_count, double* loss_mean,
                  void* stream);

/*
 * lmce_dw_sumsq -- the sum over every element of dW of dW^2 to float64 accuracy, reduced in a
 * fixed order (bitwise reproducible): the squared global norm a gradient clip
 * (clip_grad_norm_ over the tied matrix) needs.  Enqueued on `stream` after the work already
 * there, then waited for.  Reads dW as it stands (any number of micro-steps; normally after the
 * last one of a step and before the optimizer).
 *   sumsq : host -- the result
 * Errors: LMCE_ERR_ARG (null h or sumsq), LMCE_ERR_CUDA.
 */
LMCE_API int lmce_dw_sumsq(lmce_handle* h, double* sumsq, void* stream);

/*
 * lmce_clip_coef -- the global-norm clip coefficient that torch.nn.utils.clip_grad_norm_
 * applies ("Reproduce GPT-2 124M", training configuration: grad_norm_clip = 1.0):
 *   *coef = min(1, max_norm / (sqrt(sumsq) + 1e-6))   (float64, then rounded to float32)
 *   sumsq    : the sum of squares over every gradient of the model (lmce_dw_sumsq gives the
 *              tied matrix's share; add the other tensors' shares), finite and >= 0
 *   max_norm : > 0 and finite
 *   coef     : host -- the value lmce_adamw's `clip` takes
 * Host only: touches no device and no handle.
 * Errors: LMCE_ERR_ARG (null coef, sumsq < 0 or not finite, max_norm <= 0 or not finite).
 */
LMCE_API int lmce_clip_coef(double sumsq, double max_norm, float* coef);

/*
 * lmce_adamw -- one AdamW step on the tied matrix, after lmce_finalize, in one pass over the
 * elements (decoupled weight decay and Adam's bias correction, as torch.optim.AdamW):
 *   g = clip * dW
 *   m = beta1 * m + (1 - beta1) * g           v = beta2 * v + (1 - beta2) * g^2
 *   p = p * (1 - lr * weight_decay) - (lr / (1 - beta1^step)) * m / (sqrt(v) / sqrt(1 - beta2^step) + eps)
 *   W_out = p rounded to nearest-even bf16
 * in float32 (the bias corrections in float64 on the host).
 *   h            : the handle whose dW holds the step's gradient (read only)
 *   p, m, v      : device, fp32 [V, C]: master weights and the two moment estimates, updated in
 *                  place (m and v zero before the first step); caller-owned
 *   W_out        : device, bf16 [V, C] (the W the next forward reads), or NULL; caller-owned.
 *                  Any alignment; when dW, p, m, v and W_out are all 16-byte aligned the kernel
 *                  moves 16-byte vectors
 *   step         : t >= 1, the step being taken
 *   clip         : the global-norm clip coefficient, from lmce_clip_coef (1 for none)
 *   lr, beta1, beta2, eps, weight_decay : as torch.optim.AdamW; "How I trained my own GPT-2 124M",
 *                  section 6 "Implementing the Optimizer", uses 0.9, 0.95, 1e-8 and 0.1, with
 *                  decay on every tensor of two or more dimensions (W is one)
 * Enqueued on `stream`; does not block.  Counted under LMCE profile kind 1 (the finish kind).
 * Errors: LMCE_ERR_ARG (null h/p/m/v, step < 1, a beta outside [0, 1), eps < 0 or NaN, a
 *         non-finite lr, weight_decay or clip), LMCE_ERR_CUDA.
 */
LMCE_API int lmce_adamw(lmce_handle* h, float* p, float* m, float* v, void* W_out, int64_t step, float lr,
                        float beta1, float beta2, float eps, float weight_decay, float clip, void* stream);

/* lmce_destroy -- free the library scratch (not dW) and the handle.  NULL is allowed. */
LMCE_API int lmce_destroy(lmce_handle* h);

/* lmce_status_string -- static description of a status code. */
LMCE_API const char* lmce_status_string(int status);

/* lmce_launch_count -- kernels this handle has launched since create (host counter). */
LMCE_API int64_t lmce_launch_count(const lmce_handle* h);

/* lmce_selected_path -- LMCE_PATH_SIMT, LMCE_PATH_TCGEN05, LMCE_PATH_TCGEN05_TWO_PASS or
 * LMCE_PATH_TCGEN05_RECOMPUTE: the path micro-steps run. */
LMCE_API int lmce_selected_path(const lmce_handle* h);

/*
 * lmce_test_stall_next_microstep -- failure-detection test hook (not part of a training
 * step).  Arms the next micro-step of this handle so that its tensor-core gradient launches
 * start no operand load and bound every wait by `wait_ns` nanoseconds (0 < wait_ns <= 1 s)
 * instead of the normal 2 s.  Their waits then run out: each kernel records a timeout in the
 * step's error word, waits for the MMAs it issued, releases its tensor memory and returns,
 * and the context stays usable.  lmce_finalize reports the step as LMCE_ERR_CUDA; the
 * step's outputs are undefined.  One micro-step only; the hook then disarms itself.
 * Errors: LMCE_ERR_ARG (null handle, wait_ns out of range), LMCE_ERR_STATE (the handle runs
 *         the SIMT path, whose kernels have no such waits).
 */
LMCE_API int lmce_test_stall_next_microstep(lmce_handle* h, int64_t wait_ns);

/*
 * Debug build (no counterpart in the pages: a checking aid for this library).  Built with
 * LMCE_DEBUG_BOUNDS=1 (grad_lmce_microstep_gb300.build.build(debug_bounds=True) makes
 * liblmce_dbg.so beside liblmce.so), the kernels check their computed indices before the
 * accesses they guard: the row coordinates of the tensor-core passes' TMA boxes, the one-hot
 * hit list, the split-tile partial slots, the repair flags, the one-hot rows of W, and the
 * compaction's positions.  A check that fails records the site in the step's error word and
 * the access is skipped; nothing traps, and lmce_finalize returns LMCE_ERR_INTERNAL.  The
 * release build compiles the checks away.
 *
 * lmce_debug_bounds -- 1 in the debug build, 0 in the release build.  Needs no device.
 *
 * lmce_test_bounds_limit -- test hook of the debug build: the compaction's checks treat the
 * compact buffers as holding `rows` rows (0 <= rows <= max_N; max_N restores them), so a step
 * with more valid rows than that reports LMCE_ERR_INTERNAL at finalize without any access
 * outside the real buffers.  That step's outputs are undefined.
 * Errors: LMCE_ERR_ARG (null handle, rows out of range), LMCE_ERR_STATE (the release build, or
 *         a handle created without LMCE_COMPACT_VALID_ROWS).
 */
LMCE_API int lmce_debug_bounds(void);
LMCE_API int lmce_test_bounds_limit(lmce_handle* h, int64_t rows);

/* ---- kernel timing (benchmark instrumentation) --------------------------------------
 * When enabled, the library records a CUDA event pair around every kernel it launches
 * (on the stream the kernel runs on) so that per-kernel device time can be read back.
 * Kinds: */
#define LMCE_KIND_LSE     0  /* logits tiles + online logsumexp (+ per-row loss)         */
#define LMCE_KIND_FINISH  1  /* per-row passes, split-tile combines, fixed-order loss /  */
                             /* count reductions, gradient scale                        */
#define LMCE_KIND_DW      2  /* recomputed logits -> dlogits -> dW accumulation           */
#define LMCE_KIND_DH      3  /* recomputed logits -> dlogits -> dh                        */
#define LMCE_KIND_LSE_DH  4  /* logits tiles -> online softmax -> logsumexp and dh        */
#define LMCE_KIND_LN      5  /* ln_f forward, backward and parameter-gradient reduction */
#define LMCE_KIND_COMPACT 6  /* valid-row count, scan, gather and scatter               */
#define LMCE_KIND_COUNT   7

/* lmce_profile -- enable (1: clears earlier records) or disable (0) the event records. */
LMCE_API int lmce_profile(lmce_handle* h, int enable);

/*
 * lmce_profile_read -- synchronise the recorded events and return, for one kind, the
 * summed device time in milliseconds and the number of launches recorded.
 * Errors: LMCE_ERR_ARG (null handle or outputs, unknown kind), LMCE_ERR_CUDA.
 */
LMCE_API int lmce_profile_read(lmce_handle* h, int kind, double* total_ms, int64_t* launches);

/* ---- allocation-free micro-step --------------------------------------------------------
 * No counterpart on the GPT-2 training pages: this entry point exists for callers that
 * cannot call cudaMalloc -- a host runtime that hands out all device memory from its own
 * pool or arena and does not let a library allocate behind its back, or a code path that
 * must not stall (cudaFree synchronises the whole device, and cudaMalloc may too).
 *
 * lmce_microstep_noalloc -- enqueue one self-contained micro-step on `stream` with the
 * SIMT kernels, without any allocation: no cudaMalloc, no cudaFree, no allocating library
 * routine.  Its scratch (per-row logsumexp, per-block partials, accumulators) is a fixed
 * array of about 360 KB compiled into the library, which every GPU that loads the library
 * holds until the process exits.
 *   cfg             : as for lmce_create; max_N is ignored, flags must be 0 (accumulate_dW
 *                     says whether dW is written or added to), path must be AUTO or SIMT,
 *                     C <= 2048
 *   hidden, W, targets, N, global_valid, dh, row_loss : as for lmce_microstep
 *   dW              : device, fp32 [V, C]; written (accumulate_dW == 0) or added to (!= 0)
 *   loss_sum_out    : device double, or NULL: this micro-step's summed loss
 *   valid_count_out : device int64, or NULL: this micro-step's valid targets
 * Limits: N <= LMCE_NOALLOC_MAX_N; a larger N returns LMCE_ERR_ARG before anything is
 * enqueued.  hidden, W and dh must be aligned to their element size, the other pointers to
 * theirs (LMCE_ERR_ARG otherwise).
 * Errors found on the device are not returned by this call: an out-of-range target is
 * treated as ignored (it is left out of *valid_count_out, so a caller that knows its own
 * count can compare), and a non-finite loss shows as a non-finite *loss_sum_out.
 * Set-up: the first call on a device (more exactly, on a CUDA context: again after a device
 * reset) loads the code of every kernel this entry point launches, for both dtypes.  It is
 * the only call that may load code; later calls allocate nothing, whatever their dtype or
 * size.  Make it before any stream capture.  Each call looks the array's device address up
 * again with the device current, so a reset that moves the array is followed.
 * Every call on a device shares the one array and it keeps the last call's contents (the
 * accumulators are cleared by each call); calls whose work overlaps on the GPU -- on
 * different streams, or from different host threads -- race on it and must be serialised
 * by the caller.
 * Errors: LMCE_ERR_ARG, LMCE_ERR_ARCH, LMCE_ERR_NO_VALID (GLOBAL norm with
 *         global_valid <= 0: dh zeroed, dW untouched), LMCE_ERR_CUDA.
 */
#define LMCE_NOALLOC_MAX_N 65536
LMCE_API int lmce_microstep_noalloc(const lmce_config* cfg, const void* hidden, const void* W,
                                    const int32_t* targets, int64_t N, int64_t global_valid, void* dh,
                                    float* dW, int accumulate_dW, float* row_loss, double* loss_sum_out,
                                    int64_t* valid_count_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LMCE_H_ */
