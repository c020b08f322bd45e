/*
 * muon.h — C ABI of the GB300 (sm_103a) Muon optimizer step.
 *
 * The Muon step for a 2-D hidden weight matrix W with gradient G and fp32
 * momentum M is
 *
 *   M <- mu*M + G;  U = G + mu*M (Nesterov) or U = M;
 *   X0 = U / ||U||_F (on U^T when rows > cols);
 *   5 quintic Newton-Schulz iterations  X <- aX + (bA + cA^2)X,  A = XX^T,
 *     (a, b, c) = (3.4445, -4.7750, 2.0315);
 *   W <- W*(1 - lr*wd) - lr * 0.2*sqrt(max(A, B)) * O.
 *
 * Sources (web pages; titles and sections):
 *   "迎接DeepSeek开源周[Kimi先开为敬]发布开源最新Muon优化器可替代AdamW计算效率直接翻倍"
 *     (coreui.cn): §1 权重衰减机制 (decoupled decay), §2 参数更新尺度调整
 *     (0.2*sqrt(max(A,B))), §代码 (the printed Muon class: momentum,
 *     Nesterov, update order, and its AdamW backup).
 *   "DeepSpeed 集成 Muon 优化器实战从正交化原理到 ZeRO 微调配置" (lshu.cn):
 *     §核心算子牛顿-舒尔茨正交化内核 (quintic coefficients, the standard and
 *     gram methods), §use_muon 参数打标 (which parameters take Muon), TL;DR
 *     (Muon Split: per-head orthogonalisation).
 *   "Muon 优化器" (MindSpeed feature doc, gitcode.com): §TP 兼容适配 item 4
 *     (QKV split).
 *   "Muon Optimizer and the Distributed Implementation" (blog.chensy.moe):
 *     §Newton-Schulz Iteration (Frobenius normalisation, the iteration).
 *
 * Conventions for every entry point:
 *   - Tensor pointers are DEVICE pointers owned by the caller; matrices are
 *     row-major and contiguous (row stride = number of columns).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously; functions return after the
 *     launches are queued.  Host-side argument errors are reported before
 *     anything is enqueued.
 *   - A handle owns its device workspace and a device error word.  Calls on
 *     one handle must be ordered (same stream, or externally synchronised).
 *   - Errors that can only be seen on the device (a bounded wait that timed
 *     out, a non-finite gradient norm) are recorded in the error word and
 *     returned by muon_handle_check().
 *   - No C++ exception crosses this ABI; nothing aborts the process.
 */
#ifndef MUON_GB300_H_
#define MUON_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MUON_OK = 0,
  MUON_ERR_INVALID_ARG = 1,   /* bad pointer, shape, dtype or count */
  MUON_ERR_UNSUPPORTED = 2,   /* valid request this library does not run (e.g. no sm_103a device) */
  MUON_ERR_WORKSPACE = 3,     /* device or pinned workspace allocation failed */
  MUON_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed; see muon_last_error() */
  MUON_ERR_NONFINITE = 5,     /* a Frobenius norm was NaN/Inf (from muon_handle_check) */
  MUON_ERR_TIMEOUT = 6        /* a bounded device wait ran out (from muon_handle_check) */
} muon_status_t;

typedef enum { MUON_F32 = 0, MUON_BF16 = 1 } muon_dtype_t;

/* Newton-Schulz method: "standard" iterates on X; "gram" iterates on the
 * small square R = XX^T and applies the accumulated polynomial to X0 once
 * (DeepSpeed's NS_METHODS {standard, gram}).  MUON_NS_AUTO (no counterpart
 * on the pages) chooses per same-shape group, after the rows <= cols rule:
 * gram on the bf16 path when n >= 4m, where it measured faster on this GPU,
 * standard otherwise and on the fp32 paths; a call with both kinds of
 * group runs as two calls in turn on the same stream. */
typedef enum { MUON_NS_STANDARD = 0, MUON_NS_GRAM = 1, MUON_NS_AUTO = 2 } muon_ns_method_t;

typedef struct muon_handle_s* muon_handle_t;

/* One Muon parameter (2-D; callers flatten higher-rank weights to
 * (size(0), -1) and pass the original first two dims' max as scale_dim). */
typedef struct {
  void* param;            /* rows x cols, param_dtype, updated in place        */
  const void* grad;       /* rows x cols, grad_dtype, read only                */
  float* momentum;        /* rows x cols fp32, updated in place (zero at start)*/
  int64_t rows, cols;
  int32_t param_dtype;    /* muon_dtype_t */
  int32_t grad_dtype;     /* muon_dtype_t */
  int32_t split_heads;    /* >= 1; rows are split into this many equal blocks,
                             each orthogonalised on its own (Muon Split)      */
  int32_t reserved;       /* must be 0 */
  int64_t scale_dim;      /* max(A, B) of the update scale; 0 = max(rows, cols) */
} muon_param_t;

/* Create a handle on CUDA device `device`.  Checks that the device is
 * sm_103 (GB300) and resolves the tensor-map encoder.  *out is NULL on error.
 * Groups with m a multiple of 256 (or m >= 2048) run the GEMMs of the bf16
 * path on two-SM CTA pairs (256 x 256 tiles); groups with a ragged last
 * 256-row tile and m >= 1024 run their symmetric products on pairs and the
 * update products on one SM.  The environment variables, read when the
 * handle is created: MUON_TC_PAIR selects the one-SM kernels everywhere
 * ("0") or pairs for the symmetric products only ("sym");
 * MUON_TC_PAIR_MIN_M (default 1024) moves the ragged-m threshold;
 * MUON_FINAL_TMA=0 makes the last product write bf16 parameters element-wise
 * instead of through per-parameter tensor maps (same results, bit for bit). */
muon_status_t muon_handle_create(muon_handle_t* out, int device);

/* Destroy a handle: synchronises the device, frees the workspace. NULL is a no-op. */
muon_status_t muon_handle_destroy(muon_handle_t h);

/* Upper bound on the NS workspace one call may allocate (default 16 GiB);
 * same-shape groups larger than this are processed in chunks. */
muon_status_t muon_handle_set_workspace_limit(muon_handle_t h, size_t bytes);

/* Time limit of every bounded device wait (default 4 s). */
muon_status_t muon_handle_set_timeout_ns(muon_handle_t h, uint64_t timeout_ns);

/* Synchronise `stream`, read and clear the device error word: MUON_OK,
 * MUON_ERR_TIMEOUT or MUON_ERR_NONFINITE (timeout wins if both are set). */
muon_status_t muon_handle_check(muon_handle_t h, void* stream);

/* Orthogonalise `batch` independent m x n matrices in place:
 *   X[i] <- NS_steps(X[i] / ||X[i]||_F)
 * ("Muon Optimizer and the Distributed Implementation", §Newton-Schulz
 * Iteration; "DeepSpeed 集成 Muon 优化器实战", §核心算子).
 *   X       device, [batch][m][n] row-major, dtype; overwritten by O
 *   dtype   MUON_BF16: bf16 tensor-core path (bf16 operands, fp32
 *           accumulation, master X kept as a bf16 plane hi plus one byte
 *           with its next 8 bits, about 16 significant bits); MUON_F32:
 *           fp32 path (tensor cores with three bf16 planes per operand up
 *           to m = 2048, CUDA cores above)
 *   steps   >= 0 (0 returns the normalised input)
 *   coeffs  host pointer to (a, b, c); NULL = (3.4445, -4.7750, 2.0315)
 *   ns_method  muon_ns_method_t
 * Matrices with m > n are iterated on the transpose.  A zero matrix gives
 * zeros.  batch == 0, m == 0 or n == 0 is a valid no-op. */
muon_status_t muon_orthogonalize(muon_handle_t h, void* X, int32_t dtype, int64_t batch, int64_t m, int64_t n,
                                 int32_t steps, const float* coeffs, int32_t ns_method, void* stream);

/* One Muon step over `n_params` parameters (host array of descriptors):
 * momentum (+Nesterov), Frobenius normalisation, `ns_steps` Newton-Schulz
 * iterations per matrix or per row block, then
 *   W <- W*(1 - lr*wd) - lr * update_rms*sqrt(scale_dim) * O
 * ("迎接DeepSeek开源周…Muon优化器", §代码 and §2 参数更新尺度调整;
 * update_rms = 0.2 there).
 * Same-shape matrices (after the rows <= cols transpose rule, counting
 * Muon-Split blocks and transposed matrices together) are batched into
 * grouped persistent launches.
 *   ns_dtype  MUON_BF16: tensor-core path; MUON_F32: fp32 path.
 * n_params == 0 is a valid no-op.  params is read during the call only. */
muon_status_t muon_step(muon_handle_t h, const muon_param_t* params, int32_t n_params, float lr, float wd,
                        float mu, int32_t nesterov, int32_t ns_method, int32_t ns_steps, const float* coeffs,
                        float update_rms, int32_t ns_dtype, void* stream);

/* Update scale of muon_step_ex:
 *   MUON_SCALE_RMS  update_rms * sqrt(scale_dim), scale_dim = max(A, B) by
 *                   default: matches the update RMS to AdamW's
 *                   ("迎接DeepSeek开源周…Muon优化器", §2 参数更新尺度调整, 0.2);
 *                   DeepSeek-V4's sqrt(max(n, m)) * gamma is this mode with
 *                   update_rms = gamma ("Muon Optimizer and the Distributed
 *                   Implementation", §Variation).
 *   MUON_SCALE_MUP  sqrt(d_out / d_in) = sqrt(rows / cols) of the parameter
 *                   as stored (out x in): the dual of the gradient under the
 *                   RMS -> RMS operator norm has spectral norm
 *                   sqrt(d_out / d_in) (same page and section, the muP form).
 * In both modes the update is further multiplied by extra_scale (MindSpeed's
 * "--muon-extra-scale-factor", "Muon 优化器" feature doc, parameter table). */
typedef enum { MUON_SCALE_RMS = 0, MUON_SCALE_MUP = 1 } muon_scale_mode_t;

typedef struct {
  float lr;                /* learning rate */
  float wd;                /* decoupled weight decay: W <- W * (1 - lr * wd) first */
  float mu;                /* momentum */
  int32_t nesterov;        /* 1: U = G + mu * M_new; 0: U = M_new */
  int32_t ns_method;       /* muon_ns_method_t */
  int32_t ns_steps;        /* 0 .. 100 */
  const float* coeffs;     /* host (a, b, c) or NULL for (3.4445, -4.7750, 2.0315) */
  int32_t ns_dtype;        /* MUON_BF16: tensor-core path; MUON_F32: fp32 path */
  int32_t scale_mode;      /* muon_scale_mode_t */
  float update_rms;        /* MUON_SCALE_RMS factor (0.2); ignored by MUON_SCALE_MUP */
  float extra_scale;       /* multiplies the update in every mode (1.0) */
  int32_t coeffs_per_step; /* 0: coeffs is one (a, b, c) used by every step; 1: coeffs holds ns_steps
                              triples, step k uses coeffs[3k .. 3k+2] (a schedule such as the
                              hybrid iteration of DeepSeek-V4: "Muon Optimizer and the Distributed
                              Implementation", §Variation of Muon Optimizer) */
} muon_step_options_t;

/* muon_step with the update scale chosen by opts (host struct, read during
 * the call only):
 *   W <- W*(1 - lr*wd) - lr * extra_scale * scale(mode) * O
 * Everything else as muon_step, which equals muon_step_ex with
 * MUON_SCALE_RMS and extra_scale = 1.  Invalid mode or non-finite factors:
 * MUON_ERR_INVALID_ARG before anything is enqueued. */
muon_status_t muon_step_ex(muon_handle_t h, const muon_param_t* params, int32_t n_params,
                           const muon_step_options_t* opts, void* stream);

/* Device workspace, in bytes, that muon_step / muon_step_ex would need for
 * this parameter list on this handle: same-shape groups are processed in
 * chunks sized to the handle's workspace limit
 * (muon_handle_set_workspace_limit), and the workspace must hold the
 * largest chunk.  The handle allocates it on first use, rounded up to a
 * multiple of 64 MiB, keeps it until destroyed, and grows it when a later
 * call needs more; a small descriptor buffer comes on top.  Only shapes,
 * dtypes and split_heads of params are read (pointers may be NULL).
 * Host-only: enqueues nothing.  (Sizing has no counterpart on the source
 * pages; it lets a caller budget device memory before the first step.)
 *   ns_method, ns_steps, ns_dtype: as in muon_step.
 *   bytes: host pointer, receives the size (0 for an empty list). */
muon_status_t muon_workspace_size(muon_handle_t h, const muon_param_t* params, int32_t n_params, int32_t ns_method,
                                  int32_t ns_steps, int32_t ns_dtype, uint64_t* bytes);

/* AdamW fallback for non-Muon parameters (the AdamW backup of the printed
 * Muon class, "迎接DeepSeek开源周…Muon优化器", §代码):
 *   m <- m + (1-beta1)(g - m);  v <- v + (1-beta2)(g^2 - v);
 *   p <- p*(1 - lr*wd) - lr*sqrt(1-beta2^step)/(1-beta1^step) * m/(eps + sqrt(v))
 * Host arrays of `n` device pointers; numel[i] elements each.
 *   params[i]  param_dtypes[i] (MUON_F32 / MUON_BF16), updated in place
 *   grads[i]   grad_dtypes[i], read only
 *   exp_avg[i], exp_avg_sq[i]  fp32, updated in place (zero at start)
 *   step       count after this update (>= 1)
 * n == 0 is a valid no-op. */
muon_status_t adamw_step(muon_handle_t h, void* const* params, const void* const* grads, float* const* exp_avg,
                         float* const* exp_avg_sq, const int64_t* numel, const int32_t* param_dtypes,
                         const int32_t* grad_dtypes, int32_t n, int64_t step, float lr, float beta1, float beta2,
                         float eps, float wd, void* stream);

/* Launch a bounded wait on a barrier that nothing completes, limited to
 * timeout_ns; a following muon_handle_check() returns MUON_ERR_TIMEOUT.
 * Exercises the timeout path without hanging the GPU. */
muon_status_t muon_selftest_timeout(muon_handle_t h, uint64_t timeout_ns, void* stream);

/* Allocation-free orthogonalisation of ONE matrix, for callers that cannot
 * allocate device memory (code inside a CUDA graph capture that forbids
 * allocation, embedded runtimes with a fixed memory budget, processes whose
 * device memory is owned by a custom allocator).  Same result as
 * muon_orthogonalize(batch = 1, ns_method = standard); no handle needed.
 * (The source pages have no counterpart: this is a deployment variant.)
 *   X, dtype, m, n, steps, coeffs, stream: as in muon_orthogonalize.
 * Scratch: a 24 MiB file-scope device array inside the library, held by every
 * GPU that loads the library until the process exits.  Limits:
 * min(m, n) <= 1024 and m*n <= 2^20 elements; larger sizes return
 * MUON_ERR_INVALID_ARG before anything is enqueued.  Calls no cudaMalloc,
 * cudaFree or allocating library routine.  The first call on each device
 * (with that device current) resolves the array's device address
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * Every call shares the one array and leaves its contents behind: calls
 * that may overlap on the GPU (different streams without ordering) race and
 * must be serialised by the caller.  Device-side errors (a bounded wait that
 * ran out, a NaN/Inf Frobenius norm) are OR-ed into an error word at the
 * start of the array, which the first call on each device clears; they
 * collect across calls until muon_noalloc_check() reads and clears them.
 * Every bounded wait gives up after the limit set by
 * muon_noalloc_set_timeout_ns (default 4 s). */
muon_status_t muon_orthogonalize_noalloc(void* X, int32_t dtype, int64_t m, int64_t n, int32_t steps,
                                         const float* coeffs, void* stream);

/* Error readback of muon_orthogonalize_noalloc on the current device:
 * synchronise `stream`, read the error word inside the library's static
 * array, clear it (on `stream`) and return MUON_OK, MUON_ERR_TIMEOUT or
 * MUON_ERR_NONFINITE (timeout wins if both are set).  The errors reported are
 * those of every muon_orthogonalize_noalloc call on this device since the
 * previous check.  Allocates nothing: a copy into a host variable and a
 * memset of the word.  A call of muon_orthogonalize_noalloc still running on
 * another stream races with the clear.  MUON_ERR_CUDA if a CUDA call fails.
 * (No counterpart on the source pages: the handle's muon_handle_check for
 * the allocation-free path.) */
muon_status_t muon_noalloc_check(void* stream);

/* Time limit of every bounded device wait of muon_orthogonalize_noalloc,
 * process-wide, used by calls made after this one (default 4 s).
 * 0: MUON_ERR_INVALID_ARG. */
muon_status_t muon_noalloc_set_timeout_ns(uint64_t timeout_ns);

/* Kernel classes reported by muon_handle_profile(). */
enum {
  MUON_K_PREPARE = 0, /* momentum / Nesterov / norm partials / working copy */
  MUON_K_NORM = 1,    /* per-matrix 1/||U||_F                               */
  MUON_K_SYRK = 2,    /* A = X X^T                                          */
  MUON_K_POLY = 3,    /* B = bA + cA^2                                      */
  MUON_K_UPDATE = 4,  /* X = aX + BX                                        */
  MUON_K_FINAL = 5,   /* last update fused with the parameter write         */
  MUON_K_APPLY = 6,   /* parameter write when no NS iteration runs          */
  MUON_K_ADAMW = 7,   /* AdamW fallback                                     */
  MUON_K_COUNT = 8
};

/* Enable (1) or disable (0) per-launch CUDA-event timing on the launching
 * stream.  Enabling discards earlier records. */
muon_status_t muon_handle_set_profiling(muon_handle_t h, int32_t enable);

/* Wait for the recorded launches, then write per-class total milliseconds and
 * launch counts into host arrays of n_classes (<= MUON_K_COUNT) entries and
 * clear the records.  Either array may be NULL. */
muon_status_t muon_handle_profile(muon_handle_t h, double* ms, int64_t* launches, int32_t n_classes);

/* Like muon_handle_profile, but one record per launch: kernel class,
 * group tag (index of the launch's same-shape group within its call, groups
 * in ascending (m, n) order; -1 for AdamW) and milliseconds.  Writes at most
 * `capacity` records into the host arrays, stores the number of records in
 * *count (which may exceed capacity) and clears the records. */
muon_status_t muon_handle_profile_records(muon_handle_t h, int32_t* cls, int32_t* tag, float* ms, int32_t capacity,
                                          int32_t* count);

/* Number of kernels this handle has launched since it was created. */
muon_status_t muon_handle_launch_count(muon_handle_t h, uint64_t* count);

/* Static description of a status code. */
const char* muon_status_string(muon_status_t s);

/* Detail of the last failing call on this handle ("" if none). */
const char* muon_last_error(muon_handle_t h);

/* ABI version: major*10000 + minor*100 + patch. */
int32_t muon_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MUON_GB300_H_ */
