/*
 * liblla: causal Local Linear Attention (LLA) forward on one NVIDIA GB300 (sm_103a).
 *
 * Definition (the operation every entry point below serves)
 * ---------------------------------------------------------
 * "Parallax" (Tilde Research blog), section 2 "Parallax & Local Linear Attention",
 * paragraph "Canonical Formulation"; the same definition in "Parallax: Parameterized Local
 * Linear Attention for Language Modeling" (arXiv 2605.29157), section 2, LLA paragraph.
 * For each query q_i (0-based position i) over its causal prefix j <= i (diagonal included),
 * LLA fits the local linear estimator b + W (x - q_i) to the pairs (k_j, v_j) by weighted
 * least squares with kernel weights w_ij = exp(q_i . k_j / h) and ridge penalty
 * lambda * ||W||_F^2, and outputs the intercept b. In closed form
 *     o_i = vbar_i + C_vk (C_kk + lambda I)^-1 (q_i - kbar_i),
 * with kbar, vbar the w-weighted means and C_kk, C_vk the (unnormalised) w-weighted centred
 * second moments. lambda is absolute against the raw weights exp(q.k/h); h divides the logit.
 *
 * Conventions shared by all entry points
 * --------------------------------------
 * - Layout: q, k are [B, H, T, d] and v, out are [B, H, T, dv], contiguous, row-major
 *   (innermost index = feature). Element type is given by `dtype` (lla_dtype) and is the same
 *   for q, k, v and out. Sums are accumulated in fp32 (in compensated fp32 pairs for the fp32
 *   element type). For bf16 inputs the forward runs on the tensor cores: the kernel weights enter
 *   the contraction rounded to bf16, the key products k_a*k_b exactly (as an exact pair of bf16
 *   values). With d < 64 it runs on zero-padded copies of q, k and v (d = dv = 64; zero features
 *   leave the intercept unchanged: their moments are exactly zero, so the ridge system is block-
 *   diagonal with a zero right-hand side on the padded block), at the cost of the padded work.
 * - Pointers named *_host are host memory; every other data pointer is device memory of the
 *   current CUDA device, 16-byte aligned. The caller owns every buffer; `out` must not overlap
 *   an input.
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream). Calls are
 *   asynchronous on that stream unless stated otherwise; they return after validating the
 *   arguments and enqueueing work.
 * - Errors: every call returns an lla_status. Argument errors are detected on the host before
 *   any work is enqueued and leave all buffers untouched. Numerical failures inside a kernel
 *   (a non-positive pivot in a ridge solve, e.g. from non-finite inputs) are recorded in a
 *   per-device status word read by lla_stream_status(); the affected output rows are NaN. (The
 *   forward first retries such a row: in float64 from its moments on the tensor-core path, or,
 *   when its causal prefix holds at most 64 keys, exactly from q, k and v; only a row that still
 *   fails -- non-finite inputs, or a longer prefix with fewer than d + 1 affinely independent
 *   keys under a tiny effective ridge -- is reported.) No entry point aborts, traps or exits.
 * - Supported sizes: d, dv in {16, 32, 64}; B, H, T >= 0 with B*H*T < 2^31 (B*H*T == 0 is a
 *   no-op that returns LLA_OK); h > 0 and lambda > 0, both finite.
 */
#ifndef LLA_H
#define LLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LLA_VERSION_MAJOR 0
#define LLA_VERSION_MINOR 2
#define LLA_VERSION_PATCH 0

typedef enum {
  LLA_OK = 0,
  LLA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad h/lambda/dtype, negative size       */
  LLA_ERR_UNSUPPORTED = 2, /* d or dv outside {16, 32, 64}, or B*H*T >= 2^31                     */
  LLA_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed                         */
  LLA_ERR_NUMERICAL = 4,   /* a ridge solve met a non-positive pivot (rows set to NaN)            */
  LLA_ERR_TIMEOUT = 5      /* a bounded device-side wait gave up (kernel returned early)          */
} lla_status;

typedef enum { LLA_F32 = 0, LLA_BF16 = 1 } lla_dtype;

/* Implementation choices (lla_options.path). */
typedef enum {
  LLA_PATH_AUTO = 0,        /* tensor cores for bf16 (the forward: any d, zero-padded to 64 when
                               d < 64; the other ops: d = dv = 64), CUDA cores otherwise */
  LLA_PATH_CUDA_CORE = 1,   /* CUDA cores always */
  LLA_PATH_TENSOR_CORE = 2, /* tensor cores wherever supported (currently the same as AUTO) */
  LLA_PATH_CG = 3           /* lla_forward*_ex only: matrix-free conjugate gradients for the ridge
                               systems (bf16 with dv = 64 or d < 64; as AUTO elsewhere) */
} lla_path;

/* Closed form of the LLA intercept that a forward evaluates (lla_options.form). */
typedef enum { LLA_FORM_CENTRED = 0, LLA_FORM_PAGE = 1 } lla_form;

/* Test-only faults (lla_options.test_fault). */
typedef enum {
  LLA_FAULT_NONE = 0,
  LLA_FAULT_WITHHOLD_KEYS = 1 /* the tensor-core moments stage's key loader never stages its first
                                 key block, so the waits on it run out (see lla_forward_ex) */
} lla_test_fault;

/*
 * Per-call options of the *_ex entry points. An all-zero struct (or a NULL pointer) selects the
 * defaults, which are what the entry points without options use. Options belong to the one call
 * they are passed to: nothing is remembered between calls, so concurrent callers cannot change
 * each other's results.
 *   path         lla_path (the operations other than the forward accept AUTO, CUDA_CORE and
 *                TENSOR_CORE; CUDA_CORE selects their CUDA-core kernels).
 *   form         lla_form (forward only), see lla_forward_ex.
 *   cg_max_iters conjugate-gradient iteration cap, 1..1024 (0 = 1024), LLA_PATH_CG only.
 *   cg_rel_tol   CG stopping tolerance in (0, 1) (0 = 1e-3), LLA_PATH_CG only.
 *   test_fault   lla_test_fault (forward only; 0 in normal use).
 * Any other value of a field makes the call return LLA_ERR_INVALID_ARG before any work.
 */
typedef struct lla_options {
  int path;
  int form;
  int cg_max_iters;
  float cg_rel_tol;
  int test_fault;
  int reserved[3]; /* must be zero */
} lla_options;

/* Number of timed stages recorded per lla_forward call by the profiling hooks below:
 * 0 prep (per-head means, CUDA-core path; the tensor-core path's key frame runs beside stage 1
 * and is counted there), 1 weights (tensor-core path: row maxima, the weights and their sums),
 * 2 moments (the moment contraction; on the CUDA-core path also the weights), 3 solve,
 * 4 readout (with the exact pass over listed short prefixes beside it). A stage that a path does
 * not have records zero time. */
#define LLA_NUM_STAGES 5

/*
 * Causal LLA forward (the operation defined at the top of this header).
 * q, k: [B,H,T,d]; v: [B,H,T,dv]; out: [B,H,T,dv]; all device, element type `dtype`.
 * Scratch memory is taken from the CUDA stream-ordered allocator on `stream`
 * (cudaMallocAsync/cudaFreeAsync, released at the end of the call in stream order);
 * lla_workspace_size() tells how much. Use lla_forward_ws() to supply it yourself.
 * Rows whose causal prefix holds few keys may be recomputed exactly in float64 (the solve lists
 * them); that pass runs on a library-owned side stream of the current device, at its highest
 * priority, ordered after this call's solve and before the rest of the call by two events, so
 * that to the caller the whole call is still ordered on `stream`. The side stream and its events
 * are created on a device's first forward call (make that call before any stream capture); a
 * call captured into a CUDA graph forks to the side stream and joins back within the capture.
 */
int lla_forward(const void* q, const void* k, const void* v, void* out, int B, int H, int T,
                int d, int dv, float h, float lambda, int dtype, void* stream);

/* Bytes of device scratch lla_forward_ws needs for these sizes (0 for invalid sizes).
 * Host-only; touches no device. */
size_t lla_workspace_size(int B, int H, int T, int d, int dv, int dtype);

/*
 * lla_forward with caller-provided device scratch `workspace` (256-byte aligned, at least
 * lla_workspace_size(...) bytes, not used by anything else until the work on `stream` is done).
 * Allocates nothing. Returns LLA_ERR_INVALID_ARG if the workspace is missing or too small.
 */
int lla_forward_ws(const void* q, const void* k, const void* v, void* out, int B, int H, int T,
                   int d, int dv, float h, float lambda, int dtype, void* workspace,
                   size_t workspace_bytes, void* stream);

/*
 * lla_forward / lla_forward_ws with per-call options (opts may be NULL: the defaults). workspace
 * may be NULL (scratch from the stream-ordered allocator, as lla_forward) or caller-provided as
 * for lla_forward_ws (the size does not depend on the options).
 *
 * - opts->path: LLA_PATH_CUDA_CORE forces the CUDA-core moments, solve and readout for every
 *   shape; LLA_PATH_CG solves the per-query ridge systems by conjugate gradients instead of
 *   accumulating the d x d moments and factoring them: each product with C_kk is one streaming
 *   pass over the prefix, as the "Parallax" blog (s.2 "Difficulties in Scaling LLA") describes
 *   exact LLA being computed. Each query row iterates until ||r|| <= cg_rel_tol ||r_0|| (r the
 *   residual of (C_kk + lambda' I) y = q - kbar, r_0 = q - kbar) or cg_max_iters passes have run.
 *   A call on this path synchronises its stream every 8 iterations on the host to test whether any
 *   query tile is still iterating, so it blocks the calling thread and cannot be captured in a
 *   CUDA graph. Paths AUTO, CUDA_CORE and TENSOR_CORE compute the same moments; CG solves the
 *   same systems iteratively.
 * - opts->form ("Parallax" blog, s.2 Canonical Formulation and Appendix B; both forms equal the
 *   intercept of the weighted ridge regression):
 *     LLA_FORM_CENTRED (default) o = vbar + C_vk y,  (C_kk + lambda' I) y = q - kbar;
 *     LLA_FORM_PAGE  o = sum w (1 - z.rho*) v / sum w (1 - z.rho*),  z = k - q,
 *       (sum w z z^T + lambda' I) rho* = sum w z, evaluated as the exact-LLA two-branch epilogue
 *       (O1 - O2) / (d1 - d2). It runs on the tensor-core dense strategy only (bf16 with dv = 64
 *       or d < 64, path AUTO or TENSOR_CORE; otherwise LLA_ERR_UNSUPPORTED). Its system carries the rank-one
 *       term w (kbar - q)(kbar - q)^T on top of the centred one, so it is worse conditioned for
 *       queries far from the weighted key mean.
 * - opts->test_fault = LLA_FAULT_WITHHOLD_KEYS exercises the bounded device waits: the
 *   tensor-core moments stage (bf16; LLA_ERR_UNSUPPORTED on other paths) never stages
 *   its first key block, so every wait that needs it gives up after the wait limit (~2 s), the
 *   stage returns early without issuing the tensor-core work that depends on it, and
 *   LLA_ERR_TIMEOUT is recorded in the status word (lla_stream_status). The output of such a call
 *   is undefined; the stream and the device stay usable. For tests only.
 */
int lla_forward_ex(const void* q, const void* k, const void* v, void* out, int B, int H, int T,
                   int d, int dv, float h, float lambda, int dtype, const lla_options* opts,
                   void* workspace, size_t workspace_bytes, void* stream);

/* Size of the fixed device scratch that lla_forward_noalloc uses: 64 MiB. */
#define LLA_NOALLOC_SCRATCH_BYTES (64ull << 20)

/*
 * lla_forward for callers that cannot allocate device memory. (The pages have no counterpart:
 * this is a deployment convenience, not part of the method.)
 *
 * Some callers are not allowed to allocate GPU memory themselves -- a plugin that its host
 * application only hands input and output buffers, or a latency-critical loop that must not call
 * the allocator while it runs, since an allocation can block on the device or fail under memory
 * pressure at an unpredictable moment. This entry point calls no allocator at all: its scratch is
 * one fixed array of LLA_NOALLOC_SCRATCH_BYTES in device memory owned by the library, which every
 * GPU that loads this part of the library keeps until the process exits. The caller still passes
 * q, k, v and out exactly as for lla_forward, and the result is the same.
 *
 * - Size limit: returns LLA_ERR_UNSUPPORTED, before touching the device, when
 *   lla_workspace_size(B, H, T, d, dv, dtype) exceeds LLA_NOALLOC_SCRATCH_BYTES (e.g. bf16
 *   d = dv = 64 fits T <= 4343 at B*H = 1 and T <= 704 at B*H = 8; the tensor-core path's weight
 *   scratch grows with B*H*T^2). Other argument errors are those of lla_forward.
 * - Set-up: the first call on each device looks up the scratch array's device address (with that
 *   device current) and caches it, and (as any first forward call) creates the side stream of the
 *   exact short-prefix pass; make that first call before any stream capture.
 * - Sharing: all calls on a device share the one array. Calls whose work overlaps on the GPU
 *   (other streams, other host threads, without ordering between them) race on it and corrupt
 *   each other's results; order them on one stream or synchronise between them. Each call
 *   overwrites whatever an earlier call left, and nothing from an earlier call is read.
 */
int lla_forward_noalloc(const void* q, const void* k, const void* v, void* out, int B, int H,
                        int T, int d, int dv, float h, float lambda, int dtype, void* stream);

/*
 * End-to-end variant on HOST buffers: copies q_host, k_host, v_host to the device on `stream`,
 * runs the forward, copies the result to out_host and synchronises `stream` before returning.
 * Host buffers may be pageable or pinned (pinned copies overlap better). Device buffers and
 * scratch come from the stream-ordered allocator and are released before the call returns.
 * Returns the forward's status, including any device status recorded by this call's kernels.
 */
int lla_forward_host(const void* q_host, const void* k_host, const void* v_host, void* out_host,
                     int B, int H, int T, int d, int dv, float h, float lambda, int dtype,
                     void* stream);

/*
 * Debug entry: raw max-shifted kernel-weighted moments for n selected queries (the sums from
 * which the pages' omega_i, mu_i and Sigma_i follow, "Parallax" blog s.2 Canonical
 * Formulation). idx[n] (device, int64) holds flat query indices (b*H + hh)*T + i.
 * For each selected query: m = max_{j<=i} q_i.k_j/h, w_j = exp(q_i.k_j/h - m) and
 *   m[n], omega[n] = sum w_j, sk[n,d] = sum w_j k_j, sv[n,dv] = sum w_j v_j,
 *   Skk[n,d,d] = sum w_j k_j k_j^T, Svk[n,dv,d] = sum w_j v_j k_j^T   (fp32, device, row-major).
 * Any output pointer may be NULL to skip it. Accumulation is in fp64 (not a fast path).
 * An out-of-range idx entry sets LLA_ERR_INVALID_ARG in the device status word and leaves that
 * query's outputs untouched.
 */
int lla_moments(const void* q, const void* k, const void* v, const int64_t* idx, int n,
                float* m, float* omega, float* sk, float* sv, float* Skk, float* Svk,
                int B, int H, int T, int d, int dv, float h, int dtype, void* stream);

/*
 * Causal Parallax forward with a given probe ("Parallax" blog, s.2 paragraph "Parallax" and
 * Appendix B with eta = 0; streaming form in s.3 "One extra branch, no extra I/O"; output
 * combination as printed in Appendix C): for each query i over its causal prefix j <= i,
 *     o_i = o_SA_i - Sigma_KV^(i) r_i = (1 + d2/d1) O1/d1 - O2/d1,
 * where p_ij = exp(q_i . k_j / h) / sum_l exp(q_i . k_l / h) are the softmax weights, o_SA_i =
 * sum_j p_ij v_j, Sigma_KV^(i) = sum_j p_ij (v_j - vbar_i)(k_j - kbar_i)^T (dv x d), and in the
 * streaming form P1 = exp(q.k/h), P2 = P1 * (r_i . k_j), O1 = P1 V, O2 = P2 V, d1 = sum P1,
 * d2 = sum P2. r = 0 gives causal softmax attention with scale 1/h.
 * q, k, r: [B,H,T,d]; v, out: [B,H,T,dv]; all device, element type `dtype`, 16-byte aligned; the
 * conventions at the top of this header apply (lambda plays no part). bf16 inputs with
 * d = dv = 64 run on the tensor cores (weights rounded to bf16, P2 as an exact hi/lo bf16 pair,
 * fp32 accumulation); everything else runs on the CUDA cores in fp32 (lla_parallax_forward_ex
 * with path LLA_PATH_CUDA_CORE forces them for every shape). Allocates nothing. Non-finite inputs
 * give non-finite outputs; no status is recorded.
 */
int lla_parallax_forward(const void* q, const void* k, const void* v, const void* r, void* out,
                         int B, int H, int T, int d, int dv, float h, int dtype, void* stream);
int lla_parallax_forward_ex(const void* q, const void* k, const void* v, const void* r, void* out,
                            int B, int H, int T, int d, int dv, float h, int dtype,
                            const lla_options* opts, void* stream);

/*
 * Decode: one query per head against a key/value cache of L positions that the query attends to
 * in full (it is the newest token; its own key and value are already appended). The output is
 * what lla_forward returns for its last row, o = vbar + C_vk (C_kk + lambda I)^-1 (q - kbar) with
 * w_j = exp(q . k_j / h) over all L positions ("Parallax" blog, s.2 Canonical Formulation).
 * q: [B,H,d]; k: [B,H,L,d]; v: [B,H,L,dv]; out: [B,H,dv]; device, element type `dtype`, 16-byte
 * aligned; d, dv in {16, 32, 64}; B*H*L < 2^31; h, lambda finite and positive. The cache of each
 * head is split over several CTAs that reduce their chunk to partial moments (float32, shifted by
 * a maximum logit of the chunk); the last CTA of the head to finish merges them and solves the
 * ridge system in float64 (split-KV with a last-arriver merge, as the blog's decode kernel,
 * Appendix C). For bf16 with d = dv = 64 the chunk's second moments run on the tensor cores
 * (weights rounded to bf16, exact products, float32 sums) unless lla_decode_ex is given path
 * LLA_PATH_CUDA_CORE; otherwise on the CUDA cores with float32 weights. Asynchronous on `stream`; scratch from the stream-ordered pool. B*H = 0 is a
 * no-op; L = 0 with B*H > 0 is LLA_ERR_INVALID_ARG. A non-positive pivot (non-finite inputs)
 * makes that head's output NaN and records LLA_ERR_NUMERICAL.
 */
int lla_decode(const void* q, const void* k, const void* v, void* out, int B, int H, int L, int d,
               int dv, float h, float lambda, int dtype, void* stream);
int lla_decode_ex(const void* q, const void* k, const void* v, void* out, int B, int H, int L,
                  int d, int dv, float h, float lambda, int dtype, const lla_options* opts,
                  void* stream);

/*
 * Parallax decode with probe r ([B,H,d], same dtype): o = vbar - Sigma_KV r over all L cached
 * positions, as lla_parallax_forward's last row, computed as the blog's streaming combination
 * (1 + d2/d1) O1/d1 - O2/d1 (Appendix C) with the same split-KV and last-arriver merge as
 * lla_decode (float32 partials, the merge in float64). Otherwise as lla_decode (lambda plays no
 * part; no status is recorded).
 */
int lla_parallax_decode(const void* q, const void* k, const void* v, const void* r, void* out,
                        int B, int H, int L, int d, int dv, float h, int dtype, void* stream);
int lla_parallax_decode_ex(const void* q, const void* k, const void* v, const void* r, void* out,
                           int B, int H, int L, int d, int dv, float h, int dtype,
                           const lla_options* opts, void* stream);

/*
 * Causal Parallax backward ("Parallax" blog, Appendix F "Parallax backward (closed form)": a
 * forward-like pass caches per-row scalars, then a row-tile pass and a column-tile pass). Given
 * the inputs of lla_parallax_forward (q, k, r: [B,H,T,d]; v: [B,H,T,dv]) and the upstream
 * gradient dout = dL/do ([B,H,T,dv]), writes dq = dL/dq, dk, dr ([B,H,T,d]) and dv ([B,H,T,dv]).
 * The appendix's formulas were lost in extraction; the gradients are those of the forward itself
 * (o_i = sum_j p_ij (1 + tbar_i - t_ij) v_j with p_i = softmax of q_i.k_j / h over j <= i,
 * t_ij = r_i . k_j, tbar_i = sum_j p_ij t_ij). All buffers are device pointers, contiguous
 * row-major, 16-byte aligned, of the dtype given (gradients in the inputs' dtype; fp32
 * arithmetic); the caller owns them; outputs must not alias inputs. d, dv in {16, 32, 64}
 * (else LLA_ERR_UNSUPPORTED); h > 0 and finite, B, H, T >= 0 (else LLA_ERR_INVALID_ARG). Three
 * launches, asynchronous on `stream`, with a scratch of 32 bytes per query row from the
 * stream-ordered pool: for bf16 with d = dv = 64, the tensor-core forward kernel caching the row
 * records, then tensor-core row-tile and column-tile passes (tcgen05; weights rounded to bf16,
 * fp32 accumulation); for every other shape (or with path LLA_PATH_CUDA_CORE through
 * lla_parallax_backward_ex), the same three passes on the CUDA cores in fp32. Returns LLA_OK,
 * LLA_ERR_* for invalid arguments, LLA_ERR_CUDA.
 */
int lla_parallax_backward(const void* q, const void* k, const void* v, const void* r,
                          const void* dout, void* dq, void* dk, void* dv, void* dr, int B, int H,
                          int T, int d, int dv_, float h, int dtype, void* stream);
int lla_parallax_backward_ex(const void* q, const void* k, const void* v, const void* r,
                             const void* dout, void* dq, void* dk, void* dv, void* dr, int B,
                             int H, int T, int d, int dv_, float h, int dtype,
                             const lla_options* opts, void* stream);

/*
 * Synchronises `stream`, then reads and clears the current device's status word.
 * Returns LLA_OK, LLA_ERR_NUMERICAL, LLA_ERR_TIMEOUT, LLA_ERR_INVALID_ARG (bad idx in
 * lla_moments) or LLA_ERR_CUDA (a sticky CUDA error or failed synchronisation).
 */
int lla_stream_status(void* stream);

/* Static, NUL-terminated description of a status code (never NULL). */
const char* lla_status_string(int status);

/* LLA_VERSION_MAJOR*10000 + LLA_VERSION_MINOR*100 + LLA_VERSION_PATCH. */
int lla_version(void);

/* Number of kernels this library has launched in this process (all devices, all streams). */
unsigned long long lla_launch_count(void);

/*
 * Stage timing. lla_profile_enable(1) makes every later lla_forward/lla_forward_ws call record
 * CUDA events on its stream at the LLA_NUM_STAGES stage boundaries (no synchronisation is
 * added). lla_profile_collect() waits for the recorded events, writes the summed duration in
 * milliseconds of each stage over all recorded calls to stage_ms[0..min(max_stages,
 * LLA_NUM_STAGES)-1], stores the number of calls in *n_calls (if not NULL), and forgets them.
 * lla_profile_enable(0) stops recording. Returns LLA_OK or LLA_ERR_CUDA.
 */
int lla_profile_enable(int on);
int lla_profile_collect(float* stage_ms, int max_stages, int* n_calls);

#ifdef __cplusplus
}
#endif

#endif /* LLA_H */
