/*
 * libmuon -- the hybrid Muon + AdamW optimizer step on one NVIDIA GB300 (sm_103a).
 *
 * C ABI. Plain pointers and sizes; no C++ or framework types cross it.
 *
 * Sources (web pages, cited by title and section):
 *   [P1] "MuonAdamW vs DistMuonAdamW: Key Differences for Single and Multi-GPU Training in nanochat"
 *   [P2] "Optimizers: AdamW, Muon and the distributed optimizer" (AI-infra handbook)
 *   [P3] "dtensor-muon 0.1.0" package description
 *   [P4] "DMuon: Efficient Distributed Muon Training with Near-Adam Overhead" (summary of arXiv 2606.27153)
 *
 * Conventions for every call:
 *   - Matrices are row-major. A stack (K, A, B) is K matrices of A rows and B columns.
 *   - The caller allocates every buffer: parameters, gradients, optimizer state and the
 *     workspace. The library never allocates or frees device memory and keeps no pointer
 *     after a call returns.
 *   - Device work is enqueued on the caller's stream and is asynchronous: a call returns
 *     once its kernels are launched. Updates are in place.
 *   - Argument checks (null pointers, sizes, dtypes, alignment, workspace size, device
 *     capability) run on the host before anything is launched; a failed check launches
 *     nothing and changes nothing. A failed launch returns MUON_ERR_CUDA.
 *   - Every wait inside a kernel is bounded (default 2 s, muon_set_timeout_ns). A wait
 *     that runs out sets an error word in the workspace and the kernel returns early;
 *     muon_check() reports it as MUON_ERR_TIMEOUT.
 *   - Calls on one stream are ordered. Calls on different streams that share a workspace,
 *     or that touch the same parameters, race.
 */
#ifndef LIBMUON_H
#define LIBMUON_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The CUDA stream type (cudaStream_t). NULL is the legacy default stream. */
typedef struct CUstream_st *muon_stream_t;

typedef enum {
  MUON_OK = 0,
  MUON_ERR_INVALID_ARG = 1,        /* null pointer, non-positive size, bad hyperparameter */
  MUON_ERR_SHAPE = 2,              /* a dimension beyond what the kernels index */
  MUON_ERR_DTYPE = 3,              /* unsupported dtype or dtype combination */
  MUON_ERR_ALIGNMENT = 4,          /* a pointer not aligned as the call states */
  MUON_ERR_WORKSPACE = 5,          /* workspace missing or smaller than muon_workspace_bytes() */
  MUON_ERR_UNSUPPORTED_DEVICE = 6, /* current device is not compute capability 10.3 (GB300) */
  MUON_ERR_CUDA = 7,               /* a CUDA runtime/driver call failed */
  MUON_ERR_TIMEOUT = 8             /* a bounded device-side wait ran out (reported by muon_check) */
} muon_status;

typedef enum { MUON_F32 = 0, MUON_BF16 = 1 } muon_dtype;

#define MUON_MAX_NS_STEPS 32

/* Muon hyperparameters ([P2] "Muon: orthogonalising the update"; [P3] "Key options"). */
typedef struct {
  float lr;            /* eta */
  float momentum;      /* mu: M <- mu*M + G */
  float weight_decay;  /* lambda: decoupled decay p <- p - eta*lambda*p (masked if cautious) */
  int nesterov;        /* 1: orthogonalise G + mu*M (updated M); 0: orthogonalise M */
  int cautious_wd;     /* 1: decay only where u*p > 0 (u: orthogonalised update, p: pre-update param) */
  int scale_mode;      /* 0: update scale 0.2*sqrt(max(A,B)); 1: sqrt(max(1, A/B)) */
  int ns_steps;        /* N, 1..MUON_MAX_NS_STEPS */
  const float *coeffs; /* HOST array, ns_steps*3 floats: (a_t, b_t, c_t) for step t */
  float eps;           /* added to the Frobenius norm before dividing, 1e-7 on the pages */
} muon_hparams;

/* AdamW hyperparameters ([P2] "AdamW: decoupled weight decay"; [P3] "Key options", is_adamw). */
typedef struct {
  float lr, beta1, beta2, eps, weight_decay;
  int32_t l2;   /* 0: decoupled decay (AdamW). 1: L2 regularisation, wd*p joins the gradient before the
                 * moments and nothing decays separately (Adam; the is_adamw=False option) */
  int64_t step; /* t >= 1, the step count after this update; kept by the caller */
} adamw_hparams;

/* Bytes of workspace muon_step_batched / ns_orthogonalize need for a (K, A, B) stack.
 * Layout (all sections 1024-byte aligned): a header of a 256-byte control block (error word)
 * and 4*K 32-bit counters (the norm pass's per-matrix tile count, and the readiness of each
 * matrix's Gram, polynomial and iterate, through which the Newton-Schulz launches can wait per
 * matrix instead of per launch), which every call clears itself before its first launch; then K fp32
 * norm scales, per-tile norm partial sums, two bf16 iterates of (K, min, max) with rows
 * padded to a multiple of 8 elements, two bf16 (K, min, min) Gram buffers, and, for shapes that can take
 * the Gram-space path (muon_debug_gram_space), its scratch.
 * Returns 0 if K, A or B is not positive. */
size_t muon_workspace_bytes(int64_t K, int64_t A, int64_t B);

/* One Muon step on a stack of K same-shape matrices.
 * [P2] "Muon: orthogonalising the update": M <- mu*M + G; U = G + mu*M (nesterov) or M;
 * X = U / (||U||_F + eps) per matrix; if A > B work on X^T; N steps of
 * X <- a_t X + (b_t X X^T + c_t (X X^T)^2) X; transpose back; then
 * p <- p - lr*wd*p*mask - lr*scale*X with mask = 1, or [X*p > 0] if cautious ([P3] "Features").
 *   params    DEVICE array of K device pointers; each points to an A x B row-major matrix of pdt.
 *   grads     DEVICE array of K device pointers; each an A x B row-major matrix of gdt.
 *   momentum  device, fp32, contiguous (K, A, B); updated in place. Zero before the first step.
 *   pdt, gdt  MUON_F32 or MUON_BF16 each.
 *   hp        host struct; hp->coeffs host array of 3*ns_steps floats.
 *   ws        device workspace of ws_bytes >= muon_workspace_bytes(K, A, B), 256-byte aligned, zero-filled
 *             before its first use (its first bytes hold the error word, which only muon_check clears).
 * Limits: 1 <= A, B <= 65536; K * max(A,B) * min(A,B) < 2^40. */
muon_status muon_step_batched(void *const *params, muon_dtype pdt, const void *const *grads, muon_dtype gdt,
                              float *momentum, int64_t K, int64_t A, int64_t B, const muon_hparams *hp, void *ws,
                              size_t ws_bytes, muon_stream_t stream);

/* One same-shape stack of Muon matrices for muon_step_grouped (the arguments muon_step_batched takes,
 * and optionally fp32 master weights). */
typedef struct {
  void *const *params;        /* DEVICE array of K device pointers, each an A x B row-major matrix of pdt */
  const void *const *grads;   /* DEVICE array of K device pointers, each an A x B row-major matrix of gdt */
  float *momentum;            /* device fp32 (K, A, B), updated in place */
  int64_t K, A, B;
  muon_dtype pdt, gdt;
  float *const *master;       /* NULL, or (pdt must be MUON_BF16) a DEVICE array of K device pointers to fp32
                               * A x B master copies: the update (decay, cautious mask, step) is applied to
                               * the master, and the parameter becomes the master rounded to bf16 ([P2] "The
                               * optimizer's memory budget": fp32 master weights beside bf16 weights) */
} muon_bucket;

/* Workspace bytes for muon_step_grouped: one header (control block and four counters per matrix of all
 * buckets), then each bucket's sections as muon_workspace_bytes lays them out.
 * Returns 0 if n < 1, buckets is null or a dimension is not positive. */
size_t muon_workspace_bytes_grouped(const muon_bucket *buckets, int n);

/* One Muon step on n same-shape stacks at once, all with the same hyperparameters: the computation of
 * muon_step_batched on each bucket, with every Newton-Schulz step kind of all buckets issued as one
 * grouped tensor-core launch ([P4] section 2.2, batching matrices of similar shapes; [P1] the stacked
 * (K, ...) Muon groups). Results are identical to n muon_step_batched calls. The step runs in pieces of at
 * most 512 Mi matrix elements (a larger bucket cut along K into equal slices, as muon_step_batched cuts it;
 * smaller consecutive buckets packed into one piece), each piece's whole step before the next: with fewer
 * matrices in flight, consecutive launches find more of their operands in L2 and the power-capped GPU runs
 * faster (muon_debug_piece_elems). Where the launches are short
 * (muon_debug_counter_deps), each waits per matrix on counters in the workspace header that its
 * predecessor raises, rather than on the whole predecessor, so consecutive launches overlap; this
 * changes no result.
 *   buckets   HOST array of n bucket descriptors (1 <= n <= 4096).
 *   ws        device workspace of ws_bytes >= muon_workspace_bytes_grouped(buckets, n), 256-byte aligned,
 *             zero-filled before its first use; its first 256 bytes are the control block muon_check reads.
 * Errors as for muon_step_batched, checked for every bucket before anything is launched. */
muon_status muon_step_grouped(const muon_bucket *buckets, int n, const muon_hparams *hp, void *ws, size_t ws_bytes,
                              muon_stream_t stream);

/* Measured per-shape choices ([P4] section 2.4, shape-adaptive kernel autotuning: configurations searched
 * for the shapes at hand, measured once and cached for later steps). For the buckets of a grouped step with
 * these hyperparameters (the step count and coefficients set the chain's length), the call measures, on the
 * workspace alone, and records in process-wide tables:
 *   1. the Newton-Schulz path of every bucket that can take the Gram-space chain (muon_gram_space_route):
 *      that bucket's chain timed each way, keyed by (min(A,B), max(A,B), K);
 *   1b. the number of contraction slices (1 to 4) of the Gram-space buckets' fp32 Gram, which has one tile
 *      pair per matrix: their fp32 Gram launch timed with each count, keyed by each bucket's
 *      (min(A,B), max(A,B), K) (see muon_autotune_gram_split);
 *   2. the poly step's pipeline shape (mainloop stages + epilogue input slots: 4 + 5, 5 + 3, 6 + 2) for the
 *      plain buckets' grouped poly launch, keyed by its deepest contraction (without an entry, contractions
 *      up to 2048 take 4 + 5 and deeper ones 6 + 2);
 *   3. the plain chain's scheduling (per-matrix readiness counters or launch order) of a step that runs as one
 *      piece: its chains timed each way, keyed by the plain buckets' shapes and counts (a step of several pieces
 *      keeps the rule). Steps 1, 1b and 2 measure each distinct piece on its own.
 * Each candidate runs once as a warm-up and five times timed (median). Later calls use the recorded choices
 * unless a debug switch forces one. The shapes and the scheduling never change a result; the slice count
 * changes only the order of the Gram's fp32 additions; the path changes the arithmetic (both paths are
 * checked against the oracle by the tests).
 *   buckets, n, hp, ws, ws_bytes  as for muon_step_grouped. The timed chains start from whatever the
 *            workspace's iterate holds and write only workspace sections: parameters, gradients and momentum
 *            are neither read nor written.
 * Synchronous: returns after the timed launches complete. Errors as for muon_step_grouped's checks;
 * MUON_ERR_TIMEOUT if a bounded wait ran out during the measurements. */
muon_status muon_autotune(const muon_bucket *buckets, int n, const muon_hparams *hp, void *ws, size_t ws_bytes,
                          muon_stream_t stream);

/* The recorded path of K matrices of A x B: 1 Gram space, 0 plain chain, -1 none recorded. */
int32_t muon_autotune_route(int64_t K, int64_t A, int64_t B);

/* The recorded scheduling of these buckets' plain chain, as a grouped step runs them (in pieces): 1 per-matrix
 * counters, 0 launch order, for every piece with a plain chain; 2 if the pieces' records differ; -1 if a piece
 * has none (or no bucket takes the plain chain). */
int32_t muon_autotune_scheduling(const muon_bucket *buckets, int n);

/* The recorded poly shape (0: 4 + 5, 1: 5 + 3, 2: 6 + 2) for launches whose deepest contraction is
 * `contraction` (the matrices' smaller dimension), or -1 if none is recorded. */
int32_t muon_autotune_poly_shape(int64_t contraction);

/* The recorded number of contraction slices of the Gram-space path's fp32 Gram for a stack of K matrices of
 * A x B, or -1 if none is recorded. Without an entry a stack takes the most slices (up to 4) that would fill
 * one wave of SM pairs with that stack alone while each slice stays at least 1024 deep. The count belongs to
 * the stack, so a stack gets the same bits in any grouped launch and in a call of its own. */
int32_t muon_autotune_gram_split(int64_t K, int64_t A, int64_t B);

/* Empties the autotune tables. */
void muon_autotune_reset(void);

/* Newton-Schulz orthogonalisation of a stack, [P2] "Muon: orthogonalising the update" (newton_schulz):
 * out_k = NS(x_k) for k < K, with normalisation by ||x_k||_F + eps and transpose-to-wide.
 *   x    device, contiguous (K, A, B) of xdt (MUON_F32 or MUON_BF16).
 *   out  device, contiguous (K, A, B) of odt (MUON_F32 or MUON_BF16); may not alias x.
 *   coeffs HOST array of 3*ns_steps floats. ws as for muon_step_batched. */
muon_status ns_orthogonalize(const void *x, muon_dtype xdt, void *out, muon_dtype odt, int64_t K, int64_t A,
                             int64_t B, int ns_steps, const float *coeffs, float eps, void *ws, size_t ws_bytes,
                             muon_stream_t stream);

/* One AdamW step on n elements, [P2] "AdamW: decoupled weight decay":
 * p <- p*(1 - lr*wd); m <- b1*m + (1-b1)*g; v <- b2*v + (1-b2)*g^2;
 * p <- p - lr * (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps).
 * With hp->l2 = 1 (Adam with L2 regularisation, [P2] same section; [P3] is_adamw=False): g <- g + wd*p
 * first, then the same moments and update with no p*(1 - lr*wd) factor. hp->l2 other than 0 or 1 is
 * MUON_ERR_INVALID_ARG.
 *   param, grad  device, n elements of pdt / gdt (MUON_F32 or MUON_BF16 each).
 *   exp_avg, exp_avg_sq  device fp32, n elements each; zero before the first step.
 * Any alignment works; 16-byte aligned pointers take the vectorised path. */
muon_status adamw_step(void *param, muon_dtype pdt, const void *grad, muon_dtype gdt, float *exp_avg,
                       float *exp_avg_sq, int64_t n, const adamw_hparams *hp, muon_stream_t stream);

/* adamw_step for bf16 parameters kept with fp32 master weights ([P2] "The optimizer's memory budget":
 * fp32 master copy, fp32 moments, bf16 weights): the update reads and writes the master, and param
 * receives the new master rounded to bf16 (round to nearest even).
 *   master  device fp32, n elements (the values the update starts from).
 *   param   device bf16, n elements (written only).
 * Other arguments and errors as adamw_step. */
muon_status adamw_step_master(float *master, void *param, const void *grad, muon_dtype gdt, float *exp_avg,
                              float *exp_avg_sq, int64_t n, const adamw_hparams *hp, muon_stream_t stream);

/* One tensor of a grouped AdamW call: the arguments of adamw_step (master NULL) or of adamw_step_master
 * (master set; pdt must then be MUON_BF16), with its own hyperparameters, so that tensors of several
 * parameter groups (say, with and without weight decay: [P2] "AdamW: decoupled weight decay") share
 * one pass. */
typedef struct {
  void *param;               /* device, n elements of pdt */
  const void *grad;          /* device, n elements of gdt */
  float *exp_avg;            /* device fp32, n elements */
  float *exp_avg_sq;         /* device fp32, n elements */
  float *master;             /* NULL, or device fp32, n elements: the master weights taking the update */
  int64_t n;                 /* >= 1 */
  muon_dtype pdt, gdt;
  const adamw_hparams *hp;   /* HOST struct, read during the call only; tensors may share one */
} adamw_tensor;

/* Workspace bytes for adamw_step_grouped and for hybrid_step's adamw_ws: 256 for every 96 tensors
 * (one chunk counter per launch). 0 if n < 1. */
size_t adamw_workspace_bytes_grouped(int64_t n);

/* AdamW on n tensors in one launch per 96 tensors. Each tensor gets exactly the arithmetic of adamw_step
 * (or adamw_step_master), so the results are bit-identical to n separate calls; tensors must not overlap.
 *   tensors  HOST array of n descriptors (1 <= n <= 2^20).
 *   ws       device workspace of ws_bytes >= adamw_workspace_bytes_grouped(n), 256-byte aligned; needs no
 *            initialisation (the call zeroes its counters in stream order). Calls that share ws must be
 *            on one stream.
 * Errors: each tensor's checks as for adamw_step / adamw_step_master, all run before any launch;
 * MUON_ERR_WORKSPACE if ws_bytes is too small, MUON_ERR_ALIGNMENT if ws is not 256-byte aligned. */
muon_status adamw_step_grouped(const adamw_tensor *tensors, int64_t n, void *ws, size_t ws_bytes,
                               muon_stream_t stream);

/* The whole hybrid optimizer step in one call ([P1] "Usage Examples": one optimizer whose step updates the
 * hidden matrices with Muon and every other parameter with AdamW): muon_step_grouped on the buckets, then
 * adamw_step_grouped on the AdamW tensors, on the caller's stream; the results are those of the two calls.
 *   buckets, nb, hp, ws, ws_bytes   as for muon_step_grouped (nb may be 0: AdamW only).
 *   tensors, nt, adamw_ws, adamw_ws_bytes   as for adamw_step_grouped (nt may be 0: Muon only); adamw_ws
 *            may not overlap ws.
 * Errors: every check of both calls runs before anything is launched; MUON_ERR_INVALID_ARG if nb and nt
 * are both 0 or if the two workspaces overlap. */
muon_status hybrid_step(const muon_bucket *buckets, int nb, const muon_hparams *hp, void *ws, size_t ws_bytes,
                        const adamw_tensor *tensors, int64_t nt, void *adamw_ws, size_t adamw_ws_bytes,
                        muon_stream_t stream);

/* ns_orthogonalize without any device allocation. The pages have no counterpart to this call.
 * For callers that cannot allocate device memory and so cannot provide a workspace: code running
 * inside a device-memory allocator's own hooks (allocating there would re-enter the allocator),
 * plugins whose host program gives them no allocation API, runtimes whose device-memory budget is
 * fixed at start-up. Same result and arguments as ns_orthogonalize minus the workspace.
 *   Scratch: a static 64 MiB device array inside the library, held by every GPU that loads the
 *   library until the process exits, laid out as ns_orthogonalize's workspace. A stack fits if
 *   muon_workspace_bytes(K, A, B) <= 64 MiB (about 4*K*A*B + 4*K*min(A,B)^2 bytes plus padding and
 *   16 bytes of counters per matrix); larger stacks return MUON_ERR_WORKSPACE before anything is launched.
 *   The first call on a device (of this function or of the two below) looks up the array's device
 *   address and zeroes its control block (once per device, with that device current, synchronously);
 *   make that first call before any stream capture.
 *   Every call shares the array: calls whose work overlaps on the GPU (other streams, other host
 *   threads) race and must be serialised by the caller. Each call clears the array's per-matrix counters.
 *   The array's error word is sticky: a device-side wait that runs out sets it (the output is then
 *   incomplete), and only ns_orthogonalize_noalloc_check reads and clears it.
 *   The chain runs as separate launches per Newton-Schulz step for every shape.
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library routine. */
muon_status ns_orthogonalize_noalloc(const void *x, muon_dtype xdt, void *out, muon_dtype odt, int64_t K, int64_t A,
                                     int64_t B, int ns_steps, const float *coeffs, float eps, muon_stream_t stream);

/* The check that goes with ns_orthogonalize_noalloc (no counterpart on the pages): synchronises the
 * stream the calls ran on, then reads and clears the built-in scratch's error word with a 4-byte copy into
 * a host variable and a memset (nothing is allocated). Returns MUON_ERR_TIMEOUT if a bounded wait of an
 * ns_orthogonalize_noalloc call on this device ran out since the last check, else MUON_OK. */
muon_status ns_orthogonalize_noalloc_check(muon_stream_t stream);

/* muon_debug_wait_timeout for the built-in scratch: one bounded wait that nothing completes, reporting into
 * the scratch's error word, so that ns_orthogonalize_noalloc_check's report can be tested without a fault.
 * MUON_ERR_INVALID_ARG unless 0 < timeout_ns <= 1e10. */
muon_status muon_debug_wait_timeout_noalloc(uint64_t timeout_ns, muon_stream_t stream);

/* The three tensor-core steps of one Newton-Schulz iteration on contiguous bf16 stacks, exposed
 * one by one ([P2] newton_schulz loop body; [P4] section 2.2 symmetric Gram). The loop body's
 * a*X + (b*A + c*A A) X is computed as (a*I + b*A + c*A A) X, with a folded into the polynomial:
 *   ns_gram:  g = alpha * x x^T,         x (K, m, n), g (K, m, m); symmetric, both halves written.
 *   ns_poly:  h = a*I + b*g + c*g g,     g, h (K, m, m); g must be symmetric.
 *   ns_apply: out = h x,                 h (K, m, m), x and out (K, m, n); out may not alias x.
 * All rows must be 16-byte aligned (m and n multiples of 8), pointers 256-byte aligned.
 * ws: any workspace of at least 256 bytes (only the control block is used). */
muon_status ns_gram(const void *x, void *g, int64_t K, int64_t m, int64_t n, float alpha, void *ws, size_t ws_bytes,
                    muon_stream_t stream);
muon_status ns_poly(const void *g, void *h, int64_t K, int64_t m, float a, float b, float c, void *ws,
                    size_t ws_bytes, muon_stream_t stream);
muon_status ns_apply(const void *h, const void *x, void *out, int64_t K, int64_t m, int64_t n, void *ws,
                     size_t ws_bytes, muon_stream_t stream);

/* Shape bucketing, host only ([P1] "Parameter Processing and Padding": stacking into (K, ...);
 * [P4] section 2.2 "Batching"). Groups n matrices by exact (rows, cols), buckets numbered in
 * order of first appearance; members keep their order.
 *   rows, cols        host arrays of n.
 *   bucket_id, index_in_bucket   host outputs of n.
 *   n_buckets         host output.
 *   bucket_shapes     host output of 2*n (rows, cols per bucket; first 2*n_buckets used).
 *   bucket_K          host output of n (first n_buckets used).
 *   momentum_offset   host output of n: element offset of each bucket's fp32 (K, A, B) momentum
 *                     block in one concatenated buffer (running sum of K*A*B).
 * Returns MUON_ERR_INVALID_ARG for a null pointer with n > 0 or a non-positive dimension. */
muon_status muon_plan_buckets(int64_t n, const int64_t *rows, const int64_t *cols, int64_t *bucket_id,
                              int64_t *index_in_bucket, int64_t *n_buckets, int64_t *bucket_shapes, int64_t *bucket_K,
                              int64_t *momentum_offset);

/* Synchronises the stream, then reads and clears the workspace's error word.
 * Returns MUON_ERR_TIMEOUT if a bounded wait ran out since the last check, else MUON_OK. */
muon_status muon_check(void *ws, muon_stream_t stream);

/* Per-wait limit for device-side waits, in nanoseconds (default 2e9). Applies to later launches. */
void muon_set_timeout_ns(uint64_t ns);

/* Forces every poly launch onto one pipeline shape (0, 1 or 2 as in muon_autotune_poly_shape), or -1
 * to go back to the table and the rule; for tests and sweeps. MUON_ERR_INVALID_ARG outside -1..2. */
muon_status muon_debug_poly_shape(int32_t shape);

/* The Newton-Schulz iteration in the Gram space ([P4] section 2.2, "Efficient Gram Newton-Schulz Iteration"):
 * for a wide iterate X_0 (m x n, m = min(A,B) <= n) the chain runs on m x m matrices, A_0 = X_0 X_0^T,
 * Q_t = a_t I + b_t A_t + c_t A_t^2, R_{t+1} = Q_t R_t, A_{t+1} = Q_t A_t Q_t, and X_N = R_N X_0 -- the same
 * result as the plain iteration, at O(m^3) instead of O(m^2 n) per step. A_0 is accumulated in fp32 from the
 * bf16 iterate; the m x m chain stores every matrix as a bf16 hi / lo pair (16 significant bits) and forms
 * each product in three bf16 tensor-core passes accumulated in fp32; R_N goes to the final product as a bf16
 * hi / lo pair too, and that product applies the parameter update as the plain path's last step does.
 * Shapes that can take it: m <= 256 and not the fused small-matrix kernel's (m <= 128 with n <= 256); their
 * workspace (muon_workspace_bytes) includes 24*K*m*round8(m) + 4*K*m*round64(m) bytes of scratch for it.
 * muon_step_batched, muon_step_grouped, hybrid_step and ns_orthogonalize take it where
 * muon_gram_space_route says so: as measured by muon_autotune for that (m, n, K), else for n >= 4*m.
 * muon_debug_gram_space: -1 the default rule, 0 never, 1 for every shape that can take it (for tests and
 * measurements). MUON_ERR_INVALID_ARG for other values. */
muon_status muon_debug_gram_space(int32_t mode);

/* Runs every Muon call's steps in pieces of at most `elems` matrix elements (a larger stack cut along K into
 * equal slices, smaller consecutive buckets packed together), or the default (512 Mi elements) for 0. Each
 * piece runs its whole step before the next starts; results are the same for any piece size (the fp32 Gram's
 * slice count, which depends on a stack's K, aside: force it with muon_debug_gram_split to compare). For tests
 * and measurements. MUON_ERR_INVALID_ARG for negative values. */
muon_status muon_debug_piece_elems(int64_t elems);

/* Forces the fp32 Gram of the Gram-space path into `split` contraction slices (1 .. 4, clipped per stack to
 * its contraction) in every launch, or -1 to go back to the table and the rule; for tests and sweeps. The
 * slices are added in index order by a second kernel, so a given split always gives the same bits.
 * MUON_ERR_INVALID_ARG for other values. */
muon_status muon_debug_gram_split(int32_t split);

/* 1 if a stack of K matrices of A x B takes the Gram-space path under the current mode and the autotune
 * table, else 0 (also for K, A or B < 1). */
int32_t muon_gram_space_route(int64_t K, int64_t A, int64_t B);

/* Grouped chain scheduling (muon_step_grouped, hybrid_step). 1: each launch of the Newton-Schulz chain
 * waits per matrix on counters its predecessor raises, so that launches overlap. 0: each launch waits for
 * its whole predecessor. -1 (the default): counters where the launches are short (a few hundred
 * microseconds at most), the launch order elsewhere.
 * Results are the same in every mode; for measurements. MUON_ERR_INVALID_ARG for other values. */
muon_status muon_debug_counter_deps(int32_t on);

/* Storage of the symmetric m x m matrices of the Newton-Schulz chain (G = X X^T and the polynomial H).
 * 1 (the default): only their upper 256-blocks are stored, as computed (a diagonal block whole); the steps
 * that read G or H take a block below the diagonal as the transpose of the stored block above it. 0: the
 * strictly upper part is stored and mirrored, and every block is read directly. The tensor cores compute both
 * halves of a diagonal block identically, so results are the same bits either way; for tests and
 * measurements. MUON_ERR_INVALID_ARG for other values. No counterpart on the pages. */
muon_status muon_debug_half_symmetric(int32_t on);

/* Launches one kernel that waits on a barrier nothing will complete, with the given limit,
 * so that the bounded-wait path can be exercised: afterwards muon_check returns MUON_ERR_TIMEOUT. */
muon_status muon_debug_wait_timeout(void *ws, size_t ws_bytes, uint64_t timeout_ns, muon_stream_t stream);

/* Performance analysis: while a buffer is registered, the tensor-core launches that follow write, per CTA
 * and per tile they process (up to records_per_cta), ten 64-bit words: tile index, producer start (before
 * its waits) and last copy issue, MMA start (accumulator free), first and last operands ready, last MMA
 * commit, epilogue start and end, producer first copy issue (globaltimer nanoseconds; 0 = not reached). The buffer is cut into regions of (SM count) *
 * records_per_cta * 10 words; the i-th launch after registration fills region i (record r of CTA c at word
 * (c * records_per_cta + r) * 10 of it) and launches beyond the last region record nothing.
 * buf: device memory, zero-filled by the caller. buf = NULL unregisters. Returns MUON_ERR_WORKSPACE if the
 * buffer holds less than one region. No counterpart on the pages. */
muon_status muon_debug_timeline(void *buf, int64_t bytes, int32_t records_per_cta);

/* Number of kernels this library has launched since it was loaded. */
int64_t muon_launch_count(void);

/* Kernel timing with CUDA events. While enabled, every launch is bracketed by an event pair
 * on its stream (up to 65536 pairs). muon_trace_collect synchronises on the events recorded so far,
 * writes up to cap (kind, milliseconds) pairs and clears the record; it returns the number written,
 * or -1 on a CUDA error. Kinds: see muon_kernel_name. */
void muon_trace_enable(int on);
int64_t muon_trace_collect(int32_t *kinds, float *ms, int64_t cap);
const char *muon_kernel_name(int32_t kind);

const char *muon_status_string(muon_status s);

#ifdef __cplusplus
}
#endif

#endif /* LIBMUON_H */
