// Internal interfaces between the C-ABI layer (libmuon.cu) and the kernels (ns_gemm.cu, elementwise.cu).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>
#include <utility>
#include <vector>

#include "../../include/libmuon.h"

namespace muon {

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline long long round8(long long v) { return (v + 7) / 8 * 8; }

// Kernel kinds, for launch counting and the event trace.
enum KernelKind : int32_t {
  KK_ADAMW = 0,
  KK_NESTEROV_NORM = 1,
  KK_COUNTER_RESET = 2,
  KK_GRAM = 3,
  KK_POLY = 4,
  KK_APPLY = 5,
  KK_FINAL = 6,
  KK_DEBUG_WAIT = 7,
  KK_NS_SMALL = 8,
  KK_GRAM_SPACE = 9,
  KK_GRAM32 = 10,
  KK_GRAM32_REDUCE = 11,
  KK_COUNT = 12
};

// Launch bookkeeping (libmuon.cu): counts launches and, while tracing, records an event pair.
void launch_begin(int32_t kind, cudaStream_t s);
void launch_end(cudaStream_t s);
int device_sm_count();
// The current device's capability check and the per-wait limit set by muon_set_timeout_ns (libmuon.cu).
muon_status device_check();
unsigned long long wait_timeout_ns();
// The registered per-tile timeline buffer of the GEMM kernels (null unless muon_debug_timeline set one).
void debug_timeline(unsigned long long **buf, int *cap_per_cta);

// ------------------------------------------------------------------------------------------ tensor-core GEMMs

// EPI_GRAM32: the Gram matrix of a wide iterate with m <= 256 rows, accumulated in fp32 and stored as a bf16 "hi"
// plane (the value rounded) and a bf16 "lo" plane (the rest, rounded) for the Gram-space chain.
enum EpiKind : int { EPI_GRAM = 0, EPI_POLY = 1, EPI_APPLY = 2, EPI_FINAL = 3, EPI_GRAM32 = 5 };

constexpr int GEMM_MAX_PROBLEMS = 8;

// One problem of a grouped tensor-core launch: a stack of `batch` matrices whose output is rows x cols
// (128 x 256 tiles), with its own epilogue inputs and outputs.
struct GemmProblem {
  int batch;
  int rows;
  int cols;
  int m_tiles, n_tiles;
  int m_pairs;            // tile rows are processed in vertically adjacent pairs, one per CTA of a cluster
  int tiles_per_matrix;   // tile pairs per matrix
  int k_iters;            // contraction / 64, rounded up
  int k_wrap;             // 0, or: 64-deep steps kk >= k_wrap read B's rows from (kk - k_wrap) * 64 (the final
                          // step of the Gram-space path: [R_hi | R_lo] times [X; X])
  long long tile_begin;   // first tile pair of this problem in the launch's pair space
  // per-matrix readiness counters (see TileSync), indexed by the matrix within the problem; null: none
  const uint32_t *wait_ctr;
  uint32_t wait_target;
  uint32_t *sig_ctr;
  // epilogue coefficients
  float alpha;            // gram: output = alpha * s^2 * acc (s from `scale` when given)
  float coef_a, coef_b, coef_c;   // poly: output = a*I + b*G + c*acc, with G read by the epilogue
  const float *scale;     // per-matrix normalisation s_k (device), or null; apply / final: output = s * acc
  // bf16 output of gram / poly / apply
  __nv_bfloat16 *out;
  long long ld_out, mstride_out;
  // output of the Gram-space Gram (EPI_GRAM32), bf16 planes: G's hi plane (G rounded) at out, its lo plane (the
  // rest, rounded) at out + gs_plane, with the row and matrix pitches ld_out and mstride_out (elements); and
  // c * G + b * I (coef_b, coef_c) the same way at out + gs_bprime and that + gs_plane
  long long gs_plane, gs_bprime;
  // EPI_GRAM32 split along the contraction: ksplit (>= 1) slices of kper 64-deep steps, each slice a tile pair of
  // its own; slice j stores its raw fp32 sum over the two bf16 planes 2 + 2 j and 3 + 2 j (as fp32 with the same
  // element pitches, from out + (2 + 2 j) * gs_plane), and a reduce kernel adds the slices in index order and
  // forms the outputs above
  int ksplit, kper;
  // Symmetric m x m matrices (G, H) stored as their upper 256-blocks only: block (i, j), rows 256 i .., columns
  // 256 j .., is stored when j >= i, a diagonal block whole. half_out (GRAM, POLY): store only those blocks, every
  // element as computed, nothing mirrored. half_a (POLY, APPLY, FINAL) / half_b (POLY): the A / B operand is such
  // a matrix; a 64-deep step whose 256-block lies left of the operand rows' block reads the stored block above the
  // diagonal transposed (an MN-major operand through map_t), which holds the same values.
  int half_out, half_a, half_b;
  // final step: parameter update (params != null) or dense store (out_dense != null); with master, the
  // update applies to the fp32 master copies and params receive them rounded to bf16
  void *const *params;
  float *const *master;
  void *out_dense;
  int out_dtype;          // muon_dtype of params / out_dense
  int transposed;         // stored matrix is the transpose of the wide iterate
  int orig_cols;          // columns of the stored matrix
  int cautious;
  float lr_wd;            // lr * weight_decay
  float lr_scale;         // lr * update scale
};

// A bf16 matrix stack in global memory as the GEMMs see it: K matrices of rows x cols,
// row pitch ld elements (multiple of 8), matrix pitch mstride elements.
struct Bf16Stack {
  const void *ptr;
  long long rows, cols, ld, mstride, batch;
};

// Final iteration: u = s * (h x) in the wide orientation (h = a*I + b*G + c*G^2), then either the Muon parameter update
// or a dense store, transposing back when the stored matrix is tall.
struct FinalSpec {
  void *const *params;   // device array of K pointers (update) or null
  float *const *master;  // device array of K pointers to fp32 master copies of bf16 params, or null
  void *out_dense;       // contiguous (K, A, B) (store) or null
  int dtype;             // muon_dtype
  int transposed;
  int orig_cols;
  int cautious;
  float lr_wd, lr_scale;
};

// Collects the problems of one step kind (all grams, all polys, ...) of several stacks and launches
// them as few grouped kernels (up to GEMM_MAX_PROBLEMS problems per launch), deepest contraction first.
// POLY, the one step kind compiled in several pipeline shapes (mainloop stages + epilogue ring slots):
// shape 0 = 4 + 5, 1 = 5 + 3, 2 = 6 + 2. Without a measured choice, contractions up to 2048 take shape 0 and
// deeper ones shape 2. Every shape computes each tile the same way, so the choice changes only the time.
constexpr int POLY_SHAPES = 3;
// The autotune table (process-wide): the measured shape for POLY launches whose deepest contraction is
// k_iters 64-deep steps, or -1; and a forced shape for every launch (-1: none), for tests and sweeps.
int poly_shape_lookup(int k_iters);
void poly_shape_record(int k_iters, int shape);
void poly_shape_clear();
int poly_shape_forced();

// The fp32 Gram of the Gram-space path (EPI_GRAM32) has one tile pair per matrix, which leaves most SMs idle when
// a launch holds fewer matrices than there are SM pairs. Its contraction (the iterate's long side) is then split
// into up to GRAM32_MAX_SPLIT slices, each computed by a tile pair of its own. The count is a property of the
// stack, so that a stack gets the same bits in any launch it shares: the autotune table's measured count for
// its (m, contraction steps, K), else the most slices that would fill one wave of SM pairs with this stack
// alone while each slice keeps at least GRAM32_MIN_SLICE_K 64-deep steps; a forced count (-1: none) serves
// tests and sweeps. The count changes only the order of the fp32 additions.
constexpr int GRAM32_MAX_SPLIT = 4;
constexpr int GRAM32_MIN_SLICE_K = 16;
int gram_split_lookup(long long m, int k_iters, long long K);
void gram_split_record(long long m, int k_iters, long long K, int split);
void gram_split_clear();
int gram_split_forced();

// Per-matrix dependencies between the grouped launches of one Newton-Schulz chain, instead of the launch
// order: a tile of matrix b loads its operands only once wait[b] >= target (every tile of b that the
// previous step kind produced has been stored), and each epilogue warp adds 1 to sig[b] (release) when
// its part of a tile is stored. A launch whose problems all have a wait skips the grid-wide dependency on
// its predecessor, so its tiles can start on the SMs its predecessor has left while the rest finish.
struct TileSync {
  const uint32_t *wait;
  uint32_t target;
  uint32_t *sig;
};
// The signals one launch of this step kind adds to a matrix's counter (every CTA's epilogue warps, once
// per tile) for a wide iterate of m rows and n columns.
uint32_t gemm_signals_per_matrix(int epi, long long m, long long n);
// The 256 x 256 tile pairs one launch of this step kind computes per matrix (symmetric kinds: on or above
// the diagonal only).
long long gemm_tiles_per_matrix(int epi, long long m, long long n);

class GemmBatch {
 public:
  GemmBatch(int epi, uint32_t *err, unsigned long long timeout_ns) : epi_(epi), err_(err), timeout_ns_(timeout_ns) {}
  // POLY only: launch with this pipeline shape whatever the table or the rule says (-1: no override)
  void force_shape(int shape) { force_ = shape; }
  muon_status add_gram(const Bf16Stack &x, __nv_bfloat16 *g, long long ldg, long long mstride_g, float alpha,
                       const float *scale,
                       const TileSync *sync = nullptr);
  muon_status add_poly(const Bf16Stack &g, __nv_bfloat16 *h, long long ldh, long long mstride_h, float a, float b,
                       float c,
                       const TileSync *sync = nullptr);
  muon_status add_apply(const Bf16Stack &h, const Bf16Stack &x, __nv_bfloat16 *out, const float *scale,
                       const TileSync *sync = nullptr);
  // EPI_GRAM32 (x.rows <= 256): g = alpha * s^2 * x x^T as bf16 hi / lo planes, and c g + b I at g_hi + bprime;
  // planes 2 .. bprime / plane - 1 are scratch for the slices of a split contraction (two planes per slice)
  muon_status add_gram32(const Bf16Stack &x, __nv_bfloat16 *g_hi, long long ldg, long long mstride_g, long long plane,
                         long long bprime, float b, float c, float alpha, const float *scale);
  // EPI_GRAM32 only: split every contraction into this many slices (clipped to what each problem allows), whatever
  // the table or the rule says (0: no override)
  void force_split(int split) { split_ = split; }
  muon_status add_final(const Bf16Stack &h, const Bf16Stack &x, const float *scale, const FinalSpec &f,
                       const TileSync *sync = nullptr, int k_wrap = 0);
  muon_status launch(cudaStream_t s);
  // Per-matrix counter waits replace the wait for the whole previous grid unless this is set: then the
  // launches wait for both (used where the previous launch in the stream belongs to another branch)
  void force_grid_wait(bool on) { grid_wait_ = on; }
  // Items added after this read and write the symmetric G and H as their upper 256-blocks only (GemmProblem's
  // half_out, half_a, half_b): GRAM and POLY store no mirrored blocks, POLY, APPLY and the final step read the
  // blocks below the diagonal transposed. Results are the same bits either way.
  void half_symmetric(bool on) { half_ = on; }
  ~GemmBatch();

 private:
  struct Item;
  int epi_;
  uint32_t *err_;
  unsigned long long timeout_ns_;
  Item *items_ = nullptr;
  int n_ = 0, cap_ = 0;
  int force_ = -1;
  int split_ = 0;
  bool grid_wait_ = false;
  bool half_ = false;
  muon_status push(const Item &it);
  void order();                        // launch order of the items (stable for a given set)
  int group_size(int first) const;     // items from first that share one launch
};

// Single-stack conveniences (a batch of one).
muon_status launch_gram(const Bf16Stack &x, __nv_bfloat16 *g, long long ldg, long long mstride_g, float alpha,
                        const float *scale, uint32_t *err, unsigned long long timeout_ns, cudaStream_t s,
                        const TileSync *sync = nullptr);
muon_status launch_poly(const Bf16Stack &g, __nv_bfloat16 *h, long long ldh, long long mstride_h, float a, float b,
                        float c, uint32_t *err, unsigned long long timeout_ns, cudaStream_t s,
                        const TileSync *sync = nullptr);
muon_status launch_apply(const Bf16Stack &h, const Bf16Stack &x, __nv_bfloat16 *out, const float *scale,
                         uint32_t *err, unsigned long long timeout_ns, cudaStream_t s,
                        const TileSync *sync = nullptr);
muon_status launch_final(const Bf16Stack &h, const Bf16Stack &x, const float *scale, const FinalSpec &f,
                         uint32_t *err, unsigned long long timeout_ns, cudaStream_t s,
                        const TileSync *sync = nullptr);

// ------------------------------------------------------------------------------------------ small matrices

// The whole Newton-Schulz chain of each matrix of a stack in one CTA (ns_small.cu), for wide iterates of
// at most 128 x 256: from the wide U (bf16, with the per-matrix scale s) to the parameter update or the
// dense output of the large path's final step.
struct SmallNsArgs {
  const __nv_bfloat16 *u;   // wide U of matrix k at u + k * mstride_u, rows of ldu elements
  long long ldu, mstride_u;
  const float *scale;       // s_k, or null
  int K, m, n;              // matrices; wide rows and columns
  int transposed;           // stored matrix is the transpose of the wide iterate
  int orig_cols;            // columns of the stored matrix
  int ns_steps;
  float coeffs[3 * MUON_MAX_NS_STEPS];
  void *const *params;      // device array of K pointers (update), or null (dense output)
  float *const *master;     // fp32 master copies of bf16 params, or null
  void *out_dense;          // contiguous (K, A, B) output when params is null
  int out_dtype;            // muon_dtype of params / out_dense
  int cautious;
  float lr_wd, lr_scale;
  uint32_t *err;
  unsigned long long timeout_ns;
};
bool ns_small_fits(long long m, long long n);
muon_status launch_ns_small(const SmallNsArgs &a, cudaStream_t s);

// ------------------------------------------------------------------------------------------ Gram-space chain

// The Newton-Schulz iteration in the m x m Gram space (ns_gram_space.cu) for wide iterates with at most
// GS_MAX_M rows that the fused small-matrix kernel does not take. Its scratch is GS_BUFFERS m x m matrices per
// matrix of the stack (A, Q, P, two R and B), each as two bf16 planes, hi (the value rounded) and lo (the rest,
// rounded), with rows of round8(m) elements: buffer b, plane p, matrix k at ((b * 2 + p) * K + k) * m *
// round8(m) elements; before the chain runs, buffers Q .. R1 hold the fp32 Gram's slice sums when its
// contraction is split (slice j, fp32, over planes 2 + 2 j and 3 + 2 j); then R_N for the final product as two
// bf16 halves side by side, [R_hi | R_lo] (R_hi = R_N rounded, R_lo = the rest rounded), each half 64-column
// padded with zeros: K matrices of m rows x 2 * round64(m) columns.
constexpr int GS_MAX_M = 256;
constexpr int GS_BUFFERS = 6;
// GS_B holds c_t A_t + b_t I, the right operand of phase A's product A_t (c_t A_t + b_t I) = b_t A_t + c_t A_t^2,
// written wherever A_t is written
enum GsBuffer : int { GS_G = 0, GS_Q = 1, GS_P = 2, GS_R0 = 3, GS_R1 = 4, GS_B = 5 };
inline bool gram_space_eligible(long long m, long long n) { return m >= 1 && m <= GS_MAX_M && !ns_small_fits(m, n); }
size_t gram_space_plane_bytes(long long K, long long m);
inline long long round64(long long v) { return (v + 63) / 64 * 64; }
struct GramSpaceStack {
  __nv_bfloat16 *planes;     // the stack's scratch (16-byte aligned): the buffers' planes, then [R_hi | R_lo]
  int K, m;
};
// The [R_hi | R_lo] halves of a stack's scratch.
inline __nv_bfloat16 *gram_space_rsplit(__nv_bfloat16 *planes, long long K, long long m) {
  return planes + static_cast<long long>(GS_BUFFERS) * 2 * K * m * round8(m);
}
// From A_0 in buffer GS_G (written by an EPI_GRAM32 launch) to R_N in bf16, for every matrix of up to n stacks
// (one launch per 8 stacks).
muon_status launch_gram_space(const GramSpaceStack *stacks, int n, int ns_steps, const float *coeffs, uint32_t *err,
                              unsigned long long timeout_ns, cudaStream_t s);

// ------------------------------------------------------------------------------------------ elementwise

// Momentum + Nesterov + Frobenius norm scale + bf16 store in the wide orientation, for one stack.
struct NesterovArgs {
  const void *const *gptrs;  // device array of K pointers, or null (then gbase is used)
  const void *gbase;         // contiguous (K, A, B)
  int gdtype;
  float *momentum;           // (K, A, B) fp32 or null (plain normalisation, no momentum)
  __nv_bfloat16 *u;
  long long ldu, mstride_u;
  float *partials;           // [K][tiles_r * tiles_c]
  float *scale;              // [K]: s_k = 1 / (||U_k||_F + eps)
  unsigned *counters;        // [K], zero when the launch starts
  int K, A, B, tiles_r, tiles_c, transposed;
  float mu, eps;
  int nesterov;
  int wide_tiles;   // 1: tiles of 64 rows x NESTEROV_WIDE_TILE columns, or of NESTEROV_TALL_ROWS x 64 where stored
                    // tall; 0: 64 x 64
};
constexpr int NESTEROV_TILE = 64;
constexpr int NESTEROV_TALL_ROWS = 128;   // rows of a tile of a matrix stored tall (wide_tiles)
constexpr int NESTEROV_WIDE_TILE = 256;
constexpr int NESTEROV_MAX_PROBLEMS = 16;
struct NesterovGroup {
  NesterovArgs prob[NESTEROV_MAX_PROBLEMS];
  long long block_begin[NESTEROV_MAX_PROBLEMS];
  int nprob;
};
static_assert(sizeof(NesterovGroup) <= 4096, "kernel parameter block too large");

// ------------------------------------------------------------------------------------------ workspace layout
//
// A workspace (the caller's, or the no-allocation entry point's static scratch) starts with a header: the
// control block (error word at byte 0) and four 32-bit counters per matrix of the call (the norm pass's tile
// count, then the readiness of each matrix's G, H and iterate X), which every call zeroes before its first
// launch. Each stack's sections follow, stack after stack; their offsets are relative to the stack's start.
constexpr size_t CTRL_BYTES = 256;

inline size_t header_bytes(long long total_K) {
  return align_up(CTRL_BYTES + static_cast<size_t>(total_K) * 16, 1024);
}

// One stack's sections (1024-byte aligned): K fp32 scales, the norm pass's per-tile partial sums, two bf16
// iterates (K, m, ldx) and two bf16 (K, m, ldg) buffers for G and H; m = min(A, B), n = max(A, B), rows padded
// to a multiple of 8 elements (16 bytes, as TMA requires); then, for shapes that can take the Gram-space path,
// its scratch (gram_space_plane_bytes).
struct Layout {
  long long m, n, ldx, ldg, tiles_r, tiles_c;
  size_t scale, partial, x0, x1, g, h, gs, total;   // gs: the Gram-space planes (shapes that can take that path)
};

inline Layout layout(long long K, long long A, long long B) {
  Layout L{};
  L.m = A < B ? A : B;
  L.n = A < B ? B : A;
  L.ldx = round8(L.n);
  L.ldg = round8(L.m);
  L.tiles_r = (A + NESTEROV_TILE - 1) / NESTEROV_TILE;
  L.tiles_c = (B + NESTEROV_TILE - 1) / NESTEROV_TILE;
  size_t off = 0;
  L.scale = off;
  off = align_up(off + static_cast<size_t>(K) * 4, 1024);
  L.partial = off;
  off = align_up(off + static_cast<size_t>(K) * L.tiles_r * L.tiles_c * 4, 1024);
  L.x0 = off;
  off = align_up(off + static_cast<size_t>(K) * L.m * L.ldx * 2, 1024);
  L.x1 = off;
  off = align_up(off + static_cast<size_t>(K) * L.m * L.ldx * 2, 1024);
  L.g = off;
  off = align_up(off + static_cast<size_t>(K) * L.m * L.ldg * 2, 1024);
  L.h = off;
  off = align_up(off + static_cast<size_t>(K) * L.m * L.ldg * 2, 1024);
  L.gs = off;
  if (gram_space_eligible(L.m, L.n)) off = align_up(off + gram_space_plane_bytes(K, L.m), 1024);
  L.total = off;
  return L;
}

// ------------------------------------------------------------------------------------------ argument checks

inline bool valid_dtype(int d) { return d == MUON_F32 || d == MUON_BF16; }

inline muon_status check_stack_dims(int64_t K, int64_t A, int64_t B) {
  if (K < 1 || A < 1 || B < 1) return MUON_ERR_INVALID_ARG;
  if (A > 65536 || B > 65536 || K > (1ll << 31)) return MUON_ERR_SHAPE;
  const long double elems = static_cast<long double>(K) * A * B;
  if (elems >= static_cast<long double>(1ll << 40)) return MUON_ERR_SHAPE;
  return MUON_OK;
}

inline muon_status check_coeffs(int ns_steps, const float *coeffs) {
  if (ns_steps < 1 || ns_steps > MUON_MAX_NS_STEPS || coeffs == nullptr) return MUON_ERR_INVALID_ARG;
  for (int i = 0; i < 3 * ns_steps; ++i)
    if (!std::isfinite(coeffs[i])) return MUON_ERR_INVALID_ARG;
  return MUON_OK;
}

// Every check of ns_orthogonalize's arguments but the workspace's.
inline muon_status check_ns_args(const void *x, int xdt, const void *out, int odt, int64_t K, int64_t A, int64_t B,
                                 int ns_steps, const float *coeffs, float eps) {
  if (x == nullptr || out == nullptr) return MUON_ERR_INVALID_ARG;
  muon_status st = check_stack_dims(K, A, B);
  if (st != MUON_OK) return st;
  if (!valid_dtype(xdt) || !valid_dtype(odt)) return MUON_ERR_DTYPE;
  if ((st = check_coeffs(ns_steps, coeffs)) != MUON_OK) return st;
  if (!std::isfinite(eps) || eps < 0.f) return MUON_ERR_INVALID_ARG;
  return MUON_OK;
}
// All n stacks (all with momentum or all without) in as few launches as the grid and the problem table
// allow. The counters must be zero when the call's launches start; they are left at the tile counts.
muon_status launch_nesterov_norm(const NesterovArgs *probs, int n, cudaStream_t s);
// Zeroes n counters in stream order (a kernel, so that the launches around it keep overlapping).
muon_status launch_counter_reset(unsigned *counters, long long n, cudaStream_t s, unsigned *counters2 = nullptr,
                                 long long n2 = 0);

struct AdamwConst {
  int l2;               // 1: g <- g + l2_wd * p before the moments (Adam with L2); 0: decoupled decay
  float l2_wd;
  float decay;          // 1 - lr*wd (decoupled), 1 (L2)
  float beta1, one_minus_beta1, beta2, one_minus_beta2;
  float step_size;      // lr / (1 - beta1^t)
  float inv_sqrt_bc2;   // 1 / sqrt(1 - beta2^t)
  float eps;
};
muon_status launch_adamw(void *p, int pdt, const void *g, int gdt, float *m, float *v, long long n,
                         const AdamwConst &c, cudaStream_t s);
muon_status launch_adamw_master(float *master, __nv_bfloat16 *p, const void *g, int gdt, float *m, float *v,
                                long long n, const AdamwConst &c, cudaStream_t s);

// ------------------------------------------------------------------ grouped AdamW
// One launch updates up to ADAMW_GROUP_MAX tensors. Their elements are cut into chunks of `chunk` elements
// (the last chunk of a tensor may be short), numbered tensor after tensor; each warp takes the next
// chunk from a counter in the launch's region until none is left, so every chunk is updated once
// whatever the tensors' sizes. The chunk is about an eighth of a full grid's warps' share of the elements:
// a multiple of 256, at least 256, at most ADAMW_CHUNK_MAX.
constexpr int ADAMW_GROUP_MAX = 96;
constexpr long long ADAMW_CHUNK_MAX = 8192;
constexpr size_t ADAMW_REGION_BYTES = 256;       // per launch: the chunk counter (8 B)
constexpr int ADAMW_THREADS = 96;
struct AdamwTensorDesc {
  void *p;              // parameters (pdt), or bf16 when master is set
  const void *g;        // gradients (gdt)
  float *m, *v;         // moments
  float *master;        // fp32 master weights taking the update, or null
  long long n;
  long long chunk_begin;   // first chunk of this tensor in the launch's numbering
  int pdt, gdt;
  int vec;              // all pointers 16-byte aligned: 8-element vector accesses
  AdamwConst c;
};
struct AdamwGroup {
  AdamwTensorDesc t[ADAMW_GROUP_MAX];
  int ntensors;
  long long chunk;            // elements per chunk: a multiple of 256
  long long total_chunks;
  unsigned long long *next;   // the chunk counter (zero when the pass starts)
};
static_assert(sizeof(AdamwGroup) <= 16384, "kernel parameter block too large");
// A grid of ADAMW_THREADS-thread blocks filling the GPU (10 blocks per SM at 64 registers).
muon_status launch_adamw_grouped(const AdamwGroup &G, cudaStream_t s);

muon_status launch_debug_wait(uint32_t *err, unsigned long long timeout_ns, cudaStream_t s);

}  // namespace muon
