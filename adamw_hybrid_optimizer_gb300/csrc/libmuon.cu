// libmuon C ABI: argument checks, workspace layout, the order of launches of one optimizer step,
// launch counting and the optional event trace. See include/libmuon.h for the contract.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>
#include <map>
#include <set>
#include <utility>
#include <vector>

#include "../../include/libmuon.h"
#include "internal.h"

namespace muon {
namespace {

// ------------------------------------------------------------------------------------------ device state

struct DeviceInfo {
  bool probed = false;
  bool supported = false;
  int sms = 0;
};

std::mutex g_dev_mu;
DeviceInfo g_dev[64];

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return -1;
  return d;
}

muon_status check_device() {
  const int d = current_device();
  if (d < 0 || d >= 64) return MUON_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo &di = g_dev[d];
  if (!di.probed) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d) != cudaSuccess)
      return MUON_ERR_CUDA;
    di.probed = true;
    di.supported = (major == 10 && minor == 3);
    di.sms = sms;
  }
  return di.supported ? MUON_OK : MUON_ERR_UNSUPPORTED_DEVICE;
}

// ------------------------------------------------------------------------------------------ trace

std::mutex g_trace_mu;
bool g_trace_on = false;
int64_t g_launches = 0;
struct TraceRec {
  int32_t kind;
  cudaEvent_t start, stop;
};
std::vector<TraceRec> g_trace;
std::vector<cudaEvent_t> g_event_pool;
constexpr size_t TRACE_CAP = 65536;
int32_t g_pending_kind = -1;
cudaEvent_t g_pending_start = nullptr;

cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

unsigned long long g_timeout_ns = 2000000000ull;
// grouped chain: per-matrix counter dependencies between launches: -1 where the rule in enqueue_grouped
// allows them, 0 never, 1 always
std::atomic<int> g_counter_deps{-1};
// Gram-space path: -1 the rule (gram_space_route), 0 never, 1 wherever the shape is eligible
std::atomic<int> g_gram_space{-1};
// plain chain: G and H stored as their upper 256-blocks only (1, the default) or whole (0)
std::atomic<int> g_half_sym{1};

}  // namespace

void launch_begin(int32_t kind, cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  ++g_launches;
  g_pending_kind = -1;
  if (!g_trace_on || g_trace.size() >= TRACE_CAP) return;
  cudaEvent_t e = take_event();
  if (e == nullptr) return;
  cudaEventRecord(e, s);
  g_pending_kind = kind;
  g_pending_start = e;
}

void launch_end(cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (g_pending_kind < 0) return;
  cudaEvent_t e = take_event();
  if (e == nullptr) {
    g_event_pool.push_back(g_pending_start);
  } else {
    cudaEventRecord(e, s);
    g_trace.push_back({g_pending_kind, g_pending_start, e});
  }
  g_pending_kind = -1;
}

muon_status device_check() { return check_device(); }

// ------------------------------------------------------------------------------------------ autotune table

namespace {
std::mutex g_tune_mu;
std::map<int, int> g_poly_shape;   // deepest contraction (64-deep steps) of a POLY launch -> measured shape
int g_poly_forced = -1;
}  // namespace

int poly_shape_lookup(int k_iters) {
  std::lock_guard<std::mutex> lk(g_tune_mu);
  auto it = g_poly_shape.find(k_iters);
  return it == g_poly_shape.end() ? -1 : it->second;
}
void poly_shape_record(int k_iters, int shape) {
  std::lock_guard<std::mutex> lk(g_tune_mu);
  g_poly_shape[k_iters] = shape;
}
void poly_shape_clear() {
  std::lock_guard<std::mutex> lk(g_tune_mu);
  g_poly_shape.clear();
}
int poly_shape_forced() {
  std::lock_guard<std::mutex> lk(g_tune_mu);
  return g_poly_forced;
}

namespace {
std::map<std::vector<long long>, int> g_gram_split;   // (m, contraction steps, K) of a stack -> measured slices
int g_gram_split_forced = -1;
}  // namespace

int gram_split_lookup(long long m, int k_iters, long long K) {
  std::lock_guard<std::mutex> lk(g_tune_mu);
  auto it = g_gram_split.find({m, static_cast<long long>(k_iters), K});
  return it == g_gram_split.end() ? -1 : it->second;
}
void gram_split_record(long long m, int k_iters, long long K, int split) {
  std::lock_guard<std::mutex> lk(g_tune_mu);
  g_gram_split[{m, static_cast<long long>(k_iters), K}] = split;
}
void gram_split_clear() {
  std::lock_guard<std::mutex> lk(g_tune_mu);
  g_gram_split.clear();
}
int gram_split_forced() {
  std::lock_guard<std::mutex> lk(g_tune_mu);
  return g_gram_split_forced;
}

unsigned long long wait_timeout_ns() { return g_timeout_ns; }

namespace {
unsigned long long *g_timeline = nullptr;
int g_timeline_cap = 0;
int64_t g_timeline_regions = 0, g_timeline_next = 0, g_timeline_region_words = 0;
}  // namespace

// Each tensor-core launch after registration takes the next region of the buffer, until it is full.
void debug_timeline(unsigned long long **buf, int *cap_per_cta) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (g_timeline == nullptr || g_timeline_next >= g_timeline_regions) {
    *buf = nullptr;
    *cap_per_cta = 0;
    return;
  }
  *buf = g_timeline + g_timeline_next++ * g_timeline_region_words;
  *cap_per_cta = g_timeline_cap;
}

int device_sm_count() {
  const int d = current_device();
  if (d < 0 || d >= 64) return 1;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  return g_dev[d].sms > 0 ? g_dev[d].sms : 1;
}

namespace {

// ------------------------------------------------------------------------------------------ workspace

// The Nesterov/norm pass of one stack whose sections start at w; counters: the stack's K header words.
NesterovArgs nesterov_args(char *w, const Layout &L, unsigned *counters, long long K, long long A, long long B,
                           const void *const *gptrs, const void *gbase, int gdt, float *momentum, float mu,
                           bool nesterov, float eps) {
  NesterovArgs na{};
  na.gptrs = gptrs;
  na.gbase = gbase;
  na.gdtype = gdt;
  na.momentum = momentum;
  na.u = reinterpret_cast<__nv_bfloat16 *>(w + L.x0);
  na.ldu = L.ldx;
  na.mstride_u = L.m * L.ldx;
  na.partials = reinterpret_cast<float *>(w + L.partial);
  na.scale = reinterpret_cast<float *>(w + L.scale);
  na.counters = counters;
  na.K = static_cast<int>(K);
  na.A = static_cast<int>(A);
  na.B = static_cast<int>(B);
  na.tiles_r = static_cast<int>(L.tiles_r);
  na.tiles_c = static_cast<int>(L.tiles_c);
  na.transposed = A > B ? 1 : 0;
  // rows of 256 columns per block where stored wide: longer contiguous segments, and a quarter of the blocks
  // (and of their per-block reduction, fence and count) of 64 x 64 tiles; 128 x 64 tiles where stored tall,
  // so that each row of the transposed U is written 256 bytes at a time; the partial sums need less room
  na.wide_tiles = 1;
  if (!na.transposed)
    na.tiles_c = static_cast<int>((B + NESTEROV_WIDE_TILE - 1) / NESTEROV_WIDE_TILE);
  else
    na.tiles_r = static_cast<int>((A + NESTEROV_TALL_ROWS - 1) / NESTEROV_TALL_ROWS);
  na.mu = mu;
  na.eps = eps;
  na.nesterov = nesterov ? 1 : 0;
  return na;
}

// The Newton-Schulz chain on the wide iterate in x0 (unnormalised U; s_k in `scale`) of the stack whose
// sections start at ws, ending in launch_final. Iteration t reads X from one iterate buffer and writes the other.
// The fused one-CTA-per-matrix chain of a stack whose wide iterate fits ns_small (sections at ws).
SmallNsArgs small_args(uint32_t *err, char *ws, const Layout &L, long long K, int ns_steps, const float *coeffs,
                       const FinalSpec &fin) {
  SmallNsArgs a{};
  a.u = reinterpret_cast<const __nv_bfloat16 *>(ws + L.x0);
  a.ldu = L.ldx;
  a.mstride_u = L.m * L.ldx;
  a.scale = reinterpret_cast<const float *>(ws + L.scale);
  a.K = static_cast<int>(K);
  a.m = static_cast<int>(L.m);
  a.n = static_cast<int>(L.n);
  a.transposed = fin.transposed;
  a.orig_cols = fin.orig_cols;
  a.ns_steps = ns_steps;
  for (int i = 0; i < 3 * ns_steps; ++i) a.coeffs[i] = coeffs[i];
  a.params = fin.params;
  a.master = fin.master;
  a.out_dense = fin.out_dense;
  a.out_dtype = fin.dtype;
  a.cautious = fin.cautious;
  a.lr_wd = fin.lr_wd;
  a.lr_scale = fin.lr_scale;
  a.err = err;
  a.timeout_ns = g_timeout_ns;
  return a;
}

// Estimated duration of one step kind's launch over these stacks: 0.33 us per 64-deep k-step of a 256 x 256
// tile pair (the measured mainloop rate), spread over the clusters.
double launch_estimate_us(int kind, long long m, long long n, long long K) {
  const long long k = (kind == EPI_GRAM ? n + 63 : m + 63) / 64;
  const double pairs = static_cast<double>(K) * gemm_tiles_per_matrix(kind, m, n);
  return pairs * static_cast<double>(k) * 0.33 / std::max(1, device_sm_count() / 2);
}

// Whether a chain whose longest launch is estimated at est_us uses the per-matrix readiness counters.
// They pay where launch boundaries are a visible share of the chain: launches of a few hundred
// microseconds at most. Measured: GPT-2-small step 1.525 -> 1.457 ms and the 256-wide aspect set
// 1.86 -> 1.80 ms with them, but the Llama-3-8B set (launches of milliseconds) 325 -> 355 ms.
bool counter_deps_for(double est_us) {
  const int mode = g_counter_deps.load();
  return mode == 1 || (mode == -1 && est_us <= 500.0);
}

// Whether a stack of K wide m x n iterates takes the Gram-space path: never for shapes that cannot (m > 256, or
// the fused small-matrix kernel's); else as forced by muon_debug_gram_space, else as measured by muon_autotune
// for this (m, n, K), else where the long side is at least four times the short one, where the m x m chain
// (about 4 m^3 flops per step in three bf16 passes) costs a fraction of the plain step's 4 m^2 n + 2 m^3.
std::mutex g_route_mu;
std::map<std::vector<long long>, int> g_route_table;   // (m, n, K) -> measured: 1 Gram space, 0 plain chain

bool gram_space_route(long long m, long long n, long long K) {
  if (!gram_space_eligible(m, n)) return false;
  const int mode = g_gram_space.load();
  if (mode >= 0) return mode == 1;
  {
    std::lock_guard<std::mutex> lk(g_route_mu);
    auto it = g_route_table.find({m, n, K});
    if (it != g_route_table.end()) return it->second == 1;
  }
  return n >= 4 * m;
}

// The Gram-space path's launches for one stack, added to three batches: the fp32 Gram A_0 = s^2 U U^T of the
// wide U in x0, the m x m chain (into gs), and the final step with [R_hi | R_lo] times [U; U] (scaled by s).
muon_status add_gram_space(char *ws, const Layout &L, long long K, const float *coeffs, const FinalSpec &fin,
                           GemmBatch &g32, std::vector<GramSpaceStack> &gs, GemmBatch &fin_batch) {
  const float *scale = reinterpret_cast<const float *>(ws + L.scale);
  __nv_bfloat16 *planes = reinterpret_cast<__nv_bfloat16 *>(ws + L.gs);
  const long long ldm = round8(L.m), msm = L.m * ldm;
  Bf16Stack X{ws + L.x0, L.m, L.n, L.ldx, L.m * L.ldx, K};
  // A_0 into buffer GS_G and c_0 A_0 + b_0 I into buffer GS_B (plane p of buffer b starts at (2 b + p) K m ldm)
  muon_status st = g32.add_gram32(X, planes, ldm, msm, K * msm, 2LL * GS_B * K * msm, coeffs[1], coeffs[2], 1.0f,
                                  scale);
  if (st != MUON_OK) return st;
  gs.push_back(GramSpaceStack{planes, static_cast<int>(K), static_cast<int>(L.m)});
  const long long mp = round64(L.m);
  Bf16Stack Rs{gram_space_rsplit(planes, K, L.m), L.m, 2 * mp, 2 * mp, L.m * 2 * mp, K};
  return fin_batch.add_final(Rs, X, scale, fin, nullptr, static_cast<int>(mp / 64));
}

muon_status launch_gram_space_batches(GemmBatch &g32, const std::vector<GramSpaceStack> &gs, GemmBatch &fin_batch,
                                      int ns_steps, const float *coeffs, uint32_t *err, cudaStream_t s) {
  muon_status st;
  if ((st = g32.launch(s)) != MUON_OK) return st;
  if ((st = launch_gram_space(gs.data(), static_cast<int>(gs.size()), ns_steps, coeffs, err, g_timeout_ns, s)) !=
      MUON_OK)
    return st;
  return fin_batch.launch(s);
}

// The Newton-Schulz chain of one stack. counters: the workspace's four counters per matrix (the norm
// pass's, then the readiness of G, H and X), zeroed by the caller before the norm pass; norm_tiles: the
// norm pass's tiles per matrix. With counter dependencies (counter_deps_for), each launch waits per matrix
// on its predecessor's counters instead of on the whole grid.
muon_status run_ns_chain(uint32_t *err, char *ws, const Layout &L, long long K, int ns_steps, const float *coeffs,
                         const FinalSpec &fin, cudaStream_t s, uint32_t *counters, uint32_t norm_tiles) {
  if (ns_small_fits(L.m, L.n)) return launch_ns_small(small_args(err, ws, L, K, ns_steps, coeffs, fin), s);
  if (gram_space_route(L.m, L.n, K)) {
    GemmBatch g32(EPI_GRAM32, err, g_timeout_ns), fb(EPI_FINAL, err, g_timeout_ns);
    std::vector<GramSpaceStack> gs;
    muon_status st = add_gram_space(ws, L, K, coeffs, fin, g32, gs, fb);
    return st != MUON_OK ? st : launch_gram_space_batches(g32, gs, fb, ns_steps, coeffs, err, s);
  }
  double est = 0.0;
  for (int kind = EPI_GRAM; kind <= EPI_APPLY; ++kind) est = std::max(est, launch_estimate_us(kind, L.m, L.n, K));
  const bool deps = counter_deps_for(est);
  uint32_t *G_ready = counters + K, *H_ready = counters + 2 * K, *X_ready = counters + 3 * K;
  const uint32_t e_gram = gemm_signals_per_matrix(EPI_GRAM, L.m, L.n);
  const uint32_t e_poly = gemm_signals_per_matrix(EPI_POLY, L.m, L.n);
  const uint32_t e_apply = gemm_signals_per_matrix(EPI_APPLY, L.m, L.n);
  const float *scale = reinterpret_cast<const float *>(ws + L.scale);
  __nv_bfloat16 *xb[2] = {reinterpret_cast<__nv_bfloat16 *>(ws + L.x0), reinterpret_cast<__nv_bfloat16 *>(ws + L.x1)};
  __nv_bfloat16 *G = reinterpret_cast<__nv_bfloat16 *>(ws + L.g);
  __nv_bfloat16 *H = reinterpret_cast<__nv_bfloat16 *>(ws + L.h);
  const long long mstride_x = L.m * L.ldx;
  const long long mstride_g = L.m * L.ldg;
  const unsigned long long to = g_timeout_ns;
  muon_status st = MUON_OK;
  for (int t = 0; t < ns_steps; ++t) {
    const float a = coeffs[3 * t], b = coeffs[3 * t + 1], c = coeffs[3 * t + 2];
    const float *sc = (t == 0) ? scale : nullptr;
    const uint32_t tt = static_cast<uint32_t>(t);
    const TileSync sync_gram{t == 0 ? counters : X_ready, t == 0 ? norm_tiles + 1u : tt * e_apply, G_ready};
    const TileSync sync_poly{G_ready, (tt + 1) * e_gram, H_ready};
    const TileSync sync_last{H_ready, (tt + 1) * e_poly, t + 1 < ns_steps ? X_ready : nullptr};
    Bf16Stack X{xb[t & 1], L.m, L.n, L.ldx, mstride_x, K};
    if ((st = launch_gram(X, G, L.ldg, mstride_g, 1.0f, sc, err, to, s, deps ? &sync_gram : nullptr)) != MUON_OK)
      return st;
    Bf16Stack Gs{G, L.m, L.m, L.ldg, mstride_g, K};
    if ((st = launch_poly(Gs, H, L.ldg, mstride_g, a, b, c, err, to, s, deps ? &sync_poly : nullptr)) != MUON_OK)
      return st;
    Bf16Stack Hs{H, L.m, L.m, L.ldg, mstride_g, K};
    if (t + 1 < ns_steps) {
      st = launch_apply(Hs, X, xb[(t + 1) & 1], sc, err, to, s, deps ? &sync_last : nullptr);
    } else {
      st = launch_final(Hs, X, sc, fin, err, to, s, deps ? &sync_last : nullptr);
    }
    if (st != MUON_OK) return st;
  }
  return MUON_OK;
}

// Pieces of a step. Every call runs its stacks' steps piece by piece: a stack of more than the piece size
// (in elements) is cut along K into equal slices of at most that size, each running its whole step (norm
// pass, chain, final step) before the next starts. Each matrix's arithmetic is the same in any slice, so
// this changes no result; what it changes is the working set of consecutive launches. On the Llama-3-8B set
// (7 G Muon elements at the 1.4 kW power cap) one call over everything took 338 ms, one call per bucket
// 324 ms, and pieces of 0.4, 0.75 and 1.5 G elements 312-313 ms: with fewer matrices in flight, more of
// each launch's operands are still in L2 from the launch before, the step moves fewer DRAM bytes per flop,
// and the power-capped clock runs about 10% higher (1560-1610 against 1400-1470 MHz).
std::atomic<long long> g_piece_elems{512ll << 20};

// The K-slices [k0, k1) of a stack of K matrices of A x B: one if it fits a piece, else equal parts.
std::vector<std::pair<int64_t, int64_t>> stack_slices(int64_t K, int64_t A, int64_t B) {
  const long double elems = static_cast<long double>(K) * A * B;
  const long long piece = g_piece_elems.load();
  int64_t parts = elems <= piece ? 1 : static_cast<int64_t>(std::ceil(elems / piece));
  parts = std::max<int64_t>(1, std::min<int64_t>(parts, K));
  std::vector<std::pair<int64_t, int64_t>> out;
  for (int64_t i = 0; i < parts; ++i) out.emplace_back(K * i / parts, K * (i + 1) / parts);
  return out;
}

}  // namespace
}  // namespace muon

using namespace muon;

extern "C" {

size_t muon_workspace_bytes(int64_t K, int64_t A, int64_t B) {
  if (K < 1 || A < 1 || B < 1) return 0;
  return header_bytes(K) + layout(K, A, B).total;
}

muon_status muon_step_batched(void *const *params, muon_dtype pdt, const void *const *grads, muon_dtype gdt,
                              float *momentum, int64_t K, int64_t A, int64_t B, const muon_hparams *hp, void *ws,
                              size_t ws_bytes, muon_stream_t stream) {
  if (params == nullptr || grads == nullptr || momentum == nullptr || hp == nullptr || ws == nullptr)
    return MUON_ERR_INVALID_ARG;
  muon_status st = check_stack_dims(K, A, B);
  if (st != MUON_OK) return st;
  if (!valid_dtype(pdt) || !valid_dtype(gdt)) return MUON_ERR_DTYPE;
  if ((st = check_coeffs(hp->ns_steps, hp->coeffs)) != MUON_OK) return st;
  if (hp->scale_mode != 0 && hp->scale_mode != 1) return MUON_ERR_INVALID_ARG;
  if (!std::isfinite(hp->lr) || !std::isfinite(hp->momentum) || !std::isfinite(hp->weight_decay) ||
      !std::isfinite(hp->eps) || hp->eps < 0.f)
    return MUON_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return MUON_ERR_ALIGNMENT;
  const Layout L = layout(K, A, B);
  if (ws_bytes < header_bytes(K) + L.total) return MUON_ERR_WORKSPACE;
  if ((st = check_device()) != MUON_OK) return st;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char *base = static_cast<char *>(ws);
  unsigned *counters = reinterpret_cast<unsigned *>(base + CTRL_BYTES);
  const double scale = hp->scale_mode == 0 ? 0.2 * std::sqrt(static_cast<double>(A > B ? A : B))
                                           : std::sqrt(std::max(1.0, static_cast<double>(A) / static_cast<double>(B)));
  for (const auto &sl : stack_slices(K, A, B)) {
    // one piece: matrices k0 .. k1 - 1, in the workspace from its start
    const int64_t k0 = sl.first, Kp = sl.second - sl.first;
    const Layout Lp = layout(Kp, A, B);
    char *w = base + header_bytes(Kp);
    if ((st = launch_counter_reset(counters, 4 * Kp, s)) != MUON_OK) return st;
    const NesterovArgs na = nesterov_args(w, Lp, counters, Kp, A, B, grads + k0, nullptr, gdt, momentum + k0 * A * B,
                                          hp->momentum, hp->nesterov != 0, hp->eps);
    if ((st = launch_nesterov_norm(&na, 1, s)) != MUON_OK) return st;
    FinalSpec fin{};
    fin.params = params + k0;
    fin.out_dense = nullptr;
    fin.dtype = pdt;
    fin.transposed = na.transposed;
    fin.orig_cols = static_cast<int>(B);
    fin.cautious = hp->cautious_wd ? 1 : 0;
    fin.lr_wd = static_cast<float>(static_cast<double>(hp->lr) * hp->weight_decay);
    fin.lr_scale = static_cast<float>(static_cast<double>(hp->lr) * scale);
    if ((st = run_ns_chain(reinterpret_cast<uint32_t *>(base), w, Lp, Kp, hp->ns_steps, hp->coeffs, fin, s, counters,
                           static_cast<uint32_t>(na.tiles_r * na.tiles_c))) != MUON_OK)
      return st;
  }
  return MUON_OK;
}

static muon_status check_bucket(const muon_bucket &b) {
  if (b.params == nullptr || b.grads == nullptr || b.momentum == nullptr) return MUON_ERR_INVALID_ARG;
  muon_status st = check_stack_dims(b.K, b.A, b.B);
  if (st != MUON_OK) return st;
  if (!valid_dtype(b.pdt) || !valid_dtype(b.gdt)) return MUON_ERR_DTYPE;
  if (b.master != nullptr && b.pdt != MUON_BF16) return MUON_ERR_DTYPE;
  return MUON_OK;
}

size_t muon_workspace_bytes_grouped(const muon_bucket *buckets, int n) {
  if (buckets == nullptr || n < 1) return 0;
  size_t total = 0;
  long long total_K = 0;
  for (int i = 0; i < n; ++i) {
    if (buckets[i].K < 1 || buckets[i].A < 1 || buckets[i].B < 1) return 0;
    total += layout(buckets[i].K, buckets[i].A, buckets[i].B).total;
    total_K += buckets[i].K;
  }
  return header_bytes(total_K) + total;
}

// Every argument check of muon_step_grouped (the device check excepted).
static muon_status check_grouped(const muon_bucket *buckets, int n, const muon_hparams *hp, void *ws,
                                 size_t ws_bytes) {
  if (buckets == nullptr || hp == nullptr || ws == nullptr || n < 1 || n > 4096) return MUON_ERR_INVALID_ARG;
  muon_status st;
  for (int i = 0; i < n; ++i)
    if ((st = check_bucket(buckets[i])) != MUON_OK) return st;
  if ((st = check_coeffs(hp->ns_steps, hp->coeffs)) != MUON_OK) return st;
  if (hp->scale_mode != 0 && hp->scale_mode != 1) return MUON_ERR_INVALID_ARG;
  if (!std::isfinite(hp->lr) || !std::isfinite(hp->momentum) || !std::isfinite(hp->weight_decay) ||
      !std::isfinite(hp->eps) || hp->eps < 0.f)
    return MUON_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return MUON_ERR_ALIGNMENT;
  if (ws_bytes < muon_workspace_bytes_grouped(buckets, n)) return MUON_ERR_WORKSPACE;
  return MUON_OK;
}

}  // extern "C"

namespace muon_grouped_detail {
using namespace muon;

// Matrices k0 .. k1 - 1 of a bucket, as a bucket of their own.
muon_bucket bucket_slice(const muon_bucket &b, int64_t k0, int64_t k1) {
  muon_bucket s = b;
  s.params = b.params + k0;
  s.grads = b.grads + k0;
  s.momentum = b.momentum + k0 * b.A * b.B;
  s.master = b.master != nullptr ? b.master + k0 : nullptr;
  s.K = k1 - k0;
  return s;
}

// The pieces of a grouped step, in order: each slice of a bucket larger than a piece on its own (stack_slices
// cuts it exactly as a call on that bucket alone would), and runs of consecutive smaller buckets packed
// together up to the piece size.
std::vector<std::vector<muon_bucket>> grouped_pieces(const muon_bucket *buckets, int n) {
  std::vector<std::vector<muon_bucket>> out;
  std::vector<muon_bucket> cur;
  long double cur_elems = 0;
  const long long piece = g_piece_elems.load();
  auto flush = [&] {
    if (!cur.empty()) out.push_back(cur);
    cur.clear();
    cur_elems = 0;
  };
  for (int i = 0; i < n; ++i) {
    const muon_bucket &b = buckets[i];
    const auto slices = stack_slices(b.K, b.A, b.B);
    if (slices.size() > 1) {
      flush();
      for (const auto &sl : slices) out.push_back({bucket_slice(b, sl.first, sl.second)});
      continue;
    }
    const long double e = static_cast<long double>(b.K) * b.A * b.B;
    if (!cur.empty() && cur_elems + e > piece) flush();
    cur.push_back(b);
    cur_elems += e;
  }
  flush();
  return out;
}

// Where a stack's Newton-Schulz chain runs.
enum : int { PATH_SMALL = 0, PATH_GRAM = 1, PATH_PLAIN = 2 };

// One stack of a grouped call, as the chain issuer sees it.
struct ChainStack {
  Layout L;
  char *w;               // the stack's sections
  long long K, k0;       // matrices; the first one's index in the call's counters
  uint32_t norm_done;    // the norm counter's value once the stack's U and scales are stored
  FinalSpec fin;
  int path;
};

// What the chain issuer needs besides the stacks.
struct ChainCall {
  uint32_t *err;
  uint32_t *counters;    // the header's four counters per matrix
  long long total_K;
  int ns_steps;
  const float *coeffs;
  bool norm_wait;        // the first Gram launch waits on the norm counters (false: no norm pass precedes)
  int deps;              // plain chain: -1 the table or the rule, 0 launch order, 1 per-matrix counters
};

// The plain stacks' (m, n, K) in order: the key of a grouped chain's measured scheduling mode.
std::vector<long long> plain_signature(const std::vector<ChainStack> &cs) {
  std::vector<long long> sig;
  for (const ChainStack &c : cs)
    if (c.path == PATH_PLAIN) sig.insert(sig.end(), {c.L.m, c.L.n, c.K});
  return sig;
}

std::mutex g_sched_mu;
std::map<std::vector<long long>, int> g_deps_table;   // plain-chain signature -> measured scheduling mode

int deps_lookup(const std::vector<long long> &sig) {
  std::lock_guard<std::mutex> lk(g_sched_mu);
  auto it = g_deps_table.find(sig);
  return it == g_deps_table.end() ? -1 : it->second;
}

// The chains of a grouped call, after its norm pass. Launch order: the branches first (small stacks: the whole
// chain in one fused launch each; Gram-space stacks: fp32 Gram, m x m chain, final step), each launch waiting
// for the whole previous grid; then the plain chain of the other stacks. Where the plain chain's launches wait
// per matrix on counters, its first launch also waits for the previous grid, so that the step's last launch
// completes only after every branch.
muon_status issue_chains(const std::vector<ChainStack> &cs, const ChainCall &cc, cudaStream_t s) {
  muon_status st;
  const unsigned long long to = g_timeout_ns;
  const int N = cc.ns_steps;
  bool branch = false;
  for (const ChainStack &c : cs) {
    if (c.path != PATH_SMALL) continue;
    branch = true;
    if ((st = launch_ns_small(small_args(cc.err, c.w, c.L, c.K, N, cc.coeffs, c.fin), s)) != MUON_OK) return st;
  }
  {
    GemmBatch g32(EPI_GRAM32, cc.err, to), fb(EPI_FINAL, cc.err, to);
    std::vector<GramSpaceStack> gs;
    for (const ChainStack &c : cs)
      if (c.path == PATH_GRAM && (st = add_gram_space(c.w, c.L, c.K, cc.coeffs, c.fin, g32, gs, fb)) != MUON_OK)
        return st;
    if (!gs.empty()) {
      branch = true;
      if ((st = launch_gram_space_batches(g32, gs, fb, N, cc.coeffs, cc.err, s)) != MUON_OK) return st;
    }
  }
  // scheduling of the plain chain: forced, else measured for this set of stacks, else the rule (per-matrix
  // counters where the launches, all stacks of a step kind in one, are short)
  bool deps;
  if (cc.deps >= 0) {
    deps = cc.deps == 1;
  } else if (g_counter_deps.load() >= 0) {
    deps = g_counter_deps.load() == 1;
  } else {
    const int measured = deps_lookup(plain_signature(cs));
    if (measured >= 0) {
      deps = measured == 1;
    } else {
      double est_us = 0.0;
      for (int kind = EPI_GRAM; kind <= EPI_APPLY; ++kind) {
        double us = 0.0;
        for (const ChainStack &c : cs)
          if (c.path == PATH_PLAIN) us += launch_estimate_us(kind, c.L.m, c.L.n, c.K);
        est_us = std::max(est_us, us);
      }
      deps = est_us <= 500.0;
    }
  }
  uint32_t *G_ready = cc.counters + cc.total_K, *H_ready = cc.counters + 2 * cc.total_K;
  uint32_t *X_ready = cc.counters + 3 * cc.total_K;
  for (int t = 0; t < N; ++t) {
    const float a = cc.coeffs[3 * t], b = cc.coeffs[3 * t + 1], c3 = cc.coeffs[3 * t + 2];
    GemmBatch gram(EPI_GRAM, cc.err, to), poly(EPI_POLY, cc.err, to);
    GemmBatch last(t + 1 < N ? EPI_APPLY : EPI_FINAL, cc.err, to);
    const bool half = g_half_sym.load() != 0;
    gram.half_symmetric(half);
    poly.half_symmetric(half);
    last.half_symmetric(half);
    if (t == 0 && branch) gram.force_grid_wait(true);
    for (const ChainStack &c : cs) {
      if (c.path != PATH_PLAIN) continue;
      const Layout &Li = c.L;
      const long long k0 = c.k0;
      const float *sc = t == 0 ? reinterpret_cast<const float *>(c.w + Li.scale) : nullptr;
      const uint32_t e_gram = gemm_signals_per_matrix(EPI_GRAM, Li.m, Li.n);
      const uint32_t e_poly = gemm_signals_per_matrix(EPI_POLY, Li.m, Li.n);
      const uint32_t e_apply = gemm_signals_per_matrix(EPI_APPLY, Li.m, Li.n);
      const uint32_t tt = static_cast<uint32_t>(t);
      // GRAM of step 0 reads the norm pass's output: a matrix's norm counter reaches its tile count plus one
      // once its U and scale are stored
      const TileSync sync_gram{t == 0 ? (cc.norm_wait ? cc.counters + k0 : nullptr) : X_ready + k0,
                               t == 0 ? c.norm_done : tt * e_apply, G_ready + k0};
      const TileSync sync_poly{G_ready + k0, (tt + 1) * e_gram, H_ready + k0};
      const TileSync sync_last{H_ready + k0, (tt + 1) * e_poly, t + 1 < N ? X_ready + k0 : nullptr};
      __nv_bfloat16 *xb[2] = {reinterpret_cast<__nv_bfloat16 *>(c.w + Li.x0),
                              reinterpret_cast<__nv_bfloat16 *>(c.w + Li.x1)};
      __nv_bfloat16 *G = reinterpret_cast<__nv_bfloat16 *>(c.w + Li.g);
      __nv_bfloat16 *H = reinterpret_cast<__nv_bfloat16 *>(c.w + Li.h);
      const long long K = c.K, msx = Li.m * Li.ldx, msg = Li.m * Li.ldg;
      Bf16Stack X{xb[t & 1], Li.m, Li.n, Li.ldx, msx, K};
      Bf16Stack Gs{G, Li.m, Li.m, Li.ldg, msg, K};
      Bf16Stack Hs{H, Li.m, Li.m, Li.ldg, msg, K};
      if ((st = gram.add_gram(X, G, Li.ldg, msg, 1.0f, sc, deps ? &sync_gram : nullptr)) != MUON_OK) return st;
      if ((st = poly.add_poly(Gs, H, Li.ldg, msg, a, b, c3, deps ? &sync_poly : nullptr)) != MUON_OK) return st;
      if (t + 1 < N) {
        st = last.add_apply(Hs, X, xb[(t + 1) & 1], sc, deps ? &sync_last : nullptr);
      } else {
        st = last.add_final(Hs, X, sc, c.fin, deps ? &sync_last : nullptr);
      }
      if (st != MUON_OK) return st;
    }
    if ((st = gram.launch(s)) != MUON_OK || (st = poly.launch(s)) != MUON_OK || (st = last.launch(s)) != MUON_OK)
      return st;
  }
  return MUON_OK;
}

FinalSpec final_spec_of(const muon_bucket &bk, const muon_hparams *hp) {
  const double scale = hp->scale_mode == 0
                           ? 0.2 * std::sqrt(static_cast<double>(bk.A > bk.B ? bk.A : bk.B))
                           : std::sqrt(std::max(1.0, static_cast<double>(bk.A) / static_cast<double>(bk.B)));
  FinalSpec fin{};
  fin.params = bk.params;
  fin.master = bk.master;
  fin.dtype = bk.pdt;
  fin.transposed = bk.A > bk.B ? 1 : 0;
  fin.orig_cols = static_cast<int>(bk.B);
  fin.cautious = hp->cautious_wd ? 1 : 0;
  fin.lr_wd = static_cast<float>(static_cast<double>(hp->lr) * hp->weight_decay);
  fin.lr_scale = static_cast<float>(static_cast<double>(hp->lr) * scale);
  return fin;
}

// The stacks of a grouped call over workspace ws: layouts, sections, counters and paths (by the route rule,
// the measured table, or the debug switch).
std::vector<ChainStack> chain_stacks(const muon_bucket *buckets, int n, const muon_hparams *hp, char *base,
                                     long long *total_K_out) {
  long long total_K = 0;
  for (int i = 0; i < n; ++i) total_K += buckets[i].K;
  std::vector<ChainStack> cs(n);
  size_t off = header_bytes(total_K);
  for (long long i = 0, k0 = 0; i < n; k0 += buckets[i].K, ++i) {
    ChainStack &c = cs[i];
    c.L = layout(buckets[i].K, buckets[i].A, buckets[i].B);
    c.w = base + off;
    off += c.L.total;
    c.K = buckets[i].K;
    c.k0 = k0;
    c.fin = final_spec_of(buckets[i], hp);
    c.path = ns_small_fits(c.L.m, c.L.n) ? PATH_SMALL
             : gram_space_route(c.L.m, c.L.n, c.K) ? PATH_GRAM
                                                  : PATH_PLAIN;
  }
  *total_K_out = total_K;
  return cs;
}

// Median device time of five runs of fn (after one warm-up run) on stream s, in ms; <0 on a CUDA error.
template <typename F>
float median_time(F fn, cudaStream_t s, muon_status *st) {
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
    if (e0) cudaEventDestroy(e0);
    *st = MUON_ERR_CUDA;
    return -1.f;
  }
  constexpr int REPS = 5;
  float t[REPS];
  *st = fn();
  for (int r = 0; r < REPS && *st == MUON_OK; ++r) {
    if (cudaEventRecord(e0, s) != cudaSuccess) *st = MUON_ERR_CUDA;
    if (*st == MUON_OK) *st = fn();
    if (*st == MUON_OK && (cudaEventRecord(e1, s) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
                           cudaEventElapsedTime(&t[r], e0, e1) != cudaSuccess))
      *st = MUON_ERR_CUDA;
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (*st != MUON_OK) return -1.f;
  std::sort(t, t + REPS);
  return t[REPS / 2];
}

// Every timed run of the autotune works on the workspace alone: the chains start from whatever iterate x0 holds
// (no norm pass, so parameters, gradients and momentum are not read) and the final step writes a dense bf16
// output into an iterate buffer the chain no longer reads, instead of updating parameters. Times do not depend
// on the values. This sets a stack up that way for its current path (call again after changing the path).
void timing_final(ChainStack &c, int ns_steps) {
  c.norm_done = 0;
  c.fin = FinalSpec{};
  c.fin.dtype = MUON_BF16;
  c.fin.orig_cols = static_cast<int>(c.L.n);
  // plain chain: the final step reads iterate (N - 1) & 1; the Gram-space and small paths read only x0
  const bool x0_free = c.path == PATH_PLAIN && ((ns_steps - 1) & 1) == 1;
  c.fin.out_dense = c.w + (x0_free ? c.L.x0 : c.L.x1);
}

}  // namespace muon_grouped_detail

extern "C" {

// One piece of a grouped step (all of it, for a set within one piece), in the workspace from its start.
static muon_status enqueue_piece(const muon_bucket *buckets, int n, const muon_hparams *hp, void *ws, cudaStream_t s,
                                 unsigned *extra_zero, long long extra_n) {
  using namespace muon_grouped_detail;
  muon_status st;
  char *base = static_cast<char *>(ws);
  long long total_K = 0;
  std::vector<ChainStack> cs = chain_stacks(buckets, n, hp, base, &total_K);
  unsigned *counters = reinterpret_cast<unsigned *>(base + CTRL_BYTES);
  // (extra_zero: more counters to clear in the same launch, for a call that follows this chain)
  if ((st = launch_counter_reset(counters, 4 * total_K, s, extra_zero, extra_n)) != MUON_OK) return st;
  // momentum, Nesterov input, norm: all buckets in one pass
  std::vector<NesterovArgs> na(n);
  for (int i = 0; i < n; ++i) {
    const muon_bucket &bk = buckets[i];
    na[i] = nesterov_args(cs[i].w, cs[i].L, counters + cs[i].k0, bk.K, bk.A, bk.B, bk.grads, nullptr, bk.gdt,
                          bk.momentum, hp->momentum, hp->nesterov != 0, hp->eps);
    cs[i].norm_done = static_cast<uint32_t>(na[i].tiles_r * na[i].tiles_c) + 1u;
  }
  if ((st = launch_nesterov_norm(na.data(), n, s)) != MUON_OK) return st;
  ChainCall cc{reinterpret_cast<uint32_t *>(base), counters, total_K, hp->ns_steps, hp->coeffs, true, -1};
  return issue_chains(cs, cc, s);
}

// The launches of one grouped Muon step, piece by piece (grouped_pieces), on stream s (arguments already
// checked). extra_zero / extra_n: counters of a call that follows this step, cleared with the first piece's.
static muon_status enqueue_grouped(const muon_bucket *buckets, int n, const muon_hparams *hp, void *ws,
                                   cudaStream_t s, unsigned *extra_zero = nullptr, long long extra_n = 0) {
  muon_status st;
  bool first = true;
  for (const auto &piece : muon_grouped_detail::grouped_pieces(buckets, n)) {
    if ((st = enqueue_piece(piece.data(), static_cast<int>(piece.size()), hp, ws, s, first ? extra_zero : nullptr,
                            first ? extra_n : 0)) != MUON_OK)
      return st;
    first = false;
  }
  return MUON_OK;
}

muon_status muon_step_grouped(const muon_bucket *buckets, int n, const muon_hparams *hp, void *ws, size_t ws_bytes,
                              muon_stream_t stream) {
  muon_status st;
  if ((st = check_grouped(buckets, n, hp, ws, ws_bytes)) != MUON_OK || (st = check_device()) != MUON_OK) return st;
  return enqueue_grouped(buckets, n, hp, ws, reinterpret_cast<cudaStream_t>(stream));
}

muon_status ns_orthogonalize(const void *x, muon_dtype xdt, void *out, muon_dtype odt, int64_t K, int64_t A,
                             int64_t B, int ns_steps, const float *coeffs, float eps, void *ws, size_t ws_bytes,
                             muon_stream_t stream) {
  if (ws == nullptr) return MUON_ERR_INVALID_ARG;
  muon_status st = check_ns_args(x, xdt, out, odt, K, A, B, ns_steps, coeffs, eps);
  if (st != MUON_OK) return st;
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return MUON_ERR_ALIGNMENT;
  const Layout L = layout(K, A, B);
  if (ws_bytes < header_bytes(K) + L.total) return MUON_ERR_WORKSPACE;
  if ((st = check_device()) != MUON_OK) return st;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char *base = static_cast<char *>(ws);
  unsigned *counters = reinterpret_cast<unsigned *>(base + CTRL_BYTES);
  const size_t xe = xdt == MUON_F32 ? 4 : 2, oe = odt == MUON_F32 ? 4 : 2;
  for (const auto &sl : stack_slices(K, A, B)) {
    // one piece: matrices k0 .. k1 - 1, in the workspace from its start
    const int64_t k0 = sl.first, Kp = sl.second - sl.first;
    const Layout Lp = layout(Kp, A, B);
    char *w = base + header_bytes(Kp);
    if ((st = launch_counter_reset(counters, 4 * Kp, s)) != MUON_OK) return st;
    const NesterovArgs na = nesterov_args(w, Lp, counters, Kp, A, B, nullptr,
                                          static_cast<const char *>(x) + k0 * A * B * xe, xdt, nullptr, 0.f, false,
                                          eps);
    if ((st = launch_nesterov_norm(&na, 1, s)) != MUON_OK) return st;
    FinalSpec fin{};
    fin.params = nullptr;
    fin.out_dense = static_cast<char *>(out) + k0 * A * B * oe;
    fin.dtype = odt;
    fin.transposed = na.transposed;
    fin.orig_cols = static_cast<int>(B);
    if ((st = run_ns_chain(reinterpret_cast<uint32_t *>(base), w, Lp, Kp, ns_steps, coeffs, fin, s, counters,
                           static_cast<uint32_t>(na.tiles_r * na.tiles_c))) != MUON_OK)
      return st;
  }
  return MUON_OK;
}

// Validates AdamW hyperparameters and derives the kernel constants.
static muon_status adamw_constants(const adamw_hparams *hp, AdamwConst *out) {
  if (hp->step < 1 || !std::isfinite(hp->lr) || !std::isfinite(hp->beta1) || !std::isfinite(hp->beta2) ||
      !std::isfinite(hp->eps) || !std::isfinite(hp->weight_decay) || hp->beta1 < 0.f || hp->beta1 >= 1.f ||
      hp->beta2 < 0.f || hp->beta2 >= 1.f || (hp->l2 != 0 && hp->l2 != 1))
    return MUON_ERR_INVALID_ARG;
  const double t = static_cast<double>(hp->step);
  const double bc1 = 1.0 - std::pow(static_cast<double>(hp->beta1), t);
  const double bc2 = 1.0 - std::pow(static_cast<double>(hp->beta2), t);
  AdamwConst &c = *out;
  c.l2 = hp->l2;
  c.l2_wd = hp->l2 ? hp->weight_decay : 0.f;
  c.decay = hp->l2 ? 1.f : static_cast<float>(1.0 - static_cast<double>(hp->lr) * hp->weight_decay);
  c.beta1 = hp->beta1;
  c.one_minus_beta1 = static_cast<float>(1.0 - hp->beta1);
  c.beta2 = hp->beta2;
  c.one_minus_beta2 = static_cast<float>(1.0 - hp->beta2);
  c.step_size = static_cast<float>(hp->lr / bc1);
  c.inv_sqrt_bc2 = static_cast<float>(1.0 / std::sqrt(bc2));
  c.eps = hp->eps;
  return MUON_OK;
}

muon_status adamw_step(void *param, muon_dtype pdt, const void *grad, muon_dtype gdt, float *exp_avg,
                       float *exp_avg_sq, int64_t n, const adamw_hparams *hp, muon_stream_t stream) {
  if (param == nullptr || grad == nullptr || exp_avg == nullptr || exp_avg_sq == nullptr || hp == nullptr)
    return MUON_ERR_INVALID_ARG;
  if (n < 1) return MUON_ERR_INVALID_ARG;
  if (!valid_dtype(pdt) || !valid_dtype(gdt)) return MUON_ERR_DTYPE;
  AdamwConst c{};
  muon_status st = adamw_constants(hp, &c);
  if (st != MUON_OK) return st;
  if ((st = check_device()) != MUON_OK) return st;
  return launch_adamw(param, pdt, grad, gdt, exp_avg, exp_avg_sq, n, c, reinterpret_cast<cudaStream_t>(stream));
}

muon_status adamw_step_master(float *master, void *param, const void *grad, muon_dtype gdt, float *exp_avg,
                              float *exp_avg_sq, int64_t n, const adamw_hparams *hp, muon_stream_t stream) {
  if (master == nullptr || param == nullptr || grad == nullptr || exp_avg == nullptr || exp_avg_sq == nullptr ||
      hp == nullptr)
    return MUON_ERR_INVALID_ARG;
  if (n < 1) return MUON_ERR_INVALID_ARG;
  if (!valid_dtype(gdt)) return MUON_ERR_DTYPE;
  AdamwConst c{};
  muon_status st = adamw_constants(hp, &c);
  if (st != MUON_OK) return st;
  if ((st = check_device()) != MUON_OK) return st;
  return launch_adamw_master(master, static_cast<__nv_bfloat16 *>(param), grad, gdt, exp_avg, exp_avg_sq, n, c,
                             reinterpret_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------------------------------ autotune

}  // extern "C"

static muon_status autotune_piece(const muon_bucket *buckets, int n, const muon_hparams *hp, void *ws,
                                  cudaStream_t s);

extern "C" {

muon_status muon_autotune(const muon_bucket *buckets, int n, const muon_hparams *hp, void *ws, size_t ws_bytes,
                          muon_stream_t stream) {
  using namespace muon_grouped_detail;
  if (buckets == nullptr || hp == nullptr || ws == nullptr || n < 1 || n > 4096) return MUON_ERR_INVALID_ARG;
  muon_status st;
  for (int i = 0; i < n; ++i)
    if ((st = check_bucket(buckets[i])) != MUON_OK) return st;
  if ((st = check_coeffs(hp->ns_steps, hp->coeffs)) != MUON_OK) return st;
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return MUON_ERR_ALIGNMENT;
  if (ws_bytes < muon_workspace_bytes_grouped(buckets, n)) return MUON_ERR_WORKSPACE;
  if ((st = check_device()) != MUON_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the pieces the step runs (grouped_pieces), each measured once per distinct (A, B, K) list
  const auto pieces = grouped_pieces(buckets, n);
  std::set<std::vector<long long>> seen;
  for (const auto &piece : pieces) {
    std::vector<long long> sig;
    for (const muon_bucket &b : piece) sig.insert(sig.end(), {b.A, b.B, b.K});
    if (!seen.insert(sig).second) continue;
    if ((st = autotune_piece(piece.data(), static_cast<int>(piece.size()), hp, ws, s)) != MUON_OK) return st;
  }
  // 3. the plain chain's scheduling, per-matrix counters or launch order, for a step that runs as one piece: its
  // chains timed each way. A step of several pieces keeps the rule: the timed runs leave out the norm pass (they
  // may not read the state), and on the Llama-3-8B set they found the counters faster, by piece and over every
  // piece in turn, while the real step, whose first Gram launches then overlap the norm pass at the power cap,
  // was 2% slower with them.
  if (g_counter_deps.load() < 0 && pieces.size() == 1) {
    char *base = static_cast<char *>(ws);
    uint32_t *err = reinterpret_cast<uint32_t *>(base);
    unsigned *counters = reinterpret_cast<unsigned *>(base + CTRL_BYTES);
    const int N = hp->ns_steps;
    std::vector<std::vector<ChainStack>> sets;
    std::vector<long long> ks;
    bool any_plain = false;
    for (const auto &piece : pieces) {
      long long tk = 0;
      sets.push_back(chain_stacks(piece.data(), static_cast<int>(piece.size()), hp, base, &tk));
      ks.push_back(tk);
      for (ChainStack &c : sets.back()) {
        timing_final(c, N);
        any_plain = any_plain || c.path == PATH_PLAIN;
      }
    }
    if (any_plain) {
      float t_mode[2];
      for (int deps = 0; deps < 2; ++deps) {
        t_mode[deps] = median_time(
            [&]() -> muon_status {
              for (size_t i = 0; i < sets.size(); ++i) {
                muon_status r = launch_counter_reset(counters, 4 * ks[i], s);
                if (r != MUON_OK) return r;
                ChainCall cc{err, counters, ks[i], N, hp->coeffs, false, deps};
                if ((r = issue_chains(sets[i], cc, s)) != MUON_OK) return r;
              }
              return MUON_OK;
            },
            s, &st);
        if (st != MUON_OK) return st;
      }
      std::lock_guard<std::mutex> lk(g_sched_mu);
      for (const auto &set : sets) {
        const auto sig = plain_signature(set);
        if (!sig.empty()) g_deps_table[sig] = t_mode[1] < t_mode[0] ? 1 : 0;
      }
    }
  }
  return muon_check(ws, stream) == MUON_ERR_TIMEOUT ? MUON_ERR_TIMEOUT : MUON_OK;
}

}  // extern "C"

// The measurements of muon_autotune on one piece of the step, in the workspace from its start.
static muon_status autotune_piece(const muon_bucket *buckets, int n, const muon_hparams *hp, void *ws,
                                  cudaStream_t s) {
  using namespace muon_grouped_detail;
  muon_status st;
  char *base = static_cast<char *>(ws);
  uint32_t *err = reinterpret_cast<uint32_t *>(base);
  unsigned *counters = reinterpret_cast<unsigned *>(base + CTRL_BYTES);
  long long total_K = 0;
  std::vector<ChainStack> cs = chain_stacks(buckets, n, hp, base, &total_K);
  const int N = hp->ns_steps;
  for (ChainStack &c : cs) timing_final(c, N);
  auto dense_out = [&](ChainStack &c) { timing_final(c, N); };
  auto run = [&](std::vector<ChainStack> &set, int deps) -> muon_status {
    muon_status r = launch_counter_reset(counters, 4 * total_K, s);
    if (r != MUON_OK) return r;
    ChainCall cc{err, counters, total_K, N, hp->coeffs, false, deps};
    return issue_chains(set, cc, s);
  };
  // 1. the path of each stack that can take the Gram-space chain: each way, that stack alone
  for (ChainStack &c : cs) {
    if (c.path == PATH_SMALL || !gram_space_eligible(c.L.m, c.L.n) || g_gram_space.load() >= 0) continue;
    float best = -1.f;
    int best_path = c.path;
    for (int path : {PATH_GRAM, PATH_PLAIN}) {
      c.path = path;
      dense_out(c);
      std::vector<ChainStack> one{c};
      const float ms = median_time([&] { return run(one, -1); }, s, &st);
      if (st != MUON_OK) return st;
      if (best < 0.f || ms < best) {
        best = ms;
        best_path = path;
      }
    }
    c.path = best_path;
    std::lock_guard<std::mutex> lk(g_route_mu);
    g_route_table[{c.L.m, c.L.n, c.K}] = best_path == PATH_GRAM ? 1 : 0;
  }
  for (ChainStack &c : cs) dense_out(c);
  // 1b. the slices of the Gram-space stacks' fp32 Gram launch (reads the iterate, writes the Gram-space planes)
  bool any_gram = false;
  for (const ChainStack &c : cs) any_gram = any_gram || c.path == PATH_GRAM;
  if (any_gram && gram_split_forced() < 0) {
    auto gram32_batch = [&](GemmBatch &g32) -> muon_status {
      for (const ChainStack &c : cs) {
        if (c.path != PATH_GRAM) continue;
        __nv_bfloat16 *planes = reinterpret_cast<__nv_bfloat16 *>(c.w + c.L.gs);
        const long long ldm = round8(c.L.m), msm = c.L.m * ldm;
        Bf16Stack X{c.w + c.L.x0, c.L.m, c.L.n, c.L.ldx, c.L.m * c.L.ldx, c.K};
        muon_status r = g32.add_gram32(X, planes, ldm, msm, c.K * msm, 2LL * GS_B * c.K * msm, hp->coeffs[1],
                                       hp->coeffs[2], 1.0f, nullptr);
        if (r != MUON_OK) return r;
      }
      return MUON_OK;
    };
    int best = 1;
    float best_ms = -1.f;
    for (int split = 1; split <= GRAM32_MAX_SPLIT; ++split) {
      const float ms = median_time(
          [&]() -> muon_status {
            GemmBatch g32(EPI_GRAM32, err, g_timeout_ns);
            g32.force_split(split);
            muon_status r = gram32_batch(g32);
            return r != MUON_OK ? r : g32.launch(s);
          },
          s, &st);
      if (st != MUON_OK) return st;
      if (best_ms < 0.f || ms < best_ms) {
        best = split;
        best_ms = ms;
      }
    }
    for (const ChainStack &c : cs)
      if (c.path == PATH_GRAM) gram_split_record(c.L.m, static_cast<int>((c.L.n + 63) / 64), c.K, best);
  }
  // 2. the poly step's pipeline shape, on the plain stacks' grouped poly launch (reads G, writes H)
  int max_k = 0;
  bool any_plain = false;
  for (const ChainStack &c : cs)
    if (c.path == PATH_PLAIN) {
      any_plain = true;
      max_k = std::max(max_k, static_cast<int>((c.L.m + 63) / 64));
    }
  if (any_plain) {
    int best = -1;
    float best_ms = 0.f;
    for (int shape = 0; shape < POLY_SHAPES; ++shape) {
      const float ms = median_time(
          [&]() -> muon_status {
            GemmBatch poly(EPI_POLY, err, g_timeout_ns);
            poly.force_shape(shape);
            poly.half_symmetric(g_half_sym.load() != 0);   // as the chain runs it
            for (const ChainStack &c : cs) {
              if (c.path != PATH_PLAIN) continue;
              const long long msg = c.L.m * c.L.ldg;
              Bf16Stack Gs{c.w + c.L.g, c.L.m, c.L.m, c.L.ldg, msg, c.K};
              muon_status r = poly.add_poly(Gs, reinterpret_cast<__nv_bfloat16 *>(c.w + c.L.h), c.L.ldg, msg,
                                            hp->coeffs[0], hp->coeffs[1], hp->coeffs[2]);
              if (r != MUON_OK) return r;
            }
            return poly.launch(s);
          },
          s, &st);
      if (st != MUON_OK) return st;
      if (best < 0 || ms < best_ms) {
        best = shape;
        best_ms = ms;
      }
    }
    poly_shape_record(max_k, best);
  }
  return MUON_OK;
}

extern "C" {

int32_t muon_autotune_route(int64_t K, int64_t A, int64_t B) {
  if (K < 1 || A < 1 || B < 1) return -1;
  std::lock_guard<std::mutex> lk(g_route_mu);
  auto it = g_route_table.find({std::min(A, B), std::max(A, B), K});
  return it == g_route_table.end() ? -1 : it->second;
}

int32_t muon_autotune_scheduling(const muon_bucket *buckets, int n) {
  using namespace muon_grouped_detail;
  if (buckets == nullptr || n < 1 || n > 4096) return -1;
  for (int i = 0; i < n; ++i)
    if (buckets[i].K < 1 || buckets[i].A < 1 || buckets[i].B < 1) return -1;
  // the step's pieces: the record of each piece that has a plain chain
  int found = -3;   // none seen yet
  for (const auto &piece : grouped_pieces(buckets, n)) {
    std::vector<long long> sig;
    for (const muon_bucket &b : piece) {
      const long long m = std::min(b.A, b.B), nn = std::max(b.A, b.B);
      if (ns_small_fits(m, nn) || gram_space_route(m, nn, b.K)) continue;
      sig.insert(sig.end(), {m, nn, static_cast<long long>(b.K)});
    }
    if (sig.empty()) continue;
    const int r = deps_lookup(sig);
    if (r < 0) return -1;
    if (found == -3) found = r;
    else if (found != r) return 2;
  }
  return found == -3 ? -1 : found;
}

int32_t muon_autotune_poly_shape(int64_t contraction) {
  if (contraction < 1 || contraction > (1 << 20)) return -1;
  return poly_shape_lookup(static_cast<int>((contraction + 63) / 64));
}

int32_t muon_autotune_gram_split(int64_t K, int64_t A, int64_t B) {
  if (K < 1 || A < 1 || B < 1 || A > 65536 || B > 65536) return -1;
  return gram_split_lookup(std::min(A, B), static_cast<int>((std::max(A, B) + 63) / 64), K);
}

void muon_autotune_reset(void) {
  poly_shape_clear();
  gram_split_clear();
  {
    std::lock_guard<std::mutex> lk(g_route_mu);
    g_route_table.clear();
  }
  std::lock_guard<std::mutex> lk(muon_grouped_detail::g_sched_mu);
  muon_grouped_detail::g_deps_table.clear();
}

muon_status muon_debug_counter_deps(int32_t on) {
  if (on < -1 || on > 1) return MUON_ERR_INVALID_ARG;
  g_counter_deps.store(on);
  return MUON_OK;
}

muon_status muon_debug_half_symmetric(int32_t on) {
  if (on < 0 || on > 1) return MUON_ERR_INVALID_ARG;
  g_half_sym.store(on);
  return MUON_OK;
}

muon_status muon_debug_gram_space(int32_t mode) {
  if (mode < -1 || mode > 1) return MUON_ERR_INVALID_ARG;
  g_gram_space.store(mode);
  return MUON_OK;
}

int32_t muon_gram_space_route(int64_t K, int64_t A, int64_t B) {
  if (K < 1 || A < 1 || B < 1) return 0;
  return gram_space_route(std::min(A, B), std::max(A, B), K) ? 1 : 0;
}

muon_status muon_debug_piece_elems(int64_t elems) {
  if (elems < 0) return MUON_ERR_INVALID_ARG;
  g_piece_elems.store(elems == 0 ? (512ll << 20) : elems);
  return MUON_OK;
}

muon_status muon_debug_gram_split(int32_t split) {
  if (split < -1 || split == 0 || split > GRAM32_MAX_SPLIT) return MUON_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_tune_mu);
  g_gram_split_forced = split;
  return MUON_OK;
}

muon_status muon_debug_poly_shape(int32_t shape) {
  if (shape < -1 || shape >= POLY_SHAPES) return MUON_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_tune_mu);
  g_poly_forced = shape;
  return MUON_OK;
}

// ------------------------------------------------------------------------------------------ grouped AdamW

static int64_t adamw_passes(int64_t n) { return (n + ADAMW_GROUP_MAX - 1) / ADAMW_GROUP_MAX; }

// Checks every tensor and builds one launch argument block per pass of up to ADAMW_GROUP_MAX tensors, each
// with its counter region in ws.
static muon_status build_adamw_groups(const adamw_tensor *t, int64_t n, void *ws, size_t ws_bytes,
                                      std::vector<AdamwGroup> &out) {
  if (t == nullptr || ws == nullptr || n < 1 || n > (1 << 20)) return MUON_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return MUON_ERR_ALIGNMENT;
  if (ws_bytes < adamw_workspace_bytes_grouped(n)) return MUON_ERR_WORKSPACE;
  auto aligned = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
  out.assign(static_cast<size_t>(adamw_passes(n)), AdamwGroup{});
  for (int64_t i = 0; i < n; ++i) {
    const adamw_tensor &x = t[i];
    if (x.param == nullptr || x.grad == nullptr || x.exp_avg == nullptr || x.exp_avg_sq == nullptr ||
        x.hp == nullptr || x.n < 1)
      return MUON_ERR_INVALID_ARG;
    if (!valid_dtype(x.pdt) || !valid_dtype(x.gdt)) return MUON_ERR_DTYPE;
    if (x.master != nullptr && x.pdt != MUON_BF16) return MUON_ERR_DTYPE;
    AdamwGroup &G = out[static_cast<size_t>(i / ADAMW_GROUP_MAX)];
    AdamwTensorDesc &d = G.t[G.ntensors];
    muon_status st = adamw_constants(x.hp, &d.c);
    if (st != MUON_OK) return st;
    d.p = x.param;
    d.g = x.grad;
    d.m = x.exp_avg;
    d.v = x.exp_avg_sq;
    d.master = x.master;
    d.n = x.n;
    d.pdt = x.pdt;
    d.gdt = x.gdt;
    d.vec = aligned(x.param) && aligned(x.grad) && aligned(x.exp_avg) && aligned(x.exp_avg_sq) &&
            (x.master == nullptr || aligned(x.master));
    ++G.ntensors;
  }
  for (size_t k = 0; k < out.size(); ++k)
    out[k].next = reinterpret_cast<unsigned long long *>(static_cast<char *>(ws) + k * ADAMW_REGION_BYTES);
  return MUON_OK;
}

// Chunk size and numbering per launch (after the device check, which gives the SM count): about eight
// chunks per warp of a full grid (10 blocks of 3 warps per SM), so that the last chunks, which a few warps
// finish alone, are a small part of the pass; at least 256 elements, at most ADAMW_CHUNK_MAX.
static void number_adamw_chunks(std::vector<AdamwGroup> &groups) {
  const long long warps = static_cast<long long>(device_sm_count()) * 10 * (ADAMW_THREADS / 32);
  for (AdamwGroup &G : groups) {
    long long elems = 0;
    for (int k = 0; k < G.ntensors; ++k) elems += G.t[k].n;
    long long c = (elems / std::max(1LL, 8 * warps) + 255) / 256 * 256;
    G.chunk = std::min(ADAMW_CHUNK_MAX, std::max(256LL, c));
    G.total_chunks = 0;
    for (int k = 0; k < G.ntensors; ++k) {
      G.t[k].chunk_begin = G.total_chunks;
      G.total_chunks += (G.t[k].n + G.chunk - 1) / G.chunk;
    }
  }
}

size_t adamw_workspace_bytes_grouped(int64_t n) {
  if (n < 1) return 0;
  return static_cast<size_t>(adamw_passes(n)) * ADAMW_REGION_BYTES;
}

static muon_status reset_adamw_regions(void *ws, size_t passes, cudaStream_t s) {
  return launch_counter_reset(static_cast<unsigned *>(ws),
                              static_cast<long long>(passes * ADAMW_REGION_BYTES / sizeof(unsigned)), s);
}

muon_status adamw_step_grouped(const adamw_tensor *tensors, int64_t n, void *ws, size_t ws_bytes,
                               muon_stream_t stream) {
  std::vector<AdamwGroup> groups;
  muon_status st = build_adamw_groups(tensors, n, ws, ws_bytes, groups);
  if (st != MUON_OK || (st = check_device()) != MUON_OK) return st;
  number_adamw_chunks(groups);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = reset_adamw_regions(ws, groups.size(), s)) != MUON_OK) return st;
  for (const AdamwGroup &G : groups)
    if ((st = launch_adamw_grouped(G, s)) != MUON_OK) return st;
  return MUON_OK;
}

// ------------------------------------------------------------------------------------------ hybrid step

muon_status hybrid_step(const muon_bucket *buckets, int nb, const muon_hparams *hp, void *ws, size_t ws_bytes,
                        const adamw_tensor *tensors, int64_t nt, void *adamw_ws, size_t adamw_ws_bytes,
                        muon_stream_t stream) {
  if (nb < 0 || nt < 0 || (nb == 0 && nt == 0)) return MUON_ERR_INVALID_ARG;
  muon_status st;
  if (nb > 0 && (st = check_grouped(buckets, nb, hp, ws, ws_bytes)) != MUON_OK) return st;
  std::vector<AdamwGroup> groups;
  if (nt > 0 && (st = build_adamw_groups(tensors, nt, adamw_ws, adamw_ws_bytes, groups)) != MUON_OK) return st;
  if (nb > 0 && nt > 0) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(ws), a1 = a0 + muon_workspace_bytes_grouped(buckets, nb);
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(adamw_ws), b1 = b0 + adamw_workspace_bytes_grouped(nt);
    if (a0 < b1 && b0 < a1) return MUON_ERR_INVALID_ARG;
  }
  if ((st = check_device()) != MUON_OK) return st;
  number_adamw_chunks(groups);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // with both parts, the AdamW chunk counters are cleared by the Muon step's own counter reset
  const long long adamw_words =
      nt > 0 ? static_cast<long long>(groups.size() * ADAMW_REGION_BYTES / sizeof(unsigned)) : 0;
  if (nb > 0 && (st = enqueue_grouped(buckets, nb, hp, ws, s, static_cast<unsigned *>(adamw_ws), adamw_words)) !=
                    MUON_OK)
    return st;
  if (nt > 0) {
    if (nb == 0 && (st = reset_adamw_regions(adamw_ws, groups.size(), s)) != MUON_OK) return st;
    for (const AdamwGroup &G : groups)
      if ((st = launch_adamw_grouped(G, s)) != MUON_OK) return st;
  }
  return MUON_OK;
}

static muon_status check_step_stack(const void *p, int64_t K, int64_t m, int64_t n) {
  if (p == nullptr) return MUON_ERR_INVALID_ARG;
  muon_status st = check_stack_dims(K, m, n);
  if (st != MUON_OK) return st;
  if (m % 8 != 0 || n % 8 != 0) return MUON_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(p) & 255) != 0) return MUON_ERR_ALIGNMENT;
  return MUON_OK;
}

static muon_status check_ws_ctrl(void *ws, size_t ws_bytes) {
  if (ws == nullptr) return MUON_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return MUON_ERR_ALIGNMENT;
  if (ws_bytes < CTRL_BYTES) return MUON_ERR_WORKSPACE;
  return MUON_OK;
}

muon_status ns_gram(const void *x, void *g, int64_t K, int64_t m, int64_t n, float alpha, void *ws, size_t ws_bytes,
                    muon_stream_t stream) {
  muon_status st;
  if ((st = check_step_stack(x, K, m, n)) != MUON_OK || (st = check_step_stack(g, K, m, m)) != MUON_OK ||
      (st = check_ws_ctrl(ws, ws_bytes)) != MUON_OK)
    return st;
  if (!std::isfinite(alpha)) return MUON_ERR_INVALID_ARG;
  if ((st = check_device()) != MUON_OK) return st;
  Bf16Stack X{x, m, n, n, m * n, K};
  return launch_gram(X, static_cast<__nv_bfloat16 *>(g), m, m * m, alpha, nullptr, static_cast<uint32_t *>(ws),
                     g_timeout_ns, reinterpret_cast<cudaStream_t>(stream));
}

muon_status ns_poly(const void *g, void *h, int64_t K, int64_t m, float a, float b, float c, void *ws,
                    size_t ws_bytes, muon_stream_t stream) {
  muon_status st;
  if ((st = check_step_stack(g, K, m, m)) != MUON_OK || (st = check_step_stack(h, K, m, m)) != MUON_OK ||
      (st = check_ws_ctrl(ws, ws_bytes)) != MUON_OK)
    return st;
  if (!std::isfinite(a) || !std::isfinite(b) || !std::isfinite(c)) return MUON_ERR_INVALID_ARG;
  if ((st = check_device()) != MUON_OK) return st;
  Bf16Stack G{g, m, m, m, m * m, K};
  return launch_poly(G, static_cast<__nv_bfloat16 *>(h), m, m * m, a, b, c, static_cast<uint32_t *>(ws),
                     g_timeout_ns, reinterpret_cast<cudaStream_t>(stream));
}

muon_status ns_apply(const void *h, const void *x, void *out, int64_t K, int64_t m, int64_t n, void *ws,
                     size_t ws_bytes, muon_stream_t stream) {
  muon_status st;
  if ((st = check_step_stack(h, K, m, m)) != MUON_OK || (st = check_step_stack(x, K, m, n)) != MUON_OK ||
      (st = check_step_stack(out, K, m, n)) != MUON_OK || (st = check_ws_ctrl(ws, ws_bytes)) != MUON_OK)
    return st;
  if (out == x) return MUON_ERR_INVALID_ARG;
  if ((st = check_device()) != MUON_OK) return st;
  Bf16Stack Hs{h, m, m, m, m * m, K};
  Bf16Stack X{x, m, n, n, m * n, K};
  // out has x's layout: launch_apply writes with x's pitches
  return launch_apply(Hs, X, static_cast<__nv_bfloat16 *>(out), nullptr, static_cast<uint32_t *>(ws),
                      g_timeout_ns, reinterpret_cast<cudaStream_t>(stream));
}

muon_status muon_plan_buckets(int64_t n, const int64_t *rows, const int64_t *cols, int64_t *bucket_id,
                              int64_t *index_in_bucket, int64_t *n_buckets, int64_t *bucket_shapes, int64_t *bucket_K,
                              int64_t *momentum_offset) {
  if (n < 0 || n_buckets == nullptr) return MUON_ERR_INVALID_ARG;
  if (n > 0 && (rows == nullptr || cols == nullptr || bucket_id == nullptr || index_in_bucket == nullptr ||
                bucket_shapes == nullptr || bucket_K == nullptr || momentum_offset == nullptr))
    return MUON_ERR_INVALID_ARG;
  for (int64_t i = 0; i < n; ++i)
    if (rows[i] < 1 || cols[i] < 1) return MUON_ERR_INVALID_ARG;
  // exact (rows, cols) -> bucket; buckets numbered in order of first appearance
  std::map<std::pair<int64_t, int64_t>, int64_t> seen;
  int64_t nb = 0;
  for (int64_t i = 0; i < n; ++i) {
    const auto key = std::make_pair(rows[i], cols[i]);
    auto it = seen.find(key);
    int64_t b;
    if (it == seen.end()) {
      b = nb++;
      seen.emplace(key, b);
      bucket_shapes[2 * b] = rows[i];
      bucket_shapes[2 * b + 1] = cols[i];
      bucket_K[b] = 0;
    } else {
      b = it->second;
    }
    bucket_id[i] = b;
    index_in_bucket[i] = bucket_K[b]++;
  }
  int64_t off = 0;
  for (int64_t b = 0; b < nb; ++b) {
    momentum_offset[b] = off;
    off += bucket_K[b] * bucket_shapes[2 * b] * bucket_shapes[2 * b + 1];
  }
  *n_buckets = nb;
  return MUON_OK;
}

muon_status muon_check(void *ws, muon_stream_t stream) {
  if (ws == nullptr) return MUON_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MUON_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return MUON_ERR_CUDA;
  if (word == 0) return MUON_OK;
  const uint32_t zero = 0;
  if (cudaMemcpy(ws, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return MUON_ERR_CUDA;
  return MUON_ERR_TIMEOUT;
}

void muon_set_timeout_ns(uint64_t ns) { muon::g_timeout_ns = ns > 0 ? ns : 1; }

muon_status muon_debug_wait_timeout(void *ws, size_t ws_bytes, uint64_t timeout_ns, muon_stream_t stream) {
  muon_status st = check_ws_ctrl(ws, ws_bytes);
  if (st != MUON_OK) return st;
  if (timeout_ns == 0 || timeout_ns > 10000000000ull) return MUON_ERR_INVALID_ARG;
  if ((st = check_device()) != MUON_OK) return st;
  return launch_debug_wait(static_cast<uint32_t *>(ws), timeout_ns, reinterpret_cast<cudaStream_t>(stream));
}

muon_status muon_debug_timeline(void *buf, int64_t bytes, int32_t records_per_cta) {
  if (buf == nullptr || bytes <= 0 || records_per_cta <= 0) {
    muon::g_timeline = nullptr;
    muon::g_timeline_cap = 0;
    return MUON_OK;
  }
  if (muon::device_check() != MUON_OK) return MUON_ERR_UNSUPPORTED_DEVICE;
  const int64_t region = static_cast<int64_t>(muon::device_sm_count()) * records_per_cta * 10;
  if (bytes < region * 8) return MUON_ERR_WORKSPACE;
  std::lock_guard<std::mutex> lk(muon::g_trace_mu);
  muon::g_timeline = static_cast<unsigned long long *>(buf);
  muon::g_timeline_cap = records_per_cta;
  muon::g_timeline_region_words = region;
  muon::g_timeline_regions = bytes / (region * 8);
  muon::g_timeline_next = 0;
  return MUON_OK;
}

int64_t muon_launch_count(void) {
  std::lock_guard<std::mutex> lk(muon::g_trace_mu);
  return muon::g_launches;
}

void muon_trace_enable(int on) {
  std::lock_guard<std::mutex> lk(muon::g_trace_mu);
  muon::g_trace_on = on != 0;
}

int64_t muon_trace_collect(int32_t *kinds, float *ms, int64_t cap) {
  std::lock_guard<std::mutex> lk(muon::g_trace_mu);
  int64_t written = 0;
  bool failed = false;
  for (auto &r : muon::g_trace) {
    if (cudaEventSynchronize(r.stop) != cudaSuccess) failed = true;
    float t = 0.f;
    if (!failed && cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess) failed = true;
    if (written < cap && kinds != nullptr && ms != nullptr) {
      kinds[written] = r.kind;
      ms[written] = t;
      ++written;
    }
    muon::g_event_pool.push_back(r.start);
    muon::g_event_pool.push_back(r.stop);
  }
  muon::g_trace.clear();
  return failed ? -1 : written;
}

const char *muon_kernel_name(int32_t kind) {
  switch (kind) {
    case KK_ADAMW: return "adamw";
    case KK_NESTEROV_NORM: return "nesterov_norm";
    case KK_COUNTER_RESET: return "counter_reset";
    case KK_GRAM: return "ns_gram";
    case KK_POLY: return "ns_poly";
    case KK_APPLY: return "ns_apply";
    case KK_FINAL: return "ns_final";
    case KK_DEBUG_WAIT: return "debug_wait";
    case KK_NS_SMALL: return "ns_small";
    case KK_GRAM_SPACE: return "ns_gram_space";
    case KK_GRAM32: return "ns_gram_f32";
    case KK_GRAM32_REDUCE: return "ns_gram_f32_reduce";
    default: return "unknown";
  }
}

const char *muon_status_string(muon_status s) {
  switch (s) {
    case MUON_OK: return "MUON_OK";
    case MUON_ERR_INVALID_ARG: return "MUON_ERR_INVALID_ARG: null pointer, non-positive size or bad hyperparameter";
    case MUON_ERR_SHAPE: return "MUON_ERR_SHAPE: dimension outside the supported range";
    case MUON_ERR_DTYPE: return "MUON_ERR_DTYPE: unsupported dtype";
    case MUON_ERR_ALIGNMENT: return "MUON_ERR_ALIGNMENT: pointer not aligned as required";
    case MUON_ERR_WORKSPACE: return "MUON_ERR_WORKSPACE: workspace missing or too small";
    case MUON_ERR_UNSUPPORTED_DEVICE: return "MUON_ERR_UNSUPPORTED_DEVICE: current device is not a GB300 (sm_103)";
    case MUON_ERR_CUDA: return "MUON_ERR_CUDA: a CUDA call failed";
    case MUON_ERR_TIMEOUT: return "MUON_ERR_TIMEOUT: a bounded device-side wait ran out";
    default: return "unknown muon_status";
  }
}

}  // extern "C"
