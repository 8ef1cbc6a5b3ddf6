// ns_orthogonalize_noalloc: Newton-Schulz orthogonalisation of a stack without any device
// allocation, neither by the library nor by the caller.
//
// Who needs it: callers that cannot call cudaMalloc (or any allocating routine) and so cannot hand
// the library a workspace -- for example code that runs inside a device-memory allocator's own
// hooks, where allocating would re-enter the allocator; plugins of a host program that gives them no
// way to allocate device memory; or runtimes whose device-memory budget is fixed when they start.
// They pass only their input and output buffers; the scratch lives in this file's static device
// array, which every GPU that loads this code holds until the process exits.
//
// The array is shared by every call on a device and keeps the last call's contents. Each call clears
// the part that must start at zero (the control block with the error word, and one counter per
// matrix) with an asynchronous memset, which allocates nothing; every other scratch byte is written
// before it is read. Calls whose
// work overlaps on the GPU (different streams, or several host threads) race on the array.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/libmuon.h"
#include "internal.h"

namespace muon {
namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(64) << 20;   // the stated maximum: 64 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[64] = {};

// Once per device, with that device current: the device address of the scratch array. In host code
// the array's name is only a host-side stand-in, never a device address.
muon_status noalloc_scratch(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MUON_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MUON_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return MUON_OK;
}

size_t up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct ScratchLayout {
  long long m, n, ldx, ldg, tiles_r, tiles_c;
  size_t counters, scale, partial, x0, x1, g, h, total;
};

// Control block and per-matrix counters (the zeroed part), then the same sections the workspace of
// ns_orthogonalize holds.
ScratchLayout scratch_layout(long long K, long long A, long long B) {
  ScratchLayout L{};
  L.m = A < B ? A : B;
  L.n = A < B ? B : A;
  L.ldx = (L.n + 7) / 8 * 8;
  L.ldg = (L.m + 7) / 8 * 8;
  L.tiles_r = (A + NESTEROV_TILE - 1) / NESTEROV_TILE;
  L.tiles_c = (B + NESTEROV_TILE - 1) / NESTEROV_TILE;
  size_t off = 256;
  L.counters = off;
  off = up(off + size_t(K) * 4, 1024);
  L.scale = off;
  off = up(off + size_t(K) * 4, 1024);
  L.partial = off;
  off = up(off + size_t(K) * L.tiles_r * L.tiles_c * 4, 1024);
  L.x0 = off;
  off = up(off + size_t(K) * L.m * L.ldx * 2, 1024);
  L.x1 = off;
  off = up(off + size_t(K) * L.m * L.ldx * 2, 1024);
  L.g = off;
  off = up(off + size_t(K) * L.m * L.ldg * 2, 1024);
  L.h = off;
  off = up(off + size_t(K) * L.m * L.ldg * 2, 1024);
  L.total = off;
  return L;
}

}  // namespace
}  // namespace muon

using namespace muon;

extern "C" muon_status ns_orthogonalize_noalloc(const void *x, muon_dtype xdt, void *out, muon_dtype odt, int64_t K,
                                                int64_t A, int64_t B, int ns_steps, const float *coeffs, float eps,
                                                muon_stream_t stream) {
  if (x == nullptr || out == nullptr || coeffs == nullptr) return MUON_ERR_INVALID_ARG;
  if (K < 1 || A < 1 || B < 1) return MUON_ERR_INVALID_ARG;
  if (A > 65536 || B > 65536 || K > (1ll << 31)) return MUON_ERR_SHAPE;
  if ((xdt != MUON_F32 && xdt != MUON_BF16) || (odt != MUON_F32 && odt != MUON_BF16)) return MUON_ERR_DTYPE;
  if (ns_steps < 1 || ns_steps > MUON_MAX_NS_STEPS) return MUON_ERR_INVALID_ARG;
  for (int i = 0; i < 3 * ns_steps; ++i)
    if (!(coeffs[i] == coeffs[i]) || coeffs[i] > 3.4e38f || coeffs[i] < -3.4e38f) return MUON_ERR_INVALID_ARG;
  if (!(eps >= 0.f) || eps > 3.4e38f) return MUON_ERR_INVALID_ARG;
  // checked in floating point first so that huge stacks cannot overflow the layout arithmetic
  const long double approx = 4.0L * K * A * B + 4.0L * K * (long double)(A < B ? A : B) * (A < B ? A : B);
  if (approx > (long double)NOALLOC_SCRATCH_BYTES) return MUON_ERR_WORKSPACE;
  const ScratchLayout L = scratch_layout(K, A, B);
  if (L.total > NOALLOC_SCRATCH_BYTES) return MUON_ERR_WORKSPACE;
  muon_status st = device_check();
  if (st != MUON_OK) return st;
  void *scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != MUON_OK) return st;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char *w = static_cast<char *>(scratch);
  uint32_t *err = reinterpret_cast<uint32_t *>(w);
  if (cudaMemsetAsync(w, 0, L.scale, s) != cudaSuccess) return MUON_ERR_CUDA;

  NesterovArgs na{};
  na.gptrs = nullptr;
  na.gbase = x;
  na.gdtype = xdt;
  na.momentum = nullptr;
  na.u = reinterpret_cast<__nv_bfloat16 *>(w + L.x0);
  na.ldu = L.ldx;
  na.mstride_u = L.m * L.ldx;
  na.partials = reinterpret_cast<float *>(w + L.partial);
  na.scale = reinterpret_cast<float *>(w + L.scale);
  na.counters = reinterpret_cast<unsigned *>(w + L.counters);
  na.K = static_cast<int>(K);
  na.A = static_cast<int>(A);
  na.B = static_cast<int>(B);
  na.tiles_r = static_cast<int>(L.tiles_r);
  na.tiles_c = static_cast<int>(L.tiles_c);
  na.transposed = A > B ? 1 : 0;
  na.eps = eps;
  const float *scale = na.scale;
  if ((st = launch_nesterov_norm(&na, 1, s)) != MUON_OK) return st;

  FinalSpec fin{};
  fin.params = nullptr;
  fin.out_dense = out;
  fin.dtype = odt;
  fin.transposed = na.transposed;
  fin.orig_cols = static_cast<int>(B);
  __nv_bfloat16 *xb[2] = {reinterpret_cast<__nv_bfloat16 *>(w + L.x0), reinterpret_cast<__nv_bfloat16 *>(w + L.x1)};
  __nv_bfloat16 *G = reinterpret_cast<__nv_bfloat16 *>(w + L.g);
  __nv_bfloat16 *H = reinterpret_cast<__nv_bfloat16 *>(w + L.h);
  const long long msx = L.m * L.ldx, msg = L.m * L.ldg;
  const unsigned long long to = wait_timeout_ns();
  for (int t = 0; t < ns_steps; ++t) {
    const float a = coeffs[3 * t], b = coeffs[3 * t + 1], c = coeffs[3 * t + 2];
    const float *sc = t == 0 ? scale : nullptr;
    Bf16Stack X{xb[t & 1], L.m, L.n, L.ldx, msx, K};
    if ((st = launch_gram(X, G, L.ldg, msg, 1.0f, sc, err, to, s)) != MUON_OK) return st;
    Bf16Stack Gs{G, L.m, L.m, L.ldg, msg, K};
    if ((st = launch_poly(Gs, H, L.ldg, msg, a, b, c, err, to, s)) != MUON_OK) return st;
    Bf16Stack Hs{H, L.m, L.m, L.ldg, msg, K};
    if (t + 1 < ns_steps)
      st = launch_apply(Hs, X, xb[(t + 1) & 1], sc, err, to, s);
    else
      st = launch_final(Hs, X, sc, fin, err, to, s);
    if (st != MUON_OK) return st;
  }
  return MUON_OK;
}
