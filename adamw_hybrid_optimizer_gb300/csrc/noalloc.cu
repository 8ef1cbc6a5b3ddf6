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
// The array holds a workspace laid out exactly as ns_orthogonalize's (internal.h: header_bytes and
// layout), so a stack fits when muon_workspace_bytes(K, A, B) is at most its size. It is shared by every
// call on a device and keeps the last call's contents. Each call clears the part that must start at zero
// (the per-matrix counters of the header) with an asynchronous memset, which allocates nothing; every
// other scratch byte is written before it is read. The error word at its start is sticky: a bounded wait
// that runs out sets it, and only ns_orthogonalize_noalloc_check reads and clears it. Calls whose work
// overlaps on the GPU (different streams, or several host threads) race on the array.
//
// This path runs the chain as separate launches per step (Gram, polynomial, apply), also for stacks that
// ns_orthogonalize hands to the fused small-matrix kernel.
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

// Set-up, once per device, with that device current: the device address of the scratch array (in host
// code the array's name is only a host-side stand-in, never a device address), and a zeroed control
// block. The memset is synchronous, so the first call on a device should come before any stream capture.
muon_status noalloc_scratch(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MUON_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MUON_ERR_CUDA;
    if (cudaMemset(p, 0, CTRL_BYTES) != cudaSuccess) return MUON_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return MUON_OK;
}

}  // namespace
}  // namespace muon

using namespace muon;

extern "C" muon_status ns_orthogonalize_noalloc(const void *x, muon_dtype xdt, void *out, muon_dtype odt, int64_t K,
                                                int64_t A, int64_t B, int ns_steps, const float *coeffs, float eps,
                                                muon_stream_t stream) {
  muon_status st = check_ns_args(x, xdt, out, odt, K, A, B, ns_steps, coeffs, eps);
  if (st != MUON_OK) return st;
  // the bound in floating point first, so that huge stacks cannot overflow the layout arithmetic
  const long double mn = static_cast<long double>(A < B ? A : B);
  if (4.0L * K * A * B + 4.0L * K * mn * mn > static_cast<long double>(NOALLOC_SCRATCH_BYTES))
    return MUON_ERR_WORKSPACE;
  const Layout L = layout(K, A, B);
  const size_t hdr = header_bytes(K);
  if (hdr + L.total > NOALLOC_SCRATCH_BYTES) return MUON_ERR_WORKSPACE;
  if ((st = device_check()) != MUON_OK) return st;
  void *scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != MUON_OK) return st;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char *base = static_cast<char *>(scratch);
  uint32_t *err = reinterpret_cast<uint32_t *>(base);
  unsigned *counters = reinterpret_cast<unsigned *>(base + CTRL_BYTES);
  char *w = base + hdr;
  // the per-matrix counters start at zero; the error word (sticky) is left alone
  if (cudaMemsetAsync(counters, 0, hdr - CTRL_BYTES, s) != cudaSuccess) return MUON_ERR_CUDA;

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
  na.counters = counters;
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

// Reads and clears the scratch's error word after the stream's work is done. A small synchronous copy
// into a host variable and a memset: nothing is allocated.
extern "C" muon_status ns_orthogonalize_noalloc_check(muon_stream_t stream) {
  muon_status st = device_check();
  if (st != MUON_OK) return st;
  void *scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != MUON_OK) return st;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return MUON_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, scratch, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return MUON_ERR_CUDA;
  if (word == 0) return MUON_OK;
  if (cudaMemset(scratch, 0, sizeof(word)) != cudaSuccess) return MUON_ERR_CUDA;
  return MUON_ERR_TIMEOUT;
}

// The bounded-wait test kernel of muon_debug_wait_timeout, reporting into the scratch's error word.
extern "C" muon_status muon_debug_wait_timeout_noalloc(uint64_t timeout_ns, muon_stream_t stream) {
  if (timeout_ns == 0 || timeout_ns > 10000000000ull) return MUON_ERR_INVALID_ARG;
  muon_status st = device_check();
  if (st != MUON_OK) return st;
  void *scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != MUON_OK) return st;
  return launch_debug_wait(static_cast<uint32_t *>(scratch), timeout_ns, reinterpret_cast<cudaStream_t>(stream));
}
