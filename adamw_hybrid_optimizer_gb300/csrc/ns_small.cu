// The whole Newton-Schulz chain of a small matrix in one CTA ("Optimizers: AdamW, Muon and the distributed
// optimizer", section "Muon: orthogonalising the update"; the fused small-matrix execution of "DMuon",
// section 2.2, which keeps small problems resident on chip): for a wide iterate with m <= 128 rows and
// n <= 256 columns, X (bf16) and G / H (bf16) stay in shared memory and the accumulators in tensor memory
// across every step, so a stack of K matrices takes one launch of K CTAs instead of 3 launches per step.
//
// Per step t (coefficients a, b, c; s the Frobenius scale, applied at t = 0):
//     G = (t == 0 ? s^2 : 1) X X^T                 tcgen05.mma M = 128, N = m (padded), K = n
//     H = a I + b G + c G G                       M = 128, N = m, K = m (G symmetric, G G = G G^T)
//     X <- (t == 0 ? s : 1) H X   (t < N - 1)      M = 128, N = n, K = m (B = X read N-major)
//     last step: u = H X, then the parameter update (or the dense output) as the large path's final step.
// Shared-memory operands use one layout for both majornesses: 64-column chunks of 128 rows, each row 128
// bytes with a 128-byte swizzle (16-byte piece q of row r at piece position q ^ (r & 7)). Padding rows
// (>= m) and columns (>= n) hold zeros and stay zero through every step (H has no diagonal term there).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace muon {

namespace {

constexpr int SMALL_THREADS = 128;       // 4 warps: warp w owns tensor-memory lanes 32w .. 32w + 31
constexpr int SMALL_ROWS = 128;          // M of every MMA; rows of every shared-memory operand
constexpr int CHUNK_BYTES = SMALL_ROWS * 128;
constexpr uint32_t SMALL_TMEM_COLS = 256;

__device__ __forceinline__ uint32_t piece_off(int r, int c) {   // 16-byte piece holding columns c .. c+7
  return static_cast<uint32_t>((c >> 6) * CHUNK_BYTES + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4));
}

// D (128 x N, tensor memory) = A (128 x K, K-major) * B, B K-major (its rows are the N index) or N-major
// (its rows are the K index). One thread.
__device__ __forceinline__ void issue_mma(uint32_t d, uint32_t a_base, uint32_t b_base, int K, int N, bool b_mn) {
  const uint32_t idesc = idesc_bf16_f32(SMALL_ROWS, N, false, b_mn);
  for (int k = 0; k < K / 16; ++k) {
    const uint64_t adesc = smem_desc_sw128(a_base + (k >> 2) * CHUNK_BYTES + (k & 3) * 32, 16, 1024);
    const uint64_t bdesc = b_mn ? smem_desc_sw128(b_base + k * 16 * 128, CHUNK_BYTES, 1024)
                                : smem_desc_sw128(b_base + (k >> 2) * CHUNK_BYTES + (k & 3) * 32, 16, 1024);
    tc_mma_bf16(d, adesc, bdesc, idesc, k > 0 ? 1u : 0u);
  }
}

__device__ __forceinline__ void unpack8f(const uint4 &w, float *dst) {
  const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&w);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __bfloat1622float2(h[e]);
    dst[2 * e] = f.x;
    dst[2 * e + 1] = f.y;
  }
}
__device__ __forceinline__ uint4 pack8f(const float *src) {
  uint4 w;
  __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&w);
#pragma unroll
  for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(src[2 * e], src[2 * e + 1]);
  return w;
}

__device__ __forceinline__ float update_elem(float p, float u, const SmallNsArgs &a) {
  const float d = (!a.cautious || u * p > 0.f) ? a.lr_wd : 0.f;
  return fmaf(-a.lr_scale, u, fmaf(-d, p, p));
}

__global__ void __launch_bounds__(SMALL_THREADS) ns_small_kernel(const __grid_constant__ SmallNsArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int xchunks = (a.n + 63) / 64;
  uint8_t *xs = smem;                                  // X: xchunks chunks
  uint8_t *gh = smem + xchunks * CHUNK_BYTES;          // G, then H in place: 2 chunks
  uint64_t *bar = reinterpret_cast<uint64_t *>(gh + 2 * CHUNK_BYTES);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 1);
  int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int row = threadIdx.x;              // this thread's accumulator row (tensor-memory lane)
  const int k = blockIdx.x;                 // matrix of the stack
  const int m = a.m, n = a.n;
  const int mp = (m + 15) / 16 * 16;        // N of the m-wide products
  const int np = (n + 15) / 16 * 16;        // N of the n-wide product

  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, SMALL_TMEM_COLS);
    tmem_relinquish();
  }
  // operands written by earlier kernels are read only after the previous grid has completed
  pdl_wait();
  if (threadIdx.x == 0) pdl_launch_dependents();

  // X <- the matrix's wide U (rows >= m and columns >= n zero); G / H buffer zeroed
  const __nv_bfloat16 *u = a.u + static_cast<long long>(k) * a.mstride_u;
  for (int c = 0; c < xchunks * 64; c += 8) {
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (row < m) {
      const __nv_bfloat16 *src = u + static_cast<long long>(row) * a.ldu + c;
      if (c + 8 <= n) {
        w = *reinterpret_cast<const uint4 *>(src);
      } else if (c < n) {
        __nv_bfloat16 *h = reinterpret_cast<__nv_bfloat16 *>(&w);
        for (int e = 0; e < n - c; ++e) h[e] = src[e];
      }
    }
    *reinterpret_cast<uint4 *>(xs + piece_off(row, c)) = w;
  }
  for (int c = 0; c < 128; c += 8) *reinterpret_cast<uint4 *>(gh + piece_off(row, c)) = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_shared();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_lane = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  WaitCtl ctl{abort_flag, a.err, a.timeout_ns};
  const float s = a.scale != nullptr ? a.scale[k] : 1.f;
  const uint32_t xs_a = smem_u32(xs), gh_a = smem_u32(gh);
  uint32_t phase = 0;
  bool ok = true;

  // one MMA group on the tensor cores, then every thread waits for it (bounded)
  auto run = [&](uint32_t a_base, uint32_t b_base, int K, int N, bool b_mn) -> bool {
    if (threadIdx.x == 0) {
      tc_fence_after();
      issue_mma(tmem, a_base, b_base, K, N, b_mn);
      tc_commit(bar);
    }
    const bool w = wait_bounded(bar, phase, ctl, ERR_WAIT_FULL);
    phase ^= 1u;
    tc_fence_after();
    return __syncthreads_and(w) != 0;
  };
  // after the epilogue's shared-memory writes: visible to the next MMAs, and tensor-memory reads done
  auto publish = [&]() {
    fence_proxy_async_shared();
    tc_fence_before();
    __syncthreads();
  };

  for (int t = 0; ok && t < a.ns_steps; ++t) {
    const float ca = a.coeffs[3 * t], cb = a.coeffs[3 * t + 1], cc = a.coeffs[3 * t + 2];
    const bool last = t + 1 == a.ns_steps;
    // G = (t == 0 ? s^2 : 1) X X^T
    if (!(ok = run(xs_a, xs_a, np, mp, false))) break;
    {
      const float sc = t == 0 ? s * s : 1.f;
      for (int c0 = 0; c0 < mp; c0 += 32) {
        float v[32];
        tmem_ld_32x32b_x32(t_lane + c0, v);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (c0 + 8 * q >= mp) break;
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = sc * v[8 * q + e];
          *reinterpret_cast<uint4 *>(gh + piece_off(row, c0 + 8 * q)) = pack8f(f);
        }
      }
    }
    publish();
    // H = a I + b G + c G G, in place of G
    if (!(ok = run(gh_a, gh_a, mp, mp, false))) break;
    for (int c0 = 0; c0 < mp; c0 += 32) {
      float v[32];
      tmem_ld_32x32b_x32(t_lane + c0, v);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int c = c0 + 8 * q;
        if (c >= mp) break;
        uint4 *pc = reinterpret_cast<uint4 *>(gh + piece_off(row, c));
        float g[8];
        unpack8f(*pc, g);
#pragma unroll
        for (int e = 0; e < 8; ++e) g[e] = cb * g[e] + cc * v[8 * q + e] + ((c + e == row && row < m) ? ca : 0.f);
        *pc = pack8f(g);
      }
    }
    publish();
    // X' = H X (scaled by s at t = 0); the last step updates the parameters instead
    if (!(ok = run(gh_a, xs_a, mp, np, true))) break;
    const float sc = (t == 0) ? s : 1.f;
    if (!last) {
      for (int c0 = 0; c0 < np; c0 += 32) {
        float v[32];
        tmem_ld_32x32b_x32(t_lane + c0, v);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int c = c0 + 8 * q;
          if (c >= np) break;
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = sc * v[8 * q + e];
          *reinterpret_cast<uint4 *>(xs + piece_off(row, c)) = pack8f(f);
        }
      }
      publish();
      continue;
    }
    for (int c0 = 0; c0 < np; c0 += 32) {
      float v[32];
      tmem_ld_32x32b_x32(t_lane + c0, v);
      if (row >= m) continue;
#pragma unroll 4
      for (int j = 0; j < 32; ++j) {
        const int col = c0 + j;
        if (col >= n) break;
        const float uu = sc * v[j];
        // stored wide: element (row, col); stored tall: (col, row)
        const long long idx = a.transposed ? static_cast<long long>(col) * a.orig_cols + row
                                           : static_cast<long long>(row) * a.orig_cols + col;
        if (a.params == nullptr) {   // dense output of the orthogonalisation
          const long long o = static_cast<long long>(k) * m * n + idx;
          if (a.out_dtype == MUON_F32) static_cast<float *>(a.out_dense)[o] = uu;
          else static_cast<__nv_bfloat16 *>(a.out_dense)[o] = __float2bfloat16_rn(uu);
        } else if (a.master != nullptr) {
          float *mp_ = a.master[k] + idx;
          const float nv = update_elem(*mp_, uu, a);
          *mp_ = nv;
          static_cast<__nv_bfloat16 *>(a.params[k])[idx] = __float2bfloat16_rn(nv);
        } else if (a.out_dtype == MUON_F32) {
          float *p = static_cast<float *>(a.params[k]) + idx;
          *p = update_elem(*p, uu, a);
        } else {
          __nv_bfloat16 *p = static_cast<__nv_bfloat16 *>(a.params[k]) + idx;
          *p = __float2bfloat16_rn(update_elem(__bfloat162float(*p), uu, a));
        }
      }
    }
  }
  // a wait that ran out leaves an MMA group possibly in flight: it completes before tensor memory is freed
  if (!ok && threadIdx.x == 0) drain_wait(bar, phase ^ 1u, ctl);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, SMALL_TMEM_COLS);
  }
}

}  // namespace

bool ns_small_fits(long long m, long long n) { return m >= 1 && m <= 128 && n >= 1 && n <= 256; }

muon_status launch_ns_small(const SmallNsArgs &a, cudaStream_t s) {
  if (!ns_small_fits(a.m, a.n) || a.K < 1) return MUON_ERR_INVALID_ARG;
  const size_t smem = 1024 + static_cast<size_t>((a.n + 63) / 64 + 2) * CHUNK_BYTES + 64;
  static std::once_flag attr_once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  std::call_once(attr_once[dev & 63], [] {
    cudaFuncSetAttribute(ns_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(1024 + 6 * CHUNK_BYTES + 64));
  });
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.K));
  cfg.blockDim = dim3(SMALL_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  launch_begin(KK_NS_SMALL, s);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, ns_small_kernel, a);
  launch_end(s);
  return e == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
}

}  // namespace muon
