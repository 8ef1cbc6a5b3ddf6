// Bandwidth-bound kernels of the optimizer step.
//
//   nesterov_norm_kernel  momentum M <- mu M + G, Nesterov input U = G + mu M (or M), U stored bf16 in
//                         the wide orientation, and the Frobenius scale s_k = 1 / (||U_k||_F + eps)
//                         from per-tile sums of U^2 added in a fixed order by the matrix's last tile,
//                         which then counts the matrix as ready for the chain
//                         ("Optimizers: AdamW, Muon and the distributed optimizer", section "Muon:
//                         orthogonalising the update": the momentum rule and newton_schulz's first lines).
//   counter_reset_kernel  zeroes counters in stream order: the norm pass's and the chain's per-matrix
//                         counters, and the grouped AdamW pass's chunk counter.
//   adamw kernels         AdamW with bias correction and decoupled decay (same page, section "AdamW:
//                         decoupled weight decay"), or Adam with L2, 16-byte vector accesses when aligned:
//                         one tensor per launch (adamw_kernel, adamw_master_kernel) or many, warps taking
//                         element chunks from a counter (adamw_grouped_kernel).
//   debug_wait_kernel     one bounded wait on a barrier nothing completes.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <type_traits>
#include <utility>

#include "internal.h"
#include "ptx.cuh"

namespace muon {

namespace {

__device__ __forceinline__ float ld_f(const float *p, long long i) { return p[i]; }
__device__ __forceinline__ float ld_f(const __nv_bfloat16 *p, long long i) { return __bfloat162float(p[i]); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Block of 256 threads on one 64 x 64 tile (tr, tc) of matrix b of the stored (A x B) stack; thread
// (tx, ty) handles columns 4*tx..4*tx+3 of rows ty, ty+16, ty+32, ty+48. Returns the thread's sum of U^2.
template <typename GT, bool MOMENTUM, int TR>
__device__ __forceinline__ float nesterov_tile(const NesterovArgs &a, long long b, int tr, int tc,
                                               __nv_bfloat16 (*tile)[TR + 8]) {
  constexpr int T = NESTEROV_TILE;   // columns; TR rows
  const long long mat = static_cast<long long>(a.A) * a.B;
  const GT *g = a.gptrs != nullptr ? static_cast<const GT *>(a.gptrs[b])
                                   : static_cast<const GT *>(a.gbase) + b * mat;
  float *M = MOMENTUM ? a.momentum + b * mat : nullptr;
  __nv_bfloat16 *u = a.u + b * a.mstride_u;

  const int tx = threadIdx.x & 15;
  const int ty = threadIdx.x >> 4;
  const int c0 = tc * T + tx * 4;
  // vector path: the 4 columns are in range and both rows are 16-byte (M) / 4-element (G) aligned
  const bool vec = (a.B % 4 == 0) && (c0 + 4 <= a.B) &&
                   ((reinterpret_cast<uintptr_t>(g) & (4 * sizeof(GT) - 1)) == 0) &&
                   (!MOMENTUM || (reinterpret_cast<uintptr_t>(M) & 15) == 0);
  float ss = 0.f;
#pragma unroll 1
  for (int p0 = 0; p0 < TR / 16; p0 += 4) {
#pragma unroll
  for (int p = p0; p < p0 + 4; ++p) {
    const int lrow = ty + 16 * p;
    const int r = tr * TR + lrow;
    float uv[4] = {0.f, 0.f, 0.f, 0.f};
    if (r < a.A) {
      const long long base = static_cast<long long>(r) * a.B + c0;
      float gv[4], mv[4];
      if (vec) {
        if constexpr (sizeof(GT) == 4) {
          const float4 q = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(g) + base);
          gv[0] = q.x; gv[1] = q.y; gv[2] = q.z; gv[3] = q.w;
        } else {
          const uint2 q = *reinterpret_cast<const uint2 *>(reinterpret_cast<const __nv_bfloat16 *>(g) + base);
          const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&q.x));
          const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&q.y));
          gv[0] = lo.x; gv[1] = lo.y; gv[2] = hi.x; gv[3] = hi.y;
        }
        if constexpr (MOMENTUM) {
          const float4 q = *reinterpret_cast<const float4 *>(M + base);
          mv[0] = q.x; mv[1] = q.y; mv[2] = q.z; mv[3] = q.w;
        }
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const bool in = c0 + q < a.B;
          gv[q] = in ? ld_f(g, base + q) : 0.f;
          mv[q] = (MOMENTUM && in) ? M[base + q] : 0.f;
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if constexpr (MOMENTUM) {
          const float mn = fmaf(a.mu, mv[q], gv[q]);
          mv[q] = mn;
          uv[q] = a.nesterov ? fmaf(a.mu, mn, gv[q]) : mn;
        } else {
          uv[q] = gv[q];
        }
        if (c0 + q >= a.B) uv[q] = 0.f;
        ss = fmaf(uv[q], uv[q], ss);
      }
      if constexpr (MOMENTUM) {
        if (vec) {
          *reinterpret_cast<float4 *>(M + base) = make_float4(mv[0], mv[1], mv[2], mv[3]);
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (c0 + q < a.B) M[base + q] = mv[q];
        }
      }
      if (!a.transposed) {
        __nv_bfloat16 *dst = u + static_cast<long long>(r) * a.ldu + c0;
        if (c0 + 4 <= a.B) {
          __nv_bfloat162 w[2] = {__floats2bfloat162_rn(uv[0], uv[1]), __floats2bfloat162_rn(uv[2], uv[3])};
          *reinterpret_cast<uint2 *>(dst) = *reinterpret_cast<uint2 *>(w);
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (c0 + q < a.B) dst[q] = __float2bfloat16_rn(uv[q]);
        }
      }
    }
    if (a.transposed) {
#pragma unroll
      for (int q = 0; q < 4; ++q) tile[tx * 4 + q][lrow] = __float2bfloat16_rn(uv[q]);
    }
  }
  }
  if (a.transposed) {
    __syncthreads();
    // wide row = stored column, wide column = stored row: thread tx writes TR/16 consecutive elements of it
    constexpr int E = TR / 16;
    using Vec = typename std::conditional<E == 8, uint4, uint2>::type;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const int lc = ty + 16 * p;
      const int c = tc * T + lc;
      const int r0 = tr * TR + tx * E;
      if (c < a.B) {
        __nv_bfloat16 *dst = u + static_cast<long long>(c) * a.ldu + r0;
        if (r0 + E <= a.A) {
          *reinterpret_cast<Vec *>(dst) = *reinterpret_cast<const Vec *>(&tile[lc][tx * E]);
        } else {
#pragma unroll
          for (int q = 0; q < E; ++q)
            if (r0 + q < a.A) dst[q] = tile[lc][tx * E + q];
        }
      }
    }
  }
  return ss;
}

// As nesterov_tile for a matrix stored wide (not transposed), on a tile of 64 rows x 256 columns: thread
// (tx, ty) handles columns 4*tx..4*tx+3 of rows ty, ty+4, .., ty+60, four rows at a time, so that a warp
// covers 128 consecutive columns of one row. Returns the thread's sum of U^2.
template <typename GT, bool MOMENTUM>
__device__ __forceinline__ float nesterov_tile_wide(const NesterovArgs &a, long long b, int tr, int tc) {
  constexpr int TR = NESTEROV_TILE, TC = NESTEROV_WIDE_TILE;
  const long long mat = static_cast<long long>(a.A) * a.B;
  const GT *g = a.gptrs != nullptr ? static_cast<const GT *>(a.gptrs[b])
                                   : static_cast<const GT *>(a.gbase) + b * mat;
  float *M = MOMENTUM ? a.momentum + b * mat : nullptr;
  __nv_bfloat16 *u = a.u + b * a.mstride_u;
  const int tx = threadIdx.x & 63;
  const int ty = threadIdx.x >> 6;
  const int c0 = tc * TC + tx * 4;
  const bool vec = (a.B % 4 == 0) && (c0 + 4 <= a.B) &&
                   ((reinterpret_cast<uintptr_t>(g) & (4 * sizeof(GT) - 1)) == 0) &&
                   (!MOMENTUM || (reinterpret_cast<uintptr_t>(M) & 15) == 0);
  float ss = 0.f;
#pragma unroll 1
  for (int p0 = 0; p0 < TR / 4; p0 += 4) {
#pragma unroll
    for (int p = p0; p < p0 + 4; ++p) {
      const int r = tr * TR + ty + 4 * p;
      if (r >= a.A || c0 >= a.B) continue;
      const long long base = static_cast<long long>(r) * a.B + c0;
      float gv[4], mv[4], uv[4];
      if (vec) {
        if constexpr (sizeof(GT) == 4) {
          const float4 q = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(g) + base);
          gv[0] = q.x; gv[1] = q.y; gv[2] = q.z; gv[3] = q.w;
        } else {
          const uint2 q = *reinterpret_cast<const uint2 *>(reinterpret_cast<const __nv_bfloat16 *>(g) + base);
          const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&q.x));
          const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&q.y));
          gv[0] = lo.x; gv[1] = lo.y; gv[2] = hi.x; gv[3] = hi.y;
        }
        if constexpr (MOMENTUM) {
          const float4 q = *reinterpret_cast<const float4 *>(M + base);
          mv[0] = q.x; mv[1] = q.y; mv[2] = q.z; mv[3] = q.w;
        }
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const bool in = c0 + q < a.B;
          gv[q] = in ? ld_f(g, base + q) : 0.f;
          mv[q] = (MOMENTUM && in) ? M[base + q] : 0.f;
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if constexpr (MOMENTUM) {
          const float mn = fmaf(a.mu, mv[q], gv[q]);
          mv[q] = mn;
          uv[q] = a.nesterov ? fmaf(a.mu, mn, gv[q]) : mn;
        } else {
          uv[q] = gv[q];
        }
        if (c0 + q >= a.B) uv[q] = 0.f;
        ss = fmaf(uv[q], uv[q], ss);
      }
      if constexpr (MOMENTUM) {
        if (vec) {
          *reinterpret_cast<float4 *>(M + base) = make_float4(mv[0], mv[1], mv[2], mv[3]);
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (c0 + q < a.B) M[base + q] = mv[q];
        }
      }
      __nv_bfloat16 *dst = u + static_cast<long long>(r) * a.ldu + c0;
      if (c0 + 4 <= a.B) {
        __nv_bfloat162 w[2] = {__floats2bfloat162_rn(uv[0], uv[1]), __floats2bfloat162_rn(uv[2], uv[3])};
        *reinterpret_cast<uint2 *>(dst) = *reinterpret_cast<uint2 *>(w);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (c0 + q < a.B) dst[q] = __float2bfloat16_rn(uv[q]);
      }
    }
  }
  return ss;
}

// One launch over the tiles of every matrix of up to NESTEROV_MAX_PROBLEMS stacks (blocks in problem order,
// within a problem matrix by matrix). Each block stores its tile's sum of U^2 and counts itself in the
// matrix's counter; the block that completes the count sums the matrix's tile sums in index order (the
// same order whichever block finishes last) and writes s = 1 / (sqrt(sum) + eps).
template <bool MOMENTUM>
// at most 32 registers (8 blocks of 256 threads per SM): the pass needs every block it can keep resident to have
// enough loads in flight, and the two tile shapes of a transposed store would otherwise cost 48
__global__ void __launch_bounds__(256, 8) nesterov_norm_kernel(const __grid_constant__ NesterovGroup G) {
  pdl_wait();
  if (threadIdx.x == 0) pdl_launch_dependents();
  // the transposing tiles' buffer: 64 columns of up to NESTEROV_TALL_ROWS rows (+8 of padding)
  __shared__ __align__(16) __nv_bfloat16 tile_buf[NESTEROV_TILE * (NESTEROV_TALL_ROWS + 8)];
  __shared__ float red[8];
  __shared__ int last;
  int pi = 0;
  while (pi + 1 < G.nprob && static_cast<long long>(blockIdx.x) >= G.block_begin[pi + 1]) ++pi;
  const NesterovArgs &a = G.prob[pi];
  const long long tiles = static_cast<long long>(a.tiles_r) * a.tiles_c;
  const long long local = static_cast<long long>(blockIdx.x) - G.block_begin[pi];
  const long long b = local / tiles;
  const long long t = local - b * tiles;
  const int tr = static_cast<int>(t / a.tiles_c);
  const int tc = static_cast<int>(t - static_cast<long long>(tr) * a.tiles_c);
  float ss;
  if (a.wide_tiles && !a.transposed) {
    ss = a.gdtype == MUON_F32 ? nesterov_tile_wide<float, MOMENTUM>(a, b, tr, tc)
                              : nesterov_tile_wide<__nv_bfloat16, MOMENTUM>(a, b, tr, tc);
  } else if (a.wide_tiles) {   // stored tall: 128-row tiles, so that each row of U gets 256 bytes at a time
    auto tile = reinterpret_cast<__nv_bfloat16 (*)[NESTEROV_TALL_ROWS + 8]>(tile_buf);
    ss = a.gdtype == MUON_F32 ? nesterov_tile<float, MOMENTUM, NESTEROV_TALL_ROWS>(a, b, tr, tc, tile)
                              : nesterov_tile<__nv_bfloat16, MOMENTUM, NESTEROV_TALL_ROWS>(a, b, tr, tc, tile);
  } else {
    auto tile = reinterpret_cast<__nv_bfloat16 (*)[NESTEROV_TILE + 8]>(tile_buf);
    ss = a.gdtype == MUON_F32 ? nesterov_tile<float, MOMENTUM, NESTEROV_TILE>(a, b, tr, tc, tile)
                              : nesterov_tile<__nv_bfloat16, MOMENTUM, NESTEROV_TILE>(a, b, tr, tc, tile);
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float *partials = a.partials + b * tiles;
  if (threadIdx.x == 0) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) sum += red[w];
    partials[t] = sum;
    __threadfence();
    last = atomicAdd(a.counters + b, 1u) == static_cast<unsigned>(tiles - 1);
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  float s = 0.f;
  for (long long i = threadIdx.x; i < tiles; i += 256) s += __ldcg(partials + i);
  s = warp_sum(s);
  __syncthreads();   // red is reused
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) sum += red[w];
    a.scale[b] = 1.0f / (sqrtf(sum) + a.eps);
    // one count past the tiles: matrix b's input to the chain (its tiles' U and this scale) is complete
    red_release_gpu_add(a.counters + b, 1u);
  }
}

// Zeroes n counters. It lets its successor launch at once, but finishes only after its predecessor
// has: a successor that waits for this grid so also waits for everything before it.
__global__ void __launch_bounds__(256) counter_reset_kernel(unsigned *counters, long long n, unsigned *counters2,
                                                             long long n2) {
  if (threadIdx.x == 0) pdl_launch_dependents();
  pdl_wait();
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n + n2;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    if (i < n) counters[i] = 0u;
    else counters2[i - n] = 0u;
  }
}

// ------------------------------------------------------------------------------------------ AdamW

// Every rounding step is spelled out (explicit fmaf and round-to-nearest multiplies and divide), so the
// compiler has no contraction left to choose and every kernel that calls this gives the same bits.
__device__ __forceinline__ float adamw_elem(float &pf, float gf, float &mf, float &vf, const AdamwConst &c) {
  if (c.l2) gf = fmaf(c.l2_wd, pf, gf);
  pf = __fmul_rn(pf, c.decay);
  mf = fmaf(c.beta1, mf, __fmul_rn(c.one_minus_beta1, gf));
  vf = fmaf(c.beta2, vf, __fmul_rn(__fmul_rn(c.one_minus_beta2, gf), gf));
  const float denom = fmaf(sqrtf(vf), c.inv_sqrt_bc2, c.eps);
  pf = fmaf(-c.step_size, __fdiv_rn(mf, denom), pf);
  return pf;
}

template <typename T>
__device__ __forceinline__ void load8(const T *p, float *f);
template <>
__device__ __forceinline__ void load8<float>(const float *p, float *f) {
  const float4 a = reinterpret_cast<const float4 *>(p)[0];
  const float4 b = reinterpret_cast<const float4 *>(p)[1];
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16 *p, float *f) {
  const uint4 w = reinterpret_cast<const uint4 *>(p)[0];
  const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&w);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 x = __bfloat1622float2(h[e]);
    f[2 * e] = x.x;
    f[2 * e + 1] = x.y;
  }
}
template <typename T>
__device__ __forceinline__ void store8(T *p, const float *f);
template <>
__device__ __forceinline__ void store8<float>(float *p, const float *f) {
  reinterpret_cast<float4 *>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
  reinterpret_cast<float4 *>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
}
template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16 *p, const float *f) {
  uint4 w;
  __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&w);
#pragma unroll
  for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(f[2 * e], f[2 * e + 1]);
  reinterpret_cast<uint4 *>(p)[0] = w;
}

template <typename T>
__device__ __forceinline__ float load1(const T *p, long long i);
template <>
__device__ __forceinline__ float load1<float>(const float *p, long long i) { return p[i]; }
template <>
__device__ __forceinline__ float load1<__nv_bfloat16>(const __nv_bfloat16 *p, long long i) {
  return __bfloat162float(p[i]);
}
__device__ __forceinline__ void store1(float *p, long long i, float v) { p[i] = v; }
__device__ __forceinline__ void store1(__nv_bfloat16 *p, long long i, float v) { p[i] = __float2bfloat16_rn(v); }

// Groups of 8 elements from `first`, then the scalar tail; vec=false runs everything scalar.
template <typename PT, typename GT>
__global__ void __launch_bounds__(256) adamw_kernel(PT *__restrict__ p, const GT *__restrict__ g,
                                                    float *__restrict__ m, float *__restrict__ v, long long n,
                                                    int vec, AdamwConst c) {
  pdl_wait();
  if (threadIdx.x == 0) pdl_launch_dependents();
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  long long done = 0;
  if (vec) {
    const long long groups = n / 8;
    for (long long i = tid; i < groups; i += stride) {
      const long long o = i * 8;
      float pf[8], gf[8], mf[8], vf[8];
      load8(p + o, pf);
      load8(g + o, gf);
      load8(m + o, mf);
      load8(v + o, vf);
#pragma unroll
      for (int e = 0; e < 8; ++e) adamw_elem(pf[e], gf[e], mf[e], vf[e], c);
      store8(p + o, pf);
      store8(m + o, mf);
      store8(v + o, vf);
    }
    done = groups * 8;
  }
  for (long long i = done + tid; i < n; i += stride) {
    float pf = load1(p, i), mf = m[i], vf = v[i];
    adamw_elem(pf, load1(g, i), mf, vf, c);
    store1(p, i, pf);
    m[i] = mf;
    v[i] = vf;
  }
}

__global__ void debug_wait_kernel(uint32_t *err, unsigned long long timeout_ns) {
  pdl_wait();
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    WaitCtl ctl{&abort_flag, err, timeout_ns};
    wait_bounded(&bar, 0u, ctl, ERR_WAIT_DEBUG);
  }
}

// Launch with programmatic stream serialization (the kernel waits for its predecessor itself).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace

muon_status launch_counter_reset(unsigned *counters, long long n, cudaStream_t s, unsigned *counters2, long long n2) {
  if (counters2 == nullptr || n2 < 0) n2 = 0;
  if (n < 0) n = 0;
  if (n + n2 < 1) return MUON_OK;
  const long long blocks = std::min<long long>((n + n2 + 255) / 256, device_sm_count());
  launch_begin(KK_COUNTER_RESET, s);
  const cudaError_t e = launch_pdl(counter_reset_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                                   counters, n, counters2, n2);
  launch_end(s);
  return e == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
}

muon_status launch_nesterov_norm(const NesterovArgs *probs, int n, cudaStream_t s) {
  if (n < 1) return MUON_OK;
  const bool mom = probs[0].momentum != nullptr;
  NesterovGroup G{};
  long long blocks = 0;
  auto flush = [&]() -> muon_status {
    if (G.nprob == 0) return MUON_OK;
    launch_begin(KK_NESTEROV_NORM, s);
    const dim3 grid(static_cast<unsigned>(blocks));
    const cudaError_t e = mom ? launch_pdl(nesterov_norm_kernel<true>, grid, dim3(256), 0, s, G)
                              : launch_pdl(nesterov_norm_kernel<false>, grid, dim3(256), 0, s, G);
    launch_end(s);
    G.nprob = 0;
    blocks = 0;
    return e == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
  };
  constexpr long long MAX_GRID = (1ll << 31) - 1;
  for (int i = 0; i < n; ++i) {
    if ((probs[i].momentum != nullptr) != mom) return MUON_ERR_INVALID_ARG;
    const long long tiles = static_cast<long long>(probs[i].tiles_r) * probs[i].tiles_c;
    long long done = 0;   // matrices of stack i already placed in a launch
    while (done < probs[i].K) {
      if (G.nprob == NESTEROV_MAX_PROBLEMS || blocks + tiles > MAX_GRID) {
        const muon_status st = flush();
        if (st != MUON_OK) return st;
      }
      const long long fit = std::min<long long>(probs[i].K - done, (MAX_GRID - blocks) / tiles);
      NesterovArgs p = probs[i];
      // the launch sees matrices done .. done+fit-1 of the stack as its matrices 0 .. fit-1
      if (p.gptrs != nullptr) p.gptrs += done;
      else p.gbase = static_cast<const char *>(p.gbase) + done * static_cast<long long>(p.A) * p.B *
                                                              (p.gdtype == MUON_F32 ? 4 : 2);
      if (p.momentum != nullptr) p.momentum += done * static_cast<long long>(p.A) * p.B;
      p.u += done * p.mstride_u;
      p.partials += done * tiles;
      p.scale += done;
      p.counters += done;
      p.K = static_cast<int>(fit);
      G.block_begin[G.nprob] = blocks;
      G.prob[G.nprob++] = p;
      blocks += fit * tiles;
      done += fit;
    }
  }
  return flush();
}

// AdamW on fp32 master weights: the update reads and writes the master, and p receives it rounded to bf16.
template <typename GT>
__global__ void __launch_bounds__(256) adamw_master_kernel(float *__restrict__ master, __nv_bfloat16 *__restrict__ p,
                                                           const GT *__restrict__ g, float *__restrict__ m,
                                                           float *__restrict__ v, long long n, int vec,
                                                           AdamwConst c) {
  pdl_wait();
  if (threadIdx.x == 0) pdl_launch_dependents();
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  long long done = 0;
  if (vec) {
    const long long groups = n / 8;
    for (long long i = tid; i < groups; i += stride) {
      const long long o = i * 8;
      float pf[8], gf[8], mf[8], vf[8];
      load8(master + o, pf);
      load8(g + o, gf);
      load8(m + o, mf);
      load8(v + o, vf);
#pragma unroll
      for (int e = 0; e < 8; ++e) adamw_elem(pf[e], gf[e], mf[e], vf[e], c);
      store8(master + o, pf);
      store8(p + o, pf);
      store8(m + o, mf);
      store8(v + o, vf);
    }
    done = groups * 8;
  }
  for (long long i = done + tid; i < n; i += stride) {
    float pf = master[i], mf = m[i], vf = v[i];
    adamw_elem(pf, load1(g, i), mf, vf, c);
    master[i] = pf;
    store1(p, i, pf);
    m[i] = mf;
    v[i] = vf;
  }
}

// One warp's share of a grouped pass: elements [e0, e1) of tensor d, 8 per lane per step when the tensor is
// vector-aligned (e0 is a multiple of the chunk size, so the alignment holds), then the scalar rest.
template <typename PT, typename GT, bool MASTER>
__device__ __forceinline__ void adamw_span(const AdamwTensorDesc &d, long long e0, long long e1, int lane) {
  PT *p = static_cast<PT *>(d.p);
  const GT *g = static_cast<const GT *>(d.g);
  float *m = d.m, *v = d.v, *ms = d.master;
  long long e = e0;
  if (d.vec) {
    const long long ev = e0 + ((e1 - e0) & ~7LL);
#pragma unroll 1
    for (long long o = e0 + 8 * lane; o < ev; o += 256) {
      float pf[8], gf[8], mf[8], vf[8];
      if constexpr (MASTER) load8(ms + o, pf);
      else load8(p + o, pf);
      load8(g + o, gf);
      load8(m + o, mf);
      load8(v + o, vf);
#pragma unroll
      for (int k = 0; k < 8; ++k) adamw_elem(pf[k], gf[k], mf[k], vf[k], d.c);
      if constexpr (MASTER) store8(ms + o, pf);
      store8(p + o, pf);
      store8(m + o, mf);
      store8(v + o, vf);
    }
    e = ev;
  }
  for (long long i = e + lane; i < e1; i += 32) {
    float pf = MASTER ? ms[i] : load1(p, i), mf = m[i], vf = v[i];
    adamw_elem(pf, load1(g, i), mf, vf, d.c);
    if constexpr (MASTER) ms[i] = pf;
    store1(p, i, pf);
    m[i] = mf;
    v[i] = vf;
  }
}

// Grouped AdamW: warps take chunks from the pass's counter until none is left (see AdamwGroup). The
// arithmetic per element is adamw_elem, as in adamw_kernel, so both give the same bits.
__global__ void __launch_bounds__(ADAMW_THREADS, 10) adamw_grouped_kernel(const __grid_constant__ AdamwGroup G) {
  pdl_wait();
  if (threadIdx.x == 0) pdl_launch_dependents();
  const int lane = threadIdx.x % 32;
  for (;;) {
    unsigned long long chunk = 0;
    if (lane == 0) chunk = atomicAdd(G.next, 1ull);
    chunk = __shfl_sync(0xffffffffu, chunk, 0);
    if (chunk >= static_cast<unsigned long long>(G.total_chunks)) break;
    const long long ch = static_cast<long long>(chunk);
    int lo = 0, hi = G.ntensors - 1;   // the last tensor whose first chunk is <= ch
    while (lo < hi) {
      const int mid = (lo + hi + 1) / 2;
      if (G.t[mid].chunk_begin <= ch) lo = mid;
      else hi = mid - 1;
    }
    const AdamwTensorDesc &d = G.t[lo];
    const long long e0 = (ch - d.chunk_begin) * G.chunk;
    const long long e1 = min(e0 + G.chunk, d.n);
    if (d.master != nullptr) {
      if (d.gdt == MUON_F32) adamw_span<__nv_bfloat16, float, true>(d, e0, e1, lane);
      else adamw_span<__nv_bfloat16, __nv_bfloat16, true>(d, e0, e1, lane);
    } else if (d.pdt == MUON_F32) {
      if (d.gdt == MUON_F32) adamw_span<float, float, false>(d, e0, e1, lane);
      else adamw_span<float, __nv_bfloat16, false>(d, e0, e1, lane);
    } else {
      if (d.gdt == MUON_F32) adamw_span<__nv_bfloat16, float, false>(d, e0, e1, lane);
      else adamw_span<__nv_bfloat16, __nv_bfloat16, false>(d, e0, e1, lane);
    }
  }
}

long long adamw_blocks(long long work) {
  const long long sms = device_sm_count();
  long long blocks = (work + 255) / 256;
  const long long cap = sms * 8;  // 8 resident 256-thread blocks per SM, grid-stride beyond that
  if (blocks > cap) blocks = cap;
  return blocks < 1 ? 1 : blocks;
}

muon_status launch_adamw_grouped(const AdamwGroup &G, cudaStream_t s) {
  if (G.ntensors < 1 || G.total_chunks < 1) return MUON_OK;
  const long long sms = device_sm_count();
  const long long warps = ADAMW_THREADS / 32;
  const long long need = (G.total_chunks + warps - 1) / warps;   // blocks that can all find a chunk
  const long long blocks = std::max(1LL, std::min(need, sms * 10));
  launch_begin(KK_ADAMW, s);
  const dim3 grid(static_cast<unsigned>(blocks)), block(ADAMW_THREADS);
  const cudaError_t e = launch_pdl(adamw_grouped_kernel, grid, block, 0, s, G);
  launch_end(s);
  return e == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
}

muon_status launch_adamw_master(float *master, __nv_bfloat16 *p, const void *g, int gdt, float *m, float *v,
                                long long n, const AdamwConst &c, cudaStream_t s) {
  auto aligned = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
  const int vec = aligned(master) && aligned(p) && aligned(g) && aligned(m) && aligned(v);
  const dim3 gb(static_cast<unsigned>(adamw_blocks(vec ? (n / 8 + (n % 8)) : n))), tb(256);
  launch_begin(KK_ADAMW, s);
  const cudaError_t e =
      gdt == MUON_F32
          ? launch_pdl(adamw_master_kernel<float>, gb, tb, 0, s, master, p, static_cast<const float *>(g), m, v, n,
                       vec, c)
          : launch_pdl(adamw_master_kernel<__nv_bfloat16>, gb, tb, 0, s, master, p,
                       static_cast<const __nv_bfloat16 *>(g), m, v, n, vec, c);
  launch_end(s);
  return e == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
}

muon_status launch_adamw(void *p, int pdt, const void *g, int gdt, float *m, float *v, long long n,
                         const AdamwConst &c, cudaStream_t s) {
  auto aligned = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
  const int vec = aligned(p) && aligned(g) && aligned(m) && aligned(v) &&
                  (pdt == MUON_F32 || (reinterpret_cast<uintptr_t>(p) & 15) == 0);
  const long long work = vec ? (n / 8 + (n % 8)) : n;
  const long long sms = device_sm_count();
  long long blocks = (work + 255) / 256;
  const long long cap = sms * 8;  // 8 resident 256-thread blocks per SM, grid-stride beyond that
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  launch_begin(KK_ADAMW, s);
  const dim3 gb(static_cast<unsigned>(blocks)), tb(256);
  cudaError_t e;
  if (pdt == MUON_F32 && gdt == MUON_F32)
    e = launch_pdl(adamw_kernel<float, float>, gb, tb, 0, s, static_cast<float *>(p), static_cast<const float *>(g),
                   m, v, n, vec, c);
  else if (pdt == MUON_F32 && gdt == MUON_BF16)
    e = launch_pdl(adamw_kernel<float, __nv_bfloat16>, gb, tb, 0, s, static_cast<float *>(p),
                   static_cast<const __nv_bfloat16 *>(g), m, v, n, vec, c);
  else if (pdt == MUON_BF16 && gdt == MUON_F32)
    e = launch_pdl(adamw_kernel<__nv_bfloat16, float>, gb, tb, 0, s, static_cast<__nv_bfloat16 *>(p),
                   static_cast<const float *>(g), m, v, n, vec, c);
  else
    e = launch_pdl(adamw_kernel<__nv_bfloat16, __nv_bfloat16>, gb, tb, 0, s, static_cast<__nv_bfloat16 *>(p),
                   static_cast<const __nv_bfloat16 *>(g), m, v, n, vec, c);
  launch_end(s);
  return e == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
}

muon_status launch_debug_wait(uint32_t *err, unsigned long long timeout_ns, cudaStream_t s) {
  launch_begin(KK_DEBUG_WAIT, s);
  const cudaError_t e = launch_pdl(debug_wait_kernel, dim3(1), dim3(32), 0, s, err, timeout_ns);
  launch_end(s);
  return e == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
}

}  // namespace muon
