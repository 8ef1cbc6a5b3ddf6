// Tensor-core GEMMs of the Newton-Schulz iteration, one persistent grouped kernel per step kind.
//
// One Newton-Schulz step ("Optimizers: AdamW, Muon and the distributed optimizer", section
// "Muon: orthogonalising the update") on a wide iterate X (m x n, m <= n):
//     G = X X^T                     EPI_GRAM   symmetric: only tiles touching the upper triangle
//                                              are computed, every value is also stored mirrored
//                                              ("DMuon", section 2.2, symmetric Gram)
//     H = b G + c G G               EPI_POLY   G symmetric, so G G = G G^T: same operand pattern
//     X' = a X + H X                EPI_APPLY  B operand (X) is read N-major
//     last step: u = a X + H X, then p <- p - lr*wd*p*mask - lr*scale*u      EPI_FINAL
//
// Design (sm_103a): 128 x 256 output tiles, 64-deep k-slices, 4-stage TMA ring with 128-byte
// swizzle, one tcgen05.mma (M=128, N=256, K=16, bf16 -> fp32) per 16-slice issued by one thread,
// fp32 accumulators in tensor memory (2 x 256 columns, so the epilogue of one tile overlaps the
// MMAs of the next), persistent CTAs (one per SM) striding over (matrix, tile) of the whole stack.
// Warp roles: warp 0 = TMA producer, warp 1 = MMA issuer (and TMEM owner), warps 2-5 = epilogue.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace muon {

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int ACC_COLS = BN;
constexpr uint32_t TMEM_COLS = 512;
constexpr int NUM_THREADS = 192;

struct Ctrl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t SMEM_BYTES = static_cast<size_t>(STAGES) * STAGE_BYTES + sizeof(Ctrl) + 1024;

__device__ __forceinline__ void decode_tile(const GemmArgs &a, long long t, int &b, int &ti, int &tj) {
  b = static_cast<int>(t / a.tiles_per_matrix);
  int r = static_cast<int>(t - static_cast<long long>(b) * a.tiles_per_matrix);
  if (!a.symmetric) {
    tj = r / a.m_tiles;
    ti = r - tj * a.m_tiles;
    return;
  }
  // column-major over the tiles with 256*j + 255 >= 128*i, i.e. i < 2j + 2
  int j = 0;
  for (;;) {
    const int cnt = min(a.m_tiles, 2 * j + 2);
    if (r < cnt) {
      ti = r;
      tj = j;
      return;
    }
    r -= cnt;
    ++j;
  }
}

__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ void load_bf16x32(const __nv_bfloat16 *src, float *dst) {
  const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w = s4[q];
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float2 f = __bfloat1622float2(h[e]);
      dst[q * 8 + 2 * e] = f.x;
      dst[q * 8 + 2 * e + 1] = f.y;
    }
  }
}

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16 *dst, const float *src) {
  uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&w);
#pragma unroll
    for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(src[q * 8 + 2 * e], src[q * 8 + 2 * e + 1]);
    d4[q] = w;
  }
}

// Epilogue for one 32-column chunk held by one thread (its row `row`, columns col0..col0+31).
template <int EPI>
__device__ __forceinline__ void epilogue_chunk(const GemmArgs &a, int b, int row, int col0, float *v) {
  if constexpr (EPI == EPI_GRAM || EPI == EPI_POLY) {
    float sc = a.alpha;
    if (EPI == EPI_GRAM && a.scale != nullptr) {
      const float s = a.scale[b];
      sc *= s * s;
    }
    const bool row_ok = row < a.rows;
    const bool full = row_ok && (col0 >= row) && (col0 + 32 <= a.cols);
    __nv_bfloat16 *out_b = a.out + static_cast<long long>(b) * a.mstride_out;
    if constexpr (EPI == EPI_POLY) {
      const __nv_bfloat16 *g_row = a.aux + static_cast<long long>(b) * a.mstride_aux + static_cast<long long>(row) * a.ld_aux;
      if (full) {
        float gv[32];
        load_bf16x32(g_row + col0, gv);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = a.coef_b * gv[j] + a.coef_c * v[j];
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int c = col0 + j;
          const float gv = (row_ok && c < a.cols && c >= row) ? bf2f(g_row[c]) : 0.f;
          v[j] = a.coef_b * gv + a.coef_c * v[j];
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] *= sc;
    }
    // direct store of the upper-triangle part of this row
    if (full) {
      store_bf16x32(out_b + static_cast<long long>(row) * a.ld_out + col0, v);
    } else if (row_ok) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int c = col0 + j;
        if (c < a.cols && c >= row) out_b[static_cast<long long>(row) * a.ld_out + c] = __float2bfloat16_rn(v[j]);
      }
    }
    // mirrored store of the strictly-upper part: lanes hold consecutive rows, so each column's
    // 32 values land in one contiguous 64-byte segment of the mirrored row
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int c = col0 + j;
      if (row_ok && c < a.cols && c > row) out_b[static_cast<long long>(c) * a.ld_out + row] = __float2bfloat16_rn(v[j]);
    }
  } else {
    float sc = 1.f;
    if (a.scale != nullptr) sc = a.scale[b];
    if (row >= a.rows) return;
    const __nv_bfloat16 *x_row = a.aux + static_cast<long long>(b) * a.mstride_aux + static_cast<long long>(row) * a.ld_aux;
    const bool full = (col0 + 32 <= a.cols);
    float xv[32];
    if (full) {
      load_bf16x32(x_row + col0, xv);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) xv[j] = (col0 + j < a.cols) ? bf2f(x_row[col0 + j]) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = sc * (a.coef_a * xv[j] + v[j]);
    if constexpr (EPI == EPI_APPLY) {
      __nv_bfloat16 *o_row = a.out + static_cast<long long>(b) * a.mstride_out + static_cast<long long>(row) * a.ld_out;
      if (full) {
        store_bf16x32(o_row + col0, v);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (col0 + j < a.cols) o_row[col0 + j] = __float2bfloat16_rn(v[j]);
      }
    } else {
      // wide (row, c) is stored element (c, row) when transposed, else (row, c)
      const long long mat_elems = static_cast<long long>(a.rows) * a.cols;
      void *base = a.params != nullptr ? a.params[b]
                                       : static_cast<void *>(static_cast<char *>(a.out_dense) +
                                                             static_cast<long long>(b) * mat_elems *
                                                                 (a.out_dtype == MUON_F32 ? 4 : 2));
      const bool update = a.params != nullptr;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int c = col0 + j;
        if (c >= a.cols) continue;
        const long long idx = a.transposed ? static_cast<long long>(c) * a.orig_cols + row
                                           : static_cast<long long>(row) * a.orig_cols + c;
        const float u = v[j];
        if (a.out_dtype == MUON_F32) {
          float *p = static_cast<float *>(base) + idx;
          if (update) {
            const float pv = *p;
            const float mask = (!a.cautious || u * pv > 0.f) ? 1.f : 0.f;
            *p = (pv - a.lr_wd * mask * pv) - a.lr_scale * u;
          } else {
            *p = u;
          }
        } else {
          __nv_bfloat16 *p = static_cast<__nv_bfloat16 *>(base) + idx;
          if (update) {
            const float pv = bf2f(*p);
            const float mask = (!a.cautious || u * pv > 0.f) ? 1.f : 0.f;
            *p = __float2bfloat16_rn((pv - a.lr_wd * mask * pv) - a.lr_scale * u);
          } else {
            *p = __float2bfloat16_rn(u);
          }
        }
      }
    }
  }
}

template <int EPI, bool B_MN>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    ns_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                   const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctrl *ctrl = reinterpret_cast<Ctrl *>(smem + STAGES * STAGE_BYTES);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctrl->full[s], 1);
      mbar_init(&ctrl->empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ctrl->acc_full[s], 1);
      mbar_init(&ctrl->acc_empty[s], 4);
    }
    mbar_init(&ctrl->drain, 1);
    ctrl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_a);
    tma_prefetch_desc(&map_b);
  }
  if (warp == 1) {
    tmem_alloc(&ctrl->tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctrl->tmem_base;
  WaitCtl ctl{&ctrl->abort_flag, args.err, args.timeout_ns};
  WaitCtl drain_ctl{&ctrl->abort_flag, args.err, args.timeout_ns};

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      uint32_t stage = 0, phase = 0;
      int last_parity[STAGES];
      for (int s = 0; s < STAGES; ++s) last_parity[s] = -1;
      bool ok = true;
      for (long long t = blockIdx.x; ok && t < args.total_tiles; t += gridDim.x) {
        int b, ti, tj;
        decode_tile(args, t, b, ti, tj);
        for (int kk = 0; kk < args.k_iters; ++kk) {
          if (!wait_bounded(&ctrl->empty[stage], phase ^ 1u, ctl, ERR_WAIT_EMPTY)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&ctrl->full[stage], STAGE_BYTES);
          last_parity[stage] = static_cast<int>(phase);
          uint8_t *sa = smem + stage * STAGE_BYTES;
          uint8_t *sb = sa + A_BYTES;
          tma_load_3d(sa, &map_a, &ctrl->full[stage], kk * BK, ti * BM, b);
          if constexpr (!B_MN) {
            tma_load_3d(sb, &map_b, &ctrl->full[stage], kk * BK, tj * BN, b);
          } else {
#pragma unroll
            for (int c = 0; c < BN / 64; ++c)
              tma_load_3d(sb + c * (64 * BK * 2), &map_b, &ctrl->full[stage], tj * BN + 64 * c, kk * BK, b);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // every armed stage's copies have landed before the CTA may exit
      for (int s = 0; s < STAGES; ++s) {
        if (last_parity[s] < 0) continue;
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&ctrl->full[s], static_cast<uint32_t>(last_parity[s]))) {
          if (globaltimer_ns() - t0 > drain_ctl.timeout_ns) {
            if (args.err) atomicCAS(args.err, 0u, ERR_WAIT_DRAIN);
            break;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, false, B_MN);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      bool issued = false;
      for (long long t = blockIdx.x; ok && t < args.total_tiles; t += gridDim.x) {
        if (!wait_bounded(&ctrl->acc_empty[acc], acc_phase ^ 1u, ctl, ERR_WAIT_ACC_EMPTY)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
        for (int kk = 0; kk < args.k_iters; ++kk) {
          if (!wait_bounded(&ctrl->full[stage], phase, ctl, ERR_WAIT_FULL)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t adesc = smem_desc_sw128(sa + k * 32, 16, 1024);
            const uint64_t bdesc =
                B_MN ? smem_desc_sw128(sb + k * 16 * 128, 64 * BK * 2, 1024) : smem_desc_sw128(sb + k * 32, 16, 1024);
            tc_mma_bf16(d_tmem, adesc, bdesc, idesc, (kk | k) != 0 ? 1u : 0u);
          }
          issued = true;
          tc_commit(&ctrl->empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&ctrl->acc_full[acc]);
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      // all MMAs this thread issued have completed before TMEM is released
      if (issued) {
        tc_commit(&ctrl->drain);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&ctrl->drain, 0)) {
          if (globaltimer_ns() - t0 > drain_ctl.timeout_ns) {
            if (args.err) atomicCAS(args.err, 0u, ERR_WAIT_DRAIN);
            break;
          }
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 2..5)
    const int lane_base = (warp % 4) * 32;  // TMEM lanes this warp may read
    uint32_t acc = 0, acc_phase = 0;
    for (long long t = blockIdx.x; t < args.total_tiles; t += gridDim.x) {
      int b, ti, tj;
      decode_tile(args, t, b, ti, tj);
      // every lane waits; the warp proceeds only if all of them saw the accumulator complete, so the
      // warp-collective TMEM loads below never run with part of the warp gone
      const bool ok = wait_bounded(&ctrl->acc_full[acc], acc_phase, ctl, ERR_WAIT_ACC_FULL);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const int row = ti * BM + lane_base + lane;
      const int warp_row0 = ti * BM + lane_base;
#pragma unroll 1
      for (int ch = 0; ch < BN / 32; ++ch) {
        const int col0 = tj * BN + ch * 32;
        if (col0 >= args.cols) break;                                    // warp-uniform
        if (args.symmetric && col0 + 31 < warp_row0) continue;           // chunk below the diagonal for every lane
        if (warp_row0 >= args.rows) break;                               // whole warp past the last row
        float v[32];
        tmem_ld_32x32b_x32(tmem_base + acc * ACC_COLS + (static_cast<uint32_t>(lane_base) << 16) + ch * 32, v);
        epilogue_chunk<EPI>(args, b, row, col0, v);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctrl->acc_empty[acc]);
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------------------------------ host side

// The driver's tensor-map encoder, fetched through the runtime so the library needs no -lcuda.
using EncodeTiledFn = decltype(&cuTensorMapEncodeTiled);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D bf16 map (inner, rows, batch) with a box of (64, box_rows, 1) and 128-byte swizzle.
bool make_map(CUtensorMap *map, const void *base, long long inner, long long rows, long long batch, long long ld,
              long long mstride, int box_rows) {
  auto enc = get_encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(batch)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2, static_cast<cuuint64_t>(mstride) * 2};
  cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_rows), 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int EPI, bool B_MN>
muon_status launch_kernel(const CUtensorMap &ma, const CUtensorMap &mb, const GemmArgs &args, int32_t kind,
                          cudaStream_t s) {
  static std::once_flag attr_once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  std::call_once(attr_once[dev & 63], [] {
    cudaFuncSetAttribute(ns_gemm_kernel<EPI, B_MN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(SMEM_BYTES));
  });
  if (args.total_tiles <= 0) return MUON_OK;
  const long long sms = device_sm_count();
  const int grid = static_cast<int>(args.total_tiles < sms ? args.total_tiles : sms);
  launch_begin(kind, s);
  ns_gemm_kernel<EPI, B_MN><<<grid, NUM_THREADS, SMEM_BYTES, s>>>(ma, mb, args);
  launch_end(s);
  return cudaGetLastError() == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
}

void fill_tiles(GemmArgs &a, int batch, int rows, int cols, int contraction, bool symmetric) {
  a.batch = batch;
  a.rows = rows;
  a.cols = cols;
  a.m_tiles = (rows + BM - 1) / BM;
  a.n_tiles = (cols + BN - 1) / BN;
  a.symmetric = symmetric ? 1 : 0;
  if (symmetric) {
    int cnt = 0;
    for (int j = 0; j < a.n_tiles; ++j) cnt += (a.m_tiles < 2 * j + 2 ? a.m_tiles : 2 * j + 2);
    a.tiles_per_matrix = cnt;
  } else {
    a.tiles_per_matrix = a.m_tiles * a.n_tiles;
  }
  a.total_tiles = static_cast<long long>(a.tiles_per_matrix) * batch;
  a.k_iters = (contraction + BK - 1) / BK;
}

}  // namespace

muon_status launch_gram(const Bf16Stack &x, __nv_bfloat16 *g, long long ldg, long long mstride_g, float alpha,
                        const float *scale, uint32_t *err, unsigned long long timeout_ns, cudaStream_t s) {
  CUtensorMap ma, mb;
  if (!make_map(&ma, x.ptr, x.cols, x.rows, x.batch, x.ld, x.mstride, BM) ||
      !make_map(&mb, x.ptr, x.cols, x.rows, x.batch, x.ld, x.mstride, BN))
    return MUON_ERR_CUDA;
  GemmArgs a{};
  fill_tiles(a, static_cast<int>(x.batch), static_cast<int>(x.rows), static_cast<int>(x.rows),
             static_cast<int>(x.cols), true);
  a.alpha = alpha;
  a.scale = scale;
  a.scale_pow = 2;
  a.out = g;
  a.ld_out = ldg;
  a.mstride_out = mstride_g;
  a.err = err;
  a.timeout_ns = timeout_ns;
  return launch_kernel<EPI_GRAM, false>(ma, mb, a, KK_GRAM, s);
}

muon_status launch_poly(const Bf16Stack &g, __nv_bfloat16 *h, long long ldh, long long mstride_h, float b, float c,
                        uint32_t *err, unsigned long long timeout_ns, cudaStream_t s) {
  CUtensorMap ma, mb;
  if (!make_map(&ma, g.ptr, g.cols, g.rows, g.batch, g.ld, g.mstride, BM) ||
      !make_map(&mb, g.ptr, g.cols, g.rows, g.batch, g.ld, g.mstride, BN))
    return MUON_ERR_CUDA;
  GemmArgs a{};
  fill_tiles(a, static_cast<int>(g.batch), static_cast<int>(g.rows), static_cast<int>(g.rows),
             static_cast<int>(g.cols), true);
  a.alpha = 1.f;
  a.coef_b = b;
  a.coef_c = c;
  a.out = h;
  a.ld_out = ldh;
  a.mstride_out = mstride_h;
  a.aux = static_cast<const __nv_bfloat16 *>(g.ptr);
  a.ld_aux = g.ld;
  a.mstride_aux = g.mstride;
  a.err = err;
  a.timeout_ns = timeout_ns;
  return launch_kernel<EPI_POLY, false>(ma, mb, a, KK_POLY, s);
}

static bool apply_maps(const Bf16Stack &h, const Bf16Stack &x, CUtensorMap *ma, CUtensorMap *mb) {
  return make_map(ma, h.ptr, h.cols, h.rows, h.batch, h.ld, h.mstride, BM) &&
         make_map(mb, x.ptr, x.cols, x.rows, x.batch, x.ld, x.mstride, BK);
}

muon_status launch_apply(const Bf16Stack &h, const Bf16Stack &x, __nv_bfloat16 *out, float a_coef,
                         const float *scale, uint32_t *err, unsigned long long timeout_ns, cudaStream_t s) {
  CUtensorMap ma, mb;
  if (!apply_maps(h, x, &ma, &mb)) return MUON_ERR_CUDA;
  GemmArgs a{};
  fill_tiles(a, static_cast<int>(x.batch), static_cast<int>(x.rows), static_cast<int>(x.cols),
             static_cast<int>(h.cols), false);
  a.coef_a = a_coef;
  a.scale = scale;
  a.scale_pow = 1;
  a.out = out;
  a.ld_out = x.ld;
  a.mstride_out = x.mstride;
  a.aux = static_cast<const __nv_bfloat16 *>(x.ptr);
  a.ld_aux = x.ld;
  a.mstride_aux = x.mstride;
  a.err = err;
  a.timeout_ns = timeout_ns;
  return launch_kernel<EPI_APPLY, true>(ma, mb, a, KK_APPLY, s);
}

muon_status launch_final(const Bf16Stack &h, const Bf16Stack &x, float a_coef, const float *scale, const FinalSpec &f,
                         uint32_t *err, unsigned long long timeout_ns, cudaStream_t s) {
  CUtensorMap ma, mb;
  if (!apply_maps(h, x, &ma, &mb)) return MUON_ERR_CUDA;
  GemmArgs a{};
  fill_tiles(a, static_cast<int>(x.batch), static_cast<int>(x.rows), static_cast<int>(x.cols),
             static_cast<int>(h.cols), false);
  a.coef_a = a_coef;
  a.scale = scale;
  a.scale_pow = 1;
  a.aux = static_cast<const __nv_bfloat16 *>(x.ptr);
  a.ld_aux = x.ld;
  a.mstride_aux = x.mstride;
  a.params = f.params;
  a.out_dense = f.out_dense;
  a.out_dtype = f.dtype;
  a.transposed = f.transposed;
  a.orig_cols = f.orig_cols;
  a.cautious = f.cautious;
  a.lr_wd = f.lr_wd;
  a.lr_scale = f.lr_scale;
  a.err = err;
  a.timeout_ns = timeout_ns;
  return launch_kernel<EPI_FINAL, true>(ma, mb, a, KK_FINAL, s);
}

}  // namespace muon
