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
// Design (sm_103a): 128 x 256 output tiles, 64-deep k-slices, a TMA ring with 128-byte swizzle
// (4 stages, 3 for the final step), one tcgen05.mma (M=128, N=256, K=16, bf16 -> fp32) per 16-slice
// issued by one thread, fp32 accumulators in tensor memory (2 x 256 columns, so the epilogue of one
// tile overlaps the MMAs of the next), persistent CTAs (one per SM) striding over the tiles of up to
// GEMM_MAX_PROBLEMS stacks at once. CTAs run as clusters of two that compute vertically adjacent tiles
// (rows 2p and 2p+1 of one tile column): both need the same B operand, so each CTA loads one half of it
// and multicasts it to both, which cuts the operand traffic per SM by a third. Warp roles: warp 0 = TMA producer, warp 1 = MMA issuer (and TMEM
// owner), warps 2-9 = epilogue (two per tensor-memory lane quarter, each taking one 32-column half of
// every 64-column slot), warp 10 = epilogue loader: ahead of the epilogue it brings each tile's
// second input (G or X) and, for bf16 parameters, the parameters into a 2-slot shared-memory ring, so
// the epilogue never waits for a global-memory round trip.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace muon {

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int MAX_STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int ACC_COLS = BN;
constexpr uint32_t TMEM_COLS = 512;
constexpr int EPI_WARPS = 8;                                // two per TMEM lane quarter
constexpr int LOADER_WARP = 2 + EPI_WARPS;
constexpr int NUM_THREADS = 32 * (LOADER_WARP + 1);

// Epilogue input ring: a slot holds 64 columns (two 32-column chunks) of a tile's 128 rows.
constexpr int RING_SLOTS = 2;
constexpr int RING_AUX_BYTES = BM * 64 * 2;                 // bf16, 128-byte rows, 128B-swizzled (as TMA writes)
constexpr int PARAM_PITCH_WIDE = 64 * 2 + 16;               // stored row-major: [128 rows][64 cols] + pad
constexpr int PARAM_PITCH_TALL = BM * 2 + 16;               // stored transposed: [64 stored rows][128] + pad
constexpr int RING_PARAM_BYTES = BM * PARAM_PITCH_WIDE;     // >= 64 * PARAM_PITCH_TALL
static_assert(RING_PARAM_BYTES >= 64 * PARAM_PITCH_TALL, "param slot too small");

__host__ __device__ constexpr int stages_of(int epi) { return epi == EPI_FINAL ? 3 : 4; }
__host__ __device__ constexpr int ring_slot_bytes(int epi) {
  return epi == EPI_GRAM ? 0 : (epi == EPI_FINAL ? RING_AUX_BYTES + RING_PARAM_BYTES : RING_AUX_BYTES);
}

struct Ctrl {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t ring_full[RING_SLOTS];
  uint64_t ring_empty[RING_SLOTS];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int ring_param_ok[RING_SLOTS];
};

__host__ __device__ constexpr size_t smem_bytes(int epi) {
  return static_cast<size_t>(stages_of(epi)) * STAGE_BYTES + static_cast<size_t>(RING_SLOTS) * ring_slot_bytes(epi) +
         sizeof(Ctrl) + 1024;
}
static_assert(smem_bytes(EPI_APPLY) <= 232448 && smem_bytes(EPI_FINAL) <= 232448, "shared memory over budget");

// Kernel parameter: up to GEMM_MAX_PROBLEMS problems of one step kind, in order of tile_begin.
struct GemmGroup {
  CUtensorMap map_a[GEMM_MAX_PROBLEMS];
  CUtensorMap map_b[GEMM_MAX_PROBLEMS];
  GemmProblem prob[GEMM_MAX_PROBLEMS];
  int nprob;
  int symmetric;
  long long total_tiles;
  uint32_t *err;
  unsigned long long timeout_ns;
};
static_assert(sizeof(GemmGroup) <= 4096, "kernel parameter block too large");

__device__ __forceinline__ int find_problem(const GemmGroup &g, long long t) {
  int p = 0;
#pragma unroll 1
  for (int q = 1; q < g.nprob; ++q)
    if (t >= g.prob[q].tile_begin) p = q;
  return p;
}

// local tile-pair index of one problem -> (matrix, tile row of this CTA, tile column). Pair p covers tile
// rows 2p (cluster rank 0) and 2p+1 (rank 1); a rank-1 tile past the last row computes nothing useful and
// stores nothing.
__device__ __forceinline__ void decode_tile(const GemmProblem &a, int symmetric, long long t, uint32_t rank, int &b,
                                            int &ti, int &tj) {
  b = static_cast<int>(t / a.tiles_per_matrix);
  int r = static_cast<int>(t - static_cast<long long>(b) * a.tiles_per_matrix);
  if (!symmetric) {
    tj = r / a.m_pairs;
    ti = 2 * (r - tj * a.m_pairs) + static_cast<int>(rank);
    return;
  }
  // column-major over the pairs touching the upper triangle: tile (i, j) is needed iff 128 i <= 256 j + 255,
  // i.e. i < 2j + 2, so pair p is needed iff p <= j
  int j = 0;
  for (;;) {
    const int cnt = min(a.m_pairs, j + 1);
    if (r < cnt) {
      ti = 2 * r + static_cast<int>(rank);
      tj = j;
      return;
    }
    r -= cnt;
    ++j;
  }
}

// A ring slot pair of chunks is used unless the whole tile lies below the diagonal for those 64 columns.
__device__ __forceinline__ bool slot_used(int symmetric, int c0, int row0) { return !(symmetric && c0 + 63 < row0); }

__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ void unpack8(const uint4 &w, float *dst) {
  const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&w);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __bfloat1622float2(h[e]);
    dst[2 * e] = f.x;
    dst[2 * e + 1] = f.y;
  }
}

__device__ __forceinline__ uint4 pack8(const float *src) {
  uint4 w;
  __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&w);
#pragma unroll
  for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(src[2 * e], src[2 * e + 1]);
  return w;
}

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16 *dst, const float *src) {
  uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) d4[q] = pack8(src + 8 * q);
}

// 32 bf16 values of tile row r, columns 32*half .. 32*half+31 of a ring slot (128-byte rows, 128B swizzle:
// the 16-byte chunk q of row r sits at chunk position q ^ (r & 7)).
__device__ __forceinline__ void ring_aux_row(const uint8_t *slot, int r, int half, float *dst) {
  const uint8_t *row = slot + r * 128;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int qq = (4 * half + q) ^ (r & 7);
    unpack8(*reinterpret_cast<const uint4 *>(row + qq * 16), dst + 8 * q);
  }
}

// Muon parameter update of one element: decoupled decay (masked where u*p <= 0 if cautious), then the
// scaled orthogonalised step.
__device__ __forceinline__ float param_update(float pv, float u, const GemmProblem &a) {
  const float mask = (!a.cautious || u * pv > 0.f) ? 1.f : 0.f;
  return (pv - a.lr_wd * mask * pv) - a.lr_scale * u;
}

// Final step for one thread's 32 values of wide row `row`, columns col0..col0+31.
//   stored wide (row-major A x B): the thread's row segment; parameters from the ring (param_slot, laid out
//   [128 rows][64 cols] with pitch PARAM_PITCH_WIDE) when the loader staged them, else loaded directly.
//   stored tall (transposed): element (c, row); for each column the warp's lanes cover 32 consecutive stored
//   elements; ring layout [64 stored rows][128] with pitch PARAM_PITCH_TALL.
__device__ __forceinline__ void final_store(const GemmProblem &a, void *base, int row, int rloc, int col0, int half,
                                            const uint8_t *param_slot, bool staged, float *v) {
  const bool update = a.params != nullptr;
  const bool f32 = a.out_dtype == MUON_F32;
  if (!a.transposed) {
    const long long idx = static_cast<long long>(row) * a.orig_cols + col0;
    float pv[32];
    if (update) {
      if (staged) {
        const uint8_t *src = param_slot + rloc * PARAM_PITCH_WIDE + half * 64;
#pragma unroll
        for (int q = 0; q < 4; ++q) unpack8(*reinterpret_cast<const uint4 *>(src + 16 * q), pv + 8 * q);
      } else if (f32) {
        const float *p = static_cast<const float *>(base) + idx;
#pragma unroll
        for (int j = 0; j < 32; ++j) pv[j] = (col0 + j < a.cols) ? p[j] : 0.f;
      } else {
        const __nv_bfloat16 *p = static_cast<const __nv_bfloat16 *>(base) + idx;
        const bool vec = col0 + 32 <= a.cols && (reinterpret_cast<uintptr_t>(p) & 15) == 0;
        if (vec) {
#pragma unroll
          for (int q = 0; q < 4; ++q) unpack8(reinterpret_cast<const uint4 *>(p)[q], pv + 8 * q);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) pv[j] = (col0 + j < a.cols) ? bf2f(p[j]) : 0.f;
        }
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = param_update(pv[j], v[j], a);
    }
    if (f32) {
      float *p = static_cast<float *>(base) + idx;
      const bool vec = col0 + 32 <= a.cols && (reinterpret_cast<uintptr_t>(p) & 15) == 0;
      if (vec) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          reinterpret_cast<float4 *>(p)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (col0 + j < a.cols) p[j] = v[j];
      }
    } else {
      __nv_bfloat16 *p = static_cast<__nv_bfloat16 *>(base) + idx;
      const bool vec = col0 + 32 <= a.cols && (reinterpret_cast<uintptr_t>(p) & 15) == 0;
      if (vec) {
        store_bf16x32(p, v);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (col0 + j < a.cols) p[j] = __float2bfloat16_rn(v[j]);
      }
    }
    return;
  }
  // transposed: all loads are issued before the first store
  if (update) {
    float pv[32];
    if (staged) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        pv[j] = bf2f(*reinterpret_cast<const __nv_bfloat16 *>(param_slot + (32 * half + j) * PARAM_PITCH_TALL +
                                                              2 * rloc));
    } else if (f32) {
      const float *p = static_cast<const float *>(base) + row;
#pragma unroll
      for (int j = 0; j < 32; ++j) pv[j] = (col0 + j < a.cols) ? p[static_cast<long long>(col0 + j) * a.orig_cols] : 0.f;
    } else {
      const __nv_bfloat16 *p = static_cast<const __nv_bfloat16 *>(base) + row;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        pv[j] = (col0 + j < a.cols) ? bf2f(p[static_cast<long long>(col0 + j) * a.orig_cols]) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = param_update(pv[j], v[j], a);
  }
  if (f32) {
    float *p = static_cast<float *>(base) + row;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (col0 + j < a.cols) p[static_cast<long long>(col0 + j) * a.orig_cols] = v[j];
  } else {
    __nv_bfloat16 *p = static_cast<__nv_bfloat16 *>(base) + row;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (col0 + j < a.cols) p[static_cast<long long>(col0 + j) * a.orig_cols] = __float2bfloat16_rn(v[j]);
  }
}

// Epilogue for one 32-column chunk held by one thread (its row `row` = tile row `rloc`, columns
// col0..col0+31, i.e. half `half` of the ring slot). Called by every lane of the warp.
template <int EPI>
__device__ __forceinline__ void epilogue_chunk(const GemmProblem &a, int b, int row, int rloc, int col0, int half,
                                               const uint8_t *aux_slot, const uint8_t *param_slot, bool param_staged,
                                               float *v) {
  if constexpr (EPI == EPI_GRAM || EPI == EPI_POLY) {
    const bool row_ok = row < a.rows;
    const bool full = row_ok && (col0 >= row) && (col0 + 32 <= a.cols);
    __nv_bfloat16 *out_b = a.out + static_cast<long long>(b) * a.mstride_out;
    if constexpr (EPI == EPI_POLY) {
      float gv[32];
      ring_aux_row(aux_slot, rloc, half, gv);
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = a.coef_b * gv[j] + a.coef_c * v[j];
    } else {
      float sc = a.alpha;
      if (a.scale != nullptr) {
        const float s = a.scale[b];
        sc *= s * s;
      }
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
    const float sc = a.scale != nullptr ? a.scale[b] : 1.f;
    float xv[32];
    ring_aux_row(aux_slot, rloc, half, xv);
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = sc * (a.coef_a * xv[j] + v[j]);
    if (row >= a.rows) return;
    if constexpr (EPI == EPI_APPLY) {
      __nv_bfloat16 *o_row = a.out + static_cast<long long>(b) * a.mstride_out + static_cast<long long>(row) * a.ld_out;
      if (col0 + 32 <= a.cols) {
        store_bf16x32(o_row + col0, v);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (col0 + j < a.cols) o_row[col0 + j] = __float2bfloat16_rn(v[j]);
      }
    } else {
      const long long mat_elems = static_cast<long long>(a.rows) * a.cols;
      void *base = a.params != nullptr ? a.params[b]
                                       : static_cast<void *>(static_cast<char *>(a.out_dense) +
                                                             static_cast<long long>(b) * mat_elems *
                                                                 (a.out_dtype == MUON_F32 ? 4 : 2));
      final_store(a, base, row, rloc, col0, half, param_slot, param_staged, v);
    }
  }
}

// Epilogue loader's parameter staging for one slot (64 columns of a tile) of the final step: 1-D bulk
// copies of the stored rows, when every copy is a whole, 16-byte-aligned bf16 segment. Returns the
// bytes it will deliver (0: the epilogue loads the parameters itself).
__device__ __forceinline__ uint32_t stage_params_bytes(const GemmProblem &a, int b, int row0, int c0,
                                                       const void *&base) {
  if (a.params == nullptr || a.out_dtype != MUON_BF16) return 0;
  base = a.params[b];
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0 || (a.orig_cols & 7) != 0) return 0;
  if (c0 + 64 > a.cols || row0 + BM > a.rows) return 0;
  return a.transposed ? 64u * BM * 2u : static_cast<uint32_t>(BM) * 64u * 2u;
}

// Issued by all 32 lanes of the loader warp, each taking every 32nd row segment.
__device__ __forceinline__ void stage_params_issue(const GemmProblem &a, const void *base, int row0, int c0,
                                                   uint8_t *dst, uint64_t *bar, int lane) {
  const __nv_bfloat16 *p = static_cast<const __nv_bfloat16 *>(base);
  if (!a.transposed) {
    for (int r = lane; r < BM; r += 32)
      bulk_load(dst + r * PARAM_PITCH_WIDE, p + static_cast<long long>(row0 + r) * a.orig_cols + c0, 128, bar);
  } else {
    for (int j = lane; j < 64; j += 32)
      bulk_load(dst + j * PARAM_PITCH_TALL, p + static_cast<long long>(c0 + j) * a.orig_cols + row0, BM * 2, bar);
  }
}

template <int EPI, bool B_MN>
__global__ void __launch_bounds__(NUM_THREADS, 1) ns_gemm_kernel(const __grid_constant__ GemmGroup args) {
  constexpr int STAGES = stages_of(EPI);
  constexpr int SLOT_BYTES = ring_slot_bytes(EPI);
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *ring = smem + STAGES * STAGE_BYTES;
  Ctrl *ctrl = reinterpret_cast<Ctrl *>(ring + RING_SLOTS * SLOT_BYTES);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctrl->full[s], 1);
      mbar_init(&ctrl->empty[s], 2);   // both CTAs' MMAs read each stage (B halves are shared)
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ctrl->acc_full[s], 1);
      mbar_init(&ctrl->acc_empty[s], EPI_WARPS);
    }
    for (int s = 0; s < RING_SLOTS; ++s) {
      mbar_init(&ctrl->ring_full[s], 1);
      mbar_init(&ctrl->ring_empty[s], EPI_WARPS);
    }
    mbar_init(&ctrl->drain, 1);
    ctrl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane < 2 * args.nprob) {
    tma_prefetch_desc(lane & 1 ? &args.map_b[lane >> 1] : &args.map_a[lane >> 1]);
  }
  if (warp == 1) {
    tmem_alloc(&ctrl->tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncwarp();     // the cluster barrier is warp-aligned
  cluster_sync();   // both CTAs' barriers are initialised before either multicasts into the other
  tc_fence_after();
  // everything above touched only shared and tensor memory; operands, scales and parameters written by
  // earlier kernels are read only after the previous grid has completed
  pdl_wait();
  if (threadIdx.x == 0) pdl_launch_dependents();
  const uint32_t tmem_base = ctrl->tmem_base;
  WaitCtl ctl{&ctrl->abort_flag, args.err, args.timeout_ns};
  const uint32_t rank = cluster_ctarank();
  const long long first = blockIdx.x >> 1;
  const long long stride = gridDim.x >> 1;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      uint32_t stage = 0, phase = 0;
      int last_parity[MAX_STAGES];
      for (int s = 0; s < MAX_STAGES; ++s) last_parity[s] = -1;
      bool ok = true;
      for (long long t = first; ok && t < args.total_tiles; t += stride) {
        // descriptor fields copied to registers: the asm below clobbers memory, which would otherwise force a
        // reload from parameter space on every use
        const int pi = find_problem(args, t);
        const GemmProblem P = args.prob[pi];
        const CUtensorMap *map_a = &args.map_a[pi];
        const CUtensorMap *map_b = &args.map_b[pi];
        int b, ti, tj;
        decode_tile(P, args.symmetric, t - P.tile_begin, rank, b, ti, tj);
        const int k_iters = P.k_iters;
        for (int kk = 0; kk < k_iters; ++kk) {
          if (!wait_bounded(&ctrl->empty[stage], phase ^ 1u, ctl, ERR_WAIT_EMPTY)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&ctrl->full[stage], STAGE_BYTES);
          last_parity[stage] = static_cast<int>(phase);
          uint8_t *sa = smem + stage * STAGE_BYTES;
          uint8_t *sb = sa + A_BYTES;
          tma_load_3d(sa, map_a, &ctrl->full[stage], kk * BK, ti * BM, b);
          // this CTA's half of the shared B operand, delivered to both CTAs of the pair
          if constexpr (!B_MN) {
            // K-major: rows tj*256 + 128*rank .. +127 through the A map (same tensor, box 64 x 128)
            tma_load_3d_mc(sb + rank * (B_BYTES / 2), map_a, &ctrl->full[stage], kk * BK,
                           tj * BN + (BN / 2) * static_cast<int>(rank), b, 0x3);
          } else {
            // N-major: column chunks 2*rank and 2*rank+1 (64 columns each)
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              const int c = 2 * static_cast<int>(rank) + q;
              tma_load_3d_mc(sb + c * (64 * BK * 2), map_b, &ctrl->full[stage], tj * BN + 64 * c, kk * BK, b, 0x3);
            }
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // every armed stage's copies have landed before the CTA may exit
      for (int s = 0; s < STAGES; ++s)
        if (last_parity[s] >= 0) drain_wait(&ctrl->full[s], static_cast<uint32_t>(last_parity[s]), ctl);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, false, B_MN);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      bool issued = false;
      for (long long t = first; ok && t < args.total_tiles; t += stride) {
        if (!wait_bounded(&ctrl->acc_empty[acc], acc_phase ^ 1u, ctl, ERR_WAIT_ACC_EMPTY)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
        const int k_iters = args.prob[find_problem(args, t)].k_iters;
        for (int kk = 0; kk < k_iters; ++kk) {
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
          tc_commit_mc(&ctrl->empty[stage], 0x3);   // frees the stage in both CTAs of the pair
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
        drain_wait(&ctrl->drain, 0u, ctl);
      }
    }
  } else if (warp == LOADER_WARP) {
    if constexpr (EPI != EPI_GRAM) {
      // ---------------------------------------------------------------- epilogue loader (whole warp: lane 0
      // owns the ring barriers and the TMA loads, all lanes share the parameter row copies)
      uint32_t slot = 0, rphase = 0;
      int last_parity[RING_SLOTS];
      for (int s = 0; s < RING_SLOTS; ++s) last_parity[s] = -1;
      bool ok = true;
      for (long long t = first; ok && t < args.total_tiles; t += stride) {
        const int pi = find_problem(args, t);
        const GemmProblem P = args.prob[pi];
        // POLY reads G through the A-operand map (box 64 x 128); APPLY / FINAL read X through the N-major
        // B-operand map (box 64 x 64, two loads)
        const CUtensorMap *aux_map = (EPI == EPI_POLY) ? &args.map_a[pi] : &args.map_b[pi];
        int b, ti, tj;
        decode_tile(P, args.symmetric, t - P.tile_begin, rank, b, ti, tj);
        const int row0 = ti * BM;
        for (int s = 0; s < BN / 64; ++s) {
          const int c0 = tj * BN + 64 * s;
          if (c0 >= P.cols) break;
          if (!slot_used(args.symmetric, c0, row0)) continue;
          bool w = true;
          if (lane == 0) w = wait_bounded(&ctrl->ring_empty[slot], rphase ^ 1u, ctl, ERR_WAIT_RING_EMPTY);
          if (!__shfl_sync(0xffffffffu, w, 0)) {
            ok = false;
            break;
          }
          uint8_t *dst = ring + slot * SLOT_BYTES;
          uint32_t pbytes = 0;
          const void *pbase = nullptr;
          if constexpr (EPI == EPI_FINAL) pbytes = stage_params_bytes(P, b, row0, c0, pbase);
          if (lane == 0) {
            ctrl->ring_param_ok[slot] = pbytes != 0;
            mbar_arrive_expect_tx(&ctrl->ring_full[slot], RING_AUX_BYTES + pbytes);
            if constexpr (EPI == EPI_POLY) {
              tma_load_3d(dst, aux_map, &ctrl->ring_full[slot], c0, row0, b);
            } else {
              tma_load_3d(dst, aux_map, &ctrl->ring_full[slot], c0, row0, b);
              tma_load_3d(dst + 64 * 128, aux_map, &ctrl->ring_full[slot], c0, row0 + 64, b);
            }
          }
          __syncwarp();   // the expected byte count is registered before any lane's copy can complete
          if constexpr (EPI == EPI_FINAL) {
            if (pbytes) stage_params_issue(P, pbase, row0, c0, dst + RING_AUX_BYTES, &ctrl->ring_full[slot], lane);
          }
          last_parity[slot] = static_cast<int>(rphase);
          if (++slot == RING_SLOTS) {
            slot = 0;
            rphase ^= 1u;
          }
        }
      }
      if (lane == 0)
        for (int s = 0; s < RING_SLOTS; ++s)
          if (last_parity[s] >= 0) drain_wait(&ctrl->ring_full[s], static_cast<uint32_t>(last_parity[s]), ctl);
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 2..9)
    const int lane_base = (warp % 4) * 32;  // TMEM lanes this warp may read
    const int rloc = lane_base + lane;      // this thread's row within the tile
    const int my_half = (warp - 2) / 4;     // which 32-column half of each 64-column slot
    uint32_t acc = 0, acc_phase = 0, slot = 0, rphase = 0;
    for (long long t = first; t < args.total_tiles; t += stride) {
      // by value: epilogue stores could alias a reference into parameter space and force reloads
      const GemmProblem P = args.prob[find_problem(args, t)];
      int b, ti, tj;
      decode_tile(P, args.symmetric, t - P.tile_begin, rank, b, ti, tj);
      // every lane waits; the warp proceeds only if all of them saw the accumulator complete, so the
      // warp-collective TMEM loads below never run with part of the warp gone
      bool ok = wait_bounded(&ctrl->acc_full[acc], acc_phase, ctl, ERR_WAIT_ACC_FULL);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const int row0 = ti * BM;
      const int row = row0 + rloc;
      const int warp_row0 = row0 + lane_base;
      bool aborted = false;
#pragma unroll 1
      for (int s = 0; s < BN / 64; ++s) {
        const int c0 = tj * BN + 64 * s;
        if (c0 >= P.cols) break;
        if (EPI != EPI_GRAM && !slot_used(args.symmetric, c0, row0)) continue;
        const uint8_t *slot_ptr = ring + slot * SLOT_BYTES;
        bool staged = false;
        if constexpr (EPI != EPI_GRAM) {
          ok = wait_bounded(&ctrl->ring_full[slot], rphase, ctl, ERR_WAIT_RING_FULL);
          if (!__all_sync(0xffffffffu, ok)) {
            aborted = true;
            break;
          }
          staged = ctrl->ring_param_ok[slot] != 0;
        }
        {
          const int half = my_half;
          const int col0 = c0 + 32 * half;
          // warp-uniform: chunk past the last column, below the diagonal for every lane, or past the last row
          if (col0 < P.cols && !(args.symmetric && col0 + 31 < warp_row0) && warp_row0 < P.rows) {
            float v[32];
            tmem_ld_32x32b_x32(tmem_base + acc * ACC_COLS + (static_cast<uint32_t>(lane_base) << 16) +
                                   (col0 - tj * BN),
                               v);
            epilogue_chunk<EPI>(P, b, row, rloc, col0, half, slot_ptr, slot_ptr + RING_AUX_BYTES, staged, v);
          }
        }
        if constexpr (EPI != EPI_GRAM) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctrl->ring_empty[slot]);
          if (++slot == RING_SLOTS) {
            slot = 0;
            rphase ^= 1u;
          }
        }
      }
      if (aborted) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctrl->acc_empty[acc]);
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  // neither CTA leaves while the other may still multicast into it or arrive on its barriers
  tc_fence_before();
  __syncwarp();     // lanes that ran a role loop rejoin their warp before the warp-aligned barrier
  cluster_sync();
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
muon_status launch_group(const GemmGroup &g, int32_t kind, cudaStream_t s) {
  static std::once_flag attr_once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  std::call_once(attr_once[dev & 63], [] {
    cudaFuncSetAttribute(ns_gemm_kernel<EPI, B_MN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(smem_bytes(EPI)));
  });
  if (g.total_tiles <= 0) return MUON_OK;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = smem_bytes(EPI);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // persistent: as many pairs of CTAs as can be resident at once (one CTA per SM)
  static int max_clusters[64];
  if (max_clusters[dev & 63] == 0) {
    int n = 0;
    cfg.gridDim = dim3(2 * (device_sm_count() / 2));
    if (cudaOccupancyMaxActiveClusters(&n, ns_gemm_kernel<EPI, B_MN>, &cfg) != cudaSuccess || n < 1)
      n = device_sm_count() / 2;
    max_clusters[dev & 63] = n;
  }
  const long long ncl = g.total_tiles < max_clusters[dev & 63] ? g.total_tiles : max_clusters[dev & 63];
  cfg.gridDim = dim3(static_cast<unsigned>(2 * ncl));
  launch_begin(kind, s);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, ns_gemm_kernel<EPI, B_MN>, g);
  launch_end(s);
  return e == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
}

void fill_tiles(GemmProblem &a, long long batch, long long rows, long long cols, long long contraction,
                bool symmetric) {
  a.batch = static_cast<int>(batch);
  a.rows = static_cast<int>(rows);
  a.cols = static_cast<int>(cols);
  a.m_tiles = static_cast<int>((rows + BM - 1) / BM);
  a.n_tiles = static_cast<int>((cols + BN - 1) / BN);
  a.m_pairs = (a.m_tiles + 1) / 2;
  if (symmetric) {
    int cnt = 0;
    for (int j = 0; j < a.n_tiles; ++j) cnt += (a.m_pairs < j + 1 ? a.m_pairs : j + 1);
    a.tiles_per_matrix = cnt;
  } else {
    a.tiles_per_matrix = a.m_pairs * a.n_tiles;
  }
  a.k_iters = static_cast<int>((contraction + BK - 1) / BK);
}

bool apply_maps(const Bf16Stack &h, const Bf16Stack &x, CUtensorMap *ma, CUtensorMap *mb) {
  return make_map(ma, h.ptr, h.cols, h.rows, h.batch, h.ld, h.mstride, BM) &&
         make_map(mb, x.ptr, x.cols, x.rows, x.batch, x.ld, x.mstride, BK);
}

}  // namespace

struct GemmBatch::Item {
  CUtensorMap ma, mb;
  GemmProblem p;
};

GemmBatch::~GemmBatch() { delete[] items_; }

muon_status GemmBatch::push(const Item &it) {
  if (n_ == cap_) {
    const int nc = cap_ ? 2 * cap_ : GEMM_MAX_PROBLEMS;
    Item *ni = new Item[nc];
    for (int i = 0; i < n_; ++i) ni[i] = items_[i];
    delete[] items_;
    items_ = ni;
    cap_ = nc;
  }
  items_[n_++] = it;
  return MUON_OK;
}

muon_status GemmBatch::add_gram(const Bf16Stack &x, __nv_bfloat16 *g, long long ldg, long long mstride_g, float alpha,
                                const float *scale) {
  if (epi_ != EPI_GRAM) return MUON_ERR_INVALID_ARG;
  Item it{};
  if (!make_map(&it.ma, x.ptr, x.cols, x.rows, x.batch, x.ld, x.mstride, BM) ||
      !make_map(&it.mb, x.ptr, x.cols, x.rows, x.batch, x.ld, x.mstride, BN))
    return MUON_ERR_CUDA;
  fill_tiles(it.p, x.batch, x.rows, x.rows, x.cols, true);
  it.p.alpha = alpha;
  it.p.scale = scale;
  it.p.out = g;
  it.p.ld_out = ldg;
  it.p.mstride_out = mstride_g;
  return push(it);
}

muon_status GemmBatch::add_poly(const Bf16Stack &g, __nv_bfloat16 *h, long long ldh, long long mstride_h, float b,
                                float c) {
  if (epi_ != EPI_POLY) return MUON_ERR_INVALID_ARG;
  Item it{};
  if (!make_map(&it.ma, g.ptr, g.cols, g.rows, g.batch, g.ld, g.mstride, BM) ||
      !make_map(&it.mb, g.ptr, g.cols, g.rows, g.batch, g.ld, g.mstride, BN))
    return MUON_ERR_CUDA;
  fill_tiles(it.p, g.batch, g.rows, g.rows, g.cols, true);
  it.p.alpha = 1.f;
  it.p.coef_b = b;
  it.p.coef_c = c;
  it.p.out = h;
  it.p.ld_out = ldh;
  it.p.mstride_out = mstride_h;
  it.p.aux = static_cast<const __nv_bfloat16 *>(g.ptr);
  it.p.ld_aux = g.ld;
  it.p.mstride_aux = g.mstride;
  return push(it);
}

muon_status GemmBatch::add_apply(const Bf16Stack &h, const Bf16Stack &x, __nv_bfloat16 *out, float a,
                                 const float *scale) {
  if (epi_ != EPI_APPLY) return MUON_ERR_INVALID_ARG;
  Item it{};
  if (!apply_maps(h, x, &it.ma, &it.mb)) return MUON_ERR_CUDA;
  fill_tiles(it.p, x.batch, x.rows, x.cols, h.cols, false);
  it.p.coef_a = a;
  it.p.scale = scale;
  it.p.out = out;
  it.p.ld_out = x.ld;
  it.p.mstride_out = x.mstride;
  it.p.aux = static_cast<const __nv_bfloat16 *>(x.ptr);
  it.p.ld_aux = x.ld;
  it.p.mstride_aux = x.mstride;
  return push(it);
}

muon_status GemmBatch::add_final(const Bf16Stack &h, const Bf16Stack &x, float a, const float *scale,
                                 const FinalSpec &f) {
  if (epi_ != EPI_FINAL) return MUON_ERR_INVALID_ARG;
  Item it{};
  if (!apply_maps(h, x, &it.ma, &it.mb)) return MUON_ERR_CUDA;
  fill_tiles(it.p, x.batch, x.rows, x.cols, h.cols, false);
  it.p.coef_a = a;
  it.p.scale = scale;
  it.p.aux = static_cast<const __nv_bfloat16 *>(x.ptr);
  it.p.ld_aux = x.ld;
  it.p.mstride_aux = x.mstride;
  it.p.params = f.params;
  it.p.out_dense = f.out_dense;
  it.p.out_dtype = f.dtype;
  it.p.transposed = f.transposed;
  it.p.orig_cols = f.orig_cols;
  it.p.cautious = f.cautious;
  it.p.lr_wd = f.lr_wd;
  it.p.lr_scale = f.lr_scale;
  return push(it);
}

muon_status GemmBatch::launch(cudaStream_t s) {
  // deepest contraction first, so that the longest tiles start in the first wave of the persistent CTAs
  for (int i = 1; i < n_; ++i)
    for (int j = i; j > 0 && items_[j].p.k_iters > items_[j - 1].p.k_iters; --j) {
      Item t = items_[j];
      items_[j] = items_[j - 1];
      items_[j - 1] = t;
    }
  for (int first = 0; first < n_; first += GEMM_MAX_PROBLEMS) {
    const int cnt = (n_ - first) < GEMM_MAX_PROBLEMS ? (n_ - first) : GEMM_MAX_PROBLEMS;
    GemmGroup g;
    memset(&g, 0, sizeof(g));
    long long tiles = 0;
    for (int i = 0; i < cnt; ++i) {
      g.map_a[i] = items_[first + i].ma;
      g.map_b[i] = items_[first + i].mb;
      g.prob[i] = items_[first + i].p;
      g.prob[i].tile_begin = tiles;
      tiles += static_cast<long long>(g.prob[i].tiles_per_matrix) * g.prob[i].batch;
    }
    g.nprob = cnt;
    g.symmetric = (epi_ == EPI_GRAM || epi_ == EPI_POLY) ? 1 : 0;
    g.total_tiles = tiles;
    g.err = err_;
    g.timeout_ns = timeout_ns_;
    muon_status st;
    switch (epi_) {
      case EPI_GRAM: st = launch_group<EPI_GRAM, false>(g, KK_GRAM, s); break;
      case EPI_POLY: st = launch_group<EPI_POLY, false>(g, KK_POLY, s); break;
      case EPI_APPLY: st = launch_group<EPI_APPLY, true>(g, KK_APPLY, s); break;
      default: st = launch_group<EPI_FINAL, true>(g, KK_FINAL, s); break;
    }
    if (st != MUON_OK) return st;
  }
  return MUON_OK;
}

muon_status launch_gram(const Bf16Stack &x, __nv_bfloat16 *g, long long ldg, long long mstride_g, float alpha,
                        const float *scale, uint32_t *err, unsigned long long timeout_ns, cudaStream_t s) {
  GemmBatch bt(EPI_GRAM, err, timeout_ns);
  muon_status st = bt.add_gram(x, g, ldg, mstride_g, alpha, scale);
  return st != MUON_OK ? st : bt.launch(s);
}

muon_status launch_poly(const Bf16Stack &g, __nv_bfloat16 *h, long long ldh, long long mstride_h, float b, float c,
                        uint32_t *err, unsigned long long timeout_ns, cudaStream_t s) {
  GemmBatch bt(EPI_POLY, err, timeout_ns);
  muon_status st = bt.add_poly(g, h, ldh, mstride_h, b, c);
  return st != MUON_OK ? st : bt.launch(s);
}

muon_status launch_apply(const Bf16Stack &h, const Bf16Stack &x, __nv_bfloat16 *out, float a, const float *scale,
                         uint32_t *err, unsigned long long timeout_ns, cudaStream_t s) {
  GemmBatch bt(EPI_APPLY, err, timeout_ns);
  muon_status st = bt.add_apply(h, x, out, a, scale);
  return st != MUON_OK ? st : bt.launch(s);
}

muon_status launch_final(const Bf16Stack &h, const Bf16Stack &x, float a, const float *scale, const FinalSpec &f,
                         uint32_t *err, unsigned long long timeout_ns, cudaStream_t s) {
  GemmBatch bt(EPI_FINAL, err, timeout_ns);
  muon_status st = bt.add_final(h, x, a, scale, f);
  return st != MUON_OK ? st : bt.launch(s);
}

}  // namespace muon
