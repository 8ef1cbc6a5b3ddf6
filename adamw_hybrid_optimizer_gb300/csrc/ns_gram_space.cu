// The Newton-Schulz iteration in the Gram space ("DMuon: Efficient Distributed Muon Training with Near-Adam
// Overhead", section 2.2 "Efficient Gram Newton-Schulz Iteration"): for a wide iterate X_0 (m x n, m <= n) the
// chain runs on m x m matrices instead of m x n ones. With A_0 = X_0 X_0^T (computed by the tensor-core GEMM's
// fp32 Gram epilogue before this kernel), per step t with coefficients (a, b, c):
//     Q_t = a I + b A_t + c A_t A_t ;  R_{t+1} = Q_t R_t (R_1 = Q_0) ;  A_{t+1} = Q_t (Q_t A_t)
// and X_N = R_N X_0, which the final-step GEMM applies with the parameter update (as R_hi X_0 + R_lo X_0).
// Every matrix here is a polynomial in A_0, so all of them are symmetric and commute.
//
// Precision: forming A squares the condition number, so the m x m chain keeps more than bf16 accuracy. Each
// matrix is stored as two bf16 planes, hi = the value rounded to bf16 and lo = the rest rounded to bf16 (16
// significant bits together), and every product is three bf16 tensor-core passes, hi*hi + hi*lo + lo*hi,
// accumulated in fp32 in tensor memory (the lo*lo term is below that precision). The error of the result is
// then set by the bf16 iterate X_0 and by the bf16 halves of R_N, not by the chain: in fp64 simulations of the
// recurrence on the test inputs (Gaussian, Student-t(3), rank-16 spikes, log-spaced spectra) the bf16 split
// gave the same error against the plain fp64 iteration as fp32-accurate products, to three or four digits.
//
// Design (sm_103a): one cluster of 4 CTAs per matrix (m in 129..256: CTA (bi, bj) owns the 128 x 128 output
// block (bi, bj) of every product) or per 4 matrices (m <= 128: one block each). A CTA's operands are the rows
// of its block row of the left matrix (K-major) and the columns of its block column of the right one, read as
// 64-row slices of that block column (MN-major). The matrices are symmetric only up to rounding, and the
// iteration amplifies the asymmetric part, so every product takes its right operand as stored, never its
// transpose: in fp64 simulations of the recurrence on square Gaussian inputs, reading the right operand
// transposed (exact for symmetric matrices) raised the error ten times. TMA brings the operands in 64-deep
// (128-byte) slices of hi and lo planes through a 3-stage ring, one thread issues tcgen05.mma kind::f16 (bf16, M = 128, N = 128, K = 16) into
// one of two 128-column accumulators, and four epilogue warps (one per tensor-memory lane quarter) finish each
// product 64 columns at a time: the diagonal term of Q, the hi / lo split, and the stores. The CTAs of a cluster
// exchange results through global memory (L2-resident; every block leaves by TMA bulk stores of 128 x 64 bf16
// tiles staged in shared memory), one cluster barrier per phase:
//     phase A: A B = b A + c A A  -> Q = a I + A B (and R_1 = Q_0 at t = 0)
//     phase B: P = Q A, R' = Q R  -> P, R'   (P not at the last step, R' not at t = 0)
//     phase C: A' = Q P           -> A, and B = c' A' + b' I with the next step's coefficients (not at the last step)
// (B = c_0 A_0 + b_0 I comes with A_0 from the Gram epilogue), so no epilogue reads global memory.
// R_N is also stored for the final GEMM as two bf16 halves [R_hi | R_lo] (R has a wide range of magnitudes on
// ill-conditioned inputs, and one bf16 rounding of it would cost more accuracy than the whole bf16 chain): the
// final step contracts them with [X_0; X_0]. Every mbarrier wait is bounded; a wait
// that runs out sets the error word, and the CTA then skips its remaining work but keeps taking part in every
// cluster barrier (so no CTA of the cluster waits forever), drains its copies and MMAs, and frees its TMEM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace muon {

namespace {

constexpr int GS_THREADS = 192;          // warp 0 TMA, warp 1 MMA (+ TMEM owner), warps 2-5 epilogue
constexpr int GS_BLOCK = 128;            // output block side, M and N of every MMA
constexpr int GS_KC = 64;                // bf16 columns per slice: one 128-byte swizzled row
constexpr int GS_TILE_BYTES = GS_BLOCK * GS_KC * 2;          // 16 KB
constexpr int GS_STAGE_BYTES = 4 * GS_TILE_BYTES;            // A hi, A lo, B hi, B lo
constexpr int GS_STAGES = 3;
constexpr int GS_CLUSTER = 4;
constexpr uint32_t GS_TMEM_COLS = 256;   // two 128-column accumulators
constexpr int GS_MAX_PROBLEMS = 8;

struct GsProblem {
  __nv_bfloat16 *planes;    // buffer b, plane p (0 hi, 1 lo), matrix k at ((b * 2 + p) * K + k) * m * ldm
  __nv_bfloat16 *r_out;     // [R_hi | R_lo]: matrix k at r_out + k * m * ld_r, rows of ld_r = 2 * mp elements
  long long ldm, ld_r, mp;  // mp = round64(m): the offset of R_lo in a row
  long long unit_begin;     // first cluster of this problem in the launch
  int K, m, mb;             // matrices, wide rows, 128-row blocks per side (1 or 2)
};

struct GsGroup {
  CUtensorMap map[GS_MAX_PROBLEMS];   // bf16 (m, m, 12 K) over the planes, box 64 x 128, 128-byte swizzle
  CUtensorMap map_b[GS_MAX_PROBLEMS]; // the same tensor, box 64 x 64: a right-operand slice is two of them
  GsProblem prob[GS_MAX_PROBLEMS];
  int nprob;
  long long total_units;
  int ns_steps;
  float coeffs[3 * MUON_MAX_NS_STEPS];
  uint32_t *err;
  unsigned long long timeout_ns;
  unsigned long long *timeline;   // optional per-phase timestamps (performance analysis), or null
  int timeline_cap;               // records per CTA
  int timeline_ctas;              // CTAs that record (the region holds this many)
};
static_assert(sizeof(GsGroup) <= 4096, "kernel parameter block too large");

// Timeline record of one phase (globaltimer ns): phase number + 1, producer first / last copy issue, MMA first
// operands ready, last MMA commit, epilogue first accumulator ready, epilogue end, barrier passed.
constexpr int GS_TL_WORDS = 10;

struct GsCtrl {
  uint64_t full[GS_STAGES];
  uint64_t empty[GS_STAGES];
  uint64_t acc_full[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

constexpr int GS_EPI_WARPS = 4;
constexpr int GS_OUT_TILES = 2;   // double-buffered 128 x 64 bf16 output tiles for the TMA stores
constexpr size_t GS_SMEM = static_cast<size_t>(GS_STAGES) * GS_STAGE_BYTES +
                           static_cast<size_t>(GS_OUT_TILES) * GS_TILE_BYTES + sizeof(GsCtrl) + 1024;
constexpr int GS_EPI_BAR = 1;     // named barrier of the four epilogue warps
static_assert(GS_SMEM <= 232448, "shared memory over budget");

// Epilogue kinds of one product.
enum : int { EK_Q = 0, EK_P = 1, EK_A = 2, EK_R = 3 };

struct Product {
  int a_buf, b_buf, acc, kind, out_buf;
};

// The products of phase `ph` (0 = A, 1 = B, 2 = C) of step t; returns how many (0 if the phase is skipped).
__device__ __forceinline__ int phase_products(int t, int ph, int N, Product *p) {
  const int r_in = GS_R0 + ((t - 1) & 1), r_out = GS_R0 + (t & 1);
  if (ph == 0) {
    p[0] = {GS_G, GS_B, 0, EK_Q, GS_Q};   // A (c A + b I) = b A + c A^2
    return 1;
  }
  if (ph == 1) {
    int n = 0;
    if (t < N - 1) p[n++] = {GS_Q, GS_G, 0, EK_P, GS_P};
    if (t >= 1) p[n++] = {GS_Q, r_in, 1, EK_R, r_out};
    return n;
  }
  if (t < N - 1) {
    p[0] = {GS_Q, GS_P, 0, EK_A, GS_G};
    return 1;
  }
  return 0;
}

// Eight values as bf16: rounded (hi), or what rounding left over, rounded (lo).
__device__ __forceinline__ uint4 pack8_hi(const float *x) {
  uint4 w;
  __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&w);
#pragma unroll
  for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
  return w;
}
__device__ __forceinline__ uint4 pack8_lo(const float *x) {
  uint4 w;
  __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&w);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 r = __bfloat1622float2(__floats2bfloat162_rn(x[2 * e], x[2 * e + 1]));
    h[e] = __floats2bfloat162_rn(x[2 * e] - r.x, x[2 * e + 1] - r.y);
  }
  return w;
}

__device__ __forceinline__ int find_problem(const GsGroup &g, long long u) {
  int p = 0;
#pragma unroll 1
  for (int q = 1; q < g.nprob; ++q)
    if (u >= g.prob[q].unit_begin) p = q;
  return p;
}


// Epilogue output: the four epilogue warps write a 128-row x 64-column bf16 tile of one plane into shared memory
// in the layout a TMA load of that box produces (128-byte rows; 16-byte piece q of row r at position q ^ (r & 7)),
// and one thread stores it with a TMA bulk store, which writes whole rows, leaves out rows and columns past m, and
// runs asynchronously to the warps. Two tiles alternate; the storing thread waits, before a tile is written
// again, until the store two tiles back has read it, and before the phase barrier until every store is done.
struct TileOut {
  uint8_t *tiles;          // GS_OUT_TILES tiles of GS_TILE_BYTES, 1024-byte aligned
  const CUtensorMap *map;  // the planes' tensor map (box 64 x 128)
  int n;                   // tiles stored so far in this kernel
  bool issuer;             // the one thread that issues the stores
};

__device__ __forceinline__ float4 *tile_piece(uint8_t *tile, int r, int q) {
  return reinterpret_cast<float4 *>(tile + r * 128 + ((q ^ (r & 7)) << 4));
}

// Collective over the four epilogue warps: stores rows of block row bi (this lane's row: quarter * 32 + lane of
// the tile), columns col0 .. col0 + 63, of plane `pl` of buffer `buf` of matrix k; piece(q) gives the lane's
// 16-byte piece q (columns col0 + 8 q .. + 7).
template <typename Piece>
__device__ __forceinline__ void store_tile(TileOut &to, const GsProblem &P, int bi, int quarter, int lane, int buf,
                                           int pl, int k, int col0, Piece piece) {
  uint8_t *tile = to.tiles + (to.n & 1) * GS_TILE_BYTES;
  if (to.issuer) bulk_wait_group_read<1>();   // the store that last used this tile has read it
  named_barrier_sync(GS_EPI_BAR, GS_EPI_WARPS * 32);
  const int r = quarter * 32 + lane;
#pragma unroll
  for (int q = 0; q < 8; ++q) *reinterpret_cast<uint4 *>(tile_piece(tile, r, q)) = piece(q);
  fence_proxy_async_shared();                 // the generic writes are visible to the TMA engine
  named_barrier_sync(GS_EPI_BAR, GS_EPI_WARPS * 32);
  if (to.issuer) {
    tma_store_3d(to.map, tile, col0, bi * GS_BLOCK, (buf * 2 + pl) * P.K + k);
    bulk_commit_group();
  }
  ++to.n;
}

// Both planes of one buffer from the lane's 64 values: the bf16 rounding and the rounded rest.
__device__ __forceinline__ void store_split(TileOut &to, const GsProblem &P, int bi, int quarter, int lane, int buf,
                                            int k, int col0, const float *v) {
  store_tile(to, P, bi, quarter, lane, buf, 0, k, col0, [&](int q) { return pack8_hi(v + 8 * q); });
  store_tile(to, P, bi, quarter, lane, buf, 1, k, col0, [&](int q) { return pack8_lo(v + 8 * q); });
}

// R_N for the final GEMM as two bf16 halves, R_hi = rn(R) at column c and R_lo = rn(R - R_hi) at column mp + c,
// zero in the padding columns m .. mp - 1 of each half. Per warp, through a 32 x 32 fp32 staging chunk (so that
// lanes store consecutive columns of a row), with plain stores: it runs once per chain.
__device__ __forceinline__ void store_rsplit(const GsProblem &P, uint8_t *stg, int lane, int k, int row0, int col0,
                                             const float *v) {
#pragma unroll
  for (int q = 0; q < 8; ++q) *tile_piece(stg, lane, q) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  __syncwarp();
  const int q = lane & 7;
  const int c = col0 + 4 * q;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = 4 * i + (lane >> 3);
    if (row0 + r >= P.m || c >= P.mp) continue;
    const float4 x = *tile_piece(stg, r, q);
    const float e[4] = {x.x, x.y, x.z, x.w};
    __nv_bfloat16 hv[4], lv[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float val = c + j < P.m ? e[j] : 0.f;
      hv[j] = __float2bfloat16_rn(val);
      lv[j] = __float2bfloat16_rn(val - __bfloat162float(hv[j]));
    }
    __nv_bfloat16 *d = P.r_out + (static_cast<long long>(k) * P.m + row0 + r) * P.ld_r + c;
    *reinterpret_cast<uint2 *>(d) = *reinterpret_cast<const uint2 *>(hv);            // mp, c: multiples of 4
    *reinterpret_cast<uint2 *>(d + P.mp) = *reinterpret_cast<const uint2 *>(lv);
  }
  __syncwarp();
}

// The epilogue of one 64-column chunk of a product, collective over the four epilogue warps: rows of block row
// bi (lane = row quarter * 32 + lane of the block), columns col0 .. col0 + 63; v holds the lane's 64 values.
// rstage: a 4 KB staging chunk of this warp for the R_N halves (in the operand ring, idle by then).
__device__ __forceinline__ void epilogue_chunk(TileOut &to, const GsProblem &P, const Product &pr, int k, int bi,
                                               int quarter, int lane, int col0, int t, int N, const float *co,
                                               float *v, uint8_t *rstage) {
  const int row0 = bi * GS_BLOCK + quarter * 32;
  const int row = row0 + lane;
  if (col0 < P.m) {
    if (pr.kind == EK_Q) {
      // Q = a I + (b A + c A^2), the bracket from the MMA
#pragma unroll
      for (int j = 0; j < 64; ++j) v[j] += col0 + j == row ? co[3 * t] : 0.f;
      if (t == 0 && N > 1) store_split(to, P, bi, quarter, lane, GS_R0, k, col0, v);   // R_1 = Q_0
    }
    store_split(to, P, bi, quarter, lane, pr.out_buf, k, col0, v);
    if (pr.kind == EK_A) {
      // the next step's right operand c' A' + b' I
      const float bn = co[3 * (t + 1) + 1], cn = co[3 * (t + 1) + 2];
      auto bprime8 = [&](int q, float *w) {
#pragma unroll
        for (int j = 0; j < 8; ++j) w[j] = fmaf(cn, v[8 * q + j], col0 + 8 * q + j == row ? bn : 0.f);
      };
      store_tile(to, P, bi, quarter, lane, GS_B, 0, k, col0, [&](int q) {
        float w[8];
        bprime8(q, w);
        return pack8_hi(w);
      });
      store_tile(to, P, bi, quarter, lane, GS_B, 1, k, col0, [&](int q) {
        float w[8];
        bprime8(q, w);
        return pack8_lo(w);
      });
    }
  }
  // R_N: at t = 0 when N = 1 (R_1 = Q_0), else from the last R product (the phase's only product either way)
  if (row0 < P.m && ((pr.kind == EK_Q && N == 1) || (pr.kind == EK_R && t == N - 1))) {
    store_rsplit(P, rstage, lane, k, row0, col0, v);
    store_rsplit(P, rstage, lane, k, row0, col0 + 32, v + 32);
  }
}

__global__ void __cluster_dims__(GS_CLUSTER, 1, 1) __launch_bounds__(GS_THREADS, 1)
    gram_space_kernel(const __grid_constant__ GsGroup args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *out_tiles = smem + GS_STAGES * GS_STAGE_BYTES;
  GsCtrl *ctrl = reinterpret_cast<GsCtrl *>(out_tiles + GS_OUT_TILES * GS_TILE_BYTES);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();

  if (threadIdx.x == 0) {
    for (int s = 0; s < GS_STAGES; ++s) {
      mbar_init(&ctrl->full[s], 1);
      mbar_init(&ctrl->empty[s], 1);
    }
    mbar_init(&ctrl->acc_full[0], 1);
    mbar_init(&ctrl->acc_full[1], 1);
    mbar_init(&ctrl->drain, 1);
    ctrl->abort_flag = 0;
    fence_mbar_init();
  }
  // this CTA's matrix and output block
  const long long unit = blockIdx.x / GS_CLUSTER;
  const int pi = find_problem(args, unit);
  const GsProblem P = args.prob[pi];
  const long long lu = unit - P.unit_begin;
  const int k = P.mb == 2 ? static_cast<int>(lu) : static_cast<int>(lu * GS_CLUSTER + rank);
  const int bi = P.mb == 2 ? static_cast<int>(rank >> 1) : 0;
  const int bj = P.mb == 2 ? static_cast<int>(rank & 1) : 0;
  const bool active = k < P.K;
  const CUtensorMap *map = &args.map[pi];
  const CUtensorMap *map_b = &args.map_b[pi];
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(map);
    tma_prefetch_desc(map_b);
  }
  if (warp == 1) {
    tmem_alloc(&ctrl->tmem_base, GS_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // A_0 (and the scratch planes) are written by the previous kernel: read only once it has completed
  pdl_wait();
  if (threadIdx.x == 0) pdl_launch_dependents();
  const uint32_t tmem = ctrl->tmem_base;
  WaitCtl ctl{&ctrl->abort_flag, args.err, args.timeout_ns};
  const int N = args.ns_steps;
  const int kchunks = (P.m + GS_KC - 1) / GS_KC;
  constexpr uint32_t idesc = idesc_bf16_f32(GS_BLOCK, GS_BLOCK, false, true);

  // pipeline state, carried across products and phases
  TileOut tout{out_tiles, map, 0, warp == 2 && lane == 0};
  uint32_t stage = 0, sphase = 0;
  int last_parity[GS_STAGES] = {-1, -1, -1};
  uint32_t acc_uses[2] = {0u, 0u};
  bool issued = false;

  int phase_no = 0;
#pragma unroll 1
  for (int t = 0; t < N; ++t) {
#pragma unroll 1
    for (int ph = 0; ph < 3; ++ph) {
      Product prods[2];
      const int np = phase_products(t, ph, N, prods);
      if (np == 0) continue;   // the same for every CTA of the cluster: no barrier for a skipped phase
      const bool work = active && ctrl->abort_flag == 0;
      unsigned long long *rec =
          (args.timeline != nullptr && phase_no < args.timeline_cap && static_cast<int>(blockIdx.x) < args.timeline_ctas)
              ? args.timeline + (static_cast<long long>(blockIdx.x) * args.timeline_cap + phase_no) * GS_TL_WORDS
              : nullptr;
      ++phase_no;
      if (warp == 0) {
        if (lane == 0 && work) {
          // ------------------------------------------------------------ TMA producer
          fence_proxy_async_global();   // the planes were written by generic stores before the last barrier
          if (rec) {
            rec[0] = static_cast<unsigned long long>(phase_no);
            rec[1] = globaltimer_ns();
          }
          bool ok = true;
          for (int q = 0; q < np && ok; ++q) {
            const int za = (prods[q].a_buf * 2) * P.K + k, zb = (prods[q].b_buf * 2) * P.K + k;
            for (int c = 0; c < kchunks; ++c) {
              if (!wait_bounded(&ctrl->empty[stage], sphase ^ 1u, ctl, ERR_WAIT_EMPTY)) {
                ok = false;
                break;
              }
              uint8_t *st = smem + stage * GS_STAGE_BYTES;
              mbar_arrive_expect_tx(&ctrl->full[stage], GS_STAGE_BYTES);
              last_parity[stage] = static_cast<int>(sphase);
              tma_load_3d(st, map, &ctrl->full[stage], c * GS_KC, bi * GS_BLOCK, za);
              tma_load_3d(st + GS_TILE_BYTES, map, &ctrl->full[stage], c * GS_KC, bi * GS_BLOCK, za + P.K);
              // right operand: rows c * 64 .. + 63, columns of block column bj, as two 64-column halves
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int x = bj * GS_BLOCK + 64 * h;
                tma_load_3d(st + 2 * GS_TILE_BYTES + h * (GS_TILE_BYTES / 2), map_b, &ctrl->full[stage], x, c * GS_KC,
                            zb);
                tma_load_3d(st + 3 * GS_TILE_BYTES + h * (GS_TILE_BYTES / 2), map_b, &ctrl->full[stage], x, c * GS_KC,
                            zb + P.K);
              }
              if (++stage == GS_STAGES) {
                stage = 0;
                sphase ^= 1u;
              }
            }
          }
          if (rec) rec[2] = globaltimer_ns();
        }
      } else if (warp == 1) {
        if (lane == 0 && work) {
          // ------------------------------------------------------------ MMA issuer
          tc_fence_after();
          bool ok = true;
          for (int q = 0; q < np && ok; ++q) {
            const uint32_t d = tmem + static_cast<uint32_t>(prods[q].acc * GS_BLOCK);
            for (int c = 0; c < kchunks; ++c) {
              if (!wait_bounded(&ctrl->full[stage], sphase, ctl, ERR_WAIT_FULL)) {
                ok = false;
                break;
              }
              if (rec && q == 0 && c == 0) rec[3] = globaltimer_ns();
              tc_fence_after();
              const uint32_t a_hi = smem_u32(smem + stage * GS_STAGE_BYTES);
              const uint32_t a_lo = a_hi + GS_TILE_BYTES, b_hi = a_hi + 2 * GS_TILE_BYTES,
                             b_lo = a_hi + 3 * GS_TILE_BYTES;
#pragma unroll
              for (int kk = 0; kk < GS_KC / 16; ++kk) {
                const uint64_t ah = smem_desc_sw128(a_hi + kk * 32, 16, 1024);
                const uint64_t al = smem_desc_sw128(a_lo + kk * 32, 16, 1024);
                // MN-major: 16 rows of 128 bytes per step; the second 64-column half 8 KB on
                const uint64_t bh = smem_desc_sw128(b_hi + kk * 16 * 128, GS_TILE_BYTES / 2, 1024);
                const uint64_t bl = smem_desc_sw128(b_lo + kk * 16 * 128, GS_TILE_BYTES / 2, 1024);
                tc_mma_bf16(d, ah, bh, idesc, (c | kk) != 0 ? 1u : 0u);
                tc_mma_bf16(d, ah, bl, idesc, 1u);
                tc_mma_bf16(d, al, bh, idesc, 1u);
              }
              issued = true;
              tc_commit(&ctrl->empty[stage]);
              if (++stage == GS_STAGES) {
                stage = 0;
                sphase ^= 1u;
              }
            }
            if (ok) tc_commit(&ctrl->acc_full[prods[q].acc]);
          }
          if (rec) rec[4] = globaltimer_ns();
        }
      } else {
        // -------------------------------------------------------------- epilogue (warps 2..5)
        const int quarter = warp & 3;               // tensor-memory lanes this warp may read
        uint8_t *rstage = smem + (warp - 2) * (32 * 32 * 4);
        for (int q = 0; q < np; ++q) {
          const Product pr = prods[q];
          const uint32_t par = acc_uses[pr.acc] & 1u;
          acc_uses[pr.acc] += 1u;
          if (!work) continue;
          const bool ok = wait_bounded(&ctrl->acc_full[pr.acc], par, ctl, ERR_WAIT_ACC_FULL);
          // the output stores are collective over the four epilogue warps: they go on only if all saw the
          // accumulator (each thread arrives here after a bounded wait)
          if (!named_barrier_and(GS_EPI_BAR, GS_EPI_WARPS * 32, ok)) continue;
          if (rec && q == 0 && warp == 2 && lane == 0) rec[5] = globaltimer_ns();
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < GS_BLOCK / 64; ++cc) {
            const int col0 = bj * GS_BLOCK + cc * 64;
            if (col0 >= P.mp) break;   // warp-uniform (columns m .. mp - 1: zero padding of [R_hi | R_lo] only)
            const uint32_t ta = tmem + static_cast<uint32_t>(pr.acc * GS_BLOCK + cc * 64) +
                                (static_cast<uint32_t>(quarter * 32) << 16);
            uint32_t r0[32], r1[32];
            tmem_ld_32x32b_x32_async(ta, r0);
            tmem_ld_32x32b_x32_async(ta + 32, r1);
            tmem_ld_wait();
            float v[64];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              v[j] = __uint_as_float(r0[j]);
              v[32 + j] = __uint_as_float(r1[j]);
            }
            epilogue_chunk(tout, P, pr, k, bi, quarter, lane, col0, t, N, args.coeffs, v, rstage);
          }
        }
        // every store of the phase has been performed before the barrier publishes it
        if (tout.issuer) {
          bulk_wait_group_all();
          fence_proxy_async_global();
        }
        if (rec && warp == 2 && lane == 0) rec[6] = globaltimer_ns();
      }
      // ---------------------------------------------------------------- phase barrier (every thread of the cluster):
      // its release / acquire at cluster scope orders this phase's global stores before the next phase's reads,
      // whose TMA copies the producer issues after a proxy fence
      tc_fence_before();
      __syncwarp();
      cluster_sync();
      tc_fence_after();
      if (rec && threadIdx.x == 0) rec[7] = globaltimer_ns();
    }
  }

  // teardown: every armed stage's copies have landed and every MMA has completed before the CTA exits
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < GS_STAGES; ++s)
      if (last_parity[s] >= 0) drain_wait(&ctrl->full[s], static_cast<uint32_t>(last_parity[s]), ctl);
  }
  if (warp == 1 && lane == 0 && issued) {
    tc_commit(&ctrl->drain);
    drain_wait(&ctrl->drain, 0u, ctl);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, GS_TMEM_COLS);
  }
}

// The driver's tensor-map encoder, fetched through the runtime so the library needs no -lcuda.
using EncodeTiledFn = decltype(&cuTensorMapEncodeTiled);

EncodeTiledFn encode_fn() {
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

}  // namespace

size_t gram_space_plane_bytes(long long K, long long m) {
  return static_cast<size_t>(GS_BUFFERS) * 2 * static_cast<size_t>(K) * static_cast<size_t>(m) *
             static_cast<size_t>(round8(m)) * 2 +
         static_cast<size_t>(K) * static_cast<size_t>(m) * static_cast<size_t>(2 * round64(m)) * 2;
}

muon_status launch_gram_space(const GramSpaceStack *stacks, int n, int ns_steps, const float *coeffs, uint32_t *err,
                              unsigned long long timeout_ns, cudaStream_t s) {
  if (n < 1 || ns_steps < 1 || ns_steps > MUON_MAX_NS_STEPS) return MUON_ERR_INVALID_ARG;
  auto enc = encode_fn();
  if (enc == nullptr) return MUON_ERR_CUDA;
  static std::once_flag attr_once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  std::call_once(attr_once[dev & 63], [] {
    cudaFuncSetAttribute(gram_space_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(GS_SMEM));
  });
  for (int first = 0; first < n; first += GS_MAX_PROBLEMS) {
    const int cnt = n - first < GS_MAX_PROBLEMS ? n - first : GS_MAX_PROBLEMS;
    GsGroup g;
    memset(&g, 0, sizeof(g));
    long long units = 0;
    for (int i = 0; i < cnt; ++i) {
      const GramSpaceStack &st = stacks[first + i];
      if (st.m < 1 || st.m > GS_MAX_M || st.K < 1) return MUON_ERR_INVALID_ARG;
      GsProblem &P = g.prob[i];
      P.planes = st.planes;
      P.r_out = gram_space_rsplit(st.planes, st.K, st.m);
      P.ldm = round8(st.m);
      P.mp = round64(st.m);
      P.ld_r = 2 * P.mp;
      P.K = st.K;
      P.m = st.m;
      P.mb = st.m > GS_BLOCK ? 2 : 1;
      P.unit_begin = units;
      units += P.mb == 2 ? st.K : (st.K + GS_CLUSTER - 1) / GS_CLUSTER;
      cuuint64_t dims[3] = {static_cast<cuuint64_t>(st.m), static_cast<cuuint64_t>(st.m),
                            static_cast<cuuint64_t>(2 * GS_BUFFERS) * static_cast<cuuint64_t>(st.K)};
      cuuint64_t strides[2] = {static_cast<cuuint64_t>(P.ldm) * 2,
                               static_cast<cuuint64_t>(P.ldm) * static_cast<cuuint64_t>(st.m) * 2};
      cuuint32_t box[3] = {static_cast<cuuint32_t>(GS_KC), static_cast<cuuint32_t>(GS_BLOCK), 1u};
      cuuint32_t box_b[3] = {64u, static_cast<cuuint32_t>(GS_KC), 1u};
      cuuint32_t estr[3] = {1u, 1u, 1u};
      if (enc(&g.map[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, st.planes, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
          enc(&g.map_b[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, st.planes, dims, strides, box_b, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return MUON_ERR_CUDA;
    }
    g.nprob = cnt;
    g.total_units = units;
    g.ns_steps = ns_steps;
    for (int i = 0; i < 3 * ns_steps; ++i) g.coeffs[i] = coeffs[i];
    g.err = err;
    g.timeout_ns = timeout_ns;
    debug_timeline(&g.timeline, &g.timeline_cap);
    g.timeline_ctas = device_sm_count();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(GS_CLUSTER * units));
    cfg.blockDim = dim3(GS_THREADS);
    cfg.dynamicSmemBytes = GS_SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    launch_begin(KK_GRAM_SPACE, s);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, gram_space_kernel, g);
    launch_end(s);
    if (e != cudaSuccess) return MUON_ERR_CUDA;
  }
  return MUON_OK;
}

}  // namespace muon
