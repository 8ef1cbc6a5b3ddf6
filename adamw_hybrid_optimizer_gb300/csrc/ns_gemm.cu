// Tensor-core GEMMs of the Newton-Schulz iteration, one persistent grouped kernel per step kind.
//
// One Newton-Schulz step ("Optimizers: AdamW, Muon and the distributed optimizer", section
// "Muon: orthogonalising the update") on a wide iterate X (m x n, m <= n):
//     G = X X^T                     EPI_GRAM   symmetric: only tiles touching the upper triangle
//                                              are computed ("DMuon", section 2.2, symmetric Gram);
//                                              G and H are stored as their upper 256-blocks (a diagonal
//                                              block whole) and their readers take a block below the
//                                              diagonal as the transpose of the one above it (half_out,
//                                              half_a, half_b), or, for the single-step entry points,
//                                              every value is also stored mirrored
//     H = a I + b G + c G G         EPI_POLY   G symmetric, so G G = G G^T: same operand pattern
//     X' = H X                      EPI_APPLY  (= a X + (b G + c G G) X); B operand X read N-major
//     last step: u = H X, then p <- p - lr*wd*p*mask - lr*scale*u      EPI_FINAL (EPI_FINAL_MASTER: on fp32
//                                                                      master copies of bf16 parameters)
//     A_0 = s^2 X X^T for the Gram-space chain (m <= 256)  EPI_GRAM32  bf16 hi / lo planes of A_0 and of
//                                                                      c_0 A_0 + b_0 I, whole tile stored;
//                                                                      or fp32 sums of contraction slices
//
// Design (sm_103a): CTAs run as pairs (clusters of two) on vertically adjacent 128 x 256 output tiles with
// paired-SM MMAs (tcgen05 cta_group::2, M = 256): each CTA holds its 128 rows of A and one half of B, the
// even CTA issues the MMAs, and each CTA's tensor memory receives its own 128 accumulator rows (2 x 256
// fp32 columns, so the epilogue of one tile overlaps the MMAs of the next). Operands arrive by TMA
// (128-byte swizzle) through a ring of 64-deep stages of 32 KB per CTA (6 stages; POLY in three splits of
// stages and epilogue input slots, picked by a measured autotune or by the contraction depth; EPI_GRAM32, whose
// one tile pair per matrix lies on the diagonal, reads B from its A tile and keeps 12 A-only stages of 16 KB,
// and may split its contraction into slices that a small reduce kernel adds in order). The CTAs are
// persistent (one per SM) and stride over the tiles of up to GEMM_MAX_PROBLEMS stacks at once. Warp roles:
// warp 0 = TMA producer, warp 1 = MMA issuer (and TMEM owner), warps 2-9 = epilogue (two per
// tensor-memory lane quarter, each taking one 32-column half of every 64-column slot), warp 10 = loader
// (POLY: TMA of G's tile into the ring; FINAL: L2 prefetch of the parameters a tile ahead), warp 11 =
// readiness signals (TileSync: per-matrix counters that let consecutive launches overlap). Each epilogue
// warp reshapes its results in shared memory so that global stores (and the final step's parameter loads,
// fetched one chunk ahead) are coalesced 16-byte accesses; transposed outputs are transposed in place
// there (ldmatrix.trans / stmatrix).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace muon {

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int MAX_STAGES = 12;
constexpr int A_BYTES = BM * BK * 2;                  // this CTA's 128 rows of A
constexpr int B_HALF_BYTES = (BN / 2) * BK * 2;       // this CTA's half (128 of 256 columns) of B
constexpr int STAGE_BYTES = A_BYTES + B_HALF_BYTES;
// A mainloop stage holds this CTA's A tile and its half of B, except in the fp32 Gram (EPI_GRAM32), whose B is
// its A: there a stage is the A tile alone, and twice as many stages fit.
__host__ __device__ constexpr int stage_bytes(int epi) { return epi == EPI_GRAM32 ? A_BYTES : STAGE_BYTES; }
constexpr int ACC_COLS = BN;
constexpr uint32_t TMEM_COLS = 512;
constexpr int EPI_WARPS = 8;                                // two per TMEM lane quarter
constexpr int LOADER_WARP = 2 + EPI_WARPS;
constexpr int SIGNAL_WARP = LOADER_WARP + 1;                  // readiness counters' GPU-scope releases
constexpr int NUM_THREADS = 32 * (SIGNAL_WARP + 1);

// Epilogue input ring: a slot holds 64 columns (two 32-column chunks) of a tile's 128 rows, bf16, 128-byte
// lines with the 128B swizzle TMA writes. Only POLY has a second input (G, for its b*G term); the other
// kinds use one slot only as the epilogue's staging space.
constexpr int MAX_RING_SLOTS = 5;
constexpr int RING_AUX_BYTES = BM * 64 * 2;

__host__ __device__ constexpr int ring_slot_bytes(int) { return RING_AUX_BYTES; }
__host__ __device__ constexpr bool has_aux(int epi) { return epi == EPI_POLY; }
// The final step on fp32 master weights: a kernel of its own, so that the plain final step carries none of
// its registers.
constexpr int EPI_FINAL_MASTER = 4;
__host__ __device__ constexpr bool is_final(int epi) { return epi == EPI_FINAL || epi == EPI_FINAL_MASTER; }

struct Ctrl {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t ring_full[MAX_RING_SLOTS];
  uint64_t ring_empty[MAX_RING_SLOTS];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int prod_tile;   // the producer's current tile (CTA-local count), for the final step's L2 prefetch pacing
  uint32_t stored; // with readiness counters: epilogue warps whose part of a tile is stored (all tiles so far)
};

// Pipeline shapes: a long contraction wants mainloop stages, a short one leaves the epilogue as the limit
// and wants ring slots (the epilogue's second input must arrive within one tile's MMA time).
__host__ __device__ constexpr size_t smem_bytes(int epi, int stages, int slots) {
  return static_cast<size_t>(stages) * stage_bytes(epi) + static_cast<size_t>(slots) * ring_slot_bytes(epi) +
         sizeof(Ctrl) + 1024;
}
constexpr int SHORT_K_ITERS = 32;   // without a measured choice, contractions up to 2048 take the deep-ring shape
static_assert(smem_bytes(EPI_GRAM, 6, 1) <= 232448 && smem_bytes(EPI_POLY, 6, 2) <= 232448 &&
                  smem_bytes(EPI_GRAM32, 12, 2) <= 232448 &&
                  smem_bytes(EPI_POLY, 5, 3) <= 232448 && smem_bytes(EPI_POLY, 4, 5) <= 232448,
              "shared memory over budget");

// Kernel parameter: up to GEMM_MAX_PROBLEMS problems of one step kind, in order of tile_begin.
struct GemmGroup {
  CUtensorMap map_a[GEMM_MAX_PROBLEMS];
  CUtensorMap map_b[GEMM_MAX_PROBLEMS];
  // the half-stored symmetric operand (half_a / half_b) as 64 x 64 boxes, for its blocks read transposed
  CUtensorMap map_t[GEMM_MAX_PROBLEMS];
  GemmProblem prob[GEMM_MAX_PROBLEMS];
  int nprob;
  int symmetric;
  long long total_tiles;
  uint32_t *err;
  unsigned long long timeout_ns;
  unsigned long long *timeline;   // optional per-tile timestamps (performance analysis), or null
  int timeline_cap;               // records per CTA
  int counter_deps;               // every problem waits on per-matrix counters: no grid-wide dependency
};
// kernel parameters up to 32764 bytes (CUDA 12.1 and later)
static_assert(sizeof(GemmGroup) <= 32764, "kernel parameter block too large");

// Timeline record of one tile (globaltimer ns): tile index, producer first / last issue, MMA start
// (accumulator free), first / last operands ready, last commit, epilogue start (accumulator full), end.
constexpr int TL_WORDS = 10;
__device__ __forceinline__ unsigned long long *tl_rec(const GemmGroup &g, int local) {
  if (g.timeline == nullptr || local >= g.timeline_cap) return nullptr;
  return g.timeline + (static_cast<long long>(blockIdx.x) * g.timeline_cap + local) * TL_WORDS;
}

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
  // a problem's tile pairs number below 2^31 (checked at launch): 32-bit divisions, which take a fraction of the
  // 64-bit ones' instructions on the producer's path between two tiles
  const uint32_t tl = static_cast<uint32_t>(t);
  const uint32_t tpm = static_cast<uint32_t>(a.tiles_per_matrix);
  b = static_cast<int>(tl / tpm);
  int r = static_cast<int>(tl - static_cast<uint32_t>(b) * tpm);
  if (!symmetric) {
    if (a.ksplit > 1) r = static_cast<int>(static_cast<uint32_t>(r) % (tpm / static_cast<uint32_t>(a.ksplit)));
    tj = static_cast<int>(static_cast<uint32_t>(r) / static_cast<uint32_t>(a.m_pairs));
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

// The contraction slice of local tile pair t and its 64-deep steps k0 .. k1 - 1: the whole contraction unless the
// problem is split, where a matrix's pairs run slice ksplit - 1 first and slice 0 last.
__device__ __forceinline__ int tile_k_range(const GemmProblem &a, long long t, int &k0, int &k1) {
  if (a.ksplit <= 1) {
    k0 = 0;
    k1 = a.k_iters;
    return 0;
  }
  const int per_slice = a.tiles_per_matrix / a.ksplit;
  const int r = static_cast<int>(static_cast<uint32_t>(t) % static_cast<uint32_t>(a.tiles_per_matrix));
  const int slice = a.ksplit - 1 - r / per_slice;
  k0 = slice * a.kper;
  k1 = min(a.k_iters, k0 + a.kper);
  return slice;
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

// ------------------------------------------------------------------------------------------ epilogue staging
//
// Each epilogue warp owns a 32 x 32 region of the current ring slot: tile rows lane_base .. +31 (one
// 128-byte line each) and the 64-byte half `half` of those lines, with the slot's 128-byte swizzle (16-byte
// piece q of line L sits at piece position q ^ (L & 7)). The region first holds the warp's part of the
// second input (as the loader's TMA wrote it); once every lane has read that, the warp reuses it to
// reshape its results, so that every global store is a 16-byte store of 8 consecutive elements, four lanes
// covering one 64-byte row segment. Row-wise access (a thread's own row) and segment-wise access (seg_row
// below) are both free of bank conflicts beyond the 4 wavefronts 512 bytes need.

struct Region {
  uint8_t *slot;
  int lane_base, half;
  __device__ __forceinline__ uint8_t *piece(int i, int q) const {
    const int line = lane_base + i;
    return slot + line * 128 + ((((half << 2) + q) ^ (line & 7)) << 4);
  }
};

// the thread's own row i: 32 values in, 32 values out
__device__ __forceinline__ void region_read_row(const Region &g, int i, float *dst) {
#pragma unroll
  for (int q = 0; q < 4; ++q) unpack8(*reinterpret_cast<const uint4 *>(g.piece(i, q)), dst + 8 * q);
}
__device__ __forceinline__ void region_write_row(const Region &g, int i, const float *src) {
#pragma unroll
  for (int q = 0; q < 4; ++q) *reinterpret_cast<uint4 *>(g.piece(i, q)) = pack8(src + 8 * q);
}
// Transposes the warp's 32 x 32 region in place (element (i, j) moves to (j, i)): its sixteen 8 x 8 blocks
// are loaded transposed into registers (ldmatrix .trans, block (p, j) by load p) and stored back at the
// mirrored block positions (stmatrix, block (j, p) by store p). Called by every lane of the warp; the
// caller orders other accesses to the region around it with __syncwarp.
__device__ __forceinline__ void region_transpose(const Region &g, int lane) {
  const int j = lane >> 3, k = lane & 7;
  uint32_t r[4][4];
#pragma unroll
  for (int p = 0; p < 4; ++p) ldsm_x4_trans(smem_u32(g.piece(8 * p + k, j)), r[p]);
  __syncwarp();
#pragma unroll
  for (int p = 0; p < 4; ++p) stsm_x4(smem_u32(g.piece(8 * j + k, p)), r[p]);
}

// Segment-wise access: in pass k, lane l handles 16-byte piece l%4 of region row seg_row(l, k). The
// eight lanes of each quarter-warp take rows r and r+4 of the pass, whose swizzled pieces fall on eight
// distinct 16-byte bank groups, so every quarter-warp phase of a 16-byte shared access is conflict-free;
// each group of four lanes still covers one contiguous 64-byte row segment in global memory.
__device__ __forceinline__ int seg_row(int lane, int k) { return 8 * k + (lane >> 3) + 4 * ((lane >> 2) & 1); }

// Stores region row i (32 bf16) to dst_row[0..31] for each of the 32 rows, 16 bytes per lane, four lanes
// per row. ok(i, e) says whether element e of row i may be written; full(i) whether all 32 may.
template <typename Ok, typename Full>
__device__ __forceinline__ void region_store(const Region &g, int lane, __nv_bfloat16 *base, long long ld, Ok ok,
                                             Full full) {
  const int q = lane & 3;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = seg_row(lane, k);
    const uint4 w = *reinterpret_cast<const uint4 *>(g.piece(i, q));
    __nv_bfloat16 *dst = base + static_cast<long long>(i) * ld + 8 * q;
    if (full(i) && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
      *reinterpret_cast<uint4 *>(dst) = w;
    } else {
      const __nv_bfloat16 *h = reinterpret_cast<const __nv_bfloat16 *>(&w);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (ok(i, 8 * q + e)) dst[e] = h[e];
    }
  }
}

// Loads 32 rows x 32 bf16 (src row i at src + i*ld, elements 0..31) into the region, segment-wise.
template <typename Ok, typename Full>
__device__ __forceinline__ void region_load(const Region &g, int lane, const __nv_bfloat16 *base, long long ld, Ok ok,
                                            Full full) {
  const int q = lane & 3;
  uint4 w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = seg_row(lane, k);
    const __nv_bfloat16 *src = base + static_cast<long long>(i) * ld + 8 * q;
    if (full(i) && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
      w[k] = *reinterpret_cast<const uint4 *>(src);
    } else {
      __nv_bfloat16 *h = reinterpret_cast<__nv_bfloat16 *>(&w[k]);
#pragma unroll
      for (int e = 0; e < 8; ++e) h[e] = ok(i, 8 * q + e) ? src[e] : __float2bfloat16_rn(0.f);
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) *reinterpret_cast<uint4 *>(g.piece(seg_row(lane, k), q)) = w[k];
}

// A 32 x 32 block of bf16 parameters as the final step reads it: block row i at base + i*ld, elements
// 0..31; rows below ilim and elements below jlim exist.
struct ParamBlock {
  const __nv_bfloat16 *base;
  long long ld;
  int ilim, jlim;
  bool valid;
};

// Issues this lane's four 16-byte loads of a block (segment-wise, as region_load) into
// registers; they complete while the caller works on something else.
__device__ __forceinline__ void block_fetch(const ParamBlock &pb, int lane, uint4 (&w)[4]) {
  const int q = lane & 3;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = seg_row(lane, k);
    const __nv_bfloat16 *src = pb.base + static_cast<long long>(i) * pb.ld + 8 * q;
    if (i < pb.ilim && pb.jlim >= 32 && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
      w[k] = *reinterpret_cast<const uint4 *>(src);
    } else {
      __nv_bfloat16 *h = reinterpret_cast<__nv_bfloat16 *>(&w[k]);
#pragma unroll
      for (int e = 0; e < 8; ++e) h[e] = (i < pb.ilim && 8 * q + e < pb.jlim) ? src[e] : __float2bfloat16_rn(0.f);
    }
  }
}

__device__ __forceinline__ void block_commit(const Region &g, int lane, const uint4 (&w)[4]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) *reinterpret_cast<uint4 *>(g.piece(seg_row(lane, k), lane & 3)) = w[k];
}

// Muon parameter update of one element: decoupled decay (masked where u*p <= 0 if cautious), then the
// scaled orthogonalised step.
template <bool CAUTIOUS>
__device__ __forceinline__ float param_update_t(float pv, float u, float lr_wd, float lr_scale) {
  const float d = (!CAUTIOUS || u * pv > 0.f) ? lr_wd : 0.f;
  return fmaf(-lr_scale, u, fmaf(-d, pv, pv));
}

// v[j] <- update of parameter value pv(j) with u = v[j], j < 32; the cautious test is taken once per chunk.
template <typename PV>
__device__ __forceinline__ void param_update_32(float *v, PV pv, const GemmProblem &a) {
  const float lr_wd = a.lr_wd, lr_scale = a.lr_scale;
  if (a.cautious) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = param_update_t<true>(pv(j), v[j], lr_wd, lr_scale);
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = param_update_t<false>(pv(j), v[j], lr_wd, lr_scale);
  }
}

__device__ __forceinline__ float param_update(float pv, float u, const GemmProblem &a) {
  const float mask = (!a.cautious || u * pv > 0.f) ? 1.f : 0.f;
  return (pv - a.lr_wd * mask * pv) - a.lr_scale * u;
}

// Final step with fp32 master weights: this thread's row (stored wide) or column (stored tall) of 32
// master values (m: the matrix, cols x rows in the wide orientation) is updated in place, and v receives the
// new values (the caller stores them as bf16).
__device__ __forceinline__ void master_update(float *m, int rows, int cols, int orig_cols, int transposed, int cautious,
                                           float lr_wd, float lr_scale, int row, int col0, float *v) {
  if (row >= rows) return;
  auto upd = [&](float mv, float u) {
    return cautious ? param_update_t<true>(mv, u, lr_wd, lr_scale) : param_update_t<false>(mv, u, lr_wd, lr_scale);
  };
  if (!transposed) {
    float *r = m + static_cast<long long>(row) * orig_cols + col0;
    if (col0 + 32 <= cols && (reinterpret_cast<uintptr_t>(r) & 15) == 0) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float4 x = reinterpret_cast<float4 *>(r)[q];
        x.x = v[4 * q] = upd(x.x, v[4 * q]);
        x.y = v[4 * q + 1] = upd(x.y, v[4 * q + 1]);
        x.z = v[4 * q + 2] = upd(x.z, v[4 * q + 2]);
        x.w = v[4 * q + 3] = upd(x.w, v[4 * q + 3]);
        reinterpret_cast<float4 *>(r)[q] = x;
      }
      return;
    }
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (col0 + j < cols) v[j] = r[j] = upd(r[j], v[j]);
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (col0 + j >= cols) continue;
      float *e = m + static_cast<long long>(col0 + j) * orig_cols + row;
      v[j] = *e = upd(*e, v[j]);
    }
  }
}

// Final step with fp32 parameters or a dense fp32 output: plain per-thread accesses (small stacks only).
__device__ __forceinline__ void final_store_f32(const GemmProblem &a, void *base, int row, int col0, float *v) {
  const bool update = a.params != nullptr;
  float *p = static_cast<float *>(base);
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int c = col0 + j;
    if (c >= a.cols) continue;
    const long long idx = a.transposed ? static_cast<long long>(c) * a.orig_cols + row
                                       : static_cast<long long>(row) * a.orig_cols + c;
    p[idx] = update ? param_update(p[idx], v[j], a) : v[j];
  }
}

// Epilogue for one 32 x 32 chunk: warp rows warp_row0 .. +31 (this thread: row = warp_row0 + lane), columns
// col0 .. +31; v holds this thread's 32 accumulator values. Called by every lane of the warp; the region
// holds the chunk's second input on entry (POLY, APPLY, FINAL) and is free for reuse on exit.
template <int EPI>
__device__ __forceinline__ void epilogue_chunk(const GemmProblem &a, int b, int warp_row0, int lane, int col0,
                                               const Region &rg, float *v, int slice = 0) {
  const int row = warp_row0 + lane;
  const int rows = a.rows, cols = a.cols;
  if constexpr (EPI == EPI_GRAM32) {
    // Each lane writes its own row's 32 values in whole 16-byte pieces: a piece that starts inside the row ends
    // inside its padding (the pitch is a multiple of 8 elements), where every output is zero (the operand's rows
    // past m load as zeros, and the diagonal term lies inside) and nothing reads.
    if (row >= rows) return;
    const long long at = static_cast<long long>(b) * a.mstride_out + static_cast<long long>(row) * a.ld_out + col0;
    if (a.ksplit > 1) {
      // one slice of a split contraction: the raw fp32 sum into the slice's scratch; the reduce kernel scales and
      // splits the total
      float *d = reinterpret_cast<float *>(a.out + (2 + 2 * slice) * a.gs_plane) + at;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (col0 + 4 * q < cols)
          *reinterpret_cast<float4 *>(d + 4 * q) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      return;
    }
    // the whole m x m tile is computed (m <= 256: one tile pair per matrix): G = alpha s^2 acc and c G + b I,
    // each as a bf16 hi plane (rounded) and a bf16 lo plane (the rest, rounded)
    float sc = a.alpha;
    if (a.scale != nullptr) {
      const float s = a.scale[b];
      sc *= s * s;
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] *= sc;
    __nv_bfloat16 *base = a.out + at;
#pragma unroll 1
    for (int bp = 0; bp < 2; ++bp) {   // G, then c G + b I
      const float cm = bp ? a.coef_c : 1.f, dg = bp ? a.coef_b : 0.f;
      __nv_bfloat16 *dh = base + (bp ? a.gs_bprime : 0), *dl = dh + a.gs_plane;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (col0 + 8 * q >= cols) break;
        uint4 wh, wl;
        __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&wh), *l = reinterpret_cast<__nv_bfloat162 *>(&wl);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = 8 * q + 2 * e;
          const float x0 = fmaf(cm, v[j], col0 + j == row ? dg : 0.f);
          const float x1 = fmaf(cm, v[j + 1], col0 + j + 1 == row ? dg : 0.f);
          h[e] = __floats2bfloat162_rn(x0, x1);
          const float2 r = __bfloat1622float2(h[e]);
          l[e] = __floats2bfloat162_rn(x0 - r.x, x1 - r.y);
        }
        *reinterpret_cast<uint4 *>(dh + 8 * q) = wh;
        *reinterpret_cast<uint4 *>(dl + 8 * q) = wl;
      }
    }
    return;
  } else if constexpr (EPI == EPI_GRAM || EPI == EPI_POLY) {
    if constexpr (EPI == EPI_POLY) {
      float gv[32];
      region_read_row(rg, lane, gv);
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = a.coef_b * gv[j] + a.coef_c * v[j] + (col0 + j == row ? a.coef_a : 0.f);
      __syncwarp();
    } else {
      float sc = a.alpha;
      if (a.scale != nullptr) {
        const float s = a.scale[b];
        sc *= s * s;
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] *= sc;
    }
    __nv_bfloat16 *out_b = a.out + static_cast<long long>(b) * a.mstride_out;
    if (a.half_out) {
      // upper 256-blocks only, every element as computed: an off-diagonal block lies above the diagonal, and a
      // diagonal block's pair tile computed both of its halves; readers take the blocks below the diagonal
      // transposed, so nothing is mirrored
      region_write_row(rg, lane, v);
      __syncwarp();
      region_store(
          rg, lane, out_b + static_cast<long long>(warp_row0) * a.ld_out + col0, a.ld_out,
          [&](int i, int j) { return warp_row0 + i < rows && col0 + j < cols; },
          [&](int i) { return warp_row0 + i < rows && col0 + 32 <= cols; });
      return;
    }
    // upper triangle including the diagonal, stored as computed: element (row, c) with c >= row
    region_write_row(rg, lane, v);
    __syncwarp();
    const bool below_free = col0 >= warp_row0 + 31;   // no element of the chunk lies below the diagonal
    region_store(
        rg, lane, out_b + static_cast<long long>(warp_row0) * a.ld_out + col0, a.ld_out,
        [&](int i, int j) { return warp_row0 + i < rows && col0 + j < cols && col0 + j >= warp_row0 + i; },
        [&](int i) { return warp_row0 + i < rows && col0 + 32 <= cols && (below_free || col0 >= warp_row0 + i); });
    __syncwarp();
    // strictly upper part mirrored: element (row, c) also stored at (c, row); the region, transposed in
    // place, holds the transposed chunk, whose row i is output row col0 + i, columns warp_row0 .. +31
    region_transpose(rg, lane);
    __syncwarp();
    region_store(
        rg, lane, out_b + static_cast<long long>(col0) * a.ld_out + warp_row0, a.ld_out,
        [&](int i, int j) { return col0 + i < cols && warp_row0 + j < rows && col0 + i > warp_row0 + j; },
        [&](int i) { return col0 + i < cols && warp_row0 + 32 <= rows && col0 + i > warp_row0 + 31; });
  } else {
    if (a.scale != nullptr) {
      const float sc = a.scale[b];
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] *= sc;
    }
    if constexpr (EPI == EPI_APPLY) {
      region_write_row(rg, lane, v);
      __syncwarp();
      region_store(
          rg, lane, a.out + static_cast<long long>(b) * a.mstride_out + static_cast<long long>(warp_row0) * a.ld_out +
                        col0,
          a.ld_out, [&](int i, int j) { return warp_row0 + i < rows && col0 + j < cols; },
          [&](int i) { return warp_row0 + i < rows && col0 + 32 <= cols; });
    } else {
      const long long mat_elems = static_cast<long long>(rows) * cols;
      void *base = a.params != nullptr ? a.params[b]
                                       : static_cast<void *>(static_cast<char *>(a.out_dense) +
                                                             static_cast<long long>(b) * mat_elems *
                                                                 (a.out_dtype == MUON_F32 ? 4 : 2));
      if (a.out_dtype == MUON_F32) {
        if (row < rows) final_store_f32(a, base, row, col0, v);
        return;
      }
      if constexpr (EPI == EPI_FINAL_MASTER)   // v <- the new master values
        master_update(a.master[b], rows, cols, a.orig_cols, a.transposed, a.cautious, a.lr_wd, a.lr_scale, row, col0,
                      v);
      const bool update = EPI == EPI_FINAL && a.params != nullptr;
      __nv_bfloat16 *p = static_cast<__nv_bfloat16 *>(base);
      if (!a.transposed) {
        // stored wide: region row i = stored row warp_row0 + i, columns col0 ..
        __nv_bfloat16 *blk = p + static_cast<long long>(warp_row0) * a.orig_cols + col0;
        auto ok = [&](int i, int j) { return warp_row0 + i < rows && col0 + j < cols; };
        auto full = [&](int i) { return warp_row0 + i < rows && col0 + 32 <= cols; };
        if (update) {
          region_load(rg, lane, blk, a.orig_cols, ok, full);
          __syncwarp();
          float pv[32];
          region_read_row(rg, lane, pv);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = param_update(pv[j], v[j], a);
          __syncwarp();
        }
        region_write_row(rg, lane, v);
        __syncwarp();
        region_store(rg, lane, blk, a.orig_cols, ok, full);
      } else {
        // stored tall: stored row col0 + i holds wide column col0 + i; its elements warp_row0 .. are wide rows
        __nv_bfloat16 *blk = p + static_cast<long long>(col0) * a.orig_cols + warp_row0;
        auto ok = [&](int i, int j) { return col0 + i < cols && warp_row0 + j < rows; };
        auto full = [&](int i) { return col0 + i < cols && warp_row0 + 32 <= rows; };
        if (update) {
          region_load(rg, lane, blk, a.orig_cols, ok, full);
          __syncwarp();
          region_transpose(rg, lane);   // region row i: wide row warp_row0 + i
          __syncwarp();
          float pv[32];
          region_read_row(rg, lane, pv);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = param_update(pv[j], v[j], a);
          __syncwarp();
        }
        region_write_row(rg, lane, v);
        __syncwarp();
        region_transpose(rg, lane);     // region row i: stored row col0 + i
        __syncwarp();
        region_store(rg, lane, blk, a.orig_cols, ok, full);
      }
    }
  }
}

// The block of bf16 parameters one final-step chunk updates (stored wide: rows = wide rows; stored tall:
// rows = wide columns).
__device__ __forceinline__ ParamBlock param_block(const GemmProblem &a, const __nv_bfloat16 *p, int warp_row0,
                                                  int col0) {
  ParamBlock pb;
  if (!a.transposed) {
    pb.base = p + static_cast<long long>(warp_row0) * a.orig_cols + col0;
    pb.ilim = a.rows - warp_row0;
    pb.jlim = a.cols - col0;
  } else {
    pb.base = p + static_cast<long long>(col0) * a.orig_cols + warp_row0;
    pb.ilim = a.cols - col0;
    pb.jlim = a.rows - warp_row0;
  }
  pb.ld = a.orig_cols;
  pb.valid = col0 < a.cols && warp_row0 < a.rows;
  return pb;
}

// Final-step chunk for bf16 parameters: as epilogue_chunk, with this chunk's parameter block already in
// flight in pf (fetched one chunk ahead); once pf is in the staging region, the block of the chunk 64
// columns on is fetched into pf if fetch_next.
__device__ __forceinline__ void final_chunk_bf16(const GemmProblem &a, int b, int warp_row0, int lane, int col0,
                                                 const Region &rg, float *v, uint4 (&pf)[4], bool fetch_next) {
  __nv_bfloat16 *p = static_cast<__nv_bfloat16 *>(a.params[b]);
  block_commit(rg, lane, pf);
  if (fetch_next) block_fetch(param_block(a, p, warp_row0, col0 + 64), lane, pf);
  if (a.scale != nullptr) {
    const float sc = a.scale[b];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] *= sc;
  }
  __syncwarp();
  // stored tall: the block is transposed in place to the wide orientation, updated row by row, and
  // transposed back
  if (a.transposed) {
    region_transpose(rg, lane);
    __syncwarp();
  }
  {
    float pv[32];
    region_read_row(rg, lane, pv);
    param_update_32(v, [&](int j) { return pv[j]; }, a);
  }
  __syncwarp();
  region_write_row(rg, lane, v);
  __syncwarp();
  if (a.transposed) {
    region_transpose(rg, lane);
    __syncwarp();
  }
  const ParamBlock pb = param_block(a, p, warp_row0, col0);
  region_store(
      rg, lane, const_cast<__nv_bfloat16 *>(pb.base), pb.ld, [&](int i, int j) { return i < pb.ilim && j < pb.jlim; },
      [&](int i) { return i < pb.ilim && pb.jlim >= 32; });
}

template <int EPI, bool B_MN, int STAGES, int RING_SLOTS>
__global__ void __launch_bounds__(NUM_THREADS, 1) ns_gemm_kernel(const __grid_constant__ GemmGroup args) {
  static_assert(STAGES <= MAX_STAGES && RING_SLOTS <= MAX_RING_SLOTS, "pipeline shape");
  constexpr int SLOT_BYTES = ring_slot_bytes(EPI);
  // The fp32 Gram's one tile pair per matrix (m <= 256) lies on the diagonal: each CTA's half of B is the same
  // 128 rows of the same tensor as its A tile, so only A is loaded and the MMA reads B from it.
  constexpr bool SHARED_B = EPI == EPI_GRAM32;
  constexpr int SB = stage_bytes(EPI);
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *ring = smem + STAGES * SB;
  Ctrl *ctrl = reinterpret_cast<Ctrl *>(ring + RING_SLOTS * SLOT_BYTES);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctrl->full[s], 1);
      mbar_init(&ctrl->empty[s], 1);   // the pair MMA's commit, multicast to both CTAs
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ctrl->acc_full[s], 1);
      mbar_init(&ctrl->acc_empty[s], 2 * EPI_WARPS);   // both CTAs' epilogue warps (even CTA's copy used)
    }
    for (int s = 0; s < MAX_RING_SLOTS; ++s) {
      mbar_init(&ctrl->ring_full[s], 1);
      mbar_init(&ctrl->ring_empty[s], EPI_WARPS);
    }
    mbar_init(&ctrl->drain, 1);
    ctrl->abort_flag = 0;
    ctrl->prod_tile = -1;
    ctrl->stored = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane < 2 * args.nprob) {
    tma_prefetch_desc(lane & 1 ? &args.map_b[lane >> 1] : &args.map_a[lane >> 1]);
  }
  if (warp == 1) {
    tmem_alloc_pair(&ctrl->tmem_base, TMEM_COLS);   // jointly with the peer CTA's warp 1
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncwarp();     // the cluster barrier is warp-aligned
  cluster_sync();   // both CTAs' barriers are initialised before either multicasts into the other
  tc_fence_after();
  // everything above touched only shared and tensor memory; operands, scales and parameters written by
  // earlier kernels are read only after the previous grid has completed, or, with per-matrix counters,
  // after the tiles of the matrix they belong to have been stored (the waits below)
  if (!args.counter_deps) pdl_wait();
  if (threadIdx.x == 0) pdl_launch_dependents();
  const uint32_t tmem_base = ctrl->tmem_base;
  WaitCtl ctl{&ctrl->abort_flag, args.err, args.timeout_ns};
  const uint32_t rank = cluster_ctarank();
  const long long first = blockIdx.x >> 1;
  const long long stride = gridDim.x >> 1;
  // the even CTA's copies of the stage-full and accumulator-free barriers, as cluster addresses
  const uint32_t leader_full0 = mapa_shared(smem_u32(&ctrl->full[0]), 0);
  const uint32_t leader_acc_empty0 = mapa_shared(smem_u32(&ctrl->acc_empty[0]), 0);

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      uint32_t stage = 0, phase = 0;
      int last_parity[MAX_STAGES];
      for (int s = 0; s < MAX_STAGES; ++s) last_parity[s] = -1;
      bool ok = true;
      int local = 0;
      int ready_pi = -1, ready_b = -1;   // the last matrix whose inputs this thread has waited for
      for (long long t = first; ok && t < args.total_tiles; t += stride, ++local) {
        unsigned long long *rec = tl_rec(args, local);
        if (rec) {
          rec[0] = static_cast<unsigned long long>(t);
          rec[1] = globaltimer_ns();
        }
        if constexpr (is_final(EPI)) *reinterpret_cast<volatile int *>(&ctrl->prod_tile) = local;
        // descriptor fields copied to registers: the asm below clobbers memory, which would otherwise force a
        // reload from parameter space on every use
        const int pi = find_problem(args, t);
        const GemmProblem P = args.prob[pi];
        const CUtensorMap *map_a = &args.map_a[pi];
        const CUtensorMap *map_b = &args.map_b[pi];
        int b, ti, tj;
        decode_tile(P, args.symmetric, t - P.tile_begin, rank, b, ti, tj);
        if (P.wait_ctr != nullptr && (pi != ready_pi || b != ready_b)) {
          if (!wait_counter(P.wait_ctr + b, P.wait_target, ctl)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();   // the TMA loads below read what the generic stores wrote
          ready_pi = pi;
          ready_b = b;
        }
        int k0, k1;
        tile_k_range(P, t - P.tile_begin, k0, k1);
        for (int kk = k0; kk < k1; ++kk) {
          if (!wait_bounded(&ctrl->empty[stage], phase ^ 1u, ctl, ERR_WAIT_EMPTY)) {
            ok = false;
            break;
          }
          // both CTAs' copies complete on the even CTA's barrier, which the even CTA arms for both
          if (rank == 0) {
            mbar_arrive_expect_tx(&ctrl->full[stage], 2 * SB);
            last_parity[stage] = static_cast<int>(phase);
          }
          if (rec && kk == k0) rec[9] = globaltimer_ns();
          const uint32_t fb = leader_full0 + stage * static_cast<uint32_t>(sizeof(uint64_t));
          uint8_t *sa = smem + stage * SB;
          uint8_t *sb = sa + A_BYTES;
          // half-stored symmetric operands: this step's 256-block (kk / 4) left of the rows' block is read as
          // the transpose of the stored block above the diagonal, in two 64-wide MN-major chunks
          const int kblk = kk >> 2;
          if (P.half_a && kblk < (ti >> 1)) {
#pragma unroll
            for (int q = 0; q < 2; ++q)
              tma_load_3d_pair(sa + q * (64 * BK * 2), &args.map_t[pi], fb, ti * BM + 64 * q, kk * BK, b);
          } else {
            tma_load_3d_pair(sa, map_a, fb, kk * BK, ti * BM, b);
          }
          if constexpr (!SHARED_B) {
            // this CTA's half of B: columns tj*256 + 128*rank .. +127
            if constexpr (!B_MN) {
              if (P.half_b && kblk < tj) {
#pragma unroll
                for (int q = 0; q < 2; ++q)
                  tma_load_3d_pair(sb + q * (64 * BK * 2), &args.map_t[pi], fb,
                                   tj * BN + (BN / 2) * static_cast<int>(rank) + 64 * q, kk * BK, b);
              } else {
                // K-major: those rows of the same tensor through the A map (box 64 x 128)
                tma_load_3d_pair(sb, map_a, fb, kk * BK, tj * BN + (BN / 2) * static_cast<int>(rank), b);
              }
            } else {
              // N-major: column chunks 2*rank and 2*rank+1 (64 columns each); with k_wrap, the second half of the
              // contraction reads B's rows again from the top
              const int kb = (P.k_wrap > 0 && kk >= P.k_wrap) ? kk - P.k_wrap : kk;
#pragma unroll
              for (int q = 0; q < 2; ++q)
                tma_load_3d_pair(sb + q * (64 * BK * 2), map_b, fb, tj * BN + 64 * (2 * static_cast<int>(rank) + q),
                                 kb * BK, b);
            }
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (rec) rec[2] = globaltimer_ns();
      }
      // every armed stage's copies have landed before the CTA may exit
      for (int s = 0; s < STAGES; ++s)
        if (last_parity[s] >= 0) drain_wait(&ctrl->full[s], static_cast<uint32_t>(last_parity[s]), ctl);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------------------------------------------------------- MMA issuer (even CTA: M = 256 pair MMAs)
      constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, BN, false, B_MN);
      // with a half-stored symmetric operand: A transposed (MN-major) and / or B MN-major for some steps
      constexpr uint32_t idesc_kt = idesc_bf16_f32(2 * BM, BN, false, true);
      constexpr uint32_t idesc_tk = idesc_bf16_f32(2 * BM, BN, true, false);
      constexpr uint32_t idesc_tt = idesc_bf16_f32(2 * BM, BN, true, true);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      bool issued = false;
      int local = 0;
      for (long long t = first; ok && t < args.total_tiles; t += stride, ++local) {
        unsigned long long *rec = tl_rec(args, local);
        if (!wait_bounded(&ctrl->acc_empty[acc], acc_phase ^ 1u, ctl, ERR_WAIT_ACC_EMPTY)) break;
        if (rec) rec[3] = globaltimer_ns();
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
        const GemmProblem &P = args.prob[find_problem(args, t)];
        int k0, k1;
        tile_k_range(P, t - P.tile_begin, k0, k1);
        // 256-blocks of the contraction read transposed (half-stored symmetric operands): A's below its rows'
        // block, B's below its columns' block
        int a_tblk = 0, b_tblk = 0;
        if (P.half_a || P.half_b) {
          int mb, mti, mtj;
          decode_tile(P, args.symmetric, t - P.tile_begin, rank, mb, mti, mtj);
          a_tblk = P.half_a ? (mti >> 1) : 0;
          b_tblk = P.half_b ? mtj : 0;
        }
        for (int kk = k0; kk < k1; ++kk) {
          if (!wait_bounded(&ctrl->full[stage], phase, ctl, ERR_WAIT_FULL)) {
            ok = false;
            break;
          }
          if (rec && (kk == k0 || kk == k1 - 1)) rec[kk == k0 ? 4 : 5] = globaltimer_ns();
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * SB);
          const uint32_t sb = SHARED_B ? sa : sa + A_BYTES;
          const bool a_t = (kk >> 2) < a_tblk;
          const bool b_mn = B_MN || (kk >> 2) < b_tblk;
          const uint32_t id = a_t ? (b_mn ? idesc_tt : idesc_tk) : (b_mn ? idesc_kt : idesc);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t adesc =
                a_t ? smem_desc_sw128(sa + k * 16 * 128, 64 * BK * 2, 1024) : smem_desc_sw128(sa + k * 32, 16, 1024);
            const uint64_t bdesc =
                b_mn ? smem_desc_sw128(sb + k * 16 * 128, 64 * BK * 2, 1024) : smem_desc_sw128(sb + k * 32, 16, 1024);
            tc_mma_bf16_pair(d_tmem, adesc, bdesc, id, ((kk - k0) | k) != 0 ? 1u : 0u);
          }
          issued = true;
          tc_commit_pair_mc(&ctrl->empty[stage], 0x3);   // frees the stage in both CTAs of the pair
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair_mc(&ctrl->acc_full[acc], 0x3);    // both CTAs' accumulator halves are ready
        if (rec) rec[6] = globaltimer_ns();
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      // all MMAs this thread issued have completed before TMEM is released
      if (issued) {
        tc_commit_pair_mc(&ctrl->drain, 0x1);
        drain_wait(&ctrl->drain, 0u, ctl);
      }
    }
  } else if (warp == LOADER_WARP) {
    if constexpr (has_aux(EPI)) {
      // ---------------------------------------------------------------- epilogue loader (lane 0 owns the
      // ring barriers and the TMA loads; the warp stays converged for the barrier broadcasts)
      uint32_t slot = 0, rphase = 0;
      int last_parity[MAX_RING_SLOTS];
      for (int s = 0; s < MAX_RING_SLOTS; ++s) last_parity[s] = -1;
      bool ok = true;
      int ready_pi = -1, ready_b = -1;
      for (long long t = first; ok && t < args.total_tiles; t += stride) {
        const int pi = find_problem(args, t);
        const GemmProblem P = args.prob[pi];
        // POLY reads G through the A-operand map (box 64 x 128)
        const CUtensorMap *aux_map = &args.map_a[pi];
        int b, ti, tj;
        decode_tile(P, args.symmetric, t - P.tile_begin, rank, b, ti, tj);
        if (P.wait_ctr != nullptr && (pi != ready_pi || b != ready_b)) {
          bool w = true;
          if (lane == 0) {
            w = wait_counter(P.wait_ctr + b, P.wait_target, ctl);
            if (w) fence_proxy_async_global();
          }
          if (!__shfl_sync(0xffffffffu, w, 0)) break;
          ready_pi = pi;
          ready_b = b;
        }
        const int row0 = ti * BM;
        for (int s = 0; s < BN / 64; ++s) {
          const int c0 = tj * BN + 64 * s;
          if (c0 >= P.cols) break;
          if (!slot_used(args.symmetric && !P.half_out, c0, row0)) continue;
          bool w = true;
          if (lane == 0) w = wait_bounded(&ctrl->ring_empty[slot], rphase ^ 1u, ctl, ERR_WAIT_RING_EMPTY);
          if (!__shfl_sync(0xffffffffu, w, 0)) {
            ok = false;
            break;
          }
          uint8_t *dst = ring + slot * SLOT_BYTES;
          if (lane == 0) {
            mbar_arrive_expect_tx(&ctrl->ring_full[slot], RING_AUX_BYTES);
            tma_load_3d(dst, aux_map, &ctrl->ring_full[slot], c0, row0, b);
          }
          __syncwarp();
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
    } else if constexpr (EPI == EPI_FINAL) {   // (no L2 prefetch for the master kernel: parameters are only written)
      // ---------------------------------------------------------------- L2 prefetch of the parameters the
      // epilogue will update: a tile's rows are requested when the producer starts that tile's operand
      // loads, one to two tiles before its epilogue reads them. Only a hint: the pacing wait gives up after
      // 50 us, and nothing waits for the prefetches.
      volatile int *prod_tile = &ctrl->prod_tile;
      volatile int *abort_flag = &ctrl->abort_flag;
      int local = 0;
      for (long long t = first; t < args.total_tiles; t += stride, ++local) {
        const unsigned long long t0 = globaltimer_ns();
        while (*prod_tile < local && *abort_flag == 0 && globaltimer_ns() - t0 < 50000ull) __nanosleep(256);
        if (*abort_flag != 0) break;
        const GemmProblem P = args.prob[find_problem(args, t)];
        if (P.params == nullptr || P.out_dtype != MUON_BF16 || (P.orig_cols & 7) != 0) continue;
        int b, ti, tj;
        decode_tile(P, args.symmetric, t - P.tile_begin, rank, b, ti, tj);
        const char *p = static_cast<const char *>(P.params[b]);
        if ((reinterpret_cast<uintptr_t>(p) & 15) != 0) continue;
        const int row0 = ti * BM, col0 = tj * BN;
        if (row0 >= P.rows || col0 >= P.cols) continue;   // the pair's second tile row may lie past the end
        if (!P.transposed) {
          // stored wide: this CTA's rows row0 .., columns col0 .. col0 + 255
          const int ncols = min(BN, P.cols - col0);
          for (int r = row0 + lane; r < min(row0 + BM, P.rows); r += 32)
            prefetch_l2_bulk(p + (static_cast<long long>(r) * P.orig_cols + col0) * 2, static_cast<uint32_t>(ncols) * 2);
        } else {
          // stored tall: stored rows col0 .. col0 + 255, stored columns row0 .. row0 + 127
          const int nrows = min(BM, P.rows - row0);
          for (int c = col0 + lane; c < min(col0 + BN, P.cols); c += 32)
            prefetch_l2_bulk(p + (static_cast<long long>(c) * P.orig_cols + row0) * 2, static_cast<uint32_t>(nrows) * 2);
        }
      }
    }
  } else if (warp == SIGNAL_WARP) {
    // ---------------------------------------------------------------- readiness signals: once all eight
    // epilogue warps have stored their parts of this CTA's j-th signalled tile (their CTA-scope releases,
    // acquired here), add them to the tile's matrix counter with one GPU-scope release, so that no epilogue
    // warp waits for its stores to reach the GPU scope
    if (lane == 0) {
      volatile int *abort_flag = &ctrl->abort_flag;
      uint32_t j = 0;   // signalled tiles so far (the epilogue counts only those)
      for (long long t = first; t < args.total_tiles; t += stride) {
        const GemmProblem &P = args.prob[find_problem(args, t)];
        if (P.sig_ctr == nullptr) continue;
        int b, ti, tj;
        decode_tile(P, args.symmetric, t - P.tile_begin, rank, b, ti, tj);
        const uint32_t need = EPI_WARPS * ++j;
        const unsigned long long t0 = globaltimer_ns();
        bool gone = false;
        // a tile takes microseconds: poll with a growing sleep (up to half a microsecond) rather than every few
        // tens of nanoseconds for the whole launch
        unsigned sleep_ns = 32;
        while (ld_acquire_cta_shared(&ctrl->stored) < need) {
          if (*abort_flag != 0 || globaltimer_ns() - t0 > args.timeout_ns) {
            gone = true;
            break;
          }
          __nanosleep(sleep_ns);
          if (sleep_ns < 512) sleep_ns <<= 1;
        }
        if (gone) break;
        red_release_gpu_add(P.sig_ctr + b, static_cast<uint32_t>(EPI_WARPS));
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 2..9)
    const int lane_base = (warp % 4) * 32;  // TMEM lanes this warp may read
    const int my_half = (warp - 2) / 4;     // which 32-column half of each 64-column slot
    uint32_t acc = 0, acc_phase = 0, slot = 0, rphase = 0;
    int local = 0;
    for (long long t = first; t < args.total_tiles; t += stride, ++local) {
      unsigned long long *rec = (warp == 2 && lane == 0) ? tl_rec(args, local) : nullptr;
      // by value: epilogue stores could alias a reference into parameter space and force reloads
      const GemmProblem P = args.prob[find_problem(args, t)];
      int b, ti, tj;
      decode_tile(P, args.symmetric, t - P.tile_begin, rank, b, ti, tj);
      // every lane waits; the warp proceeds only if all of them saw the accumulator complete, so the
      // warp-collective TMEM loads below never run with part of the warp gone
      bool ok = wait_bounded(&ctrl->acc_full[acc], acc_phase, ctl, ERR_WAIT_ACC_FULL);
      if (!__all_sync(0xffffffffu, ok)) break;
      if (rec) rec[7] = globaltimer_ns();
      tc_fence_after();
      const int row0 = ti * BM;
      const int warp_row0 = row0 + lane_base;
      int k0, k1;
      const int slice = EPI == EPI_GRAM32 ? tile_k_range(P, t - P.tile_begin, k0, k1) : 0;
      bool aborted = false;
      // final step with bf16 parameters: their blocks are fetched one chunk ahead
      const bool prefetch_params =
          EPI == EPI_FINAL && P.params != nullptr && P.out_dtype == MUON_BF16;
      const __nv_bfloat16 *pbase = prefetch_params ? static_cast<const __nv_bfloat16 *>(P.params[b]) : nullptr;
      uint4 pf[4];
      bool pf_ready = false;
#pragma unroll 1
      for (int s = 0; s < BN / 64; ++s) {
        const int c0 = tj * BN + 64 * s;
        if (c0 >= P.cols) break;
        if (EPI != EPI_GRAM && !slot_used(args.symmetric && !P.half_out, c0, row0)) continue;
        // kinds without a second input use slot 0 only as staging space
        uint8_t *slot_ptr = ring + (has_aux(EPI) ? slot : 0) * SLOT_BYTES;
        if constexpr (has_aux(EPI)) {
          ok = wait_bounded(&ctrl->ring_full[slot], rphase, ctl, ERR_WAIT_RING_FULL);
          if (!__all_sync(0xffffffffu, ok)) {
            aborted = true;
            break;
          }
        }
        {
          const int col0 = c0 + 32 * my_half;
          // warp-uniform: chunk past the last column, below the diagonal for every lane, or past the last row
          if (col0 < P.cols && !(args.symmetric && !P.half_out && col0 + 31 < warp_row0) && warp_row0 < P.rows) {
            float v[32];
            tmem_ld_32x32b_x32(tmem_base + acc * ACC_COLS + (static_cast<uint32_t>(lane_base) << 16) +
                                   (col0 - tj * BN),
                               v);
            const Region rg{slot_ptr, lane_base, my_half};
            if (EPI == EPI_FINAL && prefetch_params) {
              if (!pf_ready) block_fetch(param_block(P, pbase, warp_row0, col0), lane, pf);
              // only this warp's next chunk of the same tile, if it exists
              const bool next = s + 1 < BN / 64 && col0 + 64 < P.cols;
              final_chunk_bf16(P, b, warp_row0, lane, col0, rg, v, pf, next);
              pf_ready = next;
            } else {
              epilogue_chunk<EPI>(P, b, warp_row0, lane, col0, rg, v, slice);
            }
            __syncwarp();   // every lane's region reads are done before the region is written again
          }
        }
        if constexpr (has_aux(EPI)) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctrl->ring_empty[slot]);
          if (++slot == RING_SLOTS) {
            slot = 0;
            rphase ^= 1u;
          }
        }
      }
      if (aborted) break;
      if (rec) rec[8] = globaltimer_ns();
      tc_fence_before();
      __syncwarp();
      // this warp's stores of the tile are done: count them (CTA-scope release) for the signal warp, which
      // passes them on to the launches that read this matrix
      if (P.sig_ctr != nullptr && lane == 0) red_release_cta_shared_add(&ctrl->stored, 1u);
      // the accumulator is free once both CTAs' epilogues have read their halves (even CTA's barrier); the
      // MMA warp reads none of this warp's global stores, so the signal need not wait for them to drain
      if (lane == 0) mbar_arrive_cluster_relaxed(leader_acc_empty0 + acc * static_cast<uint32_t>(sizeof(uint64_t)));
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
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
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

template <int EPI, bool B_MN, int STAGES, int SLOTS>
muon_status launch_shape(const GemmGroup &g, int32_t kind, cudaStream_t s) {
  constexpr size_t SMEM = smem_bytes(EPI, STAGES, SLOTS);
  static std::once_flag attr_once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  std::call_once(attr_once[dev & 63], [] {
    cudaFuncSetAttribute(ns_gemm_kernel<EPI, B_MN, STAGES, SLOTS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(SMEM));
  });
  if (g.total_tiles <= 0) return MUON_OK;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = SMEM;
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
    if (cudaOccupancyMaxActiveClusters(&n, ns_gemm_kernel<EPI, B_MN, STAGES, SLOTS>, &cfg) != cudaSuccess || n < 1)
      n = device_sm_count() / 2;
    max_clusters[dev & 63] = n;
  }
  const long long ncl = g.total_tiles < max_clusters[dev & 63] ? g.total_tiles : max_clusters[dev & 63];
  cfg.gridDim = dim3(static_cast<unsigned>(2 * ncl));
  launch_begin(kind, s);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, ns_gemm_kernel<EPI, B_MN, STAGES, SLOTS>, g);
  launch_end(s);
  return e == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
}

// ------------------------------------------------------------------------------------------ split fp32 Gram

// One problem of a split EPI_GRAM32 launch, for the reduce kernel: ksplit raw fp32 slice sums, slice j over the
// bf16 planes 2 + 2 j and 3 + 2 j from out (rows x rows, row pitch ld and matrix pitch mstride in elements, plane
// pitch plane); the outputs as the unsplit epilogue writes them.
struct Gram32Reduce {
  __nv_bfloat16 *out;
  const float *scale;
  long long plane, bprime, ld, mstride, block_begin;
  int rows, ksplit, row_blocks;
  float alpha, coef_b, coef_c;
};
struct Gram32ReduceGroup {
  Gram32Reduce prob[GEMM_MAX_PROBLEMS];
  int nprob;
};
static_assert(sizeof(Gram32ReduceGroup) <= 4096, "kernel parameter block too large");

// The outputs of the fp32 Gram from its slices: G = alpha * s^2 * (slice 0 + slice 1 + ...), added in slice
// order, and c G + b I, each as a bf16 hi plane (rounded) and a bf16 lo plane (the rest, rounded): what the
// unsplit epilogue stores. Blocks of 256 threads: 8 rows of one matrix, 32 lanes per row, lane l the 4 columns
// at 4 l and 4 l + 128 (rows <= 256).
__global__ void __launch_bounds__(256) gram32_reduce_kernel(const __grid_constant__ Gram32ReduceGroup G) {
  pdl_wait();
  if (threadIdx.x == 0) pdl_launch_dependents();
  int pi = 0;
  while (pi + 1 < G.nprob && static_cast<long long>(blockIdx.x) >= G.prob[pi + 1].block_begin) ++pi;
  const Gram32Reduce &a = G.prob[pi];
  const long long local = static_cast<long long>(blockIdx.x) - a.block_begin;
  const long long b = local / a.row_blocks;
  const int row = static_cast<int>(local - b * a.row_blocks) * 8 + static_cast<int>(threadIdx.x >> 5);
  if (row >= a.rows) return;
  float sc = a.alpha;
  if (a.scale != nullptr) {
    const float sv = a.scale[b];
    sc *= sv * sv;
  }
  const long long base = b * a.mstride + static_cast<long long>(row) * a.ld;
#pragma unroll 1
  for (int h = 0; h < 2; ++h) {
    const int c = 4 * static_cast<int>(threadIdx.x & 31) + 128 * h;
    if (c >= a.rows) break;
    const bool full = c + 4 <= a.rows;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
    for (int j = 0; j < a.ksplit; ++j) {
      const float *src = reinterpret_cast<const float *>(a.out + (2 + 2 * j) * a.plane) + base + c;
      if (full) {
        const float4 q = __ldcg(reinterpret_cast<const float4 *>(src));
        v[0] += q.x;
        v[1] += q.y;
        v[2] += q.z;
        v[3] += q.w;
      } else {
        for (int e = 0; e < 4; ++e)
          if (c + e < a.rows) v[e] += __ldcg(src + e);
      }
    }
    __nv_bfloat16 o[4][4];   // G hi, G lo, (c G + b I) hi, lo
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float x = v[e] * sc;
      const float xb = fmaf(a.coef_c, x, c + e == row ? a.coef_b : 0.f);
      o[0][e] = __float2bfloat16_rn(x);
      o[1][e] = __float2bfloat16_rn(x - __bfloat162float(o[0][e]));
      o[2][e] = __float2bfloat16_rn(xb);
      o[3][e] = __float2bfloat16_rn(xb - __bfloat162float(o[2][e]));
    }
    const long long off[4] = {0, a.plane, a.bprime, a.bprime + a.plane};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      __nv_bfloat16 *d = a.out + off[w] + base + c;
      if (full) {
        *reinterpret_cast<uint2 *>(d) = *reinterpret_cast<const uint2 *>(o[w]);
      } else {
        for (int e = 0; e < 4; ++e)
          if (c + e < a.rows) d[e] = o[w][e];
      }
    }
  }
}

muon_status launch_gram32_reduce(const Gram32ReduceGroup &g, long long blocks, cudaStream_t s) {
  if (blocks <= 0) return MUON_OK;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  launch_begin(KK_GRAM32_REDUCE, s);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, gram32_reduce_kernel, g);
  launch_end(s);
  return e == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
}

// The slices of each EPI_GRAM32 problem: an explicit count, else the measured one for the stack, else the most
// that would fill one wave of SM pairs with that stack alone while each slice keeps GRAM32_MIN_SLICE_K 64-deep
// steps; clipped to the problem's scratch planes and contraction, and evened out so that no slice is empty.
// Sets ksplit, kper and the problem's tile pairs per matrix. Depends on the problem alone.
void choose_gram_split(GemmProblem *probs, int cnt, int forced) {
  const long long pairs = device_sm_count() / 2;
  for (int i = 0; i < cnt; ++i) {
    GemmProblem &p = probs[i];
    long long sp = forced > 0 ? forced : gram_split_forced();
    if (sp <= 0) sp = gram_split_lookup(p.rows, p.k_iters, p.batch);
    if (sp <= 0) sp = std::min<long long>(pairs / std::max(1, p.batch), p.k_iters / GRAM32_MIN_SLICE_K);
    const long long planes = p.gs_plane > 0 ? (p.gs_bprime / p.gs_plane - 2) / 2 : 0;   // two per slice
    sp = std::min<long long>({sp, GRAM32_MAX_SPLIT, planes, p.k_iters});
    if (sp < 1) sp = 1;
    p.kper = static_cast<int>((p.k_iters + sp - 1) / sp);
    p.ksplit = (p.k_iters + p.kper - 1) / p.kper;
    p.tiles_per_matrix = p.m_pairs * p.n_tiles * p.ksplit;
  }
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
  a.ksplit = 1;
  a.kper = a.k_iters;
}

bool apply_maps(const Bf16Stack &h, const Bf16Stack &x, CUtensorMap *ma, CUtensorMap *mb) {
  return make_map(ma, h.ptr, h.cols, h.rows, h.batch, h.ld, h.mstride, BM) &&
         make_map(mb, x.ptr, x.cols, x.rows, x.batch, x.ld, x.mstride, BK);
}

}  // namespace

struct GemmBatch::Item {
  CUtensorMap ma, mb, mt;
  GemmProblem p;
};

GemmBatch::~GemmBatch() { delete[] items_; }

namespace {
void set_sync(GemmProblem &p, const TileSync *sync) {
  if (sync == nullptr) return;
  p.wait_ctr = sync->wait;
  p.wait_target = sync->target;
  p.sig_ctr = sync->sig;
}
}  // namespace

long long gemm_tiles_per_matrix(int epi, long long m, long long n) {
  GemmProblem p{};
  const bool symmetric = epi == EPI_GRAM || epi == EPI_POLY;
  fill_tiles(p, 1, m, symmetric ? m : n, symmetric ? n : m, symmetric);
  return p.tiles_per_matrix;
}

uint32_t gemm_signals_per_matrix(int epi, long long m, long long n) {
  return static_cast<uint32_t>(gemm_tiles_per_matrix(epi, m, n)) * 2u * EPI_WARPS;
}

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
                                const float *scale, const TileSync *sync) {
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
  it.p.half_out = half_ ? 1 : 0;
  set_sync(it.p, sync);
  return push(it);
}

muon_status GemmBatch::add_gram32(const Bf16Stack &x, __nv_bfloat16 *g_hi, long long ldg, long long mstride_g,
                                  long long plane, long long bprime, float b, float c, float alpha,
                                  const float *scale) {
  if (epi_ != EPI_GRAM32 || x.rows > 2 * BM) return MUON_ERR_INVALID_ARG;
  Item it{};
  if (!make_map(&it.ma, x.ptr, x.cols, x.rows, x.batch, x.ld, x.mstride, BM) ||
      !make_map(&it.mb, x.ptr, x.cols, x.rows, x.batch, x.ld, x.mstride, BN))
    return MUON_ERR_CUDA;
  fill_tiles(it.p, x.batch, x.rows, x.rows, x.cols, false);   // one tile pair per matrix: the whole m x m
  it.p.alpha = alpha;
  it.p.scale = scale;
  it.p.out = g_hi;
  it.p.gs_plane = plane;
  it.p.gs_bprime = bprime;
  it.p.coef_b = b;
  it.p.coef_c = c;
  it.p.ld_out = ldg;
  it.p.mstride_out = mstride_g;
  return push(it);
}

muon_status GemmBatch::add_poly(const Bf16Stack &g, __nv_bfloat16 *h, long long ldh, long long mstride_h, float a,
                                float b, float c, const TileSync *sync) {
  if (epi_ != EPI_POLY) return MUON_ERR_INVALID_ARG;
  Item it{};
  if (!make_map(&it.ma, g.ptr, g.cols, g.rows, g.batch, g.ld, g.mstride, BM) ||
      !make_map(&it.mb, g.ptr, g.cols, g.rows, g.batch, g.ld, g.mstride, BN))
    return MUON_ERR_CUDA;
  fill_tiles(it.p, g.batch, g.rows, g.rows, g.cols, true);
  it.p.alpha = 1.f;
  it.p.coef_a = a;
  it.p.coef_b = b;
  it.p.coef_c = c;
  it.p.out = h;
  it.p.ld_out = ldh;
  it.p.mstride_out = mstride_h;
  if (half_) {
    if (!make_map(&it.mt, g.ptr, g.cols, g.rows, g.batch, g.ld, g.mstride, 64)) return MUON_ERR_CUDA;
    it.p.half_out = it.p.half_a = it.p.half_b = 1;
  }
  set_sync(it.p, sync);
  return push(it);
}

muon_status GemmBatch::add_apply(const Bf16Stack &h, const Bf16Stack &x, __nv_bfloat16 *out, const float *scale,
                                 const TileSync *sync) {
  if (epi_ != EPI_APPLY) return MUON_ERR_INVALID_ARG;
  Item it{};
  if (!apply_maps(h, x, &it.ma, &it.mb)) return MUON_ERR_CUDA;
  fill_tiles(it.p, x.batch, x.rows, x.cols, h.cols, false);
  if (half_) {
    if (!make_map(&it.mt, h.ptr, h.cols, h.rows, h.batch, h.ld, h.mstride, 64)) return MUON_ERR_CUDA;
    it.p.half_a = 1;
  }
  it.p.scale = scale;
  it.p.out = out;
  it.p.ld_out = x.ld;
  it.p.mstride_out = x.mstride;
  set_sync(it.p, sync);
  return push(it);
}

muon_status GemmBatch::add_final(const Bf16Stack &h, const Bf16Stack &x, const float *scale, const FinalSpec &f,
                                 const TileSync *sync, int k_wrap) {
  if (epi_ != EPI_FINAL || k_wrap < 0 || (k_wrap > 0 && h.cols != 2LL * k_wrap * BK)) return MUON_ERR_INVALID_ARG;
  Item it{};
  if (!apply_maps(h, x, &it.ma, &it.mb)) return MUON_ERR_CUDA;
  fill_tiles(it.p, x.batch, x.rows, x.cols, h.cols, false);
  if (half_ && k_wrap == 0) {   // [R_hi | R_lo] of the Gram-space path is stored whole
    if (!make_map(&it.mt, h.ptr, h.cols, h.rows, h.batch, h.ld, h.mstride, 64)) return MUON_ERR_CUDA;
    it.p.half_a = 1;
  }
  it.p.k_wrap = k_wrap;
  it.p.scale = scale;
  it.p.params = f.params;
  it.p.master = f.master;
  it.p.out_dense = f.out_dense;
  it.p.out_dtype = f.dtype;
  it.p.transposed = f.transposed;
  it.p.orig_cols = f.orig_cols;
  it.p.cautious = f.cautious;
  it.p.lr_wd = f.lr_wd;
  it.p.lr_scale = f.lr_scale;
  set_sync(it.p, sync);
  return push(it);
}

int GemmBatch::group_size(int first) const {
  int cnt = (n_ - first) < GEMM_MAX_PROBLEMS ? (n_ - first) : GEMM_MAX_PROBLEMS;
  for (int i = 1; i < cnt; ++i)
    if ((items_[first + i].p.master != nullptr) != (items_[first].p.master != nullptr)) return i;
  return cnt;
}

void GemmBatch::order() {
  // deepest contraction first, so that the longest tiles start in the first wave of the persistent CTAs
  for (int i = 1; i < n_; ++i)
    for (int j = i; j > 0 && items_[j].p.k_iters > items_[j - 1].p.k_iters; --j) {
      Item t = items_[j];
      items_[j] = items_[j - 1];
      items_[j - 1] = t;
    }
  // final steps with fp32 master weights run in launches of their own (a kernel compiled for them)
  if (epi_ == EPI_FINAL) {
    int w = 0;
    for (int pass = 0; pass < 2; ++pass)
      for (int i = w; i < n_; ++i)
        if ((items_[i].p.master != nullptr) == (pass == 1)) {
          Item t = items_[i];
          for (int j = i; j > w; --j) items_[j] = items_[j - 1];
          items_[w++] = t;
        }
  }
}

muon_status GemmBatch::launch(cudaStream_t s) {
  order();
  for (int first = 0; first < n_;) {
    const int cnt = group_size(first);
    const bool master = items_[first].p.master != nullptr;
    GemmGroup g;
    memset(&g, 0, sizeof(g));
    for (int i = 0; i < cnt; ++i) g.prob[i] = items_[first + i].p;
    if (epi_ == EPI_GRAM32) choose_gram_split(g.prob, cnt, split_);
    long long tiles = 0;
    for (int i = 0; i < cnt; ++i) {
      g.map_a[i] = items_[first + i].ma;
      g.map_b[i] = items_[first + i].mb;
      g.map_t[i] = items_[first + i].mt;
      g.prob[i].tile_begin = tiles;
      const long long own = static_cast<long long>(g.prob[i].tiles_per_matrix) * g.prob[i].batch;
      if (own >= (1ll << 31)) return MUON_ERR_SHAPE;   // the kernel decodes a problem's tiles in 32 bits
      tiles += own;
    }
    g.nprob = cnt;
    g.counter_deps = 1;
    for (int i = 0; i < cnt; ++i)
      if (g.prob[i].wait_ctr == nullptr) g.counter_deps = 0;
    if (grid_wait_) g.counter_deps = 0;
    g.symmetric = (epi_ == EPI_GRAM || epi_ == EPI_POLY) ? 1 : 0;
    g.total_tiles = tiles;
    g.err = err_;
    g.timeout_ns = timeout_ns_;
    debug_timeline(&g.timeline, &g.timeline_cap);
    int max_k = 0;
    for (int i = 0; i < cnt; ++i) max_k = g.prob[i].k_iters > max_k ? g.prob[i].k_iters : max_k;
    // POLY's pipeline shape: an explicit override, else the autotune table's measured choice, else the rule
    int shape = force_ >= 0 ? force_ : poly_shape_forced();
    if (shape < 0) shape = poly_shape_lookup(max_k);
    if (shape < 0) shape = max_k <= SHORT_K_ITERS ? 0 : 2;
    muon_status st;
    switch (epi_) {
      case EPI_GRAM: st = launch_shape<EPI_GRAM, false, 6, 1>(g, KK_GRAM, s); break;
      case EPI_GRAM32:
        st = launch_shape<EPI_GRAM32, false, 12, 2>(g, KK_GRAM32, s);
        if (st == MUON_OK) {
          // the split problems' slices, added up
          Gram32ReduceGroup rg;
          memset(&rg, 0, sizeof(rg));
          long long blocks = 0;
          for (int i = 0; i < cnt; ++i) {
            const GemmProblem &p = g.prob[i];
            if (p.ksplit <= 1) continue;
            Gram32Reduce &r = rg.prob[rg.nprob++];
            r.out = p.out;
            r.scale = p.scale;
            r.plane = p.gs_plane;
            r.bprime = p.gs_bprime;
            r.ld = p.ld_out;
            r.mstride = p.mstride_out;
            r.rows = p.rows;
            r.ksplit = p.ksplit;
            r.row_blocks = (p.rows + 7) / 8;
            r.alpha = p.alpha;
            r.coef_b = p.coef_b;
            r.coef_c = p.coef_c;
            r.block_begin = blocks;
            blocks += static_cast<long long>(p.batch) * r.row_blocks;
          }
          st = launch_gram32_reduce(rg, blocks, s);
        }
        break;
      case EPI_POLY:
        st = shape == 0   ? launch_shape<EPI_POLY, false, 4, 5>(g, KK_POLY, s)
             : shape == 1 ? launch_shape<EPI_POLY, false, 5, 3>(g, KK_POLY, s)
                          : launch_shape<EPI_POLY, false, 6, 2>(g, KK_POLY, s);
        break;
      case EPI_APPLY: st = launch_shape<EPI_APPLY, true, 6, 1>(g, KK_APPLY, s); break;
      default:
        st = master ? launch_shape<EPI_FINAL_MASTER, true, 6, 1>(g, KK_FINAL, s)
                    : launch_shape<EPI_FINAL, true, 6, 1>(g, KK_FINAL, s);
        break;
    }
    if (st != MUON_OK) return st;
    first += cnt;
  }
  return MUON_OK;
}

muon_status launch_gram(const Bf16Stack &x, __nv_bfloat16 *g, long long ldg, long long mstride_g, float alpha,
                        const float *scale, uint32_t *err, unsigned long long timeout_ns, cudaStream_t s,
                        const TileSync *sync) {
  GemmBatch bt(EPI_GRAM, err, timeout_ns);
  muon_status st = bt.add_gram(x, g, ldg, mstride_g, alpha, scale, sync);
  return st != MUON_OK ? st : bt.launch(s);
}

muon_status launch_poly(const Bf16Stack &g, __nv_bfloat16 *h, long long ldh, long long mstride_h, float a, float b,
                        float c, uint32_t *err, unsigned long long timeout_ns, cudaStream_t s, const TileSync *sync) {
  GemmBatch bt(EPI_POLY, err, timeout_ns);
  muon_status st = bt.add_poly(g, h, ldh, mstride_h, a, b, c, sync);
  return st != MUON_OK ? st : bt.launch(s);
}

muon_status launch_apply(const Bf16Stack &h, const Bf16Stack &x, __nv_bfloat16 *out, const float *scale,
                         uint32_t *err, unsigned long long timeout_ns, cudaStream_t s, const TileSync *sync) {
  GemmBatch bt(EPI_APPLY, err, timeout_ns);
  muon_status st = bt.add_apply(h, x, out, scale, sync);
  return st != MUON_OK ? st : bt.launch(s);
}

muon_status launch_final(const Bf16Stack &h, const Bf16Stack &x, const float *scale, const FinalSpec &f,
                         uint32_t *err, unsigned long long timeout_ns, cudaStream_t s, const TileSync *sync) {
  GemmBatch bt(EPI_FINAL, err, timeout_ns);
  muon_status st = bt.add_final(h, x, scale, f, sync);
  return st != MUON_OK ? st : bt.launch(s);
}

}  // namespace muon
