// Tensor-core (tcgen05 / TMEM / TMA) grouped GEMM for the Newton-Schulz phases
// of Muon ([K2-internals] Algorithm 1 orthogonalisation step; [K2-explained]
// symbol list: "a few iterations of an odd matrix polynomial"):
//
//   phase 1  A  = s * X X^T            (A operand X rows, B operand X rows)
//   phase 2  B  = c * A A + b * A      (A symmetric: its rows serve as B^T)
//   phase 3  X' = s * (B X + a * X)    (B operand X stored [K, N]: MN-major)
//
// All three are D = s_b * (alpha * P + beta * C) with P = A_op x B_op^T.
// Split mode (default): every operand is a bf16 pair (hi, lo) and
// P = hi*hi + hi*lo + lo*hi accumulated in fp32 in TMEM, so products carry
// ~16 significand bits; D is stored again as a (hi, lo) pair.  Plain mode:
// one bf16 plane, one MMA per k-step.
//
// Kernel layout (one CTA per SM, persistent over output tiles):
//   warp 0      TMA producer (one elected lane)
//   warp 1      TMEM allocator + MMA issuer (one elected lane)
//   warps 2..5  epilogue: TMEM -> registers -> fused polynomial -> global
// Tiles are 128 x 256; K advances by BKT (64: 128-byte swizzle rows, or 32:
// 64-byte swizzle rows and twice the stages); the accumulator is
// double-buffered in TMEM (2 x 256 columns) so the epilogue of tile t overlaps
// the MMAs of tile t+1.
//
// Symmetric outputs (phases 1 and 2) are computed only on tiles that touch
// the upper triangle.  Per 128 x 128 block (I, J) of such a tile: I < J is
// stored and mirrored to (J, I); I == J is stored whole (no mirror, so each
// element has exactly one writer); I > J is dropped (its mirror comes from
// block (J, I)).
//
// Every mbarrier wait is bounded; on timeout the kernel records
// MC_STATUS_TIMEOUT, drains its own TMA copies and MMAs, frees TMEM and
// returns.
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "common.cuh"
#include "kernels.h"

namespace mc {
namespace {

constexpr int BM = 128, BN = 256;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;    // two 128 x 256 fp32 accumulators
constexpr int kOperandSmem = 192 * 1024;

// TERMS: tensor-core products per k-step (1: hi*hi, 3: hi*hi + hi*lo + lo*hi).
// LO: the iterate is stored as (hi, lo) planes (the epilogue reads and writes
// both), independently of how many products the k-loop takes.
template <int TERMS, int BKT>
struct Cfg {
  static constexpr int kABytes = BM * BKT * 2;
  static constexpr int kBBytes = BN * BKT * 2;
  static constexpr int kStageBytes = TERMS == 3 ? 2 * (kABytes + kBBytes) : (kABytes + kBBytes);
  static constexpr int kStages = kOperandSmem / kStageBytes;
  static constexpr int kSmem = kStages * kStageBytes + 1024 + 256;
  // K-major operands: rows of BKT bf16 = 128 B (swizzle 128) or 64 B (swizzle 64)
  static constexpr uint32_t kLayout = BKT == 64 ? 2u : 4u;
  static constexpr uint32_t kSbo = 8 * BKT * 2;   // one 8-row swizzle atom
  static_assert(kStages >= 2 && kStages <= 8, "stage count");
};

struct TmaArgs {
  GemmTmaps maps;
};

__device__ inline int find_group(const GemmParams& p, int t) {
  int g = 0;
  while (g + 1 < p.ngroups && p.g[g + 1].tile_begin <= t) ++g;
  return g;
}

struct TileCoord {
  int g, b, m0, n0;
};
__device__ inline TileCoord tile_coord(const GemmParams& p, int t) {
  TileCoord c;
  c.g = find_group(p, t);
  const GemmGroup& G = p.g[c.g];
  const int lt = t - G.tile_begin;
  c.b = lt / G.tiles_per_item;
  int rem = lt % G.tiles_per_item;
  if (!G.symmetric) {
    c.m0 = (rem % G.tiles_m) * BM;   // consecutive tiles share the B column block
    c.n0 = (rem / G.tiles_m) * BN;
  } else {
    // column block tn holds row blocks tm <= 2 tn + 1 (those touching i <= j)
    int tn = 0;
    for (;; ++tn) {
      const int rows = min(G.tiles_m, 2 * tn + 2);
      if (rem < rows) break;
      rem -= rows;
    }
    c.m0 = rem * BM;
    c.n0 = tn * BN;
  }
  return c;
}

template <int TERMS, bool LO, int BKT>
__global__ void __launch_bounds__(kThreads, 1)
    ns_gemm_tc_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ TmaArgs tm) {
  using C = Cfg<TERMS, BKT>;
  constexpr bool SPLIT = TERMS == 3;      // lo operands are loaded and multiplied
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  uint64_t* empty = full + C::kStages;
  uint64_t* tfull = empty + C::kStages;   // [2]
  uint64_t* tempty = tfull + 2;            // [2]
  uint64_t* drain = tempty + 2;            // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < C::kStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int a = 0; a < 2; ++a) { mbar_init(&tfull[a], 1); mbar_init(&tempty[a], 4); }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int g = 0; g < p.ngroups; ++g) {
      prefetch_tmap(&tm.maps.a_hi[g]); prefetch_tmap(&tm.maps.b_hi[g]);
      if (SPLIT) { prefetch_tmap(&tm.maps.a_lo[g]); prefetch_tmap(&tm.maps.b_lo[g]); }
    }
  }
  if (warp == 1) { tmem_alloc(tmem_slot, kTmemCols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  auto fail = [&]() {
    abort_flag = 1;
    set_status(p.status, MC_STATUS_TIMEOUT);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t it = 0;
      uint32_t last_par[8] = {};
      bool used[8] = {};
      for (int t = blockIdx.x; t < p.total_tiles && !abort_flag; t += gridDim.x) {
        const TileCoord tc = tile_coord(p, t);
        const GemmGroup& G = p.g[tc.g];
        const int nk = (G.K + BKT - 1) / BKT;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % C::kStages;
          const uint32_t use = it / C::kStages;
          if (!mbar_wait(&empty[s], (use & 1) ^ 1, &abort_flag)) { fail(); ok = false; break; }
          uint8_t* st = smem + s * C::kStageBytes;
          uint8_t* a_hi = st;
          uint8_t* a_lo = st + C::kABytes;
          uint8_t* b_hi = st + (SPLIT ? 2 * C::kABytes : C::kABytes);
          uint8_t* b_lo = b_hi + C::kBBytes;
          mbar_arrive_expect_tx(&full[s], C::kStageBytes);
          const int k0 = kb * BKT;
          tma_load_3d(a_hi, &tm.maps.a_hi[tc.g], &full[s], k0, tc.m0, tc.b);
          if (SPLIT) tma_load_3d(a_lo, &tm.maps.a_lo[tc.g], &full[s], k0, tc.m0, tc.b);
          if (!G.b_mn_major) {
            tma_load_3d(b_hi, &tm.maps.b_hi[tc.g], &full[s], k0, tc.n0, tc.b);
            if (SPLIT) tma_load_3d(b_lo, &tm.maps.b_lo[tc.g], &full[s], k0, tc.n0, tc.b);
          } else {
#pragma unroll
            for (int q = 0; q < BN / 64; ++q) {
              tma_load_3d(b_hi + q * (64 * BKT * 2), &tm.maps.b_hi[tc.g], &full[s], tc.n0 + 64 * q, k0, tc.b);
              if (SPLIT)
                tma_load_3d(b_lo + q * (64 * BKT * 2), &tm.maps.b_lo[tc.g], &full[s], tc.n0 + 64 * q, k0, tc.b);
            }
          }
          used[s] = true;
          last_par[s] = use & 1;
        }
        if (!ok) break;
      }
      // drain: every issued copy must have landed before the CTA may exit
      for (int s = 0; s < C::kStages; ++s)
        if (used[s]) mbar_wait(&full[s], last_par[s], nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_k = make_idesc_bf16(BM, BN, 0, 0);
      constexpr uint32_t idesc_mn = make_idesc_bf16(BM, BN, 0, 1);
      uint32_t it = 0, tcount = 0;
      bool issued = false;
      for (int t = blockIdx.x; t < p.total_tiles && !abort_flag; t += gridDim.x, ++tcount) {
        const TileCoord tc = tile_coord(p, t);
        const GemmGroup& G = p.g[tc.g];
        const int nk = (G.K + BKT - 1) / BKT;
        const int acc = tcount & 1;
        const uint32_t ause = tcount >> 1;
        if (!mbar_wait(&tempty[acc], (ause & 1) ^ 1, &abort_flag)) { fail(); break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        const uint32_t idesc = G.b_mn_major ? idesc_mn : idesc_k;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % C::kStages;
          const uint32_t use = it / C::kStages;
          if (!mbar_wait(&full[s], use & 1, &abort_flag)) { fail(); ok = false; break; }
          tc_fence_after();
          const uint32_t st = smem_u32(smem + s * C::kStageBytes);
          const uint32_t a_hi = st, a_lo = st + C::kABytes;
          const uint32_t b_hi = st + (SPLIT ? 2 * C::kABytes : C::kABytes), b_lo = b_hi + C::kBBytes;
#pragma unroll
          for (int kk = 0; kk < BKT / 16; ++kk) {
            // K-major: 16 elements = 32 bytes further along the swizzled row
            const uint64_t dah = make_sdesc(a_hi + kk * 32, 16, C::kSbo, C::kLayout);
            uint64_t dbh, dbl = 0, dal = 0;
            if (!G.b_mn_major) {
              dbh = make_sdesc(b_hi + kk * 32, 16, C::kSbo, C::kLayout);
              if (SPLIT) dbl = make_sdesc(b_lo + kk * 32, 16, C::kSbo, C::kLayout);
            } else {
              // MN-major (128-byte swizzle): 16 K-rows = two 1024-byte atoms;
              // 64-wide N blocks are 64*BKT*2 bytes apart
              dbh = make_sdesc(b_hi + kk * 2048, 64 * BKT * 2, 1024, 2);
              if (SPLIT) dbl = make_sdesc(b_lo + kk * 2048, 64 * BKT * 2, 1024, 2);
            }
            const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
            tc_mma(d_tmem, dah, dbh, idesc, accum);
            if (SPLIT) {
              dal = make_sdesc(a_lo + kk * 32, 16, C::kSbo, C::kLayout);
              tc_mma(d_tmem, dah, dbl, idesc, 1u);
              tc_mma(d_tmem, dal, dbh, idesc, 1u);
            }
          }
          issued = true;
          tc_commit(&empty[s]);          // stage free once these MMAs have read it
        }
        if (!ok) break;
        tc_commit(&tfull[acc]);          // accumulator ready for the epilogue
      }
      if (issued) {                      // all issued MMAs complete before teardown
        tc_commit(drain);
        mbar_wait(drain, 0, nullptr);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;              // TMEM lane quadrant of this warp
    uint32_t tcount = 0;
    for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++tcount) {
      const TileCoord tc = tile_coord(p, t);
      const GemmGroup& G = p.g[tc.g];
      const int acc = tcount & 1;
      const uint32_t ause = tcount >> 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&tfull[acc], ause & 1, &abort_flag) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) { if (lane == 0) fail(); break; }
      tc_fence_after();
      const int row = tc.m0 + q * 32 + lane;
      const float sb = p.s ? p.s[G.mat_base + tc.b] : 1.f;
      const float al = p.alpha * sb, be = p.beta * sb;
      const bool row_ok = row < G.M;
      const long long crow = (long long)tc.b * G.c_bstride + (long long)row * G.ldc;
      const long long drow = (long long)tc.b * G.d_bstride + (long long)row * G.ldd;
      const long long mbase = (long long)tc.b * G.d_bstride + row;     // mirror column
      __nv_bfloat16* dh = reinterpret_cast<__nv_bfloat16*>(G.d_hi);
      __nv_bfloat16* dl = reinterpret_cast<__nv_bfloat16*>(G.d_lo);
      bool bad = false;
#pragma unroll 1
      for (int ch = 0; ch < BN / 32; ++ch) {
        float v[32];
        tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN + ch * 32, v);
        const int col0 = tc.n0 + ch * 32;
        // block ownership of this 32-column chunk (symmetric outputs)
        bool store = true, mirror = false;
        if (G.symmetric) {
          const int I = tc.m0 / 128, J = col0 / 128;
          store = I <= J;
          mirror = I < J;
        }
        if (!row_ok || col0 >= G.N || !store) continue;
#pragma unroll
        for (int v8 = 0; v8 < 4; ++v8) {
          const int col = col0 + v8 * 8;
          float* o = v + v8 * 8;
#pragma unroll
          for (int e = 0; e < 8; ++e) o[e] *= al;
          if (p.beta != 0.f && col < G.N) {
            const uint4 ch4 = *reinterpret_cast<const uint4*>(
                reinterpret_cast<const __nv_bfloat16*>(G.c_hi) + crow + col);
            const __nv_bfloat16* chb = reinterpret_cast<const __nv_bfloat16*>(&ch4);
            if (LO) {
              const uint4 cl4 = *reinterpret_cast<const uint4*>(
                  reinterpret_cast<const __nv_bfloat16*>(G.c_lo) + crow + col);
              const __nv_bfloat16* clb = reinterpret_cast<const __nv_bfloat16*>(&cl4);
#pragma unroll
              for (int e = 0; e < 8; ++e)
                o[e] = fmaf(be, __bfloat162float(chb[e]) + __bfloat162float(clb[e]), o[e]);
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) o[e] = fmaf(be, __bfloat162float(chb[e]), o[e]);
            }
          }
        }
        __nv_bfloat16 hb[32], lb[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          bad |= !finite_f(v[e]) && (col0 + e < G.N);
          if (LO) split_bf16(v[e], hb[e], lb[e]);
          else hb[e] = __float2bfloat16_rn(v[e]);
        }
#pragma unroll
        for (int v8 = 0; v8 < 4; ++v8) {
          const int col = col0 + v8 * 8;
          if (col >= G.N) break;
          *reinterpret_cast<uint4*>(dh + drow + col) = *reinterpret_cast<const uint4*>(hb + v8 * 8);
          if (LO)
            *reinterpret_cast<uint4*>(dl + drow + col) = *reinterpret_cast<const uint4*>(lb + v8 * 8);
        }
        if (mirror) {
          // (row, col) also lands at (col, row); lanes hold consecutive rows,
          // so each store instruction covers 64 contiguous bytes
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int col = col0 + e;
            if (col < G.N) {
              dh[mbase + (long long)col * G.ldd] = hb[e];
              if (LO) dl[mbase + (long long)col * G.ldd] = lb[e];
            }
          }
        }
      }
      if (bad) set_status(p.status, MC_STATUS_NONFINITE_UPDATE);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

// 3D bf16 map over `batch` row-major [rows, cols] planes (row stride ld,
// plane stride bstride, both in elements); box = box_cols x box_rows x 1,
// swizzle 128 B (box_cols 64) or 64 B (box_cols 32), zero fill outside
// [cols, rows, batch].
bool encode_3d(CUtensorMap* m, const void* base, int cols, int rows, int batch, long long ld,
               long long bstride, int box_cols, int box_rows, char* err, size_t errlen) {
  EncodeTiledFn enc = get_encode();
  if (!enc) { snprintf(err, errlen, "cuTensorMapEncodeTiled unavailable"); return false; }
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)batch};
  cuuint64_t strides[2] = {(cuuint64_t)ld * 2, (cuuint64_t)bstride * 2};
  cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  const CUtensorMapSwizzle sw = box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(err, errlen, "cuTensorMapEncodeTiled failed (%d): cols=%d rows=%d batch=%d ld=%lld",
             (int)r, cols, rows, batch, ld);
    return false;
  }
  return true;
}

template <int TERMS, bool LO, int BKT>
cudaError_t launch_variant(const GemmParams& p, cudaStream_t s, char* err, size_t errlen) {
  constexpr bool SPLIT = TERMS == 3;
  TmaArgs tm;
  memset(&tm, 0, sizeof(tm));
  for (int g = 0; g < p.ngroups; ++g) {
    const GemmGroup& G = p.g[g];
    // A operand: rows of an [M, K] plane (K contiguous)
    if (!encode_3d(&tm.maps.a_hi[g], G.a_hi, G.K, G.M, G.batch, G.lda, G.a_bstride, BKT, BM, err, errlen))
      return cudaErrorInvalidValue;
    if (SPLIT && !encode_3d(&tm.maps.a_lo[g], G.a_lo, G.K, G.M, G.batch, G.lda, G.a_bstride, BKT, BM, err, errlen))
      return cudaErrorInvalidValue;
    if (!G.b_mn_major) {   // B operand: rows of an [N, K] plane
      if (!encode_3d(&tm.maps.b_hi[g], G.b_hi, G.K, G.N, G.batch, G.ldb, G.b_bstride, BKT, BN, err, errlen))
        return cudaErrorInvalidValue;
      if (SPLIT && !encode_3d(&tm.maps.b_lo[g], G.b_lo, G.K, G.N, G.batch, G.ldb, G.b_bstride, BKT, BN, err, errlen))
        return cudaErrorInvalidValue;
    } else {               // B operand: [K, N] plane, 64-wide N boxes of BKT rows
      if (!encode_3d(&tm.maps.b_hi[g], G.b_hi, G.N, G.K, G.batch, G.ldb, G.b_bstride, 64, BKT, err, errlen))
        return cudaErrorInvalidValue;
      if (SPLIT && !encode_3d(&tm.maps.b_lo[g], G.b_lo, G.N, G.K, G.batch, G.ldb, G.b_bstride, 64, BKT, err, errlen))
        return cudaErrorInvalidValue;
    }
  }
  const int grid = p.total_tiles < sm_count() ? p.total_tiles : sm_count();
  auto k = ns_gemm_tc_kernel<TERMS, LO, BKT>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg<TERMS, BKT>::kSmem);
  if (e != cudaSuccess) return e;
  k<<<grid, kThreads, Cfg<TERMS, BKT>::kSmem, s>>>(p, tm);
  return cudaGetLastError();
}

// K step of the tensor-core GEMM: 64 (default) or 32 (MC_NS_BK=32).
int k_step() {
  static int bk = 0;
  if (bk == 0) {
    const char* e = getenv("MC_NS_BK");
    bk = (e && atoi(e) == 32) ? 32 : 64;
  }
  return bk;
}

}  // namespace

template <int BKT>
cudaError_t launch_bk(const GemmParams& p, cudaStream_t s, char* err, size_t errlen) {
  if (p.xmode != kXSplit) return launch_variant<1, false, BKT>(p, s, err, errlen);
  if (p.terms == 3) return launch_variant<3, true, BKT>(p, s, err, errlen);
  return launch_variant<1, true, BKT>(p, s, err, errlen);
}

cudaError_t launch_ns_gemm_tc(const GemmParams& p, cudaStream_t s, char* err, size_t errlen) {
  if (p.total_tiles <= 0) return cudaSuccess;
  return k_step() == 32 ? launch_bk<32>(p, s, err, errlen) : launch_bk<64>(p, s, err, errlen);
}

}  // namespace mc
