// CUDA-core fp32 GEMM for the fp32 Newton-Schulz path (MC_NS_FP32):
//   D[b] = s_b * (alpha * A[b] x op(B[b]) + beta * C[b] + diag * I)
// op(B) = B^T when B is stored [N, K] (K contiguous), B when stored [K, N].
// Used for fp32 weights, where the update must match exact arithmetic to
// ~1e-5 of its RMS, beyond what bf16 tensor-core operands give.  Products are
// summed 16 at a time in fp32 and folded into a running sum kept as an
// unevaluated pair of fp32 values (hi + lo, by TwoSum: ~48 significand bits,
// where fp64 adds would cost far more on this part), so rounding error grows
// with sqrt(16) rather than sqrt(K); the epilogue runs in fp64.
// 64 x 64 output tiles, 32-deep k-tiles in two shared-memory buffers: the next
// k-tile's global loads (float4) are in flight while the current one is used.
#include "common.cuh"
#include "kernels.h"

namespace mc {
namespace {

constexpr int BM = 64, BN = 64, BK = 32, NT = 256;
constexpr int FOLD = 16;                 // fp32 partial sums of 16 products, folded into fp64

__device__ inline int find_group(const GemmParams& p, int t) {
  int g = 0;
  while (g + 1 < p.ngroups && p.g[g + 1].tile_begin <= t) ++g;
  return g;
}

// 8 consecutive elements of row r, columns c .. c + 7 (as two float4), zero past
// `cols`; the planes are 16-byte aligned with pitches of whole float4s.
__device__ inline void load8(const float* base, long long ld, int r, int rows, int c, int cols,
                             float4& x0, float4& x1) {
  x0 = x1 = make_float4(0.f, 0.f, 0.f, 0.f);
  if (r >= rows) return;
  const float* row = base + (long long)r * ld;
  if (c + 7 < cols) {
    x0 = *reinterpret_cast<const float4*>(row + c);
    x1 = *reinterpret_cast<const float4*>(row + c + 4);
    return;
  }
  float v[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) v[e] = c + e < cols ? row[c + e] : 0.f;
  x0 = make_float4(v[0], v[1], v[2], v[3]);
  x1 = make_float4(v[4], v[5], v[6], v[7]);
}

// s + e = a + b exactly (Knuth's TwoSum; IEEE fp32, no reassociation)
__device__ inline void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

__global__ void __launch_bounds__(NT) sgemm_kernel(const __grid_constant__ GemmParams p) {
  // double-buffered k-tiles, stored k-major: X[k][row]
  __shared__ __align__(16) float As[2][BK][BM + 4];
  __shared__ __align__(16) float Bs[2][BK][BN + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
    const int gi = find_group(p, t);
    const GemmGroup& g = p.g[gi];
    const int per = g.tiles_per_item;
    const int lt = t - g.tile_begin;
    const int b = lt / per, rem = lt % per;
    const int m0 = (rem % g.tiles_m) * BM, n0 = (rem / g.tiles_m) * BN;
    const float* A = reinterpret_cast<const float*>(g.a_hi) + (long long)b * g.a_bstride;
    const float* B = reinterpret_cast<const float*>(g.b_hi) + (long long)b * g.b_bstride;
    // per thread and k-tile: 8 consecutive elements of A and of B
    //   A [M, K]: row m0 + idx / 4, columns k0 + 8 (idx % 4) ..
    //   B [N, K] (K contiguous): the same with n; B [K, N]: row k0 + idx / 8,
    //   columns n0 + 8 (idx % 8) ..
    const int ar = threadIdx.x >> 2, ak = (threadIdx.x & 3) * 8;
    const int bkr = threadIdx.x >> 3, bkn = (threadIdx.x & 7) * 8;
    float4 a0, a1, b0, b1;
    auto fetch = [&](int k0) {
      load8(A, g.lda, m0 + ar, g.M, k0 + ak, g.K, a0, a1);
      if (g.b_mn_major) load8(B, g.ldb, k0 + bkr, g.K, n0 + bkn, g.N, b0, b1);
      else load8(B, g.ldb, n0 + ar, g.N, k0 + ak, g.K, b0, b1);
    };
    auto stash = [&](int buf) {
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) As[buf][ak + e][ar] = av[e];
      if (g.b_mn_major) {
        *reinterpret_cast<float4*>(&Bs[buf][bkr][bkn]) = b0;
        *reinterpret_cast<float4*>(&Bs[buf][bkr][bkn + 4]) = b1;
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) Bs[buf][ak + e][ar] = bv[e];
      }
    };
    // running sums as unevaluated fp32 pairs (hi + lo), ~48 significand bits
    float acc_hi[4][4] = {}, acc_lo[4][4] = {};
    fetch(0);
    stash(0);
    __syncthreads();
    int buf = 0;
    for (int k0 = 0; k0 < g.K; k0 += BK) {
      const bool more = k0 + BK < g.K;
      if (more) fetch(k0 + BK);                  // in flight while this tile computes
#pragma unroll
      for (int f = 0; f < BK; f += FOLD) {
        float acc[4][4] = {};
#pragma unroll
        for (int k = f; k < f + FOLD; ++k) {
          const float4 av = *reinterpret_cast<const float4*>(&As[buf][k][ty * 4]);
          const float4 bv = *reinterpret_cast<const float4*>(&Bs[buf][k][tx * 4]);
          const float a[4] = {av.x, av.y, av.z, av.w}, bb[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float sum, err;
            two_sum(acc_hi[i][j], acc[i][j], sum, err);
            acc_hi[i][j] = sum;
            acc_lo[i][j] += err;
          }
      }
      if (more) stash(buf ^ 1);                  // the other buffer was last read a tile ago
      __syncthreads();
      buf ^= 1;
    }
    const float s = p.s ? p.s[g.mat_base + b] : 1.f;
    const float* C = reinterpret_cast<const float*>(g.c_hi);
    float* D = reinterpret_cast<float*>(g.d_hi) + (long long)b * g.d_bstride;
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = m0 + ty * 4 + i;
      if (r >= g.M) continue;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = n0 + tx * 4 + j;
        if (c >= g.N) continue;
        double v = (double)p.alpha * ((double)acc_hi[i][j] + (double)acc_lo[i][j]);
        if (p.beta != 0.f)
          v += (double)p.beta * (double)C[(long long)b * g.c_bstride + (long long)r * g.ldc + c];
        if (r == c) v += (double)p.diag;
        const float vf = (float)(v * (double)s);
        bad |= !finite_f(vf);
        D[(long long)r * g.ldd + c] = vf;
      }
    }
    if (bad) set_status(p.status, MC_STATUS_NONFINITE_UPDATE);
  }
}

}  // namespace

cudaError_t launch_ns_gemm_f32(const GemmParams& p, cudaStream_t s) {
  if (p.total_tiles <= 0) return cudaSuccess;
  const int cap = sm_count() * 4;
  const int grid = p.total_tiles < cap ? p.total_tiles : cap;
  sgemm_kernel<<<grid, NT, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace mc
