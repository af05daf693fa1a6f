// CUDA-core fp32 GEMM for the fp32 Newton-Schulz path (MC_NS_FP32):
//   D[b] = s_b * (alpha * A[b] x op(B[b]) + beta * C[b] + diag * I)
// op(B) = B^T when B is stored [N, K] (K contiguous), B when stored [K, N].
// Used for fp32 weights, where the update must match exact arithmetic to
// ~1e-5 of its RMS, beyond what bf16 tensor-core operands give.  Each 16-wide
// k-tile is summed in fp32 and folded into fp64 accumulators, so rounding
// error grows with sqrt(16) rather than sqrt(K); the epilogue runs in fp64.
#include "common.cuh"
#include "kernels.h"

namespace mc {
namespace {

constexpr int BM = 64, BN = 64, BK = 16, NT = 256;

__device__ inline int find_group(const GemmParams& p, int t) {
  int g = 0;
  while (g + 1 < p.ngroups && p.g[g + 1].tile_begin <= t) ++g;
  return g;
}

__global__ void __launch_bounds__(NT) sgemm_kernel(const __grid_constant__ GemmParams p) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
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
    double acc64[4][4] = {};
    for (int k0 = 0; k0 < g.K; k0 += BK) {
      float acc[4][4] = {};
      // A tile [BM x BK] -> As[k][m]; 1024 elements, 4 per thread
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int idx = threadIdx.x + e * NT;
        const int r = idx / BK, k = idx % BK;
        const int gr = m0 + r, gk = k0 + k;
        As[k][r] = (gr < g.M && gk < g.K) ? A[(long long)gr * g.lda + gk] : 0.f;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int idx = threadIdx.x + e * NT;
        if (g.b_mn_major) {
          const int k = idx / BN, n = idx % BN;
          const int gk = k0 + k, gn = n0 + n;
          Bs[k][n] = (gk < g.K && gn < g.N) ? B[(long long)gk * g.ldb + gn] : 0.f;
        } else {
          const int n = idx / BK, k = idx % BK;
          const int gk = k0 + k, gn = n0 + n;
          Bs[k][n] = (gk < g.K && gn < g.N) ? B[(long long)gn * g.ldb + gk] : 0.f;
        }
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < BK; ++k) {
        float a[4], bb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = As[k][ty * 4 + i];
#pragma unroll
        for (int j = 0; j < 4; ++j) bb[j] = Bs[k][tx * 4 + j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc64[i][j] += (double)acc[i][j];
      __syncthreads();
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
        double v = (double)p.alpha * acc64[i][j];
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
