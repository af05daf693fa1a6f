// Per-head max attention logit ([K2-internals] "核心数学"):
//   S_max^h = scale * max_b max_{i, j <= i} q_{b,i,h} . k_{b,j,h}
// Flash-style tiling: the S x S logit matrix is never stored; each CTA keeps
// running maxima in registers and publishes one packed atomicMax per head.
//
// Results travel through the caller's output buffers:
//   argmax == null : smax[h] holds an order-preserving int32 image of the
//                    scaled max during the launch (init -> atomicMax -> decode)
//   argmax != null : argmax[h] holds a packed 64-bit key
//                    (ordered value << 32 | (0xffffffff - flat index)) so one
//                    atomicMax keeps the largest value and, among equal
//                    values, the smallest flat index (b*S + i)*S + j.
#include "common.cuh"
#include "kernels.h"

namespace mc {
namespace {

__device__ inline unsigned long long pack_key(float v, uint32_t idx) {
  const uint32_t u = (uint32_t)float_to_ordered(v) ^ 0x80000000u;
  return ((unsigned long long)u << 32) | (unsigned long long)(0xffffffffu - idx);
}

__global__ void ml_init_kernel(MaxLogitParams p) {
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h >= p.H) return;
  if (p.argmax) {
    reinterpret_cast<unsigned long long*>(p.argmax)[h] = 0ull;
  } else {
    int32_t* si = reinterpret_cast<int32_t*>(p.smax);
    si[h] = float_to_ordered(p.accumulate ? p.smax[h] : -INFINITY);
  }
}

__global__ void ml_final_kernel(MaxLogitParams p) {
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h >= p.H) return;
  if (p.argmax) {
    const unsigned long long key = reinterpret_cast<unsigned long long*>(p.argmax)[h];
    const int32_t ord = (int32_t)((uint32_t)(key >> 32) ^ 0x80000000u);
    p.smax[h] = ordered_to_float(ord);
    p.argmax[h] = (long long)(0xffffffffu - (uint32_t)(key & 0xffffffffull));
  } else {
    const int32_t ord = reinterpret_cast<int32_t*>(p.smax)[h];
    p.smax[h] = ordered_to_float(ord);
  }
}

__device__ inline void publish(const MaxLogitParams& p, int h, float v, uint32_t idx) {
  if (p.argmax)
    atomicMax(reinterpret_cast<unsigned long long*>(p.argmax) + h, pack_key(v, idx));
  else
    atomicMax(reinterpret_cast<int32_t*>(p.smax) + h, float_to_ordered(v));
}

// ---------------------------------------------------------------- CUDA cores
// fp32 features (and any dtype while d exceeds the tensor-core tiles):
// 64 x 64 logit tiles, 256 threads, 4 x 4 logits per thread, features staged
// transposed in shared memory.
constexpr int kT = 64;

template <typename T>
__device__ inline float ldf(const T* p) { return (float)*p; }
template <>
__device__ inline float ldf<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

template <typename T>
__global__ void __launch_bounds__(256) ml_simt_kernel(const __grid_constant__ MaxLogitParams p) {
  extern __shared__ float sm[];
  const int D = p.d_head + p.d_shared;
  float* Qs = sm;                    // [D][kT + 1]
  float* Ks = sm + D * (kT + 1);     // [D][kT + 1]
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int nib = (p.S + kT - 1) / kT;
  const long long items = (long long)p.B * p.H * nib;
  const T* q = reinterpret_cast<const T*>(p.q);
  const T* k = reinterpret_cast<const T*>(p.k);
  const T* ks = reinterpret_cast<const T*>(p.ks);
  for (long long it = blockIdx.x; it < items; it += gridDim.x) {
    // heaviest (largest i-block) first under causal masking
    const int ib = nib - 1 - (int)(it % nib);
    const int h = (int)((it / nib) % p.H), b = (int)(it / ((long long)nib * p.H));
    const int i0 = ib * kT;
    for (int e = threadIdx.x; e < kT * D; e += blockDim.x) {
      const int r = e / D, d = e % D, i = i0 + r;
      Qs[d * (kT + 1) + r] =
          i < p.S ? ldf(q + b * p.qs[0] + (long long)i * p.qs[1] + (long long)h * p.qs[2] + d) : 0.f;
    }
    float best = -INFINITY;
    uint32_t best_idx = 0xffffffffu;
    bool bad = false;
    const int njb = p.causal ? ib + 1 : nib;
    for (int jb = 0; jb < njb; ++jb) {
      const int j0 = jb * kT;
      __syncthreads();
      for (int e = threadIdx.x; e < kT * D; e += blockDim.x) {
        const int r = e / D, d = e % D, j = j0 + r;
        float v = 0.f;
        if (j < p.S) {
          v = d < p.d_head
                  ? ldf(k + b * p.kst[0] + (long long)j * p.kst[1] + (long long)h * p.kst[2] + d)
                  : ldf(ks + b * p.kss[0] + (long long)j * p.kss[1] + (d - p.d_head));
        }
        Ks[d * (kT + 1) + r] = v;
      }
      __syncthreads();
      float acc[4][4] = {};
      for (int d = 0; d < D; ++d) {
        float a[4], c[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) a[x] = Qs[d * (kT + 1) + ty * 4 + x];
#pragma unroll
        for (int y = 0; y < 4; ++y) c[y] = Ks[d * (kT + 1) + tx * 4 + y];
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
          for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(a[x], c[y], acc[x][y]);
      }
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int i = i0 + ty * 4 + x;
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          const int j = j0 + tx * 4 + y;
          if (i >= p.S || j >= p.S || (p.causal && j > i)) continue;
          const float v = acc[x][y];
          bad |= !finite_f(v);
          const uint32_t idx = (uint32_t)(((long long)b * p.S + i) * p.S + j);
          if (v > best || (v == best && idx < best_idx)) { best = v; best_idx = idx; }
        }
      }
    }
    if (bad) set_status(p.status, MC_STATUS_NONFINITE_LOGIT);
    // block reduction of (best, best_idx)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_down_sync(0xffffffffu, best, o);
      const uint32_t oi = __shfl_down_sync(0xffffffffu, best_idx, o);
      if (ov > best || (ov == best && oi < best_idx)) { best = ov; best_idx = oi; }
    }
    __shared__ float rv[8];
    __shared__ uint32_t ri[8];
    __syncthreads();
    if ((threadIdx.x & 31) == 0) { rv[threadIdx.x >> 5] = best; ri[threadIdx.x >> 5] = best_idx; }
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int w = 1; w < 8; ++w)
        if (rv[w] > best || (rv[w] == best && ri[w] < best_idx)) { best = rv[w]; best_idx = ri[w]; }
      if (best > -INFINITY) publish(p, h, best * p.scale, best_idx);
    }
  }
}

}  // namespace

cudaError_t launch_max_logit(const MaxLogitParams& p, cudaStream_t s, char* err, size_t errlen) {
  const int hb = (p.H + 127) / 128;
  ml_init_kernel<<<hb, 128, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int D = p.d_head + p.d_shared;
  const size_t smem = 2 * (size_t)D * (kT + 1) * sizeof(float);
  const int nib = (p.S + kT - 1) / kT;
  const long long items = (long long)p.B * p.H * nib;
  const int grid = (int)(items < (long long)sm_count() * 4 ? items : sm_count() * 4);
  if (p.dtype == MC_BF16) {
    cudaFuncSetAttribute(ml_simt_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    ml_simt_kernel<__nv_bfloat16><<<grid, 256, smem, s>>>(p);
  } else {
    cudaFuncSetAttribute(ml_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    ml_simt_kernel<float><<<grid, 256, smem, s>>>(p);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ml_final_kernel<<<hb, 128, 0, s>>>(p);
  (void)err; (void)errlen;
  return cudaGetLastError();
}

}  // namespace mc
