// Setup (untimed): the query/key features of an attention layer on the
// library's own kernels, so that S_max and its re-measurement after a clip run
// entirely on the library.  [K2-internals] "MLA 的特殊处理": the query splits
// into a per-head part q^C and a rotary part q^R taken from the compressed
// query latent; the keys into k^C (per head, from the compressed key/value
// latent) and one rotary k^R shared by every head.  MHA: Q = X W_q^T,
// K = X W_k^T ([K2-notes] 3.2).
//
//   mc_matmul    D = A B^T: bf16 on the Newton-Schulz GEMM core (tcgen05 CTA
//                pairs, one bf16 plane, fp32 accumulation); fp32 on the
//                CUDA-core GEMM with compensated sums.
//   mc_rms_norm  y = x / sqrt(mean(x^2) + eps) per row (weightless RMSNorm of
//                the latents), fp32 arithmetic.
//   mc_rope      rotary embedding on interleaved pairs at positions 0..S-1,
//                angles s * theta^(-2k/d) and their cosines and sines in fp64.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "../../include/muonclip.h"
#include "common.cuh"
#include "kernels.h"

namespace mc {
namespace {

template <typename T>
__device__ inline float ldv(const T* p);
template <>
__device__ inline float ldv<float>(const float* p) { return *p; }
template <>
__device__ inline float ldv<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }
template <typename T>
__device__ inline void stv(T* p, float v);
template <>
__device__ inline void stv<float>(float* p, float v) { *p = v; }
template <>
__device__ inline void stv<__nv_bfloat16>(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// One warp per row: the mean of the squares over `cols` values in fp32, then
// every value divided by sqrt(mean + eps).  In place when y == x (each value
// is read and then written by the same lane).
template <typename T>
__global__ void rms_rows_kernel(const T* x, long long ldx, T* y, long long ldy, long long rows, int cols,
                                float eps) {
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
    const T* xr = x + r * ldx;
    T* yr = y + r * ldy;
    float s = 0.f;
    for (int c = lane; c < cols; c += 32) {
      const float v = ldv(xr + c);
      s = fmaf(v, v, s);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float inv = 1.f / sqrtf(s / (float)cols + eps);
    for (int c = lane; c < cols; c += 32) stv(yr + c, ldv(xr + c) * inv);
  }
}

// One (b, s) position per iteration of a block: the d/2 cosines and sines of
// position s go to shared memory (fp64 angle, rounded to fp32), then every
// head's pairs (x[2k], x[2k+1]) rotate by them, in place.
template <typename T>
__global__ void rope_kernel(T* x, int B, int S, int nh, int d, long long sb, long long ss, long long sh,
                            double theta) {
  extern __shared__ float cs[];          // [d/2] cosines, then [d/2] sines
  const int half = d / 2;
  const long long rows = (long long)B * S;
  for (long long row = blockIdx.x; row < rows; row += gridDim.x) {
    const int b = (int)(row / S), s = (int)(row % S);
    __syncthreads();
    for (int k = threadIdx.x; k < half; k += blockDim.x) {
      const double ang = (double)s * pow(theta, -2.0 * (double)k / (double)d);
      double sn, cn;
      sincos(ang, &sn, &cn);
      cs[k] = (float)cn;
      cs[half + k] = (float)sn;
    }
    __syncthreads();
    T* xr = x + (long long)b * sb + (long long)s * ss;
    for (int i = threadIdx.x; i < nh * half; i += blockDim.x) {
      const int h = i / half, k = i - h * half;
      T* p = xr + (long long)h * sh + 2 * k;
      const float x0 = ldv(p), x1 = ldv(p + 1), c = cs[k], sn = cs[half + k];
      stv(p, x0 * c - x1 * sn);
      stv(p + 1, x0 * sn + x1 * c);
    }
  }
}

mc_status err(mc_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  return record_error(s, buf);
}

mc_status done() { return record_error(MC_OK, ""); }

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t esize(int32_t dtype) { return dtype == MC_BF16 ? 2 : 4; }

}  // namespace
}  // namespace mc

using namespace mc;

extern "C" {

mc_status mc_matmul(const void* A, int64_t lda, const void* B, int64_t ldb, void* D, int64_t ldd,
                    int32_t M, int32_t N, int32_t K, int32_t dtype, void* scratch, int32_t* status,
                    mc_stream_t stream) {
  if (dtype != MC_BF16 && dtype != MC_F32) return err(MC_ERR_INVALID_ARG, "mc_matmul: dtype %d", dtype);
  if (M < 0 || N < 0 || K < 1) return err(MC_ERR_INVALID_ARG, "mc_matmul: M %d, N %d, K %d", M, N, K);
  if (M == 0 || N == 0) return done();
  if (!A || !B || !D) return err(MC_ERR_INVALID_ARG, "mc_matmul: null operand");
  if (lda < K || ldb < K || ldd < N) return err(MC_ERR_INVALID_ARG, "mc_matmul: pitch below the row length");
  const size_t es = esize(dtype);
  if (!al16(A) || !al16(B) || !al16(D) || (lda * es) % 16 || (ldb * es) % 16 || (ldd * es) % 16)
    return err(MC_ERR_INVALID_ARG, "mc_matmul: pointers and row pitches must be 16-byte aligned");
  if (dtype == MC_BF16 && (!scratch || !al16(scratch)))
    return err(MC_ERR_INVALID_ARG, "mc_matmul: bf16 needs a 16-byte aligned device scratch of >= 16 bytes");
  GemmParams gp;
  memset(&gp, 0, sizeof gp);
  gp.xmode = dtype == MC_BF16 ? kXBf16 : kXF32;
  gp.status = status;
  gp.ngroups = 1;
  gp.terms = 1;
  gp.fmt = kFmtBf16;
  gp.alpha = 1.f;
  GemmGroup& G = gp.g[0];
  G.M = M; G.N = N; G.K = K; G.batch = 1;
  G.a_hi = A; G.lda = lda; G.a_bstride = (long long)M * lda;
  G.b_hi = B; G.ldb = ldb; G.b_bstride = (long long)N * ldb;
  G.d_hi = D; G.ldd = ldd; G.d_bstride = (long long)M * ldd;
  const int tm = dtype == MC_BF16 ? kTcTileM : 64, tn = dtype == MC_BF16 ? kTcTileN : 64;
  G.tiles_m = (int)cdiv(M, tm);
  G.tiles_n = (int)cdiv(N, tn);
  G.tiles_per_item = G.tiles_m * G.tiles_n;
  gp.total_tiles = G.tiles_per_item;
  const cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e;
  if (dtype == MC_BF16) {
    e = cudaMemsetAsync(scratch, 0, sizeof(int), s);          // the launch's tile counter
    if (e != cudaSuccess) return err(MC_ERR_CUDA, "mc_matmul: %s", cudaGetErrorString(e));
    gp.sched = static_cast<int*>(scratch);
    char msg[256] = {0};
    e = launch_ns_gemm_tc(gp, nullptr, s, msg, sizeof msg);
    if (e != cudaSuccess && msg[0]) return err(MC_ERR_CUDA, "mc_matmul: tensor-core GEMM: %s", msg);
  } else {
    e = launch_ns_gemm_f32(gp, s);
  }
  if (e != cudaSuccess) return err(MC_ERR_CUDA, "mc_matmul: %s", cudaGetErrorString(e));
  return done();
}

mc_status mc_rms_norm(const void* x, int64_t ldx, void* y, int64_t ldy, int64_t rows, int32_t cols,
                      int32_t dtype, float eps, mc_stream_t stream) {
  if (dtype != MC_BF16 && dtype != MC_F32) return err(MC_ERR_INVALID_ARG, "mc_rms_norm: dtype %d", dtype);
  if (rows < 0 || cols < 1 || ldx < cols || ldy < cols)
    return err(MC_ERR_INVALID_ARG, "mc_rms_norm: rows %lld, cols %d, pitches %lld / %lld", (long long)rows,
               cols, (long long)ldx, (long long)ldy);
  if (!(eps >= 0.f)) return err(MC_ERR_INVALID_ARG, "mc_rms_norm: eps must be >= 0");
  if (rows == 0) return done();
  if (!x || !y) return err(MC_ERR_INVALID_ARG, "mc_rms_norm: null pointer");
  const int threads = 256, rows_per_block = threads / 32;
  const long long want = (rows + rows_per_block - 1) / rows_per_block;
  const int grid = (int)(want < (long long)sm_count() * 8 ? want : (long long)sm_count() * 8);
  const cudaStream_t s = (cudaStream_t)stream;
  if (dtype == MC_BF16)
    rms_rows_kernel<__nv_bfloat16><<<grid, threads, 0, s>>>(static_cast<const __nv_bfloat16*>(x), ldx,
                                                            static_cast<__nv_bfloat16*>(y), ldy, rows, cols, eps);
  else
    rms_rows_kernel<float><<<grid, threads, 0, s>>>(static_cast<const float*>(x), ldx, static_cast<float*>(y),
                                                    ldy, rows, cols, eps);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return err(MC_ERR_CUDA, "mc_rms_norm: %s", cudaGetErrorString(e));
  return done();
}

mc_status mc_rope(void* x, int32_t B, int32_t S, int32_t nh, int32_t d, int64_t sb, int64_t ss, int64_t sh,
                  int32_t dtype, double theta, mc_stream_t stream) {
  if (dtype != MC_BF16 && dtype != MC_F32) return err(MC_ERR_INVALID_ARG, "mc_rope: dtype %d", dtype);
  if (B < 0 || S < 0 || nh < 1 || d < 2 || (d & 1) || d > 4096)
    return err(MC_ERR_INVALID_ARG, "mc_rope: B %d, S %d, heads %d, d %d (d even, 2..4096)", B, S, nh, d);
  if (!(theta > 0.0)) return err(MC_ERR_INVALID_ARG, "mc_rope: theta must be > 0");
  if ((long long)B * S == 0) return done();
  if (!x) return err(MC_ERR_INVALID_ARG, "mc_rope: null pointer");
  const long long rows = (long long)B * S;
  const int grid = (int)(rows < (long long)sm_count() * 8 ? rows : (long long)sm_count() * 8);
  const size_t smem = (size_t)d * sizeof(float);
  const cudaStream_t s = (cudaStream_t)stream;
  if (dtype == MC_BF16)
    rope_kernel<__nv_bfloat16><<<grid, 256, smem, s>>>(static_cast<__nv_bfloat16*>(x), B, S, nh, d, sb, ss, sh,
                                                        theta);
  else
    rope_kernel<float><<<grid, 256, smem, s>>>(static_cast<float*>(x), B, S, nh, d, sb, ss, sh, theta);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return err(MC_ERR_CUDA, "mc_rope: %s", cudaGetErrorString(e));
  return done();
}

}  // extern "C"
