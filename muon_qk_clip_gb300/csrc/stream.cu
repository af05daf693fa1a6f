// HBM-streaming kernels of the MuonClip step:
//   prep   : M <- mu M + G (momentum, [K2-internals] Algorithm 1), the
//            oriented Newton-Schulz iterate X0 ~ M (split bf16 / bf16 / fp32)
//            and one sum of squares per 64x64 tile (for ||M||_F).
//   norms  : per-matrix 1/(||M||_F + eps) from the tile sums, fixed order.
//   apply  : W <- W - lr (s X + wd W) (decoupled decay, Algorithm 1) or
//            O <- s X for the standalone Newton-Schulz call.
//   clip   : per-head QK-Clip rescale of weight row segments
//            ([K2-internals] "核心数学", "MLA 的特殊处理").
#include "common.cuh"
#include "kernels.h"

namespace mc {

namespace {

constexpr int kTile = 64;
constexpr int kThreads = 256;

template <class Job>
__device__ inline int find_job(const Job* jobs, int njobs, int t) {
  int lo = 0, hi = njobs - 1;
  while (lo < hi) {  // last job with tile_begin <= t
    int mid = (lo + hi + 1) >> 1;
    if (jobs[mid].tile_begin <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ inline float load_elem(const void* base, long long idx, int bf16) {
  return bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx])
              : reinterpret_cast<const float*>(base)[idx];
}

// Write one iterate element x at (r, c) of the oriented planes.
template <int XM>
__device__ inline void store_x(void* xh, void* xl, long long idx, float x) {
  if (XM == kXSplit) {
    __nv_bfloat16 h, l;
    split_bf16(x, h, l);
    reinterpret_cast<__nv_bfloat16*>(xh)[idx] = h;
    reinterpret_cast<__nv_bfloat16*>(xl)[idx] = l;
  } else if (XM == kXBf16) {
    reinterpret_cast<__nv_bfloat16*>(xh)[idx] = __float2bfloat16_rn(x);
  } else {
    reinterpret_cast<float*>(xh)[idx] = x;
  }
}

template <int XM>
__device__ inline float load_x(const void* xh, const void* xl, long long idx) {
  if (XM == kXSplit)
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(xh)[idx]) +
           __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(xl)[idx]);
  if (XM == kXBf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(xh)[idx]);
  return reinterpret_cast<const float*>(xh)[idx];
}

// Four consecutive elements (16-byte aligned fp32 or 8-byte aligned bf16).
__device__ inline void load4(const void* base, long long idx, int bf16, float (&o)[4]) {
  if (bf16) {
    const uint2 u = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(base) + idx);
    const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = __bfloat162float(b[e]);
  } else {
    const float4 f = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + idx);
    o[0] = f.x; o[1] = f.y; o[2] = f.z; o[3] = f.w;
  }
}
__device__ inline void store4(void* base, long long idx, int bf16, const float (&v)[4]) {
  if (bf16) {
    uint2 u;
    __nv_bfloat16* b = reinterpret_cast<__nv_bfloat16*>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) b[e] = __float2bfloat16_rn(v[e]);
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(base) + idx) = u;
  } else {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + idx) = make_float4(v[0], v[1], v[2], v[3]);
  }
}
template <int XM>
__device__ inline void store_x4(void* xh, void* xl, long long idx, const float (&v)[4]) {
  if (XM == kXSplit) {
    uint2 uh, ul;
    __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(&uh);
    __nv_bfloat16* l = reinterpret_cast<__nv_bfloat16*>(&ul);
#pragma unroll
    for (int e = 0; e < 4; ++e) split_bf16(v[e], h[e], l[e]);
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(xh) + idx) = uh;
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(xl) + idx) = ul;
  } else if (XM == kXBf16) {
    store4(xh, idx, 1, v);
  } else {
    store4(xh, idx, 0, v);
  }
}
template <int XM>
__device__ inline void load_x4(const void* xh, const void* xl, long long idx, float (&o)[4]) {
  if (XM == kXSplit) {
    float h[4], l[4];
    load4(xh, idx, 1, h);
    load4(xl, idx, 1, l);
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = h[e] + l[e];
  } else {
    load4(xh, idx, XM == kXBf16, o);
  }
}

// Deterministic block sum (fixed shuffle tree, then fixed order over warps).
__device__ inline double block_sum(double v, double* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  double s = 0.0;
  if (threadIdx.x == 0)
    for (int i = 0; i < kThreads / 32; ++i) s += red[i];
  return s;
}

// Thread layout inside a 64x64 tile: 16 threads x 4 columns per row,
// 16 rows per pass, 4 passes.
template <int XM>
__global__ void __launch_bounds__(kThreads) prep_kernel(const __grid_constant__ PrepParams p) {
  __shared__ float tile[kTile][kTile + 1];
  __shared__ double red[kThreads / 32];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
    const PrepJob& jb = p.jobs[find_job(p.jobs, p.njobs, t)];
    const int lt = t - jb.tile_begin;
    const int r0 = (lt / jb.tiles_c) * kTile, c0 = (lt % jb.tiles_c) * kTile;
    float ss = 0.f;
    bool bad = false;
    const int cl0 = tx * 4, cbase = c0 + cl0;
    const bool vec = cbase + 3 < jb.cols;        // 4 in-range columns: one vector access
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int rl = ty + 16 * k, r = r0 + rl;
      float m[4] = {0.f, 0.f, 0.f, 0.f};
      if (r < jb.rows) {
        const long long im = (long long)r * jb.ldM + cbase;
        if (vec) {
          load4(jb.M, im, 0, m);
          if (p.do_momentum) {
            float g[4];
            load4(jb.G, (long long)r * jb.ldG + cbase, jb.g_bf16, g);
#pragma unroll
            for (int e = 0; e < 4; ++e) m[e] = fmaf(p.mu, m[e], g[e]);
            store4(jb.M, im, 0, m);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (cbase + e >= jb.cols) continue;
            m[e] = jb.M[im + e];
            if (p.do_momentum) {
              m[e] = fmaf(p.mu, m[e], load_elem(jb.G, (long long)r * jb.ldG + cbase + e, jb.g_bf16));
              jb.M[im + e] = m[e];
            }
          }
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        bad |= !finite_f(m[e]);
        ss = fmaf(m[e], m[e], ss);
        tile[rl][cl0 + e] = m[e];
      }
    }
    if (bad) set_status(p.status, MC_STATUS_NONFINITE_UPDATE);
    if (p.write_x) {
      if (!jb.transpose) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int rl = ty + 16 * k, r = r0 + rl;
          if (r >= jb.rows) continue;
          const long long ix = (long long)r * jb.ldx + cbase;
          if (vec) {
            float v[4] = {tile[rl][cl0], tile[rl][cl0 + 1], tile[rl][cl0 + 2], tile[rl][cl0 + 3]};
            store_x4<XM>(jb.xh, jb.xl, ix, v);
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (cbase + e < jb.cols) store_x<XM>(jb.xh, jb.xl, ix + e, tile[rl][cl0 + e]);
          }
        }
      } else {
        __syncthreads();
        // oriented row = original column, oriented column = original row
        const int rbase = r0 + tx * 4;
        const bool rvec = rbase + 3 < jb.rows;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int cl = ty + 16 * k, c = c0 + cl;
          if (c >= jb.cols) continue;
          const long long ix = (long long)c * jb.ldx + rbase;
          float v[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) v[e] = tile[tx * 4 + e][cl];
          if (rvec) {
            store_x4<XM>(jb.xh, jb.xl, ix, v);
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (rbase + e < jb.rows) store_x<XM>(jb.xh, jb.xl, ix + e, v[e]);
          }
        }
      }
    }
    if (p.partials) {
      const double s = block_sum((double)ss, red);
      if (threadIdx.x == 0) p.partials[t] = s;
    }
    __syncthreads();
  }
}

__global__ void norms_kernel(const __grid_constant__ NormParams p) {
  __shared__ double red[kThreads / 32];
  const int j = blockIdx.x;
  if (j >= p.nmat) return;
  double s = 0.0;
  const int b = p.begin[j], n = p.count[j];
  for (int i = threadIdx.x; i < n; i += blockDim.x) s += p.partials[b + i];
  s = block_sum(s, red);
  if (threadIdx.x == 0) {
    const double inv = 1.0 / (sqrt(s) + (double)p.eps);
    p.inv_norm[p.mat0 + j] = (float)inv;
    p.inv_norm_sq[p.mat0 + j] = (float)(inv * inv);
  }
}

template <int XM>
__global__ void __launch_bounds__(kThreads) apply_kernel(const __grid_constant__ ApplyParams p) {
  __shared__ float tile[kTile][kTile + 1];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
    const ApplyJob& jb = p.jobs[find_job(p.jobs, p.njobs, t)];
    const int lt = t - jb.tile_begin;
    const int r0 = (lt / jb.tiles_c) * kTile, c0 = (lt % jb.tiles_c) * kTile;
    const float s = jb.scale * (p.mat_scale ? p.mat_scale[jb.mat] : 1.f);
    const int cl0 = tx * 4, cbase = c0 + cl0;
    if (jb.transpose) {
      // stage X^T tile: oriented rows c0.., oriented cols r0..
      const int rbase = r0 + tx * 4;
      const bool rvec = rbase + 3 < jb.rows;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int cl = ty + 16 * k, c = c0 + cl;
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        if (c < jb.cols) {
          const long long ix = (long long)c * jb.ldx + rbase;
          if (rvec) {
            load_x4<XM>(jb.xh, jb.xl, ix, x);
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (rbase + e < jb.rows) x[e] = load_x<XM>(jb.xh, jb.xl, ix + e);
          }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) tile[tx * 4 + e][cl] = x[e];
      }
      __syncthreads();
    }
    bool bad = false;
    const bool vec = cbase + 3 < jb.cols;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int rl = ty + 16 * k, r = r0 + rl;
      if (r >= jb.rows) continue;
      float x[4];
      const long long ixo = (long long)r * jb.ldx + cbase;
      if (jb.transpose) {
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = tile[rl][cl0 + e];
      } else if (vec) {
        load_x4<XM>(jb.xh, jb.xl, ixo, x);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = cbase + e < jb.cols ? load_x<XM>(jb.xh, jb.xl, ixo + e) : 0.f;
      }
      const long long io = (long long)r * jb.ldo + cbase;
      float w[4] = {0.f, 0.f, 0.f, 0.f}, v[4];
      if (!p.write_o) {
        if (vec) {
          load4(jb.out, io, jb.out_bf16, w);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (cbase + e < jb.cols) w[e] = load_elem(jb.out, io + e, jb.out_bf16);
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float o = s * x[e];
        v[e] = p.write_o ? o : fmaf(-p.lr, fmaf(p.wd, w[e], o), w[e]);   // w - lr (o + wd w)
        bad |= !finite_f(v[e]) && (cbase + e < jb.cols);
      }
      if (vec) {
        store4(jb.out, io, jb.out_bf16, v);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (cbase + e >= jb.cols) continue;
          if (jb.out_bf16) reinterpret_cast<__nv_bfloat16*>(jb.out)[io + e] = __float2bfloat16_rn(v[e]);
          else reinterpret_cast<float*>(jb.out)[io + e] = v[e];
        }
      }
    }
    if (bad) set_status(p.status, MC_STATUS_NONFINITE_UPDATE);
    if (jb.transpose) __syncthreads();
  }
}

// ---------------------------------------------------------------- QK-Clip
__device__ inline float clip_power(float gamma, float e) {
  if (e == 0.5f) return sqrtf(gamma);
  if (e == 1.0f) return gamma;
  if (e == 0.0f) return 1.0f;
  return powf(gamma, e);
}

// Total mode: the layer's max S_max (NaN if any head's is NaN).
__device__ inline float total_smax(const ClipParams& p) {
  float mx = -INFINITY;
  bool nan = false;
  for (int h = 0; h < p.H; ++h) {
    const float s = p.smax[h];
    nan |= s != s;
    mx = fmaxf(mx, s);
  }
  return nan ? NAN : mx;
}

__global__ void clip_stats_kernel(const __grid_constant__ ClipParams p) {
  // one block: gamma_out, nclipped and the NaN flag
  __shared__ float s_total;
  if (p.total) {
    if (threadIdx.x == 0) s_total = total_smax(p);
    __syncthreads();
  }
  int local = 0;
  for (int h = threadIdx.x; h < p.H; h += blockDim.x) {
    const float sh = p.smax[h];
    const float s = p.total ? s_total : sh;
    const bool clip = s > p.tau;
    if (sh != sh) set_status(p.status, MC_STATUS_NONFINITE_SMAX);
    if (p.gamma_out) p.gamma_out[h] = clip ? p.tau / s : 1.f;
    local += clip;
  }
  if (p.nclipped) {
    __shared__ int cnt;
    if (threadIdx.x == 0) cnt = 0;
    __syncthreads();
    atomicAdd(&cnt, local);
    __syncthreads();
    if (threadIdx.x == 0) *p.nclipped = cnt;
  }
}

// grid.x over (segment, head) pairs, grid.y over row chunks of a head.
__global__ void __launch_bounds__(kThreads) clip_rows_kernel(const __grid_constant__ ClipParams p) {
  const int pair = blockIdx.x;
  const int seg = pair / p.H, h = pair % p.H;
  if (seg >= p.nsegs) return;
  __shared__ float s_blk;
  if (threadIdx.x == 0) s_blk = p.total ? total_smax(p) : p.smax[h];
  __syncthreads();
  const float s = s_blk;
  if (!(s > p.tau)) return;                       // untouched head (and NaN)
  const ClipSegDev& sg = p.segs[seg];
  const float f = clip_power(p.tau / s, sg.exponent);
  const long long row0 = sg.row_offset + (long long)h * sg.row_stride;
  for (long long rr = blockIdx.y; rr < sg.rows; rr += gridDim.y) {
    const long long base = (row0 + rr) * sg.ld;
    if (sg.bf16) {
      __nv_bfloat16* w = reinterpret_cast<__nv_bfloat16*>(sg.w) + base;
      const int nvec = sg.cols / 8;
      for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
        uint4 raw = reinterpret_cast<uint4*>(w)[v];
        __nv_bfloat16* e = reinterpret_cast<__nv_bfloat16*>(&raw);
#pragma unroll
        for (int i = 0; i < 8; ++i) e[i] = __float2bfloat16_rn(__bfloat162float(e[i]) * f);
        reinterpret_cast<uint4*>(w)[v] = raw;
      }
      for (int c = nvec * 8 + threadIdx.x; c < sg.cols; c += blockDim.x)
        w[c] = __float2bfloat16_rn(__bfloat162float(w[c]) * f);
    } else {
      float* w = reinterpret_cast<float*>(sg.w) + base;
      const int nvec = sg.cols / 4;
      for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
        float4 x = reinterpret_cast<float4*>(w)[v];
        x.x *= f; x.y *= f; x.z *= f; x.w *= f;
        reinterpret_cast<float4*>(w)[v] = x;
      }
      for (int c = nvec * 4 + threadIdx.x; c < sg.cols; c += blockDim.x) w[c] *= f;
    }
  }
}

int grid_for(int tiles) {
  const int cap = sm_count() * 8;
  return tiles < cap ? (tiles > 0 ? tiles : 1) : cap;
}

}  // namespace

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

cudaError_t launch_prep(const PrepParams& p, cudaStream_t s) {
  if (p.total_tiles <= 0) return cudaSuccess;
  const int g = grid_for(p.total_tiles);
  switch (p.xmode) {
    case kXSplit: prep_kernel<kXSplit><<<g, kThreads, 0, s>>>(p); break;
    case kXBf16: prep_kernel<kXBf16><<<g, kThreads, 0, s>>>(p); break;
    default: prep_kernel<kXF32><<<g, kThreads, 0, s>>>(p); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_norms(const double* partials, const int* tile_begin, const int* tile_count,
                         int nmat, float eps, float* inv_norm, float* inv_norm_sq,
                         cudaStream_t s) {
  for (int j0 = 0; j0 < nmat; j0 += kMaxNormMats) {
    NormParams p;  // passed by value as the kernel parameter block
    p.nmat = nmat - j0 < kMaxNormMats ? nmat - j0 : kMaxNormMats;
    p.mat0 = j0;
    for (int j = 0; j < p.nmat; ++j) { p.begin[j] = tile_begin[j0 + j]; p.count[j] = tile_count[j0 + j]; }
    p.eps = eps;
    p.partials = partials;
    p.inv_norm = inv_norm;
    p.inv_norm_sq = inv_norm_sq;
    norms_kernel<<<p.nmat, kThreads, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_apply(const ApplyParams& p, cudaStream_t s) {
  if (p.total_tiles <= 0) return cudaSuccess;
  const int g = grid_for(p.total_tiles);
  switch (p.xmode) {
    case kXSplit: apply_kernel<kXSplit><<<g, kThreads, 0, s>>>(p); break;
    case kXBf16: apply_kernel<kXBf16><<<g, kThreads, 0, s>>>(p); break;
    default: apply_kernel<kXF32><<<g, kThreads, 0, s>>>(p); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_clip(const ClipParams& p, cudaStream_t s) {
  if (p.gamma_out || p.nclipped || p.status) clip_stats_kernel<<<1, 256, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.nsegs <= 0 || p.H <= 0) return cudaSuccess;
  long long max_rows = 1;
  for (int i = 0; i < p.nsegs; ++i) max_rows = p.segs[i].rows > max_rows ? p.segs[i].rows : max_rows;
  dim3 grid(p.nsegs * p.H, (unsigned)(max_rows < 64 ? max_rows : 64));
  clip_rows_kernel<<<grid, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace mc
