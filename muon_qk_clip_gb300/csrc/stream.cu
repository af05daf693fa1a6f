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

// Four consecutive elements (16-byte aligned fp32 or 8-byte aligned bf16).
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

// Eight consecutive bf16 (16-byte aligned); elements past n (< 8 only at a
// matrix's edge) read as zero / are not written.
__device__ inline uint4 load8_bf16(const __nv_bfloat16* src, int n) {
  if (n >= 8) return *reinterpret_cast<const uint4*>(src);
  uint4 u = make_uint4(0u, 0u, 0u, 0u);
  __nv_bfloat16* e = reinterpret_cast<__nv_bfloat16*>(&u);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (i < n) e[i] = src[i];
  return u;
}
__device__ inline void store8_bf16(__nv_bfloat16* dst, const uint4& v, int n) {
  if (n >= 8) { *reinterpret_cast<uint4*>(dst) = v; return; }
  const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&v);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (i < n) dst[i] = e[i];
}

// Raw bits of up to four consecutive elements, unconverted, so that a tile's
// loads can all be in flight before the first one is used: 16-bit elements
// packed two per word in .x/.y, fp32 elements one per word; elements past
// n (< 4 only at a matrix's right edge) are zero bits.
__device__ inline uint4 raw_load4(const void* base, long long idx, int half, bool vec, int n) {
  uint4 u = make_uint4(0u, 0u, 0u, 0u);
  if (half) {
    const uint16_t* b = reinterpret_cast<const uint16_t*>(base) + idx;
    if (vec) {
      const uint2 v = *reinterpret_cast<const uint2*>(b);
      u.x = v.x; u.y = v.y;
    } else {
      uint32_t e[4] = {0u, 0u, 0u, 0u};
      for (int i = 0; i < n && i < 4; ++i) e[i] = b[i];
      u.x = e[0] | (e[1] << 16); u.y = e[2] | (e[3] << 16);
    }
  } else {
    const uint32_t* f = reinterpret_cast<const uint32_t*>(base) + idx;
    if (vec) {
      u = *reinterpret_cast<const uint4*>(f);
    } else {
      uint32_t e[4] = {0u, 0u, 0u, 0u};
      for (int i = 0; i < n && i < 4; ++i) e[i] = f[i];
      u = make_uint4(e[0], e[1], e[2], e[3]);
    }
  }
  return u;
}
// bf16 -> fp32 is exact: the 16 bits are the high half of the fp32 word.
__device__ inline void raw_cvt4(const uint4& u, int half, float (&o)[4]) {
  if (half) {
    o[0] = __uint_as_float(u.x << 16); o[1] = __uint_as_float(u.x & 0xffff0000u);
    o[2] = __uint_as_float(u.y << 16); o[3] = __uint_as_float(u.y & 0xffff0000u);
  } else {
    o[0] = __uint_as_float(u.x); o[1] = __uint_as_float(u.y);
    o[2] = __uint_as_float(u.z); o[3] = __uint_as_float(u.w);
  }
}
// Four fp16 values packed two per word in .x/.y.
__device__ inline void raw_cvt4_f16(const uint4& u, float (&o)[4]) {
  o[0] = from16<true>((uint16_t)(u.x & 0xffffu)); o[1] = from16<true>((uint16_t)(u.x >> 16));
  o[2] = from16<true>((uint16_t)(u.y & 0xffffu)); o[3] = from16<true>((uint16_t)(u.y >> 16));
}
// The iterate's value from the raw words of its plane(s); XF16: the split
// planes hold fp16 (else bf16).
template <int XM, bool XF16>
__device__ inline void raw_cvt_x4(const uint4& a, const uint4& b, float (&o)[4]) {
  if (XM == kXSplit && XF16) raw_cvt4_f16(a, o);
  else raw_cvt4(a, XM != kXF32, o);
  if (XM == kXSplit) {
    float l[4];
    if (XF16) raw_cvt4_f16(b, l);
    else raw_cvt4(b, 1, l);
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] += l[e];
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
// 16 rows per pass, 4 passes.  Every load of a tile is issued before its
// first store (the stores to M could alias the next rows' loads as far as
// the compiler knows, which would leave one row's loads in flight at a
// time).  partials[tile] is the fp64 sum of squares of the tile: a fixed
// shuffle tree per warp, then the 8 warp sums in warp order (double-buffered
// by tile parity, so one barrier per tile suffices).
template <int XM>
__global__ void __launch_bounds__(kThreads) prep_kernel(const __grid_constant__ PrepParams p) {
  __shared__ float tile[kTile][kTile + 1];
  __shared__ double red[2][kThreads / 32];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  int parity = 0;
  for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x, parity ^= 1) {
    const PrepJob& jb = p.jobs[find_job(p.jobs, p.njobs, t)];
    const int lt = t - jb.tile_begin;
    const int r0 = (lt / jb.tiles_c) * kTile, c0 = (lt % jb.tiles_c) * kTile;
    const int cl0 = tx * 4, cbase = c0 + cl0;
    const bool vec = cbase + 3 < jb.cols;        // 4 in-range columns: one vector access
    const int nc = jb.cols - cbase;               // valid columns of this thread (may be <= 0)
    float m[4][4];
    uint4 gr[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int r = r0 + ty + 16 * k;
      gr[k] = make_uint4(0u, 0u, 0u, 0u);
      const uint4 mr = r < jb.rows ? raw_load4(jb.M, (long long)r * jb.ldM + cbase, 0, vec, nc)
                                   : make_uint4(0u, 0u, 0u, 0u);
      m[k][0] = __uint_as_float(mr.x); m[k][1] = __uint_as_float(mr.y);
      m[k][2] = __uint_as_float(mr.z); m[k][3] = __uint_as_float(mr.w);
      if (p.do_momentum && r < jb.rows)
        gr[k] = raw_load4(jb.G, (long long)r * jb.ldG + cbase, jb.g_bf16, vec, nc);
    }
    float ss = 0.f;
    bool bad = false;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int rl = ty + 16 * k, r = r0 + rl;
      if (p.do_momentum) {
        float g[4];
        raw_cvt4(gr[k], jb.g_bf16, g);
#pragma unroll
        for (int e = 0; e < 4; ++e) m[k][e] = fmaf(p.mu, m[k][e], g[e]);
        if (r < jb.rows) {
          const long long im = (long long)r * jb.ldM + cbase;
          if (vec) {
            store4(jb.M, im, 0, m[k]);
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (cbase + e < jb.cols) jb.M[im + e] = m[k][e];
          }
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        bad |= !finite_f(m[k][e]);
        ss = fmaf(m[k][e], m[k][e], ss);
      }
      if (!p.write_x || r >= jb.rows) continue;
      if (jb.transpose) {
#pragma unroll
        for (int e = 0; e < 4; ++e) tile[rl][cl0 + e] = m[k][e];
      } else {
        const long long ix = (long long)r * jb.ldx + cbase;
        if (vec) {
          store_x4<XM>(jb.xh, jb.xl, ix, m[k]);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (cbase + e < jb.cols) store_x<XM>(jb.xh, jb.xl, ix + e, m[k][e]);
        }
      }
    }
    if (bad) set_status(p.status, MC_STATUS_NONFINITE_UPDATE);
    if (p.write_x && jb.transpose) {
      __syncthreads();
      // oriented row = original column, oriented column = original row
      // (rows of the tile past jb.rows were never written and are not read)
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
      __syncthreads();
    }
    if (p.partials) {
      double v = ss;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
      if ((threadIdx.x & 31) == 0) red[parity][threadIdx.x >> 5] = v;
      __syncthreads();
      if (threadIdx.x == 0) {
        double sum = 0.0;
        for (int i = 0; i < kThreads / 32; ++i) sum += red[parity][i];
        p.partials[t] = sum;
      }
    }
  }
}

__global__ void norms_kernel(const __grid_constant__ NormParams p) {
  __shared__ double red[kThreads / 32];
  const int j = blockIdx.x;
  if (j >= p.nmat) return;
  // eight independent accumulators per thread (their loads overlap), folded
  // in a fixed order
  double acc[8] = {0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0};
  const int b = p.begin[j], n = p.count[j];
  for (int i0 = threadIdx.x; i0 < n; i0 += 8 * kThreads) {
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (i0 + u * kThreads < n) acc[u] += p.partials[b + i0 + u * kThreads];
  }
  double s = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
  s = block_sum(s, red);
  if (threadIdx.x == 0) {
    const double inv = 1.0 / (sqrt(s) + (double)p.eps);
    p.inv_norm[p.mat0 + j] = (float)inv;
    p.inv_norm_sq[p.mat0 + j] = (float)(inv * inv);
  }
}

// Same tile layout as prep_kernel (the step's split-iterate / bf16-W case
// takes 16-byte accesses instead); every load of a tile is issued before the
// first store of W.  XF16: the split iterate's planes hold fp16 (after at
// least one Newton-Schulz iteration), else bf16.
template <int XM, bool XF16>
__global__ void __launch_bounds__(kThreads) apply_kernel(const __grid_constant__ ApplyParams p) {
  __shared__ float tile[kTile][kTile + 1];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
    const ApplyJob& jb = p.jobs[find_job(p.jobs, p.njobs, t)];
    const int lt = t - jb.tile_begin;
    const int r0 = (lt / jb.tiles_c) * kTile, c0 = (lt % jb.tiles_c) * kTile;
    const float s = jb.scale * (p.mat_scale ? p.mat_scale[jb.mat] : 1.f);
    if (XM == kXSplit && !p.write_o && jb.out_bf16) {
      // the step's own case (split iterate, bf16 W): 16-byte accesses, 8
      // threads x 8 columns per row, 32 rows per pass, two passes
      const int tx8 = threadIdx.x & 7, ty8 = threadIdx.x >> 3;
      const int cb = c0 + tx8 * 8, nc8 = jb.cols - cb;
      uint4 wv[2], xh[2], xl[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int r = r0 + ty8 + 32 * k;
        wv[k] = make_uint4(0u, 0u, 0u, 0u);
        if (r < jb.rows) wv[k] = load8_bf16(reinterpret_cast<const __nv_bfloat16*>(jb.out) + (long long)r * jb.ldo + cb, nc8);
      }
      if (jb.transpose) {
        // X^T: oriented row c (a column of W) holds W rows rb .. rb + 7
        const int rb = r0 + tx8 * 8, nr8 = jb.rows - rb;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int c = c0 + ty8 + 32 * k;
          xh[k] = xl[k] = make_uint4(0u, 0u, 0u, 0u);
          if (c >= jb.cols) continue;
          const long long ix = (long long)c * jb.ldx + rb;
          xh[k] = load8_bf16(reinterpret_cast<const __nv_bfloat16*>(jb.xh) + ix, nr8);
          xl[k] = load8_bf16(reinterpret_cast<const __nv_bfloat16*>(jb.xl) + ix, nr8);
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const uint16_t* a = reinterpret_cast<const uint16_t*>(&xh[k]);
          const uint16_t* b2 = reinterpret_cast<const uint16_t*>(&xl[k]);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            tile[tx8 * 8 + e][ty8 + 32 * k] = from16<XF16>(a[e]) + from16<XF16>(b2[e]);
        }
        __syncthreads();
      } else {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int r = r0 + ty8 + 32 * k;
          xh[k] = xl[k] = make_uint4(0u, 0u, 0u, 0u);
          if (r >= jb.rows) continue;
          const long long ix = (long long)r * jb.ldx + cb;
          xh[k] = load8_bf16(reinterpret_cast<const __nv_bfloat16*>(jb.xh) + ix, nc8);
          xl[k] = load8_bf16(reinterpret_cast<const __nv_bfloat16*>(jb.xl) + ix, nc8);
        }
      }
      bool bad8 = false;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int rl = ty8 + 32 * k, r = r0 + rl;
        if (r >= jb.rows) continue;
        const uint16_t* a = reinterpret_cast<const uint16_t*>(&xh[k]);
        const uint16_t* b2 = reinterpret_cast<const uint16_t*>(&xl[k]);
        const __nv_bfloat16* w8 = reinterpret_cast<const __nv_bfloat16*>(&wv[k]);
        uint4 outv;
        __nv_bfloat16* o8 = reinterpret_cast<__nv_bfloat16*>(&outv);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float x = jb.transpose ? tile[rl][tx8 * 8 + e]
                                       : from16<XF16>(a[e]) + from16<XF16>(b2[e]);
          const float w = __bfloat162float(w8[e]);
          const float v = fmaf(-p.lr, fmaf(p.wd, w, s * x), w);   // w - lr (s x + wd w)
          bad8 |= !finite_f(v) && (e < nc8);
          o8[e] = __float2bfloat16_rn(v);
        }
        store8_bf16(reinterpret_cast<__nv_bfloat16*>(jb.out) + (long long)r * jb.ldo + cb, outv, nc8);
      }
      if (bad8) set_status(p.status, MC_STATUS_NONFINITE_UPDATE);
      if (jb.transpose) __syncthreads();
      continue;
    }
    const int cl0 = tx * 4, cbase = c0 + cl0;
    if (jb.transpose) {
      // stage X^T tile: oriented rows c0.., oriented cols r0..
      const int rbase = r0 + tx * 4;
      const bool rvec = rbase + 3 < jb.rows;
      const int nr = jb.rows - rbase;
      uint4 xa[4], xb[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int c = c0 + ty + 16 * k;
        xa[k] = xb[k] = make_uint4(0u, 0u, 0u, 0u);
        if (c >= jb.cols) continue;
        const long long ix = (long long)c * jb.ldx + rbase;
        xa[k] = raw_load4(jb.xh, ix, XM != kXF32, rvec, nr);
        if (XM == kXSplit) xb[k] = raw_load4(jb.xl, ix, 1, rvec, nr);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float x[4];
        raw_cvt_x4<XM, XF16>(xa[k], xb[k], x);
#pragma unroll
        for (int e = 0; e < 4; ++e) tile[tx * 4 + e][ty + 16 * k] = x[e];
      }
      __syncthreads();
    }
    const bool vec = cbase + 3 < jb.cols;
    const int nc = jb.cols - cbase;
    uint4 xa[4], xb[4], wr[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int r = r0 + ty + 16 * k;
      xa[k] = xb[k] = wr[k] = make_uint4(0u, 0u, 0u, 0u);
      if (r >= jb.rows) continue;
      if (!jb.transpose) {
        const long long ixo = (long long)r * jb.ldx + cbase;
        xa[k] = raw_load4(jb.xh, ixo, XM != kXF32, vec, nc);
        if (XM == kXSplit) xb[k] = raw_load4(jb.xl, ixo, 1, vec, nc);
      }
      if (!p.write_o) wr[k] = raw_load4(jb.out, (long long)r * jb.ldo + cbase, jb.out_bf16, vec, nc);
    }
    bool bad = false;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int r = r0 + ty + 16 * k;
      if (r >= jb.rows) continue;
      float x[4], w[4], v[4];
      if (jb.transpose) {
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = tile[ty + 16 * k][cl0 + e];
      } else {
        raw_cvt_x4<XM, XF16>(xa[k], xb[k], x);
      }
      raw_cvt4(wr[k], jb.out_bf16, w);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float o = s * x[e];
        v[e] = p.write_o ? o : fmaf(-p.lr, fmaf(p.wd, w[e], o), w[e]);   // w - lr (o + wd w)
        bad |= !finite_f(v[e]) && (cbase + e < jb.cols);
      }
      const long long io = (long long)r * jb.ldo + cbase;
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

// gamma_out, nclipped and the NaN flag, computed by one whole block
__device__ void clip_stats(const ClipParams& p) {
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

// grid.x over (segment, head) pairs, grid.y over chunks of a head's rows.
constexpr int kClipUnroll = 8;
__global__ void __launch_bounds__(kThreads) clip_rows_kernel(const __grid_constant__ ClipParams p) {
  if (blockIdx.x == 0 && blockIdx.y == 0 && (p.gamma_out || p.nclipped || p.status)) clip_stats(p);
  const int pair = blockIdx.x;
  const int seg = pair / p.H, h = pair % p.H;
  if (seg >= p.nsegs) return;
  float s;
  if (p.total) {
    __shared__ float s_blk;
    if (threadIdx.x == 0) s_blk = total_smax(p);
    __syncthreads();
    s = s_blk;
  } else {
    s = p.smax[h];                                // one broadcast load, no barrier
  }
  if (!(s > p.tau)) return;                       // untouched head (and NaN)
  const ClipSegDev& sg = p.segs[seg];
  const float f = clip_power(p.tau / s, sg.exponent);
  const long long row0 = sg.row_offset + (long long)h * sg.row_stride;
  const int per_vec = sg.bf16 ? 8 : 4;
  if (sg.ld == sg.cols && (sg.rows * (long long)sg.cols) % per_vec == 0) {
    // the head's rows are one contiguous range: stride over its 16-byte
    // vectors, kClipUnroll loads in flight per thread
    const long long nvec = sg.rows * (long long)sg.cols / per_vec;
    uint4* w = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(sg.w) +
                                        row0 * sg.ld * (sg.bf16 ? 2 : 4));
    const long long step = (long long)gridDim.y * blockDim.x;
    for (long long v0 = (long long)blockIdx.y * blockDim.x + threadIdx.x; v0 < nvec;
         v0 += kClipUnroll * step) {
      uint4 raw[kClipUnroll];
#pragma unroll
      for (int u = 0; u < kClipUnroll; ++u)
        if (v0 + u * step < nvec) raw[u] = w[v0 + u * step];
#pragma unroll
      for (int u = 0; u < kClipUnroll; ++u) {
        if (v0 + u * step >= nvec) continue;
        if (sg.bf16) {
          __nv_bfloat16* e = reinterpret_cast<__nv_bfloat16*>(&raw[u]);
#pragma unroll
          for (int i = 0; i < 8; ++i) e[i] = __float2bfloat16_rn(__bfloat162float(e[i]) * f);
        } else {
          float* e = reinterpret_cast<float*>(&raw[u]);
#pragma unroll
          for (int i = 0; i < 4; ++i) e[i] *= f;
        }
        w[v0 + u * step] = raw[u];
      }
    }
    return;
  }
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

// Grid of a tile-loop kernel: every block resident at once (blocks per SM
// from the kernel's own occupancy), so the tiles split evenly over one wave.
template <class Kernel>
int grid_for(Kernel kernel, int tiles) {
  static const int per_sm = [&] {
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, kThreads, 0) != cudaSuccess) {
      (void)cudaGetLastError();
      nb = 0;
    }
    return nb > 0 ? nb : 4;
  }();
  const int cap = sm_count() * per_sm;
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
  switch (p.xmode) {
    case kXSplit: prep_kernel<kXSplit><<<grid_for(prep_kernel<kXSplit>, p.total_tiles), kThreads, 0, s>>>(p); break;
    case kXBf16: prep_kernel<kXBf16><<<grid_for(prep_kernel<kXBf16>, p.total_tiles), kThreads, 0, s>>>(p); break;
    default: prep_kernel<kXF32><<<grid_for(prep_kernel<kXF32>, p.total_tiles), kThreads, 0, s>>>(p); break;
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
  switch (p.xmode) {
    case kXSplit:
      if (p.x_f16)
        apply_kernel<kXSplit, true><<<grid_for(apply_kernel<kXSplit, true>, p.total_tiles), kThreads, 0, s>>>(p);
      else
        apply_kernel<kXSplit, false><<<grid_for(apply_kernel<kXSplit, false>, p.total_tiles), kThreads, 0, s>>>(p);
      break;
    case kXBf16: apply_kernel<kXBf16, false><<<grid_for(apply_kernel<kXBf16, false>, p.total_tiles), kThreads, 0, s>>>(p); break;
    default: apply_kernel<kXF32, false><<<grid_for(apply_kernel<kXF32, false>, p.total_tiles), kThreads, 0, s>>>(p); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_clip(const ClipParams& p, cudaStream_t s) {
  // one launch: block (0, 0) also writes the statistics
  const bool stats = p.gamma_out || p.nclipped || p.status;
  if (p.H <= 0 || (p.nsegs <= 0 && !stats)) return cudaSuccess;
  // chunks per head: about kClipUnroll 16-byte vectors per thread for a
  // contiguous head block, a row per chunk (up to 64) otherwise
  long long chunks = 1;
  for (int i = 0; i < p.nsegs; ++i) {
    const ClipSegDev& sg = p.segs[i];
    const int per_vec = sg.bf16 ? 8 : 4;
    const long long want = sg.ld == sg.cols && (sg.rows * (long long)sg.cols) % per_vec == 0
                               ? cdiv(sg.rows * (long long)sg.cols / per_vec, (long long)kThreads * kClipUnroll)
                               : sg.rows;
    chunks = want > chunks ? want : chunks;
  }
  const int pairs = p.nsegs > 0 ? p.nsegs * p.H : 1;
  dim3 grid(pairs, (unsigned)(chunks < 64 ? chunks : 64));
  clip_rows_kernel<<<grid, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace mc
