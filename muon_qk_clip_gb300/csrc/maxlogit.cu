// Per-head max attention logit ([K2-internals] "核心数学"):
//   S_max^h = scale * max_b max_{i, j <= i} q_{b,i,h} . k_{b,j,h}
// Flash-style tiling: the S x S logit matrix is never stored; each CTA keeps
// running maxima in registers and publishes one packed atomicMax per head.
//
// Results travel through the caller's output buffers:
//   argmax == null : smax[h] holds the float maximum throughout: a
//                    non-negative value (sign bit clear) is max-combined as a
//                    signed int, a negative one min-combined as an unsigned
//                    int, which orders all non-NaN floats as float max does
//                    (-0 below +0); initialised to -inf unless accumulating
//   argmax != null : argmax[h] holds a packed 64-bit key
//                    (ordered value << 32 | (0xffffffff - flat index)) so one
//                    atomicMax keeps the largest value and, among equal
//                    values, the smallest flat index (b*S + i)*S + j.
#include <stdio.h>
#include <string.h>

#include "common.cuh"
#include "fastdiv.cuh"
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
  if (p.argmax)
    reinterpret_cast<unsigned long long*>(p.argmax)[h] = 0ull;
  else if (!p.accumulate)
    p.smax[h] = -INFINITY;
}

__global__ void ml_final_kernel(MaxLogitParams p) {
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h >= p.H) return;
  const unsigned long long key = reinterpret_cast<unsigned long long*>(p.argmax)[h];
  const int32_t ord = (int32_t)((uint32_t)(key >> 32) ^ 0x80000000u);
  p.smax[h] = ordered_to_float(ord);
  p.argmax[h] = (long long)(0xffffffffu - (uint32_t)(key & 0xffffffffull));
}

__device__ inline void publish(const MaxLogitParams& p, int h, float v, uint32_t idx) {
  if (p.argmax)
    atomicMax(reinterpret_cast<unsigned long long*>(p.argmax) + h, pack_key(v, idx));
  else if (__float_as_int(v) >= 0)
    atomicMax(reinterpret_cast<int*>(p.smax) + h, __float_as_int(v));
  else
    atomicMin(reinterpret_cast<unsigned int*>(p.smax) + h, __float_as_uint(v));
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


// ---------------------------------------------------------------- tensor cores
// bf16 features, q.k length in 64-wide chunks.  One work item = (b, h, 128
// query rows), in the order of next_item; its Q chunks are loaded once
// (double-buffered across items) and 256-row key blocks stream through a ring
// of 64-feature chunk stages.  For MLA the key chunks come first from the
// head's k^C, then from the shared k^R.  Each key block is one 128 x 256 x d
// product accumulated in TMEM (double buffered); 8 epilogue warps take running
// row maxima straight out of TMEM.
// With a few 128 x 256 x 16 MMAs per stage the single issuing thread is on the
// critical path, so its loop does no division (ring counters, multiply-shift
// item decoding) and builds each stage's two descriptors once.
namespace tcml {

constexpr int BM = 128, BN = 256;
constexpr int kNBuf = 512 / BN;          // TMEM accumulators (512 columns)
constexpr int kCols = BN / 2;            // columns per epilogue warp
constexpr int kThreads = 320;            // producer, MMA, 8 epilogue warps
constexpr int Q_CHUNK = BM * 64 * 2;     // 16 KB
constexpr int K_CHUNK = BN * 64 * 2;     // 32 KB
constexpr int kMaxStages = 6;
constexpr uint32_t kTmemCols = 512;

struct Maps {
  CUtensorMap q, k, ks;
};

struct Geo {
  int nch, nck;        // chunks of q.k and of the head-specific key part
  int stages;
  int nqb;             // query blocks per (b, h)
  int nunit;           // work units per (b, h) (pairs of query blocks when causal)
  uint32_t units;       // below 2^30 (checked on the host)
  FastDiv div_nunit, div_h, div_bh;   // by nunit, H and B H
  int snake;           // 1: items heaviest first, dealt to the CTAs in snake order
  uint32_t items;      // B H nqb (snake order)
};


// 3-input minimum that returns NaN when any input is NaN
__device__ inline float min3_nan(float a, float b, float c) {
  float r;
  asm("min.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ inline float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Causal: a unit pairs query blocks ib and nqb - 1 - ib of one (b, h) (equal
// work), numbered (b, h)-major so the CTAs in flight share a few heads' keys in
// L2; without the mask a unit is one block.  Iteration n of a CTA is half
// n & 1 of its (n >> 1)-th unit: 1 with coordinates, 0 for the missing half of
// an unpaired middle block, -1 when the CTA has no units left.
__device__ inline int next_item(const MaxLogitParams& p, const Geo& g, uint32_t n, int& b, int& h,
                                int& ib) {
  if (g.snake) {
    // item k = (b h, query block): blocks in decreasing order of work (the
    // query block from the last down), every head within a block; round n
    // deals G consecutive items to the G CTAs, alternately forward and back,
    // so every CTA's total stays within one item of the others'
    const uint32_t G = gridDim.x;
    const uint32_t k = n * G + ((n & 1) ? G - 1 - blockIdx.x : blockIdx.x);
    if (k >= g.items) return -1;
    const uint32_t q = fastdiv(k, g.div_bh);
    const uint32_t bh = k - q * (uint32_t)(p.B * p.H);
    ib = g.nqb - 1 - (int)q;
    b = (int)fastdiv(bh, g.div_h);
    h = (int)(bh - (uint32_t)b * (uint32_t)p.H);
    return 1;
  }
  // divisions by run-time values as multiply-shifts (fastdiv.cuh)
  const uint32_t u = blockIdx.x + (n >> 1) * gridDim.x;
  if (u >= g.units) return -1;
  const uint32_t bh = fastdiv(u, g.div_nunit);
  const int pu = (int)(u - bh * (uint32_t)g.nunit);
  b = (int)fastdiv(bh, g.div_h);
  h = (int)(bh - (uint32_t)b * (uint32_t)p.H);
  if (!p.causal) {
    ib = pu;
    return (n & 1) ? 0 : 1;
  }
  if ((n & 1) == 0) { ib = g.nqb - 1 - pu; return 1; }
  ib = pu;
  return pu < g.nqb - 1 - pu ? 1 : 0;
}

__device__ inline int kblocks(const MaxLogitParams& p, int ib) {
  const int hi = p.causal ? min(p.S, (ib + 1) * BM) : p.S;
  return (hi + BN - 1) / BN;
}

template <bool ARG>
__global__ void __launch_bounds__(kThreads, 1)
    ml_tc_kernel(const __grid_constant__ MaxLogitParams p, const __grid_constant__ Maps mp,
                 const Geo g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* qbuf = smem;                                   // [2][nch] x 16 KB
  uint8_t* kbuf = smem + 2 * g.nch * Q_CHUNK;             // [stages] x 32 KB
  uint64_t* bars = reinterpret_cast<uint64_t*>(kbuf + g.stages * K_CHUNK);
  uint64_t* q_full = bars;            // [2]
  uint64_t* q_empty = bars + 2;       // [2]
  uint64_t* t_full = bars + 4;        // [kNBuf]
  uint64_t* t_empty = t_full + kNBuf; // [kNBuf]
  uint64_t* drain = t_empty + kNBuf;  // [1]
  uint64_t* k_full = drain + 1;       // [stages]
  uint64_t* k_empty = k_full + kMaxStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(k_empty + kMaxStages);
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < 2; ++i) { mbar_init(&q_full[i], 1); mbar_init(&q_empty[i], 1); }
    for (int i = 0; i < kNBuf; ++i) { mbar_init(&t_full[i], 1); mbar_init(&t_empty[i], 8); }
    mbar_init(drain, 1);
    for (int s = 0; s < g.stages; ++s) { mbar_init(&k_full[s], 1); mbar_init(&k_empty[s], 1); }
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&mp.q); prefetch_tmap(&mp.k);
    if (g.nch > g.nck) prefetch_tmap(&mp.ks);
  }
  if (warp == 1) { tmem_alloc(tmem_slot, kTmemCols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  auto fail = [&]() { abort_flag = 1; set_status(p.status, MC_STATUS_TIMEOUT); };

  if (warp == 0) {
    if (lane == 0) {
      uint32_t ks = 0, kph = 0, li = 0;     // next key stage and its use parity
      bool used_q[2] = {false, false}, used_k[kMaxStages] = {};
      uint32_t par_q[2] = {0, 0}, par_k[kMaxStages] = {};
      for (uint32_t n = 0; !abort_flag; ++n) {
        int b, h, ib;
        const int st = next_item(p, g, n, b, h, ib);
        if (st < 0) break;
        if (st == 0) continue;
        const int qb = li & 1;
        if (!mbar_wait(&q_empty[qb], ((li >> 1) & 1) ^ 1, &abort_flag)) { fail(); break; }
        mbar_arrive_expect_tx(&q_full[qb], g.nch * Q_CHUNK);
        for (int c = 0; c < g.nch; ++c)
          tma_load_4d(qbuf + (qb * g.nch + c) * Q_CHUNK, &mp.q, &q_full[qb], 64 * c, h, ib * BM, b);
        used_q[qb] = true; par_q[qb] = (li >> 1) & 1;
        const int nkb = kblocks(p, ib);
        bool ok = true;
        for (int kb = 0; kb < nkb && ok; ++kb) {
          for (int c = 0; c < g.nch; ++c) {
            const int s = (int)ks;
            if (!mbar_wait(&k_empty[s], kph ^ 1, &abort_flag)) { fail(); ok = false; break; }
            mbar_arrive_expect_tx(&k_full[s], K_CHUNK);
            if (c < g.nck)
              tma_load_4d(kbuf + s * K_CHUNK, &mp.k, &k_full[s], 64 * c, h, kb * BN, b);
            else
              tma_load_3d(kbuf + s * K_CHUNK, &mp.ks, &k_full[s], 64 * (c - g.nck), kb * BN, b);
            used_k[s] = true; par_k[s] = kph;
            if (++ks == (uint32_t)g.stages) { ks = 0; kph ^= 1; }
          }
        }
        if (!ok) break;
        ++li;
      }
      for (int i = 0; i < 2; ++i) if (used_q[i]) mbar_wait(&q_full[i], par_q[i], nullptr);
      for (int s = 0; s < g.stages; ++s) if (used_k[s]) mbar_wait(&k_full[s], par_k[s], nullptr);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc_bf16(BM, BN, 0, 0);
      uint32_t ks = 0, kph = 0, li = 0, tcount = 0;   // key stage ring as in the producer
      bool issued = false;
      for (uint32_t n = 0; !abort_flag; ++n) {
        int b, h, ib;
        const int st = next_item(p, g, n, b, h, ib);
        if (st < 0) break;
        if (st == 0) continue;
        const int qb = li & 1;
        if (!mbar_wait(&q_full[qb], (li >> 1) & 1, &abort_flag)) { fail(); break; }
        const int nkb = kblocks(p, ib);
        bool ok = true;
        for (int kb = 0; kb < nkb && ok; ++kb, ++tcount) {
          const int acc = tcount % kNBuf;
          if (!mbar_wait(&t_empty[acc], ((tcount / kNBuf) & 1) ^ 1, &abort_flag)) { fail(); ok = false; break; }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * BN;
          for (int c = 0; c < g.nch; ++c) {
            const int s = (int)ks;
            if (!mbar_wait(&k_full[s], kph, &abort_flag)) { fail(); ok = false; break; }
            tc_fence_after();
            const uint64_t qd = make_sdesc_sw128(smem_u32(qbuf + (qb * g.nch + c) * Q_CHUNK), 16, 1024);
            const uint64_t kd = make_sdesc_sw128(smem_u32(kbuf + s * K_CHUNK), 16, 1024);
            tc_mma(d_tmem, qd, kd, idesc, c > 0 ? 1u : 0u);
#pragma unroll
            for (int kk = 1; kk < 4; ++kk) tc_mma(d_tmem, qd + 2 * kk, kd + 2 * kk, idesc, 1u);
            issued = true;
            tc_commit(&k_empty[s]);
            if (++ks == (uint32_t)g.stages) { ks = 0; kph ^= 1; }
          }
          if (ok) tc_commit(&t_full[acc]);
        }
        if (!ok) break;
        tc_commit(&q_empty[qb]);
        ++li;
      }
      if (issued) { tc_commit(drain); mbar_wait(drain, 0, nullptr); }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int e = warp - 2;              // 0..7
    const int q = warp & 3;              // TMEM lane quadrant
    const int half = e >> 2;             // columns [half*kCols, half*kCols + kCols)
    uint32_t tcount = 0;
    for (uint32_t n = 0;; ++n) {
      int b, h, ib;
      const int st = next_item(p, g, n, b, h, ib);
      if (st < 0) break;
      if (st == 0) continue;
      const int nkb = kblocks(p, ib);
      const int i = ib * BM + q * 32 + lane;          // this thread's query row
      const int i_lo = ib * BM + q * 32;              // warp's first row
      float best = -INFINITY;
      uint32_t bidx = 0xffffffffu;
      float lo4[4] = {INFINITY, INFINITY, INFINITY, INFINITY};
      int failed = 0;                    // warp-uniform
      for (int kb = 0; kb < nkb; ++kb, ++tcount) {
        if (failed) continue;            // every later wait would fail too
        const int acc = tcount % kNBuf;
        int w = 1;
        if (lane == 0) w = mbar_wait(&t_full[acc], (tcount / kNBuf) & 1, &abort_flag) ? 1 : 0;
        w = __shfl_sync(0xffffffffu, w, 0);
        if (!w) { failed = 1; if (lane == 0) fail(); continue; }
        tc_fence_after();
        const int j0 = kb * BN + half * kCols;
        // every element of this warp's 32 x kCols block valid?
        const bool interior = (j0 + kCols - 1 < p.S) && (i_lo + 31 < p.S) && (!p.causal || j0 + kCols - 1 <= i_lo);
        const bool empty = (j0 >= p.S) || (i_lo >= p.S) || (p.causal && j0 > i_lo + 31);
        // rounds of two 32-column loads in flight before each wait (the
        // warp's block is empty or not as a whole)
        if (!empty) {
          const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN + half * kCols;
#pragma unroll
          for (int hh = 0; hh < kCols / 64; ++hh) {
            uint32_t r[2][32];
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) tmem_ld_32x32b_x32_async(tbase + (hh * 2 + c2) * 32, r[c2]);
            tmem_ld_wait();
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) reg_fence32(r[c2]);
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
              float* v = reinterpret_cast<float*>(r[c2]);
              const int jc = j0 + (hh * 2 + c2) * 32;
              if (!interior) {
#pragma unroll
                for (int x = 0; x < 32; ++x) {
                  const int j = jc + x;
                  const bool valid = j < p.S && i < p.S && (!p.causal || j <= i);
                  v[x] = valid ? v[x] : -3.402823466e38f;   // finite: invisible to the non-finite check
                }
              }
              // four independent chains each for the maximum and for the
              // NaN-propagating minimum (the non-finite check): one 3-input
              // min or max per two logits
              float m4[4];
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                m4[c] = fmaxf(v[2 * c], v[2 * c + 1]);
                lo4[c] = min3_nan(lo4[c], v[2 * c], v[2 * c + 1]);
              }
#pragma unroll
              for (int x = 8; x < 32; x += 8)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                  m4[c] = max3(m4[c], v[x + 2 * c], v[x + 2 * c + 1]);
                  lo4[c] = min3_nan(lo4[c], v[x + 2 * c], v[x + 2 * c + 1]);
                }
              const float m = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
              if (m > best) {
                best = m;
                if (ARG) {
                  uint32_t jx = 31;
#pragma unroll
                  for (int x = 31; x >= 0; --x) jx = (v[x] == m) ? (uint32_t)x : jx;
                  bidx = (uint32_t)(((long long)b * p.S + i) * p.S + jc + (int)jx);
                }
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&t_empty[acc]);
      }
      // some unmasked logit was NaN or -inf iff the NaN-propagating minimum is
      // NaN or -inf; +inf iff the running maximum is
      const float lo = min3_nan(lo4[0], lo4[1], min3_nan(lo4[2], lo4[3], lo4[3]));
      const bool nonfinite = !(lo > -INFINITY) || best == INFINITY;
      // Reduce (best, bidx) over the warp; each warp publishes its own
      // maximum (the packed atomic max is order-independent, and scaling by
      // a positive factor commutes with max), so the eight epilogue warps
      // never wait for one another between items.
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_down_sync(0xffffffffu, best, o);
        const uint32_t oi = __shfl_down_sync(0xffffffffu, bidx, o);
        if (ov > best || (ov == best && oi < bidx)) { best = ov; bidx = oi; }
      }
      const int badw = __any_sync(0xffffffffu, nonfinite);
      if (lane == 0 && !failed) {
        if (badw) set_status(p.status, MC_STATUS_NONFINITE_LOGIT);
        if (best > -INFINITY) publish(p, h, best * p.scale, bidx);
      }
      if (failed) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult qr;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess && qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

bool encode(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
            const cuuint64_t* strides_bytes, const cuuint32_t* box) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return false;
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides_bytes,
             box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tcml

// The tensor-core path takes bf16 features whose rows TMA can address
// (16-byte aligned bases and strides) and whose head/shared split falls on a
// 64-feature chunk boundary.
bool tc_eligible(const MaxLogitParams& p) {
  if (p.dtype != MC_BF16) return false;
  const int D = p.d_head + p.d_shared;
  if (D > 256) return false;
  if (p.d_shared > 0 && (p.d_head % 64) != 0) return false;
  auto al16 = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; };
  if (!al16(p.q) || !al16(p.k) || (p.d_shared > 0 && !al16(p.ks))) return false;
  for (int i = 0; i < 3; ++i)
    if ((p.qs[i] % 8) != 0 || (p.kst[i] % 8) != 0) return false;
  if (p.d_shared > 0 && ((p.kss[0] % 8) != 0 || (p.kss[1] % 8) != 0)) return false;
  return true;
}

cudaError_t launch_ml_tc(const MaxLogitParams& p, cudaStream_t s, char* err, size_t errlen) {
  using namespace tcml;
  Maps mp;
  memset(&mp, 0, sizeof mp);
  const int D = p.d_head + p.d_shared;
  Geo g;
  g.nck = (p.d_head + 63) / 64;
  g.nch = p.d_shared > 0 ? g.nck + (p.d_shared + 63) / 64 : g.nck;
  g.nqb = (p.S + BM - 1) / BM;
  g.nunit = p.causal ? (g.nqb + 1) / 2 : g.nqb;
  const long long units = (long long)p.B * p.H * g.nunit;
  if (units >= (1ll << 30)) { snprintf(err, errlen, "%lld work units exceed the kernel's 2^30", units); return cudaErrorInvalidValue; }
  g.units = (uint32_t)units;
  g.div_nunit = make_fastdiv((uint32_t)g.nunit);
  g.div_h = make_fastdiv((uint32_t)p.H);
  g.div_bh = make_fastdiv((uint32_t)(p.B * p.H));
  {
    // Heaviest-first snake order balances the CTAs' work to within one item,
    // but interleaves every head, so it is taken only while all the keys
    // stay resident in L2 (at most 96 MB); beyond that the paired
    // (b, h)-major order keeps the heads in flight few.
    const long long kbytes = (long long)p.B * p.S * ((long long)p.H * p.d_head + p.d_shared) * 2;
    const long long items = (long long)p.B * p.H * g.nqb;
    g.snake = (p.causal && kbytes <= (96ll << 20) && items < (1ll << 30)) ? 1 : 0;
    g.items = g.snake ? (uint32_t)items : 0u;
  }
  const int smem_cap = 227 * 1024 - 2048;
  g.stages = (smem_cap - 2 * g.nch * Q_CHUNK) / K_CHUNK;
  if (g.stages > kMaxStages) g.stages = kMaxStages;
  if (g.stages < 2) { snprintf(err, errlen, "q.k length %d leaves no room for key stages", D); return cudaErrorInvalidValue; }
  {
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)p.H, (cuuint64_t)p.S, (cuuint64_t)p.B};
    cuuint64_t st[3] = {(cuuint64_t)p.qs[2] * 2, (cuuint64_t)p.qs[1] * 2, (cuuint64_t)p.qs[0] * 2};
    cuuint32_t box[4] = {64, 1, BM, 1};
    if (!encode(&mp.q, p.q, 4, dims, st, box)) { snprintf(err, errlen, "tensor map for q failed"); return cudaErrorInvalidValue; }
  }
  {
    cuuint64_t dims[4] = {(cuuint64_t)p.d_head, (cuuint64_t)p.H, (cuuint64_t)p.S, (cuuint64_t)p.B};
    cuuint64_t st[3] = {(cuuint64_t)p.kst[2] * 2, (cuuint64_t)p.kst[1] * 2, (cuuint64_t)p.kst[0] * 2};
    cuuint32_t box[4] = {64, 1, BN, 1};
    if (!encode(&mp.k, p.k, 4, dims, st, box)) { snprintf(err, errlen, "tensor map for k failed"); return cudaErrorInvalidValue; }
  }
  if (p.d_shared > 0) {
    cuuint64_t dims[3] = {(cuuint64_t)p.d_shared, (cuuint64_t)p.S, (cuuint64_t)p.B};
    cuuint64_t st[2] = {(cuuint64_t)p.kss[1] * 2, (cuuint64_t)p.kss[0] * 2};
    cuuint32_t box[3] = {64, BN, 1};
    if (!encode(&mp.ks, p.ks, 3, dims, st, box)) { snprintf(err, errlen, "tensor map for k_shared failed"); return cudaErrorInvalidValue; }
  }
  const size_t smem = 1024 + 2 * g.nch * Q_CHUNK + g.stages * K_CHUNK + 512;
  // one CTA per work unit (a single item in snake order), at most one per SM
  const uint32_t work = g.snake ? g.items : g.units;
  const int grid = (int)(work < (uint32_t)sm_count() ? work : (uint32_t)sm_count());
  cudaError_t e;
  if (p.argmax) {
    e = cudaFuncSetAttribute(ml_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    ml_tc_kernel<true><<<grid, kThreads, smem, s>>>(p, mp, g);
  } else {
    e = cudaFuncSetAttribute(ml_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    ml_tc_kernel<false><<<grid, kThreads, smem, s>>>(p, mp, g);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_max_logit(const MaxLogitParams& p, cudaStream_t s, char* err, size_t errlen) {
  const int hb = (p.H + 127) / 128;
  cudaError_t e = cudaSuccess;
  // an accumulating S_max needs neither the initial nor the decoding pass;
  // a plain one only the initial -inf; the argmax keys both
  if (p.argmax || !p.accumulate) {
    ml_init_kernel<<<hb, 128, 0, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (tc_eligible(p)) {
    e = launch_ml_tc(p, s, err, errlen);
    if (e != cudaSuccess) return e;
    if (p.argmax) ml_final_kernel<<<hb, 128, 0, s>>>(p);
    return cudaGetLastError();
  }
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
  if (p.argmax) ml_final_kernel<<<hb, 128, 0, s>>>(p);
  (void)err; (void)errlen;
  return cudaGetLastError();
}

}  // namespace mc
