// Causal attention forward with the per-head max logit taken on the way:
//
//   O^h = softmax(scale * Q^h K^h^T) V^h          ([K2-internals] "核心数学")
//   S_max^h = scale * max_b max_{i, j <= i} q_{b,i,h} . k_{b,j,h}
//
// This is where training finds S_max ("already computed during forward",
// [K2-internals] Algorithm 1): the softmax already needs each row's maximum
// logit, so the per-head max costs one max per row and one atomic per warp.
//
// Tiles: one work item = (b, h, 128 query rows); key/value blocks of 128.
//   warp 0      TMA producer (Q once per item; K and V rings per block)
//   warp 1      TMEM allocator + MMA issuer: S_j = Q K_j^T into one of two
//               128-column TMEM buffers, then O += P_{j-1} V_{j-1} (O: 128 x d_v
//               fp32 in TMEM, P: bf16 in shared memory)
//   warps 2..9  softmax: two threads per query row (warps w and w + 4 share a
//               TMEM lane quadrant; each takes 64 keys and half of O's
//               columns) read S from TMEM, mask, take the row maximum
//               (exchanging half-row maxima through shared memory), write
//               P = 2^(s log2e scale - m) in bf16; at the end of the item they
//               normalise O by the row sum and store it through shared memory
//               with TMA.
// The running maximum m used for the exponentials is updated lazily: only
// when a block's maximum exceeds it by more than 8 (log2 units) are O and the
// row sum rescaled (read, scale and write back the row's O in TMEM), so
// P <= 2^8 and the result is exact either way.  S_max uses the true maximum.
//
// MLA: the q.k length is d_head + d_shared; the key chunks of a block come from
// the head's k^C and then from the rotary key shared by every head, as in the
// max-logit kernel.
//
// Every mbarrier wait is bounded (MC_STATUS_TIMEOUT; the kernel drains its
// copies and MMAs, frees TMEM and returns).
#include <stdio.h>
#include <string.h>

#include "common.cuh"
#include "fastdiv.cuh"
#include "kernels.h"

namespace mc {
namespace {
namespace fa {

constexpr int BM = 128, BN = 128;
constexpr int kThreads = 320;            // producer, MMA, 8 softmax warps
constexpr int CH = 128 * 64 * 2;         // one 128-row x 64-feature bf16 chunk (128-byte swizzle)
constexpr uint32_t kTmemCols = 512;      // S x 2 (cols 0, 128), O (cols 256 ..)
constexpr uint32_t kOCol = 256;
constexpr int kMaxStages = 2;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLazy = 8.f;             // rescale O when the max grows by more than 2^8

struct Maps {
  CUtensorMap q, k, ks, v, o;
};

struct Geo {
  int nch, nck, ncv;   // chunks of q.k, of its head-specific part, of d_v
  int kst, vst;        // K and V stages
  int nqb;             // query blocks per (b, h)
  int nunit;           // units per (b, h) (pairs of query blocks when causal)
  uint32_t units;      // below 2^30 (checked on the host)
  FastDiv div_nunit, div_h;
};

// Work order.  Causal: a unit is a pair of query blocks (ib, nqb - 1 - ib) of
// one (b, h), nqb + 1 key blocks in all whatever ib is, so a static round robin
// over units is balanced; the heavy block runs first and the light one re-reads
// the same keys from L2.  Units are numbered (b, h)-major so the CTAs in flight
// share a few heads' keys and values.  Without the mask each unit is one block.
// Iteration n of a CTA is half n & 1 of its (n >> 1)-th unit: returns 1 with
// the item's coordinates, 0 for the missing half of an unpaired middle block,
// -1 when the CTA has no units left.
__device__ inline int next_item(const AttnFwdParams& p, const Geo& g, uint32_t n, int& b, int& h,
                                int& ib) {
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

__device__ inline int kv_blocks(const AttnFwdParams& p, int ib) {
  const int hi = p.causal ? min(p.S, (ib + 1) * BM) : p.S;
  return (hi + BN - 1) / BN;
}

// byte offset of (row, 16-byte unit u) in a 128-row chunk with 128-byte rows
// and the 128-byte TMA swizzle (unit index XOR row mod 8)
__device__ inline uint32_t sw128(int row, int u) {
  return (uint32_t)(row * 128 + ((u ^ (row & 7)) << 4));
}

__device__ inline float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ inline float min3f(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// S_max stays a float throughout: a non-negative value (sign bit clear) is
// max-combined as a signed int, a negative one min-combined as an unsigned
// int, which orders all non-NaN floats as float max does (-0 below +0).
__global__ void smax_init_kernel(float* smax, int H) {
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h < H) smax[h] = -INFINITY;
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ AttnFwdParams p, const __grid_constant__ Maps mp,
                    const Geo g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* qbuf = smem;                                   // nch chunks
  uint8_t* kbuf = qbuf + g.nch * CH;                      // kst x nch chunks
  uint8_t* vbuf = kbuf + g.kst * g.nch * CH;              // vst x ncv chunks
  uint8_t* pbuf = vbuf + g.vst * g.ncv * CH;              // 2 chunks: P, then O staging
  uint64_t* bars = reinterpret_cast<uint64_t*>(pbuf + 2 * CH);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* s_full = bars + 2;     // [2]
  uint64_t* s_empty = bars + 4;    // [2]
  uint64_t* p_full = bars + 6;
  uint64_t* p_empty = bars + 7;
  uint64_t* o_full = bars + 8;
  uint64_t* o_empty = bars + 9;
  uint64_t* drain = bars + 10;
  uint64_t* xbar = bars + 11;      // [4] half-row exchange per 32-row range
  uint64_t* k_full = bars + 15;    // [kMaxStages]
  uint64_t* k_empty = k_full + kMaxStages;
  uint64_t* v_full = k_empty + kMaxStages;
  uint64_t* v_empty = v_full + kMaxStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(v_empty + kMaxStages);
  __shared__ volatile int abort_flag;
  __shared__ float red[2][2][BM];    // [block parity][half][row] exchanged values

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(q_full, 1); mbar_init(q_empty, 1);
    for (int i = 0; i < 2; ++i) { mbar_init(&s_full[i], 1); mbar_init(&s_empty[i], 8); }
    mbar_init(p_full, 8); mbar_init(p_empty, 1);
    mbar_init(o_full, 1); mbar_init(o_empty, 8);
    mbar_init(drain, 1);
    for (int i = 0; i < 4; ++i) mbar_init(&xbar[i], 64);
    for (int s = 0; s < g.kst; ++s) { mbar_init(&k_full[s], 1); mbar_init(&k_empty[s], 1); }
    for (int s = 0; s < g.vst; ++s) { mbar_init(&v_full[s], 1); mbar_init(&v_empty[s], 1); }
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&mp.q); prefetch_tmap(&mp.k); prefetch_tmap(&mp.v); prefetch_tmap(&mp.o);
    if (g.nch > g.nck) prefetch_tmap(&mp.ks);
  }
  if (warp == 1) { tmem_alloc(tmem_slot, kTmemCols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  auto fail = [&]() { abort_flag = 1; set_status(p.status, MC_STATUS_TIMEOUT); };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // K and V stage rings: next stage and its use parity (counters, no division)
      uint32_t ks = 0, kph = 0, vs = 0, vph = 0, li = 0;
      bool used_q = false, used_k[kMaxStages] = {}, used_v[kMaxStages] = {};
      uint32_t par_q = 0, par_k[kMaxStages] = {}, par_v[kMaxStages] = {};
      for (uint32_t n = 0; !abort_flag; ++n) {
        int b, h, ib;
        const int st = next_item(p, g, n, b, h, ib);
        if (st < 0) break;
        if (st == 0) continue;
        if (!mbar_wait(q_empty, (li & 1) ^ 1, &abort_flag)) { fail(); break; }
        mbar_arrive_expect_tx(q_full, g.nch * CH);
        for (int c = 0; c < g.nch; ++c) tma_load_4d(qbuf + c * CH, &mp.q, q_full, 64 * c, h, ib * BM, b);
        used_q = true; par_q = li & 1;
        const int nkb = kv_blocks(p, ib);
        bool ok = true;
        for (int j = 0; j < nkb && ok; ++j) {
          {
            const int s = (int)ks;
            if (!mbar_wait(&k_empty[s], kph ^ 1, &abort_flag)) { fail(); ok = false; break; }
            mbar_arrive_expect_tx(&k_full[s], g.nch * CH);
            uint8_t* dst = kbuf + s * g.nch * CH;
            for (int c = 0; c < g.nch; ++c) {
              if (c < g.nck) tma_load_4d(dst + c * CH, &mp.k, &k_full[s], 64 * c, h, j * BN, b);
              else tma_load_3d(dst + c * CH, &mp.ks, &k_full[s], 64 * (c - g.nck), j * BN, b);
            }
            used_k[s] = true; par_k[s] = kph;
            if (++ks == (uint32_t)g.kst) { ks = 0; kph ^= 1; }
          }
          {
            const int s = (int)vs;
            if (!mbar_wait(&v_empty[s], vph ^ 1, &abort_flag)) { fail(); ok = false; break; }
            mbar_arrive_expect_tx(&v_full[s], g.ncv * CH);
            uint8_t* dst = vbuf + s * g.ncv * CH;
            for (int c = 0; c < g.ncv; ++c) tma_load_4d(dst + c * CH, &mp.v, &v_full[s], 64 * c, h, j * BN, b);
            used_v[s] = true; par_v[s] = vph;
            if (++vs == (uint32_t)g.vst) { vs = 0; vph ^= 1; }
          }
        }
        if (!ok) break;
        ++li;
      }
      // every issued copy must have landed before the CTA may exit
      if (used_q) mbar_wait(q_full, par_q, nullptr);
      for (int s = 0; s < g.kst; ++s) if (used_k[s]) mbar_wait(&k_full[s], par_k[s], nullptr);
      for (int s = 0; s < g.vst; ++s) if (used_v[s]) mbar_wait(&v_full[s], par_v[s], nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = make_idesc_bf16(BM, BN, 0, 0);   // Q (K-major) x K (K-major)
      const uint32_t idesc_o = make_idesc_bf16(BM, 64 * g.ncv, 0, 1);  // P (K-major) x V (MN-major)
      uint32_t ks = 0, kph = 0, vs = 0, vph = 0, sc = 0, pc = 0, li = 0;   // rings as in the producer
      bool issued = false;
      for (uint32_t n = 0; !abort_flag; ++n) {
        int b, h, ib;
        const int st = next_item(p, g, n, b, h, ib);
        if (st < 0) break;
        if (st == 0) continue;
        const int nkb = kv_blocks(p, ib);
        if (!mbar_wait(q_full, li & 1, &abort_flag)) { fail(); break; }
        bool ok = true;
        for (int j = 0; j <= nkb && ok; ++j) {
          if (j < nkb) {                 // S_j = Q K_j^T
            const int buf = sc & 1;
            if (!mbar_wait(&s_empty[buf], ((sc >> 1) & 1) ^ 1, &abort_flag)) { fail(); ok = false; break; }
            const int s = (int)ks;
            if (!mbar_wait(&k_full[s], kph, &abort_flag)) { fail(); ok = false; break; }
            tc_fence_after();
            const uint32_t qa = smem_u32(qbuf), ka = smem_u32(kbuf + s * g.nch * CH);
            for (int c = 0; c < g.nch; ++c)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                tc_mma(tmem_base + buf * BN, make_sdesc_sw128(qa + c * CH + kk * 32, 16, 1024),
                       make_sdesc_sw128(ka + c * CH + kk * 32, 16, 1024), idesc_s,
                       (c > 0 || kk > 0) ? 1u : 0u);
            issued = true;
            tc_commit(&k_empty[s]);
            tc_commit(&s_full[buf]);
            if (j == nkb - 1) tc_commit(q_empty);
            if (++ks == (uint32_t)g.kst) { ks = 0; kph ^= 1; }
            ++sc;
          }
          if (j >= 1) {                  // O += P_{j-1} V_{j-1}
            if (j == 1 && !mbar_wait(o_empty, (li & 1) ^ 1, &abort_flag)) { fail(); ok = false; break; }
            if (!mbar_wait(p_full, pc & 1, &abort_flag)) { fail(); ok = false; break; }
            const int s = (int)vs;
            if (!mbar_wait(&v_full[s], vph, &abort_flag)) { fail(); ok = false; break; }
            tc_fence_after();
            const uint32_t pa = smem_u32(pbuf), va = smem_u32(vbuf + s * g.ncv * CH);
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              // A: P rows, 64-key chunks of 128-byte rows; B: V rows of 64
              // features (MN-major), 16 key rows = 2048 bytes per k-step, the
              // 64-wide feature blocks one chunk apart
              tc_mma(tmem_base + kOCol, make_sdesc_sw128(pa + (kk >> 2) * CH + (kk & 3) * 32, 16, 1024),
                     make_sdesc(va + kk * 2048, CH, 1024, 2), idesc_o, (j > 1 || kk > 0) ? 1u : 0u);
            tc_commit(&v_empty[s]);
            tc_commit(p_empty);
            if (++vs == (uint32_t)g.vst) { vs = 0; vph ^= 1; }
            ++pc;
          }
        }
        if (!ok) break;
        tc_commit(o_full);
        ++li;
      }
      if (issued) { tc_commit(drain); mbar_wait(drain, 0, nullptr); }
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    // Warps 2..9: warp e = warp - 2 takes rows 32q .. 32q + 31 (q = warp & 3,
    // its TMEM lane quadrant) and keys / O columns of half hf = e >> 2.  The
    // two warps of a row range exchange their half-row maxima once per block
    // through shared memory behind a bounded mbarrier (xbar[q], both slots of
    // red alternating with the block parity); their row sums stay separate
    // until the end of the item.
    const int e = warp - 2;
    const int q = warp & 3, hf = e >> 2;
    const int row = q * 32 + lane;
    const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16);
    const int ocols = 32 * g.ncv;                  // O columns of this half
    uint8_t* mine = pbuf + hf * CH + q * 32 * 128;  // this warp's P rows / O staging (4 KB)
    const float c2 = p.scale * kLog2e;
    uint32_t sc = 0, pc = 0, li = 0, xc = 0;
    bool bad = false;
    auto exchange = [&](float v_mine, float& v_other) -> bool {
      const int slot = xc & 1;
      red[slot][hf][row] = v_mine;
      mbar_arrive(&xbar[q]);
      const bool ok = mbar_wait(&xbar[q], xc & 1, &abort_flag);
      v_other = red[slot][hf ^ 1][row];
      ++xc;
      return ok;
    };
    for (uint32_t n = 0;; ++n) {
      int b, h, ib;
      const int st = next_item(p, g, n, b, h, ib);
      if (st < 0) break;
      if (st == 0) continue;
      const int nkb = kv_blocks(p, ib);
      const int i = ib * BM + row;                   // this thread's query row
      float m_run = -INFINITY, l = 0.f, raw_max = -INFINITY;
      int failed = 0;
      for (int j = 0; j < nkb && !failed; ++j, ++sc, ++pc) {
        const int buf = sc & 1;
        int w = 1;
        if (lane == 0) w = mbar_wait(&s_full[buf], (sc >> 1) & 1, &abort_flag) ? 1 : 0;
        w = __shfl_sync(0xffffffffu, w, 0);
        if (!w) { failed = 1; break; }
        tc_fence_after();
        uint32_t r[2][32];
#pragma unroll
        for (int c = 0; c < 2; ++c) tmem_ld_32x32b_x32_async(trow + buf * BN + hf * 64 + c * 32, r[c]);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 2; ++c) reg_fence32(r[c]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_empty[buf]);   // S buffer free for block j + 2
        float v[64];
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int x = 0; x < 32; ++x) v[c * 32 + x] = __uint_as_float(r[c][x]);
        const int j0 = j * BN + hf * 64;
        const bool full = (j0 + 63 < p.S) && (i < p.S) && (!p.causal || j0 + 63 <= ib * BM);
        // half-row max and min over the valid logits, four independent chains
        // each (a non-finite valid logit shows as max = +inf, min = -inf, or a
        // NaN sum below)
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        float mn4[4] = {INFINITY, INFINITY, INFINITY, INFINITY};
        if (full) {
#pragma unroll
          for (int x = 0; x < 64; x += 8)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              mx4[c] = max3f(mx4[c], v[x + 2 * c], v[x + 2 * c + 1]);
              mn4[c] = min3f(mn4[c], v[x + 2 * c], v[x + 2 * c + 1]);
            }
        } else {
#pragma unroll
          for (int x = 0; x < 64; ++x) {
            const int jj = j0 + x;
            const bool valid = jj < p.S && i < p.S && (!p.causal || jj <= i);
            mn4[x & 3] = fminf(mn4[x & 3], valid ? v[x] : INFINITY);
            v[x] = valid ? v[x] : -INFINITY;
            mx4[x & 3] = fmaxf(mx4[x & 3], v[x]);
          }
        }
        const float mxh = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        const float mn = fminf(fminf(mn4[0], mn4[1]), fminf(mn4[2], mn4[3]));
        bad |= (mxh == INFINITY) || (mn == -INFINITY);
        raw_max = fmaxf(raw_max, mxh);
        float mxo;
        w = exchange(mxh, mxo) ? 1 : 0;
        if (!__all_sync(0xffffffffu, w)) { failed = 1; break; }
        const float mx = fmaxf(mxh, mxo);             // the full row's maximum
        // lazy running max (log2 units); both halves decide identically
        float alpha = 1.f;
        bool rescale = false;
        if (mx != -INFINITY) {
          const float m_new = mx * c2;
          if (m_run == -INFINITY || m_new > m_run + kLazy) {
            alpha = m_run == -INFINITY ? 0.f : ex2_approx(m_run - m_new);
            rescale = j > 0 && m_run != -INFINITY;
            m_run = m_new;
            l *= alpha;
          }
        }
        uint32_t pk[32];
        if (m_run == -INFINITY) {        // no valid key yet (a row past the sequence end)
#pragma unroll
          for (int x = 0; x < 32; ++x) pk[x] = 0u;
        } else {
          float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int x = 0; x < 64; x += 2) {
            const float e0 = ex2_approx(fmaf(v[x], c2, -m_run));
            const float e1 = ex2_approx(fmaf(v[x + 1], c2, -m_run));
            s4[(x >> 1) & 3] += e0 + e1;
            __nv_bfloat162 h2 = __floats2bfloat162_rn(e0, e1);
            pk[x / 2] = *reinterpret_cast<uint32_t*>(&h2);
          }
          const float sum = (s4[0] + s4[1]) + (s4[2] + s4[3]);
          bad |= sum != sum;
          l += sum;
        }
        // P buffer free and O updated once the previous block's P V is done
        if (lane == 0) w = mbar_wait(p_empty, (pc & 1) ^ 1, &abort_flag) ? 1 : 0;
        w = __shfl_sync(0xffffffffu, w, 0);
        if (!w) { failed = 1; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, rescale)) {
          const float a = rescale ? alpha : 1.f;
          for (int c = 0; c < g.ncv; ++c) {
            const uint32_t col = kOCol + hf * ocols + c * 32;
            uint32_t o[32];
            tmem_ld_32x32b_x32_async(trow + col, o);
            tmem_ld_wait();
            reg_fence32(o);
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * a);
            tmem_st_32x32b_x32(trow + col, o);
          }
          tmem_st_wait();
        }
        // this warp's previous O store must have read its staging rows
        if (lane == 0) bulk_wait_read0();
        __syncwarp();
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 val = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
          *reinterpret_cast<uint4*>(pbuf + hf * CH + sw128(row, u)) = val;
        }
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
      }
      // ---- epilogue of the item: O / l -> bf16 -> TMA store; lse; S_max
      int w = failed ? 0 : 1;
      if (!failed && lane == 0) w = mbar_wait(o_full, li & 1, &abort_flag) ? 1 : 0;
      w = __shfl_sync(0xffffffffu, w, 0);
      if (w) {
        float lo;
        w = exchange(l, lo) ? 1 : 0;               // the row sum is the two halves'
        w = __all_sync(0xffffffffu, w);
        l += lo;
      }
      if (!w) { if (lane == 0) fail(); break; }
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int r32 = lane;                          // row within this warp's 32
      for (int c = 0; c < g.ncv; ++c) {
        uint32_t o[32];
        tmem_ld_32x32b_x32_async(trow + kOCol + hf * ocols + c * 32, o);
        tmem_ld_wait();
        reg_fence32(o);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint32_t pk4[4];
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(o[8 * u + 2 * x]) * inv,
                                                      __uint_as_float(o[8 * u + 2 * x + 1]) * inv);
            pk4[x] = *reinterpret_cast<uint32_t*>(&h2);
          }
          // 32 x 32 box, 64-byte rows, 64-byte swizzle; box c at 2 KB steps
          *reinterpret_cast<uint4*>(mine + c * 2048 + r32 * 64 + ((u ^ ((r32 >> 1) & 3)) << 4)) =
              make_uint4(pk4[0], pk4[1], pk4[2], pk4[3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_empty);           // the MMA warp may overwrite O
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        for (int c = 0; c < g.ncv; ++c)
          if (hf * ocols + 32 * c < p.d_v)
            tma_store_4d(&mp.o, mine + c * 2048, hf * ocols + 32 * c, h, ib * BM + q * 32, b);
        bulk_commit();
      }
      if (hf == 0 && p.lse && i < p.S)
        p.lse[((long long)b * p.H + h) * p.S + i] = l > 0.f ? (m_run + log2f(l)) * kLn2 : -INFINITY;
      float wm = raw_max;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
      if (lane == 0 && wm > -INFINITY) {
        const float v = wm * p.scale;
        if (__float_as_int(v) >= 0) atomicMax(reinterpret_cast<int*>(p.smax) + h, __float_as_int(v));
        else atomicMin(reinterpret_cast<unsigned int*>(p.smax) + h, __float_as_uint(v));
      }
      ++li;
    }
    if (lane == 0) bulk_wait0();
    if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(p.status, MC_STATUS_NONFINITE_LOGIT);
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
            const cuuint64_t* strides_bytes, const cuuint32_t* box,
            CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return false;
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides_bytes,
             box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool geometry(const AttnFwdParams& p, Geo& g, size_t& smem, char* err, size_t errlen) {
  g.nck = (p.d_head + 63) / 64;
  g.nch = p.d_shared > 0 ? g.nck + (p.d_shared + 63) / 64 : g.nck;
  g.ncv = (p.d_v + 63) / 64;
  g.nqb = (p.S + BM - 1) / BM;
  g.nunit = p.causal ? (g.nqb + 1) / 2 : g.nqb;
  const long long units = (long long)p.B * p.H * g.nunit;
  if (units >= (1ll << 30)) { snprintf(err, errlen, "%lld work units exceed the kernel's 2^30", units); return false; }
  g.units = (uint32_t)units;
  g.div_nunit = make_fastdiv((uint32_t)g.nunit);
  g.div_h = make_fastdiv((uint32_t)p.H);
  const size_t cap = 227 * 1024 - 1024 - 256 - 2 * 2 * BM * 4 - 64;   // static: red, abort flag
  const size_t fixed = (size_t)(g.nch + 2) * CH;      // Q, P
  g.kst = g.vst = 0;
  for (int ks = kMaxStages; ks >= 1 && !g.kst; --ks)
    for (int vs = kMaxStages; vs >= 1; --vs)
      if (fixed + (size_t)ks * g.nch * CH + (size_t)vs * g.ncv * CH <= cap) { g.kst = ks; g.vst = vs; break; }
  if (!g.kst) {
    snprintf(err, errlen, "q.k length %d and d_v %d leave no room for key/value stages",
             p.d_head + p.d_shared, p.d_v);
    return false;
  }
  smem = 1024 + fixed + (size_t)g.kst * g.nch * CH + (size_t)g.vst * g.ncv * CH + 256;
  return true;
}

}  // namespace fa
}  // namespace

bool attn_fwd_supported(const AttnFwdParams& p, char* err, size_t errlen) {
  const int D = p.d_head + p.d_shared;
  if (D < 16 || D > 192) { snprintf(err, errlen, "q.k length %d outside [16, 192]", D); return false; }
  if (p.d_v < 16 || p.d_v > 128) { snprintf(err, errlen, "d_v %d outside [16, 128]", p.d_v); return false; }
  if (p.d_shared > 0 && (p.d_head % 64) != 0) {
    snprintf(err, errlen, "with a shared key part d_head must be a multiple of 64 (got %d)", p.d_head);
    return false;
  }
  auto al16 = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; };
  if (!al16(p.q) || !al16(p.k) || !al16(p.v) || !al16(p.o) || (p.d_shared > 0 && !al16(p.ks))) {
    snprintf(err, errlen, "q, k, k_shared, v and o must be 16-byte aligned");
    return false;
  }
  for (int i = 0; i < 3; ++i)
    if ((p.qs[i] % 8) || (p.kst[i] % 8) || (p.vs[i] % 8) || (p.os[i] % 8)) {
      snprintf(err, errlen, "strides must be multiples of 8 elements");
      return false;
    }
  if (p.d_shared > 0 && ((p.kss[0] % 8) || (p.kss[1] % 8))) {
    snprintf(err, errlen, "k_shared strides must be multiples of 8 elements");
    return false;
  }
  fa::Geo g;
  size_t smem;
  return fa::geometry(p, g, smem, err, errlen);
}

cudaError_t launch_attn_fwd(const AttnFwdParams& p, cudaStream_t s, char* err, size_t errlen) {
  using namespace fa;
  Geo g;
  size_t smem;
  if (!geometry(p, g, smem, err, errlen)) return cudaErrorInvalidValue;
  Maps mp;
  memset(&mp, 0, sizeof mp);
  const int D = p.d_head + p.d_shared;
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
  {
    cuuint64_t dims[4] = {(cuuint64_t)p.d_v, (cuuint64_t)p.H, (cuuint64_t)p.S, (cuuint64_t)p.B};
    cuuint64_t st[3] = {(cuuint64_t)p.vs[2] * 2, (cuuint64_t)p.vs[1] * 2, (cuuint64_t)p.vs[0] * 2};
    cuuint32_t box[4] = {64, 1, BN, 1};
    if (!encode(&mp.v, p.v, 4, dims, st, box)) { snprintf(err, errlen, "tensor map for v failed"); return cudaErrorInvalidValue; }
  }
  {
    cuuint64_t dims[4] = {(cuuint64_t)p.d_v, (cuuint64_t)p.H, (cuuint64_t)p.S, (cuuint64_t)p.B};
    cuuint64_t st[3] = {(cuuint64_t)p.os[2] * 2, (cuuint64_t)p.os[1] * 2, (cuuint64_t)p.os[0] * 2};
    cuuint32_t box[4] = {32, 1, 32, 1};               // one warp's 32 rows x 32 features
    if (!encode(&mp.o, p.o, 4, dims, st, box, CU_TENSOR_MAP_SWIZZLE_64B)) { snprintf(err, errlen, "tensor map for o failed"); return cudaErrorInvalidValue; }
  }
  const int hb = (p.H + 127) / 128;
  cudaError_t e = cudaSuccess;
  if (!p.accumulate) {
    smax_init_kernel<<<hb, 128, 0, s>>>(p.smax, p.H);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  e = cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = (int)(g.units < (uint32_t)sm_count() ? g.units : (uint32_t)sm_count());
  attn_fwd_kernel<<<grid, kThreads, smem, s>>>(p, mp, g);
  return cudaGetLastError();
}

}  // namespace mc
