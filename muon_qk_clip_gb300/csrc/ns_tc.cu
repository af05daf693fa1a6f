// Tensor-core (tcgen05 / TMEM / TMA) grouped GEMM for the Newton-Schulz phases
// of Muon ([K2-internals] Algorithm 1 orthogonalisation step; [K2-explained]
// symbol list: "a few iterations of an odd matrix polynomial"):
//
//   phase 1  A  = s * X X^T            (A operand X rows, B operand X rows)
//   phase 2  B  = c * A A + b * A      (A symmetric: its rows serve as B^T)
//   phase 3  X' = s * (B X + a * X)    (B operand X stored [K, N]: MN-major)
//
// All three are D = s_b * (alpha * P + beta * C + diag * I) with
// P = A_op x B_op^T.  In three-term iterations phase 2 adds a I and phase 3
// reads no C (X' = s * (B + a I) X).
// Split mode (default): every operand is a 16-bit pair (hi, lo) and
// P = hi*hi + hi*lo + lo*hi accumulated in fp32 in TMEM, so products carry
// ~16 significand bits (one-product launches take hi*hi alone, the last
// update of a step may take hi*hi + hi*lo_B); D is stored again as a
// (hi, lo) pair.  Plain mode: one bf16 plane, one MMA per k-step.
//
// Kernel layout (one CTA per SM, persistent over output tiles, CTAs paired
// into tcgen05 .cta_group::2 clusters of two):
//   warp 0      TMA producer (one elected lane)
//   warp 1      TMEM allocator + MMA issuer (one elected lane of the first
//               CTA of the pair)
//   warps 2..9  epilogue: TMEM -> registers -> fused polynomial -> global
// A pair computes 256 x 256 output tiles (128 rows per CTA) with K advancing
// by 64 in three-product launches and by 128 in one-product ones (operand
// rows in 128-byte swizzled boxes of 64 elements, three 64 KB stages); the
// accumulator is double-buffered in TMEM (2 x 256 columns) so the epilogue of
// tile t overlaps the MMAs of tile t+1.  The epilogue stages every 32 x 16
// chunk of D (and, for symmetric outputs, its transpose) through 4 KB of
// shared memory per warp, from where TMA bulk stores write it.
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

constexpr int BM = 128, BN = 256, BKT = 32;
constexpr int kEpiWarps = 8;           // two per TMEM lane quadrant (column halves)
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint32_t kTmemCols = 512;    // two 128 x 256 fp32 accumulators
constexpr int kEpiWarpBytes = 4096;    // per epilogue warp: two 32 x 16 hi+lo slots
constexpr int kEpiBytes = kEpiWarps * kEpiWarpBytes;
constexpr int kBarBytes = 512;
constexpr int kTS = 4;                 // tile-id ring (dynamic schedule)
constexpr int kSmemCap = 227 * 1024;

// K-major operand layout for a k-step of BK: rows of BK bf16 with the 64-byte
// (BK 32) or 128-byte (BK 64) swizzle, 8-row atoms.
template <int BK>
struct KLayout {
  static_assert(BK == 32 || BK == 64 || BK == 128, "k-step");
  static constexpr int kBX = BK < 64 ? BK : 64;           // K elements per TMA box (<= 128 bytes)
  static constexpr int kSub = BK / kBX;                   // boxes along K per operand per stage
  static constexpr uint32_t kType = kBX == 64 ? 2u : 4u;
  static constexpr uint32_t kSbo = 8 * kBX * 2;
};

// TERMS: tensor-core products per k-step (1: hi*hi; 2: hi*hi + hi*lo_B;
// 3: hi*hi + hi*lo + lo*hi).
// LO: the iterate is stored as (hi, lo) planes (the epilogue reads and writes
// both), independently of how many products the k-loop takes.
template <int TERMS, int AROWS, int BROWS, int BK = BKT>
struct Stages {
  static constexpr int kABytes = AROWS * BK * 2;
  static constexpr int kBBytes = BROWS * BK * 2;
  // three products stage both planes of A and B; two (hi*hi + hi*lo_B)
  // both planes of B; one the hi planes only
  static constexpr int kStageBytes =
      TERMS == 3 ? 2 * (kABytes + kBBytes) : (TERMS == 2 ? kABytes + 2 * kBBytes : kABytes + kBBytes);
  static constexpr int kAvail = kSmemCap - kEpiBytes - 1024 - kBarBytes - 64;
  static constexpr int kStages = kAvail / kStageBytes > 8 ? 8 : kAvail / kStageBytes;
  static constexpr int kSmem = kStages * kStageBytes + kEpiBytes + 1024 + kBarBytes;
  static_assert(kStages >= 2, "stage count");
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

// Tiles of tm_rows x 256.  Symmetric outputs keep only tiles touching the
// upper triangle: column tile tn holds row tiles tm < (tn + 1) * 256 / tm_rows.
template <int TM_ROWS>
__device__ inline TileCoord tile_coord(const GemmParams& p, int t) {
  TileCoord c;
  c.g = find_group(p, t);
  const GemmGroup& G = p.g[c.g];
  const int lt = t - G.tile_begin;
  c.b = lt / G.tiles_per_item;
  int rem = lt % G.tiles_per_item;
  if (!G.symmetric) {
    c.m0 = (rem % G.tiles_m) * TM_ROWS;   // consecutive tiles share the B column block
    c.n0 = (rem / G.tiles_m) * BN;
  } else {
    int tn = 0;
    for (;; ++tn) {
      const int rows = min(G.tiles_m, (tn + 1) * (BN / TM_ROWS));
      if (rem < rows) break;
      rem -= rows;
    }
    c.m0 = rem * TM_ROWS;
    c.n0 = tn * BN;
  }
  return c;
}

// Byte offsets in the TMA swizzle patterns (the 16-byte unit index of a row is
// XOR-ed with address bits 7 and up): 32-byte rows (32-byte swizzle, one bit)
// and 64-byte rows (64-byte swizzle, two bits).
__device__ inline uint32_t swz32(int row, int b) {
  return (uint32_t)(row * 32 + ((((b >> 4) ^ ((row >> 2) & 1)) & 1) << 4) + (b & 15));
}
__device__ inline uint32_t swz64(int row, int b) {
  return (uint32_t)(row * 64 + ((((b >> 4) ^ ((row >> 1) & 3)) & 3) << 4) + (b & 15));
}

// ------------------------------------------------------------ epilogue
// One warp's 32 rows [r0, r0 + 32) and 16-column chunks [c_begin, c_end) of an
// output tile whose accumulator sits in TMEM at `tacc` (lane quadrant q).
// D = s_b * (alpha * acc + beta * C + diag I).  Symmetric outputs: chunks in
// 128-column blocks I < J are also stored transposed (mirror); I > J are
// dropped.
//
// The warp's 4 KB of shared memory is two 2 KB slots, each a 32 x 16 chunk of
// hi and lo planes (32-byte rows, 32-byte swizzle): a chunk of D and its
// mirror (16 rows of 64 bytes, 64-byte swizzle) for symmetric outputs, else a
// ring of two D chunks, so a chunk waits only for the store group that last
// used its slot.  The small footprint leaves room for three 64 KB operand
// stages.  `ek` counts this warp's store groups across tiles.  C of a
// symmetric output (the polynomial's b A term) is read by each lane straight
// from global memory (its row's 32 contiguous bytes per plane); C of a
// non-symmetric output (the update's a X term) arrives by TMA (CSlots below).
// The next chunk's TMEM load and C loads are issued as soon as the current
// chunk's values are converted, so they are in flight while it is stored; two
// warps share each lane quadrant (one per column half), so one warp's waits
// overlap the other's work.
constexpr int kCW = 16;                         // chunk width (columns)
constexpr int kPlane = 32 * kCW * 2;            // 1 KB: one plane of a chunk
constexpr int kSlot = 2 * kPlane;               // hi + lo

// The lane's C of a chunk: 2 x 8 columns per plane, zero past the edges.
template <bool LO>
__device__ inline void load_c_chunk(const GemmGroup& G, const TileCoord& tc, int row, int ch,
                                    uint4 (&h)[2], uint4 (&l)[2]) {
  const int col0 = tc.n0 + ch * kCW;
  const bool row_ok = row < G.M;
  const long long o = (long long)tc.b * G.c_bstride + (long long)row * G.ldc + col0;
  const uint16_t* c_hi = reinterpret_cast<const uint16_t*>(G.c_hi) + o;
  const uint16_t* c_lo = reinterpret_cast<const uint16_t*>(G.c_lo) + o;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const bool ok = row_ok && col0 + 8 * j < G.N;
    h[j] = ok ? __ldg(reinterpret_cast<const uint4*>(c_hi + 8 * j)) : make_uint4(0, 0, 0, 0);
    if (LO) l[j] = ok ? __ldg(reinterpret_cast<const uint4*>(c_lo + 8 * j)) : make_uint4(0, 0, 0, 0);
  }
}

// Before a tile's accumulator is ready: pull the C rows this warp will read
// (its 32 rows, chunks [c_begin, c_end), both planes) into L2, so the
// epilogue's loads, issued one chunk ahead, wait for L2 rather than DRAM.
template <bool LO>
__device__ inline void prefetch_c_rows(const GemmParams& p, const TileCoord& tc, int r0, int c_begin,
                                       int c_end, int lane) {
  const GemmGroup& G = p.g[tc.g];
  const int row = r0 + lane;
  if (p.beta == 0.f || row >= G.M) return;
  const long long o = (long long)tc.b * G.c_bstride + (long long)row * G.ldc;
  const uint16_t* c_hi = reinterpret_cast<const uint16_t*>(G.c_hi) + o;
  const uint16_t* c_lo = reinterpret_cast<const uint16_t*>(G.c_lo) + o;
  for (int ch = c_begin; ch < c_end; ch += 4) {      // one 128-byte line per four chunks
    const int col0 = tc.n0 + ch * kCW;
    if (col0 >= G.N) break;
    prefetch_l2(c_hi + col0);
    if (LO) prefetch_l2(c_lo + col0);
  }
}

// C through TMA (non-symmetric outputs with a C term): the warp's two slots
// take the C chunks as 16 x 32 boxes (hi and lo planes), loaded two chunks
// ahead and, for a tile's first two chunks, before its accumulator is ready;
// each chunk's D is then written over its C in the same slot and leaves by
// TMA.  Chunk i of the warp's sequence uses slot ek & 1.
struct CSlots {
  uint64_t* bar;       // [2] completion of the C box loads of each slot
  uint32_t par;        // bit s: parity of the next wait on bar[s]
  uint32_t pending;    // bit s: a load into slot s has not been waited for
};

__device__ inline bool c_by_tma(const GemmParams& p, const GemmGroup& G) {
  return p.beta != 0.f && !G.symmetric;
}

// Lane 0: load C chunk `ch` of rows [r0, r0 + 32) into slot `slot`, once the
// store that last read the slot has finished reading it.
template <bool LO>
__device__ inline void c_load(const TmaArgs& tm, const TileCoord& tc, int r0, int ch, uint8_t* ebuf,
                              int slot, CSlots& cs) {
  bulk_wait_read_upto(0);
  uint8_t* sb = ebuf + slot * kSlot;
  mbar_arrive_expect_tx(&cs.bar[slot], LO ? 2 * kPlane : kPlane);
  const int col0 = tc.n0 + ch * kCW;
  tma_load_3d(sb, &tm.maps.c_hi[tc.g], &cs.bar[slot], col0, r0, tc.b);
  if (LO) tma_load_3d(sb + kPlane, &tm.maps.c_lo[tc.g], &cs.bar[slot], col0, r0, tc.b);
  cs.pending |= 1u << slot;
}

// The first two live chunks of this warp's share of a tile (issued before
// the accumulator is ready).
template <bool LO>
__device__ inline void c_prologue(const GemmParams& p, const TmaArgs& tm, const TileCoord& tc, int r0,
                                  int c_begin, int c_end, int lane, uint8_t* ebuf, uint32_t ek,
                                  CSlots& cs) {
  const GemmGroup& G = p.g[tc.g];
  if (!c_by_tma(p, G) || r0 >= G.M || lane != 0) return;
  int k = 0;
  for (int ch = c_begin; ch < c_end && k < 2; ++ch) {
    if (tc.n0 + ch * kCW >= G.N) break;
    c_load<LO>(tm, tc, r0, ch, ebuf, (int)((ek + k) & 1), cs);
    ++k;
  }
}

template <bool LO, bool IN16, bool OUT16>
__device__ bool epilogue_rows(const GemmParams& p, const TmaArgs& tm, const TileCoord& tc, int r0,
                              int c_begin, int c_end, uint32_t tacc, int q, int lane, uint8_t* ebuf,
                              uint32_t& ek, bool& bad, CSlots& cs, volatile int* abort_flag) {
  const GemmGroup& G = p.g[tc.g];
  if (r0 >= G.M) return true;                       // no valid row in this warp
  const float sb = p.s ? p.s[G.mat_base + tc.b] : 1.f;
  const float al = p.alpha * sb, be = p.beta * sb, dg = p.diag * sb;
  const bool use_c = p.beta != 0.f;
  const bool tmac = c_by_tma(p, G);                 // C arrives by TMA in the slots
  const int per = G.symmetric ? 2 : 1;              // slots per store group
  const int depth = 2 / per;                        // store groups in flight
  const int I = r0 / 128;
  auto mode_of = [&](int ch) -> int {             // 0 skip, 1 store, 2 store + mirror
    const int col0 = tc.n0 + ch * kCW;
    if (col0 >= G.N) return 0;
    if (!G.symmetric) return 1;
    const int J = col0 / 128;
    return I < J ? 2 : (I == J ? 1 : 0);
  };
  auto next_live = [&](int ch) -> int {
    for (int c = ch + 1; c < c_end; ++c)
      if (mode_of(c)) return c;
    return c_end;
  };
  const int row = r0 + lane;
  const bool row_ok = row < G.M;
  const uint32_t trow = tacc + ((uint32_t)(q * 32) << 16);
  int ch = next_live(c_begin - 1);
  if (ch >= c_end) return true;
  uint4 c_h[2], c_l[2];
  uint32_t nr[16];
  tmem_ld_32x32b_x16_async(trow + ch * kCW, nr);
  if (use_c && !tmac) load_c_chunk<LO>(G, tc, row, ch, c_h, c_l);
  while (ch < c_end) {
    const int mode = mode_of(ch);
    const int col0 = tc.n0 + ch * kCW;
    const int nx = next_live(ch);
    uint8_t* db = ebuf + (int)(ek % (uint32_t)depth) * per * kSlot;
    if (tmac) {
      // this chunk's C box: wait for it, then read the lane's row from the slot
      const int slot = (int)(ek & 1);
      int ok = 1;
      if (lane == 0) {
        ok = mbar_wait(&cs.bar[slot], (cs.par >> slot) & 1u, abort_flag) ? 1 : 0;
        if (ok) cs.pending &= ~(1u << slot);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        tmem_ld_wait();                 // the chunk's TMEM load lands before giving up
        return false;
      }
      cs.par ^= 1u << slot;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        c_h[j] = *reinterpret_cast<const uint4*>(db + swz32(lane, j * 16));
        if (LO) c_l[j] = *reinterpret_cast<const uint4*>(db + kPlane + swz32(lane, j * 16));
      }
    }
    tmem_ld_wait();
    reg_fence16(nr);
    float v[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(nr[e]);
    if (use_c) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint16_t* hh = reinterpret_cast<const uint16_t*>(&c_h[j]);
        const uint16_t* ll = reinterpret_cast<const uint16_t*>(&c_l[j]);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float cv = LO ? from16<IN16>(hh[e]) + from16<IN16>(ll[e]) : from16<IN16>(hh[e]);
          v[j * 8 + e] = fmaf(al, v[j * 8 + e], be * cv);
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] *= al;
    }
    if (dg != 0.f && row >= col0 && row < col0 + kCW) {
#pragma unroll
      for (int e = 0; e < 16; ++e)
        if (col0 + e == row) v[e] += dg;
    }
    // non-finite test: v * 0 is 0 for a finite v and NaN for Inf or NaN, so
    // four chains of fma(v, 0, acc) end in NaN iff some value is not finite
    // (the ragged edge tests its valid elements one by one)
    if (row_ok && col0 + kCW - 1 < G.N) {
      float z4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int e = 0; e < 16; ++e) z4[e & 3] = fmaf(v[e], 0.f, z4[e & 3]);
      const float z = (z4[0] + z4[1]) + (z4[2] + z4[3]);
      bad |= z != z;
    } else if (row_ok) {
#pragma unroll
      for (int e = 0; e < 16; ++e) bad |= !finite_f(v[e]) && (col0 + e < G.N);
    }
    uint16_t hb[16], lb[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      if (LO) split16<OUT16>(v[e], hb[e], lb[e]);
      else hb[e] = to16<OUT16>(v[e]);
    }
    // this chunk's accumulator and C are consumed: start the next chunk's
    // loads (warp-uniform: nx is the same in every lane)
    if (nx < c_end) {
      tmem_ld_32x32b_x16_async(trow + nx * kCW, nr);
      if (use_c && !tmac) load_c_chunk<LO>(G, tc, row, nx, c_h, c_l);
    }
    uint8_t* mb = db + kSlot;
    // the store group that last used these slots must have read them (with C
    // by TMA the slot was last read by this chunk's own C box, already used)
    if (lane == 0 && !tmac) bulk_wait_read_upto(depth - 1);
    __syncwarp();
    const bool st_lo = LO && !p.d_hi_only;          // warp-uniform
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      *reinterpret_cast<uint4*>(db + swz32(lane, j * 16)) = *reinterpret_cast<const uint4*>(hb + j * 8);
      if (st_lo)
        *reinterpret_cast<uint4*>(db + kPlane + swz32(lane, j * 16)) = *reinterpret_cast<const uint4*>(lb + j * 8);
    }
    if (mode == 2) {
      // mirror: row c of a 16 x 32 plane holds column c of this chunk, i.e.
      // lane (row) r -> byte 2r
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        *reinterpret_cast<uint16_t*>(mb + swz64(c, 2 * lane)) = hb[c];
        if (st_lo) *reinterpret_cast<uint16_t*>(mb + kPlane + swz64(c, 2 * lane)) = lb[c];
      }
    }
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(&tm.maps.d_hi[tc.g], db, col0, r0, tc.b);
      if (st_lo) tma_store_3d(&tm.maps.d_lo[tc.g], db + kPlane, col0, r0, tc.b);
      if (mode == 2) {
        tma_store_3d(&tm.maps.dm_hi[tc.g], mb, r0, col0, tc.b);
        if (st_lo) tma_store_3d(&tm.maps.dm_lo[tc.g], mb + kPlane, r0, col0, tc.b);
      }
      bulk_commit();
      // the chunk two on takes its C into this slot once the store has read it
      if (tmac) {
        const int n2 = nx < c_end ? next_live(nx) : c_end;
        if (n2 < c_end) c_load<LO>(tm, tc, r0, n2, ebuf, (int)(ek & 1), cs);
      }
    }
    ++ek;
    ch = nx;
  }
  return true;
}

// ------------------------------------------------------------ fused apply
// The last update of a step, applied in its epilogue: for chunk values v (the
// oriented iterate X5 = D / alpha), W <- rn_bf16(W - lr (scale v + wd W)).
// A chunk covers X rows r0 .. r0 + 31 and columns col0 .. col0 + 15.  When W
// is oriented like X its segment is 32 rows of 32 contiguous bytes (W rows
// r0 + k at columns col0 ..); when W is the transpose of X it is 16 rows of 64
// bytes (W rows col0 + e at columns r0 ..).  Full segments move by 1-D bulk
// copies, one per row (slot rows 48 or 80 bytes apart, which spreads the
// lanes' accesses over the banks), loaded two chunks ahead and stored back
// from the slot; segments cut by the matrix's edge are read and written by
// plain loads and stores.
struct NoApply {
  static constexpr bool kOn = false;
};

__device__ inline const FusedApplyJob& fa_job(const FusedApply& fa, const GemmGroup& G, const TileCoord& tc) {
  return fa.job[G.mat_base + tc.b];
}
__device__ inline bool w_full(const FusedApplyJob& J, const GemmGroup& G, int r0, int col0) {
  return J.transpose ? (r0 + 32 <= G.M) : (col0 + kCW <= G.N);
}
// slot rows of the segment, their bytes and their pitch in the slot
__device__ inline int w_rows(const FusedApplyJob& J, const GemmGroup& G, int r0, int col0) {
  return J.transpose ? min(kCW, G.N - col0) : min(32, G.M - r0);
}
__device__ inline int w_row_bytes(const FusedApplyJob& J) { return J.transpose ? 64 : 2 * kCW; }
__device__ inline int w_pitch(const FusedApplyJob& J) { return J.transpose ? 80 : 48; }
__device__ inline __nv_bfloat16* w_row(const FusedApplyJob& J, int r0, int col0, int k) {
  __nv_bfloat16* w = reinterpret_cast<__nv_bfloat16*>(J.w);
  return J.transpose ? w + (long long)(col0 + k) * J.ld + r0 : w + (long long)(r0 + k) * J.ld + col0;
}

// All lanes: bring chunk ch's W segment into slot `slot` (full segments only),
// once this lane's earlier stores from the slot have read it.
__device__ inline void w_load(const FusedApply& fa, const GemmParams& p, const TileCoord& tc, int r0, int ch,
                              uint8_t* ebuf, int slot, CSlots& cs, int lane) {
  const GemmGroup& G = p.g[tc.g];
  const FusedApplyJob& J = fa_job(fa, G, tc);
  const int col0 = tc.n0 + ch * kCW;
  if (!w_full(J, G, r0, col0)) return;
  const int nr = w_rows(J, G, r0, col0), rb = w_row_bytes(J);
  bulk_wait_read0();
  __syncwarp();
  if (lane == 0) {
    mbar_arrive_expect_tx(&cs.bar[slot], (uint32_t)(rb * nr));
    cs.pending |= 1u << slot;
  }
  __syncwarp();
  if (lane < nr)
    bulk_load_1d(ebuf + slot * kSlot + lane * w_pitch(J), w_row(J, r0, col0, lane), (uint32_t)rb, &cs.bar[slot]);
}

__device__ inline void w_prologue(const FusedApply& fa, const GemmParams& p, const TileCoord& tc, int r0,
                                  int c_begin, int c_end, int lane, uint8_t* ebuf, uint32_t ek, CSlots& cs) {
  const GemmGroup& G = p.g[tc.g];
  if (r0 >= G.M) return;
  int k = 0;
  for (int ch = c_begin; ch < c_end && k < 2; ++ch) {
    if (tc.n0 + ch * kCW >= G.N) break;
    w_load(fa, p, tc, r0, ch, ebuf, (int)((ek + k) & 1), cs, lane);
    ++k;
  }
}

__device__ bool epilogue_apply(const GemmParams& p, const FusedApply& fa, const TileCoord& tc, int r0,
                               int c_begin, int c_end, uint32_t tacc, int q, int lane, uint8_t* ebuf,
                               uint32_t& ek, bool& bad, CSlots& cs, volatile int* abort_flag) {
  const GemmGroup& G = p.g[tc.g];
  if (r0 >= G.M) return true;
  const FusedApplyJob& J = fa_job(fa, G, tc);
  const float sb = p.s ? p.s[G.mat_base + tc.b] : 1.f;
  const float al = p.alpha * sb * J.scale;           // O = scale * X
  const float lr = fa.lr, wd = fa.wd;
  const int row = r0 + lane;
  const bool row_ok = row < G.M;
  const uint32_t trow = tacc + ((uint32_t)(q * 32) << 16);
  auto live = [&](int ch) { return tc.n0 + ch * kCW < G.N; };
  int ch = c_begin;
  if (!live(ch)) return true;
  uint32_t nr[16];
  tmem_ld_32x32b_x16_async(trow + ch * kCW, nr);
  while (ch < c_end && live(ch)) {
    const int col0 = tc.n0 + ch * kCW;
    const int nx = ch + 1 < c_end && live(ch + 1) ? ch + 1 : c_end;
    const int slot = (int)(ek & 1);
    uint8_t* sb8 = ebuf + slot * kSlot;
    const bool full = w_full(J, G, r0, col0);
    const int nrows = w_rows(J, G, r0, col0);
    if (full) {
      int ok = mbar_wait(&cs.bar[slot], (cs.par >> slot) & 1u, abort_flag) ? 1 : 0;
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        tmem_ld_wait();
        return false;
      }
      if (lane == 0) cs.pending &= ~(1u << slot);
      cs.par ^= 1u << slot;
    }
    tmem_ld_wait();
    reg_fence16(nr);
    float v[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] = al * __uint_as_float(nr[e]);
    if (nx < c_end) tmem_ld_32x32b_x16_async(trow + nx * kCW, nr);
    if (full && !J.transpose) {
      // the lane's own row: W[row][col0 .. col0 + 15]
      uint8_t* rp = sb8 + lane * 48;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        uint4 u = *reinterpret_cast<const uint4*>(rp + 16 * j);
        __nv_bfloat16* w8 = reinterpret_cast<__nv_bfloat16*>(&u);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float w = __bfloat162float(w8[e]);
          const float nw = fmaf(-lr, fmaf(wd, w, v[8 * j + e]), w);
          bad |= row_ok && !finite_f(nw);
          w8[e] = __float2bfloat16_rn(nw);
        }
        *reinterpret_cast<uint4*>(rp + 16 * j) = u;
      }
    } else if (full) {
      // W = X^T: slot row e holds W[col0 + e][r0 .. r0 + 31]; the lane's
      // values sit in column `lane` of every row
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        __nv_bfloat16* wp = reinterpret_cast<__nv_bfloat16*>(sb8 + e * 80 + 2 * lane);
        const float w = __bfloat162float(*wp);
        const float nw = fmaf(-lr, fmaf(wd, w, v[e]), w);
        bad |= e < nrows && !finite_f(nw);
        *wp = __float2bfloat16_rn(nw);
      }
    } else {
      // a segment cut by the matrix's edge: element by element
      __nv_bfloat16* w = reinterpret_cast<__nv_bfloat16*>(J.w);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int c = col0 + e;
        if (!row_ok || c >= G.N) continue;
        __nv_bfloat16* wp = J.transpose ? w + (long long)c * J.ld + row : w + (long long)row * J.ld + c;
        const float wv = __bfloat162float(*wp);
        const float nw = fmaf(-lr, fmaf(wd, wv, v[e]), wv);
        bad |= !finite_f(nw);
        *wp = __float2bfloat16_rn(nw);
      }
    }
    if (full) {
      fence_async_smem();
      __syncwarp();
      if (lane < nrows) {
        bulk_store_1d(w_row(J, r0, col0, lane), sb8 + lane * w_pitch(J), (uint32_t)w_row_bytes(J));
        bulk_commit();
      }
    }
    // the chunk two on takes its W into this slot once these stores have read it
    const int n2 = nx < c_end && nx + 1 < c_end && live(nx + 1) ? nx + 1 : c_end;
    if (n2 < c_end) w_load(fa, p, tc, r0, n2, ebuf, slot, cs, lane);
    ++ek;
    ch = nx;
  }
  return true;
}

// ------------------------------------------------------------ the kernel
// Roles: warp 0 produces (TMA), warp 1 issues the MMAs (one thread), warps
// 2-9 are the epilogue.  The CTAs run as tcgen05 .cta_group::2 pairs
// (clusters of two): the pair owns a 256 x 256 output tile, each CTA stages
// 128 rows of A and 128 rows (N values) of B per k-step, and both CTAs'
// copies complete on the first CTA's full barrier, whose producer alone
// arrives (expecting both CTAs' bytes).  The first CTA issues M = 256 MMAs
// into both CTAs' TMEM and multicasts its commits (mbarrier arrivals) to
// both; the epilogue warps of both CTAs release the first CTA's accumulator.
// A stage is 32 KB per CTA, so five fit beside the epilogue's 64 KB.
// Tiles are handed out dynamically: the first CTA's producer claims the next
// tile id from a zeroed per-launch counter and publishes it to every role of
// both CTAs through a kTS-deep shared-memory ring.
template <int TERMS, bool LO, int BK, int FMT, class AP>
__global__ void __launch_bounds__(kThreads, 1)
    ns_gemm_tc_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ TmaArgs tm,
                      const __grid_constant__ AP ap) {
  using C = Stages<TERMS, BM, 128, BK>;
  using KL = KLayout<BK>;
  constexpr bool SPLIT = TERMS == 3;     // the A operand's lo plane is staged
  constexpr bool BLO = TERMS >= 2;       // the B operand's lo plane is staged
  constexpr bool IN16 = FMT == kFmtF16;  // fp16 operands (else bf16)
  constexpr bool OUT16 = FMT != kFmtBf16;
  constexpr int TM_ROWS = 2 * BM;
  const uint32_t crank = cluster_ctarank();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* epi = smem + C::kStages * C::kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(epi + kEpiBytes);
  uint64_t* empty = full + 8;
  uint64_t* tfull = empty + 8;             // [2]
  uint64_t* tempty = tfull + 2;            // [2]
  uint64_t* drain = tempty + 2;            // [1]
  uint64_t* sfull = drain + 1;             // [kTS] tile id published
  uint64_t* sempty = sfull + kTS;          // [kTS] tile id read by every role
  uint64_t* cbar = sempty + kTS;           // [2 kEpiWarps] C box loads per epilogue slot
  int* sid = reinterpret_cast<int*>(cbar + 2 * kEpiWarps);   // [kTS]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sid + kTS);
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * kEpiWarps);
    }
    mbar_init(drain, 1);
    // readers of a ring slot: the producer and the epilogue warps of each
    // CTA (the first CTA's producer and MMA warp, the second's producer)
    for (int i = 0; i < kTS; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&sempty[i], 2 * (1 + kEpiWarps));
    }
    for (int i = 0; i < 2 * kEpiWarps; ++i) mbar_init(&cbar[i], 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int g = 0; g < p.ngroups; ++g) {
      prefetch_tmap(&tm.maps.a_hi[g]); prefetch_tmap(&tm.maps.b_hi[g]);
      if (SPLIT) prefetch_tmap(&tm.maps.a_lo[g]);
      if (BLO) prefetch_tmap(&tm.maps.b_lo[g]);
    }
  }
  if (warp == 1) { tmem_alloc_pair(tmem_slot, kTmemCols); tmem_relinquish_pair(); }
  tc_fence_before();
  __syncwarp();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  auto fail = [&]() {
    abort_flag = 1;
    set_status(p.status, MC_STATUS_TIMEOUT);
  };

  // Tile schedule: the first CTA's producer claims the next tile from the
  // launch's global counter and publishes its id in a kTS-deep ring (in both
  // CTAs); every role reads the seq-th id from the ring.  Tiles are numbered
  // heaviest group first, so claiming in order approximates
  // longest-processing-time-first scheduling.  -1 ends the sequence, -2 is a
  // wait timeout.
  const uint32_t sempty_r0 = mapa_shared(smem_u32(&sempty[0]), 0);
  auto take = [&](uint32_t seq) -> int {
    const int slot = (int)(seq % kTS);
    if (!mbar_wait_acq_cluster(&sfull[slot], (seq / kTS) & 1, &abort_flag)) return -2;
    const int t = reinterpret_cast<volatile int*>(sid)[slot];
    mbar_arrive_cluster(sempty_r0 + slot * 8);
    return t;
  };
  auto claim = [&](uint32_t seq) -> int {      // first CTA's producer
    const int slot = (int)(seq % kTS);
    if (!mbar_wait_acq_cluster(&sempty[slot], ((seq / kTS) & 1) ^ 1, &abort_flag)) return -2;
    int t = atomicAdd(p.sched, 1);
    if (t >= p.total_tiles) t = -1;
    sid[slot] = t;
    st_shared_cluster_u32(mapa_shared(smem_u32(&sid[slot]), 1), (uint32_t)t);
    mbar_arrive_cluster(mapa_shared(smem_u32(&sfull[slot]), 1));
    mbar_arrive(&sfull[slot]);
    return t;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t it = 0;
      uint32_t last_par[8] = {};
      bool used[8] = {};
      // the first CTA claims one tile ahead of its own loads, so the id of
      // the next tile is in the ring while this one's stages are loaded
      int ahead = crank == 0 ? claim(0) : 0;
      for (uint32_t seq = 0; !abort_flag; ++seq) {
        int t;
        if (crank == 0) {
          t = ahead;
          if (t >= 0) ahead = claim(seq + 1);
        } else {
          t = take(seq);
        }
        if (t == -2) { fail(); break; }
        if (t < 0) break;
        const TileCoord tc = tile_coord<TM_ROWS>(p, t);
        const GemmGroup& G = p.g[tc.g];
        const int nk = (G.K + BK - 1) / BK;
        const int m0 = tc.m0 + BM * (int)crank;
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
          const int k0 = kb * BK;
          // this CTA's 128 rows of A and of B, counted on the first CTA's
          // barrier; only the first CTA arrives (with both CTAs' bytes), so
          // the second CTA's copies need no cross-CTA arrive per stage (its
          // copies cannot complete the phase before that arrive)
          const uint32_t fb = mapa_shared(smem_u32(&full[s]), 0);
          if (crank == 0) mbar_arrive_expect_tx(&full[s], 2 * C::kStageBytes);
          const int nb = tc.n0 + 128 * (int)crank;
#pragma unroll
          for (int sub = 0; sub < KL::kSub; ++sub) {
            const int ks = k0 + sub * KL::kBX, so = sub * 128 * KL::kBX * 2;
            tma_load_3d_pair(a_hi + so, &tm.maps.a_hi[tc.g], fb, ks, m0, tc.b);
            if (SPLIT) tma_load_3d_pair(a_lo + so, &tm.maps.a_lo[tc.g], fb, ks, m0, tc.b);
          }
          if (!G.b_mn_major) {
#pragma unroll
            for (int sub = 0; sub < KL::kSub; ++sub) {
              const int ks = k0 + sub * KL::kBX, so = sub * 128 * KL::kBX * 2;
              tma_load_3d_pair(b_hi + so, &tm.maps.b_hi[tc.g], fb, ks, nb, tc.b);
              if (BLO) tma_load_3d_pair(b_lo + so, &tm.maps.b_lo[tc.g], fb, ks, nb, tc.b);
            }
          } else {
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {
              tma_load_3d_pair(b_hi + qq * (64 * BK * 2), &tm.maps.b_hi[tc.g], fb, nb + 64 * qq, k0, tc.b);
              if (BLO)
                tma_load_3d_pair(b_lo + qq * (64 * BK * 2), &tm.maps.b_lo[tc.g], fb, nb + 64 * qq, k0, tc.b);
            }
          }
          used[s] = true;
          last_par[s] = use & 1;
        }
        if (!ok) break;
      }
      // drain: every issued copy must have landed before the CTA may exit
      // (the first CTA's barriers count both CTAs' copies, and the second
      // CTA stays until the closing cluster barrier)
      if (crank == 0)
        for (int s = 0; s < C::kStages; ++s)
          if (used[s]) mbar_wait(&full[s], last_par[s], nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && crank == 0) {
      constexpr uint32_t idesc_k = make_idesc_16(2 * BM, BN, 0, 0, IN16 ? 1u : 0u);
      constexpr uint32_t idesc_mn = make_idesc_16(2 * BM, BN, 0, 1, IN16 ? 1u : 0u);
      uint32_t it = 0, tcount = 0;
      bool issued = false;
      for (uint32_t seq = 0; !abort_flag; ++seq, ++tcount) {
        const int t = take(seq);
        if (t == -2) { fail(); break; }
        if (t < 0) break;
        const TileCoord tc = tile_coord<TM_ROWS>(p, t);
        const GemmGroup& G = p.g[tc.g];
        const int nk = (G.K + BK - 1) / BK;
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
          for (int kk = 0; kk < BK / 16; ++kk) {
            // K-major: 16 elements = 32 bytes further along the swizzled row,
            // in sub-tile kk / (kBX / 16) of the stage
            const uint32_t ko = (uint32_t)((kk / (KL::kBX / 16)) * 128 * KL::kBX * 2 + (kk % (KL::kBX / 16)) * 32);
            const uint64_t dah = make_sdesc(a_hi + ko, 16, KL::kSbo, KL::kType);
            uint64_t dbh, dbl = 0, dal = 0;
            if (!G.b_mn_major) {
              dbh = make_sdesc(b_hi + ko, 16, KL::kSbo, KL::kType);
              if (BLO) dbl = make_sdesc(b_lo + ko, 16, KL::kSbo, KL::kType);
            } else {
              // MN-major (128-byte swizzle): 16 K-rows = two 1024-byte atoms;
              // 64-wide N blocks are 64*BK*2 bytes apart
              dbh = make_sdesc(b_hi + kk * 2048, 64 * BK * 2, 1024, 2);
              if (BLO) dbl = make_sdesc(b_lo + kk * 2048, 64 * BK * 2, 1024, 2);
            }
            const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
            if (SPLIT) dal = make_sdesc(a_lo + ko, 16, KL::kSbo, KL::kType);
            tc_mma_pair(d_tmem, dah, dbh, idesc, accum);
            if (BLO) tc_mma_pair(d_tmem, dah, dbl, idesc, 1u);
            if (SPLIT) tc_mma_pair(d_tmem, dal, dbh, idesc, 1u);
          }
          issued = true;
          // stage free (in both CTAs of the pair) once these MMAs have read it
          tc_commit_pair_mc(&empty[s], 0x3);
        }
        if (!ok) break;
        // accumulator ready for the epilogue of both CTAs
        tc_commit_pair_mc(&tfull[acc], 0x3);
      }
      if (issued) {                      // all issued MMAs complete before teardown
        tc_commit_pair_mc(drain, 0x1);
        mbar_wait(drain, 0, nullptr);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int e = warp - 2;
    const int q = warp & 3;              // TMEM lane quadrant of this warp
    const int hc = e >> 2;               // column half: chunks [4 hc, 4 hc + 4)
    uint8_t* ebuf = epi + e * kEpiWarpBytes;
    uint32_t ek = 0;
    bool bad = false;
    uint32_t tcount = 0;
    CSlots cs{cbar + 2 * e, 0u, 0u};
    for (uint32_t seq = 0;; ++seq, ++tcount) {
      int t = 0;
      if (lane == 0) t = take(seq);
      t = __shfl_sync(0xffffffffu, t, 0);
      if (t == -2) { if (lane == 0) fail(); break; }
      if (t < 0) break;
      const TileCoord tc = tile_coord<TM_ROWS>(p, t);
      const int acc = tcount & 1;
      const int r0 = tc.m0 + BM * (int)crank + q * 32;
      const int c0 = hc * (BN / 2 / kCW), c1 = (hc + 1) * (BN / 2 / kCW);
      // C (or W) of this tile: the first two chunks' boxes now, every C row
      // into L2, while the MMAs still run
      if constexpr (AP::kOn) {
        w_prologue(ap, p, tc, r0, c0, c1, lane, ebuf, ek, cs);
      } else {
        c_prologue<LO>(p, tm, tc, r0, c0, c1, lane, ebuf, ek, cs);
        prefetch_c_rows<LO>(p, tc, r0, c0, c1, lane);
      }
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&tfull[acc], (tcount >> 1) & 1, &abort_flag) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) { if (lane == 0) fail(); break; }
      tc_fence_after();
      bool eok;
      if constexpr (AP::kOn)
        eok = epilogue_apply(p, ap, tc, r0, c0, c1, tmem_base + acc * BN, q, lane, ebuf, ek, bad, cs, &abort_flag);
      else
        eok = epilogue_rows<LO, IN16, OUT16>(p, tm, tc, r0, c0, c1, tmem_base + acc * BN, q, lane, ebuf, ek,
                                             bad, cs, &abort_flag);
      if (!eok) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));   // the first CTA's MMA
      }
    }
    // C boxes still in flight (only after a failed wait) land before exit
    if (lane == 0)
      for (int sl = 0; sl < 2; ++sl)
        if (cs.pending & (1u << sl)) mbar_wait(&cs.bar[sl], (cs.par >> sl) & 1u, nullptr);
    bulk_wait0();                        // every store of this warp (fused apply: every lane's) completes
    if (bad) set_status(p.status, MC_STATUS_NONFINITE_UPDATE);
  }

  tc_fence_before();
  __syncwarp();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
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
// swizzle 128 B (box_cols 64) or 64 B (box_cols 32), zero fill (loads) and
// clipping (stores) outside [cols, rows, batch].
bool encode_3d(CUtensorMap* m, const void* base, int cols, int rows, int batch, long long ld,
               long long bstride, int box_cols, int box_rows, bool f16, char* err, size_t errlen) {
  EncodeTiledFn enc = get_encode();
  if (!enc) { snprintf(err, errlen, "cuTensorMapEncodeTiled unavailable"); return false; }
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)batch};
  cuuint64_t strides[2] = {(cuuint64_t)ld * 2, (cuuint64_t)bstride * 2};
  cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  const CUtensorMapSwizzle sw = box_cols == 64   ? CU_TENSOR_MAP_SWIZZLE_128B
                                : box_cols == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                 : CU_TENSOR_MAP_SWIZZLE_32B;
  CUresult r = enc(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(err, errlen, "cuTensorMapEncodeTiled failed (%d): cols=%d rows=%d batch=%d ld=%lld",
             (int)r, cols, rows, batch, ld);
    return false;
  }
  return true;
}

// Operand maps (A rows of a_rows, B rows of b_rows per box) and the 32 x 32
// epilogue store maps for D.  a_lo: the A operand's lo plane is read; b_lo:
// the B operand's; lo: D is stored as (hi, lo); in16 / out16: operand and
// output planes hold fp16 (else bf16).
bool encode_all(const GemmParams& p, TmaArgs& tm, bool a_lo, bool b_lo, bool lo, bool in16, bool out16,
                int a_rows, int b_rows, int bk, int bx, char* err, size_t errlen) {
  memset(&tm, 0, sizeof(tm));
  for (int g = 0; g < p.ngroups; ++g) {
    const GemmGroup& G = p.g[g];
    if (!encode_3d(&tm.maps.a_hi[g], G.a_hi, G.K, G.M, G.batch, G.lda, G.a_bstride, bx, a_rows, in16, err, errlen)) return false;
    if (a_lo && !encode_3d(&tm.maps.a_lo[g], G.a_lo, G.K, G.M, G.batch, G.lda, G.a_bstride, bx, a_rows, in16, err, errlen)) return false;
    if (!G.b_mn_major) {   // B operand: rows of an [N, K] plane, boxes bx wide
      if (!encode_3d(&tm.maps.b_hi[g], G.b_hi, G.K, G.N, G.batch, G.ldb, G.b_bstride, bx, b_rows, in16, err, errlen)) return false;
      if (b_lo && !encode_3d(&tm.maps.b_lo[g], G.b_lo, G.K, G.N, G.batch, G.ldb, G.b_bstride, bx, b_rows, in16, err, errlen)) return false;
    } else {               // B operand: [K, N] plane, 64-wide N boxes of bk rows
      if (!encode_3d(&tm.maps.b_hi[g], G.b_hi, G.N, G.K, G.batch, G.ldb, G.b_bstride, 64, bk, in16, err, errlen)) return false;
      if (b_lo && !encode_3d(&tm.maps.b_lo[g], G.b_lo, G.N, G.K, G.batch, G.ldb, G.b_bstride, 64, bk, in16, err, errlen)) return false;
    }
    // D chunks of 16 columns x 32 rows; their mirrors 32 columns x 16 rows
    if (!encode_3d(&tm.maps.d_hi[g], G.d_hi, G.N, G.M, G.batch, G.ldd, G.d_bstride, 16, 32, out16, err, errlen)) return false;
    if (lo && !encode_3d(&tm.maps.d_lo[g], G.d_lo, G.N, G.M, G.batch, G.ldd, G.d_bstride, 16, 32, out16, err, errlen)) return false;
    if (G.symmetric) {
      if (!encode_3d(&tm.maps.dm_hi[g], G.d_hi, G.N, G.M, G.batch, G.ldd, G.d_bstride, 32, 16, out16, err, errlen)) return false;
      if (lo && !encode_3d(&tm.maps.dm_lo[g], G.d_lo, G.N, G.M, G.batch, G.ldd, G.d_bstride, 32, 16, out16, err, errlen)) return false;
    }
    // C of a non-symmetric output is read by the epilogue through TMA, in the
    // operands' format
    if (p.beta != 0.f && !G.symmetric) {
      if (!encode_3d(&tm.maps.c_hi[g], G.c_hi, G.N, G.M, G.batch, G.ldc, G.c_bstride, 16, 32, in16, err, errlen)) return false;
      if (lo && !encode_3d(&tm.maps.c_lo[g], G.c_lo, G.N, G.M, G.batch, G.ldc, G.c_bstride, 16, 32, in16, err, errlen)) return false;
    }
  }
  return true;
}

template <int TERMS, bool LO, int BK, int FMT, class AP = NoApply>
cudaError_t launch_pairs(const GemmParams& p, const AP& ap, cudaStream_t s, char* err, size_t errlen) {
  TmaArgs tm;
  // each CTA's B box is its 128-row half of the pair's 256 B rows
  if (!encode_all(p, tm, TERMS == 3, TERMS >= 2, LO, FMT == kFmtF16, FMT != kFmtBf16, BM, 128, BK,
                  KLayout<BK>::kBX, err, errlen))
    return cudaErrorInvalidValue;
  auto k = ns_gemm_tc_kernel<TERMS, LO, BK, FMT, AP>;
  const int smem = Stages<TERMS, BM, 128, BK>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  static int max_clusters = 0;
  if (max_clusters == 0) {
    cfg.gridDim = dim3(2 * (sm_count() / 2));
    if (cudaOccupancyMaxActiveClusters(&max_clusters, k, &cfg) != cudaSuccess || max_clusters <= 0)
      max_clusters = sm_count() / 2;
  }
  const int units = p.total_tiles < max_clusters ? p.total_tiles : max_clusters;
  cfg.gridDim = dim3(2 * units);
  e = cudaLaunchKernelEx(&cfg, k, p, tm, ap);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// One layout: CTA pairs.  Operand rows are 128-byte swizzled boxes of 64
// K-elements; three-product launches take 64-deep k-steps (three 64 KB stages,
// twelve MMAs per stage), two-product ones 64-deep k-steps too (A's hi plane
// and both planes of B: four 48 KB stages, eight MMAs per stage), one-product
// launches 128-deep ones (two boxes per operand per stage, eight MMAs, three
// 64 KB stages): the single issuing thread's per-stage cost is then spread
// over more MMAs (measured: 32-deep one-product stages took 48 % longer than
// 64-deep, 128-deep ones 4-9 % less; 64-deep three-product stages 5-9 % less
// than 32-deep).  Two products run only on fp16 planes (a last update).
template <int FMT>
cudaError_t launch_fmt(const GemmParams& p, const FusedApply* fa, cudaStream_t s, char* err, size_t errlen) {
  if (p.terms == 3) {
    if constexpr (FMT != kFmtBf16)
      if (fa) return launch_pairs<3, true, 64, FMT, FusedApply>(p, *fa, s, err, errlen);
    return launch_pairs<3, true, 64, FMT>(p, NoApply{}, s, err, errlen);
  }
  if (p.terms == 2) {
    if constexpr (FMT == kFmtF16) {
      if (fa) return launch_pairs<2, true, 64, FMT, FusedApply>(p, *fa, s, err, errlen);
      return launch_pairs<2, true, 64, FMT>(p, NoApply{}, s, err, errlen);
    }
    snprintf(err, errlen, "two products per k-step run on fp16 planes only");
    return cudaErrorInvalidValue;
  }
  return launch_pairs<1, true, 128, FMT>(p, NoApply{}, s, err, errlen);
}

}  // namespace

cudaError_t launch_ns_gemm_tc(const GemmParams& p, const FusedApply* fa, cudaStream_t s, char* err,
                              size_t errlen) {
  if (p.total_tiles <= 0) return cudaSuccess;
  if (fa && (p.xmode != kXSplit || p.terms < 2 || p.fmt == kFmtBf16 || p.beta != 0.f || p.g[0].symmetric)) {
    snprintf(err, errlen, "the fused apply runs in a two- or three-product, fp16-output update launch");
    return cudaErrorInvalidValue;
  }
  if (!p.sched) {
    snprintf(err, errlen, "tensor-core GEMM launched without a tile counter");
    return cudaErrorInvalidValue;
  }
  if (p.xmode != kXSplit) {            // one bf16 plane, one product
    if (p.terms != 1 || p.fmt != kFmtBf16) {
      snprintf(err, errlen, "plain bf16 planes take one bf16 product");
      return cudaErrorInvalidValue;
    }
    return launch_pairs<1, false, 128, kFmtBf16>(p, NoApply{}, s, err, errlen);
  }
  switch (p.fmt) {
    case kFmtBf16: return launch_fmt<kFmtBf16>(p, nullptr, s, err, errlen);
    case kFmtBf16ToF16: return launch_fmt<kFmtBf16ToF16>(p, fa, s, err, errlen);
    default: return launch_fmt<kFmtF16>(p, fa, s, err, errlen);
  }
}

}  // namespace mc
