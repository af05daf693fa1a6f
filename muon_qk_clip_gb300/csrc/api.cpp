// C ABI of the MuonClip library: argument validation, workspace planning and
// launch sequencing.  Every check runs on the host before the first launch.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <memory>
#include <string>
#include <vector>

#include "../../include/muonclip.h"
#include "kernels.h"

using namespace mc;

namespace {

thread_local std::string g_last_error;

mc_status fail(mc_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

mc_status ok() {
  g_last_error.clear();
  return MC_OK;
}

mc_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ------------------------------------------------------------------ profiler
enum ProfClass { kPrep, kNorms, kGemm, kApply, kClip, kMaxLogit, kAttnFwd, kNumProf };
const char* kProfNames[kNumProf] = {"prep", "norms", "ns_gemm", "apply", "clip", "max_logit", "attn_fwd"};

struct Profiler {
  bool on = false;
  struct Rec { int cls; int launches; cudaEvent_t a, b; };
  std::vector<Rec> pending;
  std::vector<cudaEvent_t> pool;
  double ms[kNumProf] = {0};
  long long launches[kNumProf] = {0};
  cudaEvent_t get() {
    if (!pool.empty()) { cudaEvent_t e = pool.back(); pool.pop_back(); return e; }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }
  void drain() {
    for (Rec& r : pending) {
      float t = 0.f;
      if (cudaEventSynchronize(r.b) == cudaSuccess && cudaEventElapsedTime(&t, r.a, r.b) == cudaSuccess)
        ms[r.cls] += t;
      launches[r.cls] += r.launches;
      pool.push_back(r.a);
      pool.push_back(r.b);
    }
    pending.clear();
  }
};
Profiler g_prof;

struct ProfScope {
  int cls, n;
  cudaStream_t s;
  cudaEvent_t a = nullptr;
  ProfScope(int cls_, int n_, cudaStream_t s_) : cls(cls_), n(n_), s(s_) {
    if (g_prof.on) { a = g_prof.get(); cudaEventRecord(a, s); }
  }
  ~ProfScope() {
    if (a) {
      cudaEvent_t b = g_prof.get();
      cudaEventRecord(b, s);
      g_prof.pending.push_back({cls, n, a, b});
      if (g_prof.pending.size() > 4096) g_prof.drain();
    }
  }
};

size_t dtype_size(int32_t d) { return d == MC_BF16 ? 2 : 4; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

mc_status check_mat(const mc_mat& m, const char* name, int idx, bool allow_bf16, bool allow_f32) {
  if (!m.ptr) return fail(MC_ERR_INVALID_ARG, "%s[%d]: null pointer", name, idx);
  if (m.dtype != MC_F32 && m.dtype != MC_BF16)
    return fail(MC_ERR_INVALID_ARG, "%s[%d]: unknown dtype %d", name, idx, m.dtype);
  if ((m.dtype == MC_BF16 && !allow_bf16) || (m.dtype == MC_F32 && !allow_f32))
    return fail(MC_ERR_INVALID_ARG, "%s[%d]: dtype %s not accepted here", name, idx,
                m.dtype == MC_BF16 ? "bf16" : "f32");
  if (m.rows < 1 || m.cols < 1 || m.rows > (1 << 30) || m.cols > (1 << 30))
    return fail(MC_ERR_INVALID_ARG, "%s[%d]: bad shape %lld x %lld", name, idx, (long long)m.rows,
                (long long)m.cols);
  if (m.ld < m.cols)
    return fail(MC_ERR_INVALID_ARG, "%s[%d]: ld %lld < cols %lld", name, idx, (long long)m.ld,
                (long long)m.cols);
  if (!aligned16(m.ptr) || (m.ld * (int64_t)dtype_size(m.dtype)) % 16 != 0)
    return fail(MC_ERR_INVALID_ARG, "%s[%d]: pointer and row pitch must be 16-byte aligned", name,
                idx);
  return MC_OK;
}

mc_status check_hparams(const mc_hparams* hp) {
  if (!hp) return fail(MC_ERR_INVALID_ARG, "hparams: null");
  if (!std::isfinite(hp->mu) || !std::isfinite(hp->lr) || !std::isfinite(hp->weight_decay) ||
      !std::isfinite(hp->rms_scale) || !std::isfinite(hp->ns_a) || !std::isfinite(hp->ns_b) ||
      !std::isfinite(hp->ns_c) || !std::isfinite(hp->ns_eps))
    return fail(MC_ERR_INVALID_ARG, "hparams: non-finite value");
  if (hp->ns_steps < 0 || hp->ns_steps > 32)
    return fail(MC_ERR_INVALID_ARG, "hparams: ns_steps %d outside [0, 32]", hp->ns_steps);
  if (hp->ns_eps < 0.f) return fail(MC_ERR_INVALID_ARG, "hparams: ns_eps < 0");
  if (!(hp->tau > 0.f) || !std::isfinite(hp->tau))
    return fail(MC_ERR_INVALID_ARG, "hparams: tau must be finite and > 0");
  if (!(hp->alpha >= 0.f && hp->alpha <= 1.f))
    return fail(MC_ERR_INVALID_ARG, "hparams: alpha outside [0, 1]");
  if (hp->ns_precision < MC_NS_AUTO || hp->ns_precision > MC_NS_FP32)
    return fail(MC_ERR_INVALID_ARG, "hparams: unknown ns_precision %d", hp->ns_precision);
  if (hp->scale_mode != MC_SCALE_RMS && hp->scale_mode != MC_SCALE_SPECTRAL)
    return fail(MC_ERR_INVALID_ARG, "hparams: unknown scale_mode %d", hp->scale_mode);
  if (hp->ns_fast_steps < 0 || hp->ns_fast_steps > 32)
    return fail(MC_ERR_INVALID_ARG, "hparams: ns_fast_steps %d outside [0, 32]", hp->ns_fast_steps);
  return MC_OK;
}

// ------------------------------------------------------------------ planning
constexpr size_t kAlign = 1024;
size_t al(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Group {
  int m, n, batch;
  std::vector<int> mats;                // matrix indices
  long long ldn, ldm;                   // pitches (elements) of [m, n] and [m, m] planes
  size_t x[2][2], a[2], b[2];           // byte offsets: x[iterate][plane], a[plane], b[plane]
};

struct Plan {
  int xmode = kXSplit;
  int count = 0;
  std::vector<int> m, n, transpose, group, slot;  // per matrix
  std::vector<Group> groups;
  std::vector<int> tile_begin, tile_count;        // prep tiles per matrix
  int total_tiles = 0;
  size_t off_partials = 0, off_inv = 0, off_inv_sq = 0, bytes = 0;
  size_t off_sched = 0;                           // tile counters, one per NS GEMM launch
  int nsched = 0;
};

int resolve_xmode(int prec, bool any_f32_output) {
  switch (prec) {
    case MC_NS_SPLIT_BF16: return kXSplit;
    case MC_NS_BF16: return kXBf16;
    case MC_NS_FP32: return kXF32;
    default: return any_f32_output ? kXF32 : kXSplit;
  }
}

Plan make_plan(const mc_mat* mats, int count, int xmode) {
  Plan P;
  P.xmode = xmode;
  P.count = count;
  P.m.resize(count); P.n.resize(count); P.transpose.resize(count);
  P.group.resize(count); P.slot.resize(count);
  P.tile_begin.resize(count); P.tile_count.resize(count);
  std::map<std::pair<int, int>, int> gid;
  for (int j = 0; j < count; ++j) {
    const int r = (int)mats[j].rows, c = (int)mats[j].cols;
    P.transpose[j] = r > c;
    P.m[j] = std::min(r, c);
    P.n[j] = std::max(r, c);
    auto key = std::make_pair(P.m[j], P.n[j]);
    auto it = gid.find(key);
    if (it == gid.end()) {
      Group g;
      g.m = P.m[j]; g.n = P.n[j]; g.batch = 0;
      gid[key] = (int)P.groups.size();
      P.groups.push_back(g);
      it = gid.find(key);
    }
    Group& g = P.groups[it->second];
    P.group[j] = it->second;
    P.slot[j] = g.batch++;
    g.mats.push_back(j);
    P.tile_begin[j] = P.total_tiles;
    P.tile_count[j] = (int)(cdiv(r, 64) * cdiv(c, 64));
    P.total_tiles += P.tile_count[j];
  }
  const size_t es = xmode == kXF32 ? 4 : 2;
  const int planes = xmode == kXSplit ? 2 : 1;
  size_t off = 0;
  for (Group& g : P.groups) {
    g.ldn = round_up(g.n, 8);
    g.ldm = round_up(g.m, 8);
    const size_t xb = al((size_t)g.batch * g.m * g.ldn * es);
    const size_t ab = al((size_t)g.batch * g.m * g.ldm * es);
    for (int i = 0; i < 2; ++i)
      for (int pl = 0; pl < 2; ++pl) {
        g.x[i][pl] = off;
        if (pl < planes) off += xb;
      }
    for (int pl = 0; pl < 2; ++pl) { g.a[pl] = off; if (pl < planes) off += ab; }
    for (int pl = 0; pl < 2; ++pl) { g.b[pl] = off; if (pl < planes) off += ab; }
  }
  P.off_partials = off; off += al((size_t)P.total_tiles * sizeof(double));
  P.off_inv = off; off += al((size_t)count * sizeof(float));
  P.off_inv_sq = off; off += al((size_t)count * sizeof(float));
  // up to 32 iterations x 3 phases x (ceil(groups / kMaxGroups) + 3) launches
  // (the groups may be split over two streams and by products per k-step)
  P.nsched = 3 * 32 * ((int)cdiv((long long)P.groups.size(), kMaxGroups) + 3);
  P.off_sched = off; off += al((size_t)P.nsched * sizeof(int));
  P.bytes = off;
  return P;
}

char* wsp(void* ws, size_t off) { return static_cast<char*>(ws) + off; }

// plane pointer of matrix j inside its group's batch
void* x_plane(const Plan& P, void* ws, int j, int it, int pl) {
  const Group& g = P.groups[P.group[j]];
  const size_t es = P.xmode == kXF32 ? 4 : 2;
  return wsp(ws, g.x[it][pl]) + (size_t)P.slot[j] * g.m * g.ldn * es;
}

// ------------------------------------------------------------------ launches
mc_status run_prep(const Plan& P, void* ws, mc_mat* M, const mc_mat* G, bool do_momentum,
                   bool write_x, float mu, int32_t* status, cudaStream_t s) {
  for (int j0 = 0; j0 < P.count; j0 += kMaxJobs) {
    const int nj = std::min(kMaxJobs, P.count - j0);
    PrepParams pp;
    memset(&pp, 0, sizeof pp);
    pp.njobs = nj;
    pp.do_momentum = do_momentum;
    pp.write_x = write_x;
    pp.xmode = P.xmode;
    pp.mu = mu;
    pp.status = status;
    pp.partials = write_x ? reinterpret_cast<double*>(wsp(ws, P.off_partials)) + P.tile_begin[j0]
                          : nullptr;
    int t = 0;
    for (int q = 0; q < nj; ++q) {
      const int j = j0 + q;
      PrepJob& jb = pp.jobs[q];
      jb.M = static_cast<float*>(M[j].ptr);
      jb.ldM = M[j].ld;
      if (G) { jb.G = G[j].ptr; jb.ldG = G[j].ld; jb.g_bf16 = G[j].dtype == MC_BF16; }
      jb.rows = (int)M[j].rows;
      jb.cols = (int)M[j].cols;
      jb.transpose = P.transpose[j];
      if (write_x) {
        jb.xh = x_plane(P, ws, j, 0, 0);
        jb.xl = x_plane(P, ws, j, 0, 1);
        jb.ldx = P.groups[P.group[j]].ldn;
      }
      jb.tile_begin = t;
      jb.tiles_c = (int)cdiv(jb.cols, 64);
      t += (int)(cdiv(jb.rows, 64) * jb.tiles_c);
    }
    pp.total_tiles = t;
    ProfScope ps(kPrep, 1, s);
    cudaError_t e = launch_prep(pp, s);
    if (e != cudaSuccess) return cuda_fail(e, "momentum/prep launch");
  }
  return MC_OK;
}

mc_status run_norms(const Plan& P, void* ws, float eps, cudaStream_t s) {
  ProfScope ps(kNorms, (P.count + kMaxNormMats - 1) / kMaxNormMats, s);
  cudaError_t e = launch_norms(reinterpret_cast<double*>(wsp(ws, P.off_partials)),
                               P.tile_begin.data(), P.tile_count.data(), P.count, eps,
                               reinterpret_cast<float*>(wsp(ws, P.off_inv)),
                               reinterpret_cast<float*>(wsp(ws, P.off_inv_sq)), s);
  if (e != cudaSuccess) return cuda_fail(e, "norm launch");
  return MC_OK;
}

// One Newton-Schulz phase over every group (chunks of kMaxGroups).
enum Phase { kGram = 1, kPoly = 2, kNext = 3 };

// The split Newton-Schulz plan.  Iteration 0 reads the iterate prep wrote
// from the raw momentum, whose scale is arbitrary, so it works on bf16 planes
// (fp32's exponent range); its update multiplies by 1/||M|| and stores X1 as
// fp16 (hi, lo) planes, and every later iteration works on fp16 planes:
// entries are then bounded (singular values stay below ~1.2) and fp16's 11
// significand bits make a one-product (hi*hi) step 8x more accurate than
// bf16's.  The leading iterations take one product per k-step; the trailing
// ones take one in the Gram, three (hi*hi + hi*lo + lo*hi) in the polynomial
// and two or three in the update (below).
//
// Float64 emulation of this arithmetic (max error / RMS of the exact result;
// the bound is 2e-2) over Gaussian inputs and adversarial spectra (64, 16 or 4
// unit directions over a 1e-3 rest), sides 64 to 2048 x 16384:
//   - three leading one-product iterations (ns_fast_steps = 3) with
//     three-product trailing iterations: at most 8.2e-3 from a smaller side
//     of 256 (512 x 16384 Gaussian), 1.4e-2 at 64; so the one-product
//     iterations run from a smaller side of kFastMinSide and smaller matrices
//     take three products in every phase (2.8e-3 at 64);
//   - the updates of the two trailing iterations may then drop lo(B') x hi(X),
//     B' = a I + b A + c A^2: at most 1.4e-2 from a smaller side of 512
//     (2048 x 16384 adversarial, 64 directions: 1.37e-2 against 7.9e-3 with
//     three products; 512 x 16384 Gaussian: 9.3e-3), so they take two
//     products (hi*hi + hi*lo of X) from kTrail2MinSide (1.3e-2 already at
//     256 x 2048).  Dropping hi(B') x lo(X) instead gives ~2e-2;
//   - a fourth one-product iteration is not offered: 2.0-2.3e-2 at 1024 x 4096
//     and 1024 x 16384 Gaussian, for ~1 % of a call once the trailing updates
//     take two products.
constexpr int kFastMinSide = 256;
constexpr int kTrail2MinSide = 512;

// Leading one-product iterations of a shape group whose smaller side is
// `side`: up to three, with at least two three-term iterations after them.
int ns_fast_iterations(const mc_hparams* hp, int side) {
  if (side < kFastMinSide) return 0;
  return std::min({hp->ns_fast_steps, 3, std::max(0, hp->ns_steps - 2)});
}

// Products per k-step (1: hi*hi; 2: hi*hi + hi*lo_B; 3: hi*hi + hi*lo +
// lo*hi) of phase `ph` of iteration `it` on the split iterate.  Two in the
// updates of the last two iterations (three-term: the leading one-product
// iterations always leave two), on fp16 planes (it >= 1).
int ns_terms(const mc_hparams* hp, int side, int it, int ph) {
  const int nf = ns_fast_iterations(hp, side);
  if (it < nf) return 1;
  if (ph == kGram && side >= kFastMinSide) return 1;
  if (ph == kNext && it >= 1 && it >= hp->ns_steps - 2 && side >= kTrail2MinSide) return 2;
  return 3;
}

// 16-bit formats of phase `ph` of iteration `it`: bf16 in iteration 0 (its
// update stores X1 as fp16), fp16 after it; plain bf16 planes throughout.
int ns_fmt(int xmode, int it, int ph) {
  if (xmode != kXSplit) return kFmtBf16;
  if (it == 0) return ph == kNext ? kFmtBf16ToF16 : kFmtBf16;
  return kFmtF16;
}

mc_status run_phase(const Plan& P, void* ws, Phase ph, int it, const mc_hparams* hp,
                    int32_t* status, int& launch, const std::vector<int>& groups, cudaStream_t s,
                    const FusedApply* fa) {
  const int cur = it & 1, nxt = cur ^ 1;
  const size_t es = P.xmode == kXF32 ? 4 : 2;
  // heavier K first for a better tail
  std::vector<int> order(groups);
  std::stable_sort(order.begin(), order.end(), [&](int x, int y) {
    const Group &a = P.groups[x], &b = P.groups[y];
    return (ph == kGram ? a.n : a.m) > (ph == kGram ? b.n : b.m);
  });
  // products per k-step of this launch kind (ns_terms; 1 off the split iterate)
  auto terms_of = [&](int g) {
    if (P.xmode != kXSplit) return 1;
    return ns_terms(hp, std::min(P.groups[g].m, P.groups[g].n), it, ph);
  };
  const bool sym_out = P.xmode != kXF32 && (ph == kGram || ph == kPoly);
  for (int terms : {1, 2, 3}) {
    std::vector<int> sub;                    // the groups of this launch kind
    for (int g : order)
      if (terms_of(g) == terms) sub.push_back(g);
    // output tiles: 256 x 256 per CTA pair (tensor cores), 64 x 64 (fp32)
    const int tileM = P.xmode != kXF32 ? kTcTileM : 64, tileN = P.xmode != kXF32 ? kTcTileN : 64;
    const int sym_step = 1;
    for (size_t g0 = 0; g0 < sub.size(); g0 += kMaxGroups) {
      GemmParams gp;
      memset(&gp, 0, sizeof gp);
      gp.xmode = P.xmode;
      gp.status = status;
      int t = 0, ng = 0;
      for (size_t q = g0; q < sub.size() && ng < kMaxGroups; ++q, ++ng) {
        const Group& g = P.groups[sub[q]];
        GemmGroup& G = gp.g[ng];
        const long long xs = (long long)g.m * g.ldn, as = (long long)g.m * g.ldm;
        auto X = [&](int i, int pl) { return (const void*)wsp(ws, g.x[i][pl]); };
        G.batch = g.batch;
        G.mat_base = g.mats[0];   // matrices of a group are contiguous in s[] order
        switch (ph) {
          case kGram:
            G.M = g.m; G.N = g.m; G.K = g.n;
            G.a_hi = X(cur, 0); G.a_lo = X(cur, 1); G.lda = g.ldn; G.a_bstride = xs;
            G.b_hi = X(cur, 0); G.b_lo = X(cur, 1); G.ldb = g.ldn; G.b_bstride = xs;
            G.d_hi = wsp(ws, g.a[0]); G.d_lo = wsp(ws, g.a[1]); G.ldd = g.ldm; G.d_bstride = as;
            break;
          case kPoly:
            G.M = g.m; G.N = g.m; G.K = g.m;
            G.a_hi = wsp(ws, g.a[0]); G.a_lo = wsp(ws, g.a[1]); G.lda = g.ldm; G.a_bstride = as;
            G.b_hi = G.a_hi; G.b_lo = G.a_lo; G.ldb = g.ldm; G.b_bstride = as;
            G.c_hi = G.a_hi; G.c_lo = G.a_lo; G.ldc = g.ldm; G.c_bstride = as;
            G.d_hi = wsp(ws, g.b[0]); G.d_lo = wsp(ws, g.b[1]); G.ldd = g.ldm; G.d_bstride = as;
            break;
          case kNext:
            G.M = g.m; G.N = g.n; G.K = g.m;
            G.a_hi = wsp(ws, g.b[0]); G.a_lo = wsp(ws, g.b[1]); G.lda = g.ldm; G.a_bstride = as;
            G.b_hi = X(cur, 0); G.b_lo = X(cur, 1); G.ldb = g.ldn; G.b_bstride = xs;
            G.b_mn_major = 1;
            G.c_hi = X(cur, 0); G.c_lo = X(cur, 1); G.ldc = g.ldn; G.c_bstride = xs;
            G.d_hi = wsp(ws, g.x[nxt][0]); G.d_lo = wsp(ws, g.x[nxt][1]); G.ldd = g.ldn;
            G.d_bstride = xs;
            break;
        }
        G.tiles_m = (int)cdiv(G.M, tileM);
        G.tiles_n = (int)cdiv(G.N, tileN);
        G.tiles_per_item = G.tiles_m * G.tiles_n;
        // Gram and polynomial outputs are symmetric: the tensor-core path
        // computes only the tiles touching the upper triangle
        if (sym_out) {
          G.symmetric = 1;
          G.tiles_per_item = 0;
          for (int tn = 0; tn < G.tiles_n; ++tn)
            G.tiles_per_item += std::min(G.tiles_m, (tn + 1) * sym_step);
        }
        G.tile_begin = t;
        t += G.tiles_per_item * G.batch;
        (void)es;
      }
      gp.ngroups = ng;
      gp.total_tiles = t;
      // tensor-core launches claim tiles from a zeroed counter of their own
      if (P.xmode != kXF32) {
        if (launch >= P.nsched)
          return fail(MC_ERR_UNSUPPORTED, "Newton-Schulz plan needs more than %d tile counters", P.nsched);
        gp.sched = reinterpret_cast<int*>(wsp(ws, P.off_sched)) + launch;
      }
      ++launch;
      gp.terms = terms;
      gp.fmt = ns_fmt(P.xmode, it, ph);
      // a one-product iteration's update reads only the polynomial's hi
      // plane (its a X term comes from X), so that lo plane is not stored
      gp.d_hi_only = P.xmode == kXSplit && ph == kPoly && terms == 1;
      // Three-term iterations fold a X into the polynomial: B' = c A^2 + b A + a I
      // and X' = B' X (two or three products), so the last phase reads no C.
      // (B' holds ~16 significand bits there; a one-plane B' would lose the
      // small singular values, so the other iterations keep X' = B X + a X.)
      const bool fold = P.xmode == kXSplit && gp.terms >= 2;
      switch (ph) {
        case kGram:
          gp.alpha = 1.f; gp.beta = 0.f;
          gp.s = it == 0 ? reinterpret_cast<const float*>(wsp(ws, P.off_inv_sq)) : nullptr;
          break;
        case kPoly:
          gp.alpha = hp->ns_c; gp.beta = hp->ns_b; gp.s = nullptr;
          gp.diag = fold ? hp->ns_a : 0.f;
          break;
        case kNext:
          gp.alpha = 1.f; gp.beta = fold ? 0.f : hp->ns_a;
          gp.s = it == 0 ? reinterpret_cast<const float*>(wsp(ws, P.off_inv)) : nullptr;
          break;
      }
      cudaError_t e;
      if (P.xmode == kXF32) {
        e = launch_ns_gemm_f32(gp, s);
      } else {
        char err[256] = {0};
        // the last update applies the step itself when the caller's W allow it
        const bool apply_here = fa && ph == kNext && it == hp->ns_steps - 1;
        e = launch_ns_gemm_tc(gp, apply_here ? fa : nullptr, s, err, sizeof err);
        if (e != cudaSuccess && err[0]) return fail(MC_ERR_CUDA, "tensor-core GEMM: %s", err);
      }
      if (e != cudaSuccess) return cuda_fail(e, "Newton-Schulz GEMM launch");
    }
  }
  return MC_OK;
}

// The GEMM epilogue addresses per-matrix scales as s[mat_base + slot], so the
// entry points first permute the matrices into shape-group order
// (group_order), which makes every group's members consecutive.
// A second stream for Newton-Schulz (one per host thread and device, created
// on first use and kept): shape groups are independent chains of launches, so
// running two sets of them side by side lets one set's launches fill the SMs
// that the other's launch tails leave idle.
struct AuxStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

cudaError_t aux_stream(AuxStream*& out) {
  thread_local std::map<int, AuxStream> cache;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  AuxStream& a = cache[dev];
  if (!a.s) {
    if ((e = cudaStreamCreateWithFlags(&a.s, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&a.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&a.join, cudaEventDisableTiming)) != cudaSuccess) return e;
  }
  out = &a;
  return cudaSuccess;
}

mc_status run_newton_schulz(Plan& P, void* ws, const mc_hparams* hp, int32_t* status,
                            cudaStream_t s, const FusedApply* fa = nullptr) {
  if (P.nsched > 0 && hp->ns_steps > 0) {
    cudaError_t e = cudaMemsetAsync(wsp(ws, P.off_sched), 0, (size_t)P.nsched * sizeof(int), s);
    if (e != cudaSuccess) return cuda_fail(e, "tile counters");
  }
  // split the shape groups into two sets of about equal Newton-Schulz work
  // (largest first onto the lighter set)
  std::vector<int> set[2];
  const int ng = (int)P.groups.size();
  if (ng >= 2 && P.xmode != kXF32) {
    std::vector<int> idx(ng);
    for (int g = 0; g < ng; ++g) idx[g] = g;
    auto work = [&](int g) {
      const double m = P.groups[g].m, n = P.groups[g].n;
      return P.groups[g].batch * (4.0 * m * m * n + 2.0 * m * m * m);
    };
    std::stable_sort(idx.begin(), idx.end(), [&](int a, int b) { return work(a) > work(b); });
    double load[2] = {0.0, 0.0};
    for (int g : idx) {
      const int k = load[1] < load[0] ? 1 : 0;
      set[k].push_back(g);
      load[k] += work(g);
    }
  } else {
    for (int g = 0; g < ng; ++g) set[0].push_back(g);
  }
  AuxStream* aux = nullptr;
  if (!set[1].empty()) {
    cudaError_t e = aux_stream(aux);
    if (e == cudaSuccess) e = cudaEventRecord(aux->fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(aux->s, aux->fork, 0);
    if (e != cudaSuccess) return cuda_fail(e, "Newton-Schulz second stream");
  }
  // the profiler times the whole Newton-Schulz section (launches overlap)
  mc_status st = MC_OK;
  {
    ProfScope ps(kGemm, 0, s);
    int launch = 0;
    for (int it = 0; it < hp->ns_steps && st == MC_OK; ++it) {
      for (Phase ph : {kGram, kPoly, kNext}) {
        if ((st = run_phase(P, ws, ph, it, hp, status, launch, set[0], s, fa)) != MC_OK) break;
        if (aux && (st = run_phase(P, ws, ph, it, hp, status, launch, set[1], aux->s, fa)) != MC_OK) break;
      }
    }
    ps.n = launch;
    // join the second stream even after a failed launch, so that no work it
    // already queued on the caller's workspace is left unordered against the
    // caller's stream (and a stream capture is not left with an open fork)
    if (aux) {
      cudaError_t e = cudaEventRecord(aux->join, aux->s);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(s, aux->join, 0);
      if (e != cudaSuccess && st == MC_OK) st = cuda_fail(e, "Newton-Schulz stream join");
    }
  }
  return st;
}

// Update factor on NewtonSchulz(M) for a [rows, cols] weight (update-RMS or
// spectral, mc_scale_mode).
float update_factor(const mc_hparams* hp, int rows, int cols) {
  return hp->scale_mode == MC_SCALE_SPECTRAL
             ? (float)std::sqrt(std::max(1.0, (double)rows / (double)cols))
             : (float)((double)hp->rms_scale * std::sqrt((double)std::max(rows, cols)));
}

// The last update can apply the step when the iterate is split, every W is
// bf16, the table holds every matrix and that update takes two or three
// products.
bool can_fuse_apply(const Plan& P, const mc_mat* W, const mc_hparams* hp) {
  if (P.xmode != kXSplit || hp->ns_steps < 1 || P.count > kMaxFusedApply) return false;
  for (int j = 0; j < P.count; ++j)
    if (W[j].dtype != MC_BF16) return false;
  for (const Group& g : P.groups)
    if (ns_terms(hp, std::min(g.m, g.n), hp->ns_steps - 1, kNext) < 2) return false;
  return true;
}

void fill_fused_apply(const Plan& P, const mc_mat* W, const mc_hparams* hp, FusedApply& fa) {
  fa.lr = hp->lr;
  fa.wd = hp->weight_decay;
  for (int j = 0; j < P.count; ++j) {
    FusedApplyJob& jb = fa.job[j];
    jb.w = W[j].ptr;
    jb.ld = W[j].ld;
    jb.transpose = P.transpose[j];
    jb.scale = update_factor(hp, (int)W[j].rows, (int)W[j].cols);
  }
}

mc_status run_apply(const Plan& P, void* ws, mc_mat* out, bool write_o, const mc_hparams* hp,
                    int32_t* status, cudaStream_t s) {
  const int fin = hp->ns_steps & 1;
  for (int j0 = 0; j0 < P.count; j0 += kMaxJobs) {
    const int nj = std::min(kMaxJobs, P.count - j0);
    ApplyParams ap;
    memset(&ap, 0, sizeof ap);
    ap.njobs = nj;
    ap.xmode = P.xmode;
    ap.write_o = write_o;
    // the split iterate is fp16 once an iteration has run (ns_fmt)
    ap.x_f16 = P.xmode == kXSplit && hp->ns_steps >= 1;
    ap.lr = hp->lr;
    ap.wd = hp->weight_decay;
    ap.status = status;
    ap.mat_scale = hp->ns_steps == 0 ? reinterpret_cast<const float*>(wsp(ws, P.off_inv)) : nullptr;
    int t = 0;
    for (int q = 0; q < nj; ++q) {
      const int j = j0 + q;
      ApplyJob& jb = ap.jobs[q];
      jb.xh = x_plane(P, ws, j, fin, 0);
      jb.xl = x_plane(P, ws, j, fin, 1);
      jb.ldx = P.groups[P.group[j]].ldn;
      jb.out = out[j].ptr;
      jb.ldo = out[j].ld;
      jb.rows = (int)out[j].rows;
      jb.cols = (int)out[j].cols;
      jb.transpose = P.transpose[j];
      jb.out_bf16 = out[j].dtype == MC_BF16;
      jb.tile_begin = t;
      jb.tiles_c = (int)cdiv(jb.cols, 64);
      jb.mat = j;
      jb.scale = update_factor(hp, jb.rows, jb.cols);
      t += (int)(cdiv(jb.rows, 64) * jb.tiles_c);
    }
    ap.total_tiles = t;
    ProfScope ps(kApply, 1, s);
    cudaError_t e = launch_apply(ap, s);
    if (e != cudaSuccess) return cuda_fail(e, "apply launch");
  }
  return MC_OK;
}

mc_status check_segments(const mc_clip_seg* segs, int nsegs, int H, const char* who) {
  if (H < 1) return fail(MC_ERR_INVALID_ARG, "%s: H must be >= 1", who);
  if (nsegs < 0 || nsegs > kMaxSegs)
    return fail(MC_ERR_INVALID_ARG, "%s: nsegs %d outside [0, %d]", who, nsegs, kMaxSegs);
  if (nsegs > 0 && !segs) return fail(MC_ERR_INVALID_ARG, "%s: null segment array", who);
  for (int i = 0; i < nsegs; ++i) {
    const mc_clip_seg& sg = segs[i];
    mc_status st = check_mat(sg.w, "segment weight", i, true, true);
    if (st != MC_OK) return st;
    if (sg.head_row_offset < 0 || sg.head_row_stride < 0 || sg.rows_per_head < 1)
      return fail(MC_ERR_INVALID_ARG, "%s: segment %d has a negative offset/stride or no rows",
                  who, i);
    const int64_t last = sg.head_row_offset + (int64_t)(H - 1) * sg.head_row_stride + sg.rows_per_head;
    if (last > sg.w.rows)
      return fail(MC_ERR_INVALID_ARG, "%s: segment %d reaches row %lld of a %lld-row weight", who,
                  i, (long long)last, (long long)sg.w.rows);
    if (!(sg.exponent >= 0.f && sg.exponent <= 4.f))
      return fail(MC_ERR_INVALID_ARG, "%s: segment %d exponent outside [0, 4]", who, i);
  }
  return MC_OK;
}

mc_status run_clip(const float* smax, int H, float tau, int mode, const mc_clip_seg* segs,
                   int nsegs, float* gamma_out, int32_t* nclipped, int32_t* status, cudaStream_t s) {
  ClipParams cp;
  memset(&cp, 0, sizeof cp);
  cp.nsegs = nsegs;
  cp.H = H;
  cp.total = mode == MC_CLIP_TOTAL;
  cp.tau = tau;
  cp.smax = smax;
  cp.gamma_out = gamma_out;
  cp.nclipped = nclipped;
  cp.status = status;
  for (int i = 0; i < nsegs; ++i) {
    ClipSegDev& d = cp.segs[i];
    d.w = segs[i].w.ptr;
    d.ld = segs[i].w.ld;
    d.row_offset = segs[i].head_row_offset;
    d.row_stride = segs[i].head_row_stride;
    d.rows = segs[i].rows_per_head;
    d.cols = (int)segs[i].w.cols;
    d.bf16 = segs[i].w.dtype == MC_BF16;
    d.exponent = segs[i].exponent;
  }
  ProfScope ps(kClip, 1, s);
  cudaError_t e = launch_clip(cp, s);
  if (e != cudaSuccess) return cuda_fail(e, "clip launch");
  return MC_OK;
}

mc_status check_ws(void* ws, size_t have, size_t need) {
  if (need == 0) return MC_OK;
  if (!ws) return fail(MC_ERR_WORKSPACE, "workspace is null (need %zu bytes)", need);
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return fail(MC_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (have < need) return fail(MC_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", have, need);
  return MC_OK;
}

// Reorder matrices so that each shape group is consecutive (the GEMM
// epilogue indexes per-matrix scales by group base + slot).
std::vector<int> group_order(const mc_mat* mats, int count) {
  std::map<std::pair<int, int>, int> first;  // shape -> first appearance
  std::vector<int> rank(count);
  for (int j = 0; j < count; ++j) {
    const int r = (int)mats[j].rows, c = (int)mats[j].cols;
    auto key = std::make_pair(std::min(r, c), std::max(r, c));
    auto it = first.find(key);
    if (it == first.end()) it = first.emplace(key, j).first;
    rank[j] = it->second;
  }
  std::vector<int> idx(count);
  for (int j = 0; j < count; ++j) idx[j] = j;
  std::stable_sort(idx.begin(), idx.end(), [&](int a, int b) { return rank[a] < rank[b]; });
  return idx;
}

template <class T>
std::vector<T> permute(const T* v, const std::vector<int>& idx) {
  std::vector<T> out(idx.size());
  for (size_t i = 0; i < idx.size(); ++i) out[i] = v[idx[i]];
  return out;
}

}  // namespace

namespace mc {
mc_status record_error(mc_status s, const char* msg) {
  g_last_error = msg;
  return s;
}
}  // namespace mc

// ==================================================================== C ABI
extern "C" {

void mc_default_hparams(mc_hparams* hp) {
  if (!hp) return;
  hp->mu = 0.95f;
  hp->lr = 2e-4f;
  hp->weight_decay = 0.1f;
  hp->rms_scale = 0.2f;
  hp->ns_steps = 5;
  hp->ns_a = 3.4445f;
  hp->ns_b = -4.7750f;
  hp->ns_c = 2.0315f;
  hp->ns_eps = 1e-7f;
  hp->tau = 100.f;
  hp->alpha = 0.5f;
  hp->ns_precision = MC_NS_AUTO;
  hp->ns_fast_steps = 3;
  hp->scale_mode = MC_SCALE_RMS;
}

const char* mc_last_error(void) { return g_last_error.c_str(); }

void mc_profiler_enable(int32_t on) { g_prof.on = on != 0; }

int32_t mc_profiler_read(mc_kernel_time* out, int32_t max, int32_t reset) {
  g_prof.drain();
  int n = 0;
  for (int c = 0; c < kNumProf && out && n < max; ++c) {
    if (g_prof.launches[c] == 0) continue;
    memset(out[n].name, 0, sizeof out[n].name);
    strncpy(out[n].name, kProfNames[c], sizeof out[n].name - 1);
    out[n].launches = (int32_t)g_prof.launches[c];
    out[n].ms = (float)g_prof.ms[c];
    ++n;
  }
  if (reset)
    for (int c = 0; c < kNumProf; ++c) { g_prof.ms[c] = 0; g_prof.launches[c] = 0; }
  return n;
}

const char* mc_version(void) { return "muonclip-gb300 0.1 (sm_103a)"; }

mc_status mc_selftest_bounded_wait(uint64_t budget_ns, uint64_t abort_after_ns, int32_t* status,
                                   uint64_t* waited_ns, mc_stream_t stream) {
  if (budget_ns < 1 || budget_ns > 1000000000ull)
    return fail(MC_ERR_INVALID_ARG, "mc_selftest_bounded_wait: budget_ns %llu outside [1, 1e9]",
                (unsigned long long)budget_ns);
  if (abort_after_ns > 1000000000ull)
    return fail(MC_ERR_INVALID_ARG, "mc_selftest_bounded_wait: abort_after_ns %llu above 1e9",
                (unsigned long long)abort_after_ns);
  if (!status) return fail(MC_ERR_INVALID_ARG, "mc_selftest_bounded_wait: null status");
  cudaError_t e = launch_wait_selftest(budget_ns, abort_after_ns, status,
                                       reinterpret_cast<unsigned long long*>(waited_ns),
                                       (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "bounded-wait self-test launch");
  return MC_OK;
}

mc_status mc_workspace_size(const mc_mat* M, int32_t count, const mc_hparams* hp, size_t* bytes) {
  if (!bytes) return fail(MC_ERR_INVALID_ARG, "bytes: null");
  if (!M || count < 1) return fail(MC_ERR_INVALID_ARG, "need count >= 1 matrices");
  mc_status st = check_hparams(hp);
  if (st != MC_OK) return st;
  bool any_f32 = false;
  for (int j = 0; j < count; ++j) {
    if (M[j].rows < 1 || M[j].cols < 1 || M[j].rows > (1 << 30) || M[j].cols > (1 << 30))
      return fail(MC_ERR_INVALID_ARG, "matrix %d: bad shape", j);
    any_f32 |= M[j].dtype == MC_F32;
  }
  (void)any_f32;
  // The precision the step will use depends on the weights; size for the
  // largest variant (fp32 planes and split planes take the same bytes).
  const int xm = hp->ns_precision == MC_NS_BF16 ? kXBf16 : kXSplit;
  *bytes = make_plan(M, count, xm).bytes;
  return ok();
}

mc_status mc_ns_products(const mc_hparams* hp, int64_t rows, int64_t cols, int32_t* products) {
  if (!products) return fail(MC_ERR_INVALID_ARG, "products: null");
  if (rows < 1 || cols < 1 || rows > (1 << 30) || cols > (1 << 30))
    return fail(MC_ERR_INVALID_ARG, "bad shape %lld x %lld", (long long)rows, (long long)cols);
  mc_status st = check_hparams(hp);
  if (st != MC_OK) return st;
  const int side = (int)std::min(rows, cols);
  for (int it = 0; it < hp->ns_steps; ++it)
    for (int ph = 1; ph <= 3; ++ph) products[3 * it + ph - 1] = ns_terms(hp, side, it, ph);
  return ok();
}

mc_status muon_momentum(mc_mat* M, const mc_mat* G, int32_t count, float mu, int32_t* status,
                        mc_stream_t stream) {
  if (!M || !G || count < 1) return fail(MC_ERR_INVALID_ARG, "need M, G and count >= 1");
  if (!std::isfinite(mu)) return fail(MC_ERR_INVALID_ARG, "mu must be finite");
  for (int j = 0; j < count; ++j) {
    mc_status st;
    if ((st = check_mat(M[j], "M", j, false, true)) != MC_OK) return st;
    if ((st = check_mat(G[j], "G", j, true, true)) != MC_OK) return st;
    if (G[j].rows != M[j].rows || G[j].cols != M[j].cols)
      return fail(MC_ERR_INVALID_ARG, "G[%d] shape differs from M[%d]", j, j);
  }
  Plan P = make_plan(M, count, kXF32);
  mc_status st = run_prep(P, nullptr, M, G, true, false, mu, status, (cudaStream_t)stream);
  return st == MC_OK ? ok() : st;
}

mc_status muon_newton_schulz(const mc_mat* M, mc_mat* O, int32_t count, const mc_hparams* hp,
                             void* workspace, size_t workspace_bytes, int32_t* status,
                             mc_stream_t stream) {
  if (!M || !O || count < 1) return fail(MC_ERR_INVALID_ARG, "need M, O and count >= 1");
  mc_status st = check_hparams(hp);
  if (st != MC_OK) return st;
  bool any_f32 = false;
  for (int j = 0; j < count; ++j) {
    if ((st = check_mat(M[j], "M", j, false, true)) != MC_OK) return st;
    if ((st = check_mat(O[j], "O", j, true, true)) != MC_OK) return st;
    if (O[j].rows != M[j].rows || O[j].cols != M[j].cols)
      return fail(MC_ERR_INVALID_ARG, "O[%d] shape differs from M[%d]", j, j);
    any_f32 |= O[j].dtype == MC_F32;
  }
  const std::vector<int> ord = group_order(M, count);
  std::vector<mc_mat> Mo = permute(M, ord), Oo = permute(O, ord);
  Plan P = make_plan(Mo.data(), count, resolve_xmode(hp->ns_precision, any_f32));
  if ((st = check_ws(workspace, workspace_bytes, P.bytes)) != MC_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  if ((st = run_prep(P, workspace, Mo.data(), nullptr, false, true, 0.f, status, s)) != MC_OK) return st;
  if ((st = run_norms(P, workspace, hp->ns_eps, s)) != MC_OK) return st;
  if ((st = run_newton_schulz(P, workspace, hp, status, s)) != MC_OK) return st;
  if ((st = run_apply(P, workspace, Oo.data(), true, hp, status, s)) != MC_OK) return st;
  return ok();
}

mc_status qk_max_logit(const mc_attn_desc* a, float* smax, int64_t* argmax, int32_t accumulate,
                       int32_t* status, mc_stream_t stream) {
  if (!a || !smax) return fail(MC_ERR_INVALID_ARG, "need attn descriptor and smax");
  if (a->B < 1 || a->S < 1 || a->H < 1 || a->d_head < 1 || a->d_shared < 0)
    return fail(MC_ERR_INVALID_ARG, "attn: B, S, H, d_head must be >= 1 and d_shared >= 0");
  if (a->dtype != MC_F32 && a->dtype != MC_BF16)
    return fail(MC_ERR_INVALID_ARG, "attn: unknown dtype %d", a->dtype);
  if (!a->q || !a->k || (a->d_shared > 0 && !a->k_shared))
    return fail(MC_ERR_INVALID_ARG, "attn: null feature pointer");
  if (!(a->scale > 0.f) || !std::isfinite(a->scale))
    return fail(MC_ERR_INVALID_ARG, "attn: scale must be finite and > 0");
  if (a->d_head + a->d_shared > 256)
    return fail(MC_ERR_UNSUPPORTED, "attn: q.k length %d > 256", a->d_head + a->d_shared);
  for (int i = 0; i < 3; ++i)
    if (a->q_strides[i] < 0 || a->k_strides[i] < 0)
      return fail(MC_ERR_INVALID_ARG, "attn: negative stride");
  if (argmax) {
    if (accumulate) return fail(MC_ERR_INVALID_ARG, "attn: argmax requires accumulate = 0");
    if ((double)a->B * a->S * a->S >= 4294967295.0)
      return fail(MC_ERR_UNSUPPORTED, "attn: argmax needs B*S*S < 2^32");
    if ((reinterpret_cast<uintptr_t>(argmax) & 7u) != 0)
      return fail(MC_ERR_INVALID_ARG, "attn: argmax must be 8-byte aligned");
  }
  if ((reinterpret_cast<uintptr_t>(smax) & 3u) != 0)
    return fail(MC_ERR_INVALID_ARG, "smax must be 4-byte aligned");
  MaxLogitParams p;
  memset(&p, 0, sizeof p);
  p.B = a->B; p.S = a->S; p.H = a->H; p.d_head = a->d_head; p.d_shared = a->d_shared;
  p.dtype = a->dtype; p.causal = a->causal != 0; p.scale = a->scale;
  p.q = a->q; p.k = a->k; p.ks = a->k_shared;
  for (int i = 0; i < 3; ++i) { p.qs[i] = a->q_strides[i]; p.kst[i] = a->k_strides[i]; }
  for (int i = 0; i < 2; ++i) p.kss[i] = a->ks_strides[i];
  p.smax = smax;
  p.argmax = reinterpret_cast<long long*>(argmax);
  p.accumulate = accumulate != 0;
  p.status = status;
  char err[256] = {0};
  cudaError_t e;
  {
    ProfScope ps(kMaxLogit, 3, (cudaStream_t)stream);
    e = launch_max_logit(p, (cudaStream_t)stream, err, sizeof err);
  }
  if (e != cudaSuccess) {
    if (err[0]) return fail(MC_ERR_CUDA, "max logit: %s", err);
    return cuda_fail(e, "max logit launch");
  }
  return ok();
}

mc_status qk_attention_forward(const mc_attn_desc* a, const mc_attn_out* out, float* smax,
                               int32_t accumulate, int32_t* status, mc_stream_t stream) {
  if (!a || !out || !smax) return fail(MC_ERR_INVALID_ARG, "need attn, out and smax");
  if (a->B < 1 || a->S < 1 || a->H < 1 || a->d_head < 1 || a->d_shared < 0)
    return fail(MC_ERR_INVALID_ARG, "attn: B, S, H, d_head must be >= 1 and d_shared >= 0");
  if (a->dtype != MC_F32 && a->dtype != MC_BF16)
    return fail(MC_ERR_INVALID_ARG, "attn: unknown dtype %d", a->dtype);
  if (a->dtype != MC_BF16) return fail(MC_ERR_UNSUPPORTED, "attention forward: bf16 only");
  if (!a->q || !a->k || (a->d_shared > 0 && !a->k_shared) || !out->v || !out->o)
    return fail(MC_ERR_INVALID_ARG, "attention forward: null pointer");
  if (!(a->scale > 0.f) || !std::isfinite(a->scale))
    return fail(MC_ERR_INVALID_ARG, "attn: scale must be finite and > 0");
  for (int i = 0; i < 3; ++i)
    if (a->q_strides[i] < 0 || a->k_strides[i] < 0 || out->v_strides[i] < 0 || out->o_strides[i] < 0)
      return fail(MC_ERR_INVALID_ARG, "attention forward: negative stride");
  if ((reinterpret_cast<uintptr_t>(smax) & 3u) != 0 ||
      (out->lse && (reinterpret_cast<uintptr_t>(out->lse) & 3u) != 0))
    return fail(MC_ERR_INVALID_ARG, "smax and lse must be 4-byte aligned");
  AttnFwdParams p;
  memset(&p, 0, sizeof p);
  p.B = a->B; p.S = a->S; p.H = a->H; p.d_head = a->d_head; p.d_shared = a->d_shared;
  p.d_v = out->d_v;
  p.causal = a->causal != 0; p.scale = a->scale;
  p.q = a->q; p.k = a->k; p.ks = a->k_shared; p.v = out->v; p.o = out->o;
  for (int i = 0; i < 3; ++i) {
    p.qs[i] = a->q_strides[i]; p.kst[i] = a->k_strides[i];
    p.vs[i] = out->v_strides[i]; p.os[i] = out->o_strides[i];
  }
  for (int i = 0; i < 2; ++i) p.kss[i] = a->ks_strides[i];
  p.lse = out->lse;
  p.smax = smax;
  p.accumulate = accumulate != 0;
  p.status = status;
  char err[256] = {0};
  if (!attn_fwd_supported(p, err, sizeof err)) return fail(MC_ERR_UNSUPPORTED, "attention forward: %s", err);
  cudaError_t e;
  {
    ProfScope ps(kAttnFwd, 3, (cudaStream_t)stream);
    e = launch_attn_fwd(p, (cudaStream_t)stream, err, sizeof err);
  }
  if (e != cudaSuccess) {
    if (err[0]) return fail(MC_ERR_CUDA, "attention forward: %s", err);
    return cuda_fail(e, "attention forward launch");
  }
  return ok();
}

mc_status qk_clip_apply(const float* smax, int32_t H, float tau, int32_t mode,
                        const mc_clip_seg* segs, int32_t nsegs, float* gamma_out,
                        int32_t* nclipped, int32_t* status, mc_stream_t stream) {
  if (!smax) return fail(MC_ERR_INVALID_ARG, "smax: null");
  if (!(tau > 0.f) || !std::isfinite(tau)) return fail(MC_ERR_INVALID_ARG, "tau must be finite and > 0");
  if (mode != MC_CLIP_PER_HEAD && mode != MC_CLIP_TOTAL)
    return fail(MC_ERR_INVALID_ARG, "qk_clip_apply: unknown mode %d", mode);
  mc_status st = check_segments(segs, nsegs, H, "qk_clip_apply");
  if (st != MC_OK) return st;
  st = run_clip(smax, H, tau, mode, segs, nsegs, gamma_out, nclipped, status, (cudaStream_t)stream);
  return st == MC_OK ? ok() : st;
}

mc_status muonclip_step(mc_mat* W, const mc_mat* G, mc_mat* M, int32_t count,
                        const mc_hparams* hp, const mc_clip_layer* layers, int32_t nlayers,
                        void* workspace, size_t workspace_bytes, int32_t* status,
                        mc_stream_t stream) {
  if (!W || !G || !M || count < 1) return fail(MC_ERR_INVALID_ARG, "need W, G, M and count >= 1");
  mc_status st = check_hparams(hp);
  if (st != MC_OK) return st;
  if (nlayers < 0 || (nlayers > 0 && !layers)) return fail(MC_ERR_INVALID_ARG, "bad layers");
  bool any_f32 = false;
  for (int j = 0; j < count; ++j) {
    if ((st = check_mat(W[j], "W", j, true, true)) != MC_OK) return st;
    if ((st = check_mat(G[j], "G", j, true, true)) != MC_OK) return st;
    if ((st = check_mat(M[j], "M", j, false, true)) != MC_OK) return st;
    if (G[j].rows != W[j].rows || G[j].cols != W[j].cols || M[j].rows != W[j].rows ||
        M[j].cols != W[j].cols)
      return fail(MC_ERR_INVALID_ARG, "matrix %d: W, G, M shapes differ", j);
    any_f32 |= W[j].dtype == MC_F32;
  }
  for (int l = 0; l < nlayers; ++l) {
    if (!layers[l].smax) return fail(MC_ERR_INVALID_ARG, "layer %d: smax null", l);
    if (layers[l].mode != MC_CLIP_PER_HEAD && layers[l].mode != MC_CLIP_TOTAL)
      return fail(MC_ERR_INVALID_ARG, "layer %d: unknown clip mode %d", l, layers[l].mode);
    if ((st = check_segments(layers[l].segs, layers[l].nsegs, layers[l].H, "muonclip_step")) != MC_OK)
      return st;
  }
  const std::vector<int> ord = group_order(W, count);
  std::vector<mc_mat> Wo = permute(W, ord), Go = permute(G, ord), Mo = permute(M, ord);
  Plan P = make_plan(Wo.data(), count, resolve_xmode(hp->ns_precision, any_f32));
  if ((st = check_ws(workspace, workspace_bytes, P.bytes)) != MC_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  // Algorithm 1, part 1: Muon on every matrix.  With bf16 weights on the split
  // path the last Newton-Schulz update applies the step in its epilogue (no
  // separate pass over the iterate); otherwise apply_kernel does.
  std::unique_ptr<FusedApply> fa;
  if (can_fuse_apply(P, Wo.data(), hp)) {
    fa.reset(new FusedApply());
    fill_fused_apply(P, Wo.data(), hp, *fa);
  }
  if ((st = run_prep(P, workspace, Mo.data(), Go.data(), true, true, hp->mu, status, s)) != MC_OK) return st;
  if ((st = run_norms(P, workspace, hp->ns_eps, s)) != MC_OK) return st;
  if ((st = run_newton_schulz(P, workspace, hp, status, s, fa.get())) != MC_OK) return st;
  if (!fa && (st = run_apply(P, workspace, Wo.data(), false, hp, status, s)) != MC_OK) return st;
  // Algorithm 1, part 2: per-head QK-Clip on the updated weights
  for (int l = 0; l < nlayers; ++l) {
    const mc_clip_layer& L = layers[l];
    if ((st = run_clip(L.smax, L.H, hp->tau, L.mode, L.segs, L.nsegs, L.gamma_out, L.nclipped, status, s)) != MC_OK)
      return st;
  }
  return ok();
}

}  // extern "C"
