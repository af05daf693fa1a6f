// Internal launcher interface between the host API (api.cpp) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/muonclip.h"

namespace mc {

inline constexpr int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline constexpr int64_t round_up(int64_t a, int64_t b) { return cdiv(a, b) * b; }

// 16-bit formats of a tensor-core Newton-Schulz launch: operands (A, B, C)
// and stored output D.
enum GemmFmt : int {
  kFmtBf16 = 0,       // bf16 in, bf16 out
  kFmtBf16ToF16 = 1,  // bf16 in, fp16 out
  kFmtF16 = 2         // fp16 in, fp16 out
};

// Storage of a Newton-Schulz iterate (and of its Gram / polynomial matrices).
enum XMode : int {
  kXSplit = 0,  // two bf16 planes, value = hi + lo
  kXBf16 = 1,   // one bf16 plane
  kXF32 = 2     // one fp32 plane (hi pointer is float*)
};

constexpr int kMaxJobs = 96;     // matrices per streaming-kernel launch
constexpr int kMaxGroups = 6;    // shape groups per tensor-core GEMM launch

// ---------------------------------------------------------------- streaming
// One matrix for the momentum / Newton-Schulz preparation kernel.  The
// iterate is written in the orientation with rows <= cols (transposed when
// rows > cols).
struct PrepJob {
  float* M;            // f32 momentum, updated in place when do_momentum
  const void* G;       // f32 or bf16 gradient (unused without do_momentum)
  void* xh;            // oriented iterate planes (see XMode)
  void* xl;
  long long ldM, ldG, ldx;
  int rows, cols;      // original shape
  int g_bf16;
  int transpose;
  int tile_begin;      // first 64x64 tile of this matrix in the launch
  int tiles_c;         // tiles along cols of the original
};

struct PrepParams {
  PrepJob jobs[kMaxJobs];
  int njobs;
  int total_tiles;
  int do_momentum;
  int write_x;         // 0: momentum only (public muon_momentum)
  int xmode;
  float mu;
  double* partials;    // [total_tiles] sum of squares per tile, or null
  int32_t* status;
};

// One matrix for the update / output kernel.
struct ApplyJob {
  const void* xh;      // final oriented iterate planes
  const void* xl;
  long long ldx;
  void* out;           // W (update in place) or O (write)
  long long ldo;
  int rows, cols;
  int transpose;
  int out_bf16;
  int tile_begin;
  int tiles_c;
  int mat;             // index into mat_scale
  float scale;         // rms_scale * sqrt(max(rows, cols))
};

struct ApplyParams {
  ApplyJob jobs[kMaxJobs];
  int njobs;
  int total_tiles;
  int xmode;
  int write_o;         // 1: out = scale * X; 0: W -= lr (scale X + wd W)
  int x_f16;           // split iterate planes hold fp16 (else bf16)
  float lr, wd;
  const float* mat_scale;  // per-matrix extra factor on X, or null
  int32_t* status;
};

cudaError_t launch_prep(const PrepParams& p, cudaStream_t s);
cudaError_t launch_apply(const ApplyParams& p, cudaStream_t s);
// inv_norm[j] = 1 / (sqrt(sum of partials of matrix j) + eps), inv_norm_sq = square.
// tile_begin / tile_count are HOST arrays (passed to the kernel as parameters).
constexpr int kMaxNormMats = 1024;
struct NormParams {
  int begin[kMaxNormMats];
  int count[kMaxNormMats];
  int nmat, mat0;
  float eps;
  const double* partials;
  float* inv_norm;
  float* inv_norm_sq;
};
cudaError_t launch_norms(const double* partials, const int* tile_begin, const int* tile_count,
                         int nmat, float eps, float* inv_norm, float* inv_norm_sq,
                         cudaStream_t s);

// ---------------------------------------------------------------- NS GEMMs
// One batch of same-shape matrices for a Newton-Schulz phase:
//   D[b] = s_b * (alpha * P[b] + beta * C[b] + diag * I),  P = A-operand x B-operand
// with P an M x N product over K (diag is nonzero only for square outputs).
struct GemmGroup {
  int M, N, K, batch;
  int tiles_m, tiles_n;
  int tile_begin;
  int mat_base;           // index of batch item 0 into the s_b array
  int b_mn_major;         // B operand stored [K, N] (N contiguous)
  int symmetric;          // D is symmetric (M == N): compute only tiles that touch
                          // the upper triangle and write each element's mirror
  int tiles_per_item;     // output tiles per batch item
  // plain pointers (SIMT path reads operands through these; the tensor-core
  // path reads operands through tensor maps and uses these for C and D)
  const void* a_hi; const void* a_lo; long long lda, a_bstride;
  const void* b_hi; const void* b_lo; long long ldb, b_bstride;
  const void* c_hi; const void* c_lo; long long ldc, c_bstride;
  void* d_hi; void* d_lo; long long ldd, d_bstride;
};

struct GemmTmaps {
  CUtensorMap a_hi[kMaxGroups], a_lo[kMaxGroups], b_hi[kMaxGroups], b_lo[kMaxGroups];
  CUtensorMap d_hi[kMaxGroups], d_lo[kMaxGroups];     // D chunks (16 columns x 32 rows)
  CUtensorMap dm_hi[kMaxGroups], dm_lo[kMaxGroups];   // mirrored D chunks (32 columns x 16 rows)
  CUtensorMap c_hi[kMaxGroups], c_lo[kMaxGroups];     // C of non-symmetric outputs (16 x 32 boxes)
};

struct GemmParams {
  GemmGroup g[kMaxGroups];
  int ngroups;
  int total_tiles;
  int xmode;
  int terms;              // tensor-core products per k-step: 1 (hi*hi), 2 (hi*hi + hi*lo_B)
                          // or 3 (hi*hi + hi*lo + lo*hi)
  int fmt;                // tensor-core planes: kFmtBf16, kFmtBf16ToF16 or kFmtF16
  int d_hi_only;          // split planes: store only D's hi plane (no consumer reads lo)
  float alpha, beta;
  float diag;             // added on the diagonal of each output item
  const float* s;         // per-matrix scale, or null
  int32_t* status;
  int* sched;             // zeroed tile counter of this launch (tensor-core path)
};

// The last Newton-Schulz update can apply the step itself: instead of storing
// the final iterate it writes W <- W - lr (scale_j D + wd W) for each matrix j
// (bf16 W in the caller's layout; the matrix is the transpose of its oriented
// iterate when rows > cols).  Indexed by the matrix order of the plan.
constexpr int kMaxFusedApply = 192;
struct FusedApplyJob {
  void* w;             // bf16 W [rows, cols], updated in place
  long long ld;        // row pitch in elements (16-byte multiple)
  int transpose;       // W = X^T (rows > cols)
  float scale;         // factor on the Newton-Schulz output (update-RMS or spectral)
};
struct FusedApply {
  static constexpr bool kOn = true;
  FusedApplyJob job[kMaxFusedApply];
  float lr, wd;
};

// Tensor-core path (split bf16 or bf16).  Encodes its own tensor maps.  With
// `fa` (the last update of a step whose W the launch updates) the epilogue
// applies the step instead of storing D.
cudaError_t launch_ns_gemm_tc(const GemmParams& p, const FusedApply* fa, cudaStream_t s, char* err,
                              size_t errlen);
// Output tiles of the tensor-core GEMM: 256 x 256 per CTA pair.
constexpr int kTcTileM = 256, kTcTileN = 256;
// CUDA-core fp32 path.
cudaError_t launch_ns_gemm_f32(const GemmParams& p, cudaStream_t s);

// ---------------------------------------------------------------- QK-Clip
struct ClipSegDev {
  void* w;
  long long ld;
  long long row_offset, row_stride, rows;
  int cols;
  int bf16;
  float exponent;
};
constexpr int kMaxSegs = 16;
struct ClipParams {
  ClipSegDev segs[kMaxSegs];
  int nsegs;
  int H;
  int total;               // 1: one gamma from max_h smax for every head
  float tau;
  const float* smax;
  float* gamma_out;
  int32_t* nclipped;
  int32_t* status;
};
cudaError_t launch_clip(const ClipParams& p, cudaStream_t s);

// ---------------------------------------------------------------- max logit
struct MaxLogitParams {
  int B, S, H, d_head, d_shared;
  int dtype;       // 0 f32, 1 bf16
  int causal;
  float scale;
  const void* q; const void* k; const void* ks;
  long long qs[3], kst[3], kss[2];
  float* smax;             // [H] float maxima (with argmax: written at the end)
  long long* argmax;       // packed (ordered value << 32 | ~index) scratch view
  int accumulate;
  int32_t* status;
};
cudaError_t launch_max_logit(const MaxLogitParams& p, cudaStream_t s, char* err, size_t errlen);

// Attention forward (bf16, tensor cores) with the per-head max logit.
struct AttnFwdParams {
  int B, S, H, d_head, d_shared, d_v;
  int causal;
  float scale;
  const void* q; const void* k; const void* ks; const void* v; void* o;
  long long qs[3], kst[3], kss[2], vs[3], os[3];   // element strides (batch, seq, head)
  float* lse;              // [B, H, S] or null
  float* smax;             // [H] float maxima, max-combined in place
  int accumulate;
  int32_t* status;
};
// Returns cudaErrorInvalidValue with a message in err for shapes outside the
// kernel's tiles (checked by the caller first).
cudaError_t launch_attn_fwd(const AttnFwdParams& p, cudaStream_t s, char* err, size_t errlen);
bool attn_fwd_supported(const AttnFwdParams& p, char* err, size_t errlen);

// Bounded-wait self-check (one CTA waits on a phase nothing completes).
cudaError_t launch_wait_selftest(unsigned long long budget_ns, unsigned long long abort_after_ns,
                                 int32_t* status, unsigned long long* waited_ns, cudaStream_t s);

// Device/properties helpers.
int sm_count();

// Record `msg` as the thread's last error (mc_last_error) and return `s`.
mc_status record_error(mc_status s, const char* msg);

}  // namespace mc
