/*
 * muonclip.h - C ABI of the GB300 (sm_103a) MuonClip optimizer step.
 *
 * MuonClip = the Muon update followed by per-head QK-Clip.  Sources, cited by
 * page title and section:
 *   [K2-internals] "Kimi K2 内部机制" (LLM-101-CN): "Algorithm 1 MuonClip
 *                  Optimizer", "核心数学" (S_max, gamma), "MLA 的特殊处理".
 *   [K2-notes]     "Kimi K2: Open Agentic Intelligence" notes, section 3.2
 *                  MuonClip (pseudocode muonclip_step).
 *   [K2-explained] "Kimi K2, explained": "Pretraining with MuonClip".
 *   [K2-zhihu]     zhihu Q&A on K2: MuonClip formula written with msign.
 *
 * Conventions for every call:
 *   - All pointers inside mc_mat / mc_attn_desc / mc_clip_seg are DEVICE
 *     pointers owned by the caller.  Descriptor arrays themselves (mc_mat*,
 *     mc_clip_seg*, mc_clip_layer*) are HOST memory, read only during the call.
 *   - Matrices are row-major: element (r, c) lives at ptr[r * ld + c], with
 *     ld >= cols, ld in elements.  Weights are stored [out, in].
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  The library allocates no device memory: scratch comes
 *     from the caller's `workspace` (size from the matching *_workspace_size).
 *   - Argument, shape, dtype and alignment errors are detected on the host
 *     before any launch; the call then returns MC_ERR_INVALID_ARG or
 *     MC_ERR_UNSUPPORTED and launches nothing.  A failed launch returns
 *     MC_ERR_CUDA.  mc_last_error() returns a thread-local message for the last
 *     non-OK return.
 *   - Data-dependent conditions (non-finite values, a device wait that ran
 *     out of time) are reported through the optional device word `status`:
 *     the kernels OR MC_STATUS_* bits into it; the caller reads it after
 *     synchronising the stream.  The library never traps or asserts on device.
 */
#ifndef MUONCLIP_H
#define MUONCLIP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* mc_stream_t; /* same object as cudaStream_t */

typedef enum {
  MC_OK = 0,
  MC_ERR_INVALID_ARG = 1,  /* bad pointer, shape, dtype, stride or value   */
  MC_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement  */
  MC_ERR_WORKSPACE = 3,    /* workspace missing, misaligned or too small   */
  MC_ERR_CUDA = 4,         /* a CUDA runtime/driver call or launch failed  */
  MC_ERR_NONFINITE = 5,    /* reserved for host-side reporting of status   */
  MC_ERR_TIMEOUT = 6       /* reserved for host-side reporting of status   */
} mc_status;

/* Bits OR-ed into the optional device status word. */
#define MC_STATUS_NONFINITE_UPDATE 1  /* NaN/Inf in M, G or the NS result  */
#define MC_STATUS_NONFINITE_LOGIT  2  /* NaN/Inf among the attention logits */
#define MC_STATUS_NONFINITE_SMAX   4  /* NaN/Inf S_max given to the clip     */
#define MC_STATUS_TIMEOUT          8  /* a bounded device wait gave up       */

typedef enum { MC_F32 = 0, MC_BF16 = 1 } mc_dtype;

/* Arithmetic of the Newton-Schulz products.
 *   MC_NS_SPLIT_BF16: tcgen05 tensor cores on 16-bit (hi, lo) planes, fp32
 *     accumulation.  The first iteration reads the momentum's bf16 (hi, lo)
 *     copy (bf16 keeps fp32's exponent range, whatever the scale of M); its
 *     update normalises by 1/||M|| and every later iterate, Gram and
 *     polynomial matrix is stored as an fp16 (hi, lo) pair (~22 significand
 *     bits; entries stay bounded after the normalisation).  A product takes
 *     one term (hi*hi), two (hi*hi + hi*lo of X: the trailing updates) or
 *     three (hi*hi + hi*lo + lo*hi) per k-step, as ns_fast_steps below says.
 *     Default for bf16 weights.
 *   MC_NS_BF16: tcgen05, one bf16 product, bf16 iterates (fastest, ~1e-1
 *     max-abs / 1e-2 RMS deviation from exact arithmetic).
 *   MC_NS_FP32: CUDA-core fp32 products and fp32 iterates.  Default for fp32
 *     weights.
 *   MC_NS_AUTO: SPLIT_BF16 when every weight is bf16, else FP32. */
typedef enum { MC_NS_AUTO = 0, MC_NS_SPLIT_BF16 = 1, MC_NS_BF16 = 2, MC_NS_FP32 = 3 } mc_ns_precision;

/* Factor applied to NewtonSchulz(M) for a weight stored [rows=out, cols=in].
 *   MC_SCALE_RMS: rms_scale * sqrt(max(rows, cols)) (AdamW-matched update RMS,
 *     [K2-internals] Algorithm 1; the default).
 *   MC_SCALE_SPECTRAL: sqrt(max(1, rows / cols)) (the MuP-style scale of the
 *     zhihu answer's section 3.2); rms_scale is ignored. */
typedef enum { MC_SCALE_RMS = 0, MC_SCALE_SPECTRAL = 1 } mc_scale_mode;

/* QK-Clip granularity.
 *   MC_CLIP_PER_HEAD: gamma_h = tau / S_max^h for each head over tau (K2).
 *   MC_CLIP_TOTAL: one gamma = tau / max_h S_max^h for every head when that
 *     max exceeds tau (the naive form of [K2-internals] "核心数学"). */
typedef enum { MC_CLIP_PER_HEAD = 0, MC_CLIP_TOTAL = 1 } mc_clip_mode;

typedef struct {
  void* ptr;      /* device pointer, 16-byte aligned                    */
  int32_t dtype;  /* mc_dtype                                           */
  int32_t _pad;
  int64_t rows;   /* >= 1                                               */
  int64_t cols;   /* >= 1                                               */
  int64_t ld;     /* leading dimension in elements, >= cols, ld*size%16==0 */
} mc_mat;

/* Hyper-parameters of one MuonClip step ([K2-internals] Algorithm 1;
 * [K2-notes] 3.2 pseudocode defaults: mu 0.95, weight_decay 0.1, tau 100). */
typedef struct {
  float mu;            /* momentum coefficient                               */
  float lr;            /* learning rate eta_t                                */
  float weight_decay;  /* decoupled weight decay lambda                      */
  float rms_scale;     /* 0.2: O_t = NS(M_t) * sqrt(max(n,m)) * rms_scale    */
  int32_t ns_steps;    /* Newton-Schulz iterations (5), 0..32                */
  float ns_a, ns_b, ns_c; /* X <- a X + (b A + c A^2) X, A = X X^T          */
  float ns_eps;        /* X0 = M / (||M||_F + ns_eps)                        */
  float tau;           /* QK-Clip threshold (> 0)                            */
  float alpha;         /* MHA split: W_q by gamma^alpha, W_k by gamma^(1-alpha) */
  int32_t ns_precision;/* mc_ns_precision                                    */
  int32_t ns_fast_steps;/* MC_NS_SPLIT_BF16 only: this many leading iterations
                          take one product (hi*hi) per k-step, for matrices
                          whose smaller side is at least 256: up to three
                          (larger values act as three), each run keeping at
                          least two iterations after it, whose Gram products
                          take one product and whose polynomial takes three
                          and whose update two (hi*hi + hi*lo of X; three
                          when the smaller side is under 512).  Float64
                          emulation of this arithmetic gives at most 1.4e-2
                          of RMS (2048 x 16384 adversarial spectrum, 64
                          dominant directions over a 1e-3 rest; 2048 x 7168
                          Gaussian: 3-5e-3; 512 x 16384 Gaussian: 9.3e-3).
                          Matrices whose smaller side is under 256 take three
                          products everywhere (1.4e-2 at 64 otherwise).
                          Default 3. */
  int32_t scale_mode;  /* mc_scale_mode: factor on NewtonSchulz(M)            */
} mc_hparams;

/* One head-blocked row segment of a weight that QK-Clip rescales.  Head h
 * owns rows [head_row_offset + h*head_row_stride, ... + rows_per_head) of w;
 * when S_max^h > tau those rows are multiplied by gamma_h^exponent, where
 * gamma_h = tau / S_max^h ([K2-internals] "核心数学", "MLA 的特殊处理";
 * Algorithm 1 QK-Clip branch).  MHA: W_q exponent alpha, W_k 1 - alpha.
 * MLA: q^C rows 0.5, k^C rows 0.5, q^R rows 1.0; the shared rotary key k^R
 * gets no segment, so it is never touched. */
typedef struct {
  mc_mat w;                /* bf16 or f32 weight, updated in place */
  int64_t head_row_offset;
  int64_t head_row_stride;
  int64_t rows_per_head;
  float exponent;          /* in [0, 4] */
  int32_t _pad;
} mc_clip_seg;

/* One attention layer's clip: S_max per head (device, [H]) and its segments. */
typedef struct {
  const float* smax;       /* device [H], S_max^h from this step's forward  */
  int32_t H;
  int32_t nsegs;
  const mc_clip_seg* segs; /* host array of nsegs                           */
  float* gamma_out;        /* device [H] or NULL: gamma_h (1 when no clip)  */
  int32_t* nclipped;       /* device int or NULL: heads clipped in layer    */
  int32_t mode;            /* mc_clip_mode                                  */
  int32_t _pad;
} mc_clip_layer;

/* Query/key features of one attention layer, for the per-head max logit.
 * Logit(b, h, i, j) = q_{b,i,h} . k_{b,j,h} with
 *   q_{b,i,h} = q[b*q_strides[0] + i*q_strides[1] + h*q_strides[2] + t],
 *               t in [0, d_head + d_shared)
 *   k_{b,j,h} = [ k[b*k_strides[0] + j*k_strides[1] + h*k_strides[2] + t],
 *                   t in [0, d_head)  ||
 *                 k_shared[b*ks_strides[0] + j*ks_strides[1] + t],
 *                   t in [0, d_shared) ]
 * MHA: d_shared = 0, k_shared = NULL.  MLA: q = [q^C || q^R] per head,
 * k = k^C (head-specific), k_shared = k^R (one rotary key for all heads).
 * Strides are in elements; the feature index is contiguous. */
typedef struct {
  int32_t B, S, H;
  int32_t d_head;          /* head-specific q.k length (MLA: d_nope)        */
  int32_t d_shared;        /* shared rotary length (MLA: d_rope), or 0      */
  int32_t dtype;           /* mc_dtype of q, k, k_shared                    */
  int32_t causal;          /* 1: max over j <= i only                       */
  float scale;             /* logit scale, 1/sqrt(d_head + d_shared)        */
  const void* q;
  const void* k;
  const void* k_shared;
  int64_t q_strides[3];    /* batch, sequence, head                         */
  int64_t k_strides[3];    /* batch, sequence, head                         */
  int64_t ks_strides[2];   /* batch, sequence                               */
} mc_attn_desc;

/* Fill *hp with the defaults named above (mu 0.95, lr 2e-4, weight_decay 0.1,
 * rms_scale 0.2, 5 steps of the quintic (3.4445, -4.7750, 2.0315),
 * ns_eps 1e-7, tau 100, alpha 0.5, MC_NS_AUTO, ns_fast_steps 3, MC_SCALE_RMS). */
void mc_default_hparams(mc_hparams* hp);

/* Bytes of workspace that muon_newton_schulz / muonclip_step need for these
 * `count` matrices (shapes and dtypes of M, or of W for muonclip_step). */
mc_status mc_workspace_size(const mc_mat* M, int32_t count, const mc_hparams* hp, size_t* bytes);

/* Products per k-step that the split tensor-core Newton-Schulz takes for
 * a rows x cols matrix under *hp ([K2-internals] Algorithm 1, orthogonalisation
 * step; the arithmetic of the split iterate is this library's): for iteration
 * i (0 .. ns_steps - 1), products[3 i + 0], [3 i + 1] and [3 i + 2] are those
 * of the Gram product A = X X^T, the polynomial B = b A + c A^2 and the update,
 * each 1 (hi*hi), 2 (hi*hi + hi*lo of X) or 3 (hi*hi + hi*lo + lo*hi).  products: host int32 array of
 * 3 * ns_steps entries, owned by the caller.  Host-only; no GPU work.
 * MC_ERR_INVALID_ARG for a null array, a shape outside 1 .. 2^30 or invalid
 * hyper-parameters. */
mc_status mc_ns_products(const mc_hparams* hp, int64_t rows, int64_t cols, int32_t* products);

/* M_t = mu * M_{t-1} + G_t for each of `count` matrices, in place.
 * [K2-internals] Algorithm 1, momentum step (M_0 = 0: pass a zeroed M).
 * M: f32; G: f32 or bf16, same rows/cols as M.  A NaN/Inf in M_t sets
 * MC_STATUS_NONFINITE_UPDATE. */
mc_status muon_momentum(mc_mat* M, const mc_mat* G, int32_t count, float mu, int32_t* status,
                        mc_stream_t stream);

/* O_t = NewtonSchulz(M_t) * sqrt(max(rows, cols)) * rms_scale for each matrix.
 * [K2-internals] Algorithm 1, orthogonalisation step; [K2-explained] symbol
 * list (odd matrix polynomial pushing singular values toward 1).  M: f32;
 * O: f32 or bf16, same shape as M (not in place).  The iteration runs on the
 * orientation with rows <= cols (transposed internally when rows > cols). */
mc_status muon_newton_schulz(const mc_mat* M, mc_mat* O, int32_t count, const mc_hparams* hp,
                             void* workspace, size_t workspace_bytes, int32_t* status,
                             mc_stream_t stream);

/* muon_newton_schulz without a workspace argument, for callers that cannot
 * give this library device memory: a framework whose caching allocator owns
 * the GPU's memory and must not see foreign cudaMalloc calls, a training loop
 * that cannot afford the device-wide synchronisation of cudaFree, or a plugin
 * whose host application provides no allocator.  The pages have no
 * counterpart to this call; it exists for those callers only.
 *   - Scratch comes from one fixed device array inside the library,
 *     MC_NOALLOC_SCRATCH_BYTES long, held on every GPU that loads the library
 *     until the process exits.  The call allocates nothing.
 *   - Requests whose workspace (mc_workspace_size) exceeds that size return
 *     MC_ERR_WORKSPACE with a message; use muon_newton_schulz for them.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and keeps it; make
 *     that first call before any stream capture.  The kept address is not
 *     looked up again: after cudaDeviceReset in this process the array may
 *     live elsewhere, so do not use this entry point after a device reset.
 *   - Every call shares the one array.  Nothing in it needs to start at zero
 *     (each value a kernel reads was written earlier in the same call), but
 *     calls that overlap on the GPU (different streams, or several host
 *     threads) race on it: serialise them.
 * Arguments, results and errors are otherwise those of muon_newton_schulz. */
#define MC_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
mc_status muon_newton_schulz_noalloc(const mc_mat* M, mc_mat* O, int32_t count,
                                     const mc_hparams* hp, int32_t* status, mc_stream_t stream);

/* Per-head max logit S_max^h = scale * max_{b} max_{i, j(<=i)} q.k.
 * [K2-internals] "核心数学" (S_max^h over the batch); Algorithm 1 takes it
 * from the forward pass.  smax: device float[H], written (accumulate = 0) or
 * max-combined with its current contents (accumulate = 1, for several
 * micro-batches of one step).  argmax: device int64[H] or NULL; receives the
 * flat index (b*S + i)*S + j of the maximising pair, ties to the smallest
 * index (requires B*S*S < 2^32; accumulate must be 0 with argmax).
 * A NaN/Inf logit sets MC_STATUS_NONFINITE_LOGIT. */
mc_status qk_max_logit(const mc_attn_desc* attn, float* smax, int64_t* argmax,
                       int32_t accumulate, int32_t* status, mc_stream_t stream);

/* Values and outputs of an attention forward ([K2-internals] "核心数学":
 * O^h = softmax(scale * Q^h K^h^T) V^h).  Layout [B, S, H, d_v] with unit
 * feature stride, bf16 like q and k; strides in elements, multiples of 8, and
 * 16-byte aligned pointers.  o must not overlap q, k, k_shared or v. */
typedef struct {
  const void* v;           /* device values [B, S, H, d_v]                          */
  int32_t d_v;             /* value width, 16..128                                  */
  int32_t _pad;
  int64_t v_strides[3];    /* batch, sequence, head                                 */
  void* o;                 /* device output [B, S, H, d_v] (written)                */
  int64_t o_strides[3];
  float* lse;              /* device [B, H, S]: natural log of each row's softmax
                              denominator (of the scaled logits), or NULL           */
} mc_attn_out;

/* Attention forward with the per-head max logit fused in: the S_max that
 * training takes "already computed during forward" ([K2-internals]
 * Algorithm 1).  The softmax needs each row's largest logit anyway; smax
 * receives S_max^h exactly as qk_max_logit defines it (written, or
 * max-combined when accumulate = 1).  bf16 only (MC_ERR_UNSUPPORTED
 * otherwise); q.k length d_head + d_shared in 16..192 (with a shared part,
 * d_head a multiple of 64); causal or not as attn->causal says; scale > 0.
 * Tensor cores: S = Q K^T and O += P V in fp32, P rounded to bf16 (softmax
 * numerators relative to a running row maximum), O rounded to bf16 once.
 * A NaN/Inf logit sets MC_STATUS_NONFINITE_LOGIT. */
mc_status qk_attention_forward(const mc_attn_desc* attn, const mc_attn_out* out, float* smax,
                               int32_t accumulate, int32_t* status, mc_stream_t stream);

/* QK-Clip for one attention layer.  MC_CLIP_PER_HEAD: for every head with
 * smax[h] > tau, gamma_h = tau / smax[h] and every segment's rows of head h are
 * multiplied by gamma_h^exponent; heads with smax[h] <= tau are untouched bit
 * for bit.  MC_CLIP_TOTAL: when max_h smax[h] > tau, every head's rows take
 * gamma = tau / max_h smax[h].  A NaN S_max sets MC_STATUS_NONFINITE_SMAX and
 * is never clipped on (in total mode nothing is clipped).  [K2-internals]
 * Algorithm 1 QK-Clip branch; "核心数学"; "MLA 的特殊处理".  gamma_out:
 * device float[H] or NULL; nclipped: device int or NULL (heads clipped). */
mc_status qk_clip_apply(const float* smax, int32_t H, float tau, int32_t mode,
                        const mc_clip_seg* segs, int32_t nsegs, float* gamma_out,
                        int32_t* nclipped, int32_t* status, mc_stream_t stream);

/* One MuonClip step ([K2-internals] Algorithm 1): for every matrix
 * M = mu M + G; O = NS(M) sqrt(max) rms_scale; W = W - lr (O + wd W); then for
 * every layer the per-head QK-Clip with that layer's smax (computed on the
 * forward's pre-update weights) applied to the updated weights.
 * W: bf16 or f32; G: f32 or bf16; M: f32 (the fp32 momentum state).
 * Segments in `layers` must point into matrices of W (any overlap with W is
 * allowed: the clip runs after every matrix's update). */
mc_status muonclip_step(mc_mat* W, const mc_mat* G, mc_mat* M, int32_t count,
                        const mc_hparams* hp, const mc_clip_layer* layers, int32_t nlayers,
                        void* workspace, size_t workspace_bytes, int32_t* status,
                        mc_stream_t stream);

/* Optional launch timing (observability).  While enabled, every kernel
 * launch of the library is bracketed by CUDA events recorded on the launch's
 * stream, accumulated per kernel class ("prep", "norms", "ns_gemm", "apply",
 * "clip", "max_logit").  mc_profiler_read synchronises on the recorded
 * events, writes up to `max` entries (class name, launches, total
 * milliseconds) and returns the number written; reset = 1 clears the totals.
 * Process-wide; not meant for use while several threads launch. */
typedef struct {
  char name[24];
  int32_t launches;
  float ms;
} mc_kernel_time;
void mc_profiler_enable(int32_t on);
int32_t mc_profiler_read(mc_kernel_time* out, int32_t max, int32_t reset);

/* ---- Setup (untimed): the attention layer's query/key features on the
 * library's own kernels ([K2-internals] "MLA 的特殊处理": q^C and the rotary
 * q^R from the compressed query latent, k^C from the compressed key/value
 * latent, one rotary k^R shared by every head; MHA: Q = X W_q^T, K = X W_k^T),
 * so that S_max and its re-measurement after a clip run on the library. ---- */

/* D = A B^T.  A: [M, K] row-major with pitch lda (elements), B: [N, K] with
 * pitch ldb, D: [M, N] with pitch ldd, all device memory of one dtype.
 * MC_BF16 runs on the Newton-Schulz phases' tcgen05 GEMM core (one bf16
 * plane, fp32 accumulation, D rounded to bf16); MC_F32 on the CUDA-core GEMM
 * (products summed in an unevaluated fp32 pair, D rounded to fp32).  Pointers
 * and pitches 16-byte aligned; K >= 1; M or N of 0 returns at once.
 * scratch (MC_BF16 only): device, 16-byte aligned, >= 16 bytes, caller-owned;
 * the call zeroes it as its launch's tile counter, so one call at a time may
 * use it.  A NaN/Inf in D ORs MC_STATUS_NONFINITE_UPDATE into *status
 * (device int32, nullable).  Asynchronous on `stream`. */
mc_status mc_matmul(const void* A, int64_t lda, const void* B, int64_t ldb, void* D, int64_t ldd,
                    int32_t M, int32_t N, int32_t K, int32_t dtype, void* scratch, int32_t* status,
                    mc_stream_t stream);

/* Weightless RMSNorm of each row (the MLA latents): y = x / sqrt(mean(x^2) +
 * eps) over `cols` values, fp32 arithmetic.  x, y: device, dtype MC_BF16 or
 * MC_F32, pitches ldx, ldy >= cols; in place when y == x and ldy == ldx;
 * eps >= 0; rows of 0 returns at once.  Asynchronous on `stream`. */
mc_status mc_rms_norm(const void* x, int64_t ldx, void* y, int64_t ldy, int64_t rows, int32_t cols,
                      int32_t dtype, float eps, mc_stream_t stream);

/* Rotary embedding in place on interleaved pairs.  x[b, s, h, 0..d) lives at
 * element offset b*sb + s*ss + h*sh (device, dtype MC_BF16 or MC_F32); each
 * pair (x[2k], x[2k+1]) rotates by the angle s * theta^(-2k/d) at position s
 * (0..S-1): (x0 cos - x1 sin, x0 sin + x1 cos), the angle, its cosine and sine
 * taken in fp64.  d even, 2..4096; heads nh >= 1; theta > 0.  Asynchronous
 * on `stream`. */
mc_status mc_rope(void* x, int32_t B, int32_t S, int32_t nh, int32_t d, int64_t sb, int64_t ss, int64_t sh,
                  int32_t dtype, double theta, mc_stream_t stream);

/* Diagnostic: exercises the bounded device wait that every tcgen05 kernel of
 * the library uses for its mbarrier phases.  One CTA waits on a phase that
 * nothing completes, for at most budget_ns nanoseconds of %globaltimer
 * (1 .. 1e9), or until a second warp of the CTA raises its abort flag after
 * abort_after_ns (0: never; 0 .. 1e9).  Giving up ORs MC_STATUS_TIMEOUT into
 * *status (device int32, required); *waited_ns (device uint64, nullable)
 * receives how long the wait took.  Nothing else is touched and the context
 * stays usable.  MC_ERR_INVALID_ARG (before any launch) for a budget outside
 * its range or a null status.  Asynchronous on `stream`. */
mc_status mc_selftest_bounded_wait(uint64_t budget_ns, uint64_t abort_after_ns, int32_t* status,
                                   uint64_t* waited_ns, mc_stream_t stream);

/* Thread-local description of the last non-OK return ("" if none). */
const char* mc_last_error(void);

/* Library version string. */
const char* mc_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MUONCLIP_H */
