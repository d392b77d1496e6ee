/*
 * vc_attn.h -- C ABI of the GB300 (sm_103a) ExpCast-FP8 + V-Smooth FP8 attention forward.
 *
 * The operation is the non-causal self-attention forward of
 *   "VC-Attention: Value Smoothing and Softmax Casting for Low-bit Attention"
 *   (Sec. 3.1 Eq. 1 online softmax; Sec. 3.2 Eq. 3-6 value-guided permutation, block demeaning
 *   and online mean restoration; Sec. 3.3 Eq. 7 ExpCast-FP8)
 * with the scheduling rules of
 *   "Open-VC Attention: an open-source, error-tunable variant of VC-Attention" (MachGen blog),
 *   "Scheduling around ExpCast": Q/K scaled per 128-token block, V per head, one FMA per score,
 *   running maximum on the true score with every increase applied, row sum built from the
 *   decoded FP8 probabilities that feed PV, mid-window key order, packed transposed V.
 *
 * Conventions shared by every call:
 *   - Pointers named as device pointers must be device memory on the current CUDA device
 *     (or managed memory); host pointers are plain host memory.
 *   - Tensors are dense, row-major, without padding: Q, K, V, O are bf16 [B, H, S, D].
 *   - All work is enqueued on `stream` (0 = legacy default stream) and is asynchronous: inputs
 *     must stay valid and unmodified until the stream reaches the call; outputs are ready when
 *     the stream has passed it.
 *   - Return value: VC_OK (0) or a negative VC_ERR_* code. Nothing aborts or prints. On an
 *     error the outputs are unspecified and the plan (if any) is left usable or destroyed as
 *     stated per call.
 *   - Supported shapes: D in {64, 128}; 1 <= S <= 1048576; B*H >= 1; B*H*ceil(S/128)*128*D below
 *     2^40 bytes; 1 <= k_clusters <= min(S, 1024); 1 <= iters <= 64 whenever k-means runs.
 *   - No CPU fallback: every step of the computation runs in this library's CUDA kernels.
 */
#ifndef VC_ATTN_H
#define VC_ATTN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------------------------- */
enum {
  VC_OK = 0,
  VC_ERR_INVALID_ARG = -1,   /* null pointer, bad size or flag combination                */
  VC_ERR_UNSUPPORTED = -2,   /* shape outside the supported set (e.g. D not 64/128)       */
  VC_ERR_CUDA = -3,          /* a CUDA runtime call or kernel launch failed               */
  VC_ERR_TIMEOUT = -4,       /* a kernel gave up waiting on an internal hand-off          */
  VC_ERR_PLAN_MISMATCH = -5, /* an existing plan has a different shape                    */
  VC_ERR_OOM = -6,           /* device allocation failed                                  */
  VC_ERR_NO_DEVICE = -7      /* the current device is not an sm_103 GPU                   */
};

/* ---- flags ----------------------------------------------------------------------------- */
enum {
  /* Score -> E4M3 probability code by one FMA, Eq. 7 of the VC-Attention paper (Sec. 3.3).
     Off: exponentiate in fp32 (exp2f) and convert with a rounding E4M3 cast. */
  VC_EXPCAST = 1u,
  /* V-Smooth (Sec. 3.2): k-means grouping, permutation of K and V, 128-row block means
     restored in the accumulator. Off (prepare): identity permutation and no means. */
  VC_VSMOOTH = 2u,
  /* Mid-window key order ("Open-VC Attention", mid-window key traversal): the query tiles 2m and
     2m+1 share one order that starts at key tile min(nkb-1, 2m+2), sweeps down to tile 0, then
     visits the tail. Off: 0..nkb-1. */
  VC_MIDWINDOW = 4u,
  /* Prepare only: K channel centering (VC-Attention Sec. 3.4 "Fused preprocessing", App. B). Every
     key has the head's channel mean mu (bf16 of the exact mean over the S tokens) subtracted in fp32
     before its block quantisation; the softmax is unchanged, the keys' quantisation range shrinks. */
  VC_KCENTER = 8u,
  /* Prepare only: begin the k-means rounds from the plan's centroids of its previous grouping
     instead of the rows floor(i*S/k) (VC-Attention Sec. 3.2 "Unbalanced clusters cost little":
     warm-starting from the previous step's centroids halves the grouping cost). Needs a plan that
     has been grouped before (else VC_ERR_INVALID_ARG); ignored when no k-means runs. */
  VC_WARM_START = 16u,
  /* Prepare only: keep the plan's permutation from an earlier prepare, no k-means (the grouping
     schedule's reuse steps). With VC_VSMOOTH the block means are recomputed on the new V; without it
     the permutation is kept and no means are used ("the plain low-bit kernel on the permutation the
     window left behind"). Needs a plan prepared before; not with an explicit perm. */
  VC_REUSE_PERM = 32u,
  /* Prepare only: one residual scale per channel instead of one per head (VC-Attention Sec. 3.2
     "Block demeaning": the residual is quantised per channel to E4M3; App. B: the block means the
     forward reads are stored divided by the channel scale, so one multiply per channel in the
     epilogue restores both terms of Eq. 6).  s_d = max_t |R[t, d]| / 448 over the head (1 for an
     all-zero channel); codes E4M3(R[t, d] * (448 / amax_d)); forward means bf16(mu / s_d).  The
     forward then computes O[:, d] = s_d * A[:, d] / l. */
  VC_VSCALE_CHANNEL = 64u,
  /* Prepare only: rotate every Q row and every K row (after the K centre) by the unnormalised
     Walsh-Hadamard transform before the block quantiser (VC-Attention Sec. 3.4 "Fused preprocessing",
     App. B: the Q and K passes fuse a Hadamard rotation; QK^T is unchanged since H H^T = D I). Computed
     in fp32 as the butterfly with stages 1, 2, ..., D/2 in that order; the forward's score constant
     becomes 8 log2(e) / (D sqrt(D)). */
  VC_QK_HADAMARD = 128u,
  /* Test hook: the forward kernel's first internal wait gives up at once, so the call reports
     VC_ERR_TIMEOUT through vc_plan_status() without hanging. */
  VC_DEBUG_TIMEOUT = 1u << 16
};
#define VC_FLAGS_DEFAULT (VC_EXPCAST | VC_VSMOOTH | VC_MIDWINDOW)

/* ---- the plan ----------------------------------------------------------------------------
 * Opaque object owning the device buffers the prepare step writes and the forward reads:
 * the permutation pi, the E4M3 codes of Q and of K' = K[pi] with one fp32 scale per 128-token
 * block, the E4M3 codes of the V' residual stored transposed and zero-padded as [B, H, D, S_pad]
 * (key dimension contiguous, the layout of the PV operand) with one fp32 scale per head, the
 * bf16 128-row block means, the k-means labels and centroids, and a device status word.
 * S_pad = 128 * ceil(S/128).  The library owns these buffers until vc_plan_destroy().
 * A plan belongs to the device that was current when it was created: preparing into it or running
 * the forward with another current device returns VC_ERR_INVALID_ARG.                         */
typedef struct vc_plan vc_plan;

/* vc_attn_prepare
 * Grouping and quantisation (VC-Attention Sec. 3.2 "Value-guided permutation", "Block
 * demeaning"; Sec. 3.4 "Fused preprocessing"; Open-VC "Fused input preparation"):
 *   per (b, h): k-means over the V rows (k_clusters centroids, `iters` Lloyd rounds, started
 *   from the rows floor(i*S/k)), pi = stable argsort of the labels, K' = K[pi], V' = V[pi];
 *   Q and K' quantised to E4M3 with one scale per 128-token block (scale = absmax/448);
 *   mu_j = mean of the valid rows of block j of V', stored as bf16; R = V' - mu_j quantised to
 *   E4M3 with one scale per head (absmax/448), stored transposed and padded.
 * Q, K, V: device bf16 [B, H, S, D].  k_clusters, iters: k-means size and rounds
 * (1 <= iters <= 64, else VC_ERR_INVALID_ARG; each round = assignment, argsort, centroid update).
 * *plan: NULL to allocate a new plan, or an
 * existing plan of the same (B, H, S, D, k_clusters), whose buffers are reused without any
 * allocation (VC_ERR_PLAN_MISMATCH if the shape differs; the plan is left untouched).
 * The first call allocates device memory (synchronous cudaMalloc); later calls reusing the plan
 * are fully asynchronous and can be captured in a CUDA graph. */
int vc_attn_prepare(const void* Q, const void* K, const void* V, int B, int H, int S, int D, int k_clusters,
                    int iters, cudaStream_t stream, vc_plan** plan);

/* vc_attn_prepare_ex -- vc_attn_prepare with control over grouping.
 * perm: NULL, or a device int32 [B, H, S] permutation per (b, h) to use instead of k-means
 *   (reusing the permutation across denoising steps, VC-Attention Sec. 3.4 "Amortized grouping
 *   schedule"; it is not checked to be a permutation -- every entry must lie in [0, S)).
 * flags: VC_VSMOOTH set -> group (unless perm is given) and demean; clear -> identity
 *   permutation (perm ignored), no means, R = V.  VC_KCENTER set -> subtract the keys' channel
 *   centre before their quantisation.  VC_VSCALE_CHANNEL set -> one residual scale per channel.
 *   VC_QK_HADAMARD set -> Q and K rows rotated before their quantisation.
 *   VC_WARM_START / VC_REUSE_PERM as documented with the flags.  Other bits are ignored here. */
int vc_attn_prepare_ex(const void* Q, const void* K, const void* V, int B, int H, int S, int D, int k_clusters,
                       int iters, const int32_t* perm, unsigned flags, cudaStream_t stream, vc_plan** plan);

/* vc_attn_prepare_repair -- prepare without V-Smooth, plus V residual repair rows ("Open-VC
 * Attention", "Why V residual repair").
 * Per (b, h): Q and K quantised per 128-token block, V quantised per head (or per channel with
 * VC_VSCALE_CHANNEL) as in vc_attn_prepare_ex without VC_VSMOOTH; then every token j gets the energy
 *   e_j = sum_c (s_c * (x_jc - E4M3(x_jc)))^2,  x_jc = fl32(V_jc * 448 / amax_c),
 * accumulated as fp32 fused multiply-adds in channel order; the n_repair tokens of largest energy
 * (ties to the lower index) are kept in ascending token order. Their bf16 keys are copied into
 * ceil(n_repair/128) extra key blocks, quantised like any key block (one scale per block, minus the
 * K centre with VC_KCENTER), and their residuals x - E4M3(x) are coded in E4M3 in the same code units
 * as the main residual codes. The forward visits these repair tiles after every regular tile; they
 * neither raise the running max (their codes clip at 120) nor add to the row sum, so they change the
 * numerator only.
 * n_repair: 0 <= n_repair <= S rows per head (the pages' operating point is ceil(0.005 * S)); it is
 *   part of the plan's shape (VC_ERR_PLAN_MISMATCH when an existing plan has another count).
 * flags: VC_KCENTER | VC_VSCALE_CHANNEL | VC_QK_HADAMARD; VC_VSMOOTH or VC_REUSE_PERM -> VC_ERR_INVALID_ARG.
 * Other arguments, allocation and asynchrony as vc_attn_prepare. */
int vc_attn_prepare_repair(const void* Q, const void* K, const void* V, int B, int H, int S, int D, int n_repair,
                           unsigned flags, cudaStream_t stream, vc_plan** plan);

/* vc_attn_forward
 * The fused attention forward (VC-Attention Eq. 1, 6, 7): for every query row, key tiles of
 * 128 are visited in the chosen order; S = Q K'^T on FP8 tensor cores; the running maximum is
 * kept on the true score in code units and every increase rescales the accumulator; each score
 * becomes an E4M3 code c = clip[0,120](rne(S*a_j + 119.65 - M)) with a_j = 8 log2(e)/sqrt(D)
 * * sQ * sK_j (or the exp-then-cast path without VC_EXPCAST); the codes multiply the residual
 * codes of V' on FP8 tensor cores; the row sum of the decoded codes (the denominator) and the
 * block means (VC_VSMOOTH) enter the accumulator; O = sV * A / l in bf16 (per channel,
 * O[:, d] = s_d * A[:, d] / l, when the plan was prepared with VC_VSCALE_CHANNEL).
 * plan: from vc_attn_prepare.  O: device bf16 [B, H, S, D], rows in the original token order.
 * flags: VC_EXPCAST | VC_MIDWINDOW | VC_VSMOOTH (VC_VSMOOTH is ignored when the plan was
 * prepared without means) | VC_DEBUG_TIMEOUT.  Kernel-side timeouts are reported
 * asynchronously through vc_plan_status(). Allocates nothing; can be captured in a graph. */
int vc_attn_forward(const vc_plan* plan, void* O, unsigned flags, cudaStream_t stream);

/* ---- plan inspection (tests, benchmarks, reuse of pi) ----------------------------------- */
enum {
  VC_PLAN_LABELS = 1,    /* int32 [B, H, S]       k-means labels of the last round            */
  VC_PLAN_PERM = 2,      /* int32 [B, H, S]       pi                                          */
  VC_PLAN_QCODES = 3,    /* uint8 [B, H, S_pad, D] E4M3 codes of Q (pad rows 0)              */
  VC_PLAN_QSCALES = 4,   /* fp32  [B, H, nkb]                                                 */
  VC_PLAN_KCODES = 5,    /* uint8 [B, H, S_pad, D] E4M3 codes of K' = K[pi]                  */
  VC_PLAN_KSCALES = 6,   /* fp32  [B, H, nkb]                                                 */
  VC_PLAN_VCODES = 7,    /* uint8 [B, H, D, S_pad] E4M3 codes of the residual, transposed     */
  VC_PLAN_VSCALES = 8,   /* fp32  [B, H]           per-head residual scale (with
                                                     VC_VSCALE_CHANNEL: the largest channel scale) */
  VC_PLAN_MEANS = 9,     /* bf16  [B, H, nkb, D]   block means of V'                          */
  VC_PLAN_CENTROIDS = 10, /* fp32 [B, H, k, D]     centroids after the last update           */
  VC_PLAN_KCENTER = 11,  /* bf16  [B, H, D]        K channel centre (prepared with VC_KCENTER) */
  VC_PLAN_VCHSCALES = 12, /* fp32 [B, H, D]        the residual scale of each channel (all equal
                                                     to the head's scale without VC_VSCALE_CHANNEL) */
  VC_PLAN_MEANS_T = 13,  /* bf16  [B, H, D, nkb16] the means as the forward reads them: transposed,
                                                     nkb16 = 16*ceil(nkb/16) with zero pad columns,
                                                     divided by the channel scale with
                                                     VC_VSCALE_CHANNEL, else in true units         */
  VC_PLAN_REPAIR_IDX = 14,     /* int32 [B, H, n_repair]  repaired tokens, ascending                */
  VC_PLAN_REPAIR_ENERGY = 15,  /* fp32  [B, H, S]         residual energy of every token            */
  VC_PLAN_REPAIR_KCODES = 16,  /* uint8 [B, H, R_pad, D]  E4M3 codes of the copied keys (pad rows 0),
                                                          R_pad = 128 * ceil(n_repair / 128)        */
  VC_PLAN_REPAIR_KSCALES = 17, /* fp32  [B, H, R_pad/128] one scale per repair key block           */
  VC_PLAN_REPAIR_VCODES = 18   /* uint8 [B, H, D, R_pad]  E4M3 codes of the repaired residuals,
                                                          transposed (pad 0)                        */
};
/* Size in bytes of one plan tensor (0 for an unknown `what` or a NULL plan). */
size_t vc_plan_size(const vc_plan* plan, int what);
/* Enqueue a copy of one plan tensor into dst (host or device memory, `bytes` >= its size). */
int vc_plan_get(const vc_plan* plan, int what, void* dst, size_t bytes, cudaStream_t stream);
/* Synchronise `stream`, read and clear the plan's device status word. Returns VC_OK, or
 * VC_ERR_TIMEOUT if a kernel recorded a timeout since the last call (bits in *bits if non-NULL).
 * Every wait inside the kernels is bounded; a wait that runs out sets a bit and the kernel
 * returns without touching its outputs further:
 *   1 forward: score tile wait      2 forward: P / S-buffer hand-off   4 forward: a TMA load
 *   8 forward: PV completion       16 forward: teardown drain         32 k-means assignment */
int vc_plan_status(vc_plan* plan, cudaStream_t stream, int* bits);
/* Shape of a plan; any output pointer may be NULL. */
int vc_plan_shape(const vc_plan* plan, int* B, int* H, int* S, int* D, int* k_clusters);
/* Free a plan and its device buffers (synchronises the device first). NULL is a no-op. */
void vc_plan_destroy(vc_plan* plan);

/* ---- single-step exports (unit tests of individual steps) ------------------------------ */
/* ExpCast-FP8 codes (VC-Attention Eq. 7): out[i] = clip[0,120](rne(fmaf(s[i], a[i], b[i]))),
 * computed by the forward kernel's own code path.  s, a, b: device fp32 [n]; out: device u8. */
int vc_expcast_encode(const float* s, const float* a, const float* b, int64_t n, uint8_t* out, cudaStream_t stream);
/* The same code path without the final clamp at 120: exactly the bytes the forward writes on its fast
 * path, which it takes while the running max |M| < 2^22 code units (Open-VC Attention, "Scheduling
 * around ExpCast": one FMA per score, round, clamp only at 0). With b = 119.65f - M and fl(s*a) <= M
 * there, every byte equals vc_expcast_encode's; outside that range bytes above 120 may occur (up to
 * 255). Same arguments and errors as vc_expcast_encode. */
int vc_expcast_encode_unclamped(const float* s, const float* a, const float* b, int64_t n, uint8_t* out,
                                cudaStream_t stream);

/* ---- allocation-free variant ----------------------------------------------------------- */
/* The pages have no counterpart to this call; it exists for callers that must not allocate
 * device memory (for instance a framework whose memory pool already owns the whole device, or
 * host code that may only allocate at start-up).
 * vc_residual_pack_noalloc computes the value side of the prepare step -- for each (b, h), the
 * gather V' = V[pi], the bf16 means of its 128-row blocks and the per-head E4M3 residual codes,
 * transposed and zero-padded -- exactly as vc_attn_prepare_ex writes them into a plan
 * (VC_PLAN_MEANS, VC_PLAN_VCODES, VC_PLAN_VSCALES), into buffers the caller provides.
 * V: device bf16 [B, H, S, D]; perm: device int32 [B, H, S] or NULL for the identity; means: device
 * bf16 [B, H, ceil(S/128), D]; vcodes: device uint8 [B, H, D, S_pad]; vscales: device fp32 [B, H].
 * V, means and vcodes must be 16-byte aligned, perm and vscales 4-byte aligned (else
 * VC_ERR_INVALID_ARG). Each row of perm must be a permutation of [0, S): an entry outside that range
 * is not checked and makes the gather read outside V (undefined behaviour).
 * It calls no cudaMalloc, cudaFree or allocating library routine. Its only scratch (one word per
 * batch-head) is a fixed array inside the library, VC_NOALLOC_MAX_HEADS words per GPU, kept until
 * the process exits: B*H above that limit returns VC_ERR_UNSUPPORTED. Every call looks up that
 * array's address on the current device (no allocation; it stays valid across a device reset); the
 * first call on a device also loads the library's module there, so make that first call before any
 * stream capture. Each call clears the scratch on `stream` before use, but all calls share it: calls
 * that overlap on the GPU (other streams, other host threads) race and must be serialised by the
 * caller. */
#define VC_NOALLOC_MAX_HEADS 4096
int vc_residual_pack_noalloc(const void* V, const int32_t* perm, int B, int H, int S, int D, void* means,
                             uint8_t* vcodes, float* vscales, cudaStream_t stream);

/* ---- grouping schedule ------------------------------------------------------------------ */
/* What a denoising step of an n_steps run does (VC-Attention Sec. 3.4 "Amortized grouping schedule",
 * App. A "Grouping schedule"): grouping and demeaning run on the first ceil(n_steps/4) steps; inside
 * that window the permutation is computed at every `reuse`-th step (the pages use 4: steps 0, 4, 8 of
 * a 40-step run) and reused in between; later steps run the plain kernel on the kept permutation.
 * Returns a VC_STEP_* value, or VC_ERR_INVALID_ARG for step outside [0, n_steps), n_steps < 1 or
 * reuse < 1.  Pure host logic: needs no device.  Prepare flags per action:
 *   VC_STEP_GROUP      VC_VSMOOTH                  (k-means from scratch)
 *   VC_STEP_GROUP_WARM VC_VSMOOTH | VC_WARM_START  (from the previous centroids, fewer rounds)
 *   VC_STEP_REUSE      VC_VSMOOTH | VC_REUSE_PERM  (same pi, new means)
 *   VC_STEP_PLAIN      VC_REUSE_PERM               (same pi, no means) */
enum { VC_STEP_GROUP = 0, VC_STEP_GROUP_WARM = 1, VC_STEP_REUSE = 2, VC_STEP_PLAIN = 3 };
int vc_schedule_action(int step, int n_steps, int reuse);

/* Human-readable text of a status code (static storage). */
const char* vc_strerror(int status);
/* Library version string. */
const char* vc_version(void);

#ifdef __cplusplus
}
#endif
#endif /* VC_ATTN_H */
