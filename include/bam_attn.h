/*
 * bam_attn.h - C ABI of the GB300 (sm_103a) GGD-BAM attention library.
 *
 * The method: Bayesian Attention Mechanism with a Generalized-Gaussian
 * positional prior ("Bayesian Attention Mechanism" technical summary,
 * gist.science 2505.22842, section "Solution Proposee : GGD-BAM").  Every
 * query-key logit of head h gets the additive bias
 *
 *     b_h(d) = -( u / alpha_h )^beta_h,   u = |d - mu_h|,   d = i - j,
 *
 * with u clamped to max(u, eps) when beta_h <= 0 (the eps of the BAM
 * repository README, "Implementation Details", eps = 1e-5).  Logits are
 *
 *     z_ij = c_i * q_i . k_j + b_h(i - j),
 *     c_i  = 1/sqrt(D)                           (ssmax == 0)
 *     c_i  = s_h * ln(n_i) / sqrt(D)             (ssmax != 0, Scalable-Softmax)
 *
 * where n_i is the number of keys query i sees (i+1 causal, T otherwise,
 * Tkv for decode).  The output is softmax_j(z_ij) applied to V ("ALiBi:
 * Attention with Linear Biases", section "Code": scores, softmax, weights @ V).
 *
 * The prior may instead be given in the repository's own parameterisation
 * (README, "Implementation Details": the bias equation and AttentionPrior):
 *
 *     b_h(d) = -exp(theta_alpha_h) * ( |d - mu_h| + eps )^theta_beta_h,
 *     mu_h   = exp(theta_mu_h) - exp(-theta_mu_h),
 *
 * with eps added for every theta_beta (bam_params.prior = BAM_PRIOR_THETA).
 *
 * Conventions shared by every entry point
 *  - Tensors are dense, row-major, in device memory, 16-byte aligned:
 *    q, k, v, o, dO, dq, dk, dv are [B, H, T, D]; lse is [B, H, T].
 *    bf16 tensors hold IEEE bfloat16 bit patterns.
 *  - D must be 64 (other head sizes return BAM_ERR_UNSUPPORTED).
 *  - The caller owns every buffer.  The library allocates nothing: scratch
 *    space is the caller's workspace `ws` of at least
 *    bam_attn_workspace_size(op, ...) bytes, 256-byte aligned.  A workspace
 *    may be reused by calls that do not overlap on the GPU.
 *  - Calls are asynchronous on `stream`.  Argument errors are returned
 *    before anything is launched; launch failures return BAM_ERR_CUDA.
 *  - Every on-device wait is bounded.  A kernel that gives up records
 *    BAM_ERR_TIMEOUT in the workspace status word and returns; read it with
 *    bam_attn_check_status().  A recorded error stays until it is read: a
 *    later call on the same workspace runs normally but neither erases nor
 *    overwrites it (the first error since the last check is reported).
 *  - A call runs on the device current at the call.  The kernels'
 *    shared-memory limits are raised once per device and the SM count is
 *    read once per device, so one process may drive several GPUs.
 */
#ifndef BAM_ATTN_H_
#define BAM_ATTN_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  BAM_OK = 0,
  BAM_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer      */
  BAM_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. D != 64)        */
  BAM_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed            */
  BAM_ERR_TIMEOUT = 4,     /* a device-side wait gave up (see check_status)   */
  BAM_ERR_WORKSPACE = 5,   /* workspace missing, misaligned or too small      */
  BAM_ERR_BOUNDS = 6       /* debug build only: a copy's bounds check failed  */
} bam_status;

/* Parameterisations of the prior (bam_params.prior). */
enum {
  BAM_PRIOR_ALPHA = 0, /* b = -(u/alpha)^beta; alpha > 0; eps clamps u when beta <= 0 */
  BAM_PRIOR_THETA = 1  /* b = -exp(theta_alpha)(|d - mu| + eps)^theta_beta,
                          mu = 2 sinh(theta_mu); any real thetas; eps always added */
};

/* Per-head prior and SSMax parameters.  alpha, beta, mu, s point to device
 * fp32 arrays of length H; s is read only when ssmax != 0.  With
 * BAM_PRIOR_ALPHA: alpha_h > 0, and eps (README: 1e-5) is the clamp of
 * |d - mu| used when beta_h <= 0.  With BAM_PRIOR_THETA: alpha, beta, mu hold
 * theta_alpha, theta_beta, theta_mu, eps is added to |d - mu| for every head,
 * and bam_attn_bwd's dalpha, dbeta, dmu are the gradients with respect to
 * those thetas.  eps > 0 in both. */
typedef struct {
  const float* alpha;
  const float* beta;
  const float* mu;
  const float* s;
  float eps;
  int causal; /* 1: key j visible to query i iff j <= i; 0: all keys visible */
  int ssmax;  /* 1: Scalable-Softmax logit scale s_h * ln(n_i)               */
  int prior;  /* BAM_PRIOR_ALPHA or BAM_PRIOR_THETA                         */
} bam_params;

enum { BAM_OP_FWD = 0, BAM_OP_BWD = 1, BAM_OP_DECODE = 2 };

/* Bytes of workspace that op (BAM_OP_*) needs for these sizes (T = Tkv for
 * decode).  Returns 0 for invalid sizes.  Host-only; launches nothing. */
size_t bam_attn_workspace_size(int op, int B, int H, int T, int D);

/* Forward (prefill).  q, k, v: bf16 [B,H,T,D].  o: [B,H,T,D], fp32 when
 * o_fp32 != 0, else bf16.  lse: fp32 [B,H,T] natural-log log-sum-exp of the
 * logits of each row (may be NULL; bam_attn_bwd needs it).  T >= 1.
 * Steps: per-head distance table b_h(d) into ws (fp32, with the exponent
 * beta * log2(u / alpha) carried as a two-float sum so that b keeps a few
 * 1e-7 relative error at any magnitude), then the fused tiled kernel
 * (tensor-core QK^T and PV, online softmax). */
bam_status bam_attn_fwd(const void* q, const void* k, const void* v, void* o, int o_fp32,
                        float* lse, int B, int H, int T, int D, const bam_params* p,
                        void* ws, size_t ws_bytes, cudaStream_t stream);

/* Backward of L = sum(O * dO) ("plain chain rule"; the pages give no
 * backward).  q, k, v, dO: bf16 [B,H,T,D]; o and lse: the forward's outputs
 * (o fp32 when o_fp32 != 0, else bf16).  Outputs: dq, dk, dv bf16
 * [B,H,T,D]; dalpha, dbeta, dmu, ds fp32 [H], overwritten, summed over the
 * batch (ds is written as 0 when ssmax == 0); with BAM_PRIOR_THETA the first
 * three are d/dtheta_alpha, d/dtheta_beta, d/dtheta_mu.  The call's first
 * kernel zeroes these four and later kernels add partial sums into them with
 * atomics (so their last bits depend on the order); after a device-side
 * give-up they hold partial sums. */
bam_status bam_attn_bwd(const void* q, const void* k, const void* v, const void* o,
                        int o_fp32, const float* lse, const void* dO, void* dq, void* dk,
                        void* dv, float* dalpha, float* dbeta, float* dmu, float* ds, int B,
                        int H, int T, int D, const bam_params* p, void* ws, size_t ws_bytes,
                        cudaStream_t stream);

/* Decode: one new query per (b, h) against a KV cache that already holds
 * its key and value.  q: bf16 [B,H,D]; kc, vc: bf16 [B,H,Tkv,D].  The query
 * sits at position Tkv-1, every cached key is visible and n = Tkv.
 * o: [B,H,D] fp32 when o_fp32 != 0, else bf16; lse: fp32 [B,H] or NULL.
 * p->causal is ignored.  Split-KV partials go to ws.  If a device wait of the
 * call gives up, o and lse are written as NaN (and bam_attn_check_status
 * reports BAM_ERR_TIMEOUT). */
bam_status bam_attn_decode(const void* q, const void* kc, const void* vc, void* o, int o_fp32,
                           float* lse, int B, int H, int Tkv, int D, const bam_params* p,
                           void* ws, size_t ws_bytes, cudaStream_t stream);

/* Ragged decode: as bam_attn_decode, but sequence b holds only
 * cache_lens[b] keys, at positions 0 .. cache_lens[b]-1 of its [Tmax, D]
 * cache rows (kc, vc: bf16 [B,H,Tmax,D]).  Its query sits at position
 * cache_lens[b]-1, so key j is at distance cache_lens[b]-1-j, and
 * n = cache_lens[b] for Scalable-Softmax.  cache_lens: device int32 [B],
 * read on the device; each must lie in [1, Tmax].  A length outside it is
 * clamped into it (no out-of-bounds access) and recorded, and
 * bam_attn_check_status then returns BAM_ERR_INVALID_ARG.  The workspace is
 * the one bam_attn_workspace_size(BAM_OP_DECODE, B, H, Tmax, D) gives. */
bam_status bam_attn_decode_varlen(const void* q, const void* kc, const void* vc,
                                  const int* cache_lens, void* o, int o_fp32, float* lse,
                                  int B, int H, int Tmax, int D, const bam_params* p, void* ws,
                                  size_t ws_bytes, cudaStream_t stream);

/* Paged decode: as bam_attn_decode_varlen, with the cache in pages.
 * k_pages, v_pages: bf16 [num_pages, H, page, D]; page is a multiple of 64.
 * block_table: device int32 [B, max_blocks]; logical block i of sequence b
 * (its keys i*page .. i*page+page-1) is page block_table[b*max_blocks + i].
 * cache_lens: device int32 [B], each in [1, max_blocks*page]; only the blocks
 * that hold a sequence's keys are read.  Out-of-range lengths or page numbers
 * are clamped on the device (page 0) and reported by bam_attn_check_status as
 * BAM_ERR_INVALID_ARG.  The workspace is the one
 * bam_attn_workspace_size(BAM_OP_DECODE, B, H, max_blocks*page, D) gives. */
bam_status bam_attn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                                 const int* block_table, const int* cache_lens, void* o,
                                 int o_fp32, float* lse, int B, int H, int page, int max_blocks,
                                 int num_pages, int D, const bam_params* p, void* ws,
                                 size_t ws_bytes, cudaStream_t stream);

/* Synchronises `stream`, then reads and clears the device status word of
 * `ws`.  Returns BAM_OK, BAM_ERR_TIMEOUT (a device wait gave up),
 * BAM_ERR_INVALID_ARG (a device-read argument was out of range: a ragged or
 * paged decode's cache length or page number), BAM_ERR_BOUNDS (debug build:
 * a bulk copy failed its bounds check and was not issued; the call's outputs
 * are then invalid) or BAM_ERR_CUDA.  The result is the first error recorded
 * by any call on `ws` since the previous check (errors are not cleared by
 * later calls).  A workspace no call has used reports BAM_OK. */
bam_status bam_attn_check_status(void* ws, cudaStream_t stream);

/* Debug build only (bam_attn_debug_build() == 1; BAM_ERR_UNSUPPORTED
 * otherwise): arms the give-up count of `ws`.  The next calls on `ws` count
 * their bounded device waits, and the n-th one gives up as if its time limit
 * had passed: the kernel records BAM_ERR_TIMEOUT, drains its own in-flight
 * copies and tensor-core work, frees its Tensor Memory and returns, and the
 * rest of the call follows the abort.  This drives the give-up paths of the
 * real kernels without a hang.  n = 0 disarms.  Synchronises the device.
 * Not part of any attention call. */
bam_status bam_attn_debug_arm_giveup(void* ws, int n);

/* 1 when the library was built with BAM_DEBUG, else 0.  The debug build is
 * the same library with every plain bulk copy (the distance-table windows of
 * the forward and backward, the K, V and table stages of the decode) checked
 * before it is issued: its source must lie inside its own table row (up to
 * the padding after the last row), cache row or page, and its addresses and
 * size must be multiples of 16 bytes.  The row coordinate of every tiled
 * store and reduction is checked to lie in [0, T).  A failed check records
 * BAM_ERR_BOUNDS, skips the copy and aborts the call; nothing traps. */
int bam_attn_debug_build(void);

/* Self-test of the failure detection: launches one thread that waits, with
 * the library's bounded wait, on a barrier nothing arrives at.  After the
 * wait limit (2 s) it records BAM_ERR_TIMEOUT in the status word of `ws`
 * (at least 256 bytes, 256-byte aligned) and returns; the context stays
 * usable.  Read the result with bam_attn_check_status.  Not part of any
 * attention call. */
bam_status bam_attn_selftest_wait(void* ws, size_t ws_bytes, cudaStream_t stream);

/* Static description of a status code. */
const char* bam_status_string(bam_status s);

/* Decode without a workspace argument, for callers that cannot allocate
 * device memory: plugin-style hosts that hand a library only its input and
 * output pointers and own every other byte through their own allocator, or
 * decode loops that cannot afford cudaMalloc's possible device-wide
 * synchronisation.  The pages have no counterpart; this is an interface
 * variant of bam_attn_decode (same kernels, same arguments and results).
 *
 * Scratch comes from a fixed array of BAM_DECODE_NOALLOC_SCRATCH_BYTES in
 * the library's device image, held by every GPU that loads the library until
 * the process exits.  Sizes whose scratch (the same amount that
 * bam_attn_workspace_size(BAM_OP_DECODE, ...) reports) exceeds it return
 * BAM_ERR_WORKSPACE before anything is launched.  Nothing is allocated or
 * freed.  The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture on the device.  All calls share the array:
 * calls that overlap on the GPU (for example on two streams) race on it.
 * A device-side give-up writes NaN to o and lse and is recorded in that
 * array; bam_attn_decode_noalloc_check_status reads it. */
#define BAM_DECODE_NOALLOC_SCRATCH_BYTES (4u << 20)
bam_status bam_attn_decode_noalloc(const void* q, const void* kc, const void* vc, void* o,
                                   int o_fp32, float* lse, int B, int H, int Tkv, int D,
                                   const bam_params* p, cudaStream_t stream);

/* bam_attn_check_status for bam_attn_decode_noalloc on the current device:
 * synchronises `stream`, then reads and clears the status words kept at the
 * start of the no-alloc scratch array (the first error of any no-alloc call
 * on this device since the previous check).  Allocates nothing.  The pages
 * have no counterpart. */
bam_status bam_attn_decode_noalloc_check_status(cudaStream_t stream);

/* bam_attn_debug_arm_giveup for the no-alloc scratch of the current device
 * (debug build only; BAM_ERR_UNSUPPORTED otherwise). */
bam_status bam_attn_debug_arm_giveup_noalloc(int n);

/* Work schedule of the causal backward's persistent grid (host only:
 * launches nothing, needs no GPU; for tests and tools).  With `grid` CTAs
 * (the backward uses min(grid, B*H*ceil(T/128)) of them, grid = the SM
 * count), CTA c runs items item[start[c]] .. item[start[c+1]-1] in that
 * order; item w is key tile w / (B*H) of (b, h) = w % (B*H).  `start` holds
 * at least min(grid, items) + 1 ints, `item` at least max_items.  Returns the
 * number of scheduled items; 0 when the kernel deals the items out
 * round-robin itself (non-causal, too many items, or no better makespan);
 * -1 on a bad argument or when max_items is too small. */
int bam_attn_bwd_schedule(int B, int H, int T, int causal, int grid, int* start, int* item,
                          int max_items);

/* Kernels that bam_attn_profile_events can bracket. */
enum {
  BAM_KERNEL_TABLE = 0,      /* distance-table kernel (fwd, decode)        */
  BAM_KERNEL_FWD = 1,        /* fused forward                               */
  BAM_KERNEL_BWD_PREP = 2,   /* backward preprocess (tables, Delta, zeroing) */
  BAM_KERNEL_BWD = 3,        /* fused backward                              */
  BAM_KERNEL_BWD_FINAL = 4,  /* dq conversion and scalar-gradient finish    */
  BAM_KERNEL_DECODE = 5,     /* split-KV decode                             */
  BAM_KERNEL_DECODE_COMBINE = 6,
  BAM_KERNEL_COUNT = 7
};

/* Instrumentation: while set, every launch of kernel `which` is bracketed
 * by records of `before` and `after` on the launch stream (external records,
 * so that a captured CUDA graph keeps them as event-record nodes).  Pass
 * NULL events to clear.  Not thread-safe with concurrent callers. */
bam_status bam_attn_profile_events(int which, cudaEvent_t before, cudaEvent_t after);

/* Number of kernel launches the library has issued since load (all kinds). */
uint64_t bam_attn_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* BAM_ATTN_H_ */
