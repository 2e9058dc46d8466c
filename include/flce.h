/*
 * flce.h -- C ABI of the fused linear cross-entropy + entropy library (libflce.so)
 * for NVIDIA GB300 (sm_103a).
 *
 * The operation (verl PR #462, "Equivalent compute logic" and "API"):
 *     logits  = hidden[N,H] @ weight[H,V]                (never stored)
 *     z       = softcap * tanh(logits / softcap)          (softcap > 0 only;
 *                                                          Liger-Kernel issue #127)
 *     p       = softmax(z) over the vocabulary
 *     lse_n   = logsumexp_v z_nv,   Ez_n = sum_v p_nv z_nv
 *     ce_n    = lse_n - z_{n,y_n}                         (the page returns -ce as logprobs)
 *     ent_n   = lse_n - Ez_n                              (entropy of p_n)
 *     loss_n  = ce_n + zloss_coef * lse_n^2               (z-loss: Liger-Kernel PR #435,
 *                                                          "Changes Made"; formula is a reading)
 *   With label smoothing eps and per-class weights w (options named in the
 *   Liger-Kernel PR #551 review; defined as torch's cross_entropy(weight,
 *   label_smoothing)): ce_n = (1-eps) w_{y_n} (lse_n - z_{n,y_n})
 *                             + eps/V sum_v w_v (lse_n - z_nv);
 *   the mean then divides the sum of ce_n by the sum of w_{y_n} over non-ignored
 *   rows, while z-loss and entropy stay unweighted (divided by the row count).
 *   Rows whose label equals ignore_index contribute exactly 0 to loss and entropy
 *   (Liger-Kernel PR #551, review: mean divides by the non-ignored count).
 *   Reduction (Liger-Kernel PR #435, "Summary"): NONE returns loss[N], entropy[N];
 *   SUM returns the sums over non-ignored rows; MEAN divides both sums by the
 *   number of non-ignored rows (0 when every row is ignored).
 *
 *   Backward, for upstream gradients g_loss, g_entropy (per token for NONE,
 *   scalars otherwise; scaled by 1/n_valid for MEAN; zero on ignored rows):
 *     dz_nv   = gl_n (p_nv - [v == y_n] + 2 coef lse_n p_nv) - ge_n p_nv (z_nv - Ez_n)
 *     dz'_nv  = dz_nv (1 - (z_nv/softcap)^2)              (soft-cap chain rule)
 *     dhidden = dz' @ weight^T,   dweight = hidden^T @ dz'
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers to dense row-major arrays, owned by
 *     the caller; the library allocates no device memory and keeps no state
 *     between calls apart from per-device caches (device attributes, the no-alloc
 *     scratch address) and the per-thread side streams described below.
 *   - hidden, weight, dhidden, dweight: bf16 (IEEE bfloat16 bit patterns; dhidden fp32
 *     when params->dhidden_fp32 is set); weight and dweight are [H,V] or [V,H] as
 *     params->weight_layout says.
 *     labels: int64.  Everything else: fp32.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  All work is
 *     enqueued asynchronously on it; nothing synchronises unless params->validate
 *     is set.  The backward passes run their dweight GEMM beside dhidden on an
 *     internal stream (one per host thread and device, created on first use and
 *     destroyed when the thread exits) that
 *     is forked from `stream` by an event and joined back before the call returns,
 *     so every call's work still follows the work enqueued on `stream` before it and
 *     precedes the work enqueued after it.
 *   - Return value: FLCE_OK or one of the FLCE_ERR_* codes below.  Argument errors
 *     are detected on the host before anything is enqueued.  Device-side
 *     conditions (a label outside [0,V) that is not ignore_index, a pipeline wait
 *     that timed out) are recorded in an error word inside the workspace; they
 *     are returned by flce_status(), or directly when params->validate != 0.
 *   - Requirements: N >= 0, H >= 8, V >= 1, H % 8 == 0, and V % 8 == 0 for a [H,V]
 *     weight (16-byte row strides for the TMA engine; a [V,H] weight takes any V).
 *     Row lengths that are multiples of 64 elements (whole 128-byte lines) run
 *     faster: ~11 % in the forward GEMM otherwise.  Every tensor pointer 16-byte aligned (g_loss,
 *     g_entropy and class_weight: 4-byte; an fp32 dhidden: 32-byte), every workspace
 *     256-byte aligned.
 */
#ifndef FLCE_H_
#define FLCE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Storage of weight (and of dweight, which always matches it).  WEIGHT_HV is the
 * [H,V] matrix of the pages' logits = hidden @ weight (verl PR #462, "API");
 * WEIGHT_VH is the transposed [V,H] layout of a torch nn.Linear LM head (the
 * layout Liger-Kernel issue #127 works with), logits = hidden @ weight^T. */
typedef enum {
  FLCE_WEIGHT_HV = 0,
  FLCE_WEIGHT_VH = 1
} flce_weight_layout;

typedef enum {
  FLCE_RED_NONE = 0,
  FLCE_RED_MEAN = 1,
  FLCE_RED_SUM = 2
} flce_reduction;

enum {
  FLCE_OK = 0,
  FLCE_ERR_BAD_ARG = 1,       /* NULL pointer, bad reduction, negative coefficient */
  FLCE_ERR_BAD_SHAPE = 2,     /* N, H or V out of the supported range */
  FLCE_ERR_ALIGN = 3,         /* H (or a [H,V] weight's V) not a multiple of 8, or a pointer
                               * not 16-byte aligned */
  FLCE_ERR_WS_TOO_SMALL = 4,  /* ws_bytes < flce_workspace_size(...) */
  FLCE_ERR_LABEL = 5,         /* a label outside [0, V) that is not ignore_index */
  FLCE_ERR_TIMEOUT = 6,       /* a device pipeline wait exceeded its time limit */
  FLCE_ERR_CUDA = 7,          /* a CUDA runtime/driver call failed */
  FLCE_ERR_DEVICE = 8,        /* current device is not an sm_103 GPU */
  FLCE_ERR_SCRATCH_LIMIT = 9, /* problem needs more than FLCE_NOALLOC_SCRATCH_BYTES */
  FLCE_ERR_BOUNDS = 10        /* libflce_debug.so only: an in-kernel bounds check failed
                               * (the access was skipped; results are not valid) */
};

typedef struct {
  int64_t N;             /* tokens (rows of hidden) */
  int64_t H;             /* hidden size */
  int64_t V;             /* vocabulary size */
  int64_t ignore_index;  /* label value that marks an ignored row (usually -100) */
  int32_t reduction;     /* flce_reduction */
  float zloss_coef;      /* z-loss coefficient, 0 = off */
  float softcap;         /* tanh logit soft-cap c, 0 = off */
  int32_t validate;      /* != 0: synchronise at the end and report device errors */
  int64_t chunk_v;       /* backward vocabulary chunk width (multiple of 256), 0 = auto:
                          * the widest whose bf16 dlogits [N, chunk_v] fit 2 GiB */
  int32_t weight_layout; /* flce_weight_layout: how weight and dweight are stored */
  float label_smoothing; /* eps in [0, 1], 0 = off */
  const float* class_weight; /* [V] fp32 device pointer, per-class target weights; NULL = all 1 */
  /* Vocabulary sharding (see flce_shard_stats).  v_total = 0: weight holds the whole
   * vocabulary.  v_total > 0: weight holds columns [v_offset, v_offset + V) of a
   * vocabulary of v_total entries, and labels are indices into the whole vocabulary.
   * Sharding excludes label_smoothing and class_weight. */
  int64_t v_offset;
  int64_t v_total;
  /* flce_forward_backward's token chunk (a multiple of 512), 0 = auto: the largest
   * chunk whose fp32 logits and bf16 dlogits fit in 8 GiB. */
  int64_t chunk_n;
  /* 0: dhidden is bf16 [N,H].  1: dhidden is fp32 [N,H] (32-byte aligned), the
   * unrounded fp32 accumulation -- for a vocabulary shard's dhidden term, so that the
   * sum over the shards is rounded once, after the exchange, not once per shard. */
  int32_t dhidden_fp32;
} flce_params;

/* FLCE_OK, or the status every entry point returns for these parameters (checked
 * on the host before any pointer is looked at): FLCE_ERR_BAD_ARG, FLCE_ERR_BAD_SHAPE
 * or FLCE_ERR_ALIGN. */
int flce_check_params(const flce_params* params);

/* Bytes of device workspace that flce_forward / flce_shard_stats (phase 0),
 * flce_backward (phase 1), flce_combine_shards (phase 2) or flce_forward_backward
 * (phase 3) needs for these parameters; 0 when the parameters are invalid.  The workspace is scratch: its
 * contents need not be preserved between calls. */
size_t flce_workspace_size(const flce_params* params, int phase);

/* Forward pass.
 *   hidden  [N,H] bf16, weight [H,V] (or [V,H]) bf16, labels [N] int64.
 *   loss, entropy: [N] fp32 for FLCE_RED_NONE, [1] fp32 otherwise (overwritten).
 *   lse, ez: [N] fp32, per-row logsumexp and softmax mean E_p[z] of the capped
 *     logits, written for every row (ignored ones too); flce_backward needs them.
 *   workspace: >= flce_workspace_size(params, 0) bytes, 256-byte aligned. */
int flce_forward(const flce_params* params, const void* hidden, const void* weight,
                 const int64_t* labels, float* loss, float* entropy, float* lse, float* ez,
                 void* workspace, size_t ws_bytes, void* stream);

/* Backward pass (logits are recomputed tile by tile; no [N,V] array exists).
 *   hidden, weight, labels: as given to flce_forward.
 *   lse, ez: the [N] outputs of flce_forward for the same inputs and params.
 *   g_loss, g_entropy: upstream gradients of loss and entropy, [N] for
 *     FLCE_RED_NONE, [1] otherwise; NULL means zero.
 *   dhidden [N,H] bf16 (fp32 with params->dhidden_fp32), dweight [H,V] (or [V,H], as
 *   weight) bf16: overwritten.
 *   workspace: >= flce_workspace_size(params, 1) bytes, 256-byte aligned. */
int flce_backward(const flce_params* params, const void* hidden, const void* weight,
                  const int64_t* labels, const float* lse, const float* ez,
                  const float* g_loss, const float* g_entropy, void* dhidden, void* dweight,
                  void* workspace, size_t ws_bytes, void* stream);

/* Forward and backward in one call, for callers that know the upstream gradients
 * when they run the forward (Liger-Kernel PR #551, "gradient in forward"; in a
 * training step the loss's gradient is 1, scaled by the reduction).  Per chunk of
 * params->chunk_n tokens the logits are computed once, kept in the workspace in
 * fp32 next to their online-softmax statistics, turned into dlogits once the
 * rows' logsumexp is known, and contracted into dhidden and dweight: 6*N*H*V
 * flops instead of flce_forward + flce_backward's 8*N*H*V (no recompute), at the
 * cost of an [chunk_n, V] fp32 + bf16 workspace.
 *   Arguments: as flce_forward's and flce_backward's (g_loss, g_entropy: [N] for
 *   FLCE_RED_NONE, [1] otherwise, NULL = zero).  loss, entropy, lse, ez,
 *   dhidden and dweight are all written, with the values the two-call path
 *   gives (the dlogits are bitwise the same).  Vocabulary sharding
 *   (v_total > 0 with a partial shard) is rejected with FLCE_ERR_BAD_ARG.
 *   workspace: >= flce_workspace_size(params, 3) bytes, 256-byte aligned. */
int flce_forward_backward(const flce_params* params, const void* hidden, const void* weight,
                          const int64_t* labels, const float* g_loss, const float* g_entropy,
                          float* loss, float* entropy, float* lse, float* ez, void* dhidden,
                          void* dweight, void* workspace, size_t ws_bytes, void* stream);

/* x[i] = bf16(g[0] * x[i]) for the n bf16 values at x (16-byte aligned), on
 * `stream`, with a zero product stored as +0 (so rows of zeros stay bitwise zero
 * under a negative g[0]); the kernel returns at once when g[0] == 1.  It scales
 * flce_forward_backward's dhidden and dweight when the upstream gradient of the
 * loss becomes known only after the forward (autograd's backward).  Not part of
 * the pages' method: a helper of the gradient-in-forward mode. */
int flce_scale_bf16(void* x, int64_t n, const float* g, void* stream);

/* Vocabulary-parallel forward, step 1 (the softmax statistics are split over
 * shards of the vocabulary and merged with the online-softmax max-rescale).
 *   params: V, v_offset, v_total describe this shard; weight is its slice, stored
 *   as params->weight_layout says ([H,V] or [V,H] with V the shard width).
 *   stats: [4, N] fp32, overwritten: per row, over the shard's columns, the maximum
 *   m of log2e * z, d = sum 2^(log2e z - m), s = sum 2^(log2e z - m) (log2e z - m),
 *   and the label's logit z_y if the label falls in the shard (else 0).
 *   workspace: >= flce_workspace_size(params, 0) bytes. */
int flce_shard_stats(const flce_params* params, const void* hidden, const void* weight,
                     const int64_t* labels, float* stats, void* workspace, size_t ws_bytes,
                     void* stream);

/* Vocabulary-parallel forward, step 2: merge the stats of all shards.
 *   stats: [n_shards, 4, N] fp32, each shard's flce_shard_stats output (as an
 *   all-gather across ranks produces it).  Outputs as flce_forward's, for the whole
 *   vocabulary (params->v_total entries).  workspace: >= flce_workspace_size(params, 2).
 *   Of params only N, ignore_index, reduction, zloss_coef, validate and v_total are
 *   used; the shard fields (V, v_offset, weight_layout) need only be a valid shard of
 *   v_total, e.g. the whole vocabulary as one [V,H] shard, which takes any v_total. 
 * The backward of a shard is flce_backward with the same sharded params and weight
 * slice: it writes that shard's dweight and this shard's term of dhidden, which the
 * caller sums over the shards. */
int flce_combine_shards(const flce_params* params, const float* stats, int32_t n_shards,
                        const int64_t* labels, float* loss, float* entropy, float* lse,
                        float* ez, void* workspace, size_t ws_bytes, void* stream);

/* Synchronises `stream` and returns the device-side status recorded in the
 * workspace header by the last call that used this workspace (FLCE_OK,
 * FLCE_ERR_LABEL, FLCE_ERR_TIMEOUT or, with libflce_debug.so, FLCE_ERR_BOUNDS), or
 * FLCE_ERR_CUDA. */
int flce_status(const void* workspace, void* stream);

/* Number of kernels one call with these parameters enqueues (memsets not counted):
 * phase 0 flce_forward, 1 flce_backward, 2 flce_combine_shards, 3 flce_shard_stats,
 * 4 flce_forward_backward; -1 when invalid. */
int flce_kernel_launches(const flce_params* params, int phase);

/* Self-test of the device-side failure detection (no counterpart on the pages): one
 * kernel thread waits, with the bounded wait every pipeline kernel uses, on an
 * mbarrier that nothing arrives on, gives up after limit_ns of global time
 * (0 < limit_ns <= 2 s) and records the timeout in the workspace header, then returns.
 * Afterwards flce_status(workspace, stream) reports FLCE_ERR_TIMEOUT and the CUDA
 * context stays usable.  workspace: >= 256 bytes, 256-byte aligned.  Returns
 * FLCE_OK once the kernel is enqueued (the timeout is the expected outcome). */
int flce_selftest_wait_timeout(void* workspace, size_t ws_bytes, uint64_t limit_ns, void* stream);

/* Diagnostic (no counterpart on the pages): the schedule the library plans for one of
 * its GEMMs, from the GEMM's shape in tiles and the GPU's capacity; host arithmetic
 * only, usable without a GPU.
 *   m_tiles, n_tiles: output tiles (256 rows x 256 columns); raster: 0 = the M tiles
 *   vary fastest in the persistent schedule, 1 = the N tiles; panel_bytes: bytes of the
 *   operand every tile of a raster group revisits, per tile of the fast dimension;
 *   a_hint, b_hint: the L2 policy wanted for the A / B loads (0 normal, 1 evict-first,
 *   2 evict-last); pairs: CTA pairs the GPU holds at once (76 on a 152-SM GB300).
 *   out[3] receives: tiles of the fast dimension per raster group, and the L2
 *   policies of the A and B loads.
 * Returns FLCE_OK, or FLCE_ERR_BAD_ARG for a NULL out or an out-of-range argument. */
int flce_plan_tiles(int32_t m_tiles, int32_t n_tiles, int32_t raster, int64_t panel_bytes,
                    int32_t a_hint, int32_t b_hint, int32_t pairs, int32_t* out);

/* Static, NUL-terminated description of a status code. */
const char* flce_strerror(int code);

/* Forward pass for callers that cannot allocate device memory.  (The pages have
 * no counterpart: this entry point serves callers that can't call cudaMalloc, e.g.
 * code whose device memory a framework or serving runtime hands out up front and
 * keeps, or code under an allocator it does not own, which therefore cannot
 * provide the workspace flce_forward needs.)
 *   Same arguments and results as flce_forward, minus the workspace, and the same
 *   kernels in the same order, so the results are bitwise flce_forward's.  The
 *   scratch it uses is a static device array of FLCE_NOALLOC_SCRATCH_BYTES (64 MiB)
 *   held by every GPU that loads the library until the process exits; problems
 *   whose flce_workspace_size(params, 0) exceeds it return FLCE_ERR_SCRATCH_LIMIT
 *   without enqueueing anything.  Nothing is allocated (no cudaMalloc/cudaFree).
 *   The first call on a device looks up the array's device address (once, with
 *   that device current, through the runtime's symbol lookup).  All calls
 *   share the array (its header is cleared on every call; the rest is fully
 *   rewritten), so calls that may overlap on the GPU -- other streams, other
 *   threads -- race and must be serialised by the caller.  flce_status() is not
 *   available for it; set params->validate to get device-side errors returned
 *   (the call then waits for `stream` and copies the error word to the host
 *   before it returns). */
#define FLCE_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int flce_forward_noalloc(const flce_params* params, const void* hidden, const void* weight,
                         const int64_t* labels, float* loss, float* entropy, float* lse,
                         float* ez, void* stream);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int flce_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FLCE_H_ */
