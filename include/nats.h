/*
 * nats.h - C ABI of libnats, the NAtS-L token-level hybrid attention layer
 * for NVIDIA GB300 (sm_103a): the forward (prefill), the same layer with its
 * projections from x, a decode step on a caller-owned state, and the
 * backward pass at the forward's selection.
 *
 * The operation ("Neural Attention Search Linear (NAtS-L)", technical
 * summary, section "Kernmechanismen"):
 *   item 1  The sequence is cut into 64-token chunks.  An Attention Score
 *           Layer (mean pooling, then a linear layer) gives each chunk one
 *           score per operation; the highest score picks softmax attention
 *           (0) or Gated DeltaNet (1) for that chunk.
 *   item 3  Both branches run over every chunk.  The softmax branch of a
 *           token attends to the tokens of earlier softmax-selected chunks
 *           plus its own chunk causally.  The Gated DeltaNet state
 *           S_t = a_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *           (a_t = exp(g_t), read out as o_t = S_t (scale q_t)) is
 *           pseudo-updated through every chunk and rolled back to the chunk
 *           start when the chunk chose softmax.
 *   item 4  Each branch output is RMS-normalised on its own; the output is
 *           w N_soft + (1 - w) N_lin with w = sigmoid(q . W_g[h] + b_g[h]).
 *
 * Conventions common to every entry point:
 *   - Layout: Q, K [B, H, L, dk], V and the output [B, H, L, dv], all
 *     contiguous, row-major, element type `dtype` (bf16 or fp32).  g and
 *     beta are fp32 [B, H, L].  Selection codes are uint8 [B, H, N] with
 *     N = L / 64.
 *   - Every data pointer is a DEVICE pointer owned by the caller; `dims` is
 *     a host pointer.  The library keeps no data between calls and never
 *     synchronises the host: all work is enqueued on `stream` (0 = the
 *     legacy default stream).  It allocates no device memory per call; what
 *     it does hold is listed here.  Per device, created on first use and
 *     kept until the process exits: one side stream and two events (the
 *     layer forward runs its two branches concurrently on that stream, and
 *     the bf16 backward its Gated DeltaNet state work beside the softmax
 *     branch, forked from and joined back into `stream`;
 *     nats_hybrid_fwd_streams and nats_hybrid_bwd_streams take caller-owned
 *     ones instead, or run everything on `stream`).
 *     Per loaded library, on every GPU: the fixed scratch array of
 *     nats_hybrid_fwd_noalloc.
 *   - Arguments are validated on the host before anything is launched; a
 *     violation returns its status and leaves every output untouched.
 *   - Launch failures return NATS_ERR_CUDA (from cudaGetLastError).  Errors
 *     that happen while the kernels run surface, as usual for CUDA, on the
 *     caller's next synchronising call.
 *   - No C++ exception crosses this interface.  Calls from several host
 *     threads are safe: the per-device side stream and events are used
 *     under a lock.  Because all forward and backward calls of a device
 *     share the one side stream, the side halves of concurrent calls made
 *     on different caller streams run one after the other on it (correct,
 *     but not concurrent).  Calls that share a workspace must be
 *     ordered by the caller.
 *   - Supported shapes: chunk = 64, L % 64 == 0, dk == dv in {64, 128},
 *     B, H, L >= 0 (any zero extent makes the call a no-op that returns
 *     NATS_OK), and B H L dk / 64 < 2^31 (tile coordinates are 32-bit;
 *     else NATS_ERR_UNSUPPORTED).  Q, K, V, the output and the workspace
 *     must be 16-byte aligned.
 */
#ifndef NATS_H_
#define NATS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st* nats_stream_t;

typedef enum {
  NATS_OK = 0,
  NATS_ERR_NULL = 1,        /* a required pointer is NULL */
  NATS_ERR_SHAPE = 2,       /* negative extent, L % chunk != 0, chunk != 64, dk != dv */
  NATS_ERR_DTYPE = 3,       /* dtype is not NATS_BF16 / NATS_F32 */
  NATS_ERR_ALIGN = 4,       /* a pointer is not 16-byte aligned */
  NATS_ERR_WORKSPACE = 5,   /* workspace smaller than nats_workspace_size() */
  NATS_ERR_UNSUPPORTED = 6, /* head size other than 64 / 128, or a size beyond int32 tiling */
  NATS_ERR_CUDA = 7,        /* a CUDA runtime call or kernel launch failed */
  NATS_ERR_INTERNAL = 8,
  NATS_ERR_VALUE = 9        /* scale or eps negative or not finite */
} nats_status;

typedef enum { NATS_BF16 = 0, NATS_F32 = 1 } nats_dtype;

typedef struct {
  int32_t B, H, L; /* batch, heads, tokens per sequence */
  int32_t dk, dv;  /* key / value head size (equal) */
  int32_t chunk;   /* must be 64 */
  int32_t dtype;   /* nats_dtype of Q, K, V and the output */
  float scale;     /* softmax logit and linear readout scale; 0 => 1/sqrt(dk) */
  float eps;       /* RMSNorm epsilon (1e-6 in the reference workloads) */
} nats_dims;

/* Human-readable name of a status code (static storage). */
const char* nats_status_string(nats_status s);

/* The CUDA runtime's description of the last CUDA error a libnats call on
 * this host thread met (the cause behind its NATS_ERR_CUDA), or "no error".
 * Static storage; only the calling thread's own calls update it. */
const char* nats_last_cuda_error(void);

/* Bytes of device workspace nats_hybrid_fwd needs for `dims` (0 for an
 * invalid `dims`).  The workspace holds the selection, the compacted
 * softmax-chunk lists, the per-chunk Gated DeltaNet factors and both branch
 * outputs; its contents are scratch between calls. */
size_t nats_workspace_size(const nats_dims* dims);

/* Synchronises `stream`, then reports whether a kernel of the last
 * nats_hybrid_fwd call that used `workspace` gave up on a bounded internal
 * wait (NATS_ERR_INTERNAL; its outputs are then invalid) or NATS_OK.  The
 * tensor-core kernels bound every spin-wait (about 2 s) instead of hanging. */
nats_status nats_workspace_check(const nats_dims* dims, const void* workspace, nats_stream_t stream);

/* Attention Score Layer + argmax alone ("Kernmechanismen" item 1).
 *   q, k    [B, H, L, dk] dtype
 *   w_s     fp32 [H, 2, 2*dk]: row 0 scores softmax, row 1 Gated DeltaNet,
 *           applied to the chunk mean of [q_t ; k_t] (unscaled q)
 *   b_s     fp32 [H, 2] or NULL (zero bias)
 *   sel     uint8 [B, H, N] out: 0 = softmax, 1 = Gated DeltaNet; ties -> 0
 *   scores  fp32 [B, H, N, 2] out, or NULL */
nats_status nats_select(const nats_dims* dims, const void* q, const void* k, const float* w_s,
                        const float* b_s, uint8_t* sel, float* scores, nats_stream_t stream);

/* The whole layer forward ("Kernmechanismen" items 1, 3, 4).
 *   q, k, v      dtype [B, H, L, d]
 *   g, beta      fp32 [B, H, L]: log-decay (a_t = exp(g_t)) and write strength
 *   w_s, b_s     score layer as in nats_select (w_s may be NULL when sel_in is given)
 *   w_g          fp32 [H, dk] merge-gate projection; b_g fp32 [H] or NULL
 *   norm_w_soft, norm_w_lin   fp32 [dv] RMSNorm weights, or NULL (unit)
 *   sel_in       uint8 [B, H, N] or NULL: when given, replaces the score
 *                layer's choice (values must be 0 or 1)
 *   out          dtype [B, H, L, dv] out
 *   sel_out      uint8 [B, H, N] out, or NULL
 *   state_out    fp32 [B, H, dv, dk] out, or NULL: the Gated DeltaNet state
 *                after the last chunk (after its commit or rollback)
 *   o_soft_out, o_lin_out   fp32 [B, H, L, dv] out, or NULL: the branch
 *                outputs before normalisation (diagnostics)
 *   workspace    device scratch of at least nats_workspace_size(dims) bytes */
nats_status nats_hybrid_fwd(const nats_dims* dims, const void* q, const void* k, const void* v,
                            const float* g, const float* beta, const float* w_s, const float* b_s,
                            const float* w_g, const float* b_g, const float* norm_w_soft,
                            const float* norm_w_lin, const uint8_t* sel_in, void* out,
                            uint8_t* sel_out, float* state_out, float* o_soft_out,
                            float* o_lin_out, void* workspace, size_t workspace_bytes,
                            nats_stream_t stream);

/* nats_hybrid_fwd for callers that cannot allocate device memory (the
 * pages describe no such variant; it exists for deployment).  Some callers
 * have no way to hand over a workspace: a plugin whose host application owns
 * all device memory through its own pool (a direct cudaMalloc would bypass
 * the pool and may synchronise the device), a latency-critical loop that must
 * never block on an allocation, or a plain C caller without an allocator.
 * This entry point takes the same inputs and outputs as nats_hybrid_fwd but
 * no workspace, and allocates nothing: its scratch is a 64 MiB device array
 * built into the library, held on every GPU that loads the library until
 * the process exits.
 *   - Problems whose nats_workspace_size() exceeds 64 MiB (67108864 bytes)
 *     are rejected with NATS_ERR_WORKSPACE before any launch.
 *   - The first call on a device looks up the array's device address on the
 *     current device (cudaGetSymbolAddress); make that first call before any
 *     stream capture.
 *   - All calls on a device share the one array, which keeps the last call's
 *     contents; calls that can overlap on the GPU (different streams without
 *     ordering, or several host threads) race on it and must be serialised
 *     by the caller.  Nothing in it needs to start zeroed.
 *   - The device address found by the first call on a device is kept for
 *     later calls.  cudaDeviceReset unloads the array with the rest of the
 *     library's device code, so that address is stale after a reset: do not
 *     use this entry point on a device the process has reset since its first
 *     call there.
 *   - A bounded internal wait that expired (outputs invalid) is reported by
 *     nats_noalloc_check, the counterpart of nats_workspace_check for the
 *     built-in scratch.
 * Other arguments, results and errors are those of nats_hybrid_fwd, checked
 * in the same order; the size limit is checked after them. */
nats_status nats_hybrid_fwd_noalloc(const nats_dims* dims, const void* q, const void* k,
                                    const void* v, const float* g, const float* beta,
                                    const float* w_s, const float* b_s, const float* w_g,
                                    const float* b_g, const float* norm_w_soft,
                                    const float* norm_w_lin, const uint8_t* sel_in, void* out,
                                    uint8_t* sel_out, float* state_out, float* o_soft_out,
                                    float* o_lin_out, nats_stream_t stream);

/* nats_workspace_check for nats_hybrid_fwd_noalloc: synchronises `stream`,
 * then reports NATS_ERR_INTERNAL if a kernel of the last allocation-free call
 * on the current device (with these dims) gave up on a bounded internal wait,
 * else NATS_OK.  NATS_ERR_WORKSPACE for dims beyond the built-in scratch. */
nats_status nats_noalloc_check(const nats_dims* dims, nats_stream_t stream);

/* Stages of nats_hybrid_fwd, for per-stage timing. */
typedef enum {
  NATS_STAGE_SCORE = 0,    /* Attention Score Layer + argmax (skipped with sel_in) */
  NATS_STAGE_COMPACT = 1,  /* prefix counts / compacted softmax-chunk lists */
  NATS_STAGE_SOFTMAX = 2,  /* softmax branch */
  NATS_STAGE_GDN_PREP = 3, /* Gated DeltaNet per-chunk factors (parallel over chunks) */
  NATS_STAGE_GDN_SCAN = 4, /* Gated DeltaNet chunk scan with commit / rollback */
  NATS_STAGE_MERGE = 5,    /* RMSNorm per branch + gated merge */
  NATS_STAGE_PROJ_IN = 6,  /* nats_hybrid_fwd_x: x -> q, k, v, g, beta */
  NATS_STAGE_PROJ_OUT = 7, /* nats_hybrid_fwd_x: output projection */
  NATS_NUM_STAGES = 8
} nats_stage;

/* Caller-owned timing hooks.  start[s] / stop[s] are cudaEvent_t handles
 * (or NULL); the library records them right before the first and right
 * after the last kernel of stage s, on the stream that stage runs on (the
 * softmax stage runs on a second stream, concurrently with the Gated
 * DeltaNet scan, and is joined back before the call's last kernel).
 * `launches` is set to the number of kernels the call launched and
 * stage_launches[s] to the number stage s launched (0: the stage did not
 * run and its events were not recorded). */
typedef struct {
  void* start[NATS_NUM_STAGES];
  void* stop[NATS_NUM_STAGES];
  int32_t launches;
  int32_t stage_launches[NATS_NUM_STAGES];
} nats_profile;

/* nats_hybrid_fwd plus per-stage event records (prof may be NULL, which
 * makes it identical to nats_hybrid_fwd).  Same arguments, errors and
 * results; recording an event that fails returns NATS_ERR_CUDA. */
nats_status nats_hybrid_fwd_profiled(const nats_dims* dims, const void* q, const void* k,
                                     const void* v, const float* g, const float* beta,
                                     const float* w_s, const float* b_s, const float* w_g,
                                     const float* b_g, const float* norm_w_soft,
                                     const float* norm_w_lin, const uint8_t* sel_in, void* out,
                                     uint8_t* sel_out, float* state_out, float* o_soft_out,
                                     float* o_lin_out, void* workspace, size_t workspace_bytes,
                                     nats_stream_t stream, nats_profile* prof);

/* Caller-owned concurrency for the layer forward.  With bf16 inputs the
 * forward runs its Gated DeltaNet scan on `stream` and the softmax branch on
 * a second stream, forked from `stream` before the branches and joined back
 * before the merge.  nats_hybrid_fwd and nats_hybrid_fwd_profiled take that
 * second stream and the fork / join events from the library's per-device
 * set; here the caller supplies them, and the call uses no library-held
 * stream or event (and takes no lock):
 *   side  the second stream (a cudaStream_t of the current device), or
 *         NULL, or `stream` itself: then both branches run in order on
 *         `stream` and fork / join are not used (may be NULL);
 *   fork  a cudaEvent_t the call records on `stream` and makes `side` wait
 *         for; join a cudaEvent_t it records on `side` and makes `stream`
 *         wait for.  Any creation flags; the caller keeps them alive until
 *         the call has been enqueued (they may be reused right after).
 * Concurrent calls that share `side` or the events must be ordered by the
 * caller. */
typedef struct {
  nats_stream_t side;
  void* fork;
  void* join;
} nats_streams;

/* nats_hybrid_fwd_profiled with caller-owned concurrency (streams may be
 * NULL, which makes it identical to nats_hybrid_fwd_profiled) and one more
 * saved activation for training: lse_out (or NULL), fp32 [B, H, L], each
 * token's log2 of the sum of 2^(s scale log2 e) over the keys its softmax
 * branch sees (s the scores q . k), written for bf16 layers (NATS_ERR_DTYPE
 * for fp32 ones); nats_hybrid_bwd_streams takes it to skip recomputing it.
 * Same arguments, errors and results otherwise; NATS_ERR_NULL when
 * streams->side is a stream other than `stream` and fork or join is NULL;
 * NATS_ERR_CUDA when recording or waiting on them fails. */
nats_status nats_hybrid_fwd_streams(const nats_dims* dims, const void* q, const void* k,
                                    const void* v, const float* g, const float* beta,
                                    const float* w_s, const float* b_s, const float* w_g,
                                    const float* b_g, const float* norm_w_soft,
                                    const float* norm_w_lin, const uint8_t* sel_in, void* out,
                                    uint8_t* sel_out, float* state_out, float* o_soft_out,
                                    float* o_lin_out, float* lse_out, void* workspace, size_t workspace_bytes,
                                    nats_stream_t stream, const nats_streams* streams,
                                    nats_profile* prof);

/* ---- The projections around the layer ------------------------------------
 * The layer above takes Q, K, V and the gates; a model layer makes them
 * from its hidden states x and maps the output back ("Neural Attention
 * Search Linear (NAtS-L)", technical summary, "Kernmechanismen" item 4:
 * the merge weights come from Q projections; the projections themselves
 * are not spelled out, so this follows the plain Gated DeltaNet form and
 * the definitions below are the reading).  bf16 only (dims->dtype must be
 * NATS_BF16), d = dims->dk = dims->dv, H = dims->H.  Per token t (row of x):
 *   [q_t | k'_t | v_t] = bf16(x_t W_qkv), head h at columns h d .. h d + d - 1
 *                        of each third;
 *   k_t = bf16(k'_t / |k'_t|) per head (|0| gives k = 0);
 *   [a_t | b_t] = x_t W_ab (fp32, not rounded);
 *   g_t,h    = -a_scale[h] softplus(a_t,h + b_a[h])   (log-decay, <= 0)
 *   beta_t,h = sigmoid(b_t,h + b_b[h]);
 *   o = the layer (nats_hybrid_fwd with w_s, b_s, w_g, b_g), bf16;
 *   y_t = bf16(sum_h o_t,h W_o[h d .. h d + d - 1, :]).
 * The products run on the library's own tcgen05 GEMM (bf16 operands, fp32
 * accumulate): the first one's epilogue writes q, k (normalised), v in the
 * layer's layout and forms g and beta; the second reads the layer output in
 * its [B, H, L, d] layout.
 *   hidden       width of x and y (multiple of 8)
 *   x            [B, L, hidden] bf16
 *   w_qkv        [hidden, 3 H d] bf16, row-major
 *   w_ab         [hidden, 2 H] bf16, row-major (column h: a of head h,
 *                column H + h: b of head h)
 *   b_a, b_b     [H] fp32 or NULL (zero); a_scale [H] fp32 or NULL (one)
 *   w_s .. b_g   as for nats_hybrid_fwd
 *   w_o          [H d, hidden] bf16, row-major
 *   y            [B, L, hidden] bf16 (output)
 *   sel_out      [B, H, N] u8 or NULL: the chunk selection
 *   workspace    device scratch of at least nats_x_workspace_size(dims, hidden)
 * Errors as nats_hybrid_fwd; NATS_ERR_SHAPE if hidden <= 0 or hidden % 8;
 * NATS_ERR_UNSUPPORTED if B L or 3 H d exceed int32 tiling.
 * nats_x_workspace_check synchronises `stream` and reports NATS_ERR_INTERNAL
 * if a kernel of the last call that used `workspace` gave up on a bounded
 * internal wait (its outputs are then invalid), else NATS_OK. */
size_t nats_x_workspace_size(const nats_dims* dims, int32_t hidden);
nats_status nats_hybrid_fwd_x(const nats_dims* dims, int32_t hidden, const void* x, const void* w_qkv,
                              const void* w_ab, const float* b_a, const float* a_scale, const float* b_b,
                              const float* w_s, const float* b_s, const float* w_g, const float* b_g,
                              const void* w_o, void* y, uint8_t* sel_out, void* workspace,
                              size_t workspace_bytes, nats_stream_t stream);
nats_status nats_x_workspace_check(const nats_dims* dims, int32_t hidden, const void* workspace,
                                   nats_stream_t stream);
/* nats_hybrid_fwd_x plus per-stage event records (the layer's stages and
 * NATS_STAGE_PROJ_IN / NATS_STAGE_PROJ_OUT, all on `stream` but the softmax
 * stage); prof may be NULL.  Same arguments, errors and results. */
nats_status nats_hybrid_fwd_x_profiled(const nats_dims* dims, int32_t hidden, const void* x, const void* w_qkv,
                                       const void* w_ab, const float* b_a, const float* a_scale, const float* b_b,
                                       const float* w_s, const float* b_s, const float* w_g, const float* b_g,
                                       const void* w_o, void* y, uint8_t* sel_out, void* workspace,
                                       size_t workspace_bytes, nats_stream_t stream, nats_profile* prof);

/* --------------------------------------------------------------- test hooks
 * Failure injection without a GPU fault.
 * nats_debug_fail_stage: the next layer forward on this host thread
 * (nats_hybrid_fwd, _profiled, _noalloc, _x) replaces the launch of stage
 * `stage` (a NATS_STAGE_* id) by a cudaErrorInvalidValue: it returns
 * NATS_ERR_CUDA there, nats_last_cuda_error() names the error, and the
 * stages before it have been enqueued.  -1 cancels.
 * nats_debug_bounded_wait: one device thread waits for an mbarrier phase
 * that nothing completes, gives up after limit_ns (1 .. 1e9) and sets *flag
 * (device int) to 1 -- the path every tensor-core kernel takes when one of
 * its bounded waits expires.  NATS_ERR_NULL / NATS_ERR_VALUE for bad
 * arguments. */
void nats_debug_fail_stage(int32_t stage);
nats_status nats_debug_bounded_wait(int32_t* flag, int64_t limit_ns, nats_stream_t stream);

/* ------------------------------------------------------------------ decode
 * The same layer in decode mode: one new token per (b, h) per call, at
 * position t of the sequence.  "Neural Attention Search Linear (NAtS-L)",
 * technical summary, "Kernmechanismen" items 1, 3 and 4 read token by token
 * (the decode reading DEC-1): the token joins its chunk's keys
 * and values and attends to the retained ones (those of earlier softmax
 * chunks) plus its chunk up to itself; the Gated DeltaNet state takes the
 * token's update at once (the pseudo-update) and the readout uses it; when
 * the token completes its chunk (t % chunk == chunk - 1) the chunk's score
 * (mean of [q; k] over the chunk through W_s, b_s; ties to softmax) decides:
 * softmax appends the chunk's keys and values to the retained ones and puts
 * the state back to the chunk start; Gated DeltaNet keeps the state (the new
 * chunk start) and drops them.  Stepped from the empty state over a
 * sequence, it gives the outputs nats_hybrid_fwd gives for that sequence.
 *
 * The state is the caller's device memory, updated in place by each call;
 * all zeros (S, S0, psum, n_kv, err) is the empty state (ck, cv need no
 * initialisation).  Layouts are contiguous, element type fp32 where marked,
 * else dims->dtype. */
typedef struct {
  float* S;       /* [B, H, dv, dk] fp32 state after the last token */
  float* S0;      /* [B, H, dv, dk] fp32 state at the start of the current chunk */
  void* ck;       /* [B, H, chunk, dk] keys of the current chunk */
  void* cv;       /* [B, H, chunk, dv] values of the current chunk */
  float* psum;    /* [B, H, 2 dk] fp32 sum of [q; k] over the current chunk */
  void* kv_k;     /* [B, H, cap, dk] keys of the retained chunks, in order */
  void* kv_v;     /* [B, H, cap, dv] values of the retained chunks */
  int32_t* n_kv;  /* [B, H] retained tokens per head (a multiple of chunk) */
  int64_t cap;    /* tokens per head kv_k / kv_v hold */
  int32_t* err;   /* [1] set to 1 by a step whose bounded wait for its key /
                     value copies ran out (that step's outputs and state are
                     then not valid); never cleared by the library */
} nats_decode_state;

/* One decode step.  dims: B, H, dk = dv (64 or 128), chunk (64), dtype,
 * scale, eps as for nats_hybrid_fwd; dims->L is not used.  t >= 0 is the
 * position of this token.  q, k [B, H, dk], v [B, H, dv] (dtype); g, beta
 * [B, H] fp32 (log-decay and delta-rule strength of this token); w_s, b_s,
 * w_g, b_g, norm weights as for nats_hybrid_fwd (b_s, b_g, norm weights may
 * be NULL).  out [B, H, dv] (dtype) = w RMSNorm(o_s) + (1 - w) RMSNorm(o_l).
 * sel_out [B, H] (or NULL) receives the selection of the completed chunk and
 * is written only when t % chunk == chunk - 1.  o_soft_out / o_lin_out [B, H,
 * dv] fp32 (or NULL) receive the two branch outputs.  All pointers device,
 * 16-byte aligned; asynchronous on `stream`.
 * Errors before any launch: NATS_ERR_NULL (a required pointer), NATS_ERR_SHAPE
 * / NATS_ERR_UNSUPPORTED / NATS_ERR_DTYPE / NATS_ERR_VALUE (dims, t < 0),
 * NATS_ERR_ALIGN, NATS_ERR_WORKSPACE when cap < chunk * (t / chunk + 1) (the
 * retained tokens could outgrow kv_k / kv_v); NATS_ERR_CUDA on a failed
 * launch. */
nats_status nats_decode_step(const nats_dims* dims, int64_t t, const void* q, const void* k, const void* v,
                             const float* g, const float* beta, const float* w_s, const float* b_s,
                             const float* w_g, const float* b_g, const float* norm_w_soft,
                             const float* norm_w_lin, const nats_decode_state* state, void* out,
                             uint8_t* sel_out, float* o_soft_out, float* o_lin_out, nats_stream_t stream);

/* ---------------------------------------------------------------- backward
 * The layer's backward pass at a fixed selection: the gradient of
 * <dout, out> with respect to its continuous inputs ("Neural Attention
 * Search Linear (NAtS-L)", technical summary, "Kernmechanismen" items 3 and
 * 4).  Item 5 says the choice of attention type is learned end to end, but
 * the pages give no estimator for the argmax; W_s and b_s get no gradient
 * here (nats_score_bwd adds an opt-in surrogate).  The forward's selection and its two branch outputs are the saved
 * activations: call nats_hybrid_fwd with sel_out, o_soft_out and o_lin_out.
 *
 * dims as for nats_hybrid_fwd.  q, k, v, dout [B, H, L, d] (dtype); g, beta
 * [B, H, L] fp32; w_g [H, d]; b_g [H] (or NULL: zero); norm weights [d] (or
 * NULL: unit); sel [B, H, L / chunk] uint8 (0 softmax, 1 Gated DeltaNet);
 * o_soft, o_lin [B, H, L, d] fp32, the branch outputs before RMSNorm.
 * Outputs, all fp32 and overwritten: dq, dk, dv [B, H, L, d]; dg, dbeta
 * [B, H, L]; dw_g [H, d], db_g [H], dnorm_w_soft, dnorm_w_lin [d] (each may
 * be NULL: not computed).  The workspace (nats_bwd_workspace_size bytes)
 * holds the per-token branch gradients, the row log-sum-exp of the softmax
 * branch, the Gated DeltaNet chunk-start states and the states of one chunk
 * per head (fp32).  All pointers device; q, k, v, o_soft, o_lin, dout, dq,
 * dk, dv and the workspace 16-byte aligned; asynchronous on `stream`.  With
 * bf16 inputs the Gated DeltaNet chunk-start states' recompute and the
 * adjoint's chunk factors and reverse scan (which write only the workspace)
 * run on the library's per-device side stream, forked from `stream` at the
 * call's start (the reverse scan waits for the merge stage, whose output it
 * reads) and joined back before the first kernel that writes dq, dk or dv
 * after the softmax branch.
 * Errors before any launch: NATS_ERR_NULL, NATS_ERR_SHAPE /
 * NATS_ERR_UNSUPPORTED / NATS_ERR_DTYPE / NATS_ERR_VALUE (dims),
 * NATS_ERR_ALIGN, NATS_ERR_WORKSPACE; NATS_ERR_CUDA on a failed launch. */
size_t nats_bwd_workspace_size(const nats_dims* dims);
nats_status nats_hybrid_bwd(const nats_dims* dims, const void* q, const void* k, const void* v, const float* g,
                            const float* beta, const float* w_g, const float* b_g, const float* norm_w_soft,
                            const float* norm_w_lin, const uint8_t* sel, const float* o_soft,
                            const float* o_lin, const void* dout, float* dq, float* dk, float* dv, float* dg,
                            float* dbeta, float* dw_g, float* db_g, float* dnorm_w_soft, float* dnorm_w_lin,
                            void* workspace, size_t workspace_bytes, nats_stream_t stream);

/* Stages of nats_hybrid_bwd, for per-stage timing (indices into the arrays
 * of nats_profile). */
typedef enum {
  NATS_BWD_STAGE_MERGE = 0,   /* RMSNorm + gated merge backward: branch output gradients, dW_g, db_g, dnorm_w */
  NATS_BWD_STAGE_SOFTMAX = 1, /* softmax branch: dq, then dk / dv (bf16: tcgen05) */
  NATS_BWD_STAGE_GDN = 2,     /* Gated DeltaNet: bf16, the chunk-start states' recompute and the
                                 chunkwise adjoint's factors and reverse scan (on the side stream,
                                 beside the softmax stage); fp32, the token-serial adjoint */
  NATS_BWD_STAGE_COMBINE = 3, /* bf16: every per-chunk product of the adjoint (one kernel: dq, dk,
                                 dv, dg, dbeta); fp32: the per-token sums of the adjoint's state
                                 halves */
  NATS_BWD_NUM_STAGES = 4
} nats_bwd_stage;

/* nats_hybrid_bwd plus per-stage event records, as in
 * nats_hybrid_fwd_profiled but with NATS_BWD_STAGE_* ids (prof may be NULL,
 * which makes it identical to nats_hybrid_bwd). */
nats_status nats_hybrid_bwd_profiled(const nats_dims* dims, const void* q, const void* k, const void* v,
                                     const float* g, const float* beta, const float* w_g, const float* b_g,
                                     const float* norm_w_soft, const float* norm_w_lin, const uint8_t* sel,
                                     const float* o_soft, const float* o_lin, const void* dout, float* dq,
                                     float* dk, float* dv, float* dg, float* dbeta, float* dw_g, float* db_g,
                                     float* dnorm_w_soft, float* dnorm_w_lin, void* workspace,
                                     size_t workspace_bytes, nats_stream_t stream, nats_profile* prof);

/* nats_hybrid_bwd_profiled with caller-owned concurrency, as
 * nats_hybrid_fwd_streams: `streams` (or NULL: the library's per-device set)
 * gives the second stream and the fork / join events of the bf16 backward;
 * side NULL or equal to `stream` runs every kernel in order on `stream`.
 * lse (or NULL; device, 16-byte aligned) is the forward's lse_out for the
 * same inputs and selection: with it, a bf16 backward reads each token's row
 * statistic instead of recomputing it from the scores (fp32 layers ignore
 * it).  Same arguments, errors and results otherwise; NATS_ERR_NULL when
 * streams->side is a stream other than `stream` and fork or join is NULL. */
nats_status nats_hybrid_bwd_streams(const nats_dims* dims, const void* q, const void* k, const void* v,
                                    const float* g, const float* beta, const float* w_g, const float* b_g,
                                    const float* norm_w_soft, const float* norm_w_lin, const uint8_t* sel,
                                    const float* o_soft, const float* o_lin, const float* lse, const void* dout,
                                    float* dq, float* dk, float* dv, float* dg, float* dbeta, float* dw_g,
                                    float* db_g, float* dnorm_w_soft, float* dnorm_w_lin, void* workspace,
                                    size_t workspace_bytes, nats_stream_t stream, const nats_streams* streams,
                                    nats_profile* prof);

/* The score layer's gradient, opt-in ("Kernmechanismen" item 5: the score
 * layer is trained end to end; the pages name no estimator, and
 * nats_hybrid_bwd gives W_s, b_s none).  This call adds a straight-through
 * surrogate (the reading BWD-2): every output row of chunk c is read as
 * scaled by pi_c[sel_c] / (that probability held constant), pi_c the softmax
 * of the chunk's two scores s_c = W_s[h] p_c + b_s[h] (p_c the chunk mean of
 * [q ; k], unscaled q) and sel_c the forward's argmax.  The value does not
 * change; with G_c = sum over the chunk's tokens of <dout_t, out_t> and
 * ds_c = G_c (e_sel - pi_c) it writes
 *   dw_s[h] = sum_{b, c} ds_c p_c^T  [H, 2, 2d] fp32,  db_s[h] = sum ds_c  [H, 2] fp32
 * (overwritten) and ADDS (W_s[h]^T ds_c) / 64 to dq (first d entries) and dk
 * (last d) of each token of the chunk.  Call it after nats_hybrid_bwd on the
 * same dq, dk to get the surrogate's full gradient.
 * q, k, out, dout [B, H, L, d] in the layer dtype (out: the forward's
 * output); w_s [H, 2, 2d], b_s [H, 2] (or NULL: zero) fp32; sel [B, H,
 * L / 64] the forward's selection; dq, dk [B, H, L, d] fp32.  All pointers
 * device, q, k, out, dout, dq, dk 16-byte aligned; asynchronous on
 * `stream`; dw_s, db_s are sums taken with atomics (their rounding order is
 * not fixed).  Errors before any launch: NATS_ERR_NULL, NATS_ERR_SHAPE /
 * NATS_ERR_UNSUPPORTED / NATS_ERR_DTYPE / NATS_ERR_VALUE (dims),
 * NATS_ERR_ALIGN; NATS_ERR_CUDA on a failed launch. */
nats_status nats_score_bwd(const nats_dims* dims, const void* q, const void* k, const float* w_s, const float* b_s,
                           const uint8_t* sel, const void* out, const void* dout, float* dq, float* dk, float* dw_s,
                           float* db_s, nats_stream_t stream);

/* -------------------------------------------------------------------- NHA
 * Native Hybrid Attention, the related layer of "Native Hybrid Attention
 * for Efficient Sequence Modeling" (section "2. Methodologie",
 * "Kernprincipes"): long-term slots updated by a linear RNN and a sliding
 * window of recent tokens form one key / value set under one softmax; the
 * window size w is the layer's only knob (w = 0: a pure linear RNN; w =
 * sequence length: full attention).  The page gives no update rule; the
 * reading (CONV-16) is the Gated Slot Attention slot update:
 *   a token j, when it leaves the window, writes every slot s:
 *     K~[s] <- alpha_j[s] K~[s] + (1 - alpha_j[s]) k_j,   V~[s] likewise with v_j,
 *   K~ = V~ = 0 at the start; the query at t sees the window tokens
 *   t - w < j <= t and, once t >= w, the m slots after the writes of every
 *   j <= t - w:
 *     o_t = softmax(scale q_t . [K~; k_window]) [V~; v_window].
 * dims: B, H, L (L % 64 == 0), d = 128, slots = 64, window w (0, a multiple
 * of 128, or >= L: full attention), dtype NATS_BF16, scale (0 =>
 * 1/sqrt(d)).  q, k, v, out [B, H, L, d] bf16; log_alpha [B, H, L, slots]
 * fp32 (log of the forget gate, <= 0).  The kernels hold the chunkwise form
 * to a product of factors e^{|A|} per half chunk, A a 32-token sum of
 * log_alpha of one slot: keep log_alpha >= -2.5 on average over any 32
 * tokens (alpha >= 0.08), far beyond the damped gates of Gated Slot
 * Attention.  All pointers device, 16-byte aligned; asynchronous on
 * `stream`.  The workspace (nats_nha_workspace_size bytes) holds the
 * chunk-start slot memories and the per-chunk gate factors.  Errors before
 * any launch: NATS_ERR_NULL, NATS_ERR_SHAPE, NATS_ERR_DTYPE,
 * NATS_ERR_UNSUPPORTED (d, slots or w not supported), NATS_ERR_VALUE,
 * NATS_ERR_ALIGN, NATS_ERR_WORKSPACE; NATS_ERR_CUDA on a failed launch.
 * nats_nha_workspace_check synchronises `stream` and reports
 * NATS_ERR_INTERNAL if a bounded internal wait of the last call that used
 * `workspace` expired. */
typedef struct {
  int32_t B, H, L;
  int32_t d;       /* head size (128) */
  int32_t slots;   /* m (64) */
  int32_t window;  /* w */
  int32_t dtype;   /* NATS_BF16 */
  float scale;     /* 0 => 1/sqrt(d) */
} nats_nha_dims;

size_t nats_nha_workspace_size(const nats_nha_dims* dims);
nats_status nats_nha_fwd(const nats_nha_dims* dims, const void* q, const void* k, const void* v,
                         const float* log_alpha, void* out, void* workspace, size_t workspace_bytes,
                         nats_stream_t stream);
nats_status nats_nha_workspace_check(const nats_nha_dims* dims, const void* workspace, nats_stream_t stream);
/* nats_nha_fwd with caller-owned CUDA events recorded around its kernels
 * (prof may be NULL): start[0] / stop[0] around the slot-memory stage (the
 * chunk-parallel gate factors, then the slot-memory scan: two kernels, not
 * launched when w >= L; stage_launches[0] then 0), start[1] / stop[1] around
 * the attention kernel; `launches` counts the kernels launched. */
nats_status nats_nha_fwd_profiled(const nats_nha_dims* dims, const void* q, const void* k, const void* v,
                                  const float* log_alpha, void* out, void* workspace, size_t workspace_bytes,
                                  nats_stream_t stream, nats_profile* prof);

#ifdef __cplusplus
}
#endif

#endif /* NATS_H_ */
