/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention forward library.
 *
 * The operation is the forward chunked prefill of Kimi Delta Attention (KDA),
 * the gated delta rule with a per-channel gate and head dimension K = V = 128:
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 *
 * with the in-kernel preprocessing that the FlashKDA backend enables
 * ("How to Use FlashKDA as a Backend for flash-linear-attention", section
 * "Running Inference with chunk_kda": use_gate_in_kernel, use_qk_l2norm_in_kernel,
 * use_beta_sigmoid_in_kernel, safe_gate, transpose_state_layout):
 *
 *     log alpha_t[c] = lower_bound * sigmoid(exp(A_log[h]) * (g_t[c] + dt_bias[h][c]))
 *     q_t <- q_t / sqrt(|q_t|^2 + 1e-6),  k_t likewise,   beta_t <- sigmoid(beta_t)
 *
 * The elementwise gate form is this library's reading (the pages give only the
 * flags and the bound lower_bound in [-5, 0]); the CPU test oracle uses the same.
 *
 * Call shape follows the FlashKDA binding ("How FlashKDA Integrates with CUTLASS
 * for High-Performance GEMM Operations", sections "Workspace Allocation and Memory
 * Alignment" and "Practical Implementation Example"; "How to Use FlashKDA ...",
 * section "Kernel API and Tensor Requirements"):
 *     fwd(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound,
 *         initial_state=None, final_state=None, cu_seqlens=None) + workspace,
 *     get_workspace_size(B*T, H).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers on the current CUDA device unless a
 *     name ends in _host.  The library never allocates, frees, synchronises or
 *     copies to the host; it only enqueues work on the given stream.
 *   - The caller owns every buffer, including the workspace, and must keep them
 *     alive until the enqueued work has finished.
 *   - Errors are returned as kda_status; nothing aborts and no argument is
 *     converted implicitly (a wrong dtype or layout is the caller's to fix).
 *   - kda_fwd and kda_bwd can be captured into a CUDA graph (stream capture) and replayed,
 *     with new inputs copied into the captured buffers, once one call on the
 *     device has run outside capture (that call sets the kernels' shared-memory
 *     attribute); kda_get_device_status synchronises and stays outside capture.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

#define KDA_HEAD_DIM 128

typedef enum {
  KDA_OK = 0,
  KDA_ERR_NULL_POINTER = 1,      /* a required pointer is NULL                     */
  KDA_ERR_INVALID_SHAPE = 2,     /* B, T, H or N out of range, or varlen with B!=1  */
  KDA_ERR_INVALID_ARG = 3,       /* lower_bound outside [-5,0], non-finite scale,   */
                                 /* unknown enum value                              */
  KDA_ERR_MISALIGNED = 4,        /* a tensor pointer is not 16-byte aligned, or the */
                                 /* workspace is not 128-byte aligned               */
  KDA_ERR_WORKSPACE_TOO_SMALL = 5,
  KDA_ERR_UNSUPPORTED_DEVICE = 6,/* current device is not compute capability 10.3   */
  KDA_ERR_CUDA = 7,              /* a CUDA runtime / driver call failed             */
  KDA_ERR_DEVICE_TIMEOUT = 8,    /* a kernel's bounded wait expired (device status) */
  KDA_ERR_BAD_SEQLENS = 9        /* cu_seqlens not monotone or not ending at T      */
} kda_status;

typedef enum { KDA_STATE_FP32 = 0, KDA_STATE_BF16 = 1 } kda_state_dtype;

/* Intracard context parallelism over one long sequence ("feat(kda): SM90 FlashKDA
 * prefill, intracard CP, and backend dispatch", use_intracard_cp = "auto" | True |
 * False): AUTO lets the planner decide from the shapes, OFF always runs the serial
 * chunk recurrence, FORCE splits every sequence that has at least two chunks. */
typedef enum { KDA_CP_AUTO = 0, KDA_CP_OFF = 1, KDA_CP_FORCE = 2 } kda_cp_mode;

/* Which kernel computes the forward.  CHUNKED is the chunked (WY) form of the
 * pages' prefill; RECURRENT runs the recurrence token by token, as written in
 * its definition, with the state held on chip -- the cheaper form for decode
 * steps and prompts of a few tokens.  AUTO takes RECURRENT for batched input of
 * at most 16 tokens per sequence and CHUNKED otherwise (varlen input always
 * goes CHUNKED unless RECURRENT is asked for).  cp_mode only affects CHUNKED. */
typedef enum { KDA_PATH_AUTO = 0, KDA_PATH_CHUNKED = 1, KDA_PATH_RECURRENT = 2 } kda_path;

/* Storage type of the gate input g.  The pages name an fp32 gate ("fp32g") and
 * more value than q/k heads ("HV > H") as calls their SM90 kernel leaves to the
 * fused CUDA path ("feat(kda): SM90 FlashKDA prefill, intracard CP, and backend
 * dispatch", description); both are accepted here. */
typedef enum { KDA_GATE_BF16 = 0, KDA_GATE_FP32 = 1 } kda_gate_dtype;

typedef struct {
  int32_t cp_mode;      /* kda_cp_mode                                              */
  int32_t seg_chunks;   /* segment length in 64-token chunks for CP; 0 = planner's  */
  int32_t path;         /* kda_path                                                 */
  int32_t num_v_heads;  /* HV, heads of v / g / beta / out / states; 0 means H.     */
                        /* A positive multiple of H; value head j reads q/k head    */
                        /* j / (HV / H) (consecutive value heads share q and k).    */
  int32_t g_dtype;      /* kda_gate_dtype of g                                      */
  int32_t debug_stall;  /* tests of the device timeout only; 0 otherwise.  1: a    */
                        /* barrier is never completed (chunked: no chunk is handed  */
                        /* from prep to factor; recurrent: a CTA's third unit is    */
                        /* never fetched), so a bounded wait (0.5 s) expires, the   */
                        /* kernel aborts and kda_get_device_status reports          */
                        /* KDA_ERR_DEVICE_TIMEOUT; units left unprocessed write no */
                        /* outputs or final states.                                 */
  int32_t reserved[2];  /* must be zero                                             */
  void* chunk_states;   /* NULL, or a device buffer (16-byte aligned) for the start  */
                        /* states of every 64-token chunk: kda_fwd (chunked path)   */
                        /* writes them, kda_bwd (chunked path) reads them instead  */
                        /* of running its own state-checkpoint forward.             */
  size_t chunk_states_bytes;  /* its size: at least kda_get_chunk_states_size, else */
                              /* KDA_ERR_WORKSPACE_TOO_SMALL                        */
} kda_options;

/* Human-readable text for a status code (static storage, never NULL). */
KDA_API const char* kda_status_string(kda_status s);

/*
 * kda_get_workspace_size -- bytes of device workspace that kda_fwd needs for a
 * problem of total_tokens packed tokens (B*T) and H heads, written to *bytes.
 * With grouped value heads pass HV (kda_options.num_v_heads) as H: the work
 * units and states are per value head.
 * The bound depends only on (total_tokens, H) and covers every plan, every
 * number of sequences N <= total_tokens + 1 and every cp_mode.  Pass the result
 * to cudaMalloc (which gives 256-byte alignment; 128 bytes is required).
 * Errors: KDA_ERR_NULL_POINTER (bytes), KDA_ERR_INVALID_SHAPE (negative sizes, or
 * total_tokens >= 2^31, which kda_fwd rejects as well).
 * Mirrors get_workspace_size(B*T, H) of the FlashKDA binding.
 */
KDA_API kda_status kda_get_workspace_size(int64_t total_tokens, int32_t H, size_t* bytes);

/*
 * kda_get_chunk_states_size -- bytes of the kda_options.chunk_states buffer for
 * total_tokens packed tokens, N sequences and HV value heads, written to *bytes.
 * Layout: bf16 [slots][HV][128(V)][128(K)], the start state of chunk c (64 tokens,
 * counted from the sequence's first token) of sequence n in slot
 * floor(bos_n / 64) + 2n + c, bos_n its first packed token; slots = total_tokens/64
 * + 2N + 1 bounds every index.  The buffer holds no other data and needs no
 * initialisation.  Errors: KDA_ERR_NULL_POINTER, KDA_ERR_INVALID_SHAPE (negative
 * sizes, total_tokens >= 2^31).
 */
KDA_API kda_status kda_get_chunk_states_size(int64_t total_tokens, int32_t N, int32_t HV,
                                             size_t* bytes);

/*
 * kda_fwd -- enqueue the KDA forward on `stream`.
 *
 *   q, k            bf16 [B, T, H, 128], contiguous.  For varlen B == 1 and T is
 *                   the packed token count.  With no tokens (T == 0) the token
 *                   tensors q, k, v, g, beta and out may be NULL.
 *   v               bf16 [B, T, HV, 128], contiguous; HV = opts->num_v_heads, or
 *                   H when that is 0 or opts is NULL.
 *   g               [B, T, HV, 128], contiguous; bf16, or fp32 when
 *                   opts->g_dtype is KDA_GATE_FP32.
 *   beta            bf16 [B, T, HV], contiguous (raw logits; sigmoid is applied).
 *   scale           output scale (finite).
 *   out             bf16 [B, T, HV, 128], written (rows of padded tokens untouched).
 *   A_log           fp32 [HV].   dt_bias  fp32 [HV, 128].
 *   lower_bound     gate floor, in [-5, 0]; 0 gives alpha == 1.
 *   initial_state   NULL (zero state) or [N, HV, 128(V), 128(K)] in state_dtype:
 *                   element (n, h, v, k) is S[k][v] of sequence n, value head h.
 *   final_state     NULL (not written) or [N, HV, 128, 128] in state_dtype, written.
 *                   It may be the initial_state buffer itself (an in-place update):
 *                   each state is read before it is written.
 *                   Either state may be given without the other.
 *   cu_seqlens      NULL (batched: N = B sequences of length T) or int64 [N+1]
 *                   device prefix sums with cu[0] = 0, cu[N] = T and cu non-
 *                   decreasing (empty sequences allowed: their final state equals
 *                   their initial state).  Requires B == 1.
 *   B, T, H, N      sizes (H: q/k heads); N is ignored (taken as B) when
 *                   cu_seqlens is NULL.  num_v_heads not a positive multiple of H
 *                   (and not 0) gives KDA_ERR_INVALID_SHAPE.
 *   state_dtype     kda_state_dtype of initial_state and final_state.
 *   workspace       device buffer of at least kda_get_workspace_size(B*T, HV) bytes,
 *                   128-byte aligned; contents need not be initialised.  It also
 *                   holds the device status word read by kda_get_device_status.
 *   opts            NULL for defaults (KDA_CP_AUTO, KDA_PATH_AUTO, HV = H, bf16 g).
 *                   opts->chunk_states: also write every chunk's start state (bf16,
 *                   the copy the kernel forms for its output product) for a later
 *                   kda_bwd of the same inputs.  The chunked path does this for
 *                   whole sequences and for the segments of a split one (each
 *                   segment's start state is its merged one); AUTO then takes the
 *                   chunked path at any length, and RECURRENT with chunk_states is
 *                   KDA_ERR_INVALID_ARG.
 *
 * Host-side validation (shape, range, alignment, workspace size) happens before
 * anything is enqueued.  cu_seqlens lives on the device and is not read by the
 * host; its consistency is checked by the device planner, which records
 * KDA_ERR_BAD_SEQLENS in the device status word and skips the work.
 * Determinism: results are bitwise identical run to run for the same inputs,
 * sizes, options and device.
 */
KDA_API kda_status kda_fwd(const void* q, const void* k, const void* v, const void* g,
                   const void* beta, float scale, void* out, const float* A_log,
                   const float* dt_bias, float lower_bound, const void* initial_state,
                   void* final_state, const int64_t* cu_seqlens, int64_t B, int64_t T,
                   int32_t H, int32_t N, int32_t state_dtype, void* workspace,
                   size_t workspace_bytes, const kda_options* opts, cudaStream_t stream);

/*
 * kda_get_device_status -- copy the device status word of the last kda_fwd that
 * used `workspace` into *status (KDA_OK, KDA_ERR_DEVICE_TIMEOUT or
 * KDA_ERR_BAD_SEQLENS).  This call synchronises `stream` (it is the one entry
 * point that does), so keep it off the hot path.
 */
KDA_API kda_status kda_get_device_status(const void* workspace, kda_status* status,
                                 cudaStream_t stream);

/*
 * kda_fwd_transition -- enqueue the affine form of the forward over each
 * sequence: the recurrence is affine in the state, S_end = M S_start + B, with M
 * independent of the values.  For every (sequence n, value head h) it writes
 *   M_out[n][h]  the transition M, i.e. the final state of the run from the
 *                identity with v = 0, and
 *   B_out[n][h]  the offset B, the final state of the run from zero,
 * both fp32 [N, HV, 128, 128] in the state layout (element (n, h, i, j) is
 * X[i][j] with X = M^T, B^T).  This is the pre_scan of the segment split in
 * "feat(kda): SM90 FlashKDA prefill, intracard CP, and backend dispatch" (commit
 * notes: K1 once -> pre_scan -> merge -> segment-K2), applied to a whole
 * sequence shard so that ranks holding consecutive shards of one sequence can
 * exchange (M, B) and compose their start states (the review thread's "Kimi CP
 * gives each rank a sequence shard ... nesting"); see kda_compose_states.
 *   q .. dt_bias, lower_bound, cu_seqlens, B, T, H, N, opts   as for kda_fwd
 *                   (opts->path and cp_mode are ignored: whole sequences, the
 *                   chunked kernel).
 *   M_out, B_out    fp32 device buffers of N * HV * 128 * 128 floats, 16-byte aligned.
 *   workspace       as for kda_fwd (>= kda_get_workspace_size(B*T, HV) bytes); its
 *                   status word reports bad cu_seqlens and bounded-wait timeouts.
 * Errors: those of kda_fwd for the shared arguments; KDA_ERR_NULL_POINTER
 * (M_out, B_out), KDA_ERR_MISALIGNED.
 */
KDA_API kda_status kda_fwd_transition(const void* q, const void* k, const void* v, const void* g,
                                      const void* beta, const float* A_log, const float* dt_bias,
                                      float lower_bound, const int64_t* cu_seqlens, int64_t B,
                                      int64_t T, int32_t H, int32_t N, float* M_out, float* B_out,
                                      void* workspace, size_t workspace_bytes,
                                      const kda_options* opts, cudaStream_t stream);

/*
 * kda_compose_states -- enqueue the merge of affine state maps in a fixed order:
 *     X = S_in (or zero when S_in is NULL);  X <- X M[r] + B[r],  r = 0 .. R-1;
 *     S_out = X
 * for num_states independent states at once, all fp32 in the state layout of
 * kda_fwd_transition (so X M[r] + B[r] is S <- M_r S + B_r on the states
 * themselves).  M, B: [R, num_states, 128, 128]; S_in, S_out: [num_states, 128,
 * 128]; all 16-byte aligned device buffers, S_out distinct from the inputs.
 * The merge step of the segment split ("feat(kda): SM90 FlashKDA prefill,
 * intracard CP, and backend dispatch", commit notes), used across ranks: rank r
 * composes the (M, B) of the shards before its own into its start state.
 * Errors: KDA_ERR_NULL_POINTER, KDA_ERR_INVALID_SHAPE (R < 0, num_states out of
 * [0, 2^27)), KDA_ERR_MISALIGNED, KDA_ERR_UNSUPPORTED_DEVICE, KDA_ERR_CUDA.
 */
KDA_API kda_status kda_compose_states(const float* M, const float* B, int32_t R,
                                      int64_t num_states, const float* S_in, float* S_out,
                                      cudaStream_t stream);

/*
 * kda_bwd_get_workspace_size -- bytes of device workspace that kda_bwd needs for
 * total_tokens packed tokens, N sequences, H q/k heads and num_v_heads value
 * heads (0 = H), written to *bytes: state checkpoints every 16 tokens of every
 * (sequence, value head) (64 KiB each; the chunked path keeps its bf16 chunk-start
 * states, 32 KiB per 64 tokens, in the same region), a recomputation scratch of
 * 256 KiB per CTA (at most 160 CTAs), per-unit partial sums and, for grouped value
 * heads, per-value-head dq / dk partials.  The size covers both paths.  Errors:
 * KDA_ERR_NULL_POINTER, KDA_ERR_INVALID_SHAPE (negative sizes, HV not a multiple
 * of H, total_tokens >= 2^31).
 */
KDA_API kda_status kda_bwd_get_workspace_size(int64_t total_tokens, int32_t N, int32_t H,
                                              int32_t num_v_heads, size_t* bytes);

/*
 * kda_bwd -- enqueue the backward pass: the gradients of
 *     L = <dout, out> + <dfinal_state, final_state>
 * with respect to every input of kda_fwd.  The pages' kernels are forward only
 * ("feat(kda): SM90 FlashKDA prefill, intracard CP, and backend dispatch",
 * commit notes); both paths below are reverse modes derived from the same
 * recurrence and preprocessing.
 *   opts->path KDA_PATH_AUTO / KDA_PATH_CHUNKED (default): the chunked WY form on
 *     the tensor cores.  The forward kernel first runs in a state-checkpoint mode
 *     (no outputs) and keeps each 64-token chunk's start state in bf16 -- or, when
 *     opts->chunk_states is given, the states that a kda_fwd of the same inputs
 *     with the same buffer wrote are read from it and that pass is skipped; a reverse
 *     sweep over the chunks then forms every gradient with bf16 MMA operands and
 *     fp32 accumulation (the forward kernel's arithmetic).  Gradients are accurate
 *     to about 1e-2 of each tensor's largest magnitude; q, k and v must be 16-byte
 *     aligned (KDA_ERR_MISALIGNED otherwise).
 *   opts->path KDA_PATH_RECURRENT: token by token in fp32, states recomputed from
 *     16-token checkpoints; the exact gradient of the recurrence as written, to
 *     fp32 rounding, at several times the chunked path's cost.  chunk_states must
 *     be NULL on this path (KDA_ERR_INVALID_ARG).
 *
 *   q .. state_dtype, cu_seqlens, opts   as for kda_fwd (the same call's inputs;
 *                   opts->debug_stall: 0, or 1 on the chunked path only, where the
 *                   reverse kernel then never issues a chunk's first MMAs, its bounded
 *                   wait expires and the status word reads KDA_ERR_DEVICE_TIMEOUT:
 *                   the timeout test's hook).
 *   dout            bf16 [B, T, HV, 128], the gradient of out.
 *   dfinal_state    NULL (zero) or [N, HV, 128(V), 128(K)] in state_dtype.
 *   dq, dk          fp32 [B, T, H, 128], written.
 *   dv, dg          fp32 [B, T, HV, 128], written (dg: the gradient of the raw gate
 *                   input g, whatever its storage type).
 *   dbeta           fp32 [B, T, HV] (gradient of the raw beta logits), written.
 *   dA_log          fp32 [HV], ddt_bias fp32 [HV, 128], written (sums over all
 *                   sequences and tokens).
 *   dinitial_state  NULL (not written) or fp32 [N, HV, 128, 128], written.
 *   workspace       at least kda_bwd_get_workspace_size(B*T, N, H, num_v_heads)
 *                   bytes, 128-byte aligned; its first word is the device status
 *                   read by kda_get_device_status (bad cu_seqlens).
 * Results are bitwise reproducible run to run on either path.  Host-side errors
 * are those of kda_fwd; gradient pointers dq, dk, dg must be 16-byte aligned.  On
 * the chunked path a bounded wait that expires is recorded in the status word
 * (KDA_ERR_DEVICE_TIMEOUT through kda_get_device_status).
 */
KDA_API kda_status kda_bwd(const void* q, const void* k, const void* v, const void* g,
                           const void* beta, float scale, const float* A_log,
                           const float* dt_bias, float lower_bound, const void* initial_state,
                           const void* dout, const void* dfinal_state, const int64_t* cu_seqlens,
                           float* dq, float* dk, float* dv, float* dg, float* dbeta,
                           float* dA_log, float* ddt_bias, float* dinitial_state, int64_t B,
                           int64_t T, int32_t H, int32_t N, int32_t state_dtype, void* workspace,
                           size_t workspace_bytes, const kda_options* opts, cudaStream_t stream);

/*
 * kda_fwd_static_scratch -- kda_fwd for callers that cannot allocate device
 * memory.  The pages have no counterpart of this entry point.
 *
 * Some callers cannot call cudaMalloc: a host framework that reserves all device
 * memory up front and passes a plugin only its input and output buffers, or an
 * embedded runtime with a fixed memory budget that forbids allocations after
 * start-up.  This entry point takes the same arguments as kda_fwd minus the
 * workspace, and runs the same forward with its workspace in a device array that
 * the library declares at file scope: KDA_STATIC_SCRATCH_BYTES bytes, which every
 * GPU that loads the library holds until the process exits.  It allocates
 * nothing (no cudaMalloc, no cudaFree, no allocating library routine).
 *
 *   - Limit: problems whose kda_get_workspace_size(B*T, HV) exceeds
 *     KDA_STATIC_SCRATCH_BYTES are rejected with KDA_ERR_WORKSPACE_TOO_SMALL
 *     (the five reference workloads need at most about 34 MiB).
 *   - The first call on a device looks up the array's device address with that
 *     device current; make that first call before any stream capture.  The
 *     address is kept per device and CUDA context (a call from another context
 *     looks it up again).  A device reset (cudaDeviceReset) that re-creates the
 *     primary context under the same handle leaves the kept address stale: do
 *     not use this entry point across a device reset.
 *   - Every call shares the one array, which keeps the last call's contents; each
 *     call clears what must start at zero.  Calls that overlap on the GPU (other
 *     streams, or other host threads on one device) race on the array: serialise
 *     them.
 *   - The device status word lives in the array: device-side errors (a
 *     bounded-wait timeout, inconsistent cu_seqlens) skip the affected work and
 *     are recorded there; kda_static_scratch_device_status reads them back.
 * Host-side errors are those of kda_fwd, checked in kda_fwd's order before the
 * size limit.
 */
#define KDA_STATIC_SCRATCH_BYTES (40u * 1024u * 1024u)

KDA_API kda_status kda_fwd_static_scratch(const void* q, const void* k, const void* v,
                                          const void* g, const void* beta, float scale,
                                          void* out, const float* A_log, const float* dt_bias,
                                          float lower_bound, const void* initial_state,
                                          void* final_state, const int64_t* cu_seqlens,
                                          int64_t B, int64_t T, int32_t H, int32_t N,
                                          int32_t state_dtype, const kda_options* opts,
                                          cudaStream_t stream);

/*
 * kda_static_scratch_device_status -- the device status word of the last
 * kda_fwd_static_scratch call on the current device, as kda_get_device_status
 * reads it for a caller workspace (KDA_OK, KDA_ERR_DEVICE_TIMEOUT or
 * KDA_ERR_BAD_SEQLENS) into *status.  It synchronises `stream`; the pages have no
 * counterpart.  Errors: KDA_ERR_NULL_POINTER (status), KDA_ERR_CUDA.
 */
KDA_API kda_status kda_static_scratch_device_status(kda_status* status, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
