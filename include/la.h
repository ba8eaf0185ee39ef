/*
 * la.h -- C ABI of the chunkwise linear-attention forward library (libla.so)
 * for NVIDIA GB300 (sm_103a).
 *
 * The library computes, for every batch entry b and head h independently,
 * the causal forward pass of the matrix-state recurrence
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T ,
 *     o_t = S_t^T q_t ,
 *
 * and its special cases, with S key-major ([dk][dv], float32). The pages this
 * follows state the same recurrence value-major (S = sum v k^T, o = S q;
 * "Talk Linear Attention" section 6; "LLM attention optimisation: linear
 * attention", DeltaNet and Gated DeltaNet sections); the key-major state here
 * is its transpose and gives the same o. The sequence is processed in chunks
 * of C tokens ("Talk Linear Attention" section 3.2: local attention inside a
 * chunk, state passing between chunks); the result equals the token-by-token
 * recurrence up to floating-point rounding.
 *
 * Entry points: la_chunk_fwd (the causal forward in every mode, and the
 * non-causal form), la_chunk_fwd_noalloc (its materialised variant without
 * allocation), la_chunk_fwd_gdelta (the generalised delta rule
 * S_t = (I - b_t a_t^T) S_{t-1} + k_t v_t^T), la_chunk_bwd (the backward pass
 * for LA_LINEAR, LA_RETNET, LA_SCALAR_GATE and LA_GLA), la_chunk_bwd_delta
 * (the backward pass for LA_GDN), la_recurrent_step
 * (one decode step), la_prologue (short convolution, L2 norm and gate
 * activations in front of the forward), la_stream_status, la_last_error,
 * la_version.
 *
 * Conventions for every entry point
 *   - Tensors are dense row-major: q, k [B][H][T][dk], v, o [B][H][T][dv]
 *     (d fastest). Decode steps drop the T axis.
 *   - q, k, v and o share one dtype: bfloat16 by default, float32 when the
 *     LA_F32 flag is set in `mode`. All arithmetic accumulates in float32.
 *   - Gates g are natural logarithms: the decay applied is alpha = exp(g).
 *   - The state is float32 [B][H][dk][W] with W = dv, except for
 *     LA_ELU1_NORM where W = dv + 1 and column dv holds the normaliser z.
 *   - All pointers are DEVICE pointers owned by the caller. The library never
 *     frees or retains them. Device memory of its own is taken only by the
 *     materialised variant, the two-phase delta-rule variant, the LA_KDA
 *     path and the non-causal form of la_chunk_fwd, by the bfloat16 path of
 *     la_chunk_fwd_gdelta, and by la_chunk_bwd and la_chunk_bwd_delta:
 *     workspaces allocated and freed on `stream` from a library-owned
 *     stream-ordered pool (one per device) that keeps freed memory for the
 *     next call.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream);
 *     nothing synchronises with the host.
 *   - Return value: LA_OK, or an LA_ERR_* code with a message available from
 *     la_last_error() (thread-local). Argument errors are detected on the host
 *     before anything is launched; nothing is written in that case.
 */
#ifndef LA_H
#define LA_H

#ifdef __cplusplus
extern "C" {
#endif

/* Same underlying type as cudaStream_t / CUstream: pass either directly. */
struct CUstream_st;
typedef struct CUstream_st *la_stream_t;

/* ---- status codes ------------------------------------------------------ */
#define LA_OK                0
#define LA_ERR_INVALID_ARG   1  /* null required pointer, bad size, misalignment, g/beta vs mode */
#define LA_ERR_UNSUPPORTED   2  /* valid request this build does not implement (dims, C, dtype) */
#define LA_ERR_CUDA          3  /* a CUDA runtime/driver call or launch failed */
#define LA_ERR_TIMEOUT       4  /* a kernel gave up waiting on a device barrier (see la_stream_status) */

/* ---- modes (low byte) and flags ---------------------------------------- */
/* Plain causal linear attention: S_t = S_{t-1} + k_t v_t^T, o_t = S_t^T q_t.
 * ("Talk Linear Attention", section 2.1.) g and beta must be NULL. */
#define LA_LINEAR        0
/* Kernelised attention phi(x) = elu(x) + 1 with the causal normaliser:
 * S_t = S_{t-1} + phi(k_t) v_t^T, z_t = z_{t-1} + phi(k_t),
 * o_t = S_t^T phi(q_t) / (z_t . phi(q_t)).  (Kernel-attention notes,
 * sections 13-14; "Linear Attention" glossary.) g and beta must be NULL.
 * The library applies phi; the state has dv + 1 columns (z in column dv). */
#define LA_ELU1_NORM     1
/* Fixed per-head decay (RetNet): S_t = gamma_h S_{t-1} + k_t v_t^T.
 * g = float32 [H] holding log gamma_h. beta must be NULL. */
#define LA_RETNET        2
/* GLA diagonal gate on the key axis: S_t = Diag(alpha_t) S_{t-1} + k_t v_t^T
 * ("Talk Linear Attention", section 5.1). g = float32 [B][H][T][dk]
 * (per step [B][H][dk]), 16-byte aligned. beta must be NULL. Chunked
 * evaluation factors exp(b_r - b_s) per channel around the chunk midpoint;
 * a cumulative log-gate magnitude above ~80 within half a chunk underflows. */
#define LA_GLA           3
/* Data-dependent scalar decay (Mamba-2 form): S_t = alpha_t S_{t-1} + k_t v_t^T.
 * g = float32 [B][H][T] (per step [B][H]). beta must be NULL. */
#define LA_SCALAR_GATE   4
/* Gated DeltaNet: decay, then the delta rule,
 * S_t = (I - beta_t k_t k_t^T) alpha_t S_{t-1} + beta_t k_t v_t^T
 * ("LLM attention optimisation", Gated DeltaNet section; "Talk Linear
 * Attention" section 6.2). g = float32 [B][H][T] or NULL (alpha = 1, plain
 * DeltaNet); beta = float32 [B][H][T] or NULL (beta = 1). */
#define LA_GDN           5
/* Kimi Delta Attention: Gated DeltaNet with a per-key-channel gate,
 * S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 * ("LLM attention optimisation", Kimi Delta Attention section; Diag(alpha_t)
 * acts on the key axis). g = float32 [B][H][T][dk] (per step [B][H][dk]),
 * 16-byte aligned; beta = float32 [B][H][T] or NULL (beta = 1). bfloat16
 * inputs only in la_chunk_fwd (LA_F32 is LA_ERR_UNSUPPORTED); chunked
 * evaluation folds exp(b_r - b_s) per channel around the chunk midpoint as
 * for LA_GLA, with the same range limit. la_chunk_fwd runs it in two phases
 * (every chunk's key side in parallel into a workspace of
 * B*H*ceil(T/64)*(3*64*dk*2 + 2*64*64*2 + dk*4) bytes from the library's
 * pool, then the state chain; B*H <= 65535, else LA_ERR_UNSUPPORTED);
 * LA_KDA=tc or LA_VARIANT=tc selects the fused kernel instead. */
#define LA_KDA           6
/* Outer-product gate: S_t = (alpha_t beta_t^T) ⊙ S_{t-1} + k_t v_t^T, a
 * key-axis gate alpha_t (row c of S) times a value-axis gate beta_t (column
 * j) -- the gate form "Talk Linear Attention" section 5.4 gives for gated
 * linear attention that remains a matrix product. g = float32 [B][H][T][dk]
 * holding log alpha; the beta argument carries float32 [B][H][T][dv] holding
 * log beta (both required, 16-byte aligned; per step [B][H][dk] and
 * [B][H][dv]). bfloat16 inputs only in la_chunk_fwd. Chunked evaluation
 * folds both axes' gates around the chunk midpoint; the range limit of
 * LA_GLA applies to the sum of the two axes' log-gates: for every key
 * channel c and value column j, log alpha_c + log beta_j summed over half a
 * chunk (32 tokens) must stay above about -80, else the state overflows. */
#define LA_OUTER_GATE    7
/* Flag: q, k, v and o are float32 instead of bfloat16. */
#define LA_F32           0x100
/* Flag (la_chunk_fwd only, with LA_LINEAR or LA_ELU1_NORM, bfloat16): the
 * non-causal form, every token reads the state of the whole sequence,
 *     o_t = S_T^T q_t,  S_T = S0 + sum_{s<T} k_s v_s^T
 * (elu+1: o_t = S_T^T phi(q_t) / (z_T . phi(q_t))), computed right to left as
 * Q (K^T V) (kernel-attention notes, section 3).
 * S_final is S_T, as in the causal form. Uses a stream-ordered workspace
 * from the library's pool (B*H*splits*dk*(dv + 1)*4 bytes, splits <= 2*SMs/(B*H)). */
#define LA_NONCAUSAL     0x200

/*
 * la_chunk_fwd -- causal forward pass over a whole sequence, chunkwise.
 *
 *   q, k    [B][H][T][dk]  input dtype, 16-byte aligned
 *   v       [B][H][T][dv]  input dtype, 16-byte aligned
 *   g       float32, shape per mode (see the mode list), or NULL
 *   beta    float32 [B][H][T] (LA_GDN only) or NULL
 *   o       [B][H][T][dv]  output, input dtype, 16-byte aligned; written
 *   S0      float32 [B][H][dk][W] initial state, or NULL for zero
 *   S_final float32 [B][H][dk][W] final state, or NULL to skip writing it
 *           (may alias S0: every head reads its S0 before writing S_final)
 *   B, H, T >= 1; dk, dv in {64, 128}
 *   C       chunk length: 0 (pick per shape), 64 or 128. C = 128 runs the
 *           materialised variant of LA_LINEAR, LA_ELU1_NORM, LA_RETNET and
 *           LA_SCALAR_GATE (bfloat16, causal); for any other mode or flag it
 *           returns LA_ERR_UNSUPPORTED on the host, before any CUDA call, as
 *           it does when LA_VARIANT forces another variant. Any other value
 *           is LA_ERR_INVALID_ARG.
 *   mode    one LA_* mode, optionally | LA_F32
 *
 * S_final of one call passed as S0 of the next continues the sequence
 * (the recurrent state is the whole checkpoint).
 *
 * Kernel variants ("Talk Linear Attention" section 4.1.2). Fused: one CTA per
 * head walks the chunks, keeping the state on chip; nothing but q, k, v, o and
 * the states touches memory. Materialised (unit-write modes, bfloat16): a
 * state pass writes every chunk's incoming state to a workspace of
 * B*H*ceil(T/C)*dk*256 bytes (plus B*H*ceil(T/C)*dk*4 for LA_ELU1_NORM),
 * then all chunks' outputs are computed in parallel; it wins when B*H is too
 * small to fill the GPU. The state pass walks each head's chunks in order,
 * except for LA_LINEAR and LA_ELU1_NORM, whose chunk states are prefix sums:
 * there every 64-token chunk's K^T V is formed at once into
 * B*H*ceil(T/64)*dk*dv*4 more bytes of workspace (plus B*H*ceil(T/64)*dk*4
 * for LA_ELU1_NORM) and a scan adds them up, while those take at most 2 GiB
 * (the environment variable LA_MAT_STATE=serial keeps the serial walk). The choice is made per shape: materialised for the
 * unit-write modes when T >= 512 and B*H <= SMs / 2 (GLA: SMs / 4; elu+1:
 * any B*H), fused otherwise; with C = 0 the materialised variant runs C = 128
 * for LA_LINEAR and LA_ELU1_NORM, and for LA_RETNET and LA_SCALAR_GATE when
 * T >= 2048, else C = 64. The fused kernels run C = 64. Gated DeltaNet runs fused by default; its two-phase variant (the
 * triangular solve of every chunk first, written as one 8 KB image per chunk of
 * 64 tokens to a workspace of B*H*ceil(T/64)*8192 bytes, then the state chain,
 * dk = dv = 128) is selected by LA_DELTA=wy. The environment variable
 * LA_VARIANT = tc (or nonmat) | mat | simt forces a variant.
 */
int la_chunk_fwd(const void *q, const void *k, const void *v, const float *g, const float *beta,
                 void *o, const float *S0, float *S_final,
                 int B, int H, int T, int dk, int dv, int C, int mode, la_stream_t stream);

/*
 * la_chunk_fwd_noalloc -- la_chunk_fwd's materialised variant with its
 * workspace in a static device array instead of an allocation, for callers
 * that cannot allocate device memory. The pages have no counterpart to this
 * entry point: it is an interface of this library only.
 *
 *   Arguments, layouts and results as la_chunk_fwd, restricted to the modes
 *   the materialised variant covers: LA_LINEAR, LA_ELU1_NORM, LA_RETNET,
 *   LA_GLA and LA_SCALAR_GATE, bfloat16, causal, C = 0 (64) or 64, or 128
 *   for every one of them but LA_GLA. Rejected on the host before any CUDA
 *   call: LA_GDN, LA_KDA and LA_OUTER_GATE (LA_ERR_UNSUPPORTED), LA_F32
 *   (LA_ERR_UNSUPPORTED), C = 128 with LA_GLA (LA_ERR_UNSUPPORTED),
 *   LA_NONCAUSAL or any other flag, an unknown mode, a missing or
 *   superfluous g, any beta (LA_ERR_INVALID_ARG). Scratch needed:
 *   B*H*ceil(T/C)*dk*256 bytes, plus B*H*ceil(T/C)*dk*4 for LA_ELU1_NORM. A call that needs more than LA_NOALLOC_SCRATCH_BYTES
 *   is rejected with LA_ERR_INVALID_ARG before anything is launched.
 *   Allocates nothing: no cudaMalloc, cudaFree or stream-ordered allocation.
 *   The scratch is one array per device, shared by every call on that
 *   device: calls that overlap on the GPU (several streams or host threads)
 *   race on it, so the caller orders them. Nothing in it needs to start at
 *   zero. Every call looks up the array's address on the current device
 *   (the first call on a device may load the module holding it: make that
 *   first call before any stream capture). The array is device memory held
 *   for the life of the CUDA context once its module is loaded: with lazy
 *   module loading (the CUDA default) that is the first la_chunk_fwd_noalloc
 *   call on the device; with CUDA_MODULE_LOADING=EAGER every process that
 *   loads libla.so holds the 32 MiB on every device it uses.
 */
#define LA_NOALLOC_SCRATCH_BYTES 0x2000000  /* 32 MiB */
int la_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const float *g,
                         const float *beta, void *o, const float *S0, float *S_final,
                         int B, int H, int T, int dk, int dv, int C, int mode, la_stream_t stream);

/*
 * la_prologue -- the per-token steps that turn the q/k/v/gate/beta
 * projections into la_chunk_fwd's inputs, in one pass over memory:
 *
 *   1. short convolution ("LLM attention optimisation: linear attention",
 *      DeltaNet section: a depthwise convolution over the last K tokens after
 *      the projections), on each of q, k and v:
 *          x~_t[c] = sum_{tau=0}^{K-1} w[h][c][tau] * x_{t-tau}[c]
 *      Tokens before the first come from hist_in, else are zero.
 *   2. optional L2 normalisation of q~ and/or k~ per token:
 *          x / max(||x||_2, 1e-6)   (the pages do not state it; Gated DeltaNet
 *          is used with L2-normalised q and k)
 *   3. gate activation of a_gate into natural-log gates g:
 *          LA_GATE_LOGSIGMOID    g = logsigmoid(a) / tau  (log of
 *                                sigmoid(.)^(1/tau): "Talk Linear Attention"
 *                                section 5.1, the GLA gate)
 *          LA_GATE_NEG_SOFTPLUS  g = -softplus(a) / tau  (alpha in (0, 1))
 *   4. beta = sigmoid(a_beta).
 *
 *   xq, xk  bfloat16 [B][H][T][dk]; xv bfloat16 [B][H][T][dv]; 16-byte aligned
 *   wq, wk  float32 [H][dk][K], wv float32 [H][dv][K]; w[..][0] weights the
 *           current token. NULL: no convolution for that tensor (identity).
 *   K       convolution length, 1..4
 *   hist_in / hist_out
 *           bfloat16 [B][H][K-1][2*dk + dv]: per (b, h), the K-1 raw rows
 *           (before the convolution) preceding this call's first token, oldest
 *           first, each row the q, k and v projections side by side. hist_out
 *           receives the last K-1 raw rows of hist_in ++ x, so passing it as
 *           the next call's hist_in continues the sequence. Either may be NULL
 *           (zero history / not written); they must not alias. Ignored if K = 1.
 *   a_gate  float32 [B][H][T] (gate_width 1) or [B][H][T][dk] (gate_width dk);
 *           gate_kind LA_GATE_NONE: a_gate, g unused (may be NULL)
 *   tau     finite, > 0
 *   a_beta  float32 [B][H][T] or NULL (then beta is not written)
 *   q, k, v outputs, bfloat16, shapes of xq, xk, xv, 16-byte aligned
 *   g, beta float32 outputs, shapes of a_gate, a_beta
 *   flags   LA_PRO_L2NORM_Q | LA_PRO_L2NORM_K
 *
 * Arithmetic in float32; q, k, v rounded to bfloat16 once. Outputs must not
 * overlap the inputs. The pages have no single routine for this: it bundles
 * the steps they place before the recurrence.
 */
#define LA_GATE_NONE          0
#define LA_GATE_LOGSIGMOID    1
#define LA_GATE_NEG_SOFTPLUS  2
#define LA_PRO_L2NORM_Q       1
#define LA_PRO_L2NORM_K       2
int la_prologue(const void *xq, const void *xk, const void *xv,
                const float *wq, const float *wk, const float *wv, int K,
                const void *hist_in, void *hist_out,
                const float *a_gate, int gate_kind, int gate_width, float tau,
                const float *a_beta,
                void *q, void *k, void *v, float *g, float *beta,
                int B, int H, int T, int dk, int dv, int flags, la_stream_t stream);

/*
 * la_chunk_bwd -- the backward pass of la_chunk_fwd for LA_LINEAR, LA_RETNET
 * and LA_SCALAR_GATE, optionally | LA_F32: given dO = dL/do and
 * dS_final = dL/dS_final, the gradients
 *
 *   dq_t = alpha^(t+1) S0 dO_t + sum_{s<=t} alpha^(t-s) (dO_t . v_s) k_s
 *   dk_s = sum_{t>=s} alpha^(t-s) (dO_t . v_s) q_t + alpha^(T-1-s) dS_final v_s
 *   dv_s = sum_{t>=s} alpha^(t-s) (q_t . k_s) dO_t + alpha^(T-1-s) dS_final^T k_s
 *   dS0  = sum_t alpha^(t+1) q_t dO_t^T + alpha^T dS_final
 *
 * (alpha = 1, or gamma_h = exp(g_h); for LA_SCALAR_GATE alpha^(t-s) stands
 * for the product of exp(g) over the tokens s+1 .. t, and alpha^(t+1) for
 * tokens 0 .. t), and for LA_SCALAR_GATE the gradient of the log-gates
 *
 *   dg_tau = sum_{u>=tau} (q_u . dq_u - k_u . dk_u) + sum(dS_final ⊙ S_final).
 *
 * The chunk states are recomputed, not stored ("Talk Linear Attention"
 * section 4.1.2).
 *
 *   q, k, v, g, S0  as passed to la_chunk_fwd (S0 may be NULL: zero)
 *   dO       [B][H][T][dv], input dtype; dS_final float32 [B][H][dk][dv] or NULL (zero)
 *   dq_out, dk_out [B][H][T][dk]; dv_out [B][H][T][dv]: dq, dk, dv, input dtype
 *   dS0      float32 [B][H][dk][dv] output, or NULL (not computed)
 *   dg_out   float32 [B][H][T] output for LA_SCALAR_GATE, or NULL (not
 *            computed); must be NULL for the other modes
 *   16-byte alignment for every pointer. For LA_RETNET, g_h > -80 (the
 *   passes divide dS_final by gamma_h). C = 0 or 64.
 * Runs as three chunk-forward passes on `stream` (two of them run the
 * recurrence over the time-reversed sequence, reading and writing the
 * tensors where they are), plus, for dg with dS_final, a forward pass for
 * S_final and a suffix-sum kernel; workspace from the library's pool of
 * 16*B*H*dk*dv bytes (initial states of the passes), + 4*B*H*dk*dv +
 * B*H*T*dv*esize with dg.
 */
int la_chunk_bwd(const void *q, const void *k, const void *v, const float *g, const void *dO,
                 const float *dS_final, const float *S0, void *dq_out, void *dk_out, void *dv_out,
                 float *dS0, float *dg_out, int B, int H, int T, int dk, int dv, int C, int mode,
                 la_stream_t stream);

/*
 * la_chunk_bwd_delta -- the backward pass of la_chunk_fwd for LA_GDN (Gated
 * DeltaNet) and LA_KDA (Kimi Delta Attention), bfloat16: given dO = dL/do and
 * dS_final = dL/dS_final, the gradients of L through the recurrence
 *
 *   R_t = Diag(alpha_t) S_{t-1},  r_t = v_t - R_t^T k_t,  S_t = R_t + beta_t k_t r_t^T,
 *   o_t = S_t^T q_t
 *
 * (alpha_t a scalar for LA_GDN, one value per key channel for LA_KDA; "LLM
 * attention optimisation" page, Gated DeltaNet and Kimi Delta Attention
 * sections; "Talk Linear Attention" section 6.2), i.e. with Gh_t = dL/dS_t
 * (later tokens and o_t):
 *
 *   dq_t = S_t dO_t,  dv_t = beta_t Gh_t^T k_t,  dbeta_t = (Gh_t^T k_t) . r_t,
 *   dk_t = beta_t (Gh_t r_t - R_t Gh_t^T k_t),
 *   dg_t = <(I - beta_t k_t k_t^T) Gh_t, R_t> (LA_KDA: the row sums, one per key
 *          channel),  dS0 = dL/dS_{-1}.
 *
 * Chunkwise (C = 64) through the WY form of the forward: the chunk states and
 * the state gradients at the chunk boundaries are recomputed by two serial
 * passes ("Talk Linear Attention" section 4.1.2; bf16 warp MMAs, fp32 states),
 * then every chunk's gradients are computed in parallel (tf32 warp MMAs,
 * float32 arithmetic). LA_KDA folds the per-channel gate into the keys and
 * queries around each chunk's midpoint row, as its forward does.
 *
 *   q, k, v, g, beta, S0  as passed to la_chunk_fwd for the mode (LA_GDN: g
 *            NULL means alpha = 1; LA_KDA: g [B][H][T][dk] required; beta NULL:
 *            beta = 1; S0 NULL: zero); bfloat16 q, k, v
 *   dO       [B][H][T][dv] bfloat16; dS_final float32 [B][H][dk][dv] or NULL (zero)
 *   dq_out, dk_out [B][H][T][dk]; dv_out [B][H][T][dv]: bfloat16 outputs
 *   dbeta_out float32 [B][H][T] or NULL (not written; with beta NULL it is the
 *            gradient at beta = 1)
 *   dg_out   float32, g's shape, or NULL; needs g (LA_ERR_INVALID_ARG otherwise)
 *   dS0      float32 [B][H][dk][dv] or NULL
 *   mode     LA_GDN or LA_KDA (another known mode or LA_F32: LA_ERR_UNSUPPORTED;
 *            an unknown one: LA_ERR_INVALID_ARG); C = 0 or 64
 *   16-byte alignment for every pointer; B*H <= 65535.
 * Workspace from the library's pool, per (b, h) and chunk of 64 tokens:
 * LA_GDN (2*64*64 + 2*dk*dv)*4 + 2*64*64*2 bytes (the triangular inverses and
 * masked scores in float32 and bf16, the states and state gradients at the
 * chunk boundaries); LA_KDA (2*64*64 + 2*dk*dv + dk)*4 + (2*64*64 + 3*64*dk)*2
 * bytes (the same plus the folded key and query images and e^{B_L}). Four
 * kernels on `stream`; errors as la_chunk_fwd.
 */
int la_chunk_bwd_delta(const void *q, const void *k, const void *v, const float *g, const float *beta,
                       const void *dO, const float *dS_final, const float *S0, void *dq_out, void *dk_out,
                       void *dv_out, float *dbeta_out, float *dg_out, float *dS0, int B, int H, int T,
                       int dk, int dv, int C, int mode, la_stream_t stream);

/*
 * la_chunk_fwd_gdelta -- causal forward of the generalised delta rule, an
 * identity-plus-rank-one transition between linear-attention steps ("Talk
 * Linear Attention", section 7.1, which writes the value-major
 * S_t = S_{t-1}(I - a_t b_t^T) + v_t k_t^T). In this library's key-major
 * orientation:
 *
 *   S_t = (I - b_t a_t^T) S_{t-1} + k_t v_t^T,   o_t = S_t^T q_t
 *
 * (retrieve with a_t, erase along b_t, unit write). a = b = sqrt(beta) k with
 * beta k as the write key gives DeltaNet.
 *
 *   q, k, a, b [B][H][T][dk]; v, o [B][H][T][dv]: bfloat16, or float32 with
 *            mode = LA_F32 (mode 0: bfloat16); 16-byte aligned
 *   S0, S_final  float32 [B][H][dk][dv] or NULL (zero / not written),
 *            16-byte aligned; S_final may alias S0
 *   C        0 or 64
 * Chunkwise (C = 64). bfloat16: two phases on bf16 warp MMAs (fp32
 * accumulate) -- every chunk's key side in parallel (T = (I + L_ab)^{-1}, T A,
 * T L_ak and the two masked score matrices) into bf16 images, a workspace of
 * B*H*ceil(T/64)*(64*dk + 3*64*64)*2 bytes from the library's pool, then the
 * state chain per head and 16 value columns; B*H <= 65535. float32 (LA_F32), or bfloat16 with the environment
 * variable LA_GDELTA=simt: one pass on the CUDA cores in float32, no
 * workspace. Errors as la_chunk_fwd; asynchronous on `stream`.
 */
int la_chunk_fwd_gdelta(const void *q, const void *k, const void *v, const void *a, const void *b,
                        void *o, const float *S0, float *S_final, int B, int H, int T, int dk, int dv,
                        int C, int mode, la_stream_t stream);

/*
 * la_recurrent_step -- one decode step (the recurrent form, "Talk Linear
 * Attention" section 2.1; kernel-attention notes section 14): for every
 * (b, h), apply the mode's update with this token and write o = S^T q
 * (divided by z . phi(q) for LA_ELU1_NORM).
 *
 *   q, k [B][H][dk]; v, o [B][H][dv] (input dtype, 4-byte aligned)
 *   g    LA_RETNET [H]; LA_GLA / LA_KDA / LA_OUTER_GATE [B][H][dk];
 *        LA_SCALAR_GATE / LA_GDN [B][H]
 *   beta LA_GDN / LA_KDA [B][H] or NULL; LA_OUTER_GATE [B][H][dv] (log beta)
 *   S    float32 [B][H][dk][W], updated in place
 */
int la_recurrent_step(const void *q, const void *k, const void *v, const float *g,
                      const float *beta, void *o, float *S,
                      int B, int H, int dk, int dv, int mode, la_stream_t stream);

/*
 * la_stream_status -- synchronise `stream`, then read and clear this
 * library's device status word on the current device. Returns LA_OK, or
 * LA_ERR_TIMEOUT if a kernel launched since the last call gave up on a
 * bounded device-side wait (it then skipped its remaining work and released
 * its resources; its outputs are undefined), or LA_ERR_CUDA.
 */
int la_stream_status(la_stream_t stream);

/* Message for the last error on the calling thread ("" if none). */
const char *la_last_error(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int la_version(void);

#ifdef __cplusplus
}
#endif
#endif /* LA_H */
