/*
 * efla.h -- C ABI of libefla.so, the GB300 (sm_103a) implementation of the
 * Error-Free Linear Attention (EFLA) token mixer.
 *
 * The operation (per head; notation of the pages that describe the method):
 *
 *   lambda_t = ||k_t||^2
 *   alpha_t  = (1 - exp(-beta_t lambda_t)) / lambda_t      (beta_t when lambda_t == 0)
 *   S_t      = (I - alpha_t k_t k_t^T) S_{t-1} + alpha_t k_t v_t^T
 *   o_t      = S_t^T q_t                                     (reads the UPDATED state)
 *
 *   ["Exact Flow Linear Attention: Exact Solution from Continuous-Time Dynamics"
 *    (gist.science summary), Metodologia 2-3;
 *    "Error-Free Linear Attention is a Free Lunch: Exact Solution from
 *    Continuous-Time Dynamics" (howistudyai explainer), Steps 1-3 and
 *    "Putting it all together (pipeline)".]
 *
 * No scaling of q and no normalisation of q or k is applied: the key norm is
 * the gate's input (howistudyai, "Key Norms as Dynamic Gates").
 *
 * Conventions shared by every entry point
 *   - All tensor arguments are DEVICE pointers to contiguous row-major arrays
 *     owned by the caller.  The library allocates no device memory per call.
 *   - Every call is asynchronous on `stream` (NULL = legacy default stream)
 *     and never synchronises the host.
 *   - Arguments are validated on the host before anything is launched.  A
 *     rejected call returns EFLA_ERR_INVALID_ARG or EFLA_ERR_UNSUPPORTED and
 *     launches nothing.  Launch failures return EFLA_ERR_CUDA.
 *   - Kernels that wait on other warps bound every wait; if a bound expires
 *     the kernel abandons its work, records EFLA_ERR_DEVICE_TIMEOUT in a
 *     library-owned device status word and returns.  efla_device_status()
 *     reads and clears that word.
 *   - Pointers must be 16-byte aligned.  Outputs must not alias inputs, except
 *     that S0 == S_T is allowed (each unit reads its S0 before writing S_T).
 *   - efla_last_error() gives a human-readable reason for the most recent
 *     failing call on the calling host thread.
 */
#ifndef EFLA_H
#define EFLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define EFLA_ABI_VERSION 10

typedef enum {
    EFLA_OK = 0,
    EFLA_ERR_INVALID_ARG = 1,     /* null/misaligned pointer, bad size, bad cu_seqlens shape */
    EFLA_ERR_UNSUPPORTED = 2,     /* valid but not implemented (e.g. d_k not in {32,64,128}) */
    EFLA_ERR_CUDA = 3,            /* a CUDA runtime/driver call or a launch failed */
    EFLA_ERR_DEVICE_TIMEOUT = 4   /* a bounded in-kernel wait expired (device status word) */
} efla_status;

typedef enum {
    EFLA_BF16 = 0,
    EFLA_F32 = 1
} efla_dtype;

/* The gate of the rank-1 update.
 *   EFLA_UPDATE_EXACT: alpha = (1 - exp(-beta lambda)) / lambda, the exact solution of
 *     the zero-order-hold ODE over the token window (the method itself).
 *   EFLA_UPDATE_EULER: alpha = beta, the explicit-Euler (delta rule, DeltaNet) step
 *     that the pages compare EFLA against ("Error-Free Linear Attention is a Free
 *     Lunch" (howistudyai), "Delta Rule (Linear Attention as Online Learning)").
 *     Same kernels, same layouts; provided for side-by-side measurement. */
typedef enum {
    EFLA_UPDATE_EXACT = 0,
    EFLA_UPDATE_EULER = 1
} efla_update;

/* Same object as cudaStream_t; kept opaque so that this header needs no CUDA header. */
typedef struct CUstream_st *efla_stream_t;

/*
 * efla_fwd_chunked -- EFLA forward over whole sequences, chunkwise (WY/UT form).
 *
 * Defined by: the update rule and read-out above, evaluated in chunks of
 * `chunk` tokens with the WY/UT representation of the products of rank-1
 * updates ("Exact Flow Linear Attention" (gist.science), Metodologia 3;
 * "Error-Free Linear Attention is a Free Lunch" (howistudyai), Step 4).
 * The result equals the token-by-token recurrence up to rounding.
 *
 *   q, k     [B, T, H, d_k]  dtype
 *   v        [B, T, H, d_v]  dtype
 *   beta     [B, T, H]       fp32, the per-token step size beta_t (any finite value)
 *   S0       [N, H, d_k, d_v] fp32 (d_v contiguous) initial states, or NULL for zeros
 *   cu_seqlens [N+1] int32 DEVICE array, or NULL.
 *            NULL: N must equal B; sequence b is row b, length T.
 *            non-NULL: B must be 1; sequence n covers packed tokens
 *            cu_seqlens[n] .. cu_seqlens[n+1]-1 of T; cu_seqlens[0] = 0,
 *            cu_seqlens[N] = T, non-decreasing.  It is not read on the host:
 *            a kernel that meets a sequence with bounds outside [0, T] or
 *            decreasing writes nothing for that sequence and records
 *            EFLA_ERR_INVALID_ARG in the device status word (the outputs of
 *            sequences whose ranges overlap are then unspecified).  Sequences
 *            are independent.
 *   o        [B, T, H, d_v]  dtype (the dtype of q); every token row written
 *   S_T      [N, H, d_k, d_v] fp32 final states, or NULL (not written)
 *   dtype    EFLA_BF16 or EFLA_F32, the element type of q, k, v and o
 *   chunk    chunk length: 16, 32 or 64 (0 selects 64); 128 returns
 *            EFLA_ERR_UNSUPPORTED (the chunk's fp32 buffers would not fit one
 *            CTA's shared memory)
 *
 * State and all accumulation are fp32.  Supported: d_k, d_v in {32, 64, 128}.
 * bf16 inputs with d_k = d_v = 128 and chunk 64 run on the tcgen05
 * tensor-core chunk kernel; every other supported combination runs the
 * chunkwise evaluation on CUDA cores in fp32.  T = 0 or N = 0 is valid
 * (S_T = S0, or zeros, is written).  efla_fwd_chunked_ex below takes an
 * explicit output dtype (an fp32 o for bf16 inputs) and update rule.
 */
efla_status efla_fwd_chunked(const void *q, const void *k, const void *v, const float *beta,
                             const float *S0, const int32_t *cu_seqlens, void *o, float *S_T,
                             int B, int T, int H, int d_k, int d_v, int N,
                             efla_dtype dtype, int chunk, efla_stream_t stream);

/*
 * efla_fwd_recurrent -- the same forward, evaluated token by token on CUDA
 * cores in fp32 (howistudyai, "Putting it all together (pipeline)": for each
 * token compute lambda and alpha, update S, emit o).  Same arguments and
 * layouts as efla_fwd_chunked without `chunk` (o in the dtype of q).  An
 * independent GPU evaluation of the recurrence.
 */
efla_status efla_fwd_recurrent(const void *q, const void *k, const void *v, const float *beta,
                               const float *S0, const int32_t *cu_seqlens, void *o, float *S_T,
                               int B, int T, int H, int d_k, int d_v, int N,
                               efla_dtype dtype, efla_stream_t stream);

/*
 * efla_decode_step -- one token per sequence, state updated IN PLACE.
 *
 * Defined by: one application of the update rule and read-out above
 * ("Exact Flow Linear Attention" (gist.science), Metodologia 3;
 *  "Error-Free Linear Attention is a Free Lunch" (howistudyai), Steps 1-3).
 * Evaluated in one pass over S using o = S^T q + (q.k) u with
 * u = alpha (v - S^T k), which equals S_t^T q after S_t = S + k u^T.
 *
 *   q, k  [B, H, d_k] dtype;  v [B, H, d_v] dtype;  beta [B, H] fp32
 *   S     [B, H, d_k, d_v] fp32, read and overwritten with the new state
 *   o     [B, H, d_v] dtype
 * Supported: d_k, d_v in {32, 64, 128}.  efla_decode_step_ex takes an explicit
 * output dtype and update rule.
 */
efla_status efla_decode_step(const void *q, const void *k, const void *v, const float *beta,
                             float *S, void *o, int B, int H, int d_k, int d_v,
                             efla_dtype dtype, efla_stream_t stream);

/*
 * efla_fwd_chunked_scan -- efla_fwd_chunked for few long sequences, split along time.
 *
 * Same operation and layouts as efla_fwd_chunked with cu_seqlens = NULL (N = B).
 * Over any stretch of tokens the update rule is affine in the start state,
 * S_out = M S_in + N ("Exact Flow Linear Attention" (gist.science), Metodologia 3,
 * applied token after token), so each sequence is cut into `segments` pieces at
 * chunk boundaries and evaluated in three launches: the maps (M, N) of every
 * piece but the last, all pieces in parallel; the start state of every piece by
 * a serial scan over the maps; then every piece from its start state, with
 * outputs.  The result equals the unsplit forward up to rounding; it trades
 * about three times the arithmetic for `segments` times the parallelism, which
 * pays when B*H is well below the SM count.
 *
 *   segments   pieces per sequence; 0 = SM count / (B*H).  Capped at the chunk count.
 *   workspace  device scratch owned by the caller, 16-byte aligned, at least the size
 *              efla_fwd_scan_workspace reports (0 bytes when one piece results);
 *              must not overlap any argument; its contents on return are unspecified.
 * Only bf16 inputs with d_k = d_v = 128 are split; other shapes, and a single
 * piece, run the plain efla_fwd_chunked path (the workspace is then unused).
 */
efla_status efla_fwd_chunked_scan(const void *q, const void *k, const void *v, const float *beta,
                                  const float *S0, void *o, float *S_T, int B, int T, int H,
                                  int d_k, int d_v, efla_dtype in_dtype, efla_dtype o_dtype,
                                  int segments, void *workspace, size_t workspace_bytes,
                                  efla_update update, efla_stream_t stream);

/* Workspace bytes efla_fwd_chunked_scan needs for these sizes, and the number of
 * pieces it will use (segments_used may be NULL).  segments = 0 queries the
 * current device's SM count. */
efla_status efla_fwd_scan_workspace(int B, int T, int H, int d_k, int d_v, int segments,
                                    size_t *bytes, int *segments_used);

/*
 * efla_fwd_chunked_scan_static -- efla_fwd_chunked_scan with library-owned scratch.
 *
 * The pages have no counterpart to this call: it is the same operation as
 * efla_fwd_chunked_scan (same arguments without workspace/workspace_bytes) for
 * callers that cannot provide device memory.  The scratch is a fixed 32 MiB device
 * array inside libefla.so (allocated when the module loads; this call allocates
 * nothing), enough for any automatic split (segments = 0) on GPUs of up to 170
 * SMs.  A split that needs more returns EFLA_ERR_UNSUPPORTED before any launch.
 * Nothing in the scratch has to start at zero, so it is never cleared.
 * The scratch is shared by every call in the process on the same device: calls
 * that may overlap in time (other streams, other host threads) race on it and
 * give wrong results; serialise them, or use efla_fwd_chunked_scan.
 */
efla_status efla_fwd_chunked_scan_static(const void *q, const void *k, const void *v, const float *beta,
                                         const float *S0, void *o, float *S_T, int B, int T, int H,
                                         int d_k, int d_v, efla_dtype in_dtype, efla_dtype o_dtype,
                                         int segments, efla_update update, efla_stream_t stream);

/*
 * efla_bwd_recurrent -- gradients of efla_fwd_chunked (cu_seqlens = NULL, N = B).
 *
 * Given dO = dL/do and dS_T = dL/dS_T, returns dq, dk, dv, dbeta and dS0 of any loss L
 * of the forward's outputs.  The pages give no backward formulas: this is reverse
 * mode of the update rule and read-out above ("Exact Flow Linear Attention"
 * (gist.science), Metodologia 3; "Error-Free Linear Attention is a Free Lunch"
 * (howistudyai), Steps 1-3), evaluated token by token in reverse order in fp32 on CUDA
 * cores (one CTA per (b, h); a forward sweep first recomputes the states).
 *
 *   q, k [B, T, H, d_k], v [B, T, H, d_v] in_dtype;  beta [B, T, H] fp32
 *   S0, dS_T [B, H, d_k, d_v] fp32 or NULL (zero)
 *   dO   [B, T, H, d_v] fp32
 *   dq, dk [B, T, H, d_k], dv [B, T, H, d_v], dbeta [B, T, H] fp32 outputs;
 *   dS0 [B, H, d_k, d_v] fp32 or NULL (not written)
 *   update  the gate of the forward (EFLA_UPDATE_EXACT or EFLA_UPDATE_EULER)
 * Outputs must not overlap inputs or each other.  Supported: d_k, d_v in {32, 64, 128}.
 */
efla_status efla_bwd_recurrent(const void *q, const void *k, const void *v, const float *beta,
                               const float *S0, const float *dO, const float *dS_T, float *dq,
                               float *dk, float *dv, float *dbeta, float *dS0, int B, int T, int H,
                               int d_k, int d_v, efla_dtype in_dtype, efla_update update,
                               efla_stream_t stream);

/*
 * efla_bwd_chunked -- the gradients of efla_bwd_recurrent, evaluated in chunks of 64 tokens.
 *
 * Same arguments, layouts, outputs and rules as efla_bwd_recurrent, plus a workspace.  The
 * pages give no backward formulas: this is reverse mode of the chunkwise (WY/UT) form of the
 * forward ("Error-Free Linear Attention is a Free Lunch" (howistudyai), Step 4 "Chunkwise
 * Parallelism"; "Exact Flow Linear Attention" (gist.science), Metodologia 3).  Three steps
 * on `stream`: the forward, writing the state at the start of every chunk into the
 * workspace; one CTA per (b, h) that walks the chunks in reverse for the gradient of each
 * chunk's end state (also into the workspace); then the (b, h, chunk) items, all
 * independent, for every token's gradients (fp32 on CUDA cores).  For bf16 inputs with
 * d = 128 all three steps run on the tensor cores (split-bf16 operands, fp32 accumulation;
 * the last on persistent CTAs), after a pass that writes dO as bf16 hi and lo parts into the
 * workspace; the first also writes every chunk's T'' there, the second G and -dR (bf16 hi and
 * lo) of every token.
 *
 *   workspace  device scratch owned by the caller, 16-byte aligned, at least the size
 *              efla_bwd_workspace reports (B x H x ceil(T/64) x (2 d_k d_v + 4096) x 4 bytes
 *              + B x T x H x d_v x 12 bytes);
 *              it must not overlap any argument.  Too small or NULL: EFLA_ERR_INVALID_ARG.
 * Supported: d_k = d_v in {64, 128} (other sizes: EFLA_ERR_UNSUPPORTED, use
 * efla_bwd_recurrent).
 */
efla_status efla_bwd_chunked(const void *q, const void *k, const void *v, const float *beta,
                             const float *S0, const float *dO, const float *dS_T, float *dq,
                             float *dk, float *dv, float *dbeta, float *dS0, int B, int T, int H,
                             int d_k, int d_v, efla_dtype in_dtype, efla_update update,
                             void *workspace, size_t workspace_bytes, efla_stream_t stream);

/* Workspace bytes efla_bwd_chunked needs for these sizes (into *bytes). */
efla_status efla_bwd_workspace(int B, int T, int H, int d_k, int d_v, size_t *bytes);

/*
 * efla_fwd_chunked_train -- efla_fwd_chunked (rows of [B, T], no cu_seqlens, o in q's dtype,
 * chunk 64) that also keeps what the chunked backward would otherwise recompute: the state at
 * the start of every chunk (and, for bf16 with d = 128, every chunk's T'') go into `workspace`,
 * laid out as efla_bwd_chunked lays them out.  A later efla_bwd_chunked_saved with the same
 * inputs and that workspace then skips its forward.  The reverse mode of training: the forward
 * keeps its activations for the backward ("Error-Free Linear Attention is a Free Lunch"
 * (howistudyai), Step 4 "Chunkwise Parallelism").
 *   workspace  device scratch owned by the caller, 16-byte aligned, at least the size
 *              efla_bwd_workspace reports; it must not overlap any argument.
 * Supported: d_k = d_v in {64, 128}.  Errors as efla_fwd_chunked and efla_bwd_chunked.
 */
efla_status efla_fwd_chunked_train(const void *q, const void *k, const void *v, const float *beta,
                                   const float *S0, void *o, float *S_T, int B, int T, int H, int d_k,
                                   int d_v, efla_dtype in_dtype, efla_update update, void *workspace,
                                   size_t workspace_bytes, efla_stream_t stream);

/*
 * efla_bwd_chunked_saved -- efla_bwd_chunked on a workspace that efla_fwd_chunked_train filled
 * for the same q, k, v, beta, S0, sizes, dtype and update rule, without running the forward
 * again; the same arguments, outputs and rules.  That the workspace matches the inputs is the
 * caller's contract and is not checked: other contents give unspecified gradients (every access
 * still stays inside the workspace).
 */
efla_status efla_bwd_chunked_saved(const void *q, const void *k, const void *v, const float *beta,
                                   const float *S0, const float *dO, const float *dS_T, float *dq,
                                   float *dk, float *dv, float *dbeta, float *dS0, int B, int T, int H,
                                   int d_k, int d_v, efla_dtype in_dtype, efla_update update,
                                   void *workspace, size_t workspace_bytes, efla_stream_t stream);

/*
 * efla_decode_tokens -- m tokens per sequence appended to a resident state,
 * S updated IN PLACE (multi-token decode, prefill continuation).
 *
 * Defined by: m applications, in token order, of the update rule and read-out
 * above ("Exact Flow Linear Attention" (gist.science), Metodologia 3;
 * "Error-Free Linear Attention is a Free Lunch" (howistudyai), Steps 1-3 and
 * "Putting it all together (pipeline)"); equal to m successive
 * efla_decode_step calls, with S read and written once.
 *
 *   q, k  [B, m, H, d_k] in_dtype;  v [B, m, H, d_v] in_dtype;  beta [B, m, H] fp32
 *   S     [B, H, d_k, d_v] fp32, read and overwritten with the state after token m
 *   o     [B, m, H, d_v] o_dtype
 *   update  EFLA_UPDATE_EXACT or EFLA_UPDATE_EULER
 * m = 0 or B = 0 is valid and changes nothing.  Supported: d_k, d_v in {32, 64, 128}.
 * S must not overlap any input or o; o must not overlap any input.
 */
efla_status efla_decode_tokens(const void *q, const void *k, const void *v, const float *beta,
                               float *S, void *o, int B, int m, int H, int d_k, int d_v,
                               efla_dtype in_dtype, efla_dtype o_dtype, efla_update update,
                               efla_stream_t stream);

/*
 * The three calls above with an explicit output dtype (o_dtype: EFLA_F32 gives
 * an fp32 o for bf16 inputs, free of the output's own bf16 rounding) and an
 * explicit update rule (efla_update).  The versions without the suffix use
 * o_dtype = in_dtype and EFLA_UPDATE_EXACT.  An unknown rule or dtype returns
 * EFLA_ERR_INVALID_ARG.
 */
efla_status efla_fwd_chunked_ex(const void *q, const void *k, const void *v, const float *beta,
                                const float *S0, const int32_t *cu_seqlens, void *o, float *S_T,
                                int B, int T, int H, int d_k, int d_v, int N,
                                efla_dtype in_dtype, efla_dtype o_dtype, int chunk,
                                efla_update update, efla_stream_t stream);
efla_status efla_fwd_recurrent_ex(const void *q, const void *k, const void *v, const float *beta,
                                  const float *S0, const int32_t *cu_seqlens, void *o, float *S_T,
                                  int B, int T, int H, int d_k, int d_v, int N,
                                  efla_dtype in_dtype, efla_dtype o_dtype, efla_update update,
                                  efla_stream_t stream);
efla_status efla_decode_step_ex(const void *q, const void *k, const void *v, const float *beta,
                                float *S, void *o, int B, int H, int d_k, int d_v,
                                efla_dtype in_dtype, efla_dtype o_dtype, efla_update update,
                                efla_stream_t stream);

/*
 * efla_prep -- the per-token quantities of the update, for n token-head rows.
 *
 * Defined by: lambda = ||k||^2 ("Exact Flow Linear Attention" (gist.science),
 * Metodologia 2) and the gate alpha (efla_update; exact: (1 - exp(-beta lambda))
 * / lambda, beta at lambda = 0; Metodologia 3 and howistudyai Step 1), and the
 * two gate-scaled factors of the rank-1 write alpha k v^T.
 *
 *   k     [n, d_k] dtype; v [n, d_v] dtype (may be NULL unless av is requested)
 *   beta  [n] fp32
 *   lam   [n] fp32 out, or NULL      alpha [n] fp32 out, or NULL
 *   ak    [n, d_k] dtype out = alpha k, or NULL
 *   av    [n, d_v] dtype out = alpha v, or NULL
 * A [B, T, H, d] activation tensor is n = B*T*H rows.  Supported d_k, d_v in
 * {32, 64, 128}; dtype EFLA_BF16 or EFLA_F32 (fp32 arithmetic either way).
 */
efla_status efla_prep(const void *k, const void *v, const float *beta, float *lam, float *alpha,
                      void *ak, void *av, long long n, int d_k, int d_v, efla_dtype dtype,
                      efla_update update, efla_stream_t stream);

/* Reads the calling thread's current device's status word on `stream`
 * (synchronising that stream), resets it to EFLA_OK and returns what it held:
 * EFLA_ERR_DEVICE_TIMEOUT after a bounded in-kernel wait expired, or
 * EFLA_ERR_INVALID_ARG after a kernel met malformed cu_seqlens.  Each device
 * has its own word. */
efla_status efla_device_status(efla_stream_t stream);

/* Static description of a status code; never NULL. */
const char *efla_get_error_string(efla_status status);

/* Test hook: the bound, in nanoseconds, on each wait of the tensor-core chunk
 * kernel between its warp roles (0 restores the default of 2 s).  Applies to
 * launches made after the call, from any host thread.  The waits that let a
 * kernel's own copies and tensor-core operations finish before it releases
 * tensor memory keep their 2 s bound whatever this is set to. */
void efla_debug_set_wait_limit_ns(unsigned long long ns);

/* Test hook: stall is a set of bits, each naming a tensor-core kernel: 1 the chunk
 * kernel (the forward, also the first step of efla_bwd_chunked), 2 the backward's
 * state pass, 4 the backward's per-chunk gradient kernel.  Each launch of a named
 * kernel made after the call has its tensor-core issuing thread first wait on a
 * barrier that nothing completes.  That wait runs out after the wait limit above;
 * the kernel then abandons its work, lets its own copies and tensor-core
 * operations finish, records EFLA_ERR_DEVICE_TIMEOUT in the status word and
 * returns (its outputs are unspecified).  This exercises the bounded-wait path
 * without any fault.  stall = 0 (the default) restores normal launches. */
void efla_debug_set_stall(int stall);

/* Reason for the most recent failing call on this host thread ("" if none). */
const char *efla_last_error(void);

/* EFLA_ABI_VERSION of the loaded library. */
int efla_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* EFLA_H */
