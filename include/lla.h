/*
 * lla.h -- C ABI of liblla.so: log-linear attention (Log-Linear Mamba-2 form)
 * on one NVIDIA GB300 GPU (sm_103a).
 *
 * The operator (page "Log-Linear Attention", gist.science 2506.04761,
 * technical summary §2.2 output equation, with the scalar-gate Mamba-2
 * instance of §3), for every batch b, head h and token t:
 *
 *     o_t = sum_{s <= t} lambda_t[l(t,s)] * exp(G_t - G_s) * (q_t . k_s) * v_s
 *
 *     G_t    = g_0 + ... + g_t          (inclusive running sum of the gates)
 *     l(t,s) = bit_length(t XOR s)       (0 when s == t; otherwise the
 *                                         Fenwick-tree bucket of [0,t) that
 *                                         holds s, 2^(l-1) keys per bucket)
 *     L      = 1 + bit_length(T - 1)     (lambda entries per token)
 *
 * Positions are 0-based.  Gates are log-decays, g <= 0 in the intended use
 * (the library does not require it).  Lambda entries at levels with no
 * bucket for a given t multiply an empty sum and are ignored.
 *
 * Conventions for every entry point:
 *   - Tensor pointers are DEVICE pointers to caller-owned memory, densely
 *     packed (C-contiguous) in the layout given, 16-byte aligned.  The
 *     library keeps no pointer after a call returns and allocates no device
 *     memory.  Scratch memory is a caller-provided workspace, sized by the
 *     matching *_workspace_bytes query.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call is asynchronous and stream-ordered: it enqueues
 *     kernels and returns without synchronising the host.
 *   - Arguments are validated before anything is enqueued.  A validation
 *     failure returns an error and enqueues nothing.  LLA_ERR_CUDA means a
 *     launch was rejected by the CUDA runtime (the runtime's last error is
 *     left for the caller to inspect with cudaGetLastError).
 *   - The current CUDA device must be the device that owns the pointers.
 *   - Errors found while the kernels run.  The tensor-core kernels hand work
 *     between warps and copy engines through shared-memory barriers; every
 *     wait on one is bounded (about half a second).  A wait that runs out
 *     records an lla_device_error code and the kernel carries on to its end
 *     (every later wait is bounded too), so the GPU never hangs; the output
 *     of that call is then invalid.  Entry points with such waits
 *     take `int32_t *device_error`: NULL, or one int32 of device memory owned
 *     by the caller that the kernels set (atomically, first code wins) and
 *     never clear.  Zero it before the calls it should cover and read it
 *     with lla_device_error_check once they are done.
 */
#ifndef LLA_H
#define LLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LLA_F32 = 0,  /* IEEE binary32                              */
    LLA_BF16 = 1  /* bfloat16 (8-bit exponent, 7-bit mantissa)  */
} lla_dtype;

typedef enum {
    LLA_OK = 0,
    LLA_ERR_INVALID_ARGUMENT = 1,    /* null pointer, negative size, bad enum     */
    LLA_ERR_UNSUPPORTED_SHAPE = 2,   /* a size outside the supported set          */
    LLA_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes < the query's answer       */
    LLA_ERR_CUDA = 4,                /* a kernel launch failed                     */
    LLA_ERR_DEVICE_REPORTED = 5      /* a kernel recorded an error (device_error) */
} lla_status;

/* Codes the kernels store in a caller's device_error word (forward, backward,
 * prefill, lambda producer; the decode steps store 1 + b instead, see there). */
typedef enum {
    LLA_DEVERR_NONE = 0,
    LLA_DEVERR_COPY_TIMEOUT = 1,  /* a bulk copy into shared memory did not land in time     */
    LLA_DEVERR_SYNC_TIMEOUT = 2   /* a tensor-core product or a warp hand-off did not finish */
} lla_device_error;

/* Human-readable name of a status code (static storage, never NULL). */
const char *lla_status_string(lla_status s);

/* Library version as 10000*major + 100*minor + patch. */
int lla_version(void);

/* Reads a device_error word after the work it covers: synchronises `stream`,
 * copies the int32 at device address device_error to the host and returns
 * LLA_OK when it is 0, LLA_ERR_DEVICE_REPORTED otherwise (the code is stored
 * in *code when code is non-NULL).  The word is left as it is.  NULL
 * device_error: LLA_ERR_INVALID_ARGUMENT; a failed copy: LLA_ERR_CUDA.
 * This is the one call of the library that blocks the host. */
lla_status lla_device_error_check(const int32_t *device_error, int32_t *code, void *stream);

/* Test hook for the reporting path above (the pages have no counterpart).
 * While enabled (nonzero), every tensor-core forward launch withholds the
 * first product of each tile (the intra-tile Q K^T: neither the product nor
 * its completion signal is issued, so no copy or product is left in flight)
 * and bounds the waits on that product at a few thousand polls: they run
 * out, LLA_DEVERR_SYNC_TIMEOUT is recorded and the launch finishes with an
 * invalid output.  Process-wide; 0 restores normal operation. */
void lla_debug_withhold_first_product(int enable);

/* L = 1 + bit_length(T-1): lambda entries per token for a length-T forward
 * (level 0 plus the Fenwick levels of the longest prefix).  0 for T <= 0. */
int lla_num_levels(int T);

/*
 * Chunked O(T log T) forward ("Log-Linear Attention" §2.3: the hierarchical
 * mask trained in parallel, matmul-rich).  The sequence is cut into chunks of
 * `chunk` tokens; within a chunk the masked product (Q K^T . M) V is formed
 * directly, and every earlier chunk is reached through the chunk-level
 * Fenwick-tree states of §2.2, each weighted per token by its lambda.  The
 * result does not depend on `chunk` beyond rounding.
 *
 *   q      [B,H,T,dk]  in_dt       k [B,H,T,dk] in_dt      v [B,H,T,dv] in_dt
 *   g      [B,H,T]     fp32        per-token log-gate
 *   lambda [B,H,T,L]   fp32        L = lla_num_levels(T)
 *   out    [B,H,T,dv]  out_dt      fully overwritten
 *
 * Supported: B,H >= 0; T >= 0 with T % chunk == 0 and T <= 2^24;
 * chunk in {16,32,64,128}; dk, dv in {16,32,64,128};
 * (in_dt, out_dt) in {(F32,F32), (BF16,F32), (BF16,BF16)}.
 * B*H*T == 0 is a valid no-op.  Other shapes: LLA_ERR_UNSUPPORTED_SHAPE.
 * workspace: device memory of at least lla_fwd_workspace_bytes(...) bytes,
 * 256-byte aligned; its contents on entry do not matter and are undefined on
 * return.  Calls that share a workspace must not overlap on the GPU.
 * q, k, v, g, lambda are read only; out must not alias an input.
 * device_error: NULL or a caller-owned device int32 (see the conventions
 * above); the tensor-core path (bf16, dk = dv = 128) may set it to
 * LLA_DEVERR_COPY_TIMEOUT or LLA_DEVERR_SYNC_TIMEOUT; the CUDA-core path has
 * no waits and never writes it.
 */
size_t lla_fwd_workspace_bytes(int B, int H, int T, int dk, int dv, int chunk,
                               lla_dtype in_dt);

/* Number of kernel launches (memsets included) one lla_fwd call with these
 * arguments enqueues on its stream; 0 for an empty or unsupported call. */
int lla_fwd_launches(int B, int H, int T, int dk, int dv, int chunk, lla_dtype in_dt,
                     lla_dtype out_dt);

lla_status lla_fwd(const void *q, const void *k, const void *v,
                   const float *g, const float *lambda, void *out,
                   int B, int H, int T, int dk, int dv, int chunk,
                   lla_dtype in_dt, lla_dtype out_dt,
                   void *workspace, size_t workspace_bytes, int32_t *device_error,
                   void *stream);

/*
 * lla_fwd for callers that cannot allocate device memory.  The pages have
 * no counterpart to this entry point; it exists for code that must not call
 * cudaMalloc where it runs the forward (inside an allocator or memory-pool
 * callback, a plugin handed only its input and output buffers, a runtime
 * that forbids allocation while it records or replays work).
 * Same arguments, layouts and results as lla_fwd, without the workspace:
 * the scratch is one fixed array of lla_fwd_noalloc_max_scratch_bytes()
 * bytes (64 MiB) compiled into the library, present on every GPU that loads
 * it until the process exits.  Arguments are checked in lla_fwd's order
 * (shape and dtype, pointers and alignment, the stream's device); then a
 * call that needs more scratch than the array holds
 * (lla_fwd_workspace_bytes(...) > the maximum) returns
 * LLA_ERR_WORKSPACE_TOO_SMALL.  Nothing is enqueued on any error.
 * `stream` must belong to the current device (LLA_ERR_INVALID_ARGUMENT
 * otherwise): the array's address is looked up per device.  The first call
 * on a device looks that address up with the device current; make it before
 * any stream capture.  A failed look-up returns LLA_ERR_CUDA and is tried
 * again by the next call.  All calls share the array: calls that may
 * overlap on the GPU race and must be ordered by the caller.  The library
 * allocates nothing and nothing needs clearing between calls.
 */
size_t lla_fwd_noalloc_max_scratch_bytes(void);

lla_status lla_fwd_noalloc(const void *q, const void *k, const void *v,
                           const float *g, const float *lambda, void *out,
                           int B, int H, int T, int dk, int dv, int chunk,
                           lla_dtype in_dt, lla_dtype out_dt, int32_t *device_error,
                           void *stream);

/*
 * lla_fwd with lambda produced by the two-layer MLP of "Adaptive memory decay
 * for Log-Linear Attention" (§Method, LambdaMLPSoftplus) instead of passed in:
 *     lambda_t = softplus((d_t W1) W2 + b),   width 2L hidden, L = lla_num_levels(T),
 * then out = lla_fwd(q, k, v, g, lambda).  The same MLP as lla_lambda_mlp.
 *   d  [B,H,T,Dd] in_dt     W1 [Dd,2L], W2 [2L,L], b [L] fp32 (shared by heads)
 * Other arguments, layouts and errors as lla_fwd and lla_lambda_mlp.
 * When d is the key tensor itself (d == k, Dd == dk) on the tensor-core
 * shapes (bf16, dk = dv in {64,128}) with 2L <= 32 (T <= 32768), lambda is
 * computed inside the read-out, from the key tile it already holds in shared
 * memory (the first layer on the tensor cores with W1 split into two bf16
 * parts, the second layer and softplus in fp32), and never goes to device
 * memory.  Any other call runs lla_lambda_mlp into the workspace and then
 * lla_fwd (the same results up to rounding, two passes over lambda).
 * workspace: at least lla_fwd_lambda_mlp_workspace_bytes(...) bytes, enough
 * for either way.
 */
size_t lla_fwd_lambda_mlp_workspace_bytes(int B, int H, int T, int dk, int dv, int Dd,
                                          int chunk, lla_dtype in_dt);

lla_status lla_fwd_lambda_mlp(const void *q, const void *k, const void *v, const float *g,
                              const void *d, const float *W1, const float *W2,
                              const float *b, void *out, int B, int H, int T, int dk, int dv,
                              int Dd, int chunk, lla_dtype in_dt, lla_dtype out_dt,
                              void *workspace, size_t workspace_bytes,
                              int32_t *device_error, void *stream);

/*
 * Decode state (the recurrent form of "Log-Linear Attention" §2.3: O(log T)
 * states, each step reads and updates O(log T) of them).  For one (b,h) at
 * token index t the state holds the Fenwick buckets of the prefix [0,t):
 *   state_levels   [B,H,Ls,dk,dv] fp32: slot i holds level i+1;
 *   state_logdecay [B,H,Ls]       fp32: the level's true state is
 *                                 exp(state_logdecay) * state_levels.
 * Slot i is live iff bit i of t is set; dead slots are never read.  A zeroed
 * state is the state of the empty prefix (t = 0).
 * lla_decode_state_bytes returns the size of state_levels in bytes.
 */
size_t lla_decode_state_bytes(int B, int H, int dk, int dv, int Ls);

/*
 * One decode step for B sequences x H heads; sequence b is at token index
 * t = pos[b] (the state holds [0,t) and this call consumes token t):
 *   1. logdecay += g for the live slots;
 *   2. out = lambda[0] (q.k) v + sum_{live l} lambda[l] exp(logdecay_l) q^T S_l;
 *   3. with m = trailing zeros of t+1, slot m (level m+1) becomes
 *      k v^T + sum_{l=1..m} exp(logdecay_l) S_l with logdecay 0; slots
 *      0..m-1 become dead (they are not cleared).
 *   q, k [B,H,dk] in_dt; v [B,H,dv] in_dt; g [B,H] fp32;
 *   lambda [B,H,Ls+1] fp32 (levels 0..Ls); out [B,H,dv] fp32;
 *   pos [B] int64 on the device, read by the kernel (the caller advances it).
 * Supported: dk, dv in {16,32,64,128}; 1 <= Ls <= 40; in_dt F32 or BF16.
 * A sequence with pos < 0 or bit_length(pos+1) > Ls is skipped (its out and
 * state are left untouched) and, if device_error is non-NULL, the kernel
 * stores 1 + b into *device_error (one of the offending b when several).
 * The live slots stream into shared memory by bulk copies whose waits are
 * bounded; one that runs out stores -1 (if nothing was stored before) and
 * that step's output is invalid.  The kernel never traps.  device_error is device memory owned by the caller;
 * the library only ever writes a nonzero value into it.
 */
lla_status lla_decode_step(float *state_levels, float *state_logdecay,
                           const void *q, const void *k, const void *v,
                           const float *g, const float *lambda, float *out,
                           const int64_t *pos, int B, int H, int dk, int dv,
                           int Ls, lla_dtype in_dt, int32_t *device_error,
                           void *stream);

/*
 * Prefill -> decode hand-off: the decode state after the prefix [0,T), i.e.
 * for the next token index t = T, computed from the bucket definition of
 * "Log-Linear Attention" §2.2:
 *   S_l = sum_{s<T, l(T,s)=l} exp(G_{T-1} - G_s) k_s v_s^T,   logdecay_l = 0,
 * and dead slots zeroed.  k [B,H,T,dk], v [B,H,T,dv] in_dt; g [B,H,T] fp32;
 * state_levels [B,H,Ls,dk,dv] fp32 and state_logdecay [B,H,Ls] fp32 are
 * fully overwritten.  Requires bit_length(T) <= Ls <= 40, T <= 2^30.
 * workspace: at least lla_prefill_workspace_bytes(B,H,T) bytes.
 * device_error: NULL or a caller-owned device int32, set by the tensor-core
 * path (bf16, dk = dv = 128) as for lla_fwd.
 */
size_t lla_prefill_workspace_bytes(int B, int H, int T);

lla_status lla_prefill_state(const void *k, const void *v, const float *g,
                             float *state_levels, float *state_logdecay,
                             int B, int H, int T, int dk, int dv, int Ls,
                             lla_dtype in_dt, void *workspace,
                             size_t workspace_bytes, int32_t *device_error, void *stream);

/*
 * lla_fwd on inputs and outputs in host memory (same layouts and dtypes as
 * lla_fwd, host pointers; pin them for asynchronous copies).  The pages have
 * no counterpart: this is the host-facing call of the library.  The
 * (batch, head) pairs are processed in groups of at most `group` pairs (0:
 * about an eighth of them; the first and the last group hold half as many,
 * which shortens the copies that cannot overlap), pipelined over two device
 * slots so that copying group
 * j+1 in, computing group j and copying group j-1 out overlap (two internal
 * streams, created on the first call on a device and kept until exit).
 * Ordered on `stream`: earlier work on it completes before the first copy,
 * and the stream waits for the last copy out, so synchronising the stream
 * makes the host output valid.  Results are identical to lla_fwd.
 * workspace: device memory of at least lla_fwd_host_workspace_bytes(...)
 * bytes (two slots of group-sized copies plus the forward's workspace),
 * 256-byte aligned.  Errors as lla_fwd, all before the first copy;
 * device_error (device memory, nullable) as for lla_fwd, covering every group.
 */
size_t lla_fwd_host_workspace_bytes(int B, int H, int T, int dk, int dv, int chunk,
                                    lla_dtype in_dt, lla_dtype out_dt, int group);

lla_status lla_fwd_host(const void *q, const void *k, const void *v, const float *g,
                        const float *lambda, void *out, int B, int H, int T, int dk,
                        int dv, int chunk, lla_dtype in_dt, lla_dtype out_dt, int group,
                        void *workspace, size_t workspace_bytes, int32_t *device_error,
                        void *stream);

/*
 * Log-Linear Gated DeltaNet ("Log-Linear Attention" §3 names it: the Gated
 * DeltaNet state update under the hierarchical Fenwick mask; the pages give
 * no formula).  Reading implemented: every Fenwick bucket keeps its own
 * state, all bucket states take each token's transition
 *   A_t = exp(g_t) (I - beta_t k_t k_t^T),
 * and the read-out weights them by lambda:
 *   o_t = sum_{s<=t} lambda_t[l(t,s)] beta_s v_s (k_s^T A_{s+1} ... A_t q_t).
 * With lambda = 1 it is Gated DeltaNet.  Keys should be L2-normalised and
 * beta in [0,1] for the transitions to be contractions (not checked).
 *
 * lla_gdn_fwd runs the chunkwise form (§2.3's chunked evaluation with the
 * delta rule's compact product): per chunk of 64 tokens the product of the
 * undecayed factors is I - K^T T K with
 * T = (I + strict_lower(diag(beta) K K^T))^{-1} diag(beta), so the
 * intra-chunk output, the read-out of earlier states and the chunk's
 * transition are small matrix products; the chunk-level Fenwick states are
 * then carried across chunks in order.  Two launches; the products run on
 * the tensor cores as TF32 with every fp32 operand split into a high part
 * and a remainder (about 21 bits; bf16 inputs are exact), accumulation fp32.
 *   q, k [B,H,T,dk], v [B,H,T,dv] in in_dt; g, beta [B,H,T] fp32;
 *   lambda [B,H,T,L] fp32 with L = lla_num_levels(T); out [B,H,T,dv] fp32.
 *   q, k, v and out must be 16-byte aligned (read and written in 16-byte pieces).
 *   state_out (nullable) [B,H,Ls_out,dk,dv] fp32 receives the state after the
 *   sequence in the layout of lla_gdn_decode_step (slot i = level i+1, dead
 *   slots zeroed); Ls_out >= bit_length(T) when state_out is given.
 * Supported: dk, dv in {16,32,64,128}, T <= 2^24 (and the per-CTA state of
 * the chunk scan, bit_length(ceil(T/64)) x dk x 8 floats plus staging, must
 * fit in shared memory), B, H <= 65535.
 * workspace: >= lla_gdn_fwd_workspace_bytes(B,H,T,dk,dv) bytes, 256-byte
 * aligned, owned by the caller (per chunk: q~ and w transposed, the chunk
 * state H, its total decay; fp32).  Errors as lla_fwd: a bad shape returns
 * LLA_ERR_UNSUPPORTED_SHAPE, a NULL or misaligned pointer or a short
 * workspace LLA_ERR_INVALID_ARGUMENT.  B*H*T == 0 is a no-op returning LLA_OK.
 */
size_t lla_gdn_fwd_workspace_bytes(int B, int H, int T, int dk, int dv);
lla_status lla_gdn_fwd(const void *q, const void *k, const void *v, const float *g,
                       const float *beta, const float *lambda, float *out,
                       float *state_out, int B, int H, int T, int dk, int dv,
                       int Ls_out, lla_dtype in_dt, void *workspace,
                       size_t workspace_bytes, void *stream);

/*
 * One decode step of Log-Linear Gated DeltaNet on an eager level state:
 *   state [B,H,Ls,dk,dv] fp32, slot i = level i+1, live for token t = pos[b]
 *   iff bit i of t is set (the state holds the prefix [0, t));
 *   q, k [B,H,dk], v [B,H,dv] in_dt; g, beta [B,H] fp32; lambda [B,H,Ls+1];
 *   out [B,H,dv] fp32; pos [B] int64 on the device.
 * The step transitions every live slot in place, reads out, and writes slot
 * ctz(t+1) = beta k v^T + the slots below it (which become dead; their
 * contents are left as they were).  A position without room
 * (bit_length(t+1) > Ls) sets *device_error = 1 + b (if non-NULL) and that
 * batch row is skipped.  Ls <= 40.
 */
lla_status lla_gdn_decode_step(float *state, const void *q, const void *k,
                               const void *v, const float *g, const float *beta,
                               const float *lambda, float *out, const int64_t *pos,
                               int B, int H, int dk, int dv, int Ls, lla_dtype in_dt,
                               int32_t *device_error, void *stream);

/*
 * Backward of lla_fwd: given dout = dLoss/dout, the gradients of every input.
 * "Log-Linear Attention" §2.2 defines the forward only; these are the
 * derivatives of that double sum (A_ts = lambda_t[l(t,s)] exp(G_t - G_s),
 * s <= t, G the inclusive running sum of g):
 *   dq_t = sum_s A_ts (dout_t . v_s) k_s       dk_s = sum_t A_ts (dout_t . v_s) q_t
 *   dv_s = sum_t A_ts (q_t . k_s) dout_t
 *   dlambda_t[l] = sum_{s: l(t,s)=l} exp(G_t - G_s) (q_t . k_s)(dout_t . v_s)
 *   dg_r = sum_{u >= r} (sum_l lambda_u[l] dlambda_u[l] - k_u . dk_u).
 * Computed chunkwise: the forward's chunk-level Fenwick nodes serve dq and
 * dlambda; one lambda-weighted state per (level, aligned block of later
 * chunks) serves dk and dv.  For bf16 inputs with dk = dv = 128 and chunk 64
 * the products run on the tensor cores with every fp32 operand split into
 * two or three bf16 parts (fp32-level accuracy); otherwise on CUDA cores in
 * fp32.  Sums run in a fixed order, so repeated calls give bitwise-identical
 * results.
 *   q, k [B,H,T,dk], v [B,H,T,dv] in in_dt; g [B,H,T], lambda [B,H,T,L]
 *   (L = lla_num_levels(T)), dout [B,H,T,dv] fp32; outputs (caller-owned,
 *   fully overwritten, fp32): dq, dk [B,H,T,dk], dv [B,H,T,dv], dg [B,H,T],
 *   dlambda [B,H,T,L].  All row-major and contiguous.
 * Supported: chunk in {16,32,64}, T % chunk == 0, T <= 2^24,
 * dk, dv in {16,32,64,128}.  B*H*T == 0 is a no-op returning LLA_OK.
 * workspace: >= lla_bwd_workspace_bytes(...) bytes, 256-byte aligned, owned
 * by the caller; no allocation happens inside.  Errors: a bad shape returns
 * LLA_ERR_UNSUPPORTED_SHAPE, a NULL pointer or misaligned workspace
 * LLA_ERR_INVALID_ARGUMENT, a short workspace LLA_ERR_WORKSPACE_TOO_SMALL,
 * all before any launch; a failed launch returns LLA_ERR_CUDA.
 * device_error: NULL or a caller-owned device int32, set by the tensor-core
 * parts as for lla_fwd.
 */
size_t lla_bwd_workspace_bytes(int B, int H, int T, int dk, int dv, int chunk,
                               lla_dtype in_dt);

lla_status lla_bwd(const void *q, const void *k, const void *v, const float *g,
                   const float *lambda, const float *dout, float *dq, float *dk,
                   float *dv, float *dg, float *dlambda, int B, int H, int T,
                   int dk_dim, int dv_dim, int chunk, lla_dtype in_dt,
                   void *workspace, size_t workspace_bytes, int32_t *device_error,
                   void *stream);

/*
 * Level weights from a two-layer MLP ("Adaptive memory decay for Log-Linear
 * Attention", §Method "LambdaMLPSoftplus"): for every (token, head),
 *     h = d W1 (width 2L, no activation),   lambda = softplus(h W2 + b),
 * so lambda >= 0 with every level scaled independently.  W2 = 0, b = 0.54
 * gives softplus(0.54), about 1.0, everywhere (the page's initialisation).
 *   d      [B,H,T,Dd] in_dt   the per-(token, head) input representation
 *   W1     [Dd, 2L]  fp32     W2 [2L, L] fp32     b [L] fp32 (shared by heads)
 *   lambda [B,H,T,L] fp32     output, the layout lla_fwd reads
 * Supported: 1 <= Dd <= 256, 1 <= L <= 32 (shared memory holds the weights).
 * device_error: NULL or a caller-owned device int32, set by the tensor-core
 * path (bf16 d, Dd a multiple of 64) as for lla_fwd.
 */
lla_status lla_lambda_mlp(const void *d, const float *W1, const float *W2,
                          const float *b, float *lambda, int B, int H, int T,
                          int Dd, int L, lla_dtype in_dt, int32_t *device_error,
                          void *stream);

#ifdef __cplusplus
}
#endif

#endif /* LLA_H */
