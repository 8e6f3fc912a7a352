/*
 * sss.h -- C ABI of libsss: the state-passing forward of a Mamba-2-style
 * recurrent mixer (causal depthwise conv with an explicit conv state, then a
 * scalar-decay selective scan from a non-zero initial state) and its
 * single/multi-token decode update over a circular conv-state pool, as
 * hand-written CUDA kernels for GB300 (sm_103a).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every tensor pointer is a DEVICE pointer owned by the caller; the library
 *    keeps no pointer after a call returns and allocates nothing.
 *  - Tensors are dense and row-major (last index fastest), with the layouts
 *    given per argument.  Every pointer must be aligned to its element size;
 *    16-byte alignment of every tensor (and row strides that are multiples of
 *    16 bytes) selects the vectorised and tensor-core paths.
 *  - All work is enqueued asynchronously on `stream` (NULL = the legacy
 *    default stream).  Host-detectable problems (null pointers, sizes,
 *    dtypes) return a status before anything is launched and leave every
 *    output untouched.  Problems only the device can see (an out-of-range
 *    pool row, a negative length, a wait that ran out) are OR-ed into a
 *    device status word that sss_device_status() reads.
 *  - Names follow the pages: x input, u conv output, dt step size, A per-head
 *    decay rate, B/C input/output projections, h SSM state, S/F conv state,
 *    K conv width, cache_seqlens, conv_state_indices.
 *
 * Symbols: Bz batch, L tokens in the call, D = H*P channels, H heads, P head
 * dimension, N state size, G groups of B/C (H % G == 0, head h uses group
 * h / (H/G)), K conv width.
 */
#ifndef SSS_H_
#define SSS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (the runtime and driver stream handle types are the same). */
typedef struct CUstream_st* sss_stream_t;

typedef enum {
  SSS_OK = 0,
  SSS_ERR_INVALID_ARG = 1, /* null pointer, bad size or dtype; nothing launched */
  SSS_ERR_UNSUPPORTED = 2, /* valid request this build cannot run             */
  SSS_ERR_INDEX = 4,       /* device: pool row outside [0,pool) or length < 0  */
  SSS_ERR_TIMEOUT = 8,     /* device: a bounded wait inside a kernel ran out   */
  SSS_ERR_CUDA = 16        /* a CUDA runtime call failed (launch, no device)   */
} sss_status;

typedef enum { SSS_F32 = 0, SSS_BF16 = 1 } sss_dtype;

/* Library version, major*10000 + minor*100 + patch. */
int sss_version(void);

/* Static string for a status value (bits may be OR-ed together). */
const char* sss_status_string(int status);

/* Text of the last CUDA runtime error a call of this thread turned into
 * SSS_ERR_CUDA (or SSS_ERR_UNSUPPORTED). */
const char* sss_last_cuda_error(void);

/*
 * sss_conv_state_fwd -- causal depthwise conv1d with an explicit conv state.
 *
 * Source: "Chapter 7: state, chunking and incremental inference" (causal-conv1d
 * tutorial), section "define the state with the extended sequence": with the
 * state S holding the K-1 inputs before this call, oldest first, the call
 * computes over u = [S_0..S_{K-2}, x_0..x_{L-1}]
 *     z_t = bias + sum_{k<K} w_k u_{t+k},   F = u[L : L+K-1],
 * and returns SiLU(z) (z / (1 + exp(-z))) when apply_silu != 0, else z.
 * The form holds for L < K-1 (F then keeps part of S) and L == 0 (F = S).
 *
 *  x          [Bz, L, D]   x_dtype
 *  w          [D, K]       float32
 *  bias       [D]          float32, NULL = 0
 *  state_in   [Bz, D, K-1] x_dtype, NULL = zeros (no history)
 *  state_out  [Bz, D, K-1] x_dtype, receives F; may equal state_in (the
 *                          streaming case); NULL = do not write F
 *  u          [Bz, L, D]   u_dtype (SSS_F32 keeps the conv output exact
 *                          enough for the scan's state; SSS_BF16 halves
 *                          the bytes)
 * Returns SSS_ERR_INVALID_ARG for null x/w/u (when L > 0), K < 1, negative
 * sizes, or an unknown dtype.
 */
sss_status sss_conv_state_fwd(const void* x, sss_dtype x_dtype, const float* w,
                              const float* bias, const void* state_in,
                              void* state_out, void* u, sss_dtype u_dtype,
                              int64_t Bz, int64_t L, int64_t D, int K,
                              int apply_silu, sss_stream_t stream);

/*
 * sss_conv_state_bwd -- gradient of sss_conv_state_fwd, state included.
 *
 * Source: "Chapter 7: state, chunking and incremental inference", section
 * "unified derivation of the backward pass with state": with
 * delta_t = dL/dz_t = dy_t SiLU'(z_t) (dy_t when apply_silu == 0) and
 * q = dL/dF,
 *     dL/du_j = sum_{t,k: t+k=j} delta_t w_k + [L <= j < L+K-1] q_{j-L},
 *     dS = du[0 : K-1],  dx = du[K-1 : K-1+L],
 *     dw_k = sum_{b,t} delta_t u_{t+k},  dbias = sum_{b,t} delta_t.
 * The forward is recomputed from x, w, bias and state_in.  Chunked training:
 * the dstate_in of segment B is the dstate_out of segment A (the same
 * chapter, section on chunked training and truncated backpropagation).
 *
 *  x, w, bias, state_in   as in sss_conv_state_fwd (state_in NULL = zeros)
 *  dy          [Bz, L, D]     dy_dtype, dL/d(output)
 *  dstate_out  [Bz, D, K-1]   dy_dtype, dL/dF, NULL = zeros
 *  dx          [Bz, L, D]     dx_dtype, written
 *  dstate_in   [Bz, D, K-1]   dx_dtype, dL/dS, written; must not overlap
 *                             dstate_out
 *  dw, dbias   [D, K], [D]    float32, written (not accumulated); dbias may
 *                             be NULL
 *  workspace   device scratch of at least sss_conv_state_bwd_workspace_size
 *              bytes (per-block partial sums of dw and dbias, reduced in a
 *              fixed order: the result is deterministic); may be NULL when
 *              that size is 0
 * Returns SSS_ERR_INVALID_ARG for null required pointers, misalignment,
 * overlapping dstate_in / dstate_out, a short workspace, bad sizes or an
 * unknown dtype; SSS_ERR_UNSUPPORTED for K > 8.
 */
size_t sss_conv_state_bwd_workspace_size(int64_t Bz, int64_t L, int64_t D, int K);

sss_status sss_conv_state_bwd(const void* x, sss_dtype x_dtype, const float* w,
                              const float* bias, const void* state_in,
                              const void* dy, sss_dtype dy_dtype,
                              const void* dstate_out, void* dx, sss_dtype dx_dtype,
                              void* dstate_in, float* dw, float* dbias,
                              int64_t Bz, int64_t L, int64_t D, int K,
                              int apply_silu, void* workspace,
                              size_t workspace_bytes, sss_stream_t stream);

/*
 * sss_conv_state_bwd_noalloc -- sss_conv_state_bwd without a caller-provided
 * workspace, for callers that cannot allocate device memory.  The pages have
 * no counterpart: this is a library convenience, not part of the method.
 *
 * Some callers can't call cudaMalloc (or any allocator) at the point where
 * they run the backward: a plugin inside an inference or training engine
 * whose execute step is not allowed to allocate, code that runs with a fixed
 * device-memory budget handed to it by a host framework it has no allocator
 * handle for, or a latency-critical loop that must not pay for cudaMalloc's
 * implicit synchronisation.  This entry point takes the same arguments as
 * sss_conv_state_bwd minus the workspace, computes the same dx, dstate_in,
 * dw and dbias, and keeps its partial sums in one static device array of
 * SSS_CONV_BWD_NOALLOC_SCRATCH_BYTES bytes that belongs to the library.  It
 * calls no cudaMalloc, cudaFree or allocating library routine.
 *
 *  - Size limit: it serves calls whose sss_conv_state_bwd_workspace_size()
 *    is at most SSS_CONV_BWD_NOALLOC_SCRATCH_BYTES (8 MiB: for example
 *    Bz = 32 sequences of 1024 tokens at D = 2048, K = 4 need 5 MiB)
 *    and returns SSS_ERR_UNSUPPORTED, before anything is launched, for
 *    larger ones.  Other errors are those of sss_conv_state_bwd.
 *  - Memory: every GPU that loads the library holds the 8 MiB array until
 *    the process exits.
 *  - Set-up: the first call on a device, with that device current, looks up
 *    the array's device address (cudaGetSymbolAddress) and caches it for
 *    that device's current context; a call under another context (after
 *    cudaDeviceReset, say, when the module is loaded again and the array may
 *    sit elsewhere) looks it up again.  Make the first call on a device, and
 *    the first after a reset, before any stream capture begins.  A failed
 *    lookup returns SSS_ERR_CUDA.
 *  - Sharing: all calls on a device use the same array, and it keeps the
 *    last call's partial sums.  Each call writes every partial it reads
 *    before reading it, so nothing needs clearing between calls; but two
 *    calls that can run at the same time on the GPU (different streams, no
 *    ordering between them) race on the array and give wrong dw and dbias.
 *    Serialise them, e.g. by issuing them on one stream.
 */
#define SSS_CONV_BWD_NOALLOC_SCRATCH_BYTES (8u << 20)

sss_status sss_conv_state_bwd_noalloc(const void* x, sss_dtype x_dtype, const float* w,
                                      const float* bias, const void* state_in,
                                      const void* dy, sss_dtype dy_dtype,
                                      const void* dstate_out, void* dx,
                                      sss_dtype dx_dtype, void* dstate_in, float* dw,
                                      float* dbias, int64_t Bz, int64_t L, int64_t D,
                                      int K, int apply_silu, sss_stream_t stream);

/* The size in bytes of the static array behind sss_conv_state_bwd_noalloc
 * (SSS_CONV_BWD_NOALLOC_SCRATCH_BYTES), for bindings that cannot read the
 * macro. */
size_t sss_conv_state_bwd_noalloc_scratch_bytes(void);

/*
 * sss_conv_state_fwd_packed -- sss_conv_state_fwd over rows that pack several
 * samples.  Source: "Chapter 7: state, chunking and incremental inference",
 * section "packed sequence boundaries": with samples A and B concatenated in
 * one row, B's first tokens must not read A's end; tap k of token t reads
 * the extended-sequence entry u_{t+k} only when that entry's sequence id
 * equals token t's (identity equality: a reused id, as in A, B, A, is not
 * recognised as a reset - the caller gives distinct ids within a window).
 * The state entries (positions < 0) carry token 0's id: the call continues
 * the sample its first token belongs to.  F = u[L : L+K-1] as without ids.
 *  seq_idx  [Bz, L] int32 (device); every other argument as for
 *           sss_conv_state_fwd (state_out may equal state_in).
 */
sss_status sss_conv_state_fwd_packed(const void* x, sss_dtype x_dtype, const float* w,
                                     const float* bias, const void* state_in, void* state_out,
                                     const int32_t* seq_idx, void* u, sss_dtype u_dtype,
                                     int64_t Bz, int64_t L, int64_t D, int K, int apply_silu,
                                     sss_stream_t stream);

/*
 * sss_ssm_scan_fwd -- scalar-decay selective scan from an initial state.
 *
 * Source: "Understanding and Improving Length Generalization in Recurrent
 * Models", section 2 Eq. (1) h_t = A_t h_{t-1} + B_t x_t, y_t = C_t^T h_t,
 * with one scalar decay per head A_t = exp(dt_t * A_h), started from a
 * non-zero initial state h_{-1} as in Eq. (4) (section 4.1), and returning
 * the final state so a later call can continue (state passing, TBTT).
 * Per (batch b, head h, channel p, state n):
 *     h[p,n] <- exp(dt[b,t,h] A[h]) h[p,n] + x[b,t,h,p] B[b,t,g,n]
 *     y[b,t,h,p] = sum_n h[p,n] C[b,t,g,n]
 *
 *  x       [Bz, L, H, P]  x_dtype (the conv output u)
 *  dt      [Bz, L, H]     act_dtype, already positive (post-softplus)
 *  A       [H]            float32 (negative for a decaying state)
 *  B, C    [Bz, L, G, N]  act_dtype
 *  h0_in   [Bz, H, P, N]  float32, NULL = zeros
 *  hT_out  [Bz, H, P, N]  float32, may equal h0_in; NULL = do not write
 *  y       [Bz, L, H, P]  y_dtype
 *  workspace / workspace_bytes: scratch of at least
 *          sss_ssm_scan_workspace_size() bytes (may be NULL when that is 0).
 * bf16 activations with P == 64, N == 128 run on a tcgen05 tensor-core
 * chunked scan (two heads per CTA when H / G is even, one otherwise); every
 * other case runs on the fp32 CUDA-core scan.  The state is kept in fp32
 * throughout.
 */
size_t sss_ssm_scan_workspace_size(int64_t Bz, int64_t L, int H, int P, int N,
                                   int G, sss_dtype x_dtype, sss_dtype act_dtype);

/* Which kernel sss_ssm_scan_fwd picks for these sizes and dtypes (given
 * 16-byte aligned tensors): 2 = tcgen05 chunked scan over head pairs,
 * 1 = tcgen05 chunked scan, one head per CTA, 0 = fp32 CUDA-core scan,
 * -1 = unsupported. */
int sss_ssm_scan_path(int64_t Bz, int64_t L, int H, int P, int N, int G,
                      sss_dtype x_dtype, sss_dtype act_dtype, sss_dtype y_dtype);

sss_status sss_ssm_scan_fwd(const void* x, sss_dtype x_dtype, const void* dt,
                            const float* A, const void* B, const void* C,
                            sss_dtype act_dtype, const float* h0_in,
                            float* hT_out, void* y, sss_dtype y_dtype,
                            int64_t Bz, int64_t L, int H, int P, int N, int G,
                            void* workspace, size_t workspace_bytes,
                            sss_stream_t stream);

/*
 * sss_ssm_scan_bwd -- gradient of sss_ssm_scan_fwd with state, for
 * state-passing and truncated-backpropagation training.  Sources:
 * "Understanding and Improving Length Generalization in Recurrent Models",
 * sections 4.4-4.5 (a segment starts from the previous segment's final
 * state; the gradient of that state is what flows back into the previous
 * segment), with the recurrence of section 2 Eq. (1) and the initial-state
 * form Eq. (4); "Chapter 7: state, chunking and incremental inference",
 * section "chunked training and truncated backpropagation" (the state
 * gradient of chunk B must be passed to chunk A for the chunked gradient
 * to equal the whole one).  With g_t = dL/dh_t and a_t = exp(dt_t A_h):
 *     g_{L-1} = dhT + dy_{L-1} C_{L-1}^T,  g_t = a_{t+1} g_{t+1} + dy_t C_t^T
 *     dx_t = g_t B_t,  dB_t = g_t^T x_t,  dC_t = h_t^T dy_t,
 *     ddt_t = A_h a_t <g_t, h_{t-1}>,  dA_h = sum_t dt_t a_t <g_t, h_{t-1}>,
 *     dh0 = a_0 g_0
 * (dB and dC summed over the heads of a group, dA over the batch).
 *
 *  x, dt, A, B, C, h0_in   as for sss_ssm_scan_fwd (h0_in NULL = zeros)
 *  dy      [Bz, L, H, P]  float32, dL/dy
 *  dhT     [Bz, H, P, N]  float32, dL/d(final state); NULL = zeros
 *  dx      [Bz, L, H, P]  float32 (written)
 *  ddt     [Bz, L, H]     float32 (written)
 *  dA      [H]            float32 (written, not accumulated)
 *  dB, dC  [Bz, L, G, N]  float32 (written)
 *  dh0     [Bz, H, P, N]  float32, dL/dh0; NULL = not written; may be the
 *                         same buffer as dhT (any other overlap is invalid)
 *  workspace: at least sss_ssm_scan_bwd_workspace_size() bytes, 256-byte
 *          aligned, owned by the caller (chunk-boundary states and gradients
 *          and per-head partial sums; contents need not be initialised).
 * Deterministic: every sum has a fixed order.  P <= 64 and N <= 128
 * (SSS_ERR_UNSUPPORTED otherwise); any dtype mix of x and activations.
 * The arithmetic is fp32 from the exact input values.
 */
size_t sss_ssm_scan_bwd_workspace_size(int64_t Bz, int64_t L, int H, int P, int N, int G);

sss_status sss_ssm_scan_bwd(const void* x, sss_dtype x_dtype, const void* dt,
                            const float* A, const void* B, const void* C,
                            sss_dtype act_dtype, const float* h0_in, const float* dy,
                            const float* dhT, float* dx, float* ddt, float* dA, float* dB,
                            float* dC, float* dh0, int64_t Bz, int64_t L, int H, int P,
                            int N, int G, void* workspace, size_t workspace_bytes,
                            sss_stream_t stream);

/*
 * sss_prefill_to_pool -- write the state a prompt leaves into the pool rows
 * the decode update reads.  Source: "Chapter 7: state, chunking and
 * incremental inference", sections "continuous batching" (rows addressed by
 * conv_state_indices), "circular mode" (logical position q in slot
 * q mod S_len) and "the physical cache can be longer" (non-circular rows,
 * oldest first).  For request b, r = conv_state_indices[b] (b when NULL):
 * conv_pool row r gets the newest S_len entries of the extended sequence
 * u = [conv_state_in (K-1 values), x (L values)], zeros where u has none;
 * with cache_seqlens (p = cache_seqlens[b], the length after the prompt,
 * the prompt at logical positions p - L .. p - 1) position q goes to slot
 * q mod S_len, without it (non-circular) the S_len values go oldest first.
 * ssm_pool row r gets hT[b] (hT and ssm_pool both given or both NULL).
 * The decode update on the next tokens then continues the request exactly.
 * A row with r outside [0, pool) or p < 0 is skipped and SSS_ERR_INDEX is
 * raised in the device status; two requests naming one row is a contract
 * violation.
 *
 *  x              [Bz, L, H*P]     x_dtype (the prompt's conv inputs)
 *  conv_state_in  [Bz, H*P, K-1]   x_dtype, the conv state before the prompt; NULL = zeros
 *  hT             [Bz, H, P, N]    float32, 16-byte aligned (P*N a multiple of 4)
 *  conv_pool      [pool, H*P, S_len] x_dtype, S_len >= K-1
 *  ssm_pool       [pool, H, P, N]  float32
 */
sss_status sss_prefill_to_pool(const void* x, sss_dtype x_dtype, const void* conv_state_in, int K,
                               const float* hT, void* conv_pool, int64_t pool, int S_len,
                               float* ssm_pool, const int32_t* cache_seqlens,
                               const int32_t* conv_state_indices, int64_t Bz, int64_t L,
                               int64_t D, int H, int P, int N, sss_stream_t stream);

/*
 * State-passing training utilities.  Source: "Understanding and Improving
 * Length Generalization in Recurrent Models", section 4.4 (state passing:
 * the next batch starts from the previous final states, each reset to zero
 * with probability p = 0.1), section 4.2 Eqs. (5)-(6) (fitted noise:
 * per-head mean and variance of the final states, mixed into running values
 * with weight 1 - beta = 0.9 on the new statistic, then Gaussian initial
 * states), section 3.5 (the state scale as a function of position).  The
 * random draws are inputs, so results follow the caller's generator.
 *
 * sss_state_reset: row b of h [Bz, h_row_elems] fp32 and of conv_state
 *   [Bz, conv_row_elems] (conv_dtype; either may be NULL, not both) is set to
 *   zero when u[b] < p_reset (u [Bz] fp32 uniforms in [0, 1)); other rows are
 *   not touched (not even rewritten).
 * sss_fitted_noise_update: per head h, over hT [Bz, H, P, N] fp32, the mean
 *   and the population variance of the Bz * P * N values; with has_history,
 *   mu[h] = (1 - beta) mean + beta mu[h] and var[h] likewise, else mu[h] =
 *   mean, var[h] = variance.  mu, var [H] fp32, in/out.  Sums in fp64, in a
 *   fixed order (deterministic).
 * sss_fitted_noise_sample: h0[b, h, p, n] = mu[h] + sqrt(var[h]) eps[b, h, p, n]
 *   with eps [Bz, H, P, N] fp32 standard normal draws.
 * sss_state_std_trace: runs the scan of sss_ssm_scan_fwd (inputs as there,
 *   y not produced) and writes out[b, k, h] = the standard deviation over the
 *   P x N elements of head h's state after token min(stride (k + 1), L) - 1,
 *   k < ceil(L / stride); 1 <= stride <= 64, P <= 64, N <= 128
 *   (SSS_ERR_UNSUPPORTED otherwise).
 */
sss_status sss_state_reset(const float* u, float p_reset, float* h, int64_t Bz,
                           int64_t h_row_elems, void* conv_state, sss_dtype conv_dtype,
                           int64_t conv_row_elems, sss_stream_t stream);
sss_status sss_fitted_noise_update(const float* hT, int64_t Bz, int H, int P, int N, float beta,
                                   int has_history, float* mu, float* var, sss_stream_t stream);
sss_status sss_fitted_noise_sample(const float* mu, const float* var, const float* eps,
                                   float* h0, int64_t Bz, int H, int P, int N,
                                   sss_stream_t stream);
sss_status sss_state_std_trace(const void* x, sss_dtype x_dtype, const void* dt, const float* A,
                               const void* B, sss_dtype act_dtype, const float* h0, float* out,
                               int64_t Bz, int64_t L, int H, int P, int N, int G, int stride,
                               sss_stream_t stream);

/*
 * sss_ssm_scan_fwd_packed / sss_mixer_fwd_packed -- the forward over rows
 * that pack several samples (seq_idx [Bz, L] int32, device).  Source:
 * "Chapter 7: state, chunking and incremental inference", section "packed
 * sequence boundaries" (no history crosses a sample boundary).  The conv of
 * sss_mixer_fwd_packed follows sss_conv_state_fwd_packed; in the scan a
 * token whose id differs from the previous token's restarts the state from
 * zero (its decay is exactly zero: the kernels give it log-decay -200, which
 * underflows to 0 in fp32); the first token continues from h0_in.  Arguments
 * otherwise as for sss_ssm_scan_fwd and sss_mixer_fwd; the fused packed
 * forward needs the two-heads-per-CTA kernel (H / G even), else
 * SSS_ERR_UNSUPPORTED (compose sss_conv_state_fwd_packed and
 * sss_ssm_scan_fwd_packed instead).
 */
sss_status sss_ssm_scan_fwd_packed(const void* x, sss_dtype x_dtype, const void* dt,
                                   const float* A, const void* B, const void* C,
                                   sss_dtype act_dtype, const float* h0_in, float* hT_out,
                                   const int32_t* seq_idx, void* y, sss_dtype y_dtype, int64_t Bz,
                                   int64_t L, int H, int P, int N, int G, sss_stream_t stream);
sss_status sss_mixer_fwd_packed(const void* x, sss_dtype x_dtype, const float* w,
                                const float* bias, const void* conv_state_in,
                                void* conv_state_out, const void* dt, const float* A,
                                const void* B, const void* C, const float* h0_in, float* hT_out,
                                const int32_t* seq_idx, void* y, sss_dtype y_dtype, int64_t Bz,
                                int64_t L, int H, int P, int N, int G, int K,
                                sss_stream_t stream);

/*
 * sss_mixer_fwd -- one segment of the streaming forward in a single kernel:
 * the conv with state of sss_conv_state_fwd (SiLU applied) feeding the scan
 * of sss_ssm_scan_fwd, so the conv output never goes to memory.  Sources:
 * both of the above, and "Chapter 7: state, chunking and incremental
 * inference", section "chunked training and truncated backpropagation"
 * (segment B starts from segment A's final conv state, S_B = F_A) together
 * with section 2.6 / Eq. (4) of "Understanding and Improving Length
 * Generalization in Recurrent Models" (state passing of h).
 *
 *  x                   [Bz, L, H*P]  x_dtype (bf16 on this path)
 *  w, bias             [H*P, K], [H*P]  float32 (bias NULL = 0)
 *  conv_state_in/out   [Bz, H*P, K-1] x_dtype; may be the same buffer;
 *                      NULL in = zeros, NULL out = not written
 *  dt                  [Bz, L, H]    x_dtype, positive
 *  A                   [H]           float32
 *  B, C                [Bz, L, G, N] x_dtype
 *  h0_in / hT_out      [Bz, H, P, N] float32; may be the same buffer
 *  y                   [Bz, L, H, P] y_dtype
 * Supported (sss_mixer_fwd_supported() == 1): bf16 x/dt/B/C, P == 64,
 * N == 128, K <= 4; otherwise SSS_ERR_UNSUPPORTED (compose
 * sss_conv_state_fwd and sss_ssm_scan_fwd instead).
 */
int sss_mixer_fwd_supported(int64_t Bz, int64_t L, int H, int P, int N, int G,
                            int K, sss_dtype x_dtype, sss_dtype y_dtype);

sss_status sss_mixer_fwd(const void* x, sss_dtype x_dtype, const float* w,
                         const float* bias, const void* conv_state_in,
                         void* conv_state_out, const void* dt, const float* A,
                         const void* B, const void* C, const float* h0_in,
                         float* hT_out, void* y, sss_dtype y_dtype, int64_t Bz,
                         int64_t L, int H, int P, int N, int G, int K,
                         sss_stream_t stream);

/*
 * Span-parallel forward -- the same results as sss_mixer_fwd /
 * sss_ssm_scan_fwd, for long sequences in small batches that give the
 * chunked scan too few (batch row, head pair) work items to fill the GPU.
 * Source: "Understanding and Improving Length Generalization in Recurrent
 * Models", section 2.5 Eq. (4): the state at the end of a stretch of tokens
 * is the state reached from a zero start plus the inherited state decayed by
 * the stretch's total decay, so stretches compose associatively.  Each
 * sequence is cut into ns equal spans of L / ns tokens that run as separate
 * rows: a first pass from zero states gives every span's own final state, a
 * warp-shuffle scan over the spans (fp32) gives every span its true initial
 * state and the call its final state, and a second pass from those states
 * writes y.  The conv state of span k > 0 is the K-1 inputs before it.
 *
 * sss_mixer_fwd_span_count / sss_ssm_scan_fwd_span_count: the ns the library
 * would pick for these sizes on the current device (1 = no split pays, or
 * the sizes are not supported by the span path).
 * sss_fwd_spans_workspace_size: bytes of scratch for ns spans (0 for ns < 2);
 * K = 1 for the scan alone.
 * sss_mixer_fwd_spans / sss_ssm_scan_fwd_spans: arguments as in
 * sss_mixer_fwd / sss_ssm_scan_fwd, plus ns (1..32; 1 = the one-pass call)
 * and the workspace (256-byte aligned, at least
 * sss_fwd_spans_workspace_size() bytes, not overlapping any argument).
 * h0_in / hT_out must be 16-byte aligned here.
 * Requires L % ns == 0, L / ns >= K - 1 (else SSS_ERR_INVALID_ARG) and the
 * head-pair tcgen05 scan (bf16 dt/B/C, P == 64, N == 128, H / G even; else
 * SSS_ERR_UNSUPPORTED).  h0_in / hT_out and conv_state_in / conv_state_out
 * may be the same buffers.  Numerics: y and hT come from fp32 states as in
 * the one-pass call; rounding differs by the order of the carry.
 */
int sss_mixer_fwd_span_count(int64_t Bz, int64_t L, int H, int P, int N, int G, int K,
                             sss_dtype x_dtype, sss_dtype y_dtype);
int sss_ssm_scan_fwd_span_count(int64_t Bz, int64_t L, int H, int P, int N, int G,
                                sss_dtype x_dtype, sss_dtype act_dtype, sss_dtype y_dtype);
size_t sss_fwd_spans_workspace_size(int64_t Bz, int64_t L, int H, int P, int N, int K, int ns);
sss_status sss_mixer_fwd_spans(const void* x, sss_dtype x_dtype, const float* w,
                               const float* bias, const void* conv_state_in,
                               void* conv_state_out, const void* dt, const float* A,
                               const void* B, const void* C, const float* h0_in, float* hT_out,
                               void* y, sss_dtype y_dtype, int64_t Bz, int64_t L, int H, int P,
                               int N, int G, int K, int ns, void* workspace,
                               size_t workspace_bytes, sss_stream_t stream);
sss_status sss_ssm_scan_fwd_spans(const void* x, sss_dtype x_dtype, const void* dt,
                                  const float* A, const void* B, const void* C,
                                  sss_dtype act_dtype, const float* h0_in, float* hT_out, void* y,
                                  sss_dtype y_dtype, int64_t Bz, int64_t L, int H, int P, int N,
                                  int G, int ns, void* workspace, size_t workspace_bytes,
                                  sss_stream_t stream);

/*
 * sss_mixer_update -- single/multi-token decode update over a circular
 * conv-state pool, then the same scan on the pool's SSM state.
 *
 * Source: "Chapter 7: state, chunking and incremental inference", sections
 * "single-token update", "the physical cache may be longer than the minimum
 * history", "circular mode" and "continuous batching".  For request row b:
 * r = conv_state_indices[b] (b when NULL), p = cache_seqlens[b].  History j
 * (j = 1..K-1) of channel d is read from conv_pool[r, d, (p-j) mod S_len]
 * before anything is written; token i (logical position p+i) uses the
 * register window, then its INPUT x_i (not the output) is stored at slot
 * (p+i) mod S_len.  u_i = SiLU(bias + sum_k w_k window_k).  Then for every
 * head the recurrence above runs over the L_new tokens on
 * ssm_pool[r, h] (fp32, updated in place) and writes y.
 * cache_seqlens is NOT advanced: the caller adds L_new after the call.
 * cache_seqlens NULL selects the non-circular mode of the same chapter
 * ("the physical cache may be longer than the minimum history"): each row
 * holds its newest S_len >= K-1 inputs, oldest at slot 0; the history of the
 * first new token is slots S_len-K+1 .. S_len-1, and after the call the row
 * holds the last S_len entries of [row, x_0 .. x_{L_new-1}] (the oldest L_new
 * dropped, the new inputs appended).
 * A slot reused for a new request must be cleared by the caller (p < K-1
 * reads the wrapped slots as they are).  Two rows naming the same pool row
 * is a contract violation (undefined result).  A row with r outside
 * [0, pool) or p < 0 is skipped: its pool rows are untouched, its y rows are
 * set to zero and SSS_ERR_INDEX is raised in the device status.
 *
 *  x_new              [Bz, L_new, D]      act_dtype
 *  w, bias            [D, K], [D]         float32 (bias NULL = 0)
 *  conv_pool          [pool, D, S_len]    act_dtype, S_len >= K-1, in/out
 *  cache_seqlens      [Bz]                int32 (device); NULL = non-circular
 *  conv_state_indices [Bz]                int32 (device), NULL = identity
 *  dt                 [Bz, L_new, H]      act_dtype
 *  A                  [H]                 float32
 *  B, C               [Bz, L_new, G, N]   act_dtype
 *  ssm_pool           [pool, H, P, N]     float32, in/out
 *  y                  [Bz, L_new, H, P]   act_dtype
 * L_new <= 64.  With N == 128, P a multiple of 8 (P <= 128), L_new <= 8
 * and 16-byte aligned x_new, w, bias, conv_pool, B, C and ssm_pool the
 * update streams each (request, head) state block through shared memory
 * with bulk copies (persistent kernel); other shapes run one CTA per
 * (request, head).  Both give the same result.
 */
sss_status sss_mixer_update(const void* x_new, sss_dtype act_dtype,
                            const float* w, const float* bias, void* conv_pool,
                            int64_t pool, int S_len,
                            const int32_t* cache_seqlens,
                            const int32_t* conv_state_indices, const void* dt,
                            const float* A, const void* B, const void* C,
                            float* ssm_pool, void* y, int64_t Bz, int L_new,
                            int H, int P, int N, int G, int K,
                            sss_stream_t stream);

/* Which kernel sss_mixer_update picks for these sizes (given 16-byte
 * aligned tensors and a bias): 1 = bulk-copy pipelined kernel, 0 = one CTA
 * per (request, head), -1 = unsupported. */
int sss_mixer_update_path(int L_new, int P, int N, int K, int S_len,
                          sss_dtype act_dtype);

/*
 * sss_mamba2_mixer_fwd -- one segment of the full Mamba-2 mixer wiring: the
 * conv with state over every channel of xBC, then the scan with Mamba-2's
 * discretisation, D skip and gate.  Sources: the Mamba-2 370M-1.3B layers the
 * length-generalisation study post-trains ("Understanding and Improving
 * Length Generalization in Recurrent Models", sections 1 and 4.4), whose
 * mixer convolves x, B and C together before the scan, and "Chapter 7:
 * state, chunking and incremental inference" for the conv with state.  Per
 * (batch row b, head h) and token t, with u = SiLU(conv(xBC)) split into
 * x = u[..., 0:D], B = u[..., D + g N : D + (g+1) N] and
 * C = u[..., D + G N + g N : D + G N + (g+1) N] (g the head's group):
 *   dt_t = softplus(dt_raw_t + dt_bias_h),  a_t = exp(dt_t A_h),
 *   h_t  = a_t h_{t-1} + dt_t x_t B_t^T,
 *   y_t  = (h_t C_t + D_h x_t) SiLU(z_t).
 *
 *  xBC                 [Bz, L, D + 2 G N]  act_dtype, D = H*P
 *  z                   [Bz, L, D] act_dtype, or NULL (no gate)
 *  dt_raw              [Bz, L, H] act_dtype (before bias and softplus)
 *  dt_bias, A, D_skip  [H] float32 (dt_bias / D_skip NULL = 0)
 *  conv_w, conv_b      [D + 2 G N, K], [D + 2 G N] float32 (conv_b NULL = 0)
 *  conv_state_in/out   [Bz, D + 2 G N, K-1] act_dtype; may be the same
 *                      buffer; NULL in = zeros, NULL out = not written
 *  h0_in / hT_out      [Bz, H, P, N] float32; may be the same buffer
 *  y                   [Bz, L, H, P] y_dtype
 *  workspace           caller-owned device buffer of at least
 *                      sss_mamba2_mixer_fwd_workspace_size() bytes, 16-byte
 *                      aligned: the fp32 conv output of every channel
 * The scan runs in fp32 on CUDA cores with the state in registers: B and C
 * come out of the conv and are not rounded before the scan.  K <= 8,
 * P <= 128, N <= 256 (else SSS_ERR_UNSUPPORTED).  Asynchronous on `stream`.
 */
size_t sss_mamba2_mixer_fwd_workspace_size(int64_t Bz, int64_t L, int H, int P, int N, int G);

sss_status sss_mamba2_mixer_fwd(const void* xBC, const void* z, sss_dtype act_dtype,
                                const void* dt_raw, const float* dt_bias, const float* A,
                                const float* D_skip, const float* conv_w, const float* conv_b,
                                const void* conv_state_in, void* conv_state_out,
                                const float* h0_in, float* hT_out, void* y, sss_dtype y_dtype,
                                int64_t Bz, int64_t L, int H, int P, int N, int G, int K,
                                void* workspace, size_t workspace_bytes, sss_stream_t stream);

/*
 * sss_device_status -- read the device status word (OR of SSS_ERR_INDEX /
 * SSS_ERR_TIMEOUT raised by kernels of this library on the current device)
 * after the work on `stream` has finished; clear it when `clear` != 0.
 * Synchronises `stream`.
 */
sss_status sss_device_status(int* status_out, int clear, sss_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* SSS_H_ */
