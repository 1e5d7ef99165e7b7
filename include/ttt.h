/*
 * ttt.h - C ABI of the GB300 (sm_103a) large-chunk TTT-KVB layer and its
 * chunked linear-attention reduction.
 *
 * The operation (from "5.2.1 LaCT and TTT-E2E", eqs (2)-(6) and (10), and
 * "Test-Time Training with KV Binding Is Secretly Linear Attention", sec. 5.3,
 * 6.1, App. E, H): each (batch, head) carries a bias-free SwiGLU fast-weight
 * net f_W(x) = W2 [SiLU(W1 x) o (W3 x)].  The sequence is cut into chunks of
 * `chunk` tokens.  Per chunk the layer
 *   (apply)  o_i = f_W(q_i) for every query of the chunk, and
 *   (update) g = grad_W sum_i eta_i * (-f_W(k_i)^T v_i)   (summed, no 1/b),
 *            M <- beta M + g, U = Muon(M) (Newton-Schulz) or M,
 *            W <- L2-Normalize(W - U) (rows to unit norm over the input dim),
 * in the order the mask mode sets.  For a linear fast weight the layer is the
 * chunked linear attention computed by linattn_chunked_forward.
 *
 * Conventions for every entry point:
 *   - All pointers are DEVICE pointers (cudaMalloc'd or otherwise
 *     device-accessible) unless the argument says "host".  The caller owns
 *     every buffer; the library allocates nothing on the call path.
 *   - Tensors are dense row-major with the shapes given per argument.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream).  Argument errors are found on the host and returned
 *     before anything is enqueued.  Failures detected by a kernel (a bounded
 *     wait that ran out) are recorded in a device status word that
 *     ttt_device_status() reads.
 *   - Inputs are read-only; q and k may alias (the "replace Q with K" use).
 *   - bf16 I/O computes with bf16 tensor-core operands and fp32 accumulation
 *     and fp32 fast-weight state; fp32 I/O computes in fp32 throughout (no
 *     TF32).  There is no CPU fallback.
 */
#ifndef TTT_GB300_TTT_H
#define TTT_GB300_TTT_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* ttt_stream_t; /* a cudaStream_t */

typedef enum {
  TTT_OK = 0,
  TTT_ERR_NULL = -1,        /* a required pointer is NULL */
  TTT_ERR_SHAPE = -2,       /* sizes inconsistent (e.g. N % chunk != 0) */
  TTT_ERR_ALIGN = -3,       /* a pointer is not 16-byte aligned */
  TTT_ERR_UNSUPPORTED = -4, /* valid request the library does not implement */
  TTT_ERR_WORKSPACE = -5,   /* workspace NULL or smaller than the query says */
  TTT_ERR_CUDA = -6,        /* a CUDA runtime call failed (no device, launch) */
  TTT_ERR_TIMEOUT = -7,     /* a kernel's bounded wait ran out (device word) */
  TTT_ERR_ARG = -8,         /* an argument value is out of range */
  TTT_ERR_PAGEABLE = -9     /* a host buffer is not page-locked */
} ttt_status;

typedef enum { TTT_F32 = 0, TTT_BF16 = 1 } ttt_dtype;

/* Order of apply and update per chunk ("5.2.1 LaCT and TTT-E2E", sec. 1.1 and
 * eq (10)).
 *   TTT_APPLY_THEN_UPDATE: chunk c is read with the state after chunks
 *                          0..c-1, then chunk c updates it (causal LM).
 *   TTT_BLOCK_CAUSAL:      chunk c updates first, then is read (block mask).
 *   TTT_BIDIRECTIONAL:     one chunk covering the sequence (chunk == N),
 *                          update then apply (full attention).
 *   TTT_STRIDED:           update (then apply) only on chunks flagged in
 *                          update_chunks; apply on every chunk. */
typedef enum {
  TTT_APPLY_THEN_UPDATE = 0,
  TTT_BLOCK_CAUSAL = 1,
  TTT_BIDIRECTIONAL = 2,
  TTT_STRIDED = 3
} ttt_mask_mode;

/* Forms of the chunk scan (form field of ttt_update_rule). */
typedef enum {
  TTT_FORM_AUTO = 0,       /* parallel where it is exact (see below), else recurrent */
  TTT_FORM_RECURRENT = 1,  /* chunk after chunk */
  TTT_FORM_PARALLEL = 2    /* the parallel form; TTT_ERR_ARG where it is not exact */
} ttt_form;

/* Weight-update rule ("5.2.1 LaCT and TTT-E2E", eqs (5), (6) and the
 * momentum sentence after eq (6)).
 *   l2norm        : 1 = L2-Normalize every updated row after W - U.
 *   muon_steps    : Newton-Schulz steps of Muon(M); 0 = U is M itself.
 *   momentum_beta : M <- beta M + g; 0 = no momentum (M = g).
 *   ns_a/ns_b/ns_c: Newton-Schulz coefficients X <- aX + b(XX^T)X + c(XX^T)^2X
 *                   (the Muon quintic is 3.4445, -4.7750, 2.0315).
 *   last_layer_only: 1 = only W2 updates; W1 and W3 keep their initial
 *                   values, so phi(x) = SiLU(W1 x) o (W3 x) is a static
 *                   feature map ("Test-Time Training with KV Binding Is
 *                   Secretly Linear Attention", sec. 6.1 Step 1, Variant 1).
 *   inner_steps   : update steps taken on each updating chunk (each one a
 *                   gradient at the current weights, momentum, Muon and
 *                   normalisation); 0 or 1 = one ("Test-Time Training with
 *                   KV Binding...", sec. 4.1 / Fig. 1, more inner-loop steps).
 *   form          : ttt_form.  The parallel form (App. H, sec. 6.2: static
 *                   feature map, no normalisation, so the state update is
 *                   associative; Variant 2) is exact when last_layer_only = 1,
 *                   l2norm = 0 and inner_steps <= 1; it first computes phi(q)
 *                   and phi(k) for every token, then runs the chunked linear
 *                   attention with momentum and Muon of
 *                   linattn_chunked_forward_rule (needs d_h, m_h <= 512 on
 *                   the bf16 path).
 * Muon first scales M to unit Frobenius norm (eps 1e-7) and transposes a
 * matrix with more rows than columns. */
typedef struct {
  int l2norm;
  int muon_steps;
  float momentum_beta;
  float ns_a, ns_b, ns_c;
  int last_layer_only;
  int inner_steps;
  int form;
} ttt_update_rule;

/* Human-readable name of a status code (static string, never NULL). */
const char* ttt_status_string(int status);

/* Bytes of device workspace ttt_layer_forward needs for these arguments
 * (0 if the arguments are invalid).  rule may not be NULL. */
size_t ttt_layer_workspace_size(int B, int H, int N, int d_h, int m_h, int chunk,
                                int io_dtype, int mask_mode,
                                const ttt_update_rule* rule);

/* The LaCT TTT layer forward over a whole sequence.
 *
 *   q, k, v     [B, H, N, d_h] in io_dtype (k may alias q).
 *   eta         [B, H, N] fp32: per-token learning rate eta_i (eq 2); any
 *               sign (negative eta is gradient ascent).
 *   W1, W3      fp32 initial fast weights [H, m_h, d_h] (w_per_batch = 0,
 *               shared over the batch) or [B, H, m_h, d_h] (w_per_batch = 1).
 *   W2          fp32 [H, d_h, m_h] or [B, H, d_h, m_h] likewise.
 *   chunk       tokens per chunk; N % chunk == 0; BIDIRECTIONAL needs
 *               chunk == N.
 *   update_chunks  HOST array of N/chunk bytes (nonzero = update on that
 *               chunk); read only for TTT_STRIDED, may be NULL otherwise.
 *   rule        HOST pointer to the update rule.
 *   out         [B, H, N, d_h] in io_dtype: o_i = f_W(q_i).
 *   W1_final, W3_final  fp32 [B, H, m_h, d_h]; W2_final fp32 [B, H, d_h, m_h]:
 *               the fast weights after the last chunk.  They hold the running
 *               state during the call; they may alias W1/W2/W3 only when
 *               w_per_batch = 1.
 *   momentum    NULL, or fp32 [3][B][H][m_h*d_h] in the order M1, M2, M3
 *               (M2 stored [d_h, m_h]): read as the initial momentum and
 *               overwritten with the final one.  NULL = zero start, discarded.
 *   workspace   device scratch of at least ttt_layer_workspace_size() bytes,
 *               256-byte aligned, not shared with a concurrent call.
 *
 * Supported: io_dtype TTT_BF16 with d_h, m_h multiples of 64 (<= 1024) and
 * chunk a multiple of 128; io_dtype TTT_F32 with d_h, m_h <= 1024.  Other
 * requests return TTT_ERR_UNSUPPORTED.  Device pointers must be 16-byte
 * aligned.  Returns TTT_OK when the work was enqueued. */
int ttt_layer_forward(const void* q, const void* k, const void* v, const float* eta,
                      const float* W1, const float* W2, const float* W3, int w_per_batch,
                      int B, int H, int N, int d_h, int m_h, int chunk, int io_dtype,
                      int mask_mode, const unsigned char* update_chunks,
                      const ttt_update_rule* rule,
                      void* out, float* W1_final, float* W2_final, float* W3_final,
                      float* momentum, void* workspace, size_t workspace_bytes,
                      ttt_stream_t stream);

/* Bytes of device workspace ttt_layer_forward_host needs (0 if the arguments
 * are invalid): the layer workspace plus device copies of q, k, v, eta, the
 * initial and final weights, the momentum and out. */
size_t ttt_layer_host_workspace_size(int B, int H, int N, int d_h, int m_h, int chunk,
                                     int io_dtype, int mask_mode,
                                     const ttt_update_rule* rule, int w_per_batch);

/* ttt_layer_forward with every tensor in page-locked HOST memory (allocated
 * with cudaHostAlloc / cudaMallocHost or registered with cudaHostRegister):
 * the same arguments, shapes, results and support as ttt_layer_forward, with
 * q, k, v, eta, W1, W2, W3, out, W1_final, W2_final, W3_final and momentum
 * host pointers (k may equal q; momentum may be NULL).
 *
 * The call copies the weights (and momentum) to the device, then each chunk
 * of q, k, v, eta for all (batch, head) sequences on a copy stream, in chunk
 * order; the layer's launches for a chunk wait only for that chunk's copy,
 * and each chunk's output rows go back to host memory as soon as they are
 * written, so transfers in both directions overlap the kernels.  The final
 * weights (and momentum) are copied back after the last chunk.  Everything
 * is ordered on `stream`: the host results are complete when work enqueued
 * after the call on `stream` runs (e.g. after cudaStreamSynchronize).
 *
 *   workspace  device scratch of at least ttt_layer_host_workspace_size()
 *              bytes, 256-byte aligned, not shared with a concurrent call.
 *
 * Returns TTT_ERR_PAGEABLE if a host buffer is not page-locked, otherwise the
 * codes of ttt_layer_forward. */
int ttt_layer_forward_host(const void* q, const void* k, const void* v, const float* eta,
                           const float* W1, const float* W2, const float* W3, int w_per_batch,
                           int B, int H, int N, int d_h, int m_h, int chunk, int io_dtype,
                           int mask_mode, const unsigned char* update_chunks,
                           const ttt_update_rule* rule,
                           void* out, float* W1_final, float* W2_final, float* W3_final,
                           float* momentum, void* workspace, size_t workspace_bytes,
                           ttt_stream_t stream);

/* Bytes of device workspace linattn_chunked_forward needs (0 if invalid). */
size_t linattn_workspace_size(int B, int H, int N, int d_k, int d_v, int chunk,
                              int io_dtype, int mask_mode);

/* Chunked linear attention: the TTT layer with a linear fast weight
 * f_S(x) = S x, S0 initial state, dot-product loss and no normalisation
 * ("Test-Time Training with KV Binding Is Secretly Linear Attention",
 * Thm 5.2, sec. 6.1 step 6, App. H with alpha = 0).  Per chunk
 *   S <- S + sum_i eta_i v_i k_i^T   and   o_i = S q_i,
 * in the order the mask mode sets, so with S0 = 0 and block-causal order
 * o_i = sum_{chunk(j) <= chunk(i)} eta_j (q_i . k_j) v_j.
 *
 *   q, k        [B, H, N, d_k] in io_dtype;  v [B, H, N, d_v] in io_dtype.
 *   eta         [B, H, N] fp32.
 *   S0          fp32 [B, H, d_v, d_k] initial state, or NULL for zeros.
 *   update_chunks  HOST flags for TTT_STRIDED (else may be NULL).
 *   out         [B, H, N, d_v] in io_dtype.
 *   S_final     fp32 [B, H, d_v, d_k] state after the last chunk (may be NULL).
 *   workspace   at least linattn_workspace_size() bytes, 256-byte aligned.
 *
 * Supported: io_dtype TTT_BF16 with d_k, d_v multiples of 64 (<= 512) and
 * chunk a multiple of 128; io_dtype TTT_F32 with d_k, d_v <= 1024. */
int linattn_chunked_forward(const void* q, const void* k, const void* v, const float* eta,
                            const float* S0, int B, int H, int N, int d_k, int d_v,
                            int chunk, int io_dtype, int mask_mode,
                            const unsigned char* update_chunks,
                            void* out, float* S_final,
                            void* workspace, size_t workspace_bytes, ttt_stream_t stream);

/* Momentum, per-chunk learning rate and Muon of the linear-attention state
 * update: the reducible TTT variants ("Test-Time Training with KV Binding Is
 * Secretly Linear Attention", Thm 5.3 / App. D for gradient descent with a
 * per-step momentum factor, App. H for its chunk form with per-chunk
 * learning rates, App. E.3 for Muon applied to the momentum accumulator;
 * sec. 6.1 Variants 3-6 are the single-linear-layer cases).  Per (batch,
 * head) and updating chunk t, with G_t = sum over the chunk's tokens of
 * eta_i v_i k_i^T:
 *     M_t = alpha_t M_{t-1} + G_t          (M_{-1} = M0)
 *     U_t = Muon(M_t) (muon_steps > 0) or M_t
 *     S   <- S + lr_t U_t
 * Chunks a strided mask does not update leave M and S unchanged.
 *   alpha     device fp32 [B, H, N/chunk]: momentum factor of each chunk, or
 *             NULL (0: no momentum; M_t = G_t).
 *   lr        device fp32 [B, H, N/chunk]: learning rate of each chunk, or
 *             NULL (1).
 *   M0        device fp32 [B, H, d_v, d_k] initial momentum, or NULL (zeros).
 *   M_final   device fp32 [B, H, d_v, d_k]: the momentum after the last chunk,
 *             or NULL (not written).  May alias M0.
 *   muon_steps, ns_a/ns_b/ns_c: as in ttt_update_rule (Muon scales M_t to
 *             unit Frobenius norm, eps 1e-7, and orients the smaller side). */
typedef struct {
  const float* alpha;
  const float* lr;
  const float* M0;
  float* M_final;
  int muon_steps;
  float ns_a, ns_b, ns_c;
} linattn_rule;

/* Bytes of device workspace linattn_chunked_forward_rule needs (0 if the
 * arguments are invalid).  rule may be NULL (plain linear attention). */
size_t linattn_rule_workspace_size(int B, int H, int N, int d_k, int d_v, int chunk,
                                   int io_dtype, int mask_mode, const linattn_rule* rule);

/* linattn_chunked_forward with the update rule above (HOST pointer `rule`;
 * NULL, or alpha = lr = M0 = M_final = NULL with muon_steps = 0, computes
 * exactly what linattn_chunked_forward computes).  Same tensors, shapes,
 * support and status codes; alpha and lr must be 4-byte aligned, M0 and
 * M_final 16-byte aligned.  With Muon the bf16 path rounds each M_t to bf16
 * for the Newton-Schulz products (fp32 accumulation), like the layer. */
int linattn_chunked_forward_rule(const void* q, const void* k, const void* v, const float* eta,
                                 const float* S0, int B, int H, int N, int d_k, int d_v,
                                 int chunk, int io_dtype, int mask_mode,
                                 const unsigned char* update_chunks, const linattn_rule* rule,
                                 void* out, float* S_final, void* workspace,
                                 size_t workspace_bytes, ttt_stream_t stream);

/* linattn_chunked_forward for callers that cannot allocate device memory.
 * The pages have no counterpart for this call; it exists because some
 * callers cannot call cudaMalloc (a host framework that owns the GPU memory
 * pool and forbids outside allocations, or a latency-critical loop that
 * cannot afford cudaMalloc's implicit device synchronisation), so they cannot
 * provide the workspace the regular call needs.
 *
 * Same arguments and results as linattn_chunked_forward, without the
 * workspace: the scratch comes from a fixed 16 MiB array in device memory
 * that every GPU loading the library reserves until the process exits.
 * Allocates nothing.  Problems whose linattn_workspace_size() exceeds 16 MiB
 * return TTT_ERR_WORKSPACE before anything is enqueued.  The array used is
 * the CURRENT device's (cudaGetDevice), so the current device must be the
 * device of `stream` and of every tensor.  The first call on each device
 * looks up the array's device address with a runtime call (with that device
 * current), so make it before any stream capture begins.  All
 * calls share the array: calls that overlap on the GPU (e.g. concurrently on
 * two streams) race on it and must be serialised by the caller. */
int linattn_chunked_forward_noalloc(const void* q, const void* k, const void* v,
                                    const float* eta, const float* S0, int B, int H, int N,
                                    int d_k, int d_v, int chunk, int io_dtype, int mask_mode,
                                    const unsigned char* update_chunks, void* out,
                                    float* S_final, ttt_stream_t stream);

/* Synchronises `stream`, then returns and clears the device status word:
 * TTT_OK, TTT_ERR_TIMEOUT if a kernel's bounded wait ran out since the last
 * call, or TTT_ERR_CUDA if the synchronisation itself failed. */
int ttt_device_status(ttt_stream_t stream);

/* Sets the bounded-wait limit of the library's kernels in nanoseconds
 * (default 2e9).  Takes effect for launches enqueued after the call. */
void ttt_set_wait_limit_ns(unsigned long long ns);

#ifdef __cplusplus
}
#endif

#endif /* TTT_GB300_TTT_H */
