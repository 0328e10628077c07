/*
 * ttt.h -- C ABI of libttt.so: the chunked inner-loop gradient-descent scan of
 * Test-Time Training (TTT) layers on NVIDIA B300 (sm_103a).
 *
 * What the library computes
 * -------------------------
 * Each (batch, head) carries fast weights W.  Tokens are taken in blocks
 * ("mini-batches") of `chunk` tokens.  Inside a block every token's
 * self-supervised loss  l = 1/2 ||f(k; W) - v||^2  is differentiated at the
 * block-start weights W0, the steps are applied in causal order, and each
 * token is read out through the weights after its own step.  In matrix
 * ("dual") form, for TTT-Linear (f(x; W) = x W):
 *
 *     E = K W0 - V
 *     Z = Q W0 - tril(eta . Q K^T) E       (mask includes the diagonal; column
 *                                          j is scaled by the key token's eta_j)
 *     W = W0 - K^T diag(eta) E             (state handed to the next block)
 *
 * Sources: "Test-Time Training Layers: How Inner-Loop Gradient Descent Replaces
 * the Transformer KV Cache with Expressive Hidden Models" (news.premlal.in),
 * section "The Core Mechanism" (loss with the factor 1/2, descent step,
 * readout through the updated weights) and section "Hardware Parallelization:
 * The Dual Form and Mini-Batch GPU Acceleration" (mini-batches of tokens);
 * the TTT essay (ren-xubin.github.io), paragraph on mini-batches and the dual
 * form (gradients at the block start, effects accumulated in causal order);
 * "Test-Time Training (TTT) Layers for Sequence Modeling" (dileepadev.github.io),
 * "Mathematical Formulation" and "Variants: TTT-Linear vs. TTT-MLP".
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All pointers are DEVICE pointers (cudaMalloc'd or equivalent) unless
 *    stated otherwise, owned by the caller.  The library allocates no device
 *    memory and keeps no per-call state.
 *  - Layouts are dense row-major: Q, K, V, Z are [B][H][T][d]; eta is
 *    [B][H][T] fp32; a weight matrix W is [B][H][d_in][d_out] fp32 with
 *    f(x; W) = x W (row = input dimension).
 *  - `dtype` is the element type of Q, K, V and Z (TTT_F32 or TTT_BF16).
 *    Fast weights and eta are always fp32.  Kernels accumulate in fp32; bf16
 *    contractions run on the tensor cores with fp32 accumulation; Z is rounded
 *    to the output type with round-to-nearest-even.
 *  - Every pointer must be 16-byte aligned.  Inputs must not overlap outputs,
 *    except where an entry point allows the state to be updated in place.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Calls are asynchronous on that stream: on TTT_OK the work has
 *    been enqueued, not finished.
 *  - Errors: a bad argument returns TTT_ERR_INVALID_ARG (or
 *    TTT_ERR_UNSUPPORTED for a well-formed shape outside the supported set)
 *    before anything is launched; a failed CUDA launch returns TTT_ERR_CUDA
 *    (text from ttt_last_error()).  A kernel never traps: a device-side
 *    fault it can detect (an expired bounded wait) is recorded in a device
 *    status word read by ttt_get_device_status().
 *  - Empty problems (B*H == 0, or T == 0) launch nothing except the copy of
 *    the initial state to the output state when T == 0 and they differ.
 */
#ifndef TTT_H_
#define TTT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ttt_status {
    TTT_OK = 0,
    TTT_ERR_INVALID_ARG = 1, /* null/misaligned pointer, negative size, bad chunk; nothing launched */
    TTT_ERR_UNSUPPORTED = 2, /* well-formed but outside the supported shapes; nothing launched */
    TTT_ERR_CUDA = 3,        /* a CUDA runtime call failed (see ttt_last_error) */
    TTT_ERR_TIMEOUT = 4      /* a bounded device-side wait expired (from ttt_get_device_status) */
} ttt_status;

typedef enum ttt_dtype {
    TTT_F32 = 0,  /* float32 Q/K/V/Z */
    TTT_BF16 = 1  /* bfloat16 Q/K/V/Z */
} ttt_dtype;

/*
 * TTT-Linear prefill: the whole chunked scan over T tokens.
 *
 *   Q, K, V  [B][H][T][d]  dtype     queries, keys (training inputs), values (targets)
 *   eta      [B][H][T]     fp32      per-token inner-loop step size
 *   W0       [B][H][d][d]  fp32      initial fast weights (input)
 *   Z        [B][H][T][d]  dtype     outputs z_t = q_t W_t (written)
 *   W_out    [B][H][d][d]  fp32      fast weights after the last token (written);
 *                                    may be the same buffer as W0 (in place)
 *   chunk    1..512; the last block may be shorter when chunk does not divide T
 *   d        16, 32, 64 or 128 (else TTT_ERR_UNSUPPORTED)
 *
 * Kernels: bf16 with 16 | chunk runs on warp-level tensor-core MMAs, for any T
 * (d = 64: one warp per 16-column group; d = 128: a recurrence warp and a
 * read-out warp per group); a shorter last block is fewer 16-token steps, a
 * partial last step weighs the tokens past T by zero.  Other shapes run on a
 * generic SIMT kernel.  The
 * environment variable TTT_LINEAR_PREFILL_KERNEL = "fused", "tc", "mma" or
 * "generic" starts the choice at that kernel ("tc": d = 64 with the read-out
 * as tcgen05 products; a kernel that does not cover the shape passes it on).
 * All give the same result up to rounding.  TTT_WAIT_LIMIT_NS (diagnostic,
 * 1 ns .. 4 s) bounds the barrier waits of the d = 64 fused kernel: a tiny
 * bound makes them expire, which exercises the failure path (TTT_ERR_TIMEOUT in
 * the device status word, every warp leaves, copies in flight are drained).
 *
 * Source: "Test-Time Training Layers ...", sections "The Core Mechanism" and
 * "Hardware Parallelization"; TTT essay, paragraph on the dual form.
 */
ttt_status ttt_linear_prefill(const void* Q, const void* K, const void* V, const float* eta,
                              const float* W0, void* Z, float* W_out, int B, int H, int T, int d,
                              int chunk, ttt_dtype dtype, void* stream);

/*
 * TTT-Linear prefill split along the sequence: the same results as
 * ttt_linear_prefill (same arguments, up to fp32 rounding), for a caller that
 * supplies scratch memory.  A block's update is affine in its start state,
 *     W <- (I - K^T diag(eta) K) W + K^T diag(eta) V,
 * so a run of whole blocks (a segment) maps its start state W_s to
 * W_s + Delta_s W_s + B_s.  Each (batch, head) is cut into S segments; the
 * maps of all segments but the last are formed in parallel (the recurrence
 * from zero with targets -K for Delta_s and V for B_s), combined in order into
 * every segment's start state (fp32), and every segment is then scanned from
 * its own start state: S times the parallelism of the one-pass scan.
 *
 *   workspace        device scratch of at least
 *                    ttt_linear_prefill_workspace_size(B, H, T, d, chunk, dtype)
 *                    bytes, 16-byte aligned, owned by the caller, not shared
 *                    with a call in flight; contents on return (fp32, P = B*H):
 *                      maps   [P][S-1][2][d][d]  Delta_s, B_s
 *                      starts [P][S][d][d]       the start state of every segment
 *                    (S is chosen from the shape and the SM count, about two
 *                    segments per SM and at least 256 tokens per segment; the
 *                    environment variable TTT_LINEAR_SEGMENTS = n asks for n.
 *                    With nblk = T / chunk blocks, a segment holds
 *                    L = ceil(nblk / n) blocks, the last one the rest, and
 *                    S = ceil(nblk / L) <= n)
 *   workspace_bytes  its size; smaller than needed: TTT_ERR_INVALID_ARG
 *
 * Shapes the split covers: bf16, d = 64, 16 | chunk, chunk | T.  For any other
 * shape, or when a single segment is best, the workspace size is 0 and the call
 * is ttt_linear_prefill (workspace may then be NULL).  W_out may be W0.
 * Source: "Test-Time Training Layers ...", sections "The Core Mechanism" (the
 * step) and "Hardware Parallelization"; TTT essay, paragraph on the dual form.
 * The affine segment maps are our parallelisation of that scan.
 */
size_t ttt_linear_prefill_workspace_size(int B, int H, int T, int d, int chunk, ttt_dtype dtype);
ttt_status ttt_linear_prefill_ws(const void* Q, const void* K, const void* V, const float* eta,
                                 const float* W0, void* Z, float* W_out, int B, int H, int T, int d,
                                 int chunk, ttt_dtype dtype, void* workspace, size_t workspace_bytes,
                                 void* stream);

/*
 * The split prefill of ttt_linear_prefill_ws for callers that cannot allocate
 * device memory when they run the scan: a serving loop that must never reach
 * the device allocator (cudaMalloc may synchronise the whole device), or code
 * whose device memory belongs to an allocator it may not go around.  Same
 * arguments and results as ttt_linear_prefill; no workspace argument, and
 * nothing is allocated by the caller or by the library.  The pages have no
 * counterpart: this is a property of the library, not of the method.
 *
 * The segment maps and start states live in a fixed 16 MiB array that every
 * GPU loading the library holds until the process exits.  A shape whose split
 * needs more than that (ttt_linear_prefill_workspace_size > 16 MiB) returns
 * TTT_ERR_UNSUPPORTED with the sizes in ttt_last_error(), before anything is
 * launched; a shape that is not split (workspace size 0) runs the one-pass
 * scan.  The first call on each device looks up the array's device address (a
 * runtime call; it is repeated if the device's context changed), so make that
 * first call before any stream capture.  All calls share the array, which keeps
 * the last call's contents (nothing in it has to start at zero): calls that
 * overlap on the GPU, from different streams or host threads, race and must be
 * serialised by the caller.
 */
ttt_status ttt_linear_prefill_noalloc(const void* Q, const void* K, const void* V, const float* eta,
                                      const float* W0, void* Z, float* W_out, int B, int H, int T,
                                      int d, int chunk, ttt_dtype dtype, void* stream);

/*
 * TTT-Linear prefill with momentum: gradient descent with momentum on the same
 * loss, every gradient taken at the block-start weights, and every token
 * taking its own step with the momentum carried from token to token and from
 * block to block:
 *
 *   g_i = k_i^T (k_i W_s - v_i)      (W_s, M_s: weights and momentum at the block start)
 *   M_i = beta M_{i-1} + g_i,   W_i = W_{i-1} - eta_i M_i,   z_i = q_i W_i
 *
 * (M_0 = M_s, W_0 = W_s).  Per block of n tokens this has the exact closed form
 *   Z = Q W_s - diag(c) Q M_s - (G . tril(Q K^T)) E,   E = K W_s - V,
 *   W = W_s - c_{n-1} M_s - K^T diag(G_{n-1,.}) E,    M = beta^n M_s + K^T diag(beta^(n-1-j)) E,
 * with c_i = sum_{l<=i} eta_l beta^(l+1) and G_ij = sum_{l=j..i} eta_l beta^(l-j) (0-based);
 * beta = 0 is ttt_linear_prefill.
 *
 *   M0       [B][H][d][d]  fp32   momentum at the start, or NULL for zero
 *   M_out    [B][H][d][d]  fp32   momentum after the last token (written; may be M0)
 *   W_out    may be W0; beta in [0, 1] (else TTT_ERR_INVALID_ARG)
 *   Other arguments as ttt_linear_prefill.  bf16 with d = 64 and chunk = 16 runs on warp-level
 *   tensor-core MMAs for any T (bf16 operands, fp32 state and momentum; a partial last chunk
 *   weighs its tokens past T by zero and decays the momentum by beta per token it holds); every
 *   other shape on the SIMT fp32 kernel.  TTT_LINEAR_MOMENTUM_KERNEL = "simt" forces the SIMT kernel.
 *
 * Source: E^2-TTT article (zhichai.net), section "Technical Details and Practical
 * Implications" (momentum gradient descent, squared loss, gradients at the
 * chunk start, fast weights and momentum carried between chunks; the closed form
 * itself is missing from the page, the recursion above is our reading of it).
 */
ttt_status ttt_linear_momentum_prefill(const void* Q, const void* K, const void* V, const float* eta,
                                       const float* W0, const float* M0, void* Z, float* W_out,
                                       float* M_out, int B, int H, int T, int d, int chunk, float beta,
                                       ttt_dtype dtype, void* stream);

/*
 * TTT-Linear prefill that also records the state at the start of every block
 * (the values ttt_linear_prefill_backward needs).  Same arguments and results
 * as ttt_linear_prefill, plus:
 *
 *   W_hist   [B][H][nblk][d][d]  dtype  written: W_hist[b][h][n] = the state at
 *                                       the start of block n (n = 0: W0),
 *                                       nblk = ceil(T / chunk)
 *
 * W_hist has the element type of Q/K/V: fp32 for TTT_F32; for TTT_BF16 the
 * state rounded to bf16 (RN-even), which is the operand the forward's products
 * used and all the backward reads (half the bytes of fp32 states).
 * W_hist must not overlap any other argument.  bf16 with d in {64, 128} and
 * chunk 16 runs the warp-MMA prefill kernels with the state writes added;
 * every other shape the SIMT kernel.
 * Source: as ttt_linear_prefill; the saved states serve the gradient below.
 */
ttt_status ttt_linear_prefill_hist(const void* Q, const void* K, const void* V, const float* eta,
                                   const float* W0, void* Z, float* W_out, void* W_hist, int B, int H,
                                   int T, int d, int chunk, ttt_dtype dtype, void* stream);

/*
 * Gradient of the TTT-Linear prefill, for training the outer model through the
 * inner loop (the slow weights learn the initialisation and the update rule:
 * TTT essay, ren-xubin.github.io, paragraph on the two time scales).  Given the
 * gradients of a scalar loss with respect to the outputs Z and to the final
 * state, returns them with respect to Q, K, V, eta and W0:
 *
 *   Q, K, V     [B][H][T][d]        dtype   the forward inputs
 *   eta         [B][H][T]           fp32
 *   W_hist      [B][H][nblk][d][d]  dtype   block-start states from ttt_linear_prefill_hist
 *   dZ          [B][H][T][d]        dtype   dL/dZ
 *   dW_T        [B][H][d][d]        fp32    dL/dW_out, or NULL for zero
 *   dQ, dK, dV  [B][H][T][d]        dtype   written: dL/dQ, dL/dK, dL/dV
 *   deta        [B][H][T]           fp32    written: dL/deta
 *   dW0         [B][H][d][d]        fp32    written: dL/dW0 (may be the same buffer as dW_T)
 *   chunk       1..512 with the block tiles in shared memory: (2 d (d+1) + 7 chunk (d+1)
 *               + 2 chunk (chunk+1) + chunk) * 4 bytes <= 227 KB (d = 64: chunk <= 64;
 *               d = 128: chunk <= 16), else TTT_ERR_UNSUPPORTED
 *   d           16, 32, 64 or 128
 *
 * Per block, reverse order (D = diag(eta), M the causal mask, S = Q K^T,
 * A = (M . S) D, E = K W - V, dW' the gradient of the state after the block):
 *   dE = -A^T dZ - D K dW',  dA = -dZ E^T,  dQ = dZ W^T + (M . dA D) K,
 *   dK = dE W^T - D E dW'^T + (M . dA D)^T Q,  dV = -dE,
 *   deta_j = -sum_c E_jc (K dW')_jc + sum_i M_ij dA_ij S_ij,
 *   dW = dW' + Q^T dZ + K^T dE.
 * Accumulation in fp32; outputs rounded to dtype (RN-even).  bf16 with d = 64
 * and chunk 16 runs on the tensor cores for any T (a partial last block weighs
 * its tokens past T by zero), every other shape on a SIMT fp32 kernel;
 * TTT_LINEAR_BACKWARD_KERNEL = "simt" forces the SIMT kernel.
 */
ttt_status ttt_linear_prefill_backward(const void* Q, const void* K, const void* V, const float* eta,
                                       const void* W_hist, const void* dZ, const float* dW_T, void* dQ,
                                       void* dK, void* dV, float* deta, float* dW0, int B, int H, int T,
                                       int d, int chunk, ttt_dtype dtype, void* stream);

/*
 * TTT-MLP prefill: f(x; W1, W2) = GELU(x W1) W2 with the tanh form of GELU,
 * no biases.  Per block, with start state (W1, W2):
 *
 *   Zk = K W1, Hk = GELU(Zk), E2 = Hk W2 - V, E1 = (E2 W2^T) . GELU'(Zk)
 *   Hq = GELU(Q W1 - tril(eta . Q K^T) E1)
 *   Z  = Hq W2 - tril(eta . Hq Hk^T) E2
 *   W1 <- W1 - K^T diag(eta) E1,   W2 <- W2 - Hk^T diag(eta) E2
 *
 *   W1_0, W1_out  [B][H][d][hidden]  fp32  (W1_out may equal W1_0)
 *   W2_0, W2_out  [B][H][hidden][d]  fp32  (W2_out may equal W2_0)
 *   d in {16, 32, 64}; hidden a multiple of 16 with d*hidden <= 16384;
 *   chunk 1..64 with chunk*hidden <= 4096 (last block may be shorter).
 *
 * Kernels: bf16 with d = 64, hidden = 256 and chunk 16 runs on warp-level
 * tensor-core MMAs for any T (a partial last block weighs its tokens past T by
 * zero); other shapes on a SIMT kernel.  TTT_MLP_PREFILL_KERNEL = "tc" selects
 * the tcgen05 form for that shape when 16 | T.
 *
 * Source: "Test-Time Training (TTT) Layers for Sequence Modeling", section
 * "Variants: TTT-Linear vs. TTT-MLP" (two-layer MLP inner model); loss, step
 * and readout as for TTT-Linear.
 */
ttt_status ttt_mlp_prefill(const void* Q, const void* K, const void* V, const float* eta,
                           const float* W1_0, const float* W2_0, void* Z, float* W1_out,
                           float* W2_out, int B, int H, int T, int d, int hidden, int chunk,
                           ttt_dtype dtype, void* stream);

/*
 * TTT-MLP prefill that also records the state at the start of every block (the
 * values ttt_mlp_prefill_backward needs).  Same arguments and results as
 * ttt_mlp_prefill, plus:
 *
 *   W1_hist  [B][H][nblk][d][hidden]  dtype  written: W1 at the start of block n
 *   W2_hist  [B][H][nblk][hidden][d]  dtype  written: W2 at the start of block n
 *                                            (n = 0: W1_0, W2_0; nblk = ceil(T / chunk))
 *
 * In the element type of Q: fp32 for TTT_F32; for TTT_BF16 the state rounded to
 * bf16 (RN-even), the operand the forward's products used.  Neither may overlap
 * another argument.  bf16 with d = 64, hidden = 256, chunk 16 runs the warp-MMA
 * kernel with the state writes added; every other shape the SIMT kernel.
 * Source: as ttt_mlp_prefill; the saved states serve the gradient below.
 */
ttt_status ttt_mlp_prefill_hist(const void* Q, const void* K, const void* V, const float* eta,
                                const float* W1_0, const float* W2_0, void* Z, float* W1_out,
                                float* W2_out, void* W1_hist, void* W2_hist, int B, int H, int T, int d,
                                int hidden, int chunk, ttt_dtype dtype, void* stream);

/*
 * Gradient of the TTT-MLP prefill (training the outer model through the inner
 * loop: TTT essay, ren-xubin.github.io, paragraph on the two time scales; the
 * two-layer inner model of "Test-Time Training (TTT) Layers for Sequence
 * Modeling", section "Variants: TTT-Linear vs. TTT-MLP").  Given the gradients
 * of a scalar loss with respect to Z and to the final W1, W2:
 *
 *   Q, K, V        [B][H][T][d]              dtype   forward inputs
 *   eta            [B][H][T]                 fp32
 *   W1_hist, W2_hist                         dtype   block-start states from ttt_mlp_prefill_hist
 *   dZ             [B][H][T][d]              dtype   dL/dZ
 *   dW1_T, dW2_T   [B][H][d][hidden], [B][H][hidden][d]  fp32  dL/dW1_out, dL/dW2_out, or NULL for zero
 *   dQ, dK, dV     [B][H][T][d]              dtype   written
 *   deta           [B][H][T]                 fp32    written
 *   dW1_0, dW2_0   fp32                              written: dL/dW1_0, dL/dW2_0 (may be dW1_T, dW2_T)
 *   shapes as ttt_mlp_prefill with chunk <= 16 (else TTT_ERR_UNSUPPORTED)
 *
 * Per block, in reverse (g = GELU, tanh form; D = diag(eta); M the causal mask):
 *   forward at the block start: Zk = K W1, Hk = g(Zk), E2 = Hk W2 - V, Gk = E2 W2^T,
 *   E1 = Gk . g'(Zk), Zq = Q W1 - (M . Q K^T) D E1, Hq = g(Zq);
 *   dW2 += Hq^T dZ + dGk^T E2 + Hk^T dE2,  dW1 += Q^T dZq + K^T dZk, with
 *   dE2 = -D Hk dW2' - (M . Hq Hk^T D)^T dZ + dGk W2,  dZq = (dZ W2^T + dS2 Hk) . g'(Zq),
 *   dE1 = -D K dW1' - (M . Q K^T D)^T dZq,  dGk = dE1 . g'(Zk),
 *   dZk = dE1 . Gk . g''(Zk) + (-D E2 dW2'^T + dS2^T Hq + dE2 W2^T) . g'(Zk),
 *   dQ = dZq W1^T + dS1 K,  dK = -D E1 dW1'^T + dS1^T Q + dZk W1^T,  dV = -dE2,
 *   with dS1 = M . (-dZq E1^T) D, dS2 = M . (-dZ E2^T) D, and deta from the same terms.
 * Accumulation in fp32, outputs rounded to dtype (RN-even). bf16 with d = 64, hidden = 256,
 * chunk = 16 (any T: a partial last block weighs its tokens past T by zero) runs on
 * warp-level tensor-core MMAs with bf16 operands (the recorded
 * states, the intermediates and a bf16 copy of the running state gradient); every other shape on
 * fp32 SIMT arithmetic. TTT_MLP_BACKWARD_KERNEL = "simt" forces the SIMT kernel.
 */
ttt_status ttt_mlp_prefill_backward(const void* Q, const void* K, const void* V, const float* eta,
                                    const void* W1_hist, const void* W2_hist, const void* dZ,
                                    const float* dW1_T, const float* dW2_T, void* dQ, void* dK, void* dV,
                                    float* deta, float* dW1_0, float* dW2_0, int B, int H, int T, int d,
                                    int hidden, int chunk, ttt_dtype dtype, void* stream);

/*
 * TTT-Linear decode: one online step (a block of one token) for every
 * (batch, head), updating the state in place:
 *
 *   e = k W - v;   W <- W - eta k^T e;   z = q W  (new W)
 *
 *   q, k, v, z  [B][H][d]     dtype
 *   eta         [B][H]        fp32
 *   W           [B][H][d][d]  fp32, read and written in place
 *   d           16, 32, 64 or 128
 *
 * Source: "Test-Time Training Layers ...", section "The Core Mechanism" and
 * the per-token forward step of its section "Python / PyTorch TTT-Linear Layer
 * Implementation".
 */
ttt_status ttt_linear_decode_step(const void* q, const void* k, const void* v, const float* eta,
                                  float* W, void* z, int B, int H, int d, ttt_dtype dtype,
                                  void* stream);

/*
 * TTT-MLP decode: one online step (a block of one token) for every
 * (batch, head), updating W1 and W2 in place; the output is read through the
 * updated weights:
 *
 *   u = k W1, a = GELU(u), e2 = a W2 - v, e1 = (e2 W2^T) . GELU'(u)
 *   W1 <- W1 - eta k^T e1,   W2 <- W2 - eta a^T e2
 *   z  = GELU(q W1) W2        (new W1, W2)
 *
 *   q, k, v, z  [B][H][d]         dtype
 *   eta         [B][H]            fp32
 *   W1          [B][H][d][hidden] fp32, read and written in place
 *   W2          [B][H][hidden][d] fp32, read and written in place
 *   d in {16, 32, 64}; hidden in {64, 128, 256} (else TTT_ERR_UNSUPPORTED)
 *
 * Source: "Test-Time Training (TTT) Layers for Sequence Modeling", section
 * "Variants: TTT-Linear vs. TTT-MLP" (two-layer MLP inner model);
 * "Test-Time Training Layers ...", section "The Core Mechanism" (loss, step,
 * read-out after the step).  The same step as ttt_mlp_prefill with chunk 1.
 */
ttt_status ttt_mlp_decode_step(const void* q, const void* k, const void* v, const float* eta, float* W1,
                               float* W2, void* z, int B, int H, int d, int hidden, ttt_dtype dtype,
                               void* stream);

/*
 * Reads and clears the device status word for the current device.
 * Synchronises `stream`.  Returns TTT_OK, or the first error a kernel
 * recorded since the last call (TTT_ERR_TIMEOUT for an expired bounded wait),
 * or TTT_ERR_CUDA if the read itself failed.
 */
ttt_status ttt_get_device_status(void* stream);

/*
 * Diagnostic: exercises the device-side failure path without faulting the GPU.
 * Launches one CTA that waits, with the bounded wait the prefill kernels use,
 * on a barrier nothing ever completes; after `limit_ns` nanoseconds (1 ns .. 2 s,
 * else TTT_ERR_INVALID_ARG) it records TTT_ERR_TIMEOUT in the device status
 * word and returns.  Asynchronous on `stream`; read the outcome with
 * ttt_get_device_status().  Not part of the computation; no page counterpart.
 */
ttt_status ttt_selftest_wait_timeout(uint64_t limit_ns, void* stream);

/* Static English text for a status code. */
const char* ttt_status_string(ttt_status s);

/* Text of the last TTT_ERR_* condition raised on the calling thread ("" if none). */
const char* ttt_last_error(void);

/* Library ABI version (major*10000 + minor*100 + patch). */
int ttt_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TTT_H_ */
