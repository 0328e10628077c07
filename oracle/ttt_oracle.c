/*
 * ttt_oracle.c -- plain fp64 CPU oracle of the Test-Time Training inner loop.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the CUDA library calls, links or
 * includes this file, and the two share no code.  Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg load it.
 *
 * What is computed, and where it is stated:
 *
 *  [CM]  "Test-Time Training Layers: How Inner-Loop Gradient Descent Replaces
 *        the Transformer KV Cache with Expressive Hidden Models"
 *        (news.premlal.in), section "The Core Mechanism": the per-token loss
 *        l(W; x_t) = 1/2 ||f(k_t; W) - v_t||^2 (step 1), the descent step
 *        W_t = W_{t-1} - eta * grad_W l (step 2), and the readout
 *        y_t = f(q_t; W_t) through the weights *after* the token's own step
 *        (step 3).
 *  [HP]  same page, section "Hardware Parallelization: The Dual Form and
 *        Mini-Batch GPU Acceleration": tokens are grouped into mini-batches of
 *        b tokens.
 *  [ES]  TTT essay (ren-xubin.github.io), paragraph on mini-batches and the
 *        dual form: inside a block every gradient is taken at the block-start
 *        parameters, and the effects are accumulated in causal order.
 *  [MF]  "Test-Time Training (TTT) Layers for Sequence Modeling"
 *        (dileepadev.github.io), sections "Mathematical Formulation" and
 *        "Variants: TTT-Linear vs. TTT-MLP": f is a linear map (TTT-Linear) or
 *        a two-layer MLP (TTT-MLP).
 *
 * Readings taken where the pages are silent or disagree (each one is also
 * listed in the design notes of the repository):
 *   R1  loss carries the factor 1/2 ([CM] step 1; the dileepadev page and the
 *       essay print it without), so grad = k^T (f(k;W) - v) for TTT-Linear.
 *   R2  readout after the token's own step, so the causal mask includes the
 *       diagonal.
 *   R3  the per-token step size eta_j belongs to the key/gradient token j.
 *   R4  gradients inside a mini-batch are summed, not averaged.
 *   R5  W is stored [d_in][d_out] and f(k;W) = kW (the page code's W is the
 *       transpose of this).
 *   R6  the MLP is f(x) = GELU(x W1) W2, no biases, with the tanh form of GELU
 *       and its exact derivative.
 *   R7  a final mini-batch shorter than b is processed as a shorter block.
 *   R13 (momentum variant) every token takes its own momentum step with the gradient at the chunk
 *       start: M_i = beta M_{i-1} + g_i, W_i = W_{i-1} - eta_i M_i (see the momentum section).
 *
 * Layouts (row-major, contiguous): Q,K,V,Z [B][H][T][d]; eta [B][H][T];
 * W [B][H][d][d]; W1 [B][H][d][hd]; W2 [B][H][hd][d].  All arrays are double.
 *
 * Two evaluations are provided for each prefill variant:
 *   *_primal : the token-level definition, with every intermediate W_i formed
 *              explicitly (the loop of [CM] with gradients at the block start
 *              as in [ES]);
 *   *_dual   : the matrix ("dual") form of the same mini-batch step, written
 *              from the formulas Z = Q W0 - tril(eta . Q K^T)(K W0 - V) and
 *              W <- W0 - K^T diag(eta)(K W0 - V) and their MLP counterparts.
 * Their agreement to ~1e-12 is one of the oracle's self-checks.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* GELU, tanh form (Hendrycks & Gimpel 2016), and its exact derivative */
/* ------------------------------------------------------------------ */

static const double GELU_C = 0.79788456080286535587989211986876; /* sqrt(2/pi) */
static const double GELU_A = 0.044715;

double oracle_gelu(double x)
{
    double t = tanh(GELU_C * (x + GELU_A * x * x * x));
    return 0.5 * x * (1.0 + t);
}

/* d/dx of 0.5 x (1 + tanh(c (x + a x^3))) */
double oracle_gelu_prime(double x)
{
    double t = tanh(GELU_C * (x + GELU_A * x * x * x));
    double dinner = GELU_C * (1.0 + 3.0 * GELU_A * x * x);
    return 0.5 * (1.0 + t) + 0.5 * x * (1.0 - t * t) * dinner;
}

/* ------------------------------------------------------------------ */
/* small dense helpers (plain loops)                                   */
/* ------------------------------------------------------------------ */

/* y[n] = x[m] * A[m][n] */
static void vecmat(const double *x, const double *A, double *y, int m, int n)
{
    for (int j = 0; j < n; ++j) y[j] = 0.0;
    for (int i = 0; i < m; ++i) {
        double xi = x[i];
        const double *row = A + (size_t)i * n;
        for (int j = 0; j < n; ++j) y[j] += xi * row[j];
    }
}

/* A[m][n] -= s * x[m]^T y[n]   (rank-one update) */
static void rank1_sub(double *A, double s, const double *x, const double *y, int m, int n)
{
    for (int i = 0; i < m; ++i) {
        double sx = s * x[i];
        double *row = A + (size_t)i * n;
        for (int j = 0; j < n; ++j) row[j] -= sx * y[j];
    }
}

static double dot(const double *x, const double *y, int n)
{
    double s = 0.0;
    for (int i = 0; i < n; ++i) s += x[i] * y[i];
    return s;
}

static void *xmalloc(size_t n)
{
    void *p = malloc(n ? n : 1);
    if (!p) abort();
    return p;
}

/* ------------------------------------------------------------------ */
/* TTT-Linear                                                          */
/* ------------------------------------------------------------------ */

/*
 * Per-token gradient of l = 1/2 ||k W - v||^2 at W (R1, R5):
 *   e = k W - v,  grad = k^T e.
 * Only e is returned; the caller applies the rank-one k^T e.
 */
void oracle_linear_token_error(const double *k, const double *v, const double *W,
                               double *e, int d)
{
    vecmat(k, W, e, d, d);
    for (int j = 0; j < d; ++j) e[j] -= v[j];
}

/*
 * Token-level definition ([CM] steps 1-3, [ES]) for one (batch, head):
 * for every block of `chunk` tokens starting at state Ws,
 *   for each token i of the block:  W <- W - eta_i k_i^T (k_i Ws - v_i);
 *                                   z_i = q_i W.
 */
static void linear_primal_head(const double *Q, const double *K, const double *V,
                               const double *eta, const double *W0, double *Z,
                               double *W, int T, int d, int chunk)
{
    size_t dd = (size_t)d * d;
    double *Ws = xmalloc(dd * sizeof(double));
    double *e = xmalloc((size_t)d * sizeof(double));
    if (W != W0) memcpy(W, W0, dd * sizeof(double)); /* W may alias W0 (in-place step) */
    for (int t0 = 0; t0 < T; t0 += chunk) {
        int n = (T - t0 < chunk) ? (T - t0) : chunk; /* R7 */
        memcpy(Ws, W, dd * sizeof(double));            /* block-start state */
        for (int i = t0; i < t0 + n; ++i) {
            const double *k = K + (size_t)i * d;
            oracle_linear_token_error(k, V + (size_t)i * d, Ws, e, d); /* at Ws */
            rank1_sub(W, eta[i], k, e, d, d);                          /* step */
            vecmat(Q + (size_t)i * d, W, Z + (size_t)i * d, d, d);     /* readout */
        }
    }
    free(Ws);
    free(e);
}

/*
 * Dual (matrix) form of the same block step, per block with start state W0:
 *   E = K W0 - V                         (b x d)
 *   A = tril(Q K^T) with column j scaled by eta_j, diagonal included (R2, R3)
 *   Z = Q W0 - A E
 *   W = W0 - K^T diag(eta) E
 */
static void linear_dual_head(const double *Q, const double *K, const double *V,
                             const double *eta, const double *W0, double *Z,
                             double *W, int T, int d, int chunk)
{
    size_t dd = (size_t)d * d;
    double *E = xmalloc((size_t)chunk * d * sizeof(double));
    double *A = xmalloc((size_t)chunk * chunk * sizeof(double));
    double *Wn = xmalloc(dd * sizeof(double));
    if (W != W0) memcpy(W, W0, dd * sizeof(double));
    for (int t0 = 0; t0 < T; t0 += chunk) {
        int n = (T - t0 < chunk) ? (T - t0) : chunk;
        const double *Qc = Q + (size_t)t0 * d, *Kc = K + (size_t)t0 * d;
        const double *Vc = V + (size_t)t0 * d, *ec = eta + t0;
        double *Zc = Z + (size_t)t0 * d;
        /* E = K W0 - V */
        for (int i = 0; i < n; ++i) {
            vecmat(Kc + (size_t)i * d, W, E + (size_t)i * d, d, d);
            for (int c = 0; c < d; ++c) E[(size_t)i * d + c] -= Vc[(size_t)i * d + c];
        }
        /* A = tril(eta . Q K^T) */
        for (int i = 0; i < n; ++i)
            for (int j = 0; j < n; ++j)
                A[(size_t)i * n + j] = (j <= i) ? ec[j] * dot(Qc + (size_t)i * d, Kc + (size_t)j * d, d) : 0.0;
        /* Z = Q W0 - A E */
        for (int i = 0; i < n; ++i) {
            double *z = Zc + (size_t)i * d;
            vecmat(Qc + (size_t)i * d, W, z, d, d);
            for (int j = 0; j <= i; ++j) {
                double a = A[(size_t)i * n + j];
                const double *ej = E + (size_t)j * d;
                for (int c = 0; c < d; ++c) z[c] -= a * ej[c];
            }
        }
        /* W = W0 - K^T diag(eta) E */
        memcpy(Wn, W, dd * sizeof(double));
        for (int j = 0; j < n; ++j) rank1_sub(Wn, ec[j], Kc + (size_t)j * d, E + (size_t)j * d, d, d);
        memcpy(W, Wn, dd * sizeof(double));
    }
    free(E);
    free(A);
    free(Wn);
}

typedef void (*linear_head_fn)(const double *, const double *, const double *, const double *,
                               const double *, double *, double *, int, int, int);

static void linear_all(linear_head_fn fn, const double *Q, const double *K, const double *V,
                       const double *eta, const double *W0, double *Z, double *W,
                       int B, int H, int T, int d, int chunk)
{
    long BH = (long)B * H;
    size_t td = (size_t)T * d, dd = (size_t)d * d;
#pragma omp parallel for schedule(dynamic, 1)
    for (long bh = 0; bh < BH; ++bh)
        fn(Q + bh * td, K + bh * td, V + bh * td, eta + bh * (size_t)T, W0 + bh * dd,
           Z + bh * td, W + bh * dd, T, d, chunk);
}

void oracle_linear_primal(const double *Q, const double *K, const double *V, const double *eta,
                          const double *W0, double *Z, double *W, int B, int H, int T, int d,
                          int chunk)
{
    linear_all(linear_primal_head, Q, K, V, eta, W0, Z, W, B, H, T, d, chunk);
}

void oracle_linear_dual(const double *Q, const double *K, const double *V, const double *eta,
                        const double *W0, double *Z, double *W, int B, int H, int T, int d,
                        int chunk)
{
    linear_all(linear_dual_head, Q, K, V, eta, W0, Z, W, B, H, T, d, chunk);
}

/*
 * Gradient of the TTT-Linear chunked scan, for training the outer model through the inner
 * loop.  Given the gradients of a scalar loss with respect to the outputs, dZ [B][H][T][d], and
 * to the final state, dWT [B][H][d][d] (NULL: zero), returns the gradients with respect to the
 * inputs Q, K, V [B][H][T][d], eta [B][H][T] and W0 [B][H][d][d].
 *
 * The forward definitions are those of linear_dual_head (the dual form of the mini-batch step
 * of [HP]/[ES], readings R1-R5, R7).  Their chain rule, block by block in reverse order, with
 * W = W_n the state at the start of block n, D = diag(eta), M the causal mask (j <= i),
 * S = Q K^T, A = (M . S) D, E = K W - V and dWn1 the gradient of the state after the block:
 *   from W_{n+1} = W - K^T D E:  dW += dWn1;  dE += -D K dWn1;  dK += -D E dWn1^T;
 *                                deta_j += -sum_c E_jc (K dWn1)_jc
 *   from Z = Q W - A E:          dW += Q^T dZ;  dQ += dZ W^T;  dE += -A^T dZ;  dA = -dZ E^T
 *   from A = (M . S) D:          dS = M . dA D;  deta_j += sum_i M_ij dA_ij S_ij
 *   from S = Q K^T:              dQ += dS K;  dK += dS^T Q
 *   from E = K W - V:            dK += dE W^T;  dW += K^T dE;  dV = -dE
 * The block-start states come from a forward pass over the whole sequence first.
 * Pinned by central finite differences of the token-level definition (linear_primal_head).
 */
static void linear_backward_head(const double *Q, const double *K, const double *V,
                                 const double *eta, const double *W0, const double *dZ,
                                 const double *dWT, double *dQ, double *dK, double *dV,
                                 double *deta, double *dW0, int T, int d, int chunk)
{
    int nblk = (T + chunk - 1) / chunk;
    size_t dd = (size_t)d * d;
    double *Ws = xmalloc((size_t)(nblk + 1) * dd * sizeof(double)); /* W_0 .. W_nblk */
    double *E = xmalloc((size_t)chunk * d * sizeof(double));
    double *dE = xmalloc((size_t)chunk * d * sizeof(double));
    double *KdW = xmalloc((size_t)chunk * d * sizeof(double));
    double *S = xmalloc((size_t)chunk * chunk * sizeof(double));
    double *dA = xmalloc((size_t)chunk * chunk * sizeof(double));
    double *dW = xmalloc(dd * sizeof(double));
    double *dWp = xmalloc(dd * sizeof(double));

    /* forward: the state at the start of every block */
    memcpy(Ws, W0, dd * sizeof(double));
    for (int n = 0; n < nblk; ++n) {
        int t0 = n * chunk, b = (T - t0 < chunk) ? (T - t0) : chunk;
        const double *Kc = K + (size_t)t0 * d, *Vc = V + (size_t)t0 * d, *ec = eta + t0;
        const double *W = Ws + (size_t)n * dd;
        double *Wn = Ws + (size_t)(n + 1) * dd;
        memcpy(Wn, W, dd * sizeof(double));
        for (int j = 0; j < b; ++j) {
            vecmat(Kc + (size_t)j * d, W, E + (size_t)j * d, d, d);
            for (int c = 0; c < d; ++c) E[(size_t)j * d + c] -= Vc[(size_t)j * d + c];
        }
        for (int j = 0; j < b; ++j) rank1_sub(Wn, ec[j], &Kc[(size_t)j * d], &E[(size_t)j * d], d, d);
    }

    /* reverse */
    if (dWT) memcpy(dW, dWT, dd * sizeof(double));
    else memset(dW, 0, dd * sizeof(double));
    for (int n = nblk - 1; n >= 0; --n) {
        int t0 = n * chunk, b = (T - t0 < chunk) ? (T - t0) : chunk;
        const double *Qc = Q + (size_t)t0 * d, *Kc = K + (size_t)t0 * d;
        const double *Vc = V + (size_t)t0 * d, *ec = eta + t0, *dZc = dZ + (size_t)t0 * d;
        double *dQc = dQ + (size_t)t0 * d, *dKc = dK + (size_t)t0 * d, *dVc = dV + (size_t)t0 * d;
        double *detac = deta + t0;
        const double *W = Ws + (size_t)n * dd; /* the state at the start of block n */
        /* E = K W - V, S = Q K^T, K dWn1 */
        for (int j = 0; j < b; ++j) {
            vecmat(Kc + (size_t)j * d, W, E + (size_t)j * d, d, d);
            for (int c = 0; c < d; ++c) E[(size_t)j * d + c] -= Vc[(size_t)j * d + c];
            vecmat(Kc + (size_t)j * d, dW, KdW + (size_t)j * d, d, d);
        }
        for (int i = 0; i < b; ++i)
            for (int j = 0; j < b; ++j) S[(size_t)i * b + j] = dot(Qc + (size_t)i * d, Kc + (size_t)j * d, d);
        /* dA = -dZ E^T on the mask; dE = -A^T dZ - D K dWn1 */
        for (int i = 0; i < b; ++i)
            for (int j = 0; j < b; ++j)
                dA[(size_t)i * b + j] = (j <= i) ? -dot(dZc + (size_t)i * d, E + (size_t)j * d, d) : 0.0;
        for (int j = 0; j < b; ++j)
            for (int c = 0; c < d; ++c) {
                double acc = -ec[j] * KdW[(size_t)j * d + c];
                for (int i = j; i < b; ++i) acc -= S[(size_t)i * b + j] * ec[j] * dZc[(size_t)i * d + c];
                dE[(size_t)j * d + c] = acc;
            }
        /* dQ = dZ W^T + dS K, with dS = M . dA D */
        for (int i = 0; i < b; ++i)
            for (int k = 0; k < d; ++k) {
                double acc = dot(dZc + (size_t)i * d, W + (size_t)k * d, d);
                for (int j = 0; j <= i; ++j) acc += dA[(size_t)i * b + j] * ec[j] * Kc[(size_t)j * d + k];
                dQc[(size_t)i * d + k] = acc;
            }
        /* dK = dE W^T - D E dWn1^T + dS^T Q;  dV = -dE;  deta */
        for (int j = 0; j < b; ++j) {
            for (int k = 0; k < d; ++k) {
                double acc = dot(dE + (size_t)j * d, W + (size_t)k * d, d);
                acc -= ec[j] * dot(E + (size_t)j * d, dW + (size_t)k * d, d);
                for (int i = j; i < b; ++i) acc += dA[(size_t)i * b + j] * ec[j] * Qc[(size_t)i * d + k];
                dKc[(size_t)j * d + k] = acc;
            }
            for (int c = 0; c < d; ++c) dVc[(size_t)j * d + c] = -dE[(size_t)j * d + c];
            double de = -dot(E + (size_t)j * d, KdW + (size_t)j * d, d);
            for (int i = j; i < b; ++i) de += dA[(size_t)i * b + j] * S[(size_t)i * b + j];
            detac[j] = de;
        }
        /* dW_n = dWn1 + Q^T dZ + K^T dE */
        memcpy(dWp, dW, dd * sizeof(double));
        for (int i = 0; i < b; ++i) {
            rank1_sub(dWp, -1.0, Qc + (size_t)i * d, dZc + (size_t)i * d, d, d);
            rank1_sub(dWp, -1.0, Kc + (size_t)i * d, dE + (size_t)i * d, d, d);
        }
        memcpy(dW, dWp, dd * sizeof(double));
    }
    memcpy(dW0, dW, dd * sizeof(double));
    free(Ws);
    free(E);
    free(dE);
    free(KdW);
    free(S);
    free(dA);
    free(dW);
    free(dWp);
}

void oracle_linear_backward(const double *Q, const double *K, const double *V, const double *eta,
                            const double *W0, const double *dZ, const double *dWT, double *dQ,
                            double *dK, double *dV, double *deta, double *dW0, int B, int H, int T,
                            int d, int chunk)
{
    long BH = (long)B * H;
    size_t td = (size_t)T * d, dd = (size_t)d * d;
#pragma omp parallel for schedule(dynamic, 1)
    for (long bh = 0; bh < BH; ++bh)
        linear_backward_head(Q + bh * td, K + bh * td, V + bh * td, eta + bh * (size_t)T, W0 + bh * dd,
                             dZ + bh * td, dWT ? dWT + bh * dd : NULL, dQ + bh * td, dK + bh * td,
                             dV + bh * td, deta + bh * (size_t)T, dW0 + bh * dd, T, d, chunk);
}

/*
 * One online step (b = 1) for every (batch, head), in place on W:
 *   e = k W - v;  W <- W - eta k^T e;  z = q W.
 * This is the per-token loop of [CM]/[MF] applied to a single token.
 * q,k,v,z [B][H][d]; eta [B][H]; W [B][H][d][d].
 */
void oracle_linear_decode(const double *q, const double *k, const double *v, const double *eta,
                          double *W, double *z, int B, int H, int d)
{
    linear_all(linear_primal_head, q, k, v, eta, W, z, W, B, H, 1, d, 1);
}

/* ------------------------------------------------------------------ */
/* TTT-Linear with momentum (reading R13)                              */
/* ------------------------------------------------------------------ */

/*
 * [E2] "E^2-TTT" article (zhichai.net), section "Technical Details and Practical Implications":
 * gradient descent with momentum, squared loss, gradients computed at the chunk start, fast
 * weights W and momentum M carried from chunk to chunk (the closed form itself is missing from
 * the page).  Reading R13: every token keeps its own momentum step, with its gradient taken at
 * the chunk-start state W_s:
 *     g_i = k_i^T (k_i W_s - v_i),   M_i = beta M_{i-1} + g_i,   W_i = W_{i-1} - eta_i M_i,
 *     z_i = q_i W_i   (read-out after the token's own step, R2),
 * with M_0, W_0 the chunk-start momentum and state.  beta = 0 is the plain scan above.
 * Token-level definition, one (batch, head).
 */
static void momentum_primal_head(const double *Q, const double *K, const double *V, const double *eta,
                                 const double *W0, const double *M0, double beta, double *Z, double *W,
                                 double *M, int T, int d, int chunk)
{
    size_t dd = (size_t)d * d;
    double *Ws = xmalloc(dd * sizeof(double));
    double *e = xmalloc((size_t)d * sizeof(double));
    memcpy(W, W0, dd * sizeof(double));
    if (M0) memcpy(M, M0, dd * sizeof(double)); else memset(M, 0, dd * sizeof(double));
    for (int t0 = 0; t0 < T; t0 += chunk) {
        int n = (T - t0 < chunk) ? (T - t0) : chunk;
        memcpy(Ws, W, dd * sizeof(double));
        for (int i = t0; i < t0 + n; ++i) {
            const double *k = K + (size_t)i * d;
            oracle_linear_token_error(k, V + (size_t)i * d, Ws, e, d);   /* e = k W_s - v */
            for (size_t x = 0; x < dd; ++x) M[x] *= beta;                 /* M = beta M + k^T e */
            rank1_sub(M, -1.0, k, e, d, d);
            for (size_t x = 0; x < dd; ++x) W[x] -= eta[i] * M[x];        /* W -= eta_i M */
            vecmat(Q + (size_t)i * d, W, Z + (size_t)i * d, d, d);        /* z = q W */
        }
    }
    free(Ws);
    free(e);
}

/*
 * Closed form of one chunk (indices 1..n inside the chunk), written out from the recursion above:
 *   M_i = beta^i M_s + sum_{j<=i} beta^{i-j} g_j,
 *   W_i = W_s - c_i M_s - sum_{j<=i} G_ij k_j^T e_j,   c_i = sum_{l<=i} eta_l beta^l,
 *                                                     G_ij = sum_{l=j..i} eta_l beta^{l-j}, so
 *   Z      = Q W_s - diag(c) Q M_s - (G . M . Q K^T) E          (M the causal mask, E = K W_s - V)
 *   W_end  = W_s - c_n M_s - K^T diag(G_n.) E
 *   M_end  = beta^n M_s + K^T diag(beta^{n-j}) E.
 * With beta = 0: c = 0, G_ij = eta_j, the dual form of the plain scan.
 */
static void momentum_dual_head(const double *Q, const double *K, const double *V, const double *eta,
                               const double *W0, const double *M0, double beta, double *Z, double *W,
                               double *M, int T, int d, int chunk)
{
    size_t dd = (size_t)d * d;
    double *E = xmalloc((size_t)chunk * d * sizeof(double));
    double *G = xmalloc((size_t)chunk * chunk * sizeof(double));
    double *c = xmalloc((size_t)chunk * sizeof(double));
    double *QM = xmalloc((size_t)d * sizeof(double));
    double *Wn = xmalloc(dd * sizeof(double)), *Mn = xmalloc(dd * sizeof(double));
    memcpy(W, W0, dd * sizeof(double));
    if (M0) memcpy(M, M0, dd * sizeof(double)); else memset(M, 0, dd * sizeof(double));
    for (int t0 = 0; t0 < T; t0 += chunk) {
        int n = (T - t0 < chunk) ? (T - t0) : chunk;
        const double *Qc = Q + (size_t)t0 * d, *Kc = K + (size_t)t0 * d, *Vc = V + (size_t)t0 * d;
        const double *ec = eta + t0;
        double *Zc = Z + (size_t)t0 * d;
        for (int j = 0; j < n; ++j) {
            vecmat(Kc + (size_t)j * d, W, E + (size_t)j * d, d, d);
            for (int x = 0; x < d; ++x) E[(size_t)j * d + x] -= Vc[(size_t)j * d + x];
        }
        /* c_i and G_ij with 0-based i, j: the token at position p carries beta^(p+1) in c */
        double bp = 1.0, acc = 0.0;
        for (int i = 0; i < n; ++i) {
            bp *= beta;
            acc += ec[i] * bp;
            c[i] = acc;
        }
        for (int j = 0; j < n; ++j) {
            double g = 0.0, bl = 1.0;
            for (int i = 0; i < n; ++i) {
                if (i < j) {
                    G[(size_t)i * n + j] = 0.0;
                    continue;
                }
                g += ec[i] * bl;  /* adds eta_i beta^(i-j) */
                bl *= beta;
                G[(size_t)i * n + j] = g;
            }
        }
        for (int i = 0; i < n; ++i) {
            double *z = Zc + (size_t)i * d;
            vecmat(Qc + (size_t)i * d, W, z, d, d);
            vecmat(Qc + (size_t)i * d, M, QM, d, d);
            for (int x = 0; x < d; ++x) z[x] -= c[i] * QM[x];
            for (int j = 0; j <= i; ++j) {
                double a = G[(size_t)i * n + j] * dot(Qc + (size_t)i * d, Kc + (size_t)j * d, d);
                for (int x = 0; x < d; ++x) z[x] -= a * E[(size_t)j * d + x];
            }
        }
        memcpy(Wn, W, dd * sizeof(double));
        for (size_t x = 0; x < dd; ++x) Wn[x] -= c[n - 1] * M[x];
        double bn = 1.0;
        for (int j = 0; j < n; ++j) bn *= beta;
        for (size_t x = 0; x < dd; ++x) Mn[x] = bn * M[x];
        for (int j = 0; j < n; ++j) {
            rank1_sub(Wn, G[(size_t)(n - 1) * n + j], Kc + (size_t)j * d, E + (size_t)j * d, d, d);
            double w = 1.0;
            for (int l = j + 1; l < n; ++l) w *= beta;  /* beta^(n-1-j) */
            rank1_sub(Mn, -w, Kc + (size_t)j * d, E + (size_t)j * d, d, d);
        }
        memcpy(W, Wn, dd * sizeof(double));
        memcpy(M, Mn, dd * sizeof(double));
    }
    free(E); free(G); free(c); free(QM); free(Wn); free(Mn);
}

typedef void (*momentum_head_fn)(const double *, const double *, const double *, const double *,
                                 const double *, const double *, double, double *, double *, double *,
                                 int, int, int);

static void momentum_all(momentum_head_fn fn, const double *Q, const double *K, const double *V,
                         const double *eta, const double *W0, const double *M0, double beta, double *Z,
                         double *W, double *M, int B, int H, int T, int d, int chunk)
{
    long BH = (long)B * H;
    size_t td = (size_t)T * d, dd = (size_t)d * d;
#pragma omp parallel for schedule(dynamic, 1)
    for (long bh = 0; bh < BH; ++bh)
        fn(Q + bh * td, K + bh * td, V + bh * td, eta + bh * (size_t)T, W0 + bh * dd, M0 ? M0 + bh * dd : NULL,
           beta, Z + bh * td, W + bh * dd, M + bh * dd, T, d, chunk);
}

/* M0 may be NULL (zero momentum).  Z [B][H][T][d]; W, M [B][H][d][d] are outputs. */
void oracle_linear_momentum_primal(const double *Q, const double *K, const double *V, const double *eta,
                                   const double *W0, const double *M0, double beta, double *Z, double *W,
                                   double *M, int B, int H, int T, int d, int chunk)
{
    momentum_all(momentum_primal_head, Q, K, V, eta, W0, M0, beta, Z, W, M, B, H, T, d, chunk);
}

void oracle_linear_momentum_dual(const double *Q, const double *K, const double *V, const double *eta,
                                 const double *W0, const double *M0, double beta, double *Z, double *W,
                                 double *M, int B, int H, int T, int d, int chunk)
{
    momentum_all(momentum_dual_head, Q, K, V, eta, W0, M0, beta, Z, W, M, B, H, T, d, chunk);
}

/* ------------------------------------------------------------------ */
/* TTT-MLP:  f(x; W1, W2) = GELU(x W1) W2   (R6)                        */
/* ------------------------------------------------------------------ */

/*
 * Loss and gradient of l = 1/2 ||GELU(k W1) W2 - v||^2 for one token, by the
 * chain rule:
 *   u = k W1, a = GELU(u), p = a W2, e2 = p - v,
 *   e1 = (e2 W2^T) . GELU'(u),
 *   dl/dW2 = a^T e2,   dl/dW1 = k^T e1.
 * Outputs a [hd], e1 [hd], e2 [d]; returns the loss.
 */
double oracle_mlp_token_grad(const double *k, const double *v, const double *W1, const double *W2,
                             double *a, double *e1, double *e2, int d, int hd)
{
    double *u = xmalloc((size_t)hd * sizeof(double));
    vecmat(k, W1, u, d, hd);
    for (int m = 0; m < hd; ++m) a[m] = oracle_gelu(u[m]);
    vecmat(a, W2, e2, hd, d);
    double loss = 0.0;
    for (int c = 0; c < d; ++c) {
        e2[c] -= v[c];
        loss += 0.5 * e2[c] * e2[c];
    }
    for (int m = 0; m < hd; ++m) {
        /* (e2 W2^T)[m] = sum_c e2[c] W2[m][c] */
        double s = dot(e2, W2 + (size_t)m * d, d);
        e1[m] = s * oracle_gelu_prime(u[m]);
    }
    free(u);
    return loss;
}

/* Forward f(x; W1, W2) for one row: y[d] */
void oracle_mlp_forward(const double *x, const double *W1, const double *W2, double *y, int d,
                        int hd)
{
    double *h = xmalloc((size_t)hd * sizeof(double));
    vecmat(x, W1, h, d, hd);
    for (int m = 0; m < hd; ++m) h[m] = oracle_gelu(h[m]);
    vecmat(h, W2, y, hd, d);
    free(h);
}

/* Token-level definition for one (batch, head), gradients at the block start. */
static void mlp_primal_head(const double *Q, const double *K, const double *V, const double *eta,
                            const double *W1_0, const double *W2_0, double *Z, double *W1,
                            double *W2, int T, int d, int hd, int chunk)
{
    size_t n1 = (size_t)d * hd;
    double *W1s = xmalloc(n1 * sizeof(double)), *W2s = xmalloc(n1 * sizeof(double));
    double *a = xmalloc((size_t)hd * sizeof(double)), *e1 = xmalloc((size_t)hd * sizeof(double));
    double *e2 = xmalloc((size_t)d * sizeof(double));
    memcpy(W1, W1_0, n1 * sizeof(double));
    memcpy(W2, W2_0, n1 * sizeof(double));
    for (int t0 = 0; t0 < T; t0 += chunk) {
        int n = (T - t0 < chunk) ? (T - t0) : chunk;
        memcpy(W1s, W1, n1 * sizeof(double));
        memcpy(W2s, W2, n1 * sizeof(double));
        for (int i = t0; i < t0 + n; ++i) {
            const double *k = K + (size_t)i * d;
            oracle_mlp_token_grad(k, V + (size_t)i * d, W1s, W2s, a, e1, e2, d, hd);
            rank1_sub(W1, eta[i], k, e1, d, hd);  /* W1 -= eta k^T e1 */
            rank1_sub(W2, eta[i], a, e2, hd, d);  /* W2 -= eta a^T e2 */
            oracle_mlp_forward(Q + (size_t)i * d, W1, W2, Z + (size_t)i * d, d, hd);
        }
    }
    free(W1s); free(W2s); free(a); free(e1); free(e2);
}

/*
 * Dual form of the MLP block step, per block with start state (W1, W2):
 *   Zk = K W1, Hk = GELU(Zk), E2 = Hk W2 - V, E1 = (E2 W2^T) . GELU'(Zk)
 *   A1 = tril(eta . Q K^T)            (carries the layer-1 delta)
 *   Hq = GELU(Q W1 - A1 E1)
 *   A2 = tril(eta . Hq Hk^T)          (carries the layer-2 delta)
 *   Z  = Hq W2 - A2 E2
 *   W1 <- W1 - K^T diag(eta) E1,  W2 <- W2 - Hk^T diag(eta) E2
 */
static void mlp_dual_head(const double *Q, const double *K, const double *V, const double *eta,
                          const double *W1_0, const double *W2_0, double *Z, double *W1,
                          double *W2, int T, int d, int hd, int chunk)
{
    size_t n1 = (size_t)d * hd;
    double *Zk = xmalloc((size_t)chunk * hd * sizeof(double));
    double *Hk = xmalloc((size_t)chunk * hd * sizeof(double));
    double *E1 = xmalloc((size_t)chunk * hd * sizeof(double));
    double *E2 = xmalloc((size_t)chunk * d * sizeof(double));
    double *Hq = xmalloc((size_t)chunk * hd * sizeof(double));
    double *W1n = xmalloc(n1 * sizeof(double)), *W2n = xmalloc(n1 * sizeof(double));
    memcpy(W1, W1_0, n1 * sizeof(double));
    memcpy(W2, W2_0, n1 * sizeof(double));
    for (int t0 = 0; t0 < T; t0 += chunk) {
        int n = (T - t0 < chunk) ? (T - t0) : chunk;
        const double *Qc = Q + (size_t)t0 * d, *Kc = K + (size_t)t0 * d;
        const double *Vc = V + (size_t)t0 * d, *ec = eta + t0;
        double *Zc = Z + (size_t)t0 * d;
        for (int i = 0; i < n; ++i) {
            double *zk = Zk + (size_t)i * hd, *hk = Hk + (size_t)i * hd;
            double *e2 = E2 + (size_t)i * d, *e1 = E1 + (size_t)i * hd;
            vecmat(Kc + (size_t)i * d, W1, zk, d, hd);
            for (int m = 0; m < hd; ++m) hk[m] = oracle_gelu(zk[m]);
            vecmat(hk, W2, e2, hd, d);
            for (int c = 0; c < d; ++c) e2[c] -= Vc[(size_t)i * d + c];
            for (int m = 0; m < hd; ++m)
                e1[m] = dot(e2, W2 + (size_t)m * d, d) * oracle_gelu_prime(zk[m]);
        }
        for (int i = 0; i < n; ++i) {
            /* layer 1 through the delta carried by tril(eta . Q K^T) */
            double *hq = Hq + (size_t)i * hd;
            vecmat(Qc + (size_t)i * d, W1, hq, d, hd);
            for (int j = 0; j <= i; ++j) {
                double a1 = ec[j] * dot(Qc + (size_t)i * d, Kc + (size_t)j * d, d);
                const double *e1 = E1 + (size_t)j * hd;
                for (int m = 0; m < hd; ++m) hq[m] -= a1 * e1[m];
            }
            for (int m = 0; m < hd; ++m) hq[m] = oracle_gelu(hq[m]);
            /* layer 2 through the delta carried by tril(eta . Hq Hk^T) */
            double *z = Zc + (size_t)i * d;
            vecmat(hq, W2, z, hd, d);
            for (int j = 0; j <= i; ++j) {
                double a2 = ec[j] * dot(hq, Hk + (size_t)j * hd, hd);
                const double *e2 = E2 + (size_t)j * d;
                for (int c = 0; c < d; ++c) z[c] -= a2 * e2[c];
            }
        }
        memcpy(W1n, W1, n1 * sizeof(double));
        memcpy(W2n, W2, n1 * sizeof(double));
        for (int j = 0; j < n; ++j) {
            rank1_sub(W1n, ec[j], Kc + (size_t)j * d, E1 + (size_t)j * hd, d, hd);
            rank1_sub(W2n, ec[j], Hk + (size_t)j * hd, E2 + (size_t)j * d, hd, d);
        }
        memcpy(W1, W1n, n1 * sizeof(double));
        memcpy(W2, W2n, n1 * sizeof(double));
    }
    free(Zk); free(Hk); free(E1); free(E2); free(Hq); free(W1n); free(W2n);
}

typedef void (*mlp_head_fn)(const double *, const double *, const double *, const double *,
                            const double *, const double *, double *, double *, double *, int,
                            int, int, int);

static void mlp_all(mlp_head_fn fn, const double *Q, const double *K, const double *V,
                    const double *eta, const double *W1_0, const double *W2_0, double *Z,
                    double *W1, double *W2, int B, int H, int T, int d, int hd, int chunk)
{
    long BH = (long)B * H;
    size_t td = (size_t)T * d, n1 = (size_t)d * hd;
#pragma omp parallel for schedule(dynamic, 1)
    for (long bh = 0; bh < BH; ++bh)
        fn(Q + bh * td, K + bh * td, V + bh * td, eta + bh * (size_t)T, W1_0 + bh * n1,
           W2_0 + bh * n1, Z + bh * td, W1 + bh * n1, W2 + bh * n1, T, d, hd, chunk);
}

void oracle_mlp_primal(const double *Q, const double *K, const double *V, const double *eta,
                       const double *W1_0, const double *W2_0, double *Z, double *W1, double *W2,
                       int B, int H, int T, int d, int hd, int chunk)
{
    mlp_all(mlp_primal_head, Q, K, V, eta, W1_0, W2_0, Z, W1, W2, B, H, T, d, hd, chunk);
}

void oracle_mlp_dual(const double *Q, const double *K, const double *V, const double *eta,
                     const double *W1_0, const double *W2_0, double *Z, double *W1, double *W2,
                     int B, int H, int T, int d, int hd, int chunk)
{
    mlp_all(mlp_dual_head, Q, K, V, eta, W1_0, W2_0, Z, W1, W2, B, H, T, d, hd, chunk);
}

/* Second derivative of the tanh-form GELU: with u = c (x + a x^3), t = tanh u, u' = c (1 + 3 a x^2),
 * u'' = 6 a c x:  GELU'' = (1 - t^2) u' + 1/2 x (1 - t^2) (u'' - 2 t u'^2). */
double oracle_gelu_second(double x)
{
    double t = tanh(GELU_C * (x + GELU_A * x * x * x));
    double u1 = GELU_C * (1.0 + 3.0 * GELU_A * x * x);
    double u2 = 6.0 * GELU_A * GELU_C * x;
    double s = 1.0 - t * t;
    return s * u1 + 0.5 * x * s * (u2 - 2.0 * t * u1 * u1);
}

/* y[m] = A[m][n] x[n]   (matrix times vector) */
static void matvec(const double *A, const double *x, double *y, int m, int n)
{
    for (int i = 0; i < m; ++i) y[i] = dot(A + (size_t)i * n, x, n);
}

/*
 * Gradient of the TTT-MLP scan (outer-loop training through the inner loop: the slow weights learn
 * the initialisation and the update rule, [ES] paragraph on the two time scales).  Given dZ and the
 * gradients dW1T, dW2T of the final state (NULL: zero), returns dQ, dK, dV, deta, dW1_0, dW2_0.
 *
 * The forward is mlp_dual_head (readings R1-R7), per block with start state (W1, W2), D = diag(eta),
 * M the causal mask (j <= i), g = GELU:
 *   Zk = K W1, Hk = g(Zk), E2 = Hk W2 - V, Gk = E2 W2^T, E1 = Gk . g'(Zk),
 *   A1 = (M . Q K^T) D, Zq = Q W1 - A1 E1, Hq = g(Zq), A2 = (M . Hq Hk^T) D, Z = Hq W2 - A2 E2,
 *   W1' = W1 - K^T D E1, W2' = W2 - Hk^T D E2.
 * Its chain rule, block by block in reverse order (dW1', dW2' the gradients of the state after the
 * block; every d* accumulates):
 *   W2':  dW2 += dW2';  dHk += -D E2 dW2'^T;  dE2 += -D Hk dW2';  deta_j += -(Hk dW2')_j . E2_j
 *   W1':  dW1 += dW1';  dK += -D E1 dW1'^T;   dE1 += -D K dW1';   deta_j += -(K dW1')_j . E1_j
 *   Z:    dHq += dZ W2^T;  dW2 += Hq^T dZ;  dA2 = -dZ E2^T;  dE2 += -A2^T dZ
 *   A2:   deta_j += sum_i M_ij (Hq Hk^T)_ij dA2_ij;  dHq += (M . dA2 D) Hk;  dHk += (M . dA2 D)^T Hq
 *   Hq:   dZq = dHq . g'(Zq)
 *   Zq:   dQ += dZq W1^T;  dW1 += Q^T dZq;  dA1 = -dZq E1^T;  dE1 += -A1^T dZq
 *   A1:   deta_j += sum_i M_ij (Q K^T)_ij dA1_ij;  dQ += (M . dA1 D) K;  dK += (M . dA1 D)^T Q
 *   E1:   dGk = dE1 . g'(Zk);  dZk += dE1 . Gk . g''(Zk)
 *   Gk:   dE2 += dGk W2;  dW2 += dGk^T E2
 *   E2:   dV = -dE2;  dHk += dE2 W2^T;  dW2 += Hk^T dE2
 *   Hk:   dZk += dHk . g'(Zk)
 *   Zk:   dK += dZk W1^T;  dW1 += K^T dZk
 * The block-start states come from a forward pass over the whole sequence first.
 * Pinned by central finite differences of the token-level definition (mlp_primal_head).
 */
static void mlp_backward_head(const double *Q, const double *K, const double *V, const double *eta,
                              const double *W1_0, const double *W2_0, const double *dZ,
                              const double *dW1T, const double *dW2T, double *dQ, double *dK,
                              double *dV, double *deta, double *dW1_0, double *dW2_0, int T, int d,
                              int hd, int chunk)
{
    int nblk = (T + chunk - 1) / chunk;
    size_t n1 = (size_t)d * hd, bh_ = (size_t)chunk * hd, bd = (size_t)chunk * d, bb = (size_t)chunk * chunk;
    double *W1s = xmalloc((size_t)(nblk + 1) * n1 * sizeof(double)); /* block-start W1, W2 */
    double *W2s = xmalloc((size_t)(nblk + 1) * n1 * sizeof(double));
    double *Zk = xmalloc(bh_ * sizeof(double)), *Hk = xmalloc(bh_ * sizeof(double));
    double *Gk = xmalloc(bh_ * sizeof(double)), *E1 = xmalloc(bh_ * sizeof(double));
    double *Zq = xmalloc(bh_ * sizeof(double)), *Hq = xmalloc(bh_ * sizeof(double));
    double *dHk = xmalloc(bh_ * sizeof(double)), *dHq = xmalloc(bh_ * sizeof(double));
    double *dE1 = xmalloc(bh_ * sizeof(double)), *dZq = xmalloc(bh_ * sizeof(double));
    double *dZk = xmalloc(bh_ * sizeof(double)), *dGk = xmalloc(bh_ * sizeof(double));
    double *E2 = xmalloc(bd * sizeof(double)), *dE2 = xmalloc(bd * sizeof(double));
    double *S1 = xmalloc(bb * sizeof(double)), *S2 = xmalloc(bb * sizeof(double));
    double *dA1 = xmalloc(bb * sizeof(double)), *dA2 = xmalloc(bb * sizeof(double));
    double *dW1 = xmalloc(n1 * sizeof(double)), *dW2 = xmalloc(n1 * sizeof(double));
    double *tmp = xmalloc((size_t)(hd > d ? hd : d) * sizeof(double));

    /* forward: the state at the start of every block (the dual form of mlp_dual_head) */
    memcpy(W1s, W1_0, n1 * sizeof(double));
    memcpy(W2s, W2_0, n1 * sizeof(double));
    for (int n = 0; n < nblk; ++n) {
        int t0 = n * chunk, b = (T - t0 < chunk) ? (T - t0) : chunk;
        const double *Kc = K + (size_t)t0 * d, *Vc = V + (size_t)t0 * d, *ec = eta + t0;
        const double *W1 = W1s + (size_t)n * n1, *W2 = W2s + (size_t)n * n1;
        double *W1e = W1s + (size_t)(n + 1) * n1, *W2e = W2s + (size_t)(n + 1) * n1;
        memcpy(W1e, W1, n1 * sizeof(double));
        memcpy(W2e, W2, n1 * sizeof(double));
        for (int j = 0; j < b; ++j) {
            double *zk = Zk + (size_t)j * hd, *hk = Hk + (size_t)j * hd, *e2 = E2 + (size_t)j * d;
            vecmat(Kc + (size_t)j * d, W1, zk, d, hd);
            for (int m = 0; m < hd; ++m) hk[m] = oracle_gelu(zk[m]);
            vecmat(hk, W2, e2, hd, d);
            for (int c = 0; c < d; ++c) e2[c] -= Vc[(size_t)j * d + c];
            for (int m = 0; m < hd; ++m)
                E1[(size_t)j * hd + m] = dot(e2, W2 + (size_t)m * d, d) * oracle_gelu_prime(zk[m]);
        }
        for (int j = 0; j < b; ++j) {
            rank1_sub(W1e, ec[j], Kc + (size_t)j * d, E1 + (size_t)j * hd, d, hd);
            rank1_sub(W2e, ec[j], Hk + (size_t)j * hd, E2 + (size_t)j * d, hd, d);
        }
    }

    if (dW1T) memcpy(dW1, dW1T, n1 * sizeof(double)); else memset(dW1, 0, n1 * sizeof(double));
    if (dW2T) memcpy(dW2, dW2T, n1 * sizeof(double)); else memset(dW2, 0, n1 * sizeof(double));
    for (int n = nblk - 1; n >= 0; --n) {
        int t0 = n * chunk, b = (T - t0 < chunk) ? (T - t0) : chunk;
        const double *Qc = Q + (size_t)t0 * d, *Kc = K + (size_t)t0 * d, *Vc = V + (size_t)t0 * d;
        const double *ec = eta + t0, *dZc = dZ + (size_t)t0 * d;
        double *dQc = dQ + (size_t)t0 * d, *dKc = dK + (size_t)t0 * d, *dVc = dV + (size_t)t0 * d;
        double *detac = deta + t0;
        const double *W1 = W1s + (size_t)n * n1, *W2 = W2s + (size_t)n * n1;
        /* the block's forward quantities at its start state */
        for (int j = 0; j < b; ++j) {
            double *zk = Zk + (size_t)j * hd, *hk = Hk + (size_t)j * hd, *e2 = E2 + (size_t)j * d;
            vecmat(Kc + (size_t)j * d, W1, zk, d, hd);
            for (int m = 0; m < hd; ++m) hk[m] = oracle_gelu(zk[m]);
            vecmat(hk, W2, e2, hd, d);
            for (int c = 0; c < d; ++c) e2[c] -= Vc[(size_t)j * d + c];
            for (int m = 0; m < hd; ++m) {
                Gk[(size_t)j * hd + m] = dot(e2, W2 + (size_t)m * d, d);
                E1[(size_t)j * hd + m] = Gk[(size_t)j * hd + m] * oracle_gelu_prime(zk[m]);
            }
        }
        for (int i = 0; i < b; ++i)
            for (int j = 0; j < b; ++j) S1[(size_t)i * b + j] = dot(Qc + (size_t)i * d, Kc + (size_t)j * d, d);
        for (int i = 0; i < b; ++i) {
            double *zq = Zq + (size_t)i * hd;
            vecmat(Qc + (size_t)i * d, W1, zq, d, hd);
            for (int j = 0; j <= i; ++j) {
                double a1 = ec[j] * S1[(size_t)i * b + j];
                for (int m = 0; m < hd; ++m) zq[m] -= a1 * E1[(size_t)j * hd + m];
            }
            for (int m = 0; m < hd; ++m) Hq[(size_t)i * hd + m] = oracle_gelu(zq[m]);
        }
        for (int i = 0; i < b; ++i)
            for (int j = 0; j < b; ++j)
                S2[(size_t)i * b + j] = dot(Hq + (size_t)i * hd, Hk + (size_t)j * hd, hd);

        /* the state update: W2' = W2 - Hk^T D E2, W1' = W1 - K^T D E1 (dW1, dW2 hold dW1', dW2') */
        for (int j = 0; j < b; ++j) {
            const double *hk = Hk + (size_t)j * hd, *e2 = E2 + (size_t)j * d, *e1 = E1 + (size_t)j * hd;
            const double *kj = Kc + (size_t)j * d;
            matvec(dW2, e2, dHk + (size_t)j * hd, hd, d);                  /* (E2 dW2'^T)_j */
            for (int m = 0; m < hd; ++m) dHk[(size_t)j * hd + m] *= -ec[j];
            vecmat(hk, dW2, tmp, hd, d);                                   /* (Hk dW2')_j */
            detac[j] = -dot(tmp, e2, d);
            for (int c = 0; c < d; ++c) dE2[(size_t)j * d + c] = -ec[j] * tmp[c];
            matvec(dW1, e1, dKc + (size_t)j * d, d, hd);                   /* (E1 dW1'^T)_j */
            for (int k = 0; k < d; ++k) dKc[(size_t)j * d + k] *= -ec[j];
            vecmat(kj, dW1, tmp, d, hd);                                   /* (K dW1')_j */
            detac[j] -= dot(tmp, e1, hd);
            for (int m = 0; m < hd; ++m) dE1[(size_t)j * hd + m] = -ec[j] * tmp[m];
        }
        /* Z = Hq W2 - A2 E2 */
        for (int i = 0; i < b; ++i) {
            matvec(W2, dZc + (size_t)i * d, dHq + (size_t)i * hd, hd, d);  /* dZ W2^T */
            for (int j = 0; j < b; ++j)
                dA2[(size_t)i * b + j] = (j <= i) ? -dot(dZc + (size_t)i * d, E2 + (size_t)j * d, d) : 0.0;
        }
        for (int i = 0; i < b; ++i) rank1_sub(dW2, -1.0, Hq + (size_t)i * hd, dZc + (size_t)i * d, hd, d);
        for (int j = 0; j < b; ++j)
            for (int i = j; i < b; ++i) {
                double a2 = ec[j] * S2[(size_t)i * b + j];
                for (int c = 0; c < d; ++c) dE2[(size_t)j * d + c] -= a2 * dZc[(size_t)i * d + c];
            }
        /* A2 = (M . Hq Hk^T) D */
        for (int i = 0; i < b; ++i)
            for (int j = 0; j <= i; ++j) {
                double g = dA2[(size_t)i * b + j];
                detac[j] += g * S2[(size_t)i * b + j];
                double ds = g * ec[j];
                for (int m = 0; m < hd; ++m) {
                    dHq[(size_t)i * hd + m] += ds * Hk[(size_t)j * hd + m];
                    dHk[(size_t)j * hd + m] += ds * Hq[(size_t)i * hd + m];
                }
            }
        /* Hq = g(Zq);  Zq = Q W1 - A1 E1 */
        for (int i = 0; i < b; ++i)
            for (int m = 0; m < hd; ++m)
                dZq[(size_t)i * hd + m] = dHq[(size_t)i * hd + m] * oracle_gelu_prime(Zq[(size_t)i * hd + m]);
        for (int i = 0; i < b; ++i) {
            matvec(W1, dZq + (size_t)i * hd, dQc + (size_t)i * d, d, hd);  /* dZq W1^T */
            for (int j = 0; j < b; ++j)
                dA1[(size_t)i * b + j] = (j <= i) ? -dot(dZq + (size_t)i * hd, E1 + (size_t)j * hd, hd) : 0.0;
        }
        for (int i = 0; i < b; ++i) rank1_sub(dW1, -1.0, Qc + (size_t)i * d, dZq + (size_t)i * hd, d, hd);
        for (int j = 0; j < b; ++j)
            for (int i = j; i < b; ++i) {
                double a1 = ec[j] * S1[(size_t)i * b + j];
                for (int m = 0; m < hd; ++m) dE1[(size_t)j * hd + m] -= a1 * dZq[(size_t)i * hd + m];
            }
        /* A1 = (M . Q K^T) D */
        for (int i = 0; i < b; ++i)
            for (int j = 0; j <= i; ++j) {
                double g = dA1[(size_t)i * b + j];
                detac[j] += g * S1[(size_t)i * b + j];
                double ds = g * ec[j];
                for (int k = 0; k < d; ++k) {
                    dQc[(size_t)i * d + k] += ds * Kc[(size_t)j * d + k];
                    dKc[(size_t)j * d + k] += ds * Qc[(size_t)i * d + k];
                }
            }
        /* E1 = Gk . g'(Zk);  Gk = E2 W2^T */
        for (int j = 0; j < b; ++j)
            for (int m = 0; m < hd; ++m) {
                size_t at = (size_t)j * hd + m;
                dGk[at] = dE1[at] * oracle_gelu_prime(Zk[at]);
                dZk[at] = dE1[at] * Gk[at] * oracle_gelu_second(Zk[at]);
            }
        for (int j = 0; j < b; ++j) {
            vecmat(dGk + (size_t)j * hd, W2, tmp, hd, d);                  /* dGk W2 */
            for (int c = 0; c < d; ++c) dE2[(size_t)j * d + c] += tmp[c];
        }
        for (int j = 0; j < b; ++j) rank1_sub(dW2, -1.0, dGk + (size_t)j * hd, E2 + (size_t)j * d, hd, d);
        /* E2 = Hk W2 - V;  Hk = g(Zk);  Zk = K W1 */
        for (int j = 0; j < b; ++j) {
            for (int c = 0; c < d; ++c) dVc[(size_t)j * d + c] = -dE2[(size_t)j * d + c];
            matvec(W2, dE2 + (size_t)j * d, tmp, hd, d);                   /* dE2 W2^T */
            for (int m = 0; m < hd; ++m) {
                size_t at = (size_t)j * hd + m;
                dHk[at] += tmp[m];
                dZk[at] += dHk[at] * oracle_gelu_prime(Zk[at]);
            }
        }
        for (int j = 0; j < b; ++j) {
            rank1_sub(dW2, -1.0, Hk + (size_t)j * hd, dE2 + (size_t)j * d, hd, d);
            matvec(W1, dZk + (size_t)j * hd, tmp, d, hd);                  /* dZk W1^T */
            for (int k = 0; k < d; ++k) dKc[(size_t)j * d + k] += tmp[k];
            rank1_sub(dW1, -1.0, Kc + (size_t)j * d, dZk + (size_t)j * hd, d, hd);
        }
    }
    memcpy(dW1_0, dW1, n1 * sizeof(double));
    memcpy(dW2_0, dW2, n1 * sizeof(double));
    free(W1s); free(W2s); free(Zk); free(Hk); free(Gk); free(E1); free(Zq); free(Hq);
    free(dHk); free(dHq); free(dE1); free(dZq); free(dZk); free(dGk); free(E2); free(dE2);
    free(S1); free(S2); free(dA1); free(dA2); free(dW1); free(dW2); free(tmp);
}

void oracle_mlp_backward(const double *Q, const double *K, const double *V, const double *eta,
                         const double *W1_0, const double *W2_0, const double *dZ,
                         const double *dW1T, const double *dW2T, double *dQ, double *dK, double *dV,
                         double *deta, double *dW1_0, double *dW2_0, int B, int H, int T, int d, int hd,
                         int chunk)
{
    long BH = (long)B * H;
    size_t td = (size_t)T * d, n1 = (size_t)d * hd;
#pragma omp parallel for schedule(dynamic, 1)
    for (long bh = 0; bh < BH; ++bh)
        mlp_backward_head(Q + bh * td, K + bh * td, V + bh * td, eta + bh * (size_t)T, W1_0 + bh * n1,
                          W2_0 + bh * n1, dZ + bh * td, dW1T ? dW1T + bh * n1 : NULL,
                          dW2T ? dW2T + bh * n1 : NULL, dQ + bh * td, dK + bh * td, dV + bh * td,
                          deta + bh * (size_t)T, dW1_0 + bh * n1, dW2_0 + bh * n1, T, d, hd, chunk);
}

/* Threads OpenMP will use (1 when built without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
