/*
 * Float64 CPU oracle of the four-layer bidirectional LSTM stack.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link,
 * load or call this file: only the test-suite, the package smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header, table or
 * constant with the CUDA library; it is written from the definition of the
 * method and nothing else.
 *
 * What it follows (pages of the speakrs 0.6.0 crate source on docs.rs):
 *  - lstmproj.rs, module docs: per layer, `x . W^T` for every step of each
 *    direction with the gate columns reordered so each hidden unit's four
 *    gates are adjacent, then a recurrence per direction; the reverse
 *    direction runs beside the forward one and the next layer takes both.
 *  - lstmproj.rs, `PackedLayer`: input width 60 for the first layer and 256
 *    after it; recurrent matrix `[2, 512, 128]`; bias `Wb + Rb`.
 *  - lstmproj.rs, `Oxide::with_recurrence` (the `pack` closure): source
 *    lengths per layer W = 2*512*input, R = 2*512*128, B = 4*512, i.e. per
 *    direction a W block `[512, input]`, an R block `[512, 128]` and a bias
 *    block `Wb[512] ++ Rb[512]`.
 *  - lstmproj.rs, `recur`: the reverse direction's hidden state goes to the
 *    output columns after the forward direction's 128.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - cell equations: the standard LSTM without peepholes, clipping or
 *    projection; gate row blocks in the order i, f, g, o;
 *  - h and c start at zero for every window, direction and layer;
 *  - the reverse direction at time t writes output row t (not time-flipped).
 *
 * Everything is plain float64 with libm exp/tanh; loops follow the
 * definition with no blocking or reordering.
 *
 * TF32 projection mode (lstmproj.rs `CudaMath::Tf32` and `projection_rule`:
 * the projection's products on TF32 tensor cores, the recurrence in FP32):
 * the `_tf32` entry points round both factors of every input-projection
 * product, W and the layer input, to TF32 before multiplying; the sums, the
 * recurrent term and the cell stay float64.  TF32 keeps fp32's sign and
 * 8-bit exponent and 10 explicit mantissa bits.  The pages do not say how
 * values are rounded to it; the reading taken is round to nearest with ties
 * away from zero, the rounding of the fp32-to-TF32 conversion instruction.  Windows are independent, so the
 * stack loop runs them (and the two directions) in parallel with OpenMP.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/*
 * v rounded to TF32 (11 significant bits: the implicit one and 10 stored),
 * to nearest, ties away from zero.  For zero and for finite values in the
 * normal fp32 range; the LSTM's weights, inputs and hidden states are.
 */
double oracle_tf32(double v)
{
    if (v == 0.0 || !isfinite(v))
        return v;
    int e;
    double m = frexp(v, &e);                   /* v = m * 2^e, 0.5 <= |m| < 1 */
    return ldexp(round(ldexp(m, 11)), e - 11); /* round(): halves away from 0 */
}

void oracle_tf32_array(long n, const double *v, double *out)
{
    for (long i = 0; i < n; ++i)
        out[i] = oracle_tf32(v[i]);
}

int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * One cell update for H units given the full pre-activation z[4H] in source
 * gate-block order (rows [0,H) input gate i, [H,2H) forget gate f,
 * [2H,3H) cell candidate g, [3H,4H) output gate o):
 *   c <- f*c + i*g,   h <- o*tanh(c).
 */
static void cell_update(int H, const double *z, double *c, double *h)
{
    for (int u = 0; u < H; ++u) {
        double i = sigmoid(z[u]);
        double f = sigmoid(z[H + u]);
        double g = tanh(z[2 * H + u]);
        double o = sigmoid(z[3 * H + u]);
        c[u] = f * c[u] + i * g;
        h[u] = o * tanh(c[u]);
    }
}

/*
 * One direction of one layer over one window of T steps.
 *   x     : step t's input at x[t*x_stride + j], j < in
 *   W     : [4H][in]   input weights, gate row blocks i,f,g,o
 *   R     : [4H][H]    recurrent weights, same row blocks
 *   Wb,Rb : [4H]       the two bias vectors; both are added
 *   h_out : step t's hidden state written at h_out[t*h_stride + u]
 * The forward direction visits t = 0..T-1, the reverse one t = T-1..0;
 * each visit uses the hidden state of the previously visited step.
 */
static void direction(int T, int in, int H,
                      const double *x, long x_stride,
                      const double *W, const double *R,
                      const double *Wb, const double *Rb,
                      int reverse, double *h_out, long h_stride, int tf32)
{
    double *z = malloc(sizeof(double) * 4 * H);
    double *h = calloc(H, sizeof(double));
    double *c = calloc(H, sizeof(double));
    for (int s = 0; s < T; ++s) {
        int t = reverse ? T - 1 - s : s;
        const double *xt = x + (long)t * x_stride;
        for (int r = 0; r < 4 * H; ++r) {
            double acc = Wb[r] + Rb[r];
            for (int j = 0; j < in; ++j)
                acc += tf32 ? oracle_tf32(W[(long)r * in + j]) * oracle_tf32(xt[j])
                            : W[(long)r * in + j] * xt[j];
            for (int j = 0; j < H; ++j)
                acc += R[(long)r * H + j] * h[j];
            z[r] = acc;
        }
        cell_update(H, z, c, h);
        memcpy(h_out + (long)t * h_stride, h, sizeof(double) * H);
    }
    free(z);
    free(h);
    free(c);
}

void oracle_lstm_direction(int T, int in, int H,
                           const double *x, long x_stride,
                           const double *W, const double *R,
                           const double *Wb, const double *Rb,
                           int reverse, double *h_out, long h_stride)
{
    direction(T, in, H, x, x_stride, W, R, Wb, Rb, reverse, h_out, h_stride, 0);
}

/*
 * The whole bidirectional stack.
 *   x      : [B][T][in0]
 *   w[l]   : [2][4H][in_l]   (in_0 = in0, in_l = 2H after the first layer)
 *   r[l]   : [2][4H][H]
 *   b[l]   : [2][8H]         per direction Wb[4H] then Rb[4H]
 *   y      : [B][T][2H]      last layer's concat(forward h, reverse h)
 * Layer l+1 reads layer l's [B][T][2H] output.
 */
static void stack(int B, int T, int in0, int H, int L,
                  const double *x,
                  const double *const *w, const double *const *r,
                  const double *const *b, double *y, int tf32)
{
    long plane = (long)B * T * 2 * H;
    double *cur = malloc(sizeof(double) * plane);
    double *nxt = malloc(sizeof(double) * plane);
    for (int l = 0; l < L; ++l) {
        int in = l == 0 ? in0 : 2 * H;
        const double *src = l == 0 ? x : cur;
        double *dst = l == L - 1 ? y : nxt;
        #pragma omp parallel for collapse(2) schedule(dynamic, 1)
        for (int bb = 0; bb < B; ++bb) {
            for (int d = 0; d < 2; ++d) {
                direction(
                    T, in, H,
                    src + (long)bb * T * in, in,
                    w[l] + (long)d * 4 * H * in,
                    r[l] + (long)d * 4 * H * H,
                    b[l] + (long)d * 8 * H,
                    b[l] + (long)d * 8 * H + 4 * H,
                    d, dst + (long)bb * T * 2 * H + d * H, 2 * H, tf32);
            }
        }
        double *t = cur; cur = nxt; nxt = t;
    }
    free(cur);
    free(nxt);
}

void oracle_lstm_stack(int B, int T, int in0, int H, int L, const double *x,
                       const double *const *w, const double *const *r,
                       const double *const *b, double *y)
{
    stack(B, T, in0, H, L, x, w, r, b, y, 0);
}

/* The stack with TF32 input-projection products (see the header). */
void oracle_lstm_stack_tf32(int B, int T, int in0, int H, int L, const double *x,
                            const double *const *w, const double *const *r,
                            const double *const *b, double *y)
{
    stack(B, T, in0, H, L, x, w, r, b, y, 1);
}

/*
 * The input projection of one layer for both directions, in the packed gate
 * column order the method uses (lstmproj.rs module docs: each hidden unit's
 * four gates adjacent).  Packed column n = d*4H + 4u + k holds, for unit u and
 * gate k (0=i, 1=f, 2=g, 3=o) of direction d, source row k*H + u:
 *   G[m][d*4H + 4u + k] = sum_j X[m][j] * W[d][k*H + u][j].
 * No bias is added here.
 *   X : [M][in],  W : [2][4H][in],  G : [M][8H]
 */
static void projection(long M, int in, int H, const double *X,
                       const double *W, double *G, int tf32)
{
    #pragma omp parallel for schedule(static)
    for (long m = 0; m < M; ++m) {
        for (int d = 0; d < 2; ++d) {
            for (int u = 0; u < H; ++u) {
                for (int k = 0; k < 4; ++k) {
                    const double *wr = W + ((long)d * 4 * H + (long)k * H + u) * in;
                    double acc = 0.0;
                    for (int j = 0; j < in; ++j)
                        acc += tf32 ? oracle_tf32(X[m * in + j]) * oracle_tf32(wr[j])
                                    : X[m * in + j] * wr[j];
                    G[m * 8 * H + d * 4 * H + 4 * u + k] = acc;
                }
            }
        }
    }
}

void oracle_projection(long M, int in, int H, const double *X, const double *W, double *G)
{
    projection(M, in, H, X, W, G, 0);
}

/* The projection with both factors of each product rounded to TF32. */
void oracle_projection_tf32(long M, int in, int H, const double *X, const double *W,
                            double *G)
{
    projection(M, in, H, X, W, G, 1);
}

/*
 * One layer's recurrence for both directions, given the projection G in the
 * packed column order above ([B*T][8H], row b*T + t):
 *   z[k*H + u] = G[b*T + t][d*4H + 4u + k] + Wb[d][k*H+u] + Rb[d][k*H+u]
 *              + sum_j R[d][k*H + u][j] * h[j]
 * then the cell update.  Output y : [B][T][2H] with direction d's hidden state
 * in columns d*H .. d*H + H - 1.
 *   R : [2][4H][H],  bias : [2][8H] (Wb then Rb per direction)
 */
void oracle_recurrence(int B, int T, int H, const double *G,
                       const double *R, const double *bias, double *y)
{
    #pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int bb = 0; bb < B; ++bb) {
        for (int d = 0; d < 2; ++d) {
            const double *Rd = R + (long)d * 4 * H * H;
            const double *Wb = bias + (long)d * 8 * H;
            const double *Rb = Wb + 4 * H;
            double *z = malloc(sizeof(double) * 4 * H);
            double *h = calloc(H, sizeof(double));
            double *c = calloc(H, sizeof(double));
            for (int s = 0; s < T; ++s) {
                int t = d ? T - 1 - s : s;
                const double *gt = G + ((long)bb * T + t) * 8 * H + d * 4 * H;
                for (int k = 0; k < 4; ++k) {
                    for (int u = 0; u < H; ++u) {
                        int row = k * H + u;
                        double acc = gt[4 * u + k] + Wb[row] + Rb[row];
                        for (int j = 0; j < H; ++j)
                            acc += Rd[(long)row * H + j] * h[j];
                        z[row] = acc;
                    }
                }
                cell_update(H, z, c, h);
                memcpy(y + ((long)bb * T + t) * 2 * H + d * H, h, sizeof(double) * H);
            }
            free(z);
            free(h);
            free(c);
        }
    }
}

/*
 * The segmentation model's dense heads on the stack output (segdense.rs,
 * `Site`: `Linear0` a row-major 256-to-128 projection `[k, n]` with bias and
 * LeakyReLU, `Linear1` 128-to-128 with bias and LeakyReLU, `Linear2` 128-to-7
 * with bias and log-softmax; `DenseOxide`: the epilogues fused), for every
 * row m < M of y [M][256]:
 *   h1 = leaky(y[m] . W0 + b0),  h2 = leaky(h1 . W1 + b1),
 *   z  = h2 . W2 + b2,           out[m] = z - log(sum_j exp(z_j)),
 * with leaky(v) = v for v >= 0 and slope * v below (the pages name LeakyReLU
 * without a slope; the reading taken is a caller-given slope, PyTorch's 0.01
 * by default).  The log-sum-exp is taken as max_j z_j + log(sum_j exp(z_j -
 * max)), the same value written so it cannot overflow.
 *   W0 : [256][128] (row k holds input k's weights to the 128 outputs),
 *   W1 : [128][128], W2 : [128][7],  out : [M][7]
 */
static double leaky(double v, double slope) { return v >= 0.0 ? v : slope * v; }

void oracle_heads(long M, const double *y, const double *W0, const double *b0,
                  const double *W1, const double *b1, const double *W2,
                  const double *b2, double slope, double *out)
{
    #pragma omp parallel for schedule(static)
    for (long m = 0; m < M; ++m) {
        double h1[128], h2[128], z[7];
        for (int n = 0; n < 128; ++n) {
            double acc = b0[n];
            for (int k = 0; k < 256; ++k)
                acc += y[m * 256 + k] * W0[k * 128 + n];
            h1[n] = leaky(acc, slope);
        }
        for (int n = 0; n < 128; ++n) {
            double acc = b1[n];
            for (int k = 0; k < 128; ++k)
                acc += h1[k] * W1[k * 128 + n];
            h2[n] = leaky(acc, slope);
        }
        double zmax = -INFINITY;
        for (int n = 0; n < 7; ++n) {
            double acc = b2[n];
            for (int k = 0; k < 128; ++k)
                acc += h2[k] * W2[k * 7 + n];
            z[n] = acc;
            if (acc > zmax)
                zmax = acc;
        }
        double s = 0.0;
        for (int n = 0; n < 7; ++n)
            s += exp(z[n] - zmax);
        const double lse = zmax + log(s);
        for (int n = 0; n < 7; ++n)
            out[m * 7 + n] = z[n] - lse;
    }
}
