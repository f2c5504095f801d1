/*
 * mamba_oracle.c -- plain fp64 CPU oracle for the Mamba2 recurrent-state update.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls this file:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg do.  It shares no
 * code, header, table or constant with the CUDA library.
 *
 * Everything is double precision and written as the plain definition, one loop per sum,
 * with no blocking or fusion.  Inputs arrive already upcast to fp64 from the exact values
 * the GPU receives (bf16 or fp32).
 *
 * Sources (page title, section / equation):
 *  - "Hybrid SSM / Mamba models and non-KV state" (mlinterviewnotes.com):
 *      state shapes (temporal state (H, head_dim, d_state), conv state (d_conv, W-1),
 *      d_conv = d_inner + 2*g*d_state); the slot pool indexed [layer, slot, ...] with a
 *      padding slot; the decode call selective_state_update(..., D, z, dt_bias,
 *      dt_softplus=True, state_batch_indices, out); the simplified recurrence
 *      S_t = A_t (.) S_{t-1} + x_t B_t^T, y_t = S_t C_t; chunked prefill as a state
 *      hand-off (has_initial_states); align-mode checkpoints at i*block_size; the
 *      affine-composition snippet.
 *  - echobase "Mamba" notes: the Mamba block equations
 *      x = SiLU(Conv1d(x')),  Delta_t = Softplus(.),  h_t = exp(Delta_t A) h_{t-1} + Delta_t B_t x_t,
 *      y_t = C_t h_t,  y_hat = y (.) SiLU(z);  classic SSM output y_t = C h_t + D x_t;
 *      the SSD matrix form y_i = sum_{j<=i} C_i (prod_{k=j+1..i} Abar_k) Bbar_j x_j,
 *      Y = (M (.) L) X with L the causal mask.
 *
 * Readings where the pages are open (each is listed in the design notes):
 *  - Bbar_j = Delta_j * B_j (the "Delta_t B_t x_t" term), not the exact ZOH form.
 *  - y = C.h + D*x (D nullable), then y *= SiLU(z) when z is given.
 *  - softplus is exact: log(1 + e^s), evaluated stably.
 *  - heads map to groups contiguously: g(h) = h / (H/G).
 *  - xBC channel order is [x | B | C].
 *  - the conv window is oldest-first; the newest input meets w[c, W-1].
 *  - the conv state of width Wc >= W-1 holds the last Wc inputs; a step of ntok tokens
 *    shifts it left by ntok and appends the new inputs.
 *  - checkpoint k (k >= 1) is the state after the first k*interval tokens of the
 *    sequence in this call.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_EINVAL (-1)
#define OR_ENOMEM (-2)

/* ------------------------------------------------------------------------------------ */
/* scalar functions                                                                      */
/* ------------------------------------------------------------------------------------ */

/* softplus(s) = log(1 + exp(s)); written so neither branch overflows. */
static double softplus(double s) { return s > 0.0 ? s + log1p(exp(-s)) : log1p(exp(s)); }

static double sigmoid(double v) {
    if (v >= 0.0) return 1.0 / (1.0 + exp(-v));
    double e = exp(v);
    return e / (1.0 + e);
}

/* SiLU(v) = v * sigmoid(v) */
static double silu(double v) { return v * sigmoid(v); }

/* Delta for one (token, head): Delta = softplus(dt + dt_bias) when dt_softplus, else dt + dt_bias. */
static double make_delta(double dt, const double *dt_bias, int head, int dt_softplus) {
    double s = dt + (dt_bias ? dt_bias[head] : 0.0);
    return dt_softplus ? softplus(s) : s;
}

/* ------------------------------------------------------------------------------------ */
/* a small parallel-for over independent units (rows, or (sequence, head) pairs)         */
/* ------------------------------------------------------------------------------------ */

typedef void (*unit_fn)(int64_t unit, void *ctx);

struct pf_arg {
    unit_fn fn;
    void *ctx;
    int64_t n;
    int stride;
    int first;
};

static void *pf_worker(void *p) {
    struct pf_arg *a = (struct pf_arg *)p;
    for (int64_t i = a->first; i < a->n; i += a->stride) a->fn(i, a->ctx);
    return NULL;
}

#define PF_MAX_THREADS 256

static void parallel_for(int64_t n, int nthreads, unit_fn fn, void *ctx) {
    if (nthreads > PF_MAX_THREADS) nthreads = PF_MAX_THREADS;
    if (nthreads > n) nthreads = (int)n;
    if (nthreads <= 1) {
        for (int64_t i = 0; i < n; ++i) fn(i, ctx);
        return;
    }
    pthread_t th[PF_MAX_THREADS];
    struct pf_arg args[PF_MAX_THREADS];
    int started[PF_MAX_THREADS];
    for (int t = 0; t < nthreads; ++t) {
        args[t].fn = fn;
        args[t].ctx = ctx;
        args[t].n = n;
        args[t].stride = nthreads;
        args[t].first = t;
        started[t] = pthread_create(&th[t], NULL, pf_worker, &args[t]) == 0;
        if (!started[t]) pf_worker(&args[t]); /* run that share inline */
    }
    for (int t = 0; t < nthreads; ++t)
        if (started[t]) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------------------------------ */
/* decode: causal depthwise conv1d update with SiLU, one request                          */
/* ------------------------------------------------------------------------------------ */

/*
 * One request, ntok tokens, Cd channels.
 *   state: Cd x Wc, channel-major, column 0 = oldest input (Wc >= W-1).
 *   u:     ntok x Cd raw inputs.     w: Cd x W taps.     b: Cd bias or NULL.
 *   out:   ntok x Cd, SiLU(conv).
 * Token j convolves the window [last W-1 inputs before it, u_j] with w[c, 0..W-1]
 * (oldest input times w[c, 0]).  After each token the state shifts left by one and the
 * token is appended, so after ntok tokens it holds the last Wc inputs.
 */
void oracle_conv_update(int Cd, int Wc, int W, int ntok, double *state, const double *u,
                        const double *w, const double *b, double *out) {
    for (int j = 0; j < ntok; ++j) {
        for (int c = 0; c < Cd; ++c) {
            double *st = state + (int64_t)c * Wc;
            double v = b ? b[c] : 0.0;
            for (int k = 0; k < W - 1; ++k) v += w[(int64_t)c * W + k] * st[Wc - (W - 1) + k];
            v += w[(int64_t)c * W + (W - 1)] * u[(int64_t)j * Cd + c];
            out[(int64_t)j * Cd + c] = silu(v);
            for (int k = 0; k + 1 < Wc; ++k) st[k] = st[k + 1];
            st[Wc - 1] = u[(int64_t)j * Cd + c];
        }
    }
}

/* ------------------------------------------------------------------------------------ */
/* decode: the selective state update, one request                                       */
/* ------------------------------------------------------------------------------------ */

/*
 * One request, ntok tokens in order.  For token j and head hh (group g = hh / (H/G)):
 *   Delta = softplus(dt + dt_bias) (or dt + dt_bias),   a = exp(Delta * A[hh])
 *   h[p, n] <- a * h[p, n] + Delta * B[g, n] * x[p]
 *   y[p]     = sum_n C[g, n] * h[p, n] + D[hh] * x[p];   y *= SiLU(z[p]) if z
 * h: H x P x N (in/out).  h_tok (nullable): ntok x H x P x N, the state after each token.
 * x, z, y: ntok x H x P.   Bm, Cm: ntok x G x N.   dt: ntok x H.
 */
void oracle_ssm_update(int H, int P, int N, int G, int ntok, double *h, double *h_tok,
                       const double *x, const double *Bm, const double *Cm, const double *dt,
                       const double *A, const double *D, const double *dt_bias, int dt_softplus,
                       const double *z, double *y) {
    const int heads_per_group = H / G;
    const int64_t hsz = (int64_t)H * P * N;
    for (int j = 0; j < ntok; ++j) {
        for (int hh = 0; hh < H; ++hh) {
            const int g = hh / heads_per_group;
            const double delta = make_delta(dt[(int64_t)j * H + hh], dt_bias, hh, dt_softplus);
            const double a = exp(delta * A[hh]);
            const double *Bj = Bm + ((int64_t)j * G + g) * N;
            const double *Cj = Cm + ((int64_t)j * G + g) * N;
            for (int p = 0; p < P; ++p) {
                const int64_t xi = ((int64_t)j * H + hh) * P + p;
                const double xv = x[xi];
                double *hrow = h + ((int64_t)hh * P + p) * N;
                double acc = 0.0;
                for (int n = 0; n < N; ++n) {
                    hrow[n] = a * hrow[n] + delta * Bj[n] * xv;
                    acc += Cj[n] * hrow[n];
                }
                double yv = acc + (D ? D[hh] * xv : 0.0);
                if (z) yv *= silu(z[xi]);
                y[xi] = yv;
            }
        }
        if (h_tok) memcpy(h_tok + (int64_t)j * hsz, h, sizeof(double) * (size_t)hsz);
    }
}

/* ------------------------------------------------------------------------------------ */
/* Mamba1 (S6): the selective state update with a per-channel step and a (D, N) A        */
/* ------------------------------------------------------------------------------------ */

/*
 * One request of a Mamba1 layer, ntok tokens in order (echobase "Mamba" notes: the Mamba block
 * equations with B and C input dependent, h_t = exp(Delta_t A) h_{t-1} + Delta_t B_t x_t,
 * y_t = C_t h_t, y_hat = y (.) SiLU(z); the classic output adds D x_t; "Hybrid SSM / Mamba
 * models and non-KV state": the Mamba1 recurrent state has shape (D, N)).  Here every channel
 * d of the D = d_inner channels has its own step and its own row of A:
 *   Delta = softplus(dt[d] + dt_bias[d]) (or dt + dt_bias),
 *   h[d, n] <- exp(Delta * A[d, n]) * h[d, n] + Delta * B[n] * x[d],
 *   y[d] = sum_n C[n] * h[d, n] + D[d] * x[d];   y *= SiLU(z[d]) if z.
 * h: D x N (in/out).  x, dt, z, y: ntok x D.   A: D x N.   Bm, Cm: ntok x N.
 */
void oracle_mamba1_update(int D, int N, int ntok, double *h, const double *x, const double *dt,
                          const double *A, const double *Bm, const double *Cm, const double *Dskip,
                          const double *dt_bias, int dt_softplus, const double *z, double *y) {
    for (int j = 0; j < ntok; ++j) {
        for (int d = 0; d < D; ++d) {
            const double delta = make_delta(dt[(int64_t)j * D + d], dt_bias, d, dt_softplus);
            const double xv = x[(int64_t)j * D + d];
            double *hrow = h + (int64_t)d * N;
            double acc = 0.0;
            for (int n = 0; n < N; ++n) {
                hrow[n] = exp(delta * A[(int64_t)d * N + n]) * hrow[n] + delta * Bm[(int64_t)j * N + n] * xv;
                acc += Cm[(int64_t)j * N + n] * hrow[n];
            }
            double yv = acc + (Dskip ? Dskip[d] * xv : 0.0);
            if (z) yv *= silu(z[(int64_t)j * D + d]);
            y[(int64_t)j * D + d] = yv;
        }
    }
}

/* ------------------------------------------------------------------------------------ */
/* decode over a slot pool                                                               */
/* ------------------------------------------------------------------------------------ */

struct decode_ctx {
    int H, P, N, G, W, Wc, Cd, ntok;
    double *ssm_pool;
    int64_t ssm_stride;
    double *conv_pool;
    int64_t conv_stride;
    const double *conv_w, *conv_b;
    const int32_t *slot, *scratch;
    const double *xbc, *dt, *A, *D, *dt_bias, *z;
    int dt_softplus;
    double *y;
    int failed;
};

static void decode_row(int64_t i, void *vctx) {
    struct decode_ctx *c = (struct decode_ctx *)vctx;
    const int32_t s = c->slot[i];
    if (s < 0) return; /* padding row: state and output untouched */
    const int64_t HPN = (int64_t)c->H * c->P * c->N;
    const int64_t xbc_row = (int64_t)c->ntok * c->Cd;
    double *post = (double *)malloc(sizeof(double) * (size_t)xbc_row);
    double *x = (double *)malloc(sizeof(double) * (size_t)c->ntok * c->H * c->P);
    double *Bm = (double *)malloc(sizeof(double) * (size_t)c->ntok * c->G * c->N);
    double *Cm = (double *)malloc(sizeof(double) * (size_t)c->ntok * c->G * c->N);
    double *h = (double *)malloc(sizeof(double) * (size_t)HPN);
    double *h_tok = c->scratch ? (double *)malloc(sizeof(double) * (size_t)(c->ntok * HPN)) : NULL;
    if (!post || !x || !Bm || !Cm || !h || (c->scratch && !h_tok)) {
        c->failed = 1;
        goto done;
    }
    /* conv (fused) or pass-through of already convolved inputs */
    if (c->conv_pool) {
        oracle_conv_update(c->Cd, c->Wc, c->W, c->ntok, c->conv_pool + (int64_t)s * c->conv_stride,
                           c->xbc + i * xbc_row, c->conv_w, c->conv_b, post);
    } else {
        memcpy(post, c->xbc + i * xbc_row, sizeof(double) * (size_t)xbc_row);
    }
    /* split channels [x | B | C] */
    const int HP = c->H * c->P, GN = c->G * c->N;
    for (int j = 0; j < c->ntok; ++j) {
        const double *pr = post + (int64_t)j * c->Cd;
        memcpy(x + (int64_t)j * HP, pr, sizeof(double) * (size_t)HP);
        memcpy(Bm + (int64_t)j * GN, pr + HP, sizeof(double) * (size_t)GN);
        memcpy(Cm + (int64_t)j * GN, pr + HP + GN, sizeof(double) * (size_t)GN);
    }
    memcpy(h, c->ssm_pool + (int64_t)s * c->ssm_stride, sizeof(double) * (size_t)HPN);
    oracle_ssm_update(c->H, c->P, c->N, c->G, c->ntok, h, h_tok, x, Bm, Cm,
                      c->dt + i * (int64_t)c->ntok * c->H, c->A, c->D, c->dt_bias, c->dt_softplus,
                      c->z ? c->z + i * (int64_t)c->ntok * HP : NULL, c->y + i * (int64_t)c->ntok * HP);
    if (c->scratch) {
        /* speculative tokens: the state after token j goes to scratch slot j; the main slot keeps
           the state from before the step */
        for (int j = 0; j < c->ntok; ++j) {
            const int32_t d = c->scratch[i * c->ntok + j];
            if (d >= 0)
                memcpy(c->ssm_pool + (int64_t)d * c->ssm_stride, h_tok + (int64_t)j * HPN,
                       sizeof(double) * (size_t)HPN);
        }
    } else {
        memcpy(c->ssm_pool + (int64_t)s * c->ssm_stride, h, sizeof(double) * (size_t)HPN);
    }
done:
    free(post);
    free(x);
    free(Bm);
    free(Cm);
    free(h);
    free(h_tok);
}

/*
 * Batched decode over a slot pool.
 *   ssm_pool: num_slots x ssm_stride doubles, slot s holds H x P x N at s*ssm_stride.
 *   conv_pool (nullable): num_slots x conv_stride, slot s holds Cd x Wc.  When NULL, xbc is
 *     taken as already convolved (x | B | C after SiLU) and no conv state is touched.
 *   slot[batch]: pool slot per row, -1 = padding (row skipped, y row not written).
 *   scratch (nullable, batch x ntok): the state after token j of row i goes to slot
 *     scratch[i, j] and slot[i] is not written; otherwise the state after the last token is
 *     written back to slot[i].
 *   xbc: batch x ntok x Cd; dt: batch x ntok x H; z, y: batch x ntok x H x P.
 * Slot ids must be distinct and inside the pool (the caller's precondition).
 */
int oracle_decode(int H, int P, int N, int G, int W, int Wc, int ntok, int batch, double *ssm_pool,
                  int64_t ssm_stride, double *conv_pool, int64_t conv_stride, const double *conv_w,
                  const double *conv_b, const int32_t *slot, const int32_t *scratch, const double *xbc,
                  const double *dt, const double *A, const double *D, const double *dt_bias,
                  int dt_softplus, const double *z, double *y, int nthreads) {
    if (H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G || ntok <= 0 || batch < 0) return OR_EINVAL;
    if (conv_pool && (W < 1 || Wc < W - 1)) return OR_EINVAL;
    struct decode_ctx c;
    memset(&c, 0, sizeof(c));
    c.H = H; c.P = P; c.N = N; c.G = G; c.W = W; c.Wc = Wc; c.ntok = ntok;
    c.Cd = H * P + 2 * G * N;
    c.ssm_pool = ssm_pool; c.ssm_stride = ssm_stride;
    c.conv_pool = conv_pool; c.conv_stride = conv_stride;
    c.conv_w = conv_w; c.conv_b = conv_b;
    c.slot = slot; c.scratch = scratch;
    c.xbc = xbc; c.dt = dt; c.A = A; c.D = D; c.dt_bias = dt_bias; c.z = z;
    c.dt_softplus = dt_softplus; c.y = y;
    parallel_for(batch, nthreads, decode_row, &c);
    return c.failed ? OR_ENOMEM : OR_OK;
}

/*
 * Speculative commit.  Row i (slot[i] >= 0) accepted a in 0..ntok draft tokens:
 *  - a >= 1: the state after token a (scratch[i, a-1]) is copied into slot[i];
 *    a == 0 leaves slot[i] as it was before the speculative step.
 *  - the conv state, which after the speculative step holds the last Wc inputs ending at
 *    draft token ntok, is moved right by (ntok - a) columns so that its last W-1 columns
 *    end at accepted token a; the columns this frees on the left are set to zero.
 */
int oracle_spec_commit(int64_t ssm_elems, int Cd, int Wc, int ntok, int batch, double *ssm_pool,
                       int64_t ssm_stride, double *conv_pool, int64_t conv_stride,
                       const int32_t *slot, const int32_t *scratch, const int32_t *accept) {
    for (int i = 0; i < batch; ++i) {
        const int32_t s = slot[i];
        if (s < 0) continue;
        const int a = accept[i];
        if (a < 0 || a > ntok) return OR_EINVAL;
        if (a >= 1)
            memcpy(ssm_pool + (int64_t)s * ssm_stride,
                   ssm_pool + (int64_t)scratch[(int64_t)i * ntok + (a - 1)] * ssm_stride,
                   sizeof(double) * (size_t)ssm_elems);
        if (conv_pool) {
            const int shift = ntok - a;
            for (int c = 0; c < Cd; ++c) {
                double *st = conv_pool + (int64_t)s * conv_stride + (int64_t)c * Wc;
                for (int k = Wc - 1; k >= 0; --k) st[k] = (k - shift >= 0) ? st[k - shift] : 0.0;
            }
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------------------ */
/* int8 checkpoint store: per-(head, k-channel) symmetric quantisation                   */
/* ------------------------------------------------------------------------------------ */

/*
 * A cached checkpoint of the temporal state kept in int8, one scale per (head, k-channel),
 * symmetric ("Hybrid SSM / Mamba models and non-KV state", the SGLang checkpoint-store
 * paragraph: quantised once on store, dequantised once into a fresh active slot on a hit).
 * The state is H x P x N; its k-channel is the d_state index n (B_t, the key of each update
 * x_t B_t^T, runs along n), so a scale covers the P values of one (h, n):
 *     amax = max_p |state[h,p,n]|,   s[h,n] = amax / 127,   r[h,n] = 127 / amax,
 *     q[h,p,n] = clamp(rint(state[h,p,n] * r[h,n]), -127, 127)   (amax == 0: s = 0, q = 0):
 * the nearest code on the grid of step s, reached by multiplying with the reciprocal step.
 * The codes are integers decided by floating point, so this is computed in float32, the
 * precision the quantiser runs in (rint: round half to even).
 */
void oracle_int8_quantize(int H, int P, int N, const double *state, int8_t *q, float *scale) {
    for (int h = 0; h < H; ++h) {
        for (int n = 0; n < N; ++n) {
            float amax = 0.0f;
            for (int p = 0; p < P; ++p) {
                const float v = fabsf((float)state[((int64_t)h * P + p) * N + n]);
                if (v > amax) amax = v;
            }
            const float sc = amax / 127.0f;
            const float rs = amax > 0.0f ? 127.0f / amax : 0.0f;
            scale[(int64_t)h * N + n] = sc;
            for (int p = 0; p < P; ++p) {
                const int64_t i = ((int64_t)h * P + p) * N + n;
                float r = 0.0f;
                if (amax > 0.0f) {
                    r = rintf((float)state[i] * rs);
                    if (r > 127.0f) r = 127.0f;
                    if (r < -127.0f) r = -127.0f;
                }
                q[i] = (int8_t)r;
            }
        }
    }
}

/* Dequantise: state'[h,p,n] = q[h,p,n] * s[h,n], the product in float32. */
void oracle_int8_dequantize(int H, int P, int N, const int8_t *q, const float *scale, double *out) {
    for (int h = 0; h < H; ++h)
        for (int p = 0; p < P; ++p)
            for (int n = 0; n < N; ++n) {
                const int64_t i = ((int64_t)h * P + p) * N + n;
                out[i] = (double)((float)q[i] * scale[(int64_t)h * N + n]);
            }
}

/* ------------------------------------------------------------------------------------ */
/* prefill: varlen causal conv1d + SiLU, conv state read at the start and written back   */
/* ------------------------------------------------------------------------------------ */

/*
 * The conv in front of the chunked scan (x = SiLU(Conv1d(x')) of the Mamba block, applied to a
 * whole prompt; the conv state as the FIFO of the most recent inputs, continued across prefill
 * chunks like the temporal state).  Sequence s owns rows [cu[s], cu[s+1]) of u (T x Cd raw
 * inputs).  Its input stream is e_s(q) for q = -Wc .. L-1:
 *     e_s(q) = state[s, c, Wc + q]   for q < 0 when init[s] != 0 (zero when init[s] == 0),
 *     e_s(q) = u[cu[s] + q, c]       for q >= 0.
 * Token q of the sequence convolves the W inputs ending at itself:
 *     out[cu[s] + q, c] = SiLU(b_c + sum_{k=0..W-1} w[c, k] * e_s(q - (W-1) + k)).
 * On return state[s, c, i] = e_s(L - Wc + i) for i = 0..Wc-1: the last Wc inputs of the
 * stream (for L >= Wc only new inputs; an empty sequence keeps its old window, or zeros).
 *   state: nseq x Cd x Wc (oldest column first), w: Cd x W, b: Cd or NULL, out: T x Cd.
 *   init: nseq bytes or NULL (all zero).
 */
int oracle_conv_varlen(int Cd, int Wc, int W, int nseq, const int32_t *cu, const uint8_t *init,
                       double *state, const double *u, const double *w, const double *b,
                       double *out) {
    if (Cd <= 0 || W < 1 || Wc < W - 1 || nseq < 0) return OR_EINVAL;
    for (int s = 0; s < nseq; ++s)
        if (cu[s + 1] < cu[s]) return OR_EINVAL;
    double *stream = NULL;
    for (int s = 0; s < nseq; ++s) {
        const int L = cu[s + 1] - cu[s];
        const int has = init ? init[s] != 0 : 0;
        double *ns = (double *)realloc(stream, sizeof(double) * (size_t)(Wc + L));
        if (!ns) {
            free(stream);
            return OR_ENOMEM;
        }
        stream = ns;
        for (int c = 0; c < Cd; ++c) {
            double *st = state + ((int64_t)s * Cd + c) * Wc;
            /* stream[Wc + q] = e_s(q) */
            for (int i = 0; i < Wc; ++i) stream[i] = has ? st[i] : 0.0;
            for (int q = 0; q < L; ++q) stream[Wc + q] = u[((int64_t)cu[s] + q) * Cd + c];
            for (int q = 0; q < L; ++q) {
                double v = b ? b[c] : 0.0;
                for (int k = 0; k < W; ++k) v += w[(int64_t)c * W + k] * stream[Wc + q - (W - 1) + k];
                out[((int64_t)cu[s] + q) * Cd + c] = silu(v);
            }
            for (int i = 0; i < Wc; ++i) st[i] = stream[L + i];
        }
    }
    free(stream);
    return OR_OK;
}

/* ------------------------------------------------------------------------------------ */
/* prefill (i): the step recurrence, token by token                                      */
/* ------------------------------------------------------------------------------------ */

struct steps_ctx {
    int H, P, N, G, nseq;
    const int32_t *cu;
    const double *h0;
    const double *x, *dt, *A, *Bm, *Cm, *D, *dt_bias, *z;
    int dt_softplus;
    double *y, *h_final;
    int ckpt_interval, max_ckpt;
    double *h_ckpt;
};

static void steps_unit(int64_t unit, void *vctx) {
    struct steps_ctx *c = (struct steps_ctx *)vctx;
    const int s = (int)(unit / c->H), hh = (int)(unit % c->H);
    const int g = hh / (c->H / c->G);
    const int P = c->P, N = c->N, H = c->H, G = c->G;
    const int64_t PN = (int64_t)P * N;
    double *h = (double *)malloc(sizeof(double) * (size_t)PN);
    if (!h) return;
    if (c->h0)
        memcpy(h, c->h0 + ((int64_t)s * H + hh) * PN, sizeof(double) * (size_t)PN);
    else
        memset(h, 0, sizeof(double) * (size_t)PN);
    for (int32_t t = c->cu[s]; t < c->cu[s + 1]; ++t) {
        const double delta = make_delta(c->dt[(int64_t)t * H + hh], c->dt_bias, hh, c->dt_softplus);
        const double a = exp(delta * c->A[hh]);
        const double *Bt = c->Bm + ((int64_t)t * G + g) * N;
        const double *Ct = c->Cm + ((int64_t)t * G + g) * N;
        for (int p = 0; p < P; ++p) {
            const int64_t xi = ((int64_t)t * H + hh) * P + p;
            const double xv = c->x[xi];
            double acc = 0.0;
            for (int n = 0; n < N; ++n) {
                h[(int64_t)p * N + n] = a * h[(int64_t)p * N + n] + delta * Bt[n] * xv;
                acc += Ct[n] * h[(int64_t)p * N + n];
            }
            double yv = acc + (c->D ? c->D[hh] * xv : 0.0);
            if (c->z) yv *= silu(c->z[xi]);
            c->y[xi] = yv;
        }
        const int32_t done = t - c->cu[s] + 1;
        if (c->h_ckpt && c->ckpt_interval > 0 && done % c->ckpt_interval == 0) {
            const int k = done / c->ckpt_interval;
            if (k <= c->max_ckpt)
                memcpy(c->h_ckpt + (((int64_t)s * c->max_ckpt + (k - 1)) * H + hh) * PN, h,
                       sizeof(double) * (size_t)PN);
        }
    }
    memcpy(c->h_final + ((int64_t)s * H + hh) * PN, h, sizeof(double) * (size_t)PN);
    free(h);
}

/*
 * Varlen prefill by the step recurrence.  Sequence s owns tokens [cu[s], cu[s+1]).
 *   h0 (nullable): nseq x H x P x N initial states (zeros when NULL).
 *   x, z, y: T x H x P;  dt: T x H;  Bm, Cm: T x G x N.
 *   h_final: nseq x H x P x N, each sequence's state once all its tokens are consumed.
 *   h_ckpt (nullable): nseq x max_ckpt x H x P x N; entry k-1 is the state after the
 *     first k*ckpt_interval tokens of the sequence (entries past the sequence untouched).
 */
int oracle_prefill_steps(int H, int P, int N, int G, int nseq, const int32_t *cu, const double *h0,
                         const double *x, const double *dt, const double *A, const double *Bm,
                         const double *Cm, const double *D, const double *dt_bias, int dt_softplus,
                         const double *z, double *y, double *h_final, int ckpt_interval,
                         int max_ckpt, double *h_ckpt, int nthreads) {
    if (H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G || nseq < 0) return OR_EINVAL;
    for (int s = 0; s < nseq; ++s)
        if (cu[s + 1] < cu[s]) return OR_EINVAL;
    struct steps_ctx c;
    memset(&c, 0, sizeof(c));
    c.H = H; c.P = P; c.N = N; c.G = G; c.nseq = nseq; c.cu = cu; c.h0 = h0;
    c.x = x; c.dt = dt; c.A = A; c.Bm = Bm; c.Cm = Cm; c.D = D; c.dt_bias = dt_bias; c.z = z;
    c.dt_softplus = dt_softplus; c.y = y; c.h_final = h_final;
    c.ckpt_interval = ckpt_interval; c.max_ckpt = max_ckpt; c.h_ckpt = h_ckpt;
    parallel_for((int64_t)nseq * H, nthreads, steps_unit, &c);
    return OR_OK;
}

/* ------------------------------------------------------------------------------------ */
/* prefill (ii): the materialised SSD matrix form, one sequence (tiny inputs only)        */
/* ------------------------------------------------------------------------------------ */

/*
 * Y = (M (.) L) X, with, per head (group g),
 *   Abar_k = exp(Delta_k A),  Bbar_j = Delta_j B_j,
 *   M_ij   = C_i . (prod_{k=j+1..i} Abar_k) Bbar_j   for j <= i (L keeps j <= i only).
 * The initial state h0 enters as C_i (prod_{k=0..i} Abar_k) h0, and
 *   h_T = sum_j (prod_{k=j+1..T-1} Abar_k) Bbar_j x_j^T + (prod_{k=0..T-1} Abar_k) h0.
 * Every product is formed by its own explicit loop.  Cost is O(T^3) per head.
 */
int oracle_prefill_materialised(int H, int P, int N, int G, int T, const double *h0,
                                const double *x, const double *dt, const double *A,
                                const double *Bm, const double *Cm, const double *D,
                                const double *dt_bias, int dt_softplus, const double *z, double *y,
                                double *h_final) {
    if (H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G || T < 0) return OR_EINVAL;
    const int hpg = H / G;
    double *Abar = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    double *delta = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    double *L = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * (size_t)(T > 0 ? T : 1));
    if (!Abar || !delta || !L) {
        free(Abar); free(delta); free(L);
        return OR_ENOMEM;
    }
    for (int hh = 0; hh < H; ++hh) {
        const int g = hh / hpg;
        for (int t = 0; t < T; ++t) {
            delta[t] = make_delta(dt[(int64_t)t * H + hh], dt_bias, hh, dt_softplus);
            Abar[t] = exp(delta[t] * A[hh]);
        }
        /* L[i][j] = prod_{k=j+1..i} Abar_k for j <= i, else 0 (the causal mask) */
        for (int i = 0; i < T; ++i)
            for (int j = 0; j < T; ++j) {
                double prod = 0.0;
                if (j <= i) {
                    prod = 1.0;
                    for (int k = j + 1; k <= i; ++k) prod *= Abar[k];
                }
                L[(int64_t)i * T + j] = prod;
            }
        for (int i = 0; i < T; ++i) {
            const double *Ci = Cm + ((int64_t)i * G + g) * N;
            double decay0 = 1.0; /* prod_{k=0..i} Abar_k */
            for (int k = 0; k <= i; ++k) decay0 *= Abar[k];
            for (int p = 0; p < P; ++p) {
                double acc = 0.0;
                for (int j = 0; j <= i; ++j) {
                    const double *Bj = Bm + ((int64_t)j * G + g) * N;
                    double cb = 0.0;
                    for (int n = 0; n < N; ++n) cb += Ci[n] * Bj[n];
                    const double Mij = cb * L[(int64_t)i * T + j] * delta[j];
                    acc += Mij * x[((int64_t)j * H + hh) * P + p];
                }
                if (h0) {
                    double ch = 0.0;
                    for (int n = 0; n < N; ++n) ch += Ci[n] * h0[((int64_t)hh * P + p) * N + n];
                    acc += decay0 * ch;
                }
                const int64_t xi = ((int64_t)i * H + hh) * P + p;
                double yv = acc + (D ? D[hh] * x[xi] : 0.0);
                if (z) yv *= silu(z[xi]);
                y[xi] = yv;
            }
        }
        for (int p = 0; p < P; ++p)
            for (int n = 0; n < N; ++n) {
                double acc = 0.0;
                for (int j = 0; j < T; ++j) {
                    double prod = 1.0;
                    for (int k = j + 1; k <= T - 1; ++k) prod *= Abar[k];
                    acc += prod * delta[j] * Bm[((int64_t)j * G + g) * N + n] *
                           x[((int64_t)j * H + hh) * P + p];
                }
                if (h0) {
                    double prod = 1.0;
                    for (int k = 0; k <= T - 1; ++k) prod *= Abar[k];
                    acc += prod * h0[((int64_t)hh * P + p) * N + n];
                }
                h_final[((int64_t)hh * P + p) * N + n] = acc;
            }
    }
    free(Abar);
    free(delta);
    free(L);
    return OR_OK;
}

/* ------------------------------------------------------------------------------------ */
/* prefill (iii): the chunked SSD decomposition, in fp64                                 */
/* ------------------------------------------------------------------------------------ */

/*
 * One sequence of T tokens split into chunks of Q starting at its first token (the last
 * chunk may be partial).  Per head, chunk by chunk, with cum_t = sum_{k<=t in chunk} Delta_k A:
 *   diagonal block:  Y_i += sum_{j<=i in chunk} (C_i . B_j) exp(cum_i - cum_j) Delta_j x_j
 *   off-diagonal:    Y_i += exp(cum_i) C_i . h_prev
 *   chunk state:     S = sum_j exp(cum_end - cum_j) Delta_j x_j B_j^T
 *   state passing:   h = exp(cum_end) h_prev + S      (the affine composition across chunks)
 * The tensor-core prefill computes exactly these four terms per chunk.
 */
int oracle_prefill_chunked(int H, int P, int N, int G, int T, int Q, const double *h0,
                           const double *x, const double *dt, const double *A, const double *Bm,
                           const double *Cm, const double *D, const double *dt_bias, int dt_softplus,
                           const double *z, double *y, double *h_final) {
    if (H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G || T < 0 || Q <= 0) return OR_EINVAL;
    const int hpg = H / G;
    const int64_t PN = (int64_t)P * N;
    double *cum = (double *)malloc(sizeof(double) * (size_t)Q);
    double *delta = (double *)malloc(sizeof(double) * (size_t)Q);
    double *h = (double *)malloc(sizeof(double) * (size_t)PN);
    double *S = (double *)malloc(sizeof(double) * (size_t)PN);
    if (!cum || !delta || !h || !S) {
        free(cum); free(delta); free(h); free(S);
        return OR_ENOMEM;
    }
    for (int hh = 0; hh < H; ++hh) {
        const int g = hh / hpg;
        if (h0)
            memcpy(h, h0 + (int64_t)hh * PN, sizeof(double) * (size_t)PN);
        else
            memset(h, 0, sizeof(double) * (size_t)PN);
        for (int c0 = 0; c0 < T; c0 += Q) {
            const int len = (T - c0) < Q ? (T - c0) : Q;
            double run = 0.0;
            for (int t = 0; t < len; ++t) {
                delta[t] = make_delta(dt[(int64_t)(c0 + t) * H + hh], dt_bias, hh, dt_softplus);
                run += delta[t] * A[hh];
                cum[t] = run;
            }
            for (int i = 0; i < len; ++i) {
                const double *Ci = Cm + ((int64_t)(c0 + i) * G + g) * N;
                for (int p = 0; p < P; ++p) {
                    double acc = 0.0;
                    for (int j = 0; j <= i; ++j) {
                        const double *Bj = Bm + ((int64_t)(c0 + j) * G + g) * N;
                        double cb = 0.0;
                        for (int n = 0; n < N; ++n) cb += Ci[n] * Bj[n];
                        acc += cb * exp(cum[i] - cum[j]) * delta[j] *
                               x[((int64_t)(c0 + j) * H + hh) * P + p];
                    }
                    double ch = 0.0;
                    for (int n = 0; n < N; ++n) ch += Ci[n] * h[(int64_t)p * N + n];
                    acc += exp(cum[i]) * ch;
                    const int64_t xi = ((int64_t)(c0 + i) * H + hh) * P + p;
                    double yv = acc + (D ? D[hh] * x[xi] : 0.0);
                    if (z) yv *= silu(z[xi]);
                    y[xi] = yv;
                }
            }
            const double cum_end = cum[len - 1];
            for (int p = 0; p < P; ++p)
                for (int n = 0; n < N; ++n) {
                    double acc = 0.0;
                    for (int j = 0; j < len; ++j)
                        acc += exp(cum_end - cum[j]) * delta[j] *
                               x[((int64_t)(c0 + j) * H + hh) * P + p] *
                               Bm[((int64_t)(c0 + j) * G + g) * N + n];
                    S[(int64_t)p * N + n] = acc;
                }
            for (int64_t e = 0; e < PN; ++e) h[e] = exp(cum_end) * h[e] + S[e];
        }
        memcpy(h_final + (int64_t)hh * PN, h, sizeof(double) * (size_t)PN);
    }
    free(cum);
    free(delta);
    free(h);
    free(S);
    return OR_OK;
}
