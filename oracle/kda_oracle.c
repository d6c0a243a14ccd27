/*
 * kda_oracle.c -- plain, slow, sequential fp64 CPU oracle for the Kimi Delta
 * Attention (KDA) decode / spec-verify core.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * Sources (vLLM API documentation pages for Kimi-K3 specialized decode):
 *  - "vllm.models.kimi_k3.amd.specialized_decode.mono.attention.kda" (K1
 *    kda_pre), module docstring: the kda task runs the conv update of the
 *    owned channels, f_b . f_a and the lower-bound gate, the l2norm, the
 *    recurrence over the L tokens with one state written per token, then the
 *    gated RMSNorm over the head's 128 values into core_out; rounding follows
 *    the unfused path at every bf16 hand-off between the original kernels.
 *  - "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.kda.prepared"
 *    (PreparedKda): the packed projection columns (_operands), the fp32
 *    o_norm weight and the scalars (gate_lower_bound, 128**-0.5,
 *    o_norm.eps) (__init__), verify rows = requests x tokens (run).
 *
 * Every step is written out directly, one request, one token, one head, one
 * channel at a time, in fp64.  The state pool is fp32 storage; inside a step
 * the state of a (request, head) is held in fp64 and rounded to fp32 when it
 * is stored.  bf16 values are passed as their raw uint16 bit patterns.
 *
 * Readings taken where the pages are silent (each one is listed in the
 * design notes of the repository):
 *  - gate:  g = lb * sigmoid(exp(A_log[h]) * (z + dt_bias[c])), range (lb, 0)
 *           (gate_mode 0, the reading taken); gate_mode 1 is the other form the
 *           pages leave open: g = max(-exp(A_log[h]) * softplus(z + dt_bias[c]), lb).
 *  - conv:  causal depthwise, tap W-1 multiplies the current token, window
 *           oldest first; activation SiLU (act = 1) or none (act = 0, pins).
 *  - l2norm: x / sqrt(sum x^2 + 1e-6); q is scaled by 128^-0.5 afterwards.
 *  - bf16 hand-offs: conv outputs q, k, v; z = f_b . f_a; o before the norm;
 *    the final output.  Everything else stays fp64 (state stored fp32).
 *  - verify: the start state and conv window come from slot
 *    slots[r, accepted[r] - 1]; after token t both are written to slots[r, t].
 *  - slot -1 at slots[r, 0] marks a padding row / request: nothing is read or
 *    written in the caches and its output rows are zero.
 *  - state layout [pool, H, v = 128, k = 128], k contiguous; stored as fp32,
 *    or (state_bf16 = 1, the bf16 cache variant) as bf16 rounded to nearest
 *    even when a state is written -- a step always carries it in fp64.
 *  - conv_state layout [pool, 3D, W-1] (dim_first = 1) or [pool, W-1, 3D].
 *  - o_norm weight [128] shared by the heads; A_log [H]; dt_bias [D].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define HEAD_DIM 128

#define ERR_SLOT 1u     /* a slot outside [0, pool) (other than a padding -1) */
#define ERR_ACCEPTED 2u /* accepted[r] outside 1..L */

/* bf16 bit pattern -> value (exact). */
static double bf16_value(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round an fp64 value to the nearest bf16 (ties to even), directly from fp64.
 * bf16 keeps 8 significant bits; its exponent range is fp32's, so below
 * 2^-126 the spacing stays 2^-133 (subnormals).  Values that round to 2^128
 * or beyond become infinity. */
static uint16_t bf16_round(double x) {
    if (isnan(x)) return 0x7FC0;
    double ax = fabs(x), r;
    if (ax == 0.0 || isinf(ax)) {
        r = ax;
    } else {
        int e;
        frexp(ax, &e); /* ax = m * 2^e, 0.5 <= m < 1 */
        int qexp = e - 8;
        if (qexp < -133) qexp = -133;
        double quantum = ldexp(1.0, qexp);
        r = nearbyint(ax / quantum) * quantum; /* default rounding: ties to even */
        if (r >= ldexp(1.0, 128)) r = INFINITY;
    }
    float f = (float)copysign(r, x); /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof f);
    return (uint16_t)(u >> 16);
}

static double bf16_rounded(double x) { return bf16_value(bf16_round(x)); }

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }
static double softplus(double x) { return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x)); }

/* Exported so that tests can pin the rounding rule itself. */
uint16_t kda_oracle_bf16_round(double x) { return bf16_round(x); }

/* The arguments of one step, shared by its (request, head) tasks. */
typedef struct {
    int heads, W, act, gate_mode, dim_first, state_bf16, L;
    const uint16_t *conv_w, *bias, *f_b;
    const float *A_log, *dt_bias, *o_norm;
    double lb, eps;
    const uint16_t *projected;
    int64_t pitch, pool;
    uint16_t *conv_state;
    float *state_pool;
    const int32_t *slots;
    uint16_t *out;
    double *diag;
} StepArgs;

/* Working arrays of one task. */
typedef struct {
    double *qkv;    /* [L][3][128]: conv outputs of the head's q, k, v channels, bf16-rounded */
    double *g;      /* [L][128]: the head's log-decays */
    double *beta;   /* [L] */
    double *S;      /* [128 (k)][128 (v)] */
    double *window; /* [W-1] */
} TaskBuf;

/*
 * Steps 2-6 for head h of request r (rows r L .. r L + L - 1), starting from
 * slot `start`.  Every channel the task touches belongs to head h (its q, k
 * and v conv channels, its 128 decay channels, its beta column, its state
 * block and its output columns), so the tasks of one step are independent:
 * they write disjoint cache entries (distinct slots per request; a step with
 * duplicate slots is undefined).
 */
static void run_task(const StepArgs *a, int64_t r, int64_t h, int64_t start, TaskBuf *b) {
    const int64_t D = (int64_t)HEAD_DIM * a->heads, C = 3 * D, SL = a->W - 1, W = a->W, L = a->L;
    const int64_t row0 = r * L, heads = a->heads;
    const int64_t DIAG = 5 * HEAD_DIM + 1;
    const double q_scale = 1.0 / sqrt((double)HEAD_DIM);
    const uint16_t *projected = a->projected, *conv_w = a->conv_w, *bias = a->bias, *f_b = a->f_b;
    const int64_t pitch = a->pitch;
    uint16_t *conv_state = a->conv_state;
    const int dim_first = a->dim_first;
    double *window = b->window;

    /* Step 1+2: split the packed row; causal depthwise conv of the head's
     * q|k|v channels against the window of the start slot. */
    for (int kind = 0; kind < 3; ++kind)
        for (int i = 0; i < HEAD_DIM; ++i) {
            const int64_t c = kind * D + h * HEAD_DIM + i;
            for (int64_t j = 0; j < SL; ++j) {
                int64_t ix = dim_first ? (start * C + c) * SL + j : (start * SL + j) * C + c;
                window[j] = bf16_value(conv_state[ix]);
            }
            for (int64_t t = 0; t < L; ++t) {
                const double x_t = bf16_value(projected[(row0 + t) * pitch + c]);
                double y = bias ? bf16_value(bias[c]) : 0.0;
                for (int64_t j = 0; j < W; ++j) {
                    const double x = (j < SL) ? window[j] : x_t; /* tap W-1 = current token */
                    y += bf16_value(conv_w[c * W + j]) * x;
                }
                if (a->act) y = y * sigmoid(y); /* SiLU */
                b->qkv[(t * 3 + kind) * HEAD_DIM + i] = bf16_rounded(y);
                /* shift the window by one and store it in this token's slot */
                for (int64_t j = 0; j + 1 < SL; ++j) window[j] = window[j + 1];
                if (SL > 0) window[SL - 1] = x_t;
                const int64_t dst = a->slots[row0 + t];
                for (int64_t j = 0; j < SL; ++j) {
                    int64_t ix = dim_first ? (dst * C + c) * SL + j : (dst * SL + j) * C + c;
                    conv_state[ix] = bf16_round(window[j]);
                }
            }
        }

    /* Step 3: gates.  z = f_b . f_a (bf16 hand-off), lower-bounded decay, beta. */
    const double lb = a->lb;
    for (int64_t t = 0; t < L; ++t) {
        const uint16_t *prow = projected + (row0 + t) * pitch;
        for (int i = 0; i < HEAD_DIM; ++i) {
            const int64_t c = h * HEAD_DIM + i;
            double z = 0.0;
            for (int64_t j = 0; j < HEAD_DIM; ++j)
                z += bf16_value(f_b[c * HEAD_DIM + j]) * bf16_value(prow[4 * D + j]);
            z = bf16_rounded(z);
            if (a->gate_mode == 0)
                b->g[t * HEAD_DIM + i] = (double)lb * sigmoid(exp((double)a->A_log[h]) * (z + (double)a->dt_bias[c]));
            else
                b->g[t * HEAD_DIM + i] = fmax(-exp((double)a->A_log[h]) * softplus(z + a->dt_bias[c]), (double)lb);
        }
        b->beta[t] = sigmoid(bf16_value(prow[4 * D + HEAD_DIM + h]));
    }

    /* Start state of (request, head), storage [v][k] -> S[k][v]. */
    double *S = b->S;
    const float *src = a->state_pool + (start * heads + h) * HEAD_DIM * HEAD_DIM;
    const uint16_t *src16 = (const uint16_t *)a->state_pool + (start * heads + h) * HEAD_DIM * HEAD_DIM;
    for (int v = 0; v < HEAD_DIM; ++v)
        for (int k = 0; k < HEAD_DIM; ++k) {
            if (a->state_bf16) S[k * HEAD_DIM + v] = bf16_value(src16[v * HEAD_DIM + k]);
            else S[k * HEAD_DIM + v] = (double)src[v * HEAD_DIM + k];
        }

    for (int64_t t = 0; t < L; ++t) {
        const double *qr = b->qkv + (t * 3 + 0) * HEAD_DIM;
        const double *kr = b->qkv + (t * 3 + 1) * HEAD_DIM;
        const double *vr = b->qkv + (t * 3 + 2) * HEAD_DIM;
        const double *gr = b->g + t * HEAD_DIM;
        const double bt = b->beta[t];

        /* Step 4: L2 normalisation of q and k, q scaled by 128^-0.5. */
        double qq = 0.0, kk = 0.0;
        for (int i = 0; i < HEAD_DIM; ++i) { qq += qr[i] * qr[i]; kk += kr[i] * kr[i]; }
        const double qn = 1.0 / sqrt(qq + 1e-6), kn = 1.0 / sqrt(kk + 1e-6);
        double qh[HEAD_DIM], kh[HEAD_DIM], o[HEAD_DIM], u[HEAD_DIM];
        for (int i = 0; i < HEAD_DIM; ++i) { qh[i] = qr[i] * qn * q_scale; kh[i] = kr[i] * kn; }

        /* Step 5: gated delta rule.  S <- diag(e^g) S;  u = v - S^T k^;
         * S <- S + beta k^ u^T;  o = S^T q^ (the updated state). */
        for (int k = 0; k < HEAD_DIM; ++k) {
            const double decay = exp(gr[k]);
            for (int v = 0; v < HEAD_DIM; ++v) S[k * HEAD_DIM + v] *= decay;
        }
        for (int v = 0; v < HEAD_DIM; ++v) {
            double s = 0.0;
            for (int k = 0; k < HEAD_DIM; ++k) s += S[k * HEAD_DIM + v] * kh[k];
            u[v] = vr[v] - s;
        }
        for (int k = 0; k < HEAD_DIM; ++k)
            for (int v = 0; v < HEAD_DIM; ++v) S[k * HEAD_DIM + v] += bt * kh[k] * u[v];
        for (int v = 0; v < HEAD_DIM; ++v) {
            double s = 0.0;
            for (int k = 0; k < HEAD_DIM; ++k) s += S[k * HEAD_DIM + v] * qh[k];
            o[v] = bf16_rounded(s); /* bf16 hand-off into the norm */
        }
        /* one state written per token, into slots[r, t] */
        float *dst = a->state_pool + ((int64_t)a->slots[row0 + t] * heads + h) * HEAD_DIM * HEAD_DIM;
        uint16_t *dst16 = (uint16_t *)a->state_pool + ((int64_t)a->slots[row0 + t] * heads + h) * HEAD_DIM * HEAD_DIM;
        for (int v = 0; v < HEAD_DIM; ++v)
            for (int k = 0; k < HEAD_DIM; ++k) {
                if (a->state_bf16) dst16[v * HEAD_DIM + k] = bf16_round(S[k * HEAD_DIM + v]);
                else dst[v * HEAD_DIM + k] = (float)S[k * HEAD_DIM + v];
            }

        /* Step 6: gated RMSNorm over the head's 128 -> bf16 core_out. */
        double ms = 0.0;
        for (int v = 0; v < HEAD_DIM; ++v) ms += o[v] * o[v];
        ms /= HEAD_DIM;
        const double rstd = 1.0 / sqrt(ms + a->eps);
        const uint16_t *gate = projected + (row0 + t) * pitch + 3 * D + h * HEAD_DIM;
        for (int v = 0; v < HEAD_DIM; ++v) {
            const double y = o[v] * rstd * (double)a->o_norm[v] * sigmoid(bf16_value(gate[v]));
            a->out[(row0 + t) * D + h * HEAD_DIM + v] = bf16_round(y);
        }

        if (a->diag) {
            double *dg = a->diag + ((row0 + t) * heads + h) * DIAG;
            for (int i = 0; i < HEAD_DIM; ++i) {
                dg[i] = qh[i];
                dg[HEAD_DIM + i] = kh[i];
                dg[2 * HEAD_DIM + i] = vr[i];
                dg[3 * HEAD_DIM + i] = gr[i];
                dg[4 * HEAD_DIM + i] = o[i];
            }
            dg[5 * HEAD_DIM] = bt;
        }
    }
}

/* Threads the OpenMP build may use (1 when built without OpenMP). */
int kda_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * One decode or verify step.
 *
 *   heads, W          H heads of 128 channels (D = 128 H); conv width W (state_len W-1)
 *   conv_w            [3D, 1, W] bf16 (the model's depthwise conv weight)
 *   bias              [3D] bf16 or NULL (zero bias)
 *   f_b               [D, 128] bf16
 *   A_log             [H] fp32;  dt_bias [D] fp32;  o_norm [128] fp32
 *   lb, eps           gate lower bound and o_norm epsilon (fp32 scalars)
 *   act               1 = SiLU after the conv (the model), 0 = none (pins only)
 *   gate_mode         0 = lb * sigmoid form, 1 = clamped softplus form (see above)
 *   projected         [rows, pitch] bf16: cols [0,3D) q|k|v, [3D,4D) out-gate,
 *                     [4D, 4D+128) f_a, [4D+128, 4D+128+H) beta
 *   conv_state        bf16 [pool, 3D, W-1] (dim_first) or [pool, W-1, 3D]; updated
 *   state_pool        fp32 [pool, H, 128 (v), 128 (k)]; updated (bf16 bits when state_bf16)
 *   slots             [rows] int32 (request-major [R, L] for verify)
 *   L                 tokens per request (rows = R L)
 *   accepted          [R] int32 in 1..L, or NULL for decode (then L must be 1)
 *   out               [rows, D] bf16
 *   err               OR-ed error bits (ERR_SLOT, ERR_ACCEPTED)
 *   diag              NULL or [rows, H, 5*128 + 1] fp64: q^, k^, v, g, o (bf16), beta
 *   threads           OpenMP threads over the (request, head) tasks (1 = serial);
 *                     each task runs its steps in the same order whatever the
 *                     count, so the results do not depend on it
 *
 * Returns 0, or -1 for arguments that make the step undefined.
 */
int kda_oracle_step(int heads, int W, const uint16_t *conv_w, const uint16_t *bias,
                    const uint16_t *f_b, const float *A_log, const float *dt_bias,
                    const float *o_norm, float lb, float eps, int act, int gate_mode,
                    const uint16_t *projected, int64_t rows, int64_t pitch,
                    uint16_t *conv_state, int dim_first, float *state_pool, int64_t pool, int state_bf16,
                    const int32_t *slots, int L, const int32_t *accepted, uint16_t *out,
                    uint32_t *err, double *diag, int threads) {
    if (heads < 1 || W < 2 || L < 1 || rows < 0 || pool < 0 || threads < 1) return -1;
    if (rows % L != 0) return -1;
    if (accepted == NULL && L != 1) return -1;
    const int64_t D = (int64_t)HEAD_DIM * heads;
    if (pitch < 4 * D + HEAD_DIM + heads) return -1;
    const int64_t R = rows / L;
    StepArgs a = {heads, W, act, gate_mode, dim_first, state_bf16, L, conv_w, bias, f_b, A_log, dt_bias, o_norm,
                  (double)lb, (double)eps, projected, pitch, pool, conv_state, state_pool, slots, out, diag};

    /* Step 1 per request: padding, accepted and slot checks, the start slot. */
    int64_t *start_of = malloc(sizeof(int64_t) * (size_t)(R > 0 ? R : 1));
    if (!start_of) return -1;
    for (int64_t r = 0; r < R; ++r) {
        const int64_t row0 = r * L;
        start_of[r] = -1;
        /* Padding request: slot -1 in its first position. */
        if (slots[row0] == -1) {
            for (int64_t t = 0; t < L; ++t)
                for (int64_t c = 0; c < D; ++c) out[(row0 + t) * D + c] = 0;
            continue;
        }
        int acc = 1;
        if (accepted != NULL) {
            acc = accepted[r];
            if (acc < 1 || acc > L) { *err |= ERR_ACCEPTED; continue; }
        }
        int bad = 0;
        for (int64_t t = 0; t < L; ++t)
            if (slots[row0 + t] < 0 || slots[row0 + t] >= pool) bad = 1;
        if (bad) { *err |= ERR_SLOT; continue; }
        start_of[r] = slots[row0 + acc - 1];
    }

    /* Steps 2-6, one task per (request, head). */
    const int64_t tasks = R * heads;
    int failed = 0;
#ifdef _OPENMP
#pragma omp parallel num_threads(threads) reduction(| : failed)
#endif
    {
        TaskBuf b;
        b.qkv = malloc(sizeof(double) * (size_t)(L * 3 * HEAD_DIM));
        b.g = malloc(sizeof(double) * (size_t)(L * HEAD_DIM));
        b.beta = malloc(sizeof(double) * (size_t)L);
        b.S = malloc(sizeof(double) * HEAD_DIM * HEAD_DIM);
        b.window = malloc(sizeof(double) * (size_t)W);
        const int ok = b.qkv && b.g && b.beta && b.S && b.window;
        if (!ok) failed = 1;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t k = 0; k < tasks; ++k) {
            const int64_t r = k / heads, h = k % heads;
            if (ok && start_of[r] >= 0) run_task(&a, r, h, start_of[r], &b);
        }
        free(b.qkv); free(b.g); free(b.beta); free(b.S); free(b.window);
    }
    free(start_of);
    return failed ? -1 : 0;
}
