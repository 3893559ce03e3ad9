/*
 * fp64 CPU oracle for the ReplaySSM decode path.  TEST INFRASTRUCTURE ONLY:
 * the tests, the smoke check and the benchmark's CPU-baseline leg may call
 * it; the product path never does.  It shares no code with the CUDA library.
 *
 * The method ("ReplaySSM: Cache SSM Inputs, Not State", section "How it
 * works"; abstract) produces the outputs of conventional decoding, apart from
 * rounding (same page, section "Limits").  So the oracle is
 * the conventional (eager) recurrence itself, in double precision, stepping a
 * fully materialised state S in R^{P x N} per (sequence, head):
 *
 *   Mamba-2       alpha_t = exp(dt_t * A_h),  v_t = dt_t * x_t
 *                 S_t = alpha_t S_{t-1} + v_t k_t^T          (k_t = B_t of the head's group)
 *                 y_t = S_t q_t + D_h x_t                     (q_t = C_t of the head's group)
 *   Gated DeltaNet
 *                 u_t = beta_t (v_t - alpha_t S_{t-1} k_t)    (section "How it works", GDN bullet)
 *                 S_t = alpha_t S_{t-1} + u_t k_t^T
 *                 y_t = S_t q_t
 *   per-channel decay (the reading of Kimi Delta Attention, which section
 *   "Limits" names as compatible but does not define: GDN with the scalar
 *   alpha_t replaced by one decay per key channel, alpha_t in R^N)
 *                 D_t = S_{t-1} diag(alpha_t)
 *                 u_t = beta_t (v_t - D_t k_t)
 *                 S_t = D_t + u_t k_t^T
 *                 y_t = S_t q_t
 *
 * A speculative round (section "How it works", speculative bullet and the
 * flowchart) runs the recurrence over the T drafts from the committed state,
 * emits all T outputs, and commits the state reached after the first a_b
 * drafts; the rest are discarded.
 *
 * Layouts (row-major): state S[b][h][p][n]; Mamba-2 head h reads B/C group
 * h / (H/G); GDN v-head h reads k-head h / (Hv/Hk).  bf16 inputs arrive as
 * raw uint16 bits and are widened exactly.
 */
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* One Mamba-2 step on one (P x N) state. */
static void mamba2_head_step(int P, int N, double *s, const uint16_t *x, double dt, double A,
                             const uint16_t *kb, const uint16_t *qb, double D, double *y)
{
    const double alpha = exp(dt * A);
    for (int p = 0; p < P; ++p) {
        const double v = dt * bf16(x[p]);
        double acc = 0.0;
        double *row = s + (size_t)p * N;
        for (int n = 0; n < N; ++n) {
            row[n] = alpha * row[n] + v * bf16(kb[n]);
            acc += row[n] * bf16(qb[n]);
        }
        y[p] = acc + D * bf16(x[p]);
    }
}

/* One GDN step on one (P x N) state; u_t[p] only needs row p of S_{t-1}. */
static void gdn_head_step(int P, int N, double *s, const uint16_t *qb, const uint16_t *kb,
                          const uint16_t *vb, double alpha, double beta, double *y, double *u_out)
{
    for (int p = 0; p < P; ++p) {
        double *row = s + (size_t)p * N;
        double sk = 0.0;
        for (int n = 0; n < N; ++n) sk += row[n] * bf16(kb[n]);
        const double u = beta * (bf16(vb[p]) - alpha * sk);
        double acc = 0.0;
        for (int n = 0; n < N; ++n) {
            row[n] = alpha * row[n] + u * bf16(kb[n]);
            acc += row[n] * bf16(qb[n]);
        }
        y[p] = acc;
        if (u_out) u_out[p] = u;
    }
}

/* One step with a per-key-channel decay; alpha points at the head's N decays. */
static void kda_head_step(int P, int N, double *s, const uint16_t *qb, const uint16_t *kb,
                          const uint16_t *vb, const float *alpha, double beta, double *y, double *u_out)
{
    for (int p = 0; p < P; ++p) {
        double *row = s + (size_t)p * N;
        double dk = 0.0;
        for (int n = 0; n < N; ++n) {
            row[n] *= (double)alpha[n];
            dk += row[n] * bf16(kb[n]);
        }
        const double u = beta * (bf16(vb[p]) - dk);
        double acc = 0.0;
        for (int n = 0; n < N; ++n) {
            row[n] += u * bf16(kb[n]);
            acc += row[n] * bf16(qb[n]);
        }
        y[p] = acc;
        if (u_out) u_out[p] = u;
    }
}

/*
 * Mamba-2 standard step for all sequences and heads.
 *   S  f64[B][H][P][N] (updated in place)   x u16[B][H][P]   dt f32[B][H]
 *   A  f32[H]   Bm, Cm u16[B][G][N]   D f32[H]   y f64[B][H][P]
 */
void oracle_mamba2_step(int B, int H, int G, int P, int N, double *S, const uint16_t *x,
                        const float *dt, const float *A, const uint16_t *Bm, const uint16_t *Cm,
                        const float *D, double *y)
{
    const int hpg = H / G;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            const int g = h / hpg;
            const size_t bh = (size_t)b * H + h, bg = (size_t)b * G + g;
            mamba2_head_step(P, N, S + bh * P * N, x + bh * P, dt[bh], A[h], Bm + bg * N,
                             Cm + bg * N, D[h], y + bh * P);
        }
}

/*
 * GDN standard step.  S f64[B][Hv][P][N]; q, k u16[B][Hk][N]; v u16[B][Hv][P];
 * alpha, beta f32[B][Hv]; y f64[B][Hv][P]; u (nullable) f64[B][Hv][P].
 */
void oracle_gdn_step(int B, int Hv, int Hk, int P, int N, double *S, const uint16_t *q,
                     const uint16_t *k, const uint16_t *v, const float *alpha, const float *beta,
                     double *y, double *u)
{
    const int ratio = Hv / Hk;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < Hv; ++h) {
            const size_t bh = (size_t)b * Hv + h, bk = (size_t)b * Hk + h / ratio;
            gdn_head_step(P, N, S + bh * P * N, q + bk * N, k + bk * N, v + bh * P, alpha[bh],
                          beta[bh], y + bh * P, u ? u + bh * P : NULL);
        }
}

/*
 * Mamba-2 speculative round.  Draft inputs carry a draft axis after the batch
 * axis: x u16[B][T][H][P], dt f32[B][T][H], Bm/Cm u16[B][T][G][N];
 * y f64[B][T][H][P]; accepted i32[B] in 0..T.  S holds the committed state and
 * is replaced by the state after the accepted prefix.
 */
void oracle_mamba2_spec_round(int B, int H, int G, int P, int N, int T, double *S,
                              const uint16_t *x, const float *dt, const float *A,
                              const uint16_t *Bm, const uint16_t *Cm, const float *D,
                              const int32_t *accepted, double *y)
{
    const int hpg = H / G;
#pragma omp parallel
    {
        double *work = (double *)malloc(sizeof(double) * (size_t)P * N);
#pragma omp for collapse(2) schedule(static)
        for (int b = 0; b < B; ++b)
            for (int h = 0; h < H; ++h) {
                const int g = h / hpg;
                double *s = S + ((size_t)b * H + h) * P * N;
                memcpy(work, s, sizeof(double) * (size_t)P * N);
                for (int i = 0; i < T; ++i) {
                    const size_t bth = ((size_t)b * T + i) * H + h;
                    const size_t btg = ((size_t)b * T + i) * G + g;
                    mamba2_head_step(P, N, work, x + bth * P, dt[bth], A[h], Bm + btg * N,
                                     Cm + btg * N, D[h], y + bth * P);
                    if (i + 1 == accepted[b]) memcpy(s, work, sizeof(double) * (size_t)P * N);
                }
            }
        free(work);
    }
}

/*
 * GDN speculative round.  q, k u16[B][T][Hk][N]; v u16[B][T][Hv][P];
 * alpha, beta f32[B][T][Hv]; y f64[B][T][Hv][P]; accepted i32[B].
 */
void oracle_gdn_spec_round(int B, int Hv, int Hk, int P, int N, int T, double *S,
                           const uint16_t *q, const uint16_t *k, const uint16_t *v,
                           const float *alpha, const float *beta, const int32_t *accepted,
                           double *y)
{
    const int ratio = Hv / Hk;
#pragma omp parallel
    {
        double *work = (double *)malloc(sizeof(double) * (size_t)P * N);
#pragma omp for collapse(2) schedule(static)
        for (int b = 0; b < B; ++b)
            for (int h = 0; h < Hv; ++h) {
                double *s = S + ((size_t)b * Hv + h) * P * N;
                memcpy(work, s, sizeof(double) * (size_t)P * N);
                for (int i = 0; i < T; ++i) {
                    const size_t bth = ((size_t)b * T + i) * Hv + h;
                    const size_t btk = ((size_t)b * T + i) * Hk + h / ratio;
                    gdn_head_step(P, N, work, q + btk * N, k + btk * N, v + bth * P, alpha[bth],
                                  beta[bth], y + bth * P, NULL);
                    if (i + 1 == accepted[b]) memcpy(s, work, sizeof(double) * (size_t)P * N);
                }
            }
        free(work);
    }
}

/*
 * Per-channel-decay step.  As oracle_gdn_step, with alpha f32[B][Hv][N].
 */
void oracle_kda_step(int B, int Hv, int Hk, int P, int N, double *S, const uint16_t *q,
                     const uint16_t *k, const uint16_t *v, const float *alpha, const float *beta,
                     double *y, double *u)
{
    const int ratio = Hv / Hk;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < Hv; ++h) {
            const size_t bh = (size_t)b * Hv + h, bk = (size_t)b * Hk + h / ratio;
            kda_head_step(P, N, S + bh * P * N, q + bk * N, k + bk * N, v + bh * P, alpha + bh * N,
                          beta[bh], y + bh * P, u ? u + bh * P : NULL);
        }
}

/*
 * Per-channel-decay speculative round.  As oracle_gdn_spec_round, with
 * alpha f32[B][T][Hv][N].
 */
void oracle_kda_spec_round(int B, int Hv, int Hk, int P, int N, int T, double *S,
                           const uint16_t *q, const uint16_t *k, const uint16_t *v,
                           const float *alpha, const float *beta, const int32_t *accepted,
                           double *y)
{
    const int ratio = Hv / Hk;
#pragma omp parallel
    {
        double *work = (double *)malloc(sizeof(double) * (size_t)P * N);
#pragma omp for collapse(2) schedule(static)
        for (int b = 0; b < B; ++b)
            for (int h = 0; h < Hv; ++h) {
                double *s = S + ((size_t)b * Hv + h) * P * N;
                memcpy(work, s, sizeof(double) * (size_t)P * N);
                for (int i = 0; i < T; ++i) {
                    const size_t bth = ((size_t)b * T + i) * Hv + h;
                    const size_t btk = ((size_t)b * T + i) * Hk + h / ratio;
                    kda_head_step(P, N, work, q + btk * N, k + btk * N, v + bth * P, alpha + bth * N,
                                  beta[bth], y + bth * P, NULL);
                    if (i + 1 == accepted[b]) memcpy(s, work, sizeof(double) * (size_t)P * N);
                }
            }
        free(work);
    }
}

/* Number of OpenMP threads the oracle runs with (for reporting). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
