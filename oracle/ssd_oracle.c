/*
 * ssd_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, sequential fp64 CPU implementation of the Mamba-2 SSD
 * (state-space-dual) selective scan forward.  Only the test-suite, the smoke
 * check and the CPU-baseline leg of the benchmark load this file; the product
 * path never does.  It shares no code with the CUDA library.
 *
 * What it computes (one independent recurrence per batch row b and head h,
 * with g = h / (nheads / ngroups), the "group query" mapping of B and C onto
 * heads described in the "Differences between simple_gla kernel and
 * mamba2_ssd kernel" list of fla-org/flash-linear-attention PR #49 and in the
 * ngroups repro of state-spaces/mamba issue #647):
 *
 *   dt_t  = dt_raw[b,t,h] + dt_bias[h]           (dt_bias absent -> 0)
 *   dt_t  = softplus(dt_t)                       if dt_softplus
 *   dt_t  = clamp(dt_t, lo, hi)                  unless (lo, hi) == (0, +inf)
 *   if seq_idx given and t > 0 and seq_idx[b,t] != seq_idx[b,t-1]:  h := 0
 *   h     = exp(dt_t * A[h]) * h + dt_t * x[b,t,h,:] (outer) B[b,t,g,:]
 *   y_t   = h . C[b,t,g,:]  +  D[h] * x[b,t,h,:]  (D absent -> 0)
 *   out   = y_t * silu(z[b,t,h,:])               if z given
 *
 * h starts at initial_states[b,h] (absent -> 0); final_states[b,h] is h
 * after the last token.  The state is stored [headdim][dstate].
 *
 * The dt argument order (bias, then softplus, then the dt_limit clamp) and
 * the (0, inf) default of dt_limit follow the argument list of the
 * mamba_split_conv1d_scan_combined call on the issue #647 page; initial and
 * final states follow the chunked-prefill description of state-spaces/mamba
 * PR #488.
 *
 * A compile-time switch SSD_ORACLE_MUTATION=k plants one deliberate mistake
 * (see the list at the bottom of the loop body).  It exists only so that the
 * test-suite can show that its pins catch each such mistake; the default
 * build (k = 0) has none.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef SSD_ORACLE_MUTATION
#define SSD_ORACLE_MUTATION 0
#endif

static double softplus_d(double v)
{
    /* log(1 + e^v) without overflow */
    return v > 0.0 ? v + log1p(exp(-v)) : log1p(exp(v));
}

int ssd_oracle_mutation(void) { return SSD_ORACLE_MUTATION; }

/* dt preprocessing alone, [batch, seqlen, nheads] -> same shape. */
void ssd_oracle_dt(int64_t batch, int64_t seqlen, int64_t nheads,
                   const double *dt_raw, const double *dt_bias,
                   int dt_softplus, double lo, double hi, double *dt_out)
{
    const int clamp = !(lo == 0.0 && isinf(hi) && hi > 0);
    for (int64_t i = 0; i < batch * seqlen; ++i)
        for (int64_t h = 0; h < nheads; ++h) {
            double d = dt_raw[i * nheads + h] + (dt_bias ? dt_bias[h] : 0.0);
            if (dt_softplus) d = softplus_d(d);
            if (clamp) d = d < lo ? lo : (d > hi ? hi : d);
            dt_out[i * nheads + h] = d;
        }
}

/*
 * Full scan.  Every array is dense row-major fp64 (seq_idx int32).
 *   x, z, out        [batch, seqlen, nheads, headdim]
 *   dt_raw           [batch, seqlen, nheads]
 *   B, C             [batch, seqlen, ngroups, dstate]
 *   dt_bias, A, D    [nheads]
 *   initial, final   [batch, nheads, headdim, dstate]
 *   seq_idx          [batch, seqlen]
 * Optional inputs may be NULL.  Returns 0, or -1 on bad sizes.
 */
int ssd_oracle_scan(int64_t batch, int64_t seqlen, int64_t nheads,
                    int64_t headdim, int64_t dstate, int64_t ngroups,
                    const double *x, const double *dt_raw,
                    const double *dt_bias, int dt_softplus,
                    double lo, double hi, const double *A,
                    const double *B, const double *C, const double *D,
                    const double *z, const double *initial_states,
                    const int32_t *seq_idx, double *out,
                    double *final_states, int nthreads)
{
    if (batch < 0 || seqlen < 0 || nheads <= 0 || headdim <= 0 || dstate <= 0 ||
        ngroups <= 0 || nheads % ngroups != 0)
        return -1;
    const int64_t H = nheads, P = headdim, N = dstate, G = ngroups;
    const int64_t heads_per_group = H / G;
    const int clamp = !(lo == 0.0 && isinf(hi) && hi > 0);
    if (nthreads < 1) nthreads = 1;
    (void)nthreads;

#pragma omp parallel for collapse(2) schedule(dynamic, 1) num_threads(nthreads)
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t hh = 0; hh < H; ++hh) {
#if SSD_ORACLE_MUTATION == 4
            const int64_t g = hh % G;           /* wrong head -> group map */
#else
            const int64_t g = hh / heads_per_group;
#endif
            double *state = (double *)malloc(sizeof(double) * (size_t)(P * N));
            if (initial_states)
                memcpy(state, initial_states + (b * H + hh) * P * N,
                       sizeof(double) * (size_t)(P * N));
            else
                memset(state, 0, sizeof(double) * (size_t)(P * N));

            for (int64_t t = 0; t < seqlen; ++t) {
                const int64_t bt = b * seqlen + t;
#if SSD_ORACLE_MUTATION != 5                     /* 5: seq_idx ignored */
                if (seq_idx && t > 0 && seq_idx[bt] != seq_idx[bt - 1])
                    memset(state, 0, sizeof(double) * (size_t)(P * N));
#endif
                double d = dt_raw[bt * H + hh] + (dt_bias ? dt_bias[hh] : 0.0);
                if (dt_softplus) d = softplus_d(d);
                if (clamp) d = d < lo ? lo : (d > hi ? hi : d);
#if SSD_ORACLE_MUTATION == 1
                const double decay = exp(-d * A[hh]);  /* wrong sign */
#else
                const double decay = exp(d * A[hh]);
#endif
                const double *xt = x + (bt * H + hh) * P;
                const double *Bt = B + (bt * G + g) * N;
                const double *Ct = C + (bt * G + g) * N;
                for (int64_t p = 0; p < P; ++p) {
                    double *sp = state + p * N;
#if SSD_ORACLE_MUTATION == 2
                    const double dx = xt[p];           /* dt dropped from input */
#else
                    const double dx = d * xt[p];
#endif
                    for (int64_t n = 0; n < N; ++n)
#if SSD_ORACLE_MUTATION == 3
                        sp[n] = decay * sp[n] + dx * Ct[n];   /* B and C swapped */
#else
                        sp[n] = decay * sp[n] + dx * Bt[n];
#endif
                }
                double *yt = out + (bt * H + hh) * P;
                for (int64_t p = 0; p < P; ++p) {
                    const double *sp = state + p * N;
                    double acc = 0.0;
                    for (int64_t n = 0; n < N; ++n)
#if SSD_ORACLE_MUTATION == 3
                        acc += sp[n] * Bt[n];
#else
                        acc += sp[n] * Ct[n];
#endif
#if SSD_ORACLE_MUTATION != 6                     /* 6: D-skip dropped */
                    if (D) acc += D[hh] * xt[p];
#endif
                    if (z) {
                        const double zz = z[(bt * H + hh) * P + p];
#if SSD_ORACLE_MUTATION == 7
                        acc *= zz;                     /* gate without the sigmoid */
#else
                        acc *= zz / (1.0 + exp(-zz));
#endif
                    }
                    yt[p] = acc;
                }
            }
            if (final_states)
                memcpy(final_states + (b * H + hh) * P * N, state,
                       sizeof(double) * (size_t)(P * N));
            free(state);
        }
    }
    return 0;
}
