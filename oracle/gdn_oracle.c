/*
 * Float64 CPU oracle of the Gated DeltaNet speculative verify/commit path.
 * TEST INFRASTRUCTURE ONLY: see gdn_oracle.h for who may use it.
 *
 * Written to be read against the definition, not to be fast: every token
 * builds the dk x dk matrix (I - beta k k^T) and multiplies the whole state by
 * it, exactly as the update is written.  No blocking, no fusion, no reordering.
 * Compile with -ffp-contract=off so no multiply-add is fused behind our back.
 */
#include "gdn_oracle.h"

#include <stdlib.h>
#include <string.h>

/* tile[i][j] = S[j][i]: the stored tile is the transpose of the dv x dk state. */
static void tile_to_state(const double *tile, double *S, int64_t dk, int64_t dv)
{
    for (int64_t j = 0; j < dv; ++j)
        for (int64_t i = 0; i < dk; ++i)
            S[j * dk + i] = tile[i * dv + j];
}

static void state_to_tile(const double *S, double *tile, int64_t dk, int64_t dv)
{
    for (int64_t i = 0; i < dk; ++i)
        for (int64_t j = 0; j < dv; ++j)
            tile[i * dv + j] = S[j * dk + i];
}

int gdn_oracle_run_units(int64_t heads, int64_t dk, int64_t dv, int64_t max_T,
                         const int64_t *cu_seqlens,
                         const double *q, const double *k, const double *v,
                         const double *alpha, const double *beta,
                         int64_t n_units, const int64_t *unit_ids,
                         const double *s0, const int64_t *accepted,
                         double *o, double *s_acc)
{
    double *S = (double *)malloc((size_t)(dv * dk) * sizeof(double));   /* S_{t}, dv x dk */
    double *E = (double *)malloc((size_t)(dk * dk) * sizeof(double));   /* I - beta k k^T */
    double *SE = (double *)malloc((size_t)(dv * dk) * sizeof(double));  /* S_{t-1} E      */
    int status = 0;
    if (!S || !E || !SE) {
        status = 2;
        goto done;
    }

    for (int64_t n = 0; n < n_units; ++n) {
        const int64_t u = unit_ids[n];
        const int64_t r = u / heads;
        const int64_t h = u % heads;
        const int64_t row0 = cu_seqlens[r];
        const int64_t T_r = cu_seqlens[r + 1] - cu_seqlens[r];
        const int64_t a_r = accepted ? accepted[r] : -1;
        if (T_r < 0 || T_r > max_T || (accepted && (a_r < 0 || a_r > T_r))) {
            status = 1;
            goto done;
        }

        /* S_0: the checkpoint, never written by the oracle. */
        tile_to_state(s0 + n * dk * dv, S, dk, dv);
        if (s_acc && a_r == 0)
            state_to_tile(S, s_acc + n * dk * dv, dk, dv);

        /* Without outputs only the accepted prefix needs replaying. */
        const int64_t T_run = (o == NULL && s_acc) ? a_r : T_r;
        for (int64_t t = 0; t < T_run; ++t) {
            const int64_t x = (row0 + t) * heads + h;  /* token row, head */
            const double a_t = alpha[x];
            const double b_t = beta[x];
            const double *k_t = k + x * dk;
            const double *v_t = v + x * dv;
            const double *q_t = q + x * dk;

            /* E = I - beta_t k_t k_t^T */
            for (int64_t i = 0; i < dk; ++i)
                for (int64_t l = 0; l < dk; ++l)
                    E[i * dk + l] = (i == l ? 1.0 : 0.0) - b_t * k_t[i] * k_t[l];

            /* SE = S_{t-1} E */
            for (int64_t j = 0; j < dv; ++j)
                for (int64_t l = 0; l < dk; ++l) {
                    double acc = 0.0;
                    for (int64_t i = 0; i < dk; ++i)
                        acc += S[j * dk + i] * E[i * dk + l];
                    SE[j * dk + l] = acc;
                }

            /* S_t = alpha_t SE + beta_t v_t k_t^T */
            for (int64_t j = 0; j < dv; ++j)
                for (int64_t l = 0; l < dk; ++l)
                    S[j * dk + l] = a_t * SE[j * dk + l] + b_t * v_t[j] * k_t[l];

            /* o_t = S_t q_t */
            if (o) {
                double *o_t = o + (n * max_T + t) * dv;
                for (int64_t j = 0; j < dv; ++j) {
                    double acc = 0.0;
                    for (int64_t i = 0; i < dk; ++i)
                        acc += S[j * dk + i] * q_t[i];
                    o_t[j] = acc;
                }
            }

            /* The accepted prefix ends after token a_r. */
            if (s_acc && t + 1 == a_r)
                state_to_tile(S, s_acc + n * dk * dv, dk, dv);
        }
    }

done:
    free(S);
    free(E);
    free(SE);
    return status;
}
