/*
 * Float64 CPU oracle of the Gated DeltaNet speculative verify/commit path.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark may load this library.  The CUDA library never links,
 * includes or calls it, and this file includes nothing of the CUDA library.
 *
 * What it computes (for every listed unit = one (request r, head h)):
 *   the gated delta rule of Gated DeltaNet, the per-token state update that
 *   the OCRia write-up ("OCRia 推理栈：单卡 B200 提速近 10 倍", section "Make
 *   speculative verification cheaper") says a GDN layer performs for every
 *   token, in the orientation where the state S is dv x dk:
 *
 *       S_t = alpha_t * S_{t-1} * (I - beta_t * k_t * k_t^T) + beta_t * v_t * k_t^T
 *       o_t = S_t * q_t                       (contracts the key index)
 *
 *   starting from the checkpoint S_0 (ReplaySSM's checkpoint, same section),
 *   for t = 1..T_r.  Verification reports every o_t and never changes S_0;
 *   commit keeps the accepted prefix: the state after a_r tokens.
 *
 * Storage: a state tile is stored transposed, tile[i][j] = S[j][i] (key index
 * i is the row, value index j is contiguous); q and k are [N_tok][H][dk], v is
 * [N_tok][H][dv], alpha and beta are [N_tok][H]; all float64 here.
 */
#ifndef GDN_ORACLE_H
#define GDN_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Runs the recurrence for n_units listed units.
 *   unit_ids[n]  = r * heads + h of the n-th listed unit
 *   cu_seqlens   = [B+1] token-row offsets; request r owns rows [cu[r], cu[r+1])
 *   s0           = [n_units][dk][dv] checkpoint tile of each listed unit
 *   accepted     = [B] accepted lengths, or NULL (then s_acc must be NULL)
 *   o            = [n_units][max_T][dv] outputs o_t (rows t >= T_r untouched), or NULL
 *   s_acc        = [n_units][dk][dv] state after accepted[r] tokens, or NULL
 * Returns 0, or 1 when a length exceeds max_T or an accepted length lies
 * outside [0, T_r], or 2 when memory runs out.  Pure function of its inputs.
 */
int gdn_oracle_run_units(int64_t heads, int64_t dk, int64_t dv, int64_t max_T,
                         const int64_t *cu_seqlens,
                         const double *q, const double *k, const double *v,
                         const double *alpha, const double *beta,
                         int64_t n_units, const int64_t *unit_ids,
                         const double *s0, const int64_t *accepted,
                         double *o, double *s_acc);

#ifdef __cplusplus
}
#endif

#endif /* GDN_ORACLE_H */
