/*
 * oracle/gdn_ref.c -- the CPU oracle for Gated Delta Net prefill.  TEST INFRASTRUCTURE ONLY:
 * the product path never links, loads or calls this file.  Only the tests, the package's smoke
 * check and the benchmark's CPU legs use it.
 *
 * What it computes (page "TIRx" (zixuwang.me), section "用状态递推解释 GDN"): each sequence
 * and head carries a state matrix H of shape [V, K] (dv x dk).  Token by token, in order:
 *
 *     H_decay    = alpha_t * H
 *     prediction = H_decay k_t                    (a dv-vector)
 *     update     = beta_t * (v_t - prediction)    (a dv-vector)
 *     H          = H_decay + update k_t^T         (outer product, dv x dk)
 *     o_t        = scale * H q_t                  (a dv-vector)
 *
 * Everything is evaluated in binary64 in exactly this order, one token after another, with no
 * chunking or reordering.
 *
 * Packed input (same page, packed variable-length sequences): tokens of n_seqs independent
 * sequences are stored back to back; sequence i owns tokens cu_seqlens[i] .. cu_seqlens[i+1]-1
 * and its own state, which starts from initial_state[i] (or zero) and ends in final_state[i].
 *
 * Heads (the page names three relations: MHA, GQA and GVA).  q has h_q heads, k has h_k, and v,
 * alpha, beta and the states have h_v, with h_v a multiple of h_k: state head j reads key head
 * j / (h_v / h_k).  The outputs follow one of two layouts:
 *   h_q == h_k            one output per value head (h_o = h_v); state j reads query head
 *                         j / (h_v / h_k): MHA when h_v == h_k, GVA (grouped values) when larger;
 *   h_q a multiple of h_v one output per query head (h_o = h_q); query head m reads state
 *                         m / (h_q / h_v): GQA (grouped queries), when h_q > h_v == h_k.
 *
 * Layouts (row-major): q [T][h_q][dk]; k [T][h_k][dk]; v [T][h_v][dv]; alpha, beta [T][h_v];
 * states [n_seqs][h_v][dv][dk]; o [T][h_o][dv].
 *
 * Nothing here is shared with the GPU path: no header, helper or table.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Output heads for (h_q, h_k, h_v), or -1 if the three do not form one of the layouts above. */
int64_t oracle_gdn_out_heads(int64_t h_q, int64_t h_k, int64_t h_v)
{
    if (h_q <= 0 || h_k <= 0 || h_v <= 0 || h_v % h_k != 0) return -1;
    if (h_q == h_k) return h_v;
    if (h_q % h_v == 0) return h_q;
    return -1;
}

/* Returns 0, or -1 for inconsistent sizes, -2 if a work buffer cannot be allocated. */
int oracle_gdn_heads_f64(const double* q, const double* k, const double* v, const double* alpha,
                         const double* beta, const int32_t* cu_seqlens, int64_t n_seqs,
                         int64_t h_q, int64_t h_k, int64_t h_v, int64_t dk, int64_t dv,
                         double scale, const double* initial_state, double* o,
                         double* final_state)
{
    const int64_t h_o = oracle_gdn_out_heads(h_q, h_k, h_v);
    if (n_seqs < 0 || h_o < 0 || dk <= 0 || dv <= 0) return -1;
    for (int64_t i = 0; i < n_seqs; ++i)
        if (cu_seqlens[i + 1] < cu_seqlens[i]) return -1;
    /* per state head j: its key head, and its query heads m0 .. m0 + nq - 1 with outputs at
     * output heads o0 .. o0 + nq - 1 */
    const int64_t kgroup = h_v / h_k;
    const int64_t nq = h_o == h_v ? 1 : h_q / h_v;
    int err = 0;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int64_t i = 0; i < n_seqs; ++i) {
        for (int64_t j = 0; j < h_v; ++j) {
            double* H = (double*)malloc(sizeof(double) * (size_t)(dv * dk));
            double* upd = (double*)malloc(sizeof(double) * (size_t)dv);
            if (!H || !upd) {
                free(H);
                free(upd);
#pragma omp atomic write
                err = -2;
                continue;
            }
            const double* h0 = initial_state ? initial_state + ((i * h_v + j) * dv) * dk : NULL;
            for (int64_t e = 0; e < dv * dk; ++e) H[e] = h0 ? h0[e] : 0.0;
            const int64_t jk = j / kgroup;
            const int64_t m0 = h_o == h_v ? j / kgroup : j * nq;   /* first query head */
            const int64_t o0 = h_o == h_v ? j : j * nq;            /* its output head */
            for (int64_t t = cu_seqlens[i]; t < cu_seqlens[i + 1]; ++t) {
                const double* kt = k + (t * h_k + jk) * dk;
                const double* vt = v + (t * h_v + j) * dv;
                const double a = alpha[t * h_v + j];
                const double b = beta[t * h_v + j];
                /* H_decay = alpha * H */
                for (int64_t e = 0; e < dv * dk; ++e) H[e] *= a;
                /* prediction = H_decay k; update = beta * (v - prediction) */
                for (int64_t r = 0; r < dv; ++r) {
                    double p = 0.0;
                    for (int64_t c = 0; c < dk; ++c) p += H[r * dk + c] * kt[c];
                    upd[r] = b * (vt[r] - p);
                }
                /* H = H_decay + update k^T */
                for (int64_t r = 0; r < dv; ++r)
                    for (int64_t c = 0; c < dk; ++c) H[r * dk + c] += upd[r] * kt[c];
                /* o = scale * H q, for each query head this state serves */
                for (int64_t g = 0; g < nq; ++g) {
                    const double* qt = q + (t * h_q + m0 + g) * dk;
                    double* ot = o + (t * h_o + o0 + g) * dv;
                    for (int64_t r = 0; r < dv; ++r) {
                        double s = 0.0;
                        for (int64_t c = 0; c < dk; ++c) s += H[r * dk + c] * qt[c];
                        ot[r] = scale * s;
                    }
                }
            }
            if (final_state) memcpy(final_state + ((i * h_v + j) * dv) * dk, H,
                                    sizeof(double) * (size_t)(dv * dk));
            free(H);
            free(upd);
        }
    }
    return err;
}

/* q and k sharing h_qk heads (MHA, GVA): the layout above with h_q = h_k = h_qk. */
int oracle_gdn_f64(const double* q, const double* k, const double* v, const double* alpha,
                   const double* beta, const int32_t* cu_seqlens, int64_t n_seqs, int64_t h_qk,
                   int64_t h_v, int64_t dk, int64_t dv, double scale,
                   const double* initial_state, double* o, double* final_state)
{
    return oracle_gdn_heads_f64(q, k, v, alpha, beta, cu_seqlens, n_seqs, h_qk, h_qk, h_v, dk, dv,
                                scale, initial_state, o, final_state);
}
