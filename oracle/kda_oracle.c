/*
 * KDA oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, sequential fp64 restatement of the Kimi Delta Attention (KDA)
 * gated delta-rule recurrence.  It exists so that the CUDA path can be checked
 * against something obviously correct; nothing in the product library links,
 * includes or calls this file, and this file uses nothing from the product.
 * Only tests/, __graft_entry__.smoke() and bench.py (its cpu_baseline leg and
 * its reference arm) may load it.
 *
 * Definition followed (per chain = one sequence n and one head h, state S is
 * K x V with row index = key channel, column index = value channel):
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 *
 * Source: the recurrence behind "Kimi Delta Attention (KDA) prefill" on the
 * TensorRT-LLM pull request "Kimi K3 KDA prefill: K1 warps finish reading
 * sPartialLast before the next chunk" (Description: gate prefix scan, chunk
 * total, beta sigmoid) and the cuDNN-frontend pull request for the sm90 KDA
 * prefill kernel (Conversation: BF16 Q/K/V, FP32 gate / beta / state, non-zero
 * initial_state, scoring by an fp64 oracle).  The pages do not print the
 * equation; the form above is the one the build is specified against, and the
 * step order below is the plainest reading of it:
 *
 *     S <- Diag(exp g_t) S            (decay every key row c by exp(g_t[c]))
 *     u <- v_t - S^T k_t              (what the memory currently returns for k_t)
 *     S <- S + beta_t k_t u^T         (delta-rule write)
 *     o_t <- scale * S^T q_t
 *
 * which is algebraically identical to the matrix form (expand the product)
 * but costs O(K V) per token instead of O(K^2 V).
 *
 * beta: if beta_is_logit != 0 the per-token value b is a logit and
 * beta = 1 / (1 + exp(-b)) (the "beta sigmoid" fused into prefill, page 1);
 * otherwise b is used as beta directly.
 *
 * All inputs are fp64 arrays in a canonical packed layout; the Python wrapper
 * widens bf16 / fp32 device tensors exactly before calling.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static double kda_oracle_beta(double b, int beta_is_logit) {
    if (!beta_is_logit) return b;
    return 1.0 / (1.0 + exp(-b));
}

/* One token of the recurrence on a K x V state (row-major, row = key). */
static void kda_oracle_token(double* S, int64_t K, int64_t V,
                             const double* q, const double* k, const double* v,
                             const double* g, double beta, double scale,
                             double* u /* scratch [V] */, double* o /* [V] */) {
    /* decay: S <- Diag(exp g) S */
    for (int64_t c = 0; c < K; ++c) {
        const double d = exp(g[c]);
        double* row = S + c * V;
        for (int64_t j = 0; j < V; ++j) row[j] *= d;
    }
    /* u <- v - S^T k */
    for (int64_t j = 0; j < V; ++j) u[j] = v[j];
    for (int64_t c = 0; c < K; ++c) {
        const double kc = k[c];
        const double* row = S + c * V;
        for (int64_t j = 0; j < V; ++j) u[j] -= row[j] * kc;
    }
    /* S <- S + beta k u^T */
    for (int64_t c = 0; c < K; ++c) {
        const double bk = beta * k[c];
        double* row = S + c * V;
        for (int64_t j = 0; j < V; ++j) row[j] += bk * u[j];
    }
    /* o <- scale S^T q */
    if (o) {
        for (int64_t j = 0; j < V; ++j) o[j] = 0.0;
        for (int64_t c = 0; c < K; ++c) {
            const double qc = q[c];
            const double* row = S + c * V;
            for (int64_t j = 0; j < V; ++j) o[j] += row[j] * qc;
        }
        for (int64_t j = 0; j < V; ++j) o[j] *= scale;
    }
}

/*
 * Prefill over packed variable-length sequences.
 *   cu      int64 [N+1], cu[0] = 0, non-decreasing; sequence n owns tokens
 *           cu[n] .. cu[n+1]-1 of the packed token axis.
 *   q, k, g [T_total, H, K];  v [T_total, H, V];  b [T_total, H]
 *   h0      [N, H, K, V] or NULL (zeros)
 *   out     [T_total, H, V]
 *   hT      [N, H, K, V] or NULL (not stored)
 * Returns the number of threads used.
 */
int kda_oracle_prefill(int64_t N, const int64_t* cu, int64_t H, int64_t K, int64_t V,
                       const double* q, const double* k, const double* v,
                       const double* g, const double* b, int beta_is_logit,
                       double scale, const double* h0, double* out, double* hT) {
    int used = 1;
    const int64_t chains = N * H;
#pragma omp parallel
    {
#ifdef _OPENMP
#pragma omp single
        used = omp_get_num_threads();
#endif
        double* S = (double*)malloc(sizeof(double) * (size_t)(K * V));
        double* u = (double*)malloc(sizeof(double) * (size_t)V);
#pragma omp for schedule(dynamic, 1)
        for (int64_t ch = 0; ch < chains; ++ch) {
            const int64_t n = ch / H, h = ch % H;
            if (h0)
                memcpy(S, h0 + ch * K * V, sizeof(double) * (size_t)(K * V));
            else
                memset(S, 0, sizeof(double) * (size_t)(K * V));
            for (int64_t t = cu[n]; t < cu[n + 1]; ++t) {
                const int64_t th = t * H + h;
                kda_oracle_token(S, K, V, q + th * K, k + th * K, v + th * V, g + th * K,
                                 kda_oracle_beta(b[th], beta_is_logit), scale, u,
                                 out + th * V);
            }
            if (hT) memcpy(hT + ch * K * V, S, sizeof(double) * (size_t)(K * V));
        }
        free(u);
        free(S);
    }
    return used;
}

/*
 * MTP verify: R requests, each with D draft tokens, against a state pool.
 *   q, k, g [R, D, H, K];  v [R, D, H, V];  b [R, D, H]
 *   pool    [P, H, K, V]  (read at slot[r], or r when slot is NULL)
 *   accepted int64 [R], each in 0..D: the state stored for request r is the
 *           state after its first accepted[r] drafts (accepted 0 = unchanged).
 *   out     [R, D, H, V]: outputs of every draft, computed sequentially.
 *   pool_out [R, H, K, V]: the stored state of every request.
 * The drafts of one request are one short chunk of the same recurrence
 * (TensorRT-LLM PR "Kimi K3 work for Rubin (SM107)", Description: tcgen05 KDA
 * MTP verify kernel, WY-form chunk; the replay-only commit stores only the state).
 */
int kda_oracle_verify(int64_t R, int64_t D, int64_t H, int64_t K, int64_t V,
                      const double* q, const double* k, const double* v,
                      const double* g, const double* b, int beta_is_logit, double scale,
                      const double* pool, const int64_t* slot, const int64_t* accepted,
                      double* out, double* pool_out) {
    int used = 1;
    const int64_t chains = R * H;
#pragma omp parallel
    {
#ifdef _OPENMP
#pragma omp single
        used = omp_get_num_threads();
#endif
        double* S = (double*)malloc(sizeof(double) * (size_t)(K * V));
        double* u = (double*)malloc(sizeof(double) * (size_t)V);
#pragma omp for schedule(dynamic, 1)
        for (int64_t ch = 0; ch < chains; ++ch) {
            const int64_t r = ch / H, h = ch % H;
            const int64_t s = slot ? slot[r] : r;
            memcpy(S, pool + (s * H + h) * K * V, sizeof(double) * (size_t)(K * V));
            double* dst = pool_out + (r * H + h) * K * V;
            if (accepted[r] == 0) memcpy(dst, S, sizeof(double) * (size_t)(K * V));
            for (int64_t t = 0; t < D; ++t) {
                const int64_t th = (r * D + t) * H + h;
                kda_oracle_token(S, K, V, q + th * K, k + th * K, v + th * V, g + th * K,
                                 kda_oracle_beta(b[th], beta_is_logit), scale, u,
                                 out + th * V);
                if (t + 1 == accepted[r]) memcpy(dst, S, sizeof(double) * (size_t)(K * V));
            }
        }
        free(u);
        free(S);
    }
    return used;
}
