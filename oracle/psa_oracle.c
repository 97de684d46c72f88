/*
 * psa_oracle.c -- plain fp64 CPU oracle for PSA self-attention (forward and
 * backward).  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * bench's CPU-baseline leg load this file; the product (the CUDA library) never
 * does, and the two share no code.
 *
 * What it computes.  "Struct PsaFa2Backward" (vision_rs, yolo attention psa),
 * description paragraphs: one FlashAttention-2 style self-attention backward
 * per V section, N_CTX_Q == N_CTX_K == N, with two calls ("lo" and "hi") that
 * share the Q and K sections of a packed per-(batch, head) buffer and each own a
 * V section; dQ and dK are summed over the calls ("Atomicity" paragraph).
 * The FA2 backward is exact: it returns the analytic gradient of plain softmax
 * attention.  So this oracle is that definition written out, for `nv` V
 * sections that share one softmax:
 *
 *   s_ij   = scale * <q_i, k_j>
 *   LSE_i  = log sum_j exp(s_ij)                      (natural log)
 *   P_ij   = exp(s_ij - LSE_i)
 *   O_h[i] = sum_j P_ij V_h[j]                        h = 0 .. nv-1
 *   D_i    = sum_h <dO_h[i], O_h[i]>
 *   dP_ij  = sum_h <dO_h[i], V_h[j]>
 *   dS_ij  = P_ij (dP_ij - D_i)
 *   dQ_i   = scale * sum_j dS_ij k_j
 *   dK_j   = scale * sum_i dS_ij q_i
 *   dV_h[j]= sum_i P_ij dO_h[i]
 *
 * nv = 2 is the PSA lo/hi pair; nv = 1 is one plain attention call, which the
 * tests use to check that the pair's dQ/dK is the sum of two single calls.
 * Every value is fp64; nothing is blocked, fused or reordered beyond the
 * loops above.  No N x N matrix is stored: each row of s is recomputed where
 * it is needed.  Rows are independent, so OpenMP splits rows across threads
 * (summation order inside a row is fixed, results do not depend on threads).
 *
 * Layouts (all row-major, contiguous, fp64):
 *   q, k, dq, dk          [BH, N, d]
 *   v, dout, o, dv        [nv, BH, N, d]
 *   lse, D                [BH, N]
 *
 * Pins (tests marked "not gpu"): central finite differences of
 * L = sum_h <dO_h, O_h>, closed forms for N = 1 and Q = 0, a two-key sigmoid
 * closed form, the invariants (equal V rows -> dQ = dK = 0, column sums of dV,
 * sum_j dK_j = 0, key permutation, <Q,dQ> = <K,dK>, pair = sum of singles),
 * and float64 torch SDPA autograd on tiny inputs.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double dot(const double* a, const double* b, int d) {
    double acc = 0.0;
    for (int c = 0; c < d; ++c) acc += a[c] * b[c];
    return acc;
}

/* s_ij for a whole row i of one (b,h) slice, into s[N]; returns LSE_i. */
static double score_row_lse(const double* q, const double* k, int N, int d, double scale,
                            int i, double* s) {
    double m = -INFINITY;
    for (int j = 0; j < N; ++j) {
        s[j] = scale * dot(q + (size_t)i * d, k + (size_t)j * d, d);
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int j = 0; j < N; ++j) l += exp(s[j] - m);
    return m + log(l);
}

int psa_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void psa_oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * Forward: O_h and LSE for BH independent slices.
 * Returns 0, or -1 on bad sizes / allocation failure.
 */
int psa_oracle_fwd(int BH, int N, int d, int nv, double scale,
                   const double* q, const double* k, const double* v,
                   double* o, double* lse) {
    if (BH < 0 || N < 0 || d <= 0 || nv <= 0) return -1;
    if (BH == 0 || N == 0) return 0;
    const size_t sec = (size_t)BH * N * d; /* elements of one [BH,N,d] tensor */
    int err = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)N);
        if (!s) {
#pragma omp atomic write
            err = -1;
        } else {
#pragma omp for schedule(static)
            for (long r = 0; r < (long)BH * N; ++r) {
                const int bh = (int)(r / N), i = (int)(r % N);
                const double* qb = q + (size_t)bh * N * d;
                const double* kb = k + (size_t)bh * N * d;
                const double L = score_row_lse(qb, kb, N, d, scale, i, s);
                lse[r] = L;
                for (int h = 0; h < nv; ++h) {
                    const double* vb = v + h * sec + (size_t)bh * N * d;
                    double* orow = o + h * sec + (size_t)r * d;
                    for (int c = 0; c < d; ++c) orow[c] = 0.0;
                    for (int j = 0; j < N; ++j) {
                        const double p = exp(s[j] - L);
                        for (int c = 0; c < d; ++c) orow[c] += p * vb[(size_t)j * d + c];
                    }
                }
            }
            free(s);
        }
    }
    return err;
}

/*
 * Backward: dQ, dK (summed over the nv calls) and dV_h, from the inputs alone.
 * The oracle runs its own forward for LSE and O (so D uses the oracle's own
 * fp64 O), then one pass over query rows (dQ) and one over key rows (dK, dV).
 * o_out / lse_out / D_out may be NULL; when given they receive the forward
 * outputs and D.  Returns 0, or -1 on bad sizes / allocation failure.
 */
int psa_oracle_bwd(int BH, int N, int d, int nv, double scale,
                   const double* q, const double* k, const double* v, const double* dout,
                   double* dq, double* dk, double* dv,
                   double* o_out, double* lse_out, double* D_out) {
    if (BH < 0 || N < 0 || d <= 0 || nv <= 0) return -1;
    if (BH == 0 || N == 0) return 0;
    const size_t sec = (size_t)BH * N * d;
    double* o = o_out ? o_out : (double*)malloc(sizeof(double) * sec * nv);
    double* lse = lse_out ? lse_out : (double*)malloc(sizeof(double) * (size_t)BH * N);
    double* D = D_out ? D_out : (double*)malloc(sizeof(double) * (size_t)BH * N);
    int err = 0;
    if (!o || !lse || !D) { err = -1; goto done; }

    /* 1. forward: LSE and O */
    err = psa_oracle_fwd(BH, N, d, nv, scale, q, k, v, o, lse);
    if (err) goto done;

    /* 2. D_i = sum_h <dO_h[i], O_h[i]> */
#pragma omp parallel for schedule(static)
    for (long r = 0; r < (long)BH * N; ++r) {
        double acc = 0.0;
        for (int h = 0; h < nv; ++h)
            acc += dot(dout + h * sec + (size_t)r * d, o + h * sec + (size_t)r * d, d);
        D[r] = acc;
    }

    /* 3. pass over query rows: dQ_i = scale * sum_j dS_ij k_j */
#pragma omp parallel for schedule(static)
    for (long r = 0; r < (long)BH * N; ++r) {
        const int bh = (int)(r / N), i = (int)(r % N);
        const size_t base = (size_t)bh * N * d;
        const double* qi = q + (size_t)r * d;
        double* dqi = dq + (size_t)r * d;
        for (int c = 0; c < d; ++c) dqi[c] = 0.0;
        for (int j = 0; j < N; ++j) {
            const double* kj = k + base + (size_t)j * d;
            const double p = exp(scale * dot(qi, kj, d) - lse[r]);
            double dp = 0.0;
            for (int h = 0; h < nv; ++h)
                dp += dot(dout + h * sec + (size_t)r * d, v + h * sec + base + (size_t)j * d, d);
            const double ds = p * (dp - D[r]);
            for (int c = 0; c < d; ++c) dqi[c] += ds * kj[c];
        }
        for (int c = 0; c < d; ++c) dqi[c] *= scale;
    }

    /* 4. pass over key rows: dV_h[j] = sum_i P_ij dO_h[i]; dK_j = scale * sum_i dS_ij q_i */
#pragma omp parallel for schedule(static)
    for (long r = 0; r < (long)BH * N; ++r) {
        const int bh = (int)(r / N), j = (int)(r % N);
        const size_t base = (size_t)bh * N * d;
        const double* kj = k + (size_t)r * d;
        double* dkj = dk + (size_t)r * d;
        for (int c = 0; c < d; ++c) dkj[c] = 0.0;
        for (int h = 0; h < nv; ++h)
            for (int c = 0; c < d; ++c) dv[h * sec + (size_t)r * d + c] = 0.0;
        for (int i = 0; i < N; ++i) {
            const size_t ri = (size_t)bh * N + i;
            const double* qi = q + base + (size_t)i * d;
            const double p = exp(scale * dot(qi, kj, d) - lse[ri]);
            double dp = 0.0;
            for (int h = 0; h < nv; ++h) {
                const double* doi = dout + h * sec + ri * d;
                dp += dot(doi, v + h * sec + (size_t)r * d, d);
                double* dvj = dv + h * sec + (size_t)r * d;
                for (int c = 0; c < d; ++c) dvj[c] += p * doi[c];
            }
            const double ds = p * (dp - D[ri]);
            for (int c = 0; c < d; ++c) dkj[c] += ds * qi[c];
        }
        for (int c = 0; c < d; ++c) dkj[c] *= scale;
    }

done:
    if (!o_out) free(o);
    if (!lse_out) free(lse);
    if (!D_out) free(D);
    return err;
}

/*
 * PSA attention merge ("Struct PsaMergeAttnRuntimeOp": the op after the lo/hi
 * pair; its backward takes d_merged, d_lo, d_hi, c, H, W and the head count,
 * one thread block per (batch*head, position)).  The pages do not spell the
 * channel order out; the reading taken here: the merged tensor is [B, c, H, W]
 * with c = 2 * heads * d channels, the lo outputs of every head in the low
 * half of the channels and the hi outputs in the high half, head-major inside
 * each half, positions n = y * W + x:
 *   merged[b, s*heads*d + h*d + j, n] = O_s[b*heads + h, n, j],   s = 0 (lo), 1 (hi)
 * The merge is a permutation of elements, so its backward is the inverse
 * gather:
 *   dO_s[b*heads + h, n, j] = d_merged[b, s*heads*d + h*d + j, n]
 * Layouts: o_lo, o_hi, d_lo, d_hi [B*heads, N, d]; merged [B, c, N]; fp64.
 */
int psa_oracle_merge_fwd(int B, int heads, int N, int d, const double* o_lo, const double* o_hi,
                         double* merged) {
    if (B < 0 || heads <= 0 || N < 0 || d <= 0) return -1;
    const long c = 2L * heads * d;
    for (int b = 0; b < B; ++b)
        for (int s = 0; s < 2; ++s)
            for (int h = 0; h < heads; ++h)
                for (int j = 0; j < d; ++j)
                    for (int n = 0; n < N; ++n) {
                        const double* o = s == 0 ? o_lo : o_hi;
                        merged[((size_t)b * c + (size_t)s * heads * d + (size_t)h * d + j) * N + n] =
                            o[(((size_t)b * heads + h) * N + n) * d + j];
                    }
    return 0;
}

int psa_oracle_merge_bwd(int B, int heads, int N, int d, const double* d_merged, double* d_lo,
                         double* d_hi) {
    if (B < 0 || heads <= 0 || N < 0 || d <= 0) return -1;
    const long c = 2L * heads * d;
    for (int b = 0; b < B; ++b)
        for (int s = 0; s < 2; ++s)
            for (int h = 0; h < heads; ++h)
                for (int n = 0; n < N; ++n)
                    for (int j = 0; j < d; ++j) {
                        double* g = s == 0 ? d_lo : d_hi;
                        g[(((size_t)b * heads + h) * N + n) * d + j] =
                            d_merged[((size_t)b * c + (size_t)s * heads * d + (size_t)h * d + j) * N + n];
                    }
    return 0;
}
