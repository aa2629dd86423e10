/*
 * Exact scaled-dot-product attention (forward and VJP) in double precision.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the oracle that the CUDA path is
 * checked against. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may build, load or call it; the product path never does.
 * It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes is the plain definition of attention, written out one
 * query row at a time (every row is the full definition; nothing is blocked,
 * fused or reordered):
 *
 *   S[i,j]  = scale * sum_d Q[b,h,i,d] * K[b,g,j,d]            g = h / (Hq/Hkv)
 *   allowed(i,j) = !(causal && j > i) && !(W > 0 && i >= j && i - j >= W)
 *   LSE[i]  = log sum_{j allowed} exp(S[i,j])                  (natural log)
 *   P[i,j]  = exp(S[i,j] - LSE[i]) if allowed, else 0
 *   O[i,:]  = sum_j P[i,j] * V[b,g,j,:]
 *   dP[i,j] = sum_d dO[i,d] * V[b,g,j,d]
 *   Dv[i]   = sum_d dO[i,d] * O[i,d]                           (exact O)
 *   dS[i,j] = P[i,j] * (dP[i,j] - Dv[i])
 *   dQ[i,:] = scale * sum_j dS[i,j] * K[b,g,j,:]
 *   dK[b,g,j,:] = scale * sum_{h in group g} sum_i dS[i,j] * Q[b,h,i,:]
 *   dV[b,g,j,:] =         sum_{h in group g} sum_i P[i,j]  * dO[b,h,i,:]
 *
 * Sources (page title, section):
 *  - "mlx-bun 0.0.4: package/src/model/flash-attention.ts", forward shader:
 *    score = scale * q.k, causal mask (key > query), sliding-window mask
 *    (query >= key and query - key >= window), online softmax whose result is
 *    O = o / l and L = m + log(l); GQA head map kv_head = head / reps.
 *  - same page, backward passes 1-3: D_i = rowsum(O o dO), p = exp(s - L),
 *    dp = dO.v, ds = p * (dp - D), dV += p dO, dK += ds q scale,
 *    dQ += ds k scale; dK/dV owned per KV head and summed over its reps.
 *  - same page, manualSdpa: the materialised softmax(QK^T*scale + mask) V
 *    that the flash kernels are an exact reformulation of.
 *  - "R/ag_flash_attn.R" (ggmlR), .ag_flash_mask: causal means query j sees
 *    keys 1..j (top-left alignment when the lengths differ).
 *
 * Readings where the pages leave a step open:
 *  - A row with no allowed key (possible only with a window and Tq > Tkv)
 *    has O = 0, LSE = -inf, and contributes nothing to any gradient.
 *  - The window counts the query's own key: a row sees W keys of its past.
 *  - No clamping of exponent arguments: masked entries are exactly zero.
 *
 * Layouts (all row-major, contiguous): Q, O, dO, dQ [B,Hq,Tq,D];
 * K, V, dK, dV [B,Hkv,Tkv,D]; LSE, Dv [B,Hq,Tq].
 *
 * Row restriction: every entry point takes [row_lo, row_hi). Forward outputs
 * and dQ are computed for those query rows only (others are left untouched).
 * dK and dV are the sums over those query rows only; they equal the full
 * gradient for every key row whose allowed query rows all lie in the range.
 * [0, Tq) gives the full result.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static int allowed(int64_t i, int64_t j, int causal, int window) {
    if (causal && j > i) return 0;
    if (window > 0 && i >= j && i - j >= window) return 0;
    return 1;
}

/* One query row of the forward definition. s[] (Tkv scratch) receives
 * P[i,:] on return; o_row receives O[i,:]; the return value is LSE[i]. */
static double fwd_row(const double* qi, const double* kg, const double* vg,
                      int64_t i, int Tkv, int D, double scale, int causal,
                      int window, double* s, double* o_row) {
    double m = -INFINITY;
    for (int j = 0; j < Tkv; ++j) {
        if (!allowed(i, j, causal, window)) { s[j] = -INFINITY; continue; }
        const double* kj = kg + (int64_t)j * D;
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += qi[d] * kj[d];
        s[j] = scale * acc;
        if (s[j] > m) m = s[j];
    }
    for (int d = 0; d < D; ++d) o_row[d] = 0.0;
    if (m == -INFINITY) {                       /* no allowed key */
        for (int j = 0; j < Tkv; ++j) s[j] = 0.0;
        return -INFINITY;
    }
    double sum = 0.0;
    for (int j = 0; j < Tkv; ++j)
        if (s[j] != -INFINITY) sum += exp(s[j] - m);
    const double lse = m + log(sum);
    for (int j = 0; j < Tkv; ++j) {
        s[j] = (s[j] == -INFINITY) ? 0.0 : exp(s[j] - lse);
        if (s[j] != 0.0) {
            const double* vj = vg + (int64_t)j * D;
            for (int d = 0; d < D; ++d) o_row[d] += s[j] * vj[d];
        }
    }
    return lse;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Forward: O and LSE for query rows [row_lo, row_hi) of every (b, h). */
void oracle_attn_fwd(const double* q, const double* k, const double* v,
                     double* o, double* lse,
                     int B, int Hq, int Hkv, int Tq, int Tkv, int D,
                     double scale, int causal, int window,
                     int row_lo, int row_hi) {
    const int reps = Hq / Hkv;
    #pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(Tkv > 0 ? Tkv : 1));
        #pragma omp for collapse(2) schedule(dynamic, 1)
        for (int bh = 0; bh < B * Hq; ++bh)
            for (int i = row_lo; i < row_hi; ++i) {
                const int b = bh / Hq, h = bh % Hq, g = h / reps;
                const double* qi = q + (((int64_t)b * Hq + h) * Tq + i) * D;
                const double* kg = k + ((int64_t)b * Hkv + g) * (int64_t)Tkv * D;
                const double* vg = v + ((int64_t)b * Hkv + g) * (int64_t)Tkv * D;
                double* orow = o + (((int64_t)b * Hq + h) * Tq + i) * D;
                lse[((int64_t)b * Hq + h) * Tq + i] =
                    fwd_row(qi, kg, vg, i, Tkv, D, scale, causal, window, s, orow);
            }
        free(s);
    }
}

/* VJP: dQ for query rows [row_lo, row_hi); dK, dV as the sum over those rows
 * (see the header). Optional outputs o/lse/dvec (may be NULL) receive the
 * exact O, LSE and D-vector of the covered rows. dk and dv are overwritten.
 *
 * Each output is computed straight from its own defining sum, in three
 * passes that are each parallel over independent outputs:
 *   1. per query row i: LSE_i and O_i (the forward definition), D_i = dO_i.O_i
 *   2. per query row i: dQ_i = scale * sum_j P_ij (dP_ij - D_i) K_j
 *   3. per key row j of group g: dK_j = scale * sum_{h in g} sum_i dS_ij Q_i,
 *                                dV_j = sum_{h in g} sum_i P_ij dO_i
 * with P_ij = exp(S_ij - LSE_i) on visible pairs and dP_ij = dO_i . V_j. */
static double dot(const double* a, const double* b, int D) {
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += a[d] * b[d];
    return acc;
}

void oracle_attn_bwd(const double* q, const double* k, const double* v,
                     const double* dout,
                     double* dq, double* dk, double* dv,
                     double* o, double* lse, double* dvec,
                     int B, int Hq, int Hkv, int Tq, int Tkv, int D,
                     double scale, int causal, int window,
                     int row_lo, int row_hi) {
    const int reps = Hq / Hkv;
    const int nrows = row_hi > row_lo ? row_hi - row_lo : 0;
    /* row statistics of the covered rows, indexed [b][h][i - row_lo] */
    double* L = (double*)malloc(sizeof(double) * ((size_t)B * Hq * nrows + 1));
    double* Dv = (double*)malloc(sizeof(double) * ((size_t)B * Hq * nrows + 1));

    /* pass 1: LSE, O and the D-vector of every covered row */
    #pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * (size_t)(Tkv > 0 ? Tkv : 1));
        double* orow = (double*)malloc(sizeof(double) * (size_t)D);
        #pragma omp for collapse(2) schedule(dynamic, 1)
        for (int bh = 0; bh < B * Hq; ++bh)
            for (int i = row_lo; i < row_hi; ++i) {
                const int b = bh / Hq, h = bh % Hq, g = h / reps;
                const int64_t row = ((int64_t)b * Hq + h) * Tq + i;
                const double* kg = k + ((int64_t)b * Hkv + g) * (int64_t)Tkv * D;
                const double* vg = v + ((int64_t)b * Hkv + g) * (int64_t)Tkv * D;
                const double Li = fwd_row(q + row * D, kg, vg, i, Tkv, D, scale,
                                          causal, window, p, orow);
                const double Di = dot(dout + row * D, orow, D);
                L[(int64_t)bh * nrows + (i - row_lo)] = Li;
                Dv[(int64_t)bh * nrows + (i - row_lo)] = Di;
                if (o) for (int d = 0; d < D; ++d) o[row * D + d] = orow[d];
                if (lse) lse[row] = Li;
                if (dvec) dvec[row] = Di;
            }
        free(orow);
        free(p);
    }

    /* pass 2: dQ_i = scale * sum_j dS_ij K_j */
    #pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int bh = 0; bh < B * Hq; ++bh)
        for (int i = row_lo; i < row_hi; ++i) {
            const int b = bh / Hq, h = bh % Hq, g = h / reps;
            const int64_t row = ((int64_t)b * Hq + h) * Tq + i;
            const double* qi = q + row * D;
            const double* doi = dout + row * D;
            const double Li = L[(int64_t)bh * nrows + (i - row_lo)];
            const double Di = Dv[(int64_t)bh * nrows + (i - row_lo)];
            double* dqi = dq + row * D;
            for (int d = 0; d < D; ++d) dqi[d] = 0.0;
            if (Li == -INFINITY) continue;              /* no visible key */
            for (int j = 0; j < Tkv; ++j) {
                if (!allowed(i, j, causal, window)) continue;
                const double* kj = k + (((int64_t)b * Hkv + g) * Tkv + j) * D;
                const double* vj = v + (((int64_t)b * Hkv + g) * Tkv + j) * D;
                const double pij = exp(scale * dot(qi, kj, D) - Li);
                const double ds = pij * (dot(doi, vj, D) - Di);
                for (int d = 0; d < D; ++d) dqi[d] += scale * ds * kj[d];
            }
        }

    /* pass 3: dK_j and dV_j, summed over the group's query heads and rows */
    #pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int bg = 0; bg < B * Hkv; ++bg)
        for (int j = 0; j < Tkv; ++j) {
            const int b = bg / Hkv, g = bg % Hkv;
            const double* kj = k + ((int64_t)bg * Tkv + j) * D;
            const double* vj = v + ((int64_t)bg * Tkv + j) * D;
            double* dkj = dk + ((int64_t)bg * Tkv + j) * D;
            double* dvj = dv + ((int64_t)bg * Tkv + j) * D;
            for (int d = 0; d < D; ++d) { dkj[d] = 0.0; dvj[d] = 0.0; }
            for (int h = g * reps; h < (g + 1) * reps; ++h)
                for (int i = row_lo; i < row_hi; ++i) {
                    if (!allowed(i, j, causal, window)) continue;
                    const int bh = b * Hq + h;
                    const double Li = L[(int64_t)bh * nrows + (i - row_lo)];
                    if (Li == -INFINITY) continue;
                    const int64_t row = (int64_t)bh * Tq + i;
                    const double* qi = q + row * D;
                    const double* doi = dout + row * D;
                    const double pij = exp(scale * dot(qi, kj, D) - Li);
                    const double ds = pij * (dot(doi, vj, D) - Dv[(int64_t)bh * nrows + (i - row_lo)]);
                    for (int d = 0; d < D; ++d) {
                        dkj[d] += scale * ds * qi[d];
                        dvj[d] += pij * doi[d];
                    }
                }
        }
    free(Dv);
    free(L);
}
