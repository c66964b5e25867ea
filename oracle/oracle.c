/*
 * CPU oracle for the DSpark per-cycle draft step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * definition of what the CUDA path computes.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load it; the library never does.
 * It shares no code, header or table with the CUDA side.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared oracle.c -lm
 * Arithmetic: IEEE double, one operation at a time (no FMA contraction, no SIMD,
 * no threads), loops in the order the method states them.
 *
 * Sources (web pages describing DSpark speculative decoding):
 *  - vllm.cpp issue #436 "SPEC-DSPARK W7: the sequential Markov sample loop is
 *    HOST-side", sections "Measured" and "The fix": the per-step Markov chain
 *    IndexSelect(markov_w1, prev) -> GEMV against markov_w2 -> add the step's base
 *    row -> greedy argmax with lowest-index tie-break -> d2t map (identity when the
 *    checkpoint ships none) -> prev carried to the next step; markov_w2 is
 *    [draft_vocab, markov_rank] bf16 ("W7 LANDED").
 *  - ds4 PR #772 "dspark: cut per-cycle CUDA overheads", section "Summary": the
 *    proposer's confidence probe is a 7424-wide matvec of the hidden state against
 *    Q8_0 weights whose result gates the proposal length.
 *  - SharpInference issue #441 "DSpark GPU draft round runs ~3x the bandwidth
 *    floor", sections "Observation" and "Proposed work": the draft projections are
 *    fp16 GEMMs with M = B = 7 rows, Y = X W^T with the weight read once for all rows;
 *    the weight-stationary kernels it reuses read quantized (Q8_0) weights.
 *
 * Parity pins (tests/test_oracle_*.py): exact brute force with rational
 * arithmetic on tiny inputs, the zero-markov_w2 closed form, identity vs
 * injective d2t, constructed ties, argmax certificates, batch invariance,
 * power-of-two scaling, vocab-permutation equivariance; for the probe one-hot and
 * all-ones hidden vectors and the logit-space gate; for the matvec M=1, identity W,
 * row independence of M; fp16 decode/encode against numpy's binary16 routines.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- number formats ---------------------------------------------------------- */

/* bf16 is the upper half of an IEEE binary32; the widening is exact. */
double oracle_bf16_to_f64(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t bits)
{
    int sign = bits >> 15;
    int e = (bits >> 10) & 0x1f;
    int m = bits & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);     /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* Round a double to the nearest binary16 value, ties to even; overflow gives inf. */
uint16_t oracle_f64_to_f16_rne(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x))
        return 0x7e00;
    if (a == 0.0)
        return sign;
    /* scale so that the binary16 quantum becomes 1 */
    int e;
    frexp(a, &e);              /* a = f * 2^e, f in [0.5, 1) */
    int exp16 = e - 1;         /* a in [2^exp16, 2^(exp16+1)) */
    int q;                     /* quantum exponent */
    if (exp16 < -14)
        q = -24;               /* subnormal range: quantum 2^-24 */
    else
        q = exp16 - 10;
    double s = ldexp(a, -q);   /* exact: a power-of-two scaling */
    double r = floor(s);
    double frac = s - r;       /* exact */
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0))
        r += 1.0;
    double v = ldexp(r, q);    /* rounded magnitude */
    if (v >= 65520.0 || v > 65504.0)
        return sign | 0x7c00;
    /* encode v */
    if (v < ldexp(1.0, -14)) {
        uint16_t m = (uint16_t)ldexp(v, 24);
        return sign | m;
    }
    int ev;
    frexp(v, &ev);
    int E = ev - 1;                              /* v in [2^E, 2^(E+1)) */
    uint16_t m = (uint16_t)(ldexp(v, 10 - E) - 1024.0);
    return sign | (uint16_t)((E + 15) << 10) | m;
}

/* ---- Markov block draft -------------------------------------------------------- */

/*
 * For every request r and draft position i = 0..k-1 (vllm.cpp #436, "The fix"):
 *   h[j]     = markov_w1[p, j]                                  (IndexSelect by prev p)
 *   bias[v]  = sum_{j<R} markov_w2[v, j] * h[j]                 (GEMV, j ascending)
 *   logit[v] = base[r, i, v] + bias[v]                          (the step's base row)
 *   id       = smallest v with logit[v] == max_u logit[u]       (greedy, lowest index)
 *   out[r,i] = d2t ? d2t[id] : id                               (identity without d2t)
 *   p        = id (draft-space id; forced_prev[r,i] replaces it when given)
 * p starts at prev0[r].
 *
 * Arrays are row-major: base [B,k,V] fp32; w1, w2 [V,R] bf16 bits; d2t [V] or NULL;
 * prev0 [B]; forced_prev [B,k] or NULL; out_ids, draft_ids [B,k];
 * logits_out, bias_out [B,k,V] or NULL.
 * Returns 0, or -1 on a bad argument or an out-of-range prev.
 */
int oracle_markov_draft(const float *base, const uint16_t *w1, const uint16_t *w2,
                        const int32_t *d2t, const int64_t *prev0, int B, int k, int V,
                        int R, const int64_t *forced_prev, int64_t *out_ids,
                        int64_t *draft_ids, double *logits_out, double *bias_out)
{
    if (B < 0 || k < 0 || V <= 0 || R <= 0 || !base || !w1 || !w2 || !prev0)
        return -1;
    double h[4096];
    if (R > 4096)
        return -1;
    for (int r = 0; r < B; ++r) {
        int64_t p = prev0[r];
        for (int i = 0; i < k; ++i) {
            if (p < 0 || p >= V)
                return -1;
            for (int j = 0; j < R; ++j)
                h[j] = oracle_bf16_to_f64(w1[(size_t)p * R + j]);
            const float *base_row = base + ((size_t)r * k + i) * V;
            double best = -INFINITY;
            int64_t best_v = -1;
            for (int v = 0; v < V; ++v) {
                double bias = 0.0;
                for (int j = 0; j < R; ++j)
                    bias += oracle_bf16_to_f64(w2[(size_t)v * R + j]) * h[j];
                double logit = (double)base_row[v] + bias;
                size_t o = ((size_t)r * k + i) * V + v;
                if (logits_out)
                    logits_out[o] = logit;
                if (bias_out)
                    bias_out[o] = bias;
                if (best_v < 0 || logit > best) {  /* strict: the first maximum wins */
                    best = logit;
                    best_v = v;
                }
            }
            if (draft_ids)
                draft_ids[(size_t)r * k + i] = best_v;
            if (out_ids)
                out_ids[(size_t)r * k + i] = d2t ? (int64_t)d2t[best_v] : best_v;
            p = forced_prev ? forced_prev[(size_t)r * k + i] : best_v;
        }
    }
    return 0;
}

/* ---- confidence probe ---------------------------------------------------------- */

/*
 * ds4 PR #772, "Summary": one Q8_0 weight row against the hidden vector.
 * Q8_0 block b (34 bytes): fp16 scale d_b (little endian), then 32 int8 q_{b,j};
 * weight element 32b+j = d_b * q_{b,j}.
 *   z    = bias + sum_b d_b * (sum_j q_{b,j} * x[32b+j])
 *   gate = sigmoid(z) >= threshold, evaluated as z >= log(t / (1 - t))
 * hidden [n, K] fp32; z_out, gate_out [n] (either may be NULL).
 * Returns 0, or -1 on a bad argument.
 */
int oracle_conf_probe(const uint8_t *wq, const float *hidden, int K, int n, double bias,
                      double threshold, double *z_out, int32_t *gate_out)
{
    if (K <= 0 || K % 32 || n < 0 || !wq || !hidden || !(threshold > 0.0 && threshold < 1.0))
        return -1;
    double t_logit = log(threshold / (1.0 - threshold));
    int nb = K / 32;
    for (int p = 0; p < n; ++p) {
        const float *x = hidden + (size_t)p * K;
        double z = bias;
        for (int b = 0; b < nb; ++b) {
            const uint8_t *blk = wq + (size_t)b * 34;
            uint16_t dbits = (uint16_t)(blk[0] | ((uint16_t)blk[1] << 8));
            double d = oracle_f16_to_f64(dbits);
            double s = 0.0;
            for (int j = 0; j < 32; ++j) {
                int8_t q;
                memcpy(&q, blk + 2 + j, 1);
                s += (double)q * (double)x[32 * b + j];
            }
            z += d * s;
        }
        if (z_out)
            z_out[p] = z;
        if (gate_out)
            gate_out[p] = (z >= t_logit) ? 1 : 0;
    }
    return 0;
}

/* ---- weight-stationary projection matvec ---------------------------------------- */

/*
 * SharpInference #441: Y[m, n] = sum_k X[m, k] * W[n, k]  (W is [N, K], out x in).
 * W, X fp16 bits; Y [M, N] double; Y16 [M, N] fp16 bits of RNE(Y) or NULL.
 * Returns 0, or -1 on a bad argument.
 */
int oracle_ws_matvec(const uint16_t *W, const uint16_t *X, int M, int N, int K, double *Y,
                     uint16_t *Y16)
{
    if (M < 0 || N < 0 || K < 0 || !W || !X || !Y)
        return -1;
    /* decode the fp16 operands once (exact), then sum k ascending per output */
    double *xd = malloc(sizeof(double) * ((size_t)M * K + 1));
    double *wd = malloc(sizeof(double) * ((size_t)K + 1));
    if (!xd || !wd) {
        free(xd);
        free(wd);
        return -1;
    }
    for (size_t e = 0; e < (size_t)M * K; ++e)
        xd[e] = oracle_f16_to_f64(X[e]);
    for (int n = 0; n < N; ++n) {
        for (int kk = 0; kk < K; ++kk)
            wd[kk] = oracle_f16_to_f64(W[(size_t)n * K + kk]);
        for (int m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int kk = 0; kk < K; ++kk)
                acc += xd[(size_t)m * K + kk] * wd[kk];
            Y[(size_t)m * N + n] = acc;
            if (Y16)
                Y16[(size_t)m * N + n] = oracle_f64_to_f16_rne(acc);
        }
    }
    free(xd);
    free(wd);
    return 0;
}

/* ---- quantized weight-stationary matvec ---------------------------------------- */

/*
 * SharpInference #441, "Proposed work": the weight-stationary kernels of #194 read
 * quantized weights.  With Q8_0 weights (row n, block b: fp16 scale d_{n,b} and int8 q):
 *   Y[m, n] = sum_b d_{n,b} * sum_{j<32} q_{n,b,j} * X[m, 32b + j]
 * W_q8 is [N][K/32] blocks of 34 bytes (ggml layout, as in oracle_conf_probe); X fp16 [M, K];
 * Y [M, N] double.  Returns 0, or -1 on a bad argument.
 */
int oracle_ws_matvec_q8(const uint8_t *Wq8, const uint16_t *X, int M, int N, int K, double *Y)
{
    if (M < 0 || N < 0 || K <= 0 || K % 32 || !Wq8 || !X || !Y)
        return -1;
    int nb = K / 32;
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int b = 0; b < nb; ++b) {
                const uint8_t *blk = Wq8 + ((size_t)n * nb + b) * 34;
                double d = oracle_f16_to_f64((uint16_t)(blk[0] | ((uint16_t)blk[1] << 8)));
                double s = 0.0;
                for (int j = 0; j < 32; ++j) {
                    int8_t q;
                    memcpy(&q, blk + 2 + j, 1);
                    s += (double)q * oracle_f16_to_f64(X[(size_t)m * K + 32 * b + j]);
                }
                acc += d * s;
            }
            Y[(size_t)m * N + n] = acc;
        }
    return 0;
}
