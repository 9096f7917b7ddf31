/*
 * fp64 CPU oracle for the FlashAttention-2 forward pass.
 *
 * TEST INFRASTRUCTURE ONLY. This file is compiled into oracle/liboracle.so and
 * is called by the tests, by the package's smoke check and by the benchmark's
 * CPU-baseline leg. The GPU library never links, loads or calls it, and it
 * shares no code, header or table with the GPU path.
 *
 * What it computes. The forward pass of FlashAttention-2 is exact
 * scaled-dot-product attention ("A Case Study in CUDA Kernel Fusion:
 * Implementing FlashAttention-2 on NVIDIA Hopper Architecture using the
 * CUTLASS Library", abstract: a "memory-aware scaled dot-product attention"
 * whose forward pass fuses an online softmax with two back-to-back GEMMs).
 * Tiling and the online softmax change only the rounding order, so the oracle
 * is the plain definition, with the full score row materialised:
 *
 *     s_j    = scale * sum_t q_t k_{j,t}          (j = 0 .. N-1)
 *     m      = max_j s_j
 *     p_j    = exp(s_j - m)
 *     l      = sum_j p_j
 *     o      = (sum_j p_j v_j) / l
 *     lse    = m + ln(l)
 *
 * Scope follows "FlashAttention-2 from scratch on Ampere, Part 1"
 * (lubitschian.com/flash/Part-1), section "Kernel Specification": forward
 * only, non-causal, equal query/key/value lengths, 16-bit (bf16/fp16) inputs,
 * softmax in fp32 on the GPU (fp64 here). The logsumexp output is the natural
 * log of sum_j exp(s_j) with the scale included. Grouped KV heads follow the
 * query-head packing of "FlashAttention-3 for Inference: INT8 Quantization and
 * Query Head Packing for MQA/GQA" (Colfax Research author page): query head h
 * reads KV head h / (Hq / Hkv).
 *
 * The generalised form (oracle_attention_ex_rows) covers unequal and ragged
 * query/key lengths and the causal mask, the variants the Ampere series
 * excludes from its Kernel Specification (equal lengths, non-causal,
 * lengths divisible by the block size).
 *
 * Every function here is pinned by tests/test_oracle.py against closed forms,
 * invariants, a hand-computed case and an independent library computation.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_BF16 0
#define ORACLE_FP16 1

/* Exact value of a bf16 bit pattern: the top half of an IEEE binary32. */
static double decode_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Exact value of an IEEE binary16 bit pattern (sign, 5-bit exponent with bias
 * 15, 10-bit fraction; exponent 0 encodes subnormals, 31 encodes inf/NaN). */
static double decode_fp16(uint16_t b) {
    int sign = (b >> 15) & 1;
    int e = (b >> 10) & 0x1F;
    int f = b & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

static double decode16(uint16_t b, int dtype) {
    return dtype == ORACLE_FP16 ? decode_fp16(b) : decode_bf16(b);
}

/* Widen n 16-bit patterns to double (exact). */
void oracle_decode16(const uint16_t* bits, int64_t n, int dtype, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = decode16(bits[i], dtype);
}

/*
 * Step 1 of the definition for a whole K or V tensor: every 16-bit pattern
 * widened to its exact double value once, before any row uses it, so that
 * the per-row loops below read doubles. (Decoding is exact, so doing it
 * here rather than inside the loops changes no result.) Returns NULL if the
 * memory is not available.
 */
static double* decode_all(const uint16_t* bits, int64_t n, int dtype) {
    double* out = (double*)malloc(sizeof(double) * (size_t)n);
    if (!out) return NULL;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = decode16(bits[i], dtype);
    return out;
}

/*
 * Attention forward for a list of query rows.
 *
 * q:   [B, Hq, N, d]   16-bit patterns, contiguous
 * k,v: [B, Hkv, N, d]  16-bit patterns, contiguous
 * rows: flat indices r = (b*Hq + h)*N + i of the query rows to compute, or
 *       NULL for all B*Hq*N rows in order (then nrows must equal B*Hq*N)
 * o_out:   [nrows, d] doubles, the unrounded output rows
 * lse_out: [nrows]    doubles, natural-log logsumexp of the scaled scores
 * nthreads: OpenMP threads (<= 0: library default)
 *
 * Returns 0, or -1 on invalid sizes.
 */
int oracle_attention_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                          int dtype, int64_t B, int64_t Hq, int64_t Hkv, int64_t N,
                          int64_t d, double scale, const int64_t* rows, int64_t nrows,
                          double* o_out, double* lse_out, int nthreads) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || N <= 0 || d <= 0 || Hq % Hkv) return -1;
    if (!rows && nrows != B * Hq * N) return -1;
    const int64_t G = Hq / Hkv;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    /* step 1: exact double values of K and V */
    double* kall = decode_all(k, B * Hkv * N * d, dtype);
    double* vall = decode_all(v, B * Hkv * N * d, dtype);
    if (!kall || !vall) {
        free(kall);
        free(vall);
        return -2;
    }

#pragma omp parallel
    {
        double* qrow = (double*)malloc(sizeof(double) * (size_t)d);
        double* s = (double*)malloc(sizeof(double) * (size_t)N);
        double* acc = (double*)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < nrows; ++r) {
            const int64_t flat = rows ? rows[r] : r;
            const int64_t i = flat % N;
            const int64_t h = (flat / N) % Hq;
            const int64_t b = flat / (N * Hq);
            const int64_t hk = h / G;
            const uint16_t* qp = q + ((b * Hq + h) * N + i) * d;
            const double* kp = kall + (b * Hkv + hk) * N * d;
            const double* vp = vall + (b * Hkv + hk) * N * d;

            for (int64_t t = 0; t < d; ++t) qrow[t] = decode16(qp[t], dtype);

            /* scores s_j = scale * <q, k_j> over the whole key sequence */
            double m = -INFINITY;
            for (int64_t j = 0; j < N; ++j) {
                double dot = 0.0;
                for (int64_t t = 0; t < d; ++t) dot += qrow[t] * kp[j * d + t];
                s[j] = scale * dot;
                if (s[j] > m) m = s[j];
            }
            /* max-subtracted softmax weights, their sum, and the weighted sum of V */
            double l = 0.0;
            for (int64_t t = 0; t < d; ++t) acc[t] = 0.0;
            for (int64_t j = 0; j < N; ++j) {
                const double p = exp(s[j] - m);
                l += p;
                for (int64_t t = 0; t < d; ++t) acc[t] += p * vp[j * d + t];
            }
            for (int64_t t = 0; t < d; ++t) o_out[r * d + t] = acc[t] / l;
            lse_out[r] = m + log(l);
        }
        free(qrow);
        free(s);
        free(acc);
    }
    free(kall);
    free(vall);
    return 0;
}

/*
 * The normalised softmax row P_i = exp(s - lse) of one query row, for the
 * oracle's own invariant checks (rows of P sum to one). p_out: [N] doubles.
 */
int oracle_softmax_row(const uint16_t* q, const uint16_t* k, int dtype, int64_t B,
                       int64_t Hq, int64_t Hkv, int64_t N, int64_t d, double scale,
                       int64_t row, double* p_out) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || N <= 0 || d <= 0 || Hq % Hkv) return -1;
    if (row < 0 || row >= B * Hq * N) return -1;
    const int64_t G = Hq / Hkv;
    const int64_t i = row % N, h = (row / N) % Hq, b = row / (N * Hq), hk = h / G;
    const uint16_t* qp = q + ((b * Hq + h) * N + i) * d;
    const uint16_t* kp = k + (b * Hkv + hk) * N * d;
    double m = -INFINITY;
    for (int64_t j = 0; j < N; ++j) {
        double dot = 0.0;
        for (int64_t t = 0; t < d; ++t) dot += decode16(qp[t], dtype) * decode16(kp[j * d + t], dtype);
        p_out[j] = scale * dot;
        if (p_out[j] > m) m = p_out[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < N; ++j) {
        p_out[j] = exp(p_out[j] - m);
        l += p_out[j];
    }
    for (int64_t j = 0; j < N; ++j) p_out[j] /= l;
    return 0;
}

/*
 * Generalised forward: query length Nq and key length Nk may differ and need
 * not be multiples of any block size, and an optional causal mask. Query row
 * i may attend key j iff j < kend(i), with
 *     kend(i) = Nk                          (non-causal)
 *     kend(i) = min(Nk, i + 1 + Nk - Nq)    (causal, aligned to the end of
 *                                            the key sequence)
 * which for Nq = Nk is the usual lower-triangular mask j <= i. A row with no
 * allowed key (causal with Nq > Nk) has o = 0 and lse = -inf.
 *
 * q: [B, Hq, Nq, d]; k, v: [B, Hkv, Nk, d]; rows index [B, Hq, Nq] flat
 * (NULL = all). Returns 0, or -1 on invalid sizes.
 */
int oracle_attention_ex_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v, int dtype,
                             int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d,
                             double scale, int causal, const int64_t* rows, int64_t nrows,
                             double* o_out, double* lse_out, int nthreads) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || Nk <= 0 || d <= 0 || Hq % Hkv) return -1;
    if (!rows && nrows != B * Hq * Nq) return -1;
    const int64_t G = Hq / Hkv;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    /* step 1: exact double values of K and V */
    double* kall = decode_all(k, B * Hkv * Nk * d, dtype);
    double* vall = decode_all(v, B * Hkv * Nk * d, dtype);
    if (!kall || !vall) {
        free(kall);
        free(vall);
        return -2;
    }

#pragma omp parallel
    {
        double* qrow = (double*)malloc(sizeof(double) * (size_t)d);
        double* s = (double*)malloc(sizeof(double) * (size_t)Nk);
        double* acc = (double*)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < nrows; ++r) {
            const int64_t flat = rows ? rows[r] : r;
            const int64_t i = flat % Nq;
            const int64_t h = (flat / Nq) % Hq;
            const int64_t b = flat / (Nq * Hq);
            const int64_t hk = h / G;
            const uint16_t* qp = q + ((b * Hq + h) * Nq + i) * d;
            const double* kp = kall + (b * Hkv + hk) * Nk * d;
            const double* vp = vall + (b * Hkv + hk) * Nk * d;
            int64_t kend = Nk;
            if (causal) {
                const int64_t lim = i + 1 + Nk - Nq;
                kend = lim < Nk ? lim : Nk;
            }
            if (kend <= 0) {
                for (int64_t t = 0; t < d; ++t) o_out[r * d + t] = 0.0;
                lse_out[r] = -INFINITY;
                continue;
            }
            for (int64_t t = 0; t < d; ++t) qrow[t] = decode16(qp[t], dtype);
            double m = -INFINITY;
            for (int64_t j = 0; j < kend; ++j) {
                double dot = 0.0;
                for (int64_t t = 0; t < d; ++t) dot += qrow[t] * kp[j * d + t];
                s[j] = scale * dot;
                if (s[j] > m) m = s[j];
            }
            double l = 0.0;
            for (int64_t t = 0; t < d; ++t) acc[t] = 0.0;
            for (int64_t j = 0; j < kend; ++j) {
                const double p = exp(s[j] - m);
                l += p;
                for (int64_t t = 0; t < d; ++t) acc[t] += p * vp[j * d + t];
            }
            for (int64_t t = 0; t < d; ++t) o_out[r * d + t] = acc[t] / l;
            lse_out[r] = m + log(l);
        }
        free(qrow);
        free(s);
        free(acc);
    }
    free(kall);
    free(vall);
    return 0;
}

/*
 * Backward pass of attention in fp64, by its definition (the gradient of the
 * forward above with respect to q, k and v for an upstream gradient dO):
 *     S = scale Q K^T (causal: keys j >= kend(i) excluded), P = softmax(S),
 *     O = P V, D_i = sum_t dO_it O_it, dP = dO V^T,
 *     dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO.
 * With grouped heads, dK and dV of a KV head sum over its query heads.
 * Inputs q, k, v, dout are 16-bit patterns ([B,Hq,N,d], [B,Hkv,N,d],
 * [B,Hkv,N,d], [B,Hq,N,d]); outputs are doubles of the same shapes as q, k, v.
 * Equal query/key lengths N. Rows with no allowed key contribute nothing.
 *
 * Optional bound sums (each pointer may be NULL). They are not part of the
 * gradient: they are the absolute sums that bound, element by element, how
 * far a computation that rounds P, dS and O to 16 bits and accumulates in
 * fp32 can land from the exact gradient. With a_it = sum_j P_ij |V_jt|,
 * E_i = sum_t |dO_it| (|O_it| + a_it) and F_ij = sum_t |dO_it| |V_jt|:
 *   bq [3, B,Hq,N,d]:  A = scale sum_j |dS_ij| |K_jt|,
 *                      BE = scale E_i sum_j P_ij |K_jt|,
 *                      BF = scale sum_j P_ij F_ij |K_jt|
 *   bk [3, B,Hkv,N,d]: the same three sums over the query rows i (and the
 *                      query heads of the KV head) with |Q_it| for |K_jt|
 *   bv [B,Hkv,N,d]:    A = sum_i P_ij |dO_it|
 */
int oracle_attention_bwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dout,
                         int dtype, int64_t B, int64_t Hq, int64_t Hkv, int64_t N, int64_t d,
                         double scale, int causal, double* dq, double* dk, double* dv,
                         double* bq, double* bk, double* bv) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || N <= 0 || d <= 0 || Hq % Hkv) return -1;
    const int64_t G = Hq / Hkv;
    const int64_t nq = B * Hq * N * d, nkv = B * Hkv * N * d;
    /* the 16-bit inputs as exact doubles */
    double* Q = decode_all(q, nq, dtype);
    double* K = decode_all(k, nkv, dtype);
    double* V = decode_all(v, nkv, dtype);
    double* dO = decode_all(dout, nq, dtype);
    if (!Q || !K || !V || !dO) {
        free(Q);
        free(K);
        free(V);
        free(dO);
        return -2;
    }
    for (int64_t i = 0; i < nkv; ++i) {
        dk[i] = 0.0;
        dv[i] = 0.0;
        if (bk) bk[i] = bk[nkv + i] = bk[2 * nkv + i] = 0.0;
        if (bv) bv[i] = 0.0;
    }
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t hk = 0; hk < Hkv; ++hk) {
            const int64_t kvoff = (b * Hkv + hk) * N * d;
            const double* kp = K + kvoff;
            const double* vp = V + kvoff;
            for (int64_t g = 0; g < G; ++g) {
                const int64_t h = hk * G + g;
                const int64_t qoff = (b * Hq + h) * N * d;
                const double* qp = Q + qoff;
                const double* dop = dO + qoff;
#pragma omp parallel
                {
                    double* P = (double*)malloc(sizeof(double) * (size_t)N);
                    double* dS = (double*)malloc(sizeof(double) * (size_t)N);
                    double* F = (double*)malloc(sizeof(double) * (size_t)N);
                    double* o = (double*)malloc(sizeof(double) * (size_t)d);
                    double* a = (double*)malloc(sizeof(double) * (size_t)d);
                    /* per-thread dK, dV (and bound) rows, added up at the end */
                    const int nloc = 2 + (bk ? 3 : 0) + (bv ? 1 : 0);
                    double* loc = (double*)calloc((size_t)(nloc * N * d), sizeof(double));
                    double* dkl = loc;
                    double* dvl = loc + N * d;
                    double* bkl = bk ? loc + 2 * N * d : NULL;
                    double* bvl = bv ? loc + (2 + (bk ? 3 : 0)) * N * d : NULL;
#pragma omp for schedule(dynamic, 4)
                    for (int64_t i = 0; i < N; ++i) {
                        const int64_t kend = causal ? (i + 1 < N ? i + 1 : N) : N;
                        const double* qi = qp + i * d;
                        const double* doi = dop + i * d;
                        double m = -INFINITY;
                        for (int64_t j = 0; j < kend; ++j) {
                            double dot = 0.0;
                            for (int64_t t = 0; t < d; ++t) dot += qi[t] * kp[j * d + t];
                            P[j] = scale * dot;
                            if (P[j] > m) m = P[j];
                        }
                        double l = 0.0;
                        for (int64_t j = 0; j < kend; ++j) {
                            P[j] = exp(P[j] - m);
                            l += P[j];
                        }
                        for (int64_t t = 0; t < d; ++t) o[t] = a[t] = 0.0;
                        for (int64_t j = 0; j < kend; ++j) {
                            P[j] /= l;
                            for (int64_t t = 0; t < d; ++t) {
                                o[t] += P[j] * vp[j * d + t];
                                a[t] += P[j] * fabs(vp[j * d + t]);
                            }
                        }
                        double Di = 0.0, Ei = 0.0;
                        for (int64_t t = 0; t < d; ++t) {
                            Di += doi[t] * o[t];
                            Ei += fabs(doi[t]) * (fabs(o[t]) + a[t]);
                        }
                        for (int64_t j = 0; j < kend; ++j) {
                            double dp = 0.0, f = 0.0;
                            for (int64_t t = 0; t < d; ++t) {
                                dp += doi[t] * vp[j * d + t];
                                f += fabs(doi[t]) * fabs(vp[j * d + t]);
                            }
                            dS[j] = P[j] * (dp - Di);
                            F[j] = f;
                        }
                        for (int64_t t = 0; t < d; ++t) {
                            double acc = 0.0, sa = 0.0, se = 0.0, sf = 0.0;
                            for (int64_t j = 0; j < kend; ++j) {
                                const double kk = kp[j * d + t];
                                acc += dS[j] * kk;
                                sa += fabs(dS[j]) * fabs(kk);
                                se += P[j] * fabs(kk);
                                sf += P[j] * F[j] * fabs(kk);
                            }
                            dq[qoff + i * d + t] = scale * acc;
                            if (bq) {
                                bq[qoff + i * d + t] = scale * sa;
                                bq[nq + qoff + i * d + t] = scale * Ei * se;
                                bq[2 * nq + qoff + i * d + t] = scale * sf;
                            }
                        }
                        for (int64_t j = 0; j < kend; ++j)
                            for (int64_t t = 0; t < d; ++t) {
                                dkl[j * d + t] += scale * dS[j] * qi[t];
                                dvl[j * d + t] += P[j] * doi[t];
                                if (bkl) {
                                    bkl[j * d + t] += scale * fabs(dS[j]) * fabs(qi[t]);
                                    bkl[N * d + j * d + t] += scale * P[j] * Ei * fabs(qi[t]);
                                    bkl[2 * N * d + j * d + t] += scale * P[j] * F[j] * fabs(qi[t]);
                                }
                                if (bvl) bvl[j * d + t] += P[j] * fabs(doi[t]);
                            }
                    }
#pragma omp critical
                    {
                        for (int64_t x = 0; x < N * d; ++x) {
                            dk[kvoff + x] += dkl[x];
                            dv[kvoff + x] += dvl[x];
                            if (bkl) {
                                bk[kvoff + x] += bkl[x];
                                bk[nkv + kvoff + x] += bkl[N * d + x];
                                bk[2 * nkv + kvoff + x] += bkl[2 * N * d + x];
                            }
                            if (bvl) bv[kvoff + x] += bvl[x];
                        }
                    }
                    free(P);
                    free(dS);
                    free(F);
                    free(o);
                    free(a);
                    free(loc);
                }
            }
        }
    }
    free(Q);
    free(K);
    free(V);
    free(dO);
    return 0;
}

/*
 * Forward on double inputs (no 16-bit decoding), all rows, for the
 * finite-difference pin of the backward: out o [B,Hq,N,d].
 */
int oracle_attention_f64(const double* q, const double* k, const double* v, int64_t B, int64_t Hq,
                         int64_t Hkv, int64_t N, int64_t d, double scale, int causal, double* o) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || N <= 0 || d <= 0 || Hq % Hkv) return -1;
    const int64_t G = Hq / Hkv;
    double* s = (double*)malloc(sizeof(double) * (size_t)N);
    for (int64_t r = 0; r < B * Hq * N; ++r) {
        const int64_t i = r % N, h = (r / N) % Hq, b = r / (N * Hq), hk = h / G;
        const double* qp = q + r * d;
        const double* kp = k + (b * Hkv + hk) * N * d;
        const double* vp = v + (b * Hkv + hk) * N * d;
        const int64_t kend = causal ? (i + 1 < N ? i + 1 : N) : N;
        double m = -INFINITY;
        for (int64_t j = 0; j < kend; ++j) {
            double dot = 0.0;
            for (int64_t t = 0; t < d; ++t) dot += qp[t] * kp[j * d + t];
            s[j] = scale * dot;
            if (s[j] > m) m = s[j];
        }
        double l = 0.0;
        for (int64_t t = 0; t < d; ++t) o[r * d + t] = 0.0;
        for (int64_t j = 0; j < kend; ++j) {
            const double p = exp(s[j] - m);
            l += p;
            for (int64_t t = 0; t < d; ++t) o[r * d + t] += p * vp[j * d + t];
        }
        for (int64_t t = 0; t < d; ++t) o[r * d + t] /= l;
    }
    free(s);
    return 0;
}

/*
 * FP8 (e4m3) inputs with in-kernel scaling: the variant the Character.AI /
 * Colfax article "FlashAttention-3 for Inference: INT8 Quantization and Query
 * Head Packing for MQA/GQA" (Colfax Research author page) names -- quantised
 * Q, K, V consumed directly by an attention kernel that applies their scales
 * itself. The pages give only the article's title and summary, so the form
 * here is the plainest one consistent with it:
 *
 *   inputs   e4m3 codes q, k, v with one fp32 descale per (batch, KV head)
 *            for each tensor (the query heads of a KV head share the Q one);
 *            the represented values are code * descale
 *   method   FlashAttention-2's forward over key tiles of bc keys (the
 *            online softmax of "A Case Study in CUDA Kernel Fusion:
 *            Implementing FlashAttention-2 on NVIDIA Hopper Architecture
 *            using the CUTLASS Library", abstract, and the Ampere series'
 *            algorithm): for tile T = keys [T*bc, (T+1)*bc)
 *              m_T = max(m_{T-1}, max_{j in T} s_j)
 *              p_j = exp(s_j - m_T)                       (j in T)
 *              l_T = exp(m_{T-1} - m_T) l_{T-1} + sum_{j in T} p_j
 *              o_T = exp(m_{T-1} - m_T) o_{T-1} + sum_{j in T} w_j vdeq_j
 *            with the P.V product on FP8 operands: w_j = e4m3(256 p_j) / 256,
 *            P scaled by 2^8 and rounded to e4m3 against the running max of
 *            its tile; l sums the unrounded p_j. o = o_last / l_last,
 *            lse = m_last + ln(l_last).
 *   plain    the definition on the dequantised inputs, the quantity the
 *            method approximates: p_j = exp(s_j - max_j s_j), o = sum p_j
 *            vdeq_j / sum p_j.
 * Where the rounding happens relative to a running max, the rounded weights
 * of a tile depend on the tiling, so the method output depends on bc (the
 * kernel's key tile is 128); with bc >= N it rounds against the final max.
 * Two auxiliary row sums bound the effect of rounding P (any bc):
 *   a_t = sum_j p_j |vdeq_{j,t}| / l,    b_t = sum_j |vdeq_{j,t}| / l
 * with p_j and l of the plain definition.
 */

/* Exact value of an e4m3 code (OCP 8-bit floating point, E4M3: sign, 4-bit
 * exponent with bias 7, 3-bit fraction; exponent 0 encodes subnormals
 * f/8 * 2^-6; S.1111.111 is NaN; there are no infinities). */
static double decode_e4m3(uint8_t c) {
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int f = c & 7;
    double v;
    if (e == 15 && f == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)f, -9);
    else
        v = ldexp((double)(8 + f), e - 10);
    return sign ? -v : v;
}

/* x >= 0 rounded to the nearest e4m3 value, ties to even, saturating at 448:
 * with the binade's spacing u (2^-9 below 2^-6, else 2^(floor(log2 x) - 3)),
 * round x/u to the nearest integer with rint (the default rounding mode,
 * nearest-even), whose parity is the parity of the code. */
static double round_e4m3(double x) {
    if (!(x > 0.0)) return 0.0;
    if (x >= 448.0) return 448.0;
    int ex;
    frexp(x, &ex);                  /* x = f * 2^ex, f in [0.5, 1): floor(log2 x) = ex - 1 */
    int e = ex - 1;
    if (e < -6) e = -6;             /* subnormal range shares the spacing of [2^-6, 2^-5) */
    double u = ldexp(1.0, e - 3);
    double r = rint(x / u) * u;
    return r > 448.0 ? 448.0 : r;
}

void oracle_decode_e4m3(const uint8_t* codes, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = decode_e4m3(codes[i]);
}

void oracle_round_e4m3(const double* x, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = x[i] < 0.0 ? -round_e4m3(-x[i]) : round_e4m3(x[i]);
}

/*
 * q: [B, Hq, Nq, d] e4m3 codes; k, v: [B, Hkv, Nk, d] codes; qd, kd, vd:
 * [B*Hkv] descales. causal: query row i sees keys j < kend(i) =
 * min(Nk, i + 1 + Nk - Nq) (the mask of oracle_attention_ex_rows), else all
 * Nk keys; a row that sees no key gets o = 0, lse = -inf. bc: key tile of the
 * method (>= 1), tiles start at key 0. rows: flat query rows
 * (b*Hq + h)*Nq + i or NULL for all. o_method, o_plain, a_out, b_out:
 * [nrows, d], each may be NULL; lse: [nrows] (the plain definition's).
 */
int oracle_attention_fp8_rows(const uint8_t* q, const uint8_t* k, const uint8_t* v, const double* qd,
                              const double* kd, const double* vd, int64_t B, int64_t Hq, int64_t Hkv,
                              int64_t Nq, int64_t Nk, int64_t d, double scale, int causal, int64_t bc,
                              const int64_t* rows, int64_t nrows, double* o_method, double* o_plain,
                              double* lse_out, double* a_out, double* b_out, int nthreads) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || Nk <= 0 || d <= 0 || Hq % Hkv || bc <= 0) return -1;
    if (!rows && nrows != B * Hq * Nq) return -1;
    const int64_t G = Hq / Hkv;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif

    double tab[256];               /* code -> value, so the loops below decode by lookup */
    for (int c = 0; c < 256; ++c) tab[c] = decode_e4m3((uint8_t)c);

#pragma omp parallel
    {
        double* qrow = (double*)malloc(sizeof(double) * (size_t)d);
        double* s = (double*)malloc(sizeof(double) * (size_t)Nk);
        double* acc = (double*)malloc(sizeof(double) * (size_t)d);
        double* accp = (double*)malloc(sizeof(double) * (size_t)d);
        double* aa = (double*)malloc(sizeof(double) * (size_t)d);
        double* bb = (double*)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < nrows; ++r) {
            const int64_t flat = rows ? rows[r] : r;
            const int64_t i = flat % Nq;
            const int64_t h = (flat / Nq) % Hq;
            const int64_t b = flat / (Nq * Hq);
            const int64_t g = b * Hkv + h / G;      /* the (batch, KV head) group */
            const uint8_t* qp = q + ((b * Hq + h) * Nq + i) * d;
            const uint8_t* kp = k + g * Nk * d;
            const uint8_t* vp = v + g * Nk * d;
            int64_t kend = Nk;                      /* keys j < kend are allowed */
            if (causal && i + 1 + Nk - Nq < kend) kend = i + 1 + Nk - Nq;
            if (kend <= 0) {                        /* no allowed key */
                for (int64_t t = 0; t < d; ++t) {
                    if (o_method) o_method[r * d + t] = 0.0;
                    if (o_plain) o_plain[r * d + t] = 0.0;
                    if (a_out) a_out[r * d + t] = 0.0;
                    if (b_out) b_out[r * d + t] = 0.0;
                }
                lse_out[r] = -INFINITY;
                continue;
            }

            /* dequantised inputs: code * descale */
            for (int64_t t = 0; t < d; ++t) qrow[t] = tab[qp[t]] * qd[g];
            double m = -INFINITY;
            for (int64_t j = 0; j < kend; ++j) {
                double dot = 0.0;
                for (int64_t t = 0; t < d; ++t) dot += qrow[t] * (tab[kp[j * d + t]] * kd[g]);
                s[j] = scale * dot;
                if (s[j] > m) m = s[j];
            }
            /* plain definition and the two bounding sums */
            double l = 0.0;
            for (int64_t t = 0; t < d; ++t) accp[t] = aa[t] = bb[t] = 0.0;
            for (int64_t j = 0; j < kend; ++j) {
                const double pj = exp(s[j] - m);
                l += pj;
                for (int64_t t = 0; t < d; ++t) {
                    const double vv = tab[vp[j * d + t]] * vd[g];
                    accp[t] += pj * vv;
                    aa[t] += pj * fabs(vv);
                    bb[t] += fabs(vv);
                }
            }
            /* the method: online softmax over key tiles, P rounded per tile */
            double mt = -INFINITY, lt = 0.0;
            for (int64_t t = 0; t < d; ++t) acc[t] = 0.0;
            for (int64_t j0 = 0; j0 < kend; j0 += bc) {
                const int64_t j1 = j0 + bc < kend ? j0 + bc : kend;
                double mnew = mt;
                for (int64_t j = j0; j < j1; ++j)
                    if (s[j] > mnew) mnew = s[j];
                const double alpha = mt == -INFINITY ? 0.0 : exp(mt - mnew);
                lt *= alpha;
                for (int64_t t = 0; t < d; ++t) acc[t] *= alpha;
                mt = mnew;
                for (int64_t j = j0; j < j1; ++j) {
                    const double pj = exp(s[j] - mt);
                    lt += pj;
                    const double wj = round_e4m3(256.0 * pj) / 256.0;
                    for (int64_t t = 0; t < d; ++t) acc[t] += wj * (tab[vp[j * d + t]] * vd[g]);
                }
            }
            for (int64_t t = 0; t < d; ++t) {
                if (o_method) o_method[r * d + t] = acc[t] / lt;
                if (o_plain) o_plain[r * d + t] = accp[t] / l;
                if (a_out) a_out[r * d + t] = aa[t] / l;
                if (b_out) b_out[r * d + t] = bb[t] / l;
            }
            lse_out[r] = m + log(l);
        }
        free(qrow);
        free(s);
        free(acc);
        free(accp);
        free(aa);
        free(bb);
    }
    return 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
