/*
 * oracle.c -- plain, slow, fp64 CPU oracle for exact attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call this code:
 * only the tests, the smoke check and the bench's CPU-baseline leg load it.
 * It shares no source, header, table or helper with the CUDA library; the
 * inputs it is given are the raw fp16/bf16 bit patterns that the seeded
 * generators produce, and it decodes them itself.
 *
 * What it computes (definitions, written out with no blocking, fusion or
 * online rescaling):
 *
 *   softmax attention, from "[CUDA 优化实战] fmha sm120 : 超越 torch.sdpa
 *   (flash-attention-2)" section 1 ("flash attention"): O = softmax(scale *
 *   Q K^T) V, with the naive three steps s = q k^T * scale, p = softmax(s),
 *   o = p v.  S and P are materialised, one block of query rows at a time
 *   (every entry of the block is formed explicitly; blocking rows changes no
 *   arithmetic).
 *
 *   causal mask, same page, section 2 ("fmha 实现", the kernel listing's
 *   mask): key j is visible to query i iff j <= i (top-left aligned).
 *
 *   GQA, same page, section 2: query head h reads kv head h / (Hq / Hkv).
 *
 *   per-row log-sum-exp, "CUDA 实现 Flash Decoding" section 2.2: lse = m +
 *   log(l) with natural log, here of the scaled logits: lse_i =
 *   ln sum_j exp(scale * q_i . k_j).  "Tensor Core 迁移计划" (cross-cutting
 *   concerns) fixes the LSE output as fp32 floats; the oracle keeps fp64.
 *
 *   chunked decode, "CUDA 实现 Flash Decoding" section 2.2, Step 1 (per
 *   chunk: S_c, m_c, P_c = exp(S_c - m_c), l_c, O_c = P_c V_c / l_c,
 *   lse_c = m_c + log l_c) and Step 2 (m = max_c, global_lse = m +
 *   log sum_c exp(lse_c - m), w_c = exp(lse_c - global_lse), O = sum_c w_c
 *   O_c).
 *
 *   backward, "Tensor Core 迁移计划" (phase 2: the backward's contractions
 *   dV = P^T dO, dP = dO V^T, dQ and dK from dS): the gradients of O with
 *   respect to Q, K and V by the chain rule through the softmax.
 *
 *   FP8 K/V decode: attention over K = k_scale[h] * e4m3(k8), V likewise,
 *   with the OCP E4M3 format decoded from its definition.
 *
 *   paged K/V decode: key j of sequence b gathered from page
 *   block_table[b][j / page], row j % page, for j < seq_lens[b].
 *
 * Layouts: q, o [B, N, Hq, d]; k, v [B, M, Hkv, d]; lse [B, Hq, N]; paged
 * caches [num_pages, page, Hkv, d]; all contiguous.  dtype 0 = IEEE fp16,
 * 1 = bfloat16.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_ROWS_PER_BLOCK 16

/* ---- exact decoding of the 16-bit input formats ------------------------- */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_fp16_to_double(uint16_t bits) {
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 10) & 0x1f;
    int frac = bits & 0x3ff;
    double mag;
    if (expo == 0) {
        mag = ldexp((double)frac, -24);           /* subnormal: frac * 2^-14 * 2^-10 */
    } else if (expo == 31) {
        mag = frac ? NAN : INFINITY;
    } else {
        mag = ldexp((double)(1024 + frac), expo - 25); /* (1 + frac/1024) * 2^(expo-15) */
    }
    return sign ? -mag : mag;
}

/* bfloat16: the upper half of an IEEE binary32 word. */
double oracle_bf16_to_double(uint16_t bits) {
    uint32_t word = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &word, sizeof f);
    return (double)f;
}

static void decode_array(const uint16_t* src, double* dst, size_t n, int dtype) {
    for (size_t i = 0; i < n; ++i)
        dst[i] = dtype == 0 ? oracle_fp16_to_double(src[i]) : oracle_bf16_to_double(src[i]);
}

/* Copy the (b, head) slice of a [B, S, H, d] tensor into a dense [S][d] fp64 array. */
static void gather_head(const uint16_t* x, int dtype, int b, int head, int S, int H, int d,
                        double* out) {
    for (int s = 0; s < S; ++s) {
        const uint16_t* row = x + (((size_t)b * S + s) * H + head) * (size_t)d;
        decode_array(row, out + (size_t)s * d, (size_t)d, dtype);
    }
}

/* ---- one query row, straight from the definition ------------------------ */

/*
 * Computes O row and LSE for query vector qrow against keys 0..nkeys-1 of the
 * dense head slices K, V.  srow and prow are caller scratch of length >= nkeys
 * (the materialised S and P rows).
 */
static void attend_row(const double* qrow, const double* K, const double* V, int nkeys, int d,
                       double scale, double* srow, double* prow, double* orow, double* lse) {
    /* S row: s_j = scale * q . k_j */
    for (int j = 0; j < nkeys; ++j) {
        const double* kj = K + (size_t)j * d;
        double acc = 0.0;
        for (int t = 0; t < d; ++t) acc += qrow[t] * kj[t];
        srow[j] = scale * acc;
    }
    /* softmax: m = max_j s_j, e_j = exp(s_j - m), P_j = e_j / sum e */
    double m = -INFINITY;
    for (int j = 0; j < nkeys; ++j)
        if (srow[j] > m) m = srow[j];
    double l = 0.0;
    for (int j = 0; j < nkeys; ++j) {
        prow[j] = exp(srow[j] - m);
        l += prow[j];
    }
    for (int j = 0; j < nkeys; ++j) prow[j] /= l;
    /* O row = P V */
    for (int t = 0; t < d; ++t) orow[t] = 0.0;
    for (int j = 0; j < nkeys; ++j) {
        const double* vj = V + (size_t)j * d;
        for (int t = 0; t < d; ++t) orow[t] += prow[j] * vj[t];
    }
    *lse = m + log(l);
}

static int check_shape(int B, int Hq, int Hkv, int N, int M, int d) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || N <= 0 || M <= 0 || d <= 0) return -1;
    if (Hq % Hkv != 0) return -1;
    return 0;
}

static int keys_visible(int i, int M, int causal) {
    if (!causal) return M;
    return i + 1 < M ? i + 1 : M;
}

/* ---- full forward -------------------------------------------------------- */

/*
 * O [B,N,Hq,d] and LSE [B,Hq,N] (fp64) of exact attention.  probs, when not
 * NULL, receives the full P matrix [B,Hq,N,M] (masked entries 0); only for
 * tiny problems.  Returns 0, or -1 on a bad shape / allocation failure.
 */
int oracle_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v, int dtype,
                     int B, int Hq, int Hkv, int N, int M, int d, int causal, double scale,
                     double* o, double* lse, double* probs) {
    if (check_shape(B, Hq, Hkv, N, M, d)) return -1;
    const int g = Hq / Hkv;
    double* K = malloc(sizeof(double) * (size_t)M * d);
    double* V = malloc(sizeof(double) * (size_t)M * d);
    if (!K || !V) { free(K); free(V); return -1; }
    const int nblocks = (N + ORACLE_ROWS_PER_BLOCK - 1) / ORACLE_ROWS_PER_BLOCK;
    int failed = 0;
    for (int b = 0; b < B; ++b) {
        for (int kh = 0; kh < Hkv; ++kh) {
            gather_head(k, dtype, b, kh, M, Hkv, d, K);
            gather_head(v, dtype, b, kh, M, Hkv, d, V);
            const int ntasks = g * nblocks;
#pragma omp parallel for schedule(dynamic, 1)
            for (int task = 0; task < ntasks; ++task) {
                const int h = kh * g + task / nblocks;   /* GQA: h / g == kh */
                const int i0 = (task % nblocks) * ORACLE_ROWS_PER_BLOCK;
                const int i1 = i0 + ORACLE_ROWS_PER_BLOCK < N ? i0 + ORACLE_ROWS_PER_BLOCK : N;
                /* the materialised S and P blocks for rows i0..i1-1 */
                double* Sblk = malloc(sizeof(double) * (size_t)(i1 - i0) * M);
                double* Pblk = malloc(sizeof(double) * (size_t)(i1 - i0) * M);
                double* qrow = malloc(sizeof(double) * (size_t)d);
                if (!Sblk || !Pblk || !qrow) {
#pragma omp atomic write
                    failed = 1;
                } else {
                    for (int i = i0; i < i1; ++i) {
                        const uint16_t* qsrc = q + (((size_t)b * N + i) * Hq + h) * (size_t)d;
                        decode_array(qsrc, qrow, (size_t)d, dtype);
                        const int nk = keys_visible(i, M, causal);
                        double* srow = Sblk + (size_t)(i - i0) * M;
                        double* prow = Pblk + (size_t)(i - i0) * M;
                        double* orow = o + (((size_t)b * N + i) * Hq + h) * (size_t)d;
                        double l;
                        attend_row(qrow, K, V, nk, d, scale, srow, prow, orow, &l);
                        lse[((size_t)b * Hq + h) * N + i] = l;
                        if (probs) {
                            double* pdst = probs + (((size_t)b * Hq + h) * N + i) * (size_t)M;
                            for (int j = 0; j < M; ++j) pdst[j] = j < nk ? prow[j] : 0.0;
                        }
                    }
                }
                free(Sblk);
                free(Pblk);
                free(qrow);
            }
        }
    }
    free(K);
    free(V);
    return failed ? -1 : 0;
}

/*
 * The same definition evaluated for a list of query rows only (for sampled
 * checks at sizes where the full oracle would take too long).  rows holds
 * nrows triples (b, h, i); o_rows [nrows, d] and lse_rows [nrows] fp64.
 */
int oracle_attention_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v, int dtype,
                          int B, int Hq, int Hkv, int N, int M, int d, int causal, double scale,
                          const int64_t* rows, int nrows, double* o_rows, double* lse_rows) {
    if (check_shape(B, Hq, Hkv, N, M, d) || nrows < 0) return -1;
    for (int r = 0; r < nrows; ++r) {
        int64_t b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
        if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= N) return -1;
    }
    const int g = Hq / Hkv;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < nrows; ++r) {
        const int b = (int)rows[3 * r], h = (int)rows[3 * r + 1], i = (int)rows[3 * r + 2];
        const int kh = h / g;
        const int nk = keys_visible(i, M, causal);
        double* K = malloc(sizeof(double) * (size_t)nk * d);
        double* V = malloc(sizeof(double) * (size_t)nk * d);
        double* srow = malloc(sizeof(double) * (size_t)nk);
        double* prow = malloc(sizeof(double) * (size_t)nk);
        double* qrow = malloc(sizeof(double) * (size_t)d);
        if (!K || !V || !srow || !prow || !qrow) {
#pragma omp atomic write
            failed = 1;
        } else {
            /* the first nk keys of kv head kh in batch b */
            for (int j = 0; j < nk; ++j) {
                decode_array(k + (((size_t)b * M + j) * Hkv + kh) * (size_t)d, K + (size_t)j * d,
                             (size_t)d, dtype);
                decode_array(v + (((size_t)b * M + j) * Hkv + kh) * (size_t)d, V + (size_t)j * d,
                             (size_t)d, dtype);
            }
            decode_array(q + (((size_t)b * N + i) * Hq + h) * (size_t)d, qrow, (size_t)d, dtype);
            attend_row(qrow, K, V, nk, d, scale, srow, prow, o_rows + (size_t)r * d, &lse_rows[r]);
        }
        free(K);
        free(V);
        free(srow);
        free(prow);
        free(qrow);
    }
    return failed ? -1 : 0;
}

/* ---- split-KV decode: chunk partials and their LSE-weighted merge --------- */

/*
 * q [B,1,Hq,d], k/v [B,M,Hkv,d].  For every (b, h) the M keys are cut into
 * nc = ceil(M / chunk) chunks [c*chunk, min(M, (c+1)*chunk)).  Writes
 * o_part [B,Hq,nc,d], lse_part [B,Hq,nc] (Step 1) and the merged o [B,1,Hq,d],
 * lse [B,Hq] (Step 2).  Any output pointer may be NULL.
 */
int oracle_decode_chunked(const uint16_t* q, const uint16_t* k, const uint16_t* v, int dtype,
                          int B, int Hq, int Hkv, int M, int d, int chunk, double scale,
                          double* o_part, double* lse_part, double* o, double* lse) {
    if (check_shape(B, Hq, Hkv, 1, M, d) || chunk <= 0) return -1;
    const int g = Hq / Hkv;
    const int nc = (M + chunk - 1) / chunk;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < B * Hq; ++bh) {
        const int b = bh / Hq, h = bh % Hq, kh = h / g;
        double* K = malloc(sizeof(double) * (size_t)M * d);
        double* V = malloc(sizeof(double) * (size_t)M * d);
        double* qrow = malloc(sizeof(double) * (size_t)d);
        double* srow = malloc(sizeof(double) * (size_t)chunk);
        double* prow = malloc(sizeof(double) * (size_t)chunk);
        double* Oc = malloc(sizeof(double) * (size_t)nc * d);
        double* Lc = malloc(sizeof(double) * (size_t)nc);
        if (!K || !V || !qrow || !srow || !prow || !Oc || !Lc) {
#pragma omp atomic write
            failed = 1;
        } else {
            for (int j = 0; j < M; ++j) {
                decode_array(k + (((size_t)b * M + j) * Hkv + kh) * (size_t)d, K + (size_t)j * d,
                             (size_t)d, dtype);
                decode_array(v + (((size_t)b * M + j) * Hkv + kh) * (size_t)d, V + (size_t)j * d,
                             (size_t)d, dtype);
            }
            decode_array(q + ((size_t)b * Hq + h) * (size_t)d, qrow, (size_t)d, dtype);
            /* Step 1: each chunk on its own (its softmax is normalised inside the chunk) */
            for (int c = 0; c < nc; ++c) {
                const int j0 = c * chunk;
                const int len = j0 + chunk < M ? chunk : M - j0;
                attend_row(qrow, K + (size_t)j0 * d, V + (size_t)j0 * d, len, d, scale, srow, prow,
                           Oc + (size_t)c * d, &Lc[c]);
            }
            /* Step 2: global_lse = m + log sum_c exp(lse_c - m); w_c = exp(lse_c - global_lse) */
            double m = -INFINITY;
            for (int c = 0; c < nc; ++c)
                if (Lc[c] > m) m = Lc[c];
            double L = 0.0;
            for (int c = 0; c < nc; ++c) L += exp(Lc[c] - m);
            const double glse = m + log(L);
            if (o) {
                double* orow = o + ((size_t)b * Hq + h) * (size_t)d;
                for (int t = 0; t < d; ++t) orow[t] = 0.0;
                for (int c = 0; c < nc; ++c) {
                    const double w = exp(Lc[c] - glse);
                    for (int t = 0; t < d; ++t) orow[t] += w * Oc[(size_t)c * d + t];
                }
            }
            if (lse) lse[(size_t)b * Hq + h] = glse;
            if (o_part) memcpy(o_part + (size_t)bh * nc * d, Oc, sizeof(double) * (size_t)nc * d);
            if (lse_part) memcpy(lse_part + (size_t)bh * nc, Lc, sizeof(double) * (size_t)nc);
        }
        free(K);
        free(V);
        free(qrow);
        free(srow);
        free(prow);
        free(Oc);
        free(Lc);
    }
    return failed ? -1 : 0;
}

/* ---- backward: gradients of O with respect to Q, K and V ------------------ */

/*
 * The gradients of the attention above, for an upstream gradient dO [B,N,Hq,d]
 * (the training step after the forward; "Tensor Core 迁移计划", phase 2, names
 * the backward's contractions dV = P^T dO, dP = dO V^T and dQ, dK from dS).
 * With s_ij = scale q_i . k_j over the visible keys and p_ij its softmax, the
 * chain rule through o_i = sum_j p_ij v_j and the softmax Jacobian gives
 *     dV_j  = sum_i p_ij dO_i,
 *     dP_ij = dO_i . v_j,
 *     dS_ij = p_ij (dP_ij - sum_k p_ik dP_ik),
 *     dQ_i  = scale sum_j dS_ij k_j,
 *     dK_j  = scale sum_i dS_ij q_i,
 * with dK and dV of kv head kh summed over the g query heads that read it.
 * Every P row, dP row and dS row is formed explicitly (no D_i = dO_i . O_i
 * shortcut, no online rescaling).  dq [B,N,Hq,d], dk/dv [B,M,Hkv,d], fp64.
 * Returns 0, or -1 on a bad shape or an allocation failure.
 */
int oracle_attention_backward(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                              const uint16_t* dout, int dtype, int B, int Hq, int Hkv, int N,
                              int M, int d, int causal, double scale, double* dq, double* dk,
                              double* dv) {
    if (check_shape(B, Hq, Hkv, N, M, d)) return -1;
    const int g = Hq / Hkv;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int task = 0; task < B * Hkv; ++task) {
        const int b = task / Hkv, kh = task % Hkv;
        double* K = malloc(sizeof(double) * (size_t)M * d);
        double* V = malloc(sizeof(double) * (size_t)M * d);
        double* dK = calloc((size_t)M * d, sizeof(double));
        double* dV = calloc((size_t)M * d, sizeof(double));
        double* qrow = malloc(sizeof(double) * (size_t)d);
        double* dorow = malloc(sizeof(double) * (size_t)d);
        double* P = malloc(sizeof(double) * (size_t)M);
        double* dP = malloc(sizeof(double) * (size_t)M);
        double* dS = malloc(sizeof(double) * (size_t)M);
        if (!K || !V || !dK || !dV || !qrow || !dorow || !P || !dP || !dS) {
#pragma omp atomic write
            failed = 1;
        } else {
            gather_head(k, dtype, b, kh, M, Hkv, d, K);
            gather_head(v, dtype, b, kh, M, Hkv, d, V);
            for (int h = kh * g; h < (kh + 1) * g; ++h) {
                for (int i = 0; i < N; ++i) {
                    const size_t row = (((size_t)b * N + i) * Hq + h) * (size_t)d;
                    decode_array(q + row, qrow, (size_t)d, dtype);
                    decode_array(dout + row, dorow, (size_t)d, dtype);
                    const int nk = keys_visible(i, M, causal);
                    /* P row: softmax of s_ij = scale q_i . k_j */
                    double m = -INFINITY;
                    for (int j = 0; j < nk; ++j) {
                        double acc = 0.0;
                        for (int t = 0; t < d; ++t) acc += qrow[t] * K[(size_t)j * d + t];
                        P[j] = scale * acc;
                        if (P[j] > m) m = P[j];
                    }
                    double l = 0.0;
                    for (int j = 0; j < nk; ++j) {
                        P[j] = exp(P[j] - m);
                        l += P[j];
                    }
                    for (int j = 0; j < nk; ++j) P[j] /= l;
                    /* dP row and the softmax Jacobian */
                    double pdp = 0.0;
                    for (int j = 0; j < nk; ++j) {
                        double acc = 0.0;
                        for (int t = 0; t < d; ++t) acc += dorow[t] * V[(size_t)j * d + t];
                        dP[j] = acc;
                        pdp += P[j] * dP[j];
                    }
                    for (int j = 0; j < nk; ++j) dS[j] = P[j] * (dP[j] - pdp);
                    /* dQ_i, and this row's terms of dK and dV */
                    double* dqrow = dq + row;
                    for (int t = 0; t < d; ++t) dqrow[t] = 0.0;
                    for (int j = 0; j < nk; ++j) {
                        for (int t = 0; t < d; ++t) {
                            dqrow[t] += scale * dS[j] * K[(size_t)j * d + t];
                            dK[(size_t)j * d + t] += scale * dS[j] * qrow[t];
                            dV[(size_t)j * d + t] += P[j] * dorow[t];
                        }
                    }
                }
            }
            for (int j = 0; j < M; ++j) {
                const size_t dst = (((size_t)b * M + j) * Hkv + kh) * (size_t)d;
                memcpy(dk + dst, dK + (size_t)j * d, sizeof(double) * (size_t)d);
                memcpy(dv + dst, dV + (size_t)j * d, sizeof(double) * (size_t)d);
            }
        }
        free(K);
        free(V);
        free(dK);
        free(dV);
        free(qrow);
        free(dorow);
        free(P);
        free(dP);
        free(dS);
    }
    return failed ? -1 : 0;
}

/*
 * dQ of the backward above for selected query rows only (sampled checks at
 * sizes where the full backward would take too long): dQ_i depends on row i
 * alone -- its P row, dP row and dS row -- so each listed row is the same
 * definition as in oracle_attention_backward.  rows holds nrows triples
 * (b, h, i); dq_rows [nrows, d] fp64.
 */
int oracle_attention_backward_dq_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                      const uint16_t* dout, int dtype, int B, int Hq, int Hkv,
                                      int N, int M, int d, int causal, double scale,
                                      const int64_t* rows, int nrows, double* dq_rows) {
    if (check_shape(B, Hq, Hkv, N, M, d) || nrows < 0) return -1;
    const int g = Hq / Hkv;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int rI = 0; rI < nrows; ++rI) {
        const int64_t b = rows[3 * rI], h = rows[3 * rI + 1], i = rows[3 * rI + 2];
        if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= N) {
#pragma omp atomic write
            failed = 1;
            continue;
        }
        const int kh = (int)h / g;
        const int nk = keys_visible((int)i, M, causal);
        double* qrow = malloc(sizeof(double) * (size_t)d);
        double* dorow = malloc(sizeof(double) * (size_t)d);
        double* krow = malloc(sizeof(double) * (size_t)d);
        double* vrow = malloc(sizeof(double) * (size_t)d);
        double* P = malloc(sizeof(double) * (size_t)nk);
        double* dP = malloc(sizeof(double) * (size_t)nk);
        if (!qrow || !dorow || !krow || !vrow || !P || !dP) {
#pragma omp atomic write
            failed = 1;
        } else {
            const size_t row = (((size_t)b * N + i) * Hq + h) * (size_t)d;
            decode_array(q + row, qrow, (size_t)d, dtype);
            decode_array(dout + row, dorow, (size_t)d, dtype);
            double m = -INFINITY;
            for (int j = 0; j < nk; ++j) {
                decode_array(k + (((size_t)b * M + j) * Hkv + kh) * (size_t)d, krow, (size_t)d, dtype);
                decode_array(v + (((size_t)b * M + j) * Hkv + kh) * (size_t)d, vrow, (size_t)d, dtype);
                double s = 0.0, dp = 0.0;
                for (int t = 0; t < d; ++t) {
                    s += qrow[t] * krow[t];
                    dp += dorow[t] * vrow[t];
                }
                P[j] = scale * s;
                dP[j] = dp;
                if (P[j] > m) m = P[j];
            }
            double l = 0.0;
            for (int j = 0; j < nk; ++j) {
                P[j] = exp(P[j] - m);
                l += P[j];
            }
            double pdp = 0.0;
            for (int j = 0; j < nk; ++j) {
                P[j] /= l;
                pdp += P[j] * dP[j];
            }
            double* out = dq_rows + (size_t)rI * d;
            for (int t = 0; t < d; ++t) out[t] = 0.0;
            for (int j = 0; j < nk; ++j) {
                const double ds = P[j] * (dP[j] - pdp);
                decode_array(k + (((size_t)b * M + j) * Hkv + kh) * (size_t)d, krow, (size_t)d, dtype);
                for (int t = 0; t < d; ++t) out[t] += scale * ds * krow[t];
            }
        }
        free(qrow);
        free(dorow);
        free(krow);
        free(vrow);
        free(P);
        free(dP);
    }
    return failed ? -1 : 0;
}

/* ---- FP8 (e4m3) K/V --------------------------------------------------------- */

/*
 * OCP 8-bit floating point E4M3 (the format the FP8 KV-cache quantisation of
 * the fmha sm120 page's closing "TODO" section and lever 1 of the Flash
 * Decoding page's section 8 store): 1 sign bit, 4 exponent bits (bias 7),
 * 3 mantissa bits; exponent 0 is subnormal (m/8 * 2^-6); there are no
 * infinities, and exponent 15 with mantissa 7 is NaN (so the largest finite
 * value is 1.75 * 2^8 = 448).
 */
double oracle_e4m3_to_double(uint8_t bits) {
    const int sign = (bits >> 7) & 1;
    const int expo = (bits >> 3) & 0xf;
    const int mant = bits & 0x7;
    double mag;
    if (expo == 0xf && mant == 0x7)
        mag = NAN;
    else if (expo == 0)
        mag = ldexp((double)mant, -9);            /* mant/8 * 2^(1-7) */
    else
        mag = ldexp((double)(8 + mant), expo - 10); /* (1 + mant/8) * 2^(expo-7) */
    return sign ? -mag : mag;
}

/*
 * Decode against an e4m3 K/V cache: exact attention of each query row
 * q [B,1,Hq,d] (16-bit dtype) over the dequantised cache
 *     K[b][j][h] = k_scale[h] * e4m3(k8[b][j][h]),  V likewise with v_scale,
 * k8/v8 [B,M,Hkv,d] bytes, scales [Hkv].  o [B,Hq,d], lse [B,Hq] (natural
 * log); either may be NULL.  The split into chunks and their merge reproduce
 * this result exactly up to rounding order, so the definition is the oracle.
 */
int oracle_decode_fp8(const uint16_t* q, const uint8_t* k8, const uint8_t* v8,
                      const float* k_scale, const float* v_scale, int dtype, int B, int Hq,
                      int Hkv, int M, int d, double scale, double* o, double* lse) {
    if (check_shape(B, Hq, Hkv, 1, M, d)) return -1;
    const int g = Hq / Hkv;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < B * Hq; ++bh) {
        const int b = bh / Hq, h = bh % Hq, kh = h / g;
        double* K = malloc(sizeof(double) * (size_t)M * d);
        double* V = malloc(sizeof(double) * (size_t)M * d);
        double* qrow = malloc(sizeof(double) * (size_t)d);
        double* srow = malloc(sizeof(double) * (size_t)M);
        double* prow = malloc(sizeof(double) * (size_t)M);
        double* orow = malloc(sizeof(double) * (size_t)d);
        if (!K || !V || !qrow || !srow || !prow || !orow) {
#pragma omp atomic write
            failed = 1;
        } else {
            const double ks = (double)k_scale[kh], vs = (double)v_scale[kh];
            for (int j = 0; j < M; ++j) {
                const size_t src = (((size_t)b * M + j) * Hkv + kh) * (size_t)d;
                for (int t = 0; t < d; ++t) {
                    K[(size_t)j * d + t] = ks * oracle_e4m3_to_double(k8[src + t]);
                    V[(size_t)j * d + t] = vs * oracle_e4m3_to_double(v8[src + t]);
                }
            }
            decode_array(q + ((size_t)b * Hq + h) * (size_t)d, qrow, (size_t)d, dtype);
            double l;
            attend_row(qrow, K, V, M, d, scale, srow, prow, orow, &l);
            if (o) memcpy(o + (size_t)bh * d, orow, sizeof(double) * (size_t)d);
            if (lse) lse[bh] = l;
        }
        free(K);
        free(V);
        free(qrow);
        free(srow);
        free(prow);
        free(orow);
    }
    return failed ? -1 : 0;
}

/* ---- paged K/V cache ------------------------------------------------------- */

/*
 * Decode against a paged K/V cache (the "attention with kv cache block" item
 * of the fmha sm120 page's closing "TODO" section): key j of sequence b is row
 * j % page of page block_table[b * max_pages + j / page] of the caches
 * kc/vc [num_pages, page, Hkv, d]; sequence b has L_b = min(seq_lens[b], M)
 * keys.  Gathers those rows, then takes the definition as above.  L_b <= 0
 * gives o = 0 and lse = -inf (an empty softmax).  Returns -1 on a bad shape,
 * an allocation failure or a block-table entry outside [0, num_pages) for a
 * key below L_b.
 */
int oracle_decode_paged(const uint16_t* q, const uint16_t* kc, const uint16_t* vc,
                        const int32_t* block_table, const int32_t* seq_lens, int dtype, int B,
                        int Hq, int Hkv, int M, int num_pages, int page, int max_pages, int d,
                        double scale, double* o, double* lse) {
    if (check_shape(B, Hq, Hkv, 1, M, d) || num_pages <= 0 || page <= 0 || max_pages <= 0)
        return -1;
    if ((long long)max_pages * page < M) return -1;
    const int g = Hq / Hkv;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < B * Hq; ++bh) {
        const int b = bh / Hq, h = bh % Hq, kh = h / g;
        const int L = seq_lens[b] < M ? seq_lens[b] : M;
        const int n = L > 0 ? L : 1;
        double* K = malloc(sizeof(double) * (size_t)n * d);
        double* V = malloc(sizeof(double) * (size_t)n * d);
        double* qrow = malloc(sizeof(double) * (size_t)d);
        double* srow = malloc(sizeof(double) * (size_t)n);
        double* prow = malloc(sizeof(double) * (size_t)n);
        double* orow = malloc(sizeof(double) * (size_t)d);
        int bad = !K || !V || !qrow || !srow || !prow || !orow;
        for (int j = 0; j < L && !bad; ++j) {
            const int pg = block_table[(size_t)b * max_pages + j / page];
            if (pg < 0 || pg >= num_pages) {
                bad = 1;
                break;
            }
            const size_t src = (((size_t)pg * page + j % page) * Hkv + kh) * (size_t)d;
            decode_array(kc + src, K + (size_t)j * d, (size_t)d, dtype);
            decode_array(vc + src, V + (size_t)j * d, (size_t)d, dtype);
        }
        if (bad) {
#pragma omp atomic write
            failed = 1;
        } else {
            double l = -INFINITY;
            if (L > 0) {
                decode_array(q + ((size_t)b * Hq + h) * (size_t)d, qrow, (size_t)d, dtype);
                attend_row(qrow, K, V, L, d, scale, srow, prow, orow, &l);
            } else {
                for (int t = 0; t < d; ++t) orow[t] = 0.0;
            }
            if (o) memcpy(o + (size_t)bh * d, orow, sizeof(double) * (size_t)d);
            if (lse) lse[bh] = l;
        }
        free(K);
        free(V);
        free(qrow);
        free(srow);
        free(prow);
        free(orow);
    }
    return failed ? -1 : 0;
}

/* Number of threads the oracle's parallel regions use (1 without OpenMP). */
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
