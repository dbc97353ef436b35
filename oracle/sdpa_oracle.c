/*
 * sdpa_oracle.c -- plain fp64 CPU reference for the scaled dot-product
 * attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check
 * and the benchmark's CPU-baseline / reference legs load this library.  It
 * shares no code, header, table or constant with the CUDA kernels, and the
 * product path never calls it.
 *
 * What it computes.  Codelab "Attention on GPU (cuDNN and TransformerEngine)",
 * section 1 ("How attention works"):
 *
 *     Attention(Q, K, V) = softmax(Q K^T / sqrt(d_k)) V
 *
 * in the four steps that section lists -- score, scale + softmax, attend,
 * output shaped like Q -- and in the order section 4 ("Implement attention
 * from scratch", the naive_attention cell) performs them: every score of a
 * query row is formed, the row goes through a max-subtracted softmax, and the
 * weights multiply V.  The scale is an argument (section 4 uses
 * 1/sqrt(head_dim)).  Arrays use the (B, T, N, H) layout of section 3
 * ("Create Q, K and V test arrays"): Q and O are [B][Sq][Hq][D], K and V are
 * [B][Skv][Hkv][D], D contiguous.
 *
 * Causal masking (section 7, "Add causal masking"): the mask is the lower
 * triangle of the Sq x Skv score matrix, so query row i sees keys 0..i; the
 * first position sees only itself.  For Sq != Skv the pages say nothing; this
 * oracle keeps the literal lower triangle (top-left aligned), so row i sees
 * keys 0..min(i, Skv-1) and no row is ever empty.
 *
 * Grouped heads (section 9, "Compare MHA, GQA and MQA"): with Hkv < Hq each
 * KV head serves G = Hq / Hkv consecutive query heads, i.e. query head hq
 * reads KV head hq / G (the same grouping as repeating every KV head G times
 * in place).
 *
 * Element types: the inputs are decoded here, from each format's definition,
 * to exact doubles: bfloat16, IEEE binary16, OCP FP8 E4M3 (times a per-tensor
 * descale factor, section 10 "FP8": E4M3 for the forward pass), binary32 and
 * binary64.  All arithmetic after decoding is binary64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum {
    ORACLE_BF16 = 0,
    ORACLE_FP16 = 1,
    ORACLE_E4M3 = 2,
    ORACLE_F32 = 3,
    ORACLE_F64 = 4
};

/* ---- element decoders (from the format definitions) ---------------------- */

/* bfloat16: the upper 16 bits of an IEEE binary32. */
static double decode_bf16(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double decode_fp16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* zero / subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);     /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* OCP FP8 E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits; no
 * infinities, S.1111.111 is NaN, largest finite magnitude 448. */
static double decode_e4m3(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xf;
    int f = b & 0x7;
    double v;
    if (e == 15 && f == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)f, -9);                  /* subnormal: f/8 * 2^-6 */
    else
        v = ldexp((double)(8 + f), e - 10);        /* (1 + f/8) * 2^(e-7) */
    return sign ? -v : v;
}

static double load_elem(const void *base, long idx, int dtype, double descale)
{
    switch (dtype) {
    case ORACLE_BF16: return decode_bf16(((const uint16_t *)base)[idx]);
    case ORACLE_FP16: return decode_fp16(((const uint16_t *)base)[idx]);
    case ORACLE_E4M3: return decode_e4m3(((const uint8_t *)base)[idx]) * descale;
    case ORACLE_F32:  return (double)((const float *)base)[idx];
    default:          return ((const double *)base)[idx];
    }
}

double oracle_decode(const void *base, long idx, int dtype, double descale)
{
    return load_elem(base, idx, dtype, descale);
}

/* ---- one query row --------------------------------------------------------- */

typedef struct {
    const void *Q, *K, *V;
    int dtype;
    double dq, dk, dv;               /* per-tensor descales (1 unless E4M3) */
    long B, Hq, Hkv, Sq, Skv, D;
    double scale;
    int causal;
} problem_t;

/* Flat index of element (b, s, h, d) of a [B][S][H][D] array. */
static long bshd(long b, long s, long h, long d, long S, long H, long D)
{
    return ((b * S + s) * H + h) * D + d;
}

/*
 * Output row (b, i, hq):  scores s_j = scale * sum_d Q[b,i,hq,d] K[b,j,g,d]
 * for the visible keys j, weights w_j = exp(s_j - max s) / sum exp(s - max s),
 * out = sum_j w_j V[b,j,g,:].  Masked keys get weight 0.  `scores` is scratch
 * of Skv doubles; `w_out` (optional) receives all Skv weights; `lse_out`
 * (optional) receives log(sum_j exp(s_j)) over the visible keys, the log of
 * the softmax denominator, formed as max s + log(sum exp(s - max s)).
 */
static void attend_row(const problem_t *p, long b, long hq, long i,
                       double *scores, double *out, double *w_out, double *lse_out)
{
    const long G = p->Hq / p->Hkv;          /* query heads per KV head */
    const long g = hq / G;                  /* KV head read by query head hq */
    long n_vis = p->Skv;
    if (p->causal && i + 1 < n_vis)
        n_vis = i + 1;                      /* lower triangle: keys 0..i */

    /* score */
    for (long j = 0; j < n_vis; ++j) {
        double acc = 0.0;
        for (long d = 0; d < p->D; ++d) {
            double q = load_elem(p->Q, bshd(b, i, hq, d, p->Sq, p->Hq, p->D), p->dtype, p->dq);
            double k = load_elem(p->K, bshd(b, j, g, d, p->Skv, p->Hkv, p->D), p->dtype, p->dk);
            acc += q * k;
        }
        scores[j] = acc * p->scale;
    }

    /* scale + softmax (max-subtracted) */
    double m = -INFINITY;
    for (long j = 0; j < n_vis; ++j)
        if (scores[j] > m)
            m = scores[j];
    double denom = 0.0;
    for (long j = 0; j < n_vis; ++j) {
        scores[j] = exp(scores[j] - m);
        denom += scores[j];
    }
    if (lse_out)
        *lse_out = m + log(denom);
    for (long j = 0; j < n_vis; ++j)
        scores[j] /= denom;

    if (w_out) {
        for (long j = 0; j < p->Skv; ++j)
            w_out[j] = j < n_vis ? scores[j] : 0.0;
    }

    /* attend */
    for (long d = 0; d < p->D; ++d) {
        double acc = 0.0;
        for (long j = 0; j < n_vis; ++j)
            acc += scores[j] * load_elem(p->V, bshd(b, j, g, d, p->Skv, p->Hkv, p->D), p->dtype, p->dv);
        out[d] = acc;
    }
}

static int valid_problem(const problem_t *p)
{
    if (!p->Q || !p->K || !p->V) return 0;
    if (p->B < 1 || p->Hq < 1 || p->Hkv < 1 || p->Sq < 1 || p->Skv < 1 || p->D < 1) return 0;
    if (p->Hq % p->Hkv != 0) return 0;
    if (p->dtype < ORACLE_BF16 || p->dtype > ORACLE_F64) return 0;
    return 1;
}

static int resolve_threads(int nthreads)
{
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/*
 * Compute the output rows listed in `rows` (flat indices r = (b*Sq + i)*Hq + hq
 * into the [B][Sq][Hq] row space of O); row k of `out` (D doubles) receives
 * row rows[k].  If `weights` is non-NULL it receives nrows x Skv weights, if
 * `lse` is non-NULL it receives the nrows log-sum-exp values.  Returns the
 * number of threads used, or -1 on an invalid argument.
 */
int oracle_sdpa_rows(const void *Q, const void *K, const void *V, int dtype,
                     double descale_q, double descale_k, double descale_v,
                     long B, long Hq, long Hkv, long Sq, long Skv, long D,
                     double scale, int causal, const long *rows, long nrows,
                     double *out, double *weights, double *lse, int nthreads)
{
    problem_t p = {Q, K, V, dtype, descale_q, descale_k, descale_v,
                   B, Hq, Hkv, Sq, Skv, D, scale, causal};
    if (!valid_problem(&p) || !rows || !out || nrows < 0)
        return -1;
    for (long k = 0; k < nrows; ++k)
        if (rows[k] < 0 || rows[k] >= B * Sq * Hq)
            return -1;
    int nt = resolve_threads(nthreads);
    int failed = 0;
#pragma omp parallel num_threads(nt)
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)Skv);
        if (!scores) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 8)
        for (long k = 0; k < nrows; ++k) {
            if (!scores)
                continue;
            long r = rows[k];
            long hq = r % Hq;
            long i = (r / Hq) % Sq;
            long b = r / (Hq * Sq);
            attend_row(&p, b, hq, i, scores, out + k * D,
                       weights ? weights + k * Skv : NULL, lse ? lse + k : NULL);
        }
        free(scores);
    }
    return failed ? -1 : nt;
}

/*
 * Whole forward pass: out is [B][Sq][Hq][D] doubles; `lse` (optional) is
 * [B][Hq][Sq] doubles.  Returns the number of threads used, or -1 on an
 * invalid argument.
 */
int oracle_sdpa_fwd(const void *Q, const void *K, const void *V, int dtype,
                    double descale_q, double descale_k, double descale_v,
                    long B, long Hq, long Hkv, long Sq, long Skv, long D,
                    double scale, int causal, double *out, double *lse, int nthreads)
{
    problem_t p = {Q, K, V, dtype, descale_q, descale_k, descale_v,
                   B, Hq, Hkv, Sq, Skv, D, scale, causal};
    if (!valid_problem(&p) || !out)
        return -1;
    const long nrows = B * Sq * Hq;
    int nt = resolve_threads(nthreads);
    int failed = 0;
#pragma omp parallel num_threads(nt)
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)Skv);
        if (!scores) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 8)
        for (long r = 0; r < nrows; ++r) {
            if (!scores)
                continue;
            long hq = r % Hq;
            long i = (r / Hq) % Sq;
            long b = r / (Hq * Sq);
            attend_row(&p, b, hq, i, scores, out + r * D, NULL,
                       lse ? lse + (b * Hq + hq) * Sq + i : NULL);
        }
        free(scores);
    }
    return failed ? -1 : nt;
}

/*
 * Backward pass of the same attention, for an upstream gradient dO (shaped
 * like O, same element type as Q): with the scores s_ij = scale q_i . k_j,
 * the softmax P_i. over the visible keys, O_i = sum_j P_ij v_j and the loss
 * sum_i dO_i . O_i, the chain rule through section 1's three steps gives
 *     dV_j  = sum_i P_ij dO_i
 *     dP_ij = dO_i . v_j
 *     dS_ij = P_ij (dP_ij - sum_l P_il dP_il)       (softmax Jacobian)
 *     dQ_i  = scale sum_j dS_ij k_j
 *     dK_j  = scale sum_i dS_ij q_i
 * Masked keys have P_ij = 0.  With grouped heads each KV head sums the
 * contributions of its G query heads.  dQ is [B][Sq][Hq][D], dK and dV are
 * [B][Skv][Hkv][D], all doubles.  Parallel over (b, KV head), so no two
 * threads add into the same dK / dV row.  Returns the number of threads
 * used, or -1 on an invalid argument.
 */
int oracle_sdpa_bwd(const void *Q, const void *K, const void *V, const void *dO, int dtype,
                    long B, long Hq, long Hkv, long Sq, long Skv, long D,
                    double scale, int causal, double *dQ, double *dK, double *dV, int nthreads)
{
    problem_t p = {Q, K, V, dtype, 1.0, 1.0, 1.0, B, Hq, Hkv, Sq, Skv, D, scale, causal};
    if (!valid_problem(&p) || !dO || !dQ || !dK || !dV || dtype == ORACLE_E4M3)
        return -1;
    const long G = Hq / Hkv;
    int nt = resolve_threads(nthreads);
    int failed = 0;
    memset(dK, 0, sizeof(double) * (size_t)(B * Skv * Hkv * D));
    memset(dV, 0, sizeof(double) * (size_t)(B * Skv * Hkv * D));
#pragma omp parallel num_threads(nt)
    {
        double *P = (double *)malloc(sizeof(double) * (size_t)Skv);
        double *dP = (double *)malloc(sizeof(double) * (size_t)Skv);
        if (!P || !dP) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (long bg = 0; bg < B * Hkv; ++bg) {
            if (!P || !dP)
                continue;
            const long b = bg / Hkv, g = bg % Hkv;
            for (long hq = g * G; hq < (g + 1) * G; ++hq) {
                for (long i = 0; i < Sq; ++i) {
                    /* keys 0..i under the causal mask (lower triangle) */
                    const long n_vis = (causal && i + 1 < Skv) ? i + 1 : Skv;
                    /* forward: softmax of the visible scores */
                    double m = -INFINITY;
                    for (long j = 0; j < n_vis; ++j) {
                        double acc = 0.0;
                        for (long d = 0; d < D; ++d)
                            acc += load_elem(Q, bshd(b, i, hq, d, Sq, Hq, D), dtype, 1.0) *
                                   load_elem(K, bshd(b, j, g, d, Skv, Hkv, D), dtype, 1.0);
                        P[j] = acc * scale;
                        if (P[j] > m)
                            m = P[j];
                    }
                    double denom = 0.0;
                    for (long j = 0; j < n_vis; ++j) {
                        P[j] = exp(P[j] - m);
                        denom += P[j];
                    }
                    for (long j = 0; j < n_vis; ++j)
                        P[j] /= denom;
                    /* dP_ij = dO_i . v_j and its P-weighted mean */
                    double mean = 0.0;
                    for (long j = 0; j < n_vis; ++j) {
                        double acc = 0.0;
                        for (long d = 0; d < D; ++d)
                            acc += load_elem(dO, bshd(b, i, hq, d, Sq, Hq, D), dtype, 1.0) *
                                   load_elem(V, bshd(b, j, g, d, Skv, Hkv, D), dtype, 1.0);
                        dP[j] = acc;
                        mean += P[j] * acc;
                    }
                    double *dq = dQ + bshd(b, i, hq, 0, Sq, Hq, D);
                    for (long d = 0; d < D; ++d)
                        dq[d] = 0.0;
                    for (long j = 0; j < n_vis; ++j) {
                        const double dS = P[j] * (dP[j] - mean);
                        double *dk = dK + bshd(b, j, g, 0, Skv, Hkv, D);
                        double *dv = dV + bshd(b, j, g, 0, Skv, Hkv, D);
                        for (long d = 0; d < D; ++d) {
                            dq[d] += scale * dS * load_elem(K, bshd(b, j, g, d, Skv, Hkv, D), dtype, 1.0);
                            dk[d] += scale * dS * load_elem(Q, bshd(b, i, hq, d, Sq, Hq, D), dtype, 1.0);
                            dv[d] += P[j] * load_elem(dO, bshd(b, i, hq, d, Sq, Hq, D), dtype, 1.0);
                        }
                    }
                }
            }
        }
        free(P);
        free(dP);
    }
    return failed ? -1 : nt;
}

int oracle_max_threads(void)
{
    return resolve_threads(0);
}
