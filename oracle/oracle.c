/*
 * oracle.c — CPU oracle for the lattice-PIR database scan.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this code.  The product library never
 * calls it, and the two share no source, header, table or constant generator.
 *
 * Plain, slow, obviously-correct C.  Every function restates one definition
 * from the pages it is checked against:
 *
 *   [VIPIR]  "VIPIR: a general GPU framework for integrating PIR protocols"
 *            (CSDN translation), sections 2.2-2.5 and 4.1-4.3.
 *   [GPIR]   "GPIR: Enabling Practical Private Information Retrieval with
 *            GPUs" (arXiv 2604.04696), the RowSel paragraphs of section 2
 *            (the M_out[p,m,n] formulation) and the ColTor / Dcp
 *            paragraphs of sections 2-3 (the external product, l = 5).
 *
 * Readings of points the pages leave open are stated at each function and
 * listed in the design notes.  Integer arithmetic only; no lazy reduction,
 * no blocking, no reordering beyond the definitions.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <pthread.h>

typedef unsigned __int128 u128;

/* ------------------------------------------------------------------ */
/* Modular arithmetic on residues < q < 2^32 (plain % reductions).      */
/* ------------------------------------------------------------------ */

static uint32_t mulmod(uint32_t a, uint32_t b, uint32_t q)
{
    return (uint32_t)(((uint64_t)a * (uint64_t)b) % q);
}

uint32_t orc_powmod(uint32_t base, uint64_t e, uint32_t q)
{
    uint32_t r = 1 % q;
    uint32_t b = base % q;
    while (e) {
        if (e & 1) r = mulmod(r, b, q);
        b = mulmod(b, b, q);
        e >>= 1;
    }
    return r;
}

/* Inverse by Fermat's little theorem (q prime). */
uint32_t orc_invmod(uint32_t a, uint32_t q)
{
    return orc_powmod(a, (uint64_t)q - 2, q);
}

/* Primality by trial division. */
int orc_is_prime(uint32_t q)
{
    if (q < 2) return 0;
    if (q % 2 == 0) return q == 2;
    for (uint64_t d = 3; d * d <= q; d += 2)
        if (q % d == 0) return 0;
    return 1;
}

/*
 * RNS primes: the `count` largest primes below `bound` with q = 1 (mod 2N),
 * in descending order.  [VIPIR 2.3]: q = q0*q1*q2, each q_i < 2^32 and one row
 * of the 3 x N residue matrix; [VIPIR 4.2]: q_i < 2^29 for lazy reduction.
 * q = 1 (mod 2N) is what makes a negacyclic NTT of length N exist mod q_i.
 * Returns the number found.
 */
int orc_primes(uint32_t N, uint32_t count, uint32_t bound, uint32_t *out)
{
    uint64_t twoN = 2ull * N;
    if (bound < twoN + 2) return 0;
    /* largest x < bound with x = 1 (mod 2N) */
    uint64_t x = ((uint64_t)(bound - 2) / twoN) * twoN + 1;
    int found = 0;
    while (found < (int)count && x > twoN) {
        if (orc_is_prime((uint32_t)x)) out[found++] = (uint32_t)x;
        x -= twoN;
    }
    return found;
}

/*
 * psi: the smallest g in [2, q) with g^N = -1 (mod q).  Any such g has
 * multiplicative order exactly 2N (its order divides 2N but not N, and 2N is
 * a power of two), so it is a primitive 2N-th root of unity.
 * Reading: the pages do not say which root; the smallest one is taken.
 */
uint32_t orc_min_psi(uint32_t q, uint32_t N)
{
    for (uint32_t g = 2; g < q; g++)
        if (orc_powmod(g, N, q) == q - 1) return g;
    return 0;
}

uint32_t orc_bitrev(uint32_t x, uint32_t bits)
{
    uint32_t r = 0;
    for (uint32_t i = 0; i < bits; i++) {
        r = (r << 1) | (x & 1);
        x >>= 1;
    }
    return r;
}

static uint32_t log2u(uint32_t N)
{
    uint32_t b = 0;
    while ((1u << b) < N) b++;
    return b;
}

/* ------------------------------------------------------------------ */
/* Negacyclic NTT over Z_q[X]/(X^N+1)   [VIPIR 2.3]                     */
/* ------------------------------------------------------------------ */

/*
 * Forward transform, straight from the definition (O(N^2)):
 *     out[j] = sum_t a[t] * psi^((2*brv(j)+1)*t)  mod q.
 * out[j] is the value of a(X) at the root psi^(2*brv(j)+1) of X^N+1, so the
 * transform maps a product in Z_q[X]/(X^N+1) to a point-wise product.
 * Reading: output in bit-reversed order of the odd roots (the pages are
 * silent on the order).
 */
void orc_ntt_direct(uint32_t q, uint32_t psi, uint32_t N, const uint32_t *a, uint32_t *out)
{
    uint32_t bits = log2u(N);
    for (uint32_t j = 0; j < N; j++) {
        uint32_t root = orc_powmod(psi, 2ull * orc_bitrev(j, bits) + 1, q);
        uint32_t w = 1 % q;            /* root^t */
        uint64_t acc = 0;
        for (uint32_t t = 0; t < N; t++) {
            acc = (acc + mulmod(a[t], w, q)) % q;
            w = mulmod(w, root, q);
        }
        out[j] = (uint32_t)acc;
    }
}

/*
 * Inverse transform, from the definition:
 *     a[t] = N^-1 * sum_j in[j] * psi^(-(2*brv(j)+1)*t)  mod q.
 */
void orc_intt_direct(uint32_t q, uint32_t psi, uint32_t N, const uint32_t *in, uint32_t *out)
{
    uint32_t bits = log2u(N);
    uint32_t psi_inv = orc_invmod(psi, q);
    uint32_t n_inv = orc_invmod(N % q, q);
    for (uint32_t t = 0; t < N; t++) {
        uint64_t acc = 0;
        for (uint32_t j = 0; j < N; j++) {
            uint64_t e = (2ull * orc_bitrev(j, bits) + 1) * (uint64_t)t;
            acc = (acc + mulmod(in[j], orc_powmod(psi_inv, e % (2ull * N), q), q)) % q;
        }
        out[t] = mulmod((uint32_t)acc, n_inv, q);
    }
}

/*
 * Textbook iterative forward transform (O(N log N)), same result as
 * orc_ntt_direct:
 *   1. twist:      b[t] = a[t] * psi^t            (turns negacyclic into cyclic)
 *   2. cyclic DFT  B[u] = sum_t b[t] * w^(u*t), w = psi^2, by the radix-2
 *      decimation-in-time Cooley-Tukey recursion on bit-reversed input;
 *   3. reorder:    out[j] = B[brv(j)]
 * since psi^((2*brv(j)+1)*t) = psi^t * w^(brv(j)*t).
 * In place on a[0..N).
 */
void orc_ntt_iter(uint32_t q, uint32_t psi, uint32_t N, uint32_t *a)
{
    uint32_t bits = log2u(N);
    uint32_t *tmp = (uint32_t *)malloc(sizeof(uint32_t) * N);
    /* 1. twist */
    uint32_t p = 1 % q;
    for (uint32_t t = 0; t < N; t++) {
        a[t] = mulmod(a[t] % q, p, q);
        p = mulmod(p, psi, q);
    }
    /* 2a. bit-reverse permutation of the input */
    for (uint32_t t = 0; t < N; t++) tmp[orc_bitrev(t, bits)] = a[t];
    /* 2b. DIT butterflies, natural-order output */
    uint32_t w = mulmod(psi, psi, q);
    for (uint32_t len = 2; len <= N; len <<= 1) {
        uint32_t wlen = orc_powmod(w, N / len, q);   /* primitive len-th root */
        for (uint32_t i = 0; i < N; i += len) {
            uint32_t wj = 1 % q;
            for (uint32_t j = 0; j < len / 2; j++) {
                uint32_t u = tmp[i + j];
                uint32_t v = mulmod(tmp[i + j + len / 2], wj, q);
                tmp[i + j] = (uint32_t)(((uint64_t)u + v) % q);
                tmp[i + j + len / 2] = (uint32_t)(((uint64_t)u + q - v) % q);
                wj = mulmod(wj, wlen, q);
            }
        }
    }
    /* 3. bit-reversed output order */
    for (uint32_t j = 0; j < N; j++) a[j] = tmp[orc_bitrev(j, bits)];
    free(tmp);
}

/*
 * Textbook iterative inverse: undo step 3, inverse cyclic DFT with w^-1 and
 * the factor N^-1, then undo the twist with psi^-t.  In place.
 */
void orc_intt_iter(uint32_t q, uint32_t psi, uint32_t N, uint32_t *a)
{
    uint32_t bits = log2u(N);
    uint32_t *B = (uint32_t *)malloc(sizeof(uint32_t) * N);
    uint32_t *tmp = (uint32_t *)malloc(sizeof(uint32_t) * N);
    for (uint32_t j = 0; j < N; j++) B[orc_bitrev(j, bits)] = a[j] % q;
    for (uint32_t t = 0; t < N; t++) tmp[orc_bitrev(t, bits)] = B[t];
    uint32_t psi_inv = orc_invmod(psi, q);
    uint32_t winv = mulmod(psi_inv, psi_inv, q);
    for (uint32_t len = 2; len <= N; len <<= 1) {
        uint32_t wlen = orc_powmod(winv, N / len, q);
        for (uint32_t i = 0; i < N; i += len) {
            uint32_t wj = 1 % q;
            for (uint32_t j = 0; j < len / 2; j++) {
                uint32_t u = tmp[i + j];
                uint32_t v = mulmod(tmp[i + j + len / 2], wj, q);
                tmp[i + j] = (uint32_t)(((uint64_t)u + v) % q);
                tmp[i + j + len / 2] = (uint32_t)(((uint64_t)u + q - v) % q);
                wj = mulmod(wj, wlen, q);
            }
        }
    }
    uint32_t n_inv = orc_invmod(N % q, q);
    uint32_t p = 1 % q;
    for (uint32_t t = 0; t < N; t++) {
        a[t] = mulmod(mulmod(tmp[t], n_inv, q), p, q);
        p = mulmod(p, psi_inv, q);
    }
    free(B);
    free(tmp);
}

/*
 * Schoolbook product in Z_q[X]/(X^N+1):
 *     c[t] = sum_{u+v=t} a[u]*b[v] - sum_{u+v=t+N} a[u]*b[v]  mod q
 * (X^N = -1 folds the upper half back with a minus sign).
 */
void orc_negacyclic_mul(uint32_t q, uint32_t N, const uint32_t *a, const uint32_t *b, uint32_t *c)
{
    for (uint32_t t = 0; t < N; t++) {
        uint64_t pos = 0, neg = 0;
        for (uint32_t u = 0; u < N; u++) {
            uint32_t prod = mulmod(a[u] % q, b[(t + N - u) % N] % q, q);
            if (u <= t) pos = (pos + prod) % q;    /* v = t - u */
            else        neg = (neg + prod) % q;    /* v = t + N - u */
        }
        c[t] = (uint32_t)((pos + q - neg) % q);
    }
}

/* ------------------------------------------------------------------ */
/* Batched helpers (threads over independent polynomials)              */
/* ------------------------------------------------------------------ */

typedef struct {
    uint32_t N, L;
    const uint32_t *q, *psi;
    uint64_t row0, row1;      /* rows [row0,row1) of the [cnt][L][N] array */
    const uint32_t *in;
    uint32_t *out;
    int inverse;
} ntt_job;

static void *ntt_worker(void *arg)
{
    ntt_job *j = (ntt_job *)arg;
    for (uint64_t r = j->row0; r < j->row1; r++) {
        uint32_t l = (uint32_t)(r % j->L);
        uint32_t *dst = j->out + r * j->N;
        if (dst != j->in + r * j->N) memcpy(dst, j->in + r * j->N, sizeof(uint32_t) * j->N);
        if (j->inverse) orc_intt_iter(j->q[l], j->psi[l], j->N, dst);
        else            orc_ntt_iter(j->q[l], j->psi[l], j->N, dst);
    }
    return NULL;
}

static int clamp_threads(int nthreads, uint64_t work)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((uint64_t)nthreads > work) nthreads = (int)(work ? work : 1);
    return nthreads;
}

/*
 * Transform cnt polynomials in RNS form, laid out [cnt][L][N] (row r uses
 * prime r % L).  in may equal out.
 */
void orc_ntt_polys(uint32_t N, uint32_t L, const uint32_t *q, const uint32_t *psi,
                   uint64_t cnt, const uint32_t *in, uint32_t *out, int inverse, int nthreads)
{
    uint64_t rows = cnt * L;
    nthreads = clamp_threads(nthreads, rows);
    pthread_t th[256];
    ntt_job jobs[256];
    for (int i = 0; i < nthreads; i++) {
        jobs[i] = (ntt_job){N, L, q, psi, rows * i / nthreads, rows * (i + 1) / nthreads, in, out, inverse};
        pthread_create(&th[i], NULL, ntt_worker, &jobs[i]);
    }
    for (int i = 0; i < nthreads; i++) pthread_join(th[i], NULL);
}

/*
 * DB encoding of plaintext records [VIPIR 2.4; GPIR section 2]: each record
 * is a polynomial with coefficients in [0, 2^16); it is lifted to R_q (a
 * coefficient below every q_i is its own residue, so the lift copies it into
 * each of the L RNS rows) and brought to the evaluation domain by the forward
 * NTT.  raw is [cnt][N]; out is [cnt][L][N].
 * Reading: no scaling of the plaintext (a BFV plaintext-ciphertext product
 * multiplies by the plaintext as is).
 */
void orc_encode_records(uint32_t N, uint32_t L, const uint32_t *q, const uint32_t *psi,
                        uint64_t cnt, const uint32_t *raw, uint32_t *out, int nthreads)
{
    for (uint64_t r = 0; r < cnt; r++)
        for (uint32_t l = 0; l < L; l++)
            for (uint32_t t = 0; t < N; t++)
                out[(r * L + l) * N + t] = raw[r * N + t] % q[l];
    orc_ntt_polys(N, L, q, psi, cnt, out, out, 0, nthreads);
}

/* ------------------------------------------------------------------ */
/* RowSel  [GPIR section 2]                                             */
/* ------------------------------------------------------------------ */

/*
 * M_out[p,m,n] = sum_k M_in0[p,m,k] * M_in1[p,k,n]  mod q_{l(p)}
 *
 * with p = l*N + j an evaluation point (prime l, NTT slot j), m = 2b + c
 * (query b, ciphertext polynomial c in {0,1}), k < D0 a DB row and n < D1 a
 * DB column:
 *     M_in0[p, 2b+c, k] = query[b][k][c][l][j]      (the D0 query ciphertexts)
 *     M_in1[p, k, n]    = db[k][n][l][j]            (NTT of record (k,n))
 *     M_out[p, 2b+c, n] -> out[b][i][c][l][j]       (D1 result ciphertexts)
 * The sum is exact in 128 bits and reduced once.
 *
 * Layouts (uint32, all residues < q_l):
 *   db    [D0][D1][L][N]
 *   query [B][D0][2][L][N]
 *   out   [B][ncols][2][L][N], where output column i is DB column cols[i].
 * Threads split the output columns.
 * Reading: the pages' "4N" points are L*N residues per polynomial here.
 */
typedef struct {
    uint32_t N, L, D0, D1, B;
    const uint32_t *q, *db, *query, *cols;
    uint32_t ncols, i0, i1;
    uint32_t *out;
} rowsel_job;

static void *rowsel_worker(void *arg)
{
    rowsel_job *J = (rowsel_job *)arg;
    uint64_t P = (uint64_t)J->L * J->N;
    for (uint32_t i = J->i0; i < J->i1; i++) {
        uint32_t n = J->cols[i];
        for (uint32_t b = 0; b < J->B; b++)
            for (uint32_t c = 0; c < 2; c++)
                for (uint64_t p = 0; p < P; p++) {
                    uint32_t q = J->q[p / J->N];
                    u128 acc = 0;
                    for (uint32_t k = 0; k < J->D0; k++) {
                        uint64_t in0 = J->query[(((uint64_t)b * J->D0 + k) * 2 + c) * P + p];
                        uint64_t in1 = J->db[((uint64_t)k * J->D1 + n) * P + p];
                        acc += (u128)(in0 * in1);
                    }
                    J->out[(((uint64_t)b * J->ncols + i) * 2 + c) * P + p] = (uint32_t)(acc % q);
                }
    }
    return NULL;
}

void orc_rowsel(uint32_t N, uint32_t L, const uint32_t *q, uint32_t D0, uint32_t D1, uint32_t B,
                const uint32_t *db, const uint32_t *query, uint32_t ncols, const uint32_t *cols,
                uint32_t *out, int nthreads)
{
    nthreads = clamp_threads(nthreads, ncols);
    pthread_t th[256];
    rowsel_job jobs[256];
    for (int t = 0; t < nthreads; t++) {
        jobs[t] = (rowsel_job){N, L, D0, D1, B, q, db, query, cols, ncols,
                               (uint32_t)((uint64_t)ncols * t / nthreads),
                               (uint32_t)((uint64_t)ncols * (t + 1) / nthreads), out};
        pthread_create(&th[t], NULL, rowsel_worker, &jobs[t]);
    }
    for (int t = 0; t < nthreads; t++) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------------ */
/* Scalar-HE scan  [VIPIR 2.5, 4.1]                                     */
/* ------------------------------------------------------------------ */

/*
 * out[r][b] = sum_c db[r][c] * Q[c][b]  mod 2^32
 * The DB GEMM of SimplePIR-style folding: a D1 x B x D0 GEMM of a byte DB by
 * 32-bit query words, where arithmetic mod 2^32 is plain wrap-around
 * ("the modular reduction is free").  uint32 arithmetic wraps by definition.
 * db rows are given as a list: db_rows is [nrows][C] (row i of it is DB row
 * rows[i]); out is [nrows][B].  Q is [C][B].  Threads split the rows.
 * Reading: DB bytes are unsigned, in [0, 256).
 */
typedef struct {
    uint64_t C;
    uint32_t B;
    const uint8_t *db_rows;
    const uint32_t *Q;
    uint32_t *out;
    uint64_t i0, i1;
} scalar_job;

static void *scalar_worker(void *arg)
{
    scalar_job *J = (scalar_job *)arg;
    for (uint64_t i = J->i0; i < J->i1; i++) {
        for (uint32_t b = 0; b < J->B; b++) {
            uint32_t acc = 0;
            for (uint64_t c = 0; c < J->C; c++)
                acc += (uint32_t)J->db_rows[i * J->C + c] * J->Q[c * J->B + b];
            J->out[i * J->B + b] = acc;
        }
    }
    return NULL;
}

void orc_scalar_scan(uint64_t nrows, uint64_t C, uint32_t B, const uint8_t *db_rows,
                     const uint32_t *Q, uint32_t *out, int nthreads)
{
    nthreads = clamp_threads(nthreads, nrows);
    pthread_t th[256];
    scalar_job jobs[256];
    for (int t = 0; t < nthreads; t++) {
        jobs[t] = (scalar_job){C, B, db_rows, Q, out, nrows * t / nthreads, nrows * (t + 1) / nthreads};
        pthread_create(&th[t], NULL, scalar_worker, &jobs[t]);
    }
    for (int t = 0; t < nthreads; t++) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------------ */
/* ColTor: gadget decomposition and the RGSW-RLWE external product      */
/* [GPIR section 2 and the ColTor paragraphs of section 3 (Dcp, l = 5); */
/*  VIPIR 3.6 step 7 and section 5 (q ~ 2^87 in 3 RNS primes)]          */
/* ------------------------------------------------------------------ */

/*
 * The integer X in [0, Q), Q = q_0 * ... * q_{L-1}, with X = x_l (mod q_l),
 * by Garner's mixed-radix recurrence:
 *     v_l = (((x_l - v_0) q_0^-1 - v_1) q_1^-1 - ... - v_{l-1}) q_{l-1}^-1  mod q_l
 *     X   = v_0 + q_0 (v_1 + q_1 (v_2 + ...)).
 * Requires Q < 2^128 (L <= 4 primes below 2^32).
 */
static u128 crt_garner(uint32_t L, const uint32_t *q, const uint32_t *x)
{
    uint32_t v[4];
    for (uint32_t l = 0; l < L; l++) {
        uint64_t t = x[l] % q[l];
        for (uint32_t k = 0; k < l; k++) {
            t = (t + q[l] - v[k] % q[l]) % q[l];
            t = (uint64_t)mulmod((uint32_t)t, orc_invmod(q[k] % q[l], q[l]), q[l]);
        }
        v[l] = (uint32_t)t;
    }
    u128 X = 0;
    for (int l = (int)L - 1; l >= 0; l--) X = X * q[l] + v[l];
    return X;
}

/*
 * Gadget decomposition Dcp of one polynomial of R_Q in coefficient form,
 * x[l][t] (L rows of N residues): every coefficient X (the CRT value above)
 * is written in base 2^w with ell digits,
 *     X = sum_{u < ell} d_u 2^(w u),   d_u = floor(X / 2^(w u)) mod 2^w,
 * and d[u][t] = d_u.  Readings (the pages fix only ell = 5 at Q ~ 2^87):
 * unsigned digits of the CRT value, base 2^w with w * ell >= bits of Q
 * (w = 18 for ell = 5), digit 0 the least significant.
 */
void orc_dcp(uint32_t N, uint32_t L, const uint32_t *q, uint32_t ell, uint32_t w,
             const uint32_t *x, uint32_t *d)
{
    uint32_t xs[4];
    const u128 mask = (w >= 128) ? ~(u128)0 : (((u128)1 << w) - 1);
    for (uint32_t t = 0; t < N; t++) {
        for (uint32_t l = 0; l < L; l++) xs[l] = x[(uint64_t)l * N + t];
        u128 X = crt_garner(L, q, xs);
        for (uint32_t u = 0; u < ell; u++) {
            uint32_t sh = w * u;
            d[(uint64_t)u * N + t] = sh >= 128 ? 0u : (uint32_t)((X >> sh) & mask);
        }
    }
}

/*
 * External product of an RGSW ciphertext C with an RLWE ciphertext ct:
 *     out_c = sum_{u < ell} NTT(Dcp_u(ct_0)) (.) C[u]_c
 *           + sum_{u < ell} NTT(Dcp_u(ct_1)) (.) C[ell + u]_c      (c = 0, 1)
 * point-wise mod q_l, where (.) is the point-wise product of NTT vectors.
 *   C   : [2 ell][2][L][N], NTT form (row u pairs with digit u of ct_0,
 *         row ell + u with digit u of ct_1: the layout Z + m * (I_2 x g)
 *         of an RGSW encryption of m with gadget g_u = 2^(w u)).
 *   ct  : [2][L][N], coefficient form.
 *   out : [2][L][N], NTT form.
 * Each digit is a plain integer below 2^w; it is lifted to every prime
 * (reduced mod q_l) and transformed with the iterative NTT above.
 */
void orc_ext_product(uint32_t N, uint32_t L, const uint32_t *q, const uint32_t *psi, uint32_t ell,
                     uint32_t w, const uint32_t *C, const uint32_t *ct, uint32_t *out)
{
    uint64_t PN = (uint64_t)L * N;
    uint32_t *d = (uint32_t *)malloc(sizeof(uint32_t) * ell * N);
    uint32_t *dn = (uint32_t *)malloc(sizeof(uint32_t) * 2 * ell * PN);   /* [cin][u][l][t] */
    for (uint32_t cin = 0; cin < 2; cin++) {
        orc_dcp(N, L, q, ell, w, ct + cin * PN, d);
        for (uint32_t u = 0; u < ell; u++)
            for (uint32_t l = 0; l < L; l++) {
                uint32_t *row = dn + ((uint64_t)(cin * ell + u) * L + l) * N;
                for (uint32_t t = 0; t < N; t++) row[t] = d[(uint64_t)u * N + t] % q[l];
                orc_ntt_iter(q[l], psi[l], N, row);
            }
    }
    for (uint32_t c = 0; c < 2; c++)
        for (uint32_t l = 0; l < L; l++)
            for (uint32_t j = 0; j < N; j++) {
                u128 acc = 0;
                for (uint32_t v = 0; v < 2 * ell; v++)
                    acc += (u128)dn[((uint64_t)v * L + l) * N + j] *
                           C[(((uint64_t)v * 2 + c) * L + l) * N + j];
                out[((uint64_t)c * L + l) * N + j] = (uint32_t)(acc % q[l]);
            }
    free(d);
    free(dn);
}

/*
 * One ColTor stage (the column tournament's selection by one bit):
 *     out_i = ct_{2i} + C (x) (ct_{2i+1} - ct_{2i}),   i < ceil(nin / 2),
 * with (x) the external product above, all ciphertexts in NTT form; the
 * difference is brought to coefficient form by the inverse NTT before Dcp.
 * C encrypting 0 keeps ct_{2i}, C encrypting 1 takes ct_{2i+1}.
 * Reading: when nin is odd the last ciphertext meets the zero ciphertext
 * (the tournament padded with zeros to an even count).
 *   in  : [nin][2][L][N], out : [ceil(nin/2)][2][L][N].
 */
typedef struct {
    uint32_t N, L, ell, w;
    const uint32_t *q, *psi, *C, *in;
    uint64_t nin, i0, i1;
    uint32_t *out;
} coltor_job;

static void *coltor_worker(void *arg)
{
    coltor_job *j = (coltor_job *)arg;
    uint64_t PN = (uint64_t)j->L * j->N, CT = 2 * PN;
    uint32_t *diff = (uint32_t *)malloc(sizeof(uint32_t) * CT);
    uint32_t *ext = (uint32_t *)malloc(sizeof(uint32_t) * CT);
    for (uint64_t i = j->i0; i < j->i1; i++) {
        const uint32_t *even = j->in + 2 * i * CT;
        const uint32_t *odd = (2 * i + 1 < j->nin) ? j->in + (2 * i + 1) * CT : NULL;
        for (uint32_t c = 0; c < 2; c++)
            for (uint32_t l = 0; l < j->L; l++) {
                uint32_t ql = j->q[l];
                uint64_t base = ((uint64_t)c * j->L + l) * j->N;
                for (uint32_t t = 0; t < j->N; t++) {
                    uint64_t o = odd ? odd[base + t] % ql : 0;
                    diff[base + t] = (uint32_t)((o + ql - even[base + t] % ql) % ql);
                }
                orc_intt_iter(ql, j->psi[l], j->N, diff + base);
            }
        orc_ext_product(j->N, j->L, j->q, j->psi, j->ell, j->w, j->C, diff, ext);
        uint32_t *dst = j->out + i * CT;
        for (uint32_t c = 0; c < 2; c++)
            for (uint32_t l = 0; l < j->L; l++) {
                uint64_t base = ((uint64_t)c * j->L + l) * j->N;
                for (uint32_t t = 0; t < j->N; t++)
                    dst[base + t] = (uint32_t)(((uint64_t)even[base + t] % j->q[l] + ext[base + t]) % j->q[l]);
            }
    }
    free(diff);
    free(ext);
    return NULL;
}

void orc_coltor_stage(uint32_t N, uint32_t L, const uint32_t *q, const uint32_t *psi, uint32_t ell,
                      uint32_t w, const uint32_t *C, const uint32_t *in, uint64_t nin, uint32_t *out,
                      int nthreads)
{
    uint64_t nout = (nin + 1) / 2;
    nthreads = clamp_threads(nthreads, nout);
    pthread_t th[256];
    coltor_job jobs[256];
    for (int i = 0; i < nthreads; i++) {
        jobs[i] = (coltor_job){N, L, ell, w, q, psi, C, in, nin, nout * i / nthreads,
                               nout * (i + 1) / nthreads, out};
        pthread_create(&th[i], NULL, coltor_worker, &jobs[i]);
    }
    for (int i = 0; i < nthreads; i++) pthread_join(th[i], NULL);
}

/* ------------------------------------------------------------------ */
/* ExpandQuery: Subs (automorphism + key switching) and the expansion   */
/* tree [GPIR section 2 (ExpandQuery, Subs, evk, up to log N stages)    */
/*  and section 3 (Subs touches only the a polynomial)]                 */
/* ------------------------------------------------------------------ */

/*
 * Automorphism sigma_k: a(X) -> a(X^k) in Z_q[X]/(X^N+1), k odd, in
 * coefficient form: coefficient t moves to t*k mod 2N, with a minus sign
 * when that lands in [N, 2N) (X^N = -1).  a, out: [L][N].
 */
void orc_automorph(uint32_t N, uint32_t L, const uint32_t *q, uint32_t k, const uint32_t *a, uint32_t *out)
{
    for (uint32_t l = 0; l < L; l++)
        for (uint32_t t = 0; t < N; t++) {
            uint64_t e = (uint64_t)t * k % (2ull * N);
            uint32_t v = a[(uint64_t)l * N + t] % q[l];
            if (e < N) out[(uint64_t)l * N + e] = v;
            else       out[(uint64_t)l * N + (e - N)] = (q[l] - v) % q[l];
        }
}

/*
 * Subs(ct, k) for ct = (c0, c1) decrypting as c0 + c1 s, with the
 * evaluation key evk[u] = an RLWE encryption of sigma_k(s) g_u under s:
 *     Subs(ct, k) = (NTT(sigma_k(c0)), 0)
 *                 + sum_{u<ell} NTT(Dcp_u(sigma_k(c1))) (.) evk[u]
 * Readings: only the a polynomial c1 is decomposed (GPIR section 3); Dcp is
 * the decomposition of orc_dcp; evk is [ell][2][L][N] in NTT form.
 *   ct, out : [2][L][N], NTT form.
 */
void orc_subs(uint32_t N, uint32_t L, const uint32_t *q, const uint32_t *psi, uint32_t ell, uint32_t w,
              uint32_t k, const uint32_t *evk, const uint32_t *ct, uint32_t *out)
{
    uint64_t PN = (uint64_t)L * N;
    uint32_t *c = (uint32_t *)malloc(sizeof(uint32_t) * 2 * PN);
    uint32_t *s = (uint32_t *)malloc(sizeof(uint32_t) * 2 * PN);
    uint32_t *d = (uint32_t *)malloc(sizeof(uint32_t) * ell * N);
    uint32_t *dn = (uint32_t *)malloc(sizeof(uint32_t) * ell * PN);
    memcpy(c, ct, sizeof(uint32_t) * 2 * PN);
    for (uint32_t p = 0; p < 2; p++)
        for (uint32_t l = 0; l < L; l++) orc_intt_iter(q[l], psi[l], N, c + p * PN + (uint64_t)l * N);
    orc_automorph(N, L, q, k, c, s);              /* sigma(c0) */
    orc_automorph(N, L, q, k, c + PN, s + PN);    /* sigma(c1) */
    orc_dcp(N, L, q, ell, w, s + PN, d);
    for (uint32_t u = 0; u < ell; u++)
        for (uint32_t l = 0; l < L; l++) {
            uint32_t *row = dn + ((uint64_t)u * L + l) * N;
            for (uint32_t t = 0; t < N; t++) row[t] = d[(uint64_t)u * N + t] % q[l];
            orc_ntt_iter(q[l], psi[l], N, row);
        }
    for (uint32_t l = 0; l < L; l++) orc_ntt_iter(q[l], psi[l], N, s + (uint64_t)l * N);   /* NTT(sigma(c0)) */
    for (uint32_t p = 0; p < 2; p++)
        for (uint32_t l = 0; l < L; l++)
            for (uint32_t j = 0; j < N; j++) {
                u128 acc = p == 0 ? s[(uint64_t)l * N + j] : 0;
                for (uint32_t u = 0; u < ell; u++)
                    acc += (u128)dn[((uint64_t)u * L + l) * N + j] * evk[(((uint64_t)u * 2 + p) * L + l) * N + j];
                out[p * PN + (uint64_t)l * N + j] = (uint32_t)(acc % q[l]);
            }
    free(c);
    free(s);
    free(d);
    free(dn);
}

/*
 * One expansion stage j (Galois element k = N / 2^j + 1) over M ciphertexts:
 *     out[i]     = ct_i + Subs(ct_i, k)
 *     out[i + M] = (ct_i - Subs(ct_i, k)) * X^(-2^j)
 * all in NTT form; the product by the monomial is point-wise by its NTT.
 * Reading: the expansion tree of the SealPIR/OnionPIR family in this output
 * order, so that after S stages ciphertext r carries coefficient r of the
 * query plaintext, times 2^S, as a constant polynomial.
 *   evk : [ell][2][L][N] (the key of this stage), in : [M][2][L][N],
 *   out : [2M][2][L][N].
 */
typedef struct {
    uint32_t N, L, ell, w, j;
    const uint32_t *q, *psi, *evk, *in;
    uint64_t M, i0, i1;
    uint32_t *out;
} expand_job;

static void *expand_worker(void *arg)
{
    expand_job *jb = (expand_job *)arg;
    uint32_t N = jb->N, L = jb->L;
    uint64_t PN = (uint64_t)L * N, CT = 2 * PN;
    uint32_t k = N / (1u << jb->j) + 1;
    uint32_t *sub = (uint32_t *)malloc(sizeof(uint32_t) * CT);
    uint32_t *mono = (uint32_t *)malloc(sizeof(uint32_t) * PN);
    /* NTT(X^(-2^j)) = NTT(-X^(N - 2^j)) */
    for (uint32_t l = 0; l < L; l++) {
        uint32_t *row = mono + (uint64_t)l * N;
        memset(row, 0, sizeof(uint32_t) * N);
        row[N - (1u << jb->j)] = jb->q[l] - 1;                     /* j < log2 N */
        orc_ntt_iter(jb->q[l], jb->psi[l], N, row);
    }
    for (uint64_t i = jb->i0; i < jb->i1; i++) {
        const uint32_t *ct = jb->in + i * CT;
        orc_subs(N, L, jb->q, jb->psi, jb->ell, jb->w, k, jb->evk, ct, sub);
        uint32_t *o1 = jb->out + i * CT, *o2 = jb->out + (i + jb->M) * CT;
        for (uint32_t p = 0; p < 2; p++)
            for (uint32_t l = 0; l < L; l++) {
                uint32_t ql = jb->q[l];
                for (uint32_t t = 0; t < N; t++) {
                    uint64_t x = p * PN + (uint64_t)l * N + t;
                    uint64_t a = ct[x] % ql, b = sub[x];
                    o1[x] = (uint32_t)((a + b) % ql);
                    o2[x] = (uint32_t)((((a + ql - b) % ql) * mono[(uint64_t)l * N + t]) % ql);
                }
            }
    }
    free(sub);
    free(mono);
    return NULL;
}

void orc_expand_stage(uint32_t N, uint32_t L, const uint32_t *q, const uint32_t *psi, uint32_t ell, uint32_t w,
                      uint32_t j, const uint32_t *evk, const uint32_t *in, uint64_t M, uint32_t *out,
                      int nthreads)
{
    nthreads = clamp_threads(nthreads, M);
    pthread_t th[256];
    expand_job jobs[256];
    for (int i = 0; i < nthreads; i++) {
        jobs[i] = (expand_job){N, L, ell, w, j, q, psi, evk, in, M, M * i / nthreads, M * (i + 1) / nthreads, out};
        pthread_create(&th[i], NULL, expand_worker, &jobs[i]);
    }
    for (int i = 0; i < nthreads; i++) pthread_join(th[i], NULL);
}

/* ------------------------------------------------------------------ */
/* RGSW ciphertexts from the expanded query                             */
/* [GPIR section 2: the expanded query ciphertext carries both indices,  */
/*  the expansion yields the D0 RowSel ciphertexts "and RGSW"            */
/*  ciphertexts; the conversion itself is not defined on the pages]      */
/* ------------------------------------------------------------------ */

/*
 * Reading: the client places m g_u (g_u = 2^(w u), the gadget of orc_dcp)
 * in ell query coefficients, so the expansion yields RLWE'(m) = the ell
 * ciphertexts ct_u = (c0_u, c1_u) of m g_u.  An RGSW ciphertext of m in the
 * row layout of orc_ext_product needs rows u encrypting m g_u (ct_u itself)
 * and rows ell + u encrypting m s g_u.  With a key-switching key
 * ksk[v] = RLWE(s^2 g_v) the latter is
 *     C[ell + u] = (0, c0_u) + sum_{v<ell} NTT(Dcp_v(c1_u)) (.) ksk[v]
 * which decrypts to c0_u s + c1_u s^2 = s (c0_u + c1_u s) = m s g_u + s e_u.
 *   ksk : [ell][2][L][N], NTT form.
 *   in  : [ell][2][L][N], NTT form (ct_u for u < ell).
 *   out : [2 ell][2][L][N], NTT form (out[u] = ct_u, out[ell + u] above).
 * c1_u is brought to coefficient form by the inverse NTT before Dcp.
 */
void orc_rgsw_convert(uint32_t N, uint32_t L, const uint32_t *q, const uint32_t *psi, uint32_t ell,
                      uint32_t w, const uint32_t *ksk, const uint32_t *in, uint32_t *out)
{
    uint64_t PN = (uint64_t)L * N, CT = 2 * PN;
    uint32_t *c1 = (uint32_t *)malloc(sizeof(uint32_t) * PN);
    uint32_t *d = (uint32_t *)malloc(sizeof(uint32_t) * ell * N);
    uint32_t *dn = (uint32_t *)malloc(sizeof(uint32_t) * ell * PN);
    for (uint32_t u = 0; u < ell; u++) {
        const uint32_t *ct = in + u * CT;
        memcpy(out + u * CT, ct, sizeof(uint32_t) * CT);
        memcpy(c1, ct + PN, sizeof(uint32_t) * PN);
        for (uint32_t l = 0; l < L; l++) orc_intt_iter(q[l], psi[l], N, c1 + (uint64_t)l * N);
        orc_dcp(N, L, q, ell, w, c1, d);
        for (uint32_t v = 0; v < ell; v++)
            for (uint32_t l = 0; l < L; l++) {
                uint32_t *row = dn + ((uint64_t)v * L + l) * N;
                for (uint32_t t = 0; t < N; t++) row[t] = d[(uint64_t)v * N + t] % q[l];
                orc_ntt_iter(q[l], psi[l], N, row);
            }
        uint32_t *dst = out + (ell + u) * CT;
        for (uint32_t p = 0; p < 2; p++)
            for (uint32_t l = 0; l < L; l++)
                for (uint32_t j = 0; j < N; j++) {
                    u128 acc = p == 1 ? ct[(uint64_t)l * N + j] : 0;     /* (0, c0) */
                    for (uint32_t v = 0; v < ell; v++)
                        acc += (u128)dn[((uint64_t)v * L + l) * N + j] * ksk[(((uint64_t)v * 2 + p) * L + l) * N + j];
                    dst[p * PN + (uint64_t)l * N + j] = (uint32_t)(acc % q[l]);
                }
    }
    free(c1);
    free(d);
    free(dn);
}
