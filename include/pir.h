/*
 * pir.h — C ABI of the GB300 (sm_103a) server-side scan of lattice-based
 * single-server PIR.
 *
 * Two scans are provided:
 *
 *  - RowSel, the first-dimension fold of the OnionPIR family.  Every DB record
 *    is a plaintext polynomial in R_q = Z_q[X]/(X^N+1), q held in RNS
 *    (q_i < 2^29, q_i = 1 mod 2N).  DB and query are in the evaluation
 *    (NTT) domain, where the fold becomes L*N independent point-wise GEMMs
 *        M_out[p,m,n] = sum_k M_in0[p,m,k] * M_in1[p,k,n]  mod q_{l(p)}
 *    (GPIR, arXiv 2604.04696, section 2, the RowSel formulation; VIPIR,
 *    sections 2.3 and 4.2).
 *
 *  - the scalar-HE scan, the first fold of the SimplePIR family: a byte DB
 *    times a matrix of 32-bit query words, mod 2^32 (VIPIR, sections 2.5
 *    and 4.1).
 *
 * Conventions for every call:
 *  - All buffers are owned and allocated by the caller; pointers marked
 *    "device" must be device memory of the context's GPU, 16-byte aligned.
 *    The library allocates device memory only in pir_ctx_create (its
 *    twiddle tables, the expansion stages' monomial factors and a status
 *    word) and frees it in pir_ctx_destroy.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and returns before it completes.  Inputs must stay valid and
 *    unmodified until the stream reaches the work.
 *  - Return value: PIR_OK (0) or a negative PIR_ERR_* code.  Arguments are
 *    validated on the host before anything is enqueued; a failed call
 *    enqueues nothing.  Nothing is thrown across the ABI.
 *  - Residues are uint32 values in [0, q_l).  Input values are not range
 *    checked on the device; residues >= q_l give unspecified (but memory-safe)
 *    results.
 *  - Device-side waits are bounded.  A kernel that gives up sets a bit in the
 *    context's status word (pir_status) instead of hanging.
 */
#ifndef PIR_H
#define PIR_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PIR_OK 0
#define PIR_ERR_ARG (-1)          /* invalid argument (size, pointer, parameters) */
#define PIR_ERR_CUDA (-2)         /* a CUDA runtime/driver call or launch failed */
#define PIR_ERR_UNSUPPORTED (-3)  /* valid but outside what the library implements */
#define PIR_ERR_ALLOC (-4)        /* pir_ctx_create / pir_server_create could not allocate */

/* Bits of the device status word (pir_status). */
#define PIR_STATUS_TIMEOUT 1u     /* a bounded device wait ran out */

#define PIR_MAX_RNS 4
#define PIR_SLAB 128              /* width (uint32 words) of one DB column slab */

typedef struct pir_ctx pir_ctx;

/*
 * pir_params_check — validate ring parameters on the host (no GPU needed).
 * N: ring degree, a power of two in [16, 4096] (VIPIR 2.2 uses N = 2^12).
 * L: number of RNS primes, 1..4 (VIPIR 2.3 uses #RNS = 3).
 * q: host array of L distinct primes with q_i < 2^29 and q_i = 1 (mod 2N)
 *    (VIPIR 4.2: primes below 2^29 for 64-bit lazy accumulation).
 * Returns PIR_OK or PIR_ERR_ARG.
 */
int pir_params_check(uint32_t N, uint32_t L, const uint32_t *q);

/*
 * pir_primes — the L largest primes q < 2^29 with q = 1 (mod 2N), in
 * descending order, written to q (host, L entries).  Host only.  These are
 * the RNS primes of the workloads (VIPIR 2.3: q = q0*q1*q2 ~ 2^87 with
 * #RNS = 3; VIPIR 4.2: q_i < 2^29).
 * Errors: PIR_ERR_ARG (N not a power of two in [16, 4096], L not in 1..4,
 * q NULL).
 */
int pir_primes(uint32_t N, uint32_t L, uint32_t *q);

/*
 * pir_ctx_create — build a context for ring degree N and RNS primes q[0..L)
 * on CUDA device `device`: validates the parameters (as pir_params_check),
 * selects for each q_i the smallest primitive 2N-th root of unity psi_i, and
 * uploads its twiddle tables and, for ExpandQuery, NTT(X^(-2^j)) for every
 * stage j < log2 N (log2 N * L * N words).  *out receives the context (NULL
 * on error).
 * Errors: PIR_ERR_ARG, PIR_ERR_CUDA, PIR_ERR_ALLOC.
 */
int pir_ctx_create(pir_ctx **out, uint32_t N, uint32_t L, const uint32_t *q, int device);

/* pir_ctx_destroy — free the context's device tables (synchronises the device). */
void pir_ctx_destroy(pir_ctx *ctx);

/*
 * pir_ctx_psi — copy the L roots psi_i chosen by the context into psi (host).
 * The NTT-domain convention below depends on them.
 */
int pir_ctx_psi(const pir_ctx *ctx, uint32_t *psi);

/*
 * pir_ntt_fwd — forward negacyclic NTT of cnt RNS polynomials
 * (VIPIR 2.3: the per-row transform that turns a product in R_q into a
 * point-wise product mod q_i; VIPIR 4.3: one kernel per N = 2^12 transform).
 *   in, out : device, [cnt][L][N] uint32; row l of each polynomial holds
 *             residues mod q_l.  in == out (in place) is allowed; otherwise
 *             the buffers must not overlap.
 *   Output convention: out[j] = sum_t in[t] * psi^((2*brv(j)+1)*t) mod q_l,
 *   brv = log2(N)-bit reversal; outputs are canonical residues in [0, q_l).
 * Errors: PIR_ERR_ARG (NULL/unaligned pointer, cnt*L*N overflow), PIR_ERR_CUDA.
 * cnt = 0 is a no-op.
 */
int pir_ntt_fwd(pir_ctx *ctx, const uint32_t *in, uint32_t *out, uint64_t cnt, void *stream);

/*
 * pir_ntt_inv — inverse of pir_ntt_fwd including the factor N^-1:
 *   out[t] = N^-1 * sum_j in[j] * psi^(-(2*brv(j)+1)*t) mod q_l.
 * Same layout, aliasing rules and errors as pir_ntt_fwd.
 */
int pir_ntt_inv(pir_ctx *ctx, const uint32_t *in, uint32_t *out, uint64_t cnt, void *stream);

/*
 * pir_lift_ntt — lift plain 32-bit coefficients into R_q and transform them
 * (VIPIR 3.5.2 and 3.6 step 3: the INT32 scan output, read as length-N
 * coefficient vectors, becomes polynomials that are taken to NTT form, G).
 *   raw : device, [cnt][N] uint32, any value; coefficient t of polynomial i
 *         is raw[i*N + t], lifted to its residue mod q_l for every prime l.
 *   out : device, [cnt][L][N], out[i][l] = NTT(raw[i] mod q_l) with the
 *         output convention of pir_ntt_fwd.
 *   raw and out must not overlap.
 * Errors: PIR_ERR_ARG (NULL/unaligned pointer, overlap, size overflow),
 * PIR_ERR_CUDA.  cnt = 0 is a no-op.
 */
int pir_lift_ntt(pir_ctx *ctx, const uint32_t *raw, uint32_t *out, uint64_t cnt, void *stream);

/*
 * pir_db_bytes — bytes of the encoded RowSel DB for a D0 x D1 grid of records
 * (GPIR section 2: DB[i][j], i < D0, j < D1), i.e. L*N*D0*D1p*4 with
 * D1p = D1 rounded up to a multiple of 4.  Returns 0 for invalid sizes.
 *
 * Encoded layout ("column slabs", k/n-contiguous per evaluation point):
 *   evaluation point p = l*N + j (prime l, NTT slot j), record (k, n);
 *   columns are cut into slabs of PIR_SLAB = 128 columns, s = n / 128; the
 *   last slab is W_last = D1p - 128*(S-1) wide, S = ceil(D1/128).  Word
 *       db[ p*D0*D1p + s*D0*128 + k*W_s + (n - 128*s) ]
 *   holds NTT(record(k,n))[l][j], where W_s = 128 for s < S-1, W_last for
 *   the last slab.  Each (p, slab) is one contiguous D0 x W_s block.
 *   Padding columns n in [D1, D1p) hold 0.
 */
uint64_t pir_db_bytes(const pir_ctx *ctx, uint32_t D0, uint32_t D1);

/*
 * pir_db_encode — offline DB encoding (VIPIR 2.4: lift of the plaintext to
 * R_q and NTT; GPIR section 2: DB records as NTT-domain vectors), for DB rows
 * k0 .. k0+kcnt-1 of a D0 x D1 DB.
 *   raw : device, [kcnt][D1][N] uint32 plaintext coefficients (each is
 *         lifted to R_q as its residue mod q_l; the workloads use [0, 2^16)).
 *   db  : device, pir_db_bytes(ctx, D0, D1) bytes, layout above.  Only the
 *         words of rows k0..k0+kcnt-1 (including their padding columns) are
 *         written, so the DB can be encoded in row chunks.
 * Errors: PIR_ERR_ARG (k0+kcnt > D0, zero sizes, NULL/unaligned), PIR_ERR_CUDA.
 */
int pir_db_encode(pir_ctx *ctx, const uint32_t *raw, uint32_t k0, uint32_t kcnt,
                  uint32_t D0, uint32_t D1, uint32_t *db, void *stream);

/*
 * pir_rowsel_workspace_bytes — device workspace pir_rowsel needs for a
 * D0 x D1 DB and B queries: the largest pass's query in point-major order
 * (L*N * roundup(D0*Mp, 4) words, Mp = the pass's polynomial count padded to
 * a power of two, at most 32) and its results in point-major order
 * (L*N * 2*nb * roundup(D1, 4) words, nb = queries in the pass).
 * 0 for invalid sizes.
 */
uint64_t pir_rowsel_workspace_bytes(const pir_ctx *ctx, uint32_t D0, uint32_t D1, uint32_t B);

/*
 * pir_rowsel — the RowSel scan (GPIR section 2):
 *   out[b][n][c][l][j] = sum_{k<D0} query[b][k][c][l][j] * DB(k,n)[l][j]  mod q_l
 * i.e. M_out[p, m=2b+c, n] = sum_k M_in0[p,m,k] * M_in1[p,k,n] with p = l*N+j:
 * B queries, each D0 BFV ciphertexts (2 polynomials, NTT form), fold a
 * D0 x D1 DB into D1 ciphertexts per query.
 *   db    : device, encoded by pir_db_encode for the same ctx, D0, D1.
 *   query : device, [B][D0][2][L][N] uint32 residues (NTT form).
 *   out   : device, [B][D1][2][L][N] uint32 (NTT form, canonical residues).
 *   workspace : device, >= pir_rowsel_workspace_bytes(ctx, D0, D1, B) bytes,
 *               16-byte aligned; holds the query transposed to point-major
 *               order and the results before they are transposed back
 *               (GPIR's NTT-to-GEMM layout change, both directions);
 *               contents undefined after the call.
 * The DB is read from HBM once per pass.  When every q_l >= 2^26, passes of
 * 16 queries run on the tensor cores (exact fp16 digit products, the rows
 * taken in K segments of 512) while more than 8 queries remain, any D0; a
 * last pass of 9 to 15 queries too.  Every other pass (8 queries or fewer,
 * or primes below 2^26) runs on the CUDA cores and covers as many queries
 * as fit its on-chip query buffer (16 for D0 <= 896, fewer for larger D0).
 * Both give the same canonical residues.
 * Errors: PIR_ERR_ARG (zero sizes, NULL/unaligned, workspace too small),
 * PIR_ERR_CUDA, PIR_ERR_UNSUPPORTED (D0 > 14336).
 */
int pir_rowsel(pir_ctx *ctx, const uint32_t *db, uint32_t D0, uint32_t D1,
               const uint32_t *query, uint32_t B, uint32_t *out,
               void *workspace, uint64_t workspace_bytes, void *stream);

/*
 * pir_exppack — the INT32 modular GEMM of expansion-based ring packing
 * (VIPIR 3.5.2): with H (Dr x n polynomials) and G (Dr x B polynomials), the
 * NTT-domain forms of the B-batched SimplePIR hint and answers, and C
 * (n x 2B polynomials) the expanded "special" ciphertexts of B clients,
 *     out = H * C + (0 | G),
 * i.e. for client b, output ciphertext r (one per hint row) and RNS point p:
 *     out[b][r][c][p] = sum_{k<n} H[r][k][p] * C[b][k][c][p]
 *                       + (c == 1 ? G[b][r][p] : 0)        mod q_{l(p)}.
 * This is RowSel's point-wise GEMM with the hint as the DB: record (k, r) of a
 * D0 = n by D1 = Dr DB is H[r][k].
 *   h_db : device, H encoded by pir_db_encode(ctx, ..., D0 = n, D1 = Dr),
 *          record (k, r) = polynomial H[r][k] (coefficients, lifted mod q_l).
 *   C    : device, [B][n][2][L][N] residues (NTT form).
 *   G    : device, [B][Dr][L][N] residues (NTT form), added to polynomial 1
 *          (the "b" part) of every output ciphertext; must not be NULL.
 *   out  : device, [B][Dr][2][L][N] (NTT form).
 *   workspace : as for pir_rowsel, pir_rowsel_workspace_bytes(ctx, n, Dr, B).
 * Reading: "(0 | G)" is taken as (0, G_b) per client ciphertext, G joining
 * the polynomial that carries the message.
 * Errors: as pir_rowsel; PIR_ERR_ARG for a NULL or unaligned G.
 */
int pir_exppack(pir_ctx *ctx, const uint32_t *h_db, uint32_t n, uint32_t Dr, const uint32_t *C,
                const uint32_t *G, uint32_t B, uint32_t *out, void *workspace,
                uint64_t workspace_bytes, void *stream);

/*
 * ColTor — the column tournament of the OnionPIR family (GPIR section 2;
 * GPIR section 3 for Dcp and l = 5; VIPIR 3.6 step 7 for the RGSW-RLWE
 * external products after the first folding, VIPIR 5 for q ~ 2^87).
 *
 * Gadget decomposition Dcp (reading: unsigned digits of each coefficient's
 * CRT value X in [0, Q), Q = q_0 ... q_{L-1}, base 2^w, ell digits, digit 0
 * the least significant):   X = sum_{u<ell} Dcp_u 2^(w u).
 * External product of an RGSW ciphertext C with an RLWE ciphertext ct:
 *     C (x) ct = sum_u NTT(Dcp_u(ct_0)) . C[u] + NTT(Dcp_u(ct_1)) . C[ell+u]
 * ("." point-wise mod q_l), so a noise-free RGSW of m (C[u] = (m g_u, 0),
 * C[ell+u] = (0, m g_u), g_u = 2^(w u)) gives m * ct exactly.
 * One tournament stage over n ciphertexts:
 *     out_i = ct_2i + C (x) (ct_2i+1 - ct_2i),   i < ceil(n/2),
 * a missing partner (n odd) being the zero ciphertext; C encrypting 0 keeps
 * ct_2i, C encrypting 1 takes ct_2i+1.
 *
 *   C    : device, [2 ell][2][L][N] NTT form (one stage's RGSW ciphertext);
 *          for pir_coltor, [S][2 ell][2][L][N] with S = ceil(log2 n) stages,
 *          stage s selecting by bit s of the column index.
 *   in   : device, [n][2][L][N] NTT form, canonical residues (the RowSel
 *          output of one query is such a list with n = D1).
 *   out  : device; pir_coltor_stage: [ceil(n/2)][2][L][N], pir_coltor:
 *          [2][L][N]; NTT form; must not overlap in.
 *   ell, w : 1 <= ell <= 16, 1 <= w <= 32, ell * w >= the bit length of Q
 *          (ell = 5, w = 18 for three primes below 2^29).
 *   workspace : device, >= pir_coltor_workspace_bytes(ctx, n, ell) bytes,
 *          16-byte aligned; the part the call uses (its first
 *          pir_coltor_workspace_bytes bytes) must overlap neither in nor out;
 *          contents undefined after the call.
 * The library owns nothing the caller passes; calls are asynchronous on
 * stream.  Errors: PIR_ERR_ARG (NULL/unaligned pointers, n = 0 or ceil(n/2) >= 2^31,
 * ell or w out of range, digits not covering Q, workspace too small,
 * in/out overlap, workspace overlapping in or out), PIR_ERR_CUDA.
 */
uint64_t pir_coltor_workspace_bytes(const pir_ctx *ctx, uint64_t n, uint32_t ell);

int pir_coltor_stage(pir_ctx *ctx, const uint32_t *C, uint32_t ell, uint32_t w,
                     const uint32_t *in, uint64_t n, uint32_t *out,
                     void *workspace, uint64_t workspace_bytes, void *stream);

int pir_coltor(pir_ctx *ctx, const uint32_t *C, uint32_t ell, uint32_t w,
               const uint32_t *in, uint64_t n, uint32_t *out,
               void *workspace, uint64_t workspace_bytes, void *stream);

/*
 * pir_coltor_batch — G independent tournaments of n ciphertexts each (G
 * clients served by one RowSel pass, each with its own RGSW ciphertexts),
 * run stage by stage as one tournament of G * ceil(n/2) pairs, so the small
 * late stages of G tournaments share their launches.  Tournament b is
 * exactly pir_coltor on its own inputs.
 *   C    : device, [G][S][2 ell][2][L][N], S = ceil(log2 n): client b's
 *          stages at b * S * 2 ell * 2 L N words.
 *   in   : device, [G][n][2][L][N] (the RowSel output of G queries,
 *          [B][D1][2][L][N], with G = B and n = D1).
 *   out  : device, [G][2][L][N]; must not overlap in.
 *   workspace : device, >= pir_coltor_batch_workspace_bytes(ctx, n, G,
 *          ell) bytes (0 when G * ceil(n/2) >= 2^31), 16-byte aligned.
 * Errors: as pir_coltor; PIR_ERR_ARG for G = 0 or G * ceil(n/2) >= 2^31.
 * pir_coltor(...) is pir_coltor_batch with G = 1.
 */
uint64_t pir_coltor_batch_workspace_bytes(const pir_ctx *ctx, uint64_t n, uint64_t G, uint32_t ell);

int pir_coltor_batch(pir_ctx *ctx, const uint32_t *C, uint32_t ell, uint32_t w,
                     const uint32_t *in, uint64_t n, uint64_t G, uint32_t *out,
                     void *workspace, uint64_t workspace_bytes, void *stream);

/*
 * ExpandQuery — the expansion tree of Subs operations (GPIR section 2:
 * every depth of the tree is a stage with its own evaluation key, up to
 * log2 N stages; GPIR section 3: Subs operates on the a polynomial only).
 * A ciphertext ct = (c0, c1) decrypts as c0 + c1 s.  With sigma_k(a)(X) =
 * a(X^k) and the gadget decomposition Dcp of pir_coltor:
 *     Subs(ct, k) = (sigma_k(c0), 0) + sum_u NTT(Dcp_u(sigma_k(c1))) . evk[u]
 * where evk[u] is an RLWE encryption of sigma_k(s) g_u under s.  Stage j
 * (k = N/2^j + 1) over M ciphertexts writes 2M:
 *     out[i]     = ct_i + Subs(ct_i, k)
 *     out[i + M] = (ct_i - Subs(ct_i, k)) * X^(-2^j)
 * so after S stages (pir_expand) ciphertext r carries coefficient r of the
 * query's plaintext times 2^S (reading: the SealPIR/OnionPIR tree in this
 * order; the client pre-scales by 2^-S).
 *   evk  : device, [ell][2][L][N] NTT form (one stage's key); for
 *          pir_expand, [stages][ell][2][L][N], stage j's key at j.
 *   in   : device, [M][2][L][N] NTT form; for pir_expand one ciphertext.
 *   out  : device, NTT form; pir_expand_stage: [2M][2][L][N], pir_expand:
 *          [2^stages][2][L][N]; must not overlap the input.
 *   ell, w : as for pir_coltor; j < log2 N; 1 <= stages <= log2 N.
 *   workspace : device, >= pir_expand_workspace_bytes(ctx, M, ell) bytes
 *          (pir_expand: M = 2^(stages-1)), 16-byte aligned; the part the
 *          call uses (its first pir_expand_workspace_bytes bytes) must
 *          overlap neither the input nor out; contents undefined after the
 *          call.
 * Errors: PIR_ERR_ARG (NULL/unaligned pointers, sizes or gadget parameters
 * out of range, workspace too small, input/output overlap, workspace
 * overlapping the input or out), PIR_ERR_CUDA.
 */
uint64_t pir_expand_workspace_bytes(const pir_ctx *ctx, uint64_t M, uint32_t ell);

int pir_expand_stage(pir_ctx *ctx, const uint32_t *evk, uint32_t ell, uint32_t w, uint32_t j,
                     const uint32_t *in, uint64_t M, uint32_t *out,
                     void *workspace, uint64_t workspace_bytes, void *stream);

int pir_expand(pir_ctx *ctx, const uint32_t *evks, uint32_t ell, uint32_t w, uint32_t stages,
               const uint32_t *ct, uint32_t *out,
               void *workspace, uint64_t workspace_bytes, void *stream);

/*
 * pir_expand_batch — G independent expansions (G clients, each with its own
 * query ciphertext and evaluation keys) run stage by stage as one expansion
 * of G * 2^j ciphertexts at stage j, so the small early stages of G
 * expansions share their launches.  Expansion b is exactly pir_expand on its
 * own inputs.
 *   evks : device, [G][stages][ell][2][L][N]: client b's keys at
 *          b * stages * ell * 2 L N words.
 *   ct   : device, [G][2][L][N], one query ciphertext per client.
 *   out  : device, [G][2^stages][2][L][N] (the RowSel query layout
 *          [B][D0][2][L][N] with B = G, D0 = 2^stages); must not overlap ct.
 *   workspace : device, >= pir_expand_workspace_bytes(ctx, G * 2^(stages-1),
 *          ell) bytes, 16-byte aligned.
 * Errors: as pir_expand; PIR_ERR_ARG for G = 0 or G * 2^(stages-1) >= 2^31.
 * pir_expand(...) is pir_expand_batch with G = 1.
 */
int pir_expand_batch(pir_ctx *ctx, const uint32_t *evks, uint32_t ell, uint32_t w, uint32_t stages,
                     const uint32_t *ct, uint64_t G, uint32_t *out,
                     void *workspace, uint64_t workspace_bytes, void *stream);

/*
 * pir_scalar_workspace_bytes — device workspace pir_scalar_scan needs for a
 * C x B query matrix (0 for invalid sizes).
 */
uint64_t pir_scalar_workspace_bytes(uint64_t C, uint32_t B);

/*
 * pir_rgsw_convert — the RGSW ciphertexts of the column tournament from the
 * expanded query (GPIR section 2: the query ciphertext carries both the row
 * and the column index, and the expansion yields the D0 RowSel ciphertexts
 * and RGSW ciphertexts; the pages do not define the conversion, this is a
 * reading).  The client places m g_u (g_u = 2^(w u), the gadget of
 * pir_coltor, pre-scaled by 2^-S for an S-stage expansion) in ell query
 * coefficients, so the expansion yields RLWE'(m) = the ell ciphertexts
 * ct_u = (c0_u, c1_u) of m g_u.  The RGSW ciphertext of m in pir_coltor's
 * row layout is
 *     C[u] = ct_u,    C[ell + u] = (0, c0_u) + sum_v NTT(Dcp_v(c1_u)) . ksk[v]
 * where ksk[v] is an RLWE encryption of s^2 g_v under the client's secret s
 * (a key-switching key); row ell + u decrypts to s (c0_u + c1_u s) = m s g_u.
 *   ksk  : device, [G][ell][2][L][N] NTT form, client b's key at
 *          b * ell * 2 L N words.
 *   in   : device, NTT form, canonical residues: client b's n gadget lists
 *          ([n][ell][2][L][N], e.g. its ceil(log2 D1) column bits) at
 *          b * in_stride ciphertexts; in_stride >= n ell, 0 meaning n ell
 *          (contiguous); a client's expansion output can be passed as is.
 *   out  : device, [G][n][2 ell][2][L][N] NTT form: the RGSW ciphertexts, as
 *          pir_coltor_batch takes them ([G][S][2 ell][2][L][N] with S = n).
 *   ell, w : as for pir_coltor.
 *   workspace : device, >= pir_rgsw_convert_workspace_bytes(ctx, n, G, ell)
 *          bytes (0 when n G ell >= 2^31), 16-byte aligned; the part the
 *          call uses overlaps neither in nor out; contents undefined after.
 * The library owns nothing the caller passes; asynchronous on stream.
 * Errors: PIR_ERR_ARG (NULL/unaligned pointers, n = 0, G = 0, n G ell >=
 * 2^31, in_stride below n ell or the strided input reaching 2^31
 * ciphertexts, ell or w out of range, digits not covering Q, workspace too
 * small, overlaps), PIR_ERR_CUDA.
 */
uint64_t pir_rgsw_convert_workspace_bytes(const pir_ctx *ctx, uint64_t n, uint64_t G, uint32_t ell);

int pir_rgsw_convert(pir_ctx *ctx, const uint32_t *ksk, uint32_t ell, uint32_t w,
                     const uint32_t *in, uint64_t in_stride, uint64_t n, uint64_t G, uint32_t *out,
                     void *workspace, uint64_t workspace_bytes, void *stream);

/*
 * pir_scalar_scan — scalar-HE DB fold (VIPIR 2.5 and 4.1):
 *   out[r][b] = sum_{c<C} db[r][c] * Q[c][b]  mod 2^32
 * with the 4-way byte split of Q (Q = sum_i 2^(8i) Q_i, VIPIR 4.1).
 * 5 <= B <= 64 runs on the tensor cores (exact fp16 digit products, 64
 * queries per pass whatever B is); B <= 4 runs as a GEMV on the CUDA cores
 * (4-way byte dot products, VIPIR's single-query case, bounded by the HBM
 * read of the DB).  Results are identical either way.
 *   db  : device, [R][C] uint8 row-major (bytes are unsigned).
 *   Q   : device, [C][B] uint32.
 *   out : device, [R][B] uint32 (fully overwritten).
 *   workspace : device, >= pir_scalar_workspace_bytes(C, B) bytes, 128-byte
 *               aligned; scratch for the split query, contents undefined
 *               after the call.
 * Requirements: R >= 1, C % 64 == 0, 1 <= B <= 64, R and C <= 2^31.
 * Errors: PIR_ERR_ARG, PIR_ERR_UNSUPPORTED (shape outside the requirements),
 * PIR_ERR_CUDA.
 */
int pir_scalar_scan(pir_ctx *ctx, const uint8_t *db, uint64_t R, uint64_t C,
                    const uint32_t *Q, uint32_t B, uint32_t *out,
                    void *workspace, uint64_t workspace_bytes, void *stream);

/*
 * pir_scalar_scan_noalloc — pir_scalar_scan for callers that cannot allocate
 * device memory at call time (a framework allocator owns the device pool,
 * the caller only receives its input and output buffers, or a cudaMalloc
 * and its implicit synchronisation are not acceptable on the call path).
 * The pages have no counterpart; this is a deployment variant.
 *   Same arguments, layouts, results and errors as pir_scalar_scan, minus the
 *   workspace: the split query is staged in a static device array of
 *   8 MiB that the library reserves on every GPU where it is loaded, so
 *   C <= 16384 (larger C returns PIR_ERR_UNSUPPORTED).  No device memory is
 *   allocated or freed by this call.
 *   The first call on a device looks up the array's device address (one
 *   runtime query, no allocation); make that first call before any stream
 *   capture.  All calls share the array and it keeps the last call's
 *   contents; each call rewrites what it reads, so nothing needs clearing,
 *   but calls that overlap on the GPU (different streams, no ordering
 *   between them) race on it and give undefined results.
 */
int pir_scalar_scan_noalloc(pir_ctx *ctx, const uint8_t *db, uint64_t R, uint64_t C,
                            const uint32_t *Q, uint32_t B, uint32_t *out, void *stream);

/*
 * pir_status — read the context's device status word (PIR_STATUS_* bits set
 * by kernels whose bounded waits ran out) into *flags; clear it if `clear`.
 * Synchronises the context's device.
 */
int pir_status(pir_ctx *ctx, uint32_t *flags, int clear);

/*
 * Failure-path diagnostics (no counterpart in the pages; they exist so that
 * the bounded-wait recovery path can be exercised without faulting a GPU).
 *
 * pir_ctx_set_wait_limit — limit, in nanoseconds, of the ordinary device
 *   waits of the kernels launched with this context from now on (today:
 *   the RowSel scans, pir_rowsel / pir_exppack).  0 restores the default of
 *   2 s; values above 2 s are rejected.  The waits with which a kernel
 *   drains its own bulk copies before it exits keep the full 2 s, so a
 *   kernel never exits with copies into its shared memory outstanding.
 *   Errors: PIR_ERR_ARG (NULL ctx, ns > 2e9).
 * pir_ctx_set_test_hook — PIR_HOOK_WITHHOLD_LAST_COPY makes the first CTA
 *   of either RowSel scan (CUDA cores or tensor cores) never issue the copy
 *   of its last DB chunk or tile: the wait for it runs out, the kernel sets
 *   PIR_STATUS_TIMEOUT, stops computing, drains its other copies and
 *   returns; the results of that launch are unspecified.  PIR_HOOK_NONE
 *   (the default) turns it off.  Host state only: no launch is made.
 *   Errors: PIR_ERR_ARG (NULL ctx, unknown hook).
 */
#define PIR_HOOK_NONE 0u
#define PIR_HOOK_WITHHOLD_LAST_COPY 1u
int pir_ctx_set_wait_limit(pir_ctx *ctx, uint64_t ns);
int pir_ctx_set_test_hook(pir_ctx *ctx, uint32_t hook);

/*
 * pir_server — a query stream over a resident RowSel DB (GPIR section 2,
 * the online phase NTT(query) -> RowSel -> INTT(result), once per query),
 * with host-memory queries and results.  Copies run on their own streams
 * and overlap the scan of the neighbouring queries: query i+1 is copied in
 * and the result of query i-1 is copied out while query i is scanned.  The
 * pages serve queries this way but do not specify the mechanism; this is
 * the host runtime around the three calls.
 *
 * pir_server_create: device buffers for two queries in flight (2 x query,
 *   2 x result, one NTT-domain query and result, the RowSel workspace:
 *   about 3 x (query + result) bytes), three non-blocking streams, events.
 *   db must stay valid and unchanged while the server exists; ctx must
 *   outlive it.  Errors: PIR_ERR_ARG, PIR_ERR_CUDA, PIR_ERR_ALLOC.
 * pir_server_destroy: waits for all submitted work, frees everything.
 * pir_server_submit: enqueues one query; returns at once with its ticket
 *   (0, 1, 2, ... in submission order).
 *     host_query  : [B][D0][2][L][N] coefficient-form residues (as the
 *                   input of pir_ntt_fwd); must stay unchanged until the
 *                   query's result has arrived (pir_server_wait).
 *     host_result : [B][D1][2][L][N] coefficient-form results; written by
 *                   the time pir_server_wait(ticket) returns; must not be
 *                   reused by a later submit before then.
 *   Both should be page-locked (cudaHostAlloc / cudaHostRegister); pageable
 *   memory works but its copies do not overlap.  The result slot of ticket
 *   t is reused by ticket t + 2, so at most two results are in flight per
 *   pair of host buffers the caller alternates.
 * pir_server_wait: blocks until the result of `ticket` (and of every
 *   earlier ticket) is in host memory; PIR_ERR_CUDA if a kernel reported a
 *   device-side timeout (pir_status) or CUDA failed; PIR_ERR_ARG for a
 *   ticket not yet submitted.
 * pir_server_mark / pir_server_elapsed_ms: device-clock timing of a stretch
 *   of the stream: mark(0) records a start event on the copy-in stream
 *   (before the next submitted query's copy), mark(1) an end event on the
 *   copy-out stream (after the last submitted result's copy); elapsed_ms
 *   waits for the end event and returns the time between them.
 */
typedef struct pir_server pir_server;
int pir_server_create(pir_server **srv, pir_ctx *ctx, const uint32_t *db, uint32_t D0, uint32_t D1,
                      uint32_t B);
void pir_server_destroy(pir_server *srv);
int pir_server_submit(pir_server *srv, const uint32_t *host_query, uint32_t *host_result,
                      uint64_t *ticket);
int pir_server_wait(pir_server *srv, uint64_t ticket);
int pir_server_mark(pir_server *srv, int which);
int pir_server_elapsed_ms(pir_server *srv, float *ms);

/* pir_strerror — static description of a return code. */
const char *pir_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* PIR_H */
