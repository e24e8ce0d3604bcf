/*
 * oracle.c -- plain, slow, fp64 CPU oracle for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or load this
 * file; only the tests, the smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no code, header or constant with the CUDA library.
 *
 * What it computes (the plain definition that the tiled GPU method reaches exactly,
 * up to rounding order):
 *
 *   "FlashAttention principles and engineering practice", section 2.1 (memory access):
 *   the standard implementation forms attn = (q k^T) * scale, applies softmax over the
 *   last dimension and multiplies by v.  Per (b,h) head, with Q of shape [Lq,D] and K, V of
 *   shape [Lk,D]:
 *
 *     S   = scale * Q K^T                      (S_ij = -inf for j > i + Lk - Lq when causal)
 *     m_i = max_j S_ij
 *     P   = exp(S - m) / rowsum(exp(S - m))    (materialised, fp64)
 *     O   = P V
 *     LSE_i = m_i + ln sum_j exp(S_ij - m_i)
 *
 *   "FlashAttention data-flow optimisation: MI50 memory and bandwidth bottlenecks",
 *   section 2.2, third layer (gradient re-computation): only the per-row softmax
 *   statistics are kept for the backward pass.  The backward formulas are not printed on
 *   the pages; they are the textbook softmax-Jacobian derivation:
 *
 *     dV = P^T dO
 *     dP = dO V^T
 *     Delta_i = sum_j P_ij dP_ij                (equals sum_d dO_id O_id)
 *     dS = P o (dP - Delta 1^T)
 *     dQ = scale * dS K
 *     dK = scale * dS^T Q
 *
 * Queries and keys may differ in length (Lq != Lk: a block of queries attending to a longer
 * or shorter key sequence, as the flash_attn_func interface allows, "FlashAttention data-flow
 * optimisation", section 4.1, step 3).  The pages do not say how the causal mask lines up
 * then; the reading taken here is that the queries are the LAST Lq positions of the sequence
 * whose keys are given (a block of new tokens after a cache of earlier ones), so query i sits
 * at position i + Lk - Lq and sees key j iff j <= i + Lk - Lq.  For Lq = Lk this is the usual
 * j <= i.  When Lq > Lk the first Lq - Lk query rows see no key at all: their softmax is over
 * an empty set, and the oracle gives them O = 0, LSE = -inf (the log of an empty sum) and
 * dQ = 0; they contribute nothing to dK and dV.
 *
 * Masked entries have P_ij = exp(-inf) = 0 exactly, so they are simply not visited: every
 * sum below runs over the visible keys j < n_i, n_i = clamp(i + 1 + Lk - Lq, 0, Lk) (causal)
 * or Lk.  Rows of S and P are materialised one row block at a time; a block holds every row
 * of the head whenever R*Lk doubles fit the block budget, so for test sizes the whole
 * Lq x Lk matrix is materialised at once.
 *
 * Dropout on P ("FlashAttention data-flow optimisation", section 4.1, step 3: the dropout_p
 * argument of flash_attn_func).  With probability p each entry of P is dropped and the kept ones
 * are scaled by 1/(1-p): O = (P o Z) V with Z_ij in {0, 1/(1-p)}; the LSE is that of P itself.
 * The backward then has dV = (P o Z)^T dO and dP = (dO V^T) o Z, with Delta and dS as above
 * (Delta_i = sum_j P_ij dP_ij still equals sum_d dO_id O_id).  Which entries are dropped is
 * decided by a counter-based generator, Philox-4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw,
 * "Parallel random numbers: as easy as 1, 2, 3", SC 2011), written out below from that
 * definition: entry (bh, i, j) of head bh = b*H + h reads word j % 4 of the block for counter
 * (j / 4, i, bh, 0) under the key (seed low 32 bits, seed high 32 bits), and is dropped iff that
 * word is below floor(p * 2^32).  p = 0 keeps every entry.
 *
 * Layout: every tensor is contiguous [B,H,L,D] (L = Lq for Q, O, dO, dQ and Lk for K, V,
 * dK, dV; LSE, Delta: [B,H,Lq]) in fp64.
 * Parallelism: OpenMP over rows (and over key columns for dK/dV) inside one head.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_NO_MEMORY 2

/* Default cap on doubles held by one materialised block of S/P (2^25 = 256 MiB). */
#define ORACLE_DEFAULT_BLOCK_DOUBLES (1L << 25)

/* Philox-4x32-10: ten rounds of the round function on the 4-word counter, the 2-word key
 * advanced by the Weyl constants between rounds. */
void oracle_philox4x32_10(const unsigned int ctr_in[4], const unsigned int key_in[2],
                          unsigned int out[4]) {
    const unsigned long long M0 = 0xD2511F53ull, M1 = 0xCD9E8D57ull;
    const unsigned int W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    unsigned int c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    unsigned int k0 = key_in[0], k1 = key_in[1];
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += W0;
            k1 += W1;
        }
        const unsigned long long p0 = M0 * (unsigned long long)c0;
        const unsigned long long p1 = M1 * (unsigned long long)c2;
        const unsigned int hi0 = (unsigned int)(p0 >> 32), lo0 = (unsigned int)p0;
        const unsigned int hi1 = (unsigned int)(p1 >> 32), lo1 = (unsigned int)p1;
        const unsigned int n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

/* Dropout parameters: no dropout when p_drop == 0. */
typedef struct {
    double p;                /* drop probability in [0, 1) */
    unsigned int threshold;  /* floor(p * 2^32): an entry is dropped iff its word is below it */
    unsigned int key[2];     /* the seed */
} dropout_t;

static dropout_t make_dropout(double p, unsigned long long seed) {
    dropout_t d;
    d.p = p;
    d.threshold = (unsigned int)floor(p * 4294967296.0);
    d.key[0] = (unsigned int)(seed & 0xffffffffull);
    d.key[1] = (unsigned int)(seed >> 32);
    return d;
}

/* The factor Z_ij of entry (bh, i, j): 0 if dropped, 1/(1-p) if kept (1 without dropout). */
static double dropout_factor(const dropout_t* d, long bh, long i, long j) {
    if (d->threshold == 0u) return 1.0;
    const unsigned int ctr[4] = {(unsigned int)(j >> 2), (unsigned int)i, (unsigned int)bh, 0u};
    unsigned int w[4];
    oracle_philox4x32_10(ctr, d->key, w);
    return w[j & 3] < d->threshold ? 0.0 : 1.0 / (1.0 - d->p);
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Keys visible to query row i: all Lk, or (causal) those at positions <= i + Lk - Lq. */
static long visible_keys(long i, long Lq, long Lk, int causal) {
    if (!causal) return Lk;
    long n = i + 1 + (Lk - Lq);
    if (n < 0) n = 0;
    if (n > Lk) n = Lk;
    return n;
}

/* Row i of S (scaled logits), written into s[0..n), and returns n. */
static long logits_row(const double* Q, const double* K, long i, long Lq, long Lk, long D,
                       double scale, int causal, double* s) {
    long n = visible_keys(i, Lq, Lk, causal);
    const double* q = Q + i * D;
    for (long j = 0; j < n; ++j) {
        const double* k = K + j * D;
        double dot = 0.0;
        for (long d = 0; d < D; ++d) dot += q[d] * k[d];
        s[j] = scale * dot;
    }
    return n;
}

/* Turns s[0..n) into the softmax row P in place; returns LSE = m + ln(sum exp(s - m)), or
 * -inf for an empty row (n = 0). */
static double softmax_row(double* s, long n) {
    if (n == 0) return -INFINITY;
    double m = -INFINITY;
    for (long j = 0; j < n; ++j)
        if (s[j] > m) m = s[j];
    double sum = 0.0;
    for (long j = 0; j < n; ++j) {
        s[j] = exp(s[j] - m);
        sum += s[j];
    }
    for (long j = 0; j < n; ++j) s[j] /= sum;
    return m + log(sum);
}

/* Rows of S/P materialised at once: as many rows of `row_len` doubles as fit the budget, at
 * least one and at most `rows` (the number of query rows; never 0, so the row loops advance). */
static long block_rows(long row_len, long rows, long block_doubles) {
    if (block_doubles <= 0) block_doubles = ORACLE_DEFAULT_BLOCK_DOUBLES;
    long r = block_doubles / (row_len > 0 ? row_len : 1);
    if (r > rows) r = rows;
    if (r < 1) r = 1;
    return r;
}

/* Forward pass for one head (bh = b*H + h for the dropout counter): Q, O [Lq,D], K, V [Lk,D],
 * lse [Lq]. */
static int fwd_head(const double* Q, const double* K, const double* V, double* O, double* lse,
                    long Lq, long Lk, long D, double scale, int causal, long block_doubles,
                    const dropout_t* drop, long bh) {
    long R = block_rows(Lk, Lq, block_doubles);
    double* P = (double*)malloc(sizeof(double) * (size_t)R * (size_t)(Lk > 0 ? Lk : 1));
    if (!P) return ORACLE_NO_MEMORY;
    for (long i0 = 0; i0 < Lq; i0 += R) {
        long i1 = i0 + R < Lq ? i0 + R : Lq;
#pragma omp parallel for schedule(dynamic, 4)
        for (long i = i0; i < i1; ++i) {
            double* p = P + (i - i0) * Lk;
            long n = logits_row(Q, K, i, Lq, Lk, D, scale, causal, p);
            lse[i] = softmax_row(p, n);
            double* o = O + i * D;
            for (long d = 0; d < D; ++d) o[d] = 0.0;
            for (long j = 0; j < n; ++j) {
                const double* v = V + j * D;
                const double pz = p[j] * dropout_factor(drop, bh, i, j);
                for (long d = 0; d < D; ++d) o[d] += pz * v[d];
            }
        }
    }
    free(P);
    return ORACLE_OK;
}

/* Backward pass for one head (P recomputed from the definition, nothing cached):
 * Q, dO, dQ [Lq,D], K, V, dK, dV [Lk,D], delta [Lq]. */
static int bwd_head(const double* Q, const double* K, const double* V, const double* dO,
                    double* dQ, double* dK, double* dV, double* delta, long Lq, long Lk, long D,
                    double scale, int causal, long block_doubles, const dropout_t* drop,
                    long bh) {
    long R = block_rows(Lk, Lq, block_doubles / 2);
    size_t row = (size_t)(Lk > 0 ? Lk : 1);
    double* P = (double*)malloc(sizeof(double) * (size_t)R * row);
    double* dS = (double*)malloc(sizeof(double) * (size_t)R * row);
    if (!P || !dS) {
        free(P);
        free(dS);
        return ORACLE_NO_MEMORY;
    }
    memset(dK, 0, sizeof(double) * (size_t)Lk * (size_t)D);
    memset(dV, 0, sizeof(double) * (size_t)Lk * (size_t)D);
    for (long i0 = 0; i0 < Lq; i0 += R) {
        long i1 = i0 + R < Lq ? i0 + R : Lq;
        /* Rows: P, dP, Delta, dS and dQ. */
#pragma omp parallel for schedule(dynamic, 4)
        for (long i = i0; i < i1; ++i) {
            double* p = P + (i - i0) * Lk;
            double* ds = dS + (i - i0) * Lk;
            long n = logits_row(Q, K, i, Lq, Lk, D, scale, causal, p);
            (void)softmax_row(p, n);
            const double* g = dO + i * D;
            double dlt = 0.0;
            for (long j = 0; j < n; ++j) {
                const double* v = V + j * D;
                double dp = 0.0;
                for (long d = 0; d < D; ++d) dp += g[d] * v[d];
                dp *= dropout_factor(drop, bh, i, j); /* dP = (dO V^T) o Z */
                ds[j] = dp; /* dP_ij for now */
                dlt += p[j] * dp;
            }
            delta[i] = dlt;
            for (long j = 0; j < n; ++j) ds[j] = p[j] * (ds[j] - dlt);
            double* dq = dQ + i * D;
            for (long d = 0; d < D; ++d) dq[d] = 0.0;
            for (long j = 0; j < n; ++j) {
                const double* k = K + j * D;
                for (long d = 0; d < D; ++d) dq[d] += ds[j] * k[d];
            }
            for (long d = 0; d < D; ++d) dq[d] *= scale;
        }
        /* Columns: dV_j += sum_i P_ij dO_i and dK_j += scale * sum_i dS_ij Q_i over this block. */
#pragma omp parallel for schedule(dynamic, 4)
        for (long j = 0; j < Lk; ++j) {
            double* dv = dV + j * D;
            double* dk = dK + j * D;
            for (long i = i0; i < i1; ++i) {
                if (j >= visible_keys(i, Lq, Lk, causal)) continue; /* P_ij = 0 and dS_ij = 0 */
                double pij = P[(i - i0) * Lk + j] * dropout_factor(drop, bh, i, j); /* P o Z */
                double dsij = dS[(i - i0) * Lk + j];
                const double* g = dO + i * D;
                const double* q = Q + i * D;
                for (long d = 0; d < D; ++d) {
                    dv[d] += pij * g[d];
                    dk[d] += scale * dsij * q[d];
                }
            }
        }
    }
    free(P);
    free(dS);
    return ORACLE_OK;
}

static int bad_shape(long B, long H, long Lq, long Lk, long D) {
    return B < 0 || H < 0 || Lq < 0 || Lk < 0 || D < 1;
}

/*
 * Forward over all heads.  q: [B,H,Lq,D]; k, v: [B,H,Lk,D]; o: [B,H,Lq,D]; lse: [B,H,Lq].
 * block_doubles caps the doubles of one materialised S/P block (<= 0: default).
 */
int oracle_fwd_f64(const double* q, const double* k, const double* v, double* o, double* lse,
                   long B, long H, long Lq, long Lk, long D, double scale, int causal,
                   long block_doubles, double p_drop, unsigned long long seed) {
    if (bad_shape(B, H, Lq, Lk, D) || !(p_drop >= 0.0 && p_drop < 1.0)) return ORACLE_BAD_ARG;
    const dropout_t drop = make_dropout(p_drop, seed);
    for (long bh = 0; bh < B * H; ++bh) {
        size_t oq = (size_t)bh * (size_t)Lq * (size_t)D;
        size_t ok = (size_t)bh * (size_t)Lk * (size_t)D;
        int rc = fwd_head(q + oq, k + ok, v + ok, o + oq, lse + (size_t)bh * (size_t)Lq, Lq, Lk, D,
                          scale, causal, block_doubles, &drop, bh);
        if (rc) return rc;
    }
    return ORACLE_OK;
}

/*
 * Backward over all heads.  Inputs q, dO: [B,H,Lq,D], k, v: [B,H,Lk,D]; outputs dq: [B,H,Lq,D],
 * dk, dv: [B,H,Lk,D] and delta: [B,H,Lq] (Delta_i = sum_j P_ij dP_ij).
 */
int oracle_bwd_f64(const double* q, const double* k, const double* v, const double* dO,
                   double* dq, double* dk, double* dv, double* delta, long B, long H, long Lq,
                   long Lk, long D, double scale, int causal, long block_doubles, double p_drop,
                   unsigned long long seed) {
    if (bad_shape(B, H, Lq, Lk, D) || !(p_drop >= 0.0 && p_drop < 1.0)) return ORACLE_BAD_ARG;
    const dropout_t drop = make_dropout(p_drop, seed);
    for (long bh = 0; bh < B * H; ++bh) {
        size_t oq = (size_t)bh * (size_t)Lq * (size_t)D;
        size_t ok = (size_t)bh * (size_t)Lk * (size_t)D;
        int rc = bwd_head(q + oq, k + ok, v + ok, dO + oq, dq + oq, dk + ok, dv + ok,
                          delta + (size_t)bh * (size_t)Lq, Lq, Lk, D, scale, causal,
                          block_doubles, &drop, bh);
        if (rc) return rc;
    }
    return ORACLE_OK;
}

/* The full probability matrix P [Lq,Lk] of one head (masked entries are 0; a row that sees
 * no key is all zeros). */
int oracle_probs_f64(const double* q, const double* k, double* p, long Lq, long Lk, long D,
                     double scale, int causal) {
    if (bad_shape(1, 1, Lq, Lk, D)) return ORACLE_BAD_ARG;
    for (long i = 0; i < Lq; ++i) {
        double* row = p + i * Lk;
        long n = logits_row(q, k, i, Lq, Lk, D, scale, causal, row);
        (void)softmax_row(row, n);
        for (long j = n; j < Lk; ++j) row[j] = 0.0;
    }
    return ORACLE_OK;
}

/*
 * Decode over a paged key/value cache ("FlashAttention principles and engineering practice",
 * section 4.2: served through vLLM with PagedAttention and block_size 16).  Each sequence b has
 * one new query row q[b, h, :] per head and a cache of seq_lens[b] tokens stored in pages of
 * `page` tokens: token t of sequence b lives in physical page block_tables[b*max_pages + t/page]
 * at slot t % page, head h, i.e. at k_cache[((phys*H + h)*page + t%page)*D ...].  The query is the
 * newest position, so it sees every cached token: per (b, h) this is the plain definition with
 * one query row and the sequence's tokens gathered in order as keys and values.  A sequence with
 * no cached token has O = 0 and LSE = -inf.  Returns ORACLE_BAD_ARG for a page index or length
 * out of range.
 *   q, o: [B, H, D]; lse: [B, H]; k_cache, v_cache: [num_pages, H, page, D];
 *   block_tables: [B, max_pages]; seq_lens: [B].
 */
int oracle_decode_paged_f64(const double* q, const double* k_cache, const double* v_cache,
                            const int* block_tables, const int* seq_lens, double* o, double* lse,
                            long B, long H, long D, long num_pages, long page, long max_pages,
                            double scale) {
    if (B < 0 || H < 0 || D < 1 || num_pages < 0 || page < 1 || max_pages < 0)
        return ORACLE_BAD_ARG;
    for (long b = 0; b < B; ++b) {
        const long n = seq_lens[b];
        if (n < 0 || n > max_pages * page) return ORACLE_BAD_ARG;
        for (long t = 0; t < n; t += page) {
            const long phys = block_tables[b * max_pages + t / page];
            if (phys < 0 || phys >= num_pages) return ORACLE_BAD_ARG;
        }
        double* kb = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * (size_t)D);
        double* vb = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * (size_t)D);
        if (!kb || !vb) {
            free(kb);
            free(vb);
            return ORACLE_NO_MEMORY;
        }
        for (long h = 0; h < H; ++h) {
            /* Gather the sequence's keys and values of head h in token order. */
            for (long t = 0; t < n; ++t) {
                const long phys = block_tables[b * max_pages + t / page];
                const size_t src = ((size_t)(phys * H + h) * (size_t)page + (size_t)(t % page)) *
                                   (size_t)D;
                memcpy(kb + t * D, k_cache + src, sizeof(double) * (size_t)D);
                memcpy(vb + t * D, v_cache + src, sizeof(double) * (size_t)D);
            }
            const size_t qo = (size_t)(b * H + h) * (size_t)D;
            /* One query row that sees all n keys (non-causal, Lq = 1). */
            const dropout_t none = make_dropout(0.0, 0ull);
            int rc = fwd_head(q + qo, kb, vb, o + qo, lse + b * H + h, 1, n, D, scale, 0, 0, &none,
                              b * H + h);
            if (rc) {
                free(kb);
                free(vb);
                return rc;
            }
        }
        free(kb);
        free(vb);
    }
    return ORACLE_OK;
}
