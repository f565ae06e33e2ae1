/*
 * oracle.c -- plain, slow, obviously-correct CPU oracle for the batched
 * RNS negacyclic NTT and the NTT-domain kernels built on it.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; only the tests, the package's smoke check and the bench's
 * CPU-baseline leg do.  It shares no code, header, table or constant with the
 * CUDA library: every modular operation here is an unsigned __int128 product
 * followed by the C '%' operator -- no Montgomery, Shoup or Barrett forms.
 *
 * Sources (the web pages this build follows):
 *  [FH] FHElium, "Eager, Compile, and native execution":
 *       section "Shared implementation and native path" (RNS tensor
 *       [*batch, limb, coefficient], parameter column j describes limb j),
 *       section "CUDA execution" (coefficient-wise Montgomery multiplication,
 *       mixed-radix decomposition and basis extension, NTT families, Galois
 *       automorphisms, key-switch multiply-accumulate), table "Native
 *       operator families".
 *  [KE] kestrel-llm data-flow overview (lpnh.cn news 2512365):
 *       section 3 (vllm_ntt.c: negacyclic NTT and polynomial multiplication;
 *       vllm_ckks.c: mul / relin / rotate; the "key point" paragraph: the NTT
 *       is proved against the textbook O(n^2) product), section 4.2
 *       (modraise by Garner extension; coeff_to_slot = Galois rotation +
 *       key-switch), section 5 (8 ciphertexts = 4 tokens x 2 components).
 *
 * The pages fix no root of unity, output order or basis-extension formula.
 * The readings taken here (and repeated where they are used) are:
 *  - primes: q < 2^bits, q = 1 (mod 2n), scanned downward from the largest;
 *  - psi: the smallest primitive 2n-th root of unity modulo q;
 *  - forward NTT: ahat[i] = sum_j a[j] * psi^((2*brv(i)+1)*j), i.e. the
 *    evaluation of a(X) at the n roots of X^n+1, stored in bit-reversed order;
 *  - inverse NTT: the exact inverse, including the 1/n factor;
 *  - ModUp: exact mixed-radix (Garner) CRT of a digit, then residues of that
 *    integer modulo every prime of the extended basis; the approximate
 *    variant keeps the CRT sum's overflow e Q (0 <= e < digit size);
 *  - modraise: the exact Garner extension from the first primes of the chain
 *    to the whole chain, with the value taken in [0, Q_low) (no centring);
 *  - hoisted rotations: one ModUp and NTT of the digits, then per Galois
 *    element the automorphism of the extended digits and the inner product.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <pthread.h>

typedef unsigned __int128 u128;

/* ------------------------------------------------------------------------ */
/* Scalar modular arithmetic (definitions, nothing clever).                  */
/* ------------------------------------------------------------------------ */

static uint64_t mulmod(uint64_t a, uint64_t b, uint64_t q) {
    return (uint64_t)(((u128)a * (u128)b) % q);
}

static uint64_t addmod(uint64_t a, uint64_t b, uint64_t q) {
    return (uint64_t)(((u128)a + (u128)b) % q);
}

static uint64_t submod(uint64_t a, uint64_t b, uint64_t q) {
    /* a - b mod q for a, b in [0, q) */
    return (uint64_t)(((u128)a + (u128)q - (u128)(b % q)) % q);
}

static uint64_t powmod(uint64_t b, uint64_t e, uint64_t q) {
    uint64_t r = 1 % q;
    b %= q;
    while (e) {
        if (e & 1) r = mulmod(r, b, q);
        b = mulmod(b, b, q);
        e >>= 1;
    }
    return r;
}

/* inverse by Fermat's little theorem; q must be prime and a != 0 mod q */
static uint64_t invmod(uint64_t a, uint64_t q) {
    return powmod(a % q, q - 2, q);
}

uint64_t oracle_mulmod(uint64_t a, uint64_t b, uint64_t q) { return mulmod(a, b, q); }
uint64_t oracle_powmod(uint64_t b, uint64_t e, uint64_t q) { return powmod(b, e, q); }

/* ------------------------------------------------------------------------ */
/* Primes and roots of unity.                                                */
/* ------------------------------------------------------------------------ */

/* Deterministic Miller-Rabin for 64-bit inputs: the first twelve primes as
 * witnesses are enough for every n < 3.18e23. */
int oracle_is_prime(uint64_t n) {
    static const uint64_t small[12] = {2, 3, 5, 7, 11, 13, 17, 19, 23, 29, 31, 37};
    if (n < 2) return 0;
    for (int i = 0; i < 12; i++) {
        if (n == small[i]) return 1;
        if (n % small[i] == 0) return 0;
    }
    uint64_t d = n - 1;
    int s = 0;
    while ((d & 1) == 0) { d >>= 1; s++; }
    for (int i = 0; i < 12; i++) {
        uint64_t x = powmod(small[i], d, n);
        if (x == 1 || x == n - 1) continue;
        int composite = 1;
        for (int r = 1; r < s; r++) {
            x = mulmod(x, x, n);
            if (x == n - 1) { composite = 0; break; }
        }
        if (composite) return 0;
    }
    return 1;
}

/* The `count` largest primes q < 2^bits with q = 1 (mod m), in descending
 * order, starting below `below` (pass 0 to start at 2^bits).  Returns the
 * number found (count unless the range runs out). */
int oracle_primes(uint64_t m, int bits, int count, uint64_t below, uint64_t *out) {
    uint64_t top = (bits >= 64) ? UINT64_MAX : ((uint64_t)1 << bits);
    if (below == 0 || below > top) below = top;
    /* largest value < below that is = 1 mod m */
    uint64_t c = below - 1;
    c -= (c % m + m - 1) % m;   /* now c = 1 mod m, c <= below - 1 */
    int found = 0;
    while (found < count && c > m) {
        if (oracle_is_prime(c)) out[found++] = c;
        c -= m;
    }
    return found;
}

/* Smallest primitive m-th root of unity mod q, m a power of two dividing
 * q - 1.  A primitive m-th root is g0^t for odd t, where g0 = x^((q-1)/m) and
 * x is any quadratic non-residue; this takes the least such value. */
uint64_t oracle_psi(uint64_t q, uint64_t m) {
    uint64_t x = 2;
    while (powmod(x, (q - 1) / 2, q) != q - 1) x++;
    uint64_t g0 = powmod(x, (q - 1) / m, q);
    uint64_t g2 = mulmod(g0, g0, q);
    uint64_t cur = g0, best = g0;
    for (uint64_t t = 1; t < m; t += 2) {   /* cur = g0^t */
        if (cur < best) best = cur;
        cur = mulmod(cur, g2, q);
    }
    return best;
}

/* ------------------------------------------------------------------------ */
/* Index helpers.                                                            */
/* ------------------------------------------------------------------------ */

static uint64_t brv(uint64_t x, int bits) {
    uint64_t r = 0;
    for (int i = 0; i < bits; i++) { r = (r << 1) | (x & 1); x >>= 1; }
    return r;
}

uint64_t oracle_brv(uint64_t x, int bits) { return brv(x, bits); }

/* ------------------------------------------------------------------------ */
/* NTT by definition, O(n^2).                                                */
/* ------------------------------------------------------------------------ */

/* ahat[i] = sum_j a[j] * psi^((2 brv(i) + 1) j) mod q */
void oracle_ntt_direct(const uint64_t *a, uint64_t *out, int log_n, uint64_t q, uint64_t psi) {
    uint64_t n = (uint64_t)1 << log_n;
    for (uint64_t i = 0; i < n; i++) {
        uint64_t root = powmod(psi, 2 * brv(i, log_n) + 1, q);
        uint64_t acc = 0, pw = 1;
        for (uint64_t j = 0; j < n; j++) {
            acc = addmod(acc, mulmod(a[j], pw, q), q);
            pw = mulmod(pw, root, q);
        }
        out[i] = acc;
    }
}

/* a[j] = n^-1 * sum_i ahat[i] * psi^(-(2 brv(i) + 1) j) mod q */
void oracle_intt_direct(const uint64_t *ahat, uint64_t *out, int log_n, uint64_t q, uint64_t psi) {
    uint64_t n = (uint64_t)1 << log_n;
    uint64_t psi_inv = invmod(psi, q), n_inv = invmod(n % q, q);
    for (uint64_t j = 0; j < n; j++) {
        uint64_t acc = 0;
        for (uint64_t i = 0; i < n; i++) {
            uint64_t e = ((2 * brv(i, log_n) + 1) * j) % (2 * n);
            acc = addmod(acc, mulmod(ahat[i], powmod(psi_inv, e, q), q), q);
        }
        out[j] = mulmod(acc, n_inv, q);
    }
}

/* ------------------------------------------------------------------------ */
/* NTT, O(n log n): twist by psi^j, textbook cyclic DFT with omega = psi^2   */
/* (iterative radix-2 with a bit-reversal permutation of the input), then    */
/* the bit-reversed output order of the definition above.  Written for       */
/* readability, not speed.                                                   */
/* ------------------------------------------------------------------------ */

static void bit_reverse_permute(uint64_t *a, int log_n) {
    uint64_t n = (uint64_t)1 << log_n;
    for (uint64_t i = 0; i < n; i++) {
        uint64_t j = brv(i, log_n);
        if (j > i) { uint64_t t = a[i]; a[i] = a[j]; a[j] = t; }
    }
}

/* In place cyclic DFT: A[k] = sum_j a[j] w^(jk), natural order in and out. */
static void cyclic_dft(uint64_t *a, int log_n, uint64_t q, uint64_t w) {
    uint64_t n = (uint64_t)1 << log_n;
    bit_reverse_permute(a, log_n);
    for (uint64_t len = 2; len <= n; len <<= 1) {
        uint64_t wl = powmod(w, n / len, q);   /* primitive len-th root */
        for (uint64_t start = 0; start < n; start += len) {
            uint64_t f = 1;
            for (uint64_t k = 0; k < len / 2; k++) {
                uint64_t u = a[start + k];
                uint64_t v = mulmod(a[start + k + len / 2], f, q);
                a[start + k] = addmod(u, v, q);
                a[start + k + len / 2] = submod(u, v, q);
                f = mulmod(f, wl, q);
            }
        }
    }
}

void oracle_ntt(uint64_t *a, int log_n, uint64_t q, uint64_t psi) {
    uint64_t n = (uint64_t)1 << log_n;
    uint64_t pw = 1;
    for (uint64_t j = 0; j < n; j++) { a[j] = mulmod(a[j] % q, pw, q); pw = mulmod(pw, psi, q); }
    cyclic_dft(a, log_n, q, mulmod(psi, psi, q));
    /* A[k] is the value at psi^(2k+1); the definition stores it at brv(k) */
    bit_reverse_permute(a, log_n);
}

void oracle_intt(uint64_t *a, int log_n, uint64_t q, uint64_t psi) {
    uint64_t n = (uint64_t)1 << log_n;
    uint64_t psi_inv = invmod(psi, q);
    bit_reverse_permute(a, log_n);             /* back to natural k order */
    cyclic_dft(a, log_n, q, mulmod(psi_inv, psi_inv, q));
    uint64_t n_inv = invmod(n % q, q), pw = n_inv;
    for (uint64_t j = 0; j < n; j++) { a[j] = mulmod(a[j], pw, q); pw = mulmod(pw, psi_inv, q); }
}

/* ------------------------------------------------------------------------ */
/* Negacyclic product by definition (schoolbook, O(n^2)).                    */
/* c_k = sum_{i+j=k} a_i b_j - sum_{i+j=k+n} a_i b_j  mod q                  */
/* ------------------------------------------------------------------------ */

void oracle_negacyclic_mul(const uint64_t *a, const uint64_t *b, uint64_t *c, int log_n, uint64_t q) {
    uint64_t n = (uint64_t)1 << log_n;
    for (uint64_t k = 0; k < n; k++) c[k] = 0;
    for (uint64_t i = 0; i < n; i++) {
        for (uint64_t j = 0; j < n; j++) {
            uint64_t p = mulmod(a[i], b[j], q);
            if (i + j < n) c[i + j] = addmod(c[i + j], p, q);
            else c[i + j - n] = submod(c[i + j - n], p, q);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Galois automorphism sigma_k: a(X) -> a(X^k), k odd in [1, 2n).            */
/* ------------------------------------------------------------------------ */

/* Coefficient domain: X^t -> X^(t k mod 2n) = -X^(t k mod 2n - n) when the
 * exponent is >= n, because X^n = -1. */
void oracle_automorph_coeff(const uint64_t *a, uint64_t *out, int log_n, uint64_t q, uint64_t k) {
    uint64_t n = (uint64_t)1 << log_n;
    for (uint64_t t = 0; t < n; t++) {
        uint64_t s = (t * k) % (2 * n);
        if (s < n) out[s] = a[t] % q;
        else out[s - n] = (q - a[t] % q) % q;
    }
}

/* NTT domain, by definition: NTT(sigma_k(INTT(x))).  Uses no index formula. */
void oracle_automorph_ntt(const uint64_t *ahat, uint64_t *out, int log_n, uint64_t q, uint64_t psi, uint64_t k) {
    uint64_t n = (uint64_t)1 << log_n;
    uint64_t *tmp = (uint64_t *)malloc(n * sizeof(uint64_t));
    memcpy(tmp, ahat, n * sizeof(uint64_t));
    oracle_intt(tmp, log_n, q, psi);
    oracle_automorph_coeff(tmp, out, log_n, q, k);
    oracle_ntt(out, log_n, q, psi);
    free(tmp);
}

/* ------------------------------------------------------------------------ */
/* Basis extension of one digit (mixed-radix / Garner), exact.               */
/* ------------------------------------------------------------------------ */

/* For one coefficient: residues x[0..alpha) modulo the digit primes d[0..alpha)
 * define X in [0, D), D = prod d.  Garner's mixed-radix digits v satisfy
 *   X = v0 + v1 d0 + v2 d0 d1 + ... + v_{a-1} d0...d_{a-2},  0 <= v_i < d_i,
 * with v_i = (x_i - (v0 + v1 d0 + ... + v_{i-1} d0..d_{i-2})) / (d0..d_{i-1})
 * taken mod d_i.  Then X mod p = sum_i v_i * (d0..d_{i-1} mod p) mod p. */
static void garner_digits(const uint64_t *x, const uint64_t *d, int alpha, uint64_t *v) {
    for (int i = 0; i < alpha; i++) {
        uint64_t qi = d[i];
        uint64_t partial = 0, radix = 1;   /* both mod qi */
        for (int k = 0; k < i; k++) {
            partial = addmod(partial, mulmod(v[k] % qi, radix, qi), qi);
            radix = mulmod(radix, d[k] % qi, qi);
        }
        v[i] = mulmod(submod(x[i] % qi, partial, qi), invmod(radix, qi), qi);
    }
}

static uint64_t mixed_radix_mod(const uint64_t *v, const uint64_t *d, int alpha, uint64_t p) {
    uint64_t acc = 0, radix = 1 % p;
    for (int i = 0; i < alpha; i++) {
        acc = addmod(acc, mulmod(v[i] % p, radix, p), p);
        radix = mulmod(radix, d[i] % p, p);
    }
    return acc;
}

/* Exact ModUp of one digit for one coefficient.  x: alpha residues; d: the
 * digit primes; targets: nt primes; out: nt residues of X. */
void oracle_modup_coeff(const uint64_t *x, const uint64_t *d, int alpha,
                        const uint64_t *targets, int nt, uint64_t *out) {
    uint64_t v[64];
    garner_digits(x, d, alpha, v);
    for (int t = 0; t < nt; t++) out[t] = mixed_radix_mod(v, d, alpha, targets[t]);
}

/* ------------------------------------------------------------------------ */
/* Approximate (fast) basis conversion.                                      */
/* ------------------------------------------------------------------------ */

/* With Q = q_0 ... q_{S-1} and qhat_j = Q / q_j, the CRT sum
 *   sum_j [x_j * qhat_j^-1]_{q_j} * qhat_j
 * equals X + e Q for an integer 0 <= e < S (each bracket is below q_j, so the
 * sum is below S Q).  Reducing it modulo a target prime p without the
 * correction of e Q is the approximate basis conversion: one product per
 * source limb, then one multiply-accumulate per (source, target) pair,
 * instead of Garner's quadratic digit recursion.  The constants depend only
 * on the bases: qinv[j] = qhat_j^-1 mod q_j and qhat[t][j] = qhat_j mod p_t. */
static void fast_bconv_consts(const uint64_t *src, int S, const uint64_t *dst, int T, uint64_t *qinv,
                              uint64_t *qhat) {
    for (int j = 0; j < S; j++) {
        uint64_t qj = src[j], h = 1 % qj;
        for (int i = 0; i < S; i++)
            if (i != j) h = mulmod(h, src[i] % qj, qj);
        qinv[j] = invmod(h, qj);
    }
    for (int t = 0; t < T; t++) {
        uint64_t p = dst[t];
        for (int j = 0; j < S; j++) {
            uint64_t h = 1 % p;
            for (int i = 0; i < S; i++)
                if (i != j) h = mulmod(h, src[i] % p, p);
            qhat[(long)t * S + j] = h;
        }
    }
}

static void fast_bconv_apply(const uint64_t *x, const uint64_t *src, int S, const uint64_t *dst, int T,
                             const uint64_t *qinv, const uint64_t *qhat, uint64_t *out) {
    uint64_t y[64];
    for (int j = 0; j < S; j++) y[j] = mulmod(x[j] % src[j], qinv[j], src[j]);
    for (int t = 0; t < T; t++) {
        uint64_t p = dst[t], acc = 0;
        for (int j = 0; j < S; j++) acc = addmod(acc, mulmod(y[j] % p, qhat[(long)t * S + j], p), p);
        out[t] = acc;
    }
}

/* One coefficient from basis src[S] to basis dst[T]: exact (Garner, the
 * value X in [0, Q)) or approximate (X + e Q, 0 <= e < S). */
void oracle_bconv_coeff(const uint64_t *x, const uint64_t *src, int S, const uint64_t *dst, int T, int approx,
                        uint64_t *out) {
    if (!approx) {
        oracle_modup_coeff(x, src, S, dst, T, out);
        return;
    }
    uint64_t qinv[64];
    uint64_t *qhat = (uint64_t *)malloc((size_t)T * S * sizeof(uint64_t));
    fast_bconv_consts(src, S, dst, T, qinv, qhat);
    fast_bconv_apply(x, src, S, dst, T, qinv, qhat, out);
    free(qhat);
}

/* ------------------------------------------------------------------------ */
/* Batched drivers over the [batch][L][n] layout, threaded over independent  */
/* (batch, limb) rows only.                                                  */
/* ------------------------------------------------------------------------ */

typedef struct {
    void (*fn)(void *ctx, long unit);
    void *ctx;
    long units;
    long next;
    pthread_mutex_t lock;
} pool_t;

static void *pool_worker(void *arg) {
    pool_t *p = (pool_t *)arg;
    for (;;) {
        pthread_mutex_lock(&p->lock);
        long u = p->next++;
        pthread_mutex_unlock(&p->lock);
        if (u >= p->units) break;
        p->fn(p->ctx, u);
    }
    return NULL;
}

static void run_units(void (*fn)(void *, long), void *ctx, long units, int threads) {
    if (threads <= 1 || units <= 1) {
        for (long u = 0; u < units; u++) fn(ctx, u);
        return;
    }
    if (threads > 256) threads = 256;
    pool_t p;
    p.fn = fn; p.ctx = ctx; p.units = units; p.next = 0;
    pthread_mutex_init(&p.lock, NULL);
    pthread_t tid[256];
    for (int t = 0; t < threads; t++) pthread_create(&tid[t], NULL, pool_worker, &p);
    for (int t = 0; t < threads; t++) pthread_join(tid[t], NULL);
    pthread_mutex_destroy(&p.lock);
}

typedef struct {
    uint64_t *a; const uint64_t *q; const uint64_t *psi; int log_n; int L; int inverse;
} ntt_ctx;

static void ntt_unit(void *c, long u) {
    ntt_ctx *x = (ntt_ctx *)c;
    uint64_t n = (uint64_t)1 << x->log_n;
    int l = (int)(u % x->L);
    if (x->inverse) oracle_intt(x->a + (uint64_t)u * n, x->log_n, x->q[l], x->psi[l]);
    else oracle_ntt(x->a + (uint64_t)u * n, x->log_n, x->q[l], x->psi[l]);
}

/* In-place forward (inverse != 0: inverse) NTT of every row of a[batch][L][n]. */
void oracle_ntt_batch(uint64_t *a, int log_n, int L, int batch, const uint64_t *q,
                      const uint64_t *psi, int inverse, int threads) {
    ntt_ctx c = {a, q, psi, log_n, L, inverse};
    run_units(ntt_unit, &c, (long)batch * L, threads);
}

/* out[b][l][i] = a[b][l][i] * b[b][l][i] mod q_l */
void oracle_mul_batch(const uint64_t *a, const uint64_t *b, uint64_t *out, int log_n, int L,
                      int batch, const uint64_t *q) {
    uint64_t n = (uint64_t)1 << log_n;
    for (long r = 0; r < (long)batch * L; r++) {
        uint64_t ql = q[r % L];
        for (uint64_t i = 0; i < n; i++) out[r * n + i] = mulmod(a[r * n + i], b[r * n + i], ql);
    }
}

/* Ciphertext tensor product in the NTT domain, per batch item:
 *   a = (a0, a1), b = (b0, b1)  ->  d0 = a0 b0, d1 = a0 b1 + a1 b0, d2 = a1 b1.
 * a, b: [batch][2][L][n]; d: [batch][3][L][n]. */
void oracle_tensor_batch(const uint64_t *a, const uint64_t *b, uint64_t *d, int log_n, int L,
                         int batch, const uint64_t *q) {
    uint64_t n = (uint64_t)1 << log_n;
    uint64_t plane = (uint64_t)L * n;
    for (int bi = 0; bi < batch; bi++) {
        const uint64_t *a0 = a + (uint64_t)bi * 2 * plane, *a1 = a0 + plane;
        const uint64_t *b0 = b + (uint64_t)bi * 2 * plane, *b1 = b0 + plane;
        uint64_t *d0 = d + (uint64_t)bi * 3 * plane, *d1 = d0 + plane, *d2 = d1 + plane;
        for (int l = 0; l < L; l++) {
            uint64_t ql = q[l];
            for (uint64_t i = 0; i < n; i++) {
                uint64_t o = (uint64_t)l * n + i;
                d0[o] = mulmod(a0[o], b0[o], ql);
                d1[o] = addmod(mulmod(a0[o], b1[o], ql), mulmod(a1[o], b0[o], ql), ql);
                d2[o] = mulmod(a1[o], b1[o], ql);
            }
        }
    }
}

typedef struct {
    const uint64_t *in; uint64_t *out; const uint64_t *q; const uint64_t *psi;
    int log_n; int L; uint64_t k; int ntt_domain;
} aut_ctx;

static void aut_unit(void *c, long u) {
    aut_ctx *x = (aut_ctx *)c;
    uint64_t n = (uint64_t)1 << x->log_n;
    int l = (int)(u % x->L);
    if (x->ntt_domain)
        oracle_automorph_ntt(x->in + (uint64_t)u * n, x->out + (uint64_t)u * n, x->log_n, x->q[l], x->psi[l], x->k);
    else
        oracle_automorph_coeff(x->in + (uint64_t)u * n, x->out + (uint64_t)u * n, x->log_n, x->q[l], x->k);
}

void oracle_automorph_batch(const uint64_t *in, uint64_t *out, int log_n, int L, int batch,
                            const uint64_t *q, const uint64_t *psi, uint64_t k, int ntt_domain,
                            int threads) {
    aut_ctx c = {in, out, q, psi, log_n, L, k, ntt_domain};
    run_units(aut_unit, &c, (long)batch * L, threads);
}

/* Digit ranges: alpha = ceil(L / dnum); digit j covers limbs [j alpha, min((j+1) alpha, L)). */
static void digit_range(int L, int dnum, int j, int *lo, int *hi) {
    int alpha = (L + dnum - 1) / dnum;
    *lo = j * alpha;
    *hi = (j + 1) * alpha < L ? (j + 1) * alpha : L;
}

typedef struct {
    const uint64_t *in; uint64_t *out; const uint64_t *qp; int log_n; int L; int K; int dnum; int batch;
    int approx;
} modup_ctx;

/* one unit = one (batch item, digit) pair: all n coefficients */
static void modup_unit(void *c, long u) {
    modup_ctx *x = (modup_ctx *)c;
    uint64_t n = (uint64_t)1 << x->log_n;
    int LK = x->L + x->K;
    int bi = (int)(u / x->dnum), j = (int)(u % x->dnum);
    int lo, hi;
    digit_range(x->L, x->dnum, j, &lo, &hi);
    int alpha = hi - lo;
    const uint64_t *src = x->in + (uint64_t)bi * x->L * n;
    uint64_t *dst = x->out + ((uint64_t)bi * x->dnum + j) * LK * n;
    uint64_t xs[64], res[256], qinv[64];
    uint64_t *qhat = NULL;
    if (x->approx) {
        qhat = (uint64_t *)malloc((size_t)LK * alpha * sizeof(uint64_t));
        fast_bconv_consts(x->qp + lo, alpha, x->qp, LK, qinv, qhat);
    }
    for (uint64_t i = 0; i < n; i++) {
        for (int a = 0; a < alpha; a++) xs[a] = src[(uint64_t)(lo + a) * n + i];
        if (x->approx) fast_bconv_apply(xs, x->qp + lo, alpha, x->qp, LK, qinv, qhat, res);
        else oracle_modup_coeff(xs, x->qp + lo, alpha, x->qp, LK, res);
        for (int l = 0; l < LK; l++) dst[(uint64_t)l * n + i] = res[l];
    }
    free(qhat);
}

/* ModUp of every digit: in [batch][L][n] (coefficient domain, basis q_0..q_{L-1})
 * -> out [batch][dnum][L+K][n] (coefficient domain, basis qp = q_0..q_{L-1},
 * p_0..p_{K-1}).  Limbs inside the digit reproduce the input residues. */
void oracle_modup_batch_ex(const uint64_t *in, uint64_t *out, const uint64_t *qp, int log_n, int L,
                           int K, int dnum, int batch, int approx, int threads) {
    modup_ctx c = {in, out, qp, log_n, L, K, dnum, batch, approx};
    run_units(modup_unit, &c, (long)batch * dnum, threads);
}

void oracle_modup_batch(const uint64_t *in, uint64_t *out, const uint64_t *qp, int log_n, int L,
                        int K, int dnum, int batch, int threads) {
    oracle_modup_batch_ex(in, out, qp, log_n, L, K, dnum, batch, 0, threads);
}

typedef struct {
    const uint64_t *in; uint64_t *out; const uint64_t *src; int S; const uint64_t *dst; int T;
    int log_n; int approx; const uint64_t *qinv; const uint64_t *qhat;
} bconv_ctx;

/* one unit = one batch item */
static void bconv_unit(void *c, long u) {
    bconv_ctx *x = (bconv_ctx *)c;
    uint64_t n = (uint64_t)1 << x->log_n;
    const uint64_t *src = x->in + (uint64_t)u * x->S * n;
    uint64_t *dst = x->out + (uint64_t)u * x->T * n;
    uint64_t xs[64], res[8192];
    for (uint64_t i = 0; i < n; i++) {
        for (int a = 0; a < x->S; a++) xs[a] = src[(uint64_t)a * n + i];
        if (x->approx) fast_bconv_apply(xs, x->src, x->S, x->dst, x->T, x->qinv, x->qhat, res);
        else oracle_modup_coeff(xs, x->src, x->S, x->dst, x->T, res);
        for (int t = 0; t < x->T; t++) dst[(uint64_t)t * n + i] = res[t];
    }
}

/* Basis conversion of every coefficient: in [batch][S][n] over src ->
 * out [batch][T][n] over dst (coefficient domain).  Modraise -- the
 * extension of a low-level ciphertext to the full chain that starts a
 * bootstrap -- is the exact case with src the first S primes of the chain
 * and dst the whole chain.  S <= 64, T <= 8192. */
void oracle_bconv_batch(const uint64_t *in, uint64_t *out, const uint64_t *src, int S, const uint64_t *dst,
                        int T, int log_n, int batch, int approx, int threads) {
    uint64_t qinv[64];
    uint64_t *qhat = (uint64_t *)malloc((size_t)T * S * sizeof(uint64_t));
    fast_bconv_consts(src, S, dst, T, qinv, qhat);
    bconv_ctx c = {in, out, src, S, dst, T, log_n, approx, qinv, qhat};
    run_units(bconv_unit, &c, (long)batch, threads);
    free(qhat);
}

/* ------------------------------------------------------------------------ */
/* ModDown (QP -> Q) and rescale: divide by P with rounding.                  */
/* ------------------------------------------------------------------------ */

/* For one coefficient with residues x[0..L+K) over (q_0..q_{L-1}, p_0..p_{K-1})
 * of X in [0, QP), P = p_0 ... p_{K-1}:
 *   out[l] = floor((X + h) / P) mod q_l,   h = (P - 1)/2 (nearest) or 0.
 * Identity used: with c = (X + h) mod P (a value in [0, P), obtained exactly
 * from the P residues of X + h by Garner's mixed radix),
 *   floor((X + h) / P) = (X + h - c) / P,
 * and the right side is reduced mod q_l with P^-1 mod q_l. */
static void moddown_coeff(const uint64_t *x, const uint64_t *qp, int L, int K, int nearest, uint64_t *out) {
    const uint64_t *P = qp + L;
    uint64_t y[64], v[64];
    for (int k = 0; k < K; k++) {
        /* h mod p_k = (P - 1)/2 mod p_k = (p_k - 1)/2 since P = 0 mod p_k */
        uint64_t h = nearest ? (P[k] - 1) / 2 : 0;
        y[k] = addmod(x[L + k] % P[k], h, P[k]);
    }
    garner_digits(y, P, K, v);
    for (int l = 0; l < L; l++) {
        uint64_t q = qp[l];
        uint64_t Pm = 1 % q;
        for (int k = 0; k < K; k++) Pm = mulmod(Pm, P[k] % q, q);
        /* h mod q = (P mod q - 1) / 2 mod q */
        uint64_t h = nearest ? mulmod(submod(Pm, 1 % q, q), invmod(2, q), q) : 0;
        uint64_t c = mixed_radix_mod(v, P, K, q);
        uint64_t num = submod(addmod(x[l] % q, h, q), c, q);
        out[l] = mulmod(num, invmod(Pm, q), q);
    }
}

/* in: [batch][L+K][n] coefficient domain; out: [batch][L][n] coefficient domain. */
void oracle_moddown_batch(const uint64_t *in, uint64_t *out, const uint64_t *qp, int log_n, int L, int K,
                          int batch, int nearest) {
    uint64_t n = (uint64_t)1 << log_n;
    uint64_t xs[256], r[256];
    for (int b = 0; b < batch; b++) {
        for (uint64_t i = 0; i < n; i++) {
            for (int l = 0; l < L + K; l++) xs[l] = in[((uint64_t)b * (L + K) + l) * n + i];
            moddown_coeff(xs, qp, L, K, nearest, r);
            for (int l = 0; l < L; l++) out[((uint64_t)b * L + l) * n + i] = r[l];
        }
    }
}

/* out[b][c][l] = sum_j ext[b][j][l] * keys[j][c][l] mod qp_l over the NTT-domain
 * extended digits ext [batch][dnum][L+K][n]. */
static void keyswitch_ip(const uint64_t *ext, const uint64_t *keys, uint64_t *out, const uint64_t *qp,
                         int log_n, int LK, int dnum, int batch) {
    uint64_t n = (uint64_t)1 << log_n;
    uint64_t plane = (uint64_t)LK * n;
    for (int bi = 0; bi < batch; bi++) {
        for (int c = 0; c < 2; c++) {
            for (int l = 0; l < LK; l++) {
                uint64_t p = qp[l];
                uint64_t *o = out + ((uint64_t)bi * 2 + c) * plane + (uint64_t)l * n;
                for (uint64_t i = 0; i < n; i++) {
                    uint64_t acc = 0;
                    for (int j = 0; j < dnum; j++) {
                        uint64_t dv = ext[(((uint64_t)bi * dnum + j) * LK + l) * n + i];
                        uint64_t kv = keys[(((uint64_t)j * 2 + c) * LK + l) * n + i];
                        acc = addmod(acc, mulmod(dv, kv, p), p);
                    }
                    o[i] = acc;
                }
            }
        }
    }
}

/* Hybrid key-switch inner product, before ModDown:
 *   out[b][c][l] = sum_j NTT_l(ModUp_j(in[b]))[l] * keys[j][c][l]  mod qp_l
 * in: [batch][L][n] coefficient domain; keys: [dnum][2][L+K][n] NTT domain;
 * out: [batch][2][L+K][n] NTT domain.  approx != 0 takes the approximate
 * basis conversion for ModUp instead of the exact one. */
void oracle_keyswitch_batch_ex(const uint64_t *in, const uint64_t *keys, uint64_t *out,
                               const uint64_t *qp, const uint64_t *psi_qp, int log_n, int L, int K,
                               int dnum, int batch, int approx, int threads) {
    uint64_t n = (uint64_t)1 << log_n;
    int LK = L + K;
    uint64_t plane = (uint64_t)LK * n;
    uint64_t *ext = (uint64_t *)malloc((uint64_t)batch * dnum * plane * sizeof(uint64_t));
    oracle_modup_batch_ex(in, ext, qp, log_n, L, K, dnum, batch, approx, threads);
    /* every (batch, digit) block is one row set of LK limbs */
    oracle_ntt_batch(ext, log_n, LK, batch * dnum, qp, psi_qp, 0, threads);
    keyswitch_ip(ext, keys, out, qp, log_n, LK, dnum, batch);
    free(ext);
}

void oracle_keyswitch_batch(const uint64_t *in, const uint64_t *keys, uint64_t *out,
                            const uint64_t *qp, const uint64_t *psi_qp, int log_n, int L, int K,
                            int dnum, int batch, int threads) {
    oracle_keyswitch_batch_ex(in, keys, out, qp, psi_qp, log_n, L, K, dnum, batch, 0, threads);
}

/* Hoisted key switch for R Galois elements k_r (the rotations of
 * coeff_to_slot / slot_to_coeff): ModUp and the NTT of the digits are done
 * once, then for each r the automorphism sigma_{k_r} acts on the extended
 * digits in the NTT domain and the inner product uses that rotation's keys:
 *   out[r][b][c][l] = sum_j sigma_{k_r}(NTT_l(ModUp_j(in[b])))[l] * keys[r][j][c][l]
 * in: [batch][L][n] coefficient domain; keys: [R][dnum][2][L+K][n];
 * out: [R][batch][2][L+K][n] NTT domain. */
void oracle_keyswitch_hoisted_batch(const uint64_t *in, const uint64_t *keys, const uint64_t *ks, int R,
                                    uint64_t *out, const uint64_t *qp, const uint64_t *psi_qp, int log_n,
                                    int L, int K, int dnum, int batch, int approx, int threads) {
    uint64_t n = (uint64_t)1 << log_n;
    int LK = L + K;
    uint64_t plane = (uint64_t)LK * n;
    uint64_t rows = (uint64_t)batch * dnum * plane;
    uint64_t *ext = (uint64_t *)malloc(rows * sizeof(uint64_t));
    uint64_t *rot = (uint64_t *)malloc(rows * sizeof(uint64_t));
    oracle_modup_batch_ex(in, ext, qp, log_n, L, K, dnum, batch, approx, threads);
    oracle_ntt_batch(ext, log_n, LK, batch * dnum, qp, psi_qp, 0, threads);
    for (int r = 0; r < R; r++) {
        oracle_automorph_batch(ext, rot, log_n, LK, batch * dnum, qp, psi_qp, ks[r], 1, threads);
        keyswitch_ip(rot, keys + (uint64_t)r * dnum * 2 * plane, out + (uint64_t)r * batch * 2 * plane, qp,
                     log_n, LK, dnum, batch);
    }
    free(rot);
    free(ext);
}
