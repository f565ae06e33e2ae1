// tables.cpp -- host-side table builders of libfhe_ntt.so: prime search,
// roots of unity, twiddle tables with Shoup companions, per-prime constants,
// and the Garner / mixed-radix constants of the key-switch basis extension.
// Host code only; the blobs it writes are copied to the device by the caller.
#include <cstdint>
#include <cstring>
#include <vector>

#include "fhe_arith.cuh"
#include "fhe_internal.h"
#include "ntt_shapes.h"

namespace {

using u128 = unsigned __int128;

uint64_t mul_mod(uint64_t a, uint64_t b, uint64_t m) { return (uint64_t)((u128)a * b % m); }

uint64_t pow_mod(uint64_t b, uint64_t e, uint64_t m) {
    uint64_t r = 1 % m;
    b %= m;
    for (; e; e >>= 1) {
        if (e & 1) r = mul_mod(r, b, m);
        b = mul_mod(b, b, m);
    }
    return r;
}

uint64_t inv_mod(uint64_t a, uint64_t p) { return pow_mod(a % p, p - 2, p); }

// Deterministic Miller-Rabin for all 64-bit n with the seven witnesses
// {2, 325, 9375, 28178, 450775, 9780504, 1795265022} (J. Sinclair, 2011).
bool is_prime_u64(uint64_t n) {
    if (n < 2) return false;
    for (uint64_t p : {2ull, 3ull, 5ull, 7ull, 11ull, 13ull, 17ull, 19ull, 23ull, 29ull, 31ull, 37ull}) {
        if (n % p == 0) return n == p;
    }
    uint64_t d = n - 1;
    int s = __builtin_ctzll(d);
    d >>= s;
    for (uint64_t a : {2ull, 325ull, 9375ull, 28178ull, 450775ull, 9780504ull, 1795265022ull}) {
        uint64_t x = pow_mod(a % n, d, n);
        if (a % n == 0 || x == 1 || x == n - 1) continue;
        bool witness = true;
        for (int i = 1; i < s && witness; i++) {
            x = mul_mod(x, x, n);
            if (x == n - 1) witness = false;
        }
        if (witness) return false;
    }
    return true;
}

uint64_t shoup(uint64_t w, uint64_t q) { return (uint64_t)(((u128)w << 64) / q); }

uint32_t bit_reverse(uint32_t x, int bits) {
    uint32_t r = 0;
    for (int i = 0; i < bits; i++) r |= ((x >> i) & 1u) << (bits - 1 - i);
    return r;
}

bool modulus_ok(uint64_t q, int log_n) {
    const uint64_t two_n = 2ull << log_n;
    return q > (1ull << 48) && q < (1ull << 50) && q % two_n == 1 && is_prime_u64(q);
}

// Smallest element of multiplicative order exactly 2n: every such element is
// g^t (t odd) for one g of order 2n, and g = c^((q-1)/2n) has order 2n as
// soon as c is a quadratic non-residue (then g^n = c^((q-1)/2) = -1).
uint64_t smallest_primitive_root(uint64_t q, int log_n) {
    const uint64_t two_n = 2ull << log_n, n = 1ull << log_n;
    uint64_t g = 0;
    for (uint64_t c = 2; c < q; c++) {
        g = pow_mod(c, (q - 1) / two_n, q);
        if (pow_mod(g, n, q) == q - 1) break;
    }
    const uint64_t g2 = mul_mod(g, g, q);
    uint64_t best = g, cur = g;
    for (uint64_t t = 3; t < two_n; t += 2) {
        cur = mul_mod(cur, g2, q);
        if (cur < best) best = cur;
    }
    return best;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

namespace fhe {

NttLayout ntt_layout(int log_n, int L) {
    NttLayout s;
    const size_t n = (size_t)1 << log_n;
    s.off_q = 0;
    s.off_consts = align256(s.off_q + (size_t)L * 8);
    s.off_fwd = align256(s.off_consts + (size_t)L * K_COUNT * 8);
    s.off_inv = align256(s.off_fwd + (size_t)L * n * 16);
    s.off_twist = align256(s.off_inv + (size_t)L * n * 16);
    s.bytes = align256(s.off_twist + (size_t)L * n * 16);
    return s;
}

ModupLayout modup_layout(int L, int K, int dnum) {
    ModupLayout s;
    s.alpha = (L + dnum - 1) / dnum;
    const int LK = L + K;
    s.off_digits = 0;
    s.off_garner = align256((size_t)dnum * sizeof(ModupDigit));
    s.off_mr = align256(s.off_garner + (size_t)dnum * s.alpha * s.alpha * 16);
    s.off_qinv = align256(s.off_mr + (size_t)dnum * LK * s.alpha * 16);
    s.off_qhat = align256(s.off_qinv + (size_t)dnum * s.alpha * 16);
    const size_t end = align256(s.off_qhat + (size_t)dnum * LK * s.alpha * 16);
    s.tc_tmax = s.alpha <= kTcMaxAlpha ? (LK + 1) & ~1 : 0;
    s.off_tc_tgt = end;
    s.off_tc_frac = align256(s.off_tc_tgt + (size_t)dnum * s.tc_tmax * sizeof(ModupTcTarget));
    s.off_tc_b = align256(s.off_tc_frac + (s.tc_tmax ? (size_t)dnum * (kTcMaxAlpha + 1) * sizeof(ModupTcFrac) : 0));
    s.bytes = align256(s.off_tc_b + (size_t)dnum * s.tc_tmax * 8 * kTcRowBytes);
    return s;
}

BconvLayout bconv_layout(int S, int T) {
    BconvLayout s;
    s.off_src = 0;
    s.off_dst = align256((size_t)S * 8);
    s.off_garner = align256(s.off_dst + (size_t)T * 32);
    s.off_mr = align256(s.off_garner + (size_t)S * S * 16);
    s.off_qinv = align256(s.off_mr + (size_t)T * S * 16);
    s.off_qhat = align256(s.off_qinv + (size_t)S * 16);
    s.bytes = align256(s.off_qhat + (size_t)T * S * 16);
    return s;
}

ModdownLayout moddown_layout(int L, int K) {
    ModdownLayout s;
    s.off_garner = 0;
    s.off_mr = align256((size_t)K * K * 16);
    s.off_hp = align256(s.off_mr + (size_t)L * K * 16);
    s.off_hq = align256(s.off_hp + (size_t)K * 8);
    s.off_pinv = align256(s.off_hq + (size_t)L * 8);
    const size_t end = align256(s.off_pinv + (size_t)L * 16);
    const bool tc = K <= kTcMaxAlpha;
    s.tc_tmax = tc ? (L + 1) & ~1 : 0;
    s.off_tc_qinv = end;
    s.off_tc_tgt = align256(s.off_tc_qinv + (tc ? (size_t)K * 16 : 0));
    s.off_tc_frac = align256(s.off_tc_tgt + (size_t)s.tc_tmax * sizeof(ModupTcTarget));
    s.off_tc_b = align256(s.off_tc_frac + (tc ? (size_t)(kTcMaxAlpha + 1) * sizeof(ModupTcFrac) : 0));
    s.bytes = align256(s.off_tc_b + (size_t)s.tc_tmax * 8 * kTcRowBytes);
    return s;
}

fhe_ntt_tables tables_slice(const fhe_ntt_tables *t, int first, int count) {
    fhe_ntt_tables s = *t;
    const size_t n = (size_t)1 << t->log_n;
    s.L = count;
    s.q = t->q + first;
    s.consts = t->consts + (size_t)first * K_COUNT;
    s.fwd = t->fwd + (size_t)first * n * 2;
    s.inv = t->inv + (size_t)first * n * 2;
    s.twist = t->twist + (size_t)first * n * 2;
    return s;
}

bool modup_shape_ok(int L, int K, int dnum) {
    if (L < 1 || K < 0 || dnum < 1 || dnum > L || L + K > kMaxBasis) return false;
    const int alpha = (L + dnum - 1) / dnum;
    if (alpha > kMaxAlpha) return false;
    return (dnum - 1) * alpha < L;   // every digit non-empty
}

int selftest_arith(uint64_t seed, int iters);

}  // namespace fhe

using namespace fhe;

extern "C" int fhe_find_primes(int log_n, int bits, int count, uint64_t below, uint64_t *out) {
    if (log_n < 1 || log_n > kMaxLogN || bits < 2 || bits > 62 || count < 1 || !out) return FHE_EINVAL;
    const uint64_t m = 2ull << log_n;
    const uint64_t top = 1ull << bits;
    if (below == 0 || below > top) below = top;
    if (below <= m + 1) return FHE_EINVAL;
    uint64_t c = ((below - 2) / m) * m + 1;   // largest c < below with c = 1 mod m
    int found = 0;
    for (; found < count && c > m; c -= m) {
        if (is_prime_u64(c)) out[found++] = c;
    }
    return found == count ? FHE_OK : FHE_EINVAL;
}

extern "C" int fhe_root_of_unity(uint64_t q, int log_n, uint64_t *psi) {
    if (!psi || log_n < 1 || log_n > kMaxLogN) return FHE_EINVAL;
    const uint64_t two_n = 2ull << log_n;
    if (q < 3 || q % two_n != 1 || !is_prime_u64(q)) return FHE_EINVAL;
    *psi = smallest_primitive_root(q, log_n);
    return FHE_OK;
}

extern "C" int fhe_ntt_tables_bytes(int log_n, int L, size_t *bytes) {
    if (!bytes || log_n < 1 || log_n > kMaxLogN || L < 1 || L > kMaxTableL) return FHE_EINVAL;
    *bytes = ntt_layout(log_n, L).bytes;
    return FHE_OK;
}

extern "C" int fhe_ntt_tables_build_host(int log_n, int L, const uint64_t *q, void *host_blob, size_t bytes) {
    if (!q || !host_blob || log_n < 1 || log_n > kMaxLogN || L < 1 || L > kMaxTableL) return FHE_EINVAL;
    const NttLayout lay = ntt_layout(log_n, L);
    if (bytes < lay.bytes) return FHE_ESPACE;
    for (int l = 0; l < L; l++)
        if (!modulus_ok(q[l], log_n)) return FHE_EINVAL;
    const uint64_t n = 1ull << log_n;
    char *base = (char *)host_blob;
    std::memset(base, 0, lay.bytes);
    uint64_t *qv = (uint64_t *)(base + lay.off_q);
    uint64_t *kc = (uint64_t *)(base + lay.off_consts);
    uint64_t *fwd = (uint64_t *)(base + lay.off_fwd);
    uint64_t *inv = (uint64_t *)(base + lay.off_inv);
    uint64_t *twist = (uint64_t *)(base + lay.off_twist);
    std::vector<uint64_t> pw(n), ipw(n);
    for (int l = 0; l < L; l++) {
        const uint64_t ql = q[l];
        const uint64_t psi = smallest_primitive_root(ql, log_n);
        const uint64_t psi_inv = inv_mod(psi, ql);
        pw[0] = ipw[0] = 1;
        for (uint64_t i = 1; i < n; i++) {
            pw[i] = mul_mod(pw[i - 1], psi, ql);
            ipw[i] = mul_mod(ipw[i - 1], psi_inv, ql);
        }
        uint64_t *f = fwd + (size_t)l * n * 2, *g = inv + (size_t)l * n * 2, *tw = twist + (size_t)l * n * 2;
        const uint64_t ninv = inv_mod(n % ql, ql);
        for (uint64_t k = 0; k < n; k++) {
            // forward (psi-merged, bit-reversed): fwd[k] = psi^brv(k), brv over log_n bits
            const uint64_t w = pw[bit_reverse((uint32_t)k, log_n)];
            const uint32_t slot = fwd_table_slot(log_n, (uint32_t)k);
            f[2 * slot] = w;
            f[2 * slot + 1] = shoup(w, ql);
            // twist of the inverse: twist[j] = n^-1 psi^-j
            const uint64_t tj = mul_mod(ninv, ipw[k], ql);
            tw[2 * k] = tj;
            tw[2 * k + 1] = shoup(tj, ql);
        }
        // cyclic inverse: inv[h + j] = omega_2h^-j = psi^(-j n / h) for h = 2^e < n, j < h
        g[0] = 1;
        g[1] = shoup(1, ql);
        for (uint64_t h = 1; h < n; h <<= 1) {
            for (uint64_t j = 0; j < h; j++) {
                const uint64_t wi = ipw[(j * (n / h)) % n];   // j n / h < n
                g[2 * (h + j)] = wi;
                g[2 * (h + j) + 1] = shoup(wi, ql);
            }
        }
        uint64_t *c = kc + (size_t)l * K_COUNT;
        qv[l] = ql;
        c[K_Q] = ql;
        c[K_MU12] = (uint64_t)(((u128)1 << 100) / ql) << 12;
        c[K_C58] = (uint64_t)((1ull << 58) / ql);
        c[K_NINV] = ninv;
        c[K_PSI] = psi;
    }
    return FHE_OK;
}

extern "C" int fhe_ntt_tables_bind(const void *dev_blob, size_t bytes, int log_n, int L, fhe_ntt_tables *out) {
    if (!dev_blob || !out || log_n < 1 || log_n > kMaxLogN || L < 1 || L > kMaxTableL) return FHE_EINVAL;
    const NttLayout lay = ntt_layout(log_n, L);
    if (bytes < lay.bytes) return FHE_ESPACE;
    if (((uintptr_t)dev_blob & 15) != 0) return FHE_EINVAL;
    const char *base = (const char *)dev_blob;
    out->log_n = log_n;
    out->L = L;
    out->q = (const uint64_t *)(base + lay.off_q);
    out->consts = (const uint64_t *)(base + lay.off_consts);
    out->fwd = (const uint64_t *)(base + lay.off_fwd);
    out->inv = (const uint64_t *)(base + lay.off_inv);
    out->twist = (const uint64_t *)(base + lay.off_twist);
    out->blob = dev_blob;
    out->bytes = lay.bytes;
    return FHE_OK;
}

extern "C" int fhe_modup_tables_bytes(int L, int K, int dnum, size_t *bytes) {
    if (!bytes || !modup_shape_ok(L, K, dnum)) return FHE_EINVAL;
    *bytes = modup_layout(L, K, dnum).bytes;
    return FHE_OK;
}

// Constants of the exact basis extension of digit j with primes d_0..d_{a-1}:
//  Garner (mixed radix):  v_0 = x_0,  v_i = (((x_i - v_0) d_0^-1 - v_1) d_1^-1 ...
//                          - v_{i-1}) d_{i-1}^-1  mod d_i           -> garner[i][k] = d_k^-1 mod d_i
//  Extension:             X mod p = v_0 + sum_{i>=1} v_i (d_0 ... d_{i-1} mod p)
//                                                                    -> mr[l][i] = d_0..d_{i-1} mod p_l
// Both with Shoup companions (pairs of words).
// fp16 bits of an integer 0 <= v <= 2048 (all exactly representable).
static uint16_t fp16_of_int(int v) {
    if (v == 0) return 0;
    const int e = 31 - __builtin_clz((unsigned)v);
    const int m = e <= 10 ? v << (10 - e) : v >> (e - 10);
    return (uint16_t)(((e + 15) << 10) | (m & 0x3FF));
}

// The tensor-core extension's weight operand for one digit of cnt primes and
// T targets.  With the digit's CRT brackets y_a split into bytes b_{a,e}
// (e = 0..6; y_a < 2^50) and the correction count e_c, the extension of
// target p is
//   sum_a y_a W_{a,p} - e_c D = sum_{a,e} b_{a,e} (W_{a,p} 2^(8e) mod p)
//                              + e_c ((-D) mod p)                  (mod p),
// and each constant c = W_{a,p} 2^(8e) mod p < 2^56 is split into eight
// 7-bit limbs c_s.  Operand row 8 t + s (target t, limb s), column 8 a + e,
// holds c_s; the kernel's other operand holds 1024 + b_{a,e} (the fp16 bit
// pattern 0x6400 | b) and 1024 + e_c in column 15, so accumulator column
// 8 t + s receives 1024 * (row sum) + sum_{a,e} b_{a,e} c_s + e_c m_s, with
// m_s the 7-bit limbs of (-D) mod p in column 15 (kTcCorrCol).  The other
// columns 8 a + 7 (byte 7 of y_a, always 0) hold integers <= 2048 that make
// every row sum 8192: each accumulator is then 2^23 + (a value < 2^21) and
// its f32 bit pattern minus 0x4B000000 is that value.  Rows of the odd
// target that pads T to even carry only the 8192.
static void tc_weight_image(uint8_t *img, int cnt, int T, const uint64_t *W, const uint64_t *P, const uint64_t *corr) {
    const int Tp = (T + 1) & ~1;
    for (int t = 0; t < Tp; t++) {
        for (int s = 0; s < 8; s++) {
            int val[8 * kTcMaxAlpha] = {0};
            int sum = 0;
            for (int a = 0; t < T && a < cnt; a++) {
                uint64_t c = W[(size_t)a * T + t];
                for (int e = 0; e < 7; e++, c = mul_mod(c, 256, P[t])) {
                    val[8 * a + e] = (int)((c >> (7 * s)) & 127);
                    sum += val[8 * a + e];
                }
            }
            if (t < T) {
                val[kTcCorrCol] = (int)((corr[t] >> (7 * s)) & 127);
                sum += val[kTcCorrCol];
            }
            int rem = 8192 - sum;   // sum <= 7 * 8 * 127 + 127 = 7239
            for (int a = 0; a < kTcMaxAlpha; a++) {
                if (8 * a + 7 == kTcCorrCol) continue;
                const int v = rem < 2048 ? rem : 2048;
                val[8 * a + 7] = v;
                rem -= v;
            }
            const int n = 8 * t + s;
            for (int k = 0; k < 8 * kTcMaxAlpha; k++) {
                const uint16_t h = fp16_of_int(val[k]);
                std::memcpy(img + ((size_t)(n >> 3) * kTcMaxAlpha + (k >> 3)) * 128 + (n & 7) * 16 + (k & 7) * 2, &h,
                            2);
            }
        }
    }
}

// The tensor-core extension's constants for the source basis d[0..cnt) (product
// D) and the targets p[0..T) (basis indices limb[t], output offsets aux[t]):
// the target records, the weight operand ((D/d_a) mod p and the correction
// (-D) mod p), and per source prime the reciprocal floor(2^128 / d_a) with
// the redundant-modulus constants (D/d_a) mod 2^64 and d_0 .. d_{a-1} mod 2^64
// (entry kTcMaxAlpha: D^-1 mod 2^64).
static void tc_build_basis(const uint64_t *d, int cnt, const uint64_t *p, const int *limb, const uint64_t *aux, int T,
                           ModupTcTarget *tg, ModupTcFrac *fr, uint8_t *img) {
    std::vector<uint64_t> W((size_t)cnt * T), corr(T);
    for (int t = 0; t < T; t++) {
        tg[t].p = p[t];
        tg[t].mu = (uint64_t)(((u128)1 << 64) / p[t]);
        tg[t].aux = aux ? aux[t] : 0;
        tg[t].limb = (uint64_t)limb[t];
        uint64_t Dp = 1 % p[t];
        for (int a = 0; a < cnt; a++) {
            Dp = mul_mod(Dp, d[a] % p[t], p[t]);
            uint64_t hp = 1 % p[t];
            for (int b = 0; b < cnt; b++)
                if (b != a) hp = mul_mod(hp, d[b] % p[t], p[t]);
            W[(size_t)a * T + t] = hp;            // (D / d_a) mod p
        }
        corr[t] = (p[t] - Dp) % p[t];             // (-D) mod p
    }
    tc_weight_image(img, cnt, T, W.data(), p, corr.data());
    uint64_t D64 = 1, W64 = 1;
    for (int a = 0; a < cnt; a++) D64 *= d[a];
    for (int a = 0; a < cnt; a++) {
        const u128 phi = ~(u128)0 / d[a];         // floor((2^128 - 1) / d_a) = floor(2^128 / d_a): d_a is odd
        fr[a].phi_hi = (uint64_t)(phi >> 64);
        fr[a].phi_lo = (uint64_t)phi;
        uint64_t h = 1;
        for (int b = 0; b < cnt; b++)
            if (b != a) h *= d[b];
        fr[a].dhat64 = h;                         // (D / d_a) mod 2^64
        fr[a].w64 = W64;                          // d_0 ... d_{a-1} mod 2^64
        W64 *= d[a];
    }
    uint64_t inv = D64;                           // D^-1 mod 2^64 (D odd): Newton on the 2-adic inverse
    for (int k = 0; k < 6; k++) inv *= 2 - D64 * inv;
    fr[kTcMaxAlpha].dhat64 = inv;
}

extern "C" int fhe_modup_tables_build_host(int L, int K, int dnum, const uint64_t *qp, void *host_blob,
                                           size_t bytes) {
    if (!qp || !host_blob || !modup_shape_ok(L, K, dnum)) return FHE_EINVAL;
    const ModupLayout lay = modup_layout(L, K, dnum);
    if (bytes < lay.bytes) return FHE_ESPACE;
    const int LK = L + K, alpha = lay.alpha;
    for (int l = 0; l < LK; l++) {
        if (qp[l] <= (1ull << 48) || qp[l] >= (1ull << 50) || !is_prime_u64(qp[l])) return FHE_EINVAL;
        for (int m = 0; m < l; m++)
            if (qp[m] == qp[l]) return FHE_EINVAL;
    }
    char *base = (char *)host_blob;
    std::memset(base, 0, lay.bytes);
    ModupDigit *dg = (ModupDigit *)(base + lay.off_digits);
    uint64_t *garner = (uint64_t *)(base + lay.off_garner);
    uint64_t *mr = (uint64_t *)(base + lay.off_mr);
    for (int j = 0; j < dnum; j++) {
        const int lo = j * alpha, hi = (lo + alpha < L) ? lo + alpha : L;
        dg[j].lo = lo;
        dg[j].count = hi - lo;
        uint64_t *gj = garner + (size_t)j * alpha * alpha * 2;
        for (int i = 0; i < hi - lo; i++) {
            const uint64_t di = qp[lo + i];
            for (int k = 0; k < i; k++) {
                const uint64_t c = inv_mod(qp[lo + k] % di, di);
                gj[(i * alpha + k) * 2] = c;
                gj[(i * alpha + k) * 2 + 1] = shoup(c, di);
            }
        }
        uint64_t *mj = mr + (size_t)j * LK * alpha * 2;
        for (int l = 0; l < LK; l++) {
            const uint64_t p = qp[l];
            uint64_t prod = 1 % p;
            for (int i = 0; i < hi - lo; i++) {
                split25_store(prod, mj + (l * alpha + i) * 2);
                prod = mul_mod(prod, qp[lo + i] % p, p);
            }
        }
        // approximate conversion: qinv_a = (D_j / d_a)^-1 mod d_a, qhat[l][a] = (D_j / d_a) mod qp_l
        uint64_t *qi = (uint64_t *)(base + lay.off_qinv) + (size_t)j * alpha * 2;
        uint64_t *qh = (uint64_t *)(base + lay.off_qhat) + (size_t)j * LK * alpha * 2;
        for (int a = 0; a < hi - lo; a++) {
            const uint64_t da = qp[lo + a];
            uint64_t h = 1 % da;
            for (int b = 0; b < hi - lo; b++)
                if (b != a) h = mul_mod(h, qp[lo + b] % da, da);
            const uint64_t c = inv_mod(h, da);
            qi[a * 2] = c;
            qi[a * 2 + 1] = shoup(c, da);
            for (int l = 0; l < LK; l++) {
                const uint64_t p = qp[l];
                uint64_t hp = 1 % p;
                for (int b = 0; b < hi - lo; b++)
                    if (b != a) hp = mul_mod(hp, qp[lo + b] % p, p);
                split25_store(hp, qh + (l * alpha + a) * 2);
            }
        }
        if (lay.tc_tmax > 0) {
            // the digit's targets (every prime outside it)
            const int cnt = hi - lo, T = LK - cnt;
            std::vector<uint64_t> P;
            std::vector<int> limb;
            for (int l = 0; l < LK; l++)
                if (l < lo || l >= hi) {
                    P.push_back(qp[l]);
                    limb.push_back(l);
                }
            tc_build_basis(qp + lo, cnt, P.data(), limb.data(), nullptr, T,
                           (ModupTcTarget *)(base + lay.off_tc_tgt) + (size_t)j * lay.tc_tmax,
                           (ModupTcFrac *)(base + lay.off_tc_frac) + (size_t)j * (kTcMaxAlpha + 1),
                           (uint8_t *)(base + lay.off_tc_b) + (size_t)j * lay.tc_tmax * 8 * kTcRowBytes);
        }
    }
    return FHE_OK;
}

extern "C" int fhe_bconv_tables_bytes(int S, int T, size_t *bytes) {
    if (!bytes || S < 1 || S > kMaxBconvSrc || T < 1 || T > kMaxTableL) return FHE_EINVAL;
    *bytes = bconv_layout(S, T).bytes;
    return FHE_OK;
}

// Constants of the conversion from src[S] to dst[T] (exact Garner and
// approximate CRT sum); every prime in (2^48, 2^50), the sources distinct.
extern "C" int fhe_bconv_tables_build_host(int S, const uint64_t *src, int T, const uint64_t *dst, void *host_blob,
                                           size_t bytes) {
    size_t need = 0;
    if (fhe_bconv_tables_bytes(S, T, &need) != FHE_OK || !src || !dst || !host_blob) return FHE_EINVAL;
    if (bytes < need) return FHE_ESPACE;
    auto ok = [](uint64_t q) { return q > (1ull << 48) && q < (1ull << 50) && is_prime_u64(q); };
    for (int a = 0; a < S; a++) {
        if (!ok(src[a])) return FHE_EINVAL;
        for (int b = 0; b < a; b++)
            if (src[a] == src[b]) return FHE_EINVAL;
    }
    for (int t = 0; t < T; t++)
        if (!ok(dst[t])) return FHE_EINVAL;
    const BconvLayout lay = bconv_layout(S, T);
    char *base = (char *)host_blob;
    std::memset(base, 0, lay.bytes);
    uint64_t *sp = (uint64_t *)(base + lay.off_src);
    uint64_t *dp = (uint64_t *)(base + lay.off_dst);
    uint64_t *garner = (uint64_t *)(base + lay.off_garner);
    uint64_t *mr = (uint64_t *)(base + lay.off_mr);
    uint64_t *qi = (uint64_t *)(base + lay.off_qinv);
    uint64_t *qh = (uint64_t *)(base + lay.off_qhat);
    for (int a = 0; a < S; a++) {
        sp[a] = src[a];
        for (int b = 0; b < a; b++) {
            const uint64_t c = inv_mod(src[b] % src[a], src[a]);
            garner[(a * S + b) * 2] = c;
            garner[(a * S + b) * 2 + 1] = shoup(c, src[a]);
        }
        uint64_t h = 1 % src[a];
        for (int b = 0; b < S; b++)
            if (b != a) h = mul_mod(h, src[b] % src[a], src[a]);
        const uint64_t c = inv_mod(h, src[a]);
        qi[a * 2] = c;
        qi[a * 2 + 1] = shoup(c, src[a]);
    }
    for (int t = 0; t < T; t++) {
        const uint64_t p = dst[t];
        dp[t * 4] = p;
        dp[t * 4 + 1] = (1ull << 58) / p;
        dp[t * 4 + 2] = (uint64_t)(((u128)1 << 100) / p) << 12;
        uint64_t prod = 1 % p;
        for (int a = 0; a < S; a++) {
            split25_store(prod, mr + ((size_t)t * S + a) * 2);
            prod = mul_mod(prod, src[a] % p, p);
            uint64_t hp = 1 % p;
            for (int b = 0; b < S; b++)
                if (b != a) hp = mul_mod(hp, src[b] % p, p);
            split25_store(hp, qh + ((size_t)t * S + a) * 2);
        }
    }
    return FHE_OK;
}

extern "C" int fhe_moddown_tables_bytes(int L, int K, size_t *bytes) {
    if (!bytes || L < 1 || K < 1 || K > kMaxAlpha || L + K > kMaxTableL) return FHE_EINVAL;
    *bytes = moddown_layout(L, K).bytes;
    return FHE_OK;
}

// ModDown by P = p_0 ... p_{K-1}: Garner constants over P, the mixed-radix
// weights prod_{b<a} p_b mod q_l, h = (P-1)/2 mod every prime (nearest
// rounding) and P^-1 mod q_l, with Shoup companions where used as
// multipliers.
extern "C" int fhe_moddown_tables_build_host(int L, int K, const uint64_t *qp, void *host_blob, size_t bytes) {
    if (!qp || !host_blob || L < 1 || K < 1 || K > kMaxAlpha || L + K > kMaxTableL) return FHE_EINVAL;
    const ModdownLayout lay = moddown_layout(L, K);
    if (bytes < lay.bytes) return FHE_ESPACE;
    for (int l = 0; l < L + K; l++) {
        if (qp[l] <= (1ull << 48) || qp[l] >= (1ull << 50) || !is_prime_u64(qp[l])) return FHE_EINVAL;
        for (int m = 0; m < l; m++)
            if (qp[m] == qp[l]) return FHE_EINVAL;
    }
    char *base = (char *)host_blob;
    std::memset(base, 0, lay.bytes);
    const uint64_t *P = qp + L;
    uint64_t *g = (uint64_t *)(base + lay.off_garner);
    uint64_t *mr = (uint64_t *)(base + lay.off_mr);
    uint64_t *hp = (uint64_t *)(base + lay.off_hp);
    uint64_t *hq = (uint64_t *)(base + lay.off_hq);
    uint64_t *pinv = (uint64_t *)(base + lay.off_pinv);
    for (int a = 0; a < K; a++) {
        for (int b = 0; b < a; b++) {
            const uint64_t c = inv_mod(P[b] % P[a], P[a]);
            g[(a * K + b) * 2] = c;
            g[(a * K + b) * 2 + 1] = shoup(c, P[a]);
        }
        hp[a] = (P[a] - 1) / 2;   // (P - 1)/2 mod p_a, as P = 0 mod p_a
    }
    for (int l = 0; l < L; l++) {
        const uint64_t q = qp[l];
        uint64_t prod = 1 % q;
        for (int a = 0; a < K; a++) {
            split25_store(prod, mr + (l * K + a) * 2);
            prod = mul_mod(prod, P[a] % q, q);
        }
        // prod = P mod q
        hq[l] = mul_mod((prod + q - 1) % q, inv_mod(2, q), q);
        const uint64_t pi = inv_mod(prod, q);
        pinv[l * 2] = pi;
        pinv[l * 2 + 1] = shoup(pi, q);
    }
    if (lay.tc_tmax > 0) {
        // the tensor-core conversion from P to every q_l; aux = (q_l - h) mod q_l for nearest rounding
        std::vector<int> limb(L);
        std::vector<uint64_t> aux(L);
        for (int l = 0; l < L; l++) {
            limb[l] = l;
            aux[l] = (qp[l] - hq[l]) % qp[l];
        }
        tc_build_basis(P, K, qp, limb.data(), aux.data(), L, (ModupTcTarget *)(base + lay.off_tc_tgt),
                       (ModupTcFrac *)(base + lay.off_tc_frac), (uint8_t *)(base + lay.off_tc_b));
        uint64_t *qi = (uint64_t *)(base + lay.off_tc_qinv);
        for (int a = 0; a < K; a++) {
            uint64_t h = 1 % P[a];
            for (int b = 0; b < K; b++)
                if (b != a) h = mul_mod(h, P[b] % P[a], P[a]);
            qi[a * 2] = inv_mod(h, P[a]);                 // (P / p_a)^-1 mod p_a
            qi[a * 2 + 1] = shoup(qi[a * 2], P[a]);
        }
    }
    return FHE_OK;
}

// ---- host self-test of the device arithmetic (same code, host build) ----

namespace fhe {

int selftest_arith(uint64_t seed, int iters) {
    uint64_t s = seed ? seed : 0x9E3779B97F4A7C15ull;
    auto next = [&]() {  // xorshift64*
        s ^= s >> 12; s ^= s << 25; s ^= s >> 27;
        return s * 2685821657736338717ull;
    };
    uint64_t primes[8];
    if (fhe_find_primes(17, 50, 4, 0, primes) != FHE_OK) return 1;
    if (fhe_find_primes(11, 49, 4, 0, primes + 4) != FHE_OK) return 2;
    primes[7] = primes[7];
    for (int pi = 0; pi < 8; pi++) {
        const uint64_t q = primes[pi];
        if (q <= (1ull << 48)) continue;
        const uint64_t mu12 = (uint64_t)(((u128)1 << 100) / q) << 12;
        const uint32_t c58 = (uint32_t)((1ull << 58) / q);
        for (int it = 0; it < iters; it++) {
            uint64_t a = next() % q, b = next() % q;
            if (it < 4) { a = (it & 1) ? q - 1 : 0; b = (it & 2) ? q - 1 : 1; }
            const uint64_t ref = mul_mod(a, b, q);
            if (mulmod(a, b, q, mu12) != ref) return 10;
            const uint64_t y = next() >> (2 + (it % 8));      // up to 62 bits
            const uint64_t r = shoup_lazy(y, a, shoup(a, q), q);
            if (r >= 4 * q || r % q != mul_mod(y % q, a, q)) return 11;
            const uint64_t x = next() >> 6;                     // < 2^58
            if (reduce_small(x, q, c58) != x % q) return 12;
            uint64_t h = 0, l = 0;
            for (int k = 0; k < 1 + it % 24; k++) mac128(h, l, next() % q, next() % q);
            const u128 T = ((u128)h << 64) | l;
            if (barrett_reduce128(h, l, q, mu12, c58) != (uint64_t)(T % q)) return 13;
            // sums of up to 16 products of reduced values, with an extra term
            Mac25 acc;
            u128 ref_sum = 0;
            const int terms = 1 + it % 16;
            for (int k = 0; k < terms; k++) {
                uint64_t v = next() % q, m = next() % q;
                if (it % 5 == 0) { v = q - 1; m = q - 1; }
                mac25(acc, split25(v), split25(m));
                ref_sum += (u128)v * m;
            }
            const uint64_t extra = it % 3 == 0 ? next() % q : 0;
            if (mac25_reduce(acc, extra, q, mu12, c58) != (uint64_t)((ref_sum + extra) % q)) return 14;
            // the lazy form: congruent, below (4 + terms) q
            const uint64_t lz = mac25_reduce_lazy(acc, extra, q, mu12);
            if (lz % q != (uint64_t)((ref_sum + extra) % q) || lz >= (uint64_t)(4 + terms) * q) return 15;
            // the 64-bit reduction with mu = floor(2^64 / q): congruent, below 2q, for any word
            const uint64_t w = it % 7 == 0 ? ~0ull - (uint64_t)(it % 3) : next();
            const uint64_t r64 = reduce64_small_mu(w, q, (uint64_t)(((u128)1 << 64) / q));
            if (r64 >= 2 * q || r64 % q != w % q) return 16;
        }
    }
    return 0;
}

}  // namespace fhe

extern "C" int fhe_selftest_host(uint64_t seed, int iters) {
    return fhe::selftest_arith(seed, iters) == 0 ? FHE_OK : FHE_EINVAL;
}

extern "C" int fhe_ntt_fwd_table_slot(int log_n, uint32_t k, uint32_t *slot) {
    if (!slot || log_n < 1 || log_n > kMaxLogN || k >= (1u << log_n)) return FHE_EINVAL;
    *slot = fwd_table_slot(log_n, k);
    return FHE_OK;
}
