// fhe_arith.cuh -- 64-bit modular arithmetic for primes 2^48 < q < 2^50,
// written for the integer pipes of sm_103a and usable on the host as well
// (the same code path is exercised by the library's host self-test).
//
// Cost model (measured on GB300 with a register-resident microbenchmark):
// 32-bit mul.lo issues at 64/clk/SM, mul.hi and mul.wide at ~32 and ~25/clk/SM
// (twice the cost), adds and logic run on a separate pipe.  The butterflies
// below therefore minimise hi/wide partial products and keep every reduction
// that is not strictly needed out of the inner loop (Harvey's lazy bounds).
#pragma once
#include <cstdint>

#if defined(__CUDACC__)
#define FHE_HD __host__ __device__ __forceinline__
#else
#define FHE_HD inline
#endif

namespace fhe {

FHE_HD uint32_t lo32(uint64_t x) { return (uint32_t)x; }
FHE_HD uint32_t hi32(uint64_t x) { return (uint32_t)(x >> 32); }

FHE_HD uint32_t umulhi32(uint32_t a, uint32_t b) {
#if defined(__CUDA_ARCH__)
    return __umulhi(a, b);
#else
    return (uint32_t)(((uint64_t)a * b) >> 32);
#endif
}

FHE_HD uint64_t umulhi64(uint64_t a, uint64_t b) {
#if defined(__CUDA_ARCH__)
    return __umul64hi(a, b);
#else
    return (uint64_t)(((unsigned __int128)a * b) >> 64);
#endif
}

// x - c if x >= c, else x
FHE_HD uint64_t csub(uint64_t x, uint64_t c) { return x >= c ? x - c : x; }

// Per-prime constants, one row of 16 words per prime in the table blob.
enum ConstSlot {
    K_Q = 0,          // q
    K_MU12 = 1,       // floor(2^100 / q) << 12       (Barrett, full products)
    K_C58 = 2,        // floor(2^58 / q)              (small-quotient reduction)
    K_NINV = 3,       // n^-1 mod q
    K_PSI = 4,        // psi (smallest primitive 2n-th root)
    K_COUNT = 16
};

// Lazy Shoup product.  V. Shoup's precomputed-quotient multiplication by a
// fixed w (as in NTL's MulModPrecon), with D. Harvey's lazy output range
// ("Faster arithmetic for number-theoretic transforms", J. Symb. Comp. 2014):
// for w < q, wp = floor(w 2^64 / q) and any y < 2^62, returns r = w y - Q q
// with 0 <= r < 4q.  The quotient Q uses three 32x32 partial products of
// wp * y -- the low x low term is dropped -- so Q is at most 3 below
// floor(w y / q) and never above it.
FHE_HD uint64_t shoup_lazy(uint64_t y, uint64_t w, uint64_t wp, uint64_t q) {
#if defined(__CUDA_ARCH__)
    // The same arithmetic as the host branch, written as one multiply-add
    // chain: r = (w y + Q (2^64 - q)) mod 2^64 from two wide and four low
    // products, Q from one wide and two high products (measured ~18% more
    // butterflies per clock on sm_103a than the compiler's form).
    const uint64_t nq = 0 - q;
    uint64_t r;
    asm("{\n\t"
        ".reg .u32 yl, yh, wl, wh, pl, ph, nl, nh, t1, t2, ql, qh, rl, rh;\n\t"
        ".reg .u64 Q, R;\n\t"
        "mov.b64 {yl, yh}, %1;\n\t"
        "mov.b64 {wl, wh}, %2;\n\t"
        "mov.b64 {pl, ph}, %3;\n\t"
        "mov.b64 {nl, nh}, %4;\n\t"
        "mul.hi.u32 t1, ph, yl;\n\t"
        "mul.hi.u32 t2, pl, yh;\n\t"
        "add.cc.u32 t1, t1, t2;\n\t"
        "addc.u32 t2, 0, 0;\n\t"
        "mov.b64 Q, {t1, t2};\n\t"
        "mad.wide.u32 Q, ph, yh, Q;\n\t"
        "mov.b64 {ql, qh}, Q;\n\t"
        "mul.wide.u32 R, wl, yl;\n\t"
        "mad.wide.u32 R, ql, nl, R;\n\t"
        "mov.b64 {rl, rh}, R;\n\t"
        "mad.lo.u32 rh, wl, yh, rh;\n\t"
        "mad.lo.u32 rh, wh, yl, rh;\n\t"
        "mad.lo.u32 rh, ql, nh, rh;\n\t"
        "mad.lo.u32 rh, qh, nl, rh;\n\t"
        "mov.b64 %0, {rl, rh};\n\t"
        "}"
        : "=l"(r)
        : "l"(y), "l"(w), "l"(wp), "l"(nq));
    return r;
#else
    const uint32_t yl = lo32(y), yh = hi32(y), wl = lo32(wp), wh = hi32(wp);
    const uint64_t Q = (uint64_t)wh * yh + umulhi32(wh, yl) + umulhi32(wl, yh);
    return w * y - Q * q;
#endif
}

// Reduction of x < 2^58 into [0, q) with one 32x32 high product (a Barrett
// step on the top 32 bits): Q = floor((x >> 26) * c58 / 2^32), c58 =
// floor(2^58 / q), lies in (x/q - 3, x/q], so x - Q q < 3q.
FHE_HD uint64_t reduce_small(uint64_t x, uint64_t q, uint32_t c58) {
    const uint32_t Q = umulhi32((uint32_t)(x >> 26), c58);
    uint64_t r = x - (uint64_t)Q * q;
    r = csub(r, 2 * q);
    return csub(r, q);
}

// Barrett reduction (P. Barrett, CRYPTO '86) of a 128-bit value T = hi:lo
// with T < 2^105: x = floor(T / 2^48), Q = floor(x mu / 2^52) with
// mu = floor(2^100 / q), so T - Q q < (3 + T / 2^100) q < 2^58 and the
// small-quotient step finishes the reduction.
FHE_HD uint64_t barrett_reduce128(uint64_t hi, uint64_t lo, uint64_t q, uint64_t mu12, uint32_t c58) {
    const uint64_t x = (hi << 16) | (lo >> 48);
    const uint64_t Q = umulhi64(x, mu12);
    return reduce_small(lo - Q * q, q, c58);
}

// a * b mod q exactly, for a, b < q (Barrett with mu = floor(2^100/q)):
// T = a b < 2^100, so T - Q q < 3q.
FHE_HD uint64_t mulmod(uint64_t a, uint64_t b, uint64_t q, uint64_t mu12) {
    const uint64_t lo = a * b, hi = umulhi64(a, b);
    const uint64_t x = (hi << 16) | (lo >> 48);
    const uint64_t Q = umulhi64(x, mu12);
    uint64_t r = lo - Q * q;
    r = csub(r, 2 * q);
    return csub(r, q);
}

// 128-bit multiply-accumulate: (hi:lo) += a * b
FHE_HD void mac128(uint64_t &hi, uint64_t &lo, uint64_t a, uint64_t b) {
    const uint64_t pl = a * b, ph = umulhi64(a, b);
    lo += pl;
    hi += ph + (lo < pl ? 1 : 0);
}

// Exact sums of products sum_a v_a m_a for v_a, m_a < 2^50 and at most 16
// terms, reduced once: the sums of basis extensions (ModUp, ModDown, basis
// conversion), where every product is by a different constant (stored
// pre-split in the tables).  Each factor
// is split into 25-bit halves, v = v1 2^25 + v0, and the three column sums
// s0 = sum v0 m0, s1 = sum v1 m1, s01 = sum (v0 + v1)(m0 + m1) are kept in
// 64-bit words (Karatsuba: the middle column is s01 - s0 - s1).  Every
// product is one 32x32 -> 64 multiply-add and no high half is needed, against
// two high and three wide products for a Shoup product.  Bounds: s0, s1 <
// 16 2^50 = 2^54, s01 < 16 2^52 = 2^56.
struct Split25 {
    uint32_t lo, hi, sum;   // v0, v1, v0 + v1
};
FHE_HD Split25 split25(uint64_t v) {
    const uint32_t lo = (uint32_t)v & 0x1FFFFFFu, hi = (uint32_t)(v >> 25);
    return {lo, hi, lo + hi};
}
// A constant factor m < 2^50 stored split, as the two words of a table entry:
// word 0 = m0 | m1 << 32, word 1 = m0 + m1.
FHE_HD void split25_store(uint64_t m, uint64_t *entry) {
    const Split25 s = split25(m);
    entry[0] = (uint64_t)s.lo | (uint64_t)s.hi << 32;
    entry[1] = s.sum;
}
FHE_HD Split25 split25_entry(uint64_t w0, uint64_t w1) { return {(uint32_t)w0, (uint32_t)(w0 >> 32), (uint32_t)w1}; }
struct Mac25 {
    uint64_t s0 = 0, s1 = 0, s01 = 0;
};
FHE_HD void mac25(Mac25 &acc, const Split25 &v, const Split25 &m) {
#if defined(__CUDA_ARCH__)
    asm("mad.wide.u32 %0, %3, %4, %0;\n\t"
        "mad.wide.u32 %1, %5, %6, %1;\n\t"
        "mad.wide.u32 %2, %7, %8, %2;"
        : "+l"(acc.s0), "+l"(acc.s1), "+l"(acc.s01)
        : "r"(v.lo), "r"(m.lo), "r"(v.hi), "r"(m.hi), "r"(v.sum), "r"(m.sum));
#else
    acc.s0 += (uint64_t)v.lo * m.lo;
    acc.s1 += (uint64_t)v.hi * m.hi;
    acc.s01 += (uint64_t)v.sum * m.sum;
#endif
}
// X = s1 2^50 + (s01 - s0 - s1) 2^25 + s0 + extra < 2^105 (extra < 2^60) as
// a 128-bit hi:lo.
FHE_HD void mac25_combine(const Mac25 &acc, uint64_t extra, uint64_t &hi, uint64_t &lo) {
    const uint64_t mid = acc.s01 - acc.s0 - acc.s1;
    lo = acc.s0 + extra;
    hi = 0;
    uint64_t t = mid << 25;
    lo += t;
    hi += (mid >> 39) + (lo < t ? 1 : 0);
    t = acc.s1 << 50;
    lo += t;
    hi += (acc.s1 >> 14) + (lo < t ? 1 : 0);
}

// (sum + extra) mod q, through barrett_reduce128.
FHE_HD uint64_t mac25_reduce(const Mac25 &acc, uint64_t extra, uint64_t q, uint64_t mu12, uint32_t c58) {
    uint64_t hi, lo;
    mac25_combine(acc, extra, hi, lo);
    return barrett_reduce128(hi, lo, q, mu12, c58);
}

// The Barrett step of mac25_reduce without the final small-quotient
// reduction: a value congruent to X mod q below (3 + X / 2^100) q -- e.g.
// < 11 q for the up to 8 terms of a digit's basis extension.  For results
// that feed a forward NTT, whose lazy butterflies accept inputs of this size.
FHE_HD uint64_t mac25_reduce_lazy(const Mac25 &acc, uint64_t extra, uint64_t q, uint64_t mu12) {
    uint64_t hi, lo;
    mac25_combine(acc, extra, hi, lo);
    const uint64_t x = (hi << 16) | (lo >> 48);
    return lo - umulhi64(x, mu12) * q;
}

// Forward (Cooley-Tukey) butterfly with the psi-merged twiddle w (Roy et
// al./Poppelmann et al. merged negacyclic NTT) and Harvey's lazy additive
// bound: if X, Y < B then X', Y' < B + 4q.  No comparison at all.
FHE_HD void ct_bfly(uint64_t &X, uint64_t &Y, uint64_t w, uint64_t wp, uint64_t q) {
    const uint64_t t = shoup_lazy(Y, w, wp, q);
    const uint64_t x = X;
    X = x + t;
    Y = x - t + 4 * q;
}

// Butterfly with twiddle 1 (the first stages of the cyclic inverse): if
// X, Y < b then X + Y < 2b and X - Y + b < 2b.  `b` must bound Y.
FHE_HD void ct_bfly_one(uint64_t &X, uint64_t &Y, uint64_t b) {
    const uint64_t x = X, y = Y;
    X = x + y;
    Y = x - y + b;
}

// x mod p up to 2p for any 64-bit x, with mu = floor(2^64 / p) and p > 2^48
// (so mu < 2^16): Q = floor(x mu / 2^64) is computed exactly from the 32-bit
// halves (x_hi mu + floor(x_lo mu / 2^32)) >> 32, and x/p - 2 < Q <= x/p,
// so x - Q p lies in [0, 2p).  Two wide, one high and one low product.
FHE_HD uint64_t reduce64_small_mu(uint64_t x, uint64_t p, uint64_t mu) {
    const uint32_t m = (uint32_t)mu;
    const uint64_t t = (uint64_t)hi32(x) * m + umulhi32(lo32(x), m);
    const uint32_t Q = (uint32_t)(t >> 32);
    return x - ((uint64_t)Q * lo32(p) + ((uint64_t)(Q * hi32(p)) << 32));
}

// [0, 4q) -> [0, q)
FHE_HD uint64_t reduce4(uint64_t x, uint64_t q) { return csub(csub(x, 2 * q), q); }

}  // namespace fhe
