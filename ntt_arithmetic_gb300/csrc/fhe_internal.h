// fhe_internal.h -- declarations shared by the translation units of
// libfhe_ntt.so (never installed; the public ABI is include/fhe_ntt.h).
#pragma once
#include <cstddef>
#include <cstdint>

#include "../../include/fhe_ntt.h"

namespace fhe {

constexpr int kMaxLogN = 17;      // n up to 2^17
constexpr int kMaxTableL = 8192;  // primes per table blob
constexpr int kMaxBasis = 64;     // L + K of a key switch
constexpr int kMaxAlpha = 16;     // primes per key-switch digit

struct NttLayout {
    size_t off_q, off_consts, off_fwd, off_inv, off_twist, bytes;
};
NttLayout ntt_layout(int log_n, int L);

struct ModupDigit {
    int32_t lo;      // first limb of the digit
    int32_t count;   // limbs in the digit (<= alpha)
};
// Per prime d_a of a digit, the constants of the tensor-core extension's
// exact correction (modup_tc.cu): phi = floor(2^128 / d_a) as (hi, lo) words
// for the fixed-point sum of y_a / d_a, and for the redundant-modulus
// fallback (D / d_a) mod 2^64 and d_0 ... d_{a-1} mod 2^64.  Entry
// kTcMaxAlpha of each digit holds D^-1 mod 2^64 in `dhat64`.
struct ModupTcFrac {
    uint64_t phi_hi, phi_lo, dhat64, w64;
};
// One target prime of a digit's tensor-core extension (modup_tc.cu).
struct ModupTcTarget {
    uint64_t p;      // the target prime
    uint64_t mu;     // floor(2^64 / p) (< 2^16)
    uint64_t aux;    // added to each output by ModDown with nearest rounding: (p - h) mod p; 0 for ModUp
    uint64_t limb;   // index of p in the extended basis
};
// The tensor-core extension takes digits of up to kTcMaxAlpha primes: one
// digit's mixed-radix digits are 8 alpha = 64 fp16 byte limbs (K), and the
// accumulators of up to kTcTargetsPerGroup targets (8 columns each) fill the
// 128 TMEM columns a CTA holds.
constexpr int kTcMaxAlpha = 8;
constexpr int kTcTargetsPerGroup = 16;
constexpr int kTcRowBytes = 8 * kTcMaxAlpha * 2;   // one operand row: 64 fp16
constexpr int kTcCorrCol = 15;                     // operand column of the correction count

struct ModupLayout {
    int alpha;
    size_t off_digits;   // [dnum] ModupDigit
    size_t off_garner;   // [dnum][alpha][alpha] pairs: d_b^-1 mod d_a (b < a)       (exact)
    size_t off_mr;       // [dnum][L+K][alpha] split factors: prod_{b<a} d_b mod qp_l (exact)
    size_t off_qinv;     // [dnum][alpha] pairs: (D_j / d_a)^-1 mod d_a                (approximate)
    size_t off_qhat;     // [dnum][L+K][alpha] split factors: (D_j / d_a) mod qp_l     (approximate)
    // tensor-core extension (alpha <= kTcMaxAlpha; tc_tmax = 0 otherwise):
    int tc_tmax;         // target slots per digit (L+K rounded up to even)
    size_t off_tc_tgt;   // [dnum][tc_tmax] ModupTcTarget
    size_t off_tc_frac;  // [dnum][kTcMaxAlpha + 1] ModupTcFrac
    size_t off_tc_b;     // [dnum][8 tc_tmax rows][64] fp16 weight limbs, operand layout
    size_t bytes;
};
ModupLayout modup_layout(int L, int K, int dnum);
bool modup_shape_ok(int L, int K, int dnum);

// ModDown constants for Q = (q_0..q_{L-1}), P = (p_0..p_{K-1}).
struct ModdownLayout {
    size_t off_garner;   // [K][K] pairs: p_b^-1 mod p_a (b < a)
    size_t off_mr;       // [L][K] split factors: prod_{b<a} p_b mod q_l
    // tensor-core conversion (K <= kTcMaxAlpha; tc_tmax = 0 otherwise), as ModupLayout's for one digit:
    int tc_tmax;         // target slots (L rounded up to even)
    size_t off_tc_qinv;  // [K] pairs: (P / p_a)^-1 mod p_a
    size_t off_tc_tgt;   // [tc_tmax] ModupTcTarget
    size_t off_tc_frac;  // [kTcMaxAlpha + 1] ModupTcFrac
    size_t off_tc_b;     // [8 tc_tmax rows][64] fp16 weight limbs
    size_t off_hp;       // [K] words: (P-1)/2 mod p_k
    size_t off_hq;       // [L] words: (P-1)/2 mod q_l
    size_t off_pinv;     // [L] pairs: P^-1 mod q_l
    size_t bytes;
};
ModdownLayout moddown_layout(int L, int K);

// Basis conversion from S source primes to T target primes.
constexpr int kMaxBconvSrc = 16;
struct BconvLayout {
    size_t off_src;      // [S] words: source primes
    size_t off_dst;      // [T][4] words: target prime, floor(2^58 / prime), floor(2^100 / prime) << 12, 0
    size_t off_garner;   // [S][S] pairs: q_b^-1 mod q_a (b < a)                      (exact)
    size_t off_mr;       // [T][S] split factors: prod_{b<a} q_b mod p_t              (exact)
    size_t off_qinv;     // [S] pairs: (Q / q_a)^-1 mod q_a                           (approximate)
    size_t off_qhat;     // [T][S] split factors: (Q / q_a) mod p_t                   (approximate)
    size_t bytes;
};
BconvLayout bconv_layout(int S, int T);

// "split factors" are 16-byte entries written by split25_store (fhe_arith.cuh).

// Galois elements of one hoisted key switch.
constexpr int kMaxRotations = 64;
struct GaloisSet {
    uint32_t k[kMaxRotations];
};

// ---- kernel launchers (no validation; the ABI layer validates) ----------
// Each returns the number of kernels enqueued, or -1 on a launch error.

int launch_ntt(uint64_t *res, int log_n, int L, long rows, const fhe_ntt_tables *t, bool inverse,
               void *stream);
int launch_mul(uint64_t *out, const uint64_t *a, const uint64_t *b, int log_n, int L, long rows,
               const fhe_ntt_tables *t, void *stream);
int launch_tensor(uint64_t *d, const uint64_t *a, const uint64_t *b, int log_n, int L, int batch,
                  const fhe_ntt_tables *t, void *stream);
int launch_automorph(uint64_t *out, const uint64_t *in, int log_n, int L, long rows, uint64_t k,
                     int domain, const fhe_ntt_tables *t, void *stream);
int launch_modup(uint64_t *ext, const uint64_t *in, long in_stride, int log_n, int L, int K, int dnum, int batch,
                 bool approx, const fhe_ntt_tables *t, const void *modup, void *stream);
// The tensor-core ModUp (modup_tc.cu); returns 0 without launching when the
// shape has no tensor-core form (alpha > kTcMaxAlpha, n < 128).
int launch_modup_tc(uint64_t *ext, const uint64_t *in, long in_stride, int log_n, int L, int K, int dnum, int batch,
                    bool approx, const fhe_ntt_tables *t, const void *modup, void *stream);
// ModDown's NTT-domain conversion d = ((X + h) mod P) - h mod q_l on the tensor
// cores (below 3 q_l); returns 0 without launching when K > kTcMaxAlpha or n < 128.
int launch_moddown_tc(uint64_t *d, const uint64_t *src, long src_item, int log_n, int L, int K, int batch, bool nearest,
                      const fhe_ntt_tables *t_qp, const void *md, void *stream);
// Synchronize the device, then read (and optionally clear) the status word
// of the tensor-core kernels.
int device_status(int *status, bool reset);
int launch_ks_ip_aut(uint64_t *out, const uint64_t *ext, const uint64_t *keys, int log_n, int LK, int dnum,
                     int batch, int R, const GaloisSet &g, const fhe_ntt_tables *t, void *stream);
int launch_bconv(uint64_t *out, const uint64_t *in, int log_n, int S, int T, int batch, bool approx,
                 const void *bconv, void *stream);
int launch_ks_ip(uint64_t *out, const uint64_t *ext, const uint64_t *keys, int log_n, int LK,
                 int dnum, int batch, const fhe_ntt_tables *t, void *stream);
// Forward NTT of the extended digits ext [batch][dnum][LK][n] (ModUp output,
// overwritten by the column stages) fused with the inner product into out
// [batch][2][LK][n].  Returns 0 without launching when no fused kernel
// exists for the shape (n < 2^14, dnum > 4): the caller then runs
// launch_ntt + launch_ks_ip.
// ModDown's forward NTT of its correction d [batch][L][n] (overwritten by
// the column stages) fused with the last step out = (in - NTT(d)) P^-1 mod q_l,
// in the NTT-domain input [batch][L+K][n] and pinv the blob's [L] (P^-1 mod
// q_l, Shoup companion) pairs.  Returns 0 without launching for n < 2^14: the
// caller then runs launch_ntt + its own last-step kernel.
// Inverse NTT of rows read from another buffer: row (b, l) of src at
// src + b * src_item + l * n (src unchanged), result in dst [batch][L][n].
// Returns 0 without launching for n < 2^14 (copy the rows, then launch_ntt).
int launch_ntt_inv_from(uint64_t *dst, const uint64_t *src, long src_item, int log_n, int L, int batch,
                        const fhe_ntt_tables *t, void *stream);
int launch_ntt_fwd_moddown(uint64_t *out, uint64_t *d, const uint64_t *in, int log_n, int L, int K, int batch,
                           const fhe_ntt_tables *t_q, const void *pinv, void *stream);
int launch_ntt_fwd_ip(uint64_t *out, uint64_t *ext, const uint64_t *keys, int log_n, int LK, int dnum, int batch,
                      const fhe_ntt_tables *t, void *stream);

int launch_moddown(uint64_t *out, const uint64_t *in, int log_n, int L, int K, int batch, bool ntt_domain,
                   bool nearest, const fhe_ntt_tables *t_qp, const void *md, uint64_t *ws, void *stream);

int launch_bfly_probe(uint64_t *out, int ctas, int iters, const fhe_ntt_tables *t, void *stream);

// Tables view shifted to limbs [first, first + count) of t (no copy).
fhe_ntt_tables tables_slice(const fhe_ntt_tables *t, int first, int count);

void count_launches(int k);

}  // namespace fhe
