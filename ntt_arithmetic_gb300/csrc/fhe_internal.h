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
struct ModupLayout {
    int alpha;
    size_t off_digits, off_garner, off_mr, bytes;
};
ModupLayout modup_layout(int L, int K, int dnum);
bool modup_shape_ok(int L, int K, int dnum);

// ModDown constants for Q = (q_0..q_{L-1}), P = (p_0..p_{K-1}).
struct ModdownLayout {
    size_t off_garner;   // [K][K] pairs: p_b^-1 mod p_a (b < a)
    size_t off_mr;       // [L][K] pairs: prod_{b<a} p_b mod q_l
    size_t off_hp;       // [K] words: (P-1)/2 mod p_k
    size_t off_hq;       // [L] words: (P-1)/2 mod q_l
    size_t off_pinv;     // [L] pairs: P^-1 mod q_l
    size_t bytes;
};
ModdownLayout moddown_layout(int L, int K);

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
                 const fhe_ntt_tables *t, const void *modup, void *stream);
int launch_ks_ip(uint64_t *out, const uint64_t *ext, const uint64_t *keys, int log_n, int LK,
                 int dnum, int batch, const fhe_ntt_tables *t, void *stream);

int launch_moddown(uint64_t *out, const uint64_t *in, int log_n, int L, int K, int batch, bool ntt_domain,
                   bool nearest, const fhe_ntt_tables *t_qp, const void *md, uint64_t *ws, void *stream);

// Tables view shifted to limbs [first, first + count) of t (no copy).
fhe_ntt_tables tables_slice(const fhe_ntt_tables *t, int first, int count);

void count_launches(int k);

}  // namespace fhe
