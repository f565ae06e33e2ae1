// modup.cu -- exact basis extension (ModUp) of every key-switch digit.
//
// For digit j with primes d_0..d_{a-1} and one coefficient with residues
// x_0..x_{a-1}, Garner's algorithm gives the mixed-radix digits of the CRT
// integer X in [0, d_0 ... d_{a-1}):
//   v_0 = x_0,  v_i = ((((x_i - v_0) d_0^-1 - v_1) d_1^-1 ...) - v_{i-1}) d_{i-1}^-1 mod d_i,
// and X mod p = v_0 + v_1 d_0 + v_2 d_0 d_1 + ... (mod p) for every prime p of
// the extended basis.  This is the "mixed-radix decomposition and basis
// extension" of FHElium's CUDA layer ("Eager, Compile, and native
// execution", section "CUDA execution") and the "Garner extension" of the
// kestrel-llm chain (overview, section 4.2).  All constants are fixed per
// basis: Garner's recursion uses lazy Shoup products.
//
// The approximate variant replaces Garner's recursion by the CRT sum
//   X + e D = sum_a [x_a (D / d_a)^-1]_{d_a} (D / d_a),   0 <= e < alpha,
// reduced modulo each target prime without correcting e D: alpha products
// for the brackets, then alpha multiply-accumulates per target.
// The extension sums are exact multiply-accumulates of 25-bit halves with one
// Barrett step per target (mac25 in fhe_arith.cuh), left below (4 + alpha) q.  Each CTA stages its
// digit's extension weights and the targets' reduction constants in shared
// memory, so the inner loop reads them as broadcasts.
#include <cuda_runtime.h>

#include "fhe_arith.cuh"
#include "fhe_internal.h"
#include "launch_util.h"

namespace fhe {
namespace {

constexpr int kThreads = 256;

template <int MAXA, bool APPROX>
__global__ void __launch_bounds__(kThreads)
k_modup(uint64_t *__restrict__ ext, const uint64_t *__restrict__ in, long in_stride, int log_n, int LK, int dnum, int alpha,
        const ModupDigit *__restrict__ dg, const ulonglong2 *__restrict__ garner, const ulonglong2 *__restrict__ mr,
        const uint64_t *__restrict__ consts) {
    pdl_begin();
    // APPROX: `garner` holds the bracket constants [dnum][alpha] and `mr` the
    // CRT weights [dnum][LK][alpha] of the approximate conversion.
    const long n = 1L << log_n;
    const int j = blockIdx.y, bi = blockIdx.z;
    const int lo = dg[j].lo, cnt = dg[j].count;
    const ulonglong2 *gj = garner + (long)j * alpha * (APPROX ? 1 : alpha);
    // this digit's extension weights and the targets' constants, staged in shared memory
    __shared__ ulonglong2 s_mr[kMaxBasis * MAXA];
    __shared__ ulonglong2 s_qm[kMaxBasis];     // (q, floor(2^100 / q) << 12)
    {
        const ulonglong2 *src_mr = mr + (long)j * LK * alpha;
        for (int e = threadIdx.x; e < LK * MAXA; e += blockDim.x) {
            const int l = e / MAXA, a = e - l * MAXA;
            s_mr[e] = a < alpha ? __ldg(src_mr + l * alpha + a) : make_ulonglong2(0, 0);
        }
        for (int l = threadIdx.x; l < LK; l += blockDim.x) {
            const uint64_t *kc = consts + (long)l * K_COUNT;
            s_qm[l] = make_ulonglong2(__ldg(kc + K_Q), __ldg(kc + K_MU12));
        }
        __syncthreads();
    }
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
        uint64_t x[MAXA], v[MAXA];
        const uint64_t *src = in + (long)bi * in_stride + ((long)lo << log_n) + i;
#pragma unroll
        for (int a = 0; a < MAXA; a++) x[a] = a < cnt ? __ldcs(src + ((long)a << log_n)) : 0;
        if constexpr (APPROX) {
#pragma unroll
            for (int a = 0; a < MAXA; a++) {
                v[a] = 0;
                if (a < cnt) {
                    const uint64_t d = __ldg(consts + (long)(lo + a) * K_COUNT + K_Q);
                    const ulonglong2 c = __ldg(gj + a);
                    v[a] = reduce4(shoup_lazy(x[a], c.x, c.y, d), d);
                }
            }
        } else {
        v[0] = x[0];
#pragma unroll
        for (int a = 1; a < MAXA; a++) {
            v[a] = 0;
            if (a < cnt) {
                const uint64_t d = __ldg(consts + (long)(lo + a) * K_COUNT + K_Q);
                uint64_t u = x[a];
#pragma unroll
                for (int b = 0; b < a; b++) {
                    const ulonglong2 c = __ldg(gj + a * alpha + b);
                    u = shoup_lazy(u + 4 * d - v[b], c.x, c.y, d);   // v_b < 2^50 < 4 d
                }
                v[a] = reduce4(u, d);
            }
        }
        }
        uint64_t *dst = ext + (((long)bi * dnum + j) * LK << log_n) + i;
#pragma unroll
        for (int a = 0; a < MAXA; a++)
            if (a < cnt) __stcs(dst + ((long)(lo + a) << log_n), x[a]);   // limbs of the digit are copies
        Split25 vs[MAXA];
#pragma unroll
        for (int a = 0; a < MAXA; a++) vs[a] = split25(v[a]);
        for (int l = 0; l < LK; l++) {
            if (l >= lo && l < lo + cnt) continue;
            Mac25 acc;
#pragma unroll
            for (int a = APPROX ? 0 : 1; a < MAXA; a++) {
                if (a < cnt) {
                    const ulonglong2 m = s_mr[l * MAXA + a];
                    mac25(acc, vs[a], split25_entry(m.x, m.y));
                }
            }
            const ulonglong2 qm = s_qm[l];
            // exact: the weight of v_0 is 1.  Stored below (4 + alpha) q (< 11 q at
            // alpha = 8), not fully reduced: the extended digits only feed the
            // forward NTT, whose lazy butterflies and final reduction take inputs
            // of that size (every value stays below 2^57).
            __stcs(dst + ((long)l << log_n), mac25_reduce_lazy(acc, APPROX ? 0 : v[0], qm.x, qm.y));
        }
    }
}

template <int MAXA>
void launch_modup_t(uint64_t *ext, const uint64_t *in, long in_stride, int log_n, int L, int K, int dnum, int batch,
                    bool approx, const fhe_ntt_tables *t, const void *modup, cudaStream_t st) {
    const ModupLayout lay = modup_layout(L, K, dnum);
    const char *base = (const char *)modup;
    const long n = 1L << log_n;
    // one coefficient per thread: at 4 resident CTAs per SM a capped
    // grid-stride grid left a partial last wave of long CTAs, while 2^8-
    // coefficient CTAs let the block scheduler even out the tail (measured
    // 3 % faster key switch at n = 2^16, batch 4)
    const long bx = (n + kThreads - 1) / kThreads;
    dim3 grid((unsigned)bx, (unsigned)dnum, (unsigned)batch);
    auto kern = approx ? k_modup<MAXA, true> : k_modup<MAXA, false>;
    kern<<<grid, kThreads, 0, st>>>(ext, in, in_stride, log_n, L + K, dnum, lay.alpha,
                                    (const ModupDigit *)(base + lay.off_digits),
                                    (const ulonglong2 *)(base + (approx ? lay.off_qinv : lay.off_garner)),
                                    (const ulonglong2 *)(base + (approx ? lay.off_qhat : lay.off_mr)), t->consts);
}

}  // namespace

int launch_modup(uint64_t *ext, const uint64_t *in, long in_stride, int log_n, int L, int K, int dnum, int batch,
                 bool approx, const fhe_ntt_tables *t, const void *modup, void *stream) {
    cudaStream_t st = (cudaStream_t)stream;
    const int tc = launch_modup_tc(ext, in, in_stride, log_n, L, K, dnum, batch, approx, t, modup, stream);
    if (tc != 0) return tc;   // the tensor-core extension ran (or failed to launch)
    const int alpha = modup_layout(L, K, dnum).alpha;
    if (alpha <= 1) launch_modup_t<1>(ext, in, in_stride, log_n, L, K, dnum, batch, approx, t, modup, st);
    else if (alpha <= 2) launch_modup_t<2>(ext, in, in_stride, log_n, L, K, dnum, batch, approx, t, modup, st);
    else if (alpha <= 4) launch_modup_t<4>(ext, in, in_stride, log_n, L, K, dnum, batch, approx, t, modup, st);
    else if (alpha <= 8) launch_modup_t<8>(ext, in, in_stride, log_n, L, K, dnum, batch, approx, t, modup, st);
    else launch_modup_t<16>(ext, in, in_stride, log_n, L, K, dnum, batch, approx, t, modup, st);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

}  // namespace fhe
