// automorph.cu -- Galois automorphism sigma_k: a(X) -> a(X^k), k odd.
//
// NTT domain.  Row position i holds a(zeta_i), zeta_i = psi^(2 brv(i) + 1), so
// sigma_k(a)(zeta_i) = a(zeta_i^k) = row[j] with 2 brv(j) + 1 = k (2 brv(i) + 1)
// mod 2n: a pure permutation.  Multiplying by an odd k modulo 2^(t+1) maps
// residue classes to residue classes, so the top t bits of i (the low bits of
// brv(i)) fix the top t bits of j: every contiguous output block of 2^LB
// positions reads one contiguous input block.  Each CTA stages that input
// block in shared memory with coalesced 16-byte loads and writes its output
// block with coalesced stores -- one HBM pass each way.
//
// Coefficient domain.  Coefficient t moves to s = t k mod 2n (negated when
// s >= n since X^n = -1); each output s gathers from t = s k^-1 mod 2n.
#include <cuda_runtime.h>

#include "fhe_arith.cuh"
#include "fhe_internal.h"
#include "launch_util.h"

namespace fhe {
namespace {

constexpr int kThreads = 256;
constexpr int kLogBlock = 11;   // 2048 residues = 16 KB of shared memory per CTA

__device__ __forceinline__ uint32_t brv_bits(uint32_t x, int bits) { return __brev(x) >> (32 - bits); }

// NTT-domain source position of output position i.
__device__ __forceinline__ uint32_t aut_src(uint32_t i, int log_n, uint32_t k) {
    const uint32_t m = brv_bits(i, log_n);
    const uint32_t e = (k * (2u * m + 1u)) & ((2u << log_n) - 1u);   // mod 2n (wrapping product is exact mod 2^32)
    return brv_bits((e - 1u) >> 1, log_n);
}

__global__ void __launch_bounds__(kThreads)
k_aut_ntt(uint64_t *__restrict__ out, const uint64_t *__restrict__ in, int log_n, int lb, uint32_t k) {
    pdl_begin();
    extern __shared__ __align__(16) uint64_t blk[];
    const int per_row = log_n - lb;
    const long row = (long)blockIdx.x >> per_row;
    const uint32_t ob = blockIdx.x & ((1u << per_row) - 1u);
    const uint32_t o0 = ob << lb;
    const uint32_t s0 = (aut_src(o0, log_n, k) >> lb) << lb;
    const uint64_t *src = in + (row << log_n) + s0;
    uint64_t *dst = out + (row << log_n) + o0;
    const int bs = 1 << lb;
    for (int x = 2 * threadIdx.x; x < bs; x += 2 * kThreads)
        *reinterpret_cast<ulonglong2 *>(blk + x) = __ldcs(reinterpret_cast<const ulonglong2 *>(src + x));
    __syncthreads();
    for (int x = 2 * threadIdx.x; x < bs; x += 2 * kThreads) {
        const uint64_t v0 = blk[aut_src(o0 + x, log_n, k) - s0];
        const uint64_t v1 = blk[aut_src(o0 + x + 1, log_n, k) - s0];
        __stcs(reinterpret_cast<ulonglong2 *>(dst + x), make_ulonglong2(v0, v1));
    }
}

__global__ void __launch_bounds__(kThreads)
k_aut_coeff(uint64_t *__restrict__ out, const uint64_t *__restrict__ in, long pairs, int log_n, int L,
            uint32_t kinv, const uint64_t *__restrict__ consts) {
    pdl_begin();
    const uint32_t n = 1u << log_n, mask2n = (2u << log_n) - 1u;
    const long stride = (long)gridDim.x * blockDim.x;
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < pairs; i += stride) {
        const long e = 2 * i;
        const long row = e >> log_n;
        const uint64_t q = __ldg(consts + ((uint32_t)row % (uint32_t)L) * K_COUNT + K_Q);   // rows < 2^30
        const uint64_t *src = in + (row << log_n);
        uint64_t v[2];
#pragma unroll
        for (int h = 0; h < 2; h++) {
            const uint32_t s = (uint32_t)(e & (n - 1)) + h;
            const uint32_t t1 = (s * kinv) & mask2n;
            const uint64_t a = __ldg(src + (t1 & (n - 1)));
            v[h] = (t1 & n) ? (a ? q - a : 0) : a;
        }
        __stcs(reinterpret_cast<ulonglong2 *>(out + e), make_ulonglong2(v[0], v[1]));
    }
}

}  // namespace

int launch_automorph(uint64_t *out, const uint64_t *in, int log_n, int L, long rows, uint64_t k, int domain,
                     const fhe_ntt_tables *t, void *stream) {
    cudaStream_t st = (cudaStream_t)stream;
    if (domain == FHE_DOMAIN_NTT) {
        const int lb = log_n < kLogBlock ? log_n : kLogBlock;
        const long blocks = rows << (log_n - lb);
        k_aut_ntt<<<(unsigned)blocks, kThreads, (size_t)8 << lb, st>>>(out, in, log_n, lb, (uint32_t)k);
    } else {
        // k^-1 mod 2n by Newton iteration on the 2-adic inverse (k odd).
        const uint64_t m = 2ull << log_n;
        uint64_t inv = k;                        // correct to 3 bits
        for (int i = 0; i < 5; i++) inv *= 2 - k * inv;
        inv &= m - 1;
        const long pairs = (rows << log_n) / 2;
        k_aut_coeff<<<stream_grid(pairs, kThreads, 8), kThreads, 0, st>>>(out, in, pairs, log_n, L, (uint32_t)inv,
                                                                          t->consts);
    }
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

}  // namespace fhe
