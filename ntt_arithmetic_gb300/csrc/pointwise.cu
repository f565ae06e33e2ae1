// pointwise.cu -- NTT-domain coefficient-wise kernels: pointwise product,
// ciphertext tensor product and the key-switch inner product.  All are
// HBM-streaming: one pass per operand, 16-byte accesses, persistent grids of
// a few CTAs per SM with grid-stride loops.  Variable x variable products use
// Barrett reduction (fhe_arith.cuh); sums of products are accumulated exactly
// in 128 bits and reduced once.
#include <cuda_runtime.h>

#include "fhe_arith.cuh"
#include "fhe_internal.h"
#include "launch_util.h"

namespace fhe {
namespace {

constexpr int kThreads = 256;

// out = a * b mod q_l over [rows][n], rows = batch * L; processed in pairs.
// The grid walks the pairs from the end (the kernel before it in a step
// finished there, so the first reads find L2) and stores with the L2 policy
// (the next kernel reads this output).
__global__ void __launch_bounds__(kThreads)
k_mul(uint64_t *out, const uint64_t *a, const uint64_t *b, long pairs, int log_n, int L,
      const uint64_t *__restrict__ consts) {
    pdl_begin();
    const long stride = (long)gridDim.x * blockDim.x;
    for (long i0 = (long)blockIdx.x * blockDim.x + threadIdx.x; i0 < pairs; i0 += stride) {
        const long i = pairs - 1 - i0;
        const long e = 2 * i;
        const int l = (int)((uint32_t)(e >> log_n) % (uint32_t)L);
        const uint64_t q = __ldg(consts + l * K_COUNT + K_Q), mu = __ldg(consts + l * K_COUNT + K_MU12);
        const ulonglong2 va = __ldcs(reinterpret_cast<const ulonglong2 *>(a + e));
        const ulonglong2 vb = __ldcs(reinterpret_cast<const ulonglong2 *>(b + e));
        __stcg(reinterpret_cast<ulonglong2 *>(out + e), make_ulonglong2(mulmod(va.x, vb.x, q, mu), mulmod(va.y, vb.y, q, mu)));
    }
}

// d0 = a0 b0, d1 = a0 b1 + a1 b0, d2 = a1 b1 per batch item; d1 by Karatsuba,
// ((a0 + a1)(b0 + b1) - d0 - d2) mod q: three modular products instead of four.
// Stored with the L2 policy: the inverse NTT's block kernel reads the rows
// written last first.
__global__ void __launch_bounds__(kThreads)
k_tensor(uint64_t *d, const uint64_t *a, const uint64_t *b, long pairs, int log_n, int L,
         const uint64_t *__restrict__ consts) {
    pdl_begin();
    const long plane = (long)L << log_n;
    const long stride = (long)gridDim.x * blockDim.x;
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < pairs; i += stride) {
        const long e = 2 * i;                  // flat index over [batch][L][n]
        const uint32_t row = (uint32_t)(e >> log_n);   // rows < 2^30
        const uint32_t bi = row / (uint32_t)L;
        const int l = (int)(row - bi * (uint32_t)L);
        const long in_off = e + bi * plane;    // [batch][2][L][n]
        const long out_off = e + 2 * bi * plane;  // [batch][3][L][n]
        const uint64_t *kc = consts + l * K_COUNT;
        const uint64_t q = __ldg(kc + K_Q), mu = __ldg(kc + K_MU12);
        const ulonglong2 a0 = __ldcs(reinterpret_cast<const ulonglong2 *>(a + in_off));
        const ulonglong2 a1 = __ldcs(reinterpret_cast<const ulonglong2 *>(a + in_off + plane));
        const ulonglong2 b0 = __ldcs(reinterpret_cast<const ulonglong2 *>(b + in_off));
        const ulonglong2 b1 = __ldcs(reinterpret_cast<const ulonglong2 *>(b + in_off + plane));
        const uint64_t d0x = mulmod(a0.x, b0.x, q, mu), d0y = mulmod(a0.y, b0.y, q, mu);
        const uint64_t d2x = mulmod(a1.x, b1.x, q, mu), d2y = mulmod(a1.y, b1.y, q, mu);
        const uint64_t sx = mulmod(csub(a0.x + a1.x, q), csub(b0.x + b1.x, q), q, mu);   // sums reduced below q
        const uint64_t sy = mulmod(csub(a0.y + a1.y, q), csub(b0.y + b1.y, q), q, mu);
        const uint64_t d1x = csub(sx + 2 * q - d0x - d2x, q), d1y = csub(sy + 2 * q - d0y - d2y, q);
        __stcg(reinterpret_cast<ulonglong2 *>(d + out_off), make_ulonglong2(d0x, d0y));
        __stcg(reinterpret_cast<ulonglong2 *>(d + out_off + plane), make_ulonglong2(csub(d1x, q), csub(d1y, q)));
        __stcg(reinterpret_cast<ulonglong2 *>(d + out_off + 2 * plane), make_ulonglong2(d2x, d2y));
    }
}

// out[b][c][l][i] = sum_j ext[b][j][l][i] * keys[j][c][l][i] mod p_l.
// One thread owns a pair of coefficients of one limb for every batch item,
// so each key word is fetched from HBM once per call.  DN > 0 (dnum <= 4):
// the thread's keys are held in registers across the batch loop and every
// load of a batch item is issued before its products; DN = 0: any dnum.
template <int DN>
__global__ void __launch_bounds__(kThreads)
k_ks_ip(uint64_t *out, const uint64_t *ext, const uint64_t *keys, long pairs, int log_n, int LK, int dnum_rt,
        int batch, const uint64_t *__restrict__ consts) {
    pdl_begin();
    const int dnum = DN > 0 ? DN : dnum_rt;
    const long plane = (long)LK << log_n;      // one [LK][n] block
    const long stride = (long)gridDim.x * blockDim.x;
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < pairs; i += stride) {
        const long e = 2 * i;                   // flat index over [LK][n]
        const int l = (int)(e >> log_n);
        const uint64_t *kc = consts + l * K_COUNT;
        const uint64_t q = __ldg(kc + K_Q), mu = __ldg(kc + K_MU12);
        const uint32_t c58 = (uint32_t)__ldg(kc + K_C58);
        if constexpr (DN > 0) {
            ulonglong2 k0[DN], k1[DN];
#pragma unroll
            for (int j = 0; j < DN; j++) {
                k0[j] = __ldcs(reinterpret_cast<const ulonglong2 *>(keys + (2L * j) * plane + e));
                k1[j] = __ldcs(reinterpret_cast<const ulonglong2 *>(keys + (2L * j + 1) * plane + e));
            }
            for (int bi = 0; bi < batch; bi++) {
                ulonglong2 dv[DN];
#pragma unroll
                for (int j = 0; j < DN; j++)
                    dv[j] = __ldcs(reinterpret_cast<const ulonglong2 *>(ext + ((long)bi * DN + j) * plane + e));
                uint64_t h0x = 0, l0x = 0, h0y = 0, l0y = 0, h1x = 0, l1x = 0, h1y = 0, l1y = 0;
#pragma unroll
                for (int j = 0; j < DN; j++) {
                    mac128(h0x, l0x, dv[j].x, k0[j].x);
                    mac128(h0y, l0y, dv[j].y, k0[j].y);
                    mac128(h1x, l1x, dv[j].x, k1[j].x);
                    mac128(h1y, l1y, dv[j].y, k1[j].y);
                }
                uint64_t *o = out + (long)bi * 2 * plane + e;
                __stcs(reinterpret_cast<ulonglong2 *>(o), make_ulonglong2(barrett_reduce128(h0x, l0x, q, mu, c58),
                                                                       barrett_reduce128(h0y, l0y, q, mu, c58)));
                __stcs(reinterpret_cast<ulonglong2 *>(o + plane),
                       make_ulonglong2(barrett_reduce128(h1x, l1x, q, mu, c58), barrett_reduce128(h1y, l1y, q, mu, c58)));
            }
        } else {
            for (int bi = 0; bi < batch; bi++) {
                uint64_t h0x = 0, l0x = 0, h0y = 0, l0y = 0, h1x = 0, l1x = 0, h1y = 0, l1y = 0;
                for (int j = 0; j < dnum; j++) {
                    const ulonglong2 dv =
                        __ldcs(reinterpret_cast<const ulonglong2 *>(ext + ((long)bi * dnum + j) * plane + e));
                    const ulonglong2 k0 = __ldg(reinterpret_cast<const ulonglong2 *>(keys + (2L * j) * plane + e));
                    const ulonglong2 k1 = __ldg(reinterpret_cast<const ulonglong2 *>(keys + (2L * j + 1) * plane + e));
                    mac128(h0x, l0x, dv.x, k0.x);
                    mac128(h0y, l0y, dv.y, k0.y);
                    mac128(h1x, l1x, dv.x, k1.x);
                    mac128(h1y, l1y, dv.y, k1.y);
                }
                uint64_t *o = out + (long)bi * 2 * plane + e;
                __stcs(reinterpret_cast<ulonglong2 *>(o), make_ulonglong2(barrett_reduce128(h0x, l0x, q, mu, c58),
                                                                       barrett_reduce128(h0y, l0y, q, mu, c58)));
                __stcs(reinterpret_cast<ulonglong2 *>(o + plane),
                       make_ulonglong2(barrett_reduce128(h1x, l1x, q, mu, c58), barrett_reduce128(h1y, l1y, q, mu, c58)));
            }
        }
    }
}

}  // namespace

int launch_mul(uint64_t *out, const uint64_t *a, const uint64_t *b, int log_n, int L, long rows,
               const fhe_ntt_tables *t, void *stream) {
    const long pairs = (rows << log_n) / 2;
    k_mul<<<stream_grid(pairs, kThreads, 8), kThreads, 0, (cudaStream_t)stream>>>(out, a, b, pairs, log_n, L, t->consts);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

// The tensor product's grid: two whole rounds of its resident CTAs per SM.
// At 48 registers 5 CTAs of 256 threads are resident; a grid of 8 per SM left
// a partial second round (the 2100-prime chain's tensor product 9 us slower
// per step, measured against 5 and 10 per SM).
static int tensor_ctas_per_sm() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 8;
    if (cache[dev] == 0) {
        int nb = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, k_tensor, kThreads, 0) != cudaSuccess || nb <= 0) {
            cudaGetLastError();
            nb = 4;
        }
        cache[dev] = 2 * nb;
    }
    return cache[dev];
}

int launch_tensor(uint64_t *d, const uint64_t *a, const uint64_t *b, int log_n, int L, int batch,
                  const fhe_ntt_tables *t, void *stream) {
    const long pairs = ((long)batch * L << log_n) / 2;
    k_tensor<<<stream_grid(pairs, kThreads, tensor_ctas_per_sm()), kThreads, 0, (cudaStream_t)stream>>>(
        d, a, b, pairs, log_n, L, t->consts);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

int launch_ks_ip(uint64_t *out, const uint64_t *ext, const uint64_t *keys, int log_n, int LK, int dnum, int batch,
                 const fhe_ntt_tables *t, void *stream) {
    const long pairs = ((long)LK << log_n) / 2;
    auto kern = dnum == 1 ? k_ks_ip<1> : dnum == 2 ? k_ks_ip<2> : dnum == 3 ? k_ks_ip<3> : dnum == 4 ? k_ks_ip<4>
                                                                                                     : k_ks_ip<0>;
    kern<<<stream_grid(pairs, kThreads, 8), kThreads, 0, (cudaStream_t)stream>>>(out, ext, keys, pairs, log_n, LK, dnum,
                                                                                  batch, t->consts);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

}  // namespace fhe
