// hoisted.cu -- inner product of a hoisted key switch: the automorphism of
// the extended digits fused into the key-switch multiply-accumulate.
//
// coeff_to_slot and slot_to_coeff, the two stages that the kestrel-llm boot
// profile reports as about 80% of a bootstrap (overview, section 4.2), are
// sums of Galois rotations of one ciphertext, each followed by a key switch.
// The digit decomposition, ModUp and NTT of the extended digits D_j depend only
// on the input, so they are done once; for each Galois element k_r
//   out[r][b][c][l][i] = sum_j D_j[b][l][pi_r(i)] * keys[r][j][c][l][i]  mod qp_l,
// where pi_r is the NTT-domain index map of sigma_{k_r} (row position i holds
// the value at psi^(2 brv(i) + 1)).  A contiguous output block of 2^lb
// positions reads one contiguous block of each digit row, so each CTA stages
// the dnum source blocks in shared memory with coalesced loads and gathers
// from there; keys and outputs stream through with 16-byte accesses.
//
// Grid: one CTA per (limb, output block, rotation), the rotation fastest, so
// the R CTAs reading the same digit rows run together and the rows are
// fetched from DRAM about once (later reads hit L2).  Each CTA loops over the
// batch items, so every key word is read once per call.
#include <cuda_runtime.h>

#include "fhe_arith.cuh"
#include "fhe_internal.h"
#include "launch_util.h"

namespace fhe {
namespace {

constexpr int kThreads = 256;
// Staged digit blocks per CTA and the largest output block: 2^11 positions
// for dnum <= 3 (48 KB at dnum = 3, 4 CTAs per SM).  Measured at n = 2^16,
// dnum = 3, 16 rotations: blocks of 2^11 with 256 threads 462 us, 2^9 with
// 128 threads 464 us, 2^10 with 256 or 128 threads 503 / 507 us, 2^8 or 2^9
// with one pair per thread 542 / 581 us, 512-thread CTAs 929 us.
constexpr int kSmemBudget = 48 * 1024;
constexpr int kMaxLogBlock = 11;

__device__ __forceinline__ uint32_t brv_bits(uint32_t x, int bits) { return __brev(x) >> (32 - bits); }

// NTT-domain source position of output position i under sigma_k.
__device__ __forceinline__ uint32_t aut_src(uint32_t i, int log_n, uint32_t k) {
    const uint32_t m = brv_bits(i, log_n);
    const uint32_t e = (k * (2u * m + 1u)) & ((2u << log_n) - 1u);
    return brv_bits((e - 1u) >> 1, log_n);
}

// DN > 0 (dnum <= 4): the 2 DN key pairs of each thread's first coefficient
// pair are loaded before the digit blocks are staged, so that part of the key
// stream (most of the call's bytes) overlaps the staging and its barrier
// (measured 451 -> 409 us for 16 rotations at n = 2^16, dnum = 3; prefetching
// every pair's keys as well took 98 registers and 517 us); DN = 0: any dnum.
template <int DN>
__global__ void __launch_bounds__(kThreads)
k_ks_ip_aut(uint64_t *__restrict__ out, const uint64_t *__restrict__ ext, const uint64_t *__restrict__ keys,
            int log_n, int lb, int LK, int dnum_rt, int batch, int R, const GaloisSet g,
            const uint64_t *__restrict__ consts) {
    pdl_begin();
    extern __shared__ __align__(16) uint64_t blk[];   // [dnum][2^lb]
    const int dnum = DN > 0 ? DN : dnum_rt;
    const int nb = log_n - lb;
    long u = blockIdx.x;
    const int r = (int)(u % R);
    u /= R;
    const uint32_t ob = (uint32_t)(u & ((1L << nb) - 1));
    const int l = (int)(u >> nb);
    const uint32_t k = g.k[r];
    const int bs = 1 << lb;
    const uint32_t o0 = ob << lb;
    const uint32_t s0 = (aut_src(o0, log_n, k) >> lb) << lb;
    const long plane = (long)LK << log_n;
    const long lrow = (long)l << log_n;
    const uint64_t *kc = consts + (long)l * K_COUNT;
    const uint64_t q = __ldg(kc + K_Q), mu = __ldg(kc + K_MU12);
    const uint32_t c58 = (uint32_t)__ldg(kc + K_C58);
    const uint64_t *kr = keys + (long)r * dnum * 2 * plane + lrow + o0;
    for (int b = 0; b < batch; b++) {
        constexpr int NK = DN > 0 ? DN : 1;
        ulonglong2 k0[NK], k1[NK];
        const int x0 = 2 * threadIdx.x;
        if constexpr (DN > 0) {
            if (x0 < bs) {
#pragma unroll
                for (int j = 0; j < DN; j++) {
                    k0[j] = __ldg(reinterpret_cast<const ulonglong2 *>(kr + (2L * j) * plane + x0));
                    k1[j] = __ldg(reinterpret_cast<const ulonglong2 *>(kr + (2L * j + 1) * plane + x0));
                }
            }
        }
        if (b) __syncthreads();   // the previous item's gathers are done
        for (int j = 0; j < dnum; j++) {
            const uint64_t *src = ext + ((long)b * dnum + j) * plane + lrow + s0;
            for (int x = 2 * threadIdx.x; x < bs; x += 2 * kThreads)
                *reinterpret_cast<ulonglong2 *>(blk + j * bs + x) = __ldcg(reinterpret_cast<const ulonglong2 *>(src + x));
        }
        __syncthreads();
        uint64_t *o = out + (((long)r * batch + b) * 2) * plane + lrow + o0;
        for (int x = x0; x < bs; x += 2 * kThreads) {
            const uint32_t p0 = aut_src(o0 + x, log_n, k) - s0, p1 = aut_src(o0 + x + 1, log_n, k) - s0;
            uint64_t h0x = 0, l0x = 0, h0y = 0, l0y = 0, h1x = 0, l1x = 0, h1y = 0, l1y = 0;
            if constexpr (DN > 0) {
                if (x != x0) {
#pragma unroll
                    for (int j = 0; j < DN; j++) {
                        k0[j] = __ldg(reinterpret_cast<const ulonglong2 *>(kr + (2L * j) * plane + x));
                        k1[j] = __ldg(reinterpret_cast<const ulonglong2 *>(kr + (2L * j + 1) * plane + x));
                    }
                }
#pragma unroll
                for (int j = 0; j < DN; j++) {
                    const uint64_t dx = blk[j * bs + p0], dy = blk[j * bs + p1];
                    mac128(h0x, l0x, dx, k0[j].x);
                    mac128(h0y, l0y, dy, k0[j].y);
                    mac128(h1x, l1x, dx, k1[j].x);
                    mac128(h1y, l1y, dy, k1[j].y);
                }
            } else {
                for (int j = 0; j < dnum; j++) {
                    const uint64_t dx = blk[j * bs + p0], dy = blk[j * bs + p1];
                    const ulonglong2 c0 = __ldg(reinterpret_cast<const ulonglong2 *>(kr + (2L * j) * plane + x));
                    const ulonglong2 c1 = __ldg(reinterpret_cast<const ulonglong2 *>(kr + (2L * j + 1) * plane + x));
                    mac128(h0x, l0x, dx, c0.x);
                    mac128(h0y, l0y, dy, c0.y);
                    mac128(h1x, l1x, dx, c1.x);
                    mac128(h1y, l1y, dy, c1.y);
                }
            }
            __stcs(reinterpret_cast<ulonglong2 *>(o + x),
                   make_ulonglong2(barrett_reduce128(h0x, l0x, q, mu, c58), barrett_reduce128(h0y, l0y, q, mu, c58)));
            __stcs(reinterpret_cast<ulonglong2 *>(o + plane + x),
                   make_ulonglong2(barrett_reduce128(h1x, l1x, q, mu, c58), barrett_reduce128(h1y, l1y, q, mu, c58)));
        }
    }
}

}  // namespace

int launch_ks_ip_aut(uint64_t *out, const uint64_t *ext, const uint64_t *keys, int log_n, int LK, int dnum,
                     int batch, int R, const GaloisSet &g, const fhe_ntt_tables *t, void *stream) {
    // largest block with dnum staged rows within the shared-memory budget
    int lb = log_n < kMaxLogBlock ? log_n : kMaxLogBlock;
    while (lb > 1 && ((size_t)dnum << lb) * 8 > (size_t)kSmemBudget) lb--;
    const long blocks = (long)LK * R << (log_n - lb);
    const size_t smem = ((size_t)dnum << lb) * 8;
    auto kern = dnum == 1 ? k_ks_ip_aut<1> : dnum == 2 ? k_ks_ip_aut<2> : dnum == 3 ? k_ks_ip_aut<3>
              : dnum == 4 ? k_ks_ip_aut<4> : k_ks_ip_aut<0>;
    launch_pdl(kern, (unsigned)blocks, kThreads, smem, (cudaStream_t)stream, out, ext, keys, log_n, lb, LK, dnum,
               batch, R, g, t->consts);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

}  // namespace fhe
