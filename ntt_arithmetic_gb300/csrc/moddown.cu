// moddown.cu -- ModDown (QP -> Q) and rescale: out = floor((X + h) / P) mod q_l
// for X the exact CRT value over Q u P, P = p_0 ... p_{K-1}, h = (P-1)/2
// (nearest rounding) or 0 (truncation).  Rescale is the case K = 1 with P the
// last prime of the chain.  FHElium's CUDA layer lists "key-switch
// multiply-accumulate and QP-to-Q ModDown" and "nearest and truncating rescale
// kernels" ("Eager, Compile, and native execution", section "CUDA execution");
// kestrel-llm's vllm_ckks.c has rescale (overview, section 3).
//
// With c = (X + h) mod P, floor((X + h) / P) = (X + h - c) / P, so per
// coefficient:
//   1. the P residues of X + h are converted exactly to c mod q_l by Garner's
//      mixed radix (the same construction as the key-switch ModUp; the radix
//      sum is an exact multiply-accumulate reduced once) and
//      d_l = c - h mod q_l is written (coefficient domain; in the NTT-domain
//      path as a value below (6 + K) q congruent to it, for the forward NTT);
//   2. out_l = (x_l - d_l) P^-1 mod q_l.
// In the coefficient domain both steps run in one pass (one read of every
// input limb, one write of every output limb).  In the NTT domain the P limbs
// are first brought back to coefficients (inverse NTT of a copy) and d is
// transformed forward over Q before step 2; the map is linear, so step 2 is
// the same in both domains.
#include <cuda_runtime.h>

#include "fhe_arith.cuh"
#include "fhe_internal.h"
#include "launch_util.h"

namespace fhe {
namespace {

constexpr int kThreads = 256;

// ws[b][k][i] = in[b][L + k][i]  (the P limbs of each batch item)
__global__ void __launch_bounds__(kThreads)
k_copy_limbs(uint64_t *__restrict__ ws, const uint64_t *__restrict__ in, long pairs, int log_n, int L, int K) {
    pdl_begin();
    const long stride = (long)gridDim.x * blockDim.x;
    const long per_item = (long)K << log_n;
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < pairs; i += stride) {
        const long e = 2 * i;
        const long b = e / per_item, r = e - b * per_item;
        const uint64_t *src = in + b * ((long)(L + K) << log_n) + ((long)L << log_n) + r;
        __stcg(reinterpret_cast<ulonglong2 *>(ws + e), __ldcs(reinterpret_cast<const ulonglong2 *>(src)));
    }
}

// d[b][l][i] = ((X + h) mod P) - h  mod q_l, from the P residues
// src[b * src_item + k * n + i] (k < K).  FUSED (coefficient domain): instead
// of d, write out[b][l][i] = (x_l - d_l) P^-1 mod q_l directly, reading x_l
// from src - L n (the Q limbs of the same batch item).
// STAGED (L <= kMaxBasis): the radix weights and the Q primes' reduction
// constants are staged in shared memory and read as broadcasts.
template <int MAXK, bool FUSED, bool STAGED>
__global__ void __launch_bounds__(kThreads)
k_moddown_conv(uint64_t *__restrict__ d, const uint64_t *__restrict__ src, long src_item, int log_n, int L, int K,
               int batch, int nearest, const ulonglong2 *__restrict__ garner, const ulonglong2 *__restrict__ mr,
               const uint64_t *__restrict__ hp, const uint64_t *__restrict__ hq, const ulonglong2 *__restrict__ pinv,
               const uint64_t *__restrict__ consts_q, const uint64_t *__restrict__ consts_p) {
    pdl_begin();
    const long n = 1L << log_n;
    const long total = n * batch;
    const long stride = (long)gridDim.x * blockDim.x;
    __shared__ ulonglong2 s_mr[STAGED ? kMaxBasis * MAXK : 1];
    __shared__ ulonglong2 s_qm[STAGED ? kMaxBasis : 1];     // (q, floor(2^100 / q) << 12)
    __shared__ uint32_t s_c58[STAGED ? kMaxBasis : 1];
    if constexpr (STAGED) {
        for (int e = threadIdx.x; e < L * MAXK; e += blockDim.x) {
            const int l = e / MAXK, a = e - l * MAXK;
            s_mr[e] = a < K ? __ldg(mr + l * K + a) : make_ulonglong2(0, 0);
        }
        for (int l = threadIdx.x; l < L; l += blockDim.x) {
            const uint64_t *kc = consts_q + (long)l * K_COUNT;
            s_qm[l] = make_ulonglong2(__ldg(kc + K_Q), __ldg(kc + K_MU12));
            s_c58[l] = (uint32_t)__ldg(kc + K_C58);
        }
        __syncthreads();
    }
    for (long e = (long)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += stride) {
        const long b = e >> log_n, i = e & (n - 1);
        uint64_t v[MAXK];
#pragma unroll
        for (int a = 0; a < MAXK; a++) {
            v[a] = 0;
            if (a < K) {
                const uint64_t p = __ldg(consts_p + (long)a * K_COUNT + K_Q);
                const uint64_t y = __ldcs(src + b * src_item + (long)a * n + i) + (nearest ? __ldg(hp + a) : 0);
                v[a] = csub(y, p);   // y < 2p
            }
        }
        // Garner over P: v_a <- ((((y_a - v_0) p_0^-1 - v_1) p_1^-1 ...) - v_{a-1}) p_{a-1}^-1 mod p_a
#pragma unroll
        for (int a = 1; a < MAXK; a++) {
            if (a < K) {
                const uint64_t p = __ldg(consts_p + (long)a * K_COUNT + K_Q);
                uint64_t u = v[a];
#pragma unroll
                for (int c = 0; c < a; c++) {
                    const ulonglong2 g = __ldg(garner + a * K + c);
                    u = shoup_lazy(u + 4 * p - v[c], g.x, g.y, p);   // v_c < 2^50 < 4 p
                }
                v[a] = reduce4(u, p);
            }
        }
        Split25 vs[MAXK];
#pragma unroll
        for (int a = 0; a < MAXK; a++) vs[a] = split25(v[a]);
        for (int l = 0; l < L; l++) {
            const uint64_t *kc = consts_q + (long)l * K_COUNT;
            const ulonglong2 qm = STAGED ? s_qm[l] : make_ulonglong2(__ldg(kc + K_Q), __ldg(kc + K_MU12));
            const uint64_t q = qm.x;
            Mac25 acc;   // sum_{a >= 1} v_a (p_0 ... p_{a-1}); the weight of v_0 is 1
#pragma unroll
            for (int a = 1; a < MAXK; a++) {
                if (a < K) {
                    const ulonglong2 m = STAGED ? s_mr[l * MAXK + a] : __ldg(mr + l * K + a);
                    mac25(acc, vs[a], split25_entry(m.x, m.y));
                }
            }
            uint64_t c;
            if constexpr (FUSED) {
                c = mac25_reduce(acc, v[0], q, qm.y, STAGED ? s_c58[l] : (uint32_t)__ldg(kc + K_C58));
                if (nearest) {
                    const uint64_t h = __ldg(hq + l);
                    c = c >= h ? c - h : c + q - h;
                }
            } else {
                // d only feeds the forward NTT over Q, whose lazy butterflies take
                // inputs of a few q: left below (5 + K) q, not fully reduced
                c = mac25_reduce_lazy(acc, v[0], q, qm.y);
                if (nearest) c += q - __ldg(hq + l);
            }
            if constexpr (FUSED) {
                const uint64_t x = __ldcs(src + b * src_item - ((long)(L - l) << log_n) + i);
                const ulonglong2 pi = __ldg(pinv + l);
                __stcs(d + ((b * L + l) << log_n) + i, reduce4(shoup_lazy(x + q - c, pi.x, pi.y, q), q));
            } else {
                __stcg(d + ((b * L + l) << log_n) + i, c);
            }
        }
    }
}

// out[b][l][i] = (in[b][l][i] - d[b][l][i]) P^-1 mod q_l
__global__ void __launch_bounds__(kThreads)
k_moddown_finish(uint64_t *__restrict__ out, const uint64_t *__restrict__ in, const uint64_t *__restrict__ d,
                 long pairs, int log_n, int L, int K, const ulonglong2 *__restrict__ pinv,
                 const uint64_t *__restrict__ consts) {
    pdl_begin();
    const long stride = (long)gridDim.x * blockDim.x;
    const long plane = (long)L << log_n;
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < pairs; i += stride) {
        const long e = 2 * i;                  // index over [batch][L][n]
        const long b = e / plane, r = e - b * plane;
        const int l = (int)(r >> log_n);
        const uint64_t q = __ldg(consts + (long)l * K_COUNT + K_Q);
        const ulonglong2 pi = __ldg(pinv + l);
        const ulonglong2 x = __ldcs(reinterpret_cast<const ulonglong2 *>(in + b * ((long)(L + K) << log_n) + r));
        const ulonglong2 dv = __ldcs(reinterpret_cast<const ulonglong2 *>(d + e));
        const uint64_t o0 = reduce4(shoup_lazy(x.x + q - dv.x, pi.x, pi.y, q), q);
        const uint64_t o1 = reduce4(shoup_lazy(x.y + q - dv.y, pi.x, pi.y, q), q);
        __stcs(reinterpret_cast<ulonglong2 *>(out + e), make_ulonglong2(o0, o1));
    }
}

template <int MAXK>
void launch_conv(uint64_t *d, const uint64_t *src, long src_item, int log_n, int L, int K, int batch, bool nearest,
                 bool fused, const ModdownLayout &lay, const char *md, const fhe_ntt_tables *t_qp, cudaStream_t st) {
    const long total = (long)batch << log_n;
    const unsigned grid = stream_grid(total, kThreads, 8);
    const bool staged = L <= kMaxBasis;
    auto kern = fused ? (staged ? k_moddown_conv<MAXK, true, true> : k_moddown_conv<MAXK, true, false>)
                      : (staged ? k_moddown_conv<MAXK, false, true> : k_moddown_conv<MAXK, false, false>);
    launch_pdl(kern, grid, kThreads, 0, st, d, src, src_item, log_n, L, K, batch, nearest ? 1 : 0,
               (const ulonglong2 *)(md + lay.off_garner), (const ulonglong2 *)(md + lay.off_mr),
               (const uint64_t *)(md + lay.off_hp), (const uint64_t *)(md + lay.off_hq),
               (const ulonglong2 *)(md + lay.off_pinv), t_qp->consts,
               t_qp->consts + (long)L * K_COUNT);
}

}  // namespace

int launch_moddown(uint64_t *out, const uint64_t *in, int log_n, int L, int K, int batch, bool ntt_domain,
                   bool nearest, const fhe_ntt_tables *t_qp, const void *md_blob, uint64_t *ws, void *stream) {
    cudaStream_t st = (cudaStream_t)stream;
    const ModdownLayout lay = moddown_layout(L, K);
    const char *md = (const char *)md_blob;
    int launched = 0;
    const uint64_t *src = in + ((long)L << log_n);       // P limbs of batch item 0
    long src_item = (long)(L + K) << log_n;
    uint64_t *d = ntt_domain ? ws : out;                // [batch][L][n]; the output itself when fused
    if (ntt_domain) {
        uint64_t *pl = ws + ((long)batch * L << log_n);   // [batch][K][n]
        const fhe_ntt_tables tp = tables_slice(t_qp, L, K);
        // the inverse NTT of the P limbs reads them from `in` where its block kernel can
        int r = launch_ntt_inv_from(pl, in + ((long)L << log_n), (long)(L + K) << log_n, log_n, K, batch, &tp, stream);
        if (r < 0) return -1;
        if (r == 0) {
            const long pairs = ((long)batch * K << log_n) / 2;
            launch_pdl(k_copy_limbs, stream_grid(pairs, kThreads, 8), kThreads, 0, st, pl, in, pairs, log_n, L, K);
            if (cudaGetLastError() != cudaSuccess) return -1;
            launched++;
            r = launch_ntt(pl, log_n, K, (long)batch * K, &tp, true, stream);
            if (r < 0) return -1;
        }
        launched += r;
        src = pl;
        src_item = (long)K << log_n;
    }
    // the NTT-domain conversion on the tensor cores where the shape allows (K <= 8, n >= 128)
    const int tc = ntt_domain ? launch_moddown_tc(d, src, src_item, log_n, L, K, batch, nearest, t_qp, md, stream) : 0;
    if (tc < 0) return -1;
    if (tc == 0) {
        if (K <= 1) launch_conv<1>(d, src, src_item, log_n, L, K, batch, nearest, !ntt_domain, lay, md, t_qp, st);
        else if (K <= 2) launch_conv<2>(d, src, src_item, log_n, L, K, batch, nearest, !ntt_domain, lay, md, t_qp, st);
        else if (K <= 4) launch_conv<4>(d, src, src_item, log_n, L, K, batch, nearest, !ntt_domain, lay, md, t_qp, st);
        else if (K <= 8) launch_conv<8>(d, src, src_item, log_n, L, K, batch, nearest, !ntt_domain, lay, md, t_qp, st);
        else launch_conv<16>(d, src, src_item, log_n, L, K, batch, nearest, !ntt_domain, lay, md, t_qp, st);
    }
    if (cudaGetLastError() != cudaSuccess) return -1;
    launched++;
    if (!ntt_domain) return launched;
    const fhe_ntt_tables tq = tables_slice(t_qp, 0, L);
    // the forward NTT of d fused with the last step where a fused kernel exists
    int r = launch_ntt_fwd_moddown(out, d, in, log_n, L, K, batch, &tq, md + lay.off_pinv, stream);
    if (r < 0) return -1;
    if (r > 0) return launched + r;
    r = launch_ntt(d, log_n, L, (long)batch * L, &tq, false, stream);
    if (r < 0) return -1;
    launched += r;
    const long pairs = ((long)batch * L << log_n) / 2;
    launch_pdl(k_moddown_finish, stream_grid(pairs, kThreads, 8), kThreads, 0, st, out, in, d, pairs, log_n, L, K,
               (const ulonglong2 *)(md + lay.off_pinv), t_qp->consts);
    if (cudaGetLastError() != cudaSuccess) return -1;
    return launched + 1;
}

}  // namespace fhe
