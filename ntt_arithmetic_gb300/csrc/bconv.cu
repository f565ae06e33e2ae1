// bconv.cu -- basis conversion of a polynomial from S source primes to T
// target primes, coefficient domain.  Modraise, the first step of the
// kestrel-llm bootstrap ("modraise" in the boot profile, overview section
// 4.2: the Garner extension that lifts a low-level ciphertext back to the full
// modulus chain), is the exact case with the sources the first S primes of the
// chain and the targets the whole chain.
//
// Exact: Garner's mixed-radix digits v_a of X in [0, Q), Q = q_0 ... q_{S-1},
// then X mod p = sum_a v_a (q_0 ... q_{a-1}) mod p.  Approximate: the CRT sum
// sum_a [x_a (Q / q_a)^-1]_{q_a} (Q / q_a) = X + e Q with 0 <= e < S, reduced
// modulo p without the correction.  Garner's recursion uses lazy Shoup
// products; each target's sum is an exact multiply-accumulate of 25-bit
// halves (mac25) with one Barrett reduction.
//
// Layout: in [batch][S][n], out [batch][T][n].  One thread per pair of
// coefficients computes their digits once and then a contiguous chunk of
// targets (grid y), so a long target chain (thousands of primes at n = 2^11)
// still fills the GPU.
#include <cuda_runtime.h>

#include "fhe_arith.cuh"
#include "fhe_internal.h"
#include "launch_util.h"

namespace fhe {
namespace {

constexpr int kThreads = 256;

// Digits of one coefficient from its S source residues (in place in v).
template <int MAXS, bool APPROX>
__device__ __forceinline__ void bconv_digits(uint64_t (&v)[MAXS], int S, const uint64_t *__restrict__ src,
                                             const ulonglong2 *__restrict__ garner) {
    if constexpr (APPROX) {
#pragma unroll
        for (int a = 0; a < MAXS; a++) {
            if (a < S) {
                const uint64_t q = __ldg(src + a);
                const ulonglong2 c = __ldg(garner + a);
                v[a] = reduce4(shoup_lazy(v[a], c.x, c.y, q), q);
            }
        }
    } else {
#pragma unroll
        for (int a = 1; a < MAXS; a++) {
            if (a < S) {
                const uint64_t q = __ldg(src + a);
                uint64_t u = v[a];
#pragma unroll
                for (int c = 0; c < a; c++) {
                    const ulonglong2 g = __ldg(garner + a * S + c);
                    u = shoup_lazy(u + 4 * q - v[c], g.x, g.y, q);   // v_c < 2^50 < 4 q
                }
                v[a] = reduce4(u, q);
            }
        }
    }
}

// One thread per pair of adjacent coefficients (16-byte loads and stores).
template <int MAXS, bool APPROX>
__global__ void __launch_bounds__(kThreads, 2)
k_bconv(uint64_t *__restrict__ out, const uint64_t *__restrict__ in, int log_n, int S, int T, int tchunk,
        const uint64_t *__restrict__ src, const ulonglong2 *__restrict__ dst, const ulonglong2 *__restrict__ garner,
        const ulonglong2 *__restrict__ weights) {
    pdl_begin();
    // APPROX: `garner` holds the bracket constants [S], `weights` the CRT
    // weights [T][S]; exact: Garner constants [S][S] and radix weights [T][S].
    const long n = 1L << log_n;
    const long b = blockIdx.z;
    const int t0 = blockIdx.y * tchunk;
    const int t1 = t0 + tchunk < T ? t0 + tchunk : T;
    for (long i = 2 * ((long)blockIdx.x * blockDim.x + threadIdx.x); i < n; i += 2L * gridDim.x * blockDim.x) {
        uint64_t v0[MAXS], v1[MAXS];
#pragma unroll
        for (int a = 0; a < MAXS; a++) {
            v0[a] = v1[a] = 0;
            if (a < S) {
                const ulonglong2 x = __ldcs(reinterpret_cast<const ulonglong2 *>(in + (b * S + a) * n + i));
                v0[a] = x.x;
                v1[a] = x.y;
            }
        }
        bconv_digits<MAXS, APPROX>(v0, S, src, garner);
        bconv_digits<MAXS, APPROX>(v1, S, src, garner);
        uint64_t *o = out + b * T * n + i;
        Split25 s0[MAXS], s1[MAXS];
#pragma unroll
        for (int a = 0; a < MAXS; a++) {
            s0[a] = split25(v0[a]);
            s1[a] = split25(v1[a]);
        }
        for (int t = t0; t < t1; t++) {
            const ulonglong2 pc = __ldg(dst + 2 * t);       // (p, floor(2^58 / p))
            if (!APPROX && S == 1) {   // one source prime (modraise from one limb): X = x_0 < 2^50
                __stcs(reinterpret_cast<ulonglong2 *>(o + (long)t * n),
                       make_ulonglong2(reduce_small(v0[0], pc.x, (uint32_t)pc.y), reduce_small(v1[0], pc.x, (uint32_t)pc.y)));
                continue;
            }
            const uint64_t mu12 = __ldg(reinterpret_cast<const uint64_t *>(dst + 2 * t + 1));
            const ulonglong2 *wt = weights + (long)t * S;
            Mac25 acc0, acc1;
#pragma unroll
            for (int a = APPROX ? 0 : 1; a < MAXS; a++) {
                if (a < S) {
                    const ulonglong2 w = __ldg(wt + a);
                    const Split25 m = split25_entry(w.x, w.y);
                    mac25(acc0, s0[a], m);
                    mac25(acc1, s1[a], m);
                }
            }
            // exact: the weight of v_0 is 1
            __stcs(reinterpret_cast<ulonglong2 *>(o + (long)t * n),
                   make_ulonglong2(mac25_reduce(acc0, APPROX ? 0 : v0[0], pc.x, mu12, (uint32_t)pc.y),
                                   mac25_reduce(acc1, APPROX ? 0 : v1[0], pc.x, mu12, (uint32_t)pc.y)));
        }
    }
}

template <int MAXS>
void launch_t(uint64_t *out, const uint64_t *in, int log_n, int S, int T, int batch, bool approx, const char *base,
              cudaStream_t st) {
    const BconvLayout lay = bconv_layout(S, T);
    const long n = 1L << log_n;
    const long bx = (n / 2 + kThreads - 1) / kThreads;   // one thread per coefficient pair
    // enough CTAs for 8 per SM; each chunk repeats the digit computation once
    const long want = (long)sm_count() * 8;
    long chunks = (want + bx * batch - 1) / (bx * batch);
    const long max_chunks = (T + 7) / 8;   // at least 8 targets per chunk
    if (chunks > max_chunks) chunks = max_chunks;
    if (chunks < 1) chunks = 1;
    const int tchunk = (int)((T + chunks - 1) / chunks);
    chunks = (T + tchunk - 1) / tchunk;
    dim3 grid((unsigned)bx, (unsigned)chunks, (unsigned)batch);
    auto kern = approx ? k_bconv<MAXS, true> : k_bconv<MAXS, false>;
    launch_pdl(kern, grid, kThreads, 0, st, out, in, log_n, S, T, tchunk, (const uint64_t *)(base + lay.off_src),
               (const ulonglong2 *)(base + lay.off_dst),
               (const ulonglong2 *)(base + (approx ? lay.off_qinv : lay.off_garner)),
               (const ulonglong2 *)(base + (approx ? lay.off_qhat : lay.off_mr)));
}

}  // namespace

int launch_bconv(uint64_t *out, const uint64_t *in, int log_n, int S, int T, int batch, bool approx,
                 const void *bconv, void *stream) {
    cudaStream_t st = (cudaStream_t)stream;
    const char *base = (const char *)bconv;
    if (S <= 1) launch_t<1>(out, in, log_n, S, T, batch, approx, base, st);
    else if (S <= 2) launch_t<2>(out, in, log_n, S, T, batch, approx, base, st);
    else if (S <= 4) launch_t<4>(out, in, log_n, S, T, batch, approx, base, st);
    else if (S <= 8) launch_t<8>(out, in, log_n, S, T, batch, approx, base, st);
    else launch_t<16>(out, in, log_n, S, T, batch, approx, base, st);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

}  // namespace fhe
