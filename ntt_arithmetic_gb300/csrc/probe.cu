// probe.cu -- register-resident throughput probe of the NTT butterfly.
//
// Every thread keeps 32 residues in registers and runs rounds of the forward
// transform's register pass (five radix-2 stages, 80 lazy Cooley-Tukey
// butterflies, fhe_arith.cuh) with twiddles read coalesced from prime 0 of a
// forward table, the same loads the last pass of the NTT makes.  Nothing else
// is on the path: no global data, no shared memory, no barrier.  The rate it
// reaches is the ceiling of this butterfly on the GPU it runs on, which the
// benchmark reports beside the NTT's roofline.
#include <cuda_runtime.h>

#include "fhe_arith.cuh"
#include "fhe_internal.h"

namespace fhe {
namespace {

constexpr int kProbeThreads = 256;
constexpr int kProbeE = 32;

__global__ void __launch_bounds__(kProbeThreads, 2)
k_bfly_probe(uint64_t *__restrict__ out, const ulonglong2 *__restrict__ tw, const uint64_t *__restrict__ consts,
             int iters) {
    const uint64_t q = __ldg(consts + K_Q);
    const uint64_t id = (uint64_t)blockIdx.x * kProbeThreads + threadIdx.x;
    uint64_t x[kProbeE];
#pragma unroll
    for (int i = 0; i < kProbeE; i++) x[i] = (id * 977 + (uint64_t)i * 131) % q;
    const ulonglong2 *lane_tw = tw + (threadIdx.x & 31);
    for (int it = 0; it < iters; it++) {
        // two groups of 31 twiddles, alternating between rounds; entry (g, k) at 32 (32 g + k) + lane
        const ulonglong2 *group = lane_tw + 32 * ((it & 1) << 5);
#pragma unroll
        for (int s = 0; s < 5; s++) {
            constexpr int E = kProbeE;
            const int h = E >> (s + 1);
#pragma unroll
            for (int jj = 0; jj < (1 << s); jj++) {
                const ulonglong2 w = __ldg(group + 32 * ((1 << s) + jj));
#pragma unroll
                for (int u = 0; u < h; u++) ct_bfly(x[jj * 2 * h + u], x[jj * 2 * h + u + h], w.x, w.y, q);
            }
        }
    }
    // checksum: the XOR of the fully reduced residues (x < 2^62 here)
    const uint64_t mu12 = __ldg(consts + K_MU12);
    const uint32_t c58 = (uint32_t)__ldg(consts + K_C58);
    uint64_t acc = 0;
#pragma unroll
    for (int i = 0; i < kProbeE; i++) acc ^= barrett_reduce128(0, x[i], q, mu12, c58);
    out[id] = acc;
}

}  // namespace

int launch_bfly_probe(uint64_t *out, int ctas, int iters, const fhe_ntt_tables *t, void *stream) {
    k_bfly_probe<<<ctas, kProbeThreads, 0, (cudaStream_t)stream>>>(
        out, reinterpret_cast<const ulonglong2 *>(t->fwd), t->consts, iters);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

}  // namespace fhe
