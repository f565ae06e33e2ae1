// launch_util.h -- grid sizing and launch helpers shared by the kernels.
#pragma once
#include <cuda_runtime.h>

#include <utility>

namespace fhe {

// Programmatic dependent launch.  Every library kernel begins with
// pdl_begin(): it signals that the kernel after it in the stream may be
// scheduled, then waits until the kernel before it has completed and its
// writes are visible.  No CTA touches global memory before that wait, so
// stream order holds for every buffer (tables included).  Kernels launched
// through launch_pdl carry the attribute that lets the GPU place their CTAs
// while the previous kernel's last wave is still running: what overlaps is
// the launch and the CTAs' placement, not their work.  Without the attribute
// the wait returns at once.  Measured on GB300 (n = 2^16, 24 primes): the NTT
// kernels gain about 5 us per two-kernel transform and ModDown 10 us per
// call, while the grid-stride streaming kernels (automorphism, products) and
// ModUp lose time under it (the headline step 40 us slower, the key switch
// 9 us), so those keep the plain launch.
#if defined(__CUDACC__)
__device__ __forceinline__ void pdl_begin() {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
}
#endif

template <typename... P, typename... A>
inline cudaError_t launch_pdl(void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, A &&...args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<A>(args)...);
}

// Multiprocessor count of the current device (cached per device id).
inline int sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 132;
    if (cache[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 132;
        cache[dev] = v;
    }
    return cache[dev];
}

// Persistent grid for a grid-stride loop over `items`: at most ctas_per_sm
// resident CTAs per SM (a whole number of waves), fewer for small inputs.
inline unsigned stream_grid(long items, int threads, int ctas_per_sm) {
    const long need = (items + threads - 1) / threads;
    const long cap = (long)sm_count() * ctas_per_sm;
    const long g = need < cap ? need : cap;
    return (unsigned)(g > 0 ? g : 1);
}

}  // namespace fhe
