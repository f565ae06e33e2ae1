// launch_util.h -- grid sizing helpers shared by the streaming kernels.
#pragma once
#include <cuda_runtime.h>

namespace fhe {

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
