// keyswitch_noalloc.cu -- a key switch for callers that must not allocate
// device memory.
//
// fhe_keyswitch_ip needs a caller-provided workspace of
// batch * dnum * (L+K) * n words for the extended digits.  Some callers
// cannot obtain one: code that runs where cudaMalloc/cudaFree are not
// allowed (they may synchronise the device, which a latency-critical or
// stream-ordered caller cannot afford), services whose GPU memory budget is
// fixed and partitioned at start-up, and host runtimes that embed this
// library without giving it any allocator.  fhe_keyswitch_ip_noalloc gives
// them the same operation with the workspace taken from a fixed array in
// this library's own device memory.
//
// The array is a file-scope __device__ variable of kScratchBytes.  Every GPU
// that loads the library holds it until the process exits.  In host code its
// name is only a host-side stand-in, not a device address, so it is never
// passed to a kernel directly: the device address is looked up once per
// device with cudaGetSymbolAddress, with that device current, and cached.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "fhe_internal.h"

namespace fhe {
namespace {

constexpr size_t kScratchBytes = (size_t)16 << 20;   // 16 MiB of extended digits
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint64_t g_ks_scratch[kScratchBytes / sizeof(uint64_t)];

std::mutex g_setup_mutex;
uint64_t *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_ks_scratch on device `dev` (made current by the caller);
// looked up on the first call for that device.
int scratch_for_device(int dev, uint64_t **out) {
    if (dev < 0 || dev >= kMaxDevices) return FHE_EDEVICE;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_ks_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return FHE_ECUDA;
        }
        g_scratch_ptr[dev] = (uint64_t *)p;
    }
    *out = g_scratch_ptr[dev];
    return FHE_OK;
}

}  // namespace
}  // namespace fhe

using namespace fhe;

extern "C" size_t fhe_keyswitch_noalloc_max_bytes(void) { return kScratchBytes; }

extern "C" int fhe_keyswitch_ip_noalloc(uint64_t *out, const uint64_t *in, size_t in_stride, const uint64_t *keys,
                                        int log_n, int L, int K, int dnum, int batch, const fhe_ntt_tables *t_qp,
                                        const void *modup, void *stream) {
    size_t need = 0;
    const int s = fhe_keyswitch_workspace_bytes(log_n, L, K, dnum, batch, &need);
    if (s != FHE_OK) return s;
    if (need > kScratchBytes) return FHE_ESPACE;   // beyond the fixed scratch array: use fhe_keyswitch_ip
    if (!out) return FHE_EINVAL;
    // The scratch lives on the operands' device: make that device current first.
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, out) != cudaSuccess) {
        cudaGetLastError();
        return FHE_EDEVICE;
    }
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) return FHE_EDEVICE;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) return FHE_ECUDA;
    if (cur != a.device && cudaSetDevice(a.device) != cudaSuccess) return FHE_ECUDA;
    uint64_t *scratch = nullptr;
    const int r = scratch_for_device(a.device, &scratch);
    if (r != FHE_OK) return r;
    // Same validation, kernels and launch order as the allocating entry point.
    return fhe_keyswitch_ip(out, in, in_stride, keys, log_n, L, K, dnum, batch, t_qp, modup, scratch, kScratchBytes,
                            stream);
}
