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
// passed to a kernel directly: every call looks the device address up with
// cudaGetSymbolAddress, with the operands' device current.  The address is
// not cached, because it belongs to the current context: after a
// cudaDeviceReset the runtime loads the library's device code again and the
// array may sit elsewhere.
#include <cuda_runtime.h>

#include <cstdint>

#include "fhe_internal.h"

namespace fhe {
namespace {

constexpr size_t kScratchBytes = (size_t)16 << 20;   // 16 MiB of extended digits

static __device__ __align__(256) uint64_t g_ks_scratch[kScratchBytes / sizeof(uint64_t)];

// Device address of g_ks_scratch in the current context (the operands'
// device, made current by the caller).  The first lookup on a device also
// loads this library's device code there.
int scratch_address(uint64_t **out) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_ks_scratch) != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return FHE_ECUDA;
    }
    *out = (uint64_t *)p;
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
    const int r = scratch_address(&scratch);
    if (r != FHE_OK) return r;
    // Same validation, kernels and launch order as the allocating entry point.
    return fhe_keyswitch_ip(out, in, in_stride, keys, log_n, L, K, dnum, batch, t_qp, modup, scratch, kScratchBytes,
                            stream);
}
