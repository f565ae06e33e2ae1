// abi.cu -- the extern "C" entry points of libfhe_ntt.so: host-side
// validation, device selection and launches on the caller's stream.
//
// Validation follows the rules FHElium states for its adapters ("Eager,
// Compile, and native execution", sections "Schema registration and device
// dispatch", "CUDA execution" and "Execution properties"): shape, device
// agreement, parameter-row counts and prohibited overlap are checked before
// launch; mixed-device operands fail; the operand's device is made current;
// kernels go on the given stream with no host synchronisation.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "fhe_internal.h"

namespace fhe {

static std::atomic<uint64_t> g_launches{0};

void count_launches(int k) {
    if (k > 0) g_launches.fetch_add((uint64_t)k, std::memory_order_relaxed);
}

namespace {

struct Span {
    const void *p;
    size_t bytes;
};

bool overlap(Span a, Span b) {
    const uintptr_t a0 = (uintptr_t)a.p, a1 = a0 + a.bytes, b0 = (uintptr_t)b.p, b1 = b0 + b.bytes;
    return a.bytes && b.bytes && a0 < b1 && b0 < a1;
}

bool same(Span a, Span b) { return a.p == b.p && a.bytes == b.bytes; }

// Resolve the device of every pointer; all must be device (or managed)
// memory of one device, which becomes current.  Host or unknown pointers
// are rejected so that no kernel is ever handed a host address.
int select_device(std::initializer_list<const void *> ptrs) {
    int dev = -1;
    for (const void *p : ptrs) {
        if (!p) return FHE_EINVAL;
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
            cudaGetLastError();
            return FHE_EDEVICE;
        }
        if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) return FHE_EDEVICE;
        if (dev < 0) dev = a.device;
        else if (a.device != dev) return FHE_EDEVICE;
    }
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) return FHE_ECUDA;
    if (cur != dev && cudaSetDevice(dev) != cudaSuccess) return FHE_ECUDA;
    return FHE_OK;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15) == 0; }

// The struct must be exactly what fhe_ntt_tables_bind writes for its blob:
// every sub-pointer at its layout offset from `blob` and `bytes` the layout's
// size.  Only `blob` goes through the device and overlap checks, so a
// sub-pointer anywhere else (another buffer, host memory) is refused here,
// before any launch.
int check_tables(const fhe_ntt_tables *t, int log_n, int L) {
    if (!t || !t->blob || !aligned16(t->blob)) return FHE_EINVAL;
    if (t->log_n < 1 || t->log_n > kMaxLogN || t->L < 1 || t->L > kMaxTableL) return FHE_EINVAL;
    if (t->log_n != log_n || L > t->L) return FHE_EINVAL;
    const NttLayout lay = ntt_layout(t->log_n, t->L);
    const char *base = (const char *)t->blob;
    if (t->bytes != lay.bytes || (const char *)t->q != base + lay.off_q ||
        (const char *)t->consts != base + lay.off_consts || (const char *)t->fwd != base + lay.off_fwd ||
        (const char *)t->inv != base + lay.off_inv || (const char *)t->twist != base + lay.off_twist)
        return FHE_EINVAL;
    return FHE_OK;
}

int check_shape(int log_n, int L, long batch) {
    if (log_n < 1 || log_n > kMaxLogN || L < 1 || batch < 1) return FHE_EINVAL;
    const long rows = batch * (long)L;
    if (rows > (1L << 30) / (log_n >= 14 ? (1L << (log_n - 13)) : 1)) return FHE_EINVAL;  // grid size
    return FHE_OK;
}

int finish(int launched) {
    if (launched < 0) {
        cudaGetLastError();
        return FHE_ECUDA;
    }
    count_launches(launched);
    return FHE_OK;
}

}  // namespace
}  // namespace fhe

using namespace fhe;

extern "C" int fhe_version(void) { return 100; }

extern "C" const char *fhe_status_str(int s) {
    switch (s) {
        case FHE_OK: return "ok";
        case FHE_EINVAL: return "invalid argument (size, modulus, k, null pointer, alignment or table shape)";
        case FHE_EALIAS: return "prohibited overlap between an output and another buffer";
        case FHE_ECUDA: return "CUDA runtime or kernel launch failure";
        case FHE_ESPACE: return "workspace or host buffer too small";
        case FHE_EDEVICE: return "host pointer where a device pointer is required, or operands on different devices";
        default: return "unknown status";
    }
}

extern "C" uint64_t fhe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" int fhe_device_status(int *status, int reset) {
    if (!status) return FHE_EINVAL;
    return device_status(status, reset != 0);
}

extern "C" int fhe_butterfly_probe(uint64_t *out, int ctas, int iters, const fhe_ntt_tables *t, void *stream) {
    if (!out || !aligned16(out) || ctas < 1 || ctas > (1 << 20) || iters < 1 || iters > 128) return FHE_EINVAL;
    if (!t || t->log_n < 11) return FHE_EINVAL;
    int s = check_tables(t, t->log_n, 1);
    if (s) return s;
    if ((s = select_device({out, t->blob}))) return s;
    const Span o{out, (size_t)ctas * 256 * 8}, tb{t->blob, t->bytes};
    if (overlap(o, tb)) return FHE_EALIAS;
    return finish(launch_bfly_probe(out, ctas, iters, t, stream));
}

static int ntt_call(uint64_t *res, int log_n, int L, int batch, const fhe_ntt_tables *t, void *stream, bool inverse) {
    int s = check_shape(log_n, L, batch);
    if (s) return s;
    if ((s = check_tables(t, log_n, L))) return s;
    if (!res || !aligned16(res)) return FHE_EINVAL;
    if ((s = select_device({res, t->blob}))) return s;
    const Span r{res, ((size_t)batch * L << log_n) * 8}, tb{t->blob, t->bytes};
    if (overlap(r, tb)) return FHE_EALIAS;
    return finish(launch_ntt(res, log_n, L, (long)batch * L, t, inverse, stream));
}

extern "C" int fhe_ntt_fwd(uint64_t *res, int log_n, int L, int batch, const fhe_ntt_tables *t, void *stream) {
    return ntt_call(res, log_n, L, batch, t, stream, false);
}

extern "C" int fhe_ntt_inv(uint64_t *res, int log_n, int L, int batch, const fhe_ntt_tables *t, void *stream) {
    return ntt_call(res, log_n, L, batch, t, stream, true);
}

extern "C" int fhe_mul_ntt(uint64_t *out, const uint64_t *a, const uint64_t *b, int log_n, int L, int batch,
                           const fhe_ntt_tables *t, void *stream) {
    int s = check_shape(log_n, L, batch);
    if (s) return s;
    if ((s = check_tables(t, log_n, L))) return s;
    if (!out || !a || !b || !aligned16(out) || !aligned16(a) || !aligned16(b)) return FHE_EINVAL;
    if ((s = select_device({out, a, b, t->blob}))) return s;
    const size_t bytes = ((size_t)batch * L << log_n) * 8;
    const Span o{out, bytes}, sa{a, bytes}, sb{b, bytes}, tb{t->blob, t->bytes};
    if ((overlap(o, sa) && !same(o, sa)) || (overlap(o, sb) && !same(o, sb)) || overlap(o, tb)) return FHE_EALIAS;
    return finish(launch_mul(out, a, b, log_n, L, (long)batch * L, t, stream));
}

extern "C" int fhe_tensor(uint64_t *d, const uint64_t *a, const uint64_t *b, int log_n, int L, int batch,
                          const fhe_ntt_tables *t, void *stream) {
    int s = check_shape(log_n, L, batch);
    if (s) return s;
    if ((s = check_tables(t, log_n, L))) return s;
    if (!d || !a || !b || !aligned16(d) || !aligned16(a) || !aligned16(b)) return FHE_EINVAL;
    if ((s = select_device({d, a, b, t->blob}))) return s;
    const size_t plane = ((size_t)L << log_n) * 8;
    const Span sd{d, 3 * plane * batch}, sa{a, 2 * plane * batch}, sb{b, 2 * plane * batch}, tb{t->blob, t->bytes};
    if (overlap(sd, sa) || overlap(sd, sb) || overlap(sd, tb)) return FHE_EALIAS;
    return finish(launch_tensor(d, a, b, log_n, L, batch, t, stream));
}

extern "C" int fhe_automorph(uint64_t *out, const uint64_t *in, int log_n, int L, int batch, uint64_t k, int domain,
                             const fhe_ntt_tables *t, void *stream) {
    int s = check_shape(log_n, L, batch);
    if (s) return s;
    if ((s = check_tables(t, log_n, L))) return s;
    if (domain != FHE_DOMAIN_COEFF && domain != FHE_DOMAIN_NTT) return FHE_EINVAL;
    if ((k & 1) == 0 || k >= (2ull << log_n)) return FHE_EINVAL;
    if (!out || !in || !aligned16(out) || !aligned16(in)) return FHE_EINVAL;
    if ((s = select_device({out, in, t->blob}))) return s;
    const size_t bytes = ((size_t)batch * L << log_n) * 8;
    const Span o{out, bytes}, i{in, bytes}, tb{t->blob, t->bytes};
    if (overlap(o, i) || overlap(o, tb)) return FHE_EALIAS;
    return finish(launch_automorph(out, in, log_n, L, (long)batch * L, k, domain, t, stream));
}

extern "C" int fhe_keyswitch_workspace_bytes(int log_n, int L, int K, int dnum, int batch, size_t *bytes) {
    if (!bytes || log_n < 1 || log_n > kMaxLogN || batch < 1 || !modup_shape_ok(L, K, dnum) || dnum > 32)
        return FHE_EINVAL;
    *bytes = ((size_t)batch * dnum * (L + K) << log_n) * 8;
    return FHE_OK;
}

namespace {

// Validation and ModUp + NTT of the digits shared by the plain and the hoisted
// key switch.  R = 0: plain (out [batch][2][L+K][n], keys [dnum][2][L+K][n]);
// R >= 1: hoisted (out [R][batch][2][L+K][n], keys [R][dnum][2][L+K][n]).
int keyswitch_call(uint64_t *out, const uint64_t *in, size_t in_stride, const uint64_t *keys, const uint32_t *galois,
                   int R, int log_n, int L, int K, int dnum, int batch, int modup_mode, const fhe_ntt_tables *t_qp,
                   const void *modup, uint64_t *workspace, size_t ws_bytes, void *stream) {
    size_t need = 0;
    int s = fhe_keyswitch_workspace_bytes(log_n, L, K, dnum, batch, &need);
    if (s) return s;
    const int LK = L + K;
    if ((s = check_shape(log_n, LK, (long)batch * dnum))) return s;
    if ((s = check_tables(t_qp, log_n, LK))) return s;
    if (modup_mode != FHE_MODUP_EXACT && modup_mode != FHE_MODUP_APPROX) return FHE_EINVAL;
    if (!out || !in || !keys || !modup || !workspace) return FHE_EINVAL;
    if (!aligned16(out) || !aligned16(in) || !aligned16(keys) || !aligned16(workspace) || !aligned16(modup))
        return FHE_EINVAL;
    GaloisSet g = {};
    if (R > 0) {
        if (R > kMaxRotations || !galois) return FHE_EINVAL;
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, galois) != cudaSuccess) cudaGetLastError();   // plain host memory
        else if (a.type == cudaMemoryTypeDevice) return FHE_EDEVICE;                  // must be host-readable
        const uint64_t two_n = 2ull << log_n;
        for (int r = 0; r < R; r++) {
            if (!(galois[r] & 1) || galois[r] >= two_n) return FHE_EINVAL;
            g.k[r] = galois[r];
        }
    }
    if (ws_bytes < need) return FHE_ESPACE;
    const size_t item = (size_t)L << log_n;
    if (in_stride == 0) in_stride = item;
    if (in_stride < item || (in_stride & 1)) return FHE_EINVAL;
    if ((s = select_device({out, in, keys, modup, workspace, t_qp->blob}))) return s;
    const size_t plane = ((size_t)LK << log_n) * 8;
    const size_t reps = R > 0 ? (size_t)R : 1;
    const Span so{out, 2 * plane * batch * reps}, si{in, ((size_t)(batch - 1) * in_stride + item) * 8},
        sk{keys, 2 * plane * dnum * reps}, sw{workspace, need}, tb{t_qp->blob, t_qp->bytes},
        sm{modup, modup_layout(L, K, dnum).bytes};
    const Span all[6] = {so, si, sk, sw, tb, sm};
    for (int x = 0; x < 6; x++)
        for (int y = x + 1; y < 6; y++) {
            if ((x == 1 || x == 2 || x == 4 || x == 5) && (y == 1 || y == 2 || y == 4 || y == 5)) continue;  // read-only pairs
            if (overlap(all[x], all[y])) return FHE_EALIAS;
        }
    int launched = 0, r;
    if ((r = launch_modup(workspace, in, (long)in_stride, log_n, L, K, dnum, batch, modup_mode == FHE_MODUP_APPROX,
                          t_qp, modup, stream)) < 0)
        return finish(-1);
    launched += r;
    if (R == 0) {
        // the NTT of the digits fused with the inner product where a fused kernel exists
        if ((r = launch_ntt_fwd_ip(out, workspace, keys, log_n, LK, dnum, batch, t_qp, stream)) < 0)
            return finish(-1);
        if (r > 0) return finish(launched + r);
    }
    if ((r = launch_ntt(workspace, log_n, LK, (long)batch * dnum * LK, t_qp, false, stream)) < 0) return finish(-1);
    launched += r;
    r = R > 0 ? launch_ks_ip_aut(out, workspace, keys, log_n, LK, dnum, batch, R, g, t_qp, stream)
              : launch_ks_ip(out, workspace, keys, log_n, LK, dnum, batch, t_qp, stream);
    if (r < 0) return finish(-1);
    launched += r;
    return finish(launched);
}

}  // namespace

extern "C" int fhe_keyswitch_ip_ex(uint64_t *out, const uint64_t *in, size_t in_stride, const uint64_t *keys,
                                   int log_n, int L, int K, int dnum, int batch, int modup_mode,
                                   const fhe_ntt_tables *t_qp, const void *modup, uint64_t *workspace,
                                   size_t ws_bytes, void *stream) {
    return keyswitch_call(out, in, in_stride, keys, nullptr, 0, log_n, L, K, dnum, batch, modup_mode, t_qp, modup,
                          workspace, ws_bytes, stream);
}

extern "C" int fhe_keyswitch_ip(uint64_t *out, const uint64_t *in, size_t in_stride, const uint64_t *keys, int log_n,
                                int L, int K, int dnum, int batch, const fhe_ntt_tables *t_qp, const void *modup,
                                uint64_t *workspace, size_t ws_bytes, void *stream) {
    return keyswitch_call(out, in, in_stride, keys, nullptr, 0, log_n, L, K, dnum, batch, FHE_MODUP_EXACT, t_qp,
                          modup, workspace, ws_bytes, stream);
}

extern "C" int fhe_keyswitch_hoisted(uint64_t *out, const uint64_t *in, size_t in_stride, const uint64_t *keys,
                                     const uint32_t *galois, int R, int log_n, int L, int K, int dnum, int batch,
                                     int modup_mode, const fhe_ntt_tables *t_qp, const void *modup,
                                     uint64_t *workspace, size_t ws_bytes, void *stream) {
    if (R < 1) return FHE_EINVAL;
    return keyswitch_call(out, in, in_stride, keys, galois, R, log_n, L, K, dnum, batch, modup_mode, t_qp, modup,
                          workspace, ws_bytes, stream);
}

extern "C" int fhe_keyswitch_decompose(uint64_t *digits, const uint64_t *in, size_t in_stride, int log_n, int L,
                                       int K, int dnum, int batch, int modup_mode, const fhe_ntt_tables *t_qp,
                                       const void *modup, void *stream) {
    size_t need = 0;
    int s = fhe_keyswitch_workspace_bytes(log_n, L, K, dnum, batch, &need);
    if (s) return s;
    const int LK = L + K;
    if ((s = check_shape(log_n, LK, (long)batch * dnum))) return s;
    if ((s = check_tables(t_qp, log_n, LK))) return s;
    if (modup_mode != FHE_MODUP_EXACT && modup_mode != FHE_MODUP_APPROX) return FHE_EINVAL;
    if (!digits || !in || !modup || !aligned16(digits) || !aligned16(in) || !aligned16(modup)) return FHE_EINVAL;
    const size_t item = (size_t)L << log_n;
    if (in_stride == 0) in_stride = item;
    if (in_stride < item || (in_stride & 1)) return FHE_EINVAL;
    if ((s = select_device({digits, in, modup, t_qp->blob}))) return s;
    const Span sd{digits, need}, si{in, ((size_t)(batch - 1) * in_stride + item) * 8}, tb{t_qp->blob, t_qp->bytes},
        sm{modup, modup_layout(L, K, dnum).bytes};
    if (overlap(sd, si) || overlap(sd, tb) || overlap(sd, sm)) return FHE_EALIAS;
    int launched = 0, r;
    if ((r = launch_modup(digits, in, (long)in_stride, log_n, L, K, dnum, batch, modup_mode == FHE_MODUP_APPROX, t_qp,
                          modup, stream)) < 0)
        return finish(-1);
    launched += r;
    if ((r = launch_ntt(digits, log_n, LK, (long)batch * dnum * LK, t_qp, false, stream)) < 0) return finish(-1);
    return finish(launched + r);
}

extern "C" int fhe_keyswitch_apply(uint64_t *out, const uint64_t *digits, const uint64_t *keys, const uint32_t *galois,
                                   int R, int log_n, int L, int K, int dnum, int batch, const fhe_ntt_tables *t_qp,
                                   void *stream) {
    const int LK = L + K;
    int s = check_shape(log_n, LK, (long)batch * dnum);
    if (s) return s;
    if ((s = check_tables(t_qp, log_n, LK))) return s;
    if (dnum < 1 || dnum > LK || R < 1 || R > kMaxRotations || (!galois && R != 1)) return FHE_EINVAL;
    if (!out || !digits || !keys || !aligned16(out) || !aligned16(digits) || !aligned16(keys)) return FHE_EINVAL;
    GaloisSet g = {};
    if (galois) {
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, galois) != cudaSuccess) cudaGetLastError();
        else if (a.type == cudaMemoryTypeDevice) return FHE_EDEVICE;
        const uint64_t two_n = 2ull << log_n;
        for (int r = 0; r < R; r++) {
            if (!(galois[r] & 1) || galois[r] >= two_n) return FHE_EINVAL;
            g.k[r] = galois[r];
        }
    }
    if ((s = select_device({out, digits, keys, t_qp->blob}))) return s;
    const size_t plane = ((size_t)LK << log_n) * 8;
    const Span so{out, 2 * plane * batch * R}, sd{digits, plane * dnum * batch}, sk{keys, 2 * plane * dnum * R},
        tb{t_qp->blob, t_qp->bytes};
    if (overlap(so, sd) || overlap(so, sk) || overlap(so, tb)) return FHE_EALIAS;
    const int r = galois ? launch_ks_ip_aut(out, digits, keys, log_n, LK, dnum, batch, R, g, t_qp, stream)
                         : launch_ks_ip(out, digits, keys, log_n, LK, dnum, batch, t_qp, stream);
    return finish(r);
}

extern "C" int fhe_bconv(uint64_t *out, const uint64_t *in, int log_n, int S, int T, int batch, int mode,
                         const void *bconv, void *stream) {
    size_t tb = 0;
    int s = fhe_bconv_tables_bytes(S, T, &tb);
    if (s) return s;
    if (log_n < 1 || log_n > kMaxLogN || batch < 1 || batch > 65535) return FHE_EINVAL;
    if (mode != FHE_BCONV_EXACT && mode != FHE_BCONV_APPROX) return FHE_EINVAL;
    if (!out || !in || !bconv || !aligned16(out) || !aligned16(in) || !aligned16(bconv)) return FHE_EINVAL;
    if ((s = select_device({out, in, bconv}))) return s;
    const Span so{out, ((size_t)batch * T << log_n) * 8}, si{in, ((size_t)batch * S << log_n) * 8}, st{bconv, tb};
    if (overlap(so, si) || overlap(so, st)) return FHE_EALIAS;
    return finish(launch_bconv(out, in, log_n, S, T, batch, mode == FHE_BCONV_APPROX, bconv, stream));
}


extern "C" int fhe_moddown_workspace_bytes(int log_n, int L, int K, int batch, size_t *bytes) {
    if (!bytes || log_n < 1 || log_n > kMaxLogN || L < 1 || K < 1 || K > kMaxAlpha || batch < 1) return FHE_EINVAL;
    *bytes = ((size_t)batch * (L + K) << log_n) * 8;
    return FHE_OK;
}

extern "C" int fhe_moddown(uint64_t *out, const uint64_t *in, int log_n, int L, int K, int batch, int domain,
                           int rounding, const fhe_ntt_tables *t_qp, const void *md, uint64_t *workspace,
                           size_t ws_bytes, void *stream) {
    size_t need = 0;
    int s = fhe_moddown_workspace_bytes(log_n, L, K, batch, &need);
    if (s) return s;
    if ((s = check_shape(log_n, L + K, batch))) return s;
    if ((s = check_tables(t_qp, log_n, L + K))) return s;
    if (domain != FHE_DOMAIN_COEFF && domain != FHE_DOMAIN_NTT) return FHE_EINVAL;
    if (rounding != FHE_ROUND_TRUNCATE && rounding != FHE_ROUND_NEAREST) return FHE_EINVAL;
    if (!out || !in || !md || !workspace) return FHE_EINVAL;
    if (!aligned16(out) || !aligned16(in) || !aligned16(md) || !aligned16(workspace)) return FHE_EINVAL;
    if (ws_bytes < need) return FHE_ESPACE;
    if ((s = select_device({out, in, md, workspace, t_qp->blob}))) return s;
    const Span so{out, ((size_t)batch * L << log_n) * 8}, si{in, ((size_t)batch * (L + K) << log_n) * 8},
        sw{workspace, need}, tb{t_qp->blob, t_qp->bytes}, sm{md, moddown_layout(L, K).bytes};
    if (overlap(so, si) || overlap(so, sw) || overlap(so, tb) || overlap(so, sm) || overlap(si, sw) ||
        overlap(sw, tb) || overlap(sw, sm))
        return FHE_EALIAS;
    return finish(launch_moddown(out, in, log_n, L, K, batch, domain == FHE_DOMAIN_NTT,
                                 rounding == FHE_ROUND_NEAREST, t_qp, md, workspace, stream));
}

extern "C" int fhe_rescale(uint64_t *out, const uint64_t *in, int log_n, int L, int batch, int domain, int rounding,
                           const fhe_ntt_tables *t_q, const void *rs, uint64_t *workspace, size_t ws_bytes,
                           void *stream) {
    if (L < 2) return FHE_EINVAL;
    return fhe_moddown(out, in, log_n, L - 1, 1, batch, domain, rounding, t_q, rs, workspace, ws_bytes, stream);
}
