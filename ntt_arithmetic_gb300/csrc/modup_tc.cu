// modup_tc.cu -- ModUp's basis extension as a tensor-core contraction.
//
// For digit j (primes d_0..d_{c-1}, product D) every coefficient x with
// residues x_a is extended to each target prime p outside the digit -- the
// "mixed-radix decomposition and basis extension" of FHElium's CUDA layer
// ("Eager, Compile, and native execution", section "CUDA execution") and the
// "Garner extension" of the kestrel-llm chain (overview, section 4.2).  With
// the CRT brackets y_a = [x_a (D/d_a)^-1]_{d_a},
//   sum_a y_a (D/d_a) = X + e D,   e = floor(sum_a y_a / d_a) < c,
// where X in [0, D) is the coefficient's CRT value.  The approximate
// conversion stops at X + e D; the exact one subtracts e D.  Over a tile of
// 128 coefficients and all targets this is a dense 128 x (8 targets) x (8 c)
// contraction, run on the tensor cores exactly:
//
//  * each y_a < 2^50 is split into bytes b_{a,e}; the A operand row of a
//    coefficient holds the fp16 values 1024 + b_{a,e} (bit pattern
//    0x6400 | b, one byte permute per two elements) and 1024 + e in the
//    spare column 15;
//  * the B operand (built on the host, tables.cpp: tc_weight_image) holds the
//    7-bit limbs of (D/d_a) 2^(8e) mod p, the limbs of (-D) mod p in column
//    15 and offset columns, so that every f32 accumulator is 2^23 + (an
//    integer below 2^21): products and sums of integers below 2^24 are exact
//    in f32, and the accumulator's bit pattern minus 0x4B000000 is the integer;
//  * the eight accumulators u_s of a target recombine as
//    S = sum_s u_s 2^(7s) = (u_0 + .. + u_3 2^21) + 2^28 (u_4 + .. + u_7 2^21).
//    S < 2^64: u_s <= 8 (6 * 255 + 3) 127 + 7 * 127 < 2^20.6 for s < 7 (a
//    bracket's byte 6 is below 4), and limb 7 of a constant below 2^50 is 0
//    or 1, so u_7 < 2^13.6 and S < 2^42 (2^20.6 * 1.008 + 2^13.6 2^7) < 2^63.6.
//    One Barrett step with mu = floor(2^64 / p) < 2^16 leaves S mod p below
//    2 p (the forward NTT that follows takes inputs of that size).
//
// e comes from a 64.64 fixed-point sum of y_a / d_a with the reciprocals
// floor(2^128 / d_a); every term is below the true value by less than 2, so
// the integer part is e unless the fraction lies within 2 c units of 1 (X near
// 0 or near D, i.e. small coefficients).  Those lanes compute e exactly:
// Garner's recursion gives X's mixed-radix digits w_a, X mod 2^64 =
// sum_a w_a (d_0 .. d_{a-1}) mod 2^64, and with the redundant modulus 2^64
// e = (sum_a y_a (D/d_a) - X) D^-1 mod 2^64.
//
// The integer pipes keep c Shoup products and c fixed-point products per
// coefficient and one Barrett step per output; the c multiply-accumulates
// per output of the integer kernel (modup.cu) move to the tensor cores.
//
// CTA: 128 threads, thread m owns coefficient m of the tile and row m of the
// accumulator (TMEM lane m).  Persistent over the tiles of one digit: the
// digit's B operand and constants are staged in shared memory once, and each
// thread loads its next tile's residues while the current one is converted.
// Targets are processed in groups of up to 16 (N = 128 columns), one MMA
// chain of K = 64 (4 instructions) per group into the CTA's 128 TMEM columns.
#include <cuda_runtime.h>

#include <cstdlib>

#include "fhe_arith.cuh"
#include "fhe_internal.h"
#include "launch_util.h"
#include "tc_util.cuh"

namespace fhe {

// Status word of the tensor-core kernels (FHE_STATUS_* bits), read and
// cleared by fhe_device_status.
__device__ int g_fhe_status;

namespace {

constexpr int kTcThreads = 128;                      // M = 128: one row per thread
constexpr int kTileBytesA = 128 * kTcRowBytes;       // A operand, 16 KB
constexpr uint32_t kCoreK = 128;                     // bytes between cores adjacent along K
constexpr uint32_t kCoreRows = kTcMaxAlpha * 128;    // bytes between cores adjacent along the rows
constexpr uint64_t kTcWaitNs = 200000000ull;         // give up an MMA wait after 200 ms
constexpr uint64_t kTcTestWaitNs = 1000000ull;       // the test hook's wait on a barrier nobody arrives on
constexpr uint32_t kF32Offset = 0x4B000000u;         // f32 bit pattern of 2^23

// Shared memory of one CTA for a digit with T targets (padded to even).
__host__ __device__ constexpr size_t tc_smem_bytes(int T) {
    return (size_t)kTileBytesA + (size_t)((T + 1) & ~1) * 8 * kTcRowBytes + (size_t)T * sizeof(ModupTcTarget);
}

// One source basis (a ModUp digit, or ModDown's P) of `cnt` primes extended to
// its T targets, for every coefficient of `batch` items: the body shared by
// k_modup_tc (MD = false: the digit's own limbs are copied to `out` as well)
// and k_moddown_tc (MD = true: the inputs get h added, the outputs get the
// target's `aux` added).  Source limb a of item bi is at
// in + bi in_stride + (lo + a) n; output row `limb` of item bi and digit j at
// out + ((bi dnum + j) out_rows + limb) n.
template <bool APPROX, bool MD>
__device__ __forceinline__ void ext_tc(uint8_t *sm, uint64_t *__restrict__ out, int out_rows,
                                       const uint64_t *__restrict__ in, long in_stride, int log_n, int batch,
                                       int lo, int cnt, int T, int j, int dnum, const ulonglong2 *__restrict__ qinv,
                                       const ulonglong2 *__restrict__ garner, int gstride,
                                       const ModupTcFrac *__restrict__ frac, const ModupTcTarget *__restrict__ tgt,
                                       const uint4 *__restrict__ wimg, const uint64_t *__restrict__ src_consts,
                                       const uint64_t *__restrict__ hsrc, bool test_timeout) {
    // qinv: the brackets' constants [cnt]; garner: [cnt][gstride] (the exact fallback).
    // test_timeout: every MMA wait is on `idle`, a barrier nothing arrives on, for 1 ms -- the path of a
    // wait that gives up, taken without any fault (the committed MMA still completes on `mbar`).
    __shared__ uint64_t mbar, idle;
    __shared__ uint32_t tslot;
    const int t = threadIdx.x, warp = t >> 5;
    const int Tp = (T + 1) & ~1;
    uint8_t *sA = sm, *sB = sm + kTileBytesA;
    ModupTcTarget *sT = reinterpret_cast<ModupTcTarget *>(sB + (size_t)Tp * 8 * kTcRowBytes);
    // the basis' constants, read inside the per-coefficient dependency chains
    __shared__ ulonglong2 sQ[kTcMaxAlpha];                   // bracket constants (D/d_a)^-1 mod d_a
    __shared__ ulonglong2 sG[kTcMaxAlpha * kTcMaxAlpha];     // Garner: (a, b) = d_b^-1 mod d_a, b < a
    __shared__ ModupTcFrac sF[kTcMaxAlpha + 1];              // reciprocals, redundant-modulus constants
    __shared__ uint64_t sD[kTcMaxAlpha], sH[kTcMaxAlpha];    // the source primes, h mod each (ModDown)
    {
        for (int e = t; e < Tp * 8 * kTcRowBytes / 16; e += kTcThreads)
            reinterpret_cast<uint4 *>(sB)[e] = __ldg(wimg + e);
        for (int e = t; e < T; e += kTcThreads) sT[e] = tgt[e];
        for (int e = t; e < kTcMaxAlpha * kTcMaxAlpha; e += kTcThreads) {
            const int a = e / kTcMaxAlpha, b = e - a * kTcMaxAlpha;
            sG[e] = (a < cnt && b < a) ? __ldg(garner + a * gstride + b) : make_ulonglong2(0, 0);
        }
        if (t < kTcMaxAlpha) {
            sQ[t] = t < cnt ? __ldg(qinv + t) : make_ulonglong2(0, 0);
            sD[t] = t < cnt ? __ldg(src_consts + (long)(lo + t) * K_COUNT + K_Q) : 0;
            sH[t] = (MD && hsrc && t < cnt) ? __ldg(hsrc + t) : 0;
        }
        if (t <= kTcMaxAlpha) sF[t] = frac[t];
    }
    if (warp == 0) tmem_alloc(&tslot, 128);
    if (t == 0) {
        mbar_init(&mbar, 1);
        mbar_init(&idle, 1);
    }
    fence_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tslot, lanes = (uint32_t)(32 * warp) << 16;
    const uint32_t a_addr = smem_u32(sA), b_addr = smem_u32(sB);
    uint8_t *arow = sA + (t >> 3) * kCoreRows + (t & 7) * 16;   // this thread's operand row
    const long tiles_per_item = (1L << log_n) >> 7;
    const long tiles = (long)batch * tiles_per_item;
    uint32_t phase = 0;
    bool ok = true;
    // the residues of the CTA's next tile are loaded while the current one is converted
    uint64_t xn[kTcMaxAlpha];
    auto load_tile = [&](long tile) {
        const int bi = (int)(tile / tiles_per_item);
        const uint64_t *src = in + (long)bi * in_stride + ((long)lo << log_n) +
                              ((tile - (long)bi * tiles_per_item) << 7) + t;
#pragma unroll
        for (int a = 0; a < kTcMaxAlpha; a++) xn[a] = a < cnt ? __ldcs(src + ((long)a << log_n)) : 0;
    };
    if (blockIdx.x < tiles) load_tile(blockIdx.x);
    for (long tile = blockIdx.x; ok && tile < tiles; tile += gridDim.x) {
        const int bi = (int)(tile / tiles_per_item);
        const long i = ((tile - (long)bi * tiles_per_item) << 7) + t;
        uint64_t x[kTcMaxAlpha], v[kTcMaxAlpha];
#pragma unroll
        for (int a = 0; a < kTcMaxAlpha; a++) x[a] = xn[a];
        if (tile + gridDim.x < tiles) load_tile(tile + gridDim.x);
        if constexpr (MD) {   // the residues of X + h
#pragma unroll
            for (int a = 0; a < kTcMaxAlpha; a++)
                if (a < cnt) x[a] = csub(x[a] + sH[a], sD[a]);
        }
        // CRT brackets v_a = [x_a (D/d_a)^-1]_{d_a}: sum_a v_a (D/d_a) = X + e D with
        // e = floor(sum_a v_a / d_a) < cnt
#pragma unroll
        for (int a = 0; a < kTcMaxAlpha; a++) {
            v[a] = 0;
            if (a < cnt) {
                const uint64_t d = sD[a];
                const ulonglong2 c = sQ[a];
                v[a] = reduce4(shoup_lazy(x[a], c.x, c.y, d), d);
            }
        }
        uint32_t ec = 0;   // the correction count e (0 for the approximate conversion)
        if constexpr (!APPROX) {
            // e from the 64.64 fixed-point sum of v_a / d_a (each term below the true value by < 2)
            uint64_t F = 0;
#pragma unroll
            for (int a = 0; a < kTcMaxAlpha; a++) {
                if (a < cnt) {
                    const uint64_t term = v[a] * sF[a].phi_hi + umulhi64(v[a], sF[a].phi_lo);
                    F += term;
                    ec += F < term;
                }
            }
            // X / D within 2 cnt 2^-64 of 1 (or of 0, wrapped): the sum may round either way
            const bool near = F > ~0ull - 2 * (uint64_t)cnt;
            if (__any_sync(0xffffffffu, near) && near) {
                // exact e by a redundant modulus: Garner gives X's mixed-radix digits w_a, and
                // e = (sum v_a (D/d_a) - X) D^-1 mod 2^64
                uint64_t w[kTcMaxAlpha];
                w[0] = x[0];
#pragma unroll
                for (int a = 1; a < kTcMaxAlpha; a++) {
                    w[a] = 0;
                    if (a < cnt) {
                        const uint64_t d = sD[a];
                        uint64_t u = x[a];
#pragma unroll
                        for (int b = 0; b < a; b++) {
                            const ulonglong2 c = sG[a * kTcMaxAlpha + b];
                            u = shoup_lazy(u + 4 * d - w[b], c.x, c.y, d);   // w_b < 2^50 < 4 d
                        }
                        w[a] = reduce4(u, d);
                    }
                }
                uint64_t Y = 0, X = 0;
#pragma unroll
                for (int a = 0; a < kTcMaxAlpha; a++) {
                    if (a < cnt) {
                        Y += v[a] * sF[a].dhat64;
                        X += w[a] * sF[a].w64;
                    }
                }
                ec = (uint32_t)((Y - X) * sF[kTcMaxAlpha].dhat64);
            }
        }
        uint64_t *dst = out + (((long)bi * dnum + j) * out_rows << log_n) + i;
        if constexpr (!MD) {
#pragma unroll
            for (int a = 0; a < kTcMaxAlpha; a++)
                if (a < cnt) __stcg(dst + ((long)(lo + a) << log_n), x[a]);   // limbs of the digit are copies
        }
        // A operand row: fp16 1024 + byte, eight per digit (byte 7 of v_a < 2^50 is 0);
        // column 15 (byte 7 of v_1) carries 1024 + e
#pragma unroll
        for (int a = 0; a < kTcMaxAlpha; a++) {
            const uint32_t vl = (uint32_t)v[a], vh = (uint32_t)(v[a] >> 32);
            uint4 row;
            row.x = __byte_perm(vl, 0x64646464u, 0x4140);
            row.y = __byte_perm(vl, 0x64646464u, 0x4342);
            row.z = __byte_perm(vh, 0x64646464u, 0x4140);
            row.w = __byte_perm(vh, 0x64646464u, 0x4342);
            if (8 * a + 7 == kTcCorrCol) row.w |= ec << 16;
            *reinterpret_cast<uint4 *>(arow + a * kCoreK) = row;
        }
        fence_async_smem();
        tc_fence_before_sync();
        __syncthreads();
        tc_fence_after_sync();
        for (int g0 = 0; g0 < T; g0 += kTcTargetsPerGroup) {
            const int gcnt = min(kTcTargetsPerGroup, T - g0);
            if (t == 0) {
                const uint32_t idesc = tc_idesc_f16_f32(8 * ((gcnt + 1) & ~1));
#pragma unroll
                for (int ks = 0; ks < kTcMaxAlpha / 2; ks++)
                    tc_mma_f16(tmem, tc_smem_desc(a_addr + ks * 2 * kCoreK, kCoreK, kCoreRows),
                               tc_smem_desc(b_addr + g0 * 8 * kTcRowBytes + ks * 2 * kCoreK, kCoreK, kCoreRows),
                               idesc, ks > 0);
                tc_commit(&mbar);
            }
            const bool done = test_timeout ? mbar_wait(&idle, 0, kTcTestWaitNs) : mbar_wait(&mbar, phase, kTcWaitNs);
            phase ^= 1;
            ok = __syncthreads_and(done);
            if (!ok) break;
            tc_fence_after_sync();
            for (int tt = 0; tt < gcnt; tt += 4) {
                uint32_t r[32];
                tmem_ld32(tmem + lanes + 8 * tt, r);   // targets tt .. tt + 3 (columns inside the group's N)
#pragma unroll
                for (int h = 0; h < 4; h++) {
                    if (tt + h < gcnt) {
                        const uint32_t *u = r + 8 * h;
                        // u_s = 2^23 bit pattern + d_s, d_s < 2^21: pairs d_s + d_{s+1} 2^7 < 2^29 taken
                        // mod 2^32 with the two offsets folded into one constant
                        const uint32_t p01 = u[0] + (u[1] << 7) - kF32Offset * 129u;
                        const uint32_t p23 = u[2] + (u[3] << 7) - kF32Offset * 129u;
                        const uint32_t p45 = u[4] + (u[5] << 7) - kF32Offset * 129u;
                        const uint32_t p67 = u[6] + (u[7] << 7) - kF32Offset * 129u;
                        const uint64_t l4 = (uint64_t)p23 * (1u << 14) + p01;   // d_0 + .. + d_3 2^21
                        const uint64_t h4 = (uint64_t)p67 * (1u << 14) + p45;   // d_4 + .. + d_7 2^21
                        const ModupTcTarget &tg = sT[g0 + tt + h];
                        const uint64_t r = reduce64_small_mu(l4 + (h4 << 28), tg.p, tg.mu);
                        // L2 policy: the column stages of the forward NTT read these next
                        __stcg(dst + ((long)tg.limb << log_n), MD && hsrc ? r + tg.aux : r);
                    }
                }
            }
            tc_fence_before_sync();
            __syncthreads();   // every lane's TMEM reads are done before the next MMA overwrites them
            tc_fence_after_sync();
        }
    }
    if (!ok) {
        if (t == 0) atomicOr(&g_fhe_status, FHE_STATUS_TC_TIMEOUT);
        mbar_wait(&mbar, phase ^ 1, kTcWaitNs);   // let the abandoned MMA finish before its columns are freed
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

template <bool APPROX>
__global__ void __launch_bounds__(kTcThreads, 4)
k_modup_tc(uint64_t *__restrict__ ext, const uint64_t *__restrict__ in, long in_stride, int log_n, int LK, int batch,
           int alpha, const ModupDigit *__restrict__ dg, const ulonglong2 *__restrict__ qinv,
           const ulonglong2 *__restrict__ garner, const ModupTcFrac *__restrict__ frac,
           const ModupTcTarget *__restrict__ tgt, const uint4 *__restrict__ wimg, int tmax,
           const uint64_t *__restrict__ consts, int test_timeout) {
    pdl_begin();
    extern __shared__ __align__(1024) uint8_t sm[];   // [A operand][B operand][targets]
    const int j = blockIdx.y;
    const int lo = dg[j].lo, cnt = dg[j].count;
    ext_tc<APPROX, false>(sm, ext, LK, in, in_stride, log_n, batch, lo, cnt, LK - cnt, j, gridDim.y,
                          qinv + (long)j * alpha, garner + (long)j * alpha * alpha, alpha,
                          frac + (long)j * (kTcMaxAlpha + 1), tgt + (long)j * tmax,
                          wimg + (size_t)j * tmax * 8 * kTcRowBytes / 16, consts, nullptr, test_timeout != 0);
}

// ModDown's conversion d_l = ((X + h) mod P) - h mod q_l (below 3 q_l, for the
// forward NTT) from the P limbs in[b][k][n], K <= kTcMaxAlpha.
__global__ void __launch_bounds__(kTcThreads, 4)
k_moddown_tc(uint64_t *__restrict__ d, const uint64_t *__restrict__ in, long in_stride, int log_n, int L, int K,
             int batch, const ulonglong2 *__restrict__ qinv, const ulonglong2 *__restrict__ garner,
             const ModupTcFrac *__restrict__ frac, const ModupTcTarget *__restrict__ tgt,
             const uint4 *__restrict__ wimg, const uint64_t *__restrict__ consts_p, const uint64_t *__restrict__ hp,
             int test_timeout) {
    pdl_begin();
    extern __shared__ __align__(1024) uint8_t sm[];
    ext_tc<false, true>(sm, d, L, in, in_stride, log_n, batch, 0, K, L, 0, 1, qinv, garner, K, frac, tgt, wimg,
                        consts_p, hp, test_timeout != 0);
}

// The test hook: FHE_TC_TEST_TIMEOUT=1 in the environment makes the tensor-core
// kernels take their give-up path (see ext_tc).
int tc_test_timeout() {
    const char *v = getenv("FHE_TC_TEST_TIMEOUT");
    return v && v[0] == '1' && v[1] == 0;
}

}  // namespace

int launch_modup_tc(uint64_t *ext, const uint64_t *in, long in_stride, int log_n, int L, int K, int dnum, int batch,
                    bool approx, const fhe_ntt_tables *t, const void *modup, void *stream) {
    cudaStream_t st = (cudaStream_t)stream;
    const ModupLayout lay = modup_layout(L, K, dnum);
    if (lay.tc_tmax == 0 || log_n < 7) return 0;
    const int LK = L + K;
    const int cnt_min = L - (dnum - 1) * lay.alpha;   // the last digit is the smallest
    const size_t need = tc_smem_bytes(LK - cnt_min);
    // at least 46 KB per CTA: at most 4 CTAs per SM, whose 4 x 128 TMEM columns fit the SM's 512
    const size_t smem = need > 47104 ? need : 47104;
    auto kern = approx ? k_modup_tc<true> : k_modup_tc<false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return -1;
    const int per_sm = (int)(228 * 1024 / (smem + 1024)) < 4 ? (int)(228 * 1024 / (smem + 1024)) : 4;
    const long tiles = (long)batch << (log_n - 7);
    // every CTA resident at once (a CTA left for a second wave would run its tiles alone at the end)
    long gx = (long)sm_count() * per_sm / dnum;
    if (gx < 1) gx = 1;
    if (gx > tiles) gx = tiles;
    const char *base = (const char *)modup;
    kern<<<dim3((unsigned)gx, (unsigned)dnum), kTcThreads, smem, st>>>(
        ext, in, in_stride, log_n, LK, batch, lay.alpha, (const ModupDigit *)(base + lay.off_digits),
        (const ulonglong2 *)(base + lay.off_qinv), (const ulonglong2 *)(base + lay.off_garner),
        (const ModupTcFrac *)(base + lay.off_tc_frac), (const ModupTcTarget *)(base + lay.off_tc_tgt),
        (const uint4 *)(base + lay.off_tc_b), lay.tc_tmax, t->consts, tc_test_timeout());
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

int launch_moddown_tc(uint64_t *d, const uint64_t *src, long src_item, int log_n, int L, int K, int batch, bool nearest,
                      const fhe_ntt_tables *t_qp, const void *md, void *stream) {
    cudaStream_t st = (cudaStream_t)stream;
    const ModdownLayout lay = moddown_layout(L, K);
    if (lay.tc_tmax == 0 || log_n < 7) return 0;
    const size_t need = tc_smem_bytes(L);
    const size_t smem = need > 47104 ? need : 47104;   // at most 4 CTAs per SM (TMEM)
    if (cudaFuncSetAttribute(k_moddown_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return -1;
    const int per_sm = (int)(228 * 1024 / (smem + 1024)) < 4 ? (int)(228 * 1024 / (smem + 1024)) : 4;
    const long tiles = (long)batch << (log_n - 7);
    long gx = (long)sm_count() * per_sm;
    if (gx > tiles) gx = tiles;
    const char *base = (const char *)md;
    launch_pdl(k_moddown_tc, dim3((unsigned)gx), kTcThreads, smem, st, d, src, src_item, log_n, L, K, batch,
               (const ulonglong2 *)(base + lay.off_tc_qinv), (const ulonglong2 *)(base + lay.off_garner),
               (const ModupTcFrac *)(base + lay.off_tc_frac), (const ModupTcTarget *)(base + lay.off_tc_tgt),
               (const uint4 *)(base + lay.off_tc_b), t_qp->consts + (long)L * K_COUNT,
               nearest ? (const uint64_t *)(base + lay.off_hp) : (const uint64_t *)nullptr, tc_test_timeout());
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

int device_status(int *status, bool reset) {
    if (cudaDeviceSynchronize() != cudaSuccess) return FHE_ECUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_fhe_status, sizeof(int)) != cudaSuccess) return FHE_ECUDA;
    if (reset && v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_fhe_status, &zero, sizeof(int)) != cudaSuccess) return FHE_ECUDA;
    }
    *status = v;
    return FHE_OK;
}

}  // namespace fhe
