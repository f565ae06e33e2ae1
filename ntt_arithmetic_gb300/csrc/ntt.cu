// ntt.cu -- batched negacyclic NTT / INTT over RNS primes on sm_103a.
//
// One (polynomial, prime) row of n = 2^LOGN residues is cut into C = 2^LOGC
// blocks of M = n / C residues (C = 1 for n <= 2^13), one CTA per block,
// which holds its block in registers and shared memory: the "compact
// grouped" / "fixed-radix shared-memory" execution FHElium describes for its
// CUDA NTT families ("Eager, Compile, and native execution", table "Native
// operator families").  For n >= 2^14 (the "split" shapes of ntt_shapes.h)
// the first LOGC forward stages (the last LOGC inverse stages), which mix
// the blocks, run in a column kernel over the whole row in one HBM pass, and
// the C block CTAs run independently after it (forward) or before it
// (inverse): a two-kernel decomposition.
//
// Forward (natural -> bit-reversed, psi-merged Cooley-Tukey):
//   stage s (s = 0 .. LOGN-1) pairs positions p and p + n/2^(s+1) inside blocks
//   of n/2^s and multiplies by psi^brv(2^s + block) (table fwd[2^s + block]).
//   * cross stages s < LOGC: the C elements {j1 M + j2 : j1 < C} of a column
//     j2 belong to C different blocks.  k_ntt_fwd_cols gives each column to a
//     few threads of one CTA and stores the stages' lazy results back in place;
//   * local stages s >= LOGC run in passes of up to LOGE stages: a thread
//     holds 2^LOGE residues (radix-2^LOGE in registers), with one shared-
//     memory round trip and one __syncthreads between passes (k_ntt_fwd for
//     C = 1, k_ntt_fwd_blk per block for C > 1).
// Inverse (bit-reversed -> natural): cyclic Cooley-Tukey (decimation in time)
//   with omega^-1 = psi^-2 followed by the twist n^-1 psi^-j; local passes
//   first (spans 1, 2, 4, ...), cross stages last -- the mirror image.  C = 1:
//   k_ntt_inv; C > 1: k_ntt_inv_blk runs the local passes and stores each
//   block back unreduced, then k_ntt_inv_cols runs the cross stages and the
//   twist.
//
// Twiddles: those that every thread of a CTA (or a warp) shares -- the
// forward's local passes but the last, the inverse's first two local passes,
// the inverse column kernel's per-column twiddles -- are copied into shared
// memory with cp.async at kernel start, overlapping the data load; the
// per-thread twiddles of the remaining stages are read from the table
// coalesced.
//
// Caching: residues move with the .cg (L2, no L1) policy, not the
// evict-first streaming policy: the kernel that runs next -- the other half of
// a split transform, or the product or automorphism that reads the transform's
// output -- then finds part of them in L2.
//
// Fused block kernels: the key switch's digit transform ends in the inner
// product with the keys (k_ntt_fwd_blk_ip) and ModDown's transform of its
// correction ends in the last product (x - d) P^-1 (k_ntt_fwd_blk_md); both
// keep the reduced block in shared memory instead of storing it.
//
// Arithmetic: lazy Shoup butterflies (fhe_arith.cuh).  Values grow by < 4q
// per stage with no comparisons and are reduced once, before the store.
// Forward inputs below B stay below B + 68 q after 17 stages: B = q for the
// public transform; the key switch's extended digits and ModDown's
// correction arrive below 20 q (their lazy Barrett outputs), so every value
// stays below 2^57.  Inverse: < 128 q, the twiddle-1 butterflies of its
// first pass doubling instead.
//
// Shared-memory index swizzle: index p is stored at p ^ (((p >> LOGE) & 7) << 1),
// which makes every pass's accesses bank-conflict-free (two wavefronts per
// 64-bit warp access) and keeps 16-byte pairs (2k, 2k+1) adjacent.
#include <cuda_runtime.h>

#include "fhe_arith.cuh"
#include "fhe_internal.h"
#include "launch_util.h"
#include "ntt_shapes.h"

namespace fhe {
namespace {

// 16-byte asynchronous global -> shared copy (no register holds the data in flight)
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }
// wait until at most the most recent committed group is still in flight
__device__ __forceinline__ void cp_async_wait_but_last() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }

template <int LOGN_, int LOGC_, int LOGT_, int LOGE_>
struct Shape {
    static constexpr int LOGN = LOGN_, LOGC = LOGC_, LOGT = LOGT_, LOGE = LOGE_;
    static constexpr int N = 1 << LOGN, C = 1 << LOGC, LOGM = LOGN - LOGC, M = 1 << LOGM;
    static constexpr int T = 1 << LOGT, E = 1 << LOGE;
    static constexpr int P = (LOGM + LOGE - 1) / LOGE;     // local passes
    static constexpr int EREM = LOGM - (P - 1) * LOGE;     // stages in the odd-sized pass
    static_assert(LOGM == LOGT + LOGE, "M = T * E");
    // Staged twiddles (shared memory, after the data block), copied there
    // asynchronously at kernel start so that their latency overlaps the data
    // load instead of stalling the first butterflies of each stage.
    // Forward: every local pass but the last, laid out [pass 0][pass 1]...,
    // stage I of pass PI holding the CTA's 2^(LOGM - B - EP + I) consecutive
    // table entries (the last pass reads the table directly, coalesced).
    __host__ __device__ static constexpr int pass_b(int pi) { return (P - 1 - pi) * LOGE; }
    __host__ __device__ static constexpr int pass_ep(int pi) { return pi == 0 ? EREM : LOGE; }
    __host__ __device__ static constexpr int pass_cnt(int pi) {
        return (1 << (LOGM - pass_b(pi) - pass_ep(pi))) * ((1 << pass_ep(pi)) - 1);
    }
    __host__ __device__ static constexpr int seg_off(int pi) { return pi == 0 ? 0 : seg_off(pi - 1) + pass_cnt(pi - 1); }
    static constexpr int FWD_TW = P >= 2 ? seg_off(P - 1) : 0;
    // Inverse: table entries [1, 2^ILOG) -- every twiddle of the first two
    // local passes, which depend on the position inside the block only.
    static constexpr int ILOG = LOGM < 2 * LOGE ? LOGM : 2 * LOGE;
    static constexpr int INV_TW = 1 << ILOG;
    static constexpr int smem_words(bool inverse) { return M + 2 * (inverse ? INV_TW : FWD_TW); }
};

struct Ctx {
    const ulonglong2 *tw;   // this prime's twiddle pairs (w, floor(w 2^64 / q))
    const uint64_t *kc;     // this prime's constants
    uint64_t q;
    int t;                  // thread index
    int r;                  // block index within the row
    const ulonglong2 *etw;  // staged twiddles (shared memory)
};

template <int LOGE>
__device__ __forceinline__ int swz(int p) { return p ^ (((p >> LOGE) & 7) << 1); }

// Position inside the CTA's block of the j-th residue of group g in a pass
// covering local bit positions [B, B + EP).
template <int B, int EP>
__device__ __forceinline__ int pass_pos(int g, int j) {
    return (g & ((1 << B) - 1)) | (j << B) | ((g >> B) << (B + EP));
}

template <class SH, int B, int EP>
__device__ __forceinline__ void smem_load(uint64_t (&x)[SH::E], const uint64_t *sm, int t) {
    constexpr int G = SH::E >> EP, EPN = 1 << EP;
#pragma unroll
    for (int k = 0; k < G; k++) {
        const int g = t + SH::T * k;
        if constexpr (B == 0 && EP >= 1) {
#pragma unroll
            for (int j = 0; j < EPN; j += 2) {
                const ulonglong2 v = *reinterpret_cast<const ulonglong2 *>(sm + swz<SH::LOGE>(pass_pos<B, EP>(g, j)));
                x[k * EPN + j] = v.x;
                x[k * EPN + j + 1] = v.y;
            }
        } else {
#pragma unroll
            for (int j = 0; j < EPN; j++) x[k * EPN + j] = sm[swz<SH::LOGE>(pass_pos<B, EP>(g, j))];
        }
    }
}

template <class SH, int B, int EP>
__device__ __forceinline__ void smem_store(const uint64_t (&x)[SH::E], uint64_t *sm, int t) {
    constexpr int G = SH::E >> EP, EPN = 1 << EP;
#pragma unroll
    for (int k = 0; k < G; k++) {
        const int g = t + SH::T * k;
        if constexpr (B == 0 && EP >= 1) {
#pragma unroll
            for (int j = 0; j < EPN; j += 2) {
                *reinterpret_cast<ulonglong2 *>(sm + swz<SH::LOGE>(pass_pos<B, EP>(g, j))) =
                    make_ulonglong2(x[k * EPN + j], x[k * EPN + j + 1]);
            }
        } else {
#pragma unroll
            for (int j = 0; j < EPN; j++) sm[swz<SH::LOGE>(pass_pos<B, EP>(g, j))] = x[k * EPN + j];
        }
    }
}

// HBM <-> registers for a pass; `blk` points at this CTA's block of M residues.
template <class SH, int B, int EP>
__device__ __forceinline__ void global_load(uint64_t (&x)[SH::E], const uint64_t *blk, int t) {
    constexpr int G = SH::E >> EP, EPN = 1 << EP;
#pragma unroll
    for (int k = 0; k < G; k++) {
        const int g = t + SH::T * k;
        if constexpr (B == 0 && EP >= 1) {
#pragma unroll
            for (int j = 0; j < EPN; j += 2) {
                const ulonglong2 v = __ldcg(reinterpret_cast<const ulonglong2 *>(blk + pass_pos<B, EP>(g, j)));
                x[k * EPN + j] = v.x;
                x[k * EPN + j + 1] = v.y;
            }
        } else {
#pragma unroll
            for (int j = 0; j < EPN; j++) x[k * EPN + j] = __ldcg(blk + pass_pos<B, EP>(g, j));
        }
    }
}

template <class SH, int B, int EP>
__device__ __forceinline__ void global_store(const uint64_t (&x)[SH::E], uint64_t *blk, int t) {
    constexpr int G = SH::E >> EP, EPN = 1 << EP;
#pragma unroll
    for (int k = 0; k < G; k++) {
        const int g = t + SH::T * k;
        if constexpr (B == 0 && EP >= 1) {
#pragma unroll
            for (int j = 0; j < EPN; j += 2)
                __stcg(reinterpret_cast<ulonglong2 *>(blk + pass_pos<B, EP>(g, j)),
                       make_ulonglong2(x[k * EPN + j], x[k * EPN + j + 1]));
        } else {
#pragma unroll
            for (int j = 0; j < EPN; j++) __stcg(blk + pass_pos<B, EP>(g, j), x[k * EPN + j]);
        }
    }
}

// Coalesced copies of the CTA's block between HBM (natural order) and shared
// memory (swizzled): each warp instruction moves 512 contiguous bytes.  The
// register passes that touch the lowest index bits hold 2^LOGE consecutive
// residues per thread, so reading or writing HBM straight from them would
// scatter every warp access over 32 lines; staging through shared memory
// (conflict-free under the swizzle) avoids that.
template <class SH>
__device__ __forceinline__ void block_load_coalesced(uint64_t *sm, const uint64_t *blk, int t) {
#pragma unroll
    for (int k = 0; k < SH::E / 2; k++) {
        const int p = 2 * (t + SH::T * k);
        *reinterpret_cast<ulonglong2 *>(sm + swz<SH::LOGE>(p)) = __ldcg(reinterpret_cast<const ulonglong2 *>(blk + p));
    }
}

template <class SH>
__device__ __forceinline__ void block_store_coalesced(const uint64_t *sm, uint64_t *blk, int t) {
#pragma unroll
    for (int k = 0; k < SH::E / 2; k++) {
        const int p = 2 * (t + SH::T * k);
        __stcg(reinterpret_cast<ulonglong2 *>(blk + p), *reinterpret_cast<const ulonglong2 *>(sm + swz<SH::LOGE>(p)));
    }
}

// ---------------------------------------------------------------- forward --

// Local stage I of a pass over bits [B, B+EP): global stage s = LOGN-B-EP+I,
// register distance 2^(EP-1-I), 2^I distinct twiddles per group.
template <class SH, int B, int EP, int I>
__device__ __forceinline__ void fwd_stage(uint64_t (&x)[SH::E], const Ctx &c) {
    constexpr int G = SH::E >> EP, EPN = 1 << EP;
    constexpr int S = SH::LOGN - B - EP + I;
    constexpr int HALF = 1 << (EP - 1 - I);
    constexpr int NW = 1 << I;
    if constexpr (B + EP == SH::LOGM && G > 1) {
        // first local pass: g >> B is 0 for every group, so the twiddles are
        // the same for all groups of the CTA -- load them once
        constexpr int PI = SH::P - 1 - B / SH::LOGE;
        constexpr int OFF = SH::seg_off(PI) + (1 << (SH::LOGM - B - EP)) * ((1 << I) - 1);
#pragma unroll
        for (int jj = 0; jj < NW; jj++) {
            const ulonglong2 w = c.etw[OFF + jj];
#pragma unroll
            for (int k = 0; k < G; k++) {
#pragma unroll
                for (int u = 0; u < HALF; u++) {
                    const int j = jj * 2 * HALF + u;
                    ct_bfly(x[k * EPN + j], x[k * EPN + j + HALF], w.x, w.y, c.q);
                }
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < G; k++) {
            const int g = c.t + SH::T * k;
            const int base = (1 << S) + (c.r << (SH::LOGM - B - EP + I)) + ((g >> B) << I);
#pragma unroll
            for (int jj = 0; jj < NW; jj++) {
                // the last pass (B = 0) reads its twiddles from the (r, jj, g)
                // order of the table (fwd_table_slot): coalesced across g
                const int slot = B == 0 ? (1 << S) + (c.r << (SH::LOGM - EP + I)) + (jj << (SH::LOGM - EP)) + g
                                        : base + jj;
                ulonglong2 w;
                if constexpr (B == 0) {
                    w = __ldg(c.tw + slot);
                } else {
                    constexpr int PI = SH::P - 1 - B / SH::LOGE;
                    constexpr int OFF = SH::seg_off(PI) + (1 << (SH::LOGM - B - EP)) * ((1 << I) - 1);
                    w = c.etw[OFF + ((g >> B) << I) + jj];
                }
#pragma unroll
                for (int u = 0; u < HALF; u++) {
                    const int j = jj * 2 * HALF + u;
                    ct_bfly(x[k * EPN + j], x[k * EPN + j + HALF], w.x, w.y, c.q);
                }
            }
        }
    }
}

template <class SH, int B, int EP, int I = 0>
__device__ __forceinline__ void fwd_compute(uint64_t (&x)[SH::E], const Ctx &c) {
    if constexpr (I < EP) {
        fwd_stage<SH, B, EP, I>(x, c);
        fwd_compute<SH, B, EP, I + 1>(x, c);
    }
}

// KEEP: the reduced block is left in shared memory (swizzled) instead of
// being stored to `blk` (the fused key-switch kernel consumes it there).
template <class SH, int PI, bool KEEP = false>
__device__ __forceinline__ void fwd_passes(uint64_t (&x)[SH::E], uint64_t *sm, uint64_t *blk, const Ctx &c) {
    constexpr int LOGE = SH::LOGE;
    constexpr int B = (SH::P - 1 - PI) * LOGE;
    constexpr int EP = PI == 0 ? SH::EREM : LOGE;
    fwd_compute<SH, B, EP>(x, c);
    if constexpr (PI + 1 < SH::P) {
        smem_store<SH, B, EP>(x, sm, c.t);
        __syncthreads();
        constexpr int B2 = (SH::P - 2 - PI) * LOGE;
        smem_load<SH, B2, LOGE>(x, sm, c.t);
        fwd_passes<SH, PI + 1, KEEP>(x, sm, blk, c);
    } else {
        const uint32_t c58 = (uint32_t)c.kc[K_C58];
#pragma unroll
        for (int i = 0; i < SH::E; i++) x[i] = reduce_small(x[i], c.q, c58);
        if constexpr (KEEP) {
            static_assert(B == 0, "the fused key switch runs on the split shapes");
            smem_store<SH, B, EP>(x, sm, c.t);
        } else if constexpr (B == 0 && SH::E >= 2) {
            smem_store<SH, B, EP>(x, sm, c.t);   // each thread rewrites the positions it read
            __syncthreads();
            block_store_coalesced<SH>(sm, blk, c.t);
        } else {
            global_store<SH, B, EP>(x, blk, c.t);
        }
    }
}

// Row (batch item b, limb l) of the group of C blocks of CTA index `bid`.
// Rows are numbered limb-major (all batch items of limb 0, then of limb 1,
// ...), so the CTAs resident at one time share a few primes' twiddle tables
// and a table is fetched from DRAM about once per launch however long the
// chain is.  A kernel that consumes what the kernel before it wrote in this
// order walks it backwards (bid = gridDim.x - 1 - blockIdx.x): the rows
// written last are read first, while they are still in L2.
template <int LOGC>
__device__ __forceinline__ long row_of(int L, int batch, int &l, unsigned bid = blockIdx.x) {
    const long cl = (long)(bid >> LOGC);
    l = (int)(cl / batch);
    return (cl - (long)l * batch) * L + l;
}

template <class SH, int PI>
__device__ __forceinline__ void etw_issue_pass(ulonglong2 *etw, const ulonglong2 *tw, int r, int t) {
    if constexpr (PI < SH::P - 1) {
        constexpr int B = SH::pass_b(PI), EP = SH::pass_ep(PI);
#pragma unroll
        for (int I = 0; I < EP; I++) {
            const int cnt = 1 << (SH::LOGM - B - EP + I);
            const int off = SH::seg_off(PI) + (1 << (SH::LOGM - B - EP)) * ((1 << I) - 1);
            const ulonglong2 *src = tw + (1 << (SH::LOGN - B - EP + I)) + ((long)r << (SH::LOGM - B - EP + I));
            for (int u = t; u < cnt; u += SH::T) cp_async16(etw + off + u, src + u);
        }
        etw_issue_pass<SH, PI + 1>(etw, tw, r, t);
    }
}

// One CTA per row (C = 1): every stage is local.
template <int LOGN, int LOGC, int LOGT, int LOGE, int MINB>
__global__ void __launch_bounds__(1 << LOGT, MINB)
k_ntt_fwd(uint64_t *__restrict__ res, int L, int batch, const ulonglong2 *__restrict__ tw,
          const uint64_t *__restrict__ consts) {
    pdl_begin();
    using SH = Shape<LOGN, LOGC, LOGT, LOGE>;
    static_assert(SH::C == 1, "a row of more than one block takes the split kernels");
    extern __shared__ __align__(16) uint64_t sm[];
    Ctx c;
    c.t = threadIdx.x;
    c.r = 0;
    int l;
    const long row = row_of<LOGC>(L, batch, l);
    uint64_t *data = res + row * SH::N;
    c.tw = tw + (long)l * SH::N;
    c.kc = consts + (long)l * K_COUNT;
    c.q = c.kc[K_Q];
    ulonglong2 *etw = reinterpret_cast<ulonglong2 *>(sm + SH::M);
    c.etw = etw;
    etw_issue_pass<SH, 0>(etw, c.tw, c.r, c.t);
    cp_async_commit();
    uint64_t x[SH::E];
    global_load<SH, (SH::P - 1) * LOGE, SH::EREM>(x, data, c.t);
    cp_async_wait_all();
    __syncthreads();   // the staged twiddles are visible to every thread
    fwd_passes<SH, 0>(x, sm, data, c);
}

// ------------------------------------------------------- split forward --
//
// The cross stages of a split shape as a kernel of their own.  CTA (l, chunk,
// part) owns COLS adjacent columns j2 of prime l for up to `chunk` consecutive
// batch items, and loads item b + 1 while it transforms item b.  The TPC =
// 2^LOGTPC threads of a column j2 hold its C residues j1 M + j2 (stride M,
// coalesced across the CTA's COLS adjacent columns), first as j1 = g + TPC i
// for the stages of span >= TPC, then -- after one shared-memory exchange --
// as j1 = VPT g + i for the spans below TPC.  Every twiddle depends on j1
// only (fwd[2^s + (j1 >> (LOGC - s))], warp-uniform).  The outputs are
// stored in place unreduced (< (4 LOGC + 1) q), the block kernel's input.
template <int LOGN, int LOGC, int LOGTPC>
__global__ void __launch_bounds__(256, 4)
k_ntt_fwd_cols(uint64_t *__restrict__ res, int L, int batch, int chunk, const ulonglong2 *__restrict__ tw,
               const uint64_t *__restrict__ consts) {
    pdl_begin();
    constexpr int C = 1 << LOGC, M = 1 << (LOGN - LOGC);
    constexpr int TPC = 1 << LOGTPC, LOGVPT = LOGC - LOGTPC, VPT = 1 << LOGVPT;
    constexpr int COLS = 256 / TPC, CPR = M / COLS;   // columns per CTA, CTAs per row
    static_assert(LOGTPC <= LOGVPT, "the spans below TPC lie inside one thread's run of VPT residues");
    static_assert(M % COLS == 0, "whole CTAs per row");
    __shared__ uint64_t tile[C][COLS];
    // limb-major (as row_of): the CTAs running together share a prime
    const int part = (int)(blockIdx.x % CPR);
    const int nch = (batch + chunk - 1) / chunk;
    const int rest = (int)(blockIdx.x / CPR);
    const int l = rest / nch, b0 = (rest - l * nch) * chunk;
    const int b1 = min(batch, b0 + chunk);
    const int cl = threadIdx.x % COLS, g = threadIdx.x / COLS;
    const uint64_t q = __ldg(consts + (long)l * K_COUNT + K_Q);
    const ulonglong2 *w = tw + ((long)l << LOGN);
    const long rstride = (long)L << LOGN;   // between consecutive batch items of one prime
    uint64_t *p = res + ((long)b0 * L + l) * ((long)1 << LOGN) + part * COLS + cl;
    uint64_t xn[VPT];
#pragma unroll
    for (int i = 0; i < VPT; i++) xn[i] = __ldcg(p + (long)(g + TPC * i) * M);
    for (int b = b0; b < b1; b++, p += rstride) {
        uint64_t x[VPT];
#pragma unroll
        for (int i = 0; i < VPT; i++) x[i] = xn[i];
        if (b + 1 < b1) {
#pragma unroll
            for (int i = 0; i < VPT; i++) xn[i] = __ldcg(p + rstride + (long)(g + TPC * i) * M);
        }
#pragma unroll
        for (int S = 0; S < LOGVPT; S++) {
            const int HI = VPT >> (S + 1);   // span C / 2^(S+1) = TPC HI in j1
#pragma unroll
            for (int i = 0; i < VPT; i++) {
                if (i & HI) continue;
                const ulonglong2 wt = __ldg(w + (1 << S) + ((g + TPC * i) >> (LOGC - S)));
                ct_bfly(x[i], x[i + HI], wt.x, wt.y, q);
            }
        }
        if constexpr (LOGTPC > 0) {
            if (b > b0) __syncthreads();   // the previous item's tile reads are done
#pragma unroll
            for (int i = 0; i < VPT; i++) tile[g + TPC * i][cl] = x[i];
            __syncthreads();
#pragma unroll
            for (int i = 0; i < VPT; i++) x[i] = tile[VPT * g + i][cl];
#pragma unroll
            for (int S = LOGVPT; S < LOGC; S++) {
                const int HI = 1 << (LOGC - 1 - S);   // span < TPC <= VPT
#pragma unroll
                for (int i = 0; i < VPT; i++) {
                    if (i & HI) continue;
                    const ulonglong2 wt = __ldg(w + (1 << S) + ((VPT * g + i) >> (LOGC - S)));
                    ct_bfly(x[i], x[i + HI], wt.x, wt.y, q);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < VPT; i++) __stcg(p + (long)(LOGTPC > 0 ? VPT * g + i : g + TPC * i) * M, x[i]);
    }
}

// The local stages of a split shape: CTA r of a row transforms block r
// (residues [r M, (r + 1) M)) on its own, with the same passes, twiddle
// staging and coalesced store as the one-CTA kernel.
template <int LOGN, int LOGC, int LOGT, int LOGE, int MINB>
__global__ void __launch_bounds__(1 << LOGT, MINB)
k_ntt_fwd_blk(uint64_t *__restrict__ res, int L, int batch, const ulonglong2 *__restrict__ tw,
              const uint64_t *__restrict__ consts) {
    pdl_begin();
    using SH = Shape<LOGN, LOGC, LOGT, LOGE>;
    extern __shared__ __align__(16) uint64_t sm[];
    Ctx c;
    c.t = threadIdx.x;
    // last rows first: the column kernel wrote them last, so they are still in L2
    const unsigned bid = gridDim.x - 1 - blockIdx.x;
    c.r = (int)(bid & (SH::C - 1));
    int l;
    const long row = row_of<LOGC>(L, batch, l, bid);
    uint64_t *blk = res + row * SH::N + (long)c.r * SH::M;
    c.tw = tw + (long)l * SH::N;
    c.kc = consts + (long)l * K_COUNT;
    c.q = c.kc[K_Q];
    ulonglong2 *etw = reinterpret_cast<ulonglong2 *>(sm + SH::M);
    c.etw = etw;
    etw_issue_pass<SH, 0>(etw, c.tw, c.r, c.t);   // the local passes' shared twiddles (no cross stages here)
    cp_async_commit();
    uint64_t x[SH::E];
    global_load<SH, (SH::P - 1) * LOGE, SH::EREM>(x, blk, c.t);
    cp_async_wait_all();
    __syncthreads();   // the staged twiddles are visible to every thread
    fwd_passes<SH, 0>(x, sm, blk, c);
}

// The last LOGM stages of the extended digits' forward NTT fused with the
// key-switch inner product (FHElium, "Eager, Compile, and native
// execution", section "CUDA execution": "key-switch multiply-accumulate"):
// CTA (l, r, b) transforms block r of row (b, j, l) for every digit j < DN,
// keeps the DN reduced blocks in shared memory, then computes
//   out[b][c][l][p] = sum_j D_j[p] keys[j][c][l][p]  mod q_l   (c = 0, 1)
// for the block's positions p, with each key word read once per CTA and the
// output written once: the transformed digits never return to HBM.  The
// batch index varies fastest over the grid, so the CTAs that read the same
// key blocks run together and the keys come from DRAM about once per call.
// Sums are exact multiply-accumulates of 25-bit halves reduced once.
template <int LOGN, int LOGC, int LOGT, int LOGE, int MINB, int DN>
__global__ void __launch_bounds__(1 << LOGT, MINB)
k_ntt_fwd_blk_ip(uint64_t *__restrict__ out, const uint64_t *__restrict__ ext, const uint64_t *__restrict__ keys,
                 int LK, int batch, const ulonglong2 *__restrict__ tw, const uint64_t *__restrict__ consts) {
    pdl_begin();
    using SH = Shape<LOGN, LOGC, LOGT, LOGE>;
    extern __shared__ __align__(16) uint64_t sm[];   // [DN][M] digit blocks, then the staged twiddles
    const unsigned bid = gridDim.x - 1 - blockIdx.x;   // last rows first (still in L2)
    const int b = (int)(bid % (unsigned)batch);
    const int rest = (int)(bid / (unsigned)batch);
    Ctx c;
    c.t = threadIdx.x;
    c.r = rest & (SH::C - 1);
    const int l = rest >> SH::LOGC;
    c.tw = tw + (long)l * SH::N;
    c.kc = consts + (long)l * K_COUNT;
    c.q = c.kc[K_Q];
    ulonglong2 *etw = reinterpret_cast<ulonglong2 *>(sm + DN * SH::M);
    c.etw = etw;
    etw_issue_pass<SH, 0>(etw, c.tw, c.r, c.t);
    cp_async_commit();
    const long plane = (long)LK << LOGN;   // one [LK][n] block
    const long boff = (long)l * SH::N + (long)c.r * SH::M;
    if (c.t == 0) {
        // the later digit blocks and this block's keys, fetched into L2 while the first digit is transformed
        for (int j = 1; j < DN; j++)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(ext + ((long)b * DN + j) * plane + boff),
                         "r"(SH::M * 8) : "memory");
        for (int j = 0; j < 2 * DN; j++)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(keys + (long)j * plane + boff),
                         "r"(SH::M * 8) : "memory");
    }
#pragma unroll 1
    for (int j = 0; j < DN; j++) {
        uint64_t x[SH::E];
        global_load<SH, (SH::P - 1) * LOGE, SH::EREM>(x, ext + ((long)b * DN + j) * plane + boff, c.t);
        if (j == 0) {
            cp_async_wait_all();
            __syncthreads();   // the staged twiddles are visible to every thread
        }
        fwd_passes<SH, 0, true>(x, sm + j * SH::M, nullptr, c);
    }
    __syncthreads();   // every digit block is in shared memory
    const uint64_t mu = c.kc[K_MU12];
    const uint32_t c58 = (uint32_t)c.kc[K_C58];
    uint64_t *o0 = out + (long)b * 2 * plane + boff, *o1 = o0 + plane;
#pragma unroll 2
    for (int k = 0; k < SH::E / 2; k++) {
        const int p = 2 * (c.t + SH::T * k);
        Mac25 a0x, a0y, a1x, a1y;
#pragma unroll
        for (int j = 0; j < DN; j++) {
            const ulonglong2 d = *reinterpret_cast<const ulonglong2 *>(sm + j * SH::M + swz<SH::LOGE>(p));
            const ulonglong2 k0 = __ldg(reinterpret_cast<const ulonglong2 *>(keys + (2L * j) * plane + boff + p));
            const ulonglong2 k1 = __ldg(reinterpret_cast<const ulonglong2 *>(keys + (2L * j + 1) * plane + boff + p));
            const Split25 dx = split25(d.x), dy = split25(d.y);
            mac25(a0x, dx, split25(k0.x));
            mac25(a0y, dy, split25(k0.y));
            mac25(a1x, dx, split25(k1.x));
            mac25(a1y, dy, split25(k1.y));
        }
        __stcg(reinterpret_cast<ulonglong2 *>(o0 + p),
               make_ulonglong2(mac25_reduce(a0x, 0, c.q, mu, c58), mac25_reduce(a0y, 0, c.q, mu, c58)));
        __stcg(reinterpret_cast<ulonglong2 *>(o1 + p),
               make_ulonglong2(mac25_reduce(a1x, 0, c.q, mu, c58), mac25_reduce(a1y, 0, c.q, mu, c58)));
    }
}

// The block stages of the forward NTT of ModDown's correction d fused with
// ModDown's last step (FHElium, "Eager, Compile, and native execution",
// section "CUDA execution": "QP-to-Q ModDown"): CTA (row (b, l), block r)
// transforms block r of d[b][l] and writes
//   out[b][l][p] = (in[b][l][p] - NTT(d)[b][l][p]) P^-1  mod q_l
// for the block's positions p, with in the NTT-domain input over Q u P
// (item stride L + K rows).  The transformed d never returns to HBM.
template <int LOGN, int LOGC, int LOGT, int LOGE, int MINB>
__global__ void __launch_bounds__(1 << LOGT, MINB)
k_ntt_fwd_blk_md(uint64_t *__restrict__ out, const uint64_t *__restrict__ d, const uint64_t *__restrict__ in, int L,
                 int K, int batch, const ulonglong2 *__restrict__ tw, const uint64_t *__restrict__ consts,
                 const ulonglong2 *__restrict__ pinv) {
    pdl_begin();
    using SH = Shape<LOGN, LOGC, LOGT, LOGE>;
    extern __shared__ __align__(16) uint64_t sm[];
    Ctx c;
    c.t = threadIdx.x;
    const unsigned bid = gridDim.x - 1 - blockIdx.x;   // last rows first (still in L2)
    c.r = (int)(bid & (SH::C - 1));
    int l;
    const long row = row_of<LOGC>(L, batch, l, bid);
    const long b = row / L;
    c.tw = tw + (long)l * SH::N;
    c.kc = consts + (long)l * K_COUNT;
    c.q = c.kc[K_Q];
    ulonglong2 *etw = reinterpret_cast<ulonglong2 *>(sm + SH::M);
    c.etw = etw;
    uint64_t *xs = sm + SH::M + 2 * SH::FWD_TW;   // the block of x, for the last product
    const uint64_t *src = in + ((b * (L + K) + l) << LOGN) + (long)c.r * SH::M;
    etw_issue_pass<SH, 0>(etw, c.tw, c.r, c.t);
    cp_async_commit();
    // x is only needed after the transform: its copy is a commit group of its
    // own, so the first pass waits for the staged twiddles alone
    for (int u = 2 * c.t; u < SH::M; u += 2 * SH::T) cp_async16(xs + u, src + u);
    cp_async_commit();
    uint64_t x[SH::E];
    global_load<SH, (SH::P - 1) * LOGE, SH::EREM>(x, d + row * SH::N + (long)c.r * SH::M, c.t);
    cp_async_wait_but_last();
    __syncthreads();   // the staged twiddles are visible to every thread
    fwd_passes<SH, 0, true>(x, sm, nullptr, c);
    cp_async_wait_all();
    __syncthreads();   // the reduced block and x are in shared memory
    const ulonglong2 pi = __ldg(pinv + l);
    uint64_t *dst = out + row * SH::N + (long)c.r * SH::M;
#pragma unroll
    for (int k = 0; k < SH::E / 2; k++) {
        const int p = 2 * (c.t + SH::T * k);
        const ulonglong2 dv = *reinterpret_cast<const ulonglong2 *>(sm + swz<SH::LOGE>(p));
        const ulonglong2 xv = *reinterpret_cast<const ulonglong2 *>(xs + p);
        __stcs(reinterpret_cast<ulonglong2 *>(dst + p),
               make_ulonglong2(reduce4(shoup_lazy(xv.x + c.q - dv.x, pi.x, pi.y, c.q), c.q),
                               reduce4(shoup_lazy(xv.y + c.q - dv.y, pi.x, pi.y, c.q), c.q)));
    }
}

// ---------------------------------------------------------------- inverse --
//
// Cyclic Cooley-Tukey (decimation in time) on the bit-reversed input, then the
// twist n^-1 psi^-j on natural-order output j:
//   a_j = n^-1 psi^-j sum_k A_k omega^-jk,  omega = psi^2,  A[k] stored at brv(k).
// The stage of span h = 2^e pairs p and p + h (p mod 2h < h) and multiplies the
// second by omega_2h^-(p mod h) = inv[h + (p mod h)], so all butterflies are the
// comparison-free lazy Cooley-Tukey kind; values grow by < 4q per stage.  In
// the first register pass (spans 1 .. 2^(LOGE-1)) the twiddles are the same
// for every thread and one in 2^i butterflies of stage i has twiddle 1, whose
// multiplication is skipped.

// Bound, in units of q, of the values entering stage I of the first pass:
// inputs are < q; a twiddle-1 butterfly doubles the bound, the others add 4q.
template <int I>
struct FirstBound {
    static constexpr int prev = FirstBound<I - 1>::value;
    static constexpr int value = 2 * prev > prev + 4 ? 2 * prev : prev + 4;
};
template <>
struct FirstBound<0> {
    static constexpr int value = 1;
};

// Local stage I of an inverse pass over bits [B, B+EP): span 2^(B+I), register
// distance 2^I, twiddle inv[2^(B+I) + (p mod 2^(B+I))].
template <class SH, int B, int EP, int I>
__device__ __forceinline__ void inv_stage(uint64_t (&x)[SH::E], const Ctx &c) {
    constexpr int G = SH::E >> EP, EPN = 1 << EP;
    constexpr int KB = B + I;
    constexpr int HALF = 1 << I;
    constexpr int NH = EPN / (2 * HALF);
#pragma unroll
    for (int k = 0; k < G; k++) {
        const int g = c.t + SH::T * k;
        const int gl = g & ((1 << B) - 1);
#pragma unroll
        for (int jl = 0; jl < HALF; jl++) {
            if (B == 0 && jl == 0) {
                const uint64_t bnd = (uint64_t)FirstBound<I>::value * c.q;
#pragma unroll
                for (int jh = 0; jh < NH; jh++) {
                    const int j = jh * 2 * HALF;
                    ct_bfly_one(x[k * EPN + j], x[k * EPN + j + HALF], bnd);
                }
            } else {
                ulonglong2 w;
                if constexpr (KB < SH::ILOG) w = c.etw[(1 << KB) + gl + (jl << B)];
                else w = __ldg(c.tw + (1 << KB) + gl + (jl << B));
#pragma unroll
                for (int jh = 0; jh < NH; jh++) {
                    const int j = jh * 2 * HALF + jl;
                    ct_bfly(x[k * EPN + j], x[k * EPN + j + HALF], w.x, w.y, c.q);
                }
            }
        }
    }
}

template <class SH, int B, int EP, int I = 0>
__device__ __forceinline__ void inv_compute(uint64_t (&x)[SH::E], const Ctx &c) {
    if constexpr (I < EP) {
        inv_stage<SH, B, EP, I>(x, c);
        inv_compute<SH, B, EP, I + 1>(x, c);
    }
}

// x <- x * n^-1 psi^-p mod q, fully reduced (x < 2^57 on entry)
__device__ __forceinline__ uint64_t twist(uint64_t x, ulonglong2 t, uint64_t q) {
    return reduce4(shoup_lazy(x, t.x, t.y, q), q);
}

// BLK: a split shape's block kernel -- the local passes only; the block is
// stored back in place unreduced for the column kernel (k_ntt_inv_cols).
template <class SH, int PI, bool BLK = false>
__device__ __forceinline__ void inv_passes(uint64_t (&x)[SH::E], uint64_t *sm, uint64_t *blk, const ulonglong2 *tws,
                                           const Ctx &c) {
    constexpr int LOGE = SH::LOGE;
    constexpr int B = PI * LOGE;
    constexpr int EP = PI == SH::P - 1 ? SH::EREM : LOGE;
    inv_compute<SH, B, EP>(x, c);
    if constexpr (PI + 1 < SH::P) {
        smem_store<SH, B, EP>(x, sm, c.t);
        __syncthreads();
        constexpr int EP2 = PI + 1 == SH::P - 1 ? SH::EREM : LOGE;
        smem_load<SH, B + LOGE, EP2>(x, sm, c.t);
        inv_passes<SH, PI + 1, BLK>(x, sm, blk, tws, c);
    } else if constexpr (BLK) {
        global_store<SH, B, EP>(x, blk, c.t);   // pass B holds bits >= B: coalesced
    } else {
        static_assert(SH::C == 1, "a row of more than one block takes the split kernels");
        constexpr int G = SH::E >> EP, EPN = 1 << EP;
#pragma unroll
        for (int k = 0; k < G; k++) {
            const int g = c.t + SH::T * k;
#pragma unroll
            for (int j = 0; j < EPN; j++) x[k * EPN + j] = twist(x[k * EPN + j], __ldg(tws + pass_pos<B, EP>(g, j)), c.q);
        }
        global_store<SH, B, EP>(x, blk, c.t);
    }
}

// One CTA per row (C = 1): every stage is local, then the twist.
template <int LOGN, int LOGC, int LOGT, int LOGE, int MINB>
__global__ void __launch_bounds__(1 << LOGT, MINB)
k_ntt_inv(uint64_t *__restrict__ res, int L, int batch, const ulonglong2 *__restrict__ tw,
          const uint64_t *__restrict__ consts, const ulonglong2 *__restrict__ twist_tab) {
    pdl_begin();
    using SH = Shape<LOGN, LOGC, LOGT, LOGE>;
    static_assert(SH::C == 1, "a row of more than one block takes the split kernels");
    extern __shared__ __align__(16) uint64_t sm[];
    Ctx c;
    c.t = threadIdx.x;
    c.r = 0;
    int l;
    const long row = row_of<LOGC>(L, batch, l);
    uint64_t *data = res + row * SH::N;
    c.tw = tw + (long)l * SH::N;
    c.kc = consts + (long)l * K_COUNT;
    c.q = c.kc[K_Q];
    ulonglong2 *etw = reinterpret_cast<ulonglong2 *>(sm + SH::M);
    c.etw = etw;
    for (int u = 1 + c.t; u < SH::INV_TW; u += SH::T) cp_async16(etw + u, c.tw + u);
    cp_async_commit();
    uint64_t x[SH::E];
    constexpr int EP0 = SH::P == 1 ? SH::EREM : LOGE;
    if constexpr (SH::E >= 2) {
        block_load_coalesced<SH>(sm, data, c.t);
        cp_async_wait_all();
        __syncthreads();   // the block and the staged twiddles are visible to every thread
        smem_load<SH, 0, EP0>(x, sm, c.t);
    } else {
        global_load<SH, 0, EP0>(x, data, c.t);
        cp_async_wait_all();
        __syncthreads();
    }
    inv_passes<SH, 0>(x, sm, data, twist_tab + (long)l * SH::N, c);
}

// ------------------------------------------------------- split inverse --
//
// The local stages of a split shape: CTA r of a row runs spans 1 .. M/2 on
// block r alone (the same passes and staged twiddles as the one-CTA kernel)
// and stores the block in place, unreduced.
template <int LOGN, int LOGC, int LOGT, int LOGE, int MINB>
__global__ void __launch_bounds__(1 << LOGT, MINB)
k_ntt_inv_blk(uint64_t *res, const uint64_t *src, long src_item, int L, int batch, const ulonglong2 *__restrict__ tw,
              const uint64_t *__restrict__ consts) {
    pdl_begin();
    // reads row (b, l) at src + b src_item + l N (src = res, src_item = L N:
    // in place) and writes it to res + (b L + l) N
    using SH = Shape<LOGN, LOGC, LOGT, LOGE>;
    static_assert(SH::E >= 2, "the block is loaded through shared memory");
    extern __shared__ __align__(16) uint64_t sm[];
    Ctx c;
    c.t = threadIdx.x;
    c.r = (int)(blockIdx.x & (SH::C - 1));
    int l;
    const long row = row_of<LOGC>(L, batch, l);
    uint64_t *blk = res + row * SH::N + (long)c.r * SH::M;
    const uint64_t *sblk = src + (row / L) * src_item + (long)l * SH::N + (long)c.r * SH::M;
    c.tw = tw + (long)l * SH::N;
    c.kc = consts + (long)l * K_COUNT;
    c.q = c.kc[K_Q];
    ulonglong2 *etw = reinterpret_cast<ulonglong2 *>(sm + SH::M);
    c.etw = etw;
    for (int u = 1 + c.t; u < SH::INV_TW; u += SH::T) cp_async16(etw + u, c.tw + u);
    cp_async_commit();
    uint64_t x[SH::E];
    block_load_coalesced<SH>(sm, sblk, c.t);
    cp_async_wait_all();
    __syncthreads();   // the block and the staged twiddles are visible to every thread
    smem_load<SH, 0, SH::P == 1 ? SH::EREM : LOGE>(x, sm, c.t);
    inv_passes<SH, 0, true>(x, sm, blk, nullptr, c);
}

// The cross stages of a split inverse and the twist, over whole columns.
// CTA (l, chunk, part) owns COLS adjacent columns j2 of prime l and runs them
// for up to `chunk` consecutive batch items.  The TPC = 2^LOGTPC threads of
// column j2 hold its C residues j1 M + j2, first as j1 = VPT g + i for the
// spans below VPT, then -- after one shared-memory exchange -- as
// j1 = g + TPC i for the spans >= VPT.  The span-M 2^S stage pairs j1 and
// j1 + 2^S and multiplies by inv[M (2^S + (j1 mod 2^S)) + j2]: those C - 1
// twiddles of each column depend on the column, not on the batch item, so the
// CTA copies them into shared memory once (cp.async, overlapping the first
// item's loads) and every item reads them there.  Last, every residue is
// multiplied by n^-1 psi^-p (p = j1 M + j2, loaded with the item's residues),
// reduced into [0, q) and stored.
template <int LOGN, int LOGC, int LOGTPC>
__global__ void __launch_bounds__(256)
k_ntt_inv_cols(uint64_t *__restrict__ res, int L, int batch, int chunk, const ulonglong2 *__restrict__ tw,
               const uint64_t *__restrict__ consts, const ulonglong2 *__restrict__ twist_tab) {
    pdl_begin();
    constexpr int C = 1 << LOGC, M = 1 << (LOGN - LOGC);
    constexpr int TPC = 1 << LOGTPC, LOGVPT = LOGC - LOGTPC, VPT = 1 << LOGVPT;
    constexpr int COLS = 256 / TPC, CPR = M / COLS;   // columns per CTA, CTAs per row
    static_assert(LOGTPC <= LOGVPT, "the spans >= VPT are whole multiples of TPC");
    static_assert(M % COLS == 0, "whole CTAs per row");
    __shared__ __align__(16) ulonglong2 stw[C - 1][COLS];   // twiddle 2^S + jlo of column cl at [2^S + jlo - 1][cl]
    __shared__ uint64_t tile[C][COLS];
    // limb-major (as row_of): the CTAs running together share a prime
    const unsigned bid = gridDim.x - 1 - blockIdx.x;   // last rows first (still in L2)
    const int part = (int)(bid % CPR);
    const int nch = (batch + chunk - 1) / chunk;
    const int rest = (int)(bid / CPR);
    const int l = rest / nch, b0 = (rest - l * nch) * chunk;
    const int b1 = min(batch, b0 + chunk);
    const int cl = threadIdx.x % COLS, g = threadIdx.x / COLS;
    const int j2 = part * COLS + cl;
    const ulonglong2 *wl = tw + ((long)l << LOGN) + part * COLS;
    for (int u = threadIdx.x; u < (C - 1) * COLS; u += 256)
        cp_async16(&stw[u / COLS][u % COLS], wl + (long)(u / COLS + 1) * M + u % COLS);
    cp_async_commit();
    const uint64_t q = __ldg(consts + (long)l * K_COUNT + K_Q);
    const ulonglong2 *tt = twist_tab + ((long)l << LOGN) + j2;
    for (int b = b0; b < b1; b++) {
        uint64_t *p = res + ((long)b * L + l) * ((long)1 << LOGN) + j2;
        uint64_t x[VPT];
        ulonglong2 tv[VPT];
#pragma unroll
        for (int i = 0; i < VPT; i++) x[i] = __ldcg(p + (long)(VPT * g + i) * M);
#pragma unroll
        for (int i = 0; i < VPT; i++) tv[i] = __ldg(tt + (long)(LOGTPC > 0 ? g + TPC * i : VPT * g + i) * M);
        cp_async_wait_all();
        __syncthreads();   // the staged twiddles are visible; the previous item's tile reads are done
#pragma unroll
        for (int S = 0; S < LOGVPT; S++) {
            const int H = 1 << S;   // j1 = VPT g + i, VPT g a multiple of 2^(S+1)
#pragma unroll
            for (int i = 0; i < VPT; i++) {
                if (i & H) continue;
                const ulonglong2 wt = stw[(1 << S) + (i & (H - 1)) - 1][cl];
                ct_bfly(x[i], x[i + H], wt.x, wt.y, q);
            }
        }
        if constexpr (LOGTPC > 0) {
#pragma unroll
            for (int i = 0; i < VPT; i++) tile[VPT * g + i][cl] = x[i];
            __syncthreads();
#pragma unroll
            for (int i = 0; i < VPT; i++) x[i] = tile[g + TPC * i][cl];
#pragma unroll
            for (int S = LOGVPT; S < LOGC; S++) {
                const int HI = 1 << (S - LOGTPC);   // span 2^S = TPC HI in j1 = g + TPC i
#pragma unroll
                for (int i = 0; i < VPT; i++) {
                    if (i & HI) continue;
                    const int j1 = g + TPC * i;
                    const ulonglong2 wt = stw[(1 << S) + (j1 & ((1 << S) - 1)) - 1][cl];
                    ct_bfly(x[i], x[i + HI], wt.x, wt.y, q);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < VPT; i++)
            __stcg(p + (long)(LOGTPC > 0 ? g + TPC * i : VPT * g + i) * M, twist(x[i], tv[i], q));
    }
}

// ---------------------------------------------------------------- launch --

// One CTA per row (C = 1).
template <int LOGN, int LOGC, int LOGT, int LOGE, int MINB, bool INVERSE>
int launch_shape(uint64_t *res, int L, long rows, const fhe_ntt_tables *t, cudaStream_t st) {
    using SH = Shape<LOGN, LOGC, LOGT, LOGE>;
    static_assert(SH::C == 1, "a row of more than one block takes the split kernels");
    if (rows % L) return -1;
    const int batch = (int)(rows / L);
    const size_t smem = (size_t)SH::smem_words(INVERSE) * sizeof(uint64_t);
    if constexpr (INVERSE) {
        auto kern = k_ntt_inv<LOGN, LOGC, LOGT, LOGE, MINB>;
        if (smem > 48 * 1024 &&
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return -1;
        launch_pdl(kern, (unsigned)rows, SH::T, smem, st, res, L, batch, reinterpret_cast<const ulonglong2 *>(t->inv),
                                                  t->consts, reinterpret_cast<const ulonglong2 *>(t->twist));
    } else {
        auto kern = k_ntt_fwd<LOGN, LOGC, LOGT, LOGE, MINB>;
        if (smem > 48 * 1024 &&
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return -1;
        launch_pdl(kern, (unsigned)rows, SH::T, smem, st, res, L, batch, reinterpret_cast<const ulonglong2 *>(t->fwd),
                                                  t->consts);
    }
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

// Split forward: the column kernel (first LOGC stages), then one CTA per block.
template <int LOGN, int LOGC, int LOGT, int LOGE, int MINB>
int launch_split_fwd(uint64_t *res, int L, long rows, const fhe_ntt_tables *t, cudaStream_t st) {
    using SH = Shape<LOGN, LOGC, LOGT, LOGE>;
    constexpr int LOGTPC = LOGC / 2;                  // threads per column
    constexpr int CPR = SH::M / (256 >> LOGTPC);      // column-kernel CTAs per row
    if (rows % L) return -1;
    const int batch = (int)(rows / L);
    const ulonglong2 *tw = reinterpret_cast<const ulonglong2 *>(t->fwd);
    // batch items per column CTA: up to 4, balanced (each CTA loads item
    // b + 1 while it transforms item b)
    const int nch = (batch + 3) / 4, chunk = (batch + nch - 1) / nch;
    const int nchunks = (batch + chunk - 1) / chunk;
    launch_pdl(k_ntt_fwd_cols<LOGN, LOGC, LOGTPC>, (unsigned)((long)L * nchunks * CPR), 256, 0, st, res, L, batch,
               chunk, tw, t->consts);
    if (cudaGetLastError() != cudaSuccess) return -1;
    auto kern = k_ntt_fwd_blk<LOGN, LOGC, LOGT, LOGE, MINB>;
    const size_t smem = (size_t)SH::smem_words(false) * sizeof(uint64_t);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return -1;
    launch_pdl(kern, (unsigned)(rows * SH::C), SH::T, smem, st, res, L, batch, tw, t->consts);
    if (cudaGetLastError() != cudaSuccess) return -1;
    return 2;
}

template <int LOGN, int LOGC, int LOGT, int LOGE, int MINB, int SPLIT>
int launch_fwd(uint64_t *res, int L, long rows, const fhe_ntt_tables *t, cudaStream_t st) {
    if constexpr (SPLIT) return launch_split_fwd<LOGN, LOGC, LOGT, LOGE, MINB>(res, L, rows, t, st);
    else return launch_shape<LOGN, LOGC, LOGT, LOGE, MINB, false>(res, L, rows, t, st);
}

// Split inverse: one CTA per block (the local stages), then the column kernel.
template <int LOGN, int LOGC, int LOGT, int LOGE, int MINB>
int launch_split_inv(uint64_t *res, int L, long rows, const fhe_ntt_tables *t, cudaStream_t st,
                     const uint64_t *src = nullptr, long src_item = 0) {
    using SH = Shape<LOGN, LOGC, LOGT, LOGE>;
    constexpr int LOGTPC = LOGC / 2;                  // threads per column
    constexpr int CPR = SH::M / (256 >> LOGTPC);      // column-kernel CTAs per row
    if (rows % L) return -1;
    const int batch = (int)(rows / L);
    const ulonglong2 *tw = reinterpret_cast<const ulonglong2 *>(t->inv);
    auto kern = k_ntt_inv_blk<LOGN, LOGC, LOGT, LOGE, MINB>;
    const size_t smem = (size_t)SH::smem_words(true) * sizeof(uint64_t);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return -1;
    if (!src) {
        src = res;
        src_item = (long)L << LOGN;
    }
    launch_pdl(kern, (unsigned)(rows * SH::C), SH::T, smem, st, res, src, src_item, L, batch, tw, t->consts);
    if (cudaGetLastError() != cudaSuccess) return -1;
    // batch items per column CTA: up to 4, balanced, so the staged twiddles
    // serve several items and the grid still spans several waves
    const int nch = (batch + 3) / 4, chunk = (batch + nch - 1) / nch;
    const int nchunks = (batch + chunk - 1) / chunk;
    launch_pdl(k_ntt_inv_cols<LOGN, LOGC, LOGTPC>, (unsigned)((long)L * nchunks * CPR), 256, 0, st, res, L, batch,
               chunk, tw, t->consts, reinterpret_cast<const ulonglong2 *>(t->twist));
    if (cudaGetLastError() != cudaSuccess) return -1;
    return 2;
}

template <int LOGN, int LOGC, int LOGT, int LOGE, int MINB, int SPLIT>
int launch_inv(uint64_t *res, int L, long rows, const fhe_ntt_tables *t, cudaStream_t st) {
    if constexpr (SPLIT) return launch_split_inv<LOGN, LOGC, LOGT, LOGE, MINB>(res, L, rows, t, st);
    else return launch_shape<LOGN, LOGC, LOGT, LOGE, MINB, true>(res, L, rows, t, st);
}

// Forward NTT of the extended digits fused with the inner product (split
// shapes): the column kernel on every row of ext, then k_ntt_fwd_blk_ip.
template <int LOGN, int LOGC, int LOGT, int LOGE, int MINB, int SPLIT, int DN>
int launch_fwd_ip_dn(uint64_t *out, uint64_t *ext, const uint64_t *keys, int LK, int batch, const fhe_ntt_tables *t,
                     cudaStream_t st) {
    if constexpr (!SPLIT) {
        return 0;
    } else {
        using SH = Shape<LOGN, LOGC, LOGT, LOGE>;
        constexpr int LOGTPC = LOGC / 2;
        constexpr int CPR = SH::M / (256 >> LOGTPC);
        const ulonglong2 *tw = reinterpret_cast<const ulonglong2 *>(t->fwd);
        const int items = batch * DN;   // rows of one prime in ext: [batch][DN][LK][n]
        const int nch = (items + 3) / 4, chunk = (items + nch - 1) / nch;
        const int nchunks = (items + chunk - 1) / chunk;
        launch_pdl(k_ntt_fwd_cols<LOGN, LOGC, LOGTPC>, (unsigned)((long)LK * nchunks * CPR), 256, 0, st, ext, LK,
                   items, chunk, tw, t->consts);
        if (cudaGetLastError() != cudaSuccess) return -1;
        auto kern = k_ntt_fwd_blk_ip<LOGN, LOGC, LOGT, LOGE, MINB, DN>;
        const size_t smem = (size_t)(DN * SH::M + 2 * SH::FWD_TW) * sizeof(uint64_t);
        if (smem > 48 * 1024 &&
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return -1;
        launch_pdl(kern, (unsigned)((long)LK * SH::C * batch), SH::T, smem, st, out, ext, keys, LK, batch, tw,
                   t->consts);
        if (cudaGetLastError() != cudaSuccess) return -1;
        return 2;
    }
}

// ModDown's forward NTT of d fused with its last step (split shapes): the
// column kernel on every row of d, then k_ntt_fwd_blk_md.
template <int LOGN, int LOGC, int LOGT, int LOGE, int MINB, int SPLIT>
int launch_fwd_md(uint64_t *out, uint64_t *d, const uint64_t *in, int L, int K, int batch, const fhe_ntt_tables *t,
                  const ulonglong2 *pinv, cudaStream_t st) {
    if constexpr (!SPLIT) {
        return 0;
    } else {
        using SH = Shape<LOGN, LOGC, LOGT, LOGE>;
        constexpr int LOGTPC = LOGC / 2;
        constexpr int CPR = SH::M / (256 >> LOGTPC);
        const ulonglong2 *tw = reinterpret_cast<const ulonglong2 *>(t->fwd);
        const int nch = (batch + 3) / 4, chunk = (batch + nch - 1) / nch;
        const int nchunks = (batch + chunk - 1) / chunk;
        launch_pdl(k_ntt_fwd_cols<LOGN, LOGC, LOGTPC>, (unsigned)((long)L * nchunks * CPR), 256, 0, st, d, L, batch,
                   chunk, tw, t->consts);
        if (cudaGetLastError() != cudaSuccess) return -1;
        auto kern = k_ntt_fwd_blk_md<LOGN, LOGC, LOGT, LOGE, MINB>;
        const size_t smem = (size_t)(SH::smem_words(false) + SH::M) * sizeof(uint64_t);
        if (smem > 48 * 1024 &&
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return -1;
        launch_pdl(kern, (unsigned)((long)batch * L * SH::C), SH::T, smem, st, out, d, in, L, K, batch, tw, t->consts,
                   pinv);
        if (cudaGetLastError() != cudaSuccess) return -1;
        return 2;
    }
}

template <int LOGN, int LOGC, int LOGT, int LOGE, int MINB, int SPLIT>
int launch_fwd_ip(uint64_t *out, uint64_t *ext, const uint64_t *keys, int LK, int dnum, int batch,
                  const fhe_ntt_tables *t, cudaStream_t st) {
    switch (dnum) {
        case 1: return launch_fwd_ip_dn<LOGN, LOGC, LOGT, LOGE, MINB, SPLIT, 1>(out, ext, keys, LK, batch, t, st);
        case 2: return launch_fwd_ip_dn<LOGN, LOGC, LOGT, LOGE, MINB, SPLIT, 2>(out, ext, keys, LK, batch, t, st);
        case 3: return launch_fwd_ip_dn<LOGN, LOGC, LOGT, LOGE, MINB, SPLIT, 3>(out, ext, keys, LK, batch, t, st);
        case 4: return launch_fwd_ip_dn<LOGN, LOGC, LOGT, LOGE, MINB, SPLIT, 4>(out, ext, keys, LK, batch, t, st);
        default: return 0;
    }
}

// A split inverse reading its rows from another buffer (row (b, l) at
// src + b src_item + l n) and leaving the result in dst [batch][L][n].
template <int LOGN, int LOGC, int LOGT, int LOGE, int MINB, int SPLIT>
int launch_inv_from(uint64_t *dst, const uint64_t *src, long src_item, int L, int batch, const fhe_ntt_tables *t,
                    cudaStream_t st) {
    if constexpr (!SPLIT) return 0;
    else return launch_split_inv<LOGN, LOGC, LOGT, LOGE, MINB>(dst, L, (long)batch * L, t, st, src, src_item);
}

}  // namespace

int launch_ntt_fwd_ip(uint64_t *out, uint64_t *ext, const uint64_t *keys, int log_n, int LK, int dnum, int batch,
                      const fhe_ntt_tables *t, void *stream) {
    cudaStream_t st = (cudaStream_t)stream;
    if ((long)LK * batch * (1L << (log_n - 10)) >= (1L << 31)) return 0;
    switch (log_n) {
        case 14: return launch_fwd_ip<14, FHE_SHAPE_14>(out, ext, keys, LK, dnum, batch, t, st);
        case 15: return launch_fwd_ip<15, FHE_SHAPE_15>(out, ext, keys, LK, dnum, batch, t, st);
        case 16: return launch_fwd_ip<16, FHE_SHAPE_16>(out, ext, keys, LK, dnum, batch, t, st);
        case 17: return launch_fwd_ip<17, FHE_SHAPE_17>(out, ext, keys, LK, dnum, batch, t, st);
        default: return 0;
    }
}

int launch_ntt_inv_from(uint64_t *dst, const uint64_t *src, long src_item, int log_n, int L, int batch,
                        const fhe_ntt_tables *t, void *stream) {
    cudaStream_t st = (cudaStream_t)stream;
    switch (log_n) {
        case 14: return launch_inv_from<14, FHE_INV_SHAPE_14>(dst, src, src_item, L, batch, t, st);
        case 15: return launch_inv_from<15, FHE_INV_SHAPE_15>(dst, src, src_item, L, batch, t, st);
        case 16: return launch_inv_from<16, FHE_INV_SHAPE_16>(dst, src, src_item, L, batch, t, st);
        case 17: return launch_inv_from<17, FHE_INV_SHAPE_17>(dst, src, src_item, L, batch, t, st);
        default: return 0;
    }
}

int launch_ntt_fwd_moddown(uint64_t *out, uint64_t *d, const uint64_t *in, int log_n, int L, int K, int batch,
                           const fhe_ntt_tables *t_q, const void *pinv, void *stream) {
    cudaStream_t st = (cudaStream_t)stream;
    const ulonglong2 *pi = (const ulonglong2 *)pinv;
    switch (log_n) {
        case 14: return launch_fwd_md<14, FHE_SHAPE_14>(out, d, in, L, K, batch, t_q, pi, st);
        case 15: return launch_fwd_md<15, FHE_SHAPE_15>(out, d, in, L, K, batch, t_q, pi, st);
        case 16: return launch_fwd_md<16, FHE_SHAPE_16>(out, d, in, L, K, batch, t_q, pi, st);
        case 17: return launch_fwd_md<17, FHE_SHAPE_17>(out, d, in, L, K, batch, t_q, pi, st);
        default: return 0;
    }
}

int launch_ntt(uint64_t *res, int log_n, int L, long rows, const fhe_ntt_tables *t, bool inverse, void *stream) {
    cudaStream_t st = (cudaStream_t)stream;
    switch (log_n) {
        case 1: return inverse ? launch_inv<1, FHE_INV_SHAPE_1>(res, L, rows, t, st)
                          : launch_fwd<1, FHE_SHAPE_1>(res, L, rows, t, st);
        case 2: return inverse ? launch_inv<2, FHE_INV_SHAPE_2>(res, L, rows, t, st)
                          : launch_fwd<2, FHE_SHAPE_2>(res, L, rows, t, st);
        case 3: return inverse ? launch_inv<3, FHE_INV_SHAPE_3>(res, L, rows, t, st)
                          : launch_fwd<3, FHE_SHAPE_3>(res, L, rows, t, st);
        case 4: return inverse ? launch_inv<4, FHE_INV_SHAPE_4>(res, L, rows, t, st)
                          : launch_fwd<4, FHE_SHAPE_4>(res, L, rows, t, st);
        case 5: return inverse ? launch_inv<5, FHE_INV_SHAPE_5>(res, L, rows, t, st)
                          : launch_fwd<5, FHE_SHAPE_5>(res, L, rows, t, st);
        case 6: return inverse ? launch_inv<6, FHE_INV_SHAPE_6>(res, L, rows, t, st)
                          : launch_fwd<6, FHE_SHAPE_6>(res, L, rows, t, st);
        case 7: return inverse ? launch_inv<7, FHE_INV_SHAPE_7>(res, L, rows, t, st)
                          : launch_fwd<7, FHE_SHAPE_7>(res, L, rows, t, st);
        case 8: return inverse ? launch_inv<8, FHE_INV_SHAPE_8>(res, L, rows, t, st)
                          : launch_fwd<8, FHE_SHAPE_8>(res, L, rows, t, st);
        case 9: return inverse ? launch_inv<9, FHE_INV_SHAPE_9>(res, L, rows, t, st)
                          : launch_fwd<9, FHE_SHAPE_9>(res, L, rows, t, st);
        case 10: return inverse ? launch_inv<10, FHE_INV_SHAPE_10>(res, L, rows, t, st)
                          : launch_fwd<10, FHE_SHAPE_10>(res, L, rows, t, st);
        case 11: return inverse ? launch_inv<11, FHE_INV_SHAPE_11>(res, L, rows, t, st)
                          : launch_fwd<11, FHE_SHAPE_11>(res, L, rows, t, st);
        case 12: return inverse ? launch_inv<12, FHE_INV_SHAPE_12>(res, L, rows, t, st)
                          : launch_fwd<12, FHE_SHAPE_12>(res, L, rows, t, st);
        case 13: return inverse ? launch_inv<13, FHE_INV_SHAPE_13>(res, L, rows, t, st)
                          : launch_fwd<13, FHE_SHAPE_13>(res, L, rows, t, st);
        case 14: return inverse ? launch_inv<14, FHE_INV_SHAPE_14>(res, L, rows, t, st)
                          : launch_fwd<14, FHE_SHAPE_14>(res, L, rows, t, st);
        case 15: return inverse ? launch_inv<15, FHE_INV_SHAPE_15>(res, L, rows, t, st)
                          : launch_fwd<15, FHE_SHAPE_15>(res, L, rows, t, st);
        case 16: return inverse ? launch_inv<16, FHE_INV_SHAPE_16>(res, L, rows, t, st)
                          : launch_fwd<16, FHE_SHAPE_16>(res, L, rows, t, st);
        case 17: return inverse ? launch_inv<17, FHE_INV_SHAPE_17>(res, L, rows, t, st)
                          : launch_fwd<17, FHE_SHAPE_17>(res, L, rows, t, st);
        default: return -1;
    }
}

}  // namespace fhe
