/*
 * fhe_ntt.h -- C ABI of libfhe_ntt.so: batched RNS negacyclic NTT and the
 * NTT-domain kernels of RNS-CKKS on one NVIDIA GB300 (sm_103a).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layout.  A residue tensor is row-major uint64_t[batch][L][n]: row (b, l)
 *   holds the n residues of polynomial b modulo the l-th prime (FHElium,
 *   "Eager, Compile, and native execution", section "Shared implementation
 *   and native path": an RNS tensor is [*batch, limb, coefficient] and
 *   parameter column j describes limb j).  n = 2^log_n, 1 <= log_n <= 17.
 * Values.  Inputs must be fully reduced (0 <= x < q_l); outputs always are
 *   ("For standard RNS addition, CPU and CUDA produce residues in [0, q_i)",
 *   same page, section "One operation through both use models").  Inputs
 *   outside [0, q) are not checked and give unspecified outputs.
 * Moduli.  Every prime satisfies 2^48 < q < 2^50 and q = 1 (mod 2n); the
 *   table builders reject anything else with FHE_EINVAL.
 * Memory.  Every residue, table and workspace pointer is a device pointer
 *   owned by the caller (PyTorch in the Python binding): the library never
 *   allocates, frees or copies device memory.  All device pointers of one
 *   call must live on one CUDA device; the call makes that device current
 *   (as FHElium's CUDA adapters do) and fails with FHE_EDEVICE otherwise.
 *   Host pointers where a device pointer is required fail with FHE_EDEVICE
 *   before any launch, so no kernel ever receives a host address.  Residue,
 *   table and workspace pointers must be 16-byte aligned (FHE_EINVAL).
 * Streams.  `stream` is a cudaStream_t (NULL = legacy default stream).
 *   Kernels are enqueued on it and the call returns without synchronising
 *   ("Kernels launch on the current stream ... and do not introduce an
 *   implicit host synchronization", same page, section "CUDA execution").
 *   A fault inside a kernel surfaces at the caller's next synchronisation.
 * Validation.  Arguments (sizes, pointer kinds, table shape, aliasing) are
 *   checked on the host before launch ("C++ validation checks shape, dtype,
 *   device agreement, parameter-row counts, broadcasting rules, and
 *   prohibited overlap before ... launching a CUDA kernel", same page,
 *   section "Schema registration and device dispatch").  Nothing aborts or
 *   throws; every entry point returns a status code.
 * Limb subsets.  A call with L smaller than the tables' L uses limbs [0, L).
 */
#ifndef FHE_NTT_H
#define FHE_NTT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define FHE_OK 0
#define FHE_EINVAL (-1)    /* bad size, modulus, k, null pointer or table shape */
#define FHE_EALIAS (-2)    /* prohibited overlap between an output and another buffer */
#define FHE_ECUDA (-3)     /* a CUDA runtime call or a kernel launch failed */
#define FHE_ESPACE (-4)    /* workspace or host buffer too small */
#define FHE_EDEVICE (-5)   /* host pointer where a device pointer is required, or mixed devices */

/* Bits of the device status word (fhe_device_status). */
#define FHE_STATUS_TC_TIMEOUT 1   /* a tensor-core kernel gave up waiting for its MMA: its outputs are invalid */

/* Library version: major * 10000 + minor * 100 + patch. */
int fhe_version(void);

/* Static message for a status code (never NULL). */
const char *fhe_status_str(int status);

/* Number of kernels this library has enqueued in this process (all devices,
 * all streams) -- a diagnostic for counting launches around a timed region. */
uint64_t fhe_launch_count(void);

/* Diagnostic: checks the library's modular arithmetic routines (the lazy
 * Shoup product, Barrett reductions, 128-bit accumulation) compiled for the
 * host against exact 128-bit arithmetic on `iters` pseudo-random operands
 * per prime (seeded by `seed`).  Needs no GPU.  FHE_OK when all agree. */
int fhe_selftest_host(uint64_t seed, int iters);


/* ---- primes and roots -------------------------------------------------- */

/* The `count` largest primes q < below (below = 0 means 2^bits) with
 * q = 1 (mod 2^(log_n+1)), in descending order, written to host out[count].
 * Primality: deterministic Miller-Rabin for 64-bit inputs.  This reading of
 * "the largest q < 2^50 with q = 1 mod 2n" is the one used for every
 * workload; the special primes of a key switch are the next ones after the
 * chain's primes (pass below = the last chain prime).
 * Returns FHE_EINVAL if the range holds fewer than `count` primes. */
int fhe_find_primes(int log_n, int bits, int count, uint64_t below, uint64_t *out);

/* psi = the smallest primitive 2n-th root of unity modulo prime q
 * (q = 1 mod 2n), written to *psi (host).  The transform below evaluates at
 * the odd powers of this psi.  The pages fix no root; the smallest one is
 * canonical and independent of any generator choice. */
int fhe_root_of_unity(uint64_t q, int log_n, uint64_t *psi);

/* ---- NTT tables -------------------------------------------------------- */

/* Device view of a table blob: pointers into one caller-owned device buffer.
 * FHElium passes "schedule and twiddle Tensors" to every NTT call (same page,
 * section "Shared implementation and native path"); this struct is that
 * argument.  Filled by fhe_ntt_tables_bind; treat the fields as opaque.
 * Every entry point checks, before any launch, that the struct is exactly
 * what fhe_ntt_tables_bind writes for `blob` (each array pointer at its
 * offset inside the blob, `bytes` the layout size); any other struct gives
 * FHE_EINVAL.  `blob` itself then goes through the device and overlap
 * checks, so no kernel reads tables outside the caller's device blob. */
typedef struct fhe_ntt_tables {
    int32_t log_n;            /* tables are for n = 2^log_n */
    int32_t L;                /* number of primes covered */
    const uint64_t *q;        /* [L] moduli */
    const uint64_t *consts;   /* [L][16] per-prime constants */
    const uint64_t *fwd;      /* [L][n][2] forward twiddles and Shoup companions, the value
                                 psi^brv(k) at slot fhe_ntt_fwd_table_slot(log_n, k) */
    const uint64_t *inv;      /* [L][n][2] inverse (cyclic) twiddles and companions */
    const uint64_t *twist;    /* [L][n][2] n^-1 psi^-j and companions */
    const void *blob;         /* base of the device blob */
    size_t bytes;             /* blob size */
} fhe_ntt_tables;

/* Size in bytes of the table blob for (log_n, L). */
int fhe_ntt_tables_bytes(int log_n, int L, size_t *bytes);

/* Build the blob for primes q[L] (host array) into host memory host_blob of
 * `bytes` bytes (FHE_ESPACE if smaller than fhe_ntt_tables_bytes).  Copy
 * the blob unchanged to device memory (any 16-byte aligned address), then
 * call fhe_ntt_tables_bind. */
int fhe_ntt_tables_build_host(int log_n, int L, const uint64_t *q, void *host_blob, size_t bytes);

/* Fill *out with device pointers into dev_blob (no copy, no launch). */
int fhe_ntt_tables_bind(const void *dev_blob, size_t bytes, int log_n, int L, fhe_ntt_tables *out);

/* Where the forward twiddle of index k (value psi^brv(k), 0 <= k < n) is
 * stored in a prime's fwd table: the stages of the transform's last register
 * pass keep their twiddles in the order that pass reads them (consecutive
 * threads, consecutive entries); every other entry is at slot k.  For tools
 * that read or write table blobs. */
int fhe_ntt_fwd_table_slot(int log_n, uint32_t k, uint32_t *slot);

/* ---- transforms -------------------------------------------------------- */

/* In-place forward negacyclic NTT of every row of res[batch][L][n]:
 *   res[b][l][i] <- sum_j res[b][l][j] * psi_l^((2 brv(i) + 1) j)  mod q_l,
 * i.e. the values of the row's polynomial at the n roots of X^n + 1, stored
 * in bit-reversed order (brv over log_n bits).  The NTT is the transform
 * under every CKKS multiplication, relinearisation and rotation in the
 * kestrel-llm chain (lpnh.cn news 2512365, section 3, vllm_ntt.c) and
 * FHElium's "power-of-two-radix NTT" family ("Eager, Compile, and native
 * execution", table "Native operator families").  Launches on `stream`, no
 * host sync: one kernel for n <= 2^13, two for n >= 2^14 (a kernel over
 * strided columns for the first stages, then one over contiguous blocks). */
int fhe_ntt_fwd(uint64_t *res, int log_n, int L, int batch, const fhe_ntt_tables *t, void *stream);

/* In-place exact inverse of fhe_ntt_fwd, including the 1/n factor:
 * bit-reversed evaluations in, natural-order coefficients out.  Launches as
 * fhe_ntt_fwd does, in the mirror order for n >= 2^14 (blocks, then
 * columns). */
int fhe_ntt_inv(uint64_t *res, int log_n, int L, int batch, const fhe_ntt_tables *t, void *stream);

/* Measurement aid with no counterpart on the pages: the throughput ceiling of
 * the NTT butterfly on this GPU.  Each of the `ctas` CTAs of 256 threads keeps
 * 32 residues per thread in registers and runs `iters` rounds of five radix-2
 * stages (80 lazy Cooley-Tukey butterflies per thread per round, the
 * arithmetic of fhe_ntt_fwd) with twiddles read coalesced from prime 0 of
 * `t`, then writes one word per thread to out[ctas * 256] (device memory,
 * caller-owned, 16-byte aligned): the XOR of its 32 residues reduced into
 * [0, q_0), a checksum of the butterfly network (residue i of global thread g
 * starts at (977 g + 131 i) mod q_0; round r uses, for stage s and twiddle j,
 * entry 32 (32 (r mod 2) + 2^s + j) + (g mod 32) of prime 0's forward table).
 * Butterflies per call: ctas * 256 * iters * 80.  Needs t->log_n >= 11;
 * 1 <= ctas <= 1048576, 1 <= iters <= 128 (the lazy bound of the residues),
 * else FHE_EINVAL.  One launch on `stream`, no host sync. */
int fhe_butterfly_probe(uint64_t *out, int ctas, int iters, const fhe_ntt_tables *t, void *stream);

/* Device status word.  Kernels that wait on the tensor cores (the ModUp of
 * fhe_keyswitch_ip and the other key-switch calls, for digits of at most 8
 * primes) bound every wait (200 ms); one that gives up sets a
 * FHE_STATUS_* bit here, releases its tensor memory and returns, leaving the
 * context usable.  Waits for all work on the current device
 * (cudaDeviceSynchronize), then writes the word to *status and, if reset is
 * nonzero, clears it.  FHE_EINVAL for a null status, FHE_ECUDA if the
 * synchronization or the copy fails.
 * For tests of that path: with FHE_TC_TEST_TIMEOUT=1 in the environment at
 * launch time, the tensor-core kernels wait 1 ms on a barrier nothing
 * arrives on and give up as above (their outputs are then invalid). */
int fhe_device_status(int *status, int reset);

/* ---- NTT-domain kernels ------------------------------------------------ */

/* out = a * b mod q_l elementwise over [batch][L][n] (the pointwise product
 * that turns into the negacyclic product after fhe_ntt_inv; kestrel-llm
 * section 3 "polynomial multiplication").  out may equal a or b exactly;
 * any other overlap is FHE_EALIAS. */
int fhe_mul_ntt(uint64_t *out, const uint64_t *a, const uint64_t *b, int log_n, int L, int batch,
                const fhe_ntt_tables *t, void *stream);

/* Ciphertext tensor product in the NTT domain (the CKKS multiply before
 * relinearisation; kestrel-llm section 3, vllm_ckks.c):
 *   a, b: [batch][2][L][n] (components 0 and 1),  d: [batch][3][L][n]
 *   d0 = a0 b0,  d1 = a0 b1 + a1 b0,  d2 = a1 b1   (mod q_l).
 * d must not overlap a or b (FHE_EALIAS). */
int fhe_tensor(uint64_t *d, const uint64_t *a, const uint64_t *b, int log_n, int L, int batch,
               const fhe_ntt_tables *t, void *stream);

#define FHE_DOMAIN_COEFF 0
#define FHE_DOMAIN_NTT 1

/* Galois automorphism sigma_k: a(X) -> a(X^k), k odd, 1 <= k < 2n (the
 * rotations inside coeff_to_slot / slot_to_coeff, kestrel-llm section 4.2;
 * FHElium "Galois automorphisms").  out, in: [batch][L][n].
 *   FHE_DOMAIN_COEFF: coefficient t moves to s = t k mod 2n, negated
 *     (q - a mod q) when s >= n, since X^n = -1.
 *   FHE_DOMAIN_NTT: out[i] = in[j] with 2 brv(j) + 1 = k (2 brv(i) + 1)
 *     mod 2n (a permutation of the evaluation points; no arithmetic).
 * out must not overlap in (FHE_EALIAS). */
int fhe_automorph(uint64_t *out, const uint64_t *in, int log_n, int L, int batch, uint64_t k,
                  int domain, const fhe_ntt_tables *t, void *stream);

/* ---- hybrid key switch ------------------------------------------------- */

/* Basis: qp = (q_0 .. q_{L-1}, p_0 .. p_{K-1}), L + K <= 64.  Digits: with
 * alpha = ceil(L / dnum), digit j covers limbs [j alpha, min((j+1) alpha, L)),
 * 1 <= alpha <= 16, and every digit is non-empty. */

/* Size of the ModUp constant blob (Garner and mixed-radix constants). */
int fhe_modup_tables_bytes(int L, int K, int dnum, size_t *bytes);

/* Build the ModUp blob for basis qp[L+K] (host) into host memory; copy it
 * unchanged to a 16-byte aligned device buffer and pass that pointer as
 * `modup` below. */
int fhe_modup_tables_build_host(int L, int K, int dnum, const uint64_t *qp, void *host_blob,
                                size_t bytes);

/* Workspace bytes fhe_keyswitch_ip needs: batch * dnum * (L+K) * n * 8. */
int fhe_keyswitch_workspace_bytes(int log_n, int L, int K, int dnum, int batch, size_t *bytes);

/* Hybrid key-switch inner product, before ModDown (FHElium "key-switch
 * multiply-accumulate" and "mixed-radix decomposition and basis extension",
 * "Eager, Compile, and native execution", section "CUDA execution";
 * kestrel-llm's Garner extension, section 4.2):
 *   in:   batch items of [L][n], item b at in + b * in_stride (elements;
 *         in_stride = 0 means L * n, i.e. a contiguous [batch][L][n]; it
 *         lets a call read component d2 of a [batch][3][L][n] tensor
 *         product directly), coefficient domain, basis q_0..q_{L-1}
 *   keys: [dnum][2][L+K][n]      NTT domain, basis qp
 *   out:  [batch][2][L+K][n]     NTT domain, basis qp
 * For every digit j: X_j = the exact CRT integer of the digit's residues
 * (0 <= X_j < prod of the digit's primes; mixed-radix / Garner), extended to
 * every prime of qp (limbs inside the digit are copied), transformed with
 * fhe_ntt_fwd over qp, then
 *   out[b][c][l] = sum_j NTT(X_j)[l] * keys[j][c][l]  mod qp_l.
 * t_qp: NTT tables for the L+K primes of qp in that order.
 * workspace: device buffer of at least fhe_keyswitch_workspace_bytes; its
 * contents on entry are ignored and on return are unspecified.  out, in,
 * keys and workspace must be pairwise disjoint (FHE_EALIAS); in_stride, if
 * nonzero, must be >= L * n and even.
 * Launches on `stream`, no host sync: ModUp; then, for n >= 2^14 and
 * dnum <= 4, the column stages of the digits' NTT and one kernel that runs
 * their block stages and the inner product together (the transformed digits
 * never return to memory; 3 launches in all); otherwise the digits' NTT and
 * a separate inner-product kernel.
 * For digits of at most 8 primes and n >= 128, ModUp's extension runs on the
 * tensor cores (fp16 products of byte and 7-bit limbs, f32 sums, every sum an
 * integer below 2^24, so the result is exact and identical to the integer
 * path's): a kernel that gave up a bounded wait on them sets
 * FHE_STATUS_TC_TIMEOUT in the device status word (fhe_device_status) and its
 * outputs are invalid. */
int fhe_keyswitch_ip(uint64_t *out, const uint64_t *in, size_t in_stride, const uint64_t *keys,
                     int log_n, int L, int K, int dnum, int batch, const fhe_ntt_tables *t_qp,
                     const void *modup, uint64_t *workspace, size_t ws_bytes, void *stream);

/* ModUp variants of the key switch. */
#define FHE_MODUP_EXACT 0    /* Garner: X_j exactly, as above */
#define FHE_MODUP_APPROX 1   /* approximate basis conversion (next paragraph) */

/* fhe_keyswitch_ip with a choice of ModUp.  FHE_MODUP_APPROX replaces the
 * exact X_j by the CRT sum sum_a [x_a (D_j/d_a)^-1]_{d_a} (D_j/d_a) = X_j + e D_j
 * with 0 <= e < (primes in digit j), D_j the digit's modulus: alpha products
 * and alpha multiply-accumulates per target instead of Garner's quadratic
 * recursion; the extra e D_j is a multiple of the digit modulus (zero on the
 * digit's own primes, which are copied in both variants).  The cheaper
 * inexact ModUp of FHElium's "mixed-radix decomposition and basis extension"
 * family ("Eager, Compile, and native execution", section "CUDA execution").
 * Same arguments, workspace and rules as fhe_keyswitch_ip otherwise. */
int fhe_keyswitch_ip_ex(uint64_t *out, const uint64_t *in, size_t in_stride, const uint64_t *keys,
                        int log_n, int L, int K, int dnum, int batch, int modup_mode,
                        const fhe_ntt_tables *t_qp, const void *modup, uint64_t *workspace,
                        size_t ws_bytes, void *stream);

/* Hoisted key switch for R Galois elements (the rotations of coeff_to_slot
 * and slot_to_coeff, which kestrel-llm's boot profile reports as about 80% of
 * a bootstrap; overview, section 4.2).  The digit ModUp and its NTT are
 * computed once; then for every r < R the automorphism sigma_{galois[r]} of
 * the extended digits (NTT domain, the index map of fhe_automorph) is fused
 * into the inner product with that rotation's keys:
 *   out[r][b][c][l] = sum_j sigma_{galois[r]}(NTT(X_j))[l] * keys[r][j][c][l]  mod qp_l
 *   in:     as fhe_keyswitch_ip (coefficient domain, in_stride as there)
 *   keys:   [R][dnum][2][L+K][n]    NTT domain, basis qp
 *   out:    [R][batch][2][L+K][n]   NTT domain, basis qp
 *   galois: HOST array of R odd elements in [1, 2n), 1 <= R <= 64 (a device
 *           pointer gives FHE_EDEVICE)
 * sigma_k(X_j) is congruent to the extension of sigma_k(in) modulo the digit's
 * primes, so this is a valid key switch of each rotated input.  Workspace as
 * fhe_keyswitch_ip (fhe_keyswitch_workspace_bytes, independent of R). */
int fhe_keyswitch_hoisted(uint64_t *out, const uint64_t *in, size_t in_stride, const uint64_t *keys,
                          const uint32_t *galois, int R, int log_n, int L, int K, int dnum, int batch,
                          int modup_mode, const fhe_ntt_tables *t_qp, const void *modup,
                          uint64_t *workspace, size_t ws_bytes, void *stream);

/* The two halves of fhe_keyswitch_ip / fhe_keyswitch_hoisted, for callers
 * that reuse one decomposition across several calls (more rotations or key
 * sets later) or schedule the halves on different streams.
 *
 * fhe_keyswitch_decompose: digits [batch][dnum][L+K][n] (NTT domain, basis
 * qp) = NTT(X_j) of every digit of `in` (arguments as fhe_keyswitch_ip;
 * `digits` is fhe_keyswitch_workspace_bytes long and must not overlap in or
 * the tables).
 *
 * fhe_keyswitch_apply: with galois == NULL and R == 1,
 *   out[b][c][l] = sum_j digits[b][j][l] * keys[j][c][l]            (keys [dnum][2][L+K][n])
 * otherwise (host array of R odd elements in [1, 2n), 1 <= R <= 64)
 *   out[r][b][c][l] = sum_j sigma_{galois[r]}(digits[b][j])[l] * keys[r][j][c][l]
 * out must not overlap digits, keys or the tables. */
int fhe_keyswitch_decompose(uint64_t *digits, const uint64_t *in, size_t in_stride, int log_n, int L, int K,
                            int dnum, int batch, int modup_mode, const fhe_ntt_tables *t_qp,
                            const void *modup, void *stream);
int fhe_keyswitch_apply(uint64_t *out, const uint64_t *digits, const uint64_t *keys, const uint32_t *galois,
                        int R, int log_n, int L, int K, int dnum, int batch, const fhe_ntt_tables *t_qp,
                        void *stream);

/* ---- basis conversion and modraise ------------------------------------ */

#define FHE_BCONV_EXACT 0    /* Garner: X in [0, Q) */
#define FHE_BCONV_APPROX 1   /* CRT sum without correction: X + e Q, 0 <= e < S */

/* Conversion of every coefficient from S source primes (Q = their product)
 * to T target primes, coefficient domain.  Modraise -- kestrel-llm's
 * bootstrap entry, the Garner extension that lifts a low-level ciphertext
 * back to the full chain (overview, section 4.2) -- is FHE_BCONV_EXACT with
 * the sources = the first S primes of the chain and the targets = the whole
 * chain; the value taken is X in [0, Q) (no centring).  A target equal to a
 * source reproduces the input limb in both modes.
 *   in:  [batch][S][n]; out: [batch][T][n]; 1 <= S <= 16, 1 <= T <= 8192,
 *   batch <= 65535; every prime in (2^48, 2^50), sources distinct.
 * out must not overlap in or the tables (FHE_EALIAS). */
int fhe_bconv_tables_bytes(int S, int T, size_t *bytes);
int fhe_bconv_tables_build_host(int S, const uint64_t *src, int T, const uint64_t *dst, void *host_blob,
                                size_t bytes);
int fhe_bconv(uint64_t *out, const uint64_t *in, int log_n, int S, int T, int batch, int mode,
              const void *bconv, void *stream);

/* ---- ModDown and rescale ---------------------------------------------- */

#define FHE_ROUND_TRUNCATE 0
#define FHE_ROUND_NEAREST 1

/* Division by P = p_0 ... p_{K-1} with rounding (FHElium "QP-to-Q ModDown"
 * and "nearest and truncating rescale kernels", "Eager, Compile, and native
 * execution", section "CUDA execution"; kestrel-llm vllm_ckks.c rescale,
 * overview section 3).  Basis qp = (q_0..q_{L-1}, p_0..p_{K-1}), 1 <= K <= 16.
 * Per coefficient, with X the exact CRT value in [0, QP):
 *   out_l = floor((X + h) / P) mod q_l,  h = (P-1)/2 (FHE_ROUND_NEAREST) or 0
 *   (FHE_ROUND_TRUNCATE).
 * Computed as (x_l - (((X + h) mod P) - h)) P^-1 mod q_l with (X + h) mod P
 * obtained exactly from the P residues (Garner's mixed radix; in the NTT
 * domain with K <= 8 and n >= 128 the same value from the CRT brackets and
 * an exact correction count, extended on the tensor cores as in
 * fhe_keyswitch_ip, with the same device status word). */

/* Size of the constant blob for (L, K). */
int fhe_moddown_tables_bytes(int L, int K, size_t *bytes);

/* Build the constants for basis qp[L+K] (host) into host memory; copy the
 * blob unchanged to a 16-byte aligned device buffer and pass it as `md`. */
int fhe_moddown_tables_build_host(int L, int K, const uint64_t *qp, void *host_blob, size_t bytes);

/* Workspace bytes of fhe_moddown: batch * (L + K) * n * 8. */
int fhe_moddown_workspace_bytes(int log_n, int L, int K, int batch, size_t *bytes);

/* in: [batch][L+K][n] over qp; out: [batch][L][n] over q_0..q_{L-1}; both in
 * `domain` (FHE_DOMAIN_COEFF or FHE_DOMAIN_NTT; the NTT-domain result is the
 * NTT over Q of the coefficient-domain result of the INTT over QP of `in`).
 * t_qp: NTT tables covering at least the L+K primes of qp in that order.
 * workspace: at least fhe_moddown_workspace_bytes, contents ignored.  out
 * must not overlap in, workspace or the tables; in must not overlap the
 * workspace (FHE_EALIAS). */
int fhe_moddown(uint64_t *out, const uint64_t *in, int log_n, int L, int K, int batch, int domain,
                int rounding, const fhe_ntt_tables *t_qp, const void *md, uint64_t *workspace,
                size_t ws_bytes, void *stream);

/* Rescale: drop the last of L primes, out = floor((X + h) / q_{L-1}) over
 * q_0..q_{L-2}; exactly fhe_moddown with (L-1, 1).  in: [batch][L][n];
 * out: [batch][L-1][n]; rs = fhe_moddown_tables_build_host(L-1, 1, q).
 * Workspace: fhe_moddown_workspace_bytes(log_n, L-1, 1, batch). */
int fhe_rescale(uint64_t *out, const uint64_t *in, int log_n, int L, int batch, int domain, int rounding,
                const fhe_ntt_tables *t_q, const void *rs, uint64_t *workspace, size_t ws_bytes,
                void *stream);

/* ---- key switch without device allocation ----------------------------- */

/* The pages have no counterpart to this entry point; it serves callers of
 * this library that cannot allocate device memory: code that runs where
 * cudaMalloc/cudaFree are not allowed (they can synchronise the device),
 * services whose GPU memory is partitioned once at start-up, and runtimes
 * that embed the library without an allocator.
 *
 * fhe_keyswitch_ip_noalloc computes exactly what fhe_keyswitch_ip computes
 * (same arguments minus the workspace, same validation, kernels and
 * results), taking its workspace from one fixed array in the library's own
 * device memory of fhe_keyswitch_noalloc_max_bytes() bytes (16 MiB), which
 * every GPU that loads the library holds until the process exits.
 *   - Sizes: if fhe_keyswitch_workspace_bytes(log_n, L, K, dnum, batch)
 *     exceeds that maximum the call returns FHE_ESPACE before any launch
 *     (e.g. n = 2^13, L+K = 32, dnum = 3 needs 6 MiB and fits; n = 2^16
 *     with the same basis needs 48 MiB and does not -- use
 *     fhe_keyswitch_ip with a caller workspace).
 *   - Allocation: none -- no cudaMalloc, cudaFree or allocating library
 *     routine is called.
 *   - Set-up: every call looks up the array's device address
 *     (cudaGetSymbolAddress, with the operands' device current); nothing is
 *     cached, so the address stays right after a cudaDeviceReset.  The
 *     first call on a device also loads the library's device code there:
 *     make that first call before any stream capture.
 *   - Sharing: every call on a device uses the same array, which keeps the
 *     last call's contents.  Nothing in it has to start at zero (each call
 *     writes every word it later reads), but calls whose kernels overlap on
 *     the GPU (different streams without ordering between them) race on the
 *     array and give wrong results: order them on one stream or with events. */
int fhe_keyswitch_ip_noalloc(uint64_t *out, const uint64_t *in, size_t in_stride, const uint64_t *keys,
                             int log_n, int L, int K, int dnum, int batch, const fhe_ntt_tables *t_qp,
                             const void *modup, void *stream);

/* Bytes of the fixed workspace behind fhe_keyswitch_ip_noalloc (16 MiB). */
size_t fhe_keyswitch_noalloc_max_bytes(void);

#ifdef __cplusplus
}
#endif

#endif /* FHE_NTT_H */
