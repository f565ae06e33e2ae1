// ntt_shapes.h -- launch shape of the NTT kernels per log2(n), shared by the
// kernels (ntt.cu) and the table builder (tables.cpp), which lays out the
// forward twiddles of the last register pass in the order that pass reads.
#pragma once

// Forward launch shape per log2(n): the number of blocks a row is cut into
// (log2 C), threads per CTA (log2 T), residues per thread (log2 E, = radix of
// a register pass), the minimum number of resident CTAs per SM the register
// allocation must allow, and the kernel structure:
//   0 -- one CTA per row (log2 C = 0), every stage in one kernel;
//   1 -- split: a column kernel runs the first log2 C stages over the whole
//        row, then C independent CTAs run the remaining stages on one block
//        each.
// Measured on GB300 (201 MB of residues): the split beat a thread-block
// cluster of C CTAs per row exchanging through L2 by 8 % at n = 2^16 and 20 %
// at 2^17.  Blocks of 1024 residues (64 threads x 16, 8 CTAs per SM) beat
// blocks of 2048 at n = 2^16 (245 against 250 us forward, 234 against 237 us
// inverse on 384 rows), at 2^15 (248 against 253 / 230 against 234 us) and at
// 2^14 (249 against 257 us forward); blocks of 4096 (256 threads) or 8
// residues per thread were 8 % slower.  The forward block kernels of 1024
// residues run at 10 CTAs per SM (96 registers, no spills): 247 / 244 / 249
// against 253 / 249 / 253 us at n = 2^14 / 2^15 / 2^16 with 8 per SM (126
// registers); 12 per SM (80 registers) spilled and was slower, and the
// inverse block kernels gained nothing from 10.  At 2^17 blocks of 1024 would need 127
// staged twiddle rows per inverse column CTA (65 KB), so it keeps blocks of
// 2048.
// The inverse shapes (FHE_INV_SHAPE_n) have the same five fields; a split
// inverse runs the block CTAs first (the local stages) and the column kernel
// last (the last log2 C stages and the twist n^-1 psi^-j).
#define FHE_SHAPE_1 0, 0, 1, 1, 0
#define FHE_SHAPE_2 0, 0, 2, 1, 0
#define FHE_SHAPE_3 0, 0, 3, 1, 0
#define FHE_SHAPE_4 0, 1, 3, 1, 0
#define FHE_SHAPE_5 0, 2, 3, 1, 0
#define FHE_SHAPE_6 0, 3, 3, 1, 0
#define FHE_SHAPE_7 0, 4, 3, 1, 0
#define FHE_SHAPE_8 0, 5, 3, 1, 0
#define FHE_SHAPE_9 0, 6, 3, 1, 0
#define FHE_SHAPE_10 0, 7, 3, 1, 0
#define FHE_SHAPE_11 0, 7, 4, 4, 0
#define FHE_SHAPE_12 0, 8, 4, 2, 0
#define FHE_SHAPE_13 0, 8, 5, 2, 0
#define FHE_SHAPE_14 4, 6, 4, 10, 1
#define FHE_SHAPE_15 5, 6, 4, 10, 1
#define FHE_SHAPE_16 6, 6, 4, 10, 1
#define FHE_SHAPE_17 6, 7, 4, 4, 1

// Inverse shapes: split from n = 2^14 (measured against cluster shapes: 247
// against 263 us at 2^16, 259 against 338 us at 2^17, 227 against 229 us at
// 2^14, 230 against 234 us at 2^15), one CTA per row below.
#define FHE_INV_SHAPE_1 0, 0, 1, 1, 0
#define FHE_INV_SHAPE_2 0, 0, 2, 1, 0
#define FHE_INV_SHAPE_3 0, 0, 3, 1, 0
#define FHE_INV_SHAPE_4 0, 1, 3, 1, 0
#define FHE_INV_SHAPE_5 0, 2, 3, 1, 0
#define FHE_INV_SHAPE_6 0, 3, 3, 1, 0
#define FHE_INV_SHAPE_7 0, 4, 3, 1, 0
#define FHE_INV_SHAPE_8 0, 5, 3, 1, 0
#define FHE_INV_SHAPE_9 0, 6, 3, 1, 0
#define FHE_INV_SHAPE_10 0, 7, 3, 1, 0
#define FHE_INV_SHAPE_11 0, 7, 4, 4, 0
#define FHE_INV_SHAPE_12 0, 8, 4, 2, 0
#define FHE_INV_SHAPE_13 0, 8, 5, 2, 0
#define FHE_INV_SHAPE_14 4, 6, 4, 8, 1
#define FHE_INV_SHAPE_15 5, 6, 4, 8, 1
#define FHE_INV_SHAPE_16 6, 6, 4, 8, 1
#define FHE_INV_SHAPE_17 6, 7, 4, 4, 1

namespace fhe {

struct NttShape {
    int logc, logt, loge, minb, split;
};

constexpr NttShape ntt_shape(int log_n) {
    switch (log_n) {
        case 1: return {FHE_SHAPE_1};
        case 2: return {FHE_SHAPE_2};
        case 3: return {FHE_SHAPE_3};
        case 4: return {FHE_SHAPE_4};
        case 5: return {FHE_SHAPE_5};
        case 6: return {FHE_SHAPE_6};
        case 7: return {FHE_SHAPE_7};
        case 8: return {FHE_SHAPE_8};
        case 9: return {FHE_SHAPE_9};
        case 10: return {FHE_SHAPE_10};
        case 11: return {FHE_SHAPE_11};
        case 12: return {FHE_SHAPE_12};
        case 13: return {FHE_SHAPE_13};
        case 14: return {FHE_SHAPE_14};
        case 15: return {FHE_SHAPE_15};
        case 16: return {FHE_SHAPE_16};
        case 17: return {FHE_SHAPE_17};
        default: return {0, 0, 1, 1, 0};
    }
}

// Stages in the forward transform's last register pass (local bits [0, EP)).
constexpr int fwd_last_pass_stages(int log_n) {
    const NttShape s = ntt_shape(log_n);
    const int logm = log_n - s.logc;
    const int p = (logm + s.loge - 1) / s.loge;
    return p == 1 ? logm : s.loge;
}

// Storage slot of forward twiddle k (the value psi^brv(k), brv over log_n
// bits) in a prime's fwd table.  Stage s uses k in [2^s, 2^(s+1)); inside
// the last pass's stages (s >= log_n - EP, I = s - (log_n - EP)) the offset
// k - 2^s = (r, g, jj) -- cluster rank r, group g of 2^G, G = log_n - logc - EP,
// twiddle jj of 2^I -- is stored as (r, jj, g), so that the threads of a warp
// (consecutive g) read consecutive 16-byte entries.  Other stages: slot = k.
constexpr uint32_t fwd_table_slot(int log_n, uint32_t k) {
    if (k < 2) return k;
    int s = 0;
    while ((k >> (s + 1)) != 0) s++;
    const int ep = fwd_last_pass_stages(log_n);
    if (s < log_n - ep) return k;
    const int i = s - (log_n - ep);
    const int gbits = log_n - ntt_shape(log_n).logc - ep;
    const uint32_t off = k - (1u << s);
    const uint32_t jj = off & ((1u << i) - 1);
    const uint32_t g = (off >> i) & ((1u << gbits) - 1);
    const uint32_t r = off >> (i + gbits);
    return (1u << s) + (r << (i + gbits)) + (jj << gbits) + g;
}

}  // namespace fhe
