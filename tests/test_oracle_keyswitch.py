"""Pins for the oracle's digit basis extension (ModUp), key-switch inner
product, pointwise multiply and ciphertext tensor product.

FHElium's CUDA layer provides "mixed-radix decomposition and basis
extension" and "key-switch multiply-accumulate" ("Eager, Compile, and native
execution", section "CUDA execution"); kestrel-llm raises the modulus chain
"by Garner extension" (overview, section 4.2) and multiplies ciphertexts in
vllm_ckks.c (section 3).  Pins: Python big-integer CRT by the textbook
formula (a different computation from Garner's mixed radix), special values,
a delta key, linearity, and a full small case built from Python integers only.
"""
import numpy as np
import pytest

import oracle
from ntt_arithmetic_gb300 import inputs


def crt_bigint(residues, moduli):
    """X = sum x_i * M_i * (M_i^-1 mod m_i) mod M, M_i = M / m_i (textbook CRT)."""
    M = 1
    for m in moduli:
        M *= int(m)
    X = 0
    for x, m in zip(residues, moduli):
        m = int(m)
        Mi = M // m
        X += int(x) * Mi * pow(Mi, -1, m)
    return X % M, M


def qp_basis(n, L, K):
    qp = [int(q) for q in oracle.primes(2 * n, L + K)]
    return qp


@pytest.mark.parametrize("alpha", [1, 2, 5, 8])
def test_modup_coeff_vs_bigint_crt(alpha):
    n = 1 << 16
    qp = qp_basis(n, 24, 8)
    digit, targets = qp[:alpha], qp
    rng = np.random.default_rng(alpha)
    for t in range(300):
        x = [int(rng.integers(0, q)) for q in digit]
        X, M = crt_bigint(x, digit)
        out = oracle.modup_coeff(x, digit, targets)
        assert [int(v) for v in out] == [X % p for p in targets]


def test_modup_special_values():
    qp = qp_basis(1 << 16, 24, 8)
    digit = qp[8:16]
    M = 1
    for q in digit:
        M *= q
    # zero, D - 1 and a small integer below every modulus
    for x, X in [([0] * 8, 0), ([q - 1 for q in digit], M - 1), ([12345] * 8, 12345)]:
        out = oracle.modup_coeff(x, digit, qp)
        assert [int(v) for v in out] == [X % p for p in qp]


def test_modup_batch_digits_and_copies():
    n, L, K, dnum = 64, 24, 8, 3
    qp = qp_basis(1 << 16, L, K)
    x = inputs.uniform_residues((2, L, n), qp[:L], 40)
    ext = oracle.modup_batch(x, qp, L, K, dnum, threads=2)
    assert ext.shape == (2, dnum, L + K, n)
    for b in range(2):
        for j in range(dnum):
            lo, hi = 8 * j, 8 * j + 8
            assert np.array_equal(ext[b, j, lo:hi], x[b, lo:hi])   # in-digit limbs copy the input
            for i in range(0, n, 7):
                X, _ = crt_bigint(x[b, lo:hi, i], qp[lo:hi])
                assert [int(v) for v in ext[b, j, :, i]] == [X % p for p in qp]


def test_modup_ragged_digits():
    """L not divisible by dnum: alpha = ceil(L/dnum), the last digit is short."""
    n, L, K, dnum = 16, 7, 3, 3
    qp = qp_basis(1 << 11, L, K)
    x = inputs.uniform_residues((1, L, n), qp[:L], 41)
    ext = oracle.modup_batch(x, qp, L, K, dnum, threads=1)
    for j, (lo, hi) in enumerate([(0, 3), (3, 6), (6, 7)]):
        for i in range(n):
            X, _ = crt_bigint(x[0, lo:hi, i], qp[lo:hi])
            assert [int(v) for v in ext[0, j, :, i]] == [X % p for p in qp]


def py_ntt_by_evaluation(a, q, psi, logn):
    n = 1 << logn
    out = []
    for i in range(n):
        z = pow(psi, 2 * int(format(i, f"0{logn}b")[::-1], 2) + 1, q)
        acc = 0
        for c in reversed([int(v) for v in a]):
            acc = (acc * z + c) % q
        out.append(acc)
    return out


def test_keyswitch_small_all_python():
    """Full small key switch computed from Python integers only (big-int CRT,
    evaluation at the roots of X^n+1, exact inner product)."""
    logn, L, K, dnum, batch = 4, 4, 2, 2, 2
    n = 1 << logn
    qp = qp_basis(n, L, K)
    psis = [oracle.psi(q, 2 * n) for q in qp]
    x = inputs.uniform_residues((batch, L, n), qp[:L], 50)
    keys = inputs.uniform_residues((dnum, 2, L + K, n), qp, 51)
    out = oracle.keyswitch_batch(x, keys, qp, psis, L, K, dnum, threads=2)
    for b in range(batch):
        ext = []
        for j in range(dnum):
            lo, hi = 2 * j, 2 * j + 2
            rows = []
            for l, p in enumerate(qp):
                coeffs = [crt_bigint(x[b, lo:hi, i], qp[lo:hi])[0] % p for i in range(n)]
                rows.append(py_ntt_by_evaluation(coeffs, p, psis[l], logn))
            ext.append(rows)
        for c in range(2):
            for l, p in enumerate(qp):
                expect = [sum(ext[j][l][i] * int(keys[j, c, l, i]) for j in range(dnum)) % p for i in range(n)]
                assert [int(v) for v in out[b, c, l]] == expect


def test_keyswitch_delta_key_and_linearity():
    logn, L, K, dnum = 8, 6, 2, 3
    n = 1 << logn
    qp = qp_basis(n, L, K)
    ps = oracle.psis(qp, n)
    x = inputs.uniform_residues((1, L, n), qp[:L], 60)
    ext = oracle.modup_batch(x, qp, L, K, dnum, threads=2)
    ext_ntt = oracle.ntt_batch(ext[0], qp, ps)      # [dnum][L+K][n]
    for j in range(dnum):
        keys = np.zeros((dnum, 2, L + K, n), dtype=np.uint64)
        keys[j, 0] = 1
        out = oracle.keyswitch_batch(x, keys, qp, ps, L, K, dnum, threads=2)
        assert np.array_equal(out[0, 0], ext_ntt[j]) and not out[0, 1].any()
    k1 = inputs.uniform_residues((dnum, 2, L + K, n), qp, 61)
    k2 = inputs.uniform_residues((dnum, 2, L + K, n), qp, 62)
    qcol = np.array(qp, dtype=object)[None, None, :, None]
    ksum = ((k1.astype(object) + k2.astype(object)) % qcol).astype(np.uint64)
    o1 = oracle.keyswitch_batch(x, k1, qp, ps, L, K, dnum).astype(object)
    o2 = oracle.keyswitch_batch(x, k2, qp, ps, L, K, dnum).astype(object)
    osum = oracle.keyswitch_batch(x, ksum, qp, ps, L, K, dnum)
    assert np.array_equal(osum, ((o1 + o2) % np.array(qp, dtype=object)[None, None, :, None]).astype(np.uint64))


def test_tensor_product_against_schoolbook():
    """In the NTT domain, d0 = a0 b0, d1 = a0 b1 + a1 b0, d2 = a1 b1 are the
    negacyclic products once transformed back (convolution theorem)."""
    n, L, batch = 256, 3, 2
    qs = oracle.primes(4096, L)
    ps = oracle.psis(qs, n)
    a = inputs.uniform_residues((batch, 2, L, n), qs, 70)
    b = inputs.uniform_residues((batch, 2, L, n), qs, 71)
    A = oracle.ntt_batch(a, qs, ps)
    B = oracle.ntt_batch(b, qs, ps)
    d = oracle.ntt_batch(oracle.tensor_batch(A, B, qs), qs, ps, inverse=True)
    for bi in range(batch):
        for l in range(L):
            q = int(qs[l])
            nm = lambda u, v: oracle.negacyclic_mul(u, v, q)  # noqa: E731
            assert np.array_equal(d[bi, 0, l], nm(a[bi, 0, l], b[bi, 0, l]))
            s = (nm(a[bi, 0, l], b[bi, 1, l]).astype(object) + nm(a[bi, 1, l], b[bi, 0, l]).astype(object)) % q
            assert np.array_equal(d[bi, 1, l], s.astype(np.uint64))
            assert np.array_equal(d[bi, 2, l], nm(a[bi, 1, l], b[bi, 1, l]))


def test_pointwise_mul_is_exact():
    n, L = 512, 4
    qs = oracle.primes(4096, L)
    a = inputs.uniform_residues((2, L, n), qs, 80)
    b = inputs.uniform_residues((2, L, n), qs, 81)
    # extreme values in the first row: q-1 times q-1 and zeros
    for l in range(L):
        a[0, l, :4] = [int(qs[l]) - 1, 0, 1, int(qs[l]) - 1]
        b[0, l, :4] = [int(qs[l]) - 1, int(qs[l]) - 1, int(qs[l]) - 1, 0]
    out = oracle.mul_batch(a, b, qs)
    q3 = np.array([int(q) for q in qs], dtype=object)[None, :, None]
    assert np.array_equal(out, ((a.astype(object) * b.astype(object)) % q3).astype(np.uint64))


def test_ciphertext_file_size_identity():
    """kestrel-llm overview, section 5: each hop writes 8 ciphertexts (4 token
    positions x 2 components), each about 3.5 MB, at n=2048 over 112 primes.
    A ciphertext of 2 polynomials of u64 residues [2][112][2048] is exactly
    3.5 MiB, which pins 64-bit residues and the (c0, c1) pair layout."""
    with open(__file__.replace("test_oracle_keyswitch.py", "golden/ciphertext_size.txt")) as f:
        vals = dict(line.split() for line in f if line.strip() and not line.startswith("#"))
    n, L, comps, word = (int(vals[k]) for k in ("n", "L", "components", "word_bytes"))
    assert comps * L * n * word == int(vals["bytes"]) == int(3.5 * 2 ** 20)
    assert int(vals["ciphertexts_per_hop"]) == 8
