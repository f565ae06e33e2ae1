"""Pins for the oracle's Galois automorphism sigma_k: a(X) -> a(X^k).

FHElium lists Galois automorphisms among its CKKS-local tensor primitives
("Eager, Compile, and native execution", table "Native operator families");
the kestrel-llm overview (section 4.2) builds coeff_to_slot and
slot_to_coeff from Galois rotations plus key-switching.  The pages give no
formula; sigma_k is pinned here by monomials, composition, the ring
homomorphism property and (NTT domain) the closed-form index permutation.
"""
import numpy as np
import pytest

import oracle
from ntt_arithmetic_gb300 import inputs


def py_brv(x, bits):
    return int(format(x, f"0{bits}b")[::-1], 2) if bits else 0


def setup(logn, seed=0):
    n = 1 << logn
    q = int(oracle.primes(1 << 17, 1)[0]) if logn <= 16 else int(oracle.primes(2 * n, 1)[0])
    return n, q, oracle.psi(q, 2 * n)


@pytest.mark.parametrize("logn", [1, 3, 6, 10])
def test_monomials(logn):
    n, q, _ = setup(logn)
    rng = np.random.default_rng(logn)
    for k in [1, 3, 5, 2 * n - 1] + [int(2 * rng.integers(0, n) + 1) for _ in range(4)]:
        for t in range(0, n, max(1, n // 16)):
            a = np.zeros(n, dtype=np.uint64); a[t] = 7
            out = oracle.automorph_coeff(a, q, k)
            e = (t * k) % (2 * n)
            expect = np.zeros(n, dtype=np.uint64)
            if e < n:
                expect[e] = 7
            else:
                expect[e - n] = q - 7
            assert np.array_equal(out, expect), (k, t)


@pytest.mark.parametrize("logn", [4, 9])
def test_identity_and_composition(logn):
    n, q, psi = setup(logn)
    a = inputs.uniform_row(q, n, 3, 0, logn)
    assert np.array_equal(oracle.automorph_coeff(a, q, 1), a)
    conj = oracle.automorph_coeff(a, q, 2 * n - 1)
    assert np.array_equal(oracle.automorph_coeff(conj, q, 2 * n - 1), a)
    rng = np.random.default_rng(logn)
    for _ in range(5):
        k, m = (int(2 * rng.integers(0, n) + 1) for _ in range(2))
        lhs = oracle.automorph_coeff(oracle.automorph_coeff(a, q, m), q, k)
        assert np.array_equal(lhs, oracle.automorph_coeff(a, q, (k * m) % (2 * n)))
    A = oracle.ntt(a, q, psi)
    assert np.array_equal(oracle.automorph_ntt(A, q, psi, 1), A)


@pytest.mark.parametrize("logn", [3, 7])
def test_ring_homomorphism(logn):
    n, q, _ = setup(logn)
    a = inputs.uniform_row(q, n, 4, 0, logn)
    b = inputs.uniform_row(q, n, 4, 1, logn)
    for k in [3, 5, 2 * n - 1, 2 * n - 3]:
        lhs = oracle.automorph_coeff(oracle.negacyclic_mul(a, b, q), q, k)
        rhs = oracle.negacyclic_mul(oracle.automorph_coeff(a, q, k), oracle.automorph_coeff(b, q, k), q)
        assert np.array_equal(lhs, rhs), k


@pytest.mark.parametrize("logn", [1, 2, 5, 11])
def test_ntt_domain_is_index_permutation(logn):
    """NTT(sigma_k(a))[i] = NTT(a)[j] with 2 brv(j) + 1 = k (2 brv(i) + 1) mod 2n:
    evaluating sigma_k(a) at zeta_i is evaluating a at zeta_i^k."""
    n, q, psi = setup(logn)
    a = inputs.uniform_row(q, n, 6, 0, logn)
    A = oracle.ntt(a, q, psi)
    inv_brv = {py_brv(i, logn): i for i in range(n)}
    for k in sorted({1, 3, 5, 2 * n - 1, (5 ** 3) % (2 * n), (2 * n + 1) // 2 | 1}):
        if k >= 2 * n:
            continue
        out = oracle.automorph_ntt(A, q, psi, k)
        for i in range(n):
            e = (k * (2 * py_brv(i, logn) + 1)) % (2 * n)
            j = inv_brv[(e - 1) // 2]
            assert out[i] == A[j], (k, i)


def test_galois_elements_of_the_n65536_workload():
    """k = 5^r mod 2^17 for r in {1, 2, 4, ..., 2^15}: r = 2^15 gives k = 1
    (5 has order 2^15 modulo 2^17) and r = 2^14 gives k = 2^16 + 1."""
    ks = [pow(5, 1 << j, 1 << 17) for j in range(16)]
    assert ks[-1] == 1 and ks[-2] == 65537
    assert all(k % 2 == 1 for k in ks) and len(set(ks)) == 16
