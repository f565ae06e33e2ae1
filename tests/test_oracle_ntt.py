"""Pins for the oracle's forward/inverse negacyclic NTT and schoolbook product.

The kestrel-llm overview (section 3, "key point" paragraph) validates its
negacyclic NTT bit for bit against the textbook O(n^2) product; the same pin
is used here, next to a hand-computed worked example, evaluation by Horner's
rule at the roots of X^n + 1, delta inputs and the inverse identities.
"""
import os

import numpy as np
import pytest

import oracle
from ntt_arithmetic_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_fixture(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, *v = line.split()
                vals[k] = [int(x) for x in v]
    return vals


def py_brv(x, bits):
    return int(format(x, f"0{bits}b")[::-1], 2) if bits else 0


def horner(a, x, q):
    acc = 0
    for c in reversed([int(v) for v in a]):
        acc = (acc * x + c) % q
    return acc


def test_hand_worked_example():
    g = read_fixture("ntt_q17_n4.txt")
    q, n, psi = g["q"][0], g["n"][0], g["psi"][0]
    assert oracle.psi(q, 2 * n) == psi
    a = np.array(g["a"], dtype=np.uint64)
    assert list(oracle.ntt(a, q, psi)) == g["ahat"]
    assert list(oracle.ntt_direct(a, q, psi)) == g["ahat"]
    assert list(oracle.intt(np.array(g["ahat"], dtype=np.uint64), q, psi)) == g["a"]


def _cases():
    q2048 = [int(q) for q in oracle.primes(4096, 3)]   # q = 1 mod 4096 serves every n <= 2048
    for logn in range(1, 11):
        for q in q2048:
            yield logn, q


@pytest.mark.parametrize("logn,q", list(_cases()))
def test_fast_equals_direct(logn, q):
    n = 1 << logn
    psi = oracle.psi(q, 2 * n)
    a = inputs.uniform_row(q, n, 101, logn, q % 1000)
    A = oracle.ntt(a, q, psi)
    assert np.array_equal(A, oracle.ntt_direct(a, q, psi))
    assert np.array_equal(oracle.intt(A, q, psi), a)
    assert np.array_equal(oracle.intt_direct(A, q, psi), a)


@pytest.mark.parametrize("logn", [1, 2, 3, 6, 9])
def test_evaluation_at_roots_horner(logn):
    """ahat[i] is a(zeta_i) with zeta_i = psi^(2 brv(i) + 1); the zeta_i are the
    n distinct roots of X^n + 1."""
    n = 1 << logn
    q = int(oracle.primes(4096, 1)[0])
    psi = oracle.psi(q, 2 * n)
    zetas = [pow(psi, 2 * py_brv(i, logn) + 1, q) for i in range(n)]
    assert len(set(zetas)) == n and all(pow(z, n, q) == q - 1 for z in zetas)
    a = inputs.uniform_row(q, n, 5, 0, logn)
    A = oracle.ntt(a, q, psi)
    assert [int(v) for v in A] == [horner(a, z, q) for z in zetas]


@pytest.mark.parametrize("logn", [1, 4, 11, 16])
def test_delta_inputs(logn):
    n = 1 << logn
    q = int(oracle.primes(1 << 17, 1)[0])
    psi = oracle.psi(q, 2 * n)
    e0 = np.zeros(n, dtype=np.uint64); e0[0] = 1
    assert np.all(oracle.ntt(e0, q, psi) == 1)
    e1 = np.zeros(n, dtype=np.uint64)
    if n > 1:
        e1[1] = 1
        A = oracle.ntt(e1, q, psi)
        idx = np.arange(n)
        sample = idx if n <= 64 else np.random.default_rng(1).choice(n, 64, replace=False)
        for i in sample:
            assert int(A[i]) == pow(psi, 2 * py_brv(int(i), logn) + 1, q)


@pytest.mark.parametrize("logn", [12, 14, 16, 17])
def test_inverse_identities_large(logn):
    n = 1 << logn
    q = int(oracle.primes(2 * n, 2)[1])
    psi = oracle.psi(q, 2 * n)
    a = inputs.uniform_row(q, n, 9, 1, logn)
    assert np.array_equal(oracle.intt(oracle.ntt(a, q, psi), q, psi), a)
    assert np.array_equal(oracle.ntt(oracle.intt(a, q, psi), q, psi), a)


def negacyclic_reference(a, b, q):
    """Independent product: exact integer full convolution (numpy object
    dtype, Python ints), then fold with X^n = -1."""
    n = len(a)
    full = np.convolve(np.array([int(v) for v in a], dtype=object),
                       np.array([int(v) for v in b], dtype=object))
    c = [0] * n
    for k, v in enumerate(full):
        if k < n:
            c[k] += v
        else:
            c[k - n] -= v
    return [v % q for v in c]


@pytest.mark.parametrize("logn", [1, 2, 5, 8])
def test_schoolbook_vs_integer_convolution(logn):
    n = 1 << logn
    q = int(oracle.primes(4096, 1)[0])
    a = inputs.uniform_row(q, n, 11, 0, logn)
    b = inputs.uniform_row(q, n, 11, 1, logn)
    assert [int(v) for v in oracle.negacyclic_mul(a, b, q)] == negacyclic_reference(a, b, q)


def test_schoolbook_vs_sympy_ntt_convolution():
    sympy_conv = pytest.importorskip("sympy.discrete.convolutions")
    n = 256
    q = int(oracle.primes(4096, 1)[0])
    a = inputs.uniform_row(q, n, 12, 0, 0)
    b = inputs.uniform_row(q, n, 12, 1, 0)
    full = sympy_conv.convolution_ntt([int(v) for v in a], [int(v) for v in b], prime=q)
    full = list(full) + [0] * (2 * n - len(full))
    expect = [(full[k] - full[k + n]) % q for k in range(n)]
    assert [int(v) for v in oracle.negacyclic_mul(a, b, q)] == expect


def test_x_times_x_n_minus_1_is_minus_one():
    n = 64
    q = int(oracle.primes(4096, 1)[0])
    a = np.zeros(n, dtype=np.uint64); a[1] = 1
    b = np.zeros(n, dtype=np.uint64); b[n - 1] = 1
    c = oracle.negacyclic_mul(a, b, q)
    assert int(c[0]) == q - 1 and not c[1:].any()


@pytest.mark.parametrize("L_idx", [0, 1, 2, 3])
def test_convolution_theorem_n2048(L_idx):
    """INTT(NTT(a) * NTT(b)) equals the schoolbook negacyclic product at the
    PR1 size (n=2048, each of the 4 largest q = 1 mod 4096)."""
    n = 2048
    q = int(oracle.primes(4096, 4)[L_idx])
    psi = oracle.psi(q, 2 * n)
    a = inputs.uniform_row(q, n, 1, 0, L_idx)
    b = inputs.uniform_row(q, n, 1, 1, L_idx)
    A, B = oracle.ntt(a, q, psi), oracle.ntt(b, q, psi)
    C = np.array([(int(x) * int(y)) % q for x, y in zip(A, B)], dtype=np.uint64)
    assert np.array_equal(oracle.intt(C, q, psi), oracle.negacyclic_mul(a, b, q))


def test_linearity():
    n = 1024
    q = int(oracle.primes(4096, 1)[0])
    psi = oracle.psi(q, 2 * n)
    a = inputs.uniform_row(q, n, 2, 0, 0)
    b = inputs.uniform_row(q, n, 2, 1, 0)
    s = np.array([(int(x) + int(y)) % q for x, y in zip(a, b)], dtype=np.uint64)
    A, B, S = oracle.ntt(a, q, psi), oracle.ntt(b, q, psi), oracle.ntt(s, q, psi)
    assert all(int(S[i]) == (int(A[i]) + int(B[i])) % q for i in range(n))


def test_batch_driver_matches_single_rows():
    n, L, batch = 256, 5, 3
    qs = oracle.primes(2 * n, L)
    ps = oracle.psis(qs, n)
    x = inputs.uniform_residues((batch, L, n), qs, 4)
    y = oracle.ntt_batch(x, qs, ps, threads=3)
    for b in range(batch):
        for l in range(L):
            assert np.array_equal(y[b, l], oracle.ntt(x[b, l], int(qs[l]), int(ps[l])))
    assert np.array_equal(oracle.ntt_batch(y, qs, ps, inverse=True, threads=2), x)
