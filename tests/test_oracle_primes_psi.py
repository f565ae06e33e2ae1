"""Pins for the oracle's prime search and root of unity (not gpu).

Readings pinned here: primes are the largest q < 2^50 with q = 1 (mod 2n),
descending (workload text of the n=2048/L=112 and n=2^16 configurations; the
kestrel-llm overview, sections 6-7, uses n=2048 with 112- and 2100-prime
chains); psi is the smallest primitive 2n-th root of unity (pages silent).
"""
import numpy as np
import pytest

import oracle


def trial_division_is_prime(q: int) -> bool:
    """Independent primality check: divide by every odd d <= sqrt(q)."""
    if q % 2 == 0:
        return q == 2
    lim = int(np.sqrt(float(q))) + 2
    d = np.arange(3, lim, 2, dtype=np.uint64)
    return not np.any(np.uint64(q) % d == 0)


@pytest.mark.parametrize("m,count", [(1 << 12, 4), (1 << 17, 2)])
def test_primes_trial_division(m, count):
    qs = [int(q) for q in oracle.primes(m, count)]
    for q in qs:
        assert q < 2 ** 50 and q % m == 1
        assert trial_division_is_prime(q)


@pytest.mark.parametrize("m,count", [(1 << 12, 112), (1 << 17, 32), (1 << 18, 64), (1 << 12, 4)])
def test_primes_are_the_largest(m, count):
    sympy = pytest.importorskip("sympy")
    qs = [int(q) for q in oracle.primes(m, count)]
    assert qs == sorted(qs, reverse=True) and len(set(qs)) == count
    # every candidate = 1 mod m between 2^50 and the last prime is either in the list or composite
    top = (2 ** 50 - 1) - ((2 ** 50 - 2) % m)
    listed = set(qs)
    c = top
    while c >= qs[-1]:
        assert (c in listed) == sympy.isprime(c), c
        c -= m


def test_first_primes_for_n2048_are_stable():
    # The PR1 configuration uses the 4 largest q < 2^50 with q = 1 mod 4096.
    # Fixed by sympy, independently of the oracle.
    sympy = pytest.importorskip("sympy")
    expect = []
    c = (2 ** 50 - 1) - ((2 ** 50 - 2) % 4096)
    while len(expect) < 4:
        if sympy.isprime(c):
            expect.append(c)
        c -= 4096
    assert [int(q) for q in oracle.primes(4096, 4)] == expect


def test_is_prime_special_cases():
    sympy = pytest.importorskip("sympy")
    # strong pseudoprimes to small bases and Carmichael numbers must be rejected
    for c in [2047, 1373653, 25326001, 3215031751, 2152302898747, 3474749660383,
              341550071728321, 3825123056546413051, 561, 1105, 1729, 2465, 2821, 6601]:
        assert oracle.is_prime(c) == sympy.isprime(c) == False  # noqa: E712
    rng = np.random.default_rng(7)
    for x in rng.integers(2, 2 ** 62, 300, dtype=np.uint64):
        assert oracle.is_prime(int(x)) == sympy.isprime(int(x))
    for p in [2, 3, 5, 37, 41, 2 ** 61 - 1, 18446744073709551557]:
        assert oracle.is_prime(p)


def brute_force_psi(q: int, m: int) -> int:
    """Smallest g in [2, q) with g^(m/2) = -1 (for m a power of two this is
    exactly 'g has multiplicative order m')."""
    for g in range(2, q):
        if pow(g, m // 2, q) == q - 1:
            return g
    raise AssertionError("no primitive root")


@pytest.mark.parametrize("q", [17, 97, 193, 257, 769, 7681, 12289, 40961, 65537])
def test_psi_brute_force_small(q):
    m = 2
    while (q - 1) % m == 0 and m <= 4096:
        assert oracle.psi(q, m) == brute_force_psi(q, m), (q, m)
        m *= 2


@pytest.mark.parametrize("logn,count", [(11, 112), (16, 32), (17, 64), (1, 4), (5, 4)])
def test_psi_is_primitive_2n_root(logn, count):
    n = 1 << logn
    for q in oracle.primes(2 * n, count)[:8]:
        q = int(q)
        p = oracle.psi(q, 2 * n)
        assert 2 <= p < q
        assert pow(p, n, q) == q - 1      # order exactly 2n (2n is a power of two)
        assert pow(p, 2 * n, q) == 1
