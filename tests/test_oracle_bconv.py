"""Oracle pins (not gpu): basis conversion (exact and approximate), modraise,
the approximate ModUp of the key switch and the hoisted key switch.

Exact conversion is checked against Python big-integer CRT.  The approximate
conversion has no single right value, so it is pinned by what defines it: its
output is X + e Q with one integer e in [0, S) shared by every target prime,
and e is not always 0.  The hoisted key switch is pinned by composition with
separately pinned pieces (key switch, automorphism) and by the congruence that
makes hoisting valid: sigma_k of an extended digit equals the extension of
sigma_k of the input modulo the digit's primes.
"""
import random

import numpy as np
import pytest

import oracle


def crt(res, mods):
    Q = 1
    for m in mods:
        Q *= int(m)
    X = 0
    for r, m in zip(res, mods):
        m = int(m)
        Mi = Q // m
        X += int(r) * Mi * pow(Mi, -1, m)
    return X % Q, Q


@pytest.fixture(scope="module")
def chain():
    # 12 primes = 1 mod 2^9 below 2^50 (n = 256)
    return [int(v) for v in oracle.primes(512, 12)]


@pytest.mark.parametrize("S", [1, 2, 3, 8])
def test_exact_bconv_is_crt(chain, S):
    rng = random.Random(S)
    src, dst = chain[:S], chain[S:]
    for _ in range(300):
        x = [rng.randrange(q) for q in src]
        X, _ = crt(x, src)
        got = oracle.bconv_coeff(x, src, dst, approx=False)
        assert [int(v) for v in got] == [X % p for p in dst]


@pytest.mark.parametrize("S", [2, 3, 5, 8])
def test_approx_bconv_overflow_is_one_small_multiple(chain, S):
    """out_p = X + e Q mod p for one e in [0, S), the same for every target."""
    rng = random.Random(100 + S)
    src, dst = chain[:S], chain[S:]
    seen = set()
    for _ in range(400):
        x = [rng.randrange(q) for q in src]
        X, Q = crt(x, src)
        got = oracle.bconv_coeff(x, src, dst, approx=True)
        es = {((int(g) - X) * pow(Q, -1, p)) % p for g, p in zip(got, dst)}
        assert len(es) == 1
        e = es.pop()
        assert 0 <= e < S
        seen.add(e)
    assert len(seen) > 1 and max(seen) >= 1     # the overflow is real, and not constant
    if S <= 3:
        assert 0 in seen


def test_bconv_source_primes_reproduce_input(chain):
    rng = random.Random(7)
    src = chain[:4]
    for approx in (False, True):
        for _ in range(50):
            x = [rng.randrange(q) for q in src]
            got = oracle.bconv_coeff(x, src, src + chain[4:6], approx=approx)
            assert [int(v) for v in got[:4]] == x


def test_single_source_prime_is_plain_reduction(chain):
    rng = random.Random(8)
    q = chain[0]
    for _ in range(100):
        x = rng.randrange(q)
        for approx in (False, True):
            got = oracle.bconv_coeff([x], [q], chain[1:], approx=approx)
            assert [int(v) for v in got] == [x % p for p in chain[1:]]


def test_bconv_batch_layout_and_modraise(chain):
    """Modraise: the first S limbs of a low-level polynomial extended to the
    whole chain; the layout [batch][S][n] -> [batch][T][n]."""
    n, S, batch = 64, 2, 3
    rng = np.random.default_rng(11)
    a = np.stack([np.stack([rng.integers(0, q, size=n, dtype=np.uint64) for q in chain[:S]])
                  for _ in range(batch)])
    out = oracle.bconv_batch(a, chain[:S], chain, approx=False)
    assert out.shape == (batch, len(chain), n)
    assert np.array_equal(out[:, :S], a)
    for b in range(batch):
        for i in range(0, n, 7):
            X, _ = crt(a[b, :, i], chain[:S])
            assert [int(v) for v in out[b, :, i]] == [X % p for p in chain]
    approx = oracle.bconv_batch(a, chain[:S], chain, approx=True)
    for b in range(batch):
        for i in range(n):
            assert np.array_equal(approx[b, :, i], oracle.bconv_coeff(a[b, :, i], chain[:S], chain, True))


def test_approx_modup_differs_from_exact_by_small_multiples(chain):
    n, L, K, dnum, batch = 32, 6, 3, 2, 2
    qp = chain[:L + K]
    rng = np.random.default_rng(12)
    a = np.stack([np.stack([rng.integers(0, q, size=n, dtype=np.uint64) for q in qp[:L]]) for _ in range(batch)])
    ex = oracle.modup_batch(a, qp, L, K, dnum)
    ap = oracle.modup_batch(a, qp, L, K, dnum, approx=True)
    alpha = (L + dnum - 1) // dnum
    for j in range(dnum):
        lo, hi = j * alpha, min((j + 1) * alpha, L)
        Qj = 1
        for q in qp[lo:hi]:
            Qj *= q
        assert np.array_equal(ap[:, j, lo:hi], a[:, lo:hi])          # in-digit limbs are copies
        for b in range(batch):
            for i in range(n):
                es = {((int(ap[b, j, l, i]) - int(ex[b, j, l, i])) * pow(Qj, -1, qp[l])) % qp[l]
                      for l in range(L + K) if not lo <= l < hi}
                assert len(es) == 1 and es.pop() < hi - lo


@pytest.fixture(scope="module")
def ks_setup():
    log_n, L, K, dnum, batch = 6, 6, 3, 3, 2
    n = 1 << log_n
    qp = [int(v) for v in oracle.primes(2 * n, L + K)]
    ps = oracle.psis(qp, n)
    rng = np.random.default_rng(13)
    a = np.stack([np.stack([rng.integers(0, q, size=n, dtype=np.uint64) for q in qp[:L]]) for _ in range(batch)])
    return log_n, L, K, dnum, batch, qp, ps, a, rng


def _rand_keys(rng, R, dnum, qp, n):
    return np.stack([np.stack([np.stack([np.stack([rng.integers(0, q, size=n, dtype=np.uint64) for q in qp])
                                         for _ in range(2)]) for _ in range(dnum)]) for _ in range(R)])


def test_hoisted_identity_is_keyswitch(ks_setup):
    log_n, L, K, dnum, batch, qp, ps, a, rng = ks_setup
    keys = _rand_keys(rng, 1, dnum, qp, 1 << log_n)
    for approx in (False, True):
        h = oracle.keyswitch_hoisted_batch(a, keys, [1], qp, ps, L, K, dnum, approx=approx)
        assert np.array_equal(h[0], oracle.keyswitch_batch(a, keys[0], qp, ps, L, K, dnum, approx=approx))


def test_hoisted_is_automorphism_of_extended_digit(ks_setup):
    """Key = 1 on digit j component 0, 0 elsewhere: out_r[b][0] is sigma_{k_r}
    of the NTT-domain extended digit j, out_r[b][1] is zero."""
    log_n, L, K, dnum, batch, qp, ps, a, rng = ks_setup
    n = 1 << log_n
    ks = [5, pow(5, 3, 2 * n), 2 * n - 1]
    for j in range(dnum):
        keys = np.zeros((len(ks), dnum, 2, L + K, n), dtype=np.uint64)
        keys[:, j, 0] = 1
        h = oracle.keyswitch_hoisted_batch(a, keys, ks, qp, ps, L, K, dnum)
        digit = oracle.keyswitch_batch(a, keys[0], qp, ps, L, K, dnum)[:, 0]     # NTT(ModUp_j(a))
        for r, k in enumerate(ks):
            assert np.array_equal(h[r, :, 0], oracle.automorph_batch(digit, qp, ps, k, ntt_domain=True))
            assert not h[r, :, 1].any()


def test_hoisting_congruence(ks_setup):
    """On the primes of digit j, sigma_k(ModUp_j(a)) and ModUp_j(sigma_k(a))
    agree (they differ by multiples of Q_j), so the hoisted result equals the
    key switch of the rotated input there."""
    log_n, L, K, dnum, batch, qp, ps, a, rng = ks_setup
    n = 1 << log_n
    alpha = (L + dnum - 1) // dnum
    k = pow(5, 7, 2 * n)
    rot = oracle.automorph_batch(a, qp[:L], ps[:L], k, ntt_domain=False)
    differs = False
    for j in range(dnum):
        lo, hi = j * alpha, min((j + 1) * alpha, L)
        keys = _rand_keys(rng, 1, dnum, qp, n)
        keys[:, [i for i in range(dnum) if i != j]] = 0
        h = oracle.keyswitch_hoisted_batch(a, keys, [k], qp, ps, L, K, dnum)[0]
        direct = oracle.keyswitch_batch(rot, keys[0], qp, ps, L, K, dnum)
        assert np.array_equal(h[:, :, lo:hi], direct[:, :, lo:hi])
        differs |= not np.array_equal(h, direct)
    assert differs     # outside the digit the two lifts differ: the hoisted path is not a re-run


def test_hoisted_rotations_are_independent(ks_setup):
    log_n, L, K, dnum, batch, qp, ps, a, rng = ks_setup
    n = 1 << log_n
    ks = [pow(5, 1 << r, 2 * n) for r in range(3)]
    keys = _rand_keys(rng, len(ks), dnum, qp, n)
    h = oracle.keyswitch_hoisted_batch(a, keys, ks, qp, ps, L, K, dnum)
    for r, k in enumerate(ks):
        one = oracle.keyswitch_hoisted_batch(a, keys[r:r + 1], [k], qp, ps, L, K, dnum)
        assert np.array_equal(h[r], one[0])
