"""Pins for the oracle's ModDown (QP -> Q) and rescale (division by the last
prime), nearest and truncating.  FHElium's CUDA layer lists "key-switch
multiply-accumulate and QP-to-Q ModDown" and "nearest and truncating
rescale kernels" ("Eager, Compile, and native execution", section "CUDA
execution"); kestrel-llm's vllm_ckks.c has rescale (overview, section 3).
The pages give no formula; the reading is out = floor((X + h) / P) mod q_l
with X the exact CRT value in [0, QP) and h = (P-1)/2 (nearest) or 0.
Pinned here by Python big-integer division on random and extreme values.
"""
import numpy as np
import pytest

import oracle
from ntt_arithmetic_gb300 import inputs


def crt(residues, moduli):
    M = 1
    for m in moduli:
        M *= int(m)
    X = 0
    for r, m in zip(residues, moduli):
        Mi = M // int(m)
        X += int(r) * Mi * pow(Mi, -1, int(m))
    return X % M, M


@pytest.mark.parametrize("L,K,nearest", [(4, 2, True), (4, 2, False), (7, 3, True), (24, 8, True), (24, 8, False),
                                         (5, 1, True), (5, 1, False), (1, 1, True)])
def test_moddown_vs_bigint(L, K, nearest):
    n = 32
    qp = [int(v) for v in oracle.primes(1 << 17, L + K)]
    x = inputs.uniform_residues((2, L + K, n), qp, 77 + L + K)
    # extreme coefficients: X = 0, X = QP - 1, X = P - 1, X = (P - 1)/2, X = (P + 1)/2
    P = 1
    for p in qp[L:]:
        P *= p
    QP = 1
    for p in qp:
        QP *= p
    for i, X in enumerate([0, QP - 1, P - 1, (P - 1) // 2, (P + 1) // 2]):
        x[0, :, i] = [X % m for m in qp]
    out = oracle.moddown_batch(x, qp, L, K, nearest)
    h = (P - 1) // 2 if nearest else 0
    for b in range(2):
        for i in range(n):
            X, _ = crt(x[b, :, i], qp)
            want = (X + h) // P
            assert [int(v) for v in out[b, :, i]] == [want % q for q in qp[:L]], (b, i)


def test_rescale_rounds_to_nearest_and_truncates():
    """Rescale = division by the last prime: a message m*q_last + e with
    |e| < q_last/2 rescales to m (nearest) and to m or m-1 (truncating, e < 0)."""
    L = 4
    qp = [int(v) for v in oracle.primes(1 << 17, L)]
    ql = qp[-1]
    n = 16
    import random
    rng = random.Random(3)
    Q = 1
    for q in qp[:-1]:
        Q *= q
    ms = [rng.randrange(0, Q // 2) for _ in range(n)]
    es = [rng.randrange(-(ql // 2) + 1, ql // 2) for _ in range(n)]
    x = np.zeros((1, L, n), dtype=np.uint64)
    for i, (m, e) in enumerate(zip(ms, es)):
        X = (m * ql + e) % (Q * ql)
        x[0, :, i] = [X % q for q in qp]
    near = oracle.moddown_batch(x, qp, L - 1, 1, True)
    trunc = oracle.moddown_batch(x, qp, L - 1, 1, False)
    for i, (m, e) in enumerate(zip(ms, es)):
        assert [int(v) for v in near[0, :, i]] == [m % q for q in qp[:-1]]
        want = m if e >= 0 else m - 1
        assert [int(v) for v in trunc[0, :, i]] == [want % q for q in qp[:-1]]


def test_moddown_ntt_domain_is_conjugated_coefficient_moddown():
    n, L, K = 64, 3, 2
    qp = [int(v) for v in oracle.primes(2 * n, L + K)]
    ps = oracle.psis(qp, n)
    x = inputs.uniform_residues((2, L + K, n), qp, 88)
    X = oracle.ntt_batch(x, qp, ps)
    got = oracle.moddown_ntt_batch(X, qp, ps, L, K, True)
    want = oracle.ntt_batch(oracle.moddown_batch(x, qp, L, K, True), qp[:L], ps[:L])
    assert np.array_equal(got, want)
