"""GPU parity on the long bootstrap chain: n = 2^11 with 2100 primes (the
kestrel-llm boot chain, overview sections 6-7: "np2100"), through the
forward NTT, the ciphertext tensor product and the inverse NTT of 4
ciphertext pairs (16 polynomials, 551 MB of residues), and the modraise of a
level-0 ciphertext to the whole chain.

Sampled limbs are compared element by element with the oracle (forward NTT,
tensor, inverse NTT and the schoolbook negacyclic product); on the device,
every limb of every polynomial is checked for INTT(NTT(x)) == x and for
residues below their modulus.
"""
import numpy as np
import pytest

import oracle
from ntt_arithmetic_gb300 import inputs

pytestmark = pytest.mark.gpu

LOG_N, L, PAIRS = 11, 2100, 4
N = 1 << LOG_N
SAMPLE_LIMBS = [0, 1, 2, 517, 1049, 1050, 1733, 2098, 2099]


@pytest.fixture(scope="module")
def g():
    import gpu_util
    return gpu_util


@pytest.fixture(scope="module")
def chain(g):
    import torch
    qs = list(g.primes(LOG_N, L))
    assert len(set(qs)) == L and all(q % (2 * N) == 1 and (1 << 48) < q < (1 << 50) for q in qs)
    t = g.api.NttTables(LOG_N, qs)
    x = inputs.uniform_residues((2, PAIRS, 2, L, N), qs, 900, buffer=0)
    return qs, t, x, torch.tensor(qs, dtype=torch.int64, device="cuda").view(L, 1)


def test_chain_ntt_tensor_intt(g, chain):
    import torch
    qs, t, x, qcol = chain
    X = g.dev(x)
    g.api.ntt_fwd(X, t)
    assert bool((X.view(torch.int64) < qcol).all())
    D = torch.empty((PAIRS, 3, L, N), dtype=torch.uint64, device="cuda")
    g.api.tensor(D, X[0], X[1], t)
    g.api.ntt_inv(D, t)
    assert bool((D.view(torch.int64) < qcol).all())
    Xh = g.host(X)
    Dh = g.host(D)
    for l in SAMPLE_LIMBS:
        q = qs[l]
        p = oracle.psi(q, 2 * N)
        for pair in (0, PAIRS - 1):
            a = [x[0, pair, c, l] for c in range(2)]
            b = [x[1, pair, c, l] for c in range(2)]
            for c in range(2):
                assert np.array_equal(Xh[0, pair, c, l], oracle.ntt(a[c], q, p)), (l, pair, c)
            want = oracle.tensor_batch(np.stack([oracle.ntt(v, q, p) for v in a])[None, :, None],
                                       np.stack([oracle.ntt(v, q, p) for v in b])[None, :, None], [q])[0, :, 0]
            for c in range(3):
                assert np.array_equal(Dh[pair, c, l], oracle.intt(want[c], q, p)), (l, pair, c)
        # the coefficient-domain result is the schoolbook product
        assert np.array_equal(Dh[0, 0, l], oracle.negacyclic_mul(x[0, 0, 0, l], x[1, 0, 0, l], q))
        d1 = (oracle.negacyclic_mul(x[0, 0, 0, l], x[1, 0, 1, l], q).astype(object)
              + oracle.negacyclic_mul(x[0, 0, 1, l], x[1, 0, 0, l], q).astype(object)) % q
        assert np.array_equal(Dh[0, 1, l], d1.astype(np.uint64))


def test_chain_round_trip_every_limb(g, chain):
    qs, t, x, qcol = chain
    X = g.dev(x)
    g.api.ntt_fwd(X, t)
    g.api.ntt_inv(X, t)
    assert g.same_bits(X, g.dev(x))


def test_chain_modraise(g, chain):
    """Level-0 ciphertext (c0, c1) over q_0 lifted to all 2100 primes."""
    import torch
    qs, t, x, qcol = chain
    bt = g.api.BconvTables(qs[:1], qs)
    lo = np.ascontiguousarray(x[0, 0, :, :1])                  # [2][1][n]
    out = torch.empty((2, L, N), dtype=torch.uint64, device="cuda")
    g.api.modraise(out, g.dev(lo), bt)
    got = g.host(out)
    want = np.broadcast_to(lo, (2, L, N)) % np.array(qs, dtype=np.uint64)[None, :, None]
    assert np.array_equal(got, want)
