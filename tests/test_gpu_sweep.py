"""GPU parity over the sweep workload: n in {2^11 .. 2^17}, L in {1, 8, 24,
64}, batch in {1, 16, 64} (84 points, up to 4 GiB per operand), for the
forward NTT, the fused pointwise product and the inverse NTT.

Points of up to FULL_BYTES per operand (78 of the 84) take distinct seeded
inputs on every row and compare every output row with the oracle, element by
element: the forward NTT of both operands, their pointwise product and its
inverse NTT.  The six multi-GiB points tile a seeded pool of 2 distinct batch
items on the device (host memory and oracle time would otherwise dominate the
suite) and compare the first, middle and last (batch, limb) row with the
oracle.  Every point also checks, on the device and on every row,
INTT(NTT(x)) == x and every output residue below its modulus.
"""
import os

import numpy as np
import pytest

import oracle
from ntt_arithmetic_gb300 import inputs

pytestmark = pytest.mark.gpu

LS = [1, 8, 24, 64]
BATCHES = [1, 16, 64]
FULL_BYTES = 540 << 20
THREADS = os.cpu_count() or 1


@pytest.fixture(scope="module")
def g():
    import gpu_util
    return gpu_util


def _tile(pool, batch):
    reps = (batch + pool.shape[0] - 1) // pool.shape[0]
    return pool.repeat(reps, 1, 1)[:batch].contiguous()


def _full_point(g, t, qs, ps, qcol, log_n, L, batch):
    import torch
    n = 1 << log_n
    a = inputs.uniform_residues((batch, L, n), qs, 7000 + log_n, buffer=100 * L + batch, threads=THREADS)
    b = inputs.uniform_residues((batch, L, n), qs, 8000 + log_n, buffer=100 * L + batch, threads=THREADS)
    x, y = g.dev(a), g.dev(b)
    g.api.ntt_fwd(x, t)
    g.api.ntt_fwd(y, t)
    A = oracle.ntt_batch(a, qs, ps)
    B = oracle.ntt_batch(b, qs, ps)
    assert np.array_equal(g.host(x), A), (log_n, L, batch, "fwd a")
    assert np.array_equal(g.host(y), B), (log_n, L, batch, "fwd b")
    g.api.mul_ntt(x, x, y, t)                         # fused pointwise product in the NTT domain
    P = oracle.mul_batch(A, B, qs)
    assert np.array_equal(g.host(x), P), (log_n, L, batch, "product")
    g.api.ntt_inv(x, t)
    assert np.array_equal(g.host(x), oracle.ntt_batch(P, qs, ps, inverse=True)), (log_n, L, batch, "inv")
    assert bool((x.view(torch.int64) < qcol).all())
    g.api.ntt_inv(y, t)                               # round trip of b on every row
    assert g.same_bits(y, g.dev(b)), (log_n, L, batch, "round trip")


def _sampled_point(g, t, qs, ps, qcol, log_n, L, batch):
    import torch
    n = 1 << log_n
    pool_a = g.dev(inputs.uniform_residues((2, L, n), qs, 5000 + log_n, buffer=L))
    pool_b = g.dev(inputs.uniform_residues((2, L, n), qs, 6000 + log_n, buffer=L))
    host_a, host_b = pool_a.cpu().numpy(), pool_b.cpu().numpy()
    x = _tile(pool_a, batch)
    x0 = x.clone()
    y = _tile(pool_b, batch)
    g.api.ntt_fwd(x, t)
    g.api.ntt_fwd(y, t)
    assert bool((x.view(torch.int64) < qcol).all()), (log_n, L, batch)
    rows = sorted({(0, 0), (batch // 2, L // 2), (batch - 1, L - 1)})
    xh = x.cpu().numpy()
    for b, l in rows:
        q, p = int(qs[l]), int(ps[l])
        assert np.array_equal(xh[b, l], oracle.ntt(host_a[b % 2, l], q, p)), (log_n, L, batch, b, l)
    g.api.mul_ntt(x, x, y, t)
    g.api.ntt_inv(x, t)
    xh = x.cpu().numpy()
    for b, l in rows:
        q, p = int(qs[l]), int(ps[l])
        want = oracle.intt(oracle.mul_batch(oracle.ntt(host_a[b % 2, l], q, p)[None, None],
                                            oracle.ntt(host_b[b % 2, l], q, p)[None, None], [q])[0, 0], q, p)
        assert np.array_equal(xh[b, l], want), (log_n, L, batch, b, l)
    g.api.ntt_fwd(x0, t)                              # round trip on every row, on the device
    g.api.ntt_inv(x0, t)
    assert g.same_bits(x0, _tile(pool_a, batch)), (log_n, L, batch)


@pytest.mark.parametrize("log_n", list(range(11, 18)))
def test_sweep_point_parity(g, log_n):
    import torch
    n = 1 << log_n
    for L in LS:
        qs = g.primes(log_n, L)
        t = g.tables(log_n, qs)
        ps = oracle.psis(qs, n)
        qcol = torch.tensor([int(q) for q in qs], dtype=torch.int64, device="cuda").view(1, L, 1)
        for batch in BATCHES:
            if batch * L * n * 8 <= FULL_BYTES:
                _full_point(g, t, qs, ps, qcol, log_n, L, batch)
            else:
                _sampled_point(g, t, qs, ps, qcol, log_n, L, batch)
            torch.cuda.empty_cache()
