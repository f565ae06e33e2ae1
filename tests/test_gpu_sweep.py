"""GPU parity over the sweep workload: n in {2^11 .. 2^17}, L in {1, 8, 24,
64}, batch in {1, 16, 64} (84 points, up to 4 GiB per operand), for the
forward NTT, the inverse NTT and the fused pointwise product.

At these sizes the oracle checks sampled rows (first, middle and last (batch,
limb) row of each point) element by element; properties that hold at any
size are checked on every row on the device: INTT(NTT(x)) == x and every
output residue below its modulus.  Inputs are seeded uniform residues; to
bound host time, a point's batch is a device-side tiling of a seeded pool of
up to 2 distinct batch items (every limb row of the pool is distinct).
"""
import numpy as np
import pytest

import oracle
from ntt_arithmetic_gb300 import inputs

pytestmark = pytest.mark.gpu

LS = [1, 8, 24, 64]
BATCHES = [1, 16, 64]


@pytest.fixture(scope="module")
def g():
    import gpu_util
    return gpu_util


def _tile(pool, batch):
    import torch
    reps = (batch + pool.shape[0] - 1) // pool.shape[0]
    return pool.repeat(reps, 1, 1)[:batch].contiguous()


@pytest.mark.parametrize("log_n", list(range(11, 18)))
def test_sweep_point_parity(g, log_n):
    import torch
    n = 1 << log_n
    for L in LS:
        qs = g.primes(log_n, L)
        t = g.tables(log_n, qs)
        ps = oracle.psis(qs, n)
        qcol = torch.tensor([int(q) for q in qs], dtype=torch.int64, device="cuda").view(1, L, 1)
        pool_a = g.dev(inputs.uniform_residues((2, L, n), qs, 5000 + log_n, buffer=L))
        pool_b = g.dev(inputs.uniform_residues((2, L, n), qs, 6000 + log_n, buffer=L))
        host_a = pool_a.cpu().numpy()
        host_b = pool_b.cpu().numpy()
        for batch in BATCHES:
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
            g.api.mul_ntt(x, x, y, t)                    # fused pointwise product in the NTT domain
            g.api.ntt_inv(x, t)
            xh = x.cpu().numpy()
            for b, l in rows:
                q, p = int(qs[l]), int(ps[l])
                want = oracle.intt(oracle.mul_batch(oracle.ntt(host_a[b % 2, l], q, p)[None, None],
                                                    oracle.ntt(host_b[b % 2, l], q, p)[None, None], [q])[0, 0], q, p)
                assert np.array_equal(xh[b, l], want), (log_n, L, batch, b, l)
            # round trip on every row, on the device
            g.api.ntt_fwd(x0, t)
            g.api.ntt_inv(x0, t)
            assert g.same_bits(x0, _tile(pool_a, batch)), (log_n, L, batch)
            del x, x0, y
        torch.cuda.empty_cache()
