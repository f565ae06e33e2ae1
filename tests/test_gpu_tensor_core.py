"""GPU parity of the tensor-core basis extensions on inputs that exercise
their exact fallback.

ModUp (digits of <= 8 primes) and the NTT-domain ModDown conversion (<= 8
primes of P) run on the tensor cores with a correction count e taken from a
fixed-point sum; where that sum lies within a few units of an integer -- the
coefficient's CRT value X is near 0 or near the basis product D, i.e. a small
signed integer -- the lane computes e exactly from Garner's digits and a
redundant modulus.  Uniform inputs almost never take that branch, so here the
coefficients are small signed integers (every lane takes it) or a mix of small
and uniform ones (some lanes of a warp take it).  Every output is compared with
the oracle, and the device status word must stay 0 (no tensor-core wait gave up).
"""
import numpy as np
import pytest

import oracle
from ntt_arithmetic_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import gpu_util
    return gpu_util


def small_signed(shape, qs, seed, bound=1 << 20, mix=False):
    """Residues of small signed integers c (|c| < bound), the same c in every limb; with mix=True every
    other run of 16 coefficients is uniform instead."""
    rng = np.random.default_rng(seed)
    c = rng.integers(-bound, bound, size=shape[:-2] + (shape[-1],))
    c[..., :4] = [0, 1, -1, bound - 1]
    x = np.empty(shape, dtype=np.uint64)
    for l, q in enumerate(qs):
        x[..., l, :] = np.where(c >= 0, c, c + int(q)).astype(np.uint64)
    if mix:
        u = inputs.uniform_residues(shape, qs, seed, buffer=3)
        sel = (np.arange(shape[-1]) // 16) % 2 == 1
        x[..., sel] = u[..., sel]
    return x


@pytest.mark.parametrize("mix", [False, True])
@pytest.mark.parametrize("approx", [False, True])
def test_keyswitch_small_coefficients(g, mix, approx):
    import torch
    log_n, L, K, dnum, batch = 12, 24, 8, 3, 2
    n = 1 << log_n
    qp = g.qp_basis(log_n, L, K)
    t = g.tables(log_n, tuple(qp))
    mt = g.api.ModupTables(L, K, dnum, qp)
    x = small_signed((batch, L, n), qp[:L], 71, mix=mix)
    keys = inputs.uniform_residues((dnum, 2, L + K, n), qp, 72, buffer=1)
    g.api.device_status()
    out = torch.empty((batch, 2, L + K, n), dtype=torch.uint64, device="cuda")
    g.api.keyswitch_ip(out, g.dev(x), g.dev(keys), L, K, dnum, t, mt, approx=approx)
    want = oracle.keyswitch_batch(x, keys, qp, oracle.psis(qp, n), L, K, dnum, approx=approx)
    assert np.array_equal(g.host(out), want)
    assert g.api.device_status() == 0


@pytest.mark.parametrize("log_n,L,K,dnum", [(14, 7, 3, 3), (11, 5, 1, 1), (13, 16, 4, 2)])
def test_modup_digits_small_coefficients(g, log_n, L, K, dnum):
    """The extended digits themselves (decompose: ModUp + NTT over Q u P) on ragged digit shapes, one target
    per digit, and two digits of 8 primes."""
    import torch
    n = 1 << log_n
    qp = g.qp_basis(log_n, L, K)
    t = g.tables(log_n, tuple(qp))
    mt = g.api.ModupTables(L, K, dnum, qp)
    x = small_signed((2, L, n), qp[:L], 73 + log_n, mix=True)
    digits = torch.empty((2, dnum, L + K, n), dtype=torch.uint64, device="cuda")
    g.api.keyswitch_decompose(digits, g.dev(x), L, K, dnum, t, mt)
    ext = oracle.modup_batch(x, np.array(qp, dtype=np.uint64), L, K, dnum)
    want = oracle.ntt_batch(ext.reshape(2 * dnum, L + K, n), qp, oracle.psis(qp, n)).reshape(ext.shape)
    assert np.array_equal(g.host(digits), want)
    assert g.api.device_status() == 0


@pytest.mark.parametrize("nearest", [True, False])
@pytest.mark.parametrize("mix", [False, True])
def test_moddown_ntt_small_coefficients(g, nearest, mix):
    """NTT-domain ModDown of the NTT of small signed coefficients: X is small, so with truncation the
    conversion's X + h = X is near 0 or near P in every lane (the fallback), with nearest rounding it is
    near P / 2."""
    import torch
    log_n, L, K, batch = 13, 24, 8, 3
    n = 1 << log_n
    qp = g.qp_basis(log_n, L, K)
    t = g.tables(log_n, tuple(qp))
    md = g.api.ModdownTables(L, K, qp)
    ps = oracle.psis(qp, n)
    c = small_signed((batch, L + K, n), qp, 74, mix=mix)
    x = oracle.ntt_batch(c, qp, ps)
    out = torch.empty((batch, L, n), dtype=torch.uint64, device="cuda")
    g.api.moddown(out, g.dev(x), L, K, t, md, domain="ntt", nearest=nearest)
    assert np.array_equal(g.host(out), oracle.moddown_ntt_batch(x, qp, ps, L, K, nearest))
    assert g.api.device_status() == 0


def test_tensor_core_wait_gives_up_without_fault(g, monkeypatch):
    """The bounded-wait path, taken on purpose: with FHE_TC_TEST_TIMEOUT=1 the tensor-core kernels wait
    for 1 ms on a barrier nothing arrives on, give up, set FHE_STATUS_TC_TIMEOUT, let their committed MMA
    finish, free their tensor memory and return.  The status word reports it, and the same context then
    computes the exact result again."""
    import torch
    log_n, L, K, dnum, batch = 12, 24, 8, 3, 1
    n = 1 << log_n
    qp = g.qp_basis(log_n, L, K)
    t = g.tables(log_n, tuple(qp))
    mt = g.api.ModupTables(L, K, dnum, qp)
    md = g.api.ModdownTables(L, K, qp)
    x = inputs.uniform_residues((batch, L, n), qp[:L], 91, buffer=0)
    keys = inputs.uniform_residues((dnum, 2, L + K, n), qp, 91, buffer=1)
    dx, dk = g.dev(x), g.dev(keys)
    out = torch.empty((batch, 2, L + K, n), dtype=torch.uint64, device="cuda")
    down = torch.empty((2 * batch, L, n), dtype=torch.uint64, device="cuda")
    assert g.api.device_status() == 0
    monkeypatch.setenv("FHE_TC_TEST_TIMEOUT", "1")
    g.api.keyswitch_ip(out, dx, dk, L, K, dnum, t, mt)
    assert g.api.device_status() == g.api.N.FHE_STATUS_TC_TIMEOUT     # read and cleared
    g.api.moddown(down, out.view(2 * batch, L + K, n), L, K, t, md, domain="ntt")
    assert g.api.device_status() == g.api.N.FHE_STATUS_TC_TIMEOUT
    monkeypatch.delenv("FHE_TC_TEST_TIMEOUT")
    g.api.keyswitch_ip(out, dx, dk, L, K, dnum, t, mt)
    want = oracle.keyswitch_batch(x, keys, qp, oracle.psis(qp, n), L, K, dnum)
    assert np.array_equal(g.host(out), want)
    assert g.api.device_status() == 0


@pytest.mark.parametrize("log_n", [7, 8, 9])
def test_tensor_core_smallest_rings(g, log_n):
    """The tensor-core kernels from their smallest ring (n = 128: one tile per item, a grid of a few CTAs):
    key switch (exact and approximate) and NTT-domain ModDown against the oracle."""
    import torch
    L, K, dnum, batch = 5, 2, 2, 3
    n = 1 << log_n
    qp = g.qp_basis(log_n, L, K)
    t = g.tables(log_n, tuple(qp))
    mt = g.api.ModupTables(L, K, dnum, qp)
    md = g.api.ModdownTables(L, K, qp)
    ps = oracle.psis(qp, n)
    x = small_signed((batch, L, n), qp[:L], 95 + log_n, bound=1 << 30, mix=True)
    keys = inputs.uniform_residues((dnum, 2, L + K, n), qp, 96 + log_n, buffer=1)
    out = torch.empty((batch, 2, L + K, n), dtype=torch.uint64, device="cuda")
    for approx in (False, True):
        g.api.keyswitch_ip(out, g.dev(x), g.dev(keys), L, K, dnum, t, mt, approx=approx)
        assert np.array_equal(g.host(out), oracle.keyswitch_batch(x, keys, qp, ps, L, K, dnum, approx=approx))
    xs = inputs.uniform_residues((batch, L + K, n), qp, 97 + log_n)
    down = torch.empty((batch, L, n), dtype=torch.uint64, device="cuda")
    for nearest in (True, False):
        g.api.moddown(down, g.dev(xs), L, K, t, md, domain="ntt", nearest=nearest)
        assert np.array_equal(g.host(down), oracle.moddown_ntt_batch(xs, qp, ps, L, K, nearest))
    assert g.api.device_status() == 0
