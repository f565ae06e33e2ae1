"""GPU parity of ModDown (QP -> Q) and rescale against the oracle.

out_l = floor((X + h) / P) mod q_l with h = (P-1)/2 (nearest) or 0
(truncating), in the coefficient and the NTT domain, element by element
against ``oracle.moddown_batch`` / ``oracle.moddown_ntt_batch``: the key-switch
basis of the n=2^16 workload (24 + 8 primes), rescale (K = 1) of the 24-prime
chain, every Garner width the kernel instantiates (K = 1, 2, 3, 4, 8, 16),
small and ragged shapes, inputs at the extremes, and the argument checks.
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


def _run(g, x, L, K, qp, domain, nearest):
    import torch
    n = x.shape[-1]
    log_n = n.bit_length() - 1
    t = g.tables(log_n, tuple(qp))
    md = g.api.ModdownTables(L, K, qp)
    out = torch.empty((x.shape[0], L, n), dtype=torch.uint64, device="cuda")
    g.api.moddown(out, g.dev(x), L, K, t, md, domain=domain, nearest=nearest)
    return g.host(out)


def _want(x, qp, L, K, domain, nearest):
    if domain == "coeff":
        return oracle.moddown_batch(x, qp, L, K, nearest)
    n = x.shape[-1]
    return oracle.moddown_ntt_batch(x, qp, oracle.psis(qp, n), L, K, nearest)


@pytest.mark.parametrize("domain", ["coeff", "ntt"])
@pytest.mark.parametrize("nearest", [True, False])
def test_moddown_keyswitch_basis(g, domain, nearest):
    """n = 2^16, Q = 24 primes, P = 8 primes (the key-switch basis), batch 2."""
    log_n, L, K, batch = 16, 24, 8, 2
    qp = g.qp_basis(log_n, L, K)
    x = inputs.uniform_residues((batch, L + K, 1 << log_n), qp, 700 + nearest, buffer=1)
    got = _run(g, x, L, K, qp, domain, nearest)
    assert np.array_equal(got, _want(x, qp, L, K, domain, nearest))


@pytest.mark.parametrize("domain", ["coeff", "ntt"])
@pytest.mark.parametrize("nearest", [True, False])
def test_rescale_chain(g, domain, nearest):
    """Rescale drops the last of 24 primes (n = 2^16, batch 2 ciphertext halves)."""
    import torch
    log_n, L, batch = 16, 24, 2
    n = 1 << log_n
    q = list(g.primes(log_n, L))
    t = g.tables(log_n, tuple(q))
    rs = g.api.ModdownTables(L - 1, 1, q)
    x = inputs.uniform_residues((batch, L, n), q, 710 + nearest, buffer=1)
    out = torch.empty((batch, L - 1, n), dtype=torch.uint64, device="cuda")
    g.api.rescale(out, g.dev(x), t, rs, domain=domain, nearest=nearest)
    assert np.array_equal(g.host(out), _want(x, q, L - 1, 1, domain, nearest))


@pytest.mark.parametrize("log_n,L,K,batch", [(11, 7, 3, 3), (12, 5, 16, 2), (10, 9, 2, 5), (13, 3, 4, 1),
                                             (1, 2, 1, 3), (4, 1, 16, 2), (17, 2, 8, 1), (14, 5, 3, 3),
                                             (15, 4, 2, 2)])
@pytest.mark.parametrize("domain", ["coeff", "ntt"])
def test_moddown_shapes(g, log_n, L, K, batch, domain):
    qp = g.qp_basis(log_n, L, K)
    x = inputs.uniform_residues((batch, L + K, 1 << log_n), qp, 720 + log_n + K, buffer=1)
    for nearest in (True, False):
        got = _run(g, x, L, K, qp, domain, nearest)
        assert np.array_equal(got, _want(x, qp, L, K, domain, nearest)), (log_n, L, K, batch, nearest)


def test_moddown_extremes(g):
    """All residues 0, all q-1 / p-1, and X = m P + r for known m and r."""
    log_n, L, K = 11, 6, 4
    n = 1 << log_n
    qp = g.qp_basis(log_n, L, K)
    col = np.array(qp, dtype=np.uint64)[:, None]
    zero = np.zeros((1, L + K, n), dtype=np.uint64)
    top = np.broadcast_to(col - 1, (1, L + K, n)).copy()
    for x in (zero, top):
        for nearest in (True, False):
            assert np.array_equal(_run(g, x, L, K, qp, "coeff", nearest),
                                  oracle.moddown_batch(x, qp, L, K, nearest))
    # X = m P + r: truncation gives m; nearest gives m + (r > (P-1)/2)
    P = 1
    for p in qp[L:]:
        P *= int(p)
    rng = np.random.default_rng(9)
    ms = [int(v) for v in rng.integers(0, 1 << 62, size=n)]
    rs = [0, 1, (P - 1) // 2, (P + 1) // 2, P - 1] + [int(v) % P for v in rng.integers(0, 1 << 63, size=n - 5)]
    x = np.array([[[(m * P + r) % int(p) for m, r in zip(ms, rs)] for p in qp]], dtype=np.uint64)
    trunc = _run(g, x, L, K, qp, "coeff", False)
    near = _run(g, x, L, K, qp, "coeff", True)
    for l in range(L):
        q = int(qp[l])
        assert [int(v) for v in trunc[0, l]] == [m % q for m in ms]
        assert [int(v) for v in near[0, l]] == [(m + (2 * r > P - 1)) % q for m, r in zip(ms, rs)]


def test_moddown_arguments(g):
    import torch
    log_n, L, K, batch = 10, 4, 2, 2
    n = 1 << log_n
    qp = g.qp_basis(log_n, L, K)
    t = g.tables(log_n, tuple(qp))
    md = g.api.ModdownTables(L, K, qp)
    x = g.dev(inputs.uniform_residues((batch, L + K, n), qp, 730, buffer=1))
    out = torch.empty((batch, L, n), dtype=torch.uint64, device="cuda")
    need = g.api.moddown_workspace_bytes(log_n, L, K, batch)
    assert need == batch * (L + K) * n * 8
    from ntt_arithmetic_gb300 import _native as N

    def status(fn):
        with pytest.raises(N.FheError) as e:
            fn()
        return e.value.status

    small = torch.empty(need // 8 - 2, dtype=torch.uint64, device="cuda")
    assert status(lambda: g.api.moddown(out, x, L, K, t, md, workspace=small)) == N.FHE_ESPACE
    alias_out = x.view(-1)[: batch * L * n].view(batch, L, n)
    assert status(lambda: g.api.moddown(alias_out, x, L, K, t, md)) == N.FHE_EALIAS
    ws = torch.empty(need // 8, dtype=torch.uint64, device="cuda")
    x_in_ws = ws[: batch * (L + K) * n].view(batch, L + K, n)
    assert status(lambda: g.api.moddown(out, x_in_ws, L, K, t, md, workspace=ws)) == N.FHE_EALIAS

    def raw(k=K, rounding=1, tables=t):
        N.call("fhe_moddown", out.data_ptr(), x.data_ptr(), log_n, L, k, batch, 1, rounding, tables.ref(),
               md.blob.data_ptr(), ws.data_ptr(), need, None)

    for bad_k in (0, 17):
        assert status(lambda: raw(k=bad_k)) == N.FHE_EINVAL
    assert status(lambda: raw(rounding=2)) == N.FHE_EINVAL
    t_short = g.tables(log_n, tuple(qp[:L]))          # covers fewer than L + K primes
    assert status(lambda: raw(tables=t_short)) == N.FHE_EINVAL
    raw()                                              # the same call with valid arguments succeeds


def test_moddown_launch_count(g):
    """Coefficient domain: one fused pass; NTT domain: copy of the P limbs,
    inverse NTT, conversion, forward NTT over Q and the final product (for
    n >= 2^14 without the copy, and the last two in one kernel's block
    stages)."""
    import torch
    log_n, L, K, batch = 12, 4, 2, 1
    n = 1 << log_n
    qp = g.qp_basis(log_n, L, K)
    t = g.tables(log_n, tuple(qp))
    md = g.api.ModdownTables(L, K, qp)
    x = g.dev(inputs.uniform_residues((batch, L + K, n), qp, 740, buffer=1))
    out = torch.empty((batch, L, n), dtype=torch.uint64, device="cuda")
    c0 = g.api.launch_count()
    g.api.moddown(out, x, L, K, t, md, domain="coeff")
    c1 = g.api.launch_count()
    g.api.moddown(out, x, L, K, t, md, domain="ntt")
    c2 = g.api.launch_count()
    assert c1 - c0 == 1
    assert c2 - c1 == 5
    # n >= 2^14: the inverse NTT's block kernel reads the P limbs from the input (no copy) and the forward
    # NTT's block stages carry the final product (inverse NTT in two launches, conversion, column stages,
    # block stages + product)
    log_n = 14
    n = 1 << log_n
    qp = g.qp_basis(log_n, L, K)
    t = g.tables(log_n, tuple(qp))
    md = g.api.ModdownTables(L, K, qp)
    xh = inputs.uniform_residues((batch, L + K, n), qp, 741, buffer=1)
    out = torch.empty((batch, L, n), dtype=torch.uint64, device="cuda")
    c0 = g.api.launch_count()
    g.api.moddown(out, g.dev(xh), L, K, t, md, domain="ntt")
    assert g.api.launch_count() - c0 == 5
    assert np.array_equal(g.host(out), _want(xh, qp, L, K, "ntt", True))


@pytest.mark.parametrize("domain", ["coeff", "ntt"])
def test_moddown_long_chain(g, domain):
    """More than 64 Q primes: the conversion reads its weights from global memory
    instead of staging them in shared memory (n = 2^11, 150 + 2 primes, and a
    rescale of a 130-prime chain)."""
    import torch
    log_n, n = 11, 1 << 11
    qp = g.qp_basis(log_n, 150, 2)
    x = inputs.uniform_residues((2, 152, n), qp, 740, buffer=1)
    for nearest in (True, False):
        got = _run(g, x, 150, 2, qp, domain, nearest)
        assert np.array_equal(got, _want(x, qp, 150, 2, domain, nearest)), nearest
    q = list(g.primes(log_n, 130))
    t = g.tables(log_n, tuple(q))
    rs = g.api.ModdownTables(129, 1, q)
    x = inputs.uniform_residues((2, 130, n), q, 741, buffer=1)
    out = torch.empty((2, 129, n), dtype=torch.uint64, device="cuda")
    g.api.rescale(out, g.dev(x), t, rs, domain=domain, nearest=True)
    assert np.array_equal(g.host(out), _want(x, q, 129, 1, domain, True))
