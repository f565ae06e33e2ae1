"""GPU parity: basis conversion / modraise, the approximate-ModUp key switch
and the hoisted key switch, element by element against the oracle."""
import ctypes

import numpy as np
import pytest

import oracle
from ntt_arithmetic_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import gpu_util
    return gpu_util


def _bconv(g, x, src, dst, approx):
    import torch
    t = g.api.BconvTables(src, dst)
    out = torch.empty((x.shape[0], len(dst), x.shape[-1]), dtype=torch.uint64, device="cuda")
    g.api.bconv(out, g.dev(x), t, approx=approx)
    return g.host(out)


@pytest.mark.parametrize("log_n,S,T,batch", [(16, 1, 24, 2), (16, 3, 24, 2), (12, 8, 40, 3), (10, 16, 20, 2),
                                             (1, 2, 5, 3), (13, 5, 64, 1), (11, 4, 2100, 2)])
@pytest.mark.parametrize("approx", [False, True])
def test_bconv_vs_oracle(g, log_n, S, T, batch, approx):
    """Modraise shape: sources = the first S primes of a T-prime chain."""
    n = 1 << log_n
    chain = list(g.primes(log_n, T))
    x = inputs.uniform_residues((batch, S, n), chain[:S], 800 + log_n + S, buffer=1)
    got = _bconv(g, x, chain[:S], chain, approx)
    assert np.array_equal(got[:, :S], x)                      # source limbs reproduce the input
    assert np.array_equal(got, oracle.bconv_batch(x, chain[:S], chain, approx=approx))


def test_bconv_disjoint_targets_and_extremes(g):
    log_n, S = 11, 6
    n = 1 << log_n
    chain = g.qp_basis(log_n, S, 10)
    src, dst = chain[:S], chain[S:]
    col = np.array(src, dtype=np.uint64)[:, None]
    for x in (np.zeros((1, S, n), dtype=np.uint64), np.broadcast_to(col - 1, (1, S, n)).copy(),
              inputs.uniform_residues((2, S, n), src, 812, buffer=1)):
        for approx in (False, True):
            assert np.array_equal(_bconv(g, x, src, dst, approx), oracle.bconv_batch(x, src, dst, approx=approx))


def test_bconv_arguments(g):
    import torch
    from ntt_arithmetic_gb300 import _native as N
    log_n, S, T = 10, 2, 6
    n = 1 << log_n
    chain = list(g.primes(log_n, T))
    t = g.api.BconvTables(chain[:S], chain)
    x = g.dev(inputs.uniform_residues((1, S, n), chain[:S], 813, buffer=1))
    out = torch.empty((1, T, n), dtype=torch.uint64, device="cuda")

    def st(*a):
        with pytest.raises(N.FheError) as e:
            N.call("fhe_bconv", *a)
        return e.value.status

    P = lambda v: v.data_ptr()
    assert st(P(out), P(x), log_n, 0, T, 1, 0, P(t.blob), None) == N.FHE_EINVAL          # S = 0
    assert st(P(out), P(x), log_n, 17, T, 1, 0, P(t.blob), None) == N.FHE_EINVAL         # S > 16
    assert st(P(out), P(x), log_n, S, T, 1, 2, P(t.blob), None) == N.FHE_EINVAL          # mode
    assert st(P(out), P(out), log_n, S, T, 1, 0, P(t.blob), None) == N.FHE_EALIAS        # in inside out
    host = np.zeros(16, dtype=np.uint64)
    assert st(P(out), host.ctypes.data, log_n, S, T, 1, 0, P(t.blob), None) == N.FHE_EDEVICE
    with pytest.raises(N.FheError):                                                     # not prime / repeated
        g.api.BconvTables([chain[0], chain[0]], chain)
    N.call("fhe_bconv", P(out), P(x), log_n, S, T, 1, 0, P(t.blob), None)


# ------------------------------------------------------ approximate ModUp --

@pytest.mark.parametrize("log_n,L,K,dnum,batch", [(16, 24, 8, 3, 1), (11, 7, 3, 3, 2), (12, 16, 4, 2, 2),
                                                  (10, 5, 5, 5, 1)])
def test_keyswitch_approx_vs_oracle(g, log_n, L, K, dnum, batch):
    import torch
    n = 1 << log_n
    qp = g.qp_basis(log_n, L, K)
    t = g.tables(log_n, tuple(qp))
    mt = g.api.ModupTables(L, K, dnum, qp)
    ps = oracle.psis(qp, n)
    x = inputs.uniform_residues((batch, L, n), qp[:L], 820 + log_n, buffer=0)
    keys = inputs.uniform_residues((dnum, 2, L + K, n), qp, 821 + log_n, buffer=1)
    out = torch.empty((batch, 2, L + K, n), dtype=torch.uint64, device="cuda")
    g.api.keyswitch_ip(out, g.dev(x), g.dev(keys), L, K, dnum, t, mt, approx=True)
    want = oracle.keyswitch_batch(x, keys, qp, ps, L, K, dnum, approx=True)
    assert np.array_equal(g.host(out), want)
    if (L + dnum - 1) // dnum > 1:                # one-prime digits convert exactly either way
        exact = oracle.keyswitch_batch(x, keys, qp, ps, L, K, dnum)
        assert not np.array_equal(want, exact)   # the variant really differs


# ------------------------------------------------------- hoisted rotations --

def _hoisted_case(g, log_n, L, K, dnum, batch, ks, approx, seed):
    import torch
    n = 1 << log_n
    qp = g.qp_basis(log_n, L, K)
    t = g.tables(log_n, tuple(qp))
    mt = g.api.ModupTables(L, K, dnum, qp)
    ps = oracle.psis(qp, n)
    R = len(ks)
    x = inputs.uniform_residues((batch, L, n), qp[:L], seed, buffer=0)
    keys = inputs.uniform_residues((R * dnum * 2, L + K, n), qp, seed + 1, buffer=1).reshape(R, dnum, 2, L + K, n)
    out = torch.empty((R, batch, 2, L + K, n), dtype=torch.uint64, device="cuda")
    g.api.keyswitch_hoisted(out, g.dev(x), g.dev(keys), ks, L, K, dnum, t, mt, approx=approx)
    return g.host(out), oracle.keyswitch_hoisted_batch(x, keys, ks, qp, ps, L, K, dnum, approx=approx)


@pytest.mark.parametrize("log_n,L,K,dnum,batch,R", [(12, 8, 4, 2, 2, 4), (11, 24, 2, 24, 1, 3), (6, 3, 2, 3, 2, 64),
                                                    (1, 2, 1, 2, 2, 2), (13, 10, 3, 4, 3, 5), (10, 4, 2, 1, 2, 3)])
@pytest.mark.parametrize("approx", [False, True])
def test_hoisted_vs_oracle(g, log_n, L, K, dnum, batch, R, approx):
    two_n = 2 << log_n
    # powers of 5 (rotations) and their negatives (rotation composed with conjugation), all odd
    ks = [pow(5, r + 1, two_n) if r % 3 else two_n - pow(5, r + 1, two_n) for r in range(R)]
    got, want = _hoisted_case(g, log_n, L, K, dnum, batch, ks, approx, 830 + log_n + R)
    assert np.array_equal(got, want)


def test_hoisted_full_basis(g):
    """n = 2^16, 24 + 8 primes, dnum = 3: the coeff_to_slot rotations
    k = 5^(2^r) for r < 4 plus the conjugation 2n - 1."""
    n = 1 << 16
    ks = [pow(5, 1 << r, 2 * n) for r in range(4)] + [2 * n - 1]
    got, want = _hoisted_case(g, 16, 24, 8, 3, 1, ks, False, 840)
    assert np.array_equal(got, want)


def test_hoisted_arguments_and_launches(g):
    import torch
    from ntt_arithmetic_gb300 import _native as N
    log_n, L, K, dnum, batch = 10, 4, 2, 2, 1
    n = 1 << log_n
    qp = g.qp_basis(log_n, L, K)
    t = g.tables(log_n, tuple(qp))
    mt = g.api.ModupTables(L, K, dnum, qp)
    x = g.dev(inputs.uniform_residues((batch, L, n), qp[:L], 850, buffer=0))
    keys = torch.zeros((65, dnum, 2, L + K, n), dtype=torch.uint64, device="cuda")
    out = torch.empty((65, batch, 2, L + K, n), dtype=torch.uint64, device="cuda")

    def st(ks, kk=None, oo=None):
        R = len(ks)
        with pytest.raises(N.FheError) as e:
            g.api.keyswitch_hoisted(oo if oo is not None else out[:R], x, kk if kk is not None else keys[:R], ks,
                                    L, K, dnum, t, mt)
        return e.value.status

    assert st([5, 4]) == N.FHE_EINVAL                 # even element
    assert st([5, 2 * n + 1]) == N.FHE_EINVAL         # not below 2n
    assert st(list(range(1, 131, 2))) == N.FHE_EINVAL  # R = 65 > 64
    ws = torch.empty(g.api.keyswitch_workspace_bytes(log_n, L, K, dnum, batch) // 8, dtype=torch.uint64,
                     device="cuda")
    gal_dev = torch.tensor([5, 25], dtype=torch.int32, device="cuda")
    with pytest.raises(N.FheError) as e:
        N.call("fhe_keyswitch_hoisted", out.data_ptr(), x.data_ptr(), 0, keys.data_ptr(),
               ctypes.cast(gal_dev.data_ptr(), ctypes.POINTER(ctypes.c_uint32)), 2, log_n, L, K, dnum, batch, 0,
               t.ref(), mt.blob.data_ptr(), ws.data_ptr(), ws.numel() * 8, None)
    assert e.value.status == N.FHE_EDEVICE
    c0 = g.api.launch_count()
    g.api.keyswitch_hoisted(out[:3], x, keys[:3], [1, 5, 25], L, K, dnum, t, mt)
    assert g.api.launch_count() - c0 == 3             # ModUp, NTT of the digits, fused automorphism + IP


def test_decompose_apply_equal_the_one_call_forms(g):
    import torch
    log_n, L, K, dnum, batch = 12, 8, 4, 3, 2
    n = 1 << log_n
    qp = g.qp_basis(log_n, L, K)
    t = g.tables(log_n, tuple(qp))
    mt = g.api.ModupTables(L, K, dnum, qp)
    x = g.dev(inputs.uniform_residues((batch, L, n), qp[:L], 860, buffer=0))
    keys = g.dev(inputs.uniform_residues((3 * dnum * 2, L + K, n), qp, 861, buffer=1)).view(3, dnum, 2, L + K, n)
    ks = [5, 25, 2 * n - 1]
    for approx in (False, True):
        digits = torch.empty((batch, dnum, L + K, n), dtype=torch.uint64, device="cuda")
        g.api.keyswitch_decompose(digits, x, L, K, dnum, t, mt, approx=approx)
        one = torch.empty((batch, 2, L + K, n), dtype=torch.uint64, device="cuda")
        g.api.keyswitch_apply(one, digits, keys[0], L, K, dnum, t)
        ref = torch.empty_like(one)
        g.api.keyswitch_ip(ref, x, keys[0], L, K, dnum, t, mt, approx=approx)
        assert g.same_bits(one, ref)
        rot = torch.empty((3, batch, 2, L + K, n), dtype=torch.uint64, device="cuda")
        g.api.keyswitch_apply(rot, digits, keys, L, K, dnum, t, galois=ks)
        ref = torch.empty_like(rot)
        g.api.keyswitch_hoisted(ref, x, keys, ks, L, K, dnum, t, mt, approx=approx)
        assert g.same_bits(rot, ref)
