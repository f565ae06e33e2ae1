"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle,
element by element, bit-exact, on seeded inputs.

Sizes span several tiles and ragged tails (batch * L not a multiple of
anything, every n from 2 to 2^17), the full n = 2^16 / L = 24 / batch 16
workload, the n = 2048 / L = 112 tensor-product workload, the PR1 reference
case against the schoolbook product, and the hybrid key switch at n = 2^16.
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


def assert_reduced(x: np.ndarray, qs):
    qcol = np.array([int(q) for q in qs], dtype=np.uint64).reshape((len(qs), 1))
    assert (x.reshape(-1, len(qs), x.shape[-1]) < qcol).all()


@pytest.mark.parametrize("log_n", list(range(1, 18)))
def test_ntt_fwd_inv_every_size(g, log_n):
    """Ragged batch x L (3 x 5 rows) at every supported n."""
    n = 1 << log_n
    L, batch = 5, 3
    qs = g.primes(log_n, L)
    t = g.tables(log_n, qs)
    ps = oracle.psis(qs, n)
    x = inputs.uniform_residues((batch, L, n), qs, 100 + log_n)
    d = g.dev(x)
    g.api.ntt_fwd(d, t)
    got = g.host(d)
    want = oracle.ntt_batch(x, qs, ps)
    assert np.array_equal(got, want)
    g.api.ntt_inv(d, t)
    assert np.array_equal(g.host(d), x)
    # inverse on independent NTT-domain data
    y = inputs.uniform_residues((batch, L, n), qs, 200 + log_n)
    d2 = g.dev(y)
    g.api.ntt_inv(d2, t)
    assert np.array_equal(g.host(d2), oracle.ntt_batch(y, qs, ps, inverse=True))


@pytest.mark.parametrize("log_n", [14, 16, 17])
@pytest.mark.parametrize("batch", [5, 7])
def test_split_ntt_ragged_batch_chunks(g, log_n, batch):
    """The split shapes' column kernels run up to 4 batch items of one prime
    per CTA (5 -> 3 + 2, 7 -> 4 + 3): every row of both chunks, forward and
    inverse, against the oracle."""
    n = 1 << log_n
    L = 3
    qs = g.primes(log_n, L)
    t = g.tables(log_n, qs)
    ps = oracle.psis(qs, n)
    x = inputs.uniform_residues((batch, L, n), qs, 300 + log_n + batch)
    d = g.dev(x)
    g.api.ntt_fwd(d, t)
    assert np.array_equal(g.host(d), oracle.ntt_batch(x, qs, ps))
    y = inputs.uniform_residues((batch, L, n), qs, 400 + log_n + batch)
    d2 = g.dev(y)
    g.api.ntt_inv(d2, t)
    assert np.array_equal(g.host(d2), oracle.ntt_batch(y, qs, ps, inverse=True))


def test_pr1_reference_schoolbook(g):
    """PR1 workload: n=2048, the 4 largest q < 2^50 with q = 1 mod 4096, one
    polynomial pair: NTT, pointwise product, INTT == the O(n^2) negacyclic
    product (the kestrel-llm overview's section-3 proof of its NTT)."""
    log_n, n, L = 11, 2048, 4
    qs = g.primes(log_n, L)
    assert list(qs) == [int(v) for v in oracle.primes(4096, 4)]
    t = g.tables(log_n, qs)
    a = inputs.uniform_residues((1, L, n), qs, 1, buffer=0)
    b = inputs.uniform_residues((1, L, n), qs, 1, buffer=1)
    da, db = g.dev(a), g.dev(b)
    g.api.ntt_fwd(da, t)
    g.api.ntt_fwd(db, t)
    g.api.mul_ntt(da, da, db, t)
    g.api.ntt_inv(da, t)
    got = g.host(da)
    for l, q in enumerate(qs):
        assert np.array_equal(got[0, l], oracle.negacyclic_mul(a[0, l], b[0, l], int(q)))


def test_tensor_product_n2048_L112(g):
    """4 ciphertext pairs (16 polynomials) at n=2048 over 112 primes: forward
    NTT, tensor product, INTT of the 12 outputs; every stage against the
    oracle."""
    log_n, n, L = 11, 2048, 112
    qs = g.primes(log_n, L)
    t = g.tables(log_n, qs)
    ps = oracle.psis(qs, n)
    a = inputs.uniform_residues((4, 2, L, n), qs, 2, buffer=0)
    b = inputs.uniform_residues((4, 2, L, n), qs, 2, buffer=1)
    da, db = g.dev(a), g.dev(b)
    g.api.ntt_fwd(da, t)
    g.api.ntt_fwd(db, t)
    A, Bn = oracle.ntt_batch(a, qs, ps), oracle.ntt_batch(b, qs, ps)
    assert np.array_equal(g.host(da), A) and np.array_equal(g.host(db), Bn)
    import torch
    dd = torch.empty((4, 3, L, n), dtype=torch.uint64, device="cuda")
    g.api.tensor(dd, da, db, t)
    D = oracle.tensor_batch(A, Bn, qs)
    assert np.array_equal(g.host(dd), D)
    g.api.ntt_inv(dd, t)
    assert np.array_equal(g.host(dd), oracle.ntt_batch(D, qs, ps, inverse=True))


def test_ntt_n65536_L24_batch16_full(g):
    """The n=2^16, L=24, batch-16 workload in the bench's launch
    configuration, compared element by element."""
    log_n, n, L = 16, 1 << 16, 24
    qs = g.primes(log_n, L)
    t = g.tables(log_n, qs)
    ps = oracle.psis(qs, n)
    x = inputs.uniform_residues((16, L, n), qs, 3)
    d = g.dev(x)
    g.api.ntt_fwd(d, t)
    X = oracle.ntt_batch(x, qs, ps)
    assert np.array_equal(g.host(d), X)
    g.api.ntt_inv(d, t)
    assert np.array_equal(g.host(d), x)


@pytest.mark.parametrize("domain", ["ntt", "coeff"])
def test_automorph_n65536_all_galois_elements(g, domain):
    """k = 5^r mod 2^17 for r in {1, 2, 4, ..., 2^15}: two sampled rows per k
    against the oracle and sigma_k then sigma_{k^-1} == id on the whole
    [16][24][2^16] tensor; for k = 5^32 mod 2^17 and for the conjugation
    k = 2n - 1, every one of the 384 output rows against the oracle."""
    import torch
    log_n, n, L = 16, 1 << 16, 24
    qs = g.primes(log_n, L)
    t = g.tables(log_n, qs)
    ps = oracle.psis(qs, n)
    x = inputs.uniform_residues((16, L, n), qs, 4)
    d = g.dev(x)
    out = torch.empty_like(d)
    back = torch.empty_like(d)
    rng = np.random.default_rng(9)
    for j in range(16):
        k = pow(5, 1 << j, 2 * n)
        kinv = pow(k, -1, 2 * n)
        g.api.automorph(out, d, k, t, domain=domain)
        got = g.host(out)
        rows = [(int(rng.integers(16)), int(rng.integers(L))) for _ in range(2)]
        for b, l in rows:
            q = int(qs[l])
            if domain == "ntt":
                want = oracle.automorph_ntt(x[b, l], q, int(ps[l]), k)
            else:
                want = oracle.automorph_coeff(x[b, l], q, k)
            assert np.array_equal(got[b, l], want), (k, b, l)
        if j == 5:
            assert np.array_equal(got, oracle.automorph_batch(x, qs, ps, k, domain == "ntt")), k
        g.api.automorph(back, out, kinv, t, domain=domain)
        assert g.same_bits(back, d), k
        if k == 1:
            assert g.same_bits(out, d)
    k = 2 * n - 1
    g.api.automorph(out, d, k, t, domain=domain)
    assert np.array_equal(g.host(out), oracle.automorph_batch(x, qs, ps, k, domain == "ntt")), k


def test_automorph_coeff_full_rows(g):
    """Coefficient-domain automorphism on every row (cheap in the oracle)."""
    import torch
    log_n, n, L = 12, 4096, 7
    qs = g.primes(log_n, L)
    t = g.tables(log_n, qs)
    x = inputs.uniform_residues((3, L, n), qs, 5)
    d = g.dev(x)
    out = torch.empty_like(d)
    for k in [1, 3, 5, 2 * n - 1, 1234567 % (2 * n) | 1]:
        g.api.automorph(out, d, k, t, domain="coeff")
        got = g.host(out)
        for b in range(3):
            for l in range(L):
                assert np.array_equal(got[b, l], oracle.automorph_coeff(x[b, l], int(qs[l]), k))


@pytest.mark.parametrize("log_n,L,K,dnum,batch", [(16, 24, 8, 3, 1), (11, 7, 3, 3, 2), (12, 16, 4, 2, 3),
                                                  (10, 5, 2, 5, 1)])
def test_keyswitch_vs_oracle(g, log_n, L, K, dnum, batch):
    """Hybrid key switch: exact ModUp of each digit, NTT over Q u P, inner
    product with the keys -- the n=2^16 / 24+8 primes / dnum=3 workload and
    ragged shapes (digits of 3, 3, 1 limbs; alpha = 1)."""
    import torch
    n = 1 << log_n
    qp = g.qp_basis(log_n, L, K)
    assert qp == [int(v) for v in oracle.primes(2 * n, L + K)]
    t = g.tables(log_n, tuple(qp))
    mt = g.api.ModupTables(L, K, dnum, qp)
    ps = oracle.psis(qp, n)
    x = inputs.uniform_residues((batch, L, n), qp[:L], 6, buffer=0)
    keys = inputs.uniform_residues((dnum, 2, L + K, n), qp, 6, buffer=1)
    out = torch.empty((batch, 2, L + K, n), dtype=torch.uint64, device="cuda")
    g.api.keyswitch_ip(out, g.dev(x), g.dev(keys), L, K, dnum, t, mt)
    want = oracle.keyswitch_batch(x, keys, qp, ps, L, K, dnum)
    got = g.host(out)
    assert np.array_equal(got, want)
    assert_reduced(got, qp)


@pytest.mark.parametrize("log_n,L,K,dnum,batch", [(14, 7, 3, 3, 3), (15, 8, 2, 2, 2), (17, 4, 2, 4, 1),
                                                  (14, 5, 3, 1, 2), (16, 24, 8, 3, 4)])
def test_keyswitch_fused_ntt_ip(g, log_n, L, K, dnum, batch):
    """For n >= 2^14 and dnum <= 4 the key switch runs the digits' NTT fused
    with the inner product (the block stages of every digit of one (limb,
    block, item) in one CTA, then the products with the keys).  Every output
    row is compared with the oracle, and bit for bit with the unfused path
    (decompose = ModUp + NTT of the digits, then apply = inner product), for
    the exact and the approximate ModUp; ragged digits (3, 3, 1), one- and
    four-digit shapes and the full bench shape (4 ciphertexts, 24 + 8
    primes, dnum = 3).  The call launches 3 kernels: ModUp, the column
    stages, the fused block stages + inner product."""
    import torch
    n = 1 << log_n
    qp = g.qp_basis(log_n, L, K)
    t = g.tables(log_n, tuple(qp))
    mt = g.api.ModupTables(L, K, dnum, qp)
    ps = oracle.psis(qp, n)
    x = inputs.uniform_residues((batch, L, n), qp[:L], 40 + log_n, buffer=0)
    keys = inputs.uniform_residues((dnum, 2, L + K, n), qp, 41 + log_n, buffer=1)
    dx, dk = g.dev(x), g.dev(keys)
    for approx in (False, True):
        out = torch.empty((batch, 2, L + K, n), dtype=torch.uint64, device="cuda")
        c0 = g.api.launch_count()
        g.api.keyswitch_ip(out, dx, dk, L, K, dnum, t, mt, approx=approx)
        assert g.api.launch_count() - c0 == 3
        got = g.host(out)
        assert np.array_equal(got, oracle.keyswitch_batch(x, keys, qp, ps, L, K, dnum, approx=approx)), approx
        assert_reduced(got, qp)
        digits = torch.empty((batch, dnum, L + K, n), dtype=torch.uint64, device="cuda")
        g.api.keyswitch_decompose(digits, dx, L, K, dnum, t, mt, approx=approx)
        split = torch.empty_like(out)
        g.api.keyswitch_apply(split, digits, dk, L, K, dnum, t)
        assert g.same_bits(split, out), approx


def test_pointwise_aliasing_and_extremes(g):
    import torch
    log_n, n, L = 11, 2048, 6
    qs = g.primes(log_n, L)
    t = g.tables(log_n, qs)
    a = inputs.uniform_residues((2, L, n), qs, 7, buffer=0)
    b = inputs.uniform_residues((2, L, n), qs, 7, buffer=1)
    for l in range(L):     # q-1, 0 and 1 in the first coefficients
        a[0, l, :4] = [qs[l] - 1, 0, 1, qs[l] - 1]
        b[0, l, :4] = [qs[l] - 1, qs[l] - 1, qs[l] - 1, 0]
    want = oracle.mul_batch(a, b, qs)
    da, db = g.dev(a), g.dev(b)
    out = torch.empty_like(da)
    g.api.mul_ntt(out, da, db, t)
    assert np.array_equal(g.host(out), want)
    g.api.mul_ntt(da, da, db, t)           # out aliases a
    assert np.array_equal(g.host(da), want)
    da = g.dev(a)
    g.api.mul_ntt(db, da, db, t)           # out aliases b
    assert np.array_equal(g.host(db), want)
    with pytest.raises(Exception):
        g.api.mul_ntt(out[:, :, 2:].contiguous(), da, da, t)  # shape mismatch


def test_extreme_values_through_ntt(g):
    """All-zero, all-(q-1) and single-spike rows through NTT / INTT."""
    log_n, n, L = 16, 1 << 16, 3
    qs = g.primes(log_n, L)
    t = g.tables(log_n, qs)
    ps = oracle.psis(qs, n)
    x = np.zeros((3, L, n), dtype=np.uint64)
    for l in range(L):
        x[1, l, :] = qs[l] - 1
        x[2, l, 12345] = qs[l] - 1
    d = g.dev(x)
    g.api.ntt_fwd(d, t)
    assert np.array_equal(g.host(d), oracle.ntt_batch(x, qs, ps))
    g.api.ntt_inv(d, t)
    assert np.array_equal(g.host(d), x)


def test_limb_subset_of_tables(g):
    """A call with L smaller than the tables' L uses limbs [0, L)."""
    log_n, n = 13, 8192
    qs = g.primes(log_n, 9)
    t = g.tables(log_n, qs)
    ps = oracle.psis(qs[:4], n)
    x = inputs.uniform_residues((2, 4, n), qs[:4], 8)
    d = g.dev(x)
    g.api.ntt_fwd(d, t)
    assert np.array_equal(g.host(d), oracle.ntt_batch(x, qs[:4], ps))


def test_launch_counter_counts_kernels(g):
    log_n, n, L = 12, 4096, 2
    qs = g.primes(log_n, L)
    t = g.tables(log_n, qs)
    d = g.dev(inputs.uniform_residues((1, L, n), qs, 9))
    c0 = g.api.launch_count()
    g.api.ntt_fwd(d, t)
    g.api.ntt_inv(d, t)
    assert g.api.launch_count() - c0 == 2


def test_keyswitch_strided_d2_of_tensor_output(g):
    """The relinearisation input read in place: component d2 of a
    [batch][3][L][n] tensor product (in_offset = 2 L n, in_stride = 3 L n)."""
    import torch
    log_n, L, K, dnum, batch = 12, 8, 4, 2, 3
    n = 1 << log_n
    qp = g.qp_basis(log_n, L, K)
    t = g.tables(log_n, tuple(qp))
    mt = g.api.ModupTables(L, K, dnum, qp)
    ps = oracle.psis(qp, n)
    d = inputs.uniform_residues((batch, 3, L, n), qp[:L], 12, buffer=0)
    keys = inputs.uniform_residues((dnum, 2, L + K, n), qp, 12, buffer=1)
    out = torch.empty((batch, 2, L + K, n), dtype=torch.uint64, device="cuda")
    g.api.keyswitch_ip(out, g.dev(d), g.dev(keys), L, K, dnum, t, mt, in_offset=2 * L * n, in_stride=3 * L * n,
                       batch=batch)
    want = oracle.keyswitch_batch(np.ascontiguousarray(d[:, 2]), keys, qp, ps, L, K, dnum)
    assert np.array_equal(g.host(out), want)
