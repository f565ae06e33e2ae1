"""Guard words around every output and workspace: each entry point writes only
inside the buffers it is given.

Every output (and workspace) below is the interior of a larger device buffer
whose 4096 leading and trailing words hold a sentinel; after the call, the
sentinels must be intact.  The shapes cover each kernel family's launch
shapes: tiny rows, ragged batches, single-CTA rows (n <= 2^13), clusters of
2 to 16 CTAs (n = 2^14 .. 2^17), digit counts that leave a short last digit,
and long target chains.
"""
import numpy as np
import pytest

from ntt_arithmetic_gb300 import inputs

pytestmark = pytest.mark.gpu

PAD = 4096
SENTINEL = -0x5A5A5A5A5A5A5A5B          # 0xA5A5A5A5A5A5A5A5 as int64


@pytest.fixture(scope="module")
def g():
    import gpu_util
    return gpu_util


def guarded(shape, fill=None):
    """(full buffer, interior view of `shape`); the interior starts 16-byte aligned."""
    import torch
    n = int(np.prod(shape))
    full = torch.full((PAD + n + PAD,), SENTINEL, dtype=torch.int64, device="cuda")
    inner = full[PAD:PAD + n].view(*shape)
    if fill is not None:
        inner.copy_(fill.view(torch.int64))
    return full, inner.view(torch.uint64)


def intact(full):
    import torch
    torch.cuda.synchronize()
    head, tail = full[:PAD], full[-PAD:]
    return bool((head == SENTINEL).all()) and bool((tail == SENTINEL).all())


NTT_SHAPES = [(1, 1, 3), (4, 2, 5), (11, 3, 2), (13, 2, 1), (14, 2, 1), (16, 1, 1), (17, 1, 1)]


@pytest.mark.parametrize("log_n,L,batch", NTT_SHAPES)
def test_ntt_mul_automorph_stay_inside(g, log_n, L, batch):
    n = 1 << log_n
    qs = g.primes(log_n, L)
    t = g.tables(log_n, qs)
    x = g.dev(inputs.uniform_residues((batch, L, n), qs, 900 + log_n, buffer=0))
    y = g.dev(inputs.uniform_residues((batch, L, n), qs, 900 + log_n, buffer=1))
    full, buf = guarded((batch, L, n), x)
    g.api.ntt_fwd(buf, t)
    assert intact(full), "ntt_fwd"
    g.api.ntt_inv(buf, t)
    assert intact(full), "ntt_inv"
    assert g.same_bits(buf, x)
    full, out = guarded((batch, L, n))
    g.api.mul_ntt(out, x, y, t)
    assert intact(full), "mul_ntt"
    for domain in ("ntt", "coeff"):
        full, out = guarded((batch, L, n))
        g.api.automorph(out, x, 5 % (2 * n) or 1, t, domain=domain)
        assert intact(full), f"automorph {domain}"


@pytest.mark.parametrize("log_n,L,batch", [(11, 3, 2), (14, 2, 1), (4, 2, 3)])
def test_tensor_stays_inside(g, log_n, L, batch):
    n = 1 << log_n
    qs = g.primes(log_n, L)
    t = g.tables(log_n, qs)
    a = g.dev(inputs.uniform_residues((batch, 2, L, n), qs, 910, buffer=0))
    b = g.dev(inputs.uniform_residues((batch, 2, L, n), qs, 910, buffer=1))
    full, d = guarded((batch, 3, L, n))
    g.api.tensor(d, a, b, t)
    assert intact(full)


@pytest.mark.parametrize("log_n,L,K,dnum,batch", [(12, 5, 2, 2, 2), (14, 7, 3, 3, 1), (11, 4, 1, 4, 3)])
def test_keyswitch_family_stays_inside(g, log_n, L, K, dnum, batch):
    import torch
    n = 1 << log_n
    qp = g.qp_basis(log_n, L, K)
    t = g.tables(log_n, tuple(qp))
    mt = g.api.ModupTables(L, K, dnum, qp)
    x = g.dev(inputs.uniform_residues((batch, L, n), qp[:L], 920, buffer=0))
    keys = g.dev(inputs.uniform_residues((dnum, 2, L + K, n), qp, 920, buffer=1))
    ws_words = g.api.keyswitch_workspace_bytes(log_n, L, K, dnum, batch) // 8
    for approx in (False, True):
        full_o, out = guarded((batch, 2, L + K, n))
        full_w, ws = guarded((ws_words,))
        g.api.keyswitch_ip(out, x, keys, L, K, dnum, t, mt, ws, approx=approx)
        assert intact(full_o) and intact(full_w), f"keyswitch_ip approx={approx}"
    gal = [5, 25, 2 * n - 1]
    hkeys = g.dev(inputs.uniform_residues((3, dnum, 2, L + K, n), qp, 921, buffer=1))
    full_o, out = guarded((3, batch, 2, L + K, n))
    full_w, ws = guarded((ws_words,))
    g.api.keyswitch_hoisted(out, x, hkeys, gal, L, K, dnum, t, mt, ws)
    assert intact(full_o) and intact(full_w), "keyswitch_hoisted"
    full_d, digits = guarded((batch, dnum, L + K, n))
    g.api.keyswitch_decompose(digits, x, L, K, dnum, t, mt)
    assert intact(full_d), "keyswitch_decompose"
    full_o, out = guarded((3, batch, 2, L + K, n))
    g.api.keyswitch_apply(out, digits, hkeys, L, K, dnum, t, galois=gal)
    assert intact(full_o), "keyswitch_apply"
    if ws_words * 8 <= g.api.N.lib().fhe_keyswitch_noalloc_max_bytes():
        full_o, out = guarded((batch, 2, L + K, n))
        g.api.keyswitch_ip_noalloc(out, x, keys, L, K, dnum, t, mt)
        assert intact(full_o), "keyswitch_ip_noalloc"
    torch.cuda.synchronize()


@pytest.mark.parametrize("log_n,L,K,batch", [(12, 5, 3, 2), (14, 6, 1, 1), (11, 70, 2, 1)])
def test_moddown_stays_inside(g, log_n, L, K, batch):
    n = 1 << log_n
    qp = g.qp_basis(log_n, L, K)
    t = g.tables(log_n, tuple(qp))
    md = g.api.ModdownTables(L, K, qp)
    x = g.dev(inputs.uniform_residues((batch, L + K, n), qp, 930, buffer=0))
    ws_words = g.api.moddown_workspace_bytes(log_n, L, K, batch) // 8
    for domain in ("coeff", "ntt"):
        full_o, out = guarded((batch, L, n))
        full_w, ws = guarded((max(ws_words, 2),))
        g.api.moddown(out, x, L, K, t, md, domain=domain, workspace=ws)
        assert intact(full_o) and intact(full_w), domain


@pytest.mark.parametrize("log_n,S,T,batch", [(11, 3, 20, 2), (11, 1, 2100, 1), (13, 8, 32, 1)])
def test_bconv_stays_inside(g, log_n, S, T, batch):
    n = 1 << log_n
    chain = list(g.primes(log_n, max(S, T)))
    src, dst = chain[:S], chain[:T]
    bt = g.api.BconvTables(src, dst)
    x = g.dev(inputs.uniform_residues((batch, S, n), src, 940, buffer=0))
    for approx in (False, True):
        full, out = guarded((batch, T, n))
        g.api.bconv(out, x, bt, approx=approx)
        assert intact(full), f"bconv approx={approx}"
