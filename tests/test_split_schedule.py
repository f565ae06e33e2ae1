"""Host-side check of the NTT kernels' schedules (no GPU).

For every shape in csrc/ntt_shapes.h -- the split shapes (n >= 2^14) and the
one-CTA-per-row shapes (n <= 2^13) -- the forward and the inverse are
replayed here at the production n, in exact modular arithmetic, following the
kernels' own index arithmetic:
- the column kernels: which thread slot holds which column element, the
  order of the stages, the shared-memory exchange between the two thread
  layouts and the twiddle index of every butterfly;
- the block kernels: the register passes (the positions a thread holds in
  each pass), the stages inside a pass, the twiddles staged in shared memory
  and the last pass's reads from the permuted table slots.
The twiddles come from the table blob that the library's host builder writes
(fhe_ntt_tables_build_host), so the replay also checks the table layout the
kernels rely on.  The results must equal the oracle's NTT and INTT.  A
wrong twiddle index, a stage on the wrong layout or a mismatch between the
table's slot order and the last pass's reads fails here without a GPU; the
shorter replays by textbook definition stay as a second reference.
"""
import ctypes
import os
import random
import re

import numpy as np
import pytest

import oracle
from ntt_arithmetic_gb300 import _native as N
from ntt_arithmetic_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SHAPES_H = os.path.join(ROOT, "ntt_arithmetic_gb300", "csrc", "ntt_shapes.h")


def split_shapes(prefix: str, full: bool = False):
    """(log_n, log_c) -- with full=True (log_n, log_c, log_t, log_e) -- of every
    split shape named FHE_<prefix>SHAPE_<n>."""
    text = open(SHAPES_H).read()
    out = []
    for m in re.finditer(r"#define FHE_%sSHAPE_(\d+) (\d+), (\d+), (\d+), (\d+), (\d+)" % prefix, text):
        log_n, logc, logt, loge, split = (int(m.group(i)) for i in (1, 2, 3, 4, 6))
        if split:
            out.append((log_n, logc, logt, loge) if full else (log_n, logc))
    return sorted(set(out))


def brv(x: int, bits: int) -> int:
    return int(format(x, "0%db" % bits)[::-1], 2) if bits else 0


def fwd_table(q: int, psi: int, log_n: int):
    """fwd[k] = psi^brv(k) (log_n bits): the forward stage-s twiddle of block b is fwd[2^s + b]."""
    n = 1 << log_n
    return [pow(psi, brv(k, log_n), q) for k in range(n)]


def col(x, log_n, logc):
    """Residues of the row as C arrays over the M columns: col[j1][j2] = x[j1 M + j2]."""
    m = 1 << (log_n - logc)
    return [np.array([int(v) for v in x[j1 * m:(j1 + 1) * m]], dtype=object) for j1 in range(1 << logc)]


def fwd_columns(cols, q, fwd, logc):
    """The forward column kernel: threads g < TPC of a column hold j1 = g + TPC i
    for the spans >= TPC, then (after the exchange) j1 = VPT g + i."""
    c = 1 << logc
    logtpc = logc // 2
    tpc, logvpt = 1 << logtpc, logc - logtpc
    vpt = 1 << logvpt
    for g in range(tpc):
        x = [cols[g + tpc * i] for i in range(vpt)]
        for s in range(logvpt):
            hi = vpt >> (s + 1)
            for i in range(vpt):
                if i & hi:
                    continue
                w = fwd[(1 << s) + ((g + tpc * i) >> (logc - s))]
                t = x[i + hi] * w % q
                x[i], x[i + hi] = (x[i] + t) % q, (x[i] - t) % q
        for i in range(vpt):
            cols[g + tpc * i] = x[i]
    if logtpc > 0:
        for g in range(tpc):
            x = [cols[vpt * g + i] for i in range(vpt)]
            for s in range(logvpt, logc):
                hi = 1 << (logc - 1 - s)
                for i in range(vpt):
                    if i & hi:
                        continue
                    w = fwd[(1 << s) + ((vpt * g + i) >> (logc - s))]
                    t = x[i + hi] * w % q
                    x[i], x[i + hi] = (x[i] + t) % q, (x[i] - t) % q
            for i in range(vpt):
                cols[vpt * g + i] = x[i]
    assert len(cols) == c
    return cols


def fwd_local(row, q, fwd, log_n, logc):
    """Stages s >= log_c by definition: pairs (p, p + n/2^(s+1)) in blocks of n/2^s, twiddle fwd[2^s + block]."""
    n = 1 << log_n
    a = row.reshape(1, n)
    for s in range(logc, log_n):
        half = n >> (s + 1)
        a = a.reshape(1 << s, 2, half)
        w = np.array([fwd[(1 << s) + b] for b in range(1 << s)], dtype=object).reshape(1 << s, 1)
        t = a[:, 1, :] * w % q
        a = np.stack([(a[:, 0, :] + t) % q, (a[:, 0, :] - t) % q], axis=1)
    return a.reshape(n)


def inv_tables(q: int, psi: int, log_n: int):
    """inv[h + j] = omega_2h^-j (omega_2h = psi^(n/h)); twist[p] = n^-1 psi^-p."""
    n = 1 << log_n
    inv = [0] * n
    h = 1
    while h < n:
        wi = pow(pow(psi, n // h, q), q - 2, q)
        for j in range(h):
            inv[h + j] = pow(wi, j, q)
        h *= 2
    ninv, psii = pow(n, q - 2, q), pow(psi, q - 2, q)
    return inv, [ninv * pow(psii, p, q) % q for p in range(n)]


def inv_local(row, q, inv, log_n, logc):
    """Cyclic decimation-in-time spans 1 .. M/2 by definition: pairs (p, p + h), p mod 2h < h,
    the second times inv[h + (p mod h)]."""
    n = 1 << log_n
    m = n >> logc
    a = row.copy()
    h = 1
    while h < m:
        a = a.reshape(n // (2 * h), 2, h)
        w = np.array(inv[h:2 * h], dtype=object).reshape(1, h)
        t = a[:, 1, :] * w % q
        a = np.stack([(a[:, 0, :] + t) % q, (a[:, 0, :] - t) % q], axis=1)
        h *= 2
    return a.reshape(n)


def inv_columns(cols, q, inv, twist, log_n, logc):
    """The inverse column kernel: j1 = VPT g + i for the spans below VPT, then
    j1 = g + TPC i; span-M 2^S twiddle inv[M (2^S + j1 mod 2^S) + j2]; then the twist."""
    m = 1 << (log_n - logc)
    logtpc = logc // 2
    tpc, logvpt = 1 << logtpc, logc - logtpc
    vpt = 1 << logvpt
    inv_a = np.array(inv, dtype=object)
    tw = lambda idx: inv_a[m * idx:m * idx + m]      # noqa: E731 -- the twiddles of all columns j2
    for g in range(tpc):
        x = [cols[vpt * g + i] for i in range(vpt)]
        for s in range(logvpt):
            h = 1 << s
            for i in range(vpt):
                if i & h:
                    continue
                t = x[i + h] * tw((1 << s) + (i & (h - 1))) % q
                x[i], x[i + h] = (x[i] + t) % q, (x[i] - t) % q
        for i in range(vpt):
            cols[vpt * g + i] = x[i]
    if logtpc > 0:
        for g in range(tpc):
            x = [cols[g + tpc * i] for i in range(vpt)]
            for s in range(logvpt, logc):
                hi = 1 << (s - logtpc)
                for i in range(vpt):
                    if i & hi:
                        continue
                    j1 = g + tpc * i
                    t = x[i + hi] * tw((1 << s) + (j1 & ((1 << s) - 1))) % q
                    x[i], x[i + hi] = (x[i] + t) % q, (x[i] - t) % q
            for i in range(vpt):
                cols[g + tpc * i] = x[i]
    tw_a = np.array(twist, dtype=object)
    return [cols[j1] * tw_a[j1 * m:(j1 + 1) * m] % q for j1 in range(1 << logc)]


def test_shapes_file_lists_split_shapes():
    fwd, inv = split_shapes(""), split_shapes("INV_")
    assert fwd and inv
    for log_n, logc in fwd + inv:
        assert log_n >= 14 and 1 <= logc < log_n


@pytest.mark.parametrize("log_n,logc", split_shapes(""))
def test_forward_column_schedule(log_n, logc):
    n = 1 << log_n
    q = int(oracle.primes(2 * n, 1)[0])
    psi = oracle.psi(q, 2 * n)
    rng = random.Random(log_n * 100 + logc)
    x = np.array([rng.randrange(q) for _ in range(n)], dtype=np.uint64)
    fwd = fwd_table(q, psi, log_n)
    cols = fwd_columns(col(x, log_n, logc), q, fwd, logc)
    row = np.concatenate(cols)
    got = fwd_local(row, q, fwd, log_n, logc)
    want = oracle.ntt(x, q, psi)
    assert [int(v) for v in got] == [int(v) for v in want]


@pytest.mark.parametrize("log_n,logc", split_shapes("INV_"))
def test_inverse_column_schedule(log_n, logc):
    n = 1 << log_n
    q = int(oracle.primes(2 * n, 1)[0])
    psi = oracle.psi(q, 2 * n)
    rng = random.Random(log_n * 100 + logc + 7)
    y = np.array([rng.randrange(q) for _ in range(n)], dtype=np.uint64)
    inv, twist = inv_tables(q, psi, log_n)
    row = inv_local(np.array([int(v) for v in y], dtype=object), q, inv, log_n, logc)
    out = np.concatenate(inv_columns(col(row, log_n, logc), q, inv, twist, log_n, logc))
    want = oracle.intt(y, q, psi)
    assert [int(v) for v in out] == [int(v) for v in want]


# ------------------------------------------------- block kernels, library tables --

@pytest.fixture(scope="module")
def lib():
    B.build()
    return N.lib()


def library_tables(lib, log_n: int, q: int):
    """The forward table by slot, the inverse table and the twist table (values only) of
    the blob the library builds on the host for one prime."""
    n = 1 << log_n
    nb = ctypes.c_size_t()
    assert lib.fhe_ntt_tables_bytes(log_n, 1, ctypes.byref(nb)) == 0
    blob = np.zeros(nb.value, dtype=np.uint8)
    arr = (ctypes.c_uint64 * 1)(q)
    assert lib.fhe_ntt_tables_build_host(log_n, 1, arr, blob.ctypes.data_as(ctypes.c_void_p), nb.value) == 0
    t = N.NttTables()
    base = blob.ctypes.data
    assert lib.fhe_ntt_tables_bind(ctypes.c_void_p(base), nb.value, log_n, 1, ctypes.byref(t)) == 0
    pairs = lambda ptr: np.frombuffer(blob, dtype=np.uint64, count=2 * n, offset=ptr - base).reshape(n, 2)  # noqa: E731
    vals = lambda ptr: [int(v) for v in pairs(ptr)[:, 0]]  # noqa: E731
    return vals(t.fwd), vals(t.inv), vals(t.twist)


def pass_pos(g, j, b, ep):
    """Position in the block of the j-th residue of thread group g in a pass over bits [b, b + ep)."""
    return (g & ((1 << b) - 1)) | (j << b) | ((g >> b) << (b + ep))


def fwd_block(blk, r, q, fwd_slots, log_n, logc, logt, loge):
    """k_ntt_fwd_blk on block r: passes from the high bits down; the first pass's
    twiddles are common to all groups, the middle passes' come from the staged
    copy of the table, the last pass reads the permuted slots (r, jj, g)."""
    logm = log_n - logc
    t_, e_ = 1 << logt, 1 << loge
    p_ = (logm + loge - 1) // loge
    erem = logm - (p_ - 1) * loge
    th = np.arange(t_)
    for pi in range(p_):
        b = (p_ - 1 - pi) * loge
        ep = erem if pi == 0 else loge
        g_, epn = e_ >> ep, 1 << ep
        pos = {(k, j): pass_pos(th + t_ * k, j, b, ep) for k in range(g_) for j in range(epn)}
        x = {kj: blk[p] for kj, p in pos.items()}
        for i in range(ep):
            s_ = log_n - b - ep + i
            half, nw = 1 << (ep - 1 - i), 1 << i
            for k in range(g_):
                g = th + t_ * k
                for jj in range(nw):
                    if b + ep == logm and g_ > 1:
                        w = fwd_slots[(1 << s_) + (r << i) + jj]
                    elif b == 0:
                        idx = (1 << s_) + (r << (logm - ep + i)) + (jj << (logm - ep)) + g
                        w = np.array([fwd_slots[v] for v in idx], dtype=object)
                    else:
                        idx = (1 << s_) + (r << (logm - b - ep + i)) + ((g >> b) << i) + jj
                        w = np.array([fwd_slots[v] for v in idx], dtype=object)
                    for u in range(half):
                        j = jj * 2 * half + u
                        tt = x[(k, j + half)] * w % q
                        x[(k, j)], x[(k, j + half)] = (x[(k, j)] + tt) % q, (x[(k, j)] - tt) % q
        for kj, p in pos.items():
            blk[p] = x[kj]
    return blk


def inv_block(blk, q, inv, logm, logt, loge):
    """k_ntt_inv_blk on one block: passes from the low bits up; in the first pass the
    twiddle-1 butterflies, elsewhere inv[2^(B+I) + (g mod 2^B) + (jl << B)]."""
    t_, e_ = 1 << logt, 1 << loge
    p_ = (logm + loge - 1) // loge
    erem = logm - (p_ - 1) * loge
    th = np.arange(t_)
    for pi in range(p_):
        b = pi * loge
        ep = erem if pi == p_ - 1 else loge
        g_, epn = e_ >> ep, 1 << ep
        pos = {(k, j): pass_pos(th + t_ * k, j, b, ep) for k in range(g_) for j in range(epn)}
        x = {kj: blk[p] for kj, p in pos.items()}
        for i in range(ep):
            kb, half = b + i, 1 << i
            nh = epn // (2 * half)
            for k in range(g_):
                gl = (th + t_ * k) & ((1 << b) - 1)
                for jl in range(half):
                    if b == 0 and jl == 0:
                        w = 1
                    else:
                        w = np.array([inv[v] for v in (1 << kb) + gl + (jl << b)], dtype=object)
                    for jh in range(nh):
                        j = jh * 2 * half + jl
                        tt = x[(k, j + half)] * w % q
                        x[(k, j)], x[(k, j + half)] = (x[(k, j)] + tt) % q, (x[(k, j)] - tt) % q
        for kj, p in pos.items():
            blk[p] = x[kj]
    return blk


@pytest.mark.parametrize("log_n,logc,logt,loge", split_shapes("", full=True))
def test_forward_kernels_with_library_tables(lib, log_n, logc, logt, loge):
    n, m = 1 << log_n, 1 << (log_n - logc)
    q = int(oracle.primes(2 * n, 1)[0])
    psi = oracle.psi(q, 2 * n)
    fwd_slots, _, _ = library_tables(lib, log_n, q)
    rng = random.Random(log_n * 1000 + logc)
    x = np.array([rng.randrange(q) for _ in range(n)], dtype=np.uint64)
    # the column kernel's stages read slots 2^s + block directly (identity below the last pass)
    row = np.concatenate(fwd_columns(col(x, log_n, logc), q, fwd_slots, logc))
    for r in range(1 << logc):
        row[r * m:(r + 1) * m] = fwd_block(row[r * m:(r + 1) * m].copy(), r, q, fwd_slots, log_n, logc, logt, loge)
    want = oracle.ntt(x, q, psi)
    assert [int(v) for v in row] == [int(v) for v in want]


@pytest.mark.parametrize("log_n,logc,logt,loge", split_shapes("INV_", full=True))
def test_inverse_kernels_with_library_tables(lib, log_n, logc, logt, loge):
    n, m = 1 << log_n, 1 << (log_n - logc)
    q = int(oracle.primes(2 * n, 1)[0])
    psi = oracle.psi(q, 2 * n)
    _, inv, twist = library_tables(lib, log_n, q)
    rng = random.Random(log_n * 1000 + logc + 7)
    y = np.array([rng.randrange(q) for _ in range(n)], dtype=np.uint64)
    row = np.array([int(v) for v in y], dtype=object)
    for r in range(1 << logc):
        row[r * m:(r + 1) * m] = inv_block(row[r * m:(r + 1) * m].copy(), q, inv, log_n - logc, logt, loge)
    out = np.concatenate(inv_columns(col(row, log_n, logc), q, inv, twist, log_n, logc))
    want = oracle.intt(y, q, psi)
    assert [int(v) for v in out] == [int(v) for v in want]


def one_cta_shapes(prefix: str):
    """(log_n, log_t, log_e) of every one-CTA-per-row shape named FHE_<prefix>SHAPE_<n>."""
    text = open(SHAPES_H).read()
    out = []
    for m in re.finditer(r"#define FHE_%sSHAPE_(\d+) (\d+), (\d+), (\d+), (\d+), (\d+)" % prefix, text):
        log_n, logc, logt, loge, split = (int(m.group(i)) for i in (1, 2, 3, 4, 6))
        if not split:
            assert logc == 0
            out.append((log_n, logt, loge))
    return sorted(set(out))


@pytest.mark.parametrize("log_n,logt,loge", one_cta_shapes(""))
def test_one_cta_forward_with_library_tables(lib, log_n, logt, loge):
    """k_ntt_fwd (n <= 2^13): the block kernel's passes over the whole row."""
    n = 1 << log_n
    q = int(oracle.primes(2 * n, 1)[0])
    psi = oracle.psi(q, 2 * n)
    fwd_slots, _, _ = library_tables(lib, log_n, q)
    rng = random.Random(log_n * 7 + 1)
    x = np.array([rng.randrange(q) for _ in range(n)], dtype=np.uint64)
    got = fwd_block(np.array([int(v) for v in x], dtype=object), 0, q, fwd_slots, log_n, 0, logt, loge)
    assert [int(v) for v in got] == [int(v) for v in oracle.ntt(x, q, psi)]


@pytest.mark.parametrize("log_n,logt,loge", one_cta_shapes("INV_"))
def test_one_cta_inverse_with_library_tables(lib, log_n, logt, loge):
    """k_ntt_inv (n <= 2^13): the passes over the whole row, then the twist at every position."""
    n = 1 << log_n
    q = int(oracle.primes(2 * n, 1)[0])
    psi = oracle.psi(q, 2 * n)
    _, inv, twist = library_tables(lib, log_n, q)
    rng = random.Random(log_n * 7 + 2)
    y = np.array([rng.randrange(q) for _ in range(n)], dtype=np.uint64)
    got = inv_block(np.array([int(v) for v in y], dtype=object), q, inv, log_n, logt, loge)
    got = [int(v) * twist[p] % q for p, v in enumerate(got)]
    assert got == [int(v) for v in oracle.intt(y, q, psi)]
