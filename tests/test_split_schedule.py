"""Host-side check of the split NTT's column-kernel schedules (no GPU).

For every split shape in csrc/ntt_shapes.h (n >= 2^14), the forward column
kernel's stages -- which thread slot holds which column element, in which
order the stages run, the shared-memory exchange between the two thread
layouts and the twiddle index of every butterfly -- are replayed here in
exact modular arithmetic over all columns at once, at the production n; the
remaining (block-local) stages are applied by their textbook definition.
The result must equal the oracle's NTT.  The inverse is checked the same
way: textbook block-local stages, then the inverse column kernel's schedule
and its twist, against the oracle's INTT.

This pins the index arithmetic that the GPU parity tests exercise only
through the compiled kernels: a wrong twiddle index or a stage run on the
wrong layout fails here without a GPU.
"""
import os
import random
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SHAPES_H = os.path.join(ROOT, "ntt_arithmetic_gb300", "csrc", "ntt_shapes.h")


def split_shapes(prefix: str):
    """(log_n, log_c) of every split shape named FHE_<prefix>SHAPE_<n>."""
    text = open(SHAPES_H).read()
    out = []
    for m in re.finditer(r"#define FHE_%sSHAPE_(\d+) (\d+), (\d+), (\d+), (\d+), (\d+)" % prefix, text):
        log_n, logc, split = int(m.group(1)), int(m.group(2)), int(m.group(6))
        if split:
            out.append((log_n, logc))
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
