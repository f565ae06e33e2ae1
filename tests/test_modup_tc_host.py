"""Host-side check of the tensor-core ModUp's encoding (no GPU).

The tensor-core extension (csrc/modup_tc.cu) computes each target residue of
a digit's basis extension as an exact fp16 x fp16 -> f32 contraction.  Per
coefficient it forms the CRT brackets y_a = [x_a (D/d_a)^-1]_{d_a}, for the
exact extension also the count e = floor(sum_a y_a / d_a) (from a 64.64
fixed-point sum, or -- when that sum is within 2 cnt units of an integer --
from Garner's digits and a redundant modulus 2^64); the A operand row holds
1024 + b for every byte b of the y_a and 1024 + e in column 15, the B operand
-- written by the library's host builder into the ModUp table blob -- the
7-bit limbs of (D/d_a) 2^(8e) mod p, the limbs of (-D) mod p in column 15 and
offset columns, so that every accumulator comes out as 2^23 + (an integer
below 2^21); the eight accumulators of a target recombine as
sum_s u_s 2^(7s) < 2^64, reduced with one Barrett step by
mu = floor(2^64 / p).

Here all of it is replayed in exact integer arithmetic from the blob the
library builds (fhe_modup_tables_build_host) and compared with the oracle's
ModUp (modup_batch).  A wrong weight, limb order, offset or correction
column, a wrong reciprocal or redundant-modulus constant, a wrong target list
or a near-integer test that misses a case fails here without a GPU.
"""
import ctypes
import math

import numpy as np
import pytest

import oracle
from ntt_arithmetic_gb300 import _native as N
from ntt_arithmetic_gb300 import build as B

ROWB = 128          # bytes of one operand row: 64 fp16
MAXA = 8            # digits of up to 8 primes take the tensor-core path


@pytest.fixture(scope="module")
def lib():
    B.build()
    return N.lib()


def a256(x: int) -> int:
    return (x + 255) & ~255


def layout(L: int, K: int, dnum: int) -> dict:
    """The ModUp blob's layout (the sections the tensor-core kernel reads)."""
    alpha = -(-L // dnum)
    LK = L + K
    off_garner = a256(dnum * 8)
    off_mr = a256(off_garner + dnum * alpha * alpha * 16)
    off_qinv = a256(off_mr + dnum * LK * alpha * 16)
    off_qhat = a256(off_qinv + dnum * alpha * 16)
    end = a256(off_qhat + dnum * LK * alpha * 16)
    tmax = (LK + 1) & ~1 if alpha <= MAXA else 0
    off_tgt = end
    off_frac = a256(off_tgt + dnum * tmax * 32)
    off_b = a256(off_frac + (dnum * (MAXA + 1) * 32 if tmax else 0))
    return {"alpha": alpha, "tmax": tmax, "tgt": off_tgt, "frac": off_frac, "b": off_b,
            "bytes": a256(off_b + dnum * tmax * 8 * ROWB)}


def fp16_int(bits: np.ndarray) -> np.ndarray:
    """Integer values of fp16 bit patterns holding integers (exact)."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64).astype(np.int64)


def weight_operand(blob: np.ndarray, off: int, rows: int) -> np.ndarray:
    """[rows][64] integers of an operand image: core (r/8, k/8) at ((r/8) 8 + k/8) 128, row r%8 at +16 (r%8)."""
    img = blob[off:off + rows * ROWB].view(np.uint16)
    out = np.zeros((rows, 64), dtype=np.int64)
    for r in range(rows):
        for kc in range(8):
            base = (((r >> 3) * 8 + kc) * ROWB + (r & 7) * 16) // 2
            out[r, 8 * kc:8 * kc + 8] = fp16_int(img[base:base + 8])
    return out


def build_blob(lib, L, K, dnum, qp):
    nb = ctypes.c_size_t()
    assert lib.fhe_modup_tables_bytes(L, K, dnum, ctypes.byref(nb)) == 0
    blob = np.zeros(nb.value, dtype=np.uint8)
    arr = (ctypes.c_uint64 * len(qp))(*[int(q) for q in qp])
    assert lib.fhe_modup_tables_build_host(L, K, dnum, arr, blob.ctypes.data_as(ctypes.c_void_p), nb.value) == 0
    return blob


def correction_count(xs, d, frac, approx):
    """The kernel's e: 0 for the approximate conversion; else the fixed-point
    estimate, or the redundant-modulus value when the estimate is near an integer."""
    M64 = (1 << 64) - 1
    Dj = math.prod(d)
    y = [xs[a] * pow(Dj // d[a], -1, d[a]) % d[a] for a in range(len(d))]
    if approx:
        return y, 0, False
    F, e = 0, 0
    for a in range(len(d)):
        phi = (int(frac[a, 0]) << 64) | int(frac[a, 1])
        assert phi == (1 << 128) // d[a]
        term = y[a] * int(frac[a, 0]) + ((y[a] * int(frac[a, 1])) >> 64)
        F += term
    e, F = F >> 64, F & M64
    near = F > M64 - 2 * len(d)
    if near:   # Garner's mixed-radix digits of X, then e = (sum y_a (D/d_a) - X) D^-1 mod 2^64
        X = sum(xs[a] * (Dj // d[a]) * pow(Dj // d[a], -1, d[a]) for a in range(len(d))) % Dj
        w = []
        for a in range(len(d)):
            w.append(X % d[a])
            X //= d[a]
        Y = sum(y[a] * int(frac[a, 2]) for a in range(len(d))) & M64
        Xr = sum(w[a] * int(frac[a, 3]) for a in range(len(d))) & M64
        e = ((Y - Xr) * int(frac[MAXA, 2])) & M64
    true_e = sum(y[a] * (Dj // d[a]) for a in range(len(d))) // Dj
    assert e == true_e, "the kernel's correction count is the exact one"
    return y, e, near


def replay(blob, lay, qp, L, K, dnum, x, approx):
    """The tensor-core kernel's arithmetic on coefficients x [L][m] (ints) -> [dnum][L+K][m]."""
    LK, alpha, tmax = L + K, lay["alpha"], lay["tmax"]
    m = len(x[0])
    out = np.zeros((dnum, LK, m), dtype=object)
    tg = blob[lay["tgt"]:lay["tgt"] + dnum * tmax * 32].view(np.uint64).reshape(dnum, tmax, 4)
    fr = blob[lay["frac"]:lay["frac"] + dnum * (MAXA + 1) * 32].view(np.uint64).reshape(dnum, MAXA + 1, 4)
    nears = 0
    for j in range(dnum):
        lo = j * alpha
        cnt = min(alpha, L - lo)
        d = [int(q) for q in qp[lo:lo + cnt]]
        Dj = math.prod(d)
        assert (int(fr[j, MAXA, 2]) * (Dj & ((1 << 64) - 1))) & ((1 << 64) - 1) == 1
        T = LK - cnt
        Tp = (T + 1) & ~1
        Bw = weight_operand(blob, lay["b"] + j * tmax * 8 * ROWB, 8 * Tp)
        assert (Bw.sum(axis=1) == 8192).all(), "every weight row sums to 8192 (the 2^23 offset)"
        assert (Bw <= 2048).all() and (Bw >= 0).all()
        A = np.full((m, 64), 1024, dtype=np.int64)
        for c in range(m):
            xs = [int(x[lo + a][c]) for a in range(cnt)]
            y, e, near = correction_count(xs, d, fr[j], approx)
            nears += near
            for a in range(cnt):
                assert y[a] < 1 << 50
                for k in range(7):
                    A[c, 8 * a + k] = 1024 + ((y[a] >> (8 * k)) & 255)
            A[c, 15] = 1024 + e
            for a in range(cnt):
                out[j, lo + a, c] = xs[a]
        Dacc = A @ Bw.T                         # exact: every value < 2^24
        assert (Dacc >= 1 << 23).all() and (Dacc < (1 << 23) + (1 << 21)).all()
        U = Dacc - (1 << 23)
        for t in range(T):
            p, limb = int(tg[j, t, 0]), int(tg[j, t, 3])
            assert p == int(qp[limb]) and not (lo <= limb < lo + cnt)
            mu = int(tg[j, t, 1])
            assert mu == (1 << 64) // p
            for c in range(m):
                S = sum(int(U[c, 8 * t + s]) << (7 * s) for s in range(8))
                assert S < 1 << 64, "the recombined sum fits one word"
                r = S - ((S * mu) >> 64) * p      # the kernel's Barrett step
                assert 0 <= r < 2 * p
                out[j, limb, c] = r % p
    return out, nears


@pytest.mark.parametrize("L,K,dnum,approx", [(24, 8, 3, False), (24, 8, 3, True), (7, 3, 3, False),
                                              (5, 2, 1, False), (16, 4, 2, True)])
def test_tensor_core_modup_encoding(lib, L, K, dnum, approx):
    qp = [int(v) for v in oracle.primes(1 << 12, L + K)]
    lay = layout(L, K, dnum)
    blob = build_blob(lib, L, K, dnum, qp)
    assert blob.size == lay["bytes"], "the layout replayed here matches the library's"
    assert lay["tmax"] > 0
    rng = np.random.default_rng(L * 100 + K * 10 + dnum)
    m = 16
    x = [[int(v) for v in rng.integers(0, qp[l], m, dtype=np.uint64)] for l in range(L)]
    for l in range(L):              # edge coefficients: 0, q - 1 and a small value in every limb
        x[l][0], x[l][1], x[l][2] = 0, qp[l] - 1, 1
    got, nears = replay(blob, lay, qp, L, K, dnum, x, approx)
    if not approx:
        assert nears > 0, "the edge coefficients (1 and q - 1 in every limb) take the exact fallback"
    a = np.array(x, dtype=np.uint64).reshape(1, L, m)
    want = oracle.modup_batch(a, np.array(qp, dtype=np.uint64), L, K, dnum, approx=approx)[0]
    assert np.array_equal(np.array(got, dtype=np.uint64), want)


def test_no_tensor_core_section_for_wide_digits(lib):
    """Digits of more than 8 primes keep the integer kernel: no tensor-core section."""
    lay = layout(24, 8, 2)
    assert lay["tmax"] == 0
    nb = ctypes.c_size_t()
    assert lib.fhe_modup_tables_bytes(24, 8, 2, ctypes.byref(nb)) == 0
    assert nb.value == lay["bytes"]


def moddown_layout(L: int, K: int) -> dict:
    """The ModDown blob's layout (the tensor-core sections after the integer kernel's)."""
    off_mr = a256(K * K * 16)
    off_hp = a256(off_mr + L * K * 16)
    off_hq = a256(off_hp + K * 8)
    off_pinv = a256(off_hq + L * 8)
    end = a256(off_pinv + L * 16)
    tc = K <= MAXA
    tmax = (L + 1) & ~1 if tc else 0
    off_qinv = end
    off_tgt = a256(off_qinv + (K * 16 if tc else 0))
    off_frac = a256(off_tgt + tmax * 32)
    off_b = a256(off_frac + ((MAXA + 1) * 32 if tc else 0))
    return {"tmax": tmax, "hp": off_hp, "hq": off_hq, "pinv": off_pinv, "qinv": off_qinv, "tgt": off_tgt,
            "frac": off_frac, "b": off_b, "bytes": a256(off_b + tmax * 8 * ROWB)}


@pytest.mark.parametrize("L,K,nearest", [(24, 8, True), (24, 8, False), (5, 3, True), (7, 1, True)])
def test_tensor_core_moddown_encoding(lib, L, K, nearest):
    """ModDown's tensor-core conversion d_l = ((X + h) mod P) - h mod q_l from the ModDown blob, replayed and
    finished as (x_l - d_l) P^-1 mod q_l, against the oracle's ModDown."""
    qp = [int(v) for v in oracle.primes(1 << 12, L + K)]
    lay = moddown_layout(L, K)
    nb = ctypes.c_size_t()
    assert lib.fhe_moddown_tables_bytes(L, K, ctypes.byref(nb)) == 0
    assert nb.value == lay["bytes"], "the layout replayed here matches the library's"
    blob = np.zeros(nb.value, dtype=np.uint8)
    arr = (ctypes.c_uint64 * len(qp))(*qp)
    assert lib.fhe_moddown_tables_build_host(L, K, arr, blob.ctypes.data_as(ctypes.c_void_p), nb.value) == 0
    P = qp[L:]
    Pprod = math.prod(P)
    tmax = lay["tmax"]
    tg = blob[lay["tgt"]:lay["tgt"] + tmax * 32].view(np.uint64).reshape(tmax, 4)
    fr = blob[lay["frac"]:lay["frac"] + (MAXA + 1) * 32].view(np.uint64).reshape(MAXA + 1, 4)
    qi = blob[lay["qinv"]:lay["qinv"] + K * 16].view(np.uint64).reshape(K, 2)
    hp = blob[lay["hp"]:lay["hp"] + K * 8].view(np.uint64)
    for a in range(K):
        assert int(qi[a, 0]) == pow(Pprod // P[a], -1, P[a])
    Bw = weight_operand(blob, lay["b"], 8 * tmax)
    assert (Bw.sum(axis=1) == 8192).all() and (Bw >= 0).all() and (Bw <= 2048).all()
    rng = np.random.default_rng(L * 10 + K)
    m = 16
    x = [[int(v) for v in rng.integers(0, qp[l], m, dtype=np.uint64)] for l in range(L + K)]
    for l in range(L + K):          # edge coefficients: 0 and q - 1 in every limb
        x[l][0], x[l][1] = 0, qp[l] - 1
    A = np.full((m, 64), 1024, dtype=np.int64)
    for c in range(m):
        xs = [(x[L + a][c] + (int(hp[a]) if nearest else 0)) % P[a] for a in range(K)]
        y, e, _ = correction_count(xs, P, fr, False)
        for a in range(K):
            for k in range(7):
                A[c, 8 * a + k] = 1024 + ((y[a] >> (8 * k)) & 255)
        A[c, 15] = 1024 + e
    Dacc = A @ Bw.T
    assert (Dacc >= 1 << 23).all() and (Dacc < (1 << 23) + (1 << 21)).all()
    U = Dacc - (1 << 23)
    out = np.zeros((L, m), dtype=np.uint64)
    h = (Pprod - 1) // 2 if nearest else 0
    for t in range(L):
        q, mu, aux, limb = (int(v) for v in tg[t])
        assert limb == t and q == qp[t] and mu == (1 << 64) // q
        assert aux == (q - ((Pprod - 1) // 2) % q) % q, "aux holds (q - h) mod q; truncation does not add it"
        pinv = pow(Pprod, -1, q)
        for c in range(m):
            S = sum(int(U[c, 8 * t + s]) << (7 * s) for s in range(8))
            assert S < 1 << 64
            r = S - ((S * mu) >> 64) * q
            d = r + (aux if nearest else 0)
            assert d < 3 * q, "d stays below 3 q for the forward NTT"
            out[t, c] = (x[t][c] - d) * pinv % q
    a_in = np.array(x, dtype=np.uint64).reshape(1, L + K, m)
    want = oracle.moddown_batch(a_in, np.array(qp, dtype=np.uint64), L, K, nearest)[0]
    assert np.array_equal(out, want)
