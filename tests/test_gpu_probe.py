"""The butterfly throughput probe (fhe_butterfly_probe) computes the butterfly
network its header describes: every thread's checksum equals the XOR of the
32 residues that exact modular arithmetic (Python integers) gives for the
same start values and twiddles.  This checks the probe, not the method: the
probe only measures how fast the NTT's butterfly can run."""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _expected(q, tw, ctas, iters):
    out = []
    for g in range(ctas * 256):
        x = [(977 * g + 131 * i) % q for i in range(32)]
        lane = g % 32
        for r in range(iters):
            for s in range(5):
                h = 32 >> (s + 1)
                for jj in range(1 << s):
                    w = int(tw[32 * (32 * (r % 2) + (1 << s) + jj) + lane])
                    for u in range(h):
                        j = jj * 2 * h + u
                        a, b = x[j], x[j + h]
                        x[j], x[j + h] = (a + w * b) % q, (a - w * b) % q
        acc = 0
        for v in x:
            acc ^= v
        out.append(acc)
    return np.array(out, dtype=np.uint64)


def test_butterfly_probe_matches_exact_arithmetic():
    import torch
    import gpu_util as g
    log_n = 11
    qs = g.primes(log_n, 2)
    t = g.tables(log_n, qs)
    ref = t.struct
    base = t.blob.data_ptr()
    words = t.blob.view(torch.int64)
    off = (ref.fwd - base) // 8
    tw = g.host(words[off: off + 2 * 2048].view(torch.uint64)).reshape(2048, 2)[:, 0]   # (w, Shoup) pairs
    out = torch.zeros(2 * 256, dtype=torch.uint64, device="cuda")
    n_bfly = g.api.butterfly_probe(out, 3, t)
    assert n_bfly == 2 * 256 * 3 * 80
    got = g.host(out)
    assert np.array_equal(got, _expected(qs[0], tw, 2, 3))
    out2 = torch.zeros_like(out)
    g.api.butterfly_probe(out2, 3, t)
    assert g.same_bits(out, out2)
