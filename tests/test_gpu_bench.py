"""The bench's pipelined end-to-end leg computes what the plain step does:
each step's key-switch output, read back to host memory, equals the output
of the same step run on a fresh copy of the input."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def test_e2e_pipeline_matches_plain_steps():
    import torch
    import gpu_util  # noqa: F401  (builds the library)
    import bench
    dev = torch.device("cuda", 0)
    st = bench.build_state(dev, seed=5)
    bench.e2e_steps(st, 3, dev)
    got = {2: st["ks_pinned"].numpy().copy(), 1: st["ks_pinned2"].numpy().copy()}
    for i in (1, 2):
        st["X"].copy_(st["x_pinned"])
        bench.run_step(st, i)
        torch.cuda.synchronize()
        assert np.array_equal(st["KS"].cpu().numpy(), got[i]), i


def test_pr1_row_step_is_the_negacyclic_product():
    """One step of the bench's n=2048 / 4-prime row (forward NTT of a and b,
    pointwise product, inverse NTT) leaves the schoolbook negacyclic product
    a*b in its output, prime by prime."""
    import torch
    import gpu_util  # noqa: F401  (builds the library)
    import bench
    import oracle
    from ntt_arithmetic_gb300 import inputs
    row = bench.Pr1Row()
    row.setup(torch.device("cuda", 0))
    row.step()
    torch.cuda.synchronize()
    got = row.P.cpu().numpy()
    n = 1 << row.LOG_N
    for l, q in enumerate(row.q):
        a = inputs.uniform_residues((1, row.L, n), row.q, 1, buffer=0)[0, l]
        b = inputs.uniform_residues((1, row.L, n), row.q, 1, buffer=1)[0, l]
        assert np.array_equal(got[l], oracle.negacyclic_mul(a, b, int(q))), l


def test_two_stream_step_matches_the_plain_step():
    """The bench's two-stream form of the step (two halves of 2 ciphertext
    pairs on two streams) leaves the same key-switch output as the plain
    one-stream step."""
    import torch
    import gpu_util  # noqa: F401  (builds the library)
    import bench
    dev = torch.device("cuda", 0)
    st = bench.build_state(dev, seed=6)
    bench.run_step(st, 3)
    torch.cuda.synchronize()
    want = st["KS"].cpu().numpy().copy()
    st["X"].copy_(st["x_pinned"])
    st["KS"].zero_()
    streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    torch.cuda.synchronize()
    bench.run_step_halves(st, 3, streams)
    torch.cuda.synchronize()
    assert np.array_equal(st["KS"].cpu().numpy(), want)
