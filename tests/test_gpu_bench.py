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
