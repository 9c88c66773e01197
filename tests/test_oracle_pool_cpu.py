"""The parallel oracle runs of the parity tests (spawned workers, row-block
profile for long prompts) give the serial dense oracle's results."""
import numpy as np

from parity_util import oracle_head, oracle_heads
from synth import CONFIGS, make_workload


def test_parallel_long_prompt_oracle_equals_serial_dense():
    cfg = CONFIGS["tiny"].with_(L=1, H=4, n=150, steps=6)
    w = make_workload(cfg, threads=1)
    idxs = [0, 2, 3]
    par = oracle_heads(cfg, w, idxs, long_prompt=True, procs=2)
    for i in idxs:
        want = oracle_head(cfg, w, i)
        got = par[i]
        assert got["policy"] == want["policy"]
        assert np.array_equal(got["keep"], want["keep"])
        assert np.abs(got["mass"] - want["mass"]).max() < 1e-12
        assert np.abs(got["colsum"] - want["colsum"]).max() < 1e-12
        assert np.abs(got["out"] - want["out"]).max() < 1e-12
        assert np.array_equal(got["final_pos"], want["final_pos"])
