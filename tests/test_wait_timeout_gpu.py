"""The bounded-wait error path of the tensor-core profiler passes, exercised
without a GPU fault: fastgen_profile_stall_test holds one pass's producer
back, so the pass's other warps wait for work that never comes; each wait
runs out after its limit, every CTA unwinds with nothing in flight, and the
call reports FG_EDEVICE through the device error word.  The context must stay
usable: the same stream then runs the whole path, which must match the
oracle as in the main parity tests."""
import time

import numpy as np
import pytest
import torch

from synth import CONFIGS

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("stall_pass", [1, 2])
def test_wait_that_runs_out_is_reported_and_the_context_survives(stall_pass):
    from adaptive_head_kv_gb300 import fastgen as fg
    from adaptive_head_kv_gb300.session import FastGenSession, make_params
    from parity_util import compare, run_gpu
    from synth import make_workload, punct_ids, special_ids

    cfg = CONFIGS["tiny"].with_(dtype="bf16", d=128, L=2, H=4, n=300, steps=8)
    w = make_workload(cfg)
    n, dev = cfg.n, torch.device("cuda")
    p = make_params(cfg.B, cfg.L, cfg.H, n, cfg.d, cfg.dtype, cfg.T, cfg.r_l, cfg.r_f)
    s = FastGenSession(p, special_ids(), punct_ids(), cfg.steps)
    Q, K = (w[x][:, :n].contiguous().to(dev) for x in "QK")
    ids = torch.from_numpy(w["ids"][:, :n].copy()).to(dev)
    s.profile(Q, K, ids)
    assert fg.fastgen_read_error(s.dev_err) == fg.FG_OK
    want_policy = s.policy.clone()
    t0 = time.perf_counter()
    fg.fastgen_profile_stall_test(s.p, Q, K, ids, s.special, s.punct, s.policy, s.mass, s.cost,
                                  s.colsum, s.keep, s.kept, s.ws, s.dev_err, stall_pass)
    assert fg.fastgen_read_error(s.dev_err) == fg.FG_EDEVICE
    waited = time.perf_counter() - t0
    assert 0.5 < waited < 30.0, waited  # the waits ran out after their ~1 s limit
    # the same context and stream carry on: a fresh error word, then the path
    s.dev_err.zero_()
    s.profile(Q, K, ids)
    assert fg.fastgen_read_error(s.dev_err) == fg.FG_OK
    assert torch.equal(s.policy, want_policy)
    gpu = run_gpu(cfg)
    assert gpu["dev_err"] == 0
    rep = compare(cfg, gpu, list(range(cfg.G)))
    assert rep["decode_checked"] >= cfg.G // 2, rep
    assert np.array_equal(gpu["policy"], want_policy.cpu().numpy().astype(int))
