"""The allocation-free decode entry point (fastgen_decode_attn_noalloc).

It exists for callers that cannot allocate device memory while decoding,
e.g. an engine whose pool allocator took all free device memory at start-up.
Its scratch is a fixed array inside the library instead of a caller-supplied
workspace.  The GPU test drives it through the C ABI for two generation steps
in a row, next to the ordinary entry point on an identical copy of the
caches.  Both run the same kernels on the same inputs, so the outputs, the
K/V pools, the positions and the descriptors must agree bit for bit.

The file name sorts last so that pytest collects it after every other test
file: if it fails, a run that stops at the first failure (-x) has already run
the rest of the suite.  The test makes the entry point's first call itself
(the call that sets the array aside), so it passes alone in a fresh process
and after the other tests alike.
"""
import ctypes

import numpy as np
import pytest
import torch

from adaptive_head_kv_gb300 import fastgen as fg
from synth import CONFIGS, make_workload, punct_ids, special_ids

def test_noalloc_rejects_plans_beyond_its_scratch():
    """Host-side check (no GPU needed): a plan whose partials exceed the
    library's fixed scratch is refused before anything is launched."""
    p = fg.Params(1, 2, 3, 100, 128, fg.FG_BF16, 0.95, 0.3, 0.3, 0.0)
    per_item = (128 + 2) * 4
    info = fg.PlanInfo(1000, fg.NOALLOC_SCRATCH_BYTES // per_item + 10, 256)
    assert fg.fastgen_decode_workspace_bytes(p, info) > fg.NOALLOC_SCRATCH_BYTES
    fake = 1 << 20
    st = fg.lib().fastgen_decode_attn_noalloc(ctypes.byref(p), fake, ctypes.byref(info), fake,
                                             fake, fake, fake, fake, fake, fake, fake, 1, fake,
                                             1, 100, fake, fake, None)
    assert st == fg.FG_EWORKSPACE


@pytest.mark.gpu
def test_noalloc_matches_workspace_decode_two_calls():
    from adaptive_head_kv_gb300.session import FastGenSession, make_params

    cfg = CONFIGS["tiny"].with_(dtype="bf16", d=128, L=2, H=4, n=300, steps=2)
    w = make_workload(cfg)
    n, dev = cfg.n, torch.device("cuda")
    p = make_params(cfg.B, cfg.L, cfg.H, n, cfg.d, cfg.dtype, cfg.T, cfg.r_l, cfg.r_f)
    ids = torch.from_numpy(w["ids"]).to(dev)
    Q, K, V = (w[x][:, :n].contiguous().to(dev) for x in "QKV")
    ref = FastGenSession(p, special_ids(), punct_ids(), cfg.steps)
    noa = FastGenSession(p, special_ids(), punct_ids(), cfg.steps)
    for s in (ref, noa):
        s.prefill(Q, K, V, ids[:, :n].contiguous())
    assert fg.fastgen_decode_workspace_bytes(p, noa.info) <= fg.NOALLOC_SCRATCH_BYTES
    for st in range(2):
        t = n + st
        q, k, v = (w[x][:, t].contiguous().to(dev) for x in "QKV")
        tid = ids[:, t].contiguous()
        want = ref.decode(q, k, v, tid, t).float().clone()
        got = torch.empty_like(noa.out)
        fg.fastgen_decode_attn_noalloc(noa.p, noa.plan, noa.info, noa.K_pool, noa.V_pool,
                                       noa.pos_pool, q, k, v, tid, noa.special, noa.punct, t,
                                       got, noa.dev_err)
        torch.cuda.synchronize()
        assert torch.isfinite(got.float()).all()
        # same kernels, same inputs: only the scratch address differs
        assert torch.equal(got.float(), want), st
    assert fg.fastgen_read_error(noa.dev_err) == fg.FG_OK
    assert torch.equal(ref.pos_pool, noa.pos_pool)
    live = ref.pos_pool >= 0  # rows in use; empty rows hold unspecified bytes
    assert torch.equal(ref.K_pool[live], noa.K_pool[live])
    assert torch.equal(ref.V_pool[live], noa.V_pool[live])
    assert np.array_equal(np.frombuffer(bytes(ref.descriptors()), dtype=np.uint8),
                          np.frombuffer(bytes(noa.descriptors()), dtype=np.uint8))
