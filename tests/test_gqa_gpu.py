"""Grouped-query attention on the GPU against the oracle's group extension:
per-query-head profiles, one union cache per key/value head, every member's
decode outputs."""
import pytest
import torch

from synth import CONFIGS

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from parity_util import compare_groups, run_gpu


@pytest.mark.parametrize("name,kw", [
    ("bf16_R2", dict(dtype="bf16", d=128, L=2, H=8, Hkv=4, n=300, steps=24, one_of_each=False)),
    ("bf16_R4", dict(dtype="bf16", d=128, L=2, H=8, Hkv=2, n=300, steps=24, one_of_each=False)),
    ("bf16_R8_d64", dict(dtype="bf16", d=64, L=2, H=8, Hkv=1, n=257, steps=20, one_of_each=False)),
    ("fp32_R2", dict(dtype="fp32", d=64, L=1, H=4, Hkv=2, n=200, steps=16)),
    ("bf16_R4_two_seqs", dict(dtype="bf16", d=128, B=2, L=1, H=8, Hkv=2, n=190, steps=16,
                              one_of_each=False)),
])
def test_groups_match_oracle(name, kw):
    cfg = CONFIGS["tiny"].with_(**kw)
    gpu = run_gpu(cfg)
    rep = compare_groups(cfg, gpu)
    print(name, rep)
    assert gpu["dev_err"] == 0
    assert rep["groups"] - rep["groups_exempt"] >= max(1, rep["groups"] // 2), rep


def test_groups_on_the_7b_shape():
    """The 7B attention shape with 8 key/value heads per layer (group size
    4), 4 layers, every output against the oracle."""
    cfg = CONFIGS["llama7b"].with_(L=4, Hkv=8, steps=32)
    gpu = run_gpu(cfg)
    rep = compare_groups(cfg, gpu)
    assert gpu["dev_err"] == 0
    assert rep["groups"] - rep["groups_exempt"] >= 16, rep
