"""The seeded generator: determinism, per-head independence and the
configured shapes and mixes."""
import numpy as np

from synth import CONFIGS, head_types, make_head, make_ids, make_workload, punct_ids, special_ids


def test_ids_rules():
    cfg = CONFIGS["llama7b"]
    ids = make_ids(cfg)
    assert ids.shape == (1, cfg.n + cfg.steps)
    assert ids[0, 0] == 1 and ids.min() >= 0 and ids.max() < 32000
    frac = np.isin(ids, punct_ids()).mean()
    assert 0.03 < frac < 0.07
    assert len(set(punct_ids().tolist())) == 10 and 1 not in punct_ids()
    assert np.array_equal(special_ids(), [1])
    assert np.array_equal(ids, make_ids(cfg))


def test_head_mix():
    cfg = CONFIGS["llama13b"]
    t = head_types(cfg)
    share = np.bincount(t.ravel(), minlength=4) / t.size
    assert np.allclose(share, cfg.mix, atol=0.04), share
    assert list(head_types(CONFIGS["tiny"])[0]) == [0, 1, 2, 3]


def test_head_regenerates_alone():
    cfg = CONFIGS["tiny"].with_(L=2, H=4)
    w = make_workload(cfg, seed=3, threads=4)
    ids, types = make_ids(cfg, 3), head_types(cfg, 3)
    for g in (0, 5, 7):
        q, k, v = make_head(cfg, 3, g, ids, types)
        assert np.array_equal(w["Q"][g].numpy(), q.astype(np.float32))
        assert np.array_equal(w["V"][g].numpy(), v.astype(np.float32))
    sub = make_workload(cfg, seed=3, heads=[5], threads=1)
    assert np.array_equal(sub["K"][0].numpy(), w["K"][5].numpy())


def test_normals_moments():
    cfg = CONFIGS["llama7b"]
    ids, types = make_ids(cfg), head_types(cfg)
    _, _, v = make_head(cfg, 0, 17, ids, types)
    assert abs(v.mean()) < 0.01 and abs(v.std() - 1) < 0.01


def test_split_layout_matches_heads():
    from synth import make_workload_split

    cfg = CONFIGS["tiny"].with_(L=2, H=3, n=40, steps=7)
    a = make_workload_split(cfg, seed=5, threads=3)
    b = make_workload(cfg, seed=5, threads=3)
    n = cfg.n
    for x in "QKV":
        assert np.array_equal(a[x].numpy(), b[x][:, :n].numpy())
        assert np.array_equal(a[x.lower()].numpy(), b[x][:, n:].transpose(0, 1).numpy())
