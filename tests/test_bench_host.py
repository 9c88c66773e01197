"""Host-side bookkeeping of bench.py: the per-step cache sizes used for the
decode roofline equal the oracle's cache sets."""
import numpy as np

import bench
from oracle import fastgen_oracle as O
from synth import CONFIGS, make_workload, punct_ids, special_ids


def test_cache_rows_match_oracle():
    cfg = CONFIGS["tiny"].with_(L=2, H=4, n=100, steps=30, r_l=0.2)
    w = make_workload(cfg, threads=1)
    T = float(np.float32(cfg.T))
    policy, keep, sizes = [], [], np.zeros(cfg.steps, dtype=np.int64)
    for g in range(cfg.G):
        Qa, Ka, Va = (w[x][g].double().numpy() for x in "QKV")
        r = O.profile_head(Qa[:cfg.n], Ka[:cfg.n], w["ids"][0], special_ids(), punct_ids(), T,
                           cfg.r_l, cfg.r_f)
        policy.append(r["policy"])
        keep.append(r["keep"])
        static = [int(j) for j in np.nonzero(r["keep"] == O.KEEP_STATIC)[0]]
        for st in range(cfg.steps):
            t = cfg.n + st
            tau = int(w["ids"][0][t])
            if O.stores_static(r["policy"], tau in special_ids(), tau in punct_ids()):
                static.append(t)
            sizes[st] += len(O.decode_positions(r["policy"], static, r["w"], t))
    rows, ring = bench.cache_rows_per_step(cfg, np.array(policy), np.array(keep), w["ids"],
                                           special_ids(), punct_ids())
    assert np.array_equal(rows, sizes)
    assert (ring >= 0).all()


def test_group_caches_union():
    cfg = CONFIGS["tiny"].with_(L=1, H=4, Hkv=2, n=5)
    policy = np.array([0, 3, 1, 2])
    keep = np.array([[1, 0, 0, 0, 0], [1, 1, 0, 2, 2], [1, 0, 1, 0, 0], [0, 1, 1, 0, 0]],
                    dtype=np.uint8)
    pol, k = bench.group_caches(cfg, policy, keep)
    assert list(pol) == [3, 2]
    assert k.tolist() == [[1, 1, 0, 2, 2], [1, 1, 1, 0, 0]]


def test_cpu_baseline_sample_is_bounded_and_reported():
    """The oracle sample stops once its time budget is spent (at least one
    head) and says how many heads it timed."""
    cfg = CONFIGS["tiny"].with_(n=64, steps=4)
    rep = bench.cpu_baseline(cfg, max_heads=3, budget_s=0.0)
    assert rep["kind"] == "oracle" and rep["value"] > 0 and rep["cores"] >= 1
    assert rep["sample"].startswith("1 of 4 heads")
    full = bench.cpu_baseline(cfg, max_heads=3, budget_s=None)
    assert full["sample"].startswith("3 of 4 heads")
