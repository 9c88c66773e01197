"""Host-side bookkeeping of bench.py: the per-step cache sizes used for the
decode roofline equal the oracle's cache sets, the CPU baseline's sample is
bounded, and the DRAM traffic figures are scaled, merged and voided as
their sources change."""
import json

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


def _ncu_csv(path, launches):
    """An ncu --csv log in the layout the profiler writes: notes, a header,
    then one row per (launch, metric)."""
    cols = ["ID", "Process ID", "Process Name", "Host Name", "Kernel Name", "Context", "Stream",
            "Block Size", "Grid Size", "Device", "CC", "Section Name", "Metric Name",
            "Metric Unit", "Metric Value"]
    lines = ["==PROF== Connected to process 1", ",".join(f'"{c}"' for c in cols)]
    for i, (kernel, metrics) in enumerate(launches):
        for name, unit, value in metrics:
            row = [str(i), "1", "python3", "host", kernel, "1", "7", "(256, 1, 1)", "(8, 1, 1)",
                   "0", "10.3", "Command line profiler metrics", name, unit, value]
            lines.append(",".join(f'"{c}"' for c in row))
    path.write_text("\n".join(lines) + "\n")


def test_traffic_record_scales_merges_and_expires(tmp_path, monkeypatch):
    """record_traffic: DRAM bytes per call of a kernel group (read + write of
    every kernel of the group, divided by the launches of the group's
    call-counting kernel), scaled to the full workload when captured on a
    smaller case, merged with the other groups already recorded; load_traffic
    returns the figure only for the same workload and unchanged sources."""
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "traffic.json"))
    split = "void unnamed>::split_kernel<__nv_bfloat16, 128, 1, 0>(DecodeArgs, int, int, float)"
    comb = "void unnamed>::combine_kernel<__nv_bfloat16, 128, 0>(DecodeArgs, int, int, int)"
    dram = lambda r, w, u="Mbyte": [("gpu__time_duration.sum", "us", "100"),
                                    ("dram__bytes_read.sum", u, r), ("dram__bytes_write.sum", u, w)]
    csv_path = tmp_path / "decode.csv"
    _ncu_csv(csv_path, [(split, dram("600", "4")), (comb, dram("2", "0.5")),
                        (split, dram("0.61", "0.003", "Gbyte")), (comb, dram("2,000", "500", "Kbyte"))])
    bench.record_traffic(str(csv_path), "llama65b", "cmd", scale={"decode": 10.0},
                         measured_on="llama65b_L2")
    want = ((600 + 4 + 2 + 0.5) * 1e6 + (0.61 + 0.003) * 1e9 + 2.5e6) / 2 * 10.0
    rec = json.load(open(bench.TRAFFIC_FILE))
    assert set(rec) == {"decode"}
    assert rec["decode"]["calls"] == 2 and rec["decode"]["scale"] == 10.0
    assert abs(rec["decode"]["bytes_per_call"] - want) < 1e-3 * want
    assert abs(bench.load_traffic("decode", "llama65b") - want) < 1e-3 * want
    assert bench.load_traffic("decode", "llama7b") is None  # another workload
    # a capture of another group keeps the decode figure
    sel = "void unnamed>::select_kernel(const float *, int)"
    prof = "void unnamed>::profile_tc_kernel<1, 128>(CUtensorMap_st, CUtensorMap_st, float *)"
    csv2 = tmp_path / "profile.csv"
    _ncu_csv(csv2, [(prof, dram("1000", "10")), (sel, dram("16", "0"))])
    bench.record_traffic(str(csv2), "llama65b", "cmd2", scale={"profile": 40.0},
                         measured_on="llama65b_L2")
    rec = json.load(open(bench.TRAFFIC_FILE))
    assert set(rec) == {"decode", "profile"}
    assert abs(rec["profile"]["bytes_per_call"] - 1026e6 * 40) < 1.0
    # a change to a group's sources voids its figure, not the other group's
    real = bench.source_digest
    monkeypatch.setattr(bench, "source_digest", lambda g: "changed" if g == "profile" else real(g))
    assert bench.load_traffic("profile", "llama65b") is None
    assert bench.load_traffic("decode", "llama65b") is not None
