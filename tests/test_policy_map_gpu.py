"""GPU parity of policy reuse with a saved head-policy map: a policy profiled
on one prompt (or set by hand) is saved, loaded and applied to another
prompt through fastgen_profile_with_policy; keep codes, the column sums of
the scored heads and every decode step are compared with the oracle."""
import numpy as np
import pytest
import torch

from synth import CONFIGS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    from adaptive_head_kv_gb300 import fastgen as fg

    fg.lib()  # raises if the CUDA library is missing


def _session(cfg, max_new):
    from adaptive_head_kv_gb300.session import FastGenSession, make_params
    from synth import punct_ids, special_ids

    p = make_params(cfg.B, cfg.L, cfg.H, cfg.n, cfg.d, cfg.dtype, cfg.T, cfg.r_l, cfg.r_f,
                    Hkv=cfg.Hkv)
    return p, FastGenSession(p, special_ids(), punct_ids(), max_new, guard=True)


def _device_inputs(w, n):
    dev = torch.device("cuda")
    return (w["Q"][:, :n].contiguous().to(dev), w["K"][:, :n].contiguous().to(dev),
            w["V"][:, :n].contiguous().to(dev), torch.from_numpy(w["ids"]).to(dev))


def _run_with_map(cfg, policy_map, seed):
    """Prefill prompt `seed` under the map and run its decode steps."""
    from synth import make_workload

    w = make_workload(cfg, seed)
    n = cfg.n
    p, s = _session(cfg, cfg.steps)
    Q, K, V, ids = _device_inputs(w, n)
    s.prefill_with_policy(Q, K, V, ids[:, :n].contiguous(), policy_map)
    dev = Q.device
    Qd = w["Q"][:, n:].transpose(0, 1).contiguous().to(dev)
    Kd = w["K"][:, n:].transpose(0, 1).contiguous().to(dev)
    Vd = w["V"][:, n:].transpose(0, 1).contiguous().to(dev)
    idd = ids[:, n:].transpose(0, 1).contiguous()
    outs = torch.empty(cfg.steps, s.G, cfg.d, dtype=s.tdtype, device=dev)
    for st in range(cfg.steps):
        s.decode(Qd[st], Kd[st], Vd[st], idd[st], n + st, out=outs[st])
    torch.cuda.synchronize()
    return w, s, outs.float().cpu().numpy().astype(np.float64)


def _compare(cfg, policy_map, w, s, outs):
    from oracle import fastgen_oracle as O
    from parity_util import COLSUM_ATOL, RTOL, cache_positions, close, dec_atol
    from synth import punct_ids, special_ids

    from adaptive_head_kv_gb300 import fastgen as fg

    assert fg.fastgen_read_error(s.dev_err) == fg.FG_OK
    assert s.check_guards() == 0
    n = cfg.n
    pol = np.asarray(policy_map, dtype=np.int64)
    keep = s.keep.cpu().numpy()
    kept = s.kept.cpu().numpy()
    colsum = s.colsum.cpu().numpy().astype(np.float64)
    desc = s.descriptors()
    pos = s.pos_pool.cpu().numpy()
    checked = dict(f_heads=0, decode=0, tie_exempt=0)
    for g in range(cfg.G):
        b = g // (cfg.L * cfg.H)
        Qa = w["Q"][g].double().numpy()
        Ka = w["K"][g].double().numpy()
        Va = w["V"][g].double().numpy()
        ids = w["ids"][b]
        r = O.profile_with_policy(int(pol[g]), Qa[:n], Ka[:n], ids, special_ids(), punct_ids(),
                                  cfg.r_l, cfg.r_f)
        if r["colsum"] is not None:
            checked["f_heads"] += 1
            ok = close(colsum[g], r["colsum"], RTOL, COLSUM_ATOL)
            assert ok.all(), (g, np.nonzero(~ok)[0][:5])
            k = O.ratio_count(cfg.r_f, n)
            c = np.sort(r["colsum"])[::-1]
            if 0 < k < n and c[k - 1] - c[k] <= 1e-5 * max(1.0, c[k - 1]):
                checked["tie_exempt"] += 1  # several top-k sets are correct
                assert kept[g] == r["kept"]
                continue
        assert np.array_equal(keep[g], r["keep"]), (g, int(pol[g]))
        assert kept[g] == r["kept"]
        out, fpos = O.decode_head(int(pol[g]), r["keep"], n, O.ratio_count(cfg.r_l, n), ids,
                                  Qa, Ka, Va, special_ids(), punct_ids(), cfg.steps)
        err = np.abs(outs[:, g] - out).max()
        assert err <= dec_atol(cfg.dtype), (g, err)
        assert np.array_equal(cache_positions(desc[g], pos), fpos), g
        checked["decode"] += 1
    return checked


def test_profiled_map_reused_on_another_prompt(tmp_path):
    """Profile prompt 0, save its policy map to JSON, load it and apply it to
    prompt 1 (other ids, queries and keys)."""
    from adaptive_head_kv_gb300.session import load_policy_map, save_policy_map
    from synth import make_workload

    cfg = CONFIGS["tiny"].with_(dtype="bf16", d=128, L=2, H=8, n=300, steps=12)
    w0 = make_workload(cfg, 0)
    p, s0 = _session(cfg, cfg.steps)
    Q, K, V, ids = _device_inputs(w0, cfg.n)
    s0.profile(Q, K, ids[:, :cfg.n].contiguous())
    path = tmp_path / "map.json"
    save_policy_map(path, p, s0.policy)
    pmap = load_policy_map(path, p)
    assert len(set(pmap.tolist())) >= 3, pmap
    w, s, outs = _run_with_map(cfg, pmap, seed=1)
    rep = _compare(cfg, pmap.numpy(), w, s, outs)
    assert rep["f_heads"] >= 2 and rep["decode"] >= cfg.G // 2, rep


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("fp32", 128)])
def test_every_entry_by_hand(dtype, d):
    """A hand-set map with every shortlist entry on every layer."""
    cfg = CONFIGS["tiny"].with_(dtype=dtype, d=d, L=2, H=5, n=257, steps=9)
    pmap = np.array([g % 5 for g in range(cfg.G)], dtype=np.int8)
    w, s, outs = _run_with_map(cfg, pmap, seed=2)
    rep = _compare(cfg, pmap, w, s, outs)
    assert rep["f_heads"] == 2 * cfg.G // 5 and rep["decode"] >= cfg.G - 2, rep


def test_map_without_frequent_entries_skips_the_profiler():
    """Only special / punct / full entries: no head is scored, the keep codes
    follow from the token ids alone."""
    cfg = CONFIGS["tiny"].with_(dtype="bf16", d=128, L=1, H=6, n=200, steps=5)
    pmap = np.array([0, 1, 4, 1, 0, 4], dtype=np.int8)
    w, s, outs = _run_with_map(cfg, pmap, seed=3)
    rep = _compare(cfg, pmap, w, s, outs)
    assert rep["f_heads"] == 0 and rep["decode"] == cfg.G, rep


def test_out_of_range_saved_value_is_reported():
    from adaptive_head_kv_gb300 import fastgen as fg
    from synth import make_workload

    cfg = CONFIGS["tiny"].with_(dtype="bf16", d=128, L=1, H=4, n=130, steps=2)
    w = make_workload(cfg, 0)
    p, s = _session(cfg, cfg.steps)
    Q, K, V, ids = _device_inputs(w, cfg.n)
    s.profile_with_policy(Q, K, ids[:, :cfg.n].contiguous(), [0, 7, 2, 4])
    torch.cuda.synchronize()
    assert fg.fastgen_read_error(s.dev_err) == fg.FG_EINVAL
    keep = s.keep.cpu().numpy()
    assert np.all(keep[1] == fg.FG_KEEP_STATIC)  # read as the full cache


def test_saved_map_with_grouped_keys():
    """A hand-set map on grouped keys (two query heads per key/value head):
    each query head's keep codes, and every member's decode output over the
    group's union cache (largest member policy), against the oracle."""
    from oracle import fastgen_oracle as O
    from parity_util import dec_atol, kv_rows
    from synth import make_workload, punct_ids, special_ids

    from adaptive_head_kv_gb300 import fastgen as fg

    cfg = CONFIGS["tiny"].with_(dtype="bf16", d=128, L=2, H=4, Hkv=2, n=300, steps=10)
    pmap = np.array([0, 4, 1, 2, 3, 0, 2, 1], dtype=np.int8)  # G = 8: every pairing kind
    w = make_workload(cfg, 5)
    n, dev = cfg.n, torch.device("cuda")
    p, s = _session(cfg, cfg.steps)
    sel = kv_rows(cfg)
    Q = w["Q"][:, :n].contiguous().to(dev)
    K = w["K"][sel, :n].contiguous().to(dev)
    V = w["V"][sel, :n].contiguous().to(dev)
    ids = torch.from_numpy(w["ids"]).to(dev)
    s.prefill_with_policy(Q, K, V, ids[:, :n].contiguous(), pmap)
    Qd = w["Q"][:, n:].transpose(0, 1).contiguous().to(dev)
    Kd = w["K"][sel, n:].transpose(0, 1).contiguous().to(dev)
    Vd = w["V"][sel, n:].transpose(0, 1).contiguous().to(dev)
    idd = ids[:, n:].transpose(0, 1).contiguous()
    outs = torch.empty(cfg.steps, s.G, cfg.d, dtype=s.tdtype, device=dev)
    for st in range(cfg.steps):
        s.decode(Qd[st], Kd[st], Vd[st], idd[st], n + st, out=outs[st])
    torch.cuda.synchronize()
    assert fg.fastgen_read_error(s.dev_err) == fg.FG_OK
    assert s.check_guards() == 0
    keep = s.keep.cpu().numpy()
    outs = outs.float().cpu().numpy().astype(np.float64)
    r = cfg.H // cfg.kv_heads
    ids0 = w["ids"][0]
    for c, g0 in enumerate(sel):
        members = list(range(g0, g0 + r))
        Qs = [w["Q"][g].double().numpy() for g in members]
        Ka, Va = w["K"][g0].double().numpy(), w["V"][g0].double().numpy()
        keeps = []
        for g, Qa in zip(members, Qs):
            ora = O.profile_with_policy(int(pmap[g]), Qa[:n], Ka[:n], ids0, special_ids(),
                                        punct_ids(), cfg.r_l, cfg.r_f)
            if ora["colsum"] is not None and _topk_tied(ora["colsum"], O.ratio_count(cfg.r_f, n)):
                # several top-k sets are correct: the GPU's must be one of them
                k = O.ratio_count(cfg.r_f, n)
                spec, punc = O.token_sets(ids0[:n], special_ids(), punct_ids())
                chosen = (keep[g] == O.KEEP_STATIC) & ~(spec | punc)
                others = ~(spec | punc) & ~chosen
                ck = np.sort(ora["colsum"])[::-1][k - 1]
                tol = 2e-5 * max(1.0, ck)
                assert np.all(ora["colsum"][chosen] >= ck - tol), g
                assert np.all(ora["colsum"][others] <= ck + tol), g
                # (the kept count may differ: tied keys inside the window overlap it)
                assert ((keep[g] == O.KEEP_STATIC) & ~(spec | punc)).sum() <= k, g
                keeps.append(keep[g])
                continue
            assert np.array_equal(keep[g], ora["keep"]), g
            keeps.append(ora["keep"])
        gkeep = O.union_keep(keeps)
        gpol = int(max(pmap[g] for g in members))
        out, _ = O.decode_group(gpol, gkeep, n, O.ratio_count(cfg.r_l, n), ids0, Qs, Ka, Va,
                                special_ids(), punct_ids(), cfg.steps)
        for mi, g in enumerate(members):
            err = np.abs(outs[:, g] - out[mi]).max()
            assert err <= dec_atol(cfg.dtype), (c, g, err)


def _topk_tied(colsum, k):
    c = np.sort(colsum)[::-1]
    return 0 < k < c.shape[0] and c[k - 1] - c[k] <= 1e-5 * max(1.0, c[k - 1])



def test_pools_grow_between_prompts():
    """One session, two prompts: the second needs larger pools than the
    first left (all full caches after all special-only ones), so the one-call
    plan + gather reports the size and the session grows the pools and
    gathers again; the second prompt's decode matches the oracle."""
    from synth import make_workload

    cfg = CONFIGS["tiny"].with_(dtype="bf16", d=128, L=1, H=4, n=200, steps=6)
    p, s = _session(cfg, cfg.steps)
    w0 = make_workload(cfg, 6)
    Q, K, V, ids = _device_inputs(w0, cfg.n)
    s.prefill_with_policy(Q, K, V, ids[:, :cfg.n].contiguous(), np.zeros(cfg.G, np.int8))
    small = s.pos_pool.numel()
    full = np.full(cfg.G, 4, dtype=np.int8)
    w = make_workload(cfg, 7)
    Q, K, V, ids = _device_inputs(w, cfg.n)
    s.prefill_with_policy(Q, K, V, ids[:, :cfg.n].contiguous(), full)
    assert s.pos_pool.numel() > small
    dev = Q.device
    n = cfg.n
    Qd = w["Q"][:, n:].transpose(0, 1).contiguous().to(dev)
    Kd = w["K"][:, n:].transpose(0, 1).contiguous().to(dev)
    Vd = w["V"][:, n:].transpose(0, 1).contiguous().to(dev)
    idd = ids[:, n:].transpose(0, 1).contiguous()
    o = torch.empty(cfg.steps, s.G, cfg.d, dtype=s.tdtype, device=dev)
    for st in range(cfg.steps):
        s.decode(Qd[st], Kd[st], Vd[st], idd[st], n + st, out=o[st])
    torch.cuda.synchronize()
    rep = _compare(cfg, full, w, s, o.float().cpu().numpy().astype(np.float64))
    assert rep["decode"] == cfg.G, rep
