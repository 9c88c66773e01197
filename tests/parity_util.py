"""Runs the CUDA path and the oracle on the same seeded workload and compares
them head by head.

Tolerances (stated once, used by every parity test):
  * policies, keep codes, compacted rows and cache positions: exact, except
    that a head is exempt from the policy check when one of its oracle masses
    lies within NEAR of T, and from the kept-set check when its oracle colsum
    gap at the top-k boundary is within NEAR (relative to max(1, value)).
    Exempt heads must still make a valid choice (checked).
  * colsum and masses: |gpu - oracle| <= RTOL |oracle| + ATOL, # every compare() call's counts, printed at the end of the test session
REPORTS: list = []

RTOL = 1e-4.
    The absolute floor covers values below what fp32 sums of probabilities
    resolve (e.g. 1e-40 attention on a masked-out special token).
  * decode outputs: 2e-2 absolute for bf16, 1e-5 for fp32, on every head
    whose cache matches the oracle's.
"""
from __future__ import annotations

import os

import numpy as np
import torch

from oracle import fastgen_oracle as O
from oracle_pool import oracle_job
from synth import make_workload, punct_ids, special_ids

# every compare() call's counts, printed at the end of the test session
REPORTS: list = []

RTOL = 1e-4
COLSUM_ATOL = 1e-6
MASS_ATOL = 1e-7
NEAR = 1e-5


def dec_atol(dtype: str) -> float:
    return 2e-2 if dtype == "bf16" else 1e-5


def run_gpu(cfg, seed=0, max_new=None, T=None, check_pools=True, guard=True):
    """Whole path on the GPU.  Returns host copies of everything compared.
    Every buffer the library writes is guarded by canaries (see session)."""
    from adaptive_head_kv_gb300.session import FastGenSession, make_params

    w = make_workload(cfg, seed)
    n, steps = cfg.n, cfg.steps
    dev = torch.device("cuda")
    sel = kv_rows(cfg)  # the workload lists K/V per query head: one row per cache
    Q = w["Q"][:, :n].contiguous().to(dev)
    K = w["K"][sel, :n].contiguous().to(dev)
    V = w["V"][sel, :n].contiguous().to(dev)
    ids = torch.from_numpy(w["ids"]).to(dev)
    T = cfg.T if T is None else T
    p = make_params(cfg.B, cfg.L, cfg.H, n, cfg.d, cfg.dtype, T, cfg.r_l, cfg.r_f,
                    Hkv=cfg.Hkv)
    s = FastGenSession(p, special_ids(seed), punct_ids(seed),
                       cfg.steps if max_new is None else max_new, guard=guard)
    s.prefill(Q, K, V, ids[:, :n].contiguous())
    torch.cuda.synchronize()
    res = dict(workload=w, policy=s.policy.cpu().numpy().astype(int),
               mass=s.mass.cpu().numpy().astype(np.float64), cost=s.cost.cpu().numpy(),
               colsum=s.colsum.cpu().numpy().astype(np.float64), keep=s.keep.cpu().numpy(),
               kept=s.kept.cpu().numpy(), info=s.info)
    if check_pools:
        res["desc0"] = s.descriptors()
        res["pos0"] = s.pos_pool.cpu().numpy()
        res["Kp0"] = s.K_pool.cpu()
        res["Vp0"] = s.V_pool.cpu()
    Qd = w["Q"][:, n:].transpose(0, 1).contiguous().to(dev)
    Kd = w["K"][sel, n:].transpose(0, 1).contiguous().to(dev)
    Vd = w["V"][sel, n:].transpose(0, 1).contiguous().to(dev)
    idd = ids[:, n:].transpose(0, 1).contiguous()
    outs = torch.empty(steps, s.G, cfg.d, dtype=s.tdtype, device=dev)
    for st in range(steps):
        s.decode(Qd[st], Kd[st], Vd[st], idd[st], n + st, out=outs[st])
    torch.cuda.synchronize()
    res["out"] = outs.float().cpu().numpy().astype(np.float64)
    res["dev_err"] = int(s.dev_err.item())
    res["guards_broken"] = s.check_guards() if guard else 0
    res["desc1"] = s.descriptors()
    res["pos1"] = s.pos_pool.cpu().numpy()
    res["session"] = s
    return res


def kv_rows(cfg):
    """For each cache (key/value head), the first query head of its group."""
    r = cfg.H // cfg.kv_heads
    return [(c // cfg.kv_heads) * cfg.H + (c % cfg.kv_heads) * r for c in range(cfg.Gkv)]


def oracle_head(cfg, w, idx, T=None):
    """Oracle profile + decode of the head at position idx of the workload."""
    g = int(w["heads"][idx])
    b = g // (cfg.L * cfg.H)
    n, steps = cfg.n, cfg.steps
    Qa = w["Q"][idx].double().numpy()
    Ka = w["K"][idx].double().numpy()
    Va = w["V"][idx].double().numpy()
    ids = w["ids"][b]
    T = float(np.float32(cfg.T if T is None else T))
    r = O.profile_head(Qa[:n], Ka[:n], ids, special_ids(), punct_ids(), T, cfg.r_l, cfg.r_f)
    out, pos = O.decode_head(r["policy"], r["keep"], n, r["w"], ids, Qa, Ka, Va, special_ids(),
                             punct_ids(), steps)
    r["out"], r["final_pos"] = out, pos
    r.pop("A")
    return r


def oracle_heads(cfg, w, idxs, T=None, long_prompt=False, procs=None):
    """Oracle results of several heads of the workload, computed in parallel
    by spawned worker processes (never forked: the caller holds a CUDA
    context).  long_prompt selects the row-block profile (prompts whose dense
    map does not fit in host memory).  Returns {idx: result}."""
    import multiprocessing as mp

    T = float(np.float32(cfg.T if T is None else T))
    jobs = []
    for idx in idxs:
        g = int(w["heads"][idx])
        b = g // (cfg.L * cfg.H)
        jobs.append((w["Q"][idx].double().numpy(), w["K"][idx].double().numpy(),
                     w["V"][idx].double().numpy(), w["ids"][b], cfg.n, cfg.steps, T, cfg.r_l,
                     cfg.r_f, long_prompt))
    procs = procs or max(1, min(len(jobs), (os.cpu_count() or 2) // 2))
    threads = str(max(1, (os.cpu_count() or 1) // procs))
    keys = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in keys}
    os.environ.update({k: threads for k in keys})  # read by the workers' BLAS at start-up
    try:
        with mp.get_context("spawn").Pool(procs) as pool:
            res = pool.map(oracle_job, jobs, chunksize=1)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return dict(zip(idxs, res))


def close(a, b, rtol, atol):
    return np.abs(a - b) <= rtol * np.abs(b) + atol


def policy_exempt(ora, T) -> bool:
    return bool(np.any(np.abs(ora["mass"][:4] - T) < NEAR))


def topk_exempt(ora) -> bool:
    k, c = ora["k"], np.sort(ora["colsum"])[::-1]
    if k <= 0 or k >= c.shape[0]:
        return False
    return bool(c[k - 1] - c[k] <= NEAR * max(1.0, c[k - 1]))


def cache_positions(desc, pos_pool):
    st = pos_pool[desc.off: desc.off + desc.n_static]
    ring = pos_pool[desc.win_off: desc.win_off + desc.w]
    return np.array(sorted(list(st) + [x for x in ring if x >= 0]), dtype=np.int64)


def compare(cfg, gpu, heads_idx, T=None, report=None, oracle=None):
    """Compares sampled heads (indices into the workload) and the all-head
    invariants.  `oracle` optionally holds the heads' oracle results
    ({idx: result}, e.g. from oracle_heads); otherwise each head's is
    computed here.  Returns a dict of counts; raises AssertionError on a miss."""
    w = gpu["workload"]
    T = float(np.float32(cfg.T if T is None else T))
    n = cfg.n
    rep = dict(checked=0, policy_exempt=0, topk_exempt=0, decode_checked=0)
    assert gpu.get("guards_broken", 0) == 0, "a kernel wrote outside its buffer"
    # invariants over every head
    G = gpu["policy"].shape[0]
    assert np.all((gpu["policy"] >= 0) & (gpu["policy"] <= 4))
    assert np.allclose(gpu["colsum"].sum(axis=1), n, rtol=1e-4, atol=0), "row sums of A are 1"
    assert np.all(gpu["mass"][:, 4] == 1.0)
    assert np.all(np.diff(gpu["mass"], axis=1) >= -1e-6)
    assert np.all(np.diff(gpu["cost"], axis=1) >= 0)
    assert np.array_equal(gpu["kept"], gpu["cost"][np.arange(G), gpu["policy"]])
    assert np.array_equal(gpu["kept"], (gpu["keep"] != 0).sum(axis=1))
    for p in range(4):  # the chosen entry is the first whose own mass reaches T
        chose = gpu["policy"] == p
        assert np.all(gpu["mass"][chose, p] >= T)
        assert np.all(gpu["mass"][gpu["policy"] > p, p] < T)
    atol_dec = dec_atol(cfg.dtype)
    for idx in heads_idx:
        g = int(w["heads"][idx])
        ora = oracle[idx] if oracle is not None else oracle_head(cfg, w, idx, T)
        rep["checked"] += 1
        cs_ok = close(gpu["colsum"][g], ora["colsum"], RTOL, COLSUM_ATOL)
        assert cs_ok.all(), (g, np.nonzero(~cs_ok)[0][:5])
        m_ok = close(gpu["mass"][g], ora["mass"], RTOL, MASS_ATOL)
        assert m_ok.all(), (g, gpu["mass"][g], ora["mass"])
        pe, te = policy_exempt(ora, T), topk_exempt(ora)
        rep["policy_exempt"] += pe
        rep["topk_exempt"] += te
        assert gpu["cost"][g][0] == ora["cost"][0] and gpu["cost"][g][1] == ora["cost"][1]
        assert gpu["cost"][g][4] == ora["cost"][4]
        if not te:
            assert np.array_equal(gpu["cost"][g], ora["cost"]), (g, gpu["cost"][g], ora["cost"])
        if pe:
            p = gpu["policy"][g]
            assert p == 4 or ora["mass"][p] >= T - NEAR
            assert all(ora["mass"][q] < T + NEAR for q in range(p))
            continue
        assert gpu["policy"][g] == ora["policy"], (g, gpu["policy"][g], ora["policy"], ora["mass"])
        uses_f = ora["policy"] in (O.P_SPF, O.P_SPFL)
        if te and uses_f:
            # several top-k sets are correct: the GPU's must be one of them
            spec, punc = O.token_sets(w["ids"][g // (cfg.L * cfg.H)][:n], special_ids(),
                                      punct_ids())
            chosen_f = (gpu["keep"][g] == O.KEEP_STATIC) & ~(spec | punc)
            ck = np.sort(ora["colsum"])[::-1][ora["k"] - 1]
            tol = 2 * NEAR * max(1.0, ck)
            others = ~(spec | punc) & ~chosen_f
            assert np.all(ora["colsum"][chosen_f] >= ck - tol), g
            assert np.all(ora["colsum"][others] <= ck + tol), g
            continue
        assert np.array_equal(gpu["keep"][g], ora["keep"]), g
        if "desc0" in gpu:
            d0 = gpu["desc0"][g]
            sp = np.nonzero(ora["keep"] == O.KEEP_STATIC)[0]
            assert d0.n_static == len(sp) and d0.policy == ora["policy"]
            assert np.array_equal(gpu["pos0"][d0.off: d0.off + len(sp)], sp)
            Kh = w["K"][idx]
            Vh = w["V"][idx]
            assert torch.equal(gpu["Kp0"][d0.off: d0.off + len(sp)], Kh[sp])
            assert torch.equal(gpu["Vp0"][d0.off: d0.off + len(sp)], Vh[sp])
            if ora["policy"] == O.P_SPFL and ora["w"] > 0:
                wp = np.nonzero(ora["keep"] == O.KEEP_WINDOW)[0]
                ring = gpu["pos0"][d0.win_off: d0.win_off + d0.w]
                want = np.full(d0.w, -1)
                want[wp % ora["w"]] = wp
                assert np.array_equal(ring, want), g
                assert torch.equal(gpu["Kp0"][d0.win_off + wp % ora["w"]], Kh[wp])
        # decode: every step's output and the final cache membership
        err = np.abs(gpu["out"][:, g] - ora["out"]).max() if cfg.steps else 0.0
        assert err <= atol_dec, (g, err)
        if cfg.steps:
            assert np.array_equal(cache_positions(gpu["desc1"][g], gpu["pos1"]), ora["final_pos"]), g
        rep["decode_checked"] += 1
    if report is not None:
        report.update(rep)
    REPORTS.append((f"{cfg.name} B={cfg.B} L={cfg.L} H={cfg.H} n={cfg.n} d={cfg.d} "
                    f"{cfg.dtype} T={T:g}", dict(rep)))
    return rep


def sample_heads(cfg, types, count, seed=1):
    """Head indices covering every head type, layer 0 and the last layer."""
    rng = np.random.default_rng(seed)
    G = cfg.G
    pick = set()
    for want in range(4):
        cand = [g for g in range(G) if types[(g // cfg.H) % cfg.L, g % cfg.H] == want]
        pick.update(rng.choice(cand, size=min(len(cand), max(1, count // 8)), replace=False).tolist()
                    if cand else [])
    pick.update(range(min(cfg.H, 2)))
    last = (cfg.L - 1) * cfg.H
    pick.update(range(last, min(last + 2, G)))
    while len(pick) < min(count, G):
        pick.add(int(rng.integers(0, G)))
    return sorted(pick)


def compare_groups(cfg, gpu, T=None):
    """Grouped-query parity: every query head's profile as in compare(), and
    for each cache the union of its members' caches, the group policy, the
    compacted rows and every member's decode outputs (oracle decode_group).
    A group with an exempt member is checked for its members' profiles only."""
    w = gpu["workload"]
    T = float(np.float32(cfg.T if T is None else T))
    n, r = cfg.n, cfg.H // cfg.kv_heads
    rep = dict(groups=0, groups_exempt=0)
    compare(cfg, gpu, [], T=T)  # all-head invariants, guards
    for c, g0 in enumerate(kv_rows(cfg)):
        members = list(range(g0, g0 + r))
        b = g0 // (cfg.L * cfg.H)
        Qs = [w["Q"][g].double().numpy() for g in members]
        Ka = w["K"][g0].double().numpy()
        Va = w["V"][g0].double().numpy()
        ids = w["ids"][b]
        res, keep, pol = O.profile_group([q[:n] for q in Qs], Ka[:n], ids, special_ids(),
                                         punct_ids(), T, cfg.r_l, cfg.r_f)
        exempt = False
        for g, ora in zip(members, res):
            assert close(gpu["colsum"][g], ora["colsum"], RTOL, COLSUM_ATOL).all(), g
            assert close(gpu["mass"][g], ora["mass"], RTOL, MASS_ATOL).all(), g
            if policy_exempt(ora, T) or (topk_exempt(ora) and ora["policy"] in (2, 3)):
                exempt = True
                continue
            assert gpu["policy"][g] == ora["policy"], (g, gpu["policy"][g], ora["policy"])
            assert np.array_equal(gpu["keep"][g], ora["keep"]), g
        rep["groups"] += 1
        if exempt:
            rep["groups_exempt"] += 1
            continue
        d0 = gpu["desc0"][c]
        sp = np.nonzero(keep == O.KEEP_STATIC)[0]
        assert d0.policy == pol and d0.n_static == len(sp), (c, d0.policy, pol)
        assert np.array_equal(gpu["pos0"][d0.off: d0.off + len(sp)], sp), c
        assert torch.equal(gpu["Kp0"][d0.off: d0.off + len(sp)], w["K"][g0][sp])
        wl = res[0]["w"]
        out, pos = O.decode_group(pol, keep, n, wl, ids, Qs, Ka, Va, special_ids(), punct_ids(),
                                  cfg.steps)
        for mi, g in enumerate(members):
            err = np.abs(gpu["out"][:, g] - out[mi]).max()
            assert err <= dec_atol(cfg.dtype), (c, g, err)
        assert np.array_equal(cache_positions(gpu["desc1"][c], gpu["pos1"]), pos), c
    return rep
