"""Benchmark of the FastGen hot path on the Llama-1-65B attention shape.

One step = profile every head of the prompt, plan + compact the per-head
caches, then `steps` generation steps over those caches, all on one GPU with
the inputs resident in HBM (Q/K/V and the caches are each larger than L2, so
no flush is needed between steps).  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config llama65b]
  python bench.py --impl reference ...   # the fp64 CPU oracle on the host cores

Under torchrun each rank runs its own replica (seed = rank): the heads are
independent, so there is no data-path collective; timings are reduced with
a max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "profile+compact prompt tok/s; compressed-cache decode tok/s and HBM GB/s"


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
_CSRC = os.path.join("adaptive_head_kv_gb300", "csrc")
# the kernels behind each roofline entry, and the sources that define them
KERNEL_GROUPS = {
    "decode": dict(patterns=("split_kernel", "combine_kernel"), calls="split_kernel",
                   sources=("fg_decode.cu", "fg_common.cuh", "fg_internal.h")),
    "profile": dict(patterns=("profile_tc_kernel", "select_kernel", "token_class_kernel"),
                    calls="select_kernel",
                    sources=("fg_profile_tc.cu", "fg_sm100.cuh", "fg_select.cu", "fg_common.cuh",
                             "fg_internal.h")),
}


def source_digest(group):
    import hashlib

    h = hashlib.sha256()
    for f in KERNEL_GROUPS[group]["sources"]:
        with open(os.path.join(ROOT, _CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def record_traffic(csv_path, workload, command, scale=None, measured_on=None):
    """Writes DRAM bytes per call of each kernel group from an ncu CSV (metrics
    dram__bytes_read.sum and dram__bytes_write.sum), tagged with the sources'
    digest so that a later kernel change voids the figure.  With `scale`
    ({group: factor}), the figures were captured on the smaller workload
    `measured_on` and are scaled to `workload` by the ratio of the units
    each call processes (recorded with the figure)."""
    import csv

    rows = list(csv.reader(open(csv_path)))
    hi = next(i for i, r in enumerate(rows) if "Kernel Name" in r)
    h = rows[hi]
    ki, mi, vi, ui = (h.index(x) for x in ("Kernel Name", "Metric Name", "Metric Value",
                                            "Metric Unit"))
    unit = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    out = {}
    try:  # figures of other groups recorded earlier stay
        with open(TRAFFIC_FILE) as f:
            out = json.load(f)
    except (OSError, ValueError):
        out = {}
    for group, spec in KERNEL_GROUPS.items():
        if scale and group not in scale:
            continue
        total, calls = 0.0, 0
        for r in rows[hi + 1:]:
            if len(r) != len(h) or not any(p in r[ki] for p in spec["patterns"]):
                continue
            if r[mi] in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
                total += float(r[vi].replace(",", "")) * unit[r[ui]]
            if r[mi] == "dram__bytes_read.sum" and spec["calls"] in r[ki]:
                calls += 1
        if calls:
            f = (scale or {}).get(group, 1.0)
            out[group] = {"bytes_per_call": total / calls * f, "calls": calls,
                          "workload": workload, "source_sha256": source_digest(group),
                          "command": command}
            if scale:
                out[group].update(measured_on=measured_on, measured_bytes_per_call=total / calls,
                                  scale=f)
    os.makedirs(os.path.dirname(TRAFFIC_FILE), exist_ok=True)
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(out, f, indent=1)
    print(json.dumps(out, indent=1))


def load_traffic(group, workload):
    """Measured DRAM bytes per call, or None if absent, taken on another
    workload, or taken on kernels that have changed since."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)[group]
    except (OSError, KeyError, ValueError):
        return None
    if rec.get("workload") != workload or rec.get("source_sha256") != source_digest(group):
        return None
    return rec["bytes_per_call"]


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return dict(hbm=pk["hbm_gbs"], bf16=pk["bf16_tflops"],
                    bf16_sus=pk.get("bf16_tflops_sustained", pk["bf16_tflops"]), src="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


class Clocks:
    """Samples SM clocks and throttle reasons while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)  # the sampler is running before the timed region starts
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def group_caches(cfg, policy, keep):
    """Per cache (key/value head): the group policy (largest member policy)
    and the union of the members' keep codes; without groups, the heads'."""
    r = cfg.H // cfg.kv_heads
    if r == 1:
        return policy, keep
    pol = policy.reshape(-1, r).max(axis=1)
    k = keep.reshape(-1, r, keep.shape[1])
    static = (k == 1).any(axis=1)
    window = (k == 2).any(axis=1)
    return pol, np.where(static, 1, np.where(window, 2, 0)).astype(np.uint8)


def cache_rows_per_step(cfg, policy, keep, ids, special, punct):
    """Rows each generation step attends over, summed over caches
    (bookkeeping for the roofline's algorithmic bytes; follows the documented
    placement rule from the profile's outputs).  policy/keep: per cache."""
    n, steps = cfg.n, cfg.steps
    C, HL = keep.shape[0], cfg.L * cfg.kv_heads
    w = int(np.ceil(float(np.float32(cfg.r_l)) * n))
    b_of = np.arange(C) // HL
    dec = ids[:, n:n + steps]
    is_s = np.isin(dec, special)
    is_p = np.isin(dec, punct)
    pol = policy.astype(np.int64)[:, None]
    st = np.where(pol == 4, True, np.where(pol == 0, is_s[b_of], (is_s | is_p)[b_of]))
    n_static0 = (keep == 1).sum(axis=1)
    static_t = n_static0[:, None] + np.cumsum(st, axis=1)  # [C, steps]
    ring_ind = np.zeros((C, n + steps), dtype=np.int64)
    ring_ind[:, :n] = keep == 2
    ring_ind[:, n:] = (pol == 3) & ~st & (w > 0)
    csum = np.concatenate([np.zeros((C, 1), np.int64), np.cumsum(ring_ind, axis=1)], axis=1)
    t = np.arange(n, n + steps)
    lo = np.maximum(t - w + 1, 0)
    ring_t = csum[:, t + 1] - csum[:, lo]
    ring_t = np.where(pol == 3, ring_t, 0)
    return static_t.sum(axis=0) + ring_t.sum(axis=0), ring_t.sum(axis=0)


def run_ours(args, cfg, rank, world):
    import torch

    from adaptive_head_kv_gb300 import fastgen as fg
    from adaptive_head_kv_gb300.session import FastGenSession, make_params
    from synth import make_workload_split, punct_ids, special_ids

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    dev = torch.device("cuda")
    n, steps, G, d = cfg.n, cfg.steps, cfg.G, cfg.d
    fg.lib()
    w = make_workload_split(cfg, seed=rank, pin=True)
    hQ, hK, hV, hq, hk, hv = (w[x] for x in ("Q", "K", "V", "q", "k", "v"))
    ids_np = w["ids"]
    hids = torch.from_numpy(ids_np[:, :n].copy()).pin_memory()
    hdec_ids = torch.from_numpy(np.ascontiguousarray(ids_np[:, n:].T)).pin_memory()
    del w
    Q, K, V = hQ.to(dev), hK.to(dev), hV.to(dev)
    q, k, v = hq.to(dev), hk.to(dev), hv.to(dev)
    ids, dec_ids = hids.to(dev), hdec_ids.to(dev)
    p = make_params(cfg.B, cfg.L, cfg.H, n, d, cfg.dtype, cfg.T, cfg.r_l, cfg.r_f, Hkv=cfg.Hkv)
    s = FastGenSession(p, special_ids(rank), punct_ids(rank), steps, device=dev,
                       refresh_period=args.refresh_period)
    stream = torch.cuda.current_stream()

    graph = None

    def one_step(record):
        e0, e1, e2, e3 = (torch.cuda.Event(enable_timing=True) for _ in range(4))
        e0.record(stream)
        s.profile(Q, K, ids)
        e1.record(stream)
        s.compact(K, V)
        e2.record(stream)
        if graph is not None:  # the whole decode loop as one graph launch
            graph.replay()
        else:
            for st in range(steps):
                s.decode(q[st], k[st], v[st], dec_ids[st], n + st)
        e3.record(stream)
        return e0, e1, e2, e3

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        one_step(False)
    if not args.no_graph:
        # capture the decode loop once (same plan and pools every step), then
        # warm the graph up like the rest
        torch.cuda.synchronize()
        graph, _ = s.capture_decode(q, k, v, dec_ids, n)
        for _ in range(2):
            one_step(False)
    barrier()
    per = []
    with Clocks(torch.cuda.current_device()) as clk:
        barrier()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for _ in range(args.steps):
            per.append(one_step(True))
        t_end.record(stream)
        barrier()
    total_ms = t_start.elapsed_time(t_end)
    prof_ms = np.mean([a.elapsed_time(b) for a, b, c, e in per])
    comp_ms = np.mean([b.elapsed_time(c) for a, b, c, e in per])
    decode_ms = np.mean([c.elapsed_time(e) for a, b, c, e in per])
    step_ms = np.mean([a.elapsed_time(e) for a, b, c, e in per])
    dec_ms = np.full(steps, decode_ms / steps)  # per decode call, averaged over the loop
    assert fg.fastgen_read_error(s.dev_err) == fg.FG_OK

    # algorithmic work
    policy = s.policy.cpu().numpy()
    keep = s.keep.cpu().numpy()
    cpol, ckeep = group_caches(cfg, policy, keep)
    rows_t, ring_t = cache_rows_per_step(cfg, cpol, ckeep, ids_np, special_ids(rank),
                                         punct_ids(rank))
    eb = 2 if cfg.dtype == "bf16" else 4
    Gkv = cfg.Gkv
    # K/V rows of every cache + q and out per query head + k_new, v_new per
    # cache + ring positions + descriptors
    dec_bytes_t = (rows_t * d * 2 * eb + G * d * eb * 2 + Gkv * d * eb * 2 + ring_t * 4
                   + Gkv * 40)
    if args.refresh_period:  # per cached row: its score written and read, its acc updated
        dec_bytes_t = dec_bytes_t + rows_t * 16
    dec_gbs = dec_bytes_t.sum() / (dec_ms.sum() * 1e-3) / 1e9
    prof_flops = 2.0 * n * (n + 1) * d * G
    kept_rows = int((ckeep != 0).sum())
    comp_bytes = kept_rows * d * 2 * eb * 2 + G * n + Gkv * 40
    pmap = pattn = None
    if not args.no_extras:
        pmap = run_policy_map(args, s, Q, K, V, ids, stream)
        pattn = run_prompt_attention(args, s, cfg, Q, K, V, ids, stream)
    return dict(cfg=cfg, prof_ms=prof_ms, comp_ms=comp_ms, decode_ms=decode_ms, step_ms=step_ms,
                total_ms=total_ms, dec_ms=dec_ms, dec_bytes=float(dec_bytes_t.mean()),
                dec_gbs=dec_gbs, prof_flops=prof_flops, comp_bytes=comp_bytes,
                kept_frac=kept_rows / (Gkv * n), clocks=clk.summary(), policy_map=pmap,
                prompt_attention=pattn,
                e2e=run_e2e(args, s, cfg, hQ, hK, hV, hids, hq, hk, hv, hdec_ids, stream))


def run_policy_map(args, s, Q, K, V, ids, stream):
    """The prompt phase under a saved head-policy map (the policy just
    profiled, reused on the same prompt): profile_with_policy + plan +
    compact, timed like the main loop.  Reported beside the main line; not
    part of its value."""
    import torch

    from adaptive_head_kv_gb300 import fastgen as fg

    pmap = s.policy.clone()
    keep0 = s.keep.clone()
    scored = int(((pmap == fg.FG_POLICY_SPF) | (pmap == fg.FG_POLICY_SPFL)).sum().item())
    for _ in range(3):
        s.profile_with_policy(Q, K, ids, pmap)
        s.compact(K, V)
    torch.cuda.synchronize()
    per = []
    for _ in range(max(args.steps, 3)):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record(stream)
        s.profile_with_policy(Q, K, ids, pmap)
        e[1].record(stream)
        s.compact(K, V)
        e[2].record(stream)
        per.append(e)
    torch.cuda.synchronize()
    assert fg.fastgen_read_error(s.dev_err) == fg.FG_OK
    same = float((s.keep == keep0).all(dim=1).float().mean().item())
    prof = float(np.mean([a.elapsed_time(b) for a, b, c in per]))
    comp = float(np.mean([b.elapsed_time(c) for a, b, c in per]))
    return dict(profile_ms=prof, compact_plan_ms=comp, scored_heads=scored,
                heads=int(pmap.numel()), keep_unchanged_fraction=same)


def run_prompt_attention(args, s, cfg, Q, K, V, ids, stream):
    """fastgen_profile_attn (the profile plus the prompt attention output
    A V) against fastgen_profile on the same prompt; the difference is the
    attention-output pass.  Reported beside the main line."""
    import torch

    from adaptive_head_kv_gb300 import fastgen as fg

    out = torch.empty((cfg.G, cfg.n, cfg.d), dtype=s.tdtype, device=Q.device)
    for _ in range(3):
        s.profile_attn(Q, K, V, ids, out)
        s.profile(Q, K, ids)
    torch.cuda.synchronize()
    per = []
    for _ in range(max(args.steps, 3)):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record(stream)
        s.profile_attn(Q, K, V, ids, out)
        e[1].record(stream)
        s.profile(Q, K, ids)
        e[2].record(stream)
        per.append(e)
    torch.cuda.synchronize()
    assert fg.fastgen_read_error(s.dev_err) == fg.FG_OK
    with_attn = float(np.mean([a.elapsed_time(b) for a, b, c in per]))
    plain = float(np.mean([b.elapsed_time(c) for a, b, c in per]))
    attn_ms = with_attn - plain
    # causal Q K^T and P V: 2 * d * n(n+1)/2 flops each per head
    flops = 2.0 * cfg.d * cfg.n * (cfg.n + 1) * cfg.G
    del out
    return dict(profile_attn_ms=with_attn, profile_ms=plain, attention_pass_ms=attn_ms,
                attention_pass_tflops=flops / (attn_ms * 1e-3) / 1e12 if attn_ms > 0 else None)


def run_e2e(args, s, cfg, hQ, hK, hV, hids, hq, hk, hv, hdec_ids, stream):
    """Same metric through the public calls with host buffers: every step
    copies its inputs from pinned host memory and reads its results back."""
    import torch

    dev = torch.device("cuda")
    n, steps = cfg.n, cfg.steps
    hpol = torch.empty(s.G, dtype=torch.int8).pin_memory()
    hout = torch.empty(steps, s.G, cfg.d, dtype=s.tdtype).pin_memory()
    Q, K, V = (torch.empty_like(x, device=dev) for x in (hQ, hK, hV))
    ids = torch.empty_like(hids, device=dev)
    # per-step inputs and outputs are double-buffered: the copies of step t+1
    # and the read-back of step t-1 overlap the decode of step t
    bufs = [(torch.empty(s.G, cfg.d, dtype=s.tdtype, device=dev),
             torch.empty(s.Gkv, cfg.d, dtype=s.tdtype, device=dev),
             torch.empty(s.Gkv, cfg.d, dtype=s.tdtype, device=dev),
             torch.empty(cfg.B, dtype=torch.int32, device=dev),
             torch.empty(s.G, cfg.d, dtype=s.tdtype, device=dev)) for _ in range(2)]
    cp_in, cp_out = torch.cuda.Stream(), torch.cuda.Stream()

    def step():
        a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        a.record(stream)
        s.prefill_host(hQ, hK, hV, hids, Q, K, V, ids)
        hpol.copy_(s.policy, non_blocking=True)
        b.record(stream)
        ready = [torch.cuda.Event(), torch.cuda.Event()]
        used = [torch.cuda.Event(), torch.cuda.Event()]
        read = [torch.cuda.Event(), torch.cuda.Event()]

        def stage(st, i):
            if st >= 2:  # buffer i is free once the decode of step st - 2 has read it
                cp_in.wait_event(used[i])
            with torch.cuda.stream(cp_in):
                for dst, src in zip(bufs[i][:4], (hq[st], hk[st], hv[st], hdec_ids[st])):
                    dst.copy_(src, non_blocking=True)
                ready[i].record(cp_in)

        stage(0, 0)
        for st in range(steps):
            i = st % 2
            if st + 1 < steps:
                stage(st + 1, 1 - i)
            stream.wait_event(ready[i])
            if st >= 2:
                stream.wait_event(read[i])  # the output buffer has been read back
            qb, kb, vb, ib, ob = bufs[i]
            s.decode(qb, kb, vb, ib, n + st, out=ob)
            used[i].record(stream)
            cp_out.wait_event(used[i])
            with torch.cuda.stream(cp_out):
                hout[st].copy_(ob, non_blocking=True)
                read[i].record(cp_out)
        stream.wait_stream(cp_out)
        c.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b), b.elapsed_time(c)

    for _ in range(max(1, min(args.warmup, 2))):
        step()
    pre, dec = zip(*[step() for _ in range(max(1, min(args.steps, 3)))])
    nb = lambda t: t.numel() * t.element_size()
    return dict(prefill_ms=float(np.mean(pre)), decode_ms=float(np.mean(dec)),
                h2d=nb(hQ) + nb(hK) + nb(hV) + nb(hids),
                d2h=nb(hpol),
                dec_h2d=nb(hq) + nb(hk) + nb(hv) + nb(hdec_ids),
                dec_d2h=nb(hout))


def oracle_sample(cfg, heads, seed=0, budget_s=None):
    """Times the oracle (as it stands) on `heads` of the workload: profile,
    compaction and all decode steps per head, heads one after another.
    Stops early once `budget_s` seconds of oracle time are spent (at least
    one head).  Returns (profile+compact s, decode s, heads timed)."""
    from oracle import fastgen_oracle as O
    from synth import make_workload, punct_ids, special_ids

    w = make_workload(cfg, seed, heads=heads, threads=4)
    n, steps = cfg.n, cfg.steps
    T = float(np.float32(cfg.T))
    t_pc = t_dec = 0.0
    done = 0
    for i, g in enumerate(heads):
        b = int(g) // (cfg.L * cfg.H)
        Qa, Ka, Va = (w[x][i].double().numpy() for x in "QKV")
        ids = w["ids"][b]
        t0 = time.perf_counter()
        r = O.profile_head(Qa[:n], Ka[:n], ids, special_ids(seed), punct_ids(seed), T,
                           cfg.r_l, cfg.r_f)
        O.compact_head(Ka[:n], Va[:n], r["keep"])
        t1 = time.perf_counter()
        O.decode_head(r["policy"], r["keep"], n, r["w"], ids, Qa, Ka, Va, special_ids(seed),
                      punct_ids(seed), steps)
        t2 = time.perf_counter()
        t_pc += t1 - t0
        t_dec += t2 - t1
        done += 1
        if budget_s is not None and t_pc + t_dec >= budget_s:
            break
    return t_pc, t_dec, done


def blas_threads():
    """Threads of numpy's BLAS pool: the most threads the oracle uses at a
    time (its matrix products); every other oracle step is single-threaded.
    Asked of threadpoolctl where installed, else of the OpenBLAS library
    loaded in this process (its documented openblas_get_num_threads call)."""
    try:
        from threadpoolctl import threadpool_info

        return max([i.get("num_threads", 1) for i in threadpool_info()
                    if i.get("user_api") == "blas"] + [1])
    except Exception:
        pass
    import ctypes

    np.ones((2, 2)) @ np.ones((2, 2))  # BLAS is loaded
    try:
        libs = sorted({f[-1] for f in (l.split() for l in open("/proc/self/maps"))
                       if len(f) >= 6 and "openblas" in f[-1].lower() and ".so" in f[-1]})
    except OSError:
        libs = []
    for path in libs:
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for name in ("scipy_openblas_get_num_threads64_", "openblas_get_num_threads64_",
                     "scipy_openblas_get_num_threads", "openblas_get_num_threads"):
            fn = getattr(lib, name, None)
            if fn is not None:
                fn.restype = ctypes.c_int
                return max(1, int(fn()))
    return os.cpu_count() or 1


def cpu_baseline(cfg, max_heads=48, budget_s=20.0):
    rng = np.random.default_rng(123)
    heads = rng.choice(cfg.G, size=min(max_heads, cfg.G), replace=False).tolist()
    t_pc, t_dec, done = oracle_sample(cfg, heads, budget_s=budget_s)
    scale = cfg.G / done
    return {"value": cfg.B * cfg.n / (t_pc * scale), "unit": "tok/s", "cores": blas_threads(),
            "host_cores": os.cpu_count(), "kind": "oracle",
            "threads": "heads one after another; BLAS threads inside the matrix products, "
                       "one thread elsewhere",
            "decode_tok_s": cfg.B * cfg.steps / (t_dec * scale),
            "sample": f"{done} of {cfg.G} heads of {cfg.name} (profile+compact+{cfg.steps} "
                      f"decode steps each, {t_pc + t_dec:.1f} s), extrapolated linearly in heads"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="llama65b",
                    help="workload (default: the largest single-GPU configuration, "
                         "Llama-1-65B attention: 40960 heads, n = 2048, 1024 decode steps)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--T", type=float, default=None, help="override the recover ratio")
    ap.add_argument("--hkv", type=int, default=0,
                    help="key/value heads per layer (grouped-query attention); 0 = H")
    ap.add_argument("--refresh-period", type=int, default=0,
                    help="decode with the opt-in refresh of the frequent sets every P steps "
                         "(fastgen_decode_attn_refresh); 0 = the frozen sets (default)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch every decode call from the host instead of one CUDA graph")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the side measurements (saved policy map, prompt attention "
                         "output), e.g. for DRAM captures of the main step's kernels")
    ap.add_argument("--layers", type=int, default=0,
                    help="override the layer count (smaller cases for profiler captures)")
    ap.add_argument("--record-traffic", metavar="NCU_CSV",
                    help="write profiles/traffic.json from an ncu CSV of DRAM byte counters")
    ap.add_argument("--traffic-command", default="",
                    help="the command that produced the CSV (stored with the figures)")
    ap.add_argument("--traffic-scale", default="",
                    help="group=factor,...: the CSV was captured on a smaller case of the "
                         "workload; scale each group's bytes by the ratio of units per call")
    ap.add_argument("--traffic-measured-on", default="",
                    help="the smaller workload the scaled CSV was captured on")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    from synth import CONFIGS

    cfg = CONFIGS[args.config]
    if args.layers:
        cfg = cfg.with_(L=args.layers, name=f"{cfg.name}_L{args.layers}")
    if args.T is not None:
        cfg = cfg.with_(T=args.T, name=f"{cfg.name}_T{args.T:g}")
    if args.hkv:
        cfg = cfg.with_(Hkv=args.hkv, name=f"{cfg.name}_kv{args.hkv}")
    if args.record_traffic:
        scale = {k: float(v) for k, v in (x.split("=") for x in args.traffic_scale.split(",")
                                          if x)} or None
        record_traffic(args.record_traffic, cfg.name, args.traffic_command, scale,
                       args.traffic_measured_on or None)
        return
    if args.impl == "reference":
        if rank != 0:
            return
        run_reference(args, cfg, world)
        return

    import torch

    if world > 1:
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    r = run_ours(args, cfg, rank, world)
    step_ms, prompt_ms, decode_ms, dec_launch_ms = reduce_max(
        [r["step_ms"], r["prof_ms"] + r["comp_ms"], r["decode_ms"], r["dec_ms"].mean()], world,
        "cuda")
    if rank != 0:
        torch.distributed.destroy_process_group()
        return
    pk = load_peaks()
    prompt_tok_s = world * cfg.B * cfg.n / (prompt_ms * 1e-3)
    decode_tok_s = world * cfg.B * cfg.steps / (decode_ms * 1e-3)
    dec_ach = r["dec_bytes"] / (dec_launch_ms * 1e-3) / 1e9
    prof_ach = r["prof_flops"] / (r["prof_ms"] * 1e-3) / 1e12
    dec_roof = {"kernel": "fastgen_decode_attn (split + combine)", "bound": "hbm",
                "achieved": dec_ach, "peak": pk["hbm"], "unit": "GB/s", "frac": dec_ach / pk["hbm"],
                "traffic": load_traffic("decode", cfg.name), "peak_source": pk["src"],
                "algorithmic_bytes_per_launch": r["dec_bytes"]}
    prof_roof = {"kernel": "fastgen_profile (token classes, both passes, select)",
                 "bound": "tensor", "achieved": prof_ach, "peak": pk["bf16"], "unit": "TFLOP/s",
                 "frac": prof_ach / pk["bf16"], "traffic": load_traffic("profile", cfg.name),
                 "peak_source": pk["src"], "algorithmic_flops_per_launch": r["prof_flops"],
                 # the flops of one causal Q K^T per head over the same time (the
                 # column sums need the final row LSEs, hence the second pass)
                 "one_pass_equivalent_tflops": prof_ach / 2}
    comp_gbs = r["comp_bytes"] / (r["comp_ms"] * 1e-3) / 1e9
    comp_roof = {"kernel": "fastgen_compact_plan + fastgen_compact (plan, gather)", "bound": "hbm",
                 "achieved": comp_gbs, "peak": pk["hbm"], "unit": "GB/s",
                 "frac": comp_gbs / pk["hbm"], "peak_source": pk["src"],
                 "algorithmic_bytes_per_call": r["comp_bytes"]}
    dec_total = r["decode_ms"]
    dominant, other = (dec_roof, prof_roof) if dec_total >= r["prof_ms"] else (prof_roof, dec_roof)
    e = r["e2e"]
    out = {
        "metric": METRIC, "value": prompt_tok_s, "unit": "tok/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype,
        "data": "synthetic (seeded generator, planted head types; no weights or datasets)",
        "config": {"workload": workload_name(cfg),
                   "G": cfg.G, "parallelism": f"replicas x{world}",
                   "l2": "inputs and caches larger than L2 (no flush)",
                   "step": "profile + plan + compact + all decode steps",
                   "decode_launch": "host loop" if args.no_graph else "one CUDA graph per step",
                   "frequent_refresh_period": args.refresh_period or None},
        "decode_tok_s": decode_tok_s, "decode_hbm_gbs": r["dec_gbs"],
        "phases_ms": {"profile": r["prof_ms"], "compact_plan": r["comp_ms"],
                      "decode_all_steps": r["decode_ms"], "decode_per_step": dec_launch_ms},
        "kept_fraction": r["kept_frac"],
        "saved_policy_map": None if r["policy_map"] is None else dict(
            r["policy_map"], prompt_tok_s=world * cfg.B * cfg.n / (
                (r["policy_map"]["profile_ms"] + r["policy_map"]["compact_plan_ms"]) * 1e-3)),
        "prompt_attention_output": r["prompt_attention"],
        "roofline": dominant, "roofline_other": other, "roofline_compaction": comp_roof,
        "clocks": r["clocks"],
        "e2e": {"value": world * cfg.B * cfg.n / (e["prefill_ms"] * 1e-3), "unit": "tok/s",
                "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"],
                "decode_tok_s": world * cfg.B * cfg.steps / (e["decode_ms"] * 1e-3),
                "decode_h2d_bytes_per_step": e["dec_h2d"],
                "decode_d2h_bytes_per_step": e["dec_d2h"]},
        "gpu_launches": args.steps * (
            fg_launches("profile") + fg_launches("plan") + fg_launches("compact")
            + (fg_launches("refresh_init") if args.refresh_period else 0)
            + cfg.steps * fg_launches("decode" if not args.refresh_period else "decode_acc")
            + (cfg.steps // args.refresh_period if args.refresh_period else 0)),
    }
    if world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(cfg)
    print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def fg_launches(call):
    from adaptive_head_kv_gb300.fastgen import LAUNCHES

    return LAUNCHES[call]


def workload_name(cfg):
    """The workload as both arms name it in `config.workload`."""
    return (f"{cfg.name}: B={cfg.B} L={cfg.L} H={cfg.H} Hkv={cfg.kv_heads} d={cfg.d} n={cfg.n} "
            f"decode_steps={cfg.steps} T={cfg.T} r_l={cfg.r_l} r_f={cfg.r_f}")


def run_reference(args, cfg, world):
    """The oracle timed as it stands on the host cores, on bounded samples of
    the same workload, reported in the same metric (extrapolated linearly in
    heads: every head of a configuration costs the same)."""
    heads_per_step = 2
    rng = np.random.default_rng(7)
    for _ in range(args.warmup):  # untimed: one head each
        oracle_sample(cfg, [int(rng.integers(cfg.G))])
    t_pc = t_dec = 0.0
    sampled = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        heads = sorted(rng.choice(cfg.G, size=heads_per_step, replace=False).tolist())
        a, b, done = oracle_sample(cfg, heads)
        t_pc += a
        t_dec += b
        sampled += done
    wall_ms = (time.perf_counter() - t0) * 1e3 / max(args.steps, 1)
    scale = cfg.G / sampled
    value = cfg.B * cfg.n / (t_pc * scale)
    cores = blas_threads()
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall_ms,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded generator)",
           "config": {"workload": workload_name(cfg), "G": cfg.G,
                      "step": f"{heads_per_step} sampled heads (profile+compact+{cfg.steps} "
                              f"decode steps each); value extrapolated to all {cfg.G} heads"},
           "extrapolated_ms_per_full_step": (t_pc + t_dec) * scale / max(args.steps, 1) * 1e3,
           "decode_tok_s": cfg.B * cfg.steps / (t_dec * scale),
           "cpu_baseline": {"value": value, "unit": "tok/s", "cores": cores,
                            "host_cores": os.cpu_count(), "kind": "oracle",
                            "sample": f"{heads_per_step} heads per step x {args.steps} steps of "
                                      f"{cfg.name}, extrapolated linearly in heads"},
           "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def reduce_max(values, world, device):
    """Element-wise maximum of per-rank timings (the only cross-rank step)."""
    import torch

    t = torch.tensor(values, dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


if __name__ == "__main__":
    main()
