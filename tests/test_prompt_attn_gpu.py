"""GPU parity of the prompt attention output (fastgen_profile_attn): out =
A V against the oracle for every head on small shapes (tiles, a ragged tail,
head dims 64 / 128, grouped keys, fp32), sampled heads at the 7B shape; the
profile outputs of the same call against the oracle, and its column sums
against fastgen_profile's.

Tolerance, per element, from the arithmetic.  A weight is 2^(x) with x the
base-2 score minus the row's base-2 log-sum-exp; both are fp32 sums of d
products, so x carries at most e_i = 2 (d + 4) 2^-24 max_j |s|_ij (|s| the
score with |q|, |k|), a relative weight error ln2 e_i, plus 2^-22 from the
hardware exponential.  The fp32 accumulation over at most n terms adds
n 2^-24 relative to (A |V|)_ic.  bf16 also rounds each weight to bf16 for the
P V product (2^-8) and stores the output in bf16 (2^-8 |o|):
  fp32: |err_ic| <= (ln2 e_i + 2^-22 + n 2^-24) (A |V|)_ic + 2^-24 |o_ic|
  bf16: the same with 2^-8 added to the weight term and 2^-8 |o_ic|."""
import numpy as np
import pytest
import torch

from synth import CONFIGS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    from adaptive_head_kv_gb300 import fastgen as fg

    fg.lib()  # raises if the CUDA library is missing


def _bound(cfg, Qa, Ka, Va, want):
    from oracle import fastgen_oracle as O

    n, d = Qa.shape
    sc = O.default_scale(d)
    A = O.attention_map(Qa, Ka, sc)
    av = A @ np.abs(Va)
    sabs = np.tril(sc / np.log(2.0) * (np.abs(Qa) @ np.abs(Ka).T))  # base-2 units
    e = 2 * (d + 4) * 2.0 ** -24 * sabs.max(axis=1, keepdims=True)
    w = np.log(2.0) * e + 2.0 ** -22 + n * 2.0 ** -24
    if cfg.dtype == "bf16":
        return (2.0 ** -8 + w) * av + 2.0 ** -8 * np.abs(want) + 1e-7
    return w * av + 2.0 ** -24 * np.abs(want) + 1e-7


def _run(cfg, seed=0, heads=None):
    from adaptive_head_kv_gb300.session import FastGenSession, make_params
    from parity_util import kv_rows
    from synth import make_workload, make_workload_split, punct_ids, special_ids

    n = cfg.n
    dev = torch.device("cuda")
    if heads is None:
        w = make_workload(cfg, seed)
        sel = kv_rows(cfg)
        Q = w["Q"][:, :n].contiguous().to(dev)
        K = w["K"][sel, :n].contiguous().to(dev)
        V = w["V"][sel, :n].contiguous().to(dev)
    else:
        w = make_workload_split(cfg, seed)
        Q, K, V = (w[x].to(dev) for x in "QKV")
    ids = torch.from_numpy(w["ids"][:, :n].copy()).to(dev)
    p = make_params(cfg.B, cfg.L, cfg.H, n, cfg.d, cfg.dtype, cfg.T, cfg.r_l, cfg.r_f,
                    Hkv=cfg.Hkv)
    s = FastGenSession(p, special_ids(seed), punct_ids(seed), 0, guard=True)
    out = s._empty((cfg.G, n, cfg.d), s.tdtype)
    s.profile_attn(Q, K, V, ids, out)
    torch.cuda.synchronize()
    from adaptive_head_kv_gb300 import fastgen as fg

    assert fg.fastgen_read_error(s.dev_err) == fg.FG_OK
    assert s.check_guards() == 0
    res = dict(out=out, workload=w, policy=s.policy.cpu().numpy().astype(int),
               mass=s.mass.cpu().numpy().astype(np.float64), cost=s.cost.cpu().numpy(),
               colsum=s.colsum.cpu().numpy().astype(np.float64), keep=s.keep.cpu().numpy(),
               kept=s.kept.cpu().numpy(), session=s)
    # the same prompt through fastgen_profile: the same kernels, the same
    # profile outputs bit for bit
    s.profile(Q, K, ids)
    torch.cuda.synchronize()
    for key in ("policy", "keep", "kept"):
        assert np.array_equal(res[key], getattr(s, key).cpu().numpy().astype(res[key].dtype)), key
    assert np.array_equal(res["colsum"], s.colsum.cpu().numpy().astype(np.float64))
    return w, res


def _oracle_out(cfg, w, g):
    """(oracle output, its per-element tolerance) of query head g."""
    from oracle import fastgen_oracle as O

    n = cfg.n
    if "heads" in w:  # make_workload: K/V listed per query head
        Qa, Ka, Va = (w[x][g, :n].double().numpy() for x in "QKV")
    else:
        c = (g // cfg.H) * cfg.kv_heads + (g % cfg.H) // (cfg.H // cfg.kv_heads)
        Qa = w["Q"][g].double().numpy()
        Ka, Va = w["K"][c].double().numpy(), w["V"][c].double().numpy()
    want = O.prompt_attention(Qa, Ka, Va)
    return want, _bound(cfg, Qa, Ka, Va, want)


SMALL = [
    ("bf16_d128", dict(dtype="bf16", d=128, L=2, H=4, n=300)),
    ("bf16_d64", dict(dtype="bf16", d=64, L=1, H=4, n=257)),
    ("bf16_one_tile", dict(dtype="bf16", d=128, L=1, H=2, n=128)),
    ("bf16_ragged", dict(dtype="bf16", d=128, L=1, H=3, n=129)),
    ("bf16_n1", dict(dtype="bf16", d=128, L=1, H=2, n=1)),
    ("bf16_gqa_r4", dict(dtype="bf16", d=128, L=1, H=8, Hkv=2, n=300)),
    ("fp32_d128", dict(dtype="fp32", d=128, L=1, H=4, n=200)),
    ("fp32_d64", dict(dtype="fp32", d=64, L=1, H=2, n=150)),
]


@pytest.mark.parametrize("name,kw", SMALL, ids=[x[0] for x in SMALL])
def test_every_head_small(name, kw):
    from parity_util import compare

    cfg = CONFIGS["tiny"].with_(steps=0, **kw)
    w, res = _run(cfg)
    # every profile output of the same call against the oracle
    compare(cfg, res, list(range(cfg.G)))
    got = res["out"].float().cpu().numpy().astype(np.float64)
    worst = 0.0
    for g in range(cfg.G):
        want, tol = _oracle_out(cfg, w, g)
        err = np.abs(got[g] - want)
        worst = max(worst, float((err / tol).max()))
        assert (err <= tol).all(), (g, float(err.max()), float((err / tol).max()))
    print(name, "largest error / bound", worst)


def test_llama7b_shape_sampled_heads():
    """The 7B shape (G = 1024, n = 2048): sampled heads, every row."""
    from parity_util import sample_heads
    from synth import head_types

    cfg = CONFIGS["llama7b"].with_(steps=0)
    w, res = _run(cfg, heads=True)
    for g in sample_heads(cfg, head_types(cfg), 8):
        got = res["out"][g].float().cpu().numpy().astype(np.float64)
        want, tol = _oracle_out(cfg, w, g)
        err = np.abs(got - want)
        assert (err <= tol).all(), (g, float(err.max()), float((err / tol).max()))
