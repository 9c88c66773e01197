"""Counter-based generator of the synthetic FastGen workloads.

The FastGen pages measure on Llama 1 models with real prompts; neither the
weights nor the datasets are available here, so these seeded inputs stand in
for them, with the attention shapes of the Llama configurations and the head
types the pages describe (special-token heads, punctuation heads, local heads
and broad heads: jisaku.com "FastGen" glossary, section on the four head
types; hyper.ai ICLR 2024 summary, Method, the paragraph on head behaviour).

Every value is a pure function of (seed, stream, indices): a splitmix64 hash
(Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
OOPSLA 2014) of a 64-bit counter gives uniforms, and the Box-Muller transform
(Box and Muller, 1958) in float64 turns pairs of uniforms into normals. A head
can therefore be regenerated alone, on any machine, without generating the
others. Tensors are rounded once, to the working dtype, after the float64
values are formed.

Planted structure per head type (per layer-head (l, h); noise per (b, l, h)):
  special : u ~ N(0, I_d); K_j += 4u at special-token positions, Q_i += 4u.
  punct   : v ~ N(0, I_d); K_j += 4v at punctuation positions, Q_i += 4v.
  local   : Q_i = RoPE_i(c) + N(0, I), K_j = RoPE_j(c) + N(0, I), c = 3z,
            z ~ N(0, I_d), RoPE base 10000 on interleaved pairs.
  broad   : Q, K ~ N(0, I).
V ~ N(0, I) for every head.  Positions 0..n-1 are the prompt; positions
n..n+steps-1 are the tokens fed one by one during decoding.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace

import numpy as np

HEAD_TYPES = ("special", "punct", "local", "broad")
VOCAB = 32000
BOS_ID = 1
PUNCT_FRACTION = 0.05
N_PUNCT_IDS = 10

_M64 = (1 << 64) - 1
_GAMMA = 0x9E3779B97F4A7C15
_MIX1 = 0xBF58476D1CE4E5B9
_MIX2 = 0x94D049BB133111EB

# stream tags, one per independent draw
_S_IDS, _S_PUNCT_DRAW, _S_PUNCT_SET, _S_TYPE = 1, 2, 3, 4
_S_PLANT, _S_Q, _S_K, _S_V = 5, 6, 7, 8


def _mix_scalar(x: int) -> int:
    z = (x + _GAMMA) & _M64
    z = ((z ^ (z >> 30)) * _MIX1) & _M64
    z = ((z ^ (z >> 27)) * _MIX2) & _M64
    return z ^ (z >> 31)


def _key(*parts: int) -> int:
    h = 0
    for p in parts:
        h = _mix_scalar(h ^ (int(p) & _M64))
    return h


def _mix_vec(x: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = x + np.uint64(_GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(_MIX1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(_MIX2)
        return z ^ (z >> np.uint64(31))


def _bits(key: int, count: int) -> np.ndarray:
    ctr = np.arange(count, dtype=np.uint64) + np.uint64(key)
    return _mix_vec(ctr)


def _uniform(key: int, count: int) -> np.ndarray:
    """Uniforms in [0, 1) with 53 random bits."""
    return (_bits(key, count) >> np.uint64(11)).astype(np.float64) * 2.0 ** -53


def _normal(key: int, count: int) -> np.ndarray:
    """Standard normals by Box-Muller from counter-indexed uniform pairs."""
    pairs = (count + 1) // 2
    b = _bits(key, 2 * pairs)
    u1 = ((b[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53  # (0, 1]
    u2 = (b[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * math.pi * u2
    out = np.empty(2 * pairs, dtype=np.float64)
    out[0::2] = r * np.cos(t)
    out[1::2] = r * np.sin(t)
    return out[:count]


@dataclass(frozen=True)
class Config:
    name: str
    B: int
    L: int
    H: int
    d: int
    n: int
    steps: int
    dtype: str  # "bf16" or "fp32"
    T: float
    r_l: float
    r_f: float
    mix: tuple = (0.15, 0.20, 0.35, 0.30)  # special / punct / local / broad
    one_of_each: bool = False  # tiny: head h of each layer has type h % 4
    Hkv: int = 0  # key/value heads per layer (grouped-query attention); 0 = H
    extra: dict = field(default_factory=dict, compare=False)

    @property
    def G(self) -> int:
        return self.B * self.L * self.H

    @property
    def kv_heads(self) -> int:
        return self.Hkv or self.H

    @property
    def Gkv(self) -> int:
        return self.B * self.L * self.kv_heads

    def with_(self, **kw) -> "Config":
        return replace(self, **kw)


_LONG_MIX = (0.15 * 0.6 / 0.7, 0.20 * 0.6 / 0.7, 0.35 * 0.6 / 0.7, 0.40)

CONFIGS = {
    "tiny": Config("tiny", 1, 1, 4, 64, 128, 16, "fp32", 0.95, 0.3, 0.3, one_of_each=True),
    "llama7b": Config("llama7b", 1, 32, 32, 128, 2048, 256, "bf16", 0.95, 0.3, 0.3),
    "llama13b": Config("llama13b", 4, 40, 40, 128, 4096, 512, "bf16", 0.95, 0.3, 0.3),
    "llama65b": Config("llama65b", 8, 80, 64, 128, 2048, 1024, "bf16", 0.95, 0.3, 0.3),
    "long8k": Config("long8k", 1, 32, 32, 128, 8192, 256, "bf16", 0.95, 0.1, 0.2, _LONG_MIX),
    "long16k": Config("long16k", 1, 32, 32, 128, 16384, 256, "bf16", 0.95, 0.1, 0.2, _LONG_MIX),
    "long32k": Config("long32k", 1, 32, 32, 128, 32768, 256, "bf16", 0.95, 0.1, 0.2, _LONG_MIX),
}


def special_ids(seed: int = 0) -> np.ndarray:
    """The special-token id set: the begin-of-sequence marker alone."""
    return np.array([BOS_ID], dtype=np.int32)


def punct_ids(seed: int = 0) -> np.ndarray:
    """Ten distinct stand-in punctuation ids, drawn once from [3, VOCAB)."""
    out: list[int] = []
    i = 0
    while len(out) < N_PUNCT_IDS:
        v = 3 + int(_mix_scalar(_key(seed, _S_PUNCT_SET, i)) % (VOCAB - 3))
        if v not in out:
            out.append(v)
        i += 1
    return np.array(out, dtype=np.int32)


def make_ids(cfg: Config, seed: int = 0) -> np.ndarray:
    """Token ids [B, n + steps]: uniform over the vocabulary, BOS at 0, and
    about 5 % of positions replaced by an id from the punctuation set."""
    total = cfg.n + cfg.steps
    pset = punct_ids(seed)
    ids = np.empty((cfg.B, total), dtype=np.int32)
    for b in range(cfg.B):
        u = _bits(_key(seed, _S_IDS, b), total)
        row = (u % np.uint64(VOCAB)).astype(np.int64)
        pick = _uniform(_key(seed, _S_PUNCT_DRAW, b), 2 * total)
        is_p = pick[0::2] < PUNCT_FRACTION
        which = np.minimum((pick[1::2] * len(pset)).astype(np.int64), len(pset) - 1)
        row = np.where(is_p, pset[which], row)
        row[0] = BOS_ID
        ids[b] = row.astype(np.int32)
    return ids


def head_types(cfg: Config, seed: int = 0) -> np.ndarray:
    """Head type per (layer, head) as an index into HEAD_TYPES."""
    t = np.empty((cfg.L, cfg.H), dtype=np.int32)
    cum = np.cumsum(np.asarray(cfg.mix, dtype=np.float64))
    for l in range(cfg.L):
        for h in range(cfg.H):
            if cfg.one_of_each:
                t[l, h] = h % 4
            else:
                u = _uniform(_key(seed, _S_TYPE, l, h), 1)[0]
                t[l, h] = int(min(np.searchsorted(cum, u, side="right"), 3))
    return t


def _rope(c: np.ndarray, positions: np.ndarray, base: float = 10000.0) -> np.ndarray:
    d = c.shape[0]
    k = np.arange(d // 2, dtype=np.float64)
    theta = base ** (-2.0 * k / d)
    ang = positions[:, None].astype(np.float64) * theta[None, :]
    cs, sn = np.cos(ang), np.sin(ang)
    x, y = c[0::2][None, :], c[1::2][None, :]
    out = np.empty((positions.shape[0], d), dtype=np.float64)
    out[:, 0::2] = x * cs - y * sn
    out[:, 1::2] = x * sn + y * cs
    return out


def kv_of(cfg: Config, g: int) -> int:
    """Key/value head of query head g: head h of a layer uses kv head h // (H / Hkv)."""
    b, rem = divmod(g, cfg.L * cfg.H)
    l, h = divmod(rem, cfg.H)
    return (b * cfg.L + l) * cfg.kv_heads + h // (cfg.H // cfg.kv_heads)


def _plant(cfg: Config, seed: int, l: int, kv: int, kind: int) -> np.ndarray:
    # one planted vector per (layer, head) without groups; per type in a group
    if cfg.kv_heads == cfg.H:
        return _normal(_key(seed, _S_PLANT, l, kv), cfg.d)
    return _normal(_key(seed, _S_PLANT, l, kv, 100 + kind), cfg.d)


def make_q(cfg: Config, seed: int, g: int, ids: np.ndarray, types: np.ndarray) -> np.ndarray:
    """float64 Q [n + steps, d] of query head g = (b*L + l)*H + h."""
    b, rem = divmod(g, cfg.L * cfg.H)
    l, h = divmod(rem, cfg.H)
    kv = h // (cfg.H // cfg.kv_heads)
    total, d = cfg.n + cfg.steps, cfg.d
    kind = int(types[l, h])
    Q = _normal(_key(seed, _S_Q, b, l, h), total * d).reshape(total, d)
    plant = _plant(cfg, seed, l, kv, kind)
    if HEAD_TYPES[kind] in ("special", "punct"):
        Q += 4.0 * plant
    elif HEAD_TYPES[kind] == "local":
        Q += _rope(3.0 * plant, np.arange(total))
    return Q


def make_kv(cfg: Config, seed: int, c: int, ids: np.ndarray, types: np.ndarray):
    """float64 (K, V) [n + steps, d] of key/value head c = (b*L + l)*Hkv + kv,
    carrying the planted structure of every query head type in its group."""
    b, rem = divmod(c, cfg.L * cfg.kv_heads)
    l, kv = divmod(rem, cfg.kv_heads)
    total, d = cfg.n + cfg.steps, cfg.d
    r = cfg.H // cfg.kv_heads
    K = _normal(_key(seed, _S_K, b, l, kv), total * d).reshape(total, d)
    V = _normal(_key(seed, _S_V, b, l, kv), total * d).reshape(total, d)
    for kind in sorted(set(int(t) for t in types[l, kv * r:(kv + 1) * r])):
        plant = _plant(cfg, seed, l, kv, kind)
        if HEAD_TYPES[kind] == "special":
            K[np.isin(ids[b], special_ids(seed))] += 4.0 * plant
        elif HEAD_TYPES[kind] == "punct":
            K[np.isin(ids[b], punct_ids(seed))] += 4.0 * plant
        elif HEAD_TYPES[kind] == "local":
            K += _rope(3.0 * plant, np.arange(total))
    return K, V


def make_head(cfg: Config, seed: int, g: int, ids: np.ndarray, types: np.ndarray):
    """float64 (Q, K, V), each [n + steps, d], of query head g and its
    key/value head."""
    K, V = make_kv(cfg, seed, kv_of(cfg, g), ids, types)
    return make_q(cfg, seed, g, ids, types), K, V


def _round(x: np.ndarray, dtype: str):
    import torch

    t = torch.from_numpy(x)
    return t.to(torch.bfloat16) if dtype == "bf16" else t.to(torch.float32)


def make_workload_split(cfg: Config, seed: int = 0, threads: int | None = None, pin=False):
    """The whole workload laid out as it is consumed: prompt tensors Q
    [G, n, d] and K, V [Gkv, n, d], and per-step decode tensors q [steps, G, d]
    and k, v [steps, Gkv, d], in the working dtype (pinned host memory if
    `pin`), plus ids [B, n + steps].  Each head is generated once, straight
    into its slices."""
    import torch

    ids = make_ids(cfg, seed)
    types = head_types(cfg, seed)
    n, steps, d = cfg.n, cfg.steps, cfg.d
    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    out = {}
    for k, rows in (("Q", cfg.G), ("K", cfg.Gkv), ("V", cfg.Gkv)):
        out[k] = torch.empty((rows, n, d), dtype=tdt, pin_memory=pin)
        out[k.lower()] = torch.empty((steps, rows, d), dtype=tdt, pin_memory=pin)

    def put(name, i, x):
        r = _round(x, cfg.dtype)
        out[name][i] = r[:n]
        out[name.lower()][:, i] = r[n:]

    def one(i):
        if i < cfg.G:
            put("Q", i, make_q(cfg, seed, i, ids, types))
        else:
            c = i - cfg.G
            k, v = make_kv(cfg, seed, c, ids, types)
            put("K", c, k)
            put("V", c, v)

    nthr = threads or min(32, os.cpu_count() or 1)
    with ThreadPoolExecutor(nthr) as ex:
        list(ex.map(one, range(cfg.G + cfg.Gkv)))
    return dict(out, ids=ids, types=types)


def make_workload(cfg: Config, seed: int = 0, heads=None, threads: int | None = None):
    """Rounded CPU tensors for a whole workload (or a subset of query-head
    indices).

    Returns dict(Q: [len(heads), n + steps, d]; K, V: the same rows for
    their key/value heads (one per query head listed; without groups this is
    each head's own K/V); Kg, Vg: [Gkv, n + steps, d] when heads is None;
    ids: [B, n + steps] int32, types: [L, H], heads: the query-head indices).
    """
    import torch

    heads = np.arange(cfg.G) if heads is None else np.asarray(heads, dtype=np.int64)
    ids = make_ids(cfg, seed)
    types = head_types(cfg, seed)
    total = cfg.n + cfg.steps
    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    out = {k: torch.empty((len(heads), total, cfg.d), dtype=tdt) for k in "QKV"}

    def one(i):
        q, k, v = make_head(cfg, seed, int(heads[i]), ids, types)
        out["Q"][i] = _round(q, cfg.dtype)
        out["K"][i] = _round(k, cfg.dtype)
        out["V"][i] = _round(v, cfg.dtype)

    nthr = threads or min(32, os.cpu_count() or 1)
    if nthr <= 1 or len(heads) <= 1:
        for i in range(len(heads)):
            one(i)
    else:
        with ThreadPoolExecutor(nthr) as ex:
            list(ex.map(one, range(len(heads))))
    return dict(out, ids=ids, types=types, heads=heads)
