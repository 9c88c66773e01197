"""The C ABI without a GPU: the library loads, exports every symbol the
header declares, sizes its buffers as documented and rejects bad arguments
on the host before launching anything."""
import ctypes
import os
import re
import subprocess

import pytest

from adaptive_head_kv_gb300 import fastgen as fg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fastgen.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not os.path.exists(fg.LIB_PATH):
        from adaptive_head_kv_gb300.build import build

        build()
    fg.lib()


def declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(fastgen_\w+)\s*\(", text)))


def test_header_symbols_exported():
    names = declared()
    assert len(names) >= 10
    L = fg.lib()
    for name in names:
        assert hasattr(L, name), name
    assert set(names) <= set(fg.EXPORTS) | set(names)
    out = subprocess.run(["nm", "-D", "--defined-only", fg.LIB_PATH], capture_output=True,
                         text=True).stdout
    for name in names:
        assert re.search(rf"\bT {name}\b", out), name


def test_struct_sizes():
    assert ctypes.sizeof(fg.Params) == 44
    assert ctypes.sizeof(fg.HeadDesc) == 40
    assert ctypes.sizeof(fg.PlanInfo) == 16


def test_status_strings_and_version():
    assert fg.status_string(0) == "ok"
    for s in (-1, -2, -3, -4, -5, -6):
        assert fg.status_string(s) != "unknown status"
    assert fg.fastgen_version() >= 100


def P(**kw):
    base = dict(B=1, L=2, H=3, n=100, d=128, dtype=fg.FG_BF16, T=0.95, r_l=0.3, r_f=0.3, scale=0.0,
                Hkv=0)
    base.update(kw)
    return fg.Params(**base)


def test_workspace_sizes():
    p = P()
    G, n = 6, 100
    al = lambda x: (x + 255) // 256 * 256
    assert fg.fastgen_profile_workspace_bytes(p) == (al(G * 128 * 4) + al(G * n * 4) + al(n) + 256
                                                     + al(G * 4))
    w = 30
    work = G * ((n + 7 + 255) // 256 + (w + 255) // 256)
    assert fg.fastgen_plan_bytes(p, 7) == al(G * 40) + al(G * 8) + 256 + work * 8
    info = fg.PlanInfo(1000, 13, 256)
    assert fg.fastgen_decode_workspace_bytes(p, info) == al(13 * 8) + al(13 * 128 * 4)
    assert fg.fastgen_profile_workspace_bytes(P(d=96)) == 0


FAKE = 1 << 20  # an aligned address never dereferenced: checks fail first


def profile_status(p, ws_bytes=1 << 40, ptrs=None, ns=1, np_=1):
    L = fg.lib()
    a = dict(Q=FAKE, K=FAKE, ids=FAKE, sp=FAKE, pu=FAKE, policy=FAKE, mass=FAKE, cost=FAKE,
             colsum=FAKE, keep=FAKE, kept=FAKE, ws=FAKE, err=FAKE)
    a.update(ptrs or {})
    return L.fastgen_profile(ctypes.byref(p), a["Q"], a["K"], a["ids"], a["sp"], ns, a["pu"], np_,
                             a["policy"], a["mass"], a["cost"], a["colsum"], a["keep"],
                             a["kept"], a["ws"], ws_bytes, a["err"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(T=0.0), fg.FG_EINVAL), (dict(T=1.5), fg.FG_EINVAL), (dict(T=float("nan")), fg.FG_EINVAL),
    (dict(r_l=-0.1), fg.FG_EINVAL), (dict(r_f=1.01), fg.FG_EINVAL), (dict(n=0), fg.FG_EINVAL),
    (dict(B=0), fg.FG_EINVAL), (dict(d=96), fg.FG_EDTYPE), (dict(dtype=7), fg.FG_EDTYPE),
    (dict(scale=-1.0), fg.FG_EINVAL), (dict(scale=float("inf")), fg.FG_EINVAL),
    (dict(Hkv=2), fg.FG_EINVAL), (dict(Hkv=-1), fg.FG_EINVAL),
    (dict(H=48, Hkv=4), fg.FG_EDTYPE),  # group size 12 is not supported
])
def test_profile_rejects_bad_params(kw, status):
    assert profile_status(P(**kw)) == status


def test_profile_rejects_pointers_and_workspace():
    p = P()
    assert profile_status(p, ptrs=dict(Q=None)) == fg.FG_EINVAL
    assert profile_status(p, ptrs=dict(K=FAKE + 8)) == fg.FG_EINVAL      # not 16-byte aligned
    assert profile_status(p, ptrs=dict(ws=FAKE + 16)) == fg.FG_EINVAL     # not 256-byte aligned
    assert profile_status(p, ptrs=dict(sp=None)) == fg.FG_EINVAL          # count 1, NULL set
    assert profile_status(p, ptrs=dict(err=None)) == fg.FG_EINVAL
    assert profile_status(p, ns=-1) == fg.FG_EINVAL
    assert profile_status(p, np_=5000) == fg.FG_EINVAL
    assert profile_status(p, ws_bytes=fg.fastgen_profile_workspace_bytes(p) - 1) == fg.FG_EWORKSPACE


def test_profile_with_policy_rejects_on_host():
    L = fg.lib()
    p = P()

    def call(pol=FAKE, colsum=FAKE, ws=FAKE, ws_bytes=1 << 40, q=FAKE, **kw):
        return L.fastgen_profile_with_policy(ctypes.byref(P(**kw) if kw else p), q, FAKE, FAKE,
                                             FAKE, 1, FAKE, 1, pol, colsum, FAKE, FAKE, ws,
                                             ws_bytes, FAKE, None)

    assert call(pol=None) == fg.FG_EINVAL
    assert call(colsum=None) == fg.FG_EINVAL
    assert call(q=FAKE + 8) == fg.FG_EINVAL
    assert call(ws=FAKE + 16) == fg.FG_EINVAL
    assert call(ws_bytes=fg.fastgen_profile_workspace_bytes(p) - 1) == fg.FG_EWORKSPACE
    assert call(T=0.0) == fg.FG_EINVAL
    assert call(d=96) == fg.FG_EDTYPE


def test_policy_map_json_roundtrip(tmp_path):
    import torch

    from adaptive_head_kv_gb300.session import load_policy_map, save_policy_map

    p = P(B=2, L=2, H=4, Hkv=2)
    pol = torch.tensor([0, 1, 2, 3, 4, 4, 3, 2, 1, 0, 0, 2, 3, 1, 4, 2], dtype=torch.int8)
    path = tmp_path / "map.json"
    save_policy_map(path, p, pol)
    got = load_policy_map(path, P(B=2, L=2, H=4, Hkv=2, n=37))  # another prompt length
    assert torch.equal(got, pol)
    with pytest.raises(ValueError):
        load_policy_map(path, P(B=1, L=2, H=4, Hkv=2))
    with pytest.raises(ValueError):
        save_policy_map(path, p, pol[:5])


def test_plan_compact_in_one_call_rejects_on_host():
    L = fg.lib()
    p = P()
    info = fg.PlanInfo()
    need = fg.fastgen_plan_bytes(p, 4)
    call = lambda K=FAKE, plan=FAKE, nbytes=need: L.fastgen_plan_compact(
        ctypes.byref(p), FAKE, FAKE, 4, plan, nbytes, K, FAKE, FAKE, FAKE, FAKE, 1000,
        ctypes.byref(info), None)
    assert call(K=None) == fg.FG_EINVAL
    assert call(nbytes=need - 1) == fg.FG_EWORKSPACE
    assert call(plan=FAKE + 32) == fg.FG_EINVAL


def test_plan_compact_decode_reject_on_host():
    L = fg.lib()
    p = P()
    info = fg.PlanInfo(500, 10, 256)
    need = fg.fastgen_plan_bytes(p, 4)
    assert L.fastgen_compact_plan(ctypes.byref(p), FAKE, FAKE, 4, FAKE, need - 1,
                                  ctypes.byref(info), None) == fg.FG_EWORKSPACE
    assert L.fastgen_compact_plan(ctypes.byref(p), FAKE, FAKE, -1, FAKE, need,
                                  ctypes.byref(info), None) == fg.FG_EINVAL
    assert L.fastgen_compact_plan(ctypes.byref(p), FAKE, FAKE, 4, FAKE + 32, need,
                                  ctypes.byref(info), None) == fg.FG_EINVAL
    assert L.fastgen_compact(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, ctypes.byref(info), FAKE,
                             FAKE, FAKE, 499, None) == fg.FG_EWORKSPACE
    ws = fg.fastgen_decode_workspace_bytes(p, info)

    def dec(pos=100, ws_bytes=ws, q=FAKE):
        return L.fastgen_decode_attn(ctypes.byref(p), FAKE, ctypes.byref(info), FAKE, FAKE, FAKE,
                                     q, FAKE, FAKE, FAKE, FAKE, 1, FAKE, 1, pos, FAKE, FAKE,
                                     ws_bytes, FAKE, None)

    assert dec(pos=99) == fg.FG_EINVAL                 # a generated position precedes the prompt end
    odd = fg.PlanInfo(500, 10, 300)                    # rows per item other than 256 or 512
    assert L.fastgen_decode_attn(ctypes.byref(p), FAKE, ctypes.byref(odd), FAKE, FAKE, FAKE, FAKE,
                                 FAKE, FAKE, FAKE, FAKE, 1, FAKE, 1, 100, FAKE, FAKE, ws, FAKE,
                                 None) == fg.FG_EINVAL
    assert dec(ws_bytes=ws - 1) == fg.FG_EWORKSPACE
    assert dec(q=FAKE + 4) == fg.FG_EINVAL
    assert L.fastgen_read_error(None, None) == fg.FG_EINVAL


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(fg, "_lib", None)
    monkeypatch.setattr(fg, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(FileNotFoundError):
        fg.fastgen_version()


def test_group_sizes_in_buffer_sizes():
    """With key/value groups the plan has one descriptor per key/value head
    and the decode workspace one partial per item and query head."""
    al = lambda x: (x + 255) // 256 * 256
    p = P(H=8, Hkv=2, n=100)
    Gkv = 1 * 2 * 2
    w = 30
    work = Gkv * ((100 + 7 + 255) // 256 + (w + 255) // 256)
    assert fg.fastgen_plan_bytes(p, 7) == al(Gkv * 40) + al(Gkv * 8) + 256 + work * 8
    info = fg.PlanInfo(1000, 13, 256)
    assert fg.fastgen_decode_workspace_bytes(p, info) == al(13 * 4 * 8) + al(13 * 4 * 128 * 4)


def test_refresh_calls_reject_on_host():
    """The refresh variant's limits and buffers are checked before any launch."""
    L = fg.lib()
    al = lambda x: (x + 255) // 256 * 256
    p = P()
    info = fg.PlanInfo(1000, 10, 256)
    st = fg.fastgen_refresh_state_bytes(p, info)
    assert st == 2 * al(1000 * 4) + al(1000) + al(6 * 2 * 4)  # rows' acc, score, role; heads' (M, L)
    ws = fg.fastgen_decode_workspace_bytes(p, info)

    def dec(params=p, period=4, state=FAKE, state_bytes=st):
        return L.fastgen_decode_attn_refresh(ctypes.byref(params), FAKE, ctypes.byref(info), FAKE,
                                             FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, FAKE, 1,
                                             100, period, FAKE, state, state_bytes, FAKE, ws,
                                             FAKE, None)

    def init(params=p, state=FAKE, state_bytes=st, colsum=FAKE):
        return L.fastgen_refresh_init(ctypes.byref(params), FAKE, ctypes.byref(info), FAKE, colsum,
                                      FAKE, FAKE, 1, FAKE, 1, state, state_bytes, None)

    assert dec(period=0) == fg.FG_EINVAL                      # period >= 1
    assert dec(period=-3) == fg.FG_EINVAL
    assert dec(params=P(H=4, Hkv=2)) == fg.FG_EINVAL          # groups are not supported
    assert dec(params=P(n=20000, r_l=0.5, r_f=0.5)) == fg.FG_EINVAL  # k + w > 16384
    assert dec(state=None) == fg.FG_EINVAL
    assert dec(state=FAKE + 64) == fg.FG_EINVAL               # not 256-byte aligned
    assert dec(state_bytes=st - 1) == fg.FG_EWORKSPACE
    assert init(params=P(H=4, Hkv=2)) == fg.FG_EINVAL
    assert init(state_bytes=st - 1) == fg.FG_EWORKSPACE
    assert init(colsum=None) == fg.FG_EINVAL
    assert init(params=P(T=0.0)) == fg.FG_EINVAL


def test_stall_test_rejects_on_host():
    L = fg.lib()

    def call(stall=1, **kw):
        return L.fastgen_profile_stall_test(ctypes.byref(P(**kw)), FAKE, FAKE, FAKE, FAKE, 1, FAKE,
                                            1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40,
                                            FAKE, stall, None)

    assert call(stall=0) == fg.FG_EINVAL
    assert call(stall=3) == fg.FG_EINVAL
    assert call(dtype=fg.FG_FP32) == fg.FG_EDTYPE
    assert call(T=0.0) == fg.FG_EINVAL
