"""Python binding of libfastgen.so: argument marshalling only.

Every function has the name and argument order of the C entry point in
include/fastgen.h.  Tensor arguments are torch tensors (their data_ptr() is
passed) or raw integer addresses; `stream` defaults to torch's current CUDA
stream.  A negative status raises FastGenError.  There is no fallback: if the
shared library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfastgen.so")

FG_OK, FG_EINVAL, FG_EDTYPE, FG_EWORKSPACE, FG_ECAPACITY, FG_ECUDA, FG_EDEVICE = 0, -1, -2, -3, -4, -5, -6
FG_BF16, FG_FP32 = 0, 1
FG_POLICY_S, FG_POLICY_SP, FG_POLICY_SPF, FG_POLICY_SPFL, FG_POLICY_FULL = range(5)
POLICY_NAMES = ("special", "special+punct", "special+punct+frequent",
                "special+punct+frequent+local", "full")
FG_KEEP_DROP, FG_KEEP_STATIC, FG_KEEP_WINDOW = 0, 1, 2

# kernels launched by one call of each entry point (counted in the bench)
LAUNCHES = {"profile": 4, "profile_attn": 5, "profile_with_policy": 5, "plan": 3, "compact": 1,
            "decode": 2, "decode_acc": 3, "refresh": 1, "refresh_init": 1}

EXPORTS = (
    "fastgen_status_string", "fastgen_version", "fastgen_profile_workspace_bytes",
    "fastgen_profile", "fastgen_plan_bytes", "fastgen_compact_plan", "fastgen_compact",
    "fastgen_decode_workspace_bytes", "fastgen_decode_attn", "fastgen_read_error",
    "fastgen_decode_attn_noalloc", "fastgen_profile_with_policy", "fastgen_profile_attn",
    "fastgen_plan_compact", "fastgen_refresh_state_bytes", "fastgen_refresh_init",
    "fastgen_decode_attn_refresh", "fastgen_profile_stall_test",
)

# size of the library-held scratch array used by fastgen_decode_attn_noalloc
NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024


class Params(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("L", ctypes.c_int32), ("H", ctypes.c_int32),
                ("n", ctypes.c_int32), ("d", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("T", ctypes.c_float), ("r_l", ctypes.c_float), ("r_f", ctypes.c_float),
                ("scale", ctypes.c_float), ("Hkv", ctypes.c_int32)]


class HeadDesc(ctypes.Structure):
    _fields_ = [("off", ctypes.c_int64), ("n_static", ctypes.c_int32),
                ("static_cap", ctypes.c_int32), ("win_off", ctypes.c_int64),
                ("w", ctypes.c_int32), ("policy", ctypes.c_int32),
                ("work_off", ctypes.c_int32), ("n_work", ctypes.c_int32)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("pool_rows", ctypes.c_int64), ("n_work", ctypes.c_int32),
                ("rows_per_work", ctypes.c_int32)]


class FastGenError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


_lib = None
_P = ctypes.c_void_p
_I32, _I64, _SZ = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
_SIGS = {
    "fastgen_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "fastgen_version": (_I32, []),
    "fastgen_profile_workspace_bytes": (_SZ, [ctypes.POINTER(Params)]),
    "fastgen_profile": (ctypes.c_int, [ctypes.POINTER(Params), _P, _P, _P, _P, _I32, _P, _I32,
                                       _P, _P, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "fastgen_profile_with_policy": (ctypes.c_int, [ctypes.POINTER(Params), _P, _P, _P, _P, _I32,
                                                   _P, _I32, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "fastgen_profile_attn": (ctypes.c_int, [ctypes.POINTER(Params), _P, _P, _P, _P, _P, _I32, _P,
                                            _I32, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "fastgen_plan_bytes": (_SZ, [ctypes.POINTER(Params), _I32]),
    "fastgen_compact_plan": (ctypes.c_int, [ctypes.POINTER(Params), _P, _P, _I32, _P, _SZ,
                                            ctypes.POINTER(PlanInfo), _P]),
    "fastgen_compact": (ctypes.c_int, [ctypes.POINTER(Params), _P, _P, _P, _P,
                                       ctypes.POINTER(PlanInfo), _P, _P, _P, _I64, _P]),
    "fastgen_plan_compact": (ctypes.c_int, [ctypes.POINTER(Params), _P, _P, ctypes.c_int32, _P,
                                            _SZ, _P, _P, _P, _P, _P, _I64,
                                            ctypes.POINTER(PlanInfo), _P]),
    "fastgen_decode_workspace_bytes": (_SZ, [ctypes.POINTER(Params), ctypes.POINTER(PlanInfo)]),
    "fastgen_decode_attn": (ctypes.c_int, [ctypes.POINTER(Params), _P, ctypes.POINTER(PlanInfo),
                                           _P, _P, _P, _P, _P, _P, _P, _P, _I32, _P, _I32, _I32,
                                           _P, _P, _SZ, _P, _P]),
    "fastgen_read_error": (ctypes.c_int, [_P, _P]),
    "fastgen_profile_stall_test": (ctypes.c_int, [ctypes.POINTER(Params), _P, _P, _P, _P, _I32,
                                                  _P, _I32, _P, _P, _P, _P, _P, _P, _P, _SZ, _P,
                                                  _I32, _P]),
    "fastgen_refresh_state_bytes": (_SZ, [ctypes.POINTER(Params), ctypes.POINTER(PlanInfo)]),
    "fastgen_refresh_init": (ctypes.c_int, [ctypes.POINTER(Params), _P, ctypes.POINTER(PlanInfo),
                                            _P, _P, _P, _P, _I32, _P, _I32, _P, _SZ, _P]),
    "fastgen_decode_attn_refresh": (ctypes.c_int, [ctypes.POINTER(Params), _P,
                                                   ctypes.POINTER(PlanInfo), _P, _P, _P, _P, _P,
                                                   _P, _P, _P, _I32, _P, _I32, _I32, _I32, _P, _P,
                                                   _SZ, _P, _SZ, _P, _P]),
    "fastgen_decode_attn_noalloc": (ctypes.c_int, [ctypes.POINTER(Params), _P,
                                                   ctypes.POINTER(PlanInfo), _P, _P, _P, _P, _P,
                                                   _P, _P, _P, _I32, _P, _I32, _I32, _P, _P, _P]),
}


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise FileNotFoundError(
                f"{LIB_PATH} is missing: build it with adaptive_head_kv_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _count(x) -> int:
    return 0 if x is None else int(x.numel())


def _stream(stream) -> int | None:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str) -> None:
    if status != FG_OK:
        raise FastGenError(status, where)


def status_string(status: int) -> str:
    return lib().fastgen_status_string(status).decode()


def fastgen_status_string(status: int) -> str:
    return status_string(status)


def fastgen_version() -> int:
    return lib().fastgen_version()


def fastgen_profile_workspace_bytes(params: Params) -> int:
    return lib().fastgen_profile_workspace_bytes(ctypes.byref(params))


def fastgen_profile(params, Q, K, token_ids, special_ids, punct_ids, policy, mass, cost, colsum,
                    keep, kept, workspace, dev_err, stream=None) -> None:
    ws_bytes = workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else 0
    _check(lib().fastgen_profile(ctypes.byref(params), _ptr(Q), _ptr(K), _ptr(token_ids),
                                 _ptr(special_ids), _count(special_ids), _ptr(punct_ids),
                                 _count(punct_ids), _ptr(policy), _ptr(mass), _ptr(cost),
                                 _ptr(colsum), _ptr(keep), _ptr(kept), _ptr(workspace), ws_bytes,
                                 _ptr(dev_err), _stream(stream)), "fastgen_profile")


def fastgen_profile_with_policy(params, Q, K, token_ids, special_ids, punct_ids, policy, colsum,
                                keep, kept, workspace, dev_err, stream=None) -> None:
    ws_bytes = workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else 0
    _check(lib().fastgen_profile_with_policy(
        ctypes.byref(params), _ptr(Q), _ptr(K), _ptr(token_ids), _ptr(special_ids),
        _count(special_ids), _ptr(punct_ids), _count(punct_ids), _ptr(policy), _ptr(colsum),
        _ptr(keep), _ptr(kept), _ptr(workspace), ws_bytes, _ptr(dev_err), _stream(stream)),
        "fastgen_profile_with_policy")


def fastgen_profile_attn(params, Q, K, V, token_ids, special_ids, punct_ids, policy, mass, cost,
                         colsum, keep, kept, out, workspace, dev_err, stream=None) -> None:
    ws_bytes = workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else 0
    _check(lib().fastgen_profile_attn(
        ctypes.byref(params), _ptr(Q), _ptr(K), _ptr(V), _ptr(token_ids), _ptr(special_ids),
        _count(special_ids), _ptr(punct_ids), _count(punct_ids), _ptr(policy), _ptr(mass),
        _ptr(cost), _ptr(colsum), _ptr(keep), _ptr(kept), _ptr(out), _ptr(workspace), ws_bytes,
        _ptr(dev_err), _stream(stream)), "fastgen_profile_attn")


def fastgen_plan_bytes(params: Params, max_new_tokens: int) -> int:
    return lib().fastgen_plan_bytes(ctypes.byref(params), max_new_tokens)


def fastgen_compact_plan(params, policy, keep, max_new_tokens, plan, stream=None) -> PlanInfo:
    info = PlanInfo()
    _check(lib().fastgen_compact_plan(ctypes.byref(params), _ptr(policy), _ptr(keep),
                                      max_new_tokens, _ptr(plan), plan.numel() * plan.element_size(),
                                      ctypes.byref(info), _stream(stream)), "fastgen_compact_plan")
    return info


def fastgen_compact(params, K, V, keep, plan, info, K_pool, V_pool, pos_pool, stream=None) -> None:
    _check(lib().fastgen_compact(ctypes.byref(params), _ptr(K), _ptr(V), _ptr(keep), _ptr(plan),
                                 ctypes.byref(info), _ptr(K_pool), _ptr(V_pool), _ptr(pos_pool),
                                 int(pos_pool.numel()), _stream(stream)), "fastgen_compact")


def fastgen_plan_compact(params, policy, keep, max_new_tokens, plan, K, V, K_pool, V_pool,
                         pos_pool, stream=None):
    """Plan and gather in one call.  Returns (done, info): done is False when
    the pools are smaller than info.pool_rows (nothing was gathered)."""
    info = PlanInfo()
    st = lib().fastgen_plan_compact(
        ctypes.byref(params), _ptr(policy), _ptr(keep), max_new_tokens, _ptr(plan),
        plan.numel() * plan.element_size(), _ptr(K), _ptr(V), _ptr(K_pool), _ptr(V_pool),
        _ptr(pos_pool), int(pos_pool.numel()), ctypes.byref(info), _stream(stream))
    if st == FG_EWORKSPACE and info.pool_rows > pos_pool.numel():
        return False, info
    _check(st, "fastgen_plan_compact")
    return True, info


def fastgen_decode_workspace_bytes(params: Params, info: PlanInfo) -> int:
    return lib().fastgen_decode_workspace_bytes(ctypes.byref(params), ctypes.byref(info))


def fastgen_decode_attn(params, plan, info, K_pool, V_pool, pos_pool, q, k_new, v_new, new_ids,
                        special_ids, punct_ids, pos, out, workspace, dev_err, stream=None) -> None:
    _check(lib().fastgen_decode_attn(ctypes.byref(params), _ptr(plan), ctypes.byref(info),
                                     _ptr(K_pool), _ptr(V_pool), _ptr(pos_pool), _ptr(q),
                                     _ptr(k_new), _ptr(v_new), _ptr(new_ids), _ptr(special_ids),
                                     _count(special_ids), _ptr(punct_ids), _count(punct_ids),
                                     int(pos), _ptr(out), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _ptr(dev_err),
                                     _stream(stream)), "fastgen_decode_attn")


def fastgen_read_error(dev_err, stream=None) -> int:
    return lib().fastgen_read_error(_ptr(dev_err), _stream(stream))


def fastgen_decode_attn_noalloc(params, plan, info, K_pool, V_pool, pos_pool, q, k_new, v_new,
                                new_ids, special_ids, punct_ids, pos, out, dev_err,
                                stream=None) -> None:
    """fastgen_decode_attn without a workspace: for callers that cannot
    allocate device memory while decoding (the scratch is a fixed array held
    by the library; calls must not overlap on the GPU)."""
    _check(lib().fastgen_decode_attn_noalloc(
        ctypes.byref(params), _ptr(plan), ctypes.byref(info), _ptr(K_pool), _ptr(V_pool),
        _ptr(pos_pool), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(new_ids), _ptr(special_ids),
        _count(special_ids), _ptr(punct_ids), _count(punct_ids), int(pos), _ptr(out),
        _ptr(dev_err), _stream(stream)), "fastgen_decode_attn_noalloc")


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def fastgen_refresh_state_bytes(params: Params, info: PlanInfo) -> int:
    return lib().fastgen_refresh_state_bytes(ctypes.byref(params), ctypes.byref(info))


def fastgen_refresh_init(params, plan, info, pos_pool, colsum, token_ids, special_ids, punct_ids,
                         state, stream=None) -> None:
    _check(lib().fastgen_refresh_init(
        ctypes.byref(params), _ptr(plan), ctypes.byref(info), _ptr(pos_pool), _ptr(colsum),
        _ptr(token_ids), _ptr(special_ids), _count(special_ids), _ptr(punct_ids),
        _count(punct_ids), _ptr(state), _nbytes(state), _stream(stream)), "fastgen_refresh_init")


def fastgen_decode_attn_refresh(params, plan, info, K_pool, V_pool, pos_pool, q, k_new, v_new,
                                new_ids, special_ids, punct_ids, pos, period, out, state,
                                workspace, dev_err, stream=None) -> None:
    _check(lib().fastgen_decode_attn_refresh(
        ctypes.byref(params), _ptr(plan), ctypes.byref(info), _ptr(K_pool), _ptr(V_pool),
        _ptr(pos_pool), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(new_ids), _ptr(special_ids),
        _count(special_ids), _ptr(punct_ids), _count(punct_ids), int(pos), int(period),
        _ptr(out), _ptr(state), _nbytes(state), _ptr(workspace), _nbytes(workspace),
        _ptr(dev_err), _stream(stream)), "fastgen_decode_attn_refresh")


def fastgen_profile_stall_test(params, Q, K, token_ids, special_ids, punct_ids, policy, mass,
                               cost, colsum, keep, kept, workspace, dev_err, stall_pass,
                               stream=None) -> None:
    """fastgen_profile with one tensor-core pass's producer held back, so
    that pass's bounded waits run out (a test of the error path)."""
    _check(lib().fastgen_profile_stall_test(
        ctypes.byref(params), _ptr(Q), _ptr(K), _ptr(token_ids), _ptr(special_ids),
        _count(special_ids), _ptr(punct_ids), _count(punct_ids), _ptr(policy), _ptr(mass),
        _ptr(cost), _ptr(colsum), _ptr(keep), _ptr(kept), _ptr(workspace), _nbytes(workspace),
        _ptr(dev_err), int(stall_pass), _stream(stream)), "fastgen_profile_stall_test")
