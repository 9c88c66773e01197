"""A small driver over the C ABI that owns the device buffers (through torch)
for one batch of heads: profile -> plan -> compact -> decode steps.

It only allocates and passes pointers; every step runs in the library's
kernels.
"""
from __future__ import annotations

import json

import torch

from . import fastgen as fg


def make_params(B, L, H, n, d, dtype, T, r_l, r_f, scale=0.0, Hkv=0) -> fg.Params:
    code = {"bf16": fg.FG_BF16, "fp32": fg.FG_FP32, torch.bfloat16: fg.FG_BF16,
            torch.float32: fg.FG_FP32}[dtype]
    return fg.Params(B, L, H, n, d, code, T, r_l, r_f, scale, Hkv)


GUARD_BYTES = 4096
GUARD_FILL = 0x5A


class FastGenSession:
    """Owns the buffers of one batch of heads.  With guard=True every buffer
    the library writes gets GUARD_BYTES of canary bytes on both sides, and
    check_guards() reports any that changed (a bounds check for tests).
    refresh_period > 0 selects the opt-in refresh of the frequent sets every
    that many generation steps (fastgen_decode_attn_refresh)."""

    def __init__(self, params: fg.Params, special_ids, punct_ids, max_new_tokens: int,
                 device="cuda", stream=None, guard=False, refresh_period=0):
        self.p = params
        self.refresh_period = int(refresh_period)
        self.state = None
        self._ids = None
        self.device = torch.device(device)
        self.stream = stream
        self.max_new = int(max_new_tokens)
        self.guard = guard
        self._guards = []
        G, n = params.B * params.L * params.H, params.n
        self.G = G
        self.Gkv = params.B * params.L * (params.Hkv or params.H)  # caches (key/value heads)
        self.tdtype = torch.bfloat16 if params.dtype == fg.FG_BF16 else torch.float32
        dev = self.device
        self.special = torch.as_tensor(special_ids, dtype=torch.int32, device=dev)
        self.punct = torch.as_tensor(punct_ids, dtype=torch.int32, device=dev)
        E = self._empty
        self.policy = E((G,), torch.int8)
        self.mass = E((G, 5), torch.float32)
        self.cost = E((G, 5), torch.int32)
        self.colsum = E((G, n), torch.float32)
        self.keep = E((G, n), torch.uint8)
        self.kept = E((G,), torch.int32)
        self.ws = E((fg.fastgen_profile_workspace_bytes(params),), torch.uint8)
        self.plan = E((fg.fastgen_plan_bytes(params, self.max_new),), torch.uint8)
        self.dev_err = E((1,), torch.int32)
        self.dev_err.zero_()
        self.out = E((G, params.d), self.tdtype)
        self.info = None
        self.K_pool = self.V_pool = self.pos_pool = None
        self.dws = None

    def profile(self, Q, K, token_ids):
        self._ids = token_ids
        fg.fastgen_profile(self.p, Q, K, token_ids, self.special, self.punct, self.policy,
                           self.mass, self.cost, self.colsum, self.keep, self.kept, self.ws,
                           self.dev_err, self.stream)

    def profile_attn(self, Q, K, V, token_ids, out):
        """profile() plus the prompt attention output out [G, n, d] = A V."""
        fg.fastgen_profile_attn(self.p, Q, K, V, token_ids, self.special, self.punct,
                                self.policy, self.mass, self.cost, self.colsum, self.keep,
                                self.kept, out, self.ws, self.dev_err, self.stream)
        return out

    def profile_with_policy(self, Q, K, token_ids, policy_map):
        """Phase 1 under a saved head-policy map (one FG_POLICY_* per query
        head, host or device): keep codes of each head's saved entry on this
        prompt; only heads whose entry contains C_frequent are scored."""
        self.policy.copy_(torch.as_tensor(policy_map, dtype=torch.int8).reshape(-1),
                          non_blocking=True)
        fg.fastgen_profile_with_policy(self.p, Q, K, token_ids, self.special, self.punct,
                                       self.policy, self.colsum, self.keep, self.kept, self.ws,
                                       self.dev_err, self.stream)

    def prefill_with_policy(self, Q, K, V, token_ids, policy_map):
        self.profile_with_policy(Q, K, token_ids, policy_map)
        self.compact(K, V)

    def compact(self, K, V):
        if self.pos_pool is not None:  # pools from an earlier prompt: plan and gather in one call
            done, self.info = fg.fastgen_plan_compact(self.p, self.policy, self.keep, self.max_new,
                                                      self.plan, K, V, self.K_pool, self.V_pool,
                                                      self.pos_pool, self.stream)
            self._size_decode_workspace()
            if done:
                self._init_refresh()
                return
        else:
            self.info = fg.fastgen_compact_plan(self.p, self.policy, self.keep, self.max_new,
                                                self.plan, self.stream)
        rows = int(self.info.pool_rows)
        if self.pos_pool is None or self.pos_pool.numel() < rows:
            d = self.p.d
            self.K_pool = self._empty((rows, d), self.tdtype)
            self.V_pool = self._empty((rows, d), self.tdtype)
            self.pos_pool = self._empty((rows,), torch.int32)
        self._size_decode_workspace()
        fg.fastgen_compact(self.p, K, V, self.keep, self.plan, self.info, self.K_pool,
                           self.V_pool, self.pos_pool, self.stream)
        self._init_refresh()

    def _init_refresh(self):
        """Accumulated scores and frequent slots of the new caches (refresh mode)."""
        if self.refresh_period <= 0:
            return
        need = fg.fastgen_refresh_state_bytes(self.p, self.info)
        if self.state is None or self.state.numel() < need:
            self.state = self._empty((max(need, 256),), torch.uint8)
        fg.fastgen_refresh_init(self.p, self.plan, self.info, self.pos_pool, self.colsum,
                                self._ids, self.special, self.punct, self.state, self.stream)

    def _size_decode_workspace(self):
        need = fg.fastgen_decode_workspace_bytes(self.p, self.info)
        if self.dws is None or self.dws.numel() < need:
            self.dws = self._empty((max(need, 256),), torch.uint8)

    def prefill(self, Q, K, V, token_ids):
        self.profile(Q, K, token_ids)
        self.compact(K, V)

    def prefill_host(self, hQ, hK, hV, htoken_ids, Q, K, V, token_ids):
        """prefill() from pinned host tensors: Q (with the ids), K and V are
        copied in that order on one copy stream, and profiling starts as soon
        as Q and K are on the device, so the V copy overlaps it.  One copy at
        a time keeps the host link at its full rate: on the GB300 machines used,
        three concurrent 21 GB copies shared about half of it (103 GB/s in
        all against 211 GB/s for one)."""
        main = torch.cuda.current_stream(self.device)
        if not hasattr(self, "_copy_stream"):
            self._copy_stream = torch.cuda.Stream(self.device)
        cs = self._copy_stream
        cs.wait_stream(main)  # the buffers are free once earlier work is done
        qk_ready, v_ready = torch.cuda.Event(), torch.cuda.Event()
        with torch.cuda.stream(cs):
            token_ids.copy_(htoken_ids, non_blocking=True)
            Q.copy_(hQ, non_blocking=True)
            K.copy_(hK, non_blocking=True)
            qk_ready.record(cs)
            V.copy_(hV, non_blocking=True)
            v_ready.record(cs)
        main.wait_event(qk_ready)
        self.profile(Q, K, token_ids)
        main.wait_event(v_ready)
        self.compact(K, V)

    def decode(self, q, k_new, v_new, new_ids, pos, out=None):
        """One generation step: q [G, d] per query head, k_new/v_new [Gkv, d]
        per key/value head, new_ids [B]; returns out [G, d]."""
        out = self.out if out is None else out
        if self.refresh_period > 0:
            fg.fastgen_decode_attn_refresh(self.p, self.plan, self.info, self.K_pool, self.V_pool,
                                           self.pos_pool, q, k_new, v_new, new_ids, self.special,
                                           self.punct, pos, self.refresh_period, out, self.state,
                                           self.dws, self.dev_err, self.stream)
            return out
        fg.fastgen_decode_attn(self.p, self.plan, self.info, self.K_pool, self.V_pool,
                               self.pos_pool, q, k_new, v_new, new_ids, self.special, self.punct,
                               pos, out, self.dws, self.dev_err, self.stream)
        return out

    def row_scores(self):
        """Accumulated score of every pool row (refresh mode; host copy)."""
        rows = int(self.info.pool_rows)
        return self.state[: rows * 4].view(torch.float32).cpu()

    def capture_decode(self, q, k, v, new_ids, pos0):
        """Captures len(q) consecutive decode calls (inputs q [steps, G, d],
        k, v [steps, Gkv, d] and new_ids [steps, B] on the device, positions pos0,
        pos0 + 1, ...) as one CUDA graph; returns (graph, outs [steps, G, d]).
        Replaying it runs those steps on the session's current caches.  The
        plan and pools must not be reallocated between replays."""
        steps = q.shape[0]
        outs = self._empty((steps, self.G, self.p.d), self.tdtype)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for st in range(steps):
                self.decode(q[st], k[st], v[st], new_ids[st], pos0 + st, out=outs[st])
        return graph, outs

    def _empty(self, shape, dtype):
        if not self.guard:
            return torch.empty(shape, dtype=dtype, device=self.device)
        nbytes = int(torch.Size(shape).numel()) * torch.empty((), dtype=dtype).element_size()
        body = (nbytes + 255) // 256 * 256
        raw = torch.full((GUARD_BYTES + body + GUARD_BYTES,), GUARD_FILL, dtype=torch.uint8,
                         device=self.device)
        view = raw[GUARD_BYTES:GUARD_BYTES + nbytes].view(dtype).view(shape)
        self._guards.append((raw, body))
        return view

    def check_guards(self):
        """Number of guard buffers whose canaries changed (0 when none did)."""
        bad = 0
        for raw, body in self._guards:
            lo = raw[:GUARD_BYTES]
            hi = raw[GUARD_BYTES + body:]
            if bool((lo != GUARD_FILL).any()) or bool((hi != GUARD_FILL).any()):
                bad += 1
        return bad

    def descriptors(self):
        """Host copy of the per-cache descriptors (for inspection and tests)."""
        import ctypes

        raw = self.plan[: self.Gkv * ctypes.sizeof(fg.HeadDesc)].cpu().numpy().tobytes()
        return (fg.HeadDesc * self.Gkv).from_buffer_copy(raw)


POLICY_MAP_FORMAT = "fastgen-head-policy-map"


def save_policy_map(path, params: fg.Params, policy) -> None:
    """Writes a profiled policy (one FG_POLICY_* per query head, flat index
    g = (b*L + l)*H + h) to a JSON file with the shape it was profiled on."""
    pol = [int(x) for x in torch.as_tensor(policy).reshape(-1).cpu().tolist()]
    G = params.B * params.L * params.H
    if len(pol) != G:
        raise ValueError(f"policy has {len(pol)} entries, the shape has {G} heads")
    doc = dict(format=POLICY_MAP_FORMAT, version=1, B=params.B, L=params.L, H=params.H,
               Hkv=params.Hkv or params.H, n=params.n, T=float(params.T),
               r_l=float(params.r_l), r_f=float(params.r_f),
               policies=list(fg.POLICY_NAMES), policy=pol)
    with open(path, "w") as f:
        json.dump(doc, f)


def load_policy_map(path, params: fg.Params) -> torch.Tensor:
    """Reads a map written by save_policy_map for the same B, L, H and Hkv
    (the prompt length may differ); returns int8 [G] on the CPU."""
    with open(path) as f:
        doc = json.load(f)
    if doc.get("format") != POLICY_MAP_FORMAT or doc.get("version") != 1:
        raise ValueError("not a head-policy map")
    want = dict(B=params.B, L=params.L, H=params.H, Hkv=params.Hkv or params.H)
    got = {k: doc.get(k) for k in want}
    if got != want:
        raise ValueError(f"map was saved for {got}, the shape is {want}")
    pol = doc["policy"]
    if len(pol) != params.B * params.L * params.H or any(not 0 <= p <= 4 for p in pol):
        raise ValueError("malformed policy list")
    return torch.tensor(pol, dtype=torch.int8)

