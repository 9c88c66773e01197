"""A small driver over the C ABI that owns the device buffers (through torch)
for one batch of heads: profile -> plan -> compact -> decode steps.

It only allocates and passes pointers; every step runs in the library's
kernels.
"""
from __future__ import annotations

import torch

from . import fastgen as fg


def make_params(B, L, H, n, d, dtype, T, r_l, r_f, scale=0.0) -> fg.Params:
    code = {"bf16": fg.FG_BF16, "fp32": fg.FG_FP32, torch.bfloat16: fg.FG_BF16,
            torch.float32: fg.FG_FP32}[dtype]
    return fg.Params(B, L, H, n, d, code, T, r_l, r_f, scale)


class FastGenSession:
    def __init__(self, params: fg.Params, special_ids, punct_ids, max_new_tokens: int,
                 device="cuda", stream=None):
        self.p = params
        self.device = torch.device(device)
        self.stream = stream
        self.max_new = int(max_new_tokens)
        G, n = params.B * params.L * params.H, params.n
        self.G = G
        self.tdtype = torch.bfloat16 if params.dtype == fg.FG_BF16 else torch.float32
        dev = self.device
        self.special = torch.as_tensor(special_ids, dtype=torch.int32, device=dev)
        self.punct = torch.as_tensor(punct_ids, dtype=torch.int32, device=dev)
        self.policy = torch.empty(G, dtype=torch.int8, device=dev)
        self.mass = torch.empty(G, 5, dtype=torch.float32, device=dev)
        self.cost = torch.empty(G, 5, dtype=torch.int32, device=dev)
        self.colsum = torch.empty(G, n, dtype=torch.float32, device=dev)
        self.keep = torch.empty(G, n, dtype=torch.uint8, device=dev)
        self.kept = torch.empty(G, dtype=torch.int32, device=dev)
        self.ws = torch.empty(fg.fastgen_profile_workspace_bytes(params), dtype=torch.uint8,
                              device=dev)
        self.plan = torch.empty(fg.fastgen_plan_bytes(params, self.max_new), dtype=torch.uint8,
                                device=dev)
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.out = torch.empty(G, params.d, dtype=self.tdtype, device=dev)
        self.info = None
        self.K_pool = self.V_pool = self.pos_pool = None
        self.dws = None

    def profile(self, Q, K, token_ids):
        fg.fastgen_profile(self.p, Q, K, token_ids, self.special, self.punct, self.policy,
                           self.mass, self.cost, self.colsum, self.keep, self.kept, self.ws,
                           self.dev_err, self.stream)

    def compact(self, K, V):
        self.info = fg.fastgen_compact_plan(self.p, self.policy, self.cost, self.max_new,
                                            self.plan, self.stream)
        rows = int(self.info.pool_rows)
        if self.pos_pool is None or self.pos_pool.numel() < rows:
            d = self.p.d
            self.K_pool = torch.empty(rows, d, dtype=self.tdtype, device=self.device)
            self.V_pool = torch.empty(rows, d, dtype=self.tdtype, device=self.device)
            self.pos_pool = torch.empty(rows, dtype=torch.int32, device=self.device)
        need = fg.fastgen_decode_workspace_bytes(self.p, self.info)
        if self.dws is None or self.dws.numel() < need:
            self.dws = torch.empty(max(need, 256), dtype=torch.uint8, device=self.device)
        fg.fastgen_compact(self.p, K, V, self.keep, self.plan, self.info, self.K_pool,
                           self.V_pool, self.pos_pool, self.stream)

    def prefill(self, Q, K, V, token_ids):
        self.profile(Q, K, token_ids)
        self.compact(K, V)

    def decode(self, q, k_new, v_new, new_ids, pos, out=None):
        out = self.out if out is None else out
        fg.fastgen_decode_attn(self.p, self.plan, self.info, self.K_pool, self.V_pool,
                               self.pos_pool, q, k_new, v_new, new_ids, self.special, self.punct,
                               pos, out, self.dws, self.dev_err, self.stream)
        return out

    def descriptors(self):
        """Host copy of the per-head descriptors (for inspection and tests)."""
        import ctypes

        raw = self.plan[: self.G * ctypes.sizeof(fg.HeadDesc)].cpu().numpy().tobytes()
        return (fg.HeadDesc * self.G).from_buffer_copy(raw)
