"""Buffer set and call sequence of one compaction pass through the C-ABI.

`CompactionPass` owns the device buffers of one pass (scores, selection
lists, pools, workspaces), allocated once with torch, and issues the four
library calls in order on one stream.  It does no arithmetic of its own.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import (Policy, Pools, kvc_compact_rerotate_quant, kvc_decode_attn,
               kvc_decode_workspace_bytes, kvc_score, kvc_score_workspace_bytes, kvc_select,
               kvc_select_workspace_bytes, make_shape, N_POOLS, SCORE_ACCUMULATE)


class CompactionPass:
    def __init__(self, batch: int, n_layers: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                 n_tokens: int, window: int, policy: Policy, softmax_scale: float = 0.0,
                 device="cuda"):
        self.shape = make_shape(batch, n_layers, n_q_heads, n_kv_heads, head_dim, n_tokens)
        self.window = window
        self.policy = policy
        self.scale = softmax_scale
        self.U = batch * n_layers * n_kv_heads
        self.G = n_q_heads // n_kv_heads
        U, T, P = self.U, n_tokens, policy.page_size
        dev = torch.device(device)
        e = lambda *s, dt: torch.empty(s, dtype=dt, device=dev)
        self.scores = e(U, T, dt=torch.float32)
        self.page_scores = e(U, T // P, dt=torch.float32) if P > 1 else None
        self.score_status = torch.zeros(U, dtype=torch.int32, device=dev)
        wb = kvc_score_workspace_bytes(self.shape, window)
        self.score_ws = e(max(wb, 256), dt=torch.uint8)
        self.kept_idx = e(N_POOLS, U, max(policy.capacity, 1), dt=torch.int32)
        self.kept_count = e(N_POOLS, U, dt=torch.int32)
        self.unit_status = e(U, dt=torch.int32)
        self.compact_status = torch.zeros(U, dtype=torch.int32, device=dev)
        self.floor_excess = e(U, dt=torch.int64)
        sb = kvc_select_workspace_bytes(self.shape, policy)
        self.select_ws = e(sb, dt=torch.uint8) if sb > 0 else None
        self.pools = Pools.allocate(self.shape, policy, dev)
        db = kvc_decode_workspace_bytes(self.shape, policy)
        self.decode_ws = e(db, dt=torch.uint8) if db > 0 else None
        self.out = e(U * self.G, head_dim, dt=torch.bfloat16)

    def score(self, k_cache, q_window, bonus=None, accumulate: bool = False, stream=None,
              row_lse=None):
        kvc_score(self.shape, k_cache, q_window, self.window, self.scale, bonus,
                  self.policy.page_size, SCORE_ACCUMULATE if accumulate else 0, self.scores,
                  self.page_scores, self.score_status, self.score_ws, stream=stream,
                  row_lse=row_lse)

    def select(self, scores: Optional[torch.Tensor] = None, stream=None):
        src = scores if scores is not None else (
            self.page_scores if self.policy.page_size > 1 else self.scores)
        kvc_select(self.shape, self.policy, src, self.kept_idx, self.kept_count, self.unit_status,
                   self.floor_excess, self.select_ws,
                   self.select_ws.numel() if self.select_ws is not None else 0, stream=stream)

    def compact(self, k_cache, v_cache, pos_in, rope_cos, rope_sin, stream=None):
        kvc_compact_rerotate_quant(self.shape, self.policy, k_cache, v_cache, pos_in,
                                   self.kept_idx, self.kept_count, rope_cos, rope_sin,
                                   rope_cos.shape[0], self.pools, self.compact_status,
                                   stream=stream)

    def decode(self, q, stream=None):
        kvc_decode_attn(self.shape, self.policy, q, self.pools, self.kept_count, self.scale,
                        self.out, self.decode_ws, stream=stream)
        return self.out

    def run(self, k_cache, v_cache, q_window, pos_in, rope_cos, rope_sin, bonus=None, stream=None):
        """score -> select -> compact (the timed compaction pass)."""
        self.score(k_cache, q_window, bonus, stream=stream)
        self.select(stream=stream)
        self.compact(k_cache, v_cache, pos_in, rope_cos, rope_sin, stream=stream)


def pass_for_workload(w, device="cuda", capacity: Optional[int] = None,
                      inputs: Optional[dict] = None) -> CompactionPass:
    """A CompactionPass configured with the policy of workload `w`."""
    pol = Policy(budget_tokens=w.budget_tokens, budget_bytes=w.budget_bytes, n_sink=w.n_sink,
                 n_recent=w.n_recent, page_size=w.page_size, renumber=w.renumber,
                 capacity=capacity if capacity is not None else w.capacity(),
                 quant_mode=w.quant_mode, n_layer_groups=w.n_layer_groups)
    if inputs is not None:
        pol.flags = inputs.get("flags")
        if "tags" in inputs:
            pol.tags = inputs["tags"]
            pol.action_table = inputs["action_table"]
            pol.n_tags = int(inputs["action_table"].shape[0])
            pol.n_layer_groups = int(inputs["action_table"].shape[1])
    return CompactionPass(w.batch, w.n_layers, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_tokens,
                          w.window, pol, device=device)
