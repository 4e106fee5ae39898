"""A bounded-position session: append a chunk, compact back to the budget, repeat.

PACE Sec. 3.2 ("Bounded positions", "Choosing L"): new rows are written at
the next physical positions; before the next chunk would pass the limit L
the kept rows are renumbered to 0..n-1 and their keys re-rotated, so no
position ever reaches L.  PACE Sec. 5.7 runs such sessions to a million
tokens.  This module holds the host side of that loop -- two cache buffers
used in turn and the renumber decision -- and issues the library's calls;
every step of the pass runs in the library's kernels.

Layout.  Each buffer holds T = budget + chunk rows per unit.  A cycle reads
buffer s as the cache ([U][T][d] keys and values, positions [U][T]) and
compacts it into buffer 1 - s, whose first `budget` rows of every unit then
hold the kept rows (capacity T, so the bf16 pool has exactly the cache's
layout).  The next chunk is written to rows budget..T-1 of that buffer and
the roles swap.  The session requires token mode without EXCLUDE flags and
T >= budget, so every unit keeps exactly `budget` rows and the kept rows end
where the chunk begins.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import Policy, Pools, make_shape, N_POOLS, POOL_BF16
from .passes import CompactionPass


def renumber_due(next_pos: int, limit: int, headroom: int) -> bool:
    """PACE Sec. 3.2: renumber when the next physical position is within
    `headroom` (the chunk about to be appended) of the limit L."""
    return next_pos > limit - headroom


def cycle_schedule(next_pos: int, budget: int, chunk: int, limit: int):
    """Positions of one cycle whose chunk starts at physical position
    `next_pos`: (renumber, end, next) -- whether the compaction renumbers,
    the position one past the cache's last row, and where the following
    chunk starts (the kept rows end with the cache's last row, which the
    recent window always keeps; after a renumber they sit at 0..budget-1).
    Raises ValueError if positions would pass the limit unrenumbered."""
    end = next_pos + chunk
    ren = renumber_due(end, limit, chunk)
    if not ren and end > limit:
        raise ValueError("positions would pass the limit without renumbering")
    return ren, end, (budget if ren else end)


class BoundedSession:
    """Compaction cycles of a session of B sequences x L layers x H_kv heads.

    cycle(new_k, new_v, q_window): the chunk's keys and values
    ([B][L][H_kv][chunk][d] bf16, rotated at their physical positions -- the
    positions this session assigns, see `chunk_positions`) are appended
    after the resident rows; the window queries ([B][L][H_q][W][d], the last
    W rows of the chunk) score the cache; the cache is compacted to the
    budget, renumbered when due.  resident() returns the kept rows.
    """

    def __init__(self, batch: int, n_layers: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                 budget: int, chunk: int, window: int, limit: int, n_sink: int, n_recent: int,
                 softmax_scale: float = 0.0, device="cuda"):
        if chunk < window or n_recent < 1 or budget < n_sink + n_recent:
            raise ValueError("the window must lie in the chunk, and the budget must hold the "
                             "sinks and at least one recent row")
        self.budget, self.chunk, self.limit = budget, chunk, limit
        self.T = budget + chunk
        self.U = batch * n_layers * n_kv_heads
        self.dims = (batch, n_layers, n_kv_heads, head_dim)
        dev = torch.device(device)
        pol = Policy(budget_tokens=budget, n_sink=n_sink, n_recent=n_recent, renumber=True,
                     capacity=self.T)
        # two passes whose pools are each other's cache
        self.passes = [CompactionPass(batch, n_layers, n_q_heads, n_kv_heads, head_dim, self.T, window,
                                      Policy(**{**pol.__dict__}), softmax_scale, dev)
                       for _ in range(2)]
        for p in self.passes:
            U, T, d = self.U, self.T, head_dim
            p.pools = Pools(k_bf16=torch.empty((U, T, d), dtype=torch.bfloat16, device=dev),
                            v_bf16=torch.empty((U, T, d), dtype=torch.bfloat16, device=dev),
                            pos_out=torch.empty((N_POOLS, U, T), dtype=torch.int32, device=dev))
        self.cur = 0                  # buffer holding the resident rows
        self.next_pos = 0             # physical position of the next appended row
        self.renumbered = []          # per cycle: whether the compaction renumbered

    # ------------------------------------------------------------------ state
    def _buf(self, s: int) -> Pools:
        return self.passes[s].pools

    def start(self, k0, v0, pos0: Optional[torch.Tensor] = None):
        """Resident rows before the first cycle: [B][L][H_kv][budget][d] bf16 at
        positions 0..budget-1 (or pos0 int32 [U][budget], ascending per unit)."""
        B, L, H, d = self.dims
        buf = self._buf(self.cur)
        buf.k_bf16[:, :self.budget].copy_(k0.reshape(self.U, self.budget, d))
        buf.v_bf16[:, :self.budget].copy_(v0.reshape(self.U, self.budget, d))
        pos = buf.pos_out[POOL_BF16]
        if pos0 is None:
            pos[:, :self.budget].copy_(torch.arange(self.budget, dtype=torch.int32, device=pos.device))
            self.next_pos = self.budget
        else:
            pos[:, :self.budget].copy_(pos0)
            self.next_pos = int(pos0.max()) + 1

    def chunk_positions(self) -> range:
        """Physical positions the next chunk's rows are written at."""
        return range(self.next_pos, self.next_pos + self.chunk)

    def resident(self):
        """(keys [U][budget][d], values, positions [U][budget]) of the resident rows."""
        buf = self._buf(self.cur)
        return (buf.k_bf16[:, :self.budget], buf.v_bf16[:, :self.budget],
                buf.pos_out[POOL_BF16][:, :self.budget])

    # ------------------------------------------------------------------ cycle
    def append(self, new_k, new_v, stream=None):
        """Write the chunk after the resident rows (the engine's KV write)."""
        B, L, H, d = self.dims
        buf = self._buf(self.cur)
        s = stream if stream is not None else torch.cuda.current_stream()
        with torch.cuda.stream(s):
            buf.k_bf16[:, self.budget:].copy_(new_k.reshape(self.U, self.chunk, d), non_blocking=True)
            buf.v_bf16[:, self.budget:].copy_(new_v.reshape(self.U, self.chunk, d), non_blocking=True)
            buf.pos_out[POOL_BF16][:, self.budget:].copy_(
                torch.arange(self.next_pos, self.next_pos + self.chunk, dtype=torch.int32,
                             device=buf.pos_out.device), non_blocking=True)

    def compact(self, q_window, rope_cos, rope_sin, bonus=None, stream=None) -> bool:
        """Score, select and compact the cache (resident + chunk) into the other
        buffer; returns whether the kept rows were renumbered."""
        B, L, H, d = self.dims
        src, dst = self._buf(self.cur), self.passes[1 - self.cur]
        ren, end, nxt = cycle_schedule(self.next_pos, self.budget, self.chunk, self.limit)
        dst.policy.renumber = ren
        k = src.k_bf16.view(B, L, H, self.T, d)
        v = src.v_bf16.view(B, L, H, self.T, d)
        dst.run(k, v, q_window, src.pos_out[POOL_BF16], rope_cos, rope_sin, bonus, stream=stream)
        self.cur = 1 - self.cur
        self.next_pos = nxt
        self.renumbered.append(ren)
        return ren

    def cycle(self, new_k, new_v, q_window, rope_cos, rope_sin, bonus=None, stream=None) -> bool:
        self.append(new_k, new_v, stream=stream)
        return self.compact(q_window, rope_cos, rope_sin, bonus, stream=stream)

    @property
    def last_pass(self) -> CompactionPass:
        """The pass of the latest compaction (scores, kept lists, statuses)."""
        return self.passes[self.cur]
