"""Multi-step self-speculative decoding with a static SnapKV draft cache.

MagicDec (arXiv 2408.11049v5) section A.1, Fig. 8: the draft's compressed KV
is built once at prefill; section 3.1: each step drafts gamma tokens with the
sparse KV, verifies the gamma+1 block against the full cache and keeps the
accepted prefix; section 4.4: the static draft then takes in the new
positions.  This module sequences the library's calls for that loop -- it
holds device buffers and passes pointers; every step of the arithmetic
(selection, gather, draft-cache appends and refreshes, attention,
acceptance, the length bookkeeping) runs in libmagicdec's kernels:

  prefill:  magicdec_snapkv_select -> magicdec_gather_kv  (slots [0, base))
  step:     per layer, for g in 0..gamma-1:
                magicdec_draft_cache_update  append position len+g
                magicdec_draft_attn          over the compact cache
            per layer: magicdec_verify_attn  (block at [len, len+gamma+1))
            magicdec_spec_accept             -> n_acc
            magicdec_step_lengths            len' = len + n_acc + 1
            per layer: magicdec_draft_cache_update(len, len+gamma, len')
                                             refresh verified rows, drop rejected

The full cache k, v [B, L_cap, H_kv, d] must already hold the K/V of every
position a step reads (the pending token and the drafted tokens of each
block): there is no model here to produce them.  The draft appends rows from
`k_draft`, `v_draft` (by default the full cache itself); self-speculation's
sparse-KV draft computes its own K/V for the tokens it drafts, which the
refresh after verification replaces with the verified rows.
`layers` repeats the per-layer calls over the same cache (one layer's data
stands in for each layer).
"""
from __future__ import annotations

from typing import Optional, Sequence

import torch

from . import binding as mb


class SnapKVSpecLoop:
    def __init__(self, k: torch.Tensor, v: torch.Tensor, prefill_len: torch.Tensor, H_q: int, gamma: int,
                 window: int, pool: int, budget: int, V: int, max_steps: int, layers: int = 1,
                 k_draft: Optional[torch.Tensor] = None, v_draft: Optional[torch.Tensor] = None):
        self.k, self.v = k, v
        self.kd = k if k_draft is None else k_draft
        self.vd = v if v_draft is None else v_draft
        B, L_cap, H_kv, d = k.shape
        dev = k.device
        self.B, self.L_cap, self.H_kv, self.d, self.H_q = B, L_cap, H_kv, d, H_q
        self.gamma, self.window, self.pool, self.budget, self.V = gamma, window, pool, budget, V
        self.layers = layers
        self.cap = budget + max_steps * (gamma + 1)          # selected rows + every appended position
        i32 = dict(dtype=torch.int32, device=dev)
        self.len = torch.empty((B,), **i32)
        self.len_next = torch.empty((B,), **i32)
        self.table = torch.empty((gamma + 2, B), **i32)
        self.table_next = torch.empty((gamma + 2, B), **i32)
        self.origin = torch.empty((B,), **i32)
        self.base = torch.empty((B,), **i32)
        self.draft_len = torch.empty((B,), **i32)
        self.idx = torch.empty((B, H_kv, budget), **i32)
        self.kc = torch.zeros((B, H_kv, self.cap, d), dtype=torch.bfloat16, device=dev)
        self.vc = torch.zeros_like(self.kc)
        self.out_d = [torch.empty((B, 1, H_q, d), dtype=torch.bfloat16, device=dev) for _ in range(gamma)]
        self.out_v = torch.empty((B, gamma + 1, H_q, d), dtype=torch.bfloat16, device=dev)
        self.n_acc = torch.empty((B,), **i32)
        self.out_tok = torch.empty((B, gamma + 1), **i32)
        self.n_amb = torch.empty((B,), **i32)
        shape_v = mb.kv_shape(B, H_q, H_kv, d, L_cap)
        shape_d = mb.kv_shape(B, H_q, H_kv, d, self.cap)
        self.ws_attn = torch.zeros(max(mb.magicdec_attn_workspace_size(shape_v, gamma + 1),
                                       mb.magicdec_attn_workspace_size(shape_d, 1)), dtype=torch.uint8, device=dev)
        self.ws_snap = torch.zeros(mb.magicdec_snapkv_workspace_size(shape_v, window), dtype=torch.uint8, device=dev)
        self.ws_acc = torch.zeros(mb.magicdec_spec_accept_workspace_size(B, gamma, V), dtype=torch.uint8, device=dev)
        self._prefill_len = prefill_len
        # launches per step: layers x (gamma appends + gamma drafts + verify + refresh) + accept (4) + lengths
        self.launches_per_step = layers * (2 * gamma + 2) + 4 + 1

    def prefill(self, q_win: torch.Tensor):
        """SnapKV selection from the observation-window queries and the gather, once; the
        lengths start at the prefill length."""
        mb.magicdec_step_lengths(self._prefill_len, self.gamma, self.L_cap, len_out=self.len, table=self.table)
        mb.magicdec_snapkv_select(q_win, self.k, self.len, self.window, self.pool, self.budget, idx=self.idx,
                                  n_sel=self.base, ws=self.ws_snap)
        mb.magicdec_gather_kv(self.k, self.v, self.idx, self.cap, kc=self.kc, vc=self.vc)
        # origin = the length at selection; the draft sees the `base` kept rows
        mb.magicdec_step_lengths(self.len, 0, self.L_cap, len_out=self.origin, table=self.table_next[:2])
        mb.magicdec_step_lengths(self.base, 0, self.cap, len_out=self.draft_len, table=self.table_next[:2])

    def step(self, q_draft: Sequence[torch.Tensor], q_verify: torch.Tensor, target: torch.Tensor,
             draft: torch.Tensor, tok: torch.Tensor, u_acc: torch.Tensor, u_res: torch.Tensor, greedy: bool = False):
        t, g_ = self.table, self.gamma
        for _ in range(self.layers):
            for g in range(g_):
                mb.magicdec_draft_cache_update(self.kd, self.vd, self.kc, self.vc, t[g], t[g], t[g + 1], self.origin,
                                               self.base, 0, draft_len=self.draft_len)
                mb.magicdec_draft_attn(q_draft[g], self.kc, self.vc, self.draft_len, out=self.out_d[g],
                                       ws=self.ws_attn)
            mb.magicdec_verify_attn(q_verify, self.k, self.v, t[g_ + 1], out=self.out_v, ws=self.ws_attn)
        mb.magicdec_spec_accept(target, draft, tok, u_acc, u_res, greedy, n_acc=self.n_acc, out_tok=self.out_tok,
                                n_amb=self.n_amb, ws=self.ws_acc)
        mb.magicdec_step_lengths(self.len, g_, self.L_cap, n_acc=self.n_acc, len_out=self.len_next,
                                 table=self.table_next)
        for _ in range(self.layers):
            mb.magicdec_draft_cache_update(self.k, self.v, self.kc, self.vc, t[0], t[g_], self.len_next, self.origin,
                                           self.base, 0, draft_len=self.draft_len)
        self.len, self.len_next = self.len_next, self.len
        self.table, self.table_next = self.table_next, self.table
