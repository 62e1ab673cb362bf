"""Seeded synthetic inputs for the MagicDec attention / acceptance hot path.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic.  Both the CUDA path and the CPU oracle consume what it
produces (the oracle never imports it: tests hand it the arrays).  Random draws
the method itself needs (acceptance uniforms, the draft tokens a draft model
would sample) are made here and passed to both sides as inputs.

Workloads follow the shapes and value distributions of the method's
evaluation regime (Llama-3.1-8B / Qwen-2.5-32B attention shapes, 32k-100k
contexts, batch 16-128), which stands in for the PG-19 / RULER data the paper
ran on; attention cost does not depend on the token content, only selection and
acceptance do, and those get the structured distributions below.

All generation goes through ``torch.Generator`` on the target device, so a
(config, seed, device) triple always yields the same bits.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H_q: int
    H_kv: int
    d: int
    L: int                      # prompt / cache length per sequence
    gamma: int                  # speculation length; verify sees gamma+1 queries
    V: int                      # vocabulary
    n_sink: int = 0             # StreamingLLM attention sinks
    n_recent: int = 0           # StreamingLLM recent window
    snap_window: int = 0        # SnapKV observation window w
    snap_pool: int = 7          # SnapKV max-pool kernel
    snap_budget: int = 0        # SnapKV budget (window included)
    boost_frac: float = 0.0     # fraction of positions whose keys are scaled
    boost: float = 1.0          # key scale at those positions
    heavy_frac: float = 0.0     # fraction of heavy-hitter positions (aligned to window queries)
    heavy_cos: float = 0.6      # cosine between window queries and the heavy-hitter direction
    target_sigma: float = 2.0   # target logits ~ N(0, sigma)
    draft_noise: float = 0.5    # draft logits = target + N(0, noise)
    steps: int = 1              # draft+verify steps after selection
    seed: int = 0

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv

    @property
    def n_q(self) -> int:
        return self.gamma + 1

    @property
    def stream_budget(self) -> int:
        return self.n_sink + self.n_recent


WORKLOADS = {
    # Tiny: the CPU oracle finishes in seconds.
    "tiny": Workload("tiny", B=2, H_q=4, H_kv=1, d=64, L=256, gamma=2, V=16,
                     n_sink=4, n_recent=60, snap_window=16, snap_pool=7, snap_budget=64,
                     target_sigma=2.0, draft_noise=0.5, seed=1),
    # Llama-3.1-8B attention shape, StreamingLLM 16+496 draft.
    "llama8b_b32_l32k": Workload("llama8b_b32_l32k", B=32, H_q=32, H_kv=8, d=128, L=32000, gamma=3,
                                 V=128256, n_sink=16, n_recent=496, boost_frac=0.01, boost=4.0,
                                 target_sigma=2.0, draft_noise=0.5, seed=2),
    # Same shape, B=64, SnapKV draft (w=32, pool 7, budget 2048), 16 draft+verify steps.
    "llama8b_b64_l32k_snapkv": Workload("llama8b_b64_l32k_snapkv", B=64, H_q=32, H_kv=8, d=128, L=32000,
                                        gamma=4, V=128256, snap_window=32, snap_pool=7, snap_budget=2048,
                                        heavy_frac=0.005, heavy_cos=0.6, target_sigma=2.0, draft_noise=0.5,
                                        steps=16, seed=3),
    # Throughput regime (the headline): B=128, L=32000, both drafts with budget 512.
    "llama8b_b128_l32k": Workload("llama8b_b128_l32k", B=128, H_q=32, H_kv=8, d=128, L=32000, gamma=3,
                                  V=128256, n_sink=16, n_recent=496, snap_window=32, snap_pool=7,
                                  snap_budget=512, boost_frac=0.01, boost=4.0, target_sigma=2.0,
                                  draft_noise=0.5, seed=4),
    # Long context, Qwen-2.5-32B-like attention: B=16, L=100000, H_q=40.
    "qwen32b_b16_l100k": Workload("qwen32b_b16_l100k", B=16, H_q=40, H_kv=8, d=128, L=100000, gamma=4,
                                  V=152064, snap_window=32, snap_pool=7, snap_budget=4096,
                                  heavy_frac=0.002, heavy_cos=0.6, target_sigma=2.0, draft_noise=0.7,
                                  seed=5),
}


def gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def as_u16(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 view of its bits (host copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")


def randn_bf16(shape, g: torch.Generator, device, chunk_elems: int = 1 << 28) -> torch.Tensor:
    """N(0,1) draws rounded once (round-to-nearest-even) to bf16, filled in chunks."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk_elems):
        e = min(n, s + chunk_elems)
        flat[s:e] = torch.randn(e - s, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    return out


def _pick_positions(n_pos: int, frac: float, g: torch.Generator, device) -> torch.Tensor:
    count = max(1, int(round(frac * n_pos)))
    return torch.randperm(n_pos, generator=g, device=device)[:count]


def kv_cache(w: Workload, device, L_cap: Optional[int] = None, seed: Optional[int] = None):
    """K, V bf16 [B, L_cap, H_kv, d] ~ N(0,1).

    With ``boost_frac`` > 0, that fraction of positions (drawn per sequence and
    shared by every KV head) has its key rows scaled by ``boost``.  With
    ``heavy_frac`` > 0, that fraction of positions per (sequence, KV head)
    holds a heavy-hitter key sqrt(d) * h_hat, where h_hat is a random unit
    vector per (sequence, KV head); ``heavy_dirs`` [B, H_kv, d] (fp32) returns
    those directions so the window queries can be aligned to them.
    """
    L_cap = L_cap or w.L
    seed = w.seed if seed is None else seed
    g = gen(device, seed * 1000 + 11)
    k = randn_bf16((w.B, L_cap, w.H_kv, w.d), g, device)
    v = randn_bf16((w.B, L_cap, w.H_kv, w.d), g, device)
    heavy_dirs = None
    if w.boost_frac > 0:
        for b in range(w.B):
            pos = _pick_positions(L_cap, w.boost_frac, g, device)
            k[b, pos] = (k[b, pos].float() * w.boost).to(torch.bfloat16)
    if w.heavy_frac > 0:
        hd = torch.randn((w.B, w.H_kv, w.d), generator=g, device=device, dtype=torch.float32)
        heavy_dirs = hd / hd.norm(dim=-1, keepdim=True)
        scale = math.sqrt(w.d)
        for b in range(w.B):
            for h in range(w.H_kv):
                pos = _pick_positions(max(1, w.L - max(w.snap_window, 1)), w.heavy_frac, g, device)
                k[b, pos, h] = (heavy_dirs[b, h] * scale).to(torch.bfloat16)
    return k, v, heavy_dirs


def queries(w: Workload, n_q: int, device, seed: int) -> torch.Tensor:
    """Decode / verify queries bf16 [B, n_q, H_q, d] ~ N(0,1)."""
    g = gen(device, seed)
    return randn_bf16((w.B, n_q, w.H_q, w.d), g, device)


def window_queries(w: Workload, device, heavy_dirs: Optional[torch.Tensor] = None, seed: Optional[int] = None):
    """SnapKV observation-window queries bf16 [B, w, H_q, d].

    N(0,1) when there are no heavy hitters.  Otherwise each query is
    sqrt(d) * (c * h_hat + sqrt(1-c^2) * n_hat) with c = ``heavy_cos``, h_hat
    the KV head's heavy-hitter direction and n_hat a random unit vector
    orthogonal to it, so every window query has cosine c with the heavy keys.
    """
    seed = (w.seed if seed is None else seed) * 1000 + 23
    g = gen(device, seed)
    if heavy_dirs is None:
        return randn_bf16((w.B, w.snap_window, w.H_q, w.d), g, device)
    n = torch.randn((w.B, w.snap_window, w.H_q, w.d), generator=g, device=device, dtype=torch.float32)
    h = heavy_dirs.repeat_interleave(w.G, dim=1)[:, None, :, :]           # [B,1,H_q,d]
    n = n - (n * h).sum(-1, keepdim=True) * h
    n = n / n.norm(dim=-1, keepdim=True)
    c = w.heavy_cos
    qv = math.sqrt(w.d) * (c * h + math.sqrt(1.0 - c * c) * n)
    return qv.to(torch.bfloat16)


def logits(w: Workload, device, B: Optional[int] = None, seed: Optional[int] = None):
    """target fp32 [B, gamma+1, V] ~ N(0, target_sigma); draft = target[:, :gamma] + N(0, draft_noise);
    draft tokens drawn from softmax(draft) by the Gumbel-max trick (the draft model's own sampler);
    uniforms u_acc [B, gamma], u_res [B] in [0, 1)."""
    B = B or w.B
    seed = (w.seed if seed is None else seed) * 1000 + 37
    g = gen(device, seed)
    target = torch.randn((B, w.gamma + 1, w.V), generator=g, device=device, dtype=torch.float32) * w.target_sigma
    draft = target[:, : w.gamma] + torch.randn((B, w.gamma, w.V), generator=g, device=device,
                                               dtype=torch.float32) * w.draft_noise
    u = torch.rand((B, w.gamma, w.V), generator=g, device=device, dtype=torch.float32).clamp_(1e-20, 1.0)
    gumbel = -torch.log(-torch.log(u))
    draft_tok = torch.argmax(draft + gumbel, dim=-1).to(torch.int32)
    del u, gumbel
    u_acc = torch.rand((B, w.gamma), generator=g, device=device, dtype=torch.float32)
    u_res = torch.rand((B,), generator=g, device=device, dtype=torch.float32)
    return target.contiguous(), draft.contiguous(), draft_tok, u_acc, u_res


def ragged_lengths(B: int, lo: int, hi: int, device, seed: int) -> torch.Tensor:
    """int32 [B] lengths uniform in [lo, hi]."""
    g = gen("cpu", seed)
    return torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int32).to(device)
