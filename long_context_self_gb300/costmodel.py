"""Drafting-strategy selector of MagicDec (paper section 3.1 Eq. 1-2, section 4.1 Eq. 3-4).

Given per-call times of the attention hot path -- the target's decode step T_T(B,S),
the draft step over a K-row sparse cache T_D(B,K), the verification of gamma tokens
T_V(B,S,gamma) and the selection cost T_select(B,S,K) -- and the draft acceptance rate
alpha of each (method, budget), the expected time per generated token of speculative
decoding is

    T_avg(gamma, K, method) = (gamma * (T_D(B,K) + T_select(B,S,K)) + T_V(B,S,gamma)) / Omega(gamma, alpha)
    Omega(gamma, alpha)     = (1 - alpha^(gamma+1)) / (1 - alpha)                          (Eq. 1)

and the selector returns the (method, K, gamma) that minimises T_avg / T_T (Eq. 4), with
the predicted speedup T_T / T_avg (the inverse of Eq. 2's ratio).

`calibrate()` measures the times on the current GPU through the library's entry points
(verification with n_q = 1 is the target's own decode step); `select()` is pure host
arithmetic.  Times here cover the attention part only; `other_ms` adds a fixed per-step
cost (projections, MLP) for callers that have one.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Callable, Dict, Iterable, Optional, Sequence, Tuple


def expected_tokens(gamma: int, alpha: float) -> float:
    """Eq. 1: expected tokens generated per verification step."""
    if gamma < 0:
        raise ValueError("gamma must be >= 0")
    if alpha >= 1.0:
        return float(gamma + 1)
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


def avg_time_per_token(gamma: int, alpha: float, t_draft: float, t_select: float, t_verify: float) -> float:
    """T_avg^SD = (gamma * (T_D + T_select) + T_V) / Omega (sections 3.1 and 4.1, Eq. 3)."""
    return (gamma * (t_draft + t_select) + t_verify) / expected_tokens(gamma, alpha)


@dataclasses.dataclass(frozen=True)
class Choice:
    method: str
    budget: int
    gamma: int
    t_avg: float          # expected time per generated token
    ratio: float          # T_avg / T_T (Eq. 2 / Eq. 4 objective)
    speedup: float        # T_T / T_avg


@dataclasses.dataclass
class Timings:
    """Per-call times (ms) for one (B, S): target decode, verification per gamma, draft per
    budget, and selection cost per (method, budget) charged to each draft step."""
    t_target: float
    t_verify: Dict[int, float]
    t_draft: Dict[int, float]
    t_select: Dict[Tuple[str, int], float] = dataclasses.field(default_factory=dict)
    other_ms: float = 0.0             # non-attention time of every forward pass (target, draft, verify)


def select(tim: Timings, alpha: Dict[Tuple[str, int], float], gammas: Optional[Iterable[int]] = None) -> Choice:
    """Eq. 4: argmin over (method, budget, gamma) of T_avg / T_T.  `alpha` maps
    (method, budget) -> acceptance rate; gammas default to the measured verify gammas."""
    gammas = sorted(tim.t_verify) if gammas is None else sorted(gammas)
    t_t = tim.t_target + tim.other_ms
    best: Optional[Choice] = None
    for (method, budget), a in sorted(alpha.items()):
        if budget not in tim.t_draft:
            continue
        t_d = tim.t_draft[budget] + tim.other_ms
        t_s = tim.t_select.get((method, budget), 0.0)
        for g in gammas:
            if g < 1 or g not in tim.t_verify:
                continue
            t_avg = avg_time_per_token(g, a, t_d, t_s, tim.t_verify[g] + tim.other_ms)
            c = Choice(method, budget, g, t_avg, t_avg / t_t, t_t / t_avg)
            if best is None or c.t_avg < best.t_avg:
                best = c
    if best is None:
        raise ValueError("no (method, budget, gamma) combination has timings")
    return best


def calibrate(B: int, S: int, budgets: Sequence[int], gammas: Sequence[int], H_q: int = 32, H_kv: int = 8,
              d: int = 128, reps: int = 10, device: str = "cuda:0", snapkv_window: int = 32,
              snapkv_steps: Optional[int] = None, topk: bool = False, pq: bool = False,
              pq_centroids: int = 256, pq_iters: int = 2) -> Timings:
    """Measure T_T, T_V(gamma), T_D(K) (and the SnapKV selection cost spread over
    `snapkv_steps` draft steps) for one layer on the current GPU, in ms.  With
    `topk`, the Top-K attention draft is timed too: its per-step search over the
    whole cache is charged as T_select = (measured Top-K call) - T_D(K), so that
    T_D + T_select is the call's time (section 4.4: dynamic selection pays a
    batch-dependent search at every draft step).  With `pq`, the PQCache-style
    draft is charged the same way (its codebook, built once at prefill from
    seeded key samples, is not charged per step)."""
    import torch

    from . import binding as mb

    def timed(fn) -> float:
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    g = torch.Generator(device=device).manual_seed(0)
    k = torch.randn((B, S, H_kv, d), generator=g, device=device).to(torch.bfloat16)
    v = torch.randn((B, S, H_kv, d), generator=g, device=device).to(torch.bfloat16)
    sl = torch.full((B,), S, dtype=torch.int32, device=device)
    t_verify = {}
    for gm in sorted(set(gammas) | {0}):
        q = torch.randn((B, gm + 1, H_q, d), generator=g, device=device).to(torch.bfloat16)
        t_verify[gm] = timed(lambda: mb.magicdec_verify_attn(q, k, v, sl))
    t_target = t_verify.pop(0)
    t_draft = {}
    qd = torch.randn((B, 1, H_q, d), generator=g, device=device).to(torch.bfloat16)
    for K in budgets:
        kc = torch.randn((B, H_kv, K, d), generator=g, device=device).to(torch.bfloat16)
        vc = torch.randn((B, H_kv, K, d), generator=g, device=device).to(torch.bfloat16)
        dl = torch.full((B,), K, dtype=torch.int32, device=device)
        t_draft[K] = timed(lambda: mb.magicdec_draft_attn(qd, kc, vc, dl))
        del kc, vc
    t_select: Dict[Tuple[str, int], float] = {}
    for K in budgets:
        t_select[("streaming", K)] = 0.0      # sinks + window of the current length: no search
    if topk:
        for K in budgets:
            if K > S:
                continue
            t = timed(lambda: mb.magicdec_topk_draft_attn(qd, k, v, sl, K))
            t_select[("topk", K)] = max(0.0, t - t_draft[K])
    if pq:
        M, C = d // 8, pq_centroids
        gen = torch.Generator(device="cpu").manual_seed(7)
        pick = torch.randint(0, S, (B, H_kv, C), generator=gen).to(device)
        bidx = torch.arange(B, device=device)[:, None, None]
        hidx = torch.arange(H_kv, device=device)[None, :, None]
        cb = k[bidx, pick, hidx].float().reshape(B, H_kv, C, M, 8).permute(0, 1, 3, 2, 4).contiguous()
        codes = mb.magicdec_pq_encode(k, cb)
        for _ in range(pq_iters):
            mb.magicdec_pq_update(k, sl, codes, cb)
            mb.magicdec_pq_encode(k, cb, codes=codes)
        for K in budgets:
            if K > S:
                continue
            t = timed(lambda: mb.magicdec_pq_draft_attn(qd, k, v, sl, cb, codes, K))
            t_select[("pq", K)] = max(0.0, t - t_draft[K])
        del cb, codes
    if snapkv_steps:
        q_win = torch.randn((B, snapkv_window, H_q, d), generator=g, device=device).to(torch.bfloat16)
        for K in budgets:
            if K < snapkv_window:
                continue
            t = timed(lambda: mb.magicdec_snapkv_select(q_win, k, sl, snapkv_window, 7, K))
            t_select[("snapkv", K)] = t / snapkv_steps      # once per prefill, amortised
    return Timings(t_target=t_target, t_verify=t_verify, t_draft=t_draft, t_select=t_select)


def main(argv: Optional[Sequence[str]] = None) -> None:
    import argparse
    import json

    ap = argparse.ArgumentParser(description="calibrate the attention hot path and pick a drafting strategy")
    ap.add_argument("--B", type=int, default=128)
    ap.add_argument("--S", type=int, default=32000)
    ap.add_argument("--budgets", type=int, nargs="+", default=[256, 512, 1024, 2048])
    ap.add_argument("--gammas", type=int, nargs="+", default=[1, 2, 3, 4, 5, 6])
    ap.add_argument("--alpha", type=str, default="{}",
                    help='JSON {"streaming:512": 0.8, "snapkv:2048": 0.9, ...}; default: no selection')
    ap.add_argument("--snapkv-steps", type=int, default=0)
    ap.add_argument("--topk", action="store_true", help="also time the Top-K attention draft")
    ap.add_argument("--pq", action="store_true", help="also time the PQCache-style draft")
    args = ap.parse_args(argv)
    tim = calibrate(args.B, args.S, args.budgets, args.gammas, snapkv_steps=args.snapkv_steps or None,
                    topk=args.topk, pq=args.pq)
    out = {"B": args.B, "S": args.S, "t_target_ms": tim.t_target, "t_verify_ms": tim.t_verify,
           "t_draft_ms": tim.t_draft, "T_V_over_T_T": {g: t / tim.t_target for g, t in tim.t_verify.items()},
           "T_D_over_T_T": {K: t / tim.t_target for K, t in tim.t_draft.items()},
           "t_select_ms": {f"{m}:{K}": t for (m, K), t in tim.t_select.items()}}
    alpha = {tuple((key.split(":")[0], int(key.split(":")[1]))): a for key, a in json.loads(args.alpha).items()}
    if alpha:
        out["choice"] = dataclasses.asdict(select(tim, alpha))
    print(json.dumps(out))


if __name__ == "__main__":
    main()
