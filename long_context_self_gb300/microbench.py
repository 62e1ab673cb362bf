"""Time one entry point of libmagicdec on a named synthetic workload.

    python -m long_context_self_gb300.microbench <entry> [--workload NAME] [--batch B] [--gamma G]
                                                 [--reps N] [--warmup W] [--budget K]

entry: verify | draft | topk | pq | pq_build | accept | accept_greedy | snapkv | gather | draft_cache

Inputs come from ``synth`` (seeded, resident on the GPU before timing); each
call is launched `reps` times back to back after `warmup` untimed calls and
timed with CUDA events on the current stream.  Prints one JSON line with the
mean time per call.  Meant for kernel profiling (a fixed, short sequence of
launches of one entry point) and for quick per-call measurements; the full
speculative step is timed by bench.py at the repository root.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
from typing import Callable

import torch

from . import binding as mb
from . import build, synth


def _time(fn: Callable[[], object], reps: int, warmup: int) -> float:
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / max(reps, 1)


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("entry", choices=["verify", "draft", "topk", "pq", "pq_build", "accept", "accept_greedy", "snapkv",
                                      "gather", "draft_cache"])
    ap.add_argument("--pq-centroids", type=int, default=256)
    ap.add_argument("--pq-iters", type=int, default=2)
    ap.add_argument("--workload", default="llama8b_b128_l32k", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch size")
    ap.add_argument("--gamma", type=int, default=0, help="override the workload's draft length (verify: gamma+1 rows)")
    ap.add_argument("--reps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=2)
    ap.add_argument("--budget", type=int, default=0, help="draft / Top-K / SnapKV budget (default: the workload's)")
    args = ap.parse_args(argv)

    build.build()
    mb.lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS[args.workload]
    if args.batch:
        w = dataclasses.replace(w, B=args.batch)
    if args.gamma:
        w = dataclasses.replace(w, gamma=args.gamma)
    budget = args.budget or w.stream_budget or w.snap_budget
    sl = torch.full((w.B,), w.L, dtype=torch.int32, device=dev)
    info = {"entry": args.entry, "workload": w.name, "B": w.B, "L": w.L, "H_q": w.H_q, "H_kv": w.H_kv, "d": w.d}

    if args.entry in ("verify", "topk", "snapkv", "gather", "pq", "pq_build", "draft_cache"):
        k, v, dirs = synth.kv_cache(w, dev)
    if args.entry == "verify":
        q = synth.queries(w, w.n_q, dev, seed=w.seed * 7 + 2)
        out = torch.empty_like(q)
        ws = mb.workspace(mb.magicdec_attn_workspace_size(mb.kv_shape(w.B, w.H_q, w.H_kv, w.d, w.L), w.n_q), dev, "mb")
        fn = lambda: mb.magicdec_verify_attn(q, k, v, sl, out=out, ws=ws)
        nbytes = 2.0 * w.B * w.L * w.H_kv * w.d * 2
        info["n_q"] = w.n_q
    elif args.entry == "draft":
        kc = torch.randn((w.B, w.H_kv, budget, w.d), device=dev).to(torch.bfloat16)
        vc = torch.randn_like(kc)
        q = synth.queries(w, 1, dev, seed=w.seed * 7 + 1)
        dl = torch.full((w.B,), budget, dtype=torch.int32, device=dev)
        out = torch.empty_like(q)
        ws = mb.workspace(mb.magicdec_attn_workspace_size(mb.kv_shape(w.B, w.H_q, w.H_kv, w.d, budget), 1), dev, "mb")
        fn = lambda: mb.magicdec_draft_attn(q, kc, vc, dl, out=out, ws=ws)
        nbytes = 2.0 * w.B * budget * w.H_kv * w.d * 2
        info["budget"] = budget
    elif args.entry == "topk":
        q = synth.queries(w, 1, dev, seed=w.seed * 7 + 3)
        out = torch.empty_like(q)
        idx = torch.empty((w.B, w.H_q, budget), dtype=torch.int32, device=dev)
        ws = mb.workspace(mb.magicdec_topk_attn_workspace_size(mb.kv_shape(w.B, w.H_q, w.H_kv, w.d, w.L)), dev, "mb")
        fn = lambda: mb.magicdec_topk_draft_attn(q, k, v, sl, budget, out=out, idx=idx, ws=ws)
        nbytes = float(w.B) * w.L * w.H_kv * w.d * 2 + float(w.B) * w.H_q * budget * w.d * 2
        info["budget"] = budget
    elif args.entry in ("pq", "pq_build"):
        M, C = w.d // 8, args.pq_centroids
        gen = torch.Generator(device="cpu").manual_seed(w.seed * 11 + 5)
        pick = torch.randint(0, w.L, (w.B, w.H_kv, C), generator=gen).to(dev)
        bidx = torch.arange(w.B, device=dev)[:, None, None]
        hidx = torch.arange(w.H_kv, device=dev)[None, :, None]
        init = k[bidx, pick, hidx].float().reshape(w.B, w.H_kv, C, M, 8).permute(0, 1, 3, 2, 4).contiguous()
        cb = init.clone()
        codes = torch.empty((w.B, w.H_kv, w.L, M), dtype=torch.uint8, device=dev)
        kv_bytes = float(w.B) * w.L * w.H_kv * w.d * 2

        def pq_build():
            cb.copy_(init)
            for _ in range(args.pq_iters):
                mb.magicdec_pq_encode(k, cb, codes=codes)
                mb.magicdec_pq_update(k, sl, codes, cb)
            mb.magicdec_pq_encode(k, cb, codes=codes)
        info.update(M=M, C=C, lloyd_iterations=args.pq_iters)
        if args.entry == "pq_build":
            fn = pq_build
            nbytes = (2 * args.pq_iters + 1) * kv_bytes
        else:
            pq_build()
            q = synth.queries(w, 1, dev, seed=w.seed * 7 + 3)
            out = torch.empty_like(q)
            idx = torch.empty((w.B, w.H_q, budget), dtype=torch.int32, device=dev)
            ws = mb.workspace(mb.magicdec_pq_attn_workspace_size(mb.kv_shape(w.B, w.H_q, w.H_kv, w.d, w.L)), dev,
                              "mb")
            fn = lambda: mb.magicdec_pq_draft_attn(q, k, v, sl, cb, codes, budget, out=out, idx=idx, ws=ws)
            nbytes = (float(w.B) * w.H_kv * w.L * M + float(w.B) * w.H_kv * M * C * 32
                      + 2.0 * w.B * w.H_q * budget * w.d * 2)
            info["budget"] = budget
    elif args.entry == "draft_cache":
        cap = (w.n_sink or 16) + (w.n_recent or 496)
        kc = torch.zeros((w.B, w.H_kv, cap, w.d), dtype=torch.bfloat16, device=dev)
        vc = torch.zeros_like(kc)
        i32 = lambda x: torch.full((w.B,), int(x), dtype=torch.int32, device=dev)
        L0, org, ring = w.L - w.gamma - 1, i32(w.n_sink or 16), w.n_recent or 496
        mb.magicdec_draft_cache_update(k, v, kc, vc, i32(0), i32(0), i32(L0), org, None, ring)
        app = [(i32(L0 + g), i32(L0 + g + 1)) for g in range(w.gamma)]
        back = (i32(L0), i32(L0 + w.gamma))

        def cycle():
            for lv, ln in app:
                mb.magicdec_draft_cache_update(k, v, kc, vc, lv, lv, ln, org, None, ring)
            mb.magicdec_draft_cache_update(k, v, kc, vc, back[0], back[1], back[0], org, None, ring)
        fn = cycle
        nbytes = 2.0 * w.gamma * w.B * w.H_kv * w.d * 2 * 2 * 2
        info.update(cap=cap, gamma=w.gamma)
    elif args.entry in ("accept", "accept_greedy"):
        greedy = args.entry == "accept_greedy"
        target, draft, tok, u_acc, u_res = synth.logits(w, dev)
        fn = lambda: mb.magicdec_spec_accept(target, draft, tok, u_acc, u_res, greedy)
        nbytes = 4.0 * w.B * ((w.gamma + 1) if greedy else (2 * w.gamma + 1)) * w.V
        info.update(gamma=w.gamma, V=w.V)
    elif args.entry == "snapkv":
        sb = args.budget or w.snap_budget or 512
        win = w.snap_window or 32
        sw = dataclasses.replace(w, snap_window=win, snap_budget=sb)
        q_win = synth.window_queries(sw, dev, heavy_dirs=dirs)
        fn = lambda: mb.magicdec_snapkv_select(q_win, k, sl, win, w.snap_pool, sb)
        nbytes = 2.0 * w.B * w.L * w.H_kv * w.d * 2
        info.update(budget=sb, window=win)
    else:   # gather
        idx, _ = mb.magicdec_streaming_select(sl, w.H_kv, w.n_sink or 16, w.n_recent or 496)
        cap = idx.shape[2]
        kc = torch.empty((w.B, w.H_kv, cap, w.d), dtype=torch.bfloat16, device=dev)
        vc = torch.empty_like(kc)
        fn = lambda: mb.magicdec_gather_kv(k, v, idx, cap, kc=kc, vc=vc)
        nbytes = 2.0 * 2 * w.B * cap * w.H_kv * w.d * 2
        info["cap"] = cap

    ms = _time(fn, args.reps, args.warmup)
    info.update(ms_per_call=round(ms, 5), algorithmic_bytes=nbytes, gbs=round(nbytes / (ms * 1e-3) / 1e9, 1),
                reps=args.reps, warmup=args.warmup, device_error_word=mb.magicdec_device_error())
    print(json.dumps(info))


if __name__ == "__main__":
    main()
