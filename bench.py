"""Benchmark of the MagicDec self-speculative decoding hot path on GB300.

One timed step is one speculative-decoding step of the attention-only path over
one batch, for every decoder layer (paper section 3.1: T_SD = gamma * T_D + T_V,
then acceptance):

    for each of `layers` layers:
        StreamingLLM selection (sinks + recent window of the current lengths)
        gather of the selected rows into the compact draft cache
        gamma x draft attention over the compact cache
        verification attention of the gamma+1 speculated queries over the full cache
    speculative accept / resample over the vocabulary

Each layer reuses one layer's KV cache (16.8 GB at B=128, L=32000, far larger
than the 129 MB L2, so no layer sees another's data in cache).  SnapKV selection
runs once after prefill in the method; it is timed once per run and reported
beside the step.  Inputs are synthetic (seeded; see long_context_self_gb300.synth).

`python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]` prints
one JSON line.  Under torchrun each rank runs its own batch on its own GPU (the
path shards by sequence with no exchange; weak scaling).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from long_context_self_gb300 import synth  # noqa: E402

DEFAULT_WORKLOAD = "llama8b_b128_l32k"
METRIC = "verify/draft attn achieved HBM GB/s (% of peak); spec steps/s at B=128 L=32k"
LAYERS = 32
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "verify_attn_llama8b_b128_l32k.md")
ATTN_SRC = os.path.join(ROOT, "long_context_self_gb300", "csrc", "attn_heads.cu")   # the verification kernel at this shape


# --------------------------------------------------------------------- helpers
def spec_step_time(gamma_t_draft: float, t_verify: float, omega: float) -> float:
    """Expected time per generated token, T_SD = (gamma*T_D + T_V) / Omega (paper section 3.1)."""
    return (gamma_t_draft + t_verify) / omega


def expected_tokens(alpha: float, gamma: int) -> float:
    """Eq. 1: Omega(gamma, alpha) = (1 - alpha^(gamma+1)) / (1 - alpha)."""
    if alpha >= 1.0:
        return gamma + 1.0
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


def max_over_ranks(x: float, device=None) -> float:
    """Max of a per-rank float over the process group (identity without one)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    dev = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(world: int, steps: int, ms_max: float) -> float:
    """Whole-job steps/s: every rank runs `steps` steps of its own batch; the job takes the
    slowest rank's time."""
    return world * steps / (ms_max * 1e-3)


def rank_workload(w, rank: int):
    """The workload one rank runs: rank r draws its own sequences (seed offset by 100·r), so
    N replicas process N distinct batches; rank 0 keeps the workload's own seed."""
    return w if rank == 0 else dataclasses.replace(w, seed=w.seed + 100 * rank)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def file_sha(path: str) -> str:
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(workload: str):
    """Per-launch DRAM bytes of verify_attn from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    try:
        text = open(PROFILE_TRAFFIC).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ": " in line and line.strip().startswith("- "):
            key, _, val = line.strip()[2:].partition(": ")   # keys may contain ':' (e.g. "sha256[:16]")
            vals[key.strip()] = val.strip().strip("`")
    if vals.get("workload") != workload or vals.get("attn_heads.cu sha256[:16]") != file_sha(ATTN_SRC):
        return None
    try:
        return float(vals["dram bytes per launch (full workload)"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"magicdec_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return None
        try:
            rows = [r.split(",") for r in open(self.path).read().strip().splitlines() if r.strip()]
        except OSError:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------ our arm
class Pipeline:
    """Device buffers and the per-step call sequence, all through the C-ABI binding."""

    def __init__(self, w: synth.Workload, device, layers: int):
        from long_context_self_gb300 import binding as mb
        self.mb = mb
        self.w, self.dev, self.layers = w, device, layers
        self.k, self.v, _ = synth.kv_cache(w, device)
        self.seq_len = torch.full((w.B,), w.L, dtype=torch.int32, device=device)
        self.q_draft = synth.queries(w, 1, device, seed=w.seed * 7 + 1)
        self.q_verify = synth.queries(w, w.n_q, device, seed=w.seed * 7 + 2)
        self.cap = w.stream_budget
        self.idx = torch.empty((w.B, w.H_kv, self.cap), dtype=torch.int32, device=device)
        self.n_sel = torch.empty((w.B,), dtype=torch.int32, device=device)
        self.kc = torch.zeros((w.B, w.H_kv, self.cap, w.d), dtype=torch.bfloat16, device=device)
        self.vc = torch.zeros_like(self.kc)
        self.out_d = torch.empty_like(self.q_draft)
        self.out_v = torch.empty_like(self.q_verify)
        self.target, self.draft, self.tok, self.u_acc, self.u_res = synth.logits(w, device)
        self.n_acc = torch.empty((w.B,), dtype=torch.int32, device=device)
        self.out_tok = torch.empty((w.B, w.n_q), dtype=torch.int32, device=device)
        self.n_amb = torch.empty((w.B,), dtype=torch.int32, device=device)
        shape = mb.kv_shape(w.B, w.H_q, w.H_kv, w.d, w.L)
        ws_attn = max(mb.magicdec_attn_workspace_size(shape, w.n_q),
                      mb.magicdec_attn_workspace_size(mb.kv_shape(w.B, w.H_q, w.H_kv, w.d, self.cap), 1))
        self.ws_attn = torch.zeros(ws_attn, dtype=torch.uint8, device=device)
        self.ws_acc = torch.zeros(mb.magicdec_spec_accept_workspace_size(w.B, w.gamma, w.V), dtype=torch.uint8,
                                  device=device)
        # per layer: streaming select, gather, gamma draft attentions, verification;
        # accept (sampling mode): statistics, chain, chunk sums, draw
        self.launches_per_step = layers * (3 + w.gamma) + 4
        self.verify_events = []
        # The same draft kept as a StreamingLLM ring (sinks + recent window) by
        # magicdec_draft_cache_update: built once, then per layer gamma one-row
        # appends of the drafted positions and a post-verification update that
        # restores the ring slots they displaced (length L0 = L - gamma - 1).
        i32 = lambda x: torch.full((w.B,), int(x), dtype=torch.int32, device=device)
        self.L0 = w.L - w.gamma - 1
        self.r_origin = i32(w.n_sink)
        self.rkc = torch.zeros_like(self.kc)
        self.rvc = torch.zeros_like(self.kc)
        self.r_dl = torch.empty((w.B,), dtype=torch.int32, device=device)
        self.r_app = [(i32(self.L0 + g), i32(self.L0 + g + 1)) for g in range(w.gamma)]
        self.r_back = (i32(self.L0), i32(self.L0 + w.gamma))
        zero = i32(0)
        mb.magicdec_draft_cache_update(self.k, self.v, self.rkc, self.rvc, zero, zero, i32(self.L0), self.r_origin,
                                       None, w.n_recent, draft_len=self.r_dl)
        self.launches_per_step_ring = layers * (2 * w.gamma + 2) + 4

    def step(self, record: bool = False):
        mb, w = self.mb, self.w
        for _ in range(self.layers):
            mb.magicdec_streaming_select(self.seq_len, w.H_kv, w.n_sink, w.n_recent, idx=self.idx, n_sel=self.n_sel)
            mb.magicdec_gather_kv(self.k, self.v, self.idx, self.cap, kc=self.kc, vc=self.vc)
            for _g in range(w.gamma):
                mb.magicdec_draft_attn(self.q_draft, self.kc, self.vc, self.n_sel, out=self.out_d, ws=self.ws_attn)
            if record:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
            mb.magicdec_verify_attn(self.q_verify, self.k, self.v, self.seq_len, out=self.out_v, ws=self.ws_attn)
            if record:
                e1.record()
                self.verify_events.append((e0, e1))
        mb.magicdec_spec_accept(self.target, self.draft, self.tok, self.u_acc, self.u_res, False, n_acc=self.n_acc,
                                out_tok=self.out_tok, n_amb=self.n_amb, ws=self.ws_acc)

    def ring_updates(self):
        """One layer's draft-cache maintenance: gamma appends and the post-verification update."""
        mb, w = self.mb, self.w
        for lv, ln in self.r_app:
            mb.magicdec_draft_cache_update(self.k, self.v, self.rkc, self.rvc, lv, lv, ln, self.r_origin, None,
                                           w.n_recent, draft_len=self.r_dl)
        mb.magicdec_draft_cache_update(self.k, self.v, self.rkc, self.rvc, self.r_back[0], self.r_back[1],
                                       self.r_back[0], self.r_origin, None, w.n_recent, draft_len=self.r_dl)

    def step_ring(self):
        """The step with the StreamingLLM draft cache maintained incrementally (no per-step gather)."""
        mb, w = self.mb, self.w
        for _ in range(self.layers):
            for lv, ln in self.r_app:
                mb.magicdec_draft_attn(self.q_draft, self.rkc, self.rvc, self.r_dl, out=self.out_d, ws=self.ws_attn)
                mb.magicdec_draft_cache_update(self.k, self.v, self.rkc, self.rvc, lv, lv, ln, self.r_origin, None,
                                               w.n_recent, draft_len=self.r_dl)
            mb.magicdec_verify_attn(self.q_verify, self.k, self.v, self.seq_len, out=self.out_v, ws=self.ws_attn)
            mb.magicdec_draft_cache_update(self.k, self.v, self.rkc, self.rvc, self.r_back[0], self.r_back[1],
                                           self.r_back[0], self.r_origin, None, w.n_recent, draft_len=self.r_dl)
        mb.magicdec_spec_accept(self.target, self.draft, self.tok, self.u_acc, self.u_res, False, n_acc=self.n_acc,
                                out_tok=self.out_tok, n_amb=self.n_amb, ws=self.ws_acc)

    def ring_update_bytes(self) -> float:
        """gamma appended rows + gamma restored rows per layer, K and V, read + written."""
        w = self.w
        return 2.0 * w.gamma * w.B * w.H_kv * w.d * 2 * 2 * 2

    # algorithmic bytes
    def verify_bytes(self) -> float:
        w = self.w
        kv = 2.0 * w.B * w.L * w.H_kv * w.d * 2
        return kv + 2.0 * w.B * w.n_q * w.H_q * w.d * 2

    def draft_bytes(self) -> float:
        w = self.w
        return 2.0 * w.B * self.cap * w.H_kv * w.d * 2 + 2.0 * w.B * w.H_q * w.d * 2

    def accept_bytes(self) -> float:
        w = self.w
        return 4.0 * w.B * (2 * w.gamma + 1) * w.V


def time_component(fn, reps: int) -> float:
    """Mean device ms of fn() over reps launches (CUDA events on the current stream)."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    fn()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def time_graph(fn, reps: int) -> float:
    """Mean device ms of fn() replayed from a CUDA graph (for calls short enough that the
    binding's host-side argument checks, not the GPU, would set the pace of direct launches)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    del g
    return e0.elapsed_time(e1) / reps


def run_ours(args, rank: int, world: int, local_rank: int):
    from long_context_self_gb300 import binding as mb
    from long_context_self_gb300 import build as lbuild
    lbuild.build()
    mb.lib()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    w = synth.WORKLOADS[args.workload]
    if args.batch:
        w = dataclasses.replace(w, B=args.batch)
    w = rank_workload(w, rank)
    pipe = Pipeline(w, device, args.layers)
    torch.cuda.synchronize()

    # SnapKV selection (once after prefill in the method) and its gather: timed separately.
    snap = {}
    if w.snap_budget:
        sw = synth.Workload("snap", B=w.B, H_q=w.H_q, H_kv=w.H_kv, d=w.d, L=w.L, gamma=w.gamma, V=w.V,
                            snap_window=w.snap_window, snap_pool=w.snap_pool, snap_budget=w.snap_budget,
                            seed=w.seed)
        q_win = synth.window_queries(sw, device)
        ws_snap = torch.zeros(mb.magicdec_snapkv_workspace_size(mb.kv_shape(w.B, w.H_q, w.H_kv, w.d, w.L),
                                                                 w.snap_window), dtype=torch.uint8, device=device)
        sidx = torch.empty((w.B, w.H_kv, w.snap_budget), dtype=torch.int32, device=device)
        sn = torch.empty((w.B,), dtype=torch.int32, device=device)
        skc = torch.zeros((w.B, w.H_kv, w.snap_budget, w.d), dtype=torch.bfloat16, device=device)
        svc = torch.zeros_like(skc)
        t_sel = time_component(lambda: mb.magicdec_snapkv_select(q_win, pipe.k, pipe.seq_len, w.snap_window,
                                                                  w.snap_pool, w.snap_budget, idx=sidx, n_sel=sn,
                                                                  ws=ws_snap), 3)
        t_gat = time_component(lambda: mb.magicdec_gather_kv(pipe.k, pipe.v, sidx, w.snap_budget, kc=skc, vc=svc), 5)
        snap = {"snapkv_select_ms_per_layer": round(t_sel, 4), "snapkv_gather_ms_per_layer": round(t_gat, 4),
                "snapkv_budget": w.snap_budget, "snapkv_window": w.snap_window,
                # algorithmic bytes: K read once per scoring pass (prefix for the second) + scores
                "_snap_bytes": 2.0 * w.B * w.L * w.H_kv * w.d * 2 + 8.0 * w.B * w.H_kv * w.L,
                "_snap_ms": t_sel}
        del q_win, ws_snap, sidx, sn, skc, svc
        torch.cuda.empty_cache()

    for _ in range(args.warmup):
        pipe.step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    stream = torch.cuda.current_stream(device)
    with ClockSampler(local_rank) as clocks:
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record(stream)
        for _ in range(args.steps):
            pipe.step(record=True)
        t1.record(stream)
        torch.cuda.synchronize()
    ms_total = max_over_ranks(t0.elapsed_time(t1), device)
    ms_step = ms_total / args.steps
    ver_ms = statistics.mean(a.elapsed_time(b) for a, b in pipe.verify_events)
    # draft launches are timed back to back outside the step (events between the
    # step's kernels would serialise their programmatic-dependent launches): one
    # step's gamma x layers calls replayed from a CUDA graph, so that the
    # binding's host-side checks cannot set the pace of these ~50 us calls
    n_dra = w.gamma * args.layers
    dra_ms = time_graph(lambda: [mb.magicdec_draft_attn(pipe.q_draft, pipe.kc, pipe.vc, pipe.n_sel,
                                                        out=pipe.out_d, ws=pipe.ws_attn) for _ in range(n_dra)],
                        3) / n_dra
    acc_ms = time_component(lambda: mb.magicdec_spec_accept(pipe.target, pipe.draft, pipe.tok, pipe.u_acc,
                                                            pipe.u_res, False, n_acc=pipe.n_acc,
                                                            out_tok=pipe.out_tok, n_amb=pipe.n_amb,
                                                            ws=pipe.ws_acc), 5)
    sel_ms = time_component(lambda: (mb.magicdec_streaming_select(pipe.seq_len, w.H_kv, w.n_sink, w.n_recent,
                                                                  idx=pipe.idx, n_sel=pipe.n_sel),
                                     mb.magicdec_gather_kv(pipe.k, pipe.v, pipe.idx, pipe.cap, kc=pipe.kc,
                                                           vc=pipe.vc)), 5)
    # PQCache-style draft at the same budget: codebook built once (2 Lloyd
    # iterations from seeded key samples, then the final encode), then the
    # per-draft-step search (LUT scores over the codes, select, exact attention)
    pq = {}
    if not args.no_pq:
        M, C, iters = w.d // 8, 256, 2
        gen = torch.Generator(device="cpu").manual_seed(w.seed * 11 + 5)
        pick = torch.randint(0, w.L, (w.B, w.H_kv, C), generator=gen).to(device)
        bidx = torch.arange(w.B, device=device)[:, None, None]
        hidx = torch.arange(w.H_kv, device=device)[None, :, None]
        init = pipe.k[bidx, pick, hidx].float().reshape(w.B, w.H_kv, C, M, 8).permute(0, 1, 3, 2, 4).contiguous()
        cb = init.clone()
        codes = torch.empty((w.B, w.H_kv, w.L, M), dtype=torch.uint8, device=device)

        def pq_build():
            cb.copy_(init)
            for _ in range(iters):
                mb.magicdec_pq_encode(pipe.k, cb, codes=codes)
                mb.magicdec_pq_update(pipe.k, pipe.seq_len, codes, cb)
            mb.magicdec_pq_encode(pipe.k, cb, codes=codes)
        build_ms = time_component(pq_build, 1)
        pq_idx = torch.empty((w.B, w.H_q, pipe.cap), dtype=torch.int32, device=device)
        pq_out = torch.empty_like(pipe.q_draft)
        pq_ws = torch.empty(mb.magicdec_pq_attn_workspace_size(mb.kv_shape(w.B, w.H_q, w.H_kv, w.d, w.L)),
                            dtype=torch.uint8, device=device)
        pq_ms = time_component(lambda: mb.magicdec_pq_draft_attn(pipe.q_draft, pipe.k, pipe.v, pipe.seq_len, cb, codes,
                                                                 pipe.cap, out=pq_out, idx=pq_idx, ws=pq_ws), 5)
        kv_bytes = float(w.B) * w.L * w.H_kv * w.d * 2
        pq = {"pq_draft_us_per_layer": round(pq_ms * 1e3, 2), "pq_build_ms_per_layer": round(build_ms, 3),
              "pq_M": M, "pq_C": C, "pq_lloyd_iterations": iters,
              "_pq_bytes": (float(w.B) * w.H_kv * w.L * M + float(w.B) * w.H_kv * M * C * 8 * 4
                            + 2.0 * w.B * w.H_q * pipe.cap * w.d * 2 + 2.0 * w.B * w.H_q * w.d * 2),
              "_pq_ms": pq_ms,
              # each encode and each update reads K once; codes written per encode
              "_pq_build_bytes": (2 * iters + 1) * kv_bytes + (iters + 1) * float(w.B) * w.H_kv * w.L * M,
              "_pq_build_ms": build_ms}
        del init, cb, codes, pq_idx, pq_out, pq_ws, pick
        torch.cuda.empty_cache()
    ring_ms = time_graph(pipe.ring_updates, 20)
    # the step with the ring-maintained draft cache, timed like the headline step
    for _ in range(args.warmup):
        pipe.step_ring()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    r0.record()
    for _ in range(args.steps):
        pipe.step_ring()
    r1.record()
    torch.cuda.synchronize()
    ring_total = max_over_ranks(r0.elapsed_time(r1), device)
    ring_step = {"value": round(aggregate_rate(world, args.steps, ring_total), 4), "unit": "steps/s",
                 "ms_per_step": round(ring_total / args.steps, 4), "gpu_launches": pipe.launches_per_step_ring * args.steps,
                 "draft": f"StreamingLLM {w.n_sink}+{w.n_recent} kept as a ring by magicdec_draft_cache_update "
                          f"({w.gamma} appends + 1 post-verification update per layer, no per-step gather)"}
    omega_hat = float((pipe.n_acc.float() + 1).mean().item())
    # Top-K attention draft at the same budget: the dynamic-selection draft whose
    # per-step search reads the whole K cache (timed per call, outside the step)
    topk = {}
    if not args.no_topk:
        tk_idx = torch.empty((w.B, w.H_q, pipe.cap), dtype=torch.int32, device=device)
        tk_out = torch.empty_like(pipe.q_draft)
        tk_ws = torch.empty(mb.magicdec_topk_attn_workspace_size(mb.kv_shape(w.B, w.H_q, w.H_kv, w.d, w.L)),
                            dtype=torch.uint8, device=device)
        tk_ms = time_component(lambda: mb.magicdec_topk_draft_attn(pipe.q_draft, pipe.k, pipe.v, pipe.seq_len,
                                                                   pipe.cap, out=tk_out, idx=tk_idx, ws=tk_ws), 5)
        topk = {"topk_draft_us_per_layer": round(tk_ms * 1e3, 2), "topk_budget": pipe.cap,
                "_topk_bytes": (float(w.B) * w.L * w.H_kv * w.d * 2 + float(w.B) * w.H_q * pipe.cap * w.d * 2
                                + 2.0 * w.B * w.H_q * w.d * 2),
                "_topk_ms": tk_ms}
        del tk_idx, tk_out, tk_ws
        torch.cuda.empty_cache()

    # ---------------------------------------------- end to end from host buffers
    # Every step copies that step's inputs from pinned host memory -- the
    # queries of every layer and draft step, the logits, draft tokens and
    # uniforms -- and reads n_acc / out_tok back.  The copies run on a copy
    # stream into per-layer buffers; the compute stream waits on per-layer
    # events, so the transfer overlaps the attention of earlier layers.
    h_qd = pipe.q_draft.cpu().pin_memory()
    h_qv = pipe.q_verify.cpu().pin_memory()
    h_t, h_d = pipe.target.cpu().pin_memory(), pipe.draft.cpu().pin_memory()
    h_tok, h_ua, h_ur = pipe.tok.cpu().pin_memory(), pipe.u_acc.cpu().pin_memory(), pipe.u_res.cpu().pin_memory()
    h_nacc = torch.empty_like(pipe.n_acc, device="cpu").pin_memory()
    h_out = torch.empty_like(pipe.out_tok, device="cpu").pin_memory()
    d_qd = [[torch.empty_like(pipe.q_draft) for _ in range(w.gamma)] for _ in range(args.layers)]
    d_qv = [torch.empty_like(pipe.q_verify) for _ in range(args.layers)]
    copy_stream = torch.cuda.Stream(device)
    h2d = (h_qd.numel() * 2 * w.gamma + h_qv.numel() * 2) * args.layers + \
        (h_t.numel() + h_d.numel() + h_ua.numel() + h_ur.numel()) * 4 + h_tok.numel() * 4
    d2h = (h_nacc.numel() + h_out.numel()) * 4

    def e2e_step():
        mbb = mb
        compute = torch.cuda.current_stream(device)
        layer_ready = []
        copy_stream.wait_stream(compute)            # the previous step no longer reads these buffers
        with torch.cuda.stream(copy_stream):
            for ly in range(args.layers):
                for g in range(w.gamma):
                    d_qd[ly][g].copy_(h_qd, non_blocking=True)
                d_qv[ly].copy_(h_qv, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(copy_stream)
                layer_ready.append(ev)
            pipe.target.copy_(h_t, non_blocking=True)
            pipe.draft.copy_(h_d, non_blocking=True)
            pipe.tok.copy_(h_tok, non_blocking=True)
            pipe.u_acc.copy_(h_ua, non_blocking=True)
            pipe.u_res.copy_(h_ur, non_blocking=True)
            logits_ready = torch.cuda.Event()
            logits_ready.record(copy_stream)
        for ly in range(args.layers):
            mbb.magicdec_streaming_select(pipe.seq_len, w.H_kv, w.n_sink, w.n_recent, idx=pipe.idx, n_sel=pipe.n_sel)
            mbb.magicdec_gather_kv(pipe.k, pipe.v, pipe.idx, pipe.cap, kc=pipe.kc, vc=pipe.vc)
            compute.wait_event(layer_ready[ly])
            for g in range(w.gamma):
                mbb.magicdec_draft_attn(d_qd[ly][g], pipe.kc, pipe.vc, pipe.n_sel, out=pipe.out_d, ws=pipe.ws_attn)
            mbb.magicdec_verify_attn(d_qv[ly], pipe.k, pipe.v, pipe.seq_len, out=pipe.out_v, ws=pipe.ws_attn)
        compute.wait_event(logits_ready)
        mbb.magicdec_spec_accept(pipe.target, pipe.draft, pipe.tok, pipe.u_acc, pipe.u_res, False, n_acc=pipe.n_acc,
                                 out_tok=pipe.out_tok, n_amb=pipe.n_amb, ws=pipe.ws_acc)
        h_nacc.copy_(pipe.n_acc, non_blocking=True)
        h_out.copy_(pipe.out_tok, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        e2e_step()
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), device)
    del d_qd, d_qv
    graph = None
    if args.graph:
        # The same step captured once into a CUDA graph (kernels keep their
        # programmatic-dependency edges) and replayed: no host work per step.
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(device)
        side.wait_stream(torch.cuda.current_stream(device))
        with torch.cuda.stream(side):
            pipe.step()
        torch.cuda.current_stream(device).wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            pipe.step()
        for _ in range(args.warmup):
            g.replay()
        torch.cuda.synchronize()
        ge0, ge1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ge0.record()
        for _ in range(args.steps):
            g.replay()
        ge1.record()
        torch.cuda.synchronize()
        g_ms = max_over_ranks(ge0.elapsed_time(ge1), device)
        graph = {"value": round(aggregate_rate(world, args.steps, g_ms), 4), "unit": "steps/s",
                 "ms_per_step": round(g_ms / args.steps, 4)}
        del g
    err_word = mb.magicdec_device_error()

    peak, peak_kind = load_peaks()
    vbytes, dbytes = pipe.verify_bytes(), pipe.draft_bytes()
    ver_gbs = vbytes / (ver_ms * 1e-3) / 1e9
    dra_gbs = dbytes / (dra_ms * 1e-3) / 1e9
    traffic = recorded_traffic(args.workload)

    def row(nbytes, ms, bound="hbm"):
        gbs = nbytes / (ms * 1e-3) / 1e9
        return {"gbs": round(gbs, 1), "frac": round(gbs / peak, 4), "us": round(ms * 1e3, 2),
                "algorithmic_bytes": nbytes, "bound": bound}
    sg_bytes = 2.0 * 2 * w.B * pipe.cap * w.H_kv * w.d * 2       # gather: read + write K and V rows
    rows = {"verify_attn": row(vbytes, ver_ms), "draft_attn": row(dbytes, dra_ms),
            "streaming_select+gather_kv": row(sg_bytes, sel_ms), "spec_accept": row(pipe.accept_bytes(), acc_ms),
            "draft_cache_update (gamma appends + post-verification update, per layer)":
                row(pipe.ring_update_bytes(), ring_ms, "launch latency (6 MB of row copies in 4 launches)")}
    if snap:
        rows["snapkv_select (once per prefill)"] = row(snap.pop("_snap_bytes"), snap.pop("_snap_ms"))
    if pq:
        pq_ms = pq.pop("_pq_ms")
        rows["pq_draft_attn (LUT scores + select + exact attend, per draft step)"] = row(
            pq.pop("_pq_bytes"), pq_ms, "shared-memory lookup-table reads (score pass); latency (select)")
        b_ms = pq.pop("_pq_build_ms")
        rows["pq_build (2 Lloyd iterations + encode, once per prefill)"] = row(
            pq.pop("_pq_build_bytes"), b_ms,
            "ALU issue (encode: argmin over C centroids per subspace; the dot products on the tensor cores)")
        # encode: per (position, KV head, subspace, centroid) an 8-term dot product and a norm
        # term, as FP32-FMA flops; the encoder runs the dot products as bf16 tensor-core MMAs
        # over an exact three-piece split of the centroids, so this is the equivalent rate
        fl = 3.0 * w.B * w.L * w.H_kv * pq["pq_M"] * pq["pq_C"] * 9 * 2
        alu_peak = 152 * 128 * 2 * 2.07e9 / 1e12
        rows["pq_build (2 Lloyd iterations + encode, once per prefill)"]["alu"] = {
            "tflops": round(fl / (b_ms * 1e-3) / 1e12, 2), "peak_tflops": round(alu_peak, 1),
            "frac": round(fl / (b_ms * 1e-3) / 1e12 / alu_peak, 4),
            "peak_source": "152 SMs x 128 FP32 lanes x 2 flop x 2.07 GHz (nominal); FP32-FMA-equivalent flops of "
                           "the encodes, whose dot products run on the tensor cores"}
        pq["pq_over_verify"] = round(pq_ms / ver_ms, 4)
    if topk:
        tk_ms = topk.pop("_topk_ms")
        rows["topk_draft_attn (scores + select + attend, per draft step)"] = row(
            topk.pop("_topk_bytes"), tk_ms, "hbm (score pass, 0.93); latency (select)")
        topk["topk_over_verify"] = round(tk_ms / ver_ms, 4)
    result = {
        "metric": METRIC,
        "value": round(aggregate_rate(world, args.steps, ms_total), 4),
        "unit": "steps/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": args.workload, "B": w.B, "L": w.L, "H_q": w.H_q, "H_kv": w.H_kv, "d": w.d,
                   "gamma": w.gamma, "V": w.V, "layers": args.layers,
                   "draft": f"StreamingLLM {w.n_sink}+{w.n_recent} (selection + gather every step)",
                   "per_rank_batch": w.B, "parallelism": f"replicas x{world}",
                   "rank_seeds": "workload seed + 100 x rank (distinct sequences per rank)",
                   "l2": "inputs larger than L2 (KV cache 16.8 GB per layer vs 129 MB L2)",
                   "step": "layers x (select, gather, gamma x draft_attn, verify_attn) + spec_accept"},
        "roofline": {"bound": "hbm", "kernel": "verify_heads_kernel", "achieved": round(ver_gbs, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(ver_gbs / peak, 4),
                     "traffic": traffic, "algorithmic_bytes": vbytes, "peak_source": peak_kind},
        "rows_roofline": rows,
        "verify_gbs": round(ver_gbs, 1), "verify_pct_peak": round(100 * ver_gbs / peak, 2),
        "verify_ms_per_layer": round(ver_ms, 4),
        "draft_gbs": round(dra_gbs, 1), "draft_pct_peak": round(100 * dra_gbs / peak, 2),
        "draft_us_per_layer": round(dra_ms * 1e3, 2),
        "accept_us": round(acc_ms * 1e3, 2),
        "accept_gbs": round(pipe.accept_bytes() / (acc_ms * 1e-3) / 1e9, 1),
        "select_gather_us_per_layer": round(sel_ms * 1e3, 2),
        **snap,
        **topk,
        **pq,
        "omega_hat_synthetic": round(omega_hat, 4),
        "tokens_per_s_synthetic": round(world * w.B * omega_hat * args.steps / (ms_total * 1e-3), 1),
        "gpu_launches": pipe.launches_per_step * args.steps,
        "device_error_word": err_word,
        "e2e": {"value": round(aggregate_rate(world, args.steps, e2e_ms), 4), "unit": "steps/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "clocks": clocks.summary(),
    }
    result["ring_cache_step"] = ring_step
    if graph:
        result["cuda_graph"] = graph
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        del pipe.kc, pipe.vc
        result["cpu_baseline"] = cpu_baseline(w, args.layers, pipe)
    return result


# -------------------------------------------------------------- oracle on host
def oracle_step_sample(w: synth.Workload, layers: int, host, nb_attn: int, nb_acc: int):
    """Time the CPU oracle on a bounded sample of one step and scale it to the whole step.
    host: dict of numpy inputs for the first sequences.  Returns (seconds per full step, detail)."""
    import oracle
    k, v, qd, qv, sl = host["k"][:nb_attn], host["v"][:nb_attn], host["qd"][:nb_attn], host["qv"][:nb_attn], \
        host["sl"][:nb_attn]
    t0 = time.perf_counter()
    idx, n_sel = oracle.streaming_select(sl, w.H_kv, w.n_sink, w.n_recent)
    kc, vc = oracle.gather_kv(k, v, idx, w.stream_budget)
    t1 = time.perf_counter()
    oracle.draft_attn(qd, kc, vc, n_sel)
    t2 = time.perf_counter()
    oracle.verify_attn(qv, k, v, sl, w.n_q)
    t3 = time.perf_counter()
    oracle.spec_accept(host["target"][:nb_acc], host["draft"][:nb_acc], host["tok"][:nb_acc],
                       host["u_acc"][:nb_acc], host["u_res"][:nb_acc], False)
    t4 = time.perf_counter()
    f_attn, f_acc = w.B / nb_attn, w.B / nb_acc
    per_step = layers * ((t1 - t0) + w.gamma * (t2 - t1) + (t3 - t2)) * f_attn + (t4 - t3) * f_acc
    detail = {"select_gather_s": t1 - t0, "draft_s": t2 - t1, "verify_s": t3 - t2, "accept_s": t4 - t3}
    return per_step, detail, (t4 - t0)


def host_sample(w: synth.Workload, pipe, nb_attn: int, nb_acc: int):
    def u16(t):
        return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
    return {"k": u16(pipe.k[:nb_attn]), "v": u16(pipe.v[:nb_attn]), "qd": u16(pipe.q_draft[:nb_attn]),
            "qv": u16(pipe.q_verify[:nb_attn]), "sl": pipe.seq_len[:nb_attn].cpu().numpy(),
            "target": pipe.target[:nb_acc].cpu().numpy(), "draft": pipe.draft[:nb_acc].cpu().numpy(),
            "tok": pipe.tok[:nb_acc].cpu().numpy(), "u_acc": pipe.u_acc[:nb_acc].cpu().numpy(),
            "u_res": pipe.u_res[:nb_acc].cpu().numpy()}


def cpu_baseline(w: synth.Workload, layers: int, pipe, repeats: int = 4):
    import oracle
    nb_attn, nb_acc = min(32, w.B), min(32, w.B)
    host = host_sample(w, pipe, nb_attn, nb_acc)
    per, spent, detail = [], 0.0, None
    for _ in range(repeats):
        per_step, detail, s = oracle_step_sample(w, layers, host, nb_attn, nb_acc)
        per.append(per_step)
        spent += s
    per_step = statistics.median(per)
    return {"value": round(1.0 / per_step, 8), "unit": "steps/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"one step's calls on {nb_attn} of {w.B} sequences (attention, selection, gather; all "
                      f"{layers} layers from one layer's time) and {nb_acc} sequences (accept), scaled "
                      f"linearly to B={w.B}, median of {repeats}; {spent:.1f} s of CPU time",
            "detail_s": {k: round(v, 4) for k, v in detail.items()}}


def run_reference(args, rank: int):
    """The oracle as the reference arm: each step times a bounded sample on the host cores."""
    if rank != 0:
        return None
    import oracle
    w = synth.WORKLOADS[args.workload]
    nb_attn, nb_acc = min(8, w.B), min(16, w.B)
    # inputs for the sampled sequences, drawn on the host with the same recipes
    sw = synth.Workload("sample", B=nb_attn, H_q=w.H_q, H_kv=w.H_kv, d=w.d, L=w.L, gamma=w.gamma, V=w.V,
                        n_sink=w.n_sink, n_recent=w.n_recent, boost_frac=w.boost_frac, boost=w.boost,
                        target_sigma=w.target_sigma, draft_noise=w.draft_noise, seed=w.seed)
    k, v, _ = synth.kv_cache(sw, "cpu")
    qd = synth.queries(sw, 1, "cpu", seed=1)
    qv = synth.queries(sw, w.n_q, "cpu", seed=2)
    target, draft, tok, u_acc, u_res = synth.logits(w, "cpu", B=nb_acc)

    def u16(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)
    host = {"k": u16(k), "v": u16(v), "qd": u16(qd), "qv": u16(qv), "sl": np.full(nb_attn, w.L, np.int32),
            "target": target.numpy(), "draft": draft.numpy(), "tok": tok.numpy(), "u_acc": u_acc.numpy(),
            "u_res": u_res.numpy()}
    for _ in range(args.warmup):
        oracle_step_sample(w, args.layers, host, nb_attn, nb_acc)
    times, spent = [], 0.0
    for _ in range(args.steps):
        per_step, _, s = oracle_step_sample(w, args.layers, host, nb_attn, nb_acc)
        times.append(per_step)
        spent += s
    ms_step = 1e3 * statistics.mean(times)
    value = 1e3 / ms_step
    sample = (f"per step: one step's calls on {nb_attn} of {w.B} sequences (attention, selection, gather; "
              f"{args.layers} layers from one layer's time) and {nb_acc} sequences (accept), scaled linearly "
              f"to B={w.B}")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 8), "unit": "steps/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "B": w.B, "L": w.L, "H_q": w.H_q, "H_kv": w.H_kv, "d": w.d,
                       "gamma": w.gamma, "V": w.V, "layers": args.layers},
            "cpu_baseline": {"value": round(value, 8), "unit": "steps/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample + f"; {spent:.1f} s of CPU time in total"},
            "e2e": {"value": round(value, 8), "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--layers", type=int, default=LAYERS)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-topk", action="store_true", help="skip the Top-K attention draft row")
    ap.add_argument("--no-pq", action="store_true", help="skip the PQCache-style draft rows")
    ap.add_argument("--graph", action="store_true", help="also time the step captured in a CUDA graph")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch size (profiling runs on smaller cases)")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
