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
than the 129 MB L2, so no layer sees another's data in cache).  Inputs are
synthetic (seeded; see long_context_self_gb300.synth).

Beside the headline step the line carries:
  snapkv_step   the same workload drafted by SnapKV (budget 512): selection
                once after prefill (paper section A.1, Fig. 8), then 16 steps
                of the loop in long_context_self_gb300.pipeline, whose lengths
                diverge by each sequence's accepted count;
  per_config    the other long-context configurations on the same GPU: B=32
                StreamingLLM 16+496; B=64 SnapKV 2048 (select once, 16 steps);
                B=16, L=100000, 40 query heads, SnapKV 4096 (select once,
                16 steps);
  rows_roofline every kernel row's GB/s against the measured copy peak and
                against the 8 TB/s nominal HBM bandwidth (frac, frac_8tbs).

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
TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "verify_attn_llama8b_b128_l32k.json")
NOMINAL_HBM_GBS = 8000.0    # GB300 HBM3e nominal bandwidth (8 TB/s): the second denominator of every fraction
SPEC_LOOP_STEPS = 16        # draft+verify steps after one SnapKV selection (the SnapKV-drafted legs)


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


def recorded_traffic(workload: str, record: str = TRAFFIC_RECORD):
    """Per-launch DRAM bytes of the verification kernel from the committed ncu record
    (written by long_context_self_gb300.ncu_record), if it was taken for this workload on the
    current kernel source; else None."""
    from long_context_self_gb300.ncu_record import source_sha16
    try:
        with open(record) as f:
            rec = json.load(f)
        if rec["workload"] != workload or rec["source_sha16"] != source_sha16(os.path.join(ROOT, rec["source"])):
            return None
        return float(rec["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
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
        # room past L for the positions the SnapKV-drafted loop appends
        self.L_cap = w.L + SPEC_LOOP_STEPS * (w.gamma + 1)
        self.k, self.v, self.heavy_dirs = synth.kv_cache(w, device, L_cap=self.L_cap)
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
        shape = mb.kv_shape(w.B, w.H_q, w.H_kv, w.d, self.L_cap)
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


def fractions(gbs: float, peak: float) -> dict:
    """A bandwidth against both denominators: the measured copy peak and the 8 TB/s nominal."""
    return {"frac": round(gbs / peak, 4), "frac_8tbs": round(gbs / NOMINAL_HBM_GBS, 4)}


def config_dict(w: synth.Workload, layers: int, world: int) -> dict:
    """The `config` of both arms' JSON lines."""
    return {"workload": w.name, "B": w.B, "L": w.L, "H_q": w.H_q, "H_kv": w.H_kv, "d": w.d,
            "gamma": w.gamma, "V": w.V, "layers": layers,
            "draft": f"StreamingLLM {w.n_sink}+{w.n_recent} (selection + gather every step)",
            "per_rank_batch": w.B, "parallelism": f"replicas x{world}",
            "rank_seeds": "workload seed + 100 x rank (distinct sequences per rank)",
            "l2": f"inputs larger than L2 (KV cache {2 * w.B * w.L * w.H_kv * w.d * 2 / 1e9:.1f} GB per layer "
                  f"vs 129 MB L2)",
            "step": "layers x (select, gather, gamma x draft_attn, verify_attn) + spec_accept"}


def time_streaming_step(pipe: "Pipeline", steps: int, warmup: int, world: int, device):
    """The StreamingLLM step: warm-up, then `steps` steps between barriers; returns (max-over-ranks
    ms for all steps, mean verify ms from events around its launches, draft ms per call, accept
    ms, select+gather ms)."""
    mb, w = pipe.mb, pipe.w
    for _ in range(warmup):
        pipe.step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    pipe.verify_events = []
    stream = torch.cuda.current_stream(device)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(steps):
        pipe.step(record=True)
    t1.record(stream)
    torch.cuda.synchronize()
    ms_total = max_over_ranks(t0.elapsed_time(t1), device)
    ver_ms = statistics.mean(a.elapsed_time(b) for a, b in pipe.verify_events)
    # draft launches are timed back to back outside the step (events between the
    # step's kernels would serialise their programmatic-dependent launches): one
    # step's gamma x layers calls replayed from a CUDA graph, so that the
    # binding's host-side checks cannot set the pace of these ~50 us calls
    n_dra = w.gamma * pipe.layers
    dra_ms = time_graph(lambda: [mb.magicdec_draft_attn(pipe.q_draft, pipe.kc, pipe.vc, pipe.n_sel,
                                                        out=pipe.out_d, ws=pipe.ws_attn) for _ in range(n_dra)],
                        3) / n_dra
    acc_ms = time_component(lambda: mb.magicdec_spec_accept(pipe.target, pipe.draft, pipe.tok, pipe.u_acc,
                                                            pipe.u_res, False, n_acc=pipe.n_acc,
                                                            out_tok=pipe.out_tok, n_amb=pipe.n_amb,
                                                            ws=pipe.ws_acc), 5)
    # selection + gather: one step's layers x (select, gather) replayed from a CUDA graph,
    # for the same reason as the draft (two short calls per layer)
    sel_ms = time_graph(lambda: [(mb.magicdec_streaming_select(pipe.seq_len, w.H_kv, w.n_sink, w.n_recent,
                                                               idx=pipe.idx, n_sel=pipe.n_sel),
                                  mb.magicdec_gather_kv(pipe.k, pipe.v, pipe.idx, pipe.cap, kc=pipe.kc,
                                                        vc=pipe.vc)) for _ in range(pipe.layers)],
                        3) / pipe.layers
    return ms_total, ver_ms, dra_ms, acc_ms, sel_ms


def snapkv_loop_leg(w: synth.Workload, k: torch.Tensor, v: torch.Tensor, layers: int, device, peak: float,
                    heavy_dirs=None, world: int = 1) -> dict:
    """Self-speculation with a static SnapKV draft: selection once after prefill, then
    SPEC_LOOP_STEPS steps of (per layer: gamma x (append + draft attention), verification;
    acceptance; the length bookkeeping; per layer the post-verification refresh), lengths
    diverging by each sequence's accepted count.  One warm-up pass of the whole protocol, then a
    timed one; the step rate is over the timed steps, the selection is reported beside it."""
    from long_context_self_gb300 import binding as mb
    from long_context_self_gb300.pipeline import SnapKVSpecLoop
    prefill = torch.full((w.B,), w.L, dtype=torch.int32, device=device)
    loop = SnapKVSpecLoop(k, v, prefill, w.H_q, w.gamma, w.snap_window, w.snap_pool, w.snap_budget, w.V,
                          SPEC_LOOP_STEPS, layers)
    q_win = synth.window_queries(w, device, heavy_dirs=heavy_dirs)
    qd = [synth.queries(w, 1, device, seed=w.seed * 7 + 10 + g) for g in range(w.gamma)]
    qv = synth.queries(w, w.n_q, device, seed=w.seed * 7 + 2)
    target, draft, tok, u_acc, u_res = synth.logits(w, device)

    def steps():
        for _ in range(SPEC_LOOP_STEPS):
            loop.step(qd, qv, target, draft, tok, u_acc, u_res)
    loop.prefill(q_win)
    steps()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    e0.record()
    loop.prefill(q_win)
    e1.record()
    steps()
    e2.record()
    torch.cuda.synchronize()
    sel_ms = e0.elapsed_time(e1)
    steps_ms = max_over_ranks(e1.elapsed_time(e2), device)
    # per-call component times at the loop's final state
    vlen = loop.table[w.gamma + 1]
    ver_ms = time_component(lambda: mb.magicdec_verify_attn(qv, k, v, vlen, out=loop.out_v, ws=loop.ws_attn), 5)
    n_dra = w.gamma * layers
    dra_ms = time_graph(lambda: [mb.magicdec_draft_attn(qd[0], loop.kc, loop.vc, loop.draft_len, out=loop.out_d[0],
                                                        ws=loop.ws_attn) for _ in range(n_dra)], 3) / n_dra
    acc_ms = time_component(lambda: mb.magicdec_spec_accept(target, draft, tok, u_acc, u_res, False,
                                                            n_acc=loop.n_acc, out_tok=loop.out_tok,
                                                            n_amb=loop.n_amb, ws=loop.ws_acc), 5)
    row_b = w.H_kv * w.d * 2 * 2                                   # K and V bytes of one position, all KV heads
    q_b = 2.0 * w.B * w.H_q * w.d * 2
    ver_bytes = float(vlen.sum().item()) * row_b + 2.0 * w.B * w.n_q * w.H_q * w.d * 2
    dra_bytes = float(loop.draft_len.sum().item()) * row_b + q_b
    grown = (loop.len - w.L).cpu()
    ver_gbs = ver_bytes / (ver_ms * 1e-3) / 1e9
    dra_gbs = dra_bytes / (dra_ms * 1e-3) / 1e9
    res = {"workload": w.name, "B": w.B, "L": w.L, "H_q": w.H_q, "H_kv": w.H_kv, "d": w.d, "gamma": w.gamma,
           "V": w.V, "layers": layers,
           "draft": f"SnapKV budget {w.snap_budget} (window {w.snap_window}, max-pool {w.snap_pool}), selected once",
           "steps": SPEC_LOOP_STEPS,
           "spec_steps_per_s": round(world * SPEC_LOOP_STEPS / (steps_ms * 1e-3), 4),
           "ms_per_step": round(steps_ms / SPEC_LOOP_STEPS, 4),
           "snapkv_select_gather_ms_per_layer": round(sel_ms, 4),
           "verify_us_per_layer": round(ver_ms * 1e3, 2), "verify_gbs": round(ver_gbs, 1),
           **{"verify_" + k2: v2 for k2, v2 in fractions(ver_gbs, peak).items()},
           "draft_us_per_layer": round(dra_ms * 1e3, 2), "draft_gbs": round(dra_gbs, 1),
           **{"draft_" + k2: v2 for k2, v2 in fractions(dra_gbs, peak).items()},
           "accept_us": round(acc_ms * 1e3, 2),
           "tokens_grown_per_sequence": {"min": int(grown.min()), "max": int(grown.max()),
                                         "mean": round(float(grown.float().mean()), 2)},
           "gpu_launches_per_step": loop.launches_per_step,
           "device_error_word": mb.magicdec_device_error()}
    del loop
    torch.cuda.empty_cache()
    return res


def streaming_config_leg(w: synth.Workload, layers: int, steps: int, warmup: int, device, peak: float,
                         world: int = 1) -> dict:
    pipe = Pipeline(w, device, layers)
    torch.cuda.synchronize()
    ms_total, ver_ms, dra_ms, acc_ms, sel_ms = time_streaming_step(pipe, steps, warmup, world, device)
    ver_gbs = pipe.verify_bytes() / (ver_ms * 1e-3) / 1e9
    dra_gbs = pipe.draft_bytes() / (dra_ms * 1e-3) / 1e9
    res = {"workload": w.name, "B": w.B, "L": w.L, "H_q": w.H_q, "H_kv": w.H_kv, "d": w.d, "gamma": w.gamma,
           "V": w.V, "layers": layers, "draft": f"StreamingLLM {w.n_sink}+{w.n_recent} (selection + gather every step)",
           "steps": steps, "spec_steps_per_s": round(aggregate_rate(world, steps, ms_total), 4),
           "ms_per_step": round(ms_total / steps, 4),
           "verify_us_per_layer": round(ver_ms * 1e3, 2), "verify_gbs": round(ver_gbs, 1),
           **{"verify_" + k2: v2 for k2, v2 in fractions(ver_gbs, peak).items()},
           "draft_us_per_layer": round(dra_ms * 1e3, 2), "draft_gbs": round(dra_gbs, 1),
           **{"draft_" + k2: v2 for k2, v2 in fractions(dra_gbs, peak).items()},
           "accept_us": round(acc_ms * 1e3, 2), "select_gather_us_per_layer": round(sel_ms * 1e3, 2),
           "gpu_launches_per_step": pipe.launches_per_step}
    del pipe
    torch.cuda.empty_cache()
    return res


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
        ws_snap = torch.zeros(mb.magicdec_snapkv_workspace_size(mb.kv_shape(w.B, w.H_q, w.H_kv, w.d, pipe.L_cap),
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

    with ClockSampler(local_rank) as clocks:
        ms_total, ver_ms, dra_ms, acc_ms, sel_ms = time_streaming_step(pipe, args.steps, args.warmup, world, device)
    ms_step = ms_total / args.steps
    peak, peak_kind = load_peaks()
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
        codes = torch.empty((w.B, w.H_kv, pipe.L_cap, M), dtype=torch.uint8, device=device)

        def pq_build():
            cb.copy_(init)
            for _ in range(iters):
                mb.magicdec_pq_encode(pipe.k, cb, codes=codes)
                mb.magicdec_pq_update(pipe.k, pipe.seq_len, codes, cb)
            mb.magicdec_pq_encode(pipe.k, cb, codes=codes)
        build_ms = time_component(pq_build, 1)
        pq_idx = torch.empty((w.B, w.H_q, pipe.cap), dtype=torch.int32, device=device)
        pq_out = torch.empty_like(pipe.q_draft)
        pq_ws = torch.empty(mb.magicdec_pq_attn_workspace_size(mb.kv_shape(w.B, w.H_q, w.H_kv, w.d, pipe.L_cap)),
                            dtype=torch.uint8, device=device)
        pq_ms = time_component(lambda: mb.magicdec_pq_draft_attn(pipe.q_draft, pipe.k, pipe.v, pipe.seq_len, cb, codes,
                                                                 pipe.cap, out=pq_out, idx=pq_idx, ws=pq_ws), 5)
        kv_bytes = float(w.B) * pipe.L_cap * w.H_kv * w.d * 2     # the encodes and updates cover every cache row
        pq = {"pq_draft_us_per_layer": round(pq_ms * 1e3, 2), "pq_build_ms_per_layer": round(build_ms, 3),
              "pq_M": M, "pq_C": C, "pq_lloyd_iterations": iters,
              "_pq_bytes": (float(w.B) * w.H_kv * w.L * M + float(w.B) * w.H_kv * M * C * 8 * 4
                            + 2.0 * w.B * w.H_q * pipe.cap * w.d * 2 + 2.0 * w.B * w.H_q * w.d * 2),
              "_pq_ms": pq_ms,
              # each encode and each update reads K once; codes written per encode
              "_pq_build_bytes": (2 * iters + 1) * kv_bytes + (iters + 1) * float(w.B) * w.H_kv * pipe.L_cap * M,
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
        tk_ws = torch.empty(mb.magicdec_topk_attn_workspace_size(mb.kv_shape(w.B, w.H_q, w.H_kv, w.d, pipe.L_cap)),
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

    # the same workload drafted by SnapKV (budget as the StreamingLLM draft's): selection
    # once after prefill, then the multi-step loop with diverging lengths
    snapkv_step = None
    if w.snap_budget and not args.no_snapkv_step:
        snapkv_step = snapkv_loop_leg(w, pipe.k, pipe.v, args.layers, device, peak, world=world)

    vbytes, dbytes = pipe.verify_bytes(), pipe.draft_bytes()
    ver_gbs = vbytes / (ver_ms * 1e-3) / 1e9
    dra_gbs = dbytes / (dra_ms * 1e-3) / 1e9
    traffic = recorded_traffic(args.workload)

    def row(nbytes, ms, bound="hbm"):
        gbs = nbytes / (ms * 1e-3) / 1e9
        return {"gbs": round(gbs, 1), **fractions(gbs, peak), "us": round(ms * 1e3, 2),
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
        "config": config_dict(w, args.layers, world),
        "roofline": {"bound": "hbm", "kernel": "verify_heads_kernel", "achieved": round(ver_gbs, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(ver_gbs / peak, 4),
                     "traffic": traffic, "algorithmic_bytes": vbytes, "peak_source": peak_kind,
                     "peak_8tbs": NOMINAL_HBM_GBS, "frac_8tbs": round(ver_gbs / NOMINAL_HBM_GBS, 4)},
        "rows_roofline": rows,
        "verify_gbs": round(ver_gbs, 1), "verify_pct_peak": round(100 * ver_gbs / peak, 2),
        "verify_pct_8tbs": round(100 * ver_gbs / NOMINAL_HBM_GBS, 2),
        "verify_ms_per_layer": round(ver_ms, 4),
        "draft_gbs": round(dra_gbs, 1), "draft_pct_peak": round(100 * dra_gbs / peak, 2),
        "draft_pct_8tbs": round(100 * dra_gbs / NOMINAL_HBM_GBS, 2),
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
    if snapkv_step:
        result["snapkv_step"] = snapkv_step
    if graph:
        result["cuda_graph"] = graph
    del pipe.kc, pipe.vc, pipe.rkc, pipe.rvc
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, args.layers, pipe)
    if not args.no_configs:
        # the other long-context configurations, one after another on the same GPU
        pipe.k = pipe.v = None
        torch.cuda.empty_cache()
        cfgs = {"llama8b_b32_l32k": streaming_config_leg(rank_workload(synth.WORKLOADS["llama8b_b32_l32k"], rank),
                                                         args.layers, args.steps, args.warmup, device, peak, world)}
        for name in ("llama8b_b64_l32k_snapkv", "qwen32b_b16_l100k"):
            wc = rank_workload(synth.WORKLOADS[name], rank)
            kk, vv, dirs = synth.kv_cache(wc, device, L_cap=wc.L + SPEC_LOOP_STEPS * (wc.gamma + 1))
            cfgs[name] = snapkv_loop_leg(wc, kk, vv, args.layers, device, peak, heavy_dirs=dirs, world=world)
            del kk, vv, dirs
            torch.cuda.empty_cache()
        cfgs["qwen32b_b16_l100k"]["note"] = ("the pages give no layer count for this shape: the per-layer "
                                             "figures are the measurement, the step rate assumes 32 layers")
        result["per_config"] = cfgs
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
    full, spent = [], []
    for _ in range(args.steps):
        per_step, _, s = oracle_step_sample(w, args.layers, host, nb_attn, nb_acc)
        full.append(per_step)
        spent.append(s)
    # what was run and timed: args.steps samples; the rate is their scaling to one full step
    ms_sample = 1e3 * statistics.mean(spent)
    ms_full = 1e3 * statistics.mean(full)
    value = 1e3 / ms_full
    sample = (f"per step: one step's calls on {nb_attn} of {w.B} sequences (attention, selection, gather; "
              f"{args.layers} layers from one layer's time) and {nb_acc} sequences (accept), scaled linearly "
              f"to B={w.B}")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 8), "unit": "steps/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_sample, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(w, args.layers, args.gpus),
            "extrapolated": {"sample": sample, "ms_per_sample": round(ms_sample, 4),
                             "ms_per_full_step": round(ms_full, 4), "scale": round(ms_full / ms_sample, 3),
                             "note": "steps and ms_per_step count the samples actually run; value is "
                                     "1000 / ms_per_full_step"},
            "cpu_baseline": {"value": round(value, 8), "unit": "steps/s", "cores": oracle.num_threads(),
                             "kind": "oracle",
                             "sample": sample + f"; {sum(spent):.1f} s of CPU time in total"},
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
    ap.add_argument("--no-snapkv-step", action="store_true", help="skip the SnapKV-drafted multi-step leg")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration legs (B=32 StreamingLLM, B=64 SnapKV, B=16 L=100000)")
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
