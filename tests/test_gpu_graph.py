"""A whole speculative step (selection, gather, draft and verification attention for
several layers, acceptance) captured in a CUDA graph replays to exactly the outputs of
eager execution: the C ABI allocates nothing and never synchronises inside a call, and
every kernel is deterministic."""
import pytest
import torch

from long_context_self_gb300 import binding as mb
from long_context_self_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def test_graph_replay_equals_eager_step():
    from long_context_self_gb300 import build
    build.build()
    w = synth.Workload("g", B=8, H_q=32, H_kv=8, d=128, L=3000, gamma=3, V=5000, n_sink=16, n_recent=496,
                       snap_window=32, snap_pool=7, snap_budget=512, boost_frac=0.01, boost=4.0, seed=6)
    k, v, _ = synth.kv_cache(w, DEV)
    sl = torch.tensor([3000, 2999, 1200, 64, 600, 2048, 1, 2500], dtype=torch.int32, device=DEV)
    qd = synth.queries(w, 1, DEV, seed=1)
    qv = synth.queries(w, w.n_q, DEV, seed=2)
    q_win = synth.window_queries(w, DEV)
    target, draft, tok, u_acc, u_res = synth.logits(w, DEV)
    shape = mb.kv_shape(w.B, w.H_q, w.H_kv, w.d, w.L)
    ws_attn = torch.zeros(mb.magicdec_attn_workspace_size(shape, w.n_q), dtype=torch.uint8, device=DEV)
    ws_snap = torch.zeros(mb.magicdec_snapkv_workspace_size(shape, w.snap_window), dtype=torch.uint8, device=DEV)
    ws_acc = torch.zeros(mb.magicdec_spec_accept_workspace_size(w.B, w.gamma, w.V), dtype=torch.uint8, device=DEV)
    idx = torch.empty((w.B, w.H_kv, w.stream_budget), dtype=torch.int32, device=DEV)
    n_sel = torch.empty((w.B,), dtype=torch.int32, device=DEV)
    sidx = torch.empty((w.B, w.H_kv, w.snap_budget), dtype=torch.int32, device=DEV)
    sn = torch.empty((w.B,), dtype=torch.int32, device=DEV)
    kc = torch.zeros((w.B, w.H_kv, w.stream_budget, w.d), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    out_d = torch.empty((3, w.B, 1, w.H_q, w.d), dtype=torch.bfloat16, device=DEV)
    out_v = torch.empty((3,) + tuple(qv.shape), dtype=torch.bfloat16, device=DEV)
    n_acc = torch.empty((w.B,), dtype=torch.int32, device=DEV)
    out_tok = torch.empty((w.B, w.n_q), dtype=torch.int32, device=DEV)
    n_amb = torch.empty((w.B,), dtype=torch.int32, device=DEV)

    def step():
        mb.magicdec_snapkv_select(q_win, k, sl, w.snap_window, w.snap_pool, w.snap_budget, idx=sidx, n_sel=sn,
                                  ws=ws_snap)
        for layer in range(3):
            mb.magicdec_streaming_select(sl, w.H_kv, w.n_sink, w.n_recent, idx=idx, n_sel=n_sel)
            mb.magicdec_gather_kv(k, v, idx, w.stream_budget, kc=kc, vc=vc)
            mb.magicdec_draft_attn(qd, kc, vc, n_sel, out=out_d[layer], ws=ws_attn)
            mb.magicdec_verify_attn(qv, k, v, sl, out=out_v[layer], ws=ws_attn)
        mb.magicdec_spec_accept(target, draft, tok, u_acc, u_res, False, n_acc=n_acc, out_tok=out_tok, n_amb=n_amb,
                                ws=ws_acc)

    step()
    torch.cuda.synchronize()
    ref = [t.clone() for t in (sidx, sn, idx, n_sel, kc, vc, out_d, out_v, n_acc, out_tok, n_amb)]
    for t in (sidx, sn, idx, n_sel, kc, vc, out_d, out_v, n_acc, out_tok, n_amb):
        t.fill_(-7) if t.dtype == torch.int32 else t.fill_(0)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(2):
        for t in (sidx, sn, idx, n_sel, out_d, out_v, n_acc, out_tok):
            t.fill_(-7) if t.dtype == torch.int32 else t.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        got = (sidx, sn, idx, n_sel, kc, vc, out_d, out_v, n_acc, out_tok, n_amb)
        for a, b in zip(got, ref):
            assert torch.equal(a, b)
    assert mb.magicdec_device_error() == 0
