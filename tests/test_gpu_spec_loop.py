"""The select-once / many-steps loop of self-speculation with a static SnapKV draft
(MagicDec section A.1 Fig. 8: the compressed KV is built at prefill; section 3.1: gamma
drafts, one verification, acceptance; section 4.4: the static draft takes in new tokens),
run through the library by long_context_self_gb300.pipeline and checked against an
oracle chain of the same steps.

Lengths diverge between sequences by each one's accepted count.  The draft appends the
K/V rows of its drafted positions from a different source (the full cache with K and V
swapped) than the verified rows the refresh after verification copies, so a refresh that
fails to replace them changes the compact cache bytes.  The oracle chain takes the
kernel's SnapKV selection (checked against the oracle's own under the band rule) and the
kernel's accepted counts (each checked against the oracle's acceptance under the margin
rule, with exclusions decided by the oracle alone), so both chains hold the same state."""
import numpy as np
import pytest
import torch

import oracle
from long_context_self_gb300 import binding as mb
from long_context_self_gb300 import synth
from long_context_self_gb300.pipeline import SnapKVSpecLoop
from parity_util import bf16_out_to_f64, check_accept, check_attention, check_topk, oracle_accept, to_u16

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from long_context_self_gb300 import build
    build.build()
    mb.lib()
    yield
    assert mb.magicdec_device_error() == 0


class OracleChain:
    """The same loop on the CPU oracle for a subset of sequences (numpy, bf16 as uint16)."""

    def __init__(self, k, v, kd, vd, idx, n_sel, prefill, gamma, L_cap, cap, n_q):
        self.k, self.v, self.kd, self.vd = k, v, kd, vd
        self.gamma, self.L_cap, self.n_q = gamma, L_cap, n_q
        self.kc, self.vc = oracle.gather_kv(k, v, idx, cap)
        self.base = n_sel.astype(np.int32)
        self.origin = prefill.astype(np.int32)
        self.draft_len = self.base.copy()
        self.len, self.table = oracle.step_lengths(prefill, gamma, L_cap)

    def draft_and_verify(self, q_draft, q_verify):
        t, outs = self.table, []
        for g in range(self.gamma):
            self.draft_len, skipped = oracle.draft_cache_update(self.kd, self.vd, self.kc, self.vc, t[g], t[g],
                                                                t[g + 1], self.origin, self.base, 0)
            assert skipped == 0
            outs.append(oracle.draft_attn(q_draft[g], self.kc, self.vc, self.draft_len))
        return outs, oracle.verify_attn(q_verify, self.k, self.v, t[self.gamma + 1], self.n_q)

    def advance(self, n_acc):
        t = self.table
        len_next, table_next = oracle.step_lengths(self.len, self.gamma, self.L_cap, n_acc)
        self.draft_len, skipped = oracle.draft_cache_update(self.k, self.v, self.kc, self.vc, t[0], t[self.gamma],
                                                            len_next, self.origin, self.base, 0)
        assert skipped == 0
        self.len, self.table = len_next, table_next


def step_inputs(w, B, step, device):
    qd = [synth.queries(w, 1, device, seed=1000 * step + g) for g in range(w.gamma)]
    qv = synth.queries(w, w.n_q, device, seed=1000 * step + 999)
    return qd, qv, synth.logits(w, device, B=B, seed=w.seed * 100 + step)


def test_snapkv_loop_tiny_every_sequence_every_step():
    w = synth.WORKLOADS["tiny"]
    steps = 16
    L_cap = w.L + steps * (w.gamma + 1)
    k, v, _ = synth.kv_cache(w, "cpu", L_cap=L_cap)
    prefill = np.array([w.L, w.L - 37], np.int32)
    q_win = synth.window_queries(w, "cpu")
    kd, vd = v.to(DEV), k.to(DEV)          # drafted rows differ from the verified ones
    loop = SnapKVSpecLoop(k.to(DEV), v.to(DEV), torch.from_numpy(prefill).to(DEV), w.H_q, w.gamma, w.snap_window,
                          w.snap_pool, w.snap_budget, w.V, steps, k_draft=kd, v_draft=vd)
    loop.prefill(q_win.to(DEV))
    torch.cuda.synchronize()
    ku, vu = to_u16(k), to_u16(v)
    idx_o, n_sel_o, pooled = oracle.snapkv_select(to_u16(q_win), ku, prefill, w.snap_pool, w.snap_budget)
    idx_g, base_g = loop.idx.cpu().numpy(), loop.base.cpu().numpy()
    check_topk(idx_g, base_g, idx_o, n_sel_o, pooled, prefill, w.snap_window, w.snap_budget)
    chain = OracleChain(ku, vu, vu, ku, idx_g, base_g, prefill, w.gamma, L_cap, loop.cap, w.n_q)
    assert np.array_equal(to_u16(loop.kc), chain.kc) and np.array_equal(to_u16(loop.vc), chain.vc)
    excluded = 0
    for s in range(steps):
        qd, qv, (target, draft, tok, u_acc, u_res) = step_inputs(w, w.B, s, "cpu")
        loop.step([q.to(DEV) for q in qd], qv.to(DEV), target.to(DEV), draft.to(DEV), tok.to(DEV), u_acc.to(DEV),
                  u_res.to(DEV))
        torch.cuda.synchronize()
        outs_o, ver_o = chain.draft_and_verify([to_u16(q) for q in qd], to_u16(qv))
        for g in range(w.gamma):
            check_attention(bf16_out_to_f64(loop.out_d[g]), outs_o[g], f"step {s} draft {g}")
        check_attention(bf16_out_to_f64(loop.out_v), ver_o, f"step {s} verify")
        t, d, x, ua, ur = (a.numpy() for a in (target, draft, tok, u_acc, u_res))
        got = (loop.n_acc.cpu().numpy(), loop.out_tok.cpu().numpy(), loop.n_amb.cpu().numpy())
        excluded += check_accept(got, oracle_accept(t, d, x, ua, ur, False), f"step {s}", inputs=(t, d, ur),
                                 report=False)
        chain.advance(got[0])
        assert np.array_equal(loop.len.cpu().numpy(), chain.len), f"step {s}: lengths"
        assert np.array_equal(loop.table.cpu().numpy(), chain.table), f"step {s}: length table"
        assert np.array_equal(loop.draft_len.cpu().numpy(), chain.draft_len), f"step {s}: draft lengths"
        assert np.array_equal(to_u16(loop.kc), chain.kc), f"step {s}: compact K"
        assert np.array_equal(to_u16(loop.vc), chain.vc), f"step {s}: compact V"
    grown = chain.len - prefill
    assert grown.min() >= steps and grown.max() <= steps * (w.gamma + 1)
    assert len(set(grown.tolist())) > 1 or w.B == 1, "lengths never diverged"
    assert excluded <= 2


def test_snapkv_loop_full_size_sampled():
    """B=64, L=32000, H_q=32 over 8 KV heads, d=128, gamma=4, SnapKV w=32, pool 7, budget 2048,
    vocabulary 128256: selection once, then 16 steps; three sampled sequences are followed by
    the oracle chain and compared after steps 1, 8 and 16 (attention outputs, lengths, draft
    cache bytes), acceptance over every sequence at those steps."""
    w = synth.WORKLOADS["llama8b_b64_l32k_snapkv"]
    steps = w.steps
    L_cap = w.L + steps * (w.gamma + 1)
    k, v, dirs = synth.kv_cache(w, DEV, L_cap=L_cap)
    q_win = synth.window_queries(w, DEV, heavy_dirs=dirs)
    prefill = torch.full((w.B,), w.L, dtype=torch.int32, device=DEV)
    loop = SnapKVSpecLoop(k, v, prefill, w.H_q, w.gamma, w.snap_window, w.snap_pool, w.snap_budget, w.V, steps,
                          k_draft=v, v_draft=k)
    loop.prefill(q_win)
    torch.cuda.synchronize()
    sample = [0, 29, 63]
    idx_g, base_g = loop.idx.cpu().numpy(), loop.base.cpu().numpy()
    chains = {}
    for b in sample:
        kb, vb = to_u16(k[b:b + 1]), to_u16(v[b:b + 1])
        pf = np.array([w.L], np.int32)
        idx_o, n_sel_o, pooled = oracle.snapkv_select(to_u16(q_win[b:b + 1]), kb, pf, w.snap_pool, w.snap_budget)
        check_topk(idx_g[b:b + 1], base_g[b:b + 1], idx_o, n_sel_o, pooled, pf, w.snap_window, w.snap_budget)
        chains[b] = OracleChain(kb, vb, vb, kb, idx_g[b:b + 1], base_g[b:b + 1], pf, w.gamma, L_cap, loop.cap,
                                w.n_q)
    checks = {0, 7, 15}
    for s in range(steps):
        qd, qv, (target, draft, tok, u_acc, u_res) = step_inputs(w, w.B, s, DEV)
        loop.step(qd, qv, target, draft, tok, u_acc, u_res)
        torch.cuda.synchronize()
        n_acc = loop.n_acc.cpu().numpy()
        if s in checks:
            t, d, x, ua, ur = (a.cpu().numpy() for a in (target, draft, tok, u_acc, u_res))
            got = (n_acc, loop.out_tok.cpu().numpy(), loop.n_amb.cpu().numpy())
            n_ex = check_accept(got, oracle_accept(t, d, x, ua, ur, False), f"full-size step {s}", inputs=(t, d, ur))
            assert n_ex <= max(2, w.B // 8)
        lens = loop.len.cpu().numpy()
        for b, ch in chains.items():
            if s in checks:
                outs_o, ver_o = ch.draft_and_verify([to_u16(q[b:b + 1]) for q in qd], to_u16(qv[b:b + 1]))
                for g in range(w.gamma):
                    check_attention(bf16_out_to_f64(loop.out_d[g][b:b + 1]), outs_o[g], f"step {s} seq {b} draft {g}")
                check_attention(bf16_out_to_f64(loop.out_v[b:b + 1]), ver_o, f"step {s} seq {b} verify")
            else:
                # keep the chain's cache in step without the attention (same appends)
                t = ch.table
                for g in range(w.gamma):
                    ch.draft_len, _ = oracle.draft_cache_update(ch.kd, ch.vd, ch.kc, ch.vc, t[g], t[g], t[g + 1],
                                                                ch.origin, ch.base, 0)
            ch.advance(n_acc[b:b + 1])
            assert ch.len[0] == lens[b], f"step {s} seq {b}: length"
            if s in checks:
                dl = int(ch.draft_len[0])
                assert int(loop.draft_len[b]) == dl
                assert np.array_equal(to_u16(loop.kc[b:b + 1, :, :dl]), ch.kc[:, :, :dl]), f"step {s} seq {b}: K"
                assert np.array_equal(to_u16(loop.vc[b:b + 1, :, :dl]), ch.vc[:, :, :dl]), f"step {s} seq {b}: V"
    grown = loop.len.cpu().numpy() - w.L
    assert grown.min() >= steps and grown.max() <= steps * (w.gamma + 1) and len(set(grown.tolist())) > 1
    del loop, k, v
    torch.cuda.empty_cache()
