"""CPU oracle for the MagicDec self-speculative decoding hot path.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package.  The product
library (``long_context_self_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP over independent
(sequence, head) units); this module compiles it with gcc on first use and
marshals numpy arrays through ctypes.  Each function restates a definition from
"MagicDec: Breaking the Latency-Throughput Tradeoff for Long Context Generation
with Speculative Decoding" (arXiv 2408.11049v5); the citation for each sits on
the C function.

bf16 tensors are passed as their bit patterns (``numpy.uint16``), exactly as the
GPU consumes them.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_oracle.so (gcc, -O2, OpenMP, IEEE math)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oracle_num_threads.restype = I
            lib.oracle_set_num_threads.argtypes = [I]
            lib.oracle_verify_attn.argtypes = [I, I, I, I, I, I, P, P, P, P, P]
            lib.oracle_draft_attn.argtypes = [I, I, I, I, I, P, P, P, P, P]
            lib.oracle_streaming_select.argtypes = [P, I, I, I, I, P, P]
            lib.oracle_gather_kv.argtypes = [I, I, I, I, P, P, P, I, I, P, P]
            lib.oracle_snapkv_scores.argtypes = [I, I, I, I, I, I, P, P, P, P]
            lib.oracle_maxpool1d.argtypes = [P, I, I, P]
            lib.oracle_snapkv_select.argtypes = [I, I, I, I, I, P, P, P, I, I, I, P, P, P]
            lib.oracle_spec_accept.argtypes = [I, I, I, P, P, P, P, P, I, P, P, P, P, P]
            lib.oracle_resample_weights.argtypes = [P, P, I, P]
            lib.oracle_topk_attn.argtypes = [I, I, I, I, I, P, P, P, P, I, P, P, P]
            lib.oracle_draft_cache_update.argtypes = [I, I, I, I, P, P, P, P, P, P, P, I, I, P, P, P]
            lib.oracle_step_lengths.argtypes = [I, I, I, P, P, P, P]
            lib.oracle_pq_encode.argtypes = [I, I, I, I, P, I, I, P, P, P]
            lib.oracle_pq_update.argtypes = [I, I, I, I, P, P, I, I, P, P]
            lib.oracle_pq_attn.argtypes = [I, I, I, I, I, P, P, P, P, I, I, P, P, I, P, P, P]
            for name in ("oracle_verify_attn", "oracle_draft_attn", "oracle_streaming_select",
                         "oracle_gather_kv", "oracle_snapkv_scores", "oracle_maxpool1d",
                         "oracle_snapkv_select", "oracle_spec_accept", "oracle_resample_weights",
                         "oracle_topk_attn", "oracle_draft_cache_update", "oracle_step_lengths", "oracle_pq_encode",
                         "oracle_pq_update", "oracle_pq_attn"):
                getattr(lib, name).restype = I
            _lib = lib
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, name: str):
    if rc != 0:
        raise ValueError(f"{name}: invalid arguments (rc={rc})")


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def verify_attn(q, k, v, seq_len, n_q: int) -> np.ndarray:
    """q [B,n_q,H_q,d] u16, k/v [B,L_cap,H_kv,d] u16, seq_len [B] -> fp64 [B,n_q,H_q,d]."""
    q, k, v = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    seq_len = _c(seq_len, np.int32)
    B, nq, H_q, d = q.shape
    assert nq == n_q and k.shape[0] == B and k.shape == v.shape and k.shape[3] == d
    L_cap, H_kv = k.shape[1], k.shape[2]
    out = np.zeros((B, n_q, H_q, d), np.float64)
    _check(_load().oracle_verify_attn(B, H_q, H_kv, d, L_cap, n_q, _ptr(q), _ptr(k), _ptr(v),
                                      _ptr(seq_len), _ptr(out)), "verify_attn")
    return out


def draft_attn(q, kc, vc, draft_len) -> np.ndarray:
    """q [B,1,H_q,d] u16, kc/vc [B,H_kv,cap,d] u16, draft_len [B] -> fp64 [B,1,H_q,d]."""
    q, kc, vc = _c(q, np.uint16), _c(kc, np.uint16), _c(vc, np.uint16)
    draft_len = _c(draft_len, np.int32)
    B, one, H_q, d = q.shape
    assert one == 1 and kc.shape == vc.shape and kc.shape[0] == B and kc.shape[3] == d
    H_kv, cap = kc.shape[1], kc.shape[2]
    out = np.zeros((B, 1, H_q, d), np.float64)
    _check(_load().oracle_draft_attn(B, H_q, H_kv, d, cap, _ptr(q), _ptr(kc), _ptr(vc),
                                     _ptr(draft_len), _ptr(out)), "draft_attn")
    return out


def streaming_select(seq_len, H_kv: int, n_sink: int, n_recent: int):
    """-> (idx int32 [B,H_kv,n_sink+n_recent], n_sel int32 [B])."""
    seq_len = _c(seq_len, np.int32)
    B = seq_len.shape[0]
    idx = np.empty((B, H_kv, n_sink + n_recent), np.int32)
    n_sel = np.empty((B,), np.int32)
    _check(_load().oracle_streaming_select(_ptr(seq_len), B, H_kv, n_sink, n_recent,
                                           _ptr(idx), _ptr(n_sel)), "streaming_select")
    return idx, n_sel


def gather_kv(k, v, idx, cap: int, kc=None, vc=None):
    """k/v [B,L_cap,H_kv,d] u16, idx int32 [B,H_kv,n_idx] -> (kc, vc) u16 [B,H_kv,cap,d]."""
    k, v, idx = _c(k, np.uint16), _c(v, np.uint16), _c(idx, np.int32)
    B, L_cap, H_kv, d = k.shape
    n_idx = idx.shape[2]
    if kc is None:
        kc = np.zeros((B, H_kv, cap, d), np.uint16)
    if vc is None:
        vc = np.zeros((B, H_kv, cap, d), np.uint16)
    assert kc.flags.c_contiguous and vc.flags.c_contiguous
    _check(_load().oracle_gather_kv(B, H_kv, d, L_cap, _ptr(k), _ptr(v), _ptr(idx), n_idx, cap,
                                    _ptr(kc), _ptr(vc)), "gather_kv")
    return kc, vc


def snapkv_scores(q_win, k, seq_len) -> np.ndarray:
    """q_win [B,w,H_q,d] u16, k [B,L_cap,H_kv,d] u16 -> fp64 [B,H_kv,L_cap]."""
    q_win, k, seq_len = _c(q_win, np.uint16), _c(k, np.uint16), _c(seq_len, np.int32)
    B, w, H_q, d = q_win.shape
    L_cap, H_kv = k.shape[1], k.shape[2]
    score = np.zeros((B, H_kv, L_cap), np.float64)
    _check(_load().oracle_snapkv_scores(B, H_q, H_kv, d, L_cap, w, _ptr(q_win), _ptr(k),
                                        _ptr(seq_len), _ptr(score)), "snapkv_scores")
    return score


def maxpool1d(x, kernel: int) -> np.ndarray:
    x = _c(x, np.float64)
    out = np.empty_like(x)
    _check(_load().oracle_maxpool1d(_ptr(x), x.shape[0], kernel, _ptr(out)), "maxpool1d")
    return out


def snapkv_select(q_win, k, seq_len, pool_kernel: int, budget: int):
    """-> (idx int32 [B,H_kv,budget], n_sel int32 [B], pooled fp64 [B,H_kv,L_cap])."""
    q_win, k, seq_len = _c(q_win, np.uint16), _c(k, np.uint16), _c(seq_len, np.int32)
    B, w, H_q, d = q_win.shape
    L_cap, H_kv = k.shape[1], k.shape[2]
    idx = np.empty((B, H_kv, budget), np.int32)
    n_sel = np.empty((B,), np.int32)
    pooled = np.zeros((B, H_kv, L_cap), np.float64)
    _check(_load().oracle_snapkv_select(B, H_q, H_kv, d, L_cap, _ptr(q_win), _ptr(k), _ptr(seq_len),
                                        w, pool_kernel, budget, _ptr(idx), _ptr(n_sel), _ptr(pooled)),
           "snapkv_select")
    return idx, n_sel, pooled


def topk_attn(q, k, v, seq_len, top_k: int, want_scores: bool = False):
    """Top-K attention draft.  q [B,1,H_q,d] u16, k/v [B,L_cap,H_kv,d] u16, seq_len [B]
    -> (out fp64 [B,1,H_q,d], idx int32 [B,H_q,top_k] ascending, -1 padded,
        scores fp64 [B,H_q,L_cap] or None)."""
    q, k, v = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    seq_len = _c(seq_len, np.int32)
    B, one, H_q, d = q.shape
    assert one == 1 and k.shape == v.shape and k.shape[0] == B and k.shape[3] == d
    L_cap, H_kv = k.shape[1], k.shape[2]
    out = np.zeros((B, 1, H_q, d), np.float64)
    idx = np.empty((B, H_q, top_k), np.int32)
    scores = np.zeros((B, H_q, L_cap), np.float64) if want_scores else None
    _check(_load().oracle_topk_attn(B, H_q, H_kv, d, L_cap, _ptr(q), _ptr(k), _ptr(v), _ptr(seq_len),
                                    int(top_k), _ptr(out), _ptr(idx),
                                    _ptr(scores) if scores is not None else None), "topk_attn")
    return out, idx, scores


def draft_cache_update(k, v, kc, vc, len_valid, len_old, len_new, origin, base, ring: int):
    """Update the compact draft cache kc/vc [B,H_kv,cap,d] u16 IN PLACE from the full cache
    k/v [B,L_cap,H_kv,d] u16.  ring > 0: StreamingLLM ring layout (base unused); ring == 0:
    SnapKV linear layout.  -> (draft_len int32 [B], number of writes skipped past cap)."""
    k, v = _c(k, np.uint16), _c(v, np.uint16)
    assert kc.flags.c_contiguous and vc.flags.c_contiguous and kc.dtype == np.uint16 and vc.dtype == np.uint16
    B, L_cap, H_kv, d = k.shape
    cap = kc.shape[2]
    lv, lo, ln = (_c(a, np.int32) for a in (len_valid, len_old, len_new))
    org = _c(origin, np.int32)
    bs = _c(base, np.int32) if base is not None else None
    draft_len = np.empty((B,), np.int32)
    rc = _load().oracle_draft_cache_update(B, H_kv, d, L_cap, _ptr(k), _ptr(v), _ptr(lv), _ptr(lo), _ptr(ln),
                                           _ptr(org), _ptr(bs) if bs is not None else None, int(ring), int(cap),
                                           _ptr(kc), _ptr(vc), _ptr(draft_len))
    if rc < 0:
        raise ValueError("draft_cache_update: invalid arguments")
    return draft_len, int(rc)


def step_lengths(len_in, gamma: int, L_cap: int, n_acc=None):
    """-> (len_out int32 [B], table int32 [gamma+2, B]); see oracle_step_lengths."""
    len_in = _c(len_in, np.int32)
    B = len_in.shape[0]
    na = _c(n_acc, np.int32) if n_acc is not None else None
    len_out = np.empty((B,), np.int32)
    table = np.empty((gamma + 2, B), np.int32)
    _check(_load().oracle_step_lengths(B, int(gamma), int(L_cap), _ptr(len_in), _ptr(na) if na is not None else None,
                                       _ptr(len_out), _ptr(table)), "step_lengths")
    return len_out, table


def pq_encode(k, codebook, want_gap: bool = False):
    """k [B,L_cap,H_kv,d] u16, codebook [B,H_kv,M,C,d/M] fp32 -> (codes u8 [B,H_kv,L_cap,M], gap fp64 or None)."""
    k = _c(k, np.uint16)
    cb = _c(codebook, np.float32)
    B, L_cap, H_kv, d = k.shape
    M, C = cb.shape[2], cb.shape[3]
    codes = np.empty((B, H_kv, L_cap, M), np.uint8)
    gap = np.empty((B, H_kv, L_cap, M), np.float64) if want_gap else None
    _check(_load().oracle_pq_encode(B, H_kv, d, L_cap, _ptr(k), M, C, _ptr(cb), _ptr(codes),
                                    _ptr(gap) if gap is not None else None), "pq_encode")
    return codes, gap


def pq_update(k, seq_len, codes, codebook):
    """One Lloyd update: returns a new codebook (fp32) from codes u8 [B,H_kv,L_cap,M]."""
    k, seq_len, codes = _c(k, np.uint16), _c(seq_len, np.int32), _c(codes, np.uint8)
    cb = np.array(codebook, dtype=np.float32, copy=True, order="C")
    B, L_cap, H_kv, d = k.shape
    M, C = cb.shape[2], cb.shape[3]
    _check(_load().oracle_pq_update(B, H_kv, d, L_cap, _ptr(k), _ptr(seq_len), M, C, _ptr(codes), _ptr(cb)),
           "pq_update")
    return cb


def pq_attn(q, k, v, seq_len, codebook, codes, top_k: int, want_approx: bool = False):
    """-> (out fp64 [B,1,H_q,d], idx int32 [B,H_q,top_k], approx fp64 [B,H_q,L_cap] or None)."""
    q, k, v = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    seq_len, codes, cb = _c(seq_len, np.int32), _c(codes, np.uint8), _c(codebook, np.float32)
    B, one, H_q, d = q.shape
    L_cap, H_kv = k.shape[1], k.shape[2]
    M, C = cb.shape[2], cb.shape[3]
    out = np.zeros((B, 1, H_q, d), np.float64)
    idx = np.empty((B, H_q, top_k), np.int32)
    approx = np.zeros((B, H_q, L_cap), np.float64) if want_approx else None
    _check(_load().oracle_pq_attn(B, H_q, H_kv, d, L_cap, _ptr(q), _ptr(k), _ptr(v), _ptr(seq_len), M, C, _ptr(cb),
                                  _ptr(codes), int(top_k), _ptr(out), _ptr(idx),
                                  _ptr(approx) if approx is not None else None), "pq_attn")
    return out, idx, approx


def spec_accept(target, draft, draft_tok, u_acc, u_res, greedy: bool, want_margins: bool = False):
    """target [B,g+1,V] f32, draft [B,g,V] f32, draft_tok [B,g] i32, u_acc [B,g], u_res [B]
    -> (n_acc [B], out_tok [B,g+1], n_amb [B]) int32; with want_margins also
    (acc_margin fp64 [B,g+1], draw_margin fp64 [B]): each decision's distance from its
    boundary on the path taken (NaN where none was taken; see oracle_spec_accept)."""
    target = _c(target, np.float32)
    B, gp1, V = target.shape
    gamma = gp1 - 1
    draft = _c(draft, np.float32) if draft is not None else np.zeros((B, gamma, V), np.float32)
    draft_tok, u_acc, u_res = _c(draft_tok, np.int32), _c(u_acc, np.float32), _c(u_res, np.float32)
    assert draft.shape == (B, gamma, V) and draft_tok.shape == (B, gamma)
    n_acc = np.empty((B,), np.int32)
    out_tok = np.empty((B, gamma + 1), np.int32)
    n_amb = np.empty((B,), np.int32)
    acc_m = np.empty((B, gamma + 1), np.float64) if want_margins else None
    draw_m = np.empty((B,), np.float64) if want_margins else None
    _check(_load().oracle_spec_accept(B, gamma, V, _ptr(target), _ptr(draft), _ptr(draft_tok),
                                      _ptr(u_acc), _ptr(u_res), int(bool(greedy)), _ptr(n_acc),
                                      _ptr(out_tok), _ptr(n_amb), _ptr(acc_m) if want_margins else None,
                                      _ptr(draw_m) if want_margins else None), "spec_accept")
    if want_margins:
        return n_acc, out_tok, n_amb, acc_m, draw_m
    return n_acc, out_tok, n_amb


def resample_weights(target_row, draft_row=None) -> np.ndarray:
    """fp64 resample weights of one position: max(0, p - q) (p when that is all zero or there is
    no draft row), unnormalised -- the weights the accept step draws from."""
    t = _c(target_row, np.float32)
    V = t.shape[0]
    d = None if draft_row is None else _c(draft_row, np.float32)
    w = np.empty((V,), np.float64)
    _check(_load().oracle_resample_weights(_ptr(t), None if d is None else _ptr(d), V, _ptr(w)),
           "resample_weights")
    return w
