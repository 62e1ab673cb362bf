"""Thin Python binding of libmagicdec (ctypes).

Every function here carries the name of the C entry point it calls
(include/magicdec.h) and only marshals arguments: it checks dtypes, devices,
contiguity and shapes of torch tensors, allocates outputs (and a zero-filled workspace)
when the caller passes none, and hands raw device pointers and the current
CUDA stream to the library.  All compute happens in the library's kernels.
There is no fallback: if libmagicdec.so is missing or cannot load, every call
raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

# MAGICDEC_LIBRARY=debug loads the build whose kernels also record out-of-range
# lengths and indices in the device error word (long_context_self_gb300.build --debug).
_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                         "libmagicdec_debug.so" if os.environ.get("MAGICDEC_LIBRARY") == "debug" else "libmagicdec.so")
_lib = None
_lock = threading.Lock()


class MagicdecError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")


class KVShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H_q", ctypes.c_int), ("H_kv", ctypes.c_int), ("d", ctypes.c_int),
                ("L_cap", ctypes.c_int)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_S = ctypes.c_size_t

_SIGNATURES = {
    "magicdec_status_string": ([_I], ctypes.c_char_p),
    "magicdec_device_error": ([_P], _I),
    "magicdec_streaming_select": ([_P, _I, _I, _I, _I, _P, _P, _P], _I),
    "magicdec_snapkv_workspace_size": ([KVShape, _I], _S),
    "magicdec_snapkv_select": ([KVShape, _P, _P, _P, _I, _I, _I, _P, _P, _P, _S, _P], _I),
    "magicdec_snapkv_select_budgets": ([KVShape, _P, _P, _P, _I, _I, _P, _I, _P, _P, _P, _S, _P], _I),
    "magicdec_gather_kv": ([KVShape, _P, _P, _P, _I, _I, _P, _P, _P], _I),
    "magicdec_attn_workspace_size": ([KVShape, _I], _S),
    "magicdec_draft_attn": ([KVShape, _P, _P, _P, _P, _P, _P, _S, _P], _I),
    "magicdec_verify_attn": ([KVShape, _I, _P, _P, _P, _P, _P, _P, _S, _P], _I),
    "magicdec_verify_attn_noalloc": ([KVShape, _I, _P, _P, _P, _P, _P, _P], _I),
    "magicdec_draft_cache_update": ([KVShape, _P, _P, _P, _P, _P, _P, _P, _I, _I, _P, _P, _P, _P], _I),
    "magicdec_step_lengths": ([_I, _I, _I, _P, _P, _P, _P, _P], _I),
    "magicdec_pq_encode": ([KVShape, _P, _I, _I, _P, _P, _P], _I),
    "magicdec_pq_update": ([KVShape, _P, _P, _I, _I, _P, _P, _P], _I),
    "magicdec_pq_attn_workspace_size": ([KVShape], _S),
    "magicdec_pq_draft_attn": ([KVShape, _P, _P, _P, _P, _I, _I, _P, _P, _I, _P, _P, _P, _S, _P], _I),
    "magicdec_topk_attn_workspace_size": ([KVShape], _S),
    "magicdec_topk_draft_attn": ([KVShape, _P, _P, _P, _P, _I, _P, _P, _P, _S, _P], _I),
    "magicdec_spec_accept_workspace_size": ([_I, _I, _I], _S),
    "magicdec_spec_accept": ([_I, _I, _I, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P, _S, _P], _I),
}

EXPORTED = tuple(_SIGNATURES)


def lib() -> ctypes.CDLL:
    """Load libmagicdec.so (built by long_context_self_gb300.build); raises if it is absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(f"libmagicdec.so not found at {_LIB_PATH}: build it with "
                                   "`python -m long_context_self_gb300.build` (there is no fallback)")
            h = ctypes.CDLL(_LIB_PATH)
            for name, (args, res) in _SIGNATURES.items():
                fn = getattr(h, name)
                fn.argtypes = args
                fn.restype = res
            _lib = h
    return _lib


def status_string(status: int) -> str:
    return lib().magicdec_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != 0:
        raise MagicdecError(fn, status)


def _stream(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _need(t: torch.Tensor, name: str, dtype, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _need_shape(t: torch.Tensor, name: str, dtype, device, shape):
    """_need plus an exact shape: the kernels index these tensors by the shapes the other
    arguments imply, so a mismatch is refused here rather than read out of bounds."""
    _need(t, name, dtype, device)
    if tuple(t.shape) != tuple(int(s) for s in shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


_ws_cache = {}


def workspace(nbytes: int, device, tag: str) -> torch.Tensor:
    """A zero-filled device workspace, cached per (device, tag) and grown on demand."""
    key = (str(device), tag)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def kv_shape(B, H_q, H_kv, d, L_cap) -> KVShape:
    return KVShape(int(B), int(H_q), int(H_kv), int(d), int(L_cap))


# ----------------------------------------------------------------- entry points
def magicdec_device_error() -> int:
    v = ctypes.c_int32(0)
    _check("magicdec_device_error", lib().magicdec_device_error(ctypes.byref(v)))
    return int(v.value)


def magicdec_streaming_select(seq_len: torch.Tensor, H_kv: int, n_sink: int, n_recent: int,
                              idx: Optional[torch.Tensor] = None, n_sel: Optional[torch.Tensor] = None,
                              stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    _need(seq_len, "seq_len", torch.int32)
    dev = seq_len.device
    if seq_len.dim() != 1:
        raise ValueError("seq_len must be [B]")
    B = seq_len.shape[0]
    if idx is None:
        idx = torch.empty((B, H_kv, n_sink + n_recent), dtype=torch.int32, device=dev)
    if n_sel is None:
        n_sel = torch.empty((B,), dtype=torch.int32, device=dev)
    _need_shape(idx, "idx", torch.int32, dev, (B, H_kv, n_sink + n_recent))
    _need_shape(n_sel, "n_sel", torch.int32, dev, (B,))
    _check("magicdec_streaming_select",
           lib().magicdec_streaming_select(_ptr(seq_len), B, H_kv, n_sink, n_recent, _ptr(idx), _ptr(n_sel),
                                           _stream(stream, dev)))
    return idx, n_sel


def magicdec_snapkv_workspace_size(shape: KVShape, window: int) -> int:
    return int(lib().magicdec_snapkv_workspace_size(shape, int(window)))


def magicdec_snapkv_select(q_win: torch.Tensor, k: torch.Tensor, seq_len: torch.Tensor, window: int,
                           pool_kernel: int, budget: int, idx: Optional[torch.Tensor] = None,
                           n_sel: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                           stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """q_win [B, window, H_q, d] bf16, k [B, L_cap, H_kv, d] bf16 -> idx [B, H_kv, budget], n_sel [B]."""
    _need(q_win, "q_win", torch.bfloat16)
    dev = q_win.device
    _need(k, "k", torch.bfloat16, dev)
    B, w, H_q, d = q_win.shape
    L_cap, H_kv = k.shape[1], k.shape[2]
    if w != window or k.shape[0] != B or k.shape[3] != d:
        raise ValueError("q_win / k shapes disagree")
    _need_shape(seq_len, "seq_len", torch.int32, dev, (B,))
    shape = kv_shape(B, H_q, H_kv, d, L_cap)
    if idx is None:
        idx = torch.empty((B, H_kv, budget), dtype=torch.int32, device=dev)
    if n_sel is None:
        n_sel = torch.empty((B,), dtype=torch.int32, device=dev)
    _need_shape(idx, "idx", torch.int32, dev, (B, H_kv, budget))
    _need_shape(n_sel, "n_sel", torch.int32, dev, (B,))
    need = magicdec_snapkv_workspace_size(shape, window)
    if ws is None:
        ws = workspace(need, dev, "snapkv")
    _check("magicdec_snapkv_select",
           lib().magicdec_snapkv_select(shape, _ptr(q_win), _ptr(k), _ptr(seq_len), window, pool_kernel, budget,
                                        _ptr(idx), _ptr(n_sel), _ptr(ws), ws.numel() * ws.element_size(),
                                        _stream(stream, dev)))
    return idx, n_sel


def magicdec_snapkv_select_budgets(q_win: torch.Tensor, k: torch.Tensor, seq_len: torch.Tensor, window: int,
                                   pool_kernel: int, budgets: torch.Tensor, max_budget: int,
                                   idx: Optional[torch.Tensor] = None, n_sel: Optional[torch.Tensor] = None,
                                   ws: Optional[torch.Tensor] = None,
                                   stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """SnapKV selection with per-sequence budgets (int32 [B], clamped to [window, max_budget])
    -> (idx int32 [B, H_kv, max_budget], n_sel int32 [B])."""
    _need(q_win, "q_win", torch.bfloat16)
    dev = q_win.device
    _need(k, "k", torch.bfloat16, dev)
    B, w, H_q, d = q_win.shape
    L_cap, H_kv = k.shape[1], k.shape[2]
    if w != window or k.shape[0] != B or k.shape[3] != d:
        raise ValueError("q_win / k shapes disagree")
    _need_shape(seq_len, "seq_len", torch.int32, dev, (B,))
    _need_shape(budgets, "budgets", torch.int32, dev, (B,))
    shape = kv_shape(B, H_q, H_kv, d, L_cap)
    if idx is None:
        idx = torch.empty((B, H_kv, max_budget), dtype=torch.int32, device=dev)
    if n_sel is None:
        n_sel = torch.empty((B,), dtype=torch.int32, device=dev)
    _need_shape(idx, "idx", torch.int32, dev, (B, H_kv, max_budget))
    _need_shape(n_sel, "n_sel", torch.int32, dev, (B,))
    if ws is None:
        ws = workspace(magicdec_snapkv_workspace_size(shape, window), dev, "snapkv")
    _check("magicdec_snapkv_select_budgets",
           lib().magicdec_snapkv_select_budgets(shape, _ptr(q_win), _ptr(k), _ptr(seq_len), int(window),
                                                int(pool_kernel), _ptr(budgets), int(max_budget), _ptr(idx),
                                                _ptr(n_sel), _ptr(ws), ws.numel() * ws.element_size(),
                                                _stream(stream, dev)))
    return idx, n_sel


def magicdec_gather_kv(k: torch.Tensor, v: torch.Tensor, idx: torch.Tensor, cap: int,
                       kc: Optional[torch.Tensor] = None, vc: Optional[torch.Tensor] = None,
                       stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """k, v [B, L_cap, H_kv, d], idx [B, H_kv, n_idx] -> kc, vc [B, H_kv, cap, d]."""
    _need(k, "k", torch.bfloat16)
    dev = k.device
    _need(v, "v", torch.bfloat16, dev)
    B, L_cap, H_kv, d = k.shape
    if v.shape != k.shape or idx.dim() != 3:
        raise ValueError("k / v / idx shapes disagree")
    n_idx = idx.shape[2]
    _need_shape(idx, "idx", torch.int32, dev, (B, H_kv, n_idx))
    if kc is None:
        kc = torch.zeros((B, H_kv, cap, d), dtype=torch.bfloat16, device=dev)
    if vc is None:
        vc = torch.zeros((B, H_kv, cap, d), dtype=torch.bfloat16, device=dev)
    _need_shape(kc, "kc", torch.bfloat16, dev, (B, H_kv, cap, d))
    _need_shape(vc, "vc", torch.bfloat16, dev, (B, H_kv, cap, d))
    shape = kv_shape(B, H_kv, H_kv, d, L_cap)
    _check("magicdec_gather_kv",
           lib().magicdec_gather_kv(shape, _ptr(k), _ptr(v), _ptr(idx), n_idx, cap, _ptr(kc), _ptr(vc),
                                    _stream(stream, dev)))
    return kc, vc


def magicdec_attn_workspace_size(shape: KVShape, n_q: int) -> int:
    return int(lib().magicdec_attn_workspace_size(shape, int(n_q)))


def magicdec_draft_attn(q: torch.Tensor, kc: torch.Tensor, vc: torch.Tensor, draft_len: torch.Tensor,
                        out: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                        stream=None) -> torch.Tensor:
    """q [B, 1, H_q, d], kc/vc [B, H_kv, cap, d], draft_len [B] -> out [B, 1, H_q, d] bf16."""
    _need(q, "q", torch.bfloat16)
    dev = q.device
    _need(kc, "kc", torch.bfloat16, dev)
    _need(vc, "vc", torch.bfloat16, dev)
    B, one, H_q, d = q.shape
    H_kv, cap = kc.shape[1], kc.shape[2]
    if one != 1 or kc.shape != vc.shape or kc.shape[0] != B or kc.shape[3] != d:
        raise ValueError("q / kc / vc shapes disagree")
    _need_shape(draft_len, "draft_len", torch.int32, dev, (B,))
    shape = kv_shape(B, H_q, H_kv, d, cap)
    if out is None:
        out = torch.empty_like(q)
    _need_shape(out, "out", torch.bfloat16, dev, q.shape)
    if ws is None:
        ws = workspace(magicdec_attn_workspace_size(shape, 1), dev, "attn")
    _check("magicdec_draft_attn",
           lib().magicdec_draft_attn(shape, _ptr(q), _ptr(kc), _ptr(vc), _ptr(draft_len), _ptr(out), _ptr(ws),
                                     ws.numel() * ws.element_size(), _stream(stream, dev)))
    return out


def magicdec_verify_attn(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, seq_len: torch.Tensor,
                         out: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                         stream=None) -> torch.Tensor:
    """q [B, n_q, H_q, d], k/v [B, L_cap, H_kv, d], seq_len [B] -> out [B, n_q, H_q, d] bf16."""
    _need(q, "q", torch.bfloat16)
    dev = q.device
    _need(k, "k", torch.bfloat16, dev)
    _need(v, "v", torch.bfloat16, dev)
    B, n_q, H_q, d = q.shape
    L_cap, H_kv = k.shape[1], k.shape[2]
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != d:
        raise ValueError("q / k / v shapes disagree")
    _need_shape(seq_len, "seq_len", torch.int32, dev, (B,))
    shape = kv_shape(B, H_q, H_kv, d, L_cap)
    if out is None:
        out = torch.empty_like(q)
    _need_shape(out, "out", torch.bfloat16, dev, q.shape)
    if ws is None:
        ws = workspace(magicdec_attn_workspace_size(shape, n_q), dev, "attn")
    _check("magicdec_verify_attn",
           lib().magicdec_verify_attn(shape, n_q, _ptr(q), _ptr(k), _ptr(v), _ptr(seq_len), _ptr(out), _ptr(ws),
                                      ws.numel() * ws.element_size(), _stream(stream, dev)))
    return out


def magicdec_verify_attn_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, seq_len: torch.Tensor,
                                 out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Verification attention whose scratch lives inside the library (for callers that
    cannot allocate device memory); same shapes and results as magicdec_verify_attn."""
    _need(q, "q", torch.bfloat16)
    dev = q.device
    _need(k, "k", torch.bfloat16, dev)
    _need(v, "v", torch.bfloat16, dev)
    B, n_q, H_q, d = q.shape
    L_cap, H_kv = k.shape[1], k.shape[2]
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != d:
        raise ValueError("q / k / v shapes disagree")
    _need_shape(seq_len, "seq_len", torch.int32, dev, (B,))
    if out is None:
        out = torch.empty_like(q)
    _need_shape(out, "out", torch.bfloat16, dev, q.shape)
    _check("magicdec_verify_attn_noalloc",
           lib().magicdec_verify_attn_noalloc(kv_shape(B, H_q, H_kv, d, L_cap), n_q, _ptr(q), _ptr(k), _ptr(v),
                                              _ptr(seq_len), _ptr(out), _stream(stream, dev)))
    return out


def magicdec_draft_cache_update(k: torch.Tensor, v: torch.Tensor, kc: torch.Tensor, vc: torch.Tensor,
                                len_valid: torch.Tensor, len_old: torch.Tensor, len_new: torch.Tensor,
                                origin: torch.Tensor, base: Optional[torch.Tensor], ring: int,
                                draft_len: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Update the compact draft cache kc/vc [B, H_kv, cap, d] in place from k/v [B, L_cap, H_kv, d];
    ring > 0: StreamingLLM ring layout, ring == 0: SnapKV linear layout (base required).
    Returns draft_len int32 [B]."""
    _need(k, "k", torch.bfloat16)
    dev = k.device
    _need(v, "v", torch.bfloat16, dev)
    _need(kc, "kc", torch.bfloat16, dev)
    _need(vc, "vc", torch.bfloat16, dev)
    B, L_cap, H_kv, d = k.shape
    for name, t in (("len_valid", len_valid), ("len_old", len_old), ("len_new", len_new), ("origin", origin)):
        _need_shape(t, name, torch.int32, dev, (B,))
    if base is not None:
        _need_shape(base, "base", torch.int32, dev, (B,))
    if v.shape != k.shape or kc.shape != vc.shape or kc.shape[0] != B or kc.shape[1] != H_kv or kc.shape[3] != d:
        raise ValueError("k / v / kc / vc shapes disagree")
    cap = kc.shape[2]
    if draft_len is None:
        draft_len = torch.empty((B,), dtype=torch.int32, device=dev)
    _need_shape(draft_len, "draft_len", torch.int32, dev, (B,))
    shape = kv_shape(B, H_kv, H_kv, d, L_cap)
    _check("magicdec_draft_cache_update",
           lib().magicdec_draft_cache_update(shape, _ptr(k), _ptr(v), _ptr(len_valid), _ptr(len_old), _ptr(len_new),
                                             _ptr(origin), _ptr(base), int(ring), int(cap), _ptr(kc), _ptr(vc),
                                             _ptr(draft_len), _stream(stream, dev)))
    return draft_len


def magicdec_step_lengths(len_in: torch.Tensor, gamma: int, L_cap: int, n_acc: Optional[torch.Tensor] = None,
                          len_out: Optional[torch.Tensor] = None, table: Optional[torch.Tensor] = None,
                          stream=None):
    """len_in [B] int32 (+ n_acc [B] int32) -> (len_out [B], table [gamma+2, B]) int32:
    len_out = min(len_in + n_acc + 1, L_cap) (len_in when n_acc is None), table[j] = min(len_out + j, L_cap)."""
    _need(len_in, "len_in", torch.int32)
    dev = len_in.device
    B = len_in.shape[0]
    _need_shape(len_in, "len_in", torch.int32, dev, (B,))
    if n_acc is not None:
        _need_shape(n_acc, "n_acc", torch.int32, dev, (B,))
    if len_out is None:
        len_out = torch.empty((B,), dtype=torch.int32, device=dev)
    if table is None:
        table = torch.empty((gamma + 2, B), dtype=torch.int32, device=dev)
    _need_shape(len_out, "len_out", torch.int32, dev, (B,))
    _need_shape(table, "table", torch.int32, dev, (gamma + 2, B))
    _check("magicdec_step_lengths",
           lib().magicdec_step_lengths(int(B), int(gamma), int(L_cap), _ptr(len_in), _ptr(n_acc), _ptr(len_out),
                                       _ptr(table), _stream(stream, dev)))
    return len_out, table


def _pq_dims(k: torch.Tensor, codebook: torch.Tensor):
    B, L_cap, H_kv, d = k.shape
    if codebook.dim() != 5 or codebook.shape[0] != B or codebook.shape[1] != H_kv or codebook.shape[4] != 8:
        raise ValueError("codebook must be [B, H_kv, M, C, 8]")
    return B, L_cap, H_kv, d, codebook.shape[2], codebook.shape[3]


def magicdec_pq_encode(k: torch.Tensor, codebook: torch.Tensor, codes: Optional[torch.Tensor] = None,
                       stream=None) -> torch.Tensor:
    """k [B, L_cap, H_kv, d] bf16, codebook [B, H_kv, M, C, 8] fp32 -> codes uint8 [B, H_kv, L_cap, M]."""
    _need(k, "k", torch.bfloat16)
    dev = k.device
    _need(codebook, "codebook", torch.float32, dev)
    B, L_cap, H_kv, d, M, C = _pq_dims(k, codebook)
    if codes is None:
        codes = torch.empty((B, H_kv, L_cap, M), dtype=torch.uint8, device=dev)
    _need_shape(codes, "codes", torch.uint8, dev, (B, H_kv, L_cap, M))
    _check("magicdec_pq_encode", lib().magicdec_pq_encode(kv_shape(B, H_kv, H_kv, d, L_cap), _ptr(k), M, C,
                                                          _ptr(codebook), _ptr(codes), _stream(stream, dev)))
    return codes


def magicdec_pq_update(k: torch.Tensor, seq_len: torch.Tensor, codes: torch.Tensor, codebook: torch.Tensor,
                       stream=None) -> torch.Tensor:
    """One Lloyd update of codebook [B, H_kv, M, C, 8] fp32 in place from codes [B, H_kv, L_cap, M]."""
    _need(k, "k", torch.bfloat16)
    dev = k.device
    _need(codebook, "codebook", torch.float32, dev)
    B, L_cap, H_kv, d, M, C = _pq_dims(k, codebook)
    _need_shape(seq_len, "seq_len", torch.int32, dev, (B,))
    _need_shape(codes, "codes", torch.uint8, dev, (B, H_kv, L_cap, M))
    _check("magicdec_pq_update", lib().magicdec_pq_update(kv_shape(B, H_kv, H_kv, d, L_cap), _ptr(k), _ptr(seq_len),
                                                          M, C, _ptr(codes), _ptr(codebook), _stream(stream, dev)))
    return codebook


def magicdec_pq_attn_workspace_size(shape: KVShape) -> int:
    return int(lib().magicdec_pq_attn_workspace_size(shape))


def magicdec_pq_draft_attn(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, seq_len: torch.Tensor,
                           codebook: torch.Tensor, codes: torch.Tensor, top_k: int,
                           out: Optional[torch.Tensor] = None, idx: Optional[torch.Tensor] = None,
                           ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """PQ draft attention.  q [B, 1, H_q, d] -> out [B, 1, H_q, d] bf16; idx optional int32 [B, H_q, top_k]."""
    _need(q, "q", torch.bfloat16)
    dev = q.device
    _need(k, "k", torch.bfloat16, dev)
    _need(v, "v", torch.bfloat16, dev)
    _need(codebook, "codebook", torch.float32, dev)
    B, L_cap, H_kv, d, M, C = _pq_dims(k, codebook)
    H_q = q.shape[2]
    if q.shape[0] != B or q.shape[1] != 1 or q.shape[3] != d or v.shape != k.shape:
        raise ValueError("q / k / v shapes disagree")
    _need_shape(seq_len, "seq_len", torch.int32, dev, (B,))
    _need_shape(codes, "codes", torch.uint8, dev, (B, H_kv, L_cap, M))
    shape = kv_shape(B, H_q, H_kv, d, L_cap)
    if out is None:
        out = torch.empty_like(q)
    _need_shape(out, "out", torch.bfloat16, dev, q.shape)
    if idx is not None:
        _need(idx, "idx", torch.int32, dev)
        if tuple(idx.shape) != (B, H_q, int(top_k)):
            raise ValueError("idx must be [B, H_q, top_k]")
    if ws is None:
        ws = workspace(magicdec_pq_attn_workspace_size(shape), dev, "pq")
    _check("magicdec_pq_draft_attn",
           lib().magicdec_pq_draft_attn(shape, _ptr(q), _ptr(k), _ptr(v), _ptr(seq_len), M, C, _ptr(codebook),
                                        _ptr(codes), int(top_k), _ptr(out), _ptr(idx), _ptr(ws),
                                        ws.numel() * ws.element_size(), _stream(stream, dev)))
    return out


def magicdec_topk_attn_workspace_size(shape: KVShape) -> int:
    return int(lib().magicdec_topk_attn_workspace_size(shape))


def magicdec_topk_draft_attn(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, seq_len: torch.Tensor, top_k: int,
                             out: Optional[torch.Tensor] = None, idx: Optional[torch.Tensor] = None,
                             ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Top-K attention draft.  q [B, 1, H_q, d], k/v [B, L_cap, H_kv, d], seq_len [B] -> out [B, 1, H_q, d]
    bf16.  `idx` (optional int32 [B, H_q, top_k]) receives the kept positions, ascending, -1 padded."""
    _need(q, "q", torch.bfloat16)
    dev = q.device
    _need(k, "k", torch.bfloat16, dev)
    _need(v, "v", torch.bfloat16, dev)
    B, one, H_q, d = q.shape
    L_cap, H_kv = k.shape[1], k.shape[2]
    if one != 1 or k.shape != v.shape or k.shape[0] != B or k.shape[3] != d:
        raise ValueError("q / k / v shapes disagree")
    _need_shape(seq_len, "seq_len", torch.int32, dev, (B,))
    shape = kv_shape(B, H_q, H_kv, d, L_cap)
    if out is None:
        out = torch.empty_like(q)
    _need_shape(out, "out", torch.bfloat16, dev, q.shape)
    if idx is not None:
        _need(idx, "idx", torch.int32, dev)
        if tuple(idx.shape) != (B, H_q, int(top_k)):
            raise ValueError("idx must be [B, H_q, top_k]")
    if ws is None:
        ws = workspace(magicdec_topk_attn_workspace_size(shape), dev, "topk")
    _check("magicdec_topk_draft_attn",
           lib().magicdec_topk_draft_attn(shape, _ptr(q), _ptr(k), _ptr(v), _ptr(seq_len), int(top_k), _ptr(out),
                                          _ptr(idx), _ptr(ws), ws.numel() * ws.element_size(),
                                          _stream(stream, dev)))
    return out


def magicdec_spec_accept_workspace_size(B: int, gamma: int, V: int) -> int:
    return int(lib().magicdec_spec_accept_workspace_size(int(B), int(gamma), int(V)))


def magicdec_spec_accept(target: torch.Tensor, draft: Optional[torch.Tensor], draft_tok: torch.Tensor,
                         u_acc: Optional[torch.Tensor], u_res: Optional[torch.Tensor], greedy: bool,
                         n_acc: Optional[torch.Tensor] = None, out_tok: Optional[torch.Tensor] = None,
                         n_amb: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                         stream=None):
    """target [B, g+1, V] f32, draft [B, g, V] f32 -> (n_acc [B], out_tok [B, g+1], n_amb [B]) int32."""
    _need(target, "target", torch.float32)
    dev = target.device
    if target.dim() != 3:
        raise ValueError("target must be [B, gamma+1, V]")
    B, gp1, V = target.shape
    gamma = gp1 - 1
    if draft is not None:
        _need_shape(draft, "draft", torch.float32, dev, (B, gamma, V))
    _need_shape(draft_tok, "draft_tok", torch.int32, dev, (B, gamma))
    if u_acc is not None:
        _need_shape(u_acc, "u_acc", torch.float32, dev, (B, gamma))
    if u_res is not None:
        _need_shape(u_res, "u_res", torch.float32, dev, (B,))
    if n_acc is None:
        n_acc = torch.empty((B,), dtype=torch.int32, device=dev)
    if out_tok is None:
        out_tok = torch.empty((B, gamma + 1), dtype=torch.int32, device=dev)
    if n_amb is None:
        n_amb = torch.empty((B,), dtype=torch.int32, device=dev)
    _need_shape(n_acc, "n_acc", torch.int32, dev, (B,))
    _need_shape(out_tok, "out_tok", torch.int32, dev, (B, gamma + 1))
    _need_shape(n_amb, "n_amb", torch.int32, dev, (B,))
    if ws is None:
        ws = workspace(magicdec_spec_accept_workspace_size(B, gamma, V), dev, "accept")
    _check("magicdec_spec_accept",
           lib().magicdec_spec_accept(B, gamma, V, _ptr(target), _ptr(draft), _ptr(draft_tok), _ptr(u_acc),
                                      _ptr(u_res), int(bool(greedy)), _ptr(n_acc), _ptr(out_tok), _ptr(n_amb),
                                      _ptr(ws), ws.numel() * ws.element_size(), _stream(stream, dev)))
    return n_acc, out_tok, n_amb
