"""Child process of test_gpu_debug_checks: the binding picks the library to load from
MAGICDEC_LIBRARY when it is first used, so each build runs in a process of its own.

Each case calls one entry point twice on the same inputs: once with every length and
index in range, once with one length (or gather index) out of range.  It prints one JSON
line: per case the device error word read after each call, and whether the out-of-range
call wrote exactly what the documented clamp gives (a length clamped to [0, L_cap], a
gather index outside [0, L_cap) read as a zero row)."""
import json
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
from long_context_self_gb300 import binding as mb  # noqa: E402

DEV = "cuda:0"
B, H_q, H_kv, d, L_cap = 2, 8, 2, 128, 300


def bf16(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16).to(DEV)


def i32(vals):
    return torch.tensor(vals, dtype=torch.int32, device=DEV)


def same(a, b):
    if a.dtype == torch.bfloat16:
        a, b = a.view(torch.int16), b.view(torch.int16)
    return bool(torch.equal(a, b))


def run(call_ok, call_bad, compare):
    ok = call_ok()
    torch.cuda.synchronize()
    e_ok = mb.magicdec_device_error()
    bad = call_bad()
    torch.cuda.synchronize()
    e_bad = mb.magicdec_device_error()
    return {"err_in_range": e_ok, "err_out_of_range": e_bad, "clamped_output": compare(ok, bad)}


def main():
    k, v = bf16((B, L_cap, H_kv, d), 1), bf16((B, L_cap, H_kv, d), 2)
    res = {"library": os.path.basename(mb._LIB_PATH)}

    # gather: one index past L_cap, one negative other than the -1 padding mark
    n, cap = 40, 48
    g = torch.Generator().manual_seed(3)
    idx = torch.randint(0, L_cap, (B, H_kv, n), generator=g, dtype=torch.int32)
    idx[:, :, -3:] = -1
    bad_idx = idx.clone()
    bad_idx[1, 0, 5] = L_cap + 3
    bad_idx[0, 1, 7] = -7

    def gather_cmp(ok, bad):
        ek, ev = ok[0].clone(), ok[1].clone()
        for t in (ek, ev):
            t[1, 0, 5] = 0
            t[0, 1, 7] = 0
        return same(bad[0], ek) and same(bad[1], ev)

    res["gather_kv"] = run(lambda: mb.magicdec_gather_kv(k, v, idx.to(DEV), cap),
                           lambda: mb.magicdec_gather_kv(k, v, bad_idx.to(DEV), cap), gather_cmp)

    # verification attention: a length past L_cap reads as L_cap
    q = bf16((B, 5, H_q, d), 4)
    res["verify_attn"] = run(lambda: mb.magicdec_verify_attn(q, k, v, i32([L_cap, 200])).clone(),
                             lambda: mb.magicdec_verify_attn(q, k, v, i32([L_cap + 5, 200])).clone(), same)

    # the all-heads verification kernels (eight KV heads, d = 128): 16 and 20 rows per KV head
    k8, v8 = bf16((B, L_cap, 8, d), 12), bf16((B, L_cap, 8, d), 13)
    for n_q8, name in ((4, "verify_attn_heads16"), (5, "verify_attn_heads20")):
        q8 = bf16((B, n_q8, 32, d), 14 + n_q8)
        res[name] = run(lambda: mb.magicdec_verify_attn(q8, k8, v8, i32([L_cap, 200])).clone(),
                        lambda: mb.magicdec_verify_attn(q8, k8, v8, i32([L_cap + 5, 200])).clone(), same)

    # draft attention over a compact cache: lengths below 0 and past the capacity
    kc, vc = bf16((B, H_kv, 64, d), 5), bf16((B, H_kv, 64, d), 6)
    q1 = bf16((B, 1, H_q, d), 7)
    res["draft_attn"] = run(lambda: mb.magicdec_draft_attn(q1, kc, vc, i32([0, 64])).clone(),
                            lambda: mb.magicdec_draft_attn(q1, kc, vc, i32([-2, 64 + 7])).clone(), same)

    # draft-cache append in the linear layout: the new length past L_cap
    origin, base = i32([L_cap - 10] * B), i32([5, 9])
    kc0, vc0 = bf16((B, H_kv, 64, d), 8), bf16((B, H_kv, 64, d), 9)

    def update(len_new):
        kc1, vc1 = kc0.clone(), vc0.clone()
        dl = mb.magicdec_draft_cache_update(k, v, kc1, vc1, origin, origin, i32(len_new), origin, base, 0)
        return kc1, vc1, dl

    res["draft_cache_update"] = run(lambda: update([L_cap, L_cap]), lambda: update([L_cap + 9, L_cap]),
                                    lambda a, b: all(same(x, y) for x, y in zip(a, b)))

    # SnapKV selection scores
    qw = bf16((B, 32, H_q, d), 10)
    res["snapkv_select"] = run(lambda: [t.clone() for t in mb.magicdec_snapkv_select(qw, k, i32([L_cap, 250]), 32, 7, 64)],
                               lambda: [t.clone() for t in mb.magicdec_snapkv_select(qw, k, i32([L_cap + 1, 250]), 32, 7, 64)],
                               lambda a, b: all(same(x, y) for x, y in zip(a, b)))

    # Top-K attention draft
    res["topk_draft_attn"] = run(lambda: mb.magicdec_topk_draft_attn(q1, k, v, i32([L_cap, 150]), 64).clone(),
                                 lambda: mb.magicdec_topk_draft_attn(q1, k, v, i32([L_cap + 11, 150]), 64).clone(),
                                 same)

    # PQ attention draft
    M, C = d // 8, 16
    codebook = torch.randn((B, H_kv, M, C, 8), generator=torch.Generator().manual_seed(11)).to(DEV)
    codes = mb.magicdec_pq_encode(k, codebook)
    res["pq_draft_attn"] = run(
        lambda: mb.magicdec_pq_draft_attn(q1, k, v, i32([L_cap, 120]), codebook, codes, 32).clone(),
        lambda: mb.magicdec_pq_draft_attn(q1, k, v, i32([L_cap + 2, 120]), codebook, codes, 32).clone(), same)

    print(json.dumps(res))


if __name__ == "__main__":
    main()
