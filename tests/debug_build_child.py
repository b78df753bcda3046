"""Runs in a child process with CP_ATTN_LIBRARY naming the index-checking debug
build (libcp_attn_debug.so): every kernel family on small ragged cases, each
result against the oracle, and the device status after each.  That build also
orders every attention launch in blocks of one key/value head, so the blocked
unit orders that release builds use at large sizes run here at small ones.
Exits 0 when all results meet their bounds and no index check fired; prints one
line per check."""
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import context_causal_attention_tcgen05_gb300 as cpa  # noqa: E402
import oracle  # noqa: E402
from synth import cu_seqlens_from_lengths, make_inputs, make_qkv  # noqa: E402


def err(a, b):
    a = a.detach().float().cpu().double().numpy()
    b = np.asarray(b, dtype=np.float64)
    both = np.isneginf(a) & np.isneginf(b)
    with np.errstate(invalid="ignore"):
        return float(np.nan_to_num(np.abs(np.where(both, 0.0, a - b)), nan=np.inf).max())


failures = []


def check(name, e, bound):
    st = cpa.cp_check_device_status()
    ok = e <= bound and st == 0
    print(f"{'ok  ' if ok else 'FAIL'} {name}: err {e:.3g} bound {bound:.3g} status {st}", flush=True)
    if not ok:
        failures.append(name)


def main():
    assert os.path.basename(cpa.library_path()) == "libcp_attn_debug.so", cpa.library_path()
    cpa.load_library()
    torch.cuda.set_device(0)
    # the handbook's tiny fp32 workload through every layout and Ulysses (FFMA kernels, movers, merge)
    q, k, v = make_qkv()
    ro, rl = oracle.attention(q, k, v, True)
    for layout in ("contiguous", "zigzag", "striped"):
        for mode in ("fused", "stepwise"):
            o, l = cpa.cp_ring_attention(q.cuda(), k.cuda(), v.cuda(), 4, layout, mode)
            check(f"tiny ring {layout} {mode} out", err(o, ro), 1e-4)
    o, l = cpa.cp_ulysses_attention(q.cuda(), k.cuda(), v.cuda(), 4)
    check("tiny ulysses out", err(o, ro), 1e-4)
    # bf16 tensor-core kernels: ragged ring with packed documents, fwd + bwd, both head sizes
    S, Hq, Hkv, P = 1536, 4, 2, 4
    cu = cu_seqlens_from_lengths([300, 1, 500, 611, 124])
    cu_d = torch.from_numpy(cu).cuda()
    for D in (64, 128):
        q, k, v, do = make_inputs(S, Hq, Hkv, D, torch.bfloat16, seed=31, with_dout=True)
        ro, rl = oracle.attention(q, k, v, True, cu_seqlens=cu)
        rq, rk, rv = oracle.attention_bwd(q, k, v, do, True, cu_seqlens=cu)
        for layout in ("zigzag", "striped"):
            o, l = cpa.cp_ring_attention(q.cuda(), k.cuda(), v.cuda(), P, layout, cu_seqlens=cu_d)
            check(f"ring {layout} D={D} out", err(o, ro), 2e-2)
            check(f"ring {layout} D={D} lse", err(l, rl), 5e-3)
            g = cpa.cp_ring_attention_bwd(q.cuda(), k.cuda(), v.cuda(), o, l, do.cuda(), P, layout, cu_seqlens=cu_d)
            for name, got, ref in zip(("dq", "dk", "dv"), g, (rq, rk, rv)):
                check(f"ring bwd {layout} D={D} {name}", err(got, ref), 2e-2 * max(1.0, float(np.abs(ref).max())))
    # ring without documents (GQA, both layouts): the debug build orders every launch in
    # blocks of one key/value head, so the blocked unit orders run element by element here
    S, Hq, Hkv, D, P = 2048, 8, 2, 128, 4
    q, k, v, do = make_inputs(S, Hq, Hkv, D, torch.bfloat16, seed=34, with_dout=True)
    ro, rl = oracle.attention(q, k, v, True)
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, True)
    for layout in ("zigzag", "contiguous"):
        o, l = cpa.cp_ring_attention(q.cuda(), k.cuda(), v.cuda(), P, layout)
        check(f"ring {layout} gqa out", err(o, ro), 2e-2)
        check(f"ring {layout} gqa lse", err(l, rl), 5e-3)
        g = cpa.cp_ring_attention_bwd(q.cuda(), k.cuda(), v.cuda(), o, l, do.cuda(), P, layout)
        for name, got, ref in zip(("dq", "dk", "dv"), g, (rq, rk, rv)):
            check(f"ring bwd {layout} gqa {name}", err(got, ref), 2e-2 * max(1.0, float(np.abs(ref).max())))
    # Ulysses with replicated key/value heads and a window, fwd + bwd
    S, Hq, Hkv, D, P, W = 512, 8, 2, 128, 4, 100
    q, k, v, do = make_inputs(S, Hq, Hkv, D, torch.bfloat16, seed=32, with_dout=True)
    ro, rl = oracle.attention(q, k, v, True, window=W)
    o, l = cpa.cp_ulysses_attention(q.cuda(), k.cuda(), v.cuda(), P, window=W)
    check("ulysses window out", err(o, ro), 2e-2)
    g = cpa.cp_ulysses_attention_bwd(q.cuda(), k.cuda(), v.cuda(), o, l, do.cuda(), P, window=W)
    for name, got, ref in zip(("dq", "dk", "dv"), g, oracle.attention_bwd(q, k, v, do, True, window=W)):
        check(f"ulysses bwd {name}", err(got, ref), 2e-2 * max(1.0, float(np.abs(ref).max())))
    # a block pair with offsets and strides (striped ranks), fp32 and bf16
    for dt, tol in ((torch.float32, 1e-4), (torch.bfloat16, 2e-2)):
        q, k, v, do = make_inputs(200, 4, 2, 64, dt, seed=33, with_dout=True)
        ro, rl = oracle.attention(q, k, v, True, 3, 1, q_stride=4, k_stride=4)
        o, l = cpa.cp_attn_block_fwd(q.cuda(), k.cuda(), v.cuda(), True, 3, 1, 4, 4)
        check(f"block strided {dt} out", err(o, ro), tol)
        acc = cpa.cp_attn_block_bwd(q.cuda(), k.cuda(), v.cuda(), o, do.cuda(), l, True, 3, 1, 4, 4)
        ref = oracle.attention_bwd(q, k, v, do, True, 3, 1, q_stride=4, k_stride=4)
        for name, got, r in zip(("dq", "dk", "dv"), acc, ref):
            check(f"block strided {dt} {name}", err(got, r), tol * max(1.0, float(np.abs(r).max())))
    # the merge and the Ulysses permute, bit-exact permute
    o1, o2 = (torch.randn(333, 8, 128) for _ in range(2))
    l1, l2 = (torch.randn(8, 333) for _ in range(2))
    mo, ml = cpa.cp_lse_merge(o1.cuda(), l1.cuda(), o2.cuda(), l2.cuda())
    eo, el = oracle.lse_merge(o1.double().numpy(), l1.double().numpy(), o2.double().numpy(), l2.double().numpy())
    check("merge out", err(mo, eo), 1e-5)
    x = torch.randn(4096, 8, 128).to(torch.bfloat16)
    y = cpa.cp_ulysses_seq2head(x.cuda(), 8)
    same = np.array_equal(y.cpu().view(torch.int16).numpy(), oracle.ulysses_seq2head(x.view(torch.int16).numpy(), 8))
    check("seq2head bit-exact", 0.0 if same else 1.0, 0.0)
    print("debug build: %d failures" % len(failures), flush=True)
    return 1 if failures else 0


if __name__ == "__main__":
    sys.exit(main())
