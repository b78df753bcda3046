"""Runs one hot-path case a few times on cuda:0 (for profiler captures).

    python -m context_causal_attention_tcgen05_gb300.profile_case --case ring_fwd \
        --S 8192 --Hq 32 --Hkv 32 --P 8 --reps 3

Cases: ring_fwd (reordered inputs, fused ring: one attention launch per rep),
ring_bwd (ring backward; one tcgen05 backward launch per rep), permute
(zigzag reorder of q), ulysses (seq2head of q), merge (in-place fp32 LSE
merge of two [S, Hq, D] partial outputs).  Inputs are N(0,1) bf16 from
the shared seeded generators.  Exits non-zero if the library reports an error.
"""
from __future__ import annotations

import argparse
import sys

import torch

import context_causal_attention_tcgen05_gb300 as cpa


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", choices=["ring_fwd", "ring_bwd", "permute", "reorder_qkv", "ulysses", "merge"], required=True)
    ap.add_argument("--S", type=int, default=8192)
    ap.add_argument("--Hq", type=int, default=32)
    ap.add_argument("--Hkv", type=int, default=32)
    ap.add_argument("--D", type=int, default=128)
    ap.add_argument("--P", type=int, default=8)
    ap.add_argument("--layout", default="zigzag")
    ap.add_argument("--reps", type=int, default=3)
    a = ap.parse_args(argv)
    import os
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from synth import make_inputs

    torch.cuda.set_device(0)
    cpa.load_library()
    q, k, v, do = (t.cuda() for t in make_inputs(a.S, a.Hq, a.Hkv, a.D, torch.bfloat16, 0, True))
    if a.case == "ring_fwd":
        qr = cpa.cp_zigzag_reorder(q, a.P) if a.layout == "zigzag" else q
        kr = cpa.cp_zigzag_reorder(k, a.P) if a.layout == "zigzag" else k
        vr = cpa.cp_zigzag_reorder(v, a.P) if a.layout == "zigzag" else v
        for _ in range(a.reps):
            cpa.cp_ring_attention_reordered(qr, kr, vr, a.P, a.layout, "fused")
    elif a.case == "ring_bwd":
        o, l = cpa.cp_ring_attention(q, k, v, a.P, a.layout, "fused")
        ws = torch.empty(cpa.cp_workspace_size("ring_bwd", a.S, a.Hq, a.Hkv, a.D, q.dtype, a.P),
                         dtype=torch.uint8, device=q.device)
        for _ in range(a.reps):
            cpa.cp_ring_attention_bwd(q, k, v, o, l, do, a.P, a.layout, workspace=ws)
    elif a.case == "merge":
        g = torch.Generator(device="cuda").manual_seed(1)
        o1 = torch.randn(a.S, a.Hq, a.D, device="cuda", generator=g)
        o2 = torch.randn(a.S, a.Hq, a.D, device="cuda", generator=g)
        l1 = torch.randn(a.Hq, a.S, device="cuda", generator=g)
        l2 = torch.randn(a.Hq, a.S, device="cuda", generator=g)
        for _ in range(a.reps):
            cpa.cp_lse_merge(o1, l1, o2, l2, out=o1, lse=l1)
    elif a.case == "reorder_qkv":  # the ring step's input permute: q, k, v in one launch
        ys = [torch.empty_like(x) for x in (q, k, v)]
        for _ in range(a.reps):
            cpa.cp_ring_reorder_qkv(q, k, v, a.P, a.layout, q_re=ys[0], k_re=ys[1], v_re=ys[2])
    elif a.case == "permute":
        y = torch.empty_like(q)
        for _ in range(a.reps):
            cpa.cp_zigzag_reorder(q, a.P, y=y)
    else:
        y = torch.empty(a.P, a.S, a.Hq // a.P, a.D, dtype=q.dtype, device=q.device)
        for _ in range(a.reps):
            cpa.cp_ulysses_seq2head(q, a.P, y=y)
    torch.cuda.synchronize()
    st = cpa.cp_check_device_status()
    if st != 0:
        print("device status", st, cpa.cp_last_error(), file=sys.stderr)
        return 1
    print("ok")
    return 0


if __name__ == "__main__":
    sys.exit(main())
