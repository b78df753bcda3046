"""GPU parity of the ring and Ulysses drivers (P virtual ranks on one GPU)
against UNPARTITIONED attention computed by the CPU oracle.

Small sizes are compared element by element; the full-size workloads (the
sizes and launch configuration the bench times) are compared on sampled rows
(every head; chunk-boundary rows plus random rows), which the oracle can
compute one by one.
"""
import numpy as np
import pytest
import torch

import context_causal_attention_tcgen05_gb300 as cpa
import oracle
from gpu_common import (TOL_OUT, assert_close, check_grad, check_ok, f64, max_err, need_gpu,
                        oracle_bwd_by_kv_head, sample_rows)
from synth import cu_seqlens_from_lengths, doc_lengths, make_inputs, make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


LAYOUTS = ["contiguous", "zigzag", "striped"]
MODES = ["fused", "stepwise"]


# ---------------------------------------------------------------- the handbook's tiny workload (fp32)

@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("mode", MODES)
def test_tiny_exact_ring(layout, mode):
    q, k, v = make_qkv()  # S=32, H=8, D=16, seed 0
    ref_o, ref_l = oracle.attention(q, k, v, True)
    o, l = cpa.cp_ring_attention(q.cuda(), k.cuda(), v.cuda(), 4, layout, mode)
    assert_close(o, l, ref_o, ref_l, torch.float32, f"ring {layout} {mode}")
    check_ok()


def test_tiny_exact_ulysses():
    q, k, v = make_qkv()
    ref_o, ref_l = oracle.attention(q, k, v, True)
    o, l = cpa.cp_ulysses_attention(q.cuda(), k.cuda(), v.cuda(), 4)
    assert_close(o, l, ref_o, ref_l, torch.float32, "ulysses")
    check_ok()


@pytest.mark.parametrize("layout", LAYOUTS)
def test_tiny_exact_ring_bwd(layout):
    q, k, v = make_qkv()
    g = torch.Generator().manual_seed(5)
    do = torch.randn(q.shape, generator=g)
    o, l = cpa.cp_ring_attention(q.cuda(), k.cuda(), v.cuda(), 4, layout)
    dq, dk, dv = cpa.cp_ring_attention_bwd(q.cuda(), k.cuda(), v.cuda(), o, l, do.cuda(), 4, layout)
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, True)
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        check_grad(name, got, ref, 1e-4)
    check_ok()


# ---------------------------------------------------------------- medium bf16, element by element

@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("mode", MODES)
def test_ring_bf16_medium(layout, mode):
    S, Hq, Hkv, D, P = 1024, 8, 2, 128, 4
    q, k, v = make_inputs(S, Hq, Hkv, D, torch.bfloat16, seed=3)
    ref_o, ref_l = oracle.attention(q, k, v, True)
    o, l = cpa.cp_ring_attention(q.cuda(), k.cuda(), v.cuda(), P, layout, mode)
    assert_close(o, l, ref_o, ref_l, torch.bfloat16, f"{layout} {mode}")
    check_ok()


@pytest.mark.parametrize("layout", ["zigzag", "striped"])
def test_ring_bf16_packed_medium(layout):
    S, Hq, Hkv, D, P = 2048, 4, 2, 128, 4
    q, k, v = make_inputs(S, Hq, Hkv, D, torch.bfloat16, seed=4)
    cu = cu_seqlens_from_lengths(doc_lengths(S, 64, 700, seed=2))
    ref_o, ref_l = oracle.attention(q, k, v, True, cu_seqlens=cu)
    o, l = cpa.cp_ring_attention(q.cuda(), k.cuda(), v.cuda(), P, layout, "fused",
                                 cu_seqlens=torch.from_numpy(cu).cuda())
    assert_close(o, l, ref_o, ref_l, torch.bfloat16, layout)
    check_ok()


@pytest.mark.parametrize("layout,docs", [("zigzag", False), ("zigzag", True), ("contiguous", False)])
def test_ring_reordered_to_seq(layout, docs):
    # the fused ring writing out and lse at their sequence positions (the restore done
    # by the attention's own writes), on inputs in the ranks' layout; ragged chunks
    # (C = 200 is not a multiple of the 128-row tile) and several heads per key head
    S, Hq, Hkv, D, P = 1600, 8, 2, 128, 4
    q, k, v = make_inputs(S, Hq, Hkv, D, torch.bfloat16, seed=9)
    cu = cu_seqlens_from_lengths(doc_lengths(S, 64, 700, seed=5)) if docs else None
    cu_d = None if cu is None else torch.from_numpy(cu).cuda()
    ref_o, ref_l = oracle.attention(q, k, v, True, cu_seqlens=cu)
    reo = cpa.cp_zigzag_reorder if layout == "zigzag" else (lambda x, P: x)
    qr, kr, vr = (reo(x.cuda(), P) for x in (q, k, v))
    o, l = cpa.cp_ring_attention_reordered_to_seq(qr, kr, vr, P, layout, cu_seqlens=cu_d)
    check_ok()
    assert_close(o, l, ref_o, ref_l, torch.bfloat16, f"to_seq {layout} docs={docs}")
    # the driver takes the same path for zigzag + fused: identical results
    o2, l2 = cpa.cp_ring_attention(q.cuda(), k.cuda(), v.cuda(), P, layout, "fused", cu_seqlens=cu_d)
    check_ok()
    assert torch.equal(o, o2) and torch.equal(l, l2)


def test_ring_reordered_to_seq_refuses_striped():
    q = torch.zeros(256, 2, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cpa.CpAttnError) as ei:
        cpa.cp_ring_attention_reordered_to_seq(q, q, q, 4, "striped")
    assert ei.value.status == -5  # CP_ERR_UNSUPPORTED


@pytest.mark.parametrize("Hq,Hkv,P", [(8, 8, 4), (8, 4, 4), (16, 8, 8)])
def test_ulysses_bf16_medium(Hq, Hkv, P):
    S, D = 1024, 128
    q, k, v = make_inputs(S, Hq, Hkv, D, torch.bfloat16, seed=6)
    ref_o, ref_l = oracle.attention(q, k, v, True)
    o, l = cpa.cp_ulysses_attention(q.cuda(), k.cuda(), v.cuda(), P)
    assert_close(o, l, ref_o, ref_l, torch.bfloat16, "ulysses")
    check_ok()


@pytest.mark.parametrize("Hq,Hkv,P", [(8, 2, 4), (8, 1, 8), (16, 4, 8)])
def test_ulysses_replicated_kv_bf16(Hq, Hkv, P):
    # fewer key/value heads than ranks: each is replicated P/Hkv times before the exchange
    S, D = 1024, 128
    q, k, v = make_inputs(S, Hq, Hkv, D, torch.bfloat16, seed=16)
    ref_o, ref_l = oracle.attention(q, k, v, True)
    o, l = cpa.cp_ulysses_attention(q.cuda(), k.cuda(), v.cuda(), P)
    assert_close(o, l, ref_o, ref_l, torch.bfloat16, "ulysses replicated")
    check_ok()


def test_tiny_exact_ulysses_bwd():
    # the handbook's tiny workload (fp32, exact path): Ulysses backward vs the plain gradient
    q, k, v = make_qkv()
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(5))
    o, l = cpa.cp_ulysses_attention(q.cuda(), k.cuda(), v.cuda(), 4)
    dq, dk, dv = cpa.cp_ulysses_attention_bwd(q.cuda(), k.cuda(), v.cuda(), o, l, do.cuda(), 4)
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, True)
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        check_grad(name, got, ref, TOL_OUT[torch.float32])
    check_ok()


@pytest.mark.parametrize("Hq,Hkv,P,D,docs", [(8, 8, 4, 128, False), (8, 4, 4, 128, False),
                                             (8, 2, 4, 128, False), (8, 1, 8, 128, False),
                                             (8, 4, 2, 128, True), (8, 8, 4, 64, False)])
def test_ulysses_bwd_bf16_medium(Hq, Hkv, P, D, docs):
    # the Ulysses backward against the plain gradient of unpartitioned attention
    S = 512
    q, k, v, do = make_inputs(S, Hq, Hkv, D, torch.bfloat16, seed=17, with_dout=True)
    cu = cu_seqlens_from_lengths(doc_lengths(S, 64, 300, seed=4)) if docs else None
    cu_d = None if cu is None else torch.from_numpy(cu).cuda()
    o, l = cpa.cp_ulysses_attention(q.cuda(), k.cuda(), v.cuda(), P, cu_seqlens=cu_d)
    dq, dk, dv = cpa.cp_ulysses_attention_bwd(q.cuda(), k.cuda(), v.cuda(), o, l, do.cuda(), P,
                                              cu_seqlens=cu_d)
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, True, cu_seqlens=cu)
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        check_grad(name, got, ref, 2e-2)
    check_ok()


@pytest.mark.parametrize("Pu,Pr,layout", [(2, 2, "contiguous"), (2, 2, "zigzag"), (4, 2, "striped"), (1, 4, "zigzag"),
                                          (4, 1, "contiguous")])
def test_tiny_exact_usp(Pu, Pr, layout):
    # the handbook's tiny workload (fp32) through Ulysses-inside-groups x ring-across-groups
    q, k, v = make_qkv()
    ref_o, ref_l = oracle.attention(q, k, v, True)
    o, l = cpa.cp_usp_attention(q.cuda(), k.cuda(), v.cuda(), Pu, Pr, layout)
    assert_close(o, l, ref_o, ref_l, torch.float32, f"usp {Pu}x{Pr} {layout}")
    check_ok()


@pytest.mark.parametrize("Pu,Pr,layout,Hkv,docs", [(2, 4, "zigzag", 4, False), (4, 2, "striped", 8, True),
                                                   (2, 2, "contiguous", 2, False), (2, 4, "zigzag", 2, True)])
def test_usp_bf16_medium(Pu, Pr, layout, Hkv, docs):
    S, Hq, D = 2048, 8, 128
    q, k, v = make_inputs(S, Hq, Hkv, D, torch.bfloat16, seed=18)
    cu = cu_seqlens_from_lengths(doc_lengths(S, 64, 700, seed=5)) if docs else None
    cu_d = None if cu is None else torch.from_numpy(cu).cuda()
    ref_o, ref_l = oracle.attention(q, k, v, True, cu_seqlens=cu)
    o, l = cpa.cp_usp_attention(q.cuda(), k.cuda(), v.cuda(), Pu, Pr, layout, cu_seqlens=cu_d)
    assert_close(o, l, ref_o, ref_l, torch.bfloat16, f"usp {Pu}x{Pr} {layout}")
    check_ok()


@pytest.mark.parametrize("Hq,Hkv,P,W,docs", [(8, 4, 4, 100, False), (8, 2, 4, 300, True), (8, 8, 8, 1, False)])
def test_ulysses_window_fwd_bwd(Hq, Hkv, P, W, docs):
    # the sliding-window rule through the Ulysses drivers (forward and backward)
    S, D = 512, 128
    q, k, v, do = make_inputs(S, Hq, Hkv, D, torch.bfloat16, seed=19, with_dout=True)
    cu = cu_seqlens_from_lengths(doc_lengths(S, 64, 300, seed=6)) if docs else None
    cu_d = None if cu is None else torch.from_numpy(cu).cuda()
    ref_o, ref_l = oracle.attention(q, k, v, True, cu_seqlens=cu, window=W)
    o, l = cpa.cp_ulysses_attention(q.cuda(), k.cuda(), v.cuda(), P, cu_seqlens=cu_d, window=W)
    assert_close(o, l, ref_o, ref_l, torch.bfloat16, f"ulysses window {W}")
    dq, dk, dv = cpa.cp_ulysses_attention_bwd(q.cuda(), k.cuda(), v.cuda(), o, l, do.cuda(), P,
                                              cu_seqlens=cu_d, window=W)
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, True, cu_seqlens=cu, window=W)
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        check_grad(name, got, ref, 2e-2)
    check_ok()


@pytest.mark.parametrize("layout,docs", [("zigzag", False), ("contiguous", False), ("striped", False),
                                         ("zigzag", True), ("striped", True)])
def test_ring_bwd_bf16_medium(layout, docs):
    S, Hq, Hkv, D, P = 1024, 4, 1, 128, 4
    q, k, v, do = make_inputs(S, Hq, Hkv, D, torch.bfloat16, seed=7, with_dout=True)
    cu = cu_seqlens_from_lengths(doc_lengths(S, 64, 500, seed=3)) if docs else None
    cu_d = None if cu is None else torch.from_numpy(cu).cuda()
    o, l = cpa.cp_ring_attention(q.cuda(), k.cuda(), v.cuda(), P, layout, cu_seqlens=cu_d)
    dq, dk, dv = cpa.cp_ring_attention_bwd(q.cuda(), k.cuda(), v.cuda(), o, l, do.cuda(), P, layout,
                                           cu_seqlens=cu_d)
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, True, cu_seqlens=cu)
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        check_grad(name, got, ref, 2e-2)
    check_ok()


def test_ring_bwd_lse_not_16_byte_aligned():
    # lse is only 4-byte aligned: its reorder takes the single-float column kernel
    S, Hq, Hkv, D, P = 512, 2, 1, 128, 4
    q, k, v, do = make_inputs(S, Hq, Hkv, D, torch.bfloat16, seed=8, with_dout=True)
    o, l = cpa.cp_ring_attention(q.cuda(), k.cuda(), v.cuda(), P, "zigzag")
    buf = torch.empty(Hq * S + 4, dtype=torch.float32, device="cuda")
    l_odd = buf[1:1 + Hq * S].view(Hq, S)
    l_odd.copy_(l)
    assert l_odd.data_ptr() % 16 != 0
    dq, dk, dv = cpa.cp_ring_attention_bwd(q.cuda(), k.cuda(), v.cuda(), o, l_odd, do.cuda(), P, "zigzag")
    rq, rk, rv = cpa.cp_ring_attention_bwd(q.cuda(), k.cuda(), v.cuda(), o, l, do.cuda(), P, "zigzag")
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        assert torch.equal(got, ref)
    check_ok()


# ---------------------------------------------------------------- full-size workloads, sampled rows

def _sampled_check(q, k, v, o, l, rows, cu=None, what=""):
    S = k.shape[0]
    ref_o, ref_l = oracle.attention(q[rows], k, v, True, pos_q=rows, pos_k=np.arange(S), cu_seqlens=cu)
    o_s = o[torch.from_numpy(rows).cuda()]
    l_s = l[:, torch.from_numpy(rows).cuda()]
    return assert_close(o_s, l_s, ref_o, ref_l, torch.bfloat16, what)


def test_full_ring_fwd_mha_s8192_p8_zigzag():
    S, H, D, P = 8192, 32, 128, 8
    q, k, v = make_inputs(S, H, H, D, torch.bfloat16, seed=0)
    o, l = cpa.cp_ring_attention(q.cuda(), k.cuda(), v.cuda(), P, "zigzag", "fused")
    check_ok()
    _sampled_check(q, k, v, o, l, sample_rows(S, P, "zigzag", 1024), what="ring s8192")
    o2, l2 = cpa.cp_ring_attention(q.cuda(), k.cuda(), v.cuda(), P, "zigzag", "stepwise")
    check_ok()
    _sampled_check(q, k, v, o2, l2, sample_rows(S, P, "zigzag", 64, seed=2), what="ring s8192 stepwise")


def test_full_ulysses_s32768_h32_p16():
    S, H, D, P = 32768, 32, 128, 16
    q, k, v = make_inputs(S, H, H, D, torch.bfloat16, seed=0)
    o, l = cpa.cp_ulysses_attention(q.cuda(), k.cuda(), v.cuda(), P)
    check_ok()
    _sampled_check(q, k, v, o, l, sample_rows(S, P, "contiguous", 48), what="ulysses s32768")


def test_full_packed_varlen_s131072_p8():
    S, Hq, Hkv, D, P = 131072, 32, 8, 128, 8
    q, k, v = make_inputs(S, Hq, Hkv, D, torch.bfloat16, seed=0)
    cu = cu_seqlens_from_lengths(doc_lengths(S, 512, 16384, seed=0))
    cu_d = torch.from_numpy(cu).cuda()
    rows = sample_rows(S, P, "striped", 24)
    rows = np.unique(np.concatenate([rows, cu[1:-1], cu[1:-1] - 1]))  # document boundaries
    for layout in ("striped", "zigzag"):
        o, l = cpa.cp_ring_attention(q.cuda(), k.cuda(), v.cuda(), P, layout, "fused", cu_seqlens=cu_d)
        check_ok()
        _sampled_check(q, k, v, o, l, rows, cu=cu, what=f"packed {layout}")


def test_full_gqa_ring_fwd_bwd_s65536_p4_zigzag():
    """The llama3.1-8b attention shape (Hq=32, Hkv=8), fwd + bwd through the ring.

    Checked exactly where the oracle can compute outputs one by one: forward
    rows (sampled), dQ rows (sampled; a row's gradient needs only that row),
    dK/dV of the LAST 64 key rows (only the last 64 queries see them), plus
    two identities that hold at any size: sum_j dV_j = sum of dO over the
    group's query heads (rows of P sum to 1) and sum_j dK_j = 0 (each row of
    dS sums to 0)."""
    S, Hq, Hkv, D, P = 65536, 32, 8, 128, 4
    G = Hq // Hkv
    q, k, v, do = make_inputs(S, Hq, Hkv, D, torch.bfloat16, seed=0, with_dout=True)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, l = cpa.cp_ring_attention(qd, kd, vd, P, "zigzag", "fused")
    check_ok()
    rows = sample_rows(S, P, "zigzag", 24)
    _sampled_check(q, k, v, o, l, rows, what="gqa fwd")
    dq, dk, dv = cpa.cp_ring_attention_bwd(qd, kd, vd, o, l, dod, P, "zigzag")
    check_ok()
    allpos = np.arange(S)
    # dQ on sampled rows
    rq, _, _ = oracle.attention_bwd(q[rows], k, v, do[rows], True, pos_q=rows, pos_k=allpos)
    check_grad("dq sampled rows", dq[torch.from_numpy(rows).cuda()], rq, 2e-2)
    # dK / dV of the last T key rows
    T = 64
    tail = np.arange(S - T, S)
    _, rk, rv = oracle.attention_bwd(q[S - T:], k, v, do[S - T:], True, pos_q=tail, pos_k=allpos)
    for name, got, ref in (("dk", dk[S - T:], rk[S - T:]), ("dv", dv[S - T:], rv[S - T:])):
        check_grad(f"{name} last {T} key rows", got, ref, 2e-2)
    # identities over all rows (fp64 sums of the GPU result vs of the inputs)
    dv_sum = dv.double().sum(0).cpu().numpy()             # [Hkv, D]
    do_sum = do.double().sum(0).reshape(Hkv, G, D).sum(1).numpy()
    assert np.abs(dv_sum - do_sum).max() <= 1e-2 * max(1.0, np.abs(do_sum).max()), "sum dV"
    dk_sum = dk.double().sum(0).cpu().numpy()
    dk_scale = dk.double().abs().sum(0).cpu().numpy().max()
    assert np.abs(dk_sum).max() <= 1e-3 * dk_scale, "sum dK"


def test_full_ulysses_bwd_s32768_h32_p16():
    """Ulysses forward + backward at S=32768, H=32, D=128, P=16 (the Ulysses shape
    of the pages' cp=16 runs), checked as the GQA ring backward is: dQ on
    sampled rows, dK/dV of the last key rows, and the two identities that hold
    at any size (sum_j dV_j = sum of dO; sum_j dK_j = 0)."""
    S, H, D, P = 32768, 32, 128, 16
    q, k, v, do = make_inputs(S, H, H, D, torch.bfloat16, seed=0, with_dout=True)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, l = cpa.cp_ulysses_attention(qd, kd, vd, P)
    check_ok()
    dq, dk, dv = cpa.cp_ulysses_attention_bwd(qd, kd, vd, o, l, dod, P)
    check_ok()
    allpos = np.arange(S)
    rows = sample_rows(S, P, "contiguous", 16)
    rq, _, _ = oracle.attention_bwd(q[rows], k, v, do[rows], True, pos_q=rows, pos_k=allpos)
    check_grad("dq sampled rows", dq[torch.from_numpy(rows).cuda()], rq, 2e-2)
    T = 48
    tail = np.arange(S - T, S)
    _, rk, rv = oracle.attention_bwd(q[S - T:], k, v, do[S - T:], True, pos_q=tail, pos_k=allpos)
    for name, got, ref in (("dk", dk[S - T:], rk[S - T:]), ("dv", dv[S - T:], rv[S - T:])):
        check_grad(f"{name} last {T} key rows", got, ref, 2e-2)
    dv_sum = dv.double().sum(0).cpu().numpy()
    do_sum = do.double().sum(0).numpy()
    assert np.abs(dv_sum - do_sum).max() <= 1e-2 * max(1.0, np.abs(do_sum).max()), "sum dV"
    dk_sum = dk.double().sum(0).cpu().numpy()
    dk_scale = dk.double().abs().sum(0).cpu().numpy().max()
    assert np.abs(dk_sum).max() <= 1e-3 * dk_scale, "sum dK"


# ---------------------------------------------------------------- every gradient element at the bench's tile counts

@pytest.mark.parametrize("docs", [False, True], ids=["causal", "packed_docs"])
def test_ring_bwd_gqa_s8192_p4_zigzag_every_element(docs):
    """The GQA ring backward (Hq=32, Hkv=8, D=128, P=4 zigzag) at S=8192, where the
    key-stationary kernel runs 512 CTAs (several waves, heaviest first) and walks
    runs of up to 64 query tiles through the mask-free path: every element of dQ,
    dK and dV against the oracle's gradient of unpartitioned attention."""
    S, Hq, Hkv, D, P = 8192, 32, 8, 128, 4
    q, k, v, do = make_inputs(S, Hq, Hkv, D, torch.bfloat16, seed=9, with_dout=True)
    cu = cu_seqlens_from_lengths(doc_lengths(S, 256, 2048, seed=7)) if docs else None
    cu_d = None if cu is None else torch.from_numpy(cu).cuda()
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, l = cpa.cp_ring_attention(qd, kd, vd, P, "zigzag", "fused", cu_seqlens=cu_d)
    dq, dk, dv = cpa.cp_ring_attention_bwd(qd, kd, vd, o, l, dod, P, "zigzag", cu_seqlens=cu_d)
    check_ok()
    rq, rk, rv = oracle_bwd_by_kv_head(q, k, v, do, causal=True, cu_seqlens=cu)
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        check_grad(name, got, ref, 2e-2)


def test_ulysses_bwd_s8192_hq32_hkv8_p16_every_element():
    """The Ulysses backward with 16 virtual ranks (2 query heads each; each of the 8
    key/value heads replicated twice) at S=8192: every element of dQ, dK and dV."""
    S, Hq, Hkv, D, P = 8192, 32, 8, 128, 16
    q, k, v, do = make_inputs(S, Hq, Hkv, D, torch.bfloat16, seed=10, with_dout=True)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, l = cpa.cp_ulysses_attention(qd, kd, vd, P)
    dq, dk, dv = cpa.cp_ulysses_attention_bwd(qd, kd, vd, o, l, dod, P)
    check_ok()
    rq, rk, rv = oracle_bwd_by_kv_head(q, k, v, do, causal=True)
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        check_grad(name, got, ref, 2e-2)


# ---------------------------------------------------------------- the ring backward one block pair at a time

@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 128), (torch.float32, 64), (torch.bfloat16, 64)],
                         ids=["bf16_d128", "f32_d64", "bf16_d64"])
def test_ring_bwd_composed_from_accumulating_block_calls(dtype, D):
    """The handbook's ring ("Ring Attention: passing the KV once around a ring"),
    contiguous layout, P=4: rank r's queries meet the key/value block of every
    source src <= r.  Each pair is one cp_attn_block_bwd call with the FINAL
    (unpartitioned) out and lse of rank r's rows, adding into fp32 dQ / dK / dV
    (the first contribution to a block overwrites garbage, the rest accumulate).
    The sums equal the gradient of unpartitioned attention."""
    S, Hq, Hkv, P = 1024, 4, 2, 4
    C = S // P
    q, k, v, do = make_inputs(S, Hq, Hkv, D, dtype, seed=23, with_dout=True)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, l = cpa.cp_attn_block_fwd(qd, kd, vd, True)  # the final out and lse of every row
    f32 = dict(dtype=torch.float32, device="cuda")
    dq = torch.full((S, Hq, D), float("nan"), **f32)  # garbage the first call must overwrite
    dk = torch.full((S, Hkv, D), float("nan"), **f32)
    dv = torch.full((S, Hkv, D), float("nan"), **f32)
    seen_q, seen_k = set(), set()
    for r in range(P):
        rq = slice(r * C, (r + 1) * C)
        lse_r = l[:, rq].contiguous()
        for src in range(r, -1, -1):  # ring order: own block first, then r-1, ...
            rk = slice(src * C, (src + 1) * C)
            # one call per pair; a block written for the first time is overwritten
            first_q, first_k = r not in seen_q, src not in seen_k
            if first_q != first_k:
                # the call's one accumulate flag covers all three outputs: give the block
                # seen for the first time a zeroed start instead
                if first_q:
                    dq[rq].zero_()
                else:
                    dk[rk].zero_()
                    dv[rk].zero_()
            acc = not (first_q and first_k)
            cpa.cp_attn_block_bwd(qd[rq], kd[rk], vd[rk], o[rq], dod[rq], lse_r, True, r * C, src * C,
                                  dq_acc=dq[rq], dk_acc=dk[rk], dv_acc=dv[rk], accumulate=acc)
            seen_q.add(r)
            seen_k.add(src)
    check_ok()
    ref = oracle.attention_bwd(q, k, v, do, True)
    tol = 2e-2 if dtype == torch.bfloat16 else 1e-4
    for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        check_grad(name, got, want, tol)


def test_block_bwd_accumulate_flag_adds_and_overwrites():
    """accumulate = 0 replaces what the fp32 buffers hold; accumulate = 1 adds to it."""
    S, Hq, Hkv, D = 300, 4, 2, 128
    q, k, v, do = (t.cuda() for t in make_inputs(S, Hq, Hkv, D, torch.bfloat16, seed=24, with_dout=True))
    o, l = cpa.cp_attn_block_fwd(q, k, v, True)
    base = cpa.cp_attn_block_bwd(q, k, v, o, do, l, True)
    f32 = dict(dtype=torch.float32, device="cuda")
    start = [torch.randn(t.shape, **f32) for t in base]
    bufs = [t.clone() for t in start]
    cpa.cp_attn_block_bwd(q, k, v, o, do, l, True, dq_acc=bufs[0], dk_acc=bufs[1], dv_acc=bufs[2],
                          accumulate=True)
    for b, s0, g in zip(bufs, start, base):
        assert torch.allclose(b, s0 + g, rtol=0, atol=1e-5)
    cpa.cp_attn_block_bwd(q, k, v, o, do, l, True, dq_acc=bufs[0], dk_acc=bufs[1], dv_acc=bufs[2],
                          accumulate=False)
    for b, g in zip(bufs, base):
        assert torch.equal(b, g)
    # the typed form is the accumulating form's result rounded once
    typed = cpa.cp_attn_block_bwd_typed(q, k, v, o, do, l, True)
    for t, g in zip(typed, base):
        assert torch.equal(t, g.to(torch.bfloat16))
    check_ok()


@pytest.mark.parametrize("S,P,docs", [(800, 8, False), (800, 16, True), (1000, 4, True), (4096, 8, True),
                                      (2048, 16, False)])
def test_ring_striped_position_tiles(S, P, docs):
    """The fused striped ring tiles by position (each tile = 128/P rows of every
    rank, read as one 3-D box): ragged tails (S not a multiple of 128), every
    compiled P, with and without packed documents, against unpartitioned attention."""
    Hq, Hkv, D = 4, 2, 128
    q, k, v = make_inputs(S, Hq, Hkv, D, torch.bfloat16, seed=25)
    cu = cu_seqlens_from_lengths(doc_lengths(S, 64, 400, seed=9)) if docs else None
    cu_d = None if cu is None else torch.from_numpy(cu).cuda()
    ref_o, ref_l = oracle.attention(q, k, v, True, cu_seqlens=cu)
    o, l = cpa.cp_ring_attention(q.cuda(), k.cuda(), v.cuda(), P, "striped", "fused", cu_seqlens=cu_d)
    assert_close(o, l, ref_o, ref_l, torch.bfloat16, f"striped position tiles S={S} P={P}")
    # the same buffers in the ranks' layout through the reordered entry point
    qr, kr, vr = (cpa.cp_striped_reorder(x.cuda(), P) for x in (q, k, v))
    o2, l2 = cpa.cp_ring_attention_reordered(qr, kr, vr, P, "striped", "fused", cu_seqlens=cu_d)
    o2 = cpa.cp_striped_restore(o2, P)
    l2 = cpa.cp_lse_reorder(l2, P, "striped", inverse=True)
    assert_close(o2, l2, ref_o, ref_l, torch.bfloat16, f"striped reordered S={S} P={P}")
    check_ok()
