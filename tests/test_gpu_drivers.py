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
from gpu_common import TOL_OUT, assert_close, check_ok, f64, max_err, need_gpu, sample_rows
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
        assert max_err(got, ref) <= 1e-4 * max(1.0, float(np.abs(ref).max())), name
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
        assert max_err(got, ref) <= TOL_OUT[torch.float32] * max(1.0, float(np.abs(ref).max())), name
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
        assert max_err(got, ref) <= 2e-2 * max(1.0, float(np.abs(ref).max())), name
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
        assert max_err(got, ref) <= 2e-2 * max(1.0, float(np.abs(ref).max())), name
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
        assert max_err(got, ref) <= 2e-2 * max(1.0, float(np.abs(ref).max())), name
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
    e = max_err(dq[torch.from_numpy(rows).cuda()], rq)
    assert e <= 2e-2 * max(1.0, float(np.abs(rq).max())), f"dq {e}"
    # dK / dV of the last T key rows
    T = 64
    tail = np.arange(S - T, S)
    _, rk, rv = oracle.attention_bwd(q[S - T:], k, v, do[S - T:], True, pos_q=tail, pos_k=allpos)
    for name, got, ref in (("dk", dk[S - T:], rk[S - T:]), ("dv", dv[S - T:], rv[S - T:])):
        e = max_err(got, ref)
        assert e <= 2e-2 * max(1.0, float(np.abs(ref).max())), f"{name} {e}"
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
    e = max_err(dq[torch.from_numpy(rows).cuda()], rq)
    assert e <= 2e-2 * max(1.0, float(np.abs(rq).max())), f"dq {e}"
    T = 48
    tail = np.arange(S - T, S)
    _, rk, rv = oracle.attention_bwd(q[S - T:], k, v, do[S - T:], True, pos_q=tail, pos_k=allpos)
    for name, got, ref in (("dk", dk[S - T:], rk[S - T:]), ("dv", dv[S - T:], rv[S - T:])):
        e = max_err(got, ref)
        assert e <= 2e-2 * max(1.0, float(np.abs(ref).max())), f"{name} {e}"
    dv_sum = dv.double().sum(0).cpu().numpy()
    do_sum = do.double().sum(0).numpy()
    assert np.abs(dv_sum - do_sum).max() <= 1e-2 * max(1.0, np.abs(do_sum).max()), "sum dV"
    dk_sum = dk.double().sum(0).cpu().numpy()
    dk_scale = dk.double().abs().sum(0).cpu().numpy().max()
    assert np.abs(dk_sum).max() <= 1e-3 * dk_scale, "sum dK"
