"""GPU parity of the individual kernels against the CPU oracle, through the C ABI.

Permutes and reorders must be bit-exact; attention and merge results must
meet the tolerances fixed for this method (out: 2e-2 bf16 / 1e-4 fp32 max
abs; lse: 5e-3).
"""
import numpy as np
import pytest
import torch

import context_causal_attention_tcgen05_gb300 as cpa
import oracle
from gpu_common import TOL_LSE, TOL_OUT, assert_close, check_grad, check_ok, f64, max_err, need_gpu
from synth import cu_seqlens_from_lengths, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _raw(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def _rand(shape, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(dtype)


# ---------------------------------------------------------------- reorders and permutes (bit-exact)

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("S,H,D,P", [(64, 4, 8, 4), (96, 2, 16, 3), (8192, 32, 128, 8), (131072, 8, 128, 8)])
def test_zigzag_and_striped_bitexact(dtype, S, H, D, P):
    x = _rand((S, H, D), dtype, 11)
    xd = x.cuda()
    raw = _raw(x).numpy()
    for name, layout in (("zigzag", "zigzag"), ("striped", "striped")):
        if layout == "zigzag" and S % (2 * P):
            continue
        y = getattr(cpa, f"cp_{name}_reorder")(xd, P)
        want = oracle.reorder(raw, P, layout)
        assert np.array_equal(_raw(y.cpu()).numpy(), want), name
        back = getattr(cpa, f"cp_{name}_restore")(y, P)
        assert torch.equal(_raw(back.cpu()), _raw(x)), name + " restore"
    check_ok()


@pytest.mark.parametrize("dtype,S,H,D,P", [
    (torch.float32, 32, 8, 16, 4),         # the handbook's tiny workload
    (torch.bfloat16, 32768, 32, 128, 16),  # llama2-7b attention shape, 2 heads per rank
    (torch.bfloat16, 4096, 8, 128, 8),     # one head per rank (GQA key/value side)
    (torch.float32, 48, 6, 8, 3),
])
def test_ulysses_permute_bitexact(dtype, S, H, D, P):
    x = _rand((S, H, D), dtype, 12)
    xd = x.cuda()
    y = cpa.cp_ulysses_seq2head(xd, P)
    want = oracle.ulysses_seq2head(_raw(x).numpy(), P)
    assert np.array_equal(_raw(y.cpu()).numpy(), want)
    back = cpa.cp_ulysses_head2seq(y, P)
    assert torch.equal(_raw(back.cpu()), _raw(x))
    check_ok()


# ---------------------------------------------------------------- LSE merge

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("Sq,H,D", [(1, 1, 64), (333, 8, 128), (4096, 32, 128), (77, 3, 48), (50, 96, 32)])
def test_lse_merge(dtype, Sq, H, D):
    g = torch.Generator().manual_seed(21)
    o1 = torch.randn(Sq, H, D, generator=g).to(dtype)
    o2 = torch.randn(Sq, H, D, generator=g).to(dtype)
    l1 = torch.randn(H, Sq, generator=g) * 4
    l2 = torch.randn(H, Sq, generator=g) * 4
    # empty parts: some rows only in one part, some in neither
    l1[:, ::7] = -float("inf")
    l2[:, ::5] = -float("inf")
    o1[::7] = 0
    o2[::5] = 0
    ref_o, ref_l = oracle.lse_merge(f64(o1), f64(l1), f64(o2), f64(l2))
    o, l = cpa.cp_lse_merge(o1.cuda(), l1.cuda(), o2.cuda(), l2.cuda())
    tol = 1e-5 if dtype == torch.float32 else 2e-2
    assert max_err(o, ref_o) <= tol
    assert max_err(l, ref_l) <= 1e-5
    # in place into (o1, lse1)
    a, b = o1.cuda(), l1.cuda()
    cpa.cp_lse_merge(a, b, o2.cuda(), l2.cuda(), out=a, lse=b)
    assert max_err(a, ref_o) <= tol and max_err(b, ref_l) <= 1e-5
    check_ok()


# ---------------------------------------------------------------- block attention forward

FWD_CASES = [
    # Sq, Sk, Hq, Hkv, D, q_off, k_off, q_stride, k_stride, docs
    (33, 33, 4, 4, 16, 0, 0, 1, 1, None),
    (17, 40, 4, 2, 32, 40, 0, 1, 1, None),            # later queries against an earlier block
    (1, 129, 2, 1, 64, 200, 0, 1, 1, None),           # single row
    (129, 129, 4, 1, 128, 0, 0, 1, 1, None),          # ragged tail past one 128-row tile
    (300, 260, 4, 2, 128, 100, 60, 1, 1, None),       # offsets, several tiles, ragged
    (64, 64, 2, 2, 64, 3, 1, 4, 4, None),             # striped rank 3 vs rank 1 (P=4)
    (64, 64, 2, 2, 64, 1, 3, 4, 4, None),             # striped rank 1 vs rank 3 (first row empty)
    (256, 256, 4, 2, 128, 0, 0, 1, 1, [50, 1, 77, 128]),   # packed documents
    (20, 30, 2, 2, 64, 0, 25, 1, 1, None),            # every row fully masked
    # 640 units of two query tiles for 148+ CTAs: each CTA walks several, alternating a
    # unit whose rows see no key (rows < 300) and a unit with a single query tile
    (356, 200, 320, 32, 128, 0, 300, 1, 1, None),
]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("case", FWD_CASES)
def test_block_fwd(dtype, case):
    Sq, Sk, Hq, Hkv, D, qo, ko, qs, ks, docs = case
    if dtype == torch.bfloat16 and D not in (64, 128):
        pytest.skip("bf16 path is D in {64, 128}")
    g = torch.Generator().manual_seed(31)
    q = torch.randn(Sq, Hq, D, generator=g).to(dtype)
    k = torch.randn(Sk, Hkv, D, generator=g).to(dtype)
    v = torch.randn(Sk, Hkv, D, generator=g).to(dtype)
    cu = None if docs is None else cu_seqlens_from_lengths(docs)
    ref_o, ref_l = oracle.attention(q, k, v, True, qo, ko, q_stride=qs, k_stride=ks, cu_seqlens=cu)
    cu_d = None if cu is None else torch.from_numpy(cu).cuda()
    o, l = cpa.cp_attn_block_fwd(q.cuda(), k.cuda(), v.cuda(), True, qo, ko, qs, ks, cu_d)
    assert_close(o, l, ref_o, ref_l, dtype, str(case))
    check_ok()


WINDOW_CASES = [
    # Sq, Sk, Hq, Hkv, D, q_off, k_off, window, docs
    (300, 300, 4, 2, 128, 0, 0, 64, None),            # window inside a 128-key tile
    (300, 300, 4, 2, 128, 0, 0, 1, None),             # each query sees only itself
    (520, 520, 2, 1, 128, 0, 0, 200, None),           # window spanning tiles, ragged tail
    (256, 256, 4, 2, 128, 0, 0, 100, [50, 1, 77, 128]),   # window and packed documents
    (200, 300, 2, 2, 64, 150, 0, 90, None),           # later queries against an earlier block
    (129, 129, 4, 4, 128, 0, 0, 129, None),           # window covering the whole block
]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("case", WINDOW_CASES)
def test_block_fwd_window(dtype, case):
    Sq, Sk, Hq, Hkv, D, qo, ko, W, docs = case
    g = torch.Generator().manual_seed(33)
    q = torch.randn(Sq, Hq, D, generator=g).to(dtype)
    k = torch.randn(Sk, Hkv, D, generator=g).to(dtype)
    v = torch.randn(Sk, Hkv, D, generator=g).to(dtype)
    cu = None if docs is None else cu_seqlens_from_lengths(docs)
    ref_o, ref_l = oracle.attention(q, k, v, True, qo, ko, cu_seqlens=cu, window=W)
    cu_d = None if cu is None else torch.from_numpy(cu).cuda()
    o, l = cpa.cp_attn_block_fwd(q.cuda(), k.cuda(), v.cuda(), True, qo, ko, 1, 1, cu_d, window=W)
    assert_close(o, l, ref_o, ref_l, dtype, str(case))
    check_ok()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("case", WINDOW_CASES[:4])
def test_block_bwd_window(dtype, case):
    Sq, Sk, Hq, Hkv, D, qo, ko, W, docs = case
    g = torch.Generator().manual_seed(43)
    q = torch.randn(Sq, Hq, D, generator=g).to(dtype)
    k = torch.randn(Sk, Hkv, D, generator=g).to(dtype)
    v = torch.randn(Sk, Hkv, D, generator=g).to(dtype)
    do = torch.randn(Sq, Hq, D, generator=g).to(dtype)
    cu = None if docs is None else cu_seqlens_from_lengths(docs)
    cu_d = None if cu is None else torch.from_numpy(cu).cuda()
    o, l = cpa.cp_attn_block_fwd(q.cuda(), k.cuda(), v.cuda(), True, qo, ko, 1, 1, cu_d, window=W)
    dq, dk, dv = cpa.cp_attn_block_bwd_typed(q.cuda(), k.cuda(), v.cuda(), o, do.cuda(), l, True, qo, ko, 1, 1, cu_d,
                                       window=W)
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, True, qo, ko, cu_seqlens=cu, window=W)
    tol = TOL_OUT[dtype] if dtype == torch.float32 else 2e-2
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        check_grad(f"{name} {case}", got, ref, tol)
    check_ok()


# ---------------------------------------------------------------- block attention backward

BWD_CASES = [
    # Sq, Sk, Hq, Hkv, D, q_off, k_off, docs, causal
    (33, 33, 4, 4, 16, 0, 0, None, True),
    (40, 50, 4, 2, 64, 60, 20, None, True),
    (130, 130, 4, 1, 128, 0, 0, None, True),
    (96, 96, 2, 2, 64, 0, 0, [10, 50, 36], True),
    (300, 270, 4, 2, 128, 100, 50, None, True),        # several ragged tiles, offsets
    (256, 256, 4, 2, 128, 0, 0, [70, 1, 100, 85], True),  # packed documents
    (200, 150, 2, 1, 128, 0, 0, None, False),          # no mask at all
    (192, 192, 2, 2, 128, 0, 0, [64, 128], False),     # documents without causality
]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("case", BWD_CASES)
def test_block_bwd(dtype, case):
    Sq, Sk, Hq, Hkv, D, qo, ko, docs, causal = case
    if dtype == torch.bfloat16 and D not in (64, 128):
        pytest.skip("bf16 path is D in {64, 128}")
    g = torch.Generator().manual_seed(41)
    q = torch.randn(Sq, Hq, D, generator=g).to(dtype)
    k = torch.randn(Sk, Hkv, D, generator=g).to(dtype)
    v = torch.randn(Sk, Hkv, D, generator=g).to(dtype)
    do = torch.randn(Sq, Hq, D, generator=g).to(dtype)
    cu = None if docs is None else cu_seqlens_from_lengths(docs)
    cu_d = None if cu is None else torch.from_numpy(cu).cuda()
    # forward on the GPU gives the (out, lse) the backward consumes, as in training
    o, l = cpa.cp_attn_block_fwd(q.cuda(), k.cuda(), v.cuda(), causal, qo, ko, 1, 1, cu_d)
    dq, dk, dv = cpa.cp_attn_block_bwd_typed(q.cuda(), k.cuda(), v.cuda(), o, do.cuda(), l, causal, qo, ko, 1, 1, cu_d)
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, causal, qo, ko, cu_seqlens=cu)
    tol = TOL_OUT[dtype] if dtype == torch.float32 else 2e-2
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        check_grad(f"{name} {case}", got, ref, tol)
    check_ok()


# ---------------------------------------------------------------- bounded waits

def test_bounded_wait_gives_up_and_reports():
    assert cpa.cp_check_device_status() == 0
    cpa.cp_debug_bounded_wait(20000)  # 20 ms on a barrier nothing arrives on
    st = cpa.cp_check_device_status()
    assert st == -8, st
    assert "bounded wait" in cpa.cp_last_error()
    assert cpa.cp_check_device_status() == 0  # cleared
    # the context is still usable
    x = torch.ones(16, device="cuda")
    assert float(x.sum()) == 16.0


@pytest.mark.parametrize("S,H,P", [(64, 3, 4), (8192, 32, 8)])
def test_lse_reorder_bitexact(S, H, P):
    x = torch.randn(H, S, generator=torch.Generator().manual_seed(13))
    for layout in ("zigzag", "striped"):
        y = cpa.cp_lse_reorder(x.cuda(), P, layout)
        want = oracle.reorder(x.numpy().T, P, layout).T
        assert np.array_equal(y.cpu().numpy(), want)
        back = cpa.cp_lse_reorder(y, P, layout, inverse=True)
        assert torch.equal(back.cpu(), x)
    check_ok()


@pytest.mark.parametrize("S,Hq,Hkv,D,P,dtype", [
    (64, 4, 2, 64, 4, torch.bfloat16),      # chunk of 8 rows: lse chunks of 8 floats (16-byte runs)
    (72, 4, 4, 32, 6, torch.float32),       # chunk of 6 rows: lse by the column kernel
    (8192, 32, 8, 128, 8, torch.bfloat16),  # the ring workload's shape, GQA
])
def test_batched_ring_permutes_bitexact(S, Hq, Hkv, D, P, dtype):
    # one launch for q, k, v (and one for out + lse) equals the single-tensor calls and the oracle's maps
    g = torch.Generator().manual_seed(17)
    q = torch.randn(S, Hq, D, generator=g).to(dtype)
    k = torch.randn(S, Hkv, D, generator=g).to(dtype)
    v = torch.randn(S, Hkv, D, generator=g).to(dtype)
    lse = torch.randn(Hq, S, generator=g)
    for layout in ("zigzag", "striped"):
        qr, kr, vr = cpa.cp_ring_reorder_qkv(q.cuda(), k.cuda(), v.cuda(), P, layout)
        for got, x in ((qr, q), (kr, k), (vr, v)):
            want = oracle.reorder(x.float().numpy(), P, layout)
            assert np.array_equal(got.float().cpu().numpy(), want), layout
        lre = cpa.cp_lse_reorder(lse.cuda(), P, layout)
        out, lse_back = cpa.cp_ring_restore(qr, lre, P, layout)
        assert torch.equal(out.cpu(), q) and torch.equal(lse_back.cpu(), lse), layout
        out2, none = cpa.cp_ring_restore(kr, None, P, layout)
        assert none is None and torch.equal(out2.cpu(), k)
    check_ok()


def test_block_bwd_gradient_aliasing_an_input():
    # dq written over dout's storage: the kernels still read dout, so the library
    # accumulates in fp32 and casts after them (the direct bf16 path needs disjoint
    # buffers); the result equals the ordinary call bit for bit
    import ctypes
    Sq = Sk = 256
    Hq, Hkv, D = 4, 2, 128
    g = torch.Generator().manual_seed(51)
    q, k, v, do = (torch.randn(S, H, D, generator=g).to(torch.bfloat16).cuda()
                   for S, H in ((Sq, Hq), (Sk, Hkv), (Sk, Hkv), (Sq, Hq)))
    o, l = cpa.cp_attn_block_fwd(q, k, v, True)
    dq_ref, dk_ref, dv_ref = cpa.cp_attn_block_bwd_typed(q, k, v, o, do, l, True)
    buf = do.clone()  # dout and dq share this storage
    dk, dv = torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(cpa.cp_workspace_size("block_bwd", Sq, Hq, Hkv, D, q.dtype, 1), dtype=torch.uint8,
                     device="cuda")
    m = cpa._mask(True, 0, 0, 1, 1, None, 0)
    lib = cpa.load_library()
    st = lib.cp_attn_block_bwd_typed(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), buf.data_ptr(),
                               l.data_ptr(), Sq, Sk, Hq, Hkv, D, cpa.CP_BF16, ctypes.byref(m), 0.0,
                               buf.data_ptr(), dk.data_ptr(), dv.data_ptr(), ws.data_ptr(), ws.numel(),
                               torch.cuda.current_stream().cuda_stream)
    assert st == 0, cpa.cp_last_error()
    torch.cuda.synchronize()
    assert torch.equal(buf, dq_ref) and torch.equal(dk, dk_ref) and torch.equal(dv, dv_ref)
    check_ok()
