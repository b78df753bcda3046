"""Pins for the CPU float64 oracle (no GPU).

Each check ties the oracle to something other than itself: a library routine
(torch's scaled_dot_product_attention and autograd in float64), a closed form,
brute force with scalar loops on tiny inputs, or an invariant of the method
stated in the handbook chapter "Context parallelism: Ring Attention and
Ulysses".  The mutation tests at the end show that plausible mistakes in the
oracle (a dropped scale, an off-by-one mask, swapped operands, a wrong GQA
head map, a wrong merge weight) each fail at least one pin.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import block_attention as oattn_mod
from synth import cu_seqlens_from_lengths, make_qkv

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _sdpa(q, k, v, mask=None, is_causal=False):
    """torch SDPA in float64; q [Sq,H,D], k/v [Sk,Hkv,D] with GQA by repeat_interleave."""
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]
    G = q.shape[1] // k.shape[1]
    kt = torch.from_numpy(k).repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    vt = torch.from_numpy(v).repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    m = None if mask is None else torch.from_numpy(mask)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, is_causal=is_causal)
    return o[0].permute(1, 0, 2).numpy()


def _brute_mask(pos_q, pos_k, causal, cu=None):
    """Visibility by scalar loops: key after query is hidden; other document is hidden."""
    def doc(p):
        if cu is None:
            return 0
        d = 0
        while not (cu[d] <= p < cu[d + 1]):
            d += 1
        return d
    m = np.zeros((len(pos_q), len(pos_k)), dtype=bool)
    for i, pq in enumerate(pos_q):
        for j, pk in enumerate(pos_k):
            ok = True
            if causal and pk > pq:
                ok = False
            if cu is not None and doc(pk) != doc(pq):
                ok = False
            m[i, j] = ok
    return m


# ---------------------------------------------------------------- checks (parametrised by implementation)

def check_fwd_vs_sdpa(attn):
    for (Sq, Hq, Hkv, D, seed) in [(17, 4, 4, 8, 0), (33, 8, 2, 16, 1)]:
        q, k, v = _rand((Sq, Hq, D), seed), _rand((Sq, Hkv, D), seed + 10), _rand((Sq, Hkv, D), seed + 20)
        out, _ = attn(q, k, v, True)
        ref = _sdpa(q, k, v, is_causal=True)
        assert np.abs(out - ref).max() < 1e-12
    # offsets / strides / unequal lengths against an explicit brute-force mask
    Sq, Sk, H, D = 9, 13, 3, 5
    q, k, v = _rand((Sq, H, D), 3), _rand((Sk, H, D), 4), _rand((Sk, H, D), 5)
    for (qo, ko, qs, ks) in [(20, 0, 1, 1), (20, 15, 1, 1), (3, 1, 4, 4), (12, 0, 2, 1)]:
        pq = qo + qs * np.arange(Sq)
        pk = ko + ks * np.arange(Sk)
        m = _brute_mask(pq, pk, True)
        assert m.any(axis=1).all()
        out, _ = attn(q, k, v, True, qo, ko, q_stride=qs, k_stride=ks)
        ref = _sdpa(q, k, v, mask=m)
        assert np.abs(out - ref).max() < 1e-12


def check_lse_closed_form(attn):
    # q = 0 makes every visible score 0: lse = log(#visible), out = mean of visible v rows.
    Sq, Sk, H, D = 7, 11, 2, 3
    q = np.zeros((Sq, H, D))
    k, v = _rand((Sk, H, D), 7), _rand((Sk, H, D), 8)
    cu = np.array([0, 3, 9, 30])
    for (qo, ko, cuv) in [(0, 0, None), (5, 0, None), (6, 2, cu)]:
        pq, pk = qo + np.arange(Sq), ko + np.arange(Sk)
        m = _brute_mask(pq, pk, True, cuv)
        out, lse = attn(q, k, v, True, qo, ko, cu_seqlens=cuv)
        for i in range(Sq):
            n = int(m[i].sum())
            for h in range(H):
                if n == 0:
                    assert lse[h, i] == -np.inf and np.all(out[i, h] == 0)
                else:
                    assert abs(lse[h, i] - math.log(n)) < 1e-13
                    assert np.abs(out[i, h] - v[m[i], h].mean(axis=0)).max() < 1e-13


def check_lse_bruteforce(attn):
    Sq, Sk, Hq, Hkv, D = 3, 5, 4, 2, 3
    q, k, v = _rand((Sq, Hq, D), 11), _rand((Sk, Hkv, D), 12), _rand((Sk, Hkv, D), 13)
    qo, ko = 2, 0
    out, lse = attn(q, k, v, True, qo, ko)
    for h in range(Hq):
        hk = h // (Hq // Hkv)
        for i in range(Sq):
            sc = []
            for j in range(Sk):
                if ko + j <= qo + i:
                    s = 0.0
                    for d in range(D):
                        s += q[i, h, d] * k[j, hk, d]
                    sc.append((j, s / math.sqrt(D)))
            mx = max(s for _, s in sc)
            tot = sum(math.exp(s - mx) for _, s in sc)
            L = mx + math.log(tot)
            assert abs(lse[h, i] - L) < 1e-12
            for d in range(D):
                o = sum(math.exp(s - L) * v[j, hk, d] for j, s in sc)
                assert abs(out[i, h, d] - o) < 1e-12


def check_doc_mask(attn):
    lengths = [5, 1, 9, 4]
    cu = cu_seqlens_from_lengths(lengths)
    S, Hq, Hkv, D = sum(lengths), 4, 2, 8
    q, k, v = _rand((S, Hq, D), 21), _rand((S, Hkv, D), 22), _rand((S, Hkv, D), 23)
    out, _ = attn(q, k, v, True, cu_seqlens=cu)
    for d in range(len(lengths)):
        a, b = cu[d], cu[d + 1]
        ref = _sdpa(q[a:b], k[a:b], v[a:b], is_causal=True)
        assert np.abs(out[a:b] - ref).max() < 1e-12


def check_merge(attn, merge):
    S, Hq, Hkv, D = 12, 4, 2, 6
    q, k, v = _rand((S, Hq, D), 31), _rand((S, Hkv, D), 32), _rand((S, Hkv, D), 33)
    rng = np.random.default_rng(34)
    sel = rng.random(S) < 0.5
    sel[0] = True
    pos = np.arange(S)
    A, B = pos[sel], pos[~sel]
    oA, lA = attn(q, k[A], v[A], True, pos_q=pos, pos_k=A)
    oB, lB = attn(q, k[B], v[B], True, pos_q=pos, pos_k=B)
    o, l = merge(oA, lA, oB, lB)
    ow, lw = attn(q, k, v, True)
    assert np.abs(o - ow).max() < 1e-12 and np.abs(l - lw).max() < 1e-12
    o2, l2 = merge(oB, lB, oA, lA)
    assert np.abs(o2 - o).max() < 1e-13 and np.abs(l2 - l).max() < 1e-13


# ---------------------------------------------------------------- the pins

def test_fwd_matches_torch_sdpa_f64():
    check_fwd_vs_sdpa(oracle.attention)


def test_lse_closed_form_zero_query():
    check_lse_closed_form(oracle.attention)


def test_lse_and_out_bruteforce_scalar_loops():
    check_lse_bruteforce(oracle.attention)


def test_document_mask_equals_per_document_sdpa():
    check_doc_mask(oracle.attention)


def test_single_visible_key_gives_that_key():
    # Sk = 1 visible: out = v_0, lse = the one score.
    q, k, v = _rand((4, 2, 4), 41), _rand((1, 2, 4), 42), _rand((1, 2, 4), 43)
    out, lse = oracle.attention(q, k, v, True, 10, 0)
    assert np.abs(out - np.broadcast_to(v, out.shape)).max() < 1e-15
    ref = np.einsum("qhd,hd->hq", q, k[0]) / 2.0
    assert np.abs(lse - ref).max() < 1e-14


def test_fully_masked_rows_are_empty():
    q, k, v = _rand((4, 2, 4), 44), _rand((6, 2, 4), 45), _rand((6, 2, 4), 46)
    out, lse = oracle.attention(q, k, v, True, 0, 4)  # key positions 4..9, query 0..3
    assert np.all(np.isneginf(lse)) and np.all(out == 0)
    out, lse = oracle.attention(q, k, v, True, 4, 4)  # query 4..7: row 0 sees key 4 only
    assert np.isfinite(lse).all()
    empty_q = np.zeros((0, 2, 4))
    o, l = oracle.attention(empty_q, k, v, True)
    assert o.shape == (0, 2, 4) and l.shape == (2, 0)


def test_bwd_matches_torch_autograd_f64():
    for (S, Hq, Hkv, D, seed) in [(13, 4, 4, 8, 50), (19, 8, 2, 16, 51)]:
        q, k, v, do = (_rand((S, Hq, D), seed), _rand((S, Hkv, D), seed + 1),
                       _rand((S, Hkv, D), seed + 2), _rand((S, Hq, D), seed + 3))
        dq, dk, dv = oracle.attention_bwd(q, k, v, do, True)
        qt = torch.from_numpy(q).requires_grad_()
        kt = torch.from_numpy(k).requires_grad_()
        vt = torch.from_numpy(v).requires_grad_()
        G = Hq // Hkv
        o = torch.nn.functional.scaled_dot_product_attention(
            qt.permute(1, 0, 2)[None], kt.repeat_interleave(G, 1).permute(1, 0, 2)[None],
            vt.repeat_interleave(G, 1).permute(1, 0, 2)[None], is_causal=True)[0].permute(1, 0, 2)
        (o * torch.from_numpy(do)).sum().backward()
        assert np.abs(dq - qt.grad.numpy()).max() < 1e-11
        assert np.abs(dk - kt.grad.numpy()).max() < 1e-11
        assert np.abs(dv - vt.grad.numpy()).max() < 1e-11


def test_bwd_finite_differences_with_offsets_and_docs():
    S, Hq, Hkv, D = 6, 2, 1, 3
    q, k, v, do = _rand((S, Hq, D), 60), _rand((S, Hkv, D), 61), _rand((S, Hkv, D), 62), _rand((S, Hq, D), 63)
    cu = np.array([0, 2, 6])
    kw = dict(cu_seqlens=cu)
    grads = oracle.attention_bwd(q, k, v, do, True, **kw)

    def loss(q_, k_, v_):
        o, _ = oracle.attention(q_, k_, v_, True, **kw)
        return float(np.sum(o * do))

    h = 1e-6
    for which, x in enumerate((q, k, v)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = [q, k, v]
            args_m = [q, k, v]
            args_p[which] = xp
            args_m[which] = xm
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert np.abs(num - grads[which]).max() < 1e-7


def test_merge_of_split_softmax_equals_whole():
    check_merge(oracle.attention, oracle.lse_merge)


def test_merge_with_empty_part_is_identity():
    o = _rand((5, 3, 4), 70)
    l = _rand((3, 5), 71)
    empty_o = np.zeros_like(o)
    empty_l = np.full_like(l, -np.inf)
    mo, ml = oracle.lse_merge(o, l, empty_o, empty_l)
    assert np.array_equal(mo, o) and np.array_equal(ml, l)
    mo, ml = oracle.lse_merge(empty_o, empty_l, empty_o, empty_l)
    assert np.all(np.isneginf(ml)) and np.all(mo == 0)


def test_merge_associative():
    S, H, D = 10, 2, 4
    q, k, v = _rand((S, H, D), 80), _rand((S, H, D), 81), _rand((S, H, D), 82)
    pos = np.arange(S)
    parts = [pos[0:3], pos[3:7], pos[7:10]]
    res = [oracle.attention(q, k[p], v[p], True, pos_q=pos, pos_k=p) for p in parts]
    a = oracle.lse_merge(*oracle.lse_merge(*res[0], *res[1]), *res[2])
    b = oracle.lse_merge(*res[0], *oracle.lse_merge(*res[1], *res[2]))
    assert np.abs(a[0] - b[0]).max() < 1e-13 and np.abs(a[1] - b[1]).max() < 1e-13


def test_seq2head_index_map_and_inverse():
    for (S, H, D, P) in [(8, 4, 2, 2), (12, 6, 3, 3), (32, 8, 16, 4)]:
        x = np.arange(S * H * D, dtype=np.float64).reshape(S, H, D)
        y = oracle.ulysses_seq2head(x, P)
        assert y.shape == (P, S, H // P, D)
        Hp = H // P
        for p in range(P):
            for s in range(S):
                for hh in range(Hp):
                    # rank p holds the whole sequence for its share p of the heads
                    assert np.array_equal(y[p, s, hh], x[s, p * Hp + hh])
        assert np.array_equal(oracle.ulysses_head2seq(y, P), x)
        parts = oracle.seq_to_head([x[r * (S // P):(r + 1) * (S // P)] for r in range(P)], P)
        back = oracle.head_to_seq(parts, P)
        assert np.array_equal(np.concatenate(back), x)


def test_reorder_index_maps():
    S, P = 16, 4
    x = np.arange(S)
    z = oracle.reorder(x, P, "zigzag")
    C = S // (2 * P)
    exp = []
    for r in range(P):
        exp += list(range(r * C, (r + 1) * C)) + list(range((2 * P - 1 - r) * C, (2 * P - r) * C))
    assert list(z) == exp
    st = oracle.reorder(x, P, "striped")
    assert list(st) == [i * P + r for r in range(P) for i in range(S // P)]
    for lay in ("contiguous", "zigzag", "striped"):
        y = _rand((S, 3, 2), 90)
        assert np.array_equal(oracle.restore(oracle.reorder(y, P, lay), P, lay), y)


def test_work_counts_golden():
    g = json.load(open(os.path.join(GOLDEN, "zigzag_work_p4.json")))
    P = g["P"]
    contiguous = {r: [2 * r, 2 * r + 1] for r in range(P)}
    zigzag = {r: [r, 2 * P - 1 - r] for r in range(P)}
    assert [oracle.work(contiguous[r]) for r in range(P)] == g["work_contiguous"]
    assert [oracle.work(zigzag[r]) for r in range(P)] == g["work_zigzag"]
    assert oracle.rank_visible_pairs(g["S"], P, "zigzag") == g["zigzag_visible_pairs_per_rank"]
    q, k, v = make_qkv()
    _, _, counts = oracle.ring_attention(q.numpy(), k.numpy(), v.numpy(), P, "contiguous")
    assert counts == g["ring_blocks_contiguous"]


@pytest.mark.parametrize("S,P", [(32, 4), (64, 2), (48, 3), (8192, 8)])
def test_zigzag_equal_work_closed_form(S, P):
    C = S // (2 * P)
    want = C * C * (2 * P - 1) + C * (C + 1)
    if S <= 64:
        assert oracle.rank_visible_pairs(S, P, "zigzag") == [want] * P
    # exact closed form from the mask applied block by block (cheap at any S)
    pos = oracle.rank_positions(S, P, "zigzag")
    for r in range(P):
        tot = 0
        for a in (r, 2 * P - 1 - r):
            for b in range(2 * P):
                pq = np.arange(a * C, (a + 1) * C)
                pk = np.arange(b * C, (b + 1) * C)
                if b < a:
                    tot += C * C
                elif b == a:
                    tot += oracle.visible_pairs(pq, pk)
        assert tot == want
        assert len(pos[r]) == 2 * C


@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "striped"])
@pytest.mark.parametrize("P", [2, 4])
def test_ring_restatement_equals_unpartitioned(layout, P):
    S, Hq, Hkv, D = 32, 4, 2, 8
    q, k, v = _rand((S, Hq, D), 100), _rand((S, Hkv, D), 101), _rand((S, Hkv, D), 102)
    ref_o, ref_l = oracle.attention(q, k, v, True)
    o, l, _ = oracle.ring_attention(q, k, v, P, layout)
    assert np.abs(o - ref_o).max() < 1e-12 and np.abs(l - ref_l).max() < 1e-12
    cu = cu_seqlens_from_lengths([7, 1, 13, 11])
    ref_o, ref_l = oracle.attention(q, k, v, True, cu_seqlens=cu)
    o, l, _ = oracle.ring_attention(q, k, v, P, layout, cu_seqlens=cu)
    assert np.abs(o - ref_o).max() < 1e-12 and np.abs(l - ref_l).max() < 1e-12


@pytest.mark.parametrize("Hq,Hkv,P", [(8, 8, 4), (8, 4, 2), (8, 2, 2)])
def test_ulysses_restatement_equals_unpartitioned(Hq, Hkv, P):
    S, D = 24, 8
    q, k, v = _rand((S, Hq, D), 110), _rand((S, Hkv, D), 111), _rand((S, Hkv, D), 112)
    ref_o, ref_l = oracle.attention(q, k, v, True)
    o, l = oracle.ulysses_attention(q, k, v, P)
    assert np.abs(o - ref_o).max() < 1e-12 and np.abs(l - ref_l).max() < 1e-12


@pytest.mark.parametrize("Hq,Hkv,P", [(8, 2, 4), (8, 1, 8), (4, 2, 4)])
def test_ulysses_replicated_kv_equals_unpartitioned(Hq, Hkv, P):
    # fewer key/value heads than ranks: each head is copied P/Hkv times before the exchange
    S, D = 24, 8
    q, k, v = _rand((S, Hq, D), 113), _rand((S, Hkv, D), 114), _rand((S, Hkv, D), 115)
    ref_o, ref_l = oracle.attention(q, k, v, True)
    o, l = oracle.ulysses_attention(q, k, v, P)
    assert np.abs(o - ref_o).max() < 1e-12 and np.abs(l - ref_l).max() < 1e-12


@pytest.mark.parametrize("Hq,Hkv,P,docs", [(8, 8, 4, None), (8, 4, 2, None), (8, 2, 4, None), (8, 1, 8, None),
                                           (4, 4, 2, [5, 11, 8])])
def test_ulysses_bwd_restatement_equals_unpartitioned(Hq, Hkv, P, docs):
    # the rank-by-rank Ulysses backward (replicated heads summed) is the plain gradient
    S, D = 24, 8
    q, k, v = _rand((S, Hq, D), 116), _rand((S, Hkv, D), 117), _rand((S, Hkv, D), 118)
    do = _rand((S, Hq, D), 119)
    cu = None if docs is None else cu_seqlens_from_lengths(docs)
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, True, cu_seqlens=cu)
    dq, dk, dv = oracle.ulysses_attention_bwd(q, k, v, do, P, cu_seqlens=cu)
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        assert got.shape == ref.shape
        assert np.abs(got - ref).max() < 1e-12


@pytest.mark.parametrize("Pu,Pr,layout,Hkv,docs", [(2, 2, "zigzag", 8, None), (2, 3, "contiguous", 4, None),
                                                    (4, 2, "striped", 8, None), (2, 2, "striped", 2, [9, 20, 19]),
                                                    (1, 4, "zigzag", 4, None), (4, 1, "contiguous", 4, None)])
def test_usp_restatement_equals_unpartitioned(Pu, Pr, layout, Hkv, docs):
    # Ulysses inside groups x ring across groups is plain attention; Pu = 1 is the
    # ring alone and Pr = 1 Ulysses alone
    S, Hq, D = 48, 8, 8
    q, k, v = _rand((S, Hq, D), 120), _rand((S, Hkv, D), 121), _rand((S, Hkv, D), 122)
    cu = None if docs is None else cu_seqlens_from_lengths(docs)
    ref_o, ref_l = oracle.attention(q, k, v, True, cu_seqlens=cu)
    o, l = oracle.usp_attention(q, k, v, Pu, Pr, layout, cu_seqlens=cu)
    assert np.abs(o - ref_o).max() < 1e-12 and np.abs(l - ref_l).max() < 1e-12


def _window_mask(pos_q, pos_k, window, cu=None):
    """Sliding-window visibility by scalar loops: key not after the query, fewer than
    `window` positions before it, same document."""
    m = np.zeros((len(pos_q), len(pos_k)), dtype=bool)
    for i, a in enumerate(pos_q):
        for j, b in enumerate(pos_k):
            same = True if cu is None else (np.searchsorted(cu, a, "right") == np.searchsorted(cu, b, "right"))
            m[i, j] = (b <= a) and (a - b < window) and same
    return m


@pytest.mark.parametrize("window,docs", [(1, None), (3, None), (7, [5, 9, 6]), (40, None)])
def test_sliding_window_against_sdpa_and_brute_force(window, docs):
    S, Hq, Hkv, D = 20, 4, 2, 8
    q, k, v = _rand((S, Hq, D), 130), _rand((S, Hkv, D), 131), _rand((S, Hkv, D), 132)
    cu = None if docs is None else cu_seqlens_from_lengths(docs)
    pos = np.arange(S)
    mask = _window_mask(pos, pos, window, cu)
    assert np.array_equal(oattn_mod.visible_mask(pos, pos, True, cu, window), mask)
    o, l = oracle.attention(q, k, v, True, cu_seqlens=cu, window=window)
    assert np.abs(o - _sdpa(q, k, v, mask=mask)).max() < 1e-12
    if window >= S and docs is None:  # a window longer than the sequence is plain causal attention
        ref_o, ref_l = oracle.attention(q, k, v, True)
        assert np.abs(o - ref_o).max() < 1e-13 and np.abs(l - ref_l).max() < 1e-13


def test_sliding_window_of_one_is_the_diagonal():
    # each query sees only itself: out = its own value row, lse = its own scaled score
    S, H, D = 9, 2, 4
    q, k, v = _rand((S, H, D), 133), _rand((S, H, D), 134), _rand((S, H, D), 135)
    o, l = oracle.attention(q, k, v, True, window=1)
    assert np.abs(o - v).max() < 1e-14
    assert np.abs(l - (np.sum(q * k, axis=2) / math.sqrt(D)).T).max() < 1e-13


def test_sliding_window_bwd_matches_autograd():
    S, Hq, Hkv, D, W = 15, 4, 2, 8, 5
    q, k, v, do = (_rand((S, Hq, D), 136), _rand((S, Hkv, D), 137), _rand((S, Hkv, D), 138),
                   _rand((S, Hq, D), 139))
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, True, window=W)
    mask = torch.from_numpy(_window_mask(np.arange(S), np.arange(S), W))
    qt, kt, vt = (torch.from_numpy(x).requires_grad_() for x in (q, k, v))
    G = Hq // Hkv
    o = torch.nn.functional.scaled_dot_product_attention(
        qt.permute(1, 0, 2)[None], kt.repeat_interleave(G, 1).permute(1, 0, 2)[None],
        vt.repeat_interleave(G, 1).permute(1, 0, 2)[None], attn_mask=mask)[0].permute(1, 0, 2)
    (o * torch.from_numpy(do)).sum().backward()
    for got, ref in ((dq, qt.grad), (dk, kt.grad), (dv, vt.grad)):
        assert np.abs(got - ref.numpy()).max() < 1e-11


def test_ulysses_with_window_equals_unpartitioned():
    S, Hq, Hkv, D, P, W = 24, 8, 2, 8, 4, 6
    q, k, v, do = (_rand((S, Hq, D), 140), _rand((S, Hkv, D), 141), _rand((S, Hkv, D), 142),
                   _rand((S, Hq, D), 143))
    ref_o, ref_l = oracle.attention(q, k, v, True, window=W)
    o, l = oracle.ulysses_attention(q, k, v, P, window=W)
    assert np.abs(o - ref_o).max() < 1e-12 and np.abs(l - ref_l).max() < 1e-12
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, True, window=W)
    dq, dk, dv = oracle.ulysses_attention_bwd(q, k, v, do, P, window=W)
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        assert np.abs(got - ref).max() < 1e-12


def test_ulysses_kv_replicas_counts():
    assert oracle.ulysses_kv_replicas(32, 8, 4) == 1
    assert oracle.ulysses_kv_replicas(32, 8, 16) == 2
    assert oracle.ulysses_kv_replicas(32, 1, 32) == 32
    with pytest.raises(AssertionError):
        oracle.ulysses_kv_replicas(32, 8, 12)  # 12 is neither a divisor nor a multiple of 8


def test_tiny_exact_workload_both_schemes():
    # The handbook's own data: S=32, H=8, D=16, P=4, ring and Ulysses vs unpartitioned.
    q, k, v = (t.double().numpy() for t in make_qkv())
    ref_o, ref_l = oracle.attention(q, k, v, True)
    for lay in ("contiguous", "zigzag", "striped"):
        o, l, _ = oracle.ring_attention(q, k, v, 4, lay)
        assert np.abs(o - ref_o).max() < 1e-12 and np.abs(l - ref_l).max() < 1e-12
    o, l = oracle.ulysses_attention(q, k, v, 4)
    assert np.abs(o - ref_o).max() < 1e-12 and np.abs(l - ref_l).max() < 1e-12
    # and against torch's float64 SDPA on the same values
    assert np.abs(ref_o - _sdpa(q, k, v, is_causal=True)).max() < 1e-12


# ---------------------------------------------------------------- planted mistakes (on the CPU, in the oracle)

def _mut_no_scale(q, k, v, causal=True, q_offset=0, k_offset=0, **kw):
    kw["scale"] = 1.0
    return oracle.attention(q, k, v, causal, q_offset, k_offset, **kw)


def _mut_swap_kv(q, k, v, causal=True, q_offset=0, k_offset=0, **kw):
    return oracle.attention(q, v, k, causal, q_offset, k_offset, **kw)


def _mut_gqa_modulo(q, k, v, causal=True, q_offset=0, k_offset=0, **kw):
    Hq, Hkv = np.asarray(q).shape[1], np.asarray(k).shape[1]
    if Hq == Hkv:
        return oracle.attention(q, k, v, causal, q_offset, k_offset, **kw)
    G = Hq // Hkv
    # query head h reading kv head h % Hkv instead of h // G
    idx = [(h % Hkv) for h in range(Hq)]
    kk = np.asarray(k)[:, idx]
    vv = np.asarray(v)[:, idx]
    return oracle.attention(q, kk, vv, causal, q_offset, k_offset, **kw) if G else None


def _mut_merge_weight(o1, l1, o2, l2):
    o, l = oracle.lse_merge(o1, l1, o2, l2)
    return o, l + 1e-3


def test_planted_mistakes_are_caught(monkeypatch):
    for mut in (_mut_no_scale, _mut_swap_kv, _mut_gqa_modulo):
        caught = False
        for check in (check_fwd_vs_sdpa, check_lse_closed_form, check_lse_bruteforce, check_doc_mask):
            try:
                check(mut)
            except AssertionError:
                caught = True
        assert caught, mut.__name__
    with pytest.raises(AssertionError):
        check_merge(oracle.attention, _mut_merge_weight)
    # an off-by-one causal mask (key at the query's own position hidden)
    orig = oattn_mod.visible_mask

    def shifted(pq, pk, causal=True, cu=None, window=0):
        m = orig(pq, pk, causal, cu, window)
        pq_ = np.asarray(pq)[:, None]
        pk_ = np.asarray(pk)[None, :]
        return m & ~(pk_ == pq_) | (m & False)

    monkeypatch.setattr(oattn_mod, "visible_mask", shifted)
    with pytest.raises(AssertionError):
        check_lse_closed_form(oracle.attention)
