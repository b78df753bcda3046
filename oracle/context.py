"""CPU float64 oracle for the context-parallel pieces: the log-sum-exp merge,
the Ulysses sequence<->head exchange, the load-balancing reorders, and plain
restatements of the ring and Ulysses schemes over P virtual ranks.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``); shares no code with the
CUDA path.

Sources (handbook chapter "Context parallelism: Ring Attention and Ulysses"):

* "Ring Attention: passing the KV once around a ring": at step s rank r holds
  the key/value block of rank (r - s) mod P; a block contributes only if it is
  not later than the query block; two partial results merge as
  lse = log(e^lse1 + e^lse2), o = o1 e^(lse1 - lse) + o2 e^(lse2 - lse).
* "Ulysses: transposing between the sequence and the heads": seq_to_head turns
  [S/P, H, D] on each rank (all heads, one slice of the sequence) into
  [S, H/P, D] (whole sequence, H/P heads) with one all-to-all; head_to_seq is
  its inverse.
* "The zigzag partition": 2P blocks, rank r holds blocks r and 2P-1-r; the
  ``work`` count of a rank is the sum over its query blocks of (index + 0.5).

The striped strategy is only named in the MaxText pull request "Add Packing
Support for Context Parallelism (Ring Attention) #2906" (ReorderStrategy
AUTO / DUAL_CHUNK_SWAP / STRIPED).  Reading taken: token-granular round robin,
rank r holds global positions r, r+P, r+2P, ...  DUAL_CHUNK_SWAP is the zigzag
partition above.
"""
from __future__ import annotations

import numpy as np

from .block_attention import attention, attention_bwd, visible_pairs

__all__ = [
    "lse_merge",
    "seq_to_head",
    "head_to_seq",
    "ulysses_seq2head",
    "ulysses_head2seq",
    "rank_positions",
    "reorder",
    "restore",
    "ring_attention",
    "ulysses_attention",
    "ulysses_attention_bwd",
    "ulysses_kv_replicas",
    "usp_attention",
    "work",
    "rank_visible_pairs",
]


def lse_merge(o1, lse1, o2, lse2):
    """Merge two partial attentions over disjoint key sets.

    o*: [Sq, H, D]; lse*: [H, Sq].  Returns (o, lse).  The ring section merges
    with ``logaddexp`` and the two exp weights (lse transposed to [Sq, H, 1]).
    A row where both parts are empty (-inf) stays empty: lse = -inf, o = 0.
    """
    o1 = np.asarray(o1, dtype=np.float64)
    o2 = np.asarray(o2, dtype=np.float64)
    lse1 = np.asarray(lse1, dtype=np.float64)
    lse2 = np.asarray(lse2, dtype=np.float64)
    new = np.logaddexp(lse1, lse2)
    empty = np.isneginf(new)
    safe = np.where(empty, 0.0, new)
    w1 = np.where(empty, 0.0, np.exp(lse1 - safe))
    w2 = np.where(empty, 0.0, np.exp(lse2 - safe))
    o = o1 * w1.T[..., None] + o2 * w2.T[..., None]
    return o, new


def _all_to_all(send):
    """send[r][p] is what rank r sends to rank p; returns recv[p][r]."""
    P = len(send)
    return [[send[r][p] for r in range(P)] for p in range(P)]


def seq_to_head(x_per_rank, P):
    """Ulysses first exchange, restated rank by rank.

    x_per_rank[r]: [S/P, H, D] (rank r's slice of the sequence, all heads).
    Each rank groups its heads by destination (group p = the p-th share of the
    heads) and sends group p to rank p; rank p stacks what it receives in source
    order, which is sequence order.  Returns a list of P arrays [S, H/P, D].
    """
    C, H, D = x_per_rank[0].shape
    send = [np.asarray(x).reshape(C, P, H // P, D).transpose(1, 0, 2, 3) for x in x_per_rank]
    recv = _all_to_all(send)
    return [np.concatenate(recv[p], axis=0) for p in range(P)]


def head_to_seq(x_per_rank, P):
    """Inverse of ``seq_to_head``: list of P arrays [S, H/P, D] -> list of [S/P, H, D]."""
    S, Hp, D = x_per_rank[0].shape
    C = S // P
    send = [np.asarray(x).reshape(P, C, Hp, D) for x in x_per_rank]  # group p = p-th slice of the sequence
    recv = _all_to_all(send)
    # rank p holds, from every source rank r, r's heads for p's slice: [P(src), C, H/P, D]
    return [np.stack(recv[p], axis=0).transpose(1, 0, 2, 3).reshape(C, P * Hp, D) for p in range(P)]


def ulysses_seq2head(x, P):
    """Whole-buffer form used by the library: x [S, H, D] (ranks' slices in
    order) -> y [P, S, H/P, D], y[p] = what rank p holds after the exchange."""
    S = x.shape[0]
    C = S // P
    parts = seq_to_head([x[r * C:(r + 1) * C] for r in range(P)], P)
    return np.stack(parts, axis=0)


def ulysses_head2seq(y, P):
    """Inverse whole-buffer form: y [P, S, H/P, D] -> x [S, H, D]."""
    parts = head_to_seq([y[p] for p in range(P)], P)
    return np.concatenate(parts, axis=0)


def rank_positions(S: int, P: int, layout: str):
    """Global positions held by each virtual rank, in the order the rank stores them.

    contiguous: rank r holds [rC, (r+1)C), C = S/P.
    zigzag (DUAL_CHUNK_SWAP): C = S/(2P); rank r holds block r then block 2P-1-r.
    striped: rank r holds r, r+P, r+2P, ... (S/P tokens).
    """
    if layout == "contiguous":
        assert S % P == 0
        C = S // P
        return [np.arange(r * C, (r + 1) * C, dtype=np.int64) for r in range(P)]
    if layout in ("zigzag", "dual_chunk_swap"):
        assert S % (2 * P) == 0
        C = S // (2 * P)
        return [np.concatenate([np.arange(r * C, (r + 1) * C), np.arange((2 * P - 1 - r) * C, (2 * P - r) * C)]).astype(np.int64)
                for r in range(P)]
    if layout == "striped":
        assert S % P == 0
        return [np.arange(r, S, P, dtype=np.int64) for r in range(P)]
    raise ValueError(layout)


def reorder(x, P: int, layout: str):
    """x [S, ...] in sequence order -> ranks' holdings concatenated in rank order."""
    S = x.shape[0]
    idx = np.concatenate(rank_positions(S, P, layout))
    return np.asarray(x)[idx]


def restore(y, P: int, layout: str):
    """Inverse of ``reorder``."""
    S = y.shape[0]
    idx = np.concatenate(rank_positions(S, P, layout))
    x = np.empty_like(np.asarray(y))
    x[idx] = y
    return x


def ring_attention(q, k, v, P: int, layout: str = "contiguous", causal: bool = True, cu_seqlens=None):
    """The ring scheme over P virtual ranks, restated from the ring section.

    Rank r keeps its query positions; at step s it holds the key/value block of
    rank src = (r - s) mod P, computes the partial attention of its queries
    against that block (with the block's global positions) when any pair is
    visible, and merges it into its running (out, lse).  Returns
    (out [S, Hq, D], lse [Hq, S]) in sequence order and the per-rank count of
    blocks actually computed.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    S, Hq, D = q.shape
    pos = rank_positions(S, P, layout)
    out = np.zeros((S, Hq, D))
    lse = np.full((Hq, S), -np.inf)
    counts = []
    for r in range(P):
        pr = pos[r]
        o_acc, l_acc = None, None
        computed = 0
        src = r
        for _step in range(P):
            ps = pos[src]
            if visible_pairs(pr, ps, causal, cu_seqlens) > 0:
                o, l = attention(q[pr], k[ps], v[ps], causal, pos_q=pr, pos_k=ps, cu_seqlens=cu_seqlens)
                if o_acc is None:
                    o_acc, l_acc = o, l
                else:
                    o_acc, l_acc = lse_merge(o_acc, l_acc, o, l)
                computed += 1
            src = (src - 1) % P
        counts.append(computed)
        if o_acc is not None:
            out[pr] = o_acc
            lse[:, pr] = l_acc
    return out, lse, counts


def ulysses_kv_replicas(Hq: int, Hkv: int, P: int) -> int:
    """Copies of each key/value head in the Ulysses exchange.

    The exchange gives every rank H/P heads, so with fewer key/value heads than
    ranks the key/value heads are replicated first ("replicating the KV by
    group", the handbook's note on grouped-query attention under Ulysses):
    each head is repeated R = P / Hkv times, consecutive copies, so that rank p
    receives copy p of the repeated heads, which is original head p // R -- the
    head its query heads p*Hq/P ... read under the consecutive grouping.  R = 1
    when Hkv % P == 0 (no replication)."""
    assert Hq % P == 0, "Ulysses degree is limited by the query heads"
    if Hkv % P == 0:
        return 1
    assert P % Hkv == 0, "replication needs P to be a multiple of the key/value heads"
    return P // Hkv


def _ulysses_inputs(q, k, v, P: int):
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    R = ulysses_kv_replicas(q.shape[1], k.shape[1], P)
    if R > 1:
        k = np.repeat(k, R, axis=1)
        v = np.repeat(v, R, axis=1)
    return q, k, v, R


def ulysses_attention(q, k, v, P: int, causal: bool = True, cu_seqlens=None, window: int = 0):
    """The Ulysses scheme over P virtual ranks, restated from the Ulysses section.

    Each rank's slice of q, k, v goes through ``seq_to_head``; rank p runs
    full-sequence attention over its H/P query heads (and Hkv/P key/value
    heads, or the one replicated head, ``ulysses_kv_replicas``);
    ``head_to_seq`` brings the output back.  Returns (out [S, Hq, D], lse [Hq, S]).
    """
    q, k, v, _ = _ulysses_inputs(q, k, v, P)
    S = q.shape[0]
    C = S // P
    sl = [slice(r * C, (r + 1) * C) for r in range(P)]
    qh = seq_to_head([q[s] for s in sl], P)
    kh = seq_to_head([k[s] for s in sl], P)
    vh = seq_to_head([v[s] for s in sl], P)
    outs, lses = [], []
    for p in range(P):
        o, l = attention(qh[p], kh[p], vh[p], causal, cu_seqlens=cu_seqlens, window=window)
        outs.append(o)
        lses.append(l)
    out = np.concatenate(head_to_seq(outs, P), axis=0)
    lse = np.concatenate(lses, axis=0)  # rank p holds query heads [p*Hq/P, (p+1)*Hq/P)
    return out, lse


def ulysses_attention_bwd(q, k, v, dout, P: int, causal: bool = True, cu_seqlens=None, window: int = 0):
    """Backward of the Ulysses scheme, restated rank by rank.

    head_to_seq is the backward of seq_to_head (a permutation), so the gradients
    travel the same exchange as the outputs: q, k, v and dout go through
    ``seq_to_head``; rank p takes the exact gradient of its full-sequence
    attention; ``head_to_seq`` brings dq, dk, dv back.  Replicated key/value
    heads (``ulysses_kv_replicas``) sum their copies' gradients.  Returns
    (dq [S, Hq, D], dk [S, Hkv, D], dv [S, Hkv, D])."""
    Hkv = np.asarray(k).shape[1]
    q, k, v, R = _ulysses_inputs(q, k, v, P)
    dout = np.asarray(dout, dtype=np.float64)
    S = q.shape[0]
    C = S // P
    sl = [slice(r * C, (r + 1) * C) for r in range(P)]
    qh, kh, vh, doh = (seq_to_head([x[s] for s in sl], P) for x in (q, k, v, dout))
    dqs, dks, dvs = [], [], []
    for p in range(P):
        dq_p, dk_p, dv_p = attention_bwd(qh[p], kh[p], vh[p], doh[p], causal, cu_seqlens=cu_seqlens,
                                         window=window)
        dqs.append(dq_p)
        dks.append(dk_p)
        dvs.append(dv_p)
    dq = np.concatenate(head_to_seq(dqs, P), axis=0)
    dk = np.concatenate(head_to_seq(dks, P), axis=0)
    dv = np.concatenate(head_to_seq(dvs, P), axis=0)
    if R > 1:  # the copies of a head are consecutive
        dk = dk.reshape(S, Hkv, R, -1).sum(axis=2)
        dv = dv.reshape(S, Hkv, R, -1).sum(axis=2)
    return dq, dk, dv


def usp_attention(q, k, v, P_ulysses: int, P_ring: int, layout: str = "zigzag", causal: bool = True,
                  cu_seqlens=None):
    """Ulysses inside groups of P_ulysses ranks, the ring across P_ring groups
    (the chapter's note that the two schemes compose: heads are split inside a
    group, the key/value blocks travel around the ring between groups).

    Group g holds the positions the ring layout gives ring rank g
    (``rank_positions(S, P_ring, layout)``); inside the group, Ulysses rank u
    holds the u-th contiguous share of the group's tokens with every head, and
    ``seq_to_head`` inside the group gives it all of the group's tokens for
    head share u.  For each head share the ring runs across the groups exactly
    as in ``ring_attention`` (step s: group g holds the key/value tokens of
    group (g - s) mod P_ring, merged with lse_merge), and ``head_to_seq``
    inside the group brings the output back.  Returns (out [S, Hq, D],
    lse [Hq, S]) in sequence order.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    S, Hq, D = q.shape
    Hkv = k.shape[1]
    Pu, Pr = P_ulysses, P_ring
    assert Hq % Pu == 0 and Hkv % Pu == 0, "Ulysses degree is limited by the head counts"
    pos = rank_positions(S, Pr, layout)
    n_g = len(pos[0])
    assert n_g % Pu == 0
    Cu = n_g // Pu
    # the exchange inside each group: head share u of the group's tokens
    shares = []
    for g in range(Pr):
        parts = [(x[pos[g]][r * Cu:(r + 1) * Cu]) for r in range(Pu) for x in (q, k, v)]
        qh = seq_to_head(parts[0::3], Pu)
        kh = seq_to_head(parts[1::3], Pu)
        vh = seq_to_head(parts[2::3], Pu)
        shares.append((qh, kh, vh))
    out = np.zeros((S, Hq, D))
    lse = np.full((Hq, S), -np.inf)
    Hqu = Hq // Pu
    for g in range(Pr):
        outs_g = []
        for u in range(Pu):
            qg = shares[g][0][u]
            o_acc, l_acc = None, None
            src = g
            for _step in range(Pr):  # the ring across groups, for head share u
                ks, vs = shares[src][1][u], shares[src][2][u]
                if visible_pairs(pos[g], pos[src], causal, cu_seqlens) > 0:
                    o, l = attention(qg, ks, vs, causal, pos_q=pos[g], pos_k=pos[src], cu_seqlens=cu_seqlens)
                    if o_acc is None:
                        o_acc, l_acc = o, l
                    else:
                        o_acc, l_acc = lse_merge(o_acc, l_acc, o, l)
                src = (src - 1) % Pr
            if o_acc is None:
                o_acc, l_acc = np.zeros((n_g, Hqu, D)), np.full((Hqu, n_g), -np.inf)
            outs_g.append(o_acc)
            lse[u * Hqu:(u + 1) * Hqu, pos[g]] = l_acc
        out[pos[g]] = np.concatenate(head_to_seq(outs_g, Pu), axis=0)
    return out, lse


def work(query_chunks):
    """The zigzag section's load count: each query block needs (its index) full
    key blocks plus half of the diagonal one."""
    return sum(qc + 0.5 for qc in query_chunks)


def rank_visible_pairs(S: int, P: int, layout: str, causal: bool = True, cu_seqlens=None):
    """Exact number of visible (query, key) pairs each rank computes (per head)."""
    pos = rank_positions(S, P, layout)
    allpos = np.arange(S, dtype=np.int64)
    return [visible_pairs(pos[r], allpos, causal, cu_seqlens) for r in range(P)]
