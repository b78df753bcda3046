"""CPU float64 oracle for block causal attention with log-sum-exp.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this module; only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg do.
It shares no code with the CUDA path.

The definition followed is the ``attention(q, k, v, causal, q_offset,
k_offset)`` function of the handbook chapter "Context parallelism: Ring
Attention and Ulysses", section "Which operations partition directly":

* scores[h, i, j] = (q_i . k_j) / sqrt(D)   (einsum "qhd,khd->hqk", scale 1/sqrt(D))
* causal: a key whose position is after the query's position is set to -inf
  (positions are the block's offset in the full sequence plus the row index)
* lse[h, i] = logsumexp_j scores[h, i, j]   (natural log, layout [H, Sq])
* out[i, h, :] = sum_j exp(scores[h, i, j] - lse[h, i]) v_j   (layout [Sq, H, D])

Readings where the page is silent (each is listed in the design notes):

* Positions may be any integer arrays; the affine form offset + stride*index
  covers contiguous (stride 1) and striped (stride P) blocks.
* Packed documents ("Add Packing Support for Context Parallelism (Ring
  Attention) #2906"): a key is visible only when it lies in the same document
  as the query (document boundaries from ``cu_seqlens`` over positions).
* Grouped-query attention: query head h reads key/value head h // G, G = Hq/Hkv.
* A row with no visible key has lse = -inf and out = 0 (the page's code would
  give NaN there; its ring never forms such a row).

The backward is the exact derivative of the definition above (the pages give no
backward); it uses the same visibility rule.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "positions",
    "doc_index",
    "visible_mask",
    "attention",
    "attention_bwd",
    "visible_pairs",
]


def positions(n: int, offset: int = 0, stride: int = 1) -> np.ndarray:
    """Global sequence positions of a block's rows: offset + stride * i."""
    return offset + stride * np.arange(n, dtype=np.int64)


def doc_index(pos: np.ndarray, cu_seqlens) -> np.ndarray:
    """Index of the packed document that holds each position (cu_seqlens[d] <= pos < cu_seqlens[d+1])."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    return np.searchsorted(cu, pos, side="right") - 1


def visible_mask(pos_q: np.ndarray, pos_k: np.ndarray, causal: bool = True, cu_seqlens=None,
                 window: int = 0) -> np.ndarray:
    """Boolean [Sq, Sk]: True where query i may attend to key j.

    Causal rule from the handbook's ``attention``: masked when key position > query position.
    Document rule (packing): masked when the two positions lie in different documents.
    Sliding window (window > 0, with the causal rule; the transformers pull request's
    mask tests): masked when the key lies window or more positions before the query,
    so a query sees itself and the window - 1 keys before it.
    """
    pq = np.asarray(pos_q, dtype=np.int64)[:, None]
    pk = np.asarray(pos_k, dtype=np.int64)[None, :]
    vis = np.ones((pq.shape[0], pk.shape[1]), dtype=bool)
    if causal:
        vis &= ~(pk > pq)
    if window:
        assert causal, "a sliding window is defined with the causal rule"
        vis &= (pq - pk) < window
    if cu_seqlens is not None:
        vis &= doc_index(pq, cu_seqlens) == doc_index(pk, cu_seqlens)
    return vis


def _as_f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor (bf16 included): exact upcast
        import torch

        return x.detach().to(torch.float64).cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def _resolve_positions(Sq, Sk, q_offset, k_offset, q_stride, k_stride, pos_q, pos_k):
    if pos_q is None:
        pos_q = positions(Sq, q_offset, q_stride)
    if pos_k is None:
        pos_k = positions(Sk, k_offset, k_stride)
    pos_q = np.asarray(pos_q, dtype=np.int64)
    pos_k = np.asarray(pos_k, dtype=np.int64)
    assert pos_q.shape == (Sq,) and pos_k.shape == (Sk,)
    return pos_q, pos_k


def attention(q, k, v, causal: bool = True, q_offset: int = 0, k_offset: int = 0, *,
              q_stride: int = 1, k_stride: int = 1, pos_q=None, pos_k=None,
              cu_seqlens=None, scale: float | None = None, row_block: int = 1024, window: int = 0):
    """Forward attention of one (query block, key/value block) pair.

    q: [Sq, Hq, D]; k, v: [Sk, Hkv, D] (any real dtype; computed in float64).
    Returns (out [Sq, Hq, D] float64, lse [Hq, Sq] float64).

    Rows are processed ``row_block`` at a time per head only to bound memory;
    every row's value is the definition applied to that row alone.
    """
    q = _as_f64(q)
    k = _as_f64(k)
    v = _as_f64(v)
    Sq, Hq, D = q.shape
    Sk, Hkv, _ = k.shape
    assert Hq % Hkv == 0, "query heads must be a multiple of key/value heads"
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    pos_q, pos_k = _resolve_positions(Sq, Sk, q_offset, k_offset, q_stride, k_stride, pos_q, pos_k)

    out = np.zeros((Sq, Hq, D), dtype=np.float64)
    lse = np.full((Hq, Sq), -np.inf, dtype=np.float64)
    if Sq == 0:
        return out, lse
    for i0 in range(0, Sq, row_block):
        i1 = min(Sq, i0 + row_block)
        vis = visible_mask(pos_q[i0:i1], pos_k, causal, cu_seqlens, window)
        any_vis = vis.any(axis=1)
        for h in range(Hq):
            hk = h // G
            s = (q[i0:i1, h, :] @ k[:, hk, :].T) * scale
            s = np.where(vis, s, -np.inf)
            m = np.max(s, axis=1, initial=-np.inf)
            m_safe = np.where(any_vis, m, 0.0)
            e = np.exp(s - m_safe[:, None])  # exp(-inf) = 0 on masked entries
            l = e.sum(axis=1)
            with np.errstate(divide="ignore"):
                row_lse = np.where(any_vis, m_safe + np.log(l), -np.inf)
            lse[h, i0:i1] = row_lse
            p = np.where(any_vis[:, None], np.exp(s - np.where(any_vis, row_lse, 0.0)[:, None]), 0.0)
            out[i0:i1, h, :] = p @ v[:, hk, :]
    return out, lse


def attention_bwd(q, k, v, dout, causal: bool = True, q_offset: int = 0, k_offset: int = 0, *,
                  q_stride: int = 1, k_stride: int = 1, pos_q=None, pos_k=None,
                  cu_seqlens=None, scale: float | None = None, row_block: int = 1024, window: int = 0):
    """Gradients (dq, dk, dv) of sum(dout * out) for ``attention`` above, float64.

    With P = softmax of the visible scores and O = P v:
      dV_j  = sum_i P_ij dO_i
      dP_ij = dO_i . v_j
      dS_ij = P_ij (dP_ij - Delta_i),  Delta_i = sum_d dO_id O_id = sum_j P_ij dP_ij
      dQ_i  = scale * sum_j dS_ij k_j
      dK_j  = scale * sum_i dS_ij q_i
    dK and dV of a key/value head are summed over the G query heads that read it.
    """
    q = _as_f64(q)
    k = _as_f64(k)
    v = _as_f64(v)
    do = _as_f64(dout)
    Sq, Hq, D = q.shape
    Sk, Hkv, _ = k.shape
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    pos_q, pos_k = _resolve_positions(Sq, Sk, q_offset, k_offset, q_stride, k_stride, pos_q, pos_k)

    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for i0 in range(0, Sq, row_block):
        i1 = min(Sq, i0 + row_block)
        vis = visible_mask(pos_q[i0:i1], pos_k, causal, cu_seqlens, window)
        any_vis = vis.any(axis=1)
        for h in range(Hq):
            hk = h // G
            s = (q[i0:i1, h, :] @ k[:, hk, :].T) * scale
            s = np.where(vis, s, -np.inf)
            m = np.where(any_vis, np.max(s, axis=1, initial=-np.inf), 0.0)
            e = np.exp(s - m[:, None])
            l = e.sum(axis=1)
            p = np.where(any_vis[:, None], e / np.where(any_vis, l, 1.0)[:, None], 0.0)
            o = p @ v[:, hk, :]
            dO = do[i0:i1, h, :]
            dv[:, hk, :] += p.T @ dO
            dp = dO @ v[:, hk, :].T
            delta = np.sum(dO * o, axis=1)
            ds = p * (dp - delta[:, None])
            dq[i0:i1, h, :] += scale * (ds @ k[:, hk, :])
            dk[:, hk, :] += scale * (ds.T @ q[i0:i1, h, :])
    return dq, dk, dv


def visible_pairs(pos_q, pos_k, causal: bool = True, cu_seqlens=None, window: int = 0) -> int:
    """Number of visible (query, key) pairs of one block pair (per head)."""
    return int(visible_mask(pos_q, pos_k, causal, cu_seqlens, window).sum())
