"""Oracle: plain, slow, CPU float64 restatement of causal context-parallel attention.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's CPU
baseline import this package; the library never does, and the two share no
code.  Each function cites the passage of the handbook chapter "Context
parallelism: Ring Attention and Ulysses" (or of the MaxText packing pull
request) that it follows.  Every function here is pinned by a ``-m "not gpu"``
test against something other than itself (a library routine, a closed form,
brute force on tiny inputs, or an invariant of the method).
"""
from .block_attention import attention, attention_bwd, doc_index, positions, visible_mask, visible_pairs
from .context import (
    head_to_seq,
    lse_merge,
    rank_positions,
    rank_visible_pairs,
    reorder,
    restore,
    ring_attention,
    seq_to_head,
    ulysses_attention,
    ulysses_attention_bwd,
    ulysses_head2seq,
    ulysses_kv_replicas,
    ulysses_seq2head,
    usp_attention,
    work,
)

__all__ = [
    "attention", "attention_bwd", "doc_index", "positions", "visible_mask", "visible_pairs",
    "head_to_seq", "lse_merge", "rank_positions", "rank_visible_pairs", "reorder", "restore",
    "ring_attention", "seq_to_head", "ulysses_attention", "ulysses_attention_bwd", "ulysses_head2seq",
    "ulysses_kv_replicas", "ulysses_seq2head", "usp_attention", "work",
]
