"""Plain CPU fp64 oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, links or runs
this package: it is called by ``tests/``, by ``__graft_entry__.smoke()`` and by
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``.  It shares no
code, table or constant generator with the CUDA library.

Every function materialises the full n x n score matrix S and probability
matrix P per (batch, head) in float64 and follows the definitions printed on
the "Flash Attention原理：分块计算与重计算，如何降低O(n^2)的显存占用" page:

* forward: §一 (S = Q K^T, P = softmax(S * scale), O = P V; scale = 1/sqrt(d)
  by default), with the max-subtracted stable softmax of §四;
* online recurrence: §四 (running max m and normaliser l, old contributions
  rescaled by exp(m_old - m_new) when a new block arrives);
* stored statistics: §五 keeps only the per-row m and l; here they are merged
  into one natural-log logsumexp lse = m + ln l;
* backward: §五 / FAQ Q19 state that the gradients follow the chain rule but
  print no formulas; the oracle writes out the analytic gradient of
  softmax-then-matmul (dV = P^T dO, dP = dO V^T, dS = P * (dP - rowsum(P*dP)),
  dQ = scale dS K, dK = scale dS^T Q).

Pins: ``tests/test_oracle.py`` checks every function against closed forms,
invariants, brute-force finite differences and an independent library
implementation (torch's CPU float64 SDPA with autograd).
"""
from .sdpa import (
    attention_forward,
    attention_forward_rows,
    attention_forward_online,
    attention_backward,
    attention_decode,
    attention_decode_paged,
    attention_cross_backward,
    attention_varlen_forward,
    attention_varlen_backward,
    attention_masked_forward,
    attention_masked_backward,
    visibility,
    merge_splits,
    softmax_rows,
    softmax_two_block,
    gqa_kv_head,
    score_matrix_bytes,
    row_stat_bytes,
)

__all__ = [
    "attention_forward",
    "attention_forward_rows",
    "attention_forward_online",
    "attention_backward",
    "attention_decode",
    "attention_decode_paged",
    "attention_cross_backward",
    "attention_varlen_forward",
    "attention_varlen_backward",
    "attention_masked_forward",
    "attention_masked_backward",
    "visibility",
    "merge_splits",
    "softmax_rows",
    "softmax_two_block",
    "gqa_kv_head",
    "score_matrix_bytes",
    "row_stat_bytes",
]
