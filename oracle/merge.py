"""Log-sum-exp merge of partial attention results, in float64.

Ring-style InterSP keeps each rank's queries and streams key/value blocks
past them, accumulating the partial results "in an online manner" (HSAP,
Sec. 2.2.1, citing Milakov and Gimelshein's online softmax); HSAP's
Limitations name this step the "rescale" that a fused kernel could absorb.
Given partials (out_i, lse_i) of the same queries over disjoint key sets,
the exact result over the union of the key sets is, per query row and head:

  m = max_i lse_i
  m = -inf          ->  out = 0, lse = -inf   (no key anywhere)
  otherwise         ->  lse = m + ln sum_i exp(lse_i - m)
                        out = sum_i exp(lse_i - lse) * out_i

(the softmax normaliser of the union is the sum of the partial normalisers,
and each partial output is already normalised by its own).
"""
from __future__ import annotations

import numpy as np


def lse_merge(outs, lses):
    """outs: list of [T, H, d]; lses: list of [H, T].  Returns (out, lse)."""
    O = np.stack([np.asarray(o, dtype=np.float64) for o in outs])     # [n, T, H, d]
    L = np.stack([np.asarray(l, dtype=np.float64) for l in lses])     # [n, H, T]
    m = L.max(axis=0)                                                 # [H, T]
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    with np.errstate(divide="ignore"):      # log(0) only where every lse_i is -inf
        lse = np.where(empty, -np.inf, m_safe + np.log(np.exp(L - m_safe).sum(axis=0)))
    w = np.where(empty, 0.0, np.exp(L - np.where(empty, 0.0, lse)))  # [n, H, T]
    out = np.einsum("nht,nthd->thd", w, O)
    return out, lse
