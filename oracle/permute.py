"""The Ulysses / IntraSP layout permutation, as an explicit index loop.

HSAP, Sec. 2.2.2 "Intra-group Sequence Parallelism": before attention, the
blocks Q_i, K_i, V_i in R^{n x H x d} (n = N / P sequence rows per group) are
moved by an all-to-all to blocks in R^{N x h x d} with h = H / P heads per
group; another all-to-all moves them back afterwards.  BASP, Sec. II-C
"DeepSpeed Ulysses", describes the same exchange.  With all P sequence
shards stacked on one device ([N, H, d], shard r = rows r*n .. (r+1)*n), the
all-to-all's receive side is, for head group g and local head j:

  out[g, t, j, :] = in[t, g*h + j, :]        out has shape [P, N, h, d]

and the inverse (head -> seq) is in[t, g*h + j, :] = out[g, t, j, :].
"""
from __future__ import annotations

import numpy as np


def seq2head(x, P: int):
    T, H, d = x.shape
    assert H % P == 0
    h = H // P
    out = np.empty((P, T, h, d), dtype=x.dtype)
    for g in range(P):
        for j in range(h):
            for t in range(T):
                out[g, t, j, :] = x[t, g * h + j, :]
    return out


def head2seq(y, P: int):
    Pg, T, h, d = y.shape
    assert Pg == P
    x = np.empty((T, P * h, d), dtype=y.dtype)
    for g in range(P):
        for j in range(h):
            for t in range(T):
                x[t, g * h + j, :] = y[g, t, j, :]
    return x
