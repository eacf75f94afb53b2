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

BASP, Sec. IV "Batch-aware group formation", "Batch Aware Sequence
Partitioning" (Alg. 2) and "Subgroup all-to-all": with a micro-batch of B
sequences of L tokens on N = B K ranks, rank r holds tokens
(r mod K) L/K .. of sequence floor(r / K), and each group of K ranks runs its
own K-way all-to-all on its one sequence.  With the batch stacked on one
device ([B L, H, d], sequence b = rows b L .. (b + 1) L), the receive side of
all B groups is, for local rank (head group) g and local head j (h = H / K):

  out[b, g, t, j, :] = in[b L + t, g*h + j, :]    out has shape [B, K, L, h, d]

so each group's exchange touches its own sequence only; B = 1 is seq2head
with P = K.
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


def seq2head_groups(x, B: int, K: int):
    """The B independent K-way exchanges of a batch-aware (BASP) subgroup
    all-to-all: [B L, H, d] -> [B, K, L, H / K, d]."""
    BL, H, d = x.shape
    assert BL % B == 0 and H % K == 0
    L, h = BL // B, H // K
    out = np.empty((B, K, L, h, d), dtype=x.dtype)
    for b in range(B):
        for g in range(K):
            for j in range(h):
                for t in range(L):
                    out[b, g, t, j, :] = x[b * L + t, g * h + j, :]
    return out


def head2seq_groups(y, B: int, K: int):
    """Inverse of seq2head_groups: [B, K, L, h, d] -> [B L, K h, d]."""
    Bg, Kg, L, h, d = y.shape
    assert Bg == B and Kg == K
    x = np.empty((B * L, K * h, d), dtype=y.dtype)
    for b in range(B):
        for g in range(K):
            for j in range(h):
                for t in range(L):
                    x[b * L + t, g * h + j, :] = y[b, g, t, j, :]
    return x
